// Shared host and device helpers of the MoE expert-layer library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe_topk.h"

namespace moe {

// ----------------------------------------------------------------- host side

// Records a printf-style message for moe_last_error_string() and returns `code`.
int fail(int code, const char* fmt, ...);
// Clears the calling thread's last error.
void clear_error();
// Device address of the status word for the current device (nullptr on failure).
int* status_word();
// Multiprocessor count of the current device (cached; 0 on failure).
int sm_count();
// Current device ordinal (-1 on failure).
int current_device();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launches `kern` on `s` with programmatic dependent launch allowed: the
// kernel may be scheduled while its predecessor in the stream is finishing;
// every kernel of this library starts with pdl_wait(), which returns once
// the predecessor has completed and its memory is visible.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

inline int check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return MOE_OK;
}
// the same, naming the entry point and the kernel of a multi-kernel call
inline int check_launch(const char* fn, const char* kernel) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s: %s", fn, kernel, cudaGetErrorString(e));
  return MOE_OK;
}

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kMaxSegments = 1024;
// tokens per ranking chunk: the router's top-k CTA and the dispatch row CTA
// each cover one chunk, and the route's chunk prefixes are per chunk
constexpr int kRouteChunk = 16;

// Internal entry points shared between translation units (not exported).
struct GroupedSegs {
  int num_seg;
  const int32_t* seg_offsets;
  const int32_t* seg_expert;  // may be null (identity)
};

// Dense "row" GEMM with K-major A [M,K] and K-major B [N,K], both bf16, one
// segment [0,M) and fp32 accumulation; epilogue out[m,n] = bf16(acc + add[m,n])
// with `add` fp32 [M,N] (row stride N).  Used by the router backward.
int launch_dense_add_bf16(const void* A, const void* B, const float* add, void* out, int M, int N,
                          int K, cudaStream_t stream);
// out[g] (fp32 [groups, M, N]) = sum over the K rows of segment g of A^T B,
// with A [K_rows, M] and B [K_rows, N] bf16 row-major (both MN-major).  Used
// by the router backward (split-K partials, overwrite).  `maps` is device
// scratch of dw_split_maps_bytes(num_seg) bytes, 128-byte aligned, for the
// per-segment TMA descriptors.
size_t dw_split_maps_bytes(int num_seg);
int launch_dw_split(const void* A, const void* B, int K_rows, int M, int N,
                    const int32_t* seg_offsets, int num_seg, float* out, void* maps,
                    cudaStream_t stream);

// ---------------------------------------------------------------- device side

// Programmatic dependent launch: wait for the predecessor grid (its writes
// visible), then let the successor grid be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&p);
}

__device__ __forceinline__ void set_status(int* status, int bits) {
  if (status) atomicOr(status, bits);
}

// e4m3 row quantisation ("TorchTitan FSDP2 完全指南", performance table: FP8
// matmuls; the recipe is the reading stated in moe_topk.h): the largest |a|
// of eight bf16 values, the row scale from the row's largest |a|, and eight
// codes e4m3(a / s) (IEEE division, round to nearest even, saturated).
__device__ __forceinline__ float amax_bf16x8(uint4 v, float m) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(bf16lo(w[i])), fabsf(bf16hi(w[i]))));
  return m;
}
__device__ __forceinline__ float e4m3_row_scale(float amax) { return amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f; }
__device__ __forceinline__ uint2 e4m3_codes8(uint4 v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float2 a = make_float2(__fdiv_rn(bf16lo(w[2 * h]), s), __fdiv_rn(bf16hi(w[2 * h]), s));
    const float2 b = make_float2(__fdiv_rn(bf16lo(w[2 * h + 1]), s), __fdiv_rn(bf16hi(w[2 * h + 1]), s));
    const uint32_t ca = __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3);
    const uint32_t cb = __nv_cvt_float2_to_fp8x2(b, __NV_SATFINITE, __NV_E4M3);
    out[h] = (ca & 0xFFFFu) | (cb << 16);
  }
  return make_uint2(out[0], out[1]);
}

}  // namespace moe
