// Per-row e4m3 quantisation of bf16 tensors (sm_103a).
//
// FP8 reading of "TorchTitan FSDP2 完全指南", performance table (FP8 matmuls
// in training; the page gives no recipe): one fp32 scale per stored row,
// s = amax / 448 (1 for an all-zero row), codes e4m3(a / s) rounded to
// nearest even and saturated at 448.  Rows are token rows of x, permuted
// rows of h, or output channels of the expert weights ([E * out, in]).
//
// One warp per row reads the row once into registers (NC 16-byte vectors
// per lane, NC picked from the row length so that short rows keep few
// registers and many warps per SM; rows longer than 2048 elements are read
// twice, the second time from L2), reduces |a| to amax with shuffles, then
// writes the codes with 8-byte stores and the scale.  It moves 3 bytes per
// element; the exact IEEE division per element (which makes the codes a
// pure function of the input bits) costs about as much again: h at
// 32768 x 768 takes 16 us with it and 8 us with a multiplication.
#include <algorithm>

#include "common.cuh"

namespace {

constexpr int kQuantWarps = 8;   // rows per 256-thread block

// Blocks per SM each quantiser instantiation is compiled for.
__host__ __device__ constexpr int quant_blocks_per_sm(int nc) { return nc <= 1 ? 6 : (nc <= 3 ? 4 : (nc <= 4 ? 3 : 2)); }

// NC: 16-byte vectors (8 bf16 each) a lane holds in registers per row.  The
// grid holds what is resident at once; each warp walks rows
// warp, warp + W, warp + 2W, ... (W warps in the grid) and loads its next
// row while it reduces and converts the current one.
template <int NC>
__global__ void __launch_bounds__(32 * kQuantWarps, quant_blocks_per_sm(NC))
    quantize_rows_e4m3_kernel(const __nv_bfloat16* __restrict__ a, int rows, int cols,
                              uint8_t* __restrict__ q, float* __restrict__ scale) {
  moe::pdl_wait();
  moe::pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int stride = gridDim.x * kQuantWarps;
  const int nv = cols / 8;
  auto load = [&](int row, uint4 (&c)[NC]) {
    const uint4* src = reinterpret_cast<const uint4*>(a + (size_t)row * cols);
#pragma unroll
    for (int i = 0; i < NC; ++i) {
      const int v = lane + 32 * i;
      c[i] = v < nv ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
    }
  };
  int row = blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  uint4 cur[NC], nxt[NC];
  load(row, cur);
  for (; row < rows; row += stride) {
    if (row + stride < rows) load(row + stride, nxt);
    const uint4* src = reinterpret_cast<const uint4*>(a + (size_t)row * cols);
    uint2* dst = reinterpret_cast<uint2*>(q + (size_t)row * cols);
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < NC; ++i) m = moe::amax_bf16x8(cur[i], m);
    for (int v = lane + 32 * NC; v < nv; v += 32) m = moe::amax_bf16x8(__ldg(src + v), m);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const float s = moe::e4m3_row_scale(m);
    if (lane == 0) scale[row] = s;
#pragma unroll
    for (int i = 0; i < NC; ++i) {
      const int v = lane + 32 * i;
      if (v < nv) dst[v] = moe::e4m3_codes8(cur[i], s);
    }
    for (int v = lane + 32 * NC; v < nv; v += 32) dst[v] = moe::e4m3_codes8(__ldg(src + v), s);
#pragma unroll
    for (int i = 0; i < NC; ++i) cur[i] = nxt[i];
  }
}

}  // namespace

extern "C" int moe_quantize_rows_e4m3(const void* a, int rows, int cols, void* q, float* scale,
                                      void* stream) {
  moe::clear_error();
  const char* fn = "moe_quantize_rows_e4m3";
  if (rows < 0 || cols <= 0 || cols % 8)
    return moe::fail(MOE_ERR_INVALID_ARG, "%s: need rows>=0, cols>0, cols%%8==0 (rows=%d cols=%d)", fn,
                     rows, cols);
  if (rows == 0) return MOE_OK;
  if (!a || !q || !scale) return moe::fail(MOE_ERR_INVALID_ARG, "%s: NULL pointer argument", fn);
  if (!moe::aligned16(a) || (reinterpret_cast<uintptr_t>(q) & 7u) || (reinterpret_cast<uintptr_t>(scale) & 3u))
    return moe::fail(MOE_ERR_ALIGNMENT, "%s: a must be 16-byte, q 8-byte, scale 4-byte aligned", fn);
  const int per_lane = (cols / 8 + 31) / 32;  // 16-byte vectors per lane
  const int nc = per_lane <= 1 ? 1 : per_lane <= 2 ? 2 : per_lane <= 3 ? 3 : per_lane <= 4 ? 4 : 8;
  auto kernel = nc == 1   ? quantize_rows_e4m3_kernel<1>
                : nc == 2 ? quantize_rows_e4m3_kernel<2>
                : nc == 3 ? quantize_rows_e4m3_kernel<3>
                : nc == 4 ? quantize_rows_e4m3_kernel<4>
                          : quantize_rows_e4m3_kernel<8>;
  // one resident wave of blocks (each warp then walks several rows)
  const int sms = moe::sm_count() > 0 ? moe::sm_count() : 148;
  const int blocks = std::min((rows + kQuantWarps - 1) / kQuantWarps, sms * quant_blocks_per_sm(nc));
  cudaError_t e = moe::launch_pdl(kernel, dim3(blocks), dim3(32 * kQuantWarps), 0,
                                  static_cast<cudaStream_t>(stream),
                                  static_cast<const __nv_bfloat16*>(a), rows, cols,
                                  static_cast<uint8_t*>(q), scale);
  if (e != cudaSuccess) return moe::fail(MOE_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return MOE_OK;
}
