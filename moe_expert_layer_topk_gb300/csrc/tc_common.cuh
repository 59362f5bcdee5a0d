// tcgen05 / TMA / mbarrier building blocks shared by the grouped-GEMM
// kernels (sm_103a), and the host-side tensor-map helpers.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int THREADS = 192;
constexpr int ACC_COLS = 256;
constexpr int TMEM_COLS = 512;
constexpr int CHUNK_BYTES = 64 * BK * 2;      // one 64(MN) x 64(K) MN-major box: 8 KiB
constexpr unsigned long long TIMEOUT_NS = 2000000000ull;
// Epilogue staging: each epilogue warp owns a ring of boxes of 32 rows x 64
// bytes (32 bf16 or 16 fp32 columns), written in the 64-byte swizzle pattern.
constexpr int EP_BOX_BYTES = 32 * 64;
constexpr int EP_SLOTS = 2;
constexpr size_t kSmemMax = 232448;

// ------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for phase `parity` of an mbarrier.  Returns false when the
// CTA is aborting (*abort_flag set) or the wait timed out (which sets it).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, int* abort_flag, int* status) {
  unsigned long long t0 = 0;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*reinterpret_cast<volatile int*>(abort_flag)) return false;
      const unsigned long long now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > TIMEOUT_NS) {
        *reinterpret_cast<volatile int*>(abort_flag) = 1;
        set_status(status, MOE_STATUS_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(c1)
               : "memory");
}

__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1)
      : "memory");
}

// An L2 cache policy under which the lines an access touches are evicted
// after evict-normal ones.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                                  uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_reduce_add_2d_hint(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                                       uint64_t pol) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], "
      "%4;" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "l"(pol)
      : "memory");
}

// *dst += {a, b, c, d} as one 16-byte reduction in L2 (dst 16-byte aligned).
__device__ __forceinline__ void red_add_f32x4(float* dst, float a, float b, float c, float d) {
  asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

// One epilogue warp's staging ring (see EP_*).  Lane i holds row i of a box.
template <int SLOTS = EP_SLOTS>
struct EpRing {
  uint8_t* base;
  int slot;
  int lane;
  __device__ __forceinline__ uint8_t* acquire() {
    // the store issued from this slot SLOTS boxes ago must have read it
    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(SLOTS - 1) : "memory");
    __syncwarp();
    return base + slot * EP_BOX_BYTES;
  }
  // 16-byte chunk c (0..3) of this lane's 64-byte row, 64-byte swizzle
  __device__ __forceinline__ void put(uint8_t* box, int c, uint4 v) {
    *reinterpret_cast<uint4*>(box + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) = v;
  }
  __device__ __forceinline__ void issue(uint8_t* box, const CUtensorMap* map, int x, int y,
                                        bool reduce = false) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      if (reduce)
        tma_reduce_add_2d(map, smem_u32(box), x, y);
      else
        tma_store_2d(map, smem_u32(box), x, y);
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
    slot = (slot + 1) & (SLOTS - 1);
  }
  // issue() with an L2 cache policy for the written lines
  __device__ __forceinline__ void issue_hint(uint8_t* box, const CUtensorMap* map, int x, int y, bool reduce,
                                             uint64_t pol) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      if (reduce)
        tma_reduce_add_2d_hint(map, smem_u32(box), x, y, pol);
      else
        tma_store_2d_hint(map, smem_u32(box), x, y, pol);
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
    slot = (slot + 1) & (SLOTS - 1);
  }
  __device__ __forceinline__ void drain() {
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
  }
};

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, fp32 accumulation.
__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once) on `bar` when all previously issued tcgen05 ops of this thread complete.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 layout, version 1), 128-byte swizzle.
//   K-major operand: 8-row groups of 1024 B (SBO = 1024), k advanced by +32 B per 16 elements.
//   MN-major operand: 64-element MN chunks LBO apart, 8-row K groups SBO = 1024 apart.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ float f32(uint32_t u) { return __uint_as_float(u); }

// Makes this thread's later TMA loads through `map` see a tensor map that
// was written in global memory (by the segment-map kernel).
__device__ __forceinline__ void tmap_acquire(const CUtensorMap* map) {
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(
                   reinterpret_cast<uint64_t>(map))
               : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of `local` (a shared::cta address) in CTA `rank`
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

template <int CTAS>
__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
  if constexpr (CTAS == 1) {
    tma_load_2d(dst, map, bar, c0, c1);
  } else {
    // the mbarrier may live in the peer CTA (the leader's full barrier)
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
  }
}

// MN-major operand stage: one 3-D box {64 elements, 64 K rows, nchunks} whose
// chunks land 8 KiB apart, i.e. the canonical MN-major layout with LBO = 8 KiB.
template <int CTAS>
__device__ __forceinline__ void tma_load_mn(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int krow, int chunk0) {
  if constexpr (CTAS == 1) {
    tma_load_3d(dst, map, bar, 0, krow, chunk0);
  } else {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(0), "r"(krow), "r"(chunk0)
        : "memory");
  }
}

// D[tmem] (+)= A[smem] * B[smem], e4m3 inputs (K = 32 per instruction, the
// same 32 bytes of each operand row as one bf16 step), fp32 accumulation.
__device__ __forceinline__ void mma_e4m3(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <int CTAS, bool FP8 = false>
__device__ __forceinline__ void mma_issue(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  static_assert(!FP8 || CTAS == 1, "e4m3 GEMMs run one CTA per tile");
  if constexpr (FP8) {
    mma_e4m3(d, a, b, idesc, accumulate);
  } else if constexpr (CTAS == 1) {
    mma_bf16(d, a, b, idesc, accumulate);
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// Commit previously issued MMAs to `bar` (in both CTAs of the pair for CTAS = 2).
template <int CTAS>
__device__ __forceinline__ void mma_commit_to(uint32_t bar) {
  if constexpr (CTAS == 1) {
    mma_commit(bar);
  } else {
    const uint16_t mask = 3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(mask)
        : "memory");
  }
}

template <int CTAS>
__device__ __forceinline__ void tmem_alloc_n(uint32_t dst_smem, uint32_t ncols) {
  if constexpr (CTAS == 1) {
    tmem_alloc(dst_smem, ncols);
    tmem_relinquish();
  } else {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
}

template <int CTAS>
__device__ __forceinline__ void tmem_dealloc_n(uint32_t taddr, uint32_t ncols) {
  if constexpr (CTAS == 1) {
    tmem_dealloc(taddr, ncols);
  } else {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
    else
      cudaGetLastError();
  }
  return fn;
}

// 2-D tensor [outer, inner] row-major, box {box_inner, box_outer}.  Operand
// maps are bf16 with the 128-byte swizzle; output maps use 64-byte boxes with
// the 64-byte swizzle (bf16 or fp32).
inline int make_tmap_typed(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                           uint32_t box_inner, uint32_t box_outer, CUtensorMapDataType dt, uint64_t esz,
                           CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {inner, outer > 0 ? outer : 1};
  cuuint64_t strides[1] = {inner * esz};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, dt, 2,
                  const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for [%llu x %llu] box %u x %u",
                (int)r, (unsigned long long)outer, (unsigned long long)inner, box_inner, box_outer);
  return MOE_OK;
}

inline int make_tmap(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
                     uint32_t box_outer, bool fp32 = false,
                     CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  return make_tmap_typed(m, ptr, inner, outer, box_inner, box_outer,
                         fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         fp32 ? 4 : 2, swz);
}

// e4m3 operand map (bytes), 128-byte swizzle.
inline int make_tmap_e4m3(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                          uint32_t box_inner, uint32_t box_outer) {
  return make_tmap_typed(m, ptr, inner, outer, box_inner, box_outer, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                         CU_TENSOR_MAP_SWIZZLE_128B);
}

// MN-major operand map: the bf16 tensor [rows, cols] seen as 3-D
// {64 columns, rows, cols/64 chunks} (strides: row pitch, 128 B), box
// {64, 64 rows, nck chunks}: one load fills nck 8 KiB chunks of a stage.
inline int make_tmap_mn(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t nck) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {64, rows > 0 ? rows : 1, cols / 64};
  cuuint64_t strides[2] = {cols * 2, 128};
  cuuint32_t box[3] = {64, 64, nck};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (%d) for [%llu x %llu] x %u chunks",
                (int)r, (unsigned long long)rows, (unsigned long long)cols, nck);
  return MOE_OK;
}

// Output map: 32 rows x 64 bytes per box (32 bf16 / 16 fp32 columns).
inline int make_out_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, bool fp32) {
  return make_tmap(m, ptr, inner, outer, fp32 ? 16 : 32, 32, fp32, CU_TENSOR_MAP_SWIZZLE_64B);
}

inline uint32_t make_idesc(int n, int m, bool a_mn, bool b_mn, bool e4m3 = false) {
  return (1u << 4)                    // D fp32
         | (e4m3 ? 0u : (1u << 7) | (1u << 10))  // A, B bf16 (kind::f16) or e4m3 (kind::f8f6f4: code 0)
         | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(n >> 3) << 17)   // N / 8
         | ((uint32_t)(m >> 4) << 24);  // M / 16
}

}  // namespace tc
}  // namespace moe
