// A1 + A2: router logits, top-k, softmax weights, expert histogram, offsets.
// B5: router backward (softmax-over-selected gradient, dWr, router share of dX).
//
// The router itself is not written out on the pages; the reading taken
// (logits = x.Wr + bias in fp32 with a fixed blocked summation order, top-k
// with ties to the lower expert id, softmax over the selected logits) is
// stated in moe_topk.h.  The EP-rank row ranges follow the contiguous dim-0
// expert split of "Qwen3-MoE-30B-A3B模型EP+FSDP2并行方案", section
// "完整并行流程".
#include <cfloat>

#include "common.cuh"

namespace moe {
namespace {

// ------------------------------------------------------------ logits kernel
//
// The reading's summation order makes every 256-wide h-block an independent
// fused multiply-add chain from 0; the block partials are then added left to
// right and the bias last.  This kernel computes the partials: one CTA per
// (64 tokens, one h-block, 128 experts), written to part[block][t][e]; the
// top-k kernel adds them in order.  Splitting over h-blocks gives enough
// CTAs to fill the GPU evenly and keeps only the 64 running chains of a
// thread in registers.
//
// CTA = 4 warps; thread = 8 tokens x 8 experts (tg = tid % 8, eg = tid / 8):
// tokens 4tg..4tg+3 and 32+4tg..32+4tg+3 (so the eight tg of a warp read 128
// contiguous bytes of xs per load, free of bank conflicts), experts
// 8eg..8eg+7.  The 64 chains advance by packed two-lane FMA instructions
// (fma.rn.f32x2) over pairs of experts with the token's x value in both
// lanes: every lane is an IEEE fused multiply-add rounded to nearest, so the
// chains are exactly those of one fmaf per (token, expert, h), with half the
// instructions to issue (measured 3% faster than one fmaf per chain).
// h advances in stages of 32: a double-buffered cp.async pipeline brings the Wr tile
// [32 h][128 e] (fp32) into shared memory; the x tile [64 tokens][32 h]
// (bf16) is read into registers one stage ahead, widened and stored
// transposed as xs[32 h][64 tokens] (two buffers).
constexpr int kLogitExp = 128;
constexpr int kLogitThreads = 128;
constexpr int kLogitStage = 32;   // h per stage
constexpr int kLogitBlockH = 256; // h per summation block
constexpr int kLogitDepth = 2;    // W stages in flight
// Tokens per CTA: 64 (8 per thread) or 32 (4 per thread, fewer registers,
// five CTAs per SM).  64 when those CTAs fill at least one wave of four per
// SM, else 32, so that small batches still spread over every SM: measured
// at T=4096 58.4 µs against 63.0 (512 CTAs of 64 tokens leave SMs idle), at
// T=8192 101.0 against 107.2; the partials are bit-identical either way.
template <int NT>
constexpr size_t logit_smem() { return sizeof(float) * (kLogitDepth * kLogitStage * kLogitExp + 2 * kLogitStage * NT); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(pred ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool pred) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(pred ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint64_t pair_of(float v) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ void fma2(uint64_t& acc, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

template <bool kVec, int NT>
__global__ void __launch_bounds__(kLogitThreads, NT == 32 ? 5 : 4) router_partials_kernel(
    const __nv_bfloat16* __restrict__ x, const float* __restrict__ Wr, int T, int H, int E,
    float* __restrict__ part) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) float lsm[];
  float(*ws)[kLogitStage][kLogitExp] = reinterpret_cast<float(*)[kLogitStage][kLogitExp]>(lsm);
  constexpr int TPT = NT / 8;                                  // tokens per thread
  constexpr int XV = NT * kLogitStage / 8 / kLogitThreads;     // 16-byte x vectors per thread and stage
  float(*xs)[kLogitStage][NT] =
      reinterpret_cast<float(*)[kLogitStage][NT]>(lsm + kLogitDepth * kLogitStage * kLogitExp);
  const int tid = threadIdx.x;
  const int tg = tid & 7, eg = tid >> 3;
  const int t0 = blockIdx.x * NT, blk = blockIdx.y, e0 = blockIdx.z * kLogitExp;
  const int hb0 = blk * kLogitBlockH;
  const int hb1 = min(H, hb0 + kLogitBlockH);
  const int nstage = (hb1 - hb0) / kLogitStage;
  // x staging: thread -> token tid % NT, h part (tid / NT) * 8 * XV of the stage
  const int xt = tid % NT, xh = (tid / NT) * 8 * XV;
  const bool xok = t0 + xt < T;
  const uint4* xrow = reinterpret_cast<const uint4*>(x + (size_t)(xok ? t0 + xt : 0) * H);

  auto issue_w = [&](int st) {
    const int buf = st % kLogitDepth;
    const int h0 = hb0 + st * kLogitStage;
    // 32 rows x 128 experts = 1024 x 16 bytes, 8 per thread
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int idx = tid + i * kLogitThreads;
      const int row = idx >> 5, c4 = (idx & 31) * 4;
      const int e = e0 + c4;
      const float* src = Wr + (size_t)(h0 + row) * E + e;
      const uint32_t dst = (uint32_t)__cvta_generic_to_shared(&ws[buf][row][c4]);
      if (kVec) {
        cp_async16(dst, e < E ? src : Wr, e < E);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) cp_async4(dst + 4 * j, e + j < E ? src + j : Wr, e + j < E);
      }
    }
  };
  auto load_x = [&](int st, uint4 (&r)[XV]) {
    const int hv = (hb0 + st * kLogitStage + xh) / 8;  // 16-byte vector index in the row
#pragma unroll
    for (int u = 0; u < XV; ++u) r[u] = xok ? __ldg(xrow + hv + u) : make_uint4(0, 0, 0, 0);
  };

  // chains: pp[i][q] = token i, experts (8eg + 2q, 8eg + 2q + 1)
  uint64_t pp[TPT][4];
#pragma unroll
  for (int i = 0; i < TPT; ++i)
#pragma unroll
    for (int q = 0; q < 4; ++q) pp[i][q] = 0ull;

  uint4 xr[XV];
  load_x(0, xr);
#pragma unroll
  for (int st = 0; st < kLogitDepth - 1; ++st) {
    if (st < nstage) issue_w(st);
    cp_async_commit();
  }
  for (int st = 0; st < nstage; ++st) {
    const int xb = st & 1;
    {  // widen this stage's x into xs[xb][h][token]
#pragma unroll
      for (int u = 0; u < XV; ++u) {
        const uint32_t w4[4] = {xr[u].x, xr[u].y, xr[u].z, xr[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          xs[xb][xh + 8 * u + 2 * i][xt] = bf16lo(w4[i]);
          xs[xb][xh + 8 * u + 2 * i + 1][xt] = bf16hi(w4[i]);
        }
      }
    }
    cp_async_wait<kLogitDepth - 2>();
    __syncthreads();  // xs[xb], W stage st visible; stage st-1 fully consumed
    if (st + kLogitDepth - 1 < nstage) issue_w(st + kLogitDepth - 1);
    cp_async_commit();
    if (st + 1 < nstage) load_x(st + 1, xr);
    const int buf = st % kLogitDepth;
#pragma unroll 4
    for (int hh = 0; hh < kLogitStage; ++hh) {
      const ulonglong2 wa = *reinterpret_cast<const ulonglong2*>(&ws[buf][hh][8 * eg]);
      const ulonglong2 wb = *reinterpret_cast<const ulonglong2*>(&ws[buf][hh][8 * eg + 4]);
      const uint64_t wv[4] = {wa.x, wa.y, wb.x, wb.y};
      float xf[TPT];
#pragma unroll
      for (int g4 = 0; g4 < TPT / 4; ++g4) {
        const float4 xa = *reinterpret_cast<const float4*>(&xs[xb][hh][32 * g4 + 4 * tg]);
        xf[4 * g4] = xa.x;
        xf[4 * g4 + 1] = xa.y;
        xf[4 * g4 + 2] = xa.z;
        xf[4 * g4 + 3] = xa.w;
      }
#pragma unroll
      for (int i = 0; i < TPT; ++i) {
        const uint64_t xx = pair_of(xf[i]);
#pragma unroll
        for (int q = 0; q < 4; ++q) fma2(pp[i][q], xx, wv[q]);
      }
    }
  }
  cp_async_wait<0>();
  float p[TPT][8];
#pragma unroll
  for (int i = 0; i < TPT; ++i)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 v = *reinterpret_cast<const float2*>(&pp[i][q]);
      p[i][2 * q] = v.x;
      p[i][2 * q + 1] = v.y;
    }
  float* out = part + (size_t)blk * T * E;
#pragma unroll
  for (int i = 0; i < TPT; ++i) {
    const int t = t0 + 32 * (i / 4) + 4 * tg + (i % 4);
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = e0 + 8 * eg + j;
      if (e < E) out[(size_t)t * E + e] = p[i][j];
    }
  }
}

// -------------------------------------------------------------- top-k kernel
//
// One warp per token: the token's logits are assembled in registers (lane l
// holds experts l, l+32, ...; kNQ registers per lane) from the h-block
// partials, added left to right, bias last; k rounds of a warp-wide arg-max
// over (logit descending, id ascending) pick the slots in order.  A CTA
// covers one ranking chunk of kRouteChunk tokens and counts its slots per
// expert in shared memory; the counts go to chunk_cnt[e][chunk], every
// entry written (no atomics on global memory, nothing to clear first).
constexpr int kTopkWarps = 8;
constexpr int kTopkTokPerWarp = 2;
constexpr int kTopkTokPerBlock = kTopkWarps * kTopkTokPerWarp;
static_assert(kTopkTokPerBlock == kRouteChunk, "a top-k CTA covers one ranking chunk");
// h-block partials loaded per batch (kNQ * batch <= 32 values per lane)
template <int kNQ>
__host__ __device__ constexpr int sum_batch() { return kNQ >= 32 ? 1 : (kNQ >= 16 ? 2 : (kNQ >= 8 ? 4 : 8)); }

// Order-preserving map of a logit to an unsigned key (larger float, larger
// key; the two zeros map to one key, as they compare equal); 0 is below
// every key and marks "no candidate".
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t b = f == 0.f ? 0u : __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

template <int kNQ>
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ part, int nblk,
                                                          const float* __restrict__ bias, int T,
                                                          int E, int k, int32_t* __restrict__ topk_idx,
                                                          float* __restrict__ topk_w,
                                                          int32_t* __restrict__ chunk_cnt, int nchunk) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int chist[];  // [E] slots of this chunk per expert
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x) chist[e] = 0;
  __syncthreads();
  for (int it = 0; it < kTopkTokPerWarp; ++it) {
    const int t = blockIdx.x * kTopkTokPerBlock + warp * kTopkTokPerWarp + it;
    if (t >= T) break;
    // the partials of up to kSumBatch blocks are loaded together (independent
    // loads in flight), then added in block order
    constexpr int kSumBatch = sum_batch<kNQ>();
    float v[kNQ];
#pragma unroll
    for (int q = 0; q < kNQ; ++q) v[q] = 0.f;
    for (int b0 = 0; b0 < nblk; b0 += kSumBatch) {
      float pv[kNQ][kSumBatch];
#pragma unroll
      for (int q = 0; q < kNQ; ++q) {
        const int e = lane + 32 * q;
#pragma unroll
        for (int u = 0; u < kSumBatch; ++u)
          pv[q][u] = (e < E && b0 + u < nblk) ? __ldg(part + ((size_t)(b0 + u) * T + t) * E + e) : 0.f;
      }
#pragma unroll
      for (int q = 0; q < kNQ; ++q)
#pragma unroll
        for (int u = 0; u < kSumBatch; ++u)
          if (b0 + u < nblk) v[q] = (b0 + u == 0) ? pv[q][u] : __fadd_rn(v[q], pv[q][u]);
    }
    if (bias) {
#pragma unroll
      for (int q = 0; q < kNQ; ++q) {
        const int e = lane + 32 * q;
        if (e < E) v[q] = __fadd_rn(v[q], __ldg(bias + e));
      }
    }
    uint32_t taken = 0;
#pragma unroll
    for (int q = 0; q < kNQ; ++q)
      if (lane + 32 * q >= E) taken |= 1u << q;  // padding never wins
    uint32_t key[kNQ];
#pragma unroll
    for (int q = 0; q < kNQ; ++q) key[q] = order_key(v[q]);
    float my_v = 0.f;
    int my_i = 0;
    // round j: the largest logit left, equal logits to the lower expert id
    // (a lane's own candidates in increasing id, then the warp's largest key
    // and the lowest id holding it)
    for (int j = 0; j < k; ++j) {
      uint32_t lk = 0;
      int li = INT_MAX;
#pragma unroll
      for (int q = 0; q < kNQ; ++q)
        if (!((taken >> q) & 1u) && key[q] > lk) {
          lk = key[q];
          li = lane + 32 * q;
        }
      const uint32_t mk = __reduce_max_sync(0xffffffffu, lk);
      const int bi = __reduce_min_sync(0xffffffffu, lk == mk ? li : INT_MAX);
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == j) {
        my_v = key_value(mk);
        my_i = bi;
      }
    }
    // softmax over the selected logits, shifted by the largest (slot 0)
    const float m = __shfl_sync(0xffffffffu, my_v, 0);
    const float ex = (lane < k) ? expf(my_v - m) : 0.f;
    float s = 0.f;
    for (int j = 0; j < k; ++j) s = __fadd_rn(s, __shfl_sync(0xffffffffu, ex, j));
    if (lane < k) {
      topk_idx[(size_t)t * k + lane] = my_i;
      topk_w[(size_t)t * k + lane] = __fdiv_rn(ex, s);
      atomicAdd(&chist[my_i], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_cnt[(size_t)e * nchunk + blockIdx.x] = chist[e];
}

// chunk_cnt[e][c] <- sum_{c' < c} chunk_cnt[e][c'] (in place, exclusive) and
// totals[e] = all of e's slots.  One warp per expert walks its row of chunks
// 32 at a time (coalesced): a warp scan of each batch plus the running carry.
__global__ void __launch_bounds__(256) route_chunk_scan_kernel(int32_t* __restrict__ chunk_cnt, int nchunk,
                                                               int E, int32_t* __restrict__ totals) {
  pdl_wait();
  pdl_trigger();
  const int e = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (e >= E) return;
  int32_t* row = chunk_cnt + (size_t)e * nchunk;
  int carry = 0;
  for (int c0 = 0; c0 < nchunk; c0 += 32) {
    const int c = c0 + lane;
    const int v = c < nchunk ? row[c] : 0;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (c < nchunk) row[c] = carry + incl - v;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) totals[e] = carry;
}

// ------------------------------------------------------------ offsets kernel
// One CTA: the per-expert totals -> counts[], exclusive scan -> offsets,
// EP-rank row ranges.
__global__ void __launch_bounds__(1024) router_offsets_kernel(const int32_t* __restrict__ hist,
                                                              int E, int ep_size,
                                                              int32_t* __restrict__ counts,
                                                              int32_t* __restrict__ offsets,
                                                              int32_t* __restrict__ rank_offsets) {
  pdl_wait();
  pdl_trigger();
  __shared__ int warp_sum[32];
  __shared__ int excl[kMaxExperts + 1];
  const int e = threadIdx.x;
  const int c = e < E ? hist[e] : 0;
  if (e < E) counts[e] = c;
  const int lane = e & 31, warp = e >> 5;
  int incl = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int ws = warp_sum[lane];
    int wi = ws;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += o;
    }
    warp_sum[lane] = wi - ws;  // exclusive prefix over warps
  }
  __syncthreads();
  const int ex = warp_sum[warp] + incl - c;
  if (e < E) {
    offsets[e] = ex;
    excl[e] = ex;
  }
  if (e == E - 1) {
    offsets[E] = ex + c;
    excl[E] = ex + c;
  }
  __syncthreads();
  const int per = E / ep_size;
  if (e <= ep_size) rank_offsets[e] = excl[e * per];
}

// ----------------------------------------------------------- backward prep
//
// dl[t,j] = w_j (d_w_j - sum_i w_i d_w_i).  The two router-backward
// contractions run on the tensor cores in bf16 with fp32 accumulation; to
// keep fp32-level accuracy each fp32 factor is split into hi = bf16(v) and
// lo = bf16(v - hi), and the products hi*hi + lo*hi + hi*lo are summed.
//   dl2 [T, 2*Ep] = [dl_hi | dl_lo]              (B operand of x^T . dl)
//   dl3 [T, 3*Ep] = [dl_hi | dl_lo | dl_hi]      (A operand of dl . Wr^T)
//   wr3 [H, 3*Ep] = [Wr_hi^T | Wr_hi^T | Wr_lo^T] (B operand of dl . Wr^T)
// Ep = E rounded up to 64; padding columns are zero.
__device__ __forceinline__ void split_bf16(float v, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(v);
  lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

__global__ void __launch_bounds__(256) router_bwd_dl_kernel(
    const float* __restrict__ d_w, const float* __restrict__ topk_w,
    const int32_t* __restrict__ topk_idx, int T, int E, int Ep, int k,
    __nv_bfloat16* __restrict__ dl2, __nv_bfloat16* __restrict__ dl3, int* status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float rowbuf[];  // [8 warps][Ep]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  float* row = rowbuf + (size_t)warp * Ep;
  for (int e = lane; e < Ep; e += 32) row[e] = 0.f;
  __syncwarp();
  const float w = lane < k ? topk_w[(size_t)t * k + lane] : 0.f;
  const float g = lane < k ? d_w[(size_t)t * k + lane] : 0.f;
  float s = 0.f;
  for (int j = 0; j < k; ++j)
    s = __fmaf_rn(__shfl_sync(0xffffffffu, w, j), __shfl_sync(0xffffffffu, g, j), s);
  if (lane < k) {
    const int e = topk_idx[(size_t)t * k + lane];
    if (e >= 0 && e < E)
      row[e] = w * (g - s);
    else
      set_status(status, MOE_STATUS_BAD_INDEX);
  }
  __syncwarp();
  __nv_bfloat16* o2 = dl2 + (size_t)t * 2 * Ep;
  __nv_bfloat16* o3 = dl3 + (size_t)t * 3 * Ep;
  for (int e = lane; e < Ep; e += 32) {
    __nv_bfloat16 hi, lo;
    split_bf16(row[e], hi, lo);
    o2[e] = hi;
    o2[Ep + e] = lo;
    o3[e] = hi;
    o3[Ep + e] = lo;
    o3[2 * Ep + e] = hi;
  }
}

__global__ void router_bwd_wr_kernel(const float* __restrict__ Wr, int H, int E, int Ep,
                                     __nv_bfloat16* __restrict__ wr3) {
  pdl_wait();
  pdl_trigger();
  const size_t n = (size_t)H * Ep;
  for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < n;
       q += (size_t)gridDim.x * blockDim.x) {
    const int h = (int)(q / Ep), e = (int)(q % Ep);
    const float v = e < E ? Wr[(size_t)h * E + e] : 0.f;
    __nv_bfloat16 hi, lo;
    split_bf16(v, hi, lo);
    __nv_bfloat16* o = wr3 + (size_t)h * 3 * Ep;
    o[e] = hi;
    o[Ep + e] = hi;
    o[2 * Ep + e] = lo;
  }
}

__global__ void split_table_kernel(int32_t* __restrict__ seg, int S, int T) {
  pdl_wait();
  pdl_trigger();
  const int s = threadIdx.x;
  if (s <= S) seg[s] = (int)(((long long)s * T) / S);
}

// dWr[h,e] (+)= sum_s (P[s][h][e] + P[s][h][Ep+e]), splits in order.
__global__ void router_bwd_reduce_kernel(const float* __restrict__ P, int S, int H, int E, int Ep,
                                         float* __restrict__ dWr, int accumulate) {
  pdl_wait();
  pdl_trigger();
  const size_t n = (size_t)H * E;
  for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < n;
       q += (size_t)gridDim.x * blockDim.x) {
    const int h = (int)(q / E), e = (int)(q % E);
    float hi = 0.f, lo = 0.f;
    for (int s = 0; s < S; ++s) {
      const float* p = P + ((size_t)s * H + h) * 2 * Ep;
      hi += p[e];
      lo += p[Ep + e];
    }
    const float v = hi + lo;
    dWr[q] = accumulate ? dWr[q] + v : v;
  }
}

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }


// Route workspace: the h-block partials of the logits, fp32 [nblk_h][T][E],
// then the per-expert slot totals, then (moe_route_topk only) the per-chunk
// slot counts [E][ceil(T/16)] that moe_route_topk_chunks returns instead.
int route_nchunk(int T) { return (T + kRouteChunk - 1) / kRouteChunk; }
size_t route_part_bytes(int T, int H, int E) {
  const size_t nblk_h = (size_t)((H + kLogitBlockH - 1) / kLogitBlockH);
  return align256(sizeof(float) * nblk_h * (size_t)(T > 0 ? T : 1) * E);
}
size_t route_chunk_bytes(int T, int E) { return align256(sizeof(int32_t) * (size_t)route_nchunk(T) * E); }
size_t route_ws_bytes(int T, int H, int E, bool with_chunks) {
  return route_part_bytes(T, H, E) + align256(sizeof(int32_t) * (size_t)E) +
         (with_chunks ? route_chunk_bytes(T, E) : 0);
}

struct BwdLayout {
  int Ep, S;
  size_t dl2, dl3, wr3, seg, part, maps, total;
};

BwdLayout bwd_layout(int T, int H, int E) {
  BwdLayout L;
  L.Ep = (E + 63) / 64 * 64;
  // split-K over tokens for x^T . dl2: about one wave of 128x(2Ep) tiles
  const int sms = 148;  // nominal; the exact SM count only changes the split, not the result
  const int tiles = ((H + 127) / 128) * ((2 * L.Ep + 255) / 256);
  int S = sms / (tiles > 0 ? tiles : 1);
  S = S < 1 ? 1 : (S > 64 ? 64 : S);
  while (S > 1 && (long long)T / S < 256) --S;
  L.S = S;
  size_t off = 0;
  L.dl2 = off; off += align256(sizeof(__nv_bfloat16) * (size_t)T * 2 * L.Ep);
  L.dl3 = off; off += align256(sizeof(__nv_bfloat16) * (size_t)T * 3 * L.Ep);
  L.wr3 = off; off += align256(sizeof(__nv_bfloat16) * (size_t)H * 3 * L.Ep);
  L.seg = off; off += align256(sizeof(int32_t) * (size_t)(S + 1));
  L.part = off; off += align256(sizeof(float) * (size_t)S * H * 2 * L.Ep);
  L.maps = off; off += align256(dw_split_maps_bytes(S));
  L.total = off;
  return L;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_route_topk_workspace_size(int T, int H, int E) {
  if (T < 0 || H <= 0 || E <= 0) return 0;
  return route_ws_bytes(T, H, E, true);
}

size_t moe_route_topk_chunks_workspace_size(int T, int H, int E) {
  if (T < 0 || H <= 0 || E <= 0) return 0;
  return route_ws_bytes(T, H, E, false);
}

}  // extern "C"

namespace moe {
namespace {

// Both route entry points: partial logits, top-k + per-chunk slot counts into
// `chunk` ([E][ceil(T/16)]), their per-expert scan (chunk prefixes in place,
// totals), counts / offsets / EP-rank ranges.
int route_impl(const char* fn, const void* x, const float* Wr, const float* bias, int T, int H, int E, int k,
               int ep_size, int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
               int32_t* rank_offsets, int32_t* chunk, void* ws, cudaStream_t s) {
  float* part = static_cast<float*>(ws);
  int32_t* totals = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + route_part_bytes(T, H, E));
  const int nchunk = route_nchunk(T);
  if (T > 0) {
    static bool attr_set[64] = {};
    const int dev = current_device();
    if (dev < 0 || dev >= 64) return fail(MOE_ERR_CUDA, "%s: no usable current device", fn);
    if (!attr_set[dev]) {
      cudaError_t e[4] = {
          cudaFuncSetAttribute(router_partials_kernel<true, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)logit_smem<64>()),
          cudaFuncSetAttribute(router_partials_kernel<false, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)logit_smem<64>()),
          cudaFuncSetAttribute(router_partials_kernel<true, 32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)logit_smem<32>()),
          cudaFuncSetAttribute(router_partials_kernel<false, 32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)logit_smem<32>())};
      for (cudaError_t x : e)
        if (x != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(x));
      attr_set[dev] = true;
    }
    const int nblk_h = (H + kLogitBlockH - 1) / kLogitBlockH;
    const int nexp = (E + kLogitExp - 1) / kLogitExp;
    const long long ctas64 = (long long)((T + 63) / 64) * nblk_h * nexp;
    const int sms = sm_count();
    const bool wide = ctas64 >= 4LL * (sms > 0 ? sms : 148);
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    if (wide) {
      dim3 grid((T + 63) / 64, nblk_h, nexp);
      if (E % 4 == 0)
        launch_pdl(router_partials_kernel<true, 64>, grid, kLogitThreads, logit_smem<64>(), s, xb, Wr, T, H, E, part);
      else
        launch_pdl(router_partials_kernel<false, 64>, grid, kLogitThreads, logit_smem<64>(), s, xb, Wr, T, H, E, part);
    } else {
      dim3 grid((T + 31) / 32, nblk_h, nexp);
      if (E % 4 == 0)
        launch_pdl(router_partials_kernel<true, 32>, grid, kLogitThreads, logit_smem<32>(), s, xb, Wr, T, H, E, part);
      else
        launch_pdl(router_partials_kernel<false, 32>, grid, kLogitThreads, logit_smem<32>(), s, xb, Wr, T, H, E, part);
    }
    if (int rc = check_launch("route: logits kernel")) return rc;
    const int nq = (E + 31) / 32;
    const size_t hs = sizeof(int) * (size_t)E;
    if (nq <= 1)
      launch_pdl(router_topk_kernel<1>, nchunk, 256, hs, s, part, nblk_h, bias, T, E, k, topk_idx, topk_w, chunk, nchunk);
    else if (nq <= 2)
      launch_pdl(router_topk_kernel<2>, nchunk, 256, hs, s, part, nblk_h, bias, T, E, k, topk_idx, topk_w, chunk, nchunk);
    else if (nq <= 4)
      launch_pdl(router_topk_kernel<4>, nchunk, 256, hs, s, part, nblk_h, bias, T, E, k, topk_idx, topk_w, chunk, nchunk);
    else if (nq <= 8)
      launch_pdl(router_topk_kernel<8>, nchunk, 256, hs, s, part, nblk_h, bias, T, E, k, topk_idx, topk_w, chunk, nchunk);
    else if (nq <= 16)
      launch_pdl(router_topk_kernel<16>, nchunk, 256, hs, s, part, nblk_h, bias, T, E, k, topk_idx, topk_w, chunk, nchunk);
    else
      launch_pdl(router_topk_kernel<32>, nchunk, 256, hs, s, part, nblk_h, bias, T, E, k, topk_idx, topk_w, chunk, nchunk);
    if (int rc = check_launch("route: top-k kernel")) return rc;
  }
  // with no token every total is 0 (the scan runs over no chunk)
  launch_pdl(route_chunk_scan_kernel, (E + 7) / 8, 256, 0, s, chunk, nchunk, E, totals);
  if (int rc = check_launch("route: chunk scan kernel")) return rc;
  launch_pdl(router_offsets_kernel, 1, 1024, 0, s, totals, E, ep_size, counts, offsets, rank_offsets);
  return check_launch("route: offsets kernel");
}

int route_check(const char* fn, const void* x, const float* Wr, const float* bias, int T, int H, int E, int k,
                int ep_size, int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                int32_t* rank_offsets, void* ws, size_t ws_bytes, size_t need) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0) return fail(MOE_ERR_INVALID_ARG, "%s: need T>=0, H>0, E>0, k>0", fn);
  if (E > kMaxExperts || k > kMaxTopK || k > E || H % 64 != 0 || (long long)T * k >= (1ll << 31))
    return fail(MOE_ERR_UNSUPPORTED_SHAPE, "%s: need E<=1024, k<=min(E,32), H%%64==0, T*k<2^31 (E=%d k=%d H=%d)",
                fn, E, k, H);
  if (ep_size < 1 || E % ep_size != 0)
    return fail(MOE_ERR_INVALID_ARG, "%s: ep_size=%d must divide E=%d", fn, ep_size, E);
  if (!counts || !offsets || !rank_offsets || !ws || (T > 0 && (!x || !Wr || !topk_idx || !topk_w)))
    return fail(MOE_ERR_INVALID_ARG, "%s: NULL pointer argument", fn);
  if (!aligned16(x) || !aligned16(Wr) || !aligned16(ws) || (bias && !aligned16(bias)))
    return fail(MOE_ERR_ALIGNMENT, "%s: x, Wr, bias and ws must be 16-byte aligned", fn);
  if (ws_bytes < need) return fail(MOE_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, ws_bytes, need);
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" {

int moe_route_topk(const void* x, const float* Wr, const float* bias, int T, int H, int E, int k,
                   int ep_size, int32_t* topk_idx, float* topk_w, int32_t* counts,
                   int32_t* offsets, int32_t* rank_offsets, void* ws, size_t ws_bytes,
                   void* stream) {
  clear_error();
  const char* fn = "moe_route_topk";
  if (int rc = route_check(fn, x, Wr, bias, T, H, E, k, ep_size, topk_idx, topk_w, counts, offsets, rank_offsets,
                           ws, ws_bytes, T >= 0 && H > 0 && E > 0 ? route_ws_bytes(T, H, E, true) : 0))
    return rc;
  int32_t* chunk = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + route_ws_bytes(T, H, E, false));
  return route_impl(fn, x, Wr, bias, T, H, E, k, ep_size, topk_idx, topk_w, counts, offsets, rank_offsets,
                    chunk, ws, static_cast<cudaStream_t>(stream));
}

int moe_route_topk_chunks(const void* x, const float* Wr, const float* bias, int T, int H, int E, int k,
                          int ep_size, int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                          int32_t* rank_offsets, int32_t* chunk_prefix, void* ws, size_t ws_bytes,
                          void* stream) {
  clear_error();
  const char* fn = "moe_route_topk_chunks";
  if (int rc = route_check(fn, x, Wr, bias, T, H, E, k, ep_size, topk_idx, topk_w, counts, offsets, rank_offsets,
                           ws, ws_bytes, T >= 0 && H > 0 && E > 0 ? route_ws_bytes(T, H, E, false) : 0))
    return rc;
  if (T > 0 && !chunk_prefix) return fail(MOE_ERR_INVALID_ARG, "%s: NULL pointer argument", fn);
  return route_impl(fn, x, Wr, bias, T, H, E, k, ep_size, topk_idx, topk_w, counts, offsets, rank_offsets,
                    chunk_prefix, ws, static_cast<cudaStream_t>(stream));
}

size_t moe_route_topk_bwd_workspace_size(int T, int H, int E) {
  if (T < 0 || H <= 0 || E <= 0) return 0;
  return bwd_layout(T, H, E).total;
}

int moe_route_topk_bwd(const float* d_w, const float* topk_w, const int32_t* topk_idx,
                       const void* x, const float* Wr, const float* dx_acc, int T, int H, int E,
                       int k, float* dWr, void* dx, int accumulate, void* ws, size_t ws_bytes,
                       void* stream) {
  clear_error();
  if (T < 0 || H <= 0 || E <= 0 || k <= 0)
    return fail(MOE_ERR_INVALID_ARG, "moe_route_topk_bwd: need T>=0, H>0, E>0, k>0");
  if (E > kMaxExperts || k > kMaxTopK || k > E || H % 64 != 0 || (long long)T * k >= (1ll << 31))
    return fail(MOE_ERR_UNSUPPORTED_SHAPE,
                "moe_route_topk_bwd: need E<=1024, k<=min(E,32), H%%64==0 (E=%d k=%d H=%d)", E, k, H);
  if (!dWr || !ws || (T > 0 && (!d_w || !topk_w || !topk_idx || !x || !Wr || !dx_acc || !dx)))
    return fail(MOE_ERR_INVALID_ARG, "moe_route_topk_bwd: NULL pointer argument");
  if (!aligned16(x) || !aligned16(Wr) || !aligned16(dx_acc) || !aligned16(dWr) || !aligned16(dx) ||
      (reinterpret_cast<uintptr_t>(ws) & 127u))
    return fail(MOE_ERR_ALIGNMENT,
                "moe_route_topk_bwd: tensors must be 16-byte and ws 128-byte aligned");
  const BwdLayout L = bwd_layout(T, H, E);
  if (ws_bytes < L.total)
    return fail(MOE_ERR_WORKSPACE, "moe_route_topk_bwd: workspace %zu < %zu bytes", ws_bytes, L.total);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(ws);
  auto* dl2 = reinterpret_cast<__nv_bfloat16*>(base + L.dl2);
  auto* dl3 = reinterpret_cast<__nv_bfloat16*>(base + L.dl3);
  auto* wr3 = reinterpret_cast<__nv_bfloat16*>(base + L.wr3);
  auto* seg = reinterpret_cast<int32_t*>(base + L.seg);
  auto* part = reinterpret_cast<float*>(base + L.part);
  int* status = status_word();

  if (T == 0) {  // no token: dWr gets a zero sum, dx is empty
    if (!accumulate) {
      cudaError_t e = cudaMemsetAsync(dWr, 0, sizeof(float) * (size_t)H * E, s);
      if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "moe_route_topk_bwd: %s", cudaGetErrorString(e));
    }
    return MOE_OK;
  }
  launch_pdl(router_bwd_dl_kernel, (T + 7) / 8, 256, sizeof(float) * 8 * L.Ep, s, 
      d_w, topk_w, topk_idx, T, E, L.Ep, k, dl2, dl3, status);
  if (int rc = check_launch("moe_route_topk_bwd: dl kernel")) return rc;
  const size_t nwr = (size_t)H * L.Ep;
  launch_pdl(router_bwd_wr_kernel, (int)((nwr + 255) / 256 < 4096 ? (nwr + 255) / 256 : 4096), 256, 0, s, 
      Wr, H, E, L.Ep, wr3);
  if (int rc = check_launch("moe_route_topk_bwd: Wr split kernel")) return rc;
  launch_pdl(split_table_kernel, 1, 128, 0, s, seg, L.S, T);
  if (int rc = check_launch("moe_route_topk_bwd: split table")) return rc;
  // dx = bf16(dx_acc + dl . Wr^T)
  if (int rc = launch_dense_add_bf16(dl3, wr3, dx_acc, dx, T, H, 3 * L.Ep, s)) return rc;
  // split-K partials of x^T . [dl_hi | dl_lo]
  if (int rc = launch_dw_split(x, dl2, T, H, 2 * L.Ep, seg, L.S, part, base + L.maps, s)) return rc;
  const size_t nred = (size_t)H * E;
  launch_pdl(router_bwd_reduce_kernel, (int)((nred + 255) / 256 < 4096 ? (nred + 255) / 256 : 4096), 256, 0, s, part, L.S, H, E, L.Ep, dWr, accumulate);
  return check_launch("moe_route_topk_bwd: reduce kernel");
}

}  // extern "C"
