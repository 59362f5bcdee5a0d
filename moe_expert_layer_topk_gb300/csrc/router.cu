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
// CTA = 2 warps over 32 tokens x 32 experts; thread = 4 tokens x 4 experts.
// h advances in stages of 32 positions: a 4-deep cp.async pipeline brings
// the Wr tile [32 h][32 e] (fp32) and the x tile [32 tokens][32 h] (bf16)
// into shared memory; x is widened once per stage into a transposed fp32
// tile [32 h][32 tokens].  Each thread keeps, per output, the fused
// multiply-add chain of the current 256-wide h-block and the running sum of
// the finished blocks: exactly the order of the reading (block partials in
// increasing h from 0, block sums added left to right, bias last).
constexpr int kLogitTok = 32;
constexpr int kLogitExp = 32;
constexpr int kLogitThreads = 64;
constexpr int kLogitStage = 32;   // h per stage
constexpr int kLogitBlockH = 256; // h per summation block
constexpr int kLogitDepth = 4;    // stages in flight

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

template <bool kVec>
__global__ void __launch_bounds__(kLogitThreads) router_logits_kernel(
    const __nv_bfloat16* __restrict__ x, const float* __restrict__ Wr, const float* __restrict__ bias,
    int T, int H, int E, float* __restrict__ logits) {
  __shared__ __align__(16) float ws[kLogitDepth][kLogitStage][kLogitExp];
  __shared__ __align__(16) __nv_bfloat16 xraw[kLogitDepth][kLogitTok][kLogitStage];
  __shared__ __align__(16) float xs[kLogitStage][kLogitTok];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tg = lane & 7, eg = lane >> 3;
  const int t0 = blockIdx.x * kLogitTok, e0 = blockIdx.y * kLogitExp;
  const int my_tok = tg * 4, my_exp = warp * 16 + eg * 4;
  const int nstage = H / kLogitStage;

  auto issue = [&](int st) {
    const int buf = st % kLogitDepth;
    const int h0 = st * kLogitStage;
    // Wr: 32 rows x 32 experts = 256 x 16 bytes, 4 per thread
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = tid + i * kLogitThreads;
      const int row = idx >> 3, c4 = (idx & 7) * 4;
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
    // x: 32 tokens x 32 h (bf16) = 128 x 16 bytes, 2 per thread
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int idx = tid + i * kLogitThreads;
      const int tok = idx >> 2, h8 = (idx & 3) * 8;
      const int t = t0 + tok;
      const uint32_t dst = (uint32_t)__cvta_generic_to_shared(&xraw[buf][tok][h8]);
      cp_async16(dst, t < T ? (const void*)(x + (size_t)t * H + h0 + h8) : (const void*)x, t < T);
    }
  };

  float p[4][4], run[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      p[i][j] = 0.f;
      run[i][j] = 0.f;
    }
#pragma unroll
  for (int st = 0; st < kLogitDepth - 1; ++st) {
    if (st < nstage) issue(st);
    cp_async_commit();
  }
  for (int st = 0; st < nstage; ++st) {
    const int buf = st % kLogitDepth;
    cp_async_wait<kLogitDepth - 2>();
    __syncthreads();  // stage st landed for every thread; stage st-1 fully consumed
    // widen x: thread converts 16 values [tok][h..h+15] -> xs[h][tok]
    {
      const int tok = tid >> 1, hh0 = (tid & 1) * 16;
      const uint4* src = reinterpret_cast<const uint4*>(&xraw[buf][tok][hh0]);
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        const uint4 q = src[v];
        const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          xs[hh0 + 8 * v + 2 * i][tok] = bf16lo(w4[i]);
          xs[hh0 + 8 * v + 2 * i + 1][tok] = bf16hi(w4[i]);
        }
      }
    }
    if (st + kLogitDepth - 1 < nstage) issue(st + kLogitDepth - 1);
    cp_async_commit();
    __syncthreads();
#pragma unroll 8
    for (int hh = 0; hh < kLogitStage; ++hh) {
      const float4 xv = *reinterpret_cast<const float4*>(&xs[hh][my_tok]);
      const float4 wv = *reinterpret_cast<const float4*>(&ws[buf][hh][my_exp]);
      const float xa[4] = {xv.x, xv.y, xv.z, xv.w};
      const float wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) p[i][j] = __fmaf_rn(xa[i], wa[j], p[i][j]);
    }
    const int h_end = (st + 1) * kLogitStage;
    if (h_end % kLogitBlockH == 0 || h_end == H) {
      const bool first = h_end <= kLogitBlockH;
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          run[i][j] = first ? p[i][j] : __fadd_rn(run[i][j], p[i][j]);
          p[i][j] = 0.f;
        }
    }
  }
  cp_async_wait<0>();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + my_tok + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + my_exp + j;
      if (e < E) logits[(size_t)t * E + e] = bias ? __fadd_rn(run[i][j], __ldg(bias + e)) : run[i][j];
    }
  }
}

// -------------------------------------------------------------- top-k kernel
//
// One warp per token: the token's logits sit in registers (lane l holds
// experts l, l+32, ...; kNQ registers per lane); k rounds of a warp-wide
// arg-max over (logit descending, id ascending) pick the slots in order.
// Slot counts go to counts[] with integer atomics (order-independent).
constexpr int kTopkWarps = 8;
constexpr int kTopkTokPerWarp = 2;
constexpr int kTopkTokPerBlock = kTopkWarps * kTopkTokPerWarp;

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

template <int kNQ>
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ logits, int T,
                                                          int E, int k, int32_t* __restrict__ topk_idx,
                                                          float* __restrict__ topk_w,
                                                          int32_t* __restrict__ counts) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int it = 0; it < kTopkTokPerWarp; ++it) {
    const int t = blockIdx.x * kTopkTokPerBlock + warp * kTopkTokPerWarp + it;
    if (t >= T) break;
    float v[kNQ];
#pragma unroll
    for (int q = 0; q < kNQ; ++q) {
      const int e = lane + 32 * q;
      v[q] = (e < E) ? __ldg(logits + (size_t)t * E + e) : 0.f;
    }
    uint32_t taken = 0;
#pragma unroll
    for (int q = 0; q < kNQ; ++q)
      if (lane + 32 * q >= E) taken |= 1u << q;  // padding never wins
    float my_v = 0.f;
    int my_i = 0;
    for (int j = 0; j < k; ++j) {
      float bv = 0.f;
      int bi = INT_MAX;
#pragma unroll
      for (int q = 0; q < kNQ; ++q) {
        const int e = lane + 32 * q;
        if (!((taken >> q) & 1u) && (bi == INT_MAX || better(v[q], e, bv, bi))) {
          bv = v[q];
          bi = e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (oi != INT_MAX && (bi == INT_MAX || better(ov, oi, bv, bi))) {
          bv = ov;
          bi = oi;
        }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == j) {
        my_v = bv;
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
      atomicAdd(counts + my_i, 1);
    }
  }
}

__global__ void zero_counts_kernel(int32_t* __restrict__ counts, int E) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts[e] = 0;
}

// ------------------------------------------------------------ offsets kernel
// One CTA: exclusive scan of counts -> offsets, EP-rank row ranges.
__global__ void __launch_bounds__(1024) router_offsets_kernel(const int32_t* __restrict__ counts,
                                                              int E, int ep_size,
                                                              int32_t* __restrict__ offsets,
                                                              int32_t* __restrict__ rank_offsets) {
  __shared__ int warp_sum[32];
  __shared__ int excl[kMaxExperts + 1];
  const int e = threadIdx.x;
  const int c = e < E ? counts[e] : 0;
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
  const int s = threadIdx.x;
  if (s <= S) seg[s] = (int)(((long long)s * T) / S);
}

// dWr[h,e] (+)= sum_s (P[s][h][e] + P[s][h][Ep+e]), splits in order.
__global__ void router_bwd_reduce_kernel(const float* __restrict__ P, int S, int H, int E, int Ep,
                                         float* __restrict__ dWr, int accumulate) {
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

int route_ws_layout(int T, int E, size_t* logits_bytes, size_t* hist_bytes) {
  const size_t nblk = (size_t)((T + kTopkTokPerBlock - 1) / kTopkTokPerBlock);
  *logits_bytes = align256(sizeof(float) * (size_t)(T > 0 ? T : 1) * E);
  *hist_bytes = 0;
  return (int)nblk;
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
  (void)H;
  if (T < 0 || E <= 0) return 0;
  size_t a, b;
  route_ws_layout(T, E, &a, &b);
  return a + b;
}

int moe_route_topk(const void* x, const float* Wr, const float* bias, int T, int H, int E, int k,
                   int ep_size, int32_t* topk_idx, float* topk_w, int32_t* counts,
                   int32_t* offsets, int32_t* rank_offsets, void* ws, size_t ws_bytes,
                   void* stream) {
  clear_error();
  if (T < 0 || H <= 0 || E <= 0 || k <= 0)
    return fail(MOE_ERR_INVALID_ARG, "moe_route_topk: need T>=0, H>0, E>0, k>0");
  if (E > kMaxExperts || k > kMaxTopK || k > E || H % 64 != 0 || (long long)T * k >= (1ll << 31))
    return fail(MOE_ERR_UNSUPPORTED_SHAPE,
                "moe_route_topk: need E<=1024, k<=min(E,32), H%%64==0, T*k<2^31 (E=%d k=%d H=%d)", E,
                k, H);
  if (ep_size < 1 || E % ep_size != 0)
    return fail(MOE_ERR_INVALID_ARG, "moe_route_topk: ep_size=%d must divide E=%d", ep_size, E);
  if (!counts || !offsets || !rank_offsets || !ws ||
      (T > 0 && (!x || !Wr || !topk_idx || !topk_w)))
    return fail(MOE_ERR_INVALID_ARG, "moe_route_topk: NULL pointer argument");
  if (!aligned16(x) || !aligned16(Wr) || !aligned16(ws) || (bias && !aligned16(bias)))
    return fail(MOE_ERR_ALIGNMENT, "moe_route_topk: x, Wr, bias and ws must be 16-byte aligned");
  size_t lb, hb;
  const int nblk = route_ws_layout(T, E, &lb, &hb);
  if (ws_bytes < lb + hb)
    return fail(MOE_ERR_WORKSPACE, "moe_route_topk: workspace %zu < %zu bytes", ws_bytes, lb + hb);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* logits = static_cast<float*>(ws);
  zero_counts_kernel<<<1, 256, 0, s>>>(counts, E);
  if (int rc = check_launch("moe_route_topk: zero counts")) return rc;
  if (T > 0) {
    dim3 grid((T + kLogitTok - 1) / kLogitTok, (E + kLogitExp - 1) / kLogitExp);
    if (E % 4 == 0)
      router_logits_kernel<true><<<grid, kLogitThreads, 0, s>>>(
          static_cast<const __nv_bfloat16*>(x), Wr, bias, T, H, E, logits);
    else
      router_logits_kernel<false><<<grid, kLogitThreads, 0, s>>>(
          static_cast<const __nv_bfloat16*>(x), Wr, bias, T, H, E, logits);
    if (int rc = check_launch("moe_route_topk: logits kernel")) return rc;
    const int nq = (E + 31) / 32;
    if (nq <= 1)
      router_topk_kernel<1><<<nblk, 256, 0, s>>>(logits, T, E, k, topk_idx, topk_w, counts);
    else if (nq <= 2)
      router_topk_kernel<2><<<nblk, 256, 0, s>>>(logits, T, E, k, topk_idx, topk_w, counts);
    else if (nq <= 4)
      router_topk_kernel<4><<<nblk, 256, 0, s>>>(logits, T, E, k, topk_idx, topk_w, counts);
    else if (nq <= 8)
      router_topk_kernel<8><<<nblk, 256, 0, s>>>(logits, T, E, k, topk_idx, topk_w, counts);
    else if (nq <= 16)
      router_topk_kernel<16><<<nblk, 256, 0, s>>>(logits, T, E, k, topk_idx, topk_w, counts);
    else
      router_topk_kernel<32><<<nblk, 256, 0, s>>>(logits, T, E, k, topk_idx, topk_w, counts);
    if (int rc = check_launch("moe_route_topk: top-k kernel")) return rc;
  }
  router_offsets_kernel<<<1, 1024, 0, s>>>(counts, E, ep_size, offsets, rank_offsets);
  return check_launch("moe_route_topk: offsets kernel");
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
  router_bwd_dl_kernel<<<(T + 7) / 8, 256, sizeof(float) * 8 * L.Ep, s>>>(
      d_w, topk_w, topk_idx, T, E, L.Ep, k, dl2, dl3, status);
  if (int rc = check_launch("moe_route_topk_bwd: dl kernel")) return rc;
  const size_t nwr = (size_t)H * L.Ep;
  router_bwd_wr_kernel<<<(int)((nwr + 255) / 256 < 4096 ? (nwr + 255) / 256 : 4096), 256, 0, s>>>(
      Wr, H, E, L.Ep, wr3);
  if (int rc = check_launch("moe_route_topk_bwd: Wr split kernel")) return rc;
  split_table_kernel<<<1, 128, 0, s>>>(seg, L.S, T);
  if (int rc = check_launch("moe_route_topk_bwd: split table")) return rc;
  // dx = bf16(dx_acc + dl . Wr^T)
  if (int rc = launch_dense_add_bf16(dl3, wr3, dx_acc, dx, T, H, 3 * L.Ep, s)) return rc;
  // split-K partials of x^T . [dl_hi | dl_lo]
  if (int rc = launch_dw_split(x, dl2, T, H, 2 * L.Ep, seg, L.S, part, base + L.maps, s)) return rc;
  const size_t nred = (size_t)H * E;
  router_bwd_reduce_kernel<<<(int)((nred + 255) / 256 < 4096 ? (nred + 255) / 256 : 4096), 256, 0,
                             s>>>(part, L.S, H, E, L.Ep, dWr, accumulate);
  return check_launch("moe_route_topk_bwd: reduce kernel");
}

}  // extern "C"
