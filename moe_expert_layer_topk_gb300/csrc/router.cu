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
// CTA = 8 warps over 16 tokens x 128 experts.  Warp w sums h-block (sb + w)
// of 256 consecutive h for all 16x128 outputs (each lane: 8 tokens x 8
// experts, one fused multiply-add chain per output in increasing h).  The
// eight block partials then meet in shared memory, where one thread per
// output adds them left to right into its running sum; the bias comes last.
constexpr int kLogitTok = 16;
constexpr int kLogitExp = 128;
constexpr int kLogitWarps = 8;
constexpr int kLogitBlockH = 256;
constexpr size_t kLogitSmem = sizeof(float) * kLogitWarps * kLogitTok * kLogitExp;  // 64 KiB

__device__ __forceinline__ float bf16_elem(const uint4& v, int i) {
  const uint32_t w = (i >> 1) == 0 ? v.x : (i >> 1) == 1 ? v.y : (i >> 1) == 2 ? v.z : v.w;
  return (i & 1) ? bf16hi(w) : bf16lo(w);
}

template <bool kVec>
__global__ void __launch_bounds__(256) router_logits_kernel(const __nv_bfloat16* __restrict__ x,
                                                            const float* __restrict__ Wr,
                                                            const float* __restrict__ bias, int T,
                                                            int H, int E,
                                                            float* __restrict__ logits) {
  extern __shared__ float part[];  // [warp][token][expert]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tg = lane >> 4, eg = lane & 15;
  const int t0 = blockIdx.x * kLogitTok;
  const int e0 = blockIdx.y * kLogitExp;
  const int my_e = e0 + eg * 8;
  const int nblk = (H + kLogitBlockH - 1) / kLogitBlockH;

  float run[8];
#pragma unroll
  for (int o = 0; o < 8; ++o) run[o] = 0.f;

  for (int sb = 0; sb < nblk; sb += kLogitWarps) {
    const int blk = sb + warp;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    if (blk < nblk) {
      const int h0 = blk * kLogitBlockH;
      const int h1 = min(H, h0 + kLogitBlockH);
      for (int h = h0; h < h1; h += 8) {
        uint4 xv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int t = t0 + tg * 8 + i;
          xv[i] = (t < T) ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H + h))
                          : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int hh = 0; hh < 8; ++hh) {
          float w[8];
          const float* wrow = Wr + (size_t)(h + hh) * E;
          if (kVec) {
            if (my_e < E) {
              const float4 a = __ldg(reinterpret_cast<const float4*>(wrow + my_e));
              const float4 b = __ldg(reinterpret_cast<const float4*>(wrow + my_e + 4));
              w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
              w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) w[j] = 0.f;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) w[j] = (my_e + j < E) ? __ldg(wrow + my_e + j) : 0.f;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float xf = bf16_elem(xv[i], hh);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = __fmaf_rn(xf, w[j], acc[i][j]);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float4* dst = reinterpret_cast<float4*>(
          part + ((size_t)(warp * kLogitTok + tg * 8 + i) * kLogitExp + eg * 8));
      dst[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      dst[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
    __syncthreads();
#pragma unroll
    for (int o = 0; o < 8; ++o) {
      const int idx = threadIdx.x + o * 256;
      const int tok = idx / kLogitExp, ex = idx % kLogitExp;
#pragma unroll
      for (int w = 0; w < kLogitWarps; ++w) {
        const int b = sb + w;
        if (b < nblk) {
          const float p = part[(size_t)(w * kLogitTok + tok) * kLogitExp + ex];
          run[o] = (b == 0) ? p : __fadd_rn(run[o], p);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int o = 0; o < 8; ++o) {
    const int idx = threadIdx.x + o * 256;
    const int t = t0 + idx / kLogitExp, e = e0 + idx % kLogitExp;
    if (t < T && e < E) logits[(size_t)t * E + e] = bias ? __fadd_rn(run[o], bias[e]) : run[o];
  }
}

// -------------------------------------------------------------- top-k kernel
//
// One warp per token: the token's logits sit in registers (lane l holds
// experts l, l+32, ...); k rounds of a warp-wide arg-max over
// (logit descending, id ascending) pick the slots in order.
constexpr int kTopkWarps = 8;
constexpr int kTopkTokPerWarp = 8;
constexpr int kTopkTokPerBlock = kTopkWarps * kTopkTokPerWarp;

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ logits, int T,
                                                          int E, int k, int32_t* __restrict__ topk_idx,
                                                          float* __restrict__ topk_w,
                                                          int32_t* __restrict__ blk_hist) {
  __shared__ int hist[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nq = (E + 31) / 32;
  for (int it = 0; it < kTopkTokPerWarp; ++it) {
    const int t = blockIdx.x * kTopkTokPerBlock + warp * kTopkTokPerWarp + it;
    if (t >= T) break;
    float v[32];
#pragma unroll
    for (int q = 0; q < 32; ++q) {
      const int e = lane + 32 * q;
      v[q] = (q < nq && e < E) ? logits[(size_t)t * E + e] : -FLT_MAX;
    }
    uint32_t taken = 0;
    float my_v = 0.f;
    int my_i = 0;
    for (int j = 0; j < k; ++j) {
      float bv = 0.f;
      int bi = INT_MAX;
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const int e = lane + 32 * q;
        if (q < nq && e < E && !((taken >> q) & 1u) && (bi == INT_MAX || better(v[q], e, bv, bi))) {
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
      atomicAdd(&hist[my_i], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) blk_hist[(size_t)blockIdx.x * E + e] = hist[e];
}

// ------------------------------------------------------------ offsets kernel
// One CTA: counts[e] = sum of per-block histograms, exclusive scan -> offsets,
// EP-rank row ranges.
__global__ void __launch_bounds__(1024) router_offsets_kernel(const int32_t* __restrict__ blk_hist,
                                                              int nblk, int E, int ep_size,
                                                              int32_t* __restrict__ counts,
                                                              int32_t* __restrict__ offsets,
                                                              int32_t* __restrict__ rank_offsets) {
  __shared__ int warp_sum[32];
  __shared__ int excl[kMaxExperts + 1];
  const int e = threadIdx.x;
  int c = 0;
  if (e < E)
    for (int b = 0; b < nblk; ++b) c += blk_hist[(size_t)b * E + e];
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
    int ws = warp_sum[lane];
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
    counts[e] = c;
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
  *logits_bytes = align256(sizeof(float) * (size_t)T * E);
  *hist_bytes = align256(sizeof(int32_t) * (nblk > 0 ? nblk : 1) * E);
  return (int)nblk;
}

struct BwdLayout {
  int Ep, S;
  size_t dl2, dl3, wr3, seg, part, total;
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
  L.total = off;
  return L;
}

bool g_logit_attr[64] = {};

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
  if (!x || !Wr || !topk_idx || !topk_w || !counts || !offsets || !rank_offsets || !ws)
    return fail(MOE_ERR_INVALID_ARG, "moe_route_topk: NULL pointer argument");
  if (!aligned16(x) || !aligned16(Wr) || !aligned16(ws) || (bias && !aligned16(bias)))
    return fail(MOE_ERR_ALIGNMENT, "moe_route_topk: x, Wr, bias and ws must be 16-byte aligned");
  size_t lb, hb;
  const int nblk = route_ws_layout(T, E, &lb, &hb);
  if (ws_bytes < lb + hb)
    return fail(MOE_ERR_WORKSPACE, "moe_route_topk: workspace %zu < %zu bytes", ws_bytes, lb + hb);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* logits = static_cast<float*>(ws);
  int32_t* blk_hist = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + lb);
  const int dev = current_device();
  if (dev < 0) return fail(MOE_ERR_CUDA, "moe_route_topk: no current CUDA device");
  if (!g_logit_attr[dev]) {
    cudaFuncSetAttribute(router_logits_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)kLogitSmem);
    cudaFuncSetAttribute(router_logits_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)kLogitSmem);
    g_logit_attr[dev] = true;
  }
  if (T > 0) {
    dim3 grid((T + kLogitTok - 1) / kLogitTok, (E + kLogitExp - 1) / kLogitExp);
    const bool vec = (E % 8) == 0;
    if (vec)
      router_logits_kernel<true><<<grid, 256, kLogitSmem, s>>>(
          static_cast<const __nv_bfloat16*>(x), Wr, bias, T, H, E, logits);
    else
      router_logits_kernel<false><<<grid, 256, kLogitSmem, s>>>(
          static_cast<const __nv_bfloat16*>(x), Wr, bias, T, H, E, logits);
    if (int rc = check_launch("moe_route_topk: logits kernel")) return rc;
    router_topk_kernel<<<nblk, 256, 0, s>>>(logits, T, E, k, topk_idx, topk_w, blk_hist);
    if (int rc = check_launch("moe_route_topk: top-k kernel")) return rc;
  }
  router_offsets_kernel<<<1, 1024, 0, s>>>(blk_hist, T > 0 ? nblk : 0, E, ep_size, counts,
                                           offsets, rank_offsets);
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
  if (!d_w || !topk_w || !topk_idx || !x || !Wr || !dx_acc || !dWr || !dx || !ws)
    return fail(MOE_ERR_INVALID_ARG, "moe_route_topk_bwd: NULL pointer argument");
  if (!aligned16(x) || !aligned16(Wr) || !aligned16(dx_acc) || !aligned16(dWr) || !aligned16(dx) ||
      !aligned16(ws))
    return fail(MOE_ERR_ALIGNMENT, "moe_route_topk_bwd: tensors and ws must be 16-byte aligned");
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
  if (int rc = launch_dw_split(x, dl2, T, H, 2 * L.Ep, seg, L.S, part, s)) return rc;
  const size_t nred = (size_t)H * E;
  router_bwd_reduce_kernel<<<(int)((nred + 255) / 256 < 4096 ? (nred + 255) / 256 : 4096), 256, 0,
                             s>>>(part, L.S, H, E, L.Ep, dWr, accumulate);
  return check_launch("moe_route_topk_bwd: reduce kernel");
}

}  // extern "C"
