// A3 dispatch (permute), A6 combine (unpermute), B1 combine backward,
// B4 dispatch backward.
//
// "FSDPTurbo EP/EFSDP and LlamaFactory FSDP2/CP Design", section 3: the
// expert module runs permute -> grouped matmul -> unpermute.  The row order
// (expert-contiguous, stable by token) is the reading stated in moe_topk.h;
// with experts in ascending order every EP rank's block of experts
// ("Qwen3-MoE-30B-A3B模型EP+FSDP2并行方案", "完整并行流程") is one contiguous
// row range, which is the send buffer an all-to-all would consume.
//
// All four kernels are HBM-bound copies/reductions over 16-byte vectors
// (8 bf16): every row is read and written with fully coalesced 16-byte
// accesses, and each thread keeps all k of its independent loads in flight.
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kChunkTok = kRouteChunk;  // tokens per ranking chunk
// Blocks that share one chunk in the quantising dispatch: each ranks the
// chunk again (cheap) and quantises its share of the chunk's tokens, so
// that more warps hold a row in flight than one block per chunk gives.
// With four such blocks resident per SM (64 registers a thread) the
// quantising dispatch of 4096 tokens x 2048 to 8 experts of 128 takes
// 29 us against 40 us for one block per chunk, whose warps (124
// registers, 1.7 blocks an SM) waited on their rows' loads.
constexpr int kE4M3Split = 2;
// Batches of 32 slot expert ids the ranking warp keeps loaded ahead.
constexpr int kRankAhead = 4;

// --------------------------------------------------------------- histogram
// chunk_base[e][c] = number of slots of chunk c routed to expert e.
__global__ void __launch_bounds__(256) chunk_hist_kernel(const int32_t* __restrict__ topk_idx,
                                                         int T, int E, int k, int nchunk,
                                                         int32_t* __restrict__ chunk_base,
                                                         int* status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int hist[];  // [8 warps][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * 8 + warp;
  int* h = hist + (size_t)warp * E;
  for (int e = lane; e < E; e += 32) h[e] = 0;
  __syncwarp();
  if (c < nchunk) {
    const int s0 = c * kChunkTok * k;
    const int s1 = min(T, (c + 1) * kChunkTok) * k;
    for (int q = s0 + lane; q < s1; q += 32) {
      const int e = topk_idx[q];
      if (e >= 0 && e < E)
        atomicAdd(&h[e], 1);
      else
        set_status(status, MOE_STATUS_BAD_INDEX);
    }
    __syncwarp();
    for (int e = lane; e < E; e += 32) chunk_base[(size_t)e * nchunk + c] = h[e];
  }
}

// chunk_base[e][c] <- offsets[e] + sum_{c' < c} hist[e][c']  (in place).
// One warp per expert walks its row of chunks 32 at a time (coalesced): a
// warp scan of each batch plus the running carry gives every chunk its
// starting row.
__global__ void __launch_bounds__(256) chunk_scan_kernel(int32_t* __restrict__ chunk_base,
                                                         const int32_t* __restrict__ offsets,
                                                         int nchunk, int E, int* status) {
  pdl_wait();
  pdl_trigger();
  const int e = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (e >= E) return;
  int32_t* row = chunk_base + (size_t)e * nchunk;
  int carry = offsets[e];
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
  if (lane == 0 && carry != offsets[e + 1]) set_status(status, MOE_STATUS_COUNT_MISMATCH);
}

// ------------------------------------------------------- rank and row copy
// One CTA per chunk of 16 tokens, whose first row per expert is
// chunk_base[e][chunk] (+ base_add[e] when given: the route's chunk prefixes
// count from 0 within each expert).  Warp 0 hands out rows slot by slot in
// (token, slot) order: lanes that hold the same expert in one batch of 32
// slots get consecutive rows in lane order (= token order, since a token
// picks an expert at most once).  Then all 8 warps copy the chunk's token
// rows to their k destinations; the first row of every copying warp is
// loaded while warp 0 is still ranking.
// kE4M3: the destination rows receive the token's e4m3 codes instead (its
// scale from the largest |x| of the whole row, one fp32 scale written per
// destination row to xs_perm), the same codes as quantising x per token.
// Here kE4M3Split CTAs share a chunk (all rank it, the first writes the
// slot maps), and each warp converts 256 vectors of its row to codes once
// before storing them to the row's k destinations.
template <bool kE4M3>
__global__ void __launch_bounds__(256, kE4M3 ? 4 : 1) dispatch_kernel(
    const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ topk_idx,
    const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ base_add, int T, int H, int E, int k,
    void* __restrict__ x_perm_out, float* __restrict__ xs_perm, int32_t* __restrict__ row_of_slot,
    int32_t* __restrict__ token_of_row, int* status) {
  pdl_wait();
  pdl_trigger();
  constexpr int kSplit = kE4M3 ? kE4M3Split : 1;
  extern __shared__ int sm[];
  int* cnt = sm;                // [E]
  int* rows = sm + E;           // [kChunkTok * k]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x / kSplit, sub = blockIdx.x % kSplit;
  const int t0 = c * kChunkTok;
  const int nt = min(kChunkTok, T - t0);
  const int nslot = nt * k;
  const int R = T * k;
  const int nchunk = gridDim.x / kSplit;
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    cnt[e] = chunk_base[(size_t)e * nchunk + c] + (base_add ? base_add[e] : 0);
  const int nvec = H / 8;  // 16-byte vectors per row
  const int first = sub * 8 + warp;  // this warp's first token of the chunk
  // the first 8 vectors per lane of this warp's first token, in flight during the ranking
  uint4 pre[8];
  const bool prefetch = x_perm_out != nullptr && warp > 0 && first < nt;
  if (prefetch) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(t0 + first) * H);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int v = u * 32 + lane;
      if (v < nvec) pre[u] = __ldg(src + v);
    }
  }
  // the ranking warp's expert ids of the next kRankAhead batches of 32
  // slots, in flight (the first ones already while the counts load)
  const int32_t* ids = topk_idx + (size_t)t0 * k;
  int ahead[kRankAhead];
  if (warp == 0) {
#pragma unroll
    for (int u = 0; u < kRankAhead; ++u) ahead[u] = u * 32 + lane < nslot ? ids[u * 32 + lane] : -1;
  }
  __syncthreads();
  if (warp == 0) {
    for (int b = 0; b < nslot; b += 32) {
      const int q = b + lane;
      int e = ahead[0];
#pragma unroll
      for (int u = 0; u + 1 < kRankAhead; ++u) ahead[u] = ahead[u + 1];
      const int qn = q + 32 * kRankAhead;
      ahead[kRankAhead - 1] = qn < nslot ? ids[qn] : -1;
      if (q >= nslot || e < 0 || e >= E) e = -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      int row = -1;
      if (e >= 0) row = cnt[e] + rank;
      __syncwarp();
      if (e >= 0 && rank == 0) cnt[e] += __popc(peers);
      __syncwarp();
      if (q < nslot) {
        if (e < 0 || row < 0 || row >= R) {
          if (sub == 0) set_status(status, MOE_STATUS_BAD_INDEX);
          row = -1;
        }
        rows[q] = row;
        if (sub == 0) {
          row_of_slot[(size_t)t0 * k + q] = row;
          if (row >= 0) token_of_row[row] = t0 + q / k;
        }
      }
    }
  }
  __syncthreads();
  if (!x_perm_out) return;
  if constexpr (kE4M3) {
    uint8_t* xq = static_cast<uint8_t*>(x_perm_out);
    for (int i = first; i < nt; i += 8 * kSplit) {
      const int t = t0 + i;
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
      // the row's largest |x|; its first 256 vectors stay in registers (pre)
      float m = 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int v = u * 32 + lane;
        if (v < nvec) {
          if (!(prefetch && i == first)) pre[u] = __ldg(src + v);
          m = amax_bf16x8(pre[u], m);
        }
      }
      for (int v = 256 + lane; v < nvec; v += 32) m = amax_bf16x8(__ldg(src + v), m);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      const float sc = e4m3_row_scale(m);
      // codes of 256 vectors at a time, then stored to each destination row
      for (int v0 = 0; v0 < nvec; v0 += 32 * 8) {
        uint2 cd[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < nvec) cd[u] = e4m3_codes8(v0 == 0 ? pre[u] : __ldg(src + v), sc);
        }
        for (int j = 0; j < k; ++j) {
          const int row = rows[i * k + j];
          if (row < 0) continue;
          uint2* dst = reinterpret_cast<uint2*>(xq + (size_t)row * H);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int v = v0 + u * 32 + lane;
            if (v < nvec) dst[v] = cd[u];
          }
        }
      }
      if (lane < k) {
        const int row = rows[i * k + lane];
        if (row >= 0) xs_perm[row] = sc;
      }
    }
    return;
  }
  __nv_bfloat16* x_perm = static_cast<__nv_bfloat16*>(x_perm_out);
  for (int i = warp; i < nt; i += 8) {
    const int t = t0 + i;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    for (int v0 = 0; v0 < nvec; v0 += 32 * 8) {
      uint4 buf[8];
      if (prefetch && i == warp && v0 == 0) {
#pragma unroll
        for (int u = 0; u < 8; ++u) buf[u] = pre[u];
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < nvec) buf[u] = __ldg(src + v);
        }
      }
      for (int j = 0; j < k; ++j) {
        const int row = rows[i * k + j];
        if (row < 0) continue;
        uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)row * H);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < nvec) dst[v] = buf[u];
        }
      }
    }
  }
}

// ------------------------------------------------------------------ combine
// Thread = one 16-byte vector (8 columns) of one token; k independent row
// loads, fp32 accumulation in slot order, one bf16 rounding.
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  f[0] = bf16lo(v.x); f[1] = bf16hi(v.x); f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
  f[4] = bf16lo(v.z); f[5] = bf16hi(v.z); f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

template <bool kWeighted, bool kF32Out>
__global__ void __launch_bounds__(256) gather_sum_kernel(const __nv_bfloat16* __restrict__ src,
                                                         const float* __restrict__ topk_w,
                                                         const int32_t* __restrict__ row_of_slot,
                                                         int T, int H, int k, int R,
                                                         void* __restrict__ out, int* status) {
  pdl_wait();
  pdl_trigger();
  const int nvec = H / 8;
  const size_t total = (size_t)T * nvec;
  for (size_t gid = blockIdx.x * (size_t)blockDim.x + threadIdx.x; gid < total;
       gid += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(gid / nvec), v = (int)(gid % nvec);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int j0 = 0; j0 < k; j0 += 8) {
      uint4 buf[8];
      float wv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u;
        buf[u] = make_uint4(0, 0, 0, 0);
        wv[u] = 0.f;
        if (j < k) {
          const int row = __ldg(row_of_slot + (size_t)t * k + j);
          if (row >= 0 && row < R) {
            buf[u] = __ldg(reinterpret_cast<const uint4*>(src + (size_t)row * H) + v);
            wv[u] = kWeighted ? __ldg(topk_w + (size_t)t * k + j) : 1.f;
          } else {
            set_status(status, MOE_STATUS_BAD_INDEX);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (j0 + u < k) {
          float f[8];
          unpack8(buf[u], f);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            acc[i] = kWeighted ? __fmaf_rn(wv[u], f[i], acc[i]) : __fadd_rn(acc[i], f[i]);
        }
      }
    }
    if (kF32Out) {
      float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + (size_t)t * H) + 2 * v;
      o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
      reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + (size_t)t * H)[v] = pack8(acc);
    }
  }
}

// ------------------------------------------------------------ combine bwd
// Warp per token (grid-stride over tokens): the token's dy row sits in
// registers (8 vectors of 8 bf16 columns per lane at a time); for every slot
// the warp writes dy_perm[row] = w * dy[t] and reduces dy[t] . y_perm[row]
// (per-lane fp32 partial, then a fixed butterfly); lane j keeps d_w[t,j].
__global__ void __launch_bounds__(256) combine_bwd_kernel(
    const __nv_bfloat16* __restrict__ dy, const __nv_bfloat16* __restrict__ y_perm,
    const float* __restrict__ topk_w, const int32_t* __restrict__ row_of_slot, int T, int H, int k,
    int R, __nv_bfloat16* __restrict__ dy_perm, float* __restrict__ d_w, int* status) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int nvec = H / 8;
  const int nw = (int)((gridDim.x * blockDim.x) >> 5);
  for (int t = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); t < T; t += nw) {
    int my_row = lane < k ? __ldg(row_of_slot + (size_t)t * k + lane) : -1;
    const float my_w = lane < k ? __ldg(topk_w + (size_t)t * k + lane) : 0.f;
    if (lane < k && (my_row < 0 || my_row >= R)) {
      set_status(status, MOE_STATUS_BAD_INDEX);
      my_row = -1;
    }
    float my_dw = 0.f;
    for (int v0 = 0; v0 < nvec; v0 += 256) {
      uint4 gp[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int v = v0 + u * 32 + lane;
        gp[u] = v < nvec ? __ldg(reinterpret_cast<const uint4*>(dy + (size_t)t * H) + v) : make_uint4(0, 0, 0, 0);
      }
      for (int j = 0; j < k; ++j) {
        const int row = __shfl_sync(0xffffffffu, my_row, j);
        const float w = __shfl_sync(0xffffffffu, my_w, j);
        if (row < 0) continue;  // uniform across the warp
        uint4 yb[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int v = v0 + u * 32 + lane;
          yb[u] = v < nvec ? __ldg(reinterpret_cast<const uint4*>(y_perm + (size_t)row * H) + v)
                           : make_uint4(0, 0, 0, 0);
        }
        float p = 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int v = v0 + u * 32 + lane;
          float g[8], yv[8], o[8];
          unpack8(gp[u], g);
          unpack8(yb[u], yv);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            o[i] = w * g[i];
            p = __fmaf_rn(g[i], yv[i], p);
          }
          if (v < nvec) reinterpret_cast<uint4*>(dy_perm + (size_t)row * H)[v] = pack8(o);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
        if (lane == j) my_dw += p;
      }
    }
    if (lane < k) d_w[(size_t)t * k + lane] = my_dw;
  }
}

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

int grid_for(size_t work, int per_block) {
  const size_t b = (work + per_block - 1) / per_block;
  const size_t cap = (size_t)(sm_count() > 0 ? sm_count() : 148) * 16;
  return (int)(b < cap ? (b > 0 ? b : 1) : cap);
}

// The row kernel of a dispatch whose chunk bases are ready (chunk_base, plus
// base_add[e] when given).
template <bool kE4M3>
int dispatch_rows_launch(const void* x, const int32_t* topk_idx, const int32_t* chunk_base,
                         const int32_t* base_add, int T, int H, int E, int k, void* x_perm, float* xs_perm,
                         int32_t* row_of_slot, int32_t* token_of_row, cudaStream_t s, const char* fn) {
  const int nchunk = (T + kChunkTok - 1) / kChunkTok;
  launch_pdl(dispatch_kernel<kE4M3>, nchunk * (kE4M3 ? kE4M3Split : 1), 256, sizeof(int) * (E + kChunkTok * k), s,
             static_cast<const __nv_bfloat16*>(x), topk_idx, chunk_base, base_add, T, H, E, k, x_perm, xs_perm,
             row_of_slot, token_of_row, status_word());
  return check_launch(fn, "row kernel");
}

// Ranking (per-chunk histograms, their scan) and the row kernel of a dispatch
// whose scratch (the chunk bases) is `ws`.
template <bool kE4M3>
int dispatch_launch(const void* x, const int32_t* topk_idx, const int32_t* offsets, int T, int H, int E,
                    int k, void* x_perm, float* xs_perm, int32_t* row_of_slot, int32_t* token_of_row,
                    void* ws, cudaStream_t s, const char* fn) {
  int* status = status_word();
  const int nchunk = (T + kChunkTok - 1) / kChunkTok;
  int32_t* chunk_base = static_cast<int32_t*>(ws);
  launch_pdl(chunk_hist_kernel, (nchunk + 7) / 8, 256, sizeof(int) * 8 * E, s, topk_idx, T, E, k, nchunk,
             chunk_base, status);
  if (int rc = check_launch(fn, "histogram kernel")) return rc;
  launch_pdl(chunk_scan_kernel, (E + 7) / 8, 256, 0, s, chunk_base, offsets, nchunk, E, status);
  if (int rc = check_launch(fn, "scan kernel")) return rc;
  return dispatch_rows_launch<kE4M3>(x, topk_idx, chunk_base, nullptr, T, H, E, k, x_perm, xs_perm, row_of_slot,
                                     token_of_row, s, fn);
}

int check_rows_args(const char* fn, int T, int H, int k) {
  if (T < 0 || H <= 0 || k <= 0) return fail(MOE_ERR_INVALID_ARG, "%s: need T>=0, H>0, k>0", fn);
  if (H % 64 != 0 || k > kMaxTopK || (long long)T * k >= (1ll << 31))
    return fail(MOE_ERR_UNSUPPORTED_SHAPE, "%s: need H%%64==0, k<=32, T*k<2^31", fn);
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_dispatch_workspace_size(int T, int E, int k) {
  (void)k;
  if (T < 0 || E <= 0) return 0;
  const size_t nchunk = (size_t)((T + kChunkTok - 1) / kChunkTok);
  return align256(sizeof(int32_t) * (nchunk > 0 ? nchunk : 1) * E);
}

int moe_dispatch(const void* x, const int32_t* topk_idx, const int32_t* offsets, int T, int H,
                 int E, int k, void* x_perm, int32_t* row_of_slot, int32_t* token_of_row,
                 void* ws, size_t ws_bytes, void* stream) {
  clear_error();
  if (int rc = check_rows_args("moe_dispatch", T, H, k)) return rc;
  if (E <= 0 || E > kMaxExperts || k > E)
    return fail(MOE_ERR_UNSUPPORTED_SHAPE, "moe_dispatch: need 1<=E<=1024, k<=E");
  if (!ws || (T > 0 && (!topk_idx || !offsets || !row_of_slot || !token_of_row || (x_perm && !x))))
    return fail(MOE_ERR_INVALID_ARG, "moe_dispatch: NULL pointer argument");
  if ((x && !aligned16(x)) || (x_perm && !aligned16(x_perm)) || !aligned16(ws))
    return fail(MOE_ERR_ALIGNMENT, "moe_dispatch: x, x_perm and ws must be 16-byte aligned");
  const size_t need = moe_dispatch_workspace_size(T, E, k);
  if (ws_bytes < need)
    return fail(MOE_ERR_WORKSPACE, "moe_dispatch: workspace %zu < %zu bytes", ws_bytes, need);
  if (T == 0) return MOE_OK;
  return dispatch_launch<false>(x, topk_idx, offsets, T, H, E, k, x_perm, nullptr, row_of_slot,
                                token_of_row, ws, static_cast<cudaStream_t>(stream), "moe_dispatch");
}

int moe_dispatch_e4m3(const void* x, const int32_t* topk_idx, const int32_t* offsets, int T, int H,
                      int E, int k, void* xq_perm, float* xs_perm, int32_t* row_of_slot,
                      int32_t* token_of_row, void* ws, size_t ws_bytes, void* stream) {
  clear_error();
  const char* fn = "moe_dispatch_e4m3";
  if (int rc = check_rows_args(fn, T, H, k)) return rc;
  if (E <= 0 || E > kMaxExperts || k > E) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "%s: need 1<=E<=1024, k<=E", fn);
  if (!ws || (T > 0 && (!x || !topk_idx || !offsets || !xq_perm || !xs_perm || !row_of_slot || !token_of_row)))
    return fail(MOE_ERR_INVALID_ARG, "%s: NULL pointer argument", fn);
  if (!aligned16(x) || !aligned16(xq_perm) || !aligned16(ws) || (reinterpret_cast<uintptr_t>(xs_perm) & 3u))
    return fail(MOE_ERR_ALIGNMENT, "%s: x, xq_perm and ws must be 16-byte, xs_perm 4-byte aligned", fn);
  const size_t need = moe_dispatch_workspace_size(T, E, k);
  if (ws_bytes < need) return fail(MOE_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, ws_bytes, need);
  if (T == 0) return MOE_OK;
  return dispatch_launch<true>(x, topk_idx, offsets, T, H, E, k, xq_perm, xs_perm, row_of_slot, token_of_row,
                               ws, static_cast<cudaStream_t>(stream), fn);
}

int moe_dispatch_chunked(const void* x, const int32_t* topk_idx, const int32_t* offsets,
                         const int32_t* chunk_prefix, int T, int H, int E, int k, void* x_perm,
                         int32_t* row_of_slot, int32_t* token_of_row, void* stream) {
  clear_error();
  const char* fn = "moe_dispatch_chunked";
  if (int rc = check_rows_args(fn, T, H, k)) return rc;
  if (E <= 0 || E > kMaxExperts || k > E) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "%s: need 1<=E<=1024, k<=E", fn);
  if (T > 0 && (!topk_idx || !offsets || !chunk_prefix || !row_of_slot || !token_of_row || (x_perm && !x)))
    return fail(MOE_ERR_INVALID_ARG, "%s: NULL pointer argument", fn);
  if ((x && !aligned16(x)) || (x_perm && !aligned16(x_perm)))
    return fail(MOE_ERR_ALIGNMENT, "%s: x and x_perm must be 16-byte aligned", fn);
  if (T == 0) return MOE_OK;
  return dispatch_rows_launch<false>(x, topk_idx, chunk_prefix, offsets, T, H, E, k, x_perm, nullptr, row_of_slot,
                                     token_of_row, static_cast<cudaStream_t>(stream), fn);
}

int moe_dispatch_e4m3_chunked(const void* x, const int32_t* topk_idx, const int32_t* offsets,
                              const int32_t* chunk_prefix, int T, int H, int E, int k, void* xq_perm,
                              float* xs_perm, int32_t* row_of_slot, int32_t* token_of_row, void* stream) {
  clear_error();
  const char* fn = "moe_dispatch_e4m3_chunked";
  if (int rc = check_rows_args(fn, T, H, k)) return rc;
  if (E <= 0 || E > kMaxExperts || k > E) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "%s: need 1<=E<=1024, k<=E", fn);
  if (T > 0 && (!x || !topk_idx || !offsets || !chunk_prefix || !xq_perm || !xs_perm || !row_of_slot ||
                !token_of_row))
    return fail(MOE_ERR_INVALID_ARG, "%s: NULL pointer argument", fn);
  if (!aligned16(x) || !aligned16(xq_perm) || (reinterpret_cast<uintptr_t>(xs_perm) & 3u))
    return fail(MOE_ERR_ALIGNMENT, "%s: x and xq_perm must be 16-byte, xs_perm 4-byte aligned", fn);
  if (T == 0) return MOE_OK;
  return dispatch_rows_launch<true>(x, topk_idx, chunk_prefix, offsets, T, H, E, k, xq_perm, xs_perm, row_of_slot,
                                    token_of_row, static_cast<cudaStream_t>(stream), fn);
}



int moe_combine(const void* y_perm, const float* topk_w, const int32_t* row_of_slot, int T, int H,
                int k, void* y, void* stream) {
  clear_error();
  if (int rc = check_rows_args("moe_combine", T, H, k)) return rc;
  if (T == 0) return MOE_OK;
  if (!y_perm || !topk_w || !row_of_slot || !y)
    return fail(MOE_ERR_INVALID_ARG, "moe_combine: NULL pointer argument");
  if (!aligned16(y_perm) || !aligned16(y))
    return fail(MOE_ERR_ALIGNMENT, "moe_combine: y_perm and y must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t work = (size_t)T * (H / 8);
  launch_pdl(gather_sum_kernel<true, false>, grid_for(work, 256), 256, 0, s, 
      static_cast<const __nv_bfloat16*>(y_perm), topk_w, row_of_slot, T, H, k, T * k, y,
      status_word());
  return check_launch("moe_combine");
}

int moe_dispatch_bwd(const void* dx_perm, const int32_t* row_of_slot, int T, int H, int k,
                     float* dx_acc, void* stream) {
  clear_error();
  if (int rc = check_rows_args("moe_dispatch_bwd", T, H, k)) return rc;
  if (T == 0) return MOE_OK;
  if (!dx_perm || !row_of_slot || !dx_acc)
    return fail(MOE_ERR_INVALID_ARG, "moe_dispatch_bwd: NULL pointer argument");
  if (!aligned16(dx_perm) || !aligned16(dx_acc))
    return fail(MOE_ERR_ALIGNMENT, "moe_dispatch_bwd: dx_perm and dx_acc must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t work = (size_t)T * (H / 8);
  launch_pdl(gather_sum_kernel<false, true>, grid_for(work, 256), 256, 0, s, 
      static_cast<const __nv_bfloat16*>(dx_perm), nullptr, row_of_slot, T, H, k, T * k, dx_acc,
      status_word());
  return check_launch("moe_dispatch_bwd");
}

int moe_combine_bwd(const void* dy, const void* y_perm, const float* topk_w,
                    const int32_t* row_of_slot, int T, int H, int k, void* dy_perm, float* d_w,
                    void* stream) {
  clear_error();
  if (int rc = check_rows_args("moe_combine_bwd", T, H, k)) return rc;
  if (T == 0) return MOE_OK;
  if (!dy || !y_perm || !topk_w || !row_of_slot || !dy_perm || !d_w)
    return fail(MOE_ERR_INVALID_ARG, "moe_combine_bwd: NULL pointer argument");
  if (!aligned16(dy) || !aligned16(y_perm) || !aligned16(dy_perm))
    return fail(MOE_ERR_ALIGNMENT, "moe_combine_bwd: dy, y_perm and dy_perm must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  launch_pdl(combine_bwd_kernel, grid_for((size_t)T * 32, 256), 256, 0, s, static_cast<const __nv_bfloat16*>(dy),
                                       static_cast<const __nv_bfloat16*>(y_perm), topk_w,
                                       row_of_slot, T, H, k, T * k,
                                       static_cast<__nv_bfloat16*>(dy_perm), d_w, status_word());
  return check_launch("moe_combine_bwd");
}

// ------------------------------------------------- dispatch without workspace
//
// moe_dispatch_no_alloc runs the same three kernels as moe_dispatch, but its
// per-chunk histogram / row-base scratch lives in the file-scope device array
// below instead of a caller-provided workspace.  Every device that loads the
// library holds this array (1 MiB) until the process exits; all calls on a
// device share it, so calls that overlap on the GPU (other streams) race.
// Nothing has to start at zero: each call rewrites every entry it reads.

}  // extern "C"

namespace {

constexpr size_t kNoAllocScratchInts = 262144;  // 1 MiB of int32
static __device__ __align__(256) int32_t g_dispatch_scratch[kNoAllocScratchInts];

int32_t* g_dispatch_scratch_ptr[64] = {};
std::mutex g_dispatch_scratch_mu;

// Device address of g_dispatch_scratch on the current device, looked up once
// per device (host code cannot use the symbol's name as a device pointer).
int dispatch_scratch(int32_t** out) {
  const int dev = current_device();
  if (dev < 0) return fail(MOE_ERR_CUDA, "moe_dispatch_no_alloc: no current CUDA device");
  std::lock_guard<std::mutex> lk(g_dispatch_scratch_mu);
  if (!g_dispatch_scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(MOE_ERR_CUDA, "moe_dispatch_no_alloc: cudaGetSymbolAddress failed: %s",
                  cudaGetErrorString(e));
    }
    g_dispatch_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_dispatch_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_dispatch_no_alloc_max_scratch(void) { return kNoAllocScratchInts; }

int moe_dispatch_no_alloc(const void* x, const int32_t* topk_idx, const int32_t* offsets, int T,
                          int H, int E, int k, void* x_perm, int32_t* row_of_slot,
                          int32_t* token_of_row, void* stream) {
  clear_error();
  if (int rc = check_rows_args("moe_dispatch_no_alloc", T, H, k)) return rc;
  if (E <= 0 || E > kMaxExperts || k > E)
    return fail(MOE_ERR_UNSUPPORTED_SHAPE, "moe_dispatch_no_alloc: need 1<=E<=1024, k<=E");
  if (T > 0 && (!topk_idx || !offsets || !row_of_slot || !token_of_row || (x_perm && !x)))
    return fail(MOE_ERR_INVALID_ARG, "moe_dispatch_no_alloc: NULL pointer argument");
  if ((x && !aligned16(x)) || (x_perm && !aligned16(x_perm)))
    return fail(MOE_ERR_ALIGNMENT, "moe_dispatch_no_alloc: x and x_perm must be 16-byte aligned");
  const size_t nchunk = (size_t)((T + kChunkTok - 1) / kChunkTok);
  if (nchunk * (size_t)E > kNoAllocScratchInts)
    return fail(MOE_ERR_WORKSPACE,
                "moe_dispatch_no_alloc: ceil(T/16)*E = %zu exceeds the built-in scratch of %zu "
                "entries (use moe_dispatch with a workspace)",
                nchunk * (size_t)E, kNoAllocScratchInts);
  int32_t* chunk_base = nullptr;
  if (int rc = dispatch_scratch(&chunk_base)) return rc;
  if (T == 0) return MOE_OK;
  return dispatch_launch<false>(x, topk_idx, offsets, T, H, E, k, x_perm, nullptr, row_of_slot, token_of_row,
                                chunk_base, static_cast<cudaStream_t>(stream), "moe_dispatch_no_alloc");
}

}  // extern "C"
