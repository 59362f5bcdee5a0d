/*
 * CPU oracle for the MoE expert layer -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded fp32 restatement of what the layer computes,
 * used to check the CUDA library.  Nothing in the product path may load it.
 * It shares no code with the CUDA sources.
 *
 * What the layer is, and where it is described:
 *  - "FSDPTurbo EP/EFSDP and LlamaFactory FSDP2/CP Design", section 3 (the
 *    dispatcher table): the expert module runs permute -> grouped matmul ->
 *    unpermute, with all-to-all token dispatch/combine around the grouped
 *    matmul; the fused dispatcher must cope with experts that receive no
 *    tokens.
 *  - "Qwen3-MoE-30B-A3B模型EP+FSDP2并行方案", section on the model: 128
 *    experts, hidden 2048, intermediate 768; up [E,768,2048], down
 *    [E,2048,768]; the gate tensor printed as [E,768,768] is read as
 *    [E,768,2048] like up.  Same page, "完整并行流程": experts are split over
 *    EP ranks in contiguous dim-0 blocks (128/8 = 16 per rank).
 *  - Same page, "为什么这么设计": the all-to-all carries tokens to their
 *    experts in the forward pass and gradients back in the backward pass.
 *  - "TorchTitan FSDP2 完全指南", mixed-precision section: bf16 parameters
 *    with fp32 gradient reduction -- hence fp32 weight gradients here.
 *
 * The pages never write out the router, the activation, the permutation
 * order or the backward pass.  The readings taken (plainest ones):
 *  R1. Router: logits = x.Wr (+bias), Wr stored [H,E] fp32; the k largest
 *      logits are selected in descending order, equal logits going to the
 *      lower expert id; weights are the softmax over the selected logits
 *      (identical to a full softmax renormalised over the selected experts).
 *      No capacity limit, no dropped tokens, no shared expert, no aux loss.
 *  R2. Logit summation order (needed so that selection can be compared bit
 *      for bit): the h axis is cut into blocks of ORACLE_LOGIT_BLOCK=256
 *      consecutive positions; each block is summed in increasing h with
 *      fused multiply-add starting from 0; the block sums are added left to
 *      right in fp32; the bias, if any, is added last.
 *  R3. Permutation: rows are ordered by expert, and within an expert by
 *      token index (stable), so EP rank r's block is the contiguous row
 *      range of experts [r*E/ep, (r+1)*E/ep).
 *  R4. Expert FFN: h = silu(x.Wg^T) * (x.Wu^T), silu(g) = g/(1+exp(-g));
 *      y = h.Wd^T; weights stored [E, out, in].
 *  R5. Combine: y[t] = sum over slots j = 0..k-1, in that order, of
 *      w[t,j] * y_perm[row(t,j)].
 *  R6. Backward: the exact derivative of R1..R5 with respect to x, Wr, Wg,
 *      Wu, Wd; the routing indices and the bias get no gradient; weight
 *      gradients are fp32, overwritten unless `accumulate` is set (then the
 *      freshly computed sum is added to what the buffer holds).
 *  R7. FP8 forward.  "TorchTitan FSDP2 完全指南", performance table, reports
 *      the gain of FP8 matmuls in training but gives no recipe.  Reading:
 *      e4m3 codes (1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 *      bits, no infinities, largest finite magnitude 448) with one fp32
 *      scale per row of the operand as stored: a token row of x, a
 *      permuted row of h, an output channel of one expert's weight (a row
 *      of Wg/Wu/Wd seen as [E*out, in]).  A row a[0..n) gets
 *      s = amax/448 (fp32 division; s = 1 for an all-zero row) and
 *      q[j] = e4m3(a[j] / s) (fp32 division; round to nearest, ties to
 *      even; magnitudes at or above 448 give 448; the sign is kept, also
 *      on a zero).  The FP8 GEMMs compute
 *      g[r,n] = s_a[r] * s_w[e,n] * sum_k dec(a[r,k]) * dec(w[e,n,k]),
 *      the sum taken in double (every product of two e4m3 values is exact).
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

static float widen_bf16(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static int seg_expert_of(const int32_t* seg_expert, int s) {
  return seg_expert ? seg_expert[s] : s;
}

static int check_segments(int num_seg, const int32_t* seg_offsets, const int32_t* seg_expert,
                          int R, int E) {
  if (num_seg < 0 || (num_seg > 0 && !seg_offsets)) return -1;
  for (int s = 0; s < num_seg; ++s) {
    if (seg_offsets[s] < 0 || seg_offsets[s + 1] < seg_offsets[s] || seg_offsets[s + 1] > R)
      return -1;
    int e = seg_expert_of(seg_expert, s);
    if (e < 0 || e >= E) return -1;
  }
  return 0;
}

/* ---------------------------------------------------------------- A1 router */

/* R2: blocked fp32 sum of x[t,:].Wr[:,e] for every e of one token. */
static void logits_of_token(const uint16_t* xrow, const float* Wr, const float* bias, int H,
                            int E, float* logit, float* part) {
  for (int e = 0; e < E; ++e) logit[e] = 0.0f;
  for (int h0 = 0; h0 < H; h0 += ORACLE_LOGIT_BLOCK) {
    int h1 = h0 + ORACLE_LOGIT_BLOCK < H ? h0 + ORACLE_LOGIT_BLOCK : H;
    for (int e = 0; e < E; ++e) part[e] = 0.0f;
    for (int h = h0; h < h1; ++h) {
      float xv = widen_bf16(xrow[h]);
      const float* w = Wr + (size_t)h * E;
      for (int e = 0; e < E; ++e) part[e] = fmaf(xv, w[e], part[e]);
    }
    for (int e = 0; e < E; ++e) logit[e] = (h0 == 0) ? part[e] : logit[e] + part[e];
  }
  if (bias)
    for (int e = 0; e < E; ++e) logit[e] = logit[e] + bias[e];
}

int oracle_router_logits(const uint16_t* x, const float* Wr, const float* bias, int T, int H,
                         int E, float* logits) {
  if (T < 0 || H <= 0 || E <= 0 || !x || !Wr || !logits) return -1;
  float* part = (float*)malloc(sizeof(float) * (size_t)E);
  if (!part) return -2;
  for (int t = 0; t < T; ++t)
    logits_of_token(x + (size_t)t * H, Wr, bias, H, E, logits + (size_t)t * E, part);
  free(part);
  return 0;
}

int oracle_route_topk(const uint16_t* x, const float* Wr, const float* bias, int T, int H, int E,
                      int k, int ep_size, int32_t* topk_idx, float* topk_w, int32_t* counts,
                      int32_t* offsets, int32_t* rank_offsets) {
  if (T < 0 || H <= 0 || E <= 0 || k < 1 || k > E || ep_size < 1 || E % ep_size) return -1;
  if (!x || !Wr || !topk_idx || !topk_w || !counts || !offsets || !rank_offsets) return -1;
  float* logit = (float*)malloc(sizeof(float) * (size_t)E);
  float* part = (float*)malloc(sizeof(float) * (size_t)E);
  float* ex = (float*)malloc(sizeof(float) * (size_t)k);
  unsigned char* taken = (unsigned char*)malloc((size_t)E);
  if (!logit || !part || !ex || !taken) {
    free(logit); free(part); free(ex); free(taken);
    return -2;
  }
  for (int t = 0; t < T; ++t) {
    logits_of_token(x + (size_t)t * H, Wr, bias, H, E, logit, part);
    memset(taken, 0, (size_t)E);
    /* R1: pick the largest remaining logit k times; scanning e upwards with a
       strict '>' keeps the lower id among equal logits. */
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || logit[e] > logit[best])) best = e;
      taken[best] = 1;
      topk_idx[(size_t)t * k + j] = best;
    }
    /* softmax over the selected logits, shifted by the largest one (slot 0) */
    float m = logit[topk_idx[(size_t)t * k]];
    float s = 0.0f;
    for (int j = 0; j < k; ++j) {
      ex[j] = expf(logit[topk_idx[(size_t)t * k + j]] - m);
      s = s + ex[j];
    }
    for (int j = 0; j < k; ++j) topk_w[(size_t)t * k + j] = ex[j] / s;
  }
  /* A2: histogram of expert ids over all T*k slots, exclusive prefix sum,
     and the row range of each EP rank's contiguous block of experts. */
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (size_t q = 0; q < (size_t)T * k; ++q) counts[topk_idx[q]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int per_rank = E / ep_size;
  for (int r = 0; r <= ep_size; ++r) rank_offsets[r] = offsets[r * per_rank];
  free(logit); free(part); free(ex); free(taken);
  return 0;
}

/* -------------------------------------------------------------- A3 dispatch */

int oracle_dispatch(const uint16_t* x, const int32_t* topk_idx, const int32_t* offsets, int T,
                    int H, int E, int k, uint16_t* x_perm, int32_t* row_of_slot,
                    int32_t* token_of_row) {
  if (T < 0 || H <= 0 || E <= 0 || k < 1 || !topk_idx || !offsets || !row_of_slot ||
      !token_of_row)
    return -1;
  int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  if (!fill) return -2;
  /* R3: visiting tokens in increasing order and handing out each expert's
     rows in that order makes row(t,j) = offsets[e] + #{t' < t routed to e}. */
  for (int t = 0; t < T; ++t) {
    for (int j = 0; j < k; ++j) {
      int e = topk_idx[(size_t)t * k + j];
      if (e < 0 || e >= E) { free(fill); return -1; }
      int row = offsets[e] + fill[e];
      fill[e] += 1;
      row_of_slot[(size_t)t * k + j] = row;
      token_of_row[row] = t;
      if (x && x_perm)
        memcpy(x_perm + (size_t)row * H, x + (size_t)t * H, sizeof(uint16_t) * (size_t)H);
    }
  }
  free(fill);
  return 0;
}

/* ------------------------------------------------------ A4 gate/up + SwiGLU */

int oracle_grouped_gemm_swiglu(const float* x_perm, const uint16_t* Wg, const uint16_t* Wu,
                               int num_seg, const int32_t* seg_offsets, const int32_t* seg_expert,
                               int R, int H, int I, int E, float* h, float* gu) {
  if (H <= 0 || I <= 0 || E <= 0 || !x_perm || !Wg || !Wu || !h) return -1;
  if (check_segments(num_seg, seg_offsets, seg_expert, R, E)) return -1;
  for (int s = 0; s < num_seg; ++s) {
    int e = seg_expert_of(seg_expert, s);
    for (int r = seg_offsets[s]; r < seg_offsets[s + 1]; ++r) {
      const float* a = x_perm + (size_t)r * H;
      for (int i = 0; i < I; ++i) {
        const uint16_t* wg = Wg + ((size_t)e * I + i) * H;
        const uint16_t* wu = Wu + ((size_t)e * I + i) * H;
        float g = 0.0f, u = 0.0f;
        for (int c = 0; c < H; ++c) {
          g = g + a[c] * widen_bf16(wg[c]);
          u = u + a[c] * widen_bf16(wu[c]);
        }
        float silu = g / (1.0f + expf(-g));
        h[(size_t)r * I + i] = silu * u;
        if (gu) {
          gu[(size_t)r * 2 * I + i] = g;
          gu[(size_t)r * 2 * I + I + i] = u;
        }
      }
    }
  }
  return 0;
}

/* ---------------------------------------------------------------- A5 down */

int oracle_grouped_gemm_down(const float* h, const uint16_t* Wd, int num_seg,
                             const int32_t* seg_offsets, const int32_t* seg_expert, int R, int H,
                             int I, int E, float* y_perm) {
  if (H <= 0 || I <= 0 || E <= 0 || !h || !Wd || !y_perm) return -1;
  if (check_segments(num_seg, seg_offsets, seg_expert, R, E)) return -1;
  for (int s = 0; s < num_seg; ++s) {
    int e = seg_expert_of(seg_expert, s);
    for (int r = seg_offsets[s]; r < seg_offsets[s + 1]; ++r) {
      const float* a = h + (size_t)r * I;
      for (int n = 0; n < H; ++n) {
        const uint16_t* w = Wd + ((size_t)e * H + n) * I;
        float acc = 0.0f;
        for (int i = 0; i < I; ++i) acc = acc + a[i] * widen_bf16(w[i]);
        y_perm[(size_t)r * H + n] = acc;
      }
    }
  }
  return 0;
}

/* ------------------------------------------------------------- A6 combine */

int oracle_combine(const float* y_perm, const float* topk_w, const int32_t* row_of_slot, int T,
                   int H, int k, float* y) {
  if (T < 0 || H <= 0 || k < 1 || !y_perm || !topk_w || !row_of_slot || !y) return -1;
  for (int t = 0; t < T; ++t) {
    for (int c = 0; c < H; ++c) {
      float acc = 0.0f;
      for (int j = 0; j < k; ++j) {
        size_t row = (size_t)row_of_slot[(size_t)t * k + j];
        acc = acc + topk_w[(size_t)t * k + j] * y_perm[row * H + c];
      }
      y[(size_t)t * H + c] = acc;
    }
  }
  return 0;
}

/* --------------------------------------------------------- B1 combine bwd */

int oracle_combine_bwd(const float* dy, const float* y_perm, const float* topk_w,
                       const int32_t* row_of_slot, int T, int H, int k, float* dy_perm,
                       float* d_w) {
  if (T < 0 || H <= 0 || k < 1 || !dy || !y_perm || !topk_w || !row_of_slot || !dy_perm || !d_w)
    return -1;
  for (int t = 0; t < T; ++t) {
    const float* g = dy + (size_t)t * H;
    for (int j = 0; j < k; ++j) {
      size_t row = (size_t)row_of_slot[(size_t)t * k + j];
      float w = topk_w[(size_t)t * k + j];
      float dot = 0.0f;
      for (int c = 0; c < H; ++c) {
        dy_perm[row * H + c] = w * g[c];
        dot = dot + g[c] * y_perm[row * H + c];
      }
      d_w[(size_t)t * k + j] = dot;
    }
  }
  return 0;
}

/* ------------------------------------------- B2 down bwd + SwiGLU bwd + dWd */

static void zero_or_keep(float* p, size_t n, int accumulate) {
  if (!accumulate) memset(p, 0, n * sizeof(float));
}

int oracle_grouped_gemm_down_bwd(const float* dy_perm, const float* h, const float* gu,
                                 const uint16_t* Wd, int num_seg, const int32_t* seg_offsets,
                                 const int32_t* seg_expert, int R, int H, int I, int E,
                                 float* dgu, float* dWd, int accumulate) {
  if (H <= 0 || I <= 0 || E <= 0 || !dy_perm || !h || !gu || !Wd || !dgu || !dWd) return -1;
  if (check_segments(num_seg, seg_offsets, seg_expert, R, E)) return -1;
  float* dh = (float*)malloc(sizeof(float) * (size_t)I);
  float* sum = (float*)malloc(sizeof(float) * (size_t)H * I);
  if (!dh || !sum) { free(dh); free(sum); return -2; }
  /* dh = dy_perm . Wd[e]  (dh[i] = sum_n dy[n] Wd[e][n][i], in n order) and
     the SwiGLU derivative: with s = sigmoid(g), silu'(g) = s*(1 + g*(1-s)). */
  for (int s = 0; s < num_seg; ++s) {
    int e = seg_expert_of(seg_expert, s);
    for (int r = seg_offsets[s]; r < seg_offsets[s + 1]; ++r) {
      const float* d = dy_perm + (size_t)r * H;
      for (int i = 0; i < I; ++i) dh[i] = 0.0f;
      for (int n = 0; n < H; ++n) {
        const uint16_t* w = Wd + ((size_t)e * H + n) * I;
        for (int i = 0; i < I; ++i) dh[i] = dh[i] + d[n] * widen_bf16(w[i]);
      }
      for (int i = 0; i < I; ++i) {
        float g = gu[(size_t)r * 2 * I + i];
        float u = gu[(size_t)r * 2 * I + I + i];
        float sg = 1.0f / (1.0f + expf(-g));
        dgu[(size_t)r * 2 * I + i] = dh[i] * u * sg * (1.0f + g * (1.0f - sg));
        dgu[(size_t)r * 2 * I + I + i] = dh[i] * (g * sg);
      }
    }
  }
  /* dWd[e] = sum over e's rows (segments in order, rows in order) of
     dy_perm[r]^T h[r]; experts with no rows get a zero sum. */
  for (int e = 0; e < E; ++e) {
    memset(sum, 0, sizeof(float) * (size_t)H * I);
    for (int s = 0; s < num_seg; ++s) {
      if (seg_expert_of(seg_expert, s) != e) continue;
      for (int r = seg_offsets[s]; r < seg_offsets[s + 1]; ++r) {
        const float* d = dy_perm + (size_t)r * H;
        const float* a = h + (size_t)r * I;
        for (int n = 0; n < H; ++n)
          for (int i = 0; i < I; ++i) sum[(size_t)n * I + i] = sum[(size_t)n * I + i] + d[n] * a[i];
      }
    }
    float* out = dWd + (size_t)e * H * I;
    zero_or_keep(out, (size_t)H * I, accumulate);
    for (size_t q = 0; q < (size_t)H * I; ++q) out[q] = out[q] + sum[q];
  }
  free(dh); free(sum);
  return 0;
}

/* ------------------------------------------------ B3 gate/up bwd + dWg, dWu */

int oracle_grouped_gemm_swiglu_bwd(const float* dgu, const float* x_perm, const uint16_t* Wg,
                                   const uint16_t* Wu, int num_seg, const int32_t* seg_offsets,
                                   const int32_t* seg_expert, int R, int H, int I, int E,
                                   float* dx_perm, float* dWg, float* dWu, int accumulate) {
  if (H <= 0 || I <= 0 || E <= 0 || !dgu || !x_perm || !Wg || !Wu || !dx_perm || !dWg || !dWu)
    return -1;
  if (check_segments(num_seg, seg_offsets, seg_expert, R, E)) return -1;
  float* sg = (float*)malloc(sizeof(float) * (size_t)I * H);
  float* su = (float*)malloc(sizeof(float) * (size_t)I * H);
  if (!sg || !su) { free(sg); free(su); return -2; }
  /* dx_perm = [dg du] . [Wg[e]; Wu[e]]: one reduction over 2I terms, the
     Wg half first, each half in increasing i. */
  for (int s = 0; s < num_seg; ++s) {
    int e = seg_expert_of(seg_expert, s);
    for (int r = seg_offsets[s]; r < seg_offsets[s + 1]; ++r) {
      const float* dg = dgu + (size_t)r * 2 * I;
      const float* du = dg + I;
      float* out = dx_perm + (size_t)r * H;
      for (int c = 0; c < H; ++c) out[c] = 0.0f;
      for (int i = 0; i < I; ++i) {
        const uint16_t* w = Wg + ((size_t)e * I + i) * H;
        for (int c = 0; c < H; ++c) out[c] = out[c] + dg[i] * widen_bf16(w[c]);
      }
      for (int i = 0; i < I; ++i) {
        const uint16_t* w = Wu + ((size_t)e * I + i) * H;
        for (int c = 0; c < H; ++c) out[c] = out[c] + du[i] * widen_bf16(w[c]);
      }
    }
  }
  /* dWg[e] = dg^T x_perm, dWu[e] = du^T x_perm over e's rows. */
  for (int e = 0; e < E; ++e) {
    memset(sg, 0, sizeof(float) * (size_t)I * H);
    memset(su, 0, sizeof(float) * (size_t)I * H);
    for (int s = 0; s < num_seg; ++s) {
      if (seg_expert_of(seg_expert, s) != e) continue;
      for (int r = seg_offsets[s]; r < seg_offsets[s + 1]; ++r) {
        const float* dg = dgu + (size_t)r * 2 * I;
        const float* du = dg + I;
        const float* a = x_perm + (size_t)r * H;
        for (int i = 0; i < I; ++i)
          for (int c = 0; c < H; ++c) {
            sg[(size_t)i * H + c] = sg[(size_t)i * H + c] + dg[i] * a[c];
            su[(size_t)i * H + c] = su[(size_t)i * H + c] + du[i] * a[c];
          }
      }
    }
    float* og = dWg + (size_t)e * I * H;
    float* ou = dWu + (size_t)e * I * H;
    zero_or_keep(og, (size_t)I * H, accumulate);
    zero_or_keep(ou, (size_t)I * H, accumulate);
    for (size_t q = 0; q < (size_t)I * H; ++q) {
      og[q] = og[q] + sg[q];
      ou[q] = ou[q] + su[q];
    }
  }
  free(sg); free(su);
  return 0;
}

/* -------------------------------------------------------- B4 dispatch bwd */

int oracle_dispatch_bwd(const float* dx_perm, const int32_t* row_of_slot, int T, int H, int k,
                        float* dx_acc) {
  if (T < 0 || H <= 0 || k < 1 || !dx_perm || !row_of_slot || !dx_acc) return -1;
  for (int t = 0; t < T; ++t)
    for (int c = 0; c < H; ++c) {
      float acc = 0.0f;
      for (int j = 0; j < k; ++j)
        acc = acc + dx_perm[(size_t)row_of_slot[(size_t)t * k + j] * H + c];
      dx_acc[(size_t)t * H + c] = acc;
    }
  return 0;
}

/* ---------------------------------------------------------- B5 router bwd */

int oracle_route_topk_bwd(const float* d_w, const float* topk_w, const int32_t* topk_idx,
                          const uint16_t* x, const float* Wr, const float* dx_acc, int T, int H,
                          int E, int k, float* dWr, float* dx, int accumulate) {
  if (T < 0 || H <= 0 || E <= 0 || k < 1 || k > E || !d_w || !topk_w || !topk_idx || !x ||
      !Wr || !dx_acc || !dWr || !dx)
    return -1;
  float* dl = (float*)malloc(sizeof(float) * (size_t)(T > 0 ? T : 1) * k);
  float* sum = (float*)calloc((size_t)H * E, sizeof(float));
  if (!dl || !sum) { free(dl); free(sum); return -2; }
  /* Softmax over the selected logits: d logit_j = w_j (d_w_j - sum_i w_i d_w_i);
     unselected logits get no gradient. */
  for (int t = 0; t < T; ++t) {
    const float* w = topk_w + (size_t)t * k;
    const float* g = d_w + (size_t)t * k;
    float s = 0.0f;
    for (int j = 0; j < k; ++j) s = s + w[j] * g[j];
    for (int j = 0; j < k; ++j) dl[(size_t)t * k + j] = w[j] * (g[j] - s);
  }
  /* dWr[c,e] = sum over tokens t (increasing) that selected e of x[t,c] dl[t,e] */
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      int e = topk_idx[(size_t)t * k + j];
      if (e < 0 || e >= E) { free(dl); free(sum); return -1; }
      float d = dl[(size_t)t * k + j];
      for (int c = 0; c < H; ++c)
        sum[(size_t)c * E + e] = sum[(size_t)c * E + e] + widen_bf16(x[(size_t)t * H + c]) * d;
    }
  zero_or_keep(dWr, (size_t)H * E, accumulate);
  for (size_t q = 0; q < (size_t)H * E; ++q) dWr[q] = dWr[q] + sum[q];
  /* dx[t] = dx_acc[t] + sum_j dl[t,j] Wr[:, e_j]  (the router's share of dX) */
  for (int t = 0; t < T; ++t)
    for (int c = 0; c < H; ++c) {
      float acc = dx_acc[(size_t)t * H + c];
      for (int j = 0; j < k; ++j)
        acc = acc + dl[(size_t)t * k + j] * Wr[(size_t)c * E + topk_idx[(size_t)t * k + j]];
      dx[(size_t)t * H + c] = acc;
    }
  free(dl); free(sum);
  return 0;
}

/* ------------------------------------------------------------ R7 FP8 e4m3 */

/* Value of an e4m3 code: exponent field 0 is subnormal (m * 2^-9); fields
 * 1..15 are (1 + m/8) * 2^(field-7); magnitude code 0x7F is NaN. */
static double e4m3_value(uint8_t c) {
  const int field = (c >> 3) & 15, m = c & 7;
  double v;
  if (field == 15 && m == 7) return NAN;
  if (field == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + m / 8.0, field - 7);
  return (c & 0x80) ? -v : v;
}

/* Round-to-nearest-even of |v| onto the e4m3 grid, saturating at 448. */
static uint8_t e4m3_code(float v) {
  const uint8_t sign = signbit(v) ? 0x80 : 0x00;
  const double m = fabs((double)v);
  if (m >= 448.0) return sign | 0x7E;
  int field, q;
  if (m < ldexp(1.0, -6)) {
    /* subnormal quantum 2^-9; q = 8 lands on the smallest normal (field 1) */
    q = (int)nearbyint(m / ldexp(1.0, -9));
    return sign | (uint8_t)q;
  }
  int e2;
  (void)frexp(m, &e2);  /* m = f * 2^e2, f in [0.5, 1): leading bit at 2^(e2-1) */
  const int e = e2 - 1;
  q = (int)nearbyint(m / ldexp(1.0, e - 3)); /* 8..16 quanta of 2^(e-3) */
  if (q == 16) {
    q = 8;
    field = e + 1 + 7;
  } else {
    field = e + 7;
  }
  if (field > 15 || (field == 15 && q - 8 > 6)) return sign | 0x7E;
  return sign | (uint8_t)((field << 3) | (q - 8));
}

int oracle_e4m3_decode(const uint8_t* q, int n, float* out) {
  if (n < 0 || (n > 0 && (!q || !out))) return -1;
  for (int i = 0; i < n; ++i) out[i] = (float)e4m3_value(q[i]);
  return 0;
}

int oracle_e4m3_encode(const float* v, int n, uint8_t* q) {
  if (n < 0 || (n > 0 && (!v || !q))) return -1;
  for (int i = 0; i < n; ++i) q[i] = e4m3_code(v[i]);
  return 0;
}

int oracle_quantize_rows_e4m3(const float* a, int rows, int cols, uint8_t* q, float* scale) {
  if (rows < 0 || cols <= 0 || (rows > 0 && (!a || !q || !scale))) return -1;
  for (int r = 0; r < rows; ++r) {
    const float* row = a + (size_t)r * cols;
    float amax = 0.0f;
    for (int j = 0; j < cols; ++j) amax = fmaxf(amax, fabsf(row[j]));
    const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    scale[r] = s;
    for (int j = 0; j < cols; ++j) q[(size_t)r * cols + j] = e4m3_code(row[j] / s);
  }
  return 0;
}

/* R7 with R4: h = silu(g) * u on e4m3 rows of x_perm and e4m3 weights. */
int oracle_grouped_gemm_swiglu_fp8(const uint8_t* aq, const float* a_scale, const uint8_t* Wgq,
                                   const float* Wg_scale, const uint8_t* Wuq, const float* Wu_scale,
                                   int num_seg, const int32_t* seg_offsets,
                                   const int32_t* seg_expert, int R, int H, int I, int E, float* h) {
  if (H <= 0 || I <= 0 || E <= 0 || !aq || !a_scale || !Wgq || !Wg_scale || !Wuq || !Wu_scale || !h)
    return -1;
  if (check_segments(num_seg, seg_offsets, seg_expert, R, E)) return -1;
  for (int s = 0; s < num_seg; ++s) {
    int e = seg_expert_of(seg_expert, s);
    for (int r = seg_offsets[s]; r < seg_offsets[s + 1]; ++r) {
      const uint8_t* a = aq + (size_t)r * H;
      for (int i = 0; i < I; ++i) {
        const uint8_t* wg = Wgq + ((size_t)e * I + i) * H;
        const uint8_t* wu = Wuq + ((size_t)e * I + i) * H;
        double sg = 0.0, su = 0.0;
        for (int c = 0; c < H; ++c) {
          const double av = e4m3_value(a[c]);
          sg += av * e4m3_value(wg[c]);
          su += av * e4m3_value(wu[c]);
        }
        const double g = (double)a_scale[r] * Wg_scale[(size_t)e * I + i] * sg;
        const double u = (double)a_scale[r] * Wu_scale[(size_t)e * I + i] * su;
        h[(size_t)r * I + i] = (float)(g / (1.0 + exp(-g)) * u);
      }
    }
  }
  return 0;
}

/* R7 with R4: y_perm = h . Wd^T on e4m3 rows of h and e4m3 weights. */
int oracle_grouped_gemm_down_fp8(const uint8_t* hq, const float* h_scale, const uint8_t* Wdq,
                                 const float* Wd_scale, int num_seg, const int32_t* seg_offsets,
                                 const int32_t* seg_expert, int R, int H, int I, int E,
                                 float* y_perm) {
  if (H <= 0 || I <= 0 || E <= 0 || !hq || !h_scale || !Wdq || !Wd_scale || !y_perm) return -1;
  if (check_segments(num_seg, seg_offsets, seg_expert, R, E)) return -1;
  for (int s = 0; s < num_seg; ++s) {
    int e = seg_expert_of(seg_expert, s);
    for (int r = seg_offsets[s]; r < seg_offsets[s + 1]; ++r) {
      const uint8_t* a = hq + (size_t)r * I;
      for (int n = 0; n < H; ++n) {
        const uint8_t* w = Wdq + ((size_t)e * H + n) * I;
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += e4m3_value(a[i]) * e4m3_value(w[i]);
        y_perm[(size_t)r * H + n] = (float)((double)h_scale[r] * Wd_scale[(size_t)e * H + n] * acc);
      }
    }
  }
  return 0;
}
