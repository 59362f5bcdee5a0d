/*
 * moe_topk.h -- C ABI of the GB300 (sm_103a) MoE expert-layer library.
 *
 * The layer, as one GPU runs it for the tokens it holds:
 *
 *   forward   moe_route_topk -> moe_dispatch -> moe_grouped_gemm_swiglu
 *             -> moe_grouped_gemm_down -> moe_combine
 *   backward  moe_combine_bwd -> moe_grouped_gemm_down_bwd
 *             -> moe_grouped_gemm_swiglu_bwd -> moe_dispatch_bwd
 *             -> moe_route_topk_bwd
 *
 * Where the pages describe it:
 *   - "FSDPTurbo EP/EFSDP and LlamaFactory FSDP2/CP Design", section 3, the
 *     dispatcher table: the expert module is permute -> grouped matmul ->
 *     unpermute with all-to-all token dispatch/combine around the grouped
 *     matmul; the fused dispatcher must handle experts that receive no token.
 *   - "Qwen3-MoE-30B-A3B模型EP+FSDP2并行方案", model section: 128 experts,
 *     hidden 2048, expert intermediate 768, up [E,768,2048], down
 *     [E,2048,768] (gate read as [E,768,2048] like up); section
 *     "完整并行流程": experts are split over EP ranks in contiguous dim-0
 *     blocks; section "为什么这么设计": the all-to-all moves tokens to their
 *     experts forward and gradients back backward; section "Expert
 *     Parallelism Details": after EP sharding the expert compute runs on
 *     plain local tensors (hence raw pointers here).
 *   - "TorchTitan FSDP2 完全指南", mixed-precision section: bf16 parameters,
 *     fp32 gradient reduction (hence fp32 weight gradients).
 * The router math, the activation and the permutation order are not written
 * on the pages; the readings taken are stated at each function.
 *
 * Conventions (every function):
 *   - Returns MOE_OK (0) or a negative MOE_ERR_* code; moe_last_error_string()
 *     describes the last failure of the calling thread.
 *   - Asynchronous on `stream` (a cudaStream_t passed as void*, NULL = the
 *     legacy default stream).  Never synchronises (except
 *     moe_read_device_status), never allocates, never aborts.
 *   - All tensor pointers are DEVICE pointers owned by the caller, row-major,
 *     contiguous.  "bf16" tensors are passed as void* and hold IEEE bfloat16.
 *     Every tensor pointer must be 16-byte aligned.
 *   - Shape limits checked on the host before any launch: H and I multiples
 *     of 64, 1 <= E <= 1024, 1 <= k <= min(E, 32), T*k < 2^31, ep_size >= 1
 *     dividing E, num_seg <= 1024.  Violations return MOE_ERR_INVALID_ARG /
 *     MOE_ERR_UNSUPPORTED_SHAPE / MOE_ERR_ALIGNMENT and launch nothing.
 *   - Scratch memory ("workspace", device, caller-owned) is sized by the
 *     matching *_workspace_size query; a smaller ws_bytes returns
 *     MOE_ERR_WORKSPACE.  Workspaces are 16-byte aligned, except those of
 *     the backward GEMMs and the router backward, which hold TMA
 *     descriptors and must be 128-byte aligned (else MOE_ERR_ALIGNMENT).  A workspace may be reused by later calls on the
 *     same stream; calls that overlap on the GPU need separate workspaces.
 *   - Index data that lives on the device (topk_idx, offsets, segment
 *     tables) cannot be checked on the host.  Kernels clamp every access
 *     they derive from it, skip what is out of range, and record a device
 *     status word that moe_read_device_status() returns.
 *   - Results are deterministic (no floating-point atomics), except those
 *     of moe_grouped_gemm_down_combine, which adds with L2 reductions in no
 *     fixed order.
 *   - Expert weights are read only.  Weight gradients are fp32 and are
 *     overwritten, or added to when `accumulate` != 0.
 */
#ifndef MOE_TOPK_H
#define MOE_TOPK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)
#define MOE_ERR_UNSUPPORTED_SHAPE (-2)
#define MOE_ERR_ALIGNMENT (-3)
#define MOE_ERR_WORKSPACE (-4)
#define MOE_ERR_CUDA (-5)
#define MOE_ERR_DEVICE_CHECK (-6)

/* Device status bits recorded by kernels (see moe_read_device_status). */
#define MOE_STATUS_BAD_INDEX 1      /* an expert id / row / offset was out of range */
#define MOE_STATUS_BAD_SEGMENTS 2   /* a segment table was not monotone or exceeded R */
#define MOE_STATUS_COUNT_MISMATCH 4 /* offsets disagree with the histogram of topk_idx */
#define MOE_STATUS_TIMEOUT 8        /* a pipeline wait gave up (kernel returned early) */

/* ABI version of this header (major * 100 + minor). */
int moe_abi_version(void);

/* Text of the last error returned to the calling host thread ("" if none). */
const char* moe_last_error_string(void);

/* Copies the device status word (OR of MOE_STATUS_* bits set by kernels
 * since the last reset) to *status after synchronising `stream`; if reset is
 * non-zero the word is cleared.  The only synchronising call of the library. */
int moe_read_device_status(int* status, int reset, void* stream);

/* ------------------------------------------------------------------------
 * A1 + A2  router, top-k, expert histogram and offsets.
 *
 * For every token t:
 *   logits[t,e] = sum_h x[t,h] * Wr[h,e]  (+ bias[e])
 * in fp32 with a fixed order: h is cut into blocks of 256; each block is
 * summed in increasing h with fused multiply-add starting from 0; block sums
 * are added left to right; the bias is added last.  (Reading: the pages
 * never write the router out; this order is fixed so that selection is
 * reproducible bit for bit.)
 *   topk_idx[t,0..k) = the k largest logits in descending order, equal
 *                      logits to the lower expert id;
 *   topk_w[t,j]      = softmax over the k selected logits (equivalently, a
 *                      full softmax renormalised over the selected experts).
 * Then over all T*k slots:
 *   counts[e]        = number of slots routed to e;
 *   offsets[0..E]    = exclusive prefix sum of counts (offsets[E] = T*k);
 *   rank_offsets[r]  = offsets[r*E/ep_size], r = 0..ep_size: the row range
 *                      of EP rank r's contiguous block of E/ep_size experts
 *                      (the send-buffer split an all-to-all would use).
 * x: bf16 [T,H]; Wr: fp32 [H,E]; bias: fp32 [E] or NULL (no gradient).
 * Outputs: topk_idx int32 [T,k], topk_w fp32 [T,k], counts int32 [E],
 * offsets int32 [E+1], rank_offsets int32 [ep_size+1].
 * No capacity limit: every token keeps all k experts.  T == 0 is allowed.
 * The workspace holds the fp32 block sums of the logits, ceil(H/256) x T x E,
 * the slot total of every expert and the per-chunk slot counts described at
 * moe_route_topk_chunks.
 * ---------------------------------------------------------------------- */
size_t moe_route_topk_workspace_size(int T, int H, int E);
int moe_route_topk(const void* x, const float* Wr, const float* bias, int T, int H, int E, int k,
                   int ep_size, int32_t* topk_idx, float* topk_w, int32_t* counts,
                   int32_t* offsets, int32_t* rank_offsets, void* ws, size_t ws_bytes,
                   void* stream);

/* A1 + A2 as above, also returning where dispatch starts each chunk of 16
 * tokens in each expert's rows:
 *   chunk_prefix[e][c] = number of slots routed to expert e by tokens
 *                        0 .. 16c-1   (int32 [E][ceil(T/16)], c = chunk)
 * so the first row of chunk c's slots in expert e is offsets[e] +
 * chunk_prefix[e][c] (rows stable by token, "FSDPTurbo EP/EFSDP and
 * LlamaFactory FSDP2/CP Design", section 3, the permute step).  With it,
 * moe_dispatch_chunked permutes in one kernel instead of ranking the slots
 * again.  chunk_prefix may be NULL only when T == 0.  The workspace
 * (moe_route_topk_chunks_workspace_size) holds the logit block sums and the
 * expert totals only. */
size_t moe_route_topk_chunks_workspace_size(int T, int H, int E);
int moe_route_topk_chunks(const void* x, const float* Wr, const float* bias, int T, int H, int E, int k,
                          int ep_size, int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                          int32_t* rank_offsets, int32_t* chunk_prefix, void* ws, size_t ws_bytes,
                          void* stream);

/* ------------------------------------------------------------------------
 * A3  dispatch (permute).
 *
 * Row of slot (t,j) with expert e = topk_idx[t,j]:
 *   row(t,j) = offsets[e] + #{ t' < t : token t' routed to e }
 * i.e. expert-contiguous, stable by token index (reading of "permute" in
 * the dispatcher table; expert-ascending order makes each EP rank's block
 * contiguous).  x_perm[row(t,j)] = x[t]; row_of_slot[t,j] = row(t,j);
 * token_of_row[row(t,j)] = t.
 * x: bf16 [T,H]; topk_idx int32 [T,k]; offsets int32 [E+1] (from
 * moe_route_topk).  Outputs: x_perm bf16 [T*k,H], row_of_slot int32 [T,k],
 * token_of_row int32 [T*k].  x_perm may be NULL (indices only).
 * A histogram that disagrees with offsets sets MOE_STATUS_COUNT_MISMATCH.
 * ---------------------------------------------------------------------- */
size_t moe_dispatch_workspace_size(int T, int E, int k);
int moe_dispatch(const void* x, const int32_t* topk_idx, const int32_t* offsets, int T, int H,
                 int E, int k, void* x_perm, int32_t* row_of_slot, int32_t* token_of_row,
                 void* ws, size_t ws_bytes, void* stream);

/* A3 with the chunk prefixes of moe_route_topk_chunks: the same rows,
 * row_of_slot, token_of_row and x_perm as moe_dispatch (bit for bit), in
 * one kernel and with no workspace; the route already counted the slots of
 * every chunk of 16 tokens per expert.  chunk_prefix int32 [E][ceil(T/16)]
 * and offsets from the same moe_route_topk_chunks call.  x_perm may be NULL
 * (indices only).  A row outside [0, T*k) that inconsistent inputs would
 * give is skipped and sets MOE_STATUS_BAD_INDEX. */
int moe_dispatch_chunked(const void* x, const int32_t* topk_idx, const int32_t* offsets,
                         const int32_t* chunk_prefix, int T, int H, int E, int k, void* x_perm,
                         int32_t* row_of_slot, int32_t* token_of_row, void* stream);

/* moe_dispatch without a workspace (the pages have no counterpart to this
 * entry point; it is a convenience of this library).
 *
 * Same arguments, results and status reporting as moe_dispatch, minus the
 * workspace.  It exists for callers that cannot allocate device memory for a
 * workspace: code that runs under a fixed memory plan made at start-up (no
 * device allocation allowed afterwards), or a thin C caller with no device
 * allocator of its own.  Its scratch is a 1 MiB array built into the library;
 * every GPU that loads the library holds it until the process exits.
 *   - Limit: ceil(T/16) * E <= moe_dispatch_no_alloc_max_scratch() (262144),
 *     e.g. T <= 32768 tokens at E = 128; larger sizes return
 *     MOE_ERR_WORKSPACE without launching anything (use moe_dispatch).
 *   - The first call on a device looks the array's device address up
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  No call allocates or frees memory.
 *   - All calls on a device share the array and each call rewrites every
 *     entry it reads, so nothing carries over between calls; calls that
 *     overlap on the GPU (e.g. on two streams) race and must be serialised.
 */
size_t moe_dispatch_no_alloc_max_scratch(void);
int moe_dispatch_no_alloc(const void* x, const int32_t* topk_idx, const int32_t* offsets, int T,
                          int H, int E, int k, void* x_perm, int32_t* row_of_slot,
                          int32_t* token_of_row, void* stream);

/* ------------------------------------------------------------------------
 * Segment tables (grouped GEMMs).  Rows [seg_offsets[s], seg_offsets[s+1])
 * of the grouped operand belong to expert seg_expert[s], or to expert s when
 * seg_expert is NULL.  With num_seg = E and seg_offsets = offsets this is the
 * layout moe_dispatch produces.  The general form covers the receive side of
 * expert parallelism, where rows arrive as (source rank x local expert)
 * blocks.  Segments may be empty; rows outside every segment are neither
 * read for output nor written.  seg_offsets: int32 [num_seg+1], device.
 * ---------------------------------------------------------------------- */

/* A4  grouped gate/up GEMM with SwiGLU.
 * For each row r of expert e:
 *   g = x_perm[r] . Wg[e]^T,  u = x_perm[r] . Wu[e]^T   (fp32 accumulation)
 *   h[r] = silu(g) * u,  silu(g) = g / (1 + exp(-g))  -> bf16
 * x_perm bf16 [R,H]; Wg, Wu bf16 [E,I,H] ([E,out,in]); h bf16 [R,I];
 * gu_save bf16 [R,2I] or NULL: g in columns [0,I), u in [I,2I) (kept for the
 * backward pass).  ws may be NULL (no workspace needed). */
int moe_grouped_gemm_swiglu(const void* x_perm, const void* Wg, const void* Wu, int num_seg,
                            const int32_t* seg_offsets, const int32_t* seg_expert, int R, int H,
                            int I, int E, void* h, void* gu_save, void* ws, size_t ws_bytes,
                            void* stream);

/* A3 + A4 fused (the first "next" step after the path: the dispatcher the
 * pages call fused, "FSDPTurbo EP/EFSDP and LlamaFactory FSDP2/CP Design"
 * section 3, taken one step further): moe_grouped_gemm_swiglu on the rows
 * x_perm[r] = x[token_of_row[r]] without x_perm in memory -- the GEMM loads
 * its A rows from x by token id.  Results are bit-identical to
 * moe_dispatch + moe_grouped_gemm_swiglu.  x bf16 [T,H]; token_of_row int32
 * [R] from moe_dispatch, which may then be called with x_perm = NULL.  A
 * token id outside [0,T) inside a segment reads token 0 and sets
 * MOE_STATUS_BAD_INDEX.  No workspace. */
int moe_grouped_gemm_swiglu_gather(const void* x, const int32_t* token_of_row, int T,
                                   const void* Wg, const void* Wu, int num_seg,
                                   const int32_t* seg_offsets, const int32_t* seg_expert, int R,
                                   int H, int I, int E, void* h, void* gu_save, void* stream);

/* A5  grouped down GEMM: y_perm[r] = h[r] . Wd[e]^T (fp32 accumulation) -> bf16.
 * h bf16 [R,I]; Wd bf16 [E,H,I]; y_perm bf16 [R,H].  ws may be NULL. */
int moe_grouped_gemm_down(const void* h, const void* Wd, int num_seg, const int32_t* seg_offsets,
                          const int32_t* seg_expert, int R, int H, int I, int E, void* y_perm,
                          void* ws, size_t ws_bytes, void* stream);

/* A5 + A6 fused (the second half of the pages' fused dispatcher,
 * "FSDPTurbo EP/EFSDP and LlamaFactory FSDP2/CP Design" section 3: the
 * grouped matmul and the unpermute as one operator): the down GEMM of A5
 * whose epilogue scales each row r = row_of_slot[t,j] by topk_w[t,j] and
 * adds it into y_acc[t] (fp32), then y = bf16(y_acc).  y_perm is never
 * written.  The fp32 additions into a token's row happen in no fixed order
 * (16-byte reductions in L2), so y may differ from moe_grouped_gemm_down +
 * moe_combine (which add the k rows in slot order) by the rounding of that
 * order: results are not bit-reproducible from run to run.
 * token_of_row int32 [R], row_of_slot int32 [T,k] (moe_dispatch's);
 * topk_w fp32 [T,k]; y_acc fp32 [T,H] (caller's scratch, zeroed by the call);
 * y bf16 [T,H].  A row whose token or slot does not match is skipped; a
 * token none of whose rows lies in a segment gets y = 0.  Forward only:
 * the combine backward needs the unweighted rows.  It saves the R x H
 * y_perm buffer; on GB300 it measured slower than moe_grouped_gemm_down +
 * moe_combine (one 16-byte L2 reduction per 4 outputs). */
int moe_grouped_gemm_down_combine(const void* h, const void* Wd, int num_seg, const int32_t* seg_offsets,
                                  const int32_t* seg_expert, int R, int H, int I, int E,
                                  const int32_t* token_of_row, const int32_t* row_of_slot,
                                  const float* topk_w, int T, int k, float* y_acc, void* y, void* stream);

/* ------------------------------------------------------------------------
 * FP8 (e4m3) forward GEMMs -- the second "next" step after the path.
 *
 * "TorchTitan FSDP2 完全指南", performance table: FP8 matmuls raise training
 * throughput; the page gives no recipe.  Reading taken here: one fp32 scale
 * per stored row (a token row of x, a permuted row of h, an output channel
 * of one expert's weight, i.e. a row of Wg/Wu/Wd seen as [E*out, in]),
 *   s = amax(|row|) / 448   (s = 1 for an all-zero row)
 *   q = e4m3(row / s)       (IEEE fp32 division, round to nearest even,
 *                            saturated to +-448; e4m3 = 1 sign, 4 exponent
 *                            bits with bias 7, 3 mantissa bits, no infinity)
 * and the GEMMs multiply e4m3 codes on the tensor cores with fp32
 * accumulation, the two row scales applied to the accumulator:
 *   g[r,n] = s_a[r] * s_w[e,n] * sum_k dec(a[r,k]) * dec(w[e,n,k]).
 * H and I must be multiples of 128.  Forward only (no g,u save).
 * ---------------------------------------------------------------------- */

/* A3 on e4m3 rows: moe_dispatch that writes the permuted rows as e4m3 codes.
 * Row row(t,j) of xq_perm (uint8 [T*k, H]) holds the codes of x[t] scaled by
 * token t's scale s_t = amax(|x[t]|) / 448, and xs_perm[row(t,j)] = s_t
 * (fp32 [T*k]): exactly moe_quantize_rows_e4m3 of x followed by the
 * permutation, in one pass over x.  row_of_slot and token_of_row as
 * moe_dispatch; same workspace (moe_dispatch_workspace_size).  xq_perm feeds
 * moe_grouped_gemm_swiglu_fp8 with token_of_row = NULL.  x, xq_perm and ws
 * 16-byte aligned, xs_perm 4-byte aligned (else MOE_ERR_ALIGNMENT); shape
 * and status errors as moe_dispatch. */
int moe_dispatch_e4m3(const void* x, const int32_t* topk_idx, const int32_t* offsets, int T, int H,
                      int E, int k, void* xq_perm, float* xs_perm, int32_t* row_of_slot,
                      int32_t* token_of_row, void* ws, size_t ws_bytes, void* stream);

/* moe_dispatch_e4m3 with the chunk prefixes of moe_route_topk_chunks (as
 * moe_dispatch_chunked): the same codes, scales and indices, no workspace. */
int moe_dispatch_e4m3_chunked(const void* x, const int32_t* topk_idx, const int32_t* offsets,
                              const int32_t* chunk_prefix, int T, int H, int E, int k, void* xq_perm,
                              float* xs_perm, int32_t* row_of_slot, int32_t* token_of_row, void* stream);

/* Per-row e4m3 quantisation of a bf16 matrix a [rows, cols] (cols % 8 == 0):
 * q uint8 [rows, cols], scale fp32 [rows].  Bit-exact: codes and scales are
 * a pure function of the input bits.  a 16-byte, q 8-byte and scale 4-byte
 * aligned (else MOE_ERR_ALIGNMENT); rows < 0, cols <= 0, cols % 8 != 0 or a
 * NULL pointer give MOE_ERR_INVALID_ARG; rows == 0 does nothing. */
int moe_quantize_rows_e4m3(const void* a, int rows, int cols, void* q, float* scale, void* stream);

/* A4 on e4m3 operands: h[r] = silu(g) * u -> bf16 [R,I], with g and u the
 * scaled e4m3 GEMMs above.  Wg, Wu: uint8 [E,I,H] codes with fp32 scales
 * Wg_scale, Wu_scale [E*I] (16-byte aligned).
 *   token_of_row == NULL: a is x_perm's codes uint8 [R,H], a_scale fp32 [R].
 *   token_of_row != NULL: a is x's codes uint8 [T,H] and a_scale fp32 [T]
 *     (one scale per token); row r reads token token_of_row[r] (the fused
 *     dispatch of moe_grouped_gemm_swiglu_gather; a token id outside [0,T)
 *     reads token 0 and sets MOE_STATUS_BAD_INDEX).
 * No workspace. */
int moe_grouped_gemm_swiglu_fp8(const void* a, const float* a_scale, const int32_t* token_of_row,
                                int T, const void* Wg, const float* Wg_scale, const void* Wu,
                                const float* Wu_scale, int num_seg, const int32_t* seg_offsets,
                                const int32_t* seg_expert, int R, int H, int I, int E, void* h,
                                void* stream);

/* A5 on e4m3 operands: y_perm[r,n] = s_h[r] * s_w[e,n] * sum_i dec(h[r,i]) * dec(Wd[e,n,i])
 * -> bf16 [R,H].  h: uint8 [R,I] codes with h_scale fp32 [R] (from
 * moe_quantize_rows_e4m3 of the bf16 h); Wd: uint8 [E,H,I] with Wd_scale
 * fp32 [E*H] (16-byte aligned).  No workspace. */
int moe_grouped_gemm_down_fp8(const void* h, const float* h_scale, const void* Wd,
                              const float* Wd_scale, int num_seg, const int32_t* seg_offsets,
                              const int32_t* seg_expert, int R, int H, int I, int E, void* y_perm,
                              void* stream);

/* A6  combine (unpermute): y[t] = sum_{j=0..k-1} topk_w[t,j] * y_perm[row_of_slot[t,j]],
 * accumulated in fp32 in increasing j, rounded once to bf16.
 * y_perm bf16 [R,H]; topk_w fp32 [T,k]; row_of_slot int32 [T,k]; y bf16 [T,H]. */
int moe_combine(const void* y_perm, const float* topk_w, const int32_t* row_of_slot, int T, int H,
                int k, void* y, void* stream);

/* B1  combine backward.
 *   dy_perm[row(t,j)] = topk_w[t,j] * dy[t]                  -> bf16
 *   d_w[t,j]          = sum_h dy[t,h] * y_perm[row(t,j),h]   (fp32)
 * dy bf16 [T,H]; y_perm bf16 [R,H]; outputs dy_perm bf16 [R,H], d_w fp32 [T,k]. */
int moe_combine_bwd(const void* dy, const void* y_perm, const float* topk_w,
                    const int32_t* row_of_slot, int T, int H, int k, void* dy_perm, float* d_w,
                    void* stream);

/* Workspace of B2 and B3: two 128-byte TMA descriptors per segment, which
 * let the weight-gradient GEMM read each segment's rows with the rows past
 * its end filled with zeros.  0 when num_seg <= 0. */
size_t moe_grouped_gemm_bwd_workspace_size(int num_seg);

/* B2  down backward with the SwiGLU backward in its epilogue.
 *   dh = dy_perm[r] . Wd[e]                         (fp32)
 *   with s = sigmoid(g): dg = dh * u * s * (1 + g*(1 - s)),  du = dh * g * s
 *   dgu[r] = [dg | du]                              -> bf16 [R,2I]
 *   dWd[e] = sum over e's rows of dy_perm[r]^T h[r] (fp32 [E,H,I])
 * gu_save is the [g|u] tensor written by moe_grouped_gemm_swiglu.  Experts
 * with no rows get dWd[e] = 0 (or unchanged when accumulate != 0).
 * ws: moe_grouped_gemm_bwd_workspace_size(num_seg) bytes, 128-byte aligned
 * (the weight-gradient GEMM's per-segment TMA descriptors). */
int moe_grouped_gemm_down_bwd(const void* dy_perm, const void* h, const void* gu_save,
                              const void* Wd, int num_seg, const int32_t* seg_offsets,
                              const int32_t* seg_expert, int R, int H, int I, int E, void* dgu,
                              float* dWd, int accumulate, void* ws, size_t ws_bytes, void* stream);

/* B3  gate/up backward.
 *   dx_perm[r] = dg[r] . Wg[e] + du[r] . Wu[e]   (one fp32 sum over 2I terms) -> bf16 [R,H]
 *   dWg[e] = sum over e's rows of dg[r]^T x_perm[r],  dWu[e] likewise with du  (fp32 [E,I,H])
 * dgu bf16 [R,2I] from moe_grouped_gemm_down_bwd.
 * ws: moe_grouped_gemm_bwd_workspace_size(num_seg) bytes, 128-byte aligned. */
int moe_grouped_gemm_swiglu_bwd(const void* dgu, const void* x_perm, const void* Wg,
                                const void* Wu, int num_seg, const int32_t* seg_offsets,
                                const int32_t* seg_expert, int R, int H, int I, int E,
                                void* dx_perm, float* dWg, float* dWu, int accumulate, void* ws,
                                size_t ws_bytes, void* stream);

/* B2 and B3 in two halves each, launched by the calls above back to back.
 * Issued separately, the dX half (which the all-to-all returns to the
 * source ranks, "Qwen3-MoE-30B-A3B模型EP+FSDP2并行方案", section
 * "为什么这么设计") can leave before the weight gradients are computed, and
 * the weight-gradient GEMM can be timed on its own.  Results are
 * bit-identical to the combined calls; arguments, layouts and error rules
 * are theirs.
 *   moe_grouped_gemm_down_bwd_dx:   dgu from dy_perm, gu_save, Wd (no workspace)
 *   moe_grouped_gemm_down_bwd_dw:   dWd from dy_perm, h; ws as for moe_grouped_gemm_down_bwd
 *   moe_grouped_gemm_swiglu_bwd_dx: dx_perm from dgu, Wg, Wu (no workspace)
 *   moe_grouped_gemm_swiglu_bwd_dw: dWg, dWu from dgu, x_perm; ws as for moe_grouped_gemm_swiglu_bwd
 * A dW half and a dX half may run concurrently on two streams; two dW calls
 * that overlap need separate workspaces. */
int moe_grouped_gemm_down_bwd_dx(const void* dy_perm, const void* gu_save, const void* Wd, int num_seg,
                                 const int32_t* seg_offsets, const int32_t* seg_expert, int R, int H,
                                 int I, int E, void* dgu, void* stream);
int moe_grouped_gemm_down_bwd_dw(const void* dy_perm, const void* h, int num_seg,
                                 const int32_t* seg_offsets, const int32_t* seg_expert, int R, int H,
                                 int I, int E, float* dWd, int accumulate, void* ws, size_t ws_bytes,
                                 void* stream);
int moe_grouped_gemm_swiglu_bwd_dx(const void* dgu, const void* Wg, const void* Wu, int num_seg,
                                   const int32_t* seg_offsets, const int32_t* seg_expert, int R, int H,
                                   int I, int E, void* dx_perm, void* stream);
int moe_grouped_gemm_swiglu_bwd_dw(const void* dgu, const void* x_perm, int num_seg,
                                   const int32_t* seg_offsets, const int32_t* seg_expert, int R, int H,
                                   int I, int E, float* dWg, float* dWu, int accumulate, void* ws,
                                   size_t ws_bytes, void* stream);

/* B4  dispatch backward: dx_acc[t] = sum_{j=0..k-1} dx_perm[row_of_slot[t,j]] in fp32,
 * increasing j.  dx_perm bf16 [R,H]; dx_acc fp32 [T,H]. */
int moe_dispatch_bwd(const void* dx_perm, const int32_t* row_of_slot, int T, int H, int k,
                     float* dx_acc, void* stream);

/* B5  router backward.
 *   dl[t,j] = topk_w[t,j] * (d_w[t,j] - sum_i topk_w[t,i] * d_w[t,i])
 *             (gradient of the softmax over the selected logits; the
 *             unselected logits, the indices and the bias get none)
 *   dWr[h,e] = sum_t x[t,h] * dl[t,e]                  (fp32 [H,E])
 *   dx[t,h]  = dx_acc[t,h] + sum_j dl[t,j] * Wr[h,topk_idx[t,j]]  -> bf16 [T,H]
 * The two contractions run on the tensor cores with each fp32 operand split
 * into a bf16 high part and a bf16 low part (products hi*hi + hi*lo + lo*hi,
 * relative error about 2^-16).  dx_acc fp32 [T,H] from moe_dispatch_bwd. */
size_t moe_route_topk_bwd_workspace_size(int T, int H, int E);
int moe_route_topk_bwd(const float* d_w, const float* topk_w, const int32_t* topk_idx,
                       const void* x, const float* Wr, const float* dx_acc, int T, int H, int E,
                       int k, float* dWr, void* dx, int accumulate, void* ws, size_t ws_bytes,
                       void* stream);

/* Persistent-grid limit of the grouped GEMMs (no counterpart on the pages).
 * Every grouped GEMM kernel (the forward, backward and router-backward
 * GEMMs of the calls above) runs one CTA per SM over its tiles.  After
 * this call, those launched from the calling thread use at most max_sms
 * SMs (0 = all, the default), leaving the rest to work issued on another
 * stream: the layer runs the dispatch and router backward beside the
 * gate/up weight gradient this way.  Results do not depend on the limit.
 * *previous (host, may be NULL) receives the limit in force before.
 * MOE_ERR_INVALID_ARG if max_sms < 0. */
int moe_set_gemm_sm_limit(int max_sms, int* previous);

/* Measurement aid (no counterpart on the pages): launches a kernel whose
 * threads only run independent fp32 fused multiply-add chains, per_sm CTAs
 * of 256 threads on every SM, `iters` x 128 FMAs per thread.  Timing it
 * with events on `stream` gives the fp32 FMA rate this GPU sustains, the
 * ceiling of the router's partial-logit kernel (whose summation order keeps
 * it off the tensor cores).  *fmas (host) receives the number of FMAs the
 * launch performs; out (device, >= 1 float) is written only in a case the
 * probe's inputs never reach.  packed != 0: the chains advance in pairs by
 * packed two-lane fp32 FMA instructions (fma.rn.f32x2).  1 <= per_sm <= 32,
 * 1 <= iters <= 2^20. */
int moe_probe_fma(int packed, int per_sm, int iters, float* out, long long* fmas, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_TOPK_H */
