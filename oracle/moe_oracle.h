/*
 * CPU oracle for the MoE expert layer -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this library.  The product (the CUDA library and its Python
 * binding) never calls it and shares no code with it.
 *
 * Every function takes host pointers, runs single-threaded in fp32 (the FP8
 * GEMMs sum their exact e4m3 products in double) and
 * returns 0 on success, -1 on a bad argument, -2 when a host allocation
 * fails.  bf16 tensors are passed as uint16_t bit patterns and widened
 * exactly to fp32.  Activations that the CUDA path stores in bf16 between
 * steps (h, y_perm, dy_perm, dgu, dx_perm) are fp32 here: the oracle never
 * rounds an intermediate.
 *
 * Segment tables: rows [seg_offsets[s], seg_offsets[s+1]) of the grouped
 * operand belong to expert seg_expert[s] (seg_expert == NULL means expert s).
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Width of the h-blocks of the router's fp32 logit sum (see moe_oracle.c). */
#define ORACLE_LOGIT_BLOCK 256

int oracle_route_topk(const uint16_t* x, const float* Wr, const float* bias,
                      int T, int H, int E, int k, int ep_size,
                      int32_t* topk_idx, float* topk_w, int32_t* counts,
                      int32_t* offsets, int32_t* rank_offsets);

int oracle_router_logits(const uint16_t* x, const float* Wr, const float* bias,
                         int T, int H, int E, float* logits);

int oracle_dispatch(const uint16_t* x, const int32_t* topk_idx, const int32_t* offsets,
                    int T, int H, int E, int k,
                    uint16_t* x_perm, int32_t* row_of_slot, int32_t* token_of_row);

int oracle_grouped_gemm_swiglu(const float* x_perm, const uint16_t* Wg, const uint16_t* Wu,
                               int num_seg, const int32_t* seg_offsets, const int32_t* seg_expert,
                               int R, int H, int I, int E, float* h, float* gu);

int oracle_grouped_gemm_down(const float* h, const uint16_t* Wd,
                             int num_seg, const int32_t* seg_offsets, const int32_t* seg_expert,
                             int R, int H, int I, int E, float* y_perm);

int oracle_combine(const float* y_perm, const float* topk_w, const int32_t* row_of_slot,
                   int T, int H, int k, float* y);

int oracle_combine_bwd(const float* dy, const float* y_perm, const float* topk_w,
                       const int32_t* row_of_slot, int T, int H, int k,
                       float* dy_perm, float* d_w);

int oracle_grouped_gemm_down_bwd(const float* dy_perm, const float* h, const float* gu,
                                 const uint16_t* Wd, int num_seg, const int32_t* seg_offsets,
                                 const int32_t* seg_expert, int R, int H, int I, int E,
                                 float* dgu, float* dWd, int accumulate);

int oracle_grouped_gemm_swiglu_bwd(const float* dgu, const float* x_perm,
                                   const uint16_t* Wg, const uint16_t* Wu,
                                   int num_seg, const int32_t* seg_offsets,
                                   const int32_t* seg_expert, int R, int H, int I, int E,
                                   float* dx_perm, float* dWg, float* dWu, int accumulate);

int oracle_dispatch_bwd(const float* dx_perm, const int32_t* row_of_slot, int T, int H, int k,
                        float* dx_acc);

int oracle_route_topk_bwd(const float* d_w, const float* topk_w, const int32_t* topk_idx,
                          const uint16_t* x, const float* Wr, const float* dx_acc,
                          int T, int H, int E, int k, float* dWr, float* dx, int accumulate);

/* e4m3 (R7): codes <-> values, per-row quantisation, FP8 grouped GEMMs. */
int oracle_e4m3_decode(const uint8_t* q, int n, float* out);
int oracle_e4m3_encode(const float* v, int n, uint8_t* q);
int oracle_quantize_rows_e4m3(const float* a, int rows, int cols, uint8_t* q, float* scale);
int oracle_grouped_gemm_swiglu_fp8(const uint8_t* aq, const float* a_scale, const uint8_t* Wgq,
                                   const float* Wg_scale, const uint8_t* Wuq, const float* Wu_scale,
                                   int num_seg, const int32_t* seg_offsets,
                                   const int32_t* seg_expert, int R, int H, int I, int E, float* h);
int oracle_grouped_gemm_down_fp8(const uint8_t* hq, const float* h_scale, const uint8_t* Wdq,
                                 const float* Wd_scale, int num_seg, const int32_t* seg_offsets,
                                 const int32_t* seg_expert, int R, int H, int I, int E,
                                 float* y_perm);

#ifdef __cplusplus
}
#endif
#endif
