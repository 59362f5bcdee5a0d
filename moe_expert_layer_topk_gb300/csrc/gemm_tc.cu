// Grouped GEMMs of the MoE expert layer on the 5th-generation tensor cores
// (sm_103a): tcgen05.mma with fp32 accumulators in tensor memory (TMEM),
// operands staged in shared memory by TMA (cp.async.bulk.tensor, 128-byte
// swizzle), mbarrier producer/consumer pipeline, warp-specialised persistent
// CTAs.
//
// "FSDPTurbo EP/EFSDP and LlamaFactory FSDP2/CP Design", section 3: the
// expert compute between permute and unpermute is a grouped matmul over the
// experts' row groups, and must cope with experts that receive no rows.
// Shapes: "Qwen3-MoE-30B-A3B模型EP+FSDP2并行方案", model section (gate/up
// [E,I,H], down [E,H,I]).  fp32 weight gradients: "TorchTitan FSDP2 完全指南",
// mixed-precision section.
//
// One kernel template serves ten GEMM shapes (`Kind`):
//   GATE_UP_FWD    h = silu(A Wg^T) * (A Wu^T)  (+ save g, u)     A, B K-major
//   GATE_UP_GATHER the same with A row r = x[token_of_row[r]]
//   GATE_UP_FP8, GATE_UP_GATHER_FP8, DOWN_FP8: the forward kinds on e4m3
//                  operands (tcgen05 kind::f8f6f4, fp32 accumulation) with
//                  one fp32 scale per A row and per B row (output channel),
//                  applied to the accumulator in the epilogue
//   DOWN_FWD       y = A Wd^T                                     A, B K-major
//   DOWN_COMBINE   the same, each row scaled by its routing weight and
//                  added into its token's fp32 output row (fused combine)
//   DOWN_BWD_DX    dh = A Wd; SwiGLU backward in the epilogue     B MN-major
//   GATE_UP_BWD_DX dx = dg Wg + du Wu (K = 2I, two B tensors)      B MN-major
//   DW             dW[g] = sum over group g's rows of A^T B (fp32) A, B MN-major
//   DENSE_ADD      out = bf16(A B^T + add)  (router backward)     A, B K-major
//
// CTA layout (one CTA per SM, persistent over tiles):
//   warp 0      TMA producer (one lane issues)
//   warp 1      TMEM allocator + MMA issuer (one lane issues)
//   warps 2..   epilogue: TMEM -> registers -> global (warp w reads TMEM
//               lanes 32*(w%4)..+31, i.e. accumulator rows); four warps, or
//               eight (two per lane quadrant, sharing the columns) for the
//               weight-gradient, SwiGLU-backward and down-projection kinds
//   last 4      row-gathering kinds only: they and warp 0 copy the A rows
//               from x by token id with cp.async
// Tile: 128 rows x BN columns (BN <= 256), k-block of one 128-byte swizzle
// row (64 bf16 or 128 e4m3 elements), 4-stage shared-memory ring (3 for the
// router dX kind, whose epilogue stages its addend), two 256-column
// accumulators in TMEM so the epilogue of tile i overlaps the MMAs of tile
// i+1.  GATE_UP_BWD_DX, and GATE_UP_FWD and DOWN_FWD in the dispatch layout
// (one segment per expert), run as cluster pairs (tcgen05 cta_group::2,
// 256-row tiles).  The weight-gradient kind's TMA stores carry an
// evict-last L2 policy.
//
// Every wait on an mbarrier is bounded (globaltimer): on timeout the CTA
// records MOE_STATUS_TIMEOUT, all roles leave their loops, outstanding MMAs
// are drained with a bounded wait and TMEM is freed before returning.
#include <cuda.h>

#include <initializer_list>

#include "tc_common.cuh"

namespace moe {
namespace tc {

constexpr int A_BYTES = BM * BK * 2;          // 16 KiB
constexpr int B_BYTES_MAX = 256 * BK * 2;     // 32 KiB
// DOWN_BWD_DX also loads the saved g, u boxes by TMA: 4 sets of (g, u) slots.
constexpr int EP_GU_SETS = 4;

enum Kind : int {
  GATE_UP_FWD = 0,
  DOWN_FWD = 1,
  DOWN_BWD_DX = 2,
  GATE_UP_BWD_DX = 3,
  DW = 4,
  DENSE_ADD = 5,
  GATE_UP_GATHER = 6,
  GATE_UP_FP8 = 7,
  GATE_UP_GATHER_FP8 = 8,
  DOWN_FP8 = 9,
  DOWN_COMBINE = 10
};
constexpr int kNumKinds = 11;
__host__ __device__ constexpr bool is_fp8(int k) {
  return k == GATE_UP_FP8 || k == GATE_UP_GATHER_FP8 || k == DOWN_FP8;
}
// the gate/up forward kinds (same tiles and epilogue; they differ in how A
// arrives and in the operand type)
__host__ __device__ constexpr bool is_gate_up(int k) {
  return k == GATE_UP_FWD || k == GATE_UP_GATHER || k == GATE_UP_FP8 || k == GATE_UP_GATHER_FP8;
}
__host__ __device__ constexpr bool is_gather(int k) { return k == GATE_UP_GATHER || k == GATE_UP_GATHER_FP8; }
// the down-projection kinds (same tiles and operands)
__host__ __device__ constexpr bool is_down_fwd(int k) { return k == DOWN_FWD || k == DOWN_FP8 || k == DOWN_COMBINE; }
// reduction elements per k-block: one 128-byte row of the operand type
__host__ __device__ constexpr int kblock_elems(int k) { return is_fp8(k) ? 128 : BK; }

struct Params {
  int M;             // row kinds: rows of A (R).  DW: output rows per group.
  int N;             // output columns
  int K;             // row kinds: reduction length.  DW: rows of the K-indexed operands.
  int BN;            // MMA N
  int NH;            // gate/up forward: width of each of the g and u halves
  int n_tiles;
  int m_tiles;       // DW: m-tiles per group
  int num_seg;
  const int32_t* seg_offsets;
  const int32_t* seg_expert;
  int num_groups;    // experts (B row groups) / DW output groups
  int b_group_rows;  // rows of the 2-D view of B per expert
  int split_m;       // DW: rows m < split_m -> out0, else out1 (0: all out0)
  int ldo;           // leading dimension of out0/out1 (elements)
  int I;             // intermediate size (gu / dgu layouts)
  uint32_t idesc;
  int accumulate;
  void* out0;
  void* out1;
  const void* aux;
  union {
    const CUtensorMap* seg_maps;  // DW: per segment s, the A map (2s) and the B map (2s+1)
    struct {
      const int32_t* gather_rows;  // row-gathering kinds: A row r is x[gather_rows[r]] (token_of_row)
      const float* a_scale;        // FP8 kinds: per A row (gathering: per token of x)
      const float* b_scale0;       // FP8 kinds: per row of B0 ([E * N] output channels)
      const float* b_scale1;       // GATE_UP FP8 kinds: per row of B1
      int gather_limit;            // row-gathering kinds: tokens in x
    };
  };
  int* status;
  // DOWN_COMBINE: the rows' tokens and routing weights, the fp32 output
  const int32_t* comb_token;   // token_of_row [M]
  const int32_t* comb_rows;    // row_of_slot [comb_T, comb_k]
  const float* comb_w;         // topk_w [comb_T, comb_k]
  float* comb_out;             // [comb_T, ldo]
  int comb_T;
  int comb_k;
};

struct Ctl {
  unsigned long long full[6];
  unsigned long long empty[6];
  unsigned long long tfull[2];
  unsigned long long tempty[2];
  unsigned long long drain;
  uint32_t tmem_base;
  int abort_flag;
  int total_tiles;
  // Segment tables, in the shared memory right after this struct, sized by
  // the launch: num_seg + 1, num_seg + 1, num_seg and (DW) num_groups ints.
  int* seg_off;
  int* seg_tiles;                   // prefix sum of tiles per segment (row kinds)
  int* seg_exp;
  int* grp_rows;                    // DW: rows per output group
  unsigned long long ep_bar[4][EP_GU_SETS];  // g,u / addend box loads per epilogue warp
};

// Bytes of the segment tables that follow Ctl.
__host__ __device__ constexpr size_t seg_table_bytes(int num_seg, int num_groups, bool dw) {
  return ((size_t)(3 * num_seg + 2 + (dw ? num_groups : 0)) * 4 + 15) / 16 * 16;
}
constexpr size_t kMaxTableBytes = seg_table_bytes(kMaxSegments, kMaxExperts, true);



// ----------------------------------------------------------------- the kernel

template <int KIND>
struct Traits {
  static constexpr bool a_mn = (KIND == DW);
  static constexpr bool b_mn = (KIND == DOWN_BWD_DX || KIND == GATE_UP_BWD_DX || KIND == DW);
  static constexpr bool rows = (KIND != DW);
};

// CTAS = 1: one CTA per 128-row tile, whole B tile in its shared memory.
// CTAS = 2: a cluster pair per 256-row tile (tcgen05 cta_group::2): each CTA
// holds its own 128 rows of A and half of the B tile's N range; the leader
// (cluster rank 0) issues the MMAs, which read both CTAs' shared memory and
// write each CTA's 128 accumulator rows into that CTA's TMEM.
//
// The router dX kind reads its fp32 addend by TMA into GU_SETS staging
// sets, GU_SETS/2 chunks ahead, and runs one pipeline stage fewer.
template <int KIND, int CTAS>
struct Cfg {
  static constexpr bool gu_tma = KIND == DENSE_ADD;
  static constexpr int GU_SETS = EP_GU_SETS;
  static constexpr int STAGES = CTAS == 1 ? (gu_tma ? 3 : 4) : (gu_tma ? 4 : 6);
  static constexpr int B_BYTES = B_BYTES_MAX / CTAS;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TILE_M = BM * CTAS;
  // The weight-gradient kind (fp32 output, short reductions), the
  // SwiGLU-backward kind (heavy epilogue) and the down projections (256
  // output columns per tile from a short reduction, K = I) run eight
  // epilogue warps, two per TMEM lane quadrant sharing the columns (a
  // one-box store ring each).
  static constexpr bool EP8 = KIND == DW || KIND == DOWN_BWD_DX || is_down_fwd(KIND);
  static constexpr int EPW = EP8 ? 8 : 4;
  // row-gathering kinds: four more warps share the row gather
  static constexpr int GW = is_gather(KIND) ? 4 : 0;
  static constexpr int NTHREADS = 64 + 32 * (EPW + GW);
  static constexpr int RING = EP8 ? 1 : EP_SLOTS;
  static constexpr int EP_WARP = gu_tma ? EP_BOX_BYTES * 2 * GU_SETS : EP_BOX_BYTES * RING;
  static constexpr int EP_TOTAL = EPW * EP_WARP;
  // without the segment tables
  static constexpr size_t SMEM_FIXED = 1024 + (size_t)STAGES * STAGE_BYTES + EP_TOTAL + sizeof(Ctl);
};
// the configurations launched (cluster pairs for GATE_UP_FWD, GATE_UP_BWD_DX, DOWN_FWD and DOWN_COMBINE)
static_assert(Cfg<GATE_UP_FWD, 1>::SMEM_FIXED + kMaxTableBytes <= kSmemMax &&
                  Cfg<GATE_UP_GATHER, 1>::SMEM_FIXED + kMaxTableBytes <= kSmemMax &&
                  Cfg<GATE_UP_FP8, 1>::SMEM_FIXED + kMaxTableBytes <= kSmemMax &&
                  Cfg<GATE_UP_GATHER_FP8, 1>::SMEM_FIXED + kMaxTableBytes <= kSmemMax &&
                  Cfg<DOWN_FP8, 1>::SMEM_FIXED + kMaxTableBytes <= kSmemMax &&
                  Cfg<DOWN_FWD, 1>::SMEM_FIXED + kMaxTableBytes <= kSmemMax &&
                  Cfg<DOWN_BWD_DX, 1>::SMEM_FIXED + kMaxTableBytes <= kSmemMax &&
                  Cfg<GATE_UP_BWD_DX, 1>::SMEM_FIXED + kMaxTableBytes <= kSmemMax &&
                  Cfg<GATE_UP_BWD_DX, 2>::SMEM_FIXED + kMaxTableBytes <= kSmemMax &&
                  Cfg<GATE_UP_FWD, 2>::SMEM_FIXED + kMaxTableBytes <= kSmemMax &&
                  Cfg<DOWN_FWD, 2>::SMEM_FIXED + kMaxTableBytes <= kSmemMax &&
                  Cfg<DOWN_COMBINE, 1>::SMEM_FIXED + kMaxTableBytes <= kSmemMax &&
                  Cfg<DOWN_COMBINE, 2>::SMEM_FIXED + kMaxTableBytes <= kSmemMax &&
                  Cfg<DENSE_ADD, 1>::SMEM_FIXED + kMaxTableBytes <= kSmemMax &&
                  Cfg<DW, 1>::SMEM_FIXED + kMaxTableBytes <= kSmemMax,
              "shared memory budget exceeded");

struct Tile {
  int group;   // expert (row kinds) / output group (DW)
  int m0;      // this CTA's first row (row kinds: of A; DW: of the output)
  int n0;      // first output column of the tile
  int row_end; // row kinds: end of the segment (exclusive)
  int seg;     // row kinds: segment index
};

template <int KIND, int CTAS>
__device__ __forceinline__ Tile decode_tile(int tile, const Params& p, const Ctl* ctl, int rank) {
  Tile t;
  if constexpr (Traits<KIND>::rows) {
    const int gm = tile / p.n_tiles, nt = tile % p.n_tiles;
    int lo = 0, hi = p.num_seg - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ctl->seg_tiles[mid] <= gm) lo = mid; else hi = mid - 1;
    }
    t.seg = lo;
    t.group = ctl->seg_exp[lo];
    t.m0 = ctl->seg_off[lo] + (gm - ctl->seg_tiles[lo]) * Cfg<KIND, CTAS>::TILE_M + BM * rank;
    t.row_end = ctl->seg_off[lo + 1];
    t.n0 = nt * (is_gate_up(KIND) ? p.NH : p.BN);
  } else {
    const int per = p.m_tiles * p.n_tiles;
    t.group = tile / per;
    const int rem = tile % per;
    t.m0 = (rem / p.n_tiles) * Cfg<KIND, CTAS>::TILE_M + BM * rank;
    t.n0 = (rem % p.n_tiles) * p.BN;
    t.row_end = 0;
    t.seg = 0;
  }
  return t;
}

// Calls f(k0, valid_rows, seg) for every k-block of a tile, in order.  Row
// kinds: k0 is the reduction offset.  DW: k0 is the first row of the k-block
// counted from the start of segment `seg` (the segment's own tensor maps
// address rows from there).
template <int KIND, class F>
__device__ __forceinline__ void for_each_kblock(const Tile& t, const Params& p, const Ctl* ctl, F&& f) {
  if constexpr (Traits<KIND>::rows) {
    constexpr int KB = kblock_elems(KIND);
    const int nkb = p.K / KB;
    for (int kb = 0; kb < nkb; ++kb)
      if (!f(kb * KB, KB, t.seg)) return;
  } else if (p.seg_expert == nullptr) {
    // identity table: group g owns exactly segment g (none for g >= num_seg)
    if (t.group < p.num_seg && ctl->seg_exp[t.group] >= 0) {
      const int len = ctl->seg_off[t.group + 1] - ctl->seg_off[t.group];
      for (int r = 0; r < len; r += BK)
        if (!f(r, min(BK, len - r), t.group)) return;
    }
  } else {
    for (int s = 0; s < p.num_seg; ++s) {
      if (ctl->seg_exp[s] != t.group) continue;
      const int len = ctl->seg_off[s + 1] - ctl->seg_off[s];
      for (int r = 0; r < len; r += BK)
        if (!f(r, min(BK, len - r), s)) return;
    }
  }
}

template <int KIND, int CTAS>
__global__ void __launch_bounds__(Cfg<KIND, CTAS>::NTHREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmB1,
                        const __grid_constant__ CUtensorMap tmO0,
                        const __grid_constant__ CUtensorMap tmO1, const Params p) {
  pdl_wait();
  pdl_trigger();
  using C = Cfg<KIND, CTAS>;
  constexpr int STG = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + (size_t)STG * C::STAGE_BYTES + C::EP_TOTAL);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int limit = Traits<KIND>::rows ? p.M : p.K;  // rows addressable through the segment table
  const int rank = CTAS == 2 ? (int)cluster_rank() : 0;
  const bool leader = rank == 0;
  const int unit = CTAS == 2 ? (int)blockIdx.x / 2 : (int)blockIdx.x;  // tile-processing unit
  const int nunits = CTAS == 2 ? (int)gridDim.x / 2 : (int)gridDim.x;

  // ---- segment table -> shared memory (clamped; bad entries become empty)
  {
    int* tab = reinterpret_cast<int*>(ctl + 1);
    if (threadIdx.x == 0) {
      ctl->seg_off = tab;
      ctl->seg_tiles = tab + p.num_seg + 1;
      ctl->seg_exp = tab + 2 * (p.num_seg + 1);
      ctl->grp_rows = tab + 3 * p.num_seg + 2;
    }
    __syncthreads();
  }
  for (int s = threadIdx.x; s <= p.num_seg; s += C::NTHREADS) {
    // a null table means one segment covering every row
    int o = p.seg_offsets ? p.seg_offsets[s] : (s == 0 ? 0 : limit);
    if (o < 0 || o > limit) {
      set_status(p.status, MOE_STATUS_BAD_SEGMENTS);
      o = o < 0 ? 0 : limit;
    }
    ctl->seg_off[s] = o;
  }
  __syncthreads();
  for (int s = threadIdx.x; s < p.num_seg; s += C::NTHREADS) {
    int e = p.seg_expert ? p.seg_expert[s] : s;
    if (e < 0 || e >= p.num_groups) {
      set_status(p.status, MOE_STATUS_BAD_SEGMENTS);
      e = -1;
    }
    if (ctl->seg_off[s + 1] < ctl->seg_off[s]) {
      set_status(p.status, MOE_STATUS_BAD_SEGMENTS);
      ctl->seg_off[s + 1] = ctl->seg_off[s];  // racy only for already-invalid tables
    }
    ctl->seg_exp[s] = e;
  }
  if (!Traits<KIND>::rows)
    for (int g = threadIdx.x; g < p.num_groups; g += C::NTHREADS) ctl->grp_rows[g] = 0;
  __syncthreads();
  if (!Traits<KIND>::rows)
    for (int s = threadIdx.x; s < p.num_seg; s += C::NTHREADS)
      if (ctl->seg_exp[s] >= 0) atomicAdd(&ctl->grp_rows[ctl->seg_exp[s]], ctl->seg_off[s + 1] - ctl->seg_off[s]);
  if (warp == 0) {
    if constexpr (Traits<KIND>::rows) {
      int carry = 0;
      for (int base = 0; base < p.num_seg; base += 32) {
        const int s = base + lane;
        int n = 0;
        if (s < p.num_seg && ctl->seg_exp[s] >= 0) {
          const int len = ctl->seg_off[s + 1] - ctl->seg_off[s];
          n = len > 0 ? (len + C::TILE_M - 1) / C::TILE_M : 0;
        }
        int incl = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int o = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += o;
        }
        if (s < p.num_seg) ctl->seg_tiles[s] = carry + incl - n;
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) {
        ctl->seg_tiles[p.num_seg] = carry;
        ctl->total_tiles = carry * p.n_tiles;
      }
    } else {
      if (lane == 0) ctl->total_tiles = p.num_groups * p.m_tiles * p.n_tiles;
    }
    if (lane == 0) {
      for (int i = 0; i < STG; ++i) {
        // gather mode: lane 0's arming arrival plus one cp.async arrival per gathering lane
        mbar_init(smem_u32(&ctl->full[i]), is_gather(KIND) ? 1 + 32 * (1 + C::GW) : 1);
        mbar_init(smem_u32(&ctl->empty[i]), 1);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(smem_u32(&ctl->tfull[i]), 1);
        mbar_init(smem_u32(&ctl->tempty[i]), C::EPW * CTAS);
      }
      mbar_init(smem_u32(&ctl->drain), 1);
      for (int w = 0; w < 4; ++w)
        for (int i = 0; i < EP_GU_SETS; ++i) mbar_init(smem_u32(&ctl->ep_bar[w][i]), 1);
      ctl->abort_flag = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB0);
      prefetch_tmap(&tmB1);
      prefetch_tmap(&tmO0);
      prefetch_tmap(&tmO1);
    }
  } else if (warp == 1) {
    tmem_alloc_n<CTAS>(smem_u32(&ctl->tmem_base), TMEM_COLS);
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CTAS == 2) cluster_sync();  // peer barriers initialised before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  const int total = ctl->total_tiles;
  const uint32_t b_bytes = (uint32_t)p.BN * BK * 2 / CTAS;  // this CTA's share of a B stage

  // Row-gathering kinds: warp 0 and the GW helper warps copy the
  // A tile's rows from x by token id with cp.async (per instruction a warp
  // copies four whole 128-byte rows, 8 lanes per row, into the
  // 128-byte-swizzled tile) and each lane arrives on the stage's barrier when
  // its copies land; warp 0's lane 0 also arms the barrier for the gate and
  // up tiles, which come by TMA.
  auto gather_loop = [&](int gw) {
    constexpr int NG = 32 * (1 + C::GW);            // gathering lanes
    constexpr int PIECES = BM * 8;                   // 16-byte pieces of an A tile
    constexpr int NI = (PIECES + NG - 1) / NG;
    constexpr int KB = kblock_elems(KIND);
    const uint8_t* xg = static_cast<const uint8_t*>(p.aux);
    const size_t row_bytes = (size_t)p.K * (is_fp8(KIND) ? 1 : 2);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    const int nkb = p.K / KB;
    const int c = lane & 7;  // 16-byte chunk of a row
    for (int tile = unit; ok && tile < total; tile += nunits) {
      const Tile t = decode_tile<KIND, CTAS>(tile, p, ctl, rank);
      int tok[NI];
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const int piece = i * NG + gw * 32 + lane;
        const int r = t.m0 + piece / 8;
        int v = (piece < PIECES && r < p.M) ? p.gather_rows[r] : 0;
        if (v < 0 || v >= p.gather_limit) {
          if (r < t.row_end && c == 0) set_status(p.status, MOE_STATUS_BAD_INDEX);
          v = 0;
        }
        tok[i] = v;
      }
      for (int kb = 0; kb < nkb; ++kb) {
        if (!__all_sync(0xffffffffu, wait_bar(smem_u32(&ctl->empty[stage]), phase ^ 1u, &ctl->abort_flag,
                                              p.status))) {
          ok = false;
          break;
        }
        const uint32_t fb = smem_u32(&ctl->full[stage]);
        const uint32_t sA = smem_u32(smem + (size_t)stage * C::STAGE_BYTES);
        const int k0 = kb * KB;
        if (gw == 0 && lane == 0) {
          const uint32_t sB = sA + A_BYTES;
          mbar_arrive_expect_tx(fb, b_bytes);
          const int brow = t.group * p.b_group_rows + t.n0;
          tma_load_2d(sB, &tmB0, fb, k0, brow);
          tma_load_2d(sB + (uint32_t)p.NH * BK * 2, &tmB1, fb, k0, brow);
        }
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          const int piece = i * NG + gw * 32 + lane;
          if (piece < PIECES) {
            const int row = piece / 8;
            const uint8_t* src = xg + (size_t)tok[i] * row_bytes + (size_t)kb * 128 + 16 * c;
            const uint32_t dst = sA + (uint32_t)row * 128 + (uint32_t)((c ^ (row & 7)) << 4);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
          }
        }
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(fb) : "memory");
        if (++stage == STG) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  };

  if (warp == 0) {
    // ============================ TMA producer ============================
    if constexpr (is_gather(KIND)) {
      gather_loop(0);
    } else if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      // DW: segments whose maps this thread has acquired: the one in use,
      // this tile's (acquired a tile ahead) and the next tile's
      int map_seg = -1, this_seg = -1, next_seg = -1;
      for (int tile = unit; ok && tile < total; tile += nunits) {
        const Tile t = decode_tile<KIND, CTAS>(tile, p, ctl, rank);
        if constexpr (KIND == DW) {
          // with one segment per group, the next tile's maps are acquired
          // and prefetched now, so their fetch overlaps this tile's loads
          this_seg = next_seg;
          next_seg = -1;
          if (p.seg_expert == nullptr && tile + nunits < total) {
            const int g = decode_tile<KIND, CTAS>(tile + nunits, p, ctl, rank).group;
            if (g < p.num_seg && ctl->seg_exp[g] >= 0 && g != this_seg && g != map_seg) {
              const CUtensorMap* mn = p.seg_maps + 2 * g;
              tmap_acquire(mn);
              tmap_acquire(mn + 1);
              prefetch_tmap(mn);
              prefetch_tmap(mn + 1);
              next_seg = g;
            }
          }
        }
        for_each_kblock<KIND>(t, p, ctl, [&](int row0, int, int seg) -> bool {
          if (!wait_bar(smem_u32(&ctl->empty[stage]), phase ^ 1u, &ctl->abort_flag, p.status)) {
            ok = false;
            return false;
          }
          const uint32_t fb_local = smem_u32(&ctl->full[stage]);
          const uint32_t fb = CTAS == 2 ? map_to_rank(fb_local, 0) : fb_local;
          const uint32_t sA = smem_u32(smem + (size_t)stage * C::STAGE_BYTES);
          const uint32_t sB = sA + A_BYTES;
          if (leader) mbar_arrive_expect_tx(fb_local, CTAS * (A_BYTES + b_bytes));
          const int ck0 = rank * (p.BN / 64 / CTAS);  // first MN-major B chunk of this CTA
          if constexpr (KIND == DW) {
            // the segment's own maps end at its last row: TMA fills the
            // rows of a tail k-block past it with zeros
            const CUtensorMap* ma = p.seg_maps + 2 * seg;
            if (seg != map_seg && seg != this_seg && seg != next_seg) {
              tmap_acquire(ma);
              tmap_acquire(ma + 1);
            }
            map_seg = seg;
            tma_load_mn<CTAS>(sA, ma, fb, row0, t.m0 / 64);
            tma_load_mn<CTAS>(sB, ma + 1, fb, row0, t.n0 / 64 + ck0);
          } else {
            tma_load<CTAS>(sA, &tmA, fb, row0, t.m0);
            if constexpr (is_gate_up(KIND)) {
              const int brow = t.group * p.b_group_rows + t.n0;
              if (CTAS == 1) {
                tma_load<CTAS>(sB, &tmB0, fb, row0, brow);
                tma_load<CTAS>(sB + (uint32_t)p.NH * BK * 2, &tmB1, fb, row0, brow);
              } else {
                // pair: the leader holds the gate rows, the peer the up rows
                tma_load<CTAS>(sB, rank == 0 ? &tmB0 : &tmB1, fb, row0, brow);
              }
            } else if constexpr (is_down_fwd(KIND) || KIND == DENSE_ADD) {
              tma_load<CTAS>(sB, &tmB0, fb, row0,
                             t.group * p.b_group_rows + t.n0 + rank * (p.BN / CTAS));
            } else if constexpr (KIND == DOWN_BWD_DX) {
              tma_load_mn<CTAS>(sB, &tmB0, fb, t.group * p.b_group_rows + row0, t.n0 / 64 + ck0);
            } else {  // GATE_UP_BWD_DX: k < I from Wg, k >= I from Wu
              const bool up = row0 >= p.I;
              const int krow = t.group * p.b_group_rows + (up ? row0 - p.I : row0);
              tma_load_mn<CTAS>(sB, up ? &tmB1 : &tmB0, fb, krow, t.n0 / 64 + ck0);
            }
          }
          if (++stage == STG) {
            stage = 0;
            phase ^= 1u;
          }
          return true;
        });
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer ==============================
    // (CTAS = 2: only the leader issues; the peer's warp 1 just owns its TMEM)
    if (CTAS == 1 || leader) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int tile = unit; ok && tile < total; tile += nunits, ++local) {
        const Tile t = decode_tile<KIND, CTAS>(tile, p, ctl, rank);
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!__all_sync(0xffffffffu, wait_bar(smem_u32(&ctl->tempty[buf]), (use & 1u) ^ 1u, &ctl->abort_flag, p.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(buf * ACC_COLS);
        int nk = 0;
        for_each_kblock<KIND>(t, p, ctl, [&](int, int valid, int) -> bool {
          if (!__all_sync(0xffffffffu, wait_bar(smem_u32(&ctl->full[stage]), phase, &ctl->abort_flag, p.status))) {
            ok = false;
            return false;
          }
          uint8_t* sA = smem + (size_t)stage * C::STAGE_BYTES;
          uint8_t* sB = sA + A_BYTES;
          // DW tail k-block: the rows past the segment end arrived as zeros;
          // only the 16-deep MMA steps that hold valid rows are issued.
          const int nkk = KIND == DW ? (valid + 15) / 16 : BK / 16;
          tc_fence_after();
          if (is_gather(KIND))  // A was written by cp.async (generic proxy)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          if (lane == 0) {
            const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              if (kk >= nkk) break;
              const uint64_t ad = Traits<KIND>::a_mn ? sdesc(a0 + kk * 2048, CHUNK_BYTES, 1024)
                                                     : sdesc(a0 + kk * 32, 16, 1024);
              const uint64_t bd = Traits<KIND>::b_mn ? sdesc(b0 + kk * 2048, CHUNK_BYTES, 1024)
                                                     : sdesc(b0 + kk * 32, 16, 1024);
              mma_issue<CTAS, is_fp8(KIND)>(d, ad, bd, p.idesc, (nk > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit_to<CTAS>(smem_u32(&ctl->empty[stage]));
          }
          __syncwarp();
          ++nk;
          if (++stage == STG) {
            stage = 0;
            phase ^= 1u;
          }
          return true;
        });
        if (!ok) break;
        if (lane == 0) mma_commit_to<CTAS>(smem_u32(&ctl->tfull[buf]));
        __syncwarp();
      }
      if (!ok) {
        // drain MMAs still in flight before TMEM is released
        if (lane == 0) mma_commit_to<CTAS>(smem_u32(&ctl->drain));
        __syncwarp();
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&ctl->drain), 0) && globaltimer() - t0 < TIMEOUT_NS) {
        }
      }
    }
  } else if (C::GW > 0 && warp >= 2 + C::EPW) {
    // ======================= row-gather helper warps ========================
    if constexpr (is_gather(KIND)) gather_loop(warp - (1 + C::EPW));
  } else {
    // ============================ epilogue ================================
    // Each warp owns 32 accumulator rows of the tile (TMEM lanes
    // 32*(warp%4)..+31).  Results leave in boxes of 32 rows x 64 bytes:
    // every lane writes its own row of the box into shared memory (64-byte
    // swizzle, conflict-free); then either a TMA bulk store writes the box
    // (the kinds named at kTmaOut, when all 32 rows are valid), or the warp
    // reads the box back row-segment by row-segment and writes it with
    // coalesced 16-byte stores (8 full 64-byte row segments per
    // instruction), skipping rows past the end of the expert's rows.
    const int q = warp & 3;
    uint8_t* ep_base = smem + (size_t)STG * C::STAGE_BYTES + (size_t)(warp - 2) * C::EP_WARP;
    const int sw = (lane >> 1) & 3;  // 64-byte swizzle phase of this lane's row
    auto put = [&](uint8_t* box, int c, uint4 v) {
      *reinterpret_cast<uint4*>(box + lane * 64 + ((c ^ sw) << 4)) = v;
    };
    auto get = [&](const uint8_t* box, int c) -> uint4 {
      return *reinterpret_cast<const uint4*>(box + lane * 64 + ((c ^ sw) << 4));
    };
    // box -> rows [row0, row0 + nvalid) of a row-major tensor at byte column col
    auto flush = [&](const uint8_t* box, void* base, size_t pitch, size_t col, int row0, int nvalid,
                     bool acc_f32) {
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int rr = (lane >> 2) + 8 * j, cc = lane & 3;
        uint4 v = *reinterpret_cast<const uint4*>(box + rr * 64 + ((cc ^ ((rr >> 1) & 3)) << 4));
        if (rr < nvalid) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(base) + (size_t)(row0 + rr) * pitch +
                                                col + cc * 16);
          if (acc_f32) {
            const float4 o = *reinterpret_cast<const float4*>(dst);
            v = make_uint4(__float_as_uint(__uint_as_float(v.x) + o.x), __float_as_uint(__uint_as_float(v.y) + o.y),
                           __float_as_uint(__uint_as_float(v.z) + o.z), __float_as_uint(__uint_as_float(v.w) + o.w));
          }
          *dst = v;
        }
      }
      __syncwarp();
    };
    // Full boxes of the fp32 weight gradients, of the down projection and of
    // the SwiGLU backward's dg, du go out through TMA bulk stores instead
    // (measured faster for those three; for h, g, u of the gate/up forward
    // they measured no different).
    constexpr bool kTmaOut = KIND == DW || is_down_fwd(KIND);
    EpRing<C::RING> ring{ep_base, 0, lane};
    int gu_ctr = 0;  // DENSE_ADD: running count of this warp's 32-column chunks
    const uint32_t tempty_leader[2] = {
        CTAS == 2 ? map_to_rank(smem_u32(&ctl->tempty[0]), 0) : smem_u32(&ctl->tempty[0]),
        CTAS == 2 ? map_to_rank(smem_u32(&ctl->tempty[1]), 0) : smem_u32(&ctl->tempty[1])};
    int local = 0;
    for (int tile = unit; tile < total; tile += nunits, ++local) {
      const Tile t = decode_tile<KIND, CTAS>(tile, p, ctl, rank);
      const int buf = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      const int rb = t.m0 + q * 32;
      const int lim = Traits<KIND>::rows ? t.row_end : p.M;
      const int nvalid = lim - rb < 0 ? 0 : (lim - rb > 32 ? 32 : lim - rb);
      const bool any = nvalid > 0;
      // Router dX: the fp32 addend, which does not depend on the
      // accumulator (two boxes of 32 rows x 16 columns per 32-column
      // chunk), arrives by TMA into set (chunk counter mod GU_SETS) of the
      // warp's staging, GU_SETS/2 chunks ahead; the first ones are requested
      // before waiting for the MMAs.
      const uint32_t gu_bar0 = C::gu_tma ? smem_u32(&ctl->ep_bar[warp - 2][0]) : 0u;
      auto gu_load = [&](int c, int ctr) {
        if (C::gu_tma && any && c < p.BN && lane == 0) {
          const int set = ctr & (C::GU_SETS - 1);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // earlier reads of the set
          const uint32_t bar = gu_bar0 + 8u * (uint32_t)set;
          const uint32_t g_slot = smem_u32(ep_base + (2 * set) * EP_BOX_BYTES);
          mbar_arrive_expect_tx(bar, 2 * EP_BOX_BYTES);
          tma_load_2d(g_slot, &tmB1, bar, t.n0 + c, rb);
          tma_load_2d(g_slot + EP_BOX_BYTES, &tmB1, bar, 16 + t.n0 + c, rb);
        }
      };
      constexpr int GU_AHEAD = C::GU_SETS / 2;  // chunks requested ahead
      if constexpr (C::gu_tma) {
#pragma unroll
        for (int a = 0; a < GU_AHEAD; ++a) gu_load(32 * a, gu_ctr + a);
      }
      // With eight epilogue warps the two warps of a TMEM lane quadrant
      // share the tile's 32-column chunks.  The SwiGLU-backward kind
      // alternates them (warps 2..5 the even chunks, 6..9 the odd ones), so
      // that both halves of each 128-byte row segment of g, u (read) and of
      // dg, du (written) are touched at about the same time; the other kinds
      // split the columns in halves (warps 2..5 the first, 6..9 the second).
      constexpr bool kAlt = KIND == DOWN_BWD_DX;
      const int sub = (warp - 2) >> 2, nsub = C::EPW / 4;
      const int cbeg = kAlt ? 32 * sub : sub * (p.BN / nsub);
      const int cstep = kAlt ? 32 * nsub : 32;
      const int cend = kAlt ? p.BN : cbeg + p.BN / nsub;
      // SwiGLU backward: this lane's row of the saved g, u for a 32-column chunk
      uint4 gq[4], uq[4];
      auto ld_gu = [&](int c, uint4 (&g4)[4], uint4 (&u4)[4]) {
        const bool ok = lane < nvalid;
        const uint4* row = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.aux) +
                                                          (size_t)(ok ? rb + lane : 0) * p.I * 4);
        const int v = (t.n0 + c) >> 3, vu = (p.I + t.n0 + c) >> 3;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          g4[i] = ok ? __ldg(row + v + i) : make_uint4(0, 0, 0, 0);
          u4[i] = ok ? __ldg(row + vu + i) : make_uint4(0, 0, 0, 0);
        }
      };
      if constexpr (KIND == DOWN_BWD_DX) {
        if (any) ld_gu(cbeg, gq, uq);
      }
      // FP8 kinds: this lane's row scale (the scale of its token when
      // gathering) and the expert's output-channel scales, lane L holding
      // column L of the current 32-column chunk (gate in sc0, up in sc1).
      // Loaded before the accumulator wait, later chunks one chunk ahead.
      float rs = 1.0f, sc0 = 0.0f, sc1 = 0.0f;
      const size_t cs_base = (size_t)(t.group < 0 ? 0 : t.group) * p.b_group_rows + t.n0;
      if constexpr (is_fp8(KIND)) {
        if (any) {
          if (lane < nvalid) {
            int src = rb + lane;
            if constexpr (is_gather(KIND)) {
              const int v = p.gather_rows[src];
              src = (v >= 0 && v < p.gather_limit) ? v : 0;
            }
            rs = __ldg(p.a_scale + src);
          }
          sc0 = __ldg(p.b_scale0 + cs_base + cbeg + lane);
          if constexpr (is_gate_up(KIND)) sc1 = __ldg(p.b_scale1 + cs_base + lane);
        }
      }
      if (!__all_sync(0xffffffffu, wait_bar(smem_u32(&ctl->tfull[buf]), use & 1u, &ctl->abort_flag, p.status))) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * ACC_COLS);


      if constexpr (is_gate_up(KIND)) {
        const size_t hp_pitch = (size_t)p.I * 2, gu_pitch = (size_t)p.I * 4;
        for (int c = 0; any && c < p.NH; c += 32) {
          float nx0 = 0.0f, nx1 = 0.0f;  // FP8: the next chunk's column scales
          if constexpr (is_fp8(KIND)) {
            if (c + 32 < p.NH) {
              nx0 = __ldg(p.b_scale0 + cs_base + c + 32 + lane);
              nx1 = __ldg(p.b_scale1 + cs_base + c + 32 + lane);
            }
          }
          uint32_t g[32], u[32];
          tmem_ld32(taddr + c, g);
          tmem_ld32(taddr + p.NH + c, u);
          tmem_wait_ld();
          uint32_t hp[16], gp[16], upk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float g0 = f32(g[2 * i]), g1 = f32(g[2 * i + 1]);
            float u0 = f32(u[2 * i]), u1 = f32(u[2 * i + 1]);
            if constexpr (is_fp8(KIND)) {
              g0 = g0 * rs * __shfl_sync(0xffffffffu, sc0, 2 * i);
              g1 = g1 * rs * __shfl_sync(0xffffffffu, sc0, 2 * i + 1);
              u0 = u0 * rs * __shfl_sync(0xffffffffu, sc1, 2 * i);
              u1 = u1 * rs * __shfl_sync(0xffffffffu, sc1, 2 * i + 1);
            }
            const float h0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
            const float h1 = __fdividef(g1, 1.0f + __expf(-g1)) * u1;
            hp[i] = pack_bf16x2(h0, h1);
            gp[i] = pack_bf16x2(g0, g1);
            upk[i] = pack_bf16x2(u0, u1);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) put(ep_base, i, make_uint4(hp[4 * i], hp[4 * i + 1], hp[4 * i + 2], hp[4 * i + 3]));
          flush(ep_base, p.out0, hp_pitch, (size_t)(t.n0 + c) * 2, rb, nvalid, false);
          if (!is_fp8(KIND) && p.out1) {
#pragma unroll
            for (int i = 0; i < 4; ++i) put(ep_base, i, make_uint4(gp[4 * i], gp[4 * i + 1], gp[4 * i + 2], gp[4 * i + 3]));
            flush(ep_base, p.out1, gu_pitch, (size_t)(t.n0 + c) * 2, rb, nvalid, false);
#pragma unroll
            for (int i = 0; i < 4; ++i) put(ep_base, i, make_uint4(upk[4 * i], upk[4 * i + 1], upk[4 * i + 2], upk[4 * i + 3]));
            flush(ep_base, p.out1, gu_pitch, (size_t)(p.I + t.n0 + c) * 2, rb, nvalid, false);
          }
          sc0 = nx0;
          sc1 = nx1;
        }
      } else if constexpr (KIND == DOWN_COMBINE) {
        // out[token] += w * (this lane's row): the row's token from
        // token_of_row, its routing weight from the token's slot whose row
        // it is; 16-byte fp32 reductions in L2, in no fixed order
        int tok = -1;
        float wt = 0.0f;
        if (any && lane < nvalid) {
          const int r = rb + lane;
          const int tt = __ldg(p.comb_token + r);
          if (tt >= 0 && tt < p.comb_T) {
            for (int j = 0; j < p.comb_k; ++j) {
              if (__ldg(p.comb_rows + (size_t)tt * p.comb_k + j) == r) {
                tok = tt;
                wt = __ldg(p.comb_w + (size_t)tt * p.comb_k + j);
                break;
              }
            }
          }
        }
        for (int c = cbeg; any && c < cend; c += cstep) {
          uint32_t a[32];
          tmem_ld32(taddr + c, a);
          tmem_wait_ld();
          if (tok >= 0) {
            float* dst = p.comb_out + (size_t)tok * p.ldo + t.n0 + c;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              red_add_f32x4(dst + 4 * i, wt * f32(a[4 * i]), wt * f32(a[4 * i + 1]), wt * f32(a[4 * i + 2]),
                            wt * f32(a[4 * i + 3]));
          }
        }
      } else if constexpr (is_down_fwd(KIND) || KIND == GATE_UP_BWD_DX) {
        const size_t pitch = (size_t)p.ldo * 2;
        for (int c = cbeg; any && c < cend; c += cstep) {
          float nx0 = 0.0f;  // FP8: the next chunk's column scales
          if constexpr (is_fp8(KIND)) {
            if (c + cstep < cend) nx0 = __ldg(p.b_scale0 + cs_base + c + cstep + lane);
          }
          uint32_t a[32];
          tmem_ld32(taddr + c, a);
          tmem_wait_ld();
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = f32(a[i]);
          if constexpr (is_fp8(KIND)) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = v[i] * rs * __shfl_sync(0xffffffffu, sc0, i);
            sc0 = nx0;
          }
          uint4 pk[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            pk[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                               pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
          if (kTmaOut && nvalid == 32) {
            uint8_t* bx = ring.acquire();
#pragma unroll
            for (int i = 0; i < 4; ++i) ring.put(bx, i, pk[i]);
            ring.issue(bx, &tmO0, t.n0 + c, rb);
          } else {
            // a free slot (not awaiting a TMA store's read) for the direct path
            uint8_t* bx = kTmaOut ? ring.acquire() : ep_base;
#pragma unroll
            for (int i = 0; i < 4; ++i) put(bx, i, pk[i]);
            flush(bx, p.out0, pitch, (size_t)(t.n0 + c) * 2, rb, nvalid, false);
          }
        }
      } else if constexpr (KIND == DENSE_ADD) {
        // out = bf16(acc + add): the addend's two 16-column boxes of this
        // chunk sit in set (gu_ctr mod GU_SETS); the result goes out through the
        // first box of the set.
        const size_t pitch = (size_t)p.ldo * 2;
        for (int c = 0; any && c < p.BN; c += 32, ++gu_ctr) {
          gu_load(c + 32 * GU_AHEAD, gu_ctr + GU_AHEAD);
          uint32_t a[32];
          tmem_ld32(taddr + c, a);
          const int set = gu_ctr & (C::GU_SETS - 1);
          uint8_t* lo = ep_base + (2 * set) * EP_BOX_BYTES;
          uint8_t* hi = lo + EP_BOX_BYTES;
          const bool ok = __all_sync(0xffffffffu, wait_bar(gu_bar0 + 8u * (uint32_t)set,
                                                           (uint32_t)(gu_ctr / C::GU_SETS) & 1u, &ctl->abort_flag, p.status));
          tmem_wait_ld();
          if (!ok) break;
          uint4 pk[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 w = get(i < 2 ? lo : hi, (2 * i) & 3);
            const uint4 w2 = get(i < 2 ? lo : hi, (2 * i + 1) & 3);
            const float* av = reinterpret_cast<const float*>(&a[8 * i]);
            pk[i] = make_uint4(pack_bf16x2(av[0] + __uint_as_float(w.x), av[1] + __uint_as_float(w.y)),
                               pack_bf16x2(av[2] + __uint_as_float(w.z), av[3] + __uint_as_float(w.w)),
                               pack_bf16x2(av[4] + __uint_as_float(w2.x), av[5] + __uint_as_float(w2.y)),
                               pack_bf16x2(av[6] + __uint_as_float(w2.z), av[7] + __uint_as_float(w2.w)));
          }
          __syncwarp();  // every lane has read its addend row before the box is reused
#pragma unroll
          for (int i = 0; i < 4; ++i) put(lo, i, pk[i]);
          flush(lo, p.out0, pitch, (size_t)(t.n0 + c) * 2, rb, nvalid, false);
        }
      } else if constexpr (KIND == DOWN_BWD_DX) {
        // The saved g, u of this lane's row and chunk come from global memory
        // straight into registers, one chunk ahead; dg and du leave through
        // the warp's box by TMA stores (measured 15 us faster at T=8192 than
        // coalesced row stores from the box, which only the last rows of a
        // segment still use).
        const size_t pitch = (size_t)p.I * 4;
        for (int c = cbeg; any && c < cend; c += cstep) {
          uint4 gn[4], un[4];
          if (c + cstep < cend) ld_gu(c + cstep, gn, un);
          uint32_t a[32];
          tmem_ld32(taddr + c, a);
          tmem_wait_ld();
          uint4 og4[4], ou4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t gw[4] = {gq[i].x, gq[i].y, gq[i].z, gq[i].w};
            const uint32_t uw[4] = {uq[i].x, uq[i].y, uq[i].z, uq[i].w};
            uint32_t og[4], ou[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              float dg2[2], du2[2];
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const float g = hh ? bf16hi(gw[jj]) : bf16lo(gw[jj]);
                const float u = hh ? bf16hi(uw[jj]) : bf16lo(uw[jj]);
                const float dh = f32(a[8 * i + 2 * jj + hh]);
                const float sg = __fdividef(1.0f, 1.0f + __expf(-g));
                dg2[hh] = dh * u * sg * (1.0f + g * (1.0f - sg));
                du2[hh] = dh * (g * sg);
              }
              og[jj] = pack_bf16x2(dg2[0], dg2[1]);
              ou[jj] = pack_bf16x2(du2[0], du2[1]);
            }
            og4[i] = make_uint4(og[0], og[1], og[2], og[3]);
            ou4[i] = make_uint4(ou[0], ou[1], ou[2], ou[3]);
          }
          if (nvalid == 32) {
            uint8_t* bx = ring.acquire();
#pragma unroll
            for (int i = 0; i < 4; ++i) ring.put(bx, i, og4[i]);
            ring.issue(bx, &tmO0, t.n0 + c, rb);
            bx = ring.acquire();
#pragma unroll
            for (int i = 0; i < 4; ++i) ring.put(bx, i, ou4[i]);
            ring.issue(bx, &tmO0, p.I + t.n0 + c, rb);
          } else {  // the last rows of a segment: masked row stores
            uint8_t* bx = ring.acquire();
#pragma unroll
            for (int i = 0; i < 4; ++i) put(bx, i, og4[i]);
            flush(bx, p.out0, pitch, (size_t)(t.n0 + c) * 2, rb, nvalid, false);
#pragma unroll
            for (int i = 0; i < 4; ++i) put(bx, i, ou4[i]);
            flush(bx, p.out0, pitch, (size_t)(p.I + t.n0 + c) * 2, rb, nvalid, false);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            gq[i] = gn[i];
            uq[i] = un[i];
          }
        }
      } else {  // DW: fp32 [group, M, N] (optionally split at split_m over two tensors)
        const bool nonempty = ctl->grp_rows[t.group] > 0;
        if (any && (nonempty || !p.accumulate)) {
          const bool second = p.split_m > 0 && rb >= p.split_m;
          const int y = p.split_m > 0 ? t.group * p.split_m + (second ? rb - p.split_m : rb)
                                      : t.group * p.M + rb;
          // the written fp32 lines under an evict-last L2 policy (measured
          // 414 -> 392 us for dW_gate/up at T=8192 against the default
          // policy, 422 with evict-first)
          const uint64_t pol = l2_policy_evict_last();
          for (int c = cbeg; c < cend; c += cstep) {
            uint32_t a[32];
            if (nonempty) {
              tmem_ld32(taddr + c, a);
              tmem_wait_ld();
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) a[i] = 0u;
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              uint8_t* bx = ring.acquire();
#pragma unroll
              for (int i = 0; i < 4; ++i)
                ring.put(bx, i, make_uint4(a[16 * half + 4 * i], a[16 * half + 4 * i + 1],
                                           a[16 * half + 4 * i + 2], a[16 * half + 4 * i + 3]));
              ring.issue_hint(bx, second ? &tmO1 : &tmO0, t.n0 + c + 16 * half, y, p.accumulate != 0, pol);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (CTAS == 1)
          mbar_arrive(tempty_leader[buf]);
        else
          asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                           tempty_leader[buf])
                       : "memory");
      }
    }
    ring.drain();
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (CTAS == 2) cluster_sync();  // neither CTA frees TMEM while the pair still uses it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_n<CTAS>(tmem_base, TMEM_COLS);
  }
}

// Per-segment operand maps of the weight-gradient GEMM.  Thread i writes
// map i = 2s (A) or 2s+1 (B): a copy of the MN-major template whose base
// address is moved to segment s's first row and whose row extent is the
// segment's length (rows clamped to [0, rows) like the kernel's own table).
// An empty segment keeps the template unchanged; no k-block ever reads it.
// y = bf16(acc) (round to nearest even), eight elements per step.
__global__ void __launch_bounds__(256) f32_to_bf16_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ y,
                                                          size_t n8) {
  pdl_wait();
  pdl_trigger();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    reinterpret_cast<uint4*>(y)[i] =
        make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
  }
}

__global__ void dw_segment_maps_kernel(const __grid_constant__ CUtensorMap tplA,
                                       const __grid_constant__ CUtensorMap tplB,
                                       const int32_t* seg_offsets, int num_seg, int rows,
                                       const uint8_t* baseA, size_t pitchA, const uint8_t* baseB,
                                       size_t pitchB, CUtensorMap* maps) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 2 * num_seg) return;
  const int s = i >> 1;
  const bool isB = (i & 1) != 0;
  int a = seg_offsets ? seg_offsets[s] : 0;
  int b = seg_offsets ? seg_offsets[s + 1] : rows;
  a = a < 0 ? 0 : (a > rows ? rows : a);
  b = b < 0 ? 0 : (b > rows ? rows : b);
  CUtensorMap* m = maps + i;
  const uint4* src = reinterpret_cast<const uint4*>(isB ? &tplB : &tplA);
  uint4* dst = reinterpret_cast<uint4*>(m);
#pragma unroll
  for (int j = 0; j < (int)(sizeof(CUtensorMap) / sizeof(uint4)); ++j) dst[j] = src[j];
  if (b > a) {
    const uint64_t base = reinterpret_cast<uint64_t>(isB ? baseB : baseA) + (uint64_t)a * (isB ? pitchB : pitchA);
    const uint32_t len = (uint32_t)(b - a);
    asm volatile("tensormap.replace.tile.global_address.global.b1024.b64 [%0], %1;" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "l"(base)
                 : "memory");
    asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(len)
                 : "memory");
  }
  asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
}

// --------------------------------------------------------------- host side

int pick_bn(int n) { return n % 256 == 0 ? 256 : (n % 128 == 0 ? 128 : 64); }

// Cluster pairs (256-row tiles) need at least 128 output columns per tile
// (64 per CTA).  They are used where they measured faster: the gate/up
// backward dX GEMM, and the bf16 down projection and gate/up forward GEMM
// on permuted rows in the dispatch layout with enough rows per expert
// (pair_for_rows).  Every other kind runs one CTA per 128-row tile.
bool use_pair(int bn) { return bn >= 128; }

// The forward row kinds take pairs only in the dispatch layout (one segment
// per expert) and with at least 384 rows per segment on average: a pair
// tile wastes up to 255 rows of a segment's last tile, a single CTA's up to
// 127.  Measured at T=8192 (512 rows per expert): down 187 -> 181 us as
// pairs, gate/up equal; at T=4096 (256 rows): single CTAs 1.6-1.7% faster
// for both.
bool pair_for_rows(int bn, int R, int num_seg, int E) {
  return use_pair(bn) && num_seg <= E && (long long)R >= 384LL * num_seg;
}

bool g_attr[kNumKinds][2][64] = {};
// SMs the persistent GEMM grids may use, for launches from this thread (0: all)
thread_local int g_gemm_sm_limit = 0;

// Launches grouped_gemm_kernel<KIND, CTAS>: completes the CTAS-dependent
// parameters, sizes the shared memory to the segment tables and the
// persistent grid to the SM count and, for pairs, sets the cluster
// dimension.
template <int KIND, int CTAS>
int launch(Params p, const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
           const CUtensorMap& o0, const CUtensorMap& o1, cudaStream_t s, const char* what) {
  constexpr bool a_mn = KIND == DW;
  constexpr bool b_mn = KIND == DOWN_BWD_DX || KIND == GATE_UP_BWD_DX || KIND == DW;
  p.idesc = make_idesc(p.BN, BM * CTAS, a_mn, b_mn, is_fp8(KIND));
  long long upper;
  if (KIND == DW) {
    p.m_tiles = (p.M + BM * CTAS - 1) / (BM * CTAS);
    upper = (long long)p.num_groups * p.m_tiles * p.n_tiles;
  } else {
    upper = ((long long)(p.M + BM * CTAS - 1) / (BM * CTAS) + p.num_seg) * p.n_tiles;
  }
  const int dev = current_device();
  if (dev < 0) return fail(MOE_ERR_CUDA, "%s: no current CUDA device", what);
  auto kern = grouped_gemm_kernel<KIND, CTAS>;
  const size_t smem_sz = Cfg<KIND, CTAS>::SMEM_FIXED + seg_table_bytes(p.num_seg, p.num_groups, KIND == DW);
  if (smem_sz > kSmemMax) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "%s: segment tables too large", what);
  const int smem = (int)smem_sz;
  if (!g_attr[KIND][CTAS - 1][dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemMax);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    g_attr[KIND][CTAS - 1][dev] = true;
  }
  int sms = sm_count();
  if (sms <= 0) return fail(MOE_ERR_CUDA, "%s: cannot query the SM count", what);
  if (g_gemm_sm_limit > 0 && g_gemm_sm_limit < sms) sms = g_gemm_sm_limit;
  const long long units_max = sms / CTAS;
  long long units = upper < units_max ? upper : units_max;
  if (units < 1) units = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(units * CTAS));
  cfg.blockDim = dim3(Cfg<KIND, CTAS>::NTHREADS);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // the kernel starts with pdl_wait()
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (CTAS == 2) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a, b0, b1, o0, o1, p);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return check_launch(what);
}

// Cluster pairs are built for the gate/up GEMMs on permuted rows (forward
// and backward dX) and the bf16 down projection, where they measured
// faster; the down backward dX kind measured slower as pairs.
template <int KIND>
int run(bool pair, const Params& p, const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
        const CUtensorMap& o0, const CUtensorMap& o1, cudaStream_t s, const char* what) {
  if constexpr (KIND == GATE_UP_BWD_DX || KIND == GATE_UP_FWD || KIND == DOWN_FWD || KIND == DOWN_COMBINE) {
    if (pair) return launch<KIND, 2>(p, a, b0, b1, o0, o1, s, what);
  }
  return launch<KIND, 1>(p, a, b0, b1, o0, o1, s, what);
}

constexpr size_t kSegMapBytes = 2 * sizeof(CUtensorMap);  // A and B map of one segment

// Weight-gradient GEMM dW[g] = sum over g's rows of A^T B with A bf16
// [K_rows, M] and B bf16 [K_rows, N] (both MN-major operands): writes the
// per-segment maps into `maps` (num_seg * kSegMapBytes, 128-byte aligned),
// then runs the GEMM.  p must hold M, N, K, BN, n_tiles and the outputs.
int run_dw(bool pair, Params p, const void* A, const void* B, const CUtensorMap& o0,
           const CUtensorMap& o1, void* maps, cudaStream_t s, const char* what) {
  CUtensorMap ta, tb;
  const uint32_t nckB = p.BN / 64 / (pair ? 2 : 1);
  if (int rc = make_tmap_mn(&ta, A, p.M, p.K, BM / 64)) return rc;
  if (int rc = make_tmap_mn(&tb, B, p.N, p.K, nckB)) return rc;
  const int nmaps = 2 * p.num_seg;
  launch_pdl(dw_segment_maps_kernel, (nmaps + 127) / 128, 128, 0, s, 
      ta, tb, p.seg_offsets, p.num_seg, p.K, static_cast<const uint8_t*>(A), (size_t)p.M * 2,
      static_cast<const uint8_t*>(B), (size_t)p.N * 2, static_cast<CUtensorMap*>(maps));
  if (int rc = check_launch(what)) return rc;
  p.seg_maps = static_cast<const CUtensorMap*>(maps);
  return run<DW>(pair, p, ta, tb, tb, o0, o1, s, what);
}

// The backward GEMMs' workspace: the per-segment maps.
int check_bwd_ws(const char* fn, int num_seg, const void* ws, size_t ws_bytes) {
  const size_t need = (size_t)num_seg * kSegMapBytes;
  if (num_seg > 0 && (!ws || ws_bytes < need))
    return fail(MOE_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, ws ? ws_bytes : (size_t)0, need);
  if (ws && (reinterpret_cast<uintptr_t>(ws) & 127u))
    return fail(MOE_ERR_ALIGNMENT, "%s: ws must be 128-byte aligned", fn);
  return MOE_OK;
}

int check_grouped(const char* fn, int num_seg, const int32_t* seg_offsets, int R, int H, int I, int E) {
  if (R < 0 || H <= 0 || I <= 0 || E <= 0 || num_seg < 0)
    return fail(MOE_ERR_INVALID_ARG, "%s: need R>=0, H>0, I>0, E>0, num_seg>=0", fn);
  if (H % 64 || I % 64 || E > kMaxExperts || num_seg > kMaxSegments)
    return fail(MOE_ERR_UNSUPPORTED_SHAPE, "%s: need H%%64==0, I%%64==0, num_seg<=%d (H=%d I=%d num_seg=%d)",
                fn, kMaxSegments, H, I, num_seg);
  if (num_seg > 0 && !seg_offsets) return fail(MOE_ERR_INVALID_ARG, "%s: seg_offsets is NULL", fn);
  return MOE_OK;
}

Params base_params(int num_seg, const int32_t* so, const int32_t* se, int groups) {
  Params p{};
  p.num_seg = num_seg;
  p.seg_offsets = so;
  p.seg_expert = se;
  p.num_groups = groups;
  p.status = status_word();
  return p;
}


}  // namespace tc

// Router-backward helpers (declared in common.cuh).
int launch_dense_add_bf16(const void* A, const void* B, const float* add, void* out, int M, int N,
                          int K, cudaStream_t stream) {
  using namespace tc;
  if (M == 0) return MOE_OK;
  // one segment [0, M): a null segment table stands for it
  Params p = base_params(1, nullptr, nullptr, 1);
  p.M = M;
  p.N = N;
  p.K = K;
  p.BN = pick_bn(N);
  p.n_tiles = N / p.BN;
  p.b_group_rows = 0;
  p.ldo = N;
  p.out0 = out;
  p.aux = add;
  CUtensorMap ta, tb;
  if (int rc = make_tmap(&ta, A, K, M, 64, BM)) return rc;
  if (int rc = make_tmap(&tb, B, K, N, 64, p.BN)) return rc;
  CUtensorMap to, tadd;
  if (int rc = make_out_map(&to, out, N, M, false)) return rc;
  if (int rc = make_out_map(&tadd, add, N, M, true)) return rc;  // addend boxes in
  return run<DENSE_ADD>(false, p, ta, tb, tadd, to, to, stream, "router backward dx GEMM");
}

size_t dw_split_maps_bytes(int num_seg) { return (size_t)num_seg * tc::kSegMapBytes; }


int launch_dw_split(const void* A, const void* B, int K_rows, int M, int N,
                    const int32_t* seg_offsets, int num_seg, float* out, void* maps,
                    cudaStream_t stream) {
  using namespace tc;
  Params p = base_params(num_seg, seg_offsets, nullptr, num_seg);
  p.M = M;
  p.N = N;
  p.K = K_rows;
  p.BN = pick_bn(N);
  p.n_tiles = N / p.BN;
  p.ldo = N;
  p.out0 = out;
  CUtensorMap to;
  if (int rc = make_out_map(&to, out, N, (uint64_t)num_seg * M, true)) return rc;
  return run_dw(false, p, A, B, to, to, maps, stream, "router backward dWr GEMM");
}

}  // namespace moe

using namespace moe;
using namespace moe::tc;

namespace moe {
namespace tc {

// Gate/up GEMM + SwiGLU on A rows x_perm[r] (gather_rows == nullptr) or
// x[gather_rows[r]] (rows copied by cp.async in the producer warp).
int swiglu_impl(const void* a_src, const int32_t* gather_rows, int T, const void* Wg, const void* Wu,
                int num_seg, const int32_t* seg_offsets, const int32_t* seg_expert, int R, int H,
                int I, int E, void* h, void* gu_save, cudaStream_t s, const char* fn) {
  Params p = base_params(num_seg, seg_offsets, seg_expert, E);
  p.M = R;
  p.N = I;
  p.K = H;
  p.NH = (I % 128 == 0) ? 128 : 64;
  p.BN = 2 * p.NH;
  p.n_tiles = I / p.NH;
  p.b_group_rows = I;
  p.I = I;
  p.out0 = h;
  p.out1 = gu_save;
  p.gather_rows = gather_rows;
  p.gather_limit = T;
  CUtensorMap ta, tg, tu;
  if (gather_rows) {
    p.aux = a_src;  // x rows are copied by cp.async; the A map is unused
    if (int rc = make_tmap(&ta, a_src, H, T, 64, 64)) return rc;
  } else {
    if (int rc = make_tmap(&ta, a_src, H, R, 64, BM)) return rc;
  }
  if (int rc = make_tmap(&tg, Wg, H, (uint64_t)E * I, 64, p.NH)) return rc;
  if (int rc = make_tmap(&tu, Wu, H, (uint64_t)E * I, 64, p.NH)) return rc;
  CUtensorMap th, tgu;
  if (int rc = make_out_map(&th, h, I, R, false)) return rc;
  if (int rc = make_out_map(&tgu, gu_save ? gu_save : h, gu_save ? 2 * I : I, R, false)) return rc;
  if (gather_rows) return run<GATE_UP_GATHER>(false, p, ta, tg, tu, th, tgu, s, fn);
  // Cluster pairs (the leader loads the gate rows of B, the peer the up rows)
  // by pair_for_rows.  With several segments per expert (the EP receive
  // layout) each expert's weights stay in L2 across its segments and the
  // 256-row tiles waste more rows: single CTAs measured faster there.
  const bool pair = pair_for_rows(p.BN, R, num_seg, E);
  return run<GATE_UP_FWD>(pair, p, ta, tg, tu, th, tgu, s, fn);
}

// e4m3 operands: H and I must be multiples of 128 (one 128-byte k-block).
int check_fp8(const char* fn, int H, int I) {
  if (H % 128 || I % 128)
    return fail(MOE_ERR_UNSUPPORTED_SHAPE, "%s: e4m3 GEMMs need H%%128==0 and I%%128==0 (H=%d I=%d)", fn, H, I);
  return MOE_OK;
}

// Gate/up GEMM + SwiGLU on e4m3 rows (permuted, or gathered from x's token
// rows by token_of_row) and e4m3 weights, scales applied in the epilogue.
int swiglu_fp8_impl(const void* a, const float* a_scale, const int32_t* gather_rows, int T,
                    const void* Wg, const float* Wg_scale, const void* Wu, const float* Wu_scale,
                    int num_seg, const int32_t* seg_offsets, const int32_t* seg_expert, int R, int H,
                    int I, int E, void* h, cudaStream_t s, const char* fn) {
  Params p = base_params(num_seg, seg_offsets, seg_expert, E);
  p.M = R;
  p.N = I;
  p.K = H;
  p.NH = (I % 128 == 0) ? 128 : 64;
  p.BN = 2 * p.NH;
  p.n_tiles = I / p.NH;
  p.b_group_rows = I;
  p.I = I;
  p.out0 = h;
  p.out1 = nullptr;
  p.gather_rows = gather_rows;
  p.gather_limit = T;
  p.a_scale = a_scale;
  p.b_scale0 = Wg_scale;
  p.b_scale1 = Wu_scale;
  CUtensorMap ta, tg, tu, th;
  if (gather_rows) {
    p.aux = a;  // token rows are copied by cp.async; the A map is unused
    if (int rc = make_tmap_e4m3(&ta, a, H, T, 128, 64)) return rc;
  } else {
    if (int rc = make_tmap_e4m3(&ta, a, H, R, 128, BM)) return rc;
  }
  if (int rc = make_tmap_e4m3(&tg, Wg, H, (uint64_t)E * I, 128, p.NH)) return rc;
  if (int rc = make_tmap_e4m3(&tu, Wu, H, (uint64_t)E * I, 128, p.NH)) return rc;
  if (int rc = make_out_map(&th, h, I, R, false)) return rc;
  if (gather_rows) return run<GATE_UP_GATHER_FP8>(false, p, ta, tg, tu, th, th, s, fn);
  return run<GATE_UP_FP8>(false, p, ta, tg, tu, th, th, s, fn);
}

}  // namespace tc
}  // namespace moe

extern "C" {

int moe_set_gemm_sm_limit(int max_sms, int* previous) {
  clear_error();
  if (max_sms < 0) return fail(MOE_ERR_INVALID_ARG, "moe_set_gemm_sm_limit: max_sms must be >= 0");
  if (previous) *previous = g_gemm_sm_limit;
  g_gemm_sm_limit = max_sms;
  return MOE_OK;
}

size_t moe_grouped_gemm_bwd_workspace_size(int num_seg) {
  return num_seg > 0 ? (size_t)num_seg * kSegMapBytes : 0;
}

int moe_grouped_gemm_swiglu(const void* x_perm, const void* Wg, const void* Wu, int num_seg,
                            const int32_t* seg_offsets, const int32_t* seg_expert, int R, int H,
                            int I, int E, void* h, void* gu_save, void* ws, size_t ws_bytes,
                            void* stream) {
  (void)ws; (void)ws_bytes;
  clear_error();
  const char* fn = "moe_grouped_gemm_swiglu";
  if (int rc = check_grouped(fn, num_seg, seg_offsets, R, H, I, E)) return rc;
  if (!x_perm || !Wg || !Wu || !h) return fail(MOE_ERR_INVALID_ARG, "%s: NULL pointer argument", fn);
  if (!aligned16(x_perm) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(h) ||
      (gu_save && !aligned16(gu_save)))
    return fail(MOE_ERR_ALIGNMENT, "%s: tensors must be 16-byte aligned", fn);
  if (R == 0 || num_seg == 0) return MOE_OK;
  return swiglu_impl(x_perm, nullptr, 0, Wg, Wu, num_seg, seg_offsets, seg_expert, R, H, I, E, h,
                     gu_save, static_cast<cudaStream_t>(stream), fn);
}

int moe_grouped_gemm_swiglu_gather(const void* x, const int32_t* token_of_row, int T,
                                   const void* Wg, const void* Wu, int num_seg,
                                   const int32_t* seg_offsets, const int32_t* seg_expert, int R,
                                   int H, int I, int E, void* h, void* gu_save, void* stream) {
  clear_error();
  const char* fn = "moe_grouped_gemm_swiglu_gather";
  if (int rc = check_grouped(fn, num_seg, seg_offsets, R, H, I, E)) return rc;
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "%s: need T>=0", fn);
  if (R > 0 && num_seg > 0 && (!x || !token_of_row || !Wg || !Wu || !h || T == 0))
    return fail(MOE_ERR_INVALID_ARG, "%s: NULL pointer argument or no tokens", fn);
  if (!aligned16(x) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(h) ||
      (gu_save && !aligned16(gu_save)))
    return fail(MOE_ERR_ALIGNMENT, "%s: tensors must be 16-byte aligned", fn);
  if (R == 0 || num_seg == 0) return MOE_OK;
  return swiglu_impl(x, token_of_row, T, Wg, Wu, num_seg, seg_offsets, seg_expert, R, H, I, E, h,
                     gu_save, static_cast<cudaStream_t>(stream), fn);
}

int moe_grouped_gemm_swiglu_fp8(const void* a, const float* a_scale, const int32_t* token_of_row,
                                int T, const void* Wg, const float* Wg_scale, const void* Wu,
                                const float* Wu_scale, int num_seg, const int32_t* seg_offsets,
                                const int32_t* seg_expert, int R, int H, int I, int E, void* h,
                                void* stream) {
  clear_error();
  const char* fn = "moe_grouped_gemm_swiglu_fp8";
  if (int rc = check_grouped(fn, num_seg, seg_offsets, R, H, I, E)) return rc;
  if (int rc = check_fp8(fn, H, I)) return rc;
  if (token_of_row && T <= 0) return fail(MOE_ERR_INVALID_ARG, "%s: gathering needs T>0", fn);
  if (R > 0 && num_seg > 0 && (!a || !a_scale || !Wg || !Wg_scale || !Wu || !Wu_scale || !h))
    return fail(MOE_ERR_INVALID_ARG, "%s: NULL pointer argument", fn);
  if (!aligned16(a) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(h) || !aligned16(Wg_scale) ||
      !aligned16(Wu_scale))
    return fail(MOE_ERR_ALIGNMENT, "%s: tensors and weight scales must be 16-byte aligned", fn);
  if (R == 0 || num_seg == 0) return MOE_OK;
  return swiglu_fp8_impl(a, a_scale, token_of_row, T, Wg, Wg_scale, Wu, Wu_scale, num_seg,
                         seg_offsets, seg_expert, R, H, I, E, h, static_cast<cudaStream_t>(stream), fn);
}

int moe_grouped_gemm_down_fp8(const void* h, const float* h_scale, const void* Wd,
                              const float* Wd_scale, int num_seg, const int32_t* seg_offsets,
                              const int32_t* seg_expert, int R, int H, int I, int E, void* y_perm,
                              void* stream) {
  clear_error();
  const char* fn = "moe_grouped_gemm_down_fp8";
  if (int rc = check_grouped(fn, num_seg, seg_offsets, R, H, I, E)) return rc;
  if (int rc = check_fp8(fn, H, I)) return rc;
  if (R > 0 && num_seg > 0 && (!h || !h_scale || !Wd || !Wd_scale || !y_perm))
    return fail(MOE_ERR_INVALID_ARG, "%s: NULL pointer argument", fn);
  if (!aligned16(h) || !aligned16(Wd) || !aligned16(y_perm) || !aligned16(Wd_scale))
    return fail(MOE_ERR_ALIGNMENT, "%s: tensors and weight scales must be 16-byte aligned", fn);
  if (R == 0 || num_seg == 0) return MOE_OK;
  Params p = base_params(num_seg, seg_offsets, seg_expert, E);
  p.M = R;
  p.N = H;
  p.K = I;
  p.BN = pick_bn(H);
  p.n_tiles = H / p.BN;
  p.b_group_rows = H;
  p.ldo = H;
  p.out0 = y_perm;
  p.a_scale = h_scale;
  p.b_scale0 = Wd_scale;
  CUtensorMap ta, tb, to;
  if (int rc = make_tmap_e4m3(&ta, h, I, R, 128, BM)) return rc;
  if (int rc = make_tmap_e4m3(&tb, Wd, I, (uint64_t)E * H, 128, p.BN)) return rc;
  if (int rc = make_out_map(&to, y_perm, H, R, false)) return rc;
  return run<DOWN_FP8>(false, p, ta, tb, tb, to, to, static_cast<cudaStream_t>(stream), fn);
}

int moe_grouped_gemm_down(const void* h, const void* Wd, int num_seg, const int32_t* seg_offsets,
                          const int32_t* seg_expert, int R, int H, int I, int E, void* y_perm,
                          void* ws, size_t ws_bytes, void* stream) {
  (void)ws; (void)ws_bytes;
  clear_error();
  const char* fn = "moe_grouped_gemm_down";
  if (int rc = check_grouped(fn, num_seg, seg_offsets, R, H, I, E)) return rc;
  if (!h || !Wd || !y_perm) return fail(MOE_ERR_INVALID_ARG, "%s: NULL pointer argument", fn);
  if (!aligned16(h) || !aligned16(Wd) || !aligned16(y_perm))
    return fail(MOE_ERR_ALIGNMENT, "%s: tensors must be 16-byte aligned", fn);
  if (R == 0 || num_seg == 0) return MOE_OK;
  Params p = base_params(num_seg, seg_offsets, seg_expert, E);
  p.M = R;
  p.N = H;
  p.K = I;
  p.BN = pick_bn(H);
  p.n_tiles = H / p.BN;
  p.b_group_rows = H;
  p.ldo = H;
  p.out0 = y_perm;
  CUtensorMap ta, tb;
  if (int rc = make_tmap(&ta, h, I, R, 64, BM)) return rc;
  const bool pair = pair_for_rows(p.BN, R, num_seg, E);
  if (int rc = make_tmap(&tb, Wd, I, (uint64_t)E * H, 64, p.BN / (pair ? 2 : 1))) return rc;
  CUtensorMap to;
  if (int rc = make_out_map(&to, y_perm, H, R, false)) return rc;
  return run<DOWN_FWD>(pair, p, ta, tb, tb, to, to, static_cast<cudaStream_t>(stream), fn);
}

int moe_grouped_gemm_down_combine(const void* h, const void* Wd, int num_seg, const int32_t* seg_offsets,
                                  const int32_t* seg_expert, int R, int H, int I, int E,
                                  const int32_t* token_of_row, const int32_t* row_of_slot, const float* topk_w,
                                  int T, int k, float* y_acc, void* y, void* stream) {
  clear_error();
  const char* fn = "moe_grouped_gemm_down_combine";
  if (int rc = check_grouped(fn, num_seg, seg_offsets, R, H, I, E)) return rc;
  if (T < 0 || k < 1 || k > 32) return fail(MOE_ERR_INVALID_ARG, "%s: need T>=0, 1<=k<=32", fn);
  const bool rows = R > 0 && num_seg > 0;
  if ((T > 0 && (!y_acc || !y)) || (rows && (!h || !Wd || !token_of_row || (T > 0 && (!row_of_slot || !topk_w)))))
    return fail(MOE_ERR_INVALID_ARG, "%s: NULL pointer argument", fn);
  if ((h && !aligned16(h)) || (Wd && !aligned16(Wd)) || (y_acc && !aligned16(y_acc)) || (y && !aligned16(y)))
    return fail(MOE_ERR_ALIGNMENT, "%s: tensors must be 16-byte aligned", fn);
  if (T == 0) return MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(y_acc, 0, sizeof(float) * (size_t)T * H, s);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  if (rows) {
    Params p = base_params(num_seg, seg_offsets, seg_expert, E);
    p.M = R;
    p.N = H;
    p.K = I;
    p.BN = pick_bn(H);
    p.n_tiles = H / p.BN;
    p.b_group_rows = H;
    p.ldo = H;
    p.comb_token = token_of_row;
    p.comb_rows = row_of_slot;
    p.comb_w = topk_w;
    p.comb_out = y_acc;
    p.comb_T = T;
    p.comb_k = k;
    CUtensorMap ta, tb;
    if (int rc = make_tmap(&ta, h, I, R, 64, BM)) return rc;
    const bool pair = pair_for_rows(p.BN, R, num_seg, E);
    if (int rc = make_tmap(&tb, Wd, I, (uint64_t)E * H, 64, p.BN / (pair ? 2 : 1))) return rc;
    // no output map: the epilogue adds straight into y_acc (the A map fills the slots)
    if (int rc = run<DOWN_COMBINE>(pair, p, ta, tb, tb, ta, ta, s, fn)) return rc;
  }
  const size_t n8 = (size_t)T * H / 8;
  const int sms = sm_count();
  const size_t blocks = (n8 + 255) / 256, cap = (size_t)(sms > 0 ? sms : 148) * 8;
  launch_pdl(f32_to_bf16_kernel, (unsigned)(blocks < cap ? blocks : cap), 256, 0, s, static_cast<const float*>(y_acc),
             static_cast<__nv_bfloat16*>(y), n8);
  return check_launch(fn);
}

// B2 and B3 each run as two halves: the dX GEMM (rows x weights, with the
// SwiGLU backward in the down half's epilogue) and the weight-gradient GEMM
// (the per-segment operand maps, then the DW kind).  The combined entry
// points launch both on the same stream.

static int check_bwd_ptrs(const char* fn, std::initializer_list<const void*> ptrs) {
  for (const void* q : ptrs)
    if (!q) return fail(MOE_ERR_INVALID_ARG, "%s: NULL pointer argument", fn);
  for (const void* q : ptrs)
    if (!aligned16(q)) return fail(MOE_ERR_ALIGNMENT, "%s: tensors must be 16-byte aligned", fn);
  return MOE_OK;
}

// dgu = SwiGLU'(dy_perm . Wd[e])
static int down_bwd_dx(const void* dy_perm, const void* gu_save, const void* Wd, int num_seg,
                       const int32_t* seg_offsets, const int32_t* seg_expert, int R, int H, int I, int E,
                       void* dgu, cudaStream_t s, const char* fn) {
  if (R == 0 || num_seg == 0) return MOE_OK;
  Params p = base_params(num_seg, seg_offsets, seg_expert, E);
  p.M = R;
  p.N = I;
  p.K = H;
  p.BN = pick_bn(I);
  p.n_tiles = I / p.BN;
  p.b_group_rows = H;
  p.I = I;
  p.out0 = dgu;
  p.aux = gu_save;
  CUtensorMap ta, tb;
  if (int rc = make_tmap(&ta, dy_perm, H, R, 64, BM)) return rc;
  if (int rc = make_tmap_mn(&tb, Wd, I, (uint64_t)E * H, p.BN / 64)) return rc;
  CUtensorMap to;
  if (int rc = make_out_map(&to, dgu, 2 * I, R, false)) return rc;
  return run<DOWN_BWD_DX>(false, p, ta, tb, tb, to, to, s, fn);
}

// dWd[e] = dy_perm[rows of e]^T . h[rows of e]
static int down_bwd_dw(const void* dy_perm, const void* h, int num_seg, const int32_t* seg_offsets,
                       const int32_t* seg_expert, int R, int H, int I, int E, float* dWd, int accumulate,
                       void* ws, cudaStream_t s, const char* fn) {
  if (num_seg == 0) {
    if (accumulate) return MOE_OK;
    cudaError_t e = cudaMemsetAsync(dWd, 0, sizeof(float) * (size_t)E * H * I, s);
    return e == cudaSuccess ? MOE_OK : fail(MOE_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  }
  Params p = base_params(num_seg, seg_offsets, seg_expert, E);
  p.M = H;
  p.N = I;
  p.K = R;
  p.BN = pick_bn(I);
  p.n_tiles = I / p.BN;
  p.ldo = I;
  p.accumulate = accumulate;
  p.out0 = dWd;
  CUtensorMap to;
  if (int rc = make_out_map(&to, dWd, I, (uint64_t)E * H, true)) return rc;
  return run_dw(false, p, dy_perm, h, to, to, ws, s, fn);
}

// dx_perm = [dg du] . [Wg[e]; Wu[e]]
static int swiglu_bwd_dx(const void* dgu, const void* Wg, const void* Wu, int num_seg,
                         const int32_t* seg_offsets, const int32_t* seg_expert, int R, int H, int I, int E,
                         void* dx_perm, cudaStream_t s, const char* fn) {
  if (R == 0 || num_seg == 0) return MOE_OK;
  Params p = base_params(num_seg, seg_offsets, seg_expert, E);
  p.M = R;
  p.N = H;
  p.K = 2 * I;
  p.BN = pick_bn(H);
  p.n_tiles = H / p.BN;
  p.b_group_rows = I;
  p.I = I;
  p.ldo = H;
  p.out0 = dx_perm;
  const bool pair = use_pair(p.BN);
  CUtensorMap ta, tg, tu;
  if (int rc = make_tmap(&ta, dgu, 2 * I, R, 64, BM)) return rc;
  const uint32_t nck = p.BN / 64 / (pair ? 2 : 1);
  if (int rc = make_tmap_mn(&tg, Wg, H, (uint64_t)E * I, nck)) return rc;
  if (int rc = make_tmap_mn(&tu, Wu, H, (uint64_t)E * I, nck)) return rc;
  CUtensorMap to;
  if (int rc = make_out_map(&to, dx_perm, H, R, false)) return rc;
  return run<GATE_UP_BWD_DX>(pair, p, ta, tg, tu, to, to, s, fn);
}

// [dWg[e]; dWu[e]] = dgu[rows of e]^T . x_perm[rows of e]   (M = 2I split at I)
static int swiglu_bwd_dw(const void* dgu, const void* x_perm, int num_seg, const int32_t* seg_offsets,
                         const int32_t* seg_expert, int R, int H, int I, int E, float* dWg, float* dWu,
                         int accumulate, void* ws, cudaStream_t s, const char* fn) {
  if (num_seg == 0) {
    if (accumulate) return MOE_OK;
    cudaError_t e = cudaMemsetAsync(dWg, 0, sizeof(float) * (size_t)E * I * H, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dWu, 0, sizeof(float) * (size_t)E * I * H, s);
    return e == cudaSuccess ? MOE_OK : fail(MOE_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  }
  Params p = base_params(num_seg, seg_offsets, seg_expert, E);
  p.M = 2 * I;
  p.N = H;
  p.K = R;
  p.BN = pick_bn(H);
  p.n_tiles = H / p.BN;
  p.split_m = I;
  p.ldo = H;
  p.accumulate = accumulate;
  p.out0 = dWg;
  p.out1 = dWu;
  CUtensorMap tog, tou;
  if (int rc = make_out_map(&tog, dWg, H, (uint64_t)E * I, true)) return rc;
  if (int rc = make_out_map(&tou, dWu, H, (uint64_t)E * I, true)) return rc;
  return run_dw(false, p, dgu, x_perm, tog, tou, ws, s, fn);
}

int moe_grouped_gemm_down_bwd(const void* dy_perm, const void* h, const void* gu_save,
                              const void* Wd, int num_seg, const int32_t* seg_offsets,
                              const int32_t* seg_expert, int R, int H, int I, int E, void* dgu,
                              float* dWd, int accumulate, void* ws, size_t ws_bytes, void* stream) {
  clear_error();
  const char* fn = "moe_grouped_gemm_down_bwd";
  if (int rc = check_grouped(fn, num_seg, seg_offsets, R, H, I, E)) return rc;
  if (int rc = check_bwd_ptrs(fn, {dy_perm, h, gu_save, Wd, dgu, dWd})) return rc;
  if (int rc = check_bwd_ws(fn, num_seg, ws, ws_bytes)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (int rc = down_bwd_dx(dy_perm, gu_save, Wd, num_seg, seg_offsets, seg_expert, R, H, I, E, dgu, s, fn))
    return rc;
  return down_bwd_dw(dy_perm, h, num_seg, seg_offsets, seg_expert, R, H, I, E, dWd, accumulate, ws, s, fn);
}

int moe_grouped_gemm_down_bwd_dx(const void* dy_perm, const void* gu_save, const void* Wd, int num_seg,
                                 const int32_t* seg_offsets, const int32_t* seg_expert, int R, int H,
                                 int I, int E, void* dgu, void* stream) {
  clear_error();
  const char* fn = "moe_grouped_gemm_down_bwd_dx";
  if (int rc = check_grouped(fn, num_seg, seg_offsets, R, H, I, E)) return rc;
  if (int rc = check_bwd_ptrs(fn, {dy_perm, gu_save, Wd, dgu})) return rc;
  return down_bwd_dx(dy_perm, gu_save, Wd, num_seg, seg_offsets, seg_expert, R, H, I, E, dgu,
                     static_cast<cudaStream_t>(stream), fn);
}

int moe_grouped_gemm_down_bwd_dw(const void* dy_perm, const void* h, int num_seg,
                                 const int32_t* seg_offsets, const int32_t* seg_expert, int R, int H,
                                 int I, int E, float* dWd, int accumulate, void* ws, size_t ws_bytes,
                                 void* stream) {
  clear_error();
  const char* fn = "moe_grouped_gemm_down_bwd_dw";
  if (int rc = check_grouped(fn, num_seg, seg_offsets, R, H, I, E)) return rc;
  if (int rc = check_bwd_ptrs(fn, {dy_perm, h, dWd})) return rc;
  if (int rc = check_bwd_ws(fn, num_seg, ws, ws_bytes)) return rc;
  return down_bwd_dw(dy_perm, h, num_seg, seg_offsets, seg_expert, R, H, I, E, dWd, accumulate, ws,
                     static_cast<cudaStream_t>(stream), fn);
}

int moe_grouped_gemm_swiglu_bwd(const void* dgu, const void* x_perm, const void* Wg,
                                const void* Wu, int num_seg, const int32_t* seg_offsets,
                                const int32_t* seg_expert, int R, int H, int I, int E,
                                void* dx_perm, float* dWg, float* dWu, int accumulate, void* ws,
                                size_t ws_bytes, void* stream) {
  clear_error();
  const char* fn = "moe_grouped_gemm_swiglu_bwd";
  if (int rc = check_grouped(fn, num_seg, seg_offsets, R, H, I, E)) return rc;
  if (int rc = check_bwd_ptrs(fn, {dgu, x_perm, Wg, Wu, dx_perm, dWg, dWu})) return rc;
  if (int rc = check_bwd_ws(fn, num_seg, ws, ws_bytes)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (int rc = swiglu_bwd_dx(dgu, Wg, Wu, num_seg, seg_offsets, seg_expert, R, H, I, E, dx_perm, s, fn))
    return rc;
  return swiglu_bwd_dw(dgu, x_perm, num_seg, seg_offsets, seg_expert, R, H, I, E, dWg, dWu, accumulate, ws,
                       s, fn);
}

int moe_grouped_gemm_swiglu_bwd_dx(const void* dgu, const void* Wg, const void* Wu, int num_seg,
                                   const int32_t* seg_offsets, const int32_t* seg_expert, int R, int H,
                                   int I, int E, void* dx_perm, void* stream) {
  clear_error();
  const char* fn = "moe_grouped_gemm_swiglu_bwd_dx";
  if (int rc = check_grouped(fn, num_seg, seg_offsets, R, H, I, E)) return rc;
  if (int rc = check_bwd_ptrs(fn, {dgu, Wg, Wu, dx_perm})) return rc;
  return swiglu_bwd_dx(dgu, Wg, Wu, num_seg, seg_offsets, seg_expert, R, H, I, E, dx_perm,
                       static_cast<cudaStream_t>(stream), fn);
}

int moe_grouped_gemm_swiglu_bwd_dw(const void* dgu, const void* x_perm, int num_seg,
                                   const int32_t* seg_offsets, const int32_t* seg_expert, int R, int H,
                                   int I, int E, float* dWg, float* dWu, int accumulate, void* ws,
                                   size_t ws_bytes, void* stream) {
  clear_error();
  const char* fn = "moe_grouped_gemm_swiglu_bwd_dw";
  if (int rc = check_grouped(fn, num_seg, seg_offsets, R, H, I, E)) return rc;
  if (int rc = check_bwd_ptrs(fn, {dgu, x_perm, dWg, dWu})) return rc;
  if (int rc = check_bwd_ws(fn, num_seg, ws, ws_bytes)) return rc;
  return swiglu_bwd_dw(dgu, x_perm, num_seg, seg_offsets, seg_expert, R, H, I, E, dWg, dWu, accumulate, ws,
                       static_cast<cudaStream_t>(stream), fn);
}

}  // extern "C"
