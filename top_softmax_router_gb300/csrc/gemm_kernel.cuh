// Grouped expert GEMM on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// "Training Trillion-Parameter MoE ..." blog, section 3.3: a grouped GEMM that
// organises the expert computation by expert-aggregated batches; RelayMoE
// summary, sections 1 and 3.1: dropless and padding-free -- every expert
// takes exactly the rows routed to it, however many that is.
//
// One persistent kernel per (chunk, GEMM).  Warp roles (192 threads):
//   warp 0      TMA producer: global -> 128B-swizzled shared memory stages
//   warp 1      MMA issuer: tcgen05.mma (M=128, N=BN, K=16) into TMEM;
//               also owns the TMEM allocation
//   warps 2..5  epilogue: tcgen05.ld TMEM -> registers -> fused math -> global
// Two TMEM accumulators (2 x BN fp32 columns) let the epilogue of one tile
// overlap the main loop of the next.  Work items are taken round-robin, or
// (GemmParams::work_ctr) from a device counter by the producer, which passes
// each item to the MMA and epilogue warps through a small shared-memory ring;
// either way every output tile is computed by one CTA in one fixed K order,
// so the result does not depend on which CTA takes which tile.
//
// Segment modes:
//   SEGK = false  rows of the output are the rows of an expert segment in the
//                 chunk's permuted buffer; tiles come from the chunk's tile
//                 list (128 rows of one expert each); K is a weight dimension.
//   SEGK = true   weight-gradient GEMMs: the output is one expert's weight
//                 matrix [M, N]; K runs over the expert's rows in the chunk.
//                 Rows past the segment end are zeroed in shared memory before
//                 the MMA reads them, so neighbouring experts never leak in.
//
// Operand layouts: K-major operands are loaded as [rows][64 K] boxes,
// MN-major operands as [64 K rows][64 MN] boxes; both with 128-byte swizzle,
// which is what the shared-memory descriptors describe.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int GEMM_BM = 128;
constexpr int GEMM_BK = 64;
constexpr int GEMM_WORK_RING = 4;   // work items the producer may post ahead of the slowest consumer
// Epilogue warps: 8 (two per TMEM lane quarter, splitting the column chunks) for the dActU kernel,
// whose epilogue does the most work per element; 4 (one per quarter) elsewhere.
__host__ __device__ constexpr int gemm_epi_warps(int epi) { return epi == 3 ? 8 : 4; }
__host__ __device__ constexpr int gemm_threads(int epi) { return 64 + 32 * gemm_epi_warps(epi); }

// Wait accounting (diagnostic builds, -DMOE_GEMM_WAIT_STATS; read with moe_diag_gemm_wait_stats).  The MMA
// warp adds the SM cycles it spends waiting for a stage's operands (full barrier) and for a free
// accumulator (tempty barrier), the producer the cycles it waits for a free stage (empty barrier), to
// counters of the kernel's class.  Without the macro ws_clock() is 0 and the sums fold away; the library
// is built without it, because the clock reads and atomics slow the kernels down.
#ifdef MOE_GEMM_WAIT_STATS
__device__ __forceinline__ long long ws_clock() { return clock64(); }
#else
__device__ __forceinline__ long long ws_clock() { return 0; }
#endif
// Counters of a class: [form (0 one CTA, 1 CTA pair)][EPI][TWO_PHASE] blocks of WS_FIELDS.
enum : int {
  WS_CTAS = 0,      // CTAs (pairs: clusters) that ran
  WS_LIFE,          // cycles from the MMA warp's start to its last MMA's completion
  WS_OPERANDS,      // cycles the MMA warp waited for a stage's operands
  WS_ACCUM,         // cycles the MMA warp waited for a free accumulator
  WS_STAGE,         // cycles the producer waited for a free stage
  WS_KBLOCKS,       // 64-deep K blocks multiplied
  WS_FIELDS = 8,
  WS_CLASSES = 32
};
static_assert(WS_CLASSES == MOE_GEMM_WAIT_CLASSES && WS_FIELDS == MOE_GEMM_WAIT_FIELDS, "moe.h counter layout");
__host__ __device__ constexpr int ws_class(int form, int epi, bool two_phase) {
  return form * 16 + epi * 2 + (two_phase ? 1 : 0);
}

enum Epi : int {
  EPI_SWIGLU = 0,  // act = silu(gate) * up -> bf16 out0          (dual B: gate | up halves)
  EPI_GATEUP = 1,  // gate -> out0, up -> out1 (bf16)              (dual B)
  EPI_STORE = 2,   // acc -> bf16 out0
  EPI_DACT = 3,    // SwiGLU backward epilogue (see below)
  EPI_DW = 4,      // fp32 weight gradient, stored on the expert's first chunk, added after
  // cross-entropy head (vocabulary projection; the tile's 256 columns are 256 classes)
  EPI_LSE = 5,     // per (row, tile): max and sum of exp(logit - max) over the tile's classes; target logit
  EPI_DLOGIT = 6,  // d = g (exp(logit - lse) - [class = target]) -> bf16 out0
  EPI_ACC = 7      // row tiles, fp32 out: stored when chunk == 0, added after (TMA store / reduce-add)
};

struct GemmParams {
  // SEGK = false: chunk tile list
  const int2* tiles;        // (row_begin, expert | rows << 16)
  const int* tile_count;
  const int2* tiles2;       // 256-row tiles (CTA-pair kernels)
  const int* tile2_count;
  int band;                 // 0: tile-major order (the tile's column tiles run back to back); > 0:
                            // bands of `band` row tiles, column-tile-major within a band
  int nk;                   // K blocks per phase
  int nk_total;             // K blocks of the main loop (nk, or 2 nk for two phases)
  // SEGK = true: active experts of the chunk and their row ranges
  const int* active;
  const int* active_count;
  const int* expert_off;    // [E + 1]
  int m_tiles;
  int n_problems;           // 1, or 2 (two outputs sharing the B operand)
  // both
  int n_tiles;
  int M, N;                 // valid output extent (SEGK: weight matrix; else N = columns)
  int ldo;                  // leading dimension of the outputs, in elements
  void* out0;
  void* out1;
  void* out2;
  // EPI_DACT, and the gathered operand (GATH != 0): its row r is row row_route[r] / route_k (a token) of
  // the token-major source tensor
  const float* gates;       // [N*k] by route id
  const int* row_route;     // chunk row -> route id
  int route_k;              // routes per token
  // EPI_STORE of the dX GEMM: the router-path term of each row's route, rt_dl[row] * rt_w[e, :], added to the
  // fp32 accumulator before the bf16 store (rt_dl = NULL: plain store)
  const float* rt_dl;       // [rows] router-logit gradient of each permuted row's route
  const float* rt_w;        // [E, N] fp32 router weights
  float* dgp;               // [rows, n_tiles] partial sums of dActU * act
  // EPI_DW
  int chunk;
  const int* first_touch;   // [E]: first chunk (in backward order) in which expert e has rows
  int64_t out_estride;      // elements per expert matrix
  // cross-entropy head
  const int* targets;       // [rows] class of each row
  const float* lse;         // [rows] log-sum-exp of each row's logits (EPI_DLOGIT)
  const float* rowscale;    // [rows] gradient of each row's loss (EPI_DLOGIT)
  float* part_m;            // [rows][ldp] per-tile maximum (EPI_LSE)
  float* part_z;            // [rows][ldp] per-tile sum of exp(logit - maximum) (EPI_LSE)
  float* tgt_logit;         // [rows] logit of the row's target class (EPI_LSE)
  int col0;                 // class index of output column 0
  int ldp;                  // partials per row (EPI_LSE)
  // work distribution: NULL = static (CTA b takes items b, b + grid, ...); else a zeroed device counter
  // from which the producer of each CTA takes the next item, so CTAs that finish early take more
  int* work_ctr;
  // Launch chaining (every GEMM is launched with programmatic stream serialization):
  //  pdl_late = 0: wait for the previous kernel in the stream before the first global access (the rule);
  //  pdl_late = 1: the caller guarantees that the previous kernel neither writes this GEMM's inputs nor
  //    touches its outputs, and that everything before that kernel is complete once it has started
  //    work (it waits up front and releases its dependents only after that wait); the GEMM then runs
  //    beside it and waits for it at the end, so its own completion implies that kernel's.
  //  trigger_early = 1: release the next kernel right after this GEMM's up-front wait (the next one is a
  //    pdl_late-style kernel that runs beside it); else once no work item is left to hand out.
  int pdl_late;
  int trigger_early;
  // errors
  int* status;
  int64_t limit_ns;
  // wait accounting (diagnostic builds): WS_CLASSES x WS_FIELDS counters, or NULL
  unsigned long long* wait_stats;
};

template <int BN, int EPI>
struct GemmSmem {
  static constexpr int A_BYTES = GEMM_BM * GEMM_BK * 2;       // 16 KB
  static constexpr int B_BYTES = BN * GEMM_BK * 2;            // 32 KB for BN = 256
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // The fp32 epilogues stage boxes for TMA store / reduce-add (2 x 4 KB per epilogue warp).
  static constexpr int STG_BYTES = (EPI == EPI_DW || EPI == EPI_ACC) ? 4 * 2 * 4096 : 0;
#ifndef MOE_GEMM_STAGES
#define MOE_GEMM_STAGES 4
#endif
#ifndef MOE_GEMM_DW_STAGES
#define MOE_GEMM_DW_STAGES 4   // 4 x 48 KB + 32 KB staging fits in 227 KB; 3 was 4% (mid) to 12% (vocab head) slower
#endif
  static constexpr int STAGES = (EPI == EPI_DW) ? MOE_GEMM_DW_STAGES : MOE_GEMM_STAGES;
  static constexpr int TILE_BYTES = STAGES * STAGE_BYTES;
  static constexpr int STG_OFF = TILE_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;
  // barriers and scalars after the stages and the staging buffers
  static constexpr int BAR_OFF = TILE_BYTES + STG_BYTES;
  static constexpr int TOTAL = BAR_OFF + 256 + 1024;          // + barriers + alignment slack
};

__device__ __forceinline__ void store_bf16x32(uint16_t* dst, const float (&v)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    w.x = pack_bf16(v[8 * q + 0], v[8 * q + 1]);
    w.y = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
    w.z = pack_bf16(v[8 * q + 4], v[8 * q + 5]);
    w.w = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
    d[q] = w;
  }
}
__device__ __forceinline__ void load_bf16x32(const uint16_t* src, float (&v)[32]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w = s[q];
    v[8 * q + 0] = bf16_lo(w.x); v[8 * q + 1] = bf16_hi(w.x);
    v[8 * q + 2] = bf16_lo(w.y); v[8 * q + 3] = bf16_hi(w.y);
    v[8 * q + 4] = bf16_lo(w.z); v[8 * q + 5] = bf16_hi(w.z);
    v[8 * q + 6] = bf16_lo(w.w); v[8 * q + 7] = bf16_hi(w.w);
  }
}

__device__ __forceinline__ void load_raw32(const uint16_t* src, uint4 (&w)[4]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) w[q] = s[q];
}
__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// Token of permuted row `row` (the row of the token-major source tensor that a gather reads).
__device__ __forceinline__ int gather_token(const GemmParams& p, int row) { return p.row_route[row] / p.route_k; }

// Tokens of the four rows lane (l & 15) gathers in K block kb of a weight-gradient item: rows
// 4 (l & 15) .. +3 of the block; rows past the segment take its first row (the MMA warp zeroes them).
template <class W>
__device__ __forceinline__ void segment_tokens(const GemmParams& p, const W& wk, int kb, int lane, int (&tok)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = kb * GEMM_BK + 4 * (lane & 15) + j;
    tok[j] = gather_token(p, wk.row0 + (r < wk.rows ? r : 0));
  }
}

// Work-item decoding shared by the three roles.
struct Work {
  int e;        // expert
  int row0;     // SEGK=false: first row of the tile; SEGK=true: first row of the segment
  int rows;     // rows of the tile (SEGK=false) or of the segment (SEGK=true)
  int mt, nt;   // tile coordinates
  int prob;     // problem index (SEGK)
  int nkb;      // K blocks in the main loop (over all phases)
};

template <bool SEGK>
__device__ __forceinline__ Work decode(const GemmParams& p, int w) {
  Work r;
  if constexpr (!SEGK) {
    int t;
    if (p.band > 0) {
      // bands of p.band row tiles; within a band the row tile varies fastest, so the CTAs working at
      // the same time share a few B tiles and a few A tiles (both stay in L2 while they are used)
      const int per_band = p.band * p.n_tiles;
      const int b = w / per_band;
      const int rem = w - b * per_band;
      const int in_band = min(p.band, *p.tile_count - b * p.band);
      r.nt = rem / in_band;
      t = b * p.band + (rem - r.nt * in_band);
    } else {
      t = w / p.n_tiles;
      r.nt = w - t * p.n_tiles;
    }
    const int2 tl = p.tiles[t];
    r.row0 = tl.x;
    r.e = tl.y & 0xFFFF;
    r.rows = tl.y >> 16;
    r.mt = 0;
    r.prob = 0;
    r.nkb = p.nk_total;
  } else {
    const int per_prob = p.m_tiles * p.n_tiles;
    const int per_all = (*p.active_count) * per_prob;
    r.prob = w / per_all;
    int rem = w - r.prob * per_all;
    const int a = rem / per_prob;
    rem -= a * per_prob;
    r.mt = rem / p.n_tiles;
    r.nt = rem - r.mt * p.n_tiles;
    r.e = p.active[a];
    r.row0 = p.expert_off[r.e];
    r.rows = p.expert_off[r.e + 1] - r.row0;
    r.nkb = (r.rows + GEMM_BK - 1) / GEMM_BK;
  }
  return r;
}

template <bool SEGK>
__device__ __forceinline__ int total_work(const GemmParams& p) {
  if constexpr (!SEGK) return (*p.tile_count) * p.n_tiles;
  else return (*p.active_count) * p.m_tiles * p.n_tiles * p.n_problems;
}

// Epilogue of one tile of output rows (row tiles: the gate/up, down-projection, dX and dActU GEMMs).
// Thread = row r of the tile (TMEM lane); `rows` valid rows start at output row `row0`; `half`
// selects this warp's share of the column chunks when two warps serve one TMEM lane quarter.
template <int EPI, int BN>
__device__ __forceinline__ void epilogue_rows(const GemmParams& p, int row0, int rows, int nt, int e, uint32_t tacc,
                                              int r, int half) {
  constexpr int NH = gemm_epi_warps(EPI) / 4;
  float v[32], u[32];
  if constexpr (EPI == EPI_SWIGLU || EPI == EPI_GATEUP) {
    const bool row_ok = r < rows;
    const int64_t row = (int64_t)row0 + r;
    const int i0 = nt * (BN / 2);
#pragma unroll 1
    for (int c = 32 * half; c < BN / 2; c += 32 * NH) {
      tc_ld32(tacc + c, v);
      tc_ld32(tacc + BN / 2 + c, u);
      if (row_ok && i0 + c < p.N) {
        if constexpr (EPI == EPI_SWIGLU) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = silu_f(v[j]) * u[j];
          store_bf16x32(static_cast<uint16_t*>(p.out0) + row * p.ldo + i0 + c, v);
        } else {
          store_bf16x32(static_cast<uint16_t*>(p.out0) + row * p.ldo + i0 + c, v);
          store_bf16x32(static_cast<uint16_t*>(p.out1) + row * p.ldo + i0 + c, u);
        }
      }
    }
  } else if constexpr (EPI == EPI_STORE) {
    const bool row_ok = r < rows;
    const int64_t row = (int64_t)row0 + r;
    const int n0 = nt * BN;
    // the dX GEMM adds its row's router-path term dl * Wr[e] in fp32 (one Wr row segment for the whole tile:
    // every row of a tile belongs to expert e)
    const bool router = p.rt_dl != nullptr;
    if (!router) {
#pragma unroll 1
      for (int c = 32 * half; c < BN; c += 32 * NH) {
        tc_ld32(tacc + c, v);
        if (row_ok && n0 + c < p.N) store_bf16x32(static_cast<uint16_t*>(p.out0) + row * p.ldo + n0 + c, v);
      }
    } else {
      // the next column chunk's Wr segment is loaded before this chunk's TMEM load
      const float dl = row_ok ? p.rt_dl[row] : 0.0f;
      const float4* wr = reinterpret_cast<const float4*>(p.rt_w + (int64_t)e * p.N + n0);
      float4 w[8];
      if (n0 + 32 * half < p.N) {
#pragma unroll
        for (int q = 0; q < 8; ++q) w[q] = __ldg(wr + 8 * half + q);
      }
#pragma unroll 1
      for (int c = 32 * half; c < BN; c += 32 * NH) {
        const int cn = c + 32 * NH;
        float4 wn[8];
        if (cn < BN && n0 + cn < p.N) {
#pragma unroll
          for (int q = 0; q < 8; ++q) wn[q] = __ldg(wr + cn / 4 + q);
        }
        tc_ld32(tacc + c, v);
        if (row_ok && n0 + c < p.N) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            v[4 * q + 0] = __fmaf_rn(dl, w[q].x, v[4 * q + 0]);
            v[4 * q + 1] = __fmaf_rn(dl, w[q].y, v[4 * q + 1]);
            v[4 * q + 2] = __fmaf_rn(dl, w[q].z, v[4 * q + 2]);
            v[4 * q + 3] = __fmaf_rn(dl, w[q].w, v[4 * q + 3]);
          }
          store_bf16x32(static_cast<uint16_t*>(p.out0) + row * p.ldo + n0 + c, v);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) w[q] = wn[q];
      }
    }
  } else if constexpr (EPI == EPI_DACT) {
    // acc = dActU = dYp . Wd_e   (columns i of this tile)
    // with gate/up the recomputed pre-activations, s = sigmoid(gate):
    //   act = silu(gate) * up;  partial dgate += sum_i dActU * act   (fixed column order)
    //   dAct = g * dActU;  dGate = dAct * up * s * (1 + gate * (1 - s));  dUp = dAct * silu(gate)
    //   stores dGate over gate, dUp over up, and g * act (the dWd operand)
    const bool row_ok = r < rows;
    const int64_t row = (int64_t)row0 + r;
    const int n0 = nt * BN;
    const float g = row_ok ? p.gates[p.row_route[row]] : 0.0f;
    float part = 0.0f;
    uint16_t* gate_p = static_cast<uint16_t*>(p.out0) + row * p.ldo + n0;
    uint16_t* up_p = static_cast<uint16_t*>(p.out1) + row * p.ldo + n0;
    uint16_t* gact_p = static_cast<uint16_t*>(p.out2) + row * p.ldo + n0;
    // The gate/up loads of the next column chunk are issued before this chunk's TMEM load, so their
    // latency overlaps the current chunk's arithmetic and stores.
    uint4 graw[4], uraw[4];
    if (row_ok && n0 + 32 * half < p.N) {
      load_raw32(gate_p + 32 * half, graw);
      load_raw32(up_p + 32 * half, uraw);
    }
#pragma unroll 1
    for (int c = 32 * half; c < BN; c += 32 * NH) {
      const int cn = c + 32 * NH;
      uint4 gnext[4], unext[4];
      if (row_ok && cn < BN && n0 + cn < p.N) {
        load_raw32(gate_p + cn, gnext);
        load_raw32(up_p + cn, unext);
      }
      tc_ld32(tacc + c, v);
      if (row_ok && n0 + c < p.N) {
        // eight columns at a time, so only one 16-byte group of each output is live
        uint4* gd = reinterpret_cast<uint4*>(gate_p + c);
        uint4* ud = reinterpret_cast<uint4*>(up_p + c);
        uint4* ad = reinterpret_cast<uint4*>(gact_p + c);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t gw[4] = {graw[q].x, graw[q].y, graw[q].z, graw[q].w};
          const uint32_t uw[4] = {uraw[q].x, uraw[q].y, uraw[q].z, uraw[q].w};
          uint32_t o0[4], o1[4], o2[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            float dgo[2], duo[2], ga[2];
#pragma unroll
            for (int b = 0; b < 2; ++b) {
              const int j = 8 * q + 2 * h + b;
              const float gt = b ? bf16_hi(gw[h]) : bf16_lo(gw[h]);
              const float uj = b ? bf16_hi(uw[h]) : bf16_lo(uw[h]);
              const float s = 1.0f / (1.0f + expf(-gt));
              const float sl = gt * s;
              const float act = sl * uj;
              part = fmaf(v[j], act, part);
              const float da = g * v[j];
              dgo[b] = da * uj * (s * (1.0f + gt * (1.0f - s)));
              duo[b] = da * sl;
              ga[b] = g * act;
            }
            o0[h] = pack_bf16(dgo[0], dgo[1]);
            o1[h] = pack_bf16(duo[0], duo[1]);
            o2[h] = pack_bf16(ga[0], ga[1]);
          }
          gd[q] = make_uint4(o0[0], o0[1], o0[2], o0[3]);
          ud[q] = make_uint4(o1[0], o1[1], o1[2], o1[3]);
          ad[q] = make_uint4(o2[0], o2[1], o2[2], o2[3]);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        graw[q] = gnext[q];
        uraw[q] = unext[q];
      }
    }
    if (row_ok) p.dgp[row * (p.n_tiles * NH) + nt * NH + half] = part;
  } else if constexpr (EPI == EPI_LSE) {
    // Columns are classes n0 .. n0+255 of this tile (valid below p.N).  Online over the 32-column
    // chunks: m = running maximum, z = sum of exp(y - m), rescaled when m grows (eq. (3) of the
    // bounded-streaming summary, applied within the tile).
    const bool row_ok = r < rows;
    const int64_t row = (int64_t)row0 + r;
    const int n0 = nt * BN;
    const int tcol = row_ok ? p.targets[row] - p.col0 - n0 : -1;   // target's column in this tile
    float m = -INFINITY, z = 0.0f, yt = 0.0f;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      if (n0 + c >= p.N) break;                                    // uniform across the warp
      tc_ld32(tacc + c, v);
      const int valid = p.N - n0 - c;
      float cm = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (j < valid) cm = fmaxf(cm, v[j]);
        if (c + j == tcol) yt = v[j];
      }
      const float mn = fmaxf(m, cm);
      float sz = 0.0f;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < valid) sz += expf(v[j] - mn);
      z = z * expf(m - mn) + sz;
      m = mn;
    }
    if (row_ok) {
      p.part_m[row * p.ldp + nt] = m;
      p.part_z[row * p.ldp + nt] = z;
      if (tcol >= 0 && tcol < BN && n0 + tcol < p.N) p.tgt_logit[row] = yt;
    }
  } else if constexpr (EPI == EPI_DLOGIT) {
    const bool row_ok = r < rows;
    const int64_t row = (int64_t)row0 + r;
    const int n0 = nt * BN;
    const float l = row_ok ? p.lse[row] : 0.0f;
    const float g = row_ok ? p.rowscale[row] : 0.0f;
    const int tcol = row_ok ? p.targets[row] - p.col0 - n0 : -1;
#pragma unroll 1
    for (int c = 32 * half; c < BN; c += 32 * NH) {
      if (n0 + c >= p.N) break;                                    // uniform across the warp
      tc_ld32(tacc + c, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = g * (expf(v[j] - l) - (c + j == tcol ? 1.0f : 0.0f));
      if (row_ok) store_bf16x32(static_cast<uint16_t*>(p.out0) + row * p.ldo + n0 + c, v);
    }
  }
}

// ---------------------------------------------------------------------------
// The kernel.
//   EPI       epilogue kind
//   A_MN,B_MN operand majorness (false: K-major)
//   SEGK      segment mode (see top of file)
//   BN        tile width (256)
//   DUAL_B    B tile = [BN/2 rows from tb0 ; BN/2 rows from tb1] (gate | up)
//   TWO_PHASE K loop runs over (ta0, tb0) then (ta1, tb1), p.nk blocks each
//   GATH      gather-on-load (the dispatch gather fused into the operand loads): 0 none; 1 the A operand,
//             2 the B operand is read straight from the token-major source (X or dY, map ta0 or tb0 of
//             make_map_gather) by the rows' tokens, four rows per tile::gather4, instead of from a
//             permuted copy.  Row tiles: A, K-major (32 gathers of 4 rows per stage).  Weight gradients:
//             the MN-major operand whose K rows are the segment's rows (16 gathers per 64-wide box).
// ---------------------------------------------------------------------------
template <int EPI, bool A_MN, bool B_MN, bool SEGK, int BN, bool DUAL_B, bool TWO_PHASE, int GATH = 0>
__global__ void __launch_bounds__(gemm_threads(EPI), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap ta0, const __grid_constant__ CUtensorMap ta1,
                        const __grid_constant__ CUtensorMap tb0, const __grid_constant__ CUtensorMap tb1,
                        const __grid_constant__ CUtensorMap to0, const __grid_constant__ CUtensorMap to1,
                        const GemmParams p) {
  using S = GemmSmem<BN, EPI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BAR_OFF);
  // bars[0..S) full, [S..2S) empty, [2S..2S+2) tmem full, [2S+2..2S+4) tmem empty, [2S+4] drain,
  // [2S+5..2S+5+NW) work posted, [2S+5+NW..2S+5+2NW) work taken
  constexpr int NW = GEMM_WORK_RING;
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S::STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * S::STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * S::STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S::STAGES + 4);
  auto wfull_bar = [&](int i) { return bar0 + 8u * (2 * S::STAGES + 5 + i); };
  auto wempty_bar = [&](int i) { return bar0 + 8u * (2 * S::STAGES + 5 + NW + i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::BAR_OFF + 8 * (2 * S::STAGES + 5 + 2 * NW));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* work_ring = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), gemm_epi_warps(EPI));
    }
    mbar_init(drain_bar, 1);
    for (int i = 0; i < NW; ++i) {
      mbar_init(wfull_bar(i), 1);
      mbar_init(wempty_bar(i), 1 + gemm_epi_warps(EPI));
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&ta0);
    tma_prefetch_desc(&tb0);
    if (TWO_PHASE || SEGK) tma_prefetch_desc(&ta1);
    if (DUAL_B || TWO_PHASE || SEGK) tma_prefetch_desc(&tb1);
  }
  if (warp == 1) {
    tc_alloc(smem_u32(tmem_slot), S::TMEM_COLS);
    tc_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (!p.pdl_late) pdl_wait();   // the set-up above touches no global memory; everything below may
  if (p.trigger_early) pdl_trigger();

  const int total = total_work<SEGK>(p);
  // Item of this CTA's iteration `it`, or -1 when there is none left, or -2 after an abort.
  // Producer side (lane 0 of warp 0): takes the item and posts it to the ring.
  auto produce_next = [&](int it) -> int {
    if (p.work_ctr == nullptr) {
      const int64_t w = blockIdx.x + (int64_t)it * gridDim.x;
      return w < total ? (int)w : -1;
    }
    const int slot = it % NW;
    if (!wait_bounded(wempty_bar(slot), ((it / NW) & 1) ^ 1, abort_flag, p.limit_ns, p.status, 105)) return -2;
    int w = atomicAdd(p.work_ctr, 1);
    if (w >= total) w = -1;
    work_ring[slot] = w;
    mbar_arrive(wfull_bar(slot));
    return w;
  };
  // Consumer side (a whole warp: the MMA warp or an epilogue warp): reads the posted item.
  auto consume_next = [&](int it) -> int {
    if (p.work_ctr == nullptr) {
      const int64_t w = blockIdx.x + (int64_t)it * gridDim.x;
      return w < total ? (int)w : -1;
    }
    const int slot = it % NW;
    int w = -2;
    if (lane == 0 && wait_bounded(wfull_bar(slot), (it / NW) & 1, abort_flag, p.limit_ns, p.status, 106)) {
      w = work_ring[slot];
      mbar_arrive(wempty_bar(slot));
    }
    return __shfl_sync(0xffffffffu, w, 0);
  };

  if (warp == 0 && GATH != 0) {
    // ------------------------------------------------------------ producer, gather-on-load (whole warp)
    // Lane 0 takes the work items, waits on the stage barriers and loads the other operand; every lane
    // issues gathers of four rows of the gathered operand.
    static_assert(GATH == 0 || !TWO_PHASE, "gathered operands have one K phase");
    int stage = 0;
    uint32_t phase = 0;
    int issued = 0;
    bool ok = true;
    long long ws_stage = 0;
    for (int it = 0; ok; ++it) {
      int w = 0;
      if (lane == 0) w = produce_next(it);
      w = __shfl_sync(0xffffffffu, w, 0);
      if (w < 0) {
        ok = w == -1;
        break;
      }
      const Work wk = decode<SEGK>(p, w);
      if constexpr (EPI == EPI_DW) {
        if (lane == 0 && p.first_touch != nullptr && p.first_touch[wk.e] != p.chunk) {
          const CUtensorMap* om = wk.prob ? &to1 : &to0;
          const int n0 = wk.nt * BN, m0 = wk.mt * GEMM_BM;
          for (int rr = 0; rr < GEMM_BM && m0 + rr < p.M; rr += 32)
            for (int c = 0; c < BN && n0 + c < p.N; c += 32) tma_prefetch_3d(om, n0 + c, m0 + rr, wk.e);
        }
      }
      int tok[4], tnx[4];
      if constexpr (!SEGK) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = 4 * lane + j;   // this lane's rows of the 128-row tile
          tok[j] = gather_token(p, wk.row0 + (r < wk.rows ? r : 0));
        }
      } else {
        segment_tokens(p, wk, 0, lane, tok);
      }
      for (int kb = 0; kb < wk.nkb; ++kb) {
        if constexpr (SEGK) {
          if (kb + 1 < wk.nkb) segment_tokens(p, wk, kb + 1, lane, tnx);   // in flight during this block
        }
        int good = 1;
        const long long ws0 = ws_clock();
        if (lane == 0) good = wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.limit_ns, p.status, 101);
        ws_stage += ws_clock() - ws0;
        if (!__shfl_sync(0xffffffffu, good, 0)) {
          ok = false;
          break;
        }
        const uint32_t fb = full_bar(stage);
        const uint32_t sa = sbase + stage * S::STAGE_BYTES;
        const uint32_t sb = sa + S::A_BYTES;
        if constexpr (!SEGK) {
          const int k0 = kb * GEMM_BK;
          if (lane == 0) mbar_expect_tx(fb, S::STAGE_BYTES);
          __syncwarp();
          tma_gather4(sa + 512 * lane, &ta0, fb, k0, tok[0], tok[1], tok[2], tok[3]);
          if (lane == 0) {
            if constexpr (DUAL_B) {
              tma_load_3d(sb, &tb0, fb, k0, wk.nt * (BN / 2), wk.e);
              tma_load_3d(sb + S::B_BYTES / 2, &tb1, fb, k0, wk.nt * (BN / 2), wk.e);
            } else if constexpr (!B_MN) {
              tma_load_3d(sb, &tb0, fb, k0, wk.nt * BN, wk.e);
            } else {
#pragma unroll
              for (int b = 0; b < BN / 64; ++b) tma_load_3d(sb + b * 8192, &tb0, fb, wk.nt * BN + 64 * b, k0, wk.e);
            }
          }
        } else {
          const int r0 = wk.row0 + kb * GEMM_BK;
          const int q = lane & 15, h = lane >> 4;
          if constexpr (GATH == 1) {
            // gathered A (MN-major over M): 64-wide boxes past M are skipped (their outputs are clipped)
            const int nA = min(GEMM_BM / 64, (p.M - wk.mt * GEMM_BM + 63) / 64);
            if (lane == 0) mbar_expect_tx(fb, nA * 8192 + S::B_BYTES);
            __syncwarp();
            if (h < nA) tma_gather4(sa + h * 8192 + 512 * q, &ta0, fb, wk.mt * GEMM_BM + 64 * h, tok[0], tok[1], tok[2], tok[3]);
            if (lane == 0) {
              const CUtensorMap* B = wk.prob ? &tb1 : &tb0;
#pragma unroll
              for (int b = 0; b < BN / 64; ++b) tma_load_2d(sb + b * 8192, B, fb, wk.nt * BN + 64 * b, r0);
            }
          } else {
            // gathered B (MN-major over N), shared by both problems; boxes past N are skipped
            const int nB = min(BN / 64, (p.N - wk.nt * BN + 63) / 64);
            if (lane == 0) mbar_expect_tx(fb, S::A_BYTES + nB * 8192);
            __syncwarp();
            for (int b = h; b < nB; b += 2)
              tma_gather4(sb + b * 8192 + 512 * q, &tb0, fb, wk.nt * BN + 64 * b, tok[0], tok[1], tok[2], tok[3]);
            if (lane == 0) {
              const CUtensorMap* A = wk.prob ? &ta1 : &ta0;
#pragma unroll
              for (int a = 0; a < GEMM_BM / 64; ++a) tma_load_2d(sa + a * 8192, A, fb, wk.mt * GEMM_BM + 64 * a, r0);
            }
          }
        }
        ++issued;
        if (++stage == S::STAGES) { stage = 0; phase ^= 1u; }
        if constexpr (SEGK) {
#pragma unroll
          for (int j = 0; j < 4; ++j) tok[j] = tnx[j];
        }
      }
    }
    if (lane == 0) {
      pdl_trigger();   // no work item is left to hand out: the next kernel may be scheduled
      if (p.wait_stats)
        atomicAdd(p.wait_stats + ws_class(0, EPI, TWO_PHASE) * WS_FIELDS + WS_STAGE, (unsigned long long)ws_stage);
      if (!ok) {
        // Let the copies already issued land before the block exits.
        const int n = issued < S::STAGES ? issued : S::STAGES;
        for (int q = 1; q <= n; ++q) {
          int s = stage - q;
          uint32_t ph = phase;
          if (s < 0) { s += S::STAGES; ph ^= 1u; }
          volatile int no_abort = 0;
          wait_bounded(full_bar(s), ph, &no_abort, p.limit_ns, nullptr, 0);
        }
      }
    }
    __syncwarp();
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      long long ws_stage = 0;
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;  // stages issued (for the abort drain)
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int w = produce_next(it);
        if (w < 0) {
          ok = w == -1;
          break;
        }
        const Work wk = decode<SEGK>(p, w);
        if constexpr (EPI == EPI_DW) {
          // The epilogue will reduce-add this tile into the expert's fp32 gradient: start pulling the
          // old values into L2 now, while the tile's operands stream in, so the adds find them there.
          if (p.first_touch != nullptr && p.first_touch[wk.e] != p.chunk) {
            const CUtensorMap* om = wk.prob ? &to1 : &to0;
            const int n0 = wk.nt * BN, m0 = wk.mt * GEMM_BM;
            for (int rr = 0; rr < GEMM_BM && m0 + rr < p.M; rr += 32)
              for (int c = 0; c < BN && n0 + c < p.N; c += 32) tma_prefetch_3d(om, n0 + c, m0 + rr, wk.e);
          }
        }
        for (int kb = 0; kb < wk.nkb; ++kb) {
          const long long ws0 = ws_clock();
          const bool free_stage = wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.limit_ns, p.status, 101);
          ws_stage += ws_clock() - ws0;
          if (!free_stage) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_expect_tx(fb, S::STAGE_BYTES);
          const uint32_t sa = sbase + stage * S::STAGE_BYTES;
          const uint32_t sb = sa + S::A_BYTES;
          if constexpr (!SEGK) {
            const int ph = TWO_PHASE ? (kb >= p.nk ? 1 : 0) : 0;
            const int k0 = (kb - ph * p.nk) * GEMM_BK;
            const CUtensorMap* A = ph ? &ta1 : &ta0;
            const CUtensorMap* B = ph ? &tb1 : &tb0;
            tma_load_2d(sa, A, fb, k0, wk.row0);                       // A: K-major [128 rows][64 k]
            if constexpr (DUAL_B) {
              tma_load_3d(sb, &tb0, fb, k0, wk.nt * (BN / 2), wk.e);
              tma_load_3d(sb + S::B_BYTES / 2, &tb1, fb, k0, wk.nt * (BN / 2), wk.e);
            } else if constexpr (!B_MN) {
              tma_load_3d(sb, B, fb, k0, wk.nt * BN, wk.e);
            } else {
#pragma unroll
              for (int b = 0; b < BN / 64; ++b) tma_load_3d(sb + b * 8192, B, fb, wk.nt * BN + 64 * b, k0, wk.e);
            }
          } else {
            const int r0 = wk.row0 + kb * GEMM_BK;
            const CUtensorMap* A = wk.prob ? &ta1 : &ta0;
            const CUtensorMap* B = wk.prob ? &tb1 : &tb0;
#pragma unroll
            for (int a = 0; a < GEMM_BM / 64; ++a) tma_load_2d(sa + a * 8192, A, fb, wk.mt * GEMM_BM + 64 * a, r0);
#pragma unroll
            for (int b = 0; b < BN / 64; ++b) tma_load_2d(sb + b * 8192, B, fb, wk.nt * BN + 64 * b, r0);
          }
          ++issued;
          if (++stage == S::STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      pdl_trigger();   // no work item is left to hand out: the next kernel may be scheduled
      if (p.wait_stats)
        atomicAdd(p.wait_stats + ws_class(0, EPI, TWO_PHASE) * WS_FIELDS + WS_STAGE, (unsigned long long)ws_stage);
      if (!ok) {
        // Let the copies already issued land before the block exits.
        const int n = issued < S::STAGES ? issued : S::STAGES;
        for (int q = 1; q <= n; ++q) {
          int s = stage - q;
          uint32_t ph = phase;
          if (s < 0) { s += S::STAGES; ph ^= 1u; }
          volatile int no_abort = 0;
          wait_bounded(full_bar(s), ph, &no_abort, p.limit_ns, nullptr, 0);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = instr_desc_bf16(GEMM_BM, BN, A_MN, B_MN);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    const long long ws_start = ws_clock();
    long long ws_operands = 0, ws_accum = 0, ws_kblocks = 0;
    for (int it = 0; ok; ++it) {
      const int w = consume_next(it);
      if (w < 0) break;
      const Work wk = decode<SEGK>(p, w);
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      int good = 1;
      const long long ws0 = ws_clock();
      if (lane == 0) good = wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.limit_ns, p.status, 102);
      ws_accum += ws_clock() - ws0;
      ws_kblocks += wk.nkb;
      if (!__shfl_sync(0xffffffffu, good, 0)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tacc = tmem_base + acc * BN;
      for (int kb = 0; kb < wk.nkb; ++kb) {
        const long long ws1 = ws_clock();
        if (lane == 0) good = wait_bounded(full_bar(stage), phase, abort_flag, p.limit_ns, p.status, 103);
        ws_operands += ws_clock() - ws1;
        if (!__shfl_sync(0xffffffffu, good, 0)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sa = sbase + stage * S::STAGE_BYTES;
        const uint32_t sb = sa + S::A_BYTES;
        if constexpr (SEGK) {
          const int valid = wk.rows - kb * GEMM_BK;
          if (valid < GEMM_BK) {
            // zero K rows [valid, 64) of every 64-wide MN block of A and B
            const int nblk = GEMM_BM / 64 + BN / 64;
            const int bytes = (GEMM_BK - valid) * 128;
            for (int blk = 0; blk < nblk; ++blk) {
              uint8_t* base = smem + stage * S::STAGE_BYTES + blk * 8192 + valid * 128;
              for (int off = lane * 16; off < bytes; off += 32 * 16)
                *reinterpret_cast<uint4*>(base + off) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
        }
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < GEMM_BK / 16; ++kk) {
            const uint64_t ad = A_MN ? smem_desc_sw128(sa + kk * 2048, 8192, 1024)
                                     : smem_desc_sw128(sa + kk * 32, 0, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(sb + kk * 2048, 8192, 1024)
                                     : smem_desc_sw128(sb + kk * 32, 0, 1024);
            tc_mma(tacc, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(empty_bar(stage));
        }
        __syncwarp();
        if (++stage == S::STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(tfull_bar(acc));
      __syncwarp();
    }
    // Every MMA issued by this warp completes before TMEM is released.
    if (lane == 0) {
      tc_commit(drain_bar);
      volatile int no_abort = 0;
      wait_bounded(drain_bar, 0, &no_abort, p.limit_ns, nullptr, 0);
      if (p.wait_stats) {
        unsigned long long* c = p.wait_stats + ws_class(0, EPI, TWO_PHASE) * WS_FIELDS;
        atomicAdd(c + WS_CTAS, 1ull);
        atomicAdd(c + WS_LIFE, (unsigned long long)(ws_clock() - ws_start));
        atomicAdd(c + WS_OPERANDS, (unsigned long long)ws_operands);
        atomicAdd(c + WS_ACCUM, (unsigned long long)ws_accum);
        atomicAdd(c + WS_KBLOCKS, (unsigned long long)ws_kblocks);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                       // TMEM lane quarter this warp may access
    constexpr int NH = gemm_epi_warps(EPI) / 4;   // warps sharing a quarter; they split the column chunks
    const int half = (warp - 2) >> 2;
    const int r = q * 32 + lane;                  // row of the tile
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    int stg_count = 0;   // TMA store groups issued by this warp (EPI_DW)
    for (int it = 0;; ++it) {
      const int w = consume_next(it);
      if (w < 0) break;
      const Work wk = decode<SEGK>(p, w);
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      int good = 1;
      if (lane == 0) good = wait_bounded(tfull_bar(acc), acc_phase, abort_flag, p.limit_ns, p.status, 104);
      if (!__shfl_sync(0xffffffffu, good, 0)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + lane_off + acc * BN;

      if constexpr (EPI != EPI_DW && EPI != EPI_ACC) {
        epilogue_rows<EPI, BN>(p, wk.row0, wk.rows, wk.nt, wk.e, tacc, r, half);
      } else {
        float v[32];
        // fp32 weight gradient of expert e, rows [32q, 32q+32) of this tile: each 32 x 32 box goes
        // TMEM -> registers -> swizzled shared memory -> TMA store (the expert's first chunk in
        // backward order) or TMA reduce-add (later chunks; the add happens in L2, one add per
        // element per chunk, in chunk order).  Rows / columns past the matrix are clipped by TMA.
        // (EPI_ACC: the same for a row tile of a plain fp32 output, coordinate 0 of its third dimension,
        // stored on chunk 0 and added after.)
        const int n0 = wk.nt * BN;
        const int m0 = (EPI == EPI_ACC ? wk.row0 : wk.mt * GEMM_BM) + q * 32;
        const bool first = EPI == EPI_ACC ? p.chunk == 0
                                          : (p.first_touch == nullptr || p.first_touch[wk.e] == p.chunk);
        const CUtensorMap* om = wk.prob ? &to1 : &to0;
        uint8_t* stg = smem + S::STG_OFF + q * 8192;
        // a box whose first row is past the output (the last, partial tile) is not stored at all
        const bool rows_in = EPI == EPI_ACC ? q * 32 < wk.rows : m0 < p.M;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          if (n0 + c >= p.N || !rows_in) break;           // uniform across the warp
          tc_ld32(tacc + c, v);
          const int buf = stg_count & 1;
          if (lane == 0) bulk_wait_read<1>();             // the group that used this buffer has read it
          __syncwarp();
          uint8_t* row = stg + buf * 4096 + lane * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(row + ((j ^ (lane & 7)) << 4)) =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const uint32_t src = smem_u32(stg + buf * 4096);
            const int z = EPI == EPI_ACC ? 0 : wk.e;
            if (first) tma_store_3d(om, src, n0 + c, m0, z);
            else tma_reduce_add_3d(om, src, n0 + c, m0, z);
            bulk_commit();
          }
          ++stg_count;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
    }
    if constexpr (EPI == EPI_DW || EPI == EPI_ACC) {
      if (lane == 0) bulk_wait<0>();                      // stores complete before the block exits
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tc_dealloc(tmem_base, S::TMEM_COLS);
  if (p.pdl_late) pdl_wait();
}

}  // namespace moe
