// decode_tc.cu -- steps 4-5 of the layer for decode-sized batches (T <= 8) on
// the tensor cores, with the f32 GEMV's numerics: the weights enter as their
// exact int4 codes, f32 operands as two bf16 planes (hi, lo), every 64-K group
// accumulates into its own tensor-memory slice, and its f32 scale is applied
// in f32 afterwards (gs64: colibrì engine teardown, text-matrix.pages.dev,
// "Three key engineering decisions" (1)).
//
// At T = 1 a decode layer streams the activated experts' weights once, so the
// bound is HBM.  One tcgen05.mma issuer sustains about one M=128, K=16
// instruction per ~112 clocks, ~18 weights per clock per SM, while HBM-rate
// decode needs ~43; the CTA therefore runs four MMA pipelines, each with its
// own issuing thread and its own part of tensor memory.
//
//   super-unit (SU) = 128 weight rows x 256 K (four 64-K groups) of one expert;
//   stage           = one SU's int4 tile (128 rows x 128 bytes, 128-byte
//                     swizzle), its four 16-row bf16 operand tiles (the
//                     expert's token planes; rows past them are ignored MMA
//                     columns) and its 128 x 4 scales, brought by TMA; a ring
//                     of NS stages keeps DD SUs in flight per SM;
//   pipeline p      = 4 warps (thread r owns weight row r) on group p of every
//                     SU: decode the row's 64 codes into 32 columns of tensor
//                     memory (A), issue four K=16 MMAs (N = 16) into a 16-column
//                     slice, and one SU later read the slice back and add
//                     s_g * (D_hi + D_lo) per token in f32.
// Roles: 16 decode warps (4 per pipeline: decode into A, then the epilogue),
// one MMA-issuing warp per pipeline (an issuing thread stalls for the ~450
// clocks its four MMAs take, so it must not be a decode thread), and one TMA
// producer warp.  They hand over through mbarriers only: stage full (TMA),
// A full (4 decode warps), MMAs done (commit), stage empty (16 decode warps).
//
// The CTAs split the flat SU range evenly (split-K: a row block's SUs may span
// CTAs).  Each pipeline stores its sums for every row block it touched; after
// the main loop the row blocks are finished: by this CTA alone, or, when
// several CTAs share one, by the last of them to arrive (an atomic ticket),
// which adds all partial sums in (CTA, pipeline) order -- the result does not
// depend on timing.  W13: SwiGLU into h planes; W2: times the routing weight
// into y.  Every mbarrier wait is bounded by %globaltimer; a role that gives
// up sets the CTA's abort flag and leaves its loop, the others follow at their
// next wait, and the CTA drains its copies and MMAs and frees tensor memory.
#include <algorithm>
#include <cuda.h>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int DP = kDecPipes;         // MMA pipelines per CTA
constexpr int kDecWarps = DP * 4;     // decode + epilogue warps (4 per pipeline)
constexpr int kIssWarp0 = kDecWarps;  // MMA issuer warps (one per pipeline)
constexpr int kProdWarp = kIssWarp0 + DP;   // TMA producer warp
constexpr int DT = (kProdWarp + 1) * 32;    // threads per CTA
constexpr int DD = 5;                 // SUs loaded ahead
constexpr int NS = DD + 2;            // stages
constexpr int kWTile = 128 * 128;     // 128 rows x 256 int4 codes
constexpr int kBTile = 16 * 128;      // 16 operand rows x 64 bf16
constexpr int kSTile = 128 * 4 * 4;   // 128 rows x 4 f32 scales
constexpr uint32_t kStageTx = kWTile + DP * kBTile + kSTile;
constexpr uint32_t kTmemPerPipe = 128;   // columns: 2 A buffers x 32, 2 slices x 16
constexpr uint32_t kSliceCol = 64;

struct __align__(1024) DecStage {
  uint8_t w[kWTile];          // 128-byte swizzle: 1024-byte aligned
  uint8_t b[DP][kBTile];
  float sc[128 * 4];
};
static_assert(sizeof(DecStage) % 1024 == 0, "stage alignment");

struct __align__(1024) SmemDec {
  DecStage st[NS];
  uint64_t full[NS];                // a stage landed
  uint64_t empty[NS];               // all decode warps are done with a stage
  uint64_t afull[DP][2];            // a pipeline's A buffer is written (4 warps)
  uint64_t done[DP][2];             // a pipeline's MMAs of an SU completed
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kDecSmem = sizeof(SmemDec) + 1024;
static_assert(kDecSmem <= 227 * 1024, "shared memory");
static_assert(DP * kTmemPerPipe <= 512, "TMEM columns");
static_assert(DP == 4, "an SU holds one 64-K group per pipeline");

struct DecParams {
  CUtensorMap map_w;       // routed weights [E * rows][K / 2] u8, box 128 x 128, swizzled
  CUtensorMap map_ws;      // shared expert [rows_s][K_s / 2] u8
  CUtensorMap map_s;       // routed scales [E * rows][K / 64] f32, box 4 x 128
  CUtensorMap map_ss;      // shared scales [rows_s][K_s / 64] f32
  CUtensorMap map_b;       // operand planes [R][Kmax] bf16, box 64 x 16, swizzled
  int mode;                // 0: W13 + SwiGLU, 1: W2 x routing weight
  int E, A, T, S;
  int rows, rows_s;        // weight rows of a routed expert / of the shared expert
  int K, K_s;
  const int32_t *active;   // ascending active experts, the shared expert (E) last
  const int32_t *n_active;
  const int32_t *offsets;  // [E+1]
  float *partial;          // [CTA + row block][pipeline][128][kDecTokens]
  int32_t *ticket;         // [n_rb] this launch's arrival counters
  int32_t *ticket_other;   // the other matrix's counters, cleared here
  int n_ticket_other;
  __nv_bfloat16 *he;       // W13 out: planes [2 R][h_stride]
  int h_stride;
  float *y;                // W2 out [R][H]
  int H;
  const float *wperm;      // [R]
  int32_t *status;
  L2Prefetch pf;           // W2: the next layer's router and shared expert
  unsigned long long wait_ns;   // limit of each role wait (MOE_OPT_WAIT_LIMIT_US)
};

// The grid's flat SU range: routed experts (slot a < n_r) first, then the
// shared expert; inside an expert, row block-major.
struct Geo {
  int n_r, RB, G4, RBs, G4s, P;
  long long U_r, U;
  __device__ long long start(int i) const { return (long long)i * U / P; }
  // The CTA whose range holds SU u.
  __device__ int cta_of(long long u) const { return (int)(((u + 1) * P + U - 1) / U) - 1; }
};

struct Cur {
  int a, rb, s;       // expert slot (n_r: the shared expert), row block, SU in the row block
  int e, wbase, p0;   // the slot's expert, its first weight row, its first grouped row
};

// The slot's expert and rows: read once per expert, not once per SU.
__device__ __forceinline__ void load_slot(const DecParams &p, const Geo &q, Cur &c) {
  if (c.a >= q.n_r) {
    c.e = p.E;
    c.wbase = 0;
    c.p0 = p.A;
  } else {
    c.e = __ldcg(p.active + c.a);
    c.wbase = c.e * p.rows;
    c.p0 = __ldcg(p.offsets + c.e);
  }
}

__device__ __forceinline__ Cur cur_at(const DecParams &p, const Geo &q, long long u) {
  Cur c;
  if (u < q.U_r) {
    const long long per = (long long)q.RB * q.G4;
    c.a = (int)(u / per);
    const long long rem = u - (long long)c.a * per;
    c.rb = (int)(rem / q.G4);
    c.s = (int)(rem - (long long)c.rb * q.G4);
  } else {
    const long long rem = u - q.U_r;
    c.a = q.n_r;
    c.rb = (int)(rem / q.G4s);
    c.s = (int)(rem - (long long)c.rb * q.G4s);
  }
  load_slot(p, q, c);
  return c;
}

// Advances to the next SU; `reload` false skips the slot lookup on a change
// of expert (for a cursor that has reached the end of its range).
__device__ __forceinline__ void cur_next(const DecParams &p, const Geo &q, Cur &c,
                                         bool reload = true) {
  const bool sh = c.a >= q.n_r;
  if (++c.s == (sh ? q.G4s : q.G4)) {
    c.s = 0;
    if (++c.rb == (sh ? q.RBs : q.RB)) {
      c.rb = 0;
      ++c.a;
      if (reload && c.a <= q.n_r) load_slot(p, q, c);
    }
  }
}

// First SU of the cursor's row block (U past the last one).
__device__ __forceinline__ long long rb_start(const Geo &q, const Cur &c) {
  if (c.a < q.n_r) return ((long long)c.a * q.RB + c.rb) * q.G4;
  if (c.a == q.n_r) return q.U_r + (long long)c.rb * q.G4s;
  return q.U;
}

__device__ __forceinline__ int rb_index(const Geo &q, const Cur &c) {
  return c.a < q.n_r ? c.a * q.RB + c.rb : q.n_r * q.RB + c.rb;
}

__device__ __forceinline__ bool bar_vote_or(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id)
      : "memory");
  return r != 0;
}

// TMA for SU c into stage `stage`: the int4 tile, the four operand tiles and
// the scales.  Weights and scales are read once per pass: they enter L2 as
// evict-first (policy pol), so the split-K partial sums written during the
// pass are still in L2 when the row blocks are finished.
template <int PL>
__device__ __forceinline__ void issue_su(const DecParams &p, const Geo &q, SmemDec *sm, int stage,
                                         const Cur &c, uint64_t pol) {
  const bool sh = c.a >= q.n_r;
  const int wrow0 = c.wbase + c.rb * 128;
  DecStage &st = sm->st[stage];
  uint64_t *bar = &sm->full[stage];
  mbar_expect_tx(bar, kStageTx);
  tma_load_2d_hint(st.w, sh ? &p.map_ws : &p.map_w, c.s * 128, wrow0, bar, pol);
#pragma unroll
  for (int g = 0; g < DP; ++g) tma_load_2d(st.b[g], &p.map_b, (c.s * 4 + g) * 64, PL * c.p0, bar);
  tma_load_2d_hint(st.sc, sh ? &p.map_ss : &p.map_s, c.s * 4, wrow0, bar, pol);
}

__device__ __forceinline__ float *partial_row(const DecParams &p, int cta, int rbi, int pipe,
                                              int r) {
  return p.partial + (((size_t)(cta + rbi) * DP + pipe) * 128 + r) * kDecTokens;
}

// Finishes row block c (pipeline pp's 128 threads, after the CTA's partial
// sums are all stored).
template <int NT>
__device__ void finish_rb(const DecParams &p, const Geo &q, int pp, const Cur &c) {
  const int r = threadIdx.x & 127, lane = threadIdx.x & 31;
  const bool sh = c.a >= q.n_r;
  const int rbi = rb_index(q, c);
  const long long us = rb_start(q, c);
  const int f0 = q.cta_of(us), f1 = q.cta_of(us + (sh ? q.G4s : q.G4) - 1);
  if (f0 != f1) {
    bool last = false;
    if (r == 0) {
      const int old = atomicAdd(p.ticket + rbi, 1);
      last = (old == f1 - f0);
      if (last) p.ticket[rbi] = 0;
    }
    if (!bar_vote_or(1 + pp, last)) return;
    __threadfence();
  }
  float tot[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) tot[t] = 0.f;
  for (int f = f0; f <= f1; ++f) {   // (CTA, pipeline) order: the same sum every run
#pragma unroll
    for (int g = 0; g < DP; ++g) {
      const float *src = partial_row(p, f, rbi, g, r);
#pragma unroll
      for (int t = 0; t < NT; ++t) tot[t] += __ldcg(src + t);
    }
  }
  const int cnt = sh ? p.T : __ldcg(p.offsets + c.e + 1) - c.p0;
  if (p.mode == 0) {
    // Rows of the block: quadrant qd holds the W1 rows of features rb*64 +
    // 16 qd + (lane & 15) in lanes 0-15 and the W3 rows of the same in 16-31.
    const int feat = c.rb * 64 + (r >> 5) * 16 + (lane & 15);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float u = __shfl_xor_sync(0xffffffffu, tot[t], 16);
      if (lane < 16 && t < cnt) {
        const float hval = tot[t] / (1.0f + expf(-tot[t])) * u;
        const __nv_bfloat16 hi = __float2bfloat16_rn(hval);
        const __nv_bfloat16 lo = __float2bfloat16_rn(hval - __bfloat162float(hi));
        const size_t r2 = 2 * (size_t)(c.p0 + t);
        p.he[r2 * p.h_stride + feat] = hi;
        p.he[(r2 + 1) * p.h_stride + feat] = lo;
      }
    }
  } else {
    const int o = c.rb * 128 + r;
#pragma unroll
    for (int t = 0; t < NT; ++t)
      if (t < cnt) p.y[(size_t)(c.p0 + t) * p.H + o] = tot[t] * __ldcg(p.wperm + c.p0 + t);
  }
}

// NT: tokens per expert handled (a power of two >= T); PL: operand planes per
// token (1: bf16 x; 2: hi/lo planes of f32 x or of h).
// kShortWaits: the instantiation launched when the caller set a wait limit
// below the default (MOE_OPT_WAIT_LIMIT_US); the ordinary one never tests it.
template <int NT, int PL, bool kShortWaits>
__global__ void __launch_bounds__(DT, 1) decode_tc_kernel(const __grid_constant__ DecParams p) {
  if (p.mode == 1) l2_prefetch_share(p.pf);   // init-time weights: no wait needed
  pdl_enter();
  constexpr int NC = NT * PL;                 // accumulator columns read back
  static_assert(NC <= 16, "16 MMA columns");
  extern __shared__ uint8_t smem_raw[];
  SmemDec *sm = reinterpret_cast<SmemDec *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // The other matrix's arrival counters are idle now (stream order): clear them.
  for (int i = blockIdx.x * DT + threadIdx.x; i < p.n_ticket_other; i += gridDim.x * DT)
    p.ticket_other[i] = 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&sm->full[i], 1);
      mbar_init(&sm->empty[i], kDecWarps);
    }
    for (int k = 0; k < DP; ++k)
      for (int i = 0; i < 2; ++i) {
        mbar_init(&sm->afull[k][i], 4);
        mbar_init(&sm->done[k][i], 1);
      }
    sm->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(&sm->tmem_base))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  Geo q;
  q.n_r = __ldcg(p.n_active) - p.S;
  q.RB = p.rows / 128;
  q.G4 = p.K / 256;
  q.RBs = p.rows_s / 128;
  q.G4s = p.K_s / 256;
  q.U_r = (long long)q.n_r * q.RB * q.G4;
  q.U = q.U_r + (long long)p.S * q.RBs * q.G4s;
  q.P = (int)min((long long)gridDim.x, q.U);   // CTAs with work: one SU at least each
  const long long u0 = (int)blockIdx.x < q.P ? q.start(blockIdx.x) : 0;
  const long long u1 = (int)blockIdx.x < q.P ? q.start(blockIdx.x + 1) : 0;
  const uint32_t n = (uint32_t)(u1 - u0);
  bool fail = false;

  if (n > 0 && warp == kProdWarp) {
    // ------------------------------------------------------ TMA producer
    Cur cp = cur_at(p, q, u0);
    const uint64_t pol = l2_evict_first_policy();
    uint32_t jp = 0;
    for (; jp < n; ++jp) {
      // SU jp goes into the stage SU jp - NS used, once all decode warps released it.
      const int stage = (int)(jp % NS);
      if (jp >= (uint32_t)NS &&
          !wait_role<kShortWaits>(&sm->empty[stage], ((jp / NS) & 1) ^ 1, &sm->abort, p.status, p.wait_ns)) {
        fail = true;
        break;
      }
      fence_proxy_async();
      if (elect_one()) issue_su<PL>(p, q, sm, stage, cp, pol);
      __syncwarp();
      cur_next(p, q, cp, jp + 1 < n);
    }
    const unsigned long long t0 = globaltimer();
    for (uint32_t k = (jp > (uint32_t)NS ? jp - NS : 0); k < jp; ++k)
      drain_bar(&sm->full[k % NS], (k / NS) & 1, t0);
  } else if (n > 0 && warp >= kIssWarp0) {
    // ------------------------------------------------------ MMA issuer of pipeline pp
    const int pp = warp - kIssWarp0;
    const uint32_t tmem = sm->tmem_base + pp * kTmemPerPipe;
    const uint32_t idesc = idesc_bf16(128, 16);
    uint32_t j = 0;
    for (; j < n; ++j) {
      const int stage = (int)(j % NS);
      if (!wait_role<kShortWaits>(&sm->afull[pp][j & 1], (j >> 1) & 1, &sm->abort, p.status, p.wait_ns) ||
          !wait_role<kShortWaits>(&sm->full[stage], (j / NS) & 1, &sm->abort, p.status, p.wait_ns)) {
        fail = true;
        break;
      }
      tc_fence_after();
      if (elect_one()) {
        mma_kblock_ta(tmem + kSliceCol + (j & 1) * 16, tmem + (j & 1) * 32,
                      sw128_desc(smem_u32(sm->st[stage].b[pp])), idesc, 0u);
        mma_commit(&sm->done[pp][j & 1]);
      }
      __syncwarp();
    }
    if (j > 0) drain_bar(&sm->done[pp][(j - 1) & 1], ((j - 1) >> 1) & 1, globaltimer());
  } else if (n > 0) {
    // ------------------------------------------------------ decode + epilogue
    const int pp = warp >> 2;                   // pipeline = 64-K group of each SU
    const int r = threadIdx.x & 127;            // weight row of the tile = TMEM lane
    const uint32_t tmem = sm->tmem_base + pp * kTmemPerPipe;
    const uint32_t lane_addr = (uint32_t)((r >> 5) * 32) << 16;
    Cur ce = cur_at(p, q, u0);                  // epilogue cursor (one SU behind)
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.f;
    for (uint32_t j = 0; j <= n; ++j) {
      if (j < n) {
        // This pipeline's 64 codes of row r (16-byte chunks 2 pp and 2 pp + 1
        // of the swizzled row) into 32 columns of A buffer j & 1; the MMAs
        // that read that buffer two SUs ago are complete (the epilogue of SU
        // j - 2 waited for them).
        const int stage = (int)(j % NS);
        bool go = wait_role<kShortWaits>(&sm->full[stage], (j / NS) & 1, &sm->abort, p.status, p.wait_ns);
        go = __all_sync(0xffffffffu, go);     // tcgen05.st is warp-collective
        if (!go) {
          fail = true;
          break;
        }
        const uint8_t *row = sm->st[stage].w + r * 128;
        const uint4 c0 = *reinterpret_cast<const uint4 *>(row + (((2 * pp) ^ (r & 7)) << 4));
        const uint4 c1 = *reinterpret_cast<const uint4 *>(row + (((2 * pp + 1) ^ (r & 7)) << 4));
        uint32_t o[32];
        dequant_word_q(c0.x, o + 0);
        dequant_word_q(c0.y, o + 4);
        dequant_word_q(c0.z, o + 8);
        dequant_word_q(c0.w, o + 12);
        dequant_word_q(c1.x, o + 16);
        dequant_word_q(c1.y, o + 20);
        dequant_word_q(c1.z, o + 24);
        dequant_word_q(c1.w, o + 28);
        tmem_st32(tmem + lane_addr + (j & 1) * 32, o);   // includes the wait
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->afull[pp][j & 1]);
      }
      if (j > 0) {
        // Epilogue of SU j - 1.
        const uint32_t jm = j - 1;
        const int stage = (int)(jm % NS);
        bool ok = wait_role<kShortWaits>(&sm->done[pp][jm & 1], (jm >> 1) & 1, &sm->abort, p.status, p.wait_ns);
        ok = __all_sync(0xffffffffu, ok);     // tcgen05.ld is warp-collective
        if (!ok) {
          fail = true;
          break;
        }
        tc_fence_after();
        float v[NC];
        if constexpr (NC == 16) tmem_ld16(tmem + lane_addr + kSliceCol + (jm & 1) * 16, v);
        else tmem_ld_n<NC>(tmem + lane_addr + kSliceCol + (jm & 1) * 16, v);
        tc_fence_before();
        const float s = sm->st[stage].sc[r * 4 + pp];
#pragma unroll
        for (int t = 0; t < NT; ++t)
          acc[t] = fmaf(s, PL == 2 ? v[2 * t] + v[2 * t + 1] : v[t], acc[t]);
        fence_proxy_async();   // the stage's reads before its TMA refill
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->empty[stage]);
        Cur nx = ce;
        cur_next(p, q, nx, j < n);
        if (j == n || nx.rb != ce.rb || nx.a != ce.a) {
          // This pipeline's sums over its groups of the row block.
          float *dst = partial_row(p, blockIdx.x, rb_index(q, ce), pp, r);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            dst[t] = acc[t];
            acc[t] = 0.f;
          }
        }
        ce = nx;
      }
    }
  }
  __threadfence();
  const bool any_fail = __syncthreads_or(fail || *reinterpret_cast<volatile int *>(&sm->abort));
  if (n > 0 && !any_fail && warp < kDecWarps) {
    // Finish the row blocks of this CTA's range, one pipeline per row block.
    const int pp = warp >> 2;
    Cur c = cur_at(p, q, u0);
    c.s = 0;
    for (int k = 0; rb_start(q, c) < u1; ++k) {
      if ((k & (DP - 1)) == pp) finish_rb<NT>(p, q, pp, c);
      const bool sh = c.a >= q.n_r;
      if (++c.rb == (sh ? q.RBs : q.RB)) {
        c.rb = 0;
        ++c.a;
        if (c.a <= q.n_r) load_slot(p, q, c);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(sm->tmem_base)
                 : "memory");
  }
}

template <int PL>
cudaError_t launch_pass(const DecParams &p, int T, int grid, bool pdl, cudaStream_t st) {
  cudaError_t err = cudaSuccess;
#define MOE_DEC(NT)                                                                          \
  do {                                                                                       \
    static bool attr = false;                                                                \
    if (!attr) {                                                                             \
      cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<NT, PL, false>,                  \
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,      \
                                           (int)kDecSmem);                                   \
      if (e == cudaSuccess)                                                                  \
        e = cudaFuncSetAttribute(decode_tc_kernel<NT, PL, true>,                             \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecSmem); \
      if (e != cudaSuccess) return e;                                                        \
      attr = true;                                                                           \
    }                                                                                        \
    err = launch_k(pdl, p.wait_ns < kWaitNs ? decode_tc_kernel<NT, PL, true>                  \
                                            : decode_tc_kernel<NT, PL, false>,               \
                   dim3(grid), dim3(DT), kDecSmem, st, p);                                   \
  } while (0)
  if (T <= 1) MOE_DEC(1);
  else if (T <= 2) MOE_DEC(2);
  else if (T <= 4) MOE_DEC(4);
  else MOE_DEC(8);
#undef MOE_DEC
  return err;
}

}  // namespace

cudaError_t launch_decode_tc(const moe_handle *h, const void *x, int T, float *out,
                             bool accumulate, cudaStream_t st) {
  const moe::Workspace &w = h->ws;
  const int E = h->E, H = h->H, I = h->I, k = h->k, S = h->S;
  const int Is = S ? h->Is : I;
  const int h_stride = I > Is ? I : Is;
  const int rows_x = kExactTokens * (k + S);
  if (T > kExactTokens) return cudaErrorInvalidValue;
  moe_handle *hm = const_cast<moe_handle *>(h);
  cudaError_t err = launch_gather_exact(h, x, T, st);
  if (err != cudaSuccess) return err;
  hm->launches += 1;
  if (h->profile && hm->n_ev <= moe_handle::kMaxStages) {
    hm->stage_names[hm->n_ev - 1] = "gather";
    cudaEventRecord(hm->ev[hm->n_ev++], st);
  }
  const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapDataType F32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  DecParams p{};
  const int xplanes = h->L.x_dtype == 1 ? 1 : 2;
  p.E = E;
  p.A = T * k;
  p.T = T;
  p.S = S;
  p.active = w.active;
  p.n_active = w.n_active;
  p.offsets = w.offsets;
  p.partial = w.dec_partial;
  p.he = w.he;
  p.h_stride = h_stride;
  p.y = w.y;
  p.H = H;
  p.wperm = w.wperm;
  p.status = w.status;
  p.wait_ns = h->wait_ns;
  // ---- W13 over the x planes
  bool ok = make_map(&p.map_w, h->ex.w13q, U8, 1, H / 2, (uint64_t)E * 2 * I, H / 2, 128, 128);
  ok = ok && make_map(&p.map_ws, S ? h->sh.w13q : h->ex.w13q, U8, 1, H / 2,
                      (uint64_t)2 * Is, H / 2, 128, 128);
  ok = ok && make_map(&p.map_s, h->ex.w13s, F32, 4, H / 64, (uint64_t)E * 2 * I, H / 64, 4, 128,
                      false);
  ok = ok && make_map(&p.map_ss, S ? h->sh.w13s : h->ex.w13s, F32, 4, H / 64, (uint64_t)2 * Is,
                      H / 64, 4, 128, false);
  ok = ok && make_map(&p.map_b, w.xe, BF, 2, H, (uint64_t)2 * rows_x, H, 64, 16);
  if (!ok) return cudaErrorInvalidValue;
  p.mode = 0;
  p.rows = 2 * I;
  p.rows_s = 2 * Is;
  p.K = H;
  p.K_s = H;
  p.ticket = w.dec_ticket;
  p.ticket_other = w.dec_ticket + h->dec_rb_max;
  p.n_ticket_other = h->dec_rb_max;
  err = xplanes == 1 ? launch_pass<1>(p, T, h->num_sms, h->pdl, st)
                     : launch_pass<2>(p, T, h->num_sms, h->pdl, st);
  if (err != cudaSuccess) return err;
  hm->launches += 1;
  if (h->profile && hm->n_ev <= moe_handle::kMaxStages) {
    hm->stage_names[hm->n_ev - 1] = "w13";
    cudaEventRecord(hm->ev[hm->n_ev++], st);
  }
  // ---- W2 over the h planes
  ok = make_map(&p.map_w, h->ex.w2q, U8, 1, I / 2, (uint64_t)E * H, I / 2, 128, 128);
  ok = ok && make_map(&p.map_ws, S ? h->sh.w2q : h->ex.w2q, U8, 1, Is / 2, (uint64_t)H, Is / 2, 128,
                      128);
  ok = ok && make_map(&p.map_s, h->ex.w2s, F32, 4, I / 64, (uint64_t)E * H, I / 64, 4, 128, false);
  ok = ok && make_map(&p.map_ss, S ? h->sh.w2s : h->ex.w2s, F32, 4, Is / 64, (uint64_t)H, Is / 64,
                      4, 128, false);
  ok = ok && make_map(&p.map_b, w.he, BF, 2, h_stride, (uint64_t)2 * rows_x, h_stride, 64, 16);
  if (!ok) return cudaErrorInvalidValue;
  p.mode = 1;
  p.rows = H;
  p.rows_s = H;
  p.K = I;
  p.K_s = Is;
  p.ticket = w.dec_ticket + h->dec_rb_max;
  p.ticket_other = w.dec_ticket;
  p.pf = next_layer_prefetch(h);
  err = launch_pass<2>(p, T, h->num_sms, h->pdl, st);
  if (err != cudaSuccess) return err;
  hm->launches += 1;
  if (h->profile && hm->n_ev <= moe_handle::kMaxStages) {
    hm->stage_names[hm->n_ev - 1] = "w2";
    cudaEventRecord(hm->ev[hm->n_ev++], st);
  }
  err = launch_combine(h, T, out, accumulate, st);
  hm->launches += 1;
  if (h->profile && hm->n_ev <= moe_handle::kMaxStages) {
    hm->stage_names[hm->n_ev - 1] = "combine";
    cudaEventRecord(hm->ev[hm->n_ev++], st);
  }
  return err;
}

}  // namespace moe
