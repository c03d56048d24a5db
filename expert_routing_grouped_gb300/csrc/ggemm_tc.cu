// ggemm_tc.cu -- steps 4-5 of the layer for large T (prefill) on the 5th-gen
// tensor cores: grouped GEMMs over the experts' token groups.
//
// Only this regime is a dense contraction: per expert, a group of tokens times
// its int4 weights (the pages' per-expert mini-batch GEMM -- pure-C Colibri
// tutorial, trdm.cn, §2.2 "third"; Colibri C + cuBLASLt tutorial, cf-1.com,
// §3.3 Step 4, one GEMM per non-empty expert).  Here every expert, token
// block and weight-row block is one tile of ONE persistent kernel per matrix:
//
//   ggemm_w13:  D[128 weight rows][N tokens] = W13_tile . x_grouped^T, the 128
//               rows being 64 features' W1 and W3 rows interleaved by 16, so
//               SwiGLU h = silu(g) * u pairs lanes l and l+16 of one warp;
//               h is written as fp16 in grouped order.
//   ggemm_w2:   D[128 output rows][N tokens] = W2_tile . h^T; the epilogue
//               scales each token's column by its routing weight and writes
//               y[grouped row][o] in f32.
//
// Operands are fp16 (11 significant bits; the same tensor-core rate as bf16)
// with f32 accumulation, and every quantity is brought into fp16's range by
// exact powers of two that the epilogues take out again:
//   x       per token: fp16(x * 2^ex) with |x * 2^ex| < 2^14 (exact for bf16 x);
//   weights per row:   fp16(q * fp16(s * 2^pw)) with the row's largest scale
//                      times 2^pw in [2^7, 2^8), so |w| < 2^11;
//   h       per token: fp16(h * 2^fh) with 2^fh from a bound on |h| that
//                      cannot be exceeded: |g_i| <= |W1_i| |x| (Cauchy-Schwarz,
//                      Euclidean norms), |silu(g)| <= max(|g|, 0.279), so
//                      |h| <= max(N1 |x|, 0.279) N3 |x| with N1, N3 the largest
//                      W1 / W3 row norms -- then |h * 2^fh| < 2^14.
// The bound may be loose by a few powers of two; that only moves small
// elements of h toward fp16's subnormal range, where their absolute error
// (2^-24 * 2^-fh) stays far below the rounding of the large ones.
//
// Per CTA (one per SM, 16 warps):
//   warp 0      TMA producer of raw int4 weight tiles (128 rows x 256 K, 128-byte
//               swizzled) and their gs64 scales, 4 stages deep;
//   warp 2      TMA producer of fp16 token tiles (up to 160 rows x 64 K, 128-byte
//               swizzled, several K blocks per 40 KB slot); the two producers
//               run independently.
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma kind::f16 (fp16 in,
//               f32 accumulate) M=128, N=16..160, K=16 by one elected lane
//               (the warp runs the loop, so operands stay uniform), commits
//               to mbarriers.  A is read from TMEM, B from shared memory.
//   warps 4-7   epilogue: tcgen05.ld of their TMEM lane quadrant.
//   warps 8-15  dequant: raw int4 -> fp16(q * s * 2^pw), written straight into TMEM
//               as the MMA's A operand with tcgen05.st (a warp owns one lane
//               quadrant and half of each 64-K block: one row, 32 K per thread).
// TMEM (512 columns): two 160-column accumulators, so the epilogue of one tile
// overlaps the main loop of the next, and two 64-column A groups (2 K blocks
// of 64 each), so the dequant of one group overlaps the MMAs of the other.
// One issuing thread keeps the tensor pipe full for N >= 128 (an M=128, K=16
// MMA takes N/2 clocks there; below N = 128 about 59 clocks whatever N), so
// the tile is as wide as TMEM allows while both accumulators fit.  The MMAs
// are not what sets this kernel's pace: the dequant warps and the weight
// stream are (a 128 x 64 weight block takes ~350 clocks to arrive and
// decode against ~320 clocks of MMAs at N = 160).
// Keeping A out of shared memory leaves shared-memory bandwidth to the token
// operand: per 64-K block the MMA reads N x 128 bytes of tokens that TMA wrote,
// and nothing else but the 4.5 KB raw stage passes through it.
// Every mbarrier wait is bounded by %globaltimer: a wait that gives up sets
// the device status word, flags the CTA to stop, and the kernel drains its
// outstanding copies and MMAs (bounded), frees TMEM and returns.
#include <algorithm>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "tc.cuh"

namespace moe {
namespace {

constexpr int BM = 128;          // weight rows per tile (MMA M)
constexpr int BN = kTileTokens;  // tokens per tile (MMA N, max)
constexpr int BK = 64;           // K per bf16 block (128 bytes of a row)
constexpr int RK = 256;          // K per raw int4 stage (128 bytes of a row)
constexpr int KPG = 2;           // K blocks per A group (TMEM handoff unit)
constexpr int GPS = RK / BK / KPG;  // A groups per raw stage
constexpr int NG = 2;            // A groups in TMEM
constexpr int NB = 3;            // token slots
constexpr int NR = 4;            // raw stages
constexpr int kSlotRows = 320;   // rows of 128 bytes per token slot (40 KB)
constexpr uint32_t kACol0 = 2 * BN;            // first TMEM column of the A groups
constexpr uint32_t kGroupCols = KPG * BK / 2;  // 64 columns: 2 fp16 per column
constexpr int kThreads = 512;
constexpr int kEpiWarp0 = 4;
constexpr int kDeqWarp0 = 8;
constexpr int kDeqWarps = 8;
static_assert(kACol0 + NG * kGroupCols <= 512, "TMEM columns");

struct __align__(1024) SmemTC {
  uint8_t raw[NR][BM * 128];     // 4 x 16 KB
  uint8_t b[NB][kSlotRows * 128];  // 3 x 40 KB
  float sc[NR][BM * (RK / 64)];  // 4 x 2 KB: the raw stage's gs64 scales, [row][4]
  uint64_t raw_full[NR], raw_empty[NR];
  uint64_t a_full[NG], a_empty[NG];
  uint64_t b_full[NB], b_empty[NB];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;                // the MMA warp's last commit, before TMEM is freed
  uint32_t tmem_base;
  int abort;
};

// Token boxes of 32, 64, 96 or 160 rows (the smallest that covers the tile's
// operand rows); a 40 KB slot carries 8, 4, 2 or 2 K blocks of one box, so
// small tiles keep more K blocks in flight (the counts are powers of two: K / 64
// is a multiple of 8).
constexpr int kBoxRows[4] = {32, 64, 96, BN};
static_assert(BN == 160, "the largest token box is one tile");
__device__ __forceinline__ int box_index(int nvalid) {
  return nvalid <= 32 ? 0 : nvalid <= 64 ? 1 : nvalid <= 96 ? 2 : 3;
}
__device__ __forceinline__ int box_rows(int bi) { return bi == 0 ? 32 : bi == 1 ? 64 : bi == 2 ? 96 : BN; }
__device__ __forceinline__ int box_kps(int bi) { return bi == 0 ? 8 : bi == 1 ? 4 : 2; }

struct TcParams {
  CUtensorMap map_w;       // raw weights of the routed experts [E * rows][K/2] u8
  CUtensorMap map_ws;      // raw weights of the shared expert [rows_s][K/2] u8
  CUtensorMap map_sc;      // scales of the routed experts [E * rows][K/64] f32
  CUtensorMap map_scs;     // scales of the shared expert [rows_s][K/64] f32
  CUtensorMap map_b[4];    // fp16 token operand [R][K], boxes of 32/64/96/160 rows
  int mode;                // 0: W13 + SwiGLU, 1: W2 + routing weight
  int K;                   // reduction length (H for W13, I for W2)
  int K_s;                 // the shared expert's reduction length (H, or Is for W2)
  int rows;                // weight rows per routed expert (2I or H)
  int rows_s;              // weight rows of the shared expert (2Is or H)
  int E, A, T;
  const int32_t *blocks;   // token blocks (expert << 16 | block index)
  const int32_t *n_blocks;
  const int32_t *offsets;  // [E+1]
  const float *rexp;       // per weight row 2^pw of the routed experts [E * rows]
  const float *rexp_s;     // per weight row 2^pw of the shared expert [rows_s]
  __half *hb;              // W13 output [R][h_stride]: fp16(h * 2^fh)
  int h_stride;
  float *y;                // W2 output [R][H]
  int H;
  const float *wperm;      // [R] routing weight times 2^-fh (W2 epilogue)
  const float *xcol;       // [R] 2^-ex of the row's token (W13 epilogue)
  const float *hcol;       // [R] 2^fh of the row's token (W13 epilogue)
  int32_t *status;
  unsigned long long wait_ns;   // limit of each role wait (MOE_OPT_WAIT_LIMIT_US)
};

// --------------------------------------------------------------- PTX glue --
// (mbarrier, TMA and elect helpers: ptx.cuh; tcgen05 descriptors, MMA issue,
// tensor-memory loads and stores and the int4 decodes: tc.cuh)

template <bool kShortWaits>
__device__ __forceinline__ bool wait_tc(uint64_t *bar, uint32_t parity, SmemTC *sm,
                                        const TcParams &p) {
  return moe::wait_role<kShortWaits>(bar, parity, &sm->abort, p.status, p.wait_ns);
}

// --------------------------------------------------------------- tiles --

struct Tile {
  int e, p0, nvalid, wrow0, shared, K;
};

__device__ __forceinline__ bool tile_at(const TcParams &p, int t, int n_fb, int n_blocks, Tile &tl) {
  const int blk = t / n_fb, fb = t - blk * n_fb;
  if (blk >= n_blocks) return false;
  const int packed = p.blocks[blk];
  const int e = packed >> 16, tb = packed & 0xFFFF;
  tl.e = e;
  tl.shared = (e >= p.E);
  int cnt;
  if (!tl.shared) {
    const int o0 = p.offsets[e];
    cnt = p.offsets[e + 1] - o0;
    tl.p0 = o0 + tb * BN;
    tl.wrow0 = e * p.rows + fb * BM;
    tl.K = p.K;
  } else {
    cnt = p.T;
    tl.p0 = p.A + tb * BN;
    tl.wrow0 = fb * BM;
    tl.K = p.K_s;
  }
  tl.nvalid = min(BN, cnt - tb * BN);
  // Row blocks past the expert's rows (the routed and the shared expert may
  // differ in size) have no work.
  if (fb * BM >= (tl.shared ? p.rows_s : p.rows)) tl.nvalid = 0;
  return true;
}

// --------------------------------------------------------------- kernel --
//
// A = fp16(q * s * 2^pw) per weight (the scale applied in the dequant), one
// accumulator per tile, fp16 h * 2^fh out of W13.
// kShortWaits: the instantiation launched when the caller set a wait limit
// below the default (MOE_OPT_WAIT_LIMIT_US); the ordinary one never tests it.
template <bool kShortWaits>
__global__ void __launch_bounds__(kThreads, 1) ggemm_kernel(const __grid_constant__ TcParams p) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  SmemTC *sm = reinterpret_cast<SmemTC *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_blocks = *p.n_blocks;
  const int n_fb = (p.rows > p.rows_s ? p.rows : p.rows_s) / BM;
  const int n_tiles = n_blocks * n_fb;
  constexpr int NACC = 2;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NR; ++i) {
      mbar_init(&sm->raw_full[i], 1);
      mbar_init(&sm->raw_empty[i], kDeqWarps);
    }
    for (int i = 0; i < NG; ++i) {
      mbar_init(&sm->a_full[i], kDeqWarps);
      mbar_init(&sm->a_empty[i], 1);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(&sm->b_full[i], 1);
      mbar_init(&sm->b_empty[i], 1);
    }
    for (int i = 0; i < NACC; ++i) {
      mbar_init(&sm->acc_full[i], 1);
      mbar_init(&sm->acc_empty[i], 4);
    }
    mbar_init(&sm->drain, 1);
    sm->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(&sm->tmem_base))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------ raw weight producer
    {
      uint32_t rk = 0;
      uint32_t armed = 0, par = 0;        // per stage: a copy was issued / its parity
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        Tile tl;
        if (!tile_at(p, t, n_fb, n_blocks, tl) || tl.nvalid <= 0) continue;
        const CUtensorMap *mw = tl.shared ? &p.map_ws : &p.map_w;
        const CUtensorMap *ms = tl.shared ? &p.map_scs : &p.map_sc;
        for (int r = 0; r < tl.K / RK; ++r) {
          const int s = rk % NR;
          const uint32_t ph = (rk / NR) & 1;
          if (!(ok = wait_tc<kShortWaits>(&sm->raw_empty[s], ph ^ 1, sm, p))) break;
          fence_proxy_async();
          if (elect_one()) {
            mbar_expect_tx(&sm->raw_full[s], BM * 128 + BM * (RK / 64) * 4);
            tma_load_2d(sm->raw[s], mw, r * 128, tl.wrow0, &sm->raw_full[s]);
            tma_load_2d(sm->sc[s], ms, r * (RK / 64), tl.wrow0, &sm->raw_full[s]);
          }
          __syncwarp();
          armed |= 1u << s;
          par = (par & ~(1u << s)) | (ph << s);
          ++rk;
        }
      }
      // Drain: every copy this warp issued has landed before the CTA exits.
      const unsigned long long t0 = globaltimer();
      for (int s = 0; s < NR; ++s)
        while (((armed >> s) & 1) && !mbar_try_wait(&sm->raw_full[s], (par >> s) & 1) &&
               globaltimer() - t0 < kWaitNs) {
        }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------ token tile producer
    {
      uint32_t sb = 0;                    // token slots filled so far
      uint32_t armed = 0, par = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        Tile tl;
        if (!tile_at(p, t, n_fb, n_blocks, tl) || tl.nvalid <= 0) continue;
        // Smallest box covering the tile's token rows; one slot carries
        // 256 / rows K blocks of it (K / 64 is a multiple of 8).
        const int bi = box_index(tl.nvalid);
        const int rows = box_rows(bi), kps = box_kps(bi);
        const int brow = tl.p0;
        for (int k0 = 0; k0 < tl.K / BK; k0 += kps) {
          const int s2 = sb % NB;
          const uint32_t ph2 = (sb / NB) & 1;
          if (!(ok = wait_tc<kShortWaits>(&sm->b_empty[s2], ph2 ^ 1, sm, p))) break;
          if (elect_one()) {
            mbar_expect_tx(&sm->b_full[s2], kps * rows * 128);
            for (int j = 0; j < kps; ++j)
              tma_load_2d(sm->b[s2] + j * rows * 128, &p.map_b[bi], (k0 + j) * BK, brow,
                          &sm->b_full[s2]);
          }
          __syncwarp();
          armed |= 1u << s2;
          par = (par & ~(1u << s2)) | (ph2 << s2);
          ++sb;
        }
      }
      const unsigned long long t0 = globaltimer();
      for (int s = 0; s < NB; ++s)
        while (((armed >> s) & 1) && !mbar_try_wait(&sm->b_full[s], (par >> s) & 1) &&
               globaltimer() - t0 < kWaitNs) {
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    {
      // Ring positions advance incrementally (no divisions in the loop) and
      // the token descriptor is the slot's base plus a constant per K block.
      uint32_t it = 0;
      uint32_t ga = 0, gpar = 0;          // A group and its phase
      uint32_t bs = 0, bpar = 0;          // token slot and its phase
      constexpr uint32_t kSlotDesc = (kSlotRows * 128) >> 4;   // descriptor units per slot
      const uint64_t db0 = sw128_desc(smem_u32(sm->b[0]));
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        Tile tl;
        if (!tile_at(p, t, n_fb, n_blocks, tl) || tl.nvalid <= 0) continue;
        const int buf = it & 1;
        if (!(ok = wait_tc<kShortWaits>(&sm->acc_empty[buf], ((it >> 1) & 1) ^ 1, sm, p))) break;
        tc_fence_after();
        const int ncols = tl.nvalid;
        const uint32_t idesc = idesc_f16(BM, (ncols + 15) & ~15);
        const int bi = box_index(ncols);
        const int kps_m1 = box_kps(bi) - 1;                     // K blocks per slot - 1
        const uint32_t jj_desc = (uint32_t)(box_rows(bi) * 128) >> 4;
        const uint32_t dacc = tmem + buf * BN;
        const int nkb = tl.K / BK;
        int jj = 0;
        uint32_t first = 1;
        uint64_t db_slot = db0;
        for (int k0 = 0; ok && k0 < nkb; k0 += KPG) {
          if (!(ok = wait_tc<kShortWaits>(&sm->a_full[ga], gpar, sm, p))) break;
          tc_fence_after();
          const uint32_t acol = tmem + kACol0 + ga * kGroupCols;
#pragma unroll
          for (int j = 0; j < KPG; ++j) {
            if (jj == 0) {
              if (!(ok = wait_tc<kShortWaits>(&sm->b_full[bs], bpar, sm, p))) break;
              db_slot = db0 + (uint64_t)(bs * kSlotDesc);
            }
            const bool slot_done = (jj == kps_m1);
            if (elect_one()) {
              mma_kblock_ta(dacc, acol + j * (BK / 2), db_slot + (uint64_t)(jj * jj_desc), idesc,
                            first ^ 1u);
              if (slot_done) mma_commit(&sm->b_empty[bs]);
            }
            __syncwarp();
            first = 0;
            if (slot_done) {
              jj = 0;
              if (++bs == NB) { bs = 0; bpar ^= 1; }
            } else {
              ++jj;
            }
          }
          if (!ok) break;
          if (elect_one()) mma_commit(&sm->a_empty[ga]);
          __syncwarp();
          if (++ga == NG) { ga = 0; gpar ^= 1; }
        }
        if (!ok) break;
        if (elect_one()) mma_commit(&sm->acc_full[buf]);
        __syncwarp();
        ++it;
      }
      // Drain: one more commit covers every MMA this thread issued -- also
      // those of a tile it stopped in the middle of -- and TMEM is freed only
      // once it has arrived (bounded by the full limit, whatever wait_ns is).
      if (elect_one()) mma_commit(&sm->drain);
      __syncwarp();
      {
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(&sm->drain, 0) && globaltimer() - t0 < kWaitNs) {
        }
      }
    }
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    // ------------------------------------------------------ epilogue
    const int q = warp - kEpiWarp0;       // TMEM lane quadrant
    const int row = q * 32 + lane;        // weight row of the tile
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    uint32_t it = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
      Tile tl;
      if (!tile_at(p, t, n_fb, n_blocks, tl) || tl.nvalid <= 0) continue;
      const int fb = (tl.wrow0 - (tl.shared ? 0 : tl.e * p.rows)) / BM;
      // 2^-pw of this lane's weight row (exact: a power of two).
      const float rinv = __frcp_rn(__ldg((tl.shared ? p.rexp_s : p.rexp) + tl.wrow0 + row));
      const int buf = it & 1;
      if (!(ok = wait_tc<kShortWaits>(&sm->acc_full[buf], (it >> 1) & 1, sm, p))) break;
      tc_fence_after();
      const uint32_t tbase = tmem + lane_base + buf * BN;
      for (int c0 = 0; c0 < tl.nvalid; c0 += 32) {
        // The chunk's per-column factors: lane j loads column c0 + j once and
        // the loops below take them by shuffle (a load per column would wait
        // behind the previous column's stores, which may alias it).
        const bool lane_col = c0 + lane < tl.nvalid;
        const float f0 = lane_col ? __ldcg((p.mode == 0 ? p.xcol : p.wperm) + tl.p0 + c0 + lane) : 0.f;
        const float f1 = (p.mode == 0 && lane_col) ? __ldcg(p.hcol + tl.p0 + c0 + lane) : 0.f;
        float v[32];
        tmem_ld32(tbase + c0, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= rinv;
        if (p.mode == 0) {
          // Rows: lanes 0-15 hold g of features fb*64 + 16q + (lane & 15),
          // lanes 16-31 u of the same.  One exchange per column pair: lanes
          // 0-15 finish token j (their g, the partner's u), lanes 16-31 token
          // j + 1 (the partner's g, their u).  g and u carry the token's 2^ex,
          // taken out before SwiGLU; h is rounded to fp16, so the fast
          // exponential and division are well inside its resolution.
          const int feat = fb * 64 + q * 16 + (lane & 15);
          const bool lo_half = lane < 16;
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float recv = __shfl_xor_sync(0xffffffffu, lo_half ? v[j + 1] : v[j], 16);
            const int jc = j + (lo_half ? 0 : 1);
            const float xc = __shfl_sync(0xffffffffu, f0, jc);
            const float hc = __shfl_sync(0xffffffffu, f1, jc);
            const int col = c0 + jc;
            if (col < tl.nvalid) {
              const int pr = tl.p0 + col;
              const float g = (lo_half ? v[j] : recv) * xc;
              const float u = (lo_half ? recv : v[j + 1]) * xc;
              const float e = __expf(fminf(-g, 80.0f));
              const float hval = __fdividef(g, 1.0f + e) * u * hc;
              p.hb[(size_t)pr * p.h_stride + feat] = __float2half_rn(hval);
            }
          }
        } else {
          const int o = fb * BM + row;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float wt = __shfl_sync(0xffffffffu, f0, j);
            if (c0 + j < tl.nvalid) {
              const int pr = tl.p0 + c0 + j;
              p.y[(size_t)pr * p.H + o] = v[j] * wt;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->acc_empty[buf]);
      ++it;
    }
  } else if (warp >= kDeqWarp0) {
    // ------------------------------------------------------ dequant
    // Warp w owns TMEM lane quadrant w % 4 (tile rows 32 (w % 4) .. +31, one
    // per lane) and half (w - 8) / 4 of every 64-K block: per raw stage a
    // thread turns 4 x 32 weights of its row into 4 x 16 fp16x2 columns of the
    // stage's A group.  The 32 lanes read 32 consecutive rows of the swizzled
    // raw tile, 8 distinct 16-byte bank groups per 8 lanes.
    const int dw = warp - kDeqWarp0;
    const int qd = dw & 3, hh = dw >> 2;
    const int r = qd * 32 + lane;                    // tile row 0..127
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    uint32_t rk = 0, ag = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
      Tile tl;
      if (!tile_at(p, t, n_fb, n_blocks, tl) || tl.nvalid <= 0) continue;
      const float re = __ldg((tl.shared ? p.rexp_s : p.rexp) + tl.wrow0 + r);   // 2^pw
      for (int rr = 0; rr < tl.K / RK; ++rr) {
        const int s = rk % NR;
        if (!(ok = wait_tc<kShortWaits>(&sm->raw_full[s], (rk / NR) & 1, sm, p))) break;
        const float4 sc4 = *reinterpret_cast<const float4 *>(&sm->sc[s][r * (RK / 64)]);
        const uint8_t *rrow = sm->raw[s] + r * 128;
        uint4 c[RK / BK];
#pragma unroll
        for (int j = 0; j < RK / BK; ++j)   // raw 16-byte chunk 2j + hh (128-byte swizzle)
          c[j] = *reinterpret_cast<const uint4 *>(rrow + (((2 * j + hh) ^ (r & 7)) << 4));
        fence_proxy_async();   // the raw reads before the stage's TMA refill
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->raw_empty[s]);
#pragma unroll
        for (int gi = 0; gi < GPS; ++gi) {
          const int ga = ag % NG;
          if (!(ok = wait_tc<kShortWaits>(&sm->a_empty[ga], ((ag / NG) & 1) ^ 1, sm, p))) break;
          tc_fence_after();
          const uint32_t acol = tmem + lane_base + kACol0 + ga * kGroupCols + hh * 16;
          uint32_t o[KPG][16];
#pragma unroll
          for (int jj = 0; jj < KPG; ++jj) {
            const int j = gi * KPG + jj;
            const uint32_t words[4] = {c[j].x, c[j].y, c[j].z, c[j].w};
            const float sv = (j == 0 ? sc4.x : j == 1 ? sc4.y : j == 2 ? sc4.z : sc4.w) * re;
            const __half sh = __float2half_rn(sv);
            const uint32_t s2 = f16x2_splat(sh);
            const uint32_t s16_2 = f16x2_splat(__float2half_rn(__half2float(sh) * 0.0625f));
#pragma unroll
            for (int wv = 0; wv < 4; ++wv) dequant_word_f16(words[wv], s2, s16_2, o[jj] + 4 * wv);
          }
          static_assert(KPG == 2, "two K blocks per A group");
          tmem_st16x2(acol, o[0], acol + BK / 2, o[1]);   // includes the wait
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm->a_full[ga]);
          ++ag;
        }
        if (!ok) break;
        ++rk;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

// ---------------------------------------------------- gather and combine --

// Grouped row p of the tensor-core path, for the token t it carries:
//   xp[p]    = fp16(x[t] * 2^ex), 2^ex the power of two that puts max |x[t]|
//              just under 2^14 (exact for bf16 x: 8 significant bits of 11);
//   xcol[p]  = 2^-ex (the W13 epilogue takes it out of g and u);
//   hcol[p]  = 2^fh with max(N1 |x[t]|, 0.28) N3 |x[t]| * 2^fh < 2^14, a bound
//              on |h| (Euclidean norms; N1, N3 = hnorm[0], hnorm[1], each
//              factor widened by 2% for the fp16 weights' and f32 sums'
//              rounding);
//   wperm[p] = the routing weight (1 for the shared expert) times 2^-fh.
// One warp per token: it reduces max |x[t]| and |x[t]|^2 once, then converts
// each 16-byte piece of x[t] once and stores it into every grouped row of the
// token (its kept routed slots, inv[a] >= 0, and its shared-expert row A + t),
// so x is read twice per token rather than twice per grouped row.
__global__ void __launch_bounds__(256) gather_kernel(const void *__restrict__ x, int x_is_bf16,
                                                     int T, int H, int k, int n_shared,
                                                     const int32_t *__restrict__ inv,
                                                     const float *__restrict__ w,
                                                     const float *__restrict__ hnorm,
                                                     __half *__restrict__ xp,
                                                     float *__restrict__ wperm,
                                                     float *__restrict__ xcol,
                                                     float *__restrict__ hcol) {
  pdl_enter();
  inv = after_wait(inv);
  w = after_wait(w);
  xp = after_wait(xp);
  wperm = after_wait(wperm);
  xcol = after_wait(xcol);
  hcol = after_wait(hcol);
  const int A = T * k, nrows = k + n_shared;   // nrows <= 33
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const float n1 = __ldg(hnorm) * 1.02f, n3 = __ldg(hnorm + 1) * 1.02f;
  for (int t = warp; t < T; t += nwarps) {
    const uint4 *src16 = reinterpret_cast<const uint4 *>(
        reinterpret_cast<const __nv_bfloat16 *>(x) + (size_t)t * H);
    const float4 *src32 = reinterpret_cast<const float4 *>(
        reinterpret_cast<const float *>(x) + (size_t)t * H);
    float amax = 0.f, ss = 0.f;
    if (x_is_bf16) {
      for (int i = lane; i < H / 8; i += 32) {
        const uint4 v = __ldg(src16 + i);
        const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float lo = __uint_as_float(wd[c] << 16), hi = __uint_as_float(wd[c] & 0xFFFF0000u);
          amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
          ss = fmaf(lo, lo, fmaf(hi, hi, ss));
        }
      }
    } else {
      for (int i = lane; i < H / 4; i += 32) {
        const float4 f = __ldg(src32 + i);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
        ss = fmaf(f.x, f.x, fmaf(f.y, f.y, fmaf(f.z, f.z, fmaf(f.w, f.w, ss))));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      ss += __shfl_xor_sync(0xffffffffu, ss, o);
    }
    const int ex = max(-126, min(126, 14 - pow2_above(amax)));
    const float nrm = sqrtf(ss);
    const float bound = fmaxf(n1 * nrm, 0.28f) * (n3 * nrm);
    const int fh = max(-126, min(126, 14 - pow2_above(bound)));
    // The token's grouped rows: row j < k is slot j (-1 when the top-p trim
    // dropped it), row k the shared expert's.  Lane j holds row j; row 32
    // (k = 32 with a shared expert) is the same in every lane.
    const int a0 = t * k;
    const int row_lane = lane < k ? __ldcg(inv + a0 + lane) : (lane < nrows ? A + t : -1);
    const int row_32 = nrows > 32 ? A + t : -1;
    for (int j = lane; j < nrows; j += 32) {
      const int pr = j < 32 ? row_lane : row_32;
      if (pr < 0) continue;
      const float wt = j < k ? __ldcg(w + a0 + j) : 1.0f;
      wperm[pr] = wt * pow2f(-fh);
      xcol[pr] = pow2f(-ex);
      hcol[pr] = pow2f(fh);
    }
    const float xs = pow2f(ex);
    // H is a multiple of 256, so every lane runs the same number of pieces
    // and the shuffles below see the whole warp.
    if (x_is_bf16) {
      for (int i = lane; i < H / 8; i += 32) {
        const uint4 v = __ldg(src16 + i);
        const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const __half2 hh = __floats2half2_rn(__uint_as_float(wd[c] << 16) * xs,
                                               __uint_as_float(wd[c] & 0xFFFF0000u) * xs);
          o[c] = *reinterpret_cast<const uint32_t *>(&hh);
        }
        const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
        for (int j = 0; j < nrows; ++j) {
          const int pr = j < 32 ? __shfl_sync(0xffffffffu, row_lane, j) : row_32;
          if (pr >= 0) reinterpret_cast<uint4 *>(xp + (size_t)pr * H)[i] = ov;
        }
      }
    } else {
      for (int i = lane; i < H / 4; i += 32) {
        const float4 f = __ldg(src32 + i);
        const __half2 h0 = __floats2half2_rn(f.x * xs, f.y * xs);
        const __half2 h1 = __floats2half2_rn(f.z * xs, f.w * xs);
        const uint2 ov = make_uint2(*reinterpret_cast<const uint32_t *>(&h0),
                                    *reinterpret_cast<const uint32_t *>(&h1));
        for (int j = 0; j < nrows; ++j) {
          const int pr = j < 32 ? __shfl_sync(0xffffffffu, row_lane, j) : row_32;
          if (pr >= 0) reinterpret_cast<uint2 *>(xp + (size_t)pr * H)[i] = ov;
        }
      }
    }
  }
}

// Decode tensor-core path (decode_tc.cu): grouped row pr of x as operand
// planes -- x itself when it is bf16 (one plane), else rows 2pr, 2pr+1 = bf16
// hi, bf16(x - hi) -- and the grouped routing weights.
__global__ void __launch_bounds__(256) gather_exact_kernel(const void *__restrict__ x,
                                                           int x_is_bf16, int T, int H, int k,
                                                           int n_shared,
                                                           const int32_t *__restrict__ perm,
                                                           const int32_t *__restrict__ n_assigned,
                                                           const float *__restrict__ w,
                                                           __nv_bfloat16 *__restrict__ xe,
                                                           float *__restrict__ wperm) {
  pdl_enter();
  perm = after_wait(perm);
  n_assigned = after_wait(n_assigned);
  w = after_wait(w);
  xe = after_wait(xe);
  wperm = after_wait(wperm);
  const int A = T * k, R = A + n_shared * T;
  const int n_routed = __ldcg(n_assigned);
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int pr = warp; pr < R; pr += nwarps) {
    if (pr >= n_routed && pr < A) continue;   // rows of slots the top-p trim dropped
    int t;
    float wt;
    if (pr < A) {
      const int a = perm[pr];
      t = a / k;
      wt = w[a];
    } else {
      t = pr - A;
      wt = 1.0f;
    }
    if (lane == 0) wperm[pr] = wt;
    if (x_is_bf16) {
      const uint4 *src = reinterpret_cast<const uint4 *>(
          reinterpret_cast<const __nv_bfloat16 *>(x) + (size_t)t * H);
      uint4 *dst = reinterpret_cast<uint4 *>(xe + (size_t)pr * H);
      for (int i = lane; i < H / 8; i += 32) dst[i] = __ldg(src + i);
    } else {
      const float4 *src = reinterpret_cast<const float4 *>(
          reinterpret_cast<const float *>(x) + (size_t)t * H);
      __nv_bfloat162 *hi = reinterpret_cast<__nv_bfloat162 *>(xe + (size_t)(2 * pr) * H);
      __nv_bfloat162 *lo = reinterpret_cast<__nv_bfloat162 *>(xe + (size_t)(2 * pr + 1) * H);
      for (int i = lane; i < H / 4; i += 32) {
        const float4 f = __ldg(src + i);
        const __nv_bfloat162 h0 = __floats2bfloat162_rn(f.x, f.y);
        const __nv_bfloat162 h1 = __floats2bfloat162_rn(f.z, f.w);
        hi[2 * i] = h0;
        hi[2 * i + 1] = h1;
        lo[2 * i] = __floats2bfloat162_rn(f.x - __low2float(h0), f.y - __high2float(h0));
        lo[2 * i + 1] = __floats2bfloat162_rn(f.z - __low2float(h1), f.w - __high2float(h1));
      }
    }
  }
}

// out[t] (+)= sum_j y[inv[t*k+j]] + y_shared[t]: slot order, then the shared
// expert; one owner per element, no atomics (tutorial cf-1.com §3.3 Step 5).
__global__ void __launch_bounds__(256) combine_kernel(int T, int H, int k, int n_shared,
                                                      const int32_t *__restrict__ inv,
                                                      const float *__restrict__ y,
                                                      float *__restrict__ out, int accumulate) {
  pdl_enter();
  inv = after_wait(inv);
  y = after_wait(y);
  out = after_wait(out);
  const int A = T * k;
  const int per_t = H / 4;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < (long long)T * per_t;
       i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i / per_t), c = (int)(i - (long long)t * per_t);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const int row = __ldcg(inv + t * k + j);
      if (row < 0) continue;   // a slot the top-p trim dropped
      const float4 v = __ldcg(reinterpret_cast<const float4 *>(y + (size_t)row * H) + c);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    if (n_shared) {
      const float4 v = __ldcg(reinterpret_cast<const float4 *>(y + (size_t)(A + t) * H) + c);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    float4 *o = reinterpret_cast<float4 *>(out + (size_t)t * H) + c;
    if (accumulate) {
      const float4 prev = *o;
      acc.x += prev.x;
      acc.y += prev.y;
      acc.z += prev.z;
      acc.w += prev.w;
    }
    *o = acc;
  }
}

// The combine of one token by a 1024-thread block, followed by the next
// stacked layer's RMS pre-norm of the updated row (moe_forward_residual_norm):
// out[t] (+)= sum of the token's expert rows as in combine_kernel (the same
// order, so the same bits), then norm_out[t] = bf16(rmsnorm(out[t])) exactly
// as moe_rmsnorm_bf16 computes it.  One launch in place of two; the row stays
// in registers between the two steps (float4s past 2048, H > 8192, are read
// back from out).
__global__ void __launch_bounds__(1024) combine_norm_kernel(
    int T, int H, int k, int n_shared, const int32_t *__restrict__ inv,
    const float *__restrict__ y, float *__restrict__ out, int accumulate, float eps,
    __nv_bfloat16 *__restrict__ norm_out) {
  pdl_enter();
  inv = after_wait(inv);
  y = after_wait(y);
  out = after_wait(out);
  norm_out = after_wait(norm_out);
  __shared__ float part[32];
  const int t = blockIdx.x;
  const int A = T * k;
  const int n4 = H / 4;
  float4 *orow = reinterpret_cast<float4 *>(out + (size_t)t * H);
  auto combine4 = [&](int c) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const int row = __ldcg(inv + t * k + j);
      if (row < 0) continue;   // a slot the top-p trim dropped
      const float4 v = __ldcg(reinterpret_cast<const float4 *>(y + (size_t)row * H) + c);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    if (n_shared) {
      const float4 v = __ldcg(reinterpret_cast<const float4 *>(y + (size_t)(A + t) * H) + c);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    if (accumulate) {
      const float4 prev = orow[c];
      acc.x += prev.x;
      acc.y += prev.y;
      acc.z += prev.z;
      acc.w += prev.w;
    }
    orow[c] = acc;
    return acc;
  };
  float4 v[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int i = threadIdx.x + r * 1024;
    v[r] = (i < n4) ? combine4(i) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int i = threadIdx.x + 2048; i < n4; i += 1024) combine4(i);
  rmsnorm_row_bf16(orow, v, H, eps, norm_out + (size_t)t * H, part);
}

// ------------------------------------------------- router on tensor cores --
//
// z[t][e] = sum_h x[t][h] * Wr[e][h] for bf16 x, with Wr held as three bf16
// planes hi + mid + lo (hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi -
// mid): 24 significant bits, the f32 value up to its last bit).  All three
// planes accumulate in f32 TMEM, so the logits carry f32 rounding, not bf16
// (the router stays f32: colibrì engine teardown, "System map").  The K range
// is split over 8 accumulators, summed in IEEE f32 in the epilogue: the tensor
// core's accumulation then never runs more than 1/8 of K in one chain.
// Tile: 128 experts x 64 tokens, one tile per CTA.
constexpr int RT_N = 64;         // tokens per tile
constexpr int RT_ACC = 8;        // accumulators (TMEM columns RT_ACC * RT_N)
constexpr int RT_S = 3;          // stages
constexpr uint32_t RT_STAGE_TX = 3 * BM * 128 + RT_N * 128;

struct __align__(1024) SmemRT {
  uint8_t a[RT_S][3][BM * 128];  // 3 stages x 3 planes x 16 KB
  uint8_t b[RT_S][RT_N * 128];   // 3 stages x 8 KB
  uint64_t full[RT_S], empty[RT_S], acc_full;
  uint32_t tmem_base;
  int abort;
};

struct RtParams {
  CUtensorMap map_a;       // bf16 planes [3E][H]
  CUtensorMap map_x;       // bf16 x [T][H]
  int E, T, H;
  float *z;                // [T][E]
  int32_t *status;
};

__device__ __noinline__ bool rt_wait_slow(uint64_t *bar, uint32_t parity, SmemRT *sm,
                                          int32_t *status) {
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (*reinterpret_cast<volatile int *>(&sm->abort)) return false;
      if (globaltimer() - t0 > kWaitNs) {
        atomicExch(reinterpret_cast<int *>(&sm->abort), 1);
        atomicExch(status, kStatusTimeout);
        return false;
      }
    }
  }
}

// Called by whole warps; the same result in every lane (see moe::wait_bar).
__device__ __forceinline__ bool rt_wait(uint64_t *bar, uint32_t parity, SmemRT *sm,
                                        int32_t *status) {
  return __all_sync(0xffffffffu, mbar_try_wait(bar, parity) || rt_wait_slow(bar, parity, sm, status));
}

__global__ void __launch_bounds__(256, 1) router_tc_kernel(const __grid_constant__ RtParams p) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  SmemRT *sm = reinterpret_cast<SmemRT *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = blockIdx.x * BM, t0 = blockIdx.y * RT_N;
  // Split-K over gridDim.z: this CTA's K blocks [kb0, kb0 + nk), its partial
  // logits written to z[blockIdx.z][T][E] (the top-k sums the splits in order).
  const int nk_all = p.H / BK;
  const int kb0 = (int)((long long)nk_all * blockIdx.z / gridDim.z);
  const int nk = (int)((long long)nk_all * (blockIdx.z + 1) / gridDim.z) - kb0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < RT_S; ++i) {
      mbar_init(&sm->full[i], 1);
      mbar_init(&sm->empty[i], 1);
    }
    mbar_init(&sm->acc_full, 1);
    sm->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(&sm->tmem_base))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;

  if (warp == 0) {
    uint32_t armed = 0, par = 0;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % RT_S;
      const uint32_t ph = (kb / RT_S) & 1;
      if (!rt_wait(&sm->empty[s], ph ^ 1, sm, p.status)) break;
      if (elect_one()) {
        mbar_expect_tx(&sm->full[s], RT_STAGE_TX);
#pragma unroll
        for (int pl = 0; pl < 3; ++pl)
          tma_load_2d(sm->a[s][pl], &p.map_a, (kb0 + kb) * BK, pl * p.E + e0, &sm->full[s]);
        tma_load_2d(sm->b[s], &p.map_x, (kb0 + kb) * BK, t0, &sm->full[s]);
      }
      __syncwarp();
      armed |= 1u << s;
      par = (par & ~(1u << s)) | (ph << s);
    }
    const unsigned long long tw = globaltimer();
    for (int s = 0; s < RT_S; ++s)
      while (((armed >> s) & 1) && !mbar_try_wait(&sm->full[s], (par >> s) & 1) &&
             globaltimer() - tw < kWaitNs) {
      }
  } else if (warp == 1) {
    const uint32_t idesc = idesc_bf16(BM, RT_N);
    bool ok = true;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % RT_S;
      if (!(ok = rt_wait(&sm->full[s], (kb / RT_S) & 1, sm, p.status))) break;
      tc_fence_after();
      const uint64_t db = sw128_desc(smem_u32(sm->b[s]));
      // accumulator of this k-block: the n_acc accumulators take equal runs of
      // the CTA's k-blocks (one each when there are no more k-blocks than
      // accumulators)
      const int n_acc = nk < RT_ACC ? nk : RT_ACC;
      const int acc = kb * n_acc / nk;
      const bool first = (kb == 0) || ((kb - 1) * n_acc / nk != acc);
      const uint32_t d = tmem + acc * RT_N;
      if (elect_one()) {
#pragma unroll
        for (int pl = 0; pl < 3; ++pl) {
          const uint64_t da = sw128_desc(smem_u32(sm->a[s][pl]));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_bf16(d, da + (uint64_t)(kk * 2), db + (uint64_t)(kk * 2), idesc,
                     (!first || pl || kk) ? 1u : 0u);
        }
        mma_commit(&sm->empty[s]);
      }
      __syncwarp();
    }
    if (ok) {
      if (elect_one()) mma_commit(&sm->acc_full);
      __syncwarp();
      const unsigned long long tw = globaltimer();
      while (!mbar_try_wait(&sm->acc_full, 0) && globaltimer() - tw < kWaitNs) {
      }
    }
  } else if (warp >= 4) {
    const int q = warp - 4;
    const int e = e0 + q * 32 + lane;
    if (rt_wait(&sm->acc_full, 0, sm, p.status)) {
      tc_fence_after();
      const int n_acc = nk < RT_ACC ? nk : RT_ACC;   // accumulators that received k-blocks
#pragma unroll
      for (int c0 = 0; c0 < RT_N; c0 += 32) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + c0, v);
        for (int a = 1; a < RT_ACC; ++a) {
          if (a >= n_acc) break;
          float u[32];
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + a * RT_N + c0, u);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] += u[j];
        }
        if (e < p.E) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int t = t0 + c0 + j;
            if (t < p.T) p.z[((size_t)blockIdx.z * p.T + t) * p.E + e] = v[j];
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

// hi/mid/lo bf16 planes of the transposed router weights: planes [3][E][H].
__global__ void split_planes_kernel(const float *__restrict__ w, __nv_bfloat16 *__restrict__ planes,
                                    long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const float v = w[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
    planes[i] = hi;
    planes[n + i] = mid;
    planes[2 * n + i] = lo;
  }
}

// ---------------------------------------------------------- host side --

constexpr size_t kSmemBytes = sizeof(SmemTC) + 1024;

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2D map over a row-major [rows][cols] array, box [box_rows][box_cols], 128B
// swizzle (or none).
bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, size_t elem, uint64_t cols,
              uint64_t rows, uint64_t row_stride_elems, uint32_t box_cols, uint32_t box_rows,
              bool swizzle) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_stride_elems * elem};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_path_available() { return get_encode() != nullptr; }

cudaError_t launch_split_planes(const float *wr_t, __nv_bfloat16 *planes, long long n,
                                cudaStream_t st) {
  return launch_k(false, split_planes_kernel, dim3(152 * 4), dim3(256), 0, st, wr_t, planes, n);
}

cudaError_t launch_router_tc(const moe_handle *h, const void *x, int T, float *z, int splits,
                             cudaStream_t st) {
  const int E = h->E, H = h->H;
  static bool attr = false;
  const size_t smem = sizeof(SmemRT) + 1024;
  if (!attr) {
    cudaError_t err =
        cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    attr = true;
  }
  RtParams p{};
  if (!make_map(&p.map_a, h->wr_planes, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, (uint64_t)3 * E, H,
                BK, BM) ||
      !make_map(&p.map_x, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, (uint64_t)T, H, BK, RT_N))
    return cudaErrorInvalidValue;
  p.E = E;
  p.T = T;
  p.H = H;
  p.z = z;
  p.status = h->ws.status;
  return launch_k(false, router_tc_kernel,
                  dim3((E + BM - 1) / BM, (T + RT_N - 1) / RT_N, splits), dim3(256), smem, st, p);
}

cudaError_t launch_combine(const moe_handle *h, int T, float *out, bool accumulate,
                           cudaStream_t st) {
  if (h->norm_out && T > 0)   // with the next layer's pre-norm: one block per token
    return launch_k(h->pdl, combine_norm_kernel, dim3(T), dim3(1024), 0, st, T, h->H, h->k, h->S,
                    h->ws.inv, h->ws.y, out, accumulate ? 1 : 0, h->norm_eps,
                    reinterpret_cast<__nv_bfloat16 *>(h->norm_out));
  // One float4 per thread; no more CTAs than there is work (decode: a handful).
  const long long work = (long long)T * (h->H / 4);
  const int blocks = (int)std::min<long long>((long long)h->num_sms * 8, (work + 255) / 256);
  if (blocks == 0) return cudaSuccess;
  return launch_k(h->pdl, combine_kernel, dim3(blocks), dim3(256), 0, st, T, h->H, h->k, h->S,
                  h->ws.inv, h->ws.y, out, accumulate ? 1 : 0);
}

namespace {
cudaError_t set_tc_attrs() {
  static bool attr = false;   // per process; the attribute is per function
  if (!attr) {
    cudaError_t err = cudaFuncSetAttribute(ggemm_kernel<false>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemBytes);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(ggemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    attr = true;
  }
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_gather_exact(const moe_handle *h, const void *x, int T, cudaStream_t st) {
  const moe::Workspace &w = h->ws;
  return launch_k(h->pdl, gather_exact_kernel, dim3(h->num_sms), dim3(256), 0, st, x,
                  h->L.x_dtype == 1, T, h->H, h->k, h->S, w.perm, w.offsets + h->E, w.w, w.xe,
                  w.wperm);
}

cudaError_t launch_tc_path(const moe_handle *h, const void *x, int T, float *out, bool accumulate,
                           cudaStream_t st) {
  const moe::Workspace &w = h->ws;
  const int E = h->E, H = h->H, I = h->I, k = h->k, S = h->S;
  const int Is = S ? h->Is : I;
  const int A = T * k, R = A + S * T;
  const int maxR = h->L.max_tokens * k + S * h->L.max_tokens;
  const int h_stride = I > Is ? I : Is;
  cudaError_t err = set_tc_attrs();
  if (err != cudaSuccess) return err;
  const bool short_waits = h->wait_ns < kWaitNs;
  err = launch_k(h->pdl, gather_kernel, dim3(h->num_sms * 4), dim3(256), 0, st, x,
                 h->L.x_dtype == 1, T, H, k, S, w.inv, w.w,
                 (const float *)h->hnorm, w.xp, w.wperm, w.xcol, w.hcol);
  if (err != cudaSuccess) return err;
  moe_handle *hm = const_cast<moe_handle *>(h);
  if (h->profile && hm->n_ev <= moe_handle::kMaxStages) {
    hm->stage_names[hm->n_ev - 1] = "gather";
    cudaEventRecord(hm->ev[hm->n_ev++], st);
  }
  hm->launches += 1;

  TcParams p{};
  const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapDataType F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapDataType F32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  // ---- W13
  bool ok = make_map(&p.map_w, h->ex.w13q, U8, 1, H / 2, (uint64_t)E * 2 * I, H / 2, 128, BM);
  ok = ok && make_map(&p.map_ws, S ? h->sh.w13q : h->ex.w13q, U8, 1, H / 2,
                      (uint64_t)2 * (S ? Is : I), H / 2, 128, BM);
  for (int i = 0; i < 4; ++i)
    ok = ok && make_map(&p.map_b[i], w.xp, F16, 2, H, (uint64_t)maxR, H, BK, kBoxRows[i]);
  ok = ok && make_map(&p.map_sc, h->ex.w13s, F32, 4, H / 64, (uint64_t)E * 2 * I, H / 64,
                      RK / 64, BM, false);
  ok = ok && make_map(&p.map_scs, S ? h->sh.w13s : h->ex.w13s, F32, 4, H / 64,
                      (uint64_t)2 * (S ? Is : I), H / 64, RK / 64, BM, false);
  if (!ok) return cudaErrorInvalidValue;
  p.mode = 0;
  p.K = H;
  p.K_s = H;
  p.rows = 2 * I;
  p.rows_s = 2 * Is;
  p.E = E;
  p.A = A;
  p.T = T;
  p.blocks = w.tiles;
  p.n_blocks = w.n_tiles;
  p.offsets = w.offsets;
  p.rexp = h->ex.w13e;
  p.rexp_s = S ? h->sh.w13e : h->ex.w13e;
  p.hb = w.hb;
  p.h_stride = h_stride;
  p.y = w.y;
  p.H = H;
  p.wperm = w.wperm;
  p.xcol = w.xcol;
  p.hcol = w.hcol;
  p.status = w.status;
  p.wait_ns = h->wait_ns;
  if ((err = launch_k(h->pdl, short_waits ? ggemm_kernel<true> : ggemm_kernel<false>, dim3(h->num_sms),
                      dim3(kThreads), kSmemBytes, st, p)) !=
      cudaSuccess)
    return err;
  if (h->profile && hm->n_ev <= moe_handle::kMaxStages) {
    hm->stage_names[hm->n_ev - 1] = "w13";
    cudaEventRecord(hm->ev[hm->n_ev++], st);
  }
  hm->launches += 1;
  // ---- W2: A = W2 rows [H] over K = I, B = h [R][h_stride]
  ok = make_map(&p.map_w, h->ex.w2q, U8, 1, I / 2, (uint64_t)E * H, I / 2, 128, BM);
  ok = ok && make_map(&p.map_ws, S ? h->sh.w2q : h->ex.w2q, U8, 1, Is / 2, (uint64_t)H, Is / 2, 128,
                      BM);
  for (int i = 0; i < 4; ++i)
    ok = ok && make_map(&p.map_b[i], w.hb, F16, 2, h_stride, (uint64_t)maxR, h_stride, BK,
                        kBoxRows[i]);
  ok = ok && make_map(&p.map_sc, h->ex.w2s, F32, 4, I / 64, (uint64_t)E * H, I / 64, RK / 64, BM,
                      false);
  ok = ok && make_map(&p.map_scs, S ? h->sh.w2s : h->ex.w2s, F32, 4, Is / 64, (uint64_t)H, Is / 64,
                      RK / 64, BM, false);
  if (!ok) return cudaErrorInvalidValue;
  p.mode = 1;
  p.K = I;
  p.K_s = Is;
  p.rows = H;
  p.rows_s = H;
  p.rexp = h->ex.w2e;
  p.rexp_s = S ? h->sh.w2e : h->ex.w2e;
  if ((err = launch_k(h->pdl, short_waits ? ggemm_kernel<true> : ggemm_kernel<false>, dim3(h->num_sms),
                      dim3(kThreads), kSmemBytes, st, p)) !=
      cudaSuccess)
    return err;
  if (h->profile && hm->n_ev <= moe_handle::kMaxStages) {
    hm->stage_names[hm->n_ev - 1] = "w2";
    cudaEventRecord(hm->ev[hm->n_ev++], st);
  }
  hm->launches += 1;
  err = launch_combine(h, T, out, accumulate, st);
  hm->launches += 1;
  if (h->profile && hm->n_ev <= moe_handle::kMaxStages) {
    hm->stage_names[hm->n_ev - 1] = "combine";
    cudaEventRecord(hm->ev[hm->n_ev++], st);
  }
  (void)R;
  return err;
}

}  // namespace moe
