// dispatch.cu -- step 3 of the layer: group the T*k assignments by expert.
//
// A counting sort, as the pages do it (Colibri C + cuBLASLt tutorial,
// cf-1.com, §3.3 Step 3: per-expert counts, a prefix sum into offsets, then a
// scatter, in place and with no allocation): a shared-memory histogram, a
// block-wide exclusive scan, and a stable scatter.  Assignment a = t*k + j goes
// to perm[offsets[e] + r], where r counts the assignments of expert e with a
// smaller a, so each expert's group lists its tokens in ascending order.
//
// Three launches (T > 8; the fused routing launch groups smaller batches):
// ranks and counts over contiguous ranges of assignments, one CTA per range;
// one CTA that scans the counts into offsets and per-range bases; a scatter
// over the same ranges.  Ranges and ranks both ascend, so the order is the
// stable one.
//
// Also produced here, for the expert kernels: the ascending list of experts
// that received tokens (the shared expert, id E, appended last), and the
// tensor-core token blocks: one entry per tile_m tokens of every non-empty
// group (the shared expert's included), costliest first.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;

// Exclusive scan over the block; returns the prefix and writes the total.
__device__ int block_exclusive_scan(int v, int *warp_sums, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
    int si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += n;
    }
    warp_sums[lane] = si - s;   // exclusive prefix of the warp totals
    if (lane == 31) *total = si;
  }
  __syncthreads();
  const int r = warp_sums[warp] + incl - v;
  __syncthreads();
  return r;
}

// Phase 1 of the dispatch, one CTA per contiguous range of assignments (CTA c
// takes [c A / C, (c + 1) A / C)): each assignment's rank among the earlier
// assignments of its expert inside the range goes to inv[a] (-1 for a dropped
// or invalid id), and the range's per-expert counts to part[c][e].  Inside a
// chunk of 1024, __match_any_sync ranks a lane among the lanes of its warp
// holding the same expert, and a per-(warp, expert) count table turns that
// into a rank across the chunk.
__device__ void rank_range(int c_idx, int C, const int32_t *__restrict__ idx, int A, int E,
                           int32_t *__restrict__ inv, int32_t *__restrict__ part,
                           int32_t *__restrict__ status) {
  extern __shared__ int smem[];
  int *run = smem;                 // [E] assignments of each expert so far in this range
  int *wc = run + E;               // [32][E]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int a0 = (int)((long long)A * c_idx / C);
  const int a1 = (int)((long long)A * (c_idx + 1) / C);
  for (int e = tid; e < E; e += kThreads) run[e] = 0;
  for (int i = tid; i < 32 * E; i += kThreads) wc[i] = 0;
  __syncthreads();
  const unsigned lt_mask = (1u << lane) - 1u;
  int bad = 0;
  for (int c0 = a0; c0 < a1; c0 += kThreads) {
    const int a = c0 + tid;
    int e = (a < a1) ? idx[a] : E;
    if (a < a1 && e != -1 && (e < 0 || e >= E)) bad = 1;
    if (e < 0 || e >= E) e = E;                  // dropped or invalid ids are not placed
    if (a < a1 && e == E) inv[a] = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    if (e < E && (peers & lt_mask) == 0) wc[warp * E + e] = __popc(peers);
    __syncthreads();
    for (int x = tid; x < E; x += kThreads) {
      int r = run[x];
      for (int w = 0; w < 32; ++w) {
        const int n = wc[w * E + x];
        wc[w * E + x] = r;
        r += n;
      }
      run[x] = r;
    }
    __syncthreads();
    if (e < E) inv[a] = wc[warp * E + e] + rank;
    __syncthreads();
    for (int i = tid; i < 32 * E; i += kThreads) wc[i] = 0;
    __syncthreads();
  }
  if (bad) atomicExch(status, kStatusBadExpert);
  for (int x = tid; x < E; x += kThreads) part[(size_t)c_idx * E + x] = run[x];
}

__global__ void __launch_bounds__(kThreads, 1) dispatch_rank_kernel(
    const int32_t *__restrict__ idx, int A, int E, int32_t *__restrict__ inv,
    int32_t *__restrict__ part, int32_t *__restrict__ status) {
  pdl_enter();
  rank_range(blockIdx.x, gridDim.x, after_wait(idx), A, E, after_wait(inv), after_wait(part),
             after_wait(status));
}

// Phase 2, one CTA: per-expert totals over the C ranges, counts, offsets (a
// block-wide exclusive scan), usage; part[c][e] becomes the first position of
// range c's assignments of expert e (offsets[e] plus the earlier ranges'
// counts).  Also the ascending list of experts that received tokens (the
// shared expert, id E, appended last) and the tensor-core token blocks: one
// entry per tile_m tokens of every non-empty group (the shared expert's
// included), costliest first.
__device__ void scan_ranges(int T, int E, int n_shared, int tile_m, int C,
                            int32_t *__restrict__ part, int32_t *__restrict__ counts,
                            int32_t *__restrict__ offsets, int32_t *__restrict__ active,
                            int32_t *__restrict__ n_active, int32_t *__restrict__ tiles,
                            int32_t *__restrict__ n_tiles, unsigned long long *__restrict__ usage) {
  __shared__ int warp_sums[32];
  __shared__ int total;
  const int tid = threadIdx.x;
  // Totals (E <= 1024: one expert per thread), the loads of 8 ranges at a time
  // issued before their sums.
  int c = 0;
  if (tid < E) {
    for (int r0 = 0; r0 < C; r0 += 8) {
      int v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = (r0 + u < C) ? part[(size_t)(r0 + u) * E + tid] : 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) c += v[u];
    }
  }
  const int off = block_exclusive_scan(c, warp_sums, &total);
  if (tid < E) {
    counts[tid] = c;
    offsets[tid] = off;
    if (usage && c) usage[tid] += (unsigned long long)c;   // one writer per expert
    int pos = off;
    for (int r = 0; r < C; ++r) {
      const int n = part[(size_t)r * E + tid];
      part[(size_t)r * E + tid] = pos;
      pos += n;
    }
  }
  if (tid == 0) offsets[E] = total;

  // Ascending list of non-empty experts; the shared expert (id E) goes last.
  const int flag = (tid < E && c > 0) ? 1 : 0;
  const int apos = block_exclusive_scan(flag, warp_sums, &total);
  if (flag) active[apos] = tid;
  if (tid == 0) {
    int na = total;
    if (n_shared) active[na++] = E;
    *n_active = na;
  }
  // Tensor-core token blocks, (expert << 16 | block index) in one int32.
  // Two lists: every full block (routed experts in expert order, then the
  // shared expert's), and the partial last blocks by size class (> 128
  // tokens, > 64, > 32, the rest).  They are dealt alternately (full,
  // partial, full, ...; the longer list's rest at the end), so that the
  // tensor-bound full tiles and the weight-stream-bound small ones run side by
  // side instead of one phase after the other; with the round-robin deal of
  // tiles over the CTAs each CTA gets a similar mix.
  const int nfull = (tid < E) ? c / tile_m : 0;
  const int rem = (tid < E) ? c - nfull * tile_m : 0;
  const int s_full = n_shared ? T / tile_m : 0, s_rem = n_shared ? T - s_full * tile_m : 0;
  const int base_pos = block_exclusive_scan(nfull, warp_sums, &total);
  const int n_f = total + s_full;                       // full blocks
  block_exclusive_scan(rem > 0 ? 1 : 0, warp_sums, &total);
  const int n_p = total + (s_rem > 0 ? 1 : 0);         // partial blocks
  // position of full block f and of partial block q in the dealt list
  auto pos_f = [n_f, n_p](int f) { return f < n_p ? 2 * f : n_p + f; };
  auto pos_q = [n_f, n_p](int q) { return q < n_f ? 2 * q + 1 : n_f + q; };
  for (int i = 0; i < nfull; ++i) tiles[pos_f(base_pos + i)] = (tid << 16) | i;
  if (tid == 0)
    for (int i = 0; i < s_full; ++i) tiles[pos_f(n_f - s_full + i)] = (E << 16) | i;
  int nq = 0;
  for (int cls = 0; cls < 4; ++cls) {
    const int lo = cls == 0 ? 128 : cls == 1 ? 64 : cls == 2 ? 32 : 0;
    const int hi = cls == 0 ? tile_m : cls == 1 ? 128 : cls == 2 ? 64 : 32;
    const int f = (rem > lo && rem <= hi) ? 1 : 0;
    const int pos = block_exclusive_scan(f, warp_sums, &total);
    if (f) tiles[pos_q(nq + pos)] = (tid << 16) | nfull;
    nq += total;
    if (s_rem > lo && s_rem <= hi) {
      if (tid == 0) tiles[pos_q(nq)] = (E << 16) | s_full;
      nq += 1;
    }
  }
  if (tid == 0) n_tiles[0] = n_f + n_p;
}

__global__ void __launch_bounds__(kThreads, 1) dispatch_scan_kernel(
    int T, int E, int n_shared, int tile_m, int C, int32_t *__restrict__ part,
    int32_t *__restrict__ counts, int32_t *__restrict__ offsets, int32_t *__restrict__ active,
    int32_t *__restrict__ n_active, int32_t *__restrict__ tiles, int32_t *__restrict__ n_tiles,
    unsigned long long *__restrict__ usage) {
  pdl_enter();
  scan_ranges(T, E, n_shared, tile_m, C, after_wait(part), after_wait(counts),
              after_wait(offsets), after_wait(active), after_wait(n_active), after_wait(tiles),
              after_wait(n_tiles), after_wait(usage));
}

// Phase 3, the ranges of phase 1: assignment a of range c and expert e goes to
// position part[c][e] + its rank: perm[pos] = a, inv[a] = pos.
__device__ void scatter_range(int c_idx, int C, const int32_t *__restrict__ idx, int A, int E,
                              const int32_t *__restrict__ part, int32_t *__restrict__ perm,
                              int32_t *__restrict__ inv) {
  const int a0 = (int)((long long)A * c_idx / C);
  const int a1 = (int)((long long)A * (c_idx + 1) / C);
  for (int a = a0 + threadIdx.x; a < a1; a += blockDim.x) {
    const int e = idx[a];
    const int r = inv[a];
    if (e < 0 || e >= E || r < 0) continue;
    const int pos = part[(size_t)c_idx * E + e] + r;
    perm[pos] = a;
    inv[a] = pos;
  }
}

__global__ void __launch_bounds__(kThreads) dispatch_scatter_kernel(
    const int32_t *__restrict__ idx, int A, int E, const int32_t *__restrict__ part,
    int32_t *__restrict__ perm, int32_t *__restrict__ inv) {
  pdl_enter();
  scatter_range(blockIdx.x, gridDim.x, after_wait(idx), A, E, after_wait(part), after_wait(perm),
                after_wait(inv));
}

// The three phases in one CTA, for a single range (A <= kThreads assignments):
// one launch instead of three.  A CTA barrier between the phases makes each
// phase's global writes visible to the next one's threads.
__global__ void __launch_bounds__(kThreads, 1) dispatch_small_kernel(
    const int32_t *__restrict__ idx, int T, int A, int E, int n_shared, int tile_m,
    int32_t *__restrict__ inv, int32_t *__restrict__ part, int32_t *__restrict__ perm,
    int32_t *__restrict__ counts, int32_t *__restrict__ offsets, int32_t *__restrict__ active,
    int32_t *__restrict__ n_active, int32_t *__restrict__ tiles, int32_t *__restrict__ n_tiles,
    unsigned long long *__restrict__ usage, int32_t *__restrict__ status) {
  pdl_enter();
  idx = after_wait(idx);
  inv = after_wait(inv);
  part = after_wait(part);
  perm = after_wait(perm);
  rank_range(0, 1, idx, A, E, inv, part, after_wait(status));
  __syncthreads();
  scan_ranges(T, E, n_shared, tile_m, 1, part, after_wait(counts), after_wait(offsets),
              after_wait(active), after_wait(n_active), after_wait(tiles), after_wait(n_tiles),
              after_wait(usage));
  __syncthreads();
  scatter_range(0, 1, idx, A, E, part, perm, inv);
}

}  // namespace

cudaError_t launch_dispatch(const moe_handle *h, int T, int tile_m, unsigned long long *usage,
                            cudaStream_t st) {
  const int E = h->E, A = T * h->k;
  // Ranges of at least 1024 assignments, one CTA per SM at most.
  const int C = std::max(1, std::min(h->num_sms, (A + kThreads - 1) / kThreads));
  const size_t smem = (size_t)(1 + 32) * E * sizeof(int);
  static bool attr_set = false;   // per process; the attribute is per function
  if (!attr_set) {
    const int max_smem = (int)((1 + 32) * kMaxExperts * sizeof(int));
    cudaError_t err = cudaFuncSetAttribute(dispatch_rank_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(dispatch_small_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (err != cudaSuccess) return err;
    attr_set = true;
  }
  const moe::Workspace &w = h->ws;
  // part[C][E] lives in the router's logit buffer: the top-k has read the
  // logits when the dispatch runs, and the buffer has max(max_tokens, 128) >= C
  // rows of E entries.
  int32_t *part = reinterpret_cast<int32_t *>(w.z_part);
  if (C == 1)
    return launch_k(h->pdl, dispatch_small_kernel, dim3(1), dim3(kThreads), smem, st, w.idx, T, A,
                    E, h->S, tile_m, w.inv, part, w.perm, w.counts, w.offsets, w.active,
                    w.n_active, w.tiles, w.n_tiles, usage, w.status);
  cudaError_t err = launch_k(h->pdl, dispatch_rank_kernel, dim3(C), dim3(kThreads), smem, st,
                             w.idx, A, E, w.inv, part, w.status);
  if (err == cudaSuccess)
    err = launch_k(h->pdl, dispatch_scan_kernel, dim3(1), dim3(kThreads), 0, st, T, E, h->S,
                   tile_m, C, part, w.counts, w.offsets, w.active, w.n_active, w.tiles,
                   w.n_tiles, usage);
  if (err == cudaSuccess)
    err = launch_k(h->pdl, dispatch_scatter_kernel, dim3(C), dim3(kThreads), 0, st, w.idx, A, E,
                   part, w.perm, w.inv);
  return err;
}

}  // namespace moe
