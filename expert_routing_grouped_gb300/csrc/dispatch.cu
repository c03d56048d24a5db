// dispatch.cu -- step 3 of the layer: group the T*k assignments by expert.
//
// A counting sort, as the pages do it (Colibri C + cuBLASLt tutorial,
// cf-1.com, §3.3 Step 3: per-expert counts, a prefix sum into offsets, then a
// scatter, in place and with no allocation): a shared-memory histogram, a
// block-wide exclusive scan, and a stable scatter.  Assignment a = t*k + j goes
// to perm[offsets[e] + r], where r counts the assignments of expert e with a
// smaller a, so each expert's group lists its tokens in ascending order.
//
// One CTA of 1024 threads.  Assignments are taken in chunks of 1024 in
// ascending order; inside a chunk, __match_any_sync ranks a lane among the
// lanes of its warp holding the same expert, and a per-(warp, expert) count
// table turns that into a rank across the chunk.
//
// Also produced here, for the expert kernels: the ascending list of experts
// that received tokens (the shared expert, id E, appended last), and the
// tensor-core token blocks: one entry per tile_m tokens of every non-empty
// group (the shared expert's included), costliest first.
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

__global__ void __launch_bounds__(kThreads, 1) dispatch_kernel(
    const int32_t *__restrict__ idx, int T, int k, int E, int n_shared, int tile_m,
    int32_t *__restrict__ counts, int32_t *__restrict__ offsets, int32_t *__restrict__ perm,
    int32_t *__restrict__ inv, int32_t *__restrict__ active, int32_t *__restrict__ n_active,
    int32_t *__restrict__ tiles, int32_t *__restrict__ n_tiles, int32_t *__restrict__ status,
    unsigned long long *__restrict__ usage) {
  pdl_enter();
  idx = after_wait(idx);
  counts = after_wait(counts);
  offsets = after_wait(offsets);
  perm = after_wait(perm);
  inv = after_wait(inv);
  active = after_wait(active);
  n_active = after_wait(n_active);
  tiles = after_wait(tiles);
  n_tiles = after_wait(n_tiles);
  status = after_wait(status);
  usage = after_wait(usage);
  extern __shared__ int smem[];
  int *cnt = smem;                 // [E]
  int *base = cnt + E;             // [E]
  int *wc = base + E;              // [32][E]
  __shared__ int warp_sums[32];
  __shared__ int total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int A = T * k;

  for (int e = tid; e < E; e += kThreads) cnt[e] = 0;
  for (int i = tid; i < 32 * E; i += kThreads) wc[i] = 0;
  __syncthreads();
  int bad = 0;
  for (int a = tid; a < A; a += kThreads) {
    const int e = idx[a];
    if (e == -1) continue;   // a slot the top-p trim dropped: no assignment
    if (e < 0 || e >= E) {
      bad = 1;
      continue;
    }
    atomicAdd(&cnt[e], 1);
  }
  if (bad) atomicExch(status, kStatusBadExpert);
  __syncthreads();

  // offsets = exclusive scan of counts (E <= 1024: one expert per thread).
  const int c = (tid < E) ? cnt[tid] : 0;
  const int off = block_exclusive_scan(c, warp_sums, &total);
  if (tid < E) {
    counts[tid] = c;
    offsets[tid] = off;
    base[tid] = off;
    if (usage && c) usage[tid] += (unsigned long long)c;   // one writer per expert
  }
  if (tid == 0) offsets[E] = total;
  __syncthreads();

  // Stable scatter, chunk by chunk.
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int c0 = 0; c0 < A; c0 += kThreads) {
    const int a = c0 + tid;
    int e = (a < A) ? idx[a] : E;
    if (e < 0 || e >= E) e = E;                  // dropped or invalid ids are not placed
    if (a < A && e == E) inv[a] = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    if (e < E && (peers & lt_mask) == 0) wc[warp * E + e] = __popc(peers);
    __syncthreads();
    if (tid < E) {
      int run = base[tid];
      for (int w = 0; w < 32; ++w) {
        const int n = wc[w * E + tid];
        wc[w * E + tid] = run;
        run += n;
      }
      base[tid] = run;
    }
    __syncthreads();
    if (e < E) {
      const int pos = wc[warp * E + e] + rank;
      perm[pos] = a;
      inv[a] = pos;
    }
    __syncthreads();
    for (int i = tid; i < 32 * E; i += kThreads) wc[i] = 0;
    __syncthreads();
  }

  // Ascending list of non-empty experts; the shared expert (id E) goes last.
  const int flag = (tid < E && c > 0) ? 1 : 0;
  const int apos = block_exclusive_scan(flag, warp_sums, &total);
  if (flag) active[apos] = tid;
  if (tid == 0) {
    int na = total;
    if (n_shared) active[na++] = E;
    *n_active = na;
  }
  // Tensor-core token blocks, (expert << 16 | block index) in one int32,
  // ordered by cost so that a round-robin deal of tiles over the CTAs gives
  // each a similar mix: every full block (routed experts in expert order, then
  // the shared expert's), then the partial last blocks by size class
  // (> 128 tokens, > 64, > 32, the rest).
  const int nfull = (tid < E) ? c / tile_m : 0;
  const int rem = (tid < E) ? c - nfull * tile_m : 0;
  const int base_pos = block_exclusive_scan(nfull, warp_sums, &total);
  for (int i = 0; i < nfull; ++i) tiles[base_pos + i] = (tid << 16) | i;
  int ntot = total;
  const int s_full = n_shared ? T / tile_m : 0, s_rem = n_shared ? T - s_full * tile_m : 0;
  if (tid == 0)
    for (int i = 0; i < s_full; ++i) tiles[ntot + i] = (E << 16) | i;
  ntot += s_full;
  for (int cls = 0; cls < 4; ++cls) {
    const int lo = cls == 0 ? 128 : cls == 1 ? 64 : cls == 2 ? 32 : 0;
    const int hi = cls == 0 ? tile_m : cls == 1 ? 128 : cls == 2 ? 64 : 32;
    const int f = (rem > lo && rem <= hi) ? 1 : 0;
    const int pos = block_exclusive_scan(f, warp_sums, &total);
    if (f) tiles[ntot + pos] = (tid << 16) | nfull;
    ntot += total;
    if (s_rem > lo && s_rem <= hi) {
      if (tid == 0) tiles[ntot] = (E << 16) | s_full;
      ntot += 1;
    }
  }
  if (tid == 0) n_tiles[0] = ntot;
}

}  // namespace

cudaError_t launch_dispatch(const moe_handle *h, int T, int tile_m, unsigned long long *usage,
                            cudaStream_t st) {
  const size_t smem = (size_t)(2 + 32) * h->E * sizeof(int);
  static bool attr_set = false;   // per process; the attribute is per function
  if (!attr_set) {
    cudaError_t err = cudaFuncSetAttribute(dispatch_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)((2 + 32) * kMaxExperts * sizeof(int)));
    if (err != cudaSuccess) return err;
    attr_set = true;
  }
  const moe::Workspace &w = h->ws;
  return launch_k(h->pdl, dispatch_kernel, dim3(1), dim3(kThreads), smem, st, w.idx, T, h->k, h->E,
                  h->S, tile_m, w.counts, w.offsets, w.perm, w.inv, w.active, w.n_active, w.tiles,
                  w.n_tiles, w.status, usage);
}

}  // namespace moe
