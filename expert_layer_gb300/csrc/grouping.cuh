// Stable expert grouping of routed slots by one 512-thread block, shared by
// the grouping kernels and the fused small-batch router.
//
//   counts[e]   = #{f : idx[f] == e}
//   offsets[e]  = exclusive prefix sum of counts (offsets[E] = S)
//   perm[r]     = slots sorted by expert, ascending f within an expert
//   inv_perm[f] = position of f in perm
//
// Stability comes from processing slots in 512-slot blocks in ascending f:
// within a warp, __match_any gives each slot its rank among equal experts; a
// per-(warp, expert) table scanned in warp order extends that to the block;
// block bases scanned in block order extend it to the batch.  All integer,
// all bit-exact.
#pragma once

#include "common.cuh"

namespace moe {
namespace grouping {
namespace {  // internal linkage: each translation unit gets its own copy

constexpr int kThreads = kPermBlock;   // one slot per thread per block
constexpr int kWarps = kThreads / 32;  // 16

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Exclusive scan over the 512 threads of a block; returns the prefix and the
// block total in *total.  `sw` is shared scratch of kWarps ints.
__device__ int block_exclusive_scan(int v, int* sw, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  __syncthreads();
  if (lane == 31) sw[warp] = incl;
  __syncthreads();
  int base = 0, tot = 0;
  for (int w = 0; w < kWarps; ++w) {
    const int s = sw[w];
    if (w < warp) base += s;
    tot += s;
  }
  *total = tot;
  return base + incl - v;
}

// Rank of each slot of one 512-slot block among equal experts, in f order.
// tab is [kWarps][E] shared; on return tab[w][e] is the number of slots with
// expert e in warps < w of this block (plus `base[e]` if given), and
// block_cnt[e] (if given) the block's count.  Returns the slot's rank within
// the block or -1 for an invalid slot.
__device__ int block_stable_rank(int e, bool valid, int E, int* tab, const int* base,
                                 int* block_cnt) {
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kWarps * E; i += kThreads) tab[i] = 0;
  __syncthreads();
  const int key = valid ? e : -1;
  const unsigned peers = __match_any_sync(0xffffffffu, key);
  const int rank_in_warp = __popc(peers & lanemask_lt());
  if (valid && rank_in_warp == 0) tab[warp * E + e] = __popc(peers);
  __syncthreads();
  for (int ee = threadIdx.x; ee < E; ee += kThreads) {
    int s = base ? base[ee] : 0;
    const int s0 = s;
    for (int w = 0; w < kWarps; ++w) {
      const int c = tab[w * E + ee];
      tab[w * E + ee] = s;
      s += c;
    }
    if (block_cnt) block_cnt[ee] = s - s0;
  }
  __syncthreads();
  return valid ? tab[warp * E + e] + rank_in_warp : -1;
}

// Counts -> offsets, active list, tile prefix.  Called by one 512-thread block
// with counts[] in shared memory; writes the global outputs.
__device__ void finish_scan(const int* s_counts, int E, int S, int large_threshold, int tile_rows,
                            int32_t* counts, int32_t* offsets, int32_t* active, int32_t* tiles,
                            WsHeader* hdr, int* s_off, int* sw) {
  // offsets: each thread owns experts 2t, 2t+1
  const int e0 = 2 * threadIdx.x, e1 = e0 + 1;
  const int c0 = e0 < E ? s_counts[e0] : 0, c1 = e1 < E ? s_counts[e1] : 0;
  int tot;
  const int pre = block_exclusive_scan(c0 + c1, sw, &tot);
  if (e0 < E) { s_off[e0] = pre; offsets[e0] = pre; counts[e0] = c0; }
  if (e1 < E) { s_off[e1] = pre + c0; offsets[e1] = pre + c0; counts[e1] = c1; }
  if (threadIdx.x == 0) offsets[E] = S;
  // active lists: small groups first, then large groups
  const int sm0 = (c0 > 0 && c0 < large_threshold), sm1 = (c1 > 0 && c1 < large_threshold);
  const int lg0 = (c0 >= large_threshold && c0 > 0), lg1 = (c1 >= large_threshold && c1 > 0);
  int nsmall, nlarge;
  const int ps = block_exclusive_scan(sm0 + sm1, sw, &nsmall);
  if (sm0) active[ps] = e0;
  if (sm1) active[ps + sm0] = e1;
  const int pl = block_exclusive_scan(lg0 + lg1, sw, &nlarge);
  if (lg0) active[nsmall + pl] = e0;
  if (lg1) active[nsmall + pl + lg0] = e1;
  // row-tile prefix over the large groups, in list order
  const int t0 = lg0 ? (c0 + tile_rows - 1) / tile_rows : 0;
  const int t1 = lg1 ? (c1 + tile_rows - 1) / tile_rows : 0;
  int ntiles;
  const int pt = block_exclusive_scan(t0 + t1, sw, &ntiles);
  if (lg0) tiles[pl] = pt;
  if (lg1) tiles[pl + lg0] = pt + t0;
  if (threadIdx.x == 0) {
    tiles[nlarge] = ntiles;
    hdr->num_active = nsmall + nlarge;
    hdr->num_large = nlarge;
  }
}

// Dynamic shared memory (ints) that group_single_block needs.
__host__ __device__ inline size_t single_block_smem_ints(int E) { return (size_t)E * (3 + kWarps); }

// The whole grouping for S slots in one 512-thread block.  `dyn` holds
// single_block_smem_ints(E) ints, `sw` kWarps ints.  `zero`/`nzero`: an int
// region cleared on the way (counters used later in the same call).
__device__ void group_single_block(const int32_t* __restrict__ idx, int S, int E,
                                   int large_threshold, int tile_rows, int32_t* counts,
                                   int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                                   int32_t* active, int32_t* tiles, void* ws, int* dyn, int* sw,
                                   int* zero, int nzero) {
  int* s_cnt = dyn;              // [E]
  int* s_run = s_cnt + E;        // [E]
  int* tab = s_run + E;          // [kWarps][E], then [E] block counts
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  for (int i = threadIdx.x; i < nzero; i += kThreads) zero[i] = 0;
  for (int e = threadIdx.x; e < E; e += kThreads) s_cnt[e] = 0;
  __syncthreads();
  bool bad = false;
  for (int f = threadIdx.x; f < S; f += kThreads) {
    const int e = __ldcg(&idx[f]);
    if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1); else bad = true;
  }
  if (bad) set_status(ws, kStatusBadExpert);
  __syncthreads();
  finish_scan(s_cnt, E, S, large_threshold, tile_rows, counts, offsets, active, tiles, hdr, s_run,
              sw);
  __syncthreads();
  int* s_blk = tab + kWarps * E;  // [E]
  for (int c0 = 0; c0 < S; c0 += kThreads) {
    const int f = c0 + threadIdx.x;
    int e = -1;
    if (f < S) e = __ldcg(&idx[f]);
    const bool valid = f < S && e >= 0 && e < E;
    const int pos = block_stable_rank(e, valid, E, tab, s_run, s_blk);
    if (valid) { perm[pos] = f; inv_perm[f] = pos; }
    __syncthreads();  // every thread has read its position from tab
    for (int ee = threadIdx.x; ee < E; ee += kThreads) s_run[ee] += s_blk[ee];
    __syncthreads();
  }
}

}  // namespace
}  // namespace grouping
}  // namespace moe
