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

// Exclusive scan of four independent int fields over the 512 threads of a
// block; returns the prefixes and the block totals in *total.  `sw` is shared
// scratch of kWarps int4.
__device__ int4 block_exclusive_scan4(int4 v, int4* sw, int4* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int4 incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int nx = __shfl_up_sync(0xffffffffu, incl.x, o);
    const int ny = __shfl_up_sync(0xffffffffu, incl.y, o);
    const int nz = __shfl_up_sync(0xffffffffu, incl.z, o);
    const int nw = __shfl_up_sync(0xffffffffu, incl.w, o);
    if (lane >= o) { incl.x += nx; incl.y += ny; incl.z += nz; incl.w += nw; }
  }
  __syncthreads();
  if (lane == 31) sw[warp] = incl;
  __syncthreads();
  int4 base = make_int4(0, 0, 0, 0), tot = make_int4(0, 0, 0, 0);
  for (int w = 0; w < kWarps; ++w) {
    const int4 s = sw[w];
    if (w < warp) { base.x += s.x; base.y += s.y; base.z += s.z; base.w += s.w; }
    tot.x += s.x; tot.y += s.y; tot.z += s.z; tot.w += s.w;
  }
  *total = tot;
  return make_int4(base.x + incl.x - v.x, base.y + incl.y - v.y, base.z + incl.z - v.z,
                   base.w + incl.w - v.w);
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
// with counts[] in shared memory (E <= 1024); writes the global outputs and
// the offsets to s_off.  One four-field scan carries the offsets, the
// positions in both halves of the active list and the tile prefix.
__device__ void finish_scan(const int* s_counts, int E, int S, int large_threshold, int tile_rows,
                            int32_t* counts, int32_t* offsets, int32_t* active, int32_t* tiles,
                            WsHeader* hdr, int* s_off, int4* sw) {
  // each thread owns experts 2t, 2t+1
  const int e0 = 2 * threadIdx.x, e1 = e0 + 1;
  const int c0 = e0 < E ? s_counts[e0] : 0, c1 = e1 < E ? s_counts[e1] : 0;
  // active lists: small groups first, then large groups
  const int sm0 = (c0 > 0 && c0 < large_threshold), sm1 = (c1 > 0 && c1 < large_threshold);
  const int lg0 = (c0 >= large_threshold && c0 > 0), lg1 = (c1 >= large_threshold && c1 > 0);
  // row tiles of the large groups
  const int t0 = lg0 ? (c0 + tile_rows - 1) / tile_rows : 0;
  const int t1 = lg1 ? (c1 + tile_rows - 1) / tile_rows : 0;
  int4 tot;
  const int4 pre = block_exclusive_scan4(make_int4(c0 + c1, sm0 + sm1, lg0 + lg1, t0 + t1), sw, &tot);
  if (e0 < E) { s_off[e0] = pre.x; offsets[e0] = pre.x; counts[e0] = c0; }
  if (e1 < E) { s_off[e1] = pre.x + c0; offsets[e1] = pre.x + c0; counts[e1] = c1; }
  if (threadIdx.x == 0) offsets[E] = S;
  const int nsmall = tot.y, nlarge = tot.z;
  if (sm0) active[pre.y] = e0;
  if (sm1) active[pre.y + sm0] = e1;
  if (lg0) active[nsmall + pre.z] = e0;
  if (lg1) active[nsmall + pre.z + lg0] = e1;
  if (lg0) tiles[pre.z] = pre.w;
  if (lg1) tiles[pre.z + lg0] = pre.w + t0;
  if (threadIdx.x == 0) {
    tiles[nlarge] = tot.w;
    hdr->num_active = nsmall + nlarge;
    hdr->num_large = nlarge;
  }
}

// Largest S that group_single_block serves.
constexpr int kSingleMaxChunks = 8;
constexpr int kSingleMaxSlots = kSingleMaxChunks * kThreads;

// Dynamic shared memory (ints) that group_single_block needs (an even number).
__host__ __device__ inline size_t single_block_smem_ints(int E, int S) {
  (void)S;
  return (size_t)E * (2 + kWarps);
}

// The whole grouping for S <= kSingleMaxSlots slots in one 512-thread block,
// with few block barriers (this often runs alone on one SM at the end of the
// router, where every barrier and every cold instruction line is latency).
// Warp w owns the contiguous slice of slots [w*L, (w+1)*L), L a multiple of
// 32, and walks it in rounds of 32 ascending slots: __match_any gives each
// slot its rank among equal experts in the round, and the warp's own table
// row tab[w][e] (read and advanced by each group's first lane) adds the
// earlier rounds.  A scan down the warps per expert then gives each warp's
// base, the expert offsets come from finish_scan, and position = offset[e] +
// base[w][e] + rank in the slice: ascending slot order within every expert.
// `dyn` holds single_block_smem_ints(E, S) ints, `sw` kWarps int4.
// `zero`/`nzero`: an int region cleared on the way (counters used later in
// the same call).
__device__ void group_single_block(const int32_t* __restrict__ idx, int S, int E,
                                   int large_threshold, int tile_rows, int32_t* counts,
                                   int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                                   int32_t* active, int32_t* tiles, void* ws, int* dyn, int4* sw,
                                   int* zero, int nzero) {
  int* s_cnt = dyn;              // [E] totals
  int* s_off = s_cnt + E;        // [E] offsets
  int* tab = s_off + E;          // [kWarps][E] per-warp counts, then bases
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rounds = (S + kThreads - 1) / kThreads;   // <= kSingleMaxChunks
  const int f0 = warp * rounds * 32 + lane;           // slot of round 0
  int ev[kSingleMaxChunks];      // all loads in flight before any use
#pragma unroll
  for (int r = 0; r < kSingleMaxChunks; ++r) {
    const int f = f0 + 32 * r;
    ev[r] = (r < rounds && f < S) ? __ldcg(&idx[f]) : -1;
  }
  for (int i = threadIdx.x; i < nzero; i += kThreads) zero[i] = 0;
  int* row = tab + warp * E;
  for (int e = lane; e < E; e += 32) row[e] = 0;
  __syncwarp();
  bool bad = false;
  int rel[kSingleMaxChunks];
#pragma unroll
  for (int r = 0; r < kSingleMaxChunks; ++r) {
    rel[r] = -1;
    if (r >= rounds) continue;   // uniform over the block
    const int f = f0 + 32 * r;
    const int e = ev[r];
    const bool valid = e >= 0 && e < E;
    if (f < S && !valid) bad = true;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
    const int first = __ffs(peers) - 1;
    int before = 0;
    if (valid && lane == first) {
      before = row[e];
      row[e] = before + __popc(peers);
    }
    before = __shfl_sync(0xffffffffu, before, first);
    if (valid) rel[r] = before + __popc(peers & lanemask_lt());
    __syncwarp();   // the table row is read again in the next round
  }
  if (bad) set_status(ws, kStatusBadExpert);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kThreads) {
    int s = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int c = tab[w * E + e];
      tab[w * E + e] = s;
      s += c;
    }
    s_cnt[e] = s;
  }
  __syncthreads();
  finish_scan(s_cnt, E, S, large_threshold, tile_rows, counts, offsets, active, tiles, hdr, s_off,
              sw);
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kSingleMaxChunks; ++r) {
    if (rel[r] < 0) continue;
    const int f = f0 + 32 * r;
    const int pos = s_off[ev[r]] + row[ev[r]] + rel[r];
    perm[pos] = f;
    inv_perm[f] = pos;
  }
}

}  // namespace
}  // namespace grouping
}  // namespace moe
