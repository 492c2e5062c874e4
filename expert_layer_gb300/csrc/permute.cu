// Expert grouping of the routed slots, kept on the device (page "第 9 章
// prefill：最大的瓶颈", sec. 9.9: the fused path groups by expert on the GPU
// instead of a per-layer cudaStreamSynchronize; sec. 9.5: no per-group row
// ceiling, so nothing is ever dropped).
//
// The arithmetic of the grouping is in grouping.cuh; this file holds the
// standalone kernels (one block for S <= 4096 slots, three passes above).
//
// Alongside the grouping the scan step writes the list of active experts for
// the expert GEMMs: experts with count < large_threshold first (ascending),
// then the others (ascending), plus the prefix sum of row tiles of the latter.
#include "common.cuh"
#include "grouping.cuh"
#include "kernels.h"

namespace moe {

namespace {

using grouping::kThreads;
using grouping::kWarps;
using grouping::block_stable_rank;
using grouping::finish_scan;

// ---------------------------------------------------------------- one block
__global__ void __launch_bounds__(kThreads) permute_single_kernel(
    const int32_t* __restrict__ idx, int S, int E, int large_threshold, int tile_rows,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv_perm, int32_t* __restrict__ active, int32_t* __restrict__ tiles,
    void* ws) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int smem[];
  __shared__ int4 sw[kWarps];
  grouping::group_single_block(idx, S, E, large_threshold, tile_rows, counts, offsets, perm,
                               inv_perm, active, tiles, ws, smem, sw, nullptr, 0);
}

// ---------------------------------------------------------------- many blocks
// Largest dynamic shared memory of the scan kernel's staged path.
constexpr size_t kScanSmemMax = 160 * 1024;

__global__ void __launch_bounds__(kThreads) permute_block_rank_kernel(
    const int32_t* __restrict__ idx, int S, int E, int32_t* __restrict__ blk_cnt,
    int32_t* __restrict__ lrank, void* ws) {
  pdl_wait();
  extern __shared__ int tab[];  // [kWarps][E]
  const int f = blockIdx.x * kThreads + threadIdx.x;
  int e = -1;
  if (f < S) e = idx[f];
  const bool valid = f < S && e >= 0 && e < E;
  if (f < S && !valid) set_status(ws, kStatusBadExpert);
  const int r = block_stable_rank(e, valid, E, tab, nullptr, blk_cnt + (size_t)blockIdx.x * E);
  if (f < S) lrank[f] = r;
}

// One block.  When the per-block counts fit in shared memory (`staged`) they
// are copied there with coalesced 16-byte loads first, so the per-expert walks
// over the blocks run on shared memory instead of one global load after
// another; with E <= kThreads each expert's walk is also split into
// P = kThreads / E contiguous ranges of blocks, one thread each (integer sums:
// the split changes no result).
__global__ void __launch_bounds__(kThreads) permute_scan_kernel(
    const int32_t* __restrict__ blk_cnt, int nblk, int S, int E, int large_threshold,
    int tile_rows, int32_t* __restrict__ blk_base, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ active, int32_t* __restrict__ tiles,
    void* ws, int staged) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int smem[];
  int* s_cnt = smem;       // [E]
  int* s_off = s_cnt + E;  // [E]
  int* s_blk = s_off + E;  // [nblk][E] when staged
  __shared__ int4 sw[kWarps];
  __shared__ int s_part[kThreads];   // [P][E]: sums of each thread's range of blocks
  const size_t n = (size_t)nblk * E;
  const bool vec = (n & 3) == 0 && (E & 3) == 0;   // s_blk starts 16-byte aligned when E % 4 == 0
  if (staged) {
    if (vec) {
      for (size_t i = threadIdx.x; i < n / 4; i += kThreads)
        reinterpret_cast<int4*>(s_blk)[i] = __ldcg(reinterpret_cast<const int4*>(blk_cnt) + i);
    } else {
      for (size_t i = threadIdx.x; i < n; i += kThreads) s_blk[i] = __ldcg(&blk_cnt[i]);
    }
  }
  __syncthreads();
  const bool split = staged && E <= kThreads;
  const int P = split ? kThreads / E : 1;
  const int t = threadIdx.x, pe = t % E, pp = t / E;
  const int b0 = pp * nblk / P, b1 = (pp + 1) * nblk / P;
  if (split) {
    if (t < P * E) {
      int s = 0;
      for (int b = b0; b < b1; ++b) s += s_blk[(size_t)b * E + pe];
      s_part[t] = s;
    }
    __syncthreads();
    for (int e = t; e < E; e += kThreads) {
      int s = 0;
      for (int q = 0; q < P; ++q) s += s_part[q * E + e];
      s_cnt[e] = s;
    }
  } else {
    const int32_t* src = staged ? s_blk : blk_cnt;
    for (int e = t; e < E; e += kThreads) {
      int s = 0;
      for (int b = 0; b < nblk; ++b) s += src[(size_t)b * E + e];
      s_cnt[e] = s;
    }
  }
  __syncthreads();
  finish_scan(s_cnt, E, S, large_threshold, tile_rows, counts, offsets, active, tiles,
              reinterpret_cast<WsHeader*>(ws), s_off, sw);
  __syncthreads();
  if (split) {
    if (t < P * E) {
      int s = s_off[pe];
      for (int q = 0; q < pp; ++q) s += s_part[q * E + pe];
      for (int b = b0; b < b1; ++b) {
        const int c = s_blk[(size_t)b * E + pe];
        s_blk[(size_t)b * E + pe] = s;
        s += c;
      }
    }
  } else if (staged) {
    for (int e = t; e < E; e += kThreads) {
      int s = s_off[e];
      for (int b = 0; b < nblk; ++b) {
        const int c = s_blk[(size_t)b * E + e];
        s_blk[(size_t)b * E + e] = s;
        s += c;
      }
    }
  } else {
    for (int e = t; e < E; e += kThreads) {
      int s = s_off[e];
      for (int b = 0; b < nblk; ++b) {
        blk_base[(size_t)b * E + e] = s;
        s += blk_cnt[(size_t)b * E + e];
      }
    }
  }
  if (staged) {
    __syncthreads();
    if (vec) {
      for (size_t i = threadIdx.x; i < n / 4; i += kThreads)
        reinterpret_cast<int4*>(blk_base)[i] = reinterpret_cast<const int4*>(s_blk)[i];
    } else {
      for (size_t i = threadIdx.x; i < n; i += kThreads) blk_base[i] = s_blk[i];
    }
  }
}

__global__ void __launch_bounds__(kThreads) permute_scatter_kernel(
    const int32_t* __restrict__ idx, int S, int E, const int32_t* __restrict__ blk_base,
    const int32_t* __restrict__ lrank, int32_t* __restrict__ perm, int32_t* __restrict__ inv_perm) {
  pdl_wait();
  const int f = blockIdx.x * kThreads + threadIdx.x;
  if (f >= S) return;
  const int e = idx[f];
  if (e < 0 || e >= E) return;
  const int pos = blk_base[(size_t)blockIdx.x * E + e] + lrank[f];
  perm[pos] = f;
  inv_perm[f] = pos;
}

}  // namespace

cudaError_t launch_permute(const int32_t* idx, int T, int E, int k, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv_perm, void* ws,
                           const WsLayout& L, int large_threshold, int tile_rows,
                           cudaStream_t stream, int* launches) {
  const int S = T * k;
  int32_t* active = ws_ptr<int32_t>(ws, L.active);
  int32_t* tiles = ws_ptr<int32_t>(ws, L.tiles);
  if (S <= grouping::kSingleMaxSlots) {
    const size_t smem = sizeof(int) * grouping::single_block_smem_ints(E, S);
    cudaError_t err = cudaFuncSetAttribute(permute_single_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    if (launches) *launches += 1;
    return launch_pdl(permute_single_kernel, dim3(1), dim3(kThreads), smem, stream, idx, S, E, large_threshold,
                      tile_rows, counts, offsets, perm, inv_perm, active, tiles, ws);
  }
  int32_t* blk_cnt = ws_ptr<int32_t>(ws, L.blk_cnt);
  int32_t* blk_base = ws_ptr<int32_t>(ws, L.blk_base);
  int32_t* lrank = ws_ptr<int32_t>(ws, L.lrank);
  const size_t smem_tab = sizeof(int) * (size_t)E * kWarps;
  cudaError_t err = cudaFuncSetAttribute(permute_block_rank_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_tab);
  if (err != cudaSuccess) return err;
  if (launches) *launches += 3;
  err = launch_pdl(permute_block_rank_kernel, dim3(L.nblk), dim3(kThreads), smem_tab, stream, idx, S, E, blk_cnt,
                   lrank, ws);
  if (err != cudaSuccess) return err;
  const size_t scan_smem_staged = sizeof(int) * (2 * (size_t)E + (size_t)L.nblk * E);
  const int staged = scan_smem_staged <= kScanSmemMax ? 1 : 0;
  const size_t scan_smem = staged ? scan_smem_staged : sizeof(int) * 2 * (size_t)E;
  err = cudaFuncSetAttribute(permute_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)scan_smem);
  if (err != cudaSuccess) return err;
  err = launch_pdl(permute_scan_kernel, dim3(1), dim3(kThreads), scan_smem, stream, (const int32_t*)blk_cnt,
                   L.nblk, S, E, large_threshold, tile_rows, blk_base, counts, offsets, active, tiles, ws, staged);
  if (err != cudaSuccess) return err;
  return launch_pdl(permute_scatter_kernel, dim3(L.nblk), dim3(kThreads), 0, stream, idx, S, E,
                    (const int32_t*)blk_base, (const int32_t*)lrank, perm, inv_perm);
}

}  // namespace moe
