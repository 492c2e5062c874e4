// Tensor-core grouped expert GEMMs for large groups (prefill-sized).
//
// The "expert kernel" and "activation" phases of the fused-MoE path (page
// "Decode 吞吐专项实验分析报告", section "下一步 profiling 方向", item 3) for
// experts that hold many routed rows, where the grouped GEMM is bound by the
// tensor cores.  Grouping stays on the device (page "第 9 章 prefill：最大的瓶颈",
// sec. 9.9): tile lists come from the grouping kernels' counts, no host sync.
//
// One kernel, tc_gemm_pair_kernel, on 2-CTA clusters: one
// tcgen05.mma.cta_group::2 spans both SMs of a pair with the weights as M and
// the expert's token rows as N (the layout is described above the kernel).
// Operands are K-major with the 128-byte swizzle: TMA writes them in that
// layout and the UMMA shared-memory descriptors describe it (8-row groups
// 1024 bytes apart; the K step inside a 128-byte row advances the start
// address by 32 bytes).
//
// Every wait on an mbarrier is bounded; on a timeout the CTA records
// kStatusTimeout in the workspace status word, leaves its loops, waits
// (bounded again) for the TMA loads and MMAs it has issued, frees its tensor
// memory and returns.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace tcx;

constexpr int BN = 256, BK = 64;                        // accumulator columns, K per swizzled half
constexpr uint32_t kTmemCols = 512;                     // two 256-column accumulators
constexpr int kMaxLarge = 1024;

struct TcArgs {
  int T, H, E, I, k;
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* perm;
  const int32_t* active;
  const int32_t* tiles;
  const int* num_active;
  const int* num_large;
  const float* topk_w;
  uint16_t* h;
  void* partial;
  int partial_f32;
  int* status;
};

// Per-CTA copy of the large-expert tile metadata (shared memory).
struct TileMeta {
  int* tiles;   // [nlarge+1] m-tile prefix
  int* e;       // [nlarge] expert id
  int* m;       // [nlarge] rows
  int* off;     // [nlarge] first grouped row
};

// Tile t -> (expert, n-tile, m-tile) in (expert, n, m) order, so that
// co-running CTAs share an expert's weight tile through L2.
struct TileInfo {
  int e, m, off, mtile, ntile;
};

// `prefix` is the per-expert prefix of row tiles (md.tiles: 128-row m-tiles;
// the pair kernel's prefix of 256-row m-tile pairs).
__device__ __forceinline__ TileInfo decode_tile(const TileMeta& md, const int* prefix, int nlarge,
                                                int NTN, int t) {
  int lo = 0, hi = nlarge;  // find i with prefix[i]*NTN <= t < prefix[i+1]*NTN
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] * NTN <= t) lo = mid; else hi = mid;
  }
  TileInfo ti;
  const int mt = prefix[lo + 1] - prefix[lo];
  const int local = t - prefix[lo] * NTN;
  ti.e = md.e[lo];
  ti.m = md.m[lo];
  ti.off = md.off[lo];
  ti.ntile = local / mt;
  ti.mtile = local % mt;
  return ti;
}

// ------------------------------------------------------------------ CTA pairs
// The same GEMMs on 2-CTA clusters (launched with cluster dimension 2) with
// the weights as the MMA's M side: one tcgen05.mma.cta_group::2 per 16-wide
// K step computes 256 weight rows (128 in each CTA's shared and tensor
// memory) x N token rows (N <= 256, split N/2 + N/2 between the CTAs' shared
// memory; every CTA's accumulator holds all N columns for its own 128 weight
// rows).  A pair tile is (expert, block of 256 weight rows, block of up to
// 256 of the expert's token rows); the last token block of an expert uses the
// smallest N (a multiple of 16) that covers it, so groups are padded by at
// most 15 rows instead of to a whole 128- or 256-row tile.
//   gate/up   CTA r holds gate and up rows of j = j0 + 64r .. +63
//             interleaved (row 2jj = gate, 2jj+1 = up, one 4-D TMA box), so
//             a lane pair of the epilogue holds g and u of one (j, token)
//   down      CTA r holds output features d0 + 128r .. +127
// Each CTA stages 64 KB per 128-wide K stage (32 KB of weights, 32 KB of
// token rows, each as two 64-wide halves in the 128-byte swizzle layout),
// three stages: the MMA thread polls one barrier and commits once per eight
// MMAs, which keeps its issue loop ahead of the tensor pipe.
//   producers   one thread per CTA; both CTAs' TMA loads count on CTA 0's
//               full barrier (tx bytes of the pair), each CTA waits on its
//               own empty barrier
//   MMA issuer  CTA 0 only; tcgen05.commit multicast to both CTAs' empty /
//               accumulator-full barriers
//   epilogue    both CTAs, eight warps (two per TMEM lane quadrant, taking
//               alternate 32-column chunks), lane = weight row, column =
//               token: stores of consecutive j (h) or d (partials) across a
//               warp; one arrive per warp on CTA 0's accumulator-empty
//               barrier (16 per tile)
constexpr int NS2 = 3;
constexpr int kEpiWarps = 8;                             // epilogue warps 2 .. 2 + kEpiWarps - 1
constexpr int kEpiSets = kEpiWarps / 4;                  // warps per TMEM lane quadrant
constexpr int kEpiChunks = (BN / 32) / kEpiSets;          // 32-column chunks per warp and tile
constexpr int kThreadsPair = (2 + kEpiWarps) * 32;
constexpr int kPairRows = 128;                          // weight rows, token rows per CTA
// A stage is 128 K wide, two 64-wide halves of each operand: one barrier
// poll and one commit per eight MMAs
constexpr int kHalves = 2;
constexpr int kHalfBytes = kPairRows * BK * 2;            // 16 KB: one operand, one half
constexpr int kStageBytes2 = 2 * kHalves * kHalfBytes;    // 64 KB
constexpr size_t kSmemBytes2 = (size_t)NS2 * kStageBytes2 + 1024 + 256 + 5 * 4 * (kMaxLarge + 1);

__device__ __forceinline__ uint32_t idesc_pair(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)((2 * kPairRows) >> 4) << 24);
}
// token rows of a pair tile: 256, or the rest of the group rounded up to 16
__device__ __forceinline__ int pair_n(int rem) { return rem >= 256 ? 256 : (rem + 15) & ~15; }

template <bool kDown>
__global__ void __launch_bounds__(kThreadsPair, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const TcArgs a) {
  pdl_wait();   // programmatic dependent launch: the grouping and token rows are complete
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NS2 * kStageBytes2);
  uint64_t* empty = full + NS2;
  uint64_t* tfull = empty + NS2;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;   // after a timeout: the issued MMAs are complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  TileMeta md;
  md.tiles = reinterpret_cast<int*>(smem + NS2 * kStageBytes2 + 256);   // [nlarge+1] token-block prefix
  md.e = md.tiles + (kMaxLarge + 1);
  md.m = md.e + (kMaxLarge + 1);
  md.off = md.m + (kMaxLarge + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int cid = (int)blockIdx.x >> 1, ncl = (int)gridDim.x >> 1;
  const int nlarge = *a.num_large;
  const int nsmall = *a.num_active - nlarge;
  const int NW = kDown ? a.H / (2 * kPairRows) : a.I / kPairRows;   // weight blocks per expert
  const int K = kDown ? a.I : a.H;
  const int nkb = K / (kHalves * BK);

  for (int i = threadIdx.x; i < nlarge; i += kThreadsPair) {
    int e = a.active[nsmall + i];
    if (!bounds_ok((unsigned)e < (unsigned)a.E, a.status)) e = 0;
    int m = a.counts[e], off = a.offsets[e];
    if (!bounds_ok(off >= 0 && m >= 0 && off + m <= a.T * a.k, a.status)) m = 0, off = 0;
    md.e[i] = e;
    md.m[i] = m;
    md.off[i] = off;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int i = 0; i < nlarge; ++i) {
      md.tiles[i] = acc;
      acc += (md.m[i] + 2 * kPairRows - 1) / (2 * kPairRows);
    }
    md.tiles[nlarge] = acc;
  }
  __syncthreads();
  const int total = md.tiles[nlarge] * NW;
  if (cid >= total) return;   // uniform for the pair (both read the same counts)

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS2; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&tfull[b], 1); mbar_init(&tempty[b], 2 * kEpiWarps); }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  tc_fence_before();
  cluster_sync();   // both CTAs' barriers and tensor memory exist before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (each CTA)
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int p = cid; p < total && ok; p += ncl) {
        const TileInfo ti = decode_tile(md, md.tiles, nlarge, NW, p);   // ntile = weight block
        const int n = pair_n(ti.m - ti.mtile * 2 * kPairRows);
        const int brow = ti.off + ti.mtile * 2 * kPairRows + (int)rank * (n / 2);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % NS2;
          const uint32_t ph = (it / NS2) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1)) { ok = false; break; }
          if (rank == 0) mbar_expect_tx(&full[s], 2 * kStageBytes2);
          const uint32_t fb = map_to_rank(&full[s], 0);
          // [A half 0][A half 1][B half 0][B half 1]
          unsigned char* sA = smem + s * kStageBytes2;
#pragma unroll
          for (int hh = 0; hh < kHalves; ++hh) {
            const int x = (kb * kHalves + hh) * BK;
            if (kDown)
              tma_load_2d_pair(sA + hh * kHalfBytes, &tmA, x,
                               ti.e * a.H + ti.ntile * 2 * kPairRows + (int)rank * kPairRows, fb);
            else
              tma_load_4d_pair(sA + hh * kHalfBytes, &tmA, x, 0,
                               ti.ntile * kPairRows + (int)rank * (kPairRows / 2), ti.e, fb);
            tma_load_2d_pair(sA + (kHalves + hh) * kHalfBytes, &tmB, x, brow, fb);
          }
        }
        if (*(volatile int*)abort_flag) ok = false;
      }
      if (!ok) {
        atomicOr(abort_flag, 1);
        // after a timeout: the loads already issued land before either CTA
        // may exit (CTA 0's full barriers count both CTAs' bytes; the final
        // cluster barrier holds CTA 1 until CTA 0 is done)
        if (rank == 0)
          for (uint32_t j = it > (uint32_t)NS2 ? it - NS2 : 0; j < it; ++j) mbar_wait(&full[j % NS2], (j / NS2) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (CTA 0)
    if (lane == 0 && rank == 0) {
      uint32_t it = 0, lt = 0;
      bool ok = true;
      for (int p = cid; p < total && ok; p += ncl, ++lt) {
        const TileInfo ti = decode_tile(md, md.tiles, nlarge, NW, p);
        const uint32_t idesc = idesc_pair(pair_n(ti.m - ti.mtile * 2 * kPairRows));
        const uint32_t b = lt & 1;
        const uint32_t tph = (lt >> 1) & 1;
        if (!mbar_wait(&tempty[b], tph ^ 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + b * BN;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % NS2;
          const uint32_t ph = (it / NS2) & 1;
          if (!mbar_wait(&full[s], ph)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + s * kStageBytes2);
          const uint32_t sB = sA + kHalves * kHalfBytes;
#pragma unroll
          for (int hh = 0; hh < kHalves; ++hh)
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              umma_bf16_pair(tmem_d, umma_desc(sA + hh * kHalfBytes + kk * 32),
                             umma_desc(sB + hh * kHalfBytes + kk * 32), idesc,
                             (kb | hh | kk) != 0 ? 1u : 0u);
          umma_commit_pair(&empty[s]);   // both CTAs' stage s free once these MMAs are done
        }
        if (!ok) break;
        umma_commit_pair(&tfull[b]);     // both CTAs' accumulators ready
        if (*(volatile int*)abort_flag) ok = false;
      }
      if (!ok) {
        atomicOr(abort_flag, 1);
        // after a timeout: the MMAs already issued finish before the tensor
        // memory they write is freed
        umma_commit_pair(drain);
        mbar_wait(drain, 0);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (each CTA)
    // warp w reads TMEM lanes 32(w % 4) .. +31 and the 32-column chunks
    // v = kEpiSets * i + hc of the tile (hc = (warp - 2) / 4)
    const int q = warp & 3;
    const int hc = (warp - 2) >> 2;
    const uint32_t tempty0[2] = {map_to_rank(&tempty[0], 0), map_to_rank(&tempty[1], 0)};
    // down: slots and routing weights of this warp's columns (lane c of chunk
    // i: token 32(kEpiSets i + hc) + c), one tile ahead: the next tile's slot
    // ids are requested before this tile's accumulator wait and its routing
    // weights after this tile's stores, so neither load waits on the tile
    auto tile_cols = [&](int p, int& off0, int& nc) {
      const TileInfo t2 = decode_tile(md, md.tiles, nlarge, NW, p);
      const int r0 = t2.mtile * 2 * kPairRows;
      const int rem2 = t2.m - r0;
      const int n2 = pair_n(rem2);
      off0 = t2.off + r0;
      nc = rem2 < n2 ? rem2 : n2;
    };
    int nc_next = 0;   // token columns of the next tile
    auto load_slots = [&](int p, int (&f)[kEpiChunks]) {
      int off0;
      tile_cols(p, off0, nc_next);
#pragma unroll
      for (int i = 0; i < kEpiChunks; ++i) {
        const int c = 32 * (kEpiSets * i + hc) + lane;
        f[i] = c < nc_next ? __ldg(&a.perm[off0 + c]) : 0;
      }
    };
    auto load_weights = [&](int (&f)[kEpiChunks], float (&w)[kEpiChunks]) {
#pragma unroll
      for (int i = 0; i < kEpiChunks; ++i) {
        const int c = 32 * (kEpiSets * i + hc) + lane;
        if (!bounds_ok((unsigned)f[i] < (unsigned)(a.T * a.k), a.status)) f[i] = 0;
        w[i] = c < nc_next ? __ldg(&a.topk_w[f[i]]) : 0.f;
      }
    };
    int fl_next[kEpiChunks];
    float wl_next[kEpiChunks];
    if (kDown && cid < total) {
      load_slots(cid, fl_next);
      load_weights(fl_next, wl_next);
    }
    uint32_t lt = 0;
    for (int p = cid; p < total; p += ncl, ++lt) {
      const uint32_t b = lt & 1;
      const uint32_t tph = (lt >> 1) & 1;
      const TileInfo ti = decode_tile(md, md.tiles, nlarge, NW, p);
      const int tok0 = ti.mtile * 2 * kPairRows;     // first token row of the tile (within the group)
      const int rem = ti.m - tok0;                   // token rows left in the group (> 0)
      const int n = pair_n(rem);
      const int ncols = rem < n ? rem : n;           // token columns to store
      int fl[kEpiChunks];
      float wl[kEpiChunks];
      if (kDown) {
#pragma unroll
        for (int i = 0; i < kEpiChunks; ++i) {
          fl[i] = fl_next[i];
          wl[i] = wl_next[i];
        }
        if (p + ncl < total) load_slots(p + ncl, fl_next);
      }
      if (!warp_wait(&tfull[b], tph)) { atomicOr(abort_flag, 1); break; }
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + b * BN;
      // rolled: inlined copies of the 32-column body would crowd the
      // instruction cache that the producer and MMA threads share
#pragma unroll 1
      for (int i = 0; i < kEpiChunks; ++i) {
        const int c0 = 32 * (kEpiSets * i + hc);
        if (c0 >= ncols) break;   // uniform over the warp
        uint32_t y[32];
        tmem_ld32(tb + c0, y);
        tmem_wait_ld();
        if (!kDown) {
          // lane pair (2jj, 2jj+1) holds gate and up of one j for 32 tokens;
          // the even lane forms h for tokens 0-15 of the chunk, the odd lane
          // for tokens 16-31, each with one exchange per token
          const bool odd = lane & 1;
          const int j = ti.ntile * kPairRows + (int)rank * (kPairRows / 2) + 16 * q + (lane >> 1);
          uint16_t* hcol = a.h + (size_t)(ti.off + tok0 + c0 + (odd ? 16 : 0)) * a.I + j;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float send = __uint_as_float(odd ? y[c] : y[c + 16]);
            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
            const float g = odd ? recv : __uint_as_float(y[c]);
            const float u = odd ? __uint_as_float(y[c + 16]) : recv;
            if (c0 + c + (odd ? 16 : 0) < ncols) hcol[(size_t)c * a.I] = f2bf(silu(g) * u);
          }
        } else {
          const int d = ti.ntile * 2 * kPairRows + (int)rank * kPairRows + 32 * q + lane;
          // this chunk's slot and weight (selected, not indexed: no local memory)
          int fi = fl[0];
          float wi = wl[0];
#pragma unroll
          for (int j = 1; j < kEpiChunks; ++j)
            if (i == j) fi = fl[j], wi = wl[j];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int f = __shfl_sync(0xffffffffu, fi, c);
            const float w = __shfl_sync(0xffffffffu, wi, c);
            if (c0 + c < ncols) {
              const float val = w * __uint_as_float(y[c]);
              const size_t o = (size_t)f * a.H + d;
              if (a.partial_f32) reinterpret_cast<float*>(a.partial)[o] = val;
              else reinterpret_cast<uint16_t*>(a.partial)[o] = f2bf(val);
            }
          }
        }
      }
      if (kDown && p + ncl < total) load_weights(fl_next, wl_next);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0[b]);
      if (*(volatile int*)abort_flag) break;
    }
  }

  tc_fence_before();
  cluster_sync();   // no remote arrive or multicast commit is still aimed at either CTA
  if (threadIdx.x == 0 && *abort_flag) atomicOr(a.status, kStatusTimeout);
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kTmemCols));
  }
}

// Token rows in grouped order: xp[r] = x[perm[r] / k], one warp per row,
// 16-byte vectors (x stays in L2; this is one streaming write of S*H bf16).
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ perm, int S,
                                                          int H, int k, uint16_t* __restrict__ xp,
                                                          int* status) {
  pdl_wait();   // programmatic dependent launch: the permutation is complete
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (long long r = (long long)blockIdx.x * 8 + warp; r < S; r += (long long)gridDim.x * 8) {
    int f = perm[r];
    if (!bounds_ok((unsigned)f < (unsigned)S, status)) f = 0;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(f / k) * H);
    uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)r * H);
    for (int v = lane; v < H / 8; v += 32) dst[v] = src[v];
  }
}

// ------------------------------------------------------------------ host side
// 2-D bf16 tensor map over a row-major [rows, cols] matrix, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  return make_map_2d(m, base, rows, cols, 2, BK, box_rows, true);
}

}  // namespace

cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* perm, int S, int H, int k,
                               uint16_t* xp, int* status, cudaStream_t stream, int* launches) {
  const long long blocks = ((long long)S + 7) / 8;
  if (launches) *launches += 1;
  return launch_pdl(gather_rows_kernel, dim3((unsigned)(blocks < 4096 ? blocks : 4096)), dim3(256), 0, stream, x,
                    perm, S, H, k, xp, status);
}

cudaError_t launch_tc_gemm(const TcLaunch& p, bool down, cudaStream_t stream, int* launches) {
  TcArgs a{};
  a.T = p.T; a.H = p.H; a.E = p.E; a.I = p.I; a.k = p.k;
  a.counts = p.counts; a.offsets = p.offsets; a.perm = p.perm; a.active = p.active;
  a.tiles = p.tiles; a.num_active = p.num_active; a.num_large = p.num_large;
  a.topk_w = p.topk_w; a.h = p.h; a.partial = p.partial; a.partial_f32 = p.partial_f32 ? 1 : 0;
  a.status = p.status;
  const long long S = (long long)p.T * p.k;
  if (!down) {
    const cudaError_t gerr = launch_gather_rows(p.x, p.perm, (int)S, p.H, p.k, p.xp, p.status, stream, launches);
    if (gerr != cudaSuccess) return gerr;
  }
  // CTA pairs need at least two SMs; moe_forward sends every group to the
  // weight-streaming kernel on a device with fewer
  if (p.num_sms < 2) return cudaErrorInvalidConfiguration;
  CUtensorMap tmA, tmB;
  cudaError_t err;
  // A = weights (M), B = token rows (N)
  if (!down) {
    if (!make_map_gate_up_interleaved(&tmA, p.w_gate_up, p.E, p.I, p.H)) return cudaErrorInvalidValue;
    if (!make_map(&tmB, p.xp, S, p.H, kPairRows)) return cudaErrorInvalidValue;
  } else {
    if (!make_map(&tmA, p.w_down, (uint64_t)p.E * p.H, p.I, kPairRows)) return cudaErrorInvalidValue;
    if (!make_map(&tmB, p.h, S, p.I, kPairRows)) return cudaErrorInvalidValue;
  }
  const size_t smem = kSmemBytes2;
  auto kern = down ? tc_gemm_pair_kernel<true> : tc_gemm_pair_kernel<false>;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  // as many pairs as can be resident at once (persistent kernel)
  int clusters = 0;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.num_sms & ~1));
    cfg.blockDim = dim3(kThreadsPair);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (err != cudaSuccess) return err;
  }
  if (clusters > p.num_sms / 2) clusters = p.num_sms / 2;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  if (launches) *launches += 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * clusters));
  cfg.blockDim = dim3(kThreadsPair);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, a);
}

}  // namespace moe
