// Router: "MoE gate" GEMV + "topk" with renormalised weights (page "Decode
// 吞吐专项实验分析报告", section "下一步 profiling 方向", items 2-3).
//
// logit[t,e] = sum_h x[t,h] * gate_w[e,h] (+ bias[e]).  The ranking key is the
// logit (larger first, lower expert index first on equal logits); the weights
// are the softmax over all E experts renormalised over the k selected, which
// equals exp(l_s - l_max) / sum_{s'} exp(l_s' - l_max) over the selected set.
//
// Certified ranking.  Logits accumulate in fp32.  bf16 x bf16 products are
// exact in fp32 (barring underflow, bounded separately), so the only error is
// the summation: with every product passing through at most n roundings the
// error is at most gamma_n * sum_h |x_h w_h| <= gamma_n * ||x|| * ||w_e||
// (Cauchy-Schwarz), gamma_n = n*u/(1-n*u), u = 2^-24.  Per token we take the
// uniform bound delta = gamma_n ||x|| max_e ||w_e|| (1 + 2^-10) + 2^-22 max|l|
// + H 2^-149.  Adjacent ranks closer than 2*delta inside the top region are
// recomputed in fp64 (exact products, ~1e-16 relative sums) and re-ranked, so
// the selected experts and their order equal those of the exact logits.
#include <float.h>
#include <limits.h>

#include "common.cuh"
#include "grouping.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kCandCap = 64;  // candidates a warp can hold while certifying

__host__ __device__ inline float gamma_bound(int n) {
  const double u = 5.9604644775390625e-08;  // 2^-24
  return (float)(n * u / (1.0 - n * u));
}

// Exact-product fp64 dot of two bf16 rows of length H (H % 8 == 0), whole warp.
// Every lane returns the same value (xor butterfly).
__device__ double warp_dot_f64(const uint16_t* __restrict__ a, const uint16_t* __restrict__ b,
                               int H) {
  const int lane = threadIdx.x & 31;
  double s = 0.0;
  for (int h = lane * 8; h < H; h += 256) {
    uint4 va = *reinterpret_cast<const uint4*>(a + h);
    uint4 vb = *reinterpret_cast<const uint4*>(b + h);
    const uint32_t wa[4] = {va.x, va.y, va.z, va.w};
    const uint32_t wb[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s = fma((double)bf16lo(wa[i]), (double)bf16lo(wb[i]), s);
      s = fma((double)bf16hi(wa[i]), (double)bf16hi(wb[i]), s);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

struct WarpScratch {
  int cand_e[kCandCap];
  float cand_v[kCandCap];
  double key[kCandCap];
  float ex[32];
  double kmax;
};

// Two logits whose fp32 values differ by more than this are ordered like the
// exact logits (each is within delta of its exact value).
__device__ __forceinline__ float cert_threshold(float delta) { return 2.0f * delta * 1.001f; }

// Sort key of a logit: NaN ranks below every number.
__device__ __forceinline__ float rank_key(float v) { return v != v ? -INFINITY : v; }

// (v, e) ordering: larger value first, lower index first on equal values.
__device__ __forceinline__ bool better(float v, int e, float bv, int be) {
  return v > bv || (v == bv && e < be);
}

// Sorted candidates for E > 128: cand_e/cand_v[r] = the expert of rank r
// (larger logit first, lower index first on equal logits) for
// r < min(E, kCandCap).  Each of the nthr cooperating threads (index tid)
// ranks its experts by counting the experts that come before it.  The
// caller synchronises the cooperating threads before using the result.
__device__ void rank_candidates(const float* L, int E, WarpScratch& sc, int tid, int nthr) {
  for (int e = tid; e < E; e += nthr) {
    const float v = rank_key(L[e]);
    int r = 0;
    int j = 0;
    for (; j + 4 <= E; j += 4) {
      const float4 q = *reinterpret_cast<const float4*>(L + j);
      const float q0 = rank_key(q.x), q1 = rank_key(q.y), q2 = rank_key(q.z), q3 = rank_key(q.w);
      r += (q0 > v || (q0 == v && j < e)) + (q1 > v || (q1 == v && j + 1 < e)) +
           (q2 > v || (q2 == v && j + 2 < e)) + (q3 > v || (q3 == v && j + 3 < e));
    }
    for (; j < E; ++j) {
      const float q = rank_key(L[j]);
      r += (q > v || (q == v && j < e));
    }
    if (r < kCandCap) { sc.cand_e[r] = e; sc.cand_v[r] = v; }
  }
}

// End of the certain set from fully ranked candidates: the first rank
// j >= k-1 whose gap to rank j+1 exceeds thr; everything below it is
// certainly below.  Returns -1 when no such rank lies within kCandCap.
__device__ int certain_end_ranked(const WarpScratch& sc, int E, int k, float thr) {
  const int lane = threadIdx.x & 31;
  const int nc = E < kCandCap ? E : kCandCap;
  int j = lane;
  bool ok = j >= k - 1 && j + 1 < nc && sc.cand_v[j] - sc.cand_v[j + 1] > thr;
  const unsigned g0 = __ballot_sync(0xffffffffu, ok);
  j = lane + 32;
  ok = j >= k - 1 && j + 1 < nc && sc.cand_v[j] - sc.cand_v[j + 1] > thr;
  const unsigned g1 = __ballot_sync(0xffffffffu, ok);
  if (g0) return __ffs(g0) - 1;
  if (g1) return __ffs(g1) - 1 + 32;
  return E <= kCandCap ? E - 1 : -1;
}

// Sorted candidates for E <= 128, extracted in rank order until the certain
// set is closed.  Each lane keeps its (up to) four logits sorted in
// registers; a round is one warp arg-max over the lanes' current heads.
// Writes cand_e/cand_v[0..end+1] and returns end (or -1 for the fallback).
__device__ int extract_small(const float* L, int E, int k, float thr, WarpScratch& sc) {
  const int lane = threadIdx.x & 31;
  float v[4];
  int id[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = lane + 32 * i;
    id[i] = e < E ? e : INT_MAX;
    v[i] = e < E ? rank_key(L[e]) : -INFINITY;
  }
  // sort the four (v, id) pairs, best first (5-comparator network)
#define MOE_CSWAP(a, b)                                                        \
  if (better(v[b], id[b], v[a], id[a])) {                                      \
    const float tv = v[a]; v[a] = v[b]; v[b] = tv;                             \
    const int ti = id[a]; id[a] = id[b]; id[b] = ti;                           \
  }
  MOE_CSWAP(0, 1) MOE_CSWAP(2, 3) MOE_CSWAP(0, 2) MOE_CSWAP(1, 3) MOE_CSWAP(1, 2)
#undef MOE_CSWAP
  int head = 0;
  float prev = 0.f;
  for (int r = 0; r < kCandCap; ++r) {
    float bv = head == 0 ? v[0] : head == 1 ? v[1] : head == 2 ? v[2] : head == 3 ? v[3] : -INFINITY;
    int be = head == 0 ? id[0] : head == 1 ? id[1] : head == 2 ? id[2] : head == 3 ? id[3] : INT_MAX;
    const int mylane = lane;
    int bl = mylane;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      const int ol = __shfl_xor_sync(0xffffffffu, bl, o);
      if (better(ov, oe, bv, be)) { bv = ov; be = oe; bl = ol; }
    }
    if (lane == bl) ++head;
    if (lane == 0) { sc.cand_e[r] = be; sc.cand_v[r] = bv; }
    if (r >= k && prev - bv > thr) return r - 1;   // gap closes the certain set
    if (r + 1 == E) return r;                       // every expert extracted
    prev = bv;
  }
  return -1;
}

// Certified top-k of one token from its sorted candidates cand[0..end] (the
// certain set) -- or, when fallback is set, from fp64 logits of every expert.
// Whole warp.  Writes idx_out[0..k) and w_out[0..k).
__device__ void select_token(int E, int k, float delta, int end, const uint16_t* xrow,
                             const uint16_t* gate_w, const float* bias, int H, double* l64_row,
                             WarpScratch& sc, int32_t* idx_out, float* w_out, WsHeader* hdr) {
  const int lane = threadIdx.x & 31;
  const int per_lane = (E + 31) >> 5;
  const float thr = cert_threshold(delta);
  const bool fallback = end < 0;
  __syncwarp();

  if (!fallback) {
    // Ambiguous candidates: members of an adjacent pair closer than 2*delta.
    bool amb0 = false, amb1 = false;
    for (int r = 0; r < 2; ++r) {
      const int i = lane + 32 * r;
      bool a = false;
      if (i <= end) {
        if (i > 0 && !(sc.cand_v[i - 1] - sc.cand_v[i] > thr)) a = true;
        if (i < end && !(sc.cand_v[i] - sc.cand_v[i + 1] > thr)) a = true;
      }
      if (r == 0) amb0 = a; else amb1 = a;
    }
    const unsigned bal0 = __ballot_sync(0xffffffffu, amb0);
    const unsigned bal1 = __ballot_sync(0xffffffffu, amb1);
    if ((bal0 | bal1) == 0) {
      // the fp32 order is certain: ranks are the candidate positions
      if (lane < k) {
        idx_out[lane] = sc.cand_e[lane];
        sc.ex[lane] = expf(sc.cand_v[lane] - sc.cand_v[0]);
      }
      __syncwarp();
      if (lane == 0) {
        float sum = 0.0f;
        for (int s = 0; s < k; ++s) sum += sc.ex[s];
        for (int s = 0; s < k; ++s) w_out[s] = sc.ex[s] / sum;
      }
      __syncwarp();
      return;
    }
    if (lane == 0) atomicAdd(&hdr->router_flagged, 1);
    for (int r = 0; r < 2; ++r) {
      const int i = lane + 32 * r;
      if (i <= end) sc.key[i] = (double)sc.cand_v[i];
    }
    __syncwarp();
    for (int r = 0; r < 2; ++r) {
      unsigned bal = r == 0 ? bal0 : bal1;
      while (bal) {
        const int i = __ffs(bal) - 1 + 32 * r;
        bal &= bal - 1;
        const int e = sc.cand_e[i];
        double d = warp_dot_f64(xrow, gate_w + (size_t)e * H, H);
        if (bias) d += (double)bias[e];
        if (lane == 0) sc.key[i] = d;
      }
    }
    __syncwarp();
    // rank of each candidate by (key desc, index asc)
    int rank[2] = {INT_MAX, INT_MAX};
    for (int r = 0; r < 2; ++r) {
      const int i = lane + 32 * r;
      if (i <= end) {
        const double ki = sc.key[i];
        const int ei = sc.cand_e[i];
        int rk = 0;
        for (int j = 0; j <= end; ++j) {
          const double kj = sc.key[j];
          rk += (kj > ki || (kj == ki && sc.cand_e[j] < ei)) ? 1 : 0;
        }
        rank[r] = rk;
        if (rk < k) idx_out[rk] = ei;
        if (rk == 0) sc.kmax = ki;
      }
    }
    __syncwarp();
    const double kmax = sc.kmax;
    for (int r = 0; r < 2; ++r) {
      const int i = lane + 32 * r;
      if (rank[r] < k) sc.ex[rank[r]] = expf((float)(sc.key[i] - kmax));
    }
  } else {
    // Every expert in fp64 (needs >= 64 experts within rounding of each other).
    if (lane == 0) { atomicAdd(&hdr->router_flagged, 1); atomicAdd(&hdr->router_fallback, 1); }
    for (int e = 0; e < E; ++e) {
      double d = warp_dot_f64(xrow, gate_w + (size_t)e * H, H);
      if (bias) d += (double)bias[e];
      if (lane == 0) l64_row[e] = d;
    }
    __syncwarp();
    __threadfence_block();
    uint32_t taken = 0;
    double kmax = 0.0;
    for (int s = 0; s < k; ++s) {
      double bv = 0.0;
      int be = INT_MAX;
      for (int i = 0; i < per_lane; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u)) {
          const double v = l64_row[e];
          if (be == INT_MAX || v > bv || (v == bv && e < be)) { bv = v; be = e; }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const double ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (oe != INT_MAX && (be == INT_MAX || ov > bv || (ov == bv && oe < be))) { bv = ov; be = oe; }
      }
      if (be == INT_MAX) be = 0;  // unreachable for k <= E
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      if (s == 0) kmax = bv;
      if (lane == 0) { idx_out[s] = be; sc.ex[s] = expf((float)(bv - kmax)); }
    }
  }
  __syncwarp();
  if (lane == 0) {
    float sum = 0.0f;
    for (int s = 0; s < k; ++s) sum += sc.ex[s];
    for (int s = 0; s < k; ++s) w_out[s] = sc.ex[s] / sum;
  }
  __syncwarp();
}

// ------------------------------------------------------------ small batches
// Grid (T, ceil(E/16)), 16 warps, one (token, expert) logit per warp.  Lane l
// sums the products at h = 8l + 256j + (0..7) sequentially (H/32 terms), then
// a 5-level xor tree: at most H/32 + 4 roundings per product.  The last CTA to
// finish a token (integer counter, no waiting) selects that token's top-k.
// With kGroup, the CTA that selects the batch's last token then groups all
// routed slots (grouping.cuh) in the same launch.
constexpr int kSmallWarps = 16;

template <bool kGroup>
__global__ void __launch_bounds__(kSmallWarps * 32) router_small_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ gw, const float* __restrict__ bias,
    int T, int H, int E, int k, int gamma_terms, float* __restrict__ logits,
    float* __restrict__ wnorm, double* __restrict__ l64, int* __restrict__ cnt,
    int32_t* __restrict__ idx, float* __restrict__ w, void* ws, GroupOut go) {
  extern __shared__ int gsmem[];   // grouping scratch (kGroup only)
  __shared__ WarpScratch scr;
  __shared__ __align__(16) float sl[1024];
  __shared__ int s_last, s_group;
  __shared__ int sw[grouping::kWarps];
  pdl_wait();
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.y * kSmallWarps + warp;
  const uint16_t* xr = x + (size_t)t * H;
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  if (e < E) {
    float acc = 0.f, sq = 0.f;
    const uint16_t* wr = gw + (size_t)e * H;
#pragma unroll 8
    for (int h = lane * 8; h < H; h += 256) {
      const uint4 xv = *reinterpret_cast<const uint4*>(xr + h);
      const uint4 wv = *reinterpret_cast<const uint4*>(wr + h);
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
      const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc = fmaf(bf16lo(xw[i]), bf16lo(ww[i]), acc);
        acc = fmaf(bf16hi(xw[i]), bf16hi(ww[i]), acc);
        sq = fmaf(bf16lo(ww[i]), bf16lo(ww[i]), sq);
        sq = fmaf(bf16hi(ww[i]), bf16hi(ww[i]), sq);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      acc += __shfl_xor_sync(0xffffffffu, acc, o);
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
    }
    if (lane == 0) {
      logits[(size_t)t * E + e] = bias ? acc + bias[e] : acc;
      wnorm[e] = sqrtf(sq);   // same value from every token's CTA
      __threadfence();        // the writer publishes before the CTA signals
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&cnt[t], 1) == (int)gridDim.y - 1;
  __syncthreads();
  if (!s_last) return;
  // last CTA of token t (reads other CTAs' results through L2, ld.cg):
  // logits to shared memory, certified selection
  for (int ee = threadIdx.x; ee < E; ee += blockDim.x) sl[ee] = __ldcg(&logits[(size_t)t * E + ee]);
  __syncthreads();
  if (E > 128) {   // many experts: every thread of the CTA helps rank them
    rank_candidates(sl, E, scr, threadIdx.x, blockDim.x);
    __syncthreads();
  }
  if (warp == 0) {
    // ||x_t||, max ||w_e||, max |logit| for the error bound
    float sqx = 0.f;
    for (int h = lane * 8; h < H; h += 256) {
      const uint4 xv = *reinterpret_cast<const uint4*>(xr + h);
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sqx = fmaf(bf16lo(xw[i]), bf16lo(xw[i]), sqx);
        sqx = fmaf(bf16hi(xw[i]), bf16hi(xw[i]), sqx);
      }
    }
    float wmax = 0.f, lmax = 0.f;
    for (int ee = lane; ee < E; ee += 32) {
      wmax = fmaxf(wmax, __ldcg(&wnorm[ee]));
      lmax = fmaxf(lmax, fabsf(sl[ee]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sqx += __shfl_xor_sync(0xffffffffu, sqx, o);
      wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
      lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
    }
    const float delta = gamma_bound(gamma_terms) * sqrtf(sqx) * wmax * (1.0f + 0x1p-10f) +
                        0x1p-22f * lmax + (float)H * 0x1p-149f;
    const float thr = cert_threshold(delta);
    const int end = E <= 128 ? extract_small(sl, E, k, thr, scr) : certain_end_ranked(scr, E, k, thr);
    select_token(E, k, delta, end, xr, gw, bias, H, l64 + (size_t)t * E, scr, idx + (size_t)t * k,
                 w + (size_t)t * k, hdr);
  }
  if constexpr (kGroup) {
    if (warp == 0) __threadfence();   // the selecting warp wrote idx / w
    __syncthreads();
    if (threadIdx.x == 0) s_group = atomicAdd(&hdr->tokens_done, 1) == T - 1;
    __syncthreads();
    if (!s_group) return;
    grouping::group_single_block(idx, T * k, E, go.large_threshold, go.tile_rows, go.counts,
                                 go.offsets, go.perm, go.inv_perm, go.active, go.tiles, ws, gsmem,
                                 sw, go.zero, go.nzero);
  }
}

// ------------------------------------------------------------ large batches
// Logits: one CTA = 32 tokens x all E (<= 128) experts, 128 threads; thread
// (ty, tx) owns tokens 4ty..4ty+3 and experts 4tx..4tx+3, 64+4tx..64+4tx+3.  K runs in chunks of
// 64: a chunk's 64 products are summed sequentially from zero (63 roundings)
// and the chunk sum is added to the running total (H/64 additions): at most
// 64 + H/64 roundings per product.  Selection then runs one warp per token.
constexpr int kTileT = 32, kTileE = 128, kTileK = 64;

__global__ void __launch_bounds__(128) router_tile_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ gw, const float* __restrict__ bias,
    int T, int H, int E, float* __restrict__ logits, float* __restrict__ xnorm) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* xs = reinterpret_cast<float*>(smem_raw);           // [2][kTileK][kTileT]
  float* wsm = xs + 2 * kTileK * kTileT;                    // [2][kTileK][kTileE]
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int t0 = blockIdx.x * kTileT;
  const int warp = tid >> 5, lane = tid & 31;

  // ||x_t|| for the tile's tokens: warp-level sums (H/32 + 4 roundings).
  for (int i = 0; i < kTileT / 4; ++i) {
    const int t = t0 + warp * (kTileT / 4) + i;
    float sq = 0.f;
    if (t < T) {
      for (int h = lane * 8; h < H; h += 256) {
        const uint4 v = *reinterpret_cast<const uint4*>(x + (size_t)t * H + h);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          sq = fmaf(bf16lo(u[q]), bf16lo(u[q]), sq);
          sq = fmaf(bf16hi(u[q]), bf16hi(u[q]), sq);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if (lane == 0 && t < T) xnorm[t] = sqrtf(sq);
  }

  // Global -> register staging of one K chunk: x tile 32x64 (2 uint4 per
  // thread), w tile 128x64 (8 uint4 per thread), transposed into [k][row].
  uint4 rx[2], rw[8];
  auto load_chunk = [&](int kc) {
    const int k0 = kc * kTileK;
    // vector v covers row v % rows, columns 8*(v / rows) .. +7, so that the
    // 32 lanes of a warp hold 32 consecutive rows of one column group and the
    // transposed shared-memory stores below hit 32 distinct banks
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int v = tid + 128 * i;          // 256 vectors
      const int row = v % kTileT, col = (v / kTileT) * 8;
      const int t = t0 + row;
      rx[i] = (t < T) ? *reinterpret_cast<const uint4*>(x + (size_t)t * H + k0 + col)
                      : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int v = tid + 128 * i;          // 1024 vectors
      const int row = v % kTileE, col = (v / kTileE) * 8;
      rw[i] = (row < E) ? *reinterpret_cast<const uint4*>(gw + (size_t)row * H + k0 + col)
                        : make_uint4(0, 0, 0, 0);
    }
  };
  auto store_chunk = [&](int buf) {
    float* xb = xs + buf * kTileK * kTileT;
    float* wb = wsm + buf * kTileK * kTileE;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int v = tid + 128 * i;
      const int row = v % kTileT, col = (v / kTileT) * 8;
      const uint32_t u[4] = {rx[i].x, rx[i].y, rx[i].z, rx[i].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        xb[(col + 2 * q) * kTileT + row] = bf16lo(u[q]);
        xb[(col + 2 * q + 1) * kTileT + row] = bf16hi(u[q]);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int v = tid + 128 * i;
      const int row = v % kTileE, col = (v / kTileE) * 8;
      const uint32_t u[4] = {rw[i].x, rw[i].y, rw[i].z, rw[i].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        wb[(col + 2 * q) * kTileE + row] = bf16lo(u[q]);
        wb[(col + 2 * q + 1) * kTileE + row] = bf16hi(u[q]);
      }
    }
  };

  float tot[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) tot[i][j] = 0.f;

  const int nchunks = H / kTileK;
  load_chunk(0);
  store_chunk(0);
  __syncthreads();
  for (int kc = 0; kc < nchunks; ++kc) {
    const int buf = kc & 1;
    if (kc + 1 < nchunks) load_chunk(kc + 1);
    const float* xb = xs + buf * kTileK * kTileT + ty * 4;
    // thread tx owns experts 4tx..4tx+3 and 64+4tx..64+4tx+3: a quarter-warp
    // then reads 128 contiguous bytes per vector load (no bank conflicts)
    const float* wb = wsm + buf * kTileK * kTileE + tx * 4;
    float part[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) part[i][j] = 0.f;
#pragma unroll 8
    for (int kk = 0; kk < kTileK; ++kk) {
      const float4 xa = *reinterpret_cast<const float4*>(xb + kk * kTileT);
      const float4 wa = *reinterpret_cast<const float4*>(wb + kk * kTileE);
      const float4 wb4 = *reinterpret_cast<const float4*>(wb + kk * kTileE + 64);
      const float xv[4] = {xa.x, xa.y, xa.z, xa.w};
      const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb4.x, wb4.y, wb4.z, wb4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) part[i][j] = fmaf(xv[i], wv[j], part[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) tot[i][j] += part[i][j];
    if (kc + 1 < nchunks) store_chunk(buf ^ 1);
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = (j < 4 ? 0 : 64) + tx * 4 + (j & 3);
      if (e < E) logits[(size_t)t * E + e] = bias ? tot[i][j] + bias[e] : tot[i][j];
    }
  }
}

// Selection for the tiled path: one warp per token.
__global__ void __launch_bounds__(256) router_select_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ gw, const float* __restrict__ bias,
    int T, int H, int E, int k, int gamma_terms, const float* __restrict__ logits,
    const float* __restrict__ xnorm, const float* __restrict__ wnorm, double* __restrict__ l64,
    int32_t* __restrict__ idx, float* __restrict__ w, void* ws) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WarpScratch* scr = reinterpret_cast<WarpScratch*>(smem_raw);
  float* sl = reinterpret_cast<float*>(smem_raw + sizeof(WarpScratch) * 8) + (size_t)warp * E;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  float wmax = 0.f, lmax = 0.f;
  for (int e = lane; e < E; e += 32) {
    const float v = logits[(size_t)t * E + e];
    sl[e] = v;
    wmax = fmaxf(wmax, wnorm[e]);
    lmax = fmaxf(lmax, fabsf(v));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
    lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
  }
  __syncwarp();
  const float delta = gamma_bound(gamma_terms) * xnorm[t] * wmax * (1.0f + 0x1p-10f) +
                      0x1p-22f * lmax + (float)H * 0x1p-149f;
  const int end = extract_small(sl, E, k, cert_threshold(delta), scr[warp]);   // E <= 128 here
  select_token(E, k, delta, end, x + (size_t)t * H, gw, bias, H, l64 + (size_t)t * E, scr[warp],
               idx + (size_t)t * k, w + (size_t)t * k, reinterpret_cast<WsHeader*>(ws));
}

// ||w_e|| for every expert, one warp per expert.
__global__ void __launch_bounds__(256) wnorm_kernel(const uint16_t* __restrict__ gw, int H, int E,
                                                    float* __restrict__ wnorm) {
  const int e = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (e >= E) return;
  float sq = 0.f;
  for (int h = lane * 8; h < H; h += 256) {
    const uint4 v = *reinterpret_cast<const uint4*>(gw + (size_t)e * H + h);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      sq = fmaf(bf16lo(u[q]), bf16lo(u[q]), sq);
      sq = fmaf(bf16hi(u[q]), bf16hi(u[q]), sq);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  if (lane == 0) wnorm[e] = sqrtf(sq);
}

}  // namespace

bool route_can_group(int T, int E, int k) { return !(T >= 2048 && E <= 128) && T * k <= 8 * kPermBlock; }

cudaError_t launch_route(const uint16_t* x, const uint16_t* gate_w, const float* bias, int T, int H,
                         int E, int k, int32_t* idx, float* w, void* ws, const WsLayout& L,
                         cudaStream_t stream, int* launches, const GroupOut* group) {
  float* wnorm = ws_ptr<float>(ws, L.wnorm);
  double* l64 = ws_ptr<double>(ws, L.logits64);
  const bool tiled = T >= 2048 && E <= kTileE;
  if (launches) *launches += tiled ? 3 : 1;
  if (tiled) {
    float* logits = ws_ptr<float>(ws, L.logits);
    float* xnorm = ws_ptr<float>(ws, L.xnorm);
    wnorm_kernel<<<(E + 7) / 8, 256, 0, stream>>>(gate_w, H, E, wnorm);
    const size_t smem = sizeof(float) * 2 * kTileK * (kTileT + kTileE);
    cudaError_t err = cudaFuncSetAttribute(router_tile_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    router_tile_kernel<<<(T + kTileT - 1) / kTileT, 128, smem, stream>>>(x, gate_w, bias, T, H, E,
                                                                         logits, xnorm);
    const size_t smem2 = sizeof(WarpScratch) * 8 + sizeof(float) * 8 * E;
    err = cudaFuncSetAttribute(router_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem2);
    if (err != cudaSuccess) return err;
    const int gterms = kTileK + H / kTileK + 1;
    router_select_kernel<<<(T + 7) / 8, 256, smem2, stream>>>(x, gate_w, bias, T, H, E, k, gterms,
                                                              logits, xnorm, wnorm, l64, idx, w, ws);
    return cudaGetLastError();
  }
  float* logits = ws_ptr<float>(ws, L.logits);
  int* cnt = ws_ptr<int>(ws, L.cnt);
  dim3 g1(T, (E + kSmallWarps - 1) / kSmallWarps);
  const int gterms = H / 32 + 5;
  if (group) {
    const size_t smem = sizeof(int) * grouping::single_block_smem_ints(E);
    cudaError_t err = cudaFuncSetAttribute(router_small_kernel<true>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    router_small_kernel<true><<<g1, kSmallWarps * 32, smem, stream>>>(
        x, gate_w, bias, T, H, E, k, gterms, logits, wnorm, l64, cnt, idx, w, ws, *group);
  } else {
    router_small_kernel<false><<<g1, kSmallWarps * 32, 0, stream>>>(
        x, gate_w, bias, T, H, E, k, gterms, logits, wnorm, l64, cnt, idx, w, ws, GroupOut{});
  }
  return cudaGetLastError();
}

}  // namespace moe
