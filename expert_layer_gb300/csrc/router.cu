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

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kCandCap = 64;  // candidates a warp can hold while certifying

// gamma_n as fp32, evaluated on the host (fp64 division is slow on the device)
// and passed to the kernels.
inline float gamma_bound(int n) {
  const double u = 5.9604644775390625e-08;  // 2^-24
  return (float)(n * u / (1.0 - n * u));
}

// Exact sum of bf16 x bf16 products over columns [h0, h1) (h0 % 256 == 0,
// h1 % 8 == 0) for one warp, returned as an integer part acc * 2^-48 plus an
// fp64 part r; every lane returns the same pair (xor butterflies).  A bf16 x bf16 product has at most 16
// significant bits, so its fp32 value is exact unless it under- or overflows
// fp32.  Exact products of magnitude 2^-33 .. < 1 are added as integers in a
// 64-bit fixed-point accumulator with its unit in the last place at 2^-48
// (16 significant bits shifted by exponent - 94, at most 32; a sum of up to
// 2^15 terms below 2^48 each stays below 2^63, so a warp takes at most 32768
// columns this way): those sums are exact.  A batch of 8 elements in which any
// lane meets a product outside that range (or an inexact fp32 product) is
// added in fp64 instead, for the whole warp; when no batch went that way r is
// 0 and its reduction is skipped.  The integer work runs on the full-rate
// integer pipes; GB300's fp64 pipe is slow.
__device__ __forceinline__ long long fixed_of_product(uint32_t u) {
  const int e = (int)((u >> 23) & 0xffu);
  if (e == 0) return 0;   // exact zero (an underflow was sent the fp64 way)
  const long long m16 = (long long)(((u & 0x7fffffu) | 0x800000u) >> 8);   // 16 significant bits
  const long long q = m16 << (e - 94);
  return (u & 0x80000000u) ? -q : q;
}

struct DotPart {
  long long acc;   // exact, in units of 2^-48
  double r;
};

__device__ DotPart warp_dot_f64(const uint16_t* __restrict__ a, const uint16_t* __restrict__ b,
                                int h0, int h1) {
  const int lane = threadIdx.x & 31;
  double s[4] = {0.0, 0.0, 0.0, 0.0};
  long long acc = 0;
  bool used64 = false;                      // warp-uniform
  const bool fixed_ok = h1 - h0 <= 32768;   // the accumulator's headroom
  constexpr int kB = 4;   // iterations whose loads are issued together
  for (int hb = h0; hb < h1; hb += 256 * kB) {
   uint4 va4[kB], vb4[kB];
#pragma unroll
   for (int it = 0; it < kB; ++it) {
     const int h = hb + lane * 8 + 256 * it;
     va4[it] = h < h1 ? *reinterpret_cast<const uint4*>(a + h) : make_uint4(0, 0, 0, 0);
     vb4[it] = h < h1 ? *reinterpret_cast<const uint4*>(b + h) : make_uint4(0, 0, 0, 0);
   }
#pragma unroll 1
   for (int it = 0; it < kB; ++it) {
    if (hb + 256 * it >= h1) break;   // whole warp: past the range
    const uint4 va = va4[it], vb = vb4[it];
    const uint32_t wa[4] = {va.x, va.y, va.z, va.w};
    const uint32_t wb[4] = {vb.x, vb.y, vb.z, vb.w};
    uint32_t pu[8];
    bool outside = false;
    // rolled loops throughout: this code runs rarely, from a cold
    // instruction cache, and its fetch time exceeded its execution time
    // (a traced copy: 9-12 us per dot unrolled, 6-7 us rolled)
#pragma unroll 1
    for (int i = 0; i < 4; ++i) {
#pragma unroll 1
      for (int j = 0; j < 2; ++j) {
        const float fa = j ? bf16hi(wa[i]) : bf16lo(wa[i]);
        const float fb = j ? bf16hi(wb[i]) : bf16lo(wb[i]);
        const uint32_t u = __float_as_uint(__fmul_rn(fa, fb));
        const uint32_t e = (u >> 23) & 0xffu;
        // inexact fp32 product (overflow, inf / nan, or underflow of two
        // nonzero factors), or an exact one outside the fixed-point range
        outside |= e == 0xffu || (e == 0 && fa != 0.0f && fb != 0.0f) || (e != 0 && (e < 94u || e > 126u));
        pu[2 * i + j] = u;
      }
    }
    if (__any_sync(0xffffffffu, outside || !fixed_ok)) {
      used64 = true;
#pragma unroll 1
      for (int i = 0; i < 4; ++i) {
        s[i] = fma((double)bf16lo(wa[i]), (double)bf16lo(wb[i]), s[i]);
        s[i] = fma((double)bf16hi(wa[i]), (double)bf16hi(wb[i]), s[i]);
      }
    } else {
#pragma unroll 1
      for (int i = 0; i < 8; ++i) acc += fixed_of_product(pu[i]);
    }
   }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  double r = 0.0;
  if (used64) {
    r = (s[0] + s[1]) + (s[2] + s[3]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  }
  return {acc, r};
}

struct WarpScratch {
  int cand_e[kCandCap];
  float cand_v[kCandCap];
  double key[kCandCap];
  float ex[32];
  double kmax;
  int dpos[kCandCap];   // candidate positions that need an fp64 logit
  int nd;               // fp64 logits this token needs (0: selection done)
  int end;              // last rank of the certain set, -1: every expert in fp64
};

// Two logits whose fp32 values differ by more than this are ordered like the
// exact logits (each is within delta of its exact value).
__device__ __forceinline__ float cert_threshold(float delta) { return 2.0f * delta * 1.001f; }

// Sort key of a logit: NaN ranks below every number.
__device__ __forceinline__ float rank_key(float v) { return v != v ? -INFINITY : v; }

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

// Order-preserving map of a non-NaN float to uint32 (-0 and +0 both map to
// the key of +0, as they compare equal) and its inverse.
__device__ __forceinline__ uint32_t order_bits(float v) {
  const uint32_t u = v == 0.0f ? 0u : __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float order_value(uint32_t m) {
  return __uint_as_float((m & 0x80000000u) ? (m & 0x7fffffffu) : ~m);
}

// Sorted candidates for E <= 128, extracted in rank order until the certain
// set is closed.  Lane l holds the logits of experts l + 32i (i < 4) in v[]
// (any value for e >= E).  Each lane keeps its four keys sorted in
// registers; a round is a warp max-reduction over the lanes' current heads
// followed by a min-reduction over the expert ids that reach that maximum.
// Writes cand_e/cand_v[0..end+1] and returns end (or -1 for the fallback).
__device__ int extract_regs(const float (&v)[4], int E, int k, float thr, WarpScratch& sc) {
  const int lane = threadIdx.x & 31;
  uint32_t key[4];
  uint32_t id[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = lane + 32 * i;
    id[i] = e < E ? (uint32_t)e : 0xffffffffu;
    key[i] = e < E ? order_bits(rank_key(v[i])) : 0u;   // 0 ranks below -inf
  }
  // sort the four (key, id) pairs, best first (5-comparator network)
#define MOE_CSWAP(a, b)                                                              \
  if (key[b] > key[a] || (key[b] == key[a] && id[b] < id[a])) {                      \
    const uint32_t tk = key[a]; key[a] = key[b]; key[b] = tk;                        \
    const uint32_t ti = id[a]; id[a] = id[b]; id[b] = ti;                            \
  }
  MOE_CSWAP(0, 1) MOE_CSWAP(2, 3) MOE_CSWAP(0, 2) MOE_CSWAP(1, 3) MOE_CSWAP(1, 2)
#undef MOE_CSWAP
  int head = 0;
  float prev = 0.f;
  for (int r = 0; r < kCandCap; ++r) {
    const uint32_t hk = head == 0 ? key[0] : head == 1 ? key[1] : head == 2 ? key[2] : head == 3 ? key[3] : 0u;
    const uint32_t hid = head == 0 ? id[0] : head == 1 ? id[1] : head == 2 ? id[2] : head == 3 ? id[3] : 0xffffffffu;
    const uint32_t m = __reduce_max_sync(0xffffffffu, hk);
    const uint32_t be = __reduce_min_sync(0xffffffffu, hk == m ? hid : 0xffffffffu);
    if (hk == m && hid == be) ++head;
    const float bv = order_value(m);
    if (lane == 0) { sc.cand_e[r] = (int)be; sc.cand_v[r] = bv; }
    if (r >= k && prev - bv > thr) return r - 1;   // gap closes the certain set
    if (r + 1 == E) return r;                       // every expert extracted
    prev = bv;
  }
  return -1;
}

// extract_regs over logits held in shared memory.
__device__ int extract_small(const float* L, int E, int k, float thr, WarpScratch& sc) {
  const int lane = threadIdx.x & 31;
  float v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? L[e] : 0.0f;
  }
  return extract_regs(v, E, k, thr, sc);
}

// Selection of one token from its sorted candidates cand[0..end] (the
// certain set), in three phases so that the rare fp64 work can be shared by
// every warp of the CTA:
//   select_begin  (one warp per token) certain order -> writes the top-k and
//                 the weights and sets nd = 0; else lists in dpos[0..nd) the
//                 candidates that sit within rounding of a neighbour (or, when
//                 end < 0, asks for all E experts) and sets nd
//   select_dots   (all warps of the CTA) the listed fp64 logits
//   select_end    (one warp per token with nd > 0) ranks by the fp64 keys
// Weights: softmax over all E renormalised over the k selected, i.e.
// exp(l_s - l_max) over the selected set divided by its sum.

// Renormalised weights from the unnormalised ones in lanes < k (fixed xor-tree
// sum, the same on every lane).
__device__ __forceinline__ void write_weights(float ex, int k, float* w_out) {
  const int lane = threadIdx.x & 31;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) w_out[lane] = ex / sum;
}

__device__ void select_begin(int E, int k, float delta, int end, WarpScratch& sc, int32_t* idx_out,
                             float* w_out, WsHeader* hdr) {
  const int lane = threadIdx.x & 31;
  const float thr = cert_threshold(delta);
  __syncwarp();
  if (end < 0) {
    // every expert in fp64 (needs >= 64 experts within rounding of each other)
    if (lane == 0) {
      atomicAdd(&hdr->router_flagged, 1);
      atomicAdd(&hdr->router_fallback, 1);
      sc.nd = E;
      sc.end = -1;
    }
    __syncwarp();
    return;
  }
  // ambiguous candidates: members of an adjacent pair closer than 2*delta
  bool amb[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int i = lane + 32 * r;
    bool a = false;
    if (i <= end) {
      if (i > 0 && !(sc.cand_v[i - 1] - sc.cand_v[i] > thr)) a = true;
      if (i < end && !(sc.cand_v[i] - sc.cand_v[i + 1] > thr)) a = true;
    }
    amb[r] = a;
  }
  const unsigned bal0 = __ballot_sync(0xffffffffu, amb[0]);
  const unsigned bal1 = __ballot_sync(0xffffffffu, amb[1]);
  if ((bal0 | bal1) == 0) {
    // the fp32 order is certain: ranks are the candidate positions
    float ex = 0.f;
    if (lane < k) {
      idx_out[lane] = sc.cand_e[lane];
      ex = expf(sc.cand_v[lane] - sc.cand_v[0]);
    }
    write_weights(ex, k, w_out);
    if (lane == 0) sc.nd = 0;
    __syncwarp();
    return;
  }
  if (lane == 0) atomicAdd(&hdr->router_flagged, 1);
  const unsigned lt = (1u << lane) - 1u;
  const int n0 = __popc(bal0);
  if (amb[0]) sc.dpos[__popc(bal0 & lt)] = lane;
  if (amb[1]) sc.dpos[n0 + __popc(bal1 & lt)] = lane + 32;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int i = lane + 32 * r;
    if (i <= end) sc.key[i] = (double)sc.cand_v[i];
  }
  if (lane == 0) {
    sc.nd = n0 + __popc(bal1);
    sc.end = end;
  }
  __syncwarp();
}

// The fp64 logits listed by select_begin for the tokens t0 .. t0+nt-1
// (scratch scr[0..nt)), shared by all warps of the block.  Each dot is split
// into kDotParts slices of its 256-column blocks, one warp per slice (a slice
// of up to 1024 columns is one batch of loads per lane, so a round costs one
// memory latency).  The slices' integer parts are added exactly (H <= 32768)
// and rounded to fp64 once; their fp64 parts follow in slice order.  s_part
// holds one DotPart per warp.  Called by every thread of the block.
constexpr int kDotParts = 2;

__device__ void dot_target(const WarpScratch* scr, int j, int& tt, int& r, int& e) {
  tt = 0;
  r = j;
  while (r >= scr[tt].nd) { r -= scr[tt].nd; ++tt; }
  e = scr[tt].end < 0 ? r : scr[tt].cand_e[scr[tt].dpos[r]];
}

__device__ void select_dots(WarpScratch* scr, int nt, int t0, const uint16_t* x,
                            const uint16_t* gate_w, const float* bias, int H, int E, double* l64,
                            DotPart* s_part) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int per = nw / kDotParts;   // dots per round
  const int nb = (H + 255) / 256;
  int total = 0;
  for (int tt = 0; tt < nt; ++tt) total += scr[tt].nd;
  for (int base = 0; base < total; base += per) {   // uniform trip count
    const int j = base + warp / kDotParts, q = warp % kDotParts;
    DotPart d = {0, 0.0};
    if (j < total) {
      int tt, r, e;
      dot_target(scr, j, tt, r, e);
      const int h0 = 256 * (q * nb / kDotParts), h1 = min(H, 256 * ((q + 1) * nb / kDotParts));
      d = warp_dot_f64(x + (size_t)(t0 + tt) * H, gate_w + (size_t)e * H, h0, h1);
    }
    if (lane == 0) s_part[warp] = d;
    __syncthreads();
    if (lane == 0 && warp < per && base + warp < total) {
      int tt, r, e;
      dot_target(scr, base + warp, tt, r, e);
      const DotPart* p = s_part + kDotParts * warp;
      double v = 0.0;
      if (H <= 32768) {   // fewer than 2^15 terms below 2^48 each: no overflow
        long long a = 0;
#pragma unroll
        for (int i = 0; i < kDotParts; ++i) a += p[i].acc;
        v = (double)a * 0x1p-48;   // exact scaling by a power of two
      } else {
#pragma unroll
        for (int i = 0; i < kDotParts; ++i) v += (double)p[i].acc * 0x1p-48;
      }
#pragma unroll
      for (int i = 0; i < kDotParts; ++i) v += p[i].r;
      if (bias) v += (double)bias[e];
      WarpScratch& sc = scr[tt];
      if (sc.end < 0) l64[(size_t)(t0 + tt) * E + e] = v;
      else sc.key[sc.dpos[r]] = v;
    }
    __syncthreads();
  }
}

__device__ void select_end(int E, int k, WarpScratch& sc, const double* l64_row, int32_t* idx_out,
                           float* w_out) {
  const int lane = threadIdx.x & 31;
  const int end = sc.end;
  if (end >= 0) {
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
    const int per_lane = (E + 31) >> 5;
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
  write_weights(lane < k ? sc.ex[lane] : 0.f, k, w_out);
  __syncwarp();
}

// ------------------------------------------------------------ small batches
// Grid (ceil(T / kTT), ceil(E / (16 kEPW))), 16 warps: warp w of CTA (c, y)
// computes the logits of kEPW experts (16y + w for kTT = 1; 32y + 2w, +1 for
// chunks of 4 or 8 tokens) for the kTT tokens of chunk c, holding its gate
// rows in registers.  Lane l sums the products at h = 8l + 256j + (0..7)
// in kChains sequential chains (vector j goes to chain j mod kChains: 8
// chains for one-token chunks, 2 for four-token chunks, 1 for eight, as the
// registers allow), adds the chains pairwise, then a 5-level xor tree: at
// most min(H/32, 64 ceil(H/2048) / kChains) + log2(kChains) + 5 roundings
// per product (16 at H = 2048 for one-token chunks, against 69 in one chain).  With kTT = 1 the warp reads the token row from
// global memory; larger chunks first stage the chunk's token rows (2048
// columns at a time) in shared memory, so each warp's token loads are
// shared-memory reads.  Warps w < #tokens of the y = 0 CTAs also write
// ||x_t||.  The last CTA to finish a chunk (integer counter, no waiting)
// orders each token's experts: one warp per token extracting in rank order
// (chunks of 4 or 8 tokens, E <= 128), or all threads ranking every
// (token, expert) by counting; then one warp per token selects.  With
// kGroup, each selecting CTA then gives every routed slot of its chunk its
// rank within its expert's group (an atomic per-expert counter, arrival
// order); the expert kernel builds the grouping from those ranks (no
// grouping pass and no hand-off between them).
constexpr int kSmallWarps = 16;
constexpr int kXCols = 2048;   // token-row columns staged per block

template <int kTT>
struct SmallCfg {
  static constexpr int kEPW = kTT >= 4 ? 2 : 1;            // experts per warp
  // independent accumulation chains per (expert, token) in a lane: chain
  // v % kChains takes the products of 16-byte vector v (fewer roundings per
  // product, so a tighter certified bound and fewer exact re-rankings)
  static constexpr int kChains = kTT == 1 ? 8 : kTT == 4 ? 2 : 1;
  static constexpr int kExperts = kSmallWarps * kEPW;     // experts per CTA
  static constexpr bool kStaged = kTT >= 4;                // token rows in shared memory
};

// Shared memory of the small router: for the selecting CTA, the chunk's
// sort keys [tt][E], logits [tt][E], ||w_e|| [E] and ||x_t|| [tt]; then
// (staged chunks) the token rows [tt][kXCols] bf16.
__host__ __device__ inline size_t router_small_select_bytes(int E, int tt) {
  return sizeof(uint64_t) * (size_t)tt * E + sizeof(float) * ((size_t)(tt + 1) * E + tt);
}
__host__ __device__ inline size_t router_small_smem(int E, int tt) {
  const size_t sel = (router_small_select_bytes(E, tt) + 15) & ~size_t(15);
  return tt >= 4 ? sel + sizeof(uint16_t) * (size_t)tt * kXCols : sel;
}

// Release-acquire integer add at GPU scope: the caller's earlier writes (and
// those its CTA made before a barrier) are visible to whoever observes the
// add, and the caller sees every write released to the counter before it.
__device__ __forceinline__ int atomic_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// c + a.lo * b.lo, then + a.hi * b.hi: two fp32 fmas whose factors are the
// bf16 halves of a and b (each product exact, one rounding per fma).
__device__ __forceinline__ float fma_bf16x2(uint32_t a, uint32_t b, float c) {
  asm("{\n .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
      " fma.rn.f32.bf16 %0, al, bl, %0;\n fma.rn.f32.bf16 %0, ah, bh, %0;\n}"
      : "+f"(c)
      : "r"(a), "r"(b));
  return c;
}

// Token rows t0 .. t0+kTT-1, columns [hb, hb + kXCols), into xs (zero past the
// chunk's tokens or past H).  All loads are issued before the stores.
template <int kTT>
__device__ __forceinline__ void stage_tokens(const uint16_t* __restrict__ x, int t0, int nt, int H,
                                             int hb, uint16_t* xs, uint16_t* __restrict__ x16, int* status) {
  constexpr int kRowVecs = kXCols / 8;
  constexpr int kPer = kTT * kRowVecs / (kSmallWarps * 32);
  static_assert(kTT * kRowVecs % (kSmallWarps * 32) == 0, "whole vectors per thread");
  uint4 v[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int q = threadIdx.x + i * kSmallWarps * 32;
    const int tt = q / kRowVecs, h = hb + (q % kRowVecs) * 8;
    v[i] = (tt < nt && h < H) ? *reinterpret_cast<const uint4*>(x + (size_t)(t0 + tt) * H + h)
                              : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) reinterpret_cast<uint4*>(xs)[threadIdx.x + i * kSmallWarps * 32] = v[i];
  if (x16) {   // the f16 copy of the token rows (decoded-weight expert kernels)
    bool bad = false;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int q = threadIdx.x + i * kSmallWarps * 32;
      const int tt = q / kRowVecs, h = hb + (q % kRowVecs) * 8;
      if (tt < nt && h < H)
        *reinterpret_cast<uint4*>(x16 + (size_t)(t0 + tt) * H + h) = bf16x8_to_f16x8(v[i], bad);
    }
    if (bad) atomicOr(status, kStatusRange);
  }
}

template <int kTT, bool kGroup>
__global__ void __launch_bounds__(kSmallWarps * 32) router_small_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ gw, const float* __restrict__ bias,
    int T, int H, int E, int k, float gamma, float* __restrict__ logits,
    float* __restrict__ wnorm, float* __restrict__ xnorm, double* __restrict__ l64,
    int* __restrict__ cnt, int32_t* __restrict__ idx, float* __restrict__ w, void* ws, GroupOut go,
    uint16_t* __restrict__ x16) {
  using Cfg = SmallCfg<kTT>;
  constexpr int kEPW = Cfg::kEPW;
  extern __shared__ __align__(16) int dsm[];
  __shared__ WarpScratch scr[kTT];
  __shared__ DotPart s_part[kSmallWarps];
  __shared__ int s_last;
  pdl_wait();      // the workspace counters are cleared
  pdl_trigger();   // the expert kernel may become resident; it waits for this grid
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x;
  const int t0 = chunk * kTT;
  const int nt = min(kTT, T - t0);
  const int e0 = blockIdx.y * Cfg::kExperts + warp * kEPW;
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  uint16_t* xs = reinterpret_cast<uint16_t*>(
      reinterpret_cast<unsigned char*>(dsm) +
      ((router_small_select_bytes(E, kTT) + 15) & ~size_t(15)));
  const bool xn_warp = blockIdx.y == 0 && warp < nt;   // this warp writes ||x_{t0+warp}||
  constexpr int NC = Cfg::kChains;
  float acc[kEPW][kTT][NC], sq[kEPW], sqx = 0.f;
#pragma unroll
  for (int ep = 0; ep < kEPW; ++ep) {
    sq[ep] = 0.f;
#pragma unroll
    for (int tt = 0; tt < kTT; ++tt)
#pragma unroll
      for (int c = 0; c < NC; ++c) acc[ep][tt][c] = 0.f;
  }
  for (int hb = 0; hb < H; hb += 2048) {
    uint4 wv[kEPW][8];
#pragma unroll
    for (int ep = 0; ep < kEPW; ++ep)
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const int h = hb + lane * 8 + 256 * v;
        wv[ep][v] = (e0 + ep < E && h < H) ? ldg_nc_v4(gw + (size_t)(e0 + ep) * H + h)
                                           : make_uint4(0, 0, 0, 0);
      }
    if constexpr (Cfg::kStaged) {
      if (hb > 0) __syncthreads();   // every warp is done with the previous block
      // the y = 0 CTAs also write the chunk's f16 token rows (when asked)
      stage_tokens<kTT>(x, t0, nt, H, hb, xs, blockIdx.y == 0 ? x16 : nullptr, &hdr->status);
      __syncthreads();
    }
#pragma unroll
    for (int ep = 0; ep < kEPW; ++ep)
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const uint32_t ww[4] = {wv[ep][v].x, wv[ep][v].y, wv[ep][v].z, wv[ep][v].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          sq[ep] = fmaf(bf16lo(ww[i]), bf16lo(ww[i]), sq[ep]);
          sq[ep] = fmaf(bf16hi(ww[i]), bf16hi(ww[i]), sq[ep]);
        }
      }
    if constexpr (Cfg::kStaged) {
      const uint4* xs4 = reinterpret_cast<const uint4*>(xs);
#pragma unroll
      for (int tt = 0; tt < kTT; ++tt) {
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 xv = xs4[tt * (kXCols / 8) + lane + 32 * v];
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int ep = 0; ep < kEPW; ++ep) {
            const uint32_t ww[4] = {wv[ep][v].x, wv[ep][v].y, wv[ep][v].z, wv[ep][v].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[ep][tt][v % NC] = fma_bf16x2(xw[i], ww[i], acc[ep][tt][v % NC]);
          }
        }
      }
      if (xn_warp) {   // ||x_t||^2 from the staged row, same order as the products
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 xv = xs4[warp * (kXCols / 8) + lane + 32 * v];
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) sqx = fma_bf16x2(xw[i], xw[i], sqx);
        }
      }
    } else {
      // one token: its row straight from global memory
      uint4 xv[8];
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const int h = hb + lane * 8 + 256 * v;
        xv[v] = (nt > 0 && h < H) ? *reinterpret_cast<const uint4*>(x + (size_t)t0 * H + h)
                                  : make_uint4(0, 0, 0, 0);
      }
      if (x16 && blockIdx.y == 0 && warp == 0 && nt > 0) {   // the token's f16 row (when asked)
        bool bad = false;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const int h = hb + lane * 8 + 256 * v;
          if (h < H) *reinterpret_cast<uint4*>(x16 + (size_t)t0 * H + h) = bf16x8_to_f16x8(xv[v], bad);
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&hdr->status, kStatusRange);
      }
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const uint32_t xw[4] = {xv[v].x, xv[v].y, xv[v].z, xv[v].w};
        const uint32_t ww[4] = {wv[0][v].x, wv[0][v].y, wv[0][v].z, wv[0][v].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[0][0][v % NC] = fma_bf16x2(xw[i], ww[i], acc[0][0][v % NC]);
          if (xn_warp) sqx = fma_bf16x2(xw[i], xw[i], sqx);
        }
      }
    }
  }
  // the chains pairwise (log2 NC levels), then the lanes (5 levels)
  float dot[kEPW][kTT];
#pragma unroll
  for (int ep = 0; ep < kEPW; ++ep)
#pragma unroll
    for (int tt = 0; tt < kTT; ++tt) {
#pragma unroll
      for (int w = NC / 2; w > 0; w >>= 1)
#pragma unroll
        for (int c = 0; c < w; ++c) acc[ep][tt][c] += acc[ep][tt][c + w];
      dot[ep][tt] = acc[ep][tt][0];
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sqx += __shfl_xor_sync(0xffffffffu, sqx, o);
#pragma unroll
    for (int ep = 0; ep < kEPW; ++ep) {
      sq[ep] += __shfl_xor_sync(0xffffffffu, sq[ep], o);
#pragma unroll
      for (int tt = 0; tt < kTT; ++tt) dot[ep][tt] += __shfl_xor_sync(0xffffffffu, dot[ep][tt], o);
    }
  }
#pragma unroll
  for (int ep = 0; ep < kEPW; ++ep) {
    const int e = e0 + ep;
    if (e >= E) continue;
    float mine = dot[ep][0];
#pragma unroll
    for (int tt = 1; tt < kTT; ++tt) if (lane == tt) mine = dot[ep][tt];
    if (lane < nt) logits[(size_t)(t0 + lane) * E + e] = bias ? mine + bias[e] : mine;
    if (lane == 31) wnorm[e] = sqrtf(sq[ep]);   // the same value from every chunk's CTA
  }
  if (xn_warp && lane == 0) xnorm[t0 + warp] = sqrtf(sqx);
  // Publish the CTA's results and count the CTA in; the last CTA of the
  // chunk sees every other CTA's results.
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomic_add_acq_rel(&cnt[chunk], 1) == (int)gridDim.y - 1;
  __syncthreads();
  if (!s_last) return;

  // ---- last CTA of the chunk: stage logits, ||w_e||, ||x_t|| (one L2 trip)
  // extraction in rank order, one warp per token (chunks of 4 or 8 tokens;
  // for one-token chunks the all-thread ranking is faster: 1.4 against 2.2 us)
  const bool by_warp = kTT >= 4 && E <= 128;
  uint64_t* skey = reinterpret_cast<uint64_t*>(dsm);
  float* sl = reinterpret_cast<float*>(skey + (size_t)kTT * E);
  float* swn = sl + (size_t)kTT * E;
  float* sxn = swn + E;
  // sort keys: order-preserving bits of the logit (NaN lowest, -0 = +0) above
  // the inverted expert index, so a larger key is a better (logit, index)
  for (int i = threadIdx.x; i < nt * E; i += blockDim.x) {
    const float v = __ldcg(logits + (size_t)t0 * E + i);
    sl[i] = v;
    const uint32_t e = (uint32_t)(i % E);
    if (!by_warp) skey[i] = ((uint64_t)order_bits(rank_key(v)) << 32) | (uint64_t)(0xffffffffu - e);
  }
  for (int i = threadIdx.x; i < E; i += blockDim.x) swn[i] = __ldcg(wnorm + i);
  if (threadIdx.x < nt) sxn[threadIdx.x] = __ldcg(xnorm + t0 + threadIdx.x);
  __syncthreads();
  if (!by_warp) {
    // Rank of every (token, expert) by counting the experts ahead of it:
    // larger logit first, lower index first on equal logits, NaN last.  Four
    // threads share an expert, thread q counting over j = q (mod 4).
    for (int tt = 0; tt < nt; ++tt) {
      const uint64_t* krow = skey + (size_t)tt * E;
      for (int base = 0; base < 4 * E; base += blockDim.x) {   // uniform trip count
        const int it = base + threadIdx.x;
        const int q = it & 3, ee = it >> 2;
        int r = 0;
        if (ee < E) {
          const uint64_t key = krow[ee];
#pragma unroll 8
          for (int j = q; j < E; j += 4) r += krow[j] > key ? 1 : 0;
        }
        r += __shfl_xor_sync(0xffffffffu, r, 1);
        r += __shfl_xor_sync(0xffffffffu, r, 2);
        if (ee < E && q == 0 && r < kCandCap) {
          scr[tt].cand_e[r] = ee;
          scr[tt].cand_v[r] = rank_key(sl[(size_t)tt * E + ee]);
        }
      }
    }
    __syncthreads();
  }

  if (warp < nt) {
    const int t = t0 + warp;
    WarpScratch& sc = scr[warp];
    const float* row = sl + (size_t)warp * E;
    float wmax = 0.f, lmax = 0.f;
    for (int ee = lane; ee < E; ee += 32) {
      wmax = fmaxf(wmax, swn[ee]);
      lmax = fmaxf(lmax, fabsf(row[ee]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
      lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
    }
    const float delta = gamma * sxn[warp] * wmax * (1.0f + 0x1p-10f) +
                        0x1p-22f * lmax + (float)H * 0x1p-149f;
    const float thr = cert_threshold(delta);
    const int end = by_warp ? extract_small(row, E, k, thr, sc) : certain_end_ranked(sc, E, k, thr);
    select_begin(E, k, delta, end, sc, idx + (size_t)t * k, w + (size_t)t * k, hdr);
  }
  __syncthreads();
  int ndots = 0;
  for (int tt = 0; tt < nt; ++tt) ndots += scr[tt].nd;
  if (ndots > 0) {   // uniform over the block
    select_dots(scr, nt, t0, x, gw, bias, H, E, l64, s_part);
    if (warp < nt && scr[warp].nd > 0)
      select_end(E, k, scr[warp], l64 + (size_t)(t0 + warp) * E, idx + (size_t)(t0 + warp) * k,
                 w + (size_t)(t0 + warp) * k);
  }
  if constexpr (kGroup) {
    // each routed slot of the chunk takes its rank in its expert's group
    // (arrival order); the expert kernel builds the grouping from these
    __syncthreads();   // the selecting warps' idx writes
    for (int i = threadIdx.x; i < nt * k; i += blockDim.x) {
      const int f = t0 * k + i;
      const int e = idx[f];
      go.rank[f] = (unsigned)e < (unsigned)E ? atomicAdd(&go.acnt[e], 1) : -1;
    }
  }
}

// ------------------------------------------------------------ large batches
// Logits, stream-K over a persistent grid.  A work item is (32-token block b,
// 32-wide K chunk c); the Q = nblocks * nchunks items, block-major, are split
// evenly over the G CTAs of the launch (CTA i: items [iQ/G, (i+1)Q/G)), so
// every SM gets the same number of chunk products whatever T is.  A CTA's
// range may cross block boundaries: for every block it touches it stores one
// piece, the block's partial logits over the chunks it covered, in slot
// p = i - (first CTA of the block); the select kernel adds a block's pieces
// in slot order.  The host sizes G so that a block has at most kTilePieces
// pieces.
//
// Inside a CTA: 4 warps, the even chunks of a segment to warps 0-1 and the
// odd chunks to warps 2-3 (each pair with its own double-buffered tiles and
// named barrier).  In a pair, warp w covers tokens 16(w mod 2) .. +15: lane
// l owns the 8 tokens 8(l / 16) .. +7 of them and the experts 4(l mod 16)
// .. +3 and 64 + 4(l mod 16) .. +3.  The products run on paired fp32 FMAs
// (fma.rn.f32x2: two independent fp32 fmas, each rounded as fmaf): the x
// tile holds every value twice, (x, x), so one 16-byte shared load gives two
// tokens' pairs and one f32x2 fma updates two experts of a token; a step is
// 32 paired fmas from six 16-byte shared loads.  (Four experts a lane, 16
// warps per SM at 128 registers, was slower: 10 more shared loads per 32
// paired fmas.)
//
// Roundings per product: a chunk's 32 products are summed sequentially from
// zero (31), a pair adds its chunk sums in order (at most nchunks/2), the two
// pairs' totals are added once, and the select kernel adds at most
// kTilePieces pieces: 31 + nchunks/2 + 1 + (kTilePieces - 1).
constexpr int kTileT = 32, kTileE = 128, kTileK = 32, kTileThreads = 128, kTilePieces = 4;
// floats of one chunk's tiles: x [kTileK][kTileT] as (x, x) pairs, then w [kTileK][kTileE]
constexpr int kTileXF = 2 * kTileK * kTileT;
constexpr int kTileBuf = kTileXF + kTileK * kTileE;

// The CTA whose item range holds item q (CTA i starts at floor(iQ/G)).
__host__ __device__ inline long long tile_cta_of(long long q, long long Q, long long G) {
  return ((q + 1) * G - 1) / Q;
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// c + a * b and c + a, elementwise on fp32 pairs (each half rounded as the
// scalar fmaf / fadd)
__device__ __forceinline__ float2 fma_f32x2(float2 a, float2 b, float2 c) {
  asm("{\n .reg .b64 ra, rb, rc;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%0, %1};\n fma.rn.f32x2 rc, ra, rb, rc;\n mov.b64 {%0, %1}, rc;\n}"
      : "+f"(c.x), "+f"(c.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return c;
}
__device__ __forceinline__ float2 add_f32x2(float2 a, float2 b) {
  asm("{\n .reg .b64 ra, rb;\n mov.b64 ra, {%0, %1};\n mov.b64 rb, {%2, %3};\n"
      " add.rn.f32x2 ra, ra, rb;\n mov.b64 {%0, %1}, ra;\n}"
      : "+f"(a.x), "+f"(a.y)
      : "f"(b.x), "f"(b.y));
  return a;
}

__global__ void __launch_bounds__(kTileThreads, 2) router_tile_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ gw, int T, int H, int E, int G,
    float* __restrict__ lpart, float* __restrict__ xsq, uint16_t* __restrict__ x16, int* status) {
  pdl_wait();   // programmatic dependent launch: the workspace is ready
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // [pair][buf]: x tile then w tile, fp32
  float* tiles = reinterpret_cast<float*>(smem_raw);
  __shared__ float s_sq[2][kTileT * 4];   // ||x_t||^2 partials of each pair
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int pair = warp >> 1;             // the segment's chunks c0 + pair, c0 + pair + 2, ...
  const int ptid = tid & 63;              // thread index within the pair
  const int tw = (warp & 1) * 16 + (lane >> 4) * 8;   // this lane's first token
  const int ew = 4 * (lane & 15);                     // this lane's first expert (+64)
  const int nchunks = H / kTileK;
  const long long Q = (long long)((T + kTileT - 1) / kTileT) * nchunks;
  long long q = (long long)blockIdx.x * Q / G;
  const long long q_end = (long long)(blockIdx.x + 1) * Q / G;

  // staging of one chunk by the 64 threads of a pair: x 32x32 (128 vectors,
  // 2 per thread), w 128x32 (512 vectors, 8 per thread); vector v covers row
  // v % rows and columns 8*(v / rows) .. +7 (consecutive lanes -> consecutive
  // rows: the transposed stores hit distinct banks)
  uint4 rx[2], rw[8];
  float sqacc[2];   // squares of the staged x values, per vector slot
  auto load_chunk = [&](int t0, int kc) {
    const int k0 = kc * kTileK;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int v = ptid + 64 * i;
      const int row = v % kTileT, col = (v / kTileT) * 8;
      const int t = t0 + row;
      rx[i] = (t < T) ? *reinterpret_cast<const uint4*>(x + (size_t)t * H + k0 + col) : make_uint4(0, 0, 0, 0);
    }
    if (x16) {   // the f16 copy of the token rows (each vector is loaded once in the launch)
      bool bad = false;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int v = ptid + 64 * i;
        const int row = v % kTileT, col = (v / kTileT) * 8;
        const int t = t0 + row;
        if (t < T) *reinterpret_cast<uint4*>(x16 + (size_t)t * H + k0 + col) = bf16x8_to_f16x8(rx[i], bad);
      }
      if (bad) atomicOr(status, kStatusRange);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int v = ptid + 64 * i;
      const int row = v % kTileE, col = (v / kTileE) * 8;
      rw[i] = (row < E) ? *reinterpret_cast<const uint4*>(gw + (size_t)row * H + k0 + col)
                        : make_uint4(0, 0, 0, 0);
    }
  };
  auto store_chunk = [&](int buf) {
    float* xb = tiles + (size_t)(pair * 2 + buf) * kTileBuf;
    float* wb = xb + kTileXF;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int v = ptid + 64 * i;
      const int row = v % kTileT, col = (v / kTileT) * 8;
      const uint32_t u[4] = {rx[i].x, rx[i].y, rx[i].z, rx[i].w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float lo = bf16lo(u[m]), hi = bf16hi(u[m]);
        *reinterpret_cast<float2*>(xb + 2 * ((col + 2 * m) * kTileT + row)) = make_float2(lo, lo);
        *reinterpret_cast<float2*>(xb + 2 * ((col + 2 * m + 1) * kTileT + row)) = make_float2(hi, hi);
        sqacc[i] = fmaf(lo, lo, sqacc[i]);
        sqacc[i] = fmaf(hi, hi, sqacc[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int v = ptid + 64 * i;
      const int row = v % kTileE, col = (v / kTileE) * 8;
      const uint32_t u[4] = {rw[i].x, rw[i].y, rw[i].z, rw[i].w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        wb[(col + 2 * m) * kTileE + row] = bf16lo(u[m]);
        wb[(col + 2 * m + 1) * kTileE + row] = bf16hi(u[m]);
      }
    }
  };

  while (q < q_end) {
    const long long b = q / nchunks;
    const int c0 = (int)(q - b * nchunks);
    const int c1 = (int)min((long long)nchunks, c0 + (q_end - q));
    const int t0 = (int)(b * kTileT);
    const int piece = (int)(blockIdx.x - tile_cta_of(b * nchunks, Q, G));
    __syncthreads();   // the previous segment is done with the tiles

    float2 tot[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) tot[i][j] = make_float2(0.f, 0.f);
    sqacc[0] = sqacc[1] = 0.f;
    int buf = 0;
    if (c0 + pair < c1) {
      load_chunk(t0, c0 + pair);
      store_chunk(0);
    }
    named_sync(1 + pair, 64);
    for (int kc = c0 + pair; kc < c1; kc += 2) {
      const bool more = kc + 2 < c1;
      if (more) load_chunk(t0, kc + 2);
      const float* xb = tiles + (size_t)(pair * 2 + buf) * kTileBuf + 2 * tw;
      const float* wb = tiles + (size_t)(pair * 2 + buf) * kTileBuf + kTileXF + ew;
      float2 part[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) part[i][j] = make_float2(0.f, 0.f);
#pragma unroll 4
      for (int kk = 0; kk < kTileK; ++kk) {
        float4 xv[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) xv[m] = *reinterpret_cast<const float4*>(xb + 2 * kk * kTileT + 4 * m);
        const float4 wa = *reinterpret_cast<const float4*>(wb + kk * kTileE);
        const float4 wc = *reinterpret_cast<const float4*>(wb + kk * kTileE + 64);
        const float2 wp[4] = {make_float2(wa.x, wa.y), make_float2(wa.z, wa.w), make_float2(wc.x, wc.y),
                              make_float2(wc.z, wc.w)};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 xi = (i & 1) ? make_float2(xv[i / 2].z, xv[i / 2].w) : make_float2(xv[i / 2].x, xv[i / 2].y);
#pragma unroll
          for (int j = 0; j < 4; ++j) part[i][j] = fma_f32x2(xi, wp[j], part[i][j]);
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) tot[i][j] = add_f32x2(tot[i][j], part[i][j]);
      if (more) store_chunk(buf ^ 1);
      named_sync(1 + pair, 64);
      buf ^= 1;
    }
    __syncthreads();   // both pairs are done with their tiles
    // pair 1 hands its totals to pair 0 (through the tile memory), which adds
    // them once and stores the piece
    float* xfer = tiles;   // [64 threads][64]
    if (pair == 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          xfer[(i * 8 + 2 * j) * 64 + ptid] = tot[i][j].x;
          xfer[(i * 8 + 2 * j + 1) * 64 + ptid] = tot[i][j].y;
        }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) s_sq[pair][ptid + 64 * i] = sqacc[i];
    __syncthreads();
    if (pair == 0) {
      float* dst = lpart + (size_t)piece * T * E;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int t = t0 + tw + i;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int e = (j < 2 ? 0 : 64) + ew + 2 * (j & 1);
          const float v0 = tot[i][j].x + xfer[(i * 8 + 2 * j) * 64 + ptid];
          const float v1 = tot[i][j].y + xfer[(i * 8 + 2 * j + 1) * 64 + ptid];
          if (t < T && e < E) dst[(size_t)t * E + e] = v0;
          if (t < T && e + 1 < E) dst[(size_t)t * E + e + 1] = v1;
        }
      }
    }
    // ||x_t||^2 over the segment: row t's partials are the vector slots
    // v = t + 32c (c = 0..3) of both pairs
    if (tid < kTileT && t0 + tid < T) {
      float sq = 0.f;
#pragma unroll
      for (int p2 = 0; p2 < 2; ++p2)
#pragma unroll
        for (int c = 0; c < 4; ++c) sq += s_sq[p2][tid + kTileT * c];
      xsq[(size_t)piece * T + t0 + tid] = sq;
    }
    q += c1 - c0;
  }
}

// Selection for the tiled path (E <= 128): one warp per token.  The token's
// logits are the sum of its block's stream-K pieces in slot order (then the
// bias), ||x_t|| the root of its pieces' partial squares; logits and expert
// norms are loaded in one batch (lane l: experts l + 32i) and ranked from
// registers.
__global__ void __launch_bounds__(256, 3) router_select_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ gw, const float* __restrict__ bias,
    int T, int H, int E, int k, float gamma, const float* __restrict__ lpart,
    const float* __restrict__ xsq, int G, const float* __restrict__ wnorm, double* __restrict__ l64,
    int32_t* __restrict__ idx, float* __restrict__ w, void* ws) {
  pdl_wait();   // the logits and norms are complete
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ DotPart s_part[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WarpScratch* scr = reinterpret_cast<WarpScratch*>(smem_raw);
  const int t0 = blockIdx.x * 8;
  const int nt = min(8, T - t0);
  const int t = t0 + warp;
  if (warp < nt) {
    // the token block's pieces (slot order), then the bias
    const int nchunks = H / kTileK;
    const long long Q = (long long)((T + kTileT - 1) / kTileT) * nchunks;
    const long long qb = (long long)(t / kTileT) * nchunks;
    const int np = (int)(tile_cta_of(qb + nchunks - 1, Q, G) - tile_cta_of(qb, Q, G)) + 1;
    float v[4], wn[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < E ? lpart[(size_t)t * E + e] : 0.0f;
      wn[i] = e < E ? wnorm[e] : 0.0f;
    }
    float xs = xsq[t];
    for (int p = 1; p < np; ++p) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e = lane + 32 * i;
        if (e < E) v[i] += lpart[((size_t)p * T + t) * E + e];
      }
      xs += xsq[(size_t)p * T + t];
    }
    if (bias) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e = lane + 32 * i;
        if (e < E) v[i] += bias[e];
      }
    }
    const float xn = sqrtf(xs);
    float wmax = 0.f, lmax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      wmax = fmaxf(wmax, wn[i]);
      lmax = fmaxf(lmax, fabsf(v[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
      lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
    }
    const float delta = gamma * xn * wmax * (1.0f + 0x1p-10f) +
                        0x1p-22f * lmax + (float)H * 0x1p-149f;
    const int end = extract_regs(v, E, k, cert_threshold(delta), scr[warp]);
    select_begin(E, k, delta, end, scr[warp], idx + (size_t)t * k, w + (size_t)t * k,
                 reinterpret_cast<WsHeader*>(ws));
  }
  __syncthreads();
  int ndots = 0;
  for (int tt = 0; tt < nt; ++tt) ndots += scr[tt].nd;
  if (ndots == 0) return;   // uniform over the block
  select_dots(scr, nt, t0, x, gw, bias, H, E, l64, s_part);
  if (warp < nt && scr[warp].nd > 0)
    select_end(E, k, scr[warp], l64 + (size_t)t * E, idx + (size_t)t * k, w + (size_t)t * k);
}

// ||w_e|| for every expert, one warp per expert.
__global__ void __launch_bounds__(256) wnorm_kernel(const uint16_t* __restrict__ gw, int H, int E,
                                                    float* __restrict__ wnorm) {
  pdl_wait();
  pdl_trigger();   // the logits kernel does not read ||w_e||; it may launch at once
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

bool route_can_group(int T, int E, int k) {
  // the expert kernels keep a self-grouped batch's permutation in shared
  // memory: at most 4096 slots
  return !(T >= 2048 && E <= 128) && T * k <= 4096;
}

cudaError_t launch_route(const uint16_t* x, const uint16_t* gate_w, const float* bias, int T, int H,
                         int E, int k, int32_t* idx, float* w, void* ws, const WsLayout& L,
                         cudaStream_t stream, int* launches, const GroupOut* group, uint16_t* x16) {
  float* wnorm = ws_ptr<float>(ws, L.wnorm);
  double* l64 = ws_ptr<double>(ws, L.logits64);
  const bool tiled = route_tiled(T, E);
  if (launches) *launches += tiled ? 3 : 1;
  if (tiled) {
    static_assert(kTilePieces == kRouteTilePieces && kTileE == kRouteTileMaxE, "workspace pieces");
    float* lpart = ws_ptr<float>(ws, L.lpart);
    float* xsq = ws_ptr<float>(ws, L.xsq);
    cudaError_t err = launch_pdl(wnorm_kernel, dim3((E + 7) / 8), dim3(256), 0, stream, gate_w, H, E, wnorm);
    if (err != cudaSuccess) return err;
    int dev = 0, sms = 0;
    err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    // two CTAs per SM; at least ceil((nchunks - 1) / (kTilePieces - 1)) items
    // per CTA, so that no block has more than kTilePieces pieces
    const int nchunks = H / kTileK;
    const long long Q = (long long)((T + kTileT - 1) / kTileT) * nchunks;
    const long long per_min = std::max(1, (nchunks - 1 + kTilePieces - 2) / (kTilePieces - 1));
    long long G = std::max(1LL, std::min(2LL * sms, Q / per_min));
    if (G > sms && G < 2LL * sms) G = sms;   // whole CTAs per SM: one each rather than one or two
    const size_t smem = sizeof(float) * 4 * kTileBuf;
    err = cudaFuncSetAttribute(router_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    err = launch_pdl(router_tile_kernel, dim3((unsigned)G), dim3(kTileThreads), smem, stream, x, gate_w, T, H, E, (int)G,
                     lpart, xsq, x16, &reinterpret_cast<WsHeader*>(ws)->status);
    if (err != cudaSuccess) return err;
    const size_t smem2 = sizeof(WarpScratch) * 8;
    err = cudaFuncSetAttribute(router_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem2);
    if (err != cudaSuccess) return err;
    // roundings per product: chunk sum, a pair's chunk sums, the pair
    // totals, the pieces
    const float gamma = gamma_bound(kTileK - 1 + (nchunks + 1) / 2 + 1 + (kTilePieces - 1));
    return launch_pdl(router_select_kernel, dim3((T + 7) / 8), dim3(256), smem2, stream, x, gate_w, bias, T, H,
                      E, k, gamma, (const float*)lpart, (const float*)xsq, (int)G, (const float*)wnorm, l64, idx, w,
                      ws);
  }
  const int tt = T <= 16 ? 1 : T <= 128 ? 4 : 8;
  // roundings per product: the lane's chain (at most 64 per 2048 columns
  // over the chains, and never more than the lane's H/32 products), the
  // chain tree, the 5-level lane tree
  const int nc = tt == 1 ? SmallCfg<1>::kChains : tt == 4 ? SmallCfg<4>::kChains : SmallCfg<8>::kChains;
  const int per_chain = std::min(H / 32, 64 * ((H + 2047) / 2048) / nc);
  const float gamma = gamma_bound(per_chain + (nc == 8 ? 3 : nc == 2 ? 1 : 0) + 5);
  const bool grp = group != nullptr;
  const size_t smem = router_small_smem(E, tt);
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  const int per_cta = tt >= 4 ? SmallCfg<4>::kExperts : SmallCfg<1>::kExperts;
  const dim3 grid((unsigned)((T + tt - 1) / tt), (unsigned)((E + per_cta - 1) / per_cta));
  int* cnt = ws_ptr<int>(ws, L.cnt);
  float* logits = ws_ptr<float>(ws, L.logits);
  float* xnorm = ws_ptr<float>(ws, L.xnorm);
  const GroupOut go = grp ? *group : GroupOut{};
  auto run = [&](auto kern) -> cudaError_t {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    // programmatic launch: the CTAs may become resident while the workspace
    // is being cleared and wait for it on the device
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kSmallWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, x, gate_w, bias, T, H, E, k, gamma, logits, wnorm, xnorm,
                              l64, cnt, idx, w, ws, go, x16);
  };
  if (grp) {
    if (tt == 1) return run(router_small_kernel<1, true>);
    if (tt == 4) return run(router_small_kernel<4, true>);
    return run(router_small_kernel<8, true>);
  }
  if (tt == 1) return run(router_small_kernel<1, false>);
  if (tt == 4) return run(router_small_kernel<4, false>);
  return run(router_small_kernel<8, false>);
}

}  // namespace moe
