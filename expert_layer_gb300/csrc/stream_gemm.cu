// Weight-streaming grouped expert GEMMs for small groups (decode-sized).
//
// The "expert kernel" and "activation" phases of the fused-MoE path (page
// "Decode 吞吐专项实验分析报告", section "下一步 profiling 方向", item 3) for
// experts that hold few routed rows.  At decode batch sizes these are bound by
// HBM: every active expert's weights are read once and each weight meets only
// a handful of token rows.  The kernels therefore stream the weights with
// coalesced 128-bit loads that bypass L1, keep the (small, reused) activation
// rows in L1/L2, and do the arithmetic on mma.sync m16n8k16 (bf16 in, fp32
// accumulate) with the weights as the 16-row A operand and up to 64 gathered
// token rows as the B operand ("swap AB").  This replaces the ncols <= 8 MMVQ
// templates of page "第 9 章 prefill：最大的瓶颈" (sec. 9.5): any number of rows
// per expert is served, in passes of up to 64.
//
// Work unit = (active expert, 16 weight rows over the whole K), owned by one
// warp.
//   gate/up: A rows 0-7 are gate rows j0..j0+7, rows 8-15 the matching up rows
//            I+j0..I+j0+7, so one fragment holds g and u of the same j and the
//            SwiGLU h = silu(g)*u is formed in the epilogue (h rounded to bf16).
//   down:    A rows are 16 consecutive output features d0..d0+15; the epilogue
//            scales by the routing weight and writes the slot's partial row.
// A warp sums its unit's whole K itself, so results do not depend on the
// launch shape (deterministic).
//
// K-index assignment inside one mma: thread (g, c) of a warp loads 8
// consecutive bf16 (one 16-byte vector) of rows g and g+8 at k = 8c..8c+7 of
// each 32-wide K block; step q of the block feeds pairs (8c+4q, +1) and
// (8c+4q+2, +3) to the fragment slots (2c, 2c+1) and (2c+8, 2c+9).  The B
// operand uses the same assignment, so every k meets its own partner exactly
// once: a permutation of the summation inside each 16-wide step, nothing else.
//
// NVFP4 weights (W4A16): the A fragments are decoded in registers and the
// MMA runs on f16 operands.  Thread (g, c) loads 16 bytes of codes (32
// elements, k = 32c..32c+31 of a 128-wide block) and the two e4m3 scales of
// those 32 elements; the hardware conversions cvt.rn.f16x2.e2m1x2 (a code
// byte to two f16, low nibble to the low half) and cvt.rn.f16x2.e4m3x2 (the
// scale) are exact, and so is their f16 product (an e2m1 value times an e4m3
// value has at most 6 significant bits and lies in [2^-10, 2688]); the
// per-expert fp32 global scale multiplies the fp32 accumulator in the
// epilogue.  The token rows are x converted to f16 beforehand
// (by the router) and h, which the gate/up epilogue writes in f16 on this
// path: exact for activations of magnitude 2^-14 .. 65504, below that
// rounded to the f16 subnormal grid (absolute error <= 2^-25), above it
// flagged (kStatusRange).
//
// Int8 block weights (W8A16): int8 codes with one fp16 scale per 32
// consecutive elements along K.  Thread (g, c) loads, per 64-wide K block, 8
// codes of each of the block's two scale blocks (k = 8c..8c+7 and
// 32+8c..32+8c+7), so every mma step stays inside one scale block.  Codes
// become f16 exactly (integers of magnitude <= 127), the mma sums code x
// activation over one scale block on the f16 token rows (the products are
// exact in the fp32 accumulator), and the row's scale multiplies that fp32
// partial sum before it joins the accumulator.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "nvfp4.cuh"
#include "stream_common.cuh"

namespace moe {

namespace {

using namespace stream;


// Pipeline shape per variant (NT = 8-row token tiles per pass).  A unit is
// FR fragments of 16 weight rows.  NVFP4 and int8 units are two or four
// fragments tall: each token-row fragment a thread loads then feeds FR mma
// instead of one, which matters because 4- and 8-bit weights make the token
// rows (16-bit) the larger stream whenever an expert holds more than a few
// rows.  With four token tiles (32 rows per pass, for experts averaging 24
// rows or more) the unit is two fragments tall, so that an expert of up to
// 32 rows decodes its weights once.
template <int F, int NT = 1>
struct StreamCfg {
  static constexpr bool kFp4 = F == kFmtFp4, kQ8 = F == kFmtQ8;
  static constexpr bool kDec = kFp4 || kQ8;       // decoded weights, f16 operands
  static constexpr int KB = kFp4 ? 128 : kQ8 ? 64 : 32;   // K elements per block
  static constexpr int KG = kDec ? 1 : 4;         // blocks per pipelined group
  static constexpr int FR = kDec ? (NT >= 4 ? 2 : 4) : 1;   // 16-row fragments per unit
  // groups in the ring (NS-1 in flight).  bf16: three, which leaves more of
  // the SM's unified L1 / shared memory to the token rows the warps share in
  // L1 (decode64 streaming stage 188 -> 179 us against four)
  static constexpr int NS = kDec ? (NT >= 4 ? 5 : 3) : 3;
  static constexpr int kWarps = kDec ? 8 : 12;
  // per-warp ring: [NS][KG][FR][2 rows][32 lanes] x 16 B of weights (codes),
  // plus the block scales of the decoded formats
  static constexpr int kWBytes = NS * KG * FR * 2 * 32 * 16;
  // per fragment and block the scales of each of its 16 weight rows (one
  // copy per row, read by the four lanes that use it): NVFP4 8 e4m3 bytes,
  // int8 two fp16 scales
  static constexpr int kSBytes = kFp4 ? NS * KG * FR * 16 * 8 : kQ8 ? NS * KG * FR * 16 * 4 : 0;
  static constexpr int kWarpBytes = kWBytes + kSBytes;
  static constexpr int kLutBytes = 0;
};

// B (token rows) of one K group for this thread (bf16 weights): row g of
// the pass, k = 8c..8c+7 of each 32-wide block.  Down reads h, written
// earlier in the same launch, through L2 (ld.cg).
template <int KG>
__device__ __forceinline__ void load_b(uint32_t (&b)[KG][4], const uint16_t* bsrc, int gi, int nkb,
                                       int c, bool cg) {
#pragma unroll
  for (int i = 0; i < KG; ++i) {
    const int kb = gi * KG + i;
    uint4 t = make_uint4(0, 0, 0, 0);
    if (bsrc && kb < nkb) {
      const uint4* p = reinterpret_cast<const uint4*>(bsrc + (size_t)kb * 32 + 8 * c);
      t = cg ? __ldcg(p) : *p;
    }
    b[i][0] = t.x; b[i][1] = t.y; b[i][2] = t.z; b[i][3] = t.w;
  }
}

// Gate/up and down of the small groups in one persistent launch.  Each warp
// owns whole units: no cross-warp reduction, so results do not depend on the
// launch shape.  A warp takes its first unit by its global index and every
// later one from an atomic queue counter, requested one unit early so the
// atomic's latency is hidden; the dynamic queue keeps the warps busy to the
// end of the layer instead of to the end of each projection.  A down unit of
// expert e waits until every gate/up unit of e has published its h rows (a
// per-expert counter, release / acquire).  All gate/up positions precede all
// down positions and a warp takes positions in increasing order, so no warp
// holds a gate/up unit behind a waiting down unit: every wait ends.
// Weights stream through a private per-thread ring in shared memory filled by
// cp.async (each thread copies exactly the 16-byte pieces it will later
// read), NS-1 groups ahead of the mma and across unit boundaries; the token
// rows (B) of the next group are loaded into registers one group ahead.
// Experts with more than 8*NT routed rows take several passes; later passes
// re-read the unit's weights from L2.
template <int F, int NT>
__global__ void __launch_bounds__(StreamCfg<F, NT>::kWarps * 32, 1) stream_gemm_kernel(StreamGemmArgs a) {
  using C = StreamCfg<F, NT>;
  constexpr bool kFp4 = C::kFp4, kQ8 = C::kQ8;
  constexpr int KB = C::KB, KG = C::KG, NS = C::NS, NW = C::kWarps;
  constexpr int kFifo = 8;   // > NS: unit ids the producer may hold ahead of the consumer
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int fifo[NW][kFifo];
  int4* smeta = reinterpret_cast<int4*>(smem + NW * C::kWarpBytes + C::kLutBytes);   // [E]
  int* sperm = reinterpret_cast<int*>(smeta + a.E);                                 // [S]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  uint4* ring = reinterpret_cast<uint4*>(smem + warp * C::kWarpBytes);
  uint2* sring = reinterpret_cast<uint2*>(smem + warp * C::kWarpBytes + C::kWBytes);

  // the grouping is complete once the kernel before this one is; the
  // combine may start launching
  pdl_wait();
  pdl_trigger();
  const int S = a.T * a.k;
  const bool perm_smem = a.self_group || S <= kPermSmem;
  int nsmall;
  if (a.self_group) {
    // small batch: the grouping from the router's arrival ranks, per CTA
    // (its scratch lives in the weight ring, unused until the first copy)
    nsmall = self_group(a, smeta, sperm, reinterpret_cast<int*>(smem), reinterpret_cast<int*>(smem) + a.E);
  } else {
    // the small groups' metadata, and the slot permutation when it is
    // short, once per CTA: no dependent global loads when a warp changes unit
    nsmall = *a.num_active - (a.num_large ? *a.num_large : 0);
    for (int i = threadIdx.x; i < nsmall; i += blockDim.x) {
      int e = a.active[i];
      if (!bounds_ok((unsigned)e < (unsigned)a.E, a.status)) e = 0;
      int m = a.counts[e], off = a.offsets[e];
      if (!bounds_ok(off >= 0 && m >= 0 && off + m <= a.T * a.k, a.status)) m = 0, off = 0;
      smeta[i] = make_int4(e, m, off, 0);
    }
    if (perm_smem)
      for (int i = threadIdx.x; i < S; i += blockDim.x) sperm[i] = a.perm[i];
    __syncthreads();
  }
  Queue qs;
  constexpr int FR = C::FR;
  qs.UPEg = a.I / (8 * FR);
  qs.UPEd = a.H / (16 * FR);
  qs.Ug = nsmall * qs.UPEg;
  qs.Q = qs.Ug + nsmall * qs.UPEd;
  qs.nkb_g = a.H / KB;
  qs.nkb_d = a.I / KB;
  const int nwarps = (int)gridDim.x * NW;
  const int* permp = perm_smem ? sperm : a.perm;

  // unit ids: the first by global warp index, later ones nwarps + ticket
  int pending = 0;   // lane 0: the next ticket, requested one unit early
  if (lane == 0) pending = nwarps + atomicAdd(a.queue, 1);
  int first = (int)blockIdx.x * NW + warp;
  auto fetch = [&]() -> int {
    if (first >= 0) { const int q = first; first = -1; return q; }
    const int q = __shfl_sync(0xffffffffu, pending, 0);
    if (lane == 0 && q < qs.Q) pending = nwarps + atomicAdd(a.queue, 1);
    return q;
  };
  int pw = 0, pr = 0;   // fifo push / pop counts (same in every lane)
  auto push = [&](int q) {
    if (lane == 0) fifo[warp][pw % kFifo] = q;
    ++pw;
  };

  // ---- producer side: the next group to copy
  Task it;
  {
    const int q = fetch();
    push(q);
    task_load<KG, NT>(it, smeta, qs, q);
  }
  int ig = 0;        // group index within the producer's pass
  int slot_w = 0;    // ring slot the producer fills next
  auto issue_next = [&]() {
    if (it.q >= 0) {
      const int K = it.down ? a.I : a.H;
      const int NR = it.down ? a.H : 2 * a.I;
#pragma unroll
      for (int f = 0; f < FR; ++f) {
      int rlo, rhi;
      if (it.down) { rlo = (it.blk * FR + f) * 16 + g; rhi = rlo + 8; }
      else { rlo = (it.blk * FR + f) * 8 + g; rhi = a.I + rlo; }
      const size_t Rlo = (size_t)it.e * NR + rlo, Rhi = (size_t)it.e * NR + rhi;
#pragma unroll
      for (int i = 0; i < KG; ++i) {
        const int kb = ig * KG + i;
        uint4* d = ring + (((slot_w * KG + i) * FR + f) * 2) * 32 + lane;
        if (kb < it.nkb) {
          if constexpr (kFp4) {
            const uint8_t* cb = it.down ? a.dn_codes : a.gu_codes;
            const uint8_t* sb = it.down ? a.dn_scales : a.gu_scales;
            const size_t kc = (size_t)kb * 64 + 16 * c;
            cp_async16(d, cb + Rlo * (K / 2) + kc);
            cp_async16(d + 32, cb + Rhi * (K / 2) + kc);
            // lanes 0-7: rows g = lane of the low half, lanes 8-15 the high half
            if (lane < 16) {
              const int r = lane & 7;
              const int srow = it.down ? (it.blk * FR + f) * 16 + r + (lane & 8)
                                       : (it.blk * FR + f) * 8 + r + ((lane & 8) ? a.I : 0);
              cp_async8(sring + ((slot_w * KG + i) * FR + f) * 16 + lane,
                        sb + ((size_t)it.e * NR + srow) * (K / 16) + (size_t)kb * 8);
            }
          } else if constexpr (kQ8) {
            // 8 codes of each of the block's two 32-element scale blocks:
            // k = 8c..8c+7 and 32+8c..32+8c+7, so that every mma step stays
            // inside one scale block
            const int8_t* cb = it.down ? a.dn_q8 : a.gu_q8;
            const uint16_t* sb = it.down ? a.dn_q8s : a.gu_q8s;
            const size_t kc = (size_t)kb * 64 + 8 * c;
            unsigned char* dl = reinterpret_cast<unsigned char*>(d);
            unsigned char* dh = reinterpret_cast<unsigned char*>(d + 32);
            cp_async8(dl, cb + Rlo * K + kc);
            cp_async8(dl + 8, cb + Rlo * K + kc + 32);
            cp_async8(dh, cb + Rhi * K + kc);
            cp_async8(dh + 8, cb + Rhi * K + kc + 32);
            // lanes 0-7: the two fp16 scales of row g = lane of the low half,
            // lanes 8-15 of the high half
            if (lane < 16) {
              const int r = lane & 7;
              const int srow = it.down ? (it.blk * FR + f) * 16 + r + (lane & 8)
                                       : (it.blk * FR + f) * 8 + r + ((lane & 8) ? a.I : 0);
              cp_async4(reinterpret_cast<uint32_t*>(sring) + ((slot_w * KG + i) * FR + f) * 16 + lane,
                        sb + ((size_t)it.e * NR + srow) * (K / 32) + (size_t)kb * 2);
            }
          } else {
            const uint16_t* wb = it.down ? a.w_down : a.w_gate_up;
            const size_t kc = (size_t)kb * 32 + 8 * c;
            cp_async16(d, wb + Rlo * K + kc);
            cp_async16(d + 32, wb + Rhi * K + kc);
          }
        }
      }
      }
      if (++ig == it.ngroups) {
        ig = 0;
        if (++it.pass >= it.npass) {
          const int q = fetch();
          push(q);
          task_load<KG, NT>(it, smeta, qs, q);
        }
      }
    }
    cp_async_commit();
    slot_w = slot_w + 1 == NS ? 0 : slot_w + 1;
  };

#pragma unroll 1
  for (int s = 0; s < NS - 1; ++s) issue_next();

  // ---- consumer side
  Task ct;
  auto pop = [&]() {
    __syncwarp();   // lane 0's fifo store is visible to the warp
    const int q = fifo[warp][pr % kFifo];
    ++pr;
    task_load<KG, NT>(ct, smeta, qs, q);
  };
  pop();
  int slot_r = 0;
  while (ct.q >= 0) {
    if (ct.down && ct.pass == 0) {
      // h of this expert is complete once every gate/up unit of it published
      if (lane == 0) {
        int n = 0;
        while (ld_acquire(a.dep + ct.slot) < qs.UPEg + a.wait_extra) {
          if (++n > a.spin_limit) { atomicOr(a.status, kStatusTimeout); break; }
          __nanosleep(128);
        }
      }
      __syncwarp();
    }
    const int p0 = ct.pass * 8 * NT;
    // one pass over K against NP token tiles (8 rows each) starting at p0
    auto run_pass = [&](auto np_tag) {
      constexpr int NP = decltype(np_tag)::value;
      const uint16_t* bsrc[NP];
  #pragma unroll
      for (int nt = 0; nt < NP; ++nt) {
        const int n = p0 + nt * 8 + g;
        bsrc[nt] = nullptr;
        if (n < ct.m) {
          if (ct.down) bsrc[nt] = a.h + (size_t)(ct.off + n) * a.I;
          else {
            int f = permp[ct.off + n];
            if (!bounds_ok((unsigned)f < (unsigned)(a.T * a.k), a.status)) f = 0;
            bsrc[nt] = (C::kDec ? a.x16 : a.x) + (size_t)(f / a.k) * a.H;
          }
        }
      }
      // down: the epilogue's slots and routing weights, fetched now
      int ef[NP][2];
      float ew[NP][2];
  #pragma unroll
      for (int nt = 0; nt < NP; ++nt)
  #pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int n = p0 + nt * 8 + 2 * c + h2;
          ef[nt][h2] = 0;
          ew[nt][h2] = 0.f;
          if (ct.down && n < ct.m) {
            ef[nt][h2] = permp[ct.off + n];
            if (!bounds_ok((unsigned)ef[nt][h2] < (unsigned)(a.T * a.k), a.status)) ef[nt][h2] = 0;
            ew[nt][h2] = a.topk_w[ef[nt][h2]];
          }
        }
      // tiles of the pass that hold rows: bf16 and int8 passes run with NP =
      // that count (the caller's dispatch); NVFP4 keeps one NP = NT copy of
      // its long decode loop and skips the empty tiles' mma
      const int ntiles = kFp4 ? min(NP, (ct.m - p0 + 7) / 8) : NP;
      float acc[FR][NP][4];
  #pragma unroll
      for (int f = 0; f < FR; ++f)
  #pragma unroll
        for (int nt = 0; nt < NP; ++nt) acc[f][nt][0] = acc[f][nt][1] = acc[f][nt][2] = acc[f][nt][3] = 0.f;
      if constexpr (kFp4) {
        // NVFP4: token rows double-buffered in half blocks (64 K elements = the
        // four mma steps that use one scale byte of each row)
        uint32_t bh[2][NP][8];
        auto load_half = [&](uint32_t (&b)[NP][8], int kb, int hf) {
  #pragma unroll
          for (int nt = 0; nt < NP; ++nt) {
  #pragma unroll
            for (int v = 0; v < 2; ++v) {
              uint4 t = make_uint4(0, 0, 0, 0);
              if (nt < ntiles && bsrc[nt] && kb < ct.nkb) {
                const uint4* pp = reinterpret_cast<const uint4*>(bsrc[nt] + (size_t)kb * 128 + 32 * c +
                                                                 8 * (2 * hf + v));
                t = ct.down ? __ldcg(pp) : *pp;
              }
              b[nt][4 * v + 0] = t.x; b[nt][4 * v + 1] = t.y; b[nt][4 * v + 2] = t.z; b[nt][4 * v + 3] = t.w;
            }
          }
        };
        load_half(bh[0], 0, 0);
  #pragma unroll 1
        for (int gi = 0; gi < ct.ngroups; ++gi) {   // KG = 1: group gi = block gi
          load_half(bh[1], gi, 1);
          cp_async_wait<NS - 2>();
          // the scale rows were copied by other lanes: their copies of this
          // block are complete and visible after the barrier, and every lane
          // has finished reading the slot the next copies overwrite
          __syncwarp();
  #pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            if (hf == 1) load_half(bh[0], gi + 1, 0);
            // codes and scales of all FR fragments first, then the four k
            // steps with the fragments innermost: consecutive MMAs go to
            // different accumulators, so their latencies overlap
            uint32_t sl2[FR], sh2[FR], clo[FR][2], chi[FR][2];
  #pragma unroll
            for (int f = 0; f < FR; ++f) {
              const int rs = ((slot_r * FR + f) * 2) * 32 + lane;
              const uint4 alo = ring[rs];
              const uint4 ahi = ring[rs + 32];
              const uint2 slo8 = sring[(slot_r * FR + f) * 16 + g];
              const uint2 shi8 = sring[(slot_r * FR + f) * 16 + 8 + g];
              // this thread's scale for this half: byte 2c + hf of the row's 8;
              // rows g and g+8 converted together, then each as an f16 pair {s, s}
              const uint32_t slo = (c < 2 ? slo8.x : slo8.y) >> (16 * (c & 1) + 8 * hf);
              const uint32_t shi = (c < 2 ? shi8.x : shi8.y) >> (16 * (c & 1) + 8 * hf);
              const uint32_t s2 = nvfp4::e4m3x2_f16x2((slo & 0xffu) | ((shi & 0xffu) << 8));
              sl2[f] = __byte_perm(s2, 0, 0x1010);
              sh2[f] = __byte_perm(s2, 0, 0x3232);
              clo[f][0] = hf ? alo.z : alo.x;
              clo[f][1] = hf ? alo.w : alo.y;
              chi[f][0] = hf ? ahi.z : ahi.x;
              chi[f][1] = hf ? ahi.w : ahi.y;
            }
  #pragma unroll
            for (int q = 0; q < 4; ++q) {
  #pragma unroll
              for (int f = 0; f < FR; ++f) {
                const uint32_t wl = clo[f][q >> 1] >> (16 * (q & 1));
                const uint32_t wh = chi[f][q >> 1] >> (16 * (q & 1));
                uint32_t l0, l1, h0, h1;
                nvfp4::e2m1x4_f16x2(wl, l0, l1);
                nvfp4::e2m1x4_f16x2(wh, h0, h1);
                const uint32_t a0 = nvfp4::f16x2_mul(l0, sl2[f]);
                const uint32_t a2 = nvfp4::f16x2_mul(l1, sl2[f]);
                const uint32_t a1 = nvfp4::f16x2_mul(h0, sh2[f]);
                const uint32_t a3 = nvfp4::f16x2_mul(h1, sh2[f]);
  #pragma unroll
                for (int nt = 0; nt < NP; ++nt)
                  if (nt < ntiles) mma_f16_16816(acc[f][nt], a0, a1, a2, a3, bh[hf][nt][2 * q], bh[hf][nt][2 * q + 1]);
              }
            }
          }
          slot_r = slot_r + 1 == NS ? 0 : slot_r + 1;
          issue_next();
        }
      } else if constexpr (kQ8) {
        // int8: token rows double-buffered per 32-element scale block (one
        // 16-byte piece per token tile: k = 8c..8c+7 of the block)
        uint32_t bh[2][NP][4];
        auto load_half = [&](uint32_t (&b)[NP][4], int kb, int hf) {
  #pragma unroll
          for (int nt = 0; nt < NP; ++nt) {
            uint4 t = make_uint4(0, 0, 0, 0);
            if (nt < ntiles && bsrc[nt] && kb < ct.nkb) {
              const uint4* pp = reinterpret_cast<const uint4*>(bsrc[nt] + (size_t)kb * 64 + 32 * hf + 8 * c);
              t = ct.down ? __ldcg(pp) : *pp;
            }
            b[nt][0] = t.x; b[nt][1] = t.y; b[nt][2] = t.z; b[nt][3] = t.w;
          }
        };
        const uint32_t* qring = reinterpret_cast<const uint32_t*>(sring);
        load_half(bh[0], 0, 0);
  #pragma unroll 1
        for (int gi = 0; gi < ct.ngroups; ++gi) {   // KG = 1: group gi = block gi
          load_half(bh[1], gi, 1);
          cp_async_wait<NS - 2>();
          __syncwarp();   // the scale rows were copied by other lanes
  #pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            if (hf == 1) load_half(bh[0], gi + 1, 0);
            // the block's codes and scales of all FR fragments; the mma sums
            // code x activation of one scale block (exact products, fp32
            // sums), then the scale multiplies the fp32 partial
            uint32_t clo[FR][2], chi[FR][2];
            float slo[FR], shi[FR];
  #pragma unroll
            for (int f = 0; f < FR; ++f) {
              const int rs = ((slot_r * FR + f) * 2) * 32 + lane;
              const uint4 alo = ring[rs];
              const uint4 ahi = ring[rs + 32];
              slo[f] = q8::f16_half_to_f32(qring[(slot_r * FR + f) * 16 + g], hf);
              shi[f] = q8::f16_half_to_f32(qring[(slot_r * FR + f) * 16 + 8 + g], hf);
              clo[f][0] = hf ? alo.z : alo.x;
              clo[f][1] = hf ? alo.w : alo.y;
              chi[f][0] = hf ? ahi.z : ahi.x;
              chi[f][1] = hf ? ahi.w : ahi.y;
            }
            float part[FR][NP][4];
  #pragma unroll
            for (int f = 0; f < FR; ++f)
  #pragma unroll
              for (int nt = 0; nt < NP; ++nt) part[f][nt][0] = part[f][nt][1] = part[f][nt][2] = part[f][nt][3] = 0.f;
  #pragma unroll
            for (int q = 0; q < 2; ++q) {
  #pragma unroll
              for (int f = 0; f < FR; ++f) {
                uint32_t a0, a2, a1, a3;
                q8::s8x4_f16x2(clo[f][q], a0, a2);
                q8::s8x4_f16x2(chi[f][q], a1, a3);
  #pragma unroll
                for (int nt = 0; nt < NP; ++nt)
                  if (nt < ntiles) mma_f16_16816(part[f][nt], a0, a1, a2, a3, bh[hf][nt][2 * q], bh[hf][nt][2 * q + 1]);
              }
            }
  #pragma unroll
            for (int f = 0; f < FR; ++f)
  #pragma unroll
              for (int nt = 0; nt < NP; ++nt) {
                acc[f][nt][0] = fmaf(slo[f], part[f][nt][0], acc[f][nt][0]);
                acc[f][nt][1] = fmaf(slo[f], part[f][nt][1], acc[f][nt][1]);
                acc[f][nt][2] = fmaf(shi[f], part[f][nt][2], acc[f][nt][2]);
                acc[f][nt][3] = fmaf(shi[f], part[f][nt][3], acc[f][nt][3]);
              }
          }
          slot_r = slot_r + 1 == NS ? 0 : slot_r + 1;
          issue_next();
        }
      } else {
      uint32_t bc[NP][KG][4], bn[NP][KG][4];
    #pragma unroll
        for (int nt = 0; nt < NP; ++nt)
          load_b<KG>(bc[nt], nt < ntiles ? bsrc[nt] : nullptr, 0, ct.nkb, c, ct.down);

    #pragma unroll 1
        for (int gi = 0; gi < ct.ngroups; ++gi) {
          if (gi + 1 < ct.ngroups) {
    #pragma unroll
            for (int nt = 0; nt < NP; ++nt)
              load_b<KG>(bn[nt], nt < ntiles ? bsrc[nt] : nullptr, gi + 1, ct.nkb, c, ct.down);
          }
          cp_async_wait<NS - 2>();
    #pragma unroll
          for (int i = 0; i < KG; ++i) {
            const int kb = gi * KG + i;
            if (kb >= ct.nkb) continue;
    #pragma unroll
            for (int f = 0; f < FR; ++f) {
            const uint4 alo = ring[(((slot_r * KG + i) * FR + f) * 2) * 32 + lane];
            const uint4 ahi = ring[(((slot_r * KG + i) * FR + f) * 2 + 1) * 32 + lane];
            {
    #pragma unroll
              for (int nt = 0; nt < NP; ++nt) {
                if (nt < ntiles) {
                  mma_bf16_16816(acc[f][nt], alo.x, ahi.x, alo.y, ahi.y, bc[nt][i][0], bc[nt][i][1]);
                  mma_bf16_16816(acc[f][nt], alo.z, ahi.z, alo.w, ahi.w, bc[nt][i][2], bc[nt][i][3]);
                }
              }
            }
            }
          }
          slot_r = slot_r + 1 == NS ? 0 : slot_r + 1;
          issue_next();
    #pragma unroll
          for (int nt = 0; nt < NP; ++nt)
    #pragma unroll
            for (int i = 0; i < KG; ++i)
    #pragma unroll
              for (int j = 0; j < 4; ++j) bc[nt][i][j] = bn[nt][i][j];
        }
  
      }
      // epilogue straight from the fragments: c0,c1 = row g, tokens 2c,2c+1;
      // c2,c3 = row g+8, same tokens
      float gscale = 1.0f;
      if constexpr (kFp4) gscale = ct.down ? a.dn_global[ct.e] : a.gu_global[ct.e];
  #pragma unroll
      for (int fr = 0; fr < FR; ++fr)
  #pragma unroll
      for (int nt = 0; nt < NP; ++nt) {
        if (nt >= ntiles) continue;
  #pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int n = p0 + nt * 8 + 2 * c + h2;
          if (n < ct.m) {
            if (!ct.down) {
              const float gv = acc[fr][nt][h2] * gscale, uv = acc[fr][nt][2 + h2] * gscale;
              const float hv = silu(gv) * uv;
              uint16_t hb;
              if constexpr (C::kDec) {
                hb = f2h(hv);   // the down units' f16 operand
                if ((hb & 0x7c00u) == 0x7c00u) atomicOr(a.status, kStatusRange);
              } else {
                hb = f2bf(hv);
              }
              a.h[(size_t)(ct.off + n) * a.I + (ct.blk * FR + fr) * 8 + g] = hb;
            } else {
              const int f = ef[nt][h2];
              const float wt = ew[nt][h2];
              const float y0 = wt * (acc[fr][nt][h2] * gscale), y1 = wt * (acc[fr][nt][2 + h2] * gscale);
              const size_t o = (size_t)f * a.H + (ct.blk * FR + fr) * 16 + g;
              if (a.partial_f32) {
                reinterpret_cast<float*>(a.partial)[o] = y0;
                reinterpret_cast<float*>(a.partial)[o + 8] = y1;
              } else {
                reinterpret_cast<uint16_t*>(a.partial)[o] = f2bf(y0);
                reinterpret_cast<uint16_t*>(a.partial)[o + 8] = f2bf(y1);
              }
            }
          }
        }
      }
    };
    // bf16 and int8 passes run with a compile-time number of token tiles
    // equal to the tiles that hold rows, so no mma sits behind a per-tile
    // branch (measured: int8_256 stream stage 336 -> 319 us); NVFP4 is
    // faster with one copy of its decode loop (205 us against 224 us with
    // per-count copies and 223 us with NT tiles always)
    const int tiles = min(NT, (ct.m - p0 + 7) / 8);
    if constexpr (NT == 1 || kFp4) {
      run_pass(std::integral_constant<int, NT>{});
    } else if constexpr (NT == 2) {
      if (tiles == 2) run_pass(std::integral_constant<int, 2>{});
      else run_pass(std::integral_constant<int, 1>{});
    } else {
      static_assert(NT == 4, "token tiles per pass: 1, 2 or 4");
      if (tiles == 4) run_pass(std::integral_constant<int, 4>{});
      else if (tiles == 3) run_pass(std::integral_constant<int, 3>{});
      else if (tiles == 2) run_pass(std::integral_constant<int, 2>{});
      else run_pass(std::integral_constant<int, 1>{});
    }
    if (++ct.pass < ct.npass) continue;
    if (!ct.down) {
      // publish this unit's h rows to the down units of the expert
      __syncwarp();
      if (lane == 0) red_release_add(a.dep + ct.slot, 1);
    }
    pop();
  }
  cp_async_wait<0>();
  if (a.fused_combine) {
    // every group was on this launch: once all CTAs' partials are written,
    // the combine runs here (the ring's first word carries the verdict)
    __syncthreads();
    int* flag = reinterpret_cast<int*>(smem);
    if (threadIdx.x == 0) *flag = grid_sync(a.done, (int)gridDim.x, a.status) ? 1 : 0;
    __syncthreads();
    if (*flag) combine_slice(a, (long long)blockIdx.x * blockDim.x + threadIdx.x, (long long)gridDim.x * blockDim.x);
  }
}

template <int F, int NT>
cudaError_t launch_variant(const StreamGemmArgs& a, cudaStream_t stream) {
  using C = StreamCfg<F, NT>;
  const long long S = (long long)a.T * a.k;
  const long long max_active = S < a.E ? S : a.E;
  const long long units = max_active * (a.I / (8 * C::FR) + a.H / (16 * C::FR));
  long long grid = a.num_sms;
  const long long need = (units + C::kWarps - 1) / C::kWarps;
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  // [rings][smeta E][sperm S]
  const int smem = C::kWarpBytes * C::kWarps + C::kLutBytes + 16 * a.E +
                   (S <= kPermSmem ? 4 * (int)S : 0);
  cudaError_t err = cudaFuncSetAttribute(stream_gemm_kernel<F, NT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(C::kWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, stream_gemm_kernel<F, NT>, a);
}

}  // namespace

cudaError_t launch_stream_gemm(const StreamGemmArgs& args, cudaStream_t stream, int* launches) {
  if (launches) *launches += 1;
  StreamGemmArgs a = args;
  const DebugWaits dw = debug_waits();
  a.spin_limit = dw.spin_limit > 0 ? dw.spin_limit : kSpinLimit;
  a.wait_extra = dw.force ? 1 : 0;
  // a group never holds more rows than the batch has tokens: one 8-row tile
  // per pass for T <= 8, two above; NVFP4 takes four (32-row passes) once
  // the experts average 24 rows or more (measured: 16-row passes faster at
  // 16 rows per expert, 32-row passes at 32 and 64)
  // NVFP4 and int8 weights with 256-multiple H and I: the TMA-fed kernel
  if (stream_dec_supported(a)) return launch_stream_dec(a, stream);
  const bool two = a.T > 8;
  const long long S = (long long)a.T * a.k;
  const long long avg = S / (S < a.E ? S : a.E);
  const bool four = a.T > 16 && avg >= 24;
  if (a.gu_codes != nullptr) {
    if (four) return launch_variant<kFmtFp4, 4>(a, stream);
    return two ? launch_variant<kFmtFp4, 2>(a, stream) : launch_variant<kFmtFp4, 1>(a, stream);
  }
  if (a.gu_q8 != nullptr) {
    if (four) return launch_variant<kFmtQ8, 4>(a, stream);
    return two ? launch_variant<kFmtQ8, 2>(a, stream) : launch_variant<kFmtQ8, 1>(a, stream);
  }
  return two ? launch_variant<kFmtBf16, 2>(a, stream) : launch_variant<kFmtBf16, 1>(a, stream);
}

}  // namespace moe
