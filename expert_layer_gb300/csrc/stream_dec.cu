// Weight-streaming expert kernel for the decoded weight formats (NVFP4 and
// int8 blocks), warp-specialised.
//
// The same work units, queue and arithmetic as the streaming kernel of
// stream_gemm.cu (the "expert kernel" and "activation" phases of the fused
// MoE path, page "Decode 吞吐专项实验分析报告", section "下一步 profiling 方向",
// item 3; the NVFP4 weights of page "vLLM 0.32 升级试验：TEP2 prefill 诅咒解除
// + decode 本机纪录", "背景与动机"): a unit is FR fragments of 16 weight rows of
// one expert over all of K, owned by one warp, decoded to f16 in registers
// and multiplied on mma.sync m16n8k16 against up to 8*NT token rows per pass.
// What differs is who moves the weights.  Here one producer warp per CTA
// streams every consumer warp's codes and block scales with TMA tile loads
// into that warp's ring of shared-memory stages (mbarrier full / empty
// pairs), so the consumer warps issue only the decode, the mma, the token-row
// loads and the epilogue -- no per-row copy instructions, address arithmetic
// or unit bookkeeping for the copies.  Lane w of the producer warp serves
// consumer warp w: it draws the warp's units from the queue, hands each unit
// id to the warp through a small shared-memory FIFO, and keeps up to NS
// stages of the warp's weights in flight across unit boundaries.
//
// Stage = one K block of a unit: all of its weight rows' codes (64 bytes per
// row: 128 NVFP4 or 64 int8 elements) and a 16-byte window of each row's
// block scales that holds this block's (8 e4m3 bytes for NVFP4, two fp16
// for int8).  Gate/up units load gate rows j0..j0+8FR-1 and the matching up
// rows with one 4-D box (w_gate_up viewed as [E][2][I][bytes]); down units
// 16FR consecutive rows of w_down.  In shared memory a stage is rows of 64
// code bytes (no swizzle: the 16-byte reads of 8 lanes cover 128 contiguous
// bytes) followed by rows of 16 scale bytes.
//
// Requires H and I to be multiples of 256 (the scale rows, K/16 bytes, are
// then whole 16-byte TMA strides); other shapes take stream_gemm.cu.
#include <cuda.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "nvfp4.cuh"
#include "stream_common.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace stream;

template <int F, int NT>
struct DecCfg {
  static constexpr bool kFp4 = F == kFmtFp4;
  static constexpr int FR = NT >= 4 ? 2 : 4;      // 16-row fragments per unit
  static constexpr int ROWS = 16 * FR;            // weight rows per unit
  static constexpr int SBK = kFp4 ? 8 : 4;        // scale bytes per row and block
  static constexpr int kCodeBytes = ROWS * 64;
  static constexpr int kScaleBytes = ROWS * 16;
  static constexpr int kStageBytes = kCodeBytes + kScaleBytes;
  // consumer warps, and stages per consumer ring: with the producer warp
  // three warps per SM sub-partition (168 registers each) for one or two
  // token tiles per pass; two (255 registers) for three or four tiles, which
  // spill at 168.  Measured at nvfp4_256 / int8_256 (16 rows per expert on
  // average): two tiles with 11 consumers and 3 stages 153 / 205 us, with 7
  // consumers and 4 stages 160 / 219 us; three tiles (24-row passes, so that
  // 97% of the experts decode their weights once) with 7 consumers 146 /
  // 189 us.
  static constexpr int NW = NT >= 3 ? 7 : 11;
  static constexpr int NS = FR == 4 ? 3 : 8;
  static constexpr int kThreads = (NW + 1) * 32;
  static constexpr int kRingBytes = NS * kStageBytes;
  static constexpr int kFifo = 16;                // unit ids the producer may hold ahead
};

struct DecMaps {
  CUtensorMap gu_codes, dn_codes, gu_scales, dn_scales;
};

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4, %5}], [%6];" ::"r"(tcx::smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(tcx::smem_u32(bar))
      : "memory");
}

// mma.sync m16n8k16 (f16 x f16 -> fp32) executed only when `on`: a
// predicated instruction instead of a branch around it.  `on` must be the
// same in every lane (the token-tile count of the pass is warp-uniform).
__device__ __forceinline__ void mma_f16_if(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1, bool on) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %10, 0;\n"
      " @p mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n}\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"((int)on));
}

// Four e2m1 codes of a 32-bit word -- bytes 0-1 (hi = false) or bytes 2-3
// (hi = true), low nibble to the low half -- to two f16x2, exact.
template <bool hi>
__device__ __forceinline__ void e2m1x4_f16x2_sel(uint32_t v, uint32_t& d0, uint32_t& d1) {
  if constexpr (hi)
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %2;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b2;\n cvt.rn.f16x2.e2m1x2 %1, b3;\n}"
        : "=r"(d0), "=r"(d1)
        : "r"(v));
  else
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %2;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n}"
        : "=r"(d0), "=r"(d1)
        : "r"(v));
}

// a * {s.lo, s.lo} and a * {s.hi, s.hi} (f16x2), each product exact here
__device__ __forceinline__ uint32_t mul_lo(uint32_t a, uint32_t s) {
  uint32_t d;
  asm("{\n .reg .b16 l, h;\n .reg .b32 t;\n mov.b32 {l, h}, %2;\n mov.b32 t, {l, l};\n"
      " mul.rn.f16x2 %0, %1, t;\n}"
      : "=r"(d)
      : "r"(a), "r"(s));
  return d;
}
__device__ __forceinline__ uint32_t mul_hi(uint32_t a, uint32_t s) {
  uint32_t d;
  asm("{\n .reg .b16 l, h;\n .reg .b32 t;\n mov.b32 {l, h}, %2;\n mov.b32 t, {h, h};\n"
      " mul.rn.f16x2 %0, %1, t;\n}"
      : "=r"(d)
      : "r"(a), "r"(s));
  return d;
}

// Bounded wait of one thread on an mbarrier phase: polls (with a short
// sleep after the first 32) until the phase completes or `limit` polls
// failed; false then.  The loop sits inside one asm block, so the compiler
// sees straight-line code (no divergent region to reconverge around the
// mma that follow).  The ring waits use the fixed kSpinLimit
// (StreamGemmArgs.spin_limit shortens only the down units' wait for their
// expert's h rows, as in the other streaming kernel).
__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity, int limit) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p, q;\n .reg .u32 n;\n mov.u32 n, 0;\n"
      "WAIT:\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n @p bra DONE;\n"
      " add.u32 n, n, 1;\n setp.ge.u32 q, n, %3;\n @q bra DONE;\n"
      " setp.gt.u32 q, n, 32;\n @q nanosleep.u32 32;\n bra WAIT;\n"
      "DONE:\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(tcx::smem_u32(bar)), "r"(parity), "r"((uint32_t)limit)
      : "memory");
  return ok != 0;
}

template <int F, int NT>
__global__ void __launch_bounds__(DecCfg<F, NT>::kThreads, 1)
    stream_dec_kernel(const __grid_constant__ DecMaps maps, const StreamGemmArgs a) {
  using C = DecCfg<F, NT>;
  constexpr bool kFp4 = C::kFp4;
  constexpr int FR = C::FR, NS = C::NS, NW = C::NW, kFifo = C::kFifo;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* rings = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NW * C::kRingBytes);   // [NW][NS]
  uint64_t* empty = full + NW * NS;                                           // [NW][NS]
  int* fifo = reinterpret_cast<int*>(empty + NW * NS);                        // [NW][kFifo]
  int4* smeta = reinterpret_cast<int4*>(fifo + NW * kFifo);                   // [E]
  int* sperm = reinterpret_cast<int*>(smeta + a.E);                           // [S]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NW * NS; ++i) {
      tcx::mbar_init(&full[i], 1);
      tcx::mbar_init(&empty[i], 32);   // every lane of the consumer warp arrives
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
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
    nsmall = *a.num_active - (a.num_large ? *a.num_large : 0);
    for (int i = threadIdx.x; i < nsmall; i += blockDim.x) {
      int e = a.active[i];
      if (!bounds_ok((unsigned)e < (unsigned)a.E, a.status)) e = 0;
      int m = a.counts[e], off = a.offsets[e];
      if (!bounds_ok(off >= 0 && m >= 0 && off + m <= S, a.status)) m = 0, off = 0;
      smeta[i] = make_int4(e, m, off, 0);
    }
    if (perm_smem)
      for (int i = threadIdx.x; i < S; i += blockDim.x) sperm[i] = a.perm[i];
    __syncthreads();
  }
  Queue qs;
  qs.UPEg = a.I / (8 * FR);
  qs.UPEd = a.H / (16 * FR);
  qs.Ug = nsmall * qs.UPEg;
  qs.Q = qs.Ug + nsmall * qs.UPEd;
  qs.nkb_g = a.H / (kFp4 ? 128 : 64);
  qs.nkb_d = a.I / (kFp4 ? 128 : 64);
  const int* permp = perm_smem ? sperm : a.perm;

  if (warp == NW) {
    // ------------------------------------------------------------ producer
    if (lane >= NW) return;
    const int cw = lane;                       // the consumer warp served
    uint64_t* fb = full + cw * NS;
    uint64_t* eb = empty + cw * NS;
    unsigned char* ring = rings + cw * C::kRingBytes;
    const int nwarps = (int)gridDim.x * NW;
    int first = (int)blockIdx.x * NW + cw;
    int pw = 0, slot = 0, issued = 0;
    uint32_t round = 0;
    bool ok = true;
    // a ring slot is free once its consumer released the previous round's
    // stage (the first round's wait on parity 1 passes at once)
    auto slot_free = [&]() -> bool { return bar_wait(&eb[slot], (round & 1) ^ 1, kSpinLimit); };
    auto advance = [&]() {
      ++issued;
      if (++slot == NS) { slot = 0; ++round; }
    };
    Task pt;
    while (ok) {
      int q;
      if (first >= 0) { q = first; first = -1; }
      else q = nwarps + atomicAdd(a.queue, 1);
      task_load<1, NT>(pt, smeta, qs, q);
      if (!slot_free()) { ok = false; break; }
      // the consumer reads the unit id after its first stage's full barrier
      // completes, which the arrive below (release) precedes
      fifo[cw * kFifo + (pw++ % kFifo)] = pt.q;
      if (pt.q < 0) {             // no more units: a stage without data ends the warp
        tcx::mbar_arrive(&fb[slot]);
        advance();
        break;
      }
      const int e = pt.e;
      for (int p = 0; p < pt.npass && ok; ++p) {
        for (int kb = 0; kb < pt.nkb; ++kb) {
          if ((p | kb) != 0 && !slot_free()) { ok = false; break; }
          unsigned char* st = ring + slot * C::kStageBytes;
          tcx::mbar_expect_tx(&fb[slot], C::kStageBytes);
          const int sx = (kb * C::SBK) & ~15;
          if (pt.down) {
            const int row = e * a.H + pt.blk * C::ROWS;
            tcx::tma_load_2d(st, &maps.dn_codes, kb * 64, row, &fb[slot]);
            tcx::tma_load_2d(st + C::kCodeBytes, &maps.dn_scales, sx, row, &fb[slot]);
          } else {
            const int j0 = pt.blk * 8 * FR;
            tma_load_4d(st, &maps.gu_codes, kb * 64, j0, 0, e, &fb[slot]);
            tma_load_4d(st + C::kCodeBytes, &maps.gu_scales, sx, j0, 0, e, &fb[slot]);
          }
          advance();
        }
      }
    }
    if (!ok) atomicOr(a.status, kStatusTimeout);
    // every issued stage's copies have landed before the CTA may exit
    for (int i = issued > NS ? issued - NS : 0; i < issued; ++i)
      if (!bar_wait(&fb[i % NS], (uint32_t)(i / NS) & 1, kSpinLimit)) atomicOr(a.status, kStatusTimeout);
    return;
  }

  // -------------------------------------------------------------- consumer
  uint64_t* fb = full + warp * NS;
  uint64_t* eb = empty + warp * NS;
  const unsigned char* ring = rings + warp * C::kRingBytes;
  int slot = 0, pr = 0;
  uint32_t round = 0;
  bool dead = false;
  // every lane waits itself (each gets the acquire of the TMA's writes)
  auto stage_ready = [&]() -> bool {
    const bool ok = bar_wait(&fb[slot], round & 1, kSpinLimit);
    return __all_sync(0xffffffffu, ok);
  };
  // each lane arrives after its own reads of the stage (release): no branch
  auto release = [&]() {
    tcx::mbar_arrive(&eb[slot]);
    if (++slot == NS) { slot = 0; ++round; }
  };
  Task ct;
  while (!dead) {
    if (!stage_ready()) { dead = true; break; }
    task_load<1, NT>(ct, smeta, qs, fifo[warp * kFifo + (pr++ % kFifo)]);
    if (ct.q < 0) break;
    if (ct.down) {
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
    // rows of fragment f in a stage: gate/up g and up rows 8FR + f*8 + g;
    // down 16f + g and 16f + 8 + g
    const int rlo0 = g, rhi0 = ct.down ? 8 + g : 8 * FR + g, fstep = ct.down ? 16 : 8;
    for (ct.pass = 0; ct.pass < ct.npass && !dead; ++ct.pass) {
      const int p0 = ct.pass * 8 * NT;
      const int ntiles = min(NT, (ct.m - p0 + 7) / 8);
      constexpr int NP = NT;
      const uint16_t* bsrc[NP];
#pragma unroll
      for (int nt = 0; nt < NP; ++nt) {
        const int n = p0 + nt * 8 + g;
        bsrc[nt] = nullptr;
        if (n < ct.m) {
          if (ct.down) bsrc[nt] = a.h + (size_t)(ct.off + n) * a.I;
          else {
            int f = permp[ct.off + n];
            if (!bounds_ok((unsigned)f < (unsigned)S, a.status)) f = 0;
            bsrc[nt] = a.x16 + (size_t)(f / a.k) * a.H;
          }
        }
      }
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
            if (!bounds_ok((unsigned)ef[nt][h2] < (unsigned)S, a.status)) ef[nt][h2] = 0;
            ew[nt][h2] = a.topk_w[ef[nt][h2]];
          }
        }
      float acc[FR][NP][4];
#pragma unroll
      for (int f = 0; f < FR; ++f)
#pragma unroll
        for (int nt = 0; nt < NP; ++nt) acc[f][nt][0] = acc[f][nt][1] = acc[f][nt][2] = acc[f][nt][3] = 0.f;

      if constexpr (kFp4) {
        // token rows double-buffered in half blocks (64 K elements: the
        // four mma steps that share one scale byte of each row)
        uint32_t bh[2][NP][8];
        auto load_half = [&](uint32_t (&b)[NP][8], int kb, int hf) {
#pragma unroll
          for (int nt = 0; nt < NP; ++nt)
#pragma unroll
            for (int v = 0; v < 2; ++v) {
              uint4 t = make_uint4(0, 0, 0, 0);
              if (nt < ntiles && bsrc[nt] && kb < ct.nkb) {
                const uint4* pp =
                    reinterpret_cast<const uint4*>(bsrc[nt] + (size_t)kb * 128 + 32 * c + 8 * (2 * hf + v));
                t = ct.down ? __ldcg(pp) : *pp;
              }
              b[nt][4 * v + 0] = t.x; b[nt][4 * v + 1] = t.y; b[nt][4 * v + 2] = t.z; b[nt][4 * v + 3] = t.w;
            }
        };
        load_half(bh[0], 0, 0);
#pragma unroll 1
        for (int kb = 0; kb < ct.nkb; ++kb) {
          load_half(bh[1], kb, 1);
          if ((ct.pass | kb) != 0 && !stage_ready()) { dead = true; break; }
          const unsigned char* st = ring + slot * C::kStageBytes;
          const unsigned char* sc = st + C::kCodeBytes + ((kb * C::SBK) & 15);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            if (hf == 1) load_half(bh[0], kb + 1, 0);
            // s2[f]: the f16 scales of rows g (low half) and g+8 (high half)
            // for this thread's 16-element block 2c + hf
            uint32_t s2[FR], clo[FR][2], chi[FR][2];
#pragma unroll
            for (int f = 0; f < FR; ++f) {
              const int rlo = rlo0 + f * fstep, rhi = rhi0 + f * fstep;
              // 16 bytes per row (both halves; 8 lanes read 128 contiguous
              // bytes, no bank conflict), this half's 8 used
              const uint4 a4 = *reinterpret_cast<const uint4*>(st + rlo * 64 + 16 * c);
              const uint4 b4 = *reinterpret_cast<const uint4*>(st + rhi * 64 + 16 * c);
              const uint32_t sa = *reinterpret_cast<const uint16_t*>(sc + rlo * 16 + 2 * c);
              const uint32_t sb = *reinterpret_cast<const uint16_t*>(sc + rhi * 16 + 2 * c);
              s2[f] = nvfp4::e4m3x2_f16x2(__byte_perm(sa, sb, hf ? 0x0051 : 0x0040));
              clo[f][0] = hf ? a4.z : a4.x; clo[f][1] = hf ? a4.w : a4.y;
              chi[f][0] = hf ? b4.z : b4.x; chi[f][1] = hf ? b4.w : b4.y;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
#pragma unroll
              for (int f = 0; f < FR; ++f) {
                uint32_t l0, l1, h0, h1;
                if (q & 1) {
                  e2m1x4_f16x2_sel<true>(clo[f][q >> 1], l0, l1);
                  e2m1x4_f16x2_sel<true>(chi[f][q >> 1], h0, h1);
                } else {
                  e2m1x4_f16x2_sel<false>(clo[f][q >> 1], l0, l1);
                  e2m1x4_f16x2_sel<false>(chi[f][q >> 1], h0, h1);
                }
                const uint32_t a0 = mul_lo(l0, s2[f]);
                const uint32_t a2 = mul_lo(l1, s2[f]);
                const uint32_t a1 = mul_hi(h0, s2[f]);
                const uint32_t a3 = mul_hi(h1, s2[f]);
#pragma unroll
                for (int nt = 0; nt < NP; ++nt)
                  mma_f16_if(acc[f][nt], a0, a1, a2, a3, bh[hf][nt][2 * q], bh[hf][nt][2 * q + 1], nt < ntiles);
              }
            }
          }
          release();
        }
      } else {
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
        load_half(bh[0], 0, 0);
#pragma unroll 1
        for (int kb = 0; kb < ct.nkb; ++kb) {
          load_half(bh[1], kb, 1);
          if ((ct.pass | kb) != 0 && !stage_ready()) { dead = true; break; }
          const unsigned char* st = ring + slot * C::kStageBytes;
          const unsigned char* sc = st + C::kCodeBytes + ((kb * C::SBK) & 15);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            if (hf == 1) load_half(bh[0], kb + 1, 0);
            // the mma sums code x activation of one scale block (exact
            // products, fp32 sums), then the scale multiplies the partial
            uint32_t clo[FR][2], chi[FR][2];
            float slo[FR], shi[FR];
#pragma unroll
            for (int f = 0; f < FR; ++f) {
              const int rlo = rlo0 + f * fstep, rhi = rhi0 + f * fstep;
              const uint2 alo = *reinterpret_cast<const uint2*>(st + rlo * 64 + 32 * hf + 8 * c);
              const uint2 ahi = *reinterpret_cast<const uint2*>(st + rhi * 64 + 32 * hf + 8 * c);
              slo[f] = q8::f16_half_to_f32(*reinterpret_cast<const uint32_t*>(sc + rlo * 16), hf);
              shi[f] = q8::f16_half_to_f32(*reinterpret_cast<const uint32_t*>(sc + rhi * 16), hf);
              clo[f][0] = alo.x; clo[f][1] = alo.y;
              chi[f][0] = ahi.x; chi[f][1] = ahi.y;
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
                  mma_f16_if(part[f][nt], a0, a1, a2, a3, bh[hf][nt][2 * q], bh[hf][nt][2 * q + 1], nt < ntiles);
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
          release();
        }
      }
      if (dead) break;
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
            if (n >= ct.m) continue;
            if (!ct.down) {
              const float gv = acc[fr][nt][h2] * gscale, uv = acc[fr][nt][2 + h2] * gscale;
              const uint16_t hb = f2h(silu(gv) * uv);   // the down units' f16 operand
              if ((hb & 0x7c00u) == 0x7c00u) atomicOr(a.status, kStatusRange);
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
    if (dead) break;
    if (!ct.down) {
      // publish this unit's h rows to the down units of the expert
      __syncwarp();
      if (lane == 0) red_release_add(a.dep + ct.slot, 1);
    }
  }
  if (dead) atomicOr(a.status, kStatusTimeout);
  if (a.fused_combine) {
    // every group was on this launch: once all CTAs' partials are written,
    // the consumer warps combine (named barrier 1 over the consumers; the
    // producer warp may have left; the ring's first word, idle now, carries
    // the verdict)
    asm volatile("bar.sync 1, %0;" ::"r"(NW * 32) : "memory");
    int* flag = reinterpret_cast<int*>(smem);
    if (threadIdx.x == 0) *flag = grid_sync(a.done, (int)gridDim.x, a.status) ? 1 : 0;
    asm volatile("bar.sync 1, %0;" ::"r"(NW * 32) : "memory");
    if (*flag) combine_slice(a, (long long)blockIdx.x * (NW * 32) + threadIdx.x, (long long)gridDim.x * (NW * 32));
  }
}

// Byte tensor map (uint8, no swizzle) of the given rank; strides in bytes
// for dimensions 1..rank-1.
bool make_byte_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                   const uint32_t* box) {
  tcx::EncodeTiledFn fn = tcx::encode_fn();
  if (!fn) return false;
  cuuint64_t d[4], s[3];
  cuuint32_t b[4], es[4];
  for (int i = 0; i < rank; ++i) { d[i] = dims[i]; b[i] = box[i]; es[i] = 1; }
  for (int i = 0; i + 1 < rank; ++i) s[i] = strides[i];
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void*>(base), d, s, b, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int F, int NT>
cudaError_t launch_dec(const StreamGemmArgs& a, cudaStream_t stream) {
  using C = DecCfg<F, NT>;
  const uint64_t E = a.E, H = a.H, I = a.I;
  // code bytes per row: K/2 (NVFP4) or K (int8); scale bytes per row: K/16
  const uint64_t cb_g = C::kFp4 ? H / 2 : H, cb_d = C::kFp4 ? I / 2 : I;
  const void* gc = C::kFp4 ? (const void*)a.gu_codes : (const void*)a.gu_q8;
  const void* dc = C::kFp4 ? (const void*)a.dn_codes : (const void*)a.dn_q8;
  const void* gs = C::kFp4 ? (const void*)a.gu_scales : (const void*)a.gu_q8s;
  const void* ds = C::kFp4 ? (const void*)a.dn_scales : (const void*)a.dn_q8s;
  DecMaps maps;
  {
    // w_gate_up as [E][2][I][bytes]: a box is 8FR gate rows and the same up rows
    const uint64_t dims[4] = {cb_g, I, 2, E}, str[3] = {cb_g, I * cb_g, 2 * I * cb_g};
    const uint32_t box[4] = {64, (uint32_t)(8 * C::FR), 2, 1};
    if (!make_byte_map(&maps.gu_codes, gc, 4, dims, str, box)) return cudaErrorInvalidValue;
    const uint64_t sdims[4] = {H / 16, I, 2, E}, sstr[3] = {H / 16, I * H / 16, 2 * I * H / 16};
    const uint32_t sbox[4] = {16, (uint32_t)(8 * C::FR), 2, 1};
    if (!make_byte_map(&maps.gu_scales, gs, 4, sdims, sstr, sbox)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {cb_d, E * H}, str[1] = {cb_d};
    const uint32_t box[2] = {64, (uint32_t)C::ROWS};
    if (!make_byte_map(&maps.dn_codes, dc, 2, dims, str, box)) return cudaErrorInvalidValue;
    const uint64_t sdims[2] = {I / 16, E * H}, sstr[1] = {I / 16};
    const uint32_t sbox[2] = {16, (uint32_t)C::ROWS};
    if (!make_byte_map(&maps.dn_scales, ds, 2, sdims, sstr, sbox)) return cudaErrorInvalidValue;
  }
  const long long S = (long long)a.T * a.k;
  const long long max_active = S < a.E ? S : a.E;
  const long long units = max_active * (a.I / (8 * C::FR) + a.H / (16 * C::FR));
  long long grid = a.num_sms;
  const long long need = (units + C::NW - 1) / C::NW;
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  // [rings][barriers][fifo][smeta E][sperm S]
  const int smem = C::NW * C::kRingBytes + 2 * C::NW * C::NS * 8 + C::NW * C::kFifo * 4 + 16 * a.E +
                   (S <= kPermSmem ? 4 * (int)S : 0);
  cudaError_t err =
      cudaFuncSetAttribute(stream_dec_kernel<F, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, stream_dec_kernel<F, NT>, maps, a);
}

}  // namespace

bool stream_dec_supported(const StreamGemmArgs& a) {
  return (a.gu_codes != nullptr || a.gu_q8 != nullptr) && a.H % 256 == 0 && a.I % 256 == 0;
}

cudaError_t launch_stream_dec(const StreamGemmArgs& a, cudaStream_t stream) {
  const bool two = a.T > 8;
  const long long S = (long long)a.T * a.k;
  const long long avg = S / (S < a.E ? S : a.E);
  // token tiles per pass: 32-row passes once the experts average 24 rows,
  // 24-row passes from 12, else 16 (T > 8) or 8
  const bool four = a.T > 16 && avg >= 24;
  const bool three = a.T > 16 && avg >= 12 && !four;
  if (a.gu_codes != nullptr) {
    if (four) return launch_dec<kFmtFp4, 4>(a, stream);
    if (three) return launch_dec<kFmtFp4, 3>(a, stream);
    return two ? launch_dec<kFmtFp4, 2>(a, stream) : launch_dec<kFmtFp4, 1>(a, stream);
  }
  if (four) return launch_dec<kFmtQ8, 4>(a, stream);
  if (three) return launch_dec<kFmtQ8, 3>(a, stream);
  return two ? launch_dec<kFmtQ8, 2>(a, stream) : launch_dec<kFmtQ8, 1>(a, stream);
}

}  // namespace moe
