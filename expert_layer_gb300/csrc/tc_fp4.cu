// W4A4 expert GEMMs: NVFP4 weights times NVFP4 activations on the block-scaled
// tensor cores (tcgen05.mma kind::mxf4nvf4, e2m1 x e2m1 with one ue4m3 scale
// per 16 elements along K, fp32 accumulate in tensor memory).
//
// The NVFP4 deployment on the pages is the 176B MoE served through the
// "nvfp4-sm80" graft (page "vLLM 0.32 升级试验：TEP2 prefill 诅咒解除 + decode
// 本机纪录", header and "背景与动机"); its sm_80 kernels have no FP4 tensor
// cores.  Here the activations are quantised on the fly with the format's
// own recipe, per routed row of expert e: 16-element blocks along K, block
// scale s = e4m3_rn_satfinite(amax / (6 G)), element code
// e2m1_rn_satfinite(v * r) with r = 1 / (s G) once per block, G = x_global[e]
// for the token rows and G = h_global[e] for the SwiGLU output (each
// quotient, reciprocal and product in fp32, IEEE round to nearest).
//
// Pipeline of one W4A4 layer (after routing and grouping):
//   quant x      token rows in grouped order -> e2m1 codes [S, H/2] and block
//                scales in the tensor-core layout (below)
//   gate/up      acc = sum_k A*B with A = weight codes (128 interleaved
//                gate/up rows, as the bf16 kernels) and B = 128 token rows;
//                h = bf16(silu(g') * u'), g' = acc_g * gu_global[e] * x_global[e]
//   quant h      h rows -> codes [S, I/2] and scales
//   down         partial[f, d] = topk_w[f] * acc * dn_global[e] * h_global[e]
//
// Tensor-core scale layout.  For a block of 128 rows and one MMA K step of 64
// elements (4 scales per row) the scales form one 512-byte atom of 32 rows x
// 16 bytes: atom row i, bytes 4j..4j+3 = the 4 scales (k-block order) of row
// i + 32j.  tcgen05.cp.32x128b.warpx4 copies an atom into tensor memory,
// replicated into all four lane quadrants, where the MMA reads the scales of
// A row m at (lane m, column base + m/32) and those of B column n, for the
// accumulator lanes of quadrant q, at (lane 32q + n%32, column base + n/32).
// Atoms are stored by (row block, K step): byte offset
//   ((block * (K/64) + K/64 step) * 512) + (row%32)*16 + ((row%128)/32)*4 + (k-block%4).
// Weight scales are rearranged into this layout once by moe_nvfp4_tc_scales
// (gate/up rows in the kernels' interleaved order); activation scales are
// written in it by the quantiser, with blocks of 128 rows of one expert
// (block = the expert's first block + row within the expert / 128).
//
// GEMM kernel: one persistent CTA per SM, 14 warps:
//   warp 0      one thread issues the TMA loads (codes: tiled, 128-byte
//               swizzle) and bulk copies (scale atoms) of a 5-stage ring
//   warp 1      allocates tensor memory; one thread issues four MMAs per
//               256-wide K stage (M = 128 weight rows, N = the tile's token
//               rows rounded up to 16, K = 64 each)
//   warps 2-5   scale warps, one per TMEM lane quadrant: they read a stage's
//               scale atoms from shared memory and write them into tensor
//               memory with tcgen05.st, then signal the MMA thread.  (A
//               tcgen05.cp of an atom costs ~53 cycles of the same pipe as
//               the MMAs, ~65 cycles for a 128 x 128 x 64 FP4 MMA: copying
//               the eight atoms of a stage that way took more pipe time than
//               its four MMAs.)  The MMA reads A row m's scales of K step kk
//               at (lane m, column sa + 4kk + m/32) and B column n's at
//               (lane 32q + n%32, column sb + 4kk + n/32) for the
//               accumulator lanes of quadrant q, so quadrant q writes, in its
//               own lanes, A's scales at columns sa + 4kk + q (zeros in the
//               other columns of the 16, which only other quadrants read in
//               their own lanes) and the full 16 columns of B's.
//   warps 6-13  epilogue: two warps per TMEM lane quadrant, alternate
//               32-column chunks
// Two 128-column accumulators let the epilogue of one tile overlap the
// mainloop of the next.  Every mbarrier wait is bounded; a timeout sets
// kStatusTimeout, the CTA leaves its loops, waits (bounded again) for the
// copies and MMAs it has issued, frees its tensor memory and returns.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace tcx;

constexpr int kRows = 128;                          // weight rows (M), token rows (N max) per tile
constexpr int kKStage = 256;                        // K elements per stage (128 code bytes per row)
constexpr int kCodeBytes = kRows * kKStage / 2;     // 16 KB per operand per stage
constexpr int kAtomBytes = 512;                     // scales of 128 rows x one 64-wide K step
constexpr int kSfBytes = 4 * kAtomBytes;            // per operand per stage
constexpr int kStage = 2 * kCodeBytes + 2 * kSfBytes;   // 36 KB
constexpr int NSF = 5;
constexpr int kSfWarps = 4;
constexpr int kEpiWarps = 8;
constexpr int kThreads = (2 + kSfWarps + kEpiWarps) * 32;
constexpr uint32_t kAccCols = 128;
constexpr uint32_t kSfColBase = 2 * kAccCols;       // scale columns after the two accumulators
constexpr uint32_t kSfColsStage = 32;               // SFA 16 + SFB 16 per stage
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxE = 1024;
// ring + alignment slack + barriers + per-expert metadata (e, m, off, tile prefix)
constexpr size_t kSmemBytes = (size_t)NSF * kStage + 1024 + 256 + 4 * 4 * (kMaxE + 1);

static_assert(NSF * kSfColsStage + kSfColBase <= kTmemCols, "tensor memory columns");

struct Fp4Args {
  int T, H, E, I, k;
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* perm;
  const int32_t* active;
  const int* num_active;
  const uint8_t* sfa;        // weight scales, tensor-core layout
  const uint8_t* sfb;        // activation scales, tensor-core layout
  const float* w_global;     // [E] weight global of this projection
  const float* a_global;     // [E] activation global of this projection
  const float* topk_w;       // [S]
  uint16_t* h;               // [S, I] bf16 (gate/up output)
  void* partial;             // [S, H] (down output)
  int partial_f32;
  int* status;
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void mma_fp4(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t sfa, uint32_t sfb, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n}\n" ::"r"(
          tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum), "r"(sfa), "r"(sfb));
}
// Instruction descriptor of kind::mxf4nvf4: A and B e2m1 (format 1), ue4m3
// scales (bit 23 = 0), fp32 accumulate, both K-major, N >> 3 at bit 17,
// M >> 4 at bit 24, scale-factor ids 0.
__device__ __forceinline__ uint32_t idesc_fp4(int m, int n) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// ------------------------------------------------------------------ quantiser
// e4m3 byte of an fp32 value, round to nearest even, saturating at 448
__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xffu;
}
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  uint32_t d;
  asm("{\n .reg .b16 h;\n mov.b32 {h, _}, %1;\n cvt.rn.f16x2.e4m3x2 %0, h;\n}" : "=r"(d) : "r"(b));
  return __half2float(__ushort_as_half((unsigned short)(d & 0xffffu)));
}
// (lo * r, hi * r) as one packed fp32x2 multiply: each product rounded to
// nearest even exactly as a separate fp32 multiply would be
__device__ __forceinline__ void mul2_rn(float lo, float hi, float r, float& plo, float& phi) {
  unsigned long long x, y, z;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(lo), "f"(hi));
  asm("mov.b64 %0, {%1, %1};" : "=l"(y) : "f"(r));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(z) : "l"(x), "l"(y));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(plo), "=f"(phi) : "l"(z));
}
// two e2m1 codes: lo -> low nibble, hi -> high nibble; round to nearest even,
// saturating at 6
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n mov.b16 %0, {t, 0};\n}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r & 0xffu;
}

// Byte offset of scale (row, k-block) in the tensor-core layout of a
// [rows, K/16] scale matrix whose 128-row blocks start at block index `blk`.
__device__ __forceinline__ size_t tc_scale_offset(size_t blk, int row, int kb, int K) {
  return (blk * (size_t)(K / 64) + (size_t)(kb >> 2)) * kAtomBytes + (size_t)(row & 31) * 16 +
         (size_t)((row & 127) >> 5) * 4 + (size_t)(kb & 3);
}

// One row of K values (bf16 bits) to NVFP4 with global g: one warp; lane l
// takes the 16-element blocks l, l + 32, ..., loading up to four of them
// before converting any (the rows come from L2: several requests in flight
// per lane).  Codes are written to codes[0 .. K/2); the scale bytes of 4
// consecutive blocks (one 64-wide K step) are gathered in lane 4w and
// written as one 32-bit word by put_word(step, word).
template <typename PutWord>
__device__ __forceinline__ bool quantize_row(const uint16_t* __restrict__ src, int K, float g,
                                             uint8_t* __restrict__ codes, PutWord put_word) {
  const int lane = threadIdx.x & 31;
  const float g6 = __fmul_rn(6.0f, g);
  const int nb = K / 16;
  bool bad = false;
  for (int kb0 = 0; kb0 < nb; kb0 += 128) {
    uint4 p[4][2];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int kb = kb0 + 32 * u + lane;
      p[u][0] = p[u][1] = make_uint4(0, 0, 0, 0);
      if (kb < nb) {
        p[u][0] = *reinterpret_cast<const uint4*>(src + (size_t)kb * 16);
        p[u][1] = *reinterpret_cast<const uint4*>(src + (size_t)kb * 16 + 8);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int kb = kb0 + 32 * u + lane;
      uint32_t sbyte = 0;
      if (kb < nb) {
        const uint32_t w[8] = {p[u][0].x, p[u][0].y, p[u][0].z, p[u][0].w,
                               p[u][1].x, p[u][1].y, p[u][1].z, p[u][1].w};
        float v[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) { v[2 * i] = bf16lo(w[i]); v[2 * i + 1] = bf16hi(w[i]); }
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
        bad |= !(amax <= 3.0e38f);
        sbyte = f32_to_e4m3(__fdiv_rn(amax, g6));
        const float den = __fmul_rn(e4m3_to_f32(sbyte), g);
        uint32_t c[2] = {0u, 0u};
        if (den > 0.f) {
          const float r = __frcp_rn(den);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float plo, phi;
            mul2_rn(v[2 * i], v[2 * i + 1], r, plo, phi);
            c[i >> 2] |= f32x2_to_e2m1x2(plo, phi) << (8 * (i & 3));
          }
        }
        *reinterpret_cast<uint2*>(codes + (size_t)kb * 8) = make_uint2(c[0], c[1]);
      }
      // lanes 4w .. 4w+3 hold the scales of one 64-wide K step
      const uint32_t b1 = __shfl_down_sync(0xffffffffu, sbyte, 1);
      const uint32_t b2 = __shfl_down_sync(0xffffffffu, sbyte, 2);
      const uint32_t b3 = __shfl_down_sync(0xffffffffu, sbyte, 3);
      if ((lane & 3) == 0 && kb < nb) put_word(kb >> 2, sbyte | (b1 << 8) | (b2 << 16) | (b3 << 24));
    }
  }
  return bad;
}

// Grouped rows r of the routed slots: the token row x[perm[r] / k] (gather)
// or h[r], quantised with the global of the row's expert; scales in the
// tensor-core layout by the expert's 128-row blocks.
template <bool kGather>
__global__ void __launch_bounds__(256) quant_rows_kernel(const uint16_t* __restrict__ src,
                                                         const int32_t* __restrict__ perm,
                                                         const int32_t* __restrict__ idx, int k,
                                                         const int32_t* __restrict__ counts,
                                                         const int32_t* __restrict__ offsets, int S, int K,
                                                         int E, const float* __restrict__ glob,
                                                         uint8_t* __restrict__ codes,
                                                         uint8_t* __restrict__ sf, int* status) {
  pdl_wait();   // programmatic dependent launch: the grouping (or h) is complete
  __shared__ int tpre[kMaxE + 1];
  // 128-row blocks before each expert: every thread loads counts, one warp
  // scans (lane l owns experts [32l .. 32l + 31] of at most 1024)
  for (int e = threadIdx.x; e < E; e += blockDim.x) tpre[e] = (counts[e] + kRows - 1) / kRows;
  __syncthreads();
  if (threadIdx.x < 32) {
    const int l = threadIdx.x;
    const int lo = min(E, 32 * l), hi = min(E, 32 * l + 32);
    int sum = 0;
    for (int e = lo; e < hi; ++e) sum += tpre[e];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (l >= o) incl += v;
    }
    int acc = incl - sum;
    for (int e = lo; e < hi; ++e) {
      const int nb = tpre[e];
      tpre[e] = acc;
      acc += nb;
    }
    if (l == 31) tpre[E] = incl;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  bool bad = false;
  for (long long r = (long long)blockIdx.x * 8 + warp; r < S; r += (long long)gridDim.x * 8) {
    int f = perm[r];
    if (!bounds_ok((unsigned)f < (unsigned)S, status)) f = 0;
    int e = idx[f];
    if (!bounds_ok((unsigned)e < (unsigned)E, status)) e = 0;
    int rl = (int)r - offsets[e];
    if (!bounds_ok(rl >= 0 && rl < counts[e], status)) rl = 0;
    const size_t blk = (size_t)tpre[e] + rl / kRows;
    const uint16_t* row = kGather ? src + (size_t)(f / k) * K : src + (size_t)r * K;
    uint32_t* sfw = reinterpret_cast<uint32_t*>(sf);
    bad |= quantize_row(row, K, glob[e], codes + (size_t)r * (K / 2), [&](int ks, uint32_t word) {
      sfw[tc_scale_offset(blk, rl, 4 * ks, K) / 4] = word;
    });
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(status, kStatusRange);
}

// Plain rows [R, K] to NVFP4 with one global: codes [R, K/2], scales [R, K/16]
// row-major (the standalone quantiser entry point).
__global__ void __launch_bounds__(256) quant_plain_kernel(const uint16_t* __restrict__ src, int R, int K,
                                                          float g, uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ scales, int* flag) {
  const int warp = threadIdx.x >> 5;
  bool bad = false;
  for (long long r = (long long)blockIdx.x * 8 + warp; r < R; r += (long long)gridDim.x * 8) {
    uint32_t* sw = reinterpret_cast<uint32_t*>(scales + (size_t)r * (K / 16));
    bad |= quantize_row(src + (size_t)r * K, K, g, codes + (size_t)r * (K / 2),
                        [&](int ks, uint32_t word) { sw[ks] = word; });
  }
  if (flag && __any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(flag, 1);
}

// Weight scales [E, R, K/16] row-major -> tensor-core layout, one 32-bit
// word (the 4 scales of one row and one 64-wide K step) per thread.  With
// `interleave` (gate/up, R = 2I) block b of expert e holds rows
// (rho odd ? I : 0) + 64 (b % (R/128)) + rho/2 for rho = 0..127, the order in
// which the GEMM loads the interleaved gate and up rows.
__global__ void __launch_bounds__(256) tc_scales_kernel(const uint8_t* __restrict__ in, int E, int R, int K,
                                                        int interleave, uint8_t* __restrict__ out) {
  const long long words = (long long)E * R * (K / 64);
  const int KS = K / 64;
  for (long long wi = (long long)blockIdx.x * blockDim.x + threadIdx.x; wi < words;
       wi += (long long)gridDim.x * blockDim.x) {
    // output order: (block, K step, row % 32, (row % 128) / 32)
    const int jq = (int)(wi & 3);
    const int i = (int)((wi >> 2) & 31);
    const long long rest = wi >> 7;
    const int ks = (int)(rest % KS);
    const long long blk = rest / KS;           // = e * (R/128) + b
    const int e = (int)(blk / (R / kRows));
    const int b = (int)(blk % (R / kRows));
    const int rho = i + 32 * jq;
    const int row = interleave ? ((rho & 1) ? R / 2 : 0) + (kRows / 2) * b + (rho >> 1) : kRows * b + rho;
    const uint32_t v = *reinterpret_cast<const uint32_t*>(in + ((size_t)e * R + row) * (K / 16) + 4 * ks);
    reinterpret_cast<uint32_t*>(out)[wi] = v;
  }
}

// ------------------------------------------------------------------ GEMM
struct TileF {
  int e, m, off, wblk, ttile;
  int sblk;   // the expert's first 128-row activation-scale block
};

template <bool kDown>
__global__ void __launch_bounds__(kThreads, 1)
    tc_fp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const Fp4Args a) {
  pdl_wait();   // programmatic dependent launch: the quantised token rows are complete
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NSF * kStage);
  uint64_t* empty = full + NSF;
  uint64_t* sfull = empty + NSF;    // a stage's scales are in tensor memory
  uint64_t* tfull = sfull + NSF;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;   // after a timeout: the issued MMAs are complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* s_e = reinterpret_cast<int*>(smem + NSF * kStage + 256);
  int* s_m = s_e + (kMaxE + 1);
  int* s_off = s_m + (kMaxE + 1);
  int* s_tiles = s_off + (kMaxE + 1);   // token-tile prefix over the active list

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nact = *a.num_active;
  const int NWB = kDown ? a.H / kRows : 2 * a.I / kRows;   // weight blocks per expert
  const int K = kDown ? a.I : a.H;
  const int KS = K / 64;
  const int nkc = K / kKStage;

  for (int i = threadIdx.x; i < nact; i += kThreads) {
    int e = a.active[i];
    if (!bounds_ok((unsigned)e < (unsigned)a.E, a.status)) e = 0;
    int m = a.counts[e], off = a.offsets[e];
    if (!bounds_ok(off >= 0 && m >= 0 && off + m <= a.T * a.k, a.status)) m = 0, off = 0;
    s_e[i] = e;
    s_m[i] = m;
    s_off[i] = off;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int i = 0; i < nact; ++i) {
      s_tiles[i] = acc;
      acc += (s_m[i] + kRows - 1) / kRows;
    }
    s_tiles[nact] = acc;
  }
  __syncthreads();
  const int total = s_tiles[nact] * NWB;
  if ((int)blockIdx.x >= total) return;   // uniform for the CTA

  // tile t -> (expert, weight block, token tile) in (expert, weight block,
  // token tile) order, so that co-running CTAs share an expert's weights
  auto decode = [&](int t) -> TileF {
    int lo = 0, hi = nact;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_tiles[mid] * NWB <= t) lo = mid; else hi = mid;
    }
    TileF ti;
    const int mt = s_tiles[lo + 1] - s_tiles[lo];
    const int local = t - s_tiles[lo] * NWB;
    ti.e = s_e[lo];
    ti.m = s_m[lo];
    ti.off = s_off[lo];
    ti.wblk = local / mt;
    ti.ttile = local % mt;
    ti.sblk = s_tiles[lo];
    return ti;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSF; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); mbar_init(&sfull[s], kSfWarps); }
    for (int b = 0; b < 2; ++b) { mbar_init(&tfull[b], 1); mbar_init(&tempty[b], kEpiWarps); }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const TileF ti = decode(t);
        const int brow = ti.off + ti.ttile * kRows;
        const size_t ablk = (size_t)ti.e * NWB + ti.wblk;
        // the active list is ascending and holds every expert with rows, so
        // its tile prefix is also the activation scales' block prefix
        const size_t bblk = (size_t)ti.sblk + ti.ttile;
        for (int kc = 0; kc < nkc; ++kc, ++it) {
          const int s = it % NSF;
          const uint32_t ph = (it / NSF) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1)) { ok = false; break; }
          unsigned char* sA = smem + s * kStage;
          unsigned char* sB = sA + kCodeBytes;
          unsigned char* sSA = sB + kCodeBytes;
          unsigned char* sSB = sSA + kSfBytes;
          mbar_expect_tx(&full[s], kStage);
          const int x = kc * (kKStage / 2);   // code bytes
          if (kDown) tma_load_2d(sA, &tmA, x, ti.e * a.H + ti.wblk * kRows, &full[s]);
          else tma_load_4d(sA, &tmA, x, 0, ti.wblk * (kRows / 2), ti.e, &full[s]);
          tma_load_2d(sB, &tmB, x, brow, &full[s]);
          bulk_load(sSA, a.sfa + (ablk * KS + 4 * kc) * kAtomBytes, kSfBytes, &full[s]);
          bulk_load(sSB, a.sfb + (bblk * KS + 4 * kc) * kAtomBytes, kSfBytes, &full[s]);
        }
        if (*(volatile int*)abort_flag) ok = false;
      }
      if (!ok) {
        atomicOr(abort_flag, 1);
        // after a timeout: the copies already issued land before the CTA exits
        for (uint32_t j = it > (uint32_t)NSF ? it - NSF : 0; j < it; ++j) mbar_wait(&full[j % NSF], (j / NSF) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it = 0, lt = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++lt) {
        const TileF ti = decode(t);
        const int rem = ti.m - ti.ttile * kRows;
        const int n = rem >= kRows ? kRows : (rem + 15) & ~15;
        const uint32_t idesc = idesc_fp4(kRows, n);
        const uint32_t b = lt & 1;
        const uint32_t tph = (lt >> 1) & 1;
        if (!mbar_wait(&tempty[b], tph ^ 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + b * kAccCols;
        for (int kc = 0; kc < nkc; ++kc, ++it) {
          const int s = it % NSF;
          const uint32_t ph = (it / NSF) & 1;
          // the codes have landed (full) and the scale warps have written
          // this stage's scales into tensor memory (sfull)
          if (!mbar_wait(&full[s], ph) || !mbar_wait(&sfull[s], ph)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + s * kStage);
          const uint32_t sB = sA + kCodeBytes;
          const uint32_t tsa = tmem_base + kSfColBase + s * kSfColsStage;
          const uint32_t tsb = tsa + 16;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_fp4(tmem_d, umma_desc(sA + kk * 32), umma_desc(sB + kk * 32), idesc, tsa + 4 * kk,
                    tsb + 4 * kk, (kc | kk) != 0 ? 1u : 0u);
          umma_commit(&empty[s]);   // frees the stage (shared and tensor memory) once these MMAs are done
        }
        if (!ok) break;
        umma_commit(&tfull[b]);
        if (*(volatile int*)abort_flag) ok = false;
      }
      if (!ok) {
        atomicOr(abort_flag, 1);
        // after a timeout: the MMAs already issued finish before the tensor
        // memory they write is freed
        umma_commit(drain);
        mbar_wait(drain, 0);
      }
    }
    __syncwarp();
  } else if (warp < 2 + kSfWarps) {
    // ------------------------------------------------------------ scale warps
    const int q = warp & 3;
    const uint32_t lanes = (uint32_t)(q * 32) << 16;
    uint32_t it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      for (int kc = 0; kc < nkc; ++kc, ++it) {
        const int s = it % NSF;
        const uint32_t ph = (it / NSF) & 1;
        if (!warp_wait(&full[s], ph)) { ok = false; break; }
        // atom kk, row `lane`: words j = scales of rows / columns lane + 32j
        const uint4* atA = reinterpret_cast<const uint4*>(smem + s * kStage + 2 * kCodeBytes);
        const uint4* atB = atA + kSfBytes / 16;
        uint32_t va[16], vb[16];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint4 wa = atA[kk * 32 + lane];
          va[4 * kk + 0] = q == 0 ? wa.x : 0u;
          va[4 * kk + 1] = q == 1 ? wa.y : 0u;
          va[4 * kk + 2] = q == 2 ? wa.z : 0u;
          va[4 * kk + 3] = q == 3 ? wa.w : 0u;
          const uint4 wb = atB[kk * 32 + lane];
          vb[4 * kk + 0] = wb.x; vb[4 * kk + 1] = wb.y; vb[4 * kk + 2] = wb.z; vb[4 * kk + 3] = wb.w;
        }
        const uint32_t tsa = tmem_base + lanes + kSfColBase + s * kSfColsStage;
        tmem_st16(tsa, va);
        tmem_st16(tsa + 16, vb);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfull[s]);
      }
      if (*(volatile int*)abort_flag) ok = false;
    }
    if (!ok && lane == 0) atomicOr(abort_flag, 1);
  } else {
    // ------------------------------------------------------------ epilogue
    // warp w reads TMEM lanes 32(w % 4) .. +31, 32-column chunks 2i + hc
    const int q = warp & 3;
    const int hc = (warp - 2 - kSfWarps) >> 2;
    uint32_t lt = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++lt) {
      const uint32_t b = lt & 1;
      const uint32_t tph = (lt >> 1) & 1;
      const TileF ti = decode(t);
      const int tok0 = ti.ttile * kRows;
      const int rem = ti.m - tok0;
      const int ncols = rem < kRows ? rem : kRows;
      const float scale = a.w_global[ti.e] * a.a_global[ti.e];
      int fl[2];
      float wl[2];
      if (kDown) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int c = 32 * (2 * i + hc) + lane;
          fl[i] = c < ncols ? __ldg(&a.perm[ti.off + tok0 + c]) : 0;
          if (!bounds_ok((unsigned)fl[i] < (unsigned)(a.T * a.k), a.status)) fl[i] = 0;
          wl[i] = c < ncols ? __ldg(&a.topk_w[fl[i]]) * scale : 0.f;
        }
      }
      if (!warp_wait(&tfull[b], tph)) { atomicOr(abort_flag, 1); break; }
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + b * kAccCols;
#pragma unroll 1
      for (int i = 0; i < 2; ++i) {
        const int c0 = 32 * (2 * i + hc);
        if (c0 >= ncols) break;   // uniform over the warp
        uint32_t y[32];
        tmem_ld32(tb + c0, y);
        tmem_wait_ld();
        if (!kDown) {
          // lane pair (2jj, 2jj+1) holds gate and up of one j; the even lane
          // forms h for tokens 0-15 of the chunk, the odd lane for 16-31
          const bool odd = lane & 1;
          const int j = ti.wblk * (kRows / 2) + 16 * q + (lane >> 1);
          uint16_t* hcol = a.h + (size_t)(ti.off + tok0 + c0 + (odd ? 16 : 0)) * a.I + j;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float send = __uint_as_float(odd ? y[c] : y[c + 16]);
            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
            const float g = (odd ? recv : __uint_as_float(y[c])) * scale;
            const float u = (odd ? __uint_as_float(y[c + 16]) : recv) * scale;
            if (c0 + c + (odd ? 16 : 0) < ncols) hcol[(size_t)c * a.I] = f2bf(silu(g) * u);
          }
        } else {
          const int d = ti.wblk * kRows + 32 * q + lane;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int f = __shfl_sync(0xffffffffu, fl[i], c);
            const float w = __shfl_sync(0xffffffffu, wl[i], c);
            if (c0 + c < ncols) {
              const float val = w * __uint_as_float(y[c]);
              const size_t o = (size_t)f * a.H + d;
              if (a.partial_f32) reinterpret_cast<float*>(a.partial)[o] = val;
              else reinterpret_cast<uint16_t*>(a.partial)[o] = f2bf(val);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_relaxed(&tempty[b]);   // the accumulator reads are complete
      if (*(volatile int*)abort_flag) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) atomicOr(a.status, kStatusTimeout);
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols));
  }
}

// 4-D tensor map over gate/up codes [E, 2I, H/2] viewed as (k byte, gate/up,
// j, e): a box of {128 bytes, 2, 64 j, 1} lands in shared memory as 128 rows
// of 128 bytes (row 2jj + g), with the 128-byte swizzle.
bool make_map_codes_gate_up(CUtensorMap* m, const void* base, uint64_t E, uint64_t I, uint64_t H) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {H / 2, 2, I, E};
  const cuuint64_t strides[3] = {I * H / 2, H / 2, 2 * I * H / 2};
  const cuuint32_t box[4] = {128, 2, 64, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_quant_rows(bool gather, const uint16_t* src, const int32_t* perm, const int32_t* idx, int k,
                              const int32_t* counts, const int32_t* offsets, int S, int K, int E,
                              const float* glob, uint8_t* codes, uint8_t* sf, int* status, cudaStream_t stream,
                              int* launches) {
  if (launches) *launches += 1;
  const long long blocks = ((long long)S + 7) / 8;
  int dev = 0, nsm = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  const long long cap = 3ll * nsm;   // grid-stride rows: the CTAs that are resident at once
  const unsigned grid = (unsigned)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
  if (gather)
    return launch_pdl(quant_rows_kernel<true>, dim3(grid), dim3(256), 0, stream, src, perm, idx, k, counts, offsets,
                      S, K, E, glob, codes, sf, status);
  return launch_pdl(quant_rows_kernel<false>, dim3(grid), dim3(256), 0, stream, src, perm, idx, k, counts, offsets,
                    S, K, E, glob, codes, sf, status);
}

cudaError_t launch_quant_plain(const uint16_t* src, int R, int K, float g, uint8_t* codes, uint8_t* scales,
                               int* flag, cudaStream_t stream) {
  const long long blocks = ((long long)R + 7) / 8;
  quant_plain_kernel<<<(unsigned)(blocks < 2048 ? (blocks > 0 ? blocks : 1) : 2048), 256, 0, stream>>>(
      src, R, K, g, codes, scales, flag);
  return cudaGetLastError();
}

cudaError_t launch_tc_scales(const uint8_t* in, int E, int R, int K, bool interleave, uint8_t* out,
                             cudaStream_t stream) {
  const long long words = (long long)E * R * (K / 64);
  const long long blocks = (words + 255) / 256;
  tc_scales_kernel<<<(unsigned)(blocks < 4096 ? (blocks > 0 ? blocks : 1) : 4096), 256, 0, stream>>>(
      in, E, R, K, interleave ? 1 : 0, out);
  return cudaGetLastError();
}

cudaError_t launch_tc_fp4(const Fp4Launch& p, bool down, cudaStream_t stream, int* launches) {
  Fp4Args a{};
  a.T = p.T; a.H = p.H; a.E = p.E; a.I = p.I; a.k = p.k;
  a.counts = p.counts; a.offsets = p.offsets; a.perm = p.perm; a.active = p.active;
  a.num_active = p.num_active;
  a.sfa = down ? p.dn_scales_tc : p.gu_scales_tc;
  a.sfb = down ? p.hs : p.xs;
  a.w_global = down ? p.dn_global : p.gu_global;
  a.a_global = down ? p.h_global : p.x_global;
  a.topk_w = p.topk_w; a.h = p.h; a.partial = p.partial; a.partial_f32 = p.partial_f32 ? 1 : 0;
  a.status = p.status;
  const long long S = (long long)p.T * p.k;
  CUtensorMap tmA, tmB;
  if (!down) {
    if (!make_map_codes_gate_up(&tmA, p.gu_codes, p.E, p.I, p.H)) return cudaErrorInvalidValue;
    if (!make_map_2d(&tmB, p.xq, S, p.H / 2, 1, 128, kRows, true)) return cudaErrorInvalidValue;
  } else {
    if (!make_map_2d(&tmA, p.dn_codes, (uint64_t)p.E * p.H, p.I / 2, 1, 128, kRows, true))
      return cudaErrorInvalidValue;
    if (!make_map_2d(&tmB, p.hq, S, p.I / 2, 1, 128, kRows, true)) return cudaErrorInvalidValue;
  }
  auto kern = down ? tc_fp4_kernel<true> : tc_fp4_kernel<false>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  if (launches) *launches += 1;
  return launch_pdl(kern, dim3(p.num_sms), dim3(kThreads), kSmemBytes, stream, tmA, tmB, a);
}

}  // namespace moe
