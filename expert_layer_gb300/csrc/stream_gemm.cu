// Weight-streaming grouped expert GEMMs for small groups (decode-sized).
//
// The "expert kernel" and "activation" phases of the fused-MoE path (page
// "Decode 吞吐专项实验分析报告", section "下一步 profiling 方向", item 3) for
// experts that hold few routed rows.  At decode batch sizes these are bound by
// HBM: every active expert's weights are read once and each weight meets only
// a handful of token rows.  The kernels therefore stream the weights with
// coalesced 128-bit loads that bypass L1, keep the (small, reused) activation
// rows in L1/L2, and do the arithmetic on mma.sync m16n8k16 (bf16 in, fp32
// accumulate) with the weights as the 16-row A operand and up to 32 gathered
// token rows as the B operand ("swap AB").  This replaces the ncols <= 8 MMVQ
// templates of page "第 9 章 prefill：最大的瓶颈" (sec. 9.5): any number of rows
// per expert is served, in passes of 32.
//
// Work unit = (active expert, 16 weight rows over the whole K).
//   gate/up: A rows 0-7 are gate rows j0..j0+7, rows 8-15 the matching up rows
//            I+j0..I+j0+7, so one fragment holds g and u of the same j and the
//            SwiGLU h = silu(g)*u is formed in the epilogue (h rounded to bf16).
//   down:    A rows are 16 consecutive output features d0..d0+15; the epilogue
//            scales by the routing weight and writes the slot's partial row.
// K is split across the CTA's 8 warps; warp partials are summed through
// shared memory in fixed warp order (deterministic).
//
// K-index assignment inside one mma: thread (g, c) of a warp loads 8
// consecutive bf16 (one 16-byte vector) of rows g and g+8 at k = 8c..8c+7 of
// each 32-wide K block; step q of the block feeds pairs (8c+4q, +1) and
// (8c+4q+2, +3) to the fragment slots (2c, 2c+1) and (2c+8, 2c+9).  The B
// operand uses the same assignment, so every k meets its own partner exactly
// once: a permutation of the summation inside each 16-wide step, nothing else.
//
// NVFP4 weights (W4A16): the A fragments are decoded in registers.  Thread
// (g, c) loads 16 bytes of codes (32 elements, k = 32c..32c+31 of a 128-wide
// block) and the two e4m3 scales of those 32 elements; a 256-entry table maps
// a code byte to two bf16 values, multiplied by the bf16 form of the scale.
// Both steps are exact (an e2m1 value times an e4m3 value has at most 6
// significant bits); the per-expert fp32 global scale multiplies the fp32
// accumulator in the epilogue.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kWarpsPerCta = 8;
constexpr int kThreadsPerCta = kWarpsPerCta * 32;
constexpr int kNT = 4;                 // n-tiles (8 tokens each) per pass
constexpr int kPassRows = 8 * kNT;     // 32 token rows per pass

// e2m1 code -> value, from the format: sign, 2-bit exponent (bias 1), 1-bit
// mantissa; exponent 0 is subnormal (m * 0.5).
__device__ float e2m1_value(int code) {
  const int e = (code >> 1) & 3, m = code & 1;
  const float mag = e == 0 ? 0.5f * (float)m : ldexpf(1.0f + 0.5f * (float)m, e - 1);
  return (code & 8) ? -mag : mag;
}

// e4m3 byte -> value: sign, 4-bit exponent (bias 7), 3-bit mantissa; exponent 0
// is subnormal (m/8 * 2^-6); S.1111.111 is NaN.
__device__ float e4m3_value(int b) {
  const int e = (b >> 3) & 15, m = b & 7;
  float mag;
  if (e == 15 && m == 7) mag = __int_as_float(0x7fc00000);
  else if (e == 0) mag = ldexpf((float)m / 8.0f, -6);
  else mag = ldexpf(1.0f + (float)m / 8.0f, e - 7);
  return (b & 0x80) ? -mag : mag;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

template <bool kDown, bool kFp4>
__global__ void __launch_bounds__(kThreadsPerCta, 2) stream_gemm_kernel(StreamGemmArgs a) {
  constexpr int KB = kFp4 ? 128 : 32;       // K elements per block
  constexpr int STEPS = KB / 16;            // mma k-steps per block
  constexpr int KG = kFp4 ? 2 : 4;          // K blocks per load group
  __shared__ float red[kWarpsPerCta][16][kPassRows + 1];
  __shared__ uint32_t lut_e2m1x2[kFp4 ? 256 : 1];
  __shared__ uint16_t lut_e4m3[kFp4 ? 256 : 1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int K = kDown ? a.I : a.H;
  const int NR = kDown ? a.H : 2 * a.I;     // weight rows per expert
  const int UPE = kDown ? a.H / 16 : a.I / 8;

  if constexpr (kFp4) {
    for (int i = threadIdx.x; i < 256; i += kThreadsPerCta) {
      lut_e2m1x2[i] = pack_bf16x2(e2m1_value(i & 15), e2m1_value(i >> 4));
      lut_e4m3[i] = f2bf(e4m3_value(i));
    }
    __syncthreads();
  }

  const int nsmall = *a.num_active - (a.num_large ? *a.num_large : 0);
  const long long U = (long long)nsmall * UPE;
  const long long u_begin = U * blockIdx.x / gridDim.x;
  const long long u_end = U * (blockIdx.x + 1) / gridDim.x;

  const int nkb = K / KB;
  const int kb_begin = nkb * warp / kWarpsPerCta;
  const int kb_end = nkb * (warp + 1) / kWarpsPerCta;

  for (long long u = u_begin; u < u_end; ++u) {
    const int e = a.active[u / UPE];
    const int blk = (int)(u % UPE);
    const int m = a.counts[e];
    const int off = a.offsets[e];
    int row_lo, row_hi;
    if (kDown) { row_lo = blk * 16 + g; row_hi = blk * 16 + 8 + g; }
    else { row_lo = blk * 8 + g; row_hi = a.I + blk * 8 + g; }
    const size_t rlo = (size_t)e * NR + row_lo, rhi = (size_t)e * NR + row_hi;
    float gscale = 1.0f;
    if constexpr (kFp4) gscale = kDown ? a.dn_global[e] : a.gu_global[e];

    for (int p0 = 0; p0 < m; p0 += kPassRows) {
      // token rows of this pass held by this thread: row p0 + nt*8 + g
      const uint16_t* bsrc[kNT];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        const int n = p0 + nt * 8 + g;
        bsrc[nt] = nullptr;
        if (n < m) {
          if (kDown) bsrc[nt] = a.h + (size_t)(off + n) * a.I;
          else bsrc[nt] = a.x + (size_t)(a.perm[off + n] / a.k) * a.H;
        }
      }
      const int ntiles = min(kNT, (m - p0 + 7) / 8);
      float acc[kNT][4];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

      for (int kb0 = kb_begin; kb0 < kb_end; kb0 += KG) {
        // ---- A: weights for up to KG blocks, streamed past L1
        uint4 alo[KG], ahi[KG];
        uint32_t slo[KG], shi[KG];
#pragma unroll
        for (int i = 0; i < KG; ++i) {
          const int kb = kb0 + i;
          if (kb < kb_end) {
            if constexpr (kFp4) {
              const uint8_t* cb = kDown ? a.dn_codes : a.gu_codes;
              const uint8_t* sb = kDown ? a.dn_scales : a.gu_scales;
              const size_t kc = (size_t)kb * 64 + 16 * c;
              alo[i] = ldg_nc_v4(cb + rlo * (K / 2) + kc);
              ahi[i] = ldg_nc_v4(cb + rhi * (K / 2) + kc);
              const size_t ks = (size_t)kb * 8 + 2 * c;
              slo[i] = *reinterpret_cast<const uint16_t*>(sb + rlo * (K / 16) + ks);
              shi[i] = *reinterpret_cast<const uint16_t*>(sb + rhi * (K / 16) + ks);
            } else {
              const uint16_t* wb = kDown ? a.w_down : a.w_gate_up;
              const size_t kc = (size_t)kb * 32 + 8 * c;
              alo[i] = ldg_nc_v4(wb + rlo * K + kc);
              ahi[i] = ldg_nc_v4(wb + rhi * K + kc);
            }
          }
        }
        // ---- per n-tile: B (activations) and the mma steps
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          if (nt < ntiles) {
#pragma unroll
            for (int i = 0; i < KG; ++i) {
              const int kb = kb0 + i;
              if (kb < kb_end) {
                if constexpr (kFp4) {
                  uint32_t b[16];
#pragma unroll
                  for (int v = 0; v < 4; ++v) {
                    uint4 t = make_uint4(0, 0, 0, 0);
                    if (bsrc[nt]) t = *reinterpret_cast<const uint4*>(bsrc[nt] + (size_t)kb * 128 + 32 * c + 8 * v);
                    b[4 * v + 0] = t.x; b[4 * v + 1] = t.y; b[4 * v + 2] = t.z; b[4 * v + 3] = t.w;
                  }
                  const uint32_t clo[4] = {alo[i].x, alo[i].y, alo[i].z, alo[i].w};
                  const uint32_t chi[4] = {ahi[i].x, ahi[i].y, ahi[i].z, ahi[i].w};
#pragma unroll
                  for (int q = 0; q < STEPS; ++q) {
                    const uint32_t sl = lut_e4m3[(slo[i] >> (q < 4 ? 0 : 8)) & 0xff];
                    const uint32_t sh = lut_e4m3[(shi[i] >> (q < 4 ? 0 : 8)) & 0xff];
                    const uint32_t sl2 = sl | (sl << 16), sh2 = sh | (sh << 16);
                    const uint32_t wl = clo[q >> 1] >> (16 * (q & 1));
                    const uint32_t wh = chi[q >> 1] >> (16 * (q & 1));
                    const uint32_t a0 = bf16x2_mul(lut_e2m1x2[wl & 0xff], sl2);
                    const uint32_t a2 = bf16x2_mul(lut_e2m1x2[(wl >> 8) & 0xff], sl2);
                    const uint32_t a1 = bf16x2_mul(lut_e2m1x2[wh & 0xff], sh2);
                    const uint32_t a3 = bf16x2_mul(lut_e2m1x2[(wh >> 8) & 0xff], sh2);
                    mma_bf16_16816(acc[nt], a0, a1, a2, a3, b[2 * q], b[2 * q + 1]);
                  }
                } else {
                  uint4 t = make_uint4(0, 0, 0, 0);
                  if (bsrc[nt]) t = *reinterpret_cast<const uint4*>(bsrc[nt] + (size_t)kb * 32 + 8 * c);
                  mma_bf16_16816(acc[nt], alo[i].x, ahi[i].x, alo[i].y, ahi[i].y, t.x, t.y);
                  mma_bf16_16816(acc[nt], alo[i].z, ahi[i].z, alo[i].w, ahi[i].w, t.z, t.w);
                }
              }
            }
          }
        }
      }

      // ---- cross-warp reduction (fixed warp order) and epilogue
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        red[warp][g][nt * 8 + 2 * c] = acc[nt][0];
        red[warp][g][nt * 8 + 2 * c + 1] = acc[nt][1];
        red[warp][g + 8][nt * 8 + 2 * c] = acc[nt][2];
        red[warp][g + 8][nt * 8 + 2 * c + 1] = acc[nt][3];
      }
      __syncthreads();
      if (!kDown) {
        // thread -> (token n, feature j): 32 x 8
        const int j = threadIdx.x & 7, n = threadIdx.x >> 3;
        if (p0 + n < m) {
          float gs = 0.f, us = 0.f;
#pragma unroll
          for (int w = 0; w < kWarpsPerCta; ++w) { gs += red[w][j][n]; us += red[w][j + 8][n]; }
          gs *= gscale;
          us *= gscale;
          a.h[(size_t)(off + p0 + n) * a.I + blk * 8 + j] = f2bf(silu(gs) * us);
        }
      } else {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int id = threadIdx.x + r * kThreadsPerCta;   // 512 = 32 tokens x 16 features
          const int d = id & 15, n = id >> 4;
          if (p0 + n < m) {
            float ys = 0.f;
#pragma unroll
            for (int w = 0; w < kWarpsPerCta; ++w) ys += red[w][d][n];
            ys *= gscale;
            const int f = a.perm[off + p0 + n];
            const float v = a.topk_w[f] * ys;
            const size_t o = (size_t)f * a.H + blk * 16 + d;
            if (a.partial_f32) reinterpret_cast<float*>(a.partial)[o] = v;
            else reinterpret_cast<uint16_t*>(a.partial)[o] = f2bf(v);
          }
        }
      }
      __syncthreads();
    }
  }
}

template <bool kDown>
cudaError_t launch_stream(const StreamGemmArgs& a, cudaStream_t stream, int* launches) {
  if (launches) *launches += 1;
  const bool fp4 = a.gu_codes != nullptr;
  const long long S = (long long)a.T * a.k;
  const long long max_active = S < a.E ? S : a.E;
  const long long UPE = kDown ? a.H / 16 : a.I / 8;
  long long units = max_active * UPE;
  long long grid = (long long)a.num_sms * 2;
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  if (fp4) stream_gemm_kernel<kDown, true><<<(unsigned)grid, kThreadsPerCta, 0, stream>>>(a);
  else stream_gemm_kernel<kDown, false><<<(unsigned)grid, kThreadsPerCta, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_stream_gate_up(const StreamGemmArgs& a, cudaStream_t stream, int* launches) {
  return launch_stream<false>(a, stream, launches);
}
cudaError_t launch_stream_down(const StreamGemmArgs& a, cudaStream_t stream, int* launches) {
  return launch_stream<true>(a, stream, launches);
}

}  // namespace moe
