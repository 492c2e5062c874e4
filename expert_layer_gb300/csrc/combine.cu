// Combine ("sum" phase of the fused-MoE path, page "Decode 吞吐专项实验分析报告",
// section "下一步 profiling 方向", item 3):
//   out[t, d] = bf16( sum_{s=0..k-1} partial[t*k + s, d] )
// summed in slot order in fp32, with no atomics, so the result is bitwise
// reproducible and does not depend on how slots were grouped.  The partials
// already carry the routing weight.  HBM-bound: one read of S*H partials and
// one write of T*H outputs, grid-stride over 16-byte vectors of partials.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

// Thread = V consecutive outputs of one token (one 16-byte vector of
// partials per slot: V = 4 fp32 or 8 bf16).  The k partial vectors are loaded
// in batches of 8 before any is added, so a thread waits on memory once per
// batch rather than once per slot; the additions still run in slot order
// from zero.
template <bool kF32>
__global__ void __launch_bounds__(256) combine_kernel(const void* __restrict__ partial, int T, int H,
                                                      int k, uint16_t* __restrict__ out) {
  constexpr int V = kF32 ? 4 : 8;
  if ((long long)T * (H / V) <= (long long)gridDim.x * blockDim.x) {
    // one vector per thread (small batches): while the down projection
    // finishes, bring this thread's partial row segment's address translation
    // and lines toward L2 (a prefetch returns no data; the partials are read
    // only after the wait)
    const long long v0 = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (v0 < (long long)T * (H / V)) {
      const size_t row = (size_t)(v0 / (H / V)) * k * H + (size_t)(v0 % (H / V)) * V;
      const void* pp = kF32 ? static_cast<const void*>(reinterpret_cast<const float*>(partial) + row)
                            : static_cast<const void*>(reinterpret_cast<const uint16_t*>(partial) + row);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(pp));
    }
  }
  pdl_wait();   // the partials of the down projection are complete
  const long long nvec = (long long)T * (H / V);
  for (long long v = blockIdx.x * (long long)blockDim.x + threadIdx.x; v < nvec;
       v += (long long)gridDim.x * blockDim.x) {
    const long long t = v / (H / V);
    const int d = (int)(v % (H / V)) * V;
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    for (int s0 = 0; s0 < k; s0 += 8) {
      uint4 q[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        q[j] = make_uint4(0, 0, 0, 0);
        if (s0 + j < k) {
          const size_t row = (size_t)(t * k + s0 + j) * H + d;
          q[j] = kF32 ? *reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(partial) + row)
                      : *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(partial) + row);
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (s0 + j < k) {
          const uint32_t w4[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
          if constexpr (kF32) {
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] += __uint_as_float(w4[i]);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) { acc[2 * i] += bf16lo(w4[i]); acc[2 * i + 1] += bf16hi(w4[i]); }
          }
        }
      }
    }
    if constexpr (kF32) {
      uint2 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      *reinterpret_cast<uint2*>(out + (size_t)t * H + d) = o;
    } else {
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      *reinterpret_cast<uint4*>(out + (size_t)t * H + d) = o;
    }
  }
}

}  // namespace

cudaError_t launch_combine(const void* partial, bool partial_f32, int T, int H, int k,
                           uint16_t* out, int num_sms, cudaStream_t stream, int* launches) {
  if (launches) *launches += 1;
  const long long nvec = (long long)T * (H / (partial_f32 ? 4 : 8));
  long long grid = (nvec + 255) / 256;
  // grid-stride beyond eight 256-thread CTAs per SM
  const long long cap = 8ll * (num_sms > 0 ? num_sms : 1);
  if (grid > cap) grid = cap;
  // programmatic launch: the combine's CTAs may become resident while the down
  // projection finishes and start the moment it completes
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (partial_f32) return cudaLaunchKernelEx(&cfg, combine_kernel<true>, partial, T, H, k, out);
  return cudaLaunchKernelEx(&cfg, combine_kernel<false>, partial, T, H, k, out);
}

}  // namespace moe
