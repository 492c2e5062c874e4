// Combine ("sum" phase of the fused-MoE path, page "Decode 吞吐专项实验分析报告",
// section "下一步 profiling 方向", item 3):
//   out[t, d] = bf16( sum_{s=0..k-1} partial[t*k + s, d] )
// summed in slot order in fp32, with no atomics, so the result is bitwise
// reproducible and does not depend on how slots were grouped.  The partials
// already carry the routing weight.  HBM-bound: one read of S*H partials and
// one write of T*H outputs, 16-byte vectors, grid-stride over T*H/8.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

template <bool kF32>
__global__ void __launch_bounds__(256) combine_kernel(const void* __restrict__ partial, int T, int H,
                                                      int k, uint16_t* __restrict__ out) {
  pdl_wait();   // the partials of the down projection are complete
  const long long nvec = (long long)T * (H / 8);
  for (long long v = blockIdx.x * (long long)blockDim.x + threadIdx.x; v < nvec;
       v += (long long)gridDim.x * blockDim.x) {
    const long long t = v / (H / 8);
    const int d = (int)(v % (H / 8)) * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < k; ++s) {
      const size_t row = (size_t)(t * k + s) * H + d;
      if constexpr (kF32) {
        const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(partial) + row);
        const float4 lo = p[0], hi = p[1];
        acc[0] += lo.x; acc[1] += lo.y; acc[2] += lo.z; acc[3] += lo.w;
        acc[4] += hi.x; acc[5] += hi.y; acc[6] += hi.z; acc[7] += hi.w;
      } else {
        const uint4 q = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(partial) + row);
        acc[0] += bf16lo(q.x); acc[1] += bf16hi(q.x); acc[2] += bf16lo(q.y); acc[3] += bf16hi(q.y);
        acc[4] += bf16lo(q.z); acc[5] += bf16hi(q.z); acc[6] += bf16lo(q.w); acc[7] += bf16hi(q.w);
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(out + (size_t)t * H + d) = o;
  }
}

}  // namespace

cudaError_t launch_combine(const void* partial, bool partial_f32, int T, int H, int k,
                           uint16_t* out, cudaStream_t stream, int* launches) {
  if (launches) *launches += 1;
  const long long nvec = (long long)T * (H / 8);
  long long grid = (nvec + 255) / 256;
  if (grid > 152 * 8) grid = 152 * 8;
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
