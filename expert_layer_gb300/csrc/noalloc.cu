// moe_route_noalloc: the router of moe_route, for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the
// point where they route tokens: code running while a CUDA graph is being
// captured, a runtime whose memory is pre-reserved and handed out by its own
// pool, or a host integration that forbids allocation after start-up.  They
// also may not have a workspace buffer of their own to lend to moe_route.
// This entry point keeps the router's scratch in a fixed device array that
// is part of the library image, so the caller passes only inputs, outputs
// and a stream.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes
// (about 0.8 MB).  Every GPU that loads this library holds one copy of it
// until the process exits.  Host code cannot use the array's name as a
// device address, so on the first call on each device (with that device
// current) the library looks up the array's device address with
// cudaGetSymbolAddress and caches it; make that first call before any stream
// capture begins.  The cached address stays valid while the device's primary
// context lives: after cudaDeviceReset the library image is loaded again at
// another address, so the entry point must not be called on a device that was
// reset.  All calls on a device share the one array and it keeps
// the previous call's contents: the header words that must start at zero are
// cleared on the stream at the start of each call.  Calls whose work overlaps
// on the GPU (different streams without ordering between them) race on the
// array and give undefined results.
#include <mutex>

#include "moe.h"
#include "common.cuh"
#include "kernels.h"

namespace {

// Largest T*E the array serves; T itself is also bounded (xnorm holds T floats).
constexpr long long kNoAllocMaxTE = 65536;
constexpr long long kNoAllocMaxT = 8192;
// header + scheduling counters[E+2] + counters[T] + per-expert counters[E] +
// xnorm[T] + wnorm[E] + fp32 logits[T*E] + fp64 logits[T*E] + the tiled
// router's pieces (partial logits[pieces*T*E], partial squares[pieces*T]),
// each region 256-byte aligned (the router's part of the workspace layout)
constexpr size_t kNoAllocScratchBytes =
    256 + 1026 * 4 + 2 * kNoAllocMaxT * 4 + 2 * 1024 * 4 + kNoAllocMaxTE * 4 + kNoAllocMaxTE * 8 +
    moe::kRouteTilePieces * (kNoAllocMaxTE + kNoAllocMaxT) * 4 + 9 * 256;

__device__ __align__(256) unsigned char g_route_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_route_scratch on the current device (looked up once).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" int moe_route_noalloc(const uint16_t* x, const uint16_t* gate_w, const float* bias,
                                 int T, int H, int E, int top_k, int32_t* topk_idx,
                                 float* topk_w, void* stream) {
  if (T < 0 || H <= 0 || E <= 0 || top_k <= 0 || top_k > E) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || top_k > 32 || H % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if ((long long)T * E > kNoAllocMaxTE || T > kNoAllocMaxT) return MOE_ERR_UNSUPPORTED;
  if (!x || !gate_w || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!a16(x) || !a16(gate_w) || !a16(topk_idx) || !a16(topk_w) || (bias && !a16(bias)))
    return MOE_ERR_UNSUPPORTED;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;

  // The router touches only the regions before `idx` in the workspace layout.
  const moe::WsLayout L = moe::make_layout(T, H, E, 128, top_k);
  if (L.idx > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != MOE_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (moe::launch_zero(scratch, moe::zeroed_prefix(L), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::launch_route(x, gate_w, bias, T, H, E, top_k, topk_idx, topk_w, scratch, L, s,
                        nullptr, nullptr) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
