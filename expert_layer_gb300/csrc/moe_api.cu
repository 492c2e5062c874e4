// C ABI of the MoE layer library: argument checks, workspace layout, launch
// sequence.  Nothing here allocates, synchronises or keeps state between
// calls (moe_read_status is the one call that synchronises, by design).
#include <limits.h>
#include <stdint.h>
#include <stdio.h>

#include <atomic>

#include "moe.h"
#include "common.cuh"
#include "kernels.h"

using namespace moe;

namespace moe {

namespace {
// The workspace prefix that must start at zero.  The first thing it does is
// allow the next kernel (launched as a programmatic dependent) to become
// resident; that kernel waits for this one's stores before reading anything.
__global__ void __launch_bounds__(256) zero_kernel(uint4* __restrict__ p, int n16) {
  pdl_trigger();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += gridDim.x * blockDim.x)
    p[i] = make_uint4(0, 0, 0, 0);
}
}  // namespace

namespace {
// Test-only wait settings (moe_debug_force_wait_timeout); zero in normal use.
std::atomic<int> g_debug_spin{0};
std::atomic<int> g_debug_force{0};
}  // namespace

DebugWaits debug_waits() { return DebugWaits{g_debug_spin.load(), g_debug_force.load()}; }

cudaError_t launch_zero(void* ws, size_t bytes, cudaStream_t stream) {
  const int n16 = (int)(bytes / 16);
  int grid = (n16 + 255) / 256;
  if (grid > 64) grid = 64;
  if (grid < 1) grid = 1;
  zero_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<uint4*>(ws), n16);
  return cudaGetLastError();
}

}  // namespace moe

namespace {

// Group size from which an expert runs on the tensor-core kernels: at
// prefill sizes a 32-row group already pays for a 128-row tile; at decode
// sizes the streaming kernels serve groups of up to 64 rows better.
constexpr int kLargeGroupPrefill = 32;
constexpr int kLargeGroupDecode = 65;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(long long T, long long H, long long E, long long I, long long k) {
  if (T < 0 || H <= 0 || E <= 0 || I <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
  if (k > E) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || k > 32) return MOE_ERR_UNSUPPORTED;
  if (H % 128 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (T * k >= (1ll << 31) || T * H >= (1ll << 40)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int check_device(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;
  if (num_sms &&
      cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                 \
  do {                                \
    const int _rc = (expr);           \
    if (_rc != MOE_OK) return _rc;    \
  } while (0)

#define MOE_TRY_CUDA(expr)                                 \
  do {                                                     \
    if ((expr) != cudaSuccess) return MOE_ERR_CUDA;        \
  } while (0)

int check_ptr(const void* p) {
  if (!p) return MOE_ERR_INVALID_ARG;
  if (!aligned16(p)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_version(void) { return 100; }

const char* moe_error_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: unsupported shape, alignment or device";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace too small";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: CUDA runtime or launch failure";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE: a kernel found invalid data";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT: a bounded device wait gave up";
    default: return "unknown moe_status";
  }
}

size_t moe_workspace_size(int T, int H, int E, int I, int top_k) {
  if (check_shape(T, H, E, I, top_k) != MOE_OK) return 0;
  return make_layout(T, H, E, I, top_k).total;
}

int moe_route(const uint16_t* x, const uint16_t* gate_w, const float* bias, int T, int H, int E,
              int top_k, int32_t* topk_idx, float* topk_w, void* workspace,
              size_t workspace_bytes, void* stream) {
  MOE_TRY(check_shape(T, H, E, 128, top_k));
  if (T == 0) return MOE_OK;
  MOE_TRY(check_ptr(x));
  MOE_TRY(check_ptr(gate_w));
  MOE_TRY(check_ptr(topk_idx));
  MOE_TRY(check_ptr(topk_w));
  MOE_TRY(check_ptr(workspace));
  if (bias && !aligned16(bias)) return MOE_ERR_UNSUPPORTED;
  const WsLayout L = make_layout(T, H, E, 128, top_k);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
  MOE_TRY(check_device(nullptr));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  MOE_TRY_CUDA(launch_zero(workspace, zeroed_prefix(L), s));
  return cuda_status(
      launch_route(x, gate_w, bias, T, H, E, top_k, topk_idx, topk_w, workspace, L, s, nullptr,
                   nullptr));
}

int moe_permute(const int32_t* topk_idx, int T, int E, int top_k, int32_t* counts,
                int32_t* offsets, int32_t* perm, int32_t* inv_perm, void* workspace,
                size_t workspace_bytes, void* stream) {
  MOE_TRY(check_shape(T, 128, E, 128, top_k));
  if (T == 0) return MOE_OK;
  MOE_TRY(check_ptr(topk_idx));
  MOE_TRY(check_ptr(counts));
  MOE_TRY(check_ptr(offsets));
  MOE_TRY(check_ptr(perm));
  MOE_TRY(check_ptr(inv_perm));
  MOE_TRY(check_ptr(workspace));
  const WsLayout L = make_layout(T, 128, E, 128, top_k);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
  MOE_TRY(check_device(nullptr));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  MOE_TRY_CUDA(launch_zero(workspace, zeroed_prefix(L), s));
  return cuda_status(launch_permute(topk_idx, T, E, top_k, counts, offsets, perm, inv_perm,
                                    workspace, L, INT_MAX, 128, s, nullptr));
}

static int forward_impl(const uint16_t* x, const uint16_t* gate_w, const float* bias,
                        const uint16_t* w_gate_up, const uint16_t* w_down,
                        const moe_nvfp4_weights* nvfp4, const moe_int8_weights* q8, int T, int H, int E, int I, int top_k,
                        uint16_t* out, int32_t* topk_idx, float* topk_w, void* workspace,
                        size_t workspace_bytes, void* stream, void* const* events,
                        int* launches) {
  MOE_TRY(check_shape(T, H, E, I, top_k));
  if (T == 0) return MOE_OK;
  MOE_TRY(check_ptr(x));
  MOE_TRY(check_ptr(gate_w));
  MOE_TRY(check_ptr(out));
  MOE_TRY(check_ptr(workspace));
  if (bias && !aligned16(bias)) return MOE_ERR_UNSUPPORTED;
  if (topk_idx && !aligned16(topk_idx)) return MOE_ERR_UNSUPPORTED;
  if (topk_w && !aligned16(topk_w)) return MOE_ERR_UNSUPPORTED;
  if (q8) {
    if (w_gate_up || w_down || nvfp4) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_ptr(q8->gu_codes));
    MOE_TRY(check_ptr(q8->gu_scales));
    MOE_TRY(check_ptr(q8->dn_codes));
    MOE_TRY(check_ptr(q8->dn_scales));
  } else if (nvfp4) {
    if (w_gate_up || w_down) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_ptr(nvfp4->gu_codes));
    MOE_TRY(check_ptr(nvfp4->gu_scales));
    MOE_TRY(check_ptr(nvfp4->gu_global));
    MOE_TRY(check_ptr(nvfp4->dn_codes));
    MOE_TRY(check_ptr(nvfp4->dn_scales));
    MOE_TRY(check_ptr(nvfp4->dn_global));
  } else {
    MOE_TRY(check_ptr(w_gate_up));
    MOE_TRY(check_ptr(w_down));
  }
  const WsLayout L = make_layout(T, H, E, I, top_k);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
  int num_sms = 0;
  MOE_TRY(check_device(&num_sms));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  int32_t* idx = topk_idx ? topk_idx : ws_ptr<int32_t>(workspace, L.idx);
  float* w = topk_w ? topk_w : ws_ptr<float>(workspace, L.w);
  int32_t* counts = ws_ptr<int32_t>(workspace, L.counts);
  int32_t* offsets = ws_ptr<int32_t>(workspace, L.offsets);
  int32_t* perm = ws_ptr<int32_t>(workspace, L.perm);
  int32_t* inv_perm = ws_ptr<int32_t>(workspace, L.inv_perm);
  WsHeader* hdr = ws_ptr<WsHeader>(workspace, L.hdr);

  auto mark = [&](int i) -> cudaError_t {
    return events ? cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[i]), s) : cudaSuccess;
  };
  // Experts with at least `large` rows go to the tensor-core kernels (bf16
  // weights, H a multiple of their 256-wide output tiles); a group can never
  // exceed T rows, so small batches skip them.
  const bool prefill = (long long)T * top_k >= 8192;
  const int large = prefill ? kLargeGroupPrefill : kLargeGroupDecode;
  const bool use_tc = !nvfp4 && !q8 && T >= large && H % 256 == 0 && num_sms >= 2;
  // At prefill sizes every group goes to the tensor-core kernels: a 128-row
  // tile of a small group costs the whole GPU about 0.7 us of tensor time,
  // less than streaming that expert's 9.4 MB of weights, and the streaming
  // kernel is then not launched at all.
  const bool tc_all = use_tc && prefill;
  const int large_threshold = tc_all ? 1 : use_tc ? large : INT_MAX;
  // Small batches fuse the grouping into the router.
  const bool fuse = !use_tc && route_can_group(T, E, top_k);
  // the NVFP4 and int8 expert kernels multiply in f16: the router writes x
  // converted to f16 while it reads x for the logits
  uint16_t* x16 = (nvfp4 || q8) ? ws_ptr<uint16_t>(workspace, L.x16) : nullptr;

  MOE_TRY_CUDA(mark(0));
  MOE_TRY_CUDA(launch_zero(workspace, zeroed_prefix(L), s));
  if (launches) *launches += 1;
  if (fuse) {
    GroupOut go{ws_ptr<int>(workspace, L.acnt), ws_ptr<int>(workspace, L.lrank)};
    MOE_TRY_CUDA(launch_route(x, gate_w, bias, T, H, E, top_k, idx, w, workspace, L, s, launches, &go, x16));
    MOE_TRY_CUDA(mark(1));
    MOE_TRY_CUDA(mark(2));
  } else {
    MOE_TRY_CUDA(launch_route(x, gate_w, bias, T, H, E, top_k, idx, w, workspace, L, s, launches,
                              nullptr, x16));
    MOE_TRY_CUDA(mark(1));
    MOE_TRY_CUDA(launch_permute(idx, T, E, top_k, counts, offsets, perm, inv_perm, workspace, L,
                                large_threshold, kTcRows, s, launches));
    MOE_TRY_CUDA(mark(2));
  }

  StreamGemmArgs a{};
  a.T = T; a.H = H; a.E = E; a.I = I; a.k = top_k;
  a.counts = counts; a.offsets = offsets; a.perm = perm;
  a.active = ws_ptr<int32_t>(workspace, L.active);
  a.num_active = &hdr->num_active;
  a.num_large = &hdr->num_large;
  a.x = x;
  a.w_gate_up = w_gate_up;
  a.w_down = w_down;
  if (nvfp4) {
    a.gu_codes = nvfp4->gu_codes; a.gu_scales = nvfp4->gu_scales; a.gu_global = nvfp4->gu_global;
    a.dn_codes = nvfp4->dn_codes; a.dn_scales = nvfp4->dn_scales; a.dn_global = nvfp4->dn_global;
  }
  if (q8) {
    a.gu_q8 = q8->gu_codes; a.gu_q8s = q8->gu_scales;
    a.dn_q8 = q8->dn_codes; a.dn_q8s = q8->dn_scales;
  }
  a.h = ws_ptr<uint16_t>(workspace, L.h);
  a.topk_w = w;
  a.partial = ws_ptr<void>(workspace, L.partial);
  a.partial_f32 = L.partial_f32;
  a.queue = ws_ptr<int>(workspace, L.sched);
  a.dep = a.queue + 1;
  // with every group on the streaming kernel, and a combine small enough
  // that each of its threads (at least 224 per SM) sums about one 16-byte
  // vector, the streaming kernel also does the combine (measured: decode8
  // 94.9 -> 93.2-94.0 us per step; at T = 256 the separate, wider combine
  // kernel is 2-3 us faster)
  const long long comb_vecs = (long long)T * (H / (L.partial_f32 ? 4 : 8));
  a.fused_combine = !use_tc && comb_vecs <= 224ll * num_sms;
  a.done = a.queue + 1 + E;
  a.out = out;
  a.status = &hdr->status;
  a.num_sms = num_sms;
  if (fuse) {
    // the expert kernel groups the batch itself from the router's ranks
    a.self_group = true;
    a.acnt = ws_ptr<int>(workspace, L.acnt);
    a.idx = idx;
    a.rank = ws_ptr<int>(workspace, L.lrank);
    a.counts_out = counts; a.offsets_out = offsets; a.active_out = ws_ptr<int32_t>(workspace, L.active);
    a.perm_out = perm; a.inv_perm_out = inv_perm;
    a.num_active_out = &hdr->num_active; a.num_large_out = &hdr->num_large;
  }
  TcLaunch tc{};
  tc.T = T; tc.H = H; tc.E = E; tc.I = I; tc.k = top_k;
  tc.counts = counts; tc.offsets = offsets; tc.perm = perm; tc.active = a.active;
  tc.tiles = ws_ptr<int32_t>(workspace, L.tiles);
  tc.num_active = &hdr->num_active; tc.num_large = &hdr->num_large;
  tc.x = x; tc.xp = ws_ptr<uint16_t>(workspace, L.xp); tc.w_gate_up = w_gate_up; tc.w_down = w_down; tc.topk_w = w;
  tc.h = a.h; tc.partial = a.partial; tc.partial_f32 = L.partial_f32;
  tc.status = &hdr->status; tc.num_sms = num_sms;

  a.x16 = x16;
  if (!tc_all) MOE_TRY_CUDA(launch_stream_gemm(a, s, launches));
  MOE_TRY_CUDA(mark(3));
  if (use_tc) {
    MOE_TRY_CUDA(launch_tc_gemm(tc, false, s, launches));
    MOE_TRY_CUDA(launch_tc_gemm(tc, true, s, launches));
  }
  MOE_TRY_CUDA(mark(4));
  if (!a.fused_combine)
    MOE_TRY_CUDA(launch_combine(a.partial, L.partial_f32, T, H, top_k, out, num_sms, s, launches));
  MOE_TRY_CUDA(mark(5));
  return MOE_OK;
}

int moe_forward(const uint16_t* x, const uint16_t* gate_w, const float* bias,
                const uint16_t* w_gate_up, const uint16_t* w_down, const moe_nvfp4_weights* nvfp4,
                int T, int H, int E, int I, int top_k, uint16_t* out, int32_t* topk_idx,
                float* topk_w, void* workspace, size_t workspace_bytes, void* stream) {
  return forward_impl(x, gate_w, bias, w_gate_up, w_down, nvfp4, nullptr, T, H, E, I, top_k, out,
                      topk_idx, topk_w, workspace, workspace_bytes, stream, nullptr, nullptr);
}

int moe_forward_profiled(const uint16_t* x, const uint16_t* gate_w, const float* bias,
                         const uint16_t* w_gate_up, const uint16_t* w_down,
                         const moe_nvfp4_weights* nvfp4, int T, int H, int E, int I, int top_k,
                         uint16_t* out, int32_t* topk_idx, float* topk_w, void* workspace,
                         size_t workspace_bytes, void* stream, void* const* events,
                         int32_t* kernels_launched) {
  if (!events) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 6; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  int n = 0;
  const int rc = forward_impl(x, gate_w, bias, w_gate_up, w_down, nvfp4, nullptr, T, H, E, I, top_k,
                              out, topk_idx, topk_w, workspace, workspace_bytes, stream, events, &n);
  if (kernels_launched) *kernels_launched = n;
  return rc;
}

// ------------------------------------------------------------------ int8
int moe_forward_int8(const uint16_t* x, const uint16_t* gate_w, const float* bias, const moe_int8_weights* w,
                     int T, int H, int E, int I, int top_k, uint16_t* out, int32_t* topk_idx, float* topk_w,
                     void* workspace, size_t workspace_bytes, void* stream) {
  if (!w) return MOE_ERR_INVALID_ARG;
  return forward_impl(x, gate_w, bias, nullptr, nullptr, nullptr, w, T, H, E, I, top_k, out, topk_idx,
                      topk_w, workspace, workspace_bytes, stream, nullptr, nullptr);
}

int moe_forward_int8_profiled(const uint16_t* x, const uint16_t* gate_w, const float* bias,
                              const moe_int8_weights* w, int T, int H, int E, int I, int top_k,
                              uint16_t* out, int32_t* topk_idx, float* topk_w, void* workspace,
                              size_t workspace_bytes, void* stream, void* const* events,
                              int32_t* kernels_launched) {
  if (!w || !events) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 6; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  int n = 0;
  const int rc = forward_impl(x, gate_w, bias, nullptr, nullptr, nullptr, w, T, H, E, I, top_k, out,
                              topk_idx, topk_w, workspace, workspace_bytes, stream, events, &n);
  if (kernels_launched) *kernels_launched = n;
  return rc;
}

// ------------------------------------------------------------------ W4A4
static int check_w4a4_shape(int H, int I) {
  // 256-wide K stages (H, I) and 128-row weight blocks; scale rows of H/16 and
  // I/16 bytes whose 64-wide K steps are whole 4-byte words
  return (H % 256 == 0 && I % 256 == 0) ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

static int w4a4_impl(const uint16_t* x, const uint16_t* gate_w, const float* bias, const moe_w4a4_weights* wq,
                     int T, int H, int E, int I, int top_k, uint16_t* out, int32_t* topk_idx, float* topk_w,
                     void* workspace, size_t workspace_bytes, void* stream, void* const* events, int* launches) {
  MOE_TRY(check_shape(T, H, E, I, top_k));
  if (T == 0) return MOE_OK;
  if (!wq) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_w4a4_shape(H, I));
  MOE_TRY(check_ptr(x));
  MOE_TRY(check_ptr(gate_w));
  MOE_TRY(check_ptr(out));
  MOE_TRY(check_ptr(workspace));
  if (bias && !aligned16(bias)) return MOE_ERR_UNSUPPORTED;
  if (topk_idx && !aligned16(topk_idx)) return MOE_ERR_UNSUPPORTED;
  if (topk_w && !aligned16(topk_w)) return MOE_ERR_UNSUPPORTED;
  MOE_TRY(check_ptr(wq->gu_codes));
  MOE_TRY(check_ptr(wq->gu_scales_tc));
  MOE_TRY(check_ptr(wq->gu_global));
  MOE_TRY(check_ptr(wq->dn_codes));
  MOE_TRY(check_ptr(wq->dn_scales_tc));
  MOE_TRY(check_ptr(wq->dn_global));
  MOE_TRY(check_ptr(wq->x_global));
  MOE_TRY(check_ptr(wq->h_global));
  const WsLayout L = make_layout(T, H, E, I, top_k);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
  int num_sms = 0;
  MOE_TRY(check_device(&num_sms));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const long long S = (long long)T * top_k;

  int32_t* idx = topk_idx ? topk_idx : ws_ptr<int32_t>(workspace, L.idx);
  float* w = topk_w ? topk_w : ws_ptr<float>(workspace, L.w);
  int32_t* counts = ws_ptr<int32_t>(workspace, L.counts);
  int32_t* offsets = ws_ptr<int32_t>(workspace, L.offsets);
  int32_t* perm = ws_ptr<int32_t>(workspace, L.perm);
  int32_t* inv_perm = ws_ptr<int32_t>(workspace, L.inv_perm);
  WsHeader* hdr = ws_ptr<WsHeader>(workspace, L.hdr);
  auto mark = [&](int i) -> cudaError_t {
    return events ? cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[i]), s) : cudaSuccess;
  };
  // NVFP4 activations in the token-row region: codes, then 256-aligned scales
  uint8_t* xq = ws_ptr<uint8_t>(workspace, L.xp);
  uint8_t* hq = xq + align256((size_t)S * H / 2);
  uint8_t* xs = hq + align256((size_t)S * I / 2);
  uint8_t* hs = xs + align256(fp4_act_scale_bytes(S, E, H));

  MOE_TRY_CUDA(mark(0));
  MOE_TRY_CUDA(launch_zero(workspace, zeroed_prefix(L), s));
  if (launches) *launches += 1;
  MOE_TRY_CUDA(launch_route(x, gate_w, bias, T, H, E, top_k, idx, w, workspace, L, s, launches, nullptr));
  MOE_TRY_CUDA(mark(1));
  // every active expert is served by the tensor cores (128-row blocks)
  MOE_TRY_CUDA(launch_permute(idx, T, E, top_k, counts, offsets, perm, inv_perm, workspace, L, 1, kTcRows, s,
                              launches));
  MOE_TRY_CUDA(mark(2));
  MOE_TRY_CUDA(launch_quant_rows(true, x, perm, idx, top_k, counts, offsets, (int)S, H, E, wq->x_global, xq, xs,
                                 &hdr->status, s, launches));
  MOE_TRY_CUDA(mark(3));
  Fp4Launch p{};
  p.T = T; p.H = H; p.E = E; p.I = I; p.k = top_k;
  p.counts = counts; p.offsets = offsets; p.perm = perm;
  p.active = ws_ptr<int32_t>(workspace, L.active);
  p.num_active = &hdr->num_active;
  p.gu_codes = wq->gu_codes; p.gu_scales_tc = wq->gu_scales_tc; p.gu_global = wq->gu_global;
  p.dn_codes = wq->dn_codes; p.dn_scales_tc = wq->dn_scales_tc; p.dn_global = wq->dn_global;
  p.x_global = wq->x_global; p.h_global = wq->h_global;
  p.xq = xq; p.xs = xs; p.hq = hq; p.hs = hs;
  p.topk_w = w;
  p.h = ws_ptr<uint16_t>(workspace, L.h);
  p.partial = ws_ptr<void>(workspace, L.partial);
  p.partial_f32 = L.partial_f32;
  p.status = &hdr->status;
  p.num_sms = num_sms;
  MOE_TRY_CUDA(launch_tc_fp4(p, false, s, launches));
  MOE_TRY_CUDA(launch_quant_rows(false, p.h, perm, idx, top_k, counts, offsets, (int)S, I, E, wq->h_global, hq, hs,
                                 &hdr->status, s, launches));
  MOE_TRY_CUDA(launch_tc_fp4(p, true, s, launches));
  MOE_TRY_CUDA(mark(4));
  MOE_TRY_CUDA(launch_combine(p.partial, L.partial_f32, T, H, top_k, out, num_sms, s, launches));
  MOE_TRY_CUDA(mark(5));
  return MOE_OK;
}

int moe_forward_w4a4(const uint16_t* x, const uint16_t* gate_w, const float* bias, const moe_w4a4_weights* w,
                     int T, int H, int E, int I, int top_k, uint16_t* out, int32_t* topk_idx, float* topk_w,
                     void* workspace, size_t workspace_bytes, void* stream) {
  return w4a4_impl(x, gate_w, bias, w, T, H, E, I, top_k, out, topk_idx, topk_w, workspace, workspace_bytes,
                   stream, nullptr, nullptr);
}

int moe_forward_w4a4_profiled(const uint16_t* x, const uint16_t* gate_w, const float* bias,
                              const moe_w4a4_weights* w, int T, int H, int E, int I, int top_k, uint16_t* out,
                              int32_t* topk_idx, float* topk_w, void* workspace, size_t workspace_bytes,
                              void* stream, void* const* events, int32_t* kernels_launched) {
  if (!events) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 6; ++i)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  int n = 0;
  const int rc = w4a4_impl(x, gate_w, bias, w, T, H, E, I, top_k, out, topk_idx, topk_w, workspace,
                           workspace_bytes, stream, events, &n);
  if (kernels_launched) *kernels_launched = n;
  return rc;
}

int moe_nvfp4_tc_scales(const uint8_t* scales, int E, int rows, int K, int gate_up, uint8_t* out, void* stream) {
  if (E <= 0 || rows <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (rows % 128 != 0 || K % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (gate_up && rows % 256 != 0) return MOE_ERR_UNSUPPORTED;
  MOE_TRY(check_ptr(scales));
  MOE_TRY(check_ptr(out));
  MOE_TRY(check_device(nullptr));
  return cuda_status(launch_tc_scales(scales, E, rows, K, gate_up != 0, out, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_nvfp4_quantize(const uint16_t* a, int R, int K, float global, uint8_t* codes, uint8_t* scales,
                       void* stream) {
  if (R < 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (K % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (!(global > 0.0f) || !(global < 3.0e38f)) return MOE_ERR_INVALID_ARG;
  if (R == 0) return MOE_OK;
  MOE_TRY(check_ptr(a));
  MOE_TRY(check_ptr(codes));
  MOE_TRY(check_ptr(scales));
  MOE_TRY(check_device(nullptr));
  return cuda_status(launch_quant_plain(a, R, K, global, codes, scales, nullptr,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int moe_debug_force_wait_timeout(int polls) {
  if (polls < 0) return MOE_ERR_INVALID_ARG;
  moe::g_debug_spin.store(polls);
  moe::g_debug_force.store(polls > 0 ? 1 : 0);
  return MOE_OK;
}

int moe_read_status(const void* workspace, void* stream) {
  if (!workspace) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  int st = 0;
  if (cudaMemcpy(&st, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (st & kStatusTimeout) return MOE_ERR_DEVICE_TIMEOUT;
  if (st & (kStatusBadExpert | kStatusRange | kStatusBounds)) return MOE_ERR_DEVICE;
  return MOE_OK;
}

int moe_read_diagnostics(const void* workspace, void* stream, int32_t* out4) {
  if (!workspace || !out4) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  WsHeader h;
  if (cudaMemcpy(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  out4[0] = h.num_active;
  out4[1] = h.num_large;
  out4[2] = h.router_flagged;
  out4[3] = h.router_fallback;
  return MOE_OK;
}

}  // extern "C"
