// Host-side launchers of the MoE layer kernels (one translation unit each).
// Every launcher only enqueues on `stream`, adds the number of kernels it
// launched to *launches (if non-null) and returns the launch error.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

// Outputs of the grouping when it runs fused into the small-batch router.
// Grouping fused into the small-batch router: each routed slot f takes its
// rank within its expert's group, rank[f] = atomicAdd(&acnt[idx[f]], 1)
// (arrival order; acnt starts at zero).  The expert kernel builds offsets,
// active list and permutation from acnt, idx and rank (self_group below).
struct GroupOut {
  int* acnt;     // [E] slot counts, zero at launch
  int* rank;     // [S] out
};

// moe_api.cu -- test-only settings of the bounded device waits (0, 0 in
// normal use; moe_debug_force_wait_timeout)
struct DebugWaits {
  int spin_limit;   // polls before a wait gives up (0: the default)
  int force;        // nonzero: waits aim at a count no unit reaches
};
DebugWaits debug_waits();

// moe_api.cu -- clears the first `bytes` (a multiple of 16) of the workspace;
// lets the next kernel (a programmatic dependent) start launching at once
cudaError_t launch_zero(void* ws, size_t bytes, cudaStream_t stream);

// router.cu -- logits, certified top-k, renormalised weights; with `group`
// (only where route_can_group) also the grouping, in the same launch; with
// x16 also x converted to f16 ([T, H], for the decoded-weight expert
// kernels; a value beyond the f16 range sets kStatusRange)
bool route_can_group(int T, int E, int k);
cudaError_t launch_route(const uint16_t* x, const uint16_t* gate_w, const float* bias, int T, int H,
                         int E, int k, int32_t* idx, float* w, void* ws, const WsLayout& L,
                         cudaStream_t stream, int* launches, const GroupOut* group,
                         uint16_t* x16 = nullptr);

// permute.cu -- histogram, exclusive scan, stable permutation, active list
cudaError_t launch_permute(const int32_t* idx, int T, int E, int k, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv_perm, void* ws,
                           const WsLayout& L, int large_threshold, int tile_rows,
                           cudaStream_t stream, int* launches);

// stream_gemm.cu -- weight-streaming grouped GEMV/GEMM (mma.sync), bf16 or NVFP4 weights
struct StreamGemmArgs {
  // common
  int T, H, E, I, k;
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* perm;
  const int32_t* active;     // active experts (ascending)
  const int* num_active;     // device scalar
  const int* num_large;      // device scalar: leading active experts served elsewhere (may be null)
  // gate/up
  const uint16_t* x;         // [T, H]
  const uint16_t* x16;       // [T, H] x in f16 (NVFP4 path)
  const uint16_t* w_gate_up; // [E, 2I, H] bf16 (or null)
  const uint8_t* gu_codes;   // NVFP4 (or null)
  const uint8_t* gu_scales;
  const float* gu_global;
  const int8_t* gu_q8;       // int8 block weights [E, 2I, H] (or null)
  const uint16_t* gu_q8s;    // their fp16 scales [E, 2I, H/32]
  uint16_t* h;               // [S, I] grouped order: bf16, or f16 on the NVFP4 and int8 paths
  // down
  const uint16_t* w_down;    // [E, H, I]
  const uint8_t* dn_codes;
  const uint8_t* dn_scales;
  const float* dn_global;
  const int8_t* dn_q8;       // [E, H, I]
  const uint16_t* dn_q8s;    // [E, H, I/32]
  const float* topk_w;       // [S]
  void* partial;             // [S, H] fp32 or bf16, slot order
  bool partial_f32;
  // scheduling (zero at launch): unit queue ticket counter and, per active
  // slot, the number of gate/up units whose h rows are published
  int* queue;
  int* dep;
  int* status;               // workspace status word (kStatusTimeout)
  int num_sms;
  // self-grouping (small batches: the router leaves arrival ranks instead of
  // a grouping): every CTA builds the active list, offsets and permutation
  // from acnt / idx / rank in its prologue, and CTA 0 also writes them to
  // counts / offsets / active / perm / inv_perm and the header (diagnostics)
  bool self_group;
  const int* acnt;           // [E]
  const int32_t* idx;        // [S] expert of each routed slot
  const int* rank;           // [S]
  int32_t* counts_out;
  int32_t* offsets_out;      // [E + 1]
  int32_t* active_out;
  int32_t* perm_out;
  int32_t* inv_perm_out;
  int* num_active_out;
  int* num_large_out;
  // fused combine (every group on this kernel): after its units each CTA
  // arrives on *done and waits for all CTAs (all are resident), then sums its
  // slice of out[t] = sum_s partial[t*k + s] in slot order
  bool fused_combine;
  int* done;                 // zero at launch
  uint16_t* out;             // [T, H] bf16
  // bounded waits: polls before a down unit's wait gives up; with
  // wait_extra > 0 the wait aims at a count that no unit reaches (test-only
  // forced timeout, see moe_debug_force_wait_timeout)
  int spin_limit;
  int wait_extra;
};
// gate/up then down of the small groups, one persistent launch
cudaError_t launch_stream_gemm(const StreamGemmArgs& a, cudaStream_t stream, int* launches);
// the same for NVFP4 / int8 weights with a TMA producer warp (stream_dec.cu);
// stream_dec_supported: decoded weights and H, I multiples of 256
bool stream_dec_supported(const StreamGemmArgs& a);
cudaError_t launch_stream_dec(const StreamGemmArgs& a, cudaStream_t stream);
// tc_gemm.cu -- tcgen05/TMEM grouped GEMMs for experts with many rows (bf16 weights)
struct TcLaunch {
  int T, H, E, I, k;
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* perm;
  const int32_t* active;     // small-group experts first, then the large ones
  const int32_t* tiles;      // m-tile prefix over the large experts
  const int* num_active;
  const int* num_large;
  const uint16_t* x;
  uint16_t* xp;              // [S, H] scratch: token rows in grouped order
  const uint16_t* w_gate_up;
  const uint16_t* w_down;
  const float* topk_w;
  uint16_t* h;
  void* partial;
  bool partial_f32;
  int* status;
  int num_sms;
};
constexpr int kTcRows = 128;             // token rows per tensor-core tile
cudaError_t launch_tc_gemm(const TcLaunch& p, bool down, cudaStream_t stream, int* launches);

// tc_gemm.cu -- xp[r] = x[perm[r] / k]: token rows in grouped order
cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* perm, int S, int H, int k,
                               uint16_t* xp, int* status, cudaStream_t stream, int* launches);

// tc_fp4.cu -- W4A4: NVFP4 weights x NVFP4 activations on the block-scaled
// tensor cores (tcgen05 kind::mxf4nvf4)
struct Fp4Launch {
  int T, H, E, I, k;
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* perm;
  const int32_t* active;     // active experts, ascending (all served here)
  const int* num_active;
  const uint8_t* gu_codes;   // [E, 2I, H/2]
  const uint8_t* gu_scales_tc;
  const float* gu_global;
  const uint8_t* dn_codes;   // [E, H, I/2]
  const uint8_t* dn_scales_tc;
  const float* dn_global;
  const float* x_global;     // [E]
  const float* h_global;     // [E]
  const uint8_t* xq;         // [S, H/2] token-row codes, grouped order
  const uint8_t* xs;         // token-row scales, tensor-core layout
  const uint8_t* hq;         // [S, I/2]
  const uint8_t* hs;
  const float* topk_w;
  uint16_t* h;               // [S, I] bf16
  void* partial;
  bool partial_f32;
  int* status;
  int num_sms;
};
// bytes of the activation scales of S routed rows over E experts (128-row
// blocks of each expert) for contraction length K
inline size_t fp4_act_scale_bytes(long long S, long long E, long long K) {
  return (size_t)(S / 128 + E + 1) * (size_t)(K / 64) * 512;
}
cudaError_t launch_quant_rows(bool gather, const uint16_t* src, const int32_t* perm, const int32_t* idx, int k,
                              const int32_t* counts, const int32_t* offsets, int S, int K, int E,
                              const float* glob, uint8_t* codes, uint8_t* sf, int* status, cudaStream_t stream,
                              int* launches);
cudaError_t launch_quant_plain(const uint16_t* src, int R, int K, float g, uint8_t* codes, uint8_t* scales,
                               int* flag, cudaStream_t stream);
cudaError_t launch_tc_scales(const uint8_t* in, int E, int R, int K, bool interleave, uint8_t* out,
                             cudaStream_t stream);
cudaError_t launch_tc_fp4(const Fp4Launch& p, bool down, cudaStream_t stream, int* launches);

// combine.cu -- out[t] = sum_s partial[t*k+s] in slot order
cudaError_t launch_combine(const void* partial, bool partial_f32, int T, int H, int k,
                           uint16_t* out, int num_sms, cudaStream_t stream, int* launches);

}  // namespace moe
