/*
 * moe.h -- C ABI of libmoe_gb300.so: the forward pass of a Mixture-of-Experts
 * FFN layer (router, expert grouping, grouped SwiGLU experts, combine) on one
 * NVIDIA GB300 GPU (sm_103a).
 *
 * The layer follows the phases that the serving worklogs time inside the
 * fused-MoE path -- "MoE gate", then "topk, expert kernel, activation, sum"
 * (page "Decode 吞吐专项实验分析报告", section "下一步 profiling 方向",
 * items 2-3) -- with the expert grouping done on the device, never returning
 * to the host per layer (page "第 9 章 prefill：最大的瓶颈", sec. 9.9, fused
 * path vs. the per-layer cudaStreamSynchronize of the MMQ path), and with no
 * per-expert row ceiling (sec. 9.5 records entries beyond GMAX = 8 per group
 * being dropped; here no routed row is ever dropped).
 *
 * Notation: T tokens, H hidden size, E experts, k = top_k, I expert
 * intermediate size, S = T*k routed slots, flat slot index f = t*k + s.
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers unless stated otherwise; bf16 tensors are
 *     passed as uint16_t bit patterns; all tensors are dense row-major.
 *   - Every device pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     only enqueue work on `stream`: no host synchronisation, no allocation,
 *     no global state.  Concurrent calls need distinct workspaces.
 *   - The caller owns every buffer.  `workspace` is scratch device memory of
 *     at least moe_workspace_size(...) bytes; its contents on entry do not
 *     matter.
 *   - Return value: MOE_OK (0) or a negative moe_status.  Argument errors are
 *     detected on the host before anything is enqueued.  Errors found by the
 *     kernels (e.g. an out-of-range expert id handed to moe_permute) are
 *     recorded in the workspace and reported by moe_read_status.  No kernel
 *     traps.
 *   - T == 0 is a valid empty batch: nothing is enqueued and MOE_OK returned.
 *
 * Supported shapes: 1 <= E <= 1024, 1 <= top_k <= min(E, 32), H and I
 * multiples of 128 (NVFP4: H and I multiples of 128 as well), T*top_k < 2^31.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,    /* null pointer, negative size, top_k out of range   */
  MOE_ERR_UNSUPPORTED = -2,    /* shape outside the supported set, misaligned
                                  pointer, device is not sm_103                      */
  MOE_ERR_WORKSPACE = -3,      /* workspace_bytes < moe_workspace_size(...)          */
  MOE_ERR_CUDA = -4,           /* a CUDA runtime call or kernel launch failed        */
  MOE_ERR_DEVICE = -5,         /* a kernel found invalid data, e.g. an NVFP4-path
                                  activation beyond the f16 range (moe_read_status) */
  MOE_ERR_DEVICE_TIMEOUT = -6  /* a bounded device-side wait gave up (moe_read_status) */
} moe_status;

/*
 * NVFP4 expert weights (W4A16: weights in 4 bits, activations stay bf16).
 * Element W[e,r,k] = e2m1(code) * e4m3(scale[e,r,k/16]) * global[e], with
 * e2m1 per OCP Microscaling Formats v1.0 (FP4 E2M1) and e4m3 per the OCP
 * 8-bit floating point specification.  The NVFP4 deployment on the pages is
 * the 176B MoE served through the "nvfp4-sm80" graft (page "vLLM 0.32
 * 升级试验：TEP2 prefill 诅咒解除 + decode 本机纪录", header and "背景与动机").
 *
 *   gu_codes  [E, 2I, H/2] uint8, two codes per byte, even k in the low nibble
 *   gu_scales [E, 2I, H/16] uint8 e4m3 bit patterns, 16-element blocks along H
 *   gu_global [E] fp32
 *   dn_codes  [E, H, I/2], dn_scales [E, H, I/16], dn_global [E]: same for w_down
 * Rows [0, I) of the gate/up tensor are the gate projection, rows [I, 2I) the
 * up projection.  All pointers are device pointers.
 * The expert products run on f16 operands: the decoded weights are exact in
 * f16, and the activations (x, and the SwiGLU output h) are converted to f16,
 * which is exact for magnitudes 2^-14 .. 65504; smaller ones round to the
 * f16 subnormal grid (absolute error <= 2^-25), larger ones are recorded as
 * MOE_ERR_DEVICE for moe_read_status (the output is then unspecified).
 */
typedef struct {
  const uint8_t *gu_codes;
  const uint8_t *gu_scales;
  const float *gu_global;
  const uint8_t *dn_codes;
  const uint8_t *dn_scales;
  const float *dn_global;
} moe_nvfp4_weights;

/* Bytes of device workspace that moe_route, moe_permute and moe_forward need
 * for this shape (the largest of the three).  Returns 0 for an invalid shape. */
size_t moe_workspace_size(int T, int H, int E, int I, int top_k);

/*
 * Router: "MoE gate" + "topk" (page "Decode 吞吐专项实验分析报告", section
 * "下一步 profiling 方向").
 *   logit[t,e] = sum_h x[t,h]*gate_w[e,h] (+ bias[e])
 *   experts ranked by logit, larger first, lower index first on equal logits;
 *   topk_idx[t,s] = expert in rank s (s = 0..k-1)
 *   topk_w[t,s]   = exp(logit_s) / sum_{s'<k} exp(logit_s')  (the softmax over
 *                   all E experts renormalised over the k selected ones)
 * Logits accumulate in fp32 with a rigorous per-token error bound; a token
 * whose ranking the bound cannot certify has its contested logits recomputed
 * in fp64, so topk_idx equals the ranking of the exact logits.
 *
 *   x       [T, H] bf16          gate_w [E, H] bf16
 *   bias    [E] fp32 or NULL     (added to the logits before softmax/top-k)
 *   topk_idx [T, k] int32 (out)  topk_w [T, k] fp32 (out)
 */
int moe_route(const uint16_t *x, const uint16_t *gate_w, const float *bias, int T, int H, int E,
              int top_k, int32_t *topk_idx, float *topk_w, void *workspace,
              size_t workspace_bytes, void *stream);

/*
 * Expert grouping of the routed slots (done on the device, page "第 9 章
 * prefill：最大的瓶颈", sec. 9.9, fused path):
 *   counts[e]   = number of slots f with topk_idx[f] == e
 *   offsets[e]  = sum_{e' < e} counts[e'],   offsets[E] = S      ([E+1])
 *   perm[r]     = the slot f at grouped position r: slots sorted by expert,
 *                 ascending f within an expert (a stable sort)       ([S])
 *   inv_perm[f] = r such that perm[r] == f                           ([S])
 * topk_idx is [T, k] int32 (device).  Entries outside [0, E) are skipped and
 * recorded as MOE_ERR_DEVICE for moe_read_status; the outputs are then
 * unspecified.
 */
int moe_permute(const int32_t *topk_idx, int T, int E, int top_k, int32_t *counts,
                int32_t *offsets, int32_t *perm, int32_t *inv_perm, void *workspace,
                size_t workspace_bytes, void *stream);

/*
 * The whole layer: route, group, per-expert SwiGLU, combine.
 *   g   = W_gate[e] x_t,  u = W_up[e] x_t       (rows [0,I) / [I,2I) of w_gate_up[e])
 *   h   = silu(g) * u,    silu(z) = z / (1 + exp(-z))      (rounded to bf16)
 *   y   = W_down[e] h
 *   out[t] = sum_{s=0..k-1} topk_w[t,s] * y[t,s]   summed in s order in fp32,
 *            rounded to bf16 -- no float atomics, so the result is
 *            bitwise deterministic and independent of token order.
 *
 *   x [T, H] bf16; gate_w [E, H] bf16; bias [E] fp32 or NULL
 *   w_gate_up [E, 2I, H] bf16, w_down [E, H, I] bf16 -- both NULL iff nvfp4
 *   nvfp4     NULL for bf16 weights, else the NVFP4 weights (host struct
 *             holding device pointers)
 *   out [T, H] bf16 (out)
 *   topk_idx / topk_w: optional [T, k] outputs (NULL to skip) receiving the
 *             routing that this call used.
 */
int moe_forward(const uint16_t *x, const uint16_t *gate_w, const float *bias,
                const uint16_t *w_gate_up, const uint16_t *w_down,
                const moe_nvfp4_weights *nvfp4, int T, int H, int E, int I, int top_k,
                uint16_t *out, int32_t *topk_idx, float *topk_w, void *workspace,
                size_t workspace_bytes, void *stream);

/*
 * moe_forward with timing hooks, for benchmarks and profilers: identical
 * arguments and results, and additionally records events[i] (cudaEvent_t,
 * created by the caller) on `stream` at the stage boundaries
 *   [0] start  [1] after routing  [2] after grouping
 *   [3] after the weight-streaming expert kernel (gate/up, SwiGLU and down of
 *       the experts with few rows, one launch; when no expert goes to the
 *       tensor-core kernels it also does the combine)
 *   [4] after the tensor-core expert kernels (gate/up+SwiGLU, then down, of
 *       the experts with many rows; none for small batches)  [5] after combine
 * and stores in *kernels_launched (HOST pointer, may be NULL) the number of
 * kernels this call launched.  `events` is a HOST array of 6 non-null events.
 */
int moe_forward_profiled(const uint16_t *x, const uint16_t *gate_w, const float *bias,
                         const uint16_t *w_gate_up, const uint16_t *w_down,
                         const moe_nvfp4_weights *nvfp4, int T, int H, int E, int I, int top_k,
                         uint16_t *out, int32_t *topk_idx, float *topk_w, void *workspace,
                         size_t workspace_bytes, void *stream, void *const *events,
                         int32_t *kernels_launched);

/*
 * Synchronises `stream`, then reports what the kernels of the last call that
 * used `workspace` recorded: MOE_OK, MOE_ERR_DEVICE or MOE_ERR_DEVICE_TIMEOUT.
 * `workspace` must have been passed to a moe_* call before.
 */
int moe_read_status(const void *workspace, void *stream);

/*
 * Synchronises `stream` and copies four counters of the last call that used
 * `workspace` into the HOST array out4: [0] active experts, [1] active experts
 * served by the tensor-core path, [2] tokens whose top-k needed fp64 logits,
 * [3] tokens that needed fp64 logits for every expert.  Diagnostics only.
 */
int moe_read_diagnostics(const void *workspace, void *stream, int32_t *out4);

/*
 * moe_route without a workspace, for callers that cannot allocate device
 * memory (code running under CUDA graph capture, runtimes that hand out only
 * pre-reserved pool memory, host integrations that forbid allocation after
 * start-up).  The pages describe no such entry point; it is an addition of
 * this library.  Same arguments and results as moe_route minus the
 * workspace; allocates nothing.
 *
 * Its scratch is a fixed device array inside the library (about 0.8 MB, held
 * on every GPU that loads the library until the process exits), so it serves
 * only T*E <= 65536 and T <= 8192; larger batches return MOE_ERR_UNSUPPORTED.
 * The first call on a device looks up the array's device address (make that
 * call before any stream capture) and keeps it for the life of the process:
 * after cudaDeviceReset the address is stale, so do not call this entry point
 * again on a device that was reset.  All calls on a device share the array:
 * calls whose GPU work overlaps (unordered streams) race and give undefined
 * results.  Device-side status is not reported (there is no workspace to
 * pass to moe_read_status).
 */
int moe_route_noalloc(const uint16_t *x, const uint16_t *gate_w, const float *bias, int T, int H,
                      int E, int top_k, int32_t *topk_idx, float *topk_w, void *stream);

/*
 * ------------------------------------------------------------------ W4A4
 * NVFP4 weights AND NVFP4 activations on the block-scaled tensor cores
 * (e2m1 x e2m1 products, one e4m3 scale per 16 elements along K on both
 * operands, fp32 accumulate).  The pages' NVFP4 deployment is the 176B MoE of
 * page "vLLM 0.32 升级试验：TEP2 prefill 诅咒解除 + decode 本机纪录" (header,
 * "背景与动机"); the pages give no activation numerics, so the activations are
 * quantised with the format's own recipe, per routed row of expert e:
 *   16-element blocks along K (H for the token rows, I for h),
 *   block scale  s = e4m3(amax / (6 G))           round to nearest even, <= 448
 *   element code   = e2m1(v * r), r = 1 / (s G)  round to nearest even, |.| <= 6
 *   (0 for every element of a block whose s G is 0)
 * with G = x_global[e] for the token rows and G = h_global[e] for the SwiGLU
 * output h = bf16(silu(g) * u); every quotient, reciprocal and product in
 * fp32 with IEEE rounding.  Then g, u = dequant(W_gu) dequant(x_q), y = dequant(W_dn)
 * dequant(h_q), and the combine as in moe_forward.
 *
 * Weights: codes and globals as in moe_nvfp4_weights; the block scales in the
 * tensor-core layout written by moe_nvfp4_tc_scales (done once, when the
 * weights are loaded).  x_global, h_global: [E] fp32, positive and finite
 * (device pointers), the activations' NVFP4 global scales (as NVFP4
 * checkpoints store calibrated input scales).
 * Shapes: H and I multiples of 256.  The output is out [T, H] bf16; an
 * activation that is not finite is recorded as MOE_ERR_DEVICE.
 */
typedef struct {
  const uint8_t *gu_codes;      /* [E, 2I, H/2] */
  const uint8_t *gu_scales_tc;  /* moe_nvfp4_tc_scales(gu_scales, E, 2I, H, 1, ...) */
  const float *gu_global;       /* [E] */
  const uint8_t *dn_codes;      /* [E, H, I/2] */
  const uint8_t *dn_scales_tc;  /* moe_nvfp4_tc_scales(dn_scales, E, H, I, 0, ...) */
  const float *dn_global;       /* [E] */
  const float *x_global;        /* [E] */
  const float *h_global;        /* [E] */
} moe_w4a4_weights;

/*
 * Rearranges NVFP4 block scales [E, rows, K/16] (row-major e4m3 bytes, as in
 * moe_nvfp4_weights) into the layout the W4A4 tensor-core kernels read: for
 * each block of 128 rows and each 64-wide step of K, a 512-byte atom of 32
 * rows x 16 bytes whose row i, bytes 4j..4j+3, holds the 4 scales of row
 * i + 32j; atoms ordered by (row block, K step).  With gate_up != 0 the
 * tensor is w_gate_up's (rows = 2I) and the rows of each 128-row block are
 * gate and up rows interleaved: row 2jj is gate row j0 + jj, row 2jj+1 up row
 * I + j0 + jj (j0 = 64 * block).  `out` has the same size as `scales`
 * (E * rows * K / 16 bytes).  rows % 128 == 0 (gate_up: % 256), K % 64 == 0.
 * Enqueues on `stream`.
 */
int moe_nvfp4_tc_scales(const uint8_t *scales, int E, int rows, int K, int gate_up, uint8_t *out,
                        void *stream);

/*
 * The W4A4 layer forward (see above).  Arguments as moe_forward, with the
 * W4A4 weights in place of the bf16 / NVFP4 ones; workspace of
 * moe_workspace_size(T, H, E, I, top_k) bytes.
 */
int moe_forward_w4a4(const uint16_t *x, const uint16_t *gate_w, const float *bias,
                     const moe_w4a4_weights *w, int T, int H, int E, int I, int top_k, uint16_t *out,
                     int32_t *topk_idx, float *topk_w, void *workspace, size_t workspace_bytes,
                     void *stream);

/*
 * moe_forward_w4a4 with timing hooks, as moe_forward_profiled; the events
 * mark [0] start [1] routing [2] grouping [3] token rows quantised
 * [4] gate/up, h quantised, down [5] combine.
 */
int moe_forward_w4a4_profiled(const uint16_t *x, const uint16_t *gate_w, const float *bias,
                              const moe_w4a4_weights *w, int T, int H, int E, int I, int top_k,
                              uint16_t *out, int32_t *topk_idx, float *topk_w, void *workspace,
                              size_t workspace_bytes, void *stream, void *const *events,
                              int32_t *kernels_launched);

/*
 * The activation quantiser of the W4A4 path on its own: rows a [R, K] (bf16)
 * with one global G -> codes [R, K/2] (two e2m1 codes per byte, even k in the
 * low nibble) and scales [R, K/16] (e4m3, row-major).  K % 64 == 0, G > 0.
 */
int moe_nvfp4_quantize(const uint16_t *a, int R, int K, float global, uint8_t *codes, uint8_t *scales,
                       void *stream);

/*
 * Int8 block expert weights (W8A16): the "fused int8" expert types of the
 * pages' serving stack (page "第 9 章 prefill：最大的瓶颈", sec. 9.9), taken as
 * the plain int8 block format -- one signed 8-bit code per element and one
 * fp16 scale per 32 consecutive elements along K:
 *   W[e,r,k] = code[e,r,k] * scale[e,r,k/32]
 *   gu_codes  [E, 2I, H] int8     gu_scales [E, 2I, H/32] fp16 bit patterns
 *   dn_codes  [E, H, I] int8      dn_scales [E, H, I/32]  fp16 bit patterns
 * Rows [0, I) of the gate/up tensor are the gate projection, rows [I, 2I) the
 * up projection.  All pointers are device pointers, 16-byte aligned.
 * The expert products run on f16 operands as on the NVFP4 path (codes exact
 * in f16; x and h converted to f16, out-of-range values recorded as
 * MOE_ERR_DEVICE); every expert, whatever its row count, takes the
 * weight-streaming kernel.
 */
typedef struct {
  const int8_t *gu_codes;
  const uint16_t *gu_scales;
  const int8_t *dn_codes;
  const uint16_t *dn_scales;
} moe_int8_weights;

/*
 * The layer forward with int8 block expert weights: arguments and results as
 * moe_forward, with `w` (host struct holding device pointers) in place of the
 * bf16 / NVFP4 weights; workspace of moe_workspace_size(T, H, E, I, top_k)
 * bytes.
 */
int moe_forward_int8(const uint16_t *x, const uint16_t *gate_w, const float *bias,
                     const moe_int8_weights *w, int T, int H, int E, int I, int top_k, uint16_t *out,
                     int32_t *topk_idx, float *topk_w, void *workspace, size_t workspace_bytes,
                     void *stream);

/*
 * moe_forward_int8 with the timing hooks of moe_forward_profiled (same six
 * events; [4] follows [3] directly: no tensor-core stage).
 */
int moe_forward_int8_profiled(const uint16_t *x, const uint16_t *gate_w, const float *bias,
                              const moe_int8_weights *w, int T, int H, int E, int I, int top_k,
                              uint16_t *out, int32_t *topk_idx, float *topk_w, void *workspace,
                              size_t workspace_bytes, void *stream, void *const *events,
                              int32_t *kernels_launched);

/*
 * TEST ONLY.  With polls > 0, every moe_forward launched afterwards in this
 * process makes the weight-streaming kernel's bounded waits (a down-
 * projection unit waiting for its expert's gate/up units) aim at a count
 * that no unit ever reaches and give up after `polls` polls: the call then
 * completes, its output is unspecified, and moe_read_status reports
 * MOE_ERR_DEVICE_TIMEOUT.  polls == 0 restores normal operation (the
 * default).  Process-wide setting, not thread-safe with concurrent calls;
 * it exists so that tests can exercise the timeout path without a hung or
 * faulted GPU.
 */
int moe_debug_force_wait_timeout(int polls);

/* Static, human-readable name of a moe_status value. */
const char *moe_error_string(int status);

/* Version of this library as an integer (major*10000 + minor*100 + patch). */
int moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
