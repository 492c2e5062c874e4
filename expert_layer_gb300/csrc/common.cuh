// Shared device helpers and the workspace layout of the MoE layer library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// ----------------------------------------------------------------- status
// Bits of the device status word kept in the workspace header.
enum : int {
  kStatusBadExpert = 1,   // moe_permute saw an expert id outside [0, E)
  kStatusTimeout = 2,     // a bounded device-side wait gave up
  kStatusRange = 4,       // NVFP4 path: an activation (x or h) beyond the f16 range
  kStatusBounds = 8,      // MOE_DEBUG_BOUNDS builds: an index read from a device array was out of range
};

// Index checks of MOE_DEBUG_BOUNDS builds.  Every index that an expert-GEMM,
// gather or quantiser kernel reads from a device array (the slot
// permutation, the flat expert ids, group offsets and counts) is checked
// before it addresses memory; a bad one is recorded as kStatusBounds
// (MOE_ERR_DEVICE for moe_read_status) and replaced by a safe index by the
// caller.  Normal builds compile the checks away.
#ifdef MOE_DEBUG_BOUNDS
__device__ __forceinline__ bool bounds_ok(bool ok, int* status) {
  if (!ok) atomicOr(status, kStatusBounds);
  return ok;
}
#else
__device__ __forceinline__ bool bounds_ok(bool, int*) { return true; }
#endif

// Workspace header (first 256 bytes of every workspace).
struct WsHeader {
  int status;             // OR of kStatus* bits
  int num_active;         // experts with at least one routed slot
  int num_large;          // active experts served by the tensor-core path
  int router_flagged;     // tokens whose ranking needed fp64 logits
  int router_fallback;    // tokens that needed fp64 logits for every expert
  int pad[59];
};
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte slot");

// Offsets (bytes) of every workspace region for one shape.
struct WsLayout {
  size_t hdr, sched, cnt, xnorm, wnorm, logits, logits64, lpart, xsq, idx, w, counts, offsets, active, tiles, blk_cnt,
      blk_base, lrank, perm, inv_perm, h, partial, xp, x16, acnt, total;
  int nblk;               // 512-slot blocks of the grouping kernels
  bool partial_f32;       // fp32 partials (else bf16)
};

constexpr int kPermBlock = 512;            // slots per grouping block

// Large batches route through the tiled logits kernel (stream-K over token
// blocks and K chunks; a block's partial logits come in at most
// kRouteTilePieces pieces, each with its partial ||x_t||^2).
constexpr int kRouteTilePieces = 4;
constexpr long long kRouteTileMaxE = 128;
inline bool route_tiled(long long T, long long E) { return T >= 2048 && E <= kRouteTileMaxE; }
constexpr size_t kPartialF32Limit = 32ull << 20;

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

inline WsLayout make_layout(long long T, long long H, long long E, long long I, long long k) {
  WsLayout L{};
  const long long S = T * k;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = align256(o + bytes); return r; };
  L.nblk = (int)((S + kPermBlock - 1) / kPermBlock);
  L.partial_f32 = (size_t)S * (size_t)H * 4 <= kPartialF32Limit;
  L.hdr = take(sizeof(WsHeader));
  // expert-GEMM queue counter, per-slot counters, the fused combine's counter
  L.sched = take(sizeof(int) * (E + 2));
  L.cnt = take(sizeof(int) * T);
  L.acnt = take(sizeof(int) * E);          // per-expert slot counters (ranks by arrival)
  L.xnorm = take(sizeof(float) * T);
  L.wnorm = take(sizeof(float) * E);
  L.logits = take(sizeof(float) * T * E);
  L.logits64 = take(sizeof(double) * T * E);
  const bool tiled = route_tiled(T, E);   // the tiled router's pieces
  L.lpart = take(tiled ? sizeof(float) * kRouteTilePieces * T * E : 0);
  L.xsq = take(tiled ? sizeof(float) * kRouteTilePieces * T : 0);
  L.idx = take(sizeof(int) * S);
  L.w = take(sizeof(float) * S);
  L.counts = take(sizeof(int) * E);
  L.offsets = take(sizeof(int) * (E + 1));
  L.active = take(sizeof(int) * E);
  L.tiles = take(sizeof(int) * (2 * E + 2));
  L.blk_cnt = take(sizeof(int) * (size_t)L.nblk * E);
  L.blk_base = take(sizeof(int) * (size_t)L.nblk * E);
  L.lrank = take(sizeof(int) * S);
  L.perm = take(sizeof(int) * S);
  L.inv_perm = take(sizeof(int) * S);
  L.h = take(sizeof(uint16_t) * S * I);
  L.partial = take((L.partial_f32 ? 4 : 2) * (size_t)S * H);
  // token rows in grouped order (bf16 tensor-core path), or the W4A4 path's
  // NVFP4 activations: codes [S, H/2] and [S, I/2] and their block scales in
  // 128-row blocks per expert (at most S/128 + E + 1 blocks)
  const size_t fp4 = (size_t)S * (H + I) / 2 + (size_t)(S / 128 + E + 1) * (size_t)((H + I) / 64) * 512 + 4 * 256;
  const size_t xp = sizeof(uint16_t) * (size_t)S * H;
  L.xp = take(xp > fp4 ? xp : fp4);
  L.x16 = take(sizeof(uint16_t) * (size_t)T * H);  // x in f16 (NVFP4 path)
  L.total = o;
  return L;
}

// Bytes at the start of the workspace that must be zero when a call starts
// (header, scheduling counters, per-chunk and per-expert counters); every
// entry point clears them on its stream.
inline size_t zeroed_prefix(const WsLayout& L) { return L.xnorm; }

template <typename T>
__host__ __device__ inline T* ws_ptr(void* ws, size_t off) {
  return reinterpret_cast<T*>(reinterpret_cast<char*>(ws) + off);
}

// ----------------------------------------------------------------- numerics
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint16_t f2bf(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)f2bf(lo) | ((uint32_t)f2bf(hi) << 16);
}

// silu(z) = z / (1 + e^-z) with the hardware exponential and an approximate
// division: relative error of a few 1e-7, far below the bf16 (or f16, or
// NVFP4) rounding that h receives next; for z < -87 the quotient is 0.
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// mma.sync m16n8k16, bf16 inputs, fp32 accumulate (in place).
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same MMA with f16 operands (NVFP4 path).
__device__ __forceinline__ void mma_f16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// f16 bits of a float, round to nearest even (|f| >= 65520 gives infinity)
__device__ __forceinline__ uint16_t f2h(float f) {
  uint16_t h;
  asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(f));
  return h;
}

// Eight bf16 (a 16-byte vector) to eight f16, round to nearest even; `bad`
// is set when a value rounds beyond the f16 range (or is not finite).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v, bool& bad) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint16_t lo = f2h(__uint_as_float(w[j] << 16)), hi = f2h(__uint_as_float(w[j] & 0xffff0000u));
    bad |= ((lo & 0x7c00u) == 0x7c00u) | ((hi & 0x7c00u) == 0x7c00u);
    o[j] = (uint32_t)lo | ((uint32_t)hi << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Programmatic dependent launch: wait until the grids this one depends on have
// completed and their writes are visible (a no-op for a normal launch), and
// allow the next kernel in the stream to start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch as a programmatic dependent of the previous kernel on the stream:
// the grid may be set up and become resident before its predecessor ends.
// Every kernel launched this way calls pdl_wait() before it touches any data
// (its own or its predecessors'), so the stream order of results holds.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

__device__ __forceinline__ void set_status(void* ws, int bit) {
  atomicOr(&reinterpret_cast<WsHeader*>(ws)->status, bit);
}

}  // namespace moe
