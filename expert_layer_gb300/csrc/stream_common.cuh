// Pieces shared by the two weight-streaming expert kernels (stream_gemm.cu:
// per-warp cp.async rings; stream_dec.cu: a TMA producer warp feeding
// decode-and-mma warps): the unit queue, copy and ordering primitives and
// the int8 code decoding.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace stream {
namespace {  // internal linkage: each translation unit gets its own copy

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(d), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

namespace q8 {
// Four int8 codes (byte i = element i) to two f16x2 pairs, exact: each byte,
// offset by 128 with the sign-bit flip, becomes the mantissa of the f16
// 1024 + (q + 128) (0x64 in the high byte), and 1152 is subtracted.
__device__ __forceinline__ void s8x4_f16x2(uint32_t w, uint32_t& p01, uint32_t& p23) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t lo = __byte_perm(u, 0x64646464u, 0x4140);
  const uint32_t hi = __byte_perm(u, 0x64646464u, 0x4342);
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(p01) : "r"(lo), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(p23) : "r"(hi), "r"(0x64806480u));
}
// The f16 in the low (hf = 0) or high half of v, as fp32 (exact).
__device__ __forceinline__ float f16_half_to_f32(uint32_t v, int hf) {
  float f;
  const uint32_t h = hf ? v >> 16 : v & 0xffffu;
  asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.f32.f16 %0, t;\n}" : "=f"(f) : "r"(h));
  return f;
}
}  // namespace q8

// Weight formats of the streaming kernel.
enum : int { kFmtBf16 = 0, kFmtFp4 = 1, kFmtQ8 = 2 };

// Bounded waits: polls before a wait gives up (and the kernel records
// kStatusTimeout); with the sleep between polls this is well over a second.
// (StreamGemmArgs.spin_limit overrides it in tests.)
constexpr int kSpinLimit = 1 << 22;

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Queue positions [0, Ug) are gate/up units, [Ug, Q) down units, each in
// active-list order (unit = a few 16-row fragments of one expert over all
// of K).
struct Queue {
  int UPEg, UPEd, Ug, Q, nkb_g, nkb_d;
};

// One unit of a warp, taken in passes of 8*NT of the expert's token rows
// (pass p covers rows 8NTp..).
struct Task {
  int q;         // queue position, < 0 when the warp has no more work
  bool down;
  int slot, e, blk, m, off, pass, npass, nkb, ngroups;
};

// Rows of the routed-slot permutation kept in shared memory (else read from
// global memory).
constexpr int kPermSmem = 4096;

template <int KG, int NT>
__device__ __forceinline__ void task_load(Task& t, const int4* smeta, const Queue& qs, int q) {
  if (q < 0 || q >= qs.Q) { t.q = -1; return; }
  t.q = q;
  t.down = q >= qs.Ug;
  const int r = t.down ? q - qs.Ug : q;
  const int upe = t.down ? qs.UPEd : qs.UPEg;
  t.slot = r / upe;
  t.blk = r - t.slot * upe;
  const int4 md = smeta[t.slot];   // expert, rows, first grouped row
  t.e = md.x;
  t.m = md.y;
  t.off = md.z;
  t.pass = 0;
  t.npass = (t.m + 8 * NT - 1) / (8 * NT);
  t.nkb = t.down ? qs.nkb_d : qs.nkb_g;
  t.ngroups = (t.nkb + KG - 1) / KG;
}

// The grouping of a small batch from the router's arrival ranks, built by
// every CTA of an expert kernel in its prologue (called by all threads; S <=
// kPermSmem).  Warp 0 turns the per-expert counts into offsets (exclusive
// prefix in expert order) and the active list smeta[0..nact) = (expert,
// rows, first grouped row), ascending; then every thread places its slots,
// sperm[offset[e] + rank[f]] = f.  Slots of one expert are thus in arrival
// order, not slot order: the output does not depend on it (each grouped row
// is computed on its own, with the same K order).  CTA 0 also writes the
// grouping to the workspace (counts, offsets, active list, permutation and
// its inverse, the header's expert counts) for diagnostics.  Returns nact.
// s_off ([E] ints) and s_nact may alias memory that the caller uses after
// the call (the final barrier orders every read of them before).
__device__ int self_group(const StreamGemmArgs& a, int4* smeta, int* sperm, int* s_off, int* s_nact) {
  const int E = a.E, S = a.T * a.k;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (E + 31) / 32, e0 = lane * per;
    int sum = 0, na = 0;
    for (int i = 0; i < per; ++i) {
      const int e = e0 + i;
      if (e < E) {
        const int v = a.acnt[e];
        sum += v;
        na += v > 0 ? 1 : 0;
      }
    }
    int ps = sum, pa = na;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int qs = __shfl_up_sync(0xffffffffu, ps, o), qa = __shfl_up_sync(0xffffffffu, pa, o);
      if (lane >= o) { ps += qs; pa += qa; }
    }
    int off = ps - sum, act = pa - na;
    const int total = __shfl_sync(0xffffffffu, ps, 31), nact = __shfl_sync(0xffffffffu, pa, 31);
    for (int i = 0; i < per; ++i) {
      const int e = e0 + i;
      if (e < E) {
        const int v = a.acnt[e];
        s_off[e] = off;
        if (v > 0) smeta[act++] = make_int4(e, v, off, 0);
        off += v;
      }
    }
    if (lane == 0) {
      *s_nact = nact;
      if (total != S) atomicOr(a.status, kStatusBadExpert);
    }
  }
  __syncthreads();
  for (int f = threadIdx.x; f < S; f += blockDim.x) {
    const int e = a.idx[f], r = a.rank[f];
    if ((unsigned)e < (unsigned)E && r >= 0) {
      const int pos = s_off[e] + r;
      if ((unsigned)pos < (unsigned)S) sperm[pos] = f;
      else atomicOr(a.status, kStatusBadExpert);
    } else {
      atomicOr(a.status, kStatusBadExpert);
    }
  }
  __syncthreads();
  const int nact = *s_nact;
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      a.counts_out[e] = a.acnt[e];
      a.offsets_out[e] = s_off[e];
    }
    for (int i = threadIdx.x; i < nact; i += blockDim.x) a.active_out[i] = smeta[i].x;
    for (int p = threadIdx.x; p < S; p += blockDim.x) {
      const int f = sperm[p];
      a.perm_out[p] = f;
      if ((unsigned)f < (unsigned)S) a.inv_perm_out[f] = p;
    }
    if (threadIdx.x == 0) {
      a.offsets_out[E] = S;
      *a.num_active_out = nact;
      *a.num_large_out = 0;
    }
  }
  __syncthreads();
  return nact;
}

// Grid-wide arrive and wait of one thread per CTA (every CTA of the launch
// is resident: persistent grids of at most one CTA per SM).  The caller has
// passed a CTA barrier after its CTA's last writes; the fence makes them
// visible device-wide before the arrive.  Bounded: false (and
// kStatusTimeout) after kSpinLimit polls.
__device__ bool grid_sync(int* ctr, int n, int* status) {
  __threadfence();
  atomicAdd(ctr, 1);
  int it = 0;
  while (ld_acquire(ctr) < n) {
    if (++it > kSpinLimit) {
      atomicOr(status, kStatusTimeout);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

// The combine after a grid_sync: vectors i = first, first + stride, ... of
// out viewed as [T][H / V] (V = 4 fp32 or 8 bf16 partials per 16 bytes);
// each sums the k partial vectors of its token in slot order from zero in
// fp32 and rounds to bf16 once -- the same arithmetic and order as the
// combine kernel.  The partials come from other CTAs: loads through L2.
__device__ void combine_slice(const StreamGemmArgs& a, long long first, long long stride) {
  const int H = a.H, k = a.k, V = a.partial_f32 ? 4 : 8;
  const long long nvec = (long long)a.T * (H / V);
  for (long long i = first; i < nvec; i += stride) {
    const long long t = i / (H / V);
    const int d = (int)(i % (H / V)) * V;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    // the slots' vectors in batches of 8, all loads of a batch issued first
    for (int s0 = 0; s0 < k; s0 += 8) {
      uint4 q[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        q[j] = make_uint4(0, 0, 0, 0);
        if (s0 + j < k) {
          const size_t row = (size_t)(t * k + s0 + j) * H + d;
          q[j] = a.partial_f32
                     ? __ldcg(reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(a.partial) + row))
                     : __ldcg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.partial) + row));
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (s0 + j >= k) break;
        const uint32_t w4[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
        if (a.partial_f32) {
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[i] += __uint_as_float(w4[i]);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) { acc[2 * i] += bf16lo(w4[i]); acc[2 * i + 1] += bf16hi(w4[i]); }
        }
      }
    }
    if (a.partial_f32) {
      *reinterpret_cast<uint2*>(a.out + (size_t)t * H + d) =
          make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]));
    } else {
      *reinterpret_cast<uint4*>(a.out + (size_t)t * H + d) =
          make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                     pack_bf16x2(acc[6], acc[7]));
    }
  }
}

}  // namespace
}  // namespace stream
}  // namespace moe
