// Shared device/host helpers of libkvc (sm_103a).  Nothing here is part of the
// public ABI; see include/kvc.h.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/kvc.h"

#define KVC_FULL_MASK 0xffffffffu

// ---------------------------------------------------------------- host side
namespace kvc {

// Device error word of the current device (address obtained once per device).
int32_t* err_word();
// Host counter of kernel launches made by this library.
void count_launch(int64_t n = 1);
// Records a CUDA runtime failure and maps it to KVC_ECUDA.
int cuda_status(cudaError_t e);
// Common validation of a parameter block.
int check_params(const kvc_params* p);
// Streaming multiprocessors of the current device (queried once per device; 0
// when the query fails).
int sm_count();
// Give-up limit (ns) of the first wait of every pipeline stage in the kernels
// with mbarrier pipelines, and whether their producers withhold their copies;
// set by kvc_set_wait_limit (defaults: kWaitNs, 0).  Drains after an abort keep
// their own limits.
uint64_t wait_limit_ns();
int withhold_copies();
constexpr uint64_t kWaitNs = 2000000000ull;

inline int64_t lh_count(const kvc_params* p) { return (int64_t)p->B * p->L * p->H; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace kvc

// ---------------------------------------------------------------- device side
namespace kvcd {

__device__ __forceinline__ void record_error(int32_t* err, int32_t code) {
  atomicCAS(err, 0, code);
}

// Element loads/stores for the two storage types.
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Loads N consecutive elements (N*sizeof(T) bytes, naturally aligned) as floats.
template <typename T, int N> struct VecLoad;
template <> struct VecLoad<__nv_bfloat16, 4> {
  static __device__ __forceinline__ void ld(const __nv_bfloat16* p, float* o) {
    uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    o[0] = __uint_as_float(u.x << 16); o[1] = __uint_as_float(u.x & 0xffff0000u);
    o[2] = __uint_as_float(u.y << 16); o[3] = __uint_as_float(u.y & 0xffff0000u);
  }
};
template <> struct VecLoad<__nv_bfloat16, 2> {
  static __device__ __forceinline__ void ld(const __nv_bfloat16* p, float* o) {
    uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(p));
    o[0] = __uint_as_float(u << 16); o[1] = __uint_as_float(u & 0xffff0000u);
  }
};
template <> struct VecLoad<float, 4> {
  static __device__ __forceinline__ void ld(const float* p, float* o) {
    float4 v = __ldg(reinterpret_cast<const float4*>(p));
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
};
template <> struct VecLoad<float, 2> {
  static __device__ __forceinline__ void ld(const float* p, float* o) {
    float2 v = __ldg(reinterpret_cast<const float2*>(p));
    o[0] = v.x; o[1] = v.y;
  }
};

// Generic-address loads of N consecutive elements as floats, for data that may
// live in shared memory (VecLoad's __ldg is for global memory only).
template <typename T, int N> struct VecLoadAny;
template <> struct VecLoadAny<__nv_bfloat16, 4> {
  static __device__ __forceinline__ void ld(const __nv_bfloat16* p, float* o) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    o[0] = __uint_as_float(u.x << 16); o[1] = __uint_as_float(u.x & 0xffff0000u);
    o[2] = __uint_as_float(u.y << 16); o[3] = __uint_as_float(u.y & 0xffff0000u);
  }
};
template <> struct VecLoadAny<__nv_bfloat16, 2> {
  static __device__ __forceinline__ void ld(const __nv_bfloat16* p, float* o) {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    o[0] = __uint_as_float(u << 16); o[1] = __uint_as_float(u & 0xffff0000u);
  }
};
template <> struct VecLoadAny<float, 4> {
  static __device__ __forceinline__ void ld(const float* p, float* o) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
};
template <> struct VecLoadAny<float, 2> {
  static __device__ __forceinline__ void ld(const float* p, float* o) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    o[0] = v.x; o[1] = v.y;
  }
};

// First token row of sequence b: sum_{b' < b} L*H*n_{b'}.
__device__ __forceinline__ int64_t seq_token_base(const int32_t* ctx_len, int b, int LH) {
  int64_t t = 0;
  for (int i = 0; i < b; ++i) t += (int64_t)ctx_len[i];
  return t * LH;
}

// Order-preserving map of a float to uint32 (larger float -> larger code).
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(KVC_FULL_MASK, v, o);
  return v;
}
// Warp sums of four values at once: a reduce-scatter (lanes 16..31 keep v[2..3],
// lanes 8..15 / 24..31 keep the odd one, then three butterfly levels) leaves the
// total of value g on lane 8*g, which is broadcast back.  10 shuffles instead of
// 20 for four separate reductions.
__device__ __forceinline__ void warp_sum4(float (&v)[4], int lane) {
  const bool hi16 = (lane & 16) != 0;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = hi16 ? v[i] : v[i + 2];
    const float keep = hi16 ? v[i + 2] : v[i];
    v[i] = keep + __shfl_xor_sync(KVC_FULL_MASK, send, 16);
  }
  const bool hi8 = (lane & 8) != 0;
  {
    const float send = hi8 ? v[0] : v[1];
    const float keep = hi8 ? v[1] : v[0];
    v[0] = keep + __shfl_xor_sync(KVC_FULL_MASK, send, 8);
  }
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) v[0] += __shfl_xor_sync(KVC_FULL_MASK, v[0], o);
  const float t = v[0];
#pragma unroll
  for (int g = 0; g < 4; ++g) v[g] = __shfl_sync(KVC_FULL_MASK, t, 8 * g);
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while its predecessor in the stream finishes;
// pdl_wait() blocks until the predecessor grids have completed and their
// memory is visible (immediately when there is no such predecessor), and
// pdl_trigger() lets this grid's own dependents be scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// max of three floats in one instruction (PTX three-input max).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 2^x with the PTX approximate base-2 exponential instruction; results below
// 2^-126 flush to zero (the callers sum probabilities relative to a maximum).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(KVC_FULL_MASK, v, o));
  return v;
}

// ---------------------------------------------------------------- prototype trees
// The tree of a slot [x0, y0): 15 nodes in breadth-first order, node j's
// children 2j+1 and 2j+2, nodes 7..14 the leaf prototypes.  Internal node j of
// depth k covering [a, b) is cut at x0 + cuts[j] when a cut table is given and
// that cut is valid (each child keeps 2..16 tokens per leaf below it, 2^(2-k)
// leaves), otherwise at the midpoint floor((a + b) / 2), which is valid for
// every node of a slot of 16..128 tokens.  Every kernel derives its nodes
// through these helpers, so they all see one tree.
__device__ __forceinline__ bool tree_cut_valid(int t, int depth, int a, int b) {
  const int lo = 8 >> depth, hi = 64 >> depth;
  return t - a >= lo && t - a <= hi && b - t >= lo && b - t <= hi;
}
__device__ __forceinline__ int tree_cut(const uint8_t* cuts, int j, int depth, int x0, int a,
                                        int b) {
  if (cuts) {
    const int t = x0 + (int)cuts[j];
    if (tree_cut_valid(t, depth, a, b)) return t;
  }
  return (a + b) >> 1;
}
__device__ __forceinline__ int tree_depth(int j) {
  return (j >= 7) ? 3 : (j >= 3) ? 2 : (j >= 1) ? 1 : 0;
}
// Whether depth-2 node [a, b) may isolate token t (a three-way child set [a, t),
// t, [t+1, b)): both sides keep 2..15 tokens.
__device__ __forceinline__ bool tree_extract_valid(int t, int a, int b) {
  const int l = t - a, r = b - t - 1;
  return l >= 2 && l <= 15 && r >= 2 && r <= 15;
}
// The salient token isolated by depth-2 node j (3..6) covering [a, b), or -1:
// bit j - 3 of byte 7 set and byte j = t - x0 a valid three-way cut.
__device__ __forceinline__ int tree_extract(const uint8_t* cuts, int j, int x0, int a, int b) {
  if (!cuts || j < 3 || j > 6 || !((cuts[7] >> (j - 3)) & 1)) return -1;
  const int t = x0 + (int)cuts[j];
  return tree_extract_valid(t, a, b) ? t : -1;
}
// Token range [a, b) of node j (the leaves below a three-way depth-2 node
// exclude its salient token).
__device__ __forceinline__ void tree_node_range(const uint8_t* cuts, int j, int x0, int y0,
                                                int& a, int& b) {
  const int depth = tree_depth(j);
  const int k = j - ((1 << depth) - 1);
  a = x0; b = y0;
  int node = 0;
  for (int lvl = depth - 1; lvl >= 0; --lvl) {
    const bool right = (k >> lvl) & 1;
    const int e = depth - 1 - lvl == 2 ? tree_extract(cuts, node, x0, a, b) : -1;
    if (e >= 0) {
      if (right) { a = e + 1; node = 2 * node + 2; } else { b = e; node = 2 * node + 1; }
      continue;
    }
    const int t = tree_cut(cuts, node, depth - 1 - lvl, x0, a, b);
    if (right) { a = t; node = 2 * node + 2; } else { b = t; node = 2 * node + 1; }
  }
}
// Cut table of slot s of (b,l,h) blh (8 bytes per slot, cuts of nodes 0..6 as
// offsets from the slot start), or null for midpoint trees.
__device__ __forceinline__ const uint8_t* tree_cuts_of(const kvc_params& p, long long blh,
                                                       int s) {
  return p.tree_cuts ? p.tree_cuts + ((long long)blh * p.S_max + s) * 8 : nullptr;
}

}  // namespace kvcd

// ---------------------------------------------------------------- async copy / mbarrier
namespace kvcd {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// The waiting thread is suspended until the phase completes or a hint of 1 ms
// passes (instead of returning at once), so waiters spin fewer times.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete; gives up after
// `limit_ns` nanoseconds of global time and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > limit_ns) return false;
  return true;
}

// Asynchronous prefetch of the global range [src, src + bytes) into L2 (a
// hint: nothing waits for it; 16-byte aligned, bytes % 16 == 0, in bounds).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 1-D bulk asynchronous copy global -> shared (16-byte aligned, size % 16 == 0),
// completing `bytes` transactions on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace kvcd
