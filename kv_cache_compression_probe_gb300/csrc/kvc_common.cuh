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
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(KVC_FULL_MASK, v, o));
  return v;
}

}  // namespace kvcd
