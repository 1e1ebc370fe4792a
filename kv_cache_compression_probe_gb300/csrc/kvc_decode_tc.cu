// a7 on tensor cores (bf16, d = 128): ragged GQA decode as a split-K
// flash-decode with tcgen05 (GraceKV "05 Physical cache packing": decode
// attends over each (layer, head)'s independently sized cache with the +ln m
// bias; new tokens are appended with multiplicity one).
//
// A plan kernel lists the work: every (b,l,h) with len entries contributes
// max(1, ceil(len / 512)) chunks.  One CTA of the attention kernel takes one
// chunk of up to 4 tiles of 128 cached entries:
//   QK   S^T[128 keys x 16] = K_tile x Q^T: the K tile arrives by TMA in
//        128-byte-swizzled K-major form (A operand), the G query heads are the
//        K-major B operand padded to 16 rows; fp32 accumulators in TMEM, one
//        16-column block per tile.
//   soft one epilogue thread per key row: s = S log2(e)/sqrt(d) + log2(e) ln m,
//        per-head chunk max (across the 4 epilogue warps), P = 2^(s - max)
//        rounded to bf16 into the K-major B operand of the second product; the
//        row sums add the rounded values, so the normalisation matches P.
//   PV   O^T[128 features x 16] += V_tile^T x P: the V tile is read as an
//        MN-major A operand straight from the TMA buffer.
// K and V tiles share one 2-slot ring (load order K0..Kn-1, V0..Vn-1), so a
// CTA needs 86 KB of shared memory and two CTAs fit on an SM.  The chunk
// partial (max, sum, O) goes to the workspace; the last CTA of an (l,h) to
// arrive merges the partials with the new token, appends it and increments
// len (every CTA of that (l,h) has read len by then).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "kvc_common.cuh"
#include "kvc_decode_tc.h"
#include "kvc_internal.h"

namespace {

constexpr int kD = 128;
constexpr int kTileRows = 128;
constexpr int kTiles = 4;
constexpr int kChunkTc = kvc::kDecodeTcChunk;
static_assert(kChunkTc == kTileRows * kTiles, "chunk = 4 tiles");
constexpr int kSlots = 2;
constexpr int kThreadsTc = 192;                      // producer, MMA, 4 epilogue warps
constexpr uint32_t kBlock = kTileRows * 64 * 2;      // one 64-feature block of a tile
constexpr uint32_t kTileBytes = 2 * kBlock;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint64_t desc_k(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ uint64_t desc_mn(uint32_t saddr, uint32_t lbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// M = 128, N = 16, bf16 x bf16 -> f32; QK: both operands K-major; PV: A MN-major.
constexpr uint32_t kIdQK = (1u << 4) | (1u << 7) | (1u << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdPV = kIdQK | (1u << 15);

__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   kvcd::smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// N consecutive 32-bit TMEM columns of this thread's lane (no wait).
template <int N> __device__ __forceinline__ void tld(uint32_t taddr, float (&v)[N]);
template <> __device__ __forceinline__ void tld<1>(uint32_t taddr, float (&v)[1]) {
  uint32_t r0;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r0) : "r"(taddr));
  v[0] = __uint_as_float(r0);
}
template <> __device__ __forceinline__ void tld<2>(uint32_t taddr, float (&v)[2]) {
  uint32_t r0, r1;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(taddr));
  v[0] = __uint_as_float(r0);
  v[1] = __uint_as_float(r1);
}
template <> __device__ __forceinline__ void tld<4>(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}
template <> __device__ __forceinline__ void tld<8>(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tma2d(void* dst, const CUtensorMap* m, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(kvcd::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(kvcd::smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Chunks of (b,l,h) i; -1 for a corrupt entry.
__device__ __forceinline__ int chunks_of(const kvc::DecodeTcArgs& a, int64_t i) {
  const int len = a.len_lh[i];
  const int64_t off = a.off_lh[i];
  if (len < 0 || off < 0 || off + len > a.packed_rows ||
      (len + kChunkTc) / kChunkTc > a.n_chunk_max)
    return -1;
  return len > 0 ? (len + kChunkTc - 1) / kChunkTc : 1;
}

// One CTA: the work list in (b,l,h) order.  A corrupt (b,l,h) gets no chunk
// (its output and length stay untouched) and is reported.
__global__ void __launch_bounds__(1024) decode_plan_kernel(kvc::DecodeTcArgs a, int64_t grid_items) {
  __shared__ long long wsum[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t per = (a.blh + 1023) / 1024;
  const int64_t b0 = min(a.blh, (int64_t)tid * per), b1 = min(a.blh, b0 + per);
  long long cnt = 0;
  for (int64_t i = b0; i < b1; ++i) {
    const int n = chunks_of(a, i);
    if (n < 0) kvcd::record_error(a.err, KVC_EDEVICE);
    else cnt += n;
  }
  long long incl = cnt;                             // inclusive scan over the block
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long v = __shfl_up_sync(KVC_FULL_MASK, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    long long w = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long v = __shfl_up_sync(KVC_FULL_MASK, w, o);
      if (lane >= o) w += v;
    }
    wsum[lane] = w;                                 // inclusive over warps
  }
  __syncthreads();
  const long long total = wsum[31];
  if (total > grid_items) {                          // lengths exceed the packed extent
    if (tid == 0) { kvcd::record_error(a.err, KVC_EDEVICE); *a.n_items = 0; }
    return;
  }
  long long start = incl - cnt + (warp > 0 ? wsum[warp - 1] : 0);
  for (int64_t i = b0; i < b1; ++i) {
    const int n = chunks_of(a, i);
    for (int c = 0; c < n; ++c) a.items[start + c] = ((uint32_t)c << 16) | (uint32_t)i;
    start += max(n, 0);
  }
  if (tid == 0) *a.n_items = (int32_t)total;
}

struct DecSmem {
  alignas(1024) unsigned char ring[kSlots][2][kBlock];      // K or V tile per slot
  alignas(1024) unsigned char Pt[kChunkTc / 64][16 * 128];  // P: 16 head rows x 512 keys, K-major
  alignas(1024) unsigned char Qt[2][16 * 128];              // Q: 16 head rows x 128 features
  float red_m[4][8], red_l[4][8];
  float m[8], l[8], s_new[8];
  uint64_t full[kSlots], empty[kSlots], s_ready, p_ready, o_ready, mma_done;
  uint32_t tmem;
  int abort;
  int last;
};

template <int G>
__global__ void __launch_bounds__(kThreadsTc, 2)
    decode_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                     kvc::DecodeTcArgs a) {
  extern __shared__ __align__(1024) unsigned char dec_raw[];
  if ((int)blockIdx.x >= *a.n_items) return;
  DecSmem& sm = *reinterpret_cast<DecSmem*>((reinterpret_cast<uintptr_t>(dec_raw) + 1023) &
                                            ~uintptr_t(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t item = a.items[blockIdx.x];
  const int blh = (int)(item & 0xFFFFu), c = (int)(item >> 16);
  const int len = a.len_lh[blh];                     // checked by the plan
  const int nchunks = len > 0 ? (len + kChunkTc - 1) / kChunkTc : 1;
  const int e0 = c * kChunkTc;
  const int nvalid = max(0, min(kChunkTc, len - e0));
  const int ntiles = (nvalid + kTileRows - 1) / kTileRows;
  const int64_t off = a.off_lh[blh];
  const int h = blh % a.H;
  const int64_t bl = blh / a.H;                      // b * L + l
  const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(a.q) + (bl * a.H * G + (int64_t)h * G) * kD;
  const float* lm = a.logm + off + e0;

  // Q rows into the swizzled B operand (rows >= G zero); P rows >= G zero
  for (int idx = tid; idx < 16 * 16; idx += kThreadsTc) {
    const int r = idx >> 4, ch = idx & 15;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < G) v = __ldg(reinterpret_cast<const uint4*>(qp + r * kD) + ch);
    const int kb = ch >> 3, cc = ch & 7;
    *reinterpret_cast<uint4*>(&sm.Qt[kb][r * 128 + ((cc ^ (r & 7)) << 4)]) = v;
  }
  for (int idx = tid; idx < (16 - G) * 64; idx += kThreadsTc) {
    const int r = G + (idx >> 6), kb = (idx >> 3) & 7, ch = idx & 7;
    *reinterpret_cast<uint4*>(&sm.Pt[kb][r * 128 + ch * 16]) = make_uint4(0, 0, 0, 0);
  }
  kvcd::fence_proxy_async_smem();
  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      kvcd::mbar_init(&sm.full[i], 1);
      kvcd::mbar_init(&sm.empty[i], 1);
    }
    kvcd::mbar_init(&sm.s_ready, 1);
    kvcd::mbar_init(&sm.p_ready, 4);
    kvcd::mbar_init(&sm.o_ready, 1);
    kvcd::mbar_init(&sm.mma_done, 1);
    sm.abort = 0;
    kvcd::fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     kvcd::smem_u32(&sm.tmem)), "r"(128u)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = sm.tmem;
  volatile int* abort_flag = &sm.abort;
  const int y_base = (int)(off + e0);
  int last_issue[kSlots] = {-1, -1};                 // producer: last load per slot

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      for (int i = 0; i < 2 * ntiles; ++i) {
        const int s = i & 1;
        if (i >= kSlots && !kvcd::mbar_wait(&sm.empty[s], (uint32_t)(((i >> 1) - 1) & 1))) {
          ok = false;
          break;
        }
        if (*abort_flag) break;
        const bool is_k = i < ntiles;
        const int t = is_k ? i : i - ntiles;
        kvcd::mbar_arrive_expect_tx(&sm.full[s], kTileBytes);
        tma2d(sm.ring[s][0], is_k ? &kmap : &vmap, 0, y_base + t * kTileRows, &sm.full[s]);
        tma2d(sm.ring[s][1], is_k ? &kmap : &vmap, 64, y_base + t * kTileRows, &sm.full[s]);
        last_issue[s] = i;
      }
      if (!ok) *abort_flag = 1;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (lane 0 issues)
    if (ntiles > 0) {
      bool ok = true;
      for (int i = 0; i < 2 * ntiles && ok; ++i) {
        const int s = i & 1;
        if (i == ntiles) {                           // every S block issued: hand over, wait for P
          if (lane == 0) commit(&sm.s_ready);
          ok = __all_sync(KVC_FULL_MASK, kvcd::mbar_wait(&sm.p_ready, 0));
          if (!ok) break;
        }
        ok = __all_sync(KVC_FULL_MASK, kvcd::mbar_wait(&sm.full[s], (uint32_t)((i >> 1) & 1)));
        if (!ok) break;
        if (i < ntiles) {
          fence_after();
          if (lane == 0) {
#pragma unroll
            for (int k = 0; k < kD / 16; ++k)
              mma(tmem + i * 16, desc_k(kvcd::smem_u32(sm.ring[s][k >> 2]) + (k & 3) * 32),
                  desc_k(kvcd::smem_u32(sm.Qt[k >> 2]) + (k & 3) * 32), kIdQK, k > 0 ? 1u : 0u);
            commit(&sm.empty[s]);
          }
        } else {
          const int t = i - ntiles;
          const int nrem = nvalid - t * kTileRows;   // valid rows of this V tile
          if (nrem < kTileRows) {                    // rows past the chunk: zero (P is 0 there)
            for (int z = lane; z < (kTileRows - nrem) * 16; z += 32) {
              const int r = nrem + (z >> 4), kb = (z >> 3) & 1, ch = z & 7;
              *reinterpret_cast<uint4*>(&sm.ring[s][kb][r * 128 + ch * 16]) = make_uint4(0, 0, 0, 0);
            }
            kvcd::fence_proxy_async_smem();
            __syncwarp();
          }
          fence_after();
          if (lane == 0) {
#pragma unroll
            for (int k = 0; k < kTileRows / 16; ++k) {
              const int kk = t * (kTileRows / 16) + k;           // 16-key step within the chunk
              mma(tmem + 64, desc_mn(kvcd::smem_u32(sm.ring[s][0]) + k * 2048, kBlock),
                  desc_k(kvcd::smem_u32(sm.Pt[kk >> 2]) + (kk & 3) * 32), kIdPV,
                  (t > 0 || k > 0) ? 1u : 0u);
            }
            commit(&sm.empty[s]);
          }
        }
        __syncwarp();
      }
      if (ok) {
        if (lane == 0) commit(&sm.o_ready);
      } else if (lane == 0) {
        *abort_flag = 1;
      }
    }
  } else {
    // ------------------------------------------------------------ softmax / output warps
    const int ew = warp - 2;
    const int q = warp & 3;                          // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;                   // key row within a tile / feature of O
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    float bias[kTiles];
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
      const int e = t * kTileRows + row;
      bias[t] = e < nvalid ? __ldg(lm + e) * kLog2e : -INFINITY;
    }
    float sv[kTiles][G], mh[G], lh[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      mh[g] = -INFINITY;
      lh[g] = 0.f;
    }
    if (ntiles > 0) {
      if (!*abort_flag && !kvcd::mbar_wait(&sm.s_ready, 0)) *abort_flag = 1;
      fence_after();
#pragma unroll
      for (int t = 0; t < kTiles; ++t)
        if (t < ntiles) tld<G>(tl + t * 16, sv[t]);
      wait_ld();
#pragma unroll
      for (int t = 0; t < kTiles; ++t)
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float s = (t < ntiles && bias[t] != -INFINITY) ? fmaf(sv[t][g], a.scale_log2, bias[t])
                                                               : -INFINITY;
          sv[t][g] = s;
          mh[g] = fmaxf(mh[g], s);
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      mh[g] = kvcd::warp_max(mh[g]);
      if (lane == 0) sm.red_m[ew][g] = mh[g];
    }
    named_sync(1, 128);
#pragma unroll
    for (int g = 0; g < G; ++g)
      mh[g] = fmaxf(fmaxf(sm.red_m[0][g], sm.red_m[1][g]), fmaxf(sm.red_m[2][g], sm.red_m[3][g]));
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
      if (t < ntiles) {
        const int key = t * kTileRows + row;         // within the chunk
        unsigned char* pb = &sm.Pt[key >> 6][(key & 7) * 2];
        const int cidx = (key & 63) >> 3;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pv = sv[t][g] == -INFINITY ? 0.f : exp2f(sv[t][g] - mh[g]);
          const __nv_bfloat16 p16 = __float2bfloat16_rn(pv);
          lh[g] += __bfloat162float(p16);
          *reinterpret_cast<__nv_bfloat16*>(pb + g * 128 + ((cidx ^ (g & 7)) << 4)) = p16;
        }
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      lh[g] = kvcd::warp_sum(lh[g]);
      if (lane == 0) sm.red_l[ew][g] = lh[g];
    }
    kvcd::fence_proxy_async_smem();
    fence_before();
    named_sync(1, 128);
    if (ew == 0 && lane < G) {
      sm.m[lane] = fmaxf(fmaxf(sm.red_m[0][lane], sm.red_m[1][lane]),
                         fmaxf(sm.red_m[2][lane], sm.red_m[3][lane]));
      sm.l[lane] = (sm.red_l[0][lane] + sm.red_l[1][lane]) + (sm.red_l[2][lane] + sm.red_l[3][lane]);
    }
    __syncwarp();
    if (lane == 0) kvcd::mbar_arrive(&sm.p_ready);
    float* part_out = a.partials + ((int64_t)blh * a.n_chunk_max + c) * G * (kD + 2);
    float ov[G];
#pragma unroll
    for (int g = 0; g < G; ++g) ov[g] = 0.f;
    if (ntiles > 0) {
      if (!*abort_flag && !kvcd::mbar_wait(&sm.o_ready, 0)) *abort_flag = 1;
      fence_after();
      tld<G>(tl + 64, ov);
      wait_ld();
    }
#pragma unroll
    for (int g = 0; g < G; ++g) part_out[g * (kD + 2) + 2 + row] = ov[g];
    if (ew == 0 && lane < G) {
      part_out[lane * (kD + 2)] = sm.m[lane];
      part_out[lane * (kD + 2) + 1] = sm.l[lane];
    }
  }

  fence_before();
  __syncthreads();
  if (*abort_flag) {                                 // a bounded wait gave up
    if (warp == 0 && lane == 0)                      // copies still in flight land first
      for (int s = 0; s < kSlots; ++s)
        if (last_issue[s] >= 0) kvcd::mbar_wait(&sm.full[s], (uint32_t)((last_issue[s] >> 1) & 1));
    if (warp == 1 && lane == 0) {                    // and every issued MMA completes
      commit(&sm.mma_done);
      kvcd::mbar_wait(&sm.mma_done, 0);
    }
    __syncthreads();
  }
  fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(128u)
                 : "memory");
  if (*abort_flag) {
    if (tid == 0) kvcd::record_error(a.err, KVC_ETIMEOUT);
    return;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) sm.last = (atomicAdd(a.counters + blh, 1) == nchunks - 1);
  __syncthreads();
  if (!sm.last) return;
  __threadfence();

  // ---- last chunk of this (l,h): merge with the new token, append, len += 1
  const __nv_bfloat16* kn = static_cast<const __nv_bfloat16*>(a.k_new) + (int64_t)blh * kD;
  const __nv_bfloat16* vn = static_cast<const __nv_bfloat16*>(a.v_new) + (int64_t)blh * kD;
  for (int g = warp; g < G; g += kThreadsTc / 32) {
    float acc = 0.f;
#pragma unroll
    for (int f = lane; f < kD; f += 32)
      acc = fmaf(__bfloat162float(qp[g * kD + f]), __bfloat162float(kn[f]), acc);
    acc = kvcd::warp_sum(acc);
    if (lane == 0) sm.s_new[g] = acc * a.scale_log2;
  }
  __syncthreads();
  const float* pbase = a.partials + (int64_t)blh * a.n_chunk_max * G * (kD + 2);
  __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(a.out) + (bl * a.H * G + (int64_t)h * G) * kD;
  for (int idx = tid; idx < G * kD; idx += kThreadsTc) {
    const int g = idx / kD, dd = idx % kD;
    float M = sm.s_new[g];
    for (int cc = 0; cc < nchunks; ++cc) M = fmaxf(M, __ldcg(pbase + (cc * G + g) * (kD + 2)));
    const float fn = exp2f(sm.s_new[g] - M);
    float acc = fn * __bfloat162float(vn[dd]), l = fn;
    for (int cc = 0; cc < nchunks; ++cc) {
      const float* pc = pbase + (cc * G + g) * (kD + 2);
      const float mc = __ldcg(pc);
      const float f = (mc == -INFINITY) ? 0.f : exp2f(mc - M);
      acc = fmaf(f, __ldcg(pc + 2 + dd), acc);
      l = fmaf(f, __ldcg(pc + 1), l);
    }
    outp[g * kD + dd] = __float2bfloat16_rn(acc / l);
  }
  if (len + 1 <= a.cap_lh[blh] && off + len + 1 <= a.packed_rows) {
    __nv_bfloat16* Kw = static_cast<__nv_bfloat16*>(a.Kp) + (off + len) * kD;
    __nv_bfloat16* Vw = static_cast<__nv_bfloat16*>(a.Vp) + (off + len) * kD;
    for (int i = tid; i < kD; i += kThreadsTc) {
      Kw[i] = kn[i];
      Vw[i] = vn[i];
    }
    if (tid == 0) {
      a.logm[off + len] = 0.f;
      a.pos[off + len] = a.pos_new ? a.pos_new[bl / a.L] : -1.f;
      a.len_lh[blh] = len + 1;
    }
  } else if (tid == 0) {
    kvcd::record_error(a.err, KVC_ECAPACITY);
  }
  if (tid == 0) a.counters[blh] = 0;
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 g_enc = nullptr;
std::once_flag g_enc_once;
PFN_cuTensorMapEncodeTiled_v12000 enc_fn() {
  std::call_once(g_enc_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_enc;
}

// Tensor maps of the last (K, V, rows) seen, re-encoded only when they change.
struct MapCache {
  std::mutex mu;
  const void* K = nullptr;
  const void* V = nullptr;
  int64_t rows = 0;
  CUtensorMap km, vm;
};
MapCache g_maps;

bool encode(CUtensorMap* m, void* base, int64_t rows) {
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kTileRows};
  cuuint32_t estr[2] = {1, 1};
  return enc_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int G>
cudaError_t launch_attn(const CUtensorMap& km, const CUtensorMap& vm, const kvc::DecodeTcArgs& a,
                        unsigned grid, cudaStream_t s) {
  const size_t smem = sizeof(DecSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  decode_tc_kernel<G><<<grid, kThreadsTc, smem, s>>>(km, vm, a);
  return cudaGetLastError();
}

}  // namespace

namespace kvc {

bool decode_tc_supported(const kvc_params* p, int n_chunk_max) {
  return p->dtype == KVC_BF16 && p->d == 128 && p->G >= 1 && p->G <= 8 && p->packed_rows > 0 &&
         p->packed_rows < (1LL << 31) && lh_count(p) <= 65535 && n_chunk_max <= 65535 &&
         enc_fn() != nullptr;
}

int decode_tc_launch(const DecodeTcArgs& a, cudaStream_t s) {
  CUtensorMap km, vm;
  {
    std::lock_guard<std::mutex> g(g_maps.mu);
    if (g_maps.K != a.Kp || g_maps.V != a.Vp || g_maps.rows != a.packed_rows) {
      if (!encode(&g_maps.km, a.Kp, a.packed_rows) || !encode(&g_maps.vm, a.Vp, a.packed_rows)) {
        g_maps.K = g_maps.V = nullptr;
        return KVC_ECUDA;
      }
      g_maps.K = a.Kp;
      g_maps.V = a.Vp;
      g_maps.rows = a.packed_rows;
    }
    km = g_maps.km;
    vm = g_maps.vm;
  }
  // every (l,h) has max(1, ceil(len / chunk)) <= len / chunk + 1 chunks and the
  // lengths sum to at most the packed extent
  const int64_t bound = std::min<int64_t>(a.blh * a.n_chunk_max, a.packed_rows / kChunkTc + a.blh);
  decode_plan_kernel<<<1, 1024, 0, s>>>(a, bound);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_status(e);
  switch (a.G) {
    case 1: e = launch_attn<1>(km, vm, a, (unsigned)bound, s); break;
    case 2: e = launch_attn<2>(km, vm, a, (unsigned)bound, s); break;
    case 4: e = launch_attn<4>(km, vm, a, (unsigned)bound, s); break;
    default: e = launch_attn<8>(km, vm, a, (unsigned)bound, s); break;
  }
  count_launch(2);
  return cuda_status(e);
}

}  // namespace kvc
