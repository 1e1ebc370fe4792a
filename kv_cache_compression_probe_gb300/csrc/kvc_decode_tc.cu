// a7 on tensor cores (bf16, d = 128): ragged GQA decode as a split-K
// flash-decode with tcgen05 (GraceKV "05 Physical cache packing": decode
// attends over each (layer, head)'s independently sized cache with the +ln m
// bias; new tokens are appended with multiplicity one).
//
// The work list: every (b,l,h) with len entries contributes
// max(1, ceil(len / 512)) chunks, in (b,l,h) order.  Up to 1024 (b,l,h) each
// attention CTA builds it in shared memory; beyond, a plan kernel writes it to
// the workspace.  The attention kernel is persistent (two CTAs per SM loop
// over the list); one work item is one chunk of up to 4 tiles of 128 cached
// entries:
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
// K and V tiles share one 2-slot ring (load order K0..Kn-1, V0..Vn-1 per item,
// items back to back; an item's 16 query rows arrive by TMA with its first
// tile), so a CTA needs 94 KB of shared memory and two CTAs fit on an SM.  The
// chunk partial (max, sum, O) goes to the workspace.  A merge kernel (one CTA
// per (b,l,h)) then combines the partials with the new token in log-sum-exp
// form, appends the token and increments len.  Plan, attention and merge are
// launched with programmatic dependent launch (each waits for its predecessor
// before reading its results).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <utility>

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
  const int64_t gi = kvc::lh_global(i, a.lh_span, a.lh_gap, a.lh_base);
  const int len = a.len_lh[gi];
  const int64_t off = a.off_lh[gi];
  if (len < 0 || off < 0 || off + len > a.packed_rows ||
      (len + kChunkTc) / kChunkTc > a.n_chunk_max)
    return -1;
  return len > 0 ? (len + kChunkTc - 1) / kChunkTc : 1;
}

// One CTA: the work list in (b,l,h) order.  A corrupt (b,l,h) gets no chunk
// (its output and length stay untouched) and is reported.
__global__ void __launch_bounds__(1024) decode_plan_kernel(kvc::DecodeTcArgs a, int64_t grid_items) {
  constexpr int kPer = 4;                             // entries kept in registers
  __shared__ long long wsum[32];
  kvcd::pdl_trigger();
  kvcd::pdl_wait();                                   // lengths from the previous step
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t per = (a.blh + 1023) / 1024;
  const int64_t b0 = min(a.blh, (int64_t)tid * per), b1 = min(a.blh, b0 + per);
  int nk[kPer];
  long long cnt = 0;
  for (int64_t i = b0; i < b1; ++i) {
    const int n = chunks_of(a, i);
    if (n < 0) kvcd::record_error(a.err, KVC_EDEVICE);
    if (i - b0 < kPer) nk[i - b0] = n;
    cnt += max(n, 0);
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
    const int n = i - b0 < kPer ? nk[i - b0] : chunks_of(a, i);
    for (int c = 0; c < n; ++c) a.items[start + c] = ((uint32_t)c << 16) | (uint32_t)i;
    start += max(n, 0);
  }
  if (tid == 0) *a.n_items = (int32_t)total;
}

// Up to this many (b,l,h) the attention kernel builds the work list itself
// (each CTA scans the chunk counts into shared memory); beyond, a plan kernel
// writes it to the workspace.
constexpr int kInPlanMax = 1024;

struct DecSmem {
  alignas(1024) unsigned char ring[kSlots][2][kBlock];      // K or V tile per slot
  alignas(1024) unsigned char Pt[kChunkTc / 64][16 * 128];  // P: 16 head rows x 512 keys, K-major
  alignas(1024) unsigned char Qt[2][2][16 * 128];           // Q of alternate items, per 64-feature block
  float red_m[4][8], red_l[4][8];
  float m[8], l[8];
  uint64_t full[kSlots], empty[kSlots], s_ready, p_ready, o_ready, mma_done;
  uint32_t tmem;
  int abort;
  int wsum[8];                                             // block scan of the chunk counts
  int pref[kInPlanMax + 1];                                // work items before (b,l,h) i
};

// One work-list entry: chunk c of (b,l,h) blh.
struct Item {
  int blh, c, len, nchunks, nvalid, ntiles;
  int64_t off;
};
// pref: the in-kernel work list (items before each (b,l,h)), or null to read
// the plan kernel's list.
__device__ __forceinline__ Item item_at(const kvc::DecodeTcArgs& a, int idx, const int* pref) {
  Item it;
  if (pref) {                                    // pref[lo] <= idx < pref[lo + 1]
    int lo = 0, hi = (int)a.blh;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pref[mid] <= idx) lo = mid; else hi = mid;
    }
    it.blh = lo;
    it.c = idx - pref[lo];
  } else {
    const uint32_t w = a.items[idx];
    it.blh = (int)(w & 0xFFFFu);
    it.c = (int)(w >> 16);
  }
  const int64_t gi = kvc::lh_global(it.blh, a.lh_span, a.lh_gap, a.lh_base);
  it.len = __ldcg(a.len_lh + gi);          // read before this (l,h)'s last chunk arrives
  it.off = a.off_lh[gi];
  it.nchunks = it.len > 0 ? (it.len + kChunkTc - 1) / kChunkTc : 1;
  it.nvalid = max(0, min(kChunkTc, it.len - it.c * kChunkTc));
  it.ntiles = (it.nvalid + kTileRows - 1) / kTileRows;
  return it;
}

// Persistent: CTA x takes work items x, x + gridDim.x, ...  The producer streams
// K then V tiles of consecutive items through the 2-slot ring (the item's Q
// rides on its first tile's barrier), the MMA warp runs QK(i), waits for P(i),
// runs PV(i), and the epilogue warps do softmax(i), then the chunk partial and,
// for the last chunk of an (l,h), the merge while the next item streams in.
// Registers are reserved per group of 4 warps, so the 6-warp CTA counts as 8:
// two CTAs per SM need <= 65536 / (2 * 256) = 128 registers a thread.
template <int G>
__global__ void __launch_bounds__(256, 2)
    decode_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                     const __grid_constant__ CUtensorMap qmap, kvc::DecodeTcArgs a) {
  extern __shared__ __align__(1024) unsigned char dec_raw[];
  kvcd::pdl_trigger();
  DecSmem& sm = *reinterpret_cast<DecSmem*>((reinterpret_cast<uintptr_t>(dec_raw) + 1023) &
                                            ~uintptr_t(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int idx = tid; idx < (16 - G) * 64; idx += kThreadsTc) {   // P rows >= G stay zero
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
  // the set-up above overlaps the predecessor (plan kernel or previous step)
  kvcd::pdl_wait();
  const int* pref = nullptr;
  int n_items;
  if (a.inplan) {
    // work list in shared memory: chunk counts of every (b,l,h), block scan
    const int nb = (int)a.blh;
    const int per = (nb + kThreadsTc - 1) / kThreadsTc;
    const int b0 = min(nb, tid * per), b1 = min(nb, b0 + per);
    int cnt = 0;
    for (int i = b0; i < b1; ++i) {
      int n = chunks_of(a, i);
      if (n < 0) {                                   // corrupt (b,l,h): no chunk
        if (blockIdx.x == 0) kvcd::record_error(a.err, KVC_EDEVICE);
        n = 0;
      }
      sm.pref[i + 1] = n;
      cnt += n;
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(KVC_FULL_MASK, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) sm.wsum[warp] = incl;
    __syncthreads();
    int run = incl - cnt;
    for (int w = 0; w < warp; ++w) run += sm.wsum[w];
    for (int i = b0; i < b1; ++i) {
      run += sm.pref[i + 1];
      sm.pref[i + 1] = run;
    }
    if (tid == 0) sm.pref[0] = 0;
    __syncthreads();
    n_items = sm.pref[nb];
    if (n_items > a.grid_items) {                    // lengths exceed the packed extent
      if (blockIdx.x == 0 && tid == 0) kvcd::record_error(a.err, KVC_EDEVICE);
      n_items = 0;
    }
    pref = sm.pref;
  } else {
    n_items = *a.n_items;
  }
  const uint32_t tmem = sm.tmem;
  volatile int* abort_flag = &sm.abort;
  int last_issue[kSlots] = {-1, -1};                 // producer: last load per slot

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int t = 0;                                     // tile loads issued so far
      bool ok = true;
      int li = 0;
      for (int idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x, ++li) {
        const Item it = item_at(a, idx, pref);
        const int y_base = (int)(it.off + it.c * kChunkTc);
        for (int i = 0; i < 2 * it.ntiles; ++i, ++t) {
          const int s = t & 1;
          if (t >= kSlots &&
              !kvcd::mbar_wait(&sm.empty[s], (uint32_t)(((t >> 1) - 1) & 1), a.wait_ns)) {
            ok = false;
            break;
          }
          if (*abort_flag) { ok = false; break; }
          if (a.withhold) continue;                  // test of the timeout path: no copies
          const bool is_k = i < it.ntiles;
          const int tt = is_k ? i : i - it.ntiles;
          kvcd::mbar_arrive_expect_tx(&sm.full[s], kTileBytes + (i == 0 ? 2u * 16 * 128 : 0u));
          tma2d(sm.ring[s][0], is_k ? &kmap : &vmap, 0, y_base + tt * kTileRows, &sm.full[s]);
          tma2d(sm.ring[s][1], is_k ? &kmap : &vmap, 64, y_base + tt * kTileRows, &sm.full[s]);
          if (i == 0) {                              // this item's query heads (16 rows)
            tma2d(sm.Qt[li & 1][0], &qmap, 0, it.blh * G, &sm.full[s]);
            tma2d(sm.Qt[li & 1][1], &qmap, 64, it.blh * G, &sm.full[s]);
          }
          last_issue[s] = t;
        }
      }
      if (!ok) *abort_flag = 1;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (lane 0 issues)
    // s_ready, p_ready and o_ready complete once per item with tiles (ne counts
    // them on both sides), so neither side can get two phases ahead
    int t = 0, li = 0, ne = 0;
    bool ok = true;
    for (int idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x, ++li) {
      const Item it = item_at(a, idx, pref);
      if (it.ntiles == 0) continue;
      for (int i = 0; i < it.ntiles; ++i, ++t) {     // S^T blocks
        const int s = t & 1;
        ok = __all_sync(KVC_FULL_MASK, kvcd::mbar_wait(&sm.full[s], (uint32_t)((t >> 1) & 1), a.wait_ns));
        if (!ok) break;
        fence_after();
        if (lane == 0) {
#pragma unroll
          for (int k = 0; k < kD / 16; ++k)
            mma(tmem + i * 16, desc_k(kvcd::smem_u32(sm.ring[s][k >> 2]) + (k & 3) * 32),
                desc_k(kvcd::smem_u32(sm.Qt[li & 1][k >> 2]) + (k & 3) * 32), kIdQK, k > 0 ? 1u : 0u);
          commit(&sm.empty[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) commit(&sm.s_ready);
      ok = __all_sync(KVC_FULL_MASK, kvcd::mbar_wait(&sm.p_ready, (uint32_t)(ne & 1), a.wait_ns));
      if (!ok) break;
      fence_after();
      for (int i = 0; i < it.ntiles; ++i, ++t) {     // O^T += V^T P
        const int s = t & 1;
        ok = __all_sync(KVC_FULL_MASK, kvcd::mbar_wait(&sm.full[s], (uint32_t)((t >> 1) & 1), a.wait_ns));
        if (!ok) break;
        const int nrem = it.nvalid - i * kTileRows;  // valid rows of this V tile
        if (nrem < kTileRows) {                      // rows past the chunk: zero (P is 0 there)
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
            const int kk = i * (kTileRows / 16) + k;           // 16-key step within the chunk
            mma(tmem + 64, desc_mn(kvcd::smem_u32(sm.ring[s][0]) + k * 2048, kBlock),
                desc_k(kvcd::smem_u32(sm.Pt[kk >> 2]) + (kk & 3) * 32), kIdPV,
                (i > 0 || k > 0) ? 1u : 0u);
          }
          commit(&sm.empty[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) commit(&sm.o_ready);
      ++ne;
    }
    if (!ok && lane == 0) *abort_flag = 1;
  } else {
    // ------------------------------------------------------------ softmax / output warps
    const int ew = warp - 2;
    const int q = warp & 3;                          // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;                   // key row within a tile / feature of O
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    int li = 0, ne = 0;                              // items, items with tiles
    for (int idx = blockIdx.x; idx < n_items; idx += gridDim.x, ++li) {
      const Item it = item_at(a, idx, pref);
      const int e0 = it.c * kChunkTc;
      const float* lm = a.logm + it.off + e0;
      float bias[kTiles];
#pragma unroll
      for (int t = 0; t < kTiles; ++t) {
        const int e = t * kTileRows + row;
        bias[t] = e < it.nvalid ? __ldg(lm + e) * kLog2e : -INFINITY;
      }
      float sv[kTiles][G], mh[G], lh[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        mh[g] = -INFINITY;
        lh[g] = 0.f;
      }
      if (it.ntiles > 0) {
        if (!*abort_flag && !kvcd::mbar_wait(&sm.s_ready, (uint32_t)(ne & 1), a.wait_ns)) *abort_flag = 1;
        fence_after();
#pragma unroll
        for (int t = 0; t < kTiles; ++t)
          if (t < it.ntiles) tld<G>(tl + t * 16, sv[t]);
        wait_ld();
#pragma unroll
        for (int t = 0; t < kTiles; ++t)
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float sc = (t < it.ntiles && bias[t] != -INFINITY)
                                 ? fmaf(sv[t][g], a.scale_log2, bias[t]) : -INFINITY;
            sv[t][g] = sc;
            mh[g] = fmaxf(mh[g], sc);
          }
        if (a.scores_out) {                         // the step's scores, one row per thread
#pragma unroll
          for (int t = 0; t < kTiles; ++t) {
            const int e = t * kTileRows + row;
            if (t < it.ntiles && e < it.nvalid) {
              float* so = a.scores_out + (it.off + e0 + e) * G;
#pragma unroll
              for (int g = 0; g < G; ++g) so[g] = sv[t][g];
            }
          }
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
        if (t < it.ntiles) {
          const int key = t * kTileRows + row;       // within the chunk
          unsigned char* pb = &sm.Pt[key >> 6][(key & 7) * 2];
          const int cidx = (key & 63) >> 3;
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float pv = sv[t][g] == -INFINITY ? 0.f : kvcd::ex2(sv[t][g] - mh[g]);
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
      if (lane == 0 && it.ntiles > 0) kvcd::mbar_arrive(&sm.p_ready);
      float* part_out = a.partials + ((int64_t)it.blh * a.n_chunk_max + it.c) * G * (kD + 2);
      float ov[G];
#pragma unroll
      for (int g = 0; g < G; ++g) ov[g] = 0.f;
      if (it.ntiles > 0) {
        if (!*abort_flag && !kvcd::mbar_wait(&sm.o_ready, (uint32_t)(ne & 1), a.wait_ns)) *abort_flag = 1;
        fence_after();
        tld<G>(tl + 64, ov);
        wait_ld();
        fence_before();
        ++ne;
      }
#pragma unroll
      for (int g = 0; g < G; ++g) part_out[g * (kD + 2) + 2 + row] = ov[g];
      if (ew == 0 && lane < G) {
        part_out[lane * (kD + 2)] = sm.m[lane];
        part_out[lane * (kD + 2) + 1] = sm.l[lane];
      }
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
  if (*abort_flag && tid == 0) kvcd::record_error(a.err, KVC_ETIMEOUT);
}

// One CTA (128 G threads, one per output) per (b,l,h): log-sum-exp merge of the
// chunk partials with the new token (appended with multiplicity one), then the
// append itself and len += 1 (the attention kernel has read len by now).
template <int G>
__global__ void __launch_bounds__(128 * G) decode_merge_kernel(kvc::DecodeTcArgs a) {
  __shared__ float s_new[G];
  kvcd::pdl_trigger();
  kvcd::pdl_wait();                                   // the attention kernel's partials
  const int blh = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t gblh = kvc::lh_global(blh, a.lh_span, a.lh_gap, a.lh_base);
  const int len = a.len_lh[gblh];
  const int64_t off = a.off_lh[gblh];
  if (len < 0 || off < 0 || off + len > a.packed_rows || (len + kChunkTc) / kChunkTc > a.n_chunk_max)
    return;                                          // reported by the plan
  const int nch = len > 0 ? (len + kChunkTc - 1) / kChunkTc : 1;
  const int h = blh % a.H;
  const int64_t bl = blh / a.H;
  const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(a.q) + (int64_t)blh * G * kD;
  const __nv_bfloat16* kn = static_cast<const __nv_bfloat16*>(a.k_new) + (int64_t)blh * kD;
  const __nv_bfloat16* vn = static_cast<const __nv_bfloat16*>(a.v_new) + (int64_t)blh * kD;
  const float* pbase = a.partials + (int64_t)blh * a.n_chunk_max * G * (kD + 2);
  if (warp < G) {                                    // warp g: the new token's score for head g
    float acc = 0.f;
#pragma unroll
    for (int f = lane; f < kD; f += 32)
      acc = fmaf(__bfloat162float(qp[warp * kD + f]), __bfloat162float(kn[f]), acc);
    const float sn = kvcd::warp_sum(acc) * a.scale_log2;
    if (lane == 0) s_new[warp] = sn;
    if (a.scores_out && lane == 0 && len + 1 <= a.cap_lh[gblh] && off + len + 1 <= a.packed_rows)
      a.scores_out[(off + len) * G + warp] = sn;
  }
  // thread (g, dd): partials of every chunk, 8 chunks of loads in flight at a
  // time, rescaled online to the running max (every thread of head g sees the
  // same maxima, so the sums agree across the head's threads)
  const int g = tid / kD, dd = tid % kD;
  float M = -INFINITY, acc = 0.f, l = 0.f;
  for (int c0 = 0; c0 < nch; c0 += 8) {
    float mc[8], lc[8], oc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float* pc = pbase + ((c0 + u) * G + g) * (kD + 2);
      const bool in = c0 + u < nch;
      mc[u] = in ? pc[0] : -INFINITY;
      lc[u] = in ? pc[1] : 0.f;
      oc[u] = in ? pc[2 + dd] : 0.f;
    }
    float Mb = M;
#pragma unroll
    for (int u = 0; u < 8; ++u) Mb = fmaxf(Mb, mc[u]);
    if (Mb != -INFINITY) {
      const float sc = M == -INFINITY ? 0.f : exp2f(M - Mb);
      acc *= sc;
      l *= sc;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float f = mc[u] == -INFINITY ? 0.f : exp2f(mc[u] - Mb);
        acc = fmaf(f, oc[u], acc);
        l = fmaf(f, lc[u], l);
      }
      M = Mb;
    }
  }
  __syncthreads();
  {
    const float sn = s_new[g];
    const float Mf = fmaxf(M, sn);
    const float sc = M == -INFINITY ? 0.f : exp2f(M - Mf);
    const float fn = exp2f(sn - Mf);
    const float o = fmaf(fn, __bfloat162float(vn[dd]), acc * sc);
    const float lt = fmaf(l, sc, fn);
    __nv_bfloat16* outp = static_cast<__nv_bfloat16*>(a.out) + (bl * a.H * G + (int64_t)h * G) * kD;
    outp[g * kD + dd] = __float2bfloat16_rn(o / lt);
    if (a.lse_out && dd == 0) a.lse_out[(int64_t)blh * G + g] = Mf + log2f(lt);
  }
  if (len + 1 <= a.cap_lh[gblh] && off + len + 1 <= a.packed_rows) {
    __nv_bfloat16* Kw = static_cast<__nv_bfloat16*>(a.Kp) + (off + len) * kD;
    __nv_bfloat16* Vw = static_cast<__nv_bfloat16*>(a.Vp) + (off + len) * kD;
    if (tid < kD) {
      Kw[tid] = kn[tid];
      Vw[tid] = vn[tid];
    }
    if (tid == 0) {
      a.logm[off + len] = 0.f;
      a.pos[off + len] = a.pos_new ? a.pos_new[bl / a.L] : -1.f;
      a.len_lh[gblh] = len + 1;
    }
  } else if (tid == 0) {
    kvcd::record_error(a.err, KVC_ECAPACITY);
  }
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

// Tensor maps of the last (K, V, rows) and (q, rows) seen, re-encoded only when
// they change.
struct MapCache {
  std::mutex mu;
  const void* K = nullptr;
  const void* V = nullptr;
  int64_t rows = 0;
  const void* Q = nullptr;
  int64_t qrows = 0;
  CUtensorMap km, vm, qm;
};
MapCache g_maps;

// bf16 [rows, 128] in 128-byte-swizzled boxes of 64 features x box_rows rows.
bool encode(CUtensorMap* m, const void* base, int64_t rows, int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch with programmatic stream serialization (the kernel waits for its
// predecessor with pdl_wait before reading what that predecessor writes).
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <int G>
cudaError_t launch_attn(const CUtensorMap& km, const CUtensorMap& vm, const CUtensorMap& qm,
                        const kvc::DecodeTcArgs& a, unsigned grid, cudaStream_t s) {
  const size_t smem = sizeof(DecSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(decode_tc_kernel<G>, dim3(grid), dim3(kThreadsTc), smem, s, km, vm, qm, a);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_merge_kernel<G>, dim3((unsigned)a.blh), dim3(128 * G), 0, s, a);
}

}  // namespace

namespace kvc {

bool decode_tc_supported(const kvc_params* p, int n_chunk_max) {
  return p->dtype == KVC_BF16 && p->d == 128 && p->G >= 1 && p->G <= 8 && p->packed_rows > 0 &&
         p->packed_rows < (1LL << 31) && lh_count(p) <= 65535 && n_chunk_max <= 65535 &&
         enc_fn() != nullptr;
}

int decode_tc_launch(const DecodeTcArgs& a, cudaStream_t s) {
  CUtensorMap km, vm, qm;
  const int64_t qrows = a.blh * a.G;
  {
    std::lock_guard<std::mutex> g(g_maps.mu);
    if (g_maps.K != a.Kp || g_maps.V != a.Vp || g_maps.rows != a.packed_rows) {
      g_maps.K = g_maps.V = nullptr;
      if (!encode(&g_maps.km, a.Kp, a.packed_rows, kTileRows) ||
          !encode(&g_maps.vm, a.Vp, a.packed_rows, kTileRows))
        return KVC_ECUDA;
      g_maps.K = a.Kp;
      g_maps.V = a.Vp;
      g_maps.rows = a.packed_rows;
    }
    if (g_maps.Q != a.q || g_maps.qrows != qrows) {
      g_maps.Q = nullptr;
      if (!encode(&g_maps.qm, a.q, qrows, 16)) return KVC_ECUDA;
      g_maps.Q = a.q;
      g_maps.qrows = qrows;
    }
    km = g_maps.km;
    vm = g_maps.vm;
    qm = g_maps.qm;
  }
  // every (l,h) has max(1, ceil(len / chunk)) <= len / chunk + 1 chunks and the
  // lengths sum to at most the packed extent
  const int64_t bound = std::min<int64_t>(a.blh * a.n_chunk_max, a.packed_rows / kChunkTc + a.blh);
  const int sms = kvc::sm_count();
  if (sms <= 0) return KVC_ECUDA;
  const unsigned grid = (unsigned)std::min<int64_t>(bound, 2LL * sms);   // persistent, 2 per SM
  DecodeTcArgs t = a;
  t.inplan = a.blh <= kInPlanMax ? 1 : 0;
  t.grid_items = bound;
  cudaError_t e = cudaSuccess;
  if (!t.inplan) {
    e = launch_pdl(decode_plan_kernel, dim3(1), dim3(1024), 0, s, t, bound);
    if (e != cudaSuccess) return cuda_status(e);
  }
  switch (t.G) {
    case 1: e = launch_attn<1>(km, vm, qm, t, grid, s); break;
    case 2: e = launch_attn<2>(km, vm, qm, t, grid, s); break;
    case 4: e = launch_attn<4>(km, vm, qm, t, grid, s); break;
    default: e = launch_attn<8>(km, vm, qm, t, grid, s); break;
  }
  count_launch(t.inplan ? 2 : 3);
  return cuda_status(e);
}

}  // namespace kvc
