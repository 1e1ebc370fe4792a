// Tensor-core (tcgen05 / TMEM / TMA) probe-times-key passes of kvc_score for
// bf16 caches with d = 128 (DistillCache 3.1.1 features; GraceKV "03 Bottom-up
// value flow": direct probe attention and the two relevance hops).
//
// One CTA = one (b,l,h) and a chunk of 128-key tiles.  The query rows (probe
// rows, or the hop seeds' values) are written once into shared memory in the
// 128-byte-swizzled K-major layout; one producer thread streams key tiles (128
// keys x 128 features) with 2-D TMA copies (128B swizzle) through a 3-stage
// ring; one MMA thread issues tcgen05.mma (bf16 in, fp32 out) into a
// double-buffered TMEM accumulator; epilogue warps read it with tcgen05.ld.
//   ROWSTATS (probe_tc_kernel: rows on the TMEM lanes, S[rows x 128 keys])
//            max / sum / sum p*(s - max) per row -> chunk partials
//   FEATS    (probe_tcT_kernel: keys on the lanes, S^T[128 keys x rows])
//            a = 2^(s - LSE); per key: sum a, sum a*H_row, per-head sums
//            -> alpha, sigma, H features and r0 = alpha
//   PROP     (probe_tcT_kernel) per key: sum over seeds of w_s 2^(s - LSE_s)
//            -> r = alpha + hop_weight * Prop
// Every mbarrier wait is bounded (KVC_ETIMEOUT); TMEM is always freed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "kvc_common.cuh"
#include "kvc_internal.h"
#include "kvc_score_tc.h"

namespace {

constexpr int kBM = 128;                 // rows per M tile (TMEM lanes)
constexpr int kBN = 128;                 // keys per tile (TMEM columns per tile)
constexpr int kD = 128;                  // head dim
constexpr int kStages = 3;
constexpr uint32_t kTileBytes = kBN * kD * 2;      // 32 KB per key tile (two swizzle blocks)
constexpr uint32_t kBlockBytes = kBN * 64 * 2;     // 16 KB per 64-feature swizzle block

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4)      // start address (16-byte units)
         | ((uint64_t)1 << 16)                    // leading byte offset (unused for SW128 K-major)
         | ((uint64_t)(1024 >> 4) << 32)          // stride byte offset: 8 rows x 128 B
         | ((uint64_t)1 << 46)                    // descriptor version (tcgen05)
         | ((uint64_t)2 << 61);                   // 128-byte swizzle
}

// kind::f16 instruction descriptor: D f32, A/B bf16, both K-major, M = 128, N = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                            ((uint32_t)(kBM >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(kIdesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          kvcd::smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}


__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(kvcd::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(kvcd::smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void mma_bf16_i(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                           uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// 16 consecutive TMEM columns of this thread's lane (issue only; see tmem_wait).
__device__ __forceinline__ void tmem_ld16_nw(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32 consecutive TMEM columns of this thread's lane (issue only; see tmem_wait).
__device__ __forceinline__ void tmem_ld32_nw(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}


// Packed pairs of fp32 (a in the low half): element-wise a * b + c, a * b,
// a + b on both halves with one instruction each.
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 uf2(uint64_t x) {
  float2 f;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(x));
  return f;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float hsum2(uint64_t x) {
  const float2 f = uf2(x);
  return f.x + f.y;
}

// Row-statistics passes: 16 epilogue warps; the NT row blocks' lane quarters
// are covered 4 / NT times, each copy taking its share of a tile's columns.
constexpr int kRsEpiWarps = 16;
constexpr int kRsThreads = (kRsEpiWarps + 2) * 32;
// Registers are reserved for whole groups of 4 warps: 18 warps count as 20, so
// a thread may use at most 65536 / (20 * 32) = 102, i.e. 96 registers.
constexpr int kRsMaxRegs = 96;

template <int NT>
struct TcSmem {
  alignas(1024) unsigned char A[NT][2][kBlockBytes];       // query rows, swizzled
  alignas(1024) unsigned char Bt[kStages][2][kBlockBytes]; // key tiles, swizzled
  float xch[4 / NT - 1][NT * kBM][3];                       // other column shares' (m, l, u)
  uint64_t full[kStages], empty[kStages], tfull[2], tempty[2], mma_done;
  uint32_t tmem_base;
  int abort;
  int issued;
};

template <int NT, int MODE>
__global__ void __maxnreg__(kRsMaxRegs)
    probe_tc_kernel(const __grid_constant__ CUtensorMap kmap, kvc::ProbeTcArgs a) {
  static_assert(MODE == kvc::kTcRowstatsProbes || MODE == kvc::kTcRowstatsSeeds,
                "row-statistics passes only (the per-key passes use probe_tcT_kernel)");
  extern __shared__ __align__(1024) unsigned char tc_raw[];
  // the dynamic shared memory base is aligned up to 1024 bytes by hand
  TcSmem<NT>& sm = *reinterpret_cast<TcSmem<NT>*>(
      (reinterpret_cast<uintptr_t>(tc_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kEpiWarps = kRsEpiWarps;
  constexpr int kThreads = kRsThreads;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long blh = blockIdx.y;
  const int LH = a.L * a.H;
  const int b = (int)(blh / LH);
  const int lh = (int)(blh % LH);
  const int n = a.ctx_len[b];
  const int k0 = blockIdx.x * a.chunk_tiles * kBN;
  const bool seeds = MODE == kvc::kTcRowstatsSeeds;
  const int rows = seeds ? a.P : a.G * a.P;
  float* part_out = a.part + (blh * a.n_chunks + blockIdx.x) * 256 * 3;
  if (!a.ok[blh] || k0 >= n) {
    if (part_out && tid < rows) {
      part_out[tid * 3] = -INFINITY; part_out[tid * 3 + 1] = 0.f; part_out[tid * 3 + 2] = 0.f;
    }
    return;
  }
  const int k1 = min(n, k0 + a.chunk_tiles * kBN);
  const int ntiles = (k1 - k0 + kBN - 1) / kBN;
  const int64_t row0 = kvcd::seq_token_base(a.ctx_len, b, LH) + (int64_t)lh * n;

  // ---- query rows -> swizzled K-major smem (generic stores, then a proxy fence)
  for (int idx = tid; idx < NT * kBM * 16; idx += kThreads) {
    const int r = idx >> 4, c = idx & 15;      // row, 16-byte chunk (8 per swizzle block)
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r < rows) {
      const __nv_bfloat16* src;
      if (seeds) src = static_cast<const __nv_bfloat16*>(a.V) + (row0 + a.seeds[blh * a.P + r]) * kD;
      else src = static_cast<const __nv_bfloat16*>(a.Qp) + (blh * rows + r) * kD;
      val = __ldg(reinterpret_cast<const uint4*>(src) + c);
    }
    const int mt = r >> 7, rr = r & 127, kb = c >> 3, cc = c & 7;
    *reinterpret_cast<uint4*>(&sm.A[mt][kb][rr * 128 + ((cc ^ (rr & 7)) << 4)]) = val;
  }
  kvcd::fence_proxy_async_smem();
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) { kvcd::mbar_init(&sm.full[s], 1); kvcd::mbar_init(&sm.empty[s], 1); }
    for (int s = 0; s < 2; ++s) { kvcd::mbar_init(&sm.tfull[s], 1); kvcd::mbar_init(&sm.tempty[s], kEpiWarps); }
    kvcd::mbar_init(&sm.mma_done, 1);
    sm.abort = 0;
    sm.issued = 0;
    kvcd::fence_mbar_init();
  }
  constexpr uint32_t kCols = NT == 2 ? 512u : 256u;
  if (warp == kEpiWarps + 1) {                     // MMA warp allocates TMEM
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     kvcd::smem_u32(&sm.tmem_base)), "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == kEpiWarps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % kStages;
        if (t >= kStages &&
            !kvcd::mbar_wait(&sm.empty[s], (uint32_t)(((t / kStages) - 1) & 1), a.wait_ns)) {
          sm.abort = 1;
          break;
        }
        if (a.withhold) continue;                  // test of the timeout path: no copies
        kvcd::mbar_arrive_expect_tx(&sm.full[s], kTileBytes);
        const int y = (int)(row0 + k0 + t * kBN);
        tma_load_2d(sm.Bt[s][0], &kmap, 0, y, &sm.full[s]);
        tma_load_2d(sm.Bt[s][1], &kmap, 64, y, &sm.full[s]);
        sm.issued = t + 1;
      }
    }
  } else if (warp == kEpiWarps + 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % kStages, bf = t & 1;
        if (!kvcd::mbar_wait(&sm.full[s], (uint32_t)((t / kStages) & 1), a.wait_ns)) { sm.abort = 1; break; }
        if (t >= 2 && !kvcd::mbar_wait(&sm.tempty[bf], (uint32_t)(((t >> 1) - 1) & 1), a.wait_ns)) {
          sm.abort = 1;
          break;
        }
        tc_fence_after();
        // descriptors advance by 16-byte units: a base per operand, constant steps
        const uint64_t dB = sw128_desc(kvcd::smem_u32(sm.Bt[s][0]));
#pragma unroll
        for (int mt = 0; mt < NT; ++mt) {
          const uint32_t d = tmem + (uint32_t)((bf * NT + mt) * kBN);
          const uint64_t dA = sw128_desc(kvcd::smem_u32(sm.A[mt][0]));
#pragma unroll
          for (int k = 0; k < kD / 16; ++k) {
            const uint64_t step = (uint64_t)((k >> 2) * (kBlockBytes >> 4) + (k & 3) * 2);
            mma_bf16(d, dA + step, dB + step, k > 0 ? 1u : 0u);
          }
        }
        mma_commit(&sm.empty[s]);
        mma_commit(&sm.tfull[bf]);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    // Row statistics over the keys: m (running max of s = S log2e / sqrt(d)),
    // l = sum 2^(s - m) and, for probe rows, u = sum 2^(s - m) (s - m) <= 0.
    // Warp w reads lane quarter w % 4 of row block (w / 4) % NT and column
    // share w / (4 NT) (kCW columns of every tile, in 16-column batches).  Per
    // batch the terms are summed as a tree and added to l and u with one
    // compensated (Kahan) step; masks are applied only on boundary batches.
    // The shares of a row meet once at the end (rescaled to a common max).
    constexpr bool kU = MODE == kvc::kTcRowstatsProbes;
    constexpr int kSplit = 4 / NT;
    constexpr int kCW = kBN / kSplit;
    constexpr int kCh = 16;
    const int q = warp & 3, mt = (warp >> 2) % NT, sp = warp / (4 * NT);
    const int r = mt * kBM + q * 32 + lane;
    const bool rv = r < rows;
    const int limit = seeds ? n - 1 : n - a.P + (r % a.P);
    float m = -INFINITY, l = 0.f, u = 0.f, cl = 0.f, cu = 0.f;
    volatile int* abort_flag = &sm.abort;
    const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16);
    for (int t = 0; t < ntiles; ++t) {
      // every epilogue warp runs all ntiles iterations; after an abort the
      // waits are skipped and the work is void
      const int bf = t & 1;
      if (!*abort_flag && !kvcd::mbar_wait(&sm.tfull[bf], (uint32_t)((t >> 1) & 1), a.wait_ns)) *abort_flag = 1;
      tc_fence_after();
      const int kt = k0 + t * kBN + sp * kCW;
      const uint32_t col0 = tbase + (uint32_t)((bf * NT + mt) * kBN + sp * kCW);
      float v[kCh];
      tmem_ld16_nw(col0, v);
      tmem_wait();
#pragma unroll
      for (int c = 0; c < kCW / kCh; ++c) {
        float vn[kCh];
        if (c + 1 < kCW / kCh) tmem_ld16_nw(col0 + (c + 1) * kCh, vn);   // next batch in flight
        const int i0 = kt + c * kCh;
        const bool fullc = rv && i0 + kCh - 1 < k1 && i0 + kCh - 1 <= limit;
        // One batch: the max is taken on the raw products (the scale is
        // positive), each exponent argument t = S c - m is one FMA, and the
        // masked form is separate code that only boundary batches run.
        auto batch = [&](auto masked_tag) {
          constexpr bool kMasked = decltype(masked_tag)::value;
          float raw[kCh];
#pragma unroll
          for (int j = 0; j < kCh; ++j)
            raw[j] = (!kMasked || (rv && i0 + j < k1 && i0 + j <= limit)) ? v[j] : -INFINITY;
          static_assert(kCh == 16, "three-input max tree over 16 values");
          const float r0 = kvcd::fmax3(raw[0], raw[1], raw[2]);
          const float r1 = kvcd::fmax3(raw[3], raw[4], raw[5]);
          const float r2 = kvcd::fmax3(raw[6], raw[7], raw[8]);
          const float r3 = kvcd::fmax3(raw[9], raw[10], raw[11]);
          const float r4 = kvcd::fmax3(raw[12], raw[13], raw[14]);
          const float rmax = kvcd::fmax3(kvcd::fmax3(r0, r1, r2), fmaxf(r3, r4), raw[15]);
          if (kMasked && rmax == -INFINITY) return;          // nothing valid in the batch
          const float mx = fmaxf(m, rmax * a.q_scale2);
          if (mx > m && m != -INFINITY) {
            const float sc = kvcd::ex2(m - mx);
            if (kU) { u = sc * (u + (m - mx) * l); cu *= sc; }
            l *= sc;
            cl *= sc;
          }
          m = mx;
          float esum, dsum = 0.f;
          if constexpr (!kMasked) {
            // arguments, products and the two tree sums on packed pairs
            const uint64_t c2 = f2(a.q_scale2, a.q_scale2), nm2 = f2(-mx, -mx);
            // sum e as a tree, sum e t as two fused multiply-add chains
            uint64_t e2[kCh / 2], dA = f2(0.f, 0.f), dB = f2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < kCh / 2; ++j) {
              const uint64_t t2 = fma2(f2(raw[2 * j], raw[2 * j + 1]), c2, nm2);
              const float2 tt = uf2(t2);
              e2[j] = f2(kvcd::ex2(tt.x), kvcd::ex2(tt.y));
              if (kU) {
                if (j & 1) dB = fma2(e2[j], t2, dB);
                else dA = fma2(e2[j], t2, dA);
              }
            }
#pragma unroll
            for (int w = kCh / 4; w >= 1; w >>= 1)
#pragma unroll
              for (int j = 0; j < w; ++j) e2[j] = add2(e2[j], e2[j + w]);
            esum = hsum2(e2[0]);
            if (kU) dsum = hsum2(add2(dA, dB));
          } else {
            float e[kCh], d[kCh];
#pragma unroll
            for (int j = 0; j < kCh; ++j) {
              const float tj = fmaf(raw[j], a.q_scale2, -mx);
              e[j] = kvcd::ex2(tj);                          // -inf -> 0
              if (kU) d[j] = raw[j] != -INFINITY ? e[j] * tj : 0.f;
            }
#pragma unroll
            for (int w = kCh / 2; w >= 1; w >>= 1)
#pragma unroll
              for (int j = 0; j < w; ++j) {
                e[j] += e[j + w];
                if (kU) d[j] += d[j + w];
              }
            esum = e[0];
            if (kU) dsum = d[0];
          }
          const float yl = esum - cl, tl = l + yl;
          cl = (tl - l) - yl;
          l = tl;
          if (kU) {
            const float yu = dsum - cu, tu = u + yu;
            cu = (tu - u) - yu;
            u = tu;
          }
        };
        if (fullc) batch(std::false_type{});
        else batch(std::true_type{});
        if (c + 1 < kCW / kCh) {
          tmem_wait();
#pragma unroll
          for (int j = 0; j < kCh; ++j) v[j] = vn[j];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) kvcd::mbar_arrive(&sm.tempty[bf]);
    }
    // the column shares of each row: share 0 adds the others in share order
    if (sp > 0) {
      sm.xch[sp - 1][r][0] = m;
      sm.xch[sp - 1][r][1] = l;
      sm.xch[sp - 1][r][2] = u;
    }
    named_bar(1, kEpiWarps * 32);
    if (sp == 0) {
#pragma unroll
      for (int o = 0; o < kSplit - 1; ++o) {
        const float mo = sm.xch[o][r][0], lo = sm.xch[o][r][1], uo = sm.xch[o][r][2];
        const float M = fmaxf(m, mo);
        if (M != -INFINITY) {
          const float f0 = m == -INFINITY ? 0.f : exp2f(m - M);
          const float f1 = mo == -INFINITY ? 0.f : exp2f(mo - M);
          if (kU)
            u = (m == -INFINITY ? 0.f : f0 * (u + (m - M) * l)) +
                (mo == -INFINITY ? 0.f : f1 * (uo + (mo - M) * lo));
          l = f0 * l + f1 * lo;
          m = M;
        }
      }
      if (part_out && rv) { part_out[r * 3] = m; part_out[r * 3 + 1] = l; part_out[r * 3 + 2] = u; }
    }
  }

  // ---- teardown: every role has finished; wait out copies and products of an
  // aborted run before the tensor memory is freed
  __syncthreads();
  if (sm.abort && tid == 0) {
    kvcd::record_error(a.err, KVC_ETIMEOUT);
    // bounded wait for the key tiles still in flight (the last kStages issued)
    for (int t = max(0, sm.issued - kStages); t < sm.issued; ++t)
      kvcd::mbar_wait(&sm.full[t % kStages], (uint32_t)((t / kStages) & 1), 100000000ull);
  }
  if (sm.abort && warp == kEpiWarps + 1) {
    if (lane == 0) {
      mma_commit(&sm.mma_done);
      kvcd::mbar_wait(&sm.mma_done, 0);
    }
    __syncwarp();
  }
  tc_fence_after();
  if (warp == kEpiWarps + 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols)
                 : "memory");
  }
}

// ---------------------------------------------------------------- transposed per-key passes
// FEATS and PROP reduce over the query rows for every key, so here the keys
// sit on the TMEM lanes: S^T[128 keys x N rows] = K_tile Q^T (K tile = A
// operand straight from the TMA ring, the query rows = K-major B operand; FEATS
// N = 256 probe rows as two N = 128 products, PROP N = P <= 128 seed rows).
// Sixteen epilogue warps: warp w reads lane quarter w % 4 (32 keys) and
// column share w / 4 (a quarter of the buffer's columns, in 16-column
// batches); the four shares of a key meet once per tile in shared memory and
// share 0 adds them in share order.
template <int NT>
struct TcTSmem {
  alignas(1024) unsigned char A[NT][2][kBlockBytes];       // query rows (B operand), swizzled
  alignas(1024) unsigned char Bt[kStages][2][kBlockBytes]; // key tiles (A operand), swizzled
  alignas(16) float col_a[NT * kBM];                        // per row: minus its base-2 LSE (-inf: no row)
  alignas(16) float col_b[NT * kBM];                        // per row: H (FEATS) or seed weight (PROP)
  float xch[2][3][kBN][9];                                  // shares 1..3: per-key sums, by tile parity
  uint64_t full[kStages], empty[kStages], tfull[2], tempty[2], mma_done;
  uint32_t tmem_base;
  int abort;
  int issued;
};

template <int MODE, int PN>
__global__ void __maxnreg__(kRsMaxRegs)
    probe_tcT_kernel(const __grid_constant__ CUtensorMap kmap, kvc::ProbeTcArgs a) {
  constexpr int NT = MODE == kvc::kTcFeats ? 2 : 1;          // 128-row blocks of B
  constexpr int kEpiWarps = kRsEpiWarps;
  constexpr int kThreads = kRsThreads;
  constexpr int kN = MODE == kvc::kTcFeats ? 256 : PN;       // columns per TMEM buffer (PROP: PN >= P)
  extern __shared__ __align__(1024) unsigned char tt_raw[];
  TcTSmem<NT>& sm = *reinterpret_cast<TcTSmem<NT>*>(
      (reinterpret_cast<uintptr_t>(tt_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long blh = blockIdx.y;
  const int LH = a.L * a.H;
  const int b = (int)(blh / LH);
  const int lh = (int)(blh % LH);
  const int n = a.ctx_len[b];
  const int k0 = blockIdx.x * a.chunk_tiles * kBN;
  const int rows = MODE == kvc::kTcProp ? a.P : a.G * a.P;
  if (!a.ok[blh] || k0 >= n) return;
  const int k1 = min(n, k0 + a.chunk_tiles * kBN);
  const int ntiles = (k1 - k0 + kBN - 1) / kBN;
  const int64_t row0 = kvcd::seq_token_base(a.ctx_len, b, LH) + (int64_t)lh * n;

  for (int idx = tid; idx < NT * kBM * 16; idx += kThreads) {
    const int r = idx >> 4, c = idx & 15;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r < rows) {
      const __nv_bfloat16* src;
      if (MODE == kvc::kTcProp) src = static_cast<const __nv_bfloat16*>(a.V) + (row0 + a.seeds[blh * a.P + r]) * kD;
      else src = static_cast<const __nv_bfloat16*>(a.Qp) + (blh * rows + r) * kD;
      val = __ldg(reinterpret_cast<const uint4*>(src) + c);
    }
    const int mt = r >> 7, rr = r & 127, kb = c >> 3, cc = c & 7;
    *reinterpret_cast<uint4*>(&sm.A[mt][kb][rr * 128 + ((cc ^ (rr & 7)) << 4)]) = val;
  }
  for (int c = tid; c < NT * kBM; c += kThreads) {
    const bool in = c < rows;
    if (MODE == kvc::kTcProp) {
      sm.col_a[c] = in ? -a.lse2_h[blh * a.P + c] : -INFINITY;
      sm.col_b[c] = in ? a.seed_w[blh * a.P + c] : 0.f;
    } else {
      sm.col_a[c] = in ? -a.lse2[blh * rows + c] : -INFINITY;
      sm.col_b[c] = in ? a.hrow[blh * rows + c] : 0.f;
    }
  }
  kvcd::fence_proxy_async_smem();
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) { kvcd::mbar_init(&sm.full[s], 1); kvcd::mbar_init(&sm.empty[s], 1); }
    for (int s = 0; s < 2; ++s) { kvcd::mbar_init(&sm.tfull[s], 1); kvcd::mbar_init(&sm.tempty[s], kEpiWarps); }
    kvcd::mbar_init(&sm.mma_done, 1);
    sm.abort = 0;
    sm.issued = 0;
    kvcd::fence_mbar_init();
  }
  constexpr uint32_t kCols = 2 * kN <= 128 ? 128u : (2 * kN <= 256 ? 256u : 512u);   // power of 2
  if (warp == kEpiWarps + 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     kvcd::smem_u32(&sm.tmem_base)), "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == kEpiWarps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % kStages;
        if (t >= kStages &&
            !kvcd::mbar_wait(&sm.empty[s], (uint32_t)(((t / kStages) - 1) & 1), a.wait_ns)) {
          sm.abort = 1;
          break;
        }
        if (a.withhold) continue;                  // test of the timeout path: no copies
        kvcd::mbar_arrive_expect_tx(&sm.full[s], kTileBytes);
        const int y = (int)(row0 + k0 + t * kBN);
        tma_load_2d(sm.Bt[s][0], &kmap, 0, y, &sm.full[s]);
        tma_load_2d(sm.Bt[s][1], &kmap, 64, y, &sm.full[s]);
        sm.issued = t + 1;
      }
    }
  } else if (warp == kEpiWarps + 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      // M = 128 keys, N = 128 (FEATS, twice) or N = 64 (PROP), both operands K-major
      constexpr uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                 ((uint32_t)((MODE == kvc::kTcFeats ? 128 : PN) >> 3) << 17) |
                                 ((uint32_t)(kBM >> 4) << 24);
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % kStages, bf = t & 1;
        if (!kvcd::mbar_wait(&sm.full[s], (uint32_t)((t / kStages) & 1), a.wait_ns)) { sm.abort = 1; break; }
        if (t >= 2 && !kvcd::mbar_wait(&sm.tempty[bf], (uint32_t)(((t >> 1) - 1) & 1), a.wait_ns)) {
          sm.abort = 1;
          break;
        }
        tc_fence_after();
        // descriptors advance by 16-byte units: a base per operand, constant steps
        const uint64_t dK = sw128_desc(kvcd::smem_u32(sm.Bt[s][0]));
#pragma unroll
        for (int nb = 0; nb < NT; ++nb) {
          const uint32_t d = tmem + (uint32_t)(bf * kN + nb * 128);
          const uint64_t dQ = sw128_desc(kvcd::smem_u32(sm.A[nb][0]));
#pragma unroll
          for (int k = 0; k < kD / 16; ++k) {
            const uint64_t step = (uint64_t)((k >> 2) * (kBlockBytes >> 4) + (k & 3) * 2);
            mma_bf16_i(d, dK + step, dQ + step, idesc, k > 0 ? 1u : 0u);
          }
        }
        mma_commit(&sm.empty[s]);
        mma_commit(&sm.tfull[bf]);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue: thread = key
    constexpr int kCW = kN / 4;                      // columns of one share
    constexpr int kCh = 16;                          // columns per batch
    static_assert(kCW % kCh == 0, "share width");
    const int sp = warp >> 2, q = warp & 3;
    const int kl = q * 32 + lane;                    // key within the tile (TMEM lane)
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    volatile int* abort_flag = &sm.abort;
    for (int t = 0; t < ntiles; ++t) {
      const int bf = t & 1;
      if (!*abort_flag && !kvcd::mbar_wait(&sm.tfull[bf], (uint32_t)((t >> 1) & 1), a.wait_ns)) *abort_flag = 1;
      tc_fence_after();
      const int key = k0 + t * kBN + kl;
      const bool kvalid = key < k1;
      // FEATS: probe row c sees keys <= n - P + (c % P), i.e. c % P >= thr
      const int thr = MODE == kvc::kTcFeats ? key - (n - a.P) : 0;
      const bool full_cols = kvalid && thr <= 0;
      // with P equal to the share width every share is one query head: its
      // head sum and its sum of a H are all the other shares need
      const bool one_head = MODE == kvc::kTcFeats && a.P == kCW && a.G == 4;
      float gs[8], sh = 0.f, acc = 0.f, own = 0.f;
#pragma unroll
      for (int g = 0; g < 8; ++g) gs[g] = 0.f;
      const uint32_t col0 = tmem + lane_off + (uint32_t)(bf * kN + sp * kCW);
      float v[kCh];
      tmem_ld16_nw(col0, v);
      tmem_wait();
#pragma unroll
      for (int c = 0; c < kCW / kCh; ++c) {
        float vn[kCh];
        if (c + 1 < kCW / kCh) tmem_ld16_nw(col0 + (c + 1) * kCh, vn);   // next batch in flight
        const int cb = sp * kCW + c * kCh;           // first column of the batch
        const float4* ca = reinterpret_cast<const float4*>(&sm.col_a[cb]);
        const float4* cbv = reinterpret_cast<const float4*>(&sm.col_b[cb]);
        // the same column parameters read as packed pairs (column 2i in the low half)
        const ulonglong2* ca2 = reinterpret_cast<const ulonglong2*>(&sm.col_a[cb]);
        const ulonglong2* cb2 = reinterpret_cast<const ulonglong2*>(&sm.col_b[cb]);
        float cs = 0.f, chs = 0.f;
        if (full_cols) {
          // unmasked batch on packed pairs: t = S c - LSE, e = 2^t,
          // FEATS: sum e and sum e H; PROP: sum w e
          const uint64_t c2 = f2(a.q_scale2, a.q_scale2);
          uint64_t s1 = f2(0.f, 0.f), s2 = f2(0.f, 0.f);
#pragma unroll
          for (int j4 = 0; j4 < kCh / 4; ++j4) {
            const ulonglong2 la = ca2[j4], lb = cb2[j4];
            const uint64_t t0 = fma2(f2(v[4 * j4], v[4 * j4 + 1]), c2, la.x);
            const uint64_t t1 = fma2(f2(v[4 * j4 + 2], v[4 * j4 + 3]), c2, la.y);
            const float2 u0 = uf2(t0), u1 = uf2(t1);
            const uint64_t e0 = f2(kvcd::ex2(u0.x), kvcd::ex2(u0.y));
            const uint64_t e1 = f2(kvcd::ex2(u1.x), kvcd::ex2(u1.y));
            if (MODE == kvc::kTcFeats) {
              s1 = add2(s1, add2(e0, e1));
              s2 = fma2(e0, lb.x, fma2(e1, lb.y, s2));
            } else {
              s1 = fma2(e0, lb.x, fma2(e1, lb.y, s1));
            }
          }
          if (MODE == kvc::kTcFeats) {
            cs = hsum2(s1);
            chs = hsum2(s2);
          } else {
            acc += hsum2(s1);
          }
        } else {
          // masked form (keys past the chunk, causal probe limits): boundary keys only
#pragma unroll
          for (int j4 = 0; j4 < kCh / 4; ++j4) {
            const float4 la = ca[j4], lb = cbv[j4];
            const float las[4] = {la.x, la.y, la.z, la.w}, lbs[4] = {lb.x, lb.y, lb.z, lb.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int j = j4 * 4 + u;
              float e = kvcd::ex2(fmaf(v[j], a.q_scale2, las[u]));
              const bool ok = kvalid && (MODE == kvc::kTcProp || ((cb + j) % a.P) >= thr);
              e = ok ? e : 0.f;
              if (MODE == kvc::kTcFeats) {
                cs += e;
                chs = fmaf(e, lbs[u], chs);
              } else {
                acc = fmaf(lbs[u], e, acc);
              }
            }
          }
        }
        if (MODE == kvc::kTcFeats) {
          if (one_head) {
            own += cs;
          } else {
            const int head = cb / a.P;               // P % 32 == 0: one head per batch
#pragma unroll
            for (int g = 0; g < 8; ++g)
              if (g == head) gs[g] += cs;
          }
          sh += chs;
        }
        if (c + 1 < kCW / kCh) {
          tmem_wait();
#pragma unroll
          for (int j = 0; j < kCh; ++j) v[j] = vn[j];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) kvcd::mbar_arrive(&sm.tempty[bf]);
      // the four shares of these keys: share 0 adds the others in share order.
      // The exchange buffer alternates with the tile, so one barrier per tile
      // suffices: a share writes buffer t & 1 again only after the barrier of
      // tile t + 1, which share 0 reaches after reading it.
      float (*xc)[kBN][9] = sm.xch[t & 1];
      if (sp > 0) {
        if (MODE == kvc::kTcFeats) {
          if (one_head) {
            xc[sp - 1][kl][0] = own;
            xc[sp - 1][kl][1] = sh;
          } else {
#pragma unroll
            for (int g = 0; g < 8; ++g) xc[sp - 1][kl][g] = gs[g];
            xc[sp - 1][kl][8] = sh;
          }
        } else {
          xc[sp - 1][kl][0] = acc;
        }
      }
      named_bar(1 + q, 128);                         // warps q, q + 4, q + 8, q + 12
      if (sp == 0 && kvalid) {
        if (MODE == kvc::kTcProp) {
#pragma unroll
          for (int o = 0; o < 3; ++o) acc += xc[o][kl][0];
          a.rel[row0 + key] = a.feats[(row0 + key) * 5] + a.hop_weight * acc;
        } else {
          if (one_head) {
            gs[0] = own;
#pragma unroll
            for (int o = 0; o < 3; ++o) {
              gs[1 + o] = xc[o][kl][0];
              sh += xc[o][kl][1];
            }
          } else {
#pragma unroll
            for (int o = 0; o < 3; ++o) {
#pragma unroll
              for (int g = 0; g < 8; ++g) gs[g] += xc[o][kl][g];
              sh += xc[o][kl][8];
            }
          }
          float sa = 0.f, mean = 0.f;
#pragma unroll
          for (int g = 0; g < 8; ++g) sa += gs[g];
          const float invP = 1.f / (float)a.P;
#pragma unroll
          for (int g = 0; g < 8; ++g)
            if (g < a.G) mean += gs[g] * invP;
          mean /= (float)a.G;
          float var = 0.f;
#pragma unroll
          for (int g = 0; g < 8; ++g)
            if (g < a.G) { const float dd = gs[g] * invP - mean; var += dd * dd; }
          var /= (float)a.G;
          float* f = a.feats + (row0 + key) * 5;
          const float alpha = sa / (float)rows;
          f[0] = alpha;
          f[2] = var;
          f[3] = sa > 0.f ? sh / sa : 0.f;
          a.rel[row0 + key] = alpha;
        }
      }
    }
  }

  __syncthreads();
  if (sm.abort && tid == 0) {
    kvcd::record_error(a.err, KVC_ETIMEOUT);
    for (int t = max(0, sm.issued - kStages); t < sm.issued; ++t)
      kvcd::mbar_wait(&sm.full[t % kStages], (uint32_t)((t / kStages) & 1), 100000000ull);
  }
  if (sm.abort && warp == kEpiWarps + 1) {     // issued products finish before TMEM is freed
    if (lane == 0) {
      mma_commit(&sm.mma_done);
      kvcd::mbar_wait(&sm.mma_done, 0);
    }
    __syncwarp();
  }
  tc_fence_after();
  if (warp == kEpiWarps + 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols)
                 : "memory");
  }
}

// ---------------------------------------------------------------- node statistics (a3 + a4)
// One CTA = one (b,l,h), one 128-row tile of the probe rows, and up to
// kNodeSlots consecutive slots.  Per slot:
//   phase A  S = Q K^T (keys placed leaf by leaf on 16-row boundaries) and
//            A^ = Q [k^0; k^1; k^2]^T (k^ in three bf16 parts, summed in fp32);
//   epi A    a = 2^(s - LSE) split into three bf16 parts written as the
//            K-major operand over the 128 leaf-padded key slots (each of the
//            four epilogue groups takes 32 key slots = two leaves); per-row
//            leaf masses to shared memory;
//   phase B  for each node but the root: U_N = sum over parts and over the
//            node's key slots of a_part V (V read as an MN-major operand
//            straight from TMA) into one of two TMEM buffers;
//   epi B    every group reads 32 of the 128 features of each node buffer (the
//            root's U is the sum of the two depth-1 buffers, added here) and
//            forms per-row partial sums of |U - A^ v^|^2 and |U|^2 (packed
//            f32x2 FMAs) into spare TMEM columns; once per slot the four warps
//            sharing a row quarter meet, and warp g finishes the nodes at
//            positions g, g + 4, ...: it adds the partials in a fixed order and
//            forms the row's |U - A^ v^|, |U|, |A - A^| and A, summed over its
//            32 rows.
// Per-(slot, tile) sums go to `npart`; a small kernel forms D and utilities.
constexpr int kNodeSlots = 8;
constexpr int kEpiWarps = 16;                      // 4 groups x 4 row quarters
constexpr int kNodeThreads = (kEpiWarps + 2) * 32; // + producer + MMA issuer
constexpr int kProdWarp = kEpiWarps, kMmaWarp = kEpiWarps + 1;
// Registers are reserved for whole groups of 4 warps: 18 warps count as 20, so
// a thread may use at most 65536 / (20 * 32) = 102, i.e. 96 registers.
constexpr int kNodeMaxRegs = 96;

struct NodeSmem {
  alignas(1024) unsigned char Q[2][kBlockBytes];
  alignas(1024) unsigned char Kt[2][kBlockBytes];
  alignas(1024) unsigned char Vt[2][kBlockBytes];
  alignas(1024) unsigned char Ap[3][2][kBlockBytes];
  alignas(1024) unsigned char Kh[kvc::kProtoHeadBytes]; // k^ parts (phase A operand), ln m, Rv
  alignas(16) float vh[15][128];                          // v^ of the slot's nodes
  float Al[8][128];                                       // per-row leaf masses
  float At[4][128];                                       // per-row mass of each isolated token
  uint4 vsave[4][2][8];                                   // V rows of the isolated tokens
  float red[2][4][15][4];                                 // per-quarter node sums
  uint64_t k_full, k_empty, v_full, v_empty, s_full, a_ready, b_done;
  uint64_t h_full, xch_free;                              // A^ ready; partials read
  uint64_t ap_ready;                                      // the a operand is in shared memory
  uint64_t vh_full, vh_free;
  uint64_t nfull[2], nempty[2];
  uint64_t mma_done, mid_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(NodeSmem) + 1024 <= 232448, "node kernel shared memory");

// N = 48 (three 16-row parts of the prototype keys), both operands K-major.
constexpr uint32_t kIdescN48 = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(48 >> 3) << 17) |
                               ((uint32_t)(kBM >> 4) << 24);
// N = 128 with B MN-major (values: features contiguous, key slots strided).
constexpr uint32_t kIdescVmn = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                               ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);


// MN-major 128-byte-swizzled operand: 64-feature blocks LBO apart, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr, uint32_t lbo_bytes) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo_bytes >> 4) & 0x3FFF) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}



// TMEM columns 128..247 hold, during epilogue B, the per-row partial sums of
// the node at position p from group g: (dd, uu) at 128 + 8p + 2g.  They
// overlap A^ (128..175), which epilogue A has read by then; the next slot's
// A^ product waits until these partials are read (xch_free).
__device__ __forceinline__ uint32_t part_col(int p, int g) {
  return 128u + (uint32_t)(p * 8 + 2 * g);
}
__device__ __forceinline__ void tmem_st2(uint32_t taddr, float a, float b) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(taddr),
               "r"(__float_as_uint(a)), "r"(__float_as_uint(b))
               : "memory");
}

// Leaf l of the slot [x0, y0): first token and token count (at most 16) of
// node 7 + l of the tree with cut table `cuts` (null: midpoint tree).
__device__ __forceinline__ void leaf_range(const uint8_t* cuts, int l, int x0, int y0, int& start,
                                           int& cnt) {
  int a, b;
  kvcd::tree_node_range(cuts, 7 + l, x0, y0, a, b);
  start = a; cnt = b - a;
}

// Order of the node products and their statistics: the eight leaves first
// (few products each, so the epilogue starts at once), then depth 2, depth 1
// and the root, whose products the tensor pipe runs while the epilogue works
// through the leaves.
__device__ constexpr int kNodeOrder[15] = {7, 8, 9, 10, 11, 12, 13, 14, 3, 4, 5, 6, 1, 2, 0};
// Nodes with products of their own: all but the root, whose aggregate the
// epilogue forms from the two depth-1 buffers (positions 12 and 13).
constexpr int kMmaNodes = 14;
static_assert(kMmaNodes % 2 == 0, "buffer of position pj is pj & 1");

// Leaves [l0, l1) covered by node j of the depth-3 tree.
__device__ __forceinline__ void node_leaves(int j, int& l0, int& l1) {
  const int depth = (j >= 7) ? 3 : (j >= 3) ? 2 : (j >= 1) ? 1 : 0;
  const int k = j - ((1 << depth) - 1);
  const int w = 8 >> depth;
  l0 = k * w; l1 = l0 + w;
}

__global__ void __maxnreg__(kNodeMaxRegs)
    nodes_tc_kernel(const __grid_constant__ CUtensorMap kmap16,
                    const __grid_constant__ CUtensorMap vmap16, kvc::NodeTcArgs a) {
  extern __shared__ __align__(1024) unsigned char nd_raw[];
  NodeSmem& sm = *reinterpret_cast<NodeSmem*>(
      (reinterpret_cast<uintptr_t>(nd_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long blh = blockIdx.z;
  const int mt = blockIdx.y;
  const int LH = a.L * a.H;
  const int b = (int)(blh / LH);
  const int lh = (int)(blh % LH);
  if (!a.ok[blh]) return;
  const int S = a.n_slots[b];
  const int s_begin = blockIdx.x * kNodeSlots;
  const int s_end = min(S, s_begin + kNodeSlots);
  if (s_begin >= s_end) return;
  const int nsl = s_end - s_begin;
  const int n = a.ctx_len[b];
  const int R = a.G * a.P;
  const int64_t row0 = kvcd::seq_token_base(a.ctx_len, b, LH) + (int64_t)lh * n;
  const int32_t* bd = a.bounds + (long long)b * (a.S_max + 1);

  // ---- this tile's query rows -> swizzled K-major smem
  for (int idx = tid; idx < kBM * 16; idx += kNodeThreads) {
    const int r = idx >> 4, c = idx & 15;
    const int rho = mt * kBM + r;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (rho < R)
      val = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.Qp) +
                                                 (blh * R + rho) * kD) + c);
    const int kb = c >> 3, cc = c & 7;
    *reinterpret_cast<uint4*>(&sm.Q[kb][r * 128 + ((cc ^ (r & 7)) << 4)]) = val;
  }
  kvcd::fence_proxy_async_smem();
  if (tid == 0) {
    kvcd::mbar_init(&sm.k_full, 1); kvcd::mbar_init(&sm.k_empty, 1);
    kvcd::mbar_init(&sm.v_full, 1); kvcd::mbar_init(&sm.v_empty, 1);
    kvcd::mbar_init(&sm.s_full, 1); kvcd::mbar_init(&sm.a_ready, kEpiWarps);
    kvcd::mbar_init(&sm.h_full, 1); kvcd::mbar_init(&sm.xch_free, kEpiWarps);
    kvcd::mbar_init(&sm.ap_ready, kEpiWarps);
    kvcd::mbar_init(&sm.b_done, 1);
    kvcd::mbar_init(&sm.mma_done, 1);
    kvcd::mbar_init(&sm.mid_done, 1);
    kvcd::mbar_init(&sm.vh_full, 1); kvcd::mbar_init(&sm.vh_free, kEpiWarps);
    for (int i = 0; i < 2; ++i) {
      kvcd::mbar_init(&sm.nfull[i], 1);
      kvcd::mbar_init(&sm.nempty[i], kEpiWarps);
    }
    sm.abort = 0;
    kvcd::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     kvcd::smem_u32(&sm.tmem_base)), "r"(512u)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort;

  if (warp == kProdWarp) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int nk = 0, nv = 0, nh = 0;                    // loads issued per barrier
      for (int k = 0; k < nsl; ++k) {
        const int s = s_begin + k;
        const long long tree = blh * a.S_max + s;
        const int x0 = bd[s], y0 = bd[s + 1];
        const uint8_t* cuts = a.tree_cuts ? a.tree_cuts + tree * 8 : nullptr;
        // Kt / Kh are free once phase A of the previous slot completed and its
        // epilogue read ln m from Kh (a_ready)
        if (k >= 1 && (!kvcd::mbar_wait(&sm.k_empty, (uint32_t)((k - 1) & 1), a.wait_ns) ||
                       !kvcd::mbar_wait(&sm.a_ready, (uint32_t)((k - 1) & 1), a.wait_ns))) {
          *abort_flag = 1;
          break;
        }
        if (a.withhold) continue;                      // test of the timeout path: no copies
        ++nk;
        kvcd::mbar_arrive_expect_tx(&sm.k_full, kTileBytes + kvc::kProtoHeadBytes);
        for (int l = 0; l < 8; ++l) {
          int st, cnt;
          leaf_range(cuts, l, x0, y0, st, cnt);
          for (int fb = 0; fb < 2; ++fb)
            tma_load_2d(&sm.Kt[fb][l * 2048], &kmap16, fb * 64, (int)(row0 + st), &sm.k_full);
        }
        kvcd::bulk_g2s(sm.Kh, a.proto + tree * kvc::kProtoBytes, kvc::kProtoHeadBytes, &sm.k_full);
        if (k >= 1 && !kvcd::mbar_wait(&sm.v_empty, (uint32_t)((k - 1) & 1), a.wait_ns)) { *abort_flag = 1; break; }
        ++nv;
        kvcd::mbar_arrive_expect_tx(&sm.v_full, kTileBytes);
        for (int l = 0; l < 8; ++l) {
          int st, cnt;
          leaf_range(cuts, l, x0, y0, st, cnt);
          for (int fb = 0; fb < 2; ++fb)
            tma_load_2d(&sm.Vt[fb][l * 2048], &vmap16, fb * 64, (int)(row0 + st), &sm.v_full);
        }
        if (k >= 1 && !kvcd::mbar_wait(&sm.vh_free, (uint32_t)((k - 1) & 1), a.wait_ns)) { *abort_flag = 1; break; }
        ++nh;
        kvcd::mbar_arrive_expect_tx(&sm.vh_full, 15 * 128 * 4);
        kvcd::bulk_g2s(&sm.vh[0][0], a.proto + tree * kvc::kProtoBytes + kvc::kProtoVhOff,
                       15 * 128 * 4, &sm.vh_full);
      }
      if (*abort_flag) {                               // let copies in flight land
        if (nk) kvcd::mbar_wait(&sm.k_full, (uint32_t)((nk - 1) & 1));
        if (nv) kvcd::mbar_wait(&sm.v_full, (uint32_t)((nv - 1) & 1));
        if (nh) kvcd::mbar_wait(&sm.vh_full, (uint32_t)((nh - 1) & 1));
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int nmid = 0;                                  // uses of mid_done so far
      for (int k = 0; k < nsl; ++k) {
        // key slot of each depth-2 node's isolated token in its left leaf's
        // box (-1: none); the token counts in the node and its ancestors but
        // not in the leaf, so its V rows are zeroed before the leaf products
        int salc[4];
        bool sal_any = false;
        {
          const int s = s_begin + k;
          const uint8_t* cuts = a.tree_cuts ? a.tree_cuts + (blh * a.S_max + s) * 8 : nullptr;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            int a2, b2;
            kvcd::tree_node_range(cuts, 3 + g, bd[s], bd[s + 1], a2, b2);
            const int e = kvcd::tree_extract(cuts, 3 + g, bd[s], a2, b2);
            salc[g] = e >= 0 ? e - a2 : -1;
            sal_any |= e >= 0;
          }
        }
        if (!kvcd::mbar_wait(&sm.k_full, (uint32_t)(k & 1), a.wait_ns)) { *abort_flag = 1; break; }
        tc_fence_after();
        {
          // descriptors advance by 16-byte units: one base each, constant steps
          const uint64_t dQ = sw128_desc(kvcd::smem_u32(sm.Q[0]));
          const uint64_t dK = sw128_desc(kvcd::smem_u32(sm.Kt[0]));
          const uint64_t dH = sw128_desc(kvcd::smem_u32(sm.Kh));
          static_assert(sizeof(sm.Q[0]) == kBlockBytes && sizeof(sm.Kt[0]) == kBlockBytes,
                        "operand blocks are contiguous");
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint64_t step = (uint64_t)((kk >> 2) * (kBlockBytes >> 4) + (kk & 3) * 2);
            mma_bf16_i(tmem, dQ + step, dK + step, kIdesc, kk > 0 ? 1u : 0u);
          }
          mma_commit(&sm.s_full);
          // A^ lands on the columns of the previous slot's node partials
          if (k >= 1 && !kvcd::mbar_wait(&sm.xch_free, (uint32_t)((k - 1) & 1), a.wait_ns)) {
            *abort_flag = 1;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint64_t step = (uint64_t)((kk >> 2) * (kBlockBytes >> 4) + (kk & 3) * 2);
            mma_bf16_i(tmem + 128, dQ + step,
                       dH + (uint64_t)((kk >> 2) * (6144 >> 4) + (kk & 3) * 2), kIdescN48,
                       kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(&sm.h_full);
        mma_commit(&sm.k_empty);
        // the node products need only the a operand: they start while the
        // epilogue still forms the prototype attention from A^
        if (!kvcd::mbar_wait(&sm.ap_ready, (uint32_t)(k & 1), a.wait_ns) ||
            !kvcd::mbar_wait(&sm.v_full, (uint32_t)(k & 1), a.wait_ns)) { *abort_flag = 1; break; }
        tc_fence_after();
        bool ok = true;
        // operand descriptors: the start-address field counts 16-byte units, so
        // a key step or another operand block is an addition to the base
        const uint64_t dA0 = sw128_desc(kvcd::smem_u32(sm.Ap[0][0]));
        const uint64_t dV0 = sw128_mn_desc(kvcd::smem_u32(sm.Vt[0]), kBlockBytes);
        static_assert(sizeof(sm.Ap[0][0]) == kBlockBytes, "Ap blocks are contiguous");
        // the leaf products must not see the isolated tokens: their V rows are
        // zeroed (and kept) until the leaves are done, then put back for the
        // depth-2 and higher products
        if (sal_any) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            if (salc[g] < 0) continue;
#pragma unroll
            for (int fb = 0; fb < 2; ++fb) {
              uint4* row = reinterpret_cast<uint4*>(&sm.Vt[fb][(2 * g) * 2048 + salc[g] * 128]);
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                sm.vsave[g][fb][c] = row[c];
                row[c] = make_uint4(0, 0, 0, 0);
              }
            }
          }
          kvcd::fence_proxy_async_smem();
        }
        // the root (last in the order) is the sum of the two depth-1 nodes: the
        // epilogue adds their buffers, so 14 nodes a slot have products
#pragma unroll
        for (int pj = 0; pj < kMmaNodes; ++pj) {
          const int j = kNodeOrder[pj];
          const int nn = k * kMmaNodes + pj, bf = pj & 1;
          if (pj == 8 && sal_any) {                  // leaf products done: the rows go back
            mma_commit(&sm.mid_done);
            if (!kvcd::mbar_wait(&sm.mid_done, (uint32_t)(nmid & 1), a.wait_ns)) { ok = false; break; }
            ++nmid;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              if (salc[g] < 0) continue;
#pragma unroll
              for (int fb = 0; fb < 2; ++fb) {
                uint4* row = reinterpret_cast<uint4*>(&sm.Vt[fb][(2 * g) * 2048 + salc[g] * 128]);
#pragma unroll
                for (int c = 0; c < 8; ++c) row[c] = sm.vsave[g][fb][c];
              }
            }
            kvcd::fence_proxy_async_smem();
          }
          if (nn >= 2 && !kvcd::mbar_wait(&sm.nempty[bf], (uint32_t)(((nn >> 1) - 1) & 1), a.wait_ns)) { ok = false; break; }
          tc_fence_after();
          int l0, l1;
          node_leaves(j, l0, l1);
          const uint32_t d = tmem + 256 + bf * 128;
#pragma unroll
          for (int part = 0; part < 3; ++part)
#pragma unroll
            for (int ks = l0; ks < l1; ++ks) {
              const uint64_t aa =
                  dA0 + (uint64_t)((part * 2 + (ks >> 2)) * (kBlockBytes >> 4) + (ks & 3) * 2);
              const uint64_t bb = dV0 + (uint64_t)(ks * (2048 >> 4));
              mma_bf16_i(d, aa, bb, kIdescVmn, (part > 0 || ks > l0) ? 1u : 0u);
            }
          mma_commit(&sm.nfull[bf]);
        }
        if (!ok) { *abort_flag = 1; break; }
        mma_commit(&sm.b_done);
        mma_commit(&sm.v_empty);
      }
      if (*abort_flag) {                               // issued MMAs finish before TMEM is freed
        mma_commit(&sm.mma_done);
        kvcd::mbar_wait(&sm.mma_done, 0);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue groups
    const int g = warp >> 2, q = warp & 3;          // group (feature / key quarter), row quarter
    const int rl = q * 32 + lane;                   // row within the tile (TMEM lane)
    const int rho = mt * kBM + rl;
    const bool rv = rho < R;
    const float l2 = rv ? a.lse2[blh * R + rho] : 0.f;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int qbar = 1 + q;                          // the 4 warps sharing these rows
    for (int k = 0; k < nsl; ++k) {
      const int s = s_begin + k;
      const long long tree = blh * a.S_max + s;
      const int x0 = bd[s], y0 = bd[s + 1];
      const uint8_t* cuts = a.tree_cuts ? a.tree_cuts + tree * 8 : nullptr;
      // ---- epilogue A: attention of this row to the slot's nodes and its key quarter
      if (!*abort_flag && !kvcd::mbar_wait(&sm.s_full, (uint32_t)(k & 1), a.wait_ns)) *abort_flag = 1;
      tc_fence_after();
      int cnt0, cnt1, salc;
      {
        int st;
        leaf_range(cuts, 2 * g, x0, y0, st, cnt0);
        leaf_range(cuts, 2 * g + 1, x0, y0, st, cnt1);
        int a2, b2;
        kvcd::tree_node_range(cuts, 3 + g, x0, y0, a2, b2);
        salc = kvcd::tree_extract(cuts, 3 + g, x0, a2, b2) >= 0 ? 1 : 0;   // at column cnt0
      }
      float at_acc = 0.f;                              // a of the isolated token
      if (k >= 1 && !*abort_flag && !kvcd::mbar_wait(&sm.b_done, (uint32_t)((k - 1) & 1), a.wait_ns))
        *abort_flag = 1;
      float lsum[2];
#pragma unroll
      for (int hq = 0; hq < 2; ++hq) {                 // leaf 2g + hq: key slots 32g + 16hq ..
        float v[16];
        tmem_ld16_nw(tmem + lane_off + (uint32_t)(32 * g + 16 * hq), v);
        tmem_wait();
        const int cntl = hq ? cnt1 : cnt0;
        const int cntv = hq ? cnt1 : cnt0 + salc;      // key slots that carry a
        float sacc = 0.f;
        uint32_t pk[3][8];
#pragma unroll
        for (int t = 0; t < 16; t += 2) {
          float av[2];
#pragma unroll
          for (int u = 0; u < 2; ++u)
            av[u] = (rv && t + u < cntv) ? kvcd::ex2(v[t + u] * a.q_scale2 - l2) : 0.f;
          const float in0 = t < cntl ? av[0] : 0.f, in1 = t + 1 < cntl ? av[1] : 0.f;
          sacc += in0 + in1;
          at_acc += (av[0] - in0) + (av[1] - in1);     // the isolated token's column only
          // a = p0 + p1 + p2 in bf16 pairs (element t in the low half)
          const __nv_bfloat162 p0 = __floats2bfloat162_rn(av[0], av[1]);
          const float2 f0 = __bfloat1622float2(p0);
          const float r0 = av[0] - f0.x, r1 = av[1] - f0.y;
          const __nv_bfloat162 p1 = __floats2bfloat162_rn(r0, r1);
          const float2 f1 = __bfloat1622float2(p1);
          const __nv_bfloat162 p2 = __floats2bfloat162_rn(r0 - f1.x, r1 - f1.y);
          pk[0][t >> 1] = *reinterpret_cast<const uint32_t*>(&p0);
          pk[1][t >> 1] = *reinterpret_cast<const uint32_t*>(&p1);
          pk[2][t >> 1] = *reinterpret_cast<const uint32_t*>(&p2);
        }
        lsum[hq] = sacc;
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const int kap = 32 * g + 16 * hq + ch * 8;
          const int kb = kap >> 6, cidx = (kap & 63) >> 3;
          const int off = rl * 128 + ((cidx ^ (rl & 7)) << 4);
#pragma unroll
          for (int pt = 0; pt < 3; ++pt)
            *reinterpret_cast<uint4*>(&sm.Ap[pt][kb][off]) =
                make_uint4(pk[pt][ch * 4], pk[pt][ch * 4 + 1], pk[pt][ch * 4 + 2], pk[pt][ch * 4 + 3]);
        }
      }
      sm.Al[2 * g][rl] = lsum[0];
      sm.Al[2 * g + 1][rl] = lsum[1];
      sm.At[g][rl] = at_acc;
      kvcd::fence_proxy_async_smem();                // the a operand, visible to the MMAs
      tc_fence_before();
      __syncwarp();
      if (lane == 0) kvcd::mbar_arrive(&sm.ap_ready);
      // the attention of this row to the 15 node prototypes, from A^ (its
      // product waited for the previous slot's partials, so it comes last)
      if (!*abort_flag && !kvcd::mbar_wait(&sm.h_full, (uint32_t)(k & 1), a.wait_ns)) *abort_flag = 1;
      tc_fence_after();
      float ah[15];
      {
        float d0[16], d1[16], d2[16];
        tmem_ld16_nw(tmem + lane_off + 128, d0);
        tmem_ld16_nw(tmem + lane_off + 144, d1);
        tmem_ld16_nw(tmem + lane_off + 160, d2);
        tmem_wait();
        const float* lmv = reinterpret_cast<const float*>(sm.Kh + kvc::kProtoLogmOff);
#pragma unroll
        for (int j = 0; j < 15; ++j) {
          const float sc = (d0[j] + d1[j] + d2[j]) * a.q_scale2 + lmv[j] * 1.4426950408889634f - l2;
          ah[j] = rv ? kvcd::ex2(sc) : 0.f;
        }
      }
      kvcd::fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) kvcd::mbar_arrive(&sm.a_ready);
      named_bar(qbar, 128);                          // leaf masses of these rows complete
      float an_fin[4];                               // masses of the nodes at positions g, g+4, ...
      {
        float an[15];
#pragma unroll
        for (int l = 0; l < 8; ++l) an[7 + l] = sm.Al[l][rl];
#pragma unroll
        for (int j = 6; j >= 0; --j)
          an[j] = an[2 * j + 1] + an[2 * j + 2] + (j >= 3 ? sm.At[j - 3][rl] : 0.f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float v = 0.f;
#pragma unroll
          for (int pj = i * 4; pj < i * 4 + 4 && pj < 15; ++pj)
            if ((pj & 3) == g) v = an[kNodeOrder[pj]];
          an_fin[i] = v;
        }
      }
      if (!*abort_flag && !kvcd::mbar_wait(&sm.vh_full, (uint32_t)(k & 1), a.wait_ns)) *abort_flag = 1;
      // ---- epilogue B: 32 features of every node
#pragma unroll
      for (int pj = 0; pj < 15; ++pj) {
        const int j = kNodeOrder[pj];
        const uint64_t nah = f2(-ah[j], -ah[j]);
        const ulonglong2* w2 = reinterpret_cast<const ulonglong2*>(&sm.vh[j][32 * g]);
        uint64_t dd0 = 0, dd1 = 0, uu0 = 0, uu1 = 0;
        // features 16h .. 16h + 15 of this group's 32
        auto accumulate = [&](const float (&v)[16], int h) {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const ulonglong2 w = w2[4 * h + t];
            const uint64_t ua = f2(v[4 * t], v[4 * t + 1]), ub = f2(v[4 * t + 2], v[4 * t + 3]);
            const uint64_t da = fma2(nah, w.x, ua), db = fma2(nah, w.y, ub);
            dd0 = fma2(da, da, dd0);
            dd1 = fma2(db, db, dd1);
            uu0 = fma2(ua, ua, uu0);
            uu1 = fma2(ub, ub, uu1);
          }
        };
        if (pj < kMmaNodes) {
          const int nn = k * kMmaNodes + pj, bf = pj & 1;
          if (!*abort_flag && !kvcd::mbar_wait(&sm.nfull[bf], (uint32_t)((nn >> 1) & 1), a.wait_ns)) *abort_flag = 1;
          tc_fence_after();
          float v[32];
          tmem_ld32_nw(tmem + lane_off + 256 + bf * 128 + 32 * g, v);
          tmem_wait();
          if (pj < kMmaNodes - 2) {                   // the depth-1 buffers stay for the root
            tc_fence_before();
            __syncwarp();
            if (lane == 0) kvcd::mbar_arrive(&sm.nempty[bf]);
          }
          accumulate(*reinterpret_cast<const float(*)[16]>(&v[0]), 0);
          accumulate(*reinterpret_cast<const float(*)[16]>(&v[16]), 1);
        } else {
          // root: U = U(node 1) + U(node 2), from buffers 0 and 1, in two halves
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float u1[16], u2[16];
            tmem_ld16_nw(tmem + lane_off + 256 + 32 * g + 16 * h, u1);
            tmem_ld16_nw(tmem + lane_off + 384 + 32 * g + 16 * h, u2);
            tmem_wait();
            if (h == 1) {                              // both depth-1 buffers are read
              tc_fence_before();
              __syncwarp();
              if (lane == 0) {
                kvcd::mbar_arrive(&sm.nempty[0]);
                kvcd::mbar_arrive(&sm.nempty[1]);
              }
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) u1[i] += u2[i];
            accumulate(u1, h);
          }
        }
        // this group's partial sums of the node go to TMEM; the four groups
        // meet once the slot's 15 nodes are done
        tmem_st2(tmem + lane_off + part_col(pj, g), hsum2(dd0) + hsum2(dd1), hsum2(uu0) + hsum2(uu1));
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      named_bar(qbar, 128);
      tc_fence_after();
      // group g finishes the nodes at positions g, g + 4, g + 8, g + 12: it
      // adds the groups' partials in group order and sums |A - A^|, A,
      // |U - A^ v^| and |U| over its 32 rows (16 sums reduced together)
      {
        float pp[4][8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int pos = 4 * i + g < 15 ? 4 * i + g : 4 * i;   // position 15: none (read, unused)
          uint32_t r[8];
          asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                       : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                         "=r"(r[6]), "=r"(r[7])
                       : "r"(tmem + lane_off + part_col(pos, 0)));
#pragma unroll
          for (int e = 0; e < 8; ++e) pp[i][e] = __uint_as_float(r[e]);
        }
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        float st[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const bool real = 4 * i + g < 15 && rv;
          const float ddt = (pp[i][0] + pp[i][2]) + (pp[i][4] + pp[i][6]);
          const float uut = (pp[i][1] + pp[i][3]) + (pp[i][5] + pp[i][7]);
          float ahj = 0.f;
#pragma unroll
          for (int pq = i * 4; pq < i * 4 + 4 && pq < 15; ++pq)
            if ((pq & 3) == g) ahj = ah[kNodeOrder[pq]];
          st[4 * i + 0] = real ? fabsf(an_fin[i] - ahj) : 0.f;
          st[4 * i + 1] = real ? an_fin[i] : 0.f;
          st[4 * i + 2] = real ? sqrtf(ddt) : 0.f;
          st[4 * i + 3] = real ? sqrtf(uut) : 0.f;
        }
        // reduce-scatter over the lanes: after it, lanes 2v and 2v + 1 hold
        // the warp total of value v
#pragma unroll
        for (int o = 16, n = 8; o >= 2; o >>= 1, n >>= 1) {
          const bool hi = (lane & o) != 0;
#pragma unroll
          for (int i = 0; i < n; ++i) {
            const float send = hi ? st[i] : st[i + n];
            const float keep = hi ? st[i + n] : st[i];
            st[i] = keep + __shfl_xor_sync(KVC_FULL_MASK, send, o);
          }
        }
        st[0] += __shfl_xor_sync(KVC_FULL_MASK, st[0], 1);
        const int vi = lane >> 1, ni = vi >> 2;        // value, node of the group
        if (!(lane & 1) && 4 * ni + g < 15) {
          int jj = 0;
#pragma unroll
          for (int pq = 0; pq < 15; ++pq)
            if ((pq & 3) == g && (pq >> 2) == ni) jj = kNodeOrder[pq];
          sm.red[k & 1][q][jj][vi & 3] = st[0];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) kvcd::mbar_arrive(&sm.xch_free);   // the partial columns are free
      named_bar(5, kEpiWarps * 32);                  // every node of this slot finished
      if (tid < 60) {
        const int j = tid >> 2, e = tid & 3;
        const float t = (sm.red[k & 1][0][j][e] + sm.red[k & 1][1][j][e]) +
                        (sm.red[k & 1][2][j][e] + sm.red[k & 1][3][j][e]);
        a.npart[((tree * 2 + mt) * 15 + j) * 4 + e] = t;
      }
      if (lane == 0) kvcd::mbar_arrive(&sm.vh_free);
    }
  }

  __syncthreads();
  if (*abort_flag && tid == 0) kvcd::record_error(a.err, KVC_ETIMEOUT);
  tc_fence_after();
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512u)
                 : "memory");
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

template <int MODE, int PN>
int launch_t(const CUtensorMap& map, const kvc::ProbeTcArgs& a, cudaStream_t s) {
  constexpr int NT = MODE == kvc::kTcFeats ? 2 : 1;
  constexpr int kThreads = kRsThreads;
  const size_t smem = sizeof(TcTSmem<NT>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(probe_tcT_kernel<MODE, PN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return kvc::cuda_status(e);
  dim3 grid(a.n_chunks, (unsigned)((long long)a.B * a.L * a.H));
  probe_tcT_kernel<MODE, PN><<<grid, kThreads, smem, s>>>(map, a);
  kvc::count_launch();
  return kvc::cuda_status(cudaGetLastError());
}

template <int NT, int MODE>
int launch(const CUtensorMap& map, const kvc::ProbeTcArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(TcSmem<NT>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(probe_tc_kernel<NT, MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return KVC_ECUDA;
  dim3 grid(a.n_chunks, (unsigned)((long long)a.B * a.L * a.H));
  probe_tc_kernel<NT, MODE><<<grid, kRsThreads, smem, s>>>(map, a);
  kvc::count_launch();
  return kvc::cuda_status(cudaGetLastError());
}

}  // namespace

namespace kvc {

bool probe_tc_supported(const kvc_params* p) {
  return p->dtype == KVC_BF16 && p->d == 128 && p->P % 32 == 0 && p->G * p->P <= 256 &&
         p->P <= 128 && encode_fn() != nullptr;
}

int probe_tc_pass(int mode, const ProbeTcArgs& a, int64_t total_rows, cudaStream_t s) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return KVC_ECUDA;
  CUtensorMap map;
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)total_rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kBN};
  cuuint32_t estr[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.K), dims, strides, box,
          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return KVC_ECUDA;
  const bool two = a.G * a.P > 128;
  switch (mode) {
    case kTcRowstatsProbes:
      return two ? launch<2, kTcRowstatsProbes>(map, a, s) : launch<1, kTcRowstatsProbes>(map, a, s);
    case kTcFeats:
      return launch_t<kTcFeats, 0>(map, a, s);
    case kTcRowstatsSeeds:
      return launch<1, kTcRowstatsSeeds>(map, a, s);
    default:
      return a.P <= 64 ? launch_t<kTcProp, 64>(map, a, s) : launch_t<kTcProp, 128>(map, a, s);
  }
}

}  // namespace kvc

namespace kvc {

int nodes_tc_pass(const NodeTcArgs& a, int64_t total_rows, cudaStream_t s) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return KVC_ECUDA;
  CUtensorMap km, vm;
  cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)total_rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {64, 16};
  cuuint32_t estr[2] = {1, 1};
  if (enc(&km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.K), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return KVC_ECUDA;
  if (enc(&vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.V), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return KVC_ECUDA;
  const size_t smem = sizeof(NodeSmem) + 1024;
  if (cudaFuncSetAttribute(nodes_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return KVC_ECUDA;
  const int n_mt = (a.G * a.P + kBM - 1) / kBM;
  dim3 grid((a.S_max + kNodeSlots - 1) / kNodeSlots, n_mt, (unsigned)((long long)a.B * a.L * a.H));
  nodes_tc_kernel<<<grid, kNodeThreads, smem, s>>>(km, vm, a);
  kvc::count_launch();
  return kvc::cuda_status(cudaGetLastError());
}

size_t nodes_tc_smem_bytes() { return sizeof(NodeSmem) + 1024; }

}  // namespace kvc
