// NEXT f2: per-step top-B eviction (DistillCache Algorithm 1 with the
// heuristic score alpha: the learned policy is replaced by its first feature,
// DistillCache 3.1.1).  The cache of a sequence holds the same tokens, in the
// same rows, in every (layer, KV head): len_lh is equal across the (l,h) of a
// sequence and row i is one token everywhere.
//
//   kvc_token_alpha   alpha_i = mean over (l, h, g) of the step's attention
//                     probability of row i, from the per-head base-2 LSE that
//                     kvc_decode_attn_lse wrote (the new token included).  The
//                     (l,h) of a sequence are split into groups; one CTA sums a
//                     tile of rows over one group, and a second kernel adds the
//                     group partials in group order, so the result is
//                     deterministic.  The scores come from the decode step
//                     (16 bytes per row and head for G = 4: the pass streams a
//                     sixteenth of K's bytes) or, without them, are recomputed
//                     in fp32 from K tiles staged through shared memory.
//   kvc_evict_topb    per sequence B = min(len, max(floor(r * n_seen), B_min));
//                     the B rows of largest (alpha, -position) are kept (ties go
//                     to the earlier token; one 64-bit key per row, a radix
//                     select in one CTA that stops once the cut is resolved).
//                     Eviction is in place: the kept rows beyond B move into the
//                     evicted rows below B, so only those rows are copied (one
//                     row per step in the steady state) and the row order stops
//                     following the position order.
#include <math.h>

#include <algorithm>

#include "kvc_common.cuh"
#include "kvc_internal.h"

namespace {

constexpr int kAlphaTok = 128;       // rows per alpha CTA
constexpr int kAlphaGroups = 32;     // at most this many (l,h) groups per sequence
constexpr int kPlanThreads = 1024;   // top-B CTA (one per sequence)
constexpr int kMoveRows = 32;        // row moves per CTA

struct EvictLayout {
  size_t part, dst, src, meta, total;
};

int alpha_groups(const kvc_params* p) {
  const int LH = p->L * p->H;
  const int ng = LH < kAlphaGroups ? LH : kAlphaGroups;
  const int per = (LH + ng - 1) / ng;
  return (LH + per - 1) / per;
}

EvictLayout evict_layout(const kvc_params* p, int cols) {
  EvictLayout w;
  w.part = 0;
  w.dst = kvc::align256(sizeof(float) * (size_t)p->B * alpha_groups(p) * cols);
  w.src = w.dst + kvc::align256(sizeof(int32_t) * (size_t)p->B * cols);
  w.meta = w.src + kvc::align256(sizeof(int32_t) * (size_t)p->B * cols);
  w.total = w.meta + kvc::align256(sizeof(int32_t) * 2 * (size_t)p->B);
  return w;
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(kvcd::smem_u32(smem)),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// Shared memory of one alpha CTA: two K tiles (this head, the next) and their
// scaled queries and LSEs.  A tile row is kChunks 16-byte chunks stored at
// chunk ^ (row mod kChunks), so the rows' chunk c that 32 threads read at once
// spread over all banks.
template <typename T, int D>
struct AlphaSmem {
  static constexpr int kChunks = D * (int)sizeof(T) / 16;
  uint4 tile[2][kAlphaTok * kChunks];
  float sq[2][8][D];
  float sl[2][8];
};

// Partial alpha of a 128-row tile over one group of (l,h): the group's K tiles
// stream through shared memory with asynchronous 16-byte copies (each warp
// reads whole rows), the next head's tile loading while this one is summed.
template <typename T, int D>
__global__ void __launch_bounds__(kAlphaTok) alpha_part_kernel(
    kvc_params p, const T* q, const T* Kp, const int32_t* len_lh, const int64_t* off_lh,
    const float* lse2, float* part, int cols, int n_groups, int per_group, float scale_log2,
    int32_t* err) {
  using Sm = AlphaSmem<T, D>;
  constexpr int kChunks = Sm::kChunks;
  constexpr int kElems = 16 / (int)sizeof(T);          // elements per chunk
  constexpr int G_MAX = 8;
  extern __shared__ __align__(16) unsigned char alpha_smem_raw[];
  Sm& sm = *reinterpret_cast<Sm*>(alpha_smem_raw);
  const int b = blockIdx.z, grp = blockIdx.y;
  const int LH = p.L * p.H;
  const int G = p.G;
  const int len = len_lh[(int64_t)b * LH];
  const int row0 = blockIdx.x * kAlphaTok;
  const int r = threadIdx.x, i = row0 + r;
  if (len < 0 || len > cols) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && grp == 0) kvcd::record_error(err, KVC_EDEVICE);
    return;
  }
  if (row0 >= len) return;
  const int lh0 = grp * per_group, lh1 = min(LH, lh0 + per_group);
  const int rows = min(kAlphaTok, len - row0);
  auto stage = [&](int buf, int lh) {
    const int64_t blh = (int64_t)b * LH + lh;
    const T* src = Kp + (off_lh[blh] + row0) * D;
    for (int e = threadIdx.x; e < rows * kChunks; e += kAlphaTok) {
      const int rr = e / kChunks, c = e % kChunks;
      cp_async16(&sm.tile[buf][rr * kChunks + (c ^ (rr % kChunks))], src + (int64_t)rr * D + c * kElems);
    }
    for (int t = threadIdx.x; t < G * D; t += kAlphaTok) {
      const int g = t / D, f = t % D;
      sm.sq[buf][g][f] = kvcd::to_f(q[(blh * G + g) * D + f]) * scale_log2;
    }
    if (threadIdx.x < G) sm.sl[buf][threadIdx.x] = lse2[blh * G + threadIdx.x];
    cp_async_commit();
  };
  float acc = 0.f;
  stage(0, lh0);
  for (int lh = lh0; lh < lh1; ++lh) {
    const int buf = (lh - lh0) & 1;
    if (lh + 1 < lh1) {
      stage(buf ^ 1, lh + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const int64_t blh = (int64_t)b * LH + lh;
    if (len_lh[blh] != len) {                          // lengths must agree across (l,h)
      if (threadIdx.x == 0) kvcd::record_error(err, KVC_EDEVICE);
    } else if (r < rows) {
      float s[G_MAX];
#pragma unroll
      for (int g = 0; g < G_MAX; ++g) s[g] = 0.f;
#pragma unroll 4
      for (int c = 0; c < kChunks; ++c) {
        const uint4 w = sm.tile[buf][r * kChunks + (c ^ (r % kChunks))];
        float kv[kElems];
        if constexpr (sizeof(T) == 2) {
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            kv[2 * u] = __uint_as_float(ws[u] << 16);
            kv[2 * u + 1] = __uint_as_float(ws[u] & 0xFFFF0000u);
          }
        } else {
          kv[0] = __uint_as_float(w.x); kv[1] = __uint_as_float(w.y);
          kv[2] = __uint_as_float(w.z); kv[3] = __uint_as_float(w.w);
        }
#pragma unroll
        for (int g = 0; g < G_MAX; ++g)
          if (g < G)
#pragma unroll
            for (int u = 0; u < kElems; ++u) s[g] = fmaf(sm.sq[buf][g][c * kElems + u], kv[u], s[g]);
      }
#pragma unroll
      for (int g = 0; g < G_MAX; ++g)
        if (g < G) acc += exp2f(s[g] - sm.sl[buf][g]);
    }
    __syncthreads();                                    // buf is refilled two heads on
  }
  if (i < len) part[((int64_t)b * n_groups + grp) * cols + i] = acc;
}

// Partial alpha from the scores the decode step exported: one thread per row,
// the group's (l,h) rows streamed as G-float vectors (rows of a head are
// contiguous, so a warp reads 32 consecutive vectors).
template <int G>
__global__ void __launch_bounds__(256) alpha_scores_kernel(
    kvc_params p, const float* scores, const int32_t* len_lh, const int64_t* off_lh,
    const float* lse2, float* part, int cols, int n_groups, int per_group, int32_t* err) {
  const int b = blockIdx.z, grp = blockIdx.y;
  const int LH = p.L * p.H;
  const int len = len_lh[(int64_t)b * LH];
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (len < 0 || len > cols) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && grp == 0) kvcd::record_error(err, KVC_EDEVICE);
    return;
  }
  if ((int)(blockIdx.x * blockDim.x) >= len) return;
  const int lh0 = grp * per_group, lh1 = min(LH, lh0 + per_group);
  bool bad = false;
  for (int lh = lh0; lh < lh1; ++lh) bad |= len_lh[(int64_t)b * LH + lh] != len;
  if (bad) {                                            // lengths must agree across (l,h)
    if (threadIdx.x == 0) kvcd::record_error(err, KVC_EDEVICE);
    return;
  }
  if (i >= len) return;
  float acc = 0.f;
#pragma unroll 4
  for (int lh = lh0; lh < lh1; ++lh) {
    const int64_t blh = (int64_t)b * LH + lh;
    const float* sr = scores + (off_lh[blh] + i) * G;
    float sv[G];
    if constexpr (G == 4) {
      const float4 v = __ldcs(reinterpret_cast<const float4*>(sr));
      sv[0] = v.x; sv[1] = v.y; sv[2] = v.z; sv[3] = v.w;
    } else if constexpr (G == 8) {
      const float4 v0 = __ldcs(reinterpret_cast<const float4*>(sr));
      const float4 v1 = __ldcs(reinterpret_cast<const float4*>(sr) + 1);
      sv[0] = v0.x; sv[1] = v0.y; sv[2] = v0.z; sv[3] = v0.w;
      sv[4] = v1.x; sv[5] = v1.y; sv[6] = v1.z; sv[7] = v1.w;
    } else {
#pragma unroll
      for (int g = 0; g < G; ++g) sv[g] = __ldcs(sr + g);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) acc += exp2f(sv[g] - __ldg(lse2 + blh * G + g));
  }
  part[((int64_t)b * n_groups + grp) * cols + i] = acc;
}

__global__ void alpha_sum_kernel(kvc_params p, const int32_t* len_lh, const float* part,
                                 float* alpha, int cols, int n_groups) {
  const int b = blockIdx.y;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int len = len_lh[(int64_t)b * p.L * p.H];
  if (len < 0 || len > cols || i >= len) return;
  float a = 0.f;
  for (int g = 0; g < n_groups; ++g) a += part[((int64_t)b * n_groups + g) * cols + i];
  alpha[(int64_t)b * cols + i] = a / (float)(p.L * p.H * p.G);
}

// ---------------------------------------------------------------- top-B plan
// Row key: alpha's order-preserving code above the complement of the token's
// position, so equal alphas order by the earlier token.  Keys are distinct
// while positions are.
__device__ __forceinline__ unsigned long long row_key(float a, float pos) {
  return ((unsigned long long)kvcd::float_key(a) << 32) |
         (unsigned long long)(0xffffffffu - (uint32_t)pos);
}

// Exclusive block prefix of `v` (blockDim.x == kPlanThreads); returns the total.
__device__ int block_exclusive_scan(int v, int* s_warp, int& excl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(KVC_FULL_MASK, incl, o);
    if (lane >= o) incl += u;
  }
  __syncthreads();
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(KVC_FULL_MASK, w, o);
      if (lane >= o) w += u;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  excl = incl - v + (warp > 0 ? s_warp[warp - 1] : 0);
  return s_warp[31];
}

// One CTA per sequence: the kept set and the (hole <- kept tail row) move list.
__global__ void __launch_bounds__(kPlanThreads) topb_plan_kernel(
    kvc_params p, const int32_t* len_lh, const int64_t* off_lh, const float* pos,
    const float* alpha, int cols, const int64_t* n_seen, double ratio, int b_min, int32_t* dst,
    int32_t* src, int32_t* meta, int32_t* err) {
  const int b = blockIdx.x;
  const int LH = p.L * p.H;
  const int len = len_lh[(int64_t)b * LH];
  const float* a = alpha + (int64_t)b * cols;
  const float* ps = pos + off_lh[(int64_t)b * LH];
  int32_t* db = dst + (int64_t)b * cols;
  int32_t* sb = src + (int64_t)b * cols;
  __shared__ unsigned int hist[256];
  __shared__ unsigned long long s_prefix;
  __shared__ long long s_rem;
  __shared__ int s_done;
  __shared__ int s_warp[32];
  if (len < 0 || len > cols || n_seen[b] < 0) {
    if (threadIdx.x == 0) { kvcd::record_error(err, KVC_EDEVICE); meta[2 * b] = -1; }
    return;
  }
  const long long Bq = max((long long)floor(ratio * (double)n_seen[b]), (long long)b_min);
  const int B = (int)min((long long)len, Bq);
  const bool keep_all = B >= len, keep_none = B <= 0;
  if (threadIdx.x == 0) { s_prefix = 0ull; s_rem = B; s_done = keep_all || keep_none; }
  __syncthreads();
  // the cut: the largest prefix value with at least B keys at or above it
  for (int pass = 0; pass < 8; ++pass) {
    if (s_done) break;
    const int shift = 56 - 8 * pass;
    const unsigned long long hi_mask = pass == 0 ? 0ull : (~0ull << (shift + 8));
    for (int t = threadIdx.x; t < 256; t += blockDim.x) hist[t] = 0u;
    __syncthreads();
    const unsigned long long pre = s_prefix;
    for (int i = threadIdx.x; i < len; i += blockDim.x) {
      const unsigned long long k = row_key(a[i], ps[i]);
      if ((k & hi_mask) == (pre & hi_mask)) atomicAdd(&hist[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l owns digits 255-8l .. 248-8l (descending); the lane whose running
      // count from the top first reaches rem holds the cut digit
      const int lane = threadIdx.x;
      unsigned int cnt[8];
      unsigned int mine = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) { cnt[u] = hist[255 - 8 * lane - u]; mine += cnt[u]; }
      unsigned int incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned int v = __shfl_up_sync(KVC_FULL_MASK, incl, o);
        if (lane >= o) incl += v;
      }
      const long long rem0 = s_rem;
      const unsigned int hit = __ballot_sync(KVC_FULL_MASK, (long long)incl >= rem0);
      const int ln = __ffs(hit) - 1;                 // rem0 <= keys left, so some lane hits
      if (lane == ln) {
        long long rem = rem0 - (long long)(incl - mine);
        int dsel = 255 - 8 * lane;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if ((long long)cnt[u] >= rem) { dsel = 255 - 8 * lane - u; break; }
          rem -= cnt[u];
        }
        s_prefix = pre | ((unsigned long long)dsel << shift);
        s_rem = rem;
        s_done = (long long)hist[dsel] == rem;   // every key with this prefix is kept
      }
    }
    __syncthreads();
  }
  const unsigned long long thr = s_prefix;
  auto kept = [&](int i) -> bool {
    return keep_all || (!keep_none && row_key(a[i], ps[i]) >= thr);
  };
  // holes: evicted rows below B; movers: kept rows at or above B (as many)
  const int per = (len + blockDim.x - 1) / blockDim.x;
  const int i0 = min(len, (int)threadIdx.x * per), i1 = min(len, i0 + per);
  int nh = 0, nv = 0;
  for (int i = i0; i < i1; ++i) {
    const bool k = kept(i);
    nh += (i < B) && !k;
    nv += (i < B) ? !k : k;
  }
  int ex_h, ex_v;
  const int holes = block_exclusive_scan(nh, s_warp, ex_h);
  const int total = block_exclusive_scan(nv, s_warp, ex_v);
  int r = ex_v;
  for (int i = i0; i < i1; ++i) {
    const bool k = kept(i);
    if (i < B && !k) db[r++] = i;
    else if (i >= B && k) sb[r++ - holes] = i;
  }
  if (threadIdx.x == 0) {
    meta[2 * b] = holes;
    meta[2 * b + 1] = B;
    if (total != 2 * holes) kvcd::record_error(err, KVC_EDEVICE);   // never: keys are distinct
  }
}

// Every (b,l,h): row src[j] moves to row dst[j] (K, V, log m, pos), then len = B.
template <typename T, int D>
__global__ void evict_move_kernel(kvc_params p, T* K, T* V, float* pos, float* logm,
                                  const int64_t* off_lh, int32_t* len_lh, const int32_t* dst,
                                  const int32_t* src, const int32_t* meta, int cols) {
  constexpr int kVec = D * (int)sizeof(T) / 16;       // 16-byte vectors per row
  const int64_t blh = blockIdx.y;
  const int b = (int)(blh / (p.L * p.H));
  const int np = meta[2 * b];
  if (np < 0) return;
  const int64_t off = off_lh[blh];
  const int32_t* db = dst + (int64_t)b * cols;
  const int32_t* sb = src + (int64_t)b * cols;
  for (int j0 = blockIdx.x * kMoveRows; j0 < np; j0 += gridDim.x * kMoveRows) {
    for (int e = threadIdx.x; e < kMoveRows * kVec; e += blockDim.x) {
      const int j = j0 + e / kVec, v = e % kVec;
      if (j >= np) continue;
      const int64_t s = off + sb[j], d = off + db[j];
      reinterpret_cast<uint4*>(K + d * D)[v] = reinterpret_cast<const uint4*>(K + s * D)[v];
      reinterpret_cast<uint4*>(V + d * D)[v] = reinterpret_cast<const uint4*>(V + s * D)[v];
    }
    for (int j = j0 + threadIdx.x; j < min(np, j0 + kMoveRows); j += blockDim.x) {
      const int64_t s = off + sb[j], d = off + db[j];
      pos[d] = pos[s];
      logm[d] = logm[s];
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) len_lh[blh] = meta[2 * b + 1];
}

template <typename T, int D>
void launch_alpha(const kvc_params* p, const void* q, const void* Kp, const int32_t* len_lh,
                  const int64_t* off_lh, const float* lse2, float* part, int cols, int ng,
                  int per, int32_t* err, cudaStream_t s) {
  dim3 grid((cols + kAlphaTok - 1) / kAlphaTok, ng, p->B);
  const float sc = 1.4426950408889634f / sqrtf((float)p->d);
  const int smem = (int)sizeof(AlphaSmem<T, D>);
  cudaFuncSetAttribute(alpha_part_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  alpha_part_kernel<T, D><<<grid, kAlphaTok, smem, s>>>(*p, static_cast<const T*>(q),
                                                        static_cast<const T*>(Kp), len_lh, off_lh,
                                                        lse2, part, cols, ng, per, sc, err);
}

template <typename T, int D>
void launch_move(const kvc_params* p, void* K, void* V, float* pos, float* logm,
                 const int64_t* off_lh, int32_t* len_lh, const int32_t* dst, const int32_t* src,
                 const int32_t* meta, int cols, cudaStream_t s) {
  // at most min(B, len - B) <= cols / 2 moves per (l,h), usually a handful: a
  // grid of about 4 CTAs per SM strides over them
  const int64_t blh = kvc::lh_count(p);
  const int need = (cols / 2 + kMoveRows) / kMoveRows;
  const int64_t sms = std::max(1, kvc::sm_count());
  const int x = (int)std::max<int64_t>(1, std::min<int64_t>(need, (4 * sms + blh - 1) / blh));
  dim3 grid(x, (unsigned)blh);
  evict_move_kernel<T, D><<<grid, 128, 0, s>>>(*p, static_cast<T*>(K), static_cast<T*>(V), pos,
                                               logm, off_lh, len_lh, dst, src, meta, cols);
}

}  // namespace

extern "C" size_t kvc_evict_workspace_bytes(const kvc_params* p, int32_t alpha_cols) {
  if (kvc::check_params(p) != KVC_OK || alpha_cols < 1) return 0;
  return evict_layout(p, alpha_cols).total;
}

extern "C" int kvc_token_alpha(const kvc_params* p, const void* q, const void* Kp,
                               const float* scores, const int32_t* len_lh, const int64_t* off_lh,
                               const float* lse2, float* alpha, int32_t alpha_cols,
                               void* workspace, size_t ws_bytes, void* stream) {
  int st = kvc::check_params(p);
  if (st != KVC_OK) return st;
  if ((!scores && (!q || !Kp)) || !len_lh || !off_lh || !lse2 || !alpha || alpha_cols < 1)
    return KVC_EINVAL;
  if (p->B > 65535) return KVC_EINVAL;
  const EvictLayout w = evict_layout(p, alpha_cols);
  if (!workspace || ws_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return KVC_EWORKSPACE;
  int32_t* err = kvc::err_word();
  if (!err) return KVC_ECUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* part = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.part);
  const int LH = p->L * p->H;
  const int ng = alpha_groups(p);
  const int per = (LH + ng - 1) / ng;
  if (scores) {
    dim3 grid((alpha_cols + 255) / 256, ng, p->B);
    switch (p->G) {
      case 1: alpha_scores_kernel<1><<<grid, 256, 0, s>>>(*p, scores, len_lh, off_lh, lse2, part, alpha_cols, ng, per, err); break;
      case 2: alpha_scores_kernel<2><<<grid, 256, 0, s>>>(*p, scores, len_lh, off_lh, lse2, part, alpha_cols, ng, per, err); break;
      case 4: alpha_scores_kernel<4><<<grid, 256, 0, s>>>(*p, scores, len_lh, off_lh, lse2, part, alpha_cols, ng, per, err); break;
      default: alpha_scores_kernel<8><<<grid, 256, 0, s>>>(*p, scores, len_lh, off_lh, lse2, part, alpha_cols, ng, per, err); break;
    }
  } else if (p->dtype == KVC_BF16) {
    if (p->d == 128)
      launch_alpha<__nv_bfloat16, 128>(p, q, Kp, len_lh, off_lh, lse2, part, alpha_cols, ng, per, err, s);
    else
      launch_alpha<__nv_bfloat16, 64>(p, q, Kp, len_lh, off_lh, lse2, part, alpha_cols, ng, per, err, s);
  } else {
    if (p->d == 128)
      launch_alpha<float, 128>(p, q, Kp, len_lh, off_lh, lse2, part, alpha_cols, ng, per, err, s);
    else
      launch_alpha<float, 64>(p, q, Kp, len_lh, off_lh, lse2, part, alpha_cols, ng, per, err, s);
  }
  dim3 g2((alpha_cols + 255) / 256, p->B);
  alpha_sum_kernel<<<g2, 256, 0, s>>>(*p, len_lh, part, alpha, alpha_cols, ng);
  kvc::count_launch(2);
  return kvc::cuda_status(cudaGetLastError());
}

extern "C" int kvc_evict_topb(const kvc_params* p, const float* alpha, int32_t alpha_cols,
                              const int64_t* n_seen, double ratio, int32_t b_min, void* K, void* V,
                              float* pos, float* logm, const int64_t* off_lh, int32_t* len_lh,
                              void* workspace, size_t ws_bytes, void* stream) {
  int st = kvc::check_params(p);
  if (st != KVC_OK) return st;
  if (!alpha || alpha_cols < 1 || !n_seen || !(ratio >= 0.0) || b_min < 0 || !K || !V || !pos ||
      !logm || !off_lh || !len_lh)
    return KVC_EINVAL;
  const EvictLayout w = evict_layout(p, alpha_cols);
  if (!workspace || ws_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return KVC_EWORKSPACE;
  if (kvc::lh_count(p) > 65535) return KVC_EINVAL;
  int32_t* err = kvc::err_word();
  if (!err) return KVC_ECUDA;
  char* ws = static_cast<char*>(workspace);
  int32_t* dst = reinterpret_cast<int32_t*>(ws + w.dst);
  int32_t* src = reinterpret_cast<int32_t*>(ws + w.src);
  int32_t* meta = reinterpret_cast<int32_t*>(ws + w.meta);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  topb_plan_kernel<<<p->B, kPlanThreads, 0, s>>>(*p, len_lh, off_lh, pos, alpha, alpha_cols,
                                                 n_seen, ratio, b_min, dst, src, meta, err);
  if (p->dtype == KVC_BF16) {
    if (p->d == 128)
      launch_move<__nv_bfloat16, 128>(p, K, V, pos, logm, off_lh, len_lh, dst, src, meta, alpha_cols, s);
    else
      launch_move<__nv_bfloat16, 64>(p, K, V, pos, logm, off_lh, len_lh, dst, src, meta, alpha_cols, s);
  } else {
    if (p->d == 128)
      launch_move<float, 128>(p, K, V, pos, logm, off_lh, len_lh, dst, src, meta, alpha_cols, s);
    else
      launch_move<float, 64>(p, K, V, pos, logm, off_lh, len_lh, dst, src, meta, alpha_cols, s);
  }
  kvc::count_launch(2);
  return kvc::cuda_status(cudaGetLastError());
}
