// Curvature-chosen prototype trees (GraceKV "Technical details and default
// settings": tree construction considers high-curvature split candidates plus
// the midpoint; the curvature measure of "01 Curvature-guided partition").
//
// Per (b, l, h) the keys with RoPE removed, u_i = R(-i) k_i / |R(-i) k_i|, form a
// trajectory; its multi-scale curvature is
//   kappa(t) = mean over w in {1, 2, 4, 8} with w <= t < n - w of
//              1 - cos(u_t - u_{t-w}, u_{t+w} - u_t)     (cos = 1 for a zero chord).
// Every internal node [a, b) of a slot tree (depth k, c tokens, midpoint
// m = floor((a+b)/2)) is cut, top-down, at the valid t maximising
//   kappa(t) - lam * ((t - m) / (c / 2))^2,   lam = mean kappa over [a, b),
// ties to the midpoint, then to the smaller t.  Valid: both children keep
// 2..16 tokens per leaf below them (2^(2-k) leaves), the range of the midpoint
// trees' leaves, so every leaf split stores at least 2 tokens.
//
// Kernel 1 (key_curv_kernel): one CTA per (b,l,h) and 64 positions; the unit
// rows of positions [t0 - 8, t0 + 72) are staged in shared memory (a warp per
// row, 5 rows' loads in flight at once: unrotate with the half-position table
// row 2i, one warp reduction for the norm), then every lane takes one
// position and a quarter of the features (warp = 32-position group x
// quarter) and sums the 12 chord terms of the 4 scales on packed f32x2 pairs
// with no cross-lane reduction; the quarters meet in shared memory and one
// thread per position finishes the scale terms (cos = dot * rsqrt(|a|^2 |b|^2)).
// Kernel 2 (tree_cut_kernel): one warp per slot tree; the node mean is summed
// in index order by every lane (the same fp32 sum the cut decision is checked
// against), candidates are scored 32 at a time with explicitly rounded fp32
// operations (no contraction) and the warp keeps the first maximum.
#include "kvc_common.cuh"
#include "kvc_internal.h"

namespace {

// Packed pairs of fp32 (first element in the low half): one instruction
// computes a * b + c on both halves.
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ float hsum2(uint64_t x) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
  return lo + hi;
}

constexpr int kCurvTile = 64;                 // positions per CTA
constexpr int kCurvHalo = 8;                  // largest scale
constexpr int kCurvRows = kCurvTile + 2 * kCurvHalo;

struct TreeArgs {
  const int32_t* ctx_len;
  const void* K;
  const float* cos_tab;
  const float* sin_tab;
  const int32_t* bounds;
  const int32_t* n_slots;
  float* kappa;
  uint8_t* cuts;
  int32_t* err;
};

template <typename T, int D>
__global__ void __launch_bounds__(256) key_curv_kernel(kvc_params p, TreeArgs a) {
  constexpr int VP = D / 64;                   // RoPE pairs per lane
  constexpr int HALF = D / 2;
  // unit rows, padded by 2 floats so that lanes on consecutive rows hit
  // different banks; once the rows are consumed the same memory holds the
  // chord partial sums of the 4 feature quarters
  constexpr int RS = D + 2;
  static_assert(4 * 12 * kCurvTile <= kCurvRows * RS, "partials alias the rows");
  __shared__ __align__(16) float smem_f[kCurvRows * RS];
  float (*urow)[RS] = reinterpret_cast<float (*)[RS]>(smem_f);
  float (*part)[12][kCurvTile] = reinterpret_cast<float (*)[12][kCurvTile]>(smem_f);
  const long long blh = blockIdx.y;
  const int lh = (int)(blh % ((long long)p.L * p.H));
  const int b = (int)(blh / ((long long)p.L * p.H));
  const int n = a.ctx_len[b];
  const int t0 = blockIdx.x * kCurvTile;
  if (n < 1 || n > p.n_max) {
    if (threadIdx.x == 0 && blockIdx.x == 0) kvcd::record_error(a.err, KVC_EDEVICE);
    return;
  }
  if (t0 >= n) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row0 = kvcd::seq_token_base(a.ctx_len, b, p.L * p.H) + (int64_t)lh * n;
  const T* Kh = static_cast<const T*>(a.K) + row0 * D;
  if (threadIdx.x == 0) {          // the tile's key rows (contiguous) start towards L2 at once
    const int lo = max(0, t0 - kCurvHalo), hi = min(n, t0 - kCurvHalo + kCurvRows);
    kvcd::prefetch_l2(Kh + (int64_t)lo * D, (uint32_t)((hi - lo) * D * sizeof(T)));
  }
  // unit rows u_i of positions t0 - 8 .. t0 + 71 (zero outside [0, n)); each
  // warp owns rows warp, warp + 8, ..., in batches whose loads are all issued
  // before the first use
  constexpr int kRowsPerWarp = kCurvRows / 8;
  constexpr int kBatch = 5;
  static_assert(kRowsPerWarp % kBatch == 0, "row batches");
#pragma unroll 1
  for (int r0 = 0; r0 < kRowsPerWarp; r0 += kBatch) {
    float klo[kBatch][VP], khi[kBatch][VP], cs[kBatch][VP], sn[kBatch][VP];
    bool in[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int i = t0 - kCurvHalo + warp + 8 * (r0 + q);
      in[q] = i >= 0 && i < n;
      const int ic = in[q] ? i : 0;                     // a valid row, result discarded
      const T* kr = Kh + (int64_t)ic * D;
      const float* ct = a.cos_tab + (int64_t)(2 * ic) * HALF + lane * VP;
      const float* st = a.sin_tab + (int64_t)(2 * ic) * HALF + lane * VP;
      if constexpr (VP == 2) {
        kvcd::VecLoad<T, 2>::ld(kr + lane * 2, klo[q]);
        kvcd::VecLoad<T, 2>::ld(kr + HALF + lane * 2, khi[q]);
        kvcd::VecLoad<float, 2>::ld(ct, cs[q]);
        kvcd::VecLoad<float, 2>::ld(st, sn[q]);
      } else {
        klo[q][0] = kvcd::to_f(kr[lane]);
        khi[q][0] = kvcd::to_f(kr[HALF + lane]);
        cs[q][0] = __ldg(ct);
        sn[q][0] = __ldg(st);
      }
    }
    float n2[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      n2[q] = 0.f;
#pragma unroll
      for (int t = 0; t < VP; ++t) {
        const float lo = klo[q][t] * cs[q][t] + khi[q][t] * sn[q][t];     // R(-i)
        const float hi = khi[q][t] * cs[q][t] - klo[q][t] * sn[q][t];
        klo[q][t] = in[q] ? lo : 0.f;
        khi[q][t] = in[q] ? hi : 0.f;
        n2[q] += klo[q][t] * klo[q][t] + khi[q][t] * khi[q][t];
      }
    }
    static_assert(kBatch == 5, "one four-way and one single reduction");
    kvcd::warp_sum4(*reinterpret_cast<float(*)[4]>(&n2[0]), lane);
    n2[4] = kvcd::warp_sum(n2[4]);
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int r = warp + 8 * (r0 + q);
      const float inv = n2[q] > 0.f ? 1.f / sqrtf(n2[q]) : 0.f;
#pragma unroll
      for (int t = 0; t < VP; ++t) {
        urow[r][lane * VP + t] = klo[q][t] * inv;
        urow[r][HALF + lane * VP + t] = khi[q][t] * inv;
      }
    }
  }
  __syncthreads();
  // lane = position, warp = (32-position group, feature quarter): each lane
  // sums its position's 12 chord terms over a quarter of the features on packed
  // f32x2 pairs (no cross-lane reduction), the quarters meet in shared memory
  constexpr int QF = D / 4;                    // features per quarter
  const int grp = warp & 1, quarter = warp >> 1;
  const int q = grp * 32 + lane;               // position within the tile
  const int rc = q + kCurvHalo;
  const uint64_t kNeg1 = ((uint64_t)__float_as_uint(-1.f) << 32) | __float_as_uint(-1.f);
  uint64_t dt[4], aa[4], bb[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) dt[s] = aa[s] = bb[s] = 0;
  auto ld2 = [&](int row, int f) {
    return *reinterpret_cast<const unsigned long long*>(&urow[row][f]);
  };
#pragma unroll 4
  for (int f = quarter * QF; f < quarter * QF + QF; f += 2) {
    const uint64_t uc = ld2(rc, f);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int w = 1 << s;
      const uint64_t ca = fma2(ld2(rc - w, f), kNeg1, uc);      // u_t - u_{t-w}
      const uint64_t cb = fma2(uc, kNeg1, ld2(rc + w, f));      // u_{t+w} - u_t
      dt[s] = fma2(ca, cb, dt[s]);
      aa[s] = fma2(ca, ca, aa[s]);
      bb[s] = fma2(cb, cb, bb[s]);
    }
  }
  __syncthreads();                             // every warp is done with the rows
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    part[quarter][3 * s][q] = hsum2(dt[s]);
    part[quarter][3 * s + 1][q] = hsum2(aa[s]);
    part[quarter][3 * s + 2][q] = hsum2(bb[s]);
  }
  __syncthreads();
  if (threadIdx.x < kCurvTile) {
    const int qq = threadIdx.x;
    const int t = t0 + qq;
    if (t < n) {
      float tot = 0.f;
      int cnt = 0;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int w = 1 << s;
        if (t >= w && t < n - w) {
          const float dot = part[0][3 * s][qq] + part[1][3 * s][qq] + part[2][3 * s][qq] +
                            part[3][3 * s][qq];
          const float na2 = part[0][3 * s + 1][qq] + part[1][3 * s + 1][qq] +
                            part[2][3 * s + 1][qq] + part[3][3 * s + 1][qq];
          const float nb2 = part[0][3 * s + 2][qq] + part[1][3 * s + 2][qq] +
                            part[2][3 * s + 2][qq] + part[3][3 * s + 2][qq];
          const float nn2 = na2 * nb2;
          tot += 1.f - (nn2 > 0.f ? dot * rsqrtf(nn2) : 1.f);
          ++cnt;
        }
      }
      a.kappa[row0 + t] = cnt > 0 ? tot / (float)cnt : 0.f;
    }
  }
}

// One warp per slot tree.
__global__ void __launch_bounds__(256) tree_cut_kernel(kvc_params p, TreeArgs a) {
  __shared__ float ks[8][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long tree = (long long)blockIdx.x * 8 + warp;
  if (tree >= (long long)p.B * p.L * p.H * p.S_max) return;
  const int s = (int)(tree % p.S_max);
  const long long blh = tree / p.S_max;
  const int lh = (int)(blh % ((long long)p.L * p.H));
  const int b = (int)(blh / ((long long)p.L * p.H));
  uint8_t* out = a.cuts + tree * 8;
  const int S = a.n_slots[b];
  if (s >= S) {
    if (lane < 8) out[lane] = 0;
    return;
  }
  const int n = a.ctx_len[b];
  const int x0 = a.bounds[(long long)b * (p.S_max + 1) + s];
  const int y0 = a.bounds[(long long)b * (p.S_max + 1) + s + 1];
  if (S > p.S_max || n > p.n_max || x0 < 0 || y0 - x0 < 16 || y0 - x0 > 128 || y0 > n - p.W) {
    if (lane == 0) kvcd::record_error(a.err, KVC_EDEVICE);
    return;
  }
  const int64_t row0 = kvcd::seq_token_base(a.ctx_len, b, p.L * p.H) + (int64_t)lh * n;
  float* k = ks[warp];
  for (int i = lane; i < y0 - x0; i += 32) k[i] = a.kappa[row0 + x0 + i];
  __syncwarp();
  int na[15], nb[15];                          // node ranges (relative to x0)
  na[0] = 0; nb[0] = y0 - x0;
  uint8_t cut[7];
#pragma unroll
  for (int j = 0; j < 7; ++j) {
    const int lo_n = na[j], hi_n = nb[j];
    const int depth = kvcd::tree_depth(j);
    const int lo = 8 >> depth, hi = 64 >> depth;   // 2 and 16 tokens per leaf below
    const int c = hi_n - lo_n;
    const int m = (lo_n + hi_n) >> 1;
    float acc = 0.f;                          // index-order sum, the same on every lane
    for (int i = lo_n; i < hi_n; ++i) acc = __fadd_rn(acc, k[i]);
    const float lam = __fdiv_rn(acc, (float)c);
    const float half = __fmul_rn((float)c, 0.5f);
    auto score = [&](int t) {
      const float r = __fdiv_rn((float)(t - m), half);
      return __fsub_rn(k[t], __fmul_rn(lam, __fmul_rn(r, r)));
    };
    float best = -INFINITY;
    int best_t = 0x7fffffff;
    for (int t = lo_n + lo + lane; t <= hi_n - lo; t += 32) {
      if (t - lo_n > hi || hi_n - t > hi) continue;
      const float sc = score(t);
      if (sc > best) { best = sc; best_t = t; }   // ascending t: first maximum per lane
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(KVC_FULL_MASK, best, o);
      const int ot = __shfl_xor_sync(KVC_FULL_MASK, best_t, o);
      if (ob > best || (ob == best && ot < best_t)) { best = ob; best_t = ot; }
    }
    const int t = best > score(m) ? best_t : m;
    cut[j] = (uint8_t)t;
    na[2 * j + 1] = lo_n; nb[2 * j + 1] = t;
    na[2 * j + 2] = t;    nb[2 * j + 2] = hi_n;
  }
  if (lane < 8) out[lane] = lane < 7 ? cut[lane] : (uint8_t)0;
}

}  // namespace

extern "C" int kvc_tree_cuts(const kvc_params* p, const int32_t* ctx_len, const void* K,
                             const float* rope_cos, const float* rope_sin,
                             const int32_t* slot_bounds, const int32_t* n_slots, float* kappa,
                             uint8_t* cuts, void* stream) {
  int st = kvc::check_params(p);
  if (st != KVC_OK) return st;
  if (!ctx_len || !K || !rope_cos || !rope_sin || !slot_bounds || !n_slots || !kappa || !cuts)
    return KVC_EINVAL;
  if (reinterpret_cast<uintptr_t>(K) & 15) return KVC_EINVAL;   // vector loads of key rows
  const long long blh = kvc::lh_count(p);
  if (blh > 65535) return KVC_EINVAL;
  int32_t* err = kvc::err_word();
  if (!err) return KVC_ECUDA;
  TreeArgs a;
  a.ctx_len = ctx_len; a.K = K; a.cos_tab = rope_cos; a.sin_tab = rope_sin;
  a.bounds = slot_bounds; a.n_slots = n_slots; a.kappa = kappa; a.cuts = cuts; a.err = err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const dim3 g1((unsigned)((p->n_max + kCurvTile - 1) / kCurvTile), (unsigned)blh);
  if (p->dtype == KVC_BF16) {
    if (p->d == 128) key_curv_kernel<__nv_bfloat16, 128><<<g1, 256, 0, s>>>(*p, a);
    else key_curv_kernel<__nv_bfloat16, 64><<<g1, 256, 0, s>>>(*p, a);
  } else {
    if (p->d == 128) key_curv_kernel<float, 128><<<g1, 256, 0, s>>>(*p, a);
    else key_curv_kernel<float, 64><<<g1, 256, 0, s>>>(*p, a);
  }
  const long long trees = blh * p->S_max;
  tree_cut_kernel<<<(unsigned)((trees + 7) / 8), 256, 0, s>>>(*p, a);
  kvc::count_launch(2);
  return kvc::cuda_status(cudaGetLastError());
}
