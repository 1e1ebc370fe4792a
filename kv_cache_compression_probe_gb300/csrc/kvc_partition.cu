// a0: curvature-guided slot partition (GraceKV "01 Curvature-guided
// partition": cut where the normalised hidden-state trajectory turns; slot
// lengths 16..128, target 64).  Reading of the page: one hidden-state stream,
//   kappa_w(t) = 1 - cos(h^_t - h^_{t-w}, h^_{t+w} - h^_t),  h^ = h / |h|,
// averaged over the scales w in {1, 2, 4, 8} that fit, then a dynamic program
// over cut positions in [0, n - W) maximising
//   sum_{interior cuts c} kappa(c) - lambda * sum_slots ((len - 64) / 64)^2,
// 16 <= len <= 128, lambda = mean of kappa over [0, n - W) (summed in a
// fixed order in double precision, see dp_kernel).  Ties go to the smaller
// previous cut.
//
// Kernels: norms (one warp per row), curvature (one CTA per 64 positions; the
// 80 rows it needs are staged 128 features at a time and each warp keeps the
// 12 partial dot products of its positions), and the DP (one CTA per
// sequence scoring 16 positions at a time, fp64, ring buffer of the last 256
// best scores, back-pointers in the workspace).
#include <float.h>
#include <limits.h>

#include "kvc_common.cuh"
#include "kvc_internal.h"

namespace {

constexpr int kLmin = 16, kLmax = 128, kTarget = 64;
constexpr int kPosPerCta = 64;
constexpr int kHalo = 8;
constexpr int kFeat = 128;            // features per staged chunk

template <typename T>
__global__ void norms_kernel(kvc_params p, const int32_t* ctx_len, const T* hidden, int dh,
                             float* inv_norm) {
  const int b = blockIdx.y;
  const int n = ctx_len[b];
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= n) return;
  const T* row = hidden + ((int64_t)b * p.n_max + t) * dh;
  float s = 0.f;
  for (int f = lane; f < dh; f += 32) { const float x = kvcd::to_f(row[f]); s = fmaf(x, x, s); }
  s = kvcd::warp_sum(s);
  if (lane == 0) inv_norm[(int64_t)b * p.n_max + t] = s > 0.f ? 1.f / sqrtf(s) : 0.f;
}

// One CTA = 64 positions; warp w owns positions t0 + 8w .. t0 + 8w + 7.
template <typename T>
__global__ void __launch_bounds__(256) curvature_kernel(kvc_params p, const int32_t* ctx_len,
                                                        const T* hidden, int dh,
                                                        const float* inv_norm, float* kappa) {
  __shared__ float rows[kPosPerCta + 2 * kHalo][kFeat + 1];
  const int b = blockIdx.y;
  const int n = ctx_len[b];
  const int t0 = blockIdx.x * kPosPerCta;
  if (t0 >= n) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // acc[pos][scale][0: a.b, 1: a.a, 2: b.b]
  float acc[8][4][3];
#pragma unroll
  for (int q = 0; q < 8; ++q)
#pragma unroll
    for (int w = 0; w < 4; ++w) acc[q][w][0] = acc[q][w][1] = acc[q][w][2] = 0.f;
  const float* inv = inv_norm + (int64_t)b * p.n_max;
  for (int f0 = 0; f0 < dh; f0 += kFeat) {
    __syncthreads();
    for (int idx = tid; idx < (kPosPerCta + 2 * kHalo) * kFeat; idx += 256) {
      const int r = idx / kFeat, f = idx % kFeat;
      const int t = t0 - kHalo + r;
      float x = 0.f;
      if (t >= 0 && t < n && f0 + f < dh)
        x = kvcd::to_f(hidden[((int64_t)b * p.n_max + t) * dh + f0 + f]) * inv[t];
      rows[r][f] = x;
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int r = kHalo + warp * 8 + q;                 // staged row of position t
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        const int w = 1 << wi;
        float ab = 0.f, aa = 0.f, bb = 0.f;
        for (int f = lane; f < kFeat; f += 32) {
          const float hc = rows[r][f];
          const float av = hc - rows[r - w][f];
          const float bv = rows[r + w][f] - hc;
          ab = fmaf(av, bv, ab); aa = fmaf(av, av, aa); bb = fmaf(bv, bv, bb);
        }
        acc[q][wi][0] += ab; acc[q][wi][1] += aa; acc[q][wi][2] += bb;
      }
    }
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int t = t0 + warp * 8 + q;
    float ksum = 0.f;
    int kc = 0;
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      const int w = 1 << wi;
      const float ab = kvcd::warp_sum(acc[q][wi][0]);
      const float aa = kvcd::warp_sum(acc[q][wi][1]);
      const float bb = kvcd::warp_sum(acc[q][wi][2]);
      if (n > 2 * w && t >= w && t < n - w) {
        const float den = sqrtf(aa) * sqrtf(bb);
        const float c = den > 0.f ? ab / den : 1.f;
        ksum += 1.f - c;
        ++kc;
      }
    }
    if (lane == 0 && t < n) kappa[(int64_t)b * p.n_max + t] = kc > 0 ? ksum / (float)kc : 0.f;
  }
}

// Candidate scores are compared as integers: for a double v that is not NaN
// and not -0, key(v) orders like v.  The scores here are never -0 (the gains
// and the penalties are never -0 and best[0] = +0), and -0 is mapped to +0.
__device__ __forceinline__ long long order_key(double v) {
  long long bits = __double_as_longlong(v);
  if (bits == LLONG_MIN) bits = 0;
  return bits >= 0 ? bits : bits ^ LLONG_MAX;
}
__device__ __forceinline__ double from_key(long long key) {
  return __longlong_as_double(key >= 0 ? key : key ^ LLONG_MAX);
}

// One CTA of kDpWarps warps per sequence.  Every slot is at least kLmin
// tokens long, so best[y] for the kLmin positions of a block [Y, Y + kLmin)
// depends only on best[x] with x < Y: warp w scores position Y + w, its lanes
// the candidate lengths, and the CTA synchronises once per block.  Each
// candidate is scored as (best[x] - lambda * d^2) + gain in fp64, as in the
// sequential recurrence, so the result does not depend on the blocking.
constexpr int kDpWarps = kLmin;
constexpr int kDpThreads = kDpWarps * 32;
constexpr int kRing = 256;                                  // > kLmax + kDpWarps
__global__ void __launch_bounds__(kDpThreads) dp_kernel(kvc_params p, const int32_t* ctx_len,
                                                        const float* kappa, int16_t* back,
                                                        int32_t* slot_bounds, int32_t* n_slots,
                                                        int32_t* err) {
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = ctx_len[b];
  const int end = n - p.W;
  __shared__ double ring[kRing];                          // best[x] at x % kRing
  __shared__ double pen[kLmax - kLmin + 1];               // lambda * ((len - 64) / 64)^2
  __shared__ double part[kDpThreads];
  const float* kap = kappa + (int64_t)b * p.n_max;
  int16_t* bk = back + (int64_t)b * p.n_max;
  int32_t* bd = slot_bounds + (int64_t)b * (p.S_max + 1);
  if (end < kLmin || end > p.n_max) {
    if (tid == 0) { kvcd::record_error(err, KVC_EDEVICE); n_slots[b] = 0; }
    return;
  }
  // lambda = mean kappa over [0, end): thread i sums t = i, i + 512, ... in
  // order, then the 512 partial sums are added pairwise, halving the stride
  double acc = 0.0;
  for (int t = tid; t < end; t += kDpThreads) acc += (double)kap[t];
  part[tid] = acc;
  __syncthreads();
  for (int h = kDpThreads / 2; h > 0; h >>= 1) {
    if (tid < h) part[tid] = part[tid] + part[tid + h];
    __syncthreads();
  }
  const double lam = part[0] / (double)end;
  const long long neg_bits = __double_as_longlong(-DBL_MAX);
  if (tid <= kLmax - kLmin) {
    const double d = (double)(tid + kLmin - kTarget) * (1.0 / (double)kTarget);   // exact
    pen[tid] = lam * (d * d);
  }
  for (int i = tid; i < kRing; i += kDpThreads) ring[i] = i == 0 ? 0.0 : -DBL_MAX;
  __syncthreads();
  float g_next = warp + 1 < end ? kap[warp + 1] : 0.f;
  for (int Y = 1; Y <= end; Y += kDpWarps) {
    const int y = Y + warp;
    const float g_now = g_next;
    if (y + kDpWarps < end) g_next = kap[y + kDpWarps];  // next block's gain, in flight
    if (y <= end) {                                       // warp-uniform
      const double gain = y < end ? (double)g_now : 0.0;
      // lane: lengths kLmin + lane + 32 i; the four candidates are scored
      // without branches so their loads and fp64 adds overlap
      unsigned long long bkey = 0;                        // 0: no candidate
      int bl = 0;                                         // best length (larger wins ties)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int ln = kLmin + lane + 32 * i;
        const int x = y - ln;
        const bool in = ln <= kLmax && x >= 0;
        const double bx = ring[(in ? x : 0) & (kRing - 1)];
        const double v = (bx - pen[(in ? ln : kLmin) - kLmin]) + gain;
        // unsigned key: order_key shifted so that 0 is below every score
        const unsigned long long key =
            (unsigned long long)order_key(v) ^ 0x8000000000000000ull;
        const bool ok = in && __double_as_longlong(bx) != neg_bits;
        if (ok && key >= bkey) { bkey = key; bl = ln; }   // ln ascends: ties go to the larger
      }
      // warp maximum of (key, length): the high word, then the low word among
      // the lanes holding that high word, then the largest length among the
      // lanes holding the whole key
      const unsigned hi = (unsigned)(bkey >> 32), lo = (unsigned)bkey;
      const unsigned mhi = __reduce_max_sync(KVC_FULL_MASK, hi);
      const unsigned mlo = __reduce_max_sync(KVC_FULL_MASK, hi == mhi ? lo : 0u);
      const unsigned mbl = __reduce_max_sync(KVC_FULL_MASK, (hi == mhi && lo == mlo) ? (unsigned)bl : 0u);
      if (lane == 0) {
        const unsigned long long best = ((unsigned long long)mhi << 32) | mlo;
        ring[y & (kRing - 1)] =
            mbl > 0 ? from_key((long long)(best ^ 0x8000000000000000ull)) : -DBL_MAX;
        bk[y] = (int16_t)mbl;
      }
    }
    __syncthreads();
  }
  if (tid == 0) {
    if (__double_as_longlong(ring[end & (kRing - 1)]) == neg_bits) {
      kvcd::record_error(err, KVC_EDEVICE); n_slots[b] = 0; return;
    }
    int cnt = 0;
    for (int y = end; y > 0 && cnt <= p.S_max; y -= bk[y]) {
      if (bk[y] < kLmin || bk[y] > y) { cnt = p.S_max + 1; break; }   // never for a reachable end
      ++cnt;
    }
    if (cnt > p.S_max) { kvcd::record_error(err, KVC_EDEVICE); n_slots[b] = 0; return; }
    int k = cnt;
    bd[k] = end;
    for (int y = end; y > 0; y -= bk[y]) bd[--k] = y - bk[y];
    for (int s = cnt + 1; s <= p.S_max; ++s) bd[s] = end;
    n_slots[b] = cnt;
  }
}

struct Layout {
  size_t inv, back, total;
};
Layout layout(const kvc_params* p) {
  Layout l;
  l.inv = 0;
  l.back = kvc::align256((size_t)p->B * p->n_max * sizeof(float));
  l.total = l.back + kvc::align256((size_t)p->B * p->n_max * sizeof(int16_t));
  return l;
}

template <typename T>
void launch(const kvc_params* p, const int32_t* ctx_len, const void* hidden, int dh, float* kappa,
            int32_t* bounds, int32_t* n_slots, char* ws, int32_t* err, cudaStream_t s) {
  const Layout lay = layout(p);
  float* inv = reinterpret_cast<float*>(ws + lay.inv);
  int16_t* back = reinterpret_cast<int16_t*>(ws + lay.back);
  const T* h = static_cast<const T*>(hidden);
  norms_kernel<T><<<dim3((p->n_max + 7) / 8, p->B), 256, 0, s>>>(*p, ctx_len, h, dh, inv);
  curvature_kernel<T><<<dim3((p->n_max + kPosPerCta - 1) / kPosPerCta, p->B), 256, 0, s>>>(
      *p, ctx_len, h, dh, inv, kappa);
  dp_kernel<<<p->B, kDpThreads, 0, s>>>(*p, ctx_len, kappa, back, bounds, n_slots, err);
  kvc::count_launch(3);
}

}  // namespace

namespace kvc {
size_t partition_workspace_bytes(const kvc_params* p) { return layout(p).total; }
}  // namespace kvc

extern "C" int kvc_partition(const kvc_params* p, const int32_t* ctx_len, const void* hidden,
                             int32_t dh, float* kappa, int32_t* slot_bounds, int32_t* n_slots,
                             void* workspace, size_t ws_bytes, void* stream) {
  int st = kvc::check_params(p);
  if (st != KVC_OK) return st;
  if (!ctx_len || !hidden || !kappa || !slot_bounds || !n_slots || dh < 1 || dh > 65536)
    return KVC_EINVAL;
  const size_t need = layout(p).total;
  if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return KVC_EWORKSPACE;
  int32_t* err = kvc::err_word();
  if (!err) return KVC_ECUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p->dtype == KVC_BF16)
    launch<__nv_bfloat16>(p, ctx_len, hidden, dh, kappa, slot_bounds, n_slots,
                          static_cast<char*>(workspace), err, s);
  else
    launch<float>(p, ctx_len, hidden, dh, kappa, slot_bounds, n_slots,
                  static_cast<char*>(workspace), err, s);
  return kvc::cuda_status(cudaGetLastError());
}
