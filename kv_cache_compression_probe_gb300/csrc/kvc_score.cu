// a1-a4: probe scoring and token features, relevance hops, prototype trees,
// probe-based distortion and per-entry utilities.
//
// Sources: DistillCache section 3.1.1 (features alpha, |v|, sigma, H, pos over
// the recent queries); GraceKV "03 Bottom-up value flow" (direct probes plus
// two token-to-token hops of weight 0.3; parent value = sum of child values),
// "Inside one cache entry" (RoPE-consistent key merge, relevance-weighted
// values with a 10% floor, multiplicity), technical details (distortion =
// 0.25 attention-partition error + 0.75 value-aggregate error), "04 Top-down
// budget flow" (utility = relevance x fidelity gain x head sensitivity / new
// entries).
//
// Kernels (all fp32 arithmetic on bf16/f32 inputs, scores kept in base 2):
//   rowstats   per probe row and key chunk: online max, sum p, sum p*(s - max)
//   rowcombine per row: LSE and attention entropy H(a_rho)
//   feats      per 64-key tile: a = softmax, reductions over rows -> features
//   numean     per (b,l,h): mean |v| (distortion normaliser)
//   seeds      per (b,l,h): top-P tokens by current relevance (radix select)
//   rowstats/rowcombine again with the seeds' values as queries (non-causal)
//   prop       per tile: r_k = alpha + w * sum_s r_s softmax_s(v_s . k / sqrt d)
//   nodes      per slot: 15 prototypes, per-row node mass / value aggregate,
//              distortions, the slot's 16 op utilities and costs
// The probe-times-key products use one thread per probe row with the query in
// registers and the key tile broadcast from shared memory.
#include <math.h>

#include <atomic>
#include <mutex>

#include <algorithm>
#include <type_traits>

#include "kvc_common.cuh"
#include "kvc_internal.h"
#include "kvc_score_tc.h"

namespace {

constexpr int kOps = 16;
constexpr int kTile = 64;          // keys per shared-memory tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct ScoreArgs {
  const int32_t* ctx_len;
  const void* K;
  const void* V;
  const void* Qp;
  const float* cos_tab;
  const float* sin_tab;
  const int32_t* bounds;
  const int32_t* n_slots;
  const float* head_sens;
  float* lse;          // [BLH, R] natural log
  float* feats;        // [rows, 5]
  float* rel;          // [rows]
  float* op_util;
  int32_t* op_cost;
  // workspace
  float* part;         // [BLH, n_chunks, Rmax, 3]
  float* lse2;         // [BLH, R] base-2 LSE of probe rows
  float* hrow;         // [BLH, R] entropy of probe rows
  float* nu;           // [BLH]
  int32_t* seeds;      // [BLH, P]
  float* seed_w;       // [BLH, P]
  float* lse2_h;       // [BLH, P] base-2 LSE of seed rows
  int32_t* ok;         // [BLH] 1 if the (l,h) passed its checks
  unsigned char* proto;  // [BLH * S_max] prototype records (tensor-core path)
  float* npart;        // [BLH * S_max, 2, 15, 4] node statistics (tensor-core path)
  float* nu_part;      // [BLH, S_max + 1] sums of |v| per slot, then the window (tensor-core path)
  int32_t* err;
  int chunk;           // keys per rowstats chunk
  int n_chunks;
  float q_scale2;      // log2(e) / sqrt(d)
};

__device__ __forceinline__ int seq_of(const kvc_params& p, long long blh) {
  return (int)(blh / ((long long)p.L * p.H));
}

// Loads `rows` token rows [i0, i0 + rows) of one (b,l,h) into smem as fp32
// [rows][D]; rows beyond `n` are zero-filled.
template <typename T, int D>
__device__ __forceinline__ void load_rows(float* dst, const T* src, int i0, int rows, int n) {
  constexpr int V = 4;
  for (int e = threadIdx.x * V; e < rows * D; e += blockDim.x * V) {
    const int r = e / D, c = e % D;
    float v[V];
    if (i0 + r < n) kvcd::VecLoad<T, V>::ld(src + (int64_t)(i0 + r) * D + c, v);
    else v[0] = v[1] = v[2] = v[3] = 0.f;
    *reinterpret_cast<float4*>(dst + r * D + c) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

template <typename T, int D>
__device__ __forceinline__ void load_q(float* q, const T* src, float scale) {
#pragma unroll
  for (int c = 0; c < D; c += 4) {
    float v[4];
    kvcd::VecLoad<T, 4>::ld(src + c, v);
#pragma unroll
    for (int t = 0; t < 4; ++t) q[c + t] = v[t] * scale;
  }
}

// Four dot products q . k_{j..j+3} against an fp32 smem tile [*, D].
template <int D>
__device__ __forceinline__ void dot4(const float* q, const float* tile, int j, float s[4]) {
  s[0] = s[1] = s[2] = s[3] = 0.f;
#pragma unroll
  for (int c = 0; c < D; c += 4) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float4 k = *reinterpret_cast<const float4*>(tile + (j + u) * D + c);
      s[u] = fmaf(q[c], k.x, s[u]);
      s[u] = fmaf(q[c + 1], k.y, s[u]);
      s[u] = fmaf(q[c + 2], k.z, s[u]);
      s[u] = fmaf(q[c + 3], k.w, s[u]);
    }
  }
}

__device__ __forceinline__ float dot1(const float* q, const float* k, int D) {
  float s = 0.f;
  for (int c = 0; c < D; ++c) s = fmaf(q[c], k[c], s);
  return s;
}

// ---------------------------------------------------------------- row statistics
// SEEDS = false: rows are the probes (causal: probe p sees keys <= n - P + p);
// SEEDS = true: rows are the hop seeds, queries = the seeds' values, all keys.
template <typename T, int D, bool SEEDS>
__global__ void __launch_bounds__(256, 1) rowstats_kernel(kvc_params p, ScoreArgs a) {
  extern __shared__ float4 smem4[];
  float* sK = reinterpret_cast<float*>(smem4);
  const long long blh = blockIdx.y;
  if (!a.ok[blh]) return;
  const int b = seq_of(p, blh);
  const int lh = (int)(blh % ((long long)p.L * p.H));
  const int n = a.ctx_len[b];
  const int R = SEEDS ? p.P : p.G * p.P;
  const int rho = threadIdx.x;
  const int k0 = blockIdx.x * a.chunk;
  float* out = a.part + ((blh * a.n_chunks + blockIdx.x) * 256 + rho) * 3;
  if (k0 >= n) {
    if (rho < R) { out[0] = -INFINITY; out[1] = 0.f; out[2] = 0.f; }
    return;
  }
  const int64_t row0 = kvcd::seq_token_base(a.ctx_len, b, p.L * p.H) + (int64_t)lh * n;
  const T* Kh = static_cast<const T*>(a.K) + row0 * D;
  float q[D];
  int limit = n - 1;
  if (rho < R) {
    if (SEEDS) {
      const int sidx = a.seeds[blh * p.P + rho];
      load_q<T, D>(q, static_cast<const T*>(a.V) + (row0 + sidx) * D, a.q_scale2);
    } else {
      load_q<T, D>(q, static_cast<const T*>(a.Qp) + (blh * R + rho) * D, a.q_scale2);
      limit = n - p.P + (rho % p.P);
    }
  }
  // l = sum 2^(s - m), u = sum 2^(s - m) (s - m) <= 0: both sums have terms of
  // one sign, and the entropy ln2 (log2 l - u / l) needs no subtraction of
  // nearly equal numbers.  Compensated (Kahan) accumulation.
  float m = -INFINITY, l = 0.f, u = 0.f, cl = 0.f, cu = 0.f;
  const int k1 = min(n, k0 + a.chunk);
  for (int i0 = k0; i0 < k1; i0 += kTile) {
    __syncthreads();
    load_rows<T, D>(sK, Kh, i0, kTile, k1);
    __syncthreads();
    if (rho < R) {
      const int cnt = min(kTile, k1 - i0);
      for (int j = 0; j < cnt; j += 4) {
        float s[4];
        dot4<D>(q, sK, j, s);
        float mx = m;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          if (j + v >= cnt || i0 + j + v > limit) s[v] = -INFINITY;
          mx = fmaxf(mx, s[v]);
        }
        if (mx == -INFINITY) continue;
        if (mx > m && m != -INFINITY) {
          const float sc = exp2f(m - mx);
          u = sc * (u + (m - mx) * l);
          cu = sc * cu;
          l *= sc;
          cl *= sc;
        }
        m = mx;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          if (s[v] == -INFINITY) continue;
          const float e = exp2f(s[v] - mx);
          const float yl = e - cl, tl = l + yl;
          cl = (tl - l) - yl; l = tl;
          const float yu = e * (s[v] - mx) - cu, tu = u + yu;
          cu = (tu - u) - yu; u = tu;
        }
      }
    }
  }
  if (rho < R) { out[0] = m; out[1] = l; out[2] = u; }
}

template <bool SEEDS>
__global__ void rowcombine_kernel(kvc_params p, ScoreArgs a) {
  const long long blh = blockIdx.x;
  const int rho = threadIdx.x;
  const int R = SEEDS ? p.P : p.G * p.P;
  if (rho >= R || !a.ok[blh]) return;
  const float* pp = a.part + (blh * a.n_chunks * 256 + rho) * 3;
  float M = -INFINITY;
  for (int c = 0; c < a.n_chunks; ++c) M = fmaxf(M, pp[(int64_t)c * 256 * 3]);
  float L = 0.f, U = 0.f;                          // U = sum 2^(s - M) (s - M) <= 0
  for (int c = 0; c < a.n_chunks; ++c) {
    const float* q = pp + (int64_t)c * 256 * 3;
    if (q[0] == -INFINITY) continue;
    const float f = exp2f(q[0] - M);
    L = fmaf(q[1], f, L);
    U += f * (q[2] + (q[0] - M) * q[1]);
  }
  const float lse2 = M + log2f(L);
  if (SEEDS) {
    a.lse2_h[blh * p.P + rho] = lse2;
  } else {
    a.lse2[blh * R + rho] = lse2;
    a.lse[blh * R + rho] = lse2 * kLn2;
    a.hrow[blh * R + rho] = kLn2 * (log2f(L) - U / L);
  }
}

// ---------------------------------------------------------------- features (a1)
template <typename T, int D>
__global__ void __launch_bounds__(256, 1) feats_kernel(kvc_params p, ScoreArgs a) {
  extern __shared__ float4 smem4[];
  float* sK = reinterpret_cast<float*>(smem4);            // [kTile][D]
  float* sA = sK + kTile * D;                             // [kTile][257]
  const long long blh = blockIdx.y;
  if (!a.ok[blh]) return;
  const int b = seq_of(p, blh);
  const int lh = (int)(blh % ((long long)p.L * p.H));
  const int n = a.ctx_len[b];
  const int R = p.G * p.P;
  const int i0 = blockIdx.x * kTile;
  if (i0 >= n) return;
  const int64_t row0 = kvcd::seq_token_base(a.ctx_len, b, p.L * p.H) + (int64_t)lh * n;
  const T* Kh = static_cast<const T*>(a.K) + row0 * D;
  const int cnt = min(kTile, n - i0);
  load_rows<T, D>(sK, Kh, i0, kTile, n);
  __syncthreads();
  const int rho = threadIdx.x;
  if (rho < R) {
    float q[D];
    load_q<T, D>(q, static_cast<const T*>(a.Qp) + (blh * R + rho) * D, a.q_scale2);
    const float l2 = a.lse2[blh * R + rho];
    const int limit = n - p.P + (rho % p.P);
    for (int j = 0; j < kTile; j += 4) {
      float s[4];
      dot4<D>(q, sK, j, s);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + j + u;
        sA[(j + u) * 257 + rho] = (j + u < cnt && i <= limit) ? exp2f(s[u] - l2) : 0.f;
      }
    }
  }
  __syncthreads();
  // four threads per key reduce over the rows
  const int key = threadIdx.x >> 2, part = threadIdx.x & 3;
  float sa = 0.f, sah = 0.f, sg[8];
#pragma unroll
  for (int g = 0; g < 8; ++g) sg[g] = 0.f;
  for (int r = part; r < R; r += 4) {
    const float v = sA[key * 257 + r];
    sa += v;
    sah = fmaf(v, a.hrow[blh * R + r], sah);
    const int g = r / p.P;
#pragma unroll
    for (int gg = 0; gg < 8; ++gg) if (gg == g) sg[gg] += v;
  }
  float vn2 = 0.f;
  const int i = i0 + key;
  if (key < cnt) {
    const T* vr = static_cast<const T*>(a.V) + (row0 + i) * D;
    for (int c = part; c < D; c += 4) { const float x = kvcd::to_f(vr[c]); vn2 = fmaf(x, x, vn2); }
  }
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    sa += __shfl_xor_sync(KVC_FULL_MASK, sa, o);
    sah += __shfl_xor_sync(KVC_FULL_MASK, sah, o);
    vn2 += __shfl_xor_sync(KVC_FULL_MASK, vn2, o);
#pragma unroll
    for (int g = 0; g < 8; ++g) sg[g] += __shfl_xor_sync(KVC_FULL_MASK, sg[g], o);
  }
  if (part == 0 && key < cnt) {
    float mean = 0.f;
    for (int g = 0; g < p.G; ++g) mean += sg[g] / (float)p.P;
    mean /= (float)p.G;
    float var = 0.f;
    for (int g = 0; g < p.G; ++g) { const float dlt = sg[g] / (float)p.P - mean; var += dlt * dlt; }
    var /= (float)p.G;
    float* f = a.feats + (row0 + i) * 5;
    const float alpha = sa / (float)R;
    f[0] = alpha;
    f[1] = sqrtf(vn2);
    f[2] = var;
    f[3] = sa > 0.f ? sah / sa : 0.f;
    f[4] = (float)i / (float)max(n - 1, 1);
    a.rel[row0 + i] = alpha;
  }
}

// mean |v| of one (b,l,h)
__global__ void numean_kernel(kvc_params p, ScoreArgs a) {
  const long long blh = blockIdx.x;
  if (!a.ok[blh]) return;
  const int b = seq_of(p, blh);
  const int lh = (int)(blh % ((long long)p.L * p.H));
  const int n = a.ctx_len[b];
  const int64_t row0 = kvcd::seq_token_base(a.ctx_len, b, p.L * p.H) + (int64_t)lh * n;
  float s = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) s += a.feats[(row0 + i) * 5 + 1];
  __shared__ float red[32];
  s = kvcd::warp_sum(s);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    v = kvcd::warp_sum(v);
    if (threadIdx.x == 0) a.nu[blh] = v / (float)n;
  }
}

// Tensor-core path: the slots' |v| and position features come from the
// prototype kernel (one sum of |v| per slot); this kernel covers the W window
// tokens (one thread per token) and nu_finish_slots forms the mean |v| of each
// (b,l,h) from the slot sums and the window sum in a fixed order.
template <typename T, int D>
__global__ void __launch_bounds__(128) vnorm_window_kernel(kvc_params p, ScoreArgs a) {
  const long long blh = blockIdx.x;
  if (!a.ok[blh]) return;
  const int b = seq_of(p, blh);
  const int lh = (int)(blh % ((long long)p.L * p.H));
  const int n = a.ctx_len[b];
  const int64_t row0 = kvcd::seq_token_base(a.ctx_len, b, p.L * p.H) + (int64_t)lh * n;
  __shared__ float red[4];
  float acc = 0.f;
  for (int i = n - p.W + (int)threadIdx.x; i < n; i += 128) {
    const T* vr = static_cast<const T*>(a.V) + (row0 + i) * D;
    float s2 = 0.f;
#pragma unroll 8
    for (int c = 0; c < D; c += 4) {
      float v[4];
      kvcd::VecLoad<T, 4>::ld(vr + c, v);
#pragma unroll
      for (int t = 0; t < 4; ++t) s2 = fmaf(v[t], v[t], s2);
    }
    const float nv = sqrtf(s2);
    float* f = a.feats + (row0 + i) * 5;
    f[1] = nv;
    f[4] = (float)i / (float)max(n - 1, 1);
    acc += nv;
  }
  const float ws = kvcd::warp_sum(acc);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ws;
  __syncthreads();
  if (threadIdx.x == 0)
    a.nu_part[blh * (p.S_max + 1) + p.S_max] = (red[0] + red[1]) + (red[2] + red[3]);
}

__global__ void nu_finish_slots_kernel(kvc_params p, ScoreArgs a) {
  const long long blh = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (blh >= (long long)p.B * p.L * p.H || !a.ok[blh]) return;
  const int b = seq_of(p, blh);
  const int S = a.n_slots[b];
  const float* ps = a.nu_part + blh * (p.S_max + 1);
  float t = 0.f;
  for (int s = 0; s < S; ++s) t += ps[s];
  t += ps[p.S_max];
  a.nu[blh] = t / (float)a.ctx_len[b];
}

// ---------------------------------------------------------------- hops (a2)
// Top-P tokens by relevance (ties to the lower index) via an 8-pass radix
// select on (float key, ~index); seeds written in ascending index order.
__global__ void __launch_bounds__(1024) seeds_kernel(kvc_params p, ScoreArgs a) {
  const long long blh = blockIdx.x;
  if (!a.ok[blh]) return;
  const int b = seq_of(p, blh);
  const int lh = (int)(blh % ((long long)p.L * p.H));
  const int n = a.ctx_len[b];
  const int64_t row0 = kvcd::seq_token_base(a.ctx_len, b, p.L * p.H) + (int64_t)lh * n;
  const float* r = a.rel + row0;
  const int K = min(p.P, n);
  __shared__ unsigned int hist[256];
  __shared__ unsigned long long s_prefix;
  __shared__ int s_krem;
  if (threadIdx.x == 0) { s_prefix = 0ull; s_krem = K; }
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    const unsigned long long hi_mask = pass == 0 ? 0ull : (~0ull << (shift + 8));
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const unsigned long long pref = s_prefix;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const unsigned long long k = ((unsigned long long)kvcd::float_key(r[i]) << 32) |
                                   (0xffffffffu - (uint32_t)i);
      if ((k & hi_mask) == (pref & hi_mask)) atomicAdd(&hist[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int acc = 0;
      for (int dgt = 255; dgt >= 0; --dgt) {
        const int h = (int)hist[dgt];
        if (acc + h >= s_krem) {
          s_prefix |= ((unsigned long long)dgt) << shift;
          s_krem -= acc;
          break;
        }
        acc += h;
      }
    }
    __syncthreads();
  }
  const unsigned long long thr = s_prefix;         // the K-th largest key
  // ordered compaction of keys >= thr
  __shared__ int s_cnt[1024];
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int lo = threadIdx.x * per, hi = min(n, lo + per);
  int c = 0;
  for (int i = lo; i < hi; ++i) {
    const unsigned long long k = ((unsigned long long)kvcd::float_key(r[i]) << 32) |
                                 (0xffffffffu - (uint32_t)i);
    c += k >= thr;
  }
  s_cnt[threadIdx.x] = c;
  __syncthreads();
  for (int o = 1; o < (int)blockDim.x; o <<= 1) {
    const int v = threadIdx.x >= (unsigned)o ? s_cnt[threadIdx.x - o] : 0;
    __syncthreads();
    s_cnt[threadIdx.x] += v;
    __syncthreads();
  }
  int w = s_cnt[threadIdx.x] - c;
  for (int i = lo; i < hi && w < K; ++i) {
    const unsigned long long k = ((unsigned long long)kvcd::float_key(r[i]) << 32) |
                                 (0xffffffffu - (uint32_t)i);
    if (k >= thr) {
      a.seeds[blh * p.P + w] = i;
      a.seed_w[blh * p.P + w] = r[i];
      ++w;
    }
  }
  for (int j = K + threadIdx.x; j < p.P; j += blockDim.x) {   // n < P: unused seed slots
    a.seeds[blh * p.P + j] = 0;
    a.seed_w[blh * p.P + j] = 0.f;
  }
}

// r_k(j) = alpha_j + w * sum_s r_s * softmax over all keys of (v_s . k_j / sqrt d)
template <typename T, int D>
__global__ void __launch_bounds__(256, 1) prop_kernel(kvc_params p, ScoreArgs a) {
  extern __shared__ float4 smem4[];
  float* sK = reinterpret_cast<float*>(smem4);            // [kTile][D]
  float* sA = sK + kTile * D;                             // [kTile][257]
  const long long blh = blockIdx.y;
  if (!a.ok[blh]) return;
  const int b = seq_of(p, blh);
  const int lh = (int)(blh % ((long long)p.L * p.H));
  const int n = a.ctx_len[b];
  const int S = p.P;
  const int i0 = blockIdx.x * kTile;
  if (i0 >= n) return;
  const int64_t row0 = kvcd::seq_token_base(a.ctx_len, b, p.L * p.H) + (int64_t)lh * n;
  const T* Kh = static_cast<const T*>(a.K) + row0 * D;
  const int cnt = min(kTile, n - i0);
  load_rows<T, D>(sK, Kh, i0, kTile, n);
  __syncthreads();
  const int sr = threadIdx.x;
  if (sr < S) {
    float q[D];
    const int sidx = a.seeds[blh * p.P + sr];
    load_q<T, D>(q, static_cast<const T*>(a.V) + (row0 + sidx) * D, a.q_scale2);
    const float l2 = a.lse2_h[blh * p.P + sr];
    const float wgt = a.seed_w[blh * p.P + sr];
    for (int j = 0; j < kTile; j += 4) {
      float s[4];
      dot4<D>(q, sK, j, s);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        sA[(j + u) * 257 + sr] = (j + u < cnt) ? wgt * exp2f(s[u] - l2) : 0.f;
    }
  }
  __syncthreads();
  const int key = threadIdx.x >> 2, part = threadIdx.x & 3;
  float acc = 0.f;
  for (int r = part; r < S; r += 4) acc += sA[key * 257 + r];
  acc += __shfl_xor_sync(KVC_FULL_MASK, acc, 1);
  acc += __shfl_xor_sync(KVC_FULL_MASK, acc, 2);
  if (part == 0 && key < cnt) {
    const int i = i0 + key;
    a.rel[row0 + i] = a.feats[(row0 + i) * 5] + p.hop_weight * acc;
  }
}

// ---------------------------------------------------------------- nodes (a3 + a4)
// Token range [x, y) of node j of the slot [x0, y0) (cut table `cuts`, or the
// midpoint tree when null).
__device__ __forceinline__ void node_range(const uint8_t* cuts, int j, int x0, int y0, int& x,
                                           int& y) {
  kvcd::tree_node_range(cuts, j, x0, y0, x, y);
}

// Cost of Split(node j), j < 7: a three-way depth-2 node stores three entries
// in place of one (2), every other internal node two (1).
__device__ __forceinline__ int internal_split_cost(const uint8_t* cuts, int j, int x0, int y0) {
  if (j < 3 || !cuts) return 1;
  int x, y;
  node_range(cuts, j, x0, y0, x, y);
  return kvcd::tree_extract(cuts, j, x0, x, y) >= 0 ? 2 : 1;
}

template <int D>
struct NodeSmem {
  float K[128][D];
  float V[128][D];
  float kh[15][D];
  float vh[15][D];
  float A[128][68];        // a_rho(i) for the current 64-row group (padded stride)
  float Ah[15][64];        // A_hat per node and row of the group
  float r[128];
  float logm[15];
  float Rv[15];
  float st[4][15][64];     // per node and row: |A-Ah|, A, |U-Uh|, |U|
  float acc[4][15];        // running sums over rows
};

template <int D>
__device__ __forceinline__ void finish_node(NodeSmem<D>& sm, int j, int rq, const float A[4],
                                            const float (&U)[4][D / 32], int lane) {
  constexpr int VPL = D / 32;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const float ah = sm.Ah[j][rq + r];
    float dd = 0.f, uu = 0.f;
#pragma unroll
    for (int t = 0; t < VPL; ++t) {
      const float u = U[r][t];
      const float df = u - ah * sm.vh[j][lane * VPL + t];
      dd = fmaf(df, df, dd);
      uu = fmaf(u, u, uu);
    }
    dd = kvcd::warp_sum(dd);
    uu = kvcd::warp_sum(uu);
    if (lane == 0) {
      sm.st[0][j][rq + r] = fabsf(A[r] - ah);
      sm.st[1][j][rq + r] = A[r];
      sm.st[2][j][rq + r] = sqrtf(dd);
      sm.st[3][j][rq + r] = sqrtf(uu);
    }
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(256, 1) nodes_kernel(kvc_params p, ScoreArgs a) {
  extern __shared__ float4 smem4[];
  NodeSmem<D>& sm = *reinterpret_cast<NodeSmem<D>*>(smem4);
  constexpr int VPL = D / 32;
  constexpr int HALF = D / 2;
  const long long tree = blockIdx.x;
  const int s = (int)(tree % p.S_max);
  const long long blh = tree / p.S_max;
  const int b = seq_of(p, blh);
  const int lh = (int)(blh % ((long long)p.L * p.H));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float* util_out = a.op_util + tree * kOps;
  int32_t* cost_out = a.op_cost + tree * kOps;
  if (!a.ok[blh] || s >= a.n_slots[b]) {
    if (tid < kOps) { util_out[tid] = 0.f; cost_out[tid] = 0; }
    return;
  }
  const int n = a.ctx_len[b];
  const int x0 = a.bounds[(long long)b * (p.S_max + 1) + s];
  const int y0 = a.bounds[(long long)b * (p.S_max + 1) + s + 1];
  const uint8_t* cuts = kvcd::tree_cuts_of(p, blh, s);
  const int len = y0 - x0;
  const int R = p.G * p.P;
  const int64_t row0 = kvcd::seq_token_base(a.ctx_len, b, p.L * p.H) + (int64_t)lh * n;
  load_rows<T, D>(&sm.K[0][0], static_cast<const T*>(a.K) + (row0 + x0) * D, 0, len, len);
  load_rows<T, D>(&sm.V[0][0], static_cast<const T*>(a.V) + (row0 + x0) * D, 0, len, len);
  for (int i = tid; i < len; i += blockDim.x) sm.r[i] = a.rel[row0 + x0 + i];
  if (tid < 60) (&sm.acc[0][0])[tid] = 0.f;
  __syncthreads();

  // ---- prototypes: one warp per node; lane owns RoPE pairs (j, j + D/2)
  constexpr int VP = D / 64;
  for (int j = warp; j < 15; j += 8) {
    int x, y;
    node_range(cuts, j, x0, y0, x, y);
    const int c = y - x;
    float rs = 0.f;
    for (int i = x + lane; i < y; i += 32) rs += sm.r[i - x0];
    rs = kvcd::warp_sum(rs);
    float kb_lo[VP], kb_hi[VP], vb_lo[VP], vb_hi[VP];
#pragma unroll
    for (int t = 0; t < VP; ++t) kb_lo[t] = kb_hi[t] = vb_lo[t] = vb_hi[t] = 0.f;
    const float f = p.value_floor;
    for (int i = x; i < y; ++i) {
      const float* kr = sm.K[i - x0];
      const float* vr = sm.V[i - x0];
      const float* ct = a.cos_tab + (int64_t)(2 * i) * HALF + lane * VP;
      const float* st = a.sin_tab + (int64_t)(2 * i) * HALF + lane * VP;
      const float w = rs > 0.f ? (1.f - f) * (sm.r[i - x0] / rs) + f / (float)c : 1.f / (float)c;
#pragma unroll
      for (int t = 0; t < VP; ++t) {
        const float cs = __ldg(ct + t), sn = __ldg(st + t);
        const float lo = kr[lane * VP + t], hi = kr[HALF + lane * VP + t];
        kb_lo[t] += lo * cs + hi * sn;
        kb_hi[t] += hi * cs - lo * sn;
        vb_lo[t] = fmaf(w, vr[lane * VP + t], vb_lo[t]);
        vb_hi[t] = fmaf(w, vr[HALF + lane * VP + t], vb_hi[t]);
      }
    }
    const float inv_c = 1.f / (float)c;
    float nb2 = 0.f;
#pragma unroll
    for (int t = 0; t < VP; ++t) {
      kb_lo[t] *= inv_c; kb_hi[t] *= inv_c;
      nb2 += kb_lo[t] * kb_lo[t] + kb_hi[t] * kb_hi[t];
    }
    const float nb = sqrtf(kvcd::warp_sum(nb2));
    float kap = 0.f;
    for (int i = x; i < y; ++i) {
      const float* kr = sm.K[i - x0];
      const float* ct = a.cos_tab + (int64_t)(2 * i) * HALF + lane * VP;
      const float* st = a.sin_tab + (int64_t)(2 * i) * HALF + lane * VP;
      float dot = 0.f, nk2 = 0.f;
#pragma unroll
      for (int t = 0; t < VP; ++t) {
        const float cs = __ldg(ct + t), sn = __ldg(st + t);
        const float lo = kr[lane * VP + t], hi = kr[HALF + lane * VP + t];
        const float ul = lo * cs + hi * sn, uh = hi * cs - lo * sn;
        dot += ul * kb_lo[t] + uh * kb_hi[t];
        nk2 += ul * ul + uh * uh;
      }
      dot = kvcd::warp_sum(dot);
      nk2 = kvcd::warp_sum(nk2);
      const float den = sqrtf(nk2) * nb;
      kap += den > 0.f ? dot / den : 0.f;
    }
    kap *= inv_c;
    const float m = (float)c * fminf(fmaxf(kap, inv_c), 1.f);
    const float* ct = a.cos_tab + (int64_t)(x + y - 1) * HALF + lane * VP;
    const float* st = a.sin_tab + (int64_t)(x + y - 1) * HALF + lane * VP;
#pragma unroll
    for (int t = 0; t < VP; ++t) {
      const float cs = __ldg(ct + t), sn = __ldg(st + t);
      sm.kh[j][lane * VP + t] = kb_lo[t] * cs - kb_hi[t] * sn;
      sm.kh[j][HALF + lane * VP + t] = kb_hi[t] * cs + kb_lo[t] * sn;
      sm.vh[j][lane * VP + t] = vb_lo[t];
      sm.vh[j][HALF + lane * VP + t] = vb_hi[t];
    }
    if (lane == 0) { sm.logm[j] = logf(m); sm.Rv[j] = rs; }
  }
  __syncthreads();

  // ---- per 64-row group: attention of the rows to the slot tokens and nodes
  for (int rg = 0; rg < R; rg += 64) {
    const int rl = tid & 63, sub = tid >> 6;     // row in group, token subset
    const int rho = rg + rl;
    if (rho < R) {
      float q[D];
      load_q<T, D>(q, static_cast<const T*>(a.Qp) + (blh * R + rho) * D, a.q_scale2);
      const float l2 = a.lse2[blh * R + rho];
      const int limit = n - p.P + (rho % p.P);
      for (int i = sub; i < len; i += 4) {
        const float s2 = dot1(q, sm.K[i], D);
        sm.A[i][rl] = (x0 + i <= limit) ? exp2f(s2 - l2) : 0.f;
      }
      for (int j = sub; j < 15; j += 4) {
        const float s2 = dot1(q, sm.kh[j], D) + sm.logm[j] * kLog2e - l2;
        sm.Ah[j][rl] = exp2f(s2);
      }
    } else {
      for (int i = sub; i < len; i += 4) sm.A[i][rl] = 0.f;
      for (int j = sub; j < 15; j += 4) sm.Ah[j][rl] = 0.f;
    }
    __syncthreads();
    // warp w: row quads 2w and 2w + 1 of the group; lanes own features
    for (int qd = 2 * warp; qd < 2 * warp + 2; ++qd) {
      const int rq = qd * 4;
      float Ad2[4] = {0, 0, 0, 0}, Ad1[4] = {0, 0, 0, 0}, Ar[4] = {0, 0, 0, 0};
      float Ud2[4][VPL], Ud1[4][VPL], Ur[4][VPL];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int t = 0; t < VPL; ++t) Ud2[r][t] = Ud1[r][t] = Ur[r][t] = 0.f;
      for (int j = 7; j < 15; ++j) {
        int x, y;
        node_range(cuts, j, x0, y0, x, y);
        float Al[4] = {0, 0, 0, 0};
        float Ul[4][VPL];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int t = 0; t < VPL; ++t) Ul[r][t] = 0.f;
        for (int i = x - x0; i < y - x0; ++i) {
          const float4 av = *reinterpret_cast<const float4*>(&sm.A[i][rq]);
          const float aa[4] = {av.x, av.y, av.z, av.w};
          float vv[VPL];
#pragma unroll
          for (int t = 0; t < VPL; ++t) vv[t] = sm.V[i][lane * VPL + t];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            Al[r] += aa[r];
#pragma unroll
            for (int t = 0; t < VPL; ++t) Ul[r][t] = fmaf(aa[r], vv[t], Ul[r][t]);
          }
        }
        finish_node<D>(sm, j, rq, Al, Ul, lane);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          Ad2[r] += Al[r];
#pragma unroll
          for (int t = 0; t < VPL; ++t) Ud2[r][t] += Ul[r][t];
        }
        if (j & 1) {                               // left leaf: the isolated token follows
          int x2, y2;
          node_range(cuts, (j - 1) / 2, x0, y0, x2, y2);
          const int e = kvcd::tree_extract(cuts, (j - 1) / 2, x0, x2, y2);
          if (e >= 0) {
            const float4 av = *reinterpret_cast<const float4*>(&sm.A[e - x0][rq]);
            const float aa[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              Ad2[r] += aa[r];
#pragma unroll
              for (int t = 0; t < VPL; ++t) Ud2[r][t] = fmaf(aa[r], sm.V[e - x0][lane * VPL + t], Ud2[r][t]);
            }
          }
        }
        if ((j & 1) == 0) {                        // right child: depth-2 node done
          const int j2 = (j - 1) / 2;
          finish_node<D>(sm, j2, rq, Ad2, Ud2, lane);
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            Ad1[r] += Ad2[r]; Ad2[r] = 0.f;
#pragma unroll
            for (int t = 0; t < VPL; ++t) { Ud1[r][t] += Ud2[r][t]; Ud2[r][t] = 0.f; }
          }
          if ((j2 & 1) == 0) {                     // depth-1 node done
            const int j1 = (j2 - 1) / 2;
            finish_node<D>(sm, j1, rq, Ad1, Ud1, lane);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              Ar[r] += Ad1[r]; Ad1[r] = 0.f;
#pragma unroll
              for (int t = 0; t < VPL; ++t) { Ur[r][t] += Ud1[r][t]; Ud1[r][t] = 0.f; }
            }
            if (j1 == 2) finish_node<D>(sm, 0, rq, Ar, Ur, lane);
          }
        }
      }
    }
    __syncthreads();
    // fixed-order sums over the group's valid rows
    if (tid < 60) {
      const int k = tid / 15, j = tid % 15;
      float sacc = 0.f;
      const int rows = min(64, R - rg);
      for (int r = 0; r < rows; ++r) sacc += sm.st[k][j][r];
      sm.acc[k][j] += sacc;
    }
    __syncthreads();
  }

  // ---- distortions and the 16 ops of this slot
  if (tid == 0) {
    const float nu = a.nu[blh];
    const float invR = 1.f / (float)R;
    float Dn[15], Dd[15];
    for (int j = 0; j < 15; ++j) {
      const float vt = nu > 0.f ? sm.acc[2][j] * invR / nu : 0.f;
      const float vd = nu > 0.f ? sm.acc[3][j] * invR / nu : 0.f;
      Dn[j] = p.w_part * (sm.acc[0][j] * invR) + p.w_value * vt;
      Dd[j] = p.w_part * (sm.acc[1][j] * invR) + p.w_value * vd;
    }
    const float sens = a.head_sens ? a.head_sens[lh] : 1.f;
    auto gainf = [](float num, float dd) {
      if (!(dd > 0.f)) return 0.f;
      return fminf(fmaxf(num / dd, 0.f), 1.f);
    };
    util_out[0] = sm.Rv[0] * gainf(Dd[0] - Dn[0], Dd[0]) * sens;
    cost_out[0] = 1;
    for (int j = 0; j < 15; ++j) {
      float g;
      int c;
      if (j < 7) {
        g = gainf(Dn[j] - Dn[2 * j + 1] - Dn[2 * j + 2], Dd[j]);
        c = internal_split_cost(cuts, j, x0, y0);
      } else {
        int x, y;
        node_range(cuts, j, x0, y0, x, y);
        c = y - x - 1;
        g = gainf(Dn[j], Dd[j]);
      }
      util_out[1 + j] = sm.Rv[j] * g * sens / (float)c;
      cost_out[1 + j] = c;
    }
  }
}

// ---------------------------------------------------------------- tensor-core node path
// Per slot tree: the 15 prototypes (fp32), their keys split into three bf16
// parts (k^ = p0 + p1 + p2 to fp32 accuracy) laid out as the 128-byte-swizzled
// K-major operand of the tensor-core node kernel, and each node's relevance.
//
// One warp per slot tree, one pass over its tokens in order.  Lane l owns the
// RoPE pairs (2l, 2l + 64) and (2l + 1, 2l + 65).  Per token: unrotate the
// key (u = R(-pos) k), its norm (one warp reduction), and accumulate, per
// node, sum u, sum u/|u|, sum v, sum r v and sum r.  Every node's sums are
// sums over its leaves, so the accumulators run depth-first (leaf, depth 2,
// depth 1, root) and each node is finished the moment its last leaf ends:
//   mu = sum u / c,   kappa = mean_i cos(u_i, mu) = (sum u/|u|) . mu / (c |mu|),
//   m = c clamp(kappa, 1/c, 1),   k^ = R(pbar) mu,   pbar = (x + y - 1) / 2,
//   v^ = (1 - f) sum(r v) / sum r + f sum v / c   (sum v / c when sum r = 0).
struct ProtoAcc {
  float k[4], u[4], v[4], rv[4], r;
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int t = 0; t < 4; ++t) k[t] = u[t] = v[t] = rv[t] = 0.f;
    r = 0.f;
  }
  __device__ __forceinline__ void add(const ProtoAcc& o) {
#pragma unroll
    for (int t = 0; t < 4; ++t) { k[t] += o.k[t]; u[t] += o.u[t]; v[t] += o.v[t]; rv[t] += o.rv[t]; }
    r += o.r;
  }
};

__device__ __forceinline__ uint32_t bf16_pair(float a, float b) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
}

// Writes node j's record entries from its sums (lane l: features 2l, 2l+1,
// 2l+64, 2l+65; t = 0..3 in that order).
__device__ __forceinline__ void proto_finish(const ScoreArgs& a, float value_floor, int j, int x,
                                             int y, const ProtoAcc& s, unsigned char* out,
                                             int lane) {
  const float inv_c = 1.f / (float)(y - x);
  float mu[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) mu[t] = s.k[t] * inv_c;
  const float mu2 = kvcd::warp_sum(mu[0] * mu[0] + mu[1] * mu[1] + mu[2] * mu[2] + mu[3] * mu[3]);
  const float um = kvcd::warp_sum(s.u[0] * mu[0] + s.u[1] * mu[1] + s.u[2] * mu[2] + s.u[3] * mu[3]);
  const float kbn = sqrtf(mu2);
  const float kap = kbn > 0.f ? um / kbn * inv_c : 0.f;
  const float m = (float)(y - x) * fminf(fmaxf(kap, inv_c), 1.f);
  // rerotate the mean at the half-integer position pbar (table row x + y - 1)
  const int e = x + y - 1;
  const float2 cs = __ldg(reinterpret_cast<const float2*>(a.cos_tab + (int64_t)e * 64) + lane);
  const float2 sn = __ldg(reinterpret_cast<const float2*>(a.sin_tab + (int64_t)e * 64) + lane);
  float kh[4];
  kh[0] = mu[0] * cs.x - mu[2] * sn.x;
  kh[2] = mu[2] * cs.x + mu[0] * sn.x;
  kh[1] = mu[1] * cs.y - mu[3] * sn.y;
  kh[3] = mu[3] * cs.y + mu[1] * sn.y;
  // three bf16 parts, rows 16 part + j of the two 64-feature blocks
  float r1[4], r2[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    r1[t] = kh[t] - __bfloat162float(__float2bfloat16_rn(kh[t]));
    r2[t] = r1[t] - __bfloat162float(__float2bfloat16_rn(r1[t]));
  }
  const int cc = lane >> 2, wo = (lane & 3) * 4;   // 16-byte chunk, byte within it
#pragma unroll
  for (int part = 0; part < 3; ++part) {
    const float* src = part == 0 ? kh : (part == 1 ? r1 : r2);
    const int row = 16 * part + j;
    const int off = row * 128 + ((cc ^ (row & 7)) << 4) + wo;
    *reinterpret_cast<uint32_t*>(out + off) = bf16_pair(src[0], src[1]);
    *reinterpret_cast<uint32_t*>(out + 6144 + off) = bf16_pair(src[2], src[3]);
  }
  float* vh = reinterpret_cast<float*>(out + kvc::kProtoVhOff) + j * 128;
  float vv[4];
#pragma unroll
  for (int t = 0; t < 4; ++t)
    vv[t] = s.r > 0.f ? (1.f - value_floor) * (s.rv[t] / s.r) + value_floor * s.v[t] * inv_c
                      : s.v[t] * inv_c;
  *reinterpret_cast<float2*>(vh + 2 * lane) = make_float2(vv[0], vv[1]);
  *reinterpret_cast<float2*>(vh + 64 + 2 * lane) = make_float2(vv[2], vv[3]);
  if (lane == 0) {
    reinterpret_cast<float*>(out + kvc::kProtoLogmOff)[j] = logf(m);
    reinterpret_cast<float*>(out + kvc::kProtoRvOff)[j] = s.r;
  }
}

// Accumulators of the depth-2, depth-1 and root nodes live in shared memory
// (lane-indexed, conflict-free); only the current leaf's sums are registers.
struct ProtoLevels {
  float v[3][17][32];
};

__device__ __forceinline__ void acc_to_smem(ProtoLevels& sm, int lvl, const ProtoAcc& s, int lane,
                                            bool add) {
  float* f = &sm.v[lvl][0][lane];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    f[(0 + t) * 32] = (add ? f[(0 + t) * 32] : 0.f) + s.k[t];
    f[(4 + t) * 32] = (add ? f[(4 + t) * 32] : 0.f) + s.u[t];
    f[(8 + t) * 32] = (add ? f[(8 + t) * 32] : 0.f) + s.v[t];
    f[(12 + t) * 32] = (add ? f[(12 + t) * 32] : 0.f) + s.rv[t];
  }
  f[16 * 32] = (add ? f[16 * 32] : 0.f) + s.r;
}
__device__ __forceinline__ ProtoAcc acc_from_smem(const ProtoLevels& sm, int lvl, int lane) {
  ProtoAcc s;
  const float* f = &sm.v[lvl][0][lane];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    s.k[t] = f[(0 + t) * 32];
    s.u[t] = f[(4 + t) * 32];
    s.v[t] = f[(8 + t) * 32];
    s.rv[t] = f[(12 + t) * 32];
  }
  s.r = f[16 * 32];
  return s;
}

// One warp per block: slot trees differ in length and a block retires with its
// slowest warp, so single-warp blocks let the block scheduler balance them
// (the same choice as the pack kernel).  24 blocks per SM at 80 registers:
// measured at 16K, 1.03 ms against 1.15 with 20 blocks at 96 registers and
// 1.10 with 28 at 72.
#ifndef KVC_PROTO_WARPS
#define KVC_PROTO_WARPS 1
#endif
constexpr int kProtoWarps = KVC_PROTO_WARPS;

template <typename T, int D>
__global__ void __launch_bounds__(32 * kProtoWarps, 24 / kProtoWarps)
    proto_kernel(kvc_params p, ScoreArgs a, unsigned char* proto) {
  static_assert(D == 128 && sizeof(T) == 2, "tensor-core node path is bf16, d = 128");
  __shared__ ProtoLevels levels[kProtoWarps];
  const int lane = threadIdx.x & 31;
  ProtoLevels& lv = levels[threadIdx.x >> 5];
  const long long tree = (long long)blockIdx.x * kProtoWarps + (threadIdx.x >> 5);
  if (tree >= (long long)p.B * p.L * p.H * p.S_max) return;
  const int s = (int)(tree % p.S_max);
  const long long blh = tree / p.S_max;
  const int b = seq_of(p, blh);
  const int lh = (int)(blh % ((long long)p.L * p.H));
  if (!a.ok[blh] || s >= a.n_slots[b]) return;
  const int n = a.ctx_len[b];
  const int x0 = a.bounds[(long long)b * (p.S_max + 1) + s];
  const int y0 = a.bounds[(long long)b * (p.S_max + 1) + s + 1];
  const uint8_t* cuts = kvcd::tree_cuts_of(p, blh, s);
  const int64_t row0 = kvcd::seq_token_base(a.ctx_len, b, p.L * p.H) + (int64_t)lh * n;
  const uint32_t* Kw = reinterpret_cast<const uint32_t*>(static_cast<const T*>(a.K) + row0 * D);
  const uint32_t* Vw = reinterpret_cast<const uint32_t*>(static_cast<const T*>(a.V) + row0 * D);
  const float* rel = a.rel + row0;
  unsigned char* out = proto + tree * kvc::kProtoBytes;
  const float inv_pos = 1.f / (float)max(n - 1, 1);
  float nv_sum = 0.f;                                    // sum of |v| over the slot's tokens
  // tokens [x, y) into `acc` (and their |v| and position features)
  auto stream = [&](int x, int y, ProtoAcc& leaf) {
    // tokens in groups of 4: all loads of a group first, then four interleaved
    // |u| reductions
    for (int i0 = x; i0 < y; i0 += 4) {
      const int ng = min(4, y - i0);
      uint32_t kl[4], kh[4], vl[4], vh[4];
      float2 cs[4], sn[4];
      float ri[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int i = i0 + (g < ng ? g : 0);            // a repeated row is loaded, not used
        kl[g] = __ldg(Kw + (int64_t)i * (D / 2) + lane);
        kh[g] = __ldg(Kw + (int64_t)i * (D / 2) + 32 + lane);
        vl[g] = __ldg(Vw + (int64_t)i * (D / 2) + lane);
        vh[g] = __ldg(Vw + (int64_t)i * (D / 2) + 32 + lane);
        cs[g] = __ldg(reinterpret_cast<const float2*>(a.cos_tab + (int64_t)(2 * i) * 64) + lane);
        sn[g] = __ldg(reinterpret_cast<const float2*>(a.sin_tab + (int64_t)(2 * i) * 64) + lane);
        ri[g] = __ldg(rel + i);
      }
      float u[4][4], nk2[4], nv2[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const float k0 = __uint_as_float(kl[g] << 16), k1 = __uint_as_float(kl[g] & 0xFFFF0000u);
        const float k2 = __uint_as_float(kh[g] << 16), k3 = __uint_as_float(kh[g] & 0xFFFF0000u);
        u[g][0] = k0 * cs[g].x + k2 * sn[g].x;
        u[g][2] = k2 * cs[g].x - k0 * sn[g].x;
        u[g][1] = k1 * cs[g].y + k3 * sn[g].y;
        u[g][3] = k3 * cs[g].y - k1 * sn[g].y;
        nk2[g] = u[g][0] * u[g][0] + u[g][1] * u[g][1] + u[g][2] * u[g][2] + u[g][3] * u[g][3];
        const float v0 = __uint_as_float(vl[g] << 16), v1 = __uint_as_float(vl[g] & 0xFFFF0000u);
        const float v2 = __uint_as_float(vh[g] << 16), v3 = __uint_as_float(vh[g] & 0xFFFF0000u);
        nv2[g] = v0 * v0 + v1 * v1 + v2 * v2 + v3 * v3;
      }
      kvcd::warp_sum4(nk2, lane);
      kvcd::warp_sum4(nv2, lane);
      // the value-norm and position features of these tokens (lane g writes token g)
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        if (g < ng) {
          const float nv = sqrtf(nv2[g]);
          nv_sum += nv;
          if (lane == g) {
            float* f = a.feats + (row0 + i0 + g) * 5;
            f[1] = nv;
            f[4] = (float)(i0 + g) * inv_pos;
          }
        }
      }
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        if (g < ng) {
          const float inv = nk2[g] > 0.f ? rsqrtf(nk2[g]) : 0.f;
          const float v[4] = {__uint_as_float(vl[g] << 16), __uint_as_float(vl[g] & 0xFFFF0000u),
                              __uint_as_float(vh[g] << 16), __uint_as_float(vh[g] & 0xFFFF0000u)};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            leaf.k[t] += u[g][t];
            leaf.u[t] = fmaf(u[g][t], inv, leaf.u[t]);
            leaf.v[t] += v[t];
            leaf.rv[t] = fmaf(ri[g], v[t], leaf.rv[t]);
          }
          leaf.r += ri[g];
        }
      }
    }
  };
  for (int L = 0; L < 8; ++L) {
    int x, y;
    node_range(cuts, 7 + L, x0, y0, x, y);
    ProtoAcc leaf;
    leaf.zero();
    stream(x, y, leaf);
    proto_finish(a, p.value_floor, 7 + L, x, y, leaf, out, lane);
    acc_to_smem(lv, 0, leaf, lane, (L & 1) != 0);           // depth 2 = leaf pair
    if (!(L & 1)) {                                          // and its isolated token
      int x2, y2;
      node_range(cuts, 3 + (L >> 1), x0, y0, x2, y2);
      const int e = kvcd::tree_extract(cuts, 3 + (L >> 1), x0, x2, y2);
      if (e >= 0) {
        ProtoAcc tok;
        tok.zero();
        stream(e, e + 1, tok);
        acc_to_smem(lv, 0, tok, lane, true);
      }
    }
    if (L & 1) {
      const int j2 = 3 + (L >> 1);
      node_range(cuts, j2, x0, y0, x, y);
      const ProtoAcc d2 = acc_from_smem(lv, 0, lane);
      proto_finish(a, p.value_floor, j2, x, y, d2, out, lane);
      acc_to_smem(lv, 1, d2, lane, (L & 3) == 3);            // depth 1 = depth-2 pair
      if ((L & 3) == 3) {
        const int j1 = 1 + (L >> 2);
        node_range(cuts, j1, x0, y0, x, y);
        const ProtoAcc d1 = acc_from_smem(lv, 1, lane);
        proto_finish(a, p.value_floor, j1, x, y, d1, out, lane);
        acc_to_smem(lv, 2, d1, lane, L == 7);                // root = depth-1 pair
      }
    }
  }
  const ProtoAcc root = acc_from_smem(lv, 2, lane);
  proto_finish(a, p.value_floor, 0, x0, y0, root, out, lane);
  if (lane == 0) a.nu_part[blh * (p.S_max + 1) + s] = nv_sum;
  // row 15 of every part is padding: zero key, ln m = 0, no relevance
#pragma unroll
  for (int part = 0; part < 3; ++part) {
    const int row = 16 * part + 15;
    const int off = row * 128 + lane * 4;
    *reinterpret_cast<uint32_t*>(out + off) = 0u;
    *reinterpret_cast<uint32_t*>(out + 6144 + off) = 0u;
  }
  if (lane == 0) {
    reinterpret_cast<float*>(out + kvc::kProtoLogmOff)[15] = 0.f;
    reinterpret_cast<float*>(out + kvc::kProtoRvOff)[15] = 0.f;
  }
}

// Per slot: combine the row-tile partial statistics into D, D_drop and the 16
// op utilities / costs (same formulas as the node kernel's tail).
__global__ void ops_kernel(kvc_params p, ScoreArgs a, const unsigned char* proto,
                           const float* npart, int n_mt) {
  const long long tree = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (tree >= (long long)p.B * p.L * p.H * p.S_max) return;
  const int s = (int)(tree % p.S_max);
  const long long blh = tree / p.S_max;
  const int b = seq_of(p, blh);
  const int lh = (int)(blh % ((long long)p.L * p.H));
  float* util_out = a.op_util + tree * kOps;
  int32_t* cost_out = a.op_cost + tree * kOps;
  if (!a.ok[blh] || s >= a.n_slots[b]) {
    for (int o = 0; o < kOps; ++o) { util_out[o] = 0.f; cost_out[o] = 0; }
    return;
  }
  const int x0 = a.bounds[(long long)b * (p.S_max + 1) + s];
  const int y0 = a.bounds[(long long)b * (p.S_max + 1) + s + 1];
  const uint8_t* cuts = kvcd::tree_cuts_of(p, blh, s);
  const float* rv = reinterpret_cast<const float*>(proto + tree * kvc::kProtoBytes + kvc::kProtoRvOff);
  const float nu = a.nu[blh];
  const float invR = 1.f / (float)(p.G * p.P);
  float Dn[15], Dd[15];
  for (int j = 0; j < 15; ++j) {
    float st[4] = {0.f, 0.f, 0.f, 0.f};
    for (int mt = 0; mt < n_mt; ++mt)
      for (int k = 0; k < 4; ++k) st[k] += npart[((tree * 2 + mt) * 15 + j) * 4 + k];
    const float vt = nu > 0.f ? st[2] * invR / nu : 0.f;
    const float vd = nu > 0.f ? st[3] * invR / nu : 0.f;
    Dn[j] = p.w_part * (st[0] * invR) + p.w_value * vt;
    Dd[j] = p.w_part * (st[1] * invR) + p.w_value * vd;
  }
  const float sens = a.head_sens ? a.head_sens[lh] : 1.f;
  auto gainf = [](float num, float dd) {
    if (!(dd > 0.f)) return 0.f;
    return fminf(fmaxf(num / dd, 0.f), 1.f);
  };
  util_out[0] = rv[0] * gainf(Dd[0] - Dn[0], Dd[0]) * sens;
  cost_out[0] = 1;
  for (int j = 0; j < 15; ++j) {
    float g;
    int c;
    if (j < 7) {
      g = gainf(Dn[j] - Dn[2 * j + 1] - Dn[2 * j + 2], Dd[j]);
      c = internal_split_cost(cuts, j, x0, y0);
    } else {
      int x, y;
      node_range(cuts, j, x0, y0, x, y);
      c = y - x - 1;
      g = gainf(Dn[j], Dd[j]);
    }
    util_out[1 + j] = rv[j] * g * sens / (float)c;
    cost_out[1 + j] = c;
  }
}

// Per-(b,l,h) checks of the device-side inputs.
__global__ void score_check_kernel(kvc_params p, ScoreArgs a) {
  const long long blh = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (blh >= (long long)p.B * p.L * p.H) return;
  const int b = seq_of(p, blh);
  const int n = a.ctx_len[b];
  const int S = a.n_slots[b];
  bool ok = n >= p.W + 16 && n <= p.n_max && S >= 1 && S <= p.S_max;
  if (ok) {
    const int32_t* bd = a.bounds + (long long)b * (p.S_max + 1);
    ok = bd[0] == 0 && bd[S] == n - p.W;
    for (int s = 0; ok && s < S; ++s) {
      const int ln = bd[s + 1] - bd[s];
      ok = ln >= 16 && ln <= 128;
    }
  }
  a.ok[blh] = ok ? 1 : 0;
  if (!ok) kvcd::record_error(a.err, KVC_EDEVICE);
}

// One thread per slot tree: a cut table entry that the tree helpers would
// replace by the midpoint is reported (the replacement keeps every kernel on
// one valid tree).
__global__ void cuts_check_kernel(kvc_params p, ScoreArgs a) {
  const long long tree = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (tree >= (long long)p.B * p.L * p.H * p.S_max) return;
  const int s = (int)(tree % p.S_max);
  const long long blh = tree / p.S_max;
  const int b = seq_of(p, blh);
  const int S = a.n_slots[b];
  if (s >= S || S > p.S_max) return;
  const int x0 = a.bounds[(long long)b * (p.S_max + 1) + s];
  const int y0 = a.bounds[(long long)b * (p.S_max + 1) + s + 1];
  if (x0 < 0 || y0 - x0 < 16 || y0 - x0 > 128) return;   // score_check_kernel reports it
  const uint8_t* cuts = kvcd::tree_cuts_of(p, blh, s);
  for (int j = 0; j < 7; ++j) {
    int x, y;
    kvcd::tree_node_range(cuts, j, x0, y0, x, y);
    const bool three = j >= 3 && ((cuts[7] >> (j - 3)) & 1);
    const bool ok = three ? kvcd::tree_extract_valid(x0 + (int)cuts[j], x, y)
                          : (cuts[j] == 0 ||     // unset: the midpoint
                             kvcd::tree_cut_valid(x0 + (int)cuts[j], kvcd::tree_depth(j), x, y));
    if (!ok) {
      kvcd::record_error(a.err, KVC_EDEVICE);
      return;
    }
  }
}

// Three-way salient child sets ([GK] "Technical details and default settings":
// tree construction may isolate a salient token with a three-way child set).
// One warp per slot tree, after the relevance hops: each depth-2 node j = 3..6
// covering [a, b) (at most 32 tokens, one per lane) takes its most relevant
// token t (largest relevance, ties to the smaller position); when both sides
// keep 2..15 tokens the node isolates it: byte j = t - x0 and bit j - 3 of
// byte 7 are set, otherwise the bit is cleared and byte j (the binary cut) is
// left as it is.
__global__ void salient_kernel(kvc_params p, ScoreArgs a) {
  const long long tree = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (tree >= (long long)p.B * p.L * p.H * p.S_max) return;
  const int s = (int)(tree % p.S_max);
  const long long blh = tree / p.S_max;
  const int b = seq_of(p, blh);
  const int lh = (int)(blh % ((long long)p.L * p.H));
  if (!a.ok[blh] || s >= a.n_slots[b]) return;
  const int n = a.ctx_len[b];
  const int x0 = a.bounds[(long long)b * (p.S_max + 1) + s];
  const int y0 = a.bounds[(long long)b * (p.S_max + 1) + s + 1];
  uint8_t* cuts = p.tree_cuts + ((long long)blh * p.S_max + s) * 8;
  const float* rel = a.rel + kvcd::seq_token_base(a.ctx_len, b, p.L * p.H) + (int64_t)lh * n;
  unsigned flags = 0;
#pragma unroll
  for (int j = 3; j < 7; ++j) {
    int x, y;
    node_range(cuts, j, x0, y0, x, y);           // depth-2 ranges: cuts of nodes 0..2 only
    const int i = x + lane;
    float best = i < y ? rel[i] : -INFINITY;
    int bi = i < y ? i : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(KVC_FULL_MASK, best, o);
      const int oi = __shfl_xor_sync(KVC_FULL_MASK, bi, o);
      if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
    }
    if (bi != 0x7fffffff && kvcd::tree_extract_valid(bi, x, y)) {
      flags |= 1u << (j - 3);
      if (lane == 0) cuts[j] = (uint8_t)(bi - x0);
    }
  }
  if (lane == 0) cuts[7] = (uint8_t)flags;
}

int chunk_for(const kvc_params* p) {
  int c = 1024;
  while ((p->n_max + c - 1) / c > 32) c *= 2;
  return c;
}

// tensor-core passes: 32 key tiles of 128 per CTA (measured at 16K: 16 tiles
// repeat the query-row set-up too often, 64 leave a long last wave)
constexpr int kTcChunkTiles = 32;
int tc_chunks(const kvc_params* p) { return (p->n_max + kTcChunkTiles * 128 - 1) / (kTcChunkTiles * 128); }

// Shapes the tensor-core passes handle (workspace sizing); at run time the TMA
// descriptor encoder must also be available.
bool tc_shape(const kvc_params* p) {
  return p->total_ctx > 0 && p->dtype == KVC_BF16 && p->d == 128 && p->P % 32 == 0 &&
         p->G * p->P <= 256 && p->P <= 128;
}
bool use_tc(const kvc_params* p) { return tc_shape(p) && kvc::probe_tc_supported(p); }

struct Layout {
  size_t part, lse2, hrow, nu, seeds, seed_w, lse2_h, ok, proto, npart, nu_part, total;
};
Layout layout(const kvc_params* p) {
  const size_t blh = (size_t)kvc::lh_count(p);
  const int nch = std::max((p->n_max + chunk_for(p) - 1) / chunk_for(p), tc_chunks(p));
  const int R = p->G * p->P;
  Layout l;
  size_t o = 0;
  l.part = o; o += kvc::align256(blh * nch * 256 * 3 * sizeof(float));
  l.lse2 = o; o += kvc::align256(blh * R * sizeof(float));
  l.hrow = o; o += kvc::align256(blh * R * sizeof(float));
  l.nu = o; o += kvc::align256(blh * sizeof(float));
  l.seeds = o; o += kvc::align256(blh * p->P * sizeof(int32_t));
  l.seed_w = o; o += kvc::align256(blh * p->P * sizeof(float));
  l.lse2_h = o; o += kvc::align256(blh * p->P * sizeof(float));
  l.ok = o; o += kvc::align256(blh * sizeof(int32_t));
  const size_t trees = tc_shape(p) ? blh * (size_t)p->S_max : 0;
  l.proto = o; o += kvc::align256(trees * kvc::kProtoBytes);
  l.npart = o; o += kvc::align256(trees * 2 * 15 * 4 * sizeof(float));
  l.nu_part = o;
  o += kvc::align256(blh * (size_t)std::max((p->n_max + 255) / 256, p->S_max + 1) * sizeof(float));
  l.total = o;
  return l;
}

// Optional phase timing of the tensor-core path (kvc_set_phase_timing): CUDA
// events recorded on the call's stream between its phases.
constexpr int kPhaseMarks = 7;
std::atomic<int> g_phase_on{0};
std::mutex g_phase_mu;
cudaEvent_t g_phase_ev[kPhaseMarks];
bool g_phase_made = false, g_phase_valid = false;
int g_phase_dev = -1;

void phase_mark(int i, cudaStream_t s) {
  if (g_phase_on.load(std::memory_order_relaxed)) cudaEventRecord(g_phase_ev[i], s);
}
// Called once per kvc_score: creates the events on first use (on the current
// device) and reports whether this call is timed.
bool phase_begin() {
  if (!g_phase_on.load(std::memory_order_relaxed)) return false;
  std::lock_guard<std::mutex> g(g_phase_mu);
  int dev = 0;
  cudaGetDevice(&dev);
  if (g_phase_made && dev != g_phase_dev) return false;
  if (!g_phase_made) {
    for (int i = 0; i < kPhaseMarks; ++i)
      if (cudaEventCreate(&g_phase_ev[i]) != cudaSuccess) return false;
    g_phase_made = true;
    g_phase_dev = dev;
  }
  g_phase_valid = false;
  return true;
}

template <typename T, int D>
int launch_all(const kvc_params* p, ScoreArgs& a, cudaStream_t s) {
  const long long blh = kvc::lh_count(p);
  const int R = p->G * p->P;
  int launches = 0;
  const size_t sm_rows = (size_t)kTile * D * sizeof(float);
  const size_t sm_tile = sm_rows + (size_t)kTile * 257 * sizeof(float);
  const size_t sm_nodes = sizeof(NodeSmem<D>);
  cudaFuncSetAttribute(rowstats_kernel<T, D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)sm_rows);
  cudaFuncSetAttribute(rowstats_kernel<T, D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)sm_rows);
  cudaFuncSetAttribute(feats_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_tile);
  cudaFuncSetAttribute(prop_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_tile);
  cudaFuncSetAttribute(nodes_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)sm_nodes);
  score_check_kernel<<<(unsigned)((blh + 255) / 256), 256, 0, s>>>(*p, a); ++launches;
  if (p->tree_cuts) {
    const long long trees = blh * p->S_max;
    cuts_check_kernel<<<(unsigned)((trees + 255) / 256), 256, 0, s>>>(*p, a);
    ++launches;
  }
  if constexpr (std::is_same<T, __nv_bfloat16>::value && D == 128) {
   if (use_tc(p)) {
    // tensor-core probe-times-key passes
    kvc::ProbeTcArgs t;
    t.ctx_len = a.ctx_len; t.K = a.K; t.V = a.V; t.Qp = a.Qp; t.seeds = a.seeds;
    t.seed_w = a.seed_w; t.lse2 = a.lse2; t.hrow = a.hrow; t.lse2_h = a.lse2_h; t.ok = a.ok;
    t.part = a.part; t.feats = a.feats; t.rel = a.rel; t.err = a.err;
    t.B = p->B; t.L = p->L; t.H = p->H; t.G = p->G; t.P = p->P;
    t.chunk_tiles = kTcChunkTiles; t.n_chunks = tc_chunks(p);
    t.q_scale2 = a.q_scale2; t.hop_weight = p->hop_weight;
    t.wait_ns = kvc::wait_limit_ns(); t.withhold = kvc::withhold_copies();
    a.n_chunks = t.n_chunks;                        // rowcombine loops over these partials
    const int64_t rows_total = p->total_ctx * p->L * p->H;
    const bool timed = phase_begin();
    int st;
    if (timed) phase_mark(0, s);
    if ((st = kvc::probe_tc_pass(kvc::kTcRowstatsProbes, t, rows_total, s)) != KVC_OK) return st;
    if (timed) phase_mark(1, s);
    rowcombine_kernel<false><<<(unsigned)blh, 256, 0, s>>>(*p, a);
    if (timed) phase_mark(2, s);
    if ((st = kvc::probe_tc_pass(kvc::kTcFeats, t, rows_total, s)) != KVC_OK) return st;
    if (timed) phase_mark(3, s);
    vnorm_window_kernel<T, D><<<(unsigned)blh, 128, 0, s>>>(*p, a);
    launches += 2;
    for (int hop = 0; hop < p->n_hops; ++hop) {
      seeds_kernel<<<(unsigned)blh, 1024, 0, s>>>(*p, a);
      if ((st = kvc::probe_tc_pass(kvc::kTcRowstatsSeeds, t, rows_total, s)) != KVC_OK) return st;
      rowcombine_kernel<true><<<(unsigned)blh, 256, 0, s>>>(*p, a);
      if ((st = kvc::probe_tc_pass(kvc::kTcProp, t, rows_total, s)) != KVC_OK) return st;
      launches += 2;
    }
    if (p->salient_extract) {
      salient_kernel<<<(unsigned)((blh * p->S_max * 32 + 255) / 256), 256, 0, s>>>(*p, a);
      ++launches;
    }
    // prototypes, tensor-core node statistics, utilities
    if (timed) phase_mark(4, s);
    proto_kernel<T, D><<<(unsigned)((blh * p->S_max + kProtoWarps - 1) / kProtoWarps),
                         32 * kProtoWarps, 0, s>>>(*p, a, a.proto);
    nu_finish_slots_kernel<<<(unsigned)((blh + 127) / 128), 128, 0, s>>>(*p, a);
    ++launches;
    if (timed) phase_mark(5, s);
    kvc::NodeTcArgs nd;
    nd.ctx_len = a.ctx_len; nd.K = a.K; nd.V = a.V; nd.Qp = a.Qp; nd.lse2 = a.lse2; nd.ok = a.ok;
    nd.bounds = a.bounds; nd.n_slots = a.n_slots; nd.proto = a.proto; nd.npart = a.npart;
    nd.tree_cuts = p->tree_cuts;
    nd.err = a.err; nd.B = p->B; nd.L = p->L; nd.H = p->H; nd.G = p->G; nd.P = p->P;
    nd.S_max = p->S_max; nd.q_scale2 = a.q_scale2;
    nd.wait_ns = t.wait_ns; nd.withhold = t.withhold;
    if ((st = kvc::nodes_tc_pass(nd, rows_total, s)) != KVC_OK) return st;
    if (timed) {
      phase_mark(6, s);
      std::lock_guard<std::mutex> g(g_phase_mu);
      g_phase_valid = true;
    }
    const long long trees = blh * p->S_max;
    ops_kernel<<<(unsigned)((trees + 127) / 128), 128, 0, s>>>(*p, a, a.proto, a.npart,
                                                               (p->G * p->P + 127) / 128);
    launches += 2;
    kvc::count_launch(launches);
    return kvc::cuda_status(cudaGetLastError());
   }
  }
  const dim3 g_rows(a.n_chunks, (unsigned)blh);
  rowstats_kernel<T, D, false><<<g_rows, 256, sm_rows, s>>>(*p, a);
  rowcombine_kernel<false><<<(unsigned)blh, 256, 0, s>>>(*p, a);
  const dim3 g_tiles((p->n_max + kTile - 1) / kTile, (unsigned)blh);
  feats_kernel<T, D><<<g_tiles, 256, sm_tile, s>>>(*p, a);
  numean_kernel<<<(unsigned)blh, 256, 0, s>>>(*p, a);
  launches += 4;
  for (int hop = 0; hop < p->n_hops; ++hop) {
    seeds_kernel<<<(unsigned)blh, 1024, 0, s>>>(*p, a);
    rowstats_kernel<T, D, true><<<g_rows, 256, sm_rows, s>>>(*p, a);
    rowcombine_kernel<true><<<(unsigned)blh, 256, 0, s>>>(*p, a);
    prop_kernel<T, D><<<g_tiles, 256, sm_tile, s>>>(*p, a);
    launches += 4;
  }
  if (p->salient_extract) {
    salient_kernel<<<(unsigned)((blh * p->S_max * 32 + 255) / 256), 256, 0, s>>>(*p, a);
    ++launches;
  }
  nodes_kernel<T, D><<<(unsigned)(blh * p->S_max), 256, sm_nodes, s>>>(*p, a);
  ++launches;
  kvc::count_launch(launches);
  (void)R;
  return kvc::cuda_status(cudaGetLastError());
}

}  // namespace

namespace kvc {
size_t score_workspace_bytes(const kvc_params* p) { return layout(p).total; }
}  // namespace kvc

extern "C" void kvc_set_phase_timing(int on) { g_phase_on.store(on ? 1 : 0); }

extern "C" int kvc_score_phase_ms(float* ms_out, int32_t n) {
  if (!ms_out || n < 1) return KVC_EINVAL;
  std::lock_guard<std::mutex> g(g_phase_mu);
  if (!g_phase_made || !g_phase_valid) return KVC_EINVAL;
  // phases: row statistics, per-key features, norms and hops, prototypes, node statistics
  const int pairs[5][2] = {{0, 1}, {2, 3}, {3, 4}, {4, 5}, {5, 6}};
  if (cudaEventSynchronize(g_phase_ev[kPhaseMarks - 1]) != cudaSuccess) return KVC_ECUDA;
  const int m = n < 5 ? n : 5;
  for (int i = 0; i < m; ++i)
    if (cudaEventElapsedTime(&ms_out[i], g_phase_ev[pairs[i][0]], g_phase_ev[pairs[i][1]]) !=
        cudaSuccess)
      return KVC_ECUDA;
  return m;
}

extern "C" int kvc_score(const kvc_params* p, const int32_t* ctx_len, const void* K, const void* V,
                         const void* Qp, const float* rope_cos, const float* rope_sin,
                         const int32_t* slot_bounds, const int32_t* n_slots,
                         const float* head_sens, float* lse, float* feats, float* relevance,
                         float* op_util, int32_t* op_cost, void* workspace, size_t ws_bytes,
                         void* stream) {
  int st = kvc::check_params(p);
  if (st != KVC_OK) return st;
  if (!ctx_len || !K || !V || !Qp || !rope_cos || !rope_sin || !slot_bounds || !n_slots || !lse ||
      !feats || !relevance || !op_util || !op_cost)
    return KVC_EINVAL;
  if ((reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V) |
       reinterpret_cast<uintptr_t>(Qp)) & 15)
    return KVC_EINVAL;                             // bulk copies and vector loads of rows
  const Layout lay = layout(p);
  if (!workspace || ws_bytes < lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return KVC_EWORKSPACE;
  if (kvc::lh_count(p) > 65535 || (long long)kvc::lh_count(p) * p->S_max > 0x7fffffffLL)
    return KVC_EINVAL;
  if (p->salient_extract && !p->tree_cuts) return KVC_EINVAL;   // the choice is written there
  int32_t* err = kvc::err_word();
  if (!err) return KVC_ECUDA;
  ScoreArgs a;
  a.ctx_len = ctx_len; a.K = K; a.V = V; a.Qp = Qp; a.cos_tab = rope_cos; a.sin_tab = rope_sin;
  a.bounds = slot_bounds; a.n_slots = n_slots; a.head_sens = head_sens; a.lse = lse;
  a.feats = feats; a.rel = relevance; a.op_util = op_util; a.op_cost = op_cost;
  char* w = static_cast<char*>(workspace);
  a.part = reinterpret_cast<float*>(w + lay.part);
  a.lse2 = reinterpret_cast<float*>(w + lay.lse2);
  a.hrow = reinterpret_cast<float*>(w + lay.hrow);
  a.nu = reinterpret_cast<float*>(w + lay.nu);
  a.seeds = reinterpret_cast<int32_t*>(w + lay.seeds);
  a.seed_w = reinterpret_cast<float*>(w + lay.seed_w);
  a.lse2_h = reinterpret_cast<float*>(w + lay.lse2_h);
  a.ok = reinterpret_cast<int32_t*>(w + lay.ok);
  a.proto = reinterpret_cast<unsigned char*>(w + lay.proto);
  a.npart = reinterpret_cast<float*>(w + lay.npart);
  a.nu_part = reinterpret_cast<float*>(w + lay.nu_part);
  a.err = err;
  a.chunk = chunk_for(p);
  a.n_chunks = (p->n_max + a.chunk - 1) / a.chunk;
  a.q_scale2 = kLog2e / sqrtf((float)p->d);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p->dtype == KVC_BF16)
    return p->d == 128 ? launch_all<__nv_bfloat16, 128>(p, a, s) : launch_all<__nv_bfloat16, 64>(p, a, s);
  return p->d == 128 ? launch_all<float, 128>(p, a, s) : launch_all<float, 64>(p, a, s);
}
