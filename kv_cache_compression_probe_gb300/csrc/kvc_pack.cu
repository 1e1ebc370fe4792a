// a3 + a6: merge every stored frontier node into one cache entry and pack the
// ragged per-(layer, KV head) cache (GraceKV "Inside one cache entry" and
// "05 Physical cache packing").
//
// Prototype of tokens [x, y) (c = y - x):
//   k~_i = R(-i) k_i              inverse RoPE to a shared frame
//   kbar = mean k~_i,  kappa = mean cos(k~_i, kbar)
//          (= (sum k~_i/|k~_i|) . kbar / (c |kbar|), accumulated in one pass)
//   m    = c * clamp(kappa, 1/c, 1),  stored as ln m (decode adds it to the logit)
//   k^   = R(pbar) kbar, pbar = (x + y - 1)/2; computed in the frame of the
//          node start x (rotations add up: k^ = R(pbar - x) mean R(-(i - x)) k_i),
//          so every angle is a half-position table row below 256
//   v^   = sum w_i v_i, w_i = (1-f) r_i / sum r + f / c  (uniform when sum r = 0)
// Split leaves store their tokens bit-exact (ln m = 0, pos = i); the W window
// tokens follow the slots.  Entry order per (b,l,h): slots ascending, each
// slot's frontier left to right, then the window.
//
// Layout of the work: kernel 1 counts each slot's stored entries and prefix-
// sums them per (b,l,h) (one warp per (b,l,h)); kernel 2 gives one warp per
// slot tree; a lane owns the RoPE pairs (j, j + d/2) for j = lane*VP .. so the
// rotation needs no exchange between lanes.
#include "kvc_common.cuh"
#include "kvc_internal.h"

// One warp per block: slot trees differ in length and frontier shape, and a
// block retires only with its slowest warp; single-warp blocks let the block
// scheduler balance them (measured at 16K: 0.595 ms against 0.657 with two
// warps per block and 0.67-0.71 with four), and at 64 registers they do not spill.
#ifndef KVC_PACK_WARPS
#define KVC_PACK_WARPS 1
#endif

namespace {

constexpr int kOps = 16;
constexpr int kPackWarps = KVC_PACK_WARPS;   // slot trees (warps) per block

__device__ __forceinline__ void node_range(const uint8_t* cuts, int j, int x0, int y0, int& a,
                                           int& b) {
  kvcd::tree_node_range(cuts, j, x0, y0, a, b);
}

// Stored entries of one slot tree: sum over taken ops of their cost
// (Add 1, internal Split 1, three-way depth-2 Split 2, leaf Split = leaf size - 1).
__device__ __forceinline__ int tree_entries(const uint8_t* cuts, const uint8_t* tk, int x0,
                                            int y0) {
  int n = 0;
  for (int o = 0; o < 8; ++o) n += tk[o] ? 1 : 0;
  for (int j = 3; j < 7; ++j)
    if (tk[1 + j]) {
      int a, b;
      node_range(cuts, j, x0, y0, a, b);
      n += kvcd::tree_extract(cuts, j, x0, a, b) >= 0 ? 1 : 0;
    }
  for (int j = 7; j < 15; ++j)
    if (tk[1 + j]) {
      int a, b;
      node_range(cuts, j, x0, y0, a, b);
      n += (b - a) - 1;
    }
  return n;
}

struct PackArgs {
  const int32_t* ctx_len;
  const void* K;
  const void* V;
  const float* rel;
  const float* cos_tab;
  const float* sin_tab;
  const int32_t* bounds;
  const int32_t* n_slots;
  const uint8_t* taken;
  const int32_t* len_lh;
  const int64_t* off_lh;
  void* Kp;
  void* Vp;
  float* logm;
  float* pos;
  int32_t* slot_base;   // [B, L, H, S_max]
  int32_t* lh_ok;       // [B, L, H] 1 if the (l,h) passed its checks
  int64_t capacity;
  int32_t* err;
};

// One warp per (b,l,h): per-slot entry counts -> exclusive prefix, checks.
__global__ void pack_count_kernel(kvc_params p, PackArgs a) {
  const int warps = blockDim.x >> 5;
  const long long blh = (long long)blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (blh >= (long long)p.B * p.L * p.H) return;
  const int b = (int)(blh / ((long long)p.L * p.H));
  const int n = a.ctx_len[b];
  const int S = a.n_slots[b];
  bool ok = S >= 1 && S <= p.S_max && n >= p.W + 16 && n <= p.n_max;
  const int32_t* bd = a.bounds + (long long)b * (p.S_max + 1);
  int run = 0;
  if (ok) {
    for (int s0 = 0; s0 < S; s0 += 32) {
      const int s = s0 + lane;
      int cnt = 0;
      if (s < S) {
        const int x0 = bd[s], y0 = bd[s + 1];
        if (x0 < 0 || y0 - x0 < 16 || y0 - x0 > 128 || y0 > n - p.W) ok = false;
        else cnt = tree_entries(kvcd::tree_cuts_of(p, blh, s), a.taken + (blh * p.S_max + s) * kOps,
                                x0, y0);
      }
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(KVC_FULL_MASK, incl, o);
        if (lane >= o) incl += v;
      }
      if (s < S) a.slot_base[blh * p.S_max + s] = run + incl - cnt;
      run += __shfl_sync(KVC_FULL_MASK, incl, 31);
    }
    ok = __all_sync(KVC_FULL_MASK, ok);
  }
  if (ok) {
    const int len = a.len_lh[blh];
    ok = (len == run + p.W) && a.off_lh[blh] >= 0 && a.off_lh[blh] + len <= a.capacity;
  }
  if (lane == 0) {
    a.lh_ok[blh] = ok ? 1 : 0;
    if (!ok) kvcd::record_error(a.err, KVC_EDEVICE);
  }
}

template <typename T, int D>
struct Row {
  // lane-owned features: j in [lane*VP, lane*VP + VP) and j + D/2
  static constexpr int VP = D / 64;
};

// Lane l owns the RoPE pairs (l*VP + t, D/2 + l*VP + t), t < VP = D/64.
template <typename T, int D>
__device__ __forceinline__ void load_pairs(const T* row, int lane, float* lo, float* hi) {
  constexpr int VP = D / 64;
  if constexpr (sizeof(T) == 2 && VP == 2) {            // bf16 x 2 per half: one 4-byte load each
    const uint32_t a = __ldg(reinterpret_cast<const unsigned int*>(row) + lane);
    const uint32_t b = __ldg(reinterpret_cast<const unsigned int*>(row + D / 2) + lane);
    lo[0] = __uint_as_float(a << 16); lo[1] = __uint_as_float(a & 0xFFFF0000u);
    hi[0] = __uint_as_float(b << 16); hi[1] = __uint_as_float(b & 0xFFFF0000u);
  } else {
#pragma unroll
    for (int t = 0; t < VP; ++t) {
      lo[t] = kvcd::to_f(row[lane * VP + t]);
      hi[t] = kvcd::to_f(row[D / 2 + lane * VP + t]);
    }
  }
}

// Prototype of tokens [x, y) in one pass: per token the unrotated key u (one
// warp reduction for |u|) feeds sum u and sum u/|u|; then
//   kappa = mean cos(u_i, mean u) = (sum u/|u|) . mean u / (c |mean u|),
//   v^    = (1 - f) sum(r v) / sum r + f sum v / c   (sum v / c when sum r = 0).
template <typename T, int D>
__device__ void write_prototype(const kvc_params& p, const PackArgs& a, const T* Kh, const T* Vh,
                                const float* rh, int x, int y, int64_t dst, int lane) {
  constexpr int VP = D / 64;
  constexpr int HALF = D / 2;
  const int c = y - x;
  float ku_lo[VP], ku_hi[VP], kn_lo[VP], kn_hi[VP], v_lo[VP], v_hi[VP], rv_lo[VP], rv_hi[VP];
#pragma unroll
  for (int t = 0; t < VP; ++t)
    ku_lo[t] = ku_hi[t] = kn_lo[t] = kn_hi[t] = v_lo[t] = v_hi[t] = rv_lo[t] = rv_hi[t] = 0.f;
  float rs = 0.f;
  // tokens in groups of kG: every load of a group is issued before any use and
  // the groups' |u| reductions run interleaved
  constexpr int kG = 4;
  for (int i0 = x; i0 < y; i0 += kG) {
    const int ng = min(kG, y - i0);
    float klo[kG][VP], khi[kG][VP], vlo[kG][VP], vhi[kG][VP], cs[kG][VP], sn[kG][VP], ri[kG];
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      const int i = i0 + (g < ng ? g : 0);              // a repeated row is loaded, not used
      load_pairs<T, D>(Kh + (int64_t)i * D, lane, klo[g], khi[g]);
      load_pairs<T, D>(Vh + (int64_t)i * D, lane, vlo[g], vhi[g]);
      // angles relative to the node start x (rows 0..254 of the half-position
      // table, hot in L1 for every node): the mean of R(-i) k_i is R(-x) times
      // the mean of R(-(i - x)) k_i, and R(-x) cancels in the rerotation below
      const float* ct = a.cos_tab + (int64_t)(2 * (i - x)) * HALF + lane * VP;
      const float* st = a.sin_tab + (int64_t)(2 * (i - x)) * HALF + lane * VP;
      if constexpr (VP == 2) {
        const float2 c2 = __ldg(reinterpret_cast<const float2*>(ct));
        const float2 s2 = __ldg(reinterpret_cast<const float2*>(st));
        cs[g][0] = c2.x; cs[g][1] = c2.y; sn[g][0] = s2.x; sn[g][1] = s2.y;
      } else {
#pragma unroll
        for (int t = 0; t < VP; ++t) { cs[g][t] = __ldg(ct + t); sn[g][t] = __ldg(st + t); }
      }
      ri[g] = __ldg(rh + i);
    }
    float nk2[kG];
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      nk2[g] = 0.f;
#pragma unroll
      for (int t = 0; t < VP; ++t) {
        const float ul = klo[g][t] * cs[g][t] + khi[g][t] * sn[g][t];   // R(-i)
        const float uh = khi[g][t] * cs[g][t] - klo[g][t] * sn[g][t];
        klo[g][t] = ul;
        khi[g][t] = uh;
        nk2[g] += ul * ul + uh * uh;
      }
    }
    static_assert(kG == 4, "warp_sum4");
    kvcd::warp_sum4(nk2, lane);
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      if (g < ng) {
        const float inv = nk2[g] > 0.f ? rsqrtf(nk2[g]) : 0.f;
#pragma unroll
        for (int t = 0; t < VP; ++t) {
          ku_lo[t] += klo[g][t];
          ku_hi[t] += khi[g][t];
          kn_lo[t] = fmaf(klo[g][t], inv, kn_lo[t]);
          kn_hi[t] = fmaf(khi[g][t], inv, kn_hi[t]);
          v_lo[t] += vlo[g][t];
          v_hi[t] += vhi[g][t];
          rv_lo[t] = fmaf(ri[g], vlo[g][t], rv_lo[t]);
          rv_hi[t] = fmaf(ri[g], vhi[g][t], rv_hi[t]);
        }
        rs += ri[g];
      }
    }
  }
  const float inv_c = 1.f / (float)c;
  float mu2 = 0.f, um = 0.f;
#pragma unroll
  for (int t = 0; t < VP; ++t) {
    ku_lo[t] *= inv_c;
    ku_hi[t] *= inv_c;
    mu2 += ku_lo[t] * ku_lo[t] + ku_hi[t] * ku_hi[t];
    um += kn_lo[t] * ku_lo[t] + kn_hi[t] * ku_hi[t];
  }
  const float nb = sqrtf(kvcd::warp_sum(mu2));
  um = kvcd::warp_sum(um);
  const float kap = nb > 0.f ? um / nb * inv_c : 0.f;
  const float m = (float)c * fminf(fmaxf(kap, inv_c), 1.f);
  const float f = p.value_floor;
  // rerotate the mean at pbar = (x + y - 1) / 2: half-position table row x + y - 1
  const float* ct = a.cos_tab + (int64_t)(y - x - 1) * HALF + lane * VP;   // pbar - x
  const float* st = a.sin_tab + (int64_t)(y - x - 1) * HALF + lane * VP;
  T* ko = static_cast<T*>(a.Kp) + dst * D;
  T* vo = static_cast<T*>(a.Vp) + dst * D;
#pragma unroll
  for (int t = 0; t < VP; ++t) {
    const float cs = __ldg(ct + t), sn = __ldg(st + t);
    ko[lane * VP + t] = kvcd::from_f<T>(ku_lo[t] * cs - ku_hi[t] * sn);
    ko[HALF + lane * VP + t] = kvcd::from_f<T>(ku_hi[t] * cs + ku_lo[t] * sn);
    vo[lane * VP + t] = kvcd::from_f<T>(rs > 0.f ? (1.f - f) * (rv_lo[t] / rs) + f * v_lo[t] * inv_c
                                                 : v_lo[t] * inv_c);
    vo[HALF + lane * VP + t] = kvcd::from_f<T>(rs > 0.f ? (1.f - f) * (rv_hi[t] / rs) + f * v_hi[t] * inv_c
                                                        : v_hi[t] * inv_c);
  }
  if (lane == 0) {
    a.logm[dst] = logf(m);
    a.pos[dst] = 0.5f * (float)(x + y - 1);
  }
}

// Tokens [i0, i0 + cnt) stored bit-exact at rows dst.. (16-byte vector copies:
// a row is D * sizeof(T) bytes, a multiple of 16).
template <typename T, int D>
__device__ __forceinline__ void copy_exact(const PackArgs& a, const T* Kh, const T* Vh, int i0,
                                           int cnt, int64_t dst, int lane) {
  constexpr int kRowVec = D * (int)sizeof(T) / 16;
  const uint4* ks = reinterpret_cast<const uint4*>(Kh + (int64_t)i0 * D);
  const uint4* vs = reinterpret_cast<const uint4*>(Vh + (int64_t)i0 * D);
  uint4* kd = reinterpret_cast<uint4*>(static_cast<T*>(a.Kp) + dst * D);
  uint4* vd = reinterpret_cast<uint4*>(static_cast<T*>(a.Vp) + dst * D);
  const int nvec = cnt * kRowVec;
#pragma unroll 4
  for (int e = lane; e < nvec; e += 32) {
    const uint4 kv = __ldg(ks + e), vv = __ldg(vs + e);
    kd[e] = kv;
    vd[e] = vv;
  }
  for (int r = lane; r < cnt; r += 32) {
    a.logm[dst + r] = 0.f;
    a.pos[dst + r] = (float)(i0 + r);
  }
}

// One warp per slot tree (plus one extra "slot" index S per (b,l,h) for the
// window tokens).
template <typename T, int D>
__global__ void __launch_bounds__(32 * kPackWarps, 32 / kPackWarps)
    pack_tree_kernel(kvc_params p, PackArgs a) {
  const int warps = blockDim.x >> 5;
  const long long item = (long long)blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int per = p.S_max + 1;
  if (item >= (long long)p.B * p.L * p.H * per) return;
  const int s = (int)(item % per);
  const long long blh = item / per;
  const int lh = (int)(blh % ((long long)p.L * p.H));
  const int b = (int)(blh / ((long long)p.L * p.H));
  // every per-item word is loaded up front (one round trip instead of a chain
  // of dependent ones); the window item (s == S_max) reads slot 0's words,
  // which stay in range, and ignores them
  const bool window = s == p.S_max;
  const int sl = window ? 0 : s;
  const int ok = a.lh_ok[blh];
  const int n = a.ctx_len[b];
  const int S = a.n_slots[b];
  const int64_t base = a.off_lh[blh];
  const int len = a.len_lh[blh];
  const int32_t* bd = a.bounds + (long long)b * (p.S_max + 1);
  const int x0 = bd[sl], y0 = bd[sl + 1];
  const int sbase = a.slot_base[blh * p.S_max + sl];
  const uint8_t* tk = a.taken + (blh * p.S_max + sl) * kOps;
  uint32_t taken = 0;                                   // bit o = op o taken
#pragma unroll
  for (int o = 0; o < kOps; ++o) taken |= (tk[o] != 0 ? 1u : 0u) << o;
  if (!ok) return;
  const int64_t row0 = kvcd::seq_token_base(a.ctx_len, b, p.L * p.H) + (int64_t)lh * n;
  const T* Kh = static_cast<const T*>(a.K) + row0 * D;
  const T* Vh = static_cast<const T*>(a.V) + row0 * D;
  const float* rh = a.rel + row0;
  if (window) {                                         // window tokens
    copy_exact<T, D>(a, Kh, Vh, n - p.W, p.W, base + len - p.W, lane);
    return;
  }
  if (s >= S) return;
  if (!(taken & 1u)) return;
  const uint8_t* cuts = kvcd::tree_cuts_of(p, blh, s);
  int64_t dst = base + sbase;
  // left-to-right frontier walk with an explicit stack (depth <= 4); an entry
  // -1 - t stands for the salient token t a three-way depth-2 node isolates
  int stack[8];
  int sp = 0;
  stack[sp++] = 0;
  while (sp > 0) {
    const int j = stack[--sp];
    if (j < 0) {
      copy_exact<T, D>(a, Kh, Vh, -1 - j, 1, dst, lane);
      ++dst;
      continue;
    }
    int x, y;
    node_range(cuts, j, x0, y0, x, y);
    if (!((taken >> (1 + j)) & 1u)) {
      write_prototype<T, D>(p, a, Kh, Vh, rh, x, y, dst, lane);
      ++dst;
    } else if (j < 7) {
      const int e = j >= 3 ? kvcd::tree_extract(cuts, j, x0, x, y) : -1;
      stack[sp++] = 2 * j + 2;
      if (e >= 0) stack[sp++] = -1 - e;
      stack[sp++] = 2 * j + 1;
    } else {
      copy_exact<T, D>(a, Kh, Vh, x, y - x, dst, lane);
      dst += y - x;
    }
  }
}

struct Layout {
  size_t slot_base, lh_ok, total;
};
Layout layout(const kvc_params* p) {
  Layout l;
  l.slot_base = 0;
  l.lh_ok = kvc::align256(sizeof(int32_t) * (size_t)kvc::lh_count(p) * p->S_max);
  l.total = l.lh_ok + kvc::align256(sizeof(int32_t) * (size_t)kvc::lh_count(p));
  return l;
}

}  // namespace

namespace kvc {
size_t pack_workspace_bytes(const kvc_params* p) { return layout(p).total; }
}  // namespace kvc

extern "C" int kvc_merge_pack(const kvc_params* p, const int32_t* ctx_len, const void* K,
                              const void* V, const float* relevance, const float* rope_cos,
                              const float* rope_sin, const int32_t* slot_bounds,
                              const int32_t* n_slots, const uint8_t* taken, const int32_t* len_lh,
                              const int64_t* off_lh, void* Kp, void* Vp, float* logm, float* pos,
                              int64_t capacity, void* workspace, size_t ws_bytes, void* stream) {
  int st = kvc::check_params(p);
  if (st != KVC_OK) return st;
  if (!ctx_len || !K || !V || !relevance || !rope_cos || !rope_sin || !slot_bounds || !n_slots ||
      !taken || !len_lh || !off_lh || !Kp || !Vp || !logm || !pos || capacity < 0)
    return KVC_EINVAL;
  if ((reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V) |
       reinterpret_cast<uintptr_t>(Kp) | reinterpret_cast<uintptr_t>(Vp)) & 15)
    return KVC_EINVAL;                             // 16-byte row copies
  const Layout lay = layout(p);
  if (!workspace || ws_bytes < lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return KVC_EWORKSPACE;
  int32_t* err = kvc::err_word();
  if (!err) return KVC_ECUDA;
  PackArgs a;
  a.ctx_len = ctx_len; a.K = K; a.V = V; a.rel = relevance; a.cos_tab = rope_cos;
  a.sin_tab = rope_sin; a.bounds = slot_bounds; a.n_slots = n_slots; a.taken = taken;
  a.len_lh = len_lh; a.off_lh = off_lh; a.Kp = Kp; a.Vp = Vp; a.logm = logm; a.pos = pos;
  char* w = static_cast<char*>(workspace);
  a.slot_base = reinterpret_cast<int32_t*>(w + lay.slot_base);
  a.lh_ok = reinterpret_cast<int32_t*>(w + lay.lh_ok);
  a.capacity = capacity;
  a.err = err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long blh = kvc::lh_count(p);
  pack_count_kernel<<<(unsigned)((blh + 7) / 8), 256, 0, s>>>(*p, a);
  // one warp per slot tree (+ one per window)
  const long long items = blh * (p->S_max + 1);
  const unsigned grid = (unsigned)((items + kPackWarps - 1) / kPackWarps);
  const unsigned threads = 32 * kPackWarps;
  if (p->dtype == KVC_BF16) {
    if (p->d == 128) pack_tree_kernel<__nv_bfloat16, 128><<<grid, threads, 0, s>>>(*p, a);
    else pack_tree_kernel<__nv_bfloat16, 64><<<grid, threads, 0, s>>>(*p, a);
  } else {
    if (p->d == 128) pack_tree_kernel<float, 128><<<grid, threads, 0, s>>>(*p, a);
    else pack_tree_kernel<float, 64><<<grid, threads, 0, s>>>(*p, a);
  }
  kvc::count_launch(2);
  return kvc::cuda_status(cudaGetLastError());
}
