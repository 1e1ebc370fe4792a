// a5: per-sequence budget, capped singleton floor and the global greedy
// Add/Split auction (GraceKV "Core idea" budget regions, "Exact-information
// safeguard", "04 Top-down budget flow").
//
// The auction is specified as a heap: pop the exposed op with the highest
// (utility, -op id), take it if its cost fits, expose its children.  The GPU
// reaches the identical taken set without a heap:
//   * Effective key.  For an untaken op o, e(o) = key(o) if o is exposed at
//     the start (Add of an absent slot, or Split of a present unsplit node),
//     else min(key(o), e(parent(o))).  Ops pop in descending e; ops sharing
//     one e form a connected block under its head and pop consecutively in the
//     heap order restricted to the block (its "rank").  Sort key =
//     (e, head id, rank), all distinct.
//   * Prefix cut.  Every op before the first op that does not fit is taken
//     (its parent always precedes it), so the cut is a cost-weighted radix
//     select over the 64-bit sort keys (8 passes of 8-bit digits).
//   * Tail.  After the cut the remaining budget is smaller than the cut op's
//     cost (<= 15), so at most 15 more ops can be bought; each is found as the
//     largest remaining key whose parent is taken and whose cost fits.
// The floor is specified as a scan of candidate tokens in (r * sens desc,
// index asc) order that stops at the first path that does not fit.  Inside
// the stop prefix every earlier candidate was taken, so a candidate's path
// cost is fixed by whether it is the first candidate of its tree, depth-1
// node, depth-2 node and leaf; the stop is again a weighted radix select.
#include <algorithm>

#include "kvc_common.cuh"
#include "kvc_internal.h"

namespace {

constexpr int kOps = 16;
constexpr int kPasses = 8;          // 8-bit digits of a 64-bit key
constexpr int kSelects = 3;         // floor entries, floor tokens, auction
constexpr int kTailIters = 16;

struct SeqBudget {
  long long B_alloc;      // allocatable entries (budget minus the window)
  long long cap_entries;  // floor cap in entries (min with B_alloc)
  long long cap_tokens;   // floor cap in tokens (< 0: none)
  unsigned long long floor_spent;
  unsigned long long floor_tokens;
  long long tail_rem;     // remaining budget during the tail
  unsigned long long tail_last;   // tail scans keys <= tail_last
  unsigned long long tail_best;   // best eligible key of the current tail step
  int tail_done;
  int pad;
};

struct RadixState {
  unsigned long long prefix;
  long long rem;
  int done;     // 1 once the crossing is resolved (or absent)
  int found;    // 1 if some item does not fit (prefix = its key)
};

struct SelWs {
  SeqBudget* seq;            // [B]
  RadixState* rs;            // [kSelects][B]
  unsigned long long* hist;  // [kSelects][kPasses][B][256]
  uint8_t* tok_w;            // floor weight per token row (0 = not a floor item)
  unsigned long long* keys;  // auction sort key per op (0 = not in the auction)
  double* imp;               // head-level hybrid: relevance mass per (b,l,h) outside the window
  uint8_t* full;             // head-level hybrid: 1 = the (b,l,h) keeps every token
};

__device__ __forceinline__ int op_parent(int o) {
  if (o == 0) return -1;
  const int j = o - 1;
  return j == 0 ? 0 : 1 + (j - 1) / 2;
}

// Depth-1, depth-2 and leaf node of token i in slot [x0, y0) (tree with cut
// table `cuts`, or the midpoint tree when null); leaf = -1 for the salient
// token a three-way depth-2 node isolates (its depth-2 split makes it exact).
__device__ __forceinline__ void token_path(const uint8_t* cuts, int i, int x0, int y0, int& d1,
                                           int& d2, int& leaf) {
  int a = x0, b = y0, j = 0;
  int path[3];
#pragma unroll
  for (int lvl = 0; lvl < 2; ++lvl) {
    const int t = kvcd::tree_cut(cuts, j, lvl, x0, a, b);
    if (i < t) { j = 2 * j + 1; b = t; } else { j = 2 * j + 2; a = t; }
    path[lvl] = j;
  }
  d1 = path[0]; d2 = path[1];
  const int e = kvcd::tree_extract(cuts, d2, x0, a, b);
  if (e >= 0) {
    leaf = i == e ? -1 : (i < e ? 2 * d2 + 1 : 2 * d2 + 2);
  } else {
    leaf = i < kvcd::tree_cut(cuts, d2, 2, x0, a, b) ? 2 * d2 + 1 : 2 * d2 + 2;
  }
}

__device__ __forceinline__ void node_range(const uint8_t* cuts, int j, int x0, int y0, int& a,
                                           int& b) {
  kvcd::tree_node_range(cuts, j, x0, y0, a, b);
}

__device__ __forceinline__ unsigned long long floor_key(float r, float sens, uint32_t cidx) {
  const float k = __fmul_rn(r, sens);
  return ((unsigned long long)kvcd::float_key(k) << 32) | (unsigned long long)(0xffffffffu - cidx);
}

// ---------------------------------------------------------------- budget
__global__ void sel_init_kernel(kvc_params p, const int32_t* ctx_len, const int32_t* n_slots,
                                SelWs ws, int32_t* err) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.B) return;
  const long long n = ctx_len[b];
  const long long LH = (long long)p.L * p.H;
  const long long per_lh = p.budget_entries_per_lh > 0 ? p.budget_entries_per_lh
                                                       : (long long)floor(p.budget_ratio * (double)n);
  long long B_alloc = per_lh * LH - (long long)p.W * LH;
  if (p.head_full_frac > 0.0)                          // full heads pay n - W beyond their window
    B_alloc -= (long long)floor(p.head_full_frac * (double)LH) * (n - p.W);
  bool bad = false;
  if (B_alloc < 0) { kvcd::record_error(err, KVC_EBUDGET); bad = true; }
  if (n < p.W + 16 || n > p.n_max || n_slots[b] < 1 || n_slots[b] > p.S_max) {
    kvcd::record_error(err, KVC_EDEVICE); bad = true;
  }
  if (bad) B_alloc = 0;
  long long cap = (long long)floor(p.floor_cap_frac * (double)B_alloc);
  if (cap > B_alloc) cap = B_alloc;
  if (cap < 0) cap = 0;
  SeqBudget sb;
  sb.B_alloc = B_alloc;
  sb.cap_entries = cap;
  sb.cap_tokens = p.floor_cap_tokens;
  sb.floor_spent = 0; sb.floor_tokens = 0;
  sb.tail_rem = 0; sb.tail_last = 0; sb.tail_best = 0; sb.tail_done = bad ? 1 : 0; sb.pad = bad;
  ws.seq[b] = sb;
  for (int s = 0; s < kSelects; ++s) {
    RadixState r;
    r.prefix = 0; r.found = 0;
    r.done = bad ? 1 : 0;
    r.rem = s == 0 ? cap : (s == 1 ? (p.floor_cap_tokens < 0 ? (1LL << 62) : p.floor_cap_tokens) : 0);
    ws.rs[s * p.B + b] = r;
  }
}

__global__ void zero_u64_kernel(unsigned long long* x, long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    x[i] = 0ull;
}

__global__ void zero_u8_kernel(uint8_t* x, long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    x[i] = 0;
}

// ---------------------------------------------------------------- floor weights
// One warp per (b, l, h, slot): per-token incremental path cost of the floor
// in prefix form (0 for non-candidates and for tokens whose leaf already has a
// higher-keyed candidate).
__global__ void floor_weights_kernel(kvc_params p, const int32_t* ctx_len,
                                     const int32_t* slot_bounds, const int32_t* n_slots,
                                     const float* relevance, const float* head_sens,
                                     const int32_t* op_cost, SelWs ws, int32_t* err) {
  const int warps_per_block = blockDim.x >> 5;
  const long long tree = (long long)blockIdx.x * warps_per_block + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long trees = (long long)p.B * p.L * p.H * p.S_max;
  if (tree >= trees) return;
  const int s = (int)(tree % p.S_max);
  const long long blh = tree / p.S_max;
  const int lh = (int)(blh % ((long long)p.L * p.H));
  const int b = (int)(blh / ((long long)p.L * p.H));
  if (ws.seq[b].pad) return;
  if (s >= n_slots[b]) return;
  if (p.head_full_frac > 0.0 && ws.full[blh]) return;   // already exact: not a floor item
  const int n = ctx_len[b];
  const int x0 = slot_bounds[(long long)b * (p.S_max + 1) + s];
  const int y0 = slot_bounds[(long long)b * (p.S_max + 1) + s + 1];
  const uint8_t* cuts = kvcd::tree_cuts_of(p, blh, s);
  if (x0 < 0 || y0 - x0 < 16 || y0 - x0 > 128 || y0 > n - p.W) {
    if (lane == 0) kvcd::record_error(err, KVC_EDEVICE);
    return;
  }
  const long long row0 = kvcd::seq_token_base(ctx_len, b, p.L * p.H) + (long long)lh * n;
  const float sens = head_sens ? head_sens[lh] : 1.0f;
  const int32_t* cost = op_cost + tree * kOps;
  __shared__ unsigned long long s_key[8][128];
  __shared__ unsigned long long s_gmax[8][16];
  const int w = threadIdx.x >> 5;
  for (int t = lane; t < y0 - x0; t += 32) {
    const int i = x0 + t;
    const float r = relevance[row0 + i];
    s_key[w][t] = r > 0.f ? floor_key(r, sens, (uint32_t)((long long)lh * n + i)) : 0ull;
  }
  __syncwarp();
  if (lane < 15) {
    int a, bb;
    node_range(cuts, lane, x0, y0, a, bb);
    unsigned long long m = 0;
    for (int i = a; i < bb; ++i) m = max(m, s_key[w][i - x0]);
    s_gmax[w][lane] = m;
  }
  __syncwarp();
  for (int t = lane; t < y0 - x0; t += 32) {
    const int i = x0 + t;
    const unsigned long long k = s_key[w][t];
    int c = 0;
    if (k != 0) {
      int d1, d2, leaf;
      token_path(cuts, i, x0, y0, d1, d2, leaf);
      const int ex = leaf >= 0 ? leaf : d2;            // the split that makes token i exact
      if (k == s_gmax[w][ex]) {
        c = cost[1 + ex];
        if (leaf >= 0 && k == s_gmax[w][d2]) c += cost[1 + d2];
        if (k == s_gmax[w][d1]) c += cost[1 + d1];
        if (k == s_gmax[w][0]) c += cost[0] + cost[1];
      }
    }
    ws.tok_w[row0 + i] = (uint8_t)min(c, 255);
  }
}

// ---------------------------------------------------------------- head-level hybrid
// DistillCache App. E.3: the top fraction of heads by an attention statistic
// keep the full cache.  Statistic: relevance mass outside the recent window,
// summed in float64 (one warp per (b,l,h)).
__global__ void hybrid_importance_kernel(kvc_params p, const int32_t* ctx_len,
                                         const int32_t* slot_bounds, const int32_t* n_slots,
                                         const float* relevance, SelWs ws) {
  const long long LH = (long long)p.L * p.H;
  const long long blh = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (blh >= (long long)p.B * LH) return;
  const int b = (int)(blh / LH);
  const long long lh = blh % LH;
  const int n = ctx_len[b];
  const int ns = min(max(n_slots[b], 0), p.S_max);
  const int end = min(max(slot_bounds[(long long)b * (p.S_max + 1) + ns], 0), n);
  const long long row0 = kvcd::seq_token_base(ctx_len, b, (int)LH) + lh * n;
  double acc = 0.0;
  for (int i = lane; i < end; i += 32) acc += (double)relevance[row0 + i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(KVC_FULL_MASK, acc, o);
  if (lane == 0) ws.imp[blh] = acc;
}

// One CTA per sequence: the floor(frac * L * H) heads with the largest statistic
// (ties: lower l*H + h) are full, and every op of their trees is taken.
__global__ void hybrid_mark_kernel(kvc_params p, const int32_t* n_slots, SelWs ws,
                                   uint8_t* taken) {
  const int b = blockIdx.x;
  const long long LH = (long long)p.L * p.H;
  const long long F = (long long)floor(p.head_full_frac * (double)LH);
  const double* imp = ws.imp + (long long)b * LH;
  for (long long k = threadIdx.x; k < LH; k += blockDim.x) {
    const double v = imp[k];
    long long rank = 0;
    for (long long j = 0; j < LH; ++j) {
      const double u = imp[j];
      rank += (u > v || (u == v && j < k)) ? 1 : 0;
    }
    ws.full[(long long)b * LH + k] = rank < F ? 1 : 0;
  }
  __syncthreads();
  const int S = min(max(n_slots[b], 0), p.S_max);
  const long long per = (long long)S * kOps;
  for (long long idx = threadIdx.x; idx < LH * per; idx += blockDim.x) {
    const long long lh = idx / per, rem = idx % per;
    if (ws.full[(long long)b * LH + lh])
      taken[(((long long)b * LH + lh) * p.S_max + rem / kOps) * kOps + rem % kOps] = 1;
  }
}

// ---------------------------------------------------------------- weighted radix select
// Items of sequence b: floor -> token rows of b (key recomputed from relevance,
// weight from tok_w); auction -> ops of b (stored keys, weight = cost).
struct Items {
  int kind;                 // 0 floor entries, 1 floor tokens, 2 auction
  const int32_t* ctx_len;
  const float* relevance;
  const float* head_sens;
  const int32_t* op_cost;
};

__device__ __forceinline__ bool item_at(const kvc_params& p, const Items& it, const SelWs& ws,
                                        int b, long long k, long long row0, int n,
                                        unsigned long long& key, long long& wgt) {
  if (it.kind == 2) {
    const long long idx = (long long)b * p.L * p.H * p.S_max * kOps + k;
    key = ws.keys[idx];
    wgt = it.op_cost[idx];
    return key != 0ull;
  }
  const uint8_t c = ws.tok_w[row0 + k];
  if (c == 0) return false;
  const int lh = (int)(k / n);
  const int i = (int)(k - (long long)lh * n);
  const float sens = it.head_sens ? it.head_sens[lh] : 1.0f;
  key = floor_key(it.relevance[row0 + k], sens, (uint32_t)k);
  (void)i;
  wgt = it.kind == 0 ? (long long)c : 1;
  return true;
}

__global__ void radix_hist_kernel(kvc_params p, Items it, SelWs ws, int sel, int pass) {
  const int b = blockIdx.y;
  const RadixState st = ws.rs[sel * p.B + b];
  if (st.done) return;
  __shared__ unsigned long long sh[256];
  for (int i = threadIdx.x; i < 256; i += blockDim.x) sh[i] = 0ull;
  __syncthreads();
  const int shift = 56 - 8 * pass;
  const unsigned long long hi_mask = pass == 0 ? 0ull : (~0ull << (shift + 8));
  long long count, row0 = 0;
  int n = 0;
  if (it.kind == 2) {
    count = (long long)p.L * p.H * p.S_max * kOps;
  } else {
    n = it.ctx_len[b];
    count = (long long)p.L * p.H * n;
    row0 = kvcd::seq_token_base(it.ctx_len, b, p.L * p.H);
  }
  // warp-uniform trip count; the lanes of a warp that fall in the same bin add
  // their weights first (keys of one sequence share long prefixes, so most
  // items of a pass land in a few bins)
  const int lane = threadIdx.x & 31;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long base = (long long)blockIdx.x * blockDim.x + (threadIdx.x & ~31); base < count;
       base += stride) {
    const long long k = base + lane;
    unsigned long long key = 0ull;
    long long w = 0;
    bool ok = k < count && item_at(p, it, ws, b, k, row0, n, key, w);
    ok = ok && (key & hi_mask) == (st.prefix & hi_mask) && w > 0;
    const unsigned dig = ok ? (unsigned)((key >> shift) & 255u) : 256u;
    const unsigned peers = __match_any_sync(KVC_FULL_MASK, dig);
    const unsigned sum = __reduce_add_sync(peers, ok ? (unsigned)w : 0u);   // <= 32 x a cost
    if (ok && lane == __ffs(peers) - 1) atomicAdd(&sh[dig], (unsigned long long)sum);
  }
  __syncthreads();
  unsigned long long* gh = ws.hist + (((long long)sel * kPasses + pass) * p.B + b) * 256;
  for (int i = threadIdx.x; i < 256; i += blockDim.x)
    if (sh[i]) atomicAdd(gh + i, sh[i]);
}

// One block of 256 threads per sequence: find the digit where the cumulative
// weight (from the largest digit down) crosses the remaining budget.
__global__ void radix_pick_kernel(kvc_params p, SelWs ws, int sel, int pass) {
  const int b = blockIdx.x;
  RadixState* stp = ws.rs + sel * p.B + b;
  if (stp->done) return;
  __shared__ unsigned long long sc[256];
  __shared__ int s_digit;
  const int t = threadIdx.x;                       // position in descending digit order
  const int digit = 255 - t;
  const unsigned long long* gh = ws.hist + (((long long)sel * kPasses + pass) * p.B + b) * 256;
  const unsigned long long h = gh[digit];
  sc[t] = h;
  if (t == 0) s_digit = -1;
  __syncthreads();
  for (int o = 1; o < 256; o <<= 1) {              // inclusive scan (Hillis-Steele)
    const unsigned long long v = t >= o ? sc[t - o] : 0ull;
    __syncthreads();
    sc[t] += v;
    __syncthreads();
  }
  const unsigned long long incl = sc[t], excl = incl - h;
  const unsigned long long rem = (unsigned long long)stp->rem;
  if (h > 0 && excl <= rem && rem < incl) s_digit = digit;
  __syncthreads();
  if (t == 0) {
    const int dgt = s_digit;
    if (dgt < 0) {                                 // everything fits: no crossing item
      stp->done = 1;
      stp->found = 0;
      stp->rem = (long long)(rem - sc[255]);
    } else {
      const int shift = 56 - 8 * pass;
      const int tpos = 255 - dgt;
      const unsigned long long above = tpos > 0 ? sc[tpos - 1] : 0ull;
      stp->prefix |= ((unsigned long long)dgt) << shift;
      stp->rem = (long long)(rem - above);
      if (pass == kPasses - 1) { stp->done = 1; stp->found = 1; }
    }
  }
}

// ---------------------------------------------------------------- floor marking
__global__ void floor_mark_kernel(kvc_params p, const int32_t* ctx_len,
                                  const int32_t* slot_bounds, const int32_t* n_slots,
                                  const float* relevance, const float* head_sens, SelWs ws,
                                  uint8_t* taken) {
  const int warps_per_block = blockDim.x >> 5;
  const long long tree = (long long)blockIdx.x * warps_per_block + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long trees = (long long)p.B * p.L * p.H * p.S_max;
  if (tree >= trees) return;
  const int s = (int)(tree % p.S_max);
  const long long blh = tree / p.S_max;
  const int lh = (int)(blh % ((long long)p.L * p.H));
  const int b = (int)(blh / ((long long)p.L * p.H));
  if (ws.seq[b].pad || s >= n_slots[b]) return;
  const int n = ctx_len[b];
  const int x0 = slot_bounds[(long long)b * (p.S_max + 1) + s];
  const int y0 = slot_bounds[(long long)b * (p.S_max + 1) + s + 1];
  const uint8_t* cuts = kvcd::tree_cuts_of(p, blh, s);
  if (x0 < 0 || y0 - x0 < 16 || y0 - x0 > 128 || y0 > n - p.W) return;
  const RadixState r0 = ws.rs[0 * p.B + b];
  const RadixState r1 = ws.rs[1 * p.B + b];
  unsigned long long stop = 0;
  if (r0.found) stop = r0.prefix;
  if (r1.found && r1.prefix > stop) stop = r1.prefix;
  const long long row0 = kvcd::seq_token_base(ctx_len, b, p.L * p.H) + (long long)lh * n;
  const float sens = head_sens ? head_sens[lh] : 1.0f;
  uint8_t* tk = taken + tree * kOps;
  unsigned long long spent = 0, toks = 0;
  for (int t = lane; t < y0 - x0; t += 32) {
    const int i = x0 + t;
    const int c = ws.tok_w[row0 + i];
    if (c == 0) continue;
    const unsigned long long k = floor_key(relevance[row0 + i], sens, (uint32_t)((long long)lh * n + i));
    if (k <= stop) continue;
    int d1, d2, leaf;
    token_path(cuts, i, x0, y0, d1, d2, leaf);
    tk[0] = 1; tk[1] = 1; tk[1 + d1] = 1; tk[1 + d2] = 1;
    if (leaf >= 0) tk[1 + leaf] = 1;
    spent += (unsigned long long)c;
    toks += 1;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    spent += __shfl_xor_sync(KVC_FULL_MASK, spent, o);
    toks += __shfl_xor_sync(KVC_FULL_MASK, toks, o);
  }
  if (lane == 0 && toks) {
    atomicAdd(&ws.seq[b].floor_spent, spent);
    atomicAdd(&ws.seq[b].floor_tokens, toks);
  }
}

// ---------------------------------------------------------------- auction keys
// Effective key and block rank of every untaken op of one tree.  Returns the
// sort keys in sk[16] (0 for taken ops).
__device__ void tree_sort_keys(const float* util, const uint8_t* tk, long long tree,
                               unsigned long long sk[kOps]) {
  unsigned long long key[kOps], e[kOps];
#pragma unroll
  for (int o = 0; o < kOps; ++o)
    key[o] = ((unsigned long long)kvcd::float_key(util[o]) << 32) |
             (unsigned long long)(0xffffffffu - (uint32_t)(tree * kOps + o));
  for (int o = 0; o < kOps; ++o) {           // parents precede children
    if (tk[o]) { e[o] = 0; continue; }
    const int par = op_parent(o);
    e[o] = (par < 0 || tk[par]) ? key[o] : min(key[o], e[par]);
  }
  int rank[kOps];
  for (int o = 0; o < kOps; ++o) rank[o] = -1;
  for (int a = 0; a < kOps; ++a) {
    if (tk[a] || e[a] != key[a]) continue;   // not a block head
    uint32_t pool = 1u << a;
    int r = 0;
    while (pool) {
      int best = -1;
      for (int o = 0; o < kOps; ++o)
        if ((pool >> o) & 1u) if (best < 0 || key[o] > key[best]) best = o;
      pool &= ~(1u << best);
      rank[best] = r++;
      // children ops of `best` that belong to the same block
      int c0 = -1, c1 = -1;
      if (best == 0) c0 = 1;
      else if (best - 1 < 7) { c0 = 1 + 2 * (best - 1) + 1; c1 = c0 + 1; }
      if (c0 >= 0 && !tk[c0] && e[c0] == e[a]) pool |= 1u << c0;
      if (c1 >= 0 && !tk[c1] && e[c1] == e[a]) pool |= 1u << c1;
    }
    // encode: (e utility bits, head tree*256 + head*16 + rank)
  }
  for (int o = 0; o < kOps; ++o) {
    if (tk[o]) { sk[o] = 0; continue; }
    const uint32_t head_gid = 0xffffffffu - (uint32_t)(e[o] & 0xffffffffull);  // tree*16 + head
    const uint32_t low = 0xffffffffu - (head_gid * 16u + (uint32_t)rank[o]);
    sk[o] = (e[o] & 0xffffffff00000000ull) | (unsigned long long)low;
  }
}

__global__ void auction_keys_kernel(kvc_params p, const int32_t* n_slots, const float* op_util,
                                    const uint8_t* taken, SelWs ws) {
  const long long trees = (long long)p.B * p.L * p.H * p.S_max;
  const long long tree = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (tree >= trees) return;
  const int s = (int)(tree % p.S_max);
  const int b = (int)(tree / ((long long)p.L * p.H * p.S_max));
  unsigned long long* out = ws.keys + tree * kOps;
  if (ws.seq[b].pad || s >= n_slots[b]) {
#pragma unroll
    for (int o = 0; o < kOps; ++o) out[o] = 0ull;
    return;
  }
  const long long tree_in_seq = tree - (long long)b * p.L * p.H * p.S_max;
  unsigned long long sk[kOps];
  tree_sort_keys(op_util + tree * kOps, taken + tree * kOps, tree_in_seq, sk);
#pragma unroll
  for (int o = 0; o < kOps; ++o) out[o] = sk[o];
}

// After the floor: the auction budget is B_alloc - floor spent.
__global__ void auction_budget_kernel(kvc_params p, SelWs ws) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.B) return;
  RadixState* r = ws.rs + 2 * p.B + b;
  const SeqBudget sb = ws.seq[b];
  r->rem = sb.B_alloc - (long long)sb.floor_spent;
  if (r->rem < 0) r->rem = 0;
}

__global__ void auction_mark_kernel(kvc_params p, SelWs ws, uint8_t* taken) {
  const long long total = (long long)p.B * p.L * p.H * p.S_max * kOps;
  const long long per_seq = (long long)p.L * p.H * p.S_max * kOps;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const unsigned long long k = ws.keys[i];
    if (k == 0ull) continue;
    const int b = (int)(i / per_seq);
    const RadixState r = ws.rs[2 * p.B + b];
    if (!r.found || k > r.prefix) taken[i] = 1;
  }
}

__global__ void tail_setup_kernel(kvc_params p, SelWs ws) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.B) return;
  const RadixState r = ws.rs[2 * p.B + b];
  SeqBudget* sb = ws.seq + b;
  sb->tail_rem = r.rem;
  sb->tail_last = r.prefix;
  sb->tail_best = 0;
  if (!r.found || r.rem <= 0) sb->tail_done = 1;
}

__global__ void tail_find_kernel(kvc_params p, SelWs ws, const int32_t* op_cost,
                                 const uint8_t* taken) {
  const long long total = (long long)p.B * p.L * p.H * p.S_max * kOps;
  const long long per_seq = (long long)p.L * p.H * p.S_max * kOps;
  // warp-uniform trip count; a warp's candidates of one sequence are reduced
  // to their maximum with shuffles before the one atomic.  A sequence owns a
  // multiple of 16 ops and warps start at multiples of 32, so a warp holds at
  // most two sequences split at lane 16: the xor-16 step is the only one that
  // crosses them (skipped then) and lanes 0 and 16 end with their half's max.
  const int lane = threadIdx.x & 31;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long base = (long long)blockIdx.x * blockDim.x + (threadIdx.x & ~31); base < total;
       base += stride) {
    const long long i = base + lane;
    unsigned long long cand = 0ull;
    int b = -1;
    if (i < total) {
      const unsigned long long k = ws.keys[i];
      b = (int)(i / per_seq);
      const SeqBudget& sb = ws.seq[b];
      bool ok = k != 0ull && !taken[i] && !sb.tail_done && k <= sb.tail_last &&
                op_cost[i] <= sb.tail_rem;
      const int o = (int)(i & (kOps - 1));
      const int par = op_parent(o);
      if (ok && par >= 0 && !taken[i - o + par]) ok = false;
      cand = ok ? k : 0ull;
    }
    const unsigned same = __match_any_sync(KVC_FULL_MASK, b);   // lanes of one sequence
    unsigned long long m = cand;
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long v = __shfl_xor_sync(KVC_FULL_MASK, m, o);
      const int bv = __shfl_xor_sync(KVC_FULL_MASK, b, o);
      if (bv == b && v > m) m = v;
    }
    if (b >= 0 && m != 0ull && lane == __ffs(same) - 1) atomicMax(&ws.seq[b].tail_best, m);
  }
}

__global__ void tail_take_kernel(kvc_params p, SelWs ws, const int32_t* op_cost, uint8_t* taken) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.B) return;
  SeqBudget* sb = ws.seq + b;
  if (sb->tail_done) return;
  const unsigned long long best = sb->tail_best;
  if (best == 0ull) { sb->tail_done = 1; return; }
  const uint32_t code = 0xffffffffu - (uint32_t)(best & 0xffffffffull);   // tree*256 + head*16 + rank
  const long long tree_in_seq = code >> 8;
  const long long tree = (long long)b * p.L * p.H * p.S_max + tree_in_seq;
  int op = -1;
  for (int o = 0; o < kOps; ++o) if (ws.keys[tree * kOps + o] == best) op = o;
  if (op < 0) { sb->tail_done = 1; return; }
  taken[tree * kOps + op] = 1;
  sb->tail_rem -= op_cost[tree * kOps + op];
  sb->tail_last = best - 1;
  sb->tail_best = 0;
  if (sb->tail_rem <= 0) sb->tail_done = 1;
}

// ---------------------------------------------------------------- lengths and offsets
__global__ void lens_kernel(kvc_params p, const int32_t* n_slots, const int32_t* op_cost,
                            const uint8_t* taken, int32_t* len_lh, int32_t* cap_lh) {
  const int warps_per_block = blockDim.x >> 5;
  const long long blh = (long long)blockIdx.x * warps_per_block + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (blh >= (long long)p.B * p.L * p.H) return;
  const int b = (int)(blh / ((long long)p.L * p.H));
  const int S = min(n_slots[b], p.S_max);
  long long sum = 0;
  const long long base = blh * p.S_max * kOps;
  for (int k = lane; k < S * kOps; k += 32) sum += taken[base + k] ? op_cost[base + k] : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(KVC_FULL_MASK, sum, o);
  if (lane == 0) {
    len_lh[blh] = (int32_t)(p.W + sum);
    cap_lh[blh] = (int32_t)(p.W + sum + p.decode_reserve);
  }
}

__global__ void offsets_kernel(long long n, const int32_t* cap_lh, int64_t* off_lh,
                               int64_t* total) {
  __shared__ long long s_part[1024];
  const int t = threadIdx.x;
  const long long per = (n + blockDim.x - 1) / blockDim.x;
  const long long lo = t * per, hi = min(n, lo + per);
  long long acc = 0;
  for (long long i = lo; i < hi; ++i) acc += cap_lh[i];
  s_part[t] = acc;
  __syncthreads();
  for (int o = 1; o < (int)blockDim.x; o <<= 1) {
    const long long v = t >= o ? s_part[t - o] : 0;
    __syncthreads();
    s_part[t] += v;
    __syncthreads();
  }
  long long run = s_part[t] - acc;
  for (long long i = lo; i < hi; ++i) { off_lh[i] = run; run += cap_lh[i]; }
  if (t == (int)blockDim.x - 1) *total = s_part[t];
}

struct Layout {
  size_t seq, rs, hist, tok_w, keys, imp, full, total;
};

Layout layout(const kvc_params* p) {
  Layout l;
  size_t off = 0;
  l.seq = off; off += kvc::align256(sizeof(SeqBudget) * p->B);
  l.rs = off; off += kvc::align256(sizeof(RadixState) * kSelects * p->B);
  l.hist = off; off += kvc::align256(sizeof(unsigned long long) * kSelects * kPasses * p->B * 256);
  l.tok_w = off; off += kvc::align256((size_t)p->B * p->L * p->H * p->n_max);
  l.keys = off; off += kvc::align256(sizeof(unsigned long long) * (size_t)p->B * p->L * p->H *
                                     p->S_max * kOps);
  l.imp = off; off += kvc::align256(sizeof(double) * (size_t)p->B * p->L * p->H);
  l.full = off; off += kvc::align256((size_t)p->B * p->L * p->H);
  l.total = off;
  return l;
}

}  // namespace

namespace kvc {
size_t select_workspace_bytes(const kvc_params* p) { return layout(p).total; }
}  // namespace kvc

extern "C" int kvc_select(const kvc_params* p, const int32_t* ctx_len, const int32_t* slot_bounds,
                          const int32_t* n_slots, const float* relevance, const float* head_sens,
                          const float* op_util, const int32_t* op_cost, uint8_t* taken,
                          int32_t* len_lh, int32_t* cap_lh, int64_t* off_lh,
                          int64_t* total_entries, void* workspace, size_t ws_bytes,
                          void* stream) {
  int st = kvc::check_params(p);
  if (st != KVC_OK) return st;
  if (!ctx_len || !slot_bounds || !n_slots || !relevance || !op_util || !op_cost || !taken ||
      !len_lh || !cap_lh || !off_lh || !total_entries)
    return KVC_EINVAL;
  if (p->budget_entries_per_lh > 0 && p->budget_entries_per_lh < p->W) return KVC_EBUDGET;
  const Layout lay = layout(p);
  if (!workspace || ws_bytes < lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return KVC_EWORKSPACE;
  if ((long long)p->L * p->H * p->S_max >= (1LL << 24)) return KVC_EINVAL;
  if ((long long)p->L * p->H * p->n_max >= (1LL << 32)) return KVC_EINVAL;
  int32_t* err = kvc::err_word();
  if (!err) return KVC_ECUDA;
  char* w = static_cast<char*>(workspace);
  SelWs ws;
  ws.seq = reinterpret_cast<SeqBudget*>(w + lay.seq);
  ws.rs = reinterpret_cast<RadixState*>(w + lay.rs);
  ws.hist = reinterpret_cast<unsigned long long*>(w + lay.hist);
  ws.tok_w = reinterpret_cast<uint8_t*>(w + lay.tok_w);
  ws.keys = reinterpret_cast<unsigned long long*>(w + lay.keys);
  ws.imp = reinterpret_cast<double*>(w + lay.imp);
  ws.full = reinterpret_cast<uint8_t*>(w + lay.full);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const kvc_params P = *p;
  const long long trees = (long long)p->B * p->L * p->H * p->S_max;
  const long long ops = trees * kOps;
  const int sms = std::max(1, kvc::sm_count());
  int launches = 0;

  sel_init_kernel<<<(p->B + 63) / 64, 64, 0, s>>>(P, ctx_len, n_slots, ws, err); ++launches;
  zero_u64_kernel<<<64, 256, 0, s>>>(ws.hist, (long long)kSelects * kPasses * p->B * 256);
  ++launches;
  zero_u8_kernel<<<sms * 4, 256, 0, s>>>(taken, ops); ++launches;
  zero_u8_kernel<<<sms * 4, 256, 0, s>>>(ws.tok_w, (long long)p->B * p->L * p->H * p->n_max);
  ++launches;
  if (p->head_full_frac > 0.0) {                       // head-level hybrid: full heads first
    hybrid_importance_kernel<<<(unsigned)((kvc::lh_count(p) + 7) / 8), 256, 0, s>>>(
        P, ctx_len, slot_bounds, n_slots, relevance, ws);
    hybrid_mark_kernel<<<p->B, 256, 0, s>>>(P, n_slots, ws, taken);
    launches += 2;
  }
  floor_weights_kernel<<<(unsigned)((trees + 7) / 8), 256, 0, s>>>(
      P, ctx_len, slot_bounds, n_slots, relevance, head_sens, op_cost, ws, err);
  ++launches;
  Items it{0, ctx_len, relevance, head_sens, op_cost};
  const int fsel = p->floor_cap_tokens >= 0 ? 2 : 1;
  for (int sel = 0; sel < fsel; ++sel) {
    it.kind = sel;
    for (int pass = 0; pass < kPasses; ++pass) {
      radix_hist_kernel<<<dim3(sms * 2 / std::max(1, p->B) + 1, p->B), 512, 0, s>>>(P, it, ws, sel,
                                                                                     pass);
      radix_pick_kernel<<<p->B, 256, 0, s>>>(P, ws, sel, pass);
      launches += 2;
    }
  }
  floor_mark_kernel<<<(unsigned)((trees + 7) / 8), 256, 0, s>>>(P, ctx_len, slot_bounds, n_slots,
                                                               relevance, head_sens, ws, taken);
  ++launches;
  auction_keys_kernel<<<(unsigned)((trees + 127) / 128), 128, 0, s>>>(P, n_slots, op_util, taken,
                                                                      ws);
  auction_budget_kernel<<<(p->B + 63) / 64, 64, 0, s>>>(P, ws);
  launches += 2;
  it.kind = 2;
  for (int pass = 0; pass < kPasses; ++pass) {
    radix_hist_kernel<<<dim3(sms * 2 / std::max(1, p->B) + 1, p->B), 512, 0, s>>>(P, it, ws, 2,
                                                                                   pass);
    radix_pick_kernel<<<p->B, 256, 0, s>>>(P, ws, 2, pass);
    launches += 2;
  }
  auction_mark_kernel<<<sms * 4, 256, 0, s>>>(P, ws, taken);
  tail_setup_kernel<<<(p->B + 63) / 64, 64, 0, s>>>(P, ws);
  launches += 2;
  for (int i = 0; i < kTailIters; ++i) {
    tail_find_kernel<<<sms * 4, 256, 0, s>>>(P, ws, op_cost, taken);
    tail_take_kernel<<<(p->B + 63) / 64, 64, 0, s>>>(P, ws, op_cost, taken);
    launches += 2;
  }
  lens_kernel<<<(unsigned)((kvc::lh_count(p) + 7) / 8), 256, 0, s>>>(P, n_slots, op_cost, taken,
                                                                     len_lh, cap_lh);
  offsets_kernel<<<1, 1024, 0, s>>>(kvc::lh_count(p), cap_lh, off_lh, total_entries);
  launches += 2;
  kvc::count_launch(launches);
  return kvc::cuda_status(cudaGetLastError());
}
