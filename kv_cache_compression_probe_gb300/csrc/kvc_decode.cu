// a7: ragged GQA decode attention with the +ln m multiplicity bias and the
// multiplicity-one append of the new token (GraceKV "05 Physical cache
// packing": new tokens are appended with multiplicity one; the decoder attends
// over each (layer, head)'s independently sized cache).
//
// Design (HBM-bound): one launch covers every (sequence, layer, KV head).  The
// entries of an (l,h) are split into chunks of kChunk rows; one 128-thread CTA
// streams a chunk through a kStages-deep shared-memory ring filled by 1-D bulk
// asynchronous copies (K and V rows of an (l,h) are contiguous, so a stage is
// two copies completing on one mbarrier).  Each lane owns d/32 consecutive
// features of every K/V row read from shared memory,
// the G query heads' partial dot products of 32/G rows are reduced with one
// 31-shuffle transpose, and the softmax runs online in base 2.  Chunk partials
// (max, sum, unnormalised output) go to the workspace; the last CTA of an
// (l,h) to arrive (atomic counter, no waiting) merges them in log-sum-exp form.
// A second tiny kernel commits the append (len += 1) after every chunk has read
// the old length.
#include <math.h>

#include <mutex>

#include "kvc_common.cuh"
#include "kvc_decode_tc.h"
#include "kvc_internal.h"

namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 512;       // rows per CTA (split-K chunk)
constexpr int kStage = 32;        // rows per bulk-copy stage
constexpr int kStages = 3;        // stages in the shared-memory ring
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeArgs {
  const void* q;
  const void* k_new;
  const void* v_new;
  const float* pos_new;
  void* Kp;
  void* Vp;
  float* logm;
  float* pos;
  const int32_t* len_lh;
  const int32_t* cap_lh;
  const int64_t* off_lh;
  void* out;
  float* partials;     // [BLH, n_chunk_max, G, D + 2]
  int32_t* counters;   // [BLH], zero between calls
  float* lse_out;      // [BLH, G] base-2 LSE of the step's scores, or null
  float* scores_out;   // [rows, G] base-2 score of cache row off + i per query head, or null
  int64_t lh_span, lh_gap, lh_base;   // layer range (see kvc::lh_global)
  int H, L, n_chunk_max;
  float scale_log2;    // log2(e) / sqrt(d)
  int32_t* err;
  uint64_t wait_ns;    // first-wait limit and copy withholding (kvc_set_wait_limit)
  int withhold;
};

template <typename T, int D, int G>
struct DecodeSmem {
  T ring[kStages][2][kStage][D];   // K rows, V rows of each stage
  float p[kWarps][32];
  float m[kWarps][G], l[kWarps][G];
  float o[kWarps][G][D];
  uint64_t full[kStages];
  int last;
  int abort;
};

// One warp batch: rows k < nvalid (of EB = 32/G) at kb + k*D / vb + k*D, the
// rest masked; 32 dot products, one transpose reduction, online softmax
// update.  my_lm = log2(e) * log m of row lane / G (0 when masked).  With
// s_out the batch's scores are stored there ([row][G], lane = row * G + g).
template <typename T, int D, int G>
__device__ __forceinline__ void decode_batch(const float (&qv)[G][D / 32], const T* kb,
                                             const T* vb, int nvalid, float my_lm, int lane,
                                             float* s_p, float (&m_run)[G], float& lsum,
                                             float (&o)[G][D / 32], float* s_out) {
  constexpr int VPL = D / 32;
  constexpr int EB = 32 / G;
  float kk[EB][VPL], vv[EB][VPL];
#pragma unroll
  for (int k = 0; k < EB; ++k) {
    if (k < nvalid) {                       // kb / vb: shared memory, or the new token in global
      kvcd::VecLoadAny<T, VPL>::ld(kb + k * D + lane * VPL, kk[k]);
      kvcd::VecLoadAny<T, VPL>::ld(vb + k * D + lane * VPL, vv[k]);
    } else {
#pragma unroll
      for (int t = 0; t < VPL; ++t) kk[k][t] = vv[k][t] = 0.f;
    }
  }
  float part[32];
#pragma unroll
  for (int k = 0; k < EB; ++k)
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float acc = 0.f;
#pragma unroll
      for (int t = 0; t < VPL; ++t) acc = fmaf(qv[g][t], kk[k][t], acc);
      part[k * G + g] = acc;
    }
#pragma unroll
  for (int o_ = 16, n = 32; o_ >= 1; o_ >>= 1, n >>= 1) {
    const bool upper = (lane & o_) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? part[i] : part[i + n / 2];
      const float keep = upper ? part[i + n / 2] : part[i];
      part[i] = keep + __shfl_xor_sync(KVC_FULL_MASK, send, o_);
    }
  }
  const int gj = lane % G, kj = lane / G;
  const float s = kj < nvalid ? part[0] + my_lm : -INFINITY;
  if (s_out && kj < nvalid) s_out[lane] = s;
  float gm = s;
#pragma unroll
  for (int o_ = G; o_ < 32; o_ <<= 1) gm = fmaxf(gm, __shfl_xor_sync(KVC_FULL_MASK, gm, o_));
  float alpha[G];
  float my_m = -INFINITY, my_alpha = 1.f;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float mb = __shfl_sync(KVC_FULL_MASK, gm, g);
    const float mn = fmaxf(m_run[g], mb);
    alpha[g] = (mn == -INFINITY) ? 1.f : exp2f(m_run[g] - mn);
    m_run[g] = mn;
    if (g == gj) { my_m = mn; my_alpha = alpha[g]; }
  }
  const float pr = (s == -INFINITY) ? 0.f : exp2f(s - my_m);
  lsum = lsum * my_alpha + pr;
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int t = 0; t < VPL; ++t) o[g][t] *= alpha[g];
  s_p[lane] = pr;
  __syncwarp();
#pragma unroll
  for (int k = 0; k < EB; ++k)
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float pk = s_p[k * G + g];
#pragma unroll
      for (int t = 0; t < VPL; ++t) o[g][t] = fmaf(pk, vv[k][t], o[g][t]);
    }
  __syncwarp();
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kThreads) decode_chunk_kernel(DecodeArgs a) {
  constexpr int VPL = D / 32;
  constexpr int EB = 32 / G;
  constexpr int RPW = kStage / kWarps;                   // rows of a stage per warp
  extern __shared__ __align__(128) unsigned char dsm_raw[];
  DecodeSmem<T, D, G>& sm = *reinterpret_cast<DecodeSmem<T, D, G>*>(dsm_raw);
  const int blh = blockIdx.y;
  const int c = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t gblh = kvc::lh_global(blh, a.lh_span, a.lh_gap, a.lh_base);
  const int len = a.len_lh[gblh];
  const int E = len + 1;                                 // stored rows + the new token
  const int nchunks = (E + kChunk - 1) / kChunk;
  if (len < 0 || nchunks > a.n_chunk_max) {              // corrupt length: skip this (l,h)
    if (c == 0 && tid == 0) kvcd::record_error(a.err, KVC_EDEVICE);
    return;
  }
  if (c >= nchunks) return;
  const int e0 = c * kChunk, e1 = min(e0 + kChunk, E);
  const int stored_end = min(e1, len);                   // rows [e0, stored_end) come from the cache
  const int nst = stored_end > e0 ? (stored_end - e0 + kStage - 1) / kStage : 0;
  const int64_t off = a.off_lh[gblh];
  const bool append_ok = (len + 1 <= a.cap_lh[gblh]);
  const int h = blh % a.H;
  const int64_t bl = blh / a.H;                          // b * L + l

  const T* Kp = static_cast<const T*>(a.Kp) + off * D;
  const T* Vp = static_cast<const T*>(a.Vp) + off * D;
  const float* lm = a.logm + off;
  const T* kn = static_cast<const T*>(a.k_new) + (int64_t)blh * D;
  const T* vn = static_cast<const T*>(a.v_new) + (int64_t)blh * D;
  const T* qp = static_cast<const T*>(a.q) + (bl * a.H * G + (int64_t)h * G) * D;

  auto issue = [&](int st) {                             // one thread: stage st -> slot st % kStages
    if (a.withhold) return;                              // test of the timeout path: no copies
    const int slot = st % kStages;
    const int r0 = e0 + st * kStage;
    const int rows = min(kStage, stored_end - r0);
    const uint32_t bytes = (uint32_t)(rows * D * sizeof(T));
    kvcd::mbar_arrive_expect_tx(&sm.full[slot], 2 * bytes);
    kvcd::bulk_g2s(&sm.ring[slot][0][0][0], Kp + (int64_t)r0 * D, bytes, &sm.full[slot]);
    kvcd::bulk_g2s(&sm.ring[slot][1][0][0], Vp + (int64_t)r0 * D, bytes, &sm.full[slot]);
  };
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) kvcd::mbar_init(&sm.full[i], 1);
    kvcd::fence_mbar_init();
    sm.abort = 0;
    for (int st = 0; st < min(kStages, nst); ++st) issue(st);
  }

  float qv[G][VPL];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    kvcd::VecLoad<T, VPL>::ld(qp + g * D + lane * VPL, qv[g]);
#pragma unroll
    for (int t = 0; t < VPL; ++t) qv[g][t] *= a.scale_log2;
  }
  float m_run[G], o[G][VPL];
  float lsum = 0.f;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m_run[g] = -INFINITY;
#pragma unroll
    for (int t = 0; t < VPL; ++t) o[g][t] = 0.f;
  }
  __syncthreads();

  int consumed = 0;
  for (int st = 0; st < nst; ++st) {
    const int slot = st % kStages;
    if (!kvcd::mbar_wait(&sm.full[slot], (uint32_t)((st / kStages) & 1), a.wait_ns)) sm.abort = 1;
    const int r0 = e0 + st * kStage;
    const int rows = min(kStage, stored_end - r0);
    for (int rb = warp * RPW; rb < warp * RPW + RPW; rb += EB) {
      const int nvalid = min(min(EB, rows - rb), warp * RPW + RPW - rb);
      const int my_row = rb + lane / G;
      const float my_lm = (lane / G < nvalid) ? __ldg(lm + r0 + my_row) * kLog2e : 0.f;
      decode_batch<T, D, G>(qv, &sm.ring[slot][0][rb][0], &sm.ring[slot][1][rb][0], nvalid, my_lm,
                            lane, sm.p[warp], m_run, lsum, o,
                            a.scores_out ? a.scores_out + (off + r0 + rb) * G : nullptr);
    }
    consumed = st + 1;
    __syncthreads();
    if (sm.abort) break;
    if (tid == 0 && st + kStages < nst) {
      kvcd::fence_proxy_async_smem();
      issue(st + kStages);
    }
  }
  if (sm.abort) {                                        // a bounded wait gave up
    if (tid == 0) {
      kvcd::record_error(a.err, KVC_ETIMEOUT);
      // copies still in flight: the stage whose wait failed and those issued after it
      const int first = max(0, consumed - 1);
      for (int st = first; st < min(nst, first + kStages) && !a.withhold; ++st)
        kvcd::mbar_wait(&sm.full[st % kStages], (uint32_t)((st / kStages) & 1));
    }
    return;
  }
  // the new token (row len) when this chunk holds it
  if (warp == 0 && e0 <= len && len < e1) {
    decode_batch<T, D, G>(qv, kn, vn, 1, 0.f, lane, sm.p[0], m_run, lsum, o,
                          a.scores_out && append_ok ? a.scores_out + (off + len) * G : nullptr);
  }
  // per-head row sums of this warp
#pragma unroll
  for (int o_ = G; o_ < 32; o_ <<= 1) lsum += __shfl_xor_sync(KVC_FULL_MASK, lsum, o_);
  if (lane < G) {
    sm.l[warp][lane] = lsum;
#pragma unroll
    for (int g = 0; g < G; ++g)
      if (g == lane) sm.m[warp][lane] = m_run[g];
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int t = 0; t < VPL; ++t) sm.o[warp][g][lane * VPL + t] = o[g][t];

  // the chunk holding row `len` stores the appended token
  if (append_ok && e0 <= len && len < e1) {
    T* Kw = static_cast<T*>(a.Kp) + (off + len) * D;
    T* Vw = static_cast<T*>(a.Vp) + (off + len) * D;
    for (int i = tid; i < D; i += kThreads) { Kw[i] = kn[i]; Vw[i] = vn[i]; }
    if (tid == 0) {
      a.logm[off + len] = 0.f;
      a.pos[off + len] = a.pos_new ? a.pos_new[bl / a.L] : -1.f;
    }
  }
  __syncthreads();

  // merge the warps into this chunk's partial
  float* part_out = a.partials + ((int64_t)blh * a.n_chunk_max + c) * G * (D + 2);
  for (int idx = tid; idx < G * D; idx += kThreads) {
    const int g = idx / D, dd = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.m[w][g]);
    float acc = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = (sm.m[w][g] == -INFINITY) ? 0.f : exp2f(sm.m[w][g] - M);
      acc = fmaf(f, sm.o[w][g][dd], acc);
      l = fmaf(f, sm.l[w][g], l);
    }
    part_out[g * (D + 2) + 2 + dd] = acc;
    if (dd == 0) { part_out[g * (D + 2)] = M; part_out[g * (D + 2) + 1] = l; }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) sm.last = (atomicAdd(a.counters + blh, 1) == nchunks - 1);
  __syncthreads();
  if (!sm.last) return;
  __threadfence();

  // last chunk to arrive: log-sum-exp merge of all chunk partials
  const float* pb = a.partials + (int64_t)blh * a.n_chunk_max * G * (D + 2);
  T* outp = static_cast<T*>(a.out) + (bl * a.H * G + (int64_t)h * G) * D;
  for (int idx = tid; idx < G * D; idx += kThreads) {
    const int g = idx / D, dd = idx % D;
    float M = -INFINITY;
    for (int cc = 0; cc < nchunks; ++cc) M = fmaxf(M, __ldcg(pb + (cc * G + g) * (D + 2)));
    float acc = 0.f, l = 0.f;
    for (int cc = 0; cc < nchunks; ++cc) {
      const float* pc = pb + (cc * G + g) * (D + 2);
      const float mc = __ldcg(pc);
      const float f = (mc == -INFINITY) ? 0.f : exp2f(mc - M);
      acc = fmaf(f, __ldcg(pc + 2 + dd), acc);
      l = fmaf(f, __ldcg(pc + 1), l);
    }
    outp[g * D + dd] = kvcd::from_f<T>(acc / l);
    if (a.lse_out && dd == 0) a.lse_out[(int64_t)blh * G + g] = M + log2f(l);
  }
  if (tid == 0) a.counters[blh] = 0;
}

// Commits the append once every chunk has read the old length.
__global__ void decode_commit_kernel(int32_t* len_lh, const int32_t* cap_lh, int64_t n,
                                     int n_chunk_max, int64_t span, int64_t gap, int64_t base,
                                     int32_t* err) {
  const int64_t li = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (li >= n) return;
  const int64_t i = kvc::lh_global(li, span, gap, base);
  const int len = len_lh[i];
  if (len < 0 || (len + kChunk) / kChunk > n_chunk_max) return;   // skipped by the attention
  if (len + 1 <= cap_lh[i]) len_lh[i] = len + 1;
  else kvcd::record_error(err, KVC_ECAPACITY);
}

inline int n_chunk_max(const kvc_params* p) {
  const int64_t rows = (int64_t)p->n_max + p->decode_reserve + 1;
  return (int)((rows + kChunk - 1) / kChunk);
}

template <typename T, int D, int G>
void launch_one(const DecodeArgs& a, dim3 grid, cudaStream_t s) {
  const size_t smem = sizeof(DecodeSmem<T, D, G>);
  cudaFuncSetAttribute(decode_chunk_kernel<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)smem);
  decode_chunk_kernel<T, D, G><<<grid, kThreads, smem, s>>>(a);
}

template <typename T, int D>
void launch_dg(const kvc_params* p, const DecodeArgs& a, dim3 grid, cudaStream_t s) {
  switch (p->G) {
    case 1: launch_one<T, D, 1>(a, grid, s); break;
    case 2: launch_one<T, D, 2>(a, grid, s); break;
    case 4: launch_one<T, D, 4>(a, grid, s); break;
    default: launch_one<T, D, 8>(a, grid, s); break;
  }
}

// Workspace: split-K partials, per-(b,l,h) arrival counters, and the
// tensor-core path's work list and its length.
struct DecodeLayout {
  size_t partials, counters, items, n_items, total;
};
DecodeLayout decode_layout(const kvc_params* p) {
  const int64_t blh = kvc::lh_count(p);
  DecodeLayout w;
  w.partials = 0;
  w.counters = kvc::align256((size_t)blh * n_chunk_max(p) * p->G * (p->d + 2) * sizeof(float));
  w.items = w.counters + kvc::align256((size_t)blh * sizeof(int32_t));
  w.n_items = w.items + kvc::align256((size_t)blh * n_chunk_max(p) * sizeof(uint32_t));
  w.total = w.n_items + 256;
  return w;
}

// Both entry points: validated arguments, workspace `ws` laid out as above.
int run_decode(const kvc_params* p, const void* q, const void* k_new, const void* v_new,
               const float* pos_new, void* Kp, void* Vp, float* logm, float* pos,
               int32_t* len_lh, const int32_t* cap_lh, const int64_t* off_lh, void* out,
               float* lse_out, float* scores_out, char* ws, int32_t* err, cudaStream_t s,
               int64_t lh_span = 0, int64_t lh_gap = 0, int64_t lh_base = 0,
               const kvc_params* layout_p = nullptr) {
  if (lh_span <= 0) lh_span = (int64_t)p->L * p->H;         // all layers: identity map
  const int64_t blh = kvc::lh_count(p);
  // the workspace layout always follows the full parameter block, so calls on
  // layer ranges and on all layers share the same arrival-counter words
  const DecodeLayout w = decode_layout(layout_p ? layout_p : p);
  const int ncm = n_chunk_max(p);
  if (kvc::decode_tc_supported(p, ncm)) {
    kvc::DecodeTcArgs t;
    t.q = q; t.k_new = k_new; t.v_new = v_new; t.pos_new = pos_new;
    t.Kp = Kp; t.Vp = Vp; t.logm = logm; t.pos = pos;
    t.len_lh = len_lh; t.cap_lh = cap_lh; t.off_lh = off_lh; t.out = out;
    t.partials = reinterpret_cast<float*>(ws + w.partials);
    t.counters = reinterpret_cast<int32_t*>(ws + w.counters);
    t.items = reinterpret_cast<uint32_t*>(ws + w.items);
    t.n_items = reinterpret_cast<int32_t*>(ws + w.n_items);
    t.packed_rows = p->packed_rows;
    t.blh = blh;
    t.H = p->H; t.L = p->L; t.G = p->G; t.n_chunk_max = ncm;
    t.scale_log2 = kLog2e / sqrtf((float)p->d);
    t.err = err;
    t.lse_out = lse_out;
    t.scores_out = scores_out;
    t.lh_span = lh_span; t.lh_gap = lh_gap; t.lh_base = lh_base;
    t.wait_ns = kvc::wait_limit_ns(); t.withhold = kvc::withhold_copies();
    return kvc::decode_tc_launch(t, s);
  }
  DecodeArgs a;
  a.q = q; a.k_new = k_new; a.v_new = v_new; a.pos_new = pos_new;
  a.Kp = Kp; a.Vp = Vp; a.logm = logm; a.pos = pos;
  a.len_lh = len_lh; a.cap_lh = cap_lh; a.off_lh = off_lh; a.out = out;
  a.partials = reinterpret_cast<float*>(ws + w.partials);
  a.counters = reinterpret_cast<int32_t*>(ws + w.counters);
  a.H = p->H; a.L = p->L; a.n_chunk_max = ncm;
  a.scale_log2 = kLog2e / sqrtf((float)p->d);
  a.err = err;
  a.lse_out = lse_out;
  a.scores_out = scores_out;
  a.lh_span = lh_span; a.lh_gap = lh_gap; a.lh_base = lh_base;
  a.wait_ns = kvc::wait_limit_ns(); a.withhold = kvc::withhold_copies();
  dim3 grid(a.n_chunk_max, (unsigned)blh);
  if (p->dtype == KVC_BF16) {
    if (p->d == 128) launch_dg<__nv_bfloat16, 128>(p, a, grid, s);
    else launch_dg<__nv_bfloat16, 64>(p, a, grid, s);
  } else {
    if (p->d == 128) launch_dg<float, 128>(p, a, grid, s);
    else launch_dg<float, 64>(p, a, grid, s);
  }
  decode_commit_kernel<<<(unsigned)((blh + 255) / 256), 256, 0, s>>>(
      len_lh, cap_lh, blh, a.n_chunk_max, lh_span, lh_gap, lh_base, err);
  kvc::count_launch(2);
  return kvc::cuda_status(cudaGetLastError());
}

}  // namespace

namespace kvc {
size_t decode_workspace_bytes(const kvc_params* p) { return decode_layout(p).total; }
}  // namespace kvc

extern "C" int kvc_decode_attn(const kvc_params* p, const void* q, const void* k_new,
                               const void* v_new, const float* pos_new, void* Kp, void* Vp,
                               float* logm, float* pos, int32_t* len_lh, const int32_t* cap_lh,
                               const int64_t* off_lh, void* out, void* workspace,
                               size_t ws_bytes, void* stream) {
  int st = kvc::check_params(p);
  if (st != KVC_OK) return st;
  if (!q || !k_new || !v_new || !Kp || !Vp || !logm || !pos || !len_lh || !cap_lh || !off_lh ||
      !out)
    return KVC_EINVAL;
  const size_t need = kvc::decode_workspace_bytes(p);
  if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return KVC_EWORKSPACE;
  if (kvc::lh_count(p) > 65535) return KVC_EINVAL;
  int32_t* err = kvc::err_word();
  if (!err) return KVC_ECUDA;
  return run_decode(p, q, k_new, v_new, pos_new, Kp, Vp, logm, pos, len_lh, cap_lh, off_lh, out,
                    nullptr, nullptr, static_cast<char*>(workspace), err,
                    static_cast<cudaStream_t>(stream));
}

extern "C" int kvc_decode_attn_layers(const kvc_params* p, int32_t layer_begin,
                                      int32_t layer_end, const void* q, const void* k_new,
                                      const void* v_new, const float* pos_new, void* Kp, void* Vp,
                                      float* logm, float* pos, int32_t* len_lh,
                                      const int32_t* cap_lh, const int64_t* off_lh, void* out,
                                      void* workspace, size_t ws_bytes, void* stream) {
  int st = kvc::check_params(p);
  if (st != KVC_OK) return st;
  if (!q || !k_new || !v_new || !Kp || !Vp || !logm || !pos || !len_lh || !cap_lh || !off_lh ||
      !out || layer_begin < 0 || layer_end > p->L || layer_begin >= layer_end)
    return KVC_EINVAL;
  const size_t need = kvc::decode_workspace_bytes(p);
  if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return KVC_EWORKSPACE;
  if (kvc::lh_count(p) > 65535) return KVC_EINVAL;
  int32_t* err = kvc::err_word();
  if (!err) return KVC_ECUDA;
  // the range's (b,l,h) are local to the call; the per-(b,l,h) arrays stay whole
  kvc_params pr = *p;
  pr.L = layer_end - layer_begin;
  const int64_t span = (int64_t)pr.L * p->H;
  const int64_t gap = (int64_t)(p->L - pr.L) * p->H;
  const int64_t base = (int64_t)layer_begin * p->H;
  return run_decode(&pr, q, k_new, v_new, pos_new, Kp, Vp, logm, pos, len_lh, cap_lh, off_lh, out,
                    nullptr, nullptr, static_cast<char*>(workspace), err,
                    static_cast<cudaStream_t>(stream), span, gap, base, p);
}

extern "C" int kvc_decode_attn_lse(const kvc_params* p, const void* q, const void* k_new,
                                   const void* v_new, const float* pos_new, void* Kp, void* Vp,
                                   float* logm, float* pos, int32_t* len_lh, const int32_t* cap_lh,
                                   const int64_t* off_lh, void* out, float* lse_out,
                                   float* scores_out, void* workspace, size_t ws_bytes,
                                   void* stream) {
  int st = kvc::check_params(p);
  if (st != KVC_OK) return st;
  if (!q || !k_new || !v_new || !Kp || !Vp || !logm || !pos || !len_lh || !cap_lh || !off_lh ||
      !out || !lse_out)
    return KVC_EINVAL;
  const size_t need = kvc::decode_workspace_bytes(p);
  if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return KVC_EWORKSPACE;
  if (kvc::lh_count(p) > 65535) return KVC_EINVAL;
  int32_t* err = kvc::err_word();
  if (!err) return KVC_ECUDA;
  return run_decode(p, q, k_new, v_new, pos_new, Kp, Vp, logm, pos, len_lh, cap_lh, off_lh, out,
                    lse_out, scores_out, static_cast<char*>(workspace), err,
                    static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- allocation-free variant
// Some callers cannot hand the library a workspace: a serving engine whose
// memory pool has already reserved every free byte of HBM for KV blocks, or a
// host framework whose plugin interface has no way to pass scratch and which
// forbids extensions from calling cudaMalloc / cudaFree themselves (cudaFree
// also synchronises the whole device, stalling every other stream).  For them
// kvc_decode_attn_noalloc keeps the split-K scratch in a fixed array that lives
// in this library's device image.
namespace {

constexpr size_t kStaticScratchBytes = (size_t)KVC_DECODE_STATIC_SCRATCH_BYTES;

// Decode workspace (partials, arrival counters, work list).  Every GPU that
// loads this library holds the array until the process exits.
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[256];

// Device address of g_decode_scratch on the current device (looked up once per
// device; in host code the symbol itself is only a host-side stand-in).
void* static_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return nullptr;
  std::lock_guard<std::mutex> g(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) return nullptr;
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int kvc_decode_attn_noalloc(const kvc_params* p, const void* q, const void* k_new,
                                       const void* v_new, const float* pos_new, void* Kp,
                                       void* Vp, float* logm, float* pos, int32_t* len_lh,
                                       const int32_t* cap_lh, const int64_t* off_lh, void* out,
                                       void* stream) {
  int st = kvc::check_params(p);
  if (st != KVC_OK) return st;
  if (!q || !k_new || !v_new || !Kp || !Vp || !logm || !pos || !len_lh || !cap_lh || !off_lh ||
      !out)
    return KVC_EINVAL;
  const int64_t blh = kvc::lh_count(p);
  if (blh > 65535) return KVC_EINVAL;
  const DecodeLayout w = decode_layout(p);
  if (w.total > kStaticScratchBytes) return KVC_ESCRATCH;
  int32_t* err = kvc::err_word();
  char* ws = static_cast<char*>(static_scratch());
  if (!err || !ws) return KVC_ECUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the arrival counters must start at zero (the array keeps the last call's contents)
  cudaError_t e = cudaMemsetAsync(ws + w.counters, 0, (size_t)blh * sizeof(int32_t), s);
  if (e != cudaSuccess) return KVC_ECUDA;
  return run_decode(p, q, k_new, v_new, pos_new, Kp, Vp, logm, pos, len_lh, cap_lh, off_lh, out,
                    nullptr, nullptr, ws, err, s);
}
