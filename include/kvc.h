/*
 * kvc.h - C ABI of libkvc: budgeted KV-cache compression after prefill and
 * GQA decode attention over the compressed (ragged) cache, for one GB300
 * (sm_103a).
 *
 * The method follows two public pages:
 *   [GK] "GraceKV - Every Cache Entry Earns Its Place: Global Allocation of
 *        Resolution and Coverage for KV Cache Compression" (project page),
 *   [DC] "DistillCache: KL-Guided Adaptive KV-Cache Eviction for
 *        Memory-Efficient LLM Inference", section 3.1.1 (token features).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every pointer argument is caller-owned DEVICE memory unless the comment
 *    says "host".  The library allocates nothing: scratch comes from the
 *    caller's workspace (size from kvc_workspace_bytes).
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream).  Argument errors are detected on the
 *    host before anything is launched and return a negative status.
 *  - Values the host cannot see (per-sequence lengths, slot boundaries,
 *    append capacity) are checked on the device; a violation records a code in
 *    the library's device error word and the offending unit is skipped.  Read
 *    and clear it with kvc_device_error().  No kernel traps or asserts.
 *  - Layouts (all row-major, contiguous).  "(l,h)" = (layer, KV head).
 *      token arrays   sequence b occupies a block starting at token
 *                     T_b = sum_{b'<b} L*H*n_{b'}; token i of (l,h) is row
 *                     T_b + (l*H + h)*n_b + i.  K, V: [rows, d] in `dtype`;
 *                     feats: [rows, 5] f32; relevance: [rows] f32.
 *      probes Qp      [B, L, H*G, P, d] in `dtype`; query head h*G + g serves
 *                     KV head h; probe p sits at position n_b - P + p.
 *      lse            [B, L, H, R] f32 with R = G*P, row rho = g*P + p.
 *      slot_bounds    [B, S_max + 1] int32, slots of b cover [0, n_b - W).
 *      ops            [B, L, H, S_max, 16]: op 0 = Add(slot), op 1 + j =
 *                     Split(node j) of the slot's depth-3 midpoint tree
 *                     (nodes in breadth-first order, 7..14 = leaf prototypes).
 *      per-(l,h)      [B, L, H] arrays (len_lh, cap_lh, off_lh).
 *      packed cache   Kp, Vp: [capacity, d] in `dtype`; logm, pos: [capacity]
 *                     f32.  Entries of (b,l,h) start at row off_lh[b,l,h].
 *      decode         q, out: [B, L, H*G, d]; k_new, v_new: [B, L, H, d].
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes --------------------------------------------------------- */
#define KVC_OK          0
#define KVC_EINVAL     -1   /* bad argument (null pointer, shape, unsupported size) */
#define KVC_EBUDGET    -2   /* budget smaller than the exact recent window          */
#define KVC_ECAPACITY  -3   /* append past an (l,h)'s reserved capacity             */
#define KVC_ECUDA      -4   /* a CUDA runtime call failed                           */
#define KVC_ETIMEOUT   -5   /* a bounded device wait gave up                        */
#define KVC_EWORKSPACE -6   /* workspace missing or smaller than required           */
#define KVC_EDEVICE    -7   /* device-side check failed (see kvc_device_error)      */
#define KVC_ESCRATCH   -8   /* problem too large for the built-in scratch array      */

/* ---- element types -------------------------------------------------------- */
#define KVC_F32  0
#define KVC_BF16 1

/* ---- workspace selectors for kvc_workspace_bytes --------------------------- */
#define KVC_WS_SCORE  0
#define KVC_WS_SELECT 1
#define KVC_WS_PACK   2
#define KVC_WS_DECODE 3
#define KVC_WS_PARTITION 4

/* One parameter block, passed by const pointer, owned by the caller (host). */
typedef struct kvc_params {
  int32_t B;            /* sequences in the batch                                 */
  int32_t L;            /* layers                                                 */
  int32_t H;            /* KV heads                                               */
  int32_t G;            /* query heads per KV head (GQA group), 1..8              */
  int32_t d;            /* head dim: 64 or 128                                    */
  int32_t P;            /* probe positions (last P queries), R = G*P <= 256       */
  int32_t W;            /* exact recent window (tokens per (l,h)), W >= P         */
  int32_t dtype;        /* KVC_F32 or KVC_BF16 for K, V, Qp, q, packed K/V, out   */
  int32_t n_max;        /* largest context length in the batch                    */
  int32_t S_max;        /* largest slot count in the batch (ops are padded to it) */
  float   rope_base;    /* RoPE base (rotate-half pairing), 10000 by default      */
  float   hop_weight;   /* [GK] value flow: weight of each relevance hop, 0.3     */
  int32_t n_hops;       /* [GK] value flow: number of hops, 2                     */
  float   w_part;       /* [GK] fidelity: attention-partition error weight, 0.25  */
  float   w_value;      /* [GK] fidelity: value-aggregate error weight, 0.75      */
  float   value_floor;  /* [GK] value merge: uniform share of the weights, 0.10   */
  double  budget_ratio; /* beta: floor(beta*n) entries per (l,h), pooled          */
  int64_t budget_entries_per_lh; /* > 0 overrides budget_ratio                    */
  double  floor_cap_frac;  /* [GK] singleton floor cap, fraction of B_alloc (0.6)  */
  int64_t floor_cap_tokens;/* token cap of the floor; < 0 = none                   */
  int32_t decode_reserve;  /* rows reserved per (l,h) for decode-time appends      */
  int64_t total_ctx;       /* sum of ctx_len over the batch (rows of K are
                              L*H*total_ctx); 0 = unknown, which disables the
                              tensor-core scoring passes (they need the exact
                              extent of K for their TMA descriptor)             */
  int64_t packed_rows;     /* rows of the packed cache Kp/Vp/logm/pos (the
                              capacity given to kvc_merge_pack); 0 = unknown,
                              which disables the tensor-core decode (its TMA
                              descriptor needs the extent)                      */
  double  head_full_frac;  /* [DC] App. E.3 head-level hybrid: the
                              floor(frac*L*H) heads with the largest relevance
                              mass outside the window keep every token; 0 = off */
  uint8_t* tree_cuts;      /* [GK] "Technical details": curvature-chosen trees.
                              Device array [B, L, H, S_max, 8] (row (b*L + l)*H
                              + h, slot s): byte j < 7 is the cut of internal
                              node j (breadth-first; node j covers [a, b) and
                              its children [a, t), [t, b)) as an offset t - x0
                              from the slot start x0; byte 7 holds the salient
                              flags (below, 0 without salient extraction).
                              Usually written by kvc_tree_cuts.  kvc_score,
                              kvc_select and kvc_merge_pack read it; a cut that
                              leaves a child fewer than 2 or more than 16
                              tokens per leaf below it is replaced by the
                              midpoint (and kvc_score records KVC_EDEVICE).
                              NULL = the depth-3 midpoint trees (an all-zero
                              table gives the same trees).  The three calls of
                              one compression must see the same table.        */
  int32_t salient_extract; /* [GK] "Technical details": tree construction may
                              isolate a salient token with a three-way child
                              set.  Non-zero: kvc_score decides, after the
                              relevance hops, for every depth-2 node j = 3..6
                              covering [a, b) of the binary tree, its most
                              relevant token t (largest relevance, ties to the
                              smaller position, fp32); when both sides keep
                              2..15 tokens the node's children become [a, t),
                              the token t, [t+1, b) (its split costs 2), and
                              kvc_score records the choice in tree_cuts (byte j
                              = t - x0, bit j - 3 of byte 7 set), which must
                              then be non-NULL and hold the binary cuts (a
                              fresh kvc_tree_cuts output, or zeros for the
                              midpoint trees) when kvc_score starts; kvc_select
                              and kvc_merge_pack then follow the three-way
                              trees.  0 = binary trees only (byte 7 must be 0).*/
} kvc_params;

/* Human-readable name of a status code (static string). */
const char* kvc_status_string(int status);

/* Text of the last CUDA runtime error behind a KVC_ECUDA status from any call
 * in this process ("none" if there was none); a static string. */
const char* kvc_last_cuda_error(void);

/* Reads and clears the device error word (synchronises `stream`).  Returns
 * KVC_OK and writes 0 to *code when nothing was recorded, otherwise writes the
 * first recorded code (a negative KVC_* value) to *code. */
int kvc_device_error(void* stream, int32_t* code /* host */);

/* Number of kernels this library has launched since load (host counter). */
int64_t kvc_launch_count(void);

/* Bounded device waits (no counterpart on the pages: error handling of this
 * library).  Kernels that pipeline copies and tensor-core products through
 * mbarriers (the tensor-core passes of kvc_score, both decode kernels of the
 * kvc_decode_attn family) give up a wait after first_wait_ns nanoseconds of
 * global time: the CTA then stops issuing work, waits (with its own fixed
 * limits: 2 s for copies and products already issued, 0.1 s in the probe
 * passes) for what it has in flight, frees its tensor memory, records
 * KVC_ETIMEOUT in the device error word and returns; the call's outputs are
 * then unspecified, and a decode workspace must be zeroed again before its
 * next use.  Default 2e9 ns; accepted range 1e3 .. 2e9.  withhold_copies != 0
 * makes those kernels' producers issue no copies at all, so that their
 * consumers' first waits can only end by the limit: a test of the timeout
 * path that needs no fault.  Process-wide settings read at each launch; set
 * them only while no call is in flight.  Returns KVC_OK or KVC_EINVAL. */
int kvc_set_wait_limit(uint64_t first_wait_ns, int32_t withhold_copies);

/* Bytes of workspace `which` (KVC_WS_*) needs for this parameter block.  The
 * workspace must be 256-byte aligned device memory; its contents need not be
 * initialised except for KVC_WS_DECODE, which must be zeroed once before its
 * first use and is left zeroed by every call. */
size_t kvc_workspace_bytes(int which, const kvc_params* p /* host */);

/* RoPE tables used by kvc_score and kvc_merge_pack.
 * cos_tab[e, j] = cos((e/2) * theta_j), sin_tab likewise, theta_j =
 * base^(-2j/d), for e in [0, n_half) and j < d/2; layout [n_half, d/2] f32.
 * Entry e is position e/2, so half-integer representative positions
 * ([GK] "Inside one cache entry": rerotate at the span's mean position) index
 * it exactly.  Angles are formed and evaluated in double precision on the
 * device.  n_half must be >= 2*n_max.  kvc_tree_cuts reads them too. */
int kvc_rope_table(int32_t d, float base, int64_t n_half, float* cos_tab, float* sin_tab,
                   void* stream);

/* a1-a4: probe scoring, token features, relevance hops, prototype trees,
 * distortion and per-entry utilities of every Add/Split op.
 *   [DC] 3.1.1 (features alpha, |v|, sigma, H, pos); [GK] "03 Bottom-up value
 *   flow" (direct probes + two hops, parent value = sum of children),
 *   "Inside one cache entry" (merge math), technical details (0.25 : 0.75
 *   fidelity), "04 Top-down budget flow" (utility per entry).
 * In:  ctx_len [B] int32; K, V token arrays; Qp probes; rope tables;
 *      slot_bounds [B, S_max+1]; n_slots [B] int32; head_sens [L, H] f32 or
 *      NULL (= 1).
 * Out: lse [B,L,H,R]; feats [rows,5] (alpha, |v|, sigma, H, pos);
 *      relevance [rows]; op_util [B,L,H,S_max,16] f32 (0 for padding);
 *      op_cost [B,L,H,S_max,16] int32 (0 for padding).
 * Slots must have 16..128 tokens; K, V and Qp must be 16-byte aligned
 * (KVC_EINVAL otherwise).  Errors: KVC_EINVAL, KVC_EWORKSPACE, KVC_ECUDA; bad
 * per-sequence values are reported via kvc_device_error. */
int kvc_score(const kvc_params* p, const int32_t* ctx_len, const void* K, const void* V,
              const void* Qp, const float* rope_cos, const float* rope_sin,
              const int32_t* slot_bounds, const int32_t* n_slots, const float* head_sens,
              float* lse, float* feats, float* relevance, float* op_util, int32_t* op_cost,
              void* workspace, size_t ws_bytes, void* stream);

/* Phase timing of kvc_score's tensor-core path (a measurement aid; no
 * counterpart on the pages).  With timing on, each kvc_score call on that
 * path records CUDA events on its stream between its phases (not for use
 * during stream capture); the events are created on the device current at
 * the first timed call, and calls on other devices are not timed.
 * kvc_score_phase_ms waits for the last timed call and writes up to n
 * durations in ms: [0] probe row statistics, [1] per-key features, [2] value
 * norms and relevance hops, [3] prototypes, [4] node statistics.  Returns the
 * number written, or KVC_EINVAL when no timed call completed its phases. */
void kvc_set_phase_timing(int on);
int kvc_score_phase_ms(float* ms_out /* host */, int32_t n);

/* a5: per-sequence budget, capped singleton floor, global greedy Add/Split
 * auction ([GK] "Core idea" budget regions, "Exact-information safeguard",
 * "04 Top-down budget flow").  The result is identical to processing one
 * queue of exposed ops in (utility desc, op id asc) order, taking each op
 * whose cost fits the remaining budget and discarding the rest.
 * In:  relevance (floor keys r*sens), op_util, op_cost from kvc_score.
 * With head_full_frac > 0 the floor(frac*L*H) heads of each sequence with the
 * largest relevance mass outside the window (float64 sums; ties to the lower
 * l*H+h) take every op (every token exact, len = n) and pay n - W beyond their
 * window from the same budget; the floor and auction run on the other heads.
 * Out: taken [B,L,H,S_max,16] uint8 (1 = op bought); len_lh [B,L,H] int32
 *      (stored entries incl. the W window tokens); cap_lh = len_lh +
 *      decode_reserve; off_lh [B,L,H] int64 exclusive prefix sum of cap_lh in
 *      (b,l,h) order; total_entries [1] int64 = sum of cap_lh (rows the packed
 *      cache needs).
 * Errors: KVC_EINVAL, KVC_EBUDGET (some sequence's budget < its window),
 * KVC_EWORKSPACE, KVC_ECUDA. */
int kvc_select(const kvc_params* p, const int32_t* ctx_len, const int32_t* slot_bounds,
               const int32_t* n_slots, const float* relevance, const float* head_sens,
               const float* op_util, const int32_t* op_cost, uint8_t* taken, int32_t* len_lh,
               int32_t* cap_lh, int64_t* off_lh, int64_t* total_entries, void* workspace,
               size_t ws_bytes, void* stream);

/* a3 + a6: merge each stored frontier node into one entry and pack the ragged
 * cache ([GK] "05 Physical cache packing"): per (b,l,h), slots ascending, each
 * slot's frontier left to right, then the window tokens.  A split leaf stores
 * its tokens bit-exact (log m = 0, pos = i); an unsplit node stores its
 * prototype (k_hat, v_hat, ln m, mean position).  Rows between len and cap
 * are left untouched for appends.  capacity = rows of Kp/Vp/logm/pos; a
 * sequence whose entries would overflow it is skipped and reported via
 * kvc_device_error.  K, V, Kp and Vp must be 16-byte aligned (KVC_EINVAL
 * otherwise).  Errors: KVC_EINVAL, KVC_EWORKSPACE, KVC_ECUDA. */
int kvc_merge_pack(const kvc_params* p, const int32_t* ctx_len, const void* K, const void* V,
                   const float* relevance, const float* rope_cos, const float* rope_sin,
                   const int32_t* slot_bounds, const int32_t* n_slots, const uint8_t* taken,
                   const int32_t* len_lh, const int64_t* off_lh, void* Kp, void* Vp,
                   float* logm, float* pos, int64_t capacity, void* workspace, size_t ws_bytes,
                   void* stream);

/* a7: one decode step over the ragged cache, all layers in one launch
 * ([GK] "05": new tokens are appended with multiplicity one; decode attends
 * with the +ln m bias).  For every (b,l,h) the new (k_new, v_new) is appended
 * at row off_lh + len_lh (log m = 0, pos = pos_new[b]) and the G query heads
 * attend over all len_lh + 1 entries:
 *   out = sum_e softmax_e(q . k_e / sqrt(d) + logm_e) v_e   (fp32 softmax).
 * len_lh is incremented on the device.  An (l,h) with len_lh + 1 > cap_lh
 * still attends (including the new token) but is not appended and reports
 * KVC_ECAPACITY via kvc_device_error.  pos_new may be NULL.
 * Workspace KVC_WS_DECODE holds split-K partials, per-(b,l,h) arrival
 * counters and a work list (zero before first use; every call leaves the
 * counters zero, except after a KVC_ETIMEOUT report, when the caller must zero
 * the workspace again).
 * With dtype KVC_BF16, d = 128 and packed_rows > 0 the attention runs on the
 * tensor cores (P = softmax numerators rounded to bf16 for the PV product; the
 * row sums use the same rounded values); every row the call touches must then
 * lie in [0, packed_rows), and an (l,h) whose off_lh + len_lh exceeds it is
 * skipped and reported as KVC_EDEVICE.
 * Errors: KVC_EINVAL, KVC_EWORKSPACE, KVC_ECUDA. */
int kvc_decode_attn(const kvc_params* p, const void* q, const void* k_new, const void* v_new,
                    const float* pos_new, void* Kp, void* Vp, float* logm, float* pos,
                    int32_t* len_lh, const int32_t* cap_lh, const int64_t* off_lh, void* out,
                    void* workspace, size_t ws_bytes, void* stream);

/* kvc_decode_attn over the layers [layer_begin, layer_end) only, for callers
 * that run the model layer by layer (each layer's queries exist only after the
 * previous layer).  q, k_new, v_new and out cover the range:
 * [B, layer_end - layer_begin, H*G (or H), d]; len_lh, cap_lh and off_lh are
 * the whole [B, L, H] arrays (only the range's entries are read or advanced);
 * p describes all L layers and the workspace is the one for p (shared with
 * kvc_decode_attn; the same zeroing rule).  Results equal the range's part of
 * a kvc_decode_attn call.  Errors: as kvc_decode_attn, and KVC_EINVAL unless
 * 0 <= layer_begin < layer_end <= L. */
int kvc_decode_attn_layers(const kvc_params* p, int32_t layer_begin, int32_t layer_end,
                           const void* q, const void* k_new, const void* v_new,
                           const float* pos_new, void* Kp, void* Vp, float* logm, float* pos,
                           int32_t* len_lh, const int32_t* cap_lh, const int64_t* off_lh,
                           void* out, void* workspace, size_t ws_bytes, void* stream);

/* kvc_decode_attn that also returns the base-2 log-sum-exp of each query
 * head's scores over the len_lh + 1 entries it attended:
 *   lse_out[(b,l,h), g] = log2 sum_e 2^(s_e),  s_e = (q_g . k_e / sqrt(d) + logm_e) log2 e.
 * (kvc_token_alpha needs it to form the DistillCache attention feature.)
 * On the tensor-core path the sum runs over the bf16-rounded numerators that
 * also normalise `out` (relative error of each term at most 2^-9).
 * lse_out: [B*L*H, G] f32 device, required.
 * scores_out: NULL, or f32 device rows laid out like Kp ([rows, G]): row
 * off_lh + e receives, per query head g, the base-2 score s_e of that
 * attended entry (e < len_lh + 1; the appended token's row only when it was
 * appended).  Everything else, results and errors as kvc_decode_attn. */
int kvc_decode_attn_lse(const kvc_params* p, const void* q, const void* k_new, const void* v_new,
                        const float* pos_new, void* Kp, void* Vp, float* logm, float* pos,
                        int32_t* len_lh, const int32_t* cap_lh, const int64_t* off_lh, void* out,
                        float* lse_out, float* scores_out, void* workspace, size_t ws_bytes,
                        void* stream);

/* NEXT f2, DistillCache inference with the heuristic score (DistillCache
 * Algorithm 1; the learned policy is replaced by its first feature, the
 * attention received, 3.1.1).  An evicting cache holds the same tokens in the
 * same rows of every (layer, KV head) of a sequence (row i is one token
 * everywhere; len_lh equal across the sequence's (l,h)), every entry with
 * log m = 0 and an integer position pos in [0, 2^24).
 *
 * kvc_token_alpha: per cache row i of sequence b
 *   alpha[b, i] = 1/(L H G) sum_{l,h,g} 2^(s_i - lse_out[(b,l,h), g])
 * with q the step's queries [B, L, H*G, d] and lse_out from
 * kvc_decode_attn_lse of the same step (so the rows include its appended
 * token).  With `scores` (that call's scores_out) s_i is read from it and q,
 * Kp may be NULL; with scores == NULL s_i is recomputed in fp32 from q and K
 * (every log m taken as 0).  The (l,h) are summed in fixed groups, so the
 * result is deterministic.  alpha: [B, alpha_cols] f32;
 * rows i >= len are not written.  A sequence whose len_lh differ across (l,h),
 * or exceed alpha_cols, reports KVC_EDEVICE.  Workspace: kvc_evict_workspace_bytes.
 * Errors: KVC_EINVAL, KVC_EWORKSPACE, KVC_ECUDA. */
int kvc_token_alpha(const kvc_params* p, const void* q, const void* Kp, const float* scores,
                    const int32_t* len_lh, const int64_t* off_lh, const float* lse_out,
                    float* alpha, int32_t alpha_cols, void* workspace, size_t ws_bytes,
                    void* stream);

/* Workspace bytes of kvc_token_alpha and kvc_evict_topb (one buffer may serve
 * both; 256-byte aligned device memory, no initialisation needed); 0 for
 * invalid arguments. */
size_t kvc_evict_workspace_bytes(const kvc_params* p /* host */, int32_t alpha_cols);

/* kvc_evict_topb: per sequence B_b = min(len, max(floor(ratio * n_seen[b]),
 * b_min)); keeps the B_b rows with the largest alpha, ties to the earlier
 * token (smaller pos of the sequence's first (l,h)), and sets len_lh = B_b.
 * In place: the kept rows at index >= B_b move into the evicted rows below
 * B_b (K, V, pos and logm rows of every (l,h) alike), so after the call the
 * rows are in no particular position order.  n_seen [B] int64 device: tokens
 * seen so far, this step's included.  Errors: KVC_EINVAL, KVC_EWORKSPACE,
 * KVC_ECUDA; inconsistent lengths report KVC_EDEVICE. */
int kvc_evict_topb(const kvc_params* p, const float* alpha, int32_t alpha_cols,
                   const int64_t* n_seen, double ratio, int32_t b_min, void* K, void* V,
                   float* pos, float* logm, const int64_t* off_lh, int32_t* len_lh,
                   void* workspace, size_t ws_bytes, void* stream);

/* Allocation-free variant of kvc_decode_attn (no counterpart on the pages: it
 * is an interface convenience, not part of the method).  For callers that
 * cannot allocate device memory on the library's behalf: a serving engine whose
 * pool already holds every free byte of HBM for KV blocks, or a host framework
 * whose plugin interface cannot pass a workspace and forbids cudaMalloc /
 * cudaFree inside extensions (cudaFree also synchronises the device).
 * Same arguments, results and errors as kvc_decode_attn, minus the workspace:
 * the split-K scratch lives in one file-scope device array of
 * KVC_DECODE_STATIC_SCRATCH_BYTES that every GPU loading the library holds
 * until the process exits.  The call allocates nothing (no cudaMalloc, no
 * cudaFree, no allocating library routine).
 *  - Problems whose scratch (kvc_workspace_bytes(KVC_WS_DECODE)) exceeds the
 *    array return KVC_ESCRATCH before anything is launched.
 *  - The first call on a device looks up the array's device address with that
 *    device current (cudaGetSymbolAddress); make that first call before any
 *    stream capture.
 *  - Every call clears the arrival counters it needs (cudaMemsetAsync on the
 *    stream) and reuses the same array: calls that overlap on the GPU, on any
 *    streams, race on it and must be serialised by the caller. */
#define KVC_DECODE_STATIC_SCRATCH_BYTES (48u << 20)
int kvc_decode_attn_noalloc(const kvc_params* p, const void* q, const void* k_new,
                            const void* v_new, const float* pos_new, void* Kp, void* Vp,
                            float* logm, float* pos, int32_t* len_lh, const int32_t* cap_lh,
                            const int64_t* off_lh, void* out, void* stream);

/* a0: curvature-guided slot partition ([GK] "01 Curvature-guided
 * partition"): kappa(t) = mean over w in {1,2,4,8} of
 * 1 - cos(h_t - h_{t-w}, h_{t+w} - h_t) on L2-normalised hidden states, then a
 * dynamic program over cuts in [0, n_b - W) maximising
 * sum kappa(cuts) - lambda * sum ((len - 64)/64)^2 with 16 <= len <= 128 and
 * lambda = mean kappa.  hidden: [B, n_max, dh] in `dtype` (rows beyond n_b
 * unused).  Out: kappa [B, n_max] f32, slot_bounds [B, S_max+1], n_slots [B].
 * A sequence needing more than S_max slots reports KVC_EDEVICE. */
int kvc_partition(const kvc_params* p, const int32_t* ctx_len, const void* hidden, int32_t dh,
                  float* kappa, int32_t* slot_bounds, int32_t* n_slots, void* workspace,
                  size_t ws_bytes, void* stream);

/* f3: curvature-chosen prototype trees ([GK] "Technical details and default
 * settings": tree construction considers high-curvature split candidates plus
 * the midpoint; the curvature of "01 Curvature-guided partition").  Per
 * (b,l,h), the keys with RoPE removed and normalised, u_i = R(-i)k_i/|.|, give
 *   kappa(t) = mean over w in {1,2,4,8} with w <= t < n_b - w of
 *              1 - cos(u_t - u_{t-w}, u_{t+w} - u_t)   (cos = 1 for a zero chord),
 * written to kappa (token layout, like kvc_score's features: rows
 * (l*H + h)*n_b + i of sequence b's block).  Then, per slot tree, top-down,
 * internal node j = [a, b) of depth k (c tokens, m = floor((a+b)/2)) is cut
 * at the t maximising kappa(t) - lambda*((t - m)/(c/2))^2 with lambda the mean
 * of kappa over [a, b) (summed in index order), among the t that leave each
 * child 2 .. 16 tokens per leaf below it (2^(2-k) leaves; the midpoint always
 * qualifies); ties go to the midpoint, then to the
 * smaller t.  Every step of that decision is an individually rounded fp32
 * operation in the order written.  cuts: [B, L, H, S_max, 8] bytes, the
 * table kvc_params.tree_cuts takes (byte j < 7 = cut of node j minus the slot
 * start; byte 7 = 0; all 8 bytes 0 for padding slots s >= n_slots[b]).
 * K is the token layout of kvc_score, 16-byte aligned; rope_cos / rope_sin
 * as for kvc_score (n_half >= 2*n_max).  No workspace.  B*L*H must be at most
 * 65535 and K aligned (KVC_EINVAL before any launch).  Slot bounds outside 16..128 tokens or
 * beyond n_b - W leave that slot's bytes unwritten and record KVC_EDEVICE.
 * Non-finite keys give unspecified (but valid) cuts. */
int kvc_tree_cuts(const kvc_params* p, const int32_t* ctx_len, const void* K,
                  const float* rope_cos, const float* rope_sin, const int32_t* slot_bounds,
                  const int32_t* n_slots, float* kappa, uint8_t* cuts, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* KVC_H */
