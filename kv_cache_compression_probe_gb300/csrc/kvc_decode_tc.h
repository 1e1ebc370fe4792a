// Tensor-core decode attention of kvc_decode_attn (internal).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvc.h"

namespace kvc {

struct DecodeTcArgs {
  const void* q;
  const void* k_new;
  const void* v_new;
  const float* pos_new;
  void* Kp;
  void* Vp;
  float* logm;
  float* pos;
  int32_t* len_lh;
  const int32_t* cap_lh;
  const int64_t* off_lh;
  void* out;
  float* partials;      // [BLH, n_chunk_max, G, d + 2]
  int32_t* counters;    // [BLH], zero between calls (unused by this path)
  uint32_t* items;      // [BLH * n_chunk_max] work list: chunk << 16 | (b,l,h)
  int32_t* n_items;     // [1]
  int64_t packed_rows;  // rows of Kp / Vp / logm / pos
  int64_t blh;
  int H, L, G, n_chunk_max;
  float scale_log2;     // log2(e) / sqrt(d)
  int32_t* err;
  float* lse_out;       // [BLH, G] base-2 LSE of the step's scores, or null
  float* scores_out;    // [rows, G] base-2 score of cache row off + i per query head, or null
  // set by decode_tc_launch: with inplan the attention kernel builds the work
  // list itself (no plan kernel); grid_items bounds the work-list length
  int inplan;
  int64_t grid_items;
  // layer range: local (b,l,h) i indexes the per-(b,l,h) arrays (len_lh,
  // cap_lh, off_lh) at i + (i / lh_span) * lh_gap + lh_base (identity for all
  // layers: span = L*H, gap = 0, base = 0); everything else is local
  int64_t lh_span, lh_gap, lh_base;
  // first-wait limit and copy withholding (kvc_set_wait_limit)
  uint64_t wait_ns;
  int withhold;
};

__host__ __device__ inline int64_t lh_global(int64_t i, int64_t span, int64_t gap, int64_t base) {
  return i + (i / span) * gap + base;
}

// bf16, d = 128, G <= 8, a known packed extent below 2^31 rows, at most 65535
// (b,l,h) and chunks per (l,h), and a driver that can encode tensor maps.
bool decode_tc_supported(const kvc_params* p, int n_chunk_max);
// Rows of one split-K chunk (equal to the SIMT kernel's chunk, so both share
// the workspace layout).
constexpr int kDecodeTcChunk = 512;
// Plans the work list, runs the attention kernel and the merge kernel (3
// launches); the merge kernel appends the new token and updates len.
int decode_tc_launch(const DecodeTcArgs& a, cudaStream_t s);

}  // namespace kvc
