// Tensor-core probe-times-key passes of kvc_score (internal).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvc.h"

namespace kvc {

enum { kTcRowstatsProbes = 0, kTcRowstatsSeeds = 1, kTcFeats = 2, kTcProp = 3 };

struct ProbeTcArgs {
  const int32_t* ctx_len;
  const void* K;
  const void* V;
  const void* Qp;
  const int32_t* seeds;
  const float* seed_w;
  const float* lse2;      // [BLH, R] base-2 LSE of probe rows
  const float* hrow;      // [BLH, R] entropy of probe rows
  const float* lse2_h;    // [BLH, P] base-2 LSE of seed rows
  const int32_t* ok;
  float* part;            // [BLH, n_chunks, 256, 3]
  float* feats;
  float* rel;
  int32_t* err;
  int B, L, H, G, P;
  int chunk_tiles;        // 128-key tiles per CTA
  int n_chunks;
  float q_scale2;         // log2(e) / sqrt(d)
  float hop_weight;
};

bool probe_tc_supported(const kvc_params* p);
int probe_tc_pass(int mode, const ProbeTcArgs& a, int64_t total_rows, cudaStream_t s);

}  // namespace kvc
