// Tensor-core probe-times-key passes of kvc_score (internal).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvc.h"

namespace kvc {

enum { kTcRowstatsProbes = 0, kTcRowstatsSeeds = 1, kTcFeats = 2, kTcProp = 3 };

// Per-slot prototype record written by the prototype kernel and read by the
// tensor-core node kernel: k^ split into three bf16 parts (rows 16*part + node,
// 128-byte-swizzled K-major, two 64-feature blocks of 48 rows), ln m and the
// node relevance sums (16 floats each; these three travel in one copy), then
// v^ (fp32).
constexpr int kProtoKhBytes = 2 * 48 * 128;        // 12288
constexpr int kProtoLogmOff = kProtoKhBytes;        // float[16]
constexpr int kProtoRvOff = kProtoLogmOff + 16 * 4; // float[16]
constexpr int kProtoHeadBytes = kProtoRvOff + 16 * 4;   // 12416: k^ parts, ln m, Rv
constexpr int kProtoVhOff = kProtoHeadBytes;        // float[15][128]
constexpr int kProtoBytes = 20480;
static_assert(kProtoVhOff % 16 == 0 && kProtoVhOff + 15 * 128 * 4 <= kProtoBytes, "proto record");

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
  uint64_t wait_ns;       // first-wait limit and copy withholding (kvc_set_wait_limit)
  int withhold;
};

struct NodeTcArgs {
  const int32_t* ctx_len;
  const void* K;
  const void* V;
  const void* Qp;
  const float* lse2;      // [BLH, R]
  const int32_t* ok;
  const int32_t* bounds;  // [B, S_max + 1]
  const int32_t* n_slots;
  const unsigned char* proto;   // [BLH * S_max] records of kProtoBytes
  float* npart;           // [BLH * S_max, 2 tiles, 15 nodes, 4 sums]
  const uint8_t* tree_cuts;     // [BLH * S_max, 8] cut table, or null (midpoint trees)
  int32_t* err;
  int B, L, H, G, P, S_max;
  float q_scale2;
  uint64_t wait_ns;       // first-wait limit and copy withholding (kvc_set_wait_limit)
  int withhold;
};

bool probe_tc_supported(const kvc_params* p);
int nodes_tc_pass(const NodeTcArgs& a, int64_t total_rows, cudaStream_t s);
size_t nodes_tc_smem_bytes();
int probe_tc_pass(int mode, const ProbeTcArgs& a, int64_t total_rows, cudaStream_t s);

}  // namespace kvc
