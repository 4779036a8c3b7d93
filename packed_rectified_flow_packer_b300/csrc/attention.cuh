// Varlen joint attention over a packed batch on the tcgen05 tensor cores.
#pragma once

#include "common.cuh"

namespace mf {

struct AttnParams {
  CUtensorMap tmQ, tmK, tmV;  // [N][H] bf16 joint order, box {64, 128}, 128-byte swizzle
  const int* cu;              // [S+1] joint offsets
  const int* items;           // [n_items][2] (sample, query tile), longest samples first
  const int* joint_srow;      // [N] stream-sorted row of each joint token
  bf16* out;                  // [N][H] stream-sorted output
  float* lse;                 // [heads][N] natural-log logsumexp of each query row's scaled
                              // scores, or null (not written)
  int n_tok;                  // N
  int n_seq;                  // S
  int H;
  int heads;
  int n_items;
  float scale_log2;           // log2(e) / sqrt(D)
  unsigned* status;
  unsigned long long wait_limit_ns;
};

cudaError_t launch_attention(const AttnParams& p, int head_dim, cudaStream_t stream);

}  // namespace mf
