// Backward of the varlen joint attention (tcgen05, diagonal blocks only).
#pragma once

#include "common.cuh"

namespace mf {

struct AttnBwdParams {
  CUtensorMap tmK, tmV;       // [N][H] bf16 joint order, box {64, 128}, 128-byte swizzle
  CUtensorMap tmQ, tmDO;      // [N][H] bf16 joint order, box {64, 64}, 128-byte swizzle
  CUtensorMap tmDQ;           // dq accumulator [N][H] f32, box {32, 32}, no swizzle
  const int* cu;              // [S+1] joint offsets
  const int* items;           // work list (sequence, 256-row query block), longest first
  int n_items;
  const float* lse;           // [heads][N] natural-log logsumexp of the forward's scaled scores
  const float* delta;         // [heads][N] rowsum(do * o)
  bf16* dk;                   // [N][H] joint order
  bf16* dv;                   // [N][H] joint order
  int n_tok, n_seq, H, heads, head_dim;
  float scale_log2;           // log2(e) / sqrt(D)
  float scale;                // 1 / sqrt(D)
  unsigned* status;
  unsigned long long wait_limit_ns;
};

// delta and the joint-order copy of do (do_joint null: do is already in joint order and
// dout_joint = 1), and the dq accumulator cleared.  o, and do when dout_joint = 0, are
// stream-sorted.
cudaError_t launch_attention_bwd_prep(const bf16* o, const bf16* dout, int dout_joint, const int* joint_srow,
                                      int N, int H, int head_dim, bf16* do_joint, float* delta, float* dq_acc,
                                      int num_sms, cudaStream_t st);
// n_ctas = sum over samples of ceil(L / 128), times heads.
cudaError_t launch_attention_bwd(const AttnBwdParams& p, long long n_ctas, cudaStream_t st);
cudaError_t launch_attention_bwd_dq(const float* acc, bf16* dq, long long n, int num_sms, cudaStream_t st);

}  // namespace mf
