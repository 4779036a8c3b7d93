// Row-wise and element-wise kernels of the NR-MMDiT path (memory-bound work).
#pragma once

#include "common.cuh"

namespace mf {

// phi(t) = [cos a | sin a], a_j = 1000 t 10000^(-j / (F/2)); out [S][F] f32.
cudaError_t launch_sinusoid(const float* t, int S, int F, float* out, cudaStream_t st);

// y[s][y_off + o] = act(W[o] . x[s] + b[o]) for o < O, W bf16 [O][K], x f32 [S][K];
// act 0 = identity, 1 = SiLU.  K multiple of 256, at most 4096.  *launches (if not null)
// receives the number of kernels launched (one per group of four samples).
// Wide K (at least 1024) runs a kernel with bounded waits, which report to *status.
cudaError_t launch_gemv(const bf16* W, const bf16* b, const float* x, int S, int K, int O,
                        float* y, int y_stride, int y_off, int act, unsigned* status,
                        unsigned long long wait_limit_ns, cudaStream_t st, int* launches = nullptr);

// Two GEMVs with the same x, K and O in one launch per group of four samples:
// y[s][y_off_p + o] = W_p[o] . x[s] + b_p[o] for p = 0, 1 (no activation).
cudaError_t launch_gemv2(const bf16* W0, const bf16* b0, int y_off0, const bf16* W1, const bf16* b1,
                         int y_off1, const float* x, int S, int K, int O, float* y, int y_stride,
                         unsigned* status, unsigned long long wait_limit_ns, cudaStream_t st,
                         int* launches = nullptr);

// Per-row E4M3 quantisation of x bf16 [M][K] (K multiple of 16): s[r] = amax(|x[r]|) / 448
// (1 for an all-zero row), q[r][k] = E4M3(x[r][k] / s[r]) with the division correctly rounded
// in f32 and the conversion rounding to nearest even, saturating to +-448.
cudaError_t launch_quantize_e4m3_rows(const bf16* x, int M, int K, uint8_t* q, float* s, cudaStream_t st);

// out[r] = LN(x[r]) (1 + scale) + shift for stream-sorted rows r in [0, rows), where rows
// below n_first come from x_first and the rest from x_second; (shift, scale) of row r are
// read at mod + seq(r) * seq_stride + stream(r) * stream_stride + {shift_off, scale_off},
// seq(r) = row_seq[r], stream(r) = (r >= n_first).  H multiple of 256, <= 4096.
struct LnModArgs {
  const bf16* x_first;
  const bf16* x_second;
  int n_first;
  int rows;
  int H;
  const int* row_seq;
  const float* mod;
  long long seq_stride;
  long long stream_stride;
  int shift_off;
  int scale_off;
  bf16* out;
  int n_seq;        // bound of row_seq's values
  // optional: per row r, (mean, sum of squared deviations) of each 128-column part j of x[r] at
  // stats[r * (H / 128) + j], as a GEMM epilogue with kEpiStats writes them; null = computed here
  const float2* stats;
  unsigned* status;                 // row-group kernel: bounded waits report here
  unsigned long long wait_limit_ns;
};
// Warp-per-row kernel (statistics from the row in registers).
cudaError_t launch_ln_modulate(const LnModArgs& a, cudaStream_t st);
// Row-group kernel: groups of 8 rows staged in shared memory by bulk copies several groups
// ahead; thread t owns columns 8t .. 8t + 7 and keeps their (shift, scale) in registers across
// the rows of one (sample, stream); statistics from a.stats when given, else computed per group.
cudaError_t launch_ln_group(const LnModArgs& a, cudaStream_t st);

cudaError_t launch_interpolate(const int* img_seq, const int* img_target, const float* t, int Ni,
                               int C, const float* z, const float* eps, float* zt,
                               bf16* zt_bf16, cudaStream_t st);
cudaError_t launch_cfg(const int* img_seq, const int* seq_role, const int* img_pair, int Ni, int C,
                       float w, const float* v, float* out, cudaStream_t st);
cudaError_t launch_euler(int Ni, int C, float dt, const float* v, float* z, bf16* z_bf16,
                         cudaStream_t st);
// ws: [Ni] doubles
cudaError_t launch_flow_loss(const int* cu_img, const int* img_target, int S, int Ni, int C,
                             const float* z, const float* eps, const float* v, double* ws,
                             double* loss_sum, long long* count, double* mean, cudaStream_t st);
// Diffusion-NFT loss: per-row weighted sums, then the flow loss's per-sample and mean passes.
cudaError_t launch_nft_loss(const int* cu_img, const int* img_seq, const int* img_target,
                            const float* reward, int S, int Ni, int C, const float* z,
                            const float* eps, const float* vp, const float* vn, double* ws,
                            double* loss_sum, long long* count, double* mean, cudaStream_t st);
cudaError_t launch_timeout_selftest(unsigned* status, unsigned long long limit_ns,
                                    cudaStream_t st);

}  // namespace mf
