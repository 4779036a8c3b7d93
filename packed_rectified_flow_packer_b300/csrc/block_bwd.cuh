// Row-wise and reduction kernels of the NR-MMDiT block backward (memory-bound work around the
// backward's GEMMs and attention).
#pragma once

#include "common.cuh"

namespace mf {

// Modes of the backward's row kernel.  Stream-sorted rows r; seg = (sample, stream) of r; the
// modulation row of seg is mod[seg] = mod + (sample * 2 + stream) * 6H (shift1, scale1, gate1,
// shift2, scale2, gate2); dmod has the same layout.
//  kRowGate2 : dy = gate2 * g                      -> out_bf16
//              dmod.gate2 += sum_r g * y_saved,  bias += sum_r dy
//  kRowLn2   : n = LN(x), dn = da (1 + scale2), dx = g + rstd (dn - mean dn - n mean(dn n))
//              -> out_f32 = dx, out_bf16 = gate1 * dx
//              dmod.shift2 += sum da, dmod.scale2 += sum da n, dmod.gate1 += sum dx * y_saved,
//              bias += sum gate1 * dx
//  kRowLn1   : dx = carry + rstd (dn - mean dn - n mean(dn n)) with dn = da (1 + scale1)
//              -> bf16 to out_first / out_second (the caller's split text / image buffers)
//              dmod.shift1 += sum da, dmod.scale1 += sum da n
enum RowBwdMode : int { kRowGate2 = 0, kRowLn2 = 1, kRowLn1 = 2 };

struct RowBwdArgs {
  int mode;
  int H;
  int n_first;                // rows below n_first read g / write dx in the *_first buffers
  const int* chunks;          // [n_chunks][4] (row0, row1, sample, stream)
  int n_chunks;
  const bf16* g_first;        // gradient of the block output, text rows [n_first][H]
  const bf16* g_second;       // image rows
  const bf16* da;             // [rows][H] gradient of an LN + modulate output (kRowLn*)
  const bf16* x;              // [rows][H] the LN input saved by the forward (kRowLn*)
  const bf16* y;              // [rows][H] saved ungated branch output (kRowGate2, kRowLn2)
  const float* carry;         // [rows][H] f32 residual gradient (kRowLn1)
  const float* mod;           // [S][2][6H]
  float* dmod;                // [S][2][6H], accumulated
  float* bias_grad[2];        // per stream [H], accumulated
  float* out_f32;             // kRowLn2: [rows][H]
  bf16* out_bf16;             // kRowGate2, kRowLn2: [rows][H]
  bf16* out_first;            // kRowLn1: text rows of dx
  bf16* out_second;           // kRowLn1: image rows of dx
  int n_rows, n_seq;          // stream-sorted rows and samples of the pack (bounds of the chunks)
  const int* row_seq;         // kRowLn*: [rows] sample of each stream-sorted row
  float4* stats;              // kRowLn*: [rows] scratch for the rows' LN statistics
};
// H a multiple of 256, at most 4096.
cudaError_t launch_row_bwd(const RowBwdArgs& a, cudaStream_t st);

// bias_grad[stream][c] += sum over the rows of the stream of x[r][c], x bf16 [rows][C]
// (C a multiple of 8), using the row chunks above.
cudaError_t launch_col_sum(const bf16* x, int C, const int* chunks, int n_chunks, float* bias_txt,
                           float* bias_img, cudaStream_t st);

// dqkv[r] = [RoPE^-1(dq_acc[j]) | RoPE^-1(dk[j]) | dv[j]] for stream-sorted row r, j its joint
// token, RoPE over (frame, row, col) as the forward applies it; dq_acc f32 [N][H], dk, dv bf16
// [N][H] joint order; dqkv bf16 [rows][3H].
cudaError_t launch_qkv_grad_gather(const float* dq_acc, const bf16* dk, const bf16* dv, const int* srow_joint,
                                   const int* pos, int rows, int H, int head_dim, bf16* dqkv, int num_sms,
                                   cudaStream_t st);

// Modulation backward, per stream m: dW[m][o][i] = sum_s dmod[s][m][o] c[s][i] (f32 [6H][H]),
// db[m][o] = sum_s dmod[s][m][o]; and dc[s][i] = sum_m sum_o W_mod[m][o][i] dmod[s][m][o]
// (dc f32 [S][H], overwritten).
cudaError_t launch_mod_bwd(const float* dmod, const float* c, int S, int H, const bf16* w_mod_txt,
                           const bf16* w_mod_img, float* dw_txt, float* db_txt, float* dw_img, float* db_img,
                           float* dc, cudaStream_t st);

}  // namespace mf
