// Grouped, persistent GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA) with
// the NR-MMDiT block's fused epilogues.  C[M][N] = A[M][K] B[N][K]^T for up to two problems
// (text stream, image stream) in one launch; bf16 operands, or E4M3 ones (kEpiF8) on the
// pair kernel.
#pragma once

#include "common.cuh"
#include "mageflow.h"

namespace mf {

enum GemmEpi : int {
  kEpiBiasBf16 = 0,   // out bf16 = acc + bias
  kEpiBiasF32 = 1,    // out f32  = acc + bias
  kEpiQkvRope = 2,    // q | k | v = acc + bias; RoPE on q, k; rows scattered to joint order
  kEpiGateResid = 3,  // x += gate[seq] * (acc + bias), x bf16 in place
  kEpiGelu = 4,       // out bf16 = GELU(acc + bias)
  kEpiGeluBwd = 5,    // out bf16 = acc * GELU'(aux[row][col]) (aux: the saved pre-activation)
  kEpiF8 = 8,         // flag on any of the above (pair kernel): E4M3 operands, and the
                      // accumulator is first multiplied by row_scale[row_off + row] * col_scale[col]
  kEpiSave = 16,      // flag on kEpiGelu / kEpiGateResid (pair kernel, bf16): the value before
                      // GELU / before the gate (acc + bias) is also written to aux[row][col]
  kEpiStats = 32,     // flag on kEpiGateResid (pair kernel, bf16): the LN statistics of the new x
                      // (its bf16 values) are written per 128-column part, see GemmParams::ln_stats
};

// Operand majorness of the pair kernel (bf16 only): bit 0 A, bit 1 B.  K-major (0): the matrix
// is stored [rows][K], as in C = A B^T.  MN-major (1): it is stored [K][rows] (A^T or B^T in
// memory), boxes of 64 x 64 with the MN dimension innermost; used by the backward's weight-
// gradient (both) and input-gradient (B) products.
enum GemmMajor : int { kMajKK = 0, kMajAMN = 1, kMajBMN = 2, kMajMNMN = 3 };

struct GemmProblem {
  int M, N, K;
  int row_off;            // first stream-sorted row of this problem (for the row maps)
  int stream;             // modulation stream (0 text, 1 image)
  int ldo;                // output leading dimension in elements
  const bf16* bias;       // [N] or nullptr
  const float* col_scale; // kEpiF8: [N] dequantisation scale of B's rows (output columns)
  void* out;              // output (or the residual x for kEpiGateResid)
  void* aux;              // bf16 [M][ldo]: kEpiSave output, kEpiGeluBwd input; else null
};

struct GemmParams {
  CUtensorMap tmA[2];     // A [M][K], box {64, 128}, 128-byte swizzle
  CUtensorMap tmB[2];     // B [N][K], box {64, BN}, 128-byte swizzle
  CUtensorMap tmC[2];     // bf16 output [M][N] for TMA stores, box {64, 32}, 128-byte swizzle
  int tma_store[2];       // 1: the problem's epilogue stores through tmC (bias / GELU, bf16, ldo == N)
  GemmProblem prob[2];
  int n_prob;
  int tiles_m[2], tiles_n[2];
  int group_m[2];         // tile order: 0 = N fastest, else this many row tiles fastest
  int tile_begin[3];
  // epilogue inputs shared by the problems
  const int* srow_seq;    // [rows] sample of each stream-sorted row
  const int* srow_joint;  // [rows] joint token of each stream-sorted row
  const int* pos;         // [N_tok][3]
  const float* mod;       // [S][2][6H] modulation
  int H;
  int head_dim;
  int n_tok, n_seq;       // pack sizes (bounds of the joint rows and sample ids the epilogues read)
  int gate_off;           // float offset of the gate chunk inside a (sample, stream) mod row
  const bf16* qk_norm[2][2];  // [problem][q, k]: QK-RMSNorm scales [head_dim], or null (off)
  const float* row_scale;     // kEpiF8: dequantisation scale of A's rows (indexed row_off + row)
  // kEpiStats: (mean, sum of squared deviations from it) of each row's 128-column part j of the
  // output, at ln_stats[(row_off + row) * ln_parts + j], ln_parts = N / 128 (N a multiple of 256)
  float2* ln_stats;
  int ln_parts;
  bf16* q;                // [N_tok][H] joint order
  bf16* k;
  bf16* v;
  unsigned* status;
  unsigned long long wait_limit_ns;
};

// Launches the persistent kernel for tile width BN in {128, 256}.
cudaError_t launch_gemm(const GemmParams& p, int BN, int epi, int num_sms, cudaStream_t stream);

// Launches the persistent CTA-pair kernel: 256 x 256 tiles, tmA boxes of 128 rows (each CTA's
// half of the tile's rows), tmB boxes of 128 rows (each CTA's half of the tile's columns),
// tiles_m counted in 256-row tiles.  An MN-major operand's tensor map has boxes of 64 (MN) x 64
// (K) over its [K][MN] storage; K need not be a multiple of 64 (the tail reads zeros).
cudaError_t launch_gemm_pair(const GemmParams& p, int epi, int num_sms, cudaStream_t stream, int maj = kMajKK);

}  // namespace mf
