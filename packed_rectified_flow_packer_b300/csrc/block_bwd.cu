// Memory-bound kernels of the NR-MMDiT block backward: the gated-residual and LN + adaLN
// modulate backward rows (with their per-sample modulation and per-stream bias reductions),
// bias column sums, the q / k / v gradient gather with the inverse RoPE, and the modulation
// backward.
//
// The block being differentiated is the SD3-style MMDiT block of the Mage-Flow pages
// (PaperReading review of "Mage-Flow: An Efficient Native-Resolution Foundation Model for Image
// Generation and Editing", §2.2 (3): norm, RoPE, gating and residual chains; §5: MMDiT with
// per-modality projections and norms): x1 = x0 + gate1 (o W_o^T + b_o),
// x2 = x1 + gate2 y_m, with a = LN(x)(1 + scale) + shift before the attention and the MLP.
// For a = n (1 + sc) + sh, n = (x - mu) rstd, the input gradient is
//   dx = rstd (dn - mean(dn) - n mean(dn n)),  dn = da (1 + sc),
// and the modulation gradients are dsh = sum da, dsc = sum da n, dgate = sum dx_out y.
//
// Row kernel (row_bwd_kernel): one CTA per chunk of at most 64 stream-sorted rows inside one
// (sample, stream) segment, H / 8 threads.  The segment's modulation vectors are staged in
// shared memory once.  Phase A (LN modes): warp-per-row statistics (mean, rstd, mean dn,
// mean dn n), two-pass in f32.  Phase B: each thread owns 8 columns for every row of the chunk,
// so the per-column sums accumulate in registers and leave with one atomic add per column per
// chunk.
#include "block_bwd.cuh"

namespace mf {
namespace {

constexpr float kLnEps = 1e-6f;
constexpr int kChunkRows = 64;  // must match the plan's row chunks

__device__ __forceinline__ void load8(const bf16* p, float (&v)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z), d = unpack_bf16x2(u.w);
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y; v[4] = c.x; v[5] = c.y; v[6] = d.x; v[7] = d.y;
}

__device__ __forceinline__ void store8(bf16* p, const float (&v)[8]) {
  *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                            pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

template <int MODE>
__global__ void __launch_bounds__(512) row_bwd_kernel(const RowBwdArgs a) {
  extern __shared__ float sm[];
  const int H = a.H;
  float* vec0 = sm;            // scale (LN modes) or gate2 (kRowGate2)
  float* vec1 = sm + H;        // gate1 (kRowLn2)
  float4* stats = reinterpret_cast<float4*>(sm + 2 * H);  // [64] (mean, rstd, mean dn, mean dn n)
  const int* ch = a.chunks + 4 * blockIdx.x;
  const int row0 = __ldg(ch), row1 = __ldg(ch + 1), seq = __ldg(ch + 2), stream = __ldg(ch + 3);
  if (!MF_IDX_OK(row0 >= 0 && row0 <= row1 && row1 <= a.n_rows && row1 - row0 <= kChunkRows && seq >= 0 &&
                 seq < a.n_seq && (stream == 0 || stream == 1)))
    return;  // before the block-wide barriers: the whole CTA leaves together
  const float* modrow = a.mod + ((size_t)seq * 2 + stream) * 6 * (size_t)H;
  float* dmodrow = a.dmod + ((size_t)seq * 2 + stream) * 6 * (size_t)H;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int off0 = MODE == kRowGate2 ? 5 * H : (MODE == kRowLn2 ? 4 * H : H);
  for (int c = tid; c < H; c += nthr) {
    vec0[c] = __ldg(modrow + off0 + c);
    if (MODE == kRowLn2) vec1[c] = __ldg(modrow + 2 * H + c);
  }
  __syncthreads();

  if constexpr (MODE != kRowGate2) {
    // phase A: per-row statistics, one warp per row
    const int warp = tid >> 5, lane = tid & 31, nw = nthr >> 5;
    for (int r = row0 + warp; r < row1; r += nw) {
      const bf16* xr = a.x + (size_t)r * H;
      const bf16* dr = a.da + (size_t)r * H;
      float s = 0.f;
      for (int c = lane * 8; c < H; c += 256) {
        float v[8];
        load8(xr + c, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) s += v[i];
      }
      const float mean = warp_sum(s) / H;
      float q = 0.f;
      for (int c = lane * 8; c < H; c += 256) {
        float v[8];
        load8(xr + c, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) q += (v[i] - mean) * (v[i] - mean);
      }
      const float rstd = rsqrtf(warp_sum(q) / H + kLnEps);
      float s1 = 0.f, s2 = 0.f;
      for (int c = lane * 8; c < H; c += 256) {
        float v[8], d[8];
        load8(xr + c, v);
        load8(dr + c, d);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float dn = d[i] * (1.0f + vec0[c + i]);
          s1 += dn;
          s2 += dn * (v[i] - mean) * rstd;
        }
      }
      s1 = warp_sum(s1);
      s2 = warp_sum(s2);
      if (lane == 0) stats[r - row0] = make_float4(mean, rstd, s1 / H, s2 / H);
    }
    __syncthreads();
  }

  // phase B: this thread's 8 columns over every row of the chunk
  const int c0 = tid * 8;
  float acc[4][8];
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[k][i] = 0.f;
  for (int r = row0; r < row1; ++r) {
    const size_t off = (size_t)r * H + c0;
    if constexpr (MODE == kRowGate2) {
      float g[8], y[8], dy[8];
      load8(r < a.n_first ? a.g_first + off : a.g_second + (off - (size_t)a.n_first * H), g);
      load8(a.y + off, y);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        dy[i] = vec0[c0 + i] * g[i];
        acc[0][i] += g[i] * y[i];
        acc[1][i] += dy[i];
      }
      store8(a.out_bf16 + off, dy);
    } else {
      const float4 st = stats[r - row0];
      float x[8], d[8], dx[8];
      load8(a.x + off, x);
      load8(a.da + off, d);
      if constexpr (MODE == kRowLn2) {
        float g[8], y[8], dy[8];
        load8(r < a.n_first ? a.g_first + off : a.g_second + (off - (size_t)a.n_first * H), g);
        load8(a.y + off, y);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float n = (x[i] - st.x) * st.y;
          const float dn = d[i] * (1.0f + vec0[c0 + i]);
          dx[i] = g[i] + st.y * (dn - st.z - n * st.w);
          dy[i] = vec1[c0 + i] * dx[i];
          acc[0][i] += d[i];
          acc[1][i] += d[i] * n;
          acc[2][i] += dx[i] * y[i];
          acc[3][i] += dy[i];
        }
        float4* o = reinterpret_cast<float4*>(a.out_f32 + off);
        o[0] = make_float4(dx[0], dx[1], dx[2], dx[3]);
        o[1] = make_float4(dx[4], dx[5], dx[6], dx[7]);
        store8(a.out_bf16 + off, dy);
      } else {
        const float4* cr = reinterpret_cast<const float4*>(a.carry + off);
        const float4 c_lo = __ldg(cr), c_hi = __ldg(cr + 1);
        const float carry[8] = {c_lo.x, c_lo.y, c_lo.z, c_lo.w, c_hi.x, c_hi.y, c_hi.z, c_hi.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float n = (x[i] - st.x) * st.y;
          const float dn = d[i] * (1.0f + vec0[c0 + i]);
          dx[i] = carry[i] + st.y * (dn - st.z - n * st.w);
          acc[0][i] += d[i];
          acc[1][i] += d[i] * n;
        }
        store8(r < a.n_first ? a.out_first + off : a.out_second + (off - (size_t)a.n_first * H), dx);
      }
    }
  }
  // flush: per-sample modulation gradients and per-stream bias gradients
  auto add8 = [&](float* dst, const float (&v)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) atomicAdd(dst + i, v[i]);
  };
  if constexpr (MODE == kRowGate2) {
    add8(dmodrow + 5 * H + c0, acc[0]);
    add8(a.bias_grad[stream] + c0, acc[1]);
  } else if constexpr (MODE == kRowLn2) {
    add8(dmodrow + 3 * H + c0, acc[0]);
    add8(dmodrow + 4 * H + c0, acc[1]);
    add8(dmodrow + 2 * H + c0, acc[2]);
    add8(a.bias_grad[stream] + c0, acc[3]);
  } else {
    add8(dmodrow + c0, acc[0]);
    add8(dmodrow + H + c0, acc[1]);
  }
}

// bias[stream][c..c+7] += column sums of x over the chunk's rows; grid (chunks, C / 2048).
__global__ void col_sum_kernel(const bf16* __restrict__ x, int C, const int* __restrict__ chunks,
                               float* bias_txt, float* bias_img) {
  const int* ch = chunks + 4 * blockIdx.x;
  const int row0 = __ldg(ch), row1 = __ldg(ch + 1), stream = __ldg(ch + 3);
  const int c0 = (blockIdx.y * blockDim.x + threadIdx.x) * 8;
  if (c0 >= C) return;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int r = row0; r < row1; ++r) {
    float v[8];
    load8(x + (size_t)r * C + c0, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += v[i];
  }
  float* dst = (stream ? bias_img : bias_txt) + c0;
#pragma unroll
  for (int i = 0; i < 8; ++i) atomicAdd(dst + i, acc[i]);
}

// One warp per stream-sorted row (grid-stride).  The RoPE pair table is built exactly as the
// forward's QKV epilogue builds it, so the inverse rotation uses the same angles.
__global__ void qkv_grad_gather_kernel(const float* __restrict__ dq_acc, const bf16* __restrict__ dk,
                                       const bf16* __restrict__ dv, const int* __restrict__ srow_joint,
                                       const int* __restrict__ pos, int rows, int H, int D,
                                       bf16* __restrict__ dqkv) {
  __shared__ float rope_inv[64];
  __shared__ int rope_axis[64];
  if ((int)threadIdx.x < D / 2) {
    const int g = threadIdx.x, d = 2 * g;
    const int wf = D / 8, wr = 7 * D / 16;
    int axis, j, width;
    if (d < wf) { axis = 0; j = d / 2; width = wf; }
    else if (d < wf + wr) { axis = 1; j = (d - wf) / 2; width = wr; }
    else { axis = 2; j = (d - wf - wr) / 2; width = wr; }
    rope_axis[g] = axis;
    rope_inv[g] = (float)exp(-(2.0 * j / width) * 9.210340371976184);  // ln(10000)
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
    const int j = __ldg(srow_joint + r);
    if (!MF_IDX_OK(j >= 0 && j < rows)) continue;
    const float pf = (float)__ldg(pos + 3 * j), pr = (float)__ldg(pos + 3 * j + 1), pc = (float)__ldg(pos + 3 * j + 2);
    bf16* out = dqkv + (size_t)r * 3 * H;
    for (int c = lane * 8; c < H; c += 256) {
      const int g0 = (c % D) >> 1;
      float sn[4], cs[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int ax = rope_axis[g0 + i];
        const float th = (ax == 0 ? pf : (ax == 1 ? pr : pc)) * rope_inv[g0 + i];
        // same two-constant Cody-Waite reduction modulo 2 pi and hardware sine / cosine as
        // the forward's epilogue
        const float kq = rintf(th * 0.15915494309189535f);
        const float rr = fmaf(-kq, -1.7484555314695172e-07f, fmaf(-kq, 6.2831854820251465f, th));
        __sincosf(rr, &sn[i], &cs[i]);
      }
      const float4* qa = reinterpret_cast<const float4*>(dq_acc + (size_t)j * H + c);
      const float4 q0 = __ldg(qa), q1 = __ldg(qa + 1);
      float q[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
      float k[8];
      load8(dk + (size_t)j * H + c, k);
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // transpose of the rotation: (y0 c + y1 s, -y0 s + y1 c)
        const float a0 = q[2 * i], a1 = q[2 * i + 1];
        q[2 * i] = a0 * cs[i] + a1 * sn[i];
        q[2 * i + 1] = -a0 * sn[i] + a1 * cs[i];
        const float b0 = k[2 * i], b1 = k[2 * i + 1];
        k[2 * i] = b0 * cs[i] + b1 * sn[i];
        k[2 * i + 1] = -b0 * sn[i] + b1 * cs[i];
      }
      store8(out + c, q);
      store8(out + H + c, k);
      *reinterpret_cast<uint4*>(out + 2 * H + c) = __ldg(reinterpret_cast<const uint4*>(dv + (size_t)j * H + c));
    }
  }
}

// dW[m][o][i4..] = sum_s dmod[s][m][o] c[s][i4..], db[m][o] = sum_s dmod[s][m][o]: one thread per
// 4 outputs along i, both streams (m = blockIdx.y).
__global__ void mod_dw_kernel(const float* __restrict__ dmod, const float* __restrict__ c, int S, int H,
                              float* dw_txt, float* db_txt, float* dw_img, float* db_img) {
  const int m = blockIdx.y;
  const long long n4 = 6LL * H * H / 4;
  float* dw = m ? dw_img : dw_txt;
  float* db = m ? db_img : db_txt;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < n4; t += (long long)gridDim.x * blockDim.x) {
    const int o = (int)(t / (H / 4));
    const int i = (int)(t - (long long)o * (H / 4)) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float bsum = 0.f;
    for (int s = 0; s < S; ++s) {
      const float g = __ldg(dmod + ((size_t)s * 2 + m) * 6 * H + o);
      const float4 cv = __ldg(reinterpret_cast<const float4*>(c + (size_t)s * H + i));
      acc.x = fmaf(g, cv.x, acc.x);
      acc.y = fmaf(g, cv.y, acc.y);
      acc.z = fmaf(g, cv.z, acc.z);
      acc.w = fmaf(g, cv.w, acc.w);
      bsum += g;
    }
    reinterpret_cast<float4*>(dw + (size_t)o * H + i)[0] = acc;
    if (i == 0) db[o] = bsum;
  }
}

// dc[s][i] += sum over a split of the 12H modulation rows (both streams' W_mod stacked) of
// W[o][i] dmod[s][o]; grid (H / 256, 12H / kDcRows, ceil(S / 8)), 128 threads of 2 columns.
constexpr int kDcRows = 512;
__global__ void mod_dc_kernel(const float* __restrict__ dmod, int S, int H, const bf16* __restrict__ w_txt,
                              const bf16* __restrict__ w_img, float* dc) {
  __shared__ float g_sm[kDcRows][8];
  const int i = blockIdx.x * 256 + threadIdx.x * 2;
  const int o0 = blockIdx.y * kDcRows;            // row in the stacked [12H] range
  const int s0 = blockIdx.z * 8;
  const int ns = min(8, S - s0);
  const int rows = min(kDcRows, 12 * H - o0);
  for (int t = threadIdx.x; t < kDcRows * 8; t += blockDim.x) {
    const int rr = t >> 3, ss = t & 7;
    float v = 0.f;
    if (rr < rows && ss < ns) {
      const int o = o0 + rr, m = o >= 6 * H ? 1 : 0;
      v = __ldg(dmod + ((size_t)(s0 + ss) * 2 + m) * 6 * H + (o - m * 6 * H));
    }
    g_sm[rr][ss] = v;
  }
  __syncthreads();
  float acc[8][2];
#pragma unroll
  for (int s = 0; s < 8; ++s) acc[s][0] = acc[s][1] = 0.f;
  for (int rr = 0; rr < rows; ++rr) {
    const int o = o0 + rr;
    const bf16* w = o >= 6 * H ? w_img + (size_t)(o - 6 * H) * H : w_txt + (size_t)o * H;
    const float2 wv = unpack_bf16x2(__ldg(reinterpret_cast<const uint32_t*>(w + i)));
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      acc[s][0] = fmaf(wv.x, g_sm[rr][s], acc[s][0]);
      acc[s][1] = fmaf(wv.y, g_sm[rr][s], acc[s][1]);
    }
  }
  for (int s = 0; s < ns; ++s) {
    atomicAdd(dc + (size_t)(s0 + s) * H + i, acc[s][0]);
    atomicAdd(dc + (size_t)(s0 + s) * H + i + 1, acc[s][1]);
  }
}

}  // namespace

cudaError_t launch_row_bwd(const RowBwdArgs& a, cudaStream_t st) {
  if (a.n_chunks <= 0) return cudaSuccess;
  const int threads = a.H / 8;
  const size_t smem = (2 * (size_t)a.H + 4 * kChunkRows) * sizeof(float);
  switch (a.mode) {
    case kRowGate2: row_bwd_kernel<kRowGate2><<<a.n_chunks, threads, smem, st>>>(a); break;
    case kRowLn2: row_bwd_kernel<kRowLn2><<<a.n_chunks, threads, smem, st>>>(a); break;
    case kRowLn1: row_bwd_kernel<kRowLn1><<<a.n_chunks, threads, smem, st>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_col_sum(const bf16* x, int C, const int* chunks, int n_chunks, float* bias_txt, float* bias_img,
                           cudaStream_t st) {
  if (n_chunks <= 0) return cudaSuccess;
  dim3 grid(n_chunks, (C / 8 + 255) / 256);
  col_sum_kernel<<<grid, 256, 0, st>>>(x, C, chunks, bias_txt, bias_img);
  return cudaGetLastError();
}

cudaError_t launch_qkv_grad_gather(const float* dq_acc, const bf16* dk, const bf16* dv, const int* srow_joint,
                                   const int* pos, int rows, int H, int head_dim, bf16* dqkv, int num_sms,
                                   cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const int blocks = min((rows + 7) / 8, num_sms * 8);
  qkv_grad_gather_kernel<<<blocks, 256, 0, st>>>(dq_acc, dk, dv, srow_joint, pos, rows, H, head_dim, dqkv);
  return cudaGetLastError();
}

cudaError_t launch_mod_bwd(const float* dmod, const float* c, int S, int H, const bf16* w_mod_txt,
                           const bf16* w_mod_img, float* dw_txt, float* db_txt, float* dw_img, float* db_img,
                           float* dc, cudaStream_t st) {
  if (S <= 0) return cudaSuccess;
  const long long n4 = 6LL * H * H / 4;
  dim3 g1((unsigned)min((n4 + 255) / 256, 4096LL), 2);
  mod_dw_kernel<<<g1, 256, 0, st>>>(dmod, c, S, H, dw_txt, db_txt, dw_img, db_img);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(dc, 0, (size_t)S * H * sizeof(float), st);
  if (e != cudaSuccess) return e;
  dim3 g2(H / 256, (12 * H + kDcRows - 1) / kDcRows, (S + 7) / 8);
  mod_dc_kernel<<<g2, 128, 0, st>>>(dmod, S, H, w_mod_txt, w_mod_img, dc);
  return cudaGetLastError();
}

MF_BOUNDS_EXPORT(block_bwd)

}  // namespace mf
