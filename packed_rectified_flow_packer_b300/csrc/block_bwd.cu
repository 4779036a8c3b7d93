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
// LN modes first run ln_bwd_stats_kernel (warp per row, the row of x and da in registers:
// mean, rstd, mean dn, mean dn n, two-pass in f32).  Row kernel (row_bwd_kernel): one CTA per
// half of a plan row chunk (at most 32 stream-sorted rows of one (sample, stream) segment),
// H / 8 threads, the segment's modulation vectors in shared memory; each thread owns 8 columns
// for every row, two rows per step with their loads in flight together, so the per-column sums
// accumulate in registers and leave with one atomic add per column per CTA (two or four rows
// per step with their loads in flight together).
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

__device__ __forceinline__ void unpack8v(const uint4& u, float (&v)[8]) {
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

// Per-row statistics of the LN backward, one warp per row with the row of x and of da in
// registers (H = 256 NV): stats[r] = (mean, rstd, mean dn, mean dn n), dn = da (1 + scale),
// n = (x - mean) rstd, two-pass in f32; scale is the row's (sample, stream) chunk at scale_off.
template <int NV>
__global__ void __launch_bounds__(128) ln_bwd_stats_kernel(const RowBwdArgs a, const int* __restrict__ row_seq,
                                                           int scale_off, float4* __restrict__ stats) {
  mf_pdl_enter();
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= a.n_rows) return;
  constexpr int H = 256 * NV;
  const uint4* xr = reinterpret_cast<const uint4*>(a.x + (size_t)r * H);
  const uint4* dr = reinterpret_cast<const uint4*>(a.da + (size_t)r * H);
  uint4 xu[NV], du[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    xu[i] = __ldg(xr + lane + 32 * i);
    du[i] = __ldg(dr + lane + 32 * i);
  }
  const int seq = __ldg(row_seq + r);
  if (!MF_IDX_OK(seq >= 0 && seq < a.n_seq)) return;
  const float* sc = a.mod + ((size_t)seq * 2 + (r >= a.n_first ? 1 : 0)) * 6 * (size_t)H + scale_off;
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    float v[8];
    unpack8v(xu[i], v);
#pragma unroll
    for (int k = 0; k < 8; ++k) s += v[k];
  }
  const float mean = warp_sum(s) / H;
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    float v[8];
    unpack8v(xu[i], v);
#pragma unroll
    for (int k = 0; k < 8; ++k) q += (v[k] - mean) * (v[k] - mean);
  }
  const float rstd = rsqrtf(warp_sum(q) / H + kLnEps);
  float t1 = 0.f, t2 = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    float v[8], d[8];
    unpack8v(xu[i], v);
    unpack8v(du[i], d);
    const float4* scp = reinterpret_cast<const float4*>(sc + 8 * (lane + 32 * i));
    const float4 s0 = __ldg(scp), s1 = __ldg(scp + 1);
    const float scv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float dn = d[k] * (1.0f + scv[k]);
      t1 += dn;
      t2 += dn * (v[k] - mean);
    }
  }
  t1 = warp_sum(t1);
  t2 = warp_sum(t2);
  if (lane == 0) stats[r] = make_float4(mean, rstd, t1 / H, t2 * rstd / H);
}

// Row kernel: one CTA per half chunk (at most 32 rows of one (sample, stream) segment), H / 8
// threads; thread t owns columns 8t .. 8t + 7 for every row, two rows per step with their loads
// in flight together, so the per-column sums accumulate in registers and leave with one atomic
// add per column per CTA.  The LN modes read the rows' statistics from `stats`.
template <int MODE, int kMaxThreads, int kMinBlocks>
__global__ void __launch_bounds__(kMaxThreads, kMinBlocks) row_bwd_kernel(const RowBwdArgs a,
                                                                          const float4* __restrict__ stats) {
  mf_pdl_enter();
  constexpr int RB = MODE == kRowLn2 ? 2 : 4;  // rows per step, their loads in flight together
  extern __shared__ float sm[];
  const int H = a.H;
  float* vec0 = sm;            // scale (LN modes) or gate2 (kRowGate2)
  float* vec1 = sm + H;        // gate1 (kRowLn2)
  const int* ch = a.chunks + 4 * (blockIdx.x >> 1);
  const int c_row0 = __ldg(ch), c_row1 = __ldg(ch + 1), seq = __ldg(ch + 2), stream = __ldg(ch + 3);
  if (!MF_IDX_OK(c_row0 >= 0 && c_row0 <= c_row1 && c_row1 <= a.n_rows && c_row1 - c_row0 <= kChunkRows &&
                 seq >= 0 && seq < a.n_seq && (stream == 0 || stream == 1)))
    return;  // before the block-wide barrier: the whole CTA leaves together
  const int row0 = c_row0 + (blockIdx.x & 1) * (kChunkRows / 2);
  const int row1 = min(row0 + kChunkRows / 2, c_row1);
  if (row0 >= row1) return;
  const float* modrow = a.mod + ((size_t)seq * 2 + stream) * 6 * (size_t)H;
  float* dmodrow = a.dmod + ((size_t)seq * 2 + stream) * 6 * (size_t)H;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int off0 = MODE == kRowGate2 ? 5 * H : (MODE == kRowLn2 ? 4 * H : H);
  for (int c = tid; c < H; c += nthr) {
    vec0[c] = __ldg(modrow + off0 + c);
    if (MODE == kRowLn2) vec1[c] = __ldg(modrow + 2 * H + c);
  }
  __syncthreads();

  const int c0 = tid * 8;
  float acc[4][8];
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[k][i] = 0.f;
  for (int r = row0; r < row1; r += RB) {
    uint4 gr[RB], yr[RB], xr[RB], dr[RB];
    float4 cr[RB][2];
#pragma unroll
    for (int k = 0; k < RB; ++k) {
      const int rr = min(r + k, row1 - 1);
      const size_t off = (size_t)rr * H + c0;
      if constexpr (MODE != kRowLn1) {
        gr[k] = __ldg(reinterpret_cast<const uint4*>(
            rr < a.n_first ? a.g_first + off : a.g_second + (off - (size_t)a.n_first * H)));
        yr[k] = __ldg(reinterpret_cast<const uint4*>(a.y + off));
      }
      if constexpr (MODE != kRowGate2) {
        xr[k] = __ldg(reinterpret_cast<const uint4*>(a.x + off));
        dr[k] = __ldg(reinterpret_cast<const uint4*>(a.da + off));
      }
      if constexpr (MODE == kRowLn1) {
        cr[k][0] = __ldg(reinterpret_cast<const float4*>(a.carry + off));
        cr[k][1] = __ldg(reinterpret_cast<const float4*>(a.carry + off) + 1);
      }
    }
#pragma unroll
    for (int k = 0; k < RB; ++k) {
      if (r + k >= row1) break;
      const int rr = r + k;
      const size_t off = (size_t)rr * H + c0;
      if constexpr (MODE == kRowGate2) {
        float g[8], y[8], dy[8];
        unpack8v(gr[k], g);
        unpack8v(yr[k], y);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          dy[i] = vec0[c0 + i] * g[i];
          acc[0][i] += g[i] * y[i];
          acc[1][i] += dy[i];
        }
        store8(a.out_bf16 + off, dy);
      } else {
        const float4 st = __ldg(stats + rr);
        float x[8], d[8], dx[8];
        unpack8v(xr[k], x);
        unpack8v(dr[k], d);
        if constexpr (MODE == kRowLn2) {
          float g[8], y[8], dy[8];
          unpack8v(gr[k], g);
          unpack8v(yr[k], y);
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
          const float carry[8] = {cr[k][0].x, cr[k][0].y, cr[k][0].z, cr[k][0].w,
                                  cr[k][1].x, cr[k][1].y, cr[k][1].z, cr[k][1].w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float n = (x[i] - st.x) * st.y;
            const float dn = d[i] * (1.0f + vec0[c0 + i]);
            dx[i] = carry[i] + st.y * (dn - st.z - n * st.w);
            acc[0][i] += d[i];
            acc[1][i] += d[i] * n;
          }
          store8(rr < a.n_first ? a.out_first + off : a.out_second + (off - (size_t)a.n_first * H), dx);
        }
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
  mf_pdl_enter();
  const int* ch = chunks + 4 * blockIdx.x;
  const int row0 = __ldg(ch), row1 = __ldg(ch + 1), stream = __ldg(ch + 3);
  const int c0 = (blockIdx.y * blockDim.x + threadIdx.x) * 8;
  if (c0 >= C) return;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int r = row0;
  for (; r + 4 <= row1; r += 4) {  // four rows' loads in flight
    uint4 u[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) u[k] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(r + k) * C + c0));
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float v[8];
      unpack8v(u[k], v);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += v[i];
    }
  }
  for (; r < row1; ++r) {
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
  mf_pdl_enter();
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

// dW[m][o][i..i+3] = sum_s dmod[s][m][o] c[s][i..i+3], db[m][o] = sum_s dmod[s][m][o]: a block
// per kDwRows rows o of one stream m = blockIdx.y, its threads along i (float4 each), samples
// eight at a time with their dmod values in shared memory and c in registers; the f32 stores
// are the kernel's traffic (a pack with more than eight samples adds to what the first eight
// stored).
constexpr int kDwRows = 16;
__global__ void __launch_bounds__(256) mod_dw_kernel(const float* __restrict__ dmod, const float* __restrict__ c,
                                                     int S, int H, float* dw_txt, float* db_txt, float* dw_img,
                                                     float* db_img) {
  mf_pdl_enter();
  __shared__ float g_sm[kDwRows][8];
  const int m = blockIdx.y;
  const int o0 = blockIdx.x * kDwRows;
  const int rows = min(kDwRows, 6 * H - o0);
  float* dw = m ? dw_img : dw_txt;
  float* db = m ? db_img : db_txt;
  for (int s0 = 0; s0 < S; s0 += 8) {
    const int ns = min(8, S - s0);
    __syncthreads();
    if (threadIdx.x < kDwRows * 8) {
      const int rr = threadIdx.x >> 3, ss = threadIdx.x & 7;
      g_sm[rr][ss] = (rr < rows && ss < ns) ? __ldg(dmod + ((size_t)(s0 + ss) * 2 + m) * 6 * H + o0 + rr) : 0.f;
    }
    __syncthreads();
    if ((int)threadIdx.x < rows) {
      float bs = 0.f;
#pragma unroll
      for (int ss = 0; ss < 8; ++ss) bs += g_sm[threadIdx.x][ss];
      db[o0 + threadIdx.x] = (s0 == 0 ? 0.f : db[o0 + threadIdx.x]) + bs;
    }
    for (int i = threadIdx.x * 4; i < H; i += blockDim.x * 4) {
      float4 cv[8];
#pragma unroll
      for (int ss = 0; ss < 8; ++ss)
        cv[ss] = ss < ns ? __ldg(reinterpret_cast<const float4*>(c + (size_t)(s0 + ss) * H + i))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
      for (int rr = 0; rr < rows; ++rr) {
        float4* dst = reinterpret_cast<float4*>(dw + (size_t)(o0 + rr) * H + i);
        float4 acc = s0 == 0 ? make_float4(0.f, 0.f, 0.f, 0.f) : dst[0];
#pragma unroll
        for (int ss = 0; ss < 8; ++ss) {
          const float g = g_sm[rr][ss];
          acc.x = fmaf(g, cv[ss].x, acc.x);
          acc.y = fmaf(g, cv[ss].y, acc.y);
          acc.z = fmaf(g, cv[ss].z, acc.z);
          acc.w = fmaf(g, cv[ss].w, acc.w);
        }
        dst[0] = acc;
      }
    }
  }
}

// dc[s][i] += sum over a split of the 12H modulation rows (both streams' W_mod stacked) of
// W[o][i] dmod[s][o] for NS samples s0 .. s0 + NS - 1 (those past S have dmod = 0); grid
// (H / 1024, 12H / kDcRows, ceil(S / NS)), 128 threads of 8 columns, eight rows' 16-byte loads
// in flight per step.
constexpr int kDcRows = 128;
template <int NS>
__global__ void __launch_bounds__(128) mod_dc_kernel(const float* __restrict__ dmod, int S, int H,
                                                     const bf16* __restrict__ w_txt, const bf16* __restrict__ w_img,
                                                     float* dc) {
  mf_pdl_enter();
  __shared__ float g_sm[kDcRows][NS];
  const int i = (blockIdx.x * 128 + threadIdx.x) * 8;
  const int o0 = blockIdx.y * kDcRows;            // row in the stacked [12H] range
  const int s0 = blockIdx.z * NS;
  const int ns = min(NS, S - s0);
  const int rows = min(kDcRows, 12 * H - o0);
  for (int t = threadIdx.x; t < kDcRows * NS; t += blockDim.x) {
    const int rr = t / NS, ss = t % NS;
    float v = 0.f;
    if (rr < rows && ss < ns) {
      const int o = o0 + rr, m = o >= 6 * H ? 1 : 0;
      v = __ldg(dmod + ((size_t)(s0 + ss) * 2 + m) * 6 * H + (o - m * 6 * H));
    }
    g_sm[rr][ss] = v;
  }
  __syncthreads();
  if (i >= H) return;
  float acc[NS][8];
#pragma unroll
  for (int s = 0; s < NS; ++s)
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[s][k] = 0.f;
  for (int rr = 0; rr < rows; rr += 8) {
    uint4 u[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int o = o0 + rr + k;
      const bf16* w = o >= 6 * H ? w_img + (size_t)(o - 6 * H) * H + i : w_txt + (size_t)o * H + i;
      u[k] = rr + k < rows ? __ldg(reinterpret_cast<const uint4*>(w)) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float w[8];
      unpack8v(u[k], w);
      const int r2 = min(rr + k, kDcRows - 1);  // rows past `rows` carry w = 0
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        const float g = g_sm[r2][s];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[s][e] = fmaf(w[e], g, acc[s][e]);
      }
    }
  }
  for (int s = 0; s < ns; ++s)
#pragma unroll
    for (int e = 0; e < 8; ++e) atomicAdd(dc + (size_t)(s0 + s) * H + i + e, acc[s][e]);
}

}  // namespace

cudaError_t launch_row_bwd(const RowBwdArgs& a, cudaStream_t st) {
  if (a.n_chunks <= 0) return cudaSuccess;
  if (a.mode != kRowGate2) {
    if (a.stats == nullptr || a.row_seq == nullptr) return cudaErrorInvalidValue;
    const int scale_off = a.mode == kRowLn2 ? 4 * a.H : a.H;
    const int blocks = (a.n_rows + 3) / 4;
    switch (a.H / 256) {
#define MF_STATS_CASE(nv) \
  case nv: launch_k(ln_bwd_stats_kernel<nv>, blocks, 128, 0, st, a, a.row_seq, scale_off, a.stats); break;
      MF_STATS_CASE(1) MF_STATS_CASE(2) MF_STATS_CASE(3) MF_STATS_CASE(4) MF_STATS_CASE(5) MF_STATS_CASE(6)
      MF_STATS_CASE(7) MF_STATS_CASE(8) MF_STATS_CASE(9) MF_STATS_CASE(10) MF_STATS_CASE(11) MF_STATS_CASE(12)
      MF_STATS_CASE(13) MF_STATS_CASE(14) MF_STATS_CASE(15) MF_STATS_CASE(16)
#undef MF_STATS_CASE
      default: return cudaErrorInvalidValue;
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int threads = a.H / 8;
  const size_t smem = 2 * (size_t)a.H * sizeof(float);
  const int grid = 2 * a.n_chunks;  // half chunks
  // up to H = 3072 (384 threads) the register cap lets two CTAs share an SM
  const bool two = threads <= 384;
  switch (a.mode) {
    case kRowGate2:
      if (two) launch_k(row_bwd_kernel<kRowGate2, 384, 2>, grid, threads, smem, st, a, a.stats);
      else launch_k(row_bwd_kernel<kRowGate2, 512, 1>, grid, threads, smem, st, a, a.stats);
      break;
    case kRowLn2:
      if (two) launch_k(row_bwd_kernel<kRowLn2, 384, 2>, grid, threads, smem, st, a, a.stats);
      else launch_k(row_bwd_kernel<kRowLn2, 512, 1>, grid, threads, smem, st, a, a.stats);
      break;
    case kRowLn1:
      if (two) launch_k(row_bwd_kernel<kRowLn1, 384, 2>, grid, threads, smem, st, a, a.stats);
      else launch_k(row_bwd_kernel<kRowLn1, 512, 1>, grid, threads, smem, st, a, a.stats);
      break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_col_sum(const bf16* x, int C, const int* chunks, int n_chunks, float* bias_txt, float* bias_img,
                           cudaStream_t st) {
  if (n_chunks <= 0) return cudaSuccess;
  dim3 grid(n_chunks, (C / 8 + 255) / 256);
  launch_k(col_sum_kernel, grid, 256, 0, st, x, C, chunks, bias_txt, bias_img);
  return cudaGetLastError();
}

cudaError_t launch_qkv_grad_gather(const float* dq_acc, const bf16* dk, const bf16* dv, const int* srow_joint,
                                   const int* pos, int rows, int H, int head_dim, bf16* dqkv, int num_sms,
                                   cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const int blocks = min((rows + 7) / 8, num_sms * 8);
  launch_k(qkv_grad_gather_kernel, blocks, 256, 0, st, dq_acc, dk, dv, srow_joint, pos, rows, H, head_dim, dqkv);
  return cudaGetLastError();
}

cudaError_t launch_mod_bwd(const float* dmod, const float* c, int S, int H, const bf16* w_mod_txt,
                           const bf16* w_mod_img, float* dw_txt, float* db_txt, float* dw_img, float* db_img,
                           float* dc, cudaStream_t st) {
  if (S <= 0) return cudaSuccess;
  dim3 g1((6 * H + kDwRows - 1) / kDwRows, 2);
  launch_k(mod_dw_kernel, g1, 256, 0, st, dmod, c, S, H, dw_txt, db_txt, dw_img, db_img);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(dc, 0, (size_t)S * H * sizeof(float), st);
  if (e != cudaSuccess) return e;
  // samples per launch group: the smallest of 2, 4, 8 that covers S (more groups past 8)
  const int ns = S <= 2 ? 2 : (S <= 4 ? 4 : 8);
  dim3 g2((H / 8 + 127) / 128, (12 * H + kDcRows - 1) / kDcRows, (S + ns - 1) / ns);
  if (ns == 2)
    launch_k(mod_dc_kernel<2>, g2, 128, 0, st, dmod, S, H, w_mod_txt, w_mod_img, dc);
  else if (ns == 4)
    launch_k(mod_dc_kernel<4>, g2, 128, 0, st, dmod, S, H, w_mod_txt, w_mod_img, dc);
  else
    launch_k(mod_dc_kernel<8>, g2, 128, 0, st, dmod, S, H, w_mod_txt, w_mod_img, dc);
  return cudaGetLastError();
}

MF_BOUNDS_EXPORT(block_bwd)

}  // namespace mf
