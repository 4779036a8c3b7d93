// Memory-bound kernels of the packed NR-MMDiT path: timestep conditioning GEMVs, the
// LN + adaLN-modulate prologue, and the rectified-flow epilogues (interpolation, packed CFG,
// Euler step, flow-matching loss).  Vectorised 16-byte accesses; one warp per row where a
// row reduction is needed.
//
// Definitions: PaperReading review of "Mage-Flow: An Efficient Native-Resolution Foundation
// Model for Image Generation and Editing", §2.2 (2) (z_t = (1 - t) z + t eps and the loss
// ||v - (z - eps)||^2, editing loss on the target latent only), §2.2 (3) (packed CFG, fused
// norm / gating chains) and §5 (ODE sampling from noise to data; CFG from the difference of
// the conditional and unconditional predictions); hyper.ai summary, 方法.
#include "pointwise.cuh"

#include <algorithm>

namespace mf {
namespace {

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z),
         d = unpack_bf16x2(u.w);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y; f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------------ conditioning
__global__ void sinusoid_kernel(const float* __restrict__ t, int S, int F, float* __restrict__ out) {
  mf_pdl_enter();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int half = F / 2;
  if (i >= S * half) return;
  const int s = i / half, j = i - s * half;
  // computed in double: the argument reaches 1000 rad
  const double a = 1000.0 * (double)t[s] * exp(-9.210340371976184 * (double)j / (double)half);
  out[(size_t)s * F + j] = (float)cos(a);
  out[(size_t)s * F + half + j] = (float)sin(a);
}

// Streaming 16-byte load of read-once data (weights, activations): not kept in L1.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 u;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
               : "l"(p));
  return u;
}

// (a0, a1) += (w0 * x0, w1 * x1) as one packed f32x2 FMA.
__device__ __forceinline__ void ffma2(float& a0, float& a1, float w0, float w1, float x0, float x1) {
  asm("{\n\t.reg .b64 a, w, x;\n\t"
      "mov.b64 a, {%0, %1};\n\tmov.b64 w, {%2, %3};\n\tmov.b64 x, {%4, %5};\n\t"
      "fma.rn.f32x2 a, w, x, a;\n\tmov.b64 {%0, %1}, a;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(w0), "f"(w1), "f"(x0), "f"(x1));
}

// y[s][y_off[p] + o] = act(W_p[o] . x[s] + b_p[o]) for the samples s < S <= 4 of one launch and
// the problem p = blockIdx.y.  One warp per kGemvRows consecutive output features; lane l owns
// the 8-element chunks k = 8 l + 256 i, i < NCH = K / 256.  The weights (read once, streamed past
// L1) pass through a register ring: the loads of chunk i + kGemvDepth are issued before chunk i
// is used.  Every chunk of x (f32, from L1) is loaded once for all rows of the warp; with two
// rows per warp the L1 traffic for x was four times the weight bytes and bounded the kernel.
// Products accumulate as packed f32x2 FMAs into even / odd partial sums that meet before the
// warp reduction.  Samples beyond S reuse the last sample's x (valid addresses; their sums are
// not stored), which keeps the x loads free of branches.
constexpr int kGemvRows = 4;
constexpr int kGemvDepth = 1;

struct GemvArgs {
  const bf16* W[2];
  const bf16* b[2];
  int y_off[2];
  const float* x;
  int S, O;
  float* y;
  int y_stride;
  unsigned* status;                 // bulk kernel: bounded waits report here
  unsigned long long wait_limit_ns;
};

template <int ACT, int NCH>
__global__ void __launch_bounds__(128) gemv_kernel(const GemvArgs g) {
  mf_pdl_enter();
  constexpr int K = NCH * 256;
  constexpr int R = kGemvRows, D = kGemvDepth;
  const int pb = blockIdx.y;
  const int o0 = ((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * R;
  const int lane = threadIdx.x & 31;
  if (o0 >= g.O) return;
  const int nr = min(R, g.O - o0);
  const int S = g.S;
  const bf16* wrow = (pb ? g.W[1] : g.W[0]) + (size_t)o0 * K + lane * 8;
  uint4 wv[D + 1][R];
#pragma unroll
  for (int i = 0; i < D && i < NCH; ++i)
#pragma unroll
    for (int r = 0; r < R; ++r)
      wv[i][r] = r < nr ? ld_stream16(wrow + (size_t)r * K + 256 * i) : make_uint4(0, 0, 0, 0);
  float acc[R][4][2] = {};
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    if (i + D < NCH) {
#pragma unroll
      for (int r = 0; r < R; ++r)
        wv[(i + D) % (D + 1)][r] = r < nr ? ld_stream16(wrow + (size_t)r * K + 256 * (i + D)) : make_uint4(0, 0, 0, 0);
    }
    const int k = lane * 8 + 256 * i;
    float xv[4][8];
#pragma unroll
    for (int si = 0; si < 4; ++si) {
      const float4* xp = reinterpret_cast<const float4*>(g.x + (size_t)min(si, S - 1) * K + k);
      const float4 a = __ldg(xp), c = __ldg(xp + 1);
      xv[si][0] = a.x; xv[si][1] = a.y; xv[si][2] = a.z; xv[si][3] = a.w;
      xv[si][4] = c.x; xv[si][5] = c.y; xv[si][6] = c.z; xv[si][7] = c.w;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float wf[8];
      unpack8(wv[i % (D + 1)][r], wf);
#pragma unroll
      for (int si = 0; si < 4; ++si)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          ffma2(acc[r][si][0], acc[r][si][1], wf[2 * j], wf[2 * j + 1], xv[si][2 * j], xv[si][2 * j + 1]);
    }
  }
  const bf16* bias = pb ? g.b[1] : g.b[0];
  float* y = g.y + (pb ? g.y_off[1] : g.y_off[0]) + o0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int si = 0; si < 4; ++si) {
      const float v = warp_sum(acc[r][si][0] + acc[r][si][1]);
      if (lane == 0 && r < nr && si < S) {
        const float t = v + (bias ? __bfloat162float(bias[o0 + r]) : 0.0f);
        y[(size_t)si * g.y_stride + r] = ACT == 1 ? silu_f(t) : t;
      }
    }
  }
}

// The same product for wide K (the H x H and 6H x H matrices): groups of kBulkRows rows are
// staged in shared memory by bulk copies (one per 2K-byte row), two groups per CTA in flight and
// two CTAs per SM, so the weight stream keeps HBM busy without holding the bytes in registers.
// The four warps split a group's K chunks (chunk i to warp i mod 4) over all its rows, so each
// chunk of x is read once per group from L1 for kBulkRows rows; the per-warp partial sums meet
// in shared memory.  CTAs take groups blockIdx.x, blockIdx.x + gridDim.x, ...
constexpr int kBulkRows = 8;

template <int ACT, int NCH>
__global__ void __launch_bounds__(128, 2) gemv_bulk_kernel(const GemvArgs g, int n_groups) {
  mf_pdl_enter();
  constexpr int K = NCH * 256;
  constexpr uint32_t kRowBytes = K * 2, kStage = kBulkRows * kRowBytes;
  extern __shared__ __align__(128) uint8_t gsm[];
  __shared__ uint64_t full_bar[2];
  __shared__ float part[2][4][kBulkRows][4];  // [group parity][warp][row][sample]
  __shared__ int abort_sh;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int pb = blockIdx.y;
  const bf16* W = pb ? g.W[1] : g.W[0];
  const bf16* bias = pb ? g.b[1] : g.b[0];
  float* y = g.y + (pb ? g.y_off[1] : g.y_off[0]);
  const int O = g.O, S = g.S;
  if ((int)blockIdx.x >= n_groups) return;
  if (t == 0) {
    mbar_init(&full_bar[0], 1);
    mbar_init(&full_bar[1], 1);
    abort_sh = 0;
    fence_barrier_init();
  }
  __syncthreads();
  int issued = 0;  // thread 0: groups of this CTA whose copies have been issued
  auto issue = [&](int gi, int s) {
    const int o0 = gi * kBulkRows, nr = min(kBulkRows, O - o0);
    mbar_arrive_expect_tx(&full_bar[s], nr * kRowBytes);
    for (int r = 0; r < nr; ++r)
      bulk_load(gsm + s * kStage + r * kRowBytes, W + (size_t)(o0 + r) * K, kRowBytes, &full_bar[s]);
    ++issued;
  };
  if (t == 0) {
    issue(blockIdx.x, 0);
    if ((int)(blockIdx.x + gridDim.x) < n_groups) issue(blockIdx.x + gridDim.x, 1);
  }
  int it = 0;
  for (int gi = blockIdx.x; gi < n_groups; gi += gridDim.x, ++it) {
    const int s = it & 1;
    const int o0 = gi * kBulkRows, nr = min(kBulkRows, O - o0);
    if (!mbar_wait(&full_bar[s], (uint32_t)(it >> 1) & 1u, g.wait_limit_ns)) {
      report_status(g.status, kStatusTimeout);
      abort_sh = 1;
    }
    const uint8_t* buf = gsm + s * kStage;
    float acc[kBulkRows][4][2];
#pragma unroll
    for (int r = 0; r < kBulkRows; ++r)
#pragma unroll
      for (int si = 0; si < 4; ++si) acc[r][si][0] = acc[r][si][1] = 0.f;
#pragma unroll
    for (int i0 = 0; i0 < NCH; i0 += 4) {
      const int i = i0 + warp;
      if (i < NCH) {
        const int k = lane * 8 + 256 * i;
        float xv[4][8];
#pragma unroll
        for (int si = 0; si < 4; ++si) {
          const float4* xp = reinterpret_cast<const float4*>(g.x + (size_t)min(si, S - 1) * K + k);
          const float4 a = __ldg(xp), c = __ldg(xp + 1);
          xv[si][0] = a.x; xv[si][1] = a.y; xv[si][2] = a.z; xv[si][3] = a.w;
          xv[si][4] = c.x; xv[si][5] = c.y; xv[si][6] = c.z; xv[si][7] = c.w;
        }
#pragma unroll
        for (int r = 0; r < kBulkRows; ++r) {
          // rows past nr hold stale shared memory; their sums are never stored
          const uint4 wq = *reinterpret_cast<const uint4*>(buf + r * kRowBytes + k * 2);
          float wf[8];
          unpack8(wq, wf);
#pragma unroll
          for (int si = 0; si < 4; ++si)
#pragma unroll
            for (int j = 0; j < 4; ++j)
              ffma2(acc[r][si][0], acc[r][si][1], wf[2 * j], wf[2 * j + 1], xv[si][2 * j], xv[si][2 * j + 1]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kBulkRows; ++r)
#pragma unroll
      for (int si = 0; si < 4; ++si) {
        const float v = warp_sum(acc[r][si][0] + acc[r][si][1]);
        if (lane == 0) part[it & 1][warp][r][si] = v;
      }
    __syncthreads();
    if (abort_sh) break;
    // every thread is done with stage s: it takes the group two steps ahead
    if (t == 0 && gi + 2 * (int)gridDim.x < n_groups) {
      fence_proxy_async_smem();
      issue(gi + 2 * gridDim.x, s);
    }
    if (t < kBulkRows * 4) {
      const int r = t >> 2, si = t & 3;
      if (r < nr && si < S) {
        const float v = part[it & 1][0][r][si] + part[it & 1][1][r][si] + part[it & 1][2][r][si] +
                        part[it & 1][3][r][si] + (bias ? __bfloat162float(bias[o0 + r]) : 0.0f);
        y[(size_t)si * g.y_stride + o0 + r] = ACT == 1 ? silu_f(v) : v;
      }
    }
  }
  if (t == 0 && abort_sh) {
    // stopped early: let the copies still in flight land before the CTA's shared memory goes
    for (int j = it; j < issued; ++j) (void)mbar_wait(&full_bar[j & 1], (uint32_t)(j >> 1) & 1u, g.wait_limit_ns);
  }
}

// ------------------------------------------------------------------ LN + modulate
// Persistent: warp w normalises rows w, w + W, w + 2W, ... (W = warps in the grid, two 128-thread
// blocks per SM).  A row stays in registers as packed bf16 (NV 16-byte chunks per lane) and is
// unpacked once per pass (mean, centred variance, output); the NV loads of the warp's next row
// are issued before the current row is processed, so each warp keeps a row in flight while it
// computes.  shift / scale rows (f32, shared by every row of a sample) come through L1.
template <int NV>
__device__ __forceinline__ void ln_load_row(const LnModArgs& a, int r, int lane, uint4 (&raw)[NV]) {
  const bf16* x = r >= a.n_first ? a.x_second + (size_t)(r - a.n_first) * a.H : a.x_first + (size_t)r * a.H;
#pragma unroll
  for (int i = 0; i < NV; ++i) raw[i] = ld_stream16(reinterpret_cast<const uint4*>(x) + lane + 32 * i);
}

template <int NV>
__device__ __forceinline__ void ln_row(const LnModArgs& a, int r, int lane, const uint4 (&raw)[NV]) {
  const int H = a.H;
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    float v[8];
    unpack8(raw[i], v);
#pragma unroll
    for (int u = 0; u < 8; ++u) s += v[u];
  }
  const float mean = warp_sum(s) / (float)H;
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    float v[8];
    unpack8(raw[i], v);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float d = v[u] - mean;
      q += d * d;
    }
  }
  const float rstd = rsqrtf(warp_sum(q) / (float)H + 1e-6f);
  const int seq = __ldg(a.row_seq + r);
  if (!MF_IDX_OK(seq >= 0 && seq < a.n_seq)) return;
  const float* mrow = a.mod + (size_t)seq * a.seq_stride + (r >= a.n_first ? a.stream_stride : 0);
  const float4* sh = reinterpret_cast<const float4*>(mrow + a.shift_off);
  const float4* sc = reinterpret_cast<const float4*>(mrow + a.scale_off);
  uint4* out = reinterpret_cast<uint4*>(a.out + (size_t)r * H);
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c4 = (lane + 32 * i) * 2;  // float4 index of element 8*(lane+32i)
    const float4 s0 = __ldg(sh + c4), s1 = __ldg(sh + c4 + 1);
    const float4 k0 = __ldg(sc + c4), k1 = __ldg(sc + c4 + 1);
    const float shv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    const float scv[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
    float v[8], o[8];
    unpack8(raw[i], v);
#pragma unroll
    for (int u = 0; u < 8; ++u) o[u] = (v[u] - mean) * rstd * (1.0f + scv[u]) + shv[u];
    uint4 w;
    w.x = pack_bf16x2(o[0], o[1]);
    w.y = pack_bf16x2(o[2], o[3]);
    w.z = pack_bf16x2(o[4], o[5]);
    w.w = pack_bf16x2(o[6], o[7]);
    out[lane + 32 * i] = w;
  }
}

template <int NV>
__global__ void __launch_bounds__(128) ln_modulate_kernel(const LnModArgs a) {
  mf_pdl_enter();
  const int lane = threadIdx.x & 31;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (r >= a.rows) return;
  uint4 cur[NV];
  ln_load_row<NV>(a, r, lane, cur);
  for (;;) {
    const int rn = r + nw;
    uint4 nxt[NV];
    if (rn < a.rows) ln_load_row<NV>(a, rn, lane, nxt);
    ln_row<NV>(a, r, lane, cur);
    if (rn >= a.rows) break;
#pragma unroll
    for (int i = 0; i < NV; ++i) cur[i] = nxt[i];
    r = rn;
  }
}

// ------------------------------------------------------------------ LN + modulate, row groups
// The CTA walks a contiguous range of stream-sorted rows in groups of 8 (per-element arithmetic
// in packed f32x2 pairs).  One thread stages
// each group in shared memory with bulk copies (one per row, plus the group's statistics parts
// when they are given), `stages` groups ahead: a stage is refilled as soon as every thread has
// moved its group into registers, so the copies keep HBM busy while the threads work, and two
// CTAs per SM overlap each other's barriers.  Thread t owns the columns 8t .. 8t + 7 (blockDim.x = H / 8) and keeps their
// shift and 1 + scale in registers while the rows' (sample, stream) stays the same.  A row's
// statistics are (mean, M2 = sum of squared deviations from the mean) merged from parts with
// Chan's pairwise update (Chan, Golub & LeVeque, "Updating formulae and a pairwise algorithm for
// computing sample variances"): for parts (n_a, m_a, M2_a), (n_b, m_b, M2_b) and n = n_a + n_b,
// d = m_b - m_a, m = m_a + d n_b / n, M2 = M2_a + M2_b + d^2 n_a n_b / n.
constexpr int kLnMaxStages = 4;
constexpr int kLnSmemBudget = 100 * 1024;  // per CTA; two CTAs per SM

__device__ __forceinline__ void chan_merge(float& n, float& m, float& m2, float nb, float mb, float m2b) {
  const float tot = n + nb;
  if (nb > 0.0f) {
    const float d = mb - m;
    const float f = nb / tot;
    m = fmaf(d, f, m);
    m2 += m2b + d * d * n * f;
    n = tot;
  }
}

// All lanes end with the merge of every lane's (n, m, m2).
__device__ __forceinline__ void chan_merge_warp(float& n, float& m, float& m2) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float nb = __shfl_xor_sync(0xffffffffu, n, o);
    const float mb = __shfl_xor_sync(0xffffffffu, m, o);
    const float m2b = __shfl_xor_sync(0xffffffffu, m2, o);
    if (n == 0.0f) {
      n = nb; m = mb; m2 = m2b;
    } else {
      chan_merge(n, m, m2, nb, mb, m2b);
    }
  }
}

__device__ __forceinline__ const bf16* ln_row_ptr(const LnModArgs& a, int r) {
  return r >= a.n_first ? a.x_second + (size_t)(r - a.n_first) * a.H : a.x_first + (size_t)r * a.H;
}

// One level of the warp's row-halving merge: a lane keeps half of its R rows (the upper half
// when `up`), receives the partner's values for those rows and merges them (equal counts, cnt
// per side), and sends the other half.
template <int R>
__device__ __forceinline__ void ln_halve(float (&m)[8], float (&q)[8], bool up, int mask, float cnt) {
#pragma unroll
  for (int k = 0; k < R / 2; ++k) {
    const float km = up ? m[k + R / 2] : m[k], kq = up ? q[k + R / 2] : q[k];
    const float sm = up ? m[k] : m[k + R / 2], sq = up ? q[k] : q[k + R / 2];
    const float rm = __shfl_xor_sync(0xffffffffu, sm, mask);
    const float rq = __shfl_xor_sync(0xffffffffu, sq, mask);
    const float d = rm - km;
    m[k] = 0.5f * (km + rm);
    q[k] = kq + rq + d * d * (0.5f * cnt);
  }
}

template <bool kGiven, int kMaxThreads>
__global__ void __launch_bounds__(kMaxThreads, 2) ln_group_kernel(const LnModArgs a, int rows_per_cta, int stages) {
  mf_pdl_enter();
  extern __shared__ __align__(128) uint8_t ln_smem[];
  __shared__ uint64_t full_bar[kLnMaxStages];
  __shared__ float2 part_sh[16][8];  // per warp and group row: (mean, M2) over the warp's 256 columns
  __shared__ float2 row_sh[2][8];    // per group row: (mean, rstd); double-buffered
  __shared__ int abort_sh;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, nwarps = blockDim.x >> 5;
  const int H = a.H, parts = H >> 7;
  const int r_begin = blockIdx.x * rows_per_cta;
  const int r_end = min(a.rows, r_begin + rows_per_cta);
  if (r_begin >= r_end) return;
  const int n_groups = (r_end - r_begin + 7) >> 3;
  const uint32_t row_bytes = (uint32_t)H * 2;
  const uint32_t stage_bytes = 8 * row_bytes + (kGiven ? 8u * parts * 8 : 0u);
  if (t == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(&full_bar[s], 1);
    abort_sh = 0;
    fence_barrier_init();
  }
  __syncthreads();
  int issued = 0;  // thread 0: groups whose copies have been issued
  auto issue = [&](int g) {
    const int s = g % stages, r0 = r_begin + 8 * g, nr = min(8, r_end - r0);
    uint8_t* buf = ln_smem + (size_t)s * stage_bytes;
    mbar_arrive_expect_tx(&full_bar[s], nr * row_bytes + (kGiven ? nr * parts * 8u : 0u));
    for (int i = 0; i < nr; ++i) bulk_load(buf + i * row_bytes, ln_row_ptr(a, r0 + i), row_bytes, &full_bar[s]);
    if constexpr (kGiven) bulk_load(buf + 8 * row_bytes, a.stats + (size_t)r0 * parts, nr * parts * 8u, &full_bar[s]);
    issued = g + 1;
  };
  if (t == 0)
    for (int g = 0; g < min(stages, n_groups); ++g) issue(g);
  int key = -1;  // sample * 2 + stream whose (shift, 1 + scale) are in sh, sc1
  float sh[8], sc1[8];
  int g = 0;
  for (; g < n_groups; ++g) {
    const int s = g % stages, r0 = r_begin + 8 * g, nr = min(8, r_end - r0);
    const uint8_t* buf = ln_smem + (size_t)s * stage_bytes;
    if (!mbar_wait(&full_bar[s], (uint32_t)(g / stages) & 1u, a.wait_limit_ns)) {
      report_status(a.status, kStatusTimeout);
      abort_sh = 1;
    }
    float2* ms = row_sh[g & 1];
    uint4 cur[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) cur[i] = reinterpret_cast<const uint4*>(buf + i * row_bytes)[t];
    if constexpr (kGiven) {
      const float2* st = reinterpret_cast<const float2*>(buf + 8 * row_bytes);
      for (int w = warp; w < nr; w += nwarps) {  // warp w: group row w
        float n = 0.0f, m = 0.0f, m2 = 0.0f;
        if (lane < parts) {
          const float2 v = st[w * parts + lane];
          n = 128.0f; m = v.x; m2 = v.y;
        }
        chan_merge_warp(n, m, m2);
        if (lane == 0) ms[w] = make_float2(m, rsqrtf(m2 / (float)H + 1e-6f));
      }
    } else {
      float m[8], q[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float v[8];
        unpack8(cur[i], v);
        float s0 = v[0], s1 = v[1];
        f32x2_add(s0, s1, v[2], v[3]);
        f32x2_add(s0, s1, v[4], v[5]);
        f32x2_add(s0, s1, v[6], v[7]);
        m[i] = (s0 + s1) * 0.125f;
        float q0 = 0.0f, q1 = 0.0f;
#pragma unroll
        for (int u = 0; u < 8; u += 2) {
          float d0 = v[u], d1 = v[u + 1];
          f32x2_add(d0, d1, -m[i], -m[i]);
          f32x2_fma(d0, d1, d0, d1, q0, q1);  // d * d + q
          q0 = d0;
          q1 = d1;
        }
        q[i] = q0 + q1;
      }
      ln_halve<8>(m, q, (lane & 16) != 0, 16, 8.0f);
      ln_halve<4>(m, q, (lane & 8) != 0, 8, 16.0f);
      ln_halve<2>(m, q, (lane & 4) != 0, 4, 32.0f);
#pragma unroll
      for (int o = 2, cnt = 64; o > 0; o >>= 1, cnt *= 2) {  // the four lanes of one row
        const float rm = __shfl_xor_sync(0xffffffffu, m[0], o);
        const float rq = __shfl_xor_sync(0xffffffffu, q[0], o);
        const float d = rm - m[0];
        m[0] = 0.5f * (m[0] + rm);
        q[0] = q[0] + rq + d * d * (0.5f * (float)cnt);
      }
      if ((lane & 3) == 0)
        part_sh[warp][((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1)] = make_float2(m[0], q[0]);
      __syncthreads();
      for (int w = warp; w < 8; w += nwarps) {  // warp w: group row w
        float n = 0.0f, mm = 0.0f, m2 = 0.0f;
        if (lane < nwarps) {
          const float2 v = part_sh[lane][w];
          n = 256.0f; mm = v.x; m2 = v.y;
        }
        chan_merge_warp(n, mm, m2);
        if (lane == 0) ms[w] = make_float2(mm, rsqrtf(m2 / (float)H + 1e-6f));
      }
    }
    __syncthreads();
    if (abort_sh) break;
    // every thread holds group g in registers, so its stage can take group g + stages
    if (t == 0 && g + stages < n_groups) {
      fence_proxy_async_smem();
      issue(g + stages);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i >= nr) break;
      const int r = r0 + i;
      const int st = r >= a.n_first ? 1 : 0;
      const int seq = __ldg(a.row_seq + r);
      if (!MF_IDX_OK(seq >= 0 && seq < a.n_seq)) break;
      if (seq * 2 + st != key) {
        key = seq * 2 + st;
        const float* mrow = a.mod + (size_t)seq * a.seq_stride + (st ? a.stream_stride : 0);
        const float4* shp = reinterpret_cast<const float4*>(mrow + a.shift_off) + 2 * t;
        const float4* scp = reinterpret_cast<const float4*>(mrow + a.scale_off) + 2 * t;
        const float4 s0 = __ldg(shp), s1 = __ldg(shp + 1), k0 = __ldg(scp), k1 = __ldg(scp + 1);
        sh[0] = s0.x; sh[1] = s0.y; sh[2] = s0.z; sh[3] = s0.w; sh[4] = s1.x; sh[5] = s1.y; sh[6] = s1.z; sh[7] = s1.w;
        sc1[0] = 1.0f + k0.x; sc1[1] = 1.0f + k0.y; sc1[2] = 1.0f + k0.z; sc1[3] = 1.0f + k0.w;
        sc1[4] = 1.0f + k1.x; sc1[5] = 1.0f + k1.y; sc1[6] = 1.0f + k1.z; sc1[7] = 1.0f + k1.w;
      }
      const float2 mr = ms[i];                  // (mean, rstd)
      const float nmr = -mr.x * mr.y;
      float v[8];
      unpack8(cur[i], v);
#pragma unroll
      for (int u = 0; u < 8; u += 2) {
        f32x2_fma_s(v[u], v[u + 1], mr.y, nmr);                            // (x - mean) rstd
        f32x2_fma(v[u], v[u + 1], sc1[u], sc1[u + 1], sh[u], sh[u + 1]);  // ... (1 + scale) + shift
      }
      uint4 w;
      w.x = pack_bf16x2(v[0], v[1]);
      w.y = pack_bf16x2(v[2], v[3]);
      w.z = pack_bf16x2(v[4], v[5]);
      w.w = pack_bf16x2(v[6], v[7]);
      reinterpret_cast<uint4*>(a.out + (size_t)r * H)[t] = w;
    }
  }
  if (t == 0 && g < n_groups) {
    // stopped early: let the copies still in flight land before the CTA's shared memory goes
    for (int gg = g; gg < issued; ++gg)
      (void)mbar_wait(&full_bar[gg % stages], (uint32_t)(gg / stages) & 1u, a.wait_limit_ns);
  }
}

// ------------------------------------------------------------------ fp8 quantisation
// One warp per row; lane l takes the 16-element chunks l, l + 32, ...  Pass 1 finds the row's
// largest magnitude, pass 2 (the row again, now from L1 / L2) divides and converts.
__global__ void __launch_bounds__(128) quantize_e4m3_rows_kernel(const bf16* __restrict__ x, int M, int K,
                                                                 uint8_t* __restrict__ q,
                                                                 float* __restrict__ s) {
  mf_pdl_enter();
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= M) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)r * K);
  const int nch = K / 16;
  float amax = 0.0f;
  for (int c = lane; c < nch; c += 32) {
    const uint4 a = __ldg(xr + 2 * c), b = __ldg(xr + 2 * c + 1);
    float v[16];
    unpack8(a, *reinterpret_cast<float(*)[8]>(v));
    unpack8(b, *reinterpret_cast<float(*)[8]>(v + 8));
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float sc = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  uint4* qr = reinterpret_cast<uint4*>(q + (size_t)r * K);
  for (int c = lane; c < nch; c += 32) {
    const uint4 a = __ldg(xr + 2 * c), b = __ldg(xr + 2 * c + 1);
    float v[16];
    unpack8(a, *reinterpret_cast<float(*)[8]>(v));
    unpack8(b, *reinterpret_cast<float(*)[8]>(v + 8));
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = pack_e4m3x2(__fdiv_rn(v[4 * i], sc), __fdiv_rn(v[4 * i + 1], sc));
      const uint32_t hi = pack_e4m3x2(__fdiv_rn(v[4 * i + 2], sc), __fdiv_rn(v[4 * i + 3], sc));
      w[i] = lo | (hi << 16);
    }
    qr[c] = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (lane == 0) s[r] = sc;
}

// ------------------------------------------------------------------ rectified-flow epilogues
__global__ void interpolate_kernel(const int* __restrict__ img_seq, const int* __restrict__ img_target,
                                   const float* __restrict__ t, int Ni, int C,
                                   const float* __restrict__ z, const float* __restrict__ eps,
                                   float* __restrict__ zt, bf16* __restrict__ zt_bf16) {
  mf_pdl_enter();
  const long long n4 = (long long)Ni * C / 4;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(i * 4 / C);
    const float4 a = reinterpret_cast<const float4*>(z)[i];
    float4 o = a;
    if (__ldg(img_target + r)) {
      const float tt = __ldg(t + __ldg(img_seq + r));
      const float4 e = reinterpret_cast<const float4*>(eps)[i];
      const float u = 1.0f - tt;
      o = make_float4(u * a.x + tt * e.x, u * a.y + tt * e.y, u * a.z + tt * e.z, u * a.w + tt * e.w);
    }
    if (zt) reinterpret_cast<float4*>(zt)[i] = o;
    if (zt_bf16) {
      uint2 w;
      w.x = pack_bf16x2(o.x, o.y);
      w.y = pack_bf16x2(o.z, o.w);
      reinterpret_cast<uint2*>(zt_bf16)[i] = w;
    }
  }
}

// Each conditional row writes the guided velocity to itself and to its unconditional partner,
// so in-place use is race-free (unconditional rows are only written by their partner).
__global__ void cfg_kernel(const int* __restrict__ img_seq, const int* __restrict__ seq_role,
                           const int* __restrict__ img_pair, int Ni, int C, float w,
                           const float* v, float* out) {
  mf_pdl_enter();
  const long long n4 = (long long)Ni * C / 4;
  const int c4n = C / 4;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(i / c4n);
    const int c4 = (int)(i - (long long)r * c4n);
    const int role = __ldg(seq_role + __ldg(img_seq + r));
    if (role == 0) {
      if (out != v) reinterpret_cast<float4*>(out)[i] = reinterpret_cast<const float4*>(v)[i];
    } else if (role == 1) {
      const int u = __ldg(img_pair + r);
      if (!MF_IDX_OK(u >= 0 && u < Ni)) continue;
      const long long j = (long long)u * c4n + c4;
      const float4 vc = reinterpret_cast<const float4*>(v)[i];
      const float4 vu = reinterpret_cast<const float4*>(v)[j];
      const float4 g = make_float4(vu.x + w * (vc.x - vu.x), vu.y + w * (vc.y - vu.y),
                                   vu.z + w * (vc.z - vu.z), vu.w + w * (vc.w - vu.w));
      reinterpret_cast<float4*>(out)[i] = g;
      reinterpret_cast<float4*>(out)[j] = g;
    }
  }
}

__global__ void euler_kernel(long long n4, float dt, const float* __restrict__ v, float* z,
                             bf16* __restrict__ z_bf16) {
  mf_pdl_enter();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(v)[i];
    float4 b = reinterpret_cast<float4*>(z)[i];
    b.x = fmaf(dt, a.x, b.x);
    b.y = fmaf(dt, a.y, b.y);
    b.z = fmaf(dt, a.z, b.z);
    b.w = fmaf(dt, a.w, b.w);
    reinterpret_cast<float4*>(z)[i] = b;
    if (z_bf16) {
      uint2 w;
      w.x = pack_bf16x2(b.x, b.y);
      w.y = pack_bf16x2(b.z, b.w);
      reinterpret_cast<uint2*>(z_bf16)[i] = w;
    }
  }
}

// Exact f32 building blocks for the loss rows (the FP64 pipe of this GPU is far narrower than
// its f32 pipe): Knuth's TwoSum (s + t = a + b exactly) and, with an FMA, the exact square
// (p + e = x * x).  A row's sum is carried as an unevaluated pair hi + lo of f32 values.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& t) {
  s = a + b;
  const float bb = s - a;
  t = (a - (s - bb)) + (b - bb);
}

// hi + lo += d^2 for d = u - (a - e): a - e = s + t and u - s = s2 + t2 exactly, so
// d = s2 + (t2 - t) with the second term rounded once (to 2^-24 of itself); s2^2 is split
// exactly and the cross and square terms of the small part are added with FMAs.
__device__ __forceinline__ void acc_sq_diff(float u, float a, float e, float& hi, float& lo) {
  float s, t, s2, t2;
  two_sum(a, -e, s, t);
  two_sum(u, -s, s2, t2);
  const float dl = t2 - t;
  const float p = s2 * s2;
  const float pe = fmaf(s2, s2, -p);
  const float c = fmaf(dl, dl, fmaf(2.0f * s2, dl, pe));
  float h, ht;
  two_sum(hi, p, h, ht);
  hi = h;
  lo += ht + c;
}

// per image row: sum over channels of (v - (z - eps))^2 (0 for source-frame rows), one warp per
// row, carried to within about 2^-44 of the row sum and stored as an f64
__global__ void loss_row_kernel(const int* __restrict__ img_target, int Ni, int C,
                                const float* __restrict__ z, const float* __restrict__ eps,
                                const float* __restrict__ v, double* __restrict__ ws) {
  mf_pdl_enter();
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= Ni) return;
  float hi = 0.0f, lo = 0.0f;
  if (__ldg(img_target + r)) {
    const size_t base = (size_t)r * C;
    for (int c = lane * 4; c < C; c += 128) {
      const float4 a = *reinterpret_cast<const float4*>(z + base + c);
      const float4 e = *reinterpret_cast<const float4*>(eps + base + c);
      const float4 u = *reinterpret_cast<const float4*>(v + base + c);
      acc_sq_diff(u.x, a.x, e.x, hi, lo);
      acc_sq_diff(u.y, a.y, e.y, hi, lo);
      acc_sq_diff(u.z, a.z, e.z, hi, lo);
      acc_sq_diff(u.w, a.w, e.w, hi, lo);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ho = __shfl_xor_sync(0xffffffffu, hi, o), lo2 = __shfl_xor_sync(0xffffffffu, lo, o);
    float h, t;
    two_sum(hi, ho, h, t);
    hi = h;
    lo += lo2 + t;
  }
  if (lane == 0) ws[r] = (double)hi + (double)lo;
}

// Diffusion-NFT objective, per image row: sum over channels of
// r (v+ - (z - eps))^2 + (1 - r) (v- - (z - eps))^2 in f64 with the row's sample's reward r
// (0 for source-frame rows).  The per-sample sums then take the flow loss's reductions.
__global__ void nft_row_kernel(const int* __restrict__ img_seq, const int* __restrict__ img_target,
                               const float* __restrict__ reward, int Ni, int C,
                               const float* __restrict__ z, const float* __restrict__ eps,
                               const float* __restrict__ vp, const float* __restrict__ vn,
                               double* __restrict__ ws) {
  mf_pdl_enter();
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= Ni) return;
  double acc = 0.0;
  if (__ldg(img_target + r)) {
    const double w = (double)__ldg(reward + __ldg(img_seq + r));
    const size_t base = (size_t)r * C;
    double sp = 0.0, sn = 0.0;
    for (int c = lane * 4; c < C; c += 128) {
      const float4 a = *reinterpret_cast<const float4*>(z + base + c);
      const float4 e = *reinterpret_cast<const float4*>(eps + base + c);
      const float4 p = *reinterpret_cast<const float4*>(vp + base + c);
      const float4 n = *reinterpret_cast<const float4*>(vn + base + c);
      const double t0 = (double)a.x - (double)e.x, t1 = (double)a.y - (double)e.y;
      const double t2 = (double)a.z - (double)e.z, t3 = (double)a.w - (double)e.w;
      const double p0 = (double)p.x - t0, p1 = (double)p.y - t1, p2 = (double)p.z - t2, p3 = (double)p.w - t3;
      const double n0 = (double)n.x - t0, n1 = (double)n.y - t1, n2 = (double)n.z - t2, n3 = (double)n.w - t3;
      sp += p0 * p0 + p1 * p1 + p2 * p2 + p3 * p3;
      sn += n0 * n0 + n1 * n1 + n2 * n2 + n3 * n3;
    }
    acc = w * sp + (1.0 - w) * sn;
  }
  acc = warp_sum_d(acc);
  if (lane == 0) ws[r] = acc;
}

// one block of 1024 threads per sample (four rows in flight each), fixed reduction order
__global__ void loss_seq_kernel(const int* __restrict__ cu_img, const int* __restrict__ img_target,
                                int C, const double* __restrict__ ws, double* __restrict__ loss_sum,
                                long long* __restrict__ count) {
  mf_pdl_enter();
  __shared__ double sd[1024];
  __shared__ long long sc[1024];
  const int s = blockIdx.x;
  const int lo = cu_img[s], hi = cu_img[s + 1];
  const int bd = blockDim.x;
  double a0 = 0.0, a1 = 0.0, a2 = 0.0, a3 = 0.0;  // four loads in flight per step
  long long n = 0;
  int r = lo + threadIdx.x;
  for (; r + 3 * bd < hi; r += 4 * bd) {
    a0 += ws[r];
    a1 += ws[r + bd];
    a2 += ws[r + 2 * bd];
    a3 += ws[r + 3 * bd];
    n += img_target[r] + img_target[r + bd] + img_target[r + 2 * bd] + img_target[r + 3 * bd];
  }
  for (; r < hi; r += bd) {
    a0 += ws[r];
    n += img_target[r];
  }
  sd[threadIdx.x] = (a0 + a1) + (a2 + a3);
  sc[threadIdx.x] = n;
  __syncthreads();
  for (int o = blockDim.x / 2; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o) {
      sd[threadIdx.x] += sd[threadIdx.x + o];
      sc[threadIdx.x] += sc[threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    loss_sum[s] = sd[0];
    count[s] = sc[0] * (long long)C;
  }
}

__global__ void loss_mean_kernel(int S, const double* __restrict__ loss_sum,
                                 const long long* __restrict__ count, double* __restrict__ mean) {
  mf_pdl_enter();
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  double a = 0.0;
  long long n = 0;
  for (int s = 0; s < S; ++s) {
    a += loss_sum[s];
    n += count[s];
  }
  *mean = n > 0 ? a / (double)n : 0.0;
}

__global__ void timeout_selftest_kernel(unsigned* status, unsigned long long limit_ns) {
  mf_pdl_enter();
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // nobody arrives on `bar`: the bounded wait must give up and report
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit_ns)) report_status(status, kStatusTimeout);
}

int grid_for(long long n, int threads) {
  long long g = (n + threads - 1) / threads;
  if (g > 148LL * 16) g = 148LL * 16;
  return g < 1 ? 1 : (int)g;
}

}  // namespace

cudaError_t launch_sinusoid(const float* t, int S, int F, float* out, cudaStream_t st) {
  const int n = S * (F / 2);
  if (n <= 0) return cudaSuccess;
  launch_k(sinusoid_kernel, (n + 255) / 256, 256, 0, st, t, S, F, out);
  return cudaGetLastError();
}

namespace {
// One launch per group of four samples; gridDim.y = number of problems.
cudaError_t gemv_groups(GemvArgs g, int np, int K, int act, const float* x, float* y, int S,
                        cudaStream_t st, int* launches) {
  if (launches) *launches = 0;
  if (S <= 0 || g.O <= 0) return cudaSuccess;
  const int warps = (g.O + kGemvRows - 1) / kGemvRows;
  const dim3 grid((warps + 3) / 4, np);
  const int nch = K % 256 == 0 ? K / 256 : 0;
  if (nch >= 4 && nch <= 16) {  // wide K: the bulk-copy kernel
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int n_groups = (g.O + kBulkRows - 1) / kBulkRows;
    const int per_problem = std::max(1, std::min(n_groups, 2 * sms / np));
    const dim3 bgrid(per_problem, np);
    const size_t smem = 2 * (size_t)kBulkRows * K * 2;
    for (int s0 = 0; s0 < S; s0 += 4) {
      g.S = S - s0 < 4 ? S - s0 : 4;
      g.x = x + (size_t)s0 * K;
      g.y = y + (size_t)s0 * g.y_stride;
      switch (nch * 2 + (act == 1 ? 1 : 0)) {
#define MF_GEMV_BULK_CASE(n)                                                                           \
  case 2 * n:                                                                                         \
    e = cudaFuncSetAttribute(gemv_bulk_kernel<0, n>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
    if (e == cudaSuccess) e = launch_k(gemv_bulk_kernel<0, n>, bgrid, 128, smem, st, g, n_groups);   \
    break;                                                                                            \
  case 2 * n + 1:                                                                                     \
    e = cudaFuncSetAttribute(gemv_bulk_kernel<1, n>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
    if (e == cudaSuccess) e = launch_k(gemv_bulk_kernel<1, n>, bgrid, 128, smem, st, g, n_groups);   \
    break;
        MF_GEMV_BULK_CASE(4) MF_GEMV_BULK_CASE(5) MF_GEMV_BULK_CASE(6) MF_GEMV_BULK_CASE(7)
        MF_GEMV_BULK_CASE(8) MF_GEMV_BULK_CASE(9) MF_GEMV_BULK_CASE(10) MF_GEMV_BULK_CASE(11)
        MF_GEMV_BULK_CASE(12) MF_GEMV_BULK_CASE(13) MF_GEMV_BULK_CASE(14) MF_GEMV_BULK_CASE(15)
        MF_GEMV_BULK_CASE(16)
#undef MF_GEMV_BULK_CASE
        default: return cudaErrorInvalidValue;
      }
      if (e != cudaSuccess) return e;
      if (launches) ++*launches;
    }
    return cudaGetLastError();
  }
  for (int s0 = 0; s0 < S; s0 += 4) {
    g.S = S - s0 < 4 ? S - s0 : 4;
    g.x = x + (size_t)s0 * K;
    g.y = y + (size_t)s0 * g.y_stride;
    switch (nch * 2 + (act == 1 ? 1 : 0)) {
#define MF_GEMV_CASE(n)                                 \
  case 2 * n:                                          \
    launch_k(gemv_kernel<0, n>, grid, 128, 0, st, g);        \
    break;                                             \
  case 2 * n + 1:                                      \
    launch_k(gemv_kernel<1, n>, grid, 128, 0, st, g);        \
    break;
      MF_GEMV_CASE(1) MF_GEMV_CASE(2) MF_GEMV_CASE(3) MF_GEMV_CASE(4) MF_GEMV_CASE(5) MF_GEMV_CASE(6)
      MF_GEMV_CASE(7) MF_GEMV_CASE(8) MF_GEMV_CASE(9) MF_GEMV_CASE(10) MF_GEMV_CASE(11) MF_GEMV_CASE(12)
      MF_GEMV_CASE(13) MF_GEMV_CASE(14) MF_GEMV_CASE(15) MF_GEMV_CASE(16)
#undef MF_GEMV_CASE
      default: return cudaErrorInvalidValue;  // K must be a multiple of 256, at most 4096
    }
    if (launches) ++*launches;
  }
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_gemv(const bf16* W, const bf16* b, const float* x, int S, int K, int O, float* y,
                        int y_stride, int y_off, int act, unsigned* status, unsigned long long wait_limit_ns,
                        cudaStream_t st, int* launches) {
  GemvArgs g{{W, W}, {b, b}, {y_off, y_off}, x, 0, O, y, y_stride, status, wait_limit_ns};
  return gemv_groups(g, 1, K, act, x, y, S, st, launches);
}

cudaError_t launch_gemv2(const bf16* W0, const bf16* b0, int y_off0, const bf16* W1, const bf16* b1,
                         int y_off1, const float* x, int S, int K, int O, float* y, int y_stride,
                         unsigned* status, unsigned long long wait_limit_ns, cudaStream_t st, int* launches) {
  GemvArgs g{{W0, W1}, {b0, b1}, {y_off0, y_off1}, x, 0, O, y, y_stride, status, wait_limit_ns};
  return gemv_groups(g, 2, K, 0, x, y, S, st, launches);
}

cudaError_t launch_quantize_e4m3_rows(const bf16* x, int M, int K, uint8_t* q, float* s, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  if (K <= 0 || K % 16 != 0) return cudaErrorInvalidValue;
  launch_k(quantize_e4m3_rows_kernel, (M + 3) / 4, 128, 0, st, x, M, K, q, s);
  return cudaGetLastError();
}

cudaError_t launch_ln_modulate(const LnModArgs& a, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int blocks = std::min((a.rows + 3) / 4, 2 * sms);  // two resident blocks per SM
  switch (a.H / 256) {
#define MF_LN_CASE(nv) \
  case nv: launch_k(ln_modulate_kernel<nv>, blocks, 128, 0, st, a); break;
    MF_LN_CASE(1) MF_LN_CASE(2) MF_LN_CASE(3) MF_LN_CASE(4) MF_LN_CASE(5) MF_LN_CASE(6)
    MF_LN_CASE(7) MF_LN_CASE(8) MF_LN_CASE(9) MF_LN_CASE(10) MF_LN_CASE(11) MF_LN_CASE(12)
    MF_LN_CASE(13) MF_LN_CASE(14) MF_LN_CASE(15) MF_LN_CASE(16)
#undef MF_LN_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <bool kGiven, int kMaxThreads>
cudaError_t launch_ln_group_t(const LnModArgs& a, int sms, cudaStream_t st) {
  const int stage_bytes = 8 * a.H * 2 + (kGiven ? 8 * (a.H / 128) * 8 : 0);
  const int stages = std::min(kLnMaxStages, kLnSmemBudget / stage_bytes);
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(ln_group_kernel<kGiven, kMaxThreads>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kLnSmemBudget);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // two CTAs per SM (shared memory), contiguous row ranges of a multiple of 8 rows
  const int ctas = 2 * sms;
  int per_cta = (a.rows + ctas - 1) / ctas;
  per_cta = (per_cta + 7) / 8 * 8;
  const int grid = (a.rows + per_cta - 1) / per_cta;
  launch_k(ln_group_kernel<kGiven, kMaxThreads>, grid, a.H / 8, stages * stage_bytes, st, a, per_cta, stages);
  return cudaGetLastError();
}

cudaError_t launch_ln_group(const LnModArgs& a, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  if (a.H % 256 != 0 || a.H > 4096) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (a.H <= 3072)
    return a.stats ? launch_ln_group_t<true, 384>(a, sms, st) : launch_ln_group_t<false, 384>(a, sms, st);
  return a.stats ? launch_ln_group_t<true, 512>(a, sms, st) : launch_ln_group_t<false, 512>(a, sms, st);
}

cudaError_t launch_interpolate(const int* img_seq, const int* img_target, const float* t, int Ni,
                               int C, const float* z, const float* eps, float* zt, bf16* zt_bf16,
                               cudaStream_t st) {
  const long long n4 = (long long)Ni * C / 4;
  if (n4 <= 0) return cudaSuccess;
  launch_k(interpolate_kernel, grid_for(n4, 256), 256, 0, st, img_seq, img_target, t, Ni, C, z, eps, zt,
                                                        zt_bf16);
  return cudaGetLastError();
}

cudaError_t launch_cfg(const int* img_seq, const int* seq_role, const int* img_pair, int Ni, int C,
                       float w, const float* v, float* out, cudaStream_t st) {
  const long long n4 = (long long)Ni * C / 4;
  if (n4 <= 0) return cudaSuccess;
  launch_k(cfg_kernel, grid_for(n4, 256), 256, 0, st, img_seq, seq_role, img_pair, Ni, C, w, v, out);
  return cudaGetLastError();
}

cudaError_t launch_euler(int Ni, int C, float dt, const float* v, float* z, bf16* z_bf16,
                         cudaStream_t st) {
  const long long n4 = (long long)Ni * C / 4;
  if (n4 <= 0) return cudaSuccess;
  launch_k(euler_kernel, grid_for(n4, 256), 256, 0, st, n4, dt, v, z, z_bf16);
  return cudaGetLastError();
}

cudaError_t launch_flow_loss(const int* cu_img, const int* img_target, int S, int Ni, int C,
                             const float* z, const float* eps, const float* v, double* ws,
                             double* loss_sum, long long* count, double* mean, cudaStream_t st) {
  if (Ni > 0) launch_k(loss_row_kernel, (Ni + 7) / 8, 256, 0, st, img_target, Ni, C, z, eps, v, ws);
  if (S > 0) launch_k(loss_seq_kernel, S, 1024, 0, st, cu_img, img_target, C, ws, loss_sum, count);
  launch_k(loss_mean_kernel, 1, 32, 0, st, S, loss_sum, count, mean);
  return cudaGetLastError();
}

cudaError_t launch_nft_loss(const int* cu_img, const int* img_seq, const int* img_target,
                            const float* reward, int S, int Ni, int C, const float* z,
                            const float* eps, const float* vp, const float* vn, double* ws,
                            double* loss_sum, long long* count, double* mean, cudaStream_t st) {
  if (Ni > 0)
    launch_k(nft_row_kernel, (Ni + 7) / 8, 256, 0, st, img_seq, img_target, reward, Ni, C, z, eps, vp, vn, ws);
  if (S > 0) launch_k(loss_seq_kernel, S, 1024, 0, st, cu_img, img_target, C, ws, loss_sum, count);
  launch_k(loss_mean_kernel, 1, 32, 0, st, S, loss_sum, count, mean);
  return cudaGetLastError();
}

cudaError_t launch_timeout_selftest(unsigned* status, unsigned long long limit_ns, cudaStream_t st) {
  launch_k(timeout_selftest_kernel, 1, 32, 0, st, status, limit_ns);
  return cudaGetLastError();
}

MF_BOUNDS_EXPORT(pointwise)

}  // namespace mf
