// Persistent grouped GEMMs for sm_103a: TMA (128-byte swizzle) -> shared-memory ring ->
// tcgen05.mma (f32 accumulators in TMEM, two accumulator buffers so the epilogue of one tile
// overlaps the main loop of the next) -> tcgen05.ld epilogue warps.
//
// Two kernels.  gemm_kernel (single CTA, 128-row tiles, 192 threads: warp 0 TMA producer,
// warp 1 TMEM allocator and MMA issuer, warps 2..5 epilogue) serves the narrow final projection
// and small plain GEMMs.  gemm_pair_kernel (clusters of two CTAs, 256 x 256 tiles with
// tcgen05.mma.cta_group::2, 320 threads: warp 0 producer, warp 1 MMA issuer of the even CTA,
// warps 2..9 epilogue) serves every 256-wide projection of the block; its kEpiF8 flag switches
// the operands to E4M3 (kind::f8f6f4) with per-row and per-column scales in the epilogue.
//
// The fused epilogues implement the NR-MMDiT chains that the Mage-Flow pages list as fused
// memory-bound work - norm, RoPE, gating, residual (PaperReading review of "Mage-Flow: An
// Efficient Native-Resolution Foundation Model for Image Generation and Editing", §2.2 (3);
// hyper.ai summary, 方法): bias, RoPE over (frame, row, col) with the scatter to joint order
// (and the optional per-head QK-RMSNorm), GELU, and the gated residual x += gate * y.
#include "gemm.cuh"

namespace mf {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;

// Tile order, chosen per problem on the host (GemmParams::group_m):
//  * group_m == 0, N fastest: for few N tiles (out-proj, MLP-down).  The tiles running at the
//    same time cover every N tile of a few row panels, so each A k-slice serves all of them
//    from L2 and the weight matrix stays resident in L2 from one row panel to the next.
//  * group_m > 0: group_m row tiles fastest, then N (QKV, MLP-up).  With many N tiles the
//    wide output streaming through L2 would evict a resident weight matrix; sweeping N for a
//    fixed group of row panels keeps those A panels in L2 instead.
__device__ __forceinline__ void decode_tile(const GemmParams& p, int tile, int& pi, int& m,
                                            int& n) {
  pi = (p.n_prob > 1 && tile >= p.tile_begin[1]) ? 1 : 0;
  const int t = tile - p.tile_begin[pi];
  const int tn = p.tiles_n[pi], tm = p.tiles_m[pi];
  const int gmax = p.group_m[pi];
  if (gmax == 0) {
    m = t / tn;
    n = t - m * tn;
    return;
  }
  const int group = t / (gmax * tn);
  const int first_m = group * gmax;
  const int gm = min(gmax, tm - first_m);
  const int local = t - group * gmax * tn;
  m = first_m + local % gm;
  n = local / gm;
}

__device__ __forceinline__ void load_bias32(const bf16* bias, int col0, float (&v)[32]) {
  if (bias == nullptr) return;
  const uint4* b = reinterpret_cast<const uint4*>(bias + col0);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 u = __ldg(b + i);
    float2 f0 = unpack_bf16x2(u.x), f1 = unpack_bf16x2(u.y), f2 = unpack_bf16x2(u.z),
           f3 = unpack_bf16x2(u.w);
    v[8 * i + 0] += f0.x; v[8 * i + 1] += f0.y; v[8 * i + 2] += f1.x; v[8 * i + 3] += f1.y;
    v[8 * i + 4] += f2.x; v[8 * i + 5] += f2.y; v[8 * i + 6] += f3.x; v[8 * i + 7] += f3.y;
  }
}

__device__ __forceinline__ void store_bf16x32(bf16* dst, const float (&v)[32]) {
  uint4* o = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 u;
    u.x = pack_bf16x2(v[8 * i + 0], v[8 * i + 1]);
    u.y = pack_bf16x2(v[8 * i + 2], v[8 * i + 3]);
    u.z = pack_bf16x2(v[8 * i + 4], v[8 * i + 5]);
    u.w = pack_bf16x2(v[8 * i + 6], v[8 * i + 7]);
    o[i] = u;
  }
}

template <int EPI>
__device__ __forceinline__ void epilogue_chunk(const GemmParams& p, const GemmProblem& pr,
                                               int row, int col0, const uint32_t (&r)[32],
                                               const float* rope_inv, const int* rope_axis) {
  if (row >= pr.M || col0 >= pr.N) return;
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
  load_bias32(pr.bias, col0, v);

  if constexpr (EPI == kEpiBiasBf16 || EPI == kEpiGelu) {
    if constexpr (EPI == kEpiGelu) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.5f * v[i] * (1.0f + erff(v[i] * 0.7071067811865476f));
    }
    store_bf16x32(static_cast<bf16*>(pr.out) + (size_t)row * pr.ldo + col0, v);
  } else if constexpr (EPI == kEpiBiasF32) {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(pr.out) + (size_t)row * pr.ldo + col0);
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else if constexpr (EPI == kEpiGateResid) {
    const int srow = pr.row_off + row;
    const int seq = __ldg(p.srow_seq + srow);
    if (!MF_IDX_OK(seq >= 0 && seq < p.n_seq)) return;
    const float4* g = reinterpret_cast<const float4*>(
        p.mod + ((size_t)seq * 2 + pr.stream) * 6 * (size_t)p.H + p.gate_off + col0);
    bf16* x = static_cast<bf16*>(pr.out) + (size_t)row * pr.ldo + col0;
    uint4* xv = reinterpret_cast<uint4*>(x);
    float out[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 u = xv[i];
      float4 ga = __ldg(g + 2 * i), gb = __ldg(g + 2 * i + 1);
      float2 x0 = unpack_bf16x2(u.x), x1 = unpack_bf16x2(u.y), x2 = unpack_bf16x2(u.z),
             x3 = unpack_bf16x2(u.w);
      out[8 * i + 0] = fmaf(ga.x, v[8 * i + 0], x0.x);
      out[8 * i + 1] = fmaf(ga.y, v[8 * i + 1], x0.y);
      out[8 * i + 2] = fmaf(ga.z, v[8 * i + 2], x1.x);
      out[8 * i + 3] = fmaf(ga.w, v[8 * i + 3], x1.y);
      out[8 * i + 4] = fmaf(gb.x, v[8 * i + 4], x2.x);
      out[8 * i + 5] = fmaf(gb.y, v[8 * i + 5], x2.y);
      out[8 * i + 6] = fmaf(gb.z, v[8 * i + 6], x3.x);
      out[8 * i + 7] = fmaf(gb.w, v[8 * i + 7], x3.y);
    }
    store_bf16x32(x, out);
  } else if constexpr (EPI == kEpiQkvRope) {
    const int srow = pr.row_off + row;
    const int joint = __ldg(p.srow_joint + srow);
    if (!MF_IDX_OK(joint >= 0 && joint < p.n_tok)) return;
    const int which = col0 / p.H;
    const int cc = col0 - which * p.H;
    bf16* dst = (which == 0 ? p.q : (which == 1 ? p.k : p.v)) + (size_t)joint * p.H + cc;
    if (which < 2) {
      const int* ps = p.pos + (size_t)joint * 3;
      const float pf = (float)__ldg(ps), pr_ = (float)__ldg(ps + 1), pc = (float)__ldg(ps + 2);
      const int g0 = (cc % p.head_dim) >> 1;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int ax = rope_axis[g0 + i];
        const float th = (ax == 0 ? pf : (ax == 1 ? pr_ : pc)) * rope_inv[g0 + i];
        // |th| <= max position (< 2^10): reduce modulo 2 pi with a two-constant Cody-Waite
        // step (2 pi = kHi + kLo), then the hardware sine / cosine on [-pi, pi]
        const float kq = rintf(th * 0.15915494309189535f);
        const float rr = fmaf(-kq, -1.7484555314695172e-07f, fmaf(-kq, 6.2831854820251465f, th));
        float s, c;
        __sincosf(rr, &s, &c);
        const float x0 = v[2 * i], x1 = v[2 * i + 1];
        v[2 * i] = x0 * c - x1 * s;
        v[2 * i + 1] = x0 * s + x1 * c;
      }
    }
    store_bf16x32(dst, v);
  }
}

// ---------------------------------------------------------------------------------------
// Staged epilogue of the CTA-pair kernel.  A warp owns 32 accumulator rows (its TMEM lane
// quarter) and moves them 16 columns at a time.  Phase 1, one thread per row: bias, then GELU
// or RoPE, in f32, written to the warp's staging rows in shared memory.  Phase 2, two threads
// per row, 8 columns each: the last operation (gated residual, scatter to joint order) and the
// global store, so each store instruction writes whole 32-byte sectors of 16 rows instead of
// 16 bytes of 32 rows (stores of that shape held back the tensor core's issue).
constexpr float kQkNormEps = 1e-6f;  // QK-RMSNorm epsilon (inside the root)
constexpr int kStageRow = 20;  // floats per staged row (16 + 4 padding: conflict-free 16-byte writes)

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_reg_fence16(uint32_t (&r)[16]) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
               "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
               "+r"(r[14]), "+r"(r[15]));
}

// v[i] += bias[col0 + i], i < 16 (no-op without a bias).
__device__ __forceinline__ void add_bias16(const GemmProblem& pr, int col0, float (&v)[16]) {
  if (pr.bias == nullptr) return;
  const uint4* b = reinterpret_cast<const uint4*>(pr.bias + col0);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 u = __ldg(b + i);
    const float2 f0 = unpack_bf16x2(u.x), f1 = unpack_bf16x2(u.y), f2 = unpack_bf16x2(u.z),
                 f3 = unpack_bf16x2(u.w);
    v[8 * i + 0] += f0.x; v[8 * i + 1] += f0.y; v[8 * i + 2] += f1.x; v[8 * i + 3] += f1.y;
    v[8 * i + 4] += f2.x; v[8 * i + 5] += f2.y; v[8 * i + 6] += f3.x; v[8 * i + 7] += f3.y;
  }
}

// Phase 1: 16 columns of one row, in place.  For the QKV epilogue with QK-RMSNorm, qk_g is the
// stream's scale vector of this part (q or k) and qk_rstd the row's 1 / RMS over the head of
// these columns; the norm is applied after the bias and before RoPE.
template <int EPI>
__device__ __forceinline__ void epi_row16(const GemmParams& p, const GemmProblem& pr, int row, int col0,
                                          float (&v)[16], const float* rope_inv, const int* rope_axis,
                                          const bf16* qk_g = nullptr, float qk_rstd = 0.0f) {
  constexpr int E = EPI & 7;
  if (row >= pr.M || col0 >= pr.N) return;
  if constexpr ((EPI & kEpiF8) != 0) {
    const float rs = __ldg(p.row_scale + pr.row_off + row);
    const float4* cs = reinterpret_cast<const float4*>(pr.col_scale + col0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 c = __ldg(cs + i);
      v[4 * i + 0] = v[4 * i + 0] * rs * c.x;
      v[4 * i + 1] = v[4 * i + 1] * rs * c.y;
      v[4 * i + 2] = v[4 * i + 2] * rs * c.z;
      v[4 * i + 3] = v[4 * i + 3] * rs * c.w;
    }
  }
  add_bias16(pr, col0, v);
  if constexpr (E == kEpiGelu) {
    if constexpr ((EPI & kEpiSave) != 0) {  // the pre-activation, for the backward
      uint4* a = reinterpret_cast<uint4*>(static_cast<bf16*>(pr.aux) + (size_t)row * pr.ldo + col0);
#pragma unroll
      for (int i = 0; i < 2; ++i)
        a[i] = make_uint4(pack_bf16x2(v[8 * i + 0], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                          pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.5f * v[i] * (1.0f + erff(v[i] * 0.7071067811865476f));
  } else if constexpr (E == kEpiGeluBwd) {
    // d/du GELU(u) = Phi(u) + u phi(u), phi the standard normal density
    const uint4* a = reinterpret_cast<const uint4*>(static_cast<const bf16*>(pr.aux) + (size_t)row * pr.ldo + col0);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint4 w = __ldg(a + i);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 u = unpack_bf16x2(ww[j]);
        const float g0 = 0.5f * (1.0f + erff(u.x * 0.7071067811865476f)) + u.x * 0.3989422804014327f * __expf(-0.5f * u.x * u.x);
        const float g1 = 0.5f * (1.0f + erff(u.y * 0.7071067811865476f)) + u.y * 0.3989422804014327f * __expf(-0.5f * u.y * u.y);
        v[8 * i + 2 * j] *= g0;
        v[8 * i + 2 * j + 1] *= g1;
      }
    }
  } else if constexpr (E == kEpiQkvRope) {
    const int which = col0 / p.H;
    if (qk_g != nullptr) {
      const uint4* gp = reinterpret_cast<const uint4*>(qk_g + (col0 - which * p.H) % p.head_dim);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint4 u = __ldg(gp + i);
        const float2 g0 = unpack_bf16x2(u.x), g1 = unpack_bf16x2(u.y), g2 = unpack_bf16x2(u.z),
                     g3 = unpack_bf16x2(u.w);
        v[8 * i + 0] *= qk_rstd * g0.x; v[8 * i + 1] *= qk_rstd * g0.y;
        v[8 * i + 2] *= qk_rstd * g1.x; v[8 * i + 3] *= qk_rstd * g1.y;
        v[8 * i + 4] *= qk_rstd * g2.x; v[8 * i + 5] *= qk_rstd * g2.y;
        v[8 * i + 6] *= qk_rstd * g3.x; v[8 * i + 7] *= qk_rstd * g3.y;
      }
    }
    if (which < 2) {
      const int joint = __ldg(p.srow_joint + pr.row_off + row);
      if (!MF_IDX_OK(joint >= 0 && joint < p.n_tok)) return;
      const int* ps = p.pos + (size_t)joint * 3;
      const float pf = (float)__ldg(ps), pr_ = (float)__ldg(ps + 1), pc = (float)__ldg(ps + 2);
      const int g0 = ((col0 - which * p.H) % p.head_dim) >> 1;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int ax = rope_axis[g0 + i];
        const float th = (ax == 0 ? pf : (ax == 1 ? pr_ : pc)) * rope_inv[g0 + i];
        // |th| <= max position (a few hundred): reduce modulo 2 pi with a two-constant
        // Cody-Waite step (2 pi = kHi + kLo), then the hardware sine / cosine on [-pi, pi]
        const float kq = rintf(th * 0.15915494309189535f);
        const float rr = fmaf(-kq, -1.7484555314695172e-07f, fmaf(-kq, 6.2831854820251465f, th));
        float sn, cs;
        __sincosf(rr, &sn, &cs);
        const float x0 = v[2 * i], x1 = v[2 * i + 1];
        v[2 * i] = x0 * cs - x1 * sn;
        v[2 * i + 1] = x0 * sn + x1 * cs;
      }
    }
  }
}

// Phase 2: 8 columns of one row to global memory; returns the bf16 word written (zero when the
// position lies outside the problem).
template <int EPI>
__device__ __forceinline__ uint4 epi_store8(const GemmParams& p, const GemmProblem& pr, int row, int col,
                                            const float4& a, const float4& b) {
  constexpr int E = EPI & 7;
  if (row >= pr.M || col >= pr.N) return make_uint4(0u, 0u, 0u, 0u);
  if constexpr (E == kEpiBiasF32) {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(pr.out) + (size_t)row * pr.ldo + col);
    o[0] = a;
    o[1] = b;
    return make_uint4(0u, 0u, 0u, 0u);
  }
  float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  bf16* dst;
  if constexpr (E == kEpiQkvRope) {
    const int joint = __ldg(p.srow_joint + pr.row_off + row);
    if (!MF_IDX_OK(joint >= 0 && joint < p.n_tok)) return make_uint4(0u, 0u, 0u, 0u);
    const int which = col / p.H;
    dst = (which == 0 ? p.q : (which == 1 ? p.k : p.v)) + (size_t)joint * p.H + (col - which * p.H);
  } else {
    dst = static_cast<bf16*>(pr.out) + (size_t)row * pr.ldo + col;
  }
  if constexpr (E == kEpiGateResid) {
    if constexpr ((EPI & kEpiSave) != 0)  // the ungated branch output, for the backward
      *reinterpret_cast<uint4*>(static_cast<bf16*>(pr.aux) + (size_t)row * pr.ldo + col) =
          make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                     pack_bf16x2(v[6], v[7]));
    const int seq = __ldg(p.srow_seq + pr.row_off + row);
    if (!MF_IDX_OK(seq >= 0 && seq < p.n_seq)) return make_uint4(0u, 0u, 0u, 0u);
    const float4* g = reinterpret_cast<const float4*>(
        p.mod + ((size_t)seq * 2 + pr.stream) * 6 * (size_t)p.H + p.gate_off + col);
    const float4 ga = __ldg(g), gb = __ldg(g + 1);
    const uint4 u = *reinterpret_cast<const uint4*>(dst);
    const float2 x0 = unpack_bf16x2(u.x), x1 = unpack_bf16x2(u.y), x2 = unpack_bf16x2(u.z),
                 x3 = unpack_bf16x2(u.w);
    v[0] = fmaf(ga.x, v[0], x0.x); v[1] = fmaf(ga.y, v[1], x0.y);
    v[2] = fmaf(ga.z, v[2], x1.x); v[3] = fmaf(ga.w, v[3], x1.y);
    v[4] = fmaf(gb.x, v[4], x2.x); v[5] = fmaf(gb.y, v[5], x2.y);
    v[6] = fmaf(gb.z, v[6], x3.x); v[7] = fmaf(gb.w, v[7], x3.y);
  }
  uint4 w;
  w.x = pack_bf16x2(v[0], v[1]);
  w.y = pack_bf16x2(v[2], v[3]);
  w.z = pack_bf16x2(v[4], v[5]);
  w.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(dst) = w;
  return w;
}

// Running statistics of one row's bf16 outputs in this thread (kEpiStats): sums of the values'
// deviations from a shift k (the first value seen), so that the sum of squares does not cancel
// when the row's mean is large next to its spread.
struct RowStats {
  float k, s1, s2;
};
__device__ __forceinline__ void row_stats_add(RowStats& st, const uint4& w, bool first) {
  const float2 a = unpack_bf16x2(w.x), b = unpack_bf16x2(w.y), c = unpack_bf16x2(w.z), e = unpack_bf16x2(w.w);
  const float v[8] = {a.x, a.y, b.x, b.y, c.x, c.y, e.x, e.y};
  if (first) st = RowStats{v[0], 0.0f, 0.0f};
  float s1a = 0.0f, s1b = 0.0f, s2a = 0.0f, s2b = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    float d0 = v[i], d1 = v[i + 1];
    f32x2_add(d0, d1, -st.k, -st.k);
    f32x2_add(s1a, s1b, d0, d1);
    f32x2_fma(d0, d1, d0, d1, s2a, s2b);  // d * d + s2
    s2a = d0;
    s2b = d1;
  }
  st.s1 += s1a + s1b;
  st.s2 += s2a + s2b;
}

template <int BN, int EPI>
__global__ void __launch_bounds__(192, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
  constexpr int STAGES = (BN == 256) ? 4 : 6;
  constexpr uint32_t A_BYTES = kBM * kBK * 2;
  constexpr uint32_t B_BYTES = BN * kBK * 2;
  constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr uint32_t TMEM_COLS = 2 * BN;
  constexpr uint32_t IDESC = idesc_bf16_f32(kBM, BN, false);

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[STAGES], empty_bar[STAGES], tfull_bar[2], tempty_bar[2], drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ float rope_inv[64];
  __shared__ int rope_axis[64];

  uint8_t* smem = align1024(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int total = p.tile_begin[p.n_prob];
  const uint64_t lim = p.wait_limit_ns;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 128);
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if constexpr (EPI == kEpiQkvRope) {
    // pair g of a head: axis block (frame D/8 | row 7D/16 | col 7D/16), inverse frequency
    // 10000^(-2j/width) for the pair's index j inside its block
    const int D = p.head_dim;
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
  }
  if (warp == 1) tmem_alloc(&tmem_base_sh, TMEM_COLS);
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.n_prob; ++i) {
      tma_prefetch_desc(&p.tmA[i]);
      tma_prefetch_desc(&p.tmB[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;
  mf_pdl_enter();  // the prologue above touched no global memory the previous kernel writes

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t armed = 0, armed_par = 0;  // bit s: stage s armed; its parity
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        int pi, m, n;
        decode_tile(p, tile, pi, m, n);
        const int nkb = p.prob[pi].K / kBK;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1, lim) || *(volatile int*)&abort_flag) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * STAGE_BYTES;
          mbar_arrive_expect_tx(&full_bar[stage], STAGE_BYTES);
          tma_load_2d(sa, &p.tmA[pi], kb * kBK, m * kBM, &full_bar[stage]);
          tma_load_2d(sa + A_BYTES, &p.tmB[pi], kb * kBK, n * BN, &full_bar[stage]);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) {
        *(volatile int*)&abort_flag = 1;
        report_status(p.status, kStatusTimeout);
        for (int s = 0; s < STAGES; ++s)  // let this thread's copies land before exiting
          if (armed & (1u << s)) mbar_wait(&full_bar[s], (armed_par >> s) & 1u, lim);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        int pi, m, n;
        decode_tile(p, tile, pi, m, n);
        const int nkb = p.prob[pi].K / kBK;
        if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1, lim) || *(volatile int*)&abort_flag) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_bf16(d_tmem, sdesc_sw128(a0 + k * 32, 16, 1024), sdesc_sw128(b0 + k * 32, 16, 1024),
                     IDESC, (kb | k) != 0 ? 1u : 0u);
          mma_commit(&empty_bar[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        mma_commit(&tfull_bar[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (!ok) {
        *(volatile int*)&abort_flag = 1;
        report_status(p.status, kStatusTimeout);
        mma_commit(&drain_bar);  // wait for this thread's MMAs before TMEM is freed
        mbar_wait(&drain_bar, 0, lim);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue warps
    const int q = warp & 3;
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int pi, m, n;
      decode_tile(p, tile, pi, m, n);
      const bool ok = mbar_wait(&tfull_bar[acc], acc_phase, lim);
      if (!__all_sync(0xffffffffu, ok) || __any_sync(0xffffffffu, *(volatile int*)&abort_flag)) {
        if (lane == 0) {
          *(volatile int*)&abort_flag = 1;
          report_status(p.status, kStatusTimeout);
        }
        break;
      }
      tc_fence_after();
      const GemmProblem& pr = p.prob[pi];
      const int row = m * kBM + q * 32 + lane;
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        uint32_t r[32];
        tmem_ld32(tmem_addr(tmem_base, q * 32, acc * BN + c), r);
        tmem_ld_wait();
        tmem_reg_fence(r);
        epilogue_chunk<EPI>(p, pr, row, n * BN + c, r, rope_inv, rope_axis);
      }
      tc_fence_before();
      mbar_arrive(&tempty_bar[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int BN, int EPI>
cudaError_t launch_t(const GemmParams& p, int num_sms, cudaStream_t stream) {
  constexpr int STAGES = (BN == 256) ? 4 : 6;
  const int smem = STAGES * (kBM * kBK * 2 + BN * kBK * 2) + 1024;
  auto kern = gemm_kernel<BN, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int total = p.tile_begin[p.n_prob];
  if (total <= 0) return cudaSuccess;
  const int grid = total < num_sms ? total : num_sms;
  launch_k(kern, grid, 192, smem, stream, p);
  return cudaGetLastError();
}


// ---------------------------------------------------------------------------------------
constexpr int kPairThreads = 320;  // producer warp, MMA warp, 8 epilogue warps

// CTA-pair variant: a cluster of two CTAs computes one 256 x 256 tile with
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16).  Each CTA stages its own 128 rows of
// A and its own 128 rows of B (half of the tile's N) per 64-wide K block, so a CTA moves
// 32 KB per K block instead of the 48 KB of the single-CTA 128 x 256 tile for the same MMA
// work per SM.  Both CTAs' copies complete on the even CTA's full barrier; the even CTA's
// MMA thread issues for the pair and its commits arrive on the barriers of both CTAs
// (multicast), so each CTA's producer sees its own stage freed and each CTA's epilogue sees
// its own 128 accumulator rows (TMEM lanes) ready.  Eight epilogue warps per CTA, two per TMEM
// lane quarter, each take 128 of the tile's 256 columns through the staged epilogue above; the
// epilogue warps of both CTAs release an accumulator buffer by arriving on the even CTA's
// barrier.
template <int EPI, int MAJ>
__global__ void __launch_bounds__(kPairThreads, 1) gemm_pair_kernel(const __grid_constant__ GemmParams p) {
  constexpr int STAGES = 6;
  constexpr int BN = 256;
  constexpr uint32_t A_BYTES = kBM * kBK * 2;         // this CTA's 128 rows of A
  constexpr uint32_t B_BYTES = (BN / 2) * kBK * 2;    // this CTA's 128 rows of B
  constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr uint32_t TMEM_COLS = 2 * BN;
  // E4M3 operands (kEpiF8): a 128-byte row of a K block holds 128 elements instead of 64, and
  // each MMA consumes K = 32 instead of 16; the byte layout of the stages is the same
  constexpr bool F8 = (EPI & kEpiF8) != 0;
  constexpr int E = EPI & 7;
  constexpr int KE = F8 ? 2 * kBK : kBK;  // K elements per stage
  constexpr bool AMN = (MAJ & kMajAMN) != 0, BMN = (MAJ & kMajBMN) != 0;
  static_assert(!F8 || MAJ == kMajKK, "E4M3 operands are K-major");
  constexpr uint32_t IDESC = F8 ? idesc_e4m3_f32(2 * kBM, BN) : idesc_bf16_f32_mn(2 * kBM, BN, AMN, BMN);

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[STAGES], empty_bar[STAGES], tfull_bar[2], tempty_bar[2], drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ float rope_inv[64];
  __shared__ int rope_axis[64];

  uint8_t* smem = align1024(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const int total = p.tile_begin[p.n_prob];
  const uint64_t lim = p.wait_limit_ns;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 16);  // lane 0 of the 8 epilogue warps of both CTAs
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if constexpr (E == kEpiQkvRope) {
    const int D = p.head_dim;
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
  }
  if (warp == 1) tmem_alloc_pair(&tmem_base_sh, TMEM_COLS);
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.n_prob; ++i) {
      tma_prefetch_desc(&p.tmA[i]);
      tma_prefetch_desc(&p.tmB[i]);
    }
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;
  mf_pdl_enter();  // the prologue above touched no global memory the previous kernel writes

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer (both CTAs)
    const uint32_t el = elect_one();
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    for (int tile = pair; ok && tile < total; tile += n_pairs) {
      int pi, m, n;
      decode_tile(p, tile, pi, m, n);
      const int nkb = (p.prob[pi].K + KE - 1) / KE;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!__all_sync(0xffffffffu, mbar_wait(&empty_bar[stage], phase ^ 1, lim)) ||
            __any_sync(0xffffffffu, *(volatile int*)&abort_flag)) {
          ok = false;
          break;
        }
        if (el) {
          uint8_t* sa = smem + stage * STAGE_BYTES;
          if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * STAGE_BYTES);
          const uint32_t fb = mapa_shared(&full_bar[stage], 0);
          const int a_row = m * 2 * kBM + rank * kBM, b_row = n * BN + rank * (BN / 2);
          if constexpr (AMN) {  // [K][M] storage: two 64 (M) x 64 (K) boxes
            tma_load_2d_pair(sa, &p.tmA[pi], a_row, kb * KE, fb);
            tma_load_2d_pair(sa + A_BYTES / 2, &p.tmA[pi], a_row + 64, kb * KE, fb);
          } else {
            tma_load_2d_pair(sa, &p.tmA[pi], kb * KE, a_row, fb);
          }
          if constexpr (BMN) {
            tma_load_2d_pair(sa + A_BYTES, &p.tmB[pi], b_row, kb * KE, fb);
            tma_load_2d_pair(sa + A_BYTES + B_BYTES / 2, &p.tmB[pi], b_row + 64, kb * KE, fb);
          } else {
            tma_load_2d_pair(sa + A_BYTES, &p.tmB[pi], kb * KE, b_row, fb);
          }
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    }
    if (!ok && el) {
      *(volatile int*)&abort_flag = 1;
      report_status(p.status, kStatusTimeout);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (even CTA)
    // The whole warp runs the loop; one elected lane issues each MMA and commit.
    if (leader) {
      const uint32_t el = elect_one();
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < total; tile += n_pairs) {
        int pi, m, n;
        decode_tile(p, tile, pi, m, n);
        const int nkb = (p.prob[pi].K + KE - 1) / KE;
        if (!__all_sync(0xffffffffu, mbar_wait(&tempty_bar[acc], acc_phase ^ 1, lim)) ||
            __any_sync(0xffffffffu, *(volatile int*)&abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(&full_bar[stage], phase, lim))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // K-major: 128-byte rows of K, a K = 16 step is 32 bytes into the row.  MN-major:
          // 128-byte rows of 64 MN elements per K index, the two 64-wide MN halves A_BYTES / 2
          // apart, a K = 16 step is 16 rows (2048 bytes)
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint64_t ad = AMN ? sdesc_sw128(sa, A_BYTES / 2, 1024) : sdesc_sw128(sa, 16, 1024);
          const uint64_t bd = BMN ? sdesc_sw128(sa + A_BYTES, B_BYTES / 2, 1024) : sdesc_sw128(sa + A_BYTES, 16, 1024);
          constexpr uint32_t a_step = AMN ? (2048 >> 4) : 2, b_step = BMN ? (2048 >> 4) : 2;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            if constexpr (F8)
              mma_f8_pair_if(el, d_tmem, ad + k * 2, bd + k * 2, IDESC, (kb | k) != 0 ? 1u : 0u);
            else
              mma_bf16_pair_if(el, d_tmem, ad + k * a_step, bd + k * b_step, IDESC, (kb | k) != 0 ? 1u : 0u);
          mma_commit_pair_mc_if(el, &empty_bar[stage], 0x3);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        mma_commit_pair_mc_if(el, &tfull_bar[acc], 0x3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (!ok) {
        if (el) {
          *(volatile int*)&abort_flag = 1;
          report_status(p.status, kStatusTimeout);
          mma_commit_pair_mc(&drain_bar, 0x1);  // wait for this warp's MMAs before TMEM is freed
        }
        __syncwarp();
        mbar_wait(&drain_bar, 0, lim);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue warps (both CTAs)
    const int q = warp & 3;                 // TMEM lane quarter = 32 accumulator rows
    const int c_lo = ((warp - 2) >> 2) * (BN / 2);  // first of this warp's 128 columns
    const uint32_t tempty0 = mapa_shared(&tempty_bar[0], 0), tempty1 = mapa_shared(&tempty_bar[1], 0);
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = pair; tile < total; tile += n_pairs) {
      int pi, m, n;
      decode_tile(p, tile, pi, m, n);
      const bool ok = mbar_wait(&tfull_bar[acc], acc_phase, lim);
      if (!__all_sync(0xffffffffu, ok) || __any_sync(0xffffffffu, *(volatile int*)&abort_flag)) {
        if (lane == 0) {
          *(volatile int*)&abort_flag = 1;
          report_status(p.status, kStatusTimeout);
        }
        break;
      }
      tc_fence_after();
      const GemmProblem& pr = p.prob[pi];
      const int row0 = m * 2 * kBM + rank * kBM + q * 32;  // first of this warp's 32 rows
      float* stg = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES) + (warp - 2) * 32 * kStageRow;
      if constexpr (E == kEpiBiasBf16 || E == kEpiGelu || E == kEpiGeluBwd) {
        if (p.tma_store[pi]) {
          // bf16 rows of 64 columns, 16-byte chunks swizzled as the 128-byte-swizzle tensor map
          // expects, then one TMA store of 32 rows x 64 columns per group
          uint8_t* tst = smem + STAGES * STAGE_BYTES + (warp - 2) * 4096;
          const uint32_t el = elect_one();
#pragma unroll 1
          for (int g = 0; g < BN / 2; g += 64) {
            if (el) tma_store_wait_read();  // the previous group's store has read the buffer
            __syncwarp();
#pragma unroll
            for (int cq = 0; cq < 4; ++cq) {
              const int c = c_lo + g + cq * 16;
              uint32_t r[16];
              tmem_ld16(tmem_addr(tmem_base, q * 32, acc * BN + c), r);
              tmem_ld_wait();
              tmem_reg_fence16(r);
              float v[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
              epi_row16<EPI>(p, pr, row0 + lane, n * BN + c, v, rope_inv, rope_axis);
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {
                uint4 w;
                w.x = pack_bf16x2(v[8 * h2 + 0], v[8 * h2 + 1]);
                w.y = pack_bf16x2(v[8 * h2 + 2], v[8 * h2 + 3]);
                w.z = pack_bf16x2(v[8 * h2 + 4], v[8 * h2 + 5]);
                w.w = pack_bf16x2(v[8 * h2 + 6], v[8 * h2 + 7]);
                const int ch = cq * 2 + h2;
                *reinterpret_cast<uint4*>(tst + lane * 128 + ((ch ^ (lane & 7)) << 4)) = w;
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (el) {
              tma_store_2d(&p.tmC[pi], n * BN + c_lo + g, row0, tst);
              tma_store_commit();
            }
            __syncwarp();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(acc ? tempty1 : tempty0);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
          continue;
        }
      }
      // QK-RMSNorm: a first pass over this warp's 128 columns (one head, or two when D = 64)
      // gives each row's 1 / RMS per head, from the same bias-added values the second uses
      const bf16* qk_g = nullptr;
      float qk_rstd0 = 0.0f, qk_rstd1 = 0.0f;
      if constexpr (E == kEpiQkvRope) {
        const int col_lo = n * BN + c_lo, which = col_lo / p.H;
        const bf16* g = pi ? (which ? p.qk_norm[1][1] : p.qk_norm[1][0])
                           : (which ? p.qk_norm[0][1] : p.qk_norm[0][0]);
        if (which < 2 && col_lo < pr.N && g != nullptr) {
          qk_g = g;
          float ss0 = 0.0f, ss1 = 0.0f;
#pragma unroll 1
          for (int c = c_lo; c < c_lo + BN / 2; c += 16) {
            uint32_t r[16];
            tmem_ld16(tmem_addr(tmem_base, q * 32, acc * BN + c), r);
            tmem_ld_wait();
            tmem_reg_fence16(r);
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
            add_bias16(pr, n * BN + c, v);
            float part = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) part = fmaf(v[i], v[i], part);
            if ((c - c_lo) >= p.head_dim) ss1 += part;
            else ss0 += part;
          }
          qk_rstd0 = rsqrtf(ss0 / (float)p.head_dim + kQkNormEps);
          qk_rstd1 = rsqrtf(ss1 / (float)p.head_dim + kQkNormEps);
        }
      }
      RowStats rs[2];  // kEpiStats: rows 16 it + lane / 2 of this warp's 128 columns
#pragma unroll 1
      for (int c = c_lo; c < c_lo + BN / 2; c += 16) {
        uint32_t r[16];
        tmem_ld16(tmem_addr(tmem_base, q * 32, acc * BN + c), r);
        tmem_ld_wait();
        tmem_reg_fence16(r);
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
        epi_row16<EPI>(p, pr, row0 + lane, n * BN + c, v, rope_inv, rope_axis, qk_g,
                       (c - c_lo) >= p.head_dim ? qk_rstd1 : qk_rstd0);
        float4* sp = reinterpret_cast<float4*>(stg + lane * kStageRow);
#pragma unroll
        for (int i = 0; i < 4; ++i) sp[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        __syncwarp();
#pragma unroll
        for (int it = 0; it < 2; ++it) {  // rows 16 it .. 16 it + 15, two threads per row
          const int rr = 16 * it + (lane >> 1), hh = lane & 1;
          const float4* rp = reinterpret_cast<const float4*>(stg + rr * kStageRow + hh * 8);
          const uint4 w = epi_store8<EPI>(p, pr, row0 + rr, n * BN + c + hh * 8, rp[0], rp[1]);
          if constexpr ((EPI & kEpiStats) != 0) row_stats_add(rs[it], w, c == c_lo);
        }
        __syncwarp();
      }
      if constexpr ((EPI & kEpiStats) != 0) {
        // each lane holds 64 values of its row, its partner (lane ^ 1) the other 64 of the
        // 128-column part: (mean, M2) of each, then the two merged (equal counts)
        const int part = (n * BN + c_lo) >> 7;
#pragma unroll
        for (int it = 0; it < 2; ++it) {
          const float m = rs[it].k + rs[it].s1 * (1.0f / 64.0f);
          const float m2 = fmaxf(rs[it].s2 - rs[it].s1 * rs[it].s1 * (1.0f / 64.0f), 0.0f);
          const float mo = __shfl_xor_sync(0xffffffffu, m, 1);
          const float m2o = __shfl_xor_sync(0xffffffffu, m2, 1);
          const float d = mo - m;
          const int row = row0 + 16 * it + (lane >> 1);
          if ((lane & 1) == 0 && row < pr.M)
            p.ln_stats[(size_t)(pr.row_off + row) * p.ln_parts + part] =
                make_float2(0.5f * (m + mo), m2 + m2o + 32.0f * d * d);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc ? tempty1 : tempty0);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  if (warp >= 2) tma_store_wait_all();  // this thread's bulk stores (if any) have completed
  tc_fence_before();
  cluster_sync();  // the pair's MMAs and TMEM reads are done, no remote signal is pending
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

template <int EPI, int MAJ = kMajKK>
cudaError_t launch_pair(const GemmParams& p, int num_sms, cudaStream_t stream) {
  constexpr int STAGES = 6;
  // epilogue staging: 8 warps x max(32 rows of kStageRow floats, a 32 x 64 bf16 store box)
  constexpr int kStaging = 8 * (32 * kStageRow * 4 > 4096 ? 32 * kStageRow * 4 : 4096);
  const int smem = STAGES * (kBM * kBK * 2 + 128 * kBK * 2) + kStaging + 1024;
  auto kern = gemm_pair_kernel<EPI, MAJ>;
  static int max_pairs = 0;  // clusters of two that fit on the device at once (per instantiation)
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_pairs == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    max_pairs = n < num_sms / 2 ? n : num_sms / 2;
  }
  const int total = p.tile_begin[p.n_prob];
  if (total <= 0) return cudaSuccess;
  const int pairs = total < max_pairs ? total : max_pairs;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.numAttrs = pdl_allowed() ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

cudaError_t launch_gemm_pair(const GemmParams& p, int epi, int num_sms, cudaStream_t stream, int maj) {
  if (maj == kMajBMN) {  // input gradients: dY W (W stored [K = out][N = in])
    switch (epi) {
      case kEpiBiasBf16: return launch_pair<kEpiBiasBf16, kMajBMN>(p, num_sms, stream);
      case kEpiGeluBwd: return launch_pair<kEpiGeluBwd, kMajBMN>(p, num_sms, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  if (maj == kMajMNMN) {  // weight gradients: dY^T X, both stored [K = tokens][...]
    if (epi == kEpiBiasF32) return launch_pair<kEpiBiasF32, kMajMNMN>(p, num_sms, stream);
    return cudaErrorInvalidValue;
  }
  if (maj != kMajKK) return cudaErrorInvalidValue;
  switch (epi) {
    case kEpiGelu | kEpiSave: return launch_pair<kEpiGelu | kEpiSave>(p, num_sms, stream);
    case kEpiGateResid | kEpiSave: return launch_pair<kEpiGateResid | kEpiSave>(p, num_sms, stream);
    case kEpiGateResid | kEpiStats: return launch_pair<kEpiGateResid | kEpiStats>(p, num_sms, stream);
    case kEpiBiasBf16: return launch_pair<kEpiBiasBf16>(p, num_sms, stream);
    case kEpiBiasF32: return launch_pair<kEpiBiasF32>(p, num_sms, stream);
    case kEpiQkvRope: return launch_pair<kEpiQkvRope>(p, num_sms, stream);
    case kEpiGateResid: return launch_pair<kEpiGateResid>(p, num_sms, stream);
    case kEpiGelu: return launch_pair<kEpiGelu>(p, num_sms, stream);
    case kEpiBiasBf16 | kEpiF8: return launch_pair<kEpiBiasBf16 | kEpiF8>(p, num_sms, stream);
    case kEpiQkvRope | kEpiF8: return launch_pair<kEpiQkvRope | kEpiF8>(p, num_sms, stream);
    case kEpiGateResid | kEpiF8: return launch_pair<kEpiGateResid | kEpiF8>(p, num_sms, stream);
    case kEpiGelu | kEpiF8: return launch_pair<kEpiGelu | kEpiF8>(p, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm(const GemmParams& p, int BN, int epi, int num_sms, cudaStream_t stream) {
#define MF_GEMM_CASE(bn, ep) \
  if (BN == bn && epi == ep) return launch_t<bn, ep>(p, num_sms, stream);
  MF_GEMM_CASE(256, kEpiBiasBf16)
  MF_GEMM_CASE(256, kEpiBiasF32)
  MF_GEMM_CASE(256, kEpiQkvRope)
  MF_GEMM_CASE(256, kEpiGateResid)
  MF_GEMM_CASE(256, kEpiGelu)
  MF_GEMM_CASE(128, kEpiBiasBf16)
  MF_GEMM_CASE(128, kEpiBiasF32)
  MF_GEMM_CASE(128, kEpiQkvRope)
  MF_GEMM_CASE(128, kEpiGateResid)
  MF_GEMM_CASE(128, kEpiGelu)
#undef MF_GEMM_CASE
  return cudaErrorInvalidValue;
}

MF_BOUNDS_EXPORT(gemm)

}  // namespace mf
