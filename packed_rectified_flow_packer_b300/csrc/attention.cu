// Varlen joint attention for the packed NR-MMDiT block on sm_103a.
//
// Each packed sample attends only over its own [text | image] tokens (PaperReading review of
// "Mage-Flow: An Efficient Native-Resolution Foundation Model for Image Generation and
// Editing", §2.2 (2): cumulative offsets plus a varlen kernel restricting attention to each
// sample).  Only diagonal blocks are ever scheduled: a work item is (sample, 256-row query
// block, head) and loops over that sample's own 128-row key tiles, so the cost is
// sum_i L_i^2, not (sum_i L_i)^2.
//
// CTAs are ordered sample by sample (longest first); inside a sample the query blocks run
// fastest, then the heads, so the CTAs resident at the same time share one or a few heads' K
// and V in L2 instead of streaming every head of the sample at once.
//
// One CTA per work item, 320 threads.  The 256 query rows are two 128-row tiles t = 0, 1,
// each with its own softmax warpgroup, so the tensor core works on one tile while the other
// tile's exponentials run:
//   warp 0        : TMA producer: Q_0 and Q_1 once, then K_0, V_0, K_1, V_1, ... into one
//                   shared-memory ring, in the order the tensor core consumes them.
//   warp 1        : TMEM allocator and MMA issuer (the whole warp runs the loop, one elected
//                   lane issues) of tcgen05.mma in the order
//                   S_0 = Q_0 K_0^T, S_1 = Q_1 K_0^T, then per key tile j
//                   O_0 += P_0 V_j, S_0 = Q_0 K_{j+1}^T, O_1 += P_1 V_j, S_1 = Q_1 K_{j+1}^T.
//   warps 2..5    : softmax of tile 0, warps 6..9: softmax of tile 1; one thread per query
//                   row: S from TMEM, online max / sum in f32 with exp2, P in bf16 written
//                   back to TMEM over its own S (two bf16 per 32-bit column), where the PV
//                   product reads it as the A operand; at the end O / l to global memory in
//                   stream-sorted order.
// TMEM (512 columns): S_0 @0, S_1 @128, O_0 @256, O_1 @256 + D.
// The commit that signals S_t for key tile j also covers every MMA issued before it, in
// particular O_t += P_t V_{j-1}; so once S_t is visible O_t is quiescent and may be rescaled,
// and P_t's columns may be overwritten (the PV that read them has completed).
// The running max is only moved (and O rescaled in TMEM) when a tile's max exceeds it by
// more than 8 in log2 units; the result is unchanged because numerator and denominator use
// the same stale max, and P stays <= 2^8.  Per score the softmax spends half a three-input
// max, half a packed f32x2 FMA (scale and shift), one ex2.approx, half a packed add (row sum)
// and half a bf16x2 conversion.
#include "attention.cuh"

namespace mf {
namespace {

constexpr int kT = 128;             // query rows per tile, key rows per tile
constexpr uint32_t kAtom = 16384;   // 128 rows x 128 bytes
constexpr float kRescaleLog2 = 8.0f;
constexpr int kThreads = 320;

// Three-input f32 maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (x0, x1) = (x0 * c + d, x1 * c + d) as one packed f32x2 FMA.
__device__ __forceinline__ void fma2(float& x0, float& x1, float c, float d) {
  asm("{\n\t.reg .b64 x, c, d;\n\t"
      "mov.b64 x, {%0, %1};\n\tmov.b64 c, {%2, %2};\n\tmov.b64 d, {%3, %3};\n\t"
      "fma.rn.f32x2 x, x, c, d;\n\tmov.b64 {%0, %1}, x;\n\t}"
      : "+f"(x0), "+f"(x1)
      : "f"(c), "f"(d));
}

// (a0, a1) += (x0, x1) as one packed f32x2 add.
__device__ __forceinline__ void add2(float& a0, float& a1, float x0, float x1) {
  asm("{\n\t.reg .b64 a, x;\n\t"
      "mov.b64 a, {%0, %1};\n\tmov.b64 x, {%2, %3};\n\t"
      "add.rn.f32x2 a, a, x;\n\tmov.b64 {%0, %1}, a;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(x0), "f"(x1));
}

// 8 consecutive 32-bit columns of this thread's TMEM lane.  No memory clobber, so the
// compiler may interleave the arithmetic of neighbouring chunks with the stores; the stores
// stay ordered before tcgen05.wait::st (both are volatile asm).
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]));
}

// O_t += P_t V: A operand (P, 128 x 16 bf16 per instruction) read from TMEM; issued by the
// lane whose `pred` is nonzero.
__device__ __forceinline__ void mma_bf16_ts_if(uint32_t pred, uint32_t d_tmem, uint32_t a_tmem,
                                               uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(pred)
      : "memory");
}

template <int D>
struct AttnSmem {
  static constexpr uint32_t Q = kT * D * 2;                 // one query tile
  static constexpr uint32_t KV = kT * D * 2;                // one key or value tile
  static constexpr uint32_t budget = 224u * 1024u;
  static constexpr int stages = (int)((budget - 2 * Q) / KV) > 8 ? 8 : (int)((budget - 2 * Q) / KV);
  static constexpr uint32_t off_q = 0;
  static constexpr uint32_t off_kv = 2 * Q;
  static constexpr uint32_t total = off_kv + stages * KV;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_kernel(const __grid_constant__ AttnParams p) {
  using L = AttnSmem<D>;
  constexpr int NS = L::stages;
  constexpr uint32_t IDESC_S = idesc_bf16_f32(kT, kT, false);
  constexpr uint32_t IDESC_PV = idesc_bf16_f32(kT, D, true);
  constexpr uint32_t TMEM_COLS = 512;
  constexpr uint32_t O_COL = 256;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t q_full, kv_full[NS], kv_empty[NS], s_full[2], p_full[2], o_done[2], drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  uint8_t* smem = align1024(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t lim = p.wait_limit_ns;

  // (sample, head, query block) of this CTA: the work list holds each sample's query blocks
  // contiguously, samples longest first; a sample spans (query blocks) x heads CTAs
  int seq = 0, kv0 = 0, len = 0, nqb = 1, base = 0;
  for (int it = 0; it < p.n_items;) {
    seq = __ldg(p.items + 2 * it);
    if (!MF_IDX_OK(seq >= 0 && seq < p.n_seq)) { len = 0; break; }
    kv0 = __ldg(p.cu + seq);
    len = __ldg(p.cu + seq + 1) - kv0;
    if (!MF_IDX_OK(len > 0)) break;
    nqb = (len + 2 * kT - 1) / (2 * kT);
    if ((int)blockIdx.x < base + nqb * p.heads) break;
    base += nqb * p.heads;
    it += nqb;
  }
  const int h = ((int)blockIdx.x - base) / nqb;
  const int qb = ((int)blockIdx.x - base) - h * nqb;
  if (!MF_IDX_OK(seq >= 0 && seq < p.n_seq && kv0 >= 0 && len > 0 && kv0 + len <= p.n_tok && h < p.heads))
    return;  // before any barrier or TMEM allocation: the whole CTA leaves together
  const int q0 = kv0 + qb * 2 * kT;
  const int n_kv = (len + kT - 1) / kT;
  const int n_t = (len - qb * 2 * kT) > kT ? 2 : 1;  // query tiles of this block inside the sample

  if (threadIdx.x == 0) {
    mbar_init(&q_full, 1);
    for (int b = 0; b < NS; ++b) {
      mbar_init(&kv_full[b], 1);
      mbar_init(&kv_empty[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 128);
      mbar_init(&o_done[b], 1);
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) tmem_alloc(&tmem_base_sh, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;
  mf_pdl_enter();  // the prologue above touched no global memory the previous kernel writes

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    // The whole warp runs the loop (warp-uniform state); one elected lane issues.
    const uint32_t el = elect_one();
    if (el) {
      tma_prefetch_desc(&p.tmK);
      tma_prefetch_desc(&p.tmV);
      mbar_arrive_expect_tx(&q_full, n_t * L::Q);
      for (int t = 0; t < n_t; ++t)
#pragma unroll
        for (int a = 0; a < D / 64; ++a)
          tma_load_2d(smem + L::off_q + t * L::Q + a * kAtom, &p.tmQ, h * D + a * 64, q0 + t * kT,
                      &q_full);
    }
    __syncwarp();
    bool ok = true;
    uint32_t armed = 0, armed_par = 0;  // bit s: ring slot s has a copy in flight; its parity
    // ring order = consumption order of the tensor core: K_0, V_0, K_1, V_1, ...
    for (int idx = 0; ok && idx < 2 * n_kv; ++idx) {
      const int st = idx % NS;
      const uint32_t ph = (idx / NS) & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&kv_empty[st], ph ^ 1, lim)) ||
          __any_sync(0xffffffffu, *(volatile int*)&abort_flag)) {
        ok = false;
        break;
      }
      if (el) {
        const CUtensorMap* tm = (idx & 1) ? &p.tmV : &p.tmK;
        mbar_arrive_expect_tx(&kv_full[st], L::KV);
#pragma unroll
        for (int a = 0; a < D / 64; ++a)
          tma_load_2d(smem + L::off_kv + st * L::KV + a * kAtom, tm, h * D + a * 64,
                      kv0 + (idx >> 1) * kT, &kv_full[st]);
      }
      __syncwarp();
      armed |= 1u << st;
      armed_par = (armed_par & ~(1u << st)) | (ph << st);
    }
    if (!ok) {
      if (el) {
        *(volatile int*)&abort_flag = 1;
        report_status(p.status, kStatusTimeout);
      }
      mbar_wait(&q_full, 0, lim);  // let this warp's copies land before exiting
      for (int s2 = 0; s2 < NS; ++s2)
        if (armed & (1u << s2)) mbar_wait(&kv_full[s2], (armed_par >> s2) & 1u, lim);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp runs the loop (warp-uniform state and descriptors); one elected lane
    // issues each MMA and commit.  Waits are ordered by criticality: P_t first, then the ring
    // slot (whose copy normally landed long ago).
    const uint32_t el = elect_one();
    const uint64_t qd = sdesc_sw128(smem_u32(smem + L::off_q), 16, 1024);
    const uint64_t kv0d = sdesc_sw128(smem_u32(smem + L::off_kv), 16, 1024);
    const uint64_t vv0d = sdesc_sw128(smem_u32(smem + L::off_kv), kAtom, 1024);
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, lim));
    };
    auto issue_s = [&](int t, int slot) {
      const uint64_t kd = kv0d + ((slot * L::KV) >> 4);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t o = ((kk >> 2) * kAtom + (kk & 3) * 32) >> 4;
        mma_bf16_if(el, tmem_base + t * kT, qd + ((t * L::Q) >> 4) + o, kd + o, IDESC_S, kk > 0 ? 1u : 0u);
      }
      mma_commit_if(el, &s_full[t]);
    };
    auto slot_wait = [&](int idx) -> bool { return wait_all(&kv_full[idx % NS], (idx / NS) & 1); };
    bool ok = wait_all(&q_full, 0) && slot_wait(0);
    if (ok) {
      tc_fence_after();
      for (int t = 0; t < n_t; ++t) issue_s(t, 0);
      mma_commit_if(el, &kv_empty[0]);
    }
    for (int j = 0; ok && j < n_kv; ++j) {
      const int iv = 2 * j + 1, ik = 2 * j + 2;
      const bool next = j + 1 < n_kv;
      const uint64_t vd = vv0d + (((iv % NS) * L::KV) >> 4);
      for (int t = 0; t < n_t; ++t) {
        if (!wait_all(&p_full[t], j & 1) || (t == 0 && !slot_wait(iv))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)
          mma_bf16_ts_if(el, tmem_base + O_COL + t * D, tmem_base + t * kT + kk * 8, vd + ((kk * 2048) >> 4),
                         IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
        if (next) {
          if (t == 0 && !slot_wait(ik)) {
            ok = false;
            break;
          }
          issue_s(t, ik % NS);
        }
      }
      if (!ok) break;
      mma_commit_if(el, &kv_empty[iv % NS]);
      if (next) mma_commit_if(el, &kv_empty[ik % NS]);
    }
    if (ok) {
      for (int t = 0; t < n_t; ++t) mma_commit_if(el, &o_done[t]);
    } else {
      if (el) {
        *(volatile int*)&abort_flag = 1;
        report_status(p.status, kStatusTimeout);
        mma_commit(&drain_bar);  // wait for this warp's MMAs before TMEM is freed
      }
      __syncwarp();
      mbar_wait(&drain_bar, 0, lim);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax warpgroups
    const int t = (warp - 2) >> 2;   // query tile of this warpgroup
    const int qw = warp & 3;         // TMEM lane quarter this warp may access
    const int row = qw * 32 + lane;  // query row inside the tile = TMEM lane
    const uint32_t lane_base = tmem_addr(tmem_base, qw * 32, 0);
    const uint32_t s_col = t * kT, o_col = O_COL + t * D;
    const float c = p.scale_log2;
    float m = -INFINITY;  // running max, log2 units
    float l = 0.0f;       // running sum of P
    bool ok = true;
    if (t < n_t) {
      for (int j = 0; j < n_kv; ++j) {
        // every lane polls: a completed phase is seen by each lane's own try_wait, without a
        // shuffle and warp barrier on the path from S to the exponentials
        ok = __all_sync(0xffffffffu, mbar_wait(&s_full[t], j & 1, lim));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(lane_base + s_col + cc * 32, sr[cc]);
        tmem_ld_wait();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_reg_fence(sr[cc]);

        const int valid = len - j * kT;  // key columns of this tile inside the sample
        if (valid < kT) {
#pragma unroll
          for (int i = 0; i < kT; ++i)
            if (i >= valid) sr[i >> 5][i & 31] = __float_as_uint(-INFINITY);
        }
#define MF_S(i) __uint_as_float(sr[(i) >> 5][(i) & 31])
        float mx[4] = {MF_S(0), MF_S(1), MF_S(2), MF_S(3)};
#pragma unroll
        for (int i = 4; i < kT; i += 2) mx[(i >> 1) & 3] = max3f(mx[(i >> 1) & 3], MF_S(i), MF_S(i + 1));
        const float m_tile = max3f(mx[0], mx[1], fmaxf(mx[2], mx[3])) * c;
        const bool need = (j == 0) || (m_tile > m + kRescaleLog2);
        const float alpha = (j > 0 && need) ? ex2_approx(m - m_tile) : 1.0f;
        if (need) m = m_tile;

        // P_j = exp2(S c - m) in bf16, two keys per 32-bit TMEM column, written over the
        // first 64 columns of S_t, 16 keys at a time
        const float neg_m = -m;
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            float e0 = MF_S(cc * 16 + i), e1 = MF_S(cc * 16 + i + 1);
            fma2(e0, e1, c, neg_m);
            e0 = ex2_approx(e0);  // masked columns: ex2(-inf) is exactly 0
            e1 = ex2_approx(e1);
            add2(ls[i & 2], ls[(i & 2) + 1], e0, e1);
            pk[i >> 1] = pack_bf16x2(e0, e1);
          }
          tmem_st8(lane_base + s_col + cc * 8, pk);
        }
#undef MF_S
        l = l * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
        // O_t is quiescent here (see the header): rescale it in place when a row's max moved
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t r[32];
            tmem_ld32(lane_base + o_col + cc * 32, r);
            tmem_ld_wait();
            tmem_reg_fence(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(lane_base + o_col + cc * 32, r);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[t]);
      }
      if (ok) {
        ok = __all_sync(0xffffffffu, mbar_wait(&o_done[t], 0, lim));
        if (ok) {
          tc_fence_after();
          // O / l in bf16 through this tile's Q buffer (free once o_done[t] fired: every MMA of
          // tile t has completed): each warp stages its 32 rows, 16-byte chunks XOR-swizzled by
          // row, then writes whole rows (D bf16 each) with consecutive lanes on consecutive
          // 16-byte chunks of a row
          const float inv_l = 1.0f / l;
          if (p.lse != nullptr && q0 + t * kT + row < kv0 + len)  // ln sum_k exp(s_k), s = q.k / sqrt(D)
            p.lse[(size_t)h * p.n_tok + q0 + t * kT + row] = (m + log2f(l)) * 0.6931471805599453f;
          uint8_t* stg = smem + L::off_q + t * L::Q;   // [128 rows][D bf16]
          constexpr int kChunks = D / 8;               // 16-byte chunks per row
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t r[32];
            tmem_ld32(lane_base + o_col + cc * 32, r);
            tmem_ld_wait();
            tmem_reg_fence(r);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(r[8 * i + 0]) * inv_l, __uint_as_float(r[8 * i + 1]) * inv_l);
              w.y = pack_bf16x2(__uint_as_float(r[8 * i + 2]) * inv_l, __uint_as_float(r[8 * i + 3]) * inv_l);
              w.z = pack_bf16x2(__uint_as_float(r[8 * i + 4]) * inv_l, __uint_as_float(r[8 * i + 5]) * inv_l);
              w.w = pack_bf16x2(__uint_as_float(r[8 * i + 6]) * inv_l, __uint_as_float(r[8 * i + 7]) * inv_l);
              const int ch = cc * 4 + i;
              *reinterpret_cast<uint4*>(stg + row * (D * 2) + ((ch ^ (row & 7)) << 4)) = w;
            }
          }
          __syncwarp();
          constexpr int kRowsPerStore = 32 / kChunks;  // rows one warp-wide store covers
#pragma unroll 1
          for (int r0 = 0; r0 < 32; r0 += kRowsPerStore) {
            const int rr = qw * 32 + r0 + lane / kChunks, ch = lane % kChunks;
            const int qrow = q0 + t * kT + rr;
            const int srow = qrow < kv0 + len ? __ldg(p.joint_srow + qrow) : 0;
            if (qrow < kv0 + len && MF_IDX_OK(srow >= 0 && srow < p.n_tok)) {
              const uint4 w = *reinterpret_cast<const uint4*>(stg + rr * (D * 2) + ((ch ^ (rr & 7)) << 4));
              bf16* dst = p.out + (size_t)srow * p.H + h * D;
              reinterpret_cast<uint4*>(dst)[ch] = w;
            }
          }
        }
      }
      if (!ok && lane == 0) {
        *(volatile int*)&abort_flag = 1;
        report_status(p.status, kStatusTimeout);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int D>
cudaError_t launch_d(const AttnParams& p, cudaStream_t stream) {
  const int smem = (int)AttnSmem<D>::total + 1024;
  auto kern = attn_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)p.n_items * p.heads;
  if (grid <= 0) return cudaSuccess;
  launch_k(kern, (unsigned)grid, kThreads, smem, stream, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const AttnParams& p, int head_dim, cudaStream_t stream) {
  if (head_dim == 128) return launch_d<128>(p, stream);
  if (head_dim == 64) return launch_d<64>(p, stream);
  return cudaErrorInvalidValue;
}

MF_BOUNDS_EXPORT(attention)

}  // namespace mf
