// Varlen joint attention for the packed NR-MMDiT block on sm_103a.
//
// Each packed sample attends only over its own [text | image] tokens (PaperReading review of
// "Mage-Flow: An Efficient Native-Resolution Foundation Model for Image Generation and
// Editing", §2.2 (2): cumulative offsets plus a varlen kernel restricting attention to each
// sample).  Only diagonal blocks are ever scheduled: a work item is (sample, 128-row query
// tile, head) and loops over that sample's own 128-row key tiles, so the cost is
// sum_i L_i^2, not (sum_i L_i)^2.
//
// One CTA per work item, 192 threads:
//   warp 0 lane 0 : TMA producer: Q once, then K and V tiles into two separate rings (K three
//                   deep, V two deep), in the order the tensor core consumes them.  K_j is
//                   released as soon as S_j is computed, so K runs two to three tiles ahead.
//   warp 1        : TMEM allocator; lane 0 issues tcgen05.mma
//                   S_j = Q K_j^T  into TMEM (two S buffers, so S_{j+1} overlaps softmax j)
//                   O  += P_j V_j  into TMEM (V is the MN-major B operand)
//   warps 2..5    : softmax, one thread per query row: S from TMEM, online max / sum in f32
//                   with exp2, P in bf16 to shared memory (128-byte swizzled, K-major), and
//                   the final O / l to global memory in stream-sorted order.
// The running max is only moved (and O rescaled in TMEM) when a tile's max exceeds it by
// more than 8 in log2 units; the result is unchanged because numerator and denominator use
// the same stale max, and P stays <= 2^8.  A quarter of the exponentials run on the FMA pipe
// (exp2_fma) to relieve the special-function unit.
#include "attention.cuh"

namespace mf {
namespace {

constexpr int kT = 128;             // query rows and key rows per tile
constexpr uint32_t kAtom = 16384;   // 128 rows x 128 bytes
constexpr float kRescaleLog2 = 8.0f;
constexpr int kKStages = 3;
constexpr int kVStages = 2;

// 2^x on the FMA pipe: x = n + f with n = floor(x), f in [0, 1); 2^f from a degree-3
// polynomial fitted by us (iteratively reweighted least squares on relative error over
// [0, 1]); n is then added to the result's exponent field.  Max relative error 7.6e-5, far
// inside the bf16 rounding P gets next.  Inputs below -125 give (near) zero.
__device__ __forceinline__ float exp2_fma(float x) {
  x = fmaxf(x, -125.0f);
  const float n = floorf(x);
  const float f = x - n;
  float p = fmaf(0.07802354544401169f, f, 0.22606661915779114f);
  p = fmaf(p, f, 0.6958348155021667f);
  p = fmaf(p, f, 0.9999249577522278f);
  return __int_as_float(__float_as_int(p) + (static_cast<int>(n) << 23));
}

template <int D>
struct AttnSmem {
  static constexpr uint32_t Q = kT * D * 2;
  static constexpr uint32_t KV = kT * D * 2;
  static constexpr uint32_t P = kT * kT * 2;
  static constexpr uint32_t off_q = 0;
  static constexpr uint32_t off_k = Q;
  static constexpr uint32_t off_v = off_k + kKStages * KV;
  static constexpr uint32_t off_p = off_v + kVStages * KV;
  static constexpr uint32_t total = off_p + P;
};

template <int D>
__global__ void __launch_bounds__(192, 1) attn_kernel(const __grid_constant__ AttnParams p) {
  using L = AttnSmem<D>;
  constexpr uint32_t IDESC_S = idesc_bf16_f32(kT, kT, false);
  constexpr uint32_t IDESC_PV = idesc_bf16_f32(kT, D, true);
  constexpr uint32_t TMEM_COLS = 512;  // S0 @0, S1 @128, O @256
  constexpr uint32_t O_COL = 256;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t q_full, k_full[kKStages], k_empty[kKStages], v_full[kVStages],
      v_empty[kVStages], s_full[2], s_free[2], p_full, o_ready, drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  uint8_t* smem = align1024(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t lim = p.wait_limit_ns;

  const int item = blockIdx.x / p.heads;
  const int h = blockIdx.x - item * p.heads;
  const int seq = __ldg(p.items + 2 * item);
  const int qt = __ldg(p.items + 2 * item + 1);
  const int kv0 = __ldg(p.cu + seq);
  const int len = __ldg(p.cu + seq + 1) - kv0;
  const int q0 = kv0 + qt * kT;
  const int n_kv = (len + kT - 1) / kT;

  if (threadIdx.x == 0) {
    mbar_init(&q_full, 1);
    for (int b = 0; b < kKStages; ++b) {
      mbar_init(&k_full[b], 1);
      mbar_init(&k_empty[b], 1);
    }
    for (int b = 0; b < kVStages; ++b) {
      mbar_init(&v_full[b], 1);
      mbar_init(&v_empty[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 128);
    }
    mbar_init(&p_full, 128);
    mbar_init(&o_ready, 1);
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

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      bool ok = true;
      uint32_t k_armed = 0, k_par = 0, v_armed = 0, v_par = 0;
      auto load_k = [&](int j) -> bool {
        const int st = j % kKStages;
        const uint32_t ph = (j / kKStages) & 1;
        if (!mbar_wait(&k_empty[st], ph ^ 1, lim) || *(volatile int*)&abort_flag) return false;
        mbar_arrive_expect_tx(&k_full[st], L::KV);
#pragma unroll
        for (int a = 0; a < D / 64; ++a)
          tma_load_2d(smem + L::off_k + st * L::KV + a * kAtom, &p.tmK, h * D + a * 64, kv0 + j * kT,
                      &k_full[st]);
        k_armed |= 1u << st;
        k_par = (k_par & ~(1u << st)) | (ph << st);
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int st = j % kVStages;
        const uint32_t ph = (j / kVStages) & 1;
        if (!mbar_wait(&v_empty[st], ph ^ 1, lim) || *(volatile int*)&abort_flag) return false;
        mbar_arrive_expect_tx(&v_full[st], L::KV);
#pragma unroll
        for (int a = 0; a < D / 64; ++a)
          tma_load_2d(smem + L::off_v + st * L::KV + a * kAtom, &p.tmV, h * D + a * 64, kv0 + j * kT,
                      &v_full[st]);
        v_armed |= 1u << st;
        v_par = (v_par & ~(1u << st)) | (ph << st);
        return true;
      };
      mbar_arrive_expect_tx(&q_full, L::Q);
#pragma unroll
      for (int a = 0; a < D / 64; ++a)
        tma_load_2d(smem + L::off_q + a * kAtom, &p.tmQ, h * D + a * 64, q0, &q_full);
      // consumption order of the tensor core: S_0, S_1, PV_0, S_2, PV_1, ...
      ok = load_k(0) && (n_kv < 2 || load_k(1));
      for (int j = 0; ok && j < n_kv; ++j) {
        ok = load_v(j) && (j + 2 >= n_kv || load_k(j + 2));
      }
      if (!ok) {
        *(volatile int*)&abort_flag = 1;
        report_status(p.status, kStatusTimeout);
        mbar_wait(&q_full, 0, lim);  // let this thread's copies land before exiting
        for (int s = 0; s < kKStages; ++s)
          if (k_armed & (1u << s)) mbar_wait(&k_full[s], (k_par >> s) & 1u, lim);
        for (int s = 0; s < kVStages; ++s)
          if (v_armed & (1u << s)) mbar_wait(&v_full[s], (v_par >> s) & 1u, lim);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(&q_full, 0, lim);
      const uint32_t qa = smem_u32(smem + L::off_q);
      for (int j = 0; ok && j <= n_kv; ++j) {
        if (*(volatile int*)&abort_flag) { ok = false; break; }
        if (j < n_kv) {
          const int ks = j % kKStages, sb = j & 1;
          if (!mbar_wait(&k_full[ks], (j / kKStages) & 1, lim) ||
              !mbar_wait(&s_free[sb], ((j >> 1) & 1) ^ 1, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ka = smem_u32(smem + L::off_k + ks * L::KV);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t o = (kk >> 2) * kAtom + (kk & 3) * 32;
            mma_bf16(tmem_base + sb * kT, sdesc_sw128(qa + o, 16, 1024), sdesc_sw128(ka + o, 16, 1024),
                     IDESC_S, kk > 0 ? 1u : 0u);
          }
          mma_commit(&s_full[sb]);
          mma_commit(&k_empty[ks]);
        }
        if (j >= 1) {
          const int i = j - 1;
          const int vs = i % kVStages;
          if (!mbar_wait(&v_full[vs], (i / kVStages) & 1, lim) || !mbar_wait(&p_full, i & 1, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t pa = smem_u32(smem + L::off_p);
          const uint32_t va = smem_u32(smem + L::off_v + vs * L::KV);
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk) {
            const uint32_t o = (kk >> 2) * kAtom + (kk & 3) * 32;
            mma_bf16(tmem_base + O_COL, sdesc_sw128(pa + o, 16, 1024),
                     sdesc_sw128(va + kk * 2048, kAtom, 1024), IDESC_PV, (i > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&o_ready);
          mma_commit(&v_empty[vs]);
        }
      }
      if (!ok) {
        *(volatile int*)&abort_flag = 1;
        report_status(p.status, kStatusTimeout);
        mma_commit(&drain_bar);
        mbar_wait(&drain_bar, 0, lim);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax warps
    const int qw = warp & 3;
    const int row = qw * 32 + lane;  // query row inside the tile = TMEM lane
    const uint32_t lane_base = tmem_addr(tmem_base, qw * 32, 0);
    const float c = p.scale_log2;
    float m = -INFINITY;  // running max, log2 units
    float l = 0.0f;       // running sum of P
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int sb = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[sb], (j >> 1) & 1, lim)) &&
           !__any_sync(0xffffffffu, *(volatile int*)&abort_flag);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(lane_base + sb * kT + cc * 32, sr[cc]);
      tmem_ld_wait();
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_reg_fence(sr[cc]);
      tc_fence_before();
      mbar_arrive(&s_free[sb]);

      const int valid = len - j * kT;  // key columns of this tile inside the sample
      if (valid < kT) {
#pragma unroll
        for (int i = 0; i < kT; ++i)
          if (i >= valid) sr[i >> 5][i & 31] = __float_as_uint(-INFINITY);
      }
      float mx[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx[u] = __uint_as_float(sr[0][u]);
#pragma unroll
      for (int i = 8; i < kT; ++i) mx[i & 7] = fmaxf(mx[i & 7], __uint_as_float(sr[i >> 5][i & 31]));
      const float m_tile =
          fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * c;
      const bool need = (j == 0) || (m_tile > m + kRescaleLog2);
      const float alpha = (j > 0 && need) ? ex2_approx(m - m_tile) : 1.0f;
      if (need) m = m_tile;

      // P_j = exp2(S c - m), kept in registers (in place of S) until the buffer is free
      const float neg_m = -m;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < kT; ++i) {
        const float a = fmaf(__uint_as_float(sr[i >> 5][i & 31]), c, neg_m);
        const float e = ((i & 3) == 3) ? exp2_fma(a) : ex2_approx(a);
        ls[i & 3] += e;
        sr[i >> 5][i & 31] = __float_as_uint(e);
      }
      if (valid < kT) {  // masked columns: exactly zero (the FMA path leaves a tiny value)
        ls[0] = ls[1] = ls[2] = ls[3] = 0.f;
#pragma unroll
        for (int i = 0; i < kT; ++i) {
          if (i >= valid) sr[i >> 5][i & 31] = 0u;
          ls[i & 3] += __uint_as_float(sr[i >> 5][i & 31]);
        }
      }
      if (j > 0) {
        // O += P_{j-1} V_{j-1} must be done before P's buffer is rewritten or O rescaled
        ok = __all_sync(0xffffffffu, mbar_wait(&o_ready, (uint32_t)((j - 1) & 1), lim));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t r[32];
            tmem_ld32(lane_base + O_COL + cc * 32, r);
            tmem_ld_wait();
            tmem_reg_fence(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(lane_base + O_COL + cc * 32, r);
          }
          tmem_st_wait();
        }
      }
      l = l * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
      // bf16, 128-byte swizzled K-major tile (two 64-column atoms)
      uint8_t* pbuf = smem + L::off_p;
#pragma unroll
      for (int c8 = 0; c8 < kT / 8; ++c8) {
        const uint32_t* e = &sr[(c8 * 8) >> 5][(c8 * 8) & 31];
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(e[0]), __uint_as_float(e[1]));
        w.y = pack_bf16x2(__uint_as_float(e[2]), __uint_as_float(e[3]));
        w.z = pack_bf16x2(__uint_as_float(e[4]), __uint_as_float(e[5]));
        w.w = pack_bf16x2(__uint_as_float(e[6]), __uint_as_float(e[7]));
        const int atom = c8 >> 3, chunk = c8 & 7;
        *reinterpret_cast<uint4*>(pbuf + atom * kAtom + row * 128 + ((chunk ^ (row & 7)) << 4)) = w;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full);
    }
    if (ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(&o_ready, (uint32_t)((n_kv - 1) & 1), lim));
      if (ok) {
        tc_fence_after();
        const float inv_l = 1.0f / l;
        const int qrow = q0 + row;
        const bool valid = qrow < kv0 + len;
        bf16* dst = valid ? p.out + (size_t)__ldg(p.joint_srow + qrow) * p.H + h * D : nullptr;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t r[32];
          tmem_ld32(lane_base + O_COL + cc * 32, r);
          tmem_ld_wait();
          tmem_reg_fence(r);
          if (valid) {
            uint4* o = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(r[8 * i + 0]) * inv_l, __uint_as_float(r[8 * i + 1]) * inv_l);
              w.y = pack_bf16x2(__uint_as_float(r[8 * i + 2]) * inv_l, __uint_as_float(r[8 * i + 3]) * inv_l);
              w.z = pack_bf16x2(__uint_as_float(r[8 * i + 4]) * inv_l, __uint_as_float(r[8 * i + 5]) * inv_l);
              w.w = pack_bf16x2(__uint_as_float(r[8 * i + 6]) * inv_l, __uint_as_float(r[8 * i + 7]) * inv_l);
              o[i] = w;
            }
          }
        }
      }
    }
    if (!ok && lane == 0) {
      *(volatile int*)&abort_flag = 1;
      report_status(p.status, kStatusTimeout);
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
  kern<<<(unsigned)grid, 192, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const AttnParams& p, int head_dim, cudaStream_t stream) {
  if (head_dim == 128) return launch_d<128>(p, stream);
  if (head_dim == 64) return launch_d<64>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace mf
