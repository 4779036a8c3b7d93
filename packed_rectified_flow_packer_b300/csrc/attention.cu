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
//   warp 0 lane 0 : TMA producer (Q once, then K/V tiles into a 2-deep ring)
//   warp 1        : TMEM allocator; lane 0 issues tcgen05.mma
//                   S_j = Q K_j^T  into TMEM (two S buffers, so S_{j+1} overlaps softmax j)
//                   O  += P_j V_j  into TMEM (V is the MN-major B operand)
//   warps 2..5    : softmax, one thread per query row: S from TMEM, online max / sum in f32
//                   with exp2, P in bf16 to shared memory (128-byte swizzled, K-major), and
//                   the final O / l to global memory in stream-sorted order.
// The running max is only moved (and O rescaled in TMEM) when a tile's max exceeds it by
// more than 8 in log2 units; the result is unchanged because numerator and denominator use
// the same stale max, and P stays <= 2^8.
#include "attention.cuh"

namespace mf {
namespace {

constexpr int kT = 128;             // query rows and key rows per tile
constexpr uint32_t kAtom = 16384;   // 128 rows x 128 bytes
constexpr float kRescaleLog2 = 8.0f;

template <int D>
struct AttnSmem {
  static constexpr uint32_t Q = kT * D * 2;
  static constexpr uint32_t KV = kT * D * 2;
  static constexpr uint32_t P = kT * kT * 2;
  static constexpr uint32_t off_q = 0;
  static constexpr uint32_t off_k = Q;
  static constexpr uint32_t off_v = off_k + 2 * KV;
  static constexpr uint32_t off_p = off_v + 2 * KV;
  static constexpr uint32_t total = off_p + 2 * P;
};

template <int D>
__global__ void __launch_bounds__(192, 1) attn_kernel(const __grid_constant__ AttnParams p) {
  using L = AttnSmem<D>;
  constexpr uint32_t IDESC_S = idesc_bf16_f32(kT, kT, false);
  constexpr uint32_t IDESC_PV = idesc_bf16_f32(kT, D, true);
  constexpr uint32_t TMEM_COLS = 512;  // S0 @0, S1 @128, O @256
  constexpr uint32_t O_COL = 256;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t q_full, kv_full[2], kv_empty[2], s_full[2], s_free[2], p_full[2], o_ready,
      drain_bar;
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
    for (int b = 0; b < 2; ++b) {
      mbar_init(&kv_full[b], 1);
      mbar_init(&kv_empty[b], 1);
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 128);
      mbar_init(&p_full[b], 128);
    }
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
      uint32_t armed = 0, armed_par = 0;
      mbar_arrive_expect_tx(&q_full, L::Q);
#pragma unroll
      for (int a = 0; a < D / 64; ++a)
        tma_load_2d(smem + L::off_q + a * kAtom, &p.tmQ, h * D + a * 64, q0, &q_full);
      for (int j = 0; j < n_kv; ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(&kv_empty[st], ph ^ 1, lim) || *(volatile int*)&abort_flag) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&kv_full[st], 2 * L::KV);
#pragma unroll
        for (int a = 0; a < D / 64; ++a) {
          tma_load_2d(smem + L::off_k + st * L::KV + a * kAtom, &p.tmK, h * D + a * 64, kv0 + j * kT,
                      &kv_full[st]);
          tma_load_2d(smem + L::off_v + st * L::KV + a * kAtom, &p.tmV, h * D + a * 64, kv0 + j * kT,
                      &kv_full[st]);
        }
        armed |= 1u << st;
        armed_par = (armed_par & ~(1u << st)) | (ph << st);
      }
      if (!ok) {
        *(volatile int*)&abort_flag = 1;
        report_status(p.status, kStatusTimeout);
        mbar_wait(&q_full, 0, lim);
        for (int s = 0; s < 2; ++s)
          if (armed & (1u << s)) mbar_wait(&kv_full[s], (armed_par >> s) & 1u, lim);
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
          const int st = j & 1;
          const uint32_t ph = (j >> 1) & 1;
          if (!mbar_wait(&kv_full[st], ph, lim) || !mbar_wait(&s_free[st], ph ^ 1, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ka = smem_u32(smem + L::off_k + st * L::KV);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t o = (kk >> 2) * kAtom + (kk & 3) * 32;
            mma_bf16(tmem_base + st * kT, sdesc_sw128(qa + o, 16, 1024), sdesc_sw128(ka + o, 16, 1024),
                     IDESC_S, kk > 0 ? 1u : 0u);
          }
          mma_commit(&s_full[st]);
        }
        if (j >= 1) {
          const int i = j - 1;
          const int st = i & 1;
          const uint32_t ph = (i >> 1) & 1;
          if (!mbar_wait(&p_full[st], ph, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t pa = smem_u32(smem + L::off_p + st * L::P);
          const uint32_t va = smem_u32(smem + L::off_v + st * L::KV);
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk) {
            const uint32_t o = (kk >> 2) * kAtom + (kk & 3) * 32;
            mma_bf16(tmem_base + O_COL, sdesc_sw128(pa + o, 16, 1024),
                     sdesc_sw128(va + kk * 2048, kAtom, 1024), IDESC_PV, (i > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&kv_empty[st]);
          mma_commit(&o_ready);
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
      const int st = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[st], ph, lim)) &&
           !__any_sync(0xffffffffu, *(volatile int*)&abort_flag);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(lane_base + st * kT + cc * 32, sr[cc]);
      tmem_ld_wait();
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_reg_fence(sr[cc]);
      tc_fence_before();
      mbar_arrive(&s_free[st]);

      const int valid = len - j * kT;  // key columns of this tile inside the sample
      if (valid < kT) {
#pragma unroll
        for (int i = 0; i < kT; ++i)
          if (i >= valid) sr[i >> 5][i & 31] = __float_as_uint(-INFINITY);
      }
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < kT; ++i) mx = fmaxf(mx, __uint_as_float(sr[i >> 5][i & 31]));
      const float m_tile = mx * c;
      if (j == 0) {
        m = m_tile;
      } else {
        const bool need = m_tile > m + kRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {
          const float alpha = need ? ex2_approx(m - m_tile) : 1.0f;
          // O must hold P_{j-1} V_{j-1} before it is rescaled
          ok = __all_sync(0xffffffffu, mbar_wait(&o_ready, (uint32_t)((j - 1) & 1), lim));
          if (!ok) break;
          tc_fence_after();
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
          l *= alpha;
          if (need) m = m_tile;
        }
      }
      // P_j = exp2(S * c - m) -> bf16, 128-byte swizzled K-major tile (two 64-column atoms).
      // The buffer's previous reader P_{j-2} V_{j-2} finished before S_j was signalled.
      uint8_t* pbuf = smem + L::off_p + st * L::P;
      const float neg_m = -m;
      float lsum = 0.0f;
#pragma unroll
      for (int c8 = 0; c8 < kT / 8; ++c8) {
        float e[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          e[u] = ex2_approx(fmaf(__uint_as_float(sr[(c8 * 8 + u) >> 5][(c8 * 8 + u) & 31]), c, neg_m));
          lsum += e[u];
        }
        uint4 w;
        w.x = pack_bf16x2(e[0], e[1]);
        w.y = pack_bf16x2(e[2], e[3]);
        w.z = pack_bf16x2(e[4], e[5]);
        w.w = pack_bf16x2(e[6], e[7]);
        const int atom = c8 >> 3, chunk = c8 & 7;
        *reinterpret_cast<uint4*>(pbuf + atom * kAtom + row * 128 + ((chunk ^ (row & 7)) << 4)) = w;
      }
      l += lsum;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[st]);
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
