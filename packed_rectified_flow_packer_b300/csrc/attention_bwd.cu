// Backward of the varlen joint attention on sm_103a.
//
// Forward, per packed sample and head (PaperReading review of "Mage-Flow: An Efficient
// Native-Resolution Foundation Model for Image Generation and Editing", §2.2 (2): attention
// restricted to each sample): s = q k^T / sqrt(D), P = softmax(s), o = P v.  Given do = dL/do
// and the forward's per-row logsumexp lse, the gradients are
//   P  = exp(s - lse)               (recomputed, no L x L storage)
//   dv = P^T do,   dP = do v^T,   delta = rowsum(do * o),   ds = P * (dP - delta)
//   dq = ds k / sqrt(D),   dk = ds^T q / sqrt(D).
// Only diagonal blocks exist: a CTA owns one 128-row key block of one sample and one head and
// loops over that sample's own 64-row query tiles, so the work is sum_i L_i^2.
//
// Three kernels:
//   attn_bwd_prep_kernel : per joint row, do gathered into joint order, delta per head, and the
//                          f32 dq accumulator row cleared;
//   attn_bwd_kernel      : the tcgen05 loop below;
//   attn_bwd_dq_kernel   : dq accumulator (f32, already scaled) to bf16.
//
// attn_bwd_kernel: one CTA per (sample, 128-key block, head), 320 threads, key blocks fastest,
// then heads, samples longest first.  Everything is computed transposed (keys on the TMEM
// lanes), so the key-side accumulators dV, dK stay in TMEM for the whole loop:
//   S^T  = K Q_i^T                    [128 keys x 64 queries]   (A = K, B = Q_i, both K-major)
//   P^T  = exp2(S^T log2e/sqrt(D) - lse2_i)  in f32 registers, bf16 copy into TMEM over S^T
//                                     (each warpgroup's 32 queries over the first 16 of its
//                                     own 32 columns)
//   dV  += P^T dO_i                   (A = P^T from TMEM, B = dO_i MN-major)
//   dP^T = V dO_i^T                   [128 x 64]
//   dS^T = P^T * (dP^T - delta_i)     bf16, written to one of two shared-memory buffers
//   dK  += dS^T Q_i                   (A = dS^T K-major, B = Q_i MN-major)
//   dQ_i^T = K^T dS                   [D x 64]  (A = K MN-major, B = dS^T read MN-major)
// S^T has two TMEM buffers and dP^T is computed one tile ahead, so the tensor core has queued
// work while the P / dS warps run.  Four warps read dQ_i^T (lane = head dimension), stage it
// in shared memory and add it into the f32 dq accumulator with TMA reduce-adds.
// Warp roles (448 threads): 0 TMA producer (K, V once; Q_i, dO_i per tile, plus lse_i and
// delta_i copied by the warp's lanes), 1 TMEM allocator and MMA issuer (warp-uniform loop, one
// elected lane issues), 2..5 and 10..13 the two P / dS warpgroups (thread = key row, each
// warpgroup half of the tile's query columns), 6..9 the dQ warpgroup.
// TMEM (512 columns): S^T/P^T @0 and @64, dP^T @128, dV @192 (128), dK @320 (128), dQ^T @448.
// Head dim 64 runs the same code with the head dim padded to 128: the upper half of every K
// and V tile is zero (so S^T and dP^T are unchanged) and the padded dV / dK / dQ columns are
// never stored.
#include "attention_bwd.cuh"
#include "internal.h"

namespace mf {
namespace {

constexpr int kKeys = 128;         // key rows per CTA (TMEM lanes)
constexpr int kQT = 64;            // query rows per tile
constexpr int kDP = 128;           // padded head dim inside the kernel
constexpr int kThreads = 448;     // producer, MMA, 4 dQ warps, 8 P / dS warps
constexpr int kStages = 3;
constexpr uint32_t kKVBytes = kKeys * kDP * 2;          // 32 KB: two 16 KB atoms of 128 rows
constexpr uint32_t kKVAtom = kKeys * 128;               // 16 KB
constexpr uint32_t kQTBytes = kQT * kDP * 2;            // 16 KB: two 8 KB atoms of 64 rows
constexpr uint32_t kQTAtom = kQT * 128;                 // 8 KB
constexpr uint32_t kStageBytes = 2 * kQTBytes + 1024;   // Q_i, dO_i, lse2_i[64], delta_i[64]
constexpr uint32_t kDSBytes = kKeys * kQT * 2;          // 16 KB: dS^T [128 keys][64 queries]
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kKVBytes;
constexpr uint32_t kOffStage = 2 * kKVBytes;
constexpr uint32_t kOffDS = kOffStage + kStages * kStageBytes;
constexpr uint32_t kOffDq = kOffDS + 2 * kDSBytes;
constexpr uint32_t kDqStage = 32 * 32 * 4;              // 4 KB per dQ warp: [32 queries][32 dims]
constexpr uint32_t kSmemTotal = kOffDq + 4 * kDqStage;

// TMEM columns: S^T / P^T double buffer, dP^T, the dV and dK accumulators, dQ^T.
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 192, kColDK = 320, kColDQ = 448;

// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// (sample, head, key block) of this CTA: samples in work-list order (longest first, each
// sample's query blocks contiguous), key blocks fastest, then heads.
__device__ __forceinline__ void decode_cta(const AttnBwdParams& p, int& kv0, int& len, int& h, int& kb) {
  int base = 0;
  kv0 = 0;
  len = 0;
  int nkb = 1;
  for (int it = 0; it < p.n_items;) {
    const int seq = __ldg(p.items + 2 * it);
    if (!MF_IDX_OK(seq >= 0 && seq < p.n_seq)) { len = 0; return; }
    kv0 = __ldg(p.cu + seq);
    len = __ldg(p.cu + seq + 1) - kv0;
    if (!MF_IDX_OK(len > 0)) return;
    nkb = (len + kKeys - 1) / kKeys;
    if ((int)blockIdx.x < base + nkb * p.heads) break;
    base += nkb * p.heads;
    it += (len + kQBlock - 1) / kQBlock;  // the work list's items of this sample
  }
  h = ((int)blockIdx.x - base) / nkb;
  kb = ((int)blockIdx.x - base) - h * nkb;
}

// Issue order of the MMA warp, per query tile i (b = i & 1):
//   [P_i ready]   dP_{i+1} = V dO_{i+1}^T (the P / dS warps load dP_i together with S_i, before
//                 computing P_i), then dV += P_i^T dO_i
//   [dS_i ready]  dK += dS_i^T Q_i, [dQ drained] dQ_i^T = K^T dS_i, then S_{i+2} into the S^T
//                 buffer b that dV just finished reading.
// So a tile's S^T and dP^T are both in TMEM when the P / dS warps reach it, and the tensor
// core has the next products queued while the exponentials and dS of a tile run.
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_kernel(const __grid_constant__ AttnBwdParams p) {
  constexpr uint32_t IDESC_S = idesc_bf16_f32_mn(kKeys, kQT, false, false);   // S^T, dP^T
  constexpr uint32_t IDESC_KV = idesc_bf16_f32_mn(kKeys, kDP, false, true);   // dV, dK
  constexpr uint32_t IDESC_DQ = idesc_bf16_f32_mn(kDP, kQT, true, true);      // dQ^T
  constexpr uint32_t TMEM_COLS = 512;

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t kv_full, full[kStages], empty[kStages], s_full[2], p_full[2], dp_full, ds_full;
  __shared__ uint64_t ds_free[2], dq_full, dq_free, done_bar, drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  uint8_t* smem = align1024(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t lim = p.wait_limit_ns;
  const int Dr = p.head_dim;  // 64 or 128

  int kv0, len, h, kb;
  decode_cta(p, kv0, len, h, kb);
  if (!MF_IDX_OK(kv0 >= 0 && len > 0 && kv0 + len <= p.n_tok && h < p.heads)) return;  // before any barrier
  const int k0 = kv0 + kb * kKeys;          // first key row (joint) of this CTA
  const int n_q = (len + kQT - 1) / kQT;    // query tiles of the sample

  if (Dr < kDP) {
    // head dim 64: zero the upper half (second atom) of K, V and of every stage's Q and dO
    // tile once; the TMA loads only ever fill the lower half
    uint4 z = make_uint4(0, 0, 0, 0);
    for (uint32_t i = threadIdx.x; i < kKVAtom / 16; i += blockDim.x) {
      reinterpret_cast<uint4*>(smem + kOffK + kKVAtom)[i] = z;
      reinterpret_cast<uint4*>(smem + kOffV + kKVAtom)[i] = z;
    }
    for (int st = 0; st < kStages; ++st)
      for (uint32_t i = threadIdx.x; i < kQTAtom / 16; i += blockDim.x) {
        reinterpret_cast<uint4*>(smem + kOffStage + st * kStageBytes + kQTAtom)[i] = z;
        reinterpret_cast<uint4*>(smem + kOffStage + st * kStageBytes + kQTBytes + kQTAtom)[i] = z;
      }
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 0) {
    mbar_init(&kv_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 2);  // the producer's expect-tx arrival + its lse / delta arrival
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 256);
      mbar_init(&ds_free[b], 1);
    }
    mbar_init(&dp_full, 1);
    mbar_init(&ds_full, 256);
    mbar_init(&dq_full, 1);
    mbar_init(&dq_free, 128);
    mbar_init(&done_bar, 1);
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
  auto stage_ptr = [&](int st) { return smem + kOffStage + st * kStageBytes; };

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    const uint32_t el = elect_one();
    const int natoms = Dr / 64;
    if (el) {
      tma_prefetch_desc(&p.tmK);
      tma_prefetch_desc(&p.tmV);
      tma_prefetch_desc(&p.tmQ);
      tma_prefetch_desc(&p.tmDO);
      mbar_arrive_expect_tx(&kv_full, 2u * natoms * kKVAtom);
      for (int a = 0; a < natoms; ++a) {
        tma_load_2d(smem + kOffK + a * kKVAtom, &p.tmK, h * Dr + a * 64, k0, &kv_full);
        tma_load_2d(smem + kOffV + a * kKVAtom, &p.tmV, h * Dr + a * 64, k0, &kv_full);
      }
    }
    __syncwarp();
    bool ok = true;
    uint32_t armed = 0, armed_par = 0;
    const float* lse_h = p.lse + (size_t)h * p.n_tok + kv0;
    const float* dl_h = p.delta + (size_t)h * p.n_tok + kv0;
    // lse (log2 units) and delta of tile i's 64 query rows, two per lane, loaded one tile ahead
    // so their latency overlaps the wait for the stage; rows past the sample get lse = +inf
    // (so P = 0 there) and delta = 0
    float nl[2], nd[2];
    auto load_rows = [&](int i) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int q = i * kQT + lane + 32 * u;
        nl[u] = q < len ? __ldg(lse_h + q) * 1.4426950408889634f : INFINITY;
        nd[u] = q < len ? __ldg(dl_h + q) : 0.0f;
      }
    };
    load_rows(0);
    for (int i = 0; ok && i < n_q; ++i) {
      const int st = i % kStages;
      const uint32_t ph = (i / kStages) & 1;
      uint32_t okw = 1;
      if (lane == 0) okw = mbar_wait(&empty[st], ph ^ 1, lim) && !*(volatile int*)&abort_flag ? 1u : 0u;
      if (__shfl_sync(0xffffffffu, okw, 0) == 0) {
        ok = false;
        break;
      }
      uint8_t* sp = stage_ptr(st);
      if (el) {
        mbar_arrive_expect_tx(&full[st], 2u * natoms * kQTAtom);
        for (int a = 0; a < natoms; ++a) {
          tma_load_2d(sp + a * kQTAtom, &p.tmQ, h * Dr + a * 64, kv0 + i * kQT, &full[st]);
          tma_load_2d(sp + kQTBytes + a * kQTAtom, &p.tmDO, h * Dr + a * 64, kv0 + i * kQT, &full[st]);
        }
        // the next tile into L2 while its stage is still in use, so its load starts from L2
        if (i + 1 < n_q)
          for (int a = 0; a < natoms; ++a) {
            tma_prefetch_l2_2d(&p.tmQ, h * Dr + a * 64, kv0 + (i + 1) * kQT);
            tma_prefetch_l2_2d(&p.tmDO, h * Dr + a * 64, kv0 + (i + 1) * kQT);
          }
      }
      armed |= 1u << st;
      armed_par = (armed_par & ~(1u << st)) | (ph << st);
      float* l2s = reinterpret_cast<float*>(sp + 2 * kQTBytes);
      float* dls = l2s + kQT;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        l2s[lane + 32 * u] = nl[u];
        dls[lane + 32 * u] = nd[u];
      }
      if (i + 1 < n_q) load_rows(i + 1);
      __syncwarp();
      if (el) mbar_arrive(&full[st]);
      __syncwarp();
    }
    if (!ok) {
      if (el) {
        *(volatile int*)&abort_flag = 1;
        report_status(p.status, kStatusTimeout);
      }
      mbar_wait(&kv_full, 0, lim);  // let this warp's copies land before exiting
      for (int s2 = 0; s2 < kStages; ++s2)
        if (armed & (1u << s2)) mbar_wait(&full[s2], (armed_par >> s2) & 1u, lim);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    const uint32_t el = elect_one();
    // every lane polls: a completed phase is seen by each lane's own try_wait, with no shuffle
    // and warp barrier between the barrier and the next issue
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, lim));
    };
    const uint32_t k_addr = smem_u32(smem + kOffK), v_addr = smem_u32(smem + kOffV);
    // K-major operands step 32 bytes per K = 16 (descriptor +2); MN-major ones 16 rows (+128)
    constexpr uint64_t kStepK = 2, kStepMN = 2048 >> 4;
    const uint64_t k_desc_mn = sdesc_sw128(k_addr, kKVAtom, 1024);   // K as the MN-major A of dQ^T
    // S^T (or dP^T) = A B^T: A = K (V) K-major [128 rows][128 dims], B = Q_i (dO_i) K-major;
    // the two 64-dim halves live in separate atoms
    auto issue_rowdot = [&](uint32_t a_addr, uint32_t b_addr, uint32_t d_col) {
      mma_group_ss<4>(el, tmem_base + d_col, sdesc_sw128(a_addr, 16, 1024), kStepK, sdesc_sw128(b_addr, 16, 1024),
                      kStepK, IDESC_S, 0u);
      mma_group_ss<4>(el, tmem_base + d_col, sdesc_sw128(a_addr + kKVAtom, 16, 1024), kStepK,
                      sdesc_sw128(b_addr + kQTAtom, 16, 1024), kStepK, IDESC_S, 1u);
    };
    auto stage_wait = [&](int i) { return wait_all(&full[i % kStages], (i / kStages) & 1); };
    // prologue: S_0, S_1 into both S^T buffers, dP_0
    bool ok = wait_all(&kv_full, 0) && stage_wait(0);
    if (ok) {
      tc_fence_after();
      issue_rowdot(k_addr, smem_u32(stage_ptr(0)), kColS);
      mma_commit_if(el, &s_full[0]);
      issue_rowdot(v_addr, smem_u32(stage_ptr(0)) + kQTBytes, kColDP);
      mma_commit_if(el, &dp_full);
      if (n_q > 1) {
        ok = stage_wait(1);
        if (ok) {
          tc_fence_after();
          issue_rowdot(k_addr, smem_u32(stage_ptr(1)), kColS + kQT);
          mma_commit_if(el, &s_full[1]);
        }
      }
    }
    for (int i = 0; ok && i < n_q; ++i) {
      const int st = i % kStages, b = i & 1;
      const uint32_t q_addr = smem_u32(stage_ptr(st));
      const uint32_t do_addr = q_addr + kQTBytes;
      const uint32_t ds_addr = smem_u32(smem + kOffDS + b * kDSBytes);
      // P_i is in TMEM and the P / dS warps hold dP_i in registers: dP_{i+1} may overwrite
      // dP_i (its stage was waited for when S_{i+1} was issued), then dV += P_i^T dO_i
      if (!wait_all(&p_full[b], (i >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      if (i + 1 < n_q) {
        issue_rowdot(v_addr, smem_u32(stage_ptr((i + 1) % kStages)) + kQTBytes, kColDP);
        mma_commit_if(el, &dp_full);
      }
      // P^T of queries 0..31 sits in columns 0..15 of the S^T buffer, queries 32..63 in 32..47
      mma_group2_ts(el, tmem_base + kColDV, tmem_base + kColS + b * kQT, 8, sdesc_sw128(do_addr, kQTAtom, 1024),
                    kStepMN, IDESC_KV, i > 0 ? 1u : 0u);
      mma_group2_ts(el, tmem_base + kColDV, tmem_base + kColS + b * kQT + 32, 8,
                    sdesc_sw128(do_addr + 2 * 2048, kQTAtom, 1024), kStepMN, IDESC_KV, 1u);
      // dK += dS_i^T Q_i, dQ_i^T = K^T dS_i
      if (!wait_all(&ds_full, i & 1)) { ok = false; break; }
      tc_fence_after();
      mma_group_ss<4>(el, tmem_base + kColDK, sdesc_sw128(ds_addr, 16, 1024), kStepK,
                      sdesc_sw128(q_addr, kQTAtom, 1024), kStepMN, IDESC_KV, i > 0 ? 1u : 0u);
      // dK_i is the stage's last reader (S_i, dP_i, dV_i before it; lse / delta were read before
      // dS_i was released): the producer may refill it while dQ_i waits and runs
      mma_commit_if(el, &empty[st]);
      if (i >= 1 && !wait_all(&dq_free, (i - 1) & 1)) { ok = false; break; }
      tc_fence_after();
      mma_group_ss<8>(el, tmem_base + kColDQ, k_desc_mn, kStepMN, sdesc_sw128(ds_addr, kKVAtom, 1024), kStepMN,
                      IDESC_DQ, 0u);
      mma_commit_if(el, &dq_full);
      mma_commit_if(el, &ds_free[b]);
      // S_{i+2} into buffer b (its P_i was read by the dV above)
      if (i + 2 < n_q) {
        if (!stage_wait(i + 2)) { ok = false; break; }
        tc_fence_after();
        issue_rowdot(k_addr, smem_u32(stage_ptr((i + 2) % kStages)), kColS + b * kQT);
        mma_commit_if(el, &s_full[b]);
      }
    }
    if (ok) {
      mma_commit_if(el, &done_bar);
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
  } else if (warp < 6 || warp >= 10) {
    // ---------------------------------------------------------------- P / dS warpgroups
    // Two warpgroups on the same key rows: warps 2..5 take the tile's query columns 0..31,
    // warps 10..13 columns 32..63.
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;                  // key row inside the block = TMEM lane
    const int c0 = warp >= 10 ? 32 : 0;            // this warpgroup's query columns c0 .. c0 + 31
    const bool kvalid = kb * kKeys + r < len;
    const uint32_t lane_base = tmem_addr(tmem_base, q4 * 32, 0);
    const float c = p.scale_log2;
    bool ok = true;
    // every lane polls: a completed phase is seen by each lane's own try_wait
    auto poll = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, lim));
    };
    for (int i = 0; i < n_q; ++i) {
      const int b = i & 1;
      uint8_t* sp = stage_ptr(i % kStages);
      const float* l2s = reinterpret_cast<const float*>(sp + 2 * kQTBytes);
      const float* dls = l2s + kQT;
      // the producer's lse / delta writes are acquired from the stage's own barrier (complete
      // already: S^T of this tile was computed from the same stage); S_i and dP_i are both in
      // TMEM by now (dP_i was issued one tile ahead) and are read together
      if (!(ok = poll(&full[i % kStages], (i / kStages) & 1) && poll(&s_full[b], (i >> 1) & 1) &&
                 poll(&dp_full, i & 1)))
        break;
      tc_fence_after();
      uint32_t sr[32], dr[32];
      tmem_ld32(lane_base + kColS + b * kQT + c0, sr);
      tmem_ld32(lane_base + kColDP + c0, dr);
      tmem_ld_wait();
      tmem_reg_fence(sr);
      tmem_reg_fence(dr);
      float pv[32];
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(l2s + c0 + j);
        pv[j + 0] = ex2_approx(fmaf(__uint_as_float(sr[j + 0]), c, -l4.x));
        pv[j + 1] = ex2_approx(fmaf(__uint_as_float(sr[j + 1]), c, -l4.y));
        pv[j + 2] = ex2_approx(fmaf(__uint_as_float(sr[j + 2]), c, -l4.z));
        pv[j + 3] = ex2_approx(fmaf(__uint_as_float(sr[j + 3]), c, -l4.w));
      }
      if (!kvalid) {
#pragma unroll
        for (int j = 0; j < 32; ++j) pv[j] = 0.0f;
      }
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(pv[2 * j], pv[2 * j + 1]);
      // P^T in bf16, two queries per column, over the first half of the S^T columns this
      // warpgroup read itself (the other warpgroup may still be reading its own)
      tmem_st16(lane_base + kColS + b * kQT + c0, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[b]);  // also releases the dP^T columns (read above)

      if (i >= 2 && !(ok = poll(&ds_free[b], ((i >> 1) & 1) ^ 1))) break;
      // dS^T row r over this warpgroup's queries, bf16, into dS buffer b (128-byte swizzle:
      // K-major for dK += dS^T Q_i, read MN-major by dQ^T = K^T dS)
      uint8_t* ds_row = smem + kOffDS + b * kDSBytes + r * 128;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const int j0 = ch * 8;
        const float4 d0 = *reinterpret_cast<const float4*>(dls + c0 + j0);
        const float4 d1 = *reinterpret_cast<const float4*>(dls + c0 + j0 + 4);
        const uint32_t* dp = &dr[j0];
        uint4 w;
        w.x = pack_bf16x2(pv[j0 + 0] * (__uint_as_float(dp[0]) - d0.x), pv[j0 + 1] * (__uint_as_float(dp[1]) - d0.y));
        w.y = pack_bf16x2(pv[j0 + 2] * (__uint_as_float(dp[2]) - d0.z), pv[j0 + 3] * (__uint_as_float(dp[3]) - d0.w));
        w.z = pack_bf16x2(pv[j0 + 4] * (__uint_as_float(dp[4]) - d1.x), pv[j0 + 5] * (__uint_as_float(dp[5]) - d1.y));
        w.w = pack_bf16x2(pv[j0 + 6] * (__uint_as_float(dp[6]) - d1.z), pv[j0 + 7] * (__uint_as_float(dp[7]) - d1.w));
        const int chunk = c0 / 8 + ch;
        *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (r & 7)) << 4)) = w;
      }
      fence_proxy_async_smem();
      mbar_arrive(&ds_full);
    }
    if (ok) ok = poll(&done_bar, 0);
    if (ok) {
      tc_fence_after();
      // dV (first warpgroup) or dK (second, scaled by 1 / sqrt(D)) of this thread's key row,
      // real head dims only
      const int key = k0 + r;
      {
        const int part = c0 ? 1 : 0;
        const uint32_t col = part ? kColDK : kColDV;
        const float sc = part ? p.scale : 1.0f;
        bf16* dst = (part ? p.dk : p.dv) + (size_t)key * p.H + h * Dr;
#pragma unroll 1
        for (int cc = 0; cc < kDP / 32; ++cc) {
          uint32_t v[32];
          tmem_ld32(lane_base + col + cc * 32, v);
          tmem_ld_wait();
          tmem_reg_fence(v);
          if (kvalid && cc * 32 < Dr) {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(v[8 * g + 0]) * sc, __uint_as_float(v[8 * g + 1]) * sc);
              w.y = pack_bf16x2(__uint_as_float(v[8 * g + 2]) * sc, __uint_as_float(v[8 * g + 3]) * sc);
              w.z = pack_bf16x2(__uint_as_float(v[8 * g + 4]) * sc, __uint_as_float(v[8 * g + 5]) * sc);
              w.w = pack_bf16x2(__uint_as_float(v[8 * g + 6]) * sc, __uint_as_float(v[8 * g + 7]) * sc);
              reinterpret_cast<uint4*>(dst + cc * 32)[g] = w;
            }
          }
        }
      }
    }
    if (!ok && lane == 0) {
      *(volatile int*)&abort_flag = 1;
      report_status(p.status, kStatusTimeout);
    }
  } else {
    // ---------------------------------------------------------------- dQ warpgroup
    // Lane = head dim d (TMEM lane).  The tile's 64 queries leave in two halves: a warp stages
    // [32 queries][32 dims] f32 and one lane adds the box into the f32 accumulator with a TMA
    // reduce; rows past the sample hold exact zeros (and rows past the pack are clipped).
    const int q4 = warp & 3;
    const uint32_t lane_base = tmem_addr(tmem_base, q4 * 32, 0);
    const bool real = q4 * 32 < Dr;
    float* stg = reinterpret_cast<float*>(smem + kOffDq + (warp - 6) * kDqStage);
    const uint32_t el = elect_one();
    bool ok = true;
    for (int i = 0; i < n_q; ++i) {
      uint32_t okw = 1;
      if (lane == 0) okw = mbar_wait(&dq_full, i & 1, lim) ? 1u : 0u;
      ok = __shfl_sync(0xffffffffu, okw, 0) != 0;
      __syncwarp();
      if (!ok) break;
      tc_fence_after();
      uint32_t v[2][32];
      tmem_ld32(lane_base + kColDQ, v[0]);
      tmem_ld32(lane_base + kColDQ + 32, v[1]);
      tmem_ld_wait();
      tmem_reg_fence(v[0]);
      tmem_reg_fence(v[1]);
      tc_fence_before();
      mbar_arrive(&dq_free);
      if (real) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          if (el) tma_store_wait_read();  // the previous box has been read from the staging rows
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 32; ++j) stg[j * 32 + lane] = __uint_as_float(v[half][j]) * p.scale;
          fence_proxy_async_smem();
          __syncwarp();
          if (el) {
            tma_reduce_add_2d(&p.tmDQ, h * Dr + q4 * 32, kv0 + i * kQT + half * 32, stg);
            tma_store_commit();
          }
          __syncwarp();
        }
      }
    }
    if (el) tma_store_wait_all();
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

// One warp per joint row j: do_joint[j] = do[srow(j)], delta[h][j] = sum_d do[j][h][d] o[j][h][d]
// (o, do stream-sorted), and the dq accumulator row cleared.  `do_joint` may be null when do is
// already in joint order (do_srow_map = 0), in which case it is read directly.
__global__ void attn_bwd_prep_kernel(const bf16* __restrict__ o, const bf16* __restrict__ dout,
                                     int dout_joint, const int* __restrict__ joint_srow, int N, int H,
                                     int head_dim, bf16* __restrict__ do_joint, float* __restrict__ delta,
                                     float* __restrict__ dq_acc) {
  mf_pdl_enter();
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int cph = head_dim / 8;  // 16-byte chunks per head (8 or 16), a power of two <= 16
  for (int j = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; j < N; j += warps) {
    const int sr = __ldg(joint_srow + j);
    if (!MF_IDX_OK(sr >= 0 && sr < N)) continue;
    const uint4* orow = reinterpret_cast<const uint4*>(o + (size_t)sr * H);
    const uint4* drow = reinterpret_cast<const uint4*>(dout + (size_t)(dout_joint ? j : sr) * H);
    uint4* jrow = do_joint ? reinterpret_cast<uint4*>(do_joint + (size_t)j * H) : nullptr;
    float4* qrow = reinterpret_cast<float4*>(dq_acc + (size_t)j * H);
    for (int c0 = 0; c0 < H / 8; c0 += 32) {
      const int c = c0 + lane;  // H / 8 is a multiple of 32 (H a multiple of 256)
      const uint4 a = __ldg(orow + c), d = __ldg(drow + c);
      if (jrow) jrow[c] = d;
      qrow[2 * c] = make_float4(0.f, 0.f, 0.f, 0.f);
      qrow[2 * c + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
      const float2 a0 = unpack_bf16x2(a.x), a1 = unpack_bf16x2(a.y), a2 = unpack_bf16x2(a.z),
                   a3 = unpack_bf16x2(a.w);
      const float2 d0 = unpack_bf16x2(d.x), d1 = unpack_bf16x2(d.y), d2 = unpack_bf16x2(d.z),
                   d3 = unpack_bf16x2(d.w);
      float s = a0.x * d0.x + a0.y * d0.y + a1.x * d1.x + a1.y * d1.y + a2.x * d2.x + a2.y * d2.y +
                a3.x * d3.x + a3.y * d3.y;
      for (int m = 1; m < cph; m <<= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
      if ((lane & (cph - 1)) == 0) delta[(size_t)(c / cph) * N + j] = s;
    }
  }
}

// dq[j] = bf16(dq_acc[j]) for the whole [N][H] accumulator (already scaled by 1 / sqrt(D)).
__global__ void attn_bwd_dq_kernel(const float4* __restrict__ acc, uint2* __restrict__ dq, long long n4) {
  mf_pdl_enter();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
    const float4 v = __ldg(acc + i);
    dq[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  }
}

}  // namespace

cudaError_t launch_attention_bwd_prep(const bf16* o, const bf16* dout, int dout_joint, const int* joint_srow,
                                      int N, int H, int head_dim, bf16* do_joint, float* delta, float* dq_acc,
                                      int num_sms, cudaStream_t st) {
  if (N <= 0) return cudaSuccess;
  const int blocks = min((N + 7) / 8, num_sms * 8);
  launch_k(attn_bwd_prep_kernel, blocks, 256, 0, st, o, dout, dout_joint, joint_srow, N, H, head_dim, do_joint, delta,
                                               dq_acc);
  return cudaGetLastError();
}

cudaError_t launch_attention_bwd(const AttnBwdParams& p, long long n_ctas, cudaStream_t st) {
  const int smem = (int)kSmemTotal + 1024;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (n_ctas <= 0) return cudaSuccess;
  launch_k(attn_bwd_kernel, (unsigned)n_ctas, kThreads, smem, st, p);
  return cudaGetLastError();
}

cudaError_t launch_attention_bwd_dq(const float* acc, bf16* dq, long long n, int num_sms, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const long long n4 = n / 4;
  const int blocks = (int)min((n4 + 255) / 256, (long long)num_sms * 8);
  launch_k(attn_bwd_dq_kernel, blocks, 256, 0, st, reinterpret_cast<const float4*>(acc), reinterpret_cast<uint2*>(dq), n4);
  return cudaGetLastError();
}

MF_BOUNDS_EXPORT(attention_bwd)

}  // namespace mf
