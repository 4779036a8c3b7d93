// Device helpers for sm_103a: mbarriers with bounded waits, TMA tile loads, tcgen05 MMA /
// TMEM access, shared-memory matrix descriptors and bf16 packing.  Inline PTX only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <utility>

namespace mf {

typedef __nv_bfloat16 bf16;

// ------------------------------------------------------------------ programmatic dependent launch
// Every kernel calls mf_pdl_enter() before its first access to global memory that an earlier
// kernel of the stream writes: griddepcontrol.wait returns once the previous grid has completed
// and its memory is visible (at once for a launch without the programmatic attribute), and
// griddepcontrol.launch_dependents lets the next kernel's launch begin.  With MF_PDL=1 in the
// environment every launch carries programmatic stream serialisation, so a kernel may be
// scheduled and run its prologue (barrier initialisation, TMEM allocation, descriptor
// prefetch) while the previous one finishes; on the 16K packs this measured no faster than
// plain stream order, so it is off by default.
__device__ __forceinline__ void mf_pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// MF_PDL=1 in the environment turns the attribute on; read once.
inline bool pdl_allowed() {
  static const bool on = [] {
    const char* e = std::getenv("MF_PDL");
    return e != nullptr && e[0] == '1';
  }();
  return on;
}

// kern<<<grid, block, smem, st>>>(args...), with the programmatic serialisation attribute when
// pdl_allowed().
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_allowed() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Device status word bits (OR-ed by kernels; read and cleared by mf_check).
enum : unsigned {
  kStatusTimeout = 1u,  // a bounded wait ran out
};

// Bounds checks of plan-derived indices (sample ids, joint rows, offsets), compiled in only by
// the checked build (-DMF_CHECKED, libmageflow_checked.so).  MF_IDX_OK(cond) is `cond` there:
// a failing check sets this translation unit's flag and the caller skips the access (no trap,
// no fault); mf_check() reports the flags as MF_ERR_DEVICE_BOUNDS.  Elsewhere it is `true`.
#ifdef MF_CHECKED
static __device__ unsigned g_mf_bounds;
#define MF_IDX_OK(cond) ((cond) || (atomicOr(&g_mf_bounds, 1u), false))
// Reads and clears this translation unit's flag (host).
static inline unsigned mf_tu_bounds_flag() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_mf_bounds, sizeof(v)) != cudaSuccess) return 2u;
  if (v != 0 && cudaMemcpyToSymbol(g_mf_bounds, &z, sizeof(z)) != cudaSuccess) return 2u;
  return v;
}
#define MF_BOUNDS_EXPORT(name) \
  unsigned bounds_flag_##name() { return mf_tu_bounds_flag(); }
#else
#define MF_IDX_OK(cond) true
#define MF_BOUNDS_EXPORT(name) \
  unsigned bounds_flag_##name() { return 0u; }
#endif

// ------------------------------------------------------------------ addresses and timers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits until the phase with the given parity has completed, for at most limit_ns.
// Returns false (and does not wait longer) when the limit runs out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(a, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void report_status(unsigned* status, unsigned bits) {
  if (status != nullptr) atomicOr(status, bits);
}

// ------------------------------------------------------------------ packed f32x2 arithmetic
// One instruction for a pair of f32 values.
// (a0, a1) += (x0, x1)
__device__ __forceinline__ void f32x2_add(float& a0, float& a1, float x0, float x1) {
  asm("{\n\t.reg .b64 a, x;\n\t"
      "mov.b64 a, {%0, %1};\n\tmov.b64 x, {%2, %3};\n\t"
      "add.rn.f32x2 a, a, x;\n\tmov.b64 {%0, %1}, a;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(x0), "f"(x1));
}
// (x0, x1) = (x0 * a0 + b0, x1 * a1 + b1)
__device__ __forceinline__ void f32x2_fma(float& x0, float& x1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 x, a, b;\n\t"
      "mov.b64 x, {%0, %1};\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "fma.rn.f32x2 x, x, a, b;\n\tmov.b64 {%0, %1}, x;\n\t}"
      : "+f"(x0), "+f"(x1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// (x0, x1) = (x0 * c + d, x1 * c + d)
__device__ __forceinline__ void f32x2_fma_s(float& x0, float& x1, float c, float d) {
  asm("{\n\t.reg .b64 x, c, d;\n\t"
      "mov.b64 x, {%0, %1};\n\tmov.b64 c, {%2, %2};\n\tmov.b64 d, {%3, %3};\n\t"
      "fma.rn.f32x2 x, x, c, d;\n\tmov.b64 {%0, %1}, x;\n\t}"
      : "+f"(x0), "+f"(x1)
      : "f"(c), "f"(d));
}

// ------------------------------------------------------------------ TMA
// Untiled bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from global to
// this CTA's shared memory, completing on `bar` (which expects the bytes).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// 2-D tiled load of one box into shared memory; completion is signalled on `bar` as
// transaction bytes.  x (innermost, elements) must keep x * 2 bytes a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* tm, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// L2 prefetch of one 2-D box (no shared memory, no completion): warms L2 for a later tile load.
// The same alignment rule as a load applies to x.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* tm, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(tm)),
               "r"(x), "r"(y)
               : "memory");
}

// 2-D tiled store of one box from shared memory (bulk-group completion).  The shared-memory
// data must be made visible to the async proxy first (fence_proxy_async_smem by the writers).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, int x, int y, const void* smem_src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(tm)),
               "r"(x), "r"(y), "r"(smem_u32(smem_src))
               : "memory");
}
// 2-D tiled reduce-add of one f32 box from shared memory into global memory (bulk-group
// completion); element-wise atomic with respect to other reductions of the same elements.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* tm, int x, int y, const void* smem_src) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
          reinterpret_cast<uint64_t>(tm)),
      "r"(x), "r"(y), "r"(smem_u32(smem_src))
      : "memory");
}
__device__ __forceinline__ void tma_store_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until this thread's committed stores have finished reading shared memory.
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until this thread's committed stores have completed.
__device__ __forceinline__ void tma_store_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05 / TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, f32 accumulate), one CTA.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on `bar` when every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Instruction descriptor, kind::f16: D f32, A and B bf16, A K-major, B K-major or MN-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool b_mn_major) {
  return (1u << 4)                            // D format: f32
         | (1u << 7)                          // A format: bf16
         | (1u << 10)                         // B format: bf16
         | ((b_mn_major ? 1u : 0u) << 16)     // B major-ness
         | ((uint32_t)(N >> 3) << 17)         // N / 8
         | ((uint32_t)(M >> 4) << 24);        // M / 16
}

// Instruction descriptor, kind::f16: D f32, A and B bf16, each K-major or MN-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32_mn(int M, int N, bool a_mn_major, bool b_mn_major) {
  return idesc_bf16_f32(M, N, b_mn_major) | ((a_mn_major ? 1u : 0u) << 15);  // A major-ness
}

// Instruction descriptor, kind::f8f6f4: D f32, A and B E4M3 (format code 0), both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4)                            // D format: f32
         | (0u << 7)                          // A format: E4M3
         | (0u << 10)                         // B format: E4M3
         | ((uint32_t)(N >> 3) << 17)         // N / 8
         | ((uint32_t)(M >> 4) << 24);        // M / 16
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand (tiles 1024-byte aligned).
// K-major: rows of 128 B (64 bf16 of K), 8-row groups `sbo` bytes apart; lbo unused.
// MN-major: 64 contiguous MN elements per 128 B row, K rows at 128 B, 8-row K groups `sbo`
// apart and 64-element MN groups `lbo` apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// TMEM address: lane in bits 31..16, column in bits 15..0.
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
  return base + (lane << 16) + col;
}

#define MF_R8(i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                 "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define MF_W8(i) "r"(r[i + 0]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                 "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])
#define MF_U8(i) "+r"(r[i + 0]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), \
                 "+r"(r[i + 4]), "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])

// 32 consecutive f32 columns of this thread's TMEM lane (warp w reads lanes 32*(w%4)..+31).
// The values are valid only after tmem_ld_wait() + tmem_reg_fence(r).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : MF_R8(0), MF_R8(8), MF_R8(16), MF_R8(24)
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Orders later uses of r after the preceding tcgen05.wait::ld.
__device__ __forceinline__ void tmem_reg_fence(uint32_t (&r)[32]) {
  asm volatile("" : MF_U8(0), MF_U8(8), MF_U8(16), MF_U8(24));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      MF_W8(0), MF_W8(8), MF_W8(16), MF_W8(24)
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ CTA pairs (clusters of 2)
// Rank of this CTA inside its cluster.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of the variable at `p` (a shared::cta pointer) in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  return a;
}

// Every thread of both CTAs of the cluster: release own writes, wait for the peer's.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Arrive once on an mbarrier of any CTA of the cluster (shared::cluster address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// 2-D tiled load into this CTA's shared memory whose completion is signalled on an mbarrier
// of either CTA of the pair (shared::cluster address of the barrier).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* tm, int x, int y,
                                                 uint32_t bar_cluster_addr) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar_cluster_addr)
      : "memory");
}

// TMEM allocation shared by a CTA pair: one warp of EACH CTA executes these together; both
// CTAs get the same columns.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Arrives once on the mbarrier at the same offset in every CTA of `cta_mask` when all
// tcgen05 operations issued so far by this thread are done.
__device__ __forceinline__ void mma_commit_pair_mc(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// ------------------------------------------------------------------ warp-uniform issue
// The issuing warps of the pipelined kernels run their loops with all 32 lanes (so loop state
// and descriptors stay warp-uniform) and let one elected lane execute each tcgen05 / TMA /
// mbarrier instruction that must be issued once.

// 1 in exactly one lane of the (fully active) warp, 0 in the others.
__device__ __forceinline__ uint32_t elect_one() {
  uint32_t e;
  asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(e));
  return e;
}

__device__ __forceinline__ void mma_bf16_if(uint32_t pred, uint32_t d_tmem, uint64_t a_desc,
                                            uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(pred)
      : "memory");
}

__device__ __forceinline__ void mma_commit_if(uint32_t pred, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %1, 0;\n\t"
      "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar)),
      "r"(pred)
      : "memory");
}

// D[tmem of both CTAs] (+)= A[smem of both CTAs] * B[smem of both CTAs]^T for the lane whose
// pred is non-zero (the elected lane of the even CTA's MMA warp): rows 0..M/2-1 of A and D live
// in the even CTA, the rest in the odd one; B's rows (N) are split the same way.
__device__ __forceinline__ void mma_bf16_pair_if(uint32_t pred, uint32_t d_tmem, uint64_t a_desc,
                                                 uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(pred)
      : "memory");
}

// As mma_bf16_pair_if with E4M3 operands (kind::f8f6f4, K = 32 per instruction: the same
// 32 bytes of each 128-byte swizzled row as one bf16 K = 16 step).
__device__ __forceinline__ void mma_f8_pair_if(uint32_t pred, uint32_t d_tmem, uint64_t a_desc,
                                               uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(pred)
      : "memory");
}

__device__ __forceinline__ void mma_commit_pair_mc_if(uint32_t pred, uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t"
      "@q tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "h"(cta_mask), "r"(pred)
      : "memory");
}

// ------------------------------------------------------------------ MMA groups
// A run of `n` kind::f16 MMAs into one accumulator along K, issued from one asm block by the
// lane whose pred is non-zero: step j uses descriptors a_desc + j * a_step and b_desc +
// j * b_step (the 14-bit address fields never carry: shared memory is below 256 KB), and the
// first step accumulates iff `accumulate`.  Cheaper to issue than n separate calls, which
// each rebuild both 64-bit descriptors and the predicates.
template <int n>
__device__ __forceinline__ void mma_group_ss(uint32_t pred, uint32_t d_tmem, uint64_t a_desc, uint64_t a_step,
                                             uint64_t b_desc, uint64_t b_step, uint32_t idesc, uint32_t accumulate) {
  static_assert(n == 4 || n == 8, "4 or 8 steps");
  if constexpr (n == 4) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b64 a, b;\n\t"
        "setp.ne.b32 p, %6, 0;\n\tsetp.ne.b32 q, %7, 0;\n\t"
        "mov.b64 a, %1;\n\tmov.b64 b, %3;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, p;\n\t"
        "add.s64 a, a, %2;\n\tadd.s64 b, b, %4;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, 1;\n\t"
        "add.s64 a, a, %2;\n\tadd.s64 b, b, %4;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, 1;\n\t"
        "add.s64 a, a, %2;\n\tadd.s64 b, b, %4;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %5, 1;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(a_step), "l"(b_desc), "l"(b_step), "r"(idesc), "r"(accumulate), "r"(pred)
        : "memory");
  } else {
    mma_group_ss<4>(pred, d_tmem, a_desc, a_step, b_desc, b_step, idesc, accumulate);
    mma_group_ss<4>(pred, d_tmem, a_desc + 4 * a_step, a_step, b_desc + 4 * b_step, b_step, idesc, 1u);
  }
}

// Two MMAs with A read from TMEM (columns a_tmem, a_tmem + a_step), as mma_group4_ts.
__device__ __forceinline__ void mma_group2_ts(uint32_t pred, uint32_t d_tmem, uint32_t a_tmem, uint32_t a_step,
                                              uint64_t b_desc, uint64_t b_step, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b32 a;\n\t.reg .b64 b;\n\t"
      "setp.ne.b32 p, %6, 0;\n\tsetp.ne.b32 q, %7, 0;\n\t"
      "mov.b32 a, %1;\n\tmov.b64 b, %3;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %5, p;\n\t"
      "add.u32 a, a, %2;\n\tadd.s64 b, b, %4;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %5, 1;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(a_step), "l"(b_desc), "l"(b_step), "r"(idesc), "r"(accumulate), "r"(pred)
      : "memory");
}

// ------------------------------------------------------------------ math / packing
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two f32 values to E4M3 codes, round to nearest even, saturating to +-448 (the hardware
// conversion): lo in bits 7..0, hi in bits 15..8.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  unsigned short d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(v);
}

// Advances a shared-memory pointer to the next 1024-byte boundary of the shared window.
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

}  // namespace mf
