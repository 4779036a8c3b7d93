// C ABI of libmageflow.so: argument validation, workspace layout, TMA descriptors and the
// launch sequence of each call.  The operations themselves are specified in mageflow.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>
#include <vector>

#include "attention.cuh"
#include "attention_bwd.cuh"
#include "block_bwd.cuh"
#include "gemm.cuh"
#include "internal.h"
#include "pointwise.cuh"

namespace {

using mf::bf16;

__device__ unsigned int g_mf_status;  // OR of kernel status bits since the last mf_check

// ------------------------------------------------------------------ per-device state
struct DevInfo {
  bool init = false;
  int sms = 0;
  unsigned* status = nullptr;
};
constexpr int kMaxDev = 64;
DevInfo g_dev[kMaxDev];
std::mutex g_mu;

mf_status device_info(DevInfo** out, int* dev_out = nullptr) {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDev) return MF_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& di = g_dev[d];
  if (!di.init) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess)
      return MF_ERR_CUDA;
    if (major != 10 || minor != 3) return MF_ERR_UNSUPPORTED;  // built for sm_103a only
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_mf_status) != cudaSuccess) return MF_ERR_CUDA;
    di.status = static_cast<unsigned*>(p);
    di.init = true;
  }
  *out = &di;
  if (dev_out) *dev_out = d;
  return MF_OK;
}

unsigned long long wait_limit_ns() {
  static unsigned long long v = [] {
    const char* e = std::getenv("MF_WAIT_LIMIT_MS");
    long long ms = e ? std::atoll(e) : 4000;
    if (ms < 1) ms = 1;
    if (ms > 60000) ms = 60000;
    return (unsigned long long)ms * 1000000ull;
  }();
  return v;
}

// ------------------------------------------------------------------ tracing
struct TraceRec {
  int kind;
  cudaEvent_t a, b;
  double flops, bytes;
  int nk;
};

struct TraceState {
  bool on = false;
  uint32_t mask = 0xffffffffu;  // kinds that are bracketed while tracing is on
  std::vector<TraceRec> recs;
  std::vector<cudaEvent_t> pool;
};
TraceState g_trace;
std::mutex g_trace_mu;
std::atomic<long long> g_launches{0};

cudaEvent_t trace_event() {
  if (!g_trace.pool.empty()) {
    cudaEvent_t e = g_trace.pool.back();
    g_trace.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

using mf::Trace;

// ------------------------------------------------------------------ TMA descriptors
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// bf16 matrix [rows][cols] (row-major, contiguous), boxes of box_rows x 64 columns,
// 128-byte swizzle, zero fill outside the matrix.
bool make_tmap(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E4M3 codes [rows][cols] (bytes, row-major, contiguous), boxes of box_rows x 128 columns
// (128 bytes), 128-byte swizzle, zero fill outside the matrix.
bool make_tmap_u8(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// f32 matrix [rows][cols] (row-major, contiguous), boxes of box_rows x box_cols, no swizzle.
bool make_tmap_f32(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                   uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ validation helpers
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

mf_status check_dims(const mf_dims* d) {
  if (d == nullptr) return MF_ERR_INVALID_ARG;
  if (d->hidden <= 0 || d->heads <= 0 || d->channels <= 0 || d->mlp_ratio <= 0 || d->freq_dim <= 0)
    return MF_ERR_INVALID_ARG;
  if (d->hidden % d->heads != 0) return MF_ERR_INVALID_ARG;
  const int D = d->hidden / d->heads;
  if (D != 64 && D != 128) return MF_ERR_UNSUPPORTED;
  if (d->hidden % 256 != 0 || d->hidden > 4096) return MF_ERR_UNSUPPORTED;
  if ((d->mlp_ratio * d->hidden) % 256 != 0) return MF_ERR_UNSUPPORTED;
  if (d->channels != 64 && d->channels != 128) return MF_ERR_UNSUPPORTED;
  if (d->freq_dim % 256 != 0) return MF_ERR_UNSUPPORTED;
  return MF_OK;
}

mf_status check_plan(const mf_plan* p, int dev) {
  if (p == nullptr) return MF_ERR_INVALID_ARG;
  if (p->d_blob == nullptr) return MF_ERR_NOT_UPLOADED;
  if (p->device != dev) return MF_ERR_INVALID_ARG;
  return MF_OK;
}

mf_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MF_OK : MF_ERR_CUDA; }

#define MF_TRY(x)                     \
  do {                                \
    mf_status _s = (x);               \
    if (_s != MF_OK) return _s;       \
  } while (0)
#define MF_CUDA(x)                    \
  do {                                \
    if ((x) != cudaSuccess) return MF_ERR_CUDA; \
  } while (0)

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

// ------------------------------------------------------------------ workspace layouts
struct BlockLayout {
  size_t off[9];  // c, mod, a, q, k, v, o, hidden, LN statistics parts
  size_t sinus, h1;
  size_t total;
};

BlockLayout block_layout(const mf_plan* p, const mf_dims* d) {
  BlockLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = al256(o + bytes); return r; };
  const size_t S = p->S, N = p->N, H = d->hidden, F = d->freq_dim, R = (size_t)d->mlp_ratio * H;
  L.off[0] = take(S * H * 4);
  L.off[1] = take(S * 12 * H * 4);
  L.off[2] = take(N * H * 2);
  L.off[3] = take(N * H * 2);
  L.off[4] = take(N * H * 2);
  L.off[5] = take(N * H * 2);
  L.off[6] = take(N * H * 2);
  L.off[7] = take(N * R * 2);
  L.sinus = take(S * F * 4);
  L.h1 = take(S * H * 4);
  L.off[8] = take(N * (H / 128) * 8);
  L.total = o;
  return L;
}

// fp8 block forward: E4M3 codes of one projection input at a time ([N][mlp_ratio H] bytes at
// most) and their row scales ([N] f32), after the bf16 workspace.
size_t fp8_region_bytes(const mf_plan* p, const mf_dims* d) {
  const size_t N = p->N, R = (size_t)d->mlp_ratio * d->hidden;
  return al256(N * R) + al256(N * 4);
}

// Training forward: the block workspace followed by what the backward reads - the block input
// x0 and the residual after attention x1 (stream-sorted bf16 [N][H]), the first LN + modulate
// output a1 (the block workspace's `a` keeps the second), the ungated out-projection and MLP
// outputs y_o, y_m [N][H], the MLP pre-activation u [N][rH] and the attention lse [heads][N].
struct TrainLayout {
  BlockLayout base;
  size_t x0, x1, a1, yo, ym, u, lse, total;
};

TrainLayout train_layout(const mf_plan* p, const mf_dims* d) {
  TrainLayout L{};
  L.base = block_layout(p, d);
  size_t o = L.base.total;
  auto take = [&](size_t bytes) { size_t r = o; o = al256(o + bytes); return r; };
  const size_t N = p->N, H = d->hidden, R = (size_t)d->mlp_ratio * H;
  L.x0 = take(N * H * 2);
  L.x1 = take(N * H * 2);
  L.a1 = take(N * H * 2);
  L.yo = take(N * H * 2);
  L.ym = take(N * H * 2);
  L.u = take(N * R * 2);
  L.lse = take((size_t)d->heads * N * 4);
  L.total = o;
  return L;
}

struct FinalLayout {
  size_t c, fmod, a, sinus, h1, total;
};

FinalLayout final_layout(const mf_plan* p, const mf_dims* d) {
  FinalLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = al256(o + bytes); return r; };
  const size_t S = p->S, H = d->hidden, F = d->freq_dim;
  L.c = take(S * H * 4);
  L.fmod = take(S * 2 * H * 4);
  L.a = take((size_t)p->Ni * H * 2);
  L.sinus = take(S * F * 4);
  L.h1 = take(S * H * 4);
  L.total = o;
  return L;
}

// ------------------------------------------------------------------ GEMM driver
struct GemmSpec {
  int M, N, K;
  const void* A;
  const void* B;
  const void* bias;
  void* out;
  int ldo;
  int row_off;
  int stream;
  const float* col_scale;  // E4M3 operands (kEpiF8): per-column dequantisation scale of B
  void* aux;               // kEpiSave output / kEpiGeluBwd input, bf16 [M][ldo]
};

// maj (pair kernel, bf16): mf::kMajKK for C = A B^T with A [M][K], B [N][K]; kMajBMN with B
// stored [K][N]; kMajMNMN with A stored [K][M] and B [K][N] (K may then be any length).
mf_status run_gemm(const GemmSpec* specs, int nspec, int epi, int BN, mf::GemmParams& p,
                   const DevInfo* di, cudaStream_t st, int kind, int maj = mf::kMajKK) {
  // 256-wide tiles run on CTA pairs (256 x 256 per pair), 128-wide ones on single CTAs
  const bool pair = BN == 256;
  p.n_prob = 0;
  p.tile_begin[0] = 0;
  int begin = 0;
  for (int s = 0; s < nspec; ++s) {
    const GemmSpec& g = specs[s];
    if (g.M <= 0) continue;
    const int i = p.n_prob;
    if (epi & mf::kEpiF8) {  // E4M3 operands: byte tensor maps
      if (!pair || !make_tmap_u8(&p.tmA[i], g.A, g.K, g.M, 128) || !make_tmap_u8(&p.tmB[i], g.B, g.K, g.N, BN / 2))
        return MF_ERR_CUDA;
    } else {
      const bool amn = (maj & mf::kMajAMN) != 0, bmn = (maj & mf::kMajBMN) != 0;
      if (amn ? !make_tmap(&p.tmA[i], g.A, g.M, g.K, 64) : !make_tmap(&p.tmA[i], g.A, g.K, g.M, 128))
        return MF_ERR_CUDA;
      if (bmn ? !make_tmap(&p.tmB[i], g.B, g.N, g.K, 64) : !make_tmap(&p.tmB[i], g.B, g.K, g.N, pair ? BN / 2 : BN))
        return MF_ERR_CUDA;
    }
    p.prob[i].M = g.M;
    p.prob[i].N = g.N;
    p.prob[i].K = g.K;
    p.prob[i].row_off = g.row_off;
    p.prob[i].stream = g.stream;
    p.prob[i].ldo = g.ldo;
    p.prob[i].bias = static_cast<const bf16*>(g.bias);
    p.prob[i].col_scale = g.col_scale;
    p.prob[i].out = g.out;
    p.prob[i].aux = g.aux;
    p.tiles_m[i] = pair ? (g.M + 255) / 256 : (g.M + 127) / 128;
    p.tiles_n[i] = (g.N + BN - 1) / BN;
    p.tma_store[i] = 0;
    const int base = epi & ~mf::kEpiF8;
    if (pair && (base == mf::kEpiBiasBf16 || base == mf::kEpiGelu || base == mf::kEpiGeluBwd) && g.ldo == g.N &&
        g.N % 64 == 0 &&
        aligned(g.out, 16)) {
      if (!make_tmap(&p.tmC[i], g.out, g.N, g.M, 32)) return MF_ERR_CUDA;
      p.tma_store[i] = 1;
    }
    // N fastest when a wave of tiles spans whole rows of N tiles (few N tiles: the weight
    // matrix then stays in L2); otherwise sweep N over groups of 16 row tiles
    p.group_m[i] = p.tiles_n[i] <= 16 ? 0 : 16;
    begin += p.tiles_m[i] * p.tiles_n[i];
    p.tile_begin[i + 1] = begin;
    p.n_prob++;
  }
  if (p.n_prob == 0) return MF_OK;
  if (p.n_prob == 1) p.tile_begin[2] = begin;
  p.status = di->status;
  p.wait_limit_ns = wait_limit_ns();
  double flops = 0;
  for (int i = 0; i < p.n_prob; ++i) flops += 2.0 * p.prob[i].M * (double)p.prob[i].N * p.prob[i].K;
  Trace tr(kind, st, flops, 0, 1);
  if (!pair && maj != mf::kMajKK) return MF_ERR_UNSUPPORTED;
  return cuda_status(pair ? mf::launch_gemm_pair(p, epi, di->sms, st, maj)
                          : mf::launch_gemm(p, BN, epi, di->sms, st));
}

mf_status conditioning(const mf_plan* p, const mf_dims* d, const mf_temb_weights* tw,
                       const float* t, float* sinus, float* h1, float* c, const DevInfo* di,
                       cudaStream_t st) {
  const int S = p->S, H = d->hidden, F = d->freq_dim;
  const int groups = (S + 3) / 4;  // one GEMV launch per group of four samples
  Trace tr(MF_K_COND, st, 2.0 * S * ((double)F * H + (double)H * H), 2.0 * ((double)F * H + (double)H * H),
           1 + 2 * groups);
  MF_CUDA(mf::launch_sinusoid(t, S, F, sinus, st));
  MF_CUDA(mf::launch_gemv(static_cast<const bf16*>(tw->w_t1), static_cast<const bf16*>(tw->b_t1),
                          sinus, S, F, H, h1, H, 0, 1, di->status, wait_limit_ns(), st));
  MF_CUDA(mf::launch_gemv(static_cast<const bf16*>(tw->w_t2), static_cast<const bf16*>(tw->b_t2), h1,
                          S, H, H, c, H, 0, 1, di->status, wait_limit_ns(), st));
  return MF_OK;
}

bool temb_ok(const mf_temb_weights* t) {
  return t && t->w_t1 && t->b_t1 && t->w_t2 && t->b_t2 && aligned(t->w_t1, 16) &&
         aligned(t->w_t2, 16);
}

bool stream_ok(const mf_stream_weights& s) {
  const void* ptrs[] = {s.w_mod, s.b_mod, s.w_qkv, s.b_qkv, s.w_o, s.b_o, s.w_1, s.b_1, s.w_2, s.b_2};
  for (const void* q : ptrs)
    if (q == nullptr || !aligned(q, 16)) return false;
  // QK-RMSNorm scales: both or neither
  if ((s.w_qnorm == nullptr) != (s.w_knorm == nullptr)) return false;
  if (s.w_qnorm != nullptr && (!aligned(s.w_qnorm, 16) || !aligned(s.w_knorm, 16))) return false;
  return true;
}

}  // namespace

namespace mf {

mf_status current_device(int* dev) {
  DevInfo* di = nullptr;
  return device_info(&di, dev);
}

Trace::Trace(int kind, cudaStream_t st, double flops, double bytes, int nk)
    : st_(st), kind_(kind), nk_(nk), flops_(flops), bytes_(bytes) {
  g_launches += nk;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (!g_trace.on || ((g_trace.mask >> kind) & 1u) == 0) return;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return;
  a_ = trace_event();
  b_ = trace_event();
  if (a_ == nullptr || b_ == nullptr) return;
  active_ = cudaEventRecord(a_, st) == cudaSuccess;
}

Trace::~Trace() {
  if (!active_) return;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  if (cudaEventRecord(b_, st_) == cudaSuccess) g_trace.recs.push_back(TraceRec{kind_, a_, b_, flops_, bytes_, nk_});
}

}  // namespace mf

// ====================================================================== plan upload / free
extern "C" mf_status mf_plan_upload(mf_plan* p, void* stream) {
  if (p == nullptr) return MF_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MF_ERR_CUDA;
  if (p->d_blob != nullptr) return p->device == dev ? MF_OK : MF_ERR_INVALID_ARG;

  struct Part { const void* src; size_t bytes; size_t off; };
  const int32_t* srcs[] = {p->cu.data(), p->cui.data(), p->pos.data(), p->srow_joint.data(),
                           p->srow_seq.data(), p->joint_srow.data(), p->img_seq.data(),
                           p->img_pair.data(), p->img_target.data(), p->seq_role.data(),
                           p->items.data(), p->row_chunks.data()};
  size_t counts[] = {p->cu.size(), p->cui.size(), p->pos.size(), p->srow_joint.size(),
                     p->srow_seq.size(), p->joint_srow.size(), p->img_seq.size(),
                     p->img_pair.size(), p->img_target.size(), p->seq_role.size(),
                     p->items.size(), p->row_chunks.size()};
  const int np = 12;
  size_t off[13];
  size_t o = 0;
  for (int i = 0; i < np; ++i) {
    off[i] = o;
    o = (o + counts[i] * 4 + 63) & ~size_t(63);
  }
  off[np] = o;
  o = (o + p->t.size() * 4 + 63) & ~size_t(63);
  p->blob_bytes = o > 0 ? o : 64;

  // stream-ordered allocation: neither this nor mf_plan_free waits for work on other streams
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* blob = nullptr;
  if (cudaMallocAsync(&blob, p->blob_bytes, st) != cudaSuccess) return MF_ERR_CUDA;
  // staged in one host buffer; the upload is synchronised before the buffer is released
  char* host = static_cast<char*>(std::malloc(p->blob_bytes));
  if (host == nullptr) { cudaFreeAsync(blob, st); return MF_ERR_CUDA; }
  std::memset(host, 0, p->blob_bytes);
  for (int i = 0; i < np; ++i)
    if (counts[i]) std::memcpy(host + off[i], srcs[i], counts[i] * 4);
  if (!p->t.empty()) std::memcpy(host + off[np], p->t.data(), p->t.size() * 4);
  cudaError_t e = cudaMemcpyAsync(blob, host, p->blob_bytes, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  std::free(host);
  if (e != cudaSuccess) { cudaFreeAsync(blob, st); return MF_ERR_CUDA; }

  char* b = static_cast<char*>(blob);
  p->d_cu = reinterpret_cast<const int32_t*>(b + off[0]);
  p->d_cui = reinterpret_cast<const int32_t*>(b + off[1]);
  p->d_pos = reinterpret_cast<const int32_t*>(b + off[2]);
  p->d_srow_joint = reinterpret_cast<const int32_t*>(b + off[3]);
  p->d_srow_seq = reinterpret_cast<const int32_t*>(b + off[4]);
  p->d_joint_srow = reinterpret_cast<const int32_t*>(b + off[5]);
  p->d_img_seq = reinterpret_cast<const int32_t*>(b + off[6]);
  p->d_img_pair = reinterpret_cast<const int32_t*>(b + off[7]);
  p->d_img_target = reinterpret_cast<const int32_t*>(b + off[8]);
  p->d_seq_role = reinterpret_cast<const int32_t*>(b + off[9]);
  p->d_items = reinterpret_cast<const int32_t*>(b + off[10]);
  p->d_row_chunks = reinterpret_cast<const int32_t*>(b + off[11]);
  p->d_t = reinterpret_cast<const float*>(b + off[12]);
  p->d_blob = blob;
  p->device = dev;
  return MF_OK;
}

extern "C" void mf_plan_free(mf_plan* p) {
  if (p == nullptr) return;
  if (p->d_blob != nullptr) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != p->device) cudaSetDevice(p->device);
    // released in stream order on the legacy default stream, without a device-wide wait
    cudaFreeAsync(p->d_blob, nullptr);
    if (cur != p->device && cur >= 0) cudaSetDevice(cur);
  }
  delete p;
}

// ====================================================================== block forward
extern "C" size_t mf_block_workspace_bytes(const mf_plan* p, const mf_dims* d) {
  if (p == nullptr || check_dims(d) != MF_OK) return 0;
  return block_layout(p, d).total;
}

extern "C" mf_status mf_block_workspace_layout(const mf_plan* p, const mf_dims* d, size_t* offsets,
                                               int32_t n) {
  if (p == nullptr || offsets == nullptr || n < 8) return MF_ERR_INVALID_ARG;
  MF_TRY(check_dims(d));
  BlockLayout L = block_layout(p, d);
  for (int i = 0; i < 8 || (i < 9 && i < n); ++i) offsets[i] = L.off[i];
  return MF_OK;
}

namespace {
bool stream8_ok(const mf_stream_weights_fp8& s) {
  const void* ptrs[] = {s.q_qkv, s.s_qkv, s.q_o, s.s_o, s.q_1, s.s_1, s.q_2, s.s_2};
  for (const void* q : ptrs)
    if (q == nullptr || !aligned(q, 16)) return false;
  return true;
}

// LN + modulate through the kernel `flags` selects (MF_BLOCK_LN_*; 0 = one warp per row); the
// row-group kernel also takes the statistics the out-projection's epilogue left (ln.stats).
cudaError_t launch_ln(const mf::LnModArgs& ln, int flags, cudaStream_t st) {
  return (flags & MF_BLOCK_LN_ROW_GROUPS || ln.stats != nullptr) ? mf::launch_ln_group(ln, st)
                                                                 : mf::launch_ln_modulate(ln, st);
}

// The block forward; with w8 the four projections run on E4M3 operands: each input (a, o, a,
// hidden) is quantised per row right before its GEMM, into the fp8 region after the bf16
// workspace.  `flags` (MF_BLOCK_*) select the LN + modulate variant.
// With `train`, the workspace has the training layout and the forward also keeps what the
// backward reads (TrainLayout).
mf_status block_forward(const mf_plan* p, const mf_dims* d, const mf_block_weights* w,
                        const mf_block_weights_fp8* w8, const float* d_t, void* d_x_txt, void* d_x_img,
                        void* d_ws, size_t ws_bytes, void* stream, bool train = false, int flags = 0) {
  DevInfo* di = nullptr;
  int dev = -1;
  MF_TRY(device_info(&di, &dev));
  MF_TRY(check_plan(p, dev));
  MF_TRY(check_dims(d));
  if (w == nullptr || !temb_ok(&w->temb) || !stream_ok(w->txt) || !stream_ok(w->img))
    return MF_ERR_INVALID_ARG;
  if (w8 != nullptr && (!stream8_ok(w8->txt) || !stream8_ok(w8->img))) return MF_ERR_INVALID_ARG;
  if ((flags & ~(MF_BLOCK_LN_ROW_GROUPS | MF_BLOCK_LN_STATS_FUSED | MF_BLOCK_COND_GIVEN)) != 0)
    return MF_ERR_INVALID_ARG;
  if (flags & MF_BLOCK_LN_STATS_FUSED && (w8 != nullptr || train)) return MF_ERR_UNSUPPORTED;
  if (p->N == 0) return MF_OK;
  if ((p->Nt > 0 && d_x_txt == nullptr) || (p->Ni > 0 && d_x_img == nullptr) || d_ws == nullptr)
    return MF_ERR_INVALID_ARG;
  if (!aligned(d_x_txt, 16) || !aligned(d_x_img, 16) || !aligned(d_ws, 256) || !aligned(d_t, 4))
    return MF_ERR_ALIGNMENT;
  const BlockLayout L = block_layout(p, d);
  const size_t fp8_bytes = w8 ? fp8_region_bytes(p, d) : 0;
  const TrainLayout TL = train_layout(p, d);
  if (train && (w8 != nullptr || w->txt.w_qnorm != nullptr || w->img.w_qnorm != nullptr))
    return MF_ERR_UNSUPPORTED;  // the backward covers the plain bf16 block
  if (ws_bytes < (train ? TL.total : L.total + fp8_bytes)) return MF_ERR_WORKSPACE;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(d_ws);
  const int S = p->S, N = p->N, Nt = p->Nt, Ni = p->Ni, H = d->hidden, D = H / d->heads;
  const int R = d->mlp_ratio * H;
  const float* t = d_t ? d_t : p->d_t;
  float* c = reinterpret_cast<float*>(ws + L.off[0]);
  float* mod = reinterpret_cast<float*>(ws + L.off[1]);
  bf16* a = reinterpret_cast<bf16*>(ws + L.off[2]);
  bf16* q = reinterpret_cast<bf16*>(ws + L.off[3]);
  bf16* k = reinterpret_cast<bf16*>(ws + L.off[4]);
  bf16* v = reinterpret_cast<bf16*>(ws + L.off[5]);
  bf16* o = reinterpret_cast<bf16*>(ws + L.off[6]);
  bf16* hid = reinterpret_cast<bf16*>(ws + L.off[7]);
  float2* ln_stats = reinterpret_cast<float2*>(ws + L.off[8]);
  const int STATS = (flags & MF_BLOCK_LN_STATS_FUSED) ? mf::kEpiStats : 0;
  float* sinus = reinterpret_cast<float*>(ws + L.sinus);
  float* h1 = reinterpret_cast<float*>(ws + L.h1);
  bf16* xt = static_cast<bf16*>(d_x_txt);
  bf16* xi = static_cast<bf16*>(d_x_img);
  // fp8: codes of the current projection input [N][<= R] and their row scales [N]
  uint8_t* q8 = reinterpret_cast<uint8_t*>(ws + L.total);
  float* s8 = reinterpret_cast<float*>(ws + L.total + al256((size_t)N * R));
  const int F8 = w8 ? mf::kEpiF8 : 0;
  // training: saved values (null otherwise)
  bf16* x0 = train ? reinterpret_cast<bf16*>(ws + TL.x0) : nullptr;
  bf16* x1 = train ? reinterpret_cast<bf16*>(ws + TL.x1) : nullptr;
  bf16* a1 = train ? reinterpret_cast<bf16*>(ws + TL.a1) : a;
  bf16* yo = train ? reinterpret_cast<bf16*>(ws + TL.yo) : nullptr;
  bf16* ym = train ? reinterpret_cast<bf16*>(ws + TL.ym) : nullptr;
  bf16* u = train ? reinterpret_cast<bf16*>(ws + TL.u) : nullptr;
  float* lse = train ? reinterpret_cast<float*>(ws + TL.lse) : nullptr;
  const int SAVE = train ? mf::kEpiSave : 0;
  auto copy_x = [&](bf16* dst) -> mf_status {  // stream-sorted copy of the residual
    if (Nt > 0) MF_CUDA(cudaMemcpyAsync(dst, xt, (size_t)Nt * H * 2, cudaMemcpyDeviceToDevice, st));
    if (Ni > 0) MF_CUDA(cudaMemcpyAsync(dst + (size_t)Nt * H, xi, (size_t)Ni * H * 2, cudaMemcpyDeviceToDevice, st));
    return MF_OK;
  };
  auto quantize = [&](const bf16* src, int K) -> mf_status {
    Trace tr(MF_K_FP8, st, 0, 3.0 * N * (double)K, 1);
    return cuda_status(mf::launch_quantize_e4m3_rows(src, N, K, q8, s8, st));
  };

  // 1. timestep condition c = SiLU(temb(t)) and the per-sample adaLN modulation of both streams
  if (!(flags & MF_BLOCK_COND_GIVEN)) MF_TRY(conditioning(p, d, &w->temb, t, sinus, h1, c, di, st));
  {
    // both streams' modulation GEMVs share c and run as one launch per group of four samples
    Trace tr(MF_K_COND, st, 2.0 * 2 * S * 6.0 * H * H, 2.0 * 2 * 6.0 * H * H, (S + 3) / 4);
    MF_CUDA(mf::launch_gemv2(static_cast<const bf16*>(w->txt.w_mod), static_cast<const bf16*>(w->txt.b_mod), 0,
                             static_cast<const bf16*>(w->img.w_mod), static_cast<const bf16*>(w->img.b_mod),
                             6 * H, c, S, H, 6 * H, mod, 12 * H, di->status, wait_limit_ns(), st));
  }

  // 2. a = LN(x)(1 + scale1) + shift1, stream-sorted
  if (train) MF_TRY(copy_x(x0));
  mf::LnModArgs ln{xt, xi, Nt, N, H, p->d_srow_seq, mod, 12LL * H, 6LL * H, 0, H, a1, S, nullptr,
                   di->status, wait_limit_ns()};
  {
    Trace tr(MF_K_LN, st, 0, 4.0 * N * H, 1);
    MF_CUDA(launch_ln(ln, flags, st));
  }
  ln.out = a;

  // 3. q | k | v = a W_qkv^T + b, RoPE, scattered to joint order
  mf::GemmParams gp{};
  gp.srow_seq = p->d_srow_seq;
  gp.srow_joint = p->d_srow_joint;
  gp.pos = p->d_pos;
  gp.mod = mod;
  gp.H = H;
  gp.head_dim = D;
  gp.n_tok = N;
  gp.n_seq = S;
  gp.q = q;
  gp.k = k;
  gp.v = v;
  gp.qk_norm[0][0] = static_cast<const bf16*>(w->txt.w_qnorm);
  gp.qk_norm[0][1] = static_cast<const bf16*>(w->txt.w_knorm);
  gp.qk_norm[1][0] = static_cast<const bf16*>(w->img.w_qnorm);
  gp.qk_norm[1][1] = static_cast<const bf16*>(w->img.w_knorm);
  gp.row_scale = s8;
  gp.ln_stats = ln_stats;
  gp.ln_parts = H / 128;
  if (w8) {
    MF_TRY(quantize(a, H));
    GemmSpec sp[2] = {{Nt, 3 * H, H, q8, w8->txt.q_qkv, w->txt.b_qkv, nullptr, 0, 0, 0, w8->txt.s_qkv},
                      {Ni, 3 * H, H, q8 + (size_t)Nt * H, w8->img.q_qkv, w->img.b_qkv, nullptr, 0, Nt, 1,
                       w8->img.s_qkv}};
    MF_TRY(run_gemm(sp, 2, mf::kEpiQkvRope | F8, 256, gp, di, st, MF_K_GEMM_QKV));
  } else {
    GemmSpec sp[2] = {{Nt, 3 * H, H, a1, w->txt.w_qkv, w->txt.b_qkv, nullptr, 0, 0, 0},
                      {Ni, 3 * H, H, a1 + (size_t)Nt * H, w->img.w_qkv, w->img.b_qkv, nullptr, 0, Nt, 1}};
    MF_TRY(run_gemm(sp, 2, mf::kEpiQkvRope, 256, gp, di, st, MF_K_GEMM_QKV));
  }

  // 4. joint varlen attention -> o (stream-sorted)
  {
    mf::AttnParams ap{};
    if (!make_tmap(&ap.tmQ, q, H, N, 128) || !make_tmap(&ap.tmK, k, H, N, 128) ||
        !make_tmap(&ap.tmV, v, H, N, 128))
      return MF_ERR_CUDA;
    ap.cu = p->d_cu;
    ap.items = p->d_items;
    ap.joint_srow = p->d_joint_srow;
    ap.out = o;
    ap.lse = lse;
    ap.H = H;
    ap.heads = d->heads;
    ap.n_items = p->n_items;
    ap.n_tok = N;
    ap.n_seq = S;
    ap.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    ap.status = di->status;
    ap.wait_limit_ns = wait_limit_ns();
    Trace tr(MF_K_ATTN, st, 4.0 * p->sum_L2 * H, 0, 1);
    MF_CUDA(mf::launch_attention(ap, D, st));
  }

  // 5. x += gate1 (o W_o^T + b_o)
  gp.gate_off = 2 * H;
  if (w8) {
    MF_TRY(quantize(o, H));
    GemmSpec sp[2] = {{Nt, H, H, q8, w8->txt.q_o, w->txt.b_o, xt, H, 0, 0, w8->txt.s_o},
                      {Ni, H, H, q8 + (size_t)Nt * H, w8->img.q_o, w->img.b_o, xi, H, Nt, 1, w8->img.s_o}};
    MF_TRY(run_gemm(sp, 2, mf::kEpiGateResid | F8, 256, gp, di, st, MF_K_GEMM_OPROJ));
  } else {
    GemmSpec sp[2] = {{Nt, H, H, o, w->txt.w_o, w->txt.b_o, xt, H, 0, 0, nullptr, yo},
                      {Ni, H, H, o + (size_t)Nt * H, w->img.w_o, w->img.b_o, xi, H, Nt, 1, nullptr,
                       yo ? yo + (size_t)Nt * H : nullptr}};
    MF_TRY(run_gemm(sp, 2, mf::kEpiGateResid | SAVE | STATS, 256, gp, di, st, MF_K_GEMM_OPROJ));
  }
  if (train) MF_TRY(copy_x(x1));

  // 6. a = LN(x)(1 + scale2) + shift2 (statistics from the out-projection's epilogue when fused)
  ln.shift_off = 3 * H;
  ln.scale_off = 4 * H;
  if (STATS) ln.stats = ln_stats;
  {
    Trace tr(MF_K_LN, st, 0, 4.0 * N * H, 1);
    MF_CUDA(launch_ln(ln, flags, st));
  }

  // 7. hidden = GELU(a W_1^T + b_1)
  if (w8) {
    MF_TRY(quantize(a, H));
    GemmSpec sp[2] = {{Nt, R, H, q8, w8->txt.q_1, w->txt.b_1, hid, R, 0, 0, w8->txt.s_1},
                      {Ni, R, H, q8 + (size_t)Nt * H, w8->img.q_1, w->img.b_1, hid + (size_t)Nt * R, R, Nt, 1,
                       w8->img.s_1}};
    MF_TRY(run_gemm(sp, 2, mf::kEpiGelu | F8, 256, gp, di, st, MF_K_GEMM_UP));
  } else {
    GemmSpec sp[2] = {{Nt, R, H, a, w->txt.w_1, w->txt.b_1, hid, R, 0, 0, nullptr, u},
                      {Ni, R, H, a + (size_t)Nt * H, w->img.w_1, w->img.b_1, hid + (size_t)Nt * R, R, Nt, 1, nullptr,
                       u ? u + (size_t)Nt * R : nullptr}};
    MF_TRY(run_gemm(sp, 2, mf::kEpiGelu | SAVE, 256, gp, di, st, MF_K_GEMM_UP));
  }

  // 8. x += gate2 (hidden W_2^T + b_2)
  gp.gate_off = 5 * H;
  if (w8) {
    MF_TRY(quantize(hid, R));
    GemmSpec sp[2] = {{Nt, H, R, q8, w8->txt.q_2, w->txt.b_2, xt, H, 0, 0, w8->txt.s_2},
                      {Ni, H, R, q8 + (size_t)Nt * R, w8->img.q_2, w->img.b_2, xi, H, Nt, 1, w8->img.s_2}};
    MF_TRY(run_gemm(sp, 2, mf::kEpiGateResid | F8, 256, gp, di, st, MF_K_GEMM_DOWN));
  } else {
    GemmSpec sp[2] = {{Nt, H, R, hid, w->txt.w_2, w->txt.b_2, xt, H, 0, 0, nullptr, ym},
                      {Ni, H, R, hid + (size_t)Nt * R, w->img.w_2, w->img.b_2, xi, H, Nt, 1, nullptr,
                       ym ? ym + (size_t)Nt * H : nullptr}};
    MF_TRY(run_gemm(sp, 2, mf::kEpiGateResid | SAVE, 256, gp, di, st, MF_K_GEMM_DOWN));
  }
  return MF_OK;
}
}  // namespace

extern "C" mf_status mf_block_forward(const mf_plan* p, const mf_dims* d, const mf_block_weights* w,
                                      const float* d_t, void* d_x_txt, void* d_x_img, void* d_ws,
                                      size_t ws_bytes, void* stream) {
  return block_forward(p, d, w, nullptr, d_t, d_x_txt, d_x_img, d_ws, ws_bytes, stream);
}

extern "C" mf_status mf_block_forward_ex(const mf_plan* p, const mf_dims* d, const mf_block_weights* w,
                                         const float* d_t, void* d_x_txt, void* d_x_img, void* d_ws,
                                         size_t ws_bytes, int32_t flags, void* stream) {
  return block_forward(p, d, w, nullptr, d_t, d_x_txt, d_x_img, d_ws, ws_bytes, stream, false, flags);
}

extern "C" size_t mf_block_train_workspace_bytes(const mf_plan* p, const mf_dims* d) {
  if (p == nullptr || check_dims(d) != MF_OK) return 0;
  return train_layout(p, d).total;
}

extern "C" mf_status mf_block_forward_train(const mf_plan* p, const mf_dims* d, const mf_block_weights* w,
                                            const float* d_t, void* d_x_txt, void* d_x_img, void* d_ws,
                                            size_t ws_bytes, void* stream) {
  return block_forward(p, d, w, nullptr, d_t, d_x_txt, d_x_img, d_ws, ws_bytes, stream, true);
}

// ====================================================================== block backward
namespace {
mf_status attention_args(const mf_plan* p, int32_t heads, int32_t head_dim, DevInfo** di) {
  int dev = -1;
  MF_TRY(device_info(di, &dev));
  MF_TRY(check_plan(p, dev));
  if (heads <= 0) return MF_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return MF_ERR_UNSUPPORTED;
  return MF_OK;
}

// Backward workspace: the f32 dq accumulator [N][H], delta [heads][N] f32, do in joint order
// [N][H] bf16.
struct AttnBwdLayout {
  size_t acc, delta, do_joint, total;
};
AttnBwdLayout attn_bwd_layout(const mf_plan* p, int heads, int head_dim) {
  AttnBwdLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = al256(o + bytes); return r; };
  const size_t N = p->N, H = (size_t)heads * head_dim;
  L.acc = take(N * H * 4);
  L.delta = take((size_t)heads * N * 4);
  L.do_joint = take(N * H * 2);
  L.total = o;
  return L;
}

// CTAs of the attention backward: one per (sample, 128-key block, head).
long long attn_bwd_ctas(const mf_plan* p, int heads) {
  long long n = 0;
  for (int s = 0; s < p->S; ++s) n += (p->cu[s + 1] - p->cu[s] + 127) / 128;
  return n * heads;
}

mf_status attention_backward(const mf_plan* p, int heads, int head_dim, const bf16* q, const bf16* k,
                             const bf16* v, const bf16* o, const float* lse, const bf16* dout, int dout_joint,
                             bf16* dq, bf16* dk, bf16* dv, char* ws, const DevInfo* di, cudaStream_t st) {
  const int H = heads * head_dim, N = p->N;
  const AttnBwdLayout L = attn_bwd_layout(p, heads, head_dim);
  float* acc = reinterpret_cast<float*>(ws + L.acc);
  float* delta = reinterpret_cast<float*>(ws + L.delta);
  bf16* dj = dout_joint ? nullptr : reinterpret_cast<bf16*>(ws + L.do_joint);
  {
    Trace tr(MF_K_BLOCK_BWD, st, 0, (double)N * H * (2.0 + 2.0 + (dj ? 2.0 : 0.0) + 4.0), 1);
    MF_CUDA(mf::launch_attention_bwd_prep(o, dout, dout_joint, p->d_joint_srow, N, H, head_dim, dj, delta, acc,
                                          di->sms, st));
  }
  mf::AttnBwdParams bp{};
  if (!make_tmap(&bp.tmK, k, H, N, 128) || !make_tmap(&bp.tmV, v, H, N, 128) ||
      !make_tmap(&bp.tmQ, q, H, N, 64) || !make_tmap(&bp.tmDO, dj ? dj : dout, H, N, 64) ||
      !make_tmap_f32(&bp.tmDQ, acc, H, N, 32, 32))
    return MF_ERR_CUDA;
  bp.cu = p->d_cu;
  bp.items = p->d_items;
  bp.n_items = p->n_items;
  bp.lse = lse;
  bp.delta = delta;
  bp.dk = dk;
  bp.dv = dv;
  bp.n_tok = N;
  bp.n_seq = p->S;
  bp.H = H;
  bp.heads = heads;
  bp.head_dim = head_dim;
  bp.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)head_dim));
  bp.scale = (float)(1.0 / std::sqrt((double)head_dim));
  bp.status = di->status;
  bp.wait_limit_ns = wait_limit_ns();
  {
    // S^T, dP^T, dV, dK, dQ: five products of 2 L_i^2 D flops per head
    Trace tr(MF_K_ATTN_BWD, st, 10.0 * p->sum_L2 * H, 0, 1);
    MF_CUDA(mf::launch_attention_bwd(bp, attn_bwd_ctas(p, heads), st));
  }
  if (dq != nullptr) {
    Trace tr(MF_K_BLOCK_BWD, st, 0, (double)N * H * 6.0, 1);
    MF_CUDA(mf::launch_attention_bwd_dq(acc, dq, (long long)N * H, di->sms, st));
  }
  return MF_OK;
}
}  // namespace

namespace {
// Backward workspace: dmod [S][2][6H] f32; dy (the gated-residual gradients of the MLP and then
// the attention branch) [N][H] bf16; du [N][rH] bf16; da (LN + modulate output gradients) [N][H]
// bf16; dx1 [N][H] f32; do [N][H] bf16; dqkv [N][3H] bf16; dk, dv [N][H] bf16 joint order; the
// attention backward's own workspace.
struct BwdLayout {
  size_t dmod, dy, du, da, dx1, dout, dqkv, dk, dv, attn, rstats, total;
};

BwdLayout bwd_layout(const mf_plan* p, const mf_dims* d) {
  BwdLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = al256(o + bytes); return r; };
  const size_t S = p->S, N = p->N, H = d->hidden, R = (size_t)d->mlp_ratio * H;
  L.dmod = take(S * 12 * H * 4);
  L.dy = take(N * H * 2);
  L.du = take(N * R * 2);
  L.da = take(N * H * 2);
  L.dx1 = take(N * H * 4);
  L.dout = take(N * H * 2);
  L.dqkv = take(N * 3 * H * 2);
  L.dk = take(N * H * 2);
  L.dv = take(N * H * 2);
  L.attn = take(attn_bwd_layout(p, d->heads, H / d->heads).total);
  L.rstats = take(N * 16);
  L.total = o;
  return L;
}

bool grads_ok(const mf_stream_grads& g) {
  const float* ptrs[] = {g.w_mod, g.b_mod, g.w_qkv, g.b_qkv, g.w_o, g.b_o, g.w_1, g.b_1, g.w_2, g.b_2};
  for (const float* q : ptrs)
    if (q == nullptr || !aligned(q, 16)) return false;
  return true;
}
}  // namespace

extern "C" size_t mf_block_backward_workspace_bytes(const mf_plan* p, const mf_dims* d) {
  if (p == nullptr || check_dims(d) != MF_OK) return 0;
  return bwd_layout(p, d).total;
}

extern "C" mf_status mf_block_backward(const mf_plan* p, const mf_dims* d, const mf_block_weights* w,
                                       const void* d_train_ws, size_t train_ws_bytes, void* d_dx_txt,
                                       void* d_dx_img, const mf_block_grads* g, float* d_dc, void* d_ws,
                                       size_t ws_bytes, void* stream) {
  DevInfo* di = nullptr;
  int dev = -1;
  MF_TRY(device_info(&di, &dev));
  MF_TRY(check_plan(p, dev));
  MF_TRY(check_dims(d));
  if (w == nullptr || !stream_ok(w->txt) || !stream_ok(w->img) || g == nullptr || !grads_ok(g->txt) ||
      !grads_ok(g->img))
    return MF_ERR_INVALID_ARG;
  if (w->txt.w_qnorm != nullptr || w->img.w_qnorm != nullptr) return MF_ERR_UNSUPPORTED;
  if (p->N == 0) return MF_OK;
  if ((p->Nt > 0 && d_dx_txt == nullptr) || (p->Ni > 0 && d_dx_img == nullptr) || d_train_ws == nullptr ||
      d_ws == nullptr || d_dc == nullptr)
    return MF_ERR_INVALID_ARG;
  if (!aligned(d_dx_txt, 16) || !aligned(d_dx_img, 16) || !aligned(d_train_ws, 256) || !aligned(d_ws, 256) ||
      !aligned(d_dc, 16))
    return MF_ERR_ALIGNMENT;
  const TrainLayout TL = train_layout(p, d);
  const BwdLayout L = bwd_layout(p, d);
  if (train_ws_bytes < TL.total || ws_bytes < L.total) return MF_ERR_WORKSPACE;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const char* tw = static_cast<const char*>(d_train_ws);
  char* ws = static_cast<char*>(d_ws);
  const int S = p->S, N = p->N, Nt = p->Nt, Ni = p->Ni, H = d->hidden, heads = d->heads, D = H / heads;
  const int R = d->mlp_ratio * H;
  auto T = [&](size_t off) { return reinterpret_cast<const bf16*>(tw + off); };
  const float* c = reinterpret_cast<const float*>(tw + TL.base.off[0]);
  const float* mod = reinterpret_cast<const float*>(tw + TL.base.off[1]);
  const bf16* a2 = T(TL.base.off[2]);
  const bf16 *q = T(TL.base.off[3]), *k = T(TL.base.off[4]), *v = T(TL.base.off[5]), *o = T(TL.base.off[6]);
  const bf16* hid = T(TL.base.off[7]);
  const bf16 *x0 = T(TL.x0), *x1 = T(TL.x1), *a1 = T(TL.a1), *yo = T(TL.yo), *ym = T(TL.ym), *u = T(TL.u);
  const float* lse = reinterpret_cast<const float*>(tw + TL.lse);
  float* dmod = reinterpret_cast<float*>(ws + L.dmod);
  bf16* dy = reinterpret_cast<bf16*>(ws + L.dy);
  bf16* du = reinterpret_cast<bf16*>(ws + L.du);
  bf16* da = reinterpret_cast<bf16*>(ws + L.da);
  float* dx1 = reinterpret_cast<float*>(ws + L.dx1);
  bf16* dout = reinterpret_cast<bf16*>(ws + L.dout);
  bf16* dqkv = reinterpret_cast<bf16*>(ws + L.dqkv);
  bf16* dk = reinterpret_cast<bf16*>(ws + L.dk);
  bf16* dv = reinterpret_cast<bf16*>(ws + L.dv);
  bf16* gx_t = static_cast<bf16*>(d_dx_txt);
  bf16* gx_i = static_cast<bf16*>(d_dx_img);
  const mf_stream_grads* gs[2] = {&g->txt, &g->img};
  const mf_stream_weights* wsm[2] = {&w->txt, &w->img};
  const int rows[2] = {Nt, Ni}, roff[2] = {0, Nt};

  // accumulated outputs start at zero; a stream without rows has zero weight gradients
  MF_CUDA(cudaMemsetAsync(dmod, 0, (size_t)S * 12 * H * 4, st));
  for (int m = 0; m < 2; ++m) {
    MF_CUDA(cudaMemsetAsync(gs[m]->b_o, 0, (size_t)H * 4, st));
    MF_CUDA(cudaMemsetAsync(gs[m]->b_1, 0, (size_t)R * 4, st));
    MF_CUDA(cudaMemsetAsync(gs[m]->b_2, 0, (size_t)H * 4, st));
    MF_CUDA(cudaMemsetAsync(gs[m]->b_qkv, 0, (size_t)3 * H * 4, st));
    if (rows[m] == 0) {
      MF_CUDA(cudaMemsetAsync(gs[m]->w_qkv, 0, (size_t)3 * H * H * 4, st));
      MF_CUDA(cudaMemsetAsync(gs[m]->w_o, 0, (size_t)H * H * 4, st));
      MF_CUDA(cudaMemsetAsync(gs[m]->w_1, 0, (size_t)R * H * 4, st));
      MF_CUDA(cudaMemsetAsync(gs[m]->w_2, 0, (size_t)H * R * 4, st));
    }
  }
  mf::RowBwdArgs ra{};
  ra.H = H;
  ra.n_first = Nt;
  ra.chunks = p->d_row_chunks;
  ra.n_chunks = p->n_row_chunks;
  ra.g_first = gx_t;
  ra.g_second = gx_i;
  ra.mod = mod;
  ra.dmod = dmod;
  ra.n_rows = N;
  ra.n_seq = S;
  ra.row_seq = p->d_srow_seq;
  ra.stats = reinterpret_cast<float4*>(ws + L.rstats);
  mf::GemmParams gp{};
  // input-gradient GEMM per stream: out[rows][N] = A[rows][K] W, W stored [K][N]
  auto dgrad = [&](const bf16* A, int K, int Nn, const void* W0, const void* W1, bf16* out, int epi,
                   const bf16* aux, int kind) -> mf_status {
    GemmSpec sp[2];
    int n = 0;
    for (int m = 0; m < 2; ++m) {
      if (rows[m] == 0) continue;
      sp[n++] = GemmSpec{rows[m], Nn, K, A + (size_t)roff[m] * K, m ? W1 : W0, nullptr, out + (size_t)roff[m] * Nn,
                         Nn, roff[m], m, nullptr, aux ? const_cast<bf16*>(aux) + (size_t)roff[m] * Nn : nullptr};
    }
    (void)kind;
    return run_gemm(sp, n, epi, 256, gp, di, st, MF_K_GEMM_DGRAD, mf::kMajBMN);
  };
  // weight-gradient GEMM per stream: dW[Mo][Ni] = dY^T X over the stream's rows
  auto wgrad = [&](const bf16* dY, int Mo, const bf16* X, int Nn, float* out0, float* out1, int kind) -> mf_status {
    GemmSpec sp[2];
    int n = 0;
    for (int m = 0; m < 2; ++m) {
      if (rows[m] == 0) continue;
      sp[n++] = GemmSpec{Mo, Nn, rows[m], dY + (size_t)roff[m] * Mo, X + (size_t)roff[m] * Nn, nullptr,
                         m ? out1 : out0, Nn, 0, m};
    }
    (void)kind;
    return run_gemm(sp, n, mf::kEpiBiasF32, 256, gp, di, st, MF_K_GEMM_WGRAD, mf::kMajMNMN);
  };
  auto row_kernel = [&](int mode, double bytes_per_row) -> mf_status {
    ra.mode = mode;
    Trace tr(MF_K_BLOCK_BWD, st, 0, bytes_per_row * N, 1);
    return cuda_status(mf::launch_row_bwd(ra, st));
  };

  // 1. MLP branch: dy_m = gate2 g; dgate2, db_2
  ra.y = ym;
  ra.out_bf16 = dy;
  ra.bias_grad[0] = gs[0]->b_2;
  ra.bias_grad[1] = gs[1]->b_2;
  MF_TRY(row_kernel(mf::kRowGate2, 6.0 * H));
  // 2. du = (dy_m W_2) * GELU'(u);  dW_2 = dy_m^T h
  MF_TRY(dgrad(dy, H, R, w->txt.w_2, w->img.w_2, du, mf::kEpiGeluBwd, u, MF_K_GEMM_DOWN));
  MF_TRY(wgrad(dy, H, hid, R, gs[0]->w_2, gs[1]->w_2, MF_K_GEMM_DOWN));
  // 3. da_2 = du W_1;  dW_1 = du^T a_2;  db_1
  MF_TRY(dgrad(du, R, H, w->txt.w_1, w->img.w_1, da, mf::kEpiBiasBf16, nullptr, MF_K_GEMM_UP));
  MF_TRY(wgrad(du, R, a2, H, gs[0]->w_1, gs[1]->w_1, MF_K_GEMM_UP));
  {
    Trace tr(MF_K_BLOCK_BWD, st, 0, 2.0 * N * R, 1);
    MF_CUDA(mf::launch_col_sum(du, R, p->d_row_chunks, p->n_row_chunks, gs[0]->b_1, gs[1]->b_1, st));
  }
  // 4. LN + modulate #2 backward: dx1 = g + LN'(da_2 (1 + scale2)); dy_o = gate1 dx1; dshift2,
  //    dscale2, dgate1, db_o
  ra.da = da;
  ra.x = x1;
  ra.y = yo;
  ra.out_f32 = dx1;
  ra.out_bf16 = dy;
  ra.bias_grad[0] = gs[0]->b_o;
  ra.bias_grad[1] = gs[1]->b_o;
  MF_TRY(row_kernel(mf::kRowLn2, 16.0 * H));
  // 5. do = dy_o W_o;  dW_o = dy_o^T o
  MF_TRY(dgrad(dy, H, H, w->txt.w_o, w->img.w_o, dout, mf::kEpiBiasBf16, nullptr, MF_K_GEMM_OPROJ));
  MF_TRY(wgrad(dy, H, o, H, gs[0]->w_o, gs[1]->w_o, MF_K_GEMM_OPROJ));
  // 6. attention backward (dq kept in the f32 accumulator), then dqkv with the inverse RoPE
  char* aws = ws + L.attn;
  MF_TRY(attention_backward(p, heads, D, q, k, v, o, lse, dout, 0, nullptr, dk, dv, aws, di, st));
  {
    Trace tr(MF_K_BLOCK_BWD, st, 0, (double)N * H * (4.0 + 2.0 + 2.0 + 6.0), 1);
    MF_CUDA(mf::launch_qkv_grad_gather(reinterpret_cast<const float*>(aws + attn_bwd_layout(p, heads, D).acc), dk, dv,
                                       p->d_srow_joint, p->d_pos, N, H, D, dqkv, di->sms, st));
  }
  // 7. da_1 = dqkv W_qkv;  dW_qkv = dqkv^T a_1;  db_qkv
  MF_TRY(dgrad(dqkv, 3 * H, H, w->txt.w_qkv, w->img.w_qkv, da, mf::kEpiBiasBf16, nullptr, MF_K_GEMM_QKV));
  MF_TRY(wgrad(dqkv, 3 * H, a1, H, gs[0]->w_qkv, gs[1]->w_qkv, MF_K_GEMM_QKV));
  {
    Trace tr(MF_K_BLOCK_BWD, st, 0, 2.0 * N * 3 * H, 1);
    MF_CUDA(mf::launch_col_sum(dqkv, 3 * H, p->d_row_chunks, p->n_row_chunks, gs[0]->b_qkv, gs[1]->b_qkv, st));
  }
  // 8. LN + modulate #1 backward: dx0 = dx1 + LN'(da_1 (1 + scale1)) into the caller's buffers;
  //    dshift1, dscale1
  ra.x = x0;
  ra.carry = dx1;
  ra.out_first = gx_t;
  ra.out_second = gx_i;
  MF_TRY(row_kernel(mf::kRowLn1, 14.0 * H));
  // 9. modulation: dW_mod = dmod^T c, db_mod, dc = W_mod^T dmod (both streams)
  {
    Trace tr(MF_K_BLOCK_BWD, st, 2.0 * 2 * 2 * S * 6.0 * H * H, 2.0 * 6.0 * H * H * (4.0 + 2.0), 3);
    MF_CUDA(mf::launch_mod_bwd(dmod, c, S, H, static_cast<const bf16*>(w->txt.w_mod),
                               static_cast<const bf16*>(w->img.w_mod), gs[0]->w_mod, gs[0]->b_mod, gs[1]->w_mod,
                               gs[1]->b_mod, d_dc, st));
  }
  (void)wsm;
  return MF_OK;
}

extern "C" size_t mf_block_fp8_workspace_bytes(const mf_plan* p, const mf_dims* d) {
  if (p == nullptr || check_dims(d) != MF_OK) return 0;
  return block_layout(p, d).total + fp8_region_bytes(p, d);
}

extern "C" mf_status mf_block_forward_fp8(const mf_plan* p, const mf_dims* d, const mf_block_weights* w,
                                          const mf_block_weights_fp8* w8, const float* d_t, void* d_x_txt,
                                          void* d_x_img, void* d_ws, size_t ws_bytes, void* stream) {
  if (w8 == nullptr) return MF_ERR_INVALID_ARG;
  return block_forward(p, d, w, w8, d_t, d_x_txt, d_x_img, d_ws, ws_bytes, stream);
}

// ====================================================================== embed / final
extern "C" mf_status mf_embed(const mf_plan* p, const mf_dims* d, const void* w_in, const void* b_in,
                              const void* d_zt, void* d_x_img, void* stream) {
  DevInfo* di = nullptr;
  int dev = -1;
  MF_TRY(device_info(&di, &dev));
  MF_TRY(check_plan(p, dev));
  MF_TRY(check_dims(d));
  if (w_in == nullptr || b_in == nullptr) return MF_ERR_INVALID_ARG;
  if (p->Ni == 0) return MF_OK;
  if (d_zt == nullptr || d_x_img == nullptr) return MF_ERR_INVALID_ARG;
  if (!aligned(w_in, 16) || !aligned(b_in, 16) || !aligned(d_zt, 16) || !aligned(d_x_img, 16))
    return MF_ERR_ALIGNMENT;
  const int H = d->hidden, C = d->channels;
  mf::GemmParams gp{};
  GemmSpec sp[1] = {{p->Ni, H, C, d_zt, w_in, b_in, d_x_img, H, 0, 1}};
  return run_gemm(sp, 1, mf::kEpiBiasBf16, H >= 256 ? 256 : 128, gp, di,
                  static_cast<cudaStream_t>(stream), MF_K_GEMM_EMBED);
}

extern "C" size_t mf_final_workspace_bytes(const mf_plan* p, const mf_dims* d) {
  if (p == nullptr || check_dims(d) != MF_OK) return 0;
  return final_layout(p, d).total;
}

namespace {
// The final layer; d_c (device f32 [S][H]) is the timestep condition when the caller already has
// it, else it is computed into the workspace.
mf_status final_layer(const mf_plan* p, const mf_dims* d, const mf_temb_weights* temb, const void* w_fmod,
                      const void* b_fmod, const void* w_out, const void* b_out, const float* d_t,
                      const void* d_x_img, float* d_v, void* d_ws, size_t ws_bytes, const float* d_c,
                      void* stream) {
  DevInfo* di = nullptr;
  int dev = -1;
  MF_TRY(device_info(&di, &dev));
  MF_TRY(check_plan(p, dev));
  MF_TRY(check_dims(d));
  if (!temb_ok(temb) || w_fmod == nullptr || b_fmod == nullptr || w_out == nullptr || b_out == nullptr)
    return MF_ERR_INVALID_ARG;
  if (p->Ni == 0) return MF_OK;
  if (d_x_img == nullptr || d_v == nullptr || d_ws == nullptr) return MF_ERR_INVALID_ARG;
  if (!aligned(w_fmod, 16) || !aligned(w_out, 16) || !aligned(b_out, 16) || !aligned(d_x_img, 16) ||
      !aligned(d_v, 16) || !aligned(d_ws, 256) || !aligned(d_t, 4))
    return MF_ERR_ALIGNMENT;
  const FinalLayout L = final_layout(p, d);
  if (ws_bytes < L.total) return MF_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(d_ws);
  const int S = p->S, H = d->hidden, C = d->channels;
  const float* t = d_t ? d_t : p->d_t;
  if (!aligned(d_c, 16)) return MF_ERR_ALIGNMENT;
  const float* c = d_c ? d_c : reinterpret_cast<const float*>(ws + L.c);
  float* fmod = reinterpret_cast<float*>(ws + L.fmod);
  bf16* a = reinterpret_cast<bf16*>(ws + L.a);
  if (d_c == nullptr)
    MF_TRY(conditioning(p, d, temb, t, reinterpret_cast<float*>(ws + L.sinus),
                        reinterpret_cast<float*>(ws + L.h1), reinterpret_cast<float*>(ws + L.c), di, st));
  {
    Trace tr(MF_K_COND, st, 2.0 * S * 2.0 * H * H, 2.0 * 2.0 * H * H, (S + 3) / 4);
    MF_CUDA(mf::launch_gemv(static_cast<const bf16*>(w_fmod), static_cast<const bf16*>(b_fmod), c, S, H,
                            2 * H, fmod, 2 * H, 0, 0, di->status, wait_limit_ns(), st));
  }
  mf::LnModArgs ln{static_cast<const bf16*>(d_x_img), nullptr, p->Ni, p->Ni, H,
                   p->d_srow_seq + p->Nt, fmod, 2LL * H, 0, 0, H, a, p->S, nullptr, di->status,
                   wait_limit_ns()};
  {
    Trace tr(MF_K_LN, st, 0, 4.0 * p->Ni * H, 1);
    MF_CUDA(launch_ln(ln, 0, st));
  }
  mf::GemmParams gp{};
  GemmSpec sp[1] = {{p->Ni, C, H, a, w_out, b_out, d_v, C, 0, 1}};
  return run_gemm(sp, 1, mf::kEpiBiasF32, 128, gp, di, st, MF_K_GEMM_FINAL);
}
}  // namespace

extern "C" mf_status mf_final(const mf_plan* p, const mf_dims* d, const mf_temb_weights* temb,
                              const void* w_fmod, const void* b_fmod, const void* w_out,
                              const void* b_out, const float* d_t, const void* d_x_img, float* d_v,
                              void* d_ws, size_t ws_bytes, void* stream) {
  return final_layer(p, d, temb, w_fmod, b_fmod, w_out, b_out, d_t, d_x_img, d_v, d_ws, ws_bytes, nullptr,
                     stream);
}

extern "C" mf_status mf_final_ex(const mf_plan* p, const mf_dims* d, const mf_temb_weights* temb,
                                 const void* w_fmod, const void* b_fmod, const void* w_out,
                                 const void* b_out, const float* d_t, const void* d_x_img, float* d_v,
                                 void* d_ws, size_t ws_bytes, const float* d_c, void* stream) {
  return final_layer(p, d, temb, w_fmod, b_fmod, w_out, b_out, d_t, d_x_img, d_v, d_ws, ws_bytes, d_c, stream);
}

// ====================================================================== rectified-flow epilogues
namespace {
mf_status check_latent_call(const mf_plan* p, int32_t C, DevInfo** di) {
  int dev = -1;
  MF_TRY(device_info(di, &dev));
  MF_TRY(check_plan(p, dev));
  if (C <= 0 || C % 4 != 0) return MF_ERR_INVALID_ARG;
  return MF_OK;
}
}  // namespace

extern "C" mf_status mf_interpolate(const mf_plan* p, int32_t C, const float* d_t, const float* d_z,
                                    const float* d_eps, float* d_zt, void* d_zt_bf16, void* stream) {
  DevInfo* di = nullptr;
  MF_TRY(check_latent_call(p, C, &di));
  if (p->Ni == 0) return MF_OK;
  if (d_z == nullptr || d_eps == nullptr || (d_zt == nullptr && d_zt_bf16 == nullptr))
    return MF_ERR_INVALID_ARG;
  if (!aligned(d_z, 16) || !aligned(d_eps, 16) || !aligned(d_zt, 16) || !aligned(d_zt_bf16, 16) ||
      !aligned(d_t, 4))
    return MF_ERR_ALIGNMENT;
  Trace tr(MF_K_LATENT, static_cast<cudaStream_t>(stream), 0,
           (double)p->Ni * C * (8.0 + (d_zt ? 4.0 : 0.0) + (d_zt_bf16 ? 2.0 : 0.0)), 1);
  return cuda_status(mf::launch_interpolate(p->d_img_seq, p->d_img_target, d_t ? d_t : p->d_t, p->Ni, C,
                                            d_z, d_eps, d_zt, static_cast<bf16*>(d_zt_bf16),
                                            static_cast<cudaStream_t>(stream)));
}

extern "C" mf_status mf_cfg_combine(const mf_plan* p, int32_t C, float w, const float* d_v,
                                    float* d_v_out, void* stream) {
  DevInfo* di = nullptr;
  MF_TRY(check_latent_call(p, C, &di));
  if (p->Ni == 0) return MF_OK;
  if (d_v == nullptr || d_v_out == nullptr || !std::isfinite(w)) return MF_ERR_INVALID_ARG;
  if (!aligned(d_v, 16) || !aligned(d_v_out, 16)) return MF_ERR_ALIGNMENT;
  const size_t bytes = (size_t)p->Ni * C * 4;
  const char* a = reinterpret_cast<const char*>(d_v);
  const char* b = reinterpret_cast<const char*>(d_v_out);
  if (a != b && a < b + bytes && b < a + bytes) return MF_ERR_INVALID_ARG;  // partial overlap
  Trace tr(MF_K_LATENT, static_cast<cudaStream_t>(stream), 0, (double)p->Ni * C * 8.0, 1);
  return cuda_status(mf::launch_cfg(p->d_img_seq, p->d_seq_role, p->d_img_pair, p->Ni, C, w, d_v,
                                    d_v_out, static_cast<cudaStream_t>(stream)));
}

extern "C" mf_status mf_euler_step(const mf_plan* p, int32_t C, float dt, const float* d_v, float* d_z,
                                   void* d_z_bf16, void* stream) {
  DevInfo* di = nullptr;
  MF_TRY(check_latent_call(p, C, &di));
  if (p->Ni == 0) return MF_OK;
  if (d_v == nullptr || d_z == nullptr || !std::isfinite(dt)) return MF_ERR_INVALID_ARG;
  if (!aligned(d_v, 16) || !aligned(d_z, 16) || !aligned(d_z_bf16, 16)) return MF_ERR_ALIGNMENT;
  Trace tr(MF_K_LATENT, static_cast<cudaStream_t>(stream), 0,
           (double)p->Ni * C * (12.0 + (d_z_bf16 ? 2.0 : 0.0)), 1);
  return cuda_status(mf::launch_euler(p->Ni, C, dt, d_v, d_z, static_cast<bf16*>(d_z_bf16),
                                      static_cast<cudaStream_t>(stream)));
}

extern "C" size_t mf_flow_loss_workspace_bytes(const mf_plan* p) {
  if (p == nullptr) return 0;
  return al256((size_t)(p->Ni > 0 ? p->Ni : 1) * sizeof(double));
}

extern "C" mf_status mf_flow_loss(const mf_plan* p, int32_t C, const float* d_z, const float* d_eps,
                                  const float* d_v, double* d_loss_sum, int64_t* d_count,
                                  double* d_mean, void* d_ws, size_t ws_bytes, void* stream) {
  DevInfo* di = nullptr;
  MF_TRY(check_latent_call(p, C, &di));
  if (d_loss_sum == nullptr || d_count == nullptr || d_mean == nullptr) return MF_ERR_INVALID_ARG;
  if (p->Ni > 0 && (d_z == nullptr || d_eps == nullptr || d_v == nullptr || d_ws == nullptr))
    return MF_ERR_INVALID_ARG;
  if (!aligned(d_z, 16) || !aligned(d_eps, 16) || !aligned(d_v, 16) || !aligned(d_loss_sum, 8) ||
      !aligned(d_count, 8) || !aligned(d_mean, 8) || !aligned(d_ws, 256))
    return MF_ERR_ALIGNMENT;
  if (ws_bytes < mf_flow_loss_workspace_bytes(p)) return MF_ERR_WORKSPACE;
  Trace tr(MF_K_LOSS, static_cast<cudaStream_t>(stream), 0, (double)p->Ni * C * 12.0, 3);
  return cuda_status(mf::launch_flow_loss(p->d_cui, p->d_img_target, p->S, p->Ni, C, d_z, d_eps, d_v,
                                          static_cast<double*>(d_ws), d_loss_sum,
                                          reinterpret_cast<long long*>(d_count), d_mean,
                                          static_cast<cudaStream_t>(stream)));
}

extern "C" mf_status mf_nft_loss(const mf_plan* p, int32_t C, const float* d_z, const float* d_eps,
                                 const float* d_v_pos, const float* d_v_neg, const float* d_reward,
                                 double* d_loss_sum, int64_t* d_count, double* d_mean, void* d_ws,
                                 size_t ws_bytes, void* stream) {
  DevInfo* di = nullptr;
  MF_TRY(check_latent_call(p, C, &di));
  if (d_loss_sum == nullptr || d_count == nullptr || d_mean == nullptr) return MF_ERR_INVALID_ARG;
  if (p->Ni > 0 && (d_z == nullptr || d_eps == nullptr || d_v_pos == nullptr || d_v_neg == nullptr ||
                    d_reward == nullptr || d_ws == nullptr))
    return MF_ERR_INVALID_ARG;
  if (!aligned(d_z, 16) || !aligned(d_eps, 16) || !aligned(d_v_pos, 16) || !aligned(d_v_neg, 16) ||
      !aligned(d_reward, 4) || !aligned(d_loss_sum, 8) || !aligned(d_count, 8) || !aligned(d_mean, 8) ||
      !aligned(d_ws, 256))
    return MF_ERR_ALIGNMENT;
  if (ws_bytes < mf_flow_loss_workspace_bytes(p)) return MF_ERR_WORKSPACE;
  Trace tr(MF_K_LOSS, static_cast<cudaStream_t>(stream), 0, (double)p->Ni * C * 16.0, 3);
  return cuda_status(mf::launch_nft_loss(p->d_cui, p->d_img_seq, p->d_img_target, d_reward, p->S, p->Ni,
                                         C, d_z, d_eps, d_v_pos, d_v_neg, static_cast<double*>(d_ws),
                                         d_loss_sum, reinterpret_cast<long long*>(d_count), d_mean,
                                         static_cast<cudaStream_t>(stream)));
}

// ====================================================================== building blocks
extern "C" mf_status mf_attention(const mf_plan* p, int32_t heads, int32_t head_dim, const void* d_q,
                                  const void* d_k, const void* d_v, void* d_o, void* stream) {
  DevInfo* di = nullptr;
  int dev = -1;
  MF_TRY(device_info(&di, &dev));
  MF_TRY(check_plan(p, dev));
  if (heads <= 0) return MF_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return MF_ERR_UNSUPPORTED;
  if (p->N == 0) return MF_OK;
  if (d_q == nullptr || d_k == nullptr || d_v == nullptr || d_o == nullptr) return MF_ERR_INVALID_ARG;
  if (!aligned(d_q, 16) || !aligned(d_k, 16) || !aligned(d_v, 16) || !aligned(d_o, 16))
    return MF_ERR_ALIGNMENT;
  const int H = heads * head_dim;
  mf::AttnParams ap{};
  if (!make_tmap(&ap.tmQ, d_q, H, p->N, 128) || !make_tmap(&ap.tmK, d_k, H, p->N, 128) ||
      !make_tmap(&ap.tmV, d_v, H, p->N, 128))
    return MF_ERR_CUDA;
  ap.cu = p->d_cu;
  ap.items = p->d_items;
  ap.joint_srow = p->d_joint_srow;
  ap.out = static_cast<bf16*>(d_o);
  ap.H = H;
  ap.heads = heads;
  ap.n_items = p->n_items;
  ap.n_tok = p->N;
  ap.n_seq = p->S;
  ap.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)head_dim));
  ap.status = di->status;
  ap.wait_limit_ns = wait_limit_ns();
  Trace tr(MF_K_ATTN, static_cast<cudaStream_t>(stream), 4.0 * p->sum_L2 * H, 0, 1);
  return cuda_status(mf::launch_attention(ap, head_dim, static_cast<cudaStream_t>(stream)));
}

extern "C" mf_status mf_attention_lse(const mf_plan* p, int32_t heads, int32_t head_dim, const void* d_q,
                                      const void* d_k, const void* d_v, void* d_o, float* d_lse, void* stream) {
  DevInfo* di = nullptr;
  MF_TRY(attention_args(p, heads, head_dim, &di));
  if (p->N == 0) return MF_OK;
  if (d_q == nullptr || d_k == nullptr || d_v == nullptr || d_o == nullptr || d_lse == nullptr)
    return MF_ERR_INVALID_ARG;
  if (!aligned(d_q, 16) || !aligned(d_k, 16) || !aligned(d_v, 16) || !aligned(d_o, 16) || !aligned(d_lse, 16))
    return MF_ERR_ALIGNMENT;
  const int H = heads * head_dim;
  mf::AttnParams ap{};
  if (!make_tmap(&ap.tmQ, d_q, H, p->N, 128) || !make_tmap(&ap.tmK, d_k, H, p->N, 128) ||
      !make_tmap(&ap.tmV, d_v, H, p->N, 128))
    return MF_ERR_CUDA;
  ap.cu = p->d_cu;
  ap.items = p->d_items;
  ap.joint_srow = p->d_joint_srow;
  ap.out = static_cast<bf16*>(d_o);
  ap.lse = d_lse;
  ap.H = H;
  ap.heads = heads;
  ap.n_items = p->n_items;
  ap.n_tok = p->N;
  ap.n_seq = p->S;
  ap.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)head_dim));
  ap.status = di->status;
  ap.wait_limit_ns = wait_limit_ns();
  Trace tr(MF_K_ATTN, static_cast<cudaStream_t>(stream), 4.0 * p->sum_L2 * H, 0, 1);
  return cuda_status(mf::launch_attention(ap, head_dim, static_cast<cudaStream_t>(stream)));
}

extern "C" size_t mf_attention_backward_workspace_bytes(const mf_plan* p, int32_t heads, int32_t head_dim) {
  if (p == nullptr || heads <= 0 || (head_dim != 64 && head_dim != 128)) return 0;
  return attn_bwd_layout(p, heads, head_dim).total;
}

extern "C" mf_status mf_attention_backward(const mf_plan* p, int32_t heads, int32_t head_dim, const void* d_q,
                                           const void* d_k, const void* d_v, const void* d_o, const float* d_lse,
                                           const void* d_do, void* d_dq, void* d_dk, void* d_dv, void* d_ws,
                                           size_t ws_bytes, void* stream) {
  DevInfo* di = nullptr;
  MF_TRY(attention_args(p, heads, head_dim, &di));
  if ((heads * head_dim) % 256 != 0) return MF_ERR_UNSUPPORTED;
  if (p->N == 0) return MF_OK;
  const void* ptrs[] = {d_q, d_k, d_v, d_o, d_lse, d_do, d_dq, d_dk, d_dv, d_ws};
  for (const void* x : ptrs)
    if (x == nullptr) return MF_ERR_INVALID_ARG;
  for (const void* x : ptrs)
    if (!aligned(x, 16)) return MF_ERR_ALIGNMENT;
  if (!aligned(d_ws, 256)) return MF_ERR_ALIGNMENT;
  if (ws_bytes < attn_bwd_layout(p, heads, head_dim).total) return MF_ERR_WORKSPACE;
  return attention_backward(p, heads, head_dim, static_cast<const bf16*>(d_q), static_cast<const bf16*>(d_k),
                            static_cast<const bf16*>(d_v), static_cast<const bf16*>(d_o), d_lse,
                            static_cast<const bf16*>(d_do), 0, static_cast<bf16*>(d_dq), static_cast<bf16*>(d_dk),
                            static_cast<bf16*>(d_dv), static_cast<char*>(d_ws), di, static_cast<cudaStream_t>(stream));
}

extern "C" mf_status mf_quantize_fp8_rows(int32_t M, int32_t K, const void* d_x, void* d_q, float* d_scale,
                                          void* stream) {
  DevInfo* di = nullptr;
  MF_TRY(device_info(&di));
  if (M < 0 || K <= 0 || K % 16 != 0) return MF_ERR_INVALID_ARG;
  if (M == 0) return MF_OK;
  if (d_x == nullptr || d_q == nullptr || d_scale == nullptr) return MF_ERR_INVALID_ARG;
  if (!aligned(d_x, 16) || !aligned(d_q, 16) || !aligned(d_scale, 4)) return MF_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Trace tr(MF_K_FP8, st, 0, 3.0 * M * (double)K + 4.0 * M, 1);
  return cuda_status(mf::launch_quantize_e4m3_rows(static_cast<const bf16*>(d_x), M, K,
                                                   static_cast<uint8_t*>(d_q), d_scale, st));
}

extern "C" mf_status mf_gemm_fp8(int32_t M, int32_t N, int32_t K, const void* d_a, const float* d_a_scale,
                                 const void* d_b, const float* d_b_scale, const void* d_bias, void* d_c,
                                 void* stream) {
  DevInfo* di = nullptr;
  MF_TRY(device_info(&di));
  if (M < 0 || N <= 0 || K <= 0 || K % 128 != 0 || N % 16 != 0) return MF_ERR_INVALID_ARG;
  if (M == 0) return MF_OK;
  if (d_a == nullptr || d_b == nullptr || d_c == nullptr || d_a_scale == nullptr || d_b_scale == nullptr)
    return MF_ERR_INVALID_ARG;
  if (!aligned(d_a, 16) || !aligned(d_b, 16) || !aligned(d_c, 16) || !aligned(d_bias, 16) ||
      !aligned(d_a_scale, 4) || !aligned(d_b_scale, 16))
    return MF_ERR_ALIGNMENT;
  mf::GemmParams gp{};
  gp.row_scale = d_a_scale;
  GemmSpec sp[1] = {{M, N, K, d_a, d_b, d_bias, d_c, N, 0, 0, d_b_scale}};
  return run_gemm(sp, 1, mf::kEpiBiasBf16 | mf::kEpiF8, 256, gp, di, static_cast<cudaStream_t>(stream),
                  MF_K_FP8);
}

extern "C" mf_status mf_gemm(int32_t M, int32_t N, int32_t K, const void* d_a, const void* d_b,
                             const void* d_bias, void* d_c, int32_t out_f32, void* stream) {
  DevInfo* di = nullptr;
  MF_TRY(device_info(&di));
  if (M < 0 || N <= 0 || K <= 0 || N % 32 != 0 || K % 64 != 0) return MF_ERR_INVALID_ARG;
  if (M == 0) return MF_OK;
  if (d_a == nullptr || d_b == nullptr || d_c == nullptr) return MF_ERR_INVALID_ARG;
  if (!aligned(d_a, 16) || !aligned(d_b, 16) || !aligned(d_bias, 16) || !aligned(d_c, 16))
    return MF_ERR_ALIGNMENT;
  mf::GemmParams gp{};
  GemmSpec sp[1] = {{M, N, K, d_a, d_b, d_bias, d_c, N, 0, 0}};
  return run_gemm(sp, 1, out_f32 ? mf::kEpiBiasF32 : mf::kEpiBiasBf16, N <= 128 ? 128 : 256, gp, di,
                  static_cast<cudaStream_t>(stream), MF_K_GEMM_PLAIN);
}

// ====================================================================== status
extern "C" mf_status mf_check(void* stream) {
  DevInfo* di = nullptr;
  MF_TRY(device_info(&di));
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MF_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, di->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MF_ERR_CUDA;
  // bounds-check flags of the checked build (always 0 otherwise); read and cleared
  const unsigned bounds = mf::bounds_flag_gemm() | mf::bounds_flag_attention() | mf::bounds_flag_attention_bwd() |
                          mf::bounds_flag_pointwise() | mf::bounds_flag_block_bwd();
  if (bounds & 2u) return MF_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(di->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return MF_ERR_CUDA;
  }
  if (bounds != 0) return MF_ERR_DEVICE_BOUNDS;
  if (v != 0) return MF_ERR_DEVICE_TIMEOUT;
  return MF_OK;
}

extern "C" mf_status mf_selftest_timeout(int32_t limit_us, void* stream) {
  DevInfo* di = nullptr;
  MF_TRY(device_info(&di));
  if (limit_us < 1 || limit_us > 1000000) return MF_ERR_INVALID_ARG;
  MF_TRY(mf_check(stream));  // start from a clean status word
  Trace tr(MF_K_COND, static_cast<cudaStream_t>(stream), 0, 0, 1);
  if (mf::launch_timeout_selftest(di->status, (unsigned long long)limit_us * 1000ull,
                                  static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MF_ERR_CUDA;
  return mf_check(stream);
}

// ====================================================================== tracing
extern "C" mf_status mf_trace_kinds(uint32_t mask) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace.mask = mask;
  return MF_OK;
}

extern "C" mf_status mf_trace_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace.on = on != 0;
  if (g_trace.on) {
    for (auto& r : g_trace.recs) {
      g_trace.pool.push_back(r.a);
      g_trace.pool.push_back(r.b);
    }
    g_trace.recs.clear();
  }
  return MF_OK;
}

extern "C" mf_status mf_trace_read(mf_trace_entry* e, int32_t n) {
  if (e == nullptr || n < MF_K_COUNT) return MF_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_trace_mu);
  for (int i = 0; i < n; ++i) e[i] = mf_trace_entry{0, 0.0, 0.0, 0.0};
  mf_status st = MF_OK;
  for (auto& r : g_trace.recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
      st = MF_ERR_CUDA;
    if (r.kind >= 0 && r.kind < n) {
      e[r.kind].launches += r.nk;
      e[r.kind].ms += ms;
      e[r.kind].flops += r.flops;
      e[r.kind].bytes += r.bytes;
    }
    g_trace.pool.push_back(r.a);
    g_trace.pool.push_back(r.b);
  }
  g_trace.recs.clear();
  return st;
}

extern "C" int64_t mf_launch_count(void) { return g_launches.load(); }
