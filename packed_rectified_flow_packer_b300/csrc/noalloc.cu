// mf_flow_loss_noalloc: the flow-matching loss with its scratch in a fixed, library-owned
// device array instead of a caller-provided workspace.
//
// Who needs this: callers that cannot allocate device memory at the point where they compute
// the loss - for example code running under an allocator owned by another framework that
// forbids side allocations, callers on a fixed, pre-reserved memory budget, or code paths
// where an allocation call would synchronise the device at the wrong moment.  They still pass
// their own inputs and outputs; only the per-row partial sums live here.
//
// The scratch is one file-scope array per device, held for as long as the library is loaded.
// Every call on a device shares it, so two calls that overlap on the GPU (different streams,
// no ordering between them) race on it; order such calls on one stream.  Each call writes
// every scratch row it later reads (rows 0 .. N_img-1) before reading it, so contents left by
// an earlier call never reach a result and nothing has to be cleared first.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "pointwise.cuh"

namespace {

// Per-row partial sums of the loss (one double per image row of the pack).
static __device__ __align__(256) double g_noalloc_loss_rows[MF_NOALLOC_MAX_IMG_ROWS];

constexpr int kMaxDevices = 64;
double* g_rows_addr[kMaxDevices] = {};
std::mutex g_rows_mu;

// Device address of the scratch array on the current device.  In host code the array's name
// is only a host-side stand-in, so the address is looked up once per device, with that
// device current, and cached.
mf_status scratch_address(int dev, double** out) {
  std::lock_guard<std::mutex> lk(g_rows_mu);
  if (g_rows_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_loss_rows) != cudaSuccess || p == nullptr)
      return MF_ERR_CUDA;
    g_rows_addr[dev] = static_cast<double*>(p);
  }
  *out = g_rows_addr[dev];
  return MF_OK;
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" mf_status mf_flow_loss_noalloc(const mf_plan* p, int32_t C, const float* d_z,
                                          const float* d_eps, const float* d_v, double* d_loss_sum,
                                          int64_t* d_count, double* d_mean, void* stream) {
  int dev = -1;
  mf_status st = mf::current_device(&dev);  // sm_103a check, as every other entry point
  if (st != MF_OK) return st;
  if (dev >= kMaxDevices) return MF_ERR_CUDA;
  if (p == nullptr) return MF_ERR_INVALID_ARG;
  if (p->d_blob == nullptr) return MF_ERR_NOT_UPLOADED;
  if (p->device != dev) return MF_ERR_INVALID_ARG;
  if (C <= 0 || C % 4 != 0) return MF_ERR_INVALID_ARG;
  if (d_loss_sum == nullptr || d_count == nullptr || d_mean == nullptr) return MF_ERR_INVALID_ARG;
  if (p->Ni > 0 && (d_z == nullptr || d_eps == nullptr || d_v == nullptr)) return MF_ERR_INVALID_ARG;
  if (!aligned_to(d_z, 16) || !aligned_to(d_eps, 16) || !aligned_to(d_v, 16) ||
      !aligned_to(d_loss_sum, 8) || !aligned_to(d_count, 8) || !aligned_to(d_mean, 8))
    return MF_ERR_ALIGNMENT;
  if (p->Ni > MF_NOALLOC_MAX_IMG_ROWS) return MF_ERR_WORKSPACE;
  double* rows = nullptr;
  st = scratch_address(dev, &rows);
  if (st != MF_OK) return st;
  // counted and traced like mf_flow_loss (same kind, bytes and kernel count)
  mf::Trace tr(MF_K_LOSS, static_cast<cudaStream_t>(stream), 0, (double)p->Ni * C * 12.0, 3);
  cudaError_t e = mf::launch_flow_loss(p->d_cui, p->d_img_target, p->S, p->Ni, C, d_z, d_eps, d_v, rows,
                                       d_loss_sum, reinterpret_cast<long long*>(d_count), d_mean,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MF_OK : MF_ERR_CUDA;
}
