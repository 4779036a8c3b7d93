// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

#include "mageflow.h"

// A pack and every index buffer the kernels read.  Built once by mf_pack (host only) and
// immutable afterwards; mf_plan_upload copies the buffers to the device in one blob.
struct mf_plan {
  int32_t budget = 0;
  int32_t S = 0, N = 0, Nt = 0, Ni = 0, n_items = 0;
  double sum_L2 = 0.0;  // sum over samples of (sample length)^2: attention work

  std::vector<int32_t> order;       // [S]    candidate index per packed sample
  std::vector<int32_t> cu;          // [S+1]  joint offsets (cu_seqlens)
  std::vector<int32_t> cut;         // [S+1]  text-stream offsets
  std::vector<int32_t> cui;         // [S+1]  image-stream offsets
  std::vector<int32_t> pos;         // [N*3]  (frame, row, col) per joint token
  std::vector<int32_t> txt_seq, txt_joint;   // [Nt]
  std::vector<int32_t> img_seq, img_joint;   // [Ni]
  std::vector<int32_t> img_pair;    // [Ni]  CFG partner row or -1
  std::vector<int32_t> img_target;  // [Ni]  1 = target frame
  std::vector<int32_t> seq_role;    // [S]   cfg_role
  std::vector<int32_t> items;       // [n_items*2] (sequence, query block), longest first
  std::vector<int32_t> row_chunks;  // [n_row_chunks*4] (row0, row1, sample, stream): stream-sorted
                                    // rows in pieces of <= kRowChunk inside one segment
  int32_t n_row_chunks = 0;
  std::vector<float> t;             // [S]   flow time per packed sample

  // stream-sorted rows: text rows 0..Nt-1, then image rows Nt..Nt+Ni-1
  std::vector<int32_t> srow_joint;  // [Nt+Ni] joint token of each stream-sorted row
  std::vector<int32_t> srow_seq;    // [Nt+Ni] sample of each stream-sorted row
  std::vector<int32_t> joint_srow;  // [N]     stream-sorted row of each joint token

  // device copy (one allocation, owned by the plan)
  int device = -1;
  void* d_blob = nullptr;
  size_t blob_bytes = 0;
  const int32_t* d_cu = nullptr;
  const int32_t* d_cui = nullptr;
  const int32_t* d_pos = nullptr;
  const int32_t* d_srow_joint = nullptr;
  const int32_t* d_srow_seq = nullptr;
  const int32_t* d_joint_srow = nullptr;
  const int32_t* d_img_seq = nullptr;
  const int32_t* d_img_pair = nullptr;
  const int32_t* d_img_target = nullptr;
  const int32_t* d_seq_role = nullptr;
  const int32_t* d_items = nullptr;
  const int32_t* d_row_chunks = nullptr;
  const float* d_t = nullptr;
};

namespace mf {

constexpr int kQBlock = 256;  // query rows of one attention work item (two 128-row tiles)
constexpr int kRowChunk = 64; // rows of one chunk of the backward's row kernels

// Ordinal of the current device after checking that it is an sm_103a (the library's per-device
// state is set up on first use).  MF_ERR_UNSUPPORTED on another architecture, MF_ERR_CUDA when
// no device can be queried.
mf_status current_device(int* dev);

// Bounds-check flags of the checked build, one per translation unit with device code (read and
// cleared; always 0 in the default build).
unsigned bounds_flag_gemm();
unsigned bounds_flag_attention();
unsigned bounds_flag_attention_bwd();
unsigned bounds_flag_pointwise();
unsigned bounds_flag_block_bwd();

// One library launch of `nk` kernels of kind `kind` (mf_kernel_kind): counted always and, while
// tracing is on (and the stream is not capturing), bracketed by two CUDA events on `st` -
// the constructor records the first, the destructor the second.
class Trace {
 public:
  Trace(int kind, cudaStream_t st, double flops, double bytes, int nk);
  ~Trace();
  Trace(const Trace&) = delete;
  Trace& operator=(const Trace&) = delete;

 private:
  cudaStream_t st_;
  int kind_ = 0, nk_ = 0;
  cudaEvent_t a_ = nullptr, b_ = nullptr;
  double flops_ = 0.0, bytes_ = 0.0;
  bool active_ = false;
};

}  // namespace mf
