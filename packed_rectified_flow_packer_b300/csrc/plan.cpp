// Native-resolution packer: first-fit under a fixed token budget, and the index buffers of
// the pack (cu_seqlens, (frame, row, col) positions, stream <-> joint row maps, the CFG pair
// table, target-frame flags and the attention work list).
//
// Source: PaperReading review of "Mage-Flow: An Efficient Native-Resolution Foundation Model
// for Image Generation and Editing", section 2.2 (2) (variable-length text and latent tokens
// concatenated by cumulative offsets; attention only inside each sample; a per-sample 2-D
// RoPE, plus a frame index for editing), and the hyper.ai summary, section 方法 (packing
// under a fixed token budget).  The packing rule is read as first-fit in candidate order.
//
// Host code only: no CUDA call here, so packing works (and is tested) without a GPU.
#include <algorithm>
#include <cstring>
#include <new>

#include "internal.h"

namespace {

int64_t sample_len(const mf_sample& s) {
  return (int64_t)s.txt_len + (int64_t)s.frames * s.lat_h * s.lat_w;
}

mf_status validate(const mf_sample* s, int32_t n, int32_t budget) {
  if (budget < 1) return MF_ERR_BUDGET;
  if (n < 0 || (n > 0 && s == nullptr)) return MF_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    const mf_sample& a = s[i];
    if (a.txt_len < 0 || a.lat_h < 1 || a.lat_w < 1 || (a.frames != 1 && a.frames != 2))
      return MF_ERR_INVALID_ARG;
    if (a.cfg_role < 0 || a.cfg_role > 2) return MF_ERR_INVALID_ARG;
    if (!(a.t == a.t)) return MF_ERR_INVALID_ARG;  // NaN time
    if (sample_len(a) > budget) return MF_ERR_SAMPLE_TOO_LONG;
  }
  return MF_OK;
}

}  // namespace

extern "C" mf_status mf_pack(const mf_sample* samples, int32_t n, int32_t budget, mf_plan** out) {
  if (out == nullptr) return MF_ERR_INVALID_ARG;
  mf_status st = validate(samples, n, budget);
  if (st != MF_OK) return st;

  mf_plan* p = new (std::nothrow) mf_plan();
  if (p == nullptr) return MF_ERR_INVALID_ARG;
  p->budget = budget;

  // first-fit with skip, in candidate order
  int64_t used = 0;
  std::vector<int32_t> seq_of(n > 0 ? n : 1, -1);
  for (int32_t i = 0; i < n; ++i) {
    int64_t L = sample_len(samples[i]);
    if (used + L <= budget) {
      seq_of[i] = (int32_t)p->order.size();
      p->order.push_back(i);
      used += L;
    }
  }
  const int32_t S = (int32_t)p->order.size();
  p->S = S;
  p->cu.assign(S + 1, 0);
  p->cut.assign(S + 1, 0);
  p->cui.assign(S + 1, 0);
  for (int32_t k = 0; k < S; ++k) {
    const mf_sample& a = samples[p->order[k]];
    int32_t img = a.frames * a.lat_h * a.lat_w;
    p->cu[k + 1] = p->cu[k] + a.txt_len + img;
    p->cut[k + 1] = p->cut[k] + a.txt_len;
    p->cui[k + 1] = p->cui[k] + img;
  }
  const int32_t N = p->cu[S], Nt = p->cut[S], Ni = p->cui[S];
  p->N = N;
  p->Nt = Nt;
  p->Ni = Ni;
  p->pos.assign((size_t)N * 3, 0);
  p->txt_seq.resize(Nt);
  p->txt_joint.resize(Nt);
  p->img_seq.resize(Ni);
  p->img_joint.resize(Ni);
  p->img_pair.assign(Ni, -1);
  p->img_target.resize(Ni);
  p->seq_role.resize(S);
  p->t.resize(S);
  p->srow_joint.resize((size_t)Nt + Ni);
  p->srow_seq.resize((size_t)Nt + Ni);
  p->joint_srow.resize(N);

  for (int32_t k = 0; k < S; ++k) {
    const mf_sample& a = samples[p->order[k]];
    p->seq_role[k] = a.cfg_role;
    p->t[k] = a.t;
    int32_t j = p->cu[k];
    for (int32_t x = 0; x < a.txt_len; ++x) {
      int32_t r = p->cut[k] + x;
      p->txt_seq[r] = k;
      p->txt_joint[r] = j + x;
    }
    j += a.txt_len;
    const int32_t hw = a.lat_h * a.lat_w;
    const int32_t img = a.frames * hw;
    for (int32_t l = 0; l < img; ++l) {
      int32_t r = p->cui[k] + l;
      int32_t f = l / hw, rem = l - f * hw;
      p->img_seq[r] = k;
      p->img_joint[r] = j + l;
      int32_t* q = &p->pos[(size_t)(j + l) * 3];
      q[0] = f;
      q[1] = rem / a.lat_w;
      q[2] = rem - (rem / a.lat_w) * a.lat_w;
      p->img_target[r] = (f == a.frames - 1) ? 1 : 0;
    }
    if (a.cfg_role != 0) {
      int32_t c = p->order[k];
      int32_t pc = a.cfg_pair;
      if (pc < 0 || pc >= n || seq_of[pc] < 0) { delete p; return MF_ERR_INVALID_ARG; }
      const mf_sample& b = samples[pc];
      int32_t want = (a.cfg_role == 1) ? 2 : 1;
      if (b.cfg_role != want || b.cfg_pair != c || b.frames != a.frames || b.lat_h != a.lat_h ||
          b.lat_w != a.lat_w) {
        delete p;
        return MF_ERR_INVALID_ARG;
      }
      int32_t kp = seq_of[pc];
      for (int32_t l = 0; l < img; ++l) p->img_pair[p->cui[k] + l] = p->cui[kp] + l;
    }
  }

  for (int32_t r = 0; r < Nt; ++r) {
    p->srow_joint[r] = p->txt_joint[r];
    p->srow_seq[r] = p->txt_seq[r];
  }
  for (int32_t r = 0; r < Ni; ++r) {
    p->srow_joint[(size_t)Nt + r] = p->img_joint[r];
    p->srow_seq[(size_t)Nt + r] = p->img_seq[r];
  }
  for (int32_t r = 0; r < Nt + Ni; ++r) p->joint_srow[p->srow_joint[r]] = r;

  // attention work list: (sequence, 256-row query block), longest sequences first (stable)
  std::vector<int32_t> seqs(S);
  for (int32_t k = 0; k < S; ++k) seqs[k] = k;
  std::stable_sort(seqs.begin(), seqs.end(), [&](int32_t a, int32_t b) {
    return (p->cu[a + 1] - p->cu[a]) > (p->cu[b + 1] - p->cu[b]);
  });
  for (int32_t k : seqs) {
    int32_t L = p->cu[k + 1] - p->cu[k];
    p->sum_L2 += (double)L * (double)L;
    int32_t nq = (L + mf::kQBlock - 1) / mf::kQBlock;
    for (int32_t q = 0; q < nq; ++q) {
      p->items.push_back(k);
      p->items.push_back(q);
    }
  }
  p->n_items = (int32_t)(p->items.size() / 2);

  // row chunks of the backward's row kernels: stream-sorted rows in pieces of at most
  // kRowChunk rows, each inside one (sample, stream) segment, as (row0, row1, sample, stream)
  for (int32_t m = 0; m < 2; ++m)
    for (int32_t k = 0; k < S; ++k) {
      const int32_t a = m ? Nt + p->cui[k] : p->cut[k], b = m ? Nt + p->cui[k + 1] : p->cut[k + 1];
      for (int32_t r = a; r < b; r += mf::kRowChunk) {
        p->row_chunks.push_back(r);
        p->row_chunks.push_back(std::min(b, r + mf::kRowChunk));
        p->row_chunks.push_back(k);
        p->row_chunks.push_back(m);
      }
    }
  p->n_row_chunks = (int32_t)(p->row_chunks.size() / 4);
  *out = p;
  return MF_OK;
}

extern "C" mf_status mf_plan_get_info(const mf_plan* p, mf_plan_info* info) {
  if (p == nullptr || info == nullptr) return MF_ERR_INVALID_ARG;
  info->n_seq = p->S;
  info->n_tok = p->N;
  info->n_txt = p->Nt;
  info->n_img = p->Ni;
  info->n_items = p->n_items;
  info->budget = p->budget;
  info->uploaded = p->d_blob != nullptr || (p->N == 0 && p->device >= 0);
  info->reserved = 0;
  return MF_OK;
}

extern "C" mf_status mf_plan_array(const mf_plan* p, int32_t which, const int32_t** data,
                                   int64_t* len) {
  if (p == nullptr || data == nullptr || len == nullptr) return MF_ERR_INVALID_ARG;
  const std::vector<int32_t>* v = nullptr;
  switch (which) {
    case 0: v = &p->order; break;
    case 1: v = &p->cu; break;
    case 2: v = &p->cut; break;
    case 3: v = &p->cui; break;
    case 4: v = &p->pos; break;
    case 5: v = &p->txt_seq; break;
    case 6: v = &p->txt_joint; break;
    case 7: v = &p->img_seq; break;
    case 8: v = &p->img_joint; break;
    case 9: v = &p->img_pair; break;
    case 10: v = &p->img_target; break;
    case 11: v = &p->seq_role; break;
    case 12: v = &p->items; break;
    default: return MF_ERR_INVALID_ARG;
  }
  *data = v->data();
  *len = (int64_t)v->size();
  return MF_OK;
}

extern "C" const char* mf_status_str(mf_status s) {
  switch (s) {
    case MF_OK: return "MF_OK";
    case MF_ERR_INVALID_ARG: return "MF_ERR_INVALID_ARG";
    case MF_ERR_SAMPLE_TOO_LONG: return "MF_ERR_SAMPLE_TOO_LONG";
    case MF_ERR_BUDGET: return "MF_ERR_BUDGET";
    case MF_ERR_ALIGNMENT: return "MF_ERR_ALIGNMENT";
    case MF_ERR_CUDA: return "MF_ERR_CUDA";
    case MF_ERR_DEVICE_TIMEOUT: return "MF_ERR_DEVICE_TIMEOUT";
    case MF_ERR_UNSUPPORTED: return "MF_ERR_UNSUPPORTED";
    case MF_ERR_NOT_UPLOADED: return "MF_ERR_NOT_UPLOADED";
    case MF_ERR_WORKSPACE: return "MF_ERR_WORKSPACE";
    case MF_ERR_DEVICE_BOUNDS: return "MF_ERR_DEVICE_BOUNDS";
  }
  return "MF_ERR_UNKNOWN";
}

extern "C" int32_t mf_version(void) { return (1 << 16) | 0; }
