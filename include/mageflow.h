/*
 * mageflow.h - C ABI of libmageflow.so: the packed NR-MMDiT block forward and its
 * rectified-flow epilogues on one NVIDIA B300 (sm_103a).
 *
 * Sources of the operations (page titles and sections):
 *   [PR 2.2(2)]  PaperReading review of "Mage-Flow: An Efficient Native-Resolution Foundation
 *                Model for Image Generation and Editing", section 2.2 (2): native-resolution
 *                packing by cumulative offsets, attention restricted to each sample, per-sample
 *                2-D RoPE plus a frame index for editing, the flow-matching objective and
 *                z_t = (1 - t) z + t eps, editing loss on the target latent only.
 *   [PR 2.2(3)]  same review, section 2.2 (3): packed CFG; fused norm / RoPE / gating /
 *                residual chains that leave the model function unchanged.
 *   [PR 5]       same review, section 5: MMDiT with per-modality projections and norms and
 *                joint self-attention; rectified-flow ODE sampling; CFG from the difference of
 *                the conditional and unconditional predictions.
 *   [HA M]       hyper.ai summary of the paper, section 方法 (method): packing under a fixed
 *                token budget, the loss, the frame dimension of the rotary embedding.
 *   [HA E]       hyper.ai summary, section 实验 (experiments): packed CFG keeps the denoising
 *                trajectory and raises throughput by 9-15 %.
 *
 * Conventions shared by every call
 *   - Every call returns mf_status.  Nothing aborts and nothing throws across the ABI.
 *     Arguments are validated on the host before any launch; on an error no kernel runs and
 *     no output is touched.
 *   - "device pointer" = memory the caller allocated on the current CUDA device (cudaMalloc,
 *     a PyTorch tensor ...).  The caller owns it and keeps it alive until the stream has
 *     finished the call.  Device pointers must be 16-byte aligned (256-byte aligned for
 *     workspaces); otherwise MF_ERR_ALIGNMENT.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Every
 *     call is asynchronous on that stream unless it says otherwise.
 *   - Matrices are row-major.  Weights are bf16 stored [out_features][in_features]; biases
 *     are bf16 [out_features].  Activations are bf16 [rows][features] unless stated.
 *   - Token layouts of a pack (see mf_pack):
 *       joint order   : sample by sample in pack order, each sample as
 *                       [text tokens | frame 0 image tokens | frame 1 image tokens],
 *                       image tokens row-major over the latent grid;
 *       text stream   : the text tokens of all samples, in pack order (N_txt rows);
 *       image stream  : the image tokens of all samples, in pack order (N_img rows);
 *       stream-sorted : text stream rows followed by image stream rows (N_txt + N_img rows).
 *   - Device faults are never used for error reporting.  Every wait inside a kernel is
 *     bounded; a wait that runs out records MF_ERR_DEVICE_TIMEOUT in a device status word
 *     that mf_check() returns.
 */
#ifndef MAGEFLOW_H
#define MAGEFLOW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MF_OK = 0,
  MF_ERR_INVALID_ARG = 1,      /* null pointer, bad size, bad shape or inconsistent pairing */
  MF_ERR_SAMPLE_TOO_LONG = 2,  /* one sample alone exceeds the token budget */
  MF_ERR_BUDGET = 3,           /* budget < 1 */
  MF_ERR_ALIGNMENT = 4,        /* a device pointer is not aligned as required */
  MF_ERR_CUDA = 5,             /* a CUDA runtime call failed (no device, launch failure ...) */
  MF_ERR_DEVICE_TIMEOUT = 6,   /* a bounded wait inside a kernel ran out (see mf_check) */
  MF_ERR_UNSUPPORTED = 7,      /* dims outside what the kernels implement */
  MF_ERR_NOT_UPLOADED = 8,     /* the plan has no device copy (call mf_plan_upload) */
  MF_ERR_WORKSPACE = 9,        /* workspace smaller than the *_workspace_bytes() figure */
  MF_ERR_DEVICE_BOUNDS = 10    /* checked build only: a kernel met a plan index out of range
                                  (see mf_check) */
} mf_status;

/* Human-readable name of a status; never NULL. */
const char* mf_status_str(mf_status s);

/* ABI version: (major << 16) | minor. */
int32_t mf_version(void);

/* ------------------------------------------------------------------------------------ */
/* Packing  [PR 2.2(2)], [HA M]                                                          */
/* ------------------------------------------------------------------------------------ */

/* One packing candidate.  The sample has txt_len text tokens and `frames` (1 or 2) latent
 * frames of lat_h x lat_w patch tokens; frame 0 of a 2-frame sample is the clean editing
 * source and the last frame is the target.  t is the sample's flow time in [0, 1].
 * cfg_role: 0 plain, 1 conditional branch, 2 unconditional branch; cfg_pair is the index
 * (in the candidate array) of the other branch of the same prompt, -1 for plain samples.
 * Layout: 7 x 4 bytes, little-endian, no padding. */
typedef struct {
  int32_t txt_len;
  int32_t frames;
  int32_t lat_h;
  int32_t lat_w;
  float t;
  int32_t cfg_role;
  int32_t cfg_pair;
} mf_sample;

typedef struct mf_plan mf_plan; /* opaque; owned by the library, freed with mf_plan_free */

/* Packs candidates first-fit in the order given: candidate i is taken iff its length
 * txt_len + frames*lat_h*lat_w still fits the budget left by the candidates taken before it;
 * otherwise it is skipped and packing goes on.  Taken samples keep their relative order.
 * Builds every index buffer the kernels read (cu_seqlens, per-token (frame, row, col)
 * positions, stream/joint row maps, CFG pair table, target-frame flags, the attention work
 * list).  Host only: makes no CUDA call, so it works without a GPU.
 *   samples : host array of n candidates (n >= 0; n == 0 gives an empty plan)
 *   budget  : token budget (>= 1)
 *   out     : receives a new plan; unchanged on error
 * Errors: MF_ERR_BUDGET (budget < 1), MF_ERR_SAMPLE_TOO_LONG (a candidate longer than the
 * budget), MF_ERR_INVALID_ARG (null pointer, n < 0, txt_len < 0, frames not in {1,2},
 * lat_h or lat_w < 1, cfg_role not in {0,1,2}, a packed CFG branch whose partner is not
 * packed or has another image shape). */
mf_status mf_pack(const mf_sample* samples, int32_t n, int32_t budget, mf_plan** out);

/* Copies the plan's index buffers to the current device (library-owned device memory,
 * allocated on the first upload in stream order on `stream`, freed by mf_plan_free).  The copy
 * is enqueued on `stream` and `stream` is synchronised before the call returns (work on other
 * streams is not waited for); a second upload on the same device is a no-op.
 * Errors: MF_ERR_INVALID_ARG, MF_ERR_CUDA. */
mf_status mf_plan_upload(mf_plan* plan, void* stream);

/* Frees host and device memory of the plan without waiting for the device: the device copy
 * is released in stream order on the legacy default stream.  The caller must make sure no
 * work still in flight uses it (synchronise the stream that last used the plan, or wait on an
 * event recorded after that use).  NULL is a no-op. */
void mf_plan_free(mf_plan* plan);

typedef struct {
  int32_t n_seq;      /* S: packed samples */
  int32_t n_tok;      /* N: packed tokens (<= budget) */
  int32_t n_txt;      /* text-stream rows */
  int32_t n_img;      /* image-stream rows */
  int32_t n_items;    /* attention work items (sequence, 256-row query block) */
  int32_t budget;
  int32_t uploaded;   /* 1 after mf_plan_upload */
  int32_t reserved;
} mf_plan_info;

mf_status mf_plan_get_info(const mf_plan* plan, mf_plan_info* info);

/* Host views of the plan's index buffers (int32, owned by the plan, valid until
 * mf_plan_free).  `which`:
 *   0 order[S]        candidate index of each packed sample
 *   1 cu_seqlens[S+1] joint-token offsets
 *   2 cu_txt[S+1]     text-stream row offsets
 *   3 cu_img[S+1]     image-stream row offsets
 *   4 pos[N*3]        (frame, row, col) of each joint token; text tokens (0, 0, 0)
 *   5 txt_seq[N_txt]  6 txt_joint[N_txt]   sample / joint token of each text row
 *   7 img_seq[N_img]  8 img_joint[N_img]   sample / joint token of each image row
 *   9 img_pair[N_img] CFG partner image row, -1 if none
 *  10 img_target[N_img] 1 for target-frame rows, 0 for an edit's source frame
 *  11 seq_role[S]     cfg_role of each packed sample
 *  12 items[n_items*2] attention work list (sequence, 256-row query block), longest sequences
 *                     first
 * Errors: MF_ERR_INVALID_ARG for an unknown `which` or null pointers. */
mf_status mf_plan_array(const mf_plan* plan, int32_t which, const int32_t** data, int64_t* len);

/* ------------------------------------------------------------------------------------ */
/* Model dims and weights                                                                */
/* ------------------------------------------------------------------------------------ */

typedef struct {
  int32_t hidden;     /* H; multiple of 256, at most 4096 */
  int32_t heads;      /* nh; H / nh = head dim D, D in {64, 128} */
  int32_t channels;   /* C: latent channels per patch token; 64 or 128 */
  int32_t mlp_ratio;  /* MLP width = mlp_ratio * H */
  int32_t freq_dim;   /* sinusoidal timestep features; 256 */
} mf_dims;

/* Timestep embedder, shared by every block and the final layer of a stack:
 * c = SiLU(W_t2 SiLU(W_t1 phi(t) + b_t1) + b_t2), phi(t) = [cos a | sin a],
 * a_j = 1000 t 10000^(-j / (F/2)).  W_t1 [H][F], W_t2 [H][H]. */
typedef struct {
  const void* w_t1; const void* b_t1;
  const void* w_t2; const void* b_t2;
} mf_temb_weights;

/* One stream (text or image) of one block [PR 5]: the adaLN modulation (6 chunks of H in
 * the order shift1, scale1, gate1, shift2, scale2, gate2), the fused QKV projection
 * (q | k | v, each H wide), the attention output projection and the MLP.
 * w_qnorm / w_knorm (optional, both or neither; NULL = off): the QK-RMSNorm variant, one
 * scale per head dimension [D]: each head's q (k) vector after the QKV projection becomes
 * q / sqrt(mean_d q_d^2 + 1e-6) * w_qnorm before RoPE.  The pages do not name a QK norm; the
 * plain block has none. */
typedef struct {
  const void* w_mod; const void* b_mod;   /* [6H][H], [6H] */
  const void* w_qkv; const void* b_qkv;   /* [3H][H], [3H] */
  const void* w_o;   const void* b_o;     /* [H][H],  [H]  */
  const void* w_1;   const void* b_1;     /* [rH][H], [rH] */
  const void* w_2;   const void* b_2;     /* [H][rH], [H]  */
  const void* w_qnorm; const void* w_knorm; /* [D], [D] or NULL */
} mf_stream_weights;

typedef struct {
  mf_temb_weights temb;
  mf_stream_weights txt;
  mf_stream_weights img;
} mf_block_weights;

/* ------------------------------------------------------------------------------------ */
/* The block forward  [PR 2.2(2)], [PR 2.2(3)], [PR 5]                                   */
/* ------------------------------------------------------------------------------------ */

/* Workspace the block forward needs for this plan and dims (bytes). */
size_t mf_block_workspace_bytes(const mf_plan* plan, const mf_dims* dims);

/* Byte offsets inside that workspace of the intermediates a call leaves behind, for
 * inspection: [0] c[S][H] f32, [1] mod[S][2][6H] f32 (stream 0 text, 1 image),
 * [2] a[N_txt+N_img][H] bf16 (last LN+modulate output, stream-sorted),
 * [3] q[N][H], [4] k[N][H], [5] v[N][H] bf16 in joint order (q, k after RoPE),
 * [6] o[N_txt+N_img][H] bf16 attention output, stream-sorted,
 * [7] hidden[N_txt+N_img][rH] bf16 (GELU output), stream-sorted,
 * [8] (written when n >= 9) the LN statistics parts of MF_BLOCK_LN_STATS_FUSED:
 *     [N_txt+N_img][H/128] pairs of f32 (mean, sum of squared deviations) of each 128-column
 *     part of the residual after attention.  n must be >= 8. */
mf_status mf_block_workspace_layout(const mf_plan* plan, const mf_dims* dims, size_t* offsets,
                                    int32_t n);

/* One NR-MMDiT block over the whole pack, in place on x:
 *   per sample s and stream m: (shift1, scale1, gate1, shift2, scale2, gate2) = W_mod c_s + b
 *   a  = LN(x) (1 + scale1) + shift1                      (LN without affine, eps 1e-6)
 *   q, k, v = a W_qkv^T + b_qkv, [QK-RMSNorm per head if the stream has its scales],
 *             RoPE on q and k over (frame, row, col)
 *   o  = softmax(q k^T / sqrt(D)) v, jointly over each sample's own tokens only
 *   x += gate1 (o W_o^T + b_o)
 *   x += gate2 (GELU(LN(x)(1 + scale2) + shift2) W_1^T + b_1) W_2^T + b_2)
 * Text rows use w->txt, image rows w->img.
 *   plan    : packed and uploaded plan
 *   d_t     : device f32 [S] flow time per packed sample, or NULL to use the samples' t
 *   d_x_txt : device bf16 [N_txt][H], in/out (may be NULL when N_txt == 0)
 *   d_x_img : device bf16 [N_img][H], in/out
 *   d_ws    : device workspace of mf_block_workspace_bytes() bytes, 256-byte aligned
 * Errors: MF_ERR_INVALID_ARG, MF_ERR_UNSUPPORTED (dims), MF_ERR_NOT_UPLOADED,
 * MF_ERR_WORKSPACE, MF_ERR_ALIGNMENT, MF_ERR_CUDA (launch failure). */
mf_status mf_block_forward(const mf_plan* plan, const mf_dims* dims, const mf_block_weights* w,
                           const float* d_t, void* d_x_txt, void* d_x_img, void* d_ws,
                           size_t ws_bytes, void* stream);

/* Variants of the block's LN + modulate (flags of mf_block_forward_ex).
 *  0 (default)              : one warp per row, statistics from the row held in registers
 *  MF_BLOCK_LN_ROW_GROUPS   : a row-group kernel: groups of 8 rows staged in shared memory by
 *                             bulk copies, each thread keeping its 8 columns' shift and scale in
 *                             registers across the rows of one sample and stream; statistics
 *                             merged per group with Chan's pairwise update
 *  MF_BLOCK_LN_STATS_FUSED  : the statistics of the second LN come from the out-projection's
 *                             epilogue (per 128-column part of each row of the new residual),
 *                             merged by the row-group kernel; bf16 block only, not with the
 *                             training forward  [PR 2.2(3): the norm chain fused into the
 *                             projections]
 * All compute LN(x) = (x - mean) / sqrt(var + 1e-6) with f32 statistics of the bf16 x; they
 * differ only in f32 summation order. */
#define MF_BLOCK_LN_ROW_GROUPS 1
#define MF_BLOCK_LN_STATS_FUSED 2
/* The timestep condition c [S][H] (workspace offset [0], see mf_block_workspace_layout) already
 * holds SiLU(temb(t)) for this plan, these flow times and these timestep weights, as a previous
 * block call with the same workspace left it (the blocks of a stack share the timestep
 * embedder); the timestep MLP is skipped and only the block's own modulation GEMV runs.  A
 * stale c (another plan or other t) gives wrong results, never an out-of-bounds access. */
#define MF_BLOCK_COND_GIVEN 4

/* mf_block_forward with variants: flags a combination of MF_BLOCK_LN_* (with both LN flags, the
 * first LN runs in row groups and the second takes the fused statistics) and
 * MF_BLOCK_COND_GIVEN.  Errors: as
 * mf_block_forward; MF_ERR_INVALID_ARG for unknown flags. */
mf_status mf_block_forward_ex(const mf_plan* plan, const mf_dims* dims, const mf_block_weights* w,
                              const float* d_t, void* d_x_txt, void* d_x_img, void* d_ws,
                              size_t ws_bytes, int32_t flags, void* stream);

/* ------------------------------------------------------------------------------------ */
/* Training: the block forward that keeps what the backward reads, and the block backward  */
/* (the pages' training step, PaperReading review section 3, Table 4, runs both)           */
/* ------------------------------------------------------------------------------------ */

/* Workspace of mf_block_forward_train (bytes): the mf_block_forward workspace (same offsets,
 * see mf_block_workspace_layout; `a` holds the second LN + modulate output) followed by the
 * values the backward reads: the block input and the residual after attention, the first
 * LN + modulate output, the ungated out-projection and MLP outputs, the MLP pre-activation and
 * the attention logsumexp. */
size_t mf_block_train_workspace_bytes(const mf_plan* plan, const mf_dims* dims);

/* mf_block_forward (same arguments, same result in d_x_txt / d_x_img) that also keeps, in d_ws
 * (mf_block_train_workspace_bytes() bytes), everything mf_block_backward needs.  The plain bf16
 * block only: MF_ERR_UNSUPPORTED with QK-RMSNorm scales.  Errors: as mf_block_forward. */
mf_status mf_block_forward_train(const mf_plan* plan, const mf_dims* dims, const mf_block_weights* w,
                                 const float* d_t, void* d_x_txt, void* d_x_img, void* d_ws,
                                 size_t ws_bytes, void* stream);

/* Gradients of one stream's weights, f32 device arrays shaped like the weights
 * (w_mod [6H][H], b_mod [6H], w_qkv [3H][H], b_qkv [3H], w_o [H][H], b_o [H], w_1 [rH][H],
 * b_1 [rH], w_2 [H][rH], b_2 [H]); each is overwritten. */
typedef struct {
  float* w_mod; float* b_mod;
  float* w_qkv; float* b_qkv;
  float* w_o;   float* b_o;
  float* w_1;   float* b_1;
  float* w_2;   float* b_2;
} mf_stream_grads;

typedef struct {
  mf_stream_grads txt;
  mf_stream_grads img;
} mf_block_grads;

size_t mf_block_backward_workspace_bytes(const mf_plan* plan, const mf_dims* dims);

/* Backward of one NR-MMDiT block over the pack (the block of mf_block_forward, differentiated
 * exactly: adaLN modulation, LN, fused QKV, RoPE, per-sample joint attention, gated residuals,
 * GELU MLP; attention gradients never cross samples).  Given G = dL/d(block output):
 *   d_dx_txt, d_dx_img : in: G (bf16, laid out as the forward's x); out: dL/d(block input)
 *   g                  : dL/d(every weight of both streams), f32, overwritten
 *   d_dc               : f32 [S][H], dL/dc_s for each packed sample's condition vector
 *                        c_s = SiLU(temb(t_s)) (the caller sums it over the blocks of a stack)
 *   d_train_ws         : the workspace a mf_block_forward_train call with the same plan,
 *                        dims, weights and t left behind (read only)
 *   d_ws               : mf_block_backward_workspace_bytes() bytes, 256-byte aligned
 * The QK-RMSNorm variant is not differentiated (MF_ERR_UNSUPPORTED).  Reductions over rows use
 * atomic adds, so the last bits of the weight and modulation gradients may change from run to
 * run.  Errors: MF_ERR_INVALID_ARG, MF_ERR_UNSUPPORTED, MF_ERR_NOT_UPLOADED, MF_ERR_ALIGNMENT,
 * MF_ERR_WORKSPACE, MF_ERR_CUDA. */
mf_status mf_block_backward(const mf_plan* plan, const mf_dims* dims, const mf_block_weights* w,
                            const void* d_train_ws, size_t train_ws_bytes, void* d_dx_txt, void* d_dx_img,
                            const mf_block_grads* g, float* d_dc, void* d_ws, size_t ws_bytes,
                            void* stream);

/* fp8 variant of the block (the pages name no fp8 arithmetic; see mf_gemm_fp8): the E4M3
 * codes of one stream's four projection matrices, as mf_quantize_fp8_rows writes them from the
 * bf16 weights (rows = output features), and their per-row scales. */
typedef struct {
  const void* q_qkv; const float* s_qkv;   /* [3H][H] codes, [3H] */
  const void* q_o;   const float* s_o;     /* [H][H],  [H]  */
  const void* q_1;   const float* s_1;     /* [rH][H], [rH] */
  const void* q_2;   const float* s_2;     /* [H][rH], [H]  */
} mf_stream_weights_fp8;

typedef struct {
  mf_stream_weights_fp8 txt;
  mf_stream_weights_fp8 img;
} mf_block_weights_fp8;

/* Workspace of mf_block_forward_fp8: the block workspace (same layout, same offsets) plus the
 * E4M3 codes and row scales of one projection input at a time. */
size_t mf_block_fp8_workspace_bytes(const mf_plan* plan, const mf_dims* dims);

/* mf_block_forward with the four projections on E4M3 operands: each projection input (a, the
 * attention output o, the second a, the GELU output) is quantised per row as
 * mf_quantize_fp8_rows does, right before its GEMM, and multiplied with w8's codes
 * (tcgen05 kind::f8f6f4, f32 accumulation); the row and column scales are applied in the
 * epilogue before the bias, RoPE, GELU or gated residual, which are unchanged.  w supplies
 * everything else (timestep MLP, modulation, biases, optional QK-RMSNorm scales); its bf16
 * projection matrices are not read.  d_ws: mf_block_fp8_workspace_bytes() bytes.
 * Errors: as mf_block_forward. */
mf_status mf_block_forward_fp8(const mf_plan* plan, const mf_dims* dims, const mf_block_weights* w,
                               const mf_block_weights_fp8* w8, const float* d_t, void* d_x_txt,
                               void* d_x_img, void* d_ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------ */
/* Latent embed and final layer (stack ends)  [PR 2.2(2)]                                */
/* ------------------------------------------------------------------------------------ */

/* x_img = z_t W_in^T + b_in: patch latents [N_img][C] (bf16) to hidden [N_img][H] (bf16).
 * W_in [H][C]. Errors: MF_ERR_INVALID_ARG, MF_ERR_UNSUPPORTED, MF_ERR_NOT_UPLOADED,
 * MF_ERR_ALIGNMENT, MF_ERR_CUDA. */
mf_status mf_embed(const mf_plan* plan, const mf_dims* dims, const void* w_in, const void* b_in,
                   const void* d_zt, void* d_x_img, void* stream);

size_t mf_final_workspace_bytes(const mf_plan* plan, const mf_dims* dims);

/* v = (LN(x_img)(1 + scale) + shift) W_out^T + b_out on image rows, with
 * (shift, scale) = W_fmod c_s + b_fmod (2 chunks of H), c_s the sample's timestep
 * condition.  W_fmod [2H][H], W_out [C][H].
 *   d_t : device f32 [S] or NULL (samples' t);  d_x_img : bf16 [N_img][H];
 *   d_v : device f32 [N_img][C] output velocity. */
mf_status mf_final(const mf_plan* plan, const mf_dims* dims, const mf_temb_weights* temb,
                   const void* w_fmod, const void* b_fmod, const void* w_out, const void* b_out,
                   const float* d_t, const void* d_x_img, float* d_v, void* d_ws,
                   size_t ws_bytes, void* stream);

/* mf_final with the timestep condition given: d_c, device f32 [S][H] (16-byte aligned), holds
 * c_s = SiLU(temb(t_s)) of this plan's samples for the same t and timestep weights, as a block
 * call leaves it at offset [0] of its workspace (mf_block_workspace_layout); the timestep MLP is
 * skipped.  d_c NULL behaves as mf_final.  Errors: as mf_final. */
mf_status mf_final_ex(const mf_plan* plan, const mf_dims* dims, const mf_temb_weights* temb,
                      const void* w_fmod, const void* b_fmod, const void* w_out, const void* b_out,
                      const float* d_t, const void* d_x_img, float* d_v, void* d_ws, size_t ws_bytes,
                      const float* d_c, void* stream);

/* ------------------------------------------------------------------------------------ */
/* Rectified-flow epilogues  [PR 2.2(2)], [PR 2.2(3)], [PR 5], [HA M], [HA E]            */
/* ------------------------------------------------------------------------------------ */

/* z_t = (1 - t_s) z + t_s eps on target-frame rows; source-frame rows of an edit sample
 * stay clean (z_t = z).  d_z, d_eps: f32 [N_img][C]; d_t: f32 [S] or NULL (samples' t).
 * Outputs (either may be NULL, not both): d_zt f32 [N_img][C], d_zt_bf16 bf16 [N_img][C]. */
mf_status mf_interpolate(const mf_plan* plan, int32_t channels, const float* d_t, const float* d_z,
                         const float* d_eps, float* d_zt, void* d_zt_bf16, void* stream);

/* Packed CFG [PR 2.2(3)], [PR 5]: for each conditional image row r with unconditional
 * partner u, v_out[r] = v_out[u] = v[u] + w (v[r] - v[u]); rows of plain samples are copied.
 * Both branches receive the guided velocity so that one Euler step keeps them identical.
 * d_v, d_v_out: f32 [N_img][C]; must not overlap unless equal (in place is allowed). */
mf_status mf_cfg_combine(const mf_plan* plan, int32_t channels, float w, const float* d_v,
                         float* d_v_out, void* stream);

/* Euler step of the rectified-flow ODE from t to t - dt (dt > 0 moves towards data):
 * z += dt v, since v ~ z - eps = -dz_t/dt.  d_z f32 [N_img][C] in place; d_v f32 [N_img][C];
 * d_z_bf16: optional bf16 copy of the new z (the next embed's input), may be NULL. */
mf_status mf_euler_step(const mf_plan* plan, int32_t channels, float dt, const float* d_v,
                        float* d_z, void* d_z_bf16, void* stream);

size_t mf_flow_loss_workspace_bytes(const mf_plan* plan);

/* Flow-matching loss [PR 2.2(2)]: per sample s, loss_sum[s] = sum over its target-frame
 * image elements of (v - (z - eps))^2 (f64), count[s] = number of those elements, and
 * mean[0] = sum_s loss_sum[s] / sum_s count[s].  Deterministic (fixed reduction order).
 * d_z, d_eps, d_v: f32 [N_img][C]; outputs are device arrays; d_ws: workspace of
 * mf_flow_loss_workspace_bytes() bytes. */
mf_status mf_flow_loss(const mf_plan* plan, int32_t channels, const float* d_z, const float* d_eps,
                       const float* d_v, double* d_loss_sum, int64_t* d_count, double* d_mean,
                       void* d_ws, size_t ws_bytes, void* stream);

/* Diffusion-NFT post-training objective [PR 2.2(4)]: per sample s with normalised reward
 * r[s] in [0, 1], loss_sum[s] = sum over its target-frame image elements of
 *   r[s] (v_pos - (z - eps))^2 + (1 - r[s]) (v_neg - (z - eps))^2        (f64),
 * count[s] = number of those elements, mean[0] = sum_s loss_sum[s] / sum_s count[s].  The
 * velocity target z - eps is the flow-matching target [PR 2.2(2)]; how the positive and
 * negative policy velocities are formed is left to the caller (the pages do not say).
 * d_z, d_eps, d_v_pos, d_v_neg: f32 [N_img][C]; d_reward: f32 [S] in pack order; outputs are
 * device arrays; d_ws: workspace of mf_flow_loss_workspace_bytes() bytes.  Deterministic.
 * Errors: MF_ERR_INVALID_ARG (null pointers, bad channels), MF_ERR_ALIGNMENT,
 * MF_ERR_WORKSPACE, MF_ERR_NOT_UPLOADED, MF_ERR_CUDA. */
mf_status mf_nft_loss(const mf_plan* plan, int32_t channels, const float* d_z, const float* d_eps,
                      const float* d_v_pos, const float* d_v_neg, const float* d_reward,
                      double* d_loss_sum, int64_t* d_count, double* d_mean, void* d_ws,
                      size_t ws_bytes, void* stream);

/* Image rows the scratch of mf_flow_loss_noalloc holds (8 bytes each, per device). */
#define MF_NOALLOC_MAX_IMG_ROWS 65536

/* mf_flow_loss without a workspace argument, for callers that cannot allocate device memory
 * where they compute the loss (an allocator owned by another framework that forbids side
 * allocations, a fixed pre-reserved memory budget, or a point where an allocation would
 * synchronise the device).  The paper has no counterpart: this is a library convenience.
 * Same inputs, outputs and result as mf_flow_loss; the per-row scratch lives in one
 * library-owned device array per device (MF_NOALLOC_MAX_IMG_ROWS doubles, held until the
 * library is unloaded).  The call allocates nothing.
 *   - The first call on a device looks up that array's device address (with the device
 *     current) and caches it; make that first call before any stream capture.
 *   - All calls on a device share the array: calls that overlap on the GPU (unordered
 *     streams) race; order them on one stream.  Each call writes every scratch row before it
 *     reads it, so nothing left by an earlier call reaches the result.
 * Its launches are counted and traced as MF_K_LOSS, like mf_flow_loss's.
 * Errors: as mf_flow_loss, and MF_ERR_WORKSPACE when the plan has more than
 * MF_NOALLOC_MAX_IMG_ROWS image rows (checked before any launch). */
mf_status mf_flow_loss_noalloc(const mf_plan* plan, int32_t channels, const float* d_z,
                               const float* d_eps, const float* d_v, double* d_loss_sum,
                               int64_t* d_count, double* d_mean, void* stream);

/* ------------------------------------------------------------------------------------ */
/* Building blocks, exposed for testing and reuse                                        */
/* ------------------------------------------------------------------------------------ */

/* Varlen joint attention [PR 2.2(2)]: for every packed sample and head,
 * o = softmax(q k^T / sqrt(D)) v over the sample's own tokens; nothing crosses samples.
 * d_q, d_k, d_v: bf16 [N][H] joint order (heads contiguous inside a row);
 * d_o: bf16 [N_txt + N_img][H] stream-sorted output. */
mf_status mf_attention(const mf_plan* plan, int32_t heads, int32_t head_dim, const void* d_q,
                       const void* d_k, const void* d_v, void* d_o, void* stream);

/* mf_attention that also returns each query row's logsumexp, the input the backward reads:
 * d_lse f32 [heads][N] (joint order inside each head),
 *   lse[h][j] = ln sum_k exp(q_j . k_k / sqrt(D)) over the keys k of j's own sample.
 * Same arguments, layouts and errors as mf_attention otherwise (d_lse 16-byte aligned). */
mf_status mf_attention_lse(const mf_plan* plan, int32_t heads, int32_t head_dim, const void* d_q,
                           const void* d_k, const void* d_v, void* d_o, float* d_lse, void* stream);

/* Workspace of mf_attention_backward: an f32 dq accumulator [N][H], delta [heads][N] f32 and a
 * joint-order copy of do [N][H] bf16 (bytes; 0 for bad arguments). */
size_t mf_attention_backward_workspace_bytes(const mf_plan* plan, int32_t heads, int32_t head_dim);

/* Backward of the varlen joint attention [PR 2.2(2)] (attention restricted to each sample):
 * with s = q k^T / sqrt(D), P = softmax(s) over the sample's own keys, o = P v and the output
 * gradient do, per sample and head
 *   dv = P^T do,  ds = P * (do v^T - rowsum(do * o)),  dq = ds k / sqrt(D),  dk = ds^T q / sqrt(D),
 * nothing crossing samples.  P is recomputed from q, k and the forward's lse
 * (mf_attention_lse), so no L x L matrix is stored.
 *   d_q, d_k, d_v : bf16 [N][H] joint order (the forward's inputs; q, k after RoPE)
 *   d_o, d_do     : bf16 [N_txt + N_img][H] stream-sorted (the forward's output and its gradient)
 *   d_lse         : f32 [heads][N] from mf_attention_lse
 *   d_dq, d_dk, d_dv : bf16 [N][H] joint order, written
 *   d_ws          : mf_attention_backward_workspace_bytes() bytes, 256-byte aligned
 * H = heads * head_dim must be a multiple of 256; head_dim 64 or 128.
 * Errors: MF_ERR_INVALID_ARG, MF_ERR_UNSUPPORTED, MF_ERR_NOT_UPLOADED, MF_ERR_ALIGNMENT,
 * MF_ERR_WORKSPACE, MF_ERR_CUDA. */
mf_status mf_attention_backward(const mf_plan* plan, int32_t heads, int32_t head_dim, const void* d_q,
                                const void* d_k, const void* d_v, const void* d_o, const float* d_lse,
                                const void* d_do, void* d_dq, void* d_dk, void* d_dv, void* d_ws,
                                size_t ws_bytes, void* stream);

/* fp8 variant (a knob of the block's projections; the pages name no fp8 arithmetic).
 * Per-row E4M3 quantisation: for each row r of d_x (bf16 [M][K], K a multiple of 16),
 * d_scale[r] = max_k |x[r][k]| / 448 (1 for an all-zero row) and d_q[r][k] =
 * E4M3(x[r][k] / d_scale[r]) (f32 division, round to nearest even, saturating to +-448;
 * E4M3: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, largest finite value 448).
 * d_q: device uint8 [M][K]; d_scale: device f32 [M].  16-byte aligned pointers.
 * Errors: MF_ERR_INVALID_ARG, MF_ERR_ALIGNMENT, MF_ERR_CUDA. */
mf_status mf_quantize_fp8_rows(int32_t M, int32_t K, const void* d_x, void* d_q, float* d_scale,
                               void* stream);

/* E4M3 GEMM on the tensor cores (tcgen05 kind::f8f6f4, f32 accumulation):
 * C[m][n] = (sum_k A[m][k] B[n][k]) * a_scale[m] * b_scale[n] + bias[n], C bf16 [M][N].
 * d_a: uint8 E4M3 codes [M][K], d_b: [N][K] (both K-major, as mf_quantize_fp8_rows writes
 * them); d_a_scale f32 [M], d_b_scale f32 [N] (16-byte aligned); d_bias bf16 [N] or NULL.
 * K a multiple of 128, N a multiple of 16.  Errors: MF_ERR_INVALID_ARG, MF_ERR_ALIGNMENT,
 * MF_ERR_CUDA. */
mf_status mf_gemm_fp8(int32_t M, int32_t N, int32_t K, const void* d_a, const float* d_a_scale,
                      const void* d_b, const float* d_b_scale, const void* d_bias, void* d_c,
                      void* stream);

/* Plain bf16 GEMM on the tensor cores: C[M][N] = A[M][K] B[N][K]^T (+ bias[N]).
 * out_f32 = 0: C bf16, 1: C f32.  K must be a multiple of 64.  bias may be NULL. */
mf_status mf_gemm(int32_t M, int32_t N, int32_t K, const void* d_a, const void* d_b,
                  const void* d_bias, void* d_c, int32_t out_f32, void* stream);

/* ------------------------------------------------------------------------------------ */
/* Device status                                                                         */
/* ------------------------------------------------------------------------------------ */

/* Synchronises `stream`, then returns and clears the device status word of the current
 * device: MF_OK, or MF_ERR_DEVICE_TIMEOUT if a bounded wait ran out since the last check;
 * MF_ERR_CUDA if the synchronisation itself failed.
 * The checked build (libmageflow_checked.so, compiled with -DMF_CHECKED; same ABI) also
 * checks, inside the kernels, every plan-derived index it reads (sample ids against S, joint
 * and stream-sorted rows against N, cu_seqlens bounds, CFG partner rows, backward row
 * chunks): a failing check skips the access, sets a flag, and mf_check then returns
 * MF_ERR_DEVICE_BOUNDS (before MF_ERR_DEVICE_TIMEOUT).  It never traps.  The default build
 * compiles these checks out. */
mf_status mf_check(void* stream);

/* Self-test of the bounded-wait path: launches one tiny kernel that waits on a barrier no
 * one arrives at, with a limit of limit_us microseconds (1..1000000).  Returns (after a
 * synchronisation) MF_ERR_DEVICE_TIMEOUT when the wait ran out as intended and the context
 * is still usable, MF_OK never.  The status word is cleared again before returning. */
mf_status mf_selftest_timeout(int32_t limit_us, void* stream);

/* ------------------------------------------------------------------------------------ */
/* Per-kernel timing and launch counting                                                 */
/* ------------------------------------------------------------------------------------ */

/* Kinds of kernels the library launches. */
typedef enum {
  MF_K_COND = 0,        /* timestep features and conditioning / modulation GEMVs */
  MF_K_LN = 1,          /* LN + adaLN-modulate prologue */
  MF_K_GEMM_QKV = 2,    /* QKV projection + RoPE + scatter to joint order */
  MF_K_ATTN = 3,        /* varlen joint attention */
  MF_K_GEMM_OPROJ = 4,  /* attention output projection + gated residual */
  MF_K_GEMM_UP = 5,     /* MLP up-projection + GELU */
  MF_K_GEMM_DOWN = 6,   /* MLP down-projection + gated residual */
  MF_K_GEMM_EMBED = 7,  /* latent embed C -> H */
  MF_K_GEMM_FINAL = 8,  /* final layer H -> C */
  MF_K_GEMM_PLAIN = 9,  /* mf_gemm */
  MF_K_LATENT = 10,     /* interpolate, packed CFG, Euler step */
  MF_K_LOSS = 11,       /* flow-matching loss reduction */
  MF_K_FP8 = 12,        /* fp8 variant: row quantisation and the E4M3 GEMM */
  MF_K_ATTN_BWD = 13,   /* attention backward: the tcgen05 kernel */
  MF_K_BLOCK_BWD = 14,  /* backward's memory-bound kernels: gate / LN rows, bias sums, delta and
                           do gather, dq conversion, q / k / v gradient gather, modulation */
  MF_K_GEMM_DGRAD = 15, /* backward input-gradient GEMMs (dY W) */
  MF_K_GEMM_WGRAD = 16, /* backward weight-gradient GEMMs (dY^T X) */
  MF_K_COUNT = 17
} mf_kernel_kind;

typedef struct {
  int64_t launches;  /* kernel launches of this kind since tracing was enabled */
  double ms;         /* summed device time between the events around those launches */
  double flops;      /* summed algorithmic FLOPs (dense contractions: 2 per multiply-add) */
  double bytes;      /* summed algorithmic HBM bytes (memory-bound kinds) */
} mf_trace_entry;

/* on != 0 starts recording (clearing earlier records); on == 0 stops.  While on, every
 * launch of the library outside stream capture is bracketed by two CUDA events recorded on
 * its stream; this costs two event records per launch.  Host-side, not thread-safe with
 * concurrent library calls on other threads. */
mf_status mf_trace_enable(int32_t on);

/* Which kinds are bracketed while tracing is on: bit k of `mask` selects mf_kernel_kind k
 * (all kinds by default).  Launches of other kinds are still counted by mf_launch_count but
 * get no events, so a measured region can time one kernel kind without adding event records
 * around every other launch. */
mf_status mf_trace_kinds(uint32_t mask);

/* Waits for the recorded events, writes one entry per mf_kernel_kind (n >= MF_K_COUNT) and
 * clears the records.  Errors: MF_ERR_INVALID_ARG, MF_ERR_CUDA. */
mf_status mf_trace_read(mf_trace_entry* entries, int32_t n);

/* Number of kernels the library has launched in this process (all kinds, tracing or not). */
int64_t mf_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MAGEFLOW_H */
