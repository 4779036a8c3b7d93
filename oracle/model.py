"""Oracle for one NR-MMDiT block, the timestep conditioning, the latent embed / final layer
and the rectified-flow epilogues.  float64 NumPy, one sample at a time.

Sources (page titles and sections):
* [PR 2.2(2)] PaperReading review of "Mage-Flow: An Efficient Native-Resolution Foundation
  Model for Image Generation and Editing", §2.2 (2): the flow-matching objective
  L = E || v_theta(z_t, t, tau) - (z - eps) ||^2 with z_t = (1 - t) z + t eps,
  eps ~ N(0, I); 16x-downsampled 128-channel latents flattened to variable-length tokens;
  packing by cumulative offsets with attention only inside each sample; a 2-D RoPE per
  sample, extended by a frame index f to (f, h, w) for editing; editing loss on the target
  latent only.
* [PR 2.2(3)] same review, §2.2 (3): packed CFG (cond and uncond in one packed forward,
  trajectory unchanged); norm, RoPE, gating and residual chains fused without changing the
  model function.
* [PR 5] same review, §5 concepts: MMDiT = separate projections and norms per modality with
  joint self-attention; rectified flow samples along the learned ODE from noise to data;
  CFG uses the difference of the conditional and unconditional predictions.
* [PR 2.2(4)] same review, §2.2 (4): the Diffusion-NFT post-training objective
  E[ r ||v+ - v||^2 + (1 - r) ||v- - v||^2 ] with a group-normalised reward r in [0, 1].
* [HA 方法] hyper.ai summary, 方法 (method): the same loss and interpolation; a frame dimension
  added to the 2-D rotary embedding for editing.

Readings where the pages are silent (each is a named constant below):
* block internals follow the SD3-style MMDiT the review names as its lineage: adaLN
  modulation (shift, scale, gate for attention and for the MLP) from SiLU(temb), pre-LN
  without affine (eps 1e-6), gated residuals, MLP 4x with exact-erf GELU, no QK-norm;
* timestep embedding: 256 sinusoidal features of 1000*t, [cos | sin] order, max period 1e4,
  then Linear -> SiLU -> Linear;
* RoPE: head dim split (D/8, 7D/16, 7D/16) over (frame, row, col), base 1e4, adjacent pairs
  (2j, 2j+1); text tokens at (0, 0, 0), rows and columns counted from 0;
* final layer: adaLN-modulated LN + Linear H -> C on image tokens; latent embed Linear C -> H;
* edit: every token of a sample shares t; the source frame stays clean;
* Euler: v ~ z - eps = -dz_t/dt, so stepping t_k -> t_{k+1} < t_k is z += (t_k - t_{k+1}) v;
* loss: per-sample sums over target-frame image elements, and the element-weighted mean.
* QK-RMSNorm (a variant, off unless a stream's weights carry w_qnorm / w_knorm): each head's
  query and key vector after the QKV projection is divided by its root mean square over the
  head dimension (eps 1e-6) and multiplied by a learned per-dimension scale of that stream,
  before RoPE.
"""
from __future__ import annotations

import numpy as np
from scipy.special import erf

LN_EPS = 1e-6
RMS_EPS = 1e-6
ROPE_BASE = 10000.0
T_SCALE = 1000.0
MAX_PERIOD = 10000.0
STREAMS = ("txt", "img")
MOD_CHUNKS = ("shift1", "scale1", "gate1", "shift2", "scale2", "gate2")


def f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# ------------------------------------------------------------------ elementary pieces
def linear(x, w, b):
    """x @ w^T + b with w stored [out][in]."""
    return f64(x) @ f64(w).T + f64(b)


def silu(x):
    x = f64(x)
    return x / (1.0 + np.exp(-x))


def gelu(x):
    """Exact GELU, 0.5 x (1 + erf(x / sqrt 2))."""
    x = f64(x)
    return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))


def layer_norm(x, eps: float = LN_EPS):
    """LayerNorm over the last axis without affine parameters (biased variance)."""
    x = f64(x)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def rms_norm_heads(x, g, eps: float = RMS_EPS):
    """x [L][heads][D] -> x / sqrt(mean over D of x^2 + eps) * g, g [D] (one scale per head
    dimension, shared by the heads)."""
    x = f64(x)
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps) * f64(g)


def modulate(x, shift, scale):
    return layer_norm(x) * (1.0 + f64(scale)) + f64(shift)


def timestep_embedding(t, dim: int = 256):
    """Sinusoidal features of T_SCALE * t: [cos(a_0..a_{h-1}) | sin(a_0..a_{h-1})],
    a_j = T_SCALE * t * MAX_PERIOD^(-j / h), h = dim / 2."""
    half = dim // 2
    freqs = np.exp(-np.log(MAX_PERIOD) * np.arange(half, dtype=np.float64) / half)
    args = T_SCALE * f64(t)[..., None] * freqs
    return np.concatenate([np.cos(args), np.sin(args)], axis=-1)


def condition(t, temb_w: dict, freq_dim: int = 256):
    """c = SiLU(temb(t)): the input of every adaLN modulation linear of the stack."""
    h = silu(linear(timestep_embedding(t, freq_dim), temb_w["w_t1"], temb_w["b_t1"]))
    return silu(linear(h, temb_w["w_t2"], temb_w["b_t2"]))


def modulation(c, w, b, n: int):
    return np.split(linear(c, w, b), n, axis=-1)


# ------------------------------------------------------------------ rotary positions
def rope_axis_widths(head_dim: int):
    """Widths of the (frame, row, col) blocks of one head: (D/8, 7D/16, 7D/16)."""
    return (head_dim // 8, 7 * head_dim // 16, 7 * head_dim // 16)


def rope_angles(pos, head_dim: int):
    """theta[L][D/2]: pair g of the head, inside axis block a of width d at local pair j,
    turns by pos[a] * ROPE_BASE^(-2 j / d)."""
    pos = np.asarray(pos)
    cols = []
    for a, d in enumerate(rope_axis_widths(head_dim)):
        j = np.arange(d // 2, dtype=np.float64)
        inv = ROPE_BASE ** (-2.0 * j / d)
        cols.append(pos[:, a:a + 1].astype(np.float64) * inv[None, :])
    return np.concatenate(cols, axis=1)


def apply_rope(x, pos):
    """Rotate adjacent pairs (2g, 2g+1) of every head of x [L][nh][D] by theta[L][g]."""
    x = f64(x)
    th = rope_angles(pos, x.shape[-1])[:, None, :]
    c, s = np.cos(th), np.sin(th)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def image_positions(frames: int, h: int, w: int):
    """(frame, row, col) of a sample's image tokens, frame-major then row-major."""
    f, r, c = np.meshgrid(np.arange(frames), np.arange(h), np.arange(w), indexing="ij")
    return np.stack([f.ravel(), r.ravel(), c.ravel()], axis=1).astype(np.int64)


# ------------------------------------------------------------------ attention
def attention(q, k, v, rows=None):
    """softmax(q k^T / sqrt(D)) v per head over ONE sample's tokens.  q, k, v: [L][nh][D].
    `rows` restricts the queries (the keys/values are always the whole sample)."""
    q, k, v = f64(q), f64(k), f64(v)
    if rows is not None:
        q = q[rows]
    s = np.einsum("qhd,khd->hqk", q, k) / np.sqrt(q.shape[-1])
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=-1, keepdims=True)
    return np.einsum("hqk,khd->qhd", p, v)


# ------------------------------------------------------------------ the block
def _proj(x, bw_s: dict, w8_s, name: str):
    """x W^T + b of one stream's projection `name` (qkv, o, 1, 2); with w8_s (the fp8
    variant's codes and scales of that stream) on E4M3 operands, as oracle.fp8 defines them."""
    if w8_s is None:
        return linear(x, bw_s["w_" + name], bw_s["b_" + name])
    from oracle import fp8
    return fp8.linear_fp8_act(x, w8_s, name, bw_s["b_" + name])


def block_forward(x_txt, x_img, pos_img, c, bw: dict, heads: int, rows=None, w8=None):
    """One NR-MMDiT block over ONE sample.

    x_txt [Lt][H], x_img [Li][H]: the sample's text and image tokens; pos_img [Li][3];
    c [H]: SiLU(temb) of the sample; bw[stream][name]: the stream's weights.
    Text rows use the text weights and image rows the image weights; attention is joint over
    [text | image] in that order.  `rows` (joint indices) selects which output rows to
    compute; the keys and values always cover the whole sample.  `w8` ({stream: codes and
    scales}) selects the fp8 variant of the four projections.
    Returns (x_txt_out, x_img_out), or the selected joint rows [len(rows)][H] if `rows`.
    """
    w8 = w8 or {s: None for s in STREAMS}
    x = {"txt": f64(x_txt), "img": f64(x_img)}
    Lt, Li = len(x["txt"]), len(x["img"])
    H = (x["txt"] if Lt else x["img"]).shape[1]
    D = H // heads
    L = Lt + Li
    mod = {s: dict(zip(MOD_CHUNKS, modulation(c, bw[s]["w_mod"], bw[s]["b_mod"], 6)))
           for s in STREAMS}
    a = {s: modulate(x[s], mod[s]["shift1"], mod[s]["scale1"]) for s in STREAMS}
    qkv = np.concatenate([_proj(a[s], bw[s], w8[s], "qkv") for s in STREAMS])
    q, k, v = (qkv[:, i * H:(i + 1) * H].reshape(L, heads, D) for i in range(3))
    if any("w_qnorm" in bw[s] for s in STREAMS):
        # QK-RMSNorm variant: each stream's rows with that stream's scales (text rows first)
        q, k = q.copy(), k.copy()
        for s, seg in (("txt", slice(0, Lt)), ("img", slice(Lt, L))):
            q[seg] = rms_norm_heads(q[seg], bw[s]["w_qnorm"])
            k[seg] = rms_norm_heads(k[seg], bw[s]["w_knorm"])
    pos = np.concatenate([np.zeros((Lt, 3), np.int64), np.asarray(pos_img, np.int64)])
    sel = np.arange(L) if rows is None else np.asarray(rows)
    q = apply_rope(q[sel], pos[sel])
    k = apply_rope(k, pos)
    o = attention(q, k, v).reshape(len(sel), H)
    out = np.empty((len(sel), H))
    for s in STREAMS:
        m = (sel < Lt) if s == "txt" else (sel >= Lt)
        if not m.any():
            continue
        xs = x["txt"][sel[m]] if s == "txt" else x["img"][sel[m] - Lt]
        w = bw[s]
        xs = xs + mod[s]["gate1"] * _proj(o[m], w, w8[s], "o")
        h = gelu(_proj(modulate(xs, mod[s]["shift2"], mod[s]["scale2"]), w, w8[s], "1"))
        out[m] = xs + mod[s]["gate2"] * _proj(h, w, w8[s], "2")
    if rows is not None:
        return out
    return out[:Lt], out[Lt:]


def embed(z_t, ew: dict):
    """Latent tokens [Li][C] -> hidden [Li][H]."""
    return linear(z_t, ew["w_in"], ew["b_in"])


def final_layer(x_img, c, fw: dict):
    """adaLN-modulated LN, then Linear H -> C: the velocity v_theta on image tokens."""
    shift, scale = modulation(c, fw["w_fmod"], fw["b_fmod"], 2)
    return linear(modulate(x_img, shift, scale), fw["w_out"], fw["b_out"])


def forward(x_txt, z_t, sample, t, weights, heads: int):
    """embed -> every block -> final layer for ONE sample; returns v [Li][C]."""
    c = condition(t, weights.temb, weights.dims.freq_dim)
    pos = image_positions(sample.frames, sample.lat_h, sample.lat_w)
    xt, xi = f64(x_txt), embed(z_t, weights.embed)
    for bw in weights.blocks:
        xt, xi = block_forward(xt, xi, pos, c, bw, heads)
    return final_layer(xi, c, weights.final)


# ------------------------------------------------------------------ rectified-flow epilogues
def target_mask(sample):
    """1 for image tokens of the target frame (the last frame), 0 for an edit's source frame."""
    m = np.zeros(sample.frames * sample.lat_h * sample.lat_w, dtype=bool)
    m[(sample.frames - 1) * sample.lat_h * sample.lat_w:] = True
    return m


def interpolate(z, eps, t, target=None):
    """z_t = (1 - t) z + t eps on target rows; source rows stay clean (z)."""
    z, eps = f64(z), f64(eps)
    zt = (1.0 - t) * z + t * eps
    if target is not None:
        zt[~target] = z[~target]
    return zt


def flow_loss(v, z, eps, target=None):
    """(sum over target elements of (v - (z - eps))^2, element count) for one sample."""
    d = f64(v) - (f64(z) - f64(eps))
    if target is not None:
        d = d[target]
    return float((d * d).sum()), int(d.size)


def nft_loss(v_pos, v_neg, z, eps, r, target=None):
    """Diffusion-NFT objective of one sample [PR 2.2(4)]: (sum over its target elements of
    r (v_pos - v*)^2 + (1 - r) (v_neg - v*)^2, element count), where v* = z - eps is the
    flow-matching velocity target of [PR 2.2(2)] and r in [0, 1] is the sample's
    group-normalised reward.  The pages do not say how the positive and negative policy
    velocities v_pos, v_neg are formed; they are inputs here."""
    v_star = f64(z) - f64(eps)
    dp = f64(v_pos) - v_star
    dn = f64(v_neg) - v_star
    if target is not None:
        dp, dn = dp[target], dn[target]
    return float(r * (dp * dp).sum() + (1.0 - r) * (dn * dn).sum()), int(dp.size)


def mean_loss(sums, counts):
    return float(np.sum(sums) / np.sum(counts))


def euler_step(z, v, dt):
    """z_{t - dt} = z_t + dt * v for a step from t down to t - dt (dt > 0)."""
    return f64(z) + dt * f64(v)


def cfg_combine(v_cond, v_uncond, w):
    return f64(v_uncond) + w * (f64(v_cond) - f64(v_uncond))


def sample_cfg(x_txt_cond, z0, sample_cond, sample_uncond, weights, heads: int, w: float,
               t_grid):
    """Euler sampler with CFG for one prompt: cond and uncond forwards run separately (the
    unpacked definition); returns the final latent."""
    z = f64(z0)
    empty = np.zeros((0, weights.dims.hidden))
    for k in range(len(t_grid) - 1):
        t = t_grid[k]
        vc = forward(x_txt_cond, z, sample_cond, t, weights, heads)
        vu = forward(empty, z, sample_uncond, t, weights, heads)
        z = euler_step(z, cfg_combine(vc, vu, w), t_grid[k] - t_grid[k + 1])
    return z
