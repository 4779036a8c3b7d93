"""Gradient oracle for the block backward (test infrastructure only; nothing on the product
path imports it).

The block forward is restated with plain PyTorch CPU operations in float64, step for step as
oracle.model.block_forward writes it (adaLN modulation, LN without affine, fused QKV per
stream, RoPE over (frame, row, col), joint softmax attention over the sample, gated
residuals, exact-erf GELU MLP), and PyTorch's reverse-mode differentiation of that restatement
gives the vector-Jacobian products the backward must reproduce: the gradients with respect to
the block input rows and every weight of both streams for a given output cotangent.

Pins (tests/test_oracle_grad.py): the restated forward equals oracle.model.block_forward, and
the gradients agree with central finite differences of the float64 forward along random
directions.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import model as M

F64 = torch.float64
WEIGHT_NAMES = ("w_mod", "b_mod", "w_qkv", "b_qkv", "w_o", "b_o", "w_1", "b_1", "w_2", "b_2")


def _t(a):
    return torch.as_tensor(np.asarray(a, dtype=np.float64), dtype=F64)


def _layer_norm(x):
    mu = x.mean(dim=-1, keepdim=True)
    var = ((x - mu) ** 2).mean(dim=-1, keepdim=True)
    return (x - mu) / torch.sqrt(var + M.LN_EPS)


def _modulate(x, shift, scale):
    return _layer_norm(x) * (1.0 + scale) + shift


def _gelu(x):
    return 0.5 * x * (1.0 + torch.erf(x / np.sqrt(2.0)))


def _rope(x, pos):
    """x [L][nh][D]; the angles come from the oracle (positions are not differentiated)."""
    th = _t(M.rope_angles(pos, x.shape[-1]))[:, None, :]
    c, s = torch.cos(th), torch.sin(th)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    return torch.stack([x0 * c - x1 * s, x0 * s + x1 * c], dim=-1).reshape(x.shape)


def block_forward_t(x_txt, x_img, pos_img, c, w: dict, heads: int):
    """The block over ONE sample with torch tensors (x_txt [Lt][H], x_img [Li][H], c [H];
    w[stream][name] tensors).  Returns (x_txt_out, x_img_out)."""
    Lt, Li = x_txt.shape[0], x_img.shape[0]
    H = x_txt.shape[1] if Lt else x_img.shape[1]
    D = H // heads
    L = Lt + Li
    x = {"txt": x_txt, "img": x_img}
    mod = {}
    for s in M.STREAMS:
        m = c @ w[s]["w_mod"].T + w[s]["b_mod"]
        mod[s] = dict(zip(M.MOD_CHUNKS, torch.split(m, H, dim=-1)))
    a = {s: _modulate(x[s], mod[s]["shift1"], mod[s]["scale1"]) for s in M.STREAMS}
    qkv = torch.cat([a[s] @ w[s]["w_qkv"].T + w[s]["b_qkv"] for s in M.STREAMS])
    q, k, v = (qkv[:, i * H:(i + 1) * H].reshape(L, heads, D) for i in range(3))
    pos = np.concatenate([np.zeros((Lt, 3), np.int64), np.asarray(pos_img, np.int64)])
    q, k = _rope(q, pos), _rope(k, pos)
    sc = torch.einsum("qhd,khd->hqk", q, k) / np.sqrt(D)
    p = torch.softmax(sc, dim=-1)
    o = torch.einsum("hqk,khd->qhd", p, v).reshape(L, H)
    out = []
    for s, seg in (("txt", slice(0, Lt)), ("img", slice(Lt, L))):
        ws = w[s]
        xs = x[s] + mod[s]["gate1"] * (o[seg] @ ws["w_o"].T + ws["b_o"])
        h = _gelu(_modulate(xs, mod[s]["shift2"], mod[s]["scale2"]) @ ws["w_1"].T + ws["b_1"])
        out.append(xs + mod[s]["gate2"] * (h @ ws["w_2"].T + ws["b_2"]))
    return out[0], out[1]


def block_vjp(x_txt, x_img, pos_img, c, bw: dict, heads: int, g_txt, g_img):
    """Gradients of sum(g_txt * out_txt) + sum(g_img * out_img) with respect to the block
    inputs and weights, float64 NumPy: {"x_txt", "x_img", "c", stream: {name: grad}}."""
    xt = _t(x_txt).requires_grad_(True)
    xi = _t(x_img).requires_grad_(True)
    ct = _t(c).requires_grad_(True)
    w = {s: {n: _t(bw[s][n]).requires_grad_(True) for n in WEIGHT_NAMES} for s in M.STREAMS}
    ot, oi = block_forward_t(xt, xi, pos_img, ct, w, heads)
    loss = (ot * _t(g_txt)).sum() + (oi * _t(g_img)).sum()
    leaves = [xt, xi, ct] + [w[s][n] for s in M.STREAMS for n in WEIGHT_NAMES]
    grads = torch.autograd.grad(loss, leaves, allow_unused=True)

    def np_(g, like):
        return np.zeros(like.shape) if g is None else g.detach().numpy()

    out = {"x_txt": np_(grads[0], xt), "x_img": np_(grads[1], xi), "c": np_(grads[2], ct)}
    i = 3
    for s in M.STREAMS:
        out[s] = {}
        for n in WEIGHT_NAMES:
            out[s][n] = np_(grads[i], w[s][n])
            i += 1
    return out


def attention_vjp(q, k, v, do):
    """Gradients (dq, dk, dv) of sum(do * attention(q, k, v)) for ONE sample, q, k, v, do
    [L][nh][D] float64 (reverse-mode differentiation of the restated softmax attention)."""
    qt, kt, vt = (_t(a).requires_grad_(True) for a in (q, k, v))
    D = qt.shape[-1]
    p = torch.softmax(torch.einsum("qhd,khd->hqk", qt, kt) / np.sqrt(D), dim=-1)
    o = torch.einsum("hqk,khd->qhd", p, vt)
    g = torch.autograd.grad((o * _t(do)).sum(), [qt, kt, vt])
    return tuple(x.detach().numpy() for x in g)


def attention_lse(q, k):
    """Per head and query row of ONE sample, the natural-log logsumexp of the scaled scores,
    lse[h][j] = ln sum_k exp(q_j . k_k / sqrt(D)), float64 [nh][L] (the normaliser that the
    backward uses to recompute P = exp(s - lse))."""
    from scipy.special import logsumexp
    q, k = np.asarray(q, np.float64), np.asarray(k, np.float64)
    s = np.einsum("qhd,khd->hqk", q, k) / np.sqrt(q.shape[-1])
    return logsumexp(s, axis=-1)


def attention_vjp_rows(q, k, v, do, q_rows, k_rows):
    """The attention gradients of ONE sample for selected rows, by the closed form of the
    softmax backward (per head, s = q k^T / sqrt(D), P = softmax(s), o = P v,
    delta = rowsum(do * o), dS = P * (do v^T - delta)):
      dq[j] = sum_k dS[j, k] k_k / sqrt(D)        for the query rows j in q_rows,
      dk[k] = sum_j dS[j, k] q_j / sqrt(D),  dv[k] = sum_j P[j, k] do_j   for k in k_rows.
    q, k, v, do: [L][nh][D].  Returns (dq [len(q_rows)][nh][D], dk, dv [len(k_rows)][nh][D]).
    Only the rows asked for are formed beyond the full P, so long samples stay affordable."""
    q, k, v, do = (np.asarray(a, np.float64) for a in (q, k, v, do))
    q_rows, k_rows = np.asarray(q_rows), np.asarray(k_rows)
    L, nh, D = q.shape
    dq = np.zeros((len(q_rows), nh, D))
    dk = np.zeros((len(k_rows), nh, D))
    dv = np.zeros((len(k_rows), nh, D))
    for h in range(nh):
        s = q[:, h] @ k[:, h].T / np.sqrt(D)
        s -= s.max(axis=1, keepdims=True)
        np.exp(s, out=s)
        s /= s.sum(axis=1, keepdims=True)               # s is P from here on
        delta = (do[:, h] * (s @ v[:, h])).sum(axis=1)
        ds_r = s[q_rows] * (do[q_rows, h] @ v[:, h].T - delta[q_rows, None])
        dq[:, h] = ds_r @ k[:, h] / np.sqrt(D)
        p_c = s[:, k_rows]
        dv[:, h] = p_c.T @ do[:, h]
        ds_c = p_c * (do[:, h] @ v[k_rows, h].T - delta[:, None])
        dk[:, h] = ds_c.T @ q[:, h] / np.sqrt(D)
        del s
    return dq, dk, dv
