"""Pins for the gradient oracle of the block backward (oracle/grad.py): its float64 PyTorch
restatement of the forward equals the NumPy oracle, and its gradients agree with central
finite differences of that forward along random directions, for the block inputs, the
condition and the weights of both streams."""
import numpy as np
import pytest

import synth
from oracle import model as M

torch = pytest.importorskip("torch")
from oracle import grad as G  # noqa: E402

D = synth.Dims(hidden=64, heads=2, channels=16)          # head dim 32: RoPE blocks (4, 14, 14)


def _case(seed=0, Lt=3, h=2, wd=3):
    w = synth.model_weights(D, 1, seed, std=0.1, bf16=False)
    rng = np.random.default_rng(seed)
    xt = rng.standard_normal((Lt, D.hidden))
    xi = rng.standard_normal((h * wd, D.hidden))
    pos = M.image_positions(1, h, wd)
    c = rng.standard_normal(D.hidden)
    return w.blocks[0], xt, xi, pos, c, rng


def test_restated_forward_equals_the_oracle():
    bw, xt, xi, pos, c, _ = _case()
    ref = M.block_forward(xt, xi, pos, c, bw, D.heads)
    w = {s: {n: G._t(bw[s][n]) for n in G.WEIGHT_NAMES} for s in M.STREAMS}
    got = G.block_forward_t(G._t(xt), G._t(xi), pos, G._t(c), w, D.heads)
    for r, g in zip(ref, got):
        np.testing.assert_allclose(g.numpy(), r, rtol=0, atol=1e-12)


def _objective(bw, xt, xi, pos, c, gt, gi):
    ot, oi = M.block_forward(xt, xi, pos, c, bw, D.heads)
    return float((ot * gt).sum() + (oi * gi).sum())


@pytest.mark.parametrize("seed", [0, 1])
def test_gradients_match_finite_differences(seed):
    bw, xt, xi, pos, c, rng = _case(seed)
    gt = rng.standard_normal(xt.shape)
    gi = rng.standard_normal(xi.shape)
    grads = G.block_vjp(xt, xi, pos, c, bw, D.heads, gt, gi)
    eps = 1e-5
    # inputs and condition
    for name, base in (("x_txt", xt), ("x_img", xi), ("c", c)):
        u = rng.standard_normal(base.shape)
        args = {"x_txt": xt, "x_img": xi, "c": c}
        plus, minus = dict(args), dict(args)
        plus[name], minus[name] = base + eps * u, base - eps * u
        fd = (_objective(bw, plus["x_txt"], plus["x_img"], pos, plus["c"], gt, gi) -
              _objective(bw, minus["x_txt"], minus["x_img"], pos, minus["c"], gt, gi)) / (2 * eps)
        an = float((grads[name] * u).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)
    # every weight of both streams
    for s in M.STREAMS:
        for n in G.WEIGHT_NAMES:
            u = rng.standard_normal(bw[s][n].shape)
            bp = {st: dict(bw[st]) for st in M.STREAMS}
            bm = {st: dict(bw[st]) for st in M.STREAMS}
            bp[s][n] = bw[s][n] + eps * u
            bm[s][n] = bw[s][n] - eps * u
            fd = (_objective(bp, xt, xi, pos, c, gt, gi) - _objective(bm, xt, xi, pos, c, gt, gi)) / (2 * eps)
            an = float((grads[s][n] * u).sum())
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (s, n, fd, an)


def test_gradient_special_cases():
    """Zero gates: the block is the identity, so dL/dx = g and no projection weight after the
    gates receives gradient; a sample without text tokens has no text-stream gradient."""
    bw, xt, xi, pos, c, rng = _case(3)
    for s in M.STREAMS:
        bw[s] = dict(bw[s])
        b = bw[s]["b_mod"].copy()
        wm = bw[s]["w_mod"].copy()
        H = D.hidden
        for chunk in (2, 5):                                    # gate1, gate2
            b[chunk * H:(chunk + 1) * H] = 0.0
            wm[chunk * H:(chunk + 1) * H] = 0.0
        bw[s]["b_mod"], bw[s]["w_mod"] = b, wm
    gt, gi = rng.standard_normal(xt.shape), rng.standard_normal(xi.shape)
    g = G.block_vjp(xt, xi, pos, c, bw, D.heads, gt, gi)
    np.testing.assert_allclose(g["x_txt"], gt, rtol=0, atol=1e-12)
    np.testing.assert_allclose(g["x_img"], gi, rtol=0, atol=1e-12)
    for s in M.STREAMS:
        for n in ("w_qkv", "w_o", "w_1", "w_2"):
            np.testing.assert_array_equal(g[s][n], 0.0)
    bw2, _, xi2, pos2, c2, rng2 = _case(4, Lt=0)
    g2 = G.block_vjp(np.zeros((0, D.hidden)), xi2, pos2, c2, bw2, D.heads, np.zeros((0, D.hidden)),
                     rng2.standard_normal(xi2.shape))
    for n in ("w_qkv", "w_o", "w_1", "w_2", "b_qkv", "b_o", "b_1", "b_2"):
        np.testing.assert_array_equal(g2["txt"][n], 0.0)


def test_attention_vjp_closed_form():
    """The attention gradients against the textbook closed form written out in NumPy:
    P = softmax(q k^T / sqrt(D)), dV = P^T dO, dP = dO V^T, dS = P * (dP - rowsum(dP * P)),
    dQ = dS K / sqrt(D), dK = dS^T Q / sqrt(D), per head."""
    rng = np.random.default_rng(11)
    L, nh, Dh = 7, 2, 8
    q, k, v, do = (rng.standard_normal((L, nh, Dh)) for _ in range(4))
    dq, dk, dv = G.attention_vjp(q, k, v, do)
    for h in range(nh):
        s = q[:, h] @ k[:, h].T / np.sqrt(Dh)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        dvh = p.T @ do[:, h]
        dp = do[:, h] @ v[:, h].T
        ds = p * (dp - (dp * p).sum(axis=1, keepdims=True))
        np.testing.assert_allclose(dv[:, h], dvh, rtol=0, atol=1e-12)
        np.testing.assert_allclose(dq[:, h], ds @ k[:, h] / np.sqrt(Dh), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dk[:, h], ds.T @ q[:, h] / np.sqrt(Dh), rtol=0, atol=1e-12)


def test_attention_lse_and_row_gradients():
    """attention_lse normalises the softmax (exp(s - lse) sums to 1 over the keys, and equals
    the softmax the forward oracle uses), and the selected-row gradients equal the
    reverse-mode gradients on every row asked for."""
    rng = np.random.default_rng(12)
    L, nh, Dh = 9, 3, 16
    q, k, v, do = (rng.standard_normal((L, nh, Dh)) for _ in range(4))
    lse = G.attention_lse(q, k)
    s = np.einsum("qhd,khd->hqk", q, k) / np.sqrt(Dh)
    p = np.exp(s - lse[:, :, None])
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(np.einsum("hqk,khd->qhd", p, v), M.attention(q, k, v), rtol=0, atol=1e-12)
    dq, dk, dv = G.attention_vjp(q, k, v, do)
    rows_q, rows_k = np.array([0, 4, 8]), np.array([1, 2, 7])
    gq, gk, gv = G.attention_vjp_rows(q, k, v, do, rows_q, rows_k)
    np.testing.assert_allclose(gq, dq[rows_q], rtol=0, atol=1e-12)
    np.testing.assert_allclose(gk, dk[rows_k], rtol=0, atol=1e-12)
    np.testing.assert_allclose(gv, dv[rows_k], rtol=0, atol=1e-12)
