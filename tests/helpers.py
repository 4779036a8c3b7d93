"""Shared helpers of the GPU parity tests: pack-order input marshalling, oracle runs over a
pack (one sample at a time), and the comparison statistics."""
from __future__ import annotations

import numpy as np

from oracle import model as M
from oracle import pack as opack

TOL_REL = 2e-2      # max |gpu - ref| <= 2e-2 * max |ref|
TOL_COS = 0.9999    # cosine(gpu, ref) >= 0.9999


def stats(got, ref):
    got = np.asarray(got, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    err = np.abs(got - ref).max() if got.size else 0.0
    scale = np.abs(ref).max() if ref.size else 1.0
    den = np.linalg.norm(got) * np.linalg.norm(ref)
    cos = float(got @ ref / den) if den > 0 else 1.0
    return {"rel": float(err / max(scale, 1e-30)), "cos": cos, "max_abs": float(err),
            "max_ref": float(scale)}


def assert_close(got, ref, name, rel=TOL_REL, cos=TOL_COS):
    s = stats(got, ref)
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{name}: non-finite output"
    assert s["rel"] <= rel and s["cos"] >= cos, f"{name}: {s}"
    return s


def bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (8 significand bits)."""
    a = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def assert_update_close(got, ref, x_in, name, frac=3e-2):
    """Checks a residual update out = x_in + delta stored in bf16: each element may differ
    from the exact result by one bf16 rounding of the output plus `frac` of the largest exact
    update.  (Comparing raw deltas would measure only the output rounding when the update is
    smaller than one bf16 step of the residual.)"""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    delta = ref - np.asarray(x_in, np.float64)
    bound = bf16_ulp(ref) + frac * np.abs(delta).max()
    err = np.abs(got - ref)
    worst = float((err / bound).max()) if err.size else 0.0
    assert worst <= 1.0, f"{name}: worst error / bound = {worst:.3f}, stats {stats(got - x_in, delta)}"
    return stats(got - np.asarray(x_in, np.float64), delta)


def stream_concat(parts, order, width):
    arrs = [parts[c] for c in order]
    if not arrs:
        return np.zeros((0, width), np.float32)
    return np.concatenate(arrs, axis=0).astype(np.float32) if sum(len(a) for a in arrs) else \
        np.zeros((0, width), np.float32)


def split_rows(x, cu, k):
    return x[cu[k]:cu[k + 1]]


def oracle_stack(samples, plan: opack.Plan, weights, batch, heads, zt=None, t=None, n_blocks=None,
                 x_img_in=None):
    """Per-sample oracle of embed -> blocks -> final over a pack.
    zt: stream-ordered [N_img][C] model input (default: batch z).  x_img_in: if given, the
    stream-ordered hidden image input (skips the embed).  Returns (x_txt, x_img, v) in stream
    order."""
    xs_t, xs_i, vs = [], [], []
    blocks = weights.blocks[:n_blocks]
    for k, c in enumerate(plan.order):
        s = samples[c]
        tt = s.t if t is None else t[k]
        cond = M.condition(tt, weights.temb, weights.dims.freq_dim)
        pos = M.image_positions(s.frames, s.lat_h, s.lat_w)
        xt = M.f64(batch.x_txt[c])
        if x_img_in is not None:
            xi = M.f64(split_rows(x_img_in, plan.cu_img, k))
        else:
            z = batch.z[c] if zt is None else split_rows(zt, plan.cu_img, k)
            xi = M.embed(z, weights.embed)
        for bw in blocks:
            xt, xi = M.block_forward(xt, xi, pos, cond, bw, heads)
        vs.append(M.final_layer(xi, cond, weights.final))
        xs_t.append(xt)
        xs_i.append(xi)
    cat = lambda a, w: np.concatenate(a) if a else np.zeros((0, w))     # noqa: E731
    H = weights.dims.hidden
    return cat(xs_t, H), cat(xs_i, H), cat(vs, weights.dims.channels)
