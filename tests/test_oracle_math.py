"""Pins for the oracle's arithmetic: closed forms, invariants the pages state, brute force on
tiny inputs and hand-worked values (tests/golden).  A planted mistake in any of these pieces
(a dropped term, a wrong sign or index, a transposed operand) fails at least one test here;
`test_planted_mistakes` checks that for a list of plausible mistakes."""
import copy

import numpy as np
import pytest

import synth
from oracle import brute
from oracle import model as M

R = np.random.default_rng(1234)


# ------------------------------------------------------------------ elementary closed forms
def test_layer_norm(golden):
    g = golden("elementary.json")["layer_norm"]
    y = M.layer_norm(np.array(g["x"]), g["eps"])
    np.testing.assert_allclose(y, g["y"], rtol=0, atol=1e-15)
    x = R.standard_normal((7, 33)) * 3 + 5
    y = M.layer_norm(x)
    np.testing.assert_allclose(y.mean(-1), 0, atol=1e-12)
    np.testing.assert_allclose((y ** 2).mean(-1), 1, atol=1e-5)
    for row, yr in zip(x, y):
        np.testing.assert_allclose(yr, brute.layer_norm_loops(list(row)), atol=1e-12)


def test_gelu_silu(golden):
    g = golden("elementary.json")
    np.testing.assert_allclose(M.gelu(np.array(g["gelu"]["x"])), g["gelu"]["y"], atol=1e-15)
    x = R.standard_normal(100) * 4
    np.testing.assert_allclose(M.gelu(x) - M.gelu(-x), x, atol=1e-13)     # x Phi(x) + x Phi(-x) = x
    np.testing.assert_allclose(M.silu(x) - M.silu(-x), x, atol=1e-13)
    np.testing.assert_allclose(M.gelu(np.array([30.0, -30.0])), [30.0, 0.0], atol=1e-12)
    assert M.silu(np.array([0.0]))[0] == 0.0


def test_timestep_embedding(golden):
    g = golden("elementary.json")["timestep"]
    e = M.timestep_embedding(np.array(g["t"]), g["dim"])
    for i, v in g["index_value"]:
        assert abs(e[i] - v) < 1e-14
    e0 = M.timestep_embedding(np.array(0.0), 256)
    assert np.all(e0[:128] == 1.0) and np.all(e0[128:] == 0.0)
    e = M.timestep_embedding(R.uniform(size=5), 256)
    np.testing.assert_allclose(e[:, :128] ** 2 + e[:, 128:] ** 2, 1.0, atol=1e-14)


def _golden_condition_weights(g):
    w1 = np.zeros((g["hidden"], g["freq_dim"]))
    for row, col in g["w_t1_ones"]:
        w1[row, col] = 1.0
    return {"w_t1": w1, "b_t1": np.array(g["b_t1"]), "w_t2": np.array(g["w_t2"]),
            "b_t2": np.array(g["b_t2"])}


def test_condition(golden):
    """The timestep condition c = SiLU(W_t2 SiLU(W_t1 phi(t) + b_t1) + b_t2) that feeds every
    adaLN modulation (the velocity v_theta(z_t, t, tau) takes t, PaperReading review §2.2(2);
    the block's gating, §2.2(3)): a hand-worked value with one-hot first-layer rows and an
    asymmetric second layer (a transposed W_t2, a dropped SiLU or bias, or swapped layers all
    change it), and the batch axis (one row per sample) matches per-sample calls."""
    g = golden("elementary.json")["condition"]
    tw = _golden_condition_weights(g)
    c = M.condition(np.array(g["t"]), tw, g["freq_dim"])
    np.testing.assert_allclose(c, g["c"], rtol=0, atol=1e-15)
    d = synth.Dims(hidden=32, heads=2, channels=16)
    w = synth.model_weights(d, 1, 3, bf16=False)
    ts = np.array([0.0, 0.3, 1.0])
    batch = M.condition(ts, w.temb, d.freq_dim)
    for i, t in enumerate(ts):
        np.testing.assert_allclose(batch[i], M.condition(t, w.temb, d.freq_dim), rtol=0, atol=1e-15)


def _identity_stack(H=32, C=32):
    """A one-block stack whose image path is closed-form: identity latent embed, zero gates in
    both streams (the block is the identity on x), zero final modulation and identity output
    projection, so v = LN(z_t) row by row."""
    d = synth.Dims(hidden=H, heads=1, channels=C)
    w = synth.model_weights(d, 1, 11, bf16=False)
    w.embed = {"w_in": np.eye(H, C), "b_in": np.zeros(H)}
    for s in M.STREAMS:
        for ch in ("gate1", "gate2"):
            _set_mod(w.blocks[0], s, ch, 0.0, H)
    w.final = {"w_fmod": np.zeros((2 * H, H)), "b_fmod": np.zeros(2 * H), "w_out": np.eye(C, H),
               "b_out": np.zeros(C)}
    return d, w


def test_forward_composition():
    """forward = embed -> blocks -> final layer on one sample: with the closed-form stack above
    the velocity is LN(z_t), whatever the text tokens, t or the block's other weights."""
    d, w = _identity_stack()
    smp = synth.Sample(3, 1, 2, 5, 0.4)
    z = R.standard_normal((smp.img_len, d.channels))
    v = M.forward(R.standard_normal((3, d.hidden)), z, smp, 0.4, w, d.heads)
    np.testing.assert_allclose(v, M.layer_norm(z), atol=1e-13)
    assert v.shape == z.shape


def test_sample_cfg_constant_velocity():
    """The CFG sampler on a model whose velocity is a constant b (zero output weights, bias b):
    the guided velocity is b whatever w, and the Euler steps over a grid from t = 1 to t = 0
    add up to z0 + b (the steps' dt sum to 1 and move along +v)."""
    d, w = _identity_stack()
    b = R.standard_normal(d.channels)
    w.final["w_out"] = np.zeros_like(w.final["w_out"])
    w.final["b_out"] = b
    sc, su = synth.Sample(4, 1, 2, 3, 1.0, 1, 1), synth.Sample(0, 1, 2, 3, 1.0, 2, 0)
    z0 = R.standard_normal((sc.img_len, d.channels))
    for grid in ([1.0, 0.75, 0.5, 0.25, 0.0], list(np.linspace(1.0, 0.0, 21))):
        z = M.sample_cfg(R.standard_normal((4, d.hidden)), z0, sc, su, w, d.heads, 4.0, grid)
        np.testing.assert_allclose(z, z0 + b, atol=1e-12)


# ------------------------------------------------------------------ RoPE
def test_rope_known_rotation(golden):
    g = golden("elementary.json")["rope"]
    D = g["head_dim"]
    x = np.zeros((1, 1, D))
    x[0, 0, g["in_col"]] = 1.0
    y = M.apply_rope(x, np.array([g["pos"]]))
    np.testing.assert_allclose(y[0, 0, g["in_col"]:g["in_col"] + 2], g["out"], atol=1e-15)
    assert np.count_nonzero(np.abs(y) > 1e-15) == 2


def test_rope_matches_complex_loops():
    x = R.standard_normal((5, 2, 32))
    pos = R.integers(0, 50, size=(5, 3))
    pos[:, 0] = R.integers(0, 2, size=5)
    y = M.apply_rope(x, pos)
    yb = np.array(brute.rope_loops(x.tolist(), pos.tolist()))
    np.testing.assert_allclose(y, yb, atol=1e-12)


@pytest.mark.parametrize("D", [32, 64, 128])
def test_rope_invariances(D):
    q = R.standard_normal((1, 1, D))
    k = R.standard_normal((1, 1, D))
    # position 0 is the identity; rotations preserve the norm
    np.testing.assert_array_equal(M.apply_rope(q, np.zeros((1, 3), int)), q)
    p = np.array([[1, 37, 91]])
    np.testing.assert_allclose(np.linalg.norm(M.apply_rope(q, p)), np.linalg.norm(q), rtol=1e-13)
    # scores depend only on the relative offset (PaperReading review §2.2(2): per-sample RoPE)
    pq, pk = np.array([[1, 5, 9]]), np.array([[0, 17, 2]])
    for delta in ([0, 3, 4], [1, 0, 0], [0, 100, 0], [0, 0, 63]):
        d = np.array([delta])
        a = (M.apply_rope(q, pq) * M.apply_rope(k, pk)).sum()
        b = (M.apply_rope(q, pq + d) * M.apply_rope(k, pk + d)).sum()
        assert abs(a - b) < 1e-12 * max(1.0, abs(a))
    # each axis only touches its own block of the head: (D/8, 7D/16, 7D/16)
    wf, wr, wc = M.rope_axis_widths(D)
    assert wf + wr + wc == D and wf % 2 == 0 and wr % 2 == 0
    for axis, (lo, hi) in enumerate([(0, wf), (wf, wf + wr), (wf + wr, D)]):
        pp = np.zeros((1, 3), int)
        pp[0, axis] = 3
        y = M.apply_rope(q, pp)
        moved = np.nonzero(np.abs(y - q)[0, 0] > 1e-15)[0]
        assert moved.min() >= lo and moved.max() < hi


# ------------------------------------------------------------------ attention
def test_attention_bruteforce():
    q, k, v = (R.standard_normal((6, 2, 8)) for _ in range(3))
    o = M.attention(q, k, v)
    ob = np.array(brute.attention_loops(q.tolist(), k.tolist(), v.tolist()))
    np.testing.assert_allclose(o, ob, atol=1e-13)
    # row selection computes the same rows
    np.testing.assert_allclose(M.attention(q, k, v, rows=[4, 1]), o[[4, 1]], atol=1e-15)


def test_attention_special_cases():
    k, v = R.standard_normal((9, 3, 16)), R.standard_normal((9, 3, 16))
    o = M.attention(np.zeros((9, 3, 16)), k, v)            # equal scores -> mean of V
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(0), o.shape), atol=1e-14)
    o = M.attention(R.standard_normal((1, 3, 16)), k[:1], v[:1])   # one key -> that value
    np.testing.assert_allclose(o, v[:1], atol=1e-15)
    q = np.zeros((1, 1, 16))
    q[0, 0, 0] = 200.0
    kk = np.zeros((4, 1, 16))
    kk[2, 0, 0] = 1.0                                        # one dominant key
    vv = R.standard_normal((4, 1, 16))
    np.testing.assert_allclose(M.attention(q, kk, vv)[0], vv[2], atol=1e-12)


def test_packed_masked_attention_equals_per_sample():
    """Attention inside each sample only (PaperReading review §2.2(2)): a dense attention over
    the whole pack with a block-diagonal mask equals per-sample attention."""
    lens = [3, 7, 1, 5]
    N = sum(lens)
    q, k, v = (R.standard_normal((N, 2, 8)) for _ in range(3))
    seg = np.repeat(np.arange(len(lens)), lens)
    s = np.einsum("qhd,khd->hqk", q, k) / np.sqrt(8)
    s = np.where(seg[None, :, None] == seg[None, None, :], s, -np.inf)
    p = np.exp(s - s.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    dense = np.einsum("hqk,khd->qhd", p, v)
    off = np.concatenate([[0], np.cumsum(lens)])
    per = np.concatenate([M.attention(q[a:b], k[a:b], v[a:b]) for a, b in zip(off[:-1], off[1:])])
    np.testing.assert_allclose(dense, per, atol=1e-13)


# ------------------------------------------------------------------ block structure
def _tiny_block(seed=0, H=64, heads=2):
    d = synth.Dims(hidden=H, heads=heads, channels=16)
    w = synth.model_weights(d, 1, seed, bf16=False)
    return d, w


# The reading of the adaLN modulation layout: 6 chunks of H in this order.
CHUNK_INDEX = {"shift1": 0, "scale1": 1, "gate1": 2, "shift2": 3, "scale2": 4, "gate2": 5}


def _set_mod(bw, stream, chunk, value, H):
    """Zero the stream's modulation weights and make chunk `chunk` equal `value`."""
    bw[stream]["w_mod"] = np.zeros_like(bw[stream]["w_mod"])
    b = np.zeros(6 * H)
    i = CHUNK_INDEX[chunk]
    b[i * H:(i + 1) * H] = value
    bw[stream]["b_mod"] = b


def test_block_zero_gates_is_identity():
    d, w = _tiny_block()
    bw = copy.deepcopy(w.blocks[0])
    for s in M.STREAMS:
        _set_mod(bw, s, "shift1", 0.3, d.hidden)                 # gates stay 0
    xt, xi = R.standard_normal((5, 64)), R.standard_normal((12, 64))
    pos = M.image_positions(1, 3, 4)
    ot, oi = M.block_forward(xt, xi, pos, np.ones(64), bw, d.heads)
    np.testing.assert_array_equal(ot, xt)
    np.testing.assert_array_equal(oi, xi)


@pytest.mark.parametrize("stream", M.STREAMS)
def test_block_gate_and_bias_paths(stream):
    """gate1 = 1, W_o = 0: out = x + b_o on that stream only; gate2 = 1, W_2 = 0: x + b_2."""
    d, w = _tiny_block()
    H = d.hidden
    xt, xi = R.standard_normal((5, H)), R.standard_normal((12, H))
    pos = M.image_positions(1, 3, 4)
    other = "img" if stream == "txt" else "txt"
    for gate, wname, bname in (("gate1", "w_o", "b_o"), ("gate2", "w_2", "b_2")):
        bw = copy.deepcopy(w.blocks[0])
        _set_mod(bw, stream, gate, 1.0, H)
        _set_mod(bw, other, "shift1", 0.0, H)
        bw[stream][wname] = np.zeros_like(bw[stream][wname])
        if gate == "gate2":
            bw[stream]["w_1"] = np.zeros_like(bw[stream]["w_1"])
        ot, oi = M.block_forward(xt, xi, pos, np.ones(H), bw, d.heads)
        got, x0 = (ot, xt) if stream == "txt" else (oi, xi)
        np.testing.assert_allclose(got, x0 + bw[stream][bname], atol=1e-14)
        np.testing.assert_array_equal(oi if stream == "txt" else ot, xi if stream == "txt" else xt)


def test_block_scale_minus_one_case():
    """scale1 = -1 makes every token's attention input equal shift1, so q, k, v are the same
    for all tokens and attention returns v itself: out = x + gate1 (v W_o^T + b_o), with
    v = shift1 W_v^T + b_v (the third H-slice of the fused QKV, made equal for both streams).  scale2 = -1 likewise makes the
    MLP input equal shift2.  Pins the chunk order, the QKV slicing and the residual chain."""
    d, w = _tiny_block()
    H = d.hidden
    bw = copy.deepcopy(w.blocks[0])
    rng = np.random.default_rng(7)
    sh1, sh2, g1, g2 = (rng.standard_normal(H) for _ in range(4))
    for s in M.STREAMS:
        bw[s]["w_mod"] = np.zeros_like(bw[s]["w_mod"])
        bw[s]["b_mod"] = np.concatenate([sh1, -np.ones(H), g1, sh2, -np.ones(H), g2])
    # one value projection for both streams, so every token of the sample carries the same v
    bw["txt"]["w_qkv"][2 * H:] = bw["img"]["w_qkv"][2 * H:]
    bw["txt"]["b_qkv"][2 * H:] = bw["img"]["b_qkv"][2 * H:]
    xt, xi = R.standard_normal((3, H)), R.standard_normal((8, H))
    ot, oi = M.block_forward(xt, xi, M.image_positions(1, 2, 4), np.ones(H), bw, d.heads)
    for x, o, s in ((xt, ot, "txt"), (xi, oi, "img")):
        wq = bw[s]["w_qkv"]
        v = wq[2 * H:] @ sh1 + bw[s]["b_qkv"][2 * H:]
        x1 = x + g1 * (bw[s]["w_o"] @ v + bw[s]["b_o"])
        hid = bw[s]["w_1"] @ sh2 + bw[s]["b_1"]
        hid = hid * 0.5 * (1 + M.erf(hid / np.sqrt(2)))
        np.testing.assert_allclose(o, x1 + g2 * (bw[s]["w_2"] @ hid + bw[s]["b_2"]), atol=1e-12)


def test_final_layer_scale_minus_one():
    d, w = _tiny_block()
    H, C = d.hidden, d.channels
    fw = dict(w.final)
    shift = R.standard_normal(H)
    fw["w_fmod"] = np.zeros_like(fw["w_fmod"])
    fw["b_fmod"] = np.concatenate([shift, -np.ones(H)])
    out = M.final_layer(R.standard_normal((5, H)), np.ones(H), fw)
    np.testing.assert_allclose(out, np.broadcast_to(fw["w_out"] @ shift + fw["b_out"], (5, C)),
                               atol=1e-13)


def test_block_position_shift_invariance_image_only():
    """RoPE enters only q and k, so an image-only sample's block output does not change when
    every position moves by the same offset (scores depend on relative offsets only)."""
    d, w = _tiny_block()
    xi = R.standard_normal((12, 64))
    pos = M.image_positions(1, 3, 4)
    c = R.standard_normal(64)
    _, a = M.block_forward(np.zeros((0, 64)), xi, pos, c, w.blocks[0], d.heads)
    _, b = M.block_forward(np.zeros((0, 64)), xi, pos + np.array([1, 7, 3]), c, w.blocks[0], d.heads)
    np.testing.assert_allclose(a, b, atol=1e-12)
    # but a text token sees the shift (it stays at the origin)
    xt = R.standard_normal((3, 64))
    _, a = M.block_forward(xt, xi, pos, c, w.blocks[0], d.heads)
    _, b = M.block_forward(xt, xi, pos + np.array([0, 7, 3]), c, w.blocks[0], d.heads)
    assert np.abs(a - b).max() > 1e-6


def test_block_row_selection_and_single_token():
    d, w = _tiny_block()
    xt, xi = R.standard_normal((4, 64)), R.standard_normal((6, 64))
    pos = M.image_positions(1, 2, 3)
    c = R.standard_normal(64)
    ot, oi = M.block_forward(xt, xi, pos, c, w.blocks[0], d.heads)
    rows = [0, 3, 4, 9]
    sel = M.block_forward(xt, xi, pos, c, w.blocks[0], d.heads, rows=rows)
    np.testing.assert_allclose(sel, np.concatenate([ot, oi])[rows], atol=1e-13)


def test_block_uniform_attention_case():
    """With zero q weights every score is 0, so each token attends uniformly: the result must
    equal the block evaluated with the attention output replaced by the mean value row."""
    d, w = _tiny_block()
    H = d.hidden
    bw = copy.deepcopy(w.blocks[0])
    for s in M.STREAMS:
        bw[s]["w_qkv"][:H] = 0.0
        bw[s]["b_qkv"][:H] = 0.0
    xt, xi = R.standard_normal((4, H)), R.standard_normal((6, H))
    pos = M.image_positions(1, 2, 3)
    c = R.standard_normal(H)
    ot, oi = M.block_forward(xt, xi, pos, c, bw, d.heads)
    # the mean value row is position independent, so moving the image changes nothing
    ot2, oi2 = M.block_forward(xt, xi, pos + np.array([1, 9, 9]), c, bw, d.heads)
    np.testing.assert_allclose(ot, ot2, atol=1e-13)
    np.testing.assert_allclose(oi, oi2, atol=1e-13)
    # permuting the sample's image tokens permutes the image outputs
    perm = R.permutation(6)
    _, oi3 = M.block_forward(xt, xi[perm], pos[perm], c, bw, d.heads)
    np.testing.assert_allclose(oi3, oi[perm], atol=1e-13)


def test_token_permutation_equivariance():
    """Moving tokens together with their positions permutes the block output (attention is a
    set operation once positions ride with the tokens)."""
    d, w = _tiny_block()
    xi = R.standard_normal((12, 64))
    pos = M.image_positions(2, 2, 3)
    c = R.standard_normal(64)
    xt = R.standard_normal((3, 64))
    _, a = M.block_forward(xt, xi, pos, c, w.blocks[0], d.heads)
    perm = R.permutation(12)
    _, b = M.block_forward(xt, xi[perm], pos[perm], c, w.blocks[0], d.heads)
    np.testing.assert_allclose(b, a[perm], atol=1e-12)


# ------------------------------------------------------------------ rectified flow
def test_flow_matching_hand_worked(golden):
    g = golden("flow_matching.json")
    z, e, t = np.array(g["z"]), np.array(g["eps"]), g["t"]
    np.testing.assert_allclose(M.interpolate(z, e, t), g["z_t"], atol=1e-15)
    s, n = M.flow_loss(np.array(g["v"]), z, e)
    assert abs(s - g["loss_sum"]) < 1e-15 and n == 2
    np.testing.assert_allclose(M.euler_step(M.interpolate(z, e, t), z - e, g["euler_dt"]),
                               g["euler_from_z_t_with_v_star"], atol=1e-15)
    np.testing.assert_allclose(M.cfg_combine(np.array(g["cfg_v_cond"]), np.array(g["cfg_v_uncond"]),
                                             g["cfg_w"]), g["cfg_out"], atol=1e-15)


def test_interpolation_endpoints_and_loss_zero():
    z, e = R.standard_normal((10, 4)), R.standard_normal((10, 4))
    np.testing.assert_array_equal(M.interpolate(z, e, 0.0), z)
    np.testing.assert_array_equal(M.interpolate(z, e, 1.0), e)
    assert M.flow_loss(z - e, z, e) == (0.0, 40)
    tgt = np.arange(10) >= 4                                  # edit: source rows clean
    zt = M.interpolate(z, e, 0.7, tgt)
    np.testing.assert_array_equal(zt[:4], z[:4])
    s, n = M.flow_loss(np.zeros_like(z), z, e, tgt)
    assert n == 24 and abs(s - ((z - e)[4:] ** 2).sum()) < 1e-12
    assert M.mean_loss([2.0, 4.0], [1, 3]) == 1.5


def test_euler_straight_path():
    """With the exact velocity v = z - eps, every Euler step lands on the straight path, so 4
    steps from z_1 = eps reach z (the sign/dt convention of the sampler)."""
    z, e = R.standard_normal(20), R.standard_normal(20)
    grid = [1.0, 0.75, 0.5, 0.25, 0.0]
    x = e.copy()
    for a, b in zip(grid[:-1], grid[1:]):
        x = M.euler_step(x, z - e, a - b)
        np.testing.assert_allclose(x, M.interpolate(z, e, b), atol=1e-14)
    np.testing.assert_allclose(x, z, atol=1e-14)


def test_cfg_limits():
    vc, vu = R.standard_normal(7), R.standard_normal(7)
    np.testing.assert_allclose(M.cfg_combine(vc, vu, 1.0), vc, atol=1e-15)
    np.testing.assert_array_equal(M.cfg_combine(vc, vu, 0.0), vu)


def test_nft_loss_pins():
    """Diffusion-NFT objective [PR 2.2(4)]: a hand-worked value, the reward limits (r = 1 is the
    flow loss of v+, r = 0 that of v-), equal velocities reduce to the flow loss for any r,
    linearity in r, and target-frame masking."""
    z, e = np.array([1.0, 2.0]), np.array([0.5, -1.0])          # v* = z - eps = [0.5, 3]
    vp, vn = np.array([1.0, 3.0]), np.array([0.0, 0.0])
    # 0.25 * (0.5^2 + 0^2) + 0.75 * (0.5^2 + 3^2) = 0.0625 + 6.9375
    assert M.nft_loss(vp, vn, z, e, 0.25) == (7.0, 2)
    z, e = R.standard_normal((9, 5)), R.standard_normal((9, 5))
    vp, vn = R.standard_normal((9, 5)), R.standard_normal((9, 5))
    assert M.nft_loss(vp, vn, z, e, 1.0) == M.flow_loss(vp, z, e)
    assert M.nft_loss(vp, vn, z, e, 0.0) == M.flow_loss(vn, z, e)
    s, n = M.nft_loss(vp, vp, z, e, 0.37)
    assert n == 45 and abs(s - M.flow_loss(vp, z, e)[0]) < 1e-12
    s1, s0 = M.nft_loss(vp, vn, z, e, 1.0)[0], M.nft_loss(vp, vn, z, e, 0.0)[0]
    assert abs(M.nft_loss(vp, vn, z, e, 0.6)[0] - (0.6 * s1 + 0.4 * s0)) < 1e-12
    tgt = np.arange(9) >= 3
    s, n = M.nft_loss(vp, vn, z, e, 0.6, tgt)
    assert n == 30 and abs(s - M.nft_loss(vp[3:], vn[3:], z[3:], e[3:], 0.6)[0]) < 1e-12


# ------------------------------------------------------------------ planted mistakes
def test_rms_norm_heads_pins():
    """QK-RMSNorm: a hand-worked vector, unit RMS per head whatever the heads' scales (a norm
    over the whole row, or over the heads, fails this), per-head scale invariance, and the
    scale applied per dimension."""
    y = M.rms_norm_heads(np.array([[[3.0, 4.0]]]), np.array([2.0, 0.5]), eps=0.0)
    r = np.sqrt(12.5)                                                   # sqrt((9 + 16) / 2)
    np.testing.assert_allclose(y[0, 0], [6.0 / r, 2.0 / r], rtol=1e-15)
    x = R.standard_normal((6, 4, 32)) * np.array([1e-2, 1.0, 30.0, 3.0])[None, :, None]
    y = M.rms_norm_heads(x, np.ones(32), eps=0.0)
    np.testing.assert_allclose(np.sqrt((y ** 2).mean(-1)), 1.0, rtol=1e-12)
    a = np.array([0.5, 7.0, 0.01, 2.0])[None, :, None]
    np.testing.assert_allclose(M.rms_norm_heads(x * a, np.ones(32), eps=0.0), y, rtol=1e-12)
    g = 1.0 + R.standard_normal(32)
    np.testing.assert_allclose(M.rms_norm_heads(x, g, eps=0.0), y * g, rtol=1e-12)
    # eps enters under the root: a zero head stays zero, a tiny one is damped
    z = M.rms_norm_heads(np.zeros((1, 1, 4)), np.ones(4))
    np.testing.assert_array_equal(z, 0.0)
    t = M.rms_norm_heads(np.full((1, 1, 4), 1e-3), np.ones(4), eps=1e-6)
    np.testing.assert_allclose(t, 1e-3 / np.sqrt(1e-6 + 1e-6), rtol=1e-12)


def test_block_qk_norm_invariance():
    """With QK-RMSNorm on, scaling a stream's query (or key) projection by a positive factor
    leaves the block output unchanged up to the eps term, while without it the output moves;
    with unit scales the queries and keys that reach attention have unit RMS per head (the
    norm comes before RoPE, which keeps it)."""
    d = synth.Dims(hidden=64, heads=2, channels=16)
    w = synth.model_weights(d, 1, 5, bf16=False, qk_norm=True)
    H = d.hidden
    xt, xi = R.standard_normal((5, H)), R.standard_normal((12, H))
    pos = M.image_positions(1, 3, 4)
    c = R.standard_normal(H)
    ref = np.concatenate(M.block_forward(xt, xi, pos, c, w.blocks[0], d.heads))
    for s in M.STREAMS:
        for part in (0, 1):                                              # q rows, k rows of W_qkv
            bw = copy.deepcopy(w.blocks[0])
            bw[s]["w_qkv"][part * H:(part + 1) * H] *= 20.0
            bw[s]["b_qkv"][part * H:(part + 1) * H] *= 20.0
            got = np.concatenate(M.block_forward(xt, xi, pos, c, bw, d.heads))
            np.testing.assert_allclose(got, ref, rtol=0, atol=1e-5 * np.abs(ref).max())
            off = {st: {k: v for k, v in bw[st].items() if k not in ("w_qnorm", "w_knorm")} for st in M.STREAMS}
            base = {st: {k: v for k, v in w.blocks[0][st].items() if k not in ("w_qnorm", "w_knorm")}
                    for st in M.STREAMS}
            moved = np.concatenate(M.block_forward(xt, xi, pos, c, off, d.heads)) - \
                np.concatenate(M.block_forward(xt, xi, pos, c, base, d.heads))
            assert np.abs(moved).max() > 10 * 1e-5 * np.abs(ref).max()
    bw = copy.deepcopy(w.blocks[0])
    calls = []
    orig = M.attention

    def spy(q, k, v, rows=None):
        calls.append((M.f64(q), M.f64(k)))
        return orig(q, k, v, rows)

    import unittest.mock as um
    for st in M.STREAMS:
        bw[st]["w_qnorm"] = np.ones(d.head_dim)
        bw[st]["w_knorm"] = np.ones(d.head_dim)
    with um.patch.object(M, "attention", spy):
        M.block_forward(xt, xi, pos, c, bw, d.heads)
    q, k = calls[-1]
    np.testing.assert_allclose(np.sqrt((q ** 2).mean(-1)), 1.0, rtol=1e-3)   # RoPE keeps the RMS (eps: 1e-4)
    np.testing.assert_allclose(np.sqrt((k ** 2).mean(-1)), 1.0, rtol=1e-3)


def _pins_pass():
    """A compact battery of the pins above, for the planted-mistake test."""
    from tests.conftest import load_golden
    try:
        test_layer_norm(load_golden)
        test_gelu_silu(load_golden)
        test_timestep_embedding(load_golden)
        test_condition(load_golden)
        test_rope_known_rotation(load_golden)
        test_rope_matches_complex_loops()
        for D in (32, 64):
            test_rope_invariances(D)
        test_attention_bruteforce()
        test_attention_special_cases()
        test_block_zero_gates_is_identity()
        for s in M.STREAMS:
            test_block_gate_and_bias_paths(s)
        test_block_position_shift_invariance_image_only()
        test_block_scale_minus_one_case()
        test_final_layer_scale_minus_one()
        test_forward_composition()
        test_sample_cfg_constant_velocity()
        test_flow_matching_hand_worked(load_golden)
        test_interpolation_endpoints_and_loss_zero()
        test_euler_straight_path()
        test_cfg_limits()
        test_nft_loss_pins()
        test_rms_norm_heads_pins()
        test_block_qk_norm_invariance()
    except (AssertionError, ValueError):      # a mutant that breaks a shape is caught too
        return False
    return True


ORIG = {n: getattr(M, n) for n in ("layer_norm", "gelu", "timestep_embedding", "condition", "rope_angles",
                                     "rms_norm_heads",
                                     "attention", "interpolate", "flow_loss", "euler_step",
                                     "cfg_combine", "nft_loss")}


def _mut_layer_norm(x, eps=M.LN_EPS):              # unbiased variance
    x = M.f64(x)
    mu = x.mean(-1, keepdims=True)
    return (x - mu) / np.sqrt(((x - mu) ** 2).sum(-1, keepdims=True) / (x.shape[-1] - 1) + eps)


def _mut_attention(q, k, v, rows=None):            # missing 1/sqrt(D)
    q, k, v = M.f64(q), M.f64(k), M.f64(v)
    if rows is not None:
        q = q[rows]
    s = np.einsum("qhd,khd->hqk", q, k)
    p = np.exp(s - s.max(-1, keepdims=True))
    return np.einsum("hqk,khd->qhd", p / p.sum(-1, keepdims=True), v)


def _mut_condition(kind):
    """Planted mistakes in the timestep condition (c = SiLU(W_t2 SiLU(W_t1 phi + b_t1) + b_t2))."""
    def cond(t, temb_w, freq_dim=256):
        phi = M.timestep_embedding(t, freq_dim)
        w1, b1, w2, b2 = (temb_w[k] for k in ("w_t1", "b_t1", "w_t2", "b_t2"))
        if kind == "swapped_layers":
            w1, b1, w2, b2 = w2, b2, w1, b1
        h = M.linear(phi, w1, b1)
        if kind != "no_inner_silu":
            h = M.silu(h)
        if kind == "w_t2_transposed":
            out = h @ M.f64(w2) + M.f64(b2)
        elif kind == "no_b_t2":
            out = h @ M.f64(w2).T
        else:
            out = M.linear(h, w2, b2)
        return out if kind == "no_final_silu" else M.silu(out)
    return cond


MUTANTS = {
    "layer_norm_unbiased_var": ("layer_norm", _mut_layer_norm),
    "gelu_wrong_sign": ("gelu", lambda x: 0.5 * M.f64(x) * (1.0 - M.erf(M.f64(x) / np.sqrt(2)))),
    "timestep_sin_cos_order": ("timestep_embedding",
                               lambda t, dim=256: np.roll(ORIG["timestep_embedding"](t, dim), dim // 2, -1)),
    "condition_no_final_silu": ("condition", _mut_condition("no_final_silu")),
    "condition_no_inner_silu": ("condition", _mut_condition("no_inner_silu")),
    "condition_w_t2_transposed": ("condition", _mut_condition("w_t2_transposed")),
    "condition_no_b_t2": ("condition", _mut_condition("no_b_t2")),
    "condition_swapped_layers": ("condition", _mut_condition("swapped_layers")),
    "rope_axes_swapped": ("rope_angles", lambda pos, D: ORIG["rope_angles"](np.asarray(pos)[:, [1, 0, 2]], D)),
    "rope_base_wrong": ("rope_angles", lambda pos, D: ORIG["rope_angles"](pos, D) * 1.01),
    "attention_no_scale": ("attention", _mut_attention),
    "interp_t_swapped": ("interpolate", lambda z, e, t, target=None: ORIG["interpolate"](z, e, 1.0 - t, target)),
    "loss_sign": ("flow_loss", lambda v, z, e, target=None: ORIG["flow_loss"](v, e, z, target)),
    "euler_sign": ("euler_step", lambda z, v, dt: M.f64(z) - dt * M.f64(v)),
    "cfg_swapped": ("cfg_combine", lambda vc, vu, w: ORIG["cfg_combine"](vu, vc, w)),
    "nft_reward_swapped": ("nft_loss", lambda vp, vn, z, e, r, target=None:
                           ORIG["nft_loss"](vp, vn, z, e, 1.0 - r, target)),
    "nft_target_sign": ("nft_loss", lambda vp, vn, z, e, r, target=None:
                        ORIG["nft_loss"](vp, vn, e, z, r, target)),
    "nft_no_negative_term": ("nft_loss", lambda vp, vn, z, e, r, target=None:
                             ORIG["nft_loss"](vp, vp, z, e, 1.0, target)),
    "rms_over_whole_row": ("rms_norm_heads", lambda x, g, eps=M.RMS_EPS:
                           M.f64(x) / np.sqrt((M.f64(x) ** 2).mean(axis=(-2, -1), keepdims=True) + eps) * M.f64(g)),
    "rms_eps_outside_root": ("rms_norm_heads", lambda x, g, eps=M.RMS_EPS:
                             M.f64(x) / (np.sqrt((M.f64(x) ** 2).mean(-1, keepdims=True)) + eps) * M.f64(g)),
    "rms_no_scale": ("rms_norm_heads", lambda x, g, eps=M.RMS_EPS: ORIG["rms_norm_heads"](x, np.ones_like(M.f64(g)), eps)),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes(name, monkeypatch):
    """Plant one plausible mistake in the oracle (on the CPU) and check the pins catch it."""
    fn, mutant = MUTANTS[name]
    assert _pins_pass(), "pins must pass on the unmodified oracle"
    monkeypatch.setattr(M, fn, mutant)
    assert not _pins_pass(), f"planted mistake {name} was not caught"


def test_planted_block_mistakes(monkeypatch):
    """Mistakes in the block's composition: modulation chunks in the wrong order, or the text
    rows using the image weights."""
    assert _pins_pass()
    for order in (("shift1", "scale1", "gate2", "shift2", "scale2", "gate1"),
                  ("scale1", "shift1", "gate1", "shift2", "scale2", "gate2"),
                  ("shift1", "scale1", "gate1", "scale2", "shift2", "gate2")):
        monkeypatch.setattr(M, "MOD_CHUNKS", order)
        assert not _pins_pass(), order
        monkeypatch.undo()
    orig = M.block_forward

    def crossed(x_txt, x_img, pos_img, c, bw, heads, rows=None):
        return orig(x_txt, x_img, pos_img, c, {"txt": bw["img"], "img": bw["img"]}, heads, rows)

    monkeypatch.setattr(M, "block_forward", crossed)
    assert not _pins_pass()
