"""GPU parity of the block backward through the C ABI (mf_block_forward_train, then
mf_block_backward) against the oracle's reverse-mode gradients (oracle.grad.block_vjp), one
sample at a time: the input gradients of both streams, every weight gradient of both streams
(summed over the pack's samples) and each sample's condition gradient.  Tiny configuration
(H = 256, 4 heads x 64) and ragged H = 512 packs (4 heads x 128)."""
import numpy as np
import pytest

import synth
from oracle import grad as G
from oracle import model as M
from oracle import pack as opack
from tests.helpers import assert_close, stream_concat

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import packed_rectified_flow_packer_b300 as mf
    from packed_rectified_flow_packer_b300.device import DeviceModel, to_bf16

MID = synth.Dims(hidden=512, heads=4, channels=128)


def _f(t):
    return t.double().cpu().numpy()


def _mid_samples(seed, n=6):
    g = np.random.default_rng(seed)
    return [synth.Sample(int(g.integers(0, 140)), int(g.integers(1, 3)), int(g.integers(2, 24)),
                         int(g.integers(2, 24)), float(g.uniform())) for _ in range(n)]


def _run_case(samples, dims, seed):
    H = dims.hidden
    budget = sum(s.length for s in samples)
    ref = opack.build_plan(samples, budget)
    plan = mf.mf_pack(samples, budget)
    mf.mf_plan_upload(plan)
    w = synth.model_weights(dims, 1, seed)
    model = DeviceModel(w)
    d, bs = model.dims, model.block_structs[0]
    order = ref.order
    xt_parts = [synth.round_bf16(synth.normal(seed, f"bwd.x_txt.{i}", (s.txt_len, H))) for i, s in enumerate(samples)]
    xi_parts = [synth.round_bf16(synth.normal(seed, f"bwd.x_img.{i}", (s.img_len, H))) for i, s in enumerate(samples)]
    gt_parts = [synth.round_bf16(synth.normal(seed, f"bwd.g_txt.{i}", (s.txt_len, H))) for i, s in enumerate(samples)]
    gi_parts = [synth.round_bf16(synth.normal(seed, f"bwd.g_img.{i}", (s.img_len, H))) for i, s in enumerate(samples)]
    xt, xi = stream_concat(xt_parts, order, H), stream_concat(xi_parts, order, H)
    gt, gi = stream_concat(gt_parts, order, H), stream_concat(gi_parts, order, H)
    t = torch.tensor([samples[c].t for c in order], dtype=torch.float32, device="cuda")

    # training forward (its output must equal the inference forward's bit for bit)
    X_t, X_i = to_bf16(xt if len(xt) else np.zeros((1, H), np.float32)), to_bf16(xi)
    tws = torch.empty(mf.mf_block_train_workspace_bytes(plan, d), dtype=torch.uint8, device="cuda")
    mf.mf_block_forward_train(plan, d, bs, t, X_t, X_i, tws)
    Y_t, Y_i = to_bf16(xt if len(xt) else np.zeros((1, H), np.float32)), to_bf16(xi)
    iws = torch.empty(mf.mf_block_workspace_bytes(plan, d), dtype=torch.uint8, device="cuda")
    mf.mf_block_forward(plan, d, bs, t, Y_t, Y_i, iws)
    mf.mf_check()
    assert torch.equal(X_t, Y_t) and torch.equal(X_i, Y_i)

    # backward
    DX_t, DX_i = to_bf16(gt if len(gt) else np.zeros((1, H), np.float32)), to_bf16(gi)
    grads = {s: {k: torch.full(v.shape, float("nan"), dtype=torch.float32, device="cuda")
                 for k, v in w.blocks[0][s].items()} for s in M.STREAMS}
    gstruct = mf.grads_struct(grads["txt"], grads["img"])
    dc = torch.full((len(order), H), float("nan"), dtype=torch.float32, device="cuda")
    bws = torch.empty(mf.mf_block_backward_workspace_bytes(plan, d), dtype=torch.uint8, device="cuda")
    mf.mf_block_backward(plan, d, bs, tws, DX_t, DX_i, gstruct, dc, bws)
    mf.mf_check()

    # oracle, one sample at a time
    want_wg = {s: {k: np.zeros(v.shape) for k, v in w.blocks[0][s].items()} for s in M.STREAMS}
    want_dxt, want_dxi, want_dc = [], [], []
    for k, ci in enumerate(order):
        s = samples[ci]
        c = M.condition(s.t, w.temb, dims.freq_dim)
        pos = M.image_positions(s.frames, s.lat_h, s.lat_w)
        out = G.block_vjp(xt_parts[ci], xi_parts[ci], pos, c, w.blocks[0], dims.heads, gt_parts[ci], gi_parts[ci])
        want_dxt.append(out["x_txt"])
        want_dxi.append(out["x_img"])
        want_dc.append(out["c"])
        for st in M.STREAMS:
            for name in want_wg[st]:
                want_wg[st][name] += out[st][name]
    cat = lambda a: np.concatenate(a) if a else np.zeros((0, H))          # noqa: E731
    if ref.n_txt:
        assert_close(_f(DX_t)[:ref.n_txt], cat(want_dxt), "dx text")
    assert_close(_f(DX_i), cat(want_dxi), "dx image")
    assert_close(_f(dc), np.stack(want_dc), "dc")
    for st in M.STREAMS:
        if st == "txt" and ref.n_txt == 0:
            continue
        for name, arr in want_wg[st].items():
            assert_close(_f(grads[st][name]), arr, f"d{name} ({st})")


def test_tiny_block_backward():
    _run_case(synth.tiny_samples(), synth.TINY, seed=21)


@pytest.mark.parametrize("seed", [0, 1])
def test_mid_pack_block_backward(seed):
    """Ragged H = 512 packs: GEMM row tiles with tails, edit samples (two frames), text lengths
    from 0, row chunks that end inside a sample."""
    _run_case(_mid_samples(seed + 40), MID, seed=seed + 50)


def test_h768_block_backward():
    """H = 768 (6 heads x 128): hidden sizes that are not a power of two, 3 N tiles of 256 in
    the H-wide products and 12 in the MLP."""
    _run_case(_mid_samples(70), synth.Dims(hidden=768, heads=6, channels=64), seed=71)


@pytest.mark.slow
def test_wide_block_backward():
    """H = 4096 (32 heads x 128), the widest supported hidden size: the 512-thread row kernels
    and the widest statistics and GEMV instantiations; one text + image sample and one
    two-frame edit sample without text."""
    samples = [synth.Sample(13, 1, 3, 4, 0.4), synth.Sample(0, 2, 3, 3, 0.7)]
    _run_case(samples, synth.Dims(hidden=4096, heads=32, channels=64), seed=61)
