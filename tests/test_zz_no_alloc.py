"""The allocation-free flow loss, mf_flow_loss_noalloc, against mf_flow_loss and the oracle.

mf_flow_loss_noalloc is for callers that cannot allocate device memory where they compute
the loss: their allocator belongs to another framework that forbids side allocations, their
memory budget is fixed up front, or an allocation there would synchronise the device at the
wrong moment.  It keeps its per-row scratch in a fixed array inside the library instead of
taking a workspace.  These tests call it through the C ABI several times in a row, on packs of
different sizes (so rows left by an earlier call would show up if they leaked), and compare
every result with mf_flow_loss on the same inputs and with the oracle's per-sample sums.  The
file runs last in the suite and also passes on its own in a fresh process."""
import numpy as np
import pytest

import synth
from oracle import model as M
from oracle import pack as opack

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import packed_rectified_flow_packer_b300 as mf


def _plan(samples):
    plan = mf.mf_pack(samples, sum(s.length for s in samples))
    mf.mf_plan_upload(plan)
    return plan


def _inputs(n_img, C, seed):
    g = np.random.default_rng(seed)
    return [torch.from_numpy(g.standard_normal((n_img, C)).astype(np.float32)).cuda() for _ in range(3)]


def _with_workspace(plan, C, z, e, v):
    S = plan.n_seq
    ls = torch.zeros(S, dtype=torch.float64, device="cuda")
    cnt = torch.zeros(S, dtype=torch.int64, device="cuda")
    mean = torch.zeros(1, dtype=torch.float64, device="cuda")
    ws = torch.empty(mf.mf_flow_loss_workspace_bytes(plan), dtype=torch.uint8, device="cuda")
    mf.mf_flow_loss(plan, C, z, e, v, ls, cnt, mean, ws)
    return ls, cnt, mean


def _without_workspace(plan, C, z, e, v):
    S = plan.n_seq
    ls = torch.full((S,), float("nan"), dtype=torch.float64, device="cuda")
    cnt = torch.full((S,), -1, dtype=torch.int64, device="cuda")
    mean = torch.full((1,), float("nan"), dtype=torch.float64, device="cuda")
    mf.mf_flow_loss_noalloc(plan, C, z, e, v, ls, cnt, mean)
    return ls, cnt, mean


def test_noalloc_loss_matches_workspace_loss_on_consecutive_calls():
    big = [synth.Sample(40, 2, 30, 41, 0.3), synth.Sample(7, 1, 50, 33, 0.8),
           synth.Sample(0, 1, 61, 64, 0.5)]
    small = [synth.Sample(5, 1, 3, 4, 0.3), synth.Sample(3, 2, 2, 5, 0.7)]
    cases = [(big, 128, 1), (small, 64, 2), (big, 128, 3)]
    for samples, C, seed in cases:
        plan = _plan(samples)
        z, e, v = _inputs(plan.n_img, C, seed)
        ref = _with_workspace(plan, C, z, e, v)
        got = _without_workspace(plan, C, z, e, v)
        mf.mf_check()
        np.testing.assert_allclose(got[0].cpu().numpy(), ref[0].cpu().numpy(), rtol=1e-12)
        np.testing.assert_array_equal(got[1].cpu().numpy(), ref[1].cpu().numpy())
        np.testing.assert_allclose(got[2].cpu().numpy(), ref[2].cpu().numpy(), rtol=1e-12)
        # and the oracle: per-sample sums over target-frame elements, counts, the mean
        op = opack.build_plan(samples, sum(s.length for s in samples))
        zh, eh, vh = (x.double().cpu().numpy() for x in (z, e, v))
        sums, counts = [], []
        for k, c in enumerate(op.order):
            a, b = op.cu_img[k], op.cu_img[k + 1]
            sm, n = M.flow_loss(vh[a:b], zh[a:b], eh[a:b], M.target_mask(samples[c]))
            sums.append(sm)
            counts.append(n)
        np.testing.assert_allclose(got[0].cpu().numpy(), sums, rtol=1e-12)
        np.testing.assert_array_equal(got[1].cpu().numpy(), counts)
        assert abs(got[2].item() - M.mean_loss(sums, counts)) <= 1e-12 * abs(got[2].item())


def test_noalloc_rejects_packs_beyond_its_scratch():
    """More image rows than the built-in scratch holds: a clear error, before any launch."""
    s = [synth.Sample(1, 1, 257, 256, 0.5)]          # 65792 image rows > 65536
    plan = _plan(s)
    assert plan.n_img > mf.NOALLOC_MAX_IMG_ROWS
    C = 64
    z, e, v = _inputs(plan.n_img, C, 4)
    ls = torch.zeros(1, dtype=torch.float64, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    mean = torch.zeros(1, dtype=torch.float64, device="cuda")
    st = mf.lib.mf_flow_loss_noalloc(plan.handle, C, z.data_ptr(), e.data_ptr(), v.data_ptr(),
                                     ls.data_ptr(), cnt.data_ptr(), mean.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    assert mf.STATUS[st] == "MF_ERR_WORKSPACE"
    mf.mf_check()
