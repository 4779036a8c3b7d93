"""GPU parity of the varlen attention backward through the C ABI (mf_attention_lse,
mf_attention_backward) against the oracle's gradients (oracle.grad): ragged samples of 1 to
1217 tokens with tile tails on both sides of the 64-query and 128-key tiles, head dims 64 and
128, and one sample of 16384 tokens checked on sampled rows."""
import numpy as np
import pytest

import synth
from oracle import grad as G
from oracle import pack as opack
from tests.helpers import assert_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import packed_rectified_flow_packer_b300 as mf
    from packed_rectified_flow_packer_b300.device import to_bf16

ATTN_SAMPLES = [synth.Sample(3, 1, 1, 2, 0.5), synth.Sample(0, 1, 1, 1, 0.5),
                synth.Sample(27, 1, 10, 10, 0.5), synth.Sample(28, 1, 10, 10, 0.5),
                synth.Sample(29, 1, 10, 10, 0.5), synth.Sample(44, 1, 16, 16, 0.5),
                synth.Sample(100, 2, 16, 16, 0.5), synth.Sample(17, 1, 30, 40, 0.5)]


def _plan(samples):
    budget = sum(s.length for s in samples)
    ref = opack.build_plan(samples, budget)
    plan = mf.mf_pack(samples, budget)
    mf.mf_plan_upload(plan)
    return ref, plan


def _srow_of_joint(ref):
    s = np.empty(ref.n_tok, np.int64)
    s[ref.txt_joint] = np.arange(ref.n_txt)
    s[ref.img_joint] = ref.n_txt + np.arange(ref.n_img)
    return s


def _run(plan, ref, heads, D, q, k, v, do_joint):
    """GPU forward with lse, then the backward with do (given in joint order, passed
    stream-sorted as the ABI takes it).  Returns o (joint), lse, dq, dk, dv (joint) as float64."""
    N, H = ref.n_tok, heads * D
    srow = _srow_of_joint(ref)
    do_s = np.empty_like(do_joint)
    do_s[srow] = do_joint
    Q, K, V = to_bf16(q), to_bf16(k), to_bf16(v)
    o = torch.zeros((N, H), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((heads, N), dtype=torch.float32, device="cuda")
    mf.mf_attention_lse(plan, heads, D, Q, K, V, o, lse)
    ws = torch.empty(mf.mf_attention_backward_workspace_bytes(plan, heads, D), dtype=torch.uint8, device="cuda")
    dq, dk, dv = (torch.full((N, H), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(3))
    mf.mf_attention_backward(plan, heads, D, Q, K, V, o, lse, to_bf16(do_s), dq, dk, dv, ws)
    mf.mf_check()
    f = lambda t: t.double().cpu().numpy()          # noqa: E731
    return f(o)[srow], f(lse), f(dq), f(dk), f(dv)


@pytest.mark.parametrize("heads,D", [(2, 128), (4, 64)])
def test_attention_backward_ragged(heads, D):
    ref, plan = _plan(ATTN_SAMPLES)
    N, H = ref.n_tok, heads * D
    g = np.random.default_rng(31 + D)
    q, k, v, do = (synth.round_bf16(g.standard_normal((N, H)).astype(np.float32)) for _ in range(4))
    o, lse, dq, dk, dv = _run(plan, ref, heads, D, q, k, v, do)
    want = {n: np.zeros((N, H)) for n in ("dq", "dk", "dv")}
    for s in range(ref.n_seq):
        a, b = ref.cu_seqlens[s], ref.cu_seqlens[s + 1]
        r = lambda x: x[a:b].reshape(b - a, heads, D)          # noqa: E731
        wq, wk, wv = G.attention_vjp(r(q), r(k), r(v), r(do))
        want["dq"][a:b], want["dk"][a:b], want["dv"][a:b] = (x.reshape(b - a, H) for x in (wq, wk, wv))
        np.testing.assert_allclose(lse[:, a:b], G.attention_lse(r(q), r(k)), rtol=0, atol=2e-3,
                                   err_msg=f"lse sample {s} (len {b - a}, D {D})")
    got = {"dq": dq, "dk": dk, "dv": dv}
    for n in ("dq", "dk", "dv"):
        assert_close(got[n], want[n], f"{n} whole pack (D {D})")
        # per sample as well, except where the exact gradient vanishes (a one-token sample has
        # dq = dk = 0: P = 1 and ds = dP - delta = 0 exactly); there it must stay at rounding level
        scale = np.abs(want[n]).max()
        for s in range(ref.n_seq):
            a, b = ref.cu_seqlens[s], ref.cu_seqlens[s + 1]
            if np.abs(want[n][a:b]).max() > 1e-3 * scale:
                assert_close(got[n][a:b], want[n][a:b], f"{n} sample {s} (len {b - a}, D {D})")
            else:
                assert np.abs(got[n][a:b]).max() <= 1e-4 * scale, f"{n} sample {s} (len {b - a}): not ~0"


def test_attention_backward_16k_sequence():
    """One sample filling a 16384-token budget (128 x 128 latents, no text): 256 query tiles per
    key block; dq on sampled query rows and dk, dv on sampled key rows against the oracle's
    closed-form row gradients."""
    heads, D = 2, 128
    samples = [synth.Sample(0, 1, 128, 128, 0.5)]
    ref, plan = _plan(samples)
    N, H = ref.n_tok, heads * D
    g = np.random.default_rng(5)
    q, k, v, do = (synth.round_bf16(g.standard_normal((N, H)).astype(np.float32)) for _ in range(4))
    o, lse, dq, dk, dv = _run(plan, ref, heads, D, q, k, v, do)
    rows = np.unique(np.concatenate([g.choice(N, 24, replace=False), [0, 63, 64, 127, 128, N - 1]]))
    r = lambda x: x.reshape(N, heads, D)                       # noqa: E731
    wq, wk, wv = G.attention_vjp_rows(r(q), r(k), r(v), r(do), rows, rows)
    assert_close(dq[rows], wq.reshape(len(rows), H), "dq sampled rows")
    assert_close(dk[rows], wk.reshape(len(rows), H), "dk sampled rows")
    assert_close(dv[rows], wv.reshape(len(rows), H), "dv sampled rows")
    assert np.all(np.isfinite(dq)) and np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))
