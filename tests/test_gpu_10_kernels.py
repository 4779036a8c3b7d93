"""GPU parity of the library's building blocks through the C ABI: the bounded-wait status
path, the tcgen05 GEMM, varlen attention and the rectified-flow epilogues, each against the
oracle (or, for the plain GEMM, an fp64 matmul of the same bf16 operands)."""
import numpy as np
import pytest

import synth
from oracle import model as M
from oracle import pack as opack
from tests.helpers import assert_close, stats

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import packed_rectified_flow_packer_b300 as mf
    from packed_rectified_flow_packer_b300.device import to_bf16, to_f32


def _bf16_np(t):
    return t.float().cpu().numpy()


def test_bounded_wait_reports_timeout():
    """A wait that nothing completes gives up after its limit and reports a status; the
    context stays usable afterwards."""
    st = mf.mf_selftest_timeout(2000)
    assert mf.STATUS[st] == "MF_ERR_DEVICE_TIMEOUT"
    mf.mf_check()                                  # status word is clean again
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum()) == 8.0


# the last two give 78 and 75 tiles of 256 x 256: more than one wave on 74 co-resident CTA
# pairs, with a nearly empty last wave (in the second, N = 640 ends inside the last tile)
GEMM_SHAPES = [(1, 64, 64), (100, 128, 64), (128, 256, 128), (129, 384, 256), (300, 512, 1024),
               (1000, 96, 192), (257, 256, 3072), (6656, 768, 256), (6400, 640, 128)]


@pytest.mark.parametrize("M_,N_,K_", GEMM_SHAPES)
@pytest.mark.parametrize("out_f32", [False, True])
def test_gemm(M_, N_, K_, out_f32):
    g = np.random.default_rng(M_ * 7 + N_ + K_)
    a = synth.round_bf16(g.standard_normal((M_, K_)).astype(np.float32))
    b = synth.round_bf16((g.standard_normal((N_, K_)) * 0.05).astype(np.float32))
    bias = synth.round_bf16(g.standard_normal(N_).astype(np.float32))
    ref = a.astype(np.float64) @ b.astype(np.float64).T + bias
    A, Bm, bb = to_bf16(a), to_bf16(b), to_bf16(bias)
    c = torch.zeros((M_, N_), dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    mf.mf_gemm(A, Bm, c, bias=bb, out_f32=out_f32)
    mf.mf_check()
    got = c.float().cpu().numpy()
    s = stats(got, ref)
    assert s["rel"] <= (1e-4 if out_f32 else 8e-3) and s["cos"] >= 0.99999, s


def _attn_plan(samples):
    ref = opack.build_plan(samples, sum(s.length for s in samples))
    plan = mf.mf_pack(samples, sum(s.length for s in samples))
    mf.mf_plan_upload(plan)
    return ref, plan


ATTN_SAMPLES = [synth.Sample(3, 1, 1, 2, 0.5), synth.Sample(0, 1, 1, 1, 0.5),
                synth.Sample(27, 1, 10, 10, 0.5), synth.Sample(28, 1, 10, 10, 0.5),
                synth.Sample(29, 1, 10, 10, 0.5), synth.Sample(44, 1, 16, 16, 0.5),
                synth.Sample(100, 2, 16, 16, 0.5), synth.Sample(17, 1, 30, 40, 0.5)]


@pytest.mark.parametrize("heads,D", [(2, 128), (4, 64)])
@pytest.mark.parametrize("growth", [0.0, 6.0])
def test_attention_ragged(heads, D, growth):
    """Ragged samples (1 .. 1217 tokens, tile tails on both sides of 128 and 256).  `growth` scales the
    keys up along each sample so later key tiles raise the running max by large steps (the
    rescaling path)."""
    ref, plan = _attn_plan(ATTN_SAMPLES)
    N, H = ref.n_tok, heads * D
    g = np.random.default_rng(heads + int(growth))
    q = synth.round_bf16(g.standard_normal((N, H)).astype(np.float32))
    k = g.standard_normal((N, H)).astype(np.float32)
    if growth:
        for s in range(ref.n_seq):
            a, b = ref.cu_seqlens[s], ref.cu_seqlens[s + 1]
            k[a:b] *= (1.0 + growth * np.arange(b - a) / max(1, b - a))[:, None]
    k = synth.round_bf16(k)
    v = synth.round_bf16(g.standard_normal((N, H)).astype(np.float32))
    o = torch.zeros((N, H), dtype=torch.bfloat16, device="cuda")
    mf.mf_attention(plan, heads, D, to_bf16(q), to_bf16(k), to_bf16(v), o)
    mf.mf_check()
    got = _bf16_np(o)
    # oracle, one sample at a time, mapped to stream-sorted rows
    want = np.zeros((N, H))
    srow_of_joint = np.empty(N, np.int64)
    srow_of_joint[ref.txt_joint] = np.arange(ref.n_txt)
    srow_of_joint[ref.img_joint] = ref.n_txt + np.arange(ref.n_img)
    for s in range(ref.n_seq):
        a, b = ref.cu_seqlens[s], ref.cu_seqlens[s + 1]
        os_ = M.attention(q[a:b].reshape(-1, heads, D), k[a:b].reshape(-1, heads, D),
                          v[a:b].reshape(-1, heads, D)).reshape(-1, H)
        want[srow_of_joint[a:b]] = os_
    for s in range(ref.n_seq):
        a, b = ref.cu_seqlens[s], ref.cu_seqlens[s + 1]
        rows = srow_of_joint[a:b]
        assert_close(got[rows], want[rows], f"attention sample {s} (len {b - a})")


def _latent_case():
    samples = [synth.Sample(5, 1, 3, 4, 0.3, 1, 1), synth.Sample(0, 1, 3, 4, 0.3, 2, 0),
               synth.Sample(7, 2, 2, 5, 0.8), synth.Sample(2, 1, 6, 1, 0.55)]
    budget = sum(s.length for s in samples)
    ref = opack.build_plan(samples, budget)
    plan = mf.mf_pack(samples, budget)
    mf.mf_plan_upload(plan)
    return samples, ref, plan


@pytest.mark.parametrize("C", [64, 128])
def test_rectified_flow_epilogues(C):
    samples, ref, plan = _latent_case()
    Ni = ref.n_img
    g = np.random.default_rng(C)
    z, e, v = (g.standard_normal((Ni, C)).astype(np.float32) for _ in range(3))
    Z, E, V = to_f32(z), to_f32(e), to_f32(v)
    # interpolation (edit source rows stay clean)
    zt = torch.zeros((Ni, C), device="cuda")
    ztb = torch.zeros((Ni, C), dtype=torch.bfloat16, device="cuda")
    mf.mf_interpolate(plan, C, None, Z, E, zt, ztb)
    # Euler step in place
    zz = Z.clone()
    mf.mf_euler_step(plan, C, 0.25, V, zz)
    # packed CFG
    vo = torch.zeros((Ni, C), device="cuda")
    mf.mf_cfg_combine(plan, C, 4.0, V, vo)
    vin = V.clone()
    mf.mf_cfg_combine(plan, C, 4.0, vin, vin)     # in place
    # loss
    ls = torch.zeros(ref.n_seq, dtype=torch.float64, device="cuda")
    cnt = torch.zeros(ref.n_seq, dtype=torch.int64, device="cuda")
    mean = torch.zeros(1, dtype=torch.float64, device="cuda")
    ws = torch.empty(mf.mf_flow_loss_workspace_bytes(plan), dtype=torch.uint8, device="cuda")
    mf.mf_flow_loss(plan, C, Z, E, V, ls, cnt, mean, ws)
    mf.mf_check()

    want_zt, want_cfg, sums, counts = [], np.array(v, np.float64), [], []
    for k, cidx in enumerate(ref.order):
        s = samples[cidx]
        a, b = ref.cu_img[k], ref.cu_img[k + 1]
        tgt = M.target_mask(s)
        want_zt.append(M.interpolate(z[a:b], e[a:b], np.float32(s.t), tgt))
        sm, n = M.flow_loss(v[a:b], z[a:b], e[a:b], tgt)
        sums.append(sm)
        counts.append(n)
        if s.cfg_role == 1:
            pk = list(ref.order).index(s.cfg_pair)
            pa, pb = ref.cu_img[pk], ref.cu_img[pk + 1]
            gv = M.cfg_combine(v[a:b], v[pa:pb], 4.0)
            want_cfg[a:b] = gv
            want_cfg[pa:pb] = gv
    np.testing.assert_allclose(zt.cpu().numpy(), np.concatenate(want_zt), rtol=1e-6, atol=1e-6)
    np.testing.assert_array_equal(ztb.float().cpu().numpy(),
                                  synth.round_bf16(zt.cpu().numpy()))
    np.testing.assert_allclose(zz.cpu().numpy(), M.euler_step(z, v, 0.25), rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(vo.cpu().numpy(), want_cfg, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(vin.cpu().numpy(), want_cfg, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(ls.cpu().numpy(), sums, rtol=1e-12)
    np.testing.assert_array_equal(cnt.cpu().numpy(), counts)
    assert abs(mean.item() - M.mean_loss(sums, counts)) <= 1e-12 * abs(M.mean_loss(sums, counts))
    # deterministic: a second run gives the same bits
    ls2 = torch.zeros_like(ls)
    mf.mf_flow_loss(plan, C, Z, E, V, ls2, cnt, mean, ws)
    assert torch.equal(ls, ls2)


@pytest.mark.parametrize("case", ["mixed", "native16k"])
def test_nft_loss(case):
    """Diffusion-NFT objective against the oracle, per sample: edit source frames excluded,
    rewards at the endpoints 0 and 1 and inside; sums to 1e-12 relative, counts exact."""
    if case == "mixed":
        samples, ref, plan = _latent_case()
        C = 64
    else:
        samples = synth.native_candidates(0)
        ref = opack.build_plan(samples, 16384)
        plan = mf.mf_pack(samples, 16384)
        mf.mf_plan_upload(plan)
        C = 128
    Ni, S = ref.n_img, ref.n_seq
    g = np.random.default_rng(11 + C)
    z, e, vp, vn = (g.standard_normal((Ni, C)).astype(np.float32) for _ in range(4))
    r = g.uniform(0.0, 1.0, S).astype(np.float32)
    r[0] = 1.0
    if S > 1:
        r[1] = 0.0
    ls = torch.zeros(S, dtype=torch.float64, device="cuda")
    cnt = torch.zeros(S, dtype=torch.int64, device="cuda")
    mean = torch.zeros(1, dtype=torch.float64, device="cuda")
    ws = torch.empty(mf.mf_flow_loss_workspace_bytes(plan), dtype=torch.uint8, device="cuda")
    mf.mf_nft_loss(plan, C, to_f32(z), to_f32(e), to_f32(vp), to_f32(vn), to_f32(r), ls, cnt, mean, ws)
    mf.mf_check()
    sums, counts = [], []
    for k, cidx in enumerate(ref.order):
        a, b = ref.cu_img[k], ref.cu_img[k + 1]
        sm, n = M.nft_loss(vp[a:b], vn[a:b], z[a:b], e[a:b], float(r[k]), M.target_mask(samples[cidx]))
        sums.append(sm)
        counts.append(n)
    np.testing.assert_allclose(ls.cpu().numpy(), sums, rtol=1e-12)
    np.testing.assert_array_equal(cnt.cpu().numpy(), counts)
    want = M.mean_loss(sums, counts)
    assert abs(mean.item() - want) <= 1e-12 * abs(want)


# ------------------------------------------------------------------ fp8 variant
@pytest.mark.parametrize("M_,K_", [(1, 16), (300, 1024), (77, 3072)])
def test_quantize_fp8_rows(M_, K_):
    """Per-row E4M3 quantisation: scales and codes equal the oracle's exactly (codes compared
    as values, so -0 and +0 agree), with an all-zero row, a row of huge and a row of tiny
    values."""
    from oracle import fp8 as F
    g = np.random.default_rng(M_ + K_)
    x = synth.round_bf16(g.normal(0, 2, (M_, K_)).astype(np.float32))
    if M_ > 3:
        x[1] = 0.0
        x[2] = synth.round_bf16(x[2] * 1e3)
        x[3] = synth.round_bf16(x[3] * 1e-4)
    xd = to_bf16(x)
    q = torch.empty((M_, K_), dtype=torch.uint8, device="cuda")
    s = torch.empty(M_, dtype=torch.float32, device="cuda")
    mf.mf_quantize_fp8_rows(xd, q, s)
    mf.mf_check()
    codes, scale = F.quantize_rows(x)
    np.testing.assert_array_equal(s.cpu().numpy(), scale)
    np.testing.assert_array_equal(F.e4m3_decode(q.cpu().numpy()), F.e4m3_decode(codes))


@pytest.mark.parametrize("M_,N_,K_,with_bias", [(1, 256, 128, False), (257, 384, 512, True),
                                                (1000, 512, 1024, True), (300, 3072, 3072, True)])
def test_gemm_fp8(M_, N_, K_, with_bias):
    """E4M3 GEMM (kind::f8f6f4 on CTA pairs) against the oracle's fp64 product of the same codes
    and scales.  N = 384 takes the staged epilogue (no 64-column TMA store boxes), the others the
    TMA-store one; M = 1 and 257 leave ragged row tiles."""
    from oracle import fp8 as F
    g = np.random.default_rng(M_ * 7 + N_)
    a, sa = F.quantize_rows(synth.round_bf16(g.normal(0, 1, (M_, K_)).astype(np.float32)))
    b, sb = F.quantize_rows(synth.round_bf16(g.normal(0, 0.02, (N_, K_)).astype(np.float32)))
    bias = synth.round_bf16(g.normal(0, 0.1, N_).astype(np.float32)) if with_bias else None
    c = torch.empty((M_, N_), dtype=torch.bfloat16, device="cuda")
    mf.mf_gemm_fp8(torch.from_numpy(a).cuda(), torch.from_numpy(sa).cuda(), torch.from_numpy(b).cuda(),
                   torch.from_numpy(sb).cuda(), c, None if bias is None else to_bf16(bias))
    mf.mf_check()
    ref = F.linear_fp8(a, sa, b, sb, bias)
    got = _bf16_np(c).astype(np.float64)
    assert_close(got, ref, "fp8 gemm")
    bound = 2.0 ** -8 * np.abs(ref) + 1e-3 * np.abs(ref).max()   # one bf16 rounding + f32 sums
    assert np.all(np.abs(got - ref) <= bound)
