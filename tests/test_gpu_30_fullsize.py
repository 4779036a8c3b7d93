"""Full-size GPU checks (H=3072, 24 heads x 128, C=128) in the launch configuration the bench
times.  Where the oracle cannot run the whole configuration in seconds it computes sampled
output rows one by one (keys and values of the whole sample, queries and the row-local rest
only for the sampled rows); the stacked configurations are checked through properties that hold
at any size (packed == unpacked, CFG branches stay tied, loss counts)."""
import numpy as np
import pytest

import synth
from oracle import model as M
from oracle import pack as opack
from tests.helpers import assert_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import packed_rectified_flow_packer_b300 as mf
    from packed_rectified_flow_packer_b300.device import DeviceModel, Workspace, run_stack, to_bf16, to_f32

D = synth.FULL


@pytest.fixture(scope="module")
def model1():
    w = synth.model_weights(D, 1, seed=0)
    return w, DeviceModel(w)


def _run(samples, budget, w, model, seed, t=None, interpolate=True, inputs=None):
    """Pack, then interpolate -> embed -> blocks -> final -> loss on the GPU.  `inputs`
    (x_txt, z, eps in stream order) overrides the seeded draw."""
    ref = opack.build_plan(samples, budget)
    plan = mf.mf_pack(samples, budget)
    mf.mf_plan_upload(plan)
    x, z, e = inputs if inputs is not None else synth.pack_inputs(samples, ref.order, D, seed)
    ws = Workspace(plan, model.dims)
    Z, E = to_f32(z), to_f32(e)
    ztb = torch.empty((ref.n_img, D.channels), dtype=torch.bfloat16, device="cuda")
    if interpolate:
        mf.mf_interpolate(plan, D.channels, t, Z, E, None, ztb)
    else:
        ztb.copy_(Z)
    x_txt = to_bf16(x)
    x_img = torch.empty((ref.n_img, D.hidden), dtype=torch.bfloat16, device="cuda")
    v = torch.empty((ref.n_img, D.channels), dtype=torch.float32, device="cuda")
    run_stack(plan, model, x_txt, ztb, x_img, v, ws, t=t)
    ls = torch.zeros(ref.n_seq, dtype=torch.float64, device="cuda")
    cnt = torch.zeros(ref.n_seq, dtype=torch.int64, device="cuda")
    mean = torch.zeros(1, dtype=torch.float64, device="cuda")
    mf.mf_flow_loss(plan, D.channels, Z, E, v, ls, cnt, mean, ws.loss)
    mf.mf_check()
    return {"ref": ref, "x": x, "z": z, "e": e, "v": v.cpu().numpy().astype(np.float64),
            "x_img": x_img.float().cpu().numpy(), "x_txt": x_txt.float().cpu().numpy(),
            "ztb": ztb.float().cpu().numpy(), "loss": ls.cpu().numpy(), "count": cnt.cpu().numpy(),
            "mean": mean.item()}


def _sampled_rows(L_txt, L_img, n=12, seed=0):
    g = np.random.default_rng(seed)
    L = L_txt + L_img
    rows = {0, L_txt - 1 if L_txt else 0, L_txt, L - 1, L_txt + 127, L_txt + 128}
    rows |= set(g.integers(0, L, size=n).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < L))


def _check_sampled(samples, out, w, seed=0):
    """Oracle on sampled rows of every packed sample of a 1-block stack: the block output and
    the velocity v (image rows)."""
    assert len(w.blocks) == 1
    ref = out["ref"]
    for k, c in enumerate(ref.order):
        s = samples[c]
        a, b = ref.cu_img[k], ref.cu_img[k + 1]
        ta, tb = ref.cu_txt[k], ref.cu_txt[k + 1]
        zt = out["ztb"][a:b]                                    # the GPU's bf16 model input
        cond = M.condition(np.float32(s.t), w.temb, D.freq_dim)
        xi = M.embed(zt, w.embed)
        pos = M.image_positions(s.frames, s.lat_h, s.lat_w)
        rows = _sampled_rows(s.txt_len, s.img_len, seed=seed + k)
        got = M.block_forward(out["x"][ta:tb], xi, pos, cond, w.blocks[0], D.heads, rows=rows)
        lt = s.txt_len
        gpu_rows = np.concatenate([out["x_txt"][ta:tb], out["x_img"][a:b]])[rows]
        assert_close(gpu_rows, got, f"block output rows, sample {k}")
        img_sel = rows[rows >= lt]
        vr = M.final_layer(got[rows >= lt], cond, w.final)
        assert_close(out["v"][a:b][img_sel - lt], vr, f"velocity rows, sample {k}")


def test_gen1024_sampled_rows(model1):
    """1024^2 generation pack: 256 text + 64x64 latent tokens, t = 0.5."""
    w, model = model1
    samples = synth.gen1024_samples()
    out = _run(samples, 4352, w, model, seed=3, interpolate=False)
    _check_sampled(samples, out, w)


def test_native_pack_sampled_rows_and_loss(model1):
    """16384-token native-resolution pack (seed 0): sampled rows of every sample, and the
    loss of the whole pack recomputed in fp64 from the GPU's own velocity."""
    w, model = model1
    cands = synth.native_candidates(0)
    out = _run(cands, 16384, w, model, seed=0)
    ref = out["ref"]
    assert ref.n_tok <= 16384
    _check_sampled(cands, out, w)
    for k, c in enumerate(ref.order):
        a, b = ref.cu_img[k], ref.cu_img[k + 1]
        sm, n = M.flow_loss(out["v"][a:b], out["z"][a:b], out["e"][a:b], M.target_mask(cands[c]))
        assert out["count"][k] == n
        assert abs(out["loss"][k] - sm) <= 1e-9 * sm
    assert abs(out["mean"] - M.mean_loss(out["loss"], out["count"])) <= 1e-12 * out["mean"]


@pytest.fixture(scope="module")
def model4():
    w = synth.model_weights(D, 4, seed=1)
    return w, DeviceModel(w)


def test_edit_pack_full(model4):
    """Editing pack, 2 x (512 text + source frame + target frame at 64x64) = 17408 tokens, 4
    blocks: packed result equals each sample run alone; loss counts only target frames; and a
    1-block sampled-row oracle check pins the 3-axis RoPE at full size."""
    w, model = model4
    samples = synth.edit_samples()
    out = _run(samples, 17408, w, model, seed=4)
    assert out["ref"].n_tok == 17408
    assert list(out["count"]) == [4096 * D.channels, 4096 * D.channels]
    ref = out["ref"]
    for k in range(2):
        a, b = ref.cu_img[k], ref.cu_img[k + 1]
        ta, tb = ref.cu_txt[k], ref.cu_txt[k + 1]
        alone = _run([samples[k]], samples[k].length, w, model, seed=4,
                     inputs=(out["x"][ta:tb], out["z"][a:b], out["e"][a:b]))
        np.testing.assert_allclose(alone["v"], out["v"][a:b], rtol=0, atol=1e-5 * np.abs(alone["v"]).max())
        assert alone["loss"][0] == pytest.approx(out["loss"][k], rel=1e-9)
    # one block, sampled rows, against the oracle
    w1 = synth.ModelWeights(D, w.temb, w.embed, w.blocks[:1], w.final, True)
    m1 = DeviceModel(w1)
    out1 = _run(samples, 17408, w1, m1, seed=4)
    _check_sampled(samples, out1, w1)


def test_cfg_pack_full(model4):
    """Packed CFG sampler at full size (4 blocks, 4 Euler steps, w = 4): the two branches of a
    prompt stay identical, and the packed run equals the cond-only and uncond-only packs run
    separately (the pages: packing the branches does not change the trajectory)."""
    w, model = model4
    samples = synth.cfg_samples()
    C, H = D.channels, D.hidden
    grid = [1.0, 0.75, 0.5, 0.25, 0.0]

    def sampler(cands, pairs_packed):
        ref = opack.build_plan(cands, sum(s.length for s in cands))
        plan = mf.mf_pack(cands, ref.n_tok)
        mf.mf_plan_upload(plan)
        ws = Workspace(plan, model.dims)
        x = np.concatenate([synth.round_bf16(synth.normal(5, f"x_txt.p{c // 2}", (cands[c].txt_len, H)))
                            for c in ref.order]) if ref.n_txt else np.zeros((0, H), np.float32)
        z0 = np.concatenate([synth.round_bf16(synth.normal(5, f"z0.p{pairs_packed[c]}",
                                                           (cands[c].img_len, C))) for c in ref.order])
        z = to_f32(z0)
        zb = z.to(torch.bfloat16)
        x_img = torch.empty((ref.n_img, H), dtype=torch.bfloat16, device="cuda")
        v = torch.empty((ref.n_img, C), dtype=torch.float32, device="cuda")
        vs = torch.empty_like(v)
        tt = torch.empty(ref.n_seq, dtype=torch.float32, device="cuda")
        for a, b in zip(grid[:-1], grid[1:]):
            tt.fill_(a)
            run_stack(plan, model, to_bf16(x), zb, x_img, v, ws, t=tt)
            mf.mf_cfg_combine(plan, C, 4.0, v, vs)
            mf.mf_euler_step(plan, C, a - b, vs, z, zb)
        mf.mf_check()
        return ref, z.cpu().numpy(), v.cpu().numpy()

    ref, zp, vp = sampler(samples, {0: 0, 1: 0, 2: 1, 3: 1})
    for c in (0, 2):
        k, kp = list(ref.order).index(c), list(ref.order).index(c + 1)
        np.testing.assert_array_equal(zp[ref.cu_img[k]:ref.cu_img[k + 1]],
                                      zp[ref.cu_img[kp]:ref.cu_img[kp + 1]])
    # the same sampler with the branches in separate packs: combine on the host
    cond = [synth.Sample(256, 1, 64, 64, 1.0), synth.Sample(256, 1, 48, 84, 1.0)]
    unc = [synth.Sample(0, 1, 64, 64, 1.0), synth.Sample(0, 1, 48, 84, 1.0)]
    rc = opack.build_plan(cond, 10**6)
    pc = mf.mf_pack(cond, 10**6)
    pu = mf.mf_pack(unc, 10**6)
    mf.mf_plan_upload(pc)
    mf.mf_plan_upload(pu)
    wsc, wsu = Workspace(pc, model.dims), Workspace(pu, model.dims)
    xc = np.concatenate([synth.round_bf16(synth.normal(5, f"x_txt.p{i}", (256, H))) for i in range(2)])
    z0 = np.concatenate([synth.round_bf16(synth.normal(5, f"z0.p{i}", (cond[i].img_len, C))) for i in range(2)])
    z = to_f32(z0)
    zb = z.to(torch.bfloat16)
    xi = torch.empty((rc.n_img, H), dtype=torch.bfloat16, device="cuda")
    vc = torch.empty((rc.n_img, C), dtype=torch.float32, device="cuda")
    vu = torch.empty_like(vc)
    tt = torch.empty(2, dtype=torch.float32, device="cuda")
    for a, b in zip(grid[:-1], grid[1:]):
        tt.fill_(a)
        run_stack(pc, model, to_bf16(xc), zb, xi, vc, wsc, t=tt)
        run_stack(pu, model, torch.empty((0, H), dtype=torch.bfloat16, device="cuda"), zb, xi, vu, wsu, t=tt)
        g = vu + 4.0 * (vc - vu)
        mf.mf_euler_step(pc, C, a - b, g, z, zb)
    mf.mf_check()
    zs = z.cpu().numpy()
    for i, c in enumerate((0, 2)):
        k = list(ref.order).index(c)
        got = zp[ref.cu_img[k]:ref.cu_img[k + 1]]
        want = zs[rc.cu_img[i]:rc.cu_img[i + 1]]
        assert_close(got, want, f"packed vs separate CFG, prompt {i}", rel=1e-3, cos=0.999999)
