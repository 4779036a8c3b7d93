"""Full-size oracle checks of the two 4-block configurations (H = 3072, 24 heads x 128,
C = 128): the editing pack (2 x (512 text + source and target 64 x 64 frames), 17408 tokens)
and the packed-CFG pack (cond and uncond branches of a 1024 x 1024 and a 768 x 1344 prompt,
16768 tokens, first Euler step from t = 1 with w = 4).

The GPU runs embed -> 4 blocks -> final layer (-> CFG combine -> Euler step) and every stage
is compared with the oracle applied to the GPU's own input to that stage: the latent embed and
the final layer on every row, each of the four blocks on sampled rows of every sample (the
oracle computes each sample's keys and values in full and the queried rows only), the guided
velocity and the Euler step on every row.  Together with the packed == separate check of
test_gpu_30_fullsize this covers each computation of the stacked configurations at full size.
The oracle work (float64 NumPy on the host) takes a few minutes."""
import numpy as np
import pytest

import synth
from oracle import model as M
from oracle import pack as opack
from tests.helpers import assert_close

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

if torch.cuda.is_available():
    import packed_rectified_flow_packer_b300 as mf
    from packed_rectified_flow_packer_b300.device import DeviceModel, Workspace, to_bf16, to_f32

D = synth.FULL


@pytest.fixture(scope="module")
def model4():
    w = synth.model_weights(D, 4, seed=1)
    return w, DeviceModel(w)


def _rows(L_txt, L_img, seed, n=6):
    g = np.random.default_rng(seed)
    L = L_txt + L_img
    rows = {0, L_txt, L - 1}
    if L_txt:
        rows.add(L_txt - 1)
    rows |= set(g.integers(0, L, size=n).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < L))


def _stack_stages(samples, budget, w, model, x_txt, zt_f32, t):
    """Runs the stack on the GPU and returns the host copy of every stage's input and output."""
    ref = opack.build_plan(samples, budget)
    plan = mf.mf_pack(samples, budget)
    mf.mf_plan_upload(plan)
    ws = Workspace(plan, model.dims)
    d = model.dims
    ztb = to_bf16(synth.round_bf16(zt_f32))
    xt = to_bf16(x_txt if len(x_txt) else np.zeros((1, D.hidden), np.float32))
    xi = torch.empty((ref.n_img, D.hidden), dtype=torch.bfloat16, device="cuda")
    tt = torch.tensor([samples[c].t for c in ref.order] if t is None else [t] * ref.n_seq,
                      dtype=torch.float32, device="cuda")
    mf.mf_embed(plan, d, model.embed["w_in"], model.embed["b_in"], ztb, xi)
    f = lambda a: a.double().cpu().numpy()                   # noqa: E731
    stages = {"zt": f(ztb), "embed": f(xi), "blocks": []}
    for bs in model.block_structs:
        before = (f(xt)[:ref.n_txt], f(xi))
        mf.mf_block_forward(plan, d, bs, tt, xt, xi, ws.block)
        stages["blocks"].append((before, (f(xt)[:ref.n_txt], f(xi))))
    v = torch.empty((ref.n_img, D.channels), dtype=torch.float32, device="cuda")
    fm = model.final
    mf.mf_final(plan, d, model.temb_struct, fm["w_fmod"], fm["b_fmod"], fm["w_out"], fm["b_out"], tt, xi, v,
                ws.final)
    mf.mf_check()
    stages["v"] = f(v)
    return ref, plan, stages, v


def _check_stages(samples, ref, stages, w, t=None):
    H = D.hidden
    assert_close(stages["embed"], M.embed(stages["zt"], w.embed), "latent embed (all rows)")
    for b, ((xt_in, xi_in), (xt_out, xi_out)) in enumerate(stages["blocks"]):
        for k, c in enumerate(ref.order):
            s = samples[c]
            tk = s.t if t is None else t
            cond = M.condition(np.float32(tk), w.temb, D.freq_dim)
            ta, tb = ref.cu_txt[k], ref.cu_txt[k + 1]
            a, bb = ref.cu_img[k], ref.cu_img[k + 1]
            pos = M.image_positions(s.frames, s.lat_h, s.lat_w)
            rows = _rows(s.txt_len, s.img_len, seed=100 * b + k)
            want = M.block_forward(xt_in[ta:tb], xi_in[a:bb], pos, cond, w.blocks[b], D.heads, rows=rows)
            got = np.concatenate([xt_out[ta:tb], xi_out[a:bb]])[rows] if s.txt_len else xi_out[a:bb][rows]
            assert_close(got, want, f"block {b} rows, sample {k} ({s.txt_len} text, {s.frames} frames)")
    # final layer on every image row, from the GPU's output of the last block
    xi_last = stages["blocks"][-1][1][1]
    want_v = np.zeros((ref.n_img, D.channels))
    for k, c in enumerate(ref.order):
        s = samples[c]
        cond = M.condition(np.float32(s.t if t is None else t), w.temb, D.freq_dim)
        a, bb = ref.cu_img[k], ref.cu_img[k + 1]
        want_v[a:bb] = M.final_layer(xi_last[a:bb], cond, w.final)
    assert_close(stages["v"], want_v, "final layer velocity (all rows)")
    assert H == w.dims.hidden


def test_edit_pack_every_stage(model4):
    """Editing pack: 3-axis RoPE (frame, row, col), clean source frame, all four blocks."""
    w, model = model4
    samples = synth.edit_samples()
    ref0 = opack.build_plan(samples, 17408)
    x, z, e = synth.pack_inputs(samples, ref0.order, D, seed=4)
    # z_t with the source frame clean, as mf_interpolate forms it (checked elsewhere)
    zt = np.concatenate([M.interpolate(z[ref0.cu_img[k]:ref0.cu_img[k + 1]], e[ref0.cu_img[k]:ref0.cu_img[k + 1]],
                                       samples[c].t, M.target_mask(samples[c]))
                         for k, c in enumerate(ref0.order)])
    ref, plan, stages, _ = _stack_stages(samples, 17408, w, model, x, zt, None)
    _check_stages(samples, ref, stages, w)


def test_cfg_pack_every_stage_and_euler_step(model4):
    """Packed CFG: both branches of both prompts through all four blocks at t = 1, then the
    guided velocity v_u + 4 (v_c - v_u) and one Euler step of dt = 0.25 on every row."""
    w, model = model4
    samples = synth.cfg_samples()
    C, H = D.channels, D.hidden
    budget = sum(s.length for s in samples)
    ref0 = opack.build_plan(samples, budget)
    x = np.concatenate([synth.round_bf16(synth.normal(6, f"x_txt.{c}", (samples[c].txt_len, H)))
                        for c in ref0.order if samples[c].txt_len])
    z0 = np.concatenate([synth.round_bf16(synth.normal(6, f"z0.p{c // 2}", (samples[c].img_len, C)))
                         for c in ref0.order])
    ref, plan, stages, v = _stack_stages(samples, budget, w, model, x, z0, 1.0)
    _check_stages(samples, ref, stages, w, t=1.0)
    vg = torch.empty_like(v)
    mf.mf_cfg_combine(plan, C, 4.0, v, vg)
    z = to_f32(z0)
    mf.mf_euler_step(plan, C, 0.25, vg, z, None)
    mf.mf_check()
    vh, vgh, zh = stages["v"], vg.double().cpu().numpy(), z.double().cpu().numpy()
    order = list(ref.order)
    for c in (0, 2):                                   # cond c, uncond c + 1
        k, ku = order.index(c), order.index(c + 1)
        rc, ru = slice(ref.cu_img[k], ref.cu_img[k + 1]), slice(ref.cu_img[ku], ref.cu_img[ku + 1])
        want = M.cfg_combine(vh[rc], vh[ru], 4.0)
        assert_close(vgh[rc], want, f"guided velocity, prompt {c // 2} (cond rows)")
        assert_close(vgh[ru], want, f"guided velocity, prompt {c // 2} (uncond rows)")
        assert_close(zh[rc], M.euler_step(z0[rc], want, 0.25), f"Euler step, prompt {c // 2}")
        np.testing.assert_array_equal(zh[rc], zh[ru])
