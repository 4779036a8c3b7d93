"""GPU parity of the packed block forward and the stack paths through the C ABI, against the
fp64 oracle run one sample at a time (so every check is also a packed == unpacked check)."""
import numpy as np
import pytest

import synth
from oracle import model as M
from oracle import pack as opack
from tests.helpers import assert_close, assert_update_close, oracle_stack, stream_concat

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import packed_rectified_flow_packer_b300 as mf
    from packed_rectified_flow_packer_b300.device import (DeviceModel, Workspace, run_stack, to_bf16,
                                                          to_f32)


def _f(t):
    return t.float().cpu().numpy().astype(np.float64)


class Case:
    def __init__(self, samples, dims, n_blocks, seed, budget=None, qk_norm=False, rounded=True):
        self.samples, self.dims = samples, dims
        self.budget = budget or sum(s.length for s in samples)
        # rounded=False keeps the fp32 originals (the device copies still round to bf16)
        self.w = synth.model_weights(dims, n_blocks, seed, qk_norm=qk_norm, bf16=rounded)
        self.batch = synth.batch_inputs(samples, dims, seed, bf16=rounded)
        self.ref = opack.build_plan(samples, self.budget)
        self.plan = mf.mf_pack(samples, self.budget)
        mf.mf_plan_upload(self.plan)
        self.model = DeviceModel(self.w)
        self.ws = Workspace(self.plan, self.model.dims)
        H, C = dims.hidden, dims.channels
        self.x_txt_np = stream_concat(self.batch.x_txt, self.ref.order, H)
        self.z_np = stream_concat(self.batch.z, self.ref.order, C)
        self.eps_np = stream_concat(self.batch.eps, self.ref.order, C)
        self.t_np = np.array([samples[c].t for c in self.ref.order], np.float32)


def _block_intermediates(case, x_txt, x_img, k):
    """Oracle intermediates of block 0 for packed sample k (joint order inside the sample)."""
    s = case.samples[case.ref.order[k]]
    d, bw = case.dims, case.w.blocks[0]
    H, nh = d.hidden, d.heads
    c = M.condition(s.t, case.w.temb, d.freq_dim)
    mods = {st: M.modulation(c, bw[st]["w_mod"], bw[st]["b_mod"], 6) for st in M.STREAMS}
    xt = x_txt[case.ref.cu_txt[k]:case.ref.cu_txt[k + 1]]
    xi = x_img[case.ref.cu_img[k]:case.ref.cu_img[k + 1]]
    a = {"txt": M.modulate(xt, mods["txt"][0], mods["txt"][1]),
         "img": M.modulate(xi, mods["img"][0], mods["img"][1])}
    qkv = np.concatenate([M.linear(a[st], bw[st]["w_qkv"], bw[st]["b_qkv"]) for st in M.STREAMS])
    L = len(qkv)
    pos = np.concatenate([np.zeros((len(xt), 3), np.int64), M.image_positions(s.frames, s.lat_h, s.lat_w)])
    q = M.apply_rope(qkv[:, :H].reshape(L, nh, -1), pos).reshape(L, H)
    kk = M.apply_rope(qkv[:, H:2 * H].reshape(L, nh, -1), pos).reshape(L, H)
    v = qkv[:, 2 * H:]
    o = M.attention(q.reshape(L, nh, -1), kk.reshape(L, nh, -1), v.reshape(L, nh, -1)).reshape(L, H)
    return {"c": c, "mod_txt": np.concatenate(mods["txt"]), "mod_img": np.concatenate(mods["img"]),
            "q": q, "k": kk, "v": v, "o": o}


def test_tiny_block_and_intermediates():
    """The tiny configuration (H=256, 4 heads x 64, two samples 16+8x8 and 16+4x12): the
    block alone on the GPU's own embed output, and every intermediate the call leaves."""
    d = synth.TINY
    case = Case(synth.tiny_samples(), d, 1, seed=0)
    ref, H, C = case.ref, d.hidden, d.channels
    x_txt = to_bf16(case.x_txt_np)
    x_img = torch.empty((ref.n_img, H), dtype=torch.bfloat16, device="cuda")
    mf.mf_embed(case.plan, case.model.dims, case.model.embed["w_in"], case.model.embed["b_in"],
                to_bf16(case.z_np), x_img)
    mf.mf_check()
    emb = _f(x_img)
    assert_close(emb, M.embed(case.z_np, case.w.embed), "embed")
    x_txt0 = _f(x_txt)
    mf.mf_block_forward(case.plan, case.model.dims, case.model.block_structs[0], None, x_txt, x_img,
                        case.ws.block)
    mf.mf_check()
    # intermediates left in the workspace
    off = mf.mf_block_workspace_layout(case.plan, case.model.dims)
    wsb = case.ws.block
    S, N = ref.n_seq, ref.n_tok
    view = lambda i, n, dt: wsb[off[i]:off[i] + n * (4 if dt == torch.float32 else 2)].view(dt)  # noqa: E731
    cgpu = view(0, S * H, torch.float32).cpu().numpy().reshape(S, H)
    modg = view(1, S * 12 * H, torch.float32).cpu().numpy().reshape(S, 2, 6 * H)
    qg = _f(view(3, N * H, torch.bfloat16).reshape(N, H))
    kg = _f(view(4, N * H, torch.bfloat16).reshape(N, H))
    vg = _f(view(5, N * H, torch.bfloat16).reshape(N, H))
    og = _f(view(6, N * H, torch.bfloat16).reshape(N, H))
    for k in range(S):
        it = _block_intermediates(case, x_txt0, emb, k)
        a, b = ref.cu_seqlens[k], ref.cu_seqlens[k + 1]
        assert_close(cgpu[k], it["c"], f"c[{k}]")
        assert_close(modg[k, 0], it["mod_txt"], f"mod_txt[{k}]")
        assert_close(modg[k, 1], it["mod_img"], f"mod_img[{k}]")
        assert_close(qg[a:b], it["q"], f"q[{k}]")
        assert_close(kg[a:b], it["k"], f"k[{k}]")
        assert_close(vg[a:b], it["v"], f"v[{k}]")
        rows = np.concatenate([np.arange(ref.cu_txt[k], ref.cu_txt[k + 1]),
                               ref.n_txt + np.arange(ref.cu_img[k], ref.cu_img[k + 1])])
        assert_close(og[rows], it["o"], f"o[{k}]")
    # the block output vs the oracle on the same inputs; also on the update (out - in)
    xt_ref, xi_ref, _ = oracle_stack(case.samples, ref, case.w, case.batch, d.heads,
                                     x_img_in=emb, n_blocks=1)
    got_t, got_i = _f(x_txt), _f(x_img)
    assert_close(got_t, xt_ref, "block x_txt")
    assert_close(got_i, xi_ref, "block x_img")
    assert_update_close(got_t, xt_ref, x_txt0, "block update txt")
    assert_update_close(got_i, xi_ref, emb, "block update img")


def test_wide_conditioning_intermediates():
    """H = 1024 (the conditioning GEMVs take the bulk-copy kernel from K = 1024 on) with six
    samples (two launches of at most four samples each): the timestep condition c and both
    streams' modulation rows left in the workspace, and the block output, against the oracle."""
    d = synth.Dims(hidden=1024, heads=8, channels=64)
    samples = [synth.Sample(5 + 7 * i, 1, 3 + i, 4, 0.1 + 0.15 * i) for i in range(6)]
    case = Case(samples, d, 1, seed=5)
    ref, H = case.ref, d.hidden
    g = np.random.default_rng(12)
    xi0 = synth.round_bf16(g.standard_normal((ref.n_img, H)).astype(np.float32))
    xt = to_bf16(case.x_txt_np)
    xi = to_bf16(xi0)
    x_txt0 = _f(xt)
    mf.mf_block_forward(case.plan, case.model.dims, case.model.block_structs[0], None, xt, xi, case.ws.block)
    mf.mf_check()
    off = mf.mf_block_workspace_layout(case.plan, case.model.dims)
    S = ref.n_seq
    wsb = case.ws.block
    cg = wsb[off[0]:off[0] + S * H * 4].view(torch.float32).cpu().numpy().reshape(S, H)
    mg = wsb[off[1]:off[1] + S * 12 * H * 4].view(torch.float32).cpu().numpy().reshape(S, 2, 6 * H)
    for k in range(S):
        it = _block_intermediates(case, x_txt0, xi0, k)
        assert_close(cg[k], it["c"], f"c[{k}]")
        assert_close(mg[k, 0], it["mod_txt"], f"mod_txt[{k}]")
        assert_close(mg[k, 1], it["mod_img"], f"mod_img[{k}]")
    xt_ref, xi_ref, _ = oracle_stack(case.samples, ref, case.w, case.batch, d.heads, x_img_in=xi0, n_blocks=1)
    assert_close(_f(xt)[:ref.n_txt], xt_ref, "block x_txt")
    assert_close(_f(xi), xi_ref, "block x_img")


def _stack_and_loss(case, n_blocks, round_zt=True):
    d, ref = case.dims, case.ref
    H, C = d.hidden, d.channels
    Z, E = to_f32(case.z_np), to_f32(case.eps_np)
    ztb = torch.empty((ref.n_img, C), dtype=torch.bfloat16, device="cuda")
    mf.mf_interpolate(case.plan, C, None, Z, E, None, ztb)
    x_txt = to_bf16(case.x_txt_np)
    x_img = torch.empty((ref.n_img, H), dtype=torch.bfloat16, device="cuda")
    v = torch.empty((ref.n_img, C), dtype=torch.float32, device="cuda")
    run_stack(case.plan, case.model, x_txt, ztb, x_img, v, case.ws, n_blocks=n_blocks)
    ls = torch.zeros(ref.n_seq, dtype=torch.float64, device="cuda")
    cnt = torch.zeros(ref.n_seq, dtype=torch.int64, device="cuda")
    mean = torch.zeros(1, dtype=torch.float64, device="cuda")
    mf.mf_flow_loss(case.plan, C, Z, E, v, ls, cnt, mean, case.ws.loss)
    mf.mf_check()
    # oracle: interpolate (source frames clean), then the stack, one sample at a time
    zt = []
    for k, c in enumerate(ref.order):
        s = case.samples[c]
        a, b = ref.cu_img[k], ref.cu_img[k + 1]
        zt.append(M.interpolate(case.z_np[a:b], case.eps_np[a:b], np.float32(s.t), M.target_mask(s)))
    zt = np.concatenate(zt)
    # the model input as the GPU rounds it (bf16), unless the check is against the fp32 originals
    zt_in = synth.round_bf16(zt.astype(np.float32)) if round_zt else zt
    _, _, v_ref = oracle_stack(case.samples, ref, case.w, case.batch, d.heads, zt=zt_in, n_blocks=n_blocks)
    vg = v.cpu().numpy()
    assert_close(vg, v_ref, "velocity v")
    sums = [M.flow_loss(v_ref[ref.cu_img[k]:ref.cu_img[k + 1]], case.z_np[ref.cu_img[k]:ref.cu_img[k + 1]],
                        case.eps_np[ref.cu_img[k]:ref.cu_img[k + 1]],
                        M.target_mask(case.samples[c]))[0] for k, c in enumerate(ref.order)]
    assert_close(ls.cpu().numpy(), sums, "loss sums", rel=2e-2)
    return vg, v_ref


def test_tiny_stack_with_loss():
    case = Case(synth.tiny_samples(), synth.TINY, 1, seed=1)
    _stack_and_loss(case, 1)


def test_tiny_stack_fp32_originals():
    """The tiny configuration against the oracle run on the fp32 original weights, text, latents
    and noise (the GPU rounds weights and text to bf16 and z_t to bf16 as it consumes them): the
    whole error of the path including the inputs' quantisation, which moves v by about 0.3 % of
    its largest value here, stays within the same tolerance."""
    case = Case(synth.tiny_samples(), synth.TINY, 1, seed=1, rounded=False)
    _stack_and_loss(case, 1, round_zt=False)


MID = synth.Dims(hidden=512, heads=4, channels=128)


def _mid_samples(seed, n=6):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        out.append(synth.Sample(int(g.integers(0, 140)), 1, int(g.integers(2, 24)), int(g.integers(2, 24)),
                                float(g.uniform())))
    return out


@pytest.mark.parametrize("seed", [0, 1])
def test_mid_pack_block(seed):
    """A ragged pack at H=512 (4 heads x 128): several GEMM row tiles with tails, samples that
    span several attention tiles, text lengths from 0 up."""
    samples = _mid_samples(seed)
    case = Case(samples, MID, 1, seed=seed + 10)
    _stack_and_loss(case, 1)


def _part_stats(x):
    """(mean, sum of squared deviations) of each 128-column part of each row, float64."""
    r = x.reshape(len(x), -1, 128)
    m = r.mean(axis=2)
    return m, ((r - m[..., None]) ** 2).sum(axis=2)


@pytest.mark.parametrize("size", ["tiny", "mid", "h768", "wide"])
def test_ln_variants(size):
    """The LN + modulate variants of mf_block_forward_ex - one warp per row (the default), row
    groups, and the second LN's statistics fused into the out-projection's epilogue - each match the
    oracle's block.  The fused statistics themselves match (mean, M2) of every 128-column part of
    the residual after attention, x + gate1 (o W_o^T + b_o), formed by the oracle's functions from
    the GPU's own attention output o."""
    if size == "tiny":
        case = Case(synth.tiny_samples(), synth.TINY, 1, seed=3)
    elif size == "mid":
        case = Case(_mid_samples(7), MID, 1, seed=17)
    elif size == "h768":  # 6 heads x 128: an N tile count (3) that leaves a ragged last column
        case = Case(_mid_samples(9), synth.Dims(hidden=768, heads=6, channels=64), 1, seed=29)
    else:  # the widest supported hidden size: 512-thread row kernels, three shared-memory stages
        case = Case([synth.Sample(19, 1, 3, 5, 0.3), synth.Sample(0, 2, 4, 3, 0.8)],
                    synth.Dims(hidden=4096, heads=32, channels=64), 1, seed=23)
    d, ref = case.dims, case.ref
    H = d.hidden
    g = np.random.default_rng(40)
    xi0 = synth.round_bf16(g.standard_normal((ref.n_img, H)).astype(np.float32) + 0.5)
    xt0 = case.x_txt_np
    xt_ref, xi_ref, _ = oracle_stack(case.samples, ref, case.w, case.batch, d.heads, x_img_in=xi0, n_blocks=1)
    off = mf.mf_block_workspace_layout(case.plan, case.model.dims)
    outs = {}
    for name, flags in (("warp rows", 0), ("row groups", mf.BLOCK_LN_ROW_GROUPS),
                        ("fused stats", mf.BLOCK_LN_STATS_FUSED),
                        ("row groups + fused stats", mf.BLOCK_LN_ROW_GROUPS | mf.BLOCK_LN_STATS_FUSED)):
        xt = to_bf16(xt0 if len(xt0) else np.zeros((1, H), np.float32))
        xi = to_bf16(xi0)
        case.ws.block.zero_()
        mf.mf_block_forward_ex(case.plan, case.model.dims, case.model.block_structs[0], None, xt, xi,
                               case.ws.block, flags)
        mf.mf_check()
        got_t, got_i = _f(xt)[:ref.n_txt], _f(xi)
        if ref.n_txt:
            assert_close(got_t, xt_ref, f"{name}: block x_txt")
        assert_close(got_i, xi_ref, f"{name}: block x_img")
        outs[name] = np.concatenate([got_t, got_i])
        if flags & mf.BLOCK_LN_STATS_FUSED:
            N = ref.n_txt + ref.n_img
            wsb = case.ws.block
            st = wsb[off[8]:off[8] + N * (H // 128) * 8].view(torch.float32).cpu().numpy().astype(np.float64)
            st = st.reshape(N, H // 128, 2)
            o = _f(wsb[off[6]:off[6] + N * H * 2].view(torch.bfloat16).reshape(N, H))
            x_in = np.concatenate([xt0[:ref.n_txt], xi0]).astype(np.float64)
            x1 = np.empty((N, H))
            for k, c in enumerate(ref.order):
                cond = M.condition(case.samples[c].t, case.w.temb, d.freq_dim)
                rows = {"txt": np.arange(ref.cu_txt[k], ref.cu_txt[k + 1]),
                        "img": ref.n_txt + np.arange(ref.cu_img[k], ref.cu_img[k + 1])}
                for s_ in M.STREAMS:
                    bw = case.w.blocks[0][s_]
                    gate1 = M.modulation(cond, bw["w_mod"], bw["b_mod"], 6)[2]
                    r = rows[s_]
                    x1[r] = x_in[r] + gate1 * M.linear(o[r], bw["w_o"], bw["b_o"])
            m_ref, q_ref = _part_stats(x1)
            assert_close(st[..., 0], m_ref, "fused statistics: part means")
            assert_close(st[..., 1], q_ref, "fused statistics: part M2")
    # the variants differ only in the f32 order of the statistics' sums
    for name in ("row groups", "fused stats", "row groups + fused stats"):
        assert_close(outs[name], outs["warp rows"], f"{name} vs warp rows", rel=1e-2, cos=0.99999)


def test_cond_given_reuse():
    """Two blocks on a ragged H = 512 pack: the second block reusing the first block's timestep
    condition from the shared workspace (MF_BLOCK_COND_GIVEN) gives the same output bit for bit
    as recomputing it, and so does the final layer given that condition (mf_final_ex)."""
    case = Case(_mid_samples(3), MID, 2, seed=21)
    ref, H = case.ref, case.dims.hidden
    g = np.random.default_rng(8)
    xi0 = synth.round_bf16(g.standard_normal((ref.n_img, H)).astype(np.float32))
    outs = []
    for flags in ((0, 0), (0, mf.BLOCK_COND_GIVEN)):
        xt = to_bf16(case.x_txt_np if len(case.x_txt_np) else np.zeros((1, H), np.float32))
        xi = to_bf16(xi0)
        for b, fl in enumerate(flags):
            mf.mf_block_forward_ex(case.plan, case.model.dims, case.model.block_structs[b], None, xt, xi,
                                   case.ws.block, fl)
        mf.mf_check()
        outs.append((xt.cpu(), xi.cpu()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    # the final layer with the condition the blocks left (mf_final_ex) equals mf_final
    f = case.model.final
    vs = []
    for given in (False, True):
        v = torch.empty((ref.n_img, case.dims.channels), dtype=torch.float32, device="cuda")
        args = (case.plan, case.model.dims, case.model.temb_struct, f["w_fmod"], f["b_fmod"], f["w_out"],
                f["b_out"], None, xi, v, case.ws.final)
        if given:
            off = mf.mf_block_workspace_layout(case.plan, case.model.dims)
            mf.mf_final_ex(*args, case.ws.block.data_ptr() + off[0])
        else:
            mf.mf_final(*args)
        mf.mf_check()
        vs.append(v.cpu())
    assert torch.equal(vs[0], vs[1])


def test_tiny_stack_qk_norm():
    """QK-RMSNorm variant at the tiny size (D = 64: each epilogue warp's 128 columns hold two
    heads, each normalised on its own)."""
    case = Case(synth.tiny_samples(), synth.TINY, 1, seed=11, qk_norm=True)
    _stack_and_loss(case, 1)


@pytest.mark.parametrize("seed", [0, 1])
def test_mid_pack_qk_norm(seed):
    """QK-RMSNorm variant on a ragged H=512 pack (D = 128, one head per epilogue warp), two
    blocks, text lengths from 0 up."""
    samples = _mid_samples(seed + 20)
    case = Case(samples, MID, 2, seed=seed + 30, qk_norm=True)
    _stack_and_loss(case, 2)


def test_degenerate_samples_stack():
    """Degenerate samples in one pack: a single image token and no text, one text token and
    one image token, a 1x3 latent behind 37 text tokens, and flow times at both ends (t = 0:
    z_t = z; t = 1: z_t = eps)."""
    samples = [synth.Sample(0, 1, 1, 1, 0.5), synth.Sample(1, 1, 1, 1, 0.2), synth.Sample(37, 1, 1, 3, 0.9),
               synth.Sample(0, 1, 2, 1, 0.0), synth.Sample(5, 1, 1, 1, 1.0)]
    case = Case(samples, synth.TINY, 1, seed=13)
    _stack_and_loss(case, 1)


def test_single_sample_full_budget():
    """One sample that fills the 16384-token budget exactly (no text, 128 x 128 latents) at
    H=512: attention over a single 16K-token sequence, the largest the budget allows.  Sampled
    rows of the block output (the oracle computes keys and values of the whole sample and the
    queried rows only)."""
    d = MID
    samples = [synth.Sample(0, 1, 128, 128, 0.35)]
    case = Case(samples, d, 1, seed=17, budget=16384)
    ref, H, C = case.ref, d.hidden, d.channels
    assert ref.n_tok == 16384
    Z, E = to_f32(case.z_np), to_f32(case.eps_np)
    ztb = torch.empty((ref.n_img, C), dtype=torch.bfloat16, device="cuda")
    mf.mf_interpolate(case.plan, C, None, Z, E, None, ztb)
    x_img = torch.empty((ref.n_img, H), dtype=torch.bfloat16, device="cuda")
    mf.mf_embed(case.plan, case.model.dims, case.model.embed["w_in"], case.model.embed["b_in"], ztb, x_img)
    mf.mf_check()
    emb = _f(x_img)
    mf.mf_block_forward(case.plan, case.model.dims, case.model.block_structs[0], None, None, x_img,
                        case.ws.block)
    mf.mf_check()
    s = samples[0]
    c = M.condition(np.float32(s.t), case.w.temb, d.freq_dim)
    rows = np.array([0, 1, 127, 128, 4095, 8191, 8192, 12345, 16255, 16256, 16383])
    got = M.block_forward(np.zeros((0, H)), emb, M.image_positions(1, 128, 128), c, case.w.blocks[0],
                          d.heads, rows=rows)
    assert_close(_f(x_img)[rows], got, "block output rows of the 16K sample")


@pytest.mark.parametrize("size", ["tiny", "mid"])
def test_block_fp8(size):
    """fp8 variant of the block (mf_block_forward_fp8): the four projections on E4M3 operands,
    weights quantised per output row by the oracle and uploaded, activations quantised per row
    on the GPU; against the oracle's fp8 block on the GPU's own embed output.  Tiny: H=256,
    D=64, K = 256 / 1024; mid: a ragged H=512 pack, K = 512 / 2048."""
    from oracle import fp8 as F
    d = synth.TINY if size == "tiny" else MID
    samples = synth.tiny_samples() if size == "tiny" else _mid_samples(3)
    case = Case(samples, d, 1, seed=31)
    ref, H = case.ref, d.hidden
    x_img = torch.empty((ref.n_img, H), dtype=torch.bfloat16, device="cuda")
    mf.mf_embed(case.plan, case.model.dims, case.model.embed["w_in"], case.model.embed["b_in"],
                to_bf16(case.z_np), x_img)
    emb = _f(x_img)
    x_txt = to_bf16(case.x_txt_np)
    x_txt0 = _f(x_txt)
    bw = case.w.blocks[0]
    w8 = {st: F.quantize_weights(bw[st]) for st in M.STREAMS}
    w8d = {st: {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in w8[st].items()} for st in M.STREAMS}
    ws = torch.empty(mf.mf_block_fp8_workspace_bytes(case.plan, case.model.dims), dtype=torch.uint8, device="cuda")
    mf.mf_block_forward_fp8(case.plan, case.model.dims, case.model.block_structs[0],
                            mf.block_struct_fp8(w8d["txt"], w8d["img"]), None, x_txt, x_img, ws)
    mf.mf_check()
    xt_ref, xi_ref = [], []
    for k, c in enumerate(ref.order):
        s = samples[c]
        cond = M.condition(np.float32(s.t), case.w.temb, d.freq_dim)
        xt = x_txt0[ref.cu_txt[k]:ref.cu_txt[k + 1]]
        xi = emb[ref.cu_img[k]:ref.cu_img[k + 1]]
        ot, oi = M.block_forward(xt, xi, M.image_positions(s.frames, s.lat_h, s.lat_w), cond, bw, d.heads, w8=w8)
        xt_ref.append(ot)
        xi_ref.append(oi)
    xt_ref, xi_ref = np.concatenate(xt_ref), np.concatenate(xi_ref)
    got_t, got_i = _f(x_txt), _f(x_img)
    assert_close(got_t, xt_ref, "fp8 block x_txt")
    assert_close(got_i, xi_ref, "fp8 block x_img")
    assert_update_close(got_t, xt_ref, x_txt0, "fp8 block update txt")
    assert_update_close(got_i, xi_ref, emb, "fp8 block update img")


def test_mid_edit_stack():
    """Editing structure at H=512: 2 frames (clean source, noisy target), 3-axis RoPE, loss on
    target frames only, 2 blocks."""
    samples = [synth.Sample(40, 2, 8, 12, 0.37), synth.Sample(77, 2, 10, 10, 0.81)]
    case = Case(samples, MID, 2, seed=5)
    _stack_and_loss(case, 2)


def test_mid_cfg_sampler():
    """Packed CFG sampler at H=512: cond + uncond branches of two prompts in one pack, 2 blocks,
    4 Euler steps from t=1 with w=4, against separate (unpacked) cond / uncond oracle runs."""
    d = MID
    samples = [synth.Sample(20, 1, 8, 8, 1.0, 1, 1), synth.Sample(0, 1, 8, 8, 1.0, 2, 0),
               synth.Sample(20, 1, 6, 11, 1.0, 1, 3), synth.Sample(0, 1, 6, 11, 1.0, 2, 2)]
    budget = sum(s.length for s in samples)
    w = synth.model_weights(d, 2, 7)
    batch = synth.cfg_batch(samples, d, 7)
    ref = opack.build_plan(samples, budget)
    plan = mf.mf_pack(samples, budget)
    mf.mf_plan_upload(plan)
    model = DeviceModel(w)
    ws = Workspace(plan, model.dims)
    H, C = d.hidden, d.channels
    grid = [1.0, 0.75, 0.5, 0.25, 0.0]
    z = to_f32(stream_concat(batch.z, ref.order, C))
    zb = z.to(torch.bfloat16)
    x_txt0 = to_bf16(stream_concat(batch.x_txt, ref.order, H))
    x_img = torch.empty((ref.n_img, H), dtype=torch.bfloat16, device="cuda")
    v = torch.empty((ref.n_img, C), dtype=torch.float32, device="cuda")
    tt = torch.empty(ref.n_seq, dtype=torch.float32, device="cuda")
    for a, b in zip(grid[:-1], grid[1:]):
        tt.fill_(a)
        x_txt = x_txt0.clone()
        run_stack(plan, model, x_txt, zb, x_img, v, ws, t=tt)
        mf.mf_cfg_combine(plan, C, 4.0, v, v)
        mf.mf_euler_step(plan, C, a - b, v, z, zb)
    mf.mf_check()
    zg = z.cpu().numpy()
    for k, c in enumerate(ref.order):
        s = samples[c]
        if s.cfg_role != 1:
            continue
        zref = M.sample_cfg(batch.x_txt[c], batch.z[c], s, samples[s.cfg_pair], w, d.heads, 4.0, grid)
        a, b = ref.cu_img[k], ref.cu_img[k + 1]
        assert_close(zg[a:b], zref, f"cfg sample {c}")
        pk = list(ref.order).index(s.cfg_pair)
        np.testing.assert_array_equal(zg[a:b], zg[ref.cu_img[pk]:ref.cu_img[pk + 1]])
