"""A fixed workload run through whichever library MAGEFLOW_LIB selects (the default build or
the bounds-checked one); tests/test_gpu_40_checked_build.py runs it once with each build in a
child process and compares.  Usage: python -m tests._checked_workload OUT.npz"""
import sys

import numpy as np
import torch

import synth
import packed_rectified_flow_packer_b300 as mf
from packed_rectified_flow_packer_b300.device import DeviceModel, Workspace, run_stack, to_bf16, to_f32


def main(out_path):
    out = {}
    # tiny stack + loss, and packed CFG epilogues on the tiny dims
    d = synth.TINY
    samples = synth.tiny_samples() + [synth.Sample(0, 2, 3, 5, 0.4), synth.Sample(3, 1, 1, 1, 0.9)]
    budget = sum(s.length for s in samples)
    plan = mf.mf_pack(samples, budget)
    mf.mf_plan_upload(plan)
    w = synth.model_weights(d, 2, seed=9)
    model = DeviceModel(w)
    order = plan.array("order")
    x, z, e = synth.pack_inputs(samples, order, d, 9)
    ws = Workspace(plan, model.dims)
    Z, E = to_f32(z), to_f32(e)
    ztb = torch.empty((plan.n_img, d.channels), dtype=torch.bfloat16, device="cuda")
    mf.mf_interpolate(plan, d.channels, None, Z, E, None, ztb)
    xt = to_bf16(x)
    xi = torch.empty((plan.n_img, d.hidden), dtype=torch.bfloat16, device="cuda")
    v = torch.empty((plan.n_img, d.channels), dtype=torch.float32, device="cuda")
    run_stack(plan, model, xt, ztb, xi, v, ws)
    ls = torch.zeros(plan.n_seq, dtype=torch.float64, device="cuda")
    cnt = torch.zeros(plan.n_seq, dtype=torch.int64, device="cuda")
    mean = torch.zeros(1, dtype=torch.float64, device="cuda")
    mf.mf_flow_loss(plan, d.channels, Z, E, v, ls, cnt, mean, ws.loss)
    out.update(stack_v=v.cpu().numpy(), stack_x_txt=xt.float().cpu().numpy(), loss=ls.cpu().numpy(),
               count=cnt.cpu().numpy())
    cfg = synth.cfg_samples()
    cfg = [synth.Sample(min(s.txt_len, 7), 1, s.lat_h // 8, s.lat_w // 8, s.t, s.cfg_role, s.cfg_pair) for s in cfg]
    pc = mf.mf_pack(cfg, sum(s.length for s in cfg))
    mf.mf_plan_upload(pc)
    vv = to_f32(np.random.default_rng(3).standard_normal((pc.n_img, d.channels)).astype(np.float32))
    vg = torch.empty_like(vv)
    mf.mf_cfg_combine(pc, d.channels, 4.0, vv, vg)
    out["cfg"] = vg.cpu().numpy()
    # training forward + backward on a ragged H = 512 pack (D = 128)
    mid = synth.Dims(hidden=512, heads=4, channels=128)
    g = np.random.default_rng(5)
    ms = [synth.Sample(int(g.integers(0, 90)), int(g.integers(1, 3)), int(g.integers(2, 18)),
                       int(g.integers(2, 18)), float(g.uniform())) for _ in range(5)]
    mp = mf.mf_pack(ms, sum(s.length for s in ms))
    mf.mf_plan_upload(mp)
    mw = synth.model_weights(mid, 1, seed=11)
    mm = DeviceModel(mw)
    H = mid.hidden
    X_t = to_bf16(g.standard_normal((max(mp.n_txt, 1), H)).astype(np.float32))
    X_i = to_bf16(g.standard_normal((mp.n_img, H)).astype(np.float32))
    tws = torch.empty(mf.mf_block_train_workspace_bytes(mp, mm.dims), dtype=torch.uint8, device="cuda")
    mf.mf_block_forward_train(mp, mm.dims, mm.block_structs[0], None, X_t, X_i, tws)
    out.update(train_x_txt=X_t.float().cpu().numpy(), train_x_img=X_i.float().cpu().numpy())
    G_t = to_bf16(g.standard_normal((max(mp.n_txt, 1), H)).astype(np.float32))
    G_i = to_bf16(g.standard_normal((mp.n_img, H)).astype(np.float32))
    grads = {s: {k: torch.zeros(a.shape, dtype=torch.float32, device="cuda") for k, a in mw.blocks[0][s].items()}
             for s in ("txt", "img")}
    dc = torch.zeros((mp.n_seq, H), dtype=torch.float32, device="cuda")
    bws = torch.empty(mf.mf_block_backward_workspace_bytes(mp, mm.dims), dtype=torch.uint8, device="cuda")
    mf.mf_block_backward(mp, mm.dims, mm.block_structs[0], tws, G_t, G_i,
                         mf.grads_struct(grads["txt"], grads["img"]), dc, bws)
    out.update(bwd_dx_txt=G_t.float().cpu().numpy(), bwd_dx_img=G_i.float().cpu().numpy(),
               bwd_dc=dc.cpu().numpy(), bwd_dw_qkv=grads["img"]["w_qkv"].cpu().numpy(),
               bwd_dw_mod=grads["txt"]["w_mod"].cpu().numpy())
    out["status"] = np.array([mf.lib.mf_check(torch.cuda.current_stream().cuda_stream)])
    np.savez(out_path, **out)


if __name__ == "__main__":
    main(sys.argv[1])
