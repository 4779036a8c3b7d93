#!/usr/bin/env python
"""Throughput of the packed NR-MMDiT hot path on B300: packed tokens/s per block forward.

Workload (default): the native-resolution pack - eight seeded packs of up to 16384 tokens
(candidates with H, W uniform over multiples of 16 in [512, 2048], 32-512 text tokens,
logit-normal t, first-fit), one NR-MMDiT block (H=3072, 24 heads x 128, MLP 4x, bf16 weights
N(0, 0.02)).  One step = one pack through the whole path: z_t interpolation, latent embed,
the block (conditioning, LN+modulate, QKV+RoPE, varlen attention, out-proj+gate, LN+modulate,
MLP+GELU, MLP+gate), the final layer and the flow-matching loss.  Step k uses pack k mod 8.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {mageflow,reference}]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on bounded samples of
the same workload.  Multi-GPU: one process per GPU (torchrun), each rank its own packs (weak
scaling); the only collectives are the timing barrier and the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "packed tokens/s per NR-MMDiT block fwd (1×B300) and % of bf16 tensor peak"
BUDGET = 16384
N_PACKS = 8


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=240)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["mageflow", "reference"], default="mageflow")
    ap.add_argument("--e2e-steps", type=int, default=120)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-baseline sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=["native16k", "cfg", "gemm", "fp8block", "train", "attn", "lnvariants"], default="native16k",
                    help="native16k: the headline block-forward pack; cfg: packed vs unpacked CFG sampler; "
                         "gemm: bf16 and fp8 GEMMs alone at the block's shapes; fp8block: the block "
                         "forward with fp8 projections against the bf16 one on the 16K packs; train: the "
                         "block's training forward + backward on the 16K packs; attn: varlen attention "
                         "forward and backward alone on the 16K packs; lnvariants: the block forward with each LN + "
                         "modulate variant")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def rank_seeds(rank, n_packs=N_PACKS):
    """Pack seeds of one rank: ranks never share a pack (weak scaling, no data exchange)."""
    return [rank * n_packs + i for i in range(n_packs)]


def combine_over_ranks(elapsed_s, tokens, dist=None, device="cpu"):
    """Whole-job timing of a multi-rank run: the slowest rank's elapsed time and the tokens of
    all ranks.  With no process group (one rank) the inputs come back unchanged."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return elapsed_s, tokens
    import torch
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    n = torch.tensor([float(tokens)], dtype=torch.float64, device=device)
    dist.all_reduce(n)
    return float(t.item()), int(n.item())


def config_dict(dims):
    return {"workload": "native-resolution pack, 16384-token budget, 8 seeded packs (first-fit over 64 "
                        "candidates each), 1 NR-MMDiT block + latent embed/final layer + flow loss",
            "budget": BUDGET, "packs": N_PACKS, "hidden": dims.hidden, "heads": dims.heads,
            "head_dim": dims.head_dim, "mlp_ratio": dims.mlp_ratio, "latent_channels": dims.channels,
            "l2": "working set > L2 (0.68 GB block weights + ~1.1 GB activations per step); no flush"}


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d["bf16_tflops_sustained"], "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# ---------------------------------------------------------------- CPU oracle sample
def oracle_sample(dims, weights, cands, order, n_tokens):
    """A bounded sample of the workload for the CPU oracle: the first packed sample of a pack,
    cut to its text plus its first image rows so that it holds about n_tokens tokens."""
    s = cands[order[0]]
    rows = max(1, min(s.lat_h, (n_tokens - s.txt_len) // s.lat_w))
    sub = synth.Sample(s.txt_len, 1, rows, s.lat_w, s.t)
    x = synth.round_bf16(synth.normal(0, "cpu.x_txt", (sub.txt_len, dims.hidden)))
    z = synth.round_bf16(synth.normal(0, "cpu.z", (sub.img_len, dims.channels)))
    return sub, x, z


def time_oracle(dims, weights, sub, x, z, budget_s):
    from oracle import model as M
    n, t0 = 0, time.perf_counter()
    while True:
        M.forward(x, z, sub, sub.t, weights, dims.heads)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= 50:
            return n * sub.length / el, el, n


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            return max(int(i.get("num_threads", 1)) for i in info)
    except Exception:
        pass
    return os.cpu_count()


def _tiny_tokens_per_s(seconds):
    """The oracle on the tiny configuration (2 samples, 144 tokens, H = 256): tokens/s and the
    number of passes timed, with whatever BLAS threads this process has."""
    from oracle import model as M
    d = synth.TINY
    w = synth.model_weights(d, 1, seed=0, bf16=False)
    samples = synth.tiny_samples()
    batch = synth.batch_inputs(samples, d, 0, bf16=False)
    tok, n = 0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds or n == 0:
        for i, smp in enumerate(samples):
            M.forward(batch.x_txt[i], batch.z[i], smp, smp.t, w, d.heads)
            tok += smp.length
        n += 1
    return tok / (time.perf_counter() - t0), n


def tiny_single_thread(seconds=1.0):
    """_tiny_tokens_per_s in a child process whose BLAS runs one thread (the thread count is
    fixed when NumPy loads its BLAS, so it is set in the child's environment)."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = "1"
    code = f"import json, bench; print(json.dumps(bench._tiny_tokens_per_s({float(seconds)})))"
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=120)
    if r.returncode != 0:
        raise RuntimeError("tiny single-thread oracle run failed: " + r.stderr[-300:])
    tps, n = json.loads(r.stdout.strip().splitlines()[-1])
    return tps, n


def cpu_baseline(dims, weights, cands, order, seconds):
    sub, x, z = oracle_sample(dims, weights, cands, order, 2048)
    tps, el, n = time_oracle(dims, weights, sub, x, z, seconds)
    try:
        tiny_tps, tiny_n = tiny_single_thread()
        tiny = {"value": round(tiny_tps, 1), "unit": "tokens/s", "cores": 1,
                "sample": f"tiny configuration (2 samples, 144 tokens, H = 256), {tiny_n} passes"}
    except Exception as e:  # the main baseline stands without it
        tiny = {"unavailable": str(e)[:200]}
    return {"value": tps, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"fp64 NumPy oracle: embed + 1 block + final layer on one sample of pack 0 cut to "
                      f"{sub.txt_len} text + {sub.lat_h}x{sub.lat_w} image tokens ({sub.length} tokens), "
                      f"{n} runs in {el:.1f} s",
            "config": {"workload": sample_workload(sub)},
            "tiny_1thread": tiny}


def sample_workload(sub):
    """What a bounded oracle sample of the native-resolution workload actually runs."""
    return (f"bounded sample of the native-resolution 16K pack workload: one sample of pack 0 cut to "
            f"{sub.length} tokens ({sub.txt_len} text + {sub.lat_h}x{sub.lat_w} image) per step, "
            f"H = {synth.FULL.hidden}, embed + 1 NR-MMDiT block + final layer; attention over "
            f"{sub.length} tokens instead of the packs' ~5K-token samples, so the oracle's per-token cost is "
            f"lower than on the real packs")


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(gpu_id)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- the GPU arm
def run_mageflow(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import packed_rectified_flow_packer_b300 as mf
    from packed_rectified_flow_packer_b300.device import DeviceModel, to_bf16, to_f32

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    dims = synth.FULL
    H, C = dims.hidden, dims.channels
    weights = synth.model_weights(dims, 1, seed=0)
    model = DeviceModel(weights, device=dev)
    d = model.dims

    packs = []
    for seed in rank_seeds(rank):
        cands = synth.native_candidates(seed)
        plan = mf.mf_pack(cands, BUDGET)
        mf.mf_plan_upload(plan)
        x, z, e = synth.pack_inputs(cands, plan.array("order"), dims, seed)
        packs.append({"seed": seed, "cands": cands, "plan": plan, "n_tok": plan.n_tok, "n_img": plan.n_img,
                      "n_seq": plan.n_seq, "x_txt": to_bf16(x, dev), "z": to_f32(z, dev), "eps": to_f32(e, dev),
                      "x_np": x, "z_np": z, "e_np": e})
    wsb = max(mf.mf_block_workspace_bytes(p["plan"], d) for p in packs)
    wsf = max(mf.mf_final_workspace_bytes(p["plan"], d) for p in packs)
    wsl = max(mf.mf_flow_loss_workspace_bytes(p["plan"]) for p in packs)
    ws_block = torch.empty(wsb, dtype=torch.uint8, device=dev)
    ws_final = torch.empty(wsf, dtype=torch.uint8, device=dev)
    ws_loss = torch.empty(wsl, dtype=torch.uint8, device=dev)
    x_txt = torch.empty((BUDGET, H), dtype=torch.bfloat16, device=dev)
    x_img = torch.empty((BUDGET, H), dtype=torch.bfloat16, device=dev)
    ztb = torch.empty((BUDGET, C), dtype=torch.bfloat16, device=dev)
    v = torch.empty((BUDGET, C), dtype=torch.float32, device=dev)
    ls = torch.zeros(64, dtype=torch.float64, device=dev)
    cnt = torch.zeros(64, dtype=torch.int64, device=dev)
    mean = torch.zeros(1, dtype=torch.float64, device=dev)
    stream = torch.cuda.current_stream(dev)
    emb, fin, blk = model.embed, model.final, model.block_structs[0]

    def device_step(p, timed_block=None):
        plan = p["plan"]
        nt = p["x_txt"].shape[0]
        x_txt[:nt].copy_(p["x_txt"])
        mf.mf_interpolate(plan, C, None, p["z"], p["eps"], None, ztb)
        mf.mf_embed(plan, d, emb["w_in"], emb["b_in"], ztb, x_img)
        if timed_block is not None:
            timed_block[0].record(stream)
        mf.mf_block_forward(plan, d, blk, None, x_txt, x_img, ws_block)
        if timed_block is not None:
            timed_block[1].record(stream)
        # the final layer reuses the timestep condition the block left at offset 0 of its workspace
        mf.mf_final_ex(plan, d, model.temb_struct, fin["w_fmod"], fin["b_fmod"], fin["w_out"], fin["b_out"],
                       None, x_img, v, ws_final, ws_block)
        mf.mf_flow_loss(plan, C, p["z"], p["eps"], v, ls, cnt, mean, ws_loss)

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()

    for i in range(args.warmup):
        device_step(packs[i % N_PACKS])
    mf.mf_check()
    barrier()

    # ---- per-kernel breakdown: every library launch bracketed by events, one pass over the
    # packs before the timed region; it also names the dominant kernel
    mf.mf_trace_kinds(None)
    mf.mf_trace_enable(True)
    for i in range(N_PACKS):
        device_step(packs[i % N_PACKS])
    breakdown = mf.mf_trace_read()
    mf.mf_trace_enable(False)
    barrier()
    dom = max((k for k in breakdown if breakdown[k]["flops"] > 0), key=lambda k: breakdown[k]["ms"])

    # ---- timed region: K steps, device-resident inputs; only the dominant kernel's launches
    # carry events (for the roofline's achieved rate), the rest run unbracketed
    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "") or "")
    sampler = ClockSampler(("GPU-" + uuid if uuid and not uuid.startswith("GPU-") else uuid) or local_rank)
    time.sleep(0.3)
    mf.mf_trace_kinds([dom])
    mf.mf_trace_enable(True)
    l0 = mf.mf_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    ev0.record(stream)
    tokens = 0
    for i in range(args.steps):
        p = packs[i % N_PACKS]
        device_step(p)
        tokens += p["n_tok"]
    ev1.record(stream)
    barrier()
    launches = mf.mf_launch_count() - l0
    trace = mf.mf_trace_read()
    mf.mf_trace_enable(False)
    mf.mf_trace_kinds(None)
    clocks = sampler.stop()
    mf.mf_check()
    elapsed = ev0.elapsed_time(ev1) / 1e3
    elapsed, tokens = combine_over_ranks(elapsed, tokens, dist if world > 1 else None, dev)

    # ---- block-only timing (untraced): events around each block call
    block_ms, block_tok = 0.0, 0
    pairs = []
    for i in range(min(args.steps, 4 * N_PACKS)):
        p = packs[i % N_PACKS]
        pr = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        device_step(p, pr)
        pairs.append((pr, p))
    torch.cuda.synchronize(dev)
    block_flops = 0.0
    for (a, b), p in pairs:
        block_ms += a.elapsed_time(b)
        block_tok += p["n_tok"]
        cu = p["plan"].array("cu_seqlens").astype(np.float64)
        block_flops += 24.0 * H * H * p["n_tok"] + 4.0 * H * float((np.diff(cu) ** 2).sum()) \
            + 2.0 * 2 * 6.0 * H * H * p["n_seq"]

    # ---- end to end through the public API with host buffers.  Each step packs its
    # candidates on the host, uploads the plan and copies that step's text, latents and noise
    # from pinned host memory, runs the path and reads the per-sample loss back.  The host work
    # and the copies of step i + 1 run on a side stream while the GPU computes step i (inputs
    # double-buffered, events between the streams); step i's loss is read once step i + 1 has
    # been queued.  Every step's copies and readback lie inside the timed region.
    e2e = None
    if args.e2e_steps > 0:
        pinned = []
        for p in packs:
            pinned.append({"x": torch.from_numpy(p["x_np"]).to(torch.bfloat16).pin_memory(),
                           "z": torch.from_numpy(p["z_np"]).pin_memory(),
                           "e": torch.from_numpy(p["e_np"]).pin_memory()})
        side = torch.cuda.Stream(dev)
        bufs = [{"x": torch.empty((BUDGET, H), dtype=torch.bfloat16, device=dev),
                 "z": torch.empty((BUDGET, C), dtype=torch.float32, device=dev),
                 "e": torch.empty((BUDGET, C), dtype=torch.float32, device=dev)} for _ in range(2)]
        host_out = [torch.empty(64 * 2 + 1, dtype=torch.float64).pin_memory() for _ in range(2)]
        ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        warm = 2
        total_steps = args.e2e_steps + warm

        def stage(i):
            """Host packing, plan upload and input copies of step i on the side stream."""
            slot = i % 2
            p, hp, b = packs[i % N_PACKS], pinned[i % N_PACKS], bufs[slot]
            plan = mf.mf_pack(p["cands"], BUDGET)                        # host packer
            mf.mf_plan_upload(plan, side)                                # index buffers H2D
            with torch.cuda.stream(side):
                side.wait_event(done[slot])                              # step i - 2 left this slot
                nt, ni = hp["x"].shape[0], hp["z"].shape[0]
                b["x"][:nt].copy_(hp["x"], non_blocking=True)
                b["z"][:ni].copy_(hp["z"], non_blocking=True)
                b["e"][:ni].copy_(hp["e"], non_blocking=True)
                ready[slot].record(side)
            info = plan.info()
            S = plan.n_seq
            plan_bytes = 4 * (2 * (S + 1) + 3 * info.n_tok + 3 * info.n_tok + 3 * info.n_img + 2 * S +
                              2 * info.n_items)
            h2d = hp["x"].numel() * 2 + hp["z"].numel() * 4 + hp["e"].numel() * 4 + plan_bytes
            return plan, h2d

        def compute(i, plan):
            slot = i % 2
            b = bufs[slot]
            stream.wait_event(ready[slot])
            mf.mf_interpolate(plan, C, None, b["z"], b["e"], None, ztb)
            mf.mf_embed(plan, d, emb["w_in"], emb["b_in"], ztb, x_img)
            mf.mf_block_forward(plan, d, blk, None, b["x"], x_img, ws_block)
            mf.mf_final_ex(plan, d, model.temb_struct, fin["w_fmod"], fin["b_fmod"], fin["w_out"], fin["b_out"],
                           None, x_img, v, ws_final, ws_block)
            mf.mf_flow_loss(plan, C, b["z"], b["e"], v, ls, cnt, mean, ws_loss)
            S = plan.n_seq
            ho = host_out[slot]
            ho[:S].copy_(ls[:S], non_blocking=True)
            ho[64:64 + S].copy_(cnt[:S].double(), non_blocking=True)
            ho[128:129].copy_(mean, non_blocking=True)
            done[slot].record(stream)
            return 16 * S + 8

        def retire(j, pj):
            done[j % 2].synchronize()
            return host_out[j % 2][128].item()                          # step j's mean loss

        h2d = d2h = e_tok = 0
        t_start = None
        staged = stage(0)
        inflight = None                                                  # (step, plan) on the GPU
        for i in range(total_steps):
            plan, hb = staged
            ob = compute(i, plan)
            if i >= warm:
                h2d += hb
                d2h += ob
                e_tok += plan.n_tok
            if i + 1 == warm:
                # timing starts with the GPU idle, before step `warm` is packed and copied
                torch.cuda.synchronize(dev)
                t_start = time.perf_counter()
            if i + 1 < total_steps:
                staged = stage(i + 1)
            if inflight is not None:
                retire(*inflight)
            inflight = (i, plan)
        retire(*inflight)
        del inflight, plan, staged
        e_el = time.perf_counter() - t_start
        e2e = {"value": e_tok / e_el, "unit": "tokens/s", "h2d_bytes_per_step": int(h2d / args.e2e_steps),
               "d2h_bytes_per_step": int(d2h / args.e2e_steps),
               "includes": "host first-fit packing, plan upload, pinned H2D of text/latents/noise, "
                           "device path, D2H of per-sample loss sums, counts and mean; the host work "
                           "and copies of step i + 1 overlap the GPU work of step i"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None

    # ---- roofline of the dominant kernel, from its events inside the timed region
    peaks = read_peaks()
    kernels = {}
    for k, e in breakdown.items():
        if e["launches"] == 0:
            continue
        row = {"launches": e["launches"], "ms_total": round(e["ms"], 3),
               "ms_avg": round(e["ms"] / e["launches"], 4), "share": None}
        if e["flops"] > 0 and e["ms"] > 0:
            row["tflops"] = round(e["flops"] / (e["ms"] / 1e3) / 1e12, 1)
        if e["bytes"] > 0 and e["ms"] > 0:
            row["gbs"] = round(e["bytes"] / (e["ms"] / 1e3) / 1e9, 1)
        kernels[k] = row
    tot_ms = sum(e["ms"] for e in breakdown.values())
    for k in kernels:
        kernels[k]["share"] = round(breakdown[k]["ms"] / tot_ms, 4) if tot_ms else None
    de = trace[dom]
    achieved = de["flops"] / (de["ms"] / 1e3) / 1e12
    gemm_kinds = ("gemm_qkv", "gemm_oproj", "gemm_up", "gemm_down")
    g_fl = sum(breakdown[k]["flops"] for k in gemm_kinds)
    g_ms = sum(breakdown[k]["ms"] for k in gemm_kinds)
    traffic = None
    tfile = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tfile):
        with open(tfile) as f:
            traffic = json.load(f).get(dom)
    avg_ms = de["ms"] / de["launches"]
    roofline = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 1),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved / peaks["bf16_tflops"], 4),
                "peak_kind": f"dense bf16 burst ({peaks['source']}: cuBLAS bf16 GEMM, best of 10)",
                "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                "avg_ms": round(avg_ms, 4),
                "avg_ms_x_sm_mhz": round(avg_ms * clocks["sm_mhz"], 1) if clocks.get("sm_mhz") else None,
                "traffic": traffic,
                "flops_per_launch": de["flops"] / de["launches"],
                "all_gemms_tflops": round(g_fl / (g_ms / 1e3) / 1e12, 1) if g_ms else None,
                "attention_tflops": kernels.get("attn", {}).get("tflops"),
                "measured": f"CUDA events around every {dom} launch inside the timed region; "
                            "the other kernels of the step carry no events there"}
    blk_tflops = block_flops / (block_ms / 1e3) / 1e12
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(dims, weights, packs[0]["cands"], packs[0]["plan"].array("order"), args.cpu_seconds)
    value = tokens / elapsed
    line = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed / args.steps * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) text embeddings, latents and noise; N(0,0.02) weights)",
            "config": config_dict(dims), "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": int(launches), "clocks": clocks,
            "block": {"ms_avg": round(block_ms / len(pairs), 4), "tokens_per_s": round(block_tok / (block_ms / 1e3), 1),
                      "tflops": round(blk_tflops, 1), "frac_of_burst": round(blk_tflops / peaks["bf16_tflops"], 4),
                      "frac_of_sustained": round(blk_tflops / peaks["bf16_tflops_sustained"], 4),
                      "flops_note": "24 H^2 N + 4 H sum L_i^2 + modulation; diagonal attention blocks only"},
            "kernels": kernels,
            "kernels_note": "per-kernel events around every launch, one pass over the 8 packs before the timed region",
            "peaks": peaks}
    if world > 1:
        dist.destroy_process_group()
    return line


# ---------------------------------------------------------------- packed vs unpacked CFG sampler
def run_gemm_shapes(args, rank, world, local_rank):
    """The block's four projections as plain GEMMs at the 16K pack's row count (M = 15744, the
    mean of the seeded packs), bf16 (`mf_gemm`) and fp8 (`mf_gemm_fp8` on operands the library
    quantised per row), CUDA events around K launches after W warm-up launches each; the
    quantiser is timed on its own.  Random N(0, 0.5) activations and N(0, 0.02) weights."""
    import torch
    import packed_rectified_flow_packer_b300 as mf
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    H, M = synth.FULL.hidden, 15744
    g = torch.Generator(device=dev).manual_seed(0)
    peaks = read_peaks()
    shapes = {"qkv": (3 * H, H), "oproj": (H, H), "up": (4 * H, H), "down": (H, 4 * H)}
    out = {}
    for name, (N, K) in shapes.items():
        a = (torch.randn((M, K), device=dev, generator=g) * 0.5).to(torch.bfloat16)
        b = (torch.randn((N, K), device=dev, generator=g) * 0.02).to(torch.bfloat16)
        aq = torch.empty((M, K), dtype=torch.uint8, device=dev)
        bq = torch.empty((N, K), dtype=torch.uint8, device=dev)
        sa = torch.empty(M, dtype=torch.float32, device=dev)
        sb = torch.empty(N, dtype=torch.float32, device=dev)
        mf.mf_quantize_fp8_rows(b, bq, sb)
        c8 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        c16 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        mf.mf_quantize_fp8_rows(a, aq, sa)
        row = {}
        for tag, fn in (("fp8", lambda: mf.mf_gemm_fp8(aq, sa, bq, sb, c8)),
                        ("bf16", lambda: mf.mf_gemm(a, b, c16)),
                        ("quantize", lambda: mf.mf_quantize_fp8_rows(a, aq, sa))):
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(args.steps):
                fn()
            e1.record()
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1) / args.steps
            if tag == "quantize":
                row["quantize_us"] = round(ms * 1e3, 2)
                row["quantize_gbs"] = round(3.0 * M * K / ms / 1e6, 1)
            else:
                row[f"{tag}_ms"] = round(ms, 4)
                row[f"{tag}_tflops"] = round(2.0 * M * N * K / ms / 1e9, 1)
        mf.mf_check()
        row["M"], row["N"], row["K"] = M, N, K
        out[name] = row
    if rank != 0:
        return None
    bf = peaks["bf16_tflops"]
    return {"metric": "GEMM TFLOP/s at the block's shapes (bf16 and fp8 E4M3), 1xB300", "workload": "gemm",
            "steps": args.steps, "warmup": args.warmup, "shapes": out,
            "peaks": {"bf16_tflops": bf, "fp8_tflops_from_bf16x2": round(2 * bf, 1), "source": peaks["source"]},
            "data": "synthetic (N(0,0.5) activations, N(0,0.02) weights)"}


def run_fp8_block(args, rank, world, local_rank):
    """The block forward on the eight seeded 16K packs, bf16 (`mf_block_forward`) and fp8
    (`mf_block_forward_fp8`, weights quantised per row by the library at setup), block calls
    only, K timed calls each after W warm-up calls, CUDA events around the whole run."""
    import torch
    import packed_rectified_flow_packer_b300 as mf
    from packed_rectified_flow_packer_b300.device import DeviceModel, to_bf16
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dims = synth.FULL
    H = dims.hidden
    model = DeviceModel(synth.model_weights(dims, 1, seed=0), device=dev)
    d = model.dims
    w8 = {}
    for st in ("txt", "img"):
        w8[st] = {}
        for name in ("qkv", "o", "1", "2"):
            wt = model.blocks[0][st]["w_" + name]
            q = torch.empty(wt.shape, dtype=torch.uint8, device=dev)
            sc = torch.empty(wt.shape[0], dtype=torch.float32, device=dev)
            mf.mf_quantize_fp8_rows(wt, q, sc)
            w8[st]["q_" + name], w8[st]["s_" + name] = q, sc
    s8 = mf.block_struct_fp8(w8["txt"], w8["img"])
    packs = []
    for seed in rank_seeds(rank):
        cands = synth.native_candidates(seed)
        plan = mf.mf_pack(cands, BUDGET)
        mf.mf_plan_upload(plan)
        x, _, _ = synth.pack_inputs(cands, plan.array("order"), dims, seed)
        xi = torch.randn((plan.n_img, H), device=dev, generator=torch.Generator(device=dev).manual_seed(seed))
        packs.append({"plan": plan, "x_txt": to_bf16(x, dev), "x_img": xi.to(torch.bfloat16)})
    ws = torch.empty(max(mf.mf_block_fp8_workspace_bytes(p["plan"], d) for p in packs), dtype=torch.uint8,
                     device=dev)
    xt = torch.empty((BUDGET, H), dtype=torch.bfloat16, device=dev)
    xi = torch.empty((BUDGET, H), dtype=torch.bfloat16, device=dev)
    out = {}
    for tag in ("bf16", "fp8"):
        def call(p):
            nt, ni = p["x_txt"].shape[0], p["x_img"].shape[0]
            xt[:nt].copy_(p["x_txt"])
            xi[:ni].copy_(p["x_img"])
            if tag == "fp8":
                mf.mf_block_forward_fp8(p["plan"], d, model.block_structs[0], s8, None, xt, xi, ws)
            else:
                mf.mf_block_forward(p["plan"], d, model.block_structs[0], None, xt, xi, ws)
        for i in range(args.warmup):
            call(packs[i % N_PACKS])
        torch.cuda.synchronize(dev)
        ms, tok = 0.0, 0
        for i in range(args.steps):
            p = packs[i % N_PACKS]
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            nt, ni = p["x_txt"].shape[0], p["x_img"].shape[0]
            xt[:nt].copy_(p["x_txt"])
            xi[:ni].copy_(p["x_img"])
            e0.record()
            if tag == "fp8":
                mf.mf_block_forward_fp8(p["plan"], d, model.block_structs[0], s8, None, xt, xi, ws)
            else:
                mf.mf_block_forward(p["plan"], d, model.block_structs[0], None, xt, xi, ws)
            e1.record()
            torch.cuda.synchronize(dev)
            ms += e0.elapsed_time(e1)
            tok += p["plan"].n_tok
        mf.mf_check()
        out[tag] = {"ms_per_block": round(ms / args.steps, 4), "tokens_per_s": round(tok / (ms / 1e3), 1)}
    if rank != 0:
        return None
    return {"metric": "packed tokens/s per NR-MMDiT block fwd, bf16 vs fp8 projections (1xB300)",
            "workload": "fp8block", "steps": args.steps, "warmup": args.warmup, "bf16": out["bf16"],
            "fp8": out["fp8"], "fp8_speedup": round(out["bf16"]["ms_per_block"] / out["fp8"]["ms_per_block"], 4),
            "data": "synthetic (seeded packs; N(0,1) hidden image states instead of the latent embed)"}


def run_ln_variants(args, rank, world, local_rank):
    """The block forward on the eight seeded 16K packs with each LN + modulate variant of
    mf_block_forward_ex: one warp per row (the default), row groups, and the second LN's
    statistics fused into the out-projection's epilogue.  Per variant: K block calls timed with
    CUDA events after W warm-up calls, then one pass over the packs with every launch traced
    for the LN and out-projection kernel times."""
    import torch
    import packed_rectified_flow_packer_b300 as mf
    from packed_rectified_flow_packer_b300.device import DeviceModel, to_bf16
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dims = synth.FULL
    H = dims.hidden
    model = DeviceModel(synth.model_weights(dims, 1, seed=0), device=dev)
    d = model.dims
    packs = []
    for seed in rank_seeds(rank):
        cands = synth.native_candidates(seed)
        plan = mf.mf_pack(cands, BUDGET)
        mf.mf_plan_upload(plan)
        x, _, _ = synth.pack_inputs(cands, plan.array("order"), dims, seed)
        xi = torch.randn((plan.n_img, H), device=dev, generator=torch.Generator(device=dev).manual_seed(seed))
        packs.append({"plan": plan, "x_txt": to_bf16(x, dev), "x_img": xi.to(torch.bfloat16)})
    ws = torch.empty(max(mf.mf_block_workspace_bytes(p["plan"], d) for p in packs), dtype=torch.uint8, device=dev)
    xt = torch.empty((BUDGET, H), dtype=torch.bfloat16, device=dev)
    xi = torch.empty((BUDGET, H), dtype=torch.bfloat16, device=dev)
    variants = (("warp_rows", 0), ("row_groups", mf.BLOCK_LN_ROW_GROUPS), ("stats_fused", mf.BLOCK_LN_STATS_FUSED))
    out = {}

    def call(p, flags):
        nt, ni = p["x_txt"].shape[0], p["x_img"].shape[0]
        xt[:nt].copy_(p["x_txt"])
        xi[:ni].copy_(p["x_img"])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        mf.mf_block_forward_ex(p["plan"], d, model.block_structs[0], None, xt, xi, ws, flags)
        e1.record()
        return e0, e1

    for rep_ in range(2):  # the variants twice, interleaved, so a clock drift shows
        for tag, flags in variants:
            for i in range(args.warmup):
                call(packs[i % N_PACKS], flags)
            torch.cuda.synchronize(dev)
            ms, tok = 0.0, 0
            for i in range(args.steps):
                p = packs[i % N_PACKS]
                e0, e1 = call(p, flags)
                torch.cuda.synchronize(dev)
                ms += e0.elapsed_time(e1)
                tok += p["plan"].n_tok
            mf.mf_trace_kinds(["ln", "gemm_oproj"])
            mf.mf_trace_enable(True)
            for i in range(N_PACKS):
                call(packs[i], flags)
            tr = mf.mf_trace_read()
            mf.mf_trace_enable(False)
            mf.mf_trace_kinds(None)
            mf.mf_check()
            ln, op = tr["ln"], tr["gemm_oproj"]
            out.setdefault(tag, []).append({
                "ms_per_block": round(ms / args.steps, 4), "tokens_per_s": round(tok / (ms / 1e3), 1),
                "ln_us_avg": round(1e3 * ln["ms"] / ln["launches"], 2),
                "ln_gbs": round(ln["bytes"] / (ln["ms"] / 1e3) / 1e9, 1),
                "oproj_us_avg": round(1e3 * op["ms"] / op["launches"], 2)})
    # a plain device copy of the same bytes (read [N][H] bf16, write [N][H] bf16) on the same box,
    # the bandwidth an LN pass could reach
    n_rows = max(p["plan"].n_tok for p in packs)
    src = torch.randn((n_rows, H), device=dev).to(torch.bfloat16)
    dst = torch.empty_like(src)
    for _ in range(args.warmup):
        dst.copy_(src)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        dst.copy_(src)
    e1.record()
    torch.cuda.synchronize(dev)
    copy_us = 1e3 * e0.elapsed_time(e1) / args.steps
    copy = {"rows": n_rows, "us": round(copy_us, 2), "gbs": round(4.0 * n_rows * H / (copy_us / 1e6) / 1e9, 1)}
    if rank != 0:
        return None
    return {"metric": "packed tokens/s per NR-MMDiT block fwd by LN + modulate variant (1xB300)",
            "workload": "lnvariants", "steps": args.steps, "warmup": args.warmup, "variants": out,
            "copy_same_bytes": copy,
            "config": {"workload": "8 seeded native-resolution 16K packs, 1 block, H = 3072"},
            "data": "synthetic (seeded packs; N(0,1) hidden image states instead of the latent embed)"}


def run_train(args, rank, world, local_rank):
    """Training step of one NR-MMDiT block on the eight seeded 16K packs: mf_block_forward_train
    (the forward that keeps what the backward reads), then mf_block_backward with a seeded
    output gradient (input, weight, modulation and condition gradients of both streams).
    Inputs resident in HBM; CUDA events around K steps after W warm-up steps; one traced pass
    before the timed region gives the per-kernel table and names the dominant kernel, whose
    launches alone carry events inside the timed region."""
    import torch
    import packed_rectified_flow_packer_b300 as mf
    from packed_rectified_flow_packer_b300.device import DeviceModel, to_bf16
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dims = synth.FULL
    H, R = dims.hidden, dims.mlp_ratio * dims.hidden
    weights = synth.model_weights(dims, 1, seed=0)
    model = DeviceModel(weights, device=dev)
    d, bs = model.dims, model.block_structs[0]
    packs = []
    for seed in rank_seeds(rank):
        cands = synth.native_candidates(seed)
        plan = mf.mf_pack(cands, BUDGET)
        mf.mf_plan_upload(plan)
        x, _, _ = synth.pack_inputs(cands, plan.array("order"), dims, seed)
        gen = torch.Generator(device=dev).manual_seed(1000 + seed)
        ni, nt = plan.n_img, plan.n_txt
        cu = plan.array("cu_seqlens").astype(np.float64)
        packs.append({"plan": plan, "n_tok": plan.n_tok, "n_seq": plan.n_seq, "x_txt": to_bf16(x, dev),
                      "x_img": torch.randn((ni, H), device=dev, generator=gen).to(torch.bfloat16),
                      "g_txt": torch.randn((max(nt, 1), H), device=dev, generator=gen).to(torch.bfloat16),
                      "g_img": torch.randn((ni, H), device=dev, generator=gen).to(torch.bfloat16),
                      "sum_L2": float((np.diff(cu) ** 2).sum())})
    tws = torch.empty(max(mf.mf_block_train_workspace_bytes(p["plan"], d) for p in packs), dtype=torch.uint8, device=dev)
    bws = torch.empty(max(mf.mf_block_backward_workspace_bytes(p["plan"], d) for p in packs), dtype=torch.uint8,
                      device=dev)
    xt = torch.empty((BUDGET, H), dtype=torch.bfloat16, device=dev)
    xi = torch.empty((BUDGET, H), dtype=torch.bfloat16, device=dev)
    grads = {s: {k: torch.empty(v.shape, dtype=torch.float32, device=dev) for k, v in weights.blocks[0][s].items()}
             for s in ("txt", "img")}
    gstruct = mf.grads_struct(grads["txt"], grads["img"])
    dc = torch.empty((64, H), dtype=torch.float32, device=dev)

    def step(p):
        nt, ni = p["x_txt"].shape[0], p["x_img"].shape[0]
        xt[:nt].copy_(p["x_txt"])
        xi[:ni].copy_(p["x_img"])
        mf.mf_block_forward_train(p["plan"], d, bs, None, xt, xi, tws)
        xt[:p["g_txt"].shape[0]].copy_(p["g_txt"])
        xi[:ni].copy_(p["g_img"])
        mf.mf_block_backward(p["plan"], d, bs, tws, xt, xi, gstruct, dc, bws)

    def flops(p):
        N, S, L2 = p["n_tok"], p["n_seq"], p["sum_L2"]
        fwd = 24.0 * H * H * N + 4.0 * H * L2 + 2.0 * 2 * 6.0 * H * H * S
        bwd = 48.0 * H * H * N + 10.0 * H * L2 + 2.0 * 2 * 2 * 6.0 * H * H * S
        return fwd, bwd

    for i in range(args.warmup):
        step(packs[i % N_PACKS])
    torch.cuda.synchronize(dev)
    mf.mf_check()
    mf.mf_trace_kinds(None)
    mf.mf_trace_enable(True)
    for i in range(N_PACKS):
        step(packs[i])
    breakdown = mf.mf_trace_read()
    mf.mf_trace_enable(False)
    torch.cuda.synchronize(dev)
    dom = max((k for k in breakdown if breakdown[k]["flops"] > 0), key=lambda k: breakdown[k]["ms"])
    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "") or "")
    sampler = ClockSampler(("GPU-" + uuid if uuid and not uuid.startswith("GPU-") else uuid) or local_rank)
    time.sleep(0.3)
    mf.mf_trace_kinds([dom])
    mf.mf_trace_enable(True)
    l0 = mf.mf_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record()
    tokens, fl_f, fl_b = 0, 0.0, 0.0
    for i in range(args.steps):
        p = packs[i % N_PACKS]
        step(p)
        tokens += p["n_tok"]
        f, b = flops(p)
        fl_f += f
        fl_b += b
    e1.record()
    torch.cuda.synchronize(dev)
    launches = mf.mf_launch_count() - l0
    trace = mf.mf_trace_read()
    mf.mf_trace_enable(False)
    mf.mf_trace_kinds(None)
    clocks = sampler.stop()
    mf.mf_check()
    if rank != 0:
        return None
    el = e0.elapsed_time(e1) / 1e3
    peaks = read_peaks()
    tot_ms = sum(e["ms"] for e in breakdown.values())
    kernels = {}
    for k, e in breakdown.items():
        if e["launches"] == 0:
            continue
        row = {"launches": e["launches"], "ms_total": round(e["ms"], 3), "share": round(e["ms"] / tot_ms, 4)}
        if e["flops"] > 0 and e["ms"] > 0:
            row["tflops"] = round(e["flops"] / (e["ms"] / 1e3) / 1e12, 1)
        if e["bytes"] > 0 and e["ms"] > 0:
            row["gbs"] = round(e["bytes"] / (e["ms"] / 1e3) / 1e9, 1)
        kernels[k] = row
    de = trace[dom]
    achieved = de["flops"] / (de["ms"] / 1e3) / 1e12
    tflops = (fl_f + fl_b) / el / 1e12
    traffic = None
    tfile = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tfile):
        with open(tfile) as f:
            traffic = json.load(f).get(dom)
    return {"metric": "packed tokens/s per NR-MMDiT block training step (fwd + bwd, 1xB300)",
            "value": round(tokens / el, 1), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic (seeded packs; N(0,1) hidden states and output gradients)",
            "config": dict(config_dict(dims), workload="native-resolution pack, 16384-token budget, 8 seeded packs, "
                           "1 NR-MMDiT block: training forward + backward (all weight, input and condition "
                           "gradients)"),
            "tflops": round(tflops, 1), "mfu_of_burst": round(tflops / peaks["bf16_tflops"], 4),
            "flops_note": "fwd 24 H^2 N + 4 H sum L_i^2, bwd 48 H^2 N + 10 H sum L_i^2, + modulation; "
                          "diagonal attention blocks only",
            "fwd_flops_share": round(fl_f / (fl_f + fl_b), 4),
            "roofline": {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                         "peak_kind": f"dense bf16 burst ({peaks['source']})", "traffic": traffic,
                         "avg_ms": round(de["ms"] / de["launches"], 4)},
            "gpu_launches": int(launches), "clocks": clocks, "kernels": kernels,
            "pages_context": "training step 1.9259 s -> 0.7748 s, MFU 33.20 % -> 77.26 % on 8xB200 "
                             "(PaperReading review, section 3, Table 4; whole model, 50K-token packs)"}


def run_attention(args, rank, world, local_rank):
    """Varlen attention alone on the eight seeded 16K packs (24 heads x 128): the forward with
    its logsumexp (mf_attention_lse) and the backward (mf_attention_backward), seeded N(0,1)
    q, k, v and output gradients; CUDA events around each launch, K launches after W warm-up
    launches per pack cycle.  FLOPs over the sample diagonals only: 4 H sum L_i^2 forward,
    10 H sum L_i^2 backward (S^T, dP^T, dV, dK, dQ)."""
    import torch
    import packed_rectified_flow_packer_b300 as mf
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dims = synth.FULL
    H, heads, D = dims.hidden, dims.heads, dims.head_dim
    packs = []
    for seed in rank_seeds(rank):
        cands = synth.native_candidates(seed)
        plan = mf.mf_pack(cands, BUDGET)
        mf.mf_plan_upload(plan)
        cu = plan.array("cu_seqlens").astype(np.float64)
        packs.append({"plan": plan, "n_tok": plan.n_tok, "sum_L2": float((np.diff(cu) ** 2).sum())})
    gen = torch.Generator(device=dev).manual_seed(77)
    q, k, v, do = (torch.randn((BUDGET, H), device=dev, generator=gen).to(torch.bfloat16) for _ in range(4))
    o = torch.empty((BUDGET, H), dtype=torch.bfloat16, device=dev)
    dq, dk, dv = (torch.empty((BUDGET, H), dtype=torch.bfloat16, device=dev) for _ in range(3))
    lse = torch.empty((heads, BUDGET), dtype=torch.float32, device=dev)
    ws = torch.empty(max(mf.mf_attention_backward_workspace_bytes(p["plan"], heads, D) for p in packs),
                     dtype=torch.uint8, device=dev)
    out = {}
    for tag in ("fwd", "bwd"):
        def call(p):
            if tag == "fwd":
                mf.mf_attention_lse(p["plan"], heads, D, q, k, v, o, lse)
            else:
                mf.mf_attention_backward(p["plan"], heads, D, q, k, v, o, lse, do, dq, dk, dv, ws)
        for i in range(max(args.warmup, N_PACKS)):
            p = packs[i % N_PACKS]
            mf.mf_attention_lse(p["plan"], heads, D, q, k, v, o, lse)
            call(p)
        torch.cuda.synchronize(dev)
        mf.mf_check()
        mf.mf_trace_kinds(["attn" if tag == "fwd" else "attn_bwd"])
        mf.mf_trace_enable(True)
        fl = 0.0
        for i in range(args.steps):
            p = packs[i % N_PACKS]
            if tag == "bwd":   # the backward reads the lse of the same pack (not bracketed)
                mf.mf_attention_lse(p["plan"], heads, D, q, k, v, o, lse)
            call(p)
            fl += (4.0 if tag == "fwd" else 10.0) * H * p["sum_L2"]
        tr = mf.mf_trace_read()
        mf.mf_trace_enable(False)
        mf.mf_trace_kinds(None)
        mf.mf_check()
        e = tr["attn" if tag == "fwd" else "attn_bwd"]
        out[tag] = {"launches": e["launches"], "ms_avg": round(e["ms"] / e["launches"], 4),
                    "tflops": round(fl / (e["ms"] / 1e3) / 1e12, 1)}
    if rank != 0:
        return None
    peaks = read_peaks()
    for tag in out:
        out[tag]["frac_of_burst"] = round(out[tag]["tflops"] / peaks["bf16_tflops"], 4)
    return {"metric": "varlen joint attention TFLOP/s, forward and backward (1xB300)", "workload": "attn",
            "steps": args.steps, "warmup": args.warmup, "fwd": out["fwd"], "bwd": out["bwd"],
            "config": {"workload": "8 seeded native-resolution 16K packs, 24 heads x 128, diagonal blocks only"},
            "data": "synthetic (N(0,1) q, k, v, output gradients)", "peaks": peaks}


def run_cfg_sampler(args, rank, world, local_rank):
    """4-block stack, two prompts (1024x1024 and 768x1344, 256 text tokens when conditional),
    Euler steps on a uniform grid from t = 1 to 0, guidance w = 4, for 4 steps (the Turbo
    setting) and 20 steps (the base model's, where the pages see the largest packed-CFG gain).
    Packed: cond and uncond branches of both prompts in one pack (16768 tokens); the library
    combines the branches in place.  Unpacked: the cond pack and the uncond pack run one after
    the other, and the guided step z += dt (v_u + w (v_c - v_u)) is applied as
    z += dt (1 - w) v_u, then z += dt w v_c.  Each arm's whole sampler is captured once as a
    CUDA graph and replayed."""
    import torch

    import packed_rectified_flow_packer_b300 as mf
    from packed_rectified_flow_packer_b300.device import DeviceModel, Workspace, run_stack, to_bf16, to_f32

    if rank != 0:
        return None
    torch.cuda.set_device(local_rank)
    dims = synth.FULL
    H, C = dims.hidden, dims.channels
    weights = synth.model_weights(dims, 4, seed=3)
    model = DeviceModel(weights)
    w = 4.0

    def arm(samples):
        plan = mf.mf_pack(samples, sum(s.length for s in samples))
        mf.mf_plan_upload(plan)
        order = plan.array("order")
        n_txt, n_img = plan.n_txt, plan.n_img
        x0 = np.concatenate([synth.round_bf16(synth.normal(7, f"x_txt.{c}", (samples[c].txt_len, H)))
                             for c in order]) if n_txt else np.zeros((0, H), np.float32)
        return {"plan": plan, "ws": Workspace(plan, model.dims), "x0": to_bf16(x0),
                "x": torch.empty((max(n_txt, 1), H), dtype=torch.bfloat16, device="cuda"),
                "x_img": torch.empty((n_img, H), dtype=torch.bfloat16, device="cuda"),
                "v": torch.empty((n_img, C), dtype=torch.float32, device="cuda"),
                "n_tok": plan.n_tok, "n_img": n_img}

    packed = arm(synth.cfg_samples())
    cond = arm([synth.Sample(256, 1, 64, 64, 1.0), synth.Sample(256, 1, 48, 84, 1.0)])
    unc = arm([synth.Sample(0, 1, 64, 64, 1.0), synth.Sample(0, 1, 48, 84, 1.0)])
    z0p = to_f32(synth.normal(8, "z0.packed", (packed["n_img"], C)))
    z0u = to_f32(synth.normal(8, "z0.unpacked", (cond["n_img"], C)))
    zp, zbp = z0p.clone(), z0p.to(torch.bfloat16)
    zu, zbu = z0u.clone(), z0u.to(torch.bfloat16)
    vg = torch.empty_like(packed["v"])

    def stack(a, zb, t):
        n = a["x0"].shape[0]
        if n:
            a["x"][:n].copy_(a["x0"])
        run_stack(a["plan"], model, a["x"], zb, a["x_img"], a["v"], a["ws"], t=t)

    runs = {}
    for n_steps in (4, 20):
        grid = [float(x) for x in np.linspace(1.0, 0.0, n_steps + 1)]
        tt = {id(a): [torch.full((a["plan"].n_seq,), g, dtype=torch.float32, device="cuda") for g in grid[:-1]]
              for a in (packed, cond, unc)}

        def sampler_packed():
            zp.copy_(z0p)
            zbp.copy_(zp)
            for k in range(n_steps):
                stack(packed, zbp, tt[id(packed)][k])
                mf.mf_cfg_combine(packed["plan"], C, w, packed["v"], vg)
                mf.mf_euler_step(packed["plan"], C, grid[k] - grid[k + 1], vg, zp, zbp)

        def sampler_unpacked():
            zu.copy_(z0u)
            zbu.copy_(zu)
            for k in range(n_steps):
                dt = grid[k] - grid[k + 1]
                stack(cond, zbu, tt[id(cond)][k])
                stack(unc, zbu, tt[id(unc)][k])
                mf.mf_euler_step(unc["plan"], C, dt * (1.0 - w), unc["v"], zu, None)
                mf.mf_euler_step(cond["plan"], C, dt * w, cond["v"], zu, zbu)

        result = {}
        reps = max(1, args.steps if n_steps == 4 else max(1, args.steps // 5))
        for name, fn, n_tok in (("packed", sampler_packed, packed["n_tok"]),
                                ("unpacked", sampler_unpacked, cond["n_tok"] + unc["n_tok"])):
            fn()                                   # first calls: library set-up outside the capture
            torch.cuda.synchronize()
            mf.mf_check()
            l0 = mf.mf_launch_count()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            launches = mf.mf_launch_count() - l0
            for _ in range(max(3, args.warmup)):
                g.replay()
            torch.cuda.synchronize()
            mf.mf_check()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            mf.mf_check()
            ms = e0.elapsed_time(e1) / reps
            z_out = zp if name == "packed" else zu
            z_graph = z_out.clone()
            fn()                                   # eager run: the replay must give the same bits
            torch.cuda.synchronize()
            mf.mf_check()
            result[name] = {"ms_per_sampler": round(ms, 3), "images_per_s": round(2 / (ms / 1e3), 2),
                            "tokens_per_block_fwd": n_tok, "library_launches_per_sampler": int(launches),
                            "replays_timed": reps,
                            "graph_replay_equals_eager": bool(torch.equal(z_graph, z_out))}
            del g
        result["packed_speedup"] = round(result["unpacked"]["ms_per_sampler"] / result["packed"]["ms_per_sampler"], 4)
        runs[f"steps{n_steps}"] = result
    return {"metric": "packed-CFG sampler throughput (2 prompts, 4 NR-MMDiT blocks)",
            "value": runs["steps4"]["packed"]["images_per_s"], "unit": "images/s", "n_gpus": 1,
            "steps": args.steps, "warmup": max(3, args.warmup), "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic", "graph": "whole sampler captured once per arm and step count",
            "config": {"workload": "packed CFG: 1024x1024 + 768x1344, cond (256 text) + uncond, "
                                   "4 blocks, 4 and 20 Euler steps, w = 4", "hidden": H, "heads": dims.heads},
            "steps4": runs["steps4"], "steps20": runs["steps20"],
            "packed_speedup_4": runs["steps4"]["packed_speedup"],
            "packed_speedup_20": runs["steps20"]["packed_speedup"],
            "pages_context": "1.09x-1.15x on one A100, largest for the 20-step base model (hyper.ai summary, 实验)"}


# ---------------------------------------------------------------- the reference (oracle) arm
def run_reference(args, rank, world):
    if rank != 0:
        return None
    dims = synth.FULL
    weights = synth.model_weights(dims, 1, seed=0)
    cands = synth.native_candidates(0)
    from oracle import pack as opack
    order = opack.build_plan(cands, BUDGET).order
    # size each step so that the whole run stays within about two minutes
    sub, x, z = oracle_sample(dims, weights, cands, order, 256)
    t0 = time.perf_counter()
    from oracle import model as M
    M.forward(x, z, sub, sub.t, weights, dims.heads)
    t256 = time.perf_counter() - t0
    per_step = 120.0 / max(1, args.steps + args.warmup)
    n_tok = int(min(4096, max(64, 256 * per_step / max(t256, 1e-3))))
    sub, x, z = oracle_sample(dims, weights, cands, order, n_tok)
    for _ in range(args.warmup):
        M.forward(x, z, sub, sub.t, weights, dims.heads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        M.forward(x, z, sub, sub.t, weights, dims.heads)
    el = time.perf_counter() - t0
    value = args.steps * sub.length / el
    sample = (f"fp64 NumPy oracle: embed + 1 block + final layer on one sample of pack 0 cut to "
              f"{sub.txt_len} text + {sub.lat_h}x{sub.lat_w} image tokens ({sub.length} tokens) per step")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": dict(config_dict(dims), workload=sample_workload(sub),
                                                sample_tokens=sub.length),
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    elif args.workload == "cfg":
        line = run_cfg_sampler(args, rank, world, local_rank)
    elif args.workload == "gemm":
        line = run_gemm_shapes(args, rank, world, local_rank)
    elif args.workload == "fp8block":
        line = run_fp8_block(args, rank, world, local_rank)
    elif args.workload == "train":
        line = run_train(args, rank, world, local_rank)
    elif args.workload == "lnvariants":
        line = run_ln_variants(args, rank, world, local_rank)
    elif args.workload == "attn":
        line = run_attention(args, rank, world, local_rank)
    else:
        line = run_mageflow(args, rank, world, local_rank)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
