"""Replica (weak-scaling) path of bench.py on two CPU ranks over gloo: each rank packs its own
seeds with the library's host packer, the ranks' packs are disjoint, and the whole-job figures
are the slowest rank's time and the tokens of all ranks.  The forward itself never exchanges
data between ranks (attention stays inside each sample), so these are the only collectives."""
import json
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402
import synth  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import packed_rectified_flow_packer_b300 as mf
        seeds = bench.rank_seeds(rank, n_packs=2)
        tokens = 0
        for seed in seeds:
            plan = mf.mf_pack(synth.native_candidates(seed), bench.BUDGET)
            tokens += plan.n_tok
        elapsed = 1.0 + rank  # the slower rank must win the max
        job_elapsed, job_tokens = bench.combine_over_ranks(elapsed, tokens, dist)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"seeds": seeds, "tokens": tokens, "job_elapsed": job_elapsed,
                       "job_tokens": job_tokens}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_packs_and_reduce(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert set(res[0]["seeds"]).isdisjoint(res[1]["seeds"])
    total = res[0]["tokens"] + res[1]["tokens"]
    for r in res:
        assert r["job_elapsed"] == 2.0
        assert r["job_tokens"] == total
    # the same packs packed in one process give the same token count
    import packed_rectified_flow_packer_b300 as mf
    single = sum(mf.mf_pack(synth.native_candidates(s), bench.BUDGET).n_tok
                 for s in res[0]["seeds"] + res[1]["seeds"])
    assert single == total


def test_one_rank_needs_no_process_group():
    assert bench.combine_over_ranks(3.5, 1234, None) == (3.5, 1234)
