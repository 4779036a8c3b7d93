"""Host-side checks of libmageflow.so that need no GPU: it loads, it exports every entry point
mageflow.h declares, and its native packer agrees bit for bit with the oracle's packer."""
import os
import re

import numpy as np
import pytest

import synth
from oracle import pack as opack
from tests.conftest import ROOT

B = pytest.importorskip("packed_rectified_flow_packer_b300.binding")

HEADER = os.path.join(ROOT, "include", "mageflow.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mf_[a-z0-9_]+)\s*\(", src)))


def test_header_and_exports():
    names = declared_functions()
    assert len(names) >= 20
    syms = os.popen(f"nm -D --defined-only {B.LIB_PATH}").read()
    exported = set(re.findall(r" T (mf_\w+)", syms))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    assert sorted(B.EXPORTED) == names            # the binding covers exactly the header


def test_status_strings():
    for code, name in B.STATUS.items():
        assert B.mf_status_str(code) == name
    assert B.mf_version() >> 16 == 1


def _same_plan(samples, budget):
    ref = opack.build_plan(samples, budget)
    got = B.mf_pack(samples, budget)
    pairs = {"order": ref.order, "cu_seqlens": ref.cu_seqlens, "cu_txt": ref.cu_txt,
             "cu_img": ref.cu_img, "pos": ref.pos.reshape(-1), "txt_seq": ref.txt_seq,
             "txt_joint": ref.txt_joint, "img_seq": ref.img_seq, "img_joint": ref.img_joint,
             "img_pair": ref.img_pair, "img_target": ref.img_target}
    for name, want in pairs.items():
        have = got.array(name)
        assert have.dtype == np.int32
        np.testing.assert_array_equal(have, want.astype(np.int32), err_msg=name)
    roles = np.array([samples[c].cfg_role for c in ref.order], np.int32)
    np.testing.assert_array_equal(got.array("seq_role"), roles)
    i = got.info()
    assert (i.n_seq, i.n_tok, i.n_txt, i.n_img) == (ref.n_seq, ref.n_tok, ref.n_txt, ref.n_img)
    # attention work list: every (sample, 256-row query block) once, longest samples first
    items = got.array("items").reshape(-1, 2)
    lens = np.diff(ref.cu_seqlens)
    want = sorted((s, q) for s in range(ref.n_seq) for q in range(-(-lens[s] // 256)))
    assert sorted(map(tuple, items.tolist())) == want
    assert np.all(np.diff(lens[items[:, 0]]) <= 0) if len(items) else True
    return got


def test_pack_golden(golden):
    g = golden("pack_first_fit.json")
    _same_plan([synth.Sample(**c) for c in g["candidates"]], g["budget"])


@pytest.mark.parametrize("seed", range(8))
def test_pack_native_configs(seed):
    _same_plan(synth.native_candidates(seed), 16384)


def test_pack_other_configs():
    _same_plan(synth.tiny_samples(), 144)
    _same_plan(synth.gen1024_samples(), 4352)
    _same_plan(synth.cfg_samples(), 16768)
    _same_plan(synth.edit_samples(), 17408)


@pytest.mark.parametrize("seed", range(200))
def test_pack_random(seed):
    g = np.random.default_rng(1000 + seed)
    budget = int(g.integers(1, 400))
    samples = []
    for _ in range(int(g.integers(0, 16))):
        s = synth.Sample(int(g.integers(0, 40)), int(g.integers(1, 3)), int(g.integers(1, 12)),
                         int(g.integers(1, 12)), float(g.uniform()))
        if s.length <= budget:
            samples.append(s)
    _same_plan(samples, budget)


def test_pack_errors_match_oracle():
    ok = synth.Sample(4, 1, 2, 2, 0.5)
    cases = [([ok], 0, "MF_ERR_BUDGET"),
             ([ok, synth.Sample(100, 1, 1, 1, 0.5)], 50, "MF_ERR_SAMPLE_TOO_LONG"),
             ([synth.Sample(4, 3, 2, 2, 0.5)], 50, "MF_ERR_INVALID_ARG"),
             ([synth.Sample(-1, 1, 2, 2, 0.5)], 50, "MF_ERR_INVALID_ARG"),
             ([synth.Sample(4, 1, 0, 2, 0.5)], 50, "MF_ERR_INVALID_ARG"),
             ([synth.Sample(4, 1, 2, 2, 0.5, 3)], 50, "MF_ERR_INVALID_ARG"),
             ([synth.Sample(4, 1, 4, 4, 0.5, 1, 1), synth.Sample(0, 1, 4, 4, 0.5, 2, 0)], 25,
              "MF_ERR_INVALID_ARG"),
             ([synth.Sample(4, 1, 4, 4, 0.5, 1, 1), synth.Sample(0, 1, 4, 5, 0.5, 2, 0)], 99,
              "MF_ERR_INVALID_ARG")]
    for samples, budget, want in cases:
        assert B.STATUS[B.mf_pack_status(samples, budget)] == want
        with pytest.raises(opack.PackError):
            opack.build_plan(samples, budget)


def test_empty_pack():
    p = B.mf_pack([], 10)
    assert p.n_seq == 0 and p.n_tok == 0
    assert p.array("cu_seqlens").tolist() == [0]


def test_device_calls_fail_cleanly_without_gpu():
    import torch
    if torch.cuda.is_available():
        pytest.skip("has a GPU")
    p = B.mf_pack(synth.tiny_samples(), 144)
    st = B.lib.mf_plan_upload(p.handle, None)
    assert B.STATUS[st] == "MF_ERR_CUDA"
    d = B.mf_dims(256, 4, 64, 4, 256)
    assert B.mf_block_workspace_bytes(p, d) > 0
    # the fp8 block needs the bf16 workspace plus the codes and row scales of one
    # projection input (N x 4H bytes at most)
    extra = B.mf_block_fp8_workspace_bytes(p, d) - B.mf_block_workspace_bytes(p, d)
    assert extra >= p.n_tok * 4 * 256 + 4 * p.n_tok
