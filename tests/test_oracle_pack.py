"""Pins for the oracle's packer: a hand-worked pack, first-fit characterisation, row-map
invariants and the error cases."""
import numpy as np
import pytest

import synth
from oracle import pack as opack


def _cands(g):
    return [synth.Sample(**c) for c in g["candidates"]]


def test_hand_worked_pack(golden):
    g = golden("pack_first_fit.json")
    p = opack.build_plan(_cands(g), g["budget"])
    assert p.order.tolist() == g["order"]
    assert p.cu_seqlens.tolist() == g["cu_seqlens"]
    assert p.cu_txt.tolist() == g["cu_txt"]
    assert p.cu_img.tolist() == g["cu_img"]
    for c in g["pos_checks"]:
        assert p.pos[c["joint"]].tolist() == c["pos"], c["why"]
    assert p.txt_joint.tolist() == g["txt_joint"]
    for r, j in g["img_joint_first_last"]:
        assert p.img_joint[r] == j
    for r, t in g["img_target_checks"]:
        assert p.img_target[r] == t


def _check_first_fit(samples, budget, order):
    """First-fit with skip is characterised by: taken indices increase, and each candidate is
    taken iff it fits the budget left by the candidates taken before it."""
    taken = set(order)
    used = 0
    for i, s in enumerate(samples):
        fits = used + opack.sample_length(s) <= budget
        assert fits == (i in taken), (i, used, budget)
        if fits:
            used += opack.sample_length(s)
    assert list(order) == sorted(order)
    # greedy maximality: nothing skipped fits the final slack
    for i, s in enumerate(samples):
        if i not in taken:
            assert opack.sample_length(s) > budget - used


def _check_plan_invariants(samples, p):
    N = p.n_tok
    assert p.cu_seqlens[0] == 0 and np.all(np.diff(p.cu_seqlens) > 0)
    joint = np.concatenate([p.txt_joint, p.img_joint])
    assert np.array_equal(np.sort(joint), np.arange(N))          # a partition of [0, N)
    assert np.all(p.pos[p.txt_joint] == 0)
    for k, c in enumerate(p.order):
        s = samples[c]
        lo, hi = p.cu_seqlens[k], p.cu_seqlens[k + 1]
        assert hi - lo == opack.sample_length(s)
        assert np.all(p.txt_seq[p.cu_txt[k]:p.cu_txt[k + 1]] == k)
        assert np.all(p.img_seq[p.cu_img[k]:p.cu_img[k + 1]] == k)
        # text first, then image tokens in frame-major, row-major order
        assert np.array_equal(p.txt_joint[p.cu_txt[k]:p.cu_txt[k + 1]],
                              np.arange(lo, lo + s.txt_len))
        rows = np.arange(p.cu_img[k], p.cu_img[k + 1])
        assert np.array_equal(p.img_joint[rows], np.arange(lo + s.txt_len, hi))
        local = rows - p.cu_img[k]
        hw = s.lat_h * s.lat_w
        exp = np.stack([local // hw, (local % hw) // s.lat_w, local % s.lat_w], 1)
        assert np.array_equal(p.pos[p.img_joint[rows]], exp)
        assert np.array_equal(p.img_target[rows], (local // hw == s.frames - 1).astype(np.int32))


@pytest.mark.parametrize("seed", range(40))
def test_first_fit_random(seed):
    g = np.random.default_rng(seed)
    n = int(g.integers(0, 12))
    budget = int(g.integers(1, 200))
    samples = []
    while len(samples) < n:
        s = synth.Sample(int(g.integers(0, 20)), int(g.integers(1, 3)), int(g.integers(1, 8)),
                         int(g.integers(1, 8)), 0.5)
        if s.length <= budget:
            samples.append(s)
    p = opack.build_plan(samples, budget)
    _check_first_fit(samples, budget, p.order.tolist())
    _check_plan_invariants(samples, p)
    assert p.n_tok <= budget


@pytest.mark.parametrize("seed", range(8))
def test_native_pack_fills_budget(seed):
    cands = synth.native_candidates(seed)
    p = opack.build_plan(cands, 16384)
    _check_first_fit(cands, 16384, p.order.tolist())
    assert 12000 <= p.n_tok <= 16384


def test_cfg_pack_pairs():
    s = synth.cfg_samples()
    p = opack.build_plan(s, 17000)
    assert p.n_seq == 4 and p.n_tok == 16768
    nz = p.img_pair >= 0
    assert nz.all()
    assert np.array_equal(p.img_pair[p.img_pair], np.arange(p.n_img))   # an involution
    assert p.img_pair[0] == 4096 and p.img_pair[8192] == 8192 + 4032


def test_edit_pack():
    p = opack.build_plan(synth.edit_samples(), 17408)
    assert p.n_tok == 17408 and p.n_seq == 2
    assert p.img_target.sum() == 2 * 4096


def test_errors():
    ok = synth.Sample(4, 1, 2, 2, 0.5)
    with pytest.raises(opack.PackError) as e:
        opack.build_plan([ok], 0)
    assert e.value.code == "budget"
    with pytest.raises(opack.PackError) as e:
        opack.build_plan([ok, synth.Sample(100, 1, 1, 1, 0.5)], 50)
    assert e.value.code == "sample_too_long"
    with pytest.raises(opack.PackError):
        opack.build_plan([synth.Sample(4, 3, 2, 2, 0.5)], 50)
    with pytest.raises(opack.PackError):         # cond whose uncond partner does not fit
        opack.build_plan([synth.Sample(4, 1, 4, 4, 0.5, 1, 1), synth.Sample(0, 1, 4, 4, 0.5, 2, 0)], 25)
    with pytest.raises(opack.PackError):         # pair shapes differ
        opack.build_plan([synth.Sample(4, 1, 4, 4, 0.5, 1, 1), synth.Sample(0, 1, 4, 5, 0.5, 2, 0)], 99)


def test_empty():
    p = opack.build_plan([], 10)
    assert p.n_seq == 0 and p.n_tok == 0 and p.cu_seqlens.tolist() == [0]
