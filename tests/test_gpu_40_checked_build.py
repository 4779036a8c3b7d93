"""The bounds-checked build (libmageflow_checked.so, kernels compiled with -DMF_CHECKED, which
check every plan-derived index they read and report through mf_check instead of faulting) on
a workload that touches every checked kernel: the tiny stack with its loss and packed CFG, and
the training forward and backward of a ragged H = 512 pack.  It runs once with each build in a
child process: the checked build must report no bounds failure (mf_check = MF_OK) and give the
default build's results - bit for bit where the computation is deterministic, and to rounding
where reductions use atomic adds (the backward's dq accumulation and its weight, modulation and
condition gradients)."""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CHECKED = os.path.join(ROOT, "packed_rectified_flow_packer_b300", "libmageflow_checked.so")


def _run(tmp_path, checked):
    out = tmp_path / ("checked.npz" if checked else "default.npz")
    env = dict(os.environ)
    env.pop("MAGEFLOW_LIB", None)
    if checked:
        env["MAGEFLOW_LIB"] = "checked"
    r = subprocess.run([sys.executable, "-m", "tests._checked_workload", str(out)], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return dict(np.load(out))


@pytest.mark.skipif(not os.path.exists(CHECKED), reason="checked build absent (run __graft_entry__.build())")
def test_checked_build_reports_nothing_and_matches(tmp_path):
    ref = _run(tmp_path, False)
    got = _run(tmp_path, True)
    assert int(got["status"][0]) == 0 and int(ref["status"][0]) == 0
    exact = ["stack_v", "stack_x_txt", "loss", "count", "cfg", "train_x_txt", "train_x_img"]
    for k in exact:
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
    for k in ("bwd_dx_txt", "bwd_dx_img", "bwd_dc", "bwd_dw_qkv", "bwd_dw_mod"):
        scale = np.abs(ref[k]).max()
        np.testing.assert_allclose(got[k], ref[k], rtol=0, atol=1e-5 * scale, err_msg=k)
