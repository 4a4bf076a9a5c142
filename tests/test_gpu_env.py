"""RMSNORM_FORCE_VARIANT: the environment variable that replaces the automatic
choice of every device call, read once per process -- so each case runs in a
fresh child process -- and checked against the oracle there."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")

# The child: one call through rms_norm, the variant that ran, and the
# comparison with the oracle (the same helper every GPU parity test uses).
CHILD = r"""
import json, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import torch
import rmsnorm_fwd_gb300 as rn
from rmsnorm_fwd_gb300 import inputs
from _parity import compare, from_device, to_device
rows, hidden, dtype = {rows}, {hidden}, {dtype!r}
x, w = inputs.random_case(rows, hidden, dtype, seed=hidden)
rn.ensure_context(0)
out = {{}}
try:
    y = rn.rms_norm(to_device(x, dtype), to_device(w, dtype), 1e-6)
    torch.cuda.synchronize()
    out["variant"] = rn.rmsnorm_last_variant()
    compare(from_device(y, dtype), x, w, 1e-6, dtype)
    out["parity"] = True
except rn.RmsnormError as e:
    out["status"] = e.status
print(json.dumps(out))
"""


def run_child(env_value, rows, hidden, dtype):
    env = dict(os.environ)
    if env_value is None:
        env.pop("RMSNORM_FORCE_VARIANT", None)
    else:
        env["RMSNORM_FORCE_VARIANT"] = env_value
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), rows=rows, hidden=hidden,
                        dtype=dtype)
    res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    return json.loads(res.stdout.strip().splitlines()[-1]), res.stderr


@pytest.mark.parametrize("value,expect", [("generic", 5), ("staged", 3), ("persistent", 4),
                                          ("1", 1), ("cta_per_row", 2)])
def test_forced_variant_runs_that_body(value, expect):
    out, _ = run_child(value, 96, 1024, "bf16")
    assert out == {"variant": expect, "parity": True}


@pytest.mark.parametrize("value,rows,hidden,status", [
    ("grid", 96, 1024, 9),          # RMSNORM_ERR_VARIANT: the grid barrier takes rows > 256 KiB
    ("cta_per_row", 64, 33, 7)])    # RMSNORM_ERR_MISALIGNED: 66-byte rows, no 16-byte vectors
def test_forced_variant_that_cannot_take_the_shape_is_refused(value, rows, hidden, status):
    import rmsnorm_fwd_gb300 as rn
    assert status in (rn.ERR_VARIANT, rn.ERR_MISALIGNED)
    out, _ = run_child(value, rows, hidden, "bf16")
    assert out == {"status": status}


def test_unset_or_unknown_value_leaves_the_automatic_choice():
    auto, _ = run_child(None, 96, 1024, "bf16")
    assert auto["parity"] is True
    out, err = run_child("fastest", 96, 1024, "bf16")
    assert out == auto and "RMSNORM_FORCE_VARIANT=fastest not understood" in err
