"""The persisted calibration profile on the GPU.

One process calibrates and tunes a shape, then saves its profile; a second
process, given the file through CREDIT_PROFILE, plans that shape with
credit_plan alone -- no calibration, no timing -- and gets the tuned plan
(an L2-tail plan here, which the static rule never chooses).  The same file
made stale (another SM count) is rejected, and the second process falls
back to the static rule.  CREDIT_FORCE overrides the automatic plan where
the named plan is legal and is ignored where it is not."""
import json
import os
import subprocess
import sys

import pytest
import torch

from dsmem_thread_block_gb300 import _credit as C

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SHAPE = (C.RMSNORM, 64, 786432, C.BF16)  # 1.5 MB rows: only clusters can stage them

CHILD = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
from dsmem_thread_block_gb300 import _credit as C
op, rows, cols, dt = (int(a) for a in sys.argv[2:6])
p = C.credit_plan(op, rows, cols, dt, 0)
print(json.dumps({k: (float(v) if isinstance(v, float) else int(v)) for k, v in p.as_dict().items()}))
"""


def _child(env_extra):
    env = dict(os.environ)
    env.pop("CREDIT_PROFILE", None)
    env.pop("CREDIT_FORCE", None)
    env.update(env_extra)
    out = subprocess.run([sys.executable, "-c", CHILD, ROOT, *(str(a) for a in SHAPE)], env=env,
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    return json.loads(out.stdout.strip().splitlines()[-1])


def test_second_process_plans_from_the_saved_profile(tmp_path):
    dev = torch.cuda.current_device()
    path = str(tmp_path / "profile.json")
    C.credit_calibrate(dev, 3, path)  # raises on failure
    assert C.credit_profile_check(path, C.credit_device_key(dev)) == C.OK
    op, rows, cols, dt = SHAPE
    tuned, _ = C.credit_plan_profiled(op, rows, cols, dt, C.BF16, dev, 5, 16)
    assert C.credit_save_profile(dev, path) == C.OK
    d = json.load(open(path))
    assert d["library"] == C.credit_version() and len(d["plans"]) >= 1
    assert len(d["dsmem"]["barrier_ns"]) == 17

    got = _child({"CREDIT_PROFILE": path})
    for f in ("variant", "cluster_size", "threads", "staged_elems", "slice_elems", "smem_bytes",
              "rows_per_cluster", "exchange"):
        assert got[f] == getattr(tuned, f), (f, got, tuned)
    assert abs(got["pred_us"] - tuned.pred_us) <= 1e-3 * tuned.pred_us

    # the same profile, stale: another SM count -> rejected; the static rule
    d["device"]["sms"] += 1
    stale = str(tmp_path / "stale.json")
    json.dump(d, open(stale, "w"))
    assert C.credit_load_profile(dev, stale) == C.ERR_NOT_CALIBRATED
    static = _child({"CREDIT_PROFILE": stale})
    plain = _child({})
    assert static == plain
    # a process given a missing profile plans statically as well, and the
    # file it names is only written once it calibrates or tunes
    missing = str(tmp_path / "missing.json")
    assert _child({"CREDIT_PROFILE": missing}) == plain
    assert not os.path.exists(missing)


def test_force_switch():
    got = _child({"CREDIT_FORCE": "cluster:12"})
    assert got["variant"] == C.CLUSTER and got["cluster_size"] == 12
    got = _child({"CREDIT_FORCE": "cluster:10:s36864"})
    assert got["cluster_size"] == 10 and got["staged_elems"] == 36864
    got = _child({"CREDIT_FORCE": "cluster:12:s8192:t128"})
    assert got["cluster_size"] == 12 and got["staged_elems"] == 8192 and got["threads"] == 128
    got = _child({"CREDIT_FORCE": "twopass"})
    assert got["variant"] == C.TWO_PASS
    # illegal for this shape (a 1.5 MB row in one CTA) or malformed: ignored
    plain = _child({})
    assert _child({"CREDIT_FORCE": "cluster:1"}) == plain
    assert _child({"CREDIT_FORCE": "cluster:banana"}) == plain
    assert _child({"CREDIT_FORCE": "cluster:12:s8192:t100"}) == plain  # not whole warps
