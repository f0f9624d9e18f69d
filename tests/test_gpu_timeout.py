"""The bounded pipeline waits of the main kernels, driven to run out.

A test-only build of the library (build.build_starve: waits give up after
2 ms; msa_test_starve(k) makes CTA 0 of kernel k leave out its first Q tile)
runs in a subprocess.  For each of fwd_group, fwd_main and bwd_main the
call must report MSA_ERR_TIMEOUT within a second, the CTAs must drain and
exit (the subprocess finishes), and the same process must then run a normal
forward and backward with status OK.  A fresh process with the product
library then passes the smoke parity check against the oracle.

No wait here is unbounded: a starved wait gives up after 2 ms, every role
leaves its loop on the CTA's abort flag, and copies already armed are
drained with bounded waits before TMEM is released.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys, time, ctypes
sys.path.insert(0, ROOT)
import torch
from block_sparse_gqa_msa_gb300 import api, build, inputs
api.LIB_PATH = build.build_starve()
lib = api.lib()
lib.msa_test_starve.argtypes = [ctypes.c_int32]
lib.msa_test_starve.restype = ctypes.c_int32
dev = "cuda:0"
# documents with grouped octets (dense first blocks) and pooled tasks (the
# sparse blocks of the 2500-token document)
w = inputs.custom([2500, 700], 17)
q, k, v, do = (x.to(dev) for x in (w.q, w.k, w.v, w.do))
out = {}
def run(which, backward):
    # without dense octets the 2500-token document's later blocks go through
    # the pooled tasks, so fwd_main has work
    dense = -1 if which == 2 else 0
    plan = api.msa_build_plan(w.q2k.to(dev), w.doc_offsets.to(dev), dense_blocks=dense)
    counts = api.msa_plan_counts(plan)
    assert lib.msa_test_starve(0) == 0
    o, lse = api.msa_forward(plan, q, k, v, w.scale)
    if backward:
        assert api.msa_read_status(plan) == 0
    assert lib.msa_test_starve(which) == 0
    torch.cuda.synchronize()
    t0 = time.time()
    if backward:
        api.msa_backward(plan, q, k, v, o, lse, do, w.scale)
    else:
        plan = api.msa_build_plan(w.q2k.to(dev), w.doc_offsets.to(dev), dense_blocks=dense)
        api.msa_forward(plan, q, k, v, w.scale)
    st = api.msa_read_status(plan)
    return {"status": st, "seconds": time.time() - t0, "items": counts["items"],
            "ftasks": counts["ftasks"]}
out["fwd_group"] = run(1, False)
out["fwd_main"] = run(2, False)
out["bwd_main"] = run(3, True)
# the context is still usable: a normal forward and backward
assert lib.msa_test_starve(0) == 0
plan = api.msa_build_plan(w.q2k.to(dev), w.doc_offsets.to(dev))
o, lse = api.msa_forward(plan, q, k, v, w.scale)
api.msa_backward(plan, q, k, v, o, lse, do, w.scale)
out["after"] = api.msa_read_status(plan)
out["matmul"] = float((torch.ones(256, 256, device=dev) @ torch.ones(256, 256, device=dev))[0, 0])
print("RESULT " + json.dumps(out))
"""


def test_starved_waits_report_timeout():
    r = subprocess.run([sys.executable, "-c", CHILD.replace("ROOT", repr(ROOT))],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    line = [x for x in r.stdout.splitlines() if x.startswith("RESULT ")][-1]
    res = json.loads(line[len("RESULT "):])
    for name in ("fwd_group", "fwd_main", "bwd_main"):
        assert res[name]["status"] == 8, (name, res[name])   # MSA_ERR_TIMEOUT
        assert res[name]["seconds"] < 1.0, (name, res[name])
    assert res["fwd_group"]["items"] > 0 and res["fwd_main"]["ftasks"] > 0
    assert res["after"] == 0
    assert res["matmul"] == 256.0
    # a fresh process with the product library passes the parity check
    r = subprocess.run([sys.executable, "-c",
                        "import __graft_entry__ as g; g.smoke()"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "smoke OK" in r.stdout
