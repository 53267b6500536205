"""Bounded waits end a kernel with a status instead of hanging it.

Every mbarrier wait of the tensor-core kernels gives up after the library's
wait budget (FA_WAIT_LIMIT_MS, read once per process).  A wait that runs out
records FA_ERR_TIMEOUT in the library's status word and raises the CTA's abort
flag.  Every role then stops, the drains wait for the CTA's own copies and
MMAs in flight, and TMEM is freed.  The host reads the status with
fa_device_status(), and the CUDA context stays usable.

Each case runs in a child process whose budget is 0.2 us. The MMA warp's first
wait, for the Q tile, needs a copy from device memory and cannot be met that
fast, so the budget always runs out. No fault is injected and nothing is
left to hang: the drains keep a budget of their own.
"""
import json
import os
import subprocess
import sys

import pytest

import exact_tiled_attention_23_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FA_ERR_TIMEOUT = 4
STATUS_TIMEOUT_BIT = 0x1

CHILD = r"""
import json, sys
sys.path.insert(0, sys.argv[2])
import torch
import exact_tiled_attention_23_gb300 as fa
import workloads

case = sys.argv[1]
inp = workloads.make_case(1, 4, 2048, 128, dtype="bf16", causal=True, seed=11)
q, k, v = (x.cuda() for x in (inp.q, inp.k, inp.v))
if case == "bwd":
    # any O and finite LSE do: the kernel gives up before their values matter
    o = torch.randn_like(q)
    d_o = torch.randn_like(q)
    lse = torch.zeros(q.shape[:3], device="cuda")
    fa.backward(q, k, v, o, d_o, lse, causal=True)
elif case == "splitkv":
    fa.forward(q, k, v, causal=True, splits=2)
else:
    fa.forward(q, k, v, causal=True)
torch.cuda.synchronize()
status = fa.fa_device_status(None)
detail = fa.fa_last_error_detail()
total = torch.ones(1 << 20, device="cuda").sum().item()
status_after = fa.fa_device_status(None)
print(json.dumps({"status": status, "detail": detail, "sum": total, "status_after": status_after}))
"""


@pytest.fixture(scope="module", autouse=True)
def built():
    fa.build()
    fa.load()


@pytest.mark.gpu
@pytest.mark.parametrize("case, tiles", [("fwd", "2"), ("fwd", "1"), ("fwd", "3"), ("splitkv", ""), ("bwd", "")],
                         ids=["two_tile", "one_tile", "split_rows", "splitkv", "bwd"])
def test_a_wait_that_runs_out_reports_a_timeout(case, tiles):
    env = dict(os.environ, FA_WAIT_LIMIT_MS="0.0002")
    env.pop("FA_FWD_TILES", None)
    if tiles:
        env["FA_FWD_TILES"] = tiles
    run = subprocess.run([sys.executable, "-c", CHILD, case, ROOT], env=env, capture_output=True,
                         text=True, timeout=120)
    assert run.returncode == 0, run.stderr[-2000:]
    result = json.loads(run.stdout.strip().splitlines()[-1])
    assert result["status"] == FA_ERR_TIMEOUT, result
    assert result["detail"] & STATUS_TIMEOUT_BIT, result
    # the context still runs work, and reading the status cleared it
    assert result["sum"] == float(1 << 20), result
    assert result["status_after"] == 0, result
