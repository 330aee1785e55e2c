"""Failure detection without a GPU fault: a bounded device wait that runs out must
come back as CSA2_ERR_TIMEOUT through the device status word, and leave the
context usable. The wait is the streaming kernels' own bounded mbarrier wait, made
to run out on a barrier that nothing arrives at (a short limit, no trap, no hang).

The tcgen05 form of the indexer scan (selected by an environment variable read
once per process) is checked here too, by running the scan parity tests in a
child process with that form selected.
"""
import os
import subprocess
import sys

import pytest
import torch

import fp4_compressed_kv_append_b300 as K
from fp4_compressed_kv_append_b300 import _abi as A

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_timeout():
    stream = torch.cuda.current_stream().cuda_stream
    assert K.sync_status() == 0
    st = A.lib().csa2_selftest_wait_timeout(5_000_000, stream)  # 5 ms
    assert st == A.OK, A.status_str(st)
    assert K.sync_status() == A.ERR_TIMEOUT
    assert K.sync_status() == 0  # read and cleared
    # the context is still usable
    s = torch.arange(1000, dtype=torch.float32, device="cuda")[None]
    out = K.topk_select(s, 10)
    torch.cuda.synchronize()
    assert out[0].tolist() == list(range(990, 1000))
    assert K.sync_status() == 0


def test_selftest_refuses_a_budget_over_a_second():
    assert A.lib().csa2_selftest_wait_timeout(2_000_000_000, None) == A.ERR_ARG


def test_tcgen05_scan_form_parity():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, CSA2_SCAN_KERNEL="tc")
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_gpu_parity.py", "-q", "-x", "-m", "gpu",
                        "-k", "indexer_scores_within or indexer_scores_long"],
                       cwd=root, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
