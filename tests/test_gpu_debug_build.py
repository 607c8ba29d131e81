"""The debug build (GB300 only): libd3d_debug.so is the same library compiled
with device-side internal index checks (TMA tile rows inside the request,
output rows inside the tensor, record and token indices inside their
arrays), each of which records D3D_ERR_INTERNAL in the workspace status word
and skips the access instead of trapping.  A selection of the parity tests
runs against it in a child process (D3D_LIBRARY=debug); those tests check the
results against the oracle and that every status word stays D3D_OK, so no
check may fire on valid inputs."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SELECTION = ("attn_async8b or attn_many_splits or attn_plans_under_cta_budgets or verify_async8b_full_size or "
             "verify_slice_launch or verify_one_item_per_cta or verify_sm_limit_same_results or match_planted or "
             "accept_probs_and_tau or round_on_one_stream or greedy_verify_matches_oracle")


def test_debug_build_passes_parity_subset():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    env = dict(os.environ, D3D_LIBRARY="debug")
    probe = subprocess.run([sys.executable, "-c", "import diffusion_drafted_speculative_gb300 as m; print(m.LIB_PATH)"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert probe.returncode == 0, probe.stderr
    assert probe.stdout.strip().endswith("libd3d_debug.so")
    res = subprocess.run([sys.executable, "-m", "pytest", "tests/test_gpu_parity.py", "-m", "gpu", "-q", "-x",
                          "-p", "no:cacheprovider", "-k", SELECTION], cwd=ROOT, env=env, capture_output=True,
                         text=True, timeout=1800)
    tail = (res.stdout + res.stderr)[-3000:]
    assert res.returncode == 0, tail
    assert " passed" in res.stdout and " failed" not in res.stdout, tail
