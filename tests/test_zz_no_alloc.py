"""The verification entry point that allocates nothing (GB300 only).

Callers that cannot allocate device memory (a server whose memory manager
has already reserved the whole GPU, a latency-critical loop that cannot pay
for cudaMalloc's device synchronisation, a C caller with no allocator) use
d3d_spec_verify_noalloc, whose scratch is a fixed array inside the library.
This test calls it through the C ABI twice in a row, on different inputs,
and checks each result against d3d_spec_verify with a caller workspace on
the same inputs, within the tolerances of the other verification tests, and
the sampled tokens against the oracle under the same near-tie rule as the
other verification tests.  The size limit is checked at its exact edge.
The file sorts last so that a stop-at-first-failure run has already run
every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import PROB_RTOL, bf16, compare_verify, f32, i32, oracle_verify, run_verify

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def d3d():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import diffusion_drafted_speculative_gb300 as mod

    return mod


def _noalloc_via_abi(d3d, v):
    """One call of the no-allocation entry point through the raw C ABI."""
    R, B = v["R"], v["B"]
    tg, dr = (bf16(v["target"]), bf16(v["draft"])) if v["dtype"] == W.DT_BF16 else \
        (f32(v["target"]), f32(v["draft"]))
    y, ua, us = i32(v["y"]), f32(v["u_accept"]), f32(v["u_sample"])
    out = dict(accept_len=torch.full((R,), -7, dtype=torch.int32, device="cuda"),
               out_tokens=torch.full((R, B), -7, dtype=torch.int32, device="cuda"),
               num_tokens=torch.full((R,), -7, dtype=torch.int32, device="cuda"),
               alpha=torch.full((R, B - 1), float("nan"), device="cuda"),
               p=torch.full((R, B - 1), float("nan"), device="cuda"),
               q=torch.full((R, B - 1), float("nan"), device="cuda"))
    stream = torch.cuda.current_stream().cuda_stream
    rc = d3d.lib.d3d_spec_verify_noalloc(
        tg.data_ptr(), dr.data_ptr(), v["dtype"], y.data_ptr(), ua.data_ptr(), us.data_ptr(), R, B, v["V"],
        ctypes.c_float(v["temperature"]), out["accept_len"].data_ptr(), out["out_tokens"].data_ptr(),
        out["num_tokens"].data_ptr(), out["alpha"].data_ptr(), out["p"].data_ptr(), out["q"].data_ptr(), stream)
    assert rc == d3d.D3D_OK, d3d.d3d_status_string(rc)
    torch.cuda.synchronize()
    return {k: t.cpu().numpy() for k, t in out.items()}


def _same(got, ref):
    for k in ("accept_len", "num_tokens", "out_tokens"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
    for k in ("alpha", "p", "q"):
        np.testing.assert_allclose(got[k], ref[k], rtol=PROB_RTOL, atol=1e-30, err_msg=k)


def test_noalloc_matches_workspace_entry_point_twice(d3d):
    # call 1: the 16-request serving batch; call 2: another shape, dtype and
    # temperature, so anything the first call left behind would show; call 3:
    # one request, which takes the vocabulary-slice launch
    calls = [W.verify_inputs(**W.CONFIGS["serve32b"], seed=21),
             W.verify_inputs(R=64, B=5, V=12345, logits=W.DT_F32, seed=22, temperature=0.7),
             W.verify_inputs(**W.CONFIGS["async8b"], seed=24)]
    for v in calls:
        ref, _ = run_verify(d3d, v)
        got = _noalloc_via_abi(d3d, v)
        _same(got, ref)
        compare_verify(got, oracle_verify(v), min_kept=0.85, what="no-allocation entry point")


def _call_sized(d3d, R):
    """A call of R requests at B = 16, V = 151936 on placeholder pointers:
    sizes are checked before anything is enqueued."""
    x = torch.zeros(1, dtype=torch.int32, device="cuda")
    return d3d.lib.d3d_spec_verify_noalloc(x.data_ptr(), x.data_ptr(), d3d.D3D_DTYPE_BF16, x.data_ptr(), x.data_ptr(),
                                           x.data_ptr(), R, 16, 151936, ctypes.c_float(1.0), x.data_ptr(),
                                           x.data_ptr(), x.data_ptr(), None, None, None, None)


def test_noalloc_rejects_problems_beyond_its_scratch(d3d):
    # 211 requests at B = 16, V = 151936 fit the 2 MiB array, 212 do not
    assert d3d.d3d_spec_verify_workspace_size(211, 16, 151936) <= 2 << 20 < \
        d3d.d3d_spec_verify_workspace_size(212, 16, 151936)
    assert _call_sized(d3d, 212) == d3d.D3D_ERR_UNSUPPORTED
    assert _call_sized(d3d, 4096) == d3d.D3D_ERR_UNSUPPORTED


def test_noalloc_largest_batch(d3d):
    # the largest batch that fits (211 requests) runs and matches the oracle
    v = W.verify_inputs(**dict(W.CONFIGS["async8b"], R=211), seed=23)
    ref, _ = run_verify(d3d, v)
    got = _noalloc_via_abi(d3d, v)
    _same(got, ref)
    compare_verify(got, oracle_verify(v), min_kept=0.85, what="no-allocation entry point, R = 211")
