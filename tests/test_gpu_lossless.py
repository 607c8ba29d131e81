"""Losslessness of the CUDA verification (GB300 only).

D3D and DScout, "Background: speculative decoding": the output distribution
equals the target's.  Over >= 10^6 seeded trials of one fixed problem
(vocabulary 16), the first emitted token must follow P_1 and the second,
given the first draft was accepted, P_2 (chi-square, flag at p < 1e-4)."""
import numpy as np
import pytest
import scipy.special
import scipy.stats
import torch

import workloads as W
from gpu_util import run_verify

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def d3d():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import diffusion_drafted_speculative_gb300 as mod

    return mod


def _chi2_p(tokens, probs):
    obs = np.bincount(tokens, minlength=len(probs)).astype(np.float64)
    assert obs[probs == 0].sum() == 0
    keep = probs > 0
    return scipy.stats.chisquare(obs[keep], probs[keep] * obs.sum()).pvalue


@pytest.mark.parametrize("T,dt,sm_limit", [(1.0, W.DT_F32, 0), (1.0, W.DT_BF16, 0), (0.5, W.DT_F32, 0),
                                            (1.0, W.DT_BF16, 56)])
def test_gpu_lossless_chi_square(d3d, T, dt, sm_limit):
    V, B, R = 16, 3, 65536
    rng = np.random.default_rng(77)
    x = (rng.standard_normal((B, V)) * 1.5).astype(np.float32)
    z = (x[: B - 1] + rng.standard_normal((B - 1, V))).astype(np.float32)
    if dt == W.DT_BF16:
        x, z = W.bf16_to_f32(W.bf16_bits(x)), W.bf16_to_f32(W.bf16_bits(z))
    P = scipy.special.softmax(x.astype(np.float64) / T, axis=-1)
    Q = scipy.special.softmax(z.astype(np.float64) / T, axis=-1)
    first, second = [], []
    ws = None
    for call in range(16):
        r2 = np.random.default_rng(1000 + call)
        y = np.stack([r2.choice(V, size=R, p=Q[j]) for j in range(B - 1)], axis=1).astype(np.int32)
        u = W.uniform24(r2, (R, B))
        tg = np.broadcast_to(x, (R, B, V))
        dr = np.broadcast_to(z, (R, B - 1, V))
        if dt == W.DT_BF16:
            tg, dr = W.bf16_bits(tg), W.bf16_bits(dr)
        v = dict(target=np.ascontiguousarray(tg), draft=np.ascontiguousarray(dr), dtype=dt, y=y,
                 u_accept=np.ascontiguousarray(u[:, : B - 1]), u_sample=np.ascontiguousarray(u[:, B - 1]),
                 R=R, B=B, V=V, temperature=T)
        got, ws = run_verify(d3d, v, ws=ws, want_probs=False, sm_limit=sm_limit)
        first.append(got["out_tokens"][:, 0])
        second.append(got["out_tokens"][got["accept_len"] >= 1, 1])
    first, second = np.concatenate(first), np.concatenate(second)
    assert len(first) >= 1_000_000
    assert _chi2_p(first, P[0]) > 1e-4
    assert _chi2_p(second, P[1]) > 1e-4


@pytest.mark.parametrize("dt", [W.DT_F32, W.DT_BF16])
def test_gpu_lossless_chi_square_slice_launch(d3d, dt):
    # the vocabulary-slice launch (38 requests of 4 slices of 64 entries over
    # the whole device): >= 190,000 seeded trials; the sample's crossing falls
    # in any of the four slices, so the decision across slices is exercised
    V, B, R, T = 256, 3, 38, 1.0
    assert d3d.d3d_spec_verify_slice_ctas(R, B, V, dt, T, 0) == 4 * R
    rng = np.random.default_rng(78)
    x = (rng.standard_normal((B, V)) * 1.5).astype(np.float32)
    z = (x[: B - 1] + rng.standard_normal((B - 1, V))).astype(np.float32)
    if dt == W.DT_BF16:
        x, z = W.bf16_to_f32(W.bf16_bits(x)), W.bf16_to_f32(W.bf16_bits(z))
    P = scipy.special.softmax(x.astype(np.float64) / T, axis=-1)
    Q = scipy.special.softmax(z.astype(np.float64) / T, axis=-1)
    tg = np.ascontiguousarray(np.broadcast_to(x, (R, B, V)))
    dr = np.ascontiguousarray(np.broadcast_to(z, (R, B - 1, V)))
    if dt == W.DT_BF16:
        tg, dr = W.bf16_bits(tg), W.bf16_bits(dr)
    first, second = [], []
    ws = None
    for call in range(5000):
        r2 = np.random.default_rng(5000 + call)
        y = np.stack([r2.choice(V, size=R, p=Q[j]) for j in range(B - 1)], axis=1).astype(np.int32)
        u = W.uniform24(r2, (R, B))
        v = dict(target=tg, draft=dr, dtype=dt, y=y, u_accept=np.ascontiguousarray(u[:, : B - 1]),
                 u_sample=np.ascontiguousarray(u[:, B - 1]), R=R, B=B, V=V, temperature=T)
        got, ws = run_verify(d3d, v, ws=ws, want_probs=False)
        first.append(got["out_tokens"][:, 0])
        second.append(got["out_tokens"][got["accept_len"] >= 1, 1])
    first, second = np.concatenate(first), np.concatenate(second)
    assert len(first) >= 190_000
    assert _chi2_p(first, P[0]) > 1e-4
    assert _chi2_p(second, P[1]) > 1e-4
