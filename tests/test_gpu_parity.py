"""CUDA path vs oracle, element by element, on seeded inputs (GB300 only).

Sizes span several tiles and ragged tails; the full workloads of the
benchmark shapes are checked on all tokens of sampled heads (attention) and
on whole rows (verification)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import (NEAR_TIE, PROB_RTOL, SAMPLE_BAND, assert_attn_close, compare_verify, oracle_verify, run_attn,
                      run_match, run_verify)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def d3d():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import diffusion_drafted_speculative_gb300 as mod

    return mod


def _oracle_heads(a, heads):
    ref = np.zeros((a["q"].shape[0], a["Hq"], a["d"]))
    for h in heads:
        ref[:, h] = oracle.packed_attn(a, heads=(h, h + 1))[:, h]
    return ref


# ------------------------------------------------------------------ attention
@pytest.mark.parametrize("seed", [0, 1])
def test_attn_tiny_config(d3d, seed):
    a = W.attn_inputs(**W.CONFIGS["tiny"], seed=seed)
    got, ws = run_attn(d3d, a)
    assert_attn_close(got, oracle.packed_attn(a), "tiny")
    assert d3d.d3d_workspace_status(ws) == 0


@pytest.mark.parametrize("B,C,F,L,Hq,Hkv,d", [
    (16, 12, 2, 300, 4, 1, 128),    # async layout, GQA 4, ragged prefix tail
    (16, 4, 1, 129, 8, 2, 64),      # N = 80
    (8, 3, 2, 0, 2, 2, 64),         # no prefix at all, G = 1
    (16, 2, 2, 1000, 16, 2, 128),   # G = 8
    (4, 5, 3, 77, 4, 4, 128),       # tiny blocks
    (32, 1, 1, 513, 2, 1, 64),      # C = 1: current + all-accept only
])
def test_attn_async_layouts(d3d, B, C, F, L, Hq, Hkv, d):
    a = W.attn_inputs(R=1, L=L, Hq=Hq, Hkv=Hkv, d=d, B=B, C=C, F=F, layout="async", seed=3)
    got, _ = run_attn(d3d, a)
    assert_attn_close(got, oracle.packed_attn(a), "async B%d C%d F%d" % (B, C, F))


def test_attn_peaky_softmax(d3d):
    a = W.attn_inputs(R=1, L=700, Hq=4, Hkv=2, d=128, B=16, C=3, F=2, layout="async", seed=4, k_scale=4.0)
    got, _ = run_attn(d3d, a)
    assert_attn_close(got, oracle.packed_attn(a), "k x 4")


def test_attn_ragged_batch_with_empty_request(d3d):
    segs = W.async_segments(8, 3, 2)
    a = W.attn_inputs(R=3, L=(0, 400), Hq=8, Hkv=2, d=128, seed=5, segs=segs)
    # make request 1 empty (no packed tokens, no segments)
    n = int(segs[:, 1].sum())
    keep_q = np.r_[0:n, 2 * n:3 * n]
    a["q"], a["kn"], a["vn"] = a["q"][keep_q], a["kn"][keep_q], a["vn"][keep_q]
    a["segs"] = np.concatenate([segs, segs]).astype(np.int32)
    a["cu_q"] = np.array([0, n, n, 2 * n], np.int32)
    a["cu_seg"] = np.array([0, len(segs), len(segs), 2 * len(segs)], np.int32)
    got, ws = run_attn(d3d, a)
    assert_attn_close(got, oracle.packed_attn(a), "ragged")
    assert d3d.d3d_workspace_status(ws) == 0


def test_attn_random_segment_tables(d3d):
    rng = np.random.default_rng(6)
    for t in range(6):
        rows, q, causal = [], 0, []
        for s in range(int(rng.integers(1, 12))):
            ln = int(rng.integers(1, 40))
            mode = int(rng.integers(0, 2))
            par, plen = -1, 0
            if causal and rng.random() < 0.7:
                par = int(rng.choice(causal))
                plen = int(rng.integers(0, rows[par][1] + 1))
            rows.append([q, ln, mode, par, plen])
            if mode == 0 and par == -1:
                causal.append(s)
            q += ln
        a = W.attn_inputs(R=1, L=int(rng.integers(0, 300)), Hq=4, Hkv=2, d=64, seed=t,
                          segs=np.array(rows, np.int32))
        got, _ = run_attn(d3d, a)
        assert_attn_close(got, oracle.packed_attn(a), "random table %d" % t)


def test_attn_async8b_full_size_sampled_heads(d3d):
    a = W.attn_inputs(**W.CONFIGS["async8b"], seed=0)
    got, ws = run_attn(d3d, a)
    heads = [0, 5, 31]
    ref = _oracle_heads(a, heads)
    assert_attn_close(got[:, heads], ref[:, heads], "async8b")
    assert np.isfinite(got).all()
    assert d3d.d3d_workspace_status(ws) == 0


def test_attn_long_block_full_size_sampled_heads(d3d):
    a = W.attn_inputs(**W.CONFIGS["long_block"], seed=1)
    got, _ = run_attn(d3d, a)
    heads = [0, 17]
    assert_attn_close(got[:, heads], _oracle_heads(a, heads)[:, heads], "long_block")


def test_attn_serve32b_full_size_sampled_head(d3d):
    a = W.attn_inputs(**W.CONFIGS["serve32b"], seed=2)
    got, _ = run_attn(d3d, a)
    heads = [37]
    assert_attn_close(got[:, heads], _oracle_heads(a, heads)[:, heads], "serve32b")
    assert np.isfinite(got).all()


@pytest.mark.parametrize("C,F", [(4, 1), (16, 5)])
def test_attn_sweep_full_size_sampled_head(d3d, C, F):
    a = W.attn_inputs(**dict(W.CONFIGS["sweep"], C=C, F=F), seed=3)
    assert a["q"].shape[0] == oracle.n_async(16, C, F)
    got, _ = run_attn(d3d, a)
    heads = [9]
    assert_attn_close(got[:, heads], _oracle_heads(a, heads)[:, heads], "sweep C%d F%d" % (C, F))


@pytest.mark.parametrize("cfg,heads", [("target_verify", [0, 13, 31]), ("train_mask", [0, 22])])
def test_attn_target_verify_and_training_layouts(d3d, cfg, heads):
    # the same kernel on two more layouts: the target's verification pass
    # (one causal block over an 8192-token KV, key splits) and the
    # training-time packed pass (a causal 2048-token response plus 128 anchor
    # blocks that see the response before their anchor; 129 segments, more
    # than the kernel stages in shared memory)
    a = W.attn_inputs(**W.CONFIGS[cfg], seed=60)
    got, ws = run_attn(d3d, a)
    assert np.isfinite(got).all()
    assert_attn_close(got[:, heads], _oracle_heads(a, heads)[:, heads], cfg)
    assert d3d.d3d_workspace_status(ws) == 0


def test_attn_wait_runs_out_reports_status_and_context_survives(d3d):
    # failure detection without a GPU fault: the producer skips the first key
    # tile, the consumer's bounded wait runs out, the kernel records the
    # timeout in the status word and returns; the next call is correct
    a = W.attn_inputs(**W.CONFIGS["tiny"], seed=9)
    d3d.d3d_debug_inject_fault(1)
    try:
        _, ws = run_attn(d3d, a)
    finally:
        d3d.d3d_debug_inject_fault(0)
    assert d3d.d3d_workspace_status(ws, clear=True) == d3d.D3D_ERR_DEVICE_TIMEOUT
    got, ws2 = run_attn(d3d, a)
    assert_attn_close(got, oracle.packed_attn(a), "after a timed-out call")
    assert d3d.d3d_workspace_status(ws2) == 0


def test_attn_bad_device_descriptor_sets_status(d3d):
    a = W.attn_inputs(R=1, L=64, Hq=2, Hkv=1, d=64, B=8, C=3, F=2, layout="async", seed=7)
    a["segs"] = a["segs"].copy()
    a["segs"][1, 4] = 99  # parent_len longer than the parent: only the device can see it
    got, ws = run_attn(d3d, a)
    assert d3d.d3d_workspace_status(ws, clear=True) == d3d.D3D_ERR_DEVICE_INPUT
    assert d3d.d3d_workspace_status(ws) == d3d.D3D_OK
    rows = slice(int(a["segs"][1, 0]), int(a["segs"][1, 0] + a["segs"][1, 1]))
    assert (got[rows] == 0).all()


def test_attn_many_splits_and_bad_descriptor(d3d):
    # one query-tile pair over a long prefix: the planner cuts the key list
    # into many splits, so the merge path runs with a large split count
    a = W.attn_inputs(R=1, L=4096, Hq=4, Hkv=1, d=128, B=8, C=3, F=2, layout="async", seed=8)
    got, ws = run_attn(d3d, a)
    assert_attn_close(got, oracle.packed_attn(a), "many splits")
    assert d3d.d3d_workspace_status(ws) == 0
    # the same with a descriptor only the device can see is wrong: the rows of
    # that segment come out as zeros, every other row is still correct
    bad = dict(a, segs=a["segs"].copy())
    bad["segs"][2, 4] = 99
    got2, ws2 = run_attn(d3d, bad)
    assert d3d.d3d_workspace_status(ws2, clear=True) == d3d.D3D_ERR_DEVICE_INPUT
    rows = np.zeros(got2.shape[0], bool)
    rows[int(bad["segs"][2, 0]):int(bad["segs"][2, 0] + bad["segs"][2, 1])] = True
    assert (got2[rows] == 0).all()
    assert_attn_close(got2[~rows], oracle.packed_attn(a)[~rows], "other rows")


# ------------------------------------------------------------------ each attention kernel
KERNELS = {1: "one tile per CTA", 2: "two tiles per CTA", 3: "CTA pairs"}


@pytest.fixture
def force_kernel(d3d):
    yield d3d.d3d_debug_force_attn_kernel
    d3d.d3d_debug_force_attn_kernel(0)


def _ragged_with_empty_request():
    segs = W.async_segments(8, 3, 2)
    a = W.attn_inputs(R=3, L=(0, 400), Hq=8, Hkv=2, d=128, seed=5, segs=segs)
    n = int(segs[:, 1].sum())
    keep_q = np.r_[0:n, 2 * n:3 * n]
    a["q"], a["kn"], a["vn"] = a["q"][keep_q], a["kn"][keep_q], a["vn"][keep_q]
    a["segs"] = np.concatenate([segs, segs]).astype(np.int32)
    a["cu_q"] = np.array([0, n, n, 2 * n], np.int32)
    a["cu_seg"] = np.array([0, len(segs), len(segs), 2 * len(segs)], np.int32)
    return a


def _kernel_case(case):
    if case == "async8b":  # the benchmark shape: 12 query tiles per KV head
        return W.attn_inputs(**W.CONFIGS["async8b"], seed=3), [0, 13, 31]
    if case == "odd_tiles":  # 3 query tiles per request and KV head: a pair with one tile past the request
        return W.attn_inputs(R=2, L=(100, 700), Hq=32, Hkv=8, d=128, B=16, C=4, F=1, layout="async", seed=4), \
            [0, 7, 30]
    if case == "empty_request":
        return _ragged_with_empty_request(), list(range(8))
    if case == "g8":  # 8 query heads per KV head, 16 tokens per tile, ragged prefix tail
        return W.attn_inputs(R=1, L=1000, Hq=16, Hkv=2, d=128, B=16, C=2, F=2, layout="async", seed=6), [0, 9, 15]
    if case == "peaky":  # large logits: the running max grows by more than 2^8 between tiles
        return W.attn_inputs(R=1, L=700, Hq=4, Hkv=2, d=128, B=16, C=3, F=2, layout="async", seed=4,
                             k_scale=4.0), [0, 1, 2, 3]
    raise ValueError(case)


@pytest.mark.parametrize("kind", sorted(KERNELS))
@pytest.mark.parametrize("case", ["async8b", "odd_tiles", "empty_request", "g8", "peaky"])
def test_attn_each_kernel(d3d, force_kernel, kind, case):
    # every kernel the plan may pick gives the oracle's result on the same
    # inputs; the CTA-pair kernel rounds each request's query tiles up to
    # pairs, so its CTA count is even
    a, heads = _kernel_case(case)
    force_kernel(kind)
    n = d3d.d3d_packed_draft_attn_ctas(a["R"], a["Hq"], a["Hkv"], a["d"], a["max_q"], a["max_prefix"], 0)
    if kind == 3:
        TQ = 128 // (a["Hq"] // a["Hkv"])
        MT = (a["max_q"] + TQ - 1) // TQ
        assert n == a["R"] * a["Hkv"] * ((MT + 1) // 2 * 2), "CTA pairs not planned"
    got, ws = run_attn(d3d, a)
    assert d3d.d3d_workspace_status(ws) == 0
    assert_attn_close(got[:, heads], _oracle_heads(a, heads)[:, heads], "%s, %s" % (case, KERNELS[kind]))


def test_attn_pair_kernel_wait_runs_out(d3d, force_kernel):
    # the failure-injection path on the CTA-pair kernel: both CTAs of every
    # pair skip their first key-tile half, the issuing CTA's bounded wait
    # runs out and both give up theirs; the next call is correct
    a = W.attn_inputs(R=1, L=256, Hq=4, Hkv=1, d=128, B=16, C=3, F=2, layout="async", seed=9)
    force_kernel(3)
    d3d.d3d_debug_inject_fault(1)
    try:
        _, ws = run_attn(d3d, a)
    finally:
        d3d.d3d_debug_inject_fault(0)
    assert d3d.d3d_workspace_status(ws, clear=True) == d3d.D3D_ERR_DEVICE_TIMEOUT
    got, ws2 = run_attn(d3d, a)
    assert_attn_close(got, oracle.packed_attn(a), "after a timed-out call")
    assert d3d.d3d_workspace_status(ws2) == 0


@pytest.mark.parametrize("Hq", [32, 64])
def test_attn_single_request_offsets_checked(d3d, Hq):
    # one request: the kernel takes its offsets from the totals (the contract
    # fixes them) and checks the device arrays afterwards; 32 query heads run
    # the one-tile kernel, 64 the two-tile one.  Offsets that disagree with
    # the totals void the whole output and set the status
    a = W.attn_inputs(R=1, L=1024, Hq=Hq, Hkv=8, d=128, B=16, C=12, F=2, layout="async", seed=9)
    got, ws = run_attn(d3d, a)
    heads = [0, 5, Hq - 1]
    assert_attn_close(got[:, heads], _oracle_heads(a, heads)[:, heads], "single request")
    assert d3d.d3d_workspace_status(ws) == 0
    for key, val in (("cu_prefix", [0, int(a["cu_prefix"][1]) - 128]), ("cu_q", [0, int(a["cu_q"][1]) - 16]),
                     ("cu_seg", [0, int(a["cu_seg"][1]) - 1])):
        bad = dict(a, **{key: np.array(val, dtype=np.int32)})
        got2, ws2 = run_attn(d3d, bad)
        assert d3d.d3d_workspace_status(ws2, clear=True) == d3d.D3D_ERR_DEVICE_INPUT, key
        assert (got2 == 0).all(), key


@pytest.mark.parametrize("cfg", [W.CONFIGS["async8b"],  # one request, the one-tile kernel
                                 dict(R=4, L=(100, 900), Hq=64, Hkv=8, d=128, B=16, C=12, F=2, layout="async")])
def test_attn_after_dependent_reads_the_previous_output(d3d, cfg):
    # D3D_ATTN_AFTER_DEPENDENT: the second attention takes the first one's
    # output as its queries and may start while the first still runs (the
    # first leaves SMs free); it must read those queries only once they are
    # written: the chained result equals the one of two plain launches
    from gpu_util import bf16, i32
    a = W.attn_inputs(**cfg, seed=31)
    t = {k: bf16(a[k]) for k in ("q", "kp", "vp", "kn", "vn")}
    ix = {k: i32(a[k]) for k in ("segs", "cu_prefix", "cu_q", "cu_seg")}
    ws = d3d.new_workspace(d3d.d3d_packed_draft_attn_workspace_size(a["R"], a["Hq"], a["Hkv"], a["d"], a["max_q"],
                                                                    a["max_prefix"]))
    budget = d3d.d3d_packed_draft_attn_ctas(a["R"], a["Hq"], a["Hkv"], a["d"], a["max_q"], a["max_prefix"], 0)
    budget = max(1, min(budget, torch.cuda.get_device_properties(0).multi_processor_count // 2))

    def att(q, out, dep):
        d3d.d3d_packed_draft_attn(q, t["kp"], t["vp"], t["kn"], t["vn"], ix["segs"], ix["cu_prefix"], ix["cu_q"],
                                  ix["cu_seg"], a["max_q"], a["max_prefix"], a["scale"], out, ws,
                                  max_ctas=budget, after_dependent=dep)
    mid = torch.full_like(t["q"], float("nan"))
    att(t["q"], mid, False)
    want = torch.full_like(t["q"], float("nan"))
    att(mid.clone(), want, False)
    torch.cuda.synchronize()
    assert torch.isfinite(want.float()).all()
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for _ in range(4):
            mid2 = torch.full_like(t["q"], float("nan"))
            got = torch.full_like(t["q"], float("nan"))
            att(t["q"], mid2, False)
            att(mid2, got, True)
            att(got, torch.empty_like(got), True)  # a third in the chain; its output is not checked
            st.synchronize()
            assert torch.equal(mid2, mid)
            assert torch.equal(got, want)
    assert d3d.d3d_workspace_status(ws) == 0


# ------------------------------------------------------------------ verification
@pytest.mark.parametrize("seed", range(3))
def test_verify_tiny_config_batched(d3d, seed):
    v = W.verify_inputs(**dict(W.CONFIGS["tiny"], R=256), seed=seed)
    got, ws = run_verify(d3d, v)
    compare_verify(got, oracle_verify(v), what="tiny")
    assert d3d.d3d_workspace_status(ws) == 0


@pytest.mark.parametrize("seed", range(3))
def test_verify_async8b_full_size(d3d, seed):
    # the benchmark's verification shape (B = 16, V = 151936) over 64 requests,
    # so that the bit-exact comparison covers many draws
    v = W.verify_inputs(**dict(W.CONFIGS["async8b"], R=64), seed=seed)
    got, _ = run_verify(d3d, v)
    compare_verify(got, oracle_verify(v), min_kept=0.9, what="async8b x64")


def test_verify_serve32b_batch(d3d):
    v = W.verify_inputs(**dict(W.CONFIGS["serve32b"], R=64), seed=1)
    got, _ = run_verify(d3d, v)
    compare_verify(got, oracle_verify(v), min_kept=0.9, what="serve32b x64")


@pytest.mark.parametrize("sigma", [0.25, 0.5, 1.0])
def test_verify_long_block_sigma_sweep(d3d, sigma):
    v = W.verify_inputs(**dict(W.CONFIGS["long_block"], R=32, sigma=sigma), seed=2)
    got, _ = run_verify(d3d, v)
    compare_verify(got, oracle_verify(v), min_kept=0.9, what="long block sigma %g" % sigma)


@pytest.mark.parametrize("V", [1, 7, 1000, 8191, 8193, 12345, 16384])
@pytest.mark.parametrize("dt", [W.DT_F32, W.DT_BF16])
def test_verify_ragged_vocab(d3d, V, dt):
    v = W.verify_inputs(R=64, B=5, V=V, logits=dt, seed=V)
    got, _ = run_verify(d3d, v)
    compare_verify(got, oracle_verify(v), min_kept=0.9, what="V=%d" % V)


@pytest.mark.parametrize("B,T", [(2, 1.0), (3, 0.7), (16, 2.0), (64, 1.0)])
def test_verify_block_sizes_and_temperature(d3d, B, T):
    v = W.verify_inputs(R=128, B=B, V=2048, logits=W.DT_BF16, seed=B, temperature=T)
    got, _ = run_verify(d3d, v)
    compare_verify(got, oracle_verify(v), min_kept=0.9, what="B=%d T=%g" % (B, T))


def test_verify_high_acceptance_and_bonus_path(d3d):
    # draft == target rows: every draft accepted, the bonus comes from P_B
    v = W.verify_inputs(R=256, B=8, V=3000, logits=W.DT_F32, sigma=0.0, seed=9)
    got, _ = run_verify(d3d, v)
    ref = oracle_verify(v)
    assert (ref["accept_len"] == 7).all()
    compare_verify(got, ref)


@pytest.mark.parametrize("R,B,V,dt,sigma", [(1, 16, 151936, W.DT_BF16, 0.5), (2, 5, 12345, W.DT_F32, 0.5),
                                             (2, 16, 70001, W.DT_BF16, 1.0), (3, 2, 8193, W.DT_F32, 0.5),
                                             (1, 64, 16384, W.DT_BF16, 0.25), (5, 7, 9, W.DT_F32, 0.5),
                                             (2, 8, 3000, W.DT_F32, 0.0)])
def test_verify_one_item_per_cta(d3d, R, B, V, dt, sigma):
    # few requests: every (request, position, chunk) item has a CTA of its own,
    # and the sample reuses phase A's exponentials from registers
    kept = total = 0
    for seed in range(8):
        v = W.verify_inputs(R=R, B=B, V=V, logits=dt, sigma=sigma, seed=seed + 31 * B)
        got, ws = run_verify(d3d, v)
        ref = oracle_verify(v)
        if sigma == 0.0:
            assert (ref["accept_len"] == B - 1).all()
        kept += compare_verify(got, ref, min_kept=0.0, what="R=%d B=%d V=%d seed %d" % (R, B, V, seed))[0]
        total += R
        assert d3d.d3d_workspace_status(ws) == 0
    assert kept >= 0.75 * total, "compared %d of %d draws" % (kept, total)


@pytest.mark.parametrize("sm_limit", [1, 7, 56, 151])
def test_verify_sm_limit_same_results(d3d, sm_limit):
    # an SM limit changes how the work is spread: 512-thread CTAs over
    # 16384-entry chunks, one CTA per SM.  Probabilities may differ from the
    # unlimited launch in the last bit (another summation order); both meet
    # the oracle under the same tolerances
    for v in (W.verify_inputs(**dict(W.CONFIGS["async8b"], R=24), seed=3),
              W.verify_inputs(R=40, B=6, V=9000, logits=W.DT_F32, seed=4)):
        ref = oracle_verify(v)
        free, ws = run_verify(d3d, v)
        lim, ws2 = run_verify(d3d, v, sm_limit=sm_limit)
        compare_verify(free, ref, min_kept=0.85, what="R=%d unlimited" % v["R"])
        compare_verify(lim, ref, min_kept=0.85, what="R=%d sm_limit %d" % (v["R"], sm_limit))
        for k in ("alpha", "p", "q"):
            np.testing.assert_allclose(lim[k], free[k], rtol=1e-6, atol=1e-30, err_msg=k)
        assert d3d.d3d_workspace_status(ws2) == 0


@pytest.mark.parametrize("cfg,over,sm_limit", [("async8b", {}, 0), ("async8b", {}, 56), ("async8b", dict(R=2), 0),
                                              ("async8b", dict(R=4, B=4), 56), ("tiny", dict(R=38, V=256), 0),
                                              ("long_block", {}, 0), ("async8b", dict(logits=W.DT_F32, V=32000), 0)])
def test_verify_slice_launch_matches_oracle_and_chunked(d3d, cfg, over, sm_limit):
    # one CTA per (request, vocabulary slice) with the slice's rows resident in
    # shared memory; the same inputs under an SM limit of 8 (too few SMs for
    # resident slices) take the chunked launch.  Both meet the oracle, and
    # their probabilities agree to the last bits
    v = W.verify_inputs(**dict(W.CONFIGS[cfg], **over), seed=71)
    R, B, V, dt, T = v["R"], v["B"], v["V"], v["dtype"], v.get("temperature", 1.0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = d3d.d3d_spec_verify_slice_ctas(R, B, V, dt, T, sm_limit)
    assert 0 < n <= (sm_limit or sms) and n % R == 0
    got, ws = run_verify(d3d, v, sm_limit=sm_limit)
    ref = oracle_verify(v)
    compare_verify(got, ref, min_kept=0.75, what="%s slices %d" % (cfg, n))
    assert d3d.d3d_workspace_status(ws) == 0
    assert d3d.d3d_spec_verify_slice_ctas(R, B, V, dt, T, 8) == 0
    chunked, _ = run_verify(d3d, v, sm_limit=8)
    compare_verify(chunked, ref, min_kept=0.75, what="%s chunked" % cfg)
    for k in ("alpha", "p", "q"):
        np.testing.assert_allclose(got[k], chunked[k], rtol=1e-6, atol=1e-30, err_msg=k)


def test_verify_slice_shapes(d3d):
    # the slice launch needs 16-byte aligned rows and each slice's rows in one
    # CTA's shared memory; otherwise (and at temperature 0) the chunked or
    # greedy launch runs
    bf, f = W.DT_BF16, W.DT_F32
    assert d3d.d3d_spec_verify_slice_ctas(1, 16, 151936, bf, 1.0, 56) == 56
    assert d3d.d3d_spec_verify_slice_ctas(1, 16, 151936, bf, 0.0, 56) == 0
    assert d3d.d3d_spec_verify_slice_ctas(2, 16, 70001, bf, 1.0, 0) == 0    # rows not 16-byte aligned
    assert d3d.d3d_spec_verify_slice_ctas(24, 16, 151936, bf, 1.0, 0) == 0  # slices too wide for shared memory
    assert d3d.d3d_spec_verify_slice_ctas(0, 16, 151936, bf, 1.0, 0) == 0
    small = d3d.d3d_spec_verify_workspace_size(1, 16, 151936) // 8
    assert d3d.d3d_spec_verify_slice_ctas(1, 16, 151936, bf, 1.0, 0, ws_bytes=small) == 0  # too little workspace
    assert d3d.d3d_spec_verify_slice_ctas(3, 5, 1000, f, 0.7, 0) > 0


def test_verify_slice_wait_runs_out_reports_status_and_context_survives(d3d):
    # failure detection without a GPU fault: in the slice launch CTA 0 never
    # issues its first row's copy, its bounded wait runs out, it records the
    # timeout, waits out its other copies and leaves; the other CTAs give up
    # their bounded waits.  The next call, on a re-initialised workspace, is correct
    v = W.verify_inputs(**W.CONFIGS["async8b"], seed=13)
    assert d3d.d3d_spec_verify_slice_ctas(1, 16, 151936, W.DT_BF16, 1.0, 56) > 0
    d3d.d3d_debug_inject_fault(2)
    try:
        _, ws = run_verify(d3d, v, sm_limit=56)
    finally:
        d3d.d3d_debug_inject_fault(0)
    assert d3d.d3d_workspace_status(ws, clear=True) == d3d.D3D_ERR_DEVICE_TIMEOUT
    d3d.d3d_workspace_init(ws)
    got, _ = run_verify(d3d, v, ws=ws, sm_limit=56)
    compare_verify(got, oracle_verify(v), min_kept=1.0, what="slices, after a timed-out call")
    assert d3d.d3d_workspace_status(ws) == 0


def _heads_hitting(ref, B, V, M, seed):
    """Branch heads for a verification batch: random heads of every length plus,
    for most requests, one copy of the oracle's verified tokens (a planted hit)
    and for some a copy placed twice (lowest index wins)."""
    rng = np.random.default_rng(seed)
    R = ref["out_tokens"].shape[0]
    heads = rng.integers(0, V, size=(R, M, B)).astype(np.int32)
    head_len = rng.integers(0, B + 1, size=(R, M)).astype(np.int32)
    for r in range(R):
        n = int(ref["num_tokens"][r])
        if r == 0 or rng.random() < 0.7:
            for k in sorted(rng.choice(M, size=2 if rng.random() < 0.3 else 1, replace=False)):
                heads[r, k, :n] = ref["out_tokens"][r, :n]
                head_len[r, k] = n
    return dict(heads=heads, head_len=head_len)


@pytest.mark.parametrize("cfg,sm_limit", [("async8b", 0), ("async8b", 56), ("serve32b", 0), ("serve32b", 40),
                                          ("tiny", 0)])
def test_verify_fused_match(d3d, cfg, sm_limit):
    # the match fused into the verification equals the match of the tokens the
    # verification produced (oracle), hits planted from the oracle's tokens
    c = dict(W.CONFIGS[cfg])
    c["R"] = {"tiny": 300, "async8b": 24, "serve32b": 32}[cfg]
    v = W.verify_inputs(**c, seed=8)
    ref = oracle_verify(v)
    hb = _heads_hitting(ref, c["B"], c["V"], 24, seed=9)
    got, ws = run_verify(d3d, v, sm_limit=sm_limit, heads=hb)
    compare_verify(got, ref, min_kept=0.85, what="%s fused match" % cfg)
    want = oracle.branch_match(dict(verified=got["out_tokens"], verified_len=got["num_tokens"], **hb))
    np.testing.assert_array_equal(got["branch"], want)
    assert want[0] >= 0 and (want >= 0).mean() > 0.3  # hits are exercised
    assert d3d.d3d_workspace_status(ws) == 0


@pytest.mark.parametrize("attention_first", [False, True])
def test_round_on_one_stream_overlapping(d3d, attention_first):
    # one stream, the two parts of a round overlapping: the verification on
    # the SMs the attention leaves and the attention as its programmatic
    # dependent, or the attention first and the verification as its
    # dependent; repeated, both outputs meet the oracle and a later reader
    # sees both complete
    cfg = W.CONFIGS["async8b"]
    a = W.attn_inputs(**cfg, seed=21)
    v = W.verify_inputs(**cfg, seed=21)
    ref_v = oracle_verify(v)
    ref_a = oracle.packed_attn(a, heads=(28, 32))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # the attention in one wave of at most 96 CTAs, the verification on the rest
    budget = 96
    side = sms - d3d.d3d_packed_draft_attn_ctas(1, cfg["Hq"], cfg["Hkv"], cfg["d"], a["max_q"], a["max_prefix"],
                                                budget)
    assert side >= sms - budget
    from gpu_util import bf16, f32, i32
    t = {k: bf16(a[k]) for k in ("q", "kp", "vp", "kn", "vn")}
    ix = {k: i32(a[k]) for k in ("segs", "cu_prefix", "cu_q", "cu_seg")}
    wsa = d3d.new_workspace(d3d.d3d_packed_draft_attn_workspace_size(1, cfg["Hq"], cfg["Hkv"], cfg["d"], a["max_q"],
                                                                      a["max_prefix"]))
    wsv = d3d.new_workspace(d3d.d3d_spec_verify_workspace_size(1, cfg["B"], cfg["V"]))
    tg, dr = bf16(v["target"]), bf16(v["draft"])
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    toks = torch.empty(1, cfg["B"], dtype=torch.int32, device="cuda")
    nt = torch.empty(1, dtype=torch.int32, device="cuda")
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for _ in range(5):
            out = torch.full_like(t["q"], float("nan"))
            toks.fill_(-7)
            def ver():
                d3d.d3d_spec_verify(tg, dr, i32(v["y"]), f32(v["u_accept"]), f32(v["u_sample"]), 1.0, acc, toks, nt,
                                    wsv, sm_limit=side, after_independent=attention_first)

            def att():
                d3d.d3d_packed_draft_attn(t["q"], t["kp"], t["vp"], t["kn"], t["vn"], ix["segs"], ix["cu_prefix"],
                                          ix["cu_q"], ix["cu_seg"], a["max_q"], a["max_prefix"], a["scale"], out, wsa,
                                          after_independent=not attention_first, max_ctas=budget,
                                          after_dependent=attention_first)
            if attention_first:
                att()
                ver()
            else:
                ver()
                att()
            got_t, got_o = toks.cpu().numpy(), out.float().cpu().numpy()  # read after both, same stream
            keep = (ref_v["margin_accept"] >= NEAR_TIE) & (ref_v["margin_sample"] >= SAMPLE_BAND)
            assert keep.all()  # the round's one draw (seed 21) has no near tie
            np.testing.assert_array_equal(got_t[keep], ref_v["out_tokens"][keep])
            assert_attn_close(got_o[:, 28:32], ref_a[:, 28:32], "overlapped attention")
    assert d3d.d3d_workspace_status(wsa) == 0 and d3d.d3d_workspace_status(wsv) == 0


def _round_calls(d3d, cfg, seed):
    """Device inputs and outputs of one round (attention + verification with
    the fused match) as the keyword dicts d3d_async_round takes."""
    from gpu_util import bf16, f32, i32
    a = W.attn_inputs(**cfg, seed=seed)
    v = W.verify_inputs(**cfg, seed=seed)
    ref_v = oracle_verify(v)
    hb = _heads_hitting(ref_v, cfg["B"], cfg["V"], 24, seed=seed + 1)
    R, B = v["R"], v["B"]
    attn = dict(q=bf16(a["q"]), k_prefix=bf16(a["kp"]), v_prefix=bf16(a["vp"]), k_packed=bf16(a["kn"]),
                v_packed=bf16(a["vn"]), segs=i32(a["segs"]), cu_prefix=i32(a["cu_prefix"]), cu_q=i32(a["cu_q"]),
                cu_seg=i32(a["cu_seg"]), max_q=a["max_q"], max_prefix=a["max_prefix"], scale=a["scale"])
    attn["out"] = torch.full_like(attn["q"], float("nan"))
    attn["ws"] = d3d.new_workspace(d3d.d3d_packed_draft_attn_workspace_size(a["R"], a["Hq"], a["Hkv"], a["d"],
                                                                            a["max_q"], a["max_prefix"]))
    verify = dict(target_logits=bf16(v["target"]), draft_logits=bf16(v["draft"]), draft_tokens=i32(v["y"]),
                  u_accept=f32(v["u_accept"]), u_sample=f32(v["u_sample"]), temperature=1.0,
                  accept_len=torch.full((R,), -7, dtype=torch.int32, device="cuda"),
                  out_tokens=torch.full((R, B), -7, dtype=torch.int32, device="cuda"),
                  num_tokens=torch.full((R,), -7, dtype=torch.int32, device="cuda"),
                  heads=i32(hb["heads"]), head_len=i32(hb["head_len"]),
                  branch=torch.full((R,), -7, dtype=torch.int32, device="cuda"),
                  ws=d3d.new_workspace(d3d.d3d_spec_verify_workspace_size(R, B, v["V"])))
    return a, v, ref_v, hb, attn, verify


def test_async_round_in_one_launch(d3d):
    # the drafting attention and the verification (with the fused match) of
    # the 384-token async round as one cooperative launch, three times over
    # the same workspaces: every output meets the oracle
    cfg = W.CONFIGS["async8b"]
    a, v, ref_v, hb, attn, verify = _round_calls(d3d, cfg, seed=33)
    ref_a = oracle.packed_attn(a, heads=(0, 4))
    for _ in range(3):
        attn["out"].fill_(float("nan"))
        for k in ("accept_len", "out_tokens", "num_tokens", "branch"):
            verify[k].fill_(-7)
        d3d.d3d_async_round(attn, verify)
        torch.cuda.synchronize()
        got = {k: verify[k].cpu().numpy() for k in ("accept_len", "out_tokens", "num_tokens", "branch")}
        # one request: its draw must be compared (seed 33 has no near tie)
        compare_verify(got, ref_v, min_kept=1.0, what="fused round")
        want = oracle.branch_match(dict(verified=got["out_tokens"], verified_len=got["num_tokens"], **hb))
        np.testing.assert_array_equal(got["branch"], want)
        assert_attn_close(attn["out"].float().cpu().numpy()[:, 0:4], ref_a[:, 0:4], "fused round attention")
    assert d3d.d3d_workspace_status(attn["ws"]) == 0 and d3d.d3d_workspace_status(verify["ws"]) == 0


def test_async_round_declines_key_splits(d3d):
    # a long prefix with few query tiles splits keys across a cluster: the
    # fused launch declines and the two calls do the round
    cfg = dict(W.CONFIGS["long_block"], V=4096)
    a, v, ref_v, hb, attn, verify = _round_calls(d3d, cfg, seed=34)
    with pytest.raises(d3d.D3DError) as e:
        d3d.d3d_async_round(attn, verify)
    assert e.value.rc == d3d.D3D_ERR_UNSUPPORTED


def test_attention_cta_count_matches_plan(d3d):
    # one CTA per query tile (or tile pair) and key split, all in one wave on
    # this GPU, and within the CTA budget when one is given; the unsplit
    # two-tile plan (R * Hkv * ceil(MT / 2) = 1 * 8 * 6 CTAs, MT = 384 / 32
    # query tiles) is the floor below which no budget goes
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = d3d.d3d_packed_draft_attn_ctas(1, 32, 8, 128, 384, 2048)
    assert 0 < n <= sms
    floor = d3d.d3d_packed_draft_attn_ctas(1, 32, 8, 128, 384, 2048, 1)
    assert floor >= 48
    for budget in (24, 48, 96, 120):
        assert 0 < d3d.d3d_packed_draft_attn_ctas(1, 32, 8, 128, 384, 2048, budget) <= max(budget, floor)


@pytest.mark.parametrize("budget", [0, 120, 96, 48, 12])
def test_attn_plans_under_cta_budgets(d3d, budget):
    # the CTA budget changes the plan (one or two query tiles per CTA, the key
    # split); every plan meets the oracle on the async8b layout (sampled heads)
    a = W.attn_inputs(**W.CONFIGS["async8b"], seed=17)
    from gpu_util import bf16, i32
    t = {k: bf16(a[k]) for k in ("q", "kp", "vp", "kn", "vn")}
    ix = {k: i32(a[k]) for k in ("segs", "cu_prefix", "cu_q", "cu_seg")}
    out = torch.full_like(t["q"], float("nan"))
    ws = d3d.new_workspace(d3d.d3d_packed_draft_attn_workspace_size(1, 32, 8, 128, a["max_q"], a["max_prefix"]))
    d3d.d3d_packed_draft_attn(t["q"], t["kp"], t["vp"], t["kn"], t["vn"], ix["segs"], ix["cu_prefix"], ix["cu_q"],
                              ix["cu_seg"], a["max_q"], a["max_prefix"], a["scale"], out, ws, max_ctas=budget)
    torch.cuda.synchronize()
    heads = [0, 13, 31]
    got = out.float().cpu().numpy()
    assert_attn_close(got[:, heads], _oracle_heads(a, heads)[:, heads], "budget %d" % budget)
    assert d3d.d3d_workspace_status(ws) == 0


# ------------------------------------------------------------------ greedy (temperature 0)
def _greedy_inputs(cfg, seed, plant=True, **over):
    """Verification inputs whose draft tokens follow the greedy drafter (the
    draft rows' argmax, lowest index); with plant, request r's first r % B
    tokens are replaced by the target's argmax so that every accepted length
    occurs."""
    v = W.verify_inputs(**dict(W.CONFIGS[cfg], **over), seed=seed)
    dec = (lambda x: W.bf16_to_f32(x)) if v["dtype"] == W.DT_BF16 else (lambda x: x)
    y = dec(v["draft"]).argmax(-1).astype(np.int32)
    if plant:
        g = oracle.greedy_verify(dict(v, y=y))["argmax"]
        for r in range(v["R"]):
            k = r % v["B"]
            y[r, :k] = g[r, :k]
    v["y"] = np.ascontiguousarray(y)
    return v


def _run_greedy(d3d, v, sm_limit=0, heads=None, noalloc=False, probs=True):
    from gpu_util import bf16, f32, i32
    R, B = v["R"], v["B"]
    tgt = bf16(v["target"]) if v["dtype"] == W.DT_BF16 else f32(v["target"])
    out = dict(accept_len=torch.full((R,), -7, dtype=torch.int32, device="cuda"),
               out_tokens=torch.full((R, B), -7, dtype=torch.int32, device="cuda"),
               num_tokens=torch.full((R,), -7, dtype=torch.int32, device="cuda"))
    pr = {k: torch.full((R, B - 1), float("nan"), device="cuda") for k in ("alpha", "p")} if probs else {}
    if probs and not noalloc:
        pr["awl"] = torch.full((R, B - 1), float("nan"), device="cuda")
    if noalloc:
        d3d.d3d_spec_verify_noalloc(tgt, None, i32(v["y"]), None, None, 0.0, out["accept_len"], out["out_tokens"],
                                    out["num_tokens"], alpha=pr.get("alpha"), p_draft=pr.get("p"))
        ws = None
    else:
        ws = d3d.new_workspace(d3d.d3d_spec_verify_workspace_size(R, B, v["V"]))
        extra = {}
        if heads is not None:
            out["branch"] = torch.full((R,), -7, dtype=torch.int32, device="cuda")
            extra = dict(heads=i32(heads["heads"]), head_len=i32(heads["head_len"]), branch=out["branch"])
        d3d.d3d_spec_verify(tgt, None, i32(v["y"]), None, None, 0.0, out["accept_len"], out["out_tokens"],
                            out["num_tokens"], ws, alpha=pr.get("alpha"), p_draft=pr.get("p"),
                            awl_weight=pr.get("awl"), sm_limit=sm_limit, **extra)
    torch.cuda.synchronize()
    got = {k: t.cpu().numpy() for k, t in out.items()}
    got.update({k: t.cpu().numpy() for k, t in pr.items()})
    return got, ws


def _check_greedy(got, ref):
    np.testing.assert_array_equal(got["accept_len"], ref["accept_len"])
    np.testing.assert_array_equal(got["num_tokens"], ref["num_tokens"])
    np.testing.assert_array_equal(got["out_tokens"], ref["out_tokens"])
    if "alpha" in got:
        np.testing.assert_array_equal(got["alpha"], ref["accept"].astype(np.float32))
        np.testing.assert_array_equal(got["p"], ref["accept"].astype(np.float32))
    if "awl" in got:  # the product of the acceptance indicators before each position
        np.testing.assert_array_equal(got["awl"], oracle.awl_weights(ref["accept"]).astype(np.float32))


@pytest.mark.parametrize("cfg,over", [
    ("tiny", {}),
    ("tiny", dict(R=40)),
    ("async8b", {}),
    ("async8b", dict(R=5)),
    ("long_block", {}),
    ("serve32b", {}),
    ("tiny", dict(R=9, V=1001)),                      # f32, V % 8 != 0: scalar loads
    ("async8b", dict(R=3, V=151939)),                 # bf16, V % 8 != 0
    ("async8b", dict(R=2, V=8192 * 3)),               # whole chunks only
    ("async8b", dict(R=2, V=17)),                     # one short chunk
])
def test_greedy_verify_matches_oracle(d3d, cfg, over):
    v = _greedy_inputs(cfg, seed=40, **over)
    ref = oracle.greedy_verify(v)
    got, ws = _run_greedy(d3d, v)
    _check_greedy(got, ref)
    assert d3d.d3d_workspace_status(ws) == 0
    if v["R"] >= v["B"]:
        assert len(set(ref["accept_len"].tolist())) > 3  # many accepted lengths occur


@pytest.mark.parametrize("dt", [W.DT_F32, W.DT_BF16])
def test_greedy_ties_go_to_the_lowest_index(d3d, dt):
    # integer logits in a tiny range: most rows have their maximum many times
    rng = np.random.default_rng(41)
    R, B, V = 24, 16, 40000
    vals = rng.integers(0, 3, size=(R, B, V)).astype(np.float32)
    vals[:, :, rng.integers(0, V, size=7)] = 3.0  # a few columns hold the maximum in every row
    tgt = W.bf16_bits(vals) if dt == W.DT_BF16 else vals
    g = vals.argmax(-1)
    y = np.where(rng.random((R, B - 1)) < 0.8, g[:, : B - 1], (g[:, : B - 1] + 1) % V).astype(np.int32)
    v = dict(target=tgt, dtype=dt, y=y, R=R, B=B, V=V)
    ref = oracle.greedy_verify(v)
    got, _ = _run_greedy(d3d, v)
    _check_greedy(got, ref)


@pytest.mark.parametrize("cfg,sm_limit", [("async8b", 0), ("async8b", 56), ("serve32b", 40)])
def test_greedy_fused_match_and_sm_limit(d3d, cfg, sm_limit):
    v = _greedy_inputs(cfg, seed=42)
    ref = oracle.greedy_verify(v)
    hb = _heads_hitting(ref, v["B"], v["V"], 24, seed=43)
    got, _ = _run_greedy(d3d, v, sm_limit=sm_limit, heads=hb)
    _check_greedy(got, ref)
    want = oracle.branch_match(dict(verified=ref["out_tokens"], verified_len=ref["num_tokens"], **hb))
    np.testing.assert_array_equal(got["branch"], want)


def test_greedy_bad_draft_token_and_noalloc(d3d):
    v = _greedy_inputs("tiny", seed=44, R=6)
    ref = oracle.greedy_verify(v)
    got, _ = _run_greedy(d3d, v, noalloc=True)  # the library's own scratch
    _check_greedy(got, ref)
    # a draft token outside [0, V) is rejected there and reported
    bad = dict(v, y=v["y"].copy())
    bad["y"][2, 0] = v["V"] + 5
    got, ws = _run_greedy(d3d, bad, probs=False)
    assert d3d.d3d_workspace_status(ws) == d3d.D3D_ERR_DEVICE_INPUT
    assert got["accept_len"][2] == 0 and got["out_tokens"][2, 0] == ref["argmax"][2, 0]
    keep = np.arange(v["R"]) != 2
    np.testing.assert_array_equal(got["out_tokens"][keep], ref["out_tokens"][keep])


# ------------------------------------------------------------------ branch construction
def _run_branches(d3d, v, C, F, bonus=None, full=True):
    from gpu_util import bf16, f32, i32
    R, B = v["R"], v["B"]
    M = (C - 1) * F + 2
    dr = bf16(v["draft"]) if v["dtype"] == W.DT_BF16 else f32(v["draft"])
    o = dict(anchors=torch.full((R, C - 1, F), -7, dtype=torch.int32, device="cuda"),
             heads=torch.full((R, M, B), -7, dtype=torch.int32, device="cuda"),
             head_len=torch.full((R, M), -7, dtype=torch.int32, device="cuda"))
    if full:
        o.update(segs=torch.full((R * M, 5), -7, dtype=torch.int32, device="cuda"),
                 cu_q=torch.full((R + 1,), -7, dtype=torch.int32, device="cuda"),
                 cu_seg=torch.full((R + 1,), -7, dtype=torch.int32, device="cuda"))
    ws = d3d.new_workspace(d3d.d3d_build_branches_workspace_size(R, B, v["V"], C, F))
    d3d.d3d_build_branches(dr, i32(v["y"]), C, F, o["heads"], o["head_len"], ws, anchors=o["anchors"],
                           bonus_guess=None if bonus is None else i32(bonus), segs=o.get("segs"),
                           cu_q=o.get("cu_q"), cu_seg=o.get("cu_seg"))
    torch.cuda.synchronize()
    return {k: t.cpu().numpy() for k, t in o.items()}, ws


@pytest.mark.parametrize("cfg,C,F,over,bonus", [
    ("async8b", 12, 2, {}, True),
    ("async8b", 12, 2, {}, False),
    ("serve32b", 12, 2, {}, True),
    ("sweep", 16, 5, {}, True),
    ("sweep", 8, 3, dict(R=3), False),
    ("tiny", 12, 2, dict(R=7), True),                 # f32, V = 1024
    ("async8b", 5, 4, dict(R=2, V=151939), True),     # V % 8 != 0
    ("async8b", 16, 8, dict(R=2, V=9), True),         # every token but y is an anchor
    ("async8b", 1, 2, dict(R=3), True),               # C = 1: no anchors
    ("async8b", 12, 0, dict(R=2), True),              # F = 0
])
def test_build_branches_matches_oracle(d3d, cfg, C, F, over, bonus):
    v = W.verify_inputs(**dict(W.CONFIGS[cfg], **over), seed=50)
    bg = np.random.default_rng(51).integers(0, v["V"], size=v["R"]).astype(np.int32) if bonus else None
    ref = oracle.build_branches(dict(draft=v["draft"], dtype=v["dtype"], y=v["y"], bonus_guess=bg, R=v["R"],
                                     B=v["B"], V=v["V"], C=C, F=F))
    got, ws = _run_branches(d3d, v, C, F, bonus=bg)
    for k in ("anchors", "heads", "head_len", "segs", "cu_q", "cu_seg"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
    assert d3d.d3d_workspace_status(ws) == 0
    # a second call on the same workspace (its counters reset themselves)
    got2, _ = _run_branches(d3d, v, C, F, bonus=bg, full=False)
    np.testing.assert_array_equal(got2["heads"], ref["heads"])


@pytest.mark.parametrize("dt", [W.DT_F32, W.DT_BF16])
def test_build_branches_ties_and_bad_token(d3d, dt):
    rng = np.random.default_rng(52)
    R, B, V, C, F = 6, 16, 20000, 12, 3
    vals = rng.integers(0, 3, size=(R, B - 1, V)).astype(np.float32)
    vals[:, :, rng.integers(0, V, size=5)] = 3.0
    y = vals.argmax(-1).astype(np.int32)  # the drafted token is the first maximum: the anchors are the next ones
    v = dict(draft=W.bf16_bits(vals) if dt == W.DT_BF16 else vals, dtype=dt, y=y, R=R, B=B, V=V)
    ref = oracle.build_branches(dict(v, C=C, F=F, bonus_guess=None))
    got, ws = _run_branches(d3d, v, C, F)
    np.testing.assert_array_equal(got["anchors"], ref["anchors"])
    np.testing.assert_array_equal(got["heads"], ref["heads"])
    bad = dict(v, y=y.copy())
    bad["y"][1, 3] = V + 2
    got, ws = _run_branches(d3d, bad, C, F)
    assert d3d.d3d_workspace_status(ws) == d3d.D3D_ERR_DEVICE_INPUT


def test_built_branches_drive_attention_and_match(d3d):
    # the segment rows and heads built on the device are what the packed
    # attention and the fused match consume: both against the oracle
    from gpu_util import bf16, i32
    cfg = W.CONFIGS["async8b"]
    C, F = cfg["C"], cfg["F"]
    v = W.verify_inputs(**cfg, seed=53)
    ref_v = oracle_verify(v)
    bg = ref_v["out_tokens"][:, -1].copy()  # any guess; on full acceptance a matching one makes a hit
    got, _ = _run_branches(d3d, v, C, F, bonus=bg)
    a = W.attn_inputs(**cfg, seed=53, segs=got["segs"])
    out, _ = run_attn(d3d, a)
    assert_attn_close(out[:, 4:8], oracle.packed_attn(a, heads=(4, 8))[:, 4:8], "device-built segments")
    hb = dict(heads=got["heads"], head_len=got["head_len"])
    res = run_verify(d3d, v, heads=hb)[0]
    want = oracle.branch_match(dict(verified=res["out_tokens"], verified_len=res["num_tokens"], **hb))
    np.testing.assert_array_equal(res["branch"], want)


# ------------------------------------------------------------------ acceptance probabilities and tau
@pytest.mark.parametrize("cfg,over", [
    ("tiny", {}), ("tiny", dict(R=5, temperature=0.7)), ("async8b", {}), ("serve32b", {}),
    ("long_block", dict(sigma=1.0)), ("tiny", dict(R=3, V=1001)), ("async8b", dict(R=2, V=151939)),
])
def test_accept_probs_and_tau_match_oracle(d3d, cfg, over):
    from gpu_util import bf16, f32
    v = W.verify_inputs(**dict(W.CONFIGS[cfg], **over), seed=70)
    ref = oracle.accept_probs(v)
    R, B = v["R"], v["B"]
    tg, dr = (bf16(v["target"]), bf16(v["draft"])) if v["dtype"] == W.DT_BF16 else (f32(v["target"]), f32(v["draft"]))
    ws = d3d.new_workspace(d3d.d3d_accept_probs_workspace_size(R, B, v["V"]))
    outs = []
    for _ in range(2):  # twice on one workspace: the counters reset themselves; the sums are in a fixed order
        a = torch.full((R, B - 1), float("nan"), device="cuda")
        sv = torch.full((R, B - 1), float("nan"), device="cuda")
        tau = torch.full((R,), float("nan"), device="cuda")
        d3d.d3d_accept_probs(tg, dr, v.get("temperature", 1.0), a, ws, survival=sv, tau=tau)
        torch.cuda.synchronize()
        outs.append((a.cpu().numpy(), sv.cpu().numpy(), tau.cpu().numpy()))
    a, sv, tau = outs[0]
    # the probabilities' relative tolerance (1e-5) for all three; measured on
    # GB300 over these cases and seeds 70-72: a 2.3e-7, S(k) 1.7e-6, tau 4.4e-7
    np.testing.assert_allclose(a, ref["accept_prob"], rtol=PROB_RTOL, atol=0)
    np.testing.assert_allclose(sv, ref["survival"], rtol=PROB_RTOL, atol=0)
    np.testing.assert_allclose(tau, ref["tau"], rtol=PROB_RTOL)
    for x, y in zip(outs[0], outs[1]):
        np.testing.assert_array_equal(x, y)


def test_accept_probs_slice_and_two_launch_shapes_agree(d3d):
    # one request: the slice launch (rows read once) with the full workspace;
    # a workspace that holds only the two launches' chunk records takes those
    from gpu_util import bf16
    v = W.verify_inputs(**W.CONFIGS["async8b"], seed=72)
    R, B, V = v["R"], v["B"], v["V"]
    tg, dr = bf16(v["target"]), bf16(v["draft"])
    full = d3d.d3d_accept_probs_workspace_size(R, B, V)
    res = []
    for nbytes in (full, full // 8):
        ws = d3d.new_workspace(nbytes)
        a = torch.full((R, B - 1), float("nan"), device="cuda")
        tau = torch.full((R,), float("nan"), device="cuda")
        d3d.d3d_accept_probs(tg, dr, 1.0, a, ws, tau=tau)
        torch.cuda.synchronize()
        assert d3d.d3d_workspace_status(ws) == 0
        res.append((a.cpu().numpy(), tau.cpu().numpy()))
    ref = oracle.accept_probs(v)
    for a, tau in res:
        np.testing.assert_allclose(a, ref["accept_prob"], rtol=PROB_RTOL, atol=0)
        np.testing.assert_allclose(tau, ref["tau"], rtol=PROB_RTOL)
    np.testing.assert_allclose(res[0][0], res[1][0], rtol=1e-5, atol=1e-7)


def test_verify_workspace_reuse_and_many_requests(d3d):
    v = W.verify_inputs(R=4096, B=4, V=64, logits=W.DT_F32, seed=10)
    got1, ws = run_verify(d3d, v)
    got2, _ = run_verify(d3d, v, ws=ws)
    for k in got1:
        np.testing.assert_array_equal(got1[k], got2[k])
    compare_verify(got1, oracle_verify(v), what="R=4096")


def test_verify_ring_wait_runs_out_reports_status_and_context_survives(d3d):
    # failure detection without a GPU fault: with an SM limit the bf16 rows
    # stream through a shared-memory ring; CTA 0 never issues its first
    # item's copies, its bounded wait runs out, it records the timeout, waits
    # out its other copies and leaves; the other CTAs give up their bounded
    # waits.  The next call, on a re-initialised workspace, is correct
    v = W.verify_inputs(**dict(W.CONFIGS["async8b"], R=2), seed=12)
    d3d.d3d_debug_inject_fault(2)
    try:
        _, ws = run_verify(d3d, v, sm_limit=56)
    finally:
        d3d.d3d_debug_inject_fault(0)
    assert d3d.d3d_workspace_status(ws, clear=True) == d3d.D3D_ERR_DEVICE_TIMEOUT
    d3d.d3d_workspace_init(ws)
    got, _ = run_verify(d3d, v, ws=ws, sm_limit=56)
    compare_verify(got, oracle_verify(v), min_kept=1.0, what="after a timed-out call")
    assert d3d.d3d_workspace_status(ws) == 0


def test_verify_bad_draft_token_sets_status(d3d):
    v = W.verify_inputs(R=2, B=4, V=100, seed=11)
    v["y"] = v["y"].copy()
    v["y"][1, 0] = 100
    got, ws = run_verify(d3d, v)
    assert d3d.d3d_workspace_status(ws, clear=True) == d3d.D3D_ERR_DEVICE_INPUT
    assert got["alpha"][1, 0] == 0 and got["accept_len"][1] == 0
    assert got["out_tokens"][1, 0] != 100


# ------------------------------------------------------------------ branch match
def test_match_planted_hits(d3d):
    m = W.match_inputs(R=4096, seed=12)
    got = run_match(d3d, m)
    np.testing.assert_array_equal(got, oracle.branch_match(m))


@pytest.mark.parametrize("M,B", [(5, 3), (70, 6), (33, 40), (0, 4)])
def test_match_tiny_alphabet(d3d, M, B):
    rng = np.random.default_rng(M * 100 + B)
    R = 3000
    m = dict(verified=rng.integers(0, 2, (R, B)).astype(np.int32),
             verified_len=rng.integers(-1, B + 2, R).astype(np.int32),
             heads=rng.integers(0, 2, (R, M, B)).astype(np.int32),
             head_len=rng.integers(0, B + 1, (R, M)).astype(np.int32))
    if M == 0:
        m["heads"] = np.zeros((R, 0, B), np.int32)
        m["head_len"] = np.zeros((R, 0), np.int32)
    ref = np.where((m["verified_len"] < 0) | (m["verified_len"] > B), -1,
                   oracle.branch_match(dict(m, verified_len=np.clip(m["verified_len"], 0, B))))
    np.testing.assert_array_equal(run_match(d3d, m), ref)


# ------------------------------------------------------------------ whole step
def test_step_verify_then_match_async8b(d3d):
    v = W.verify_inputs(**dict(W.CONFIGS["async8b"], R=8), seed=13)
    got, _ = run_verify(d3d, v, want_probs=False)
    hb = W.branch_heads(v["y"], 16, 12, 2, v["V"], seed=13)
    m = dict(verified=got["out_tokens"], verified_len=got["num_tokens"], heads=hb["heads"], head_len=hb["head_len"])
    np.testing.assert_array_equal(run_match(d3d, m), oracle.branch_match(m))
