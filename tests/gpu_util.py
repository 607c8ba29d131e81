"""Helpers shared by the GPU tests: move seeded inputs to the device and call
the library through its binding."""
import numpy as np
import torch

ATT_ATOL = 2e-2   # bf16 inputs, fp32 accumulate, bf16 output: |d| <= 2e-2 + 2e-2 |ref|
ATT_RTOL = 2e-2
PROB_RTOL = 1e-5  # p_j, q_j, alpha_j
# Draws excluded from the bit-exact comparison of accepted lengths and tokens:
# |u_j - alpha_j| < 1e-5 at a test that decided the accepted length (the rule
# the comparison contract states), and sample draws whose u*S lies within
# SAMPLE_BAND * S of a step of the oracle's CDF.  The second band is set from
# measurement: across seeded runs at every workload shape the largest margin
# at which the fp32 device sample differed from the fp64 oracle was below a
# tenth of it.
NEAR_TIE = 1e-5
SAMPLE_BAND = 1e-6


def oracle_verify(v):
    """The oracle's verification of a batch: one oracle call per request on
    all host cores when the OpenMP build is available (identical results),
    else the one-thread oracle."""
    import oracle

    try:
        return oracle.spec_verify_par(v)
    except RuntimeError:
        return oracle.spec_verify(v)


def bf16(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def i32(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).to(dev)


def f32(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.float32))).to(dev)


def run_attn(d3d, a, ws=None):
    dev = "cuda"
    t = {k: bf16(a[k]) for k in ("q", "kp", "vp", "kn", "vn")}
    ix = {k: i32(a[k]) for k in ("segs", "cu_prefix", "cu_q", "cu_seg")}
    out = torch.full_like(t["q"], float("nan"))
    if ws is None:
        ws = d3d.new_workspace(d3d.d3d_packed_draft_attn_workspace_size(
            a["R"], a["Hq"], a["Hkv"], a["d"], a["max_q"], a["max_prefix"]), dev)
    d3d.d3d_packed_draft_attn(t["q"], t["kp"], t["vp"], t["kn"], t["vn"], ix["segs"], ix["cu_prefix"], ix["cu_q"],
                              ix["cu_seg"], a["max_q"], a["max_prefix"], a["scale"], out, ws)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), ws


def assert_attn_close(got, ref, what=""):
    assert np.isfinite(got).all(), "non-finite attention output " + what
    excess = np.abs(got - ref) - (ATT_ATOL + ATT_RTOL * np.abs(ref))
    assert (excess <= 0).all(), "%s: max excess %g at %s" % (what, excess.max(), np.unravel_index(excess.argmax(),
                                                                                                  excess.shape))


def run_verify(d3d, v, ws=None, want_probs=True, sm_limit=0, heads=None):
    dev = "cuda"
    R, B = v["R"], v["B"]
    if v["dtype"] == 1:
        tgt, dr = bf16(v["target"]), bf16(v["draft"])
    else:
        tgt, dr = f32(v["target"]), f32(v["draft"])
    out = dict(accept_len=torch.full((R,), -7, dtype=torch.int32, device=dev),
               out_tokens=torch.full((R, B), -7, dtype=torch.int32, device=dev),
               num_tokens=torch.full((R,), -7, dtype=torch.int32, device=dev))
    probs = {k: torch.full((R, B - 1), float("nan"), device=dev) for k in ("alpha", "p", "q", "awl")} \
        if want_probs else {}
    if ws is None:
        ws = d3d.new_workspace(d3d.d3d_spec_verify_workspace_size(R, B, v["V"]), dev)
    fused = {}
    if heads is not None:  # the branch match fused into the verification
        out["branch"] = torch.full((R,), -7, dtype=torch.int32, device=dev)
        fused = dict(heads=i32(heads["heads"]), head_len=i32(heads["head_len"]), branch=out["branch"])
    d3d.d3d_spec_verify(tgt, dr, i32(v["y"]), f32(v["u_accept"]), f32(v["u_sample"]), v.get("temperature", 1.0),
                        out["accept_len"], out["out_tokens"], out["num_tokens"], ws, alpha=probs.get("alpha"),
                        p_draft=probs.get("p"), q_draft=probs.get("q"), awl_weight=probs.get("awl"),
                        sm_limit=sm_limit, **fused)
    torch.cuda.synchronize()
    res = {k: t.cpu().numpy() for k, t in {**out, **probs}.items()}
    return res, ws


def compare_verify(got, ref, min_kept=0.9, what=""):
    """Bit-exact a / tokens / counts outside the near-tie bands; probabilities
    to 1e-5 relative.  Prints and returns (compared, excluded at alpha,
    excluded at the sample); fails when fewer than min_kept of the draws are
    compared."""
    for k in ("alpha", "p", "q"):
        if k in got:
            np.testing.assert_allclose(got[k], ref[k], rtol=PROB_RTOL, atol=1e-30, err_msg=k)
    if "awl" in got:  # the acceptance-weighted loss weights, prod_{j<k} alpha_j
        import oracle

        np.testing.assert_allclose(got["awl"], oracle.awl_weights(ref["alpha"]), rtol=PROB_RTOL, atol=1e-30,
                                   err_msg="awl")
    tie_a = ref["margin_accept"] < NEAR_TIE
    tie_s = ~tie_a & (ref["margin_sample"] < SAMPLE_BAND)
    keep = ~tie_a & ~tie_s
    for k in ("accept_len", "num_tokens", "out_tokens"):
        np.testing.assert_array_equal(got[k][keep], ref[k][keep], err_msg=k)
    n = len(keep)
    print("verify %s: %d of %d draws compared, %d excluded at |u - alpha| < %g, %d at the sample band %g"
          % (what, int(keep.sum()), n, int(tie_a.sum()), NEAR_TIE, int(tie_s.sum()), SAMPLE_BAND))
    assert keep.sum() >= min_kept * n, "too many near ties: %d of %d" % (n - keep.sum(), n)
    return int(keep.sum()), int(tie_a.sum()), int(tie_s.sum())


def run_match(d3d, m):
    R = m["heads"].shape[0]
    branch = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    d3d.d3d_branch_match(i32(m["verified"]), i32(m["verified_len"]), i32(m["heads"]), i32(m["head_len"]), branch)
    torch.cuda.synchronize()
    return branch.cpu().numpy()
