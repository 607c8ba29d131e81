"""Oracle of the hot path — TEST INFRASTRUCTURE ONLY.

A plain, slow, double-precision CPU statement of what the three steps of
diffusion-drafted speculative decoding compute (packed drafting attention,
speculative-sampling verification, branch cache-hit match), plus the pages'
two closed forms (N_async and the mean acceptance length).  Only the tests,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg
may import it.  It shares no code with the CUDA library and never calls it;
the product path never calls this.

The arithmetic lives in ``d3d_oracle.c`` (plain C99, single thread, no
vectorisation or reordering), compiled with gcc into ``_build/`` on first
use.  Function-level citations are in that file and below.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "d3d_oracle.c")
_OUT = os.path.join(_HERE, "_build", "libd3d_oracle.so")
_lock = threading.Lock()
_lib = None

OK = 0


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, -O2, IEEE arithmetic: no fast-math)."""
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    if force or not os.path.exists(_OUT) or os.path.getmtime(_OUT) < os.path.getmtime(_SRC):
        tmp = _OUT + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _OUT)
    return _OUT


_SRC_PAR = os.path.join(_HERE, "d3d_oracle_par.c")
_OUT_PAR = os.path.join(_HERE, "_build", "libd3d_oracle_par.so")
_lib_par = None


def build_par(force: bool = False):
    """Compile the all-cores driver (d3d_oracle_par.c, OpenMP) together with
    the unchanged oracle into its own library; None if the compiler has no
    OpenMP."""
    os.makedirs(os.path.dirname(_OUT_PAR), exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_SRC_PAR))
    if force or not os.path.exists(_OUT_PAR) or os.path.getmtime(_OUT_PAR) < newest:
        tmp = _OUT_PAR + ".%d.tmp" % os.getpid()
        try:
            subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
                                   "-ffp-contract=off", "-fopenmp", _SRC, _SRC_PAR, "-o", tmp, "-lm"])
        except (OSError, subprocess.CalledProcessError):
            return None
        os.replace(tmp, _OUT_PAR)
    return _OUT_PAR


def _load_par():
    global _lib_par
    with _lock:
        if _lib_par is None:
            path = build_par()
            if path is None:
                raise RuntimeError("the all-cores oracle needs gcc with OpenMP")
            _lib_par = ctypes.CDLL(path)
            for name in ("oracle_packed_attn_par", "oracle_spec_verify_par", "oracle_par_threads"):
                getattr(_lib_par, name).restype = ctypes.c_int
    return _lib_par


def par_threads(n: int = 0) -> int:
    """Set (n > 0) and return the thread count of the all-cores oracle."""
    return _load_par().oracle_par_threads(ctypes.c_int(n))


def packed_attn_par(inp: dict) -> np.ndarray:
    """packed_attn on all cores: one oracle call per (request, query head)."""
    q, kp, vp, kn, vn = (_c(inp[k], np.uint16) for k in ("q", "kp", "vp", "kn", "vn"))
    segs, cu_p, cu_q, cu_s = (_c(inp[k], np.int32) for k in ("segs", "cu_prefix", "cu_q", "cu_seg"))
    NT, Hq, d = q.shape
    out = np.zeros((NT, Hq, d), np.float64)
    rc = _load_par().oracle_packed_attn_par(
        _p(q), _p(kp), _p(vp), _p(kn), _p(vn), _p(segs), _p(cu_p), _p(cu_q), _p(cu_s), ctypes.c_int(inp["R"]),
        ctypes.c_int(Hq), ctypes.c_int(inp["Hkv"]), ctypes.c_int(d), ctypes.c_double(inp["scale"]), _p(out))
    if rc != OK:
        raise ValueError("oracle_packed_attn_par: invalid arguments (rc=%d)" % rc)
    return out


def spec_verify_par(inp: dict) -> dict:
    """spec_verify on all cores: one oracle call per request; the same outputs."""
    R, B, V = inp["R"], inp["B"], inp["V"]
    dt = np.uint16 if inp["dtype"] == 1 else np.float32
    tgt, dr = _c(inp["target"], dt), _c(inp["draft"], dt)
    y = _c(inp["y"], np.int32)
    ua, us = _c(inp["u_accept"], np.float32), _c(inp["u_sample"], np.float32)
    out = dict(accept_len=np.zeros(R, np.int32), out_tokens=np.zeros((R, B), np.int32),
               num_tokens=np.zeros(R, np.int32), alpha=np.zeros((R, B - 1)),
               p=np.zeros((R, B - 1)), q=np.zeros((R, B - 1)), margin_accept=np.zeros(R),
               margin_sample=np.zeros(R), used_fallback=np.zeros(R, np.int32))
    rc = _load_par().oracle_spec_verify_par(
        _p(tgt), _p(dr), ctypes.c_int(inp["dtype"]), _p(y), _p(ua), _p(us), ctypes.c_int(R), ctypes.c_int(B),
        ctypes.c_int(V), ctypes.c_double(inp.get("temperature", 1.0)), _p(out["accept_len"]),
        _p(out["out_tokens"]), _p(out["num_tokens"]), _p(out["alpha"]), _p(out["p"]), _p(out["q"]),
        _p(out["margin_accept"]), _p(out["margin_sample"]), _p(out["used_fallback"]))
    if rc != OK:
        raise ValueError("oracle_spec_verify_par: invalid arguments (rc=%d)" % rc)
    return out


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            for name in ("oracle_packed_attn", "oracle_packed_attn_sel", "oracle_dense_attn",
                         "oracle_dense_mask", "oracle_spec_verify", "oracle_greedy_verify", "oracle_build_branches",
                         "oracle_accept_probs", "oracle_awl_weights",
                         "oracle_branch_match",
                         "oracle_check_segments"):
                getattr(_lib, name).restype = ctypes.c_int
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _c(a, dt):
    return np.ascontiguousarray(np.asarray(a, dtype=dt))


# ---------------------------------------------------------------------------
# Closed forms printed on the pages.
# ---------------------------------------------------------------------------
def n_async(B: int, C: int, F: int) -> int:
    """Packed query tokens of one asynchronous drafting pass.

    D3D, "Method steps", step 4: C-1 rejection positions times F
    alternative anchors, plus the all-accept block and the block being
    verified, each B tokens: N_async = B[(C-1)F + 2].
    """
    return B * ((C - 1) * F + 2)


def expected_tau(a) -> float:
    """Mean acceptance length of one round (DScout, "Background / MAT").

    tau = 1 + E[N] = 1 + sum_{k=1}^{bs-1} S(k), with the prefix survival
    S(k) = prod_{j<=k} a_j of the per-position acceptance probabilities
    a_1 .. a_{bs-1}.
    """
    tau, surv = 1.0, 1.0
    for aj in np.asarray(a, dtype=np.float64).ravel():
        surv *= float(aj)
        tau += surv
    return tau


# ---------------------------------------------------------------------------
# The three steps.
# ---------------------------------------------------------------------------
def check_segments(segs, cu_q, cu_seg) -> int:
    """0 if the segment table is well formed (see d3d_oracle.c), else -1."""
    segs, cu_q, cu_seg = _c(segs, np.int32), _c(cu_q, np.int32), _c(cu_seg, np.int32)
    return _load().oracle_check_segments(_p(segs), _p(cu_q), _p(cu_seg), ctypes.c_int(len(cu_q) - 1))


def packed_attn(inp: dict, heads=None, tokens=None) -> np.ndarray:
    """Packed drafting attention, visibility-predicate form, fp64 output [NT, Hq, d].

    D3D, "Core method" and "Method steps" step 2/4: each block attends to the
    shared prefix, to the hypothesised accepted tokens of its branch, and
    bidirectionally inside itself; the block under verification is causal.
    ``heads=(lo, hi)`` / ``tokens=(lo, hi)`` compute only those query heads /
    global packed rows (other outputs stay 0).
    """
    q, kp, vp, kn, vn = (_c(inp[k], np.uint16) for k in ("q", "kp", "vp", "kn", "vn"))
    segs, cu_p, cu_q, cu_s = (_c(inp[k], np.int32) for k in ("segs", "cu_prefix", "cu_q", "cu_seg"))
    NT, Hq, d = q.shape
    lo, hi = heads if heads is not None else (0, Hq)
    tlo, thi = tokens if tokens is not None else (0, NT)
    out = np.zeros((NT, Hq, d), np.float64)
    rc = _load().oracle_packed_attn_sel(
        _p(q), _p(kp), _p(vp), _p(kn), _p(vn), _p(segs), _p(cu_p), _p(cu_q), _p(cu_s),
        ctypes.c_int(inp["R"]), ctypes.c_int(Hq), ctypes.c_int(inp["Hkv"]), ctypes.c_int(d),
        ctypes.c_double(inp["scale"]), ctypes.c_int(lo), ctypes.c_int(hi), ctypes.c_int(tlo),
        ctypes.c_int(thi), _p(out))
    if rc != OK:
        raise ValueError("oracle_packed_attn: invalid arguments (rc=%d)" % rc)
    return out


def dense_mask(segs, L: int, N: int) -> np.ndarray:
    """Explicit [N, L+N] visibility matrix of one request (uint8)."""
    segs = _c(segs, np.int32)
    m = np.zeros((N, L + N), np.uint8)
    rc = _load().oracle_dense_mask(_p(segs), ctypes.c_int(len(segs)), ctypes.c_int(L),
                                   ctypes.c_int(N), _p(m))
    if rc != OK:
        raise ValueError("oracle_dense_mask: invalid segments")
    return m


def dense_attn(inp: dict) -> np.ndarray:
    """Dense masked attention of a single request (explicit mask), fp64."""
    assert inp["R"] == 1
    q, kp, vp, kn, vn = (_c(inp[k], np.uint16) for k in ("q", "kp", "vp", "kn", "vn"))
    segs = _c(inp["segs"], np.int32)
    NT, Hq, d = q.shape
    L = int(inp["cu_prefix"][1])
    out = np.zeros((NT, Hq, d), np.float64)
    rc = _load().oracle_dense_attn(_p(q), _p(kp), _p(vp), _p(kn), _p(vn), _p(segs),
                                   ctypes.c_int(len(segs)), ctypes.c_int(L), ctypes.c_int(NT),
                                   ctypes.c_int(Hq), ctypes.c_int(inp["Hkv"]), ctypes.c_int(d),
                                   ctypes.c_double(inp["scale"]), _p(out))
    if rc != OK:
        raise ValueError("oracle_dense_attn: invalid arguments")
    return out


def spec_verify(inp: dict) -> dict:
    """Speculative-sampling verification of R requests, fp64.

    D3D, "Background / speculative decoding" and DScout, "Background":
    alpha_j = min(1, P_j(y_j)/Q_j(y_j)); accept while u_j < alpha_j; at the
    first rejection resample from norm(max(0, P - Q)), or add a bonus token
    from P_B when all B-1 drafts are accepted.
    """
    R, B, V = inp["R"], inp["B"], inp["V"]
    dt = np.uint16 if inp["dtype"] == 1 else np.float32
    tgt, dr = _c(inp["target"], dt), _c(inp["draft"], dt)
    y = _c(inp["y"], np.int32)
    ua, us = _c(inp["u_accept"], np.float32), _c(inp["u_sample"], np.float32)
    out = dict(accept_len=np.zeros(R, np.int32), out_tokens=np.zeros((R, B), np.int32),
               num_tokens=np.zeros(R, np.int32), alpha=np.zeros((R, B - 1)),
               p=np.zeros((R, B - 1)), q=np.zeros((R, B - 1)), margin_accept=np.zeros(R),
               margin_sample=np.zeros(R), used_fallback=np.zeros(R, np.int32))
    rc = _load().oracle_spec_verify(
        _p(tgt), _p(dr), ctypes.c_int(inp["dtype"]), _p(y), _p(ua), _p(us), ctypes.c_int(R),
        ctypes.c_int(B), ctypes.c_int(V), ctypes.c_double(inp.get("temperature", 1.0)),
        _p(out["accept_len"]), _p(out["out_tokens"]), _p(out["num_tokens"]), _p(out["alpha"]),
        _p(out["p"]), _p(out["q"]), _p(out["margin_accept"]), _p(out["margin_sample"]),
        _p(out["used_fallback"]))
    if rc != OK:
        raise ValueError("oracle_spec_verify: invalid arguments (rc=%d)" % rc)
    return out


def awl_weights(alpha) -> np.ndarray:
    """Acceptance-weighted loss weights w [R, B-1] from alpha [R, B-1]
    (DScout, "Background: AWL and the acceptance rule"): w_k = prod_{j<k}
    alpha_j, w_0 = 1 -- the probability that verification reaches k."""
    a = _c(alpha, np.float64)
    if a.ndim != 2:
        raise ValueError("alpha must be [R, B-1]")
    w = np.zeros_like(a)
    rc = _load().oracle_awl_weights(_p(a), ctypes.c_int(a.shape[0]), ctypes.c_int(a.shape[1]), _p(w))
    if rc != OK:
        raise ValueError("oracle_awl_weights: invalid arguments (rc=%d)" % rc)
    return w


def accept_probs(inp: dict) -> dict:
    """Per-position acceptance probabilities a_j = sum_v min(P_j, Q_j), the
    prefix survivals S(k) = a_1 ... a_k and tau = 1 + sum_k S(k) of every
    request (DScout, "Background: acceptance length tau", "Background: AWL
    and the acceptance rule"); fp64 softmax at temperature T."""
    R, B, V = inp["R"], inp["B"], inp["V"]
    dt = np.uint16 if inp["dtype"] == 1 else np.float32
    tgt, dr = _c(inp["target"], dt), _c(inp["draft"], dt)
    out = dict(accept_prob=np.zeros((R, B - 1)), survival=np.zeros((R, B - 1)), tau=np.zeros(R))
    rc = _load().oracle_accept_probs(_p(tgt), _p(dr), ctypes.c_int(inp["dtype"]), ctypes.c_int(R), ctypes.c_int(B),
                                     ctypes.c_int(V), ctypes.c_double(inp.get("temperature", 1.0)),
                                     _p(out["accept_prob"]), _p(out["survival"]), _p(out["tau"]))
    if rc != OK:
        raise ValueError("oracle_accept_probs: invalid arguments (rc=%d)" % rc)
    return out


def build_branches(inp: dict) -> dict:
    """Branch construction for the asynchronous packed pass (D3D, "Background:
    asynchronous drafting and cache hits", "Method steps" step 4).

    Anchors of rejection position r: the F most likely tokens of the draft row
    Q_r (largest logit first, ties to the lowest index), y_r excluded; heads,
    head lengths and the packed pass's segment rows (see d3d_oracle.c).
    ``bonus_guess`` [R] is optional.
    """
    R, B, V, C, F = inp["R"], inp["B"], inp["V"], inp["C"], inp["F"]
    dt = np.uint16 if inp["dtype"] == 1 else np.float32
    dr, y = _c(inp["draft"], dt), _c(inp["y"], np.int32)
    bg = inp.get("bonus_guess")
    bg = None if bg is None else _c(bg, np.int32)
    M = (C - 1) * F + 2
    out = dict(anchors=np.zeros((R, max(C - 1, 0), F), np.int32), heads=np.zeros((R, M, B), np.int32),
               head_len=np.zeros((R, M), np.int32), segs=np.zeros((R * M, 5), np.int32),
               cu_q=np.zeros(R + 1, np.int32), cu_seg=np.zeros(R + 1, np.int32))
    rc = _load().oracle_build_branches(
        _p(dr), ctypes.c_int(inp["dtype"]), _p(y), None if bg is None else _p(bg), ctypes.c_int(R), ctypes.c_int(B),
        ctypes.c_int(V), ctypes.c_int(C), ctypes.c_int(F), _p(out["anchors"]), _p(out["heads"]),
        _p(out["head_len"]), _p(out["segs"]), _p(out["cu_q"]), _p(out["cu_seg"]))
    if rc != OK:
        raise ValueError("oracle_build_branches: invalid arguments (rc=%d)" % rc)
    return out


def greedy_verify(inp: dict) -> dict:
    """Greedy (temperature 0) verification of R requests.

    D3D, "Experiments" and DScout, "Experiments" (greedy decoding): the T -> 0
    limit of the sampling rule.  Accept y_j iff it is the target's argmax
    (ties to the lowest index); emit the target's argmax at the first
    rejection, or the bonus argmax of row B-1.  Only the target logits are read.
    """
    R, B, V = inp["R"], inp["B"], inp["V"]
    dt = np.uint16 if inp["dtype"] == 1 else np.float32
    tgt = _c(inp["target"], dt)
    y = _c(inp["y"], np.int32)
    out = dict(accept_len=np.zeros(R, np.int32), out_tokens=np.zeros((R, B), np.int32),
               num_tokens=np.zeros(R, np.int32), accept=np.zeros((R, B - 1)), argmax=np.zeros((R, B), np.int32))
    rc = _load().oracle_greedy_verify(
        _p(tgt), ctypes.c_int(inp["dtype"]), _p(y), ctypes.c_int(R), ctypes.c_int(B), ctypes.c_int(V),
        _p(out["accept_len"]), _p(out["out_tokens"]), _p(out["num_tokens"]), _p(out["accept"]), _p(out["argmax"]))
    if rc != OK:
        raise ValueError("oracle_greedy_verify: invalid arguments (rc=%d)" % rc)
    return out


def branch_match(inp: dict) -> np.ndarray:
    """Branch cache-hit match (D3D, "Background / asynchronous drafting and cache hits")."""
    v, vl = _c(inp["verified"], np.int32), _c(inp["verified_len"], np.int32)
    h, hl = _c(inp["heads"], np.int32), _c(inp["head_len"], np.int32)
    R, M, B = h.shape
    out = np.zeros(R, np.int32)
    rc = _load().oracle_branch_match(_p(v), _p(vl), _p(h), _p(hl), ctypes.c_int(R), ctypes.c_int(M),
                                     ctypes.c_int(B), _p(out))
    if rc != OK:
        raise ValueError("oracle_branch_match: invalid arguments")
    return out
