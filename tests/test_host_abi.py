"""The C-ABI library on the host (no GPU): it loads, exports every symbol the
header declares, rejects bad arguments before touching the device, and its
host-side segment check agrees with the oracle's rules."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest
import torch

import oracle
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def d3d():
    import __graft_entry__

    __graft_entry__._build_module().build()
    import diffusion_drafted_speculative_gb300 as mod

    return mod


def _header_functions():
    src = open(os.path.join(ROOT, "include", "d3d.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(d3d_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_three_calls():
    names = _header_functions()
    for n in ("d3d_packed_draft_attn", "d3d_spec_verify", "d3d_branch_match"):
        assert n in names


def test_every_declared_symbol_is_exported(d3d):
    names = _header_functions()
    out = subprocess.run(["nm", "-D", "--defined-only", d3d.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (d3d_\w+)", out))
    for n in names:
        assert n in exported, n
        assert hasattr(d3d.lib, n)
    # the binding covers every declared function
    assert set(d3d.EXPORTED) == set(names)


def test_status_strings(d3d):
    for rc in (0, -1, -2, -3, -4, -5, -6, 17):
        assert isinstance(d3d.d3d_status_string(rc), str)
    assert d3d.d3d_status_string(0) == "ok"
    assert d3d.d3d_version() >= 100


def test_workspace_sizes(d3d):
    assert d3d.d3d_spec_verify_workspace_size(1, 16, 151936) > 256
    assert d3d.d3d_spec_verify_workspace_size(1, 1, 10) == 0
    assert d3d.d3d_packed_draft_attn_workspace_size(1, 32, 8, 128, 384, 2048) >= 256
    big = d3d.d3d_spec_verify_workspace_size(16, 16, 151936)
    assert big > d3d.d3d_spec_verify_workspace_size(1, 16, 151936)


def test_invalid_arguments_rejected_on_host(d3d):
    L = d3d.lib
    fake = ctypes.c_void_p(256)  # never dereferenced: the checks fail first
    # verify: B < 2, V < 1, T <= 0, bad dtype, missing workspace
    args = lambda R, B, V, T, dt, ws, wsb, sm=0, M=0, heads=None, br=None, fl=0, q=None: (  # noqa
        fake, fake, dt, fake, fake, fake, R, B, V, T, fake, fake, fake, None, None, q, None, heads, heads, M, br, ws,
        wsb, sm, fl, None)
    assert L.d3d_spec_verify(*args(1, 1, 10, 1.0, 1, fake, 1 << 20)) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_spec_verify(*args(1, 4, 10, 1.0, 1, fake, 1 << 20, fl=2)) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_spec_verify(*args(1, 4, 0, 1.0, 1, fake, 1 << 20)) == d3d.D3D_ERR_INVALID_ARG
    # temperature 0 is greedy verification, which reads no draft logits: q_draft must be NULL
    assert L.d3d_spec_verify(*args(1, 4, 10, 0.0, 1, fake, 1 << 20, q=fake)) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_spec_verify(*args(1, 4, 10, -0.5, 1, fake, 1 << 20)) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_spec_verify(*args(1, 4, 10, -1.0, 1, fake, 1 << 20)) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_spec_verify(*args(1, 4, 10, float("nan"), 1, fake, 1 << 20)) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_spec_verify(*args(1, 4, 10, 1.0, 7, fake, 1 << 20)) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_spec_verify(*args(1, 4, 10, 1.0, 1, None, 1 << 20)) == d3d.D3D_ERR_WORKSPACE
    assert L.d3d_spec_verify(*args(1, 4, 10, 1.0, 1, fake, 16)) == d3d.D3D_ERR_WORKSPACE
    assert L.d3d_spec_verify(*args(1, 4, 10, 1.0, 1, ctypes.c_void_p(264), 1 << 20)) == d3d.D3D_ERR_WORKSPACE
    assert L.d3d_spec_verify(*args(1, 300, 10, 1.0, 1, fake, 1 << 30)) == d3d.D3D_ERR_UNSUPPORTED
    assert L.d3d_spec_verify(*args(1, 257, 10, 1.0, 1, fake, 1 << 30)) == d3d.D3D_ERR_UNSUPPORTED
    assert L.d3d_spec_verify(*args(1, 4, 8388609, 1.0, 1, fake, 1 << 40)) == d3d.D3D_ERR_UNSUPPORTED
    assert d3d.d3d_spec_verify_workspace_size(1, 257, 10) == 0
    assert d3d.d3d_spec_verify_workspace_size(1, 4, 8388609) == 0
    assert d3d.d3d_spec_verify_workspace_size(1, 256, 8388608) > 256
    assert L.d3d_spec_verify(*args(0, 4, 10, 1.0, 1, None, 0)) == d3d.D3D_OK  # nothing to do
    assert L.d3d_spec_verify(*args(1, 4, 10, 1.0, 1, fake, 1 << 20, -1)) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_spec_verify(*args(1, 4, 10, 1.0, 1, fake, 1 << 20, 0, -1)) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_spec_verify(*args(1, 4, 10, 1.0, 1, fake, 1 << 20, 0, 3, None, fake)) == d3d.D3D_ERR_INVALID_ARG

    def attn(R=1, Hq=32, Hkv=8, d=128, max_q=16, scale=0.1, ws=fake, wsb=1 << 30, flags=0, max_ctas=0):
        return L.d3d_packed_draft_attn(fake, fake, fake, fake, fake, fake, fake, fake, fake, R, Hq, Hkv, d, max_q,
                                       64, 16, 64, 1, scale, fake, ws, wsb, max_ctas, flags, None)
    assert attn(flags=3) == d3d.D3D_ERR_INVALID_ARG  # the two placement bits are exclusive
    assert attn(flags=4) == d3d.D3D_ERR_INVALID_ARG
    assert attn(max_ctas=-1) == d3d.D3D_ERR_INVALID_ARG
    assert attn(Hq=30, Hkv=8) == d3d.D3D_ERR_INVALID_ARG
    assert attn(d=96) == d3d.D3D_ERR_UNSUPPORTED
    assert attn(Hq=24, Hkv=8) == d3d.D3D_ERR_UNSUPPORTED  # G = 3 does not divide 128
    assert attn(max_q=8193) == d3d.D3D_ERR_UNSUPPORTED
    assert L.d3d_packed_draft_attn(ctypes.c_void_p(264), fake, fake, fake, fake, fake, fake, fake, fake, 1, 32, 8,
                                   128, 16, 64, 16, 64, 1, 0.1, fake, fake, 1 << 30, 0, 0, None) == d3d.D3D_ERR_INVALID_ARG
    assert attn(scale=0.0) == d3d.D3D_ERR_INVALID_ARG
    assert attn(scale=float("inf")) == d3d.D3D_ERR_INVALID_ARG
    assert attn(ws=None) == d3d.D3D_ERR_WORKSPACE
    assert attn(R=0) == d3d.D3D_OK
    ctas = L.d3d_packed_draft_attn_ctas
    assert ctas(1, 32, 8, 128, 16, 64, -1) == d3d.D3D_ERR_INVALID_ARG
    assert ctas(1, 30, 8, 128, 16, 64, 0) == d3d.D3D_ERR_INVALID_ARG
    assert ctas(1, 32, 8, 96, 16, 64, 0) == d3d.D3D_ERR_UNSUPPORTED
    assert ctas(1, 24, 8, 128, 16, 64, 0) == d3d.D3D_ERR_UNSUPPORTED
    assert ctas(0, 32, 8, 128, 16, 64, 0) == 0 and ctas(1, 32, 8, 128, 0, 64, 0) == 0

    # the fused round: missing calls, then each part's own argument checks
    assert L.d3d_async_round(None, None, None) == d3d.D3D_ERR_INVALID_ARG
    ac = d3d.AttnCall(*([fake] * 9 + [1, 30, 8, 128, 16, 64, 16, 64, 1, 0.1, fake, fake, 1 << 30]))
    vc = d3d.VerifyCall(fake, fake, 1, fake, fake, fake, 1, 4, 10, 1.0, fake, fake, fake, None, None, None, None,
                        None, None, 0, None, fake, 1 << 20)
    assert L.d3d_async_round(ctypes.byref(ac), ctypes.byref(vc), None) == d3d.D3D_ERR_INVALID_ARG  # Hq % Hkv
    ac.Hq = 32
    vc.temperature = -1.0
    assert L.d3d_async_round(ctypes.byref(ac), ctypes.byref(vc), None) == d3d.D3D_ERR_INVALID_ARG  # T < 0
    vc.temperature = 0.0  # greedy verification has a launch of its own
    assert L.d3d_async_round(ctypes.byref(ac), ctypes.byref(vc), None) == d3d.D3D_ERR_UNSUPPORTED
    vc.temperature = 1.0
    ac.d = 96
    assert L.d3d_async_round(ctypes.byref(ac), ctypes.byref(vc), None) == d3d.D3D_ERR_UNSUPPORTED

    # acceptance probabilities: argument checks before any device work
    ap = lambda R=1, B=16, V=100, T=1.0, out=fake, ws=fake, wsb=1 << 20: (  # noqa
        fake, fake, d3d.D3D_DTYPE_BF16, R, B, V, T, out, None, None, ws, wsb, None)
    assert L.d3d_accept_probs(*ap(T=0.0)) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_accept_probs(*ap(T=float("inf"))) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_accept_probs(*ap(B=1)) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_accept_probs(*ap(out=None)) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_accept_probs(*ap(B=300)) == d3d.D3D_ERR_UNSUPPORTED
    assert L.d3d_accept_probs(*ap(ws=None)) == d3d.D3D_ERR_WORKSPACE
    assert L.d3d_accept_probs(*ap(R=0)) == d3d.D3D_OK
    assert d3d.d3d_accept_probs_workspace_size(1, 16, 151936) > 256

    # branch construction: shapes and flags checked before any device work
    bb = lambda R=1, B=16, V=100, C=12, F=2, anc=fake, h=fake, hl=fake, cq=None, cs=None, ws=fake, wsb=1 << 20: (  # noqa
        fake, d3d.D3D_DTYPE_BF16, fake, None, R, B, V, C, F, anc, h, hl, None, cq, cs, ws, wsb, None)
    assert L.d3d_build_branches(*bb(C=17)) == d3d.D3D_ERR_INVALID_ARG        # C > B
    assert L.d3d_build_branches(*bb(C=0)) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_build_branches(*bb(F=-1)) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_build_branches(*bb(V=2)) == d3d.D3D_ERR_INVALID_ARG         # F > V - 1
    assert L.d3d_build_branches(*bb(F=9)) == d3d.D3D_ERR_UNSUPPORTED
    assert L.d3d_build_branches(*bb(B=257)) == d3d.D3D_ERR_UNSUPPORTED
    assert L.d3d_build_branches(*bb(cq=fake)) == d3d.D3D_ERR_INVALID_ARG     # cu_q without cu_seg
    assert L.d3d_build_branches(*bb(h=None)) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_build_branches(*bb(anc=None)) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_build_branches(*bb(ws=None)) == d3d.D3D_ERR_WORKSPACE
    assert L.d3d_build_branches(*bb(R=0)) == d3d.D3D_OK
    assert d3d.d3d_build_branches_workspace_size(1, 16, 151936, 12, 2) > 256
    assert d3d.d3d_build_branches_workspace_size(1, 16, 151936, 17, 2) == 0

    assert L.d3d_branch_match(fake, fake, fake, fake, 1, 2, 0, fake, None) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_branch_match(None, fake, fake, fake, 1, 2, 4, fake, None) == d3d.D3D_ERR_INVALID_ARG
    assert L.d3d_branch_match(fake, fake, fake, fake, 0, 2, 4, fake, None) == d3d.D3D_OK


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32)))


@pytest.mark.parametrize("bad", [None, "overlap", "gap", "shifted", "later_parent", "bidir_parent",
                                 "bidir_parent_alone", "long_parent", "nested", "len_without_parent", "empty_seg",
                                 "short_total", "bad_mode", "neg_parent_len", "cu_start"])
def test_validate_segments_matches_oracle_rules(d3d, bad):
    segs = W.async_segments(4, 3, 2).astype(np.int64)
    N = int(segs[:, 1].sum())
    cu_q, cu_seg = [0, N], [0, len(segs)]
    if bad == "overlap":
        segs[2, 0] -= 1
    elif bad == "gap":
        segs[2:, 0] += 1
        cu_q = [0, N + 1]
    elif bad == "shifted":
        segs[2, 0] += 1
    elif bad == "later_parent":
        segs[1, 3] = 2
    elif bad == "bidir_parent":
        segs[2, 3] = 1
    elif bad == "bidir_parent_alone":
        segs[1, 3], segs[1, 4] = -1, 0
        segs[2, 3], segs[2, 4] = 1, 1
    elif bad == "long_parent":
        segs[1, 4] = 5
    elif bad == "nested":
        segs[1, 2] = W.SEG_CAUSAL
        segs[2, 3], segs[2, 4] = 1, 1
    elif bad == "len_without_parent":
        segs[0, 4] = 1
    elif bad == "empty_seg":
        segs[3, 1] = 0
        segs[4:, 0] -= 4
        cu_q = [0, N - 4]
    elif bad == "short_total":
        cu_q = [0, N + 3]
    elif bad == "bad_mode":
        segs[1, 2] = 7
    elif bad == "neg_parent_len":
        segs[1, 4] = -1
    elif bad == "cu_start":
        cu_q, cu_seg = [1, N + 1], [0, len(segs)]
    got = d3d.d3d_validate_segments(_t(segs), _t(cu_q), _t(cu_seg))
    exp = oracle.check_segments(segs, cu_q, cu_seg)
    assert (got == 0) == (exp == 0)
    assert (got == 0) == (bad is None)


def test_validate_segments_random_tables_agree_with_oracle(d3d):
    rng = np.random.default_rng(5)
    for _ in range(300):
        R = int(rng.integers(1, 4))
        rows, cu_q, cu_seg = [], [0], [0]
        for _r in range(R):
            n_seg = int(rng.integers(1, 6))
            q = 0
            for s in range(n_seg):
                ln = int(rng.integers(0, 5))
                rows.append([q + int(rng.integers(-1, 2)) * (rng.random() < 0.1), ln, int(rng.integers(0, 3)) % 2
                             if rng.random() < 0.95 else 5, int(rng.integers(-1, s + 1)) if s else -1,
                             int(rng.integers(0, 4))])
                if rows[-1][3] == -1 and rng.random() < 0.9:
                    rows[-1][4] = 0
                q += ln
            cu_q.append(cu_q[-1] + q + (1 if rng.random() < 0.05 else 0))
            cu_seg.append(cu_seg[-1] + n_seg)
        segs = np.array(rows, np.int64)
        got = d3d.d3d_validate_segments(_t(segs), _t(cu_q), _t(cu_seg))
        exp = oracle.check_segments(segs, cu_q, cu_seg)
        assert (got == 0) == (exp == 0), (segs, cu_q, cu_seg)


def test_binding_rejects_cpu_tensors(d3d):
    x = torch.zeros(1, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        d3d.d3d_packed_draft_attn(x, x, x, x, x, torch.zeros(1, 5, dtype=torch.int32),
                                  *(torch.zeros(2, dtype=torch.int32),) * 3, 1, 1, 0.1, x,
                                  torch.zeros(256, dtype=torch.uint8))


def test_noalloc_limit_edge_in_workspace_sizes(d3d):
    # the no-allocation entry point's fixed scratch (2 MiB) holds the
    # workspace of 211 requests at B = 16, V = 151936 but not of 212
    assert d3d.d3d_spec_verify_workspace_size(211, 16, 151936) <= 2 << 20
    assert d3d.d3d_spec_verify_workspace_size(212, 16, 151936) > 2 << 20



def test_debug_build_exports_every_symbol(d3d):
    # the build with device-side internal index checks has the same entry points
    import __graft_entry__

    path = __graft_entry__._build_module().build(debug=True)
    assert os.path.basename(path) == "libd3d_debug.so"
    so = ctypes.CDLL(path)
    for name in _header_functions():
        assert hasattr(so, name), name
    fn = so.d3d_status_string
    fn.restype = ctypes.c_char_p
    fn.argtypes = [ctypes.c_int]
    assert b"internal index check" in fn(d3d.D3D_ERR_INTERNAL)
