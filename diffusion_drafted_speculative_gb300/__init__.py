"""GB300 (sm_103a) hot path of diffusion-drafted speculative decoding.

Thin Python binding of the C ABI in ``include/d3d.h`` (library
``libd3d.so`` built from ``csrc/`` by :mod:`.build`).  The functions carry the
C names and only marshal arguments: shapes, dtypes and devices are checked,
sizes are read off the tensors, pointers and the current CUDA stream are
passed through.  Every step runs in the library's kernels; there is no
fallback of any kind.  If the library is missing, importing this package
raises ImportError.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "D3DError", "lib", "d3d_status_string", "d3d_version", "d3d_validate_segments",
    "d3d_packed_draft_attn", "d3d_packed_draft_attn_workspace_size", "d3d_packed_draft_attn_ctas",
    "d3d_spec_verify", "d3d_spec_verify_workspace_size", "d3d_spec_verify_slice_ctas", "d3d_spec_verify_noalloc",
    "d3d_async_round",
    "AttnCall", "VerifyCall", "d3d_build_branches", "d3d_build_branches_workspace_size",
    "d3d_accept_probs", "d3d_accept_probs_workspace_size", "d3d_branch_match", "d3d_workspace_status", "d3d_workspace_init", "d3d_debug_inject_fault", "d3d_debug_force_attn_kernel", "new_workspace", "EXPORTED",
    "D3D_OK", "D3D_ERR_INVALID_ARG", "D3D_ERR_UNSUPPORTED", "D3D_ERR_WORKSPACE", "D3D_ERR_CUDA",
    "D3D_ERR_DEVICE_TIMEOUT", "D3D_ERR_DEVICE_INPUT", "D3D_ERR_INTERNAL", "D3D_DTYPE_F32", "D3D_DTYPE_BF16",
    "D3D_SEG_CAUSAL", "D3D_SEG_BIDIR", "D3D_ATTN_AFTER_INDEPENDENT", "D3D_ATTN_AFTER_DEPENDENT",
    "D3D_VERIFY_AFTER_INDEPENDENT",
]

D3D_OK = 0
D3D_ERR_INVALID_ARG = -1
D3D_ERR_UNSUPPORTED = -2
D3D_ERR_WORKSPACE = -3
D3D_ERR_CUDA = -4
D3D_ERR_DEVICE_TIMEOUT = -5
D3D_ERR_DEVICE_INPUT = -6
D3D_ERR_INTERNAL = -7
D3D_DTYPE_F32 = 0
D3D_DTYPE_BF16 = 1
D3D_SEG_CAUSAL = 0
D3D_SEG_BIDIR = 1
D3D_ATTN_AFTER_INDEPENDENT = 1
D3D_ATTN_AFTER_DEPENDENT = 2
D3D_VERIFY_AFTER_INDEPENDENT = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
# D3D_LIBRARY=debug selects the build with device-side internal index checks
# (libd3d_debug.so, built beside libd3d.so; same entry points and results)
LIB_PATH = os.path.join(_HERE, "libd3d_debug.so" if os.environ.get("D3D_LIBRARY") == "debug" else "libd3d.so")

_P, _I, _F, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
# name -> (restype, argtypes): every symbol declared in include/d3d.h
EXPORTED = {
    "d3d_status_string": (ctypes.c_char_p, [_I]),
    "d3d_version": (_I, []),
    "d3d_workspace_init": (_I, [_P, _Z, _P]),
    "d3d_workspace_status": (_I, [_P, _P, _I, _P]),
    "d3d_validate_segments": (_I, [_P, _P, _P, _I]),
    "d3d_packed_draft_attn_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I]),
    "d3d_packed_draft_attn": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                                   _F, _P, _P, _Z, _I, _I, _P]),
    "d3d_spec_verify_workspace_size": (_Z, [_I, _I, _I]),
    "d3d_spec_verify_slice_ctas": (_I, [_I, _I, _I, _I, _F, _I, _Z]),
    "d3d_packed_draft_attn_ctas": (_I, [_I, _I, _I, _I, _I, _I, _I]),
    "d3d_spec_verify": (_I, [_P, _P, _I, _P, _P, _P, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I,
                             _P, _P, _Z, _I, _I, _P]),
    "d3d_branch_match": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "d3d_debug_inject_fault": (None, [_I]),
    "d3d_debug_force_attn_kernel": (None, [_I]),
    "d3d_spec_verify_noalloc": (_I, [_P, _P, _I, _P, _P, _P, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _P]),
    "d3d_async_round": (_I, [_P, _P, _P]),
    "d3d_build_branches_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "d3d_accept_probs_workspace_size": (_Z, [_I, _I, _I]),
    "d3d_accept_probs": (_I, [_P, _P, _I, _I, _I, _I, _F, _P, _P, _P, _P, _Z, _P]),
    "d3d_build_branches": (_I, [_P, _I, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _Z, _P]),
}


class D3DError(RuntimeError):
    """A libd3d call returned a non-OK status."""

    def __init__(self, name: str, rc: int):
        super().__init__("%s failed: %s (%d)" % (name, d3d_status_string(rc), rc))
        self.rc = rc


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError("%s is not built (expected at %s); run "
                          "`python diffusion_drafted_speculative_gb300/build.py` (or __graft_entry__.build())"
                          % (os.path.basename(LIB_PATH), LIB_PATH))
    so = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in EXPORTED.items():
        fn = getattr(so, name)
        fn.restype, fn.argtypes = res, args
    return so


lib = _load()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need(t, name, dtype, ndim=None, cuda=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dims, got shape %s" % (name, ndim, tuple(t.shape)))
    if cuda and not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _check(name, rc):
    if rc != D3D_OK:
        raise D3DError(name, rc)


def d3d_status_string(rc: int) -> str:
    return lib.d3d_status_string(int(rc)).decode()


def d3d_version() -> int:
    return lib.d3d_version()


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """Zero-filled uint8 device buffer for a workspace (torch allocations are 256-byte aligned)."""
    ws = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")
    if ws.data_ptr() % 256:
        raise RuntimeError("workspace allocation is not 256-byte aligned")
    return ws


def d3d_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check("d3d_workspace_init", lib.d3d_workspace_init(_ptr(ws), ws.numel(), _stream(stream)))


def d3d_workspace_status(ws: torch.Tensor, clear: bool = False, stream=None) -> int:
    out = ctypes.c_int32(0)
    _check("d3d_workspace_status",
           lib.d3d_workspace_status(_ptr(ws), ctypes.addressof(out), int(bool(clear)), _stream(stream)))
    return out.value


def d3d_validate_segments(segs: torch.Tensor, cu_q: torch.Tensor, cu_seg: torch.Tensor) -> int:
    """Host-side check of a segment table (CPU int32 tensors); returns the status code."""
    _need(segs, "segs", torch.int32, 2, cuda=False)
    _need(cu_q, "cu_q", torch.int32, 1, cuda=False)
    _need(cu_seg, "cu_seg", torch.int32, 1, cuda=False)
    if segs.is_cuda or cu_q.is_cuda or cu_seg.is_cuda:
        raise ValueError("d3d_validate_segments takes host (CPU) tensors")
    if segs.numel() and segs.shape[1] != 5:
        raise ValueError("segs must be [n, 5]")
    return lib.d3d_validate_segments(_ptr(segs) if segs.numel() else None, _ptr(cu_q), _ptr(cu_seg),
                                     cu_q.numel() - 1)


def d3d_debug_inject_fault(mode: int) -> None:
    """Failure-detection hook: 1 makes later attention launches time out on purpose, 0 restores."""
    lib.d3d_debug_inject_fault(int(mode))


def d3d_debug_force_attn_kernel(kind: int) -> None:
    """Restrict later attention plans to one kernel: 1 one tile per CTA, 2 two tiles per CTA, 3 CTA pairs
    (where it applies); 0 restores the plan's own choice."""
    lib.d3d_debug_force_attn_kernel(int(kind))


def d3d_packed_draft_attn_workspace_size(R, Hq, Hkv, d, max_q, max_prefix) -> int:
    return int(lib.d3d_packed_draft_attn_workspace_size(R, Hq, Hkv, d, max_q, max_prefix))


def d3d_spec_verify_slice_ctas(R, B, V, logits_dtype, temperature, sm_limit: int = 0, ws_bytes=None) -> int:
    """CTAs of the vocabulary-slice verification launch for these sizes (0: the
    call takes the chunked or greedy launch); ws_bytes defaults to
    d3d_spec_verify_workspace_size."""
    if ws_bytes is None:
        ws_bytes = lib.d3d_spec_verify_workspace_size(R, B, V)
    n = int(lib.d3d_spec_verify_slice_ctas(R, B, V, int(logits_dtype), float(temperature), int(sm_limit),
                                           int(ws_bytes)))
    if n < 0:
        _check("d3d_spec_verify_slice_ctas", n)
    return n


def d3d_packed_draft_attn_ctas(R, Hq, Hkv, d, max_q, max_prefix, max_ctas: int = 0) -> int:
    """CTAs (one SM each) the attention launch uses on the current device."""
    n = int(lib.d3d_packed_draft_attn_ctas(R, Hq, Hkv, d, max_q, max_prefix, int(max_ctas)))
    if n < 0:
        _check("d3d_packed_draft_attn_ctas", n)
    return n


def _attn_args(q, k_prefix, v_prefix, k_packed, v_packed, segs, cu_prefix, cu_q, cu_seg, max_q, max_prefix, scale,
               out, ws):
    """Checked argument tuple of d3d_packed_draft_attn (without flags and stream)."""
    for t, n in ((q, "q"), (k_prefix, "k_prefix"), (v_prefix, "v_prefix"), (k_packed, "k_packed"),
                 (v_packed, "v_packed"), (out, "out")):
        _need(t, n, torch.bfloat16, 3)
    _need(segs, "segs", torch.int32, 2)
    for t, n in ((cu_prefix, "cu_prefix"), (cu_q, "cu_q"), (cu_seg, "cu_seg")):
        _need(t, n, torch.int32, 1)
    _need(ws, "ws", torch.uint8, 1)
    NT, Hq, d = q.shape
    LT, Hkv = k_prefix.shape[0], k_prefix.shape[1]
    if (k_packed.shape != (NT, Hkv, d) or v_packed.shape != (NT, Hkv, d) or v_prefix.shape != k_prefix.shape
            or k_prefix.shape[2] != d or out.shape != q.shape or segs.shape[1] != 5):
        raise ValueError("inconsistent attention shapes")
    R = cu_q.numel() - 1
    if cu_prefix.numel() != R + 1 or cu_seg.numel() != R + 1:
        raise ValueError("cu_prefix, cu_q and cu_seg must all have R+1 entries")
    return (_ptr(q), _ptr(k_prefix), _ptr(v_prefix), _ptr(k_packed), _ptr(v_packed), _ptr(segs), _ptr(cu_prefix),
            _ptr(cu_q), _ptr(cu_seg), R, Hq, Hkv, d, int(max_q), int(max_prefix), NT, LT, segs.shape[0],
            float(scale), _ptr(out), _ptr(ws), ws.numel())


def d3d_packed_draft_attn(q, k_prefix, v_prefix, k_packed, v_packed, segs, cu_prefix, cu_q, cu_seg,
                          max_q: int, max_prefix: int, scale: float, out, ws, after_independent: bool = False,
                          stream=None, max_ctas: int = 0, after_dependent: bool = False) -> None:
    """Packed drafting attention; shapes as in include/d3d.h (bf16 tensors, int32 tables).
    max_ctas > 0 bounds the launch to one wave of that many CTAs (SMs).  after_independent /
    after_dependent set D3D_ATTN_AFTER_INDEPENDENT / D3D_ATTN_AFTER_DEPENDENT (not both)."""
    args = _attn_args(q, k_prefix, v_prefix, k_packed, v_packed, segs, cu_prefix, cu_q, cu_seg, max_q, max_prefix,
                      scale, out, ws)
    flags = (D3D_ATTN_AFTER_INDEPENDENT if after_independent else 0) | \
        (D3D_ATTN_AFTER_DEPENDENT if after_dependent else 0)
    rc = lib.d3d_packed_draft_attn(*args, int(max_ctas), flags, _stream(stream))
    _check("d3d_packed_draft_attn", rc)


def d3d_spec_verify_workspace_size(R, B, V) -> int:
    return int(lib.d3d_spec_verify_workspace_size(R, B, V))


def _verify_args(target_logits, draft_logits, draft_tokens, u_accept, u_sample, temperature, accept_len, out_tokens,
                 num_tokens, ws, alpha, p_draft, q_draft, heads, head_len, branch, awl_weight=None):
    """Checked argument tuple of d3d_spec_verify (without sm_limit and stream).

    temperature 0 is greedy verification: draft_logits, u_accept and u_sample
    may then be None (they are not read) and q_draft must be None.
    """
    greedy = float(temperature) == 0.0
    if target_logits.dtype == torch.bfloat16:
        dt = D3D_DTYPE_BF16
    elif target_logits.dtype == torch.float32:
        dt = D3D_DTYPE_F32
    else:
        raise TypeError("logits must be float32 or bfloat16")
    _need(target_logits, "target_logits", target_logits.dtype, 3)
    R, B, V = target_logits.shape
    if not greedy or draft_logits is not None:
        _need(draft_logits, "draft_logits", target_logits.dtype, 3)
        if draft_logits.shape != (R, B - 1, V):
            raise ValueError("draft_logits must be [R, B-1, V]")
    _need(draft_tokens, "draft_tokens", torch.int32, 2)
    if not greedy or u_accept is not None or u_sample is not None:
        _need(u_accept, "u_accept", torch.float32, 2)
        _need(u_sample, "u_sample", torch.float32, 1)
        if u_accept.shape != (R, B - 1) or u_sample.shape != (R,):
            raise ValueError("u_accept must be [R, B-1], u_sample [R]")
    for t, n, shp in ((accept_len, "accept_len", (R,)), (out_tokens, "out_tokens", (R, B)),
                      (num_tokens, "num_tokens", (R,))):
        _need(t, n, torch.int32, len(shp))
        if tuple(t.shape) != shp:
            raise ValueError("%s must be %s" % (n, shp))
    for t, n in ((alpha, "alpha"), (p_draft, "p_draft"), (q_draft, "q_draft"), (awl_weight, "awl_weight")):
        if t is not None:
            _need(t, n, torch.float32, 2)
            if tuple(t.shape) != (R, B - 1):
                raise ValueError("%s must be [R, B-1]" % n)
    if draft_tokens.shape != (R, B - 1):
        raise ValueError("draft_tokens must be [R, B-1]")
    M = 0
    if branch is not None:
        _need(branch, "branch", torch.int32, 1)
        _need(heads, "heads", torch.int32, 3)
        _need(head_len, "head_len", torch.int32, 2)
        M = heads.shape[1]
        if tuple(heads.shape) != (R, M, B) or tuple(head_len.shape) != (R, M) or tuple(branch.shape) != (R,):
            raise ValueError("heads must be [R, M, B], head_len [R, M], branch [R]")
    if ws is not None:
        _need(ws, "ws", torch.uint8, 1)
    return (_ptr(target_logits), _ptr(draft_logits), dt, _ptr(draft_tokens), _ptr(u_accept), _ptr(u_sample), R, B, V,
            float(temperature), _ptr(accept_len), _ptr(out_tokens), _ptr(num_tokens), _ptr(alpha), _ptr(p_draft),
            _ptr(q_draft), _ptr(awl_weight), _ptr(heads) if branch is not None else None,
            _ptr(head_len) if branch is not None else None, M, _ptr(branch), _ptr(ws),
            ws.numel() if ws is not None else 0)


def d3d_spec_verify(target_logits, draft_logits, draft_tokens, u_accept, u_sample, temperature: float,
                    accept_len, out_tokens, num_tokens, ws, alpha=None, p_draft=None, q_draft=None,
                    heads=None, head_len=None, branch=None, sm_limit: int = 0, after_independent: bool = False,
                    stream=None, awl_weight=None) -> None:
    """Speculative-sampling verification; logits f32 or bf16 [R,B,V] / [R,B-1,V]."""
    args = _verify_args(target_logits, draft_logits, draft_tokens, u_accept, u_sample, temperature, accept_len,
                        out_tokens, num_tokens, ws, alpha, p_draft, q_draft, heads, head_len, branch, awl_weight)
    rc = lib.d3d_spec_verify(*args, int(sm_limit), D3D_VERIFY_AFTER_INDEPENDENT if after_independent else 0,
                             _stream(stream))
    _check("d3d_spec_verify", rc)


def d3d_build_branches_workspace_size(R, B, V, C, F) -> int:
    return int(lib.d3d_build_branches_workspace_size(R, B, V, C, F))


def d3d_build_branches(draft_logits, draft_tokens, C: int, F: int, heads, head_len, ws, anchors=None,
                       bonus_guess=None, segs=None, cu_q=None, cu_seg=None, stream=None) -> None:
    """Anchors, branch heads and the packed pass's segment rows (include/d3d.h).

    draft_logits [R, B-1, V] f32/bf16, draft_tokens [R, B-1] int32; outputs
    anchors [R, C-1, F], heads [R, M, B], head_len [R, M], segs [R*M, 5],
    cu_q / cu_seg [R+1] (int32), M = (C-1)F + 2.
    """
    if draft_logits.dtype == torch.bfloat16:
        dt = D3D_DTYPE_BF16
    elif draft_logits.dtype == torch.float32:
        dt = D3D_DTYPE_F32
    else:
        raise TypeError("logits must be float32 or bfloat16")
    _need(draft_logits, "draft_logits", draft_logits.dtype, 3)
    R, Bm1, V = draft_logits.shape
    B = Bm1 + 1
    M = (C - 1) * F + 2
    _need(draft_tokens, "draft_tokens", torch.int32, 2)
    if tuple(draft_tokens.shape) != (R, B - 1):
        raise ValueError("draft_tokens must be [R, B-1]")
    for t, n, shp in ((heads, "heads", (R, M, B)), (head_len, "head_len", (R, M)),
                      (anchors, "anchors", (R, C - 1, F)), (bonus_guess, "bonus_guess", (R,)),
                      (segs, "segs", (R * M, 5)), (cu_q, "cu_q", (R + 1,)), (cu_seg, "cu_seg", (R + 1,))):
        if t is None:
            continue
        _need(t, n, torch.int32, len(shp))
        if tuple(t.shape) != shp:
            raise ValueError("%s must be %s" % (n, shp))
    _need(ws, "ws", torch.uint8, 1)
    rc = lib.d3d_build_branches(_ptr(draft_logits), dt, _ptr(draft_tokens), _ptr(bonus_guess), R, B, V, C, F,
                                _ptr(anchors), _ptr(heads), _ptr(head_len), _ptr(segs), _ptr(cu_q), _ptr(cu_seg),
                                _ptr(ws), ws.numel(), _stream(stream))
    _check("d3d_build_branches", rc)


def d3d_accept_probs_workspace_size(R, B, V) -> int:
    return int(lib.d3d_accept_probs_workspace_size(R, B, V))


def d3d_accept_probs(target_logits, draft_logits, temperature: float, accept_prob, ws, survival=None, tau=None,
                     stream=None) -> None:
    """a_j = sum min(P_j, Q_j), survivals S(k) and tau (include/d3d.h); float32 outputs."""
    if target_logits.dtype == torch.bfloat16:
        dt = D3D_DTYPE_BF16
    elif target_logits.dtype == torch.float32:
        dt = D3D_DTYPE_F32
    else:
        raise TypeError("logits must be float32 or bfloat16")
    _need(target_logits, "target_logits", target_logits.dtype, 3)
    _need(draft_logits, "draft_logits", target_logits.dtype, 3)
    R, B, V = target_logits.shape
    if tuple(draft_logits.shape) != (R, B - 1, V):
        raise ValueError("draft_logits must be [R, B-1, V]")
    for t, n, shp in ((accept_prob, "accept_prob", (R, B - 1)), (survival, "survival", (R, B - 1)),
                      (tau, "tau", (R,))):
        if t is None:
            continue
        _need(t, n, torch.float32, len(shp))
        if tuple(t.shape) != shp:
            raise ValueError("%s must be %s" % (n, shp))
    _need(ws, "ws", torch.uint8, 1)
    rc = lib.d3d_accept_probs(_ptr(target_logits), _ptr(draft_logits), dt, R, B, V, float(temperature),
                              _ptr(accept_prob), _ptr(survival), _ptr(tau), _ptr(ws), ws.numel(), _stream(stream))
    _check("d3d_accept_probs", rc)


class AttnCall(ctypes.Structure):
    """d3d_attn_call_t (include/d3d.h)."""
    _fields_ = [(n, _P) for n in ("q", "k_prefix", "v_prefix", "k_packed", "v_packed", "segs", "cu_prefix", "cu_q",
                                  "cu_seg")] + \
               [(n, _I) for n in ("R", "Hq", "Hkv", "d", "max_q", "max_prefix", "total_q", "total_prefix",
                                  "total_segs")] + \
               [("scale", _F), ("out", _P), ("ws", _P), ("ws_bytes", _Z)]


class VerifyCall(ctypes.Structure):
    """d3d_verify_call_t (include/d3d.h)."""
    _fields_ = [("target_logits", _P), ("draft_logits", _P), ("logits_dtype", _I), ("draft_tokens", _P),
                ("u_accept", _P), ("u_sample", _P), ("R", _I), ("B", _I), ("V", _I), ("temperature", _F),
                ("accept_len", _P), ("out_tokens", _P), ("num_tokens", _P), ("alpha", _P), ("p_draft", _P),
                ("q_draft", _P), ("awl_weight", _P), ("heads", _P), ("head_len", _P), ("M", _I), ("branch", _P),
                ("ws", _P), ("ws_bytes", _Z)]


def d3d_async_round(attn: dict, verify: dict, stream=None) -> None:
    """The drafting attention and the verification of one round in one launch.

    ``attn`` holds d3d_packed_draft_attn's keyword arguments (q, k_prefix, ...,
    out, ws) and ``verify`` d3d_spec_verify's (target_logits, ..., ws, and the
    optional alpha/p_draft/q_draft/awl_weight/heads/head_len/branch)."""
    a = _attn_args(**attn)
    vkw = dict(alpha=None, p_draft=None, q_draft=None, heads=None, head_len=None, branch=None)
    vkw.update(verify)
    v = _verify_args(**vkw)
    ac, vc = AttnCall(*a), VerifyCall(*v)
    rc = lib.d3d_async_round(ctypes.byref(ac), ctypes.byref(vc), _stream(stream))
    _check("d3d_async_round", rc)


def d3d_spec_verify_noalloc(target_logits, draft_logits, draft_tokens, u_accept, u_sample, temperature: float,
                            accept_len, out_tokens, num_tokens, alpha=None, p_draft=None, q_draft=None,
                            stream=None) -> None:
    """d3d_spec_verify without a workspace: scratch lives inside the library (see include/d3d.h).
    Every tensor is checked for dtype, device, contiguity and shape exactly as
    d3d_spec_verify checks it."""
    args = _verify_args(target_logits, draft_logits, draft_tokens, u_accept, u_sample, temperature, accept_len,
                        out_tokens, num_tokens, None, alpha, p_draft, q_draft, None, None, None)
    rc = lib.d3d_spec_verify_noalloc(*args[:16], _stream(stream))
    _check("d3d_spec_verify_noalloc", rc)


def d3d_branch_match(verified, verified_len, heads, head_len, branch, stream=None) -> None:
    """Branch cache-hit match; int32 tensors as in include/d3d.h."""
    _need(verified, "verified", torch.int32, 2)
    _need(verified_len, "verified_len", torch.int32, 1)
    _need(heads, "heads", torch.int32, 3)
    _need(head_len, "head_len", torch.int32, 2)
    _need(branch, "branch", torch.int32, 1)
    R, M, B = heads.shape
    if verified.shape != (R, B) or verified_len.shape != (R,) or head_len.shape != (R, M) or branch.shape != (R,):
        raise ValueError("inconsistent match shapes")
    rc = lib.d3d_branch_match(_ptr(verified), _ptr(verified_len), _ptr(heads), _ptr(head_len), R, M, B,
                              _ptr(branch), _stream(stream))
    _check("d3d_branch_match", rc)
