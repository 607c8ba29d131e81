"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds input *synthesis* only: shapes, random draws, bf16 encoding
of the draws, and the structural layout of the packed drafting sequence
(which segment is which branch).  It computes none of the method's arithmetic
(no attention, no acceptance ratio, no residual, no match).  The one piece of
sampling here is the drafter's own draw of the draft tokens y_j ~ Q_j, which
happens upstream of the verified path (the drafter proposes, the verifier
checks); it is needed so that the synthetic draft tokens have the statistics
the losslessness argument assumes.

Draw order.  Every tensor has its own stream, ``np.random.default_rng
(SeedSequence([seed, STREAM_ID]))``, so adding or resizing one tensor never
changes another.  Stream ids are the ``_S_*`` constants below.

Workload shapes follow the pages: block size B = 16, C = 12 rejection
positions, F = 2 alternative anchors, N_async = B[(C-1)F+2] = 384
(D3D, "Method steps", step 4), DScout's bs = 32 block (DScout, "Core method"),
and 16 concurrent requests (D3D, "Experimental results").  Head shapes
(32q/8kv and 64q/8kv heads, head_dim 128) and the vocabulary 151936 are
Qwen3-class shapes of the target/drafter models named on the pages.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_bits", "bf16_to_f32", "uniform24", "async_segments", "block_segments", "verify_segments",
    "train_segments", "layout_segments", "prefix_lengths",
    "attn_inputs", "verify_inputs", "branch_heads", "match_inputs", "CONFIGS",
    "SEG_CAUSAL", "SEG_BIDIR", "DT_F32", "DT_BF16",
]

# Segment modes (packed drafting layout) and logit dtypes, as plain integers.
SEG_CAUSAL = 0
SEG_BIDIR = 1
DT_F32 = 0
DT_BF16 = 1

# Stream ids (one per drawn tensor).
_S_Q, _S_KP, _S_VP, _S_KN, _S_VN = 1, 2, 3, 4, 5
_S_LPREF = 6
_S_XT, _S_XD, _S_YU, _S_UACC = 10, 11, 12, 13
_S_ANCH, _S_MATCH = 20, 21
_S_TRAIN = 22


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), int(stream)]))


def bf16_bits(x) -> np.ndarray:
    """Encode float32 values as bf16 bit patterns (uint16), round to nearest even.

    NaN/Inf are not produced by the generators; finite values only.
    """
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) >> 16
    return u.astype(np.uint16)


def bf16_to_f32(b) -> np.ndarray:
    """Decode bf16 bit patterns (uint16) to float32 (exact)."""
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32)


def uniform24(rng: np.random.Generator, shape) -> np.ndarray:
    """Uniforms u = k * 2^-24, k uniform in [0, 2^24): float32 in [0, 1), exact."""
    k = rng.integers(0, 1 << 24, size=shape, dtype=np.int64)
    return (k.astype(np.float64) * (2.0 ** -24)).astype(np.float32)


# ----------------------------------------------------------------------------
# Packed drafting layout (structure only).
# A segment row is (q_start, len, mode, parent, parent_len), request-local.
# ----------------------------------------------------------------------------
def block_segments(B: int) -> np.ndarray:
    """One synchronous draft block (anchor + B-1 masks), bidirectional, no branches."""
    return np.array([[0, B, SEG_BIDIR, -1, 0]], dtype=np.int32)


def verify_segments(B: int) -> np.ndarray:
    """The target's verification pass over one drafted block: B tokens, causal
    (each position sees the prefix and the earlier tokens of the block)."""
    return np.array([[0, B, SEG_CAUSAL, -1, 0]], dtype=np.int32)


def train_segments(T: int, n_anchor: int, B: int, seed: int = 0) -> np.ndarray:
    """Training-time packed layout (forward only): segment 0 is the clean
    response of T tokens, causal; then one bidirectional block of B tokens
    (anchor + B-1 masks) per anchor, which sees the response tokens before its
    anchor (parent 0, parent_len = the anchor's position).  Anchor positions
    are distinct, drawn uniformly from [1, T) and sorted (input synthesis)."""
    pos = np.sort(_rng(seed, _S_TRAIN).choice(np.arange(1, T), size=n_anchor, replace=False))
    rows = [[0, T, SEG_CAUSAL, -1, 0]]
    q = T
    for p in pos.tolist():
        rows.append([q, B, SEG_BIDIR, 0, int(p)])
        q += B
    return np.array(rows, dtype=np.int32)


def async_segments(B: int, C: int, F: int) -> np.ndarray:
    """Layout of D3D's asynchronous packed pass (D3D, "Method steps", step 4).

    Segment 0 is the block under verification [c_0 .. c_{B-1}], encoded
    causally; its keys are the hypothesised accepted tokens the branches see.
    Then, for rejection position r+1 (r = 0 .. C-2 accepted drafts) and
    alternative anchor f = 0 .. F-1, one bidirectional branch block that sees
    c_0 .. c_r of segment 0 (parent_len = r + 1).  Last, the all-accept block,
    which sees the whole current block (parent_len = B).
    """
    rows = [[0, B, SEG_CAUSAL, -1, 0]]
    q = B
    for r in range(C - 1):
        for _f in range(F):
            rows.append([q, B, SEG_BIDIR, 0, r + 1])
            q += B
    rows.append([q, B, SEG_BIDIR, 0, B])
    return np.array(rows, dtype=np.int32)


CONFIGS = {
    # name: shapes of one workload (see the module docstring for the sources)
    "tiny": dict(R=1, L=256, Hq=2, Hkv=1, d=64, B=16, layout="block",
                 V=1024, logits=DT_F32, sigma=0.5),
    "async8b": dict(R=1, L=2048, Hq=32, Hkv=8, d=128, B=16, C=12, F=2, layout="async",
                    V=151936, logits=DT_BF16, sigma=0.5),
    "long_block": dict(R=1, L=8192, Hq=32, Hkv=8, d=128, B=32, layout="block",
                       V=151936, logits=DT_BF16, sigma=0.5),
    "serve32b": dict(R=16, L=(1024, 4096), Hq=64, Hkv=8, d=128, B=16, C=12, F=2,
                     layout="async", V=151936, logits=DT_BF16, sigma=0.5),
    "sweep": dict(R=1, L=32768, Hq=32, Hkv=8, d=128, B=16, C=12, F=2, layout="async",
                  V=151936, logits=DT_BF16, sigma=0.5),
    # the target's verification attention: one causal block over a long KV
    "target_verify": dict(R=1, L=8192, Hq=32, Hkv=8, d=128, B=16, layout="verify",
                          V=151936, logits=DT_BF16, sigma=0.5),
    # training-time packed pass: a 2048-token response with 128 anchor blocks
    "train_mask": dict(R=1, L=512, Hq=32, Hkv=8, d=128, B=16, T=2048, anchors=128, layout="train",
                       V=151936, logits=DT_BF16, sigma=0.5),
}


def prefix_lengths(R: int, L, seed: int) -> np.ndarray:
    """Per-request prefix lengths: ``L`` for every request, or uniform in the
    inclusive range ``L = (lo, hi)`` (seeded)."""
    if isinstance(L, tuple):
        lo, hi = L
        return _rng(seed, _S_LPREF).integers(lo, hi + 1, size=R).astype(np.int32)
    return np.full(R, int(L), dtype=np.int32)


def layout_segments(layout: str, B: int, C: int = 12, F: int = 2, T: int = 2048, anchors: int = 128,
                    seed: int = 0) -> np.ndarray:
    """Segment rows of one request for a named layout."""
    if layout == "block":
        return block_segments(B)
    if layout == "verify":
        return verify_segments(B)
    if layout == "train":
        return train_segments(T, anchors, B, seed)
    return async_segments(B, C, F)


def attn_inputs(R=1, L=256, Hq=2, Hkv=1, d=64, B=16, C=12, F=2, layout="block",
                seed=0, k_scale=1.0, segs=None, T=2048, anchors=128, **_unused) -> dict:
    """Inputs of one packed drafting attention call.

    Q, K, V ~ N(0, 1) rounded to bf16 (K multiplied by ``k_scale`` first: the
    adversarial variant uses 4 for peaky softmax).  ``L`` is an int (same
    prefix for every request) or a (lo, hi) range drawn per request.
    ``segs`` overrides the per-request segment table.
    """
    if segs is None:  # the layout is fixed by its shapes; seed varies the tensors only
        segs = layout_segments(layout, B, C, F, T, anchors)
    segs = np.asarray(segs, dtype=np.int32).reshape(-1, 5)
    n_q = int(segs[-1, 0] + segs[-1, 1]) if len(segs) else 0
    Ls = prefix_lengths(R, L, seed)
    cu_prefix = np.zeros(R + 1, np.int32)
    cu_prefix[1:] = np.cumsum(Ls)
    cu_q = (np.arange(R + 1) * n_q).astype(np.int32)
    cu_seg = (np.arange(R + 1) * len(segs)).astype(np.int32)
    all_segs = np.tile(segs, (R, 1)).astype(np.int32)
    NT, LT = int(cu_q[-1]), int(cu_prefix[-1])
    q = _rng(seed, _S_Q).standard_normal((NT, Hq, d), dtype=np.float32)
    kp = _rng(seed, _S_KP).standard_normal((LT, Hkv, d), dtype=np.float32) * k_scale
    vp = _rng(seed, _S_VP).standard_normal((LT, Hkv, d), dtype=np.float32)
    kn = _rng(seed, _S_KN).standard_normal((NT, Hkv, d), dtype=np.float32) * k_scale
    vn = _rng(seed, _S_VN).standard_normal((NT, Hkv, d), dtype=np.float32)
    return dict(q=bf16_bits(q), kp=bf16_bits(kp), vp=bf16_bits(vp), kn=bf16_bits(kn),
                vn=bf16_bits(vn), segs=all_segs, cu_prefix=cu_prefix, cu_q=cu_q,
                cu_seg=cu_seg, R=R, Hq=Hq, Hkv=Hkv, d=d, scale=float(1.0 / np.sqrt(d)),
                max_q=n_q, max_prefix=int(Ls.max()) if R else 0)


def _draw_from(rows64: np.ndarray, u: np.ndarray) -> np.ndarray:
    """The drafter's own token draw: y ~ softmax(row) by inverse CDF (input synthesis)."""
    m = rows64.max(axis=-1, keepdims=True)
    w = np.exp(rows64 - m)
    c = np.cumsum(w, axis=-1)
    tgt = u[..., None].astype(np.float64) * c[..., -1:]
    y = (c <= tgt).sum(axis=-1)
    return np.minimum(y, rows64.shape[-1] - 1).astype(np.int32)


def verify_inputs(R=1, B=16, V=1024, logits=DT_F32, sigma=0.5, seed=0, x_std=3.0,
                  temperature=1.0, **_unused) -> dict:
    """Inputs of one batched verification call.

    Target logits x ~ N(0, x_std^2) for B positions; draft logits
    z = x[:B-1] + N(0, sigma^2); both stored in ``logits`` dtype (f32 or bf16
    bits).  Draft tokens y_j are drawn by the drafter from softmax(z_j / T)
    (over the stored, rounded z) on their own uniform stream.  Per request,
    B-1 acceptance uniforms and 1 sample uniform, all k * 2^-24.
    """
    x = _rng(seed, _S_XT).standard_normal((R, B, V), dtype=np.float32) * np.float32(x_std)
    z = x[:, : B - 1, :] + _rng(seed, _S_XD).standard_normal((R, B - 1, V), dtype=np.float32) * np.float32(sigma)
    if logits == DT_BF16:
        xs, zs = bf16_bits(x), bf16_bits(z)
        z_val = bf16_to_f32(zs)
    else:
        xs, zs = x.astype(np.float32), z.astype(np.float32)
        z_val = zs
    y = _draw_from(z_val.astype(np.float64) / float(temperature),
                   uniform24(_rng(seed, _S_YU), (R, B - 1)))
    u = uniform24(_rng(seed, _S_UACC), (R, B))
    return dict(target=xs, draft=zs, dtype=logits, y=y, u_accept=np.ascontiguousarray(u[:, : B - 1]),
                u_sample=np.ascontiguousarray(u[:, B - 1]), R=R, B=B, V=V, temperature=float(temperature))


def branch_heads(y: np.ndarray, B: int, C: int, F: int, V: int, seed=0) -> dict:
    """Heads of the pre-drafted branches, indexed like ``async_segments`` (M = (C-1)F + 2).

    Head 0 is the current block (length 0: it never matches).  Branch
    (r, f) hypothesises r accepted drafts and the f-th alternative anchor
    at position r+1: head = [y_1 .. y_r, anchor], length r + 1.  The
    all-accept head is [y_1 .. y_{B-1}, bonus guess], length B.  Anchors are
    distinct tokens different from y_{r+1}; positions past a head's length
    hold junk so that a compare that runs too far is caught.
    """
    y = np.asarray(y, dtype=np.int32).reshape(-1, B - 1)
    R = y.shape[0]
    M = (C - 1) * F + 2
    rng = _rng(seed, _S_ANCH)
    heads = rng.integers(0, V, size=(R, M, B)).astype(np.int32)
    head_len = np.zeros((R, M), np.int32)
    for r_ in range(R):
        k = 1
        for r in range(C - 1):
            banned = {int(y[r_, r])}
            for _f in range(F):
                a = int(rng.integers(0, V))
                while a in banned:
                    a = int(rng.integers(0, V))
                banned.add(a)
                heads[r_, k, :r] = y[r_, :r]
                heads[r_, k, r] = a
                head_len[r_, k] = r + 1
                k += 1
        heads[r_, k, : B - 1] = y[r_]
        heads[r_, k, B - 1] = int(rng.integers(0, V))
        head_len[r_, k] = B
    return dict(heads=heads, head_len=head_len, M=M)


def match_inputs(R=64, B=16, C=12, F=2, V=151936, seed=0, hit_rate=0.713, dup_rate=0.1) -> dict:
    """Verified prefixes and branch heads with planted hits, misses and duplicate heads.

    A verified prefix [y_1 .. y_a, t] has a drawn a in [0, B-1]; t is
    planted from a branch whose head has that length with probability
    ``hit_rate`` (the 71.3% hit rate the D3D pages report at C=12, F=2 is
    the default), else drawn at random.  With probability ``dup_rate`` a
    later head is overwritten with a copy of an earlier one, so the
    lowest-index rule is exercised.  Lengths are ragged by construction.
    """
    rng = _rng(seed, _S_MATCH)
    y = rng.integers(0, V, size=(R, B - 1)).astype(np.int32)
    hb = branch_heads(y, B, C, F, V, seed)
    heads, head_len, M = hb["heads"], hb["head_len"], hb["M"]
    verified = rng.integers(0, V, size=(R, B)).astype(np.int32)
    vlen = np.zeros(R, np.int32)
    for r_ in range(R):
        a = int(rng.integers(0, B))
        verified[r_, :a] = y[r_, :a]
        cands = [k for k in range(M) if head_len[r_, k] == a + 1]
        if cands and rng.random() < hit_rate:
            k = cands[int(rng.integers(0, len(cands)))]
            verified[r_, a] = heads[r_, k, a]
        vlen[r_] = a + 1
        if rng.random() < dup_rate and M >= 3:
            src = int(rng.integers(1, M - 1))
            dst = int(rng.integers(src + 1, M))
            heads[r_, dst] = heads[r_, src]
            head_len[r_, dst] = head_len[r_, src]
    return dict(verified=verified, verified_len=vlen, heads=heads, head_len=head_len,
                R=R, M=M, B=B)
