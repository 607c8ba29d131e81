#!/usr/bin/env python3
"""Benchmark of the diffusion-drafted speculative decoding hot path on GB300.

One step = one pass of the whole path over one round of synthetic input:
packed drafting attention (one drafter layer, all heads) over the async
packed sequence, batched speculative-sampling verification over the
vocabulary, and the branch cache-hit match of the verified tokens.  The
default workload is D3D's asynchronous packed pass at 8B-class shapes:
1 request, prefix 2048, 32 query / 8 KV heads, head_dim 128, B=16, C=12,
F=2 (N_async = 384 packed query tokens), verification of 16 positions over a
151936-entry vocabulary, and a match against 24 branch heads.  Within a
round the packed drafting pass and the verification are independent (the
drafter prepares the successor blocks while the current block is verified),
so they run concurrently: the verification on the SMs the attention leaves
and the attention as its programmatic dependent on the same stream
(``--round fused``: one cooperative launch holding both); the branch match
runs inside the verification's last phase (``parts.match_us`` times the
stand-alone match entry point).

Timing: inputs resident in HBM; steps rotate over input sets whose total
size exceeds twice the L2 cache, so no step finds its inputs in L2; each
step is captured once in a CUDA graph and the K timed steps are graph
replays, bracketed by a barrier and synchronisation, timed with CUDA events
on the launching stream, max over ranks.  ``value`` is packed query tokens
per second of whole steps, over all ranks (weak scaling: each rank runs its
own request).  Per-part device times come from separate graph-replayed
loops of each part alone over the same rotation.

``--impl reference`` times the plain CPU oracle on this host instead (a
bounded sample per step, scaled to the same unit).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "packed-draft query tokens/s + verified positions/s; % HBM/tensor roofline"
UNIT = "packed-draft query tokens/s"
# our kernel launches per step: one fused round launch, or the attention and
# the verification (with the branch match fused into its last phase)
LAUNCHES = {"fused": 1, "attention-first": 2, "verify-first": 2}
CSRC = os.path.join(ROOT, "diffusion_drafted_speculative_gb300", "csrc")
# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one
# ncu capture of this bench's workload, keyed by a hash of the sources the
# kernel is built from: reported only while those sources are unchanged.
NCU_TRAFFIC = {
    ("async8b", "attn"): {"sources": ("attn.cu", "attn_common.cuh", "sm100_ptx.cuh", "d3d_common.cuh",
                                      "verify_body.cuh"),
                          "sha": "f4e3d13cd7896800", "bytes": 13178368},
    ("async8b", "verify"): {"sources": ("verify.cu", "verify_slice.cuh", "verify_body.cuh", "sm100_ptx.cuh",
                                        "d3d_common.cuh"),
                            "sha": "ce99d02e41d2ef67", "bytes": 9490176},
    ("async8b", "greedy"): {"sources": ("verify.cu", "greedy_body.cuh", "verify_body.cuh", "verify_slice.cuh",
                                        "sm100_ptx.cuh", "d3d_common.cuh"),
                            "sha": "81498f57f4483e7e", "bytes": 4903936},
    ("async8b", "branches"): {"sources": ("branches.cu", "sm100_ptx.cuh", "d3d_common.cuh"),
                              "sha": "1db77ce822f14171", "bytes": 3425536},
    ("async8b", "accept"): {"sources": ("accept.cu", "sm100_ptx.cuh", "d3d_common.cuh"),
                            "sha": "9d59b7469b95e2b9", "bytes": 9162112},
}


def sources_sha(names) -> str:
    import hashlib

    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(CSRC, n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def hbm_part(nbytes: float, ms: float, peak: float, traffic) -> dict:
    """HBM roofline entry of a part timed alone: algorithmic bytes over its time."""
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"achieved": round(gbs, 1), "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
            "bytes": nbytes, "traffic": traffic}


def ncu_traffic(wl_name: str, part: str):
    t = NCU_TRAFFIC.get((wl_name, part))
    if t is None or sources_sha(t["sources"]) != t["sha"]:
        return None
    return t["bytes"]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 20000 for this library, 5 for the reference arm)")
    ap.add_argument("--warmup", type=int, default=None, help="warm-up steps (default: 200, reference arm 3)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="async8b", choices=["async8b", "long_block", "serve32b"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--round-attn-ctas", type=int, default=96,
                    help="SMs the attention may hold in the split round (the verification takes the rest; "
                         "0: the whole device)")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the long-block, serving-batch and C/F-sweep measurements")
    ap.add_argument("--no-layout-parts", action="store_true",
                    help="skip timing the attention on the target-verify and training layouts")
    ap.add_argument("--round", choices=["attention-first", "verify-first", "fused"], default="attention-first",
                    help="attention-first: the attention (set up while the round before ends), then the "
                         "verification as its programmatic dependent; verify-first: the verification, then "
                         "the attention as its programmatic dependent; "
                         "fused: both in one cooperative launch (d3d_async_round)")
    return ap.parse_args()


# ----------------------------------------------------------------------------
# Workload description (shapes and algorithmic work; no method arithmetic).
# ----------------------------------------------------------------------------
def workload(name: str) -> dict:
    cfg = dict(W.CONFIGS[name])
    segs = W.layout_segments(cfg["layout"], cfg["B"], cfg.get("C", 12), cfg.get("F", 2), cfg.get("T", 2048),
                             cfg.get("anchors", 128))
    n_q = int(segs[:, 1].sum())
    # visible packed keys per query token, from the segment rows
    vis_packed = 0
    for q0, ln, mode, par, plen in segs.tolist():
        own = ln * ln if mode == W.SEG_BIDIR else ln * (ln + 1) // 2
        vis_packed += own + ln * plen
    R = cfg["R"]
    L_mean = float(np.mean(cfg["L"])) if isinstance(cfg["L"], tuple) else float(cfg["L"])
    Hq, Hkv, d, B, V = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["B"], cfg["V"]
    flops = 4.0 * d * Hq * R * (n_q * L_mean + vis_packed)
    attn_bytes = 2.0 * R * (2 * L_mean * Hkv * d + 2 * n_q * Hq * d + 2 * n_q * Hkv * d)
    verify_bytes = 2.0 * R * ((2 * B - 1) * V + 2 * V)
    greedy_bytes = 2.0 * R * B * V  # greedy verification reads the target logits only
    # branch construction reads draft rows 0..C-2; the acceptance
    # probabilities read target and draft rows 0..B-2 (bf16)
    branch_bytes = 2.0 * R * max(cfg.get("C", 1) - 1, 0) * V
    accept_bytes = 2.0 * R * 2 * (B - 1) * V
    return dict(cfg=cfg, segs=segs, n_q=n_q, R=R, flops=flops, attn_bytes=attn_bytes, verify_bytes=verify_bytes,
                greedy_bytes=greedy_bytes, branch_bytes=branch_bytes, accept_bytes=accept_bytes, positions=R * B,
                vis_packed=vis_packed)


def workload_label(name: str) -> str:
    """The workload as both arms name it in config.workload."""
    wl = workload(name)
    cfg = wl["cfg"]
    return "%s: R=%d, prefix %s, %d/%d heads, d=%d, B=%d%s, N_async=%d, V=%d, M=%d heads" % (
        name, cfg["R"], cfg["L"], cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["B"],
        (", C=%d, F=%d" % (cfg["C"], cfg["F"])) if cfg["layout"] == "async" else " block",
        wl["n_q"], cfg["V"], (cfg.get("C", 1) - 1) * cfg.get("F", 1) + 2)


# ----------------------------------------------------------------------------
# Rank logic (weak scaling: every rank runs its own requests, no data exchange).
# ----------------------------------------------------------------------------
def rank_seed(rank: int, set_index: int) -> int:
    """Seed of input set `set_index` on `rank`: ranks never share a request."""
    return 1000 * rank + set_index


def reduce_max(x: float, dist, device) -> float:
    """Max over ranks of a host float (the slowest rank sets the job time)."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, ms_per_step_max: float) -> float:
    """Units all ranks processed per second, timed by the slowest rank."""
    return world * units_per_rank / (ms_per_step_max * 1e-3)


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    source="of measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="of fallback")


# ----------------------------------------------------------------------------
# Clock sampling during the timed region.
# ----------------------------------------------------------------------------
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.proc = None
        cmd = ["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits", "-lms", "100"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out = self.proc.communicate(timeout=5)[0]
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out = self.proc.communicate()[0]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# Our arm.
# ----------------------------------------------------------------------------
def run_ours(args, rank: int, world: int, local_rank: int):
    import torch

    import __graft_entry__

    __graft_entry__._build_module().build()
    import diffusion_drafted_speculative_gb300 as d3d

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    wl = workload(args.workload)
    cfg = wl["cfg"]
    R, B, V, Hq, Hkv, d = cfg["R"], cfg["B"], cfg["V"], cfg["Hq"], cfg["Hkv"], cfg["d"]
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 << 20) or (126 << 20)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)

    def host_set(seed):
        a = W.attn_inputs(**cfg, seed=seed)
        v = W.verify_inputs(**cfg, seed=seed)
        hb = W.branch_heads(v["y"], B, cfg.get("C", 1), cfg.get("F", 1), V, seed=seed) if cfg["layout"] == "async" \
            else W.branch_heads(v["y"], B, 1, 1, V, seed=seed)
        ins = dict(q=bf(a["q"]), kp=bf(a["kp"]), vp=bf(a["vp"]), kn=bf(a["kn"]), vn=bf(a["vn"]),
                   segs=torch.from_numpy(a["segs"]), cu_prefix=torch.from_numpy(a["cu_prefix"]),
                   cu_q=torch.from_numpy(a["cu_q"]), cu_seg=torch.from_numpy(a["cu_seg"]),
                   target=bf(v["target"]), draft=bf(v["draft"]), y=torch.from_numpy(v["y"]),
                   u_accept=torch.from_numpy(v["u_accept"]), u_sample=torch.from_numpy(v["u_sample"]),
                   heads=torch.from_numpy(hb["heads"]), head_len=torch.from_numpy(hb["head_len"]))
        return ins, a["max_q"], a["max_prefix"], a["scale"]

    def outputs(NT):
        return dict(out=torch.empty(NT, Hq, d, dtype=torch.bfloat16, device=dev),
                    accept_len=torch.empty(R, dtype=torch.int32, device=dev),
                    out_tokens=torch.empty(R, B, dtype=torch.int32, device=dev),
                    num_tokens=torch.empty(R, dtype=torch.int32, device=dev),
                    branch=torch.empty(R, dtype=torch.int32, device=dev))

    first, max_q, max_prefix, scale = host_set(rank_seed(rank, 0))
    set_bytes = sum(t.numel() * t.element_size() for t in first.values()) + first["q"].numel() * 2
    n_sets = max(2, math.ceil(2.2 * l2 / set_bytes))
    sets = []
    for s in range(n_sets):
        hs = first if s == 0 else host_set(rank_seed(rank, s))[0]
        dset = {k: t.to(dev) for k, t in hs.items()}
        dset.update(outputs(hs["q"].shape[0]))
        sets.append(dset)
    ws_a = d3d.new_workspace(d3d.d3d_packed_draft_attn_workspace_size(R, Hq, Hkv, d, max_q, max_prefix), dev)
    ws_v = d3d.new_workspace(d3d.d3d_spec_verify_workspace_size(R, B, V), dev)
    # the attention holds one SM per CTA; in the round it gets at most
    # --round-attn-ctas of them and the verification beside it takes the SMs
    # it leaves (0: the attention fills the GPU, no limit).  Timed alone, the
    # attention uses the whole device.
    round_budget = max(0, args.round_attn_ctas)
    attn_ctas = d3d.d3d_packed_draft_attn_ctas(R, Hq, Hkv, d, max_q, max_prefix, round_budget)
    side_sms = props.multi_processor_count - attn_ctas
    verify_sms = side_sms if 0 < attn_ctas and side_sms > 0 else 0

    def attn(s, after_independent=False, max_ctas=0, after_dependent=False):
        d3d.d3d_packed_draft_attn(s["q"], s["kp"], s["vp"], s["kn"], s["vn"], s["segs"], s["cu_prefix"], s["cu_q"],
                                  s["cu_seg"], max_q, max_prefix, scale, s["out"], ws_a,
                                  after_independent=after_independent, max_ctas=max_ctas,
                                  after_dependent=after_dependent)

    def verify(s, sm_limit=0, fused_match=False, after_independent=False):
        extra = dict(heads=s["heads"], head_len=s["head_len"], branch=s["branch"]) if fused_match else {}
        d3d.d3d_spec_verify(s["target"], s["draft"], s["y"], s["u_accept"], s["u_sample"], 1.0, s["accept_len"],
                            s["out_tokens"], s["num_tokens"], ws_v, sm_limit=sm_limit,
                            after_independent=after_independent, **extra)

    def greedy(s):  # temperature 0: argmax verification of the same rows
        d3d.d3d_spec_verify(s["target"], None, s["y"], None, None, 0.0, s["accept_len"], s["out_tokens"],
                            s["num_tokens"], ws_v)

    def match(s):
        d3d.d3d_branch_match(s["out_tokens"], s["num_tokens"], s["heads"], s["head_len"], s["branch"])

    # branch construction for the next round's packed pass (async layouts):
    # anchors, heads and segment rows from this round's draft rows
    bC, bF = (cfg["C"], cfg["F"]) if cfg["layout"] == "async" else (1, 0)
    bM = (bC - 1) * bF + 2
    ws_b = d3d.new_workspace(d3d.d3d_build_branches_workspace_size(R, B, V, bC, bF), dev)
    b_out = dict(anchors=torch.empty((R, bC - 1, bF), dtype=torch.int32, device=dev),
                 heads=torch.empty((R, bM, B), dtype=torch.int32, device=dev),
                 head_len=torch.empty((R, bM), dtype=torch.int32, device=dev),
                 segs=torch.empty((R * bM, 5), dtype=torch.int32, device=dev),
                 cu_q=torch.empty(R + 1, dtype=torch.int32, device=dev),
                 cu_seg=torch.empty(R + 1, dtype=torch.int32, device=dev))

    ws_p = d3d.new_workspace(d3d.d3d_accept_probs_workspace_size(R, B, V), dev)
    p_out = dict(a=torch.empty((R, B - 1), device=dev), sv=torch.empty((R, B - 1), device=dev),
                 tau=torch.empty(R, device=dev))

    def accept_probs(s):  # a_j = sum min(P_j, Q_j), survivals and tau of the same rows
        d3d.d3d_accept_probs(s["target"], s["draft"], 1.0, p_out["a"], ws_p, survival=p_out["sv"], tau=p_out["tau"])

    def branches(s):
        d3d.d3d_build_branches(s["draft"], s["y"], bC, bF, b_out["heads"], b_out["head_len"], ws_b,
                               anchors=b_out["anchors"], bonus_guess=None, segs=b_out["segs"], cu_q=b_out["cu_q"],
                               cu_seg=b_out["cu_seg"])

    stream = torch.cuda.Stream(device=dev)

    def round_calls(s):
        a = dict(q=s["q"], k_prefix=s["kp"], v_prefix=s["vp"], k_packed=s["kn"], v_packed=s["vn"], segs=s["segs"],
                 cu_prefix=s["cu_prefix"], cu_q=s["cu_q"], cu_seg=s["cu_seg"], max_q=max_q, max_prefix=max_prefix,
                 scale=scale, out=s["out"], ws=ws_a)
        v = dict(target_logits=s["target"], draft_logits=s["draft"], draft_tokens=s["y"], u_accept=s["u_accept"],
                 u_sample=s["u_sample"], temperature=1.0, accept_len=s["accept_len"], out_tokens=s["out_tokens"],
                 num_tokens=s["num_tokens"], ws=ws_v, heads=s["heads"], head_len=s["head_len"], branch=s["branch"])
        return a, v

    # one launch per round (on request) when the attention leaves SMs and
    # needs no key splits
    fused_round = args.round == "fused" and verify_sms > 0
    if fused_round:
        try:
            d3d.d3d_async_round(*round_calls(sets[0]))
            torch.cuda.synchronize()
        except d3d.D3DError as e:
            if e.rc != d3d.D3D_ERR_UNSUPPORTED:
                raise
            fused_round = False

    def step(s):
        # the asynchronous round: the packed drafting pass and the verification
        # of the current block are independent and run concurrently: the
        # attention, launched as a programmatic dependent of the round before
        # (it sets up while that round ends and reads its inputs once it has
        # finished), then the verification on the SMs the attention leaves as
        # the attention's programmatic dependent (--round verify-first: the
        # other way round; --round fused: both in one cooperative launch); the
        # branch match runs inside the verification's last phase (it needs the
        # verified tokens and the round's branch heads only)
        if fused_round:
            d3d.d3d_async_round(*round_calls(s))
        elif args.round == "attention-first":
            attn(s, max_ctas=round_budget, after_dependent=verify_sms > 0)
            verify(s, verify_sms, fused_match=True, after_independent=verify_sms > 0)
        else:
            verify(s, verify_sms, fused_match=True)
            attn(s, after_independent=verify_sms > 0, max_ctas=round_budget)

    torch.cuda.synchronize()

    def graphs(fn, n):
        """Graphs that together run fn over exactly n consecutive rotation steps."""
        full, tail = divmod(n, n_sets)
        out = []
        for count, reps in ((n_sets, full), (tail, 1)):
            if count == 0 or reps == 0:
                continue
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(count):
                    fn(sets[i])
            out.append((g, reps))
        return out

    def replay(gs):
        for g, reps in gs:
            for _ in range(reps):
                g.replay()

    def hold():
        # keep the device busy (about 0.1 ms) while the host enqueues the
        # start event and the graphs behind it: the timed region then starts
        # with the first step, not with the host's first graph launch
        torch.cuda._sleep(200000)

    def timed(fn, n):
        gs = graphs(fn, n)
        replay(gs)  # untimed pass of the same graphs
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            hold()
            e0.record(stream)
            replay(gs)
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    # eager warm-up (validates every call), then graph warm-up of W steps
    with torch.cuda.stream(stream):
        for i in range(min(args.warmup, n_sets)):
            step(sets[i % n_sets])
    torch.cuda.synchronize()
    for w in (ws_a, ws_v):
        st = d3d.d3d_workspace_status(w)
        if st != 0:
            raise RuntimeError("device status after warm-up: %s" % d3d.d3d_status_string(st))
    g_warm = graphs(step, max(args.warmup, 1))
    g_timed = graphs(step, args.steps)
    replay(g_warm)
    torch.cuda.synchronize()

    uuid = None
    try:
        uuid = "GPU-" + str(props.uuid) if getattr(props, "uuid", None) is not None else None
    except Exception:
        uuid = None
    clocks = Clocks(uuid)
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall = time.perf_counter()
    with torch.cuda.stream(stream):
        hold()
        e0.record(stream)
        replay(g_timed)
        e1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    ms_step = e0.elapsed_time(e1) / args.steps
    ms_step = reduce_max(ms_step, dist, dev)
    for w in (ws_a, ws_v):
        st = d3d.d3d_workspace_status(w)
        if st != 0:
            raise RuntimeError("device status after timed region: %s" % d3d.d3d_status_string(st))

    # per-part device time (each part alone, same rotation, graph replays)
    n_part = max(n_sets, min(args.steps, 2000))
    t_attn = timed(attn, n_part)
    t_verify = timed(verify, n_part)
    t_verify_side = timed(lambda s: verify(s, verify_sms, fused_match=True), n_part)
    t_match = timed(match, n_part)
    t_greedy = timed(greedy, n_part)
    t_branches = timed(branches, n_part)
    t_accept = timed(accept_probs, n_part)

    peaks = load_peaks()
    layout_parts = {} if args.no_layout_parts else {
        n: time_attention(d3d, torch, dev, stream, dict(W.CONFIGS[n]), l2, peaks) for n in ("target_verify", "train_mask")}
    # the other workloads of the comparison contract: attention and verification
    # of the long synchronous block and of the 16-request serving batch, and the
    # attention over the C/F budget sweep at a 32768-token prefix
    other = {} if args.no_other_workloads else other_workloads(d3d, torch, dev, stream, l2, peaks)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(torch, d3d, sets, n_sets, step, dev, stream, args, R, B, dist)
        eager = run_e2e(torch, d3d, sets, n_sets, step, dev, stream, args, R, B, dist, graphs=False)
        e2e["no_graph"] = {k: eager[k] for k in ("value", "ms_per_step", "pipeline")}

    # attention and verification are each timed alone in a short loop: the
    # burst peaks apply (sustained is for a kernel inside a seconds-long step)
    achieved_tf = wl["flops"] / (t_attn * 1e-3) / 1e12
    att_ai = wl["flops"] / wl["attn_bytes"]
    ridge = peaks["bf16"] * 1e12 / (peaks["hbm"] * 1e9)
    if att_ai >= ridge:
        roof = {"bound": "tensor", "achieved": round(achieved_tf, 2), "peak": peaks["bf16"], "unit": "TFLOP/s",
                "frac": round(achieved_tf / peaks["bf16"], 4)}
    else:
        gbs = wl["attn_bytes"] / (t_attn * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm"], "unit": "GB/s",
                "frac": round(gbs / peaks["hbm"], 4)}
    roof.update({"kernel": "packed draft attention", "traffic": ncu_traffic(args.workload, "attn"),
                 "peak_source": peaks["source"] + (" (burst bf16)" if roof["bound"] == "tensor" else " (copy bandwidth)"),
                 "algorithmic": {"flops": wl["flops"], "bytes": wl["attn_bytes"]}})
    verify_gbs = wl["verify_bytes"] / (t_verify * 1e-3) / 1e9
    greedy_gbs = wl["greedy_bytes"] / (t_greedy * 1e-3) / 1e9

    value = whole_job_rate(wl["n_q"] * R, world, ms_step)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded numpy; random bf16 tensors and logits)",
        "config": {"workload": workload_label(args.workload),
                   "l2": "inputs rotate over %d sets (%.0f MB > 2x L2 %.0f MB)" % (
                       n_sets, n_sets * set_bytes / 1e6, l2 / 1e6),
                   "timing": "CUDA graph replays, CUDA events on the launching stream"},
        "verified_positions_per_s": round(world * wl["positions"] / (ms_step * 1e-3), 1),
        "parts": {"attn_us": round(t_attn * 1e3, 3), "verify_us": round(t_verify * 1e3, 3),
                  "attn_ctas": d3d.d3d_packed_draft_attn_ctas(R, Hq, Hkv, d, max_q, max_prefix),
                  "round_attn_ctas": attn_ctas, "verify_side_sms": verify_sms, "round_launch": "fused" if fused_round
                  else args.round,
                  "verify_side_us": round(t_verify_side * 1e3, 3),
                  "verify_launch": {"whole_device_slice_ctas": d3d.d3d_spec_verify_slice_ctas(R, B, V, cfg["logits"], 1.0, 0),
                                    "side_slice_ctas": d3d.d3d_spec_verify_slice_ctas(R, B, V, cfg["logits"], 1.0,
                                                                                      verify_sms),
                                    "rule": "CTAs of the vocabulary-slice launch (0: the chunked launch)"},
                  "match_us": round(t_match * 1e3, 3),
                  "attn_query_tokens_per_s": round(wl["n_q"] * R / (t_attn * 1e-3), 1),
                  "verify_positions_per_s": round(wl["positions"] / (t_verify * 1e-3), 1),
                  "verify_hbm": {"achieved": round(verify_gbs, 1), "peak": peaks["hbm"], "unit": "GB/s",
                                 "frac": round(verify_gbs / peaks["hbm"], 4),
                                 "bytes": wl["verify_bytes"], "traffic": ncu_traffic(args.workload, "verify")},
                  "greedy_verify_us": round(t_greedy * 1e3, 3),
                  "build_branches_us": round(t_branches * 1e3, 3),
                  "accept_probs_us": round(t_accept * 1e3, 3),
                  "attn_layouts": layout_parts,
                  "other_workloads": other,
                  "greedy_hbm": {"achieved": round(greedy_gbs, 1), "peak": peaks["hbm"], "unit": "GB/s",
                                 "frac": round(greedy_gbs / peaks["hbm"], 4), "bytes": wl["greedy_bytes"],
                                 "traffic": ncu_traffic(args.workload, "greedy")},
                  "branches_hbm": hbm_part(wl["branch_bytes"], t_branches, peaks["hbm"],
                                           ncu_traffic(args.workload, "branches")),
                  "accept_hbm": hbm_part(wl["accept_bytes"], t_accept, peaks["hbm"],
                                         ncu_traffic(args.workload, "accept"))},
        "roofline": roof,
        "gpu_launches": args.steps * LAUNCHES["fused" if fused_round else args.round],
        "clocks": clk, "wall_s_timed_region": round(wall, 4),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload)
        line["parity"] = workload_parity(torch, sets, cfg, rank, verify)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def _graph_time(torch, stream, calls, reps_total=48, rounds=4):
    """Mean device time (ms) of one call, from CUDA graphs replaying the calls
    (each a closure over one input set) round-robin, CUDA events on the stream."""
    with torch.cuda.stream(stream):
        for c in calls:
            c()  # eager pass validates the calls
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    reps = max(1, reps_total // len(calls))
    with torch.cuda.graph(g, stream=stream):
        for _ in range(reps):
            for c in calls:
                c()
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(rounds):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (rounds * reps * len(calls))


def attn_roofline(flops, nbytes, us, peaks):
    """Bound (tensor above the ridge, HBM below) and the fraction of it reached."""
    ridge = peaks["bf16"] * 1e12 / (peaks["hbm"] * 1e9)
    tf = flops / (us * 1e-6) / 1e12
    gbs = nbytes / (us * 1e-6) / 1e9
    if flops / nbytes >= ridge:
        return {"bound": "tensor", "tflops": round(tf, 1), "gbs": round(gbs, 1), "frac": round(tf / peaks["bf16"], 4)}
    return {"bound": "hbm", "tflops": round(tf, 1), "gbs": round(gbs, 1), "frac": round(gbs / peaks["hbm"], 4)}


def time_attention(d3d, torch, dev, stream, cfg, l2, peaks, seed=7000, segs=None):
    """Device time of d3d_packed_draft_attn on one workload shape.  Input sets
    (seeded normal bf16 tensors drawn on the device, the layout's segment
    table) rotate until they exceed 2.2x L2.  Returns time, throughput and
    roofline fraction."""
    R, Hq, Hkv, d = cfg["R"], cfg["Hq"], cfg["Hkv"], cfg["d"]
    if segs is None:
        segs = W.layout_segments(cfg["layout"], cfg["B"], cfg.get("C", 12), cfg.get("F", 2), cfg.get("T", 2048),
                                 cfg.get("anchors", 128))
    segs = np.asarray(segs, np.int32).reshape(-1, 5)
    n_q = int(segs[:, 1].sum())
    Ls = W.prefix_lengths(R, cfg["L"], seed)
    cu_prefix = np.concatenate([[0], np.cumsum(Ls)]).astype(np.int32)
    NT, LT = R * n_q, int(cu_prefix[-1])
    ix = {"segs": torch.from_numpy(np.tile(segs, (R, 1))).to(dev), "cu_prefix": torch.from_numpy(cu_prefix).to(dev),
          "cu_q": torch.from_numpy((np.arange(R + 1) * n_q).astype(np.int32)).to(dev),
          "cu_seg": torch.from_numpy((np.arange(R + 1) * len(segs)).astype(np.int32)).to(dev)}
    gen = torch.Generator(device=dev)
    sets, tot = [], 0
    for k in range(16):
        gen.manual_seed(seed + k)
        t = {n: torch.randn(shape, generator=gen, device=dev).to(torch.bfloat16)
             for n, shape in (("q", (NT, Hq, d)), ("kp", (max(LT, 1), Hkv, d)), ("vp", (max(LT, 1), Hkv, d)),
                              ("kn", (NT, Hkv, d)), ("vn", (NT, Hkv, d)))}
        t["out"] = torch.empty_like(t["q"])
        sets.append(t)
        tot += sum(x.numel() * x.element_size() for x in t.values())
        if tot > 2.2 * l2 and k >= 1:
            break
    max_q, max_prefix = n_q, int(Ls.max()) if R else 0
    ws = d3d.new_workspace(d3d.d3d_packed_draft_attn_workspace_size(R, Hq, Hkv, d, max_q, max_prefix), dev)
    scale = 1.0 / math.sqrt(d)

    def call(t):
        return lambda: d3d.d3d_packed_draft_attn(t["q"], t["kp"], t["vp"], t["kn"], t["vn"], ix["segs"],
                                                 ix["cu_prefix"], ix["cu_q"], ix["cu_seg"], max_q, max_prefix,
                                                 scale, t["out"], ws)
    ms = _graph_time(torch, stream, [call(t) for t in sets])
    if d3d.d3d_workspace_status(ws) != 0:
        raise RuntimeError("attention device status %d" % d3d.d3d_workspace_status(ws))
    vis = 0
    for q0, ln, mode, par, plen in segs.tolist():
        vis += (ln * ln if mode == W.SEG_BIDIR else ln * (ln + 1) // 2) + ln * plen
    flops = 4.0 * d * Hq * R * (n_q * float(np.mean(Ls)) + vis)
    nbytes = 2.0 * (2 * LT * Hkv * d + 2 * NT * Hq * d + 2 * NT * Hkv * d)
    res = {"attn_us": round(ms * 1e3, 3), "query_tokens": NT, "prefix": cfg["L"], "flops": flops, "bytes": nbytes,
           "ctas": d3d.d3d_packed_draft_attn_ctas(R, Hq, Hkv, d, max_q, max_prefix)}
    res.update(attn_roofline(flops, nbytes, ms * 1e3, peaks))
    return res


def time_verify(d3d, torch, dev, stream, cfg, l2, peaks, seed=8000):
    """Device time of d3d_spec_verify (whole device, temperature 1) on one
    workload's verification shape, over rotating logit sets drawn on the
    device (target ~ N(0, 3^2), draft = target + N(0, 0.5^2), bf16)."""
    R, B, V = cfg["R"], cfg["B"], cfg["V"]
    gen = torch.Generator(device=dev)
    sets, tot = [], 0
    for k in range(16):
        gen.manual_seed(seed + k)
        x = torch.randn((R, B, V), generator=gen, device=dev) * 3.0
        z = x[:, : B - 1] + torch.randn((R, B - 1, V), generator=gen, device=dev) * 0.5
        t = {"target": x.to(torch.bfloat16), "draft": z.to(torch.bfloat16),
             "y": torch.randint(0, V, (R, B - 1), generator=gen, device=dev, dtype=torch.int32),
             "ua": torch.rand((R, B - 1), generator=gen, device=dev), "us": torch.rand((R,), generator=gen, device=dev),
             "acc": torch.empty(R, dtype=torch.int32, device=dev),
             "tok": torch.empty((R, B), dtype=torch.int32, device=dev),
             "n": torch.empty(R, dtype=torch.int32, device=dev)}
        del x, z
        sets.append(t)
        tot += t["target"].numel() * 2 + t["draft"].numel() * 2
        if tot > 2.2 * l2 and k >= 1:
            break
    ws = d3d.new_workspace(d3d.d3d_spec_verify_workspace_size(R, B, V), dev)

    def call(t):
        return lambda: d3d.d3d_spec_verify(t["target"], t["draft"], t["y"], t["ua"], t["us"], 1.0, t["acc"],
                                           t["tok"], t["n"], ws)
    ms = _graph_time(torch, stream, [call(t) for t in sets])
    nbytes = 2.0 * R * ((2 * B - 1) * V + 2 * V)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"verify_us": round(ms * 1e3, 3), "positions": R * B, "bytes": nbytes, "gbs": round(gbs, 1),
            "frac": round(gbs / peaks["hbm"], 4), "bound": "hbm"}


def other_workloads(d3d, torch, dev, stream, l2, peaks) -> dict:
    """long_block and serve32b (attention and verification), and the C/F
    budget sweep of the async pass at a 32768-token prefix (attention), with
    the measured KV-read-bound to tensor-bound crossover."""
    out = {}
    for name in ("long_block", "serve32b"):
        cfg = dict(W.CONFIGS[name])
        a = time_attention(d3d, torch, dev, stream, cfg, l2, peaks)
        v = time_verify(d3d, torch, dev, stream, cfg, l2, peaks)
        out[name] = {"attn": a, "verify": v, "attn_query_tokens_per_s": round(a["query_tokens"] / (a["attn_us"] * 1e-6), 1),
                     "verified_positions_per_s": round(v["positions"] / (v["verify_us"] * 1e-6), 1)}
    cfg = dict(W.CONFIGS["sweep"])
    points = []
    for C, F in ((1, 1), (2, 1), (3, 1), (4, 1), (4, 2), (8, 1), (4, 3), (8, 2), (12, 1), (4, 5), (16, 1),
                 (12, 2), (8, 3), (16, 2), (12, 3), (8, 5), (16, 3), (12, 5), (16, 5)):
        segs = W.async_segments(cfg["B"], C, F)
        r = time_attention(d3d, torch, dev, stream, cfg, l2, peaks, segs=segs)
        points.append({"C": C, "F": F, "N": int(segs[:, 1].sum()), "attn_us": r["attn_us"], "bound": r["bound"],
                       "tflops": r["tflops"], "gbs": r["gbs"], "frac": r["frac"], "ctas": r["ctas"],
                       "tensor_frac": round(r["tflops"] / peaks["bf16"], 4),
                       "hbm_frac": round(r["gbs"] / peaks["hbm"], 4)})
    points.sort(key=lambda p: p["N"])
    # measured crossover: the packed length at which the attention's tensor
    # utilisation overtakes its HBM utilisation (linear interpolation)
    cross = None
    for p0, p1 in zip(points, points[1:]):
        d0 = p0["tensor_frac"] - p0["hbm_frac"]
        d1 = p1["tensor_frac"] - p1["hbm_frac"]
        if d0 < 0 <= d1:
            cross = round(p0["N"] + (p1["N"] - p0["N"]) * (-d0) / (d1 - d0), 1)
            break
    ridge = peaks["bf16"] * 1e12 / (peaks["hbm"] * 1e9)
    G = cfg["Hq"] // cfg["Hkv"]
    out["sweep"] = {"prefix": cfg["L"], "points": points, "crossover_N_measured": cross,
                    "crossover_N_analytic": round(ridge / G, 1),
                    "crossover_rule": "N at which tensor utilisation (of the bf16 peak) overtakes HBM utilisation "
                                      "(of the copy bandwidth); analytic: arithmetic intensity ~ G*N flop/B "
                                      "reaches the ridge peak_bf16/peak_hbm"}
    return out


def run_e2e(torch, d3d, sets, n_sets, step, dev, stream, args, R, B, dist, graphs=True):
    """Same metric through the public API, inputs from pinned host memory and
    results read back every step; copies inside the timed region.

    A serving loop: each set's inputs live in one device buffer (views keep
    every tensor's shape and dtype) with a matching pinned host buffer, so a
    step is one host-to-device copy, the step's kernels and one device-to-host
    copy of the results.  With graphs=True the kernels are one CUDA graph per
    set, captured from the public calls; with graphs=False every step calls
    the C ABI entry points themselves (argument checks, workspace carving,
    tensor-map encoding and launches on the host each step).  The copies run
    on their own streams: step i+1's inputs move while step i computes, step
    i-1's results move back meanwhile, and a set is refilled only after its
    previous results have left."""
    in_keys = ["q", "kp", "vp", "kn", "vn", "segs", "cu_prefix", "cu_q", "cu_seg", "target", "draft", "y",
               "u_accept", "u_sample", "heads", "head_len"]
    out_keys = ["out", "out_tokens", "num_tokens", "branch"]

    def layout(keys):
        offs, o = {}, 0
        for k in keys:
            nb = sets[0][k].numel() * sets[0][k].element_size()
            offs[k] = (o, nb)
            o = (o + nb + 255) // 256 * 256  # every view starts 256-byte aligned
        return offs, o

    offs_in, tot_in = layout(in_keys)
    offs_out, tot_out = layout(out_keys)

    def views(buf, offs, ref):
        return {k: buf[o:o + nb].view(ref[k].dtype).view(ref[k].shape) for k, (o, nb) in offs.items()}

    packs = []
    for s in sets:
        din = torch.empty(tot_in, dtype=torch.uint8, device=dev)
        dout = torch.empty(tot_out, dtype=torch.uint8, device=dev)
        hin = torch.empty(tot_in, dtype=torch.uint8).pin_memory()
        hout = torch.empty(tot_out, dtype=torch.uint8).pin_memory()
        hv = views(hin, offs_in, s)
        for k in in_keys:
            hv[k].copy_(s[k].cpu())  # the set's inputs, staged on the host
        dset = dict(s)
        dset.update(views(din, offs_in, s))
        dset.update(views(dout, offs_out, s))
        packs.append(dict(din=din, dout=dout, hin=hin, hout=hout, dset=dset))
    h2d, d2h = tot_in, tot_out
    # the step's kernels as one graph per set (captured from the public calls)
    with torch.cuda.stream(stream):
        for pk in packs:
            pk["din"].copy_(pk["hin"], non_blocking=True)
            step(pk["dset"])  # eager pass: validates the calls on the new buffers
    torch.cuda.synchronize()
    for pk in packs if graphs else []:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(pk["dset"])
        pk["graph"] = g
    torch.cuda.synchronize()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in packs]
    ev_done = [torch.cuda.Event() for _ in packs]
    ev_out = [torch.cuda.Event() for _ in packs]
    used = [False] * len(packs)
    n = max(n_sets, min(args.steps, 2000))

    def one(i):
        j = i % n_sets
        pk = packs[j]
        if used[j]:
            s_in.wait_event(ev_out[j])  # the set's previous results have left
        with torch.cuda.stream(s_in):
            pk["din"].copy_(pk["hin"], non_blocking=True)
            ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        with torch.cuda.stream(stream):
            if graphs:
                pk["graph"].replay()
            else:
                step(pk["dset"])
            ev_done[j].record(stream)
        s_out.wait_event(ev_done[j])
        with torch.cuda.stream(s_out):
            pk["hout"].copy_(pk["dout"], non_blocking=True)
            ev_out[j].record(s_out)
        used[j] = True

    for i in range(n_sets):  # untimed pass of the loop
        one(i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    for i in range(n):
        one(i)
    stream.wait_stream(s_out)  # the last results are on the host
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    ms = reduce_max(ms, dist, dev)
    # the last step's results equal those of the same step run without the copies
    last = packs[(n - 1) % n_sets]
    ref = sets[(n - 1) % n_sets]
    hv_out = views(last["hout"], offs_out, ref)
    step(ref)
    torch.cuda.synchronize()
    for k in ("out_tokens", "num_tokens", "branch"):
        if not torch.equal(hv_out[k], ref[k].cpu()):
            raise RuntimeError("e2e: %s read back differs from the same step run in place" % k)
    world = dist.get_world_size() if dist is not None else 1
    n_q = sets[0]["q"].shape[0]
    return {"value": round(whole_job_rate(n_q, world, ms), 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 5), "steps": n,
            "pipeline": "one copy each way per step on their own streams, overlapped with the previous and "
                        "next steps; step kernels " + ("as one CUDA graph per input set" if graphs else
                                                       "launched by the C ABI calls themselves every step")}


# ----------------------------------------------------------------------------
# CPU oracle baseline / reference arm.
# ----------------------------------------------------------------------------
def host_cpu() -> dict:
    """Core count (usable by this process) and CPU model of the host."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None and os.path.exists("/proc/cpuinfo"):
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    return {"cores": cores, "cpu_model": model or "unknown"}


class OracleRound:
    """One whole round of the workload through the oracle (every packed token
    and query head, the full vocabulary, the branch match), on one thread or
    on all cores.  Inputs are generated once."""

    def __init__(self, wl_name: str, seed: int = 0):
        import oracle

        self.oracle = oracle
        self.wl = workload(wl_name)
        self.cfg = self.wl["cfg"]
        self.attn = W.attn_inputs(**self.cfg, seed=seed)
        self.v = W.verify_inputs(**self.cfg, seed=seed)
        self.hb = W.branch_heads(self.v["y"], self.cfg["B"], self.cfg.get("C", 1), self.cfg.get("F", 1),
                                 self.cfg["V"], seed=seed)

    def run(self, parallel: bool) -> float:
        o = self.oracle
        t0 = time.perf_counter()
        if parallel:
            o.packed_attn_par(self.attn)
            r = o.spec_verify_par(self.v)
        else:
            o.packed_attn(self.attn)
            r = o.spec_verify(self.v)
        o.branch_match(dict(verified=r["out_tokens"], verified_len=r["num_tokens"], heads=self.hb["heads"],
                            head_len=self.hb["head_len"]))
        return time.perf_counter() - t0


# The parity tests' near-tie rule: a draw whose |u_j - alpha_j| at the
# deciding test is below NEAR_TIE, or whose u*S lies within SAMPLE_BAND * S of
# a step of the oracle's CDF, is counted but not compared.
NEAR_TIE = 1e-5
SAMPLE_BAND = 1e-6


def workload_parity(torch, sets, cfg, rank, verify) -> dict:
    """The verification of every input set of the run (the step's call, fresh
    outputs) against the oracle in fp64: accepted lengths, token counts and
    tokens compared draw by draw outside the near-tie bands, which are
    counted and reported."""
    import oracle

    compared = ex_a = ex_s = mismatched = 0
    for i, s in enumerate(sets):
        s2 = dict(s)
        for k in ("accept_len", "out_tokens", "num_tokens", "branch"):
            s2[k] = torch.empty_like(s[k])
        verify(s2, 0, fused_match=True)
        torch.cuda.synchronize()
        v = W.verify_inputs(**cfg, seed=rank_seed(rank, i))
        try:
            ref = oracle.spec_verify_par(v)
        except RuntimeError:
            ref = oracle.spec_verify(v)
        tie_a = ref["margin_accept"] < NEAR_TIE
        tie_s = ~tie_a & (ref["margin_sample"] < SAMPLE_BAND)
        keep = ~tie_a & ~tie_s
        got = {k: s2[k].cpu().numpy() for k in ("accept_len", "num_tokens", "out_tokens")}
        for r in np.nonzero(keep)[0]:
            if any(not np.array_equal(got[k][r], ref[k][r]) for k in got):
                mismatched += 1
        compared += int(keep.sum())
        ex_a += int(tie_a.sum())
        ex_s += int(tie_s.sum())
    return {"kind": "oracle (fp64), every input set of the run", "draws": compared + ex_a + ex_s,
            "compared": compared, "mismatched": mismatched, "excluded_near_alpha": ex_a,
            "excluded_sample_band": ex_s, "rule": "|u - alpha| < %g at the deciding test; u*S within %g*S of a CDF step"
            % (NEAR_TIE, SAMPLE_BAND)}


def cpu_baseline(wl_name: str) -> dict:
    """The oracle on one whole round: one thread (threads_1) and all cores
    (threads_all: the same oracle functions on disjoint (request, head) and
    request slices from an OpenMP loop).  No sampling, no scaling."""
    import oracle

    s = OracleRound(wl_name)
    n_q = s.wl["n_q"] * s.wl["R"]
    hc = host_cpu()
    t1 = s.run(parallel=False)
    res = {"unit": UNIT, "kind": "oracle", "cores": hc["cores"], "cpu_model": hc["cpu_model"],
           "sample": "one whole round of %s (all %d packed tokens x %d query heads, verification over V=%d, "
                     "match); plain C oracle, fp64" % (wl_name, n_q, s.cfg["Hq"], s.cfg["V"]),
           "threads_1": {"value": round(n_q / t1, 3), "s_per_round": round(t1, 3), "threads": 1}}
    value = n_q / t1
    try:
        th = oracle.par_threads(hc["cores"])
        s.run(parallel=True)  # first call builds and warms the parallel library
        ta = min(s.run(parallel=True) for _ in range(3))
        res["threads_all"] = {"value": round(n_q / ta, 3), "s_per_round": round(ta, 3), "threads": th}
        value = n_q / ta
    except RuntimeError as e:
        res["threads_all"] = {"unavailable": str(e)}
    res["value"] = round(value, 3)  # the faster of the two
    return res


def run_reference(args, rank: int, world: int):
    """The reference arm: the oracle on this host's cores, one whole round per
    step (all packed tokens and heads, the full vocabulary, the match)."""
    if rank != 0:
        return
    import oracle

    K, Wm = args.steps, args.warmup
    s = OracleRound(args.workload)
    hc = host_cpu()
    threads = 1
    try:
        threads = oracle.par_threads(hc["cores"])
        parallel = True
        s.run(parallel=True)
    except RuntimeError:
        parallel = False
    for _ in range(Wm):
        s.run(parallel)
    t0 = time.perf_counter()
    per = [s.run(parallel) for _ in range(K)]
    wall = time.perf_counter() - t0
    ms = 1e3 * wall / K
    n_q = s.wl["n_q"] * s.wl["R"]
    value = n_q / (ms * 1e-3)
    desc = ("plain C oracle, fp64, %d thread(s) on %s: one whole round per step (%d packed tokens x %d query heads, "
            "verification over V=%d, match)" % (threads, hc["cpu_model"], n_q, s.cfg["Hq"], s.cfg["V"]))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": Wm, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded numpy)",
        "config": {"workload": workload_label(args.workload)},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "cpu_model": hc["cpu_model"],
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": round(wall, 2), "s_per_round_min": round(min(per), 3)}), flush=True)


def main():
    args = parse_args()
    if args.steps is None:
        args.steps = 5 if args.impl == "reference" else 20000
    if args.warmup is None:
        args.warmup = 3 if args.impl == "reference" else 200
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
