#!/usr/bin/env python3
"""Benchmark of the hybrid-tree verify step on one or more GPUs.

One step = graft_build_tree (prune, retrieve, merge) + graft_tree_attention
for every layer + graft_accept_compact + graft_update_M, on synthetic inputs
resident in HBM, replayed from one CUDA graph.  Default workload: the
LLaMA-3-8B-shaped verify step (batch 1, 32 layers, 32/8 heads, prefix 4096,
Kmax 64, vocab 128256, M 128256x16).

Prints one JSON line (rank 0).  Under torchrun every rank runs an
independent replica of the step on its own GPU (no collective on the data
path); ``value`` is the steps all ranks completed divided by the slowest
rank's time.

``--impl reference`` times the CPU oracle (a plain NumPy restatement of the
method) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "tree-verify steps/s; tree-attention HBM GB/s vs GB300 peak; retrieval fill µs"
UNIT = "steps/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
ATTN_SOURCES = ["attention_tc.cu", "attention_tcp.cu", "attention_tc1.cu", "attention_mma.cu", "attention.cuh",
                "attention_api.cu",
                "tc_ptx.cuh", "common.cuh"]


def parse_args():
    p = argparse.ArgumentParser(description=__doc__)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["graft", "reference"], default="graft")
    p.add_argument("--workload", default="llama3_8b")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-budget-s", type=float, default=20.0)
    p.add_argument("--secondary-reps", type=int, default=20,
                   help="replays of the attention / retrieval / tree-build graphs (0 skips them)")
    return p.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def slowest_over_ranks(seconds: float, device, world: int) -> float:
    """The longest of every rank's time (the job's time for weak-scaled replicas)."""
    if world <= 1:
        return seconds
    import torch
    import torch.distributed as dist
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                                          "-i", self.gpu, "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense bf16 TFLOP/s as a burst (the attention call is timed on its own)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["bf16_tflops"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_BF16_TFLOPS, "fallback"


# exp2 results per clock per SM of the special-function unit (four per SM sub-partition)
EX2_PER_CLOCK_PER_SM = 16


def attention_roofline(wl, L0, t_call, clocks, sms):
    """The three ideal times of one attention call and the fraction of each that the call achieves:
    HBM (compulsory bytes), tensor cores (4 Hq Kmax 128 sum L flops of the prefix part) and the
    exponential unit (Hq Kmax sum L exp2).  The bound is whichever of HBM and tensor is longer."""
    nbytes = attention_bytes_per_call(wl, L0)
    sum_l = int(L0.sum())
    flops = 4.0 * wl.Hq * wl.Kmax * wl.head_dim * sum_l
    ex2 = float(wl.Hq * wl.Kmax * sum_l)
    hbm, hbm_kind = measured_peaks()
    tc, tc_kind = measured_tensor_peak()
    mhz = (clocks or {}).get("sm_mhz") or 2070.0
    sfu = EX2_PER_CLOCK_PER_SM * sms * mhz * 1e6
    t_hbm, t_tc, t_sfu = nbytes / (hbm * 1e9), flops / (tc * 1e12), ex2 / sfu
    fractions = {"hbm": t_hbm / t_call, "tensor": t_tc / t_call, "sfu": t_sfu / t_call}
    if t_tc > t_hbm:
        r = {"bound": "tensor", "achieved": flops / t_call / 1e12, "peak": tc, "unit": "TFLOP/s",
             "peak_source": f"{tc_kind} bf16_tflops"}
    else:
        r = {"bound": "hbm", "achieved": nbytes / t_call / 1e9, "peak": hbm, "unit": "GB/s",
             "peak_source": f"{hbm_kind} hbm_gbs"}
    r["frac"] = r["achieved"] / r["peak"]
    r["fractions"] = fractions
    r["fractions_basis"] = (f"ideal time over the call's time: compulsory bytes at {hbm:.0f} GB/s, prefix flops at "
                            f"{tc:.0f} TFLOP/s, exp2 at {EX2_PER_CLOCK_PER_SM}/clock/SM x {sms} SMs x {mhz:.0f} MHz")
    r["bytes_per_call"], r["flops_per_call"], r["ex2_per_call"] = nbytes, flops, ex2
    return r


def attn_source_hash() -> str:
    h = hashlib.sha256()
    for fn in ATTN_SOURCES:
        with open(os.path.join(ROOT, "tree_verification_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per attention call from the committed ncu summary, if it matches this kernel source."""
    path = os.path.join(ROOT, "profiles", "attention_traffic.json")
    try:
        with open(path) as f:
            j = json.load(f)
        ent = j.get(workload)
        if ent and ent.get("source_hash") == attn_source_hash():
            return float(ent["dram_bytes_per_call"])
    except (OSError, ValueError):
        pass
    return None


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads", 0) for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


# ----------------------------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline leg)
# ----------------------------------------------------------------------------------------------

class OracleSample:
    """The oracle's step on host copies of a workload's inputs, timed piecewise.

    A sample runs the whole tree build, acceptance and M update for the
    sampled requests, the attention of one layer on ``attn_kv_heads`` KV
    heads, and the compaction of one layer; the step time is extrapolated to
    every request, KV head and layer.
    """

    def __init__(self, wl, inputs, max_requests=4):
        import numpy as np
        from oracle import config as oconfig
        self.np = np
        self.wl = wl
        self.cfg = oconfig.make_config(Kmax=wl.Kmax, D=wl.D, k=wl.k, V=wl.V, W=wl.W, checkpoints=wl.checkpoints,
                                       tau=wl.tau)
        self.reqs = list(range(min(wl.B, max_requests)))
        dl, tl, roots, L, succ, cnt, layer0 = inputs
        self.dl = dl[self.reqs].float().cpu().numpy()
        self.tl = tl[self.reqs].cpu().numpy()
        self.roots = roots[self.reqs].cpu().numpy()
        self.L = L[self.reqs].cpu().numpy()
        self.succ = succ.cpu().numpy()
        self.cnt = cnt.cpu().numpy()
        Q, Kc, Vc, Kt, Vt = layer0
        r = self.reqs
        self.Q = Q[r].float().cpu().numpy()
        self.Kc = Kc[r].float().cpu().numpy()
        self.Vc = Vc[r].float().cpu().numpy()
        self.Kt = Kt[r].float().cpu().numpy()
        self.Vt = Vt[r].float().cpu().numpy()

    def step(self, attn_kv_heads: int):
        """Run one sampled step; returns (extrapolated seconds, seconds actually spent)."""
        np = self.np
        from oracle import accept as oacc
        from oracle import attention as oatt
        from oracle import tree as otree
        from oracle import update_m as oupd
        wl, cfg = self.wl, self.cfg
        t0 = time.perf_counter()
        tree = otree.build_tree_batch(self.dl, self.roots, self.succ, self.L, cfg)
        t1 = time.perf_counter()
        group = wl.Hq // wl.Hkv
        heads = list(range(attn_kv_heads * group))
        for b in range(len(self.reqs)):
            lb = int(self.L[b])
            oatt.tree_attention_one(self.Q[b], self.Kc[b, :lb], self.Vc[b, :lb], self.Kt[b], self.Vt[b], lb,
                                    tree["mask"][b], 1 / math.sqrt(wl.head_dim), heads=heads)
        t2 = time.perf_counter()
        a = oacc.accept_batch(self.tl, tree)
        Kc, Vc = self.Kc.copy(), self.Vc.copy()
        oacc.compact(Kc, Vc, self.Kt, self.Vt, self.L.astype(np.int64), a["path"], a["acc_len"])
        t3 = time.perf_counter()
        oupd.update_M(self.succ, self.cnt, tree["tok"].reshape(-1), a["argmax"].reshape(-1))
        t4 = time.perf_counter()
        scale_req = wl.B / len(self.reqs)
        attn = (t2 - t1) * (wl.Hkv / attn_kv_heads) * wl.n_layers
        est = (t1 - t0) * scale_req + attn * scale_req + (t3 - t2) * scale_req + (t4 - t3) * scale_req
        return est, t4 - t0

    def describe(self, attn_kv_heads, n_steps):
        return (f"oracle (NumPy, float64 attention) on {len(self.reqs)} of {self.wl.B} requests: full tree build, "
                f"acceptance, compaction of one layer and M update; attention of layer 0 on {attn_kv_heads} of "
                f"{self.wl.Hkv} KV heads; extrapolated to all requests, heads and {self.wl.n_layers} layers; "
                f"{n_steps} sampled steps")


def oracle_timing(wl, inputs, budget_s: float, n_steps: int):
    samp = OracleSample(wl, inputs)
    est, spent = samp.step(1)  # one untimed pass sizes the sample
    kvh = wl.Hkv
    per = spent * max(1, wl.Hkv)  # rough cost of a step with every KV head
    if per * n_steps > budget_s:
        kvh = 1
    ests = []
    t_start = time.perf_counter()
    for _ in range(n_steps):
        e, _ = samp.step(kvh)
        ests.append(e)
        if time.perf_counter() - t_start > budget_s:
            break
    value = len(ests) / sum(ests)
    return value, samp.describe(kvh, len(ests))


# ----------------------------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------------------------

def make_inputs(wl, dev, gb, synth):
    import torch
    cfg = gb.graft_config_init(wl.Kmax, wl.D, wl.k, wl.V, wl.W, list(wl.checkpoints), wl.tau)
    Lcap = wl.lcap(1)
    dl = synth.draft_logits(wl, dev)
    roots = synth.root_tokens(wl).to(dev)
    L0 = synth.prefix_lengths(wl).to(dev)
    if wl.M_init == "zipf":
        s, c = synth.zipf_M(wl.V, wl.W, wl.seed + 5)
    else:
        s, c = synth.empty_M(wl.V, wl.W)
    M_succ, M_cnt = torch.from_numpy(s).to(dev), torch.from_numpy(c).to(dev)
    if wl.M_init == "warm":
        src, dst = synth.stream_pairs(synth.token_stream(wl.Lmax, wl.V, wl.seed + 41))
        sd, dd = torch.from_numpy(src).to(dev), torch.from_numpy(dst).to(dev)
        for _ in range(5):
            gb.graft_update_M(M_succ, M_cnt, sd, dd)
    layers = [synth.layer_tensors(wl, l, dev, Lcap=Lcap) for l in range(wl.n_layers)]
    tl = synth.target_logits(wl, dev)
    tree = gb.graft_build_tree(cfg, dl, roots, M_succ, L0)
    torch.cuda.synchronize()
    synth.plant_paths(tl, tree["tok"].cpu().numpy(), tree["parent"].cpu().numpy(), tree["depth"].cpu().numpy(),
                      synth.planted_lengths(wl))
    return cfg, Lcap, dl, roots, L0, M_succ, M_cnt, layers, tl


def input_arena(seg_tensors, dev):
    """Copies the tensors of each (key, [tensors]) segment into one device buffer, 256-byte aligned,
    segments contiguous.  Returns the buffer, each segment's byte range and the tensors' views."""
    import torch
    align = lambda x: (x + 255) // 256 * 256
    off, plan = 0, []
    for key, ts in seg_tensors:
        s0 = off
        offs = []
        for t in ts:
            offs.append(off)
            off = align(off + t.numel() * t.element_size())
        plan.append((key, ts, offs, s0, off))
    arena = torch.empty(off, dtype=torch.uint8, device=dev)
    segs, views = {}, {}
    for key, ts, offs, s0, s1 in plan:
        vs = []
        for t, o in zip(ts, offs):
            v = arena[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
            v.copy_(t)
            vs.append(v)
        segs[key] = (s0, s1)
        views[key] = vs
    return arena, segs, views


def attention_bytes_per_call(wl, L0) -> float:
    """Compulsory bytes of one layer call: prefix K and V, tree K and V, Q in, O out (bf16)."""
    d = wl.head_dim
    prefix = 2 * int(L0.sum()) * wl.Hkv * d * 2
    tree_kv = 2 * wl.B * wl.Kmax * wl.Hkv * d * 2
    q_o = 2 * wl.B * wl.Kmax * wl.Hq * d * 2
    return float(prefix + tree_kv + q_o)


def run_graft(args):
    import torch
    import torch.distributed as dist
    from tree_verification_gb300 import _build, synth
    from tree_verification_gb300 import binding as gb
    from tree_verification_gb300.step import VerifyStep

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    _build.build()
    wl = synth.WORKLOADS[args.workload]
    cfg, Lcap, dl, roots, L0, M_succ, M_cnt, layers, tl = make_inputs(wl, dev, gb, synth)
    # Every per-step input lives in one device arena, segment by segment in the order the step
    # consumes them (drafter logits, roots and lengths; then each layer's Q and tree K/V; then the
    # target logits), mirrored by one pinned host arena: the end-to-end step streams each segment
    # in with one copy while earlier stages run.
    seg_tensors = [("tree", [dl, roots, L0])] + [(l, [layers[l][0], layers[l][3], layers[l][4]])
                                                  for l in range(wl.n_layers)] + [("accept", [tl])]
    arena, segs, views = input_arena(seg_tensors, dev)
    dl, roots, L0 = views["tree"]
    tl = views["accept"][0]
    layers = [(views[l][0], layers[l][1], layers[l][2], views[l][1], views[l][2]) for l in range(wl.n_layers)]
    Q = [x[0] for x in layers]
    step = VerifyStep(cfg, wl.B, wl.Hq, wl.Hkv, wl.n_layers, Lcap, dev, [x[1] for x in layers],
                      [x[2] for x in layers], [x[3] for x in layers], [x[4] for x in layers])
    L = L0.clone()

    def body():
        L.copy_(L0)
        step.run(dl, roots, M_succ, M_cnt, L, Q, tl)

    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        body()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    n0 = gb.graft_launch_count()
    with torch.cuda.graph(graph):
        body()
    launches_per_step = gb.graft_launch_count() - n0

    # attention alone (every layer call of a step), for the roofline
    attn_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(attn_graph):
        for l in range(wl.n_layers):
            gb.graft_tree_attention(Q[l], step.Kc[l], step.Vc[l], step.Kt[l], step.Vt[l], L0, step.tree["mask"],
                                    step.scale, O=step.O, status=step.status, ws=step.ws_attn)
    # retrieval fill alone and the whole tree build
    n_rep = 100
    ret_out = torch.empty(wl.B, max(1, cfg.n_tmpl), dtype=torch.int32, device=dev)
    ret_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ret_graph):
        for _ in range(n_rep):
            gb.graft_retrieve(cfg, roots, M_succ, ret_tok=ret_out)
    tree_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(tree_graph):
        for _ in range(n_rep):
            gb.graft_build_tree(cfg, dl, roots, M_succ, L0, out=step.tree, ws=step.ws_tree)

    def timed(g, reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s.record()
        for _ in range(reps):
            g.replay()
        e.record()
        e.synchronize()
        return s.elapsed_time(e) / 1000.0

    def timed_steps(g, reps):
        """Total seconds of reps back-to-back replays, and each replay's milliseconds (an event
        before every replay and one after the last)."""
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        torch.cuda.synchronize()
        for i in range(reps):
            ev[i].record()
            g.replay()
        ev[reps].record()
        ev[reps].synchronize()
        per = [ev[i].elapsed_time(ev[i + 1]) for i in range(reps)]
        return ev[0].elapsed_time(ev[reps]) / 1000.0, per

    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x for x in vis.split(",") if x.strip()]
    sampler = ClockSampler(ids[local] if local < len(ids) else str(local))
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_main, per_step_ms = timed_steps(graph, args.steps)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    t_max = slowest_over_ranks(t_main, dev, world)
    status = int(step.status.item())

    # secondary timings (after the main timed region)
    t_attn = t_ret = t_tree = float("nan")
    if args.secondary_reps > 0:
        reps_attn = max(args.secondary_reps, min(args.steps, 300))
        t_attn = timed(attn_graph, reps_attn) / (reps_attn * wl.n_layers)
        t_ret = timed(ret_graph, args.secondary_reps) / (args.secondary_reps * n_rep)
        t_tree = timed(tree_graph, args.secondary_reps) / (args.secondary_reps * n_rep)

    # End to end through the public step API: every step copies its inputs in from pinned host
    # memory (one copy per segment, on a copy stream, each stage waiting only for its own segment)
    # and reads its accepted tokens and lengths back; the whole thing is one captured graph.
    host_arena = arena.cpu().pin_memory()
    out_host = torch.empty(wl.B, wl.Kmax, dtype=torch.int32).pin_memory()
    len_host = torch.empty(wl.B, dtype=torch.int32).pin_memory()
    h2d = sum(s1 - s0 for s0, s1 in segs.values())
    d2h = out_host.numel() * 4 + len_host.numel() * 4
    copy_stream = torch.cuda.Stream(device=dev)
    seg_ready = {k: torch.cuda.Event() for k in segs}

    def e2e_body():
        main = torch.cuda.current_stream()
        copy_stream.wait_stream(main)
        with torch.cuda.stream(copy_stream):
            for k, (s0, s1) in segs.items():
                arena[s0:s1].copy_(host_arena[s0:s1], non_blocking=True)
                seg_ready[k].record()
        main.wait_event(seg_ready["tree"])
        L.copy_(L0)
        step.run(dl, roots, M_succ, M_cnt, L, Q, tl, inputs_ready=lambda k: main.wait_event(seg_ready[k]))
        out_host.copy_(step.acc["out_tok"], non_blocking=True)
        len_host.copy_(step.acc["acc_len"], non_blocking=True)

    e2e_body()
    torch.cuda.synchronize()
    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph):
        e2e_body()

    def e2e_step():
        e2e_graph.replay()
        torch.cuda.current_stream().synchronize()

    n_e2e = min(args.e2e_steps, args.steps)
    t_e2e = float("nan")
    if n_e2e > 0:
        for _ in range(3):
            e2e_step()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        t_e2e = time.perf_counter() - t0
    t_e2e = slowest_over_ranks(t_e2e, dev, world)

    # the fused lm_head argmax (greedy tokens straight from final hidden states) on this workload's rows
    lmh = sample_from_logits = None
    if args.secondary_reps > 0:
        H, W_lm = synth.lm_head_inputs(wl, dev)
        g_out = torch.empty(H.shape[0], dtype=torch.int32, device=dev)
        m_out = torch.empty(H.shape[0], dtype=torch.float32, device=dev)
        lws = torch.empty(max(1, gb.graft_lm_head_argmax_workspace_size(H.shape[0])), dtype=torch.uint8, device=dev)
        lmh_graph = torch.cuda.CUDAGraph()
        gb.graft_lm_head_argmax(H, W_lm, g_out, m_out, step.status, lws)
        torch.cuda.synchronize()
        with torch.cuda.graph(lmh_graph):
            gb.graft_lm_head_argmax(H, W_lm, g_out, m_out, step.status, lws)
        for _ in range(3):
            lmh_graph.replay()
        t_lmh = timed(lmh_graph, args.secondary_reps) / args.secondary_reps
        flops = 2.0 * H.shape[0] * wl.d_model * wl.V
        nbytes = (H.numel() + W_lm.numel()) * 2 + H.shape[0] * 8
        lmh = {"rows": H.shape[0], "d_model": wl.d_model, "vocab": wl.V, "us": t_lmh * 1e6,
               "tflops": flops / t_lmh / 1e12, "gbs": nbytes / t_lmh / 1e9}
        # sampling acceptance: the target's sample per node, fused into the lm_head and from given logits
        pos = step.tree["pos"]
        smp_graph = torch.cuda.CUDAGraph()
        gb.graft_lm_head_sample(H, W_lm, pos, 1.0, 1234, sampled=g_out, status=step.status, ws=lws)
        torch.cuda.synchronize()
        with torch.cuda.graph(smp_graph):
            gb.graft_lm_head_sample(H, W_lm, pos, 1.0, 1234, sampled=g_out, status=step.status, ws=lws)
        for _ in range(3):
            smp_graph.replay()
        t_smp = timed(smp_graph, args.secondary_reps) / args.secondary_reps
        lmh["sample_us"] = t_smp * 1e6
        sws = torch.empty(max(1, gb.graft_sample_tokens_workspace_size(wl.B, wl.Kmax, wl.V)), dtype=torch.uint8,
                          device=dev)
        st_graph = torch.cuda.CUDAGraph()
        gb.graft_sample_tokens(tl, pos, 1.0, 1234, sampled=step.acc["argmax"], ws=sws)
        torch.cuda.synchronize()
        with torch.cuda.graph(st_graph):
            gb.graft_sample_tokens(tl, pos, 1.0, 1234, sampled=step.acc["argmax"], ws=sws)
        for _ in range(3):
            st_graph.replay()
        t_st = timed(st_graph, args.secondary_reps) / args.secondary_reps
        sample_from_logits = {"us": t_st * 1e6, "gbs": tl.numel() * 4 / t_st / 1e9}
        del H, W_lm

    # attention alone on the other workloads' shapes (the long-context and batched configurations
    # carry the HBM target), four distinct layers per replay so every call streams from DRAM
    attn_other = {}
    if args.secondary_reps > 0 and world == 1:
        from tree_verification_gb300 import attn_bench
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        for name in ("llama31_8b_long", "qwen3_8b_batch", "qwen3_235b"):
            owl = synth.WORKLOADS[name]
            us, nb, st = attn_bench.time_calls(owl, 4, 10, dev=dev)
            r = attention_roofline(owl, synth.prefix_lengths(owl), us * 1e-6, clocks, sms)
            attn_other[name] = {"call_us": us, "gbs": nb / us / 1e3, "bound": r["bound"], "frac": r["frac"],
                                "fractions": r["fractions"], "status": st}
        torch.cuda.empty_cache()

    bytes_call = attention_bytes_per_call(wl, L0.cpu())
    peak, peak_kind = measured_peaks()
    achieved = bytes_call / t_attn / 1e9
    traffic = recorded_traffic(args.workload)
    roof = attention_roofline(wl, L0.cpu(), t_attn, clocks, torch.cuda.get_device_properties(dev).multi_processor_count)
    roof.update({"traffic": traffic, "kernel": "graft_tree_attention (one layer call)", "call_us": t_attn * 1e6})
    q = statistics.quantiles(per_step_ms, n=10) if len(per_step_ms) >= 10 else [float("nan")] * 9
    result = {
        "metric": METRIC, "value": world * args.steps / t_max, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1000.0 * t_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.B, "layers": wl.n_layers, "heads_q_kv": [wl.Hq, wl.Hkv],
                   "head_dim": wl.head_dim, "prefix": list(wl.L), "Kmax": wl.Kmax, "draft_depth_topk": [wl.D, wl.k],
                   "vocab": wl.V, "M_width": wl.W, "tau": wl.tau, "checkpoints": list(wl.checkpoints),
                   "l2": f"inputs larger than L2: {bytes_call * wl.n_layers / 1e6:.0f} MB of attention operands "
                         f"per step in distinct per-layer buffers",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "accumulate": "fp32"},
        "roofline": roof,
        "step_ms": {"median": statistics.median(per_step_ms), "p10": q[0], "p90": q[8]},
        "e2e": {"value": world * n_e2e / t_e2e if n_e2e > 0 else None, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "secondary": {"tree_attention_gbs": achieved, "tree_attention_frac_of_peak": achieved / peak,
                      "retrieval_fill_us": t_ret * 1e6, "build_tree_us": t_tree * 1e6,
                      "launches_per_step": launches_per_step, "device_status": status,
                      "lm_head_argmax": lmh, "sample_tokens_from_logits": sample_from_logits,
                      "attention_other_workloads": attn_other},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        inputs = (dl, tl, roots, L0, M_succ, M_cnt, layers[0])
        v, desc = oracle_timing(wl, inputs, args.cpu_budget_s, n_steps=50)
        result["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                                  "sample": desc}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args):
    import torch
    from tree_verification_gb300 import _build, synth
    from tree_verification_gb300 import binding as gb

    world, rank, local = dist_env()
    if rank != 0:
        return  # the reference arm runs once, on rank 0
    wl = synth.WORKLOADS[args.workload]
    # inputs are drawn exactly as the GPU arm draws them (on the GPU when one is present)
    if torch.cuda.is_available():
        dev = torch.device(f"cuda:{local}")
        torch.cuda.set_device(dev)
        _build.build()
        cfg, Lcap, dl, roots, L0, M_succ, M_cnt, layers, tl = make_inputs(wl.scaled(n_layers=1), dev, gb, synth)
        inputs = (dl, tl, roots, L0, M_succ, M_cnt, layers[0])
    else:
        dev = torch.device("cpu")
        small = wl
        Lcap = wl.lcap(1)
        s, c = synth.empty_M(wl.V, wl.W) if wl.M_init != "zipf" else synth.zipf_M(wl.V, wl.W, wl.seed + 5)
        inputs = (synth.draft_logits(small, dev), synth.target_logits(small, dev), synth.root_tokens(small),
                  synth.prefix_lengths(small), torch.from_numpy(s), torch.from_numpy(c),
                  synth.layer_tensors(small, 0, dev, Lcap=Lcap))
    samp = OracleSample(wl, inputs)
    for _ in range(max(0, min(args.warmup, 3))):
        samp.step(1)
    budget = 150.0
    _, spent = samp.step(1)
    n_run = max(1, min(args.steps, int(budget / max(spent, 1e-3))))
    ests = [samp.step(1)[0] for _ in range(n_run)]
    value = len(ests) / sum(ests)
    desc = samp.describe(1, n_run) + f" (of {args.steps} requested steps, bounded to about {budget:.0f} s)"
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 / value, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": wl.name, "batch": wl.B, "layers": wl.n_layers, "prefix": list(wl.L),
                      "Kmax": wl.Kmax, "vocab": wl.V},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle", "sample": desc},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_graft(args)


if __name__ == "__main__":
    main()
