#!/usr/bin/env python3
"""Benchmark of the hybrid-tree verify step on one or more GPUs.

    python bench.py [--gpus N] [--steps K] [--warmup W]

One step = graft_build_tree (prune, retrieve, merge) + graft_tree_attention
for every layer + graft_accept_compact + graft_update_M, on synthetic inputs
resident in HBM, replayed from one CUDA graph.  The headline line times K
steps of the largest single-GPU workload, the Qwen3-235B-shaped step (batch
16, 64/4 heads, 94 layer calls over 8192-token prefixes, Kmax 64, vocab
151936, M 151936x32; 25 GB of KV per step).  The line's ``configs`` object
times the whole step of the four other workloads the same way (tiny,
llama3_8b, qwen3_8b_batch, llama31_8b_long), each with its steps/s, its
attention call against the roofline, tree attention plus KV compaction
against the HBM roofline, the tree build, the retrieval fill and an
end-to-end step.

Every measured workload also runs end to end through the public step API
(``e2e``): each step copies its inputs in from pinned host memory and reads
the accepted tokens and lengths back, all inside the timed region.

Under torchrun every rank runs an independent replica of the step on its own
GPU (no collective on the data path); ``value`` is the steps all ranks
completed divided by the slowest rank's time.

``--impl reference`` times the CPU oracle (a plain NumPy restatement of the
method) on the host cores, on bounded samples of the same workload; it never
loads the CUDA library.  ``cpu_baseline`` in the GPU arm's line is the same
oracle on a sample of the headline workload, and ``cpu_full_steps`` times
whole oracle steps of the tiny and LLaMA-3-8B workloads on one host thread
and on all of them.

Other modes:
    --mode attention --workload W [--layers N --reps R --lcap C]
        microseconds per graft_tree_attention call of a workload
    --mode lm_head [--rows N --d-model D --vocab V --reps R]
        the fused lm_head argmax and sampling kernels
    --mode tree --workload W [--drafts flat|confident --reps R]
        microseconds per graft_build_tree call of a workload
    --mode cpu_step --workload W
        one whole oracle step on the host (run by the default mode in a
        subprocess, to fix the BLAS thread count)
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
HEADLINE = "qwen3_235b"
OTHER_CONFIGS = ["tiny", "llama3_8b", "qwen3_8b_batch", "llama31_8b_long"]
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
ATTN_SOURCES = ["attention_tc.cu", "attention_tcp.cu", "attention_tcs.cu", "attention_tc1.cu", "attention_mma.cu",
                "attention.cuh", "attention_api.cu", "tc_ptx.cuh", "common.cuh"]
BLAS_ENV = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["graft", "reference"], default="graft")
    p.add_argument("--mode", choices=["step", "attention", "lm_head", "tree", "cpu_step"], default="step")
    p.add_argument("--workload", default=HEADLINE)
    p.add_argument("--configs", default=",".join(OTHER_CONFIGS),
                   help="comma-separated workloads timed beside the headline ('none' for none)")
    p.add_argument("--e2e-steps", type=int, default=0,
                   help="end-to-end steps (0: the same as --steps; negative: none)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-budget-s", type=float, default=20.0)
    p.add_argument("--reference-budget-s", type=float, default=150.0)
    p.add_argument("--secondary-reps", type=int, default=10,
                   help="replays of the attention / compaction / tree-build graphs (0 skips them and the lm_head)")
    # --mode attention / lm_head / tree
    p.add_argument("--drafts", choices=["flat", "confident"], default="flat",
                   help="--mode tree: the workload's drafter logits (flat: pruned at the first checkpoint) or "
                        "confident rows that draft through every call")
    p.add_argument("--layers", type=int, default=4)
    p.add_argument("--reps", type=int, default=20)
    p.add_argument("--lcap", type=int, default=0)
    p.add_argument("--rows", type=int, default=64)
    p.add_argument("--d-model", type=int, default=4096)
    p.add_argument("--vocab", type=int, default=128256)
    return p.parse_args(argv)


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


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def measured_peaks():
    j = _peaks()
    if "hbm_gbs" in j:
        return float(j["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak(sustained: bool = False):
    """Dense bf16 TFLOP/s: the burst figure (a kernel timed on its own) or the sustained one."""
    j = _peaks()
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    if key in j:
        return float(j[key]), "measured"
    return FALLBACK_BF16_TFLOPS, "fallback"


# exp2 results per clock per SM of the special-function unit (four per SM sub-partition)
EX2_PER_CLOCK_PER_SM = 16


def attention_bytes_per_call(wl, L0) -> float:
    """Compulsory bytes of one layer call: prefix K and V, tree K and V, Q in, O out (bf16)."""
    d = wl.head_dim
    prefix = 2 * int(L0.sum()) * wl.Hkv * d * 2
    tree_kv = 2 * wl.B * wl.Kmax * wl.Hkv * d * 2
    q_o = 2 * wl.B * wl.Kmax * wl.Hq * d * 2
    return float(prefix + tree_kv + q_o)


def compaction_bytes_per_step(wl, acc_len) -> float:
    """Bytes one step's KV compaction must move: every accepted node's K and V row (Hkv x 128 bf16) read
    from the tree KV and written into the cache, in every layer."""
    rows = int(sum(int(x) for x in acc_len))
    return float(rows * 2 * 2 * wl.Hkv * wl.head_dim * 2 * wl.n_layers)


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
             "peak_source": f"{tc_kind} bf16_tflops (burst)"}
        tcs, _ = measured_tensor_peak(sustained=True)
        r["frac_of_sustained"] = r["achieved"] / tcs
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
    for k in BLAS_ENV:
        v = os.environ.get(k)
        if v and v.isdigit():
            return int(v)
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads", 0) for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


# ----------------------------------------------------------------------------------------------
# CPU oracle (the reference arm, cpu_baseline and cpu_full_steps).  Nothing here loads the CUDA
# library: inputs come from the seeded generators and the oracle's own tree.
# ----------------------------------------------------------------------------------------------

def oracle_inputs(wl, dev, layers):
    """Host copies of one step's inputs for the oracle: drafter and target logits (the target's planted
    on the oracle's tree), roots, lengths, M and the listed layers' Q / caches / tree KV (float32)."""
    import numpy as np
    from oracle import config as oconfig
    from oracle import tree as otree
    from oracle import update_m as oupd
    from tree_verification_gb300 import synth
    cfg = oconfig.make_config(Kmax=wl.Kmax, D=wl.D, k=wl.k, V=wl.V, W=wl.W, checkpoints=wl.checkpoints, tau=wl.tau)
    dl = synth.draft_logits(wl, dev).cpu().numpy()
    roots = synth.root_tokens(wl).numpy()
    L = synth.prefix_lengths(wl).numpy()
    if wl.M_init == "zipf":
        succ, cnt = synth.zipf_M(wl.V, wl.W, wl.seed + 5)
    else:
        succ, cnt = synth.empty_M(wl.V, wl.W)
        if wl.M_init == "warm":
            src, dst = synth.stream_pairs(synth.token_stream(wl.Lmax, wl.V, wl.seed + 41))
            for _ in range(5):
                succ, cnt = oupd.update_M(succ, cnt, src, dst)
    tree = otree.build_tree_batch(dl, roots, succ, L, cfg)
    tl_t = synth.target_logits(wl, dev)
    synth.plant_paths(tl_t, tree["tok"], tree["parent"], tree["depth"], synth.planted_lengths(wl))
    tl = tl_t.cpu().numpy()
    del tl_t
    Lcap = wl.lcap(1)
    lay = {}
    for l in layers:
        lay[l] = [x.float().cpu().numpy() for x in synth.layer_tensors(wl, l, dev, Lcap=Lcap)]
    return dict(cfg=cfg, dl=dl, roots=roots, L=L.astype(np.int64), succ=succ, cnt=cnt, tl=tl, layers=lay)


def oracle_step_sample(wl, inp, attn_requests, compact_layers):
    """One sampled oracle step: the whole tree build, acceptance and M update for every request, the
    attention of one layer call for ``attn_requests`` requests (all heads), and the compaction of
    ``compact_layers`` layers.  Returns (estimated seconds of a whole step, seconds spent, seconds of the
    sampled attention): attention scales by requests and layers, compaction by layers."""
    from oracle import accept as oacc
    from oracle import attention as oatt
    from oracle import tree as otree
    from oracle import update_m as oupd
    l0 = min(inp["layers"])
    Q, Kc, Vc, Kt, Vt = inp["layers"][l0]
    scale = 1 / math.sqrt(wl.head_dim)
    t0 = time.perf_counter()
    tree = otree.build_tree_batch(inp["dl"], inp["roots"], inp["succ"], inp["L"], inp["cfg"])
    t1 = time.perf_counter()
    for b in attn_requests:
        lb = int(inp["L"][b])
        oatt.tree_attention_one(Q[b], Kc[b, :lb], Vc[b, :lb], Kt[b], Vt[b], lb, tree["mask"][b], scale)
    t2 = time.perf_counter()
    a = oacc.accept_batch(inp["tl"], tree)
    t3 = time.perf_counter()
    for l in sorted(inp["layers"])[:compact_layers]:
        _, Kc_l, Vc_l, Kt_l, Vt_l = inp["layers"][l]
        oacc.compact(Kc_l.copy(), Vc_l.copy(), Kt_l, Vt_l, inp["L"], a["path"], a["acc_len"])
    t4 = time.perf_counter()
    oupd.update_M(inp["succ"], inp["cnt"], tree["tok"].reshape(-1), a["argmax"].reshape(-1))
    t5 = time.perf_counter()
    attn = (t2 - t1) * (wl.B / max(1, len(attn_requests))) * wl.n_layers
    compact = (t4 - t3) * (wl.n_layers / max(1, compact_layers))
    est = (t1 - t0) + attn + (t3 - t2) + compact + (t5 - t4)
    return est, t5 - t0, t2 - t1


def oracle_whole_step(wl, inp):
    """One whole oracle step (every request, every layer's attention and compaction); seconds."""
    from oracle import step as ostep
    n = wl.n_layers
    lay = [inp["layers"][l] for l in range(n)]
    Kc = [x[1].copy() for x in lay]
    Vc = [x[2].copy() for x in lay]
    t0 = time.perf_counter()
    ostep.verify_step(inp["cfg"], inp["dl"], inp["roots"], inp["succ"], inp["cnt"], inp["L"], [x[0] for x in lay],
                      Kc, Vc, [x[3] for x in lay], [x[4] for x in lay], inp["tl"], 1 / math.sqrt(wl.head_dim))
    return time.perf_counter() - t0


def calibrated_requests(wl, inp, seconds: float):
    """How many requests' attention (of one layer call) a sample may include to take about `seconds`
    (one calibration sample with one request; the stages other than attention always run whole)."""
    _, spent, t_attn = oracle_step_sample(wl, inp, [0], 1)
    per_req = max(t_attn, 1e-4)
    n = int(max(1, min(wl.B, (seconds - (spent - t_attn)) / per_req)))
    return n, spent


def run_cpu_step(args):
    """--mode cpu_step: whole oracle steps of one workload on this process's BLAS threads (one JSON line)."""
    import torch
    from tree_verification_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    dev = torch.device("cpu")
    inp = oracle_inputs(wl, dev, range(wl.n_layers))
    n = max(1, args.steps)
    secs = [oracle_whole_step(wl, inp) for _ in range(n)]
    t = statistics.median(secs)
    print(json.dumps({"workload": wl.name, "steps_per_s": 1.0 / t, "seconds_per_step": t, "steps": n,
                      "threads": blas_threads(), "kind": "oracle", "sample": "whole steps"}), flush=True)


def cpu_full_steps(budget_s: float):
    """Whole oracle steps of the tiny and LLaMA-3-8B workloads on one host thread and on every host thread,
    each in a subprocess whose BLAS thread count is fixed before NumPy loads."""
    out = {}
    for name, steps in (("tiny", 5), ("llama3_8b", 1)):
        for label, threads in (("one_thread", 1), ("all_threads", os.cpu_count() or 1)):
            env = dict(os.environ)
            for k in BLAS_ENV:
                env[k] = str(threads)
            cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--mode", "cpu_step", "--workload", name,
                   "--steps", str(steps)]
            try:
                r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=budget_s)
                line = [x for x in r.stdout.splitlines() if x.startswith("{")]
                out.setdefault(name, {})[label] = json.loads(line[-1]) if line else {"error": r.stderr[-300:]}
            except subprocess.TimeoutExpired:
                out.setdefault(name, {})[label] = {"error": f"over {budget_s:.0f} s"}
    return out


def run_reference(args):
    """The reference arm: the CPU oracle on the host cores (rank 0 only), never the CUDA library."""
    world, rank, local = dist_env()
    if rank != 0:
        return  # the reference arm runs once, on rank 0
    import torch
    from tree_verification_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    # the same seeded inputs as the GPU arm: drawn with torch's generator on the GPU when there is one
    # (torch plumbing only), then copied to the host
    dev = torch.device(f"cuda:{local}") if torch.cuda.is_available() else torch.device("cpu")
    inp = oracle_inputs(wl, dev, [0])
    if dev.type == "cuda":
        torch.cuda.empty_cache()
    # each step is a bounded sample: the whole tree build, acceptance and M update, the compaction of one
    # layer, and one layer call's attention for as many requests as fit this run's time budget
    per_step = args.reference_budget_s / max(1, args.steps + min(args.warmup, 1))
    n_req, _ = calibrated_requests(wl, inp, per_step)
    reqs = list(range(n_req))
    for _ in range(min(args.warmup, 1)):
        oracle_step_sample(wl, inp, reqs, 1)
    ests, spent = [], []
    for _ in range(args.steps):
        e, s, _ = oracle_step_sample(wl, inp, reqs, 1)
        ests.append(e)
        spent.append(s)
    value = len(ests) / sum(ests)
    ms_sample = 1000.0 * sum(spent) / len(spent)
    desc = (f"oracle (NumPy, float64 attention) on {os.cpu_count()} host cores; each timed step is one sample: the "
            f"whole tree build, acceptance and M update for all {wl.B} requests, the compaction of 1 of "
            f"{wl.n_layers} layers, and one layer call's attention for {n_req} of {wl.B} requests (all heads)")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_sample, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": workload_config(wl, world),
           "extrapolated": {"value_is": "whole-step throughput estimated from the samples",
                            "ms_per_step_is": "measured wall time of one timed sample",
                            "attention_scale": wl.B / n_req * wl.n_layers, "compaction_scale": wl.n_layers,
                            "estimated_ms_per_whole_step": 1000.0 / value},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle", "sample": desc},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ----------------------------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------------------------

def workload_config(wl, world=1):
    """The workload's sizes as the JSON line's config (the same object in both arms)."""
    from tree_verification_gb300 import synth
    gb_step = attention_bytes_per_call(wl, synth.prefix_lengths(wl)) * wl.n_layers / 1e9
    return {"workload": wl.name, "batch": wl.B, "layers": wl.n_layers, "heads_q_kv": [wl.Hq, wl.Hkv],
            "head_dim": wl.head_dim, "prefix": list(wl.L), "Kmax": wl.Kmax, "draft_depth_topk": [wl.D, wl.k],
            "vocab": wl.V, "M_width": wl.W, "tau": wl.tau, "checkpoints": list(wl.checkpoints),
            "parallelism": "replicas" if world > 1 else "single GPU", "accumulate": "fp32",
            "l2": f"inputs larger than L2: {gb_step:.2f} GB of attention operands per step in distinct per-layer "
                  f"buffers"}


def make_inputs(wl, dev, gb, synth):
    """A workload's device inputs; the target logits get their planted paths on the GPU's own tree."""
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


def _timed(g, reps):
    """Seconds of reps back-to-back replays of graph g (CUDA events on the current stream)."""
    import torch
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record()
    for _ in range(reps):
        g.replay()
    e.record()
    e.synchronize()
    return s.elapsed_time(e) / 1000.0


def _timed_steps(g, reps):
    """Total seconds of reps back-to-back replays, and each replay's milliseconds (an event before every
    replay and one after the last, on the current stream)."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    torch.cuda.synchronize()
    for i in range(reps):
        ev[i].record()
        g.replay()
    ev[reps].record()
    ev[reps].synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(reps)]
    return ev[0].elapsed_time(ev[reps]) / 1000.0, per


def _capture(fn):
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()  # warm the launch path outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


class WorkloadBench:
    """One workload's whole step on the GPU: inputs resident in HBM (one device arena for every per-step
    input, mirrored by a pinned host arena for the end-to-end step), the step and its parts captured in
    CUDA graphs."""

    def __init__(self, wl, dev):
        import torch
        from tree_verification_gb300 import binding as gb
        from tree_verification_gb300 import synth
        from tree_verification_gb300.step import VerifyStep
        self.wl, self.dev, self.gb = wl, dev, gb
        cfg, Lcap, dl, roots, L0, M_succ, M_cnt, layers, tl = make_inputs(wl, dev, gb, synth)
        self.cfg, self.Lcap, self.M_succ, self.M_cnt = cfg, Lcap, M_succ, M_cnt
        # every per-step input in one arena, segment by segment in the order the step consumes them
        # (drafter logits, roots and lengths; then each layer's Q and tree K/V; then the target logits)
        seg_tensors = [("tree", [dl, roots, L0])] + [(l, [layers[l][0], layers[l][3], layers[l][4]])
                                                      for l in range(wl.n_layers)] + [("accept", [tl])]
        self.arena, self.segs, views = input_arena(seg_tensors, dev)
        del dl, tl
        self.dl, self.roots, self.L0 = views["tree"]
        self.tl = views["accept"][0]
        self.Q = [views[l][0] for l in range(wl.n_layers)]
        Kc = [layers[l][1] for l in range(wl.n_layers)]
        Vc = [layers[l][2] for l in range(wl.n_layers)]
        Kt = [views[l][1] for l in range(wl.n_layers)]
        Vt = [views[l][2] for l in range(wl.n_layers)]
        del layers
        torch.cuda.empty_cache()
        self.step = VerifyStep(cfg, wl.B, wl.Hq, wl.Hkv, wl.n_layers, Lcap, dev, Kc, Vc, Kt, Vt)
        self.L = self.L0.clone()
        n0 = gb.graft_launch_count()
        self.graph = _capture(self._body)
        self.launches_per_step = gb.graft_launch_count() - n0

    def _body(self):
        self.L.copy_(self.L0)
        self.step.run(self.dl, self.roots, self.M_succ, self.M_cnt, self.L, self.Q, self.tl)

    def time_steps(self, reps, warmup):
        for _ in range(max(3, warmup)):
            self.graph.replay()
        return _timed_steps(self.graph, reps)

    def parts(self, reps):
        """Seconds per attention call, per acceptance + compaction call (the argmax given), per tree build
        and per retrieval fill, each from its own captured graph."""
        import torch
        gb, st, wl = self.gb, self.step, self.wl

        def attn():
            for l in range(wl.n_layers):
                gb.graft_tree_attention(self.Q[l], st.Kc[l], st.Vc[l], st.Kt[l], st.Vt[l], self.L0, st.tree["mask"],
                                        st.scale, O=st.O, status=st.status, ws=st.ws_attn)

        def compact():
            self.L.copy_(self.L0)
            gb.graft_accept_compact(None, st.tree["tok"], st.tree["parent"], st.tree["depth"], st.Kc_ptrs,
                                    st.Vc_ptrs, st.Kt_ptrs, st.Vt_ptrs, wl.n_layers, wl.Hkv, self.Lcap, self.L,
                                    out=st.acc, status=st.status, ws=st.ws_acc, argmax=st.acc["argmax"], V=wl.V)

        n_rep = 20
        ret_out = torch.empty(wl.B, max(1, self.cfg.n_tmpl), dtype=torch.int32, device=self.dev)

        def retrieve():
            for _ in range(n_rep):
                gb.graft_retrieve(self.cfg, self.roots, self.M_succ, ret_tok=ret_out)

        def tree():
            for _ in range(n_rep):
                gb.graft_build_tree(self.cfg, self.dl, self.roots, self.M_succ, self.L0, out=st.tree, ws=st.ws_tree)

        self.graph.replay()  # one step fills the tree, argmax and lengths the parts read
        torch.cuda.synchronize()
        out = {}
        for name, fn, per in (("attention", attn, wl.n_layers), ("compaction", compact, 1),
                              ("retrieval", retrieve, n_rep), ("tree", tree, n_rep)):
            g = _capture(fn)
            g.replay()
            out[name] = _timed(g, reps) / (reps * per)
            del g
        # the compaction graph advanced L and rewrote the accept outputs; one more step restores them
        self.graph.replay()
        torch.cuda.synchronize()
        return out

    def e2e(self, steps):
        """Seconds for `steps` end-to-end steps through VerifyStep.run: every step copies its inputs from
        pinned host memory (one copy per stage segment on a copy stream, each stage waiting only for its
        own segment) and reads the accepted tokens and lengths back; one captured graph per step."""
        import torch
        wl, st = self.wl, self.step
        host_arena = self.arena.cpu().pin_memory()
        out_host = torch.empty(wl.B, wl.Kmax, dtype=torch.int32).pin_memory()
        len_host = torch.empty(wl.B, dtype=torch.int32).pin_memory()
        h2d = sum(s1 - s0 for s0, s1 in self.segs.values())
        d2h = out_host.numel() * 4 + len_host.numel() * 4
        copy_stream = torch.cuda.Stream(device=self.dev)
        seg_ready = {k: torch.cuda.Event() for k in self.segs}
        arena = self.arena

        def body():
            main = torch.cuda.current_stream()
            copy_stream.wait_stream(main)
            with torch.cuda.stream(copy_stream):
                for k, (s0, s1) in self.segs.items():
                    arena[s0:s1].copy_(host_arena[s0:s1], non_blocking=True)
                    seg_ready[k].record()
            main.wait_event(seg_ready["tree"])
            self.L.copy_(self.L0)
            st.run(self.dl, self.roots, self.M_succ, self.M_cnt, self.L, self.Q, self.tl,
                   inputs_ready=lambda k: main.wait_event(seg_ready[k]))
            out_host.copy_(st.acc["out_tok"], non_blocking=True)
            len_host.copy_(st.acc["acc_len"], non_blocking=True)

        body()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            body()

        def one():
            g.replay()
            torch.cuda.current_stream().synchronize()

        for _ in range(3):
            one()
        t0 = time.perf_counter()
        for _ in range(steps):
            one()
        t = time.perf_counter() - t0
        # the same host-to-device copies alone, back to back on the copy stream: the host link's rate on
        # this machine, which bounds how much of them the step can hide
        torch.cuda.synchronize()
        n_copy = 3
        c0 = time.perf_counter()
        for _ in range(n_copy):
            with torch.cuda.stream(copy_stream):
                for k, (s0, s1) in self.segs.items():
                    arena[s0:s1].copy_(host_arena[s0:s1], non_blocking=True)
            copy_stream.synchronize()
        self.h2d_copy_s = (time.perf_counter() - c0) / n_copy
        del g, host_arena
        return t, h2d, d2h

    def acc_len(self):
        return self.step.acc["acc_len"].cpu().tolist()

    def status(self):
        return int(self.step.status.item())

    def release(self):
        import torch
        del self.graph, self.step, self.arena, self.dl, self.tl, self.Q, self.roots, self.L0, self.L
        del self.M_succ, self.M_cnt
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


def workload_report(wb, parts, clocks, sms, t_e2e, n_e2e, h2d, d2h, per_ms=None):
    """The per-workload object: step times, the attention call's roofline, attention + compaction against
    the HBM roofline, tree build and retrieval fill, and the end-to-end step."""
    import torch
    wl = wb.wl
    L0 = wb.L0.cpu()
    rep = {}
    if per_ms:
        q = statistics.quantiles(per_ms, n=10) if len(per_ms) >= 10 else [min(per_ms)] + [float("nan")] * 7 + [max(per_ms)]
        med = statistics.median(per_ms)
        rep.update({"steps_per_s": 1000.0 / med, "step_ms": {"median": med, "p10": q[0], "p90": q[8]},
                    "timed_steps": len(per_ms)})
    if parts is None:  # the parts were not timed
        rep["launches_per_step"] = wb.launches_per_step
        rep["device_status"] = wb.status()
        rep["config"] = workload_config(wl)
        return rep
    t_attn = parts["attention"]
    roof = attention_roofline(wl, L0, t_attn, clocks, sms)
    roof.update({"kernel": "graft_tree_attention (one layer call)", "call_us": t_attn * 1e6,
                 "traffic": recorded_traffic(wl.name)})
    rep["attention"] = roof
    hbm, hbm_kind = measured_peaks()
    b_attn = attention_bytes_per_call(wl, L0) * wl.n_layers
    b_comp = compaction_bytes_per_step(wl, wb.acc_len())
    t_ac = t_attn * wl.n_layers + parts["compaction"]
    rep["attention_compaction"] = {"bound": "hbm", "bytes_per_step": b_attn + b_comp,
                                   "compaction_bytes_per_step": b_comp, "seconds_per_step": t_ac,
                                   "compaction_us": parts["compaction"] * 1e6,
                                   "achieved": (b_attn + b_comp) / t_ac / 1e9, "peak": hbm, "unit": "GB/s",
                                   "frac": (b_attn + b_comp) / t_ac / 1e9 / hbm, "peak_source": f"{hbm_kind} hbm_gbs"}
    rep["build_tree_us"] = parts["tree"] * 1e6
    rep["retrieval_fill_us"] = parts["retrieval"] * 1e6
    if n_e2e > 0 and t_e2e == t_e2e:
        rep["e2e"] = {"value": n_e2e / t_e2e, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        copy_s = getattr(wb, "h2d_copy_s", None)
        if copy_s:
            rep["e2e"]["h2d_copies_alone_ms"] = copy_s * 1e3
            rep["e2e"]["h2d_gbs"] = h2d / copy_s / 1e9
    rep["launches_per_step"] = wb.launches_per_step
    rep["device_status"] = wb.status()
    rep["config"] = workload_config(wl)
    return rep


def run_graft(args):
    import torch
    import torch.distributed as dist
    from tree_verification_gb300 import _build, synth

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    _build.build()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    wl = synth.WORKLOADS[args.workload]
    n_e2e = args.e2e_steps if args.e2e_steps > 0 else (args.steps if args.e2e_steps == 0 else 0)

    # ---------------------------------------------------------------- headline: K timed steps
    wb = WorkloadBench(wl, dev)
    for _ in range(max(3, args.warmup)):
        wb.graph.replay()
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
    t_main, per_step_ms = _timed_steps(wb.graph, args.steps)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    t_max = slowest_over_ranks(t_main, dev, world)
    status = wb.status()
    reps = args.secondary_reps
    parts = wb.parts(reps) if reps > 0 else None
    t_e2e, h2d, d2h = wb.e2e(n_e2e) if n_e2e > 0 else (float("nan"), 0, 0)
    t_e2e = slowest_over_ranks(t_e2e, dev, world)
    head = workload_report(wb, parts, clocks, sms, t_e2e, n_e2e, h2d, d2h, per_step_ms)
    launches = wb.launches_per_step
    cpu_inputs_needed = rank == 0 and world == 1 and not args.no_cpu_baseline
    wb.release()
    del wb

    # ---------------------------------------------------------------- the other workloads' whole steps
    configs = {}
    names = [] if args.configs.strip() in ("", "none") else [x.strip() for x in args.configs.split(",")]
    for name in names:
        if name == wl.name:
            continue
        owl = synth.WORKLOADS[name]
        ob = WorkloadBench(owl, dev)
        ob.graph.replay()
        torch.cuda.synchronize()
        t_one = _timed(ob.graph, 3) / 3
        n = int(min(3000, max(args.steps, 0.5 / max(t_one, 1e-6))))
        _, per = ob.time_steps(n, args.warmup)
        oparts = ob.parts(reps) if reps > 0 else None
        ne = int(min(n, max(args.steps, 0.5 / max(t_one, 1e-6)))) if n_e2e > 0 else 0
        te, oh, od = ob.e2e(ne) if ne > 0 else (float("nan"), 0, 0)
        configs[name] = workload_report(ob, oparts, clocks, sms, te, ne, oh, od, per)
        ob.release()
        del ob

    # ---------------------------------------------------------------- the rest of the line
    lmh = lm_head_timing(wl, dev, reps) if args.secondary_reps > 0 else None
    roof = dict(head["attention"]) if "attention" in head else None
    if roof is not None:
        roof["kernel"] = "graft_tree_attention (one layer call of the headline step)"
    result = {
        "metric": METRIC, "value": world * args.steps / t_max, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1000.0 * t_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(wl, world),
        "roofline": roof,
        "step_ms": head.get("step_ms"),
        "e2e": head.get("e2e"),
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
        "secondary": {"attention_compaction": head.get("attention_compaction"),
                      "retrieval_fill_us": head.get("retrieval_fill_us"), "build_tree_us": head.get("build_tree_us"),
                      "launches_per_step": launches, "device_status": status, "lm_head_argmax": lmh},
        "configs": configs,
    }
    if cpu_inputs_needed:
        inp = oracle_inputs(wl, dev, [0])
        torch.cuda.empty_cache()
        n_req, _ = calibrated_requests(wl, inp, args.cpu_budget_s / 3)
        ests = []
        t0 = time.perf_counter()
        while len(ests) < 3 and (not ests or time.perf_counter() - t0 < args.cpu_budget_s):
            ests.append(oracle_step_sample(wl, inp, list(range(n_req)), 1)[0])
        v = len(ests) / sum(ests)
        result["cpu_baseline"] = {
            "value": v, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": (f"oracle (NumPy, float64 attention): {len(ests)} samples, each the whole tree build, "
                       f"acceptance and M update for all {wl.B} requests, the compaction of 1 of {wl.n_layers} "
                       f"layers and one layer call's attention for {n_req} of {wl.B} requests; the value scales "
                       f"attention by requests and layers and compaction by layers (extrapolated)")}
        del inp
        result["cpu_full_steps"] = cpu_full_steps(budget_s=120.0)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()


def lm_head_timing(wl, dev, reps):
    """The fused lm_head argmax and sampling kernels at this workload's rows (B Kmax), its vocabulary and
    a 4096-wide hidden state, plus sampling from given logits."""
    import torch
    from tree_verification_gb300 import binding as gb
    from tree_verification_gb300 import synth
    H, W_lm = synth.lm_head_inputs(wl, dev)
    N = H.shape[0]
    g_out = torch.empty(N, dtype=torch.int32, device=dev)
    m_out = torch.empty(N, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    lws = torch.empty(max(1, gb.graft_lm_head_argmax_workspace_size(N)), dtype=torch.uint8, device=dev)
    pos = torch.arange(N, dtype=torch.int32, device=dev).view(wl.B, wl.Kmax)
    res = {"rows": N, "d_model": wl.d_model, "vocab": wl.V}
    for name, fn in (("argmax", lambda: gb.graft_lm_head_argmax(H, W_lm, g_out, m_out, status, lws)),
                     ("sample", lambda: gb.graft_lm_head_sample(H, W_lm, pos, 1.0, 1234, sampled=g_out,
                                                                status=status, ws=lws))):
        g = _capture(fn)
        g.replay()
        t = _timed(g, reps) / reps
        res[f"{name}_us"] = t * 1e6
        del g
    flops = 2.0 * N * wl.d_model * wl.V
    nbytes = (H.numel() + W_lm.numel()) * 2 + N * 8
    res["tflops"] = flops / (res["argmax_us"] * 1e-6) / 1e12
    res["gbs"] = nbytes / (res["argmax_us"] * 1e-6) / 1e9
    # sampling from given fp32 logits (the same products, materialised once by torch for the input)
    logits = (H.float() @ W_lm.float().t()).view(wl.B, wl.Kmax, wl.V)
    sampled = torch.empty(wl.B, wl.Kmax, dtype=torch.int32, device=dev)
    sws = torch.empty(max(1, gb.graft_sample_tokens_workspace_size(wl.B, wl.Kmax, wl.V)), dtype=torch.uint8,
                      device=dev)
    g = _capture(lambda: gb.graft_sample_tokens(logits, pos, 1.0, 1234, sampled=sampled, ws=sws))
    g.replay()
    t = _timed(g, reps) / reps
    res["sample_tokens_us"] = t * 1e6
    res["sample_tokens_gbs"] = logits.numel() * 4 / t / 1e9  # the logits, read once
    del g, logits
    del H, W_lm
    torch.cuda.empty_cache()
    return res


def run_attention(args):
    """--mode attention: microseconds per graft_tree_attention call of a workload (distinct buffers per
    layer so calls stream from DRAM; the layer calls captured in one CUDA graph); one JSON line."""
    import numpy as np
    import torch
    from tree_verification_gb300 import _build, synth
    from tree_verification_gb300 import binding as gb
    _build.build()
    dev = torch.device("cuda")
    wl = synth.WORKLOADS[args.workload]
    Lcap = max(args.lcap, wl.lcap()) if args.lcap else wl.lcap()
    L = synth.prefix_lengths(wl).to(dev)
    layers = [synth.layer_tensors(wl, l, dev, Lcap=Lcap) for l in range(args.layers)]
    chain = np.array([[(1 << (i + 1)) - 1 for i in range(wl.Kmax)]] * wl.B, dtype=np.uint64)
    mask = torch.from_numpy(chain.view(np.int64)).to(dev)
    ws = torch.zeros(max(1, gb.graft_tree_attention_workspace_size(wl.B, wl.Hq, wl.Hkv, wl.Kmax, Lcap)),
                     dtype=torch.uint8, device=dev)
    O = torch.empty_like(layers[0][0])
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    scale = 1.0 / math.sqrt(gb.HEAD_DIM)

    def run():
        for (Q, Kc, Vc, Kt, Vt) in layers:
            gb.graft_tree_attention(Q, Kc, Vc, Kt, Vt, L, mask, scale, O=O, ws=ws, status=status)

    g = _capture(run)
    for _ in range(3):
        g.replay()
    us = _timed(g, args.reps) * 1e6 / (args.reps * args.layers)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    r = attention_roofline(wl, L.cpu(), us * 1e-6, None, sms)
    print(json.dumps({"mode": "attention", "workload": wl.name, "layers": args.layers, "lcap": Lcap, "call_us": us,
                      "bytes_per_call": r["bytes_per_call"], "gbs": r["bytes_per_call"] / us / 1e3,
                      "bound": r["bound"], "frac": r["frac"], "fractions": r["fractions"],
                      "status": int(status.item())}), flush=True)


def run_lm_head(args):
    """--mode lm_head: the fused lm_head argmax / sampling kernels on H [rows][d_model] and W [vocab][d_model]
    bf16 N(0,1); one JSON line."""
    import torch
    from tree_verification_gb300 import _build, synth
    _build.build()
    dev = torch.device("cuda")
    kmax = 64 if args.rows % 64 == 0 else args.rows
    wl = synth.WORKLOADS["llama3_8b"].scaled(B=args.rows // kmax, Kmax=kmax, V=args.vocab, d_model=args.d_model)
    res = lm_head_timing(wl, dev, args.reps)
    print(json.dumps(dict(mode="lm_head", **res)), flush=True)


def run_tree(args):
    """--mode tree: microseconds per graft_build_tree call of a workload (the calls captured in one CUDA
    graph, the workspace zero-filled once); one JSON line with the stages the calls reached."""
    import torch
    from tree_verification_gb300 import _build, synth
    from tree_verification_gb300 import binding as gb
    _build.build()
    dev = torch.device("cuda")
    wl = synth.WORKLOADS[args.workload]
    cfg = gb.graft_config_init(wl.Kmax, wl.D, wl.k, wl.V, wl.W, list(wl.checkpoints), wl.tau)
    dl = synth.draft_logits(wl, dev) if args.drafts == "flat" else synth.peaked_draft_logits(wl, dev, [12.0] * wl.B)
    roots, L = synth.root_tokens(wl).to(dev), synth.prefix_lengths(wl).to(dev)
    s_np, _ = synth.zipf_M(wl.V, wl.W, wl.seed + 5) if wl.M_init == "zipf" else synth.empty_M(wl.V, wl.W)
    M_succ = torch.from_numpy(s_np).to(dev)
    ws = torch.zeros(max(1, gb.graft_build_tree_workspace_size(cfg, wl.B)), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = gb.graft_build_tree(cfg, dl, roots, M_succ, L, ws=ws, status=status)
    n_rep = 20

    def run():
        for _ in range(n_rep):
            gb.graft_build_tree(cfg, dl, roots, M_succ, L, out=out, ws=ws, status=status)

    g = _capture(run)
    for _ in range(3):
        g.replay()
    us = _timed(g, args.reps) * 1e6 / (args.reps * n_rep)
    torch.cuda.synchronize()
    print(json.dumps({"mode": "tree", "workload": wl.name, "drafts": args.drafts, "batch": wl.B, "vocab": wl.V,
                      "call_us": us, "stages": sorted(set(out["stage"].cpu().tolist())),
                      "status": int(status.item())}), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.mode == "cpu_step":
        run_cpu_step(args)
    elif args.mode == "attention":
        run_attention(args)
    elif args.mode == "lm_head":
        run_lm_head(args)
    elif args.mode == "tree":
        run_tree(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_graft(args)


if __name__ == "__main__":
    main()
