"""Benchmark of the STILL layer on GB300: one JSON line.

A step is one chunk-parallel prefill forward of the Llama-3-8B-shaped layer at
16K context (B=1, 32 query / 8 kv heads, d = d_f = 128, W=64, C=256, m=288,
T_max=64, lambda=3): score -> select -> linear state -> hybrid attention, all
in libstill's kernels, on seeded synthetic inputs resident in HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

The headline steps run as a caller runs them (one CUDA event pair per step);
a second pass of the same steps with an event pair around every kernel gives
the per-kernel times and the roofline of the dominant kernel.  Further legs:
end to end through pinned host buffers, the 128-sequence decode step, the
routing metrics of the ablation (score kernel per metric and the layer routed
by it), the other prefill workloads (the Llama-3.2-1B-shaped layer at 4K and
the training-shaped batch of eight 1K sequences, each with its roofline, its
CPU-oracle time and its parity), and the CPU oracle on the 16K layer with the
parity of the benchmarked output against it.

Under torchrun (N > 1) every rank runs its own layer (its own seed): weak
scaling, no collective on the data path; value = all ranks' tokens / the max
over ranks of the timed region.  --impl reference times the CPU oracle (the
fp64 streaming recurrence) on the host cores instead; with N > 1 only rank 0
runs it.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "llama3_8b_layer_prefill_16k"
DECODE_WORKLOAD = "llama31_8b_decode_b128_ctx16k"
METRIC = "prefill tokens/s on 1 GB300 (16K, Llama-3-8B layer); % of BF16/HBM roofline"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=500)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-decode", action="store_true", help="skip the decode-step measurement")
    p.add_argument("--decode-seqs", type=int, default=0,
                   help="sequences of the decode workload (default: the workload's 128); a smaller batch "
                        "keeps an ncu capture of the decode kernel to a few GB of device memory")
    p.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    p.add_argument("--no-routing", action="store_true", help="skip the routing-metric measurements")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the 1B-shaped 4K and training-shaped prefill legs")
    p.add_argument("--no-backward", action="store_true", help="skip the backward-pass leg (training-shaped batch)")
    p.add_argument("--cpu-tokens", type=int, default=16384, help="tokens of the CPU-baseline sample")
    p.add_argument("--seed", type=int, default=0)
    return p.parse_args(argv)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# algorithmic work (what the method must do; no padded or masked work)
# ---------------------------------------------------------------------------

def algorithmic(w, sel_idx):
    """FLOPs and bytes of one prefill, the selection counted exactly."""
    import numpy as np
    N, d, df, Hq, Hkv, B = w.N, w.d, w.df, w.Hq, w.Hkv, w.B
    t = np.arange(N)
    win = np.minimum(t + 1, w.W).astype(np.float64)
    # kept tokens visible to query t: chunk(j) < chunk(t) and j <= t - W
    sel = sel_idx.reshape(B, Hkv, -1)
    n_sa_sel = 0.0
    la_keys = 0.0
    for b in range(B):
        for g in range(Hkv):
            s = np.sort(sel[b, g][sel[b, g] >= 0])
            ct = t // w.C
            # per query: count kept j with j // C < ct and j <= t - W
            lim_chunk = np.searchsorted(s // w.C, ct, side="left")       # kept in earlier chunks
            lim_pos = np.searchsorted(s, t - w.W, side="right")          # kept with j <= t - W
            vis = np.minimum(lim_chunk, lim_pos)
            n_sa_sel += vis.sum()
            la_keys += N - w.W - len(s) if N > w.W else 0
    sa_keys = Hq * B * win.sum() + (Hq // Hkv) * n_sa_sel
    F_score = 2.0 * d * Hq * B * win.sum()
    F_feat = 2.0 * d * df * (Hq + Hkv) * B * N
    F_fold = 2.0 * df * d * la_keys
    F_read = 2.0 * df * (d + 1) * Hq * B * N
    F_sa = 4.0 * d * sa_keys
    bytes_io = 2.0 * B * N * d * (2 * Hq + 2 * Hkv) + 4.0 * d * df
    return dict(F_score=F_score, F_feat=F_feat, F_fold=F_fold, F_readout=F_read, F_sa=F_sa,
                flops=F_score + F_feat + F_fold + F_read + F_sa, bytes=bytes_io,
                attn_flops=F_sa + F_read + 2.0 * d * df * Hq * B * N,
                mean_sa_keys=sa_keys / (Hq * B * N))


def kernel_bytes(w):
    """Algorithmic HBM bytes per launch of each kernel."""
    B, N, d, df, Hq, Hkv = w.B, w.N, w.d, w.df, w.Hq, w.Hkv
    q = 2.0 * B * Hq * N * d
    kv = 2.0 * B * Hkv * N * d
    return {"hybrid_attn": 2 * q + 2 * kv, "score": q + kv + 4.0 * B * Hkv * N,
            "features_linstate": 2 * kv, "select": 4.0 * B * Hkv * N, "scan": 0.0}


def profile_traffic(kernel):
    """dram bytes per launch from the committed ncu summary, if it was taken
    from the current source of that kernel's file."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    src_of = {"hybrid_attn": "hybrid_tc.cu", "score": "score_tc.cu", "select": "score_select.cu",
              "prep": "features.cu", "features_linstate": "linstate_tc.cu", "scan": "linstate.cu",
              "decode_step": "decode.cu"}
    f = src_of.get(kernel)
    if not f:
        return None
    sha = hashlib.sha256(open(os.path.join(ROOT, "linear_attention_linearization_gb300", "csrc", f),
                              "rb").read()).hexdigest()[:16]
    for line in open(path):
        m = re.match(r"\s*(\w+)\s+sha=(\w+)\s+bytes_per_launch=([0-9.eE+]+)", line)
        if m and m.group(1) == kernel and m.group(2) == sha:
            return float(m.group(3))
    return None


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle
# ---------------------------------------------------------------------------

def oracle_sample(q, k, v, Wf, w, tokens, threads, keep=None, gate=None):
    """Run the fp64 streaming oracle over `tokens` tokens of every kv head; the
    time it took.  With a dict `keep`, the oracle's output and scores are
    stored there (key "y", "scores") for the parity check."""
    from linear_attention_linearization_gb300.inputs import to_f64
    from oracle import ref
    qa = to_f64(q[:, :, :tokens])
    ka = to_f64(k[:, :, :tokens])
    va = to_f64(v[:, :, :tokens])
    Wa = to_f64(Wf)
    t0 = time.perf_counter()
    ga = to_f64(gate[:, :, :tokens]) if gate is not None else None
    y, sc, _ = ref.prefill(qa, ka, va, Wa, w.W, w.C, w.m, w.T_max, threads=threads, gate=ga)
    secs = time.perf_counter() - t0
    if keep is not None:
        keep.update(y=y, scores=sc, inputs=(qa, ka, va, Wa), gate=ga)
    return secs


def parity_vs_oracle(out, sel, w, toks, keep, threads):
    """The benchmarked layer's output and selection against the oracle's run of
    the CPU-baseline leg on the same inputs (tokens 0..toks-1): the largest
    output error relative to the largest oracle output; selected sets exact
    outside near-tie chunks (lambda-th and (lambda+1)-th oracle scores within
    1e-5 relative), where the GPU's set must be a valid top-lambda and the
    oracle is re-run with it."""
    import numpy as np
    from linear_attention_linearization_gb300.inputs import to_f64
    from oracle import brute, ref
    y_ref, sc = keep["y"], keep["scores"]
    sel_g = sel.cpu().numpy()
    n_ties = n_diff = 0
    exact_outside = True
    n_chunks = min(toks // w.C, w.T_max)
    for b in range(w.B):
        ties = set(brute.near_ties(sc[b], w.C, w.lam, w.T_max))
        n_ties += len(ties)
        sref = brute.select(sc[b], w.C, w.lam, w.T_max)
        for g, c in np.argwhere((sel_g[b, :, :n_chunks] != sref[:, :n_chunks]).any(axis=-1)):
            n_diff += 1
            if (g, c) not in ties:
                exact_outside = False
    if n_diff and exact_outside and toks == w.N:
        qa, ka, va, Wa = keep["inputs"]
        y_ref, _, _ = ref.prefill(qa, ka, va, Wa, w.W, w.C, w.m, w.T_max, sel_override=sel_g, threads=threads,
                                  gate=keep.get("gate"))
    y = to_f64(out[:, :, :toks])
    err = float(np.abs(y - y_ref).max() / np.abs(y_ref).max())
    return {"max_err_rel": err, "tolerance": 1e-2, "within_tolerance": err <= 1e-2,
            "near_tie_chunks": n_ties, "sel_differs_in_near_ties": n_diff if exact_outside else None,
            "sel_exact_outside_ties": exact_outside,
            "compared": f"every output element and selected index of tokens 0..{toks - 1}, all heads"}


def cpu_threads(units):
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(n, units))


def cpu_baseline(q, k, v, Wf, w, toks, gate=None):
    """The oracle on the host cores over tokens 0..toks-1 of every kv head (one
    thread per kv head), and on one core: the first kv head with its query
    heads on one thread, its time scaled by the number of kv heads and
    sequences (the units are independent and cost the same)."""
    thr = cpu_threads(w.B * w.Hkv)
    keep = {}
    secs = oracle_sample(q, k, v, Wf, w, toks, thr, keep, gate=gate)
    G = w.Hq // w.Hkv
    w1 = dataclasses.replace(w, B=1, Hq=G, Hkv=1)
    secs1 = oracle_sample(q[:1, :G], k[:1, :1], v[:1, :1], Wf, w1, toks, 1) * w.B * w.Hkv
    return {"value": w.B * toks / secs, "unit": "tokens/s", "cores": thr, "kind": "oracle",
            "sample": f"fp64 streaming oracle over tokens 0..{toks - 1} of all {w.Hkv} kv heads "
                      f"({w.Hq} query heads) of the same inputs, one thread per kv head",
            "seconds": secs,
            "one_core": {"value": w.B * toks / secs1, "unit": "tokens/s", "cores": 1,
                         "sample": f"kv head 0 of sequence 0 with its {G} query heads over the same tokens on one "
                                   f"thread, time x {w.B * w.Hkv} units"}}, keep, thr


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def reduce_max(pg, x, device):
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def aggregate(pg, seconds, tokens_per_rank, steps, device):
    """Whole-job throughput of `steps` timed steps: every rank processes
    `tokens_per_rank` tokens per step; the job takes as long as its slowest
    rank.  Returns (tokens/s over all ranks, ms per step, slowest seconds)."""
    world = pg.get_world_size() if pg is not None else 1
    t_max = reduce_max(pg, seconds, device)
    return world * tokens_per_rank * steps / t_max, 1e3 * t_max / steps, t_max


def run_reference(args):
    world, rank, local, pg = dist_setup()
    if rank != 0:
        return
    import torch
    from linear_attention_linearization_gb300 import inputs
    w = inputs.WORKLOADS[WORKLOAD]
    tokens = 1024
    q, k, v, Wf = inputs.make_inputs(w, seed=args.seed, N=tokens)
    thr = cpu_threads(w.B * w.Hkv)
    for _ in range(args.warmup):
        oracle_sample(q, k, v, Wf, w, tokens, thr)
    total = 0.0
    for _ in range(args.steps):
        total += oracle_sample(q, k, v, Wf, w, tokens, thr)
    tps = tokens * args.steps / total
    sample = (f"fp64 streaming oracle, all {w.Hkv} kv heads x {w.Hq} query heads, tokens 0..{tokens - 1} of the "
              f"16K layer per step (early tokens see fewer kept keys than the layer average)")
    line = {"impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, **w.asdict()},
            "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": thr, "kind": "oracle", "sample": sample},
            "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    del torch


def run_ours(args):
    import torch
    from linear_attention_linearization_gb300 import build, inputs
    build.build()
    from linear_attention_linearization_gb300 import still

    world, rank, local, pg = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = inputs.WORKLOADS[WORKLOAD]
    seed = args.seed + 1000 * rank
    q, k, v, Wf = inputs.make_inputs(w, seed=seed, device=dev)
    out = torch.empty_like(q)
    lam = w.lam
    sel = torch.empty((w.B, w.Hkv, w.T_max, lam), dtype=torch.int32, device=dev)
    ws = torch.empty(still.workspace_size(q, k, Wf, w.W, w.C, w.m, w.T_max), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        still.prefill(q, k, v, Wf, w.W, w.C, w.m, w.T_max, out=out, sel_idx=sel, workspace=ws, stream=stream)

    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    with ClockSampler(local) as clk:
        for _ in range(max(3, args.warmup)):
            step()
        torch.cuda.synchronize(dev)
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        # the headline: the step as a caller runs it (the library's per-kernel
        # timers put an event between launches, which would serialise the
        # programmatic dependent launches; they run in a second pass below)
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(float(i))              # evict the previous step's data from L2
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
        if pg is not None:
            pg.barrier()
    # the same steps again with a CUDA event pair around every kernel: the
    # per-kernel times and the roofline of the dominant kernel
    still.timing_read()
    still.timing_enable(True)
    ev_k = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(float(i))
        ev_k[i][0].record(stream)
        step()
        ev_k[i][1].record(stream)
    torch.cuda.synchronize(dev)
    still.timing_enable(False)
    ktimes = still.timing_read()
    step_ms_timed_kernels = statistics.mean(a.elapsed_time(b) for a, b in ev_k)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    t_total = sum(step_ms) / 1e3
    value, ms_per_step, t_max = aggregate(pg, t_total, w.B * w.N, args.steps, dev)

    # -------- roofline of the dominant kernel --------
    pk, pk_kind = peaks()
    alg = algorithmic(w, sel.cpu().numpy())
    kb = kernel_bytes(w)
    dom = max(ktimes.items(), key=lambda kv: kv[1][1])[0] if ktimes else None
    launches = sum(n for n, _ in ktimes.values())
    roof = None
    if dom:
        n, ms = ktimes[dom]
        per = ms / n / 1e3
        if dom == "hybrid_attn":
            t_hbm = kb[dom] / (pk["hbm_gbs"] * 1e9)
            t_flop = alg["attn_flops"] / (pk["bf16_tflops"] * 1e12)
            bound = "hbm" if t_hbm >= t_flop else "tensor"
        else:
            bound = "hbm"
        if bound == "hbm":
            ach = kb.get(dom, 0.0) / per / 1e9
            peak_v, unit = pk["hbm_gbs"], "GB/s"
        else:
            ach = alg["attn_flops"] / per / 1e12
            peak_v, unit = pk["bf16_tflops"], "TFLOP/s"
        roof = {"kernel": dom, "bound": bound, "achieved": ach, "peak": peak_v, "unit": unit,
                "frac": ach / peak_v, "peak_source": pk_kind, "traffic": profile_traffic(dom),
                "algorithmic_bytes_per_launch": kb.get(dom), "algorithmic_flops_per_launch": alg["attn_flops"],
                "launch_ms": per * 1e3}
    step_roof_s = max(alg["flops"] / (pk["bf16_tflops"] * 1e12), alg["bytes"] / (pk["hbm_gbs"] * 1e9))

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, **w.asdict(), "l2": "L2 flushed (258 MB write) before every timed "
                       "step; working set 336 MB > 129 MB L2", "parallelism": f"replicas x{world}"},
            "roofline": roof,
            "step_roofline": {"algorithmic_flops": alg["flops"], "algorithmic_bytes": alg["bytes"],
                              "roofline_ms": step_roof_s * 1e3, "frac_of_roofline": step_roof_s * 1e3 / ms_per_step,
                              "mean_softmax_keys_per_query": alg["mean_sa_keys"], "peak_source": pk_kind},
            "kernels": {k2: {"launches": n, "ms_per_launch": ms / n} for k2, (n, ms) in ktimes.items()},
            # the kernel pass runs the same steps through the same path, so it
            # launches what the headline pass did
            "gpu_launches": launches, "wall_s_timed_region": wall,
            "ms_per_step_with_kernel_timers": step_ms_timed_kernels,
            "clocks": clk.summary()}

    # -------- end to end through host buffers --------
    # Every step copies its inputs from pinned host memory and reads its output
    # and selection back, inside the timed region.  The three parts run on
    # their own streams so that step i+1's upload, step i's layer and step
    # i-1's download overlap (device inputs and outputs double-buffered, events
    # guarding each buffer's reuse), as a caller streaming layers would run it.
    if not args.no_e2e:
        hq = q.cpu().pin_memory()
        hk = k.cpu().pin_memory()
        hv = v.cpu().pin_memory()
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hsel = torch.empty(sel.shape, dtype=sel.dtype).pin_memory()
        dins = [(torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)) for _ in range(2)]
        douts = [(torch.empty_like(out), torch.empty_like(sel)) for _ in range(2)]
        s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("up", "comp", "down")}
        used = [False, False]

        def e2e_step(i):
            bi = i % 2
            dq, dk, dv = dins[bi]
            dout, dsel = douts[bi]
            with torch.cuda.stream(s_up):
                if used[bi]:
                    s_up.wait_event(ev["comp"][bi])     # the layer of step i-2 has read these inputs
                dq.copy_(hq, non_blocking=True)
                dk.copy_(hk, non_blocking=True)
                dv.copy_(hv, non_blocking=True)
                ev["up"][bi].record(s_up)
            stream.wait_event(ev["up"][bi])
            if used[bi]:
                stream.wait_event(ev["down"][bi])       # step i-2's output has been read back
            still.prefill(dq, dk, dv, Wf, w.W, w.C, w.m, w.T_max, out=dout, sel_idx=dsel, workspace=ws,
                          stream=stream)
            ev["comp"][bi].record(stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(ev["comp"][bi])
                hout.copy_(dout, non_blocking=True)
                hsel.copy_(dsel, non_blocking=True)
                ev["down"][bi].record(s_down)
            used[bi] = True

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        n_e2e = max(3, min(args.steps, 20))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_up)
        for i in range(n_e2e):
            e2e_step(3 + i)
        b.record(s_down)
        torch.cuda.synchronize(dev)
        v_e2e, _, _ = aggregate(pg, a.elapsed_time(b) / 1e3, w.B * w.N, n_e2e, dev)
        line["e2e"] = {"value": v_e2e, "unit": "tokens/s",
                       "h2d_bytes_per_step": int(hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2),
                       "d2h_bytes_per_step": int(hout.numel() * 2 + hsel.numel() * 4), "steps": n_e2e,
                       "overlap": "upload, layer and download on three streams, double-buffered"}

    # -------- routing metrics of the ablation (16K layer) --------
    if not args.no_routing and rank == 0:
        line["routing_metrics"] = bench_routing(still, w, (q, k, v, Wf), dev, stream, pk, pk_kind)

    # -------- the other prefill workloads --------
    if not args.no_backward and rank == 0:
        line["backward"] = bench_backward(still, dev, stream, pk, pk_kind, args.seed + 13, cpu=not args.no_cpu)
        line["backward_llama32_1b_layer_prefill_4k"] = bench_backward(
            still, dev, stream, pk, pk_kind, args.seed + 14, cpu=not args.no_cpu, name="llama32_1b_layer_prefill_4k")
    if not args.no_workloads and rank == 0:
        line["workloads"] = {nm: bench_workload(still, nm, dev, stream, pk, pk_kind, args.seed + 11,
                                                cpu=not args.no_cpu)
                             for nm in ("llama32_1b_layer_prefill_4k", "train_b8_n1k_chunk_parallel")}
        line["workloads"]["llama3_8b_layer_prefill_16k_gated"] = bench_workload(
            still, WORKLOAD, dev, stream, pk, pk_kind, args.seed + 12, steps=20, cpu=not args.no_cpu, gated=True)

    # -------- decode step (128 sequences at 16K) --------
    if not args.no_decode and rank == 0:
        line["decode_step"] = bench_decode(still, inputs, dev, stream, pk, pk_kind, args)

    # -------- CPU oracle baseline --------
    if not args.no_cpu and rank == 0 and world == 1:
        toks = min(args.cpu_tokens, w.N)
        line["cpu_baseline"], keep, thr = cpu_baseline(q.cpu(), k.cpu(), v.cpu(), Wf.cpu(), w, toks)
        # the last timed step's output against that oracle run (outside the timed regions)
        line["parity"] = parity_vs_oracle(out, sel, w, toks, keep, thr)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def bench_routing(still, w, qkvw, dev, stream, pk, pk_kind, launches=10):
    """Each routing metric's score kernel on the 16K layer (library event timers,
    L2 flushed before every launch) against its algorithmic bytes, and the whole
    layer routed by it (CUDA events around the call)."""
    import torch
    q, k, v, Wf = qkvw
    qb, kb, sb = 2.0 * w.B * w.Hq * w.N * w.d, 2.0 * w.B * w.Hkv * w.N * w.d, 4.0 * w.B * w.Hkv * w.N
    need = {"diagonal": qb + kb, "qk": qb + kb, "key_norm": kb, "uniform": 0.0, "random": 0.0}
    scores = torch.empty((w.B, w.Hkv, w.N), dtype=torch.float32, device=dev)
    out = torch.empty_like(q)
    sel = torch.empty((w.B, w.Hkv, w.T_max, w.lam), dtype=torch.int32, device=dev)
    ws = torch.empty(still.workspace_size(q, k, Wf, w.W, w.C, w.m, w.T_max), dtype=torch.uint8, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    res = {}
    for metric, inb in need.items():
        for i in range(3):
            still.score_metric(q, k, w.W, w.C, w.m, w.T_max, metric, seed=i, scores=scores, stream=stream)
        torch.cuda.synchronize(dev)
        still.timing_read()
        still.timing_enable(True)
        for i in range(launches):
            flush.fill_(float(i))
            still.score_metric(q, k, w.W, w.C, w.m, w.T_max, metric, seed=i, scores=scores, stream=stream)
        torch.cuda.synchronize(dev)
        still.timing_enable(False)
        t = still.timing_read()
        n, ms = t.get("routing_metric", t.get("score", (0, 0.0)))
        per = ms / max(n, 1) / 1e3
        by = inb + sb
        ach = by / per / 1e9
        pre = []
        for i in range(5):
            flush.fill_(float(i))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            still.prefill_routed(q, k, v, Wf, w.W, w.C, w.m, w.T_max, metric, seed=i, out=out, sel_idx=sel,
                                 workspace=ws, stream=stream)
            b.record(stream)
            pre.append((a, b))
        torch.cuda.synchronize(dev)
        res[metric] = {"ms_per_launch": per * 1e3, "launches": n, "algorithmic_bytes": by,
                       "roofline": {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                                    "frac": ach / pk["hbm_gbs"], "peak_source": pk_kind},
                       "routed_prefill_ms": statistics.median(a.elapsed_time(b) for a, b in pre[2:])}
    return res


def bench_workload(still, name, dev, stream, pk, pk_kind, seed, steps=50, cpu=True, gated=False):
    """Another prefill workload of the pages' set (the 1B-shaped layer at 4K, the
    training-shaped batch of eight 1K sequences): `steps` timed prefills after 3
    warm-up ones, L2 flushed before each (CUDA events around every call), the
    step against its roofline, the kernels' times from a second pass with the
    library's event timers, and -- unless cpu is False -- the oracle over the
    whole workload on the host cores and the parity of the GPU's output with it.
    gated: the layer with the per-channel sigmoid gate on the linear branch
    (still_prefill_gated), its pre-activations drawn by inputs.make_gate."""
    import torch
    from linear_attention_linearization_gb300 import inputs
    w = inputs.WORKLOADS[name]
    q, k, v, Wf = inputs.make_inputs(w, seed=seed, device=dev)
    gate = inputs.make_gate(w, seed=seed, device=dev) if gated else None
    out = torch.empty_like(q)
    sel = torch.empty((w.B, w.Hkv, w.T_max, w.lam), dtype=torch.int32, device=dev)
    ws = torch.empty(still.workspace_size(q, k, Wf, w.W, w.C, w.m, w.T_max), dtype=torch.uint8, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def step():
        if gated:
            still.prefill_gated(q, k, v, gate, Wf, w.W, w.C, w.m, w.T_max, out=out, sel_idx=sel, workspace=ws,
                                stream=stream)
        else:
            still.prefill(q, k, v, Wf, w.W, w.C, w.m, w.T_max, out=out, sel_idx=sel, workspace=ws, stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    ev = []
    for i in range(steps):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        ev.append((a, b))
    torch.cuda.synchronize(dev)
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    still.timing_read()
    still.timing_enable(True)
    for i in range(10):
        flush.fill_(float(i))
        step()
    torch.cuda.synchronize(dev)
    still.timing_enable(False)
    kt = still.timing_read()
    alg = algorithmic(w, sel.cpu().numpy())
    t_roof = max(alg["flops"] / (pk["bf16_tflops"] * 1e12), alg["bytes"] / (pk["hbm_gbs"] * 1e9))
    kb = kernel_bytes(w)
    att_name = "hybrid_attn_gated" if gated else "hybrid_attn"
    n_att, ms_att = kt.get(att_name, (0, 0.0))
    att = None
    if n_att:
        per = ms_att / n_att / 1e3
        by = kb["hybrid_attn"] + (2.0 * w.B * w.Hq * w.N * w.d if gated else 0.0)   # + the gate read once
        att = {"ms_per_launch": per * 1e3, "achieved": by / per / 1e9, "peak": pk["hbm_gbs"], "algorithmic_bytes": by,
               "unit": "GB/s", "frac": by / per / 1e9 / pk["hbm_gbs"], "bound": "hbm", "peak_source": pk_kind}
    res = {"config": {"workload": name, **w.asdict()}, "metric": "prefill tokens/s", "unit": "tokens/s",
           "value": w.B * w.N / (ms / 1e3), "ms_per_step": ms, "steps": steps,
           "l2": "flushed (258 MB write) before every timed step",
           "step_roofline": {"algorithmic_flops": alg["flops"], "algorithmic_bytes": alg["bytes"],
                             "roofline_ms": t_roof * 1e3, "frac_of_roofline": t_roof * 1e3 / ms, "peak_source": pk_kind},
           "attention_roofline": att,
           "kernels": {k2: {"launches": n, "ms_per_launch": m / n} for k2, (n, m) in kt.items()},
           "attention_on_tensor_cores": att_name in kt and not any(n.startswith("hybrid_attn_general") for n in kt)}
    if gated:
        res["layer"] = "gated: per-channel sigmoid gate on the linear branch's numerator"
    if cpu:
        toks = w.N
        if gated:
            res["cpu_baseline"], keep, thr = cpu_baseline(q.cpu(), k.cpu(), v.cpu(), Wf.cpu(), w, toks,
                                                          gate=gate.cpu())
        else:
            res["cpu_baseline"], keep, thr = cpu_baseline(q.cpu(), k.cpu(), v.cpu(), Wf.cpu(), w, toks)
        res["parity"] = parity_vs_oracle(out, sel, w, toks, keep, thr)
    return res


BACKWARD_WORKLOAD = "train_b8_n1k_chunk_parallel"


def backward_algorithmic(w, sel_idx):
    """Algorithmic work of one backward pass (routing fixed): per softmax pair
    (t, j) the logit recomputation and the four gradient contractions (dP, dq,
    dk, dv: 2d flops each), per query row phi(q) S for y, S g for dphi(q) and
    its share of the reverse state sum phi(q) g^T, per linear key phi(k) v^T
    for the forward state, R v and R^T phi(k), per q and k row the NP-Map
    (x Wf, dl Wf^T, x dl^T); bytes: q, k, v, dy read once (bf16), dq, dk, dv
    written once (fp32), Wf read and dWf written."""
    a = algorithmic(w, sel_idx)
    N, d, df, Hq, Hkv, B = w.N, w.d, w.df, w.Hq, w.Hkv, w.B
    sa_keys = a["mean_sa_keys"] * Hq * B * N
    kept = float((sel_idx >= 0).sum())
    rows_q, rows_k = Hq * B * N, Hkv * B * N
    lin_keys = max(rows_k - kept - Hkv * B * w.W, 0.0)
    F_soft = 10.0 * d * sa_keys
    F_lin = 3 * 2.0 * df * d * rows_q + 3 * 2.0 * df * d * lin_keys
    F_np = 6.0 * d * df * (rows_q + rows_k)
    by = 2.0 * d * (2 * rows_q + 2 * rows_k) + 4.0 * d * (rows_q + 2 * rows_k) + 8.0 * d * df
    return {"flops": F_soft + F_lin + F_np, "F_softmax": F_soft, "F_linear": F_lin, "F_npmap": F_np, "bytes": by}


def bench_backward(still, dev, stream, pk, pk_kind, seed, steps=20, cpu=True, name=BACKWARD_WORKLOAD):
    """The backward pass (still_backward, routing held fixed) of a workload (the
    training-shaped batch by default): `steps` timed calls after 3 warm-up ones, L2 flushed
    before each (CUDA events around every call), the step against its roofline,
    its kernels' times from the library's event timers, and -- unless cpu is
    False -- the gradient oracle on one sequence of the batch on the host
    cores, with the parity of the GPU's dq, dk, dv for that sequence."""
    import numpy as np
    import torch
    from linear_attention_linearization_gb300 import inputs
    from linear_attention_linearization_gb300.inputs import to_f64
    w = inputs.WORKLOADS[name]
    q, k, v, Wf = inputs.make_inputs(w, seed=seed, device=dev)
    dy = inputs.make_dout(w, seed=seed, device=dev)
    _, sel = still.prefill(q, k, v, Wf, w.W, w.C, w.m, w.T_max, stream=stream)
    grads = (torch.empty(q.shape, dtype=torch.float32, device=dev), torch.empty(k.shape, dtype=torch.float32, device=dev),
             torch.empty(v.shape, dtype=torch.float32, device=dev), torch.empty(Wf.shape, dtype=torch.float32, device=dev))
    ws = torch.empty(still.backward_workspace_size(q, k, Wf, w.W, w.C, w.m, w.T_max), dtype=torch.uint8, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def step():
        still.backward(q, k, v, Wf, w.W, w.C, w.m, w.T_max, sel, dy, grads=grads, workspace=ws, stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    ev = []
    for i in range(steps):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        ev.append((a, b))
    torch.cuda.synchronize(dev)
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    still.timing_read()
    still.timing_enable(True)
    for i in range(5):
        flush.fill_(float(i))
        step()
    torch.cuda.synchronize(dev)
    still.timing_enable(False)
    kt = still.timing_read()
    sel_h = sel.cpu().numpy()
    alg = backward_algorithmic(w, sel_h)
    t_flop = alg["flops"] / (pk["bf16_tflops"] * 1e12)
    t_hbm = alg["bytes"] / (pk["hbm_gbs"] * 1e9)
    res = {"config": {"workload": w.name, **w.asdict()}, "metric": "backward tokens/s", "unit": "tokens/s",
           "value": w.B * w.N / (ms / 1e3), "ms_per_step": ms, "steps": steps, "dtype": "bf16 operands, fp32 gradients",
           "l2": "flushed (258 MB write) before every timed step",
           "roofline": {"bound": "tensor" if t_flop >= t_hbm else "hbm", "algorithmic_flops": alg["flops"],
                        "algorithmic_bytes": alg["bytes"], "roofline_ms": max(t_flop, t_hbm) * 1e3,
                        "achieved_tflops": alg["flops"] / (ms / 1e3) / 1e12, "peak_tflops": pk["bf16_tflops"],
                        "frac": max(t_flop, t_hbm) * 1e3 / ms, "peak_source": pk_kind,
                        "split": {k2: alg[k2] for k2 in ("F_softmax", "F_linear", "F_npmap")}},
           "kernels": {k2: {"launches": n, "ms_per_launch": m / n} for k2, (n, m) in kt.items()},
           "gpu_launches_per_step": 10 + (1 if w.W < w.C else 0)}
    if cpu:
        from oracle import grad
        torch_threads = torch.get_num_threads()
        # the sample: sequence 0 and its first two kv heads (with their query heads); the kv
        # heads are independent units, so the tokens/s of the sample scales to the batch
        nkv = min(2, w.Hkv)
        nq = nkv * (w.Hq // w.Hkv)
        hq, hdy = (to_f64(t[:1, :nq]) for t in (q, dy))
        hk, hv = (to_f64(t[:1, :nkv]) for t in (k, v))
        hW = to_f64(Wf)
        cidx = torch.empty((w.B, w.Hq, w.N), dtype=torch.int32, device=dev)
        still.backward(q, k, v, Wf, w.W, w.C, w.m, w.T_max, sel, dy, grads=grads, cmax_idx=cidx, workspace=ws,
                       stream=stream)
        torch.cuda.synchronize(dev)
        sel_s = sel_h[:1, :nkv]
        t0 = time.perf_counter()
        _, dq_r, dk_r, dv_r, _, c_r = grad.layer_grad(hq, hk, hv, hW, w.W, w.C, sel_s, hdy)
        sec = time.perf_counter() - t0
        c_g = cidx[:1, :nq].cpu().numpy().astype(np.int64)
        moved = int((c_g != c_r).sum())
        if moved:   # near-equal row maxima: the oracle takes the GPU's choice of the key that holds c
            _, dq_r, dk_r, dv_r, _, _ = grad.layer_grad(hq, hk, hv, hW, w.W, w.C, sel_s, hdy, cidx=c_g)
        res["cpu_baseline"] = {"value": w.N * nkv / w.Hkv / sec, "unit": "tokens/s", "cores": torch_threads,
                               "kind": "oracle",
                               "sample": f"the gradient oracle (fp64) on sequence 0, kv heads 0..{nkv - 1} of "
                                         f"{w.Hkv} ({nq} query heads, {w.N} tokens): {sec:.2f} s, scaled to all "
                                         f"kv heads"}
        par = {}
        for nm, g_gpu, g_ref in (("dq", grads[0][:1, :nq], dq_r), ("dk", grads[1][:1, :nkv], dk_r),
                                 ("dv", grads[2][:1, :nkv], dv_r)):
            par[f"{nm}_err_rel"] = float(np.abs(g_gpu.cpu().double().numpy() - g_ref).max() / np.abs(g_ref).max())
        par["rows_row_max_differs"] = moved
        par["tolerance"] = "max|g_gpu - g_ref| <= 1e-2 max|g_ref| per tensor"
        res["parity"] = par
    return res


def cpu_decode_baseline(w, seed, steps=10):
    """The oracle's decode step on the host cores: one sequence's state built by
    the oracle's prefill over the workload's context, then `steps` decode steps
    of that sequence (its kv heads over the host threads); the decode state is
    bounded, so a step costs the same at any sequence of the batch, and the
    batch's step is the sequence's time x B."""
    import numpy as np
    from linear_attention_linearization_gb300.inputs import to_f64
    from oracle import ref
    q, k, v, Wf = (to_f64(t) for t in inputs_cpu(w, seed))
    thr = cpu_threads(w.Hkv)
    _, _, st = ref.prefill(q, k, v, Wf, w.W, w.C, w.m, w.T_max, threads=thr)
    rng = np.random.default_rng(seed + 1)
    rows = lambda h: rng.standard_normal((steps, 1, h, w.d)).astype(np.float64)
    qt, kt, vt = rows(w.Hq), rows(w.Hkv), rows(w.Hkv)
    t0 = time.perf_counter()
    for i in range(steps):
        ref.decode_step(st, qt[i], kt[i], vt[i], Wf, w.W, w.C, w.m, w.T_max, threads=thr)
    per_seq = (time.perf_counter() - t0) / steps
    return {"value": 1.0 / per_seq, "unit": "tokens/s", "cores": thr, "kind": "oracle",
            "ms_per_step": per_seq * w.B * 1e3,
            "sample": f"one sequence's state from the oracle's prefill over {w.N} tokens, {steps} decode steps of it "
                      f"({w.Hkv} kv heads over {thr} threads); a step of the {w.B}-sequence batch = its time x {w.B}"}


def inputs_cpu(w, seed):
    from linear_attention_linearization_gb300 import inputs
    return inputs.make_inputs(w, seed=seed, B=1)


def bench_decode(still, inputs, dev, stream, pk, pk_kind, args):
    import torch
    w = inputs.WORKLOADS[DECODE_WORKLOAD]
    if args.decode_seqs > 0:
        w = dataclasses.replace(w, B=args.decode_seqs)
    q, k, v, Wf = inputs.make_inputs(w, seed=args.seed + 7, device=dev)
    st = still.DecodeState(w.B, w.Hkv, w.d, w.df, w.C, w.m, device=dev)
    still.prefill(q, k, v, Wf, w.W, w.C, w.m, w.T_max, export_state=st, stream=stream)
    del q, k, v
    torch.cuda.synchronize(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(args.seed + 8)
    steps = 20
    qt = torch.randn((steps, w.B, w.Hq, w.d), generator=gen, device=dev).to(torch.bfloat16)
    kt = torch.randn((steps, w.B, w.Hkv, w.d), generator=gen, device=dev).to(torch.bfloat16)
    vt = torch.randn((steps, w.B, w.Hkv, w.d), generator=gen, device=dev).to(torch.bfloat16)
    yt = torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16, device=dev)
    valid = int((st.slot_pos[0, 0] >= 0).sum().item())
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    times = []
    warm = 3
    still.timing_read()
    for i in range(steps):
        if i == warm:
            torch.cuda.synchronize(dev)
            still.timing_read()
            still.timing_enable(True)
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        still.decode_step(st, qt[i], kt[i], vt[i], Wf, w.W, w.C, w.m, w.T_max, out_t=yt, stream=stream)
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize(dev)
    still.timing_enable(False)
    kt_launches, kt_ms = still.timing_read().get("decode_step", (0, 0.0))
    # the bracket around the call includes the host's launch work whenever
    # the GPU is idle waiting for it; the kernel's own events exclude it
    ms = [a.elapsed_time(b) for a, b in times][warm:]
    step_ms = statistics.median(ms)
    per = (kt_ms / kt_launches if kt_launches else step_ms) / 1e3
    # bytes a step must move: valid K,V slots, S read + write, z, q, k, v, out
    units = w.B * w.Hkv
    by_valid = units * (2.0 * valid * w.d * 2 + 2.0 * w.df * w.d * 4 + 2.0 * w.df * 4) + \
        w.B * (2.0 * w.Hq * w.d * 2 + 2.0 * w.Hkv * w.d * 2)
    ach = by_valid / per / 1e9
    res = {"workload": DECODE_WORKLOAD, "sequences": w.B, "context": w.N, "ms_per_step": per * 1e3,
            "ms_per_call_with_host_launch": step_ms, "kernel_launches_timed": kt_launches,
            "tokens_per_s": w.B / per, "valid_slots": valid, "algorithmic_bytes_per_step": by_valid,
            "roofline": {"kernel": "decode_step", "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": ach / pk["hbm_gbs"], "peak_source": pk_kind,
                         "traffic": profile_traffic("decode_step")},
            "state_bytes": st.nbytes()}
    if not args.no_cpu:
        res["cpu_baseline"] = cpu_decode_baseline(w, args.seed + 7)
    return res


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
