"""Benchmark of the hyper-connection call on GB300.

Workload (one GPU): the full-shape decode call, M=1 token, H=2560, C=4
(wide 10240), hc_lowrank=320, bf16 weights: one attn_hc-style call and its
inject-add, each call depending on the previous one through the residual, as
in a decoder stack.

One step = one replay of a CUDA graph that holds CALLS_PER_STEP dependent
calls, each with its inject-add, cycling through WEIGHT_SETS distinct seeded
weight sets (634 MB per pass, far larger than the 129 MB L2, so every call
streams its weights from HBM). Two sequences of the same work are timed:
  * fused (the headline): ts_hc_call, then ts_hc_inject_call for every later
    call (the previous inject-add folded into the call), then one final
    ts_hc_inject_add;
  * separate: ts_hc_call + ts_hc_inject_add for every call.
Inputs are resident in HBM when the timed region starts; ``e2e`` repeats the
headline with the step's inputs copied from pinned host memory and its
results read back inside the timed region.

``other_configs`` (skipped with --no-configs) times the rest of the workload
family the same way, each over distinct weight sets: the M=128 prefill
micro-batch (attn_hc + mlp_hc per batch, tensor-core path), a 2-token decode
batch (two-token kernels) and an 8-token one (tensor cores), the INT4-affine full shape at M=1 and M=64, the decoder's exit (mixer +
lm_head at a synthetic vocabulary of 32768) and the PLE gate at M=1 and M=16,
and the 40-layer stack (entry fused into layer 0, 80 fused calls, exit mixer)
at M=1 and M=16.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). Under torchrun each rank runs an independent
replica (no collective on the data path); value = calls of all ranks / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "hyper-connection calls/s and tokens/s at H=2560,C=4; achieved HBM GB/s vs peak"
H, C, L, M = 2560, 4, 320, 1
WEIGHT_SETS = 48
CALLS_PER_STEP = 960
CONFIG_SEED = 1  # the full-shape decode workload's seed

# Algorithmic bytes of one call + inject-add at M = 1 (every tensor once):
# down 6,553,600 + up 6,553,600 + inject 81,920 + g 20,480 + raw read 20,480
# + mixed write 5,120 + gates 16 ; inject-add: raw read+write 40,960 + out 5,120 + gates 16.
BYTES_PER_CALL = (2 * L * C * H + 2 * C * H * L + 2 * C * C * H + 2 * C * H + 2 * M * C * H
                  + 2 * M * H + 4 * M * C) + (2 * 2 * M * C * H + 2 * M * H + 4 * M * C)
assert BYTES_PER_CALL == 13_281_312


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# Sources of the kernels the headline times (the one-token path): the recorded
# DRAM traffic is reported only while their code is unchanged.
HEADLINE_KERNEL_SOURCES = ("hc_gemv.cu", "hc_kernels.h", "ptx.cuh")


def _code_only(text: str) -> str:
    """C/C++ source without its comments and blank lines (string and character
    literals kept), so that editing a comment does not count as a code change."""
    out, i, n = [], 0, len(text)
    while i < n:
        ch = text[i]
        if ch in "\"'":
            j = i + 1
            while j < n and text[j] != ch and text[j] != "\n":
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(ch)
            i += 1
    lines = (l.rstrip() for l in "".join(out).split("\n"))
    return "\n".join(l for l in lines if l)


def _kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "hyper_connection_residual_call_gb300", "csrc")
    for name in HEADLINE_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def _recorded_traffic():
    """DRAM bytes per call from the committed ncu summary, if taken on these sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("kernel_source_hash") != _kernel_source_hash():
        return None
    return d.get("dram_bytes_per_call")


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.dev), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            time.sleep(0.25)
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [l for (t, l) in self.lines if t0 - 0.15 <= t <= t1 + 0.15]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate_ranks(local_ms: float, calls_per_rank: int, device="cpu"):
    """Whole-job throughput of independent replicas: the slowest rank's time
    (max over ranks) and the calls of all ranks. Returns (max_ms, calls/s)."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    ms = float(local_ms)
    if world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, calls_per_rank * world / (ms / 1e3)


def _config(reference: bool = False):
    base = {"workload": "full-shape decode hyper-connection call + inject-add: M=1, H=2560, C=4 "
                        "(wide 10240), hc_lowrank=320, bf16 weights",
            "M": M, "H": H, "C": C, "hc_lowrank": L, "parallelism": "replicas"}
    if reference:
        return {**base, "calls_per_step": 1, "weight_sets": 1,
                "sequence": "one fp64 oracle call + inject-add per step, each call on the previous "
                            "call's residual",
                "l2": "not applicable (host cores)"}
    return {**base, "calls_per_step": CALLS_PER_STEP, "weight_sets": WEIGHT_SETS,
            "sequence": "ts_hc_call, then ts_hc_inject_call (previous inject-add fused) for each later "
                        "call, then a final ts_hc_inject_add",
            "l2": "inputs larger than L2: 48 distinct weight sets, 634 MB per pass, cycled"}


def run_reference(args):
    """The fp64 CPU oracle on this host's cores, timed on a bounded sample per step."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    from hyper_connection_residual_call_gb300 import inputs

    orc = oracle.get()
    threads = oracle.default_threads()
    w = inputs.make_hc_weights(H, C, L, CONFIG_SEED)
    raw = inputs.make_residual(M, H, C, CONFIG_SEED)
    out = inputs.make_sublayer_out(M, H, CONFIG_SEED)

    def step(r):
        res = orc.hc_call(r, w.g, w.down, w.up, w.inject, H=H, C=C, L=L, threads=threads)
        return orc.inject_add(r, out, res["gate"], H=H, C=C)

    r = raw.double().numpy()
    for _ in range(args.warmup):
        r = step(r)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r = step(r)
    dt = time.perf_counter() - t0
    value = args.steps / dt
    sample = f"{args.steps} x 1 full-shape call + inject-add (M=1, H=2560, C=4, L=320), fp64 oracle"
    line = {
        "metric": METRIC, "value": value, "unit": "calls/s", "impl": "reference", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": _config(reference=True),
        "cpu_baseline": {"value": value, "unit": "calls/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "calls/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(budget_s: float = 12.0, single_budget_s: float = 6.0, runs: int = 3):
    """The fp64 oracle on the host cores (OpenMP over output rows), and once on
    one thread, each on a bounded sample of chained full-shape calls: the median
    calls/s of `runs` timed runs that share the budget."""
    import oracle
    from hyper_connection_residual_call_gb300 import inputs

    orc = oracle.get()
    threads = oracle.default_threads()
    w = inputs.make_hc_weights(H, C, L, CONFIG_SEED)
    raw0 = inputs.make_residual(M, H, C, CONFIG_SEED).double().numpy()
    out = inputs.make_sublayer_out(M, H, CONFIG_SEED)

    def run(nthreads, budget):
        raw, n = raw0, 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < budget and n < 20000:
            res = orc.hc_call(raw, w.g, w.down, w.up, w.inject, H=H, C=C, L=L, threads=nthreads)
            raw = orc.inject_add(raw, out, res["gate"], H=H, C=C)
            n += 1
        return n, time.perf_counter() - t0

    def median_of_runs(nthreads, budget):
        res = sorted((n / dt, n, dt) for n, dt in (run(nthreads, budget / runs) for _ in range(runs)))
        rate = res[len(res) // 2][0]
        return rate, sum(r[1] for r in res), sum(r[2] for r in res)

    rate, n, dt = median_of_runs(threads, budget_s)
    rate1, n1, dt1 = median_of_runs(1, single_budget_s)
    return {"value": rate, "unit": "calls/s", "cores": threads, "kind": "oracle",
            "sample": f"median of {runs} runs, {n} full-shape calls + inject-adds (M=1, H=2560, C=4, L=320) "
                      f"in {dt:.1f} s in all, fp64 oracle, OpenMP over output rows",
            "single_thread": {"value": rate1, "unit": "calls/s", "cores": 1,
                              "sample": f"median of {runs} runs, {n1} calls + inject-adds in {dt1:.1f} s "
                                        f"in all, on one thread"}}


def parity_check(B, w0_d, w0, raw0, out0):
    """The full-shape call on weight set 0 against the oracle, before timing."""
    import numpy as np
    import torch
    import oracle

    orc = oracle.get()
    ref = orc.hc_call(raw0, w0.g, w0.down, w0.up, w0.inject, H=H, C=C, L=L)
    ref_raw = orc.inject_add(raw0, out0, ref["gate"], H=H, C=C)
    raw_d = raw0.cuda()
    mixed, gates = B.hc_call(raw_d, w0_d, H=H, C=C)
    B.hc_inject_add(raw_d, out0.cuda(), gates, H=H, C=C)
    torch.cuda.synchronize()

    def worst(g, r, atol, rtol):
        g = g.detach().double().cpu().numpy().reshape(np.shape(r))
        return float(np.max(np.abs(g - r) / (atol + rtol * np.abs(r))))

    rms = float(np.sqrt(np.mean(ref["gate"] ** 2)))
    res = {"mixed": worst(mixed, ref["mixed"], 1e-2, 1e-2),
           "raw": worst(raw_d, ref_raw, 1e-2, 1e-2),
           "gate": worst(gates, ref["gate"], 1e-5 * rms, 1e-3)}
    if not all(v <= 1.0 for v in res.values()):
        raise SystemExit(f"parity check failed before timing: {res}")
    return {"checked": "full-shape call + inject-add vs fp64 oracle", "worst_err_over_limit": max(res.values())}


def bytes_per_call(M: int, weight_bytes: int, inject: bool = True) -> int:
    """Algorithmic bytes of one call (+ its inject-add) on M tokens: weights once,
    raw read, mixed written, gates written; inject-add: raw read + written, the
    sublayer output read, the gates read."""
    b = weight_bytes + 2 * M * C * H + 2 * M * H
    if inject:
        b += 4 * M * C + (2 * 2 * M * C * H + 2 * M * H + 4 * M * C)
    return b


def fused_chain(B, raw, outs, sets, n_calls, mixed, ws, slots):
    """A body of n_calls dependent fused calls (each applies the previous call's
    inject-add), then the last inject-add; call i writes its gates to slot i % 2."""
    def body():
        for i in range(n_calls):
            w = sets[i % len(sets)]
            sl, st = slots[i % 2]
            if i == 0:
                B.hc_call(raw, w, H=H, C=C, mixed=mixed, inject_w=sl, inject_stride=st, ws=ws)
            else:
                psl, pst = slots[(i - 1) % 2]
                B.hc_inject_call(raw, outs[(i - 1) % len(outs)], psl, w, H=H, C=C, prev_inject_stride=pst,
                                 mixed=mixed, inject_w=sl, inject_stride=st, ws=ws)
        psl, pst = slots[(n_calls - 1) % 2]
        B.hc_inject_add(raw, outs[(n_calls - 1) % len(outs)], psl, H=H, C=C, inject_stride=pst)
    return body


def measure_other_configs(B, inputs, torch, dev, stream, sets_bf16, peak):
    """The workload family's other configurations, each a CUDA graph over
    distinct weight sets (every pass is larger than the 129 MB L2), timed with
    CUDA events after three warm-up replays: the M=128 prefill micro-batch
    (tensor-core path), the INT4-affine full shape at M=1 and M=64, and the
    40-layer stack (entry replication, 80 fused calls, exit mixer) at M=1 and
    M=16."""
    out = {}

    def graph_ms(body, reps):
        with torch.cuda.stream(stream):
            body()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body()
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    def chain(raw, outs, gates, sets, n_calls, mixed, ws, slots):
        return fused_chain(B, raw, outs, sets, n_calls, mixed, ws, slots)

    def record(name, Mx, ms, n_calls, bytes_call, extra=None):
        gbs = bytes_call * n_calls / (ms / 1e3) / 1e9
        out[name] = {"M": Mx, "calls_per_s": n_calls / (ms / 1e3), "tokens_per_s": Mx * n_calls / (ms / 1e3),
                     "us_per_call": 1e3 * ms / n_calls, "bytes_per_call": bytes_call, "hbm_gbs": gbs,
                     "frac": gbs / peak, **(extra or {})}

    # A 2-token decode batch (the few-token kernels): fused calls over distinct weight sets.
    Md2 = 2
    raw = inputs.make_residual(Md2, H, C, 7).to(dev)
    outs = [inputs.make_sublayer_out(Md2, H, 7, i).to(dev) for i in range(4)]
    gates = torch.zeros((2, Md2, C), dtype=torch.float32, device=dev)
    slots = [(gates[0], C), (gates[1], C)]
    mixed = torch.empty((Md2, H), dtype=torch.bfloat16, device=dev)
    ws = B.workspace(Md2, H, C, L, dev)
    n = 2 * len(sets_bf16)
    ms = graph_ms(chain(raw, outs, gates, sets_bf16, n, mixed, ws, slots), 5)
    record(f"decode_m{Md2}_bf16", Md2, ms, n, bytes_per_call(Md2, sets_bf16[0].nbytes),
           {"path": "few-token kernels (the one-token layout with a token loop)"})

    # Prefill micro-batch: M = 128, attn_hc + inject then mlp_hc + inject per batch,
    # token t's gates at t*2C (attn) and t*2C + C (mlp).
    Mp = 128
    raw = inputs.make_residual(Mp, H, C, 2).to(dev)
    outs = [inputs.make_sublayer_out(Mp, H, 2, i).to(dev) for i in range(4)]
    gates = torch.zeros((Mp, 2 * C), dtype=torch.float32, device=dev)
    slots = [(gates[:, :C], 2 * C), (gates[:, C:], 2 * C)]
    mixed = torch.empty((Mp, H), dtype=torch.bfloat16, device=dev)
    ws = B.workspace(Mp, H, C, L, dev)
    n = 2 * len(sets_bf16)
    ms = graph_ms(chain(raw, outs, gates, sets_bf16, n, mixed, ws, slots), 5)
    record("prefill_m128_bf16", Mp, ms, n, bytes_per_call(Mp, sets_bf16[0].nbytes),
           {"path": "tensor-core (tcgen05) kernels", "sequence": "attn_hc + mlp_hc per batch, fused inject"})
    del raw, outs, ws, mixed

    # INT4-affine (group 64), full shape, M = 1 and M = 64.
    # A small decode batch (8 tokens, e.g. 8 sequences decoding together): fused calls.
    Md = 8
    raw = inputs.make_residual(Md, H, C, 1).to(dev)
    outs = [inputs.make_sublayer_out(Md, H, 1, i).to(dev) for i in range(4)]
    gates = torch.zeros((2, Md, C), dtype=torch.float32, device=dev)
    slots = [(gates[0], C), (gates[1], C)]
    mixed = torch.empty((Md, H), dtype=torch.bfloat16, device=dev)
    ws = B.workspace(Md, H, C, L, dev)
    n = 2 * len(sets_bf16)
    ms = graph_ms(chain(raw, outs, gates, sets_bf16, n, mixed, ws, slots), 5)
    record(f"decode_m{Md}_bf16", Md, ms, n, bytes_per_call(Md, sets_bf16[0].nbytes),
           {"path": "tensor-core (tcgen05) kernels, one 16-token tile"})

    sets_q = [inputs.make_hc_weights(H, C, L, 4, i, kind="int4").to(dev) for i in range(len(sets_bf16))]
    for Mq in (1, 64):
        raw = inputs.make_residual(Mq, H, C, 4).to(dev)
        outs = [inputs.make_sublayer_out(Mq, H, 4, i).to(dev) for i in range(4)]
        gates = torch.zeros((2, Mq, C), dtype=torch.float32, device=dev)
        slots = [(gates[0], C), (gates[1], C)]
        mixed = torch.empty((Mq, H), dtype=torch.bfloat16, device=dev)
        ws = B.workspace(Mq, H, C, L, dev)
        n = 4 * len(sets_q) if Mq == 1 else 2 * len(sets_q)
        ms = graph_ms(chain(raw, outs, gates, sets_q, n, mixed, ws, slots), 5)
        record(f"int4_m{Mq}", Mq, ms, n, bytes_per_call(Mq, sets_q[0].nbytes),
               {"path": "CUDA-core one-token kernels" if Mq == 1
                else "tensor-core (tcgen05) kernels, INT4 dequantised to bf16 hi + lo per tile"})
    del sets_q

    # The decoder's exit: the last inject-add fused into the exit mixer, then lm_head
    # (ts_hc_exit_logits), at a synthetic vocabulary of 32768 rows (the pages give
    # none). Two lm_head copies of 168 MB alternate, so every call streams its
    # lm_head from HBM; calls depend on each other through the residual.
    V = 32768
    lm = [inputs.bf16_normal((V, H), 9000 + i, std=0.02).to(dev) for i in range(2)]
    mixers = [inputs.HCWeights(w.g, w.down, w.up, None) for w in sets_bf16[:8]]
    for Me in (1, 16):
        raw = inputs.make_residual(Me, H, C, 5).to(dev)
        oute = [inputs.make_sublayer_out(Me, H, 5, i).to(dev) for i in range(2)]
        gate = torch.full((Me, C), 0.5, dtype=torch.float32, device=dev)
        mixed = torch.empty((Me, H), dtype=torch.bfloat16, device=dev)
        logits = torch.empty((Me, V), dtype=torch.float32, device=dev)
        ws = B.workspace(Me, H, C, L, dev)
        n = 16

        def exits():
            for i in range(n):
                B.hc_exit_logits(raw, mixers[i % len(mixers)], lm[i % 2], H=H, C=C, out=oute[i % 2], prev_inject_w=gate,
                                 mixed=mixed, logits=logits, ws=ws)

        ms = graph_ms(exits, 5)
        # mixer bytes + the write-back of raw, the sublayer output and the gates read,
        # lm_head once and the logits written
        b = (bytes_per_call(Me, mixers[0].nbytes, inject=False) + 2 * Me * C * H + 2 * Me * H + 4 * Me * C
             + V * H * 2 + 4 * Me * V)
        record(f"exit_logits_m{Me}_v{V}", Me, ms, n, b,
               {"path": "inject-add fused into the exit mixer, then the tensor-core lm_head GEMM (dependent launch)",
                "vocab": V})
    del lm

    # PLE on the wide residual (ts_hc_ple), four weight sets of 66 MB cycled (264 MB,
    # more than the 129 MB L2), each call on the residual the previous one left.
    psets = [inputs.make_ple_weights(H, C, 60 + i, n_rows=4096).to(dev) for i in range(4)]
    for Mq in (1, 16):
        hid = inputs.make_residual(Mq, H, C, 6).to(dev)
        rows = inputs.make_ple_rows(Mq, 4096, 6).to(dev)
        state = torch.zeros((9, C * H), dtype=torch.float32, device=dev)
        pws = torch.empty(B.ts_hc_ple_workspace_bytes(Mq, H, C), dtype=torch.uint8, device=dev)
        n = 8

        def ples():
            for i in range(n):
                B.hc_ple(hid, rows, psets[i % 4], state, C=C, ws=pws)

        ms = graph_ms(ples, 5)
        # key_proj, value_proj, the table rows picked, the three norm scales, the conv
        # taps, the conv state read and written, the residual read and written, the ids
        W = C * H
        b = (W * H * 2 + H * H * 2 + Mq * H * 2 + 3 * W * 2 + W * 4 * 2 + 2 * 9 * W * 4 + 2 * Mq * W * 2
             + Mq * 16 * 4)
        record(f"ple_m{Mq}", Mq, ms, n, b,
               {"path": "row gather, key and value projections (one tensor-core GEMM launch), gate, causal conv + residual add"})
    del psets

    # Full-depth stack through the native driver (ts_hc_stack): entry replication,
    # 40 x (attn_hc + inject, mlp_hc + inject), exit mixer fused with the last inject-add.
    # The sublayer callback hands back stored outputs (the sublayers are not part of this path).
    n_layers = 40
    mixer_w = inputs.HCWeights(sets_bf16[0].g, sets_bf16[0].down, sets_bf16[0].up, None)
    layers = [(sets_bf16[(2 * l) % len(sets_bf16)], sets_bf16[(2 * l + 1) % len(sets_bf16)])
              for l in range(n_layers)]
    for Ms in (1, 16):
        emb = inputs.make_embedding(Ms, H, 3).to(dev)
        outs = [inputs.make_sublayer_out(Ms, H, 3, i).to(dev) for i in range(8)]
        final = torch.empty((Ms, H), dtype=torch.bfloat16, device=dev)
        sws = B.stack_workspace(Ms, H, C, L, dev)

        def stack():
            B.hc_stack(emb, layers, mixer_w, lambda l, w, t0, mixed: outs[(2 * l + w) % len(outs)], C=C,
                       max_chunk=Ms, mixed_out=final, ws=sws)

        ms = graph_ms(stack, 5)
        wb = sets_bf16[0].nbytes
        total = (2 * n_layers * bytes_per_call(Ms, wb) + bytes_per_call(Ms, mixer_w.nbytes, inject=False)
                 + 2 * Ms * H + 2 * Ms * C * H)
        gbs = total / (ms / 1e3) / 1e9
        out[f"stack40_m{Ms}"] = {"M": Ms, "tokens_per_s": Ms / (ms / 1e3), "us_per_token_step": 1e3 * ms,
                                 "bytes_per_step": total, "hbm_gbs": gbs, "frac": gbs / peak,
                                 "calls_per_step": 2 * n_layers + 1, "driver": "ts_hc_stack"}
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    from hyper_connection_residual_call_gb300 import binding as B
    from hyper_connection_residual_call_gb300 import inputs
    from hyper_connection_residual_call_gb300.build import build

    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    build()
    B.library()
    dev = torch.device("cuda", local)

    # Seeded inputs: weight sets, sublayer outputs, the initial residual.
    sets_h = [inputs.make_hc_weights(H, C, L, CONFIG_SEED, i) for i in range(WEIGHT_SETS)]
    outs_h = [inputs.make_sublayer_out(M, H, CONFIG_SEED, i) for i in range(WEIGHT_SETS)]
    raw_h = inputs.make_residual(M, H, C, CONFIG_SEED)
    sets = [w.to(dev) for w in sets_h]
    outs = torch.stack([o.to(dev) for o in outs_h])          # [sets, M, H]

    parity = None
    if rank == 0 and not (args.profile_calls or args.profile_prefill or args.profile_graph or args.profile_exit
                          or args.profile_ple):
        parity = parity_check(B, sets[0], sets_h[0], raw_h, outs_h[0])

    raw = raw_h.to(dev)
    mixed = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    gates = torch.empty((2, M, C), dtype=torch.float32, device=dev)  # two slots, alternating
    wsp = B.workspace(M, H, C, L, dev)

    def separate_step():
        for i in range(CALLS_PER_STEP):
            k = i % WEIGHT_SETS
            B.hc_call(raw, sets[k], H=H, C=C, mixed=mixed, inject_w=gates[0], inject_stride=C, ws=wsp)
            B.hc_inject_add(raw, outs[k], gates[0], H=H, C=C)

    def fused_step(n_calls=CALLS_PER_STEP):
        for i in range(n_calls):
            k = i % WEIGHT_SETS
            slot = gates[i % 2]
            if i == 0:
                B.hc_call(raw, sets[k], H=H, C=C, mixed=mixed, inject_w=slot, inject_stride=C, ws=wsp)
            else:
                kp = (i - 1) % WEIGHT_SETS
                B.hc_inject_call(raw, outs[kp], gates[(i - 1) % 2], sets[k], H=H, C=C, prev_inject_stride=C,
                                 mixed=mixed, inject_w=slot, inject_stride=C, ws=wsp)
        last = n_calls - 1
        B.hc_inject_add(raw, outs[last % WEIGHT_SETS], gates[last % 2], H=H, C=C)

    stream = torch.cuda.Stream(device=dev)
    if args.profile_prefill:
        # A short eager run of M-token calls (M=128 by default: the tensor-core
        # path; --profile-int4 for INT4-affine weights) for a profiler.
        Mp = args.profile_tokens
        psets = sets if not args.profile_int4 else [
            inputs.make_hc_weights(H, C, L, 4, i, kind="int4").to(dev) for i in range(8)]
        rawp = inputs.make_residual(Mp, H, C, 2).to(dev)
        mixedp = torch.empty((Mp, H), dtype=torch.bfloat16, device=dev)
        wsp2 = B.workspace(Mp, H, C, L, dev)
        with torch.cuda.stream(stream):
            for i in range(args.profile_prefill):
                B.hc_call(rawp, psets[i % len(psets)], H=H, C=C, mixed=mixedp, ws=wsp2)
        stream.synchronize()
        if rank == 0:
            print(f"ran {args.profile_prefill} M={Mp} calls (profiling run)")
        return
    if args.profile_exit or args.profile_ple:
        # Eager exits (mixer + lm_head, vocabulary 32768) or PLE gates at M =
        # --profile-tokens, for a profiler that captures single launches.
        Mx = args.profile_tokens
        hid = inputs.make_residual(Mx, H, C, 5).to(dev)
        with torch.cuda.stream(stream):
            if args.profile_exit:
                lm = inputs.bf16_normal((32768, H), 9000, std=0.02).to(dev)
                mixer_w = inputs.HCWeights(sets[0].g, sets[0].down, sets[0].up, None)
                mixedx = torch.empty((Mx, H), dtype=torch.bfloat16, device=dev)
                logits = torch.empty((Mx, 32768), dtype=torch.float32, device=dev)
                wsx = B.workspace(Mx, H, C, L, dev)
                for _ in range(args.profile_exit):
                    B.hc_exit_logits(hid, mixer_w, lm, H=H, C=C, mixed=mixedx, logits=logits, ws=wsx)
            else:
                pw = inputs.make_ple_weights(H, C, 60, n_rows=4096).to(dev)
                rows = inputs.make_ple_rows(Mx, 4096, 6).to(dev)
                state = torch.zeros((9, C * H), dtype=torch.float32, device=dev)
                for _ in range(args.profile_ple):
                    B.hc_ple(hid, rows, pw, state, C=C)
        stream.synchronize()
        if rank == 0:
            what = "exits" if args.profile_exit else "PLE gates"
            print(f"ran {args.profile_exit or args.profile_ple} M={Mx} {what} (profiling run)")
        return
    if args.profile_graph:
        # Replays of one CUDA graph of dependent fused M-token calls, for a profiler
        # that measures whole graphs: DRAM traffic of the chain as the kernels
        # overlap in it. One distinct weight set per call, more bytes of them than
        # the 129 MB L2 holds (16 bf16 sets of 13.2 MB, 48 INT4 sets of 3.8 MB), so
        # that a replay does not find the previous replay's weights in L2.
        Mp = args.profile_tokens
        psets = sets[:16] if not args.profile_int4 else [
            inputs.make_hc_weights(H, C, L, 4, i, kind="int4").to(dev) for i in range(48)]
        rawp = inputs.make_residual(Mp, H, C, 2).to(dev)
        outp = [inputs.make_sublayer_out(Mp, H, 2, i).to(dev) for i in range(2)]
        gatep = torch.zeros((Mp, 2 * C), dtype=torch.float32, device=dev)
        slots = [(gatep[:, :C], 2 * C), (gatep[:, C:], 2 * C)]
        mixedp = torch.empty((Mp, H), dtype=torch.bfloat16, device=dev)
        wsp2 = B.workspace(Mp, H, C, L, dev)
        body = fused_chain(B, rawp, outp, psets, len(psets), mixedp, wsp2, slots)
        with torch.cuda.stream(stream):
            body()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body()
        with torch.cuda.stream(stream):
            for _ in range(args.profile_graph):
                g.replay()
        stream.synchronize()
        if rank == 0:
            print(f"replayed a graph of {len(psets)} M={Mp} fused calls {args.profile_graph} times (profiling run)")
        return
    if args.profile_calls:
        # A short eager chain of the fused call for a profiler that captures
        # single launches: no graphs, no timing, no JSON line.
        with torch.cuda.stream(stream):
            fused_step(args.profile_calls)
        stream.synchronize()
        if rank == 0:
            print(f"ran {args.profile_calls} fused calls (profiling run)")
        return
    graphs = {}
    for name, body in (("fused", fused_step), ("separate", separate_step)):
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            body()  # eager warm-up (also initialises the library's per-device state)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body()
        graphs[name] = g
    torch.cuda.synchronize()
    launches_per_step = {"fused": 2 * CALLS_PER_STEP + 1, "separate": 3 * CALLS_PER_STEP}

    def timed(n_steps, body):
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n_steps):
                body()
            e1.record(stream)
        torch.cuda.synchronize()
        ms, _ = aggregate_ranks(e0.elapsed_time(e1), n_steps * CALLS_PER_STEP, device=dev)
        return ms

    for g in graphs.values():
        with torch.cuda.stream(stream):
            for _ in range(max(args.warmup, 3)):
                g.replay()
    torch.cuda.synchronize()

    ms_sep = timed(args.steps, graphs["separate"].replay)
    sampler = ClockSampler(local)
    sampler.start()
    t0 = time.time()
    ms = timed(args.steps, graphs["fused"].replay)
    t1 = time.time()
    clocks = sampler.stop(t0, t1)

    # Per-call time distribution: each replay (CALLS_PER_STEP calls) timed on its own.
    reps = []
    with torch.cuda.stream(stream):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(40)]
        for a, b in evs:
            a.record(stream)
            graphs["fused"].replay()
            b.record(stream)
    torch.cuda.synchronize()
    reps = sorted(1e3 * a.elapsed_time(b) / CALLS_PER_STEP for a, b in evs)
    pick = lambda q: reps[min(len(reps) - 1, int(round(q * (len(reps) - 1))))]
    per_call = {"median": pick(0.5), "p10": pick(0.1), "p90": pick(0.9), "unit": "us",
                "replays": len(reps), "calls_per_replay": CALLS_PER_STEP}

    # e2e: per step, the step's inputs (initial residual + the 48 sublayer
    # outputs) from pinned host memory, the graph, and the results read back.
    raw_pin = raw_h.pin_memory()
    outs_pin = torch.stack(outs_h).pin_memory()
    mixed_pin = torch.empty((M, H), dtype=torch.bfloat16).pin_memory()
    res_pin = torch.empty((M, C * H), dtype=torch.bfloat16).pin_memory()

    def e2e_step():
        raw.copy_(raw_pin, non_blocking=True)
        outs.copy_(outs_pin, non_blocking=True)
        graphs["fused"].replay()
        mixed_pin.copy_(mixed, non_blocking=True)
        res_pin.copy_(raw, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
    e2e_steps = max(1, args.steps // 2)
    ms_e2e = timed(e2e_steps, e2e_step)
    h2d = raw_pin.numel() * 2 + outs_pin.numel() * 2
    d2h = mixed_pin.numel() * 2 + res_pin.numel() * 2

    # One call with a host round trip: this token's residual and sublayer output
    # from pinned host memory, one fused call + inject-add, mixed and the new
    # residual read back, synchronised on the host every call.
    out_pin1 = outs_h[0].pin_memory()
    raw1 = torch.empty_like(raw)
    out1 = torch.empty((M, H), dtype=torch.bfloat16, device=dev)

    def one_call():
        raw1.copy_(raw_pin, non_blocking=True)
        out1.copy_(out_pin1, non_blocking=True)
        B.hc_call(raw1, sets[0], H=H, C=C, mixed=mixed, inject_w=gates[0], inject_stride=C, ws=wsp)
        B.hc_inject_add(raw1, out1, gates[0], H=H, C=C)
        mixed_pin.copy_(mixed, non_blocking=True)
        res_pin.copy_(raw1, non_blocking=True)
        stream.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(20):
            one_call()
        t_host = time.perf_counter()
        n_single = 400
        for _ in range(n_single):
            one_call()
        t_host = time.perf_counter() - t_host
    # The same round trip captured once in a CUDA graph (copies in, call, inject-add,
    # copies out) and replayed: what a host loop pays per token without the
    # per-call Python and launch work.
    def one_call_body():
        raw1.copy_(raw_pin, non_blocking=True)
        out1.copy_(out_pin1, non_blocking=True)
        B.hc_call(raw1, sets[0], H=H, C=C, mixed=mixed, inject_w=gates[0], inject_stride=C, ws=wsp)
        B.hc_inject_add(raw1, out1, gates[0], H=H, C=C)
        mixed_pin.copy_(mixed, non_blocking=True)
        res_pin.copy_(raw1, non_blocking=True)

    g1 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1, stream=stream):
        one_call_body()
    with torch.cuda.stream(stream):
        for _ in range(20):
            g1.replay()
            stream.synchronize()
        t_graph = time.perf_counter()
        for _ in range(n_single):
            g1.replay()
            stream.synchronize()
        t_graph = time.perf_counter() - t_graph
    single_call = {"value": n_single / t_host, "unit": "calls/s", "us_per_call": 1e6 * t_host / n_single,
                   "h2d_bytes_per_call": raw_pin.numel() * 2 + out_pin1.numel() * 2,
                   "d2h_bytes_per_call": mixed_pin.numel() * 2 + res_pin.numel() * 2,
                   "timing": "host wall clock, a stream synchronisation after every call",
                   "graph_us_per_call": 1e6 * t_graph / n_single,
                   "graph": "the same copies and calls captured once in a CUDA graph, replayed and synchronised "
                            "per call"}

    n_calls = args.steps * CALLS_PER_STEP
    value = n_calls * ws / (ms / 1e3)
    achieved = BYTES_PER_CALL / ((ms / 1e3) / n_calls) / 1e9
    achieved_sep = BYTES_PER_CALL / ((ms_sep / 1e3) / n_calls) / 1e9
    peak, peak_kind = _peaks()
    e2e_value = e2e_steps * CALLS_PER_STEP * ws / (ms_e2e / 1e3)

    others = None
    if rank == 0 and not args.no_configs:
        others = measure_other_configs(B, inputs, torch, dev, stream, sets, peak)

    if rank == 0:
        base = cpu_baseline() if ws == 1 else None
        line = {
            "metric": METRIC, "value": value, "unit": "calls/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": _config(),
            "tokens_per_s": value * M,
            "hbm_gbs": achieved,
            "us_per_call": 1e3 * ms / n_calls,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": _recorded_traffic(),
                         "kernel": "one hyper-connection call with its inject-add (down + up kernels, "
                                   "PDL-overlapped); 13,281,312 algorithmic bytes per call",
                         "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                         else "fallback 6.8 TB/s"},
            "separate_inject": {"value": n_calls * ws / (ms_sep / 1e3), "unit": "calls/s",
                                "us_per_call": 1e3 * ms_sep / n_calls, "hbm_gbs": achieved_sep,
                                "frac": achieved_sep / peak,
                                "sequence": "ts_hc_call + ts_hc_inject_add per call"},
            "per_call_us": per_call,
            "e2e": {"value": e2e_value, "unit": "calls/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "e2e_single_call": single_call,
            "gpu_launches": launches_per_step["fused"] * args.steps,
            "clocks": clocks,
            "cpu_baseline": base,
            "other_configs": others,
            "parity": parity,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the timing of the other workload configurations")
    ap.add_argument("--profile-prefill", type=int, default=0,
                    help="run this many eager M-token calls and exit (for ncu captures)")
    ap.add_argument("--profile-tokens", type=int, default=128, help="M for --profile-prefill")
    ap.add_argument("--profile-int4", action="store_true", help="INT4-affine weights for --profile-prefill")
    ap.add_argument("--profile-exit", type=int, default=0,
                    help="eager exits (mixer + lm_head at vocabulary 32768) at M = --profile-tokens, for a profiler")
    ap.add_argument("--profile-ple", type=int, default=0,
                    help="eager PLE gates at M = --profile-tokens, for a profiler")
    ap.add_argument("--profile-graph", type=int, default=0,
                    help="replays of a CUDA graph of fused M-token calls over distinct weight sets larger than "
                         "L2 in all (--profile-tokens, --profile-int4), for a profiler that measures whole graphs; "
                         "no timing")
    ap.add_argument("--profile-calls", type=int, default=0,
                    help="run this many eager fused calls of the workload and exit (for ncu captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
