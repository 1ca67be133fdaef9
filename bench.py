#!/usr/bin/env python3
"""Benchmark of the int4 group-quantized decode matvec path on GB300.

One step = one decode step of a 7B-shaped stack of 32 layers at M lanes
(default M = 1), each layer four calls through the C ABI:

    quad   : QKV 4096 -> 4096 + 1024 + 1024 (routed to q, k, v)
    matvec : O 4096 -> 4096 on q (a stand-in for the attention output)
    gated  : gate/up 4096 -> 2 x 11008 with the residual + RMSNorm prologue
             x = h + o, a = RMSNorm(x) * W_norm (writes residual_out = x)
    matvec : down 11008 -> 4096; its output is the next layer's h

with int4 weights at group size 128 (3.19 GB of packed weights, scales and
zeros per step, every step streams them from HBM: the working set is far
larger than the 129 MB L2).  Weights and inputs are seeded synthetic data.

Output: one JSON line (metric, value in GB/s of algorithmic bytes, roofline
of the dominant kernel, CPU oracle baseline, end-to-end through the API).
``--impl reference`` times the plain C oracle on the host instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "int4 matvec HBM GB/s and % of GB300 peak; 7B-stack decode µs/step at M=1"
HIDDEN, FFN, GS = 4096, 11008, 128
QKV = (4096, 1024, 1024)
EPS = 1e-6
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------------------
# Algorithmic bytes: K*N/2 + 8*N*K/gs per matrix + activations + outputs (f32)
# ---------------------------------------------------------------------------

def matrix_bytes(K, N, gs=GS):
    return K * N // 2 + 8 * N * (K // gs)


def layer_call_bytes(M):
    """Algorithmic bytes of the four calls of one layer at M lanes."""
    nq = sum(QKV)
    f = 4 * M  # bytes per f32 element per lane
    return {
        "quad": matrix_bytes(HIDDEN, nq) + f * HIDDEN + f * nq,
        "o": matrix_bytes(HIDDEN, HIDDEN) + f * HIDDEN + f * HIDDEN,
        # A, A_b, W_norm, residual_out, out
        "gated": 2 * matrix_bytes(HIDDEN, FFN) + 3 * f * HIDDEN + 4 * HIDDEN + f * FFN,
        "down": matrix_bytes(FFN, HIDDEN) + f * FFN + f * HIDDEN,
    }


def step_bytes(M, layers):
    return layers * sum(layer_call_bytes(M).values())


def stack_config(layers, M, world):
    """The bench line's `config` (the same for both arms)."""
    return {
        "workload": f"7B-shaped decode layer stack, {layers} layers, int4 group 128, M={M}",
        "lanes": M, "layers": layers, "hidden": HIDDEN, "ffn": FFN, "qkv": list(QKV),
        "group_size": GS, "bytes_per_step": step_bytes(M, layers),
        "l2": "inputs larger than L2: each step streams 3.2 GB of weights (L2 129 MB)",
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
    }


# ---------------------------------------------------------------------------
# Distributed helpers (replicas: each rank runs its own stack)
# ---------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_throughput(bytes_per_rank_step: float, ms_local: float, steps: int, world: int,
                   device="cpu"):
    """(ms per step of the slowest rank, whole-job GB/s).

    Every rank runs its own replica of the stack over the same number of
    steps, so the job moves world * bytes_per_rank_step bytes per step and
    takes as long as its slowest rank."""
    ms_step = max_over_ranks(ms_local, world, device) / steps
    return ms_step, world * bytes_per_rank_step / (ms_step / 1e3) / 1e9


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="gq4_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu_index)],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        busy = [s for s in sm if smax and s >= 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# Peaks and profile-derived traffic
# ---------------------------------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


def kernel_source_hash(names=None):
    """First 16 hex digits of the SHA-256 of the named kernel sources (all when None)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "int4_group_quantized_quant_gb300", "csrc")
    if names is None:
        names = [n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh", ".h"))]
    for name in sorted(names):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_tag: str):
    """DRAM bytes per launch recorded by an ncu capture, if the kernel's sources (the
    files the summary lists) are unchanged since."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_bytes = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", text)
    m_src = re.search(r"kernel_sources:\s*([^\n]+)", text)
    if not m_bytes or not m_hash or not m_src:
        return None
    try:
        digest = kernel_source_hash(m_src.group(1).split())
    except OSError:
        return None
    if m_hash.group(1) != digest:
        return None
    return int(m_bytes.group(1))


# ---------------------------------------------------------------------------
# The device-resident stack
# ---------------------------------------------------------------------------

def to_device(a):
    import torch
    a = np.ascontiguousarray(a)
    return torch.from_numpy(a.view(np.int32) if a.dtype == np.uint32 else a).cuda()


class Stack:
    def __init__(self, gq4, layers: int, M: int, seed: int = 4, weights=None):
        """The stack at M lanes; `weights` (another Stack's .layers) shares the
        device-resident weights instead of uploading them again."""
        import torch
        from int4_group_quantized_quant_gb300 import inputs as I
        self.gq4 = gq4
        self.M = M
        dev = torch.device("cuda")
        up = to_device
        if weights is not None:
            self.layers = weights
        else:
            self.layers = []
            for li in range(layers):
                L = I.stack_layer(li, seed)
                self.layers.append({k: (up(v.Bq), up(v.scales), up(v.zeros)) if k != "W_norm" else up(v)
                                    for k, v in L.items()})
        f32 = dict(dtype=torch.float32, device=dev)
        nq = sum(QKV)
        self.h0 = up(I.stack_input(M, seed))
        self.q = torch.empty((M, QKV[0]), **f32)
        self.k = torch.empty((M, QKV[1]), **f32)
        self.v = torch.empty((M, QKV[2]), **f32)
        self.o = torch.empty((M, HIDDEN), **f32)
        self.res = torch.empty((M, HIDDEN), **f32)
        self.f = torch.empty((M, FFN), **f32)
        # ping-pong residual-stream buffers: down output of layer l is h of layer l+1
        self.hbuf = [torch.empty((M, HIDDEN), **f32) for _ in range(2)]
        self.n0, self.n1, self.n2 = QKV[0], QKV[0] + QKV[1], nq

    def launches_per_step(self):
        return 4 * len(self.layers)

    def sequence(self):
        """The step as one call sequence (one lane): the calls of layer() in
        order, for gq4_run_sequence."""
        gq4, calls = self.gq4, []
        h = self.h0
        for li in range(len(self.layers)):
            L, h_next = self.layers[li], self.hbuf[li % 2]
            calls += [
                gq4.seq_quad(h, *L["qkv"], GS, self.n0, self.n1, self.n2, [self.q, self.k, self.v, None]),
                gq4.seq_matvec(self.q, *L["o"], GS, self.o),
                gq4.seq_gated(h, *L["gate"], *L["up"], GS, self.f, W_norm=L["W_norm"], eps=EPS,
                              A_b=self.o, residual_out=self.res),
                gq4.seq_matvec(self.f, *L["down"], GS, h_next),
            ]
            h = h_next
        return calls, h

    def layer(self, li, h, h_next, stream):
        gq4, L = self.gq4, self.layers[li]
        gq4.quad_matvec(h, *L["qkv"], GS, self.n0, self.n1, self.n2,
                        outs=[self.q, self.k, self.v, None], stream=stream)
        gq4.matvec(self.q, *L["o"], GS, C=self.o, stream=stream)
        gq4.gated_matvec(h, *L["gate"], *L["up"], GS, W_norm=L["W_norm"], eps=EPS, A_b=self.o,
                         residual_out=self.res, out=self.f, stream=stream)
        gq4.matvec(self.f, *L["down"], GS, C=h_next, stream=stream)

    def step(self, stream):
        h = self.h0
        for li in range(len(self.layers)):
            h_next = self.hbuf[li % 2]
            self.layer(li, h, h_next, stream)
            h = h_next
        return h


# ---------------------------------------------------------------------------
# Per-config lines: configs 0-3 at their stated shapes, the stack at more
# lanes, the prefill GEMM, and the sequence kernel against the graph of calls
# ---------------------------------------------------------------------------

def lane_path(M):
    """(kernel description, profile tag prefix) of the path an M-lane call takes."""
    if M == 1:
        return "one-lane streaming kernel, CUDA cores", "M1"
    if M <= 4:
        return ("2-4-lane kernel: exact fp16 products on the warp-level MMA (the 11008-long down "
                "projection with K split over a 4-CTA cluster)"), f"M{M}"
    if M < 16:
        return "multi-lane fp32 kernel, CUDA cores", f"M{M}"
    return "tensor-core kernel (tcgen05, bf16 operands, f32 accumulate)", f"M{M}"


def graph_time_us(body, steps, warmup, stream):
    """µs per replay of a CUDA graph of body(stream), CUDA events on the replay stream."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(2):
            body(stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        body(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for _ in range(max(warmup, 3)):
            g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / steps
    del g
    return us


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(fn_cols, N, reps=3):
    """(median µs single-threaded, median µs on all host cores, cores) of an
    oracle call split by columns: fn_cols(c0, c1) runs the oracle on columns
    [c0, c1).  The C oracle releases the GIL, so threads run it in parallel;
    the oracle itself is unchanged (each column's sum is still sequential)."""
    from concurrent.futures import ThreadPoolExecutor
    cores = host_cores()
    one = []
    for _ in range(reps):
        t0 = time.perf_counter()
        fn_cols(0, N)
        one.append(time.perf_counter() - t0)
    bounds = [N * i // cores for i in range(cores + 1)]
    parts = [(bounds[i], bounds[i + 1]) for i in range(cores) if bounds[i + 1] > bounds[i]]
    par = []
    with ThreadPoolExecutor(max_workers=len(parts)) as pool:
        for _ in range(reps):
            t0 = time.perf_counter()
            list(pool.map(lambda b: fn_cols(*b), parts))
            par.append(time.perf_counter() - t0)
    return statistics.median(one) * 1e6, statistics.median(par) * 1e6, len(parts)


def config_cases(gq4):
    """Configs 0-3 at their stated shapes and distributions: for each, a
    description, the algorithmic bytes of one call, the bytes of one weight
    set, a device-call maker over rotating weight sets, and the oracle over
    a column range."""
    import torch
    from int4_group_quantized_quant_gb300 import inputs as I
    cases = []

    def dev_w(w):
        return (to_device(w.Bq), to_device(w.scales), to_device(w.zeros))

    def mat_bytes(K, N, gs):
        return K * N // 2 + 8 * N * (K // gs)

    def wslice(w, c0, c1):
        return w.Bq[c0:c1], w.scales[c0:c1], w.zeros[c0:c1]

    # config 0: single matvec 1024 x 1024, gs 32
    d = I.single_matvec()
    K, N, gs = d["K"], d["N"], d["gs"]
    A, C = to_device(d["A"]), torch.empty((1, N), dtype=torch.float32, device="cuda")
    cases.append(dict(
        name="c0", workload=f"single int4 matvec M=1, K={K}, N={N}, group_size={gs}",
        call_bytes=mat_bytes(K, N, gs) + 4 * K + 4 * N, set_bytes=mat_bytes(K, N, gs),
        w0=dev_w(d["w"]), N=N,
        call=lambda W, s, A=A, C=C, gs=gs: gq4.matvec(A, *W, gs, C=C, stream=s),
        oracle=lambda orc, c0, c1, d=d: orc.matvec(d["A"], *wslice(d["w"], c0, c1), d["K"], c1 - c0,
                                                   d["gs"])))

    # config 1: quad QKV 2560 -> 10240 split 4096/5120/6144, gs 64
    d = I.quad_qkv()
    K, N, gs, n0, n1, n2 = d["K"], d["N"], d["gs"], d["n0"], d["n1"], d["n2"]
    A = to_device(d["A"])
    outs = [torch.empty((1, n), dtype=torch.float32, device="cuda")
            for n in (n0, n1 - n0, n2 - n1, N - n2)]

    def quad_oracle(orc, c0, c1, d=d):
        cl = lambda v: min(max(v - c0, 0), c1 - c0)
        return orc.quad_matvec(d["A"], *wslice(d["w"], c0, c1), d["K"], c1 - c0, d["gs"],
                               cl(d["n0"]), cl(d["n1"]), cl(d["n2"]))
    cases.append(dict(
        name="c1", workload=f"quad-output QKV matvec M=1, K={K}, N={N}, split {n0}/{n1}/{n2}, "
                            f"group_size={gs}",
        call_bytes=mat_bytes(K, N, gs) + 4 * K + 4 * N, set_bytes=mat_bytes(K, N, gs),
        w0=dev_w(d["w"]), N=N,
        call=lambda W, s, A=A, outs=outs, gs=gs, sp=(n0, n1, n2):
            gq4.quad_matvec(A, *W, gs, *sp, outs=outs, stream=s),
        oracle=quad_oracle))

    # config 2: norm-prologue matvec 4096 -> 4096, gs 64, eps 1e-6
    d = I.norm_prologue()
    K, N, gs = d["K"], d["N"], d["gs"]
    A, Ab, Wn = to_device(d["A"]), to_device(d["A_b"]), to_device(d["W_norm"])
    C = torch.empty((1, N), dtype=torch.float32, device="cuda")
    cases.append(dict(
        name="c2", workload=f"norm-prologue matvec M=1, K={K}, N={N}, group_size={gs}, eps=1e-6",
        call_bytes=mat_bytes(K, N, gs) + 3 * 4 * K + 4 * N, set_bytes=mat_bytes(K, N, gs),
        w0=dev_w(d["w"]), N=N,
        call=lambda W, s, A=A, Ab=Ab, Wn=Wn, C=C, gs=gs, eps=d["eps"]:
            gq4.norm_matvec(A, *W, gs, W_norm=Wn, eps=eps, A_b=Ab, C=C, stream=s),
        oracle=lambda orc, c0, c1, d=d: orc.norm_matvec(d["A"], d["A_b"], d["W_norm"], d["eps"],
                                                        *wslice(d["w"], c0, c1), d["K"], c1 - c0,
                                                        d["gs"])))

    # config 3: SiLU-gated gate/up 4096 -> 2 x 11008, gs 128
    d = I.gated_gate_up()
    K, N, gs = d["K"], d["N"], d["gs"]
    A = to_device(d["A"])
    out = torch.empty((1, N), dtype=torch.float32, device="cuda")
    cases.append(dict(
        name="c3", workload=f"SiLU-gated gate/up matvec M=1, K={K}, N={N} x 2, group_size={gs}",
        call_bytes=2 * mat_bytes(K, N, gs) + 4 * K + 4 * N, set_bytes=2 * mat_bytes(K, N, gs),
        w0=dev_w(d["wg"]) + dev_w(d["wu"]), N=N,
        call=lambda W, s, A=A, out=out, gs=gs: gq4.gated_matvec(A, *W, gs, out=out, stream=s),
        oracle=lambda orc, c0, c1, d=d: orc.gated_matvec(d["A"], *wslice(d["wg"], c0, c1),
                                                         *wslice(d["wu"], c0, c1), d["K"],
                                                         c1 - c0, d["gs"])))
    return cases


def measure_per_config(gq4, stack, args, peak, with_oracle):
    """One entry per config; each config's calls replayed in a CUDA graph over
    rotating weight sets of at least 4x L2, so that every call reads HBM."""
    import torch
    out = {}
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    stream = torch.cuda.Stream()
    orc = None
    if with_oracle:
        import oracle
        orc = oracle.load()
    for case in config_cases(gq4):
        R = max(2, -(-4 * l2 // case["set_bytes"]))
        sets = [case["w0"]] + [tuple(t.clone() for t in case["w0"]) for _ in range(R - 1)]

        def body(s, sets=sets, call=case["call"]):
            for W in sets:
                call(W, s)
        us = graph_time_us(body, max(args.steps, 20), args.warmup, stream) / R
        gbs = case["call_bytes"] / (us * 1e-6) / 1e9
        e = {"workload": case["workload"], "us_per_call": round(us, 3),
             "bytes_per_call": case["call_bytes"], "GB/s": round(gbs, 1),
             "frac_of_hbm_peak": round(gbs / peak, 4), "weight_sets": R,
             "kernel": lane_path(1)[0],
             "timing": f"CUDA graph of {R} calls over distinct weight sets "
                       f"({R * case['set_bytes'] / 1e6:.0f} MB > 4x L2), CUDA events"}
        if orc is not None:
            one, par, cores = time_oracle(lambda c0, c1, o=case["oracle"]: o(orc, c0, c1), case["N"])
            e["oracle"] = {"us_single_thread": round(one, 1), "us_all_cores": round(par, 1),
                           "cores": cores, "kind": "C fp64 oracle, columns split over threads",
                           "GB/s_all_cores": round(case["call_bytes"] / (par * 1e-6) / 1e9, 4)}
        out[case["name"]] = e
        del sets
    torch.cuda.empty_cache()

    # the stack at more lanes (same device weights as the one-lane stack)
    for M in args.stack_lanes:
        st = Stack(gq4, len(stack.layers), M, weights=stack.layers)
        us = graph_time_us(lambda s, st=st: st.step(s), max(args.steps, 10), args.warmup, stream)
        sb = step_bytes(M, len(stack.layers))
        gbs = sb / (us * 1e-6) / 1e9
        kern, _ = lane_path(M)
        e = {"workload": f"7B-shaped decode layer stack, {len(stack.layers)} layers, int4 group 128, "
                         f"M={M}",
             "us_per_step": round(us, 2), "bytes_per_step": sb, "GB/s": round(gbs, 1),
             "frac_of_hbm_peak": round(gbs / peak, 4), "vs_M1_step": None, "kernel": kern,
             "timing": "CUDA graph of one step (128 C-ABI calls), CUDA events"}
        if orc is not None:
            e["oracle"] = stack_oracle_sample(orc, M)
        out[f"c4_M{M}"] = e
        del st
    return out


def stack_oracle_sample(orc, M):
    """The oracle on a bounded sample of the M-lane stack: layer 0's O
    projection (4096 -> 4096) at M lanes, one thread and all cores, scaled to
    a whole 32-layer step by algorithmic bytes."""
    from int4_group_quantized_quant_gb300 import inputs as I
    L = I.stack_layer(0)
    w = L["o"]
    A = I.stack_input(M)[:, :HIDDEN].copy()
    fn = lambda c0, c1: orc.matvec(A, w.Bq[c0:c1], w.scales[c0:c1], w.zeros[c0:c1], HIDDEN,
                                   c1 - c0, GS)
    one, par, cores = time_oracle(fn, HIDDEN, reps=1)
    scale = step_bytes(M, 32) / layer_call_bytes(M)["o"]
    return {"us_per_step_single_thread": round(one * scale, 0),
            "us_per_step_all_cores": round(par * scale, 0), "cores": cores,
            "sample": f"layer 0's O projection 4096 -> 4096 at M={M} (C fp64 oracle), scaled to "
                      f"a 32-layer step by algorithmic bytes"}


def measure_gemm(gq4, args):
    """Prefill GEMM, 2048 rows through a 4096 x 4096 projection (gs 128), two
    alternating weight sets, against the measured bf16 peak."""
    import torch
    from int4_group_quantized_quant_gb300 import inputs as I
    Mg, K, N = 2048, 4096, 4096
    ws = [tuple(to_device(a) for a in (w.Bq, w.scales, w.zeros))
          for w in (I.quant_weights(K, N, GS, 1600, 90 + r) for r in range(2))]
    A = to_device(I.activations(Mg, K, 1600, 91))
    C = torch.empty((Mg, N), dtype=torch.float32, device="cuda")
    work = torch.empty(gq4.gemm_workspace_bytes(Mg, K), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()

    def body(s):
        for W in ws:
            gq4.gemm(A, *W, GS, C=C, workspace=work, stream=s)
    us = graph_time_us(body, max(args.steps, 20), args.warmup, stream) / 2
    tpeak, tsrc = bf16_peak()
    tf = 2.0 * Mg * K * N / (us * 1e-6) / 1e12
    return {"workload": f"prefill GEMM {Mg} x {K} -> {N}, int4 group {GS}", "us_per_call": round(us, 2),
            "TFLOP/s": round(tf, 1), "frac_of_bf16_peak": round(tf / tpeak, 4), "peak": tpeak,
            "peak_source": tsrc, "bound": "tensor",
            "kernel": "tcgen05 GEMM (bf16 operands dequantized in registers, f32 accumulate)",
            "timing": "CUDA graph of 2 calls over 2 weight sets, CUDA events"}


def measure_sequence(gq4, stack, args, graph_us):
    """The M = 1 step as one gq4_run_sequence launch (persistent kernel with a
    grid barrier between calls) against the graph of single calls."""
    import torch
    calls, _ = stack.sequence()
    ws = gq4.sequence_workspace()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            gq4.run_sequence(calls, ws, stream=stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(args.steps, 10)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n):
            gq4.run_sequence(calls, ws, stream=stream)
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / n
    return {"workload": "7B-shaped stack, 32 layers, M=1, as gq4_run_sequence",
            "us_per_step": round(us, 2), "graph_of_calls_us_per_step": round(graph_us, 2),
            "ratio_to_graph": round(us / graph_us, 4),
            "timing": "one persistent launch per step (128 calls), eager, CUDA events"}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import torch
    torch.cuda.set_device(local_rank)
    dist_init(world, "nccl")
    from int4_group_quantized_quant_gb300 import build as b
    if rank == 0 or world == 1:
        b.build()
    barrier(world)
    from int4_group_quantized_quant_gb300 import gq4

    M, layers = args.lanes, args.layers
    stack = Stack(gq4, layers, M)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    # warm-up (eager), then capture one step into a CUDA graph
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 1)):
            out = stack.step(stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        out = stack.step(torch.cuda.current_stream())
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    # ---- timed region: K graph replays, events on the replay stream ----
    clocks = ClockSampler(local_rank)
    clocks.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = ev0.elapsed_time(ev1)
    sbytes = step_bytes(M, layers)
    ms_step, value = job_throughput(sbytes, ms, args.steps, world, device="cuda")

    # ---- roofline: average launch duration of the dominant kernel ----
    # the gated gate/up call with its norm prologue (about half the step's
    # bytes) over the 32 layers' own weights (1.6 GB, larger than L2): a CUDA
    # graph of the 32 launches back to back, replayed between CUDA events on
    # its stream (avg = time / 32); and, for reference, each launch alone
    # between events
    def gated_all(s):
        for li in range(layers):
            L = stack.layers[li]
            gq4.gated_matvec(stack.h0, *L["gate"], *L["up"], GS, W_norm=L["W_norm"], eps=EPS,
                             A_b=stack.o, residual_out=stack.res, out=stack.f, stream=s)
    rounds = max(args.roofline_rounds, 3)
    gated_graph_us = graph_time_us(gated_all, rounds, args.warmup, stream) / layers
    durs = []
    with torch.cuda.stream(stream):
        for _ in range(args.roofline_rounds):
            for li in range(layers):
                L = stack.layers[li]
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                gq4.gated_matvec(stack.h0, *L["gate"], *L["up"], GS, W_norm=L["W_norm"], eps=EPS,
                                 A_b=stack.o, residual_out=stack.res, out=stack.f, stream=stream)
                e1.record(stream)
                durs.append((e0, e1))
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    gated_ms = [a.elapsed_time(b_) for a, b_ in durs]
    gated_alone_us = statistics.mean(gated_ms) * 1e3
    gated_avg_s = gated_graph_us / 1e6
    gated_bytes = layer_call_bytes(M)["gated"]

    # ---- end to end through the API: pinned H2D of h, replay, D2H of the output ----
    h_host = torch.empty_like(stack.h0, device="cpu").pin_memory()
    h_host.copy_(stack.h0.cpu())
    out_host = torch.empty_like(out, device="cpu").pin_memory()
    e2e_steps = args.steps
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            stack.h0.copy_(h_host, non_blocking=True)
            graph.replay()
            out_host.copy_(out, non_blocking=True)
            stream.synchronize()
    t1 = time.perf_counter()
    e2e_s = max_over_ranks((t1 - t0) / e2e_steps, world, device="cuda")

    peak, peak_src = hbm_peak()
    achieved = gated_bytes / gated_avg_s / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "us_per_step": round(ms_step * 1e3, 2),
        "pct_of_hbm_peak": round(100.0 * value / world / peak, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded; int4 codes uniform 0..15, scales U[0.005,0.02], zeros U[6,9], "
                "activations N(0,1), norm gain U[0.5,1.5])",
        "config": stack_config(layers, M, world),
        "timing": "CUDA graph of one step (128 C-ABI calls), replayed; CUDA events on the replay stream",
        "roofline": {
            "kernel": f"gq4 gated gate/up + RMSNorm prologue, 4096 -> 2 x 11008, M={M} ({lane_path(M)[0]})",
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
            else "fallback 6.8 TB/s",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": profiled_traffic(f"gated_norm_4096x2x11008_{lane_path(M)[1]}"),
            "bytes_per_launch": gated_bytes,
            "avg_launch_us": round(gated_avg_s * 1e6, 3),
            "timing": f"CUDA graph of the {layers} layers' gate/up calls back to back (their own "
                      f"weights, larger than L2), replayed {rounds}x between CUDA events",
            "launches_timed": layers * rounds,
            "alone_avg_launch_us": round(gated_alone_us, 3),
            "alone_timing": f"each launch alone between CUDA events ({len(gated_ms)} launches)",
        },
        "e2e": {
            "value": round(world * sbytes / e2e_s / 1e9, 2),
            "unit": "GB/s",
            "us_per_step": round(e2e_s * 1e6, 2),
            "h2d_bytes_per_step": int(stack.h0.numel() * 4),
            "d2h_bytes_per_step": int(out.numel() * 4),
            "how": "pinned host h -> device, graph replay of the step's C-ABI calls, "
                   "output -> pinned host, stream sync; host wall clock",
        },
        "gpu_launches": args.steps * stack.launches_per_step(),
        "clocks": clock_info,
    }
    # per-config lines (rank 0 of a replica run measures them on its own GPU)
    if rank == 0 and not args.no_per_config:
        pc = measure_per_config(gq4, stack, args, peak, with_oracle=not args.no_cpu_baseline)
        for key in list(pc):
            if key.startswith("c4_M"):
                pc[key]["vs_M1_step"] = round(pc[key]["us_per_step"] / (ms_step * 1e3), 3)
        pc["gemm_2048"] = measure_gemm(gq4, args)
        if M == 1:
            pc["sequence_M1"] = measure_sequence(gq4, stack, args, ms_step * 1e3)
        line["per_config"] = pc
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(M, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_layer(orc, L, h, M):
    """One layer through the C oracle (same data flow as the GPU step)."""
    n0, n1, n2 = QKV[0], QKV[0] + QKV[1], sum(QKV)
    outs, _ = orc.quad_matvec(h, L["qkv"].Bq, L["qkv"].scales, L["qkv"].zeros, HIDDEN, n2, GS,
                              n0, n1, n2)
    q = outs[0].astype(np.float32)
    o, _ = orc.matvec(q, L["o"].Bq, L["o"].scales, L["o"].zeros, HIDDEN, HIDDEN, GS)
    g = orc.gated_matvec(h, L["gate"].Bq, L["gate"].scales, L["gate"].zeros, L["up"].Bq,
                         L["up"].scales, L["up"].zeros, HIDDEN, FFN, GS,
                         A_b=o.astype(np.float32), W_norm=L["W_norm"], eps=EPS)
    d, _ = orc.matvec(g["out"].astype(np.float32), L["down"].Bq, L["down"].scales,
                      L["down"].zeros, FFN, HIDDEN, GS)
    return d.astype(np.float32)


def oracle_layer_parallel(orc, L, h, M, pool, cores):
    """oracle_layer with each call's columns split over `cores` threads (the C
    oracle releases the GIL; its arithmetic is unchanged, every column's sum
    still sequential, so the results are the same bits)."""
    n0, n1, n2 = QKV[0], QKV[0] + QKV[1], sum(QKV)

    def split(N):
        b = [N * i // cores for i in range(cores + 1)]
        return [(b[i], b[i + 1]) for i in range(cores) if b[i + 1] > b[i]]

    def cols(fn, N):
        parts = list(pool.map(lambda r: fn(*r), split(N)))
        return np.concatenate(parts, axis=1)

    def mv(A, w, K, N):
        return cols(lambda c0, c1: orc.matvec(A, w.Bq[c0:c1], w.scales[c0:c1], w.zeros[c0:c1], K,
                                              c1 - c0, GS)[0], N)
    qkv = mv(h, L["qkv"], HIDDEN, n2)
    q = np.ascontiguousarray(qkv[:, :n0]).astype(np.float32)
    o = mv(q, L["o"], HIDDEN, HIDDEN).astype(np.float32)
    g = cols(lambda c0, c1: orc.gated_matvec(
        h, L["gate"].Bq[c0:c1], L["gate"].scales[c0:c1], L["gate"].zeros[c0:c1],
        L["up"].Bq[c0:c1], L["up"].scales[c0:c1], L["up"].zeros[c0:c1], HIDDEN, c1 - c0, GS,
        A_b=o, W_norm=L["W_norm"], eps=EPS)["out"], FFN)
    return mv(g.astype(np.float32), L["down"], FFN, HIDDEN).astype(np.float32)


def cpu_baseline(M, seconds):
    """The oracle as it stands on the host over whole layers of the stack:
    on all host cores (each call's columns split over threads) for about
    `seconds`, and single-threaded for about `seconds`."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    from int4_group_quantized_quant_gb300 import inputs as I
    orc = oracle.load()
    lbytes = sum(layer_call_bytes(M).values())
    cores = host_cores()
    layers = [I.stack_layer(li) for li in range(4)]

    def timed(run_layer):
        h = I.stack_input(M)
        done, t_total = 0, 0.0
        while True:
            t0 = time.perf_counter()
            h = run_layer(layers[done % len(layers)], h)
            t_total += time.perf_counter() - t0
            done += 1
            if t_total >= seconds or done >= 32:
                return done, t_total, h
    with ThreadPoolExecutor(max_workers=cores) as pool:
        dp, tp, _ = timed(lambda L, h: oracle_layer_parallel(orc, L, h, M, pool, cores))
        # the split changes no bits: layer 0 both ways
        h0 = I.stack_input(M)
        same = bool(np.array_equal(oracle_layer_parallel(orc, layers[0], h0, M, pool, cores)
                                   .view(np.uint32), oracle_layer(orc, layers[0], h0, M).view(np.uint32)))
    d1, t1, _ = timed(lambda L, h: oracle_layer(orc, L, h, M))
    return {"value": round(dp * lbytes / tp / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{dp} layers of the same stack at M={M} (4 calls each, the first 4 layers' "
                      f"weights in turn), C fp64 oracle with each call's columns split over "
                      f"{cores} threads, {tp:.1f} s",
            "us_per_layer": round(tp / dp * 1e6, 1),
            "single_thread": {"value": round(d1 * lbytes / t1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                              "us_per_layer": round(t1 / d1 * 1e6, 1),
                              "sample": f"{d1} layers, single-threaded, {t1:.1f} s"},
            "threaded_equals_single": same}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    from int4_group_quantized_quant_gb300 import inputs as I
    from concurrent.futures import ThreadPoolExecutor
    orc = oracle.load()
    M = args.lanes
    cores = host_cores()
    pool = ThreadPoolExecutor(max_workers=cores)
    h = I.stack_input(M)
    li = 0
    # warm-up layers (untimed), then K timed steps of one layer each (a bounded
    # sample), each call's columns split over the host's cores
    for _ in range(args.warmup):
        h = oracle_layer_parallel(orc, I.stack_layer(li % args.layers), h, M, pool, cores)
        li += 1
    t_total = 0.0
    for _ in range(args.steps):
        L = I.stack_layer(li % args.layers)
        t0 = time.perf_counter()
        h = oracle_layer_parallel(orc, L, h, M, pool, cores)
        t_total += time.perf_counter() - t0
        li += 1
    pool.shutdown()
    lbytes = sum(layer_call_bytes(M).values())
    value = args.steps * lbytes / t_total / 1e9
    sample = (f"{args.steps} timed layers (of the {args.layers}-layer stack) at M={M}, 4 calls "
              f"each, C fp64 oracle with each call's columns split over {cores} threads")
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_total / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded, same generator and distributions as the GPU arm)",
        "config": stack_config(args.layers, M, world),
        "timing": "host wall clock over a bounded sample: one layer per step, scaled to GB/s by "
                  "the layer's algorithmic bytes",
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# Profile cases (small, for ncu): a few launches of one kernel
# ---------------------------------------------------------------------------

def run_profile_case(args):
    import torch
    from int4_group_quantized_quant_gb300 import build as b
    b.build()
    from int4_group_quantized_quant_gb300 import gq4
    torch.cuda.set_device(0)
    if args.profile == "gemm":
        # prefill GEMM: 2048 rows through one 4096 x 4096 projection (gs 128)
        from int4_group_quantized_quant_gb300 import inputs as I
        Mg, K = 2048, 4096
        w = I.quant_weights(K, 4096, GS, 1600, 90)
        Wd = tuple(torch.from_numpy(a.view(np.int32) if a.dtype == np.uint32 else a).cuda()
                   for a in (w.Bq, w.scales, w.zeros))
        A = torch.from_numpy(I.activations(Mg, K, 1600, 91)).cuda()
        C = torch.empty((Mg, 4096), dtype=torch.float32, device="cuda")
        ws = torch.empty(gq4.gemm_workspace_bytes(Mg, K), dtype=torch.uint8, device="cuda")
        for _ in range(args.steps):
            gq4.gemm(A, *Wd, GS, C=C, workspace=ws)
        torch.cuda.synchronize()
        print(json.dumps({"profile_case": "gemm", "rows": Mg, "launch_rounds": args.steps}))
        return
    stack = Stack(gq4, args.layers, args.lanes)
    stream = torch.cuda.current_stream()
    for _ in range(args.steps):
        for li in range(args.layers):
            if args.profile == "step":
                stack.layer(li, stack.h0, stack.hbuf[0], stream)
            elif args.profile == "gated":
                L = stack.layers[li]
                gq4.gated_matvec(stack.h0, *L["gate"], *L["up"], GS, W_norm=L["W_norm"], eps=EPS,
                                 A_b=stack.o, residual_out=stack.res, out=stack.f, stream=stream)
            elif args.profile == "down":
                L = stack.layers[li]
                gq4.matvec(stack.f, *L["down"], GS, C=stack.hbuf[0], stream=stream)
            elif args.profile == "quad":
                L = stack.layers[li]
                gq4.quad_matvec(stack.h0, *L["qkv"], GS, stack.n0, stack.n1, stack.n2,
                                outs=[stack.q, stack.k, stack.v, None], stream=stream)
            elif args.profile == "o":
                L = stack.layers[li]
                gq4.matvec(stack.q, *L["o"], GS, C=stack.o, stream=stream)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": args.profile, "layers": args.layers, "lanes": args.lanes,
                      "launch_rounds": args.steps}))


def run_extras(args):
    """Time the widened entry points, one JSON line per op: the dual projection
    and the gated-input matvecs (one lane, 4096 x 4096, in a CUDA graph over
    rotating weight sets larger than 4x L2, against the plain matvec), the
    prefill GEMM (512 and 2048 rows through 4096 x 4096, against the bf16
    peak), the quantizer and the MLX converter (4096 x 11008) and the
    embedding gather (8192 ids from a 32000 x 4096 table)."""
    import torch
    from int4_group_quantized_quant_gb300 import build as b
    b.build()
    from int4_group_quantized_quant_gb300 import gq4
    from int4_group_quantized_quant_gb300 import inputs as I
    torch.cuda.set_device(0)
    K = N = 4096
    gs = GS
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    mat_bytes = K * N // 2 + 8 * N * (K // gs)
    R = max(8, -(-4 * l2 // mat_bytes))
    mats = []
    for r in range(R):
        w = I.quant_weights(K, N, gs, 1600, r)
        mats.append(tuple(torch.from_numpy(a).cuda() for a in (w.Bq, w.scales, w.zeros)))
    X = torch.from_numpy(I.activations(1, K, 1600, 0)).cuda()
    G = torch.from_numpy(I.activations(1, K, 1600, 1)).cuda()
    C0 = torch.empty((1, N), dtype=torch.float32, device="cuda")
    C1 = torch.empty((1, N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    peak, peak_src = hbm_peak()

    def time_graph(body):
        with torch.cuda.stream(stream):
            for _ in range(2):
                body(stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body(torch.cuda.current_stream())
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1000.0 / args.steps

    def dual(s):
        for r in range(0, R - 1, 2):
            gq4.dual_matvec(X, *mats[r], *mats[r + 1], gs, C0=C0, C1=C1, stream=s)

    def two_matvecs(s):
        for r in range(0, R - 1, 2):
            gq4.matvec(X, *mats[r], gs, C=C0, stream=s)
            gq4.matvec(X, *mats[r + 1], gs, C=C1, stream=s)

    def plain(s):
        for r in range(R):
            gq4.matvec(X, *mats[r], gs, C=C0, stream=s)

    def sigmoid(s):
        for r in range(R):
            gq4.sigmoid_gated_matvec(X, G, *mats[r], gs, C=C0, stream=s)

    def swiglu(s):
        for r in range(R):
            gq4.swiglu_gated_matvec(X, G, *mats[r], gs, C=C0, stream=s)

    # producing the format: the quantizer over the 4096 -> 11008 gate/up
    # projection (f32 weights, 180 MB each, two rotating copies) and the MLX
    # converter over rotating MLX matrices of the same shape
    Kq, Nq = 4096, 11008
    Gq = Kq // gs
    Wf = [torch.from_numpy(I.float_weights(Nq, Kq, 1600, r)).cuda() for r in range(2)]
    qout = [gq4.quantize(Wf[r], gs) for r in range(2)]
    mlx_set = Kq * Nq // 2 + 8 * Nq * Gq
    Rm = max(8, -(-4 * l2 // (2 * mlx_set)))
    mlx_in, mlx_out = [], []
    for r in range(Rm):
        m = I.mlx_weights(Kq, Nq, gs, 1600, r)
        mlx_in.append(tuple(torch.from_numpy(a.view(np.int32) if a.dtype == np.uint32 else a)
                            .cuda() for a in (m.packed, m.scales, m.biases)))
        mlx_out.append(gq4.from_mlx(*mlx_in[r], gs))

    def quantize(s):
        for r in range(2):
            gq4.quantize(Wf[r], gs, *qout[r], stream=s)

    def convert(s):
        for r in range(Rm):
            gq4.from_mlx(*mlx_in[r], gs, *mlx_out[r], stream=s)

    # embedding gather: 8192 tokens from a 32000 x 4096 table (gs 128); the
    # 128 MB output exceeds L2, the 74 MB table does not (ids are random)
    Te, Ve = 8192, 32000
    we = I.quant_weights(Kq, Ve, gs, 1600, 77)
    emb_w = tuple(torch.from_numpy(a.view(np.int32) if a.dtype == np.uint32 else a).cuda()
                  for a in (we.Bq, we.scales, we.zeros))
    emb_ids = [torch.from_numpy(I.rng(1600, 78, r).integers(0, Ve, size=Te, dtype=np.int32))
               .cuda() for r in range(2)]
    emb_out = [torch.empty((Te, Kq), dtype=torch.float32, device="cuda") for _ in range(2)]

    def embed(s):
        for r in range(2):
            gq4.embedding(emb_ids[r], *emb_w, gs, out=emb_out[r], stream=s)

    # prefill GEMM: 512 and 2048 prompt rows through a 4096 x 4096 projection
    gemm_w = [tuple(torch.from_numpy(a.view(np.int32) if a.dtype == np.uint32 else a).cuda()
                    for a in (w.Bq, w.scales, w.zeros))
              for w in (I.quant_weights(4096, 4096, gs, 1600, 90 + r) for r in range(2))]
    gemm_rows = (512, 2048)
    gemm_A = {Mg: torch.from_numpy(I.activations(Mg, 4096, 1600, 91)).cuda() for Mg in gemm_rows}
    gemm_C = {Mg: torch.empty((Mg, 4096), dtype=torch.float32, device="cuda") for Mg in gemm_rows}
    t_gemm = {}
    for Mg in gemm_rows:
        ws = torch.empty(gq4.gemm_workspace_bytes(Mg, 4096), dtype=torch.uint8, device="cuda")

        def gemm(s, Mg=Mg, ws=ws):
            for r in range(2):
                gq4.gemm(gemm_A[Mg], *gemm_w[r], gs, C=gemm_C[Mg], workspace=ws, stream=s)
        t_gemm[Mg] = time_graph(gemm) / 2

    pairs = R // 2
    t_emb = time_graph(embed) / 2
    t_quant = time_graph(quantize) / 2
    t_mlx = time_graph(convert) / Rm
    t_dual = time_graph(dual) / pairs
    t_two = time_graph(two_matvecs) / pairs
    t_plain = time_graph(plain) / R
    t_sig = time_graph(sigmoid) / R
    t_swi = time_graph(swiglu) / R
    rows = [
        ("dual 4096 -> 2 x 4096", t_dual, 2 * mat_bytes + 4 * K + 8 * N,
         {"two_matvecs_us": round(t_two, 3)}),
        ("sigmoid-gated input 4096 -> 4096", t_sig, mat_bytes + 8 * K + 4 * N,
         {"plain_matvec_us": round(t_plain, 3)}),
        ("swiglu-gated input 4096 -> 4096", t_swi, mat_bytes + 8 * K + 4 * N,
         {"plain_matvec_us": round(t_plain, 3)}),
        ("quantize f32 4096 -> 11008 (gs %d)" % gs, t_quant,
         Kq * Nq * 4 + Kq * Nq // 2 + 8 * Nq * Gq, {"weight_sets": 2}),
        ("MLX convert 4096 -> 11008 (gs %d)" % gs, t_mlx, 2 * mlx_set,
         {"weight_sets": Rm}),
        ("embedding 8192 tokens from 32000 x 4096 (gs %d)" % gs, t_emb,
         Te * (Kq // 2 + 8 * (Kq // gs) + 4 * Kq + 4), {"weight_sets": 1, "outputs": 2}),
    ]
    tpeak, tpeak_src = bf16_peak()
    for Mg in gemm_rows:
        flops = 2.0 * Mg * 4096 * 4096
        tf = flops / (t_gemm[Mg] * 1e-6) / 1e12
        print(json.dumps({"extra": f"gemm {Mg} x 4096 -> 4096 (gs {gs})", "rows": Mg,
                          "group_size": gs, "us_per_call": round(t_gemm[Mg], 3),
                          "TFLOP/s": round(tf, 1), "frac_of_bf16_peak": round(tf / tpeak, 4),
                          "peak": tpeak, "peak_source": tpeak_src, "weight_sets": 2,
                          "timing": "CUDA graph of 2 calls, CUDA events"}))
    for name, us, nbytes, extra in rows:
        gbs = nbytes / (us * 1e-6) / 1e9
        print(json.dumps({"extra": name, "lanes": 1, "group_size": gs, "us_per_call": round(us, 3),
                          "bytes_per_call": nbytes, "GB/s": round(gbs, 1),
                          "frac_of_hbm_peak": round(gbs / peak, 4), "peak": peak,
                          "peak_source": peak_src, "weight_sets": R,
                          "timing": "CUDA graph over rotating weight sets > 4x L2, CUDA events",
                          **extra}))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--lanes", type=int, default=1, help="decode lanes M (1..32)")
    ap.add_argument("--layers", type=int, default=32)
    ap.add_argument("--roofline-rounds", type=int, default=3)
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-config entries (configs 0-3, the stack at more lanes, "
                         "the prefill GEMM, the sequence kernel)")
    ap.add_argument("--stack-lanes", type=int, nargs="*", default=[4, 16, 32],
                    help="lane counts of the extra stack entries")
    ap.add_argument("--profile", choices=["gated", "down", "quad", "o", "step", "gemm"], default=None,
                    help="run a small launch sequence of one kernel for ncu (no timing)")
    ap.add_argument("--extras", action="store_true",
                    help="time the dual, gated-input, GEMM, quantizer, MLX and embedding "
                         "entry points (one JSON line each)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours" and args.profile is None:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    rank, world, local_rank = dist_env()
    if args.extras:
        run_extras(args)
    elif args.profile:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
