"""Decode-step benchmark of the quantized KV cache on GB300.

One step = one pass of the decode hot path over the whole batch:
kvq_append (the new token; the residual flush every R tokens is part of it)
followed by kvq_decode_attention over the packed cache.  The prompt is
quantized once per cache before timing (kvq_quantize_prefill, also timed
separately and reported under "prefill").

Workload (default): the Llama-2-7B-shaped layer -- batch 8, 32 heads,
head_dim 128, 4096-token prompt, 2-bit, G=32, v_group=32, R=128, then 256
streamed appends, each followed by a decode.  The appended steps replay in
epochs of 256: a CUDA graph holds one epoch for every cache copy with the
counters of that epoch, so every replay rewrites the same residual slots and
flushes (the cache returns to its post-prompt state, context 4097..4352).
Several cache copies are used in rotation so the bytes touched between two
uses of one copy exceed 3x the L2 size (no L2 flush needed).

Prints one JSON line.  --impl reference times the CPU oracle instead (the
plain C reference of the method, on the host cores, bounded sample).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_kv_cache_14_gb300 import synth  # noqa: E402

METRIC = "quantized-KV decode attention: KV GB/s read (% of GB300 HBM peak), µs/step"
EPOCH = 256  # streamed appends per replayed epoch


# ---------------------------------------------------------------------------
# bytes of one decode step (algorithmic: what the kernel must read)
# ---------------------------------------------------------------------------

def head_counts(w, n, prompt=None):
    """(n_quant, n_resid, n_sink, n_vq) of one sequence holding n tokens (the
    cache's counting rules: KIVI residual n mod R, value queue max(0, n-R+1);
    InnerQ sinks, then window, then quantized)."""
    if w.scheme == synth.KIVI:
        nr = n % w.residual
        nq = n - nr
        nvq = max(0, n - w.residual + 1) if w.v_queue else nq
        return nq, nr, 0, nvq
    ns = min(n, w.n_sink)
    nw = min(n - ns, w.residual)
    return n - ns - nw, nw, ns, n - ns - nw


def head_bytes(w, nq, nr, ns, nvq=None):
    """Algorithmic bytes one decode reads for one KV head: key and value codes,
    their scales and zeros (fp32, or fp16 with fp16 statistics), outlier lists
    (4 bytes an entry), and the fp16 rows (sinks, residual / window, and under
    the value queue the values still waiting)."""
    nvq = nq if nvq is None else nvq
    d, b = w.head_dim, w.bits
    m = 2 if w.meta_f16 else 4
    if w.scheme == synth.KIVI:
        kmeta = (nq // w.k_group) * d * 2 * m
    else:
        kmeta = nq * (d // w.k_group) * 2 * m
    keys = nq * d * b // 8 + kmeta + nq * w.outliers * 4 + (nr + ns) * d * 2
    n = nq + nr + ns
    values = nvq * d * b // 8 + nvq * (d // w.v_group) * 2 * m + nvq * w.outliers * 4 + \
        (n - nvq) * d * 2
    return keys + values


def decode_bytes(w, n_quant, n_resid, n_sink):
    """All heads at uniform counters (the value queue's count follows)."""
    n = n_quant + n_resid + n_sink
    nvq = head_counts(w, n)[3] if w.v_queue else n_quant
    return w.batch * w.n_kv_heads * head_bytes(w, n_quant, n_resid, n_sink, nvq)


def decode_bytes_ragged(w, lengths):
    """All heads, each sequence with its own length."""
    return w.n_kv_heads * sum(head_bytes(w, *head_counts(w, int(n))) for n in lengths)


def kivi_states(w, n0, r0, steps):
    """(n_quant, n_resid) after each append, starting from (n0, r0)."""
    out, nq, nr = [], n0, r0
    for _ in range(steps):
        if nr + 1 == w.residual:
            nq, nr = nq + w.residual, 0
        else:
            nr += 1
        out.append((nq, nr))
    return out


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.lines = index, None, []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [l for t, l in self.lines if t0 - 0.15 <= t <= t1 + 0.15] or [l for _, l in self.lines]
        sm, smax, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# sources of the timed kernels (their hash ties a committed ncu summary to them)
DECODE_SOURCES = ("kvq_decode_tc.cuh", "kvq_decode_tc.cu", "kvq_tc_common.cuh", "kvq_rope.cuh",
                  "kvq_internal.cuh")
ROPE_SOURCES = ("kvq_decode_tc.cuh", "kvq_decode_tc_rope.cu", "kvq_tc_common.cuh", "kvq_rope.cuh",
                "kvq_internal.cuh")
GQA_SOURCES = ("kvq_decode_gqa.cuh", "kvq_decode_gqa.cu", "kvq_decode_gqa_iq.cu",
               "kvq_decode_gqa_f16.cu", "kvq_decode_gqa_iq16.cu", "kvq_tc_common.cuh",
               "kvq_internal.cuh")


def decode_source_sha(names=DECODE_SOURCES):
    h = hashlib.sha256()
    for name in names:
        if not os.path.exists(os.path.join(ROOT, "bit_kv_cache_14_gb300", "csrc", name)):
            continue
        with open(os.path.join(ROOT, "bit_kv_cache_14_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def decode_kernel_name(w, rope=False):
    """The decode kernel the library launches for this shape (its own answer,
    kvq_decode_kernel_name / kvq_rope_kernel_name, without the template
    arguments)."""
    from bit_kv_cache_14_gb300 import kvq
    cfg = kvq.config_of(w)
    name = kvq.rope_kernel_name(cfg, 1) if rope else kvq.decode_kernel_name(cfg, 1)
    return name.split("<")[0]


def profiled_traffic(workload, per_launch_units, rope=False, kernel="tc_decode_kernel"):
    """DRAM bytes per decode launch from the committed ncu summary, or None when
    the kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", ("decode_rope_%s.md" if rope else "decode_%s.md")
                        % workload)
    try:
        text = open(path).read()
    except OSError:
        return None
    sha = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    tb = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    sources = (ROPE_SOURCES if rope else GQA_SOURCES if kernel == "tc_gqa_kernel"
               else DECODE_SOURCES)
    if not sha or not tb or sha.group(1) != decode_source_sha(sources):
        return None
    return float(tb.group(1))


# ---------------------------------------------------------------------------
# whole-job figures over ranks (one process per GPU, weak scaling)
# ---------------------------------------------------------------------------

def max_over_ranks(values, world, device):
    """Each rank's timings -> their maxima over all ranks (one all_reduce MAX;
    NCCL on the GPUs, gloo in the CPU tests)."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_gbs(bytes_per_rank, world, elapsed_ms):
    """Every rank streams bytes_per_rank (replicas: per-GPU work fixed as N
    grows); the job lasts as long as its slowest rank."""
    return bytes_per_rank * world / (elapsed_ms * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------

def oracle_decode_rate(w, seconds=12.0, n_heads=None, rope_base=None, threads=None):
    """Times the CPU oracle's decode step (append + fp64 attention; with
    rope_base, attention over keys cached before the rotary embedding) on a
    sample of KV heads for about `seconds`; returns (bytes/s scaled to the
    whole batch, threads, description)."""
    import oracle  # only the CPU-baseline leg imports the oracle
    from concurrent.futures import ThreadPoolExecutor

    threads = threads or max(1, len(os.sched_getaffinity(0)))
    BH = w.batch * w.n_kv_heads
    n_heads = min(BH, n_heads or max(threads, 16))
    heads = [(i // w.n_kv_heads, i % w.n_kv_heads) for i in
             np.linspace(0, BH - 1, n_heads).astype(int)]
    cap = w.ctx + EPOCH
    objs = {}

    def make(bh):
        b, h = bh
        o = oracle.OracleHead.for_workload(w, cap=cap)
        K, V = synth.head_tokens(w, b, h, 0, w.ctx)
        o.prefill(K, V)
        k, v = synth.head_tokens(w, b, h, 1, EPOCH, first_token=w.ctx)
        objs[bh] = (o, k, v)

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(make, heads))
    tau = 1.0 / math.sqrt(w.head_dim)
    rg = w.group_ratio
    qs = [synth.queries(w, s) for s in range(4)]

    def one_step(bh, s):
        o, k, v = objs[bh]
        o.append(k[s], v[s])
        b, h = bh
        for hq in range(h * rg, (h + 1) * rg):
            if rope_base is None:
                o.attend(qs[s % 4][b, hq], tau)
            else:
                o.attend_rope(qs[s % 4][b, hq], tau, rope_base)

    steps, t0 = 0, time.perf_counter()
    byte_sum = 0.0
    with ThreadPoolExecutor(threads) as ex:
        while time.perf_counter() - t0 < seconds and steps < EPOCH:
            list(ex.map(lambda bh: one_step(bh, steps), heads))
            o0 = objs[heads[0]][0]
            byte_sum += decode_bytes(w, o0.n_quant, o0.n_resid, o0.n_sink_used) * n_heads / BH
            steps += 1
    dt = time.perf_counter() - t0
    desc = ("%d decode steps (append + fp64 attention%s) of %d of the %d KV heads "
            "(%d query heads each), %d threads, scaled to the whole batch by bytes"
            % (steps, "" if rope_base is None else " over keys rotated by position", n_heads,
               BH, rg, threads))
    return byte_sum / dt, threads, desc, steps


def oracle_reference_rate(w, steps, warmup, rope_base=None):
    """The reference arm: `warmup` untimed then `steps` timed decode steps of
    the CPU oracle.  A step is one append + fp64 attention on a bounded sample
    of KV heads, one head per host thread; the heads rewind to their prompt
    state every EPOCH steps like the GPU arm's replayed epochs.  Returns
    (bytes/s scaled to the whole batch, threads, description)."""
    import oracle  # only the reference arm and the CPU-baseline leg import the oracle
    from concurrent.futures import ThreadPoolExecutor

    threads = max(1, len(os.sched_getaffinity(0)))
    BH = w.batch * w.n_kv_heads
    n_heads = min(BH, threads)
    heads = [(i // w.n_kv_heads, i % w.n_kv_heads) for i in
             np.linspace(0, BH - 1, n_heads).astype(int)]
    cap = w.ctx + EPOCH
    objs = {}

    def make(bh):
        b, h = bh
        o = oracle.OracleHead.for_workload(w, cap=cap)
        K, V = synth.head_tokens(w, b, h, 0, w.ctx)
        o.prefill(K, V)
        k, v = synth.head_tokens(w, b, h, 1, EPOCH, first_token=w.ctx)
        objs[bh] = (o, k, v, o.save_state())

    tau = 1.0 / math.sqrt(w.head_dim)
    rg = w.group_ratio
    qs = [synth.queries(w, s) for s in range(4)]

    def one_step(bh, e):
        o, k, v, st = objs[bh]
        if e == 0:
            o.load_state(st)
        o.append(k[e], v[e])
        b, h = bh
        for hq in range(h * rg, (h + 1) * rg):
            if rope_base is None:
                o.attend(qs[e % 4][b, hq], tau)
            else:
                o.attend_rope(qs[e % 4][b, hq], tau, rope_base)

    byte_sum, t0 = 0.0, None
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(make, heads))
        for i in range(warmup + steps):
            if i == warmup:
                t0 = time.perf_counter()
            e = i % EPOCH
            list(ex.map(lambda bh: one_step(bh, e), heads))
            if i >= warmup:
                o0 = objs[heads[0]][0]
                byte_sum += decode_bytes(w, o0.n_quant, o0.n_resid, o0.n_sink_used) * n_heads / BH
    dt = time.perf_counter() - t0
    desc = ("%d timed decode steps (append + fp64 attention) of %d of the %d KV heads "
            "(%d query heads each), one per thread, %d threads, scaled to the whole batch "
            "by bytes" % (steps, n_heads, BH, rg, threads))
    return byte_sum / dt, threads, desc


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args, w, rank, world):
    import torch
    from bit_kv_cache_14_gb300 import kvq

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    max_ctx = w.ctx + EPOCH
    cfg = kvq.config_of(w, max_ctx)
    K, V = synth.prompt(w)
    Kd, Vd = torch.from_numpy(K).to(dev), torch.from_numpy(V).to(dev)
    torch.cuda.synchronize(dev)  # (copied on the default stream; the prefill uses `stream`)
    del K, V
    prompt_bytes_in = 2 * Kd.numel() * 2

    one = kvq.QuantizedKVCache(cfg, dev)
    cache_bytes = sum(t.numel() for t in one.bufs.values())
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    copies = max(2, math.ceil(3 * l2 / max(1, decode_bytes(w, w.ctx, 0, 0))) + 1)
    # small parity workloads: at most 64 copies, and the line says the working
    # set stays in L2 (see l2_policy)
    copies = min(copies, 64)
    caches = [one] + [kvq.QuantizedKVCache(cfg, dev) for _ in range(copies - 1)]

    # prefill (timed once per copy, plain launches)
    pre_ms = []
    with torch.cuda.stream(stream):
        for c in caches:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            c.prefill(Kd, Vd, stream)
            e1.record(stream)
            e1.synchronize()
            pre_ms.append(e0.elapsed_time(e1))
    del Kd, Vd
    n0, r0, s0 = caches[0].n_quant, caches[0].n_resid, caches[0].n_sink
    states = [(c.n_quant, c.n_resid, c.n_sink, c.ring_head, c.n_appended) for c in caches]

    Ks, Vs = synth.streamed(w, EPOCH)
    ks = torch.from_numpy(Ks).to(dev)
    vs = torch.from_numpy(Vs).to(dev)
    qs = torch.from_numpy(np.stack([synth.queries(w, s) for s in range(8)])).to(dev)
    outs = [torch.empty(qs.shape[1:], dtype=torch.float32, device=dev) for _ in caches]
    scale = 1.0 / math.sqrt(w.head_dim)

    def restore():
        for c, st in zip(caches, states):
            (c.view.n_quant, c.view.n_resid, c.view.n_sink, c.view.ring_head,
             c.view.n_appended) = st

    rope = args.rope_base

    def step(i):
        """One decode step (append + attend); returns the kernels it launched."""
        c = i % copies
        e = (i // copies) % EPOCH
        if rope is None:
            caches[c].append_decode(ks[e], vs[e], qs[e % 8], outs[c], scale, stream)
            return caches[c].last_launch_count()
        caches[c].append(ks[e], vs[e], stream)
        n = caches[c].last_launch_count()
        caches[c].decode_rope(qs[e % 8], rope, outs[c], scale, stream)
        return n + caches[c].last_launch_count()

    # per-step algorithmic bytes over one epoch (identical for every copy)
    if w.scheme == synth.KIVI:
        ep_states = kivi_states(w, n0, r0, EPOCH)
        ep_bytes = [decode_bytes(w, nq, nr, 0) for nq, nr in ep_states]
    else:
        ep_bytes = [decode_bytes(w, n0 + i + 1, r0, s0) for i in range(EPOCH)]

    # graph of one epoch for every copy: EPOCH * copies steps
    P = EPOCH * copies
    graph = torch.cuda.CUDAGraph()
    restore()
    with torch.cuda.stream(stream):
        step(0)  # warm the library (function attributes) outside capture
    stream.synchronize()
    restore()
    ep_launches = 0
    with torch.cuda.graph(graph, stream=stream):
        for i in range(P):
            ep_launches += step(i)
    restore()

    K_steps, W_steps = args.steps, args.warmup
    n_full, rem = divmod(K_steps, P)
    rem_graph = None
    rem_launches = 0
    if rem:
        rem_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(rem_graph, stream=stream):
            for i in range(rem):
                rem_launches += step(i)
        restore()
    timed_launches = n_full * ep_launches + rem_launches

    # warm-up: at least W steps, in whole epochs, then the remainder graph
    # once (a graph's first launch uploads it to the device: not a step's cost)
    warm_replays = max(1, math.ceil(W_steps / P))
    with torch.cuda.stream(stream):
        for _ in range(warm_replays):
            graph.replay()
        if rem_graph is not None:
            rem_graph.replay()
    stream.synchronize()

    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n_full):
            graph.replay()
        if rem_graph is not None:
            rem_graph.replay()
        e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = e0.elapsed_time(e1)

    # bytes of exactly the K timed steps
    total_bytes = sum(ep_bytes[(i // copies) % EPOCH] for i in range(K_steps))

    # decode kernel alone: a graph of decode launches over the copies (state:
    # post-prompt + one appended token), timed with events on the same stream
    restore()
    with torch.cuda.stream(stream):
        for c in caches:
            c.append(ks[0], vs[0], stream)
    stream.synchronize()
    dstate_bytes = decode_bytes(w, caches[0].n_quant, caches[0].n_resid, caches[0].n_sink)
    M = max(copies * 32, 256)
    dgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(dgraph, stream=stream):
        for i in range(M):
            if rope is None:
                caches[i % copies].decode(qs[i % 8], outs[i % copies], scale, stream)
            else:
                caches[i % copies].decode_rope(qs[i % 8], rope, outs[i % copies], scale, stream)
    with torch.cuda.stream(stream):
        dgraph.replay()
        stream.synchronize()
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        for _ in range(4):
            dgraph.replay()
        d1.record(stream)
    d1.synchronize()
    decode_ms = d0.elapsed_time(d1) / (4 * M)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)

    # plain launches (no graph), one step per Python call: host-launch cost
    restore()
    n_plain = min(K_steps, 2 * P) if K_steps >= 8 else K_steps
    with torch.cuda.stream(stream):
        stream.synchronize()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        for i in range(n_plain):
            if i % P == 0:
                restore()
            step(i)
        p1.record(stream)
    p1.synchronize()
    plain_ms = p0.elapsed_time(p1) / max(1, n_plain)

    # end to end through the host-buffer entry point: every step copies one
    # pinned host block [k | v | q] in and the output rows back out, rotating
    # over the same cache copies as the timed steps (an HBM-sized working set)
    restore()
    nin = caches[0].step_input_halves()
    d_in = torch.empty(nin, dtype=torch.float16, device=dev)
    d_out = torch.empty(qs.shape[1:], dtype=torch.float32, device=dev)
    qs_host = qs.cpu()
    h_in = torch.empty((EPOCH, nin), dtype=torch.float16).pin_memory()
    for e in range(EPOCH):
        h_in[e] = torch.cat([torch.from_numpy(Ks[e]).reshape(-1),
                             torch.from_numpy(Vs[e]).reshape(-1), qs_host[e % 8].reshape(-1)])
    h_out = torch.empty(qs.shape[1:], dtype=torch.float32).pin_memory()
    n_e2e = min(P, max(K_steps, 256))
    kvn = ks[0].numel()

    def host_step(i):
        c = caches[i % copies]
        e = (i // copies) % EPOCH
        if rope is None:
            c.decode_step_host(h_in[e], h_out, d_in, d_out, scale, stream)
            return
        # the same single copy in and out around the binding's two calls
        d_in.copy_(h_in[e], non_blocking=True)
        c.append(d_in[:kvn].view(ks.shape[1:]), d_in[kvn:2 * kvn].view(ks.shape[1:]), stream)
        c.decode_rope(d_in[2 * kvn:].view(qs.shape[1:]), rope, d_out, scale, stream)
        h_out.copy_(d_out, non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(8):  # warm-up
            host_step(i)
        stream.synchronize()
        restore()
        # plain calls, one per step (each a library call enqueueing its two
        # copies and its kernels)
        x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x0.record(stream)
        e2e_bytes = 0
        for i in range(n_e2e):
            host_step(i)
            e2e_bytes += ep_bytes[(i // copies) % EPOCH]
        x1.record(stream)
    x1.synchronize()
    e2e_plain_ms = x0.elapsed_time(x1)
    # a serving loop's form: every step still copies its [k|v|q] block from
    # pinned host memory and its output rows back, but the copies run on two
    # side streams with double-buffered staging (step i+1's input copy and
    # step i-1's output copy overlap step i's kernels), ordered by events;
    # the steps are captured in a CUDA graph and replayed
    cs_in, cs_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    d_ins = [torch.empty(nin, dtype=torch.float16, device=dev) for _ in range(2)]
    d_outs = [torch.empty(qs.shape[1:], dtype=torch.float32, device=dev) for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_k = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def piped_step(i):
        b = i % 2
        c = caches[i % copies]
        e = (i // copies) % EPOCH
        if i >= 2:
            cs_in.wait_event(ev_k[b])  # step i-2's kernels are done with d_ins[b]
        with torch.cuda.stream(cs_in):
            d_ins[b].copy_(h_in[e], non_blocking=True)
            ev_in[b].record(cs_in)
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])  # step i-2's output copy is done with d_outs[b]
        k_ = d_ins[b][:kvn].view(ks.shape[1:])
        v_ = d_ins[b][kvn:2 * kvn].view(ks.shape[1:])
        q_ = d_ins[b][2 * kvn:].view(qs.shape[1:])
        if rope is None:
            c.append_decode(k_, v_, q_, d_outs[b], scale, stream)
        else:
            c.append(k_, v_, stream)
            c.decode_rope(q_, rope, d_outs[b], scale, stream)
        ev_k[b].record(stream)
        cs_out.wait_event(ev_k[b])
        with torch.cuda.stream(cs_out):
            h_out.copy_(d_outs[b], non_blocking=True)
            ev_out[b].record(cs_out)

    restore()
    egraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(egraph, stream=stream):
        cs_in.wait_stream(stream)  # fork the side streams into the capture
        cs_out.wait_stream(stream)
        for i in range(n_e2e):
            piped_step(i)
        stream.wait_stream(cs_in)
        stream.wait_stream(cs_out)
    restore()
    with torch.cuda.stream(stream):
        egraph.replay()
        stream.synchronize()
        y0, y1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        y0.record(stream)
        egraph.replay()
        y1.record(stream)
    y1.synchronize()
    e2e_ms = y0.elapsed_time(y1)
    h2d = nin * 2
    d2h = qs[0].numel() * 4
    for c in caches:
        assert c.device_status() == 0

    # secondary figures: kvq_append alone, plain launches with events around
    # each over one epoch per cache copy, split into steps that store the
    # token and steps that flush (quantize) the residual.  Taken after every
    # figure above; a failure here drops only these.
    def time_appends():
        restore()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        times = {"store": [], "flush": []}
        with torch.cuda.stream(stream):
            for e in range(EPOCH):
                for c in caches:
                    kind = ("flush" if w.scheme == synth.KIVI and c.n_resid + 1 == w.residual
                            else "store")
                    ev0.record(stream)
                    c.append(ks[e], vs[e], stream)
                    ev1.record(stream)
                    ev1.synchronize()
                    times[kind].append(ev0.elapsed_time(ev1) * 1e3)
        restore()
        return {k: {"us_median": float(np.median(v)), "launches": len(v)}
                for k, v in times.items() if v}

    # the same appends captured in a CUDA graph (one epoch of every copy):
    # the kernels without the host launch cost
    def time_append_graph():
        restore()
        ag = torch.cuda.CUDAGraph()
        n = 0
        with torch.cuda.graph(ag, stream=stream):
            for e in range(EPOCH):
                for c in caches:
                    c.append(ks[e], vs[e], stream)
                    n += 1
        restore()
        with torch.cuda.stream(stream):
            ag.replay()
            stream.synchronize()
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            ag.replay()
            g1.record(stream)
        g1.synchronize()
        restore()
        return {"us_per_append": g0.elapsed_time(g1) * 1e3 / n, "launches": n,
                "mix": "every R-th append of a cache flushes (KIVI)"}

    try:
        append_stats = time_appends()
        append_stats["graph"] = time_append_graph()
    except Exception as exc:  # noqa: BLE001 -- secondary figure only
        append_stats = {"error": str(exc)[:200]}
    return dict(warmup_steps=warm_replays * P + rem, elapsed_ms=elapsed_ms, total_bytes=total_bytes,
                decode_ms=decode_ms, timed_launches=timed_launches,
                dstate_bytes=dstate_bytes, plain_ms=plain_ms, e2e_ms=e2e_ms,
                e2e_plain_ms=e2e_plain_ms,
                e2e_bytes=e2e_bytes, n_e2e=n_e2e, h2d=h2d, d2h=d2h, clocks=clocks,
                append=append_stats,
                copies=copies, cache_bytes=cache_bytes, prefill_ms=float(np.median(pre_ms)),
                prompt_bytes_in=prompt_bytes_in, l2=l2,
                ws_cache_total=cache_bytes * copies)


# ---------------------------------------------------------------------------
# the other named workloads: decode kernel alone, one line each
# ---------------------------------------------------------------------------

def prompt_on_device(w, dev):
    """The workload's prompt K, V ([B][H][T][d] fp16) generated head by head on
    the host cores (synth's seeded streams) and copied into device tensors."""
    import torch
    from concurrent.futures import ThreadPoolExecutor

    shape = (w.batch, w.n_kv_heads, w.ctx, w.head_dim)
    Kd = torch.empty(shape, dtype=torch.float16, device=dev)
    Vd = torch.empty(shape, dtype=torch.float16, device=dev)

    def one(idx):
        b, h = divmod(idx, w.n_kv_heads)
        k, v = synth.head_tokens(w, b, h, 0, w.ctx)
        Kd[b, h].copy_(torch.from_numpy(k))
        Vd[b, h].copy_(torch.from_numpy(v))

    with ThreadPoolExecutor(max(1, min(16, len(os.sched_getaffinity(0))))) as ex:
        list(ex.map(one, range(w.batch * w.n_kv_heads)))
    # the copies ran on the default stream; the prefill runs on another one
    torch.cuda.synchronize(dev)
    return Kd, Vd


def measure_config(w, dev, stream, peak):
    """Prefill once per cache copy, append the workload's streamed token, then
    time a CUDA graph of decode launches rotating over the copies (enough
    copies that 3x the L2 is touched between two uses of one, at most 64)."""
    import torch
    from bit_kv_cache_14_gb300 import kvq

    cfg = kvq.config_of(w)
    t0 = time.time()
    Kd, Vd = prompt_on_device(w, dev)
    gen_s = time.time() - t0
    lens = synth.prompt_lengths(w)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_copy = decode_bytes_ragged(w, lens) if w.ragged else decode_bytes(w, w.ctx, 0, 0)
    copies = min(64, max(2, math.ceil(3 * l2 / max(1, per_copy)) + 1))
    caches = [kvq.QuantizedKVCache(cfg, dev) for _ in range(copies)]
    pre_ms = []
    with torch.cuda.stream(stream):
        for c in caches:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if w.ragged:
                c.prefill_ragged(Kd, Vd, lens, stream)
            else:
                c.prefill(Kd, Vd, stream)
            e1.record(stream)
            e1.synchronize()
            pre_ms.append(e0.elapsed_time(e1))
    prompt_bytes = 2 * Kd.numel() * 2 if not w.ragged else \
        2 * int(np.sum(lens)) * w.n_kv_heads * w.head_dim * 2
    del Kd, Vd
    Ks, Vs = synth.streamed(w, max(1, w.n_append))
    k, v = torch.from_numpy(Ks[0]).to(dev), torch.from_numpy(Vs[0]).to(dev)
    q = torch.from_numpy(synth.queries(w, 0)).to(dev)
    outs = [torch.empty(q.shape, dtype=torch.float32, device=dev) for _ in caches]
    scale = 1.0 / math.sqrt(w.head_dim)
    with torch.cuda.stream(stream):
        for c in caches:
            c.append(k, v, stream)
    stream.synchronize()
    c0 = caches[0]
    nbytes = (decode_bytes_ragged(w, c0.seq_lengths()) if w.ragged
              else decode_bytes(w, c0.n_quant, c0.n_resid, c0.n_sink))
    ideal_s = nbytes / (peak * 1e9)
    M = max(2 * copies, min(256, int(0.05 / max(ideal_s, 1e-7))))
    with torch.cuda.stream(stream):
        for i in range(copies):  # warm the library outside capture
            caches[i].decode(q, outs[i], scale, stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(M):
            caches[i % copies].decode(q, outs[i % copies], scale, stream)
    with torch.cuda.stream(stream):
        g.replay()
        stream.synchronize()
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 3
        d0.record(stream)
        for _ in range(reps):
            g.replay()
        d1.record(stream)
    d1.synchronize()
    us = d0.elapsed_time(d1) / (reps * M) * 1e3
    for c in caches:
        assert c.device_status() == 0
    gbs = nbytes / (us * 1e-6) / 1e9
    touched = (copies - 1) * per_copy
    return {
        "kernel": kvq.decode_kernel_name(cfg, c0.n_quant),
        "us": us, "gbs": gbs, "frac": gbs / peak, "algorithmic_bytes_per_launch": nbytes,
        "state": {"n_quant": c0.n_quant, "n_resid": c0.n_resid, "n_sink": c0.n_sink},
        "launches_timed": reps * M,
        "l2_policy": "rotating %d cache copies (%.0f MB touched between uses of one copy vs %.0f "
                     "MB L2)%s" % (copies, touched / 1e6, l2 / 1e6,
                                   "" if touched > l2 else
                                   "; smaller than L2: L2-resident, latency-bound, not an HBM "
                                   "number"),
        "prefill": {"ms": float(np.median(pre_ms)), "bytes_in": prompt_bytes,
                    "gbs_in": prompt_bytes / (float(np.median(pre_ms)) * 1e-3) / 1e9},
        "host_generation_s": gen_s,
    }


# Cache-format options timed on the headline layer (decode kernel alone).
FORMATS = {"meta_f16": dict(meta_f16=True), "outliers_2": dict(outliers=2),
           "value_queue": dict(v_queue=True), "ragged": dict(ragged=True)}


# Derived shapes of the named workloads (decode kernel alone): the
# grouped-query layer with 4-bit codes, and the InnerQ cache on the
# grouped-query layer's shape (B64, 32 query / 8 KV heads, 16384 tokens).
VARIANTS = {"gqa_4bit": ("gqa_2bit", dict(bits=4)),
            "innerq_gqa": ("innerq_1m", dict(batch=64, n_q_heads=32, n_kv_heads=8, ctx=16384))}


def run_configs(names, peak, base=None):
    """names: workloads (base None), FORMATS keys (a base workload), or
    VARIANTS keys (base "variants")."""
    import torch
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    stream = torch.cuda.Stream(dev)
    out = {}
    for name in names:
        if base is None:
            w = synth.WORKLOADS[name]
        elif base == "variants":
            w = synth.scaled(synth.WORKLOADS[VARIANTS[name][0]], **VARIANTS[name][1])
        else:
            w = synth.scaled(base, **FORMATS[name])
        try:
            out[name] = measure_config(w, dev, stream, peak)
            if base == "variants":
                out[name]["workload"] = "%s with %s" % (VARIANTS[name][0], ", ".join(
                    "%s=%s" % kv for kv in sorted(VARIANTS[name][1].items())))
        except Exception as exc:  # noqa: BLE001 -- one config's failure drops only its line
            out[name] = {"error": ("%s: %s" % (type(exc).__name__, exc))[:300]}
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=512)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--workload", default="llama2_7b_2bit", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--skip-cpu", action="store_true", help="omit the cpu_baseline leg")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--configs", default="others",
                    help="comma-separated workloads whose decode kernel is also timed alone "
                         "(one GPU only); 'others' = every named workload but the headline one, "
                         "'none' = skip")
    ap.add_argument("--formats", default="all",
                    help="comma-separated cache-format options timed on the headline workload "
                         "(decode kernel alone; one GPU only): " + ", ".join(sorted(FORMATS)) +
                         "; 'all' or 'none'")
    ap.add_argument("--variants", default="all",
                    help="comma-separated derived shapes timed alone (one GPU only): " +
                         ", ".join(sorted(VARIANTS)) + "; 'all' or 'none'")
    ap.add_argument("--rope-base", type=float, default=None,
                    help="time the variant whose keys are cached before the rotary embedding "
                         "(kvq_decode_attention_rope with this base) instead of the plain decode")
    args = ap.parse_args()
    w = synth.WORKLOADS[args.workload]
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    peak, peak_kind = measured_peak()
    config = {"workload": w.name, "batch": w.batch, "n_q_heads": w.n_q_heads,
              "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "ctx": w.ctx, "bits": w.bits,
              "k_group": w.k_group, "v_group": w.v_group, "residual": w.residual,
              "n_sink": w.n_sink, "appends_per_epoch": EPOCH}
    if args.rope_base is not None:
        config["variant"] = ("keys cached before the rotary embedding (base %g), rotated inside "
                             "the decode kernel" % args.rope_base)

    if args.impl == "reference":
        if rank != 0:
            return
        rate, threads, desc = oracle_reference_rate(w, args.steps, args.warmup, args.rope_base)
        gbs = rate / 1e9
        bytes_step = decode_bytes(w, w.ctx, 1, 0)
        line = {"metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": bytes_step / rate * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic", "impl": "reference",
                "config": config,
                "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads,
                                 "kind": "oracle", "sample": desc},
                "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl")
    r = run_gpu(args, w, rank, world)
    elapsed_ms, e2e_ms = max_over_ranks([r["elapsed_ms"], r["e2e_ms"]], world, "cuda")
    value = whole_job_gbs(r["total_bytes"], world, elapsed_ms)
    decode_gbs = r["dstate_bytes"] / (r["decode_ms"] * 1e-3) / 1e9
    rope = args.rope_base is not None
    traffic = profiled_traffic(w.name, 1, rope=rope, kernel=decode_kernel_name(w, rope))
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": r["warmup_steps"], "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": dict(config, l2_policy=("rotating %d cache copies (%.0f MB touched between "
                       "uses of one copy vs %.0f MB L2)" % (
                           r["copies"], (r["copies"] - 1) * decode_bytes(w, w.ctx, 0, 0) / 1e6,
                           r["l2"] / 1e6)) + (
                           "" if (r["copies"] - 1) * decode_bytes(w, w.ctx, 0, 0) > r["l2"]
                           else "; smaller than L2: L2-resident, not an HBM number"),
                       storage="%d-bit codes + fp32 scale/zero" % w.bits,
                       parallelism="replicas" if world > 1 else "single"),
        "us_per_step": elapsed_ms / args.steps * 1e3,
        "roofline": {"bound": "hbm", "achieved": decode_gbs, "peak": peak, "unit": "GB/s",
                     "frac": decode_gbs / peak, "traffic": traffic,
                     "kernel": decode_kernel_name(w, rope),
                     "kernel_us": r["decode_ms"] * 1e3,
                     "algorithmic_bytes_per_launch": r["dstate_bytes"],
                     "peak_kind": peak_kind},
        "plain_launch_us_per_step": r["plain_ms"] * 1e3,
        "prefill": {"ms": r["prefill_ms"], "bytes_in": r["prompt_bytes_in"],
                    "gbs_in": r["prompt_bytes_in"] / (r["prefill_ms"] * 1e-3) / 1e9},
        "e2e": {"value": whole_job_gbs(r["e2e_bytes"], world, e2e_ms), "unit": "GB/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "us_per_step": e2e_ms / r["n_e2e"] * 1e3, "steps": r["n_e2e"],
                "how": "every step one host-to-device copy of its [k|v|q] block from pinned "
                       "memory, kvq_append_decode, one device-to-host copy of the output; copies "
                       "on two side streams with double-buffered staging so they overlap the "
                       "neighbouring steps' kernels; the steps captured in a CUDA graph and "
                       "replayed.  serial_us_per_step: kvq_decode_step_host (the same copies and "
                       "step in one call on one stream), issued step by step",
                "serial_us_per_step": r.get("e2e_plain_ms", e2e_ms) / r["n_e2e"] * 1e3},
        "append": r.get("append"),
        "gpu_launches": r["timed_launches"],
        "clocks": r["clocks"],
    }
    if world == 1 and args.configs != "none" and args.rope_base is None:
        names = ([n for n in synth.WORKLOADS if n != w.name] if args.configs == "others"
                 else [n for n in args.configs.split(",") if n])
        line["configs"] = run_configs(names, peak)
    if world == 1 and args.formats != "none" and args.rope_base is None:
        names = (sorted(FORMATS) if args.formats == "all"
                 else [n for n in args.formats.split(",") if n])
        line["formats"] = run_configs(names, peak, base=w)
    if world == 1 and args.variants != "none" and args.rope_base is None:
        names = (sorted(VARIANTS) if args.variants == "all"
                 else [n for n in args.variants.split(",") if n])
        line["variants"] = run_configs(names, peak, base="variants")
    if rank == 0 and world == 1 and not args.skip_cpu:
        rate, threads, desc, _ = oracle_decode_rate(w, seconds=args.cpu_seconds,
                                                    rope_base=args.rope_base)
        line["cpu_baseline"] = {"value": rate / 1e9, "unit": "GB/s", "cores": threads,
                                "kind": "oracle", "sample": desc}
        if threads > 1:
            rate1, _, desc1, _ = oracle_decode_rate(w, seconds=args.cpu_seconds / 4,
                                                    rope_base=args.rope_base, threads=1,
                                                    n_heads=16)
            line["cpu_baseline"]["single_thread"] = {"value": rate1 / 1e9, "unit": "GB/s",
                                                     "sample": desc1}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
