#!/usr/bin/env python
"""Decode-step benchmark of the quantized KV-cache library on one node.

One step = for every layer's cache: one kvq_append_decode_attn call, which
quantizes one new K/V token per sequence into the cache and attends over the
whole cache, the new row included (--separate-append: kvq_append then
kvq_decode_attn, the same work in two launches).
Workload (7B-class MHA layer): batch 8, 4096 cached tokens per sequence,
32 query = 32 KV heads, head_dim 128, INT4 group-32 cache, 32 distinct layer
caches per step (5.4 GB working set, far above the 129 MB L2).

value      tokens/s, one token = one sequence through one attention layer
           (B x layers per step), device-timed with CUDA events over a
           CUDA-graph replay of the step, inputs resident in HBM.
e2e        the same metric end to end through the C ABI: every step copies
           its q/k/v from pinned host memory, issues each layer's
           kvq_append_decode_attn call (eagerly, no graph) and copies the
           outputs back, all inside the timed region.  e2e_graph: the same
           with the step's calls replayed from a CUDA graph.
roofline   algorithmic bytes of one step call (cache rows read, the new row
           written, k/v/q in, out) / its average duration, from events around
           a CUDA graph of every layer's call back to back; the fraction is
           given of the measured copy bandwidth and of the nominal 8 TB/s.
cpu_baseline  the CPU oracle on this host's cores: one worker process per
           core over the (sequence, KV head) units of one full layer-step
           (all 8 sequences, 32 heads, 4097 rows), plus a one-thread run on
           one sequence.  Its outputs are also compared with the GPU's.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kvq|reference]
Under torchrun (N > 1) each rank runs its own replica of the workload on its
own GPU (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn tokens/s and achieved KV HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "tokens/s"
WORKLOAD = "mha7b"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def rank_info():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def workload_config(w, bits, layers):
    return {
        "workload": f"{w.name}: batch {w.batch} x {w.ctx[0]} cached tokens (+1 appended), "
                    f"{w.num_q_heads} q / {w.num_kv_heads} kv heads, head_dim {w.head_dim}, "
                    f"{'fp16' if bits == 16 else f'INT{bits} group {w.group_size}'} dense cache, "
                    f"{layers} layer caches per step",
        "batch": w.batch,
        "context": w.ctx[0] + 1,
        "num_q_heads": w.num_q_heads,
        "num_kv_heads": w.num_kv_heads,
        "head_dim": w.head_dim,
        "cache_bits": bits,
        "group_size": w.group_size if bits != 16 else None,
        "layers_per_step": layers,
        "token": "one sequence through one attention layer (append + decode attention)",
        "l2": "inputs larger than L2: every step walks all layer caches",
    }


def kivi_decode_bytes(w, bits, rows, sink):
    """Algorithmic bytes of one fused step call on an axis-aware cache of
    `rows` tokens after the append: quantized rows (codes + V headers), one
    K scale + zero per channel per block, fp16 sink and residual rows, the
    new token's K/V (read, then written to the window), q and out."""
    D, g = w.head_dim, w.group_size
    nb = (rows - sink) // g
    quant = nb * g * (2 * D * bits // 8 + 4 * (D // g)) + nb * 4 * D
    fp16_rows = rows - nb * g
    kv = w.batch * w.num_kv_heads * (quant + fp16_rows * 2 * D * 2 + 2 * D * 2)
    return kv + 2 * w.batch * w.num_q_heads * D * 2


def decode_bytes(w, bits, rows, fused=True, symmetric=False, group_size=None):
    """Algorithmic bytes of one step call.  Decode alone: `rows` cache rows
    (codes + scale/zero, K and V) read, q read, out written.  Fused append:
    rows - 1 cache rows read, the new row written, the new fp16 K/V read."""
    D = w.head_dim
    g = group_size or w.group_size
    per_row = D * bits // 8 + (0 if bits == 16 else (2 if symmetric else 4) * (D // g))
    kv = 2 * w.batch * w.num_kv_heads * rows * per_row
    if fused:
        kv += 2 * w.batch * w.num_kv_heads * D * 2
    return kv + 2 * w.batch * w.num_q_heads * D * 2


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.dev = device_index

    def start(self):
        try:
            import torch
            ident = None
            try:
                ident = "GPU-" + str(torch.cuda.get_device_properties(self.dev).uuid)
            except Exception:
                ident = str(self.dev)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", ident, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline and reference arm)
# ---------------------------------------------------------------------------

NOMINAL_HBM_GBS = 8000.0  # the ~8 TB/s nominal HBM3e bandwidth of one GB300
MODEL_LAYERS = {"mha7b": 32, "gqa_mix": 32, "long": 32, "paged": 24}


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_units(w, k, v, kn, vn, q):
    """The (sequence, KV head) units of one layer-step from fp16 numpy arrays
    k, v [B][L][Hkv][D], kn, vn [B][1][Hkv][D], q [B][Hq][D]."""
    G = w.num_q_heads // w.num_kv_heads
    return [(np.ascontiguousarray(k[b, :, h]), np.ascontiguousarray(v[b, :, h]),
             kn[b, 0, h].copy(), vn[b, 0, h].copy(), q[b, h * G:(h + 1) * G].copy())
            for b in range(k.shape[0]) for h in range(k.shape[2])]


def _oracle_prepare(unit, bits, g):
    """Quantize a unit's cached context once (untimed): the cache the step
    reads."""
    import oracle as O
    k, v, kn, vn, q = unit
    return dict(ctx=[O.quantize_groups(x[None], bits, g) for x in (k, v)], new=(kn, vn), q=q)


def _oracle_step(st, bits, g):
    """The oracle's decode step for one unit: quantize the new token, append
    it, dequantize the cache and attend ([G][D] fp64)."""
    import oracle as O
    hats = []
    for r, new in zip(st["ctx"], st["new"]):
        n = O.quantize_groups(new[None, None], bits, g)
        codes = np.concatenate([r["codes"], n["codes"]], axis=1)
        scale = np.concatenate([r["scale"], n["scale"]], axis=1)
        zero = np.concatenate([r["zero"], n["zero"]], axis=1)
        hats.append(O.dequantize(codes, scale, zero, g)[0])
    q = st["q"].astype(np.float64)
    return O.attend(q, hats[0], hats[1], 1.0 / np.sqrt(q.shape[-1]))


def _oracle_worker(conn, units, bits, g):
    """One host core: prepares its units, then runs one step over all of
    them per request until told to stop."""
    states = [_oracle_prepare(u, bits, g) for u in units]
    conn.send(len(states))
    while conn.recv():
        conn.send([_oracle_step(st, bits, g) for st in states])
    conn.close()


class OraclePool:
    """The oracle over many units on `procs` worker processes (spawned, so
    none inherits a CUDA context; one BLAS thread each).  Unit i runs on
    worker i % procs; step() returns every unit's output in unit order."""

    def __init__(self, units, procs, bits, g):
        import multiprocessing as mp
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        ctx = mp.get_context("spawn")
        self.n = len(units)
        self.procs = max(1, min(procs, self.n))
        self.conns, self.workers = [], []
        for i in range(self.procs):
            parent, child = ctx.Pipe()
            pr = ctx.Process(target=_oracle_worker, args=(child, units[i::self.procs], bits, g),
                             daemon=True)
            pr.start()
            child.close()
            self.conns.append(parent)
            self.workers.append(pr)
        for c in self.conns:
            c.recv()

    def step(self):
        for c in self.conns:
            c.send(True)
        parts = [c.recv() for c in self.conns]
        out = [None] * self.n
        for i, part in enumerate(parts):
            out[i::self.procs] = part
        return out

    def time(self, steps, warmup=1):
        for _ in range(warmup):
            self.step()
        t0 = time.perf_counter()
        for _ in range(steps):
            out = self.step()
        return (time.perf_counter() - t0) / steps, out

    def close(self):
        for c in self.conns:
            try:
                c.send(False)
            except Exception:
                pass
        for pr in self.workers:
            pr.join(timeout=10)


def host_layer(w, seed):
    """One layer-step of host-drawn fp16 inputs of workload w (the reference
    arm; the GPU arm's baseline uses the GPU's own layer-0 inputs)."""
    from quantized_kv_decode_gb300 import synth
    rng = synth.rng_for(seed)
    outl = synth.outlier_channels(rng, w.num_kv_heads, w.head_dim)
    k, v = synth.host_kv(rng, w.batch, w.ctx[0], w.num_kv_heads, w.head_dim, outl)
    kn, vn = synth.host_kv(rng, w.batch, 1, w.num_kv_heads, w.head_dim, outl)
    q = synth.host_q(rng, w.batch, w.num_q_heads, w.head_dim)
    return k, v, kn, vn, q


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on this host's cores,
    over the same workload and metric as the GPU arm.  Each step is one full
    layer-step of the workload (every sequence and head; the cached context
    quantized by the oracle before timing)."""
    rank, world, _ = rank_info()
    if rank != 0:
        return
    from quantized_kv_decode_gb300 import synth
    w = synth.WORKLOADS[WORKLOAD]
    bits = 4
    layers = args.layers or w.layers
    cores = host_cores()
    pool = OraclePool(oracle_units(w, *host_layer(w, w.seed)), cores, bits, w.group_size)
    try:
        t, _ = pool.time(args.steps, args.warmup)
    finally:
        pool.close()
    value = w.batch / t
    sample = (f"one full layer-step per step ({w.batch} sequences x {w.num_kv_heads} KV heads, "
              f"{w.ctx[0] + 1} rows, host-drawn inputs), the context quantized by the oracle "
              f"before timing; {pool.procs} worker processes, one per host core")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(workload_config(w, bits, layers),
                       parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": pool.procs, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(w, bits, layer0, gpu_out0, steps):
    """The oracle on this host: every unit of the GPU's layer-0 step on one
    worker per core (also checked against the GPU's outputs), and the units of
    sequence 0 on one worker."""
    k, v, kn, vn, q = layer0
    units = oracle_units(w, k, v, kn, vn, q)
    cores = host_cores()
    pool = OraclePool(units, cores, bits, w.group_size)
    try:
        t_all, outs = pool.time(steps)
    finally:
        pool.close()
    G = w.num_q_heads // w.num_kv_heads
    ref = np.stack(outs).reshape(w.batch, w.num_kv_heads * G, w.head_dim)
    err = float(np.abs(gpu_out0 - ref).max())
    rel = float(np.linalg.norm(gpu_out0 - ref) / np.linalg.norm(ref))
    one = OraclePool(units[:w.num_kv_heads], 1, bits, w.group_size)
    try:
        t_one, _ = one.time(max(2, steps // 2))
    finally:
        one.close()
    base = {
        "value": w.batch / t_all, "unit": UNIT, "cores": pool.procs, "kind": "oracle",
        "sample": (f"one full layer-step per step (layer 0: {w.batch} sequences x "
                   f"{w.num_kv_heads} KV heads, {w.ctx[0] + 1} rows), {steps} steps, the context "
                   f"quantized by the oracle before timing; one worker process per host core"),
        "one_thread": {"value": 1.0 / t_one, "unit": UNIT, "cores": 1,
                       "sample": "sequence 0 of layer 0 (all heads) per step"}}
    parity = {"max_abs": err, "rel_l2": rel,
              "what": f"layer 0, all {w.batch} sequences and {w.num_q_heads} heads vs the oracle"}
    return base, parity


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def build_layers(w, bits, layers, dev, seed, torch, K, synth, symmetric=False, kivi_sink=None,
                 nf4=False, group_size=None, keep_layer0=False):
    """Populate one cache per layer with device-drawn fp16 K/V; per-layer
    step inputs q, k_new, v_new.  kivi_sink: an axis-aware cache with that
    many fp16 sink tokens; nf4: normal-quantile levels; keep_layer0: also
    return layer 0's fp16 inputs on the host (for the CPU oracle)."""
    import numpy as np
    g = group_size or w.group_size
    align = g if kivi_sink is not None else 16
    cap = ((w.ctx[0] + 1 + align - 1) // align) * align
    desc = K.make_desc(bits, g if bits != 16 else 0, w.num_kv_heads, w.head_dim,
                       K.KVQ_DENSE, cap, symmetric=symmetric, k_per_channel=kivi_sink is not None,
                       sink_tokens=kivi_sink or 0, nf4=nf4)
    zeros = torch.zeros(w.batch, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    caches, qs, kns, vns, host_slices = [], [], [], [], None
    for l in range(layers):
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed * 100003 + l)
        outl = synth.outlier_channels(np.random.default_rng(seed * 100003 + l), w.num_kv_heads,
                                      w.head_dim)
        k, v = synth.device_kv(gen, w.batch, w.ctx[0], w.num_kv_heads, w.head_dim, outl, dev)
        kn, vn = synth.device_kv(gen, w.batch, 1, w.num_kv_heads, w.head_dim, outl, dev)
        q = torch.randn((w.batch, w.num_q_heads, w.head_dim), generator=gen, device=dev).half()
        cache = K.KVCache.allocate(desc, w.batch, dev)
        K.kvq_append(cache, k, v, zeros, status)
        if l == 0 and keep_layer0:
            host_slices = (k.cpu().numpy(), v.cpu().numpy(), kn.cpu().numpy(),
                           vn.cpu().numpy(), q.cpu().numpy())
        del k, v
        caches.append(cache)
        qs.append(q)
        kns.append(kn)
        vns.append(vn)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"populate flagged status {int(status.item()):#x}")
    return desc, caches, qs, kns, vns, host_slices


def run_gpu_arm(args):
    import numpy as np
    import torch

    rank, world, local = rank_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    from quantized_kv_decode_gb300 import build as kbuild
    kbuild.build()
    import quantized_kv_decode_gb300 as K
    from quantized_kv_decode_gb300 import synth

    w = synth.WORKLOADS[WORKLOAD]
    bits = 4
    layers = args.layers or w.layers
    rows = w.ctx[0] + 1
    seed = w.seed + 7919 * rank

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    def max_over_ranks(x):
        return reduce_max_over_ranks(x, world, dev)

    results = {}
    # formats: the headline asymmetric cache first, then the comparators
    kivi_sink = 4
    nf4_group = 64  # the NF4 block size of the weight-quantization page
    formats = [(bits, False, None, False, None)]
    if not args.no_symmetric:
        formats.append((bits, True, None, False, None))
    if not args.no_kivi:
        formats.append((bits, False, kivi_sink, False, None))
    if not args.no_lowbit:
        formats.append((4, False, None, True, nf4_group))
        formats.append((2, False, None, False, None))
    if not args.no_fp16:
        formats.append((16, False, None, False, None))
    for fmt, sym, ksink, nf4, fgroup in formats:
        headline = (fmt == bits and not sym and ksink is None and not nf4)
        desc, caches, qs, kns, vns, host_slices = build_layers(
            w, fmt, layers, dev, seed, torch, K, synth, symmetric=sym, kivi_sink=ksink, nf4=nf4,
            group_size=fgroup, keep_layer0=headline and world == 1 and not args.no_cpu_baseline)
        key = ("sym" if sym else "kivi" if ksink is not None else "nf4" if nf4 else
               "int2" if fmt == 2 else fmt)
        stream = torch.cuda.Stream(device=dev)
        lens_before = torch.full((w.batch,), w.ctx[0], dtype=torch.int32, device=dev)
        lens = lens_before + 1
        splits = K.kvq_decode_num_splits(desc, w.batch, w.num_q_heads, rows, 0)
        ws_bytes = K.kvq_decode_workspace_size(desc, w.batch, w.num_q_heads, rows, 0)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        # per-layer step inputs as views of one buffer (q, then k, then v of
        # every layer), so that a step's inputs arrive in one copy; outputs
        # contiguous across layers
        q_st, k_st, v_st = torch.stack(qs), torch.stack(kns), torch.stack(vns)
        in_all = torch.cat([q_st.reshape(-1), k_st.reshape(-1), v_st.reshape(-1)])
        nq, nk = q_st.numel(), k_st.numel()
        q_all = in_all[:nq].view(q_st.shape)
        k_all = in_all[nq:nq + nk].view(k_st.shape)
        v_all = in_all[nq + nk:].view(v_st.shape)
        del q_st, k_st, v_st
        qs, kns, vns = list(q_all.unbind(0)), list(k_all.unbind(0)), list(v_all.unbind(0))
        o_all = torch.empty_like(q_all)
        outs = list(o_all.unbind(0))

        kn1 = [k[:, 0] for k in kns]   # [B][Hkv][D] views of the step's new K/V
        vn1 = [v[:, 0] for v in vns]

        def call(l, s):
            if args.separate_append:
                K.kvq_decode_attn(caches[l], qs[l], lens, rows, outs[l], ws, status, stream=s)
            else:
                K.kvq_append_decode_attn(caches[l], kn1[l], vn1[l], qs[l], lens_before, rows,
                                         outs[l], ws, status, stream=s)

        def step(s):
            for l in range(layers):
                if args.separate_append:
                    K.kvq_append(caches[l], kns[l], vns[l], lens_before, status, stream=s)
                call(l, s)

        with torch.cuda.stream(stream):
            for _ in range(2):
                step(stream)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step(stream)
        torch.cuda.synchronize()

        with torch.cuda.stream(stream):
            for _ in range(max(args.warmup, 3)):
                graph.replay()
        torch.cuda.synchronize()
        barrier()

        clocks = ClockSampler(dev.index)
        if key == bits:
            # the sampler starts under load: untimed replays for --clock-preroll
            # seconds, then the timed steps, with nvidia-smi sampling throughout
            clocks.start()
            t_end = time.time() + args.clock_preroll
            with torch.cuda.stream(stream):
                while time.time() < t_end:
                    for _ in range(8):
                        graph.replay()
                    torch.cuda.current_stream().synchronize()
            torch.cuda.synchronize()
            barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ms_total = max_over_ranks(e0.elapsed_time(e1))
        clk = clocks.stop() if key == bits else None

        # per-call duration of the step call (kernel + split merge): a graph of
        # every layer's call back to back, timed with events on its stream
        # (repeating a fused call re-writes the same row with the same codes)
        dgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(dgraph, stream=stream):
            for l in range(layers):
                call(l, stream)
        torch.cuda.synchronize()
        reps = max(3, args.steps // 2)
        d0 = torch.cuda.Event(enable_timing=True)
        d1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            dgraph.replay()
            d0.record(stream)
            for _ in range(reps):
                dgraph.replay()
            d1.record(stream)
        torch.cuda.synchronize()
        call_ms = d0.elapsed_time(d1) / (reps * layers)

        # fp16 caches: the same attention by PyTorch's SDPA on the same fp16
        # K/V (a tuned library kernel, for an even INT4-vs-FP16 comparison)
        sdpa_ms = None
        if fmt == 16:
            import torch.nn.functional as F
            kv_views = [(c.k_codes.view(torch.float16)[:, :, :rows],
                         c.v_codes.view(torch.float16)[:, :, :rows]) for c in caches]
            q4 = [q.unsqueeze(2) for q in qs]
            souts = [None] * layers

            def sdpa_all():
                for l in range(layers):
                    souts[l] = F.scaled_dot_product_attention(q4[l], kv_views[l][0], kv_views[l][1])

            with torch.cuda.stream(stream):
                sdpa_all()
            torch.cuda.synchronize()
            sgraph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(sgraph, stream=stream):
                sdpa_all()
            torch.cuda.synchronize()
            g0 = torch.cuda.Event(enable_timing=True)
            g1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                sgraph.replay()
                g0.record(stream)
                for _ in range(reps):
                    sgraph.replay()
                g1.record(stream)
            torch.cuda.synchronize()
            sdpa_ms = g0.elapsed_time(g1) / (reps * layers)
            sdpa_err = float((souts[0].squeeze(2).float() - outs[0].float()).abs().max())
            del sgraph, kv_views
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item()):#x}")

        # end to end: inputs from pinned host memory, outputs back, per step
        h_in = in_all.cpu().pin_memory()
        h_o = torch.empty(o_all.shape, dtype=o_all.dtype, pin_memory=True)
        h2d = h_in.numel() * h_in.element_size()
        d2h = h_o.numel() * h_o.element_size()

        # The step's inputs (q, k, v of every layer) share one buffer and its
        # outputs another, so a step moves them with two copies.
        def e2e_step():
            in_all.copy_(h_in, non_blocking=True)
            graph.replay()
            h_o.copy_(o_all, non_blocking=True)

        # The same step with each layer's call issued through the C ABI every
        # step (no graph): the host path a caller without graphs pays.  The
        # arguments are marshalled once; each call validates, plans and
        # launches.
        from ctypes import byref
        cabi = K._lib.lib()
        sptr = stream.cuda_stream
        ws_b = ws.numel() * ws.element_size()
        cache_ptrs = [c.ptrs for c in caches]
        if args.separate_append:
            eager_calls = []
            for l in range(layers):
                eager_calls.append((cabi.kvq_append, (
                    byref(desc), byref(cache_ptrs[l]), w.batch, 1, kns[l].data_ptr(),
                    vns[l].data_ptr(), lens_before.data_ptr(), status.data_ptr(), sptr)))
                eager_calls.append((cabi.kvq_decode_attn, (
                    byref(desc), byref(cache_ptrs[l]), w.batch, w.num_q_heads, qs[l].data_ptr(),
                    lens.data_ptr(), rows, 0, 0.0, outs[l].data_ptr(), ws.data_ptr(), ws_b,
                    status.data_ptr(), sptr)))
        else:
            eager_calls = [(cabi.kvq_append_decode_attn, (
                byref(desc), byref(cache_ptrs[l]), w.batch, w.num_q_heads, kn1[l].data_ptr(),
                vn1[l].data_ptr(), qs[l].data_ptr(), lens_before.data_ptr(), rows, 0, 0.0,
                outs[l].data_ptr(), ws.data_ptr(), ws_b, status.data_ptr(), sptr))
                for l in range(layers)]

        def e2e_eager_step():
            in_all.copy_(h_in, non_blocking=True)
            for fn, a in eager_calls:
                if fn(*a) != 0:
                    raise RuntimeError("C ABI call failed")
            h_o.copy_(o_all, non_blocking=True)

        def timed(step_fn):
            with torch.cuda.stream(stream):
                for _ in range(2):
                    step_fn()
            torch.cuda.synchronize()
            barrier()
            f0 = torch.cuda.Event(enable_timing=True)
            f1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                f0.record(stream)
                for _ in range(args.steps):
                    step_fn()
                f1.record(stream)
            torch.cuda.synchronize()
            barrier()
            return max_over_ranks(f0.elapsed_time(f1))

        e2e_ms = timed(e2e_eager_step)
        e2e_graph_ms = timed(e2e_step)
        # host time to issue one call through the C ABI (validation, planning,
        # launch), the calls enqueued back to back without waiting
        torch.cuda.synchronize()
        n_issue = 0
        h0 = time.perf_counter()
        for _ in range(max(1, min(args.steps, 10))):
            for fn, a in eager_calls:
                fn(*a)
                n_issue += 1
        host_us = (time.perf_counter() - h0) / n_issue * 1e6
        torch.cuda.synchronize()

        tokens = w.batch * layers * args.steps  # per rank
        results[key] = dict(
            value=job_throughput(tokens, world, ms_total), ms_per_step=ms_total / args.steps,
            e2e=job_throughput(tokens, world, e2e_ms),
            e2e_graph=job_throughput(tokens, world, e2e_graph_ms), host_us=host_us, h2d=h2d, d2h=d2h,
            call_ms=call_ms,
            splits=splits,
            bytes=(kivi_decode_bytes(w, fmt, rows, ksink) if ksink is not None else
                   decode_bytes(w, fmt, rows, not args.separate_append, sym or nf4, fgroup)),
            clocks=clk,
            host_slices=host_slices, out0=outs[0].float().cpu().numpy(),
            sdpa_ms=sdpa_ms, sdpa_err=sdpa_err if sdpa_ms is not None else None,
            launches=args.steps * layers * ((2 if args.separate_append else 1) +
                                            (1 if splits > 1 else 0)))
        del caches, graph, dgraph
        torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    r = results[bits]
    peak, peak_kind = measured_peaks()
    workloads = (run_workloads(dev, torch, K, synth, peak, args.steps)
                 if world == 1 and not args.no_workloads else None)
    achieved = r["bytes"] / (r["call_ms"] / 1e3) / 1e9
    traffic = load_profiled_traffic()
    line = {
        "metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": dict(workload_config(w, bits, layers),
                       parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "peak_nominal": NOMINAL_HBM_GBS, "frac_nominal": achieved / NOMINAL_HBM_GBS,
                     "traffic": traffic,
                     "kernel": ("kvq_decode_attn" if args.separate_append else
                                "kvq_append_decode_attn") + " (decode kernel + split merge)",
                     "splits": r["splits"],
                     "bytes_per_launch": r["bytes"], "avg_launch_us": r["call_ms"] * 1e3},
        "model_tokens_per_s": {
            "value": r["value"] / MODEL_LAYERS[WORKLOAD], "layers": MODEL_LAYERS[WORKLOAD],
            "what": "value / the 7B-class model's layer count: decode tokens per second of a "
                    "whole model's attention (one token = one sequence through every layer)"},
        "e2e": {"value": r["e2e"], "unit": UNIT, "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"],
                "host_us_per_call": r["host_us"],
                "what": "eager C-ABI calls per layer, host copies in and out, per step; "
                        "host_us_per_call: host time to issue one call through ctypes"},
        "e2e_graph": {"value": r["e2e_graph"], "unit": UNIT, "h2d_bytes_per_step": r["h2d"],
                      "d2h_bytes_per_step": r["d2h"],
                      "what": "the same with the step's calls replayed from a CUDA graph"},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    if "sym" in results:
        f = results["sym"]
        line["symmetric_cache"] = {
            "value": f["value"], "unit": UNIT, "ms_per_step": f["ms_per_step"],
            "achieved_gbs": f["bytes"] / (f["call_ms"] / 1e3) / 1e9,
            "frac": f["bytes"] / (f["call_ms"] / 1e3) / 1e9 / peak,
            "frac_nominal": f["bytes"] / (f["call_ms"] / 1e3) / 1e9 / NOMINAL_HBM_GBS,
            "bytes_per_launch": f["bytes"], "avg_launch_us": f["call_ms"] * 1e3,
            "e2e": f["e2e"], "speedup_vs_asymmetric": f["value"] / r["value"],
            "what": "the same step over symmetric INT4 g32 caches (2-byte scale per group, "
                    "no zero-point)"}
    if "kivi" in results:
        f = results["kivi"]
        line["kivi_cache"] = {
            "value": f["value"], "unit": UNIT, "ms_per_step": f["ms_per_step"],
            "achieved_gbs": f["bytes"] / (f["call_ms"] / 1e3) / 1e9,
            "frac": f["bytes"] / (f["call_ms"] / 1e3) / 1e9 / peak,
            "frac_nominal": f["bytes"] / (f["call_ms"] / 1e3) / 1e9 / NOMINAL_HBM_GBS,
            "bytes_per_launch": f["bytes"], "avg_launch_us": f["call_ms"] * 1e3,
            "e2e": f["e2e"], "speedup_vs_asymmetric": f["value"] / r["value"],
            "what": f"the same step over axis-aware INT4 caches: K per channel over blocks of "
                    f"{w.group_size} tokens, V per token, {kivi_sink} fp16 sink tokens and the fp16 "
                    f"residual window; the step call is the append kernels + decode"}
    for key, what in (("nf4", f"NF4-style caches: 4-bit codes indexing 16 normal-quantile levels, "
                               f"one fp16 absmax scale per {nf4_group} channels; tensor-core decode "
                               f"kernel, codes to fp16 levels by a byte-permute lookup"),
                      ("int2", f"asymmetric INT2 g{w.group_size} caches (four codes per byte); "
                               f"tensor-core decode kernel")):
        if key in results:
            f = results[key]
            line[f"{key}_cache"] = {
                "value": f["value"], "unit": UNIT, "ms_per_step": f["ms_per_step"],
                "achieved_gbs": f["bytes"] / (f["call_ms"] / 1e3) / 1e9,
                "frac": f["bytes"] / (f["call_ms"] / 1e3) / 1e9 / peak,
                "frac_nominal": f["bytes"] / (f["call_ms"] / 1e3) / 1e9 / NOMINAL_HBM_GBS,
            "frac_nominal": f["bytes"] / (f["call_ms"] / 1e3) / 1e9 / NOMINAL_HBM_GBS,
                "bytes_per_launch": f["bytes"], "avg_launch_us": f["call_ms"] * 1e3,
                "e2e": f["e2e"], "speedup_vs_asymmetric": f["value"] / r["value"], "what": what}
    if 16 in results:
        f = results[16]
        sdpa_bytes = decode_bytes(w, 16, rows, fused=False)
        line["fp16_cache"] = {
            "value": f["value"], "unit": UNIT, "ms_per_step": f["ms_per_step"],
            "achieved_gbs": f["bytes"] / (f["call_ms"] / 1e3) / 1e9,
            "frac": f["bytes"] / (f["call_ms"] / 1e3) / 1e9 / peak,
            "frac_nominal": f["bytes"] / (f["call_ms"] / 1e3) / 1e9 / NOMINAL_HBM_GBS,
            "bytes_per_launch": f["bytes"], "avg_launch_us": f["call_ms"] * 1e3,
            "what": "the same step over fp16 caches through this library (tensor-core fp16 kernel)",
            "sdpa": {"avg_launch_us": f["sdpa_ms"] * 1e3,
                     "achieved_gbs": sdpa_bytes / (f["sdpa_ms"] / 1e3) / 1e9,
                     "frac": sdpa_bytes / (f["sdpa_ms"] / 1e3) / 1e9 / peak,
                     "max_abs_vs_library_fp16": f["sdpa_err"],
                     "what": "torch.nn.functional.scaled_dot_product_attention on the same fp16 "
                             "K/V (decode only, no append), per layer call"},
            "speedup_int4_vs_fp16_sdpa_per_call": f["sdpa_ms"] / r["call_ms"],
            "speedup_int4_vs_fp16_library_step": r["value"] / f["value"]}
    if workloads:
        line["workloads"] = workloads
    if world == 1 and not args.no_cpu_baseline:
        base, parity = cpu_baseline(w, bits, r["host_slices"], r["out0"], args.cpu_steps)
        line["cpu_baseline"] = base
        line["parity_sample"] = parity
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_workloads(dev, torch, K, synth, peak, steps):
    """The other workloads of the build, one fused step call per layer cache
    (append the step's token, then attend), timed in a CUDA graph over enough
    layer caches to exceed L2.  Ragged lengths and paged block tables follow
    the seeded recipe of each workload; a paged sequence maps exactly the
    pages its rows need."""
    import numpy as np
    plan = [("gqa_mix", 4, 8), ("long", 4, 8), ("long", 8, 6), ("paged", 4, 12)]
    out = {}
    for name, bits, layers in plan:
        w = synth.WORKLOADS[name]
        rng = synth.rng_for(w.seed)
        lens = synth.context_lengths(rng, w.batch, *w.ctx)
        B, Hq, Hkv, D, g = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.group_size
        Lmax = int(lens.max())
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        if w.layout == "paged":
            table, num_pages = synth.block_table(rng, lens + 1, w.page_size)
            desc = K.make_desc(bits, g, Hkv, D, K.KVQ_PAGED, w.page_size, num_pages,
                               table.shape[1])
            bt = torch.from_numpy(table)
        else:
            desc = K.make_desc(bits, g, Hkv, D, K.KVQ_DENSE, ((Lmax + 1 + 15) // 16) * 16)
            bt = None
        caches, qs, kns, vns = [], [], [], []
        for l in range(layers):
            gen = torch.Generator(device=dev)
            gen.manual_seed(w.seed * 100003 + l)
            outl = synth.outlier_channels(np.random.default_rng(w.seed * 100003 + l), Hkv, D)
            cache = K.KVCache.allocate(desc, B, dev, block_table=bt)
            if bt is None:
                k, v = synth.device_kv(gen, B, Lmax, Hkv, D, outl, dev)
                K.kvq_append(cache, k, v, torch.zeros(B, dtype=torch.int32, device=dev), status)
                del k, v
            else:
                zero1 = torch.zeros(1, dtype=torch.int32, device=dev)
                for b in range(B):  # each sequence fills only its own pages
                    view = K.KVCache(desc, 1, cache.k_codes, cache.v_codes, cache.k_scale,
                                     cache.k_zero, cache.v_scale, cache.v_zero,
                                     cache.block_table[b:b + 1])
                    k, v = synth.device_kv(gen, 1, int(lens[b]), Hkv, D, outl, dev)
                    K.kvq_append(view, k, v, zero1, status)
                del k, v
            caches.append(cache)
            kn, vn = synth.device_kv(gen, B, 1, Hkv, D, outl, dev)
            kns.append(kn[:, 0])
            vns.append(vn[:, 0])
            qs.append(torch.randn((B, Hq, D), generator=gen, device=dev).half())
        torch.cuda.synchronize()
        if int(status.item()) != 0:
            raise RuntimeError(f"{name}: populate flagged status {int(status.item()):#x}")
        lens_before = torch.from_numpy(lens).to(dev)
        rows = Lmax + 1
        splits = K.kvq_decode_num_splits(desc, B, Hq, rows, 0)
        ws = torch.empty(max(16, K.kvq_decode_workspace_size(desc, B, Hq, rows, 0)),
                         dtype=torch.uint8, device=dev)
        outs = [torch.empty_like(q) for q in qs]
        stream = torch.cuda.Stream(device=dev)

        def step():
            for l in range(layers):
                K.kvq_append_decode_attn(caches[l], kns[l], vns[l], qs[l], lens_before, rows,
                                         outs[l], ws, status, stream=stream)

        with torch.cuda.stream(stream):
            step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        with torch.cuda.stream(stream):
            for _ in range(3):
                graph.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        reps = max(3, steps // 2)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        if int(status.item()) != 0:
            raise RuntimeError(f"{name}: device status {int(status.item()):#x}")
        call_s = e0.elapsed_time(e1) / 1e3 / (reps * layers)
        per_row = D * bits // 8 + 4 * (D // g)
        nbytes = (2 * Hkv * int((lens + 1).sum()) * per_row + 2 * B * Hkv * D * 2 +
                  2 * B * Hq * D * 2)
        out[f"{name}_int{bits}"] = {
            "what": f"{w.note}; INT{bits} group {g}; fused append + decode per layer cache",
            "layers": layers, "splits": splits, "avg_launch_us": call_s * 1e6,
            "tokens_per_s": B / call_s, "model_tokens_per_s": B / call_s / MODEL_LAYERS[name],
            "model_layers": MODEL_LAYERS[name], "bytes_per_launch": nbytes,
            "achieved_gbs": nbytes / call_s / 1e9, "frac": nbytes / call_s / 1e9 / peak,
            "frac_nominal": nbytes / call_s / 1e9 / NOMINAL_HBM_GBS}
        del caches, graph, ws, outs
        torch.cuda.empty_cache()
    return out


def reduce_max_over_ranks(x, world, device):
    """The largest of every rank's x (the job's time is its slowest rank's)."""
    if world == 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank, world, ms_max):
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / (ms_max / 1e3)


def load_profiled_traffic():
    """DRAM bytes per launch of the step kernel from the committed ncu
    summary, or None when any of the kernel's sources changed since that
    capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)[WORKLOAD]
        for src, digest in d["kernel_sources"].items():
            with open(os.path.join(ROOT, src), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != digest:
                    return None
        return int(d["dram_bytes_per_launch"])
    except Exception:
        return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--clock-preroll", type=float, default=0.4,
                    help="seconds of untimed step replays between starting the clock sampler "
                         "and the timed steps (0 under a profiler)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--layers", type=int, default=0)
    ap.add_argument("--cpu-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp16", action="store_true",
                    help="skip the fp16-cache comparator (this library and PyTorch SDPA)")
    ap.add_argument("--no-symmetric", action="store_true",
                    help="skip the symmetric-cache comparator")
    ap.add_argument("--no-kivi", action="store_true",
                    help="skip the axis-aware-cache comparator")
    ap.add_argument("--no-lowbit", action="store_true",
                    help="skip the NF4 and INT2 comparators")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the GQA-mix, long-context and paged workloads")
    ap.add_argument("--separate-append", action="store_true",
                    help="append and attend in two calls instead of the fused call")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu_arm(args)


if __name__ == "__main__":
    main()
