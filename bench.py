"""Benchmark of the quantised-KV-cache decode hot path on GB300.

One step = the whole hot path over one batch: append one new bf16 token per sequence
(quantising and packing a full group whenever the window fills) and run single-query
decode attention over the packed cache, for every layer of the workload.

The headline workload (`--workload`, default the KIVI 2-bit Llama-3-8B layer: 32 query /
8 KV heads, head_dim 128, batch 8, context 4096, groups of 32, 128-token bf16 window) gives
the line's `value`; the other workloads of the suite (`--suite`) are measured the same way
and reported under `workloads`.

Timing: steps are captured in a CUDA graph; consecutive steps rotate over cache replicas
whose total size exceeds the L2 cache, so every step reads its cache from HBM.  The step
graph (K steps) is replayed `--replays` times and the median replay gives `value` and
`ms_per_step`; the decode kernels alone (the roofline's kernel: decode + merge) are timed
by replaying a K-launch decode graph for at least `--decode-seconds`, median again.  Every
replay is bracketed by CUDA events on the launching stream.  The end-to-end leg drives the
public C ABI from pinned host buffers.  `--impl reference` times the CPU oracle instead.

Prints one JSON line (rank 0).
"""
import argparse
import concurrent.futures as cf
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("quantised-cache decode attention tokens/s and achieved HBM GB/s (% of peak), 1 GB300")
L2_BYTES = 129 * 2 ** 20
# the timed workloads (the tiny INT8 one is a correctness case, checked by the tests)
SUITE = ("kivi2_llama3_8b", "kivi4_128k", "fp8_32layer", "serve_mix", "serve_mix_paged", "kivi2_llama3_8b_rope",
         "kivi4_128k_sparse")


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 200 ms) while the timed work runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------- byte model
def decode_bytes(w, lengths):
    """Algorithmic bytes one decode launch (one layer) reads for sequences holding
    `lengths[b]` tokens: packed group records + bf16 window rows + the queries."""
    H, D, gqa = w.kv_heads, w.head_dim, w.gqa
    qbytes = gqa * D * (2 if w.in_dtype == "bf16" else 4)
    total = 0
    for n_tokens in lengths:
        if w.scheme == 0:
            G, b, R = w.group_k, w.bits, w.residual
            qn = G * ((n_tokens - R) // G) if n_tokens >= R + G else 0
            r = n_tokens - qn
            rec = G * D * b // 8 * 2 + 4 * D + 4 * G * (D // w.group_v)
            rec += 4 * w.outliers * (D + G * (D // w.group_v))      # dense-and-sparse side lists
            cache = (qn // G) * rec + r * 4 * D
        elif w.scheme == 1:
            cache = n_tokens * (2 * D + 8)
        else:
            cache = n_tokens * 2 * D
        total += H * (cache + qbytes)
    return total


DECODE_SOURCES = ("kvq_api.cu", "kvq_decode.cuh", "kvq_decode_rows.cu", "kvq_internal.cuh", "kvq_launch.h",
                  "kvq_rope.cuh")
SCHEME_SOURCES = {0: tuple("kvq_decode_kivi%d%s.cu" % (b, v) for b in (2, 4, 8)
                            for v in ("", "_steal", "_paged", "_paged_steal", "_sparse", "_sparse_paged", "_rope",
                                      "_rope_paged"))
                 + ("kvq_decode_rope.cu",),
                  1: (), 2: ("kvq_decode_fp8.cu",), 3: ("kvq_decode_fp8.cu",), 4: ()}


def sources_sha256(scheme):
    """Digest of the CUDA sources (file names and contents) that decide a scheme's decode
    kernels: the plan, the shared decode code and the scheme's own translation units."""
    import hashlib
    d = os.path.join(ROOT, "quantised_kv_cache_kvq_gb300", "csrc")
    h = hashlib.sha256()
    for n in sorted(DECODE_SOURCES + SCHEME_SOURCES[scheme]):
        h.update(n.encode())
        with open(os.path.join(d, n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(workload, scheme):
    """DRAM bytes per decode launch (both kernels) from the committed ncu summary of this
    workload; None without one, or when the kernels' sources changed since its capture."""
    import re
    try:
        with open(os.path.join(ROOT, "profiles", "k_decode_%s.md" % workload)) as f:
            text = f.read()
    except OSError:
        return None
    t = re.search(r"^traffic_bytes_per_launch: (\d+)$", text, re.M)
    h = re.search(r"^sources_sha256: ([0-9a-f]+)$", text, re.M)
    if not (t and h) or h.group(1) != sources_sha256(scheme):
        return None
    return int(t.group(1))


def max_over_ranks(values, world, device="cpu"):
    """Element-wise maximum of per-rank timings (the job is as slow as its slowest rank)."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def host_cores():
    return len(os.sched_getaffinity(0))


# ---------------------------------------------------------------------------- GPU arm
def run_gpu(args, w, world, all_layers, nsteps, sampler_on):
    """Fill the workload's caches, then time the step graph, the decode graph and the
    end-to-end leg.  Returns a dict of raw timings and byte counts (this rank)."""
    import torch
    import quantised_kv_cache_kvq_gb300 as K
    from quantised_kv_cache_kvq_gb300 import workloads as W

    dev = torch.device("cuda", torch.cuda.current_device())
    lens0 = [int(x) for x in W.context_lengths(w).tolist()]
    layers = w.layers if all_layers else 1
    per_cache = layers * decode_bytes(w, lens0)
    # replicas rotated per step so that consecutive steps read their caches from HBM
    reps = max(1, math.ceil(4 * L2_BYTES / per_cache)) if args.replicas <= 0 else args.replicas
    reps = max(reps, 2) if per_cache < 4 * L2_BYTES else reps
    e2e_runs, e2e_steps = 5, min(nsteps, 200)
    # step replays grow every context by about nsteps / reps tokens each: keep the growth
    # within 2% of the mean context (at least 5 replays)
    mean0 = sum(lens0) / len(lens0)
    replays = min(args.replays, max(5, int(0.02 * mean0 * reps / nsteps)))
    # steps go to replica i % reps in each of: the warm-up, every replay of the step graph,
    # every run of the two end-to-end graphs
    appends_per_rep = (math.ceil(args.warmup / reps) + replays * math.ceil(nsteps / reps)
                       + 2 * e2e_runs * math.ceil(e2e_steps / reps) + 1)
    max_tokens = max(lens0) + appends_per_rep + 16
    paging = {}
    if w.page_groups:   # one block table for every replica (each has its own pool)
        pool, table = W.block_table(w, max_tokens, device=dev)
        paging = dict(page_groups=w.page_groups, num_pages=pool, block_table=table)
    cfg = K.make_config(w.scheme, layers, w.batch, w.q_heads, w.kv_heads, w.head_dim, max_tokens,
                        bits=w.bits, group_k=w.group_k, group_v=w.group_v, residual=w.residual,
                        in_dtype=w.in_dtype, rope_base=w.rope_base, outliers=w.outliers, **paging)
    caches = []
    fp8 = None
    if w.scheme == 2:   # static per-(kv head) scales from the first replica's fill
        k, v = W.kv_tokens(w, 0, 0, min(8, w.batch), 0, min(lens0[:8]), device=dev, tag="rep0")
        fp8 = W.fp8_scales(w, k, v)
        del k, v
    t_fill = time.perf_counter()
    for r in range(reps):
        c = K.QuantizedKVCache(cfg, dev)
        for s0 in range(0, w.batch, 8):
            ns = min(8, w.batch - s0)
            nl = lens0[s0:s0 + ns]
            k, v = W.kv_tokens(w, 0, s0, ns, 0, max(nl), device=dev, tag="rep%d" % r)
            nv = torch.tensor(nl, dtype=torch.int32, device=dev)
            # every layer is filled from the same seeded draw (the timing does not depend on
            # the values; each layer is a separate cache region read from HBM)
            for layer in range(layers):
                c.append(layer, k, v, seq_begin=s0, n_valid=nv, fp8_scales=fp8)
            del k, v
        caches.append(c)
    torch.cuda.synchronize()
    t_fill = time.perf_counter() - t_fill

    def check_status(phase):
        status = 0
        for c in caches:
            status |= c.status(stream=None)
        if status:
            raise RuntimeError("%s: device status word %#x after the %s" % (w.name, status, phase))

    check_status("fill")
    ws = caches[0].workspace
    # per-step inputs: one new token per sequence (shared by the layers) and the step's queries
    nin = args.warmup + nsteps + e2e_steps
    kn, vn = W.kv_tokens(w, 0, 0, w.batch, max(lens0), nin, device=dev, tag="steps")
    k_steps = kn.permute(1, 0, 2, 3).contiguous().unsqueeze(2)   # [step][batch][1][H][D]
    v_steps = vn.permute(1, 0, 2, 3).contiguous().unsqueeze(2)
    del kn, vn
    qdt = torch.bfloat16 if w.in_dtype == "bf16" else torch.float32
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed * 7919 + 17)
    q_steps = (torch.randn(nin, w.batch, w.q_heads, w.head_dim, generator=g, device=dev) * w.q_mult).to(qdt)
    outs = [torch.empty(w.batch, w.q_heads, w.head_dim, dtype=torch.float32, device=dev) for _ in range(reps)]
    scale = w.scale
    stream = torch.cuda.Stream(dev)
    # the inputs were made on the default stream: the timed work runs on `stream`
    stream.wait_stream(torch.cuda.current_stream())
    visits = [0] * reps          # steps appended to each replica so far

    def step(i, c):
        for layer in range(layers):
            K.kvq_quantize_append(cfg, c.cache, layer, 0, w.batch, k_steps[i], v_steps[i], 1, fp8_scales=fp8,
                                  stream=stream)
            K.kvq_decode_attention(cfg, c.cache, layer, q_steps[i], scale, outs[caches.index(c)], ws,
                                   stream=stream)

    def lengths(r):
        return [n + visits[r] for n in lens0]

    # warm-up (eager), then the timed steps as one graph of nsteps steps
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i, caches[i % reps])
            visits[i % reps] += 1
    stream.synchronize()
    check_status("warm-up steps")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(nsteps):
            step(args.warmup + i, caches[i % reps])
    launches_per_step = 3 * layers   # per layer: append (one kernel for one token), decode, merge
    # decode-only graph over the same rotation: the roofline's kernels alone
    dgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(dgraph, stream=stream):
        for i in range(nsteps):
            c = caches[i % reps]
            for layer in range(layers):
                K.kvq_decode_attention(cfg, c.cache, layer, q_steps[args.warmup + i], scale, outs[i % reps], ws,
                                       stream=stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    def replay(gr):
        with torch.cuda.stream(stream):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            gr.replay()
            e1.record(stream)
        return e0, e1

    sampler = ClockSampler(dev.index) if sampler_on else None
    if sampler:
        sampler.__enter__()
    try:
        time.sleep(0.3 if sampler else 0.0)
        barrier()
        step_ms, step_bytes = [], []
        for rep_i in range(replays):
            before = [list(lengths(r)) for r in range(reps)]
            e0, e1 = replay(graph)
            for i in range(nsteps):
                visits[i % reps] += 1
            stream.synchronize()
            step_ms.append(e0.elapsed_time(e1))
            nb = 0
            seen = [0] * reps
            for i in range(nsteps):
                r = i % reps
                seen[r] += 1
                nb += layers * decode_bytes(w, [n + seen[r] for n in before[r]])
            step_bytes.append(nb)
        barrier()
        # decode-only replays (the cache does not change): at least --decode-seconds
        dec_bytes = sum(layers * decode_bytes(w, lengths(i % reps)) for i in range(nsteps))
        dec_ms = []
        t_end = time.perf_counter() + args.decode_seconds
        while len(dec_ms) < replays or time.perf_counter() < t_end:
            e0, e1 = replay(dgraph)
            stream.synchronize()
            dec_ms.append(e0.elapsed_time(e1))
        time.sleep(0.3 if sampler else 0.0)
    finally:
        if sampler:
            sampler.__exit__(None, None, None)
    check_status("timed steps")

    # end to end through the C ABI with host buffers: per step the new token and the queries
    # come from pinned host memory (keys, values and queries side by side in one row per
    # step, each part at a 256-byte offset), then the append and decode of every layer, then
    # the step's result (the last layer's outputs) goes back to pinned host memory.  Two
    # ways, each captured as one graph of e2e_steps steps:
    #   mapped: the host rows are passed to the C ABI as they are (page-locked memory is
    #     mapped into the device's address space): the append kernel reads the new token and
    #     the decode reads the queries across the host link, and the last layer's merge
    #     writes the outputs into the host buffer;
    #   staged: copies on a second stream move each step's row into device memory and the
    #     outputs back; the inputs of step i + 1 arrive and the outputs of step i - 1 leave
    #     while step i computes (two device input rows and two output buffers).
    base = args.warmup + nsteps
    parts = [k_steps[base:base + e2e_steps], v_steps[base:base + e2e_steps], q_steps[base:base + e2e_steps]]
    sizes = [t[0].numel() * t.element_size() for t in parts]
    offs = [0]
    for n in sizes[:-1]:
        offs.append(offs[-1] + (n + 255) // 256 * 256)
    row_bytes = (offs[-1] + sizes[-1] + 255) // 256 * 256
    hin = torch.zeros(e2e_steps, row_bytes, dtype=torch.uint8).pin_memory()
    for t, o, n in zip(parts, offs, sizes):
        hin[:, o:o + n].copy_(t.reshape(e2e_steps, -1).view(torch.uint8).cpu())
    hviews = [[hin[i, o:o + n].view(t.dtype).view(t.shape[1:]) for t, o, n in zip(parts, offs, sizes)]
              for i in range(e2e_steps)]
    din = [torch.empty(row_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    views = [[d[o:o + n].view(t.dtype).view(t.shape[1:]) for t, o, n in zip(parts, offs, sizes)] for d in din]
    hout = torch.empty(e2e_steps, w.batch, w.q_heads, w.head_dim, dtype=torch.float32).pin_memory()
    dout = [torch.empty(layers, w.batch, w.q_heads, w.head_dim, dtype=torch.float32, device=dev) for _ in range(2)]
    last = e2e_steps - 1

    def mapped_graph():
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for i in range(e2e_steps):
                c = caches[i % reps]
                hk, hv, hq = hviews[i]
                for layer in range(layers):
                    K.kvq_quantize_append(cfg, c.cache, layer, 0, w.batch, hk, hv, 1, fp8_scales=fp8, stream=stream)
                    o = hout[i] if layer == layers - 1 else dout[i % 2][layer]
                    K.kvq_decode_attention(cfg, c.cache, layer, hq, scale, o, ws, stream=stream)
        return gr

    def staged_graph():
        gr = torch.cuda.CUDAGraph()
        copy_stream = torch.cuda.Stream(dev)
        with torch.cuda.graph(gr, stream=stream):
            copy_stream.wait_stream(stream)
            ev_in = [torch.cuda.Event() for _ in range(e2e_steps)]
            ev_done = [torch.cuda.Event() for _ in range(e2e_steps)]
            ev_out = [torch.cuda.Event() for _ in range(e2e_steps)]
            with torch.cuda.stream(copy_stream):
                din[0].copy_(hin[0], non_blocking=True)
                ev_in[0].record(copy_stream)
            for i in range(e2e_steps):
                c = caches[i % reps]
                dk, dv, dq = views[i % 2]
                stream.wait_event(ev_in[i])
                if i >= 2:
                    stream.wait_event(ev_out[i - 2])     # outputs of step i - 2 have left
                for layer in range(layers):
                    K.kvq_quantize_append(cfg, c.cache, layer, 0, w.batch, dk, dv, 1, fp8_scales=fp8, stream=stream)
                    K.kvq_decode_attention(cfg, c.cache, layer, dq, scale, dout[i % 2][layer], ws, stream=stream)
                ev_done[i].record(stream)
                with torch.cuda.stream(copy_stream):
                    if i + 1 < e2e_steps:
                        if i >= 1:
                            copy_stream.wait_event(ev_done[i - 1])   # input row of step i - 1 is free
                        din[(i + 1) % 2].copy_(hin[i + 1], non_blocking=True)
                        ev_in[i + 1].record(copy_stream)
                    copy_stream.wait_event(ev_done[i])
                    hout[i].copy_(dout[i % 2][layers - 1], non_blocking=True)
                    ev_out[i].record(copy_stream)
            stream.wait_stream(copy_stream)
        return gr

    e2e_med = {}
    for mode, make in (("mapped", mapped_graph), ("staged", staged_graph)):
        egraph = make()
        ms = []
        barrier()
        for run in range(e2e_runs):
            e0, e1 = replay(egraph)
            stream.synchronize()
            ms.append(e0.elapsed_time(e1))
            for i in range(e2e_steps):
                visits[i % reps] += 1
        barrier()
        del egraph
        # the last run's outputs came back to the host: check them against a decode of the
        # same cache state from device copies of the same queries (chunks taken on demand
        # split the context differently from launch to launch: compare within the attention
        # tolerance), and the copied-back ones against the device buffer they came from
        cl = caches[last % reps]
        ref = torch.empty(w.batch, w.q_heads, w.head_dim, dtype=torch.float32, device=dev)
        with torch.cuda.stream(stream):
            K.kvq_decode_attention(cfg, cl.cache, layers - 1, parts[2][last], scale, ref, ws, stream=stream)
        stream.synchronize()
        ref = ref.cpu()
        err = float((hout[last] - ref).abs().max())
        print("%s e2e %s: max |host - device decode| %.3g" % (w.name, mode, err), file=sys.stderr)
        if not torch.allclose(hout[last], ref, rtol=1e-2, atol=2e-3) or (
                mode == "staged" and not torch.equal(hout[last], dout[last % 2][layers - 1].cpu())):
            raise RuntimeError("end-to-end outputs (%s) did not come back to the host" % mode)
        check_status("end-to-end steps (%s)" % mode)
        e2e_med[mode] = statistics.median(ms)
    h2d = row_bytes
    d2h = w.batch * w.q_heads * w.head_dim * 4
    del graph, dgraph
    # the job is as slow as its slowest rank
    step_med, dec_med, e2e_mapped, e2e_staged = max_over_ranks(
        [statistics.median(step_ms), statistics.median(dec_ms), e2e_med["mapped"], e2e_med["staged"]], world, dev)
    res = dict(step_ms=step_med, step_ms_all=step_ms,
               step_bytes=statistics.median(step_bytes), decode_ms=dec_med,
               decode_replays=len(dec_ms), dec_bytes=dec_bytes, e2e_ms=e2e_mapped, e2e_staged_ms=e2e_staged,
               e2e_steps=e2e_steps, reps=reps, layers=layers, cache_mb=per_cache / 1e6,
               launches=(launches_per_step * nsteps * replays + 2 * layers * nsteps * len(dec_ms)
                         + 2 * launches_per_step * e2e_steps * e2e_runs),
               clocks=sampler.summary() if sampler else None, h2d=h2d,
               d2h=d2h, max_tokens=max_tokens, fill_s=t_fill, mean_context=sum(lens0) / len(lens0),
               nsteps=nsteps)
    caches.clear()
    del ws, outs, k_steps, v_steps, q_steps, hin, hout, din, dout
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------- CPU oracle
def oracle_setup(w, nseq):
    import numpy as np
    import torch
    import oracle as O
    from quantised_kv_cache_kvq_gb300 import workloads as W
    lens = [int(x) for x in W.context_lengths(w).tolist()[:nseq]]
    n0 = max(lens)
    kw = dict(scheme=w.scheme, layers=1, batch=nseq, q_heads=w.q_heads, kv_heads=w.kv_heads,
              head_dim=w.head_dim, bits=w.bits if w.scheme == 0 else 8, group_k=w.group_k, group_v=w.group_v,
              residual=w.residual, max_tokens=n0 + 4096, in_dtype=0 if w.in_dtype == "bf16" else 1,
              rope_base=w.rope_base, outliers=w.outliers)
    if w.page_groups:
        pool, table = W.block_table(w, kw["max_tokens"])
        kw.update(page_groups=w.page_groups, num_pages=pool, block_table=table[:nseq].numpy())
    img = O.Image(O.make_config(**kw))
    k, v = W.kv_tokens(w, 0, 0, nseq, 0, n0, device="cpu", tag="cpu")
    to = (lambda t: t.view(torch.int16).numpy().view(np.uint16)) if w.in_dtype == "bf16" else (lambda t: t.numpy())
    sc = W.fp8_scales(w, k, v).numpy() if w.scheme == 2 else None
    img.append(0, 0, to(k), to(v), n_valid=np.asarray(lens, np.int32), fp8_scales=sc)
    q = W.queries(w, 0, device="cpu").float().numpy()[:nseq]
    kn, vn = W.kv_tokens(w, 0, 0, nseq, n0, 4096, device="cpu", tag="cpu-steps")
    return img, q, to(kn), to(vn), sc


def run_oracle(w, budget_s, max_steps=None, warmup=1):
    """Time the oracle on a bounded sample of the workload: the first min(batch, 8)
    sequences of one layer; each step appends one token to every sampled sequence and
    decodes all of them, one task per (sequence, kv head) on a pool of every host core.
    After `warmup` untimed steps, steps run until `budget_s` seconds have passed (at most
    `max_steps`).  Returns a dict."""
    import numpy as np
    nseq = min(w.batch, 8)
    cores = host_cores()
    img, q, kn, vn, sc = oracle_setup(w, nseq)
    out = np.zeros((nseq, w.q_heads, w.head_dim))
    tasks = [(b, h) for b in range(nseq) for h in range(w.kv_heads)]
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        for i in range(warmup):     # untimed
            img.append(0, 0, kn[:, i:i + 1], vn[:, i:i + 1], fp8_scales=sc)
            list(ex.map(lambda t: img.decode_head(0, q, w.scale, t[0], t[1], out), tasks))
        steps, t0 = 0, time.perf_counter()
        while True:
            j = (warmup + steps) % kn.shape[1]
            img.append(0, 0, kn[:, j:j + 1], vn[:, j:j + 1], fp8_scales=sc)
            list(ex.map(lambda t: img.decode_head(0, q, w.scale, t[0], t[1], out), tasks))
            steps += 1
            el = time.perf_counter() - t0
            if el >= budget_s or (max_steps is not None and steps >= max_steps):
                break
    return {"tokens_per_s": steps * nseq / el, "seconds": el, "steps": steps, "nseq": nseq, "cores": cores,
            "tasks": len(tasks)}


def cpu_record(w, res, layers):
    return {"value": res["tokens_per_s"] / layers, "unit": "tokens/s", "cores": res["cores"], "kind": "oracle",
            "sample": "%d oracle steps on the first %d sequences of one layer (%.1f s): each appends one token "
                      "to every sequence and decodes all of them, %d (sequence, kv head) tasks on %d host "
                      "threads%s" % (res["steps"], res["nseq"], res["seconds"], res["tasks"], res["cores"],
                                     "; divided by the %d layers a token needs" % layers if layers > 1 else "")}


# ---------------------------------------------------------------------------- records
def workload_config(w, layers):
    ragged = w.context[0] != w.context[1]
    cfg = {"workload": w.name, "scheme": ["kivi", "int8", "fp8", "fp8e5m2", "int4"][w.scheme], "bits": w.bits,
           "batch": w.batch, "q_heads": w.q_heads, "kv_heads": w.kv_heads, "head_dim": w.head_dim,
           "context": list(w.context) if ragged else w.context[0], "group_k": w.group_k,
           "group_v": w.group_v, "residual": w.residual, "layers": layers}
    if w.page_groups:
        cfg["layout"] = "paged: %d group records (%d tokens) a page, shuffled block table" % (
            w.page_groups, w.page_groups * w.group_k)
    if w.rope_base:
        cfg["keys"] = "cached before the rotary embedding (base %g), rotated in the decode" % w.rope_base
    if w.outliers:
        cfg["outliers"] = ("dense-and-sparse: %d element(s) of largest magnitude per quantisation vector kept "
                           "in bf16 in a side list" % w.outliers)
    return cfg


def gpu_record(w, r, world, peak, peak_kind):
    tokens = w.batch * r["nsteps"] * world
    value = tokens / (r["step_ms"] / 1e3)
    launches = r["nsteps"] * r["layers"]                 # decode calls in the decode-only graph
    dec_avg_ms = r["decode_ms"] / launches
    achieved = (r["dec_bytes"] / launches) / (dec_avg_ms / 1e3) / 1e9
    step_gbs = r["step_bytes"] / (r["step_ms"] / 1e3) / 1e9
    from quantised_kv_cache_kvq_gb300 import workloads as W
    # the profile summaries hold the traffic of one decode call (one layer) of the workload as
    # defined (its batch); every launch of the line, one per layer, is such a call
    traffic = profiled_traffic(w.name, w.scheme) if w == W.WORKLOADS[w.name] else None
    cfg = workload_config(w, r["layers"])
    cfg.update({"steps_per_replay": r["nsteps"], "replicas": r["reps"],
                "cache_mb_per_replica": round(r["cache_mb"], 2), "mean_context": round(r["mean_context"], 1),
                "fill_s": round(r["fill_s"], 1),
                "l2": "inputs larger than L2: %d cache replica(s) rotated per step (%.0f MB > 129 MB)"
                      % (r["reps"], r["reps"] * r["cache_mb"]),
                "timing": "CUDA graph of the steps replayed %d times (median), decode graph replayed %d "
                          "times (median); CUDA events on the launch stream"
                          % (len(r["step_ms_all"]), r["decode_replays"])})
    rec = {
        "value": value, "unit": "tokens/s", "ms_per_step": r["step_ms"] / r["nsteps"],
        "hbm_gbs": step_gbs, "hbm_pct_of_peak": 100.0 * step_gbs / peak, "config": cfg,
        "roofline": {"kernel": "kvq decode attention (decode kernel + merge)", "bound": "hbm",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "traffic": traffic,
                     "traffic_source": ("ncu dram__bytes_read.sum + dram__bytes_write.sum of both kernels, from "
                                        "profiles/k_decode_%s.md (same kernel sources)" % w.name)
                     if traffic is not None else None,
                     "avg_launch_us": 1e3 * dec_avg_ms, "bytes_per_launch": r["dec_bytes"] / launches},
        "e2e": {"value": w.batch * r["e2e_steps"] * world / (r["e2e_ms"] / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"], "steps": r["e2e_steps"],
                "how": "public C ABI (kvq_quantize_append, kvq_decode_attention) in one CUDA graph per run, "
                       "called with pinned host buffers: every step the append kernel reads the new token "
                       "and the decode reads the queries from host memory across the host link, and the "
                       "last layer's merge writes the outputs into host memory; median of 5 runs",
                "staged": {"value": w.batch * r["e2e_steps"] * world / (r["e2e_staged_ms"] / 1e3),
                           "unit": "tokens/s",
                           "how": "the same steps with copies on a second stream: each step's inputs "
                                  "copied into device memory while the previous step computes, the "
                                  "outputs copied back; median of 5 runs"}},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    return rec


# ---------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="kivi2_llama3_8b", help="the headline workload")
    ap.add_argument("--suite", default="all",
                    help="other workloads to report under `workloads`: all, none, or a comma list")
    ap.add_argument("--replicas", type=int, default=0, help="cache replicas (0: enough to exceed 4x L2)")
    ap.add_argument("--replays", type=int, default=20, help="timed replays of the step graph (median)")
    ap.add_argument("--decode-seconds", type=float, default=1.0,
                    help="minimum duration of the decode-only replays (median)")
    ap.add_argument("--cpu-budget", type=float, default=8.0, help="seconds of oracle work per workload")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's number of sequences (smaller cases for ncu captures)")
    ap.add_argument("--all-layers", action="store_true",
                    help="time every layer of the headline workload in each step (default: one layer)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    from quantised_kv_cache_kvq_gb300 import workloads as W
    w = W.WORKLOADS[args.workload]
    if args.batch > 0:
        import dataclasses
        w = dataclasses.replace(w, batch=args.batch)
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    peak, peak_kind = peaks()
    if args.suite == "all":
        suite = [n for n in SUITE if n != w.name]
    elif args.suite == "none":
        suite = []
    else:
        suite = [n for n in args.suite.split(",") if n and n != w.name]

    if args.impl == "reference":
        if rank != 0:
            return
        import __graft_entry__  # noqa: F401  (oracle build)
        from oracle import build as ob
        ob.build()
        # each of the K timed steps is a bounded oracle step of the workload: one token
        # appended to every sampled sequence and all of them decoded
        res = run_oracle(w, budget_s=1e9, max_steps=args.steps, warmup=args.warmup)
        layers = w.layers if args.all_layers else 1
        cpu = cpu_record(w, res, layers)
        line = {"impl": "reference", "metric": METRIC, "value": cpu["value"], "unit": "tokens/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * res["seconds"] / res["steps"], "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": workload_config(w, layers),
                "cpu_baseline": cpu,
                "e2e": {"value": cpu["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    import __graft_entry__
    __graft_entry__.build()
    import quantised_kv_cache_kvq_gb300 as K
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    K.load()
    layers = w.layers if args.all_layers else 1
    r = run_gpu(args, w, world, args.all_layers, args.steps, sampler_on=True)
    others = {}
    for name in suite:
        ow = W.WORKLOADS[name]
        osteps = max(args.steps, ow.steps)
        try:
            others[name] = (ow, run_gpu(args, ow, world, ow.layers > 1, osteps, sampler_on=True))
        except Exception as exc:     # the other lines stand without it; the error is reported
            others[name] = (ow, {"error": str(exc)})
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
    if rank != 0:
        return
    head = gpu_record(w, r, world, peak, peak_kind)
    try:
        cpu = cpu_record(w, run_oracle(w, args.cpu_budget), layers)
    except Exception as exc:  # the GPU number stands without it
        cpu = {"value": None, "unit": "tokens/s", "cores": 0, "kind": "oracle", "sample": "failed: %s" % exc}
    head["config"]["parallelism"] = "replicas" if world > 1 else "single"
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": head["config"],
        "hbm_gbs": head["hbm_gbs"], "hbm_pct_of_peak": head["hbm_pct_of_peak"], "roofline": head["roofline"],
        "cpu_baseline": cpu, "e2e": head["e2e"], "gpu_launches": head["gpu_launches"],
        "gpu_launches_counts": "every launch of the library's kernels in all timed regions of this line "
                               "(step, decode-only and end-to-end replays of every workload)",
        "clocks": r["clocks"],
    }
    wl = {}
    for name, (ow, orr) in others.items():
        if "error" in orr:
            wl[name] = {"error": orr["error"]}
            continue
        rec = gpu_record(ow, orr, world, peak, peak_kind)
        try:
            rec["cpu_baseline"] = cpu_record(ow, run_oracle(ow, args.cpu_budget), orr["layers"])
        except Exception as exc:
            rec["cpu_baseline"] = {"value": None, "unit": "tokens/s", "cores": 0, "kind": "oracle",
                                   "sample": "failed: %s" % exc}
        line["gpu_launches"] += rec["gpu_launches"]
        wl[name] = rec
    if wl:
        line["workloads"] = wl
    print(json.dumps(line))


if __name__ == "__main__":
    main()
