"""Benchmark of the quantised-KV-cache decode hot path on GB300.

One step = the whole hot path over one batch: append one new bf16 token per sequence
(quantising and packing a full group whenever the window fills) and run single-query
decode attention over the packed cache.  Default workload: KIVI 2-bit keys/values,
Llama-3-8B attention layer shape (32 query / 8 KV heads, head_dim 128), batch 8,
context 4096, groups of 32, 128-token bf16 window.

Timing: steps are captured in a CUDA graph and replayed; consecutive steps rotate over
cache replicas whose total size exceeds the L2 cache, so every step reads its cache from
HBM.  The dominant kernel (decode attention) is also timed alone for the roofline.
`--impl reference` times the CPU oracle (tests' reference implementation) instead.

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
            cache = (qn // G) * rec + r * 4 * D
        elif w.scheme == 1:
            cache = n_tokens * (2 * D + 8)
        else:
            cache = n_tokens * 2 * D
        total += H * (cache + qbytes)
    return total


DECODE_SOURCES = ("kvq_api.cu", "kvq_decode.cuh", "kvq_decode_rows.cu", "kvq_internal.cuh", "kvq_launch.h")
SCHEME_SOURCES = {0: ("kvq_decode_kivi2.cu", "kvq_decode_kivi4.cu", "kvq_decode_kivi8.cu"),
                  1: (), 2: ("kvq_decode_fp8.cu",)}


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


# ---------------------------------------------------------------------------- GPU arm
def run_gpu(args, w, rank, world):
    import torch
    import quantised_kv_cache_kvq_gb300 as K
    from quantised_kv_cache_kvq_gb300 import workloads as W

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    K.load()
    lens0 = [int(x) for x in W.context_lengths(w).tolist()]
    layers = w.layers if args.all_layers else 1
    per_cache = layers * decode_bytes(w, lens0)
    # replicas rotated per step so that consecutive steps read their caches from HBM
    reps = max(1, math.ceil(4 * L2_BYTES / per_cache)) if args.replicas <= 0 else args.replicas
    reps = max(reps, 2) if per_cache < 4 * L2_BYTES else reps
    total_steps = args.warmup + args.steps
    e2e_steps = min(args.steps, 200)
    appends_per_rep = math.ceil((total_steps + e2e_steps) / reps) + 1
    max_tokens = max(lens0) + appends_per_rep + 64
    cfg = K.make_config(w.scheme, layers, w.batch, w.q_heads, w.kv_heads, w.head_dim, max_tokens,
                        bits=w.bits, group_k=w.group_k, group_v=w.group_v, residual=w.residual,
                        in_dtype=w.in_dtype)
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
    ws = caches[0].workspace
    # per-step inputs: one new token per sequence (shared by the layers) and the step's queries
    kn, vn = W.kv_tokens(w, 0, 0, w.batch, max(lens0), total_steps, device=dev, tag="steps")
    k_steps = kn.permute(1, 0, 2, 3).contiguous().unsqueeze(2)   # [step][batch][1][H][D]
    v_steps = vn.permute(1, 0, 2, 3).contiguous().unsqueeze(2)
    del kn, vn
    qdt = torch.bfloat16 if w.in_dtype == "bf16" else torch.float32
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed * 7919 + 17)
    q_steps = (torch.randn(total_steps, w.batch, w.q_heads, w.head_dim, generator=g, device=dev)
               * w.q_mult).to(qdt)
    outs = [torch.empty(w.batch, w.q_heads, w.head_dim, dtype=torch.float32, device=dev) for _ in range(reps)]
    scale = w.scale
    stream = torch.cuda.Stream(dev)

    def step(i):
        c = caches[i % reps]
        for layer in range(layers):
            K.kvq_quantize_append(cfg, c.cache, layer, 0, w.batch, k_steps[i], v_steps[i], 1, fp8_scales=fp8,
                                  stream=stream)
            K.kvq_decode_attention(cfg, c.cache, layer, q_steps[i], scale, outs[i % reps], ws, stream=stream)

    launches_per_step = 3 * layers  # per layer: append (one kernel for a one-token append), decode, merge
    # warm-up (eager), then the timed steps as one graph
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(args.warmup, total_steps):
            step(i)
    # decode-only graph over the same rotation, for the dominant kernel's duration
    dgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(dgraph, stream=stream):
        for i in range(args.steps):
            c = caches[i % reps]
            for layer in range(layers):
                K.kvq_decode_attention(cfg, c.cache, layer, q_steps[i], scale, outs[i % reps], ws, stream=stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    sampler = ClockSampler(dev.index)
    with sampler:
        time.sleep(0.3)
        barrier()
        # graphs replay on the current stream: make it the stream the events are recorded on
        with torch.cuda.stream(stream):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        barrier()
        step_ms = e0.elapsed_time(e1)
        # dominant kernel alone (same replicas, L2-cold by rotation)
        with torch.cuda.stream(stream):
            d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            d0.record(stream)
            dgraph.replay()
            d1.record(stream)
        stream.synchronize()
        decode_ms = d0.elapsed_time(d1)
        time.sleep(0.3)
    status = 0
    for c in caches:
        status |= c.status()
    if status:
        raise RuntimeError("device status word %#x after the benchmark" % status)

    # bytes of the timed steps (every replica's sequences grow by one token per visit)
    def lengths_after(visits):
        return [n + visits for n in lens0]

    def visits(r, steps_done):
        return steps_done // reps + (1 if r < steps_done % reps else 0)

    bytes_steps = 0
    for i in range(args.warmup, total_steps):
        r = i % reps
        bytes_steps += layers * decode_bytes(w, lengths_after(visits(r, i) + 1))
    bytes_decode = sum(layers * decode_bytes(w, lengths_after(visits(i % reps, total_steps)))
                       for i in range(args.steps))

    # end to end through the C ABI with host buffers: per step copy the new token and the
    # queries from pinned host memory, append, decode every layer, copy the outputs back.
    # A step's keys, values and queries sit side by side in one pinned row (each part at a
    # 256-byte offset), so a step makes one host-to-device copy into a device row whose
    # views are the library's inputs.
    parts = [k_steps[:e2e_steps], v_steps[:e2e_steps], q_steps[:e2e_steps]]
    sizes = [t[0].numel() * t.element_size() for t in parts]
    offs = [0]
    for n in sizes[:-1]:
        offs.append(offs[-1] + (n + 255) // 256 * 256)
    row_bytes = offs[-1] + sizes[-1]
    hin = torch.zeros(e2e_steps, row_bytes, dtype=torch.uint8).pin_memory()
    for t, o, n in zip(parts, offs, sizes):
        hin[:, o:o + n].copy_(t.reshape(e2e_steps, -1).view(torch.uint8).cpu())
    din = torch.empty(row_bytes, dtype=torch.uint8, device=dev)
    dk, dv, dq = (din[o:o + n].view(t.dtype).view(t.shape[1:]) for t, o, n in zip(parts, offs, sizes))
    hout = torch.empty(e2e_steps, layers, w.batch, w.q_heads, w.head_dim, dtype=torch.float32).pin_memory()
    hin_rows = [hin[i] for i in range(e2e_steps)]
    hout_rows = [[hout[i, layer] for layer in range(layers)] for i in range(e2e_steps)]
    barrier()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        x0.record(stream)
        for i in range(e2e_steps):
            c = caches[i % reps]
            din.copy_(hin_rows[i], non_blocking=True)
            for layer in range(layers):
                K.kvq_quantize_append(cfg, c.cache, layer, 0, w.batch, dk, dv, 1, fp8_scales=fp8, stream=stream)
                K.kvq_decode_attention(cfg, c.cache, layer, dq, scale, outs[0], ws, stream=stream)
                hout_rows[i][layer].copy_(outs[0], non_blocking=True)
        x1.record(stream)
    barrier()
    e2e_ms = x0.elapsed_time(x1)
    h2d = row_bytes
    d2h = layers * outs[0].numel() * 4

    step_ms, decode_ms, e2e_ms = max_over_ranks([step_ms, decode_ms, e2e_ms], world, dev)
    return dict(step_ms=step_ms, decode_ms=decode_ms, e2e_ms=e2e_ms, e2e_steps=e2e_steps,
                bytes_steps=bytes_steps, bytes_decode=bytes_decode, reps=reps, layers=layers,
                cache_mb=per_cache / 1e6, launches=launches_per_step * args.steps,
                clocks=sampler.summary(), h2d=h2d, d2h=d2h, max_tokens=max_tokens, fill_s=t_fill,
                mean_context=sum(lens0) / len(lens0))


# ---------------------------------------------------------------------------- CPU oracle
def oracle_setup(w, nseq):
    import numpy as np
    import oracle as O
    from quantised_kv_cache_kvq_gb300 import workloads as W
    lens = [int(x) for x in W.context_lengths(w).tolist()[:nseq]]
    n0 = max(lens)
    kw = dict(scheme=w.scheme, layers=1, batch=nseq, q_heads=w.q_heads, kv_heads=w.kv_heads,
              head_dim=w.head_dim, bits=w.bits, group_k=w.group_k, group_v=w.group_v,
              residual=w.residual, max_tokens=n0 + 4096, in_dtype=0 if w.in_dtype == "bf16" else 1)
    img = O.Image(O.make_config(**kw))
    import torch
    k, v = W.kv_tokens(w, 0, 0, nseq, 0, n0, device="cpu", tag="cpu")
    to = (lambda t: t.view(torch.int16).numpy().view(np.uint16)) if w.in_dtype == "bf16" else (lambda t: t.numpy())
    sc = W.fp8_scales(w, k, v).numpy() if w.scheme == 2 else None
    img.append(0, 0, to(k), to(v), n_valid=np.asarray(lens, np.int32), fp8_scales=sc)
    q = W.queries(w, 0, device="cpu").float().numpy()[:nseq]
    kn, vn = W.kv_tokens(w, 0, 0, nseq, n0, 4096, device="cpu", tag="cpu-steps")
    return img, q, to(kn), to(vn), sc


def oracle_steps(w, img, q, kn, vn, sc, nsteps, seqs_per_step, threads, t_index):
    """nsteps oracle steps; each appends one token to every sequence and decodes
    `seqs_per_step` of them (one thread per sequence).  Returns decoded sequences."""
    nseq = q.shape[0]
    done = 0
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        for s in range(nsteps):
            j = (t_index + s) % kn.shape[1]
            img.append(0, 0, kn[:, j:j + 1], vn[:, j:j + 1], fp8_scales=sc)
            seqs = [(t_index + s + i) % nseq for i in range(seqs_per_step)]
            list(ex.map(lambda b: img.decode(0, q, w.scale, seq_begin=b, seq_count=1), seqs))
            done += seqs_per_step
    return done


def run_oracle(w, steps, warmup, budget_s, adapt_steps=False):
    """Time the oracle on a bounded sample of the workload.  Returns (tokens/s, seconds,
    threads, sequences decoded per step, sequences in the image, steps run)."""
    nseq = min(w.batch, 8)
    cores = len(os.sched_getaffinity(0))
    img, q, kn, vn, sc = oracle_setup(w, nseq)
    threads = min(cores, nseq)
    t = time.perf_counter()
    oracle_steps(w, img, q, kn, vn, sc, max(1, warmup), 1, 1, 0)
    per_seq = (time.perf_counter() - t) / max(1, warmup)
    if adapt_steps:
        steps = int(max(1, min(steps, budget_s / max(1e-9, per_seq * nseq / threads))))
    spp = int(max(1, min(nseq, budget_s / max(1e-9, steps * per_seq) * threads)))
    t = time.perf_counter()
    done = oracle_steps(w, img, q, kn, vn, sc, steps, spp, threads, warmup)
    el = time.perf_counter() - t
    return done / el, el, threads, spp, nseq, steps


# ---------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="kivi2_llama3_8b")
    ap.add_argument("--replicas", type=int, default=0, help="cache replicas (0: enough to exceed 4x L2)")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work per run")
    ap.add_argument("--all-layers", action="store_true",
                    help="time every layer of a multi-layer workload in each step (default: one layer)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    from quantised_kv_cache_kvq_gb300 import workloads as W
    w = W.WORKLOADS[args.workload]
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    peak, peak_kind = peaks()
    ragged = w.context[0] != w.context[1]
    config = {"workload": w.name, "scheme": ["kivi", "int8", "fp8"][w.scheme], "bits": w.bits,
              "batch": w.batch, "q_heads": w.q_heads, "kv_heads": w.kv_heads, "head_dim": w.head_dim,
              "context": list(w.context) if ragged else w.context[0], "group_k": w.group_k,
              "group_v": w.group_v, "residual": w.residual,
              "layers": w.layers if args.all_layers else 1}

    if args.impl == "reference":
        if rank != 0:
            return
        import __graft_entry__  # noqa: F401  (oracle build)
        from oracle import build as ob
        ob.build()
        tps, el, threads, spp, nseq, _ = run_oracle(w, args.steps, args.warmup, args.cpu_budget)
        sample = ("%d steps; each appends one token to %d sequences and decodes %d of them "
                  "(%d KV heads, contexts of the workload's first %d sequences, one layer)"
                  % (args.steps, nseq, spp, w.kv_heads, nseq))
        line = {"impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    import __graft_entry__
    __graft_entry__.build()
    r = run_gpu(args, w, rank, world)
    if rank != 0:
        return
    tokens = w.batch * args.steps * world
    value = tokens / (r["step_ms"] / 1e3)
    launches = args.steps * r["layers"]                 # decode calls in the decode-only graph
    dec_avg_ms = r["decode_ms"] / launches
    achieved = (r["bytes_decode"] / launches) / (dec_avg_ms / 1e3) / 1e9
    step_gbs = r["bytes_steps"] / (r["step_ms"] / 1e3) / 1e9
    cpu = None
    try:
        tps, el, threads, spp, nseq, ns = run_oracle(w, 8, 1, args.cpu_budget, adapt_steps=True)
        cpu = {"value": tps / r["layers"], "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": "%d oracle steps of the same workload on %d sequences, each appending one token "
                         "to all and decoding %d of them (%.1f s)%s"
                         % (ns, nseq, spp, el, "; one layer timed, divided by the %d layers a token "
                            "needs" % r["layers"] if r["layers"] > 1 else "")}
    except Exception as exc:  # the GPU number stands without it
        cpu = {"value": None, "unit": "tokens/s", "cores": 0, "kind": "oracle", "sample": "failed: %s" % exc}
    cfg = dict(config)
    cfg.update({"replicas": r["reps"], "cache_mb_per_replica": round(r["cache_mb"], 2),
                "mean_context": round(r["mean_context"], 1), "fill_s": round(r["fill_s"], 1),
                "l2": "inputs larger than L2: %d cache replica(s) rotated per step (%.0f MB > 129 MB)"
                      % (r["reps"], r["reps"] * r["cache_mb"]),
                "timing": "CUDA graph of the timed steps, CUDA events on the launch stream",
                "parallelism": "replicas" if world > 1 else "single"})
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["step_ms"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": cfg,
        "hbm_gbs": step_gbs, "hbm_pct_of_peak": 100.0 * step_gbs / peak,
        "roofline": {"kernel": "kvq decode attention (split-context kernel + merge)", "bound": "hbm",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "traffic": profiled_traffic(w.name, w.scheme),
                     "avg_launch_us": 1e3 * dec_avg_ms,
                     "bytes_per_launch": r["bytes_decode"] / launches},
        "cpu_baseline": cpu,
        "e2e": {"value": w.batch * r["e2e_steps"] * world / (r["e2e_ms"] / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"], "steps": r["e2e_steps"]},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
