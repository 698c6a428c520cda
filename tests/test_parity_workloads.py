"""Parity at the shapes of the five benchmark workloads, through the C ABI.

Each workload is built on the GPU from `workloads.py` at its real size (the seeded draws
are made on the device and the slices the oracle needs are copied to the host), then
compared with the oracle:

* KIVI 2-bit Llama-3-8B layer (8 sequences x 4096 tokens): the whole cache image byte for
  byte after the prefill and after one decode step, and every output element.
* KIVI 4-bit, one 131072-token sequence: the whole image and every output element, also
  with one outlier per quantisation vector kept aside in bf16 (dense-and-sparse).
* FP8, 32 layers x 64 sequences x 8192 tokens: the cache is filled for every layer; the
  byte ranges, token counts, scales and outputs of layers {0, 31} x 4 sampled sequences
  are compared.
* Serving mix, 256 ragged sequences, 64 steps of (append one token, flush, decode): every
  sequence runs on the GPU; the oracle mirrors 8 sampled sequences.  Their group records,
  windows and token counts are compared after steps with flushes, and their outputs every
  8 steps.

Outputs must satisfy |gpu - oracle| <= 2e-3 + 1e-2 |oracle| per element (harness.ATOL,
RTOL).
"""
import concurrent.futures as cf
import ctypes as C

import numpy as np
import pytest
import torch

import oracle as O
from harness import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _np_bits(t):
    """bf16 tensor -> uint16 bit patterns (host); fp32 -> float32."""
    t = t.contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _kw(w, batch, layers, max_tokens):
    return dict(scheme=w.scheme, layers=layers, batch=batch, q_heads=w.q_heads, kv_heads=w.kv_heads,
                head_dim=w.head_dim, bits=w.bits if w.scheme == 0 else 8, group_k=w.group_k,
                group_v=w.group_v, residual=w.residual, max_tokens=max_tokens,
                in_dtype=0 if w.in_dtype == "bf16" else 1, outliers=w.outliers)


def _regions(kw):
    """Region offsets of a cache layout (oracle arithmetic, no allocation)."""
    out = np.zeros(6, np.int64)
    O.lib().kvqo_image_regions(C.byref(O.make_config(**kw)), out.ctypes.data_as(C.c_void_p))
    return dict(state=int(out[0]), scales=int(out[1]), data=int(out[2]), ring=int(out[3]),
                total=int(out[4]), unit=int(out[5]))


def _decode_layer(img, layer, q, scale, seqs, threads=16):
    """Oracle outputs of the given sequences of one layer, one thread per sequence (the C
    oracle releases the interpreter lock); other rows stay zero."""
    out = np.zeros((img.cfg.batch, img.cfg.q_heads, img.cfg.head_dim))
    with cf.ThreadPoolExecutor(max_workers=min(threads, len(seqs))) as ex:
        rows = ex.map(lambda b: img.decode(layer, q, scale, seq_begin=b, seq_count=1), seqs)
        for b, o in zip(seqs, rows):
            out[b] = o[b]
    return out


class GpuCache:
    def __init__(self, kw):
        import quantised_kv_cache_kvq_gb300 as K
        self.K = K
        self.cfg = K.KvqConfig(**kw)
        self.nbytes = K.kvq_cache_bytes(self.cfg, kw["max_tokens"])
        self.cache = torch.zeros(self.nbytes, dtype=torch.uint8, device="cuda")
        K.kvq_cache_init(self.cfg, self.cache)
        self.ws = torch.zeros(K.kvq_workspace_bytes(self.cfg), dtype=torch.uint8, device="cuda")

    def append(self, layer, k, v, seq_begin=0, n_valid=None, fp8_scales=None):
        nv = None if n_valid is None else torch.tensor(n_valid, dtype=torch.int32, device="cuda")
        self.K.kvq_quantize_append(self.cfg, self.cache, layer, seq_begin, k.shape[0], k.contiguous(),
                                   v.contiguous(), k.shape[1], nv, fp8_scales)

    def decode(self, layer, q, scale):
        out = torch.empty(self.cfg.batch, self.cfg.q_heads, self.cfg.head_dim, dtype=torch.float32,
                          device="cuda")
        self.K.kvq_decode_attention(self.cfg, self.cache, layer, q.contiguous(), scale, out, self.ws)
        torch.cuda.synchronize()
        return out.cpu().numpy().astype(np.float64)

    def status(self):
        return self.K.kvq_read_status(self.cache, self.ws)

    def bytes(self, off, n):
        return self.cache[off:off + n].cpu().numpy()


def _assert_bytes(got, ref, what):
    if not np.array_equal(got, ref):
        bad = np.nonzero(got != ref)[0]
        raise AssertionError("%s: %d bytes differ, first at %d (gpu %#x, oracle %#x)"
                             % (what, bad.size, bad[0], got[bad[0]], ref[bad[0]]))


# --------------------------------------------------------------------------- whole images
@pytest.mark.parametrize("name", ["kivi2_llama3_8b", "kivi4_128k", "kivi4_128k_sparse"])
def test_workload_whole_image_and_outputs(name):
    from quantised_kv_cache_kvq_gb300 import workloads as W
    w = W.WORKLOADS[name]
    n0 = w.context[0]
    kw = _kw(w, w.batch, 1, n0 + 16)
    gpu = GpuCache(kw)
    img = O.Image(O.make_config(**kw))
    assert gpu.nbytes == img.nbytes
    # prefill: the workload's context through the bulk path, 8 sequences per call
    for s0 in range(0, w.batch, 8):
        ns = min(8, w.batch - s0)
        k, v = W.kv_tokens(w, 0, s0, ns, 0, n0, device="cuda", tag="ctx")
        gpu.append(0, k, v, seq_begin=s0)
        img.append(0, s0, _np_bits(k), _np_bits(v))
        del k, v
    torch.cuda.synchronize()
    _assert_bytes(gpu.bytes(0, gpu.nbytes), img.buf, "%s image after prefill" % name)
    seqs = list(range(w.batch))
    for step in range(2):
        # one decode step: append one token per sequence (the one-kernel path), then decode
        k, v = W.kv_tokens(w, 0, 0, w.batch, n0 + step, 1, device="cuda", tag="step")
        gpu.append(0, k, v)
        img.append(0, 0, _np_bits(k), _np_bits(v))
        q = W.queries(w, 0, step, device="cuda")
        out = gpu.decode(0, q, w.scale)
        _assert_bytes(gpu.bytes(0, gpu.nbytes), img.buf, "%s image after step %d" % (name, step))
        ref = _decode_layer(img, 0, q.float().cpu().numpy(), w.scale, seqs)
        mabs, mrel = assert_close(out, ref, what="%s step %d" % (name, step))
        print("%s step %d: max abs %.3g, max rel %.3g" % (name, step, mabs, mrel))
    assert gpu.status() == 0 and img.status == 0


# --------------------------------------------------------------------------- FP8, 32 layers
def test_workload_fp8_32layer_sampled():
    from quantised_kv_cache_kvq_gb300 import workloads as W
    w = W.WORKLOADS["fp8_32layer"]
    n0 = w.context[0]
    T = n0 + 16
    kw = _kw(w, w.batch, w.layers, T)
    gpu = GpuCache(kw)
    reg = _regions(kw)
    layers = [0, w.layers - 1]
    seqs = [0, 21, 42, 63]
    okw = _kw(w, len(seqs), len(layers), T)
    img = O.Image(O.make_config(**okw))
    oreg = img.regions()
    assert oreg["unit"] == reg["unit"]
    for layer in range(w.layers):
        scales = None
        for s0 in range(0, w.batch, 8):
            k, v = W.kv_tokens(w, layer, s0, 8, 0, n0, device="cuda", tag="ctx")
            if scales is None:   # static per-(kv head) scales from the layer's first fill
                scales = W.fp8_scales(w, k, v)
            gpu.append(layer, k, v, seq_begin=s0, fp8_scales=scales)
            if layer in layers:
                li = layers.index(layer)
                for i, b in enumerate(seqs):
                    if s0 <= b < s0 + 8:
                        img.append(li, i, _np_bits(k[b - s0:b - s0 + 1]), _np_bits(v[b - s0:b - s0 + 1]),
                                   fp8_scales=scales.cpu().numpy())
            del k, v
    torch.cuda.synchronize()
    H, unit = w.kv_heads, reg["unit"]
    for li, layer in enumerate(layers):
        # the layer's scale table row
        _assert_bytes(gpu.bytes(reg["scales"] + layer * H * 8, H * 8),
                      img.buf[oreg["scales"] + li * H * 8: oreg["scales"] + (li + 1) * H * 8],
                      "fp8 scales layer %d" % layer)
        for i, b in enumerate(seqs):
            st = reg["state"] + 16 * (layer * w.batch + b)
            ost = oreg["state"] + 16 * (li * len(seqs) + i)
            _assert_bytes(gpu.bytes(st, 8), img.buf[ost:ost + 8], "state l%d s%d" % (layer, b))
            u = (layer * w.batch + b) * H
            ou = (li * len(seqs) + i) * H
            _assert_bytes(gpu.bytes(reg["data"] + u * unit, H * unit),
                          img.buf[oreg["data"] + ou * unit: oreg["data"] + (ou + H) * unit],
                          "fp8 codes layer %d seq %d" % (layer, b))
    for li, layer in enumerate(layers):
        q = W.queries(w, layer, 0, device="cuda")
        out = gpu.decode(layer, q, w.scale)
        qs = q.float().cpu().numpy()[seqs]
        ref = _decode_layer(img, li, qs, w.scale, list(range(len(seqs))))
        mabs, mrel = assert_close(out[seqs], ref, what="fp8 layer %d" % layer)
        print("fp8 layer %d: max abs %.3g, max rel %.3g" % (layer, mabs, mrel))
    assert gpu.status() == 0


# --------------------------------------------------------------------------- serving mix
def test_workload_serve_mix_steps_sampled():
    from quantised_kv_cache_kvq_gb300 import workloads as W
    w = W.WORKLOADS["serve_mix"]
    lens = [int(x) for x in W.context_lengths(w).tolist()]
    T = max(lens) + w.steps + 16
    kw = _kw(w, w.batch, 1, T)
    gpu = GpuCache(kw)
    reg = _regions(kw)
    seqs = [0, 37, 74, 111, 148, 185, 222, 255]
    okw = _kw(w, len(seqs), 1, T)
    img = O.Image(O.make_config(**okw))
    oreg = img.regions()
    assert oreg["unit"] == reg["unit"]
    for s0 in range(0, w.batch, 8):
        nl = lens[s0:s0 + 8]
        k, v = W.kv_tokens(w, 0, s0, 8, 0, max(nl), device="cuda", tag="ctx")
        gpu.append(0, k, v, seq_begin=s0, n_valid=nl)
        for i, b in enumerate(seqs):
            if s0 <= b < s0 + 8:
                img.append(0, i, _np_bits(k[b - s0:b - s0 + 1, :lens[b]]), _np_bits(v[b - s0:b - s0 + 1, :lens[b]]))
        del k, v
    torch.cuda.synchronize()
    H, D, unit = w.kv_heads, w.head_dim, reg["unit"]
    rec = unit // ((T - w.residual) // w.group_k)
    ring_unit = (w.residual + w.group_k) * 4 * D

    def compare_sampled(step):
        for i, b in enumerate(seqs):
            st = reg["state"] + 16 * b
            ost = oreg["state"] + 16 * i
            _assert_bytes(gpu.bytes(st, 8), img.buf[ost:ost + 8], "state seq %d step %d" % (b, step))
            n, qn = img.state(0, i)
            for h in range(H):
                u, ou = b * H + h, i * H + h
                used = (qn // w.group_k) * rec
                _assert_bytes(gpu.bytes(reg["data"] + u * unit, used),
                              img.buf[oreg["data"] + ou * unit: oreg["data"] + ou * unit + used],
                              "groups seq %d head %d step %d" % (b, h, step))
                _assert_bytes(gpu.bytes(reg["ring"] + u * ring_unit, ring_unit),
                              img.buf[oreg["ring"] + ou * ring_unit: oreg["ring"] + (ou + 1) * ring_unit],
                              "window seq %d head %d step %d" % (b, h, step))

    compare_sampled(-1)
    flushed = False
    for step in range(w.steps):
        k, v = W.kv_tokens(w, 0, 0, w.batch, max(lens) + step, 1, device="cuda", tag="step")
        gpu.append(0, k, v)
        ks, vs = _np_bits(k[seqs]), _np_bits(v[seqs])
        before = [img.state(0, i)[1] for i in range(len(seqs))]
        img.append(0, 0, ks, vs)
        flushed |= any(img.state(0, i)[1] != before[i] for i in range(len(seqs)))
        q = W.queries(w, 0, step, device="cuda")
        out = gpu.decode(0, q, w.scale)
        if step % 8 == 7:
            if flushed:
                compare_sampled(step)
                flushed = False
            ref = _decode_layer(img, 0, q.float().cpu().numpy()[seqs], w.scale, list(range(len(seqs))))
            mabs, mrel = assert_close(out[seqs], ref, what="serve mix step %d" % step)
            print("serve mix step %d: max abs %.3g, max rel %.3g" % (step, mabs, mrel))
    compare_sampled(w.steps)
    assert gpu.status() == 0 and img.status == 0
