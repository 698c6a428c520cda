"""Test harness: drives the CUDA library and the oracle with the same seeded inputs.

Both caches start from zeroed memory, so after the same calls their whole images
(header, status word, token counts, group records, bf16 window) must be byte-identical.
"""
import math

import numpy as np
import torch

import oracle as O
import quantised_kv_cache_kvq_gb300 as K

# tolerance of the attention outputs against the binary64 oracle: per element
# |gpu - oracle| <= ATOL + RTOL * |oracle|  (max-abs 2e-3, max-rel 1e-2)
ATOL, RTOL = 2e-3, 1e-2


def to_np_input(x: torch.Tensor):
    x = x.contiguous().cpu()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    return x.numpy().astype(np.float32)


def q_as_float(q: torch.Tensor) -> np.ndarray:
    return q.float().cpu().numpy().astype(np.float32)


class Pair:
    def __init__(self, scheme="kivi", layers=1, batch=2, q_heads=8, kv_heads=2, head_dim=128,
                 max_tokens=256, bits=2, group_k=32, group_v=32, residual=32, in_dtype="bf16",
                 page_groups=0, num_pages=0, block_table=None, rope_base=0.0, outliers=0):
        sch = {"kivi": 0, "int8": 1, "fp8": 2, "fp8e5m2": 3, "int4": 4}[scheme]
        dt = 0 if in_dtype == "bf16" else 1
        self.kw = dict(scheme=sch, layers=layers, batch=batch, q_heads=q_heads, kv_heads=kv_heads,
                       head_dim=head_dim, bits=bits if sch == 0 else (4 if sch == 4 else 8), group_k=group_k,
                       group_v=group_v, residual=residual, max_tokens=max_tokens, in_dtype=dt,
                       page_groups=page_groups, num_pages=num_pages, outliers=outliers)
        self.lib_cfg = K.KvqConfig(**self.kw)
        self.lib_cfg.rope_base = rope_base
        self.kw["rope_base"] = rope_base
        self.orc_cfg = O.make_config(**self.kw)
        if block_table is not None:
            self.set_block_table(block_table)
        self.torch_dtype = torch.bfloat16 if dt == 0 else torch.float32
        self.nbytes = K.kvq_cache_bytes(self.lib_cfg, max_tokens)
        self.img = O.Image(self.orc_cfg)
        assert self.nbytes == self.img.nbytes
        self.gpu = torch.zeros(self.nbytes, dtype=torch.uint8, device="cuda")
        K.kvq_cache_init(self.lib_cfg, self.gpu)
        self.ws = torch.zeros(K.kvq_workspace_bytes(self.lib_cfg), dtype=torch.uint8, device="cuda")

    def set_block_table(self, table):
        """Paged layout: the same block table (int32 [batch][max_pages]) on both sides."""
        table = np.ascontiguousarray(table, dtype=np.int32)
        self.lib_cfg.set_block_table(torch.from_numpy(table).cuda())
        O.set_block_table(self.orc_cfg, table)

    # ------------------------------------------------------------------ inputs
    def rand_kv(self, seq_count, n_new, gen, scale=1.0, outliers=True):
        H, D = self.kw["kv_heads"], self.kw["head_dim"]
        k = torch.randn(seq_count, n_new, H, D, generator=gen) * scale
        v = torch.randn(seq_count, n_new, H, D, generator=gen) * scale
        if outliers:
            k[..., 3] *= 12.0
            k[..., D // 2 + 1] *= 9.0
            hit = torch.rand(seq_count, n_new, generator=gen) < 0.05
            v *= torch.where(hit, 8.0, 1.0)[..., None, None]
        return k.to(self.torch_dtype), v.to(self.torch_dtype)

    def rand_q(self, gen, scale=1.0):
        q = torch.randn(self.kw["batch"], self.kw["q_heads"], self.kw["head_dim"], generator=gen) * scale
        return q.to(self.torch_dtype)

    # ------------------------------------------------------------------ calls on both sides
    def append(self, layer, k, v, seq_begin=0, n_valid=None, fp8_scales=None, flags=0):
        nv_gpu = None if n_valid is None else torch.tensor(n_valid, dtype=torch.int32, device="cuda")
        sc_gpu = None if fp8_scales is None else fp8_scales.to(torch.float32).contiguous().cuda()
        kg, vg = k.contiguous().cuda(), v.contiguous().cuda()
        K.kvq_quantize_append(self.lib_cfg, self.gpu, layer, seq_begin, k.shape[0], kg, vg, k.shape[1],
                              nv_gpu, sc_gpu, flags)
        self.img.append(layer, seq_begin, to_np_input(k), to_np_input(v),
                        None if n_valid is None else np.asarray(n_valid, np.int32),
                        None if fp8_scales is None else fp8_scales.float().numpy(), flags)
        torch.cuda.synchronize()

    def flush(self, layer):
        K.kvq_flush_group(self.lib_cfg, self.gpu, layer)
        self.img.flush(layer)
        torch.cuda.synchronize()

    def assert_same_image(self):
        torch.cuda.synchronize()
        g = self.gpu.cpu().numpy()
        o = self.img.buf
        if not np.array_equal(g, o):
            bad = np.nonzero(g != o)[0]
            reg = self.img.regions()
            raise AssertionError(
                "cache images differ at %d bytes; first at %d (gpu %#x, oracle %#x); regions %s"
                % (bad.size, bad[0], g[bad[0]], o[bad[0]], reg))

    def decode(self, layer, q, scale=None):
        if scale is None:
            scale = 1.0 / math.sqrt(self.kw["head_dim"])
        out = torch.empty(self.kw["batch"], self.kw["q_heads"], self.kw["head_dim"], dtype=torch.float32,
                          device="cuda")
        self.ws[:4].zero_()
        K.kvq_decode_attention(self.lib_cfg, self.gpu, layer, q.contiguous().cuda(), scale, out, self.ws)
        torch.cuda.synchronize()
        ref = self.img.decode(layer, q_as_float(q), scale)
        return out.cpu().numpy().astype(np.float64), ref

    def status(self):
        return K.kvq_read_status(self.gpu, self.ws)


def assert_close(got, ref, atol=ATOL, rtol=RTOL, what=""):
    err = np.abs(got - ref)
    ok = err <= atol + rtol * np.abs(ref)
    if not ok.all():
        i = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(ref))), err.shape)
        raise AssertionError("%s: %d elements outside tolerance; worst at %s: gpu %r oracle %r"
                             % (what, int((~ok).sum()), i, got[i], ref[i]))
    big = np.abs(ref) > 1e-2
    return float(err.max()), float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
