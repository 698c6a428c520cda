"""GB300 quantised KV cache: packed KIVI / INT8 / FP8 caches and single-query decode
attention over them, in CUDA kernels behind the C ABI of include/kvq.h.

`QuantizedKVCache` is a convenience holder: it allocates the cache and the decode
workspace as torch device tensors (torch serves only as the device allocator and stream
source) and forwards every call to libkvq.so.
"""
import math

from ._native import (  # noqa: F401
    EXPORTS, KVQ_BYTES_FORMULA, KVQ_BYTES_LAYOUT, KVQ_DTYPE_BF16, KVQ_DTYPE_F32,
    KVQ_NO_AUTOFLUSH, KVQ_SCHEME_FP8_E4M3, KVQ_SCHEME_FP8_E5M2, KVQ_SCHEME_INT4, KVQ_SCHEME_INT8,
    KVQ_SCHEME_KIVI,
    KVQ_STATUS_BAD_PAGE, KVQ_STATUS_CAPACITY, KVQ_STATUS_NONFINITE, KVQ_STATUS_RING_FULL, KVQ_STATUS_TIMEOUT,
    KvqConfig, KvqError, kvq_cache_bytes, kvq_cache_init, kvq_decode_attention,
    kvq_decode_attention_noalloc,
    kvq_flush_group, kvq_quantize_append, kvq_read_status, kvq_sequence_lengths,
    kvq_workspace_bytes, library_path, load, status_string,
)

_SCHEMES = {"kivi": KVQ_SCHEME_KIVI, "int8": KVQ_SCHEME_INT8, "fp8": KVQ_SCHEME_FP8_E4M3,
            "fp8e5m2": KVQ_SCHEME_FP8_E5M2, "int4": KVQ_SCHEME_INT4}


def make_config(scheme, layers, batch, q_heads, kv_heads, head_dim, max_tokens, bits=None,
                group_k=32, group_v=32, residual=0, in_dtype="bf16", page_groups=0, num_pages=0,
                block_table=None, rope_base=0.0, outliers=0) -> KvqConfig:
    """block_table: paged KIVI layout, a device int32 tensor [batch][max_pages]; rope_base:
    KIVI keys cached before the rotary embedding (its base; 0 for keys cached as given);
    outliers: KIVI dense-and-sparse, elements per quantisation vector kept aside in bf16."""
    s = _SCHEMES[scheme] if isinstance(scheme, str) else int(scheme)
    if bits is None:
        bits = {KVQ_SCHEME_KIVI: 2, KVQ_SCHEME_INT4: 4}.get(s, 8)
    c = KvqConfig()
    c.scheme, c.layers, c.batch, c.q_heads, c.kv_heads = s, layers, batch, q_heads, kv_heads
    c.head_dim, c.bits, c.group_k, c.group_v, c.residual = head_dim, bits, group_k, group_v, residual
    c.max_tokens = max_tokens
    c.in_dtype = KVQ_DTYPE_BF16 if in_dtype in ("bf16", KVQ_DTYPE_BF16) else KVQ_DTYPE_F32
    c.page_groups, c.num_pages = page_groups, num_pages
    c.rope_base = float(rope_base)
    c.outliers = int(outliers)
    c.set_block_table(block_table)
    return c


def max_pages(cfg) -> int:
    """Block-table entries per sequence of a paged configuration."""
    ng = (cfg.max_tokens - cfg.residual) // cfg.group_k if cfg.max_tokens > cfg.residual else 0
    return (ng + cfg.page_groups - 1) // cfg.page_groups if cfg.page_groups > 0 else 0


class QuantizedKVCache:
    """A cache and its decode workspace on one GPU."""

    def __init__(self, cfg: KvqConfig, device="cuda"):
        import torch
        load()
        self.cfg = cfg
        self.device = torch.device(device)
        self.nbytes = kvq_cache_bytes(cfg, cfg.max_tokens, KVQ_BYTES_LAYOUT)
        self.cache = torch.empty(self.nbytes, dtype=torch.uint8, device=self.device)
        kvq_cache_init(cfg, self.cache)
        self.workspace = torch.zeros(kvq_workspace_bytes(cfg), dtype=torch.uint8, device=self.device)

    def append(self, layer, k_new, v_new, seq_begin=0, n_valid=None, fp8_scales=None, flags=0,
               stream=None):
        """k_new, v_new: [seq_count][n_new][kv_heads][head_dim] device tensors."""
        seq_count, n_new = k_new.shape[0], k_new.shape[1]
        kvq_quantize_append(self.cfg, self.cache, layer, seq_begin, seq_count, k_new, v_new, n_new,
                            n_valid, fp8_scales, flags, stream)

    def flush(self, layer, stream=None):
        kvq_flush_group(self.cfg, self.cache, layer, stream)

    def decode(self, layer, q, softmax_scale=None, out=None, stream=None):
        import torch
        if softmax_scale is None:
            softmax_scale = 1.0 / math.sqrt(self.cfg.head_dim)
        if out is None:
            out = torch.empty(self.cfg.batch, self.cfg.q_heads, self.cfg.head_dim,
                              dtype=torch.float32, device=self.device)
        kvq_decode_attention(self.cfg, self.cache, layer, q, softmax_scale, out, self.workspace,
                             stream=stream)
        return out

    def status(self, stream=None):
        return kvq_read_status(self.cache, self.workspace, stream)

    def lengths(self, layer, stream=None):
        import torch
        n = torch.empty(self.cfg.batch, dtype=torch.int32, device=self.device)
        qn = torch.empty(self.cfg.batch, dtype=torch.int32, device=self.device)
        kvq_sequence_lengths(self.cfg, self.cache, layer, n, qn, stream)
        return n, qn
