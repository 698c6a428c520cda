"""ctypes binding of libkvq.so (include/kvq.h): the same entry points, argument
marshalling only.  Every step of the cache runs in the library's CUDA kernels; there is
no Python or CPU fallback, and loading fails loudly if the library was not built."""
import ctypes as C
import os

from . import build as _build

KVQ_SCHEME_KIVI, KVQ_SCHEME_INT8, KVQ_SCHEME_FP8_E4M3, KVQ_SCHEME_FP8_E5M2, KVQ_SCHEME_INT4 = 0, 1, 2, 3, 4
KVQ_DTYPE_BF16, KVQ_DTYPE_F32 = 0, 1
KVQ_BYTES_FORMULA, KVQ_BYTES_LAYOUT = 0, 1
KVQ_NO_AUTOFLUSH = 1
KVQ_OK, KVQ_ERR_ARG, KVQ_ERR_ALIGN, KVQ_ERR_CAPACITY = 0, -1, -2, -3
KVQ_ERR_WORKSPACE, KVQ_ERR_CUDA, KVQ_ERR_UNSUPPORTED = -4, -5, -6
KVQ_STATUS_CAPACITY, KVQ_STATUS_RING_FULL, KVQ_STATUS_NONFINITE, KVQ_STATUS_TIMEOUT = 1, 2, 4, 8
KVQ_STATUS_BAD_PAGE = 16

# every symbol include/kvq.h declares
EXPORTS = (
    "kvq_cache_bytes", "kvq_cache_init", "kvq_quantize_append", "kvq_flush_group",
    "kvq_workspace_bytes", "kvq_decode_attention", "kvq_decode_attention_noalloc", "kvq_read_status",
    "kvq_sequence_lengths", "kvq_status_string",
)
KVQ_NOALLOC_SCRATCH_BYTES = 16 << 20
KVQ_MAX_DECODE_BLOCKS = 2048
KVQ_SELFTEST_WAIT_MAGIC = 0x4b56515449434b31


class KvqConfig(C.Structure):
    """struct kvq_config"""
    _fields_ = [(n, C.c_int32) for n in (
        "scheme", "layers", "batch", "q_heads", "kv_heads", "head_dim", "bits", "group_k",
        "group_v", "residual", "max_tokens", "in_dtype", "page_groups", "num_pages")] + [
        ("block_table", C.c_void_p), ("rope_base", C.c_float), ("outliers", C.c_int32)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}

    def set_block_table(self, table):
        """Paged layout: point the configuration at a device int32 [batch][max_pages] tensor
        (kept alive here) or None."""
        self._table = table
        self.block_table = None if table is None else int(table.data_ptr())


class KvqError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__("%s failed: %d (%s)" % (fn, code, status_string(code)))
        self.code = code


_lib = None


def library_path():
    return _build.LIB


def load():
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(
            "libkvq.so is not built (expected at %s): build it with "
            "`python -m quantised_kv_cache_kvq_gb300.build` or __graft_entry__.build()" % path)
    L = C.CDLL(path)
    P, i32, i64, u32, u64 = C.c_void_p, C.c_int32, C.c_int64, C.c_uint32, C.c_uint64
    cfgp = C.POINTER(KvqConfig)
    sig = {
        "kvq_cache_bytes": [cfgp, i64, i32, C.POINTER(u64)],
        "kvq_cache_init": [cfgp, P, P],
        "kvq_quantize_append": [cfgp, P, i32, i32, i32, P, P, i32, P, P, u32, P],
        "kvq_flush_group": [cfgp, P, i32, P],
        "kvq_workspace_bytes": [cfgp, C.POINTER(u64)],
        "kvq_decode_attention": [cfgp, P, i32, P, C.c_float, P, P, u64, P],
        "kvq_decode_attention_noalloc": [cfgp, P, i32, P, C.c_float, P, P],
        "kvq_read_status": [P, P, C.POINTER(u32), P],
        "kvq_sequence_lengths": [cfgp, P, i32, P, P, P],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = C.c_int
    L.kvq_status_string.argtypes = [C.c_int]
    L.kvq_status_string.restype = C.c_char_p
    _lib = L
    return L


def status_string(code):
    return load().kvq_status_string(int(code)).decode()


def _ptr(x):
    """Device pointer of a torch tensor, or an integer address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, code):
    if code != KVQ_OK:
        raise KvqError(fn, code)


# ---------------------------------------------------------------------------- entry points
def kvq_cache_bytes(cfg, tokens, mode=KVQ_BYTES_LAYOUT):
    out = C.c_uint64(0)
    _check("kvq_cache_bytes", load().kvq_cache_bytes(C.byref(cfg), int(tokens), int(mode), C.byref(out)))
    return out.value


def kvq_cache_init(cfg, cache, stream=None):
    _check("kvq_cache_init", load().kvq_cache_init(C.byref(cfg), _ptr(cache), _stream(stream)))


def kvq_quantize_append(cfg, cache, layer, seq_begin, seq_count, k_new, v_new, n_new,
                        n_valid=None, fp8_scales=None, flags=0, stream=None):
    _check("kvq_quantize_append", load().kvq_quantize_append(
        C.byref(cfg), _ptr(cache), int(layer), int(seq_begin), int(seq_count), _ptr(k_new),
        _ptr(v_new), int(n_new), _ptr(n_valid), _ptr(fp8_scales), int(flags), _stream(stream)))


def kvq_flush_group(cfg, cache, layer, stream=None):
    _check("kvq_flush_group", load().kvq_flush_group(C.byref(cfg), _ptr(cache), int(layer), _stream(stream)))


def kvq_workspace_bytes(cfg):
    out = C.c_uint64(0)
    _check("kvq_workspace_bytes", load().kvq_workspace_bytes(C.byref(cfg), C.byref(out)))
    return out.value


def kvq_decode_attention(cfg, cache, layer, q, softmax_scale, out, workspace, workspace_bytes=None,
                         stream=None):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("kvq_decode_attention", load().kvq_decode_attention(
        C.byref(cfg), _ptr(cache), int(layer), _ptr(q), float(softmax_scale), _ptr(out),
        _ptr(workspace), int(workspace_bytes), _stream(stream)))


def kvq_decode_attention_noalloc(cfg, cache, layer, q, softmax_scale, out, stream=None):
    """Decode with the library's own fixed scratch (no workspace argument; see kvq.h)."""
    _check("kvq_decode_attention_noalloc", load().kvq_decode_attention_noalloc(
        C.byref(cfg), _ptr(cache), int(layer), _ptr(q), float(softmax_scale), _ptr(out), _stream(stream)))


def kvq_read_status(cache=None, workspace=None, stream=None):
    out = C.c_uint32(0)
    _check("kvq_read_status", load().kvq_read_status(_ptr(cache), _ptr(workspace), C.byref(out),
                                                     _stream(stream)))
    return out.value


def kvq_sequence_lengths(cfg, cache, layer, n_out=None, qn_out=None, stream=None):
    _check("kvq_sequence_lengths", load().kvq_sequence_lengths(
        C.byref(cfg), _ptr(cache), int(layer), _ptr(n_out), _ptr(qn_out), _stream(stream)))
