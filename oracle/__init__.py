"""Python access to the quantised-KV-cache ORACLE (test infrastructure only).

The oracle is the plain C file ``kvq_oracle.c`` beside this module: a slow,
single-threaded CPU restatement of the method, pinned by
``tests/test_oracle_pins.py``.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg import this package; the CUDA library never does,
and the two share no code.

This module only marshals numpy arrays into the C functions.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None

SCHEME_KIVI, SCHEME_INT8, SCHEME_FP8, SCHEME_FP8_E5M2, SCHEME_INT4 = 0, 1, 2, 3, 4
DT_BF16, DT_F32 = 0, 1
ST_CAPACITY, ST_RING_FULL, ST_NONFINITE, ST_BAD_PAGE = 1, 2, 4, 16
FLAG_NO_AUTOFLUSH = 1


class OracleConfig(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "scheme", "layers", "batch", "q_heads", "kv_heads", "head_dim", "bits",
        "group_k", "group_v", "residual", "max_tokens", "in_dtype", "page_groups", "num_pages")] + [
        ("block_table", C.c_void_p), ("rope_base", C.c_float), ("outliers", C.c_int32)]


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        P = C.c_void_p
        i32, i64, u16, f32, f64, u32 = C.c_int32, C.c_int64, C.c_uint16, C.c_float, C.c_double, C.c_uint32
        sig = {
            "kvqo_kv_bytes": (f64, [f64] * 5),
            "kvqo_concurrency": (i64, [f64] * 8),
            "kvqo_half_to_float": (f32, [u16]),
            "kvqo_half_round": (u16, [f32, C.c_int]),
            "kvqo_e4m3_to_float": (f32, [C.c_uint8]),
            "kvqo_e4m3_from_float": (C.c_uint8, [f32]),
            "kvqo_e5m2_to_float": (f32, [C.c_uint8]),
            "kvqo_e5m2_from_float": (C.c_uint8, [f32]),
            "kvqo_int4_token": (None, [P, C.c_int, P, P]),
            "kvqo_qb_group": (None, [P, C.c_int, C.c_int, C.c_int, P, P, P]),
            "kvqo_qb_group_sparse": (None, [P, C.c_int, C.c_int, C.c_int, C.c_int, P, P, P, P]),
            "kvqo_qb_dequant": (f32, [C.c_int, u16, u16]),
            "kvqo_int8_token": (None, [P, C.c_int, P, P]),
            "kvqo_image_bytes": (i64, [P]),
            "kvqo_image_regions": (None, [P, P]),
            "kvqo_record_offset": (i64, [P, C.c_int, C.c_int, C.c_int, i64]),
            "kvqo_rope_key": (None, [C.c_int, f64, i64, P, P]),
            "kvqo_image_init": (None, [P, P]),
            "kvqo_append": (u32, [P, P, C.c_int, C.c_int, C.c_int, P, P, C.c_int, P, P, u32]),
            "kvqo_flush": (None, [P, P, C.c_int]),
            "kvqo_dequant_token": (None, [P, P, C.c_int, C.c_int, C.c_int, i64, P, P]),
            "kvqo_decode": (None, [P, P, C.c_int, C.c_int, C.c_int, P, f64, P]),
            "kvqo_decode_head": (None, [P, P, C.c_int, C.c_int, C.c_int, P, f64, P]),
            "kvqo_lse_merge": (None, [C.c_int, C.c_int, P, P, P, P]),
            "kvqo_partial": (None, [P, P, C.c_int, C.c_int, C.c_int, i64, i64, P, f64, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


# ----------------------------------------------------------------------------- scalars
def kv_bytes(layers, kv_heads, head_size, tokens, bytes_per_value):
    return lib().kvqo_kv_bytes(layers, kv_heads, head_size, tokens, bytes_per_value)


def concurrency(gpu_bytes, use_fraction, weight_bytes, layers, kv_heads, head_size, tokens,
                bytes_per_value):
    return lib().kvqo_concurrency(gpu_bytes, use_fraction, weight_bytes, layers, kv_heads,
                                  head_size, tokens, bytes_per_value)


def half_round(x, mode):
    """binary16 bits of float32 x rounded nearest-even (0), down (-1) or up (+1)."""
    return lib().kvqo_half_round(float(np.float32(x)), mode)


def half_to_float(h):
    return lib().kvqo_half_to_float(int(h))


def e4m3_from_float(x):
    return lib().kvqo_e4m3_from_float(float(np.float32(x)))


def e4m3_to_float(c):
    return lib().kvqo_e4m3_to_float(int(c))


def qb_group(x, bits):
    """Q_b over one group: returns (scale bits, zero bits, codes uint8)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    s = np.zeros(1, np.uint16)
    z = np.zeros(1, np.uint16)
    codes = np.zeros(x.size, np.uint8)
    lib().kvqo_qb_group(_p(x), x.size, 1, bits, _p(s), _p(z), _p(codes))
    return int(s[0]), int(z[0]), codes


def qb_group_sparse(x, bits, k):
    """Dense-and-sparse Q_b over one vector (bf16-exact float32 values): returns (scale
    bits, zero bits, codes uint8, side entries uint32 [k])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert 0 <= k < x.size
    s = np.zeros(1, np.uint16)
    z = np.zeros(1, np.uint16)
    codes = np.zeros(x.size, np.uint8)
    ent = np.zeros(max(k, 1), np.uint32)
    lib().kvqo_qb_group_sparse(_p(x), x.size, 1, bits, k, _p(s), _p(z), _p(codes), _p(ent))
    return int(s[0]), int(z[0]), codes, ent[:k]


def qb_dequant(code, scale_bits, zero_bits):
    return lib().kvqo_qb_dequant(int(code), int(scale_bits), int(zero_bits))


def e5m2_from_float(x):
    return lib().kvqo_e5m2_from_float(float(np.float32(x)))


def e5m2_to_float(c):
    return lib().kvqo_e5m2_to_float(int(c))


def int4_token(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    s = np.zeros(1, np.float32)
    codes = np.zeros(x.size, np.int8)
    lib().kvqo_int4_token(_p(x), x.size, _p(s), _p(codes))
    return float(s[0]), codes


def int8_token(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    s = np.zeros(1, np.float32)
    codes = np.zeros(x.size, np.int8)
    lib().kvqo_int8_token(_p(x), x.size, _p(s), _p(codes))
    return float(s[0]), codes


# ----------------------------------------------------------------------------- the cache image
def make_config(block_table=None, **kw):
    """block_table (paged KIVI layout): int32 [batch][max_pages], kept alive on the config."""
    c = OracleConfig()
    defaults = dict(scheme=0, layers=1, batch=1, q_heads=1, kv_heads=1, head_dim=64, bits=2,
                    group_k=32, group_v=32, residual=0, max_tokens=64, in_dtype=DT_BF16, page_groups=0,
                    num_pages=0, outliers=0)
    defaults.update(kw)
    k = int(defaults["outliers"])
    if k and not (0 < k <= 4 and k < defaults["group_k"] and k < defaults["group_v"]
                  and defaults["scheme"] == SCHEME_KIVI):
        raise ValueError("outliers: KIVI only, 1..4 and fewer than group_k and group_v")
    rope = float(defaults.pop("rope_base", 0.0))
    for k, v in defaults.items():
        setattr(c, k, int(v))
    c.rope_base = rope
    set_block_table(c, block_table)
    return c


def rope_key(k, pos, base):
    """The oracle's rotary embedding of one key row (float32 [D]) at position pos."""
    k = np.ascontiguousarray(k, np.float32)
    out = np.zeros(k.shape[0])
    lib().kvqo_rope_key(k.shape[0], float(base), int(pos), _p(k), _p(out))
    return out


def set_block_table(cfg, table):
    """Point the config at a (new) block table: int32 [batch][max_pages] or None."""
    cfg._table = None if table is None else np.ascontiguousarray(table, dtype=np.int32)
    cfg.block_table = None if cfg._table is None else cfg._table.ctypes.data


def record_offset(cfg, layer, seq, kv_head, group):
    """Byte offset of a KIVI group record in the image (either layout)."""
    return int(lib().kvqo_record_offset(C.byref(cfg), layer, seq, kv_head, group))


class Image:
    """A host cache image in the documented byte layout, driven by the oracle."""

    def __init__(self, cfg: OracleConfig):
        self.cfg = cfg
        self.nbytes = lib().kvqo_image_bytes(C.byref(cfg))
        self.buf = np.zeros(self.nbytes, np.uint8)
        lib().kvqo_image_init(C.byref(cfg), _p(self.buf))

    def regions(self):
        out = np.zeros(6, np.int64)
        lib().kvqo_image_regions(C.byref(self.cfg), _p(out))
        return dict(state=int(out[0]), scales=int(out[1]), data=int(out[2]), ring=int(out[3]),
                    total=int(out[4]), unit=int(out[5]))

    @property
    def status(self):
        return int(self.buf[:4].view(np.uint32)[0])

    def state(self, layer, seq):
        off = 256 + 16 * (layer * self.cfg.batch + seq)
        n, qn = self.buf[off:off + 8].view(np.int32)
        return int(n), int(qn)

    def _input(self, x):
        if self.cfg.in_dtype == DT_BF16:
            assert x.dtype == np.uint16, "bf16 inputs are passed as their uint16 bit patterns"
        else:
            assert x.dtype == np.float32
        return np.ascontiguousarray(x)

    def append(self, layer, seq_begin, k, v, n_valid=None, fp8_scales=None, flags=0):
        """k, v: [seq_count][n_new][kv_heads][head_dim] (uint16 bf16 bits or float32)."""
        k = self._input(k)
        v = self._input(v)
        seq_count, n_new = k.shape[0], k.shape[1]
        nv = None if n_valid is None else np.ascontiguousarray(n_valid, dtype=np.int32)
        sc = None if fp8_scales is None else np.ascontiguousarray(fp8_scales, dtype=np.float32)
        return lib().kvqo_append(C.byref(self.cfg), _p(self.buf), layer, seq_begin, seq_count,
                                 _p(k), _p(v), n_new, _p(nv), _p(sc), flags)

    def flush(self, layer):
        lib().kvqo_flush(C.byref(self.cfg), _p(self.buf), layer)

    def dequant_token(self, layer, seq, kvh, t):
        D = self.cfg.head_dim
        k = np.zeros(D, np.float32)
        v = np.zeros(D, np.float32)
        lib().kvqo_dequant_token(C.byref(self.cfg), _p(self.buf), layer, seq, kvh, t, _p(k), _p(v))
        return k, v

    def decode(self, layer, q, softmax_scale, seq_begin=0, seq_count=None):
        """q: float32 [batch][q_heads][head_dim] (full batch); returns float64 rows for the
        requested sequences (others left zero)."""
        q = np.ascontiguousarray(q, dtype=np.float32)
        if seq_count is None:
            seq_count = self.cfg.batch - seq_begin
        out = np.zeros((self.cfg.batch, self.cfg.q_heads, self.cfg.head_dim), np.float64)
        lib().kvqo_decode(C.byref(self.cfg), _p(self.buf), layer, seq_begin, seq_count, _p(q),
                          float(softmax_scale), _p(out))
        return out

    def decode_head(self, layer, q, softmax_scale, seq, kv_head, out):
        """Writes the outputs of the query heads of (seq, kv_head) into `out` (float64
        [batch][q_heads][head_dim], C-contiguous); q as for decode."""
        q = np.ascontiguousarray(q, dtype=np.float32)
        assert out.dtype == np.float64 and out.flags["C_CONTIGUOUS"]
        lib().kvqo_decode_head(C.byref(self.cfg), _p(self.buf), layer, seq, kv_head, _p(q),
                               float(softmax_scale), _p(out))

    def partial(self, layer, seq, hq, t0, t1, qrow, softmax_scale):
        D = self.cfg.head_dim
        qrow = np.ascontiguousarray(qrow, dtype=np.float32)
        m = np.zeros(1)
        lsum = np.zeros(1)
        o = np.zeros(D)
        lib().kvqo_partial(C.byref(self.cfg), _p(self.buf), layer, seq, hq, t0, t1, _p(qrow),
                           float(softmax_scale), _p(m), _p(lsum), _p(o))
        return float(m[0]), float(lsum[0]), o


def lse_merge(m, lsum, o):
    m = np.ascontiguousarray(m, np.float64)
    lsum = np.ascontiguousarray(lsum, np.float64)
    o = np.ascontiguousarray(o, np.float64)
    out = np.zeros(o.shape[1])
    lib().kvqo_lse_merge(len(m), o.shape[1], _p(m), _p(lsum), _p(o), _p(out))
    return out
