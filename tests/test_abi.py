"""The C ABI without a GPU: the library loads, exports every entry point include/kvq.h
declares, sizes caches as the pages' formula and the layout specification say, and
rejects bad arguments on the host before any device work."""
import ctypes as C
import os
import re
import subprocess

import pytest

import oracle as O
import quantised_kv_cache_kvq_gb300 as K
from quantised_kv_cache_kvq_gb300 import _native as N

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def declared():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol():
    names = declared()
    assert set(names) == set(N.EXPORTS)
    lib = K.load()
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", K.library_path()], capture_output=True, text=True).stdout
    for n in names:
        assert re.search(r"\bT %s$" % n, out, flags=re.M), n


def _cfg(**kw):
    base = dict(scheme=0, layers=1, batch=2, q_heads=8, kv_heads=2, head_dim=128, bits=2, group_k=32,
                group_v=32, residual=128, max_tokens=4096, in_dtype=0)
    base.update(kw)
    return K.KvqConfig(**base)


def test_formula_mode_reproduces_the_pages_numbers():
    # "Quantizing the KV cache": 128 KiB per token for Llama 3 8B in 16-bit, 16 GiB at 128k
    # tokens, halved by FP8 and quartered by 4 bits; the glossary's LLaMA-7B 524 KB per token
    llama3 = _cfg(layers=32, batch=1, kv_heads=8, head_dim=128, bits=16)
    assert K.kvq_cache_bytes(llama3, 1, K.KVQ_BYTES_FORMULA) == 131072
    assert K.kvq_cache_bytes(llama3, 131072, K.KVQ_BYTES_FORMULA) == 16 * 2 ** 30
    llama3.bits = 8
    assert K.kvq_cache_bytes(llama3, 131072, K.KVQ_BYTES_FORMULA) == 8 * 2 ** 30
    llama3.bits = 4
    assert K.kvq_cache_bytes(llama3, 131072, K.KVQ_BYTES_FORMULA) == 4 * 2 ** 30
    llama3.bits, llama3.batch = 16, 8
    assert K.kvq_cache_bytes(llama3, 32768, K.KVQ_BYTES_FORMULA) == 32 * 2 ** 30
    llama7 = _cfg(layers=32, batch=1, q_heads=32, kv_heads=32, head_dim=128, bits=16)
    assert K.kvq_cache_bytes(llama7, 1, K.KVQ_BYTES_FORMULA) == 524288


@pytest.mark.parametrize("kw", [
    dict(),
    dict(bits=4, group_k=128, group_v=128, residual=128, max_tokens=131072, batch=1),
    dict(bits=8, group_k=48, group_v=64, residual=20, head_dim=64, max_tokens=777),
    dict(scheme=1, head_dim=32, q_heads=4, kv_heads=4, max_tokens=256, in_dtype=1),
    dict(scheme=2, layers=32, batch=64, q_heads=32, kv_heads=8, max_tokens=8192),
    dict(scheme=3, layers=2, batch=3, q_heads=32, kv_heads=8, max_tokens=1000),
    dict(scheme=4, head_dim=64, q_heads=8, kv_heads=2, max_tokens=333, in_dtype=1),
    dict(residual=0, max_tokens=10),
    dict(page_groups=4, num_pages=10),                                       # paged KIVI layouts
    dict(bits=4, group_k=128, group_v=128, max_tokens=20000, page_groups=1, num_pages=300, layers=3),
    dict(residual=0, max_tokens=10, page_groups=3, num_pages=1),
    dict(rope_base=500000.0),                                # pre-RoPE keys change no byte of the layout
    dict(outliers=1),                                        # dense-and-sparse side lists
    dict(outliers=4, bits=4, group_k=128, group_v=128, max_tokens=3000, batch=1),
    dict(outliers=2, bits=8, group_k=48, group_v=16, residual=20, head_dim=64, max_tokens=777,
         page_groups=3, num_pages=7),
])
def test_layout_size_matches_the_specification(kw):
    c = _cfg(**kw)
    o = O.make_config(**c.as_dict())
    assert K.kvq_cache_bytes(c, c.max_tokens, K.KVQ_BYTES_LAYOUT) == O.lib().kvqo_image_bytes(C.byref(o))


BAD = [
    (dict(scheme=5), N.KVQ_ERR_ARG),
    (dict(q_heads=6, kv_heads=4), N.KVQ_ERR_ARG),
    (dict(q_heads=48, kv_heads=2), N.KVQ_ERR_UNSUPPORTED),
    (dict(head_dim=96), N.KVQ_ERR_UNSUPPORTED),
    (dict(head_dim=32), N.KVQ_ERR_UNSUPPORTED),            # KIVI needs head_dim >= 64
    (dict(bits=3), N.KVQ_ERR_ARG),
    (dict(group_k=24), N.KVQ_ERR_ARG),
    (dict(group_v=48), N.KVQ_ERR_ARG),                    # must divide head_dim
    (dict(residual=-1), N.KVQ_ERR_ARG),
    (dict(in_dtype=1), N.KVQ_ERR_ARG),                    # KIVI window keeps bf16 inputs
    (dict(max_tokens=0), N.KVQ_ERR_ARG),
    (dict(batch=0), N.KVQ_ERR_ARG),
    (dict(page_groups=-1), N.KVQ_ERR_ARG),
    (dict(page_groups=2, num_pages=0), N.KVQ_ERR_ARG),        # a paged cache needs a pool
    (dict(scheme=1, head_dim=32, q_heads=4, kv_heads=4, in_dtype=1, page_groups=2, num_pages=4),
     N.KVQ_ERR_UNSUPPORTED),                                   # pages hold KIVI group records
    (dict(rope_base=-1.0), N.KVQ_ERR_ARG),
    (dict(rope_base=float("nan")), N.KVQ_ERR_ARG),
    (dict(rope_base=float("inf")), N.KVQ_ERR_ARG),
    (dict(scheme=2, head_dim=128, rope_base=10000.0), N.KVQ_ERR_UNSUPPORTED),   # pre-RoPE keys: KIVI
    (dict(outliers=5), N.KVQ_ERR_ARG),                                          # at most 4 per vector
    (dict(outliers=-1), N.KVQ_ERR_ARG),
    (dict(scheme=2, head_dim=128, outliers=1), N.KVQ_ERR_UNSUPPORTED),          # dense-and-sparse: KIVI
]


@pytest.mark.parametrize("kw,code", BAD)
def test_bad_configurations_are_rejected(kw, code):
    lib = K.load()
    c = _cfg(**kw)
    out = C.c_uint64(0)
    assert lib.kvq_cache_bytes(C.byref(c), c.max_tokens, K.KVQ_BYTES_LAYOUT, C.byref(out)) == code
    assert lib.kvq_workspace_bytes(C.byref(c), C.byref(out)) == code


def test_host_side_argument_checks_before_any_launch():
    lib = K.load()
    c = _cfg()
    fake = 1 << 20                      # never dereferenced: every call below fails on the host
    q = C.c_void_p(fake)
    assert lib.kvq_quantize_append(None, q, 0, 0, 1, q, q, 1, None, None, 0, None) == N.KVQ_ERR_ARG
    assert lib.kvq_quantize_append(C.byref(c), q, 1, 0, 1, q, q, 1, None, None, 0, None) == N.KVQ_ERR_ARG
    assert lib.kvq_quantize_append(C.byref(c), q, 0, 1, 2, q, q, 1, None, None, 0, None) == N.KVQ_ERR_ARG
    assert lib.kvq_quantize_append(C.byref(c), q, 0, 0, 1, q, q, 5000, None, None, 0, None) == N.KVQ_ERR_CAPACITY
    assert lib.kvq_quantize_append(C.byref(c), C.c_void_p(fake + 16), 0, 0, 1, q, q, 1, None, None, 0,
                                   None) == N.KVQ_ERR_ALIGN
    assert lib.kvq_quantize_append(C.byref(c), q, 0, 0, 1, C.c_void_p(fake + 2), q, 1, None, None, 0,
                                   None) == N.KVQ_ERR_ALIGN
    assert lib.kvq_quantize_append(C.byref(c), q, 0, 0, 1, q, q, 1, None, None, 4, None) == N.KVQ_ERR_ARG
    f8 = _cfg(scheme=2, head_dim=128)
    assert lib.kvq_quantize_append(C.byref(f8), q, 0, 0, 1, q, q, 1, None, None, 0, None) == N.KVQ_ERR_ARG
    assert lib.kvq_decode_attention(C.byref(c), q, 0, q, C.c_float(1.0), q, q, 16, None) == N.KVQ_ERR_WORKSPACE
    ws = C.c_uint64(0)
    lib.kvq_workspace_bytes(C.byref(c), C.byref(ws))
    assert lib.kvq_decode_attention(C.byref(c), q, 0, q, C.c_float(1.0), q, C.c_void_p(fake + 16), ws.value,
                                    None) == N.KVQ_ERR_ALIGN
    assert lib.kvq_decode_attention(C.byref(c), q, 3, q, C.c_float(1.0), q, q, ws.value, None) == N.KVQ_ERR_ARG
    assert lib.kvq_flush_group(C.byref(c), q, -1, None) == N.KVQ_ERR_ARG
    assert lib.kvq_read_status(None, None, None, None) == N.KVQ_ERR_ARG
    # zero-size appends are accepted and do nothing
    assert lib.kvq_quantize_append(C.byref(c), q, 0, 0, 0, None, None, 1, None, None, 0, None) == N.KVQ_OK
    # a paged cache without its block table, or with a misaligned one
    pg = _cfg(page_groups=4, num_pages=64)
    lib.kvq_workspace_bytes(C.byref(pg), C.byref(ws))
    assert lib.kvq_quantize_append(C.byref(pg), q, 0, 0, 1, q, q, 1, None, None, 0, None) == N.KVQ_ERR_ARG
    assert lib.kvq_flush_group(C.byref(pg), q, 0, None) == N.KVQ_ERR_ARG
    assert lib.kvq_decode_attention(C.byref(pg), q, 0, q, C.c_float(1.0), q, q, ws.value, None) == N.KVQ_ERR_ARG
    assert lib.kvq_decode_attention_noalloc(C.byref(pg), q, 0, q, C.c_float(1.0), q, None) == N.KVQ_ERR_ARG
    pg.block_table = fake + 2
    assert lib.kvq_quantize_append(C.byref(pg), q, 0, 0, 1, q, q, 1, None, None, 0, None) == N.KVQ_ERR_ALIGN
    assert lib.kvq_flush_group(C.byref(pg), q, 0, None) == N.KVQ_ERR_ALIGN
    assert lib.kvq_decode_attention(C.byref(pg), q, 0, q, C.c_float(1.0), q, q, ws.value, None) == N.KVQ_ERR_ALIGN


def test_status_strings():
    for code in (0, -1, -2, -3, -4, -5, -6, -99):
        assert isinstance(K.status_string(code), str) and K.status_string(code)


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    # the binding has no fallback: without libkvq.so every entry point raises instead of
    # computing anything on the host
    monkeypatch.setattr(N, "_lib", None)
    monkeypatch.setattr(N._build, "LIB", str(tmp_path / "libkvq.so"))
    with pytest.raises(RuntimeError, match="not built"):
        N.load()
    cfg = K.make_config(0, 1, 1, 4, 4, 64, 64, bits=2, group_k=16, group_v=16, residual=0)
    with pytest.raises(RuntimeError, match="not built"):
        N.kvq_cache_bytes(cfg, 64)


def test_config_struct_layout_matches_the_header(tmp_path):
    # the binding's ctypes struct must lay kvq_config out as a C compiler does from
    # include/kvq.h (size and every field offset)
    fields = [n for n, _ in N.KvqConfig._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "kvq.h"\nint main(void) {\n'
                   '    printf("%zu\\n", sizeof(kvq_config));\n'
                   + "".join('    printf("%%zu\\n", offsetof(kvq_config, %s));\n' % f for f in fields)
                   + '    return 0;\n}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert out[0] == C.sizeof(N.KvqConfig)
    assert out[1:] == [getattr(N.KvqConfig, f).offset for f in fields]


def test_layout_size_matches_the_specification_on_random_configurations():
    # a seeded sweep over valid KIVI, INT8, INT4 and FP8 configurations (paged, pre-RoPE and
    # dense-and-sparse ones included): the library's allocation size is the oracle's
    import random
    rng = random.Random(2024)
    lib = O.lib()
    for _ in range(300):
        scheme = rng.choice([0, 0, 0, 1, 2, 3, 4])
        kv = rng.choice([1, 2, 8])
        kw = dict(scheme=scheme, layers=rng.randint(1, 3), batch=rng.randint(1, 9), kv_heads=kv,
                  q_heads=kv * rng.choice([1, 2, 4, 8]), max_tokens=rng.randint(1, 3000))
        if scheme == 0:
            D = rng.choice([64, 128, 256])
            G = 16 * rng.randint(1, 8)
            Gv = rng.choice([g for g in (16, 32, 64, 128, 256) if D % g == 0])
            kw.update(head_dim=D, bits=rng.choice([2, 4, 8]), group_k=G, group_v=Gv, residual=rng.randint(0, 200),
                      in_dtype=0, outliers=rng.choice([0, 0, 1, 2, 4]),
                      rope_base=rng.choice([0.0, 10000.0]))
            if rng.random() < 0.3:
                kw.update(page_groups=rng.randint(1, 6), num_pages=rng.randint(1, 50))
        else:
            kw.update(head_dim=rng.choice([32, 64, 128, 256]), bits=8, in_dtype=rng.choice([0, 1]))
        c = _cfg(**{k: v for k, v in kw.items() if k not in ("rope_base", "outliers")})
        c.rope_base = kw.get("rope_base", 0.0)
        c.outliers = kw.get("outliers", 0)
        got = K.kvq_cache_bytes(c, c.max_tokens, K.KVQ_BYTES_LAYOUT)
        assert got == lib.kvqo_image_bytes(C.byref(O.make_config(**kw))), kw
