"""Host-side logic of bench.py (no GPU): the algorithmic bytes a decode launch reads, and
the lookup of the profiled DRAM traffic that is tied to the kernels' source digest."""
import os
import shutil

import pytest

import bench
from quantised_kv_cache_kvq_gb300 import workloads as W


def test_decode_bytes_llama3_8b_2bit_per_token_figures():
    # 2-bit KIVI, D = 128, G = Gv = 32: a packed token costs 32 B of key codes, 32 B of
    # value codes, 16 B of key scale/zero (4 D bytes per 32 tokens) and 16 B of value
    # scale/zero (4 B per token and value group, 4 groups) = 96 B; a window token 512 B
    # (bf16 key and value rows); each (sequence, kv head) also reads 4 query heads in bf16.
    w = W.WORKLOADS["kivi2_llama3_8b"]
    n = 4096
    qn = 32 * ((n - 128) // 32)          # 3968 packed, 128 in the window
    per_unit = qn * 96 + (n - qn) * 512 + 4 * 128 * 2
    assert bench.decode_bytes(w, [n] * 8) == 8 * 8 * per_unit


def test_decode_bytes_4bit_and_fp8_per_token_figures():
    # 4-bit, G = Gv = 128: 64 + 64 B of codes, 512 B of key params per 128 tokens (4 B per
    # token) and 4 B of value params per token = 136 B; FP8: 2 * 128 B per token
    w4 = W.WORKLOADS["kivi4_128k"]
    n = 131072
    qn = 128 * ((n - 128) // 128)
    assert bench.decode_bytes(w4, [n]) == 8 * (qn * 136 + (n - qn) * 512 + 4 * 128 * 2)
    w3 = W.WORKLOADS["fp8_32layer"]
    assert bench.decode_bytes(w3, [8192, 100]) == 8 * ((8192 + 100) * 256 + 2 * 4 * 128 * 2)


def test_decode_bytes_sparse_side_lists():
    # one outlier per vector at G = Gv = 128: a 4-byte key entry per channel and a 4-byte
    # value entry per token, 8 bytes a token on top of the dense 136
    w = W.WORKLOADS["kivi4_128k_sparse"]
    n = 131072
    qn = 128 * ((n - 128) // 128)
    assert bench.decode_bytes(w, [n]) == 8 * (qn * 144 + (n - qn) * 512 + 4 * 128 * 2)
    # the oracle's record agrees: K side 4 K D, V side 4 K (D / Gv) G
    import ctypes as C
    import oracle as O
    kw = dict(scheme=0, layers=1, batch=1, q_heads=32, kv_heads=8, head_dim=128, bits=4, group_k=128,
              group_v=128, residual=128, max_tokens=128 + 128 * 3)
    dense = O.lib().kvqo_image_bytes(C.byref(O.make_config(**kw)))
    sparse = O.lib().kvqo_image_bytes(C.byref(O.make_config(outliers=1, **kw)))
    assert sparse - dense == 8 * 3 * (4 * 128 + 4 * 128)


def test_decode_bytes_ragged_is_a_sum_and_short_sequences_are_window_only():
    w = W.WORKLOADS["serve_mix"]
    lens = [1024, 5000, 32768, 159, 160, 0]
    assert bench.decode_bytes(w, lens) == sum(bench.decode_bytes(w, [n]) for n in lens)
    q = 8 * 4 * 128 * 2
    # below R + G = 160 tokens nothing is packed yet
    assert bench.decode_bytes(w, [159]) == 8 * 159 * 512 + q
    assert bench.decode_bytes(w, [160]) == 8 * (32 * 96 + 128 * 512) + q
    assert bench.decode_bytes(w, [0]) == q


def _tree_copy(tmp_path):
    root = tmp_path / "tree"
    shutil.copytree(os.path.join(bench.ROOT, "quantised_kv_cache_kvq_gb300", "csrc"),
                    root / "quantised_kv_cache_kvq_gb300" / "csrc")
    (root / "profiles").mkdir()
    return root


def test_sources_digest_follows_the_scheme_sources(tmp_path, monkeypatch):
    root = _tree_copy(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    kivi, fp8 = bench.sources_sha256(0), bench.sources_sha256(2)
    assert kivi != fp8
    # an FP8-only source moves only the FP8 digest; a shared one moves both
    p = root / "quantised_kv_cache_kvq_gb300" / "csrc" / "kvq_decode_fp8.cu"
    p.write_bytes(p.read_bytes() + b"\n")
    assert bench.sources_sha256(0) == kivi and bench.sources_sha256(2) != fp8
    p = root / "quantised_kv_cache_kvq_gb300" / "csrc" / "kvq_decode.cuh"
    p.write_bytes(p.read_bytes() + b"\n")
    assert bench.sources_sha256(0) != kivi


def test_profiled_traffic_only_for_the_captured_sources(tmp_path, monkeypatch):
    root = _tree_copy(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    prof = root / "profiles" / "k_decode_kivi4_128k.md"
    assert bench.profiled_traffic("kivi4_128k", 0) is None          # no summary
    prof.write_text("# x\n\ntraffic_bytes_per_launch: 123456\nsources_sha256: %s\n" % bench.sources_sha256(0))
    assert bench.profiled_traffic("kivi4_128k", 0) == 123456
    prof.write_text("traffic_bytes_per_launch: 123456\nsources_sha256: %s\n" % ("0" * 64))
    assert bench.profiled_traffic("kivi4_128k", 0) is None          # kernels changed since
    prof.write_text("sources_sha256: %s\n" % bench.sources_sha256(0))
    assert bench.profiled_traffic("kivi4_128k", 0) is None          # no traffic figure


@pytest.mark.parametrize("wl", ["kivi2_llama3_8b", "kivi4_128k", "fp8_32layer"])
def test_committed_profiles_carry_traffic_and_digest(wl):
    with open(os.path.join(bench.ROOT, "profiles", "k_decode_%s.md" % wl)) as f:
        text = f.read()
    assert "traffic_bytes_per_launch: " in text and "sources_sha256: " in text
    assert "--clock-control none" in text
