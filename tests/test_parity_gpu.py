"""Parity of the CUDA path (through the C ABI) with the oracle, element by element.

Packed caches are compared byte for byte (the whole cache image, status word included);
attention outputs within |gpu - oracle| <= 2e-3 + 1e-2 |oracle| per element.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import quantised_kv_cache_kvq_gb300 as K
from harness import Pair, assert_close, q_as_float, to_np_input

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def gen(seed):
    return torch.Generator().manual_seed(seed)


# ------------------------------------------------------------------------- KIVI
KIVI_CASES = [
    # bits, D, gqa, G, Gv, R
    (2, 128, 4, 32, 32, 128),
    (2, 128, 4, 32, 16, 32),
    (4, 128, 4, 128, 128, 128),
    (4, 64, 2, 16, 16, 0),
    (8, 128, 8, 64, 64, 40),
    (2, 256, 1, 32, 64, 16),
    (4, 256, 8, 16, 32, 48),
    (8, 64, 4, 48, 64, 20),
]


@pytest.mark.parametrize("bits,D,gqa,G,Gv,R", KIVI_CASES)
def test_kivi_bulk_then_steps(bits, D, gqa, G, Gv, R):
    H = 2
    p = Pair("kivi", layers=2, batch=3, q_heads=H * gqa, kv_heads=H, head_dim=D, max_tokens=700,
             bits=bits, group_k=G, group_v=Gv, residual=R)
    g = gen(bits * 1000 + D + gqa)
    # ragged prefill of layer 1 through the bulk path, then single-token decode steps
    k, v = p.rand_kv(3, 517, g)
    p.append(1, k, v, n_valid=[517, 300, 1])
    p.assert_same_image()
    for step in range(G + 3):
        k, v = p.rand_kv(3, 1, g)
        p.append(1, k, v)
        if step % 7 == 0 or step == G + 2:
            p.assert_same_image()
            out, ref = p.decode(1, p.rand_q(g))
            assert_close(out, ref, what="kivi step %d" % step)
    # layer 0 untouched: zero output
    out, ref = p.decode(0, p.rand_q(g))
    assert not out.any() and not ref.any()
    assert p.status() == 0


def test_kivi_small_appends_and_window_edges():
    # appends of 1..16 tokens (the single-kernel path) across window fills and flushes
    p = Pair("kivi", batch=2, q_heads=8, kv_heads=2, head_dim=128, max_tokens=400, bits=2,
             group_k=32, group_v=32, residual=64)
    g = gen(5)
    total = 0
    for m in [1, 16, 5, 16, 16, 16, 13, 1, 1, 9, 16, 16, 16, 16, 16, 3]:
        k, v = p.rand_kv(2, m, g)
        p.append(0, k, v)
        total += m
        p.assert_same_image()
        out, ref = p.decode(0, p.rand_q(g))
        assert_close(out, ref, what="after %d tokens" % total)


def test_kivi_no_autoflush_and_explicit_flush():
    p = Pair("kivi", batch=3, q_heads=4, kv_heads=1, head_dim=64, max_tokens=300, bits=4,
             group_k=16, group_v=16, residual=24)
    g = gen(6)
    for step in range(90):
        k, v = p.rand_kv(3, 1, g)
        p.append(0, k, v, n_valid=[1, step % 2, 1], flags=1)
        if step % 3 == 2:
            p.flush(0)
        if step % 10 == 9:
            p.assert_same_image()
            out, ref = p.decode(0, p.rand_q(g))
            assert_close(out, ref, what="no-autoflush step %d" % step)
    # flushing only every third step lets the R + G window overflow now and then; the
    # skipped appends are flagged identically on both sides (the status word is part of
    # the compared image)
    assert p.status() == p.img.status == 2


def test_kivi_ring_full_and_capacity_status():
    p = Pair("kivi", batch=2, q_heads=4, kv_heads=2, head_dim=64, max_tokens=120, bits=2,
             group_k=16, group_v=16, residual=16)
    g = gen(7)
    k, v = p.rand_kv(2, 32, g)
    p.append(0, k, v, flags=1)                  # window holds R + G = 32 tokens: full
    k, v = p.rand_kv(2, 1, g)
    p.append(0, k, v, flags=1)                  # overflow: skipped, RING_FULL
    p.assert_same_image()
    assert p.status() == 2
    p.flush(0)
    k, v = p.rand_kv(2, 100, g)
    p.append(0, k, v, n_valid=[88, 89])         # 32 + 89 > 120: sequence 1 skipped, CAPACITY
    p.assert_same_image()
    assert p.status() == 3
    out, ref = p.decode(0, p.rand_q(g))
    assert_close(out, ref, what="after skips")


def test_kivi_nonfinite_flag():
    p = Pair("kivi", batch=1, q_heads=4, kv_heads=1, head_dim=64, max_tokens=64, bits=2,
             group_k=16, group_v=16, residual=8)
    g = gen(8)
    k, v = p.rand_kv(1, 20, g)
    k[0, 19, 0, 5] = float("nan")               # stays in the window: flagged, stored as is
    p.append(0, k, v)
    assert p.status() == 4
    p.assert_same_image()


def test_kivi_long_context_split():
    # many packed chunks per (sequence, kv head): exercises the split context and the merge
    p = Pair("kivi", batch=1, q_heads=32, kv_heads=8, head_dim=128, max_tokens=20000, bits=4,
             group_k=128, group_v=128, residual=128)
    g = gen(9)
    k, v = p.rand_kv(1, 19000, g)
    p.append(0, k, v)
    p.assert_same_image()
    out, ref = p.decode(0, p.rand_q(g))
    assert_close(out, ref, what="long context")


@pytest.mark.parametrize("bits,D,G,Gv,batch,tokens", [
    (2, 128, 32, 32, 2, 12200),    # several chunks per item, one stage
    (2, 64, 16, 16, 8, 3000),      # several chunks per item, double-buffered stages
    (4, 128, 128, 128, 1, 60000),  # long items (several chunks), warps sharing a group
])
def test_kivi_multi_chunk_items(bits, D, G, Gv, batch, tokens):
    # enough packed chunks over all (sequence, kv head) units that the decode gives every
    # block a run of chunks, with the online softmax carried across them
    p = Pair("kivi", batch=batch, q_heads=32, kv_heads=8, head_dim=D, max_tokens=tokens + 100, bits=bits,
             group_k=G, group_v=Gv, residual=128)
    g = gen(bits * 7 + D + G)
    k, v = p.rand_kv(batch, tokens, g)
    p.append(0, k, v, n_valid=[tokens - 37 * i for i in range(batch)])
    out, ref = p.decode(0, p.rand_q(g))
    assert_close(out, ref, what="multi-chunk items")


def test_kivi_peaky_attention_with_value_outliers():
    # large logits concentrate attention on few tokens, where value-outlier tokens (x8) and
    # key outlier channels stress the precision of the score and value contractions
    p = Pair("kivi", batch=2, q_heads=8, kv_heads=2, head_dim=128, max_tokens=1200, bits=2,
             group_k=32, group_v=32, residual=128)
    g = gen(10)
    k, v = p.rand_kv(2, 1100, g, scale=3.0)
    p.append(0, k, v)
    out, ref = p.decode(0, p.rand_q(g, scale=3.0), scale=1.0)
    assert_close(out, ref, what="peaky")


# ------------------------------------------------------------------------- INT8 / FP8
def test_int8_tiny_workload():
    # 1 layer, batch 1, 4 heads, head_dim 32, 256 fp32 tokens, two key channels x10,
    # q ~ N(0,1)/sqrt(32), softmax scale 1
    from quantised_kv_cache_kvq_gb300 import workloads as W
    w = W.WORKLOADS["int8_tiny"]
    p = Pair("int8", batch=1, q_heads=4, kv_heads=4, head_dim=32, max_tokens=256, in_dtype="f32")
    k, v = W.kv_tokens(w, 0, 0, 1, 0, 256)
    p.append(0, k[:, :200], v[:, :200])
    for t in range(200, 256, 8):
        p.append(0, k[:, t:t + 8], v[:, t:t + 8])
    p.assert_same_image()
    q = W.queries(w, 0)
    out, ref = p.decode(0, q, scale=1.0)
    assert_close(out, ref, what="int8 tiny")


@pytest.mark.parametrize("D,gqa,dtype", [(128, 4, "bf16"), (64, 8, "f32"), (256, 1, "bf16"), (32, 2, "f32")])
def test_int8_and_fp8_ragged(D, gqa, dtype):
    for scheme in ("int8", "fp8", "fp8e5m2", "int4"):
        p = Pair(scheme, layers=2, batch=3, q_heads=2 * gqa, kv_heads=2, head_dim=D, max_tokens=333,
                 in_dtype=dtype)
        g = gen(D + gqa)
        k, v = p.rand_kv(3, 250, g)
        sc = None
        if scheme.startswith("fp8"):
            fmax = 448.0 if scheme == "fp8" else 57344.0
            sc = torch.stack([k.float().abs().amax(dim=(0, 1, 3)), v.float().abs().amax(dim=(0, 1, 3))], 1) / fmax
        p.append(1, k, v, n_valid=[250, 17, 0], fp8_scales=sc)
        for _ in range(5):
            k2, v2 = p.rand_kv(3, 1, g)
            p.append(1, k2, v2, fp8_scales=sc)
        p.assert_same_image()
        out, ref = p.decode(1, p.rand_q(g))
        assert_close(out, ref, what=scheme)
        k3, v3 = p.rand_kv(3, 100, g)
        p.append(1, k3, v3, n_valid=[100, 0, 0], fp8_scales=sc)  # 255 + 100 > 333
        assert p.status() == 1
        p.assert_same_image()


def test_fp8_saturation_and_subnormals():
    p = Pair("fp8", batch=1, q_heads=4, kv_heads=1, head_dim=128, max_tokens=32)
    g = gen(12)
    k, v = p.rand_kv(1, 20, g)
    k[0, 0, 0, :8] = torch.tensor([1e4, -1e4, 1e-6, -1e-6, 449.0, 447.0, 0.0, -0.0])
    sc = torch.tensor([[1.0, 0.5]])
    p.append(0, k, v, fp8_scales=sc)
    p.assert_same_image()


def test_fp8_e5m2_saturation_nonfinite_and_subnormals():
    # E5M2 saturates at +-57344 (infinities included), keeps NaN as 0x7f and reaches
    # subnormals down to 2^-16 of the scale; the codes must match the oracle byte for byte
    p = Pair("fp8e5m2", batch=1, q_heads=4, kv_heads=1, head_dim=128, max_tokens=32)
    g = gen(14)
    k, v = p.rand_kv(1, 20, g)
    k[0, 0, 0, :10] = torch.tensor([1e6, -1e6, 6e4, 57344.0, 3e-5, -2e-5, 0.0, -0.0, float("inf"), float("-inf")])
    v[0, 1, 0, :2] = torch.tensor([float("nan"), 1.5e-5])
    sc = torch.tensor([[1.0, 0.5]])
    p.append(0, k, v, fp8_scales=sc)
    p.assert_same_image()
    assert p.status() == 4      # the non-finite inputs are flagged (and stored)


def test_fp8_long_context_separate_merge():
    # enough row chunks that the per-chunk merge weights exceed the decode block's scratch, so
    # the split context is merged by the separate merge kernel
    p = Pair("fp8", batch=1, q_heads=4, kv_heads=1, head_dim=128, max_tokens=80000)
    g = gen(13)
    k, v = p.rand_kv(1, 79000, g)
    sc = torch.stack([k.float().abs().amax(dim=(0, 1, 3)), v.float().abs().amax(dim=(0, 1, 3))], 1) / 448
    p.append(0, k, v, fp8_scales=sc)
    p.assert_same_image()
    out, ref = p.decode(0, p.rand_q(g))
    assert_close(out, ref, what="fp8 long")


@pytest.mark.parametrize("max_tokens", [512, 600])
def test_int8_merge_paths_at_the_boundary(max_tokens):
    # INT8 rows come in items of 128 tokens: 512 tokens of capacity give four items per
    # (sequence, kv head), merged by the one-thread-per-output merge; 600 give five, merged
    # by the warp-per-chunk merge.  Ragged fills leave some items empty.
    p = Pair("int8", batch=3, q_heads=8, kv_heads=2, head_dim=64, max_tokens=max_tokens, in_dtype="bf16")
    g = gen(max_tokens)
    k, v = p.rand_kv(3, max_tokens - 8, g)
    p.append(0, k, v, n_valid=[max_tokens - 8, 130, 5])
    p.assert_same_image()
    out, ref = p.decode(0, p.rand_q(g))
    assert_close(out, ref, what="int8 merge boundary %d" % max_tokens)


# ------------------------------------------------------------------------- decode scheduling
# The decode grid is one wave of resident blocks that split the layer's bytes evenly, so a
# block may take the end of one unit and the start of the next, or nothing at all.  These
# cases mix empty, one-token, window-only and long sequences in one batch.
RAGGED_LENS = [0, 1, 5, 31, 32, 33, 160, 161, 700, 0, 2047, 3000, 17, 129, 64, 1000]


@pytest.mark.parametrize("scheme,bits,G,R", [("kivi", 2, 32, 128), ("kivi", 4, 16, 8), ("fp8", 8, 32, 0),
                                             ("int8", 8, 32, 0), ("fp8e5m2", 8, 32, 0), ("int4", 4, 32, 0)])
def test_decode_schedule_ragged_batch(scheme, bits, G, R):
    B = len(RAGGED_LENS)
    p = Pair(scheme, batch=B, q_heads=16, kv_heads=4, head_dim=128, max_tokens=max(RAGGED_LENS) + 8,
             bits=bits, group_k=G, group_v=32, residual=R)
    g = gen(21 + bits + G)
    k, v = p.rand_kv(B, max(RAGGED_LENS), g)
    sc = None
    if scheme.startswith("fp8"):
        sc = torch.stack([k.float().abs().amax(dim=(0, 1, 3)), v.float().abs().amax(dim=(0, 1, 3))], 1) / 448
    p.append(0, k, v, n_valid=RAGGED_LENS, fp8_scales=sc)
    p.assert_same_image()
    out, ref = p.decode(0, p.rand_q(g))
    assert_close(out, ref, what="ragged %s" % scheme)
    assert not out[0].any() and not out[9].any()       # empty sequences give 0
    # a step later (every sequence one token longer)
    k, v = p.rand_kv(B, 1, g)
    p.append(0, k, v, fp8_scales=sc)
    out, ref = p.decode(0, p.rand_q(g))
    assert_close(out, ref, what="ragged %s after a step" % scheme)
    assert p.status() == 0


def test_decode_schedule_many_units_cost_ranges():
    # 160 ragged sequences x 4 kv heads: more units than half the grid, so the decode splits
    # the layer's bytes into equal cost ranges that cross unit boundaries (the other tests
    # with few units give every unit whole blocks)
    lens = [(37 * i * i + 11 * i) % 1900 for i in range(160)]
    lens[5] = 0
    p = Pair("kivi", batch=160, q_heads=16, kv_heads=4, head_dim=128, max_tokens=1920, bits=2, group_k=32,
             group_v=32, residual=64)
    g = gen(26)
    for s0 in range(0, 160, 40):
        k, v = p.rand_kv(40, max(lens[s0:s0 + 40]), g)
        p.append(0, k, v, seq_begin=s0, n_valid=lens[s0:s0 + 40])
    p.assert_same_image()
    out, ref = p.decode(0, p.rand_q(g))
    assert_close(out, ref, what="many units")
    assert not out[5].any()
    k, v = p.rand_kv(160, 1, g)
    p.append(0, k, v)
    out, ref = p.decode(0, p.rand_q(g))
    assert_close(out, ref, what="many units after a step")


def test_decode_schedule_chunks_on_demand():
    # few units with long contexts: at least 4 packed chunks per block, so the blocks of a
    # unit take its chunks from a counter (the window rows first, on the last blocks); a
    # second decode checks that the merge set the counters back to zero
    # (the third sequence is short: its units get a single block, which takes the window
    # first and then every packed chunk from the counter)
    lens = [400000, 300007, 1000]
    p = Pair("kivi", batch=3, q_heads=4, kv_heads=2, head_dim=64, max_tokens=max(lens) + 64, bits=2,
             group_k=32, group_v=32, residual=100)
    g = gen(27)
    k, v = p.rand_kv(3, max(lens), g)
    p.append(0, k, v, n_valid=lens)
    del k, v
    p.assert_same_image()
    for step in range(2):
        out, ref = p.decode(0, p.rand_q(g))
        assert_close(out, ref, what="chunks on demand, step %d" % step)
        assert not p.ws[256:256 + 24].any()      # the six unit counters are back at zero
        k, v = p.rand_kv(3, 1, g)
        p.append(0, k, v)
    assert p.status() == 0


# ------------------------------------------------------------------------- paged layout
def _table(rng, batch, mp, spare):
    """A block table over a shuffled pool with `spare` pages nobody uses."""
    return rng.permutation(batch * mp + spare)[:batch * mp].reshape(batch, mp).astype(np.int32)


@pytest.mark.parametrize("bits,G,PG", [(2, 32, 4), (4, 16, 1), (8, 64, 3)])
def test_paged_kivi_append_flush_and_decode(bits, G, PG):
    # the group records live in a pool of pages found through a per-sequence block table;
    # the image (pool included) must match the oracle's byte for byte, and the decode must
    # give exactly what the same cache in the contiguous layout gives
    lens = [333, 0, 517]
    kw = dict(batch=3, q_heads=8, kv_heads=2, head_dim=128, max_tokens=600, bits=bits, group_k=G, group_v=32,
              residual=24)
    ng = (600 - 24) // G
    mp = (ng + PG - 1) // PG
    rng = np.random.default_rng(bits * 100 + G)
    p = Pair("kivi", page_groups=PG, num_pages=3 * mp + 5, block_table=_table(rng, 3, mp, 5), **kw)
    f = Pair("kivi", **kw)
    g = gen(40 + bits)
    k, v = p.rand_kv(3, max(lens), g)
    for x in (p, f):
        x.append(0, k, v, n_valid=lens)
    p.assert_same_image()
    for step in range(40):
        k, v = p.rand_kv(3, 1, g)
        for x in (p, f):
            x.append(0, k, v, flags=K.KVQ_NO_AUTOFLUSH if step % 7 == 3 else 0)
        if step % 13 == 5:
            for x in (p, f):
                x.flush(0)
    p.assert_same_image()
    q = p.rand_q(g)
    out, ref = p.decode(0, q)
    out_f, _ = f.decode(0, q)
    assert_close(out, ref, what="paged %d-bit" % bits)
    assert np.array_equal(out, out_f)
    assert p.status() == 0


def test_paged_decode_chunks_on_demand():
    # long sequences in a paged cache: the blocks take their chunks on demand and every
    # chunk's groups may straddle pages
    lens = [400000, 300007]
    kw = dict(batch=2, q_heads=4, kv_heads=2, head_dim=64, max_tokens=max(lens) + 64, bits=2, group_k=32,
              group_v=32, residual=100)
    ng = (kw["max_tokens"] - 100) // 32
    PG = 5
    mp = (ng + PG - 1) // PG
    p = Pair("kivi", page_groups=PG, num_pages=2 * mp + 3, block_table=_table(np.random.default_rng(3), 2, mp, 3),
             **kw)
    g = gen(28)
    k, v = p.rand_kv(2, max(lens), g)
    p.append(0, k, v, n_valid=lens)
    del k, v
    p.assert_same_image()
    out, ref = p.decode(0, p.rand_q(g))
    assert_close(out, ref, what="paged, chunks on demand")
    assert p.status() == 0


def test_paged_page_outside_the_pool_is_reported():
    kw = dict(batch=2, q_heads=8, kv_heads=2, head_dim=128, max_tokens=256, bits=2, group_k=32, group_v=32,
              residual=16)
    ng = (256 - 16) // 32
    mp = (ng + 1) // 2
    table = _table(np.random.default_rng(9), 2, mp, 0)
    table[1, 1] = 2 * mp + 7                  # sequence 1's second page is outside the pool
    p = Pair("kivi", page_groups=2, num_pages=2 * mp, block_table=table, **kw)
    g = gen(29)
    k, v = p.rand_kv(2, 140, g)
    p.append(0, k, v)              # groups 0..2 of each: sequence 1's group 2 needs the bad page
    assert p.img.status & O.ST_BAD_PAGE
    p.assert_same_image()          # sequence 1 unchanged on both sides, status word included
    assert p.status() & K.KVQ_STATUS_BAD_PAGE
    # a decode that reads through a bad entry reports it (its output is invalid)
    table2 = table.copy()
    table2[1, 1] = table[1, 0]
    table2[0, 0] = -3
    p.set_block_table(table2)
    p.decode(0, p.rand_q(g))
    assert K.kvq_read_status(None, p.ws) & K.KVQ_STATUS_BAD_PAGE


# ------------------------------------------------------------------------- keys before RoPE
@pytest.mark.parametrize("bits,D,gqa,G,Gv,R,base", [(2, 128, 4, 32, 32, 128, 500000.0),
                                                     (4, 64, 8, 128, 64, 32, 10000.0),
                                                     (8, 256, 1, 16, 16, 16, 10000.0),
                                                     (2, 256, 8, 32, 64, 64, 10000.0)])
def test_rope_keys_cached_before_the_embedding(bits, D, gqa, G, Gv, R, base):
    # the cache holds keys before the rotary embedding; the decode turns every dequantised
    # key (packed groups and bf16 window) by its position
    lens = [0, 5, R + 3, 777, 2 * G + R, 3000]
    p = Pair("kivi", batch=6, q_heads=2 * gqa, kv_heads=2, head_dim=D, max_tokens=3100, bits=bits, group_k=G,
             group_v=Gv, residual=R, rope_base=base)
    g = gen(50 + bits)
    k, v = p.rand_kv(6, max(lens), g)
    p.append(0, k, v, n_valid=lens)
    p.assert_same_image()
    for step in range(3):
        out, ref = p.decode(0, p.rand_q(g))
        assert_close(out, ref, what="rope %d-bit, step %d" % (bits, step))
        assert not out[0].any() or step > 0
        k, v = p.rand_kv(6, 1, g)
        p.append(0, k, v)
    assert p.status() == 0


def test_rope_long_context_large_angles_and_pages():
    # positions past 100000: the fastest pair turns by more than 10^5 radians (the long
    # argument reduction of sin and cos); the records in a paged pool
    lens = [120000, 70001]
    kw = dict(batch=2, q_heads=4, kv_heads=1, head_dim=64, max_tokens=120064, bits=2, group_k=32, group_v=32,
              residual=64, rope_base=10000.0)
    ng = (120064 - 64) // 32
    mp = (ng + 7) // 8
    table = np.random.default_rng(13).permutation(2 * mp + 1)[:2 * mp].reshape(2, mp).astype(np.int32)
    p = Pair("kivi", page_groups=8, num_pages=2 * mp + 1, block_table=table, **kw)
    g = gen(55)
    k, v = p.rand_kv(2, max(lens), g)
    p.append(0, k, v, n_valid=lens)
    del k, v
    p.assert_same_image()
    out, ref = p.decode(0, p.rand_q(g))
    assert_close(out, ref, what="rope, long context, paged")
    assert p.status() == 0


def test_decode_schedule_total_smaller_than_the_grid():
    # a few tokens in all: most blocks of the wave get no chunk, some units get one block
    p = Pair("kivi", batch=3, q_heads=8, kv_heads=2, head_dim=64, max_tokens=64, bits=2, group_k=16,
             group_v=16, residual=4)
    g = gen(23)
    k, v = p.rand_kv(3, 30, g)
    p.append(0, k, v, n_valid=[30, 0, 3])
    out, ref = p.decode(0, p.rand_q(g))
    assert_close(out, ref, what="tiny total")
    assert not out[1].any()


def test_decode_all_sequences_empty():
    p = Pair("kivi", batch=2, q_heads=8, kv_heads=2, head_dim=128, max_tokens=256, bits=2)
    out, ref = p.decode(0, p.rand_q(gen(24)))
    assert not out.any() and not ref.any()
    assert p.status() == 0


# ------------------------------------------------------------------------- bounded waits
def test_bounded_wait_gives_up_and_reports_timeout():
    # the workspace self-test word makes every decode block wait once on a barrier that
    # nothing completes: the wait must give up (about a second), report
    # KVQ_STATUS_TIMEOUT, leave empty partials (outputs 0) and keep the GPU usable
    import quantised_kv_cache_kvq_gb300 as K
    from quantised_kv_cache_kvq_gb300 import _native as N
    p = Pair("kivi", batch=2, q_heads=8, kv_heads=2, head_dim=128, max_tokens=3000, bits=2, group_k=32,
             group_v=32, residual=128)
    g = gen(25)
    k, v = p.rand_kv(2, 2900, g)
    p.append(0, k, v)
    q = p.rand_q(g)
    p.ws.zero_()
    p.ws[8:16].copy_(torch.tensor([N.KVQ_SELFTEST_WAIT_MAGIC], dtype=torch.int64).view(torch.uint8))
    out = torch.full((2, 8, 128), float("nan"), device="cuda")
    K.kvq_decode_attention(p.lib_cfg, p.gpu, 0, q.cuda(), 1.0 / math.sqrt(128), out, p.ws)
    torch.cuda.synchronize()
    assert K.kvq_read_status(None, p.ws) == N.KVQ_STATUS_TIMEOUT
    assert not out.cpu().numpy().any()
    # the context stays usable: with the header cleared the same decode is correct
    p.ws[:16].zero_()
    got, ref = p.decode(0, q)
    assert_close(got, ref, what="after the self-test")
    assert p.status() == 0


@pytest.mark.parametrize("scheme,bits,G,R", [("kivi", 2, 32, 128), ("kivi", 4, 128, 128), ("fp8", 8, 32, 0),
                                             ("int8", 8, 32, 0)])
def test_mapped_host_inputs_and_outputs(scheme, bits, G, R):
    # the new tokens and the queries passed as page-locked host memory, the outputs written
    # into page-locked host memory: the kernels move them across the host link themselves,
    # and the cache and the outputs are those of the oracle
    p = Pair(scheme, batch=4, q_heads=16, kv_heads=4, head_dim=128, max_tokens=3000, bits=bits, group_k=G,
             group_v=min(G, 128), residual=R)
    g = gen(31 + bits)
    k, v = p.rand_kv(4, 2000, g)
    sc = None
    if scheme == "fp8":
        sc = torch.stack([k.float().abs().amax(dim=(0, 1, 3)), v.float().abs().amax(dim=(0, 1, 3))], 1) / 448
    p.append(0, k, v, n_valid=[2000, 1500, 733, 64], fp8_scales=sc)
    sc_gpu = None if sc is None else sc.float().contiguous().cuda()
    for step in range(G + 2):
        k1, v1 = p.rand_kv(4, 1, g)
        hk, hv = k1.contiguous().pin_memory(), v1.contiguous().pin_memory()
        K.kvq_quantize_append(p.lib_cfg, p.gpu, 0, 0, 4, hk, hv, 1, None, sc_gpu, 0)
        p.img.append(0, 0, to_np_input(k1), to_np_input(v1), None,
                     None if sc is None else sc.float().numpy(), 0)
        torch.cuda.synchronize()
        if step % 11 == 0 or step == G + 1:
            p.assert_same_image()
            q = p.rand_q(g)
            hq = q.contiguous().pin_memory()
            hout = torch.full((4, 16, 128), float("nan"), dtype=torch.float32).pin_memory()
            p.ws[:4].zero_()
            K.kvq_decode_attention(p.lib_cfg, p.gpu, 0, hq, 1.0 / math.sqrt(128), hout, p.ws)
            torch.cuda.synchronize()
            ref = p.img.decode(0, q_as_float(q), 1.0 / math.sqrt(128))
            assert_close(hout.numpy().astype(np.float64), ref, what="%s mapped step %d" % (scheme, step))
            dev_out, _ = p.decode(0, q)
            np.testing.assert_allclose(hout.numpy(), dev_out, rtol=1e-5, atol=1e-6)
    assert p.status() == 0


# ------------------------------------------------------------------------- dense-and-sparse
# "KVQuant ...", "Summary": a small fraction of outlier values is moved, per vector, into a
# separate sparse representation; the dense part is fitted to the rest.
@pytest.mark.parametrize("bits,D,gqa,G,Gv,R,nout", [(2, 128, 4, 32, 32, 128, 1),
                                                    (4, 128, 4, 128, 128, 128, 4),
                                                    (8, 64, 8, 16, 16, 16, 2),
                                                    (2, 256, 2, 64, 32, 40, 3),
                                                    (4, 64, 1, 48, 64, 20, 1),
                                                    (4, 256, 8, 64, 64, 32, 2)])
def test_sparse_outliers_bulk_steps_and_decode(bits, D, gqa, G, Gv, R, nout):
    lens = [0, 7, R + G - 1, 700, 1203]
    p = Pair("kivi", batch=5, q_heads=2 * gqa, kv_heads=2, head_dim=D, max_tokens=1400, bits=bits, group_k=G,
             group_v=Gv, residual=R, outliers=nout)
    g = gen(60 + bits + nout)
    k, v = p.rand_kv(5, max(lens), g)
    p.append(0, k, v, n_valid=lens)
    p.assert_same_image()
    for step in range(G + 2):
        k, v = p.rand_kv(5, 1, g)
        p.append(0, k, v)
        if step % 11 == 0 or step == G + 1:
            p.assert_same_image()
            out, ref = p.decode(0, p.rand_q(g))
            assert_close(out, ref, what="sparse %d-bit, %d outliers, step %d" % (bits, nout, step))
    assert p.status() == 0


def test_sparse_outliers_rescales_across_chunks():
    # more units than half the grid, so every block runs through many chunks of several
    # units; values double every 1024 tokens and keys grow late, so the value-scale
    # exponent and the running maximum both move between a block's chunks and the
    # outliers' corrections must follow the rescales.  (Much larger values make the output
    # a small difference of large terms, finer than the tolerance allows the scores to be
    # rounded.)
    n, B = 5000, 40
    p = Pair("kivi", batch=B, q_heads=16, kv_heads=8, head_dim=64, max_tokens=n, bits=2, group_k=32,
             group_v=32, residual=64, outliers=2)
    g = gen(71)
    k, v = p.rand_kv(B, n, g)
    grow = (2.0 ** (torch.arange(n) // 1024).float())[None, :, None, None]
    v = (v.float() * grow).to(torch.bfloat16)
    k = k.float()
    k[:, 3500:] *= 1.5
    k = k.to(torch.bfloat16)
    p.append(0, k, v, n_valid=[n - 37 * i for i in range(B)])
    del k, v
    p.assert_same_image()
    out, ref = p.decode(0, p.rand_q(g))
    assert_close(out, ref, what="sparse, rescales across chunks")
    assert p.status() == 0


def test_sparse_outliers_paged_with_flushes():
    kw = dict(batch=3, q_heads=8, kv_heads=2, head_dim=128, max_tokens=600, bits=4, group_k=32, group_v=64,
              residual=24, outliers=2)
    ng = (600 - 24) // 32
    mp = (ng + 2) // 3
    rng = np.random.default_rng(77)
    p = Pair("kivi", page_groups=3, num_pages=3 * mp + 4, block_table=_table(rng, 3, mp, 4), **kw)
    f = Pair("kivi", **kw)
    g = gen(78)
    lens = [333, 1, 517]
    k, v = p.rand_kv(3, max(lens), g)
    for x in (p, f):
        x.append(0, k, v, n_valid=lens)
    for step in range(40):
        k, v = p.rand_kv(3, 1, g)
        for x in (p, f):
            x.append(0, k, v, flags=K.KVQ_NO_AUTOFLUSH if step % 5 == 2 else 0)
        if step % 9 == 4:
            for x in (p, f):
                x.flush(0)
    p.assert_same_image()
    f.assert_same_image()
    q = p.rand_q(g)
    out, ref = p.decode(0, q)
    out_f, _ = f.decode(0, q)
    assert_close(out, ref, what="sparse, paged")
    assert np.array_equal(out, out_f)
    assert p.status() == 0


@pytest.mark.parametrize("bits,nout", [(2, 1), (4, 3)])
def test_sparse_outliers_with_keys_before_rope(bits, nout):
    # KVQuant's pre-RoPE keys and its sparse outliers together: the outlier's bf16 value
    # replaces the dequantised element before the rotation
    lens = [5, 700, 1500]
    p = Pair("kivi", batch=3, q_heads=8, kv_heads=2, head_dim=128, max_tokens=1600, bits=bits, group_k=32,
             group_v=32, residual=32, rope_base=10000.0, outliers=nout)
    g = gen(80 + bits)
    k, v = p.rand_kv(3, max(lens), g)
    p.append(0, k, v, n_valid=lens)
    p.assert_same_image()
    out, ref = p.decode(0, p.rand_q(g))
    assert_close(out, ref, what="sparse + rope %d-bit" % bits)
    assert p.status() == 0


def test_sparse_outliers_keys_before_rope_in_pages():
    # all three together: dense-and-sparse records of keys cached before the rotary
    # embedding, in a shuffled page pool
    kw = dict(batch=2, q_heads=8, kv_heads=2, head_dim=64, max_tokens=900, bits=2, group_k=32, group_v=32,
              residual=40, rope_base=10000.0, outliers=2)
    ng = (900 - 40) // 32
    mp = (ng + 3) // 4
    p = Pair("kivi", page_groups=4, num_pages=2 * mp + 2, block_table=_table(np.random.default_rng(88), 2, mp, 2),
             **kw)
    g = gen(89)
    k, v = p.rand_kv(2, 850, g)
    p.append(0, k, v, n_valid=[850, 333])
    for step in range(3):
        k, v = p.rand_kv(2, 1, g)
        p.append(0, k, v)
    p.assert_same_image()
    out, ref = p.decode(0, p.rand_q(g))
    assert_close(out, ref, what="sparse + rope, paged")
    assert p.status() == 0
