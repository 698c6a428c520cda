"""kvq_decode_attention_noalloc, the decode for callers that cannot allocate device memory.

Code that runs inside an allocator or memory-pool callback, or in a plugin whose host owns
all device memory, cannot call cudaMalloc to make the decode workspace.  This entry point
keeps its scratch in a fixed array the library holds on the device instead.  These tests
call it through the C ABI and check it against the workspace-taking
kvq_decode_attention on the same cache, twice in a row (the scratch is shared by all calls
and keeps the previous call's contents).  The file is named so that pytest runs it last.
"""
import ctypes as C
import math

import numpy as np
import pytest
import torch

from harness import ATOL, RTOL, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _filled_cache(K, scheme, seed):
    gen = torch.Generator().manual_seed(seed)
    if scheme == "kivi":
        cfg = K.make_config("kivi", 1, 3, 32, 8, 128, 1500, bits=2, group_k=32, group_v=32, residual=128)
        dt = torch.bfloat16
    else:
        cfg = K.make_config("int8", 1, 2, 8, 2, 64, 900, in_dtype="f32")
        dt = torch.float32
    cache = K.QuantizedKVCache(cfg)
    k = torch.randn(cfg.batch, 1300 if scheme == "kivi" else 850, cfg.kv_heads, cfg.head_dim, generator=gen)
    v = torch.randn(k.shape, generator=gen)
    k[..., 5] *= 10.0
    cache.append(0, k.to(dt).cuda(), v.to(dt).cuda(), n_valid=torch.tensor(
        [k.shape[1], k.shape[1] // 2, 7][:cfg.batch], dtype=torch.int32).cuda())
    torch.cuda.synchronize()
    return cfg, cache, dt, gen


@pytest.mark.parametrize("scheme", ["kivi", "int8"])
def test_noalloc_matches_workspace_decode_two_calls(scheme):
    import quantised_kv_cache_kvq_gb300 as K
    cfg, cache, dt, gen = _filled_cache(K, scheme, 31 if scheme == "kivi" else 32)
    scale = 1.0 / math.sqrt(cfg.head_dim)
    for call in range(2):
        q = torch.randn(cfg.batch, cfg.q_heads, cfg.head_dim, generator=gen).to(dt).cuda()
        ref = torch.empty(cfg.batch, cfg.q_heads, cfg.head_dim, dtype=torch.float32, device="cuda")
        got = torch.full_like(ref, float("nan"))
        K.kvq_decode_attention(cfg, cache.cache, 0, q, scale, ref, cache.workspace)
        K.kvq_decode_attention_noalloc(cfg, cache.cache, 0, q, scale, got)
        torch.cuda.synchronize()
        r = ref.cpu().numpy().astype(np.float64)
        assert_close(got.cpu().numpy().astype(np.float64), r, ATOL, RTOL, what="no-alloc call %d" % call)
        assert np.abs(r).max() > 0


def test_noalloc_rejects_configurations_beyond_its_scratch():
    # 1024 sequences x 8 kv heads need room for two partial results per (sequence, kv head),
    # far more split-context scratch than the fixed 16 MiB: rejected on the host, before any
    # device work
    import quantised_kv_cache_kvq_gb300 as K
    from quantised_kv_cache_kvq_gb300 import _native as N
    cfg = K.make_config("int8", 1, 1024, 32, 8, 128, 8192)
    assert K.kvq_workspace_bytes(cfg) > N.KVQ_NOALLOC_SCRATCH_BYTES
    fake = C.c_void_p(1 << 20)
    rc = K.load().kvq_decode_attention_noalloc(C.byref(cfg), fake, 0, fake, C.c_float(1.0), fake, None)
    assert rc == N.KVQ_ERR_WORKSPACE
