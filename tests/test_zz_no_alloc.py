"""dms_decode_attention_noalloc: decode attention for callers that cannot
allocate device memory when they decode (their memory is reserved up front by
their own pool, or they only receive pointers to buffers owned elsewhere).

The test builds a cache through the normal API, lays its K/V pools out the way
the no-allocation call expects (caller-owned buffers), and checks that two
calls in a row -- at two consecutive decode steps -- give the same outputs as
dms_decode_attention within the tolerance of the other GPU tests.  It lives in
a file of its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

from learned_kv_cache_eviction_b300 import dms, workload as W

pytestmark = pytest.mark.gpu

TOL_MAX_ABS = 1e-4
TOL_MEAN_REL = 1e-4


def _library_k_layout(k_logical: torch.Tensor) -> torch.Tensor:
    """K rows in the layout the kernels read: 16-byte chunk c of slot s is
    stored at chunk c ^ (s & 7)."""
    B, H, cap, D = k_logical.shape
    ch = k_logical.view(B, H, cap, D // 8, 8)
    s = torch.arange(cap, device=k_logical.device).view(cap, 1)
    c = torch.arange(D // 8, device=k_logical.device).view(1, D // 8)
    src = (c ^ (s & 7)).view(1, 1, cap, D // 8, 1).expand(B, H, cap, D // 8, 8)
    return torch.gather(ch, 3, src).reshape(B, H, cap, D).contiguous()


def _close(got: torch.Tensor, ref: torch.Tensor):
    d = (got.double() - ref.double()).abs()
    return float(d.max()), float(d.sum() / ref.double().abs().sum())


@pytest.mark.parametrize("B,Hq,Hkv,D,cap,T", [(4, 32, 8, 128, 700, 600), (2, 4, 2, 64, 300, 280),
                                            (2, 16, 2, 128, 400, 350)])  # G 8: one eight-head group here
def test_noalloc_matches_decode_attention_twice(B, Hq, Hkv, D, cap, T):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    lib = dms.load_library()
    wl = W.Workload("noalloc", B=B, Hq=Hq, Hkv=Hkv, D=D, w=16, cap=cap, seed=21, logits=("normal", 0.8, 1.0))
    k, v, lg = W.kv_range(wl, 0, 0, T + 2)
    q = W.q_range(wl, 0, T, T + 2)
    cache = dms.DmsCache(B, Hkv, cap, D, wl.w)
    cache.append_chunk(k[:, :, :T].contiguous().cuda(), v[:, :, :T].contiguous().cuda(),
                       lg[:, :, :T].contiguous().cuda())
    stream = torch.cuda.current_stream().cuda_stream
    for step in range(2):  # two calls in a row, at two consecutive decode steps
        t = T + step
        cache.append(k[:, :, t].contiguous().cuda(), v[:, :, t].contiguous().cuda(), lg[:, :, t].contiguous().cuda())
        q_t = q[:, :, step].contiguous().cuda()
        ref = cache.decode_attention(q_t, scale=wl.scale)
        # caller-owned copies of the cache's state
        k_log, v_log = cache.export_kv()
        k_pool = _library_k_layout(k_log)
        v_pool = v_log.contiguous()
        lens = cache.lengths()
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        rc = lib.dms_decode_attention_noalloc(k_pool.data_ptr(), v_pool.data_ptr(), lens.data_ptr(), B, Hkv, cap, D,
                                              q_t.data_ptr(), out.data_ptr(), ctypes.c_float(wl.scale), Hq, stream)
        assert rc == dms.DMS_OK, lib.dms_error_string(rc)
        torch.cuda.synchronize()
        assert bool(torch.isfinite(out).all())
        mx, rel = _close(out, ref)
        assert mx <= TOL_MAX_ABS and rel <= TOL_MEAN_REL, (step, mx, rel)
    assert cache.status() == dms.DMS_OK
    cache.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    lib = dms.load_library()
    buf = torch.zeros(1024, dtype=torch.float32, device="cuda")
    p = buf.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    # more heads than the fixed scratch allows
    assert lib.dms_decode_attention_noalloc(p, p, p, 4096, 8, 16, 128, p, p, 0.1, 32, s) == dms.DMS_ERR_SCRATCH_LIMIT
    # within the head limit, but G = 8 partials at head_dim 128 overflow the scratch
    assert lib.dms_decode_attention_noalloc(p, p, p, 256, 8, 4096, 128, p, p, 0.1, 64, s) == dms.DMS_ERR_SCRATCH_LIMIT
    # plain argument errors
    assert lib.dms_decode_attention_noalloc(p, p, p, 1, 8, 16, 96, p, p, 0.1, 32, s) == dms.DMS_ERR_INVALID_ARG
    assert lib.dms_decode_attention_noalloc(p, p, p, 1, 8, 16, 128, p, p, 0.1, 12, s) == dms.DMS_ERR_INVALID_ARG
    host = np.zeros(64, dtype=np.float32)
    assert lib.dms_decode_attention_noalloc(host.ctypes.data, p, p, 1, 8, 16, 128, p, p, 0.1, 32, s) == \
        dms.DMS_ERR_INVALID_ARG


def test_noalloc_full_heads_and_clamped_lengths():
    """Heads filled exactly to capacity (len == capacity) decode like
    dms_decode_attention.  Lengths outside [0, capacity] come from the caller
    and are clamped: a length above the capacity reads the full pool, a
    negative one reads nothing and leaves that head's output rows unwritten."""
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    lib = dms.load_library()
    B, Hq, Hkv, D, cap = 2, 8, 2, 128, 300
    wl = W.Workload("noalloc-full", B=B, Hq=Hq, Hkv=Hkv, D=D, w=16, cap=cap, seed=23, logits=("const", -10.0))
    k, v, lg = W.kv_range(wl, 0, 0, cap)
    q = W.q_range(wl, 0, cap - 1, cap)[:, :, 0].contiguous().cuda()
    cache = dms.DmsCache(B, Hkv, cap, D, wl.w)
    cache.append_chunk(k.contiguous().cuda(), v.contiguous().cuda(), lg.contiguous().cuda())
    lens = cache.lengths()
    assert bool((lens == cap).all())
    ref = cache.decode_attention(q, scale=wl.scale)
    k_log, v_log = cache.export_kv()
    k_pool, v_pool = _library_k_layout(k_log), v_log.contiguous()
    stream = torch.cuda.current_stream().cuda_stream
    G = Hq // Hkv
    for bad in (False, True):
        ln = lens.clone()
        if bad:
            ln[0, 0] = cap + 5    # clamped to cap: same as the full head
            ln[1, 1] = -3         # clamped to 0: no keys, rows left as they were
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        rc = lib.dms_decode_attention_noalloc(k_pool.data_ptr(), v_pool.data_ptr(), ln.data_ptr(), B, Hkv, cap, D,
                                              q.data_ptr(), out.data_ptr(), ctypes.c_float(wl.scale), Hq, stream)
        assert rc == dms.DMS_OK, lib.dms_error_string(rc)
        torch.cuda.synchronize()
        keep = torch.ones((B, Hq), dtype=torch.bool, device="cuda")
        if bad:
            keep[1, G:2 * G] = False
            assert bool(torch.isnan(out[1, G:2 * G]).all())
        mx, rel = _close(out[keep], ref[keep])
        assert mx <= TOL_MAX_ABS and rel <= TOL_MEAN_REL, (bad, mx, rel)
    cache.close()
