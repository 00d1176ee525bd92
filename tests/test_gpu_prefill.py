"""GPU parity of the chunked prefill (dms_prefill) against the CPU oracle.

The prefill's attention runs on the tensor cores: bf16 Q K^T, fp32 softmax,
P V with each probability carried as two bf16 terms (about 16 bits), fp32
accumulation.  Expected error against the float64 oracle: about 2^-17
relative per probability plus fp32 rounding, well inside both the stated bar
(max-abs 1e-2, mean relative 1e-3) and the tighter one the decode tests use
(1e-4, 1e-4), which both are asserted.  Bookkeeping after a prefill must be
bit-identical to the same tokens appended one by one.
"""
import numpy as np
import pytest
import torch

import oracle.dms_oracle as O
from learned_kv_cache_eviction_b300 import dms, workload as W

pytestmark = pytest.mark.gpu

TOL_STATED = (1e-2, 1e-3)
TOL_TIGHT = (1e-4, 1e-4)


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    dms.load_library()


def _close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.abs(got - ref)
    mx, rel = float(d.max()), float(d.sum() / np.abs(ref).sum())
    assert mx <= TOL_STATED[0] and rel <= TOL_STATED[1], f"{what}: max-abs {mx:.3e} mean-rel {rel:.3e}"
    assert mx <= TOL_TIGHT[0] and rel <= TOL_TIGHT[1], f"{what}: max-abs {mx:.3e} mean-rel {rel:.3e}"
    return mx, rel


def _wl(B, Hq, Hkv, D, w, cap, logits, seed=31):
    return W.Workload("prefill", B=B, Hq=Hq, Hkv=Hkv, D=D, w=w, cap=cap, seed=seed, logits=logits)


@pytest.mark.parametrize("case", [
    # B, Hq, Hkv, D, w, history T0, chunk C, logits
    (2, 8, 2, 128, 16, 300, 150, ("normal", 0.5, 1.0)),     # G 4: 2 cache tiles + ragged chunk tiles
    (1, 16, 2, 64, 16, 0, 200, ("normal", 1.0, 1.0)),       # G 8, empty cache, 13 query tiles
    (2, 10, 2, 128, 16, 130, 60, ("normal", 1.15, 1.0)),    # G 5: 25 positions per tile, padded rows
    (3, 3, 3, 64, 16, 257, 33, ("normal", 0.0, 1.0)),       # MHA, cache length just past two tiles
    (2, 4, 2, 128, 16, 200, 140, ("const", -10.0)),         # all keep: causal attention
    (2, 4, 2, 128, 16, 200, 140, ("const", 10.0)),          # all evict: sliding window of w
    (2, 8, 4, 64, 1, 90, 70, ("normal", 0.0, 1.0)),         # eager eviction, w = 1
    (1, 8, 1, 128, 16, 40, 5, ("normal", 0.3, 2.0)),        # chunk shorter than the window
    (2, 4, 2, 128, 16, 100, 1, ("normal", 0.5, 1.0)),       # a chunk of one token
    (1, 12, 2, 128, 16, 256, 90, ("normal", 0.8, 1.0)),     # G 6: 21 positions per tile; cache exactly two tiles
    (1, 14, 2, 64, 16, 70, 100, ("normal", 0.8, 1.0)),      # G 7: 18 positions per tile, padded rows
    (1, 4, 2, 64, 64, 120, 100, ("normal", 0.5, 1.0)),      # window 64: marks pending across the whole chunk
    (1, 4, 1, 128, 16, 0, 600, ("normal", 1.0, 1.0)),       # empty cache, 5 chunk key tiles, ragged end
])
def test_prefill_matches_oracle(case):
    B, Hq, Hkv, D, w, T0, C, logits = case
    wl = _wl(B, Hq, Hkv, D, w, T0 + C + 8, logits)
    T = T0 + C
    k, v, lg = W.kv_range(wl, 0, 0, T)
    q = W.q_range(wl, 0, T0, T)
    e = O.eviction_decisions(lg.numpy())
    cache = dms.DmsCache(B, Hkv, wl.cap, D, w)
    if T0:
        cache.append_chunk(k[:, :, :T0].contiguous().cuda(), v[:, :, :T0].contiguous().cuda(),
                           lg[:, :, :T0].contiguous().cuda())
    out = cache.prefill(q.cuda(), k[:, :, T0:].contiguous().cuda(), v[:, :, T0:].contiguous().cuda(),
                        lg[:, :, T0:].contiguous().cuda(), scale=wl.scale)
    assert cache.status() == dms.DMS_OK
    assert cache.position == T
    ref = O.prefill_attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), e, T0, w, wl.scale)
    _close(out.cpu().numpy(), ref, f"prefill {case}")
    # bookkeeping equals T single appends
    sim = O.SlotSimulator(B, Hkv, wl.cap, w)
    sim.append_chunk(e)
    assert np.array_equal(cache.lengths().cpu().numpy(), sim.len)
    assert np.array_equal(cache.slot_positions().cpu().numpy(), sim.slot_pos)
    cache.close()


def test_prefill_equals_rounds_of_append_and_decode():
    """dms_prefill of C tokens against C rounds of dms_append + dms_decode_attention
    on a second cache: the same outputs (within the tolerance) and the same
    cache state, byte for byte."""
    wl = _wl(2, 8, 2, 128, 16, 700, ("normal", 0.7, 1.0), seed=8)
    T0, C = 400, 180
    k, v, lg = W.kv_range(wl, 0, 0, T0 + C)
    q = W.q_range(wl, 0, T0, T0 + C)
    a = dms.DmsCache(wl.B, wl.Hkv, wl.cap, wl.D, wl.w)
    b = dms.DmsCache(wl.B, wl.Hkv, wl.cap, wl.D, wl.w)
    for c in (a, b):
        c.append_chunk(k[:, :, :T0].contiguous().cuda(), v[:, :, :T0].contiguous().cuda(),
                       lg[:, :, :T0].contiguous().cuda())
    out_a = a.prefill(q.cuda(), k[:, :, T0:].contiguous().cuda(), v[:, :, T0:].contiguous().cuda(),
                      lg[:, :, T0:].contiguous().cuda(), scale=wl.scale).cpu()
    rows = []
    for j in range(C):
        t = T0 + j
        b.append(k[:, :, t].contiguous().cuda(), v[:, :, t].contiguous().cuda(), lg[:, :, t].contiguous().cuda())
        rows.append(b.decode_attention(q[:, :, j].contiguous().cuda(), scale=wl.scale).cpu())
    out_b = torch.stack(rows, dim=2)
    _close(out_a.numpy(), out_b.numpy().astype(np.float64), "prefill vs decode rounds")
    assert torch.equal(a.lengths(), b.lengths())
    assert torch.equal(a.slot_positions(), b.slot_positions())
    ka, va = a.export_kv()
    kb, vb = b.export_kv()
    assert torch.equal(ka, kb) and torch.equal(va, vb)
    assert a.status() == b.status() == dms.DMS_OK


def test_prefill_argument_errors():
    c = dms.DmsCache(1, 2, 64, 64, 16)
    lib = dms.load_library()
    q = torch.zeros(1, 4, 8, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16, device="cuda")
    lg = torch.zeros(1, 2, 8, dtype=torch.float32, device="cuda")
    out = torch.empty(1, 4, 8, 64, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    h = c.handle
    assert lib.dms_prefill(h, q.data_ptr(), k.data_ptr(), k.data_ptr(), lg.data_ptr(), 0, out.data_ptr(), 0.1, 4,
                           s) == dms.DMS_ERR_INVALID_ARG
    assert lib.dms_prefill(h, q.data_ptr(), k.data_ptr(), k.data_ptr(), lg.data_ptr(), 8, out.data_ptr(), 0.1, 3,
                           s) == dms.DMS_ERR_INVALID_ARG
    assert lib.dms_prefill(h, q.data_ptr() + 2, k.data_ptr(), k.data_ptr(), lg.data_ptr(), 8, out.data_ptr(), 0.1,
                           4, s) == dms.DMS_ERR_INVALID_ARG
    assert lib.dms_prefill(None, q.data_ptr(), k.data_ptr(), k.data_ptr(), lg.data_ptr(), 8, out.data_ptr(), 0.1, 4,
                           s) == dms.DMS_ERR_BAD_HANDLE
    assert c.position == 0
    assert lib.dms_prefill(h, q.data_ptr(), k.data_ptr(), k.data_ptr(), lg.data_ptr(), 8, out.data_ptr(), 0.1, 4,
                           s) == dms.DMS_OK
    assert c.status() == dms.DMS_OK and c.position == 8
    c.close()


def test_long_context_layer_prefill_sampled():
    """One layer of the long-context stack (B4, Hq64/Hkv8, d128, 5% forced keep):
    32768 tokens prefilled in chunks of 512; the last chunk's outputs are checked
    on 6 positions of every row against the oracle's decode at those positions,
    and the bookkeeping of all rows against the slot simulator."""
    wl = W.WORKLOADS["long-context"]
    layer, C = 2, wl.chunk
    T = wl.prefill
    k, v, lg = W.kv_range(wl, layer, 0, T)
    e = O.eviction_decisions(lg.numpy())
    cache = dms.DmsCache(wl.B, wl.Hkv, wl.cap, wl.D, wl.w)
    last = None
    for t0 in range(0, T, C):
        q = W.q_range(wl, layer, t0, t0 + C)
        out = cache.prefill(q.cuda(), k[:, :, t0:t0 + C].contiguous().cuda(), v[:, :, t0:t0 + C].contiguous().cuda(),
                            lg[:, :, t0:t0 + C].contiguous().cuda(), scale=wl.scale)
        last = (t0, q, out)
    assert cache.status() == dms.DMS_OK
    sim = O.SlotSimulator(wl.B, wl.Hkv, wl.cap, wl.w)
    sim.append_chunk(e)
    assert np.array_equal(cache.lengths().cpu().numpy(), sim.len)
    t0, q, out = last
    out = out.cpu().numpy()
    k_np, v_np = k.float().numpy(), v.float().numpy()
    for c in (0, 1, 15, 16, 300, C - 1):
        ref = O.decode_attention(q[:, :, c].float().numpy(), k_np, v_np, e, t0 + c, wl.w, wl.scale)
        _close(out[:, :, c], ref, f"long-context layer {layer} position {t0 + c}")
    cache.close()
