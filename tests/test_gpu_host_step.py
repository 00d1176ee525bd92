"""GPU parity of dms_step_host: steps whose rows come from, and whose output
goes to, host memory.  Each call copies its inputs in on the cache's own copy
stream, runs the same fused step kernel as dms_step on device copies, and
copies its output out on a second copy stream, with two sets of device rows so
that the copies of one call overlap the steps of its neighbours.  The result
must be dms_step's, bit for bit, whatever the interleaving with device-row
calls, and the last step's output must match the float64 oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle.dms_oracle as O
from learned_kv_cache_eviction_b300 import dms, workload as W

pytestmark = pytest.mark.gpu

TOL_TIGHT = (1e-4, 1e-4)


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    dms.load_library()


def _host(x, pinned):
    x = x.contiguous().cpu()
    return x.pin_memory() if pinned else x.clone()


@pytest.mark.parametrize("case", [
    # B, Hq, Hkv, D, w, cap, T, logits, kv_format, pinned, device_every
    (4, 16, 4, 128, 16, 700, 420, ("normal", 0.6, 1.0), "bf16", True, 0),
    (2, 16, 2, 64, 2, 500, 300, ("normal", 0.3, 1.0), "bf16", False, 0),   # G 8, d64, pageable memory
    (3, 12, 3, 128, 16, 600, 360, ("normal", 0.6, 1.0), "bf16", True, 7),  # every 7th step with device rows
    (4, 16, 4, 128, 16, 700, 300, ("normal", 0.6, 1.0), "fp8", True, 5),
])
def test_step_host_equals_step(case):
    B, Hq, Hkv, D, w, cap, T, logits, kvf, pinned, device_every = case
    wl = W.Workload("host-step", B=B, Hq=Hq, Hkv=Hkv, D=D, w=w, cap=cap, seed=29, logits=logits)
    k_all, v_all, lg_all = W.kv_range(wl, 0, 0, T)
    q_all = W.q_range(wl, 0, 0, T)
    a = dms.DmsCache(B, Hkv, cap, D, w, kv_format=kvf)
    b = dms.DmsCache(B, Hkv, cap, D, w, kv_format=kvf)
    T0 = 40
    for c in (a, b):
        c.append_chunk(k_all[:, :, :T0].contiguous().cuda(), v_all[:, :, :T0].contiguous().cuda(),
                       lg_all[:, :, :T0].contiguous().cuda())
    n = T - T0
    kk = [k_all[:, :, t] for t in range(T0, T)]
    vv = [v_all[:, :, t] for t in range(T0, T)]
    ll = [lg_all[:, :, t] for t in range(T0, T)]
    qq = [q_all[:, :, t] for t in range(T0, T)]
    # device rows for cache a (and for b's device-row steps)
    kd, vd, ld, qd = ([x.contiguous().cuda() for x in xs] for xs in (kk, vv, ll, qq))
    out_a = torch.zeros((n, B, Hq, D), dtype=torch.float32, device="cuda")
    # host rows for cache b: every step its own input and output buffers
    kh, vh, lh, qh = ([_host(x, pinned) for x in xs] for xs in (kk, vv, ll, qq))
    out_h = [_host(torch.full((B, Hq, D), float("nan")), pinned) for _ in range(n)]
    out_bd = torch.zeros((n, B, Hq, D), dtype=torch.float32, device="cuda")
    used_dev = []
    for j in range(n):
        a.step(kd[j], vd[j], ld[j], qd[j], out_a[j], scale=wl.scale)
        if device_every and j % device_every == device_every - 1:
            b.step(kd[j], vd[j], ld[j], qd[j], out_bd[j], scale=wl.scale)
            used_dev.append(j)
        else:
            b.step_host(kh[j], vh[j], lh[j], qh[j], out_h[j], scale=wl.scale)
    b.host_join()
    torch.cuda.synchronize()
    got = torch.stack([out_bd[j].cpu() if j in used_dev else out_h[j] for j in range(n)])
    assert torch.equal(got, out_a.cpu())
    assert torch.equal(a.lengths(), b.lengths())
    assert torch.equal(a.slot_positions(), b.slot_positions())
    ka, va = a.export_kv()
    kb, vb = b.export_kv()
    assert torch.equal(ka, kb) and torch.equal(va, vb)
    assert a.position == b.position == T
    assert a.status() == b.status() == dms.DMS_OK
    if kvf == "bf16":
        # the last step against the float64 oracle
        e = O.eviction_decisions(lg_all.numpy())
        ref = O.decode_attention(q_all[:, :, T - 1].float().numpy(), k_all.float().numpy(), v_all.float().numpy(),
                                 e, T - 1, w, wl.scale)
        g = got[-1].double().numpy()
        d = np.abs(g - ref)
        mx, rel = float(d.max()), float(d.sum() / np.abs(ref).sum())
        assert mx <= TOL_TIGHT[0] and rel <= TOL_TIGHT[1], (mx, rel)
    a.close()
    b.close()


def test_step_host_refuses_device_rows():
    """Device pointers are refused before anything is enqueued; the cache does
    not advance."""
    lib = dms.load_library()
    B, Hq, Hkv, D = 2, 8, 2, 128
    c = dms.DmsCache(B, Hkv, 64, D, 16)
    k = torch.zeros((B, Hkv, D), dtype=torch.bfloat16, device="cuda")
    lg = torch.zeros((B, Hkv), dtype=torch.float32, device="cuda")
    q = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((B, Hq, D), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    rc = lib.dms_step_host(c.handle, k.data_ptr(), k.data_ptr(), lg.data_ptr(), q.data_ptr(), out.data_ptr(),
                           ctypes.c_float(0.1), Hq, st)
    assert rc == dms.DMS_ERR_INVALID_ARG
    assert c.position == 0
    assert lib.dms_step_host_join(c.handle, st) == dms.DMS_OK  # nothing to wait for
    with pytest.raises(ValueError):
        c.step_host(k, k, lg, q, out)  # the binding checks the device too
    c.close()


def test_step_host_full_size_equals_step():
    """The benchmark's end-to-end configuration (Qwen3-8B-like: B32, Hq32/Hkv8,
    d128, CR 8, context 16384): 8 host-buffer steps after a 16376-token
    history, against 8 device-row dms_step calls on a second cache with the
    same history; outputs and bookkeeping bit-exact."""
    wl = W.WORKLOADS["qwen3-8b"]
    n_dec = 8
    T0 = wl.cap - n_dec
    a = dms.DmsCache(wl.B, wl.Hkv, wl.cap, wl.D, wl.w)
    b = dms.DmsCache(wl.B, wl.Hkv, wl.cap, wl.D, wl.w)
    for t0 in range(0, T0, wl.chunk):
        t1 = min(T0, t0 + wl.chunk)
        k, v, lg = W.kv_range(wl, 0, t0, t1, device="cuda")
        a.append_chunk(k, v, lg)
        b.append_chunk(k, v, lg)
        del k, v, lg
    k, v, lg = W.kv_range(wl, 0, T0, wl.cap)
    q = W.q_range(wl, 0, T0, wl.cap)
    out_a = torch.empty((n_dec, wl.B, wl.Hq, wl.D), dtype=torch.float32, device="cuda")
    out_h = [torch.full((wl.B, wl.Hq, wl.D), float("nan")).pin_memory() for _ in range(n_dec)]
    # the pinned inputs stay referenced until the copies are done
    rows_h = [tuple(x[:, :, j].contiguous().pin_memory() for x in (k, v, lg, q)) for j in range(n_dec)]
    for j in range(n_dec):
        kj, vj, lj, qj = rows_h[j]
        a.step(kj.cuda(), vj.cuda(), lj.cuda(), qj.cuda(), out_a[j], scale=wl.scale)
        b.step_host(kj, vj, lj, qj, out_h[j], scale=wl.scale)
    b.host_join()
    torch.cuda.synchronize()
    assert torch.equal(torch.stack(out_h), out_a.cpu())
    assert torch.equal(a.lengths(), b.lengths())
    assert torch.equal(a.slot_positions(), b.slot_positions())
    assert a.position == b.position == wl.cap
    assert a.status() == b.status() == dms.DMS_OK
    a.close()
    b.close()
