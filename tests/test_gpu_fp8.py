"""GPU parity of the FP8 (E4M3) KV storage against the CPU oracles.

Bar:
* quantization (an integer decision made in float32 on both sides): every
  stored code and scale bit-exact against ``oracle.fp8_oracle``;
* bookkeeping (lengths, slot map): bit-exact against the slot simulator;
* attention: against the float64 oracle evaluated on the dequantized rows
  (code * scale), within the same bars as the bf16 path (max-abs 1e-2 /
  mean relative 1e-3 stated, 1e-4 / 1e-4 asserted): the kernel's arithmetic is
  fp32 on exact E4M3 values, so only fp32 rounding separates the two.
"""
import numpy as np
import pytest
import torch

import oracle.dms_oracle as O
import oracle.fp8_oracle as F
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


class Fp8Run:
    """One fp8 cache driven through appends, with the oracle's quantized rows
    and slot simulator alongside."""

    def __init__(self, wl: W.Workload, T: int, rows=None, layer: int = 0):
        self.wl, self.layer = wl, layer
        k, v, lg = W.kv_range(wl, layer, 0, T)
        self.k, self.v, self.lg = k, v, lg
        self.e = O.eviction_decisions(lg.numpy())
        self.rows = list(range(wl.B)) if rows is None else list(rows)
        self.kc, self.ks = F.quantize_rows(k[self.rows].float().numpy())
        self.vc, self.vs = F.quantize_rows(v[self.rows].float().numpy())
        self.k_deq = F.dequantize_rows(self.kc, self.ks)
        self.v_deq = F.dequantize_rows(self.vc, self.vs)
        self.cache = dms.DmsCache(wl.B, wl.Hkv, wl.cap, wl.D, wl.w, kv_format="fp8")
        self.sim = O.SlotSimulator(wl.B, wl.Hkv, wl.cap, wl.w)
        self.t = 0

    def append(self):
        t = self.t
        self.cache.append(self.k[:, :, t].contiguous().cuda(), self.v[:, :, t].contiguous().cuda(),
                          self.lg[:, :, t].contiguous().cuda())
        self.sim.append(self.e[:, :, t])
        self.t += 1

    def append_chunk(self, n):
        sl = slice(self.t, self.t + n)
        self.cache.append_chunk(self.k[:, :, sl].contiguous().cuda(), self.v[:, :, sl].contiguous().cuda(),
                                self.lg[:, :, sl].contiguous().cuda())
        self.sim.append_chunk(self.e[:, :, sl])
        self.t += n

    def check_state(self):
        assert np.array_equal(self.cache.lengths().cpu().numpy(), self.sim.len), f"lengths at t={self.t}"
        assert np.array_equal(self.cache.slot_positions().cpu().numpy(), self.sim.slot_pos), f"slots at t={self.t}"
        kk, vv = (x.cpu().numpy() for x in self.cache.export_kv())
        ks, vs = (x.cpu().numpy() for x in self.cache.export_scales())
        for j, b in enumerate(self.rows):
            for h in range(self.wl.Hkv):
                n = int(self.sim.len[b, h])
                pos = self.sim.slot_pos[b, h, :n].astype(np.int64)
                assert np.array_equal(kk[b, h, :n], self.kc[j, h, pos]), ("K codes", b, h)
                assert np.array_equal(vv[b, h, :n], self.vc[j, h, pos]), ("V codes", b, h)
                assert np.array_equal(ks[b, h, :n], self.ks[j, h, pos]), ("K scales", b, h)
                assert np.array_equal(vs[b, h, :n], self.vs[j, h, pos]), ("V scales", b, h)

    def decode_and_compare(self, q, what=""):
        """q: bf16 [B][Hq][D] (CPU) of the token appended last."""
        out = self.cache.decode_attention(q.cuda(), scale=self.wl.scale)
        assert self.cache.status() == dms.DMS_OK
        ref = O.decode_attention(q[self.rows].float().numpy(), self.k_deq, self.v_deq, self.e[self.rows],
                                 self.t - 1, self.wl.w, self.wl.scale)
        _close(out.cpu().numpy()[self.rows], ref, f"{what} t={self.t - 1}")


def _wl(B, Hq, Hkv, D, w, cap, logits, seed=21):
    return W.Workload("fp8", B=B, Hq=Hq, Hkv=Hkv, D=D, w=w, cap=cap, seed=seed, logits=logits)


@pytest.mark.parametrize("case", [
    # B, Hq, Hkv, D, w, cap, T, logits
    (2, 8, 2, 128, 16, 200, 90, ("normal", 0.5, 1.0)),    # G 4
    (3, 3, 3, 64, 16, 120, 70, ("normal", 0.0, 1.0)),     # MHA, d64
    (2, 16, 2, 128, 1, 80, 60, ("normal", 1.15, 1.0)),    # G 8, eager eviction
    (1, 10, 2, 64, 5, 100, 60, ("normal", 0.3, 2.0)),     # G 5, window 5
])
def test_fp8_appends_and_decode(case):
    B, Hq, Hkv, D, w, cap, T, logits = case
    wl = _wl(B, Hq, Hkv, D, w, cap, logits)
    run = Fp8Run(wl, T)
    q = W.q_range(wl, 0, 0, T)
    for t in range(T):
        run.append()
        if t < 20 or t % 7 == 0 or t == T - 1:
            run.decode_and_compare(q[:, :, t].contiguous(), f"fp8 {case}")
    run.check_state()
    run.cache.close()


@pytest.mark.parametrize("chunk,w", [(1, 16), (33, 16), (100, 16), (64, 4), (100, 1)])
def test_fp8_chunk_append_equals_single_appends(chunk, w):
    """Chunk appends store the same codes, scales and bookkeeping as single
    appends, and both match the oracle."""
    wl = _wl(2, 8, 2, 128, w, 400, ("normal", 0.6, 1.0), seed=5)
    T = 300
    a = Fp8Run(wl, T)
    b = dms.DmsCache(wl.B, wl.Hkv, wl.cap, wl.D, wl.w, kv_format="fp8")
    for t in range(T):
        a.append()
    for t0 in range(0, T, chunk):
        n = min(chunk, T - t0)
        b.append_chunk(a.k[:, :, t0:t0 + n].contiguous().cuda(), a.v[:, :, t0:t0 + n].contiguous().cuda(),
                       a.lg[:, :, t0:t0 + n].contiguous().cuda())
    a.check_state()
    assert torch.equal(a.cache.lengths(), b.lengths())
    assert torch.equal(a.cache.slot_positions(), b.slot_positions())
    for x, y in zip(a.cache.export_kv() + a.cache.export_scales(), b.export_kv() + b.export_scales()):
        assert torch.equal(x, y)
    assert a.cache.status() == b.status() == dms.DMS_OK


def test_fp8_step_equals_append_then_decode():
    wl = _wl(2, 8, 2, 128, 16, 200, ("normal", 0.6, 1.0), seed=13)
    T = 120
    k_all, v_all, lg_all = (x.cuda() for x in W.kv_range(wl, 0, 0, T))
    q = W.q_range(wl, 0, 0, T).cuda()
    a = dms.DmsCache(wl.B, wl.Hkv, wl.cap, wl.D, wl.w, kv_format="fp8")
    b = dms.DmsCache(wl.B, wl.Hkv, wl.cap, wl.D, wl.w, kv_format="fp8")
    out = torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.float32, device="cuda")
    for t in range(T):
        k, v, lg = (k_all[:, :, t].contiguous(), v_all[:, :, t].contiguous(), lg_all[:, :, t].contiguous())
        a.append(k, v, lg)
        ref = a.decode_attention(q[:, :, t].contiguous(), scale=wl.scale)
        b.step(k, v, lg, q[:, :, t].contiguous(), out, scale=wl.scale)
        assert torch.equal(out, ref), t
    for x, y in zip(a.export_kv() + a.export_scales(), b.export_kv() + b.export_scales()):
        assert torch.equal(x, y)
    assert a.status() == b.status() == dms.DMS_OK


def test_fp8_back_to_back_steps_and_graph():
    """FP8 storage through the one-launch step: dms_step calls with no host
    synchronisation between them (each started early under the previous one),
    and a 2-layer step graph replayed per token, give outputs, codes and scales
    equal, bit for bit, to dms_append + dms_decode_attention per token."""
    wl = _wl(2, 16, 2, 128, 16, 400, ("normal", 0.8, 1.0), seed=29)
    T0, T = 40, 240
    L = 2
    data = [tuple(x.cuda() for x in W.kv_range(wl, layer, 0, T)) + (W.q_range(wl, layer, 0, T).cuda(),)
            for layer in range(L)]
    ref = [dms.DmsCache(wl.B, wl.Hkv, wl.cap, wl.D, wl.w, kv_format="fp8") for _ in range(L)]
    got = [dms.DmsCache(wl.B, wl.Hkv, wl.cap, wl.D, wl.w, kv_format="fp8") for _ in range(L)]
    for layer in range(L):
        k, v, lg, _ = data[layer]
        for c in (ref[layer], got[layer]):
            c.append_chunk(k[:, :, :T0].contiguous(), v[:, :, :T0].contiguous(), lg[:, :, :T0].contiguous())
    kb = [torch.empty((wl.B, wl.Hkv, wl.D), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    vb = [torch.empty_like(x) for x in kb]
    lb = [torch.empty((wl.B, wl.Hkv), dtype=torch.float32, device="cuda") for _ in range(L)]
    qb = [torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    ob = [torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.float32, device="cuda") for _ in range(L)]
    graph = dms.DmsStepGraph(got, kb, vb, lb, qb, ob, wl.scale)
    hist_got = torch.zeros((T, L, wl.B, wl.Hq, wl.D), dtype=torch.float32, device="cuda")
    hist_ref = torch.zeros_like(hist_got)
    for t in range(T0, T):
        if t < (T0 + T) // 2:  # first half: dms_step per layer, back to back
            for layer in range(L):
                k, v, lg, q = data[layer]
                got[layer].step(k[:, :, t].contiguous(), v[:, :, t].contiguous(), lg[:, :, t].contiguous(),
                                q[:, :, t].contiguous(), hist_got[t, layer], scale=wl.scale)
        else:  # second half: the graph
            for layer in range(L):
                k, v, lg, q = data[layer]
                kb[layer].copy_(k[:, :, t])
                vb[layer].copy_(v[:, :, t])
                lb[layer].copy_(lg[:, :, t])
                qb[layer].copy_(q[:, :, t])
            graph.launch()
            for layer in range(L):
                hist_got[t, layer].copy_(ob[layer])
        for layer in range(L):
            k, v, lg, q = data[layer]
            ref[layer].append(k[:, :, t].contiguous(), v[:, :, t].contiguous(), lg[:, :, t].contiguous())
            ref[layer].decode_attention(q[:, :, t].contiguous(), out=hist_ref[t, layer], scale=wl.scale)
    torch.cuda.synchronize()
    assert torch.equal(hist_got, hist_ref)
    for layer in range(L):
        for x, y in zip(ref[layer].export_kv() + ref[layer].export_scales(),
                        got[layer].export_kv() + got[layer].export_scales()):
            assert torch.equal(x, y)
        assert torch.equal(ref[layer].lengths(), got[layer].lengths())
        assert ref[layer].status() == got[layer].status() == dms.DMS_OK
    graph.close()
    for c in ref + got:
        c.close()


def test_fp8_capacity_overflow_is_reported():
    wl = _wl(1, 4, 2, 64, 4, 10, ("const", -10.0))
    run = Fp8Run(wl, 14)
    for _ in range(10):
        run.append()
    assert run.cache.status() == dms.DMS_OK
    run.append()
    assert run.cache.status() == dms.DMS_ERR_CAPACITY
    run.append()
    run.check_state()


def test_fp8_format_queries_and_scale_export_refused_on_bf16():
    c = dms.DmsCache(1, 2, 64, 64, 16, kv_format="fp8")
    lib = dms.load_library()
    assert lib.dms_cache_kv_format(c.handle) == dms.DMS_KV_FP8_E4M3
    s = torch.cuda.current_stream().cuda_stream
    b = dms.DmsCache(1, 2, 64, 64, 16)
    ks = torch.empty(1, 2, 64, dtype=torch.float32, device="cuda")
    assert lib.dms_cache_export_scales(b.handle, ks.data_ptr(), ks.data_ptr(), s) == dms.DMS_ERR_INVALID_ARG
    assert lib.dms_cache_kv_format(b.handle) == dms.DMS_KV_BF16
    c.close()
    b.close()


@pytest.mark.parametrize("case", [
    # B, Hq, Hkv, D, w, history T0, chunk C, logits
    (2, 8, 2, 128, 16, 150, 70, ("normal", 0.5, 1.0)),   # G 4
    (2, 16, 2, 64, 4, 40, 33, ("normal", 0.0, 1.0)),     # G 8 (two groups of 4), window 4
    (1, 3, 3, 64, 16, 0, 20, ("const", -10.0)),          # MHA, empty cache, all keep
])
def test_fp8_prefill_equals_rounds_and_matches_oracle(case):
    """dms_prefill on an FP8 cache runs its definition, C rounds of append +
    decode: outputs and state equal those rounds done through the API, bit for
    bit, and the outputs match the oracle on dequantized rows."""
    B, Hq, Hkv, D, w, T0, C, logits = case
    wl = _wl(B, Hq, Hkv, D, w, T0 + C + 4, logits, seed=9)
    T = T0 + C
    run = Fp8Run(wl, T)
    twin = dms.DmsCache(wl.B, wl.Hkv, wl.cap, wl.D, wl.w, kv_format="fp8")
    if T0:
        run.append_chunk(T0)
        twin.append_chunk(run.k[:, :, :T0].contiguous().cuda(), run.v[:, :, :T0].contiguous().cuda(),
                          run.lg[:, :, :T0].contiguous().cuda())
    q = W.q_range(wl, 0, T0, T)
    out = run.cache.prefill(q.cuda(), run.k[:, :, T0:].contiguous().cuda(), run.v[:, :, T0:].contiguous().cuda(),
                            run.lg[:, :, T0:].contiguous().cuda(), scale=wl.scale)
    run.sim.append_chunk(run.e[:, :, T0:T])
    run.t = T
    assert run.cache.position == T
    for j in range(C):
        t = T0 + j
        twin.append(run.k[:, :, t].contiguous().cuda(), run.v[:, :, t].contiguous().cuda(),
                    run.lg[:, :, t].contiguous().cuda())
        ref = twin.decode_attention(q[:, :, j].contiguous().cuda(), scale=wl.scale)
        assert torch.equal(out[:, :, j], ref), j
        if j % 7 == 0 or j == C - 1:
            oref = O.decode_attention(q[:, :, j].float().numpy(), run.k_deq, run.v_deq, run.e, t, wl.w, wl.scale)
            _close(out[:, :, j].cpu().numpy(), oref, f"fp8 prefill {case} t={t}")
    run.check_state()
    for x, y in zip(run.cache.export_kv() + run.cache.export_scales(), twin.export_kv() + twin.export_scales()):
        assert torch.equal(x, y)
    assert run.cache.status() == twin.status() == dms.DMS_OK
    run.cache.close()
    twin.close()


def test_fp8_qwen3_8b_full_size_sampled():
    """The benchmark's shapes with FP8 storage (B32, Hq32/Hkv8, d128, n=16384,
    CR 8), in the benchmark's launch configuration: a 16380-token history filled
    in chunks, then 4 decode steps; outputs of rows {0, 31} against the oracle
    on dequantized rows; codes, scales and bookkeeping of those rows bit-exact."""
    wl = W.WORKLOADS["qwen3-8b"]
    rows = [0, wl.B - 1]
    T0 = wl.cap - 4
    run = Fp8Run(wl, wl.cap, rows=rows)
    while run.t < T0:
        run.append_chunk(min(wl.chunk, T0 - run.t))
    q = W.q_range(wl, 0, T0, wl.cap)
    for j in range(4):
        run.append()
        run.decode_and_compare(q[:, :, j].contiguous(), "fp8 qwen3-8b")
    run.check_state()
    lens = run.sim.len
    assert 7.0 < wl.cap / lens.mean() < 9.0
    run.cache.close()
    torch.cuda.empty_cache()
