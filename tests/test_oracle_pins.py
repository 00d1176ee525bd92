"""Pins of the CPU oracle to facts fixed outside it (no GPU).

Each ``check_*`` function compares the oracle against something it does not
share code with -- PyTorch's scaled-dot-product attention (a library
routine), a closed form, or a brute-force queue simulation -- and raises
AssertionError on a mismatch.  ``test_*`` functions run them on the real
oracle; ``test_planted_*`` plant plausible mistakes in a copy of the oracle's
functions and require that at least one check fails.

Rule being pinned ("Inference-Time Hyper-Scaling with KV Cache Compression",
AI research-map summary, "Approach"; window of 16 tokens from its
"Measured effects reported in the paper" table): a per-(token, KV head)
binary eviction decision whose eviction is carried out after a delay window.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle.dms_oracle as O


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16).float().numpy()


def _problem(B=2, Hq=6, Hkv=2, D=16, T=40, seed=0):
    q = _rand((B, Hq, T, D), seed)
    k = _rand((B, Hkv, T, D), seed + 1)
    v = _rand((B, Hkv, T, D), seed + 2)
    return q, k, v


def _sdpa(q, k, v, mask, scale):
    """Library attention in float64: q [B][Hq][T][D], k/v [B][Hkv][T][D],
    mask bool [T][T] (True = attend)."""
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).double(), torch.from_numpy(k).double(), torch.from_numpy(v).double(),
        attn_mask=torch.from_numpy(mask), scale=scale, enable_gqa=True).numpy()


def _oracle_all_steps(q, k, v, e, w, scale, decode=None):
    decode = decode or O.decode_attention
    T = q.shape[2]
    return np.stack([decode(q[:, :, t], k, v, e, t, w, scale) for t in range(T)], axis=2)


# ---------------------------------------------------------------------------
# checks
# ---------------------------------------------------------------------------

def check_all_keep_is_causal(decode=None, decisions=None):
    decisions = decisions or O.eviction_decisions
    q, k, v = _problem()
    B, Hkv, T = k.shape[0], k.shape[1], k.shape[2]
    logits = -np.abs(_rand((B, Hkv, T), 7)) - 0.5
    e = decisions(logits)
    scale = 0.37
    got = _oracle_all_steps(q, k, v, e, 16, scale, decode)
    causal = np.tril(np.ones((T, T), dtype=bool))
    ref = _sdpa(q, k, v, causal, scale)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def check_all_evict_is_sliding_window(decode=None, decisions=None):
    decisions = decisions or O.eviction_decisions
    q, k, v = _problem(seed=3)
    B, Hkv, T = k.shape[0], k.shape[1], k.shape[2]
    scale = 0.25
    for w in (1, 4, 16):
        logits = np.abs(_rand((B, Hkv, T), 11)) + 0.5
        e = decisions(logits)
        got = _oracle_all_steps(q, k, v, e, w, scale, decode)
        ones = torch.ones(T, T, dtype=torch.bool)
        band = (torch.tril(ones) & ~torch.tril(ones, diagonal=-w)).numpy()  # keys t-w+1..t
        ref = _sdpa(q, k, v, band, scale)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def check_long_window_is_causal(decode=None):
    q, k, v = _problem(seed=5, T=24)
    B, Hkv, T = k.shape[0], k.shape[1], k.shape[2]
    e = _rand((B, Hkv, T), 13) > 0
    scale = 0.5
    got = _oracle_all_steps(q, k, v, e, T, scale, decode)
    ref = _sdpa(q, k, v, np.tril(np.ones((T, T), dtype=bool)), scale)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def check_first_step_returns_v0(decode=None):
    decode = decode or O.decode_attention
    q, k, v = _problem(seed=9)
    e = np.ones(k.shape[:3], dtype=bool)
    out = decode(q[:, :, 0], k, v, e, 0, 16, 1.0)
    G = q.shape[1] // k.shape[1]
    expect = np.repeat(v[:, :, 0], G, axis=1)  # query head g reads KV head g // G
    assert np.array_equal(out, expect.astype(np.float64))


def _queue_visible(e_row, w):
    """Brute force: tokens enter a list in order; a token marked for eviction
    leaves exactly w steps after it entered.  Returns the set present after
    each step."""
    present, sets = [], []
    for t, flag in enumerate(e_row):
        present = [(j, f) for (j, f) in present if not (f and t - j >= w)]
        present.append((t, bool(flag)))
        sets.append(frozenset(j for j, _ in present))
    return sets


def check_bruteforce_masks(T=12, windows=(1, 2, 3, 5), visibility=None, retained=None, sim_cls=None):
    visibility = visibility or O.visibility_mask
    retained = retained or O.retained_length
    sim_cls = sim_cls or O.SlotSimulator
    for w in windows:
        for bits in itertools.product((False, True), repeat=T):
            e = np.array(bits)
            qsets = _queue_visible(e, w)
            sim = sim_cls(1, 1, T, w)
            for t in range(T):
                sim.append(e[t:t + 1].reshape(1, 1))
                mask_set = frozenset(np.nonzero(visibility(e, t, w))[0].tolist())
                assert mask_set == qsets[t], (w, bits, t)
                assert retained(e, t + 1, w) == len(qsets[t]), (w, bits, t)
                occ = sim.occupied_positions(0, 0)
                assert int(sim.len[0, 0]) == len(qsets[t])
                assert (occ >= 0).all() and frozenset(occ.tolist()) == qsets[t], (w, bits, t)


def check_zero_keys_give_visible_mean(decode=None):
    """With every key zero, softmax is uniform over the visible keys, so the
    output is the plain mean of the visible values (closed form)."""
    decode = decode or O.decode_attention
    rng = np.random.default_rng(4)
    B, Hq, Hkv, D, T, w = 2, 4, 2, 8, 30, 5
    q = rng.standard_normal((B, Hq, D))
    k = np.zeros((B, Hkv, T, D))
    v = rng.standard_normal((B, Hkv, T, D))
    e = rng.random((B, Hkv, T)) < 0.6
    G = Hq // Hkv
    for t in range(T):
        out = decode(q, k, v, e, t, w, 0.3)
        for b in range(B):
            for h in range(Hkv):
                vis = sorted(_queue_visible(e[b, h], w)[t])
                mean = v[b, h, vis].mean(axis=0)
                for g in range(G):
                    np.testing.assert_allclose(out[b, h * G + g], mean, rtol=1e-12, atol=1e-13)


def check_kv_token_reads_closed_forms():
    n, w = 50, 16
    keep = np.zeros((3, n), dtype=bool)
    evict = np.ones((3, n), dtype=bool)
    assert O.kv_token_reads(keep, n, w) == 3 * n * (n + 1) // 2
    assert O.kv_token_reads(evict, n, w) == 3 * sum(min(t, w) for t in range(1, n + 1))



# ---------------------------------------------------------------------------
# chunked prefill: C queries at positions t0 .. t0 + C - 1 of one call
# ---------------------------------------------------------------------------

_PF_T0, _PF_C = 13, 20  # rows 13 .. 32 of a 40-token problem


def _prefill_rows(q, k, v, e, t0, C, w, scale, prefill=None):
    prefill = prefill or O.prefill_attention
    return prefill(q[:, :, t0:t0 + C], k, v, e, t0, w, scale)


def check_prefill_all_keep_is_causal(prefill=None):
    """Every decision 'keep': the chunk's rows equal rows t0 .. t0 + C - 1 of
    causal attention over the whole sequence (library SDPA, float64)."""
    q, k, v = _problem(seed=21)
    B, Hkv, T = k.shape[0], k.shape[1], k.shape[2]
    e = O.eviction_decisions(-np.abs(_rand((B, Hkv, T), 22)) - 0.5)
    scale = 0.41
    t0, C = _PF_T0, _PF_C
    got = _prefill_rows(q, k, v, e, t0, C, 16, scale, prefill)
    ref = _sdpa(q, k, v, np.tril(np.ones((T, T), dtype=bool)), scale)[:, :, t0:t0 + C]
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def check_prefill_all_evict_is_band(prefill=None):
    """Every decision 'evict': the chunk's rows equal those rows of attention
    restricted to the last w keys (the band t - w + 1 .. t)."""
    q, k, v = _problem(seed=23)
    B, Hkv, T = k.shape[0], k.shape[1], k.shape[2]
    e = O.eviction_decisions(np.abs(_rand((B, Hkv, T), 24)) + 0.5)
    scale = 0.29
    t0, C = _PF_T0, _PF_C
    ones = torch.ones(T, T, dtype=torch.bool)
    for w in (1, 4, 16):
        got = _prefill_rows(q, k, v, e, t0, C, w, scale, prefill)
        band = (torch.tril(ones) & ~torch.tril(ones, diagonal=-w)).numpy()
        ref = _sdpa(q, k, v, band, scale)[:, :, t0:t0 + C]
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def check_prefill_matches_queue(prefill=None):
    """Random decisions: row c of the chunk attends exactly to the tokens the
    brute-force queue holds after step t0 + c (a token marked for eviction
    leaves w steps after it entered).  The reference is SDPA with a per-head
    mask built from the queue, not from the oracle's visibility rule."""
    q, k, v = _problem(seed=25)
    B, Hq, T = q.shape[0], q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    G = Hq // Hkv
    rng = np.random.default_rng(26)
    e = rng.random((B, Hkv, T)) < 0.6
    scale = 0.33
    t0, C = _PF_T0, _PF_C
    for w in (1, 3, 5):
        mask = np.zeros((B, Hq, C, T), dtype=bool)
        for b in range(B):
            for h in range(Hkv):
                sets = _queue_visible(e[b, h], w)
                for c in range(C):
                    mask[b, h * G:(h + 1) * G, c, sorted(sets[t0 + c])] = True
        got = _prefill_rows(q, k, v, e, t0, C, w, scale, prefill)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[:, :, t0:t0 + C]).double(), torch.from_numpy(k).double(),
            torch.from_numpy(v).double(), attn_mask=torch.from_numpy(mask), scale=scale, enable_gqa=True).numpy()
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)

# ---------------------------------------------------------------------------
# pins on the real oracle
# ---------------------------------------------------------------------------

def test_all_keep_equals_causal_attention():
    check_all_keep_is_causal()


def test_all_evict_equals_sliding_window():
    check_all_evict_is_sliding_window()


def test_window_longer_than_sequence_is_causal():
    check_long_window_is_causal()


def test_first_step_returns_first_value():
    check_first_step_returns_v0()


def test_bruteforce_all_patterns():
    check_bruteforce_masks()


def test_zero_keys_closed_form():
    check_zero_keys_give_visible_mean()


def test_kv_token_reads_closed_forms():
    check_kv_token_reads_closed_forms()


def test_retained_length_all_evict_is_min_n_w():
    e = np.ones(100, dtype=bool)
    for n in range(0, 100):
        assert O.retained_length(e, n, 16) == min(n, 16)


def test_decision_threshold_edges():
    x = np.array([0.0, -0.0, np.nan, 1e-45, 2.9e-8, -1e-45, 1.0, -1.0, np.inf, -np.inf], dtype=np.float32)
    got = O.eviction_decisions(x)
    assert got.tolist() == [False, False, False, True, True, False, True, False, True, False]
    # Away from 0 the threshold equals sigmoid > 0.5 (library sigmoid, float64).
    y = np.linspace(-6, 6, 1001).astype(np.float32)
    y = y[np.abs(y) > 1e-3]
    assert np.array_equal(O.eviction_decisions(y), torch.sigmoid(torch.from_numpy(y).double()).numpy() > 0.5)
    # Why the oracle does not threshold a float32 sigmoid: it rounds to 0.5 here.
    assert float(torch.sigmoid(torch.tensor(2.9e-8, dtype=torch.float32))) == 0.5


def test_permutation_invariance():
    rng = np.random.default_rng(1)
    qv = rng.standard_normal(32)
    keys = rng.standard_normal((200, 32))
    vals = rng.standard_normal((200, 32))
    perm = rng.permutation(200)
    a = O.softmax_attention(qv, keys, vals, 0.2)
    b = O.softmax_attention(qv, keys[perm], vals[perm], 0.2)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_slot_capacity_overflow():
    sim = O.SlotSimulator(1, 2, 4, 3)
    for _ in range(4):
        s = sim.append(np.zeros((1, 2), dtype=bool))
        assert (s >= 0).all()
    assert not sim.overflow
    s = sim.append(np.zeros((1, 2), dtype=bool))
    assert sim.overflow and (s == -1).all()
    # all-evict with capacity == window never overflows
    sim = O.SlotSimulator(1, 1, 3, 3)
    for _ in range(50):
        sim.append(np.ones((1, 1), dtype=bool))
    assert not sim.overflow and int(sim.len[0, 0]) == 3


def test_chunk_append_matches_single_appends():
    rng = np.random.default_rng(2)
    e = rng.random((2, 3, 70)) < 0.7
    a = O.SlotSimulator(2, 3, 64, 16)
    b = O.SlotSimulator(2, 3, 64, 16)
    a.append_chunk(e[:, :, :33])
    a.append_chunk(e[:, :, 33:])
    for t in range(70):
        b.append(e[:, :, t])
    assert np.array_equal(a.slot_pos, b.slot_pos) and np.array_equal(a.len, b.len)



def test_prefill_all_keep_equals_causal_rows():
    check_prefill_all_keep_is_causal()


def test_prefill_all_evict_equals_band_rows():
    check_prefill_all_evict_is_band()


def test_prefill_rows_match_bruteforce_queue():
    check_prefill_matches_queue()

# ---------------------------------------------------------------------------
# planted mistakes: each one must be caught by at least one check
# ---------------------------------------------------------------------------

def _fails(fn, *a, **kw):
    try:
        fn(*a, **kw)
    except AssertionError:
        return True
    return False


def test_planted_off_by_one_window():
    def bad_vis(e_col, t, w):
        e = np.asarray(e_col, dtype=bool)[: t + 1]
        j = np.arange(t + 1)
        return (j >= t - w) | (~e)
    assert _fails(check_bruteforce_masks, T=6, windows=(2,), visibility=bad_vis)


def test_planted_wrong_retained_formula():
    def bad_ret(e_col, n, w):
        e = np.asarray(e_col, dtype=bool)
        return int(n - np.count_nonzero(e[: max(n - w + 1, 0)]))
    assert _fails(check_bruteforce_masks, T=6, windows=(2,), retained=bad_ret)


def test_planted_write_then_retire_slot_policy():
    class BadSim(O.SlotSimulator):
        def append(self, e_t):
            e_t = np.asarray(e_t, dtype=bool).reshape(self.B, self.H)
            t, w = self.t, self.w
            r = t % w
            for b in range(self.B):
                for h in range(self.H):
                    s = int(self.len[b, h])  # write first into a fresh slot ...
                    self.len[b, h] = s + 1
                    if t >= w and self.ring_flag[b, h, r]:
                        old = int(self.ring_slot[b, h, r])  # ... then free the retired one
                        self.slot_pos[b, h, old] = -1
                        self.len[b, h] -= 1
                    self.slot_pos[b, h, s] = t
                    self.ring_slot[b, h, r] = s
                    self.ring_flag[b, h, r] = bool(e_t[b, h])
            self.t = t + 1
    assert _fails(check_bruteforce_masks, T=8, windows=(2,), sim_cls=BadSim)


def test_planted_wrong_head_mapping():
    def bad_decode(q_t, k_hist, v_hist, e_hist, t, w, scale):
        B, Hq, D = q_t.shape
        Hkv = k_hist.shape[1]
        out = np.empty((B, Hq, D))
        for b in range(B):
            for g in range(Hq):
                h = g % Hkv  # interleaved instead of contiguous groups
                vis = O.visibility_mask(e_hist[b, h], t, w)
                out[b, g] = O.softmax_attention(q_t[b, g], k_hist[b, h, : t + 1][vis], v_hist[b, h, : t + 1][vis], scale)
        return out
    assert _fails(check_all_keep_is_causal, decode=bad_decode)


def test_planted_missing_scale_and_swapped_kv():
    def no_scale(q_t, k_hist, v_hist, e_hist, t, w, scale):
        return O.decode_attention(q_t, k_hist, v_hist, e_hist, t, w, 1.0)

    def swapped(q_t, k_hist, v_hist, e_hist, t, w, scale):
        return O.decode_attention(q_t, v_hist, k_hist, e_hist, t, w, scale)
    assert _fails(check_all_keep_is_causal, decode=no_scale)
    assert _fails(check_all_keep_is_causal, decode=swapped)


def test_planted_decision_inverted():
    def inverted(logits):
        return np.asarray(logits, dtype=np.float32) < 0
    assert _fails(check_all_evict_is_sliding_window, decisions=inverted)


def test_golden_worked_examples():
    """tests/golden/delayed_eviction_examples.txt: the oracle still produces the
    recorded rows, and each row's visible set agrees with the brute-force queue."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "delayed_eviction_examples.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    cases = {}
    for name, w, t, d, vis, ret, slots in rows:
        cases.setdefault((name, int(w)), []).append((int(t), int(d), vis, int(ret), slots))
    assert len(cases) == 3
    for (name, w), steps in cases.items():
        e = np.array([d for _, d, _, _, _ in steps], dtype=bool)
        qsets = _queue_visible(e, w)
        sim = O.SlotSimulator(1, 1, 64, w)
        for t, _, vis, ret, slots in steps:
            sim.append(e[t:t + 1].reshape(1, 1))
            want_vis = [int(x) for x in vis.split(",")]
            assert sorted(qsets[t]) == want_vis
            assert O.retained_length(e, t + 1, w) == ret == len(want_vis)
            assert sim.occupied_positions(0, 0).tolist() == [int(x) for x in slots.split(",")]


def test_planted_prefill_position_and_chunk_index_slips():
    """A query row evaluated one position early, a query taken from the wrong
    row of the chunk, and every row evaluated at t0 are each caught."""
    def early(q_chunk, k_hist, v_hist, e_hist, t0, w, scale):
        C = q_chunk.shape[2]
        return np.stack([O.decode_attention(q_chunk[:, :, c], k_hist, v_hist, e_hist, t0 + c - 1, w, scale)
                         for c in range(C)], axis=2)

    def wrong_row(q_chunk, k_hist, v_hist, e_hist, t0, w, scale):
        C = q_chunk.shape[2]
        return np.stack([O.decode_attention(q_chunk[:, :, (c + 1) % C], k_hist, v_hist, e_hist, t0 + c, w, scale)
                         for c in range(C)], axis=2)

    def frozen(q_chunk, k_hist, v_hist, e_hist, t0, w, scale):
        C = q_chunk.shape[2]
        return np.stack([O.decode_attention(q_chunk[:, :, c], k_hist, v_hist, e_hist, t0, w, scale)
                         for c in range(C)], axis=2)
    for bad in (early, wrong_row, frozen):
        assert _fails(check_prefill_all_keep_is_causal, prefill=bad)
        assert _fails(check_prefill_matches_queue, prefill=bad)
