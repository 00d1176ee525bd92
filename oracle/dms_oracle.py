"""CPU oracle for Dynamic Memory Sparsification (DMS) decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run this module; the product
path (the C-ABI library and its Python binding) never does.  It shares no code
with the CUDA path: inputs reach it as plain arrays produced by the seeded
workload generator, and every value it returns is computed here, in float64,
from the definitions below.

Sources (web pages on the method; cited by title and section):

* "Inference-Time Hyper-Scaling with KV Cache Compression", AI research-map
  summary, section "Approach": each KV head of every token carries a learned
  binary eviction decision, and the eviction is carried out only after a delay
  window.  Sections "Measured effects reported in the paper" and "Surprising
  findings" fix that window at 16 tokens.
* Same summary, section "Experimental setup" (metrics): "KV-cache token reads"
  and "peak tokens in memory" are the method's own cost measures.
* Same paper, English abstract (chatpaper page): DMS delays token eviction
  rather than discarding tokens early.

Readings taken where the pages are silent:

* Decision at inference: ``e = (logit > 0)`` evaluated on the float32 logit,
  which is the threshold ``sigmoid(logit) > 0.5`` without the rounding of a
  float32 sigmoid near 0.5.  A logit of exactly 0 (or -0, or NaN) keeps.
* Delay: the decision of token j takes effect at step j + w.  Key j is visible
  to the query at step t iff ``j <= t`` and (``j >= t - w + 1`` or not e_j).
* Slot policy: at the append of token t, if t >= w and token t - w was marked,
  t - w leaves first and t takes its slot; otherwise t takes slot ``len`` and
  ``len`` grows by one.  Appending past the capacity is an error: the token is
  not stored, its ring entry records "no slot, keep", the error is sticky.
* Query head g reads KV head ``g // (Hq // Hkv)`` (contiguous GQA groups).
* ``scale`` is supplied by the caller; the workloads use ``1/sqrt(D)``.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
against library routines (PyTorch scaled-dot-product attention), closed forms
and brute-force enumeration; see the test file for which pin covers which
function.
"""
from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------------------
# Decision and visibility (summary page, "Approach")
# ---------------------------------------------------------------------------

def eviction_decisions(logits) -> np.ndarray:
    """Binary eviction decision per (token, KV head): ``logit > 0`` in float32.

    The summary page ("Approach") describes a learned per-head binary decision
    relaxed with a Gumbel-sigmoid during training; at inference the relaxation
    is replaced by the hard threshold sigmoid(logit) > 0.5, i.e. logit > 0.
    """
    x = np.asarray(logits, dtype=np.float32)
    return x > np.float32(0.0)


def visibility_mask(e_col, t: int, w: int) -> np.ndarray:
    """Keys visible to the query at step ``t`` for one (sequence, KV head).

    ``e_col[j]`` is token j's decision.  Returns ``bool[t + 1]`` over
    positions 0..t: key j is visible iff it is inside the delay window
    (``j >= t - w + 1``) or it was not marked for eviction.  The token of step
    t itself is always visible because w >= 1.
    """
    if w < 1:
        raise ValueError("window must be >= 1")
    e = np.asarray(e_col, dtype=bool)[: t + 1]
    j = np.arange(t + 1)
    return (j >= t - w + 1) | (~e)


def retained_length(e_col, n: int, w: int) -> int:
    """Number of tokens held for one (sequence, KV head) after ``n`` appends.

    Every token is retained except those marked for eviction whose delay has
    run out: ``n - #{j <= n - 1 - w : e_j}``.
    """
    e = np.asarray(e_col, dtype=bool)
    last = n - w  # tokens 0..n-1-w have been in the cache for >= w steps
    if last <= 0:
        return int(n)
    return int(n - np.count_nonzero(e[:last]))


def kv_token_reads(e, n_steps: int, w: int) -> int:
    """"KV-cache token reads" (summary page, "Experimental setup") of a decode
    run of ``n_steps`` steps: the sum over steps t = 1..n_steps and over all
    (sequence, KV head) of the retained length after t appends.

    ``e`` is ``bool[..., T]`` with positions on the last axis.
    """
    e = np.asarray(e, dtype=bool)
    flat = e.reshape(-1, e.shape[-1])
    total = 0
    for row in flat:
        for t in range(1, n_steps + 1):
            total += retained_length(row, t, w)
    return total


# ---------------------------------------------------------------------------
# Attention (plain softmax attention restricted to the visible keys)
# ---------------------------------------------------------------------------

def softmax_attention(qv, keys, values, scale: float) -> np.ndarray:
    """``softmax(scale * keys @ qv) @ values`` in float64 (max-subtracted)."""
    q = np.asarray(qv, dtype=np.float64)
    k = np.asarray(keys, dtype=np.float64)
    v = np.asarray(values, dtype=np.float64)
    s = (k @ q) * float(scale)
    s = s - s.max()
    p = np.exp(s)
    return (p @ v) / p.sum()


def decode_attention(q_t, k_hist, v_hist, e_hist, t: int, w: int, scale: float) -> np.ndarray:
    """DMS decode attention for the query of step ``t``.

    Shapes (float arrays hold bf16 values widened exactly):
      q_t     [B][Hq][D]       query of step t
      k_hist  [B][Hkv][T][D]   keys of positions 0..T-1 (T >= t + 1)
      v_hist  [B][Hkv][T][D]
      e_hist  [B][Hkv][T]      eviction decisions (bool)
    Returns ``float64 [B][Hq][D]``.  Query head g uses KV head g // (Hq/Hkv).
    """
    q_t = np.asarray(q_t)
    B, Hq, D = q_t.shape
    Hkv = k_hist.shape[1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    out = np.empty((B, Hq, D), dtype=np.float64)
    for b in range(B):
        for h in range(Hkv):
            vis = visibility_mask(e_hist[b, h], t, w)
            ks = np.asarray(k_hist[b, h, : t + 1])[vis]
            vs = np.asarray(v_hist[b, h, : t + 1])[vis]
            for g in range(G):
                out[b, h * G + g] = softmax_attention(q_t[b, h * G + g], ks, vs, scale)
    return out


def prefill_attention(q_chunk, k_hist, v_hist, e_hist, t0: int, w: int, scale: float) -> np.ndarray:
    """Attention of a chunk of C queries at steps t0..t0+C-1, each with the same
    per-step visibility rule as :func:`decode_attention`.

    q_chunk [B][Hq][C][D] -> float64 [B][Hq][C][D].
    """
    q_chunk = np.asarray(q_chunk)
    C = q_chunk.shape[2]
    out = np.empty(q_chunk.shape, dtype=np.float64)
    for c in range(C):
        out[:, :, c] = decode_attention(q_chunk[:, :, c], k_hist, v_hist, e_hist, t0 + c, w, scale)
    return out


# ---------------------------------------------------------------------------
# Slot bookkeeping of the compacted per-(sequence, KV head) cache
# ---------------------------------------------------------------------------

class SlotSimulator:
    """Sequential model of the compacted cache's slot map.

    State per (b, h): ``len`` (slots in use), ``slot_pos[cap]`` (position held
    by each slot, -1 = never written), a ring of the last w appends holding
    (slot, decision).  ``append`` follows the slot policy in the module
    docstring; ``append_chunk`` is defined as that many single appends.
    """

    def __init__(self, batch: int, kv_heads: int, capacity: int, window: int):
        if min(batch, kv_heads, capacity, window) < 1:
            raise ValueError("all sizes must be >= 1")
        self.B, self.H, self.cap, self.w = batch, kv_heads, capacity, window
        self.t = 0
        self.len = np.zeros((batch, kv_heads), dtype=np.int64)
        self.slot_pos = np.full((batch, kv_heads, capacity), -1, dtype=np.int64)
        self.ring_slot = np.full((batch, kv_heads, window), -1, dtype=np.int64)
        self.ring_flag = np.zeros((batch, kv_heads, window), dtype=bool)
        self.overflow = False

    def append(self, e_t) -> np.ndarray:
        """Append token ``self.t`` to every (b, h); returns its slot per head
        (-1 where it overflowed the capacity).  Heads are independent, so the
        rule is applied to all of them at once."""
        e_t = np.asarray(e_t, dtype=bool).reshape(self.B, self.H)
        t, w = self.t, self.w
        r = t % w
        retire = (t >= w) & self.ring_flag[:, :, r]      # token t - w was marked: it leaves now
        s = np.where(retire, self.ring_slot[:, :, r], self.len)  # ... and t takes its slot
        over = ~retire & (self.len >= self.cap)
        self.len = self.len + (~retire & ~over)
        s = np.where(over, -1, s)
        bi, hi = np.nonzero(s >= 0)
        self.slot_pos[bi, hi, s[bi, hi]] = t
        self.ring_slot[:, :, r] = s
        self.ring_flag[:, :, r] = e_t & (s >= 0)
        if over.any():
            self.overflow = True
        self.t = t + 1
        return s

    def append_chunk(self, e_chunk) -> np.ndarray:
        """``e_chunk [B][Hkv][C]``: C appends in position order."""
        e_chunk = np.asarray(e_chunk, dtype=bool)
        C = e_chunk.shape[-1]
        out = np.empty((self.B, self.H, C), dtype=np.int64)
        for c in range(C):
            out[:, :, c] = self.append(e_chunk[:, :, c])
        return out

    def occupied_positions(self, b: int, h: int) -> np.ndarray:
        """Positions held in slots 0..len-1, in slot order."""
        return self.slot_pos[b, h, : self.len[b, h]].copy()
