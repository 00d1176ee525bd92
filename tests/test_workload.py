"""The seeded input generator (no GPU): draws are reproducible and independent
of which rows or positions are drawn together, and the logit distributions give
the eviction rates their workloads are built for (the decision itself is the
oracle's, logit > 0)."""
import numpy as np
import torch

import oracle.dms_oracle as O
from learned_kv_cache_eviction_b300 import workload as W


def test_rows_and_positions_are_drawn_independently():
    wl = W.WORKLOADS["qwen3-8b"].with_(B=4)
    k_all, v_all, l_all = W.kv_range(wl, 0, 100, 300)
    k_r, v_r, l_r = W.kv_range(wl, 0, 150, 200, rows=[2])
    assert torch.equal(k_all[2:3, :, 50:100], k_r)
    assert torch.equal(v_all[2:3, :, 50:100], v_r)
    assert torch.equal(l_all[2:3, :, 50:100], l_r)
    q1 = W.q_range(wl, 0, 60, 70)
    q2 = W.q_range(wl, 0, 0, 128)
    assert torch.equal(q1, q2[:, :, 60:70])


def test_eviction_rates_match_their_workloads():
    def rate(name, t0, t1, rows=(0, 1, 2, 3)):
        _, _, lg = W.kv_range(W.WORKLOADS[name], 0, t0, t1, rows=list(rows))
        return float(O.eviction_decisions(lg.numpy()).mean())
    assert abs(rate("tiny", 0, 256, rows=(0,)) - 0.5) < 0.06
    assert abs(rate("llama-3.2-1b", 0, 1024) - 0.75) < 0.02
    assert abs(rate("qwen3-8b", 0, 1024) - 0.875) < 0.02
    assert rate("qwen3-8b-cr1", 0, 512) == 0.0
    # drifting compression: ~75% early, ~93.75% well past 10K tokens
    assert abs(rate("qwen3-8b-drift", 0, 2048) - 0.75) < 0.03
    assert abs(rate("qwen3-8b-drift", 14000, 16000) - 0.9375) < 0.02


def test_width_workload_spans_the_stated_rates():
    wl = W.WORKLOADS["qwen-r1-32b"]
    mu = W.head_logit_bias(wl, 0)
    from scipy.stats import norm
    rates = norm.sf(-mu)  # P(N(mu, 1) > 0)
    assert rates.min() > 0.45 and rates.max() < 0.975
    kept = 1.0 - rates
    assert 6.0 < 1.0 / kept.mean() < 10.0  # aggregate compression ~8
