"""Pins of the oracle's cache append and of sliding-window attention read from a rolling
cache ("All the attentions", section 4: the window's cache is a rolling buffer of W entries,
the newest replacing the oldest; "Attention Optimizations", Sliding-window and Attention
sinks; DSA / Computation Path: the new token's row is written before attention).

* A rolling cache filled one token at a time by the oracle's append, then read by the
  ring oracle, gives the same outputs as the plain sliding-window oracle over the whole
  history, at every length: before the ring fills, exactly full, and after several wraps
  (bit-identical: both visit the same positions in the same order with the same values).
* The paged append restores a removed row exactly where the block table says; rows of every
  other token stay untouched.
* A ring without sinks keeps only the last W tokens: a token W positions older is gone.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W


def _row(pool, bt, t, P):
    return pool[int(bt[t // P]), :, t % P]


def _fill_ring_and_compare(B, Hq, Hkv, D, P, window, n_sink, T, checks, learned, dtype):
    full = W.make_gqa(B, Hq, Hkv, D, [T] * B, page_size=P, shuffle=True, extra_pages=3,
                      seed=4242 + window + n_sink, window=window, n_sink=n_sink,
                      learned_sink=learned, dtype=dtype)
    ring = W.make_ring(B, Hq, Hkv, D, [1] * B, window, n_sink=n_sink, page_size=P,
                       extra_pages=2, seed=4343 + window, dtype=dtype)
    k_ring, v_ring = ring.k_pool, ring.v_pool
    for t in range(1, T + 1):
        lens = torch.full((B,), t, dtype=torch.int32)
        k_new = torch.stack([_row(full.k_pool, full.block_table[b], t - 1, P) for b in range(B)])
        v_new = torch.stack([_row(full.v_pool, full.block_table[b], t - 1, P) for b in range(B)])
        k_ring = oracle.cache_append(k_ring, k_new, ring.block_table, lens, window, n_sink)
        v_ring = oracle.cache_append(v_ring, v_new, ring.block_table, lens, window, n_sink)
        if t in checks:
            want, want_lse = oracle.gqa(full.q, full.k_pool, full.v_pool, full.block_table, lens,
                                        full.scale, window, n_sink, full.sink_logit)
            got, got_lse = oracle.gqa(full.q, k_ring, v_ring, ring.block_table, lens,
                                      full.scale, window, n_sink, full.sink_logit, ring=True)
            assert np.array_equal(got, want), t
            assert np.array_equal(got_lse, want_lse), t


@pytest.mark.parametrize("window,n_sink,P", [(24, 4, 16), (37, 0, 16), (16, 3, 8)])
def test_ring_equals_window_over_full_history(window, n_sink, P):
    cap = window + n_sink
    T = 3 * cap + 5
    checks = {1, 2, n_sink + 1, cap - 1, cap, cap + 1, 2 * cap + 3, T}
    _fill_ring_and_compare(2, 4, 2, 16, P, window, n_sink, T, checks, learned=False,
                           dtype=torch.float32)


def test_ring_with_learned_sink_bf16():
    _fill_ring_and_compare(2, 8, 2, 16, 16, 20, 2, 70, {5, 22, 23, 70}, learned=True,
                           dtype=torch.bfloat16)


def test_paged_append_restores_the_row():
    x = W.make_gqa(3, 4, 2, 16, [1, 17, 64], page_size=16, shuffle=True, extra_pages=2, seed=77)
    k_new = torch.stack([_row(x.k_pool, x.block_table[b], L - 1, 16)
                         for b, L in enumerate([1, 17, 64])])
    holed = x.k_pool.clone()
    for b, L in enumerate([1, 17, 64]):
        holed[int(x.block_table[b][(L - 1) // 16]), :, (L - 1) % 16] = 0
    back = oracle.cache_append(holed, k_new, x.block_table, x.seq_lens)
    assert torch.equal(back, x.k_pool)
    # one row per (sequence, KV head) changed, nothing else
    other = oracle.cache_append(x.k_pool, torch.zeros_like(k_new), x.block_table, x.seq_lens)
    assert int((other != x.k_pool).any(-1).sum()) == 3 * 2


def test_ring_forgets_the_token_a_window_back():
    window, P = 8, 4
    ring = W.make_ring(1, 2, 1, 16, [1], window, page_size=P, seed=5, dtype=torch.float32)
    k = ring.k_pool
    rows = [torch.full((1, 1, 16), float(t)) for t in range(20)]
    for t in range(20):
        k = oracle.cache_append(k, rows[t], ring.block_table, torch.tensor([t + 1], dtype=torch.int32),
                                window, 0)
    held = sorted(float(k[int(ring.block_table[0][s // P]), 0, s % P, 0]) for s in range(window))
    assert held == [float(t) for t in range(12, 20)]
