"""Pins of the oracle's Quest decode step ("Long context, KV eviction and sparse attention",
Sparse attention: per-page key minimum and maximum, the bound sum_d max(q_d kmin_d,
q_d kmax_d), the pages with the largest bounds plus the trailing partial page, attention over
them).

* The bound is the maximum of q.x over the box [kmin, kmax] (brute force over its corners)
  and so bounds every key of the page; with one dimension it is the page's best score.
* The chosen pages are the n_sel largest bounds with ties to the lower page (a stable
  library sort).
* The output is plain attention over the chosen pages' tokens and the tail (NumPy brute
  force), and with n_sel covering every full page it is the dense oracle, bit for bit.
* The summaries are the library min / max over each page.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
import workloads as W


def _keys_of_page(x, b, g, m):
    P = x.page_size
    pg = int(x.block_table[b][m])
    return x.k_pool[pg, g].double().numpy()          # [P, D]


def test_bound_is_the_box_maximum_and_bounds_every_key():
    x = W.make_gqa(2, 4, 2, 5, [48, 37], page_size=8, shuffle=True, seed=11,
                   dtype=torch.float32)
    _, _, _, ub = oracle.quest(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale, 2)
    q = x.q.double().numpy()
    for b, L in enumerate([48, 37]):
        for h in range(4):
            g = h // 2
            for m in range(L // 8):
                K = _keys_of_page(x, b, g, m)
                lo, hi = K.min(0), K.max(0)
                corners = max(float(np.dot(q[b, h], np.where(c, hi, lo)))
                              for c in itertools.product([0, 1], repeat=5))
                assert ub[b, h, m] == pytest.approx(corners, rel=1e-12, abs=1e-12)
                assert (K @ q[b, h]).max() <= ub[b, h, m] + 1e-12
            assert np.isnan(ub[b, h, L // 8:]).all()


def test_one_dimension_bound_is_the_best_score():
    x = W.make_gqa(1, 2, 1, 1, [64], page_size=16, seed=12, dtype=torch.float32)
    _, _, _, ub = oracle.quest(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale, 1)
    for h in range(2):
        for m in range(4):
            K = _keys_of_page(x, 0, 0, m)
            assert ub[0, h, m] == (K[:, 0] * float(x.q[0, h, 0])).max()


def _brute(x, n_sel):
    """Selection by a stable sort of the bounds, attention by NumPy over the chosen tokens."""
    _, _, _, ub = oracle.quest(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale, n_sel)
    P, G = x.page_size, x.Hq // x.Hkv
    q = x.q.double().numpy()
    outs, sels = np.zeros((x.B, x.Hq, x.D)), np.full((x.B, x.Hq, n_sel), -1)
    for b in range(x.B):
        L = int(x.seq_lens[b])
        full = L // P
        for h in range(x.Hq):
            u = ub[b, h, :full]
            order = np.argsort(-u, kind="stable")[:n_sel]
            chosen = np.sort(order)
            sels[b, h, :len(chosen)] = chosen
            toks = [t for m in chosen for t in range(m * P, (m + 1) * P)] + list(range(full * P, L))
            rows = [(int(x.block_table[b][t // P]), t % P) for t in toks]
            K = np.stack([x.k_pool[pg, h // G, s].double().numpy() for pg, s in rows])
            V = np.stack([x.v_pool[pg, h // G, s].double().numpy() for pg, s in rows])
            sc = x.scale * (K @ q[b, h])
            e = np.exp(sc - sc.max())
            outs[b, h] = (e[:, None] * V).sum(0) / e.sum()
    return outs, sels


@pytest.mark.parametrize("lens,n_sel", [([100, 33, 16, 7], 3), ([257, 64], 5)])
def test_selection_and_attention_brute_force(lens, n_sel):
    x = W.make_gqa(len(lens), 4, 2, 8, lens, page_size=16, shuffle=True, seed=13,
                   dtype=torch.float32)
    out, _, sel, _ = oracle.quest(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale,
                                  n_sel)
    want_out, want_sel = _brute(x, n_sel)
    assert np.array_equal(sel, want_sel)
    assert np.allclose(out, want_out, rtol=1e-12, atol=1e-12)


def test_ties_go_to_the_lower_page():
    # every page holds the same keys: all bounds are equal, the first n_sel pages win
    x = W.make_gqa(1, 2, 1, 4, [80], page_size=16, seed=14, dtype=torch.float32)
    pg0 = int(x.block_table[0][0])
    for m in range(5):
        x.k_pool[int(x.block_table[0][m])] = x.k_pool[pg0]
    _, _, sel, _ = oracle.quest(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale, 2)
    assert sel[0, 0].tolist() == [0, 1] and sel[0, 1].tolist() == [0, 1]


def test_every_page_chosen_is_dense_attention():
    lens = [100, 64, 5]
    x = W.make_gqa(3, 8, 2, 16, lens, page_size=16, shuffle=True, seed=15)
    out, lse, _, _ = oracle.quest(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale,
                                  64)
    ref, ref_lse = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)


def test_minmax_summaries():
    x = W.make_gqa(2, 4, 2, 32, [64, 64], page_size=16, seed=16)
    kmin, kmax = oracle.quest_minmax(x.k_pool)
    k = x.k_pool.double()
    assert np.array_equal(kmin, k.amin(2).numpy()) and np.array_equal(kmax, k.amax(2).numpy())
