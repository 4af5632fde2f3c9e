"""GPU parity of Quest page selection (summaries, choice, attention over the chosen pages)
against the oracle, through the C ABI.

* Summaries: bit-exact (minimum and maximum of stored values).
* Bounds: the GPU sums d products in float32, the oracle in fp64: |dU| <= 2^-20 * sum|terms|
  (the float32 sum of D terms, each term exact or rounded once).
* Choice: the GPU's pages must equal the oracle's, except across a near-tie of the n_sel-th
  bound (within the bound's tolerance), where any page whose oracle bound reaches the
  n_sel-th bound minus that tolerance is valid.
* Attention: every (sequence, head) is held to the attention bar of the other decode
  kernels (tests/parity.py): against the oracle's Quest output where the choice equals the
  oracle's, else against the oracle's plain attention over the GPU's validated pages.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.parity import assert_attn_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def kvd():
    import kv_cache_decode_split_gb300 as m
    return m


def _gpu(kvd, x, n_sel):
    q, kp, vp = x.q.to(DEV), x.k_pool.to(DEV), x.v_pool.to(DEV)
    bt, sl = x.block_table.to(DEV), x.seq_lens.to(DEV)
    kmin, kmax, err = kvd.quest_page_minmax(kp)
    ub = torch.full((x.B, x.Hq, x.max_pages), 7.0, device=DEV)
    sel = kvd.quest_select_pages(q, kmin, kmax, bt, sl, n_sel, x.page_size, ub_out=ub, err=err)
    lse = torch.empty(x.B, x.Hq, device=DEV)
    out = kvd.attn_decode_quest(q, kp, vp, bt, sl, sel, scale=x.scale, lse_out=lse, err=err)
    # the split path: bounds alone, then choice and attention in one launch -- same pages,
    # same outputs
    ub2 = kvd.quest_page_bounds(q, kmin, kmax, bt, sl, x.page_size, err=err)
    lse2 = torch.empty(x.B, x.Hq, device=DEV)
    out2, sel2 = kvd.attn_decode_quest_from_bounds(q, kp, vp, bt, sl, ub2, n_sel, scale=x.scale,
                                                   lse_out=lse2, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(sel2, sel) and torch.equal(out2, out) and torch.equal(lse2, lse)
    assert torch.equal(torch.isnan(ub2), torch.isnan(ub)) and \
        torch.equal(torch.nan_to_num(ub2), torch.nan_to_num(ub))
    return kmin.cpu(), kmax.cpu(), sel.cpu().numpy(), ub.cpu().double().numpy(), out, lse


def _bound_tol(x):
    # sum over d of |q_d| max(|kmin_d|, |kmax_d|) bounds the terms of every page's bound
    q = x.q.double().abs().numpy()
    kabs = x.k_pool.double().abs().amax(2).numpy()       # [pages, Hkv, D] >= |kmin|, |kmax|
    G = x.Hq // x.Hkv
    worst = np.einsum("bhd,phd->bhp", q, kabs[:, np.arange(x.Hq) // G]).max()
    return 2.0 ** -20 * worst + 1e-30


def _attend_chosen(x, pairs, chosen):
    """The oracle's plain attention of query head h of sequence b over the given logical
    pages plus the tail past the last full page: the same cache read through a block table
    that lists only those pages (softmax over a set does not depend on the order)."""
    P = x.page_size
    rows, lens = [], []
    for (b, h), pages in zip(pairs, chosen):
        L = int(x.seq_lens[b])
        full, tail = L // P, L % P
        row = [int(x.block_table[b, pg]) for pg in pages]
        if tail:
            row.append(int(x.block_table[b, full]))
        rows.append(row)
        lens.append(len(pages) * P + tail)
    width = max(len(r) for r in rows)
    bt = torch.zeros(len(rows), width, dtype=torch.int32)
    for i, r in enumerate(rows):
        bt[i, :len(r)] = torch.tensor(r, dtype=torch.int32)
    q = x.q[[b for b, _ in pairs]]
    sub = [(i, h) for i, (_, h) in enumerate(pairs)]
    return oracle.gqa(q, x.k_pool, x.v_pool, bt, torch.tensor(lens, dtype=torch.int32),
                      x.scale, pairs=sub)


def _verify(x, n_sel, tol, pairs, sel, out, lse, ref_out, ref_lse, ref_sel, ref_ub):
    """Every listed (sequence, head): the GPU's pages equal the oracle's, or differ only
    across a near-tie of the n_sel-th bound (the same count, no page twice, every chosen
    page's oracle bound within 2 tol of the n_sel-th); the output is held to the attention
    bar against the oracle's Quest output, or, where the choice differs, against the
    oracle's attention over the GPU's (validated) pages."""
    same, differ = [], []
    for i, (b, h) in enumerate(pairs):
        if np.array_equal(sel[b, h], ref_sel[i]):
            same.append(i)
            continue
        full = int(x.seq_lens[b]) // x.page_size
        got = sel[b, h][sel[b, h] >= 0]
        assert full > 0, (b, h, got)  # no full page: nothing to choose, both lists empty
        u = ref_ub[i, :full]
        kth = np.sort(u)[::-1][min(n_sel, full) - 1]
        assert len(got) == min(n_sel, full) and len(set(got.tolist())) == len(got), (b, h)
        assert (got < full).all() and (u[got] >= kth - 2 * tol).all(), (b, h)
        assert np.array_equal(np.sort(got), got), (b, h)
        differ.append(i)
    out_np = out.cpu()
    lse_np = lse.cpu().double().numpy()
    if same:
        idx = np.array(same)
        bi, hi = np.array(pairs)[idx].T
        assert_attn_close(out_np[bi, hi], ref_out[idx], what="quest, the oracle's pages")
        assert np.abs(lse_np[bi, hi] - ref_lse[idx]).max() < 2e-3
    if differ:
        dp = [tuple(pairs[i]) for i in differ]
        chosen = [sel[b, h][sel[b, h] >= 0].tolist() for b, h in dp]
        r_out, r_lse = _attend_chosen(x, dp, chosen)
        bi, hi = np.array(dp).T
        assert_attn_close(out_np[bi, hi], r_out, what="quest, near-tie pages")
        assert np.abs(lse_np[bi, hi] - r_lse).max() < 2e-3
    return len(same), len(differ)


def _check(kvd, x, n_sel):
    kmin, kmax, sel, ub, out, lse = _gpu(kvd, x, n_sel)
    rmin, rmax = oracle.quest_minmax(x.k_pool)
    assert np.array_equal(kmin.double().numpy(), rmin) and np.array_equal(kmax.double().numpy(), rmax)
    ref, ref_lse, ref_sel, ref_ub = oracle.quest(x.q, x.k_pool, x.v_pool, x.block_table,
                                                 x.seq_lens, x.scale, n_sel)
    tol = _bound_tol(x)
    finite = ~np.isnan(ref_ub)
    assert np.array_equal(np.isnan(ub), ~finite)
    assert np.abs(ub[finite] - ref_ub[finite]).max(initial=0.0) <= tol
    pairs = [(b, h) for b in range(x.B) for h in range(x.Hq)]
    flat = lambda a: a.reshape(x.B * x.Hq, *a.shape[2:])
    _verify(x, n_sel, tol, pairs, sel, out, lse, flat(ref), flat(ref_lse), flat(ref_sel),
            flat(ref_ub))


@pytest.mark.parametrize("D,P,n_sel", [(128, 16, 16), (64, 16, 4), (128, 32, 1), (64, 8, 64)])
def test_quest_bf16(kvd, D, P, n_sel):
    lens = [1, 7, P, P + 1, 5 * P, 300, 1000, 2047]
    x = W.make_gqa(len(lens), 16, 4, D, lens, page_size=P, shuffle=True, extra_pages=4,
                   seed=9000 + D + P + n_sel)
    _check(kvd, x, n_sel)


@pytest.mark.parametrize("n_sel", [16, 64])
def test_quest_choice_both_paths(kvd, n_sel):
    # heads with at most 512 full pages choose with their keys in registers, longer ones with
    # the keys in shared memory: lengths on both sides of 512 pages of 16 tokens
    lens = [16 * 512, 16 * 512 + 15, 16 * 513, 9000, 300]
    x = W.make_gqa(len(lens), 8, 2, 64, lens, page_size=16, shuffle=True, extra_pages=3,
                   seed=9200 + n_sel)
    _check(kvd, x, n_sel)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (16, 2), (32, 2), (12, 4)])
def test_quest_group_sizes(kvd, hq, hkv):
    # every bound-kernel width (group sizes 1, 2, 8, 16 and a padded 3)
    lens = [40, 500, 1111]
    x = W.make_gqa(3, hq, hkv, 128, lens, page_size=16, shuffle=True, extra_pages=2,
                   seed=9050 + hq + hkv)
    _check(kvd, x, 8)


def test_quest_fp32(kvd):
    lens = [5, 64, 333]
    x = W.make_gqa(3, 8, 2, 64, lens, page_size=16, shuffle=True, seed=9100,
                   dtype=torch.float32)
    _check(kvd, x, 6)


def test_quest_every_page_is_dense(kvd):
    lens = [100, 64, 1000]
    x = W.make_gqa(3, 32, 8, 128, lens, page_size=16, shuffle=True, seed=9200)
    _, _, _, _, out, _ = _gpu(kvd, x, 64)
    ref, _ = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale)
    assert_attn_close(out, ref, what="all pages (at most 64 full pages)")


def test_quest_full_size_sampled(kvd):
    x = W.build("quest_llama3")
    n_sel = W.WORKLOADS["quest_llama3"].params["n_sel"]
    kmin, kmax, sel, ub, out, lse = _gpu(kvd, x, n_sel)
    pairs = [(b, h) for b in (0, 13, 31) for h in (0, 5, 31)]
    ref, ref_lse, ref_sel, ref_ub = oracle.quest(x.q, x.k_pool, x.v_pool, x.block_table,
                                                 x.seq_lens, x.scale, n_sel, pairs=pairs)
    tol = _bound_tol(x)
    for i, (b, h) in enumerate(pairs):
        full = int(x.seq_lens[b]) // x.page_size
        assert np.abs(ub[b, h, :full] - ref_ub[i, :full]).max() <= tol
    n_same, n_differ = _verify(x, n_sel, tol, pairs, sel, out, lse, ref, ref_lse, ref_sel,
                               ref_ub)
    assert n_same + n_differ == len(pairs)


def test_quest_summaries_of_listed_pages_only(kvd):
    x = W.make_gqa(2, 8, 2, 64, [64, 64], page_size=16, seed=9300)
    kp = x.k_pool.to(DEV)
    kmin = torch.full((x.num_pages, 2, 64), 5.0, dtype=torch.bfloat16, device=DEV)
    kmax = kmin.clone()
    pages = torch.tensor([1, 6], dtype=torch.int32, device=DEV)
    _, _, err = kvd.quest_page_minmax(kp, kmin, kmax, pages=pages)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rmin, rmax = oracle.quest_minmax(x.k_pool, [1, 6])
    got = kmin.cpu().double().numpy()
    assert np.array_equal(got[[1, 6]], rmin)
    assert (got[[0, 2, 3, 4, 5, 7]] == 5.0).all()


def test_quest_bad_selection_entry_is_flagged(kvd):
    x = W.make_gqa(1, 4, 1, 64, [64], page_size=16, seed=9400)
    sel = torch.tensor([[[0, 9], [1, 2], [0, 3], [2, 3]]], dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kvd.attn_decode_quest(x.q.to(DEV), x.k_pool.to(DEV), x.v_pool.to(DEV),
                          x.block_table.to(DEV), x.seq_lens.to(DEV), sel, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == -6
