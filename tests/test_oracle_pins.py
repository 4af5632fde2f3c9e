"""Pins for the oracle: brute force on tiny inputs, closed forms, the pages' worked
examples and the invariants the method states. CPU only.

Each test names the mistake it is there to catch.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests import bruteforce as bf


def _close(a, b, tol=1e-12):
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert err <= tol * max(1.0, float(np.max(np.abs(b))) if b.size else 1.0), err


# ----------------------------------------------------------------------------- GQA family
@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("hq,hkv", [(4, 4), (4, 2), (6, 1), (8, 2)])
def test_gqa_dense_matches_bruteforce(seed, hq, hkv):
    lens = [1 + (seed * 7 + 5 * i) % 40 for i in range(3)]
    x = W.make_gqa(3, hq, hkv, 16, lens, page_size=8, shuffle=True, extra_pages=3, seed=seed,
                   dtype=torch.float32)
    o, l = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale)
    ob, lb = bf.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale)
    _close(o, ob)
    _close(l, lb)


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("window,n_sink,learned", [(5, 0, False), (5, 2, False), (9, 4, False),
                                                   (3, 0, True), (6, 3, True), (50, 2, False),
                                                   (1, 0, False), (1, 1, True)])
def test_swa_sink_matches_bruteforce(seed, window, n_sink, learned):
    lens = [1, 4, 7, 23]
    x = W.make_gqa(4, 4, 2, 8, lens, page_size=4, shuffle=True, seed=10 + seed, window=window,
                   n_sink=n_sink, learned_sink=learned, dtype=torch.float32)
    o, l = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale, x.window,
                      x.n_sink, x.sink_logit)
    ob, lb = bf.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale, x.window,
                    x.n_sink, x.sink_logit)
    _close(o, ob)
    _close(l, lb)


def test_bf16_inputs_are_widened_exactly():
    # catches: reading bf16 bits as something else, or rounding the inputs again
    x = W.make_gqa(2, 4, 2, 16, [9, 13], page_size=4, seed=3)
    o, _ = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale)
    ob, _ = bf.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale)
    _close(o, ob)


def test_single_token_returns_its_value():
    # closed form: L = 1 => o = v_0, lse = scale * q.k_0
    x = W.make_gqa(2, 4, 2, 8, [1, 1], page_size=4, seed=1, dtype=torch.float32)
    o, l = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale)
    for b in range(2):
        page = int(x.block_table[b, 0])
        for h in range(4):
            g = h // 2
            _close(o[b, h], x.v_pool[page, g, 0].double().numpy())
            _close(l[b, h], x.scale * float((x.q[b, h].double() * x.k_pool[page, g, 0].double()).sum()))


def test_zero_query_averages_visible_values():
    # closed form: q = 0 => uniform weights => mean of the visible values
    x = W.make_gqa(1, 2, 1, 4, [11], page_size=4, seed=2, dtype=torch.float32, window=5, n_sink=2)
    x.q.zero_()
    o, l = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale, x.window,
                      x.n_sink)
    vis = [0, 1, 6, 7, 8, 9, 10]
    V = bf.gather_tokens(x.v_pool, x.block_table, 0, 11, 4, 0)
    _close(o[0, 0], V[vis].mean(axis=0))
    _close(l[0, 0], math.log(len(vis)))


def test_two_token_closed_form_scale_and_sign():
    # hand-worked: D=4, scale=1/2, q=(2,0,0,0), k0=(1,0,0,0), k1=0 -> logits (1, 0),
    # p0 = e/(e+1). Catches a dropped or squared scale and a flipped sign.
    q = torch.tensor([[[2.0, 0, 0, 0]]])
    k = torch.zeros(1, 1, 2, 4)
    v = torch.zeros(1, 1, 2, 4)
    k[0, 0, 0, 0] = 1.0
    v[0, 0, 0] = torch.tensor([1.0, 2.0, 0, 0])
    v[0, 0, 1] = torch.tensor([0, 0, 4.0, 0])
    bt = torch.tensor([[0]], dtype=torch.int32)
    sl = torch.tensor([2], dtype=torch.int32)
    o, l = oracle.gqa(q, k, v, bt, sl, 0.5)
    e = math.e
    _close(o[0, 0], [e / (e + 1), 2 * e / (e + 1), 4 / (e + 1), 0.0])
    _close(l[0, 0], math.log(e + 1))
    # with a learned sink logit of 1: p = (e, 1, e) / (2e + 1) over (k0, k1, sink)
    o, l = oracle.gqa(q, k, v, bt, sl, 0.5, sink_logit=np.array([1.0], np.float32))
    _close(o[0, 0], [e / (2 * e + 1), 2 * e / (2 * e + 1), 4 / (2 * e + 1), 0.0])
    _close(l[0, 0], math.log(2 * e + 1))


def test_sliding_window_worked_example(golden_dir):
    # the page's example: T=6, W=3, token 3 sees {1,2,3}. With q=0 and one-hot values,
    # o equals the indicator of the visible set divided by its size.
    ex = json.load(open(os.path.join(golden_dir, "swa_mask_example.json")))
    T, Wn, i = ex["T"], ex["W"], ex["query"]
    L = i + 1
    D = T
    q = torch.zeros(1, 1, D)
    k = torch.zeros(1, 1, T, D)
    v = torch.eye(T, D).reshape(1, 1, T, D)
    bt = torch.tensor([[0]], dtype=torch.int32)
    o, _ = oracle.gqa(q, k, v, bt, torch.tensor([L], dtype=torch.int32), 1.0, window=Wn)
    expect = np.zeros(D)
    expect[ex["visible"]] = 1.0 / len(ex["visible"])
    _close(o[0, 0], expect)


def test_gqa_head_mapping_equals_repeated_mha():
    # invariant: GQA equals MHA over K/V repeated per group (repeat_kv order: head h uses
    # KV head h // n_rep). Catches h % Hkv and other index slips.
    x = W.make_gqa(2, 8, 2, 8, [13, 30], page_size=4, seed=5, dtype=torch.float32)
    o, l = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale)
    k_rep = x.k_pool.repeat_interleave(4, dim=1)
    v_rep = x.v_pool.repeat_interleave(4, dim=1)
    om, lm = oracle.gqa(x.q, k_rep, v_rep, x.block_table, x.seq_lens, x.scale)
    _close(o, om)
    _close(l, lm)


def test_mqa_is_single_shared_head():
    x = W.make_gqa(2, 5, 1, 8, [9, 17], page_size=4, seed=6, dtype=torch.float32)
    o, _ = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale)
    for h in range(5):
        oh, _ = oracle.gqa(x.q[:, h:h + 1], x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale)
        _close(o[:, h], oh[:, 0])


def test_paging_does_not_change_output():
    # invariant (PagedAttention): permuting physical pages with the table is bit-identical
    x = W.make_gqa(3, 4, 2, 8, [5, 17, 32], page_size=4, seed=7, dtype=torch.float32)
    o, l = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale, 6, 2)
    perm = torch.randperm(x.num_pages, generator=torch.Generator().manual_seed(0))
    inv = torch.argsort(perm)
    bt2 = torch.where(x.block_table >= 0, inv[x.block_table.clamp(min=0).long()].int(),
                      x.block_table)
    o2, l2 = oracle.gqa(x.q, x.k_pool[perm], x.v_pool[perm], bt2, x.seq_lens, x.scale, 6, 2)
    assert np.array_equal(o, o2) and np.array_equal(l, l2)


def test_window_at_least_length_equals_dense():
    x = W.make_gqa(3, 4, 2, 8, [5, 17, 32], page_size=4, seed=8, dtype=torch.float32)
    od, ld = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale)
    ow, lw = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale, window=32)
    _close(od, ow)
    _close(ld, lw)


def test_no_sink_tokens_is_pure_window_and_sinks_union():
    x = W.make_gqa(1, 2, 1, 4, [20], page_size=4, seed=9, dtype=torch.float32)
    x.q.zero_()
    o0, _ = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale, 5, 0)
    V = bf.gather_tokens(x.v_pool, x.block_table, 0, 20, 4, 0)
    _close(o0[0, 0], V[15:20].mean(axis=0))
    # sinks overlapping the window are counted once
    o1, _ = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, torch.tensor([6], dtype=torch.int32),
                       x.scale, 5, 3)
    V6 = bf.gather_tokens(x.v_pool, x.block_table, 0, 6, 4, 0)
    _close(o1[0, 0], V6.mean(axis=0))


def test_sink_logit_to_minus_infinity_is_no_sink():
    x = W.make_gqa(2, 4, 2, 8, [9, 17], page_size=4, seed=11, dtype=torch.float32, window=6,
                   learned_sink=True)
    on, ln = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale, 6, 0)
    om, lm = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale, 6, 0,
                        np.full(4, -np.inf))
    _close(on, om)
    _close(ln, lm)
    o9, _ = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale, 6, 0,
                       np.full(4, -1e4))
    _close(on, o9)


def test_zero_sink_logit_equals_zero_key_zero_value_token():
    # softmax-off-by-one: a sink logit of 0 is a token whose key and value are zero
    x = W.make_gqa(1, 2, 1, 4, [7], page_size=8, seed=12, dtype=torch.float32)
    o, l = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale,
                      sink_logit=np.zeros(2))
    k2 = x.k_pool.clone()
    v2 = x.v_pool.clone()
    k2[0, 0, 7] = 0.0
    v2[0, 0, 7] = 0.0
    oz, lz = oracle.gqa(x.q, k2, v2, x.block_table, torch.tensor([8], dtype=torch.int32), x.scale)
    _close(o, oz)
    _close(l, lz)


def test_split_and_lse_combine_is_exact():
    # the combine rule the GPU uses: o = sum_i e^{lse_i - M} o_i / sum_i e^{lse_i - M}.
    # Splitting the visible set with the sparse-MLA oracle and recombining equals the whole.
    x = W.make_mla(1, 3, [40], d_qk=16, d_v=8, page_size=8, seed=13, factor=1.0, scale=0.3)
    od, ld = oracle.mla(x.q, x.c_pool, x.block_table, x.seq_lens, x.scale, d_v=8)
    rng = np.random.default_rng(0)
    perm = rng.permutation(40)
    parts = [np.sort(perm[:7]), np.sort(perm[7:25]), np.sort(perm[25:])]
    os_, ls_ = [], []
    for p in parts:
        idx = np.full((1, 40), -1, np.int32)
        idx[0, :len(p)] = p
        o, l = oracle.mla(x.q, x.c_pool, x.block_table, x.seq_lens, x.scale, d_v=8, idx=idx,
                          idx_count=np.array([len(p)], np.int32))
        os_.append(o)
        ls_.append(l)
    L = np.stack(ls_)                      # [3, 1, H]
    M = L.max(axis=0)
    wgt = np.exp(L - M)
    comb = (wgt[..., None] * np.stack(os_)).sum(axis=0) / wgt.sum(axis=0)[..., None]
    _close(comb, od, 1e-13)
    _close(M + np.log(wgt.sum(axis=0)), ld, 1e-13)


# ----------------------------------------------------------------------------- MLA
@pytest.mark.parametrize("seed", range(4))
def test_mla_matches_bruteforce(seed):
    x = W.make_mla(2, 4, [9, 30], d_qk=24, d_v=16, page_size=8, shuffle=True, extra_pages=2,
                   seed=20 + seed, factor=1.0, scale=0.25)
    o, l = oracle.mla(x.q, x.c_pool, x.block_table, x.seq_lens, x.scale, d_v=16)
    ob, lb = bf.mla(x.q, x.c_pool, x.block_table, x.seq_lens, x.scale, d_v=16)
    _close(o, ob)
    _close(l, lb)


def test_mla_absorbed_equals_explicit_up_projection():
    # invariant: caching c_t and folding W_UK into the query / W_UV into the output equals
    # attention over the explicit per-head keys [W_UK c_t ; k^R_t] and values W_UV c_t
    # ("Overview of Attention Mechanism", MLA / Decoupled Position Embedding; "Attention
    # Optimizations", DSA / Computation Path). Both forms are stored in float32, so they agree
    # to float32 storage rounding; a wrong value slice, a dropped RoPE part or a missing
    # scale differs at O(1).
    rng = np.random.default_rng(1)
    H, dl, dr, dn, dv, L = 4, 32, 8, 16, 12, 21
    c = rng.standard_normal((L, dl))
    kr = rng.standard_normal((L, dr))
    W_UK = rng.standard_normal((H, dn, dl)) / math.sqrt(dl)
    W_UV = rng.standard_normal((H, dv, dl)) / math.sqrt(dl)
    q_nope = rng.standard_normal((H, dn))
    q_pe = rng.standard_normal((H, dr))
    scale = 1.0 / math.sqrt(dn + dr)
    # explicit form: an MHA problem with per-head 24-wide keys and 12-wide values
    K = np.concatenate([np.einsum("hnl,tl->htn", W_UK, c), np.repeat(kr[None], H, 0)], axis=2)
    V = np.zeros((H, L, dn + dr))
    V[..., :dv] = np.einsum("hvl,tl->htv", W_UV, c)
    Q = np.concatenate([q_nope, q_pe], axis=1)
    f32 = lambda a: torch.tensor(a, dtype=torch.float32)
    bt = torch.tensor([[0]], dtype=torch.int32)
    sl = torch.tensor([L], dtype=torch.int32)
    oe, le = oracle.gqa(f32(Q)[None], f32(K)[None], f32(V)[None], bt, sl, scale)
    # absorbed form: one shared (latent + RoPE) row per token, value = latent part
    q_abs = np.concatenate([np.einsum("hnl,hn->hl", W_UK, q_nope), q_pe], axis=1)
    rows = np.concatenate([c, kr], axis=1)
    ol, ll = oracle.mla(f32(q_abs)[None], f32(rows)[None], bt, sl, scale, d_v=dl)
    o_abs = np.einsum("hvl,hl->hv", W_UV, ol[0])
    _close(o_abs, oe[0][:, :dv], 1e-5)
    _close(ll, le, 1e-5)


def test_sparse_mla_all_tokens_equals_dense_and_order_free():
    x = W.make_mla(2, 4, [13, 29], d_qk=24, d_v=16, page_size=8, seed=30, factor=1.0, scale=0.25)
    od, ld = oracle.mla(x.q, x.c_pool, x.block_table, x.seq_lens, x.scale, d_v=16)
    idx = np.full((2, 32), -1, np.int32)
    rng = np.random.default_rng(2)
    idx[0, :13] = rng.permutation(13)
    idx[1, :29] = rng.permutation(29)
    os_, ls_ = oracle.mla(x.q, x.c_pool, x.block_table, x.seq_lens, x.scale, d_v=16, idx=idx,
                          idx_count=np.array([13, 29], np.int32))
    _close(os_, od)
    _close(ls_, ld)


@pytest.mark.parametrize("seed", range(3))
def test_sparse_mla_matches_bruteforce(seed):
    x = W.make_mla(2, 3, [20, 33], d_qk=24, d_v=16, page_size=8, shuffle=True, seed=40 + seed,
                   factor=1.0, scale=0.25)
    rng = np.random.default_rng(seed)
    idx = np.full((2, 10), -1, np.int32)
    cnt = np.array([7, 10], np.int32)
    idx[0, :7] = np.sort(rng.choice(20, 7, replace=False))
    idx[1, :10] = np.sort(rng.choice(33, 10, replace=False))
    o, l = oracle.mla(x.q, x.c_pool, x.block_table, x.seq_lens, x.scale, d_v=16, idx=idx,
                      idx_count=cnt)
    ob, lb = bf.mla(x.q, x.c_pool, x.block_table, x.seq_lens, x.scale, d_v=16, idx=idx,
                    idx_count=cnt)
    _close(o, ob)
    _close(l, lb)


# ----------------------------------------------------------------------------- indexer + top-k
def test_indexer_hand_worked(golden_dir):
    ex = json.load(open(os.path.join(golden_dir, "indexer_hand.json")))
    q = torch.tensor([ex["q"]], dtype=torch.bfloat16)
    kp = torch.tensor([ex["k"]], dtype=torch.bfloat16)               # one page of 4 tokens
    w = torch.tensor([ex["w"]], dtype=torch.float32)
    bt = torch.tensor([[0]], dtype=torch.int32)
    sl = torch.tensor([len(ex["k"])], dtype=torch.int32)
    s = oracle.indexer_scores(q, kp, w, bt, sl)
    _close(s[0], ex["expect_scores"])
    assert list(oracle.topk(s[0], ex["k_top"])) == ex["expect_topk"]


@pytest.mark.parametrize("seed", range(3))
def test_indexer_matches_bruteforce(seed):
    x = W.make_indexer(2, [37, 90], Hi=4, Di=16, k=8, page_size=8, shuffle=True, seed=50 + seed)
    s = oracle.indexer_scores(x.q, x.k_pool, x.w, x.block_table, x.seq_lens)
    for b in range(2):
        L = int(x.seq_lens[b])
        _close(s[b, :L], bf.indexer_scores(x.q, x.k_pool, x.w, x.block_table, x.seq_lens, b))
        assert np.all(np.isnan(s[b, L:]))


def test_topk_hand_built_ties(golden_dir):
    ex = json.load(open(os.path.join(golden_dir, "topk_ties.json")))
    for c in ex["cases"]:
        assert list(oracle.topk(np.array(c["scores"], np.float64), c["k"])) == c["expect"], c


@pytest.mark.parametrize("seed", range(5))
def test_topk_matches_full_sort_with_duplicates(seed):
    rng = np.random.default_rng(seed)
    s = rng.integers(-20, 20, size=300).astype(np.float64)     # many exact ties
    for k in (1, 7, 64, 299, 300, 500):
        assert list(oracle.topk(s, k)) == bf.topk_full_sort(list(s), k)


def test_topk_single_head_positive_weight_is_topk_of_dot():
    # with one head and w > 0, the ReLU only clips; the top-k of I equals the top-k of q.k
    # among positive dots (all dots here are made positive by construction)
    x = W.make_indexer(1, [200], Hi=1, Di=8, k=16, page_size=8, seed=60)
    x.w.abs_()
    x.w.add_(0.5)
    kp = x.k_pool.float()
    kp = kp * torch.sign((kp * x.q[0, 0].float()).sum(-1, keepdim=True) + 1e-9)
    x.k_pool = kp.to(torch.bfloat16)
    s = oracle.indexer_scores(x.q, x.k_pool, x.w, x.block_table, x.seq_lens)
    dots = (x.k_pool.double().reshape(-1, 8)[:200] @ x.q[0, 0].double()).numpy()
    assert np.all(dots > 0)
    assert list(oracle.topk(s[0], 16)) == bf.topk_full_sort(list(dots), 16)


# ----------------------------------------------------------------------------- FP8 indexer
def test_e4m3_decode_format_points():
    # format facts: a wrong exponent bias, subnormal rule, sign or NaN pattern fails one
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x3F: 1.875, 0x40: 2.0, 0x77: 240.0, 0x7E: 448.0, 0xFE: -448.0, 0xB8: -1.0}
    got = oracle.e4m3_decode(list(cases))
    assert list(got) == list(cases.values())
    assert np.all(np.isnan(oracle.e4m3_decode([0x7F, 0xFF])))


def test_e4m3_decode_matches_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().double().numpy()
    got = oracle.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])


def test_e4m3_encode_matches_torch_rounding():
    # nearest code, ties to the even code: a truncating or ties-away encoder fails the
    # midpoints, a wrong binade boundary fails the random values
    g = torch.Generator().manual_seed(970)
    vals = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    mids = (vals[:-1] + vals[1:]) / 2
    x = torch.cat([torch.randn(20000, generator=g) * s for s in (0.003, 1.0, 30.0, 150.0)] +
                  [torch.tensor(mids, dtype=torch.float32), -torch.tensor(mids, dtype=torch.float32)])
    x = x.clamp(-448.0, 448.0)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(x.numpy())
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturates():
    # magnitudes beyond the largest finite value clamp to it (no NaN, no wrap)
    got = oracle.e4m3_encode([448.0, 449.0, 464.0, 1e6, -500.0, np.inf, -np.inf])
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0xFE]


def test_quantize_rows_amax_lands_on_448_and_error_bound():
    x = W.normal((64, 128), 971)
    codes, s = oracle.quantize_e4m3_rows(x)
    dec = oracle.e4m3_decode(codes)
    # a scale off by a factor (or taken from the wrong row) moves the row maximum off 448
    assert np.all(np.max(np.abs(dec), axis=1) == 448.0)
    xf = x.float().numpy().astype(np.float64)
    err = np.abs(dec * s[:, None] - xf)
    # half a code step: 2^-4 relative for normals, 2^-10 of the scale below them
    bound = np.maximum(np.abs(xf) * 2.0 ** -4, s[:, None] * 2.0 ** -10)
    assert np.all(err <= bound * (1 + 1e-6))
    z, sz = oracle.quantize_e4m3_rows(torch.zeros(2, 16, dtype=torch.bfloat16))
    assert np.all(z == 0) and np.all(sz == 1.0)


def _fp8_case(seed):
    x = W.make_indexer(2, [37, 70], Hi=4, Di=32, page_size=16, shuffle=True, extra_pages=2,
                       seed=seed)
    rng = np.random.default_rng(seed)
    cq = rng.integers(0, 256, size=tuple(x.q.shape)).astype(np.uint8)
    ck = rng.integers(0, 256, size=tuple(x.k_pool.shape)).astype(np.uint8)
    cq[(cq & 0x7F) == 0x7F] = 0x38  # no NaN codes
    ck[(ck & 0x7F) == 0x7F] = 0x38
    return x, cq, ck


@pytest.mark.parametrize("seed", [972, 973])
def test_indexer_fp8_unit_scales_equals_bf16_indexer(seed):
    # every e4m3 value is a bf16 value: with unit scales the FP8 score is the (pinned) bf16
    # indexer on the decoded codes; a mis-decoded code or a wrong row mapping fails
    x, cq, ck = _fp8_case(seed)
    qb = torch.from_numpy(oracle.e4m3_decode(cq)).to(torch.bfloat16)
    kb = torch.from_numpy(oracle.e4m3_decode(ck)).to(torch.bfloat16)
    ref = oracle.indexer_scores(qb, kb, x.w, x.block_table, x.seq_lens)
    ones_q = np.ones(tuple(x.q.shape[:2]), np.float32)
    ones_k = np.ones(tuple(x.k_pool.shape[:2]), np.float32)
    got = oracle.indexer_scores_fp8(cq, ones_q, ck, ones_k, x.w, x.block_table, x.seq_lens)
    fin = ~np.isnan(ref)
    assert np.array_equal(fin, ~np.isnan(got))
    _close(got[fin], ref[fin], 1e-12)


def test_indexer_fp8_scales_factor_out():
    # ReLU is positively homogeneous: a head's scale multiplies that head's weight and a
    # token's scale multiplies its score; a scale on the wrong operand or row fails
    x, cq, ck = _fp8_case(974)
    rng = np.random.default_rng(975)
    sq = rng.uniform(0.01, 2.0, size=tuple(x.q.shape[:2])).astype(np.float32)
    sk = rng.uniform(0.01, 2.0, size=tuple(x.k_pool.shape[:2])).astype(np.float32)
    got = oracle.indexer_scores_fp8(cq, sq, ck, sk, x.w, x.block_table, x.seq_lens)
    w2 = (x.w.double() * torch.from_numpy(sq).double()).float()
    base = oracle.indexer_scores_fp8(cq, np.ones_like(sq), ck, np.ones_like(sk), w2,
                                     x.block_table, x.seq_lens)
    bt = x.block_table.numpy()
    for b, L in enumerate(x.seq_lens.tolist()):
        rows = np.array([bt[b, t // 16] * 16 + t % 16 for t in range(L)])
        ref = base[b, :L] * sk.reshape(-1)[rows].astype(np.float64)
        # the weights product w*sq is rounded to float32 on this side only
        _close(got[b, :L], ref, 1e-6)
