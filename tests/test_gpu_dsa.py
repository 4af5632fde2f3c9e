"""GPU parity of the DSA indexer and top-k selection against the fp64 oracle.

* Indexer scores (fp32 on the GPU) are compared with the oracle's fp64 scores.
* The selection step alone (dsa_topk) is bit-exact against the oracle's top-k on the same
  seeded float32 score arrays, including arrays full of exact ties (lower position wins).
* The full path (dsa_indexer_topk) is compared with the oracle's selection taken on its
  own scores rounded to float32: any index in the symmetric difference must score within
  1e-5 relative of the oracle's k-th score (a near-tie), and the sets have equal size.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.parity import assert_attn_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvd():
    import kv_cache_decode_split_gb300 as m
    return m


def _check_selection(idx, cnt, ref_scores, L, k):
    """GPU selection (ascending, -1 padded) vs the oracle's on fp32-rounded fp64 scores."""
    idx = idx.cpu().numpy()
    n = min(k, L)
    assert int(cnt) == n
    sel = idx[:n]
    assert np.all(np.diff(sel) > 0), "not strictly ascending"
    assert np.all(idx[n:] == -1)
    assert sel.min() >= 0 and sel.max() < L
    s32 = ref_scores[:L].astype(np.float32).astype(np.float64)
    ref = oracle.topk(s32, k)
    diff = np.setxor1d(sel, ref)
    if diff.size:
        kth = np.sort(s32)[::-1][n - 1]
        tol = 1e-5 * abs(kth)
        assert np.all(np.abs(ref_scores[diff] - kth) <= tol), (diff, ref_scores[diff], kth)


def _run_indexer(kvd, x, k):
    # table slots past a sequence's last page hold -1; the indexer reads some of them ahead of
    # the length and must neither use nor report them
    dev = "cuda"
    ws = kvd.Workspace(dev)
    scores = torch.full((x.B, x.max_pages * x.page_size), float("nan"), device=dev)
    idx, cnt = kvd.dsa_indexer_topk(x.q.to(dev), x.k_pool.to(dev), x.w.to(dev),
                                    x.block_table.to(dev), x.seq_lens.to(dev), k=k,
                                    scores_out=scores, workspace=ws)
    torch.cuda.synchronize()
    assert kvd.kvd_check_device_error(ws) == 0
    return idx, cnt, scores


@pytest.mark.parametrize("P", [64, 16, 128])
@pytest.mark.parametrize("k", [1, 16, 300])
def test_indexer_scores_and_topk_small(kvd, P, k):
    lens = [1, 100, 129, 1000, 2500]
    x = W.make_indexer(len(lens), lens, k=k, page_size=P, shuffle=True, extra_pages=3,
                       seed=500 + P + k)
    idx, cnt, scores = _run_indexer(kvd, x, k)
    ref = oracle.indexer_scores(x.q, x.k_pool, x.w, x.block_table, x.seq_lens)
    sc = scores.cpu().double().numpy()
    for b, L in enumerate(lens):
        err = np.abs(sc[b, :L] - ref[b, :L])
        assert err.max() <= 1e-4 * np.abs(ref[b, :L]).max() + 1e-3, err.max()
        _check_selection(idx[b], cnt[b], ref[b], L, k)


def test_indexer_without_scores_out(kvd):
    x = W.make_indexer(2, [700, 3000], k=256, page_size=64, shuffle=True, seed=77)
    dev = "cuda"
    idx, cnt = kvd.dsa_indexer_topk(x.q.to(dev), x.k_pool.to(dev), x.w.to(dev),
                                    x.block_table.to(dev), x.seq_lens.to(dev), k=256)
    ref = oracle.indexer_scores(x.q, x.k_pool, x.w, x.block_table, x.seq_lens)
    for b, L in enumerate([700, 3000]):
        _check_selection(idx[b], cnt[b], ref[b], L, 256)


@pytest.mark.parametrize("case", ["normal", "ties", "all_equal", "few_values", "k_ge_L"])
def test_topk_alone_bit_exact(kvd, case):
    B, stride = 3, 20000
    lens = torch.tensor([20000, 7777, 3], dtype=torch.int32)
    if case == "normal":
        s = W.normal((B, stride), 900, 1.0, torch.float32)
    elif case == "ties":
        s = torch.randint(-50, 50, (B, stride), generator=torch.Generator().manual_seed(901)).float()
    elif case == "all_equal":
        s = torch.full((B, stride), 2.5)
    elif case == "few_values":
        s = torch.randint(0, 3, (B, stride), generator=torch.Generator().manual_seed(902)).float()
    else:
        s = W.normal((B, stride), 903, 1.0, torch.float32)
    k = 50000 if case == "k_ge_L" else 2048
    k = min(k, 4096)
    if case == "k_ge_L":
        lens = torch.tensor([4000, 10, 1], dtype=torch.int32)
    idx, cnt = kvd.dsa_topk(s.cuda(), lens.cuda(), k=k)
    torch.cuda.synchronize()
    for b in range(B):
        L = int(lens[b])
        ref = oracle.topk(s[b, :L].numpy().astype(np.float64), k)
        n = min(k, L)
        assert int(cnt[b]) == n
        got = idx[b].cpu().numpy()
        assert np.array_equal(got[:n], ref), (case, b)
        assert np.all(got[n:] == -1)


@pytest.mark.parametrize("case", ["normal", "ties"])
def test_topk_long_sequences(kvd, case):
    # past 262,144 tokens the chosen-position bitmap lives in the workspace, not in shared
    # memory; a second call checks that the first left it clear
    B, stride = 2, 300000
    lens = torch.tensor([300000, 270001], dtype=torch.int32)
    if case == "normal":
        s = W.normal((B, stride), 905, 1.0, torch.float32)
    else:
        s = torch.randint(-30, 30, (B, stride), generator=torch.Generator().manual_seed(906)).float()
    ws = kvd.Workspace(torch.device("cuda"))
    for _ in range(2):
        idx, cnt = kvd.dsa_topk(s.cuda(), lens.cuda(), k=2048, workspace=ws)
        torch.cuda.synchronize()
        for b in range(B):
            L = int(lens[b])
            ref = oracle.topk(s[b, :L].numpy().astype(np.float64), 2048)
            assert int(cnt[b]) == 2048
            assert np.array_equal(idx[b].cpu().numpy(), ref), (case, b)


def test_topk_repeat_calls(kvd):
    s = W.normal((2, 50000), 904, 1.0, torch.float32).cuda()
    lens = torch.tensor([50000, 40000], dtype=torch.int32).cuda()
    a, _ = kvd.dsa_topk(s, lens, k=2048)
    b, _ = kvd.dsa_topk(s, lens, k=2048)
    assert torch.equal(a, b)


def test_dsa_full_size_indexer_sampled(kvd):
    idx_in, _ = W.build("dsa_sparse_mla")
    x = idx_in
    idx, cnt, scores = _run_indexer(kvd, x, x.k)
    ref = oracle.indexer_scores(x.q, x.k_pool, x.w, x.block_table, x.seq_lens, batches=[0, 3])
    sc = scores.cpu().double().numpy()
    for r, b in enumerate([0, 3]):
        L = int(x.seq_lens[b])
        err = np.abs(sc[b, :L] - ref[r, :L])
        assert err.max() <= 1e-4 * np.abs(ref[r, :L]).max() + 1e-3, err.max()
        _check_selection(idx[b], cnt[b], ref[r], L, x.k)


def test_workspace_shared_with_mla(kvd):
    # one Workspace object handed first to the MLA decode (which leaves its partials in the
    # buffer) and then to the selection: the binding zero-fills it on the change of family
    ws = kvd.Workspace("cuda")
    xm = W.make_mla(2, 128, [300, 2000], page_size=64, seed=905)
    kvd.attn_decode_mla(xm.q.cuda(), xm.c_pool.cuda(), xm.block_table.cuda(),
                        xm.seq_lens.cuda(), scale=xm.scale, workspace=ws)
    s = W.normal((2, 20000), 906, 1.0, torch.float32)
    lens = torch.tensor([20000, 9000], dtype=torch.int32)
    idx, cnt = kvd.dsa_topk(s.cuda(), lens.cuda(), k=2048, workspace=ws)
    assert kvd.kvd_check_device_error(ws) == 0
    for b in range(2):
        L = int(lens[b])
        ref = oracle.topk(s[b, :L].numpy().astype(np.float64), 2048)
        assert np.array_equal(idx[b].cpu().numpy(), ref)


def test_topk_non_zeroed_workspace_is_reported(kvd):
    # a raw workspace whose counters and histograms hold another kernel's data: the
    # selection stays inside its buffers, records KVD_ERR_DEVICE_STATE and leaves its
    # state zeroed, so that the next call is exact again
    B, k = 2, 256
    s = W.normal((B, 3000), 907, 1.0, torch.float32)
    lens = torch.tensor([3000, 2000], dtype=torch.int32)
    nbytes = kvd.kvd_workspace_size("dsa_topk", B, 1, max_len=3000, k=k)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")
    ws[:256] = 0  # the error flag starts clear
    kvd.dsa_topk(s.cuda(), lens.cuda(), k=k, workspace=ws)
    assert kvd.kvd_check_device_error(ws) == -7
    idx, cnt = kvd.dsa_topk(s.cuda(), lens.cuda(), k=k, workspace=ws)
    assert kvd.kvd_check_device_error(ws) == 0
    for b in range(B):
        L = int(lens[b])
        ref = oracle.topk(s[b, :L].numpy().astype(np.float64), k)
        assert np.array_equal(idx[b].cpu().numpy(), ref)


def test_workspace_reused_across_shapes(kvd):
    # one workspace, large from the start, serving selections of other batch sizes, lengths
    # and k in turn: the layout moves with them, so stale lists from one call must not be
    # read as the next call's zeroed histogram
    ws = kvd.Workspace(torch.device("cuda"))
    ws.get(64 << 20)
    for B, L, k in [(2, 50000, 2048), (4, 20000, 300), (3, 7000, 2048), (4, 20000, 300)]:
        s = W.normal((B, L), 999 + B + k, 1.0, torch.float32)
        lens = torch.full((B,), L, dtype=torch.int32)
        idx, cnt = kvd.dsa_topk(s.cuda(), lens.cuda(), k=k, workspace=ws)
        torch.cuda.synchronize()
        for b in range(B):
            ref = oracle.topk(s[b].numpy().astype(np.float64), k)
            assert int(cnt[b]) == min(k, L)
            assert np.array_equal(idx[b].cpu().numpy()[:len(ref)], ref), (B, L, k, b)
        assert kvd.kvd_check_device_error(ws) == 0


def _chain(kvd, xi, xm, batches, n_pairs, seed):
    """The DSA step as one pipeline ("Attention Optimizations", DSA / Computation Path:
    indexer scores, top-k, then attention over the selected cache rows): the indexer's own
    output (ascending positions, -1 padded, count) goes straight into the sparse MLA. The
    oracle runs the same chain: its fp64 scores, its top-k on them rounded to float32, its
    MLA over that selection. Where the GPU's selection differs only by near-ties (checked
    first), the output is compared with the oracle's MLA over the GPU's selection."""
    dev = "cuda"
    bt, sl = xm.block_table.to(dev), xm.seq_lens.to(dev)
    ws_i, ws_m = kvd.Workspace(dev), kvd.Workspace(dev)
    idx, cnt = kvd.dsa_indexer_topk(xi.q.to(dev), xi.k_pool.to(dev), xi.w.to(dev), bt, sl,
                                    k=xi.k, workspace=ws_i)
    lse = torch.empty(xm.B, xm.H, dtype=torch.float32, device=dev)
    out = kvd.attn_decode_mla_sparse(xm.q.to(dev), xm.c_pool.to(dev), bt, sl, idx, cnt,
                                     scale=xm.scale, lse_out=lse, workspace=ws_m)
    torch.cuda.synchronize()
    assert kvd.kvd_check_device_error(ws_i) == 0 and kvd.kvd_check_device_error(ws_m) == 0
    scores = oracle.indexer_scores(xi.q, xi.k_pool, xi.w, xi.block_table, xi.seq_lens,
                                   batches=batches)
    idx_h, cnt_h = idx.cpu().numpy(), cnt.cpu().numpy()
    ref_idx = np.full((xm.B, xi.k), -1, np.int32)
    ref_cnt = np.zeros(xm.B, np.int32)
    use_idx, use_cnt = ref_idx.copy(), ref_cnt.copy()
    for r, b in enumerate(batches):
        L = int(xm.seq_lens[b])
        _check_selection(idx[b], cnt[b], scores[r], L, xi.k)
        sel = oracle.topk(scores[r, :L].astype(np.float32).astype(np.float64), xi.k)
        ref_idx[b, :len(sel)], ref_cnt[b] = sel, len(sel)
        same = np.array_equal(idx_h[b], ref_idx[b])
        use_idx[b], use_cnt[b] = (ref_idx[b], ref_cnt[b]) if same else (idx_h[b], cnt_h[b])
    rng = np.random.default_rng(seed)
    pr = np.stack([rng.choice(batches, n_pairs), rng.integers(0, xm.H, n_pairs)], 1)
    pr = pr.astype(np.int32)
    ref, ref_lse = oracle.mla(xm.q, xm.c_pool, xm.block_table, xm.seq_lens, xm.scale,
                              idx=use_idx, idx_count=use_cnt, pairs=pr)
    assert_attn_close(out[pr[:, 0], pr[:, 1]], ref, what="indexer -> top-k -> sparse MLA")
    got_lse = lse.cpu().double().numpy()[pr[:, 0], pr[:, 1]]
    assert np.max(np.abs(got_lse - ref_lse)) < 2e-3 * max(1.0, np.abs(ref_lse).max())


def test_dsa_chain_ragged(kvd):
    # sequences shorter than k (every token kept, count < k, -1 padding), exactly k, and
    # longer; sharp entries so that the selection decides the output
    lens = [1, 100, 2047, 2048, 2049, 30000]
    xm = W.make_mla(len(lens), 128, lens, page_size=64, shuffle=True, extra_pages=3, seed=910,
                    factor=1.0)
    xi = W.make_indexer(len(lens), lens, k=2048, page_size=64, seed=911,
                        block_table=xm.block_table)
    _chain(kvd, xi, xm, list(range(len(lens))), 96, 912)


def test_dsa_chain_full_size(kvd):
    # the DSA workload (B=4, L=131072, k=2048) in the launch configuration the bench times,
    # sampled (sequence, head) outputs of two sequences
    xi, xm = W.build("dsa_sparse_mla")
    _chain(kvd, xi, xm, [0, 2], 48, 913)
