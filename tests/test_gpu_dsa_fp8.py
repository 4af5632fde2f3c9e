"""GPU parity of the FP8 lightning indexer, the e4m3 row quantizer and the indexer cache
append against the fp64 oracle.

* Quantizer and cache append: codes and scales bit-exact (both sides divide in float32 and
  round to the nearest e4m3 code, ties to even).
* Indexer scores (fp32 accumulation of exact e4m3 products on the GPU) against the oracle's
  fp64 scores on the same codes and scales: max error <= 1e-4 of the largest |score| + 1e-3.
* Selection: as for the bf16 indexer, the oracle's top-k on its own scores rounded to
  float32; any index in the symmetric difference must be a near-tie of the k-th score.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.test_gpu_dsa import _check_selection

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvd():
    import kv_cache_decode_split_gb300 as m
    return m


def _run(kvd, x, k, workspace=None):
    # table slots past a sequence's last page hold -1; the indexer reads some of them ahead of
    # the length and must neither use nor report them
    dev = "cuda"
    ws = kvd.Workspace(dev) if workspace is None else workspace
    scores = torch.full((x.B, x.max_pages * x.page_size), float("nan"), device=dev)
    idx, cnt = kvd.dsa_indexer_topk_fp8(x.q8.to(dev), x.q_scale.to(dev), x.k8_pool.to(dev),
                                        x.k_scale.to(dev), x.w.to(dev), x.block_table.to(dev),
                                        x.seq_lens.to(dev), k=k, scores_out=scores,
                                        workspace=ws)
    torch.cuda.synchronize()
    assert kvd.kvd_check_device_error(ws) == 0
    return idx, cnt, scores


def _ref(x, batches=None):
    return oracle.indexer_scores_fp8(x.q8.numpy(), x.q_scale.numpy(), x.k8_pool.numpy(),
                                     x.k_scale.numpy(), x.w, x.block_table, x.seq_lens,
                                     batches=batches)


def _check_scores(got, ref, L):
    err = np.abs(got[:L] - ref[:L])
    assert err.max() <= 1e-4 * np.abs(ref[:L]).max() + 1e-3, err.max()


@pytest.mark.parametrize("P", [64, 16, 128])
@pytest.mark.parametrize("k", [1, 16, 300])
def test_fp8_indexer_scores_and_topk_small(kvd, P, k):
    lens = [700, 3000, 1, 129]
    x = W.make_indexer_fp8(len(lens), lens, k=k, page_size=P, shuffle=True, extra_pages=2,
                           seed=980 + P + k)
    idx, cnt, scores = _run(kvd, x, k)
    ref = _ref(x)
    sc = scores.cpu().double().numpy()
    for b, L in enumerate(lens):
        _check_scores(sc[b], ref[b], L)
        _check_selection(idx[b], cnt[b], ref[b], L, k)


def test_fp8_indexer_full_size_sampled(kvd):
    x, _ = W.build("dsa_fp8_sparse_mla")
    idx, cnt, scores = _run(kvd, x, x.k)
    ref = _ref(x, batches=[0, 3])
    sc = scores.cpu().double().numpy()
    for r, b in enumerate([0, 3]):
        L = int(x.seq_lens[b])
        _check_scores(sc[b], ref[r], L)
        _check_selection(idx[b], cnt[b], ref[r], L, x.k)


def test_fp8_indexer_shares_workspace_with_bf16_indexer(kvd):
    # both precisions are one workspace family: alternating calls stay exact
    ws = kvd.Workspace(torch.device("cuda"))
    lens = [5000, 2500]
    x8 = W.make_indexer_fp8(2, lens, k=256, seed=990)
    xb = W.make_indexer(2, lens, k=256, seed=991)
    for _ in range(2):
        idx, cnt, scores = _run(kvd, x8, 256, workspace=ws)
        ref = _ref(x8)
        for b, L in enumerate(lens):
            _check_selection(idx[b], cnt[b], ref[b], L, 256)
        idxb, cntb = kvd.dsa_indexer_topk(xb.q.cuda(), xb.k_pool.cuda(), xb.w.cuda(),
                                          xb.block_table.cuda(), xb.seq_lens.cuda(), k=256,
                                          workspace=ws)
        refb = oracle.indexer_scores(xb.q, xb.k_pool, xb.w, xb.block_table, xb.seq_lens)
        for b, L in enumerate(lens):
            _check_selection(idxb[b], cntb[b], refb[b], L, 256)


@pytest.mark.parametrize("shape", [(64, 128), (3, 1000), (5, 7)])
def test_quantize_rows_bit_exact(kvd, shape):
    x = W.normal(shape, 992 + shape[1], 3.0)
    x[0] = 0  # a row of zeros: scale 1, codes 0
    x[-1, 0] = 1e4  # a large value next to small ones
    codes, scales = kvd.quantize_e4m3_rows(x.cuda())
    torch.cuda.synchronize()
    rc, rs = oracle.quantize_e4m3_rows(x)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


@pytest.mark.parametrize("P", [64, 16])
def test_cache_append_writes_the_newest_row_only(kvd, P):
    lens = [1, 64, 65, 300, 4096]
    x = W.make_indexer_fp8(len(lens), lens, page_size=P, shuffle=True, extra_pages=3, seed=995)
    k_new = W.normal((len(lens), 128), 996, 2.0)
    pool = x.k8_pool.clone().cuda()
    ks = x.k_scale.clone().cuda()
    err = kvd.dsa_indexer_cache_append_fp8(k_new.cuda(), x.block_table.cuda(),
                                           x.seq_lens.cuda(), pool, ks)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rc, rs = oracle.quantize_e4m3_rows(k_new)
    exp_pool = x.k8_pool.clone().numpy()
    exp_ks = x.k_scale.clone().numpy()
    bt = x.block_table.numpy()
    for b, L in enumerate(lens):
        t = L - 1
        pg, sl = bt[b, t // P], t % P
        exp_pool[pg, sl] = rc[b]
        exp_ks[pg, sl] = rs[b]
    assert np.array_equal(pool.cpu().numpy(), exp_pool)
    assert np.array_equal(ks.cpu().numpy(), exp_ks)


def test_cache_append_then_indexer_sees_the_new_token(kvd):
    # the appended token is scored like every other: the GPU indexer on the GPU-updated cache
    # matches the oracle on the cache updated by the oracle's quantizer
    lens = [2000, 777]
    P = 64
    x = W.make_indexer_fp8(2, lens, page_size=P, seed=997)
    k_new = W.normal((2, 128), 998, 1.0)
    pool, ks = x.k8_pool.clone().cuda(), x.k_scale.clone().cuda()
    kvd.dsa_indexer_cache_append_fp8(k_new.cuda(), x.block_table.cuda(), x.seq_lens.cuda(),
                                     pool, ks)
    rc, rs = oracle.quantize_e4m3_rows(k_new)
    exp_pool, exp_ks = x.k8_pool.clone(), x.k_scale.clone()
    bt = x.block_table.numpy()
    for b, L in enumerate(lens):
        t = L - 1
        exp_pool[bt[b, t // P], t % P] = torch.from_numpy(rc[b])
        exp_ks[bt[b, t // P], t % P] = float(rs[b])
    dev = "cuda"
    scores = torch.full((x.B, x.max_pages * P), float("nan"), device=dev)
    idx, cnt = kvd.dsa_indexer_topk_fp8(x.q8.to(dev), x.q_scale.to(dev), pool, ks, x.w.to(dev),
                                        x.block_table.to(dev), x.seq_lens.to(dev), k=64,
                                        scores_out=scores)
    torch.cuda.synchronize()
    ref = oracle.indexer_scores_fp8(x.q8.numpy(), x.q_scale.numpy(), exp_pool.numpy(),
                                    exp_ks.numpy(), x.w, x.block_table, x.seq_lens)
    sc = scores.cpu().double().numpy()
    for b, L in enumerate(lens):
        _check_scores(sc[b], ref[b], L)
        _check_selection(idx[b], cnt[b], ref[b], L, 64)
