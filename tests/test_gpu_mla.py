"""GPU parity of attn_decode_mla / attn_decode_mla_sparse against the fp64 oracle.

Covers ragged and partial tiles, page sizes, the sharp-logit case (entries ~ N(0,1) times
a factor, so the softmax is peaked and the running max moves by more than 2^8 between
tiles), gathered (sparse) rows in any order, the full-size DeepSeek-V3-shaped decode on
sampled (sequence, head) outputs, and the invariant that selecting every token equals
the dense decode.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.parity import RTOL_STRESS, assert_attn_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvd():
    import kv_cache_decode_split_gb300 as m
    return m


# Block-table slots past a sequence's last page hold -1 in every workload: the kernels read
# some of them ahead of the length (one memory round trip less) and must neither use nor
# report them, so every call here also checks the device error flag.
def _dense(kvd, x):
    dev = "cuda"
    ws = kvd.Workspace(dev)
    lse = torch.empty(x.B, x.H, dtype=torch.float32, device=dev)
    out = kvd.attn_decode_mla(x.q.to(dev), x.c_pool.to(dev), x.block_table.to(dev),
                              x.seq_lens.to(dev), scale=x.scale, lse_out=lse, workspace=ws)
    torch.cuda.synchronize()
    assert kvd.kvd_check_device_error(ws) == 0
    return out, lse


def _sparse(kvd, x, idx, cnt):
    dev = "cuda"
    ws = kvd.Workspace(dev)
    lse = torch.empty(x.B, x.H, dtype=torch.float32, device=dev)
    out = kvd.attn_decode_mla_sparse(x.q.to(dev), x.c_pool.to(dev), x.block_table.to(dev),
                                     x.seq_lens.to(dev), torch.as_tensor(idx).to(dev),
                                     torch.as_tensor(cnt).to(dev), scale=x.scale, lse_out=lse,
                                     workspace=ws)
    torch.cuda.synchronize()
    assert kvd.kvd_check_device_error(ws) == 0
    return out, lse


@pytest.mark.parametrize("P", [64, 16])
@pytest.mark.parametrize("factor", [0.1, 1.0, 3.0])
def test_mla_dense_small(kvd, P, factor):
    lens = [1, 63, 64, 65, 700, 3000]
    x = W.make_mla(len(lens), 128, lens, page_size=P, shuffle=True, extra_pages=3,
                   seed=int(600 + P + 10 * factor), factor=factor)
    out, lse = _dense(kvd, x)
    ref, ref_lse = oracle.mla(x.q, x.c_pool, x.block_table, x.seq_lens, x.scale)
    assert_attn_close(out, ref, what=f"mla P={P} f={factor}",
                      rtol=RTOL_STRESS if factor > 1 else 0.0)
    assert np.max(np.abs(to_np(lse) - ref_lse)) < 2e-3 * max(1.0, np.abs(ref_lse).max())


def test_mla_rising_scores_rescale(kvd):
    # later tokens score much higher, so the running max climbs tile after tile
    x = W.make_mla(2, 128, [1000, 2000], page_size=64, seed=621, factor=1.0)
    ramp = torch.linspace(0.5, 3.0, x.c_pool.shape[0] * 64).reshape(-1, 64, 1)
    x.c_pool = (x.c_pool.float() * ramp).to(torch.bfloat16)
    out, _ = _dense(kvd, x)
    ref, _ = oracle.mla(x.q, x.c_pool, x.block_table, x.seq_lens, x.scale)
    assert_attn_close(out, ref, what="rising", rtol=RTOL_STRESS)


@pytest.mark.parametrize("factor", [0.1, 1.0])
def test_mla_sparse_small(kvd, factor):
    lens = [5, 300, 4000, 9000]
    k = 2048
    x = W.make_mla(len(lens), 128, lens, page_size=64, shuffle=True, seed=630, factor=factor)
    rng = np.random.default_rng(7)
    idx = np.full((len(lens), k), -1, np.int32)
    cnt = np.zeros(len(lens), np.int32)
    for b, L in enumerate(lens):
        n = min(k, L)
        sel = rng.choice(L, n, replace=False)          # any order
        idx[b, :n] = sel
        cnt[b] = n
    out, lse = _sparse(kvd, x, idx, cnt)
    ref, ref_lse = oracle.mla(x.q, x.c_pool, x.block_table, x.seq_lens, x.scale, idx=idx,
                              idx_count=cnt)
    assert_attn_close(out, ref, what="sparse")
    assert np.max(np.abs(to_np(lse) - ref_lse)) < 2e-3 * max(1.0, np.abs(ref_lse).max())


def test_mla_sparse_all_tokens_equals_dense(kvd):
    lens = [100, 1500]
    x = W.make_mla(2, 128, lens, page_size=64, shuffle=True, seed=640, factor=1.0)
    idx = np.full((2, 1500), -1, np.int32)
    rng = np.random.default_rng(1)
    for b, L in enumerate(lens):
        idx[b, :L] = rng.permutation(L)
    # both paths against the exact dense result: two bf16 approximations of it may differ
    # from each other by up to twice the tolerance (different P roundings per tile)
    ref, ref_lse = oracle.mla(x.q, x.c_pool, x.block_table, x.seq_lens, x.scale)
    dense, _ = _dense(kvd, x)
    sparse, sparse_lse = _sparse(kvd, x, idx, np.array(lens, np.int32))
    assert_attn_close(dense, ref, what="dense")
    assert_attn_close(sparse, ref, what="all-selected sparse vs dense oracle")
    assert np.max(np.abs(to_np(sparse_lse) - ref_lse)) < 2e-3 * max(1.0, np.abs(ref_lse).max())


def _pairs(B, H, n, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.integers(0, B, n), rng.integers(0, H, n)], 1).astype(np.int32)


@pytest.mark.parametrize("sharp", [False, True])
def test_mla_full_size_sampled(kvd, sharp):
    x = W.build("mla_dsv3", sharp=sharp)
    out, lse = _dense(kvd, x)
    pr = _pairs(x.B, x.H, 48, 3)
    ref, ref_lse = oracle.mla(x.q, x.c_pool, x.block_table, x.seq_lens, x.scale, pairs=pr)
    assert_attn_close(out[pr[:, 0], pr[:, 1]], ref, what="mla full size")
    assert np.max(np.abs(to_np(lse)[pr[:, 0], pr[:, 1]] - ref_lse)) < 2e-3 * max(1.0, np.abs(ref_lse).max())


def test_mla_ragged_many_tiles_every_head(kvd):
    # enough tiles that the ranges are cut with a gap before every later sequence, and
    # lengths that put sequence boundaries, tiny sequences and partial tiles inside ranges;
    # every (sequence, head) output is checked
    lens = [60001, 1, 30000, 64, 65, 20000, 7, 5000]
    x = W.make_mla(len(lens), 128, lens, page_size=64, shuffle=True, extra_pages=5, seed=640)
    out, lse = _dense(kvd, x)
    ref, ref_lse = oracle.mla(x.q, x.c_pool, x.block_table, x.seq_lens, x.scale)
    assert_attn_close(out, ref, what="mla ragged many tiles")
    assert np.max(np.abs(to_np(lse) - ref_lse)) < 2e-3 * max(1.0, np.abs(ref_lse).max())


def test_dsa_full_size_sparse_mla_sampled(kvd):
    idx_in, x = W.build("dsa_sparse_mla")
    rng = np.random.default_rng(11)
    k = idx_in.k
    idx = np.stack([np.sort(rng.choice(int(L), k, replace=False)) for L in x.seq_lens]).astype(np.int32)
    cnt = np.full(x.B, k, np.int32)
    out, _ = _sparse(kvd, x, idx, cnt)
    pr = _pairs(x.B, x.H, 48, 4)
    ref, _ = oracle.mla(x.q, x.c_pool, x.block_table, x.seq_lens, x.scale, idx=idx, idx_count=cnt,
                        pairs=pr)
    assert_attn_close(out[pr[:, 0], pr[:, 1]], ref, what="sparse mla full size")


def _poison_past_end(pool, bt, lens, P):
    """A copy of a [num_pages, P, ...] pool whose slots past each sequence's last token
    hold NaN, +Inf and -Inf in turn, and whose pages no sequence uses hold NaN: none of them
    is visible, so the output must not change ("All the attentions", section 8)."""
    pool = pool.clone()
    used = set()
    bad = [float("nan"), float("inf"), float("-inf")]
    for b, L in enumerate(int(v) for v in lens):
        n = -(-L // P)
        used.update(int(v) for v in bt[b, :n])
        last, r = int(bt[b, n - 1]), L - (n - 1) * P
        for slot in range(r, P):
            pool[last, slot] = bad[slot % 3]
    for pg in range(pool.shape[0]):
        if pg not in used:
            pool[pg] = float("nan")
    return pool


@pytest.mark.parametrize("P", [64, 16])
def test_mla_dense_non_finite_slots_past_end(kvd, P):
    lens = [1, 63, 65, 127, 700, 3001]
    x = W.make_mla(len(lens), 128, lens, page_size=P, shuffle=True, extra_pages=3,
                   seed=650 + P)
    x.c_pool = _poison_past_end(x.c_pool, x.block_table, lens, P)
    out, lse = _dense(kvd, x)
    ref, ref_lse = oracle.mla(x.q, x.c_pool, x.block_table, x.seq_lens, x.scale)
    assert np.isfinite(ref).all()
    assert_attn_close(out, ref, what=f"mla, non-finite slots past the end, P={P}")
    assert np.max(np.abs(to_np(lse) - ref_lse)) < 2e-3 * max(1.0, np.abs(ref_lse).max())
