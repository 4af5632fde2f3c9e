"""GPU parity of the cache append (paged, rolling, MLA latent) and of sliding-window
attention read from a rolling cache, against the oracle, through the C ABI.

* Appends are byte copies: bit-exact against the oracle's append.
* Ring attention: the attention bar of the other decode kernels (tests/parity.py) against
  the oracle reading the same ring; in the decode loop, against the plain window oracle over
  the whole history, with the ring filled by the GPU append one token at a time.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.parity import assert_attn_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def kvd():
    import kv_cache_decode_split_gb300 as m
    return m


def _append_gpu(kvd, k_new, v_new, k_pool, v_pool, bt, sl, window=0, n_sink=0):
    kp, vp = k_pool.clone().to(DEV), (v_pool.clone().to(DEV) if v_pool is not None else None)
    err = kvd.cache_append(k_new.to(DEV), v_new.to(DEV) if v_new is not None else None, kp, vp,
                           bt.to(DEV), sl.to(DEV), window=window, n_sink=n_sink)
    torch.cuda.synchronize()
    return kp.cpu(), (vp.cpu() if vp is not None else None), int(err.item())


@pytest.mark.parametrize("dtype,D,P", [(torch.bfloat16, 128, 64), (torch.bfloat16, 64, 16),
                                       (torch.float32, 64, 16)])
def test_append_paged_bit_exact(kvd, dtype, D, P):
    lens = [1, 64, 65, 300, 4096]
    x = W.make_gqa(len(lens), 16, 8, D, lens, page_size=P, shuffle=True, extra_pages=3,
                   seed=8000 + D + P, dtype=dtype)
    k_new = W.normal((len(lens), 8, D), 8100, 1.0, dtype)
    v_new = W.normal((len(lens), 8, D), 8101, 1.0, dtype)
    kp, vp, err = _append_gpu(kvd, k_new, v_new, x.k_pool, x.v_pool, x.block_table, x.seq_lens)
    assert err == 0
    assert torch.equal(kp, oracle.cache_append(x.k_pool, k_new, x.block_table, x.seq_lens))
    assert torch.equal(vp, oracle.cache_append(x.v_pool, v_new, x.block_table, x.seq_lens))


def test_append_mla_latent_rows(kvd):
    lens = [1, 100, 1000]
    x = W.make_mla(3, 128, lens, page_size=64, shuffle=True, extra_pages=2, seed=8200)
    c_new = W.normal((3, 576), 8201, 0.1)
    cp, _, err = _append_gpu(kvd, c_new, None, x.c_pool, None, x.block_table, x.seq_lens)
    assert err == 0
    assert torch.equal(cp, oracle.cache_append(x.c_pool, c_new, x.block_table, x.seq_lens))


@pytest.mark.parametrize("window,n_sink,P", [(4096, 4, 64), (100, 0, 16), (37, 3, 16)])
def test_append_ring_bit_exact(kvd, window, n_sink, P):
    cap = window + n_sink
    lens = [1, 2, n_sink + 1, cap - 1, cap, cap + 1, 3 * cap + 7, 100000]
    r = W.make_ring(len(lens), 8, 8, 64, lens, window, n_sink=n_sink, page_size=P,
                    extra_pages=2, seed=8300 + window)
    k_new = W.normal((len(lens), 8, 64), 8301)
    v_new = W.normal((len(lens), 8, 64), 8302)
    kp, vp, err = _append_gpu(kvd, k_new, v_new, r.k_pool, r.v_pool, r.block_table, r.seq_lens,
                              window, n_sink)
    assert err == 0
    assert torch.equal(kp, oracle.cache_append(r.k_pool, k_new, r.block_table, r.seq_lens,
                                               window, n_sink))
    assert torch.equal(vp, oracle.cache_append(r.v_pool, v_new, r.block_table, r.seq_lens,
                                               window, n_sink))


def test_append_bad_page_is_flagged_and_skipped(kvd):
    x = W.make_gqa(2, 8, 2, 64, [100, 100], page_size=64, seed=8400)
    bt = x.block_table.clone()
    bt[1, 1] = x.num_pages + 5          # the page of position 99 of sequence 1
    k_new = W.normal((2, 2, 64), 8401)
    v_new = W.normal((2, 2, 64), 8402)
    kp, vp, err = _append_gpu(kvd, k_new, v_new, x.k_pool, x.v_pool, bt, x.seq_lens)
    assert err == -6
    # sequence 0 written, sequence 1 not written anywhere
    good = oracle.cache_append(x.k_pool, k_new, x.block_table,
                               torch.tensor([100, 100], dtype=torch.int32))
    b0 = int(x.block_table[0, 1])
    assert torch.equal(kp[b0], good[b0])
    others = [p for p in range(x.num_pages) if p != b0]
    assert torch.equal(kp[others], x.k_pool[others])


def _ring_gpu(kvd, r, ws=None):
    sink = r.sink_logit.to(DEV) if r.sink_logit is not None else None
    out = kvd.attn_decode_swa_ring(r.q.to(DEV), r.k_pool.to(DEV), r.v_pool.to(DEV),
                                   r.block_table.to(DEV), r.seq_lens.to(DEV), r.window, r.n_sink,
                                   sink, scale=r.scale, workspace=ws)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("window,n_sink,learned,D,P", [(256, 4, False, 64, 64),
                                                       (100, 0, True, 128, 16),
                                                       (37, 3, True, 64, 16)])
def test_ring_attention_matches_oracle(kvd, window, n_sink, learned, D, P):
    cap = window + n_sink
    lens = [1, 3, n_sink + 1, cap - 1, cap, cap + 1, 10 * cap + 3]
    r = W.make_ring(len(lens), 16, 4, D, lens, window, n_sink=n_sink, page_size=P,
                    extra_pages=2, seed=8500 + window, learned_sink=learned)
    ws = kvd.Workspace(DEV)
    out = _ring_gpu(kvd, r, ws)
    assert kvd.kvd_check_device_error(ws) == 0
    ref, _ = oracle.gqa(r.q, r.k_pool, r.v_pool, r.block_table, r.seq_lens, r.scale, window,
                        n_sink, r.sink_logit, ring=True)
    assert_attn_close(out, ref, what="ring")


def test_ring_attention_fp32(kvd):
    lens = [5, 70, 300]
    r = W.make_ring(3, 8, 2, 64, lens, 64, n_sink=2, page_size=16, seed=8600,
                    dtype=torch.float32)
    out = _ring_gpu(kvd, r)
    ref, _ = oracle.gqa(r.q, r.k_pool, r.v_pool, r.block_table, r.seq_lens, r.scale, 64, 2,
                        None, ring=True)
    assert_attn_close(out, ref, max_abs=1e-4, mean_abs=1e-4, rel_l2=1e-4, what="ring fp32")


def test_ring_full_size_sampled(kvd):
    r = W.build("swa_ring_sink_tokens")
    out = _ring_gpu(kvd, r)
    rng = np.random.default_rng(3)
    pairs = [(int(b), int(h)) for b, h in zip(rng.integers(0, r.B, 64), rng.integers(0, r.Hq, 64))]
    ref, _ = oracle.gqa(r.q, r.k_pool, r.v_pool, r.block_table, r.seq_lens, r.scale, r.window,
                        r.n_sink, r.sink_logit, pairs=pairs, ring=True)
    pi = np.asarray(pairs)
    assert_attn_close(out[pi[:, 0], pi[:, 1]], ref, what="ring full size")


def _two_calls_and_one(kvd, r, k_new, v_new, chunk=0):
    """The append then the ring attention (two calls), and the same step as one call, each on
    its own copy of the ring: outputs, lse and the updated rings."""
    sink = r.sink_logit.to(DEV) if r.sink_logit is not None else None
    bt, sl, q = r.block_table.to(DEV), r.seq_lens.to(DEV), r.q.to(DEV)
    kvd.kvd_set_option("gqa_chunk", chunk)
    try:
        k2, v2 = r.k_pool.clone().to(DEV), r.v_pool.clone().to(DEV)
        err = kvd.cache_append(k_new, v_new, k2, v2, bt, sl, window=r.window, n_sink=r.n_sink)
        ws2 = kvd.Workspace(DEV)
        lse2 = torch.empty(r.B, r.Hq, device=DEV)
        out2 = kvd.attn_decode_swa_ring(q, k2, v2, bt, sl, r.window, r.n_sink, sink,
                                        scale=r.scale, lse_out=lse2, workspace=ws2)
        k1, v1 = r.k_pool.clone().to(DEV), r.v_pool.clone().to(DEV)
        ws1 = kvd.Workspace(DEV)
        lse1 = torch.empty(r.B, r.Hq, device=DEV)
        out1 = kvd.attn_decode_swa_ring_append(q, k_new, v_new, k1, v1, bt, sl, r.window,
                                               r.n_sink, sink, scale=r.scale, lse_out=lse1,
                                               workspace=ws1)
        torch.cuda.synchronize()
    finally:
        kvd.kvd_set_option("gqa_chunk", 0)
    assert int(err.item()) == 0 and kvd.kvd_check_device_error(ws2) == 0
    assert kvd.kvd_check_device_error(ws1) == 0
    return (out1, lse1, k1, v1), (out2, lse2, k2, v2)


@pytest.mark.parametrize("dtype,D,P,window,n_sink,chunk", [
    (torch.bfloat16, 64, 64, 256, 4, 0),     # two KV heads per tile
    (torch.bfloat16, 64, 16, 300, 4, 64),    # many chunks: one of them holds the newest slot
    (torch.bfloat16, 128, 16, 100, 0, 0),    # one KV head per tile, no sinks
    (torch.float32, 64, 16, 64, 2, 0)])      # float32: the append's launch, then attention
def test_ring_append_one_call_equals_two_calls(kvd, dtype, D, P, window, n_sink, chunk):
    # "Attention Optimizations", DSA / Computation Path (the new token's row written before
    # attention); "All the attentions", section 4 (the newest entry replaces the oldest):
    # one call is the append followed by the ring attention, bit for bit
    cap = window + n_sink
    lens = [1, 2, n_sink + 1, cap - 1, cap, cap + 1, 7 * cap + 5]
    r = W.make_ring(len(lens), 16, 4, D, lens, window, n_sink=n_sink, page_size=P,
                    extra_pages=2, seed=8900 + D + P + window, learned_sink=True, dtype=dtype)
    k_new = W.normal((r.B, r.Hkv, D), 8950 + D, 1.0, dtype).to(DEV)
    v_new = W.normal((r.B, r.Hkv, D), 8951 + D, 1.0, dtype).to(DEV)
    (o1, l1, k1, v1), (o2, l2, k2, v2) = _two_calls_and_one(kvd, r, k_new, v_new, chunk)
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # and the output is the ring oracle's over the updated ring
    ref, _ = oracle.gqa(r.q, k1.cpu(), v1.cpu(), r.block_table, r.seq_lens, r.scale, window,
                        n_sink, r.sink_logit, ring=True)
    tol = dict(max_abs=1e-4, mean_abs=1e-4, rel_l2=1e-4) if dtype == torch.float32 else {}
    assert_attn_close(o1, ref, what="ring append + attention, one call", **tol)


def test_ring_append_one_call_bad_page_is_flagged(kvd):
    # the newest slot's page id out of range: recorded in the workspace's error flag, and the
    # pool is left as it was there
    r = W.make_ring(2, 8, 2, 64, [10, 40], 32, n_sink=2, page_size=16, seed=8990)
    bt = r.block_table.clone()
    slot = 2 + (40 - 1 - 2) % 32  # sequence 1's newest token
    bt[1, slot // 16] = r.num_pages + 7
    k_new = W.normal((2, 2, 64), 8991, 1.0, torch.bfloat16).to(DEV)
    v_new = W.normal((2, 2, 64), 8992, 1.0, torch.bfloat16).to(DEV)
    kp, vp = r.k_pool.clone().to(DEV), r.v_pool.clone().to(DEV)
    ws = kvd.Workspace(DEV)
    kvd.attn_decode_swa_ring_append(r.q.to(DEV), k_new, v_new, kp, vp, bt.to(DEV),
                                    r.seq_lens.to(DEV), 32, 2, None, workspace=ws)
    assert kvd.kvd_check_device_error(ws) == -6
    # sequence 0's row is in place; nothing else of the pool changed but that one row
    pg0 = int(r.block_table[0, 9 // 16])
    assert torch.equal(kp[pg0, :, 9 % 16].cpu(), k_new[0].cpu())
    changed = (kp.cpu() != r.k_pool).any(dim=(1, 2, 3)).nonzero().flatten().tolist()
    assert changed in ([pg0], [])


@pytest.mark.parametrize("one_call", [False, True])
def test_decode_loop_ring_equals_window_over_history(kvd, one_call):
    # every step: the GPU appends the token's K/V into the ring, then attends from the ring
    # (two calls, or the one-call step); the outputs follow the plain window oracle over the
    # whole history
    B, Hq, Hkv, D, P, window, n_sink, T = 2, 8, 2, 64, 16, 48, 4, 180
    full = W.make_gqa(B, Hq, Hkv, D, [T] * B, page_size=P, shuffle=True, seed=8700,
                      window=window, n_sink=n_sink, learned_sink=True)
    ring = W.make_ring(B, Hq, Hkv, D, [1] * B, window, n_sink=n_sink, page_size=P, seed=8701)
    kr, vr = ring.k_pool.to(DEV), ring.v_pool.to(DEV)
    bt_r = ring.block_table.to(DEV)
    q, sink = full.q.to(DEV), full.sink_logit.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = kvd.Workspace(DEV)
    checks = {1, 2, n_sink + 1, window, window + n_sink, window + n_sink + 1, 2 * window + 9, T}
    for t in range(1, T + 1):
        rows = [(int(full.block_table[b][(t - 1) // P]), (t - 1) % P) for b in range(B)]
        k_new = torch.stack([full.k_pool[pg, :, s] for pg, s in rows]).to(DEV)
        v_new = torch.stack([full.v_pool[pg, :, s] for pg, s in rows]).to(DEV)
        lens = torch.full((B,), t, dtype=torch.int32, device=DEV)
        if one_call:
            out = kvd.attn_decode_swa_ring_append(q, k_new, v_new, kr, vr, bt_r, lens, window,
                                                  n_sink, sink, scale=full.scale, workspace=ws)
        else:
            kvd.cache_append(k_new, v_new, kr, vr, bt_r, lens, window=window, n_sink=n_sink,
                             err=err)
            out = kvd.attn_decode_swa_ring(q, kr, vr, bt_r, lens, window, n_sink, sink,
                                           scale=full.scale, workspace=ws)
        if t in checks:
            torch.cuda.synchronize()
            ref, _ = oracle.gqa(full.q, full.k_pool, full.v_pool, full.block_table,
                                torch.full((B,), t, dtype=torch.int32), full.scale, window,
                                n_sink, full.sink_logit)
            assert_attn_close(out, ref, what=f"step {t}")
    assert int(err.item()) == 0
    assert kvd.kvd_check_device_error(ws) == 0


def test_ring_rejects_a_ring_larger_than_its_table(kvd):
    r = W.make_ring(1, 8, 2, 64, [10], 64, page_size=16, seed=8800)
    with pytest.raises(kvd.KvdError) as e:
        kvd.attn_decode_swa_ring(r.q.to(DEV), r.k_pool.to(DEV), r.v_pool.to(DEV),
                                 r.block_table.to(DEV), r.seq_lens.to(DEV), 64, 5, None)
    assert e.value.status == -1
