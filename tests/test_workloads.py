"""The seeded input generators: deterministic, and shaped as their workloads say."""
import math

import torch

import workloads as W


def test_generators_are_deterministic():
    a = W.make_delta(3, 64, 32, seed=5)
    b = W.make_delta(3, 64, 32, seed=5)
    for f in ("S", "q", "k", "v", "a", "beta"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f
    r1 = W.make_ring(2, 8, 2, 64, [10, 900], 128, n_sink=4, page_size=16, seed=6)
    r2 = W.make_ring(2, 8, 2, 64, [10, 900], 128, n_sink=4, page_size=16, seed=6)
    assert torch.equal(r1.k_pool, r2.k_pool) and torch.equal(r1.block_table, r2.block_table)


def test_delta_inputs_follow_the_recipe():
    x = W.make_delta(16, 128, 128, seed=7)
    assert x.S.shape == (16, 128, 128) and x.S.dtype == torch.float32
    assert torch.allclose(x.k.norm(dim=1), torch.ones(16), atol=1e-5)
    assert torch.allclose(x.q.norm(dim=1), torch.full((16,), 1 / math.sqrt(128)), atol=1e-6)
    assert float(x.a.min()) >= 0.9 and float(x.a.max()) < 1.0
    assert float(x.beta.min()) >= 0.0 and float(x.beta.max()) < 1.0
    g = W.make_delta(4, 64, 64, per_channel=False, seed=8)
    assert g.a.shape == (4,)


def test_ring_inputs_hold_capacity_pages_per_sequence():
    window, n_sink, P = 100, 4, 16
    r = W.make_ring(3, 8, 2, 64, [1, 50, 100000], window, n_sink=n_sink, page_size=P,
                    extra_pages=5, seed=9)
    pages = -(-(window + n_sink) // P)
    assert r.block_table.shape == (3, pages) and r.ring
    used = r.block_table.flatten()
    assert int(used.min()) >= 0 and len(set(used.tolist())) == 3 * pages   # distinct pages
    assert r.k_pool.shape[0] == 3 * pages + 5
    assert r.seq_lens.tolist() == [1, 50, 100000]


def test_named_small_workloads():
    x = W.build("tiny_gqa_fp32")
    assert x.q.dtype == torch.float32 and x.seq_lens.tolist() == [256, 256]
    p = W.WORKLOADS["kda_decode"].params
    assert p["B"] * p["H"] * p["dk"] * p["dv"] * 4 > 129e6          # larger than L2
    q = W.WORKLOADS["quest_llama3"].params
    assert q["page_size"] == 16 and q["n_sel"] * q["page_size"] == 256
    s = W.WORKLOADS["swa_ring_sink_tokens"].params
    assert s["ring"] and s["window"] == 4096 and s["n_sink"] == 4
