"""GPU parity of attn_decode_gqa_paged / attn_decode_swa_sink against the fp64 oracle.

Small cases compare every output; the full-size Llama-3-8B-shaped and sliding-window
workloads compare a seeded sample of (sequence, head) outputs, in the same launch
configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.parity import assert_attn_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvd():
    import kv_cache_decode_split_gb300 as m
    return m


_WS = {}


def _run(kvd, x, lse=True):
    dev = "cuda"
    ws = _WS.setdefault("ws", kvd.Workspace(dev))
    q, kp, vp = x.q.to(dev), x.k_pool.to(dev), x.v_pool.to(dev)
    bt, sl = x.block_table.to(dev), x.seq_lens.to(dev)
    lse_out = torch.empty(x.B, x.Hq, dtype=torch.float32, device=dev) if lse else None
    if x.window > 0 or x.n_sink > 0 or x.sink_logit is not None:
        sink = x.sink_logit.to(dev) if x.sink_logit is not None else None
        out = kvd.attn_decode_swa_sink(q, kp, vp, bt, sl, max(x.window, 1) if x.window > 0 else 1 << 30,
                                       x.n_sink, sink, scale=x.scale, lse_out=lse_out,
                                       workspace=ws)
    else:
        out = kvd.attn_decode_gqa_paged(q, kp, vp, bt, sl, scale=x.scale, lse_out=lse_out,
                                        workspace=ws)
    torch.cuda.synchronize()
    assert kvd.kvd_check_device_error(ws) == 0
    return out, lse_out


def _compare(kvd, x, tol=None, pairs=None):
    out, lse = _run(kvd, x)
    ref, ref_lse = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale,
                              x.window, x.n_sink, x.sink_logit, pairs=pairs)
    if pairs is not None:
        pi = np.asarray(pairs)
        out = out[pi[:, 0], pi[:, 1]]
        lse = lse[pi[:, 0], pi[:, 1]]
    kw = {} if tol is None else dict(max_abs=tol, mean_abs=tol, rel_l2=tol)
    assert_attn_close(out, ref, what="out", **kw)
    assert np.max(np.abs(to_np(lse) - ref_lse)) < 2e-3


def test_tiny_fp32_workload(kvd):
    x = W.build("tiny_gqa_fp32")
    _compare(kvd, x, tol=1e-4)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(8, 2), (32, 8), (4, 4), (16, 1), (32, 1), (12, 4)])
def test_bf16_paged_ragged(kvd, D, hq, hkv):
    lens = [1, 63, 64, 65, 200, 1000, 1500, 2047]
    x = W.make_gqa(len(lens), hq, hkv, D, lens, page_size=64, shuffle=True, extra_pages=5,
                   seed=100 + D + hq)
    _compare(kvd, x)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("P", [16, 32, 128, 256])
def test_page_sizes(kvd, P, D):
    # D = 64 with an even KV-head count and pages of <= 64 tokens moves two KV heads per
    # tile; larger pages split into 64-token pieces
    lens = [5, 130, 777]
    x = W.make_gqa(3, 8, 2, D, lens, page_size=P, shuffle=True, seed=200 + P + D)
    _compare(kvd, x)


@pytest.mark.parametrize("chunk", [64, 192])
@pytest.mark.parametrize("D", [64, 128])
def test_many_chunks(kvd, chunk, D):
    # short chunks: up to 126 chunk partials per head block in the final combine
    lens = [1, 100, 4000, 8000]
    x = W.make_gqa(len(lens), 16, 4, D, lens, page_size=64, shuffle=True, seed=400 + chunk + D)
    kvd.kvd_set_option("gqa_chunk", chunk)
    try:
        _compare(kvd, x)
    finally:
        kvd.kvd_set_option("gqa_chunk", 0)


def test_fp32_paged_shuffled(kvd):
    x = W.make_gqa(3, 8, 2, 128, [3, 300, 700], page_size=32, shuffle=True, seed=7,
                   dtype=torch.float32)
    _compare(kvd, x, tol=1e-4)


@pytest.mark.parametrize("window,n_sink,learned", [(1, 0, False), (64, 4, False), (100, 4, True),
                                                   (300, 0, True), (5000, 4, False),
                                                   (700, 70, False), (129, 200, True)])
def test_swa_sink(kvd, window, n_sink, learned):
    lens = [1, 3, 64, 190, 1000, 3000]
    x = W.make_gqa(len(lens), 16, 2, 64, lens, page_size=64, shuffle=True, seed=300 + window,
                   window=window, n_sink=n_sink, learned_sink=learned)
    _compare(kvd, x)


def test_learned_sink_values(kvd):
    # softmax-off-by-one (sink logit 0) and a strongly dominant sink
    x = W.make_gqa(2, 8, 2, 64, [50, 300], page_size=64, seed=9, window=128)
    x.sink_logit = torch.zeros(8)
    _compare(kvd, x)
    x.sink_logit = torch.full((8,), 30.0)
    _compare(kvd, x)


def test_window_at_least_length_equals_dense(kvd):
    x = W.make_gqa(4, 32, 8, 128, [100, 1000, 4000, 8000], page_size=64, shuffle=True, seed=11)
    dense, _ = _run(kvd, x)
    x.window = 8192
    win, _ = _run(kvd, x)
    assert torch.equal(dense, win) or torch.allclose(dense.float(), win.float(), atol=1e-2)


def _sample_pairs(B, H, n, seed):
    rng = np.random.default_rng(seed)
    b = rng.integers(0, B, n)
    h = rng.integers(0, H, n)
    return np.stack([b, h], axis=1).astype(np.int32)


def test_llama3_8b_full_size_sampled(kvd):
    x = W.build("llama3_8b_gqa_paged")
    _compare(kvd, x, pairs=_sample_pairs(x.B, x.Hq, 96, 1))


@pytest.mark.parametrize("name", ["swa_sink_tokens", "swa_learned_sink"])
def test_swa_full_size_sampled(kvd, name):
    x = W.build(name)
    _compare(kvd, x, pairs=_sample_pairs(x.B, x.Hq, 96, 2))


def test_repeat_calls_reuse_workspace(kvd):
    x = W.make_gqa(4, 32, 8, 128, [100, 1000, 4000, 8000], page_size=64, shuffle=True, seed=12)
    a, _ = _run(kvd, x)
    b, _ = _run(kvd, x)
    assert torch.equal(a, b)


def test_out_of_range_page_is_recorded_not_faulted(kvd):
    x = W.make_gqa(2, 8, 2, 64, [100, 100], page_size=64, seed=13)
    x.block_table[1, 0] = 10_000      # past num_pages: clamped on device, flagged
    dev = "cuda"
    ws = kvd.Workspace(dev)
    kvd.attn_decode_gqa_paged(x.q.to(dev), x.k_pool.to(dev), x.v_pool.to(dev),
                              x.block_table.to(dev), x.seq_lens.to(dev), workspace=ws)
    assert kvd.kvd_check_device_error(ws) == -6
    assert kvd.kvd_check_device_error(ws) == 0   # cleared


@pytest.mark.parametrize("D,P", [(128, 64), (64, 16), (64, 64)])
def test_non_finite_slots_past_end(kvd, D, P):
    # slots past each sequence's last token hold NaN, +Inf and -Inf in turn, unused pages
    # NaN: none is visible, so the output must not change ("All the attentions", section 8)
    lens = [1, 63, 65, 127, 700, 3001]
    x = W.make_gqa(len(lens), 16, 4, D, lens, page_size=P, shuffle=True, extra_pages=3,
                   seed=460 + D + P)
    used = set()
    bad = [float("nan"), float("inf"), float("-inf")]
    for pool in (x.k_pool, x.v_pool):
        for b, L in enumerate(lens):
            n = -(-L // P)
            used.update(int(v) for v in x.block_table[b, :n])
            last, r = int(x.block_table[b, n - 1]), L - (n - 1) * P
            for slot in range(r, P):
                pool[last, :, slot] = bad[slot % 3]
        for pg in range(pool.shape[0]):
            if pg not in used:
                pool[pg] = float("nan")
    _compare(kvd, x)


@pytest.mark.parametrize("D,lens", [(128, [100, 2000, 4000, 7000]), (64, [3, 64, 130])])
def test_bounded_wait_gives_up_and_reports_timeout(kvd, D, lens):
    # One call whose copy-ring waits are limited to ~1000 cycles and whose consumer warps
    # first wait on a barrier nothing completes: the wait runs out, the call records
    # KVD_ERR_TIMEOUT instead of hanging, waits for the copies it issued and returns. The
    # next call on the same workspace is exact again (its counters were left at zero).
    x = W.make_gqa(len(lens), 16, 4, D, lens, page_size=64, shuffle=True, seed=470 + D)
    dev = "cuda"
    ws = kvd.Workspace(dev)
    args = (x.q.to(dev), x.k_pool.to(dev), x.v_pool.to(dev), x.block_table.to(dev),
            x.seq_lens.to(dev))
    kvd.kvd_set_option("wait_timeout_test", 1)
    try:
        kvd.attn_decode_gqa_paged(*args, scale=x.scale, workspace=ws)
        assert kvd.kvd_check_device_error(ws) == -4
    finally:
        kvd.kvd_set_option("wait_timeout_test", 0)
    for _ in range(2):
        lse = torch.empty(x.B, x.Hq, dtype=torch.float32, device=dev)
        out = kvd.attn_decode_gqa_paged(*args, scale=x.scale, lse_out=lse, workspace=ws)
        assert kvd.kvd_check_device_error(ws) == 0
        ref, ref_lse = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale)
        assert_attn_close(out, ref, what="after a timed-out call")
        assert np.max(np.abs(to_np(lse) - ref_lse)) < 2e-3


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("case", ["ragged128", "ragged64", "swa_sinks", "swa_learned", "short"])
def test_combine_paths(kvd, mode, case):
    # the chunk partials combined through the workspace by the last CTA of each group (0), or
    # inside a thread-block cluster over distributed shared memory (1: when groups are few;
    # 2: whenever a group needs at most 8 chunks); chunks past a short sequence's end take
    # part in the cluster combine with nothing
    spec = {
        "ragged128": dict(B=8, hq=32, hkv=8, D=128, lens=[1, 63, 64, 65, 200, 1000, 1500, 4097]),
        "ragged64": dict(B=6, hq=16, hkv=4, D=64, lens=[1, 2, 129, 640, 3000, 9000]),
        "swa_sinks": dict(B=3, hq=64, hkv=8, D=64, lens=[50, 4100, 9000], window=4096, n_sink=4),
        "swa_learned": dict(B=2, hq=32, hkv=8, D=128, lens=[5000, 700], window=1000,
                            learned=True),
        "short": dict(B=2, hq=8, hkv=2, D=128, lens=[1, 3]),
    }[case]
    x = W.make_gqa(spec["B"], spec["hq"], spec["hkv"], spec["D"], spec["lens"], page_size=64,
                   shuffle=True, extra_pages=3, seed=480 + mode + len(case),
                   window=spec.get("window", 0), n_sink=spec.get("n_sink", 0),
                   learned_sink=spec.get("learned", False))
    kvd.kvd_set_option("gqa_cluster", mode)
    try:
        _compare(kvd, x)
        _compare(kvd, x)   # the same workspace again
    finally:
        kvd.kvd_set_option("gqa_cluster", 1)


@pytest.mark.parametrize("D,window,n_sink", [(64, 1024, 4), (128, 0, 0)])
def test_lengths_and_table_rewritten_by_the_previous_kernel(kvd, D, window, n_sink):
    """The bf16 kernel reads the lengths and block-table entries before its dependency wait
    (L2 prefetch hints, and its first copies once the same values are read again after the
    wait). Here the kernel just before it on the stream rewrites both, alternating two sets
    of values over one pool: every call must follow the values that kernel wrote."""
    dev = "cuda"
    B, Hq, Hkv = 4, 16, 4
    lens_new = [3000, 2500, 1900, 3100]
    x = W.make_gqa(B, Hq, Hkv, D, lens_new, page_size=64, shuffle=True, extra_pages=3,
                   seed=900 + D, window=window, n_sink=n_sink)
    # the other set: each sequence takes the next one's block-table row, shorter lengths
    bt_old = torch.roll(x.block_table, 1, dims=0)
    lens_old = torch.tensor([1500, 2900, 700, 1800], dtype=torch.int32)  # within the rows
    refs = {}
    for name, bt, sl in (("new", x.block_table, x.seq_lens), ("old", bt_old, lens_old)):
        refs[name] = oracle.gqa(x.q, x.k_pool, x.v_pool, bt, sl, x.scale, x.window, x.n_sink,
                                None)
    q, kp, vp = x.q.to(dev), x.k_pool.to(dev), x.v_pool.to(dev)
    src = {"new": (x.block_table.to(dev), x.seq_lens.to(dev)),
           "old": (bt_old.to(dev), lens_old.to(dev))}
    bt_d = torch.empty_like(src["new"][0])
    sl_d = torch.empty_like(src["new"][1])
    ws = kvd.Workspace(dev)
    outs = []
    for it in range(12):
        name = "new" if it % 2 == 0 else "old"
        # elementwise kernels (not copies) write the inputs just before the attention launch
        torch.add(src[name][0], 0, out=bt_d)
        torch.add(src[name][1], 0, out=sl_d)
        if window > 0:
            out = kvd.attn_decode_swa_sink(q, kp, vp, bt_d, sl_d, window, n_sink, None,
                                           scale=x.scale, workspace=ws)
        else:
            out = kvd.attn_decode_gqa_paged(q, kp, vp, bt_d, sl_d, scale=x.scale, workspace=ws)
        outs.append((name, out))
    torch.cuda.synchronize()
    assert kvd.kvd_check_device_error(ws) == 0
    for name, out in outs:
        assert_attn_close(out, refs[name][0], what=f"{name} values")
