"""attn_decode_gqa_paged_static_ws: the GQA decode for callers that cannot allocate.

Some callers of this library hold only their input and output buffers and may not call
cudaMalloc (a plugin whose host engine owns all device memory, or a decode loop that
must not take cudaMalloc's device-wide synchronisation). For them the library keeps its
split-KV scratch in a fixed-size device array of its own. This file checks, through the
C ABI, that calls in a row of that entry point (with other shapes, so that each finds the
previous call's contents in the array) give the oracle's results within the parity
tolerance of the other GPU tests, and the workspace entry point's; that bad arguments are
refused as the workspace entry point refuses them; and that a shape needing more scratch
than the array holds is refused before any launch.

The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.parity import assert_attn_close, to_np

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.fixture(scope="module")
def lib():
    import kv_cache_decode_split_gb300 as kvd
    return kvd.lib


def _call_static(lib, x, d, out, lse):
    return lib.attn_decode_gqa_paged_static_ws(
        _p(d["q"]), _p(d["k"]), _p(d["v"]), _p(d["bt"]), _p(d["sl"]), _p(out), _p(lse), x.B, x.Hq,
        x.Hkv, x.D, x.page_size, x.max_pages, x.num_pages, x.scale, 1, _stream())


def _call_ws(lib, x, d, out, lse):
    nbytes = lib.kvd_workspace_size(0, x.B, x.Hq, x.Hkv, x.D, x.max_pages * x.page_size, 0, 0, 0)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    st = lib.attn_decode_gqa_paged(
        _p(d["q"]), _p(d["k"]), _p(d["v"]), _p(d["bt"]), _p(d["sl"]), _p(out), _p(lse), x.B, x.Hq,
        x.Hkv, x.D, x.page_size, x.max_pages, x.num_pages, x.scale, 1, _p(ws), nbytes, _stream())
    return st


def _inputs(x):
    return {"q": x.q.cuda(), "k": x.k_pool.cuda(), "v": x.v_pool.cuda(),
            "bt": x.block_table.cuda(), "sl": x.seq_lens.cuda()}


def test_static_scratch_matches_oracle_and_workspace_entry_point(lib):
    # Calls in a row with other shapes, so that each finds the previous call's partials and
    # counters in the shared array: longer sequences and more chunks first, then a smaller
    # batch of short ones, then the first shape again. Each output is held to the oracle
    # (the parity bar of the other GPU tests) and to the workspace entry point.
    xa = W.make_gqa(8, 32, 8, 128, [1, 64, 65, 700, 1500, 3000, 4096, 8192], page_size=64,
                    shuffle=True, extra_pages=7, seed=4242)
    xb = W.make_gqa(3, 16, 2, 64, [5, 130, 999], page_size=16, shuffle=True, extra_pages=2,
                    seed=4243)
    for x in (xa, xb, xa):
        d = _inputs(x)
        ref, ref_lse = oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale)
        ws_out = torch.empty_like(d["q"])
        ws_lse = torch.empty(x.B, x.Hq, dtype=torch.float32, device="cuda")
        assert _call_ws(lib, x, d, ws_out, ws_lse) == 0
        out = torch.full_like(d["q"], float("nan"))
        lse = torch.full((x.B, x.Hq), float("nan"), dtype=torch.float32, device="cuda")
        assert _call_static(lib, x, d, out, lse) == 0
        torch.cuda.synchronize()
        assert_attn_close(out, ref, what=f"static scratch vs oracle, B={x.B}")
        assert np.max(np.abs(to_np(lse) - ref_lse)) < 2e-3
        assert_attn_close(out, ws_out.double().cpu().numpy(), what="static vs workspace")


def test_static_scratch_rejects_bad_arguments_like_the_workspace_entry_point(lib):
    # argument checks come first (before the shared array is touched) and return what the
    # workspace entry point returns
    x = W.make_gqa(2, 8, 2, 64, [100, 200], page_size=64, seed=4244)
    d = _inputs(x)
    out = torch.empty_like(d["q"])
    for D, page_size, dtype, want in [(96, 64, 1, -2), (64, 48, 1, -2), (64, 64, 7, -2)]:
        st = lib.attn_decode_gqa_paged_static_ws(
            _p(d["q"]), _p(d["k"]), _p(d["v"]), _p(d["bt"]), _p(d["sl"]), _p(out), None, x.B,
            x.Hq, x.Hkv, D, page_size, x.max_pages, x.num_pages, x.scale, dtype, _stream())
        ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
        st_ws = lib.attn_decode_gqa_paged(
            _p(d["q"]), _p(d["k"]), _p(d["v"]), _p(d["bt"]), _p(d["sl"]), _p(out), None, x.B,
            x.Hq, x.Hkv, D, page_size, x.max_pages, x.num_pages, x.scale, dtype, _p(ws),
            ws.numel(), _stream())
        assert st == st_ws == want, (D, page_size, dtype, st, st_ws)
    st = lib.attn_decode_gqa_paged_static_ws(
        None, _p(d["k"]), _p(d["v"]), _p(d["bt"]), _p(d["sl"]), _p(out), None, x.B, x.Hq, x.Hkv,
        x.D, 64, x.max_pages, x.num_pages, x.scale, 1, _stream())
    assert st == -1


def test_static_scratch_rejects_oversized_plans(lib):
    # B=1024 sequences x 8 KV heads x up to 64K tokens needs far more than the array holds
    st = lib.attn_decode_gqa_paged_static_ws(
        ctypes.c_void_p(256), ctypes.c_void_p(256), ctypes.c_void_p(256), ctypes.c_void_p(256),
        ctypes.c_void_p(256), ctypes.c_void_p(256), None, 1024, 64, 8, 128, 64, 1024, 4096,
        0.088, 1, _stream())
    assert st == -5
