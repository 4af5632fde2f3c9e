"""attn_decode_gqa_paged_static_ws: the GQA decode for callers that cannot allocate.

Some callers of this library hold only their input and output buffers and may not call
cudaMalloc (a plugin whose host engine owns all device memory, or a decode loop that
must not take cudaMalloc's device-wide synchronisation). For them the library keeps its
split-KV scratch in a fixed-size device array of its own. This file checks, through the
C ABI, that two calls in a row of that entry point give the same results as the
workspace entry point, within the parity tolerance of the other GPU tests, and that a
shape needing more scratch than the array holds is refused before any launch.

The file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import workloads as W
from tests.parity import assert_attn_close

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


def test_static_scratch_matches_workspace_entry_point(lib):
    x = W.make_gqa(8, 32, 8, 128, [1, 64, 65, 700, 1500, 3000, 4096, 8192], page_size=64,
                   shuffle=True, extra_pages=7, seed=4242)
    d = {"q": x.q.cuda(), "k": x.k_pool.cuda(), "v": x.v_pool.cuda(),
         "bt": x.block_table.cuda(), "sl": x.seq_lens.cuda()}
    ref = torch.empty_like(d["q"])
    ref_lse = torch.empty(x.B, x.Hq, dtype=torch.float32, device="cuda")
    assert _call_ws(lib, x, d, ref, ref_lse) == 0
    torch.cuda.synchronize()
    for _ in range(2):   # the second call finds the first call's contents in the array
        out = torch.full_like(d["q"], float("nan"))
        lse = torch.full((x.B, x.Hq), float("nan"), dtype=torch.float32, device="cuda")
        assert _call_static(lib, x, d, out, lse) == 0
        torch.cuda.synchronize()
        assert_attn_close(out, ref.double().cpu().numpy(), what="static scratch vs workspace")
        assert torch.allclose(lse, ref_lse, atol=1e-3, rtol=0)


def test_static_scratch_rejects_oversized_plans(lib):
    # B=1024 sequences x 8 KV heads x up to 64K tokens needs far more than the array holds
    st = lib.attn_decode_gqa_paged_static_ws(
        ctypes.c_void_p(256), ctypes.c_void_p(256), ctypes.c_void_p(256), ctypes.c_void_p(256),
        ctypes.c_void_p(256), ctypes.c_void_p(256), None, 1024, 64, 8, 128, 64, 1024, 4096,
        0.088, 1, _stream())
    assert st == -5
