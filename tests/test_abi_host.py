"""The C ABI without a GPU: the library builds, loads, exports every entry point the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    src = open(os.path.join(ROOT, "include", "kvdecode.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    import importlib.util
    import sys
    sys.path.insert(0, ROOT)
    import __graft_entry__ as g
    path = g._builder().build()
    spec = importlib.util.spec_from_file_location(
        "kvdecode_lib", os.path.join(ROOT, "kv_cache_decode_split_gb300", "_lib.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.load(path)


def test_header_declares_the_entry_points():
    names = _header_functions()
    for n in ("attn_decode_gqa_paged", "attn_decode_swa_sink", "attn_decode_mla",
              "dsa_indexer_topk", "attn_decode_mla_sparse", "dsa_topk", "kvd_workspace_size",
              "kvd_check_device_error", "kvd_status_string", "dsa_indexer_topk_fp8",
              "kvd_quantize_e4m3_rows", "dsa_indexer_cache_append_fp8", "kvd_delta_decode_step"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _header_functions():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert lib.kvd_status_string(0) == b"ok"
    assert lib.kvd_status_string(-5) == b"workspace too small"


def _gqa(lib, **kw):
    a = dict(q=16, k=16, v=16, bt=16, sl=16, out=16, lse=None, B=2, Hq=8, Hkv=2, D=64, P=64,
             max_pages=4, num_pages=8, scale=0.125, dtype=1, ws=256, ws_bytes=1 << 30)
    a.update(kw)
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.attn_decode_gqa_paged(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["bt"]), vp(a["sl"]),
                                     vp(a["out"]), vp(a["lse"]), a["B"], a["Hq"], a["Hkv"], a["D"],
                                     a["P"], a["max_pages"], a["num_pages"], a["scale"], a["dtype"],
                                     vp(a["ws"]), a["ws_bytes"], None)


def test_gqa_argument_checks(lib):
    assert _gqa(lib, q=None) == -1
    assert _gqa(lib, Hq=6, Hkv=4) == -1
    assert _gqa(lib, B=0) == -1
    assert _gqa(lib, D=96) == -2
    assert _gqa(lib, P=48) == -2
    assert _gqa(lib, dtype=7) == -2
    assert _gqa(lib, q=24) == -1                 # not 16-byte aligned
    assert _gqa(lib, scale=float("nan")) == -1
    assert _gqa(lib, ws_bytes=16) == -5


def test_swa_requires_positive_window(lib):
    vp = ctypes.c_void_p
    st = lib.attn_decode_swa_sink(vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), None, 2, 8, 2, 64,
                                  64, 4, 8, 0.125, 1, 0, 4, None, vp(256), 1 << 30, None)
    assert st == -1


def test_workspace_size_queries(lib):
    assert lib.kvd_workspace_size(0, 32, 32, 8, 128, 8192, 0, 0, 0) > 0
    assert lib.kvd_workspace_size(1, 8, 64, 8, 64, 32768, 4096, 4, 0) > 0
    assert lib.kvd_workspace_size(0, 2, 6, 4, 64, 256, 0, 0, 0) == 0   # Hq % Hkv != 0
    assert lib.kvd_workspace_size(99, 2, 8, 2, 64, 256, 0, 0, 0) == 0


def test_delta_step_argument_checks(lib):
    # rejected on the host, before any launch (the pointers are never dereferenced)
    vp = ctypes.c_void_p
    def call(S=1 << 20, q=2 << 20, k=3 << 20, v=4 << 20, a=5 << 20, beta=6 << 20, o=7 << 20,
             n=4, dk=128, dv=128, per_channel=1):
        return lib.kvd_delta_decode_step(vp(S) if S else None, vp(q), vp(k), vp(v), vp(a),
                                         vp(beta), vp(o), n, dk, dv, per_channel, None)
    assert call(S=0) == -1                       # null state
    assert call(n=0) == -1
    assert call(dk=96) == -2 and call(dk=512) == -2
    assert call(dv=0) == -2
    assert call(S=(1 << 20) + 4) == -1           # state not 16-byte aligned
    assert call(a=(5 << 20) + 4) == -1           # per-channel decays not 16-byte aligned
    assert call(o=(1 << 20) + 64) == -1          # output inside the state


def test_append_ring_and_quest_argument_checks(lib):
    # every call below breaks exactly one host-side rule, so none reaches a launch
    vp = ctypes.c_void_p
    A = 1 << 20   # a 16-byte aligned stand-in address, never dereferenced

    def append(k_new=A, v_new=A, err=A, D=64, dtype=1, P=64, max_pages=4, window=0, n_sink=0):
        return lib.kvd_cache_append(vp(k_new) if k_new else None, vp(v_new) if v_new else None,
                                    vp(A), vp(A) if v_new else None, vp(A), vp(A), 2, 8, D, P,
                                    max_pages, 16, dtype, window, n_sink,
                                    vp(err) if err else None, None)
    assert append(k_new=0) == -1
    assert append(err=0) == -1
    assert append(D=6) == -2                       # 12-byte rows
    assert append(dtype=5) == -2
    assert append(window=250, n_sink=7) == -1      # ring larger than the table's 256 slots
    assert append(k_new=A + 8) == -1               # not 16-byte aligned

    def ring(window=64, n_sink=4, max_pages=4):
        return lib.attn_decode_swa_ring(vp(A), vp(A), vp(A), vp(A), vp(A), vp(A), None, 2, 8, 2,
                                        64, 16, max_pages, 16, 0.125, 1, window, n_sink, None,
                                        vp(A), 1 << 30, None)
    assert ring(window=0) == -1
    assert ring(n_sink=-1) == -1
    assert ring(window=64, n_sink=4, max_pages=4) == -1   # 68 slots > 4 pages of 16

    def ring_append(k_new=A, v_new=A, window=64, n_sink=4, max_pages=8, D=64, dtype=1,
                    ws_bytes=1 << 30):
        return lib.attn_decode_swa_ring_append(
            vp(A), vp(k_new) if k_new else None, vp(v_new) if v_new else None, vp(A), vp(A),
            vp(A), vp(A), vp(A), None, 2, 8, 2, D, 16, max_pages, 16, 0.125, dtype, window,
            n_sink, None, vp(A), ws_bytes, None)
    assert ring_append(k_new=0) == -1
    assert ring_append(v_new=0) == -1
    assert ring_append(window=0) == -1
    assert ring_append(n_sink=-1) == -1
    assert ring_append(window=64, n_sink=4, max_pages=4) == -1   # 68 slots > 4 pages of 16
    assert ring_append(k_new=A + 8) == -1           # not 16-byte aligned
    assert ring_append(D=96) == -2
    assert ring_append(dtype=7) == -2
    assert ring_append(ws_bytes=16) == -5           # checked before anything is written

    def select(n_sel=16, Hq=8, Hkv=2, ub=A, D=128):
        return lib.quest_select_pages(vp(A), vp(A), vp(A), vp(A), vp(A), vp(A),
                                      vp(ub) if ub else None, 2, Hq, Hkv, D, 16, 64, 128, n_sel,
                                      1, vp(A), None)
    assert select(n_sel=0) == -2 and select(n_sel=65) == -2
    assert select(Hq=64, Hkv=2) == -2              # group of 32 query heads
    assert select(ub=0) == -1
    assert select(D=96) == -2

    def fused(max_pages=64, n_sel=16):
        return lib.attn_decode_quest_from_bounds(vp(A), vp(A), vp(A), vp(A), vp(A), vp(A), vp(A),
                                                 vp(A), None, 2, 8, 2, 128, 16, max_pages, 128,
                                                 n_sel, 0.125, 1, vp(A), None)
    assert fused(max_pages=30000) == -2            # bound keys beyond shared memory
    assert fused(n_sel=100) == -2
