"""The oracle: a plain fp64 CPU reference for decode attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package. It shares no
code with the CUDA path (``kv_cache_decode_split_gb300``) and neither imports
the other; both read the same seeded inputs from ``workloads``.

The arithmetic lives in ``oracle.c`` (plain C loops in double precision, see
its header for the passages each function follows). This module only loads
the compiled library and marshals arrays. Inputs are passed exactly as stored
(bf16 bit patterns or float32) and widened to double inside the C code.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``,
``tests/test_worked_numbers.py``, ``tests/test_oracle_ring.py`` (cache append and
rolling caches), ``tests/test_oracle_quest.py`` (Quest) and
``tests/test_oracle_delta.py`` (the gated delta rule): brute force on tiny inputs,
closed forms, the pages' printed numbers, independent formulations (the chunk-wise
delta rule, the box maximum) and the invariants the method states.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (OpenMP over independent rows)."""
    src = os.path.join(_HERE, "oracle.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i, l, d = ctypes.c_int, ctypes.c_long, ctypes.c_double
        lib.oracle_kv_cache_bytes.restype = d
        lib.oracle_kv_cache_bytes.argtypes = [d, d, d, d, d]
        lib.oracle_mla_cache_bytes.restype = d
        lib.oracle_mla_cache_bytes.argtypes = [d, d, d, d, d]
        lib.oracle_attention_flops.restype = d
        lib.oracle_attention_flops.argtypes = [d, d, d, d]
        lib.oracle_gqa.restype = None
        lib.oracle_gqa.argtypes = [P, P, P, i, P, P, i, i, i, i, i, i, d, l, l, P, P, i, P, P]
        lib.oracle_gqa_ring.restype = None
        lib.oracle_gqa_ring.argtypes = lib.oracle_gqa.argtypes
        lib.oracle_mla.restype = None
        lib.oracle_mla.argtypes = [P, P, i, P, P, P, P, i, i, i, i, i, i, i, d, P, i, P, P]
        lib.oracle_indexer_scores.restype = None
        lib.oracle_indexer_scores.argtypes = [P, P, P, P, P, i, i, i, i, P, i, l, P]
        lib.oracle_topk.restype = i
        lib.oracle_topk.argtypes = [P, l, i, P]
        lib.oracle_e4m3_decode.restype = d
        lib.oracle_e4m3_decode.argtypes = [i]
        lib.oracle_e4m3_encode.restype = i
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_quantize_e4m3_rows.restype = None
        lib.oracle_quantize_e4m3_rows.argtypes = [P, l, i, P, P]
        lib.oracle_indexer_scores_fp8.restype = None
        lib.oracle_indexer_scores_fp8.argtypes = [P, P, P, P, P, P, P, i, i, i, i, P, i, l, P]
        lib.oracle_quest_minmax.restype = None
        lib.oracle_quest_minmax.argtypes = [P, i, P, i, i, i, i, P, P]
        lib.oracle_quest.restype = None
        lib.oracle_quest.argtypes = [P, P, P, i, P, P, i, i, i, i, i, i, d, i, P, i, P, P, P, P]
        lib.oracle_cache_append.restype = None
        lib.oracle_cache_append.argtypes = [P, P, P, P, i, i, l, i, i, i, i]
        lib.oracle_delta_step.restype = None
        lib.oracle_delta_step.argtypes = [P, P, P, P, P, P, i, i, i, i, P, P]
        _lib = lib
    return _lib


def _arr(x):
    """Contiguous numpy view of a CPU tensor/array, keeping bf16 as raw uint16 bits.

    Returns (array, dtype_code) with dtype_code 0 = float32, 1 = bf16, -1 = other.
    """
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return np.ascontiguousarray(x.view(torch.int16).numpy().view(np.uint16)), 1
            x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return x, 1
    if x.dtype == np.float32:
        return x, 0
    return x, -1


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def kv_cache_bytes(tokens, layers, kv_heads, d_head, bytes_per_elem):
    """KV cache size in bytes ("Attention Optimizations", KV cache size)."""
    return _load().oracle_kv_cache_bytes(float(tokens), float(layers), float(kv_heads),
                                         float(d_head), float(bytes_per_elem))


def mla_cache_bytes(tokens, layers, d_latent, d_rope, bytes_per_elem):
    """MLA latent cache size in bytes: one (latent + RoPE key) row per token per layer."""
    return _load().oracle_mla_cache_bytes(float(tokens), float(layers), float(d_latent),
                                          float(d_rope), float(bytes_per_elem))


def attention_flops(S, layers, heads, head_dim):
    """Attention FLOPs of one token seeing S tokens: 4*S*heads*head_dim per layer."""
    return _load().oracle_attention_flops(float(S), float(layers), float(heads), float(head_dim))


def _pairs_arg(pairs):
    if pairs is None:
        return None, 0
    p = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    return p, p.shape[0]


def gqa(q, k_pool, v_pool, block_table, seq_lens, scale, window=0, n_sink=0, sink_logit=None,
        pairs=None, ring=False):
    """GQA / MHA / MQA decode with optional sliding window, sink tokens and learned sink.

    Shapes: q [B,Hq,D]; k_pool, v_pool [num_pages,Hkv,P,D]; block_table [B,max_pages];
    seq_lens [B]. Returns (out, lse) in float64: out [B,Hq,D] and lse [B,Hq], or
    [n_pairs,D] and [n_pairs] when ``pairs`` lists (b, h) pairs. ``ring``: the pools are
    rolling caches of n_sink + window slots (seq_lens the true lengths), position t read
    from the slot cache append writes it to.
    """
    assert not ring or window > 0
    qa, dt = _arr(q)
    ka, dtk = _arr(k_pool)
    va, dtv = _arr(v_pool)
    assert dt in (0, 1) and dt == dtk == dtv
    bt = np.ascontiguousarray(np.asarray(_arr(block_table)[0], dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(_arr(seq_lens)[0], dtype=np.int32))
    B, Hq, D = qa.shape
    _, Hkv, P, D2 = ka.shape
    assert D2 == D and Hq % Hkv == 0
    sink = None
    if sink_logit is not None:
        sink = np.ascontiguousarray(np.asarray(_arr(sink_logit)[0], dtype=np.float64))
    pa, n_pairs = _pairs_arg(pairs)
    n = n_pairs if pa is not None else B * Hq
    out = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    fn = _load().oracle_gqa_ring if ring else _load().oracle_gqa
    fn(_ptr(qa), _ptr(ka), _ptr(va), dt, _ptr(bt), _ptr(sl), B, Hq, Hkv, D, P, bt.shape[1],
       float(scale), int(window), int(n_sink), _ptr(sink), _ptr(pa), n_pairs, _ptr(out),
       _ptr(lse))
    if pa is None:
        return out.reshape(B, Hq, D), lse.reshape(B, Hq)
    return out, lse


def mla(q, c_pool, block_table, seq_lens, scale, d_v=512, idx=None, idx_count=None, pairs=None):
    """Absorbed-latent MLA decode, dense (idx None) or over selected token indices.

    q [B,H,d_qk], c_pool [num_pages,P,d_qk] (both bf16 or both float32); idx [B,k] int32 logical token
    indices with idx_count[b] valid entries. Returns (out [B,H,d_v], lse [B,H]) float64,
    or per-pair arrays when ``pairs`` is given.
    """
    qa, dt = _arr(q)
    ca, dtc = _arr(c_pool)
    assert dt in (0, 1) and dt == dtc
    bt = np.ascontiguousarray(np.asarray(_arr(block_table)[0], dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(_arr(seq_lens)[0], dtype=np.int32))
    B, H, d_qk = qa.shape
    P = ca.shape[1]
    ia = ic = None
    stride = 0
    if idx is not None:
        ia = np.ascontiguousarray(np.asarray(_arr(idx)[0], dtype=np.int32))
        ic = np.ascontiguousarray(np.asarray(_arr(idx_count)[0], dtype=np.int32))
        stride = ia.shape[1]
    pa, n_pairs = _pairs_arg(pairs)
    n = n_pairs if pa is not None else B * H
    out = np.zeros((n, d_v), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    _load().oracle_mla(_ptr(qa), _ptr(ca), dt, _ptr(bt), _ptr(sl), _ptr(ia), _ptr(ic), stride, B, H,
                       d_qk, d_v, P, bt.shape[1], float(scale), _ptr(pa), n_pairs, _ptr(out),
                       _ptr(lse))
    if pa is None:
        return out.reshape(B, H, d_v), lse.reshape(B, H)
    return out, lse


def indexer_scores(q, k_pool, w, block_table, seq_lens, batches=None):
    """fp64 indexer scores [n_b, max L] for the listed batch rows (NaN past L_b)."""
    qa, dt = _arr(q)
    ka, dtk = _arr(k_pool)
    assert dt == 1 and dtk == 1
    wa = np.ascontiguousarray(np.asarray(_arr(w)[0], dtype=np.float32))
    bt = np.ascontiguousarray(np.asarray(_arr(block_table)[0], dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(_arr(seq_lens)[0], dtype=np.int32))
    B, Hi, Di = qa.shape
    P = ka.shape[1]
    bl = np.arange(B, dtype=np.int32) if batches is None else np.asarray(batches, dtype=np.int32)
    bl = np.ascontiguousarray(bl)
    stride = int(sl[bl].max())
    out = np.full((len(bl), stride), np.nan, dtype=np.float64)
    _load().oracle_indexer_scores(_ptr(qa), _ptr(ka), _ptr(wa), _ptr(bt), _ptr(sl), Hi, Di, P,
                                  bt.shape[1], _ptr(bl), len(bl), stride, _ptr(out))
    return out


def e4m3_decode(codes):
    """Exact value (float64) of each e4m3 code (uint8 array-like; NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.int64)
    lib = _load()
    return np.vectorize(lambda v: lib.oracle_e4m3_decode(int(v)), otypes=[np.float64])(c)


def e4m3_encode(x):
    """Nearest e4m3 code (uint8) to each float32 value, saturating at +-448."""
    xs = np.asarray(x, dtype=np.float32)
    lib = _load()
    return np.vectorize(lambda v: lib.oracle_e4m3_encode(float(v)), otypes=[np.uint8])(xs)


def quantize_e4m3_rows(x):
    """bf16 x [..., C] -> (e4m3 codes uint8 [..., C], float32 scale per row [...])."""
    xa, dt = _arr(x)
    assert dt == 1
    C = xa.shape[-1]
    rows = int(np.prod(xa.shape[:-1]))
    codes = np.zeros(xa.shape, dtype=np.uint8)
    scales = np.zeros(xa.shape[:-1], dtype=np.float32)
    _load().oracle_quantize_e4m3_rows(_ptr(xa), rows, C, _ptr(codes), _ptr(scales))
    return codes, scales


def indexer_scores_fp8(q8, q_scale, k8_pool, k_scale, w, block_table, seq_lens, batches=None):
    """fp64 FP8-indexer scores [n_b, max L] for the listed batch rows (NaN past L_b).

    q8 [B,Hi,Di] and k8_pool [num_pages,P,Di] hold e4m3 codes (uint8), q_scale [B,Hi] and
    k_scale [num_pages,P] their float32 row scales.
    """
    qa = np.ascontiguousarray(np.asarray(q8, dtype=np.uint8))
    ka = np.ascontiguousarray(np.asarray(k8_pool, dtype=np.uint8))
    qs = np.ascontiguousarray(np.asarray(q_scale, dtype=np.float32))
    ks = np.ascontiguousarray(np.asarray(k_scale, dtype=np.float32))
    wa = np.ascontiguousarray(np.asarray(_arr(w)[0], dtype=np.float32))
    bt = np.ascontiguousarray(np.asarray(_arr(block_table)[0], dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(_arr(seq_lens)[0], dtype=np.int32))
    B, Hi, Di = qa.shape
    P = ka.shape[1]
    bl = np.arange(B, dtype=np.int32) if batches is None else np.asarray(batches, dtype=np.int32)
    bl = np.ascontiguousarray(bl)
    stride = int(sl[bl].max())
    out = np.full((len(bl), stride), np.nan, dtype=np.float64)
    _load().oracle_indexer_scores_fp8(_ptr(qa), _ptr(qs), _ptr(ka), _ptr(ks), _ptr(wa), _ptr(bt),
                                      _ptr(sl), Hi, Di, P, bt.shape[1], _ptr(bl), len(bl), stride,
                                      _ptr(out))
    return out


def quest_minmax(k_pool, pages=None):
    """Elementwise (min, max) over each page's keys: k_pool [num_pages, Hkv, P, D] ->
    two float64 arrays [n, Hkv, D] for the listed physical pages (all by default)."""
    ka, dt = _arr(k_pool)
    num_pages, Hkv, P, D = ka.shape
    pl = np.arange(num_pages, dtype=np.int32) if pages is None else \
        np.ascontiguousarray(np.asarray(pages, dtype=np.int32))
    kmin = np.zeros((len(pl), Hkv, D)); kmax = np.zeros((len(pl), Hkv, D))
    _load().oracle_quest_minmax(_ptr(ka), dt, _ptr(pl), len(pl), Hkv, P, D, _ptr(kmin),
                                _ptr(kmax))
    return kmin, kmax


def quest(q, k_pool, v_pool, block_table, seq_lens, scale, n_sel, pairs=None):
    """Quest decode per query head: page bounds, the n_sel best full pages plus the tail,
    attention over them. Returns (out, lse, sel, ub) in float64 / int32:
    out [B,Hq,D], lse [B,Hq], sel [B,Hq,n_sel] (ascending logical pages, -1 padded),
    ub [B,Hq,max_pages] (NaN past the full pages); flattened over ``pairs`` when given."""
    qa, dt = _arr(q)
    ka, dtk = _arr(k_pool)
    va, dtv = _arr(v_pool)
    assert dt in (0, 1) and dt == dtk == dtv
    bt = np.ascontiguousarray(np.asarray(_arr(block_table)[0], dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(_arr(seq_lens)[0], dtype=np.int32))
    B, Hq, D = qa.shape
    _, Hkv, P, _ = ka.shape
    pa, n_pairs = _pairs_arg(pairs)
    n = n_pairs if pa is not None else B * Hq
    mp = bt.shape[1]
    out = np.zeros((n, D)); lse = np.zeros((n,))
    sel = np.zeros((n, n_sel), dtype=np.int32); ub = np.zeros((n, mp))
    _load().oracle_quest(_ptr(qa), _ptr(ka), _ptr(va), dt, _ptr(bt), _ptr(sl), B, Hq, Hkv, D, P,
                         mp, float(scale), int(n_sel), _ptr(pa), n_pairs, _ptr(out), _ptr(lse),
                         _ptr(sel), _ptr(ub))
    if pa is None:
        return (out.reshape(B, Hq, D), lse.reshape(B, Hq), sel.reshape(B, Hq, n_sel),
                ub.reshape(B, Hq, mp))
    return out, lse, sel, ub


def cache_append(pool, new, block_table, seq_lens, window=0, n_sink=0):
    """A copy of `pool` [num_pages, H, P, D] (or [num_pages, P, D]) with each sequence's
    newest token row new[b] ([B, H, D] or [B, D]) written to its paged (window == 0) or
    rolling (window > 0, n_sink + window slots) cache slot. Tensors in, tensor out."""
    import torch
    out = torch.as_tensor(pool).detach().cpu().contiguous().clone()
    src = torch.as_tensor(new).detach().cpu().contiguous().reshape(-1).view(torch.uint8).numpy()
    dst = out.reshape(-1).view(torch.uint8).numpy()     # shares memory with out
    H = out.shape[1] if out.dim() == 4 else 1
    P = out.shape[-2]
    row_bytes = out.shape[-1] * out.element_size()
    bt = np.ascontiguousarray(np.asarray(_arr(block_table)[0], dtype=np.int32))
    sl = np.ascontiguousarray(np.asarray(_arr(seq_lens)[0], dtype=np.int32))
    B = sl.shape[0]
    assert src.size == B * H * row_bytes
    _load().oracle_cache_append(_ptr(dst), _ptr(src), _ptr(bt), _ptr(sl), B, H, row_bytes, P,
                                bt.shape[1], int(window), int(n_sink))
    return out


def delta_step(S, q, k, v, a, beta):
    """One gated delta-rule decode step per head -> (S_new, o), both float64.

    S [n, dv, dk], q and k [n, dk], v [n, dv], beta [n] (float32). a is [n, dk] (one decay
    per key channel, KDA) or [n] (one decay per head, Gated DeltaNet).
    """
    f32 = lambda x: np.ascontiguousarray(np.asarray(_arr(x)[0], dtype=np.float32))
    Sa, qa, ka, va, aa, ba = f32(S), f32(q), f32(k), f32(v), f32(a), f32(beta)
    n, dv, dk = Sa.shape
    per_channel = 1 if aa.ndim == 2 else 0
    assert qa.shape == (n, dk) and ka.shape == (n, dk) and va.shape == (n, dv)
    assert ba.shape == (n,) and (aa.shape == (n, dk) if per_channel else aa.shape == (n,))
    S_out = np.zeros((n, dv, dk), dtype=np.float64)
    o = np.zeros((n, dv), dtype=np.float64)
    _load().oracle_delta_step(_ptr(Sa), _ptr(qa), _ptr(ka), _ptr(va), _ptr(aa), _ptr(ba), n, dk,
                              dv, per_channel, _ptr(S_out), _ptr(o))
    return S_out, o


def topk(scores, k):
    """Indices (ascending) of the min(k, L) largest scores; ties go to the lower index.

    ``scores`` is a 1-D array whose comparisons are taken in its own precision: pass
    float32 values to decide in float32, float64 values to decide in float64.
    """
    s = np.ascontiguousarray(np.asarray(scores, dtype=np.float64).reshape(-1))
    out = np.zeros((max(1, min(int(k), s.shape[0])),), dtype=np.int32)
    cnt = _load().oracle_topk(_ptr(s), s.shape[0], int(k), _ptr(out))
    return out[:cnt].copy()
