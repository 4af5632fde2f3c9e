"""kv_cache_decode_split_gb300 -- single-token decode attention over a long, paged KV cache
on one GB300 GPU.

A thin Python binding over the C ABI of ``libkvdecode.so`` (``include/kvdecode.h``): each
function has the name of its C entry point, takes torch CUDA tensors, and only marshals
pointers, sizes and the current stream. Every step of the computation runs in the
library's CUDA kernels; PyTorch provides device memory and streams.

Operations:
  attn_decode_gqa_paged   GQA / MHA / MQA over a paged cache
  attn_decode_swa_sink    sliding window + sink tokens / learned sink logit
  attn_decode_mla         absorbed-latent MLA (576-wide rows, value = first 512)
  dsa_indexer_topk        indexer scores + top-k selection
  dsa_topk                top-k selection over given scores
  attn_decode_mla_sparse  MLA over the selected tokens
  dsa_indexer_topk_fp8    the indexer on e4m3 keys and queries with row scales
  quantize_e4m3_rows      e4m3 row quantizer; dsa_indexer_cache_append_fp8 its cache append
  delta_decode_step       one gated delta-rule (Gated DeltaNet / KDA) decode step
  cache_append            the new token's K/V (or latent row) into a paged or rolling cache
  attn_decode_swa_ring    sliding window + sinks over a rolling cache
  attn_decode_swa_ring_append   cache_append of the newest token, then attn_decode_swa_ring
  quest_page_minmax, quest_select_pages, attn_decode_quest   Quest page selection
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _lib
from ._lib import KvdError, OP, OPTION

lib = _lib.load()

__all__ = [
    "attn_decode_gqa_paged", "attn_decode_swa_sink", "attn_decode_mla", "dsa_indexer_topk",
    "dsa_indexer_topk_fp8", "quantize_e4m3_rows", "dsa_indexer_cache_append_fp8",
    "delta_decode_step", "attn_decode_swa_ring", "attn_decode_swa_ring_append", "cache_append",
    "quest_page_minmax",
    "quest_select_pages", "attn_decode_quest", "quest_page_bounds",
    "attn_decode_quest_from_bounds",
    "dsa_topk", "attn_decode_mla_sparse", "kvd_workspace_size", "kvd_check_device_error",
    "kvd_set_option", "Workspace", "KvdError",
]

_DT = {torch.float32: 0, torch.bfloat16: 1}


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(status, where):
    if status != 0:
        raise KvdError(status, where)


def _need(t, name, dtype=None, dim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dims")


def kvd_workspace_size(op, B, H, Hkv=1, D=0, max_len=1, window=0, n_sink=0, k=0):
    return int(lib.kvd_workspace_size(OP[op] if isinstance(op, str) else int(op), int(B), int(H),
                                      int(Hkv), int(D), int(max_len), int(window), int(n_sink),
                                      int(k)))


def kvd_check_device_error(ws, stream=None):
    """Synchronise and return the device error recorded in a workspace (0 if none)."""
    buf = ws.buffer if isinstance(ws, Workspace) else ws
    return int(lib.kvd_check_device_error(_p(buf), _stream(stream)))


def kvd_set_option(option, value):
    """Process-wide library option (measurement and tests of the library; see kvdecode.h):
    "pdl", "gqa_chunk", "mla_min_tiles", "wait_timeout_test" or "gqa_cluster"."""
    _check(lib.kvd_set_option(OPTION[option] if isinstance(option, str) else int(option),
                              int(value)), "kvd_set_option")


class Workspace:
    """A zero-filled device buffer reused across calls (grown on demand).

    The kernels of one operation family (GQA / SWA; MLA; DSA indexer / top-k) leave the
    parts they rely on zeroed for the family's next call with the same shape arguments (the
    layout of the buffer follows them), so the buffer is zeroed only when it is
    (re)allocated, handed to another family, or used with other shape arguments. Calls
    sharing one workspace must be ordered on one stream.
    """

    def __init__(self, device=None):
        self.device = torch.device(device) if device is not None else torch.device("cuda")
        self.buffer = torch.zeros(0, dtype=torch.uint8, device=self.device)
        self.family = None
        self.layout = None

    def get(self, nbytes: int, family=None, layout=None) -> torch.Tensor:
        key = (family, layout)
        if self.buffer.numel() < nbytes:
            self.buffer = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=self.device)
        elif family is not None and self.family is not None and key != (self.family, self.layout):
            # another family's kernels, or the same family with another layout, may have
            # left non-zero state where this call's kernels expect zeros
            self.buffer.zero_()
        if family is not None:
            self.family, self.layout = family, layout
        return self.buffer


_default_ws = {}


def _ws(workspace, nbytes, device, family, layout=None):
    """Workspace buffer for one call of an operation family ("gqa", "mla" or "dsa");
    `layout` names the shape arguments the buffer's layout follows."""
    if workspace is None:
        key = (torch.device(device).index, family)
        workspace = _default_ws.setdefault(key, Workspace(device))
    if isinstance(workspace, Workspace):
        buf = workspace.get(nbytes, family, layout)
    else:
        buf = workspace
    if buf.numel() < nbytes:
        raise KvdError(-5, "workspace")
    return buf


def _gqa_args(q, k_pool, v_pool, block_table, seq_lens):
    _need(q, "q", dim=3)
    _need(k_pool, "k_pool", q.dtype, 4)
    _need(v_pool, "v_pool", q.dtype, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    if q.dtype not in _DT:
        raise TypeError("q must be float32 or bfloat16")
    B, Hq, D = q.shape
    num_pages, Hkv, P, D2 = k_pool.shape
    if D2 != D or tuple(v_pool.shape) != tuple(k_pool.shape):
        raise ValueError("k_pool / v_pool must be [num_pages, Hkv, page_size, D]")
    if block_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("block_table / seq_lens batch mismatch")
    return B, Hq, Hkv, D, P, block_table.shape[1], num_pages


def attn_decode_gqa_paged(q, k_pool, v_pool, block_table, seq_lens, scale=None, out=None,
                          lse_out=None, workspace=None, stream=None):
    """Decode attention of q [B,Hq,D] over a paged K/V pool [num_pages,Hkv,P,D]."""
    B, Hq, Hkv, D, P, max_pages, num_pages = _gqa_args(q, k_pool, v_pool, block_table, seq_lens)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    nbytes = kvd_workspace_size("gqa", B, Hq, Hkv, D, max_pages * P)
    ws = _ws(workspace, nbytes, q.device, "gqa", layout=("gqa", B, Hq, Hkv, D, max_pages * P))
    st = lib.attn_decode_gqa_paged(_p(q), _p(k_pool), _p(v_pool), _p(block_table), _p(seq_lens),
                                   _p(out), _p(lse_out), B, Hq, Hkv, D, P, max_pages, num_pages,
                                   scale, _DT[q.dtype], _p(ws), ws.numel(), _stream(stream))
    _check(st, "attn_decode_gqa_paged")
    return out


def attn_decode_swa_sink(q, k_pool, v_pool, block_table, seq_lens, window, n_sink_tokens=0,
                         sink_logit=None, scale=None, out=None, lse_out=None, workspace=None,
                         stream=None):
    """Sliding-window (+ sink tokens, + learned sink logit [Hq]) decode attention."""
    B, Hq, Hkv, D, P, max_pages, num_pages = _gqa_args(q, k_pool, v_pool, block_table, seq_lens)
    if sink_logit is not None:
        _need(sink_logit, "sink_logit", torch.float32, 1)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    nbytes = kvd_workspace_size("swa", B, Hq, Hkv, D, max_pages * P, window, n_sink_tokens)
    ws = _ws(workspace, nbytes, q.device, "gqa",
             layout=("swa", B, Hq, Hkv, D, max_pages * P, window, n_sink_tokens))
    st = lib.attn_decode_swa_sink(_p(q), _p(k_pool), _p(v_pool), _p(block_table), _p(seq_lens),
                                  _p(out), _p(lse_out), B, Hq, Hkv, D, P, max_pages, num_pages,
                                  scale, _DT[q.dtype], int(window), int(n_sink_tokens),
                                  _p(sink_logit), _p(ws), ws.numel(), _stream(stream))
    _check(st, "attn_decode_swa_sink")
    return out


def attn_decode_swa_ring(q, k_ring, v_ring, block_table, seq_lens, window, n_sink_tokens=0,
                         sink_logit=None, scale=None, out=None, lse_out=None, workspace=None,
                         stream=None):
    """Sliding-window (+ sinks) decode over a rolling cache of n_sink_tokens + window slots
    per sequence (written by cache_append with the same window); seq_lens are the true
    sequence lengths."""
    B, Hq, Hkv, D, P, max_pages, num_pages = _gqa_args(q, k_ring, v_ring, block_table, seq_lens)
    if sink_logit is not None:
        _need(sink_logit, "sink_logit", torch.float32, 1)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    # the ring is read like a dense cache of max_pages * P slots
    nbytes = kvd_workspace_size("gqa", B, Hq, Hkv, D, max_pages * P)
    ws = _ws(workspace, nbytes, q.device, "gqa", layout=("gqa", B, Hq, Hkv, D, max_pages * P))
    st = lib.attn_decode_swa_ring(_p(q), _p(k_ring), _p(v_ring), _p(block_table), _p(seq_lens),
                                  _p(out), _p(lse_out), B, Hq, Hkv, D, P, max_pages, num_pages,
                                  scale, _DT[q.dtype], int(window), int(n_sink_tokens),
                                  _p(sink_logit), _p(ws), ws.numel(), _stream(stream))
    _check(st, "attn_decode_swa_ring")
    return out


def attn_decode_swa_ring_append(q, k_new, v_new, k_ring, v_ring, block_table, seq_lens, window,
                                n_sink_tokens=0, sink_logit=None, scale=None, out=None,
                                lse_out=None, workspace=None, stream=None):
    """One decode step on a rolling cache: cache_append of each sequence's newest token
    (k_new, v_new [B, Hkv, D]) into k_ring / v_ring (updated in place), then
    attn_decode_swa_ring over the updated ring, in one call (one launch for bf16 rings). A
    bad length or page id of the newest slot is recorded in the workspace's error flag."""
    B, Hq, Hkv, D, P, max_pages, num_pages = _gqa_args(q, k_ring, v_ring, block_table, seq_lens)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, n, q.dtype, 3)
        if tuple(t.shape) != (B, Hkv, D):
            raise ValueError(f"{n} must be [B, Hkv, D]")
    if sink_logit is not None:
        _need(sink_logit, "sink_logit", torch.float32, 1)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    nbytes = kvd_workspace_size("gqa", B, Hq, Hkv, D, max_pages * P)
    ws = _ws(workspace, nbytes, q.device, "gqa", layout=("gqa", B, Hq, Hkv, D, max_pages * P))
    st = lib.attn_decode_swa_ring_append(
        _p(q), _p(k_new), _p(v_new), _p(k_ring), _p(v_ring), _p(block_table), _p(seq_lens),
        _p(out), _p(lse_out), B, Hq, Hkv, D, P, max_pages, num_pages, scale, _DT[q.dtype],
        int(window), int(n_sink_tokens), _p(sink_logit), _p(ws), ws.numel(), _stream(stream))
    _check(st, "attn_decode_swa_ring_append")
    return out


def cache_append(k_new, v_new, k_pool, v_pool, block_table, seq_lens, window=0, n_sink=0,
                 err=None, stream=None):
    """Write each sequence's newest token (position seq_lens[b] - 1) into its cache slot.

    k_new / v_new [B, H, D] into k_pool / v_pool [num_pages, H, page_size, D]; for the MLA
    latent cache pass v_new = v_pool = None, k_new [B, 576] and k_pool [num_pages, P, 576].
    window > 0: a rolling cache of n_sink + window slots. `err` (int32 [1], device) receives
    a device error code and is returned.
    """
    _need(k_new, "k_new")
    _need(k_pool, "k_pool", k_new.dtype)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    if k_new.dtype not in _DT:
        raise TypeError("k_new must be float32 or bfloat16")
    if (v_new is None) != (v_pool is None):
        raise ValueError("v_new and v_pool go together")
    if v_new is not None:
        _need(v_new, "v_new", k_new.dtype)
        _need(v_pool, "v_pool", k_new.dtype)
        if v_new.shape != k_new.shape or v_pool.shape != k_pool.shape:
            raise ValueError("v_new / v_pool must match k_new / k_pool")
    B, D = k_new.shape[0], k_new.shape[-1]
    if k_pool.dim() == 4:
        num_pages, H, P, D2 = k_pool.shape
    elif k_pool.dim() == 3:
        (num_pages, P, D2), H = k_pool.shape, 1
    else:
        raise ValueError("k_pool must be [num_pages, H, P, D] or [num_pages, P, D]")
    if D2 != D or k_new.numel() != B * H * D:
        raise ValueError("k_new must be [B, H, D] matching the pool")
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=k_new.device)
    st = lib.kvd_cache_append(_p(k_new), _p(v_new), _p(k_pool), _p(v_pool), _p(block_table),
                              _p(seq_lens), B, H, D, P, block_table.shape[1], num_pages,
                              _DT[k_new.dtype], int(window), int(n_sink), _p(err),
                              _stream(stream))
    _check(st, "kvd_cache_append")
    return err


def _err(err, device):
    return torch.zeros(1, dtype=torch.int32, device=device) if err is None else err


def quest_page_minmax(k_pool, kmin=None, kmax=None, pages=None, err=None, stream=None):
    """Per-page elementwise key minimum and maximum: k_pool [num_pages, Hkv, P, D] ->
    (kmin, kmax) [num_pages, Hkv, D] in the pool's dtype, for the physical pages listed in
    `pages` (int32, device; None = all). Returns (kmin, kmax, err)."""
    _need(k_pool, "k_pool", dim=4)
    if k_pool.dtype not in _DT:
        raise TypeError("k_pool must be float32 or bfloat16")
    num_pages, Hkv, P, D = k_pool.shape
    shape = (num_pages, Hkv, D)
    kmin = torch.empty(shape, dtype=k_pool.dtype, device=k_pool.device) if kmin is None else kmin
    kmax = torch.empty(shape, dtype=k_pool.dtype, device=k_pool.device) if kmax is None else kmax
    _need(kmin, "kmin", k_pool.dtype)
    _need(kmax, "kmax", k_pool.dtype)
    if pages is not None:
        _need(pages, "pages", torch.int32, 1)
    err = _err(err, k_pool.device)
    st = lib.quest_page_minmax(_p(k_pool), _p(kmin), _p(kmax), _p(pages),
                               0 if pages is None else pages.numel(), num_pages, Hkv, P, D,
                               _DT[k_pool.dtype], _p(err), _stream(stream))
    _check(st, "quest_page_minmax")
    return kmin, kmax, err


def quest_select_pages(q, kmin, kmax, block_table, seq_lens, n_sel, page_size, sel=None,
                       ub_out=None, err=None, stream=None):
    """Each query head's n_sel full pages with the largest score bound (ascending logical
    page ids, -1 padded): sel [B, Hq, n_sel] int32."""
    _need(q, "q", dim=3)
    _need(kmin, "kmin", q.dtype, 3)
    _need(kmax, "kmax", q.dtype, 3)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, Hq, D = q.shape
    num_pages, Hkv, _ = kmin.shape
    max_pages = block_table.shape[1]
    sel = torch.empty(B, Hq, n_sel, dtype=torch.int32, device=q.device) if sel is None else sel
    if ub_out is None:
        ub_out = torch.empty(B, Hq, max_pages, dtype=torch.float32, device=q.device)
    err = _err(err, q.device)
    st = lib.quest_select_pages(_p(q), _p(kmin), _p(kmax), _p(block_table), _p(seq_lens),
                                _p(sel), _p(ub_out), B, Hq, Hkv, D, int(page_size), max_pages,
                                num_pages, int(n_sel), _DT[q.dtype], _p(err), _stream(stream))
    _check(st, "quest_select_pages")
    return sel


def attn_decode_quest(q, k_pool, v_pool, block_table, seq_lens, sel, scale=None, out=None,
                      lse_out=None, err=None, stream=None):
    """Attention of each query head over its chosen pages (sel from quest_select_pages)
    and the tokens past the last full page."""
    B, Hq, Hkv, D, P, max_pages, num_pages = _gqa_args(q, k_pool, v_pool, block_table, seq_lens)
    _need(sel, "sel", torch.int32, 3)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    err = _err(err, q.device)
    st = lib.attn_decode_quest(_p(q), _p(k_pool), _p(v_pool), _p(block_table), _p(seq_lens),
                               _p(sel), _p(out), _p(lse_out), B, Hq, Hkv, D, P, max_pages,
                               num_pages, sel.shape[2], scale, _DT[q.dtype], _p(err),
                               _stream(stream))
    _check(st, "attn_decode_quest")
    return out


def quest_page_bounds(q, kmin, kmax, block_table, seq_lens, page_size, ub=None, err=None,
                      stream=None):
    """Each query head's page bounds: ub [B, Hq, max_pages] float32 (NaN past full pages)."""
    _need(q, "q", dim=3)
    _need(kmin, "kmin", q.dtype, 3)
    _need(kmax, "kmax", q.dtype, 3)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, Hq, D = q.shape
    num_pages, Hkv, _ = kmin.shape
    max_pages = block_table.shape[1]
    ub = torch.empty(B, Hq, max_pages, dtype=torch.float32, device=q.device) if ub is None else ub
    err = _err(err, q.device)
    st = lib.quest_page_bounds(_p(q), _p(kmin), _p(kmax), _p(block_table), _p(seq_lens), _p(ub),
                               B, Hq, Hkv, D, int(page_size), max_pages, num_pages, _DT[q.dtype],
                               _p(err), _stream(stream))
    _check(st, "quest_page_bounds")
    return ub


def attn_decode_quest_from_bounds(q, k_pool, v_pool, block_table, seq_lens, ub, n_sel,
                                  scale=None, sel_out=None, out=None, lse_out=None, err=None,
                                  stream=None):
    """Choice of each head's n_sel best pages from ub and attention over them, one launch.
    Returns (out, sel_out)."""
    B, Hq, Hkv, D, P, max_pages, num_pages = _gqa_args(q, k_pool, v_pool, block_table, seq_lens)
    _need(ub, "ub", torch.float32, 3)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    sel_out = (torch.empty(B, Hq, n_sel, dtype=torch.int32, device=q.device)
               if sel_out is None else sel_out)
    err = _err(err, q.device)
    st = lib.attn_decode_quest_from_bounds(_p(q), _p(k_pool), _p(v_pool), _p(block_table),
                                           _p(seq_lens), _p(ub), _p(sel_out), _p(out),
                                           _p(lse_out), B, Hq, Hkv, D, P, max_pages, num_pages,
                                           int(n_sel), scale, _DT[q.dtype], _p(err),
                                           _stream(stream))
    _check(st, "attn_decode_quest_from_bounds")
    return out, sel_out


def _mla_args(q, c_pool, block_table, seq_lens):
    _need(q, "q", torch.bfloat16, 3)
    _need(c_pool, "c_pool", torch.bfloat16, 3)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, H, d_qk = q.shape
    num_pages, P, d2 = c_pool.shape
    if d2 != d_qk:
        raise ValueError("c_pool must be [num_pages, page_size, d_qk]")
    return B, H, d_qk, P, block_table.shape[1], num_pages


def attn_decode_mla(q, c_pool, block_table, seq_lens, scale=1.0 / math.sqrt(192), d_v=512,
                    out=None, lse_out=None, workspace=None, stream=None):
    """Absorbed-latent MLA decode: q [B,H,576] over latent rows [num_pages,P,576]."""
    B, H, d_qk, P, max_pages, num_pages = _mla_args(q, c_pool, block_table, seq_lens)
    out = torch.empty(B, H, d_v, dtype=torch.bfloat16, device=q.device) if out is None else out
    nbytes = kvd_workspace_size("mla", B, H, 1, d_v, max_pages * P)
    ws = _ws(workspace, nbytes, q.device, "mla", layout=("mla", B, H, max_pages * P))
    st = lib.attn_decode_mla(_p(q), _p(c_pool), _p(block_table), _p(seq_lens), _p(out),
                             _p(lse_out), B, H, d_qk, d_v, P, max_pages, num_pages, float(scale),
                             _p(ws), ws.numel(), _stream(stream))
    _check(st, "attn_decode_mla")
    return out


def dsa_indexer_topk(q_idx, k_idx_pool, w, block_table, seq_lens, k=2048, topk_idx=None,
                     topk_count=None, scores_out=None, workspace=None, stream=None):
    """Indexer scores of every cached token and the indices of the k largest (ascending)."""
    _need(q_idx, "q_idx", torch.bfloat16, 3)
    _need(k_idx_pool, "k_idx_pool", torch.bfloat16, 3)
    _need(w, "w", torch.float32, 2)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, Hi, Di = q_idx.shape
    num_pages, P, _ = k_idx_pool.shape
    max_pages = block_table.shape[1]
    dev = q_idx.device
    topk_idx = torch.empty(B, k, dtype=torch.int32, device=dev) if topk_idx is None else topk_idx
    topk_count = torch.empty(B, dtype=torch.int32, device=dev) if topk_count is None else topk_count
    nbytes = kvd_workspace_size("dsa_topk", B, Hi, 1, Di, max_pages * P, k=k)
    ws = _ws(workspace, nbytes, dev, "dsa", layout=(B, max_pages * P, int(k)))
    st = lib.dsa_indexer_topk(_p(q_idx), _p(k_idx_pool), _p(w), _p(block_table), _p(seq_lens),
                              _p(topk_idx), _p(topk_count), _p(scores_out), B, Hi, Di, P,
                              max_pages, num_pages, int(k), _p(ws), ws.numel(), _stream(stream))
    _check(st, "dsa_indexer_topk")
    return topk_idx, topk_count


def dsa_indexer_topk_fp8(q8, q_scale, k8_pool, k_scale, w, block_table, seq_lens, k=2048,
                         topk_idx=None, topk_count=None, scores_out=None, workspace=None,
                         stream=None):
    """FP8 indexer: e4m3 codes (uint8) with float32 row scales; same outputs as the bf16 one."""
    _need(q8, "q8", torch.uint8, 3)
    _need(q_scale, "q_scale", torch.float32, 2)
    _need(k8_pool, "k8_pool", torch.uint8, 3)
    _need(k_scale, "k_scale", torch.float32, 2)
    _need(w, "w", torch.float32, 2)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, Hi, Di = q8.shape
    num_pages, P, _ = k8_pool.shape
    max_pages = block_table.shape[1]
    dev = q8.device
    topk_idx = torch.empty(B, k, dtype=torch.int32, device=dev) if topk_idx is None else topk_idx
    topk_count = torch.empty(B, dtype=torch.int32, device=dev) if topk_count is None else topk_count
    nbytes = kvd_workspace_size("dsa_topk", B, Hi, 1, Di, max_pages * P, k=k)
    ws = _ws(workspace, nbytes, dev, "dsa", layout=(B, max_pages * P, int(k)))
    st = lib.dsa_indexer_topk_fp8(_p(q8), _p(q_scale), _p(k8_pool), _p(k_scale), _p(w),
                                  _p(block_table), _p(seq_lens), _p(topk_idx), _p(topk_count),
                                  _p(scores_out), B, Hi, Di, P, max_pages, num_pages, int(k),
                                  _p(ws), ws.numel(), _stream(stream))
    _check(st, "dsa_indexer_topk_fp8")
    return topk_idx, topk_count


def quantize_e4m3_rows(x, codes=None, scales=None, stream=None):
    """bf16 x [..., C] -> (e4m3 codes uint8 [..., C], float32 scale per row [...])."""
    _need(x, "x", torch.bfloat16)
    C = x.shape[-1]
    rows = x.numel() // C
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device) if codes is None else codes
    scales = (torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
              if scales is None else scales)
    st = lib.kvd_quantize_e4m3_rows(_p(x), _p(codes), _p(scales), rows, C, _stream(stream))
    _check(st, "kvd_quantize_e4m3_rows")
    return codes, scales


def dsa_indexer_cache_append_fp8(k_new, block_table, seq_lens, k8_pool, k_scale, err=None,
                                 stream=None):
    """Quantize each sequence's new indexer key k_new [B, Di] bf16 into its cache row at
    position seq_lens[b] - 1. `err` (int32 [1] on the device) receives a device error code."""
    _need(k_new, "k_new", torch.bfloat16, 2)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(k8_pool, "k8_pool", torch.uint8, 3)
    _need(k_scale, "k_scale", torch.float32, 2)
    B, Di = k_new.shape
    num_pages, P, _ = k8_pool.shape
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=k_new.device)
    st = lib.dsa_indexer_cache_append_fp8(_p(k_new), _p(block_table), _p(seq_lens), _p(k8_pool),
                                          _p(k_scale), B, Di, P, block_table.shape[1], num_pages,
                                          _p(err), _stream(stream))
    _check(st, "dsa_indexer_cache_append_fp8")
    return err


def delta_decode_step(S, q, k, v, a, beta, o=None, stream=None):
    """One gated delta-rule decode step per head, in place on S.

    S [..., dv, dk] float32 (updated), q and k [..., dk], v [..., dv], beta [...] float32;
    a is [..., dk] (one decay per key channel, KDA) or [...] (one per head, Gated DeltaNet).
    Returns o [..., dv] float32 = S_new q.
    """
    _need(S, "S", torch.float32)
    dv, dk = S.shape[-2], S.shape[-1]
    n = S.numel() // (dv * dk)
    for t, name, width in ((q, "q", dk), (k, "k", dk), (v, "v", dv)):
        _need(t, name, torch.float32)
        if t.numel() != n * width:
            raise ValueError(f"{name} must hold {n} x {width} values")
    _need(a, "a", torch.float32)
    _need(beta, "beta", torch.float32)
    if beta.numel() != n:
        raise ValueError(f"beta must hold {n} values")
    if a.numel() == n * dk:
        per_channel = 1
    elif a.numel() == n:
        per_channel = 0
    else:
        raise ValueError(f"a must hold {n} x {dk} (per channel) or {n} (per head) values")
    o = torch.empty(S.shape[:-1], dtype=torch.float32, device=S.device) if o is None else o
    _need(o, "o", torch.float32)
    st = lib.kvd_delta_decode_step(_p(S), _p(q), _p(k), _p(v), _p(a), _p(beta), _p(o), n, dk,
                                   dv, per_channel, _stream(stream))
    _check(st, "kvd_delta_decode_step")
    return o


def dsa_topk(scores, lens, k=2048, topk_idx=None, topk_count=None, workspace=None, stream=None):
    """Top-k selection over scores [B, stride] float32 with lens [B] valid entries per row."""
    _need(scores, "scores", torch.float32, 2)
    _need(lens, "lens", torch.int32, 1)
    B, stride = scores.shape
    dev = scores.device
    topk_idx = torch.empty(B, k, dtype=torch.int32, device=dev) if topk_idx is None else topk_idx
    topk_count = torch.empty(B, dtype=torch.int32, device=dev) if topk_count is None else topk_count
    nbytes = kvd_workspace_size("dsa_topk", B, 1, 1, 0, stride, k=k)
    ws = _ws(workspace, nbytes, dev, "dsa", layout=(B, stride, int(k)))
    st = lib.dsa_topk(_p(scores), _p(lens), _p(topk_idx), _p(topk_count), B, stride, int(k),
                      _p(ws), ws.numel(), _stream(stream))
    _check(st, "dsa_topk")
    return topk_idx, topk_count


def attn_decode_mla_sparse(q, c_pool, block_table, seq_lens, topk_idx, topk_count,
                           scale=1.0 / math.sqrt(192), d_v=512, out=None, lse_out=None,
                           workspace=None, stream=None):
    """MLA over the selected tokens: topk_idx [B,k] logical positions, topk_count [B]."""
    B, H, d_qk, P, max_pages, num_pages = _mla_args(q, c_pool, block_table, seq_lens)
    _need(topk_idx, "topk_idx", torch.int32, 2)
    _need(topk_count, "topk_count", torch.int32, 1)
    k = topk_idx.shape[1]
    out = torch.empty(B, H, d_v, dtype=torch.bfloat16, device=q.device) if out is None else out
    nbytes = kvd_workspace_size("mla_sparse", B, H, 1, d_v, max_pages * P, k=k)
    ws = _ws(workspace, nbytes, q.device, "mla", layout=("mla_sparse", B, H, int(k)))
    st = lib.attn_decode_mla_sparse(_p(q), _p(c_pool), _p(block_table), _p(seq_lens),
                                    _p(topk_idx), _p(topk_count), _p(out), _p(lse_out), B, H,
                                    d_qk, d_v, k, P, max_pages, num_pages, float(scale), _p(ws),
                                    ws.numel(), _stream(stream))
    _check(st, "attn_decode_mla_sparse")
    return out
