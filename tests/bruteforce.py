"""Brute-force fp64 checkers written in matrix form with materialised masks.

Independent of ``oracle/`` (a different formulation, in NumPy): the KV heads are
repeated to every query head the way the GQA code on "Overview of Attention
Mechanism" does (``repeat_kv``), the sliding-window mask is the full T x T mask
of "All the attentions", section 4 (``(j <= i) & (j > i - W)``), the sink mask
is the one "Long context, KV eviction and sparse attention" builds for its
sink_window selection (window part OR ``j < sinks``), and a learned sink is an
extra score column whose value row is zero ("Overview of Attention Mechanism",
StreamingLLM, softmax-off-by-one). Tiny inputs only.
"""
import numpy as np
import torch


def f64(t):
    return t.to(torch.float64).numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def gather_tokens(pool, block_table, b, L, page_size, head=None):
    """Logical tokens 0..L-1 of sequence b as an [L, D] array."""
    pool = f64(pool)
    bt = np.asarray(block_table)
    rows = []
    for t in range(L):
        page = bt[b, t // page_size]
        rows.append(pool[page, head, t % page_size] if head is not None else pool[page, t % page_size])
    return np.stack(rows)


def sliding_window_mask(T, W):
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    return (j <= i) & (j > i - W)


def gqa(q, k_pool, v_pool, block_table, seq_lens, scale, window=0, n_sink=0, sink_logit=None):
    q = f64(q)
    B, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    P = k_pool.shape[2]
    n_rep = Hq // Hkv
    out = np.zeros((B, Hq, D))
    lse = np.zeros((B, Hq))
    for b in range(B):
        L = int(seq_lens[b])
        K = np.stack([gather_tokens(k_pool, block_table, b, L, P, g) for g in range(Hkv)])  # [Hkv,L,D]
        V = np.stack([gather_tokens(v_pool, block_table, b, L, P, g) for g in range(Hkv)])
        K = K[:, None].repeat(n_rep, axis=1).reshape(Hq, L, D)   # repeat_kv
        V = V[:, None].repeat(n_rep, axis=1).reshape(Hq, L, D)
        causal = np.tril(np.ones((L, L), dtype=bool))
        if window > 0:
            mask = sliding_window_mask(L, window)
        else:
            mask = causal.copy()
        if n_sink > 0:
            mask = (mask | (np.arange(L)[None, :] < n_sink)) & causal
        row = mask[L - 1]                                         # the decoded token is the last one
        S = np.einsum("hd,hld->hl", q[b], K) * scale
        S = np.where(row[None, :], S, -np.inf)
        Vx = V
        if sink_logit is not None:
            S = np.concatenate([S, f64(sink_logit)[:, None]], axis=1)
            Vx = np.concatenate([V, np.zeros((Hq, 1, D))], axis=1)
        mx = S.max(axis=1, keepdims=True)
        E = np.exp(S - mx)
        Z = E.sum(axis=1, keepdims=True)
        out[b] = np.einsum("hl,hld->hd", E / Z, Vx)
        lse[b] = (mx + np.log(Z))[:, 0]
    return out, lse


def mla(q, c_pool, block_table, seq_lens, scale, d_v=512, idx=None, idx_count=None):
    q = f64(q)
    B, H, dqk = q.shape
    P = c_pool.shape[1]
    out = np.zeros((B, H, d_v))
    lse = np.zeros((B, H))
    for b in range(B):
        L = int(seq_lens[b])
        C = gather_tokens(c_pool, block_table, b, L, P)          # [L, 576]
        if idx is not None:
            sel = np.zeros(L, dtype=bool)
            sel[np.asarray(idx)[b, :int(idx_count[b])]] = True
        else:
            sel = np.ones(L, dtype=bool)
        S = np.where(sel[None, :], q[b] @ C.T * scale, -np.inf)
        mx = S.max(axis=1, keepdims=True)
        E = np.exp(S - mx)
        Z = E.sum(axis=1, keepdims=True)
        out[b] = (E / Z) @ C[:, :d_v]
        lse[b] = (mx + np.log(Z))[:, 0]
    return out, lse


def indexer_scores(q, k_pool, w, block_table, seq_lens, b):
    L = int(seq_lens[b])
    K = gather_tokens(k_pool, block_table, b, L, k_pool.shape[1])   # [L, Di]
    dots = f64(q)[b] @ K.T                                            # [Hi, L]
    return (f64(w)[b][:, None] * np.maximum(dots, 0.0)).sum(axis=0)


def topk_full_sort(scores, k):
    order = sorted(range(len(scores)), key=lambda t: (-scores[t], t))
    return sorted(order[:min(k, len(scores))])
