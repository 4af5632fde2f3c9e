"""Seeded synthetic inputs for single-token decode attention over a paged KV cache.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests. It holds shapes, seeds and random draws only: no attention,
indexer or selection arithmetic lives here.

Recipe (every workload): a CPU ``torch.Generator`` seeded with
``1000 * workload_id + tensor_id`` draws float32 normals, which are scaled by
the workload's factor and rounded once to the storage dtype (bf16, or kept
float32 for the tiny fp32 case). Both the GPU path and the oracle read these
same rounded values.

Cache layouts (one layer):
  * GQA / SWA pool  ``[num_pages, Hkv, page_size, D]``  (K and V separately)
  * MLA latent pool ``[num_pages, page_size, 576]``     (512 latent + 64 RoPE key)
  * indexer key pool ``[num_pages, page_size, 128]``
  * ``block_table [B, max_pages]`` int32 maps a sequence's logical page to a
    physical page; ``seq_lens [B]`` int32 counts cached tokens including the
    token being decoded (its K/V are appended before attention runs).

Unused pool pages are filled with normals too, so a wrong page index reads
plausible-looking garbage rather than zeros.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(shape, seed: int, factor: float = 1.0, dtype=torch.bfloat16) -> torch.Tensor:
    """float32 N(0,1) draws times ``factor``, rounded once to ``dtype``."""
    x = torch.randn(*shape, generator=_gen(seed), dtype=torch.float32)
    if factor != 1.0:
        x.mul_(factor)
    return x.to(dtype)


def uniform_int(lo: int, hi: int, n: int, seed: int) -> torch.Tensor:
    """n integers uniform in [lo, hi] (inclusive), int32."""
    return torch.randint(lo, hi + 1, (n,), generator=_gen(seed), dtype=torch.int32)


def block_table_for(seq_lens, page_size: int, max_pages: int, shuffle: bool, seed: int,
                    extra_pages: int = 0):
    """Assign physical pages to every sequence's logical pages.

    Returns ``(block_table [B, max_pages] int32, num_pages)``. Without
    ``shuffle`` the assignment is the identity layout (sequence b's pages are
    contiguous, in order, at ``b * max_pages``). With ``shuffle`` the pool holds
    exactly the pages in use plus ``extra_pages`` spare ones, handed out in a
    random permutation. Table slots past a sequence's last page hold -1.
    """
    lens = [int(x) for x in seq_lens]
    B = len(lens)
    bt = torch.full((B, max_pages), -1, dtype=torch.int32)
    if not shuffle:
        for b, L in enumerate(lens):
            n = -(-L // page_size)
            bt[b, :n] = torch.arange(b * max_pages, b * max_pages + n, dtype=torch.int32)
        return bt, B * max_pages
    used = [-(-L // page_size) for L in lens]
    num_pages = sum(used) + extra_pages
    perm = torch.randperm(num_pages, generator=_gen(seed), dtype=torch.int64).to(torch.int32)
    pos = 0
    for b, n in enumerate(used):
        bt[b, :n] = perm[pos:pos + n]
        pos += n
    return bt, num_pages


@dataclass
class GQAInputs:
    q: torch.Tensor            # [B, Hq, D]
    k_pool: torch.Tensor       # [num_pages, Hkv, P, D]
    v_pool: torch.Tensor       # [num_pages, Hkv, P, D]
    block_table: torch.Tensor  # [B, max_pages] int32
    seq_lens: torch.Tensor     # [B] int32
    page_size: int
    scale: float
    window: int = 0            # 0: no window (dense)
    n_sink: int = 0            # sink tokens always kept
    sink_logit: torch.Tensor | None = None  # [Hq] float32, learned sink logit
    ring: bool = False         # pools are rolling caches of n_sink + window slots

    @property
    def B(self): return self.q.shape[0]
    @property
    def Hq(self): return self.q.shape[1]
    @property
    def Hkv(self): return self.k_pool.shape[1]
    @property
    def D(self): return self.q.shape[2]
    @property
    def max_pages(self): return self.block_table.shape[1]
    @property
    def num_pages(self): return self.k_pool.shape[0]


def make_gqa(B, Hq, Hkv, D, seq_lens, *, page_size=64, max_pages=None, dtype=torch.bfloat16,
             shuffle=False, extra_pages=0, seed=0, factor=1.0, scale=None, window=0,
             n_sink=0, learned_sink=False) -> GQAInputs:
    lens = torch.as_tensor(seq_lens, dtype=torch.int32).reshape(B)
    if max_pages is None:
        max_pages = max(1, -(-int(lens.max()) // page_size))
    bt, num_pages = block_table_for(lens.tolist(), page_size, max_pages, shuffle, seed + 3,
                                    extra_pages)
    q = normal((B, Hq, D), seed + 0, factor, dtype)
    k = normal((num_pages, Hkv, page_size, D), seed + 1, factor, dtype)
    v = normal((num_pages, Hkv, page_size, D), seed + 2, factor, dtype)
    sink = normal((Hq,), seed + 4, 1.0, torch.float32) if learned_sink else None
    return GQAInputs(q, k, v, bt, lens, page_size,
                     float(scale if scale is not None else 1.0 / math.sqrt(D)),
                     int(window), int(n_sink), sink)


def make_ring(B, Hq, Hkv, D, seq_lens, window, *, n_sink=0, page_size=64, dtype=torch.bfloat16,
              shuffle=True, extra_pages=0, seed=0, factor=1.0, learned_sink=False) -> GQAInputs:
    """Sliding-window inputs on rolling caches: every sequence owns n_sink + window slots
    (all its pages allocated up front), filled with normals; seq_lens are the true lengths
    and may exceed the capacity."""
    cap = n_sink + window
    max_pages = -(-cap // page_size)
    bt, num_pages = block_table_for([cap] * B, page_size, max_pages, shuffle, seed + 3,
                                    extra_pages)
    lens = torch.as_tensor(seq_lens, dtype=torch.int32).reshape(B)
    q = normal((B, Hq, D), seed + 0, factor, dtype)
    k = normal((num_pages, Hkv, page_size, D), seed + 1, factor, dtype)
    v = normal((num_pages, Hkv, page_size, D), seed + 2, factor, dtype)
    sink = normal((Hq,), seed + 4, 1.0, torch.float32) if learned_sink else None
    return GQAInputs(q, k, v, bt, lens, page_size, 1.0 / math.sqrt(D), int(window), int(n_sink),
                     sink, ring=True)


@dataclass
class MLAInputs:
    q: torch.Tensor            # [B, H, 576] absorbed query (latent part already W_UK-folded)
    c_pool: torch.Tensor       # [num_pages, P, 576]
    block_table: torch.Tensor  # [B, max_pages] int32
    seq_lens: torch.Tensor     # [B] int32
    page_size: int
    scale: float
    d_v: int = 512

    @property
    def B(self): return self.q.shape[0]
    @property
    def H(self): return self.q.shape[1]
    @property
    def d_qk(self): return self.q.shape[2]
    @property
    def max_pages(self): return self.block_table.shape[1]
    @property
    def num_pages(self): return self.c_pool.shape[0]


def make_mla(B, H, seq_lens, *, d_qk=576, d_v=512, page_size=64, max_pages=None, shuffle=False,
             extra_pages=0, seed=0, factor=0.1, scale=1.0 / math.sqrt(192)) -> MLAInputs:
    lens = torch.as_tensor(seq_lens, dtype=torch.int32).reshape(B)
    if max_pages is None:
        max_pages = max(1, -(-int(lens.max()) // page_size))
    bt, num_pages = block_table_for(lens.tolist(), page_size, max_pages, shuffle, seed + 3,
                                    extra_pages)
    q = normal((B, H, d_qk), seed + 0, factor)
    c = normal((num_pages, page_size, d_qk), seed + 1, factor)
    return MLAInputs(q, c, bt, lens, page_size, float(scale), d_v)


@dataclass
class IndexerInputs:
    q: torch.Tensor            # [B, Hi, Di] bf16
    k_pool: torch.Tensor       # [num_pages, P, Di] bf16
    w: torch.Tensor            # [B, Hi] float32 head weights
    block_table: torch.Tensor  # [B, max_pages] int32
    seq_lens: torch.Tensor     # [B] int32
    page_size: int
    k: int

    @property
    def B(self): return self.q.shape[0]
    @property
    def Hi(self): return self.q.shape[1]
    @property
    def Di(self): return self.q.shape[2]
    @property
    def max_pages(self): return self.block_table.shape[1]
    @property
    def num_pages(self): return self.k_pool.shape[0]


def make_indexer(B, seq_lens, *, Hi=64, Di=128, k=2048, page_size=64, max_pages=None,
                 shuffle=False, extra_pages=0, seed=0, block_table=None) -> IndexerInputs:
    lens = torch.as_tensor(seq_lens, dtype=torch.int32).reshape(B)
    if max_pages is None:
        max_pages = max(1, -(-int(lens.max()) // page_size))
    if block_table is None:
        bt, num_pages = block_table_for(lens.tolist(), page_size, max_pages, shuffle, seed + 3,
                                        extra_pages)
    else:
        bt = block_table
        num_pages = int(bt.max()) + 1
    q = normal((B, Hi, Di), seed + 5)
    kp = normal((num_pages, page_size, Di), seed + 6)
    w = normal((B, Hi), seed + 7, 1.0, torch.float32)
    return IndexerInputs(q, kp, w, bt, lens, page_size, int(k))


# ----------------------------------------------------------------------------------------
# The named workloads. Each is shaped like a model family the pages use as their example.
# ----------------------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    wid: int
    kind: str               # "gqa" | "swa" | "mla" | "dsa" | "dsa_fp8" | "delta" | "quest"
    params: dict = field(default_factory=dict)
    description: str = ""


WORKLOADS = {
    "tiny_gqa_fp32": Workload(
        "tiny_gqa_fp32", 1, "gqa",
        dict(B=2, Hq=8, Hkv=2, D=64, L=256, dtype="fp32", page_size=64),
        "tiny GQA decode, fp32, B=2 Hq=8 Hkv=2 D=64 L=256, contiguous cache"),
    "llama3_8b_gqa_paged": Workload(
        "llama3_8b_gqa_paged", 2, "gqa",
        dict(B=32, Hq=32, Hkv=8, D=128, L_lo=4096, L_hi=8192, page_size=64, max_pages=128,
             shuffle=True, extra_pages=64),
        "Llama-3-8B-shaped GQA decode, one layer, bf16, B=32 Hq=32 Hkv=8 D=128, "
        "64-token pages with a shuffled block table, L ~ U[4096, 8192]"),
    "swa_sink_tokens": Workload(
        "swa_sink_tokens", 3, "swa",
        dict(B=8, Hq=64, Hkv=8, D=64, L=32768, window=4096, n_sink=4, learned_sink=False,
             page_size=64),
        "sliding window W=4096 plus the first 4 tokens, bf16, B=8 Hq=64 Hkv=8 D=64 L=32768"),
    "swa_learned_sink": Workload(
        "swa_learned_sink", 3, "swa",
        dict(B=8, Hq=64, Hkv=8, D=64, L=32768, window=4096, n_sink=0, learned_sink=True,
             page_size=64),
        "sliding window W=4096 with a learned per-head sink logit ~ N(0,1), bf16, "
        "B=8 Hq=64 Hkv=8 D=64 L=32768"),
    "swa_ring_sink_tokens": Workload(
        "swa_ring_sink_tokens", 8, "swa",
        dict(B=8, Hq=64, Hkv=8, D=64, L=32768, window=4096, n_sink=4, learned_sink=False,
             page_size=64, ring=True),
        "sliding window W=4096 plus the first 4 tokens on rolling caches of 4100 slots "
        "(O(W) memory), bf16, B=8 Hq=64 Hkv=8 D=64, true length 32768"),
    "quest_llama3": Workload(
        "quest_llama3", 9, "quest",
        dict(B=32, Hq=32, Hkv=8, D=128, L_lo=4096, L_hi=8192, page_size=16, max_pages=512,
             shuffle=True, extra_pages=64, n_sel=16),
        "Quest page selection on the Llama-3-8B-shaped GQA cache with 16-token pages "
        "(L ~ U[4096, 8192]): per-head bounds from page min/max keys, the best 16 pages "
        "(256 tokens) plus the partial tail, attention over them"),
    "mla_dsv3": Workload(
        "mla_dsv3", 4, "mla",
        dict(B=16, H=128, L=16384, page_size=64, factor=0.1),
        "MLA absorbed decode, DeepSeek-V3 shapes, bf16, B=16 H=128, 576-wide latent rows, "
        "L=16384, entries N(0,1)*0.1, scale 1/sqrt(192)"),
    "dsa_sparse_mla": Workload(
        "dsa_sparse_mla", 5, "dsa",
        dict(B=4, H=128, L=131072, Hi=64, Di=128, k=2048, page_size=64, factor=0.1),
        "DSA: indexer (64 heads x 128) over L=131072, top-2048, then 128-head sparse MLA, B=4"),
    "kda_decode": Workload(
        "kda_decode", 7, "delta",
        dict(B=128, H=32, dk=128, dv=128, per_channel=True),
        "KDA decode step, Kimi Linear shapes (32 heads, 128 x 128 float32 state per head), "
        "per-channel decay, B=128 sequences (4096 states, 268 MB)"),
    "dsa_fp8_sparse_mla": Workload(
        "dsa_fp8_sparse_mla", 6, "dsa_fp8",
        dict(B=4, H=128, L=131072, Hi=64, Di=128, k=2048, page_size=64, factor=0.1),
        "DSA with the FP8 indexer: e4m3 keys and queries with float32 row scales (64 heads x "
        "128) over L=131072, top-2048, then 128-head sparse MLA, B=4"),
}


@dataclass
class IndexerFp8Inputs:
    q8: torch.Tensor           # [B, Hi, Di] uint8 e4m3 codes
    q_scale: torch.Tensor      # [B, Hi] float32
    k8_pool: torch.Tensor      # [num_pages, P, Di] uint8 e4m3 codes
    k_scale: torch.Tensor      # [num_pages, P] float32
    w: torch.Tensor            # [B, Hi] float32
    block_table: torch.Tensor  # [B, max_pages] int32
    seq_lens: torch.Tensor     # [B] int32
    page_size: int
    k: int

    @property
    def B(self): return self.q8.shape[0]
    @property
    def max_pages(self): return self.block_table.shape[1]
    @property
    def num_pages(self): return self.k8_pool.shape[0]


def e4m3_codes(shape, seed: int, factor: float = 1.0) -> torch.Tensor:
    """uint8 e4m3 codes of seeded N(0,1) * factor draws (torch's float8 conversion)."""
    return normal(shape, seed, factor, torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)


def uniform_f32(shape, lo: float, hi: float, seed: int) -> torch.Tensor:
    """float32 draws uniform in [lo, hi)."""
    return lo + (hi - lo) * torch.rand(*shape, generator=_gen(seed), dtype=torch.float32)


def make_indexer_fp8(B, seq_lens, *, Hi=64, Di=128, k=2048, page_size=64, max_pages=None,
                     shuffle=False, extra_pages=0, seed=0, block_table=None) -> IndexerFp8Inputs:
    """FP8 indexer inputs: codes of N(0,1) draws, per-row scales uniform in [0.25, 1)."""
    base = make_indexer(B, seq_lens, Hi=Hi, Di=Di, k=k, page_size=page_size,
                        max_pages=max_pages, shuffle=shuffle, extra_pages=extra_pages, seed=seed,
                        block_table=block_table)
    num_pages = base.k_pool.shape[0]
    return IndexerFp8Inputs(
        e4m3_codes((B, Hi, Di), seed + 8), uniform_f32((B, Hi), 0.25, 1.0, seed + 10),
        e4m3_codes((num_pages, page_size, Di), seed + 9),
        uniform_f32((num_pages, page_size), 0.25, 1.0, seed + 11), base.w, base.block_table,
        base.seq_lens, page_size, int(k))


@dataclass
class DeltaInputs:
    S: torch.Tensor      # [n, dv, dk] float32 state
    q: torch.Tensor      # [n, dk] float32, unit norm times dk^-1/2
    k: torch.Tensor      # [n, dk] float32, unit norm
    v: torch.Tensor      # [n, dv] float32
    a: torch.Tensor      # [n, dk] (per key channel) or [n] (per head) float32 in [0.9, 1)
    beta: torch.Tensor   # [n] float32 in [0, 1)

    @property
    def n(self):
        return self.S.shape[0]


def make_delta(n, dk=128, dv=128, *, per_channel=True, seed=0, state_factor=0.1):
    """Gated delta-rule step inputs for n heads: state N(0,1)*state_factor, keys and queries
    scaled to unit norm (queries then by dk^-1/2), values N(0,1), decays uniform in
    [0.9, 1), write strengths uniform in [0, 1)."""
    S = normal((n, dv, dk), seed + 1, state_factor, torch.float32)
    k = normal((n, dk), seed + 2, 1.0, torch.float32)
    k = k / k.norm(dim=1, keepdim=True)
    q = normal((n, dk), seed + 3, 1.0, torch.float32)
    q = q / q.norm(dim=1, keepdim=True) / math.sqrt(dk)
    v = normal((n, dv), seed + 4, 1.0, torch.float32)
    a = uniform_f32((n, dk) if per_channel else (n,), 0.9, 1.0, seed + 5)
    beta = uniform_f32((n,), 0.0, 1.0, seed + 6)
    return DeltaInputs(S.contiguous(), q.contiguous(), k.contiguous(), v, a, beta)


def build(name: str, *, sharp: bool = False):
    """Materialise a named workload on the CPU (deterministic)."""
    w = WORKLOADS[name]
    p = w.params
    base = 1000 * w.wid
    if w.kind == "gqa" and p.get("dtype") == "fp32":
        return make_gqa(p["B"], p["Hq"], p["Hkv"], p["D"], [p["L"]] * p["B"],
                        page_size=p["page_size"], dtype=torch.float32, seed=base)
    if w.kind in ("gqa", "quest"):
        lens = uniform_int(p["L_lo"], p["L_hi"], p["B"], base + 9)
        return make_gqa(p["B"], p["Hq"], p["Hkv"], p["D"], lens, page_size=p["page_size"],
                        max_pages=p["max_pages"], shuffle=p["shuffle"],
                        extra_pages=p["extra_pages"], seed=base)
    if w.kind == "swa" and p.get("ring"):
        return make_ring(p["B"], p["Hq"], p["Hkv"], p["D"], [p["L"]] * p["B"], p["window"],
                         n_sink=p["n_sink"], page_size=p["page_size"], seed=base,
                         learned_sink=p["learned_sink"])
    if w.kind == "swa":
        return make_gqa(p["B"], p["Hq"], p["Hkv"], p["D"], [p["L"]] * p["B"],
                        page_size=p["page_size"], seed=base, window=p["window"],
                        n_sink=p["n_sink"], learned_sink=p["learned_sink"])
    if w.kind == "delta":
        return make_delta(p["B"] * p["H"], p["dk"], p["dv"], per_channel=p["per_channel"],
                          seed=base)
    factor = 1.0 if sharp else p["factor"]
    if w.kind == "mla":
        return make_mla(p["B"], p["H"], [p["L"]] * p["B"], page_size=p["page_size"], seed=base,
                        factor=factor)
    if w.kind == "dsa":
        mla = make_mla(p["B"], p["H"], [p["L"]] * p["B"], page_size=p["page_size"], seed=base,
                       factor=factor)
        idx = make_indexer(p["B"], [p["L"]] * p["B"], Hi=p["Hi"], Di=p["Di"], k=p["k"],
                           page_size=p["page_size"], seed=base, block_table=mla.block_table)
        return idx, mla
    if w.kind == "dsa_fp8":
        mla = make_mla(p["B"], p["H"], [p["L"]] * p["B"], page_size=p["page_size"], seed=base,
                       factor=factor)
        idx = make_indexer_fp8(p["B"], [p["L"]] * p["B"], Hi=p["Hi"], Di=p["Di"], k=p["k"],
                               page_size=p["page_size"], seed=base, block_table=mla.block_table)
        return idx, mla
    raise KeyError(name)
