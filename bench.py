"""Benchmark: decode-attention KV-cache bandwidth (GB/s) and attention steps/s.

One step = one decode-attention call over one batch of synthetic, seeded inputs whose
KV cache is already resident in HBM. The headline workload is the Llama-3-8B-shaped GQA
decode over a 64-token paged cache with a shuffled block table (B=32, Hq=32, Hkv=8,
D=128, L ~ U[4096, 8192]); its KV bytes (~805 MB) exceed L2, so consecutive steps cannot
be served from cache. The sliding-window, MLA, DSA, Quest and delta-rule workloads are
measured too and reported under "workloads": steps back to back over ceil(2 L2 / bytes) + 1
rotating copies of the cache (L2 size from the device; a CUDA graph of the steps, so no
host launch overhead), and single steps between L2 flushes (flush excluded). Each one's
configuration, byte and FLOP counts and roofline go on a "workload {...}" line before the
result line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {kvdecode,reference}]

`--impl reference` times the fp64 CPU oracle on the host cores instead (a bounded sample
of the same workload per step, same metric and unit).
Under torchrun each rank runs the same workload on its own GPU (independent sequences:
weak scaling, no collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

NOMINAL_HBM_GBS = 8000.0
HEADLINE = "llama3_8b_gqa_paged"


def l2_bytes(dev):
    """L2 size of the device, as the CUDA runtime reports it."""
    return int(torch.cuda.get_device_properties(dev).L2_cache_size)


# DRAM traffic (read + write bytes per launch) of each workload's dominant kernel from one ncu
# capture (summaries in profiles/, one per workload and kernel), reported only while what the
# kernel is compiled from -- its source file, the device header and its argument struct --
# still hashes to the value recorded with the capture: a changed kernel reports null.
NCU_TRAFFIC = {
    "llama3_8b_gqa_paged": {  # gqa_decode_bf16_kernel<128, 1, 1, 0>
        "bytes": 794.209280e6 + 3.381504e6,
        "sources": ('gqa_decode.cu', 'kvd_device.cuh'),
        "structs": ('GqaParams',),
        "sha256": "c0c24a8b630924cc7e5bd8d48f2a7081a33e87842b6a55136d613008fbfb3764",
    },
    "swa_sink_tokens": {  # gqa_decode_bf16_kernel<64, 1, 2, 1>
        "bytes": 68.300032e6 + 0.942592e6,
        "sources": ('gqa_decode.cu', 'kvd_device.cuh'),
        "structs": ('GqaParams',),
        "sha256": "c0c24a8b630924cc7e5bd8d48f2a7081a33e87842b6a55136d613008fbfb3764",
    },
    "swa_learned_sink": {  # gqa_decode_bf16_kernel<64, 1, 2, 1>
        "bytes": 67.251456e6 + 0.820736e6,
        "sources": ('gqa_decode.cu', 'kvd_device.cuh'),
        "structs": ('GqaParams',),
        "sha256": "c0c24a8b630924cc7e5bd8d48f2a7081a33e87842b6a55136d613008fbfb3764",
    },
    "swa_ring_sink_tokens": {  # gqa_decode_bf16_kernel<64, 1, 2, 1>
        "bytes": 68.299520e6 + 0.531200e6,
        "sources": ('gqa_decode.cu', 'kvd_device.cuh'),
        "structs": ('GqaParams',),
        "sha256": "c0c24a8b630924cc7e5bd8d48f2a7081a33e87842b6a55136d613008fbfb3764",
    },
    "mla_dsv3": {  # mla_decode_kernel<0>
        "bytes": 304.526848e6 + 4.448512e6,
        "sources": ('mla_decode.cu', 'mla_common.cuh', 'kvd_device.cuh'),
        "structs": ('MlaParams',),
        "sha256": "d4b9bbb43ff86fe732242a854b8375e50caaa2c0d204472c494a518c630f7f02",
    },
    "dsa_sparse_mla": {  # dsa_indexer_kernel
        "bytes": 134.377472e6 + 3.474688e6,
        "sources": ('dsa_indexer.cu', 'kvd_device.cuh'),
        "structs": ('IdxParams',),
        "sha256": "105e9959e518d84302f7680b51b8cd862d0ae73f3815924a3fe932b68a0ebb70",
    },
    "dsa_fp8_sparse_mla": {  # dsa_indexer_fp8_kernel
        "bytes": 69.331456e6 + 0.750080e6,
        "sources": ('dsa_indexer_fp8.cu', 'kvd_device.cuh'),
        "structs": ('IdxParams',),
        "sha256": "de9e49f6b6f46d0374108ed8d03f9b6e9b8b10c5f89b6f69a9da8ef6f42d955b",
    },
    "quest_llama3": {  # quest_attn_kernel<4, 1, 1>
        "bytes": 115.033600e6 + 3.841792e6,
        "sources": ('quest.cu', 'kvd_device.cuh'),
        "structs": ('QuestParams',),
        "sha256": "7716a52f75ab4165dd9b75304e0038b3badd1680dc098ec5e7c25e5fd9be914f",
    },
    "kda_decode": {  # delta_step_kernel<4>
        "bytes": 276.864768e6 + 210.739456e6,
        "sources": ('delta_decode.cu', 'kvd_device.cuh'),
        "structs": ('DeltaParams',),
        "sha256": "928b5aa034833b4918ac1cead8c2b1765687ceba11cd2c645b6c3dfc0b705282",
    },
}


def ncu_traffic(workload):
    import hashlib
    import re
    e = NCU_TRAFFIC.get(workload)
    if e is None:
        return None
    csrc = os.path.join(ROOT, "kv_cache_decode_split_gb300", "csrc")
    h = hashlib.sha256()
    try:
        for f in e["sources"]:
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
        with open(os.path.join(csrc, "kvd_host.h")) as fh:
            host = fh.read()
        for name in e.get("structs", ()):
            m = re.search(r"struct %s \{.*?\n\};" % name, host, re.S)
            if m is None:
                return None
            h.update(m.group(0).encode())
    except OSError:
        return None
    return e["bytes"] if h.hexdigest() == e["sha256"] else None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


# ---------------------------------------------------------------------------------------
# Workload runners (device side)
# ---------------------------------------------------------------------------------------
class GqaRunner:
    """attn_decode_gqa_paged / attn_decode_swa_sink on a named workload; on rolling caches,
    attn_decode_swa_ring_append (the step's new token appended, then attention: one call)."""
    launches_per_step = 1          # split-KV kernel; its last CTA per group combines
    kernel = "gqa_decode_bf16_kernel"
    cache_attrs = ("k", "v")       # the cache a step reads (copied for rotation)

    def __init__(self, name, dev):
        import kv_cache_decode_split_gb300 as kvd
        self.kvd = kvd
        self.name = name
        self.x = x = W.build(name)
        self.dev = dev
        self.q = x.q.to(dev)
        self.k = x.k_pool.to(dev)
        self.v = x.v_pool.to(dev)
        self.bt = x.block_table.to(dev)
        self.sl = x.seq_lens.to(dev)
        self.sink = x.sink_logit.to(dev) if x.sink_logit is not None else None
        self.out = torch.empty_like(self.q)
        self.ws = kvd.Workspace(dev)
        self.swa = x.window > 0 or x.n_sink > 0 or x.sink_logit is not None
        self.ring = x.ring
        if self.ring:
            # the step's new token (K and V rows of every sequence), appended before attention
            wid = W.WORKLOADS[name].wid
            self.h_knew = W.normal((x.B, x.Hkv, x.D), 1000 * wid + 20, 1.0, x.q.dtype)
            self.h_vnew = W.normal((x.B, x.Hkv, x.D), 1000 * wid + 21, 1.0, x.q.dtype)
            self.knew, self.vnew = self.h_knew.to(dev), self.h_vnew.to(dev)
            self.launches_per_step = 1  # the attention launch writes the new rows itself
        self._config, self.bytes, self.flops = self.describe(name, x)

    @staticmethod
    def describe(name, x):
        """(config, algorithmic KV bytes, FLOPs) of one step, from the CPU inputs."""
        swa = x.window > 0 or x.n_sink > 0 or x.sink_logit is not None
        tok = 0
        for L in x.seq_lens.tolist():
            if swa:
                tok += len(set(range(min(x.n_sink, L))) | set(range(max(0, L - x.window), L)))
            else:
                tok += L
        nbytes = tok * x.Hkv * x.D * 2 * x.q.element_size()   # K and V rows the method reads
        if x.ring:   # plus the new token's K and V rows, read once and written once
            nbytes += 2 * 2 * x.B * x.Hkv * x.D * x.q.element_size()
        flops = 4.0 * tok * x.Hkv * (x.Hq // x.Hkv) * x.D
        cfg = {"workload": name, "B": x.B, "Hq": x.Hq, "Hkv": x.Hkv, "D": x.D,
               "page_size": x.page_size, "window": x.window, "n_sink": x.n_sink,
               "learned_sink": x.sink_logit is not None,
               "seq_len_mean": float(x.seq_lens.float().mean()), "kv_bytes": nbytes}
        if x.ring:
            cfg["cache"] = f"rolling, {x.n_sink + x.window} slots per sequence"
            cfg["step"] = "the new token appended, then attention (attn_decode_swa_ring_append)"
        return cfg, nbytes, flops

    def step(self, q=None, out=None):
        x = self.x
        q = self.q if q is None else q
        out = self.out if out is None else out
        if self.ring:
            return self.kvd.attn_decode_swa_ring_append(q, self.knew, self.vnew, self.k, self.v,
                                                        self.bt, self.sl, x.window, x.n_sink,
                                                        self.sink, scale=x.scale, out=out,
                                                        workspace=self.ws)
        if self.swa:
            return self.kvd.attn_decode_swa_sink(q, self.k, self.v, self.bt, self.sl, x.window,
                                                 x.n_sink, self.sink, scale=x.scale, out=out,
                                                 workspace=self.ws)
        return self.kvd.attn_decode_gqa_paged(q, self.k, self.v, self.bt, self.sl, scale=x.scale,
                                              out=out, workspace=self.ws)

    def config(self):
        return self._config

    # --- end-to-end through the public API from pinned host buffers
    def e2e_setup(self):
        self.h_q = self.x.q.pin_memory()
        self.h_bt = self.x.block_table.pin_memory()
        self.h_sl = self.x.seq_lens.pin_memory()
        self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.d_q = torch.empty_like(self.q)
        h2d = (self.h_q.numel() * self.h_q.element_size() + self.h_bt.numel() * 4 +
               self.h_sl.numel() * 4)
        if self.ring:
            self.h_knew, self.h_vnew = self.h_knew.pin_memory(), self.h_vnew.pin_memory()
            h2d += 2 * self.h_knew.numel() * self.h_knew.element_size()
        return h2d, self.h_out.numel() * self.h_out.element_size()

    def e2e_step(self):
        if self.ring:
            self.knew.copy_(self.h_knew, non_blocking=True)
            self.vnew.copy_(self.h_vnew, non_blocking=True)
        self.d_q.copy_(self.h_q, non_blocking=True)
        self.bt.copy_(self.h_bt, non_blocking=True)
        self.sl.copy_(self.h_sl, non_blocking=True)
        self.step(q=self.d_q)
        self.h_out.copy_(self.out, non_blocking=True)

    # --- the oracle on host cores, over a bounded sample of the same workload
    def oracle_sample(self, budget_s):
        import numpy as np
        import oracle
        x = self.x
        G = x.Hq // x.Hkv
        rng = np.random.default_rng(0)
        units = [(b, g) for b in range(x.B) for g in range(x.Hkv)]
        rng.shuffle(units)
        t0 = time.perf_counter()
        done_bytes, n = 0, 0
        lens = x.seq_lens.tolist()
        for b, g in units:
            pairs = [(b, g * G + j) for j in range(G)]
            oracle.gqa(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale, x.window,
                       x.n_sink, x.sink_logit, pairs=pairs, ring=x.ring)
            L = lens[b]
            if self.swa:
                vis = len(set(range(min(x.n_sink, L))) | set(range(max(0, L - x.window), L)))
            else:
                vis = L
            done_bytes += vis * x.D * 2 * x.q.element_size()
            n += 1
            if time.perf_counter() - t0 > budget_s:
                break
        el = time.perf_counter() - t0
        return done_bytes, el, f"{n} of {len(units)} (sequence, KV head) groups, all {G} query heads each"


class MlaRunner:
    """attn_decode_mla on the DeepSeek-V3-shaped workload (128 heads, 576-wide rows)."""
    launches_per_step = 2          # split kernel (2-CTA clusters) + combine kernel
    kernel = "mla_decode_kernel"
    cache_attrs = ("c",)
    tensor_path = True             # score and value products on tcgen05

    def __init__(self, name, dev, sharp=False):
        import kv_cache_decode_split_gb300 as kvd
        self.kvd = kvd
        self.name = name
        self.x = x = W.build(name, sharp=sharp)
        self.dev = dev
        self.q = x.q.to(dev)
        self.c = x.c_pool.to(dev)
        self.bt = x.block_table.to(dev)
        self.sl = x.seq_lens.to(dev)
        self.out = torch.empty(x.B, x.H, 512, dtype=torch.bfloat16, device=dev)
        self.ws = kvd.Workspace(dev)
        self._config, self.bytes, self.flops = self.describe(name, x)

    @staticmethod
    def describe(name, x):
        tok = int(x.seq_lens.sum())
        nbytes = tok * x.d_qk * 2
        flops = 2.0 * tok * x.H * (x.d_qk + 512)
        cfg = {"workload": name, "B": x.B, "H": x.H, "d_qk": x.d_qk, "d_v": 512,
               "page_size": x.page_size, "seq_len_mean": float(x.seq_lens.float().mean()),
               "kv_bytes": nbytes, "flops": flops}
        return cfg, nbytes, flops

    def step(self, q=None):
        x = self.x
        return self.kvd.attn_decode_mla(self.q if q is None else q, self.c, self.bt, self.sl,
                                        scale=x.scale, out=self.out, workspace=self.ws)

    def config(self):
        return self._config

    def e2e_setup(self):
        self.h_q = self.x.q.pin_memory()
        self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.d_q = torch.empty_like(self.q)
        return self.h_q.numel() * 2, self.h_out.numel() * 2

    def e2e_step(self):
        self.d_q.copy_(self.h_q, non_blocking=True)
        self.step(q=self.d_q)
        self.h_out.copy_(self.out, non_blocking=True)

    def oracle_sample(self, budget_s):
        import oracle
        x = self.x
        t0 = time.perf_counter()
        done, n = 0, 0
        for b in range(x.B):
            for h0 in range(0, x.H, 16):
                pairs = [(b, h) for h in range(h0, h0 + 16)]
                oracle.mla(x.q, x.c_pool, x.block_table, x.seq_lens, x.scale, pairs=pairs)
                done += int(x.seq_lens[b]) * x.d_qk * 2 * 16 / x.H
                n += 16
                if time.perf_counter() - t0 > budget_s:
                    break
            if time.perf_counter() - t0 > budget_s:
                break
        el = time.perf_counter() - t0
        return done, el, f"{n} of {x.B * x.H} (sequence, head) outputs, bytes counted pro rata"


class DsaRunner:
    """dsa_indexer_topk then attn_decode_mla_sparse (indexer, top-2048, sparse MLA)."""
    launches_per_step = 4          # indexer, selection, sparse MLA, combine
    kernel = "dsa_indexer_kernel"
    cache_attrs = ("ki", "c")
    tensor_path = True             # indexer and sparse MLA products on tcgen05

    def __init__(self, name, dev, sharp=False):
        import kv_cache_decode_split_gb300 as kvd
        self.kvd = kvd
        self.name = name
        self.xi, self.xm = xi, xm = W.build(name, sharp=sharp)
        self.dev = dev
        self.qi = xi.q.to(dev)
        self.ki = xi.k_pool.to(dev)
        self.w = xi.w.to(dev)
        self.q = xm.q.to(dev)
        self.c = xm.c_pool.to(dev)
        self.bt = xm.block_table.to(dev)
        self.sl = xm.seq_lens.to(dev)
        self.k = xi.k
        self.idx = torch.empty(xi.B, xi.k, dtype=torch.int32, device=dev)
        self.cnt = torch.empty(xi.B, dtype=torch.int32, device=dev)
        self.out = torch.empty(xm.B, xm.H, 512, dtype=torch.bfloat16, device=dev)
        self.ws1 = kvd.Workspace(dev)
        self.ws2 = kvd.Workspace(dev)
        self._config, self.bytes, self.flops = self.describe(name, (xi, xm))

    @staticmethod
    def describe(name, x):
        xi, xm = x
        lens = [int(v) for v in xm.seq_lens]
        sel = sum(min(xi.k, L) for L in lens)
        nbytes = sum(lens) * xi.Di * 2 + sel * xm.d_qk * 2
        flops = 2.0 * sum(lens) * xi.Hi * xi.Di + 2.0 * sel * xm.H * (xm.d_qk + 512)
        cfg = {"workload": name, "B": xm.B, "H": xm.H, "Hi": xi.Hi, "Di": xi.Di, "k": xi.k,
               "seq_len": lens[0], "page_size": xm.page_size, "kv_bytes": nbytes, "flops": flops}
        return cfg, nbytes, flops

    def step(self, qi=None, q=None):
        xm = self.xm
        self.kvd.dsa_indexer_topk(self.qi if qi is None else qi, self.ki, self.w, self.bt,
                                  self.sl, k=self.k, topk_idx=self.idx, topk_count=self.cnt,
                                  workspace=self.ws1)
        return self.kvd.attn_decode_mla_sparse(self.q if q is None else q, self.c, self.bt,
                                               self.sl, self.idx, self.cnt, scale=xm.scale,
                                               out=self.out, workspace=self.ws2)

    def config(self):
        return self._config

    def e2e_setup(self):
        self.h_qi = self.xi.q.pin_memory()
        self.h_q = self.xm.q.pin_memory()
        self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.d_qi = torch.empty_like(self.qi)
        self.d_q = torch.empty_like(self.q)
        return (self.h_qi.numel() + self.h_q.numel()) * 2, self.h_out.numel() * 2

    def e2e_step(self):
        self.d_qi.copy_(self.h_qi, non_blocking=True)
        self.d_q.copy_(self.h_q, non_blocking=True)
        self.step(qi=self.d_qi, q=self.d_q)
        self.h_out.copy_(self.out, non_blocking=True)

    def oracle_sample(self, budget_s):
        import numpy as np
        import oracle
        xi, xm = self.xi, self.xm
        t0 = time.perf_counter()
        done, n = 0, 0
        for b in range(xm.B):
            sc = oracle.indexer_scores(xi.q, xi.k_pool, xi.w, xi.block_table, xi.seq_lens,
                                       batches=[b])[0]
            L = int(xm.seq_lens[b])
            idx = oracle.topk(sc[:L].astype(np.float32), self.k)
            full = np.full((xm.B, self.k), -1, np.int32)
            full[b, :len(idx)] = idx
            cnt = np.zeros(xm.B, np.int32)
            cnt[b] = len(idx)
            oracle.mla(xm.q, xm.c_pool, xm.block_table, xm.seq_lens, xm.scale, idx=full,
                       idx_count=cnt, pairs=[(b, h) for h in range(xm.H)])
            done += L * xi.Di * 2 + len(idx) * xm.d_qk * 2
            n += 1
            if time.perf_counter() - t0 > budget_s:
                break
        el = time.perf_counter() - t0
        return done, el, f"{n} of {xm.B} sequences (indexer, top-k and sparse MLA, all heads)"


class DsaFp8Runner(DsaRunner):
    """dsa_indexer_topk_fp8 then attn_decode_mla_sparse (FP8 indexer, top-2048, sparse MLA)."""
    kernel = "dsa_indexer_fp8_kernel"
    cache_attrs = ("ki", "ks", "c")

    def __init__(self, name, dev, sharp=False):
        import kv_cache_decode_split_gb300 as kvd
        self.kvd = kvd
        self.name = name
        self.xi, self.xm = xi, xm = W.build(name, sharp=sharp)
        self.dev = dev
        self.qi = xi.q8.to(dev)
        self.qs = xi.q_scale.to(dev)
        self.ki = xi.k8_pool.to(dev)
        self.ks = xi.k_scale.to(dev)
        self.w = xi.w.to(dev)
        self.q = xm.q.to(dev)
        self.c = xm.c_pool.to(dev)
        self.bt = xm.block_table.to(dev)
        self.sl = xm.seq_lens.to(dev)
        self.k = xi.k
        self.idx = torch.empty(xi.B, xi.k, dtype=torch.int32, device=dev)
        self.cnt = torch.empty(xi.B, dtype=torch.int32, device=dev)
        self.out = torch.empty(xm.B, xm.H, 512, dtype=torch.bfloat16, device=dev)
        self.ws1 = kvd.Workspace(dev)
        self.ws2 = kvd.Workspace(dev)
        self._config, self.bytes, self.flops = self.describe(name, (xi, xm))

    @staticmethod
    def describe(name, x):
        xi, xm = x
        lens = [int(v) for v in xm.seq_lens]
        Hi, Di = xi.q8.shape[1], xi.q8.shape[2]
        sel = sum(min(xi.k, L) for L in lens)
        # one-byte key codes and a float32 scale per token, then the selected latent rows
        nbytes = sum(lens) * (Di + 4) + sel * xm.d_qk * 2
        flops = 2.0 * sum(lens) * Hi * Di + 2.0 * sel * xm.H * (xm.d_qk + 512)
        cfg = {"workload": name, "B": xm.B, "H": xm.H, "Hi": Hi, "Di": Di, "k": xi.k,
               "seq_len": lens[0], "page_size": xm.page_size, "indexer": "e4m3 + f32 row scales",
               "kv_bytes": nbytes, "flops": flops}
        return cfg, nbytes, flops

    def step(self, qi=None, q=None):
        xm = self.xm
        self.kvd.dsa_indexer_topk_fp8(self.qi if qi is None else qi, self.qs, self.ki, self.ks,
                                      self.w, self.bt, self.sl, k=self.k, topk_idx=self.idx,
                                      topk_count=self.cnt, workspace=self.ws1)
        return self.kvd.attn_decode_mla_sparse(self.q if q is None else q, self.c, self.bt,
                                               self.sl, self.idx, self.cnt, scale=xm.scale,
                                               out=self.out, workspace=self.ws2)

    def e2e_setup(self):
        self.h_qi = self.xi.q8.pin_memory()
        self.h_q = self.xm.q.pin_memory()
        self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.d_qi = torch.empty_like(self.qi)
        self.d_q = torch.empty_like(self.q)
        return self.h_qi.numel() + self.h_q.numel() * 2, self.h_out.numel() * 2

    def oracle_sample(self, budget_s):
        import numpy as np
        import oracle
        xi, xm = self.xi, self.xm
        t0 = time.perf_counter()
        done, n = 0, 0
        for b in range(xm.B):
            sc = oracle.indexer_scores_fp8(xi.q8.numpy(), xi.q_scale.numpy(), xi.k8_pool.numpy(),
                                           xi.k_scale.numpy(), xi.w, xi.block_table,
                                           xi.seq_lens, batches=[b])[0]
            L = int(xm.seq_lens[b])
            idx = oracle.topk(sc[:L].astype(np.float32), self.k)
            full = np.full((xm.B, self.k), -1, np.int32)
            full[b, :len(idx)] = idx
            cnt = np.zeros(xm.B, np.int32)
            cnt[b] = len(idx)
            oracle.mla(xm.q, xm.c_pool, xm.block_table, xm.seq_lens, xm.scale, idx=full,
                       idx_count=cnt, pairs=[(b, h) for h in range(xm.H)])
            done += L * (xi.q8.shape[2] + 4) + len(idx) * xm.d_qk * 2
            n += 1
            if time.perf_counter() - t0 > budget_s:
                break
        el = time.perf_counter() - t0
        return done, el, f"{n} of {xm.B} sequences (FP8 indexer, top-k and sparse MLA, all heads)"


class DeltaRunner:
    """delta_decode_step: one gated delta-rule (KDA) token step over every head's state."""
    launches_per_step = 1
    kernel = "delta_step_kernel"
    cache_attrs = ("S",)
    dtype = "f32"
    data = "synthetic: seeded float32 draws (state, unit-norm keys and queries), Kimi Linear shapes"

    def __init__(self, name, dev, sharp=False):
        import kv_cache_decode_split_gb300 as kvd
        self.kvd = kvd
        self.name = name
        self.x = x = W.build(name)
        self.dev = dev
        self.S = x.S.to(dev)
        self.q, self.k, self.v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
        self.a, self.beta = x.a.to(dev), x.beta.to(dev)
        self.o = torch.empty(x.v.shape, dtype=torch.float32, device=dev)
        self._config, self.bytes, self.flops = self.describe(name, x)

    @staticmethod
    def describe(name, x):
        n, dv, dk = x.S.shape
        # the state read and written once; q, k, a, v, beta read and o written per head
        nbytes = n * (2 * dv * dk + 2 * dk + x.a[0].numel() + 2 * dv + 1) * 4
        flops = n * dv * dk * 7.0
        p = W.WORKLOADS[name].params
        cfg = {"workload": name, "B": p["B"], "H": p["H"], "dk": dk, "dv": dv,
               "gate": "per key channel" if x.a.dim() == 2 else "per head",
               "state_bytes": n * dv * dk * 4, "kv_bytes": nbytes, "flops": flops}
        return cfg, nbytes, flops

    def step(self, q=None):
        return self.kvd.delta_decode_step(self.S, self.q if q is None else q, self.k, self.v,
                                          self.a, self.beta, o=self.o)

    def config(self):
        return self._config

    def e2e_setup(self):
        # the per-token inputs come from the host every step; the states stay resident
        self.h_in = [t.pin_memory() for t in (self.x.q, self.x.k, self.x.v, self.x.a,
                                               self.x.beta)]
        self.d_in = [torch.empty_like(t, device=self.dev) for t in self.h_in]
        self.h_out = torch.empty(self.o.shape, dtype=torch.float32).pin_memory()
        return sum(t.numel() * 4 for t in self.h_in), self.h_out.numel() * 4

    def e2e_step(self):
        for d, h in zip(self.d_in, self.h_in):
            d.copy_(h, non_blocking=True)
        q, k, v, a, beta = self.d_in
        self.kvd.delta_decode_step(self.S, q, k, v, a, beta, o=self.o)
        self.h_out.copy_(self.o, non_blocking=True)

    def oracle_sample(self, budget_s):
        import oracle
        x = self.x
        n, dv, dk = x.S.shape
        t0 = time.perf_counter()
        done, heads = 0, 0
        per_head = (2 * dv * dk + 2 * dk + x.a[0].numel() + 2 * dv + 1) * 4
        while heads < n and time.perf_counter() - t0 < budget_s:
            sl = slice(heads, min(n, heads + 64))
            oracle.delta_step(x.S[sl], x.q[sl], x.k[sl], x.v[sl], x.a[sl], x.beta[sl])
            done += (sl.stop - sl.start) * per_head
            heads = sl.stop
        el = time.perf_counter() - t0
        return done, el, f"{heads} of {n} heads (one token step each)"


class QuestRunner(GqaRunner):
    """quest_select_pages then attn_decode_quest (page summaries computed once, at set-up,
    as pages fill in a real decode)."""
    launches_per_step = 2          # bounds; choice + attention
    kernel = "quest_attn_kernel"
    cache_attrs = ("k", "v", "kmin", "kmax")

    def __init__(self, name, dev):
        super().__init__(name, dev)
        self.n_sel = W.WORKLOADS[name].params["n_sel"]
        self.kmin, self.kmax, self.err = self.kvd.quest_page_minmax(self.k)
        self.sel = torch.empty(self.x.B, self.x.Hq, self.n_sel, dtype=torch.int32, device=dev)
        self.ub = torch.empty(self.x.B, self.x.Hq, self.x.max_pages, dtype=torch.float32,
                              device=dev)
        self._config, self.bytes, self.flops = self.describe(name, self.x)

    @staticmethod
    def describe(name, x):
        n_sel = W.WORKLOADS[name].params["n_sel"]
        P, esz = x.page_size, x.q.element_size()
        summ, rows = 0, 0
        for L in x.seq_lens.tolist():
            full = L // P
            summ += full * x.Hkv * 2 * x.D * esz                  # kmin and kmax rows read
            rows += x.Hq * (min(full, n_sel) * P + L - full * P)  # K/V rows each head reads
        nbytes = summ + rows * x.D * 2 * esz + x.q.numel() * esz
        flops = 4.0 * rows * x.D
        cfg = {"workload": name, "B": x.B, "Hq": x.Hq, "Hkv": x.Hkv, "D": x.D, "page_size": P,
               "n_sel": n_sel, "budget_tokens": n_sel * P,
               "seq_len_mean": float(x.seq_lens.float().mean()), "kv_bytes": nbytes,
               "dense_kv_bytes": int(x.seq_lens.sum()) * x.Hkv * x.D * 2 * esz}
        return cfg, nbytes, flops

    def step(self, q=None, out=None):
        x = self.x
        q = self.q if q is None else q
        out = self.out if out is None else out
        self.kvd.quest_page_bounds(q, self.kmin, self.kmax, self.bt, self.sl, x.page_size,
                                   ub=self.ub, err=self.err)
        return self.kvd.attn_decode_quest_from_bounds(q, self.k, self.v, self.bt, self.sl,
                                                      self.ub, self.n_sel, scale=x.scale,
                                                      sel_out=self.sel, out=out, err=self.err)[0]

    def oracle_sample(self, budget_s):
        import numpy as np
        import oracle
        x = self.x
        rng = np.random.default_rng(0)
        pairs_all = [(b, h) for b in range(x.B) for h in range(x.Hq)]
        rng.shuffle(pairs_all)
        t0 = time.perf_counter()
        done, n = 0, 0
        P = x.page_size
        for i in range(0, len(pairs_all), 8):
            pairs = pairs_all[i:i + 8]
            oracle.quest(x.q, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.scale,
                         self.n_sel, pairs=pairs)
            for b, h in pairs:
                L = int(x.seq_lens[b])
                full = L // P
                done += (full * 2 * x.D + (min(full, self.n_sel) * P + L - full * P) * x.D * 2) \
                    * x.q.element_size()
            n += len(pairs)
            if time.perf_counter() - t0 > budget_s:
                break
        el = time.perf_counter() - t0
        return done, el, f"{n} of {len(pairs_all)} (sequence, query head) pairs"


RUNNERS = {"gqa": GqaRunner, "swa": GqaRunner, "mla": MlaRunner, "dsa": DsaRunner,
           "dsa_fp8": DsaFp8Runner, "delta": DeltaRunner, "quest": QuestRunner}


def make_runner(name, dev):
    return RUNNERS[W.WORKLOADS[name].kind](name, dev)


# ---------------------------------------------------------------------------------------
# Timing helpers
# ---------------------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def shard_range(n, rank, world):
    """Contiguous share [lo, hi) of n independent units (sequences) for one rank."""
    per, extra = divmod(n, world)
    lo = rank * per + min(rank, extra)
    return lo, lo + per + (1 if rank < extra else 0)


def aggregate(local_ms, bytes_per_rank, world, dist=None):
    """Whole-job throughput: every rank's bytes over the slowest rank's time (max over
    ranks). Returns (max_ms, GB/s)."""
    t = torch.tensor([float(local_ms)], dtype=torch.float64)
    if dist is not None and world > 1:
        if t.device.type == "cpu" and dist.get_backend() == "nccl":
            t = t.cuda()
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms = float(t.item())
    return ms, world * bytes_per_rank / (ms * 1e-3) / 1e9


def flush_l2(buf):
    """Evict the workload from L2 by READING a buffer larger than L2 (a write-based flush
    would leave dirty lines whose write-back the next timed step would pay for)."""
    buf.sum()


def time_steps(fn, steps, stream):
    """Total CUDA-event duration (ms) of `steps` back-to-back steps on `stream`, and the mean
    per step. Only the two bracketing events are recorded: an event between steps would sit
    between two kernels and keep the second from launching while the first finishes."""
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    total = a.elapsed_time(b)
    return total, [total / steps] * steps


def time_flushed(fn, iters, stream, flush):
    per = []
    for _ in range(iters):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        per.append(a.elapsed_time(b))
    return per


def rotation_copies(nbytes, l2):
    """Independent cache copies to rotate through so that no step finds its data in L2:
    ceil(2 L2 / bytes) + 1 (two L2 sizes of other data between two reads of one copy)."""
    return max(1, math.ceil(2 * l2 / max(1, nbytes)) + 1)


def time_rotating(runner, copies, stream, steps_min=40, repeats=5):
    """Per-step time (ms, median of `repeats`) of steps run back to back, step i reading
    cache copy i mod `copies` (the runner's cache_attrs swapped in), captured once into a
    CUDA graph and replayed, so that host-side launch overhead is not in the number (a
    caller launching from C++ or from its own graph pays none either). Falls back to an
    eager loop if the capture fails; returns (ms, how)."""
    attrs = runner.cache_attrs
    orig = {a: getattr(runner, a) for a in attrs}
    sets = [orig] + [{a: t.clone() for a, t in orig.items()} for _ in range(copies - 1)]
    n = max(steps_min, copies) // copies * copies

    def run_all():
        for i in range(n):
            for a, t in sets[i % copies].items():
                setattr(runner, a, t)
            runner.step()

    run_all()          # every copy once, eagerly (workspaces sized before capture)
    torch.cuda.synchronize()
    how = "cuda graph"
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run_all()
        replay = g.replay
        replay()
        torch.cuda.synchronize()
    except Exception:  # noqa: BLE001 -- capture unsupported: time the same loop eagerly
        g, replay, how = None, run_all, "eager"
        torch.cuda.synchronize()
    per = []
    for _ in range(repeats):
        total, _ = time_steps(replay, 1, stream)
        per.append(total / n)
    for a, t in orig.items():
        setattr(runner, a, t)
    del sets, g
    return statistics.median(per), how


# ---------------------------------------------------------------------------------------
def oracle_runner(name):
    """A runner holding only the CPU inputs of a workload, for timing the oracle."""
    cls = RUNNERS[W.WORKLOADS[name].kind]
    r = cls.__new__(cls)
    r.name = name
    if cls in (DsaRunner, DsaFp8Runner):
        r.xi, r.xm = W.build(name)
        r.k = r.xi.k
    else:
        r.x = x = W.build(name)
        if cls is QuestRunner:
            r.n_sel = W.WORKLOADS[name].params["n_sel"]
        if cls in (GqaRunner, QuestRunner):
            r.swa = x.window > 0 or x.n_sink > 0 or x.sink_logit is not None
    return r


def run_reference(args, rank, world):
    if rank != 0:
        return
    name = args.workload
    wl = W.WORKLOADS[name]
    x_runner = oracle_runner(name)
    per_step = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    vals, secs = [], []
    desc = ""
    for i in range(args.warmup + args.steps):
        nbytes, el, desc = x_runner.oracle_sample(per_step)
        if i >= args.warmup:
            vals.append(nbytes / el / 1e9)
            secs.append(el)
    v = statistics.median(vals)
    cls = RUNNERS[wl.kind]
    xin = (x_runner.xi, x_runner.xm) if cls in (DsaRunner, DsaFp8Runner) else x_runner.x
    cfg, _, _ = cls.describe(name, xin)
    cfg = dict(cfg, l2="KV bytes larger than L2; steps back to back", parallelism="single")
    line = {"impl": "reference", "metric": "decode-attn KV GB/s", "value": v, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.median(secs), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": getattr(cls, "data", "synthetic: seeded N(0,1) rounded to bf16, shapes of "
                                         "the named workload"),
            "config": cfg,
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"per step: {desc}, {statistics.median(secs):.2f} s of CPU work "
                                       f"(budget {per_step:.0f} s)"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="kvdecode", choices=["kvdecode", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(W.WORKLOADS))
    ap.add_argument("--extra", default="all", help="comma list of extra workloads, 'all' or 'none'")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import torch.distributed as dist
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    peaks, peak_src = measured_peaks()

    r = make_runner(args.workload, dev)
    # a workload whose data would stay in L2 between steps rotates through independent
    # copies of its cache; larger ones run back to back on one copy
    l2 = l2_bytes(dev)
    copies = rotation_copies(r.bytes, l2) if r.bytes < 2 * l2 else 1
    if copies > 1:
        for a, t in {a: getattr(r, a) for a in r.cache_attrs}.items():
            setattr(r, a + "_rot", [t] + [t.clone() for _ in range(copies - 1)])
        i_step = [0]

        def step_main():
            i = i_step[0] % copies
            for a in r.cache_attrs:
                setattr(r, a, getattr(r, a + "_rot")[i])
            i_step[0] += 1
            r.step()
    else:
        step_main = r.step
    for _ in range(args.warmup):
        step_main()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        total_ms, per = time_steps(step_main, args.steps, stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    total_ms, _ = aggregate(total_ms, r.bytes, world, dist if world > 1 else None)
    ms = total_ms / args.steps
    value = world * r.bytes / (ms * 1e-3) / 1e9
    clocks = clk.summary()

    # end-to-end through the public API with pinned host buffers
    h2d, d2h = r.e2e_setup()
    for _ in range(3):
        r.e2e_step()
    torch.cuda.synchronize()
    e2e_total, _ = time_steps(r.e2e_step, args.steps, stream)
    e2e_ms = e2e_total / args.steps
    e2e_ms, _ = aggregate(e2e_ms, r.bytes, world, dist if world > 1 else None)

    kern_ms = statistics.mean(per)
    achieved = r.bytes / (kern_ms * 1e-3) / 1e9
    line = {
        "metric": "decode-attn KV GB/s", "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": getattr(r, "dtype", "bf16"),
        "data": getattr(r, "data", "synthetic: seeded N(0,1) rounded to bf16, workload shapes"),
        "config": dict(r.config(), l2=(f"{copies} cache copies rotated, steps back to back"
                                       if copies > 1 else
                                       "KV bytes larger than L2; steps back to back"),
                       parallelism=f"replicas{world}" if world > 1 else "single"),
        "steps_per_s": 1000.0 / ms,
        "frac_of_nominal_8tbs": value / world / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "kernel": r.kernel,
                     "achieved_over": ("the kernel's launches" if r.launches_per_step == 1 else
                                       f"whole steps ({r.launches_per_step} launches each)"),
                     "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "peak_source": peak_src, "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic(args.workload),
                     "algorithmic_bytes": r.bytes},
        "e2e": {"value": world * r.bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": r.launches_per_step * args.steps,
        "clocks": clocks,
    }
    del r, step_main
    torch.cuda.empty_cache()

    # The other workloads: each step's roofline against the measured peaks, from steps run
    # back to back over rotating cache copies (us), and from single steps between L2
    # flushes, flush excluded (us_flushed). Their configurations and byte / FLOP counts go
    # on lines of their own before the result line, which stays short.
    extras = [] if args.extra == "none" else (
        [n for n in W.WORKLOADS if n not in (args.workload, "tiny_gqa_fp32")] if args.extra == "all"
        else [n for n in args.extra.split(",") if n])
    if extras and rank == 0:
        flush_buf = torch.zeros(2 * l2 // 4 + (1 << 20), dtype=torch.float32, device=dev)
        res = {}
        for name in extras:
            try:
                rr = make_runner(name, dev)
                for _ in range(3):
                    rr.step()
                torch.cuda.synchronize()
                per = time_flushed(rr.step, max(10, args.steps // 2), stream,
                                   lambda: flush_l2(flush_buf))
                n_copies = rotation_copies(rr.bytes, l2)
                rot_ms, how = time_rotating(rr, n_copies, stream)
            except Exception as e:  # an entry point that fails reports, not crashes
                res[name] = {"status": f"error: {e}"[:120]}
                continue
            flushed_ms = statistics.median(per)
            gbs = rr.bytes / (rot_ms * 1e-3) / 1e9
            entry = {"us": round(rot_ms * 1e3, 2), "us_flushed": round(flushed_ms * 1e3, 2),
                     "GBps": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4)}
            t = ncu_traffic(name)
            entry["dram_MB"] = round(t / 1e6, 1) if t is not None else None
            tfl = rr.flops / (rot_ms * 1e-3) / 1e12
            if getattr(rr, "tensor_path", False):
                entry["TFLOPs"] = round(tfl, 1)
                entry["tensor_frac"] = round(tfl / peaks["bf16_tflops_sustained"], 4)
            res[name] = entry
            print("workload " + json.dumps({
                "name": name, "config": rr.config(), "kernel": rr.kernel,
                "launches_per_step": rr.launches_per_step, "algorithmic_bytes": rr.bytes,
                "flops": rr.flops, "rotation": f"{n_copies} copies, {how}",
                "flush": f"{flush_buf.numel() * 4 >> 20} MiB read between steps",
                "roofline": {"bound": "hbm", "achieved_GBps": gbs, "peak_GBps": peaks["hbm_gbs"],
                             "frac": gbs / peaks["hbm_gbs"], "achieved_TFLOPs": tfl,
                             "peak_TFLOPs": peaks["bf16_tflops_sustained"],
                             "traffic": ncu_traffic(name)},
                "us_per_step": rot_ms * 1e3, "us_flushed": flushed_ms * 1e3}), flush=True)
            del rr
            torch.cuda.empty_cache()
        line["workloads"] = res
        line["workloads_note"] = ("us: back to back over rotating cache copies; frac: algorithmic "
                                  "bytes / us over measured HBM; tensor_frac: FLOPs / us over "
                                  "measured sustained bf16")

    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        rr = oracle_runner(args.workload)
        nbytes, el, desc = rr.oracle_sample(args.cpu_seconds)
        line["cpu_baseline"] = {"value": nbytes / el / 1e9, "unit": "GB/s",
                                "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"{desc}, {el:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
