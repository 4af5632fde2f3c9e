"""The pages' printed byte and FLOP figures, reproduced by the oracle's size model."""
import json
import os

import oracle


def _load(golden_dir):
    return json.load(open(os.path.join(golden_dir, "worked_numbers.json")))


def _as_printed(value, unit, digits):
    return round(value / unit, digits)


def test_kv_cache_bytes(golden_dir):
    for e in _load(golden_dir)["kv_cache_bytes"]:
        v = oracle.kv_cache_bytes(e["tokens"], e["layers"], e["kv_heads"], e["d_head"],
                                  e["bytes_per_elem"])
        assert _as_printed(v, e["unit"], e["digits"]) == e["printed"], (e["what"], v)


def test_llama3_8b_bytes_per_token_is_exact(golden_dir):
    e = _load(golden_dir)["kv_cache_bytes"][0]
    assert oracle.kv_cache_bytes(1, 32, 8, 128, 2) == 131072 == e["printed"]


def test_mla_cache_bytes(golden_dir):
    for e in _load(golden_dir)["mla_cache_bytes"]:
        v = oracle.mla_cache_bytes(e["tokens"], e["layers"], e["d_latent"], e["d_rope"],
                                   e["bytes_per_elem"])
        assert _as_printed(v, e["unit"], e["digits"]) == e["printed"], (e["what"], v)


def test_mla_is_nine_halves_head_dim():
    # d_c = 4 d_h and d_h^R = d_h / 2 give 9/2 d_h elements per token per layer
    for d_h in (64, 128, 256):
        assert oracle.mla_cache_bytes(1, 1, 4 * d_h, d_h // 2, 1) == 4.5 * d_h


def test_attention_flops_crossover(golden_dir):
    for e in _load(golden_dir)["attention_flops"]:
        per_ctx_token = oracle.attention_flops(1, e["layers"], e["heads"], e["head_dim"])
        crossover = 2 * e["params"] / per_ctx_token
        assert _as_printed(crossover, e["unit"], e["digits"]) == e["printed"], (e["what"], crossover)
