"""The Python binding without a GPU: it loads the built library (no fallback), exposes every
operation, and refuses host tensors before any call into the library."""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvd():
    sys.path.insert(0, ROOT)
    import __graft_entry__ as g
    g._builder().build()          # the library is built in-tree (no GPU needed)
    import kv_cache_decode_split_gb300 as m
    return m


def test_every_public_name_is_callable(kvd):
    for name in kvd.__all__:
        assert hasattr(kvd, name), name
    assert kvd.lib is not None


def _z(*shape, dtype=torch.float32):
    return torch.zeros(*shape, dtype=dtype)


I32 = torch.int32
CALLS = {
    "gqa": lambda m: m.attn_decode_gqa_paged(_z(1, 8, 64), _z(1, 2, 16, 64), _z(1, 2, 16, 64),
                                             _z(1, 1, dtype=I32), _z(1, dtype=I32)),
    "ring": lambda m: m.attn_decode_swa_ring(_z(1, 8, 64), _z(1, 2, 16, 64), _z(1, 2, 16, 64),
                                             _z(1, 1, dtype=I32), _z(1, dtype=I32), 8),
    "append": lambda m: m.cache_append(_z(1, 2, 64), _z(1, 2, 64), _z(1, 2, 16, 64),
                                       _z(1, 2, 16, 64), _z(1, 1, dtype=I32), _z(1, dtype=I32)),
    "delta": lambda m: m.delta_decode_step(_z(2, 32, 64), _z(2, 64), _z(2, 64), _z(2, 32),
                                           _z(2, 64), _z(2)),
    "minmax": lambda m: m.quest_page_minmax(_z(4, 2, 16, 64)),
    "bounds": lambda m: m.quest_page_bounds(_z(1, 8, 64), _z(4, 2, 64), _z(4, 2, 64),
                                            _z(1, 4, dtype=I32), _z(1, dtype=I32), 16),
    "quantize": lambda m: m.quantize_e4m3_rows(_z(4, 128, dtype=torch.bfloat16)),
}


@pytest.mark.parametrize("name", sorted(CALLS))
def test_host_tensors_are_refused(kvd, name):
    with pytest.raises(TypeError, match="CUDA tensor"):
        CALLS[name](kvd)
