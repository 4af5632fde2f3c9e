"""ctypes loader for libkvdecode.so (built in-tree by ``build.py``).

There is no fallback: if the library is missing or does not load, importing the
package raises, so nothing can silently run another implementation.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvdecode.so")

EXPORTS = (
    "attn_decode_gqa_paged",
    "attn_decode_gqa_paged_static_ws",
    "attn_decode_swa_sink",
    "attn_decode_mla",
    "dsa_indexer_topk",
    "dsa_indexer_topk_fp8",
    "kvd_quantize_e4m3_rows",
    "dsa_indexer_cache_append_fp8",
    "kvd_delta_decode_step",
    "attn_decode_swa_ring",
    "attn_decode_swa_ring_append",
    "kvd_cache_append",
    "quest_page_minmax",
    "quest_select_pages",
    "attn_decode_quest",
    "quest_page_bounds",
    "attn_decode_quest_from_bounds",
    "dsa_topk",
    "attn_decode_mla_sparse",
    "kvd_workspace_size",
    "kvd_check_device_error",
    "kvd_status_string",
    "kvd_set_option",
)

STATUS = {
    0: "KVD_OK", -1: "KVD_ERR_INVALID_ARG", -2: "KVD_ERR_UNSUPPORTED", -3: "KVD_ERR_CUDA",
    -4: "KVD_ERR_TIMEOUT", -5: "KVD_ERR_WORKSPACE_TOO_SMALL", -6: "KVD_ERR_DEVICE_OOB", -7: "KVD_ERR_DEVICE_STATE",
}
OP = {"gqa": 0, "swa": 1, "mla": 2, "dsa_topk": 3, "mla_sparse": 4}
OPTION = {"pdl": 0, "gqa_chunk": 1, "mla_min_tiles": 2, "wait_timeout_test": 3,
          "gqa_cluster": 4}


class KvdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status})")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    gqa = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I]
    lib.attn_decode_gqa_paged.argtypes = gqa + [P, Z, P]
    lib.attn_decode_gqa_paged_static_ws.argtypes = gqa + [P]
    lib.attn_decode_swa_sink.argtypes = gqa + [I, I, P, P, Z, P]
    lib.attn_decode_mla.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, F, P, Z, P]
    lib.dsa_indexer_topk.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, Z, P]
    lib.dsa_indexer_topk_fp8.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, Z,
                                         P]
    lib.kvd_quantize_e4m3_rows.argtypes = [P, P, P, I, I, P]
    lib.dsa_indexer_cache_append_fp8.argtypes = [P, P, P, P, P, I, I, I, I, I, P, P]
    lib.kvd_delta_decode_step.argtypes = [P, P, P, P, P, P, P, I, I, I, I, P]
    lib.attn_decode_swa_ring.argtypes = gqa + [I, I, P, P, Z, P]
    lib.attn_decode_swa_ring_append.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I,
                                                F, I, I, I, P, P, Z, P]
    lib.kvd_cache_append.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, P, P]
    lib.quest_page_minmax.argtypes = [P, P, P, P, I, I, I, I, I, I, P, P]
    lib.quest_select_pages.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, P, P]
    lib.attn_decode_quest.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, P,
                                      P]
    lib.quest_page_bounds.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, P, P]
    lib.attn_decode_quest_from_bounds.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I,
                                                  I, I, F, I, P, P]
    lib.dsa_topk.argtypes = [P, P, P, P, I, I, I, P, Z, P]
    lib.attn_decode_mla_sparse.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, P,
                                           Z, P]
    for name in ("attn_decode_gqa_paged", "attn_decode_gqa_paged_static_ws", "attn_decode_swa_sink", "attn_decode_mla",
                 "dsa_indexer_topk", "dsa_indexer_topk_fp8", "kvd_quantize_e4m3_rows",
                 "dsa_indexer_cache_append_fp8", "kvd_delta_decode_step",
                 "attn_decode_swa_ring", "attn_decode_swa_ring_append", "kvd_cache_append",
                 "quest_page_minmax",
                 "quest_select_pages", "attn_decode_quest", "quest_page_bounds",
                 "attn_decode_quest_from_bounds", "dsa_topk",
                 "attn_decode_mla_sparse",
                 "kvd_check_device_error"):
        getattr(lib, name).restype = I
    lib.kvd_check_device_error.argtypes = [P, P]
    lib.kvd_workspace_size.restype = Z
    lib.kvd_workspace_size.argtypes = [I] * 9
    lib.kvd_status_string.restype = ctypes.c_char_p
    lib.kvd_status_string.argtypes = [I]
    lib.kvd_set_option.restype = I
    lib.kvd_set_option.argtypes = [I, ctypes.c_longlong]
    return lib
