"""ctypes binding of libsa.so (the C ABI in include/sparse_attn.h).

Argument marshalling only: tensors are passed as device pointers with their sizes and the
current CUDA stream; every step of the computation runs in the library's kernels.  If the
library has not been built this module raises -- there is no fallback path.
"""

from __future__ import annotations

import ctypes
import glob
import os
import re
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsa.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "sparse_attn.h")

(SA_OK, SA_ERR_INVALID_ARG, SA_ERR_UNSUPPORTED, SA_ERR_CUDA, SA_ERR_INDEX, SA_ERR_WORKSPACE,
 SA_ERR_TIMEOUT) = range(7)
SA_KV_BF16, SA_KV_FP8_E4M3 = 0, 1
SA_FAMILY_AUTO, SA_FAMILY_TCGEN05, SA_FAMILY_MMA_SYNC = 0, 1, 2
SA_SCORE_F32, SA_SCORE_BF16 = 0, 1
SA_INDEXER_MAX_POSITIONS = 49152
SA_STATUS_BYTES = 256

_lock = threading.Lock()
_lib = None


class SparseAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def load() -> ctypes.CDLL:
    """Load libsa.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m sparse_latent_attention_gb300.build` "
                "(or __graft_entry__.build()); there is no non-CUDA fallback")
        lib = ctypes.CDLL(LIB_PATH)
        P, i64, i32, f32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                ctypes.c_size_t)
        lib.sa_sparse_attn.restype = i32
        lib.sa_sparse_attn.argtypes = [P, P, P, i32, P, P, f32, i64, i64, i32, i32, i64, i32, P, P,
                                       sz, P]
        lib.sa_sparse_attn_family.restype = i32
        lib.sa_sparse_attn_family.argtypes = [P, P, P, i32, P, P, f32, i64, i64, i32, i32, i64, i32,
                                              P, P, sz, i32, P]
        lib.sa_sparse_attn_rope.restype = i32
        lib.sa_sparse_attn_rope.argtypes = [P, P, P, i32, P, P, f32, i64, i64, i32, i32, i64, i32,
                                            P, P, sz, P, i64, i32, i64, P]
        lib.sa_indexer_topk.restype = i32
        lib.sa_indexer_topk.argtypes = [P, i32, P, i64, i64, i64, i64, i32, i32, ctypes.c_int32,
                                        P, i64, i64, P]
        lib.sa_hc_split_sinkhorn.restype = i32
        lib.sa_hc_split_sinkhorn.argtypes = [P, i64, i32, P, P, i32, f32, P, P, P, P]
        lib.sa_candidate_blocks.restype = i32
        lib.sa_candidate_blocks.argtypes = [P, i32, i64, i64, i64, i64, i32, i32, i32, P, P]
        lib.sa_sparse_attn_workspace_size.restype = sz
        lib.sa_sparse_attn_workspace_size.argtypes = [i64, i64, i32, i32, i64, i32, i32]
        lib.sa_window_idxs.restype = i32
        lib.sa_window_idxs.argtypes = [i64, i64, i32, P, i64, i64, i64, P]
        lib.sa_act_quant_fp8.restype = i32
        lib.sa_act_quant_fp8.argtypes = [P, i64, i32, i64, P, i64, P, i64, P, i64, P]
        lib.sa_window_write.restype = i32
        lib.sa_window_write.argtypes = [P, i64, i64, i32, i64, i64, i32, P, i64, i64, P, i64, i64,
                                        P, i64, i64, P]
        lib.sa_read_status.restype = i32
        lib.sa_read_status.argtypes = [P, i32, P]
        lib.sa_status_string.restype = ctypes.c_char_p
        lib.sa_status_string.argtypes = [i32]
        lib.sa_version.restype = i32
        lib.sa_version.argtypes = []
        _lib = lib
        return lib


def declared_symbols() -> list[str]:
    """Names of the functions the headers under include/ declare."""
    names = set()
    for header in sorted(glob.glob(os.path.join(os.path.dirname(HEADER), "*.h"))):
        text = re.sub(r"/\*.*?\*/", "", open(header).read(), flags=re.S)
        names.update(re.findall(r"\b(sa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def status_string(status: int) -> str:
    return load().sa_status_string(int(status)).decode()


def check(status: int, what: str) -> None:
    if status != SA_OK:
        raise SparseAttnError(status, what)


def version() -> int:
    return int(load().sa_version())
