"""ctypes binding of libsmla.so (see include/smla.h).

Argument marshalling only: every step of the decode runs in the CUDA kernel
behind ``smla_decode``.  There is no fallback: if the library is missing,
``load_library`` raises.
"""
from __future__ import annotations

import ctypes
import threading
from ctypes import POINTER, c_char_p, c_double, c_float, c_int, c_int32, c_int64, c_size_t, c_uint32, c_void_p
from pathlib import Path
from typing import Optional

from ._build import lib_path

SMLA_OK = 0
SMLA_ERR_NULL_POINTER = 1
SMLA_ERR_MISALIGNED = 2
SMLA_ERR_BAD_SHAPE = 3
SMLA_ERR_WORKSPACE_TOO_SMALL = 4
SMLA_ERR_UNSUPPORTED_DEVICE = 5
SMLA_ERR_CUDA = 6

SMLA_DEV_BAD_INDEX = 0x1
SMLA_DEV_BAD_CMP = 0x2
SMLA_DEV_BAD_LENGTH = 0x4
SMLA_DEV_TIMEOUT = 0x8

MAX_HEADS = 128
MAX_ROWS = 1024
MAX_SPLITS = 32


class SmlaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: smla status {status} ({smla_status_string(status)})")


class smla_decode_args(ctypes.Structure):
    _fields_ = [
        ("q_nope", c_void_p), ("q_rope", c_void_p), ("kv_pool", c_void_p), ("kv_scales", c_void_p),
        ("n_main", c_int64), ("block_table", c_void_p), ("pages_per_seq", c_int32), ("row_seq", c_void_p),
        ("main_idx", c_void_p), ("topk", c_int32), ("swa_start", c_void_p), ("swa_len", c_void_p),
        ("cmp_pool", c_void_p), ("cmp_scales", c_void_p), ("n_cmp", c_int64), ("cmp_start", c_void_p),
        ("cmp_len", c_void_p), ("sink", c_void_p), ("sm_scale", c_float), ("out", c_void_p), ("lse", c_void_p),
        ("num_rows", c_int32), ("num_heads", c_int32), ("num_splits", c_int32),
    ]


class smla_plan_coeffs(ctypes.Structure):
    _fields_ = [("slots", c_double), ("t0", c_double), ("c_entry", c_double), ("c_byte", c_double),
                ("c_merge", c_double)]


_lib = None
_lock = threading.Lock()


def load_library(path: Optional[Path] = None) -> ctypes.CDLL:
    """Load libsmla.so once; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = Path(path) if path is not None else lib_path()
        if not p.exists():
            raise RuntimeError(f"{p} is missing: build it first (sparse_mla_decode_04_gb300._build.build())")
        lib = ctypes.CDLL(str(p))
        lib.smla_plan_num_splits.argtypes = [c_int, c_int, c_int64]
        lib.smla_plan_num_splits.restype = c_int
        lib.smla_plan_num_splits_ex.argtypes = [c_int, c_int, c_int64, POINTER(smla_plan_coeffs), c_int]
        lib.smla_plan_num_splits_ex.restype = c_int
        lib.smla_plan_default_coeffs.argtypes = [POINTER(smla_plan_coeffs)]
        lib.smla_plan_default_coeffs.restype = c_int
        lib.smla_workspace_bytes.argtypes = [c_int, c_int, c_int]
        lib.smla_workspace_bytes.restype = c_size_t
        lib.smla_decode.argtypes = [POINTER(smla_decode_args), c_void_p, c_size_t, c_void_p]
        lib.smla_decode.restype = c_int
        lib.smla_read_device_error.argtypes = [c_void_p, POINTER(c_uint32), c_void_p]
        lib.smla_read_device_error.restype = c_int
        lib.smla_status_string.argtypes = [c_int]
        lib.smla_status_string.restype = c_char_p
        _lib = lib
        return lib


# ---------------------------------------------------------------------------
# the C ABI, one Python function per entry point
# ---------------------------------------------------------------------------
def smla_plan_num_splits(num_rows: int, num_heads: int, kv_len: int) -> int:
    return load_library().smla_plan_num_splits(num_rows, num_heads, kv_len)


def smla_plan_num_splits_ex(num_rows: int, num_heads: int, kv_len: int, coeffs: Optional[dict] = None,
                            s_max: int = MAX_SPLITS) -> int:
    c = None
    if coeffs is not None:
        c = smla_plan_coeffs(**{k: float(coeffs[k]) for k in ("slots", "t0", "c_entry", "c_byte", "c_merge")})
    return load_library().smla_plan_num_splits_ex(num_rows, num_heads, kv_len,
                                                  ctypes.byref(c) if c is not None else None, s_max)


def smla_plan_default_coeffs() -> dict:
    c = smla_plan_coeffs()
    st = load_library().smla_plan_default_coeffs(ctypes.byref(c))
    if st != SMLA_OK:
        raise SmlaError(st, "smla_plan_default_coeffs")
    return {k: getattr(c, k) for k, _ in smla_plan_coeffs._fields_}


def smla_workspace_bytes(max_rows: int, num_heads: int, max_splits: int) -> int:
    return int(load_library().smla_workspace_bytes(max_rows, num_heads, max_splits))


def smla_decode(args: smla_decode_args, workspace: int, ws_bytes: int, stream: int = 0) -> int:
    """Enqueue one decode on `stream` (a raw cudaStream_t value).  Returns the status."""
    return load_library().smla_decode(ctypes.byref(args), c_void_p(workspace), c_size_t(ws_bytes),
                                      c_void_p(stream))


def smla_read_device_error(workspace: int, stream: int = 0) -> int:
    flags = c_uint32(0)
    st = load_library().smla_read_device_error(c_void_p(workspace), ctypes.byref(flags), c_void_p(stream))
    if st != SMLA_OK:
        raise SmlaError(st, "smla_read_device_error")
    return int(flags.value)


def smla_status_string(status: int) -> str:
    return load_library().smla_status_string(status).decode()


# ---------------------------------------------------------------------------
# marshalling from torch tensors
# ---------------------------------------------------------------------------
def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def make_args(*, q_nope, q_rope, kv_pool, kv_scales, main_idx, topk, swa_start, swa_len, cmp_pool, cmp_scales,
              cmp_start, cmp_len, sink, sm_scale, out, lse, num_splits, block_table=None, row_seq=None,
              n_main=None, n_cmp=None) -> smla_decode_args:
    """Fill smla_decode_args from device tensors (shapes as in include/smla.h)."""
    a = smla_decode_args()
    a.q_nope, a.q_rope = _ptr(q_nope), _ptr(q_rope)
    a.kv_pool, a.kv_scales = _ptr(kv_pool), _ptr(kv_scales)
    a.n_main = int(kv_pool.shape[0]) if n_main is None else int(n_main)
    a.block_table = _ptr(block_table)
    a.pages_per_seq = int(block_table.shape[1]) if block_table is not None else 0
    a.row_seq = _ptr(row_seq)
    a.main_idx, a.topk = _ptr(main_idx), int(topk)
    a.swa_start, a.swa_len = _ptr(swa_start), _ptr(swa_len)
    a.cmp_pool, a.cmp_scales = _ptr(cmp_pool), _ptr(cmp_scales)
    a.n_cmp = (int(cmp_pool.shape[0]) if cmp_pool is not None else 0) if n_cmp is None else int(n_cmp)
    a.cmp_start, a.cmp_len = _ptr(cmp_start), _ptr(cmp_len)
    a.sink = _ptr(sink)
    a.sm_scale = float(sm_scale)
    a.out, a.lse = _ptr(out), _ptr(lse)
    a.num_rows, a.num_heads = int(q_nope.shape[0]), int(q_nope.shape[1])
    a.num_splits = int(num_splits)
    return a


def smla_decode_static_scratch(args: smla_decode_args, stream: int = 0) -> int:
    """smla_decode with the library's built-in scratch array instead of a
    caller-allocated workspace (for callers that cannot allocate device
    memory; see include/smla.h).  Returns the status."""
    lib = load_library()
    fn = lib.smla_decode_static_scratch
    fn.argtypes = [POINTER(smla_decode_args), c_void_p]
    fn.restype = c_int
    return fn(ctypes.byref(args), c_void_p(stream))


def smla_cache_write(latent: int, num_rows: int, slots: int, pool: int, scales: int, n_pool: int,
                     dev_error: Optional[int] = None, stream: int = 0) -> int:
    """Quantise latent rows into the cache (raw device addresses).  Returns the status."""
    fn = load_library().smla_cache_write
    fn.argtypes = [c_void_p, c_int64, c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_void_p]
    fn.restype = c_int
    return fn(c_void_p(latent), num_rows, c_void_p(slots), c_void_p(pool), c_void_p(scales), n_pool,
              c_void_p(dev_error) if dev_error else None, c_void_p(stream))


def smla_topk_indices(scores: int, stride: int, lens: int, num_rows: int, k: int, out: int, stream: int = 0) -> int:
    """Per-row top-k positions of a score matrix (raw device addresses).  Returns the status."""
    fn = load_library().smla_topk_indices
    fn.argtypes = [c_void_p, c_int64, c_void_p, c_int32, c_int32, c_void_p, c_void_p]
    fn.restype = c_int
    return fn(c_void_p(scores), stride, c_void_p(lens), num_rows, k, c_void_p(out), c_void_p(stream))


def cache_write(latent, slots, pool, scales, dev_error=None, stream: Optional[int] = None) -> None:
    """smla_cache_write on torch device tensors: latent bf16 [n, 512], slots int64
    [n], pool uint8 [N, 576], scales uint8 [N, 8] (written in place)."""
    import torch

    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    st = smla_cache_write(latent.data_ptr(), int(latent.shape[0]), slots.data_ptr(), pool.data_ptr(),
                          scales.data_ptr(), int(pool.shape[0]),
                          dev_error.data_ptr() if dev_error is not None else None, s)
    if st != SMLA_OK:
        raise SmlaError(st, "smla_cache_write")


def topk_indices(scores, lens, k: int, out=None, stream: Optional[int] = None):
    """smla_topk_indices on torch device tensors: scores float32 [R, stride],
    lens int32 [R].  Returns int32 [R, k]."""
    import torch

    R = int(scores.shape[0])
    if out is None:
        out = torch.empty((R, k), dtype=torch.int32, device=scores.device)
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    st = smla_topk_indices(scores.data_ptr(), int(scores.stride(0)), lens.data_ptr(), R, k, out.data_ptr(), s)
    if st != SMLA_OK:
        raise SmlaError(st, "smla_topk_indices")
    return out


def smla_set_wait_limit_ns(ns: int) -> int:
    """Set the decode kernel's wait limit for later launches (0 = default 2 s);
    returns the previous limit (a diagnostic for tests of the timeout path)."""
    fn = load_library().smla_set_wait_limit_ns
    fn.argtypes = [ctypes.c_uint64]
    fn.restype = ctypes.c_uint64
    return int(fn(ns))
