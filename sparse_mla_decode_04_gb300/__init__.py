"""GB300 (sm_103a) sparse multi-head latent attention decode.

The compute path is libsmla.so (include/smla.h): a host split planner, a
persistent tcgen05 decode kernel and a GPU-wide merge kernel for rows that the
in-kernel split plan cuts into several partials.  This
package is its Python binding: the C entry points under the same names
(``smla_decode``, ``smla_plan_num_splits``, ...), plus ``Workspace`` and
``decode`` helpers that take torch device tensors.  PyTorch supplies device
memory and streams only; there is no CPU fallback.
"""
from __future__ import annotations

from typing import Optional

from ._build import build, lib_path  # noqa: F401
from .smla import (  # noqa: F401
    MAX_HEADS, MAX_ROWS, MAX_SPLITS, SMLA_DEV_BAD_CMP, SMLA_DEV_BAD_INDEX, SMLA_DEV_BAD_LENGTH,
    SMLA_DEV_TIMEOUT, SMLA_ERR_BAD_SHAPE, SMLA_ERR_CUDA, SMLA_ERR_MISALIGNED, SMLA_ERR_NULL_POINTER,
    SMLA_ERR_UNSUPPORTED_DEVICE, SMLA_ERR_WORKSPACE_TOO_SMALL, SMLA_OK, SmlaError, load_library, make_args,
    smla_decode, smla_decode_args, smla_plan_default_coeffs, smla_plan_num_splits, smla_plan_num_splits_ex,
    smla_read_device_error, smla_status_string, smla_workspace_bytes, smla_cache_write, smla_topk_indices,
    cache_write, topk_indices,
)


class Workspace:
    """A zeroed device workspace sized by smla_workspace_bytes (allocate it
    outside graph capture; calls sharing it must be ordered on one stream)."""

    def __init__(self, max_rows: int, num_heads: int, max_splits: int, device="cuda"):
        import torch

        self.nbytes = smla_workspace_bytes(max_rows, num_heads, max_splits)
        if self.nbytes == 0:
            raise SmlaError(SMLA_ERR_BAD_SHAPE, "smla_workspace_bytes")
        self.buf = torch.zeros(self.nbytes + 256, dtype=torch.uint8, device=device)
        self.ptr = (self.buf.data_ptr() + 255) // 256 * 256

    def read_error(self, stream: Optional[int] = None) -> int:
        import torch

        s = torch.cuda.current_stream().cuda_stream if stream is None else stream
        return smla_read_device_error(self.ptr, s)


def decode(p, *, num_splits: Optional[int] = None, out=None, lse=None, workspace: Optional[Workspace] = None,
           stream: Optional[int] = None):
    """Run smla_decode on the tensors of `p` (any object with the attributes of
    the C argument struct: q_nope, q_rope, kv_pool, ...).  Returns (out, lse)."""
    import torch

    R, H = p.q_nope.shape[0], p.q_nope.shape[1]
    if num_splits is None:
        kv = p.topk + int(p.swa_len.max().item() if p.swa_len is not None else 0) + \
            int(p.cmp_len.max().item() if p.cmp_len is not None else 0)
        num_splits = smla_plan_num_splits(R, H, kv)
        if num_splits < 0:
            raise SmlaError(-num_splits, "smla_plan_num_splits")
    if out is None:
        out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=p.q_nope.device)
    if lse is None:
        lse = torch.empty((R, H), dtype=torch.float32, device=p.q_nope.device)
    if workspace is None:
        workspace = Workspace(R, H, num_splits, device=p.q_nope.device)
    args = make_args(q_nope=p.q_nope, q_rope=p.q_rope, kv_pool=p.kv_pool, kv_scales=p.kv_scales,
                     main_idx=p.main_idx, topk=p.topk, swa_start=p.swa_start, swa_len=p.swa_len,
                     cmp_pool=p.cmp_pool, cmp_scales=p.cmp_scales, cmp_start=p.cmp_start, cmp_len=p.cmp_len,
                     sink=p.sink, sm_scale=p.sm_scale, out=out, lse=lse, num_splits=num_splits,
                     block_table=p.block_table, row_seq=p.row_seq)
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    st = smla_decode(args, workspace.ptr, workspace.nbytes, s)
    if st != SMLA_OK:
        raise SmlaError(st, "smla_decode")
    return out, lse
