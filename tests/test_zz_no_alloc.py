"""The no-allocation entry point, smla_decode_static_scratch.

It serves callers that cannot call cudaMalloc (plugin interfaces that only
pass inputs, outputs and a stream; code running during CUDA-graph capture;
processes whose device memory belongs to another allocator): its scratch is
a fixed array inside the library.  Its output must agree with smla_decode's,
with a caller-owned workspace, within the tolerance used everywhere else,
on two calls in a row (the second call finds the array as the first left it).
This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import smla_inputs as I
import sparse_mla_decode_04_gb300 as smla
from sparse_mla_decode_04_gb300 import smla as S

OUT_ATOL, OUT_RTOL, LSE_ATOL = 1e-2, 1e-2, 1e-3


def _args(p, out, lse, splits):
    return S.make_args(q_nope=p.q_nope, q_rope=p.q_rope, kv_pool=p.kv_pool, kv_scales=p.kv_scales,
                       main_idx=p.main_idx, topk=p.topk, swa_start=p.swa_start, swa_len=p.swa_len,
                       cmp_pool=p.cmp_pool, cmp_scales=p.cmp_scales, cmp_start=p.cmp_start, cmp_len=p.cmp_len,
                       sink=p.sink, sm_scale=p.sm_scale, out=out, lse=lse, num_splits=splits,
                       block_table=p.block_table, row_seq=p.row_seq)


def _close(a_out, a_lse, b_out, b_lse):
    a = a_out.float().cpu().numpy().astype(np.float64)
    b = b_out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(a - b) <= OUT_ATOL + OUT_RTOL * np.abs(b))
    la, lb = a_lse.cpu().numpy(), b_lse.cpu().numpy()
    assert np.all(np.abs(la - lb) <= LSE_ATOL)


def test_static_scratch_rejects_oversized_calls(smla_lib):
    a = S.smla_decode_args()
    a.num_rows, a.num_heads, a.num_splits = 1024, 128, 32  # needs far more than the built-in array
    assert S.smla_workspace_bytes(1024, 128, 32) > 32 * 1024 * 1024
    assert S.smla_decode_static_scratch(a, 0) == S.SMLA_ERR_WORKSPACE_TOO_SMALL
    assert S.smla_decode_static_scratch(S.smla_decode_args(), 0) == S.SMLA_ERR_BAD_SHAPE


def test_static_scratch_limit_matches_the_header(smla_lib):
    # 32 rows x 128 heads (the DeepSeek-V4-like decode) fits at up to 5 splits;
    # 96 rows never fit at 128 heads, whatever the split count
    assert S.smla_workspace_bytes(32, 128, 5) <= 48 * 1024 * 1024 < S.smla_workspace_bytes(32, 128, 6)
    assert S.smla_workspace_bytes(95, 128, 2) <= 48 * 1024 * 1024 < S.smla_workspace_bytes(96, 128, 1)


def _small(seed, lens):
    return I.build_problem(name="noalloc", seq_lens=list(lens), rows=[(i, L) for i, L in enumerate(lens)], H=128,
                           topk=512, invalid_frac=0.05, swa=128, seed=seed, device="cuda")


def _static_call(p, splits):
    R, H = p.num_rows, p.num_heads
    out = torch.full((R, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((R, H), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = S.smla_decode_static_scratch(_args(p, out, lse, splits), stream)
    assert st == S.SMLA_OK, S.smla_status_string(st)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.gpu
@pytest.mark.parametrize("splits", [1, 3])
def test_static_scratch_matches_workspace_entry_point(cuda_device, splits):
    p = _small(31, (9000, 3000, 700))
    ref_out, ref_lse = smla.decode(p, num_splits=splits)  # existing entry point, caller-owned workspace
    torch.cuda.synchronize()
    for _ in range(2):  # two calls in a row share the array
        out, lse = _static_call(p, splits)
        _close(out, lse, ref_out, ref_lse)


@pytest.mark.gpu
def test_static_scratch_alternating_shapes(cuda_device):
    """Consecutive calls of different shapes and split counts: each finds the
    array as the previous, different call left it."""
    big, one = _small(32, (20000, 9000, 3000)), _small(33, (15000,))
    refs = {}
    for name, p, s in (("big", big, 3), ("one", one, 1)):
        refs[name] = smla.decode(p, num_splits=s)
    torch.cuda.synchronize()
    for name, p, s in (("big", big, 3), ("one", one, 1), ("big", big, 3), ("one", one, 1)):
        out, lse = _static_call(p, s)
        _close(out, lse, *refs[name])


@pytest.mark.gpu
def test_static_scratch_dsv4_size(cuda_device):
    """The largest standard workload that fits the array: 32 rows x 128 heads."""
    p = I.dsv4(device="cuda")
    s = smla.smla_plan_num_splits(p.num_rows, p.num_heads, p.kv_len_estimate())
    assert S.smla_workspace_bytes(p.num_rows, p.num_heads, s) <= 48 * 1024 * 1024
    ref_out, ref_lse = smla.decode(p, num_splits=s)
    torch.cuda.synchronize()
    for _ in range(2):
        out, lse = _static_call(p, s)
        _close(out, lse, ref_out, ref_lse)
