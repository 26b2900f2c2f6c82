"""The T x context shape sweep (T in {1..64} rows, context 4K..1M, H = 128,
top-k 2048 with 5% -1, window 128, compressed context // 4): every shape runs
through the C ABI with the planner's split count; up to four rows of each
shape (the first, the last and two between them: with 76 CTA pairs the split
plan cuts every row of a long-context shape at one or more places) are
compared with the oracle element by element, and every output is checked
finite."""
import gc

import pytest
import torch

import smla_inputs as I
import sparse_mla_decode_04_gb300 as smla
from helpers import assert_close, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

SHAPES = [(T, ctx) for T in I.SWEEP_T for ctx in I.SWEEP_CTX]


@pytest.mark.parametrize("T,ctx", SHAPES, ids=[f"T{T}_ctx{c}" for T, c in SHAPES])
def test_sweep_shape(cuda_device, T, ctx):
    p = I.sweep(T, ctx, device="cuda")
    S = smla.smla_plan_num_splits(p.num_rows, p.num_heads, p.kv_len_estimate())
    out, lse = run_gpu(p, num_splits=S)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    rows = sorted({0, T // 3, (2 * T) // 3, T - 1})
    ro, rl = run_oracle(p, rows=rows)
    assert_close(out, lse, ro, rl, rows=rows, what=f"sweep T{T} ctx{ctx} (S={S})")
    del p, out, lse
    gc.collect()
    torch.cuda.empty_cache()
