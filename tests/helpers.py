"""Shared test helpers: run the CUDA path, run the oracle, compare."""
import numpy as np
import torch

import oracle
import sparse_mla_decode_04_gb300 as smla

OUT_ATOL = 1e-2
OUT_RTOL = 1e-2
LSE_ATOL = 1e-3


def run_gpu(p, num_splits=None, workspace=None):
    out, lse = smla.decode(p, num_splits=num_splits, workspace=workspace)
    torch.cuda.synchronize()
    return out, lse


def run_oracle(p, rows=None):
    return oracle.decode(rows=rows, **p.oracle_kwargs())


def assert_close(out_gpu, lse_gpu, out_ref, lse_ref, rows=None, what=""):
    """|gpu - ref| <= 1e-2 + 1e-2 |ref| on bf16 out; |dLSE| <= 1e-3."""
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    l = lse_gpu.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        o, l = o[rows], l[rows]
    assert o.shape == out_ref.shape, (o.shape, out_ref.shape)
    err = np.abs(o - out_ref)
    bound = OUT_ATOL + OUT_RTOL * np.abs(out_ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: out mismatch at {tuple(i)}: gpu {o[tuple(i)]} ref {out_ref[tuple(i)]} "
                             f"({int(bad.sum())} of {bad.size} outside tolerance)")
    both_inf = np.isneginf(l) & np.isneginf(lse_ref)
    dl = np.where(both_inf, 0.0, np.abs(l - lse_ref))
    badl = ~(dl <= LSE_ATOL)
    if badl.any():
        i = np.argwhere(badl)[0]
        raise AssertionError(f"{what}: lse mismatch at {tuple(i)}: gpu {l[tuple(i)]} ref {lse_ref[tuple(i)]}")
    return float(err.max(initial=0.0)), float(dl.max(initial=0.0))
