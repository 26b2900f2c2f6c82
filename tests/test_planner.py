"""Host split planner: the C implementation against the oracle's statement of
the cost model (bit-exact integer choice), and its properties."""
import numpy as np
import pytest

import oracle
from sparse_mla_decode_04_gb300 import smla as S


def test_planner_matches_oracle_cost_model_random_coefficients(smla_lib):
    rng = np.random.default_rng(0)
    for _ in range(400):
        c = dict(slots=float(rng.integers(1, 300)), t0=float(rng.uniform(0, 20)),
                 c_entry=float(rng.uniform(1e-4, 0.1)), c_byte=float(10 ** rng.uniform(-9, -5)),
                 c_merge=float(rng.uniform(0, 30)))
        R = int(rng.integers(1, 1025))
        H = int(rng.choice([16, 32, 64, 128, 8, 100]))
        kv = int(rng.integers(0, 1 << 21))
        smax = int(rng.integers(1, 33))
        assert S.smla_plan_num_splits_ex(R, H, kv, c, smax) == oracle.plan_num_splits(R, H, kv, c, smax), (c, R, H, kv)


def test_planner_builtin_coefficients_match_oracle(smla_lib):
    c = S.smla_plan_default_coeffs()
    for R in [1, 2, 4, 16, 32, 64, 256, 1024]:
        for kv in [0, 100, 3000, 10327, 50000, 264000, 1 << 20]:
            assert S.smla_plan_num_splits(R, 128, kv) == oracle.plan_num_splits(R, 128, kv, c, 32)


def test_planner_properties(smla_lib):
    for R in [1, 4, 32, 128]:
        prev = 0
        for kv in [0, 64, 1000, 10000, 100000, 1 << 20]:
            s = S.smla_plan_num_splits(R, 128, kv)
            assert 1 <= s <= 32
            assert s >= prev  # monotone in kv_len at fixed rows
            assert s == S.smla_plan_num_splits(R, 128, kv)  # deterministic
            prev = s
    # one wave already full of long rows: no split
    assert S.smla_plan_num_splits(1024, 128, 10000) == 1
    assert S.smla_plan_num_splits(2, 16, 0) == 1


@pytest.mark.parametrize("args", [(0, 128, 10), (1, 0, 10), (1, 129, 10), (1, 128, -1)])
def test_planner_rejects_bad_arguments(smla_lib, args):
    assert S.smla_plan_num_splits(*args) == -S.SMLA_ERR_BAD_SHAPE


def test_planner_ex_rejects_bad_smax(smla_lib):
    assert S.smla_plan_num_splits_ex(4, 128, 1000, None, 0) == -S.SMLA_ERR_BAD_SHAPE
    assert S.smla_plan_num_splits_ex(4, 128, 1000, None, 33) == -S.SMLA_ERR_BAD_SHAPE
