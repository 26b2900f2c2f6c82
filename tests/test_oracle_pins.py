"""Pins of the float64 oracle against things other than itself: spec values,
hand-evaluated closed forms, library routines (torch float8 decoding, torch
SDPA and logsumexp in float64), invariants, and a negative control."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import smla_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=0):
    return np.random.default_rng(seed)


def _rand_entries(n, rng, codes=(120, 135)):
    """Random raw entries: e4m3 bytes avoiding the NaN codes, bf16 RoPE, UE8M0 codes."""
    nope = rng.integers(0, 256, size=(n, 448), dtype=np.uint8)
    nope[(nope & 0x7F) == 0x7F] = 0x38
    rope = torch.randn(n, 64, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint8)
    raw = np.concatenate([nope, rope.reshape(n, 128)], axis=1)
    sc = np.zeros((n, 8), dtype=np.uint8)
    sc[:, :7] = rng.integers(codes[0], codes[1], size=(n, 7))
    return raw, sc


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------
def test_e4m3_against_ocp_spec_values():
    fx = json.load(open(os.path.join(GOLD, "e4m3_ocp_values.json")))
    for code, val in fx["codes"].items():
        got = O.e4m3_decode(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), code


def test_e4m3_table_matches_torch_float8_decode_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.E4M3_TABLE
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_ue8m0():
    assert O.ue8m0_scale(127) == 1.0
    assert O.ue8m0_scale(128) == 2.0
    assert O.ue8m0_scale(120) == 2.0 ** -7
    assert O.ue8m0_scale(0) == 2.0 ** -127
    assert O.ue8m0_scale(254) == 2.0 ** 127
    assert np.isnan(O.ue8m0_scale(255))


def test_bf16_decode_matches_torch():
    x = torch.randn(1000, dtype=torch.float32).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.bf16_bits_to_f64(bits), x.to(torch.float64).numpy())


def test_dequant_matches_torch_decode_and_scale_groups():
    rng = _rng(1)
    raw, sc = _rand_entries(37, rng)
    X = O.dequant_entries(raw, sc)
    t_nope = torch.from_numpy(raw[:, :448].copy()).view(torch.float8_e4m3fn).to(torch.float64)
    scale = torch.pow(2.0, torch.from_numpy(sc[:, :7].astype(np.float64)) - 127.0)
    ref_nope = t_nope * scale.repeat_interleave(64, dim=1)
    ref_rope = torch.from_numpy(raw[:, 448:].copy()).view(torch.bfloat16).to(torch.float64)
    assert np.array_equal(X[:, :448], ref_nope.numpy())
    assert np.array_equal(X[:, 448:], ref_rope.numpy())


def test_dequant_exact_in_bf16_for_configured_codes():
    """e4m3 value x 2^(-7..7) is exactly representable in bf16: the kernel's
    bf16 dequant adds no error at the configured scale codes."""
    rng = _rng(2)
    raw, sc = _rand_entries(64, rng, codes=(120, 135))
    X = O.dequant_entries(raw, sc)
    rt = torch.from_numpy(X).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(rt, X)


# ---------------------------------------------------------------------------
# entry selection and addressing
# ---------------------------------------------------------------------------
def test_page_table_mapping_hand_cases():
    fx = json.load(open(os.path.join(GOLD, "page_table_cases.json")))
    bt = np.array(fx["block_table"], dtype=np.int64)
    for c in fx["cases"]:
        got = O._logical_to_physical(c["pos"], c["seq"], bt, 1 << 40)
        assert got == c["phys"], c


def test_row_entries_order_and_masking():
    # one sequence, identity pages, 300 rows in the pool
    main = np.array([[5, -1, 7, 299, 300, -1, 5]], dtype=np.int32)  # 300 is out of the pool
    mrows, crows = O.row_entries(0, main, np.array([290]), np.array([4]), np.array([10]), np.array([3]),
                                 None, None, 300, 12)
    assert mrows.tolist() == [5, 7, 299, 5, 290, 291, 292, 293]
    assert crows.tolist() == [10, 11]  # 12 is outside the compressed pool


def test_window_goes_through_page_table():
    bt = np.array([[3, 1]], dtype=np.int32)
    mrows, _ = O.row_entries(0, None, np.array([62]), np.array([4]), None, None, bt, None, 1000, 0)
    assert mrows.tolist() == [3 * 64 + 62, 3 * 64 + 63, 64, 65]


def test_compressed_masked_tail():
    _, crows = O.row_entries(0, None, None, None, np.array([100]), np.array([96]), None, None, 0, 1000)
    assert crows.tolist() == list(range(100, 196))


# ---------------------------------------------------------------------------
# attention: closed forms, library routines, invariants
# ---------------------------------------------------------------------------
def _qx(H, n, rng, scale=1.0):
    return rng.standard_normal((H, 512)) * scale, rng.standard_normal((n, 512)) * scale


def test_one_entry_closed_form_golden():
    fx = json.load(open(os.path.join(GOLD, "one_entry_closed_form.json")))
    for c in fx["cases"]:
        q = np.zeros((1, 512))
        x = np.zeros((1, 512))
        for k, v in c["q_nonzero"].items():
            q[0, int(k)] = v
        for k, v in c["x_nonzero"].items():
            x[0, int(k)] = v
        out, lse = O.decode_row(q, x, np.array([c["sink"]]), c["sm_scale"])
        exp = np.zeros(512)
        for k, v in c["out_nonzero"].items():
            exp[int(k)] = v
        np.testing.assert_allclose(out[0], exp, rtol=1e-15, atol=1e-15)
        assert abs(lse[0] - c["lse"]) < 1e-14


def test_dense_equivalence_with_torch_sdpa():
    """Top-k = a permutation of every position, no window, no compressed
    entries, no sink: the result is softmax attention with K = V = X."""
    rng = _rng(3)
    L, H = 200, 8
    raw, sc = _rand_entries(L, rng, codes=(125, 130))
    perm = rng.permutation(L).astype(np.int32)[None, :]
    q = torch.randn(1, H, 512, dtype=torch.float32).to(torch.bfloat16)
    qb = q.view(torch.int16).numpy().view(np.uint16)
    out, lse = O.decode(q_nope=qb[:, :, :448], q_rope=qb[:, :, 448:], kv_pool=raw, kv_scales=sc, main_idx=perm,
                        swa_start=None, swa_len=None, cmp_pool=None, cmp_scales=None, cmp_start=None,
                        cmp_len=None, sink=np.full(H, -np.inf), sm_scale=0.07)
    X = torch.from_numpy(O.dequant_entries(raw, sc))
    qf = q.to(torch.float64)
    ref = torch.nn.functional.scaled_dot_product_attention(qf[:, :, None, :], X[None, None], X[None, None],
                                                           scale=0.07)[:, :, 0, :]
    ref_lse = torch.logsumexp(0.07 * (qf[0] @ X.T), dim=-1)
    np.testing.assert_allclose(out[0], ref[0].numpy(), rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(lse[0], ref_lse.numpy(), rtol=0, atol=1e-10)


def test_duplicate_entry_equals_logit_plus_ln2():
    """An index listed twice counts twice: same as one copy with an additive
    mask of ln 2 on it (torch SDPA with attn_mask)."""
    rng = _rng(4)
    L, H = 50, 4
    q, X = _qx(H, L, rng, 0.3)
    Xd = np.concatenate([X, X[7:8]], axis=0)
    out, _ = O.decode_row(q, Xd, np.full(H, -np.inf), 1.0)
    mask = torch.zeros(H, 1, L, dtype=torch.float64)
    mask[:, :, 7] = math.log(2.0)
    Xt = torch.from_numpy(X)
    ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q)[None, :, None, :], Xt[None, None],
                                                           Xt[None, None], attn_mask=mask[None], scale=1.0)
    np.testing.assert_allclose(out, ref[0, :, 0, :].numpy(), rtol=1e-10, atol=1e-12)


def test_sink_closed_form():
    rng = _rng(5)
    H, n = 6, 40
    q, X = _qx(H, n, rng, 0.2)
    sink = rng.standard_normal(H) * 2
    o0, l0 = O.decode_row(q, X, np.full(H, -np.inf), 1.0)
    o1, l1 = O.decode_row(q, X, sink, 1.0)
    sig = 1.0 / (1.0 + np.exp(sink - l0))
    np.testing.assert_allclose(o1, o0 * sig[:, None], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l1, np.logaddexp(l0, sink), rtol=0, atol=1e-12)


def test_all_invalid_row_reduces_to_sink():
    rng = _rng(6)
    raw, sc = _rand_entries(10, rng)
    sink = np.array([0.3, -1.2], dtype=np.float32)
    q = np.zeros((1, 2, 512), dtype=np.uint16)
    out, lse = O.decode(q_nope=q[:, :, :448], q_rope=q[:, :, 448:], kv_pool=raw, kv_scales=sc,
                        main_idx=np.full((1, 16), -1, dtype=np.int32), swa_start=np.array([0]),
                        swa_len=np.array([0]), cmp_pool=raw, cmp_scales=sc, cmp_start=np.array([0]),
                        cmp_len=np.array([0]), sink=sink, sm_scale=1.0)
    assert np.array_equal(out, np.zeros_like(out))
    np.testing.assert_array_equal(lse[0], sink.astype(np.float64))


def test_permutation_invariance():
    rng = _rng(7)
    raw, sc = _rand_entries(64, rng, codes=(126, 129))
    idx = rng.permutation(64)[:40].astype(np.int32)
    idx[::5] = -1
    q = torch.randn(1, 3, 512).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    kw = dict(q_nope=q[:, :, :448], q_rope=q[:, :, 448:], kv_pool=raw, kv_scales=sc, swa_start=None, swa_len=None,
              cmp_pool=None, cmp_scales=None, cmp_start=None, cmp_len=None, sink=np.array([0.1, 0.2, 0.3]),
              sm_scale=0.05)
    a = O.decode(main_idx=idx[None], **kw)
    b = O.decode(main_idx=rng.permutation(idx)[None], **kw)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-12)


@pytest.mark.parametrize("cuts", [[0, 1, 40], [0, 13, 14, 29, 40], [0, 40, 40]])
def test_split_and_merge_equals_unsplit(cuts):
    rng = _rng(8)
    H = 5
    q, X = _qx(H, 40, rng, 0.4)
    sink = rng.standard_normal(H)
    ref_o, ref_l = O.decode_row(q, X, sink, 0.9)
    parts = [O.partial_row(q, X[a:b], 0.9) for a, b in zip(cuts[:-1], cuts[1:])]
    out, lse = O.merge_partials(parts, sink)
    np.testing.assert_allclose(out, ref_o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)


def test_constant_v_scaled_by_one_minus_sink_mass():
    rng = _rng(9)
    H, n = 4, 30
    q = rng.standard_normal((H, 512))
    v = rng.standard_normal(512)
    X = np.tile(v, (n, 1))
    sink = rng.standard_normal(H)
    out, lse = O.decode_row(q, X, sink, 0.01)
    np.testing.assert_allclose(out, v[None, :] * (1 - np.exp(sink - lse))[:, None], rtol=1e-12, atol=1e-13)


def test_brute_force_tiny_loops():
    """Plain python loops over a 2-head, 3-entry case."""
    rng = _rng(10)
    q, X = _qx(2, 3, rng, 0.5)
    sink = np.array([0.2, -0.4])
    out, lse = O.decode_row(q, X, sink, 0.3)
    for h in range(2):
        s = [0.3 * sum(q[h, d] * X[e, d] for d in range(512)) for e in range(3)]
        Z = math.exp(sink[h]) + sum(math.exp(v) for v in s)
        assert abs(lse[h] - math.log(Z)) < 1e-12
        for d in range(0, 512, 37):
            ref = sum(math.exp(s[e]) / Z * X[e, d] for e in range(3))
            assert abs(out[h, d] - ref) < 1e-12


def test_nan_in_masked_memory_does_not_leak():
    rng = _rng(11)
    raw, sc = _rand_entries(32, rng)
    poisoned = raw.copy()
    poisoned[[3, 9, 20]] = 0x7F  # NaN e4m3 bytes / NaN bf16 in entries nobody selects
    idx = np.array([[1, 2, -1, 5, 31]], dtype=np.int32)
    q = torch.randn(1, 2, 512).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    kw = dict(q_nope=q[:, :, :448], q_rope=q[:, :, 448:], kv_scales=sc, main_idx=idx, swa_start=np.array([6]),
              swa_len=np.array([2]), cmp_pool=raw, cmp_scales=sc, cmp_start=np.array([10]),
              cmp_len=np.array([5]), sink=np.zeros(2), sm_scale=0.05)
    a = O.decode(kv_pool=raw, **kw)
    b = O.decode(kv_pool=poisoned, **kw)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---------------------------------------------------------------------------
# negative control: a planted oracle mistake must be caught by the pins
# ---------------------------------------------------------------------------
def test_negative_control_dropped_sink_in_merge_is_caught(monkeypatch):
    rng = _rng(12)
    H = 3
    q, X = _qx(H, 20, rng, 0.3)
    sink = rng.standard_normal(H)
    ref_o, _ = O.decode_row(q, X, sink, 1.0)
    parts = [O.partial_row(q, X[:7], 1.0), O.partial_row(q, X[7:], 1.0)]
    out, _ = O.merge_partials(parts, np.full(H, -np.inf))  # planted: sink dropped
    assert not np.allclose(out, ref_o, rtol=1e-6, atol=1e-8)


def test_negative_control_wrong_scale_group_is_caught():
    rng = _rng(13)
    raw, sc = _rand_entries(8, rng)
    X = O.dequant_entries(raw, sc)
    sc_bad = sc.copy()
    sc_bad[:, :7] = sc[:, [1, 0, 2, 3, 4, 5, 6]]  # planted: groups 0 and 1 swapped
    assert not np.array_equal(O.dequant_entries(raw, sc_bad), X)


# ---------------------------------------------------------------------------
# planner reference (the cost model itself)
# ---------------------------------------------------------------------------
COEFFS = dict(slots=76, t0=3.0, c_entry=0.02, c_byte=3e-7, c_merge=3.0)


def test_planner_one_wave_single_split_when_kv_short():
    assert oracle.plan_num_splits(64, 128, 100, COEFFS) == 1


def test_planner_monotone_in_kv_len():
    prev = 1
    for kv in [0, 1000, 4000, 16000, 64000, 256000, 1 << 20]:
        s = oracle.plan_num_splits(4, 128, kv, COEFFS)
        assert 1 <= s <= 32 and s >= prev
        prev = s


def test_planner_prefers_one_wave_over_two():
    # 32 rows: s = 2 fills 64 of 76 slots in one wave; s = 3 would need two waves
    assert oracle.plan_num_splits(32, 128, 10327, COEFFS) == 2


# ---------------------------------------------------------------------------
# the cost model's value, pinned by hand-evaluated cases
# ---------------------------------------------------------------------------
def _plan_cases():
    fx = json.load(open(os.path.join(GOLD, "plan_cost_cases.json")))
    return fx, [dict(c, coeffs=c.get("coeffs", fx["coeffs"])) for c in fx["cases"]]


def test_plan_cost_matches_hand_evaluated_cases():
    _, cases = _plan_cases()
    for c in cases:
        got = O.plan_cost(c["s"], c["R"], c["H"], c["kv"], c["coeffs"])
        assert got == pytest.approx(c["cost"], rel=1e-12, abs=1e-12), c["what"]


def test_plan_argmin_matches_hand_evaluated_case():
    fx, _ = _plan_cases()
    for c in fx["argmin"]:
        assert O.plan_num_splits(c["R"], c["H"], c["kv"], fx["coeffs"], c["s_max"]) == c["s"], c["what"]


def _cost_mutants():
    """Plausible mistakes in the cost model, planted in copies of it."""
    def waves(R, s, co):
        return -(-(R * s) // int(co["slots"]))

    def no_split_term(s, R, H, kv, co):
        return waves(R, s, co) * (co["t0"] + co["c_entry"] * float(-(-kv // s)))

    def split_term_without_s(s, R, H, kv, co):
        c = no_split_term(s, R, H, kv, co)
        return c + (co["c_byte"] * float(R * H * 512 * 4) + co["c_merge"] if s > 1 else 0.0)

    def floor_kv(s, R, H, kv, co):
        c = waves(R, s, co) * (co["t0"] + co["c_entry"] * float(kv // s))
        return c + (co["c_byte"] * float(R * H * 512 * 4 * s) + co["c_merge"] if s > 1 else 0.0)

    def floor_waves(s, R, H, kv, co):
        c = max(1, (R * s) // int(co["slots"])) * (co["t0"] + co["c_entry"] * float(-(-kv // s)))
        return c + (co["c_byte"] * float(R * H * 512 * 4 * s) + co["c_merge"] if s > 1 else 0.0)

    def merge_always(s, R, H, kv, co):
        return no_split_term(s, R, H, kv, co) + co["c_byte"] * float(R * H * 512 * 4 * s) + co["c_merge"]

    return [no_split_term, split_term_without_s, floor_kv, floor_waves, merge_always]


@pytest.mark.parametrize("mutant", _cost_mutants(), ids=lambda f: f.__name__)
def test_negative_control_plan_cost_mistakes_are_caught(mutant):
    """Each planted mistake disagrees with at least one hand-evaluated case,
    so the same mistake in the oracle would fail the pin above."""
    _, cases = _plan_cases()
    wrong = [c["what"] for c in cases
             if mutant(c["s"], c["R"], c["H"], c["kv"], c["coeffs"]) != pytest.approx(c["cost"], rel=1e-12)]
    assert wrong, f"{mutant.__name__} passes every golden case"
