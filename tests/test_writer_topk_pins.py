"""Pins of the oracle's cache writer and top-k selection against hand-evaluated
cases (tests/golden/cache_writer_cases.json), the OCP e4m3 format through torch's
float8 conversion, round trips through the oracle's own dequantiser, a sort in
torch, and negative controls with planted mistakes."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import smla_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")
FX = json.load(open(os.path.join(GOLD, "cache_writer_cases.json")))


def _f(v):
    return float(v) if not isinstance(v, str) else float(v.replace("inf", "inf"))


def test_ue8m0_code_hand_cases():
    for c in FX["codes"]:
        assert O.ue8m0_code_for(_f(c["amax"])) == c["code"], c["work"]


def test_e4m3_encode_hand_cases():
    for v in FX["values"]:
        code = O.ue8m0_code_for(v["amax"])
        assert O.e4m3_encode(v["x"] * math.ldexp(1.0, 127 - code)) == int(v["byte"], 16), v["work"]


def test_e4m3_encode_inverts_decode_on_every_finite_code():
    for c in range(256):
        val = O.E4M3_TABLE[c]
        if math.isnan(val):
            continue
        expect = 0x00 if val == 0.0 else c  # zero is stored as +0
        assert O.e4m3_encode(val) == expect, hex(c)


def test_e4m3_encode_matches_torch_float8_rounding():
    # torch rounds to nearest even on the e4m3fn grid; inside [-448, 448]
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(4000) * 50, rng.standard_normal(2000) * 0.01,
                        (O.E4M3_TABLE[:0x7E] + O.E4M3_TABLE[1:0x7F]) / 2])  # every midpoint
    x = np.clip(x, -448, 448)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([O.e4m3_encode(float(v)) for v in x], dtype=np.uint8)
    ref = np.where((ref & 0x7F) == 0, 0, ref)  # a rounded zero is +0 here
    assert np.array_equal(got, ref)


def test_rope_nan_canonicalisation_hand_cases():
    for c in FX["rope"]:
        bits = np.zeros(512, dtype=np.uint16)
        bits[448] = int(c["bits"], 16)
        entry, _ = O.cache_write_row(bits)
        assert int(entry[448:450].view("<u2")[0]) == int(c["out"], 16), c["work"]


def _latent(n, rng, spread=8):
    x = rng.standard_normal((n, 512)) * np.exp2(rng.integers(-spread, spread, size=(n, 1)))
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_write_then_dequant_round_trip():
    """Dequantising a written entry gives back every value to within e4m3's
    half-unit (relative 2^-4 in the normal range), codes stay in [0, 254], and
    the RoPE half comes back bit-exact."""
    rng = np.random.default_rng(4)
    bits = _latent(40, rng)
    for i in range(bits.shape[0]):
        entry, sc = O.cache_write_row(bits[i])
        assert sc[:7].max() <= 254 and sc[7] == 0
        back = O.dequant_entries(entry[None], sc[None])[0]
        x = O.bf16_bits_to_f64(bits[i])
        for g in range(7):
            grp = slice(64 * g, 64 * g + 64)
            scale = math.ldexp(1.0, int(sc[g]) - 127)
            tol = np.maximum(np.abs(x[grp]) * 2.0 ** -4, 2.0 ** -10 * scale)
            assert np.all(np.abs(back[grp] - x[grp]) <= tol)
            assert np.max(np.abs(x[grp])) / scale <= 448.0
        assert np.array_equal(entry[448:].view("<u2"), bits[i][448:])


def test_values_on_the_grid_are_stored_exactly():
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 0x7F, size=(3, 448))
    bits = np.zeros((3, 512), dtype=np.uint16)
    x = O.E4M3_TABLE[codes] * 2.0 ** 3  # e4m3 values times a power of two
    x[:, ::64] = 448 * 2.0 ** 3          # every group reaches the top of the range
    bits[:, :448] = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for i in range(3):
        entry, sc = O.cache_write_row(bits[i])
        assert np.all(sc[:7] == 130)
        assert np.array_equal(O.dequant_entries(entry[None], sc[None])[0][:448], x[i])


def test_cache_write_skips_bad_slots():
    rng = np.random.default_rng(6)
    bits = _latent(4, rng)
    pool = np.full((3, 576), 0xAB, dtype=np.uint8)
    sc = np.full((3, 8), 0xCD, dtype=np.uint8)
    bad = O.cache_write(bits, np.array([2, -1, 7, 0]), pool, sc)
    assert bad == 1
    assert np.all(pool[1] == 0xAB) and np.all(sc[1] == 0xCD)
    assert np.array_equal(pool[2], O.cache_write_row(bits[0])[0])
    assert np.array_equal(pool[0], O.cache_write_row(bits[3])[0])


def test_topk_hand_cases():
    for c in FX["topk"]:
        s = np.array([[_f(v) if v != "nan" else np.nan for v in c["scores"]]], dtype=np.float32)
        got = O.topk_indices(s, [c["len"]], c["k"])
        assert got[0].tolist() == c["out"], c["work"]


def test_topk_matches_torch_topk_on_distinct_scores():
    rng = np.random.default_rng(7)
    s = rng.permutation(50000).astype(np.float32).reshape(5, 10000) * 0.5
    lens = [10000, 7777, 3000, 2048, 100]
    got = O.topk_indices(s, lens, 2048)
    for r, L in enumerate(lens):
        k = min(2048, L)
        ref = torch.topk(torch.from_numpy(s[r, :L]), k).indices.numpy()
        assert got[r, :k].tolist() == ref.tolist()
        assert np.all(got[r, k:] == -1)


def test_negative_control_writer_mistakes_are_caught():
    """Planted mistakes in copies of the writer's steps each fail a hand case."""
    def encode_half_away(q):  # ties away from zero instead of to even
        mag = min(abs(q), 448.0)
        i = int(np.searchsorted(O._E4M3_POS, mag))
        if i < len(O._E4M3_POS) and O._E4M3_POS[i] == mag:
            c = i
        else:
            c = i if (O._E4M3_POS[i] - mag) <= (mag - O._E4M3_POS[i - 1]) else i - 1
        return 0 if c == 0 else c | (0x80 if q < 0 else 0)

    def code_floor(amax):  # floor instead of the smallest fitting power of two
        return 0 if amax <= 0 else max(0, min(254, 127 + math.floor(math.log2(amax / 448.0)))) if math.isfinite(amax) else 254

    wrong_enc = [v for v in FX["values"]
                 if encode_half_away(v["x"] * math.ldexp(1.0, 127 - O.ue8m0_code_for(v["amax"]))) != int(v["byte"], 16)]
    wrong_code = [c for c in FX["codes"] if code_floor(_f(c["amax"])) != c["code"]]
    assert wrong_enc and wrong_code
