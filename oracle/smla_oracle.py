"""Float64 reference for DeepSeek-V4-style sparse MLA decode.

TEST INFRASTRUCTURE ONLY: imported by the tests, the package smoke check and
the benchmark's CPU-baseline leg, never by the library.  Plain NumPy, float64
throughout, one row at a time, no blocking and no fusion, so that each step
can be checked against the sources by eye:

* "[ROCm][DSV4][Perf] Optimize Triton sparse-MLA decode on gfx950" (vLLM pull
  request 52212), section "Design": one 512-wide QK dot over 448 NoPE + 64
  RoPE dims, a 512-wide PV, main/sliding-window work and compressed-cache
  64-entry groups with masked tails, attention sinks, and invalid indices that
  contribute zero probability; section "Design", last paragraph: UE8M0 codes
  are capped at 254, invalid indices give zero probability, and block address
  arithmetic is 64-bit.
* "[ASM] [HIP] [MLA v4 nm] Split plan helper and persistent decode kernel with
  in-kernel split and merge" (ROCm/aiter pull request 6126), summary part 1
  (the split-count cost model) and part 2 (split rows merged from fp32
  partials plus LSE).

Readings taken where the cited pull-request pages are silent: the sink is a logit in the already-scaled domain; the returned LSE is
natural-log and includes the sink; top-k / window / compressed entries form a
multiset (no de-duplication); V is the whole 512-wide dequantised entry; the
dim order is [NoPE 0..447 | RoPE 448..511]; scale g covers NoPE dims
64g..64g+63 and equals 2**(code-127); a row with no valid entry returns
out = 0 and lse = sink.

Data layout read here (the same bytes the CUDA path reads):
  q_nope  uint16 (bf16 bits) [R, H, 448];  q_rope uint16 [R, H, 64]
  kv_pool uint8 [N_main, 576] = 448 fp8-e4m3 NoPE bytes + 64 bf16 RoPE values
  kv_scales uint8 [N_main, 8]  (7 UE8M0 codes + 1 pad byte)
  main_idx int32 [R, topk] logical token positions, -1 = invalid slot
  block_table int32 [S, P] (64-token pages) or None (logical == physical)
  row_seq int32 [R] or None (row r reads sequence r)
  swa_start, swa_len int32 [R]  (logical positions, mapped like main_idx)
  cmp_pool uint8 [N_cmp, 576], cmp_scales uint8 [N_cmp, 8],
  cmp_start, cmp_len int32 [R]  (row-dense: entries cmp_start .. +cmp_len-1)
  sink float32 [H], sm_scale float

Pools may be any object that returns uint8 rows for ``pool[int64 array]``.
"""
from __future__ import annotations

import math
from typing import Sequence

import numpy as np

PAGE_SIZE = 64
NOPE_DIMS = 448
ROPE_DIMS = 64
HEAD_DIM = NOPE_DIMS + ROPE_DIMS  # 512: QK width and PV width
ENTRY_BYTES = NOPE_DIMS + 2 * ROPE_DIMS  # 576
SCALE_GROUP = 64
N_SCALES = NOPE_DIMS // SCALE_GROUP  # 7


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------
def e4m3_decode(code: int) -> float:
    """OCP FP8 E4M3 ("fn" variant): 1 sign, 4 exponent bits (bias 7),
    3 mantissa bits, subnormals m/8 * 2**-6, S.1111.111 is NaN, no infinity."""
    sign = -1.0 if (code >> 7) & 1 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def ue8m0_scale(code):
    """UE8M0: an unsigned biased exponent, value 2**(code - 127); 255 is NaN
    (the cache writers cap codes at 254, so it never appears in valid data)."""
    code = np.asarray(code, dtype=np.int64)
    out = np.ldexp(1.0, code - 127).astype(np.float64)
    return np.where(code == 255, np.nan, out)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 is the upper half of an IEEE binary32.  NaN patterns are valid
    inputs (they stay NaN; the widening only warns about signalling ones)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# dequantisation of KV entries
# ---------------------------------------------------------------------------
def dequant_entries(raw: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Entry bytes [n, 576] + UE8M0 codes [n, 8] -> float64 [n, 512].

    x[d] = e4m3(b[d]) * 2**(code[d // 64] - 127) for d < 448, and
    x[448 + i] = the i-th bf16 RoPE value (bytes 448 + 2i, little-endian)."""
    raw = np.asarray(raw, dtype=np.uint8).reshape(-1, ENTRY_BYTES)
    scales = np.asarray(scales, dtype=np.uint8).reshape(-1, 8)
    n = raw.shape[0]
    out = np.empty((n, HEAD_DIM), dtype=np.float64)
    nope = E4M3_TABLE[raw[:, :NOPE_DIMS]]
    group_scale = ue8m0_scale(scales[:, :N_SCALES])  # [n, 7]
    for g in range(N_SCALES):
        cols = slice(g * SCALE_GROUP, (g + 1) * SCALE_GROUP)
        out[:, cols] = nope[:, cols] * group_scale[:, g:g + 1]
    rope_bits = raw[:, NOPE_DIMS:].copy().view("<u2")  # [n, 64]
    out[:, NOPE_DIMS:] = bf16_bits_to_f64(rope_bits)
    return out


# ---------------------------------------------------------------------------
# which entries a row attends to
# ---------------------------------------------------------------------------
def _logical_to_physical(pos: int, seq: int, block_table, n_rows: int):
    """Logical token position of a sequence -> physical pool row, or None when
    the position does not resolve to a row inside the pool."""
    if pos < 0:
        return None
    if block_table is None:
        phys = int(pos)
    else:
        page = pos // PAGE_SIZE
        if page >= block_table.shape[1]:
            return None
        pid = int(block_table[seq, page])
        if pid < 0:
            return None
        phys = pid * PAGE_SIZE + pos % PAGE_SIZE  # python int: 64-bit safe
    if phys >= n_rows:
        return None
    return phys


def row_entries(r: int, main_idx, swa_start, swa_len, cmp_start, cmp_len,
                block_table, row_seq, n_main: int, n_cmp: int):
    """The multiset of entries row r attends to, in order: valid top-k slots,
    then the sliding window, then the compressed entries.

    Returns (main_rows, cmp_rows): physical rows into kv_pool and cmp_pool.
    An index of -1 (or anything that does not resolve) contributes nothing."""
    seq = int(row_seq[r]) if row_seq is not None else r
    main_rows = []
    if main_idx is not None:
        for idx in np.asarray(main_idx[r]).tolist():
            if idx == -1:
                continue
            phys = _logical_to_physical(int(idx), seq, block_table, n_main)
            if phys is not None:
                main_rows.append(phys)
    if swa_len is not None:
        start = int(swa_start[r])
        for pos in range(start, start + int(swa_len[r])):
            phys = _logical_to_physical(pos, seq, block_table, n_main)
            if phys is not None:
                main_rows.append(phys)
    cmp_rows = []
    if cmp_len is not None:
        base = int(cmp_start[r])
        for j in range(int(cmp_len[r])):
            phys = base + j
            if 0 <= phys < n_cmp:
                cmp_rows.append(phys)
    return np.asarray(main_rows, dtype=np.int64), np.asarray(cmp_rows, dtype=np.int64)


# ---------------------------------------------------------------------------
# attention for one row
# ---------------------------------------------------------------------------
def decode_row(q: np.ndarray, X: np.ndarray, sink: np.ndarray, sm_scale: float):
    """q [H, 512], X [n, 512] (float64), sink [H] -> out [H, 512], lse [H].

    s[h, e] = sm_scale * <q_h, x_e>;  M = max(sink_h, max_e s);
    Z = exp(sink_h - M) + sum_e exp(s[h, e] - M);  lse = M + ln Z;
    out_h = sum_e exp(s[h, e] - lse) * x_e."""
    q = np.asarray(q, dtype=np.float64)
    X = np.asarray(X, dtype=np.float64).reshape(-1, HEAD_DIM)
    sink = np.asarray(sink, dtype=np.float64)
    H = q.shape[0]
    s = sm_scale * (q @ X.T)  # [H, n]
    m = np.max(s, axis=1) if s.shape[1] else np.full(H, -np.inf)
    M = np.maximum(m, sink)
    out = np.zeros((H, HEAD_DIM), dtype=np.float64)
    lse = np.full(H, -np.inf, dtype=np.float64)
    for h in range(H):
        if M[h] == -np.inf:  # no entry and no sink: nothing to normalise
            continue
        w = np.exp(s[h] - M[h])
        Z = np.exp(sink[h] - M[h]) + np.sum(w)
        lse[h] = M[h] + np.log(Z)
        out[h] = (w / Z) @ X
    return out, lse


def partial_row(q: np.ndarray, X: np.ndarray, sm_scale: float):
    """One split's contribution without the sink: (O, m, l) with
    m = max_e s, l = sum_e exp(s - m), O = sum_e exp(s - m) x_e."""
    q = np.asarray(q, dtype=np.float64)
    X = np.asarray(X, dtype=np.float64).reshape(-1, HEAD_DIM)
    H = q.shape[0]
    if X.shape[0] == 0:
        return np.zeros((H, HEAD_DIM)), np.full(H, -np.inf), np.zeros(H)
    s = sm_scale * (q @ X.T)
    m = np.max(s, axis=1)
    w = np.exp(s - m[:, None])
    return w @ X, m, np.sum(w, axis=1)


def merge_partials(parts: Sequence, sink: np.ndarray):
    """Merge split partials [(O_i, m_i, l_i)] with the sink, in split order:
    M = max(max_i m_i, sink); L = sum_i l_i e^(m_i - M) + e^(sink - M);
    out = sum_i e^(m_i - M) O_i / L; lse = M + ln L."""
    sink = np.asarray(sink, dtype=np.float64)
    H = sink.shape[0]
    M = sink.copy()
    for _, m, _ in parts:
        M = np.maximum(M, m)
    out = np.zeros((H, HEAD_DIM))
    lse = np.full(H, -np.inf)
    for h in range(H):
        if M[h] == -np.inf:
            continue
        L = np.exp(sink[h] - M[h])
        acc = np.zeros(HEAD_DIM)
        for O, m, l in parts:
            if m[h] == -np.inf:
                continue
            w = np.exp(m[h] - M[h])
            L += l[h] * w
            acc += w * O[h]
        out[h] = acc / L
        lse[h] = M[h] + np.log(L)
    return out, lse


def _row_q(q_nope, q_rope, r):
    return np.concatenate([bf16_bits_to_f64(q_nope[r]), bf16_bits_to_f64(q_rope[r])], axis=1)


def gather_row_X(r, *, kv_pool, kv_scales, main_idx, swa_start, swa_len, cmp_pool, cmp_scales,
                 cmp_start, cmp_len, block_table=None, row_seq=None, n_main=None, n_cmp=None):
    """Dequantised entries of row r, float64 [n, 512], in attention order."""
    n_main = kv_pool.shape[0] if n_main is None else n_main
    n_cmp = (cmp_pool.shape[0] if cmp_pool is not None else 0) if n_cmp is None else n_cmp
    mrows, crows = row_entries(r, main_idx, swa_start, swa_len, cmp_start, cmp_len,
                               block_table, row_seq, n_main, n_cmp)
    parts = []
    if mrows.size:
        parts.append(dequant_entries(kv_pool[mrows], kv_scales[mrows]))
    if crows.size:
        parts.append(dequant_entries(cmp_pool[crows], cmp_scales[crows]))
    if not parts:
        return np.zeros((0, HEAD_DIM))
    return np.concatenate(parts, axis=0)


def decode(*, q_nope, q_rope, kv_pool, kv_scales, main_idx, swa_start, swa_len, cmp_pool,
           cmp_scales, cmp_start, cmp_len, sink, sm_scale, block_table=None, row_seq=None,
           rows=None, n_main=None, n_cmp=None):
    """Whole decode step (or the listed rows): out float64 [len(rows), H, 512],
    lse float64 [len(rows), H]."""
    R = q_nope.shape[0]
    rows = list(range(R)) if rows is None else list(rows)
    H = q_nope.shape[1]
    outs = np.zeros((len(rows), H, HEAD_DIM))
    lses = np.zeros((len(rows), H))
    sink = np.asarray(sink, dtype=np.float64)
    for i, r in enumerate(rows):
        X = gather_row_X(r, kv_pool=kv_pool, kv_scales=kv_scales, main_idx=main_idx,
                         swa_start=swa_start, swa_len=swa_len, cmp_pool=cmp_pool,
                         cmp_scales=cmp_scales, cmp_start=cmp_start, cmp_len=cmp_len,
                         block_table=block_table, row_seq=row_seq, n_main=n_main, n_cmp=n_cmp)
        outs[i], lses[i] = decode_row(_row_q(q_nope, q_rope, r), X, sink, float(sm_scale))
    return outs, lses


# ---------------------------------------------------------------------------
# split-count planner (host-side cost model)
# ---------------------------------------------------------------------------
def plan_cost(s: int, num_rows: int, num_heads: int, kv_len: int, coeffs: dict) -> float:
    """Modelled time of a call with s splits per row:
    waves(R * s) * (t0 + c_entry * ceil(kv_len / s))
      + [s > 1] * (c_byte * R * H * 512 * 4 * s + c_merge),
    waves(u) = ceil(u / slots): work-group waves times per-wave KV time, plus
    the partial-write / merge cost that splitting adds."""
    waves = -(-(num_rows * s) // int(coeffs["slots"]))
    per_wave = coeffs["t0"] + coeffs["c_entry"] * float(-(-kv_len // s))
    cost = waves * per_wave
    if s > 1:
        cost += coeffs["c_byte"] * float(num_rows * num_heads * HEAD_DIM * 4 * s) + coeffs["c_merge"]
    return cost


def plan_num_splits(num_rows: int, num_heads: int, kv_len: int, coeffs: dict, s_max: int = 32) -> int:
    """argmin over s in [1, s_max] of plan_cost; ties go to the smaller s.
    Depends only on (rows, heads, kv_len) and the per-device coefficients."""
    best_s, best = 1, None
    for s in range(1, s_max + 1):
        c = plan_cost(s, num_rows, num_heads, kv_len, coeffs)
        if best is None or c < best:
            best_s, best = s, c
    return best_s


# ---------------------------------------------------------------------------
# cache writer: latent rows -> FP8 + UE8M0 cache entries
# ---------------------------------------------------------------------------
# "[ROCm][DSV4][Perf] Optimize Triton sparse-MLA decode on gfx950", section
# "Design", last paragraph: the cache writers store NoPE dims as FP8 with one
# UE8M0 scale per 64 dims, cap the UE8M0 codes at 254 and canonicalise RoPE
# NaNs.  Readings: the scale of a group is the
# smallest power of two that brings the group's largest magnitude within the
# e4m3 range (448); codes are clamped to [0, 254]; values are rounded to
# nearest, ties to even, saturating at +-448; a NaN NoPE value is stored as
# 0x7F, a value that rounds to zero as 0x00 (+0), and a NaN RoPE value as the
# canonical bf16 NaN 0x7FC0.
E4M3_MAX = 448.0
BF16_CANONICAL_NAN = 0x7FC0

# the 127 non-negative finite e4m3 codes 0x00..0x7E, ascending in value
_E4M3_POS = E4M3_TABLE[:0x7F]


def ue8m0_code_for(amax: float) -> int:
    """Smallest code c in [0, 254] with amax <= 448 * 2**(c - 127); 254 when
    none fits (an infinite amax)."""
    if not amax > 0.0:  # zero (or an all-NaN group)
        return 0
    for c in range(0, 255):
        if amax <= E4M3_MAX * math.ldexp(1.0, c - 127):
            return c
    return 254


def e4m3_encode(q: float) -> int:
    """Round to the nearest e4m3 value, ties to the even code, saturating at
    +-448; NaN -> 0x7F; a result of zero -> 0x00."""
    if math.isnan(q):
        return 0x7F
    mag = min(abs(q), E4M3_MAX)
    i = int(np.searchsorted(_E4M3_POS, mag))  # first value >= mag
    if i < len(_E4M3_POS) and _E4M3_POS[i] == mag:
        code = i
    else:
        lo, hi = i - 1, i
        dlo, dhi = mag - _E4M3_POS[lo], _E4M3_POS[hi] - mag
        code = lo if (dlo < dhi or (dlo == dhi and lo % 2 == 0)) else hi
    if code == 0:
        return 0x00
    return code | (0x80 if q < 0 else 0)


def cache_write_row(bits) -> tuple:
    """One latent row (uint16 bf16 bits [512]) -> (entry bytes [576], scale
    bytes [8])."""
    bits = np.asarray(bits, dtype=np.uint16)
    x = bf16_bits_to_f64(bits)
    entry = np.zeros(ENTRY_BYTES, dtype=np.uint8)
    sc = np.zeros(8, dtype=np.uint8)
    for g in range(N_SCALES):
        grp = x[g * SCALE_GROUP:(g + 1) * SCALE_GROUP]
        finite_or_inf = grp[~np.isnan(grp)]
        amax = float(np.max(np.abs(finite_or_inf))) if finite_or_inf.size else 0.0
        c = ue8m0_code_for(amax)
        sc[g] = c
        for d in range(SCALE_GROUP):
            entry[g * SCALE_GROUP + d] = e4m3_encode(grp[d] * math.ldexp(1.0, 127 - c))
    rope = bits[NOPE_DIMS:].copy()
    nan = ((rope & 0x7F80) == 0x7F80) & ((rope & 0x007F) != 0)
    rope[nan] = BF16_CANONICAL_NAN
    entry[NOPE_DIMS:] = rope.astype("<u2").view(np.uint8)
    return entry, sc


def cache_write(latent_bits, slots, pool, scales):
    """Write rows i with 0 <= slots[i] < len(pool) into pool / scales (numpy
    arrays, modified in place); other slots are skipped.  Returns the number of
    rows skipped for an out-of-range slot (slot -1 is a deliberate skip)."""
    bad = 0
    for i, s in enumerate(np.asarray(slots).tolist()):
        if s == -1:
            continue
        if s < -1 or s >= pool.shape[0]:
            bad += 1
            continue
        pool[s], scales[s] = cache_write_row(latent_bits[i])
    return bad


# ---------------------------------------------------------------------------
# top-k selection: the producer of main_idx
# ---------------------------------------------------------------------------
# The step before the decode: each row's top-k index list (-1 = invalid slot)
# is the k positions of [0, L_r) with the largest scores.  The vLLM page names
# the producer (the indexer top-k path and its cp-gather, "8k/1k TP8 follow-up",
# item 2) but not how scores are made, so scores are an input here.
# Readings: order by score descending, ties by position ascending; NaN scores
# are never selected; rows with fewer than k selectable positions are padded
# with -1.
def topk_indices(scores, lens, k: int) -> np.ndarray:
    scores = np.asarray(scores, dtype=np.float32)
    R = scores.shape[0]
    out = np.full((R, k), -1, dtype=np.int32)
    for r in range(R):
        L = int(lens[r])
        s = scores[r, :L].astype(np.float64)
        pos = np.arange(L)
        keep = ~np.isnan(s)
        s, pos = s[keep], pos[keep]
        order = np.lexsort((pos, -s))  # last key first: score descending, then position
        take = order[:k]
        out[r, :take.size] = pos[take]
    return out
