"""Seeded synthetic inputs for sparse-MLA decode.

Shared by the tests, the smoke check and the benchmark: it builds the input
tensors of a decode step and knows nothing of the attention arithmetic.

Recipe (one generator per problem, ``torch.Generator(device)`` seeded with
the problem's seed; values are drawn on the device that will hold them):
  * FP8 payload: e4m3 round-to-nearest-even of N(0, 1) (448 bytes / entry);
  * UE8M0 scale codes: uniform integers in [120, 134] (7 per entry, pad 0);
    the "mild" variant sets every code to 127 (scale 1);
  * RoPE: N(0, 1) rounded to bf16 (64 values / entry, little-endian);
  * q: N(0, 1) in bf16, [R, H, 512] split as NoPE 448 | RoPE 64;
  * sink: N(0, 1) float32 per head;  sm_scale = 1 / sqrt(512);
  * top-k: per row, sampled without replacement from [0, L_row); then a given
    fraction of the slots (rounded) is set to -1 at random positions;
  * pages: 64-token pages; the physical page ids of all sequences are one
    random permutation (random page table);
  * sliding window: the last `swa` positions [L_row - swa, L_row);
  * compressed cache: row-dense, L_seq // 4 entries per sequence; a row uses
    its sequence's region with length L_row // 4.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

ENTRY_BYTES = 576
SCALE_BYTES = 8
NOPE = 448
ROPE = 64
PAGE = 64

SWEEP_T = (1, 2, 4, 8, 16, 32, 48, 64)
SWEEP_CTX = (4096, 32768, 102400, 512000, 1048576)


@dataclass
class Problem:
    name: str
    q_nope: torch.Tensor            # bf16 [R, H, 448]
    q_rope: torch.Tensor            # bf16 [R, H, 64]
    kv_pool: torch.Tensor           # uint8 [N, 576]
    kv_scales: torch.Tensor         # uint8 [N, 8]
    block_table: Optional[torch.Tensor]  # int32 [S, P] or None
    row_seq: Optional[torch.Tensor]      # int32 [R] or None
    main_idx: Optional[torch.Tensor]     # int32 [R, topk] or None
    topk: int
    swa_start: Optional[torch.Tensor]    # int32 [R]
    swa_len: Optional[torch.Tensor]      # int32 [R]
    cmp_pool: Optional[torch.Tensor]     # uint8 [Nc, 576]
    cmp_scales: Optional[torch.Tensor]   # uint8 [Nc, 8]
    cmp_start: Optional[torch.Tensor]    # int32 [R]
    cmp_len: Optional[torch.Tensor]      # int32 [R]
    sink: Optional[torch.Tensor]         # float32 [H]
    sm_scale: float
    meta: dict = field(default_factory=dict)

    @property
    def num_rows(self) -> int:
        return self.q_nope.shape[0]

    @property
    def num_heads(self) -> int:
        return self.q_nope.shape[1]

    @property
    def device(self) -> torch.device:
        return self.q_nope.device

    # -- host-side counts (no attention arithmetic) --------------------------
    def valid_entries_per_row(self) -> np.ndarray:
        """Entries each row attends to (valid top-k + window + compressed),
        assuming every non -1 index resolves (true for generated inputs)."""
        R = self.num_rows
        e = np.zeros(R, dtype=np.int64)
        if self.main_idx is not None and self.topk > 0:
            e += (self.main_idx != -1).sum(dim=1).cpu().numpy().astype(np.int64)
        if self.swa_len is not None:
            e += self.swa_len.cpu().numpy().astype(np.int64)
        if self.cmp_len is not None:
            e += self.cmp_len.cpu().numpy().astype(np.int64)
        return e

    def kv_len_estimate(self) -> int:
        """Per-row entry count a caller would hand to the planner: the
        longest row's top-k slots + window + compressed entries."""
        tot = np.full(self.num_rows, self.topk, dtype=np.int64)
        if self.swa_len is not None:
            tot += self.swa_len.cpu().numpy()
        if self.cmp_len is not None:
            tot += self.cmp_len.cpu().numpy()
        return int(tot.max())

    def algorithmic_bytes(self) -> int:
        """Gathered entry bytes (576 data + 8 scale) of valid entries, q in,
        out, lse and the index list."""
        R, H = self.num_rows, self.num_heads
        E = int(self.valid_entries_per_row().sum())
        return E * (ENTRY_BYTES + SCALE_BYTES) + R * H * 512 * 2 * 2 + R * H * 4 + R * self.topk * 4

    def algorithmic_flops(self) -> int:
        """2*512 (QK) + 2*512 (PV) per head per valid entry."""
        return int(self.valid_entries_per_row().sum()) * self.num_heads * 2048

    # -- host copies for the oracle -----------------------------------------
    def oracle_kwargs(self) -> dict:
        """Numpy views of the inputs.  Pools stay where they are and are read
        row-wise on demand (``pool[rows]``), so large device pools are never
        copied whole."""
        def np_or_none(t, dtype=None):
            if t is None:
                return None
            a = t.detach().cpu().numpy()
            return a if dtype is None else a.astype(dtype)

        return dict(
            q_nope=self.q_nope.detach().view(torch.int16).cpu().numpy().view(np.uint16),
            q_rope=self.q_rope.detach().view(torch.int16).cpu().numpy().view(np.uint16),
            kv_pool=RowReader(self.kv_pool), kv_scales=RowReader(self.kv_scales),
            main_idx=np_or_none(self.main_idx), swa_start=np_or_none(self.swa_start),
            swa_len=np_or_none(self.swa_len),
            cmp_pool=RowReader(self.cmp_pool) if self.cmp_pool is not None else None,
            cmp_scales=RowReader(self.cmp_scales) if self.cmp_scales is not None else None,
            cmp_start=np_or_none(self.cmp_start), cmp_len=np_or_none(self.cmp_len),
            sink=np_or_none(self.sink) if self.sink is not None else np.full(self.num_heads, -np.inf),
            sm_scale=self.sm_scale, block_table=np_or_none(self.block_table),
            row_seq=np_or_none(self.row_seq),
        )


class RowReader:
    """``reader[int64 rows]`` -> numpy uint8 rows of a (possibly device) tensor."""

    def __init__(self, t: torch.Tensor):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, rows):
        idx = torch.as_tensor(np.asarray(rows, dtype=np.int64), device=self.t.device)
        return self.t.index_select(0, idx).cpu().numpy()


# ---------------------------------------------------------------------------
# building blocks
# ---------------------------------------------------------------------------
def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_pool(n: int, g: torch.Generator, device, mild: bool = False, chunk: int = 1 << 20):
    """n entries of [448 fp8 | 64 bf16] bytes plus [7 UE8M0 codes | pad]."""
    pool = torch.empty((n, ENTRY_BYTES), dtype=torch.uint8, device=device)
    scales = torch.zeros((n, SCALE_BYTES), dtype=torch.uint8, device=device)
    for s in range(0, n, chunk):
        m = min(chunk, n - s)
        nope = torch.randn((m, NOPE), generator=g, device=device).to(torch.float8_e4m3fn)
        pool[s:s + m, :NOPE] = nope.view(torch.uint8)
        rope = torch.randn((m, ROPE), generator=g, device=device).to(torch.bfloat16)
        pool[s:s + m, NOPE:] = rope.view(torch.uint8).reshape(m, 2 * ROPE)
        if mild:
            scales[s:s + m, :7] = 127
        else:
            scales[s:s + m, :7] = torch.randint(120, 135, (m, 7), generator=g, device=device, dtype=torch.uint8)
    return pool, scales


def sample_topk(L: int, topk: int, invalid_frac: float, g: torch.Generator, device) -> torch.Tensor:
    """topk distinct positions from [0, L) (padded with -1 when L < topk),
    then round(invalid_frac * topk) random slots set to -1."""
    idx = torch.full((topk,), -1, dtype=torch.int32, device=device)
    take = min(L, topk)
    if take > 0:
        idx[:take] = torch.randperm(L, generator=g, device=device)[:take].to(torch.int32)
    n_inv = int(round(invalid_frac * topk))
    if n_inv > 0:
        slots = torch.randperm(topk, generator=g, device=device)[:n_inv]
        idx[slots] = -1
    return idx


def build_problem(*, name: str, seq_lens: Sequence[int], rows: Sequence[Tuple[int, int]], H: int,
                  topk: int, invalid_frac: float, swa: int, seed: int, device="cpu", mild: bool = False,
                  paged: bool = True, pool_entries: Optional[int] = None, cmp_ratio: int = 4,
                  cmp_override: Optional[Tuple[List[int], List[int], int]] = None,
                  with_sink: bool = True, row_seq: bool = False) -> Problem:
    """Generic builder.  rows = [(sequence, causal length L_row)]."""
    device = torch.device(device)
    g = _gen(seed, device)
    R = len(rows)
    S = len(seq_lens)
    # main pool + page table
    if paged:
        pages = [math.ceil(L / PAGE) for L in seq_lens]
        total_pages = sum(pages)
        perm = torch.randperm(total_pages, generator=g, device=device).to(torch.int32)
        P = max(pages)
        bt = torch.full((S, P), -1, dtype=torch.int32, device=device)
        o = 0
        for s, ps in enumerate(pages):
            bt[s, :ps] = perm[o:o + ps]
            o += ps
        n_main = total_pages * PAGE
    else:
        bt = None
        n_main = pool_entries if pool_entries is not None else max(seq_lens)
    kv_pool, kv_scales = make_pool(n_main, g, device, mild)
    # compressed pool
    if cmp_override is not None:
        c_start, c_len, n_cmp = cmp_override
    else:
        bases, b = [], 0
        for L in seq_lens:
            bases.append(b)
            b += L // cmp_ratio
        n_cmp = b
        c_start = [bases[s] for s, _ in rows]
        c_len = [Lr // cmp_ratio for _, Lr in rows]
    cmp_pool, cmp_scales = make_pool(max(n_cmp, 1), g, device, mild)
    # queries, sink
    q = torch.randn((R, H, NOPE + ROPE), generator=g, device=device).to(torch.bfloat16)
    q_nope = q[:, :, :NOPE].contiguous()
    q_rope = q[:, :, NOPE:].contiguous()
    sink = torch.randn((H,), generator=g, device=device, dtype=torch.float32) if with_sink else None
    # index lists
    main = torch.stack([sample_topk(Lr, topk, invalid_frac, g, device) for _, Lr in rows]) if topk > 0 else None
    swa_start = torch.tensor([max(0, Lr - swa) for _, Lr in rows], dtype=torch.int32, device=device)
    swa_len = torch.tensor([min(swa, Lr) for _, Lr in rows], dtype=torch.int32, device=device)
    seqs = torch.tensor([s for s, _ in rows], dtype=torch.int32, device=device)
    return Problem(
        name=name, q_nope=q_nope, q_rope=q_rope, kv_pool=kv_pool, kv_scales=kv_scales,
        block_table=bt, row_seq=seqs if row_seq else None, main_idx=main, topk=topk,
        swa_start=swa_start, swa_len=swa_len, cmp_pool=cmp_pool, cmp_scales=cmp_scales,
        cmp_start=torch.tensor(c_start, dtype=torch.int32, device=device),
        cmp_len=torch.tensor(c_len, dtype=torch.int32, device=device),
        sink=sink, sm_scale=1.0 / math.sqrt(512.0),
        meta=dict(seq_lens=list(seq_lens), rows=list(rows), live_rows=list(rows), seed=seed, mild=mild,
                  swa=swa, cmp_ratio=cmp_ratio),
    )


# ---------------------------------------------------------------------------
# the named workloads
# ---------------------------------------------------------------------------
def tiny(device="cpu", seed: int = 0, mild: bool = False) -> Problem:
    """2 rows x 16 heads over one 1024-entry pool (identity pages); top-k 128
    with 10% -1; window 64 ([960, 1024)); 96 compressed entries per row (one
    full 64-group + a 32-entry tail) in separate regions."""
    return build_problem(name="tiny", seq_lens=[1024], rows=[(0, 1024), (0, 1024)], H=16, topk=128,
                         invalid_frac=0.10, swa=64, seed=seed, device=device, mild=mild, paged=False,
                         pool_entries=1024, cmp_override=([0, 96], [96, 96], 192), row_seq=True)


def dsv4(device="cuda", seed: int = 1, mild: bool = False) -> Problem:
    """32 sequences x 1 token, 128 heads, 32K context in 64-token pages (random
    page table), top-k 2048 with 2% -1, window 128, 8192 compressed entries."""
    return build_problem(name="dsv4_decode_32x32k_h128", seq_lens=[32768] * 32,
                         rows=[(s, 32768) for s in range(32)], H=128, topk=2048, invalid_frac=0.02,
                         swa=128, seed=seed, device=device, mild=mild)


def mtp(device="cuda", seed: int = 2, mild: bool = False) -> Problem:
    """16 sequences x 4 query tokens (64 rows), 64 heads, context 8K; token t
    of a sequence sees L_t = 8192 - 4 + 1 + t positions; per-token top-k 1024;
    window 128 ending at L_t; compressed L_t // 4."""
    T, ctx = 4, 8192
    rows = [(s, ctx - T + 1 + t) for s in range(16) for t in range(T)]
    return build_problem(name="mtp_decode_16x4_h64_8k", seq_lens=[ctx] * 16, rows=rows, H=64, topk=1024,
                         invalid_frac=0.0, swa=128, seed=seed, device=device, mild=mild, row_seq=True)


RAGGED_CTX = (4096, 102400, 512000, 1048576)


def ragged(device="cuda", seed: int = 3, mild: bool = False, ctx: Sequence[int] = RAGGED_CTX) -> Problem:
    """4 sequences x 1 token, 128 heads, contexts {4K, 100K, 500K, 1M} in one
    call; top-k 2048; window 128; compressed context // 4."""
    return build_problem(name="ragged_long_4x_h128", seq_lens=list(ctx), rows=[(s, L) for s, L in enumerate(ctx)],
                         H=128, topk=2048, invalid_frac=0.0, swa=128, seed=seed, device=device, mild=mild)


def sweep(T: int, ctx: int, device="cuda", mild: bool = False) -> Problem:
    """One shape of the T x context matrix: T rows (one sequence each), 128
    heads, top-k 2048 with 5% -1, window 128, compressed context // 4;
    seed 1000 + the shape's index (T-major)."""
    index = SWEEP_T.index(T) * len(SWEEP_CTX) + SWEEP_CTX.index(ctx)
    return build_problem(name=f"sweep_T{T}_ctx{ctx}", seq_lens=[ctx] * T, rows=[(s, ctx) for s in range(T)],
                         H=128, topk=2048, invalid_frac=0.05, swa=128, seed=1000 + index, device=device, mild=mild)


def redraw_lengths(p: Problem, seed: int, min_frac: float = 0.25) -> None:
    """In place: draw a new live length L2 in [min_frac * L, L] for every row,
    L its construction-time length, and rebuild that row's window, compressed
    length and top-k positions from it (all within the construction-time
    maxima).  Used for graph replays with changing lengths."""
    g = _gen(seed, p.device)
    swa, ratio = p.meta["swa"], p.meta["cmp_ratio"]
    live = []
    for r, (s, Lr) in enumerate(p.meta["rows"]):
        lo = max(1, int(Lr * min_frac))
        L2 = int(torch.randint(lo, Lr + 1, (1,), generator=g, device=p.device).item())
        live.append((s, L2))
        if p.swa_len is not None:
            w = min(swa, L2)
            p.swa_start[r] = L2 - w
            p.swa_len[r] = w
        if p.cmp_len is not None:
            p.cmp_len[r] = L2 // ratio
        if p.main_idx is not None:
            p.main_idx[r] = sample_topk(L2, p.topk, 0.0, g, p.device)
    p.meta["live_rows"] = live
