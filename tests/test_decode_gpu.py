"""CUDA path (through the C ABI) against the float64 oracle, element by element.

Tolerance: |out_gpu - out_ref| <= 1e-2 + 1e-2 |out_ref| (bf16 out) and
|lse_gpu - lse_ref| <= 1e-3, on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
import smla_inputs as I
import sparse_mla_decode_04_gb300 as smla
from helpers import assert_close, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def small(H=64, seed=7, seq_lens=(3000, 1500, 700), topk=100, swa=70, invalid=0.1, mild=False, **kw):
    rows = [(s, L) for s, L in enumerate(seq_lens)]
    return I.build_problem(name="small", seq_lens=list(seq_lens), rows=rows, H=H, topk=topk, invalid_frac=invalid,
                           swa=swa, seed=seed, device="cuda", mild=mild, **kw)


def check(p, num_splits=None, rows=None, what="", workspace=None):
    out, lse = run_gpu(p, num_splits=num_splits, workspace=workspace)
    ro, rl = run_oracle(p, rows=rows)
    return assert_close(out, lse, ro, rl, rows=rows, what=what or p.name)


# ---------------------------------------------------------------------------
def test_tiny(cuda_device):
    check(I.tiny(device="cuda"))


def test_tiny_mild(cuda_device):
    check(I.tiny(device="cuda", mild=True))


@pytest.mark.parametrize("H", [16, 32, 64, 128, 8, 100])
@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("mild", [False, True])
def test_small_heads_and_splits(cuda_device, H, splits, mild):
    check(small(H=H, mild=mild), num_splits=splits, what=f"H{H} s{splits} mild{mild}")


@pytest.mark.parametrize("splits", [1, 2, 5, 8, 17, 32])
def test_forced_splits(cuda_device, splits):
    p = small(H=128, seq_lens=(20000, 12000, 9000, 4000), topk=2048, swa=128, invalid=0.02, seed=11)
    check(p, num_splits=splits, what=f"splits {splits}")


def test_mixed_split_and_unsplit_rows(cuda_device):
    # one long row takes most of the split budget; the short rows stay unsplit
    p = small(H=128, seq_lens=(200000, 300, 64, 5000, 1), topk=512, swa=128, invalid=0.05, seed=12)
    check(p, num_splits=6, what="mixed")
    check(p, num_splits=1, what="mixed s1")


def test_one_very_long_row_takes_the_split_budget(cuda_device):
    # 8 rows at 128 heads with a budget of 8 x 32 units: the chunked plan gives
    # the long row (64000 compressed entries, ~1000 tiles) as many partials as
    # the per-row cap allows; its final merge combines them all
    R = 8
    p = small(H=128, seq_lens=(2000,) * R, topk=32, swa=16, invalid=0.0, seed=21,
              cmp_override=([0] * R, [64000] + [16] * (R - 1), 64000))
    check(p, num_splits=32, what="long row, 32 splits")


def test_every_row_one_split_on_wide_grid(cuda_device):
    # grid of rows*splits units where the live lengths give every row one split
    p = small(H=128, seq_lens=(200, 150, 100, 90), topk=32, swa=16, seed=13)
    check(p, num_splits=16, what="one split per row on a wide grid")


def test_empty_and_degenerate_rows(cuda_device):
    p = small(H=32, seq_lens=(4000, 4000, 4000, 4000, 4000), topk=256, swa=64, seed=14)
    p.main_idx[0] = -1          # row 0: no valid top-k, no window, no compressed -> sink only
    p.swa_len[0] = 0
    p.cmp_len[0] = 0
    p.main_idx[1] = -1          # row 1: compressed only (ragged tail)
    p.swa_len[1] = 0
    p.cmp_len[1] = 77
    p.swa_len[2] = 0            # row 2: top-k only
    p.cmp_len[2] = 0
    p.main_idx[3] = -1          # row 3: window only
    p.cmp_len[3] = 0
    p.cmp_len[4] = 64           # row 4: exactly one full compressed group
    out, lse = run_gpu(p, num_splits=2)
    ro, rl = run_oracle(p)
    assert_close(out, lse, ro, rl, what="degenerate rows")
    assert torch.count_nonzero(out[0]).item() == 0
    assert torch.equal(lse[0].cpu(), p.sink.cpu())


def test_topk_disabled_and_no_sink(cuda_device):
    p = small(H=16, seq_lens=(900, 2000), topk=0, swa=100, seed=15, with_sink=False)
    check(p, num_splits=1, what="no top-k, no sink")
    check(p, num_splits=4, what="no top-k, no sink, split")


def test_duplicate_indices(cuda_device):
    p = small(H=64, seq_lens=(3000,), topk=128, swa=64, seed=16)
    p.main_idx[0, 64:] = p.main_idx[0, :64]  # every top-k slot listed twice
    p.main_idx[0, 5] = int(p.swa_start[0].item()) + 3  # and one also in the window
    check(p, num_splits=1, what="duplicates")


def test_poisoned_unreferenced_memory_is_bit_identical(cuda_device):
    p = I.build_problem(name="poison", seq_lens=[1024], rows=[(0, 1024), (0, 1024)], H=32, topk=128,
                        invalid_frac=0.25, swa=64, seed=17, device="cuda", paged=False, pool_entries=1024,
                        cmp_override=([0, 128], [96, 96], 256), row_seq=True)
    out_a, lse_a = run_gpu(p, num_splits=2)
    ref = set()
    for r in range(2):
        ref.update(v for v in p.main_idx[r].tolist() if v != -1)
        s, n = int(p.swa_start[r]), int(p.swa_len[r])
        ref.update(range(s, s + n))
    unref = torch.tensor(sorted(set(range(1024)) - ref), device="cuda", dtype=torch.long)
    assert unref.numel() > 0
    p.kv_pool[unref] = 0xFF   # NaN e4m3 / NaN bf16 bytes
    p.kv_scales[unref] = 255  # NaN scale code
    tail = torch.tensor(list(range(96, 128)) + list(range(224, 256)), device="cuda")
    p.cmp_pool[tail] = 0xFF
    p.cmp_scales[tail] = 255
    out_b, lse_b = run_gpu(p, num_splits=2)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(lse_a, lse_b)
    assert not torch.isnan(out_b.float()).any()


def test_determinism_20_launches(cuda_device):
    p = small(H=128, seq_lens=(30000, 8000), topk=2048, swa=128, seed=18)
    ws = smla.Workspace(2, 128, 6)
    out0, lse0 = run_gpu(p, num_splits=6, workspace=ws)
    for _ in range(19):
        out, lse = run_gpu(p, num_splits=6, workspace=ws)
        assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
        assert torch.equal(lse, lse0)
    assert ws.read_error() == 0


def test_bad_device_data_sets_error_bits_and_is_dropped(cuda_device):
    p = small(H=16, seq_lens=(2000, 2000, 2000), topk=64, swa=32, seed=19)
    p.main_idx[0, 3] = -7                 # < -1
    p.main_idx[0, 4] = 10 ** 6            # beyond the page table
    p.cmp_start[1] = int(p.cmp_pool.shape[0]) - 10  # compressed range runs off the pool
    ws = smla.Workspace(3, 16, 2)
    out, lse = run_gpu(p, num_splits=2, workspace=ws)
    ro, rl = run_oracle(p)
    assert_close(out, lse, ro, rl, what="bad data")
    flags = ws.read_error()
    assert flags & smla.SMLA_DEV_BAD_INDEX and flags & smla.SMLA_DEV_BAD_CMP
    assert ws.read_error() == 0  # cleared by the read
    p.swa_len[2] = -5
    run_gpu(p, num_splits=2, workspace=ws)
    assert ws.read_error() & smla.SMLA_DEV_BAD_LENGTH


def test_workspace_reuse_across_batch_sizes(cuda_device):
    ws = smla.Workspace(32, 128, 8)
    big = small(H=128, seq_lens=tuple([6000] * 12), topk=512, swa=128, seed=20)
    little = small(H=128, seq_lens=(40000, 100), topk=512, swa=128, seed=21)
    check(big, num_splits=4, workspace=ws, what="big")
    check(little, num_splits=8, workspace=ws, what="little")
    check(big, num_splits=2, workspace=ws, what="big again")
    assert ws.read_error() == 0


def test_graph_replay_with_changing_lengths(cuda_device):
    p = small(H=128, seq_lens=(2000, 9000, 30000, 60000), topk=1024, swa=128, invalid=0.0, seed=22)
    R, H = p.num_rows, p.num_heads
    S = 8
    ws = smla.Workspace(R, H, S)
    out = torch.empty((R, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((R, H), dtype=torch.float32, device="cuda")
    smla.decode(p, num_splits=S, out=out, lse=lse, workspace=ws)  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            smla.decode(p, num_splits=S, out=out, lse=lse, workspace=ws)
    for i in range(6):
        I.redraw_lengths(p, seed=100 + i)
        g.replay()
        torch.cuda.synchronize()
        ro, rl = run_oracle(p)
        assert_close(out, lse, ro, rl, what=f"replay {i}")
    assert ws.read_error() == 0


def test_int64_addressing_large_pool(cuda_device):
    # > 2^31 bytes of main pool; indices near its end (identity mapping) and
    # through a page table whose page ids put rows past 2^31 / 576
    n = 4_000_000
    g = torch.Generator(device="cuda")
    g.manual_seed(23)
    pool, scales = I.make_pool(n, g, "cuda")
    assert n * 576 > 2 ** 31
    R, H, topk = 2, 64, 256
    q = torch.randn((R, H, 512), generator=g, device="cuda").to(torch.bfloat16)
    main = torch.randint(n - 50_000, n, (R, topk), generator=g, device="cuda", dtype=torch.int32)

    class P:  # plain attribute bag for smla.decode / the oracle kwargs below
        pass

    p = P()
    p.q_nope, p.q_rope = q[:, :, :448].contiguous(), q[:, :, 448:].contiguous()
    p.kv_pool, p.kv_scales, p.block_table, p.row_seq = pool, scales, None, None
    p.main_idx, p.topk = main, topk
    p.swa_start = torch.tensor([n - 100, n - 64], dtype=torch.int32, device="cuda")
    p.swa_len = torch.tensor([64, 64], dtype=torch.int32, device="cuda")
    p.cmp_pool, p.cmp_scales, p.cmp_start, p.cmp_len = None, None, None, None
    p.sink = torch.randn((H,), generator=g, device="cuda")
    p.sm_scale = 512 ** -0.5
    out, lse = run_gpu(p, num_splits=2)
    kw = dict(q_nope=p.q_nope.view(torch.int16).cpu().numpy().view(np.uint16),
              q_rope=p.q_rope.view(torch.int16).cpu().numpy().view(np.uint16),
              kv_pool=I.RowReader(pool), kv_scales=I.RowReader(scales), main_idx=main.cpu().numpy(),
              swa_start=p.swa_start.cpu().numpy(), swa_len=p.swa_len.cpu().numpy(), cmp_pool=None,
              cmp_scales=None, cmp_start=None, cmp_len=None, sink=p.sink.cpu().numpy(), sm_scale=p.sm_scale)
    ro, rl = oracle.decode(**kw)
    assert_close(out, lse, ro, rl, what="int64 identity")
    # paged: 2 sequences whose pages sit at the top of the pool
    pages = n // 64
    p.block_table = torch.tensor([[pages - 1, pages - 3], [pages - 2, 5]], dtype=torch.int32, device="cuda")
    p.main_idx = torch.randint(0, 128, (R, topk), generator=g, device="cuda", dtype=torch.int32)
    p.swa_start = torch.tensor([60, 100], dtype=torch.int32, device="cuda")
    p.swa_len = torch.tensor([64, 28], dtype=torch.int32, device="cuda")
    out, lse = run_gpu(p, num_splits=1)
    kw.update(main_idx=p.main_idx.cpu().numpy(), swa_start=p.swa_start.cpu().numpy(),
              swa_len=p.swa_len.cpu().numpy(), block_table=p.block_table.cpu().numpy())
    ro, rl = oracle.decode(**kw)
    assert_close(out, lse, ro, rl, what="int64 paged")


# ---------------------------------------------------------------------------
# full-size workloads, every row against the oracle
# ---------------------------------------------------------------------------
def test_dsv4_decode_all_rows(cuda_device):
    p = I.dsv4(device="cuda")
    S = smla.smla_plan_num_splits(p.num_rows, p.num_heads, p.kv_len_estimate())
    out, lse = run_gpu(p, num_splits=S)
    ro, rl = run_oracle(p)
    assert_close(out, lse, ro, rl, what="dsv4")
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


def test_mtp_decode_all_rows(cuda_device):
    p = I.mtp(device="cuda")
    S = smla.smla_plan_num_splits(p.num_rows, p.num_heads, p.kv_len_estimate())
    out, lse = run_gpu(p, num_splits=S)
    ro, rl = run_oracle(p)
    assert_close(out, lse, ro, rl, what="mtp")


def test_ragged_long_context_all_rows(cuda_device):
    p = I.ragged(device="cuda")
    S = smla.smla_plan_num_splits(p.num_rows, p.num_heads, p.kv_len_estimate())
    out, lse = run_gpu(p, num_splits=S)
    ro, rl = run_oracle(p)
    assert_close(out, lse, ro, rl, what="ragged")


@pytest.mark.parametrize("splits", [8, 32])
@pytest.mark.parametrize("name", ["dsv4", "ragged"])
def test_full_size_mild_forced_splits(cuda_device, name, splits):
    """Scale codes all 127 (logit std about 1): the softmax mixes many
    entries, so the rescales and the merge of many partials are exercised
    where their rounding matters."""
    p = (I.dsv4 if name == "dsv4" else I.ragged)(device="cuda", mild=True)
    out, lse = run_gpu(p, num_splits=splits)
    ro, rl = run_oracle(p)
    assert_close(out, lse, ro, rl, what=f"{name} mild s{splits}")


def test_ragged_graph_capture_replayed_with_redrawn_lengths(cuda_device):
    """The long-context ragged call (contexts 4K/100K/500K/1M) captured once at
    its full lengths, then replayed with new live lengths drawn for every row
    before each replay; every row of every replay against the oracle."""
    p = I.ragged(device="cuda")
    R, H = p.num_rows, p.num_heads
    S = smla.smla_plan_num_splits(R, H, p.kv_len_estimate())
    ws = smla.Workspace(R, H, S)
    out = torch.empty((R, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((R, H), dtype=torch.float32, device="cuda")
    smla.decode(p, num_splits=S, out=out, lse=lse, workspace=ws)  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            smla.decode(p, num_splits=S, out=out, lse=lse, workspace=ws)
    for i in range(5):
        I.redraw_lengths(p, seed=300 + i)
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ro, rl = run_oracle(p)
        assert_close(out, lse, ro, rl, what=f"ragged replay {i}")
    assert ws.read_error() == 0


def _referenced_main_entries(p, row):
    """Physical main-pool rows that `row` reads through its top-k slots."""
    idx = [v for v in p.main_idx[row].tolist() if v != -1]
    bt = p.block_table
    seq = int(p.row_seq[row]) if p.row_seq is not None else row
    out = []
    for pos in idx:
        if bt is None:
            out.append(pos)
        else:
            out.append(int(bt[seq, pos // 64]) * 64 + pos % 64)
    return sorted(set(out))


def test_scale_codes_outside_the_fast_range(cuda_device):
    # Scale codes 0..9 and 135..254 are converted by the exact path; the
    # bytes under the large codes are kept to small subnormal e4m3 values so
    # that the scores stay in a range where fp32 accumulation is accurate.
    p = small(H=64, seq_lens=(3000, 2000), topk=256, swa=64, invalid=0.05, seed=21)
    ents = _referenced_main_entries(p, 0)
    g = torch.Generator().manual_seed(5)
    pick = torch.tensor(ents, dtype=torch.long)[torch.randperm(len(ents), generator=g)[:48]].cuda()
    big, tiny_ = pick[:24], pick[24:]
    grp = 3  # dims 192..255
    small_bytes = torch.randint(0, 8, (big.numel(), 64), generator=g, dtype=torch.uint8)
    small_bytes |= (torch.randint(0, 2, small_bytes.shape, generator=g, dtype=torch.uint8) << 7)
    p.kv_pool[big, 64 * grp:64 * grp + 64] = small_bytes.cuda()
    p.kv_scales[big, grp] = 140
    p.kv_scales[tiny_, 1] = 4
    p.kv_scales[tiny_, 5] = 0
    check(p, num_splits=1, what="codes s1")
    check(p, num_splits=3, what="codes s3")


@pytest.mark.parametrize("dim", [10, 300])
def test_nan_byte_in_a_selected_entry_propagates(cuda_device, dim):
    # e4m3 0x7F is NaN: every row that reads the entry gets NaN, as in the
    # oracle; rows that do not read it stay finite and close.
    p = small(H=32, seq_lens=(2000, 1500), topk=128, swa=64, invalid=0.05, seed=22)
    e = _referenced_main_entries(p, 0)[3]
    p.kv_pool[e, dim] = 0x7F
    out, lse = run_gpu(p, num_splits=2)
    ro, rl = run_oracle(p)
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.float().cpu().numpy().astype(np.float64)
    assert np.isnan(ro[0]).all() and np.isnan(rl[0]).all()
    assert np.array_equal(np.isnan(o), np.isnan(ro)), "NaN pattern differs from the oracle"
    assert np.array_equal(np.isnan(l), np.isnan(rl))
    fin = ~np.isnan(ro)
    assert (np.abs(o[fin] - ro[fin]) <= 1e-2 + 1e-2 * np.abs(ro[fin])).all()


def test_wait_limit_runs_out_and_the_next_call_is_clean(cuda_device):
    """With a wait limit far below what the pipeline needs, the call still
    returns, the workspace error word reports SMLA_DEV_TIMEOUT, and the next
    call with the default limit matches the oracle: the kernel's give-up path
    (every role leaves its loop, issued copies and MMAs are waited for, TMEM is
    freed) leaves nothing behind."""
    from sparse_mla_decode_04_gb300 import smla as S

    p = small(H=128, seq_lens=(20000, 9000, 3000), topk=1024, swa=128, seed=41)
    ws = smla.Workspace(p.num_rows, p.num_heads, 4)
    prev = S.smla_set_wait_limit_ns(100)  # 100 ns: far below one tile
    try:
        for _ in range(3):
            run_gpu(p, num_splits=4, workspace=ws)
        flags = ws.read_error()
    finally:
        S.smla_set_wait_limit_ns(0)
    assert prev == 2_000_000_000
    assert flags & smla.SMLA_DEV_TIMEOUT
    check(p, num_splits=4, workspace=ws, what="after timeouts")
    assert ws.read_error() == 0


@pytest.mark.parametrize("case", ["A-only NoPE", "B-only RoPE", "shared window"])
def test_paired_rows_keep_a_nan_to_the_rows_that_select_it(cuda_device, case):
    """Two rows of one sequence at 64 heads share a work row (their windows and
    compressed entries are gathered once).  A NaN in an entry that only one row
    selects reaches that row alone; one in an entry both select reaches both."""
    p = I.build_problem(name="pair", seq_lens=[3000], rows=[(0, 2999), (0, 3000)], H=64, topk=256,
                        invalid_frac=0.05, swa=64, seed=51, device="cuda", row_seq=True)
    if case == "A-only NoPE":
        only = sorted(set(_referenced_main_entries(p, 0)) - set(_referenced_main_entries(p, 1)))
        p.kv_pool[only[2], 40] = 0x7F
    elif case == "B-only RoPE":
        only = sorted(set(_referenced_main_entries(p, 1)) - set(_referenced_main_entries(p, 0)))
        p.kv_pool[only[5], 470:472] = torch.tensor([0xC0, 0x7F], dtype=torch.uint8, device="cuda")  # bf16 NaN
    else:
        pos = int(p.swa_start[1].item()) + 3  # inside both windows
        e = int(p.block_table[0, pos // 64].item()) * 64 + pos % 64
        p.kv_pool[e, 100] = 0x7F
    out, lse = run_gpu(p, num_splits=2)
    ro, rl = run_oracle(p)
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.float().cpu().numpy().astype(np.float64)
    assert np.isnan(rl).any()
    assert np.array_equal(np.isnan(o), np.isnan(ro)), "NaN pattern differs from the oracle"
    assert np.array_equal(np.isnan(l), np.isnan(rl))
    fin = ~np.isnan(ro)
    assert (np.abs(o[fin] - ro[fin]) <= 1e-2 + 1e-2 * np.abs(ro[fin])).all()
    finl = ~np.isnan(rl)
    assert (np.abs(l[finl] - rl[finl]) <= 1e-3).all()
