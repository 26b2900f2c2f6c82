"""The cache writer and the top-k producer (through the C ABI) against the
oracle: byte-exact cache entries and scale codes, exact index lists."""
import math

import numpy as np
import pytest
import torch

import oracle
import smla_inputs as I
import sparse_mla_decode_04_gb300 as smla
from oracle import smla_oracle as O
from helpers import assert_close

pytestmark = pytest.mark.gpu


def _latent(n, seed, extremes=True):
    """bf16 rows whose groups span many binades; with `extremes`, NaN, +-inf,
    zeros, subnormals and huge values are planted."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((n, 512), generator=g) * torch.exp2(torch.randint(-20, 20, (n, 8), generator=g).float()
                                                        ).repeat_interleave(64, dim=1)
    if extremes:
        x[0, :64] = 0.0                                  # an all-zero group
        x[1, 3] = float("nan")                           # NaN in NoPE
        x[2, 70] = float("inf")                          # inf: code capped at 254
        x[3, 130] = -float("inf")
        x[4, 200:264] = 1e-40                            # bf16 subnormals
        x[5, 300] = 3.0e38                               # near the top of bf16
        x[6, 450] = float("nan")                         # NaN in RoPE
        x[7, :448] = torch.tensor(O.E4M3_TABLE[np.arange(448) % 0x7F]).float() * 2.0 ** -5  # on the grid
        x[8, 100] = 448.0 * 2.0 ** 3                     # exactly a power of two times 448
    bits = x.to(torch.bfloat16)
    return bits


def test_cache_writer_byte_exact(cuda_device):
    n, n_pool = 1200, 1500
    lat = _latent(n, 11)
    g = torch.Generator().manual_seed(12)
    slots = torch.randperm(n_pool, generator=g)[:n].to(torch.int64)
    slots[5] = -1     # a deliberate skip
    slots[9] = n_pool + 3  # out of range: skipped and flagged
    pool = torch.full((n_pool, 576), 0xAB, dtype=torch.uint8, device="cuda")
    scales = torch.full((n_pool, 8), 0xCD, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    smla.cache_write(lat.cuda(), slots.cuda(), pool, scales, dev_error=err)
    torch.cuda.synchronize()
    ref_pool = np.full((n_pool, 576), 0xAB, dtype=np.uint8)
    ref_sc = np.full((n_pool, 8), 0xCD, dtype=np.uint8)
    bad = O.cache_write(lat.view(torch.int16).numpy().view(np.uint16), slots.numpy(), ref_pool, ref_sc)
    assert bad == 1
    assert (int(err.item()) & smla.SMLA_DEV_BAD_INDEX) != 0
    got_pool, got_sc = pool.cpu().numpy(), scales.cpu().numpy()
    diff = np.argwhere(got_pool != ref_pool)
    assert diff.size == 0, f"pool bytes differ at {diff[:5].tolist()}: gpu {got_pool[tuple(diff[0])]:#x} ref {ref_pool[tuple(diff[0])]:#x}"
    assert np.array_equal(got_sc, ref_sc)


def test_cache_writer_feeds_the_decode(cuda_device):
    """Entries written by the writer decode like the oracle's decode of the
    same bytes (the writer and the reader agree on the layout)."""
    p = I.build_problem(name="writer", seq_lens=[4000, 3000], rows=[(0, 4000), (1, 3000)], H=64, topk=256,
                        invalid_frac=0.05, swa=64, seed=13, device="cuda")
    n = p.kv_pool.shape[0]
    g = torch.Generator(device="cuda").manual_seed(14)
    lat = (torch.randn((n, 512), generator=g, device="cuda") * 4).to(torch.bfloat16)
    smla.cache_write(lat, torch.arange(n, device="cuda", dtype=torch.int64), p.kv_pool, p.kv_scales)
    torch.cuda.synchronize()
    out, lse = smla.decode(p, num_splits=2)
    torch.cuda.synchronize()
    ro, rl = oracle.decode(**p.oracle_kwargs())
    assert_close(out, lse, ro, rl, what="decode of written entries")


def test_cache_writer_empty_and_rejects(cuda_device):
    pool = torch.zeros((4, 576), dtype=torch.uint8, device="cuda")
    sc = torch.zeros((4, 8), dtype=torch.uint8, device="cuda")
    lat = torch.zeros((0, 512), dtype=torch.bfloat16, device="cuda")
    smla.cache_write(lat, torch.zeros(0, dtype=torch.int64, device="cuda"), pool, sc)
    st = smla.smla_cache_write(pool.data_ptr() + 8, 1, sc.data_ptr(), pool.data_ptr(), sc.data_ptr(), 4)
    assert st == smla.SMLA_ERR_MISALIGNED


def _scores(R, L, seed, ties=True):
    g = torch.Generator().manual_seed(seed)
    s = torch.randn((R, L), generator=g)
    if ties:
        s = torch.round(s * 8) / 8  # many equal scores
    return s


@pytest.mark.parametrize("k", [1, 100, 2048, 4096])
def test_topk_exact(cuda_device, k):
    R, L = 6, 20000
    s = _scores(R, L, 20 + k)
    s[0, 5] = float("nan")
    s[1, :] = float("nan")                       # nothing selectable: all -1
    s[2, 7] = float("inf")
    s[2, 8] = -float("inf")
    s[3, 100:200] = -0.0
    s[3, 200:300] = 0.0
    lens = torch.tensor([L, L, 5000, 3000, 1000, 10], dtype=torch.int32)
    got = smla.topk_indices(s.cuda(), lens.cuda(), k).cpu().numpy()
    ref = O.topk_indices(s.numpy(), lens.numpy(), k)
    assert np.array_equal(got, ref)


def test_topk_lengths_beyond_the_row_are_cut(cuda_device):
    s = _scores(2, 200, 31)
    lens = torch.tensor([250, 120], dtype=torch.int32)  # row 0 claims more than its 200 positions
    got = smla.topk_indices(s.cuda(), lens.cuda(), 64).cpu().numpy()
    ref = O.topk_indices(s.numpy(), [200, 120], 64)
    assert np.array_equal(got, ref)


def test_topk_full_size_sampled_rows(cuda_device):
    """The decode's largest shape: 64 rows x 1M positions, k = 2048."""
    R, L = 64, 1 << 20
    g = torch.Generator(device="cuda").manual_seed(40)
    s = torch.randn((R, L), generator=g, device="cuda")
    lens = torch.full((R,), L, dtype=torch.int32, device="cuda")
    lens[1] = 777_777
    got = smla.topk_indices(s, lens, 2048)
    torch.cuda.synchronize()
    for r in (0, 1, 63):
        ref = O.topk_indices(s[r:r + 1].cpu().numpy(), [int(lens[r])], 2048)
        assert np.array_equal(got[r:r + 1].cpu().numpy(), ref)


def test_topk_many_ties_at_the_threshold(cuda_device):
    """More keys tied at the k-th score than the selection buffer holds: the
    ordered collection takes the smallest positions among the ties."""
    R, L = 3, 30000
    s = torch.zeros((R, L))
    s[0, ::7] = 1.0                      # 4286 ones, then 25714 zeros tied for the rest
    s[1, :] = 2.5                        # every score equal
    s[2, 5000:] = torch.randn(L - 5000, generator=torch.Generator().manual_seed(3)).round()  # integer ties
    lens = torch.full((R,), L, dtype=torch.int32)
    for k in (100, 4096):
        got = smla.topk_indices(s.cuda(), lens.cuda(), k).cpu().numpy()
        assert np.array_equal(got, O.topk_indices(s.numpy(), lens.numpy(), k))


def test_topk_unaligned_rows_and_ordered_scores(cuda_device):
    """Rows that do not start on a 16-byte boundary (a stride that is not a
    multiple of 4 floats: the scalar path) and scores sorted along the row
    (the sample must still place the threshold)."""
    R, L, stride = 5, 50001, 50003
    g = torch.Generator().manual_seed(61)
    s = torch.randn((R, stride), generator=g)
    s[1] = torch.arange(stride, dtype=torch.float32)          # ascending: the top k sit at the end
    s[2] = -torch.arange(stride, dtype=torch.float32)         # descending: at the start
    s[3, : stride // 2] = float("nan")                        # half the row never selectable
    lens = torch.tensor([L, L, L, L, 77], dtype=torch.int32)
    flat = s.cuda().contiguous()
    for k in (1, 2048, 4096):
        got = smla.smla_topk_indices  # raw entry point: stride in elements, unaligned rows
        out = torch.empty((R, k), dtype=torch.int32, device="cuda")
        st = got(flat.data_ptr(), stride, lens.cuda().data_ptr(), R, k, out.data_ptr(), 0)
        assert st == smla.SMLA_OK
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), O.topk_indices(s.numpy(), lens.numpy(), k)), k


def test_topk_large_rows_sampled_guess(cuda_device):
    """Rows of 4M scores (the sample keeps its density) from three
    distributions, k = 2048, checked in full."""
    R, L = 3, 4 << 20
    g = torch.Generator(device="cuda").manual_seed(62)
    s = torch.randn((R, L), generator=g, device="cuda")
    s[1] = torch.rand((L,), generator=g, device="cuda")            # uniform
    s[2] = torch.exp(4 * torch.randn((L,), generator=g, device="cuda"))  # heavy right tail
    lens = torch.full((R,), L, dtype=torch.int32, device="cuda")
    got = smla.topk_indices(s, lens, 2048).cpu().numpy()
    ref = O.topk_indices(s.cpu().numpy(), lens.cpu().numpy(), 2048)
    assert np.array_equal(got, ref)
