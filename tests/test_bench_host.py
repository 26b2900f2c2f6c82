"""Host-side measurement plumbing of bench.py, on CPU: the roofline
arithmetic of the JSON line (which bound applies, achieved and its fraction
of the peak) and the rule that DRAM counters from a committed ncu summary are
used only while the summary's recorded source hash matches the decode
kernel's sources (comments and whitespace left out)."""
import os

import pytest

import bench

PEAKS = {"hbm_gbs": 8000.0, "bf16_tflops": 2000.0}


def test_roofline_tensor_bound():
    # 4e12 flop at 2000 TFLOP/s = 2 ms; 8e9 B at 8000 GB/s = 1 ms: tensor-bound.
    # Measured 8 ms: achieved 4e12 / 8e-3 = 500 TFLOP/s, a quarter of the peak.
    r = bench.roofline(4e12, 8e9, 8e-3, PEAKS)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(500.0)
    assert r["peak"] == 2000.0
    assert r["frac"] == pytest.approx(0.25)
    assert r["t_roofline_us"] == pytest.approx(2000.0)


def test_roofline_hbm_bound():
    # 1e12 flop = 0.5 ms at the tensor peak; 16e9 B = 2 ms at HBM speed: HBM-bound.
    # Measured 4 ms: achieved 16e9 / 4e-3 = 4000 GB/s, half of the peak.
    r = bench.roofline(1e12, 16e9, 4e-3, PEAKS)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(4000.0)
    assert r["frac"] == pytest.approx(0.5)
    assert r["t_roofline_us"] == pytest.approx(2000.0)


def _fake_tree(tmp_path, decode_src):
    csrc = tmp_path / "sparse_mla_decode_04_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "include").mkdir()
    (tmp_path / "profiles").mkdir()
    (csrc / "smla_decode.cu").write_text(decode_src)
    (csrc / "sm103_ptx.cuh").write_text("int ptx_helper();\n")
    (csrc / "smla_internal.h").write_text("int internal_helper();\n")
    (tmp_path / "include" / "smla.h").write_text("int smla_api();\n")
    return csrc


@pytest.fixture
def fake_root(tmp_path, monkeypatch):
    csrc = _fake_tree(tmp_path, "int kernel() { return 1; }\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SRC", str(csrc / "smla_decode.cu"))
    return tmp_path, csrc


def test_source_hash_ignores_comments_and_whitespace_only(fake_root):
    _, csrc = fake_root
    h0 = bench.kernel_source_hash()
    (csrc / "smla_decode.cu").write_text("// a comment\nint  kernel()\n{ /* block */ return 1; }\n")
    assert bench.kernel_source_hash() == h0
    (csrc / "smla_decode.cu").write_text("int kernel() { return 2; }\n")
    assert bench.kernel_source_hash() != h0
    (csrc / "smla_decode.cu").write_text("int kernel() { return 1; }\n")
    (csrc / "sm103_ptx.cuh").write_text("int ptx_helper(int);\n")  # an included header counts too
    assert bench.kernel_source_hash() != h0


def test_profiled_traffic_only_while_the_hash_matches(fake_root):
    root, csrc = fake_root
    path = root / "profiles" / f"ncu_{bench.KERNEL_NAME}_someworkload.txt"
    assert bench.profiled_traffic("someworkload") is None  # no summary
    path.write_text(f"summary\nsource_hash: {bench.kernel_source_hash()}   (note)\n"
                    "dram_bytes_per_launch: 123456789\n")
    assert bench.profiled_traffic("someworkload") == 123456789.0
    (csrc / "smla_decode.cu").write_text("int kernel() { return 3; }\n")  # the kernel changed since
    assert bench.profiled_traffic("someworkload") is None
    path.write_text("summary without a hash\ndram_bytes_per_launch: 5\n")
    assert bench.profiled_traffic("someworkload") is None


def test_committed_profiles_parse():
    # every committed decode summary names a hash and a byte count in the form
    # profiled_traffic reads
    prof = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles")
    names = [n for n in os.listdir(prof) if n.startswith(f"ncu_{bench.KERNEL_NAME}_")]
    assert names
    for n in names:
        txt = open(os.path.join(prof, n)).read()
        assert "\nsource_hash: " in txt and "\ndram_bytes_per_launch: " in txt, n
