"""Host logic of bench.py that needs no GPU: the GEMM source hash that ties a
committed ncu summary to the kernel it was taken on, and the lookup of the
summary's DRAM traffic.  A comment-only edit must keep the hash (the summary
still describes the same code); any code edit must change it (the traffic is
then reported as null rather than attributed to a different kernel).  Also
the single-core timing of the oracle's quantizers."""
from __future__ import annotations

import os

import bench


def _tree(tmp_path, gemm: str, ptx: str):
    d = tmp_path / "fp8_fine_grained_act_gb300" / "csrc"
    d.mkdir(parents=True, exist_ok=True)
    (d / "gemm.cu").write_text(gemm)
    (d / "ptx.cuh").write_text(ptx)


GEMM = "int f(int x) {\n    return x + 1;  // add one\n}\n"
PTX = "#define A 1\n"


def test_hash_ignores_comments_and_blank_lines(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _tree(tmp_path, GEMM, PTX)
    h0 = bench.gemm_source_sha()
    _tree(tmp_path, "// header\n\n" + GEMM.replace("// add one", "// increment"), PTX + "\n// note\n")
    assert bench.gemm_source_sha() == h0


def test_hash_changes_with_code(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _tree(tmp_path, GEMM, PTX)
    h0 = bench.gemm_source_sha()
    _tree(tmp_path, GEMM.replace("x + 1", "x + 2"), PTX)
    h1 = bench.gemm_source_sha()
    _tree(tmp_path, GEMM, PTX.replace("1", "2"))
    h2 = bench.gemm_source_sha()
    assert len({h0, h1, h2}) == 3


def test_traffic_only_from_a_summary_of_the_current_code(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _tree(tmp_path, GEMM, PTX)
    summary = tmp_path / "summary.md"
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(summary))
    assert bench.profiled_traffic() is None                        # no summary
    summary.write_text(f"kernel source sha256[:16]: {bench.gemm_source_sha()}\n"
                       "dram bytes per launch (read + write): 123456\n")
    assert bench.profiled_traffic() == 123456
    _tree(tmp_path, GEMM.replace("x + 1", "x - 1"), PTX)              # the kernel changed since
    assert bench.profiled_traffic() is None


def test_committed_summary_names_a_hash_and_traffic():
    text = open(os.path.join(os.path.dirname(bench.__file__), "profiles",
                             "gemm_blockscaled_fprop_4096x18432x7168.md")).read()
    assert "kernel source sha256[:16]:" in text
    assert "dram bytes per launch (read + write):" in text


def test_single_core_quantizer_timing_restores_threads():
    """The oracle's quantizers timed on one core report positive rates and
    leave the oracle's thread count as it was."""
    import oracle
    n0 = oracle.num_threads()
    r = bench.cpu_quantizers_1core(128)
    assert r["cores"] == 1
    assert r["quant_act_1x128"]["GB/s"] > 0 and r["quant_w_128x128"]["GB/s"] > 0
    assert oracle.num_threads() == n0


def test_committed_summaries_describe_the_current_gemm_source():
    """Every committed GEMM summary names the hash of the GEMM source as it
    stands, so the bench reports its DRAM traffic (a stale summary would
    make the traffic null)."""
    prof = os.path.join(os.path.dirname(bench.__file__), "profiles")
    names = [n for n in os.listdir(prof) if n.startswith(("gemm_", "launches_"))]
    assert names
    h = bench.gemm_source_sha()
    for n in names:
        assert h in open(os.path.join(prof, n)).read(), f"{n} was taken on another GEMM source"
