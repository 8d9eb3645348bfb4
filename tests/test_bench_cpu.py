"""The benchmark's host-side contract, checked without a GPU: the reference
arm (the CPU oracle) prints one JSON line with the keys the measurement
contract asks for, and the committed ncu summaries carry what bench.py needs
to match them to the sources they were taken on."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                         capture_output=True, text=True, timeout=600, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out
    return json.loads(lines[0])


@pytest.mark.parametrize("args", [
    ("--workload", "C1_M4_H256_bf16_nvfp4_rowmajor"),
    ("--op", "gemm", "--gemm", "G1_M41_N4608_K1536"),
])
def test_reference_arm_line(args):
    d = _run("--impl", "reference", "--steps", "1", "--warmup", "0", *args)
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] in args


def test_committed_profiles_are_well_formed():
    """Each kernel summary under profiles/ names its workload, the hash of the
    sources it was taken on and the DRAM bytes per launch; where the hash is
    that of the current sources, bench.py reports those bytes, and they are of
    the order of the algorithmic bytes (no re-read blow-up)."""
    import glob
    import re
    import workloads
    found = 0
    for p in glob.glob(os.path.join(ROOT, "profiles", "*kernel__*.md")):
        text = open(p).read()
        assert re.search(r"^workload:\s*\S+", text, re.M), p
        assert re.search(r"^source_sha256:\s*[0-9a-f]{64}\s*$", text, re.M), p
        assert re.search(r"^dram_bytes_per_launch:\s*[0-9]+\s*$", text, re.M), p
        found += 1
    assert found >= 3
    traffic, _ = bench.recorded_traffic("C3_M8192_H7168_bf16_mxfp4_swizzled_outliers")
    if traffic is not None:
        assert 0.5 < traffic / workloads.C3.algorithmic_bytes() < 1.1


def test_gemm_profile_keys_name_format_kernel_and_tile():
    """Each GEMM capture is keyed by shape, operand format, kernel and tile
    width, so a line never reports another schedule's or format's DRAM bytes."""
    import glob
    import re
    for p in glob.glob(os.path.join(ROOT, "profiles", "gemm_*kernel__*.md")):
        key = re.search(r"^workload:\s*(\S+)", open(p).read(), re.M).group(1)
        kernel = os.path.basename(p).split("__")[0]
        assert re.fullmatch(r".*_" + kernel + r"_n(128|256)", key), p
        assert "_nvfp4_" in key or "_mxfp4_" in key, p
    assert bench.gemm_profile_key("G4", "nvfp4", "k", 256) == "G4_nvfp4_k_n256"


def test_kernel_source_hash_covers_only_each_kernels_files():
    assert bench.kernel_source_sha("fused") != bench.kernel_source_sha("gemm")
    for op, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(ROOT, "rmsnorm_fp4_quant_gb300", "csrc", f)), f
