"""bench.py's reference arm on CPU: the oracle timed on the host cores, one
JSON line with the contract's keys (rank 0 only), and the row-parallel
oracle figure beside the single-thread value."""
import io
import json
from contextlib import redirect_stdout

import bench


def _run(argv):
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(argv)
    return rc, buf.getvalue()


def test_reference_arm_prints_one_contract_line():
    rc, out = _run(["--impl", "reference", "--steps", "2", "--warmup", "1",
                    "--cpu-seconds", "0.3", "--reference-budget-s", "1"])
    assert rc == 0
    lines = [l for l in out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 2
    assert d["config"]["workload"] == "prefill_bf16_16384x4096"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"]
    assert cb["row_parallel"]["cores"] >= 1 and cb["row_parallel"]["value"] > 0
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_print_nothing():
    import argparse
    args = argparse.Namespace(workload="prefill_bf16_16384x4096", steps=1, warmup=1,
                              reference_budget_s=1.0, cpu_seconds=0.0)
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args, 2, 1) == 0
    assert buf.getvalue() == ""


def test_traffic_record_follows_the_kernel_code_not_its_comments(tmp_path, monkeypatch):
    """roofline.traffic is reported only while the row-kernel sources match the
    capture: a changed comment keeps the hash, a changed statement does not."""
    import shutil
    h_repo = bench.kernel_source_hash("bf16")
    root = tmp_path / "repo"
    for d in ("rmsnorm_fwd_gb300/csrc", "include"):
        (root / d).mkdir(parents=True)
    for n in ["rowreg_bf16.cu", *bench.ROWREG_SOURCES]:
        shutil.copy(f"{bench.ROOT}/rmsnorm_fwd_gb300/csrc/{n}", root / "rmsnorm_fwd_gb300/csrc" / n)
    shutil.copy(f"{bench.ROOT}/include/rmsnorm.h", root / "include/rmsnorm.h")
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.kernel_source_hash("bf16") == h_repo
    p = root / "rmsnorm_fwd_gb300/csrc/rowreg.cuh"
    src = p.read_text()
    p.write_text(src + "\n// a new comment\n/* and a\n   block comment */\n")
    assert bench.kernel_source_hash("bf16") == h_repo
    p.write_text(src.replace("__syncthreads();", "__syncthreads(); __syncthreads();", 1))
    assert bench.kernel_source_hash("bf16") != h_repo
