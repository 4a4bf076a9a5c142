"""Host-side logic of the tuning sweep and the benchmark, on the CPU: the
sweep's shared-memory formula agrees with the library's planner, its
summary table, the benchmark's clock-sample reading (nvidia-smi lines and
NVML reason bits) and its lookup of the committed DRAM traffic figure."""
import json

import bench
import rmsnorm_fwd_gb300 as rn
from rmsnorm_fwd_gb300 import inputs, tune

SMS, OPTIN = 152, 232448
BASE = 1 << 40


def test_sweep_staged_smem_matches_the_planner():
    """The sweep sizes staged-ring candidates with its own copy of the
    layout (mbarriers and reduction scratch, then the slots and the weight
    row); every staged plan the library makes must agree with it."""
    checked = 0
    for dtype, es in (("bf16", 2), ("f16", 2), ("f32", 4)):
        for hidden in (1024, 4096, 8192, 16384, 20480, 24576, 32768):
            if hidden * es > 72 * 1024:
                continue
            for rows in (1, 300, 4000):
                rc, p = rn.rmsnorm_plan_status(BASE, 3 * BASE, 5 * BASE, rows, hidden,
                                               rn.DTYPE_CODES[dtype], SMS, OPTIN,
                                               rn.VARIANT_STAGED)
                if rc != rn.OK:
                    continue
                assert p.smem_bytes == tune.staged_smem(hidden * es, p.stages), p.as_dict()
                checked += 1
    assert checked >= 20


def test_sweep_candidates_are_mostly_plans_the_library_takes():
    """Every non-staged candidate of the sweep validates; staged ones may ask
    for rings the library refuses (they are skipped when timed), never for
    another status."""
    lib = rn._load()
    for rows, hidden, dtype in ((16384, 4096, "bf16"), (8192, 1024, "bf16"),
                                (4000, 24576, "bf16"), (8, 65536, "bf16"), (64, 128, "f32"),
                                (1, 1 << 20, "bf16"), (300, 4097, "f16")):
        cands = tune.candidates(rows, hidden, dtype, SMS, OPTIN)
        assert cands
        for c in cands:
            p = rn.Plan(**c)
            rc = lib.rmsnorm_validate_plan(rn.ctypes.byref(p), BASE, 3 * BASE, 5 * BASE, rows,
                                           hidden, rn.DTYPE_CODES[dtype], SMS, OPTIN)
            if c["variant"] == rn.VARIANT_STAGED:
                assert rc in (rn.OK, rn.ERR_VARIANT), (rc, c)
            else:
                assert rc == rn.OK, (rc, c)


def test_sweep_summary_table(tmp_path):
    k = rn.kernels()[0]
    plan = dict(variant=k["variant"] if k["variant"] != 0 else 1, vec_bytes=k["vec_bytes"],
                threads_per_row=32, vecs_per_thread=k["nv"], block_threads=256,
                rows_per_block=8, stages=0, grid=608, smem_bytes=0, kernel_index=k["index"])
    rec = {"hidden_bf16": 1024, "row_bytes": 2048, "class": "mid", "rows": 8192,
           "top": [{"us": 7.0, "GBps": 4792.0, "plan": plan}],
           "auto": {"us": 7.28, "GBps": 4612.0, "plan": plan}}
    path = tmp_path / "grid.jsonl"
    path.write_text(json.dumps(rec) + "\n")
    table = tune.summarize(str(path)).splitlines()
    assert len(table) == 3 and table[0].startswith("| bf16 hidden")
    cells = [c.strip() for c in table[2].strip("|").split("|")]
    assert cells[:5] == ["1024 (2048)", "mid", "8192", "7.00", "4792"]
    assert cells[-1] == "1.040"


def _sampler_with(lines):
    s = bench.ClockSampler(0)
    s.lines = lines
    return s


def test_clock_summary_reads_reasons_inside_the_window():
    ok = "2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active"
    slow = "1500, 2070, 1390.0, 0x8, Active, Not Active, Not Active, Active"
    s = _sampler_with([(9.0, slow), (10.1, ok), (10.2, ok), (10.3, slow), (11.5, slow)])
    c = s.summary(10.0, 10.35)
    assert c["samples"] == 3 and c["sm_max_mhz"] == 2070.0
    assert c["sm_mhz"] == 2070.0                      # median of 2070, 2070, 1500
    assert c["reasons"] == ["hw_slowdown", "sw_power_cap"]
    c = _sampler_with([(10.1, ok), (10.2, ok)]).summary(10.0, 10.3)
    assert c["reasons"] == [] and c["samples"] == 2


def test_clock_summary_short_region_and_no_samples():
    ok = "2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active"
    c = _sampler_with([(9.0, ok), (12.0, ok)]).summary(10.0, 10.001)
    assert c["samples"] == 1 and c["sm_mhz"] == 2070.0   # the nearest sample stands in
    c = _sampler_with([(9.0, "garbled line")]).summary(10.0, 10.1)
    assert c == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}


def test_traffic_lookup_follows_workload_variant_and_sources():
    wl = inputs.WORKLOADS[inputs.HEADLINE]
    v = bench.ncu_traffic(wl, "cta_per_row")
    assert v is not None and abs(v / wl.bytes_per_call - 1) < 0.01
    assert bench.ncu_traffic(wl, "staged") is None
    assert bench.ncu_traffic(inputs.WORKLOADS["embed_bf16_8192x1024"], "cta_per_row") is None


def test_nvml_summary_names_the_reason_bits_inside_the_window():
    p = bench.NvmlPoller(None)          # no NVML here: a poller that reports nothing
    assert p.summary(0.0, 1e12) is None
    p.lib, p.max_mhz = object(), 2070   # stand-ins: summary() only reads the samples
    p.samples = [(1.0, 1000, 0x8), (2.0, 2070, 0x0), (2.5, 2055, 0x4 | 0x20), (9.0, 900, 0x40)]
    c = p.summary(1.5, 3.0)
    assert c["samples"] == 2 and c["sm_mhz"] == 2062.5 and c["sm_mhz_min"] == 2055
    assert c["reasons"] == ["sw_power_cap", "sw_thermal_slowdown"] and c["sm_max_mhz"] == 2070
    assert p.summary(3.0, 4.0) is None
