"""The benchmark's work accounting and clock parsing, on the CPU.

The roofline numbers bench.py reports are algorithmic work divided by
measured time; these tests pin the work side to closed forms of the 128K
workloads (tile-granular counting, as the paper counts executed slots) and
check the clock-sample parsing that decides whether a run is kept."""
import json
import os

import bench
from mass_adaptive_sparse_gb300 import synthetic


def test_prefill_work_closed_forms():
    cfg = synthetic.CONFIGS["prefill_128k"]
    u = bench.prefill_units(cfg)
    t = 131072 // 128
    assert u["legal_tiles"] == 8 * t * (t + 1) // 2 == 4_198_400
    assert u["tile_flops"] == 2 * 128 * 128 * 128
    legal = u["legal_tiles"]
    # dense: Q K^T and P V on every legal tile; the backward adds dP, dV, dK, dQ
    assert bench.fwd_flops(cfg, legal) == 4 * 128 ** 3 * legal
    assert bench.bwd_flops(cfg, legal) == 10 * 128 ** 3 * legal
    # nothing kept: score discovery only (§2.3: QK stays on every legal tile)
    assert bench.fwd_flops(cfg, 0) == bench.bwd_flops(cfg, 0) == 2 * 128 ** 3 * legal


def test_decode_bytes_closed_form():
    cfg = synthetic.CONFIGS["decode_128k"]
    tiles = 8 * 8 * (131072 // 128)
    tile = 128 * 128 * 2
    q_and_o = 8 * 32 * 128 * 2 * 2
    partials = 16 * 8 * 32 * (128 + 4) * 4 * 2          # written by the splits, read by the merge
    assert bench.decode_bytes(cfg, tiles) == 2 * tiles * tile + q_and_o + partials == 4_299_423_744
    assert bench.decode_bytes(cfg, 0) == tiles * tile + q_and_o + partials      # K only


def test_traffic_records_follow_their_sources():
    """A record counts only while its kernel's code is the one it was taken
    on: current records give their bytes, stale ones give None."""
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    for kernel, by_workload in rec.items():
        if kernel.startswith("_"):
            continue
        for workload, r in by_workload.items():
            src = os.path.join(bench.ROOT, "mass_adaptive_sparse_gb300", "csrc", r["source"])
            current = bench.code_sha1(open(src).read()) == r["code_sha1"]
            assert bench._traffic(kernel, workload) == (r["bytes_per_launch"] if current else None)
    assert bench._traffic("no_such_kernel", "prefill_128k") is None


def test_code_hash_ignores_comments_only():
    """Comments, trailing blanks and empty lines do not change the code hash;
    any change to the code does."""
    code = "int f(int x) {\n  return x + 1;  // one more\n}\n"
    same = "/* a header\n   comment */\nint f(int x) {   \n\n  return x + 1;\n}  // end\n"
    other = "int f(int x) {\n  return x + 2;  // one more\n}\n"
    assert bench.code_sha1(code) == bench.code_sha1(same)
    assert bench.code_sha1(code) != bench.code_sha1(other)


class _Done:
    def terminate(self):
        pass

    def wait(self):
        pass


def test_clock_samples(tmp_path):
    s = bench.ClockSampler("GPU-abc")
    s.path = str(tmp_path / "clocks.csv")
    rows = ["0, GPU-abc, 2070, 2070, 900, 0x0, Not Active, Not Active, Not Active, Active",
            "0, GPU-abc, 2070, 2070, 950, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, GPU-abc, 1965, 2070, 990, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, GPU-abc, 345, 2070, 120, 0x0, Not Active, Not Active, Not Active, Not Active",   # idle: dropped
            "1, GPU-other, 1000, 2070, 500, 0x0, Active, Not Active, Not Active, Not Active"]   # other GPU
    open(s.path, "w").write("\n".join(rows) + "\n")
    s.proc = _Done()
    c = s.stop()
    assert c["sm_mhz"] == 2070 and c["sm_max_mhz"] == 2070 and c["samples"] == 4
    assert c["reasons"] == ["sw_power_cap"]
