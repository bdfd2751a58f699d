"""bench.py's bookkeeping on CPU, against figures worked out independently.

The algorithmic bytes of a step are checked against the per-config totals
computed by hand for the measurement plan (packed Q4_K at 144 B per 256
weights, fp32 X, Y at its dtype); the launch count against the tile and wave
arithmetic of the 7B shapes on a 152-SM part (a GEMM whose last wave of
tiles is split along k also launches the fixup).
"""
import pytest

import bench


def _mb(x):
    return x / 1e6


def test_step_footprint_stack_config():
    tokens, mats, out, _ = bench.WORKLOADS["stack"]
    w, x, y = bench.step_footprint(tokens, mats, out, 144)
    # 32 layers x 202,375,168 weights x 144/256; 2048 tokens x (6 x 4096 + 11008) x 4 B per layer;
    # 2048 x (4 x 4096 + 2 x 11008 + 4096) x 2 B per layer
    assert w == 32 * 202_375_168 * 144 / 256
    assert _mb(w) == pytest.approx(3642.8, abs=0.1)
    assert _mb(x) == pytest.approx(9328.1, abs=0.1)
    assert _mb(y) == pytest.approx(5570.0, abs=0.1)


def test_step_footprint_qproj_and_ffn_configs():
    w, x, y = bench.step_footprint(512, [(4096, 4096)], "f32", 144)
    assert (_mb(w), _mb(x), _mb(y)) == pytest.approx((9.437, 8.389, 8.389), abs=1e-3)
    w, x, y = bench.step_footprint(2048, [(11008, 4096), (11008, 4096), (4096, 11008)], "bf16", 144)
    assert (_mb(w), _mb(x), _mb(y)) == pytest.approx((76.09, 157.3, 107.0), abs=0.1)
    # Q6_K weights at 210 B per 256
    w6, _, _ = bench.step_footprint(2048, [(4096, 11008)], "bf16", 210)
    assert w6 == 4096 * 11008 * 210 / 256


@pytest.mark.parametrize("m,n,k,want", [
    (2048, 4096, 4096, 3),     # 512 tiles: 3 waves + 56, split 2 ways -> quantizer, GEMM, fixup
    (2048, 11008, 4096, 3),    # 1376 tiles: 9 waves + 8, split 8 ways (parts of two super-blocks)
    (2048, 4096, 11008, 3),    # 512 tiles, split 2 ways (43 super-blocks)
    (512, 4096, 4096, 2),      # 128 tiles: one partial wave that cannot split (152 // 128 = 1)
    (2432, 4096, 4096, 2),     # 19 x 32 = 608 tiles: exactly 4 waves, nothing left over
    (256, 1024, 1024, 3),      # 16 tiles, split min(152 // 16, 4) = 4 ways
    (256, 1024, 512, 2),       # two super-blocks: not split (the fixup would cost more than it saves)
    (256, 1024, 256, 2),       # one super-block: no split possible
])
def test_gemm_launches(m, n, k, want):
    assert bench.gemm_launches(m, n, k, 152) == want


def test_hbm_view_fraction():
    v = bench.hbm_view({"hbm_gbs": 6669.5}, "measured", 26.2e6, 0.0608, "x")
    assert v["achieved"] == pytest.approx(26.2e6 / 60.8e-6 / 1e9)
    assert v["frac"] == pytest.approx(v["achieved"] / 6669.5)


def test_copy_groups():
    g = bench.copy_groups(224, 7)            # the 7B stack: one layer per copy
    assert len(g) == 32 and all(len(x) == 7 for x in g)
    assert [i for x in g for i in x] == list(range(224))
    assert bench.copy_groups(8, 7) == [[i] for i in range(8)]       # too few layers: per projection
    assert bench.copy_groups(3, 7) == [[0], [1], [2]]
    g = bench.copy_groups(30, 7)             # a partial last group keeps every index once, in order
    assert [len(x) for x in g] == [7, 7, 7, 7, 2] and [i for x in g for i in x] == list(range(30))


def test_clock_record_parsing():
    fields = bench.ClockSampler.FIELDS.split(",")
    assert len(fields) == 8
    line = "{}, 2070, {}, 0x0000000000000000, Not Active, Not Active, Not Active, {}"
    out = "\n".join([line.format(2070, "350.10", "Not Active"), line.format(1980, "1390.00", "Active"),
                     line.format(2070, "371.2", "Not Active"), "[N/A], [N/A]"])
    rec = bench.ClockSampler.parse(out)
    assert rec["sm_mhz"] == 2070 and rec["sm_max_mhz"] == 2070 and rec["samples"] == 3
    assert rec["reasons"] == ["sw_power_cap"] and rec["power_w_max"] == 1390.0
    hot = "1500, 2070, 300.0, 0x8, Not Active, Active, Not Active, Not Active"
    assert bench.ClockSampler.parse(hot)["reasons"] == ["hw_thermal_slowdown"]
    assert bench.ClockSampler.parse("")["sm_mhz"] is None


def test_gemm_digest_follows_code_not_comments(tmp_path):
    """The GEMM traffic table is keyed by a hash of the GEMM's code: the files
    it includes count, comments and blank space do not."""
    from quantized_prefill_gemm_gb300 import build

    def write(main, header):
        (tmp_path / "gemm.cu").write_text('#include "h.cuh"\n' + main)
        (tmp_path / "h.cuh").write_text(header)
        return build.gemm_digest(str(tmp_path))

    base = write("int f() { return 1; }  // one\n", "/* a */ int g();\n")
    assert build._local_includes("gemm.cu", str(tmp_path)) == ["gemm.cu", "h.cuh"]
    assert write("int f() {\n  return 1;   // another comment\n}\n", "/* b\n c */ int g();\n") == base
    assert write("int f() { return 2; }\n", "int g();\n") != base
    assert write("int f() { return 1; }\n", "int g(int);\n") != base
