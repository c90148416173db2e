"""Host-side logic of bench.py: the algorithmic byte count of a frame, the clock-sample
summary and the rule that reports a profile's DRAM traffic only for the kernel source it
was captured on.  No GPU is needed."""
import os

import pytest

import bench
from rq_transformer_frame_gb300 import configs


def test_frame_bytes_of_the_moshi_shape():
    # matrices of the Moshi-7B shape in bf16 (dim 4096, 32 layers, hidden 11264, text card
    # 32000; depformer dim 1024, 6 layers, hidden 2816; 2048 audio codes):
    #   temporal 32 x (qkv 12288x4096 + out 4096x4096 + gate_in 22528x4096 + gate_out
    #   4096x11264) x 2 B = 13 153 337 344; head 262 144 000; depformer 8 x 6 x (...) x 2 B
    #   = 1 233 125 376; inputs 67 108 864; heads 33 554 432
    c = configs.MOSHI7B
    fb = bench.frame_bytes(c, [0])
    assert fb["temporal"] == 13_153_337_344
    assert fb["weights"] == 13_153_337_344 + 262_144_000 + 1_233_125_376 + 67_108_864 + 33_554_432
    # one position of K and V per layer read (bf16) and one row of each written
    row = 2 * c.dim * 2 * c.layers
    assert fb["kv"] == row + row
    # the window stops growing at the context
    assert bench.frame_bytes(c, [10 ** 6])["kv"] == c.context * row + row
    # embedding rows: 17 temporal tables and 8 depformer tables per session
    emb = 17 * c.dim * 2 + 8 * c.ddim * 2
    assert fb["total"] == fb["weights"] + fb["kv"] + emb


def test_frame_bytes_scale_with_sessions_not_weights():
    c = configs.MOSHI7B.with_(batch=4)
    one = bench.frame_bytes(configs.MOSHI7B, [100])
    four = bench.frame_bytes(c, [100] * 4)
    assert four["weights"] == one["weights"]
    assert four["kv"] == 4 * one["kv"]


def _summary_of(lines):
    s = bench.ClockSampler(0)  # not entered: no nvidia-smi process
    s.f.write("\n".join(lines) + "\n")
    return s.summary()


def test_clock_summary_median_max_and_reasons():
    rows = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1200.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    out = _summary_of(rows)
    assert out["samples"] == 3
    assert out["sm_mhz"] == 2070.0
    assert out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]


def test_clock_summary_reports_thermal_slowdown():
    rows = ["0, 1500, 2070, 1000, 0x40, Not Active, Active, Not Active, Not Active"]
    out = _summary_of(rows)
    assert out["reasons"] == ["hw_thermal_slowdown"]


def test_clock_summary_of_no_samples():
    out = _summary_of([])
    assert out == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_profiled_traffic_needs_the_current_source(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "rq_transformer_frame_gb300" / "csrc"
    src.mkdir(parents=True)
    for n in bench.KERNEL_SOURCES["attn"]:
        (src / n).write_text("// " + n + "\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    h = bench.source_hash("attn")
    (prof / "p.md").write_text("traffic_bytes_per_launch: 2.0e8\n"
                               "algorithmic_bytes_per_launch: 1.0e8\n"
                               "source_hash: %s\n" % h)
    assert bench.profiled_traffic("p.md", "attn") == pytest.approx(2.0e8)
    # a capture of a smaller case scales with the algorithmic bytes of the full launch
    assert bench.profiled_traffic("p.md", "attn", 3.0e8) == pytest.approx(6.0e8)
    # any change to a source the kernel is built from voids the figure
    (src / "attn.cu").write_text("// changed\n")
    assert bench.profiled_traffic("p.md", "attn") is None
    assert bench.profiled_traffic("missing.md", "attn") is None


def test_committed_profiles_name_a_kernel_source_hash():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for name in ("frame_persistent_moshi7b.md", "gemv_moshi7b_b1.md",
                 "tc_gemm_moshi7b_b16.md", "attn_moshi7b_b64.md"):
        txt = open(os.path.join(root, "profiles", name)).read()
        assert "source_hash:" in txt and "traffic_bytes_per_launch:" in txt, name
        assert "--clock-control none" in txt, name
