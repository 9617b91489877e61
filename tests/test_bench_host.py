"""Host-side checks of bench.py's bookkeeping (no GPU): the roofline bound it
reports, the issued-MMA factor of each activation mode, and that a recorded
ncu traffic figure is used only for the sources it was taken on."""
import json
import os

import pytest

import bench

PEAKS = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0}


@pytest.fixture(autouse=True)
def fixed_peaks(monkeypatch):
    monkeypatch.setattr(bench, "load_peaks", lambda: (dict(PEAKS), "measured"))


def alg(bytes_, flops):
    return dict(active=128, ffn_bytes=bytes_, layer_bytes=bytes_, ffn_flops=flops, layer_flops=flops)


def test_decode_is_hbm_bound():
    roof, layer = bench.roofline(alg(1.6e9, 1.0e10), 0.32, 0.40, "decode")
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert roof["achieved"] == pytest.approx(1.6e9 / 0.32e-3 / 1e9)
    assert roof["frac"] == pytest.approx(roof["achieved"] / 6000.0)
    assert layer == pytest.approx((1.6e9 / 6000e9) / 0.40e-3)


def test_prefill_reports_the_tensor_bound_and_issued_flops():
    roof, _ = bench.roofline(alg(2.6e9, 1.44e12), 1.3, 1.6, "prefill", "e4m3")
    assert roof["bound"] == "tensor" and roof["peak"] == pytest.approx(4000.0)     # FP8 = 2 x bf16
    assert roof["achieved"] == pytest.approx(1.44e12 / 1.3e-3 / 1e12)
    assert roof["issued"]["tflops"] == pytest.approx(2 * roof["achieved"])           # two E4M3 terms
    one, _ = bench.roofline(alg(2.6e9, 1.44e12), 0.9, 1.1, "prefill", "e4m3", False, 1)
    assert one["issued"]["tflops"] == pytest.approx(one["achieved"])                 # one term
    fp4, _ = bench.roofline(alg(2.6e9, 3.7e12), 4.9, 5.2, "100b_prefill", "nvfp4")
    assert fp4["peak"] == pytest.approx(8000.0)                                      # FP4 = 4 x bf16
    assert fp4["issued"]["tflops"] == pytest.approx(4 * fp4["achieved"])             # four NVFP4 terms
    assert fp4["issued"]["peak"] == pytest.approx(8000.0)
    w4a4, _ = bench.roofline(alg(2.6e9, 3.7e12), 2.0, 2.2, "100b_prefill", "nvfp4", False, 1)
    assert w4a4["issued"]["tflops"] == pytest.approx(w4a4["achieved"])               # one term
    f16, _ = bench.roofline(alg(2.6e9, 3.7e12), 4.9, 5.2, "100b_prefill", "nvfp4", nvfp4_f16=True)
    assert f16["issued"]["peak"] == pytest.approx(2000.0)                            # f16 MMAs


def test_traffic_only_for_matching_sources(tmp_path, monkeypatch):
    kernel = "moe_expert_ffn (grouped SwiGLU GEMMs + shared expert)"
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda files=None: "abc")
    rec = {"decode": {"kernel": kernel, "source_hash": "abc", "dram_bytes_per_launch": 123}}
    (prof / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("decode", kernel) == 123
    assert bench.recorded_traffic("prefill", kernel) is None
    rec["decode"]["source_hash"] = "other"
    (prof / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("decode", kernel) is None


def test_source_hash_covers_the_kernel_sources():
    h = bench.source_hash()
    assert len(h) == 16 and int(h, 16) >= 0
    csrc = os.path.join(bench.ROOT, "top_routed_expert_gb300", "csrc")
    assert any(fn.endswith(".cu") for fn in os.listdir(csrc))


def test_single_rank_aggregation_is_the_identity():
    assert bench.max_over_ranks(1.25, 1, "cpu") == 1.25
    assert bench.job_value(1, 64, 0.5) == pytest.approx(64 / 0.5e-3)
    assert bench.job_value(4, 64, 0.5) == pytest.approx(4 * 64 / 0.5e-3)


def test_skew_reports_the_slower_bound():
    # the skewed batch is not forced onto the tensor bound: HBM when bytes dominate
    roof, _ = bench.roofline(alg(1.73e9, 0.73e12), 0.4, 0.5, "skew", "e4m3")
    assert roof["bound"] == "hbm"
    roof, _ = bench.roofline(alg(0.5e9, 2.0e12), 0.6, 0.7, "skew", "e4m3")
    assert roof["bound"] == "tensor"


def test_nvfp4_path_choice_follows_the_library():
    from types import SimpleNamespace as NS
    dec = NS(T=64, k=8, E=128)
    pre = NS(T=8192, k=8, E=128)
    assert not bench.nvfp4_on_f16_path(dec, 0) and bench.nvfp4_on_f16_path(pre, 0)
    assert bench.nvfp4_on_f16_path(dec, 0x20) and not bench.nvfp4_on_f16_path(pre, 0x10)


def test_traffic_records_are_per_variant():
    """A flag that changes the expert-stage kernels gets no traffic record
    recorded for the default path of the same workload."""
    import bench
    from top_routed_expert_gb300 import abi
    assert bench.traffic_key("prefill", 0) == "prefill"
    assert bench.traffic_key("prefill", abi.MOE_FLAG_ACT_E4M3) == "prefill+MOE_FLAG_ACT_E4M3"
    assert bench.traffic_key("100b_decode", abi.MOE_FLAG_NVFP4_F16 | abi.MOE_FLAG_NO_OVERLAP) == \
        "100b_decode+MOE_FLAG_NVFP4_F16"
    k = "moe_expert_ffn (grouped SwiGLU GEMMs + shared expert)"
    assert bench.recorded_traffic(bench.traffic_key("100b_prefill", abi.MOE_FLAG_ACT_NVFP4), k) is None


def test_traffic_records_name_their_sources():
    """Each DRAM-traffic record lists the kernel sources it was measured on;
    a change to one of them (a different hash) retires the record."""
    import bench
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    csrc = os.path.join(bench.ROOT, "top_routed_expert_gb300", "csrc")
    for name, r in rec.items():
        assert r["sources"], name
        for fn in r["sources"]:
            assert os.path.exists(os.path.join(csrc, fn)), (name, fn)
        assert len(r["source_hash"]) == 16 and int(r["source_hash"], 16) >= 0
        assert r["dram_bytes_per_launch"] > 0


def test_traffic_record_retired_when_its_sources_change(monkeypatch):
    import bench
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    r = rec["decode"]
    monkeypatch.setattr(bench, "source_hash", lambda files=None: r["source_hash"])
    assert bench.recorded_traffic("decode", r["kernel"]) == r["dram_bytes_per_launch"]
    monkeypatch.setattr(bench, "source_hash", lambda files=None: "0" * 16)
    assert bench.recorded_traffic("decode", r["kernel"]) is None
