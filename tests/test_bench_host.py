"""Host-side logic of bench.py (no GPU): the list of workloads a run times,
the recorded-traffic lookup, the source hash it is keyed by, and the
clock-corrected utilisation arithmetic."""
import os

import pytest

import bench
from attention_forward_flashattention_gb300 import inputs as I


def test_other_workloads_cover_every_config_once():
    names = bench.other_workload_names(bench.DEFAULT_WORKLOAD, "forward")
    base = [bench._base_name(n) for n in names if ":" not in n]
    assert bench.DEFAULT_WORKLOAD not in base
    assert len(base) == len(set(base))
    assert set(base) | {bench.DEFAULT_WORKLOAD} == set(I.WORKLOAD_ORDER) | set(I.FP8_WORKLOADS)
    # the other kernel of every 16-bit head-dimension-128 workload, the headline's included
    d128 = [n for n in I.WORKLOAD_ORDER if I.WORKLOADS[n].d == 128]
    other = [n for n in names if ":" in n]
    assert sorted(bench._base_name(n) for n in other) == sorted(d128)


@pytest.mark.parametrize("picks", [lambda n: True, lambda n: False,
                                   lambda n: I.WORKLOADS[n].N >= 16384])
def test_other_kernel_prefix_follows_the_choice(picks):
    names = bench.other_workload_names(bench.DEFAULT_WORKLOAD, "forward", picks_pair=picks)
    for n in names:
        if ":" in n:
            b = bench._base_name(n)
            # fa_fwd picks the pair there -> the one-CTA kernel is the other one
            assert n.startswith(bench.ONE_PREFIX if picks(b) else bench.PAIR_PREFIX)


def test_backward_pass_times_no_kernel_variants():
    names = bench.other_workload_names(bench.DEFAULT_WORKLOAD, "backward")
    assert all(":" not in n for n in names)
    assert not any(n in I.FP8_WORKLOADS for n in names)


def test_source_hash_ignores_comments_and_blank_lines():
    text = "int a;  // one\n\n// two\nint b;\n"
    assert bench._code_only(text) == bench._code_only("int a;\nint b;  // other words\n")
    assert bench._code_only(text) != bench._code_only("int a;\nint c;\n")
    hashes = {k: bench.kernel_source_sha256(k) for k in bench.KERNEL_SOURCES}
    assert len(set(hashes.values())) == 3 and all(len(h) == 64 for h in hashes.values())


def test_recorded_traffic_lookup(tmp_path, monkeypatch):
    one, pair = bench.kernel_source_sha256("one_cta"), bench.kernel_source_sha256("pair")
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "fa_fwd_traffic.txt").write_text(
        "# comment: workload: ignored\n"
        f"kernel_source_sha256: {'0' * 64}\n"            # stale block: never matched
        "workload: mha_b4_h16_n4096_d128_fp16\ndram_bytes_per_launch: 1\n"
        f"kernel_source_sha256: {one}\n"
        "workload: mha_b4_h16_n4096_d128_fp16\ndram_bytes_per_launch: 245000000\n"
        f"kernel_source_sha256: {pair}\n"
        "workload: cta_pair:mha_b4_h16_n4096_d128_fp16\ndram_bytes_per_launch: 246000000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("mha_b4_h16_n4096_d128_fp16") == 245000000
    assert bench.recorded_traffic("cta_pair:mha_b4_h16_n4096_d128_fp16") == 246000000
    assert bench.recorded_traffic("causal_b4_h16_n4096_d128_bf16") is None
    assert bench.recorded_traffic("mha_b4_h16_n4096_d128_e4m3") is None   # no e4m3 block
    monkeypatch.setattr(bench, "ROOT", str(tmp_path / "nowhere"))
    assert bench.recorded_traffic("mha_b4_h16_n4096_d128_fp16") is None


def test_committed_traffic_record_parses():
    path = os.path.join(os.path.dirname(bench.__file__), "profiles", "fa_fwd_traffic.txt")
    lines = [ln for ln in open(path).read().splitlines() if ln and not ln.startswith("#")]
    keys = [ln.split(":", 1)[0] for ln in lines]
    assert set(keys) <= {"kernel_source_sha256", "workload", "dram_bytes_per_launch"}
    assert keys.count("workload") == keys.count("dram_bytes_per_launch") > 0


def test_clock_corrected_fraction():
    # 1 PFLOP/s on 152 SMs at 2 GHz, 8192 FLOP per clock and SM (16-bit), 16384 (e4m3)
    f16 = bench.clock_corrected_frac(1000.0, "fp16", 152, 2000.0)
    assert f16 == pytest.approx(1e15 / (152 * 8192 * 2e9))
    assert bench.clock_corrected_frac(1000.0, "e4m3", 152, 2000.0) == pytest.approx(f16 / 2)
    assert bench.clock_corrected_frac(1000.0, "bf16", 152, None) is None


def test_hbm_figure():
    # C1: Q, K, V, O of B1 H2 N256 d64 fp16 (4 x 65536 bytes) and the fp32 LSE (2048 bytes)
    plan = bench.Plan(h2d=3 * 65536, d2h=65536 + 2048)
    f = bench.hbm_figure(plan, 0.0106, {"hbm_gbs": 6789.0})
    assert f["bytes"] == 264192
    assert f["gbs"] == pytest.approx(264192 / 10.6e-6 / 1e9)
    assert f["frac"] == pytest.approx(f["gbs"] / 6789.0) and f["peak_source"] == "measured copy"
    assert bench.hbm_figure(plan, 1.0, {})["peak_gbs"] == bench.FALLBACK_HBM_GBS
