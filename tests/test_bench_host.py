"""Host-side logic of bench.py, run without a GPU: the algorithmic work per token-head that
the roofline divides by, the choice of the bound, the summary of the clock samples that
decides whether a run is rejected, the rule that drops a DRAM-traffic capture once the
kernel's source has changed, and the JSON line of the reference (oracle) arm.
"""
import json
import os

import pytest

import bench

D = DV = 64
C = 256
TOKENS = 2 * 16 * 8192            # token-heads per launch at B=2, H=16, T=8192
PK = {"hbm_gbs": 6507.5, "bf16_tflops": 1739.7, "bf16_tflops_sustained": 1353.7, "sm_max_mhz": 2032.0,
      "source": "measured"}


def test_chunk_state_bytes_per_token_head():
    # one chunk state: two fp16 planes of the d^2 x dv state (hi and residual) and the fp32
    # normaliser column of d^2 entries, written once per chunk of C = 256 tokens
    per_chunk = 2 * 2 * (64 * 64) * 64 + 4 * (64 * 64)
    assert per_chunk == 1_064_960
    assert per_chunk / 256 == 4160
    # the forward walk also reads each token's k and v rows (bf16, 64 + 64 values)
    assert bench.packed_rows(D) == 2560   # 10 of the 16 blocks of 16 x 16
    assert bench.kernel_bytes("tc_state_scan_fwd", D, DV, C, 1) == 2624 + 256   # packed planes + z
    assert bench.kernel_bytes("tc_state_scan_bwd", D, DV, C, 1) == 2624 + 256 + 8   # packed gradient state


def test_algorithmic_units_per_token_head():
    # flops: the d^2 x (dv+1) contraction of one token is 2 * 4096 * 65 = 532,480; the walks add
    # one state update per chunk (2 * 4096 * 65 / 256 = 2,080 per token); a readout adds the
    # causal pairs of its chunk, (C+1)/2 per token on average, each a 64-dot and a 64-axpy
    assert bench.kernel_flops("tc_state_scan_fwd", D, DV, C, 1) == 2 * 2560 * 65 + 2 * 2560 * 65 / 256
    assert bench.kernel_flops("tc_state_scan_bwd", D, DV, C, 1) == 2 * 2560 * 65 + 2 * 2560 * 65 / 256
    assert bench.kernel_flops("tc_chunk_out", D, DV, C, 1) == 2 * 2560 * 65 + 257 * 128
    assert bench.kernel_flops("tc_bwd_dq", D, DV, C, 1) == 2 * 2560 * 65 + 257 * 128
    assert bench.kernel_flops("tc_bwd_dkdv", D, DV, C, 1) == 532_480 + 2 * 64 * 64 + 257 * 192
    # bytes: the chunk state (4,160) plus the token rows each kernel must move
    assert bench.kernel_bytes("tc_chunk_out", D, DV, C, 1) == 2624 + 2 * 192 + 4 * 65       # q k v in; o, Z out
    assert bench.kernel_bytes("tc_bwd_dq", D, DV, C, 1) == 2624 + 2 * 256 + 2 * 64 + 4 * 2   # q k v dO in; dq (bf16), two scalars
    assert bench.kernel_bytes("tc_bwd_dkdv", D, DV, C, 1) == 2624 + 2 * 256 + 2 * 128 + 4 * 4
    # decode: the fp32 state read and written once, full (d^2 rows) or symmetric-packed (d(d+1)/2)
    assert bench.decode_bytes_per_head(64, 64) - bench.decode_bytes_per_head(64, 64, packed=True) == \
        2 * (4096 - 2080) * (64 + 1) * 4
    assert bench.kernel_flops("not_a_kernel", D, DV, C, 1) is None
    assert bench.kernel_bytes("not_a_kernel", D, DV, C, 1) is None


def test_roofline_picks_the_slower_bound():
    # the forward walk: 1.16 GB at 6.5 TB/s (0.178 ms) outlasts 140 GFLOP at 1.35 PFLOP/s (0.104 ms)
    kf = bench.kernel_flops("tc_state_scan_fwd", D, DV, C, TOKENS)
    kb = bench.kernel_bytes("tc_state_scan_fwd", D, DV, C, TOKENS)
    r = bench.roofline("tc_state_scan_fwd", kf, kb, 0.616, PK, tc=True)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == PK["hbm_gbs"]
    assert r["achieved"] == pytest.approx(kb / 0.616e-3 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / PK["hbm_gbs"])
    assert r["tensor_frac"] == pytest.approx(kf / 0.616e-3 / 1e12 / PK["bf16_tflops_sustained"])
    # dk/dv (one contraction of the full gradient state per token, the key term taken from the
    # same product, the packed state read) is HBM-bound against either tensor figure: 0.89 GB at
    # 6.5 TB/s (0.14 ms) against 155 GFLOP (0.11 ms sustained, 0.09 ms burst)
    kf = bench.kernel_flops("tc_bwd_dkdv", D, DV, C, TOKENS)
    kb = bench.kernel_bytes("tc_bwd_dkdv", D, DV, C, TOKENS)
    for key in ("bf16_tflops_sustained", "bf16_tflops"):
        r = bench.roofline("tc_bwd_dkdv", kf, kb, 0.553, PK, tc=True, peak_key=key)
        assert r["bound"] == "hbm" and r["frac"] == pytest.approx(kb / 0.553e-3 / 1e9 / PK["hbm_gbs"])
        assert r["tensor_frac"] == pytest.approx(kf / 0.553e-3 / 1e12 / PK[key])
    # the tensor figure follows the length of the timed region
    assert bench.tensor_peak_key(53.0) == "bf16_tflops" and bench.tensor_peak_key(1200.0) == "bf16_tflops_sustained"
    # the same work with twice the bandwidth is tensor-bound, with half of it HBM-bound
    assert bench.roofline("k", kf, kb, 1.0, dict(PK, hbm_gbs=2 * PK["hbm_gbs"]), tc=True)["bound"] == "tensor"
    assert bench.roofline("k", kf, kb, 1.0, dict(PK, hbm_gbs=PK["hbm_gbs"] / 2), tc=True)["bound"] == "hbm"


def test_roofline_of_cuda_core_kernels_and_uncounted_work():
    r = bench.roofline("chunk_out", 1e12, None, 10.0, PK, tc=False)
    peak = 148 * 128 * 2 * 2032e6 / 1e12          # fp32 FMA rate of 148 SMs at 2032 MHz
    assert r["bound"] == "alu" and r["peak"] == pytest.approx(peak)
    assert r["frac"] == pytest.approx(1e12 / 10e-3 / 1e12 / peak)
    assert bench.roofline("x", None, None, 1.0, PK, tc=True) is None


def test_clock_summary_flags_throttling():
    lines = [
        "2032, 2032, 850.1, Not Active, Not Active, Not Active, Not Active\n",
        "1980, 2032, 1090.0, Not Active, Not Active, Not Active, Active\n",
        "garbage line\n",
        "[N/A], 2032, 1.0, Not Active, Not Active, Not Active, Not Active\n",
        "2010, 2032, 900.0, Not Active, Active, Not Active, Not Active\n",
    ]
    s = bench.parse_clocks(lines)
    assert s["samples"] == 3
    assert s["sm_mhz"] == 2010 and s["sm_max_mhz"] == 2032
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert bench.parse_clocks(["no samples\n"]) is None
    clean = bench.parse_clocks(["2032, 2032, 800, Not Active, Not Active, Not Active, Not Active\n"])
    assert clean["reasons"] == []


def test_traffic_capture_is_dropped_when_the_kernel_changes(tmp_path, monkeypatch):
    csrc = tmp_path / "ssm_sequence_mixer_chunked_b300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = csrc / "k.cu"
    src.write_text("// version 1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"k": {"file": "k.cu", "file_sha": bench.file_sha("k.cu"), "dram_bytes_per_unit": 2.5,
                 "unit": "one token-head"}}
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(rec))
    assert bench.ncu_traffic("k", 1000) == 2500.0
    assert bench.ncu_traffic("other", 1000) is None
    src.write_text("// version 2\n")
    assert bench.ncu_traffic("k", 1000) is None


def test_committed_traffic_records_name_existing_sources():
    with open(os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")) as f:
        recs = json.load(f)
    for name, rec in recs.items():
        assert os.path.exists(os.path.join(bench.ROOT, "ssm_sequence_mixer_chunked_b300", "csrc", rec["file"])), name
        assert rec["dram_bytes_per_unit"] > 0 and rec["unit"]


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` times the fp64 oracle on the CPU (one head of the bench
    workload per step) and prints the same JSON line as the CUDA arm, marked as reference."""
    import subprocess
    import sys
    out = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True, timeout=600,
                         cwd=bench.ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True and line["value"] > 0
    assert line["warmup"] >= 3 and line["steps"] == 1 and line["n_gpus"] == 1
    assert line["config"]["B"] == 2 and line["config"]["T"] == 8192 and line["config"]["d"] == 64
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
