"""Host-side bookkeeping of bench.py (no GPU): the DRAM traffic lookup, which must
only report a captured figure while the kernel's sources are unchanged, and the
algorithmic byte counts the HBM rooflines divide by."""

import dataclasses
import os

import bench
import workloads


def test_traffic_lookup_follows_the_source_hash(tmp_path, monkeypatch):
    cur = bench.source_hash(*bench.KERNEL_SOURCES["nvfp4_requant"])
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "dram_traffic.txt").write_text(
        "# comment line nvfp4_requant flux_up x 1\n"
        f"nvfp4_requant flux_up {cur} 12345\n"
        "nvfp4_act_quant flux_up 0000000000000000 999\n")
    hashes = {k: bench.source_hash(*v) for k, v in bench.KERNEL_SOURCES.items()}
    by_files = {tuple(v): hashes[k] for k, v in bench.KERNEL_SOURCES.items()}
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda *rel: by_files[tuple(rel)])
    assert bench.dram_traffic("nvfp4_requant", "flux_up") == 12345.0
    assert bench.dram_traffic("nvfp4_act_quant", "flux_up") is None  # stale capture
    assert bench.dram_traffic("nvfp4_gemm", "flux_up") is None       # none captured
    assert bench.dram_traffic("nvfp4_requant", "sana") is None        # other workload


def test_source_hash_changes_with_the_sources(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("x")
    h1 = bench.source_hash(str(a))
    a.write_text("y")
    assert bench.source_hash(str(a)) != h1


def test_algorithmic_bytes_flux():
    cfg = workloads.LINEARS["flux_up"]
    ab = bench.algorithmic_bytes(cfg)
    M, K, N = cfg.M, cfg.K, cfg.N
    sf_w = (N + 127) // 128 * 128 * (K // 16)
    sf_a = (M + 127) // 128 * 128 * (K // 16)
    # W once (bf16), A and B (fp32, rank 32), codes, scales, s_t
    assert ab["nvfp4_requant"] == 2 * N * K + 4 * 32 * K + 4 * N * 32 + N * K // 2 + sf_w + 4
    # X once (bf16), codes, scales, one fp32 per row
    assert ab["nvfp4_act_quant"] == 2 * M * K + M * K // 2 + sf_a + 4 * M
    assert ab["act_quant_per_tensor"] == ab["nvfp4_act_quant"] - 4 * M + 4
    # 2.5625 bytes per element of W (N is a multiple of 128), plus the LoRA factors and s_t
    assert ab["nvfp4_requant"] - (4 * 32 * K + 4 * N * 32 + 4) == 2.5625 * N * K


def test_algorithmic_bytes_scale_with_rows():
    cfg = workloads.LINEARS["flux_up"]
    small = dataclasses.replace(cfg, M=8192)
    a, b = bench.algorithmic_bytes(cfg), bench.algorithmic_bytes(small)
    assert a["nvfp4_requant"] == b["nvfp4_requant"]  # independent of the activations
    assert a["nvfp4_act_quant"] > 4 * b["nvfp4_act_quant"]


def test_clock_summary_from_nvidia_smi_lines():
    lines = [
        "0, 2070, 2070, 950.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1980, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1200.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    got = bench.ClockSampler.summarize(lines)
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "samples": 3, "reasons": ["sw_power_cap"]}
    hot = lines[:1] + ["0, 1500, 2070, 900, 0x8, Active, Not Active, Active, Not Active"]
    reasons = bench.ClockSampler.summarize(hot)["reasons"]
    assert reasons == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    assert bench.ClockSampler.summarize([]) is None


def test_clock_samples_are_taken_from_the_timed_region():
    """Lines stamped with their arrival time: the region keeps those that arrived from
    its start to one interval after its end; a region shorter than the interval keeps
    the first sample after its start; no bracket keeps everything."""
    stamped = [(0.90, "a"), (1.00, "b"), (1.02, "c"), (1.04, "d"), (1.07, "e"), (1.50, "f")]
    pick = bench.ClockSampler.in_region
    assert pick(stamped, 1.00, 1.03, 0.02) == ["b", "c", "d"]
    assert pick(stamped, 1.045, 1.046, 0.02) == ["e"]   # nothing inside: the next sample
    assert pick(stamped, 1.60, 1.70, 0.02) == []        # nothing after the start
    assert pick(stamped, None, None, 0.02) == ["a", "b", "c", "d", "e", "f"]


def test_clock_sampler_runs_a_fake_nvidia_smi(tmp_path, monkeypatch):
    """The sampler end to end against a stand-in nvidia-smi that prints a CSV line every
    20 ms: start() returns once sampling runs, the bracket keeps the samples of the
    region, stop() ends the child."""
    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!/bin/sh\n"
                    "i=0\n"
                    "while [ $i -lt 250 ]; do\n"
                    "  echo '0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active'\n"
                    "  i=$((i+1)); sleep 0.02\n"
                    "done\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}:{os.environ.get('PATH', '')}")
    import time
    cs = bench.ClockSampler(0)
    cs.start()
    assert cs.lines, "start() returns once the first sample is in"
    cs.begin()
    time.sleep(0.2)
    cs.end()
    got = cs.stop()
    assert cs.proc.poll() is not None
    assert got["sm_mhz"] == 2070.0 and got["reasons"] == []
    assert 2 <= got["samples"] < len(cs.lines)


def test_clock_sampler_falls_back_to_the_longer_interval(tmp_path, monkeypatch):
    """A stand-in nvidia-smi that refuses -lms 20 (exits at once, no output) and samples
    at -lms 200: the sampler retries with 200 ms and still summarises."""
    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!/bin/sh\n"
                    "for a in \"$@\"; do [ \"$a\" = 20 ] && exit 1; done\n"
                    "i=0\n"
                    "while [ $i -lt 50 ]; do\n"
                    "  echo '0, 1980, 2070, 1000.0, 0x4, Not Active, Not Active, Not Active, Active'\n"
                    "  i=$((i+1)); sleep 0.2\n"
                    "done\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}:{os.environ.get('PATH', '')}")
    cs = bench.ClockSampler(0)
    cs.start()
    assert cs.interval_ms == 200 and cs.lines
    cs.begin()
    cs.end()
    got = cs.stop()
    assert got == {"sm_mhz": 1980.0, "sm_max_mhz": 2070.0, "samples": 1, "reasons": ["sw_power_cap"]}


def test_report_line_has_the_contract_keys():
    """The JSON line bench.py prints, from made-up timings (no GPU): every key of the
    contract is there and the derived numbers follow from the timings."""
    import argparse
    cfg = workloads.LINEARS["flux_up"]
    rcfg = workloads.REWARDS[bench.REWARD_CFG]
    args = argparse.Namespace(steps=10, warmup=3, rows=None, no_e2e=False, no_cpu_baseline=True,
                              config="flux_up")
    per = {"nvfp4_requant": 0.1, "nvfp4_act_quant": 0.08, "nvfp4_gemm": 0.5, "bf16_gemm": 1.5,
           "select_contrastive": 0.016}
    clk = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "samples": 5, "reasons": []}
    out = bench.report(args, cfg, rcfg, None, per, 22.0, 50.0, 304, 906, 0, clk, 1, 0,
                       {"nvfp4_requant": 3, "nvfp4_act_quant": 1, "nvfp4_gemm": 1, "bf16_gemm": 1,
                        "select_contrastive": 2}, 0.12, {},
                       {"act_quant_prescaled": 0.05, "nvfp4_gemm_rowamax": 0.51})
    for k in ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches",
              "clocks"]:
        assert k in out, k
    flops = 2.0 * cfg.M * cfg.N * cfg.K
    assert abs(out["value"] - flops / 0.5e-3 / 1e12) < 0.01
    assert out["ms_per_step"] == 2.2 and out["gpu_launches"] == 80
    assert out["config"]["workload"].startswith("FLUX.1-shaped MLP up-projection")
    assert set(out["roofline"]) == {"bound", "achieved", "peak", "unit", "frac", "traffic"}
    assert abs(out["roofline"]["frac"] - out["roofline"]["achieved"] / out["roofline"]["peak"]) < 1e-3
    assert out["e2e"]["h2d_bytes_per_step"] == 304 and out["e2e"]["ms_per_step"] == 5.0
    assert out["variants"]["act_quant_per_tensor"]["ms"] == 0.12
    ab = bench.algorithmic_bytes(cfg)["act_quant_prescaled"]
    assert abs(out["variants"]["act_quant_prescaled"]["gbs"] - ab / 0.05e-3 / 1e9) < 0.1
    small = argparse.Namespace(**{**vars(args), "rows": 8192})
    out2 = bench.report(small, cfg, rcfg, None, per, 22.0, 50.0, 304, 906, 0, clk, 1, 0, {}, 0.12, {},
                        {"act_quant_prescaled": 0.05, "nvfp4_gemm_rowamax": 0.51})
    assert all(r["traffic"] is None for r in out2["rooflines"].values())  # no capture of that workload


def test_parse_args_defaults_and_config():
    a = bench.parse_args([])
    assert (a.gpus, a.config, a.impl) == (1, "flux_up", "ours") and a.warmup >= 3
    assert bench.parse_args(["--config", "sd35_qkv", "--warmup", "1"]).warmup == 3


def test_replica_command_is_a_local_torchrun():
    cmd = bench.replica_command(4, ["--gpus", "4", "--steps", "5"])
    assert cmd[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"]
    assert "--nproc-per-node=4" in cmd and cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[-3:] == ["--gpus", "4", "--steps", "5"][-3:] and cmd[-5].endswith("bench.py")
