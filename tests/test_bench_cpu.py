"""Host-side arithmetic of bench.py (CPU only): the algorithmic bytes the roofline divides by,
the clock record parsed from nvidia-smi's CSV, the choice of the committed ncu traffic and the
peaks file.  No GPU and no kernel run here."""
import json
import types

import pytest

import bench


def _shape(B, H, V, dtype="bf16"):
    return types.SimpleNamespace(B=B, H=H, V=V, hidden_dtype=dtype)


def test_algorithmic_bytes_of_the_gbs8_step():
    # worked by hand: W is 2 * 2880 * 201088 bytes; the step adds the bf16 hidden rows
    # (8 * 2880 * 2), gamma (2880 * 4), four fp32 params and one int32 token per row (8 * 20)
    ab = bench.algorithmic_bytes(_shape(8, 2880, 201088), emit=False)
    assert ab["lm_head"] == 1_158_266_880
    assert ab["step"] == 1_158_266_880 + 46_080 + 11_520 + 160 == 1_158_324_640


def test_algorithmic_bytes_count_emitted_logits_and_wide_hidden():
    plain = bench.algorithmic_bytes(_shape(8, 2880, 201088), emit=False)
    emit = bench.algorithmic_bytes(_shape(8, 2880, 201088), emit=True)
    assert emit["lm_head"] - plain["lm_head"] == 4 * 8 * 201088  # fp32 logits written once
    assert emit["step"] - plain["step"] == 4 * 8 * 201088
    f32 = bench.algorithmic_bytes(_shape(8, 2880, 201088, "f32"), emit=False)
    assert f32["lm_head"] == plain["lm_head"]
    assert f32["step"] - plain["step"] == 8 * 2880 * 2  # 4-byte instead of 2-byte hidden elements


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def _sampler_with(tmp_path, lines):
    path = tmp_path / "clocks.csv"
    path.write_text("")
    s = bench.ClockSampler(0)
    s.proc = _FakeProc()
    s.path = str(path)
    s.out = open(path, "a")
    s.out.write("".join(line + "\n" for line in lines))
    s.out.flush()
    return s


def test_clock_record_is_the_median_under_sampling_and_the_active_reasons(tmp_path):
    lines = [
        "0, 2070, 2070, 950.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1995, 2070, 1201.4, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2040, 2070, 1100.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",  # skipped
        "garbage line",  # skipped
    ]
    rec = _sampler_with(tmp_path, lines).stop()
    assert rec == {"sm_mhz": 2040.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert not (tmp_path / "clocks.csv").exists()


def test_clock_record_names_thermal_and_hardware_slowdowns(tmp_path):
    lines = ["0, 1500, 2070, 1390.0, 0x48, Active, Not Active, Active, Not Active"]
    rec = _sampler_with(tmp_path, lines).stop()
    assert rec["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_record_without_samples_is_none(tmp_path):
    assert _sampler_with(tmp_path, []).stop() is None
    assert bench.ClockSampler(0).stop() is None  # never started


def test_committed_traffic_is_used_only_while_the_sources_match(monkeypatch):
    with open(bench.os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")) as f:
        committed = json.load(f)
    ent = committed["gptoss_g8"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel="lmhead_tail_kernel": ent["source_hash"])
    assert bench.ncu_traffic("gptoss_g8", False, ent["kernel"]) == ent["dram_bytes_per_launch"]
    assert bench.ncu_traffic("gptoss_g8", False, "some_other_kernel") is None
    emit_ent = committed.get("gptoss_g8_emit")
    if emit_ent is not None and emit_ent["source_hash"] == ent["source_hash"]:  # the emitting form's own capture
        assert bench.ncu_traffic("gptoss_g8", True, ent["kernel"]) == emit_ent["dram_bytes_per_launch"]
    else:
        assert bench.ncu_traffic("gptoss_g8", True, ent["kernel"]) is None
    assert bench.ncu_traffic("tiny", True, ent["kernel"]) is None  # no capture of that form
    assert bench.ncu_traffic("no_such_workload", False, ent["kernel"]) is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel="lmhead_tail_kernel": "0" * 16)
    assert bench.ncu_traffic("gptoss_g8", False, ent["kernel"]) is None


def test_committed_traffic_is_close_to_the_algorithmic_bytes():
    # a capture far above the algorithmic bytes would mean re-reads of W; below them, a wrong capture
    with open(bench.os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")) as f:
        committed = json.load(f)
    shapes = {"gptoss_g8": (8, 2880, 201088), "padded_g64": (64, 3072, 201088),
              "adversarial_g32": (32, 2880, 201088), "large_g1024": (1024, 2880, 201088), "tiny": (1, 256, 4096)}
    for name, ent in committed.items():
        emit = name.endswith("_emit")
        B, H, V = shapes[name[:-len("_emit")] if emit else name]
        w_bytes = 2 * H * V
        assert w_bytes <= ent["dram_bytes_per_launch"]
        # the tensor-core path writes its fp32 logits (to scratch for the merge's rescans, when the caller
        # takes none); the emitting form writes the caller's
        logits = 4 * B * V if emit or ent["kernel"] == "lmhead_tc_kernel" else 0
        assert ent["dram_bytes_per_launch"] <= 1.1 * (w_bytes + logits), name


def test_source_hash_covers_the_kernel_and_its_headers():
    for kernel, files in bench.ROOFLINE_KERNEL_SOURCES.items():
        assert any(f.endswith(".cu") for f in files)
        h = bench.kernel_source_hash(kernel)
        assert len(h) == 16 and int(h, 16) >= 0


def test_peaks_come_from_the_measured_file():
    pk, kind = bench.peaks()
    if not bench.os.path.exists(bench.os.path.join(bench.ROOT, "MEASURED_PEAKS.json")):
        pytest.skip("no measured peaks here")
    assert kind == "measured"
    assert pk["hbm_gbs"] > 1000 and pk["bf16_tflops_sustained"] > 100


def test_cpu_baseline_times_the_oracle_on_all_cores_and_on_one():
    import gen
    w = gen.make("tiny")
    rec = bench.cpu_baseline(w, budget_s=0.5, max_steps=3)
    assert rec["kind"] == "oracle" and rec["unit"] == "rows/s" and rec["value"] > 0
    assert rec["cores"] >= 1 and "tiny" in rec["sample"]
    one = rec["single_thread"]
    assert one["cores"] == 1 and one["value"] > 0 and one["unit"] == "rows/s"


def test_gpus_n_without_torchrun_starts_n_ranks(monkeypatch):
    # --gpus 2 outside torchrun re-launches the bench as 2 ranks on one node (rendezvous on 127.0.0.1)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    calls = []
    monkeypatch.setattr(bench.subprocess, "call", lambda cmd: calls.append(cmd) or 0)
    with pytest.raises(SystemExit) as ex:
        bench.main(["--gpus", "2", "--steps", "5", "--warmup", "3"])
    assert ex.value.code == 0 and len(calls) == 1
    cmd = calls[0]
    assert cmd[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"]
    assert "--nproc-per-node=2" in cmd and "--master-addr=127.0.0.1" in cmd
    assert cmd[cmd.index(bench.os.path.abspath(bench.__file__)) + 1:] == ["--gpus", "2", "--steps", "5", "--warmup", "3"]


def test_world_size_must_match_gpus(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "4")
    monkeypatch.setenv("RANK", "0")
    with pytest.raises(SystemExit) as ex:
        bench.main(["--gpus", "2"])
    assert "WORLD_SIZE=4" in str(ex.value.code)
    assert bench.world_mismatch(2, 2) is None and bench.world_mismatch(1, 1) is None


def test_config_records_cover_the_workloads_and_the_small_path():
    names = {n for n, _, _ in bench.CONFIGS}
    assert {"gptoss_g8", "tiny", "padded_g64", "adversarial_g32", "large_g1024"} <= names
    assert ("tiny", False, "small") in bench.CONFIGS  # tiny also on the one-launch small path
    assert all(p in ("auto", "gemv", "tensor", "small") for _, _, p in bench.CONFIGS)
    fake = types.SimpleNamespace
    assert bench.path_name(fake(small=True, tc_path=False)) == "small"
    assert bench.path_name(fake(small=False, tc_path=True)) == "tensor"
    assert bench.path_name(fake(small=False, tc_path=False)) == "mma.sync"
