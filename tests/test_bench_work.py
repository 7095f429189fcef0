"""Host-side figures the benchmark reports: the operator-sweep shapes, the
algorithmic bytes of one replay call, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
import bench  # noqa: E402


def test_sweep_shapes_span_the_pages_ranges():
    # OneLA §3 (operator experiments): R 4/8/16, W 128/256/512, T 2..6 and
    # nine geometries with H_K 4-32, H_V 4-64, K 128-256, V 128-512; 405 shapes
    shapes = [(g, R, W, T) for g in synth.SWEEP_GEOMETRIES for R in synth.SWEEP_R
              for W in synth.SWEEP_W for T in synth.SWEEP_T]
    assert len(shapes) == 405 and len(set(synth.SWEEP_GEOMETRIES)) == 9
    for Hk, H, K, V in synth.SWEEP_GEOMETRIES:
        assert 4 <= Hk <= 32 and 4 <= H <= 64 and 128 <= K <= 256 and 128 <= V <= 512
        assert H % Hk == 0  # value heads share key heads in whole groups
    assert (16, 16, 128, 128) in synth.SWEEP_GEOMETRIES  # the pages' Qwen geometry
    # every end of every range is reached
    for i, ends in enumerate([(4, 32), (4, 64), (128, 256), (128, 512)]):
        vals = {g[i] for g in synth.SWEEP_GEOMETRIES}
        assert min(vals) == ends[0] and max(vals) == ends[1]


def test_replay_bytes_of_the_batched_depth_two_call():
    # 64 requests x 512 beams, 16 heads of width 128, bf16, two ancestors:
    # per beam q,k 8192 + v 4096 + gates 128 + 2 x (k_j 4096 + delta_j 4096 +
    # alpha_j 64) + delta_t,o_t 8192 = 37120 bytes, plus S_ctx (fp32) once
    # per request and head: 64 * 16 * 128 * 128 * 4 bytes
    assert bench.replay_bytes(64, 512, 16, 16, 128, 128, 2, 2) == 32768 * 37120 + 67108864
    # grouped key heads read one key row per key head
    assert (bench.replay_bytes(1, 1, 16, 4, 128, 128, 0, 2)
            == 2 * 4 * 128 * 2 + 16 * 128 * 2 + 2 * 16 * 4 + 2 * 16 * 128 * 2 + 16 * 128 * 128 * 4)


def test_replay_bytes_with_a_residual_stream():
    # stacked layers: delta_t is stored (bf16) but o_t only updates the fp32
    # residual row, read and written: 8 heads x 128 values x (2 + 4 + 4) bytes
    # in place of delta_t and o_t's 2 x 2 bytes
    plain = bench.replay_bytes(32, 1024, 8, 8, 128, 128, 1, 2)
    resid = bench.replay_bytes(32, 1024, 8, 8, 128, 128, 1, 2, residual=True)
    assert resid - plain == 32 * 1024 * 8 * 128 * (10 - 4)


def _reference_run(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--steps", "1", "--warmup", "1"], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_the_contract_line():
    # the oracle timed on the host cores, on the same workload description
    # as the CUDA arm's line
    run = _reference_run({"RANK": "0", "WORLD_SIZE": "1"})
    assert run.returncode == 0, run.stderr[-2000:]
    line = json.loads(run.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == bench.UNIT and line["higher_is_better"] is True
    assert line["value"] > 0 and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": bench.UNIT,
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    wl = synth.WORKLOADS["batched_r64_w512"]
    cfg = dict(line["config"])
    assert cfg.pop("sample")
    assert cfg == bench.workload_config(wl)


def test_reference_arm_prints_nothing_on_other_ranks():
    run = _reference_run({"RANK": "1", "WORLD_SIZE": "2"})
    assert run.returncode == 0, run.stderr[-2000:]
    assert run.stdout.strip() == ""


def test_gemm_and_selection_work_of_a_metric_decode_call():
    # 64 requests x 512 beams: the projection GEMM is 32768 x 2048 x 6176
    # (q, k, v of 16 heads of 128, and 2 x 16 gate logits) = 829 GFLOP, the
    # codebook logits 32768 x 2048 x 8192 = 1.10 TFLOP; the selection reads the
    # 32 tile statistics of each row (8 B each), each row's lse and cumulative
    # score, and W_next = 512 listed tiles of 256 bf16 logits per request
    wl = synth.WORKLOADS["batched_r64_w512"]
    w = bench.stage_work(wl, 1)
    n = 64 * 512
    assert w["project"] == 2.0 * n * 2048 * 6176
    assert abs(w["project"] / 829e9 - 1) < 2e-3
    assert w["logits"] == 2.0 * n * 2048 * 8192
    assert abs(w["logits"] / 1.0995e12 - 1) < 1e-4
    assert w["select"] == n * 32 * 8 + n * 8 + 64 * 512 * 256 * 2
    assert abs(w["select"] / 25.4e6 - 1) < 1e-2


def test_stacked_layers_multiply_the_projection_work():
    # four layers of 8 heads (d_model 1024): one projection GEMM per layer,
    # one codebook head
    wl = synth.WORKLOADS["deep4_w1024"]
    w = bench.stage_work(wl, 0)
    n = 32 * 1024
    assert w["project"] == 4 * 2.0 * n * 1024 * (3 * 8 * 128 + 2 * 8)
    assert w["logits"] == 2.0 * n * 1024 * 4096


def test_clock_summary_takes_the_loaded_samples():
    # idle samples (low power) around the timed region do not set the median;
    # any throttle reason seen in any sample is reported
    rows = [
        ["0", "2070", "2070", "120.5", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"],
        ["0", "1800", "2070", "1390.1", "0x4", "Not Active", "Not Active", "Not Active", "Active"],
        ["0", "1850", "2070", "1385.0", "0x4", "Not Active", "Not Active", "Not Active", "Active"],
        ["0", "1900", "2070", "1200.0", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"],
        ["0", "2070", "2070", "[N/A]", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"],
    ]
    c = bench.summarize_clock_rows(rows)
    assert c["sm_mhz"] == 1850.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 5 and c["samples_under_load"] == 3
    idle = bench.summarize_clock_rows([["0", "345", "2070", "[N/A]"] + ["Not Active"] * 5])
    assert idle["sm_mhz"] == 345.0 and idle["samples_under_load"] == 0


def _ours_run(args, env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          env=env, capture_output=True, text=True, timeout=300)


def test_more_than_one_gpu_is_refused_before_any_gpu_work():
    # the decode runs on one GPU (replicas are not built): a torchrun launch
    # (WORLD_SIZE > 1) or --gpus > 1 exits with a reason and does no work
    for args, env in ((["--steps", "1"], {"RANK": "0", "WORLD_SIZE": "2", "LOCAL_RANK": "0"}),
                      (["--gpus", "2", "--steps", "1"], {"WORLD_SIZE": "1"}),
                      (["--stage", "logits", "--gpus", "4"], {})):
        run = _ours_run(args, env)
        assert run.returncode == 2, (args, run.stderr[-2000:])
        line = json.loads(run.stdout.strip().splitlines()[-1])
        assert line["metric"] == bench.METRIC and "one GPU" in line["unavailable"]
        assert "one GPU" in run.stderr
    other = _ours_run(["--steps", "1"], {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert other.returncode == 2 and other.stdout.strip() == ""


def test_one_gpu_run_is_not_refused():
    ns = type("A", (), {"gpus": 1})
    assert bench.multi_gpu_refusal(ns, {"WORLD_SIZE": "1"}) is None
    assert bench.multi_gpu_refusal(ns, {}) is None
    assert bench.multi_gpu_refusal(ns, {"WORLD_SIZE": "2"}) is not None
