"""The benchmark's byte model and its JSON contract, without a GPU.

The byte model is pinned to the pages: "MARLIN: Mixed-Precision Auto-Regressive
Parallel Inference on Large Language Models" note, key results, quotes a 3.87x
ideal speed-up over FP16 for INT4 weights with group 128, which is the ratio of
bytes per weight, 2 / (0.5 + 2/128). The reference arm (the CPU oracle) runs here,
so its JSON line is checked for every key the contract asks for."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_byte_model_reproduces_the_ideal_speedup():
    r = bench.fp16_over_int4_byte_ratio(128)
    assert 3.87 <= r < 3.88
    assert bench.fp16_over_int4_byte_ratio(32) < r < bench.fp16_over_int4_byte_ratio(4096)


def test_algorithmic_bytes_and_flops():
    # 4096 x 4096, G = 128: codes K*N/2, scales ceil(K/G)*N*2, X 2MK, Y 2MN
    assert bench.weight_bytes(4096, 4096, 128) == 4096 * 4096 // 2 + 32 * 4096 * 2
    assert bench.algorithmic_bytes(16, 4096, 4096, 128) == bench.weight_bytes(4096, 4096, 128) + 2 * 16 * 4096 * 2
    # a partial last group is padded to a whole group of codes
    assert bench.weight_bytes(4000, 256, 128) == 32 * 128 * 256 // 2 + 32 * 256 * 2
    assert bench.flops(16, 4096, 4096) == 2 * 16 * 4096 * 4096


def test_roofline_picks_the_binding_resource():
    peaks = {"hbm_gbs": 6688.8, "bf16_tflops": 1939.9}
    small = bench.roofline_seconds(1, 4096, 4096, 128, peaks)
    assert small == pytest.approx(bench.algorithmic_bytes(1, 4096, 4096, 128) / 6688.8e9)
    big = bench.roofline_seconds(4096, 5120, 15360, 128, peaks)
    assert big == pytest.approx(bench.flops(4096, 5120, 15360) / 1939.9e12)


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "single_m16_4096x4096", "--steps", "2", "--warmup", "3"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] >= 3 and d["value"] > 0
    assert d["config"]["workload"] == "single_m16_4096x4096"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    out = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                          "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                          "--impl", "reference", "--workload", "single_m16_4096x4096", "--gpus", "2",
                          "--steps", "1", "--warmup", "3"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


def test_gpu_arm_refuses_more_than_one_gpu():
    """The GPU arm is single-GPU: asked for several GPUs (by flag or by a launcher's
    WORLD_SIZE) it exits non-zero with a plain message, before any CUDA work."""
    assert bench.single_gpu_refusal(1, {}) is None
    assert bench.single_gpu_refusal(1, {"WORLD_SIZE": "1"}) is None
    assert "one GPU" in bench.single_gpu_refusal(2, {})
    assert "one GPU" in bench.single_gpu_refusal(1, {"WORLD_SIZE": "2"})
    for argv, env in ((["--gpus", "2"], {}), ([], {"WORLD_SIZE": "2", "RANK": "0"})):
        out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + argv + ["--steps", "1"],
                             capture_output=True, text=True, timeout=300, cwd=ROOT,
                             env=dict(os.environ, CUDA_VISIBLE_DEVICES="", **env))
        assert out.returncode != 0
        assert "one GPU only" in out.stderr
        assert not [l for l in out.stdout.splitlines() if l.startswith("{")]


def test_warmup_below_three_is_an_error():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--warmup", "2"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode != 0 and "at least 3" in out.stderr


def test_source_digest_ignores_comments_but_not_code():
    """The key of the committed DRAM counters follows the code: a comment or layout edit
    keeps it, any change of code (string literals included) does not."""
    a = 'int f(int x) { // one\n  return x + 1; /* two */ }\nconst char* s = "// not a comment";\n'
    b = 'int f(int x)\n{\n    return x + 1;   // changed comment\n}\nconst char* s = "// not a comment";\n'
    c = 'int f(int x) { return x + 2; }\nconst char* s = "// not a comment";\n'
    d = 'int f(int x) { return x + 1; }\nconst char* s = "// not a  comment";\n'
    sa, sb, sc, sd = (bench.strip_comments(t) for t in (a, b, c, d))
    assert sa.replace("{ ", "{").replace(" }", "}") == sb.replace("{ ", "{").replace(" }", "}")
    assert sa != sc and sa != sd
    assert '"// not a comment"' in sa
