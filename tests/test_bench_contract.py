"""The bench's reference arm (the CPU oracle on the headline workload) prints
one JSON line with the keys the bench contract requires.  CPU only."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1", "--oracle-threads", "2"], capture_output=True, text=True, cwd=ROOT,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["higher_is_better"] is True and d["steps"] == 1
    assert d["value"] > 0 and d["unit"] == "draft steps/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 2
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["Vc"] == 65_536 and d["config"]["H"] == 2048 and d["config"]["B"] == 1


def test_command_line_offers_configs_and_oracle_threads():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--help"], capture_output=True, text=True,
                       cwd=ROOT, timeout=120)
    assert r.returncode == 0
    for flag in ("--gpus", "--steps", "--warmup", "--impl", "--config", "--workload", "--oracle-threads"):
        assert flag in r.stdout, flag


def test_reference_arm_under_torchrun_prints_once():
    """Launched as a multi-GPU run is launched (torchrun, 127.0.0.1): rank 0
    alone times the oracle and prints the line; the other rank exits 0."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1", "--oracle-threads", "2"],
                       capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


def test_profile_key_ignores_comments_only(tmp_path, monkeypatch):
    """A profile stays keyed to its kernel through comment and blank-line edits;
    a code edit changes the key."""
    sys.path.insert(0, ROOT)
    import bench
    src = os.path.join(ROOT, "verify_head_gb300", "csrc")
    csrc = tmp_path / "verify_head_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in ("gemv_argmax.cu",) + bench.KERNEL_HEADERS:
        (csrc / name).write_text(open(os.path.join(src, name), encoding="utf-8").read(), encoding="utf-8")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.source_sha("gemv_argmax.cu")
    k = csrc / "gemv_argmax.cu"
    text = k.read_text(encoding="utf-8")
    k.write_text("// a new comment\n\n" + text.replace("\n", "  \n", 3) + "\n/* block\n comment */\n", encoding="utf-8")
    assert bench.source_sha("gemv_argmax.cu") == base
    k.write_text(text + "\nstatic int vh_unused_for_test = 1;\n", encoding="utf-8")
    assert bench.source_sha("gemv_argmax.cu") != base
