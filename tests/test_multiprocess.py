"""Multi-process (world size 2) checks of the bench's host-side rank logic on
CPU with the gloo backend: every (sequence, head) chain is independent, so N
GPUs run N replicas with no data-path collective; the only collectives are the
timing barrier and the max over ranks of the elapsed time.  The reference arm
under torchrun must print one line, from rank 0, with every rank exiting 0.
Also the bench's other host logic: the verify reference arm, the clock
sampler's parsing and the traffic record lookup."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2",
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, ws, _ = bench.dist_init(2)
    bench.barrier(ws)
    m = bench.max_over_ranks(10.0 + r, ws)
    q.put((r, ws, m, dist.get_backend()))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2 and g[2] == 11.0 and g[3] == "gloo" for g in got)


def test_reference_arm_under_torchrun_prints_once_from_rank_zero():
    port = _free_port()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--config", "tiny"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0


def test_verify_reference_arm_prints_one_line():
    """bench.py --config verify --impl reference: the oracle's verify on a
    bounded sample of the verify workload, one JSON line in draft tokens/s."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "verify",
           "--pool", "bf16", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "draft tokens/s" and rec["value"] > 0
    assert rec["config"]["workload"] == "verify" and rec["config"]["pool"] == "bf16"
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["e2e"]["h2d_bytes_per_step"] == 0


def test_clock_sampler_reads_median_clock_and_throttle_reasons(tmp_path):
    """The bench's nvidia-smi sampler: median SM clock under load, the maximum
    clock, and every throttle reason seen Active in any sample (fed a recorded
    CSV instead of a live nvidia-smi)."""
    sys.path.insert(0, ROOT)
    import bench
    csv = tmp_path / "clocks.csv"
    csv.write_text(
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n"
        "0, 1980, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, Active\n"
        "0, 2070, 2070, 1100.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
        "garbled line\n")

    class _Done:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    s = bench.ClockSampler(0)
    s.proc, s.path = _Done(), str(csv)
    clk = s.stop()
    assert clk["sm_mhz"] == 2070.0 and clk["sm_max_mhz"] == 2070.0 and clk["samples"] == 3
    assert clk["reasons"] == ["sw_power_cap"]
    assert not csv.exists()


def test_captured_traffic_only_for_the_profiled_kernel_source(tmp_path, monkeypatch):
    """The bench's roofline `traffic` comes from a committed ncu record only
    while the kernel source still has the hash the record names; scaled by
    token-heads."""
    import hashlib
    sys.path.insert(0, ROOT)
    import bench
    (tmp_path / "profiles").mkdir()
    src_dir = tmp_path / "kda_chunked_prefill_02_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    src = src_dir / "kda_prep.cu"
    src.write_bytes(b"// kernel v1\n")
    sha = hashlib.sha256(b"// kernel v1\n").hexdigest()[:16]
    (tmp_path / "profiles" / "prep_kernel_traffic.txt").write_text(
        "kernel: prep_kernel\nsource_sha256_prefix: %s\ndram_bytes_per_token_head: 2500.0\n" % sha)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.captured_traffic("prep", 1000) == 2500.0 * 1000
    assert bench.captured_traffic("state", 1000) is None      # no record
    src.write_bytes(b"// kernel v2\n")
    assert bench.captured_traffic("prep", 1000) is None       # source changed since the capture
