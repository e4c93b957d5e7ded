"""Host-side logic of bench.py (no GPU): byte accounting, clock-sample parsing,
and the max-over-ranks / sum-over-ranks reduction on two gloo ranks."""
import json
import os
import socket
import subprocess
import sys
import textwrap

import bench


def test_algorithmic_bytes():
    # codes + scales + zero points + x + y of the 0.5B LM head at M = 1
    assert bench.algorithmic_bytes(1, 151936, 896, 32) == 68067328 + 8508416 + 2127104 + 896 * 4 + 151936 * 4
    assert bench.algorithmic_bytes(2, 4096, 4096, 128, symmetric=True) == 4096 * 2048 + 4096 * 32 * 2 + 2 * 4096 * 4 * 2


def test_clock_sampler_parsing_without_nvidia_smi():
    cs = bench.ClockSampler(0)
    cs.proc = None
    assert cs.stop()["sm_mhz"] is None
    cs = bench.ClockSampler(0)

    class P:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0
    cs.proc = P()
    cs.lines = [(1.0, "0, 1900, 2070, 800.0, 0x0, Not Active, Not Active, Not Active, Active"),
                (2.0, "0, 2000, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active")]
    r = cs.stop(0.5, 3.0)
    assert r["sm_mhz"] == 1950.0 and r["sm_max_mhz"] == 2070.0 and r["reasons"] == ["sw_power_cap"]
    r = cs.stop(10.0, 11.0)          # no sample inside the window: falls back to all samples
    assert r["samples_in_timed_region"] == 0 and r["sm_mhz"] == 1950.0


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_reduce_over_two_gloo_ranks(tmp_path):
    script = tmp_path / "ranks.py"
    script.write_text(textwrap.dedent(f"""
        import os, sys
        sys.path.insert(0, {os.path.dirname(os.path.dirname(os.path.abspath(__file__)))!r})
        import bench
        rank, world, _ = bench.dist_env()
        dist = bench.dist_init(world, "gloo")
        mx = bench.reduce_over_ranks(dist, float(rank + 1) * 10.0, "max")
        sm = bench.reduce_over_ranks(dist, float(rank + 1), "sum")
        bench.barrier(dist)
        print(f"rank={{rank}} max={{mx}} sum={{sm}}", flush=True)
        dist.destroy_process_group()
    """))
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE="2", LOCAL_RANK=str(r),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.STDOUT, text=True))
    outs = [p.communicate(timeout=120)[0] for p in procs]
    assert all(p.returncode == 0 for p in procs), outs
    for o in outs:
        assert "max=20.0 sum=3.0" in o, o


def test_reference_arm_runs_the_oracle(tmp_path):
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
                          "--ref-seconds", "1"], cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr
    import json
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0
    assert "row slices" in line["cpu_baseline"]["sample"]


def test_reference_arm_shares_many_steps_over_cores():
    # with at least four steps per core, whole steps go to one worker thread per core
    steps = 4 * (os.cpu_count() or 1)
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", str(steps), "--warmup", "1",
                          "--ref-seconds", "2"], cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr
    import json
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["steps"] == steps and line["value"] > 0
    assert "worker threads" in line["cpu_baseline"]["sample"]
    assert line["cpu_baseline"]["cores"] == (os.cpu_count() or 1)


def test_sweep_checkpoint_round_trip(tmp_path):
    # the --sweep-out file is JSON lines; a rerun skips the cells it finds, and a last
    # line cut short by an interrupted run is ignored
    import bench
    path = tmp_path / "sweep.jsonl"
    cells = [{"M": 1, "N": 4096, "K": 896, "group": 32, "symmetric": False, "us_per_call": 2.0},
             {"M": 16, "N": 4096, "K": 896, "group": 32, "symmetric": True, "us_per_call": 9.0},
             {"kind": "f32", "M": 1, "N": 4096, "K": 896, "us_per_call": 3.0},
             {"kind": "probe", "bytes": 16384, "us_per_call": 1.5}]
    path.write_text("".join(json.dumps(c) + "\n" for c in cells) + '{"M": 1, "N": 51')
    done = bench.load_sweep_checkpoint(str(path))
    assert set(done) == {(1, 4096, 896, 32, False), (16, 4096, 896, 32, True), ("f32", 1, 4096, 896),
                         ("probe", 16384)}
    assert done[(16, 4096, 896, 32, True)]["us_per_call"] == 9.0
    assert done[("f32", 1, 4096, 896)]["us_per_call"] == 3.0
    assert bench.load_sweep_checkpoint(str(tmp_path / "missing.jsonl")) == {}
    assert bench.load_sweep_checkpoint(None) == {}
