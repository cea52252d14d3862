"""The benchmark's reference arm runs on the CPU (it times the oracle): its
JSON line carries the contract's keys, and under torchrun only rank 0
prints.  The hash that ties the stored ncu counters to the device code
ignores comments only."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           *args], capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)


def test_reference_arm_line():
    out = _run({}, "--steps", "2", "--warmup", "3", "--workload", "toy_1000",
               "--cpu-threads", "2")
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 2
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] and d["config"]["workload"] == "toy_1000"


def test_reference_arm_only_rank_zero_prints():
    out = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--steps", "1",
               "--workload", "toy_1000", "--cpu-threads", "1")
    assert out.returncode == 0, out.stderr
    assert not [l for l in out.stdout.splitlines() if l.startswith("{")]


def test_kernel_hash_ignores_comments_only():
    """The stored ncu counters stay valid across comment edits of the device
    code and are voided by any code change."""
    sys.path.insert(0, ROOT)
    import bench

    code = 'int f(int x) { return x + 1; }  // one\n/* two */ const char *s = "a // b";\n'
    same = '// header\nint f(int x)\n{\n    return x + 1;  /* inline */\n}\nconst char *s = "a // b";'
    other = 'int f(int x) { return x + 2; }\nconst char *s = "a // b";'
    strip = bench.strip_c_comments
    assert strip(code) == strip(same)
    assert strip(code) != strip(other)
    assert '"a // b"' in strip(code)
    assert len(bench.kernel_source_hash()) == 16


def test_reference_arm_config_is_the_gpu_arms():
    """Both arms print the same `config` object for a workload: the
    reference arm's comes from the oracle's layout, the GPU arm's from the
    library's (host-only calls), and the two layouts agree."""
    sys.path.insert(0, ROOT)
    import bench
    from zero_distributed_optimizer_gb300 import binding as B

    out = _run({}, "--steps", "1", "--warmup", "3", "--workload", "toy_1000",
               "--cpu-threads", "1")
    assert out.returncode == 0, out.stderr
    d = json.loads([l for l in out.stdout.splitlines() if l.startswith("{")][0])
    w = bench.workload_by_name("toy_1000")
    L = B.dopt_build_range_map(list(w.sizes), w.D, w.bucket_elems, w.pad_unit, list(w.wd_mask))
    assert d["config"] == bench.workload_config(w, L.padded_numel, L.n_buckets, 1)
