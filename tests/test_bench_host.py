"""Host-side logic of bench.py that needs no GPU.

The roofline's `traffic` figure comes from DRAM counters committed under
profiles/, valid only while the kernel they were taken on is unchanged: the
check hashes the kernel sources with their comments stripped, so a comment
edit keeps the counters and any code edit drops them.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_strip_comments_keeps_code_and_literals():
    src = ('int a = 1; // note\n'
           '/* block\n   comment */ int b = 2;\n'
           'const char* s = "// not a comment";\n'
           "char c = '/';\n"
           '\n'
           'asm volatile("bar.sync %0, %1;" ::"r"(x));  /* trailing */\n')
    out = bench.strip_comments(src)
    assert out.splitlines() == ['int a = 1;', ' int b = 2;', 'const char* s = "// not a comment";',
                                "char c = '/';", 'asm volatile("bar.sync %0, %1;" ::"r"(x));']


def test_comment_edit_keeps_hash_code_edit_changes_it():
    base = "__global__ void k(float* y) {\n    y[0] = 1.f;  // store\n}\n"
    reworded = "// a kernel\n__global__ void k(float* y) {\n    y[0] = 1.f;  /* the store */\n}\n"
    changed = "__global__ void k(float* y) {\n    y[1] = 1.f;  // store\n}\n"
    s = bench.strip_comments
    assert s(base) == s(reworded)
    assert s(base) != s(changed)


def test_traffic_counters_only_for_the_kernel_they_were_taken_on(tmp_path):
    # counters recorded under the current sources' hash are returned; under
    # any other hash (the kernel changed since) the figure is None
    import json
    srcs = ["k_gemv.cu", "decode.cuh", "sm100_async.cuh"]
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps({"k_gemv<Q8_0>": {"dram_bytes_per_launch": 123, "src_sha": bench.src_hash(*srcs)},
                             "k_gemv<Q4_0>": {"dram_bytes_per_launch": 456, "src_sha": "0" * 16}}))
    assert bench.traffic_for("k_gemv<Q8_0>", srcs, str(p)) == 123
    assert bench.traffic_for("k_gemv<Q4_0>", srcs, str(p)) is None
    assert bench.traffic_for("k_gemv<Q5_0>", srcs, str(p)) is None


def test_reference_arm_json_line_keeps_the_contract():
    # the CPU oracle arm: one JSON line with the keys the bench contract names,
    # its cpu_baseline and e2e describing this same run
    import json
    import subprocess
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 0 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["value"] > 0 and d["unit"] == "GB/s"
    assert "workload" in d["config"] and "model" not in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
