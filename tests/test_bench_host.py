"""Host logic of bench.py that needs no GPU: the device-code hash that ties
the recorded ncu traffic to the kernels it was taken on, and the oracle's
column split over host threads."""
import numpy as np

import bench
import oracle
import synth


def test_code_text_drops_comments_only():
    src = ('int a = 1; // note\n'
           '/* block\n   comment */ const char* s = "a//b /* c */";\n'
           "\n"
           "char q = '/'; char e = '\\'';   \n"
           "x = a / 2;\n")
    assert bench.code_text(src) == ('int a = 1;\n'
                                    ' const char* s = "a//b /* c */";\n'
                                    "char q = '/'; char e = '\\'';\n"
                                    "x = a / 2;")


def test_kernel_hash_sees_code_not_comments(tmp_path, monkeypatch):
    d = tmp_path / "few_row_packed_gb300" / "csrc"
    d.mkdir(parents=True)
    (d / "k.cuh").write_text("// v1\n__global__ void k() { int x = 1; }\n")
    (d / "api.cpp").write_text("int host = 1;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_hash()
    (d / "k.cuh").write_text("/* v2, reworded */\n\n__global__ void k() { int x = 1; }  // same\n")
    (d / "api.cpp").write_text("int host = 2;\n")          # host code is not hashed
    assert bench.kernel_hash() == h0
    (d / "k.cuh").write_text("__global__ void k() { int x = 2; }\n")
    assert bench.kernel_hash() != h0


def test_oracle_over_threads_equals_one_thread(monkeypatch):
    """The all-cores baseline runs the unchanged oracle on column ranges;
    gathering those ranges gives the single call's result bit for bit."""
    oracle.build()
    mat = synth.Matrix("w", synth.AFFINE2, 512, 200, 64, "f16", sigma_scale=0.01)
    parts, xb = synth.gen_matrix(mat, 3, rows=8)
    Xf = oracle.x_to_f64(xb, "f16")
    Y1, _ = oracle.verify(1, parts, Xf, 512, 200, 64)
    got = {}
    real = oracle.verify

    def record(fmt, p, X, K, N, group, cols=None):
        Y, A = real(fmt, p, X, K, N, group, cols=cols)
        got[int(cols[0])] = (cols, Y)
        return Y, A

    monkeypatch.setattr(oracle, "verify", record)
    bench.oracle_columns(oracle, 1, parts, Xf, mat, np.arange(200), 3)
    assert len(got) == 3
    Y = np.empty_like(Y1)
    for cols, Yc in got.values():
        Y[:, cols] = Yc
    assert np.array_equal(Y, Y1)


def test_packed_bytes_formula_matches_library():
    """The bench's algorithmic byte counts (from the formats' bits per weight)
    equal the library's packed sizes on every configuration."""
    import few_row_packed_gb300 as lbv
    for wl in synth.WORKLOADS.values():
        for m in wl.matrices:
            assert bench.packed_weight_bytes(m) == lbv.packed_bytes(
                bench.FMT_IDS[m.fmt], m.K, m.N, m.group), m.name


def test_reference_arm_does_not_load_the_library():
    """`bench.py --impl reference` times the oracle alone: the CUDA library's
    package is never imported."""
    import json
    import subprocess
    import sys
    code = ("import sys, json, bench\n"
            "class A: pass\n"
            "a = A(); a.workload = 'sign1_tiny_512x256'; a.M = 8; a.steps = 1; a.warmup = 0\n"
            "a.head = 'fused'; a.gpus = 1\n"
            "line = bench.run_reference(a)\n"
            "assert 'few_row_packed_gb300' not in sys.modules\n"
            "print(json.dumps(line))\n")
    out = subprocess.run([sys.executable, "-c", code], cwd=bench.ROOT, capture_output=True,
                         text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
