"""Host code under AddressSanitizer and UndefinedBehaviorSanitizer: the CUDA
library's host-only planning and checks (pskv_plan.cpp) and the CPU oracle,
each built with the system compiler and run on small cases."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.join(ROOT, "tests", "sanitize")
SAN = ["-fsanitize=address,undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer",
       "-g", "-O1"]


def _build_and_run(tmp_path, compiler, sources, includes, name, extra=()):
    exe = str(tmp_path / name)
    cmd = [compiler, *SAN, *extra, *[f"-I{i}" for i in includes], *sources, "-o", exe, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0 and "asan" in res.stderr.lower():
        pytest.skip("sanitizer runtime not available: " + res.stderr[-300:])
    assert res.returncode == 0, res.stderr
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1", UBSAN_OPTIONS="print_stacktrace=1")
    run = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    return run.stdout


@pytest.mark.skipif(shutil.which("g++") is None, reason="no C++ compiler")
def test_library_host_planning_under_sanitizers(tmp_path):
    csrc = os.path.join(ROOT, "paged_split_kv_attn_gb300", "csrc")
    out = _build_and_run(tmp_path, "g++", [os.path.join(HERE, "plan_driver.cpp"),
                                           os.path.join(csrc, "pskv_plan.cpp")],
                         [csrc, os.path.join(ROOT, "include")], "plan_driver", ["-std=c++17"])
    assert "plan driver ok" in out


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_oracle_under_sanitizers(tmp_path):
    odir = os.path.join(ROOT, "oracle")
    out = _build_and_run(tmp_path, "gcc", [os.path.join(HERE, "oracle_driver.c"),
                                           os.path.join(odir, "pskv_oracle.c")],
                         [odir], "oracle_driver", ["-std=c11"])
    assert "oracle driver ok" in out
