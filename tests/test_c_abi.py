"""The C-ABI from C itself: include/kvx.h compiles as C11 and C++17, a plain C client
(tests/c/kvx_c_demo.c) links against libkvx.so and the CUDA runtime, pushes two requests and checks
every consumer byte on the host, plus the error path; and a plain C driver of the host connector
(tests/c/kvx_conn_rate.c) takes requests through the whole protocol, no GPU needed."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
PKG = os.path.join(ROOT, "disaggregated_prefill_decode_gb300")
DEMO = os.path.join(ROOT, "tests", "c", "kvx_c_demo.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def cuda_include():
    inc = os.path.join(CUDA, "include")
    if not os.path.exists(os.path.join(inc, "cuda_runtime_api.h")):
        pytest.skip("CUDA headers not found")
    return inc


@pytest.mark.parametrize("lang,std,cc", [("c", "c11", "gcc"), ("c++", "c++17", "g++")])
def test_header_compiles(lang, std, cc, tmp_path):
    if not shutil.which(cc):
        pytest.skip(f"{cc} not found")
    src = tmp_path / ("use." + ("c" if lang == "c" else "cpp"))
    src.write_text('#include "kvx.h"\nint main(void) { kvx_pool p; (void)p; return kvx_status_str(KVX_OK) == 0; }\n')
    r = subprocess.run([cc, "-x", lang, f"-std={std}", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-fsyntax-only", "-I", INCLUDE, "-I", cuda_include(), str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def build_demo(tmp_path, source=DEMO):
    if not shutil.which("gcc"):
        pytest.skip("gcc not found")
    if not os.path.exists(os.path.join(PKG, "libkvx.so")):
        pytest.skip("libkvx.so not built")
    lib64 = os.path.join(CUDA, "lib64")
    exe = tmp_path / os.path.splitext(os.path.basename(source))[0]
    r = subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", source, "-o", str(exe),
                        "-I", INCLUDE, "-I", cuda_include(), "-L", PKG, "-lkvx", "-L", lib64, "-lcudart",
                        f"-Wl,-rpath,{PKG}:{lib64}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_demo_links(tmp_path):
    build_demo(tmp_path)


@pytest.mark.gpu
def test_c_demo_runs(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    exe = build_demo(tmp_path)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c demo ok" in r.stdout


def test_connector_protocol_from_c(tmp_path):
    """Every request through registration, prefill, start, write, seal, report and release reaches DONE."""
    exe = build_demo(tmp_path, os.path.join(ROOT, "tests", "c", "kvx_conn_rate.c"))
    r = subprocess.run([str(exe), "20000"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert float(r.stdout.split()[-1]) > 0
