"""The C ABI from a plain C99 program: both headers compile as strict C
(-std=c99 -pedantic -Werror), the struct layouts the C compiler gives equal
the Python binding's ctypes structures, and the host-only entry points give
the same answers from C as through the binding and the oracle."""
import ctypes
import os
import shutil
import subprocess

import pytest

from block_diffusion_lm_gb300 import csbp
from oracle import csbp_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "block_diffusion_lm_gb300")


@pytest.fixture(scope="module")
def c_output(tmp_path_factory):
    from block_diffusion_lm_gb300 import build
    build.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path_factory.mktemp("cabi") / "c_abi_check")
    cmd = [cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi_check.c"),
           "-L", PKG, "-lcsbp", f"-Wl,-rpath,{PKG}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    out = {}
    for line in r.stdout.splitlines():
        key, _, val = line.rpartition(" ") if line.startswith(("offset", "sizeof")) \
            else line.partition(" ")
        out[key] = val
    return out


def test_struct_layouts_match_the_binding(c_output):
    o = c_output
    assert int(o["sizeof csbp_problem"]) == ctypes.sizeof(csbp.Problem)
    for f in ("scale", "window", "bwd_chunk", "per_rank", "rank"):
        assert int(o[f"offset csbp_problem.{f}"]) == getattr(csbp.Problem, f).offset, f
    assert int(o["sizeof csbp_inputs"]) == ctypes.sizeof(csbp.Inputs)
    for f in ("v_corr", "stride_tok", "stride_batch"):
        assert int(o[f"offset csbp_inputs.{f}"]) == getattr(csbp.Inputs, f).offset, f
    assert int(o["sizeof csbp_schedule_info"]) == ctypes.sizeof(csbp.ScheduleInfo)
    for f in ("tile_pairs", "bytes", "problem_key"):
        assert int(o[f"offset csbp_schedule_info.{f}"]) == getattr(csbp.ScheduleInfo, f).offset
    assert int(o["sizeof csbp_ce_problem"]) == ctypes.sizeof(csbp.CeProblem)
    for f in ("d_model", "grad_scale"):
        assert int(o[f"offset csbp_ce_problem.{f}"]) == getattr(csbp.CeProblem, f).offset, f


def test_host_entry_points_agree_with_the_binding_and_the_oracle(c_output):
    o = c_output
    assert int(o["version"]) == csbp.lib().csbp_version()
    prob = csbp.make_problem(1, 1024, 32, 4, 2, 128, P=2)
    bo, co, _, info = csbp.block_schedule(prob)
    assert int(o["tile_pairs"]) == info.tile_pairs == len(O.tile_pairs(1024, 32, 128, 128, 2))
    assert [int(x) for x in o["owner_first_last"].split()] == [bo[0], bo[31]]
    assert [int(x) for x in o["chunk_owner"].split()] == list(co) == list(O.chunk_owner(1024, 2))
    assert int(o["fwd_workspace"]) == csbp.workspace_bytes(prob, 0)
    assert int(o["bwd_workspace"]) == csbp.workspace_bytes(prob, 1)
    assert o["status_workspace"] == csbp.lib().csbp_status_string(-3).decode()
    assert int(o["fwd_without_inputs"]) == -1
    assert int(o["fwd_bad_stride"]) == -1
    assert int(o["fwd_other_problem"]) == -1
    assert int(o["fwd_small_workspace"]) == -3
    ce = csbp.make_ce_problem(1000, 256, 4096, 0, True, 0.001)
    assert int(o["ce_workspace"]) == csbp.ce_workspace_bytes(ce) > 0
    assert int(o["ce_workspace_invalid"]) == 0
    assert int(o["rank_size_query"]) == -6      # CSBP_ERR_CAPACITY: the size query of a valid list
    assert int(o["rank_out_of_range"]) == -1
    assert [int(o[k]) for k in ("e4m3_null", "e4m3_zero_scale", "e4m3_misaligned")] == [-1] * 3
    assert int(o["e4m3_empty"]) == 0


def test_schedule_builder_compiles_without_warnings():
    """The host schedule builder is plain C++17: it compiles warning-free
    with -Wall -Wextra -Wpedantic -Wshadow as errors."""
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    cmd = [cxx, "-std=c++17", "-Wall", "-Wextra", "-Wpedantic", "-Wshadow", "-Werror",
           "-fsyntax-only", "-I", os.path.join(ROOT, "include"),
           "-I", "/usr/local/cuda/include", os.path.join(PKG, "csrc", "schedule.cpp")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_headers_compile_as_strict_cpp():
    """C++ callers (framework plugins, custom ops) include the headers too."""
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    src = '#include "csbp.h"\n#include "csbp_vocab_ce.h"\nint main() { return csbp_version() > 0 ? 0 : 1; }\n'
    r = subprocess.run([cxx, "-std=c++17", "-Wall", "-Wextra", "-Wpedantic", "-Werror",
                        "-fsyntax-only", "-x", "c++", "-I", os.path.join(ROOT, "include"), "-"],
                       input=src, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_kernel_setup_runs_once_per_device(tmp_path):
    """The launchers set a kernel's shared-memory limit once per device
    ordinal (csrc/device_once.h): a second device gets its own set-up, a
    failed set-up is retried, and racing threads run it once."""
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = str(tmp_path / "device_once_check")
    cmd = [cxx, "-std=c++17", "-Wall", "-Wextra", "-Werror", "-pthread",
           "-I", os.path.join(PKG, "csrc"), os.path.join(ROOT, "tests", "device_once_check.cpp"),
           "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    lines = r.stdout.splitlines()
    assert lines[0] == "first 1 1 1 calls 1 1 done2 0"
    assert lines[1] == "retry 0 1 1 tries 2"
    assert lines[2] == "outside 0 0 runs 0"
    assert lines[3] == "race calls 1 ok 16"
