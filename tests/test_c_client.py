"""The C ABI called from a plain C program (tests/eas_c_client.c): the
header must compile as C, the library must link into a C executable, and a C
caller's spans, forward and backward must match the oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from entropy_active_span_gb300 import _lib
from gpu_helpers import BF16_TOL, small_inputs, rel_fro
from entropy_active_span_gb300 import workloads as W
import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def build_client(out_dir):
    if shutil.which("gcc") is None or not os.path.exists(os.path.join(CUDA, "include",
                                                                        "cuda_runtime_api.h")):
        pytest.skip("gcc or the CUDA runtime headers are missing")
    lib_dir = os.path.dirname(_lib.LIB_PATH)
    cuda_lib = os.path.join(CUDA, "lib64")
    exe = os.path.join(out_dir, "eas_c_client")
    # C11: the CUDA runtime headers use anonymous unions (eas.h alone is C99,
    # test_header_is_pedantic_c99)
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           os.path.join(HERE, "eas_c_client.c"), "-o", exe,
           "-L", lib_dir, "-leas", "-L", cuda_lib, "-lcudart",
           f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{cuda_lib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_header_is_pedantic_c99(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc is missing")
    src = tmp_path / "only_header.c"
    src.write_text('#include "eas.h"\nint main(void) { return eas_version() > 0 ? 0 : 1; }\n')
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-fsyntax-only", "-I", os.path.join(ROOT, "include"), str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_client_host_checks(libeas, tmp_path):
    exe = build_client(str(tmp_path))
    r = subprocess.run([exe, "host"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "host checks ok" in r.stdout


@pytest.mark.gpu
def test_c_client_matches_oracle(libeas, tmp_path):
    T, H, V = 700, 256, 1300
    inp = small_inputs(T, H, V, seed=77, mask_kind="bernoulli0.6", w_std=3.0)
    d = str(tmp_path)
    inp["hidden"].tofile(os.path.join(d, "hidden.bf16"))
    inp["weight"].tofile(os.path.join(d, "weight.bf16"))
    inp["targets"].astype(np.int32).tofile(os.path.join(d, "targets.i32"))
    inp["mask"].astype(np.uint8).tofile(os.path.join(d, "mask.u8"))
    inp["g_logprob"].astype(np.float32).tofile(os.path.join(d, "glp.f32"))
    inp["g_entropy"].astype(np.float32).tofile(os.path.join(d, "gh.f32"))
    exe = build_client(d)
    r = subprocess.run([exe, "run", d, str(T), str(H), str(V)], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr

    def load(name, dt, shape):
        return np.fromfile(os.path.join(d, name), dtype=dt).reshape(shape)

    sp = np.fromfile(os.path.join(d, "spans.i32"), dtype=np.int32)
    np.testing.assert_array_equal(sp[1:].reshape(-1, 2), oracle.active_spans(inp["mask"], 128))
    h64, w64 = W.to_f64(inp["hidden"]), W.to_f64(inp["weight"])
    rlp, rent, rlse = oracle.lmhead_forward(h64, w64, inp["targets"], inp["mask"])
    rdh, rdw = oracle.lmhead_backward(h64, w64, inp["targets"], inp["mask"], inp["g_logprob"],
                                      inp["g_entropy"])
    assert np.max(np.abs(load("logprob.f32", np.float32, T) - rlp)) <= BF16_TOL["lp"]
    assert np.max(np.abs(load("entropy.f32", np.float32, T) - rent)) <= BF16_TOL["ent"]
    assert np.max(np.abs(load("lse.f32", np.float32, T) - rlse)) <= BF16_TOL["lp"]
    dh = W.bf16_bits_to_f32(load("dhidden.bf16", np.uint16, (T, H)))
    assert rel_fro(dh, rdh) <= BF16_TOL["fro"]
    assert np.all(dh[inp["mask"] == 0] == 0)
    assert rel_fro(load("dweight.f32", np.float32, (V, H)), rdw) <= BF16_TOL["fro"]
