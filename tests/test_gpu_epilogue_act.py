"""The grouped GEMM epilogue's activations, run on the GPU over a dense sweep of
inputs and compared with their exact fp64 definitions.

The epilogue computes GELU with erf from Abramowitz & Stegun 7.1.28 and SwiGLU's
silu(a) * b with the hardware's base-2 exponential and reciprocal; the layer
tests see them only through the bf16 rounding of the hidden activations, so this
test drives the same device code (``csrc/act.cuh``, compiled into a small test
kernel) directly in fp32.

Bounds asserted:
* GELU: |GELU_gpu(u) - GELU(u)| <= 1e-6 on [-20, 20]. The erf formula's error is
  at most 3e-7, which moves u * Phi(u) by at most |u| * 1.5e-7 where Phi(-|u|) is
  not negligible (|u| <~ 6); fp32 rounding of the polynomial, of its 16th power
  and of the reciprocal adds a few 1e-8. Beyond |u| ~ 6 the result is max(u, 0)
  up to Phi(-|u|) < 1e-9.
* SiLU x b: relative error <= (|a| + 8) * 2^-23 of |silu(a) b|. The exponent
  -a log2(e) is rounded to fp32 (relative 2^-24), which e^-a turns into an
  absolute exponent error of |a| 2^-24 and so a relative error of that size; the
  approximate exponential and reciprocal and three roundings add a few ulps.
  Checked for a >= -80; below that 1 + e^-a passes 2^115 and the reciprocal
  nears the flush-to-zero range, so the result lies between 0 and the exact
  value (|silu(a) b| < 1.5e-33 |b| there), which is what is asserted.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch
from scipy.special import erf, expit

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "sparse_expert_ffn_softmax_b300", "csrc")


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    so = str(tmp_path_factory.mktemp("act_probe") / "libact_probe.so")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-shared",
           "-Xcompiler", "-fPIC", f"-I{CSRC}", "-o", so, os.path.join(HERE, "cuda", "act_probe.cu")]
    subprocess.run(cmd, check=True)
    lib = ctypes.CDLL(so)
    lib.act_probe.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_longlong,
                              ctypes.c_void_p]
    lib.act_probe.restype = ctypes.c_int
    return lib


def run(lib, which, a, b=None):
    a_d = torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    b_d = torch.from_numpy(np.ascontiguousarray(b if b is not None else a, np.float32)).cuda()
    out = torch.empty_like(a_d)
    assert a_d.numel() % 2 == 0
    code = lib.act_probe(which, a_d.data_ptr(), b_d.data_ptr(), out.data_ptr(), a_d.numel() // 2,
                         torch.cuda.current_stream().cuda_stream)
    assert code == 0
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def test_gelu_matches_erf_definition(probe):
    u = np.linspace(-20.0, 20.0, 4_000_002).astype(np.float32)
    # every fp32 value in [-1/64, 1/64] around zero's neighbourhood and the largest magnitudes too
    u = np.concatenate([u, np.float32([0.0, -0.0, 1e-30, -1e-30, 5.0, -5.0, 30.0, -30.0])])
    u64 = u.astype(np.float64)
    ref = 0.5 * u64 * (1.0 + erf(u64 / np.sqrt(2.0)))
    got = run(probe, 0, u)
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    assert err.max() <= 1e-6, (err.max(), u[err.argmax()])
    assert got[np.flatnonzero(u == 0.0)].tolist() == [0.0, 0.0]
    print("GELU max abs error", err.max(), "at u =", u[err.argmax()])


def test_silu_times_gate_matches_definition(probe):
    a = np.linspace(-100.0, 100.0, 4_000_000).astype(np.float32)
    rs = np.random.RandomState(0)
    b = rs.standard_normal(a.size).astype(np.float32)
    a64, b64 = a.astype(np.float64), b.astype(np.float64)
    ref = a64 * expit(a64) * b64
    got = run(probe, 1, a, b)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    main = a64 >= -80.0
    bound = (np.abs(a64) + 8.0) * 2.0 ** -23 * np.abs(ref)
    assert np.all(err[main] <= bound[main]), np.max(err[main] / np.maximum(bound[main], 1e-300))
    # far left tail: between zero and the exact value
    assert np.all(err[~main] <= np.abs(ref[~main]) * (1 + 1e-6) + 1e-45)
    nz = main & (ref != 0)
    rel = err[nz] / np.abs(ref[nz])
    print("silu*b max relative error", rel.max(), "at a =", a[nz][rel.argmax()])
