"""CPU tests of the C-ABI library: it builds for sm_103a, loads, exports every
symbol include/mxfp4.h declares, and rejects bad arguments before touching a
GPU.  No compute call is made here."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

import precision_bf16_mxfp4_gb300 as mx
from precision_bf16_mxfp4_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxfp4.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mxfp4_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def test_header_declares_the_documented_entry_points():
    names = _declared_functions()
    for required in ("mxfp4_quant", "mxfp4_prepack_b", "mxfp4_gemm", "mxfp4_prepacked_b_bytes",
                     "mxfp4_gemm_workspace_bytes", "mxfp4_status_string", "mxfp4_device_status"):
        assert required in names
    assert set(names) == set(_lib.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\bT\s+(mxfp4_\w+)", out.stdout))
    for name in _declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_library_is_built_for_sm_103a_only():
    # every translation unit and the link get exactly one -gencode, for
    # sm_103a (the GPU tests check the loaded kernel's binaryVersion)
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert not any("arch" in f or "gencode" in f for f in build.FLAGS)


def test_debug_options_reject_values_outside_their_sets(lib):
    assert mx.mxfp4_set_debug_options(-1, 0) == _lib.MXFP4_ERR_INVALID_ARG
    assert mx.mxfp4_set_debug_options(0, 2) == _lib.MXFP4_ERR_INVALID_ARG
    assert mx.mxfp4_set_debug_options(9, 0) == _lib.MXFP4_ERR_INVALID_ARG
    for s in range(9):
        assert mx.mxfp4_set_debug_options(s, 0) == _lib.MXFP4_OK
    assert mx.mxfp4_set_debug_options(0, 0) == _lib.MXFP4_OK


def test_binary_version_rejects_a_null_pointer(lib):
    assert mx.mxfp4_kernel_binary_version(None) == _lib.MXFP4_ERR_INVALID_ARG


def test_status_strings_and_version(lib):
    assert mx.mxfp4_status_string(0) == "MXFP4_OK"
    assert mx.mxfp4_status_string(5) == "MXFP4_ERR_TIMEOUT"
    assert mx.mxfp4_status_string(99) == "MXFP4_ERR_UNKNOWN"
    assert mx.mxfp4_version() >= 100


def _image_bytes(rows, k):
    return -(-rows // 128) * -(-k // 256) * (16384 + 1024)


@pytest.mark.parametrize("n,k", [(2880, 512), (2112, 7168), (1, 32), (129, 288), (7168, 2048)])
def test_prepacked_size(n, k):
    assert mx.mxfp4_prepacked_b_bytes(n, k) == _image_bytes(n, k)


def test_prepacked_size_rejects_bad_shapes():
    assert mx.mxfp4_prepacked_b_bytes(0, 512) == 0
    assert mx.mxfp4_prepacked_b_bytes(16, 48) == 0
    assert mx.mxfp4_prepacked_b_bytes(16, -32) == 0


@pytest.mark.parametrize("m,n,k", [(4, 2880, 512), (32, 4096, 512), (16, 2112, 7168), (1, 1, 32)])
def test_small_m_needs_no_workspace(m, n, k):
    assert mx.mxfp4_gemm_workspace_bytes(m, n, k) == 0


@pytest.mark.parametrize("m,n,k", [(64, 7168, 2048), (33, 100, 64), (256, 3072, 1536), (4096, 7168, 2048),
                                   (65, 8, 32)])
def test_large_m_workspace_is_the_activation_image(m, n, k):
    assert mx.mxfp4_gemm_workspace_bytes(m, n, k) == _image_bytes(m, k)


P = ctypes.c_void_p


def test_gemm_rejects_bad_arguments_without_a_gpu():
    fake = P(0x10000)  # aligned, never dereferenced: validation fails first
    E = _lib.MXFP4_ERR_INVALID_ARG
    assert mx.mxfp4_gemm(fake, 4, 48, 48, fake, 16, fake, 16, None, 0, None) == E       # k % 32
    assert mx.mxfp4_gemm(fake, 0, 64, 64, fake, 16, fake, 16, None, 0, None) == E       # m == 0
    assert mx.mxfp4_gemm(fake, 4, 64, 32, fake, 16, fake, 16, None, 0, None) == E       # lda < k
    assert mx.mxfp4_gemm(fake, 4, 64, 68, fake, 16, fake, 16, None, 0, None) == E       # lda % 8
    assert mx.mxfp4_gemm(fake, 4, 64, 64, fake, 16, fake, 12, None, 0, None) == E       # ldc < n
    assert mx.mxfp4_gemm(None, 4, 64, 64, fake, 16, fake, 16, None, 0, None) == E       # null A
    assert mx.mxfp4_gemm(P(0x10008), 4, 64, 64, fake, 16, fake, 16, None, 0, None) == E  # unaligned A
    assert mx.mxfp4_gemm(fake, 256, 64, 64, fake, 16, fake, 16, None, 0, None) == _lib.MXFP4_ERR_WORKSPACE
    assert mx.mxfp4_gemm(fake, 33, 64, 64, fake, 16, fake, 16, fake, 100, None) == _lib.MXFP4_ERR_WORKSPACE


def test_quant_and_prepack_reject_bad_arguments_without_a_gpu():
    fake = P(0x10000)
    E = _lib.MXFP4_ERR_INVALID_ARG
    assert mx.mxfp4_quant(fake, 4, 40, 40, fake, fake, None) == E
    assert mx.mxfp4_quant(fake, -1, 64, 64, fake, fake, None) == E
    assert mx.mxfp4_quant(fake, 0, 64, 64, fake, fake, None) == _lib.MXFP4_OK  # empty is a no-op
    assert mx.mxfp4_prepack_b(fake, fake, 16, 64, fake, 10, None) == E          # buffer too small
    assert mx.mxfp4_prepack_b(fake, fake, 0, 64, fake, 1 << 20, None) == E


@pytest.mark.parametrize("m,k", [(4, 512), (33, 64), (4096, 2048), (129, 288)])
def test_act_image_size(m, k):
    assert mx.mxfp4_act_image_bytes(m, k) == _image_bytes(m, k)
    assert mx.mxfp4_act_image_bytes(0, k) == 0
    assert mx.mxfp4_act_image_bytes(m, 48) == 0


def test_image_entry_points_reject_bad_arguments_without_a_gpu():
    fake = P(0x10000)
    E = _lib.MXFP4_ERR_INVALID_ARG
    big = 1 << 30
    assert mx.mxfp4_prepack_b_bf16(fake, 16, 64, 32, fake, big, None) == E           # ldb < k
    assert mx.mxfp4_prepack_b_bf16(fake, 16, 64, 68, fake, big, None) == E           # ldb % 8
    assert mx.mxfp4_prepack_b_bf16(fake, 16, 48, 48, fake, big, None) == E           # k % 32
    assert mx.mxfp4_prepack_b_bf16(fake, 16, 64, 64, fake, 10, None) == E            # buffer too small
    assert mx.mxfp4_prepack_b_bf16(P(0x10008), 16, 64, 64, fake, big, None) == E     # unaligned B
    assert mx.mxfp4_quant_image(fake, 0, 64, 64, fake, big, None) == E               # m == 0
    assert mx.mxfp4_quant_image(fake, 4, 64, 64, fake, 10, None) == E                # image too small
    assert mx.mxfp4_quant_image(None, 4, 64, 64, fake, big, None) == E               # null A
    assert mx.mxfp4_gemm_image(fake, 4, 64, fake, 16, fake, 12, None) == E           # ldc < n
    assert mx.mxfp4_gemm_image(fake, 4, 48, fake, 16, fake, 16, None) == E           # k % 32
    assert mx.mxfp4_gemm_image(None, 4, 64, fake, 16, fake, 16, None) == E           # null image
    assert mx.mxfp4_gemm_image(fake, 4, 64, fake, 16, P(0x10008), 16, None) == E     # unaligned C


def test_host_entry_point_rejects_bad_arguments_without_a_gpu():
    fake = P(0x10000)  # never dereferenced: every check runs before the first copy is enqueued
    E = _lib.MXFP4_ERR_INVALID_ARG
    args = dict(a=fake, m=4, k=64, lda=64, b=fake, n=16, c=fake, ldc=16, ad=fake, cd=fake, ws=None, wsb=0)

    def call(**kw):
        a = {**args, **kw}
        return mx.mxfp4_gemm_host(a["a"], a["m"], a["k"], a["lda"], a["b"], a["n"], a["c"], a["ldc"], a["ad"],
                                  a["cd"], a["ws"], a["wsb"], None)

    assert call(k=48, lda=48) == E                  # k % 32
    assert call(m=0) == E                           # m == 0
    assert call(lda=32) == E                        # lda < k
    assert call(ldc=12) == E                        # ldc < n
    assert call(a=None) == E                        # null host A
    assert call(c=None) == E                        # null host C
    assert call(ad=P(0x10008)) == E                 # unaligned device staging
    assert call(b=P(0x10008)) == E                  # unaligned packed B
    assert call(m=256) == _lib.MXFP4_ERR_WORKSPACE  # the GEMM's workspace is checked before any copy
    # host rows need no alignment: an odd host stride passes validation (only
    # the workspace check then stops this fake call)
    assert call(m=256, lda=67) == _lib.MXFP4_ERR_WORKSPACE


def test_fp4_peak_rejects_bad_arguments_without_a_gpu():
    import ctypes
    out = ctypes.c_double(0.0)
    E = _lib.MXFP4_ERR_INVALID_ARG
    assert mx.mxfp4_measure_fp4_peak(0, ctypes.byref(out), None) == E
    assert mx.mxfp4_measure_fp4_peak(1 << 25, ctypes.byref(out), None) == E
    assert mx.mxfp4_measure_fp4_peak(100, None, None) == E


def test_launch_empty_rejects_bad_arguments_without_a_gpu():
    E = _lib.MXFP4_ERR_INVALID_ARG
    assert mx.mxfp4_launch_empty(0, 32, None) == E
    assert mx.mxfp4_launch_empty(17, 32, None) == E
    assert mx.mxfp4_launch_empty(1, 0, None) == E
    assert mx.mxfp4_launch_minimal(0, 32, None) == E
    assert mx.mxfp4_launch_minimal(17, 32, None) == E
    assert mx.mxfp4_launch_minimal(1, 0, None) == E
    assert mx.mxfp4_launch_minimal(1, 65536, None) == E


def test_product_path_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "precision_bf16_mxfp4_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.replace("the oracle", "").lower() or f == "inputs.py", f
