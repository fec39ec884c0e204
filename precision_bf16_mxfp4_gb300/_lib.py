"""ctypes binding of libmxfp4.so (the C ABI declared in include/mxfp4.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  PyTorch supplies device memory and the current
stream.  If the library is missing or fails to load, every call raises: there
is no CPU or PyTorch fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

MXFP4_OK = 0
MXFP4_ERR_INVALID_ARG = 1
MXFP4_ERR_UNSUPPORTED = 2
MXFP4_ERR_WORKSPACE = 3
MXFP4_ERR_CUDA = 4
MXFP4_ERR_TIMEOUT = 5

EXPORTED = (
    "mxfp4_status_string", "mxfp4_version", "mxfp4_quant", "mxfp4_prepacked_b_bytes", "mxfp4_prepack_b",
    "mxfp4_gemm_workspace_bytes", "mxfp4_gemm", "mxfp4_gemm_noalloc", "mxfp4_device_status",
    "mxfp4_prepack_b_bf16", "mxfp4_act_image_bytes", "mxfp4_quant_image", "mxfp4_gemm_image",
    "mxfp4_gemm_host", "mxfp4_measure_fp4_peak", "mxfp4_launch_empty", "mxfp4_launch_minimal", "mxfp4_set_debug_options",
    "mxfp4_kernel_binary_version",
)

# size of the scratch array compiled into the library for mxfp4_gemm_noalloc
NOALLOC_SCRATCH_BYTES = 8 << 20


class Mxfp4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libmxfp4.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"MXFP4 CUDA library not built: {path}")
        lib = ctypes.CDLL(path)
        p, i64, sz, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
        lib.mxfp4_status_string.argtypes = [i32]
        lib.mxfp4_status_string.restype = ctypes.c_char_p
        lib.mxfp4_version.argtypes = []
        lib.mxfp4_version.restype = i32
        lib.mxfp4_quant.argtypes = [p, i64, i64, i64, p, p, p]
        lib.mxfp4_quant.restype = i32
        lib.mxfp4_prepacked_b_bytes.argtypes = [i64, i64]
        lib.mxfp4_prepacked_b_bytes.restype = sz
        lib.mxfp4_prepack_b.argtypes = [p, p, i64, i64, p, sz, p]
        lib.mxfp4_prepack_b.restype = i32
        lib.mxfp4_gemm_workspace_bytes.argtypes = [i64, i64, i64]
        lib.mxfp4_gemm_workspace_bytes.restype = sz
        lib.mxfp4_gemm.argtypes = [p, i64, i64, i64, p, i64, p, i64, p, sz, p]
        lib.mxfp4_gemm.restype = i32
        lib.mxfp4_gemm_noalloc.argtypes = [p, i64, i64, i64, p, i64, p, i64, p]
        lib.mxfp4_gemm_noalloc.restype = i32
        lib.mxfp4_gemm_host.argtypes = [p, i64, i64, i64, p, i64, p, i64, p, p, p, sz, p]
        lib.mxfp4_gemm_host.restype = i32
        lib.mxfp4_measure_fp4_peak.argtypes = [i64, ctypes.POINTER(ctypes.c_double), p]
        lib.mxfp4_measure_fp4_peak.restype = i32
        lib.mxfp4_launch_empty.argtypes = [ctypes.c_int, ctypes.c_int, p]
        lib.mxfp4_launch_empty.restype = i32
        lib.mxfp4_launch_minimal.argtypes = [ctypes.c_int, ctypes.c_int, p]
        lib.mxfp4_launch_minimal.restype = i32
        lib.mxfp4_set_debug_options.argtypes = [i32, i32]
        lib.mxfp4_set_debug_options.restype = i32
        lib.mxfp4_kernel_binary_version.argtypes = [ctypes.POINTER(ctypes.c_int)]
        lib.mxfp4_kernel_binary_version.restype = i32
        lib.mxfp4_device_status.argtypes = [p]
        lib.mxfp4_device_status.restype = i32
        lib.mxfp4_prepack_b_bf16.argtypes = [p, i64, i64, i64, p, sz, p]
        lib.mxfp4_prepack_b_bf16.restype = i32
        lib.mxfp4_act_image_bytes.argtypes = [i64, i64]
        lib.mxfp4_act_image_bytes.restype = sz
        lib.mxfp4_quant_image.argtypes = [p, i64, i64, i64, p, sz, p]
        lib.mxfp4_quant_image.restype = i32
        lib.mxfp4_gemm_image.argtypes = [p, i64, i64, p, i64, p, i64, p]
        lib.mxfp4_gemm_image.restype = i32
        _lib = lib
        return lib


# ------------------------------------------------------------ raw C ABI (same names)
def mxfp4_status_string(status: int) -> str:
    return load().mxfp4_status_string(int(status)).decode()


status_string = mxfp4_status_string


def mxfp4_version() -> int:
    return int(load().mxfp4_version())


def mxfp4_quant(a_bf16, m, k, lda, a_fp4, a_scale, stream) -> int:
    return int(load().mxfp4_quant(a_bf16, m, k, lda, a_fp4, a_scale, stream))


def mxfp4_prepacked_b_bytes(n, k) -> int:
    return int(load().mxfp4_prepacked_b_bytes(n, k))


def mxfp4_prepack_b(b_fp4, b_scale, n, k, b_packed, b_packed_bytes, stream) -> int:
    return int(load().mxfp4_prepack_b(b_fp4, b_scale, n, k, b_packed, b_packed_bytes, stream))


def mxfp4_gemm_workspace_bytes(m, n, k) -> int:
    return int(load().mxfp4_gemm_workspace_bytes(m, n, k))


def mxfp4_gemm(a_bf16, m, k, lda, b_packed, n, c_bf16, ldc, workspace, workspace_bytes, stream) -> int:
    return int(load().mxfp4_gemm(a_bf16, m, k, lda, b_packed, n, c_bf16, ldc, workspace, workspace_bytes, stream))


def mxfp4_gemm_noalloc(a_bf16, m, k, lda, b_packed, n, c_bf16, ldc, stream) -> int:
    return int(load().mxfp4_gemm_noalloc(a_bf16, m, k, lda, b_packed, n, c_bf16, ldc, stream))


def mxfp4_gemm_host(a_host, m, k, lda, b_packed, n, c_host, ldc, a_dev, c_dev, workspace, workspace_bytes,
                    stream) -> int:
    return int(load().mxfp4_gemm_host(a_host, m, k, lda, b_packed, n, c_host, ldc, a_dev, c_dev, workspace,
                                      workspace_bytes, stream))


def mxfp4_measure_fp4_peak(kblocks_per_sm, tflops, stream) -> int:
    return int(load().mxfp4_measure_fp4_peak(kblocks_per_sm, tflops, stream))


def mxfp4_launch_empty(count, ctas, stream) -> int:
    return int(load().mxfp4_launch_empty(count, ctas, stream))


def mxfp4_launch_minimal(count, ctas, stream) -> int:
    return int(load().mxfp4_launch_minimal(count, ctas, stream))


def mxfp4_set_debug_options(split_k, drop_copies) -> int:
    return int(load().mxfp4_set_debug_options(split_k, drop_copies))


def mxfp4_kernel_binary_version(version) -> int:
    return int(load().mxfp4_kernel_binary_version(version))


def mxfp4_device_status(stream) -> int:
    return int(load().mxfp4_device_status(stream))


def mxfp4_prepack_b_bf16(b_bf16, n, k, ldb, b_packed, b_packed_bytes, stream) -> int:
    return int(load().mxfp4_prepack_b_bf16(b_bf16, n, k, ldb, b_packed, b_packed_bytes, stream))


def mxfp4_act_image_bytes(m, k) -> int:
    return int(load().mxfp4_act_image_bytes(m, k))


def mxfp4_quant_image(a_bf16, m, k, lda, a_image, a_image_bytes, stream) -> int:
    return int(load().mxfp4_quant_image(a_bf16, m, k, lda, a_image, a_image_bytes, stream))


def mxfp4_gemm_image(a_image, m, k, b_packed, n, c_bf16, ldc, stream) -> int:
    return int(load().mxfp4_gemm_image(a_image, m, k, b_packed, n, c_bf16, ldc, stream))
