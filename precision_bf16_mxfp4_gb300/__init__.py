"""GB300 (sm_103a) MXFP4 GEMM:  C[m,n] = quant(A) . B^T.

A is bf16 and is quantized on the fly to MXFP4 (e2m1 values, one e8m0 scale
per 32 K elements); B is MXFP4, prepacked once into the tensor-core layout; C
is bf16.  The computation lives in hand-written CUDA kernels behind a C ABI
(include/mxfp4.h, built into _build/libmxfp4.so); this package is the thin
PyTorch-facing binding: it allocates outputs with torch, passes device
pointers and the current stream, and raises on any non-OK status.

    import precision_bf16_mxfp4_gb300 as mx
    bq, bs = mx.quant(b_bf16)                 # MXFP4 weights (linear layout)
    packed = mx.prepack_b(bq, bs)             # one-time repack
    c = mx.gemm(a_bf16, packed, n)            # fused quant + GEMM
"""
from __future__ import annotations

from . import _lib
from ._lib import (  # noqa: F401  (raw C-ABI names)
    Mxfp4Error,
    mxfp4_act_image_bytes,
    mxfp4_device_status,
    mxfp4_gemm,
    mxfp4_gemm_host,
    mxfp4_gemm_image,
    mxfp4_gemm_noalloc,
    mxfp4_gemm_workspace_bytes,
    mxfp4_launch_empty,
    mxfp4_launch_minimal,
    mxfp4_measure_fp4_peak,
    mxfp4_prepack_b,
    mxfp4_prepack_b_bf16,
    mxfp4_prepacked_b_bytes,
    mxfp4_quant,
    mxfp4_kernel_binary_version,
    mxfp4_quant_image,
    mxfp4_set_debug_options,
    mxfp4_status_string,
    mxfp4_version,
)


def _torch():
    import torch
    return torch


def _stream_handle(device):
    torch = _torch()
    return ctypes_void(torch.cuda.current_stream(device).cuda_stream)


def ctypes_void(v):
    import ctypes
    return ctypes.c_void_p(v)


def _check(status: int, where: str):
    if status != _lib.MXFP4_OK:
        raise Mxfp4Error(status, where)


def _require_cuda(t, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")


class PackedB:
    """Prepacked MXFP4 weights: an opaque uint8 device buffer valid for (n, k)."""

    def __init__(self, buf, n: int, k: int):
        self.buf, self.n, self.k = buf, n, k

    @property
    def device(self):
        return self.buf.device


def quant(a, out_q=None, out_scale=None):
    """bf16 [m,k] CUDA tensor -> (fp4x2 uint8 [m,k/2], e8m0 uint8 [m,k/32])."""
    torch = _torch()
    _require_cuda(a, "a")
    if a.dtype != torch.bfloat16 or a.dim() != 2 or a.stride(1) != 1:
        raise ValueError("a must be a 2-D bf16 tensor with unit column stride")
    m, k = a.shape
    q = out_q if out_q is not None else torch.empty((m, k // 2), dtype=torch.uint8, device=a.device)
    s = out_scale if out_scale is not None else torch.empty((m, k // 32), dtype=torch.uint8, device=a.device)
    st = mxfp4_quant(ctypes_void(a.data_ptr()), m, k, a.stride(0), ctypes_void(q.data_ptr()),
                     ctypes_void(s.data_ptr()), _stream_handle(a.device))
    _check(st, "mxfp4_quant")
    return q, s


def prepack_b(b_q, b_scale) -> PackedB:
    """MXFP4 B (fp4x2 uint8 [n,k/2], e8m0 uint8 [n,k/32]) -> PackedB."""
    torch = _torch()
    _require_cuda(b_q, "b_q")
    _require_cuda(b_scale, "b_scale")
    b_q = b_q.contiguous()
    b_scale = b_scale.contiguous()
    n, k = b_q.shape[0], b_q.shape[1] * 2
    if tuple(b_scale.shape) != (n, k // 32):
        raise ValueError("b_scale must be [n, k/32]")
    nbytes = mxfp4_prepacked_b_bytes(n, k)
    if nbytes == 0:
        raise ValueError("unsupported (n, k)")
    buf = torch.empty(nbytes, dtype=torch.uint8, device=b_q.device)
    st = mxfp4_prepack_b(ctypes_void(b_q.data_ptr()), ctypes_void(b_scale.data_ptr()), n, k,
                         ctypes_void(buf.data_ptr()), nbytes, _stream_handle(b_q.device))
    _check(st, "mxfp4_prepack_b")
    return PackedB(buf, n, k)


def prepack_b_bf16(b) -> PackedB:
    """bf16 B [n,k] CUDA tensor -> PackedB in one call (quantized on the
    device with the same rule as A; bit-identical to prepack_b(*quant(b)))."""
    torch = _torch()
    _require_cuda(b, "b")
    if b.dtype != torch.bfloat16 or b.dim() != 2 or b.stride(1) != 1:
        raise ValueError("b must be a 2-D bf16 tensor with unit column stride")
    n, k = b.shape
    nbytes = mxfp4_prepacked_b_bytes(n, k)
    if nbytes == 0:
        raise ValueError("unsupported (n, k)")
    buf = torch.empty(nbytes, dtype=torch.uint8, device=b.device)
    st = mxfp4_prepack_b_bf16(ctypes_void(b.data_ptr()), n, k, b.stride(0), ctypes_void(buf.data_ptr()), nbytes,
                              _stream_handle(b.device))
    _check(st, "mxfp4_prepack_b_bf16")
    return PackedB(buf, n, k)


class ActImage:
    """A quantized activation in the tensor-core operand layout: an opaque
    uint8 device buffer valid for (m, k), reusable by several GEMMs."""

    def __init__(self, buf, m: int, k: int):
        self.buf, self.m, self.k = buf, m, k


def quant_image(a, out=None) -> ActImage:
    """bf16 A [m,k] CUDA tensor -> ActImage (MXFP4, operand layout).

    `out` (optional) is the image buffer to overwrite: an ActImage of the same
    (m, k) or a uint8 device tensor of at least act_image_bytes(m, k) bytes."""
    torch = _torch()
    _require_cuda(a, "a")
    if a.dtype != torch.bfloat16 or a.dim() != 2 or a.stride(1) != 1:
        raise ValueError("a must be a 2-D bf16 tensor with unit column stride")
    m, k = a.shape
    nbytes = mxfp4_act_image_bytes(m, k)
    if nbytes == 0:
        raise ValueError("unsupported (m, k)")
    if isinstance(out, ActImage):
        if (out.m, out.k) != (m, k):
            raise ValueError("out is an image of another (m, k)")
        out = out.buf
    buf = out if out is not None else torch.empty(nbytes, dtype=torch.uint8, device=a.device)
    st = mxfp4_quant_image(ctypes_void(a.data_ptr()), m, k, a.stride(0), ctypes_void(buf.data_ptr()),
                           buf.numel() * buf.element_size(), _stream_handle(a.device))
    _check(st, "mxfp4_quant_image")
    return ActImage(buf, m, k)


def gemm_image(img: ActImage, packed: PackedB, out=None):
    """C = A_image . B^T as bf16 [m, n] for a quantized activation image."""
    torch = _torch()
    if img.k != packed.k:
        raise ValueError("the activation image and packed B disagree on k")
    m, n = img.m, packed.n
    c = out if out is not None else torch.empty((m, n), dtype=torch.bfloat16, device=img.buf.device)
    st = mxfp4_gemm_image(ctypes_void(img.buf.data_ptr()), m, img.k, ctypes_void(packed.buf.data_ptr()), n,
                          ctypes_void(c.data_ptr()), c.stride(0), _stream_handle(img.buf.device))
    _check(st, "mxfp4_gemm_image")
    return c


def workspace_bytes(m: int, n: int, k: int) -> int:
    return mxfp4_gemm_workspace_bytes(m, n, k)


def gemm(a, packed: PackedB, out=None, workspace=None):
    """C = quant(a) . B^T as bf16 [m, n]; `out` and `workspace` may be preallocated."""
    torch = _torch()
    _require_cuda(a, "a")
    if a.dtype != torch.bfloat16 or a.dim() != 2 or a.stride(1) != 1:
        raise ValueError("a must be a 2-D bf16 tensor with unit column stride")
    m, k = a.shape
    if k != packed.k:
        raise ValueError("a and packed B disagree on k")
    n = packed.n
    c = out if out is not None else torch.empty((m, n), dtype=torch.bfloat16, device=a.device)
    need = mxfp4_gemm_workspace_bytes(m, n, k)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=a.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = mxfp4_gemm(ctypes_void(a.data_ptr()), m, k, a.stride(0), ctypes_void(packed.buf.data_ptr()), n,
                    ctypes_void(c.data_ptr()), c.stride(0), ctypes_void(ws_ptr), ws_bytes,
                    _stream_handle(a.device))
    _check(st, "mxfp4_gemm")
    return c


def gemm_host(a_host, packed: PackedB, out=None, a_dev=None, c_dev=None, workspace=None):
    """C = quant(a_host) . B^T for a host-memory A, into host memory, through
    mxfp4_gemm_host, on the current stream of B's device.  With page-locked
    buffers the kernels work on host memory directly, except for the large-m
    CTA-pair plan and the fused plan at k > 512, which copy A up and C down
    through the device staging buffers (in row chunks whose downloads
    overlap the later chunks when C is 8 MiB or more).  `out` (bf16 [m, n],
    host) is created page-locked when not given; the staging buffers and the
    workspace are allocated when not given.  The result is in `out` once the
    stream has passed the call (synchronize before reading it)."""
    torch = _torch()
    if a_host.is_cuda:
        raise ValueError("a_host must be a host tensor (use gemm for device tensors)")
    if a_host.dtype != torch.bfloat16 or a_host.dim() != 2 or a_host.stride(1) != 1:
        raise ValueError("a_host must be a 2-D bf16 tensor with unit column stride")
    m, k = a_host.shape
    if k != packed.k:
        raise ValueError("a_host and packed B disagree on k")
    n, dev = packed.n, packed.buf.device
    n8 = (n + 7) // 8 * 8
    c = out if out is not None else torch.empty((m, n), dtype=torch.bfloat16).pin_memory()
    if c.is_cuda or c.dtype != torch.bfloat16 or c.dim() != 2 or c.stride(1) != 1 or tuple(c.shape) != (m, n):
        raise ValueError("out must be a host bf16 [m, n] tensor with unit column stride")
    if a_dev is None:
        a_dev = torch.empty((m, k), dtype=torch.bfloat16, device=dev)
    if c_dev is None:
        c_dev = torch.empty((m, n8), dtype=torch.bfloat16, device=dev)
    if a_dev.numel() < m * k or c_dev.numel() < m * n8 or not (a_dev.is_cuda and c_dev.is_cuda):
        raise ValueError("a_dev needs m*k and c_dev m*round_up(n, 8) bf16 elements on the device")
    need = mxfp4_gemm_workspace_bytes(m, n, k)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = mxfp4_gemm_host(ctypes_void(a_host.data_ptr()), m, k, a_host.stride(0), ctypes_void(packed.buf.data_ptr()),
                         n, ctypes_void(c.data_ptr()), c.stride(0), ctypes_void(a_dev.data_ptr()),
                         ctypes_void(c_dev.data_ptr()), ctypes_void(ws_ptr), ws_bytes, _stream_handle(dev))
    _check(st, "mxfp4_gemm_host")
    return c


def measure_fp4_peak(kblocks_per_sm: int = 2000, device=None) -> float:
    """Dense block-scaled FP4 tensor-core rate of the device in TFLOP/s,
    measured by mxfp4_measure_fp4_peak (blocks until it has run)."""
    import ctypes
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    out = ctypes.c_double(0.0)
    _check(mxfp4_measure_fp4_peak(int(kblocks_per_sm), ctypes.byref(out), _stream_handle(dev)),
           "mxfp4_measure_fp4_peak")
    return out.value


def launch_empty(count: int = 1, ctas: int = 32, device=None):
    """Enqueue `count` empty kernels on the current stream (the launch floor)."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _check(mxfp4_launch_empty(int(count), int(ctas), _stream_handle(dev)), "mxfp4_launch_empty")


def launch_minimal(count: int = 1, ctas: int = 32, device=None):
    """Enqueue `count` minimal kernels (a global read, a tensor-memory
    allocation, a global write per CTA) on the current stream: the launch
    floor of a tcgen05 GEMM."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _check(mxfp4_launch_minimal(int(count), int(ctas), _stream_handle(dev)), "mxfp4_launch_minimal")


def gemm_noalloc(a, packed: PackedB, out=None):
    """Same as :func:`gemm` through mxfp4_gemm_noalloc: for callers that
    cannot allocate device memory, the scratch comes from an array built into
    the library (8 MiB per device); larger shapes raise Mxfp4Error."""
    torch = _torch()
    _require_cuda(a, "a")
    if a.dtype != torch.bfloat16 or a.dim() != 2 or a.stride(1) != 1:
        raise ValueError("a must be a 2-D bf16 tensor with unit column stride")
    m, k = a.shape
    if k != packed.k:
        raise ValueError("a and packed B disagree on k")
    n = packed.n
    c = out if out is not None else torch.empty((m, n), dtype=torch.bfloat16, device=a.device)
    st = mxfp4_gemm_noalloc(ctypes_void(a.data_ptr()), m, k, a.stride(0), ctypes_void(packed.buf.data_ptr()), n,
                            ctypes_void(c.data_ptr()), c.stride(0), _stream_handle(a.device))
    _check(st, "mxfp4_gemm_noalloc")
    return c


def set_debug_options(split_k: int = 0, drop_copies: bool = False):
    """Testing and tuning overrides: force the K split (0 = the planner's
    choice, else 1, 2, 4 or 8) and make the GEMM kernels drop their operand
    copies so that their bounded waits run out (failure-detection tests)."""
    _check(mxfp4_set_debug_options(int(split_k), 1 if drop_copies else 0), "mxfp4_set_debug_options")


def kernel_binary_version() -> int:
    """binaryVersion of the library's GEMM kernel as loaded on the current
    device (major * 10 + minor: 103 for sm_103a)."""
    import ctypes
    v = ctypes.c_int(0)
    _check(mxfp4_kernel_binary_version(ctypes.byref(v)), "mxfp4_kernel_binary_version")
    return v.value


def device_status(device=None):
    """Synchronize the current stream and raise if a kernel's bounded wait ran out."""
    torch = _torch()
    dev = device if device is not None else torch.cuda.current_device()
    _check(mxfp4_device_status(_stream_handle(dev)), "mxfp4_device_status")
