"""mxfp4_gemm_noalloc: the GEMM entry point for callers that cannot allocate.

Some callers of this library cannot give it device memory: a plugin whose
host interface has no workspace argument, or an engine that committed all
device memory before its first call.  mxfp4_gemm_noalloc serves them from a
scratch array built into the library.  These tests call it through the C ABI
and check, on two calls in a row with different inputs (so a stale scratch
would show), that it returns what mxfp4_gemm returns, within the tolerance
used for the GEMM parity tests.  The file is named to be collected last.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import precision_bf16_mxfp4_gb300 as mx
from precision_bf16_mxfp4_gb300 import _lib, inputs
from tests.helpers import assert_close_to_ref

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p


def _noalloc(a, packed, c):
    stream = P(torch.cuda.current_stream().cuda_stream)
    return _lib.load().mxfp4_gemm_noalloc(P(a.data_ptr()), a.shape[0], a.shape[1], a.stride(0),
                                          P(packed.buf.data_ptr()), packed.n, P(c.data_ptr()), c.stride(0), stream)


@pytest.mark.parametrize("m,n,k", [(64, 7168, 2048), (256, 3072, 1536), (4096, 7168, 2048), (16, 2112, 7168),
                                   (100, 304, 544)])
def test_noalloc_matches_gemm_on_two_calls_in_a_row(m, n, k):
    assert mx.mxfp4_gemm_workspace_bytes(m, n, k) <= _lib.NOALLOC_SCRATCH_BYTES
    b = inputs.random_bf16(n, k, seed=n + k, std=0.05)
    bq, bs = mx.quant(b.cuda())
    packed = mx.prepack_b(bq, bs)
    for call in range(2):
        a = inputs.random_bf16(m, k, seed=1000 * call + m).cuda()
        want = mx.gemm(a, packed)
        c = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(a, packed, c) == _lib.MXFP4_OK
        torch.cuda.synchronize()
        mx.device_status()
        assert_close_to_ref(c.float().cpu().numpy(), want.double().cpu().numpy(), what=f"call {call}")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    m, n, k = 4096, 128, 4096
    assert mx.mxfp4_gemm_workspace_bytes(m, n, k) > _lib.NOALLOC_SCRATCH_BYTES
    a = torch.zeros((m, k), dtype=torch.bfloat16, device="cuda")
    bq = torch.zeros((n, k // 2), dtype=torch.uint8, device="cuda")
    bs = torch.zeros((n, k // 32), dtype=torch.uint8, device="cuda")
    packed = mx.prepack_b(bq, bs)
    c = torch.zeros((m, n), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(a, packed, c) == _lib.MXFP4_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert not c.any()  # nothing was enqueued


def test_noalloc_python_wrapper():
    a = inputs.random_bf16(48, 512, seed=3).cuda()
    b = inputs.random_bf16(640, 512, seed=4).cuda()
    packed = mx.prepack_b(*mx.quant(b))
    got = mx.gemm_noalloc(a, packed)
    want = mx.gemm(a, packed)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got.view(torch.int16).cpu().numpy(), want.view(torch.int16).cpu().numpy())
