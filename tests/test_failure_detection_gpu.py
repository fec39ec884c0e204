"""Failure detection without a GPU fault: every pipeline wait in the GEMM is
bounded.  With the copy-dropping hook of mxfp4_set_debug_options (also set
by MXFP4_DEBUG_DROP_COPIES=1 at load) the generic kernel issues no bulk
copies (the CTA-pair kernel's relay forwards nothing), so the MMA issuer's
wait for its first stage runs out (about a second); the kernel raises the
device-side timeout flag and returns normally.  The host
reads MXFP4_ERR_TIMEOUT from mxfp4_device_status, and the context stays
usable: the next call computes the right result."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import precision_bf16_mxfp4_gb300 as mx
from precision_bf16_mxfp4_gb300 import _lib, inputs
from tests.helpers import assert_close_to_ref, packed_from_oracle
import oracle
from tests.helpers import bf16_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("m,n,k,split", [(8, 256, 1024, "1"), (16, 256, 1024, "4"), (48, 256, 1024, "2"),
                                         (1024, 4864, 256, "1"), (1024, 4864, 2304, "1")])
def test_wait_timeout_is_reported_and_recoverable(m, n, k, split):
    """(1024, 4864, 256) and (1024, 4864, 2304): 152 output tiles of 128 x 256
    select the CTA-pair kernel (one and five stages per tile), whose odd CTAs
    then forward no "stage landed": the even CTAs' MMA waits run out, both
    CTAs of every pair wind down and meet at their final cluster barrier."""
    a = inputs.random_bf16(m, k, seed=m)
    b = inputs.random_bf16(n, k, seed=n, std=0.3)
    packed, bq, bs = packed_from_oracle(b)
    a_dev = a.cuda()
    try:
        mx.set_debug_options(split_k=int(split), drop_copies=True)
        mx.gemm(a_dev, packed)
        with pytest.raises(mx.Mxfp4Error) as e:
            mx.device_status()
        assert e.value.status == _lib.MXFP4_ERR_TIMEOUT
        mx.set_debug_options(split_k=int(split), drop_copies=False)
        mx.device_status()  # the flag was cleared by the previous read
        c = mx.gemm(a_dev, packed)
    finally:
        mx.set_debug_options()
    mx.device_status()
    aq, a_s = oracle.quant(bf16_bits(a))
    assert_close_to_ref(c.float().cpu().numpy(), oracle.gemm_via_dequant(aq, a_s, bq, bs))
