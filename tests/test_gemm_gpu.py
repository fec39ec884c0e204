"""GPU parity of mxfp4_gemm against the fp64 oracle.

C must satisfy |C - ref| <= 2^-7 |ref| + 1e-3 max|ref| everywhere the oracle
is evaluated; quantized A inside the fused kernel is checked bit-exactly
through an identity-B product, which makes C equal dequant(quant(A)).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import precision_bf16_mxfp4_gb300 as mx
from precision_bf16_mxfp4_gb300 import inputs
from tests.helpers import assert_close_to_ref, bf16_bits, packed_from_oracle

pytestmark = pytest.mark.gpu


def _run(a_cpu, packed, lda=None, ldc=None, poison=True):
    m, k = a_cpu.shape
    n = packed.n
    if lda is not None and lda != k:
        big = torch.zeros((m, lda), dtype=torch.bfloat16)
        big[:, :k] = a_cpu
        a_dev = big.cuda()[:, :k]
    else:
        a_dev = a_cpu.cuda()
    ldc = ldc or n
    c_full = torch.full((m, ldc), float("nan") if poison else 0.0, dtype=torch.bfloat16, device="cuda")
    c = c_full[:, :n]
    mx.gemm(a_dev, packed, out=c)
    mx.device_status()
    return c.float().cpu().numpy(), c_full


def _oracle_full(a_cpu, bq, bs):
    aq, a_s = oracle.quant(bf16_bits(a_cpu))
    return oracle.gemm_via_dequant(aq, a_s, bq, bs)


SMALL_FULL = ["m4_n2880_k512", "m32_n4096_k512", "m32_n2880_k512", "m16_n2112_k7168", "m64_n7168_k2048",
              "m256_n3072_k1536"]


@pytest.mark.parametrize("name", SMALL_FULL)
def test_gemm_workload_full_output(name):
    a, b = inputs.make_inputs(name)
    packed, bq, bs = packed_from_oracle(b)
    got, _ = _run(a, packed)
    ref = _oracle_full(a, bq, bs)
    assert_close_to_ref(got, ref, what=name)


@pytest.mark.parametrize("name", list(inputs.TEST_SHAPES))
def test_gemm_page_test_shapes_full_output(name):
    a, b = inputs.make_inputs(name)
    packed, bq, bs = packed_from_oracle(b)
    got, _ = _run(a, packed)
    assert_close_to_ref(got, _oracle_full(a, bq, bs), what=name)


def test_gemm_large_workload_full_output():
    """m=4096, n=7168, k=2048 (quantizer kernel + CTA-pair GEMM): all 29.4 M
    outputs against the oracle's definition (fp64 products of the dequantized
    values, summed by the library matmul), C poisoned with NaN beforehand;
    a few entries also against the plain oracle loop."""
    name = "m4096_n7168_k2048"
    a, b = inputs.make_inputs(name)
    packed, bq, bs = packed_from_oracle(b)
    got, _ = _run(a, packed, poison=True)
    aq, a_s = oracle.quant(bf16_bits(a))
    ref = oracle.gemm_via_dequant(aq, a_s, bq, bs)
    assert_close_to_ref(got, ref, what=name)
    rows = np.array([0, 127, 128, 255, 256, 4095, 2047, 3000])
    cols = np.array([0, 255, 256, 7167, 128, 129, 4000, 6143])
    np.testing.assert_allclose(oracle.gemm_entries(aq, a_s, bq, bs, rows, cols), ref[rows, cols], rtol=1e-12)


LARGEST = [
    (32768, 7168, 2048),  # CTA-pair kernel, 3584 tiles: 47 rounds per pair
    (2048, 4096, 16384),  # CTA-pair kernel, 32 stages per tile
    (8, 2112, 65536),     # fused kernel, K split over 8-CTA clusters, 32 K blocks per rank
    (8, 7168, 65536),     # fused kernel, 2 ranks (56 column tiles fill the SMs), 128 K blocks per rank
    (64, 65536, 2048),    # quantizer + image swap-AB, 512 CTAs in several waves
    (32, 65536, 512),     # fused kernel unsplit, 512 CTAs in several waves
    (256, 1024, 32768),   # quantizer + image plain, K split over 8-CTA clusters
]


@pytest.mark.parametrize("m,n,k", LARGEST)
def test_gemm_largest_shapes_sampled(m, n, k):
    """Shapes far beyond the benchmark's, on every plan: C poisoned with NaN
    must come back finite everywhere, and sampled entries (the last whole
    column, 2000 random positions, and the first and last whole rows where
    the oracle's budget of ~1.5e8 multiply-adds allows) must match the
    oracle.  B is a random valid MXFP4 matrix (every e2m1 code, scales
    2^-9..2^9): quantizing a bf16 B of this size in the oracle would take
    minutes."""
    rng = np.random.default_rng(m * 131 + n * 7 + k)
    bq = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    bs = rng.integers(118, 137, (n, k // 32), dtype=np.uint8)
    packed = mx.prepack_b(torch.from_numpy(bq).cuda(), torch.from_numpy(bs).cuda())
    a = inputs.random_bf16(m, k, seed=m + n + k)
    c = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    mx.gemm(a.cuda(), packed, out=c)
    mx.device_status()
    assert not torch.isnan(c).any().item(), "entries of C were not written"
    rows = [np.arange(m, dtype=np.int64), rng.integers(0, m, 2000)]
    cols = [np.full(m, n - 1, np.int64), rng.integers(0, n, 2000)]
    budget = int(1.5e8 // k) - m - 2000
    for r in (0, m - 1):
        if budget >= n:
            rows.append(np.full(n, r, np.int64))
            cols.append(np.arange(n, dtype=np.int64))
            budget -= n
    rows, cols = np.concatenate(rows), np.concatenate(cols)
    got = c[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].float().cpu().numpy()
    aq, a_s = oracle.quant(bf16_bits(a))
    ref = oracle.gemm_entries(aq, a_s, bq, bs, rows, cols)
    assert_close_to_ref(got, ref, what=f"{m}x{n}x{k}")


def _selection_weights(n, k, cols):
    """MXFP4 weights whose row j is 1.0 at K column cols[j] (no entry where
    cols[j] < 0) and zero elsewhere, every scale 2^0: row j of B^T picks
    column cols[j] of dequant(quant(A)), so C shows each quantized element."""
    bq = np.zeros((n, k // 2), np.uint8)
    for j, c in enumerate(cols):
        if 0 <= c < k:
            bq[j, c // 2] = 0x2 if c % 2 == 0 else 0x20  # code 2 = 1.0
    bs = np.full((n, k // 32), 127, np.uint8)
    return bq, bs


def _quantized_a(a):
    aq, a_s = oracle.quant(bf16_bits(a))
    return torch.from_numpy(oracle.dequant(aq, a_s)).to(torch.bfloat16).float().numpy()


def test_fused_split4_quantizer_bit_exact_at_k7168():
    """m=16, n=2112, k=7168 with the wide-exponent, zero-block activation of
    that workload: the fused kernel with BN = 16 (two quantizer groups taking
    a stage's K blocks in turn), K split over 4-CTA clusters.  Four launches
    whose weights select K columns j + 2112 r make every quantized element of
    A appear in C exactly."""
    a, _ = inputs.make_inputs("m16_n2112_k7168")
    m, k, n = 16, 7168, 2112
    want = _quantized_a(a)
    for r in range(4):
        cols = [j + n * r for j in range(n)]
        bq, bs = _selection_weights(n, k, cols)
        packed = mx.prepack_b(torch.from_numpy(bq).cuda(), torch.from_numpy(bs).cuda())
        got, _ = _run(a, packed)
        for j, c in enumerate(cols):
            if c < k:
                np.testing.assert_array_equal(got[:, j], want[:, c], err_msg=f"column {c}")
            else:
                assert not np.any(got[:, j])


@pytest.mark.parametrize("m", [64, 4096])
def test_image_quantizer_bit_exact_at_k2048(m):
    """k=2048 through the activation-image path: m=64 on the swap-AB image
    kernel (BN = 64), m=4096 (the large workload's activation) on the CTA-pair
    kernel; an identity weight (n = k) makes C = dequant(quant(A)) exactly."""
    k = n = 2048
    a = inputs.make_inputs("m4096_n7168_k2048")[0][:m] if m == 4096 else inputs.make_inputs("m64_n7168_k2048")[0]
    bq, bs = _selection_weights(n, k, list(range(n)))
    packed = mx.prepack_b(torch.from_numpy(bq).cuda(), torch.from_numpy(bs).cuda())
    got, _ = _run(a.contiguous(), packed)
    np.testing.assert_array_equal(got, _quantized_a(a))


@pytest.mark.parametrize("m,n,k,ldb", [(32, 2880, 512, 512), (16, 2112, 7168, 7168), (256, 1500, 2336, 2344),
                                       (64, 7168, 2048, 2048)])
def test_prepack_b_bf16_then_gemm_matches_the_oracle(m, n, k, ldb):
    """The one-call weight path (bf16 B -> prepacked image on the device)
    followed by mxfp4_gemm, against the oracle's quantization of the same B
    and the oracle's GEMM."""
    a = inputs.random_bf16(m, k, seed=m + k)
    big = torch.zeros((n, ldb), dtype=torch.bfloat16)
    big[:, :k] = inputs.random_bf16(n, k, seed=n + 7 * k, std=0.05)
    packed = mx.prepack_b_bf16(big.cuda()[:, :k])
    got, _ = _run(a, packed, ldc=(n + 7) // 8 * 8)
    bq, bs = oracle.quant(bf16_bits(big[:, :k]))
    assert_close_to_ref(got, _oracle_full(a, bq, bs), what=f"{m}x{n}x{k}")


@pytest.mark.parametrize("m", [1, 4, 16, 17, 32, 64, 65, 200, 256])
def test_fused_and_image_quant_bit_exact_through_identity(m):
    """B = identity (code 1.0, scale 2^0): C[i, j] = dequant(quant(A))[i, j]
    exactly, so every in-kernel quantized element is visible in C."""
    k = 512
    n = k
    bq = np.zeros((n, k // 2), np.uint8)
    for j in range(n):
        bq[j, j // 2] = 0x2 if j % 2 == 0 else 0x20
    bs = np.full((n, k // 32), 127, np.uint8)
    packed = mx.prepack_b(torch.from_numpy(bq).cuda(), torch.from_numpy(bs).cuda())
    a = inputs.random_bf16(m, k, seed=100 + m, std=2.0)
    got, _ = _run(a, packed)
    aq, a_s = oracle.quant(bf16_bits(a))
    want = torch.from_numpy(oracle.dequant(aq, a_s)).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(got, want)


RAGGED = [(1, 1, 32), (3, 100, 96), (4, 129, 288), (16, 300, 544), (17, 128, 256), (33, 257, 160),
          (64, 1000, 2080), (65, 131, 96), (130, 260, 544), (200, 520, 1024), (384, 384, 256)]


@pytest.mark.parametrize("m,n,k", RAGGED)
def test_gemm_ragged_shapes_with_padded_strides(m, n, k):
    a = inputs.random_bf16(m, k, seed=m * 7 + n * 3 + k)
    b = inputs.random_bf16(n, k, seed=m + n + k, std=0.5)
    packed, bq, bs = packed_from_oracle(b)
    lda = k + 8 * ((m % 3) + 1)
    ldc = n + (8 - n % 8) % 8 + 8
    got, c_full = _run(a, packed, lda=lda, ldc=ldc)
    assert_close_to_ref(got, _oracle_full(a, bq, bs), what=f"{m}x{n}x{k}")
    assert torch.isnan(c_full[:, n:]).all(), "wrote outside the [m, n] window"


def _random_shapes(count=40, seed=20261202, budget=3e9):
    """A fixed, seeded spread of (m, n, k) over every plan of the library:
    fused (m <= 32, with and without a K split), image swap (m <= 128),
    image plain and the CTA-pair kernel (many 256 x 256 tiles), each with an
    oracle cost below `budget` multiply-adds."""
    rng = np.random.default_rng(seed)
    out = []
    bands = [(1, 32), (33, 128), (129, 640), (641, 2200)]
    while len(out) < count:
        band = len(out) % len(bands)
        lo, hi = bands[band]
        m = int(rng.integers(lo, hi + 1))
        if band == 3:  # enough 256 x 256 tiles for the CTA-pair plan
            n_min = -(-152 // -(-m // 256)) * 256 - 255
            n = int(rng.integers(n_min, n_min + 2000))
        else:
            n = int(rng.integers(1, 5200))
        k_max = min(120, int(budget // (m * n * 32)))
        if k_max < 1:
            continue
        out.append((m, n, 32 * int(rng.integers(1, k_max + 1))))
    return out


RANDOM_SHAPES = _random_shapes()


@pytest.mark.parametrize("m,n,k", RANDOM_SHAPES)
def test_gemm_random_shapes_sweep(m, n, k):
    # a seeded sweep of shapes with odd sizes everywhere, padded strides and a
    # NaN-poisoned C: every plan the library has, against the fp64 oracle
    a = inputs.random_bf16(m, k, seed=m + 31 * n + 7 * k)
    b = inputs.random_bf16(n, k, seed=3 * m + n + k, std=0.3)
    packed, bq, bs = packed_from_oracle(b)
    lda = k + 8 * (n % 3)
    ldc = n + (8 - n % 8) % 8 + 8 * (m % 2)
    got, c_full = _run(a, packed, lda=lda, ldc=ldc)
    assert_close_to_ref(got, _oracle_full(a, bq, bs), what=f"{m}x{n}x{k}")
    if ldc > n:
        assert torch.isnan(c_full[:, n:]).all(), "wrote outside the [m, n] window"


def test_random_shapes_cover_every_plan():
    # the sweep above reaches the fused, split, image and CTA-pair plans
    sms = 152
    kinds = set()
    for m, n, k in RANDOM_SHAPES:
        if m <= 32:
            kinds.add("fused")
        elif m <= 128:
            kinds.add("image swap")
        elif n >= 256 and -(-m // 128) * -(-n // 256) >= sms:
            kinds.add("pair")
        else:
            kinds.add("image plain")
    assert kinds == {"fused", "image swap", "image plain", "pair"}, kinds


# the last two have a C of at least 8 MiB: the chunked round trip (4 chunks
# of 256 rows; 512, 512 and a ragged 76)
HOST_CASES = [(32, 2880, 512), (4, 129, 288), (17, 136, 1024), (16, 640, 7168), (64, 2000, 2048), (200, 1003, 544),
              (1024, 4864, 256), (1100, 4856, 512)]


@pytest.mark.parametrize("m,n,k", HOST_CASES)
@pytest.mark.parametrize("layout", ["aligned", "odd_strides", "pageable"])
def test_gemm_host_round_trip(m, n, k, layout):
    # C lands in a wider NaN-filled host buffer, equal bit for bit to the
    # device call, with nothing outside the [m, n] window written.  Aligned
    # page-locked rows let every plan but the CTA-pair one and the fused one
    # at k > 512 work on host memory directly; row strides that are not
    # multiples of 8 elements, or pageable memory, take the copies through
    # the device staging buffers.
    a = inputs.random_bf16(m, k, seed=m + 3 * n + 5 * k)
    b = inputs.random_bf16(n, k, seed=n + k, std=0.5)
    packed, bq, bs = packed_from_oracle(b)
    n8 = (n + 7) // 8 * 8
    lda, ldc = (k + 5, n + 3) if layout == "odd_strides" else (k + 8, n8 + 8)
    pin = (lambda t: t) if layout == "pageable" else (lambda t: t.pin_memory())
    a_big = pin(torch.zeros((m, lda), dtype=torch.bfloat16))
    a_big[:, :k] = a
    c_big = pin(torch.full((m, ldc), float("nan"), dtype=torch.bfloat16))
    out = mx.gemm_host(a_big[:, :k], packed, out=c_big[:, :n])
    torch.cuda.synchronize()
    mx.device_status()
    want = torch.empty((m, n8), dtype=torch.bfloat16, device="cuda")[:, :n]  # ldc % 8 == 0
    want = mx.gemm(a.cuda(), packed, out=want).cpu()
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))
    assert torch.isnan(c_big[:, n:]).all(), "wrote outside the [m, n] window"
    assert_close_to_ref(out.float().numpy(), _oracle_full(a, bq, bs), what=f"{m}x{n}x{k}")


def test_gemm_host_reuses_its_buffers_across_calls():
    # the same host buffers, staging and workspace through several calls in a row
    m, n, k = 32, 2880, 512
    a1, a2 = inputs.random_bf16(m, k, seed=1), inputs.random_bf16(m, k, seed=2)
    packed, _, _ = packed_from_oracle(inputs.random_bf16(n, k, seed=3))
    a_host = torch.empty((m, k), dtype=torch.bfloat16).pin_memory()
    c_host = torch.empty((m, n), dtype=torch.bfloat16).pin_memory()
    a_dev = torch.empty((m, k), dtype=torch.bfloat16, device="cuda")
    c_dev = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    for a in (a1, a2, a1):
        a_host.copy_(a)
        mx.gemm_host(a_host, packed, out=c_host, a_dev=a_dev, c_dev=c_dev)
        torch.cuda.synchronize()
        want = mx.gemm(a.cuda(), packed).cpu()
        assert torch.equal(c_host.view(torch.int16), want.view(torch.int16))


def test_gemm_host_chunked_round_trip_in_a_captured_cuda_graph():
    # the chunked form forks its downloads onto the library's helper stream
    # and joins them back; captured (after an uncaptured call made the helper
    # stream) and replayed with new A, it must give the device call's C
    m, n, k = 1024, 4864, 512
    packed, _, _ = packed_from_oracle(inputs.random_bf16(n, k, seed=7))
    a_host = inputs.random_bf16(m, k, seed=8).pin_memory()
    c_host = torch.empty((m, n), dtype=torch.bfloat16).pin_memory()
    a_dev = torch.empty((m, k), dtype=torch.bfloat16, device="cuda")
    c_dev = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(mx.workspace_bytes(m, n, k), 16), dtype=torch.uint8, device="cuda")
    call = lambda: mx.gemm_host(a_host, packed, out=c_host, a_dev=a_dev, c_dev=c_dev, workspace=ws)
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    torch.cuda.synchronize()
    for seed in (9, 10):
        a = inputs.random_bf16(m, k, seed=seed)
        a_host.copy_(a)
        c_host.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        want = mx.gemm(a.cuda(), packed).cpu()
        assert torch.equal(c_host.view(torch.int16), want.view(torch.int16))
    mx.device_status()


def test_gemm_deterministic_and_reusable_workspace():
    for name in ("m16_n2112_k7168", "m256_n3072_k1536"):
        a, b = inputs.make_inputs(name)
        packed, _, _ = packed_from_oracle(b)
        a_dev = a.cuda()
        ws_bytes = mx.workspace_bytes(*a.shape[:1], packed.n, a.shape[1])
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda") if ws_bytes else None
        c1 = mx.gemm(a_dev, packed, workspace=ws)
        c2 = mx.gemm(a_dev, packed, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


def test_gemm_on_a_side_stream_matches():
    a, b = inputs.make_inputs("m32_n2880_k512")
    packed, bq, bs = packed_from_oracle(b)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c = mx.gemm(a.cuda(), packed)
    s.synchronize()
    assert_close_to_ref(c.float().cpu().numpy(), _oracle_full(a, bq, bs))


def test_gemm_from_several_host_threads():
    # the entry points are reentrant: four host threads, each on its own
    # stream, run the fused, split, image and CTA-pair plans at once and get
    # what a single thread gets
    import threading
    shapes = [(32, 2880, 512), (16, 2112, 7168), (256, 3072, 1536), (1024, 4864, 256)]
    cases = []
    for i, (m, n, k) in enumerate(shapes):
        a = inputs.random_bf16(m, k, seed=100 + i).cuda()
        packed, _, _ = packed_from_oracle(inputs.random_bf16(n, k, seed=200 + i, std=0.5))
        cases.append((a, packed, mx.gemm(a, packed)))
    torch.cuda.synchronize()
    errors = []

    def worker(a, packed, want):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(5):
                    got = mx.gemm(a, packed)
                    s.synchronize()
                    if not torch.equal(got.view(torch.int16), want.view(torch.int16)):
                        errors.append("mismatch")
        except Exception as e:  # surfaced below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=c) for c in cases]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    mx.device_status()


def test_fp4_peak_microbenchmark_is_plausible():
    # a dense FP4 rate between a tenth of NVIDIA's nominal 13.5 PFLOP/s and
    # a little above it, and roughly proportional to the work asked for
    small, big = mx.measure_fp4_peak(500), mx.measure_fp4_peak(4000)
    assert 1350.0 < big < 15000.0, big
    assert small < big * 1.2
    mx.device_status()


def test_launch_floor_kernels_run():
    mx.launch_empty(2, 32)
    # more CTAs than the SMs' tensor memory can hold at 32 columns each at
    # once: allocations wait for other CTAs' frees, which always come
    mx.launch_minimal(2, 32)
    mx.launch_minimal(1, 4096)
    torch.cuda.synchronize()
    mx.device_status()


def test_gemm_reports_small_workspace():
    a = inputs.random_bf16(256, 512, seed=1).cuda()
    b = inputs.random_bf16(128, 512, seed=2)
    packed, _, _ = packed_from_oracle(b)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(mx.Mxfp4Error) as e:
        mx.gemm(a, packed, workspace=ws)
    assert e.value.status == 3


def test_prepack_roundtrip_through_gemm_columns():
    """Each weight row j reappears as column j of C when A = one-hot rows."""
    n, k = 300, 544
    b = inputs.random_bf16(n, k, seed=9)
    packed, bq, bs = packed_from_oracle(b)
    m = 8
    a = torch.zeros((m, k), dtype=torch.bfloat16)
    picks = [0, 1, 31, 32, 255, 256, 288, 543]
    for i, p in enumerate(picks):
        a[i, p] = 1.0
    got, _ = _run(a, packed, ldc=304)
    deq_b = oracle.dequant(bq, bs)
    want = torch.from_numpy(deq_b[:, picks].T.copy()).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(got, want)


SPLIT_CASES = [(4, 256, 1024), (16, 300, 2048), (32, 520, 2080), (64, 384, 2048), (200, 256, 2048)]


@pytest.fixture
def forced_split():
    """Set the planner's K split through mxfp4_set_debug_options; restored after the test."""
    yield lambda s: mx.set_debug_options(split_k=s)
    mx.set_debug_options(split_k=0)


@pytest.mark.parametrize("split", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("m,n,k", SPLIT_CASES)
def test_gemm_every_split_factor(m, n, k, split, forced_split):
    """The planner's K split is overridden (mxfp4_set_debug_options) to run
    every cluster size through the reduce-scatter epilogue: owners of 16
    rows (split 8) and uneven owners (splits 3, 5, 6, 7: 42-43, 25-26, 21-22
    and 18-19 rows)."""
    forced_split(split)
    a = inputs.random_bf16(m, k, seed=m + split)
    b = inputs.random_bf16(n, k, seed=n + split, std=0.3)
    packed, bq, bs = packed_from_oracle(b)
    ldc = n + (8 - n % 8) % 8
    got, c_full = _run(a, packed, ldc=ldc)
    assert_close_to_ref(got, _oracle_full(a, bq, bs), what=f"split {split}")
    a_dev = a.cuda()
    c1 = mx.gemm(a_dev, packed, out=torch.empty((m, ldc), dtype=torch.bfloat16, device="cuda")[:, :n])
    c2 = mx.gemm(a_dev, packed, out=torch.empty((m, ldc), dtype=torch.bfloat16, device="cuda")[:, :n])
    torch.cuda.synchronize()
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


@pytest.mark.parametrize("n,k,ldb", [(300, 544, 544), (2880, 512, 512), (129, 288, 288), (2112, 7168, 7168),
                                     (1500, 2336, 2344)])
def test_prepack_b_bf16_equals_quant_then_prepack(n, k, ldb):
    """The one-call weight path writes the same image bytes as mxfp4_quant
    followed by mxfp4_prepack_b (padding rows and the K tail zero); 1500 x
    2336 with a row stride of 2344 ends in a K block of 32 and 36 padding
    rows."""
    big = torch.full((n, ldb), float("nan"), dtype=torch.bfloat16)
    big[:, :k] = inputs.random_bf16(n, k, seed=n + k, std=0.5)
    b = big.cuda()[:, :k]
    one = mx.prepack_b_bf16(b)
    two = mx.prepack_b(*mx.quant(b))
    torch.cuda.synchronize()
    assert torch.equal(one.buf, two.buf)


def test_quant_image_into_an_existing_image():
    """quant_image(a, out=img) overwrites img in place and multiplies exactly
    like a fresh image of the same activation (the padding rows of an
    activation image are left unwritten, so the bytes there may differ); an
    image of another shape is refused."""
    a1 = inputs.random_bf16(200, 544, seed=5).cuda()
    a2 = inputs.random_bf16(200, 544, seed=6).cuda()
    packed, _, _ = packed_from_oracle(inputs.random_bf16(256, 544, seed=8, std=0.3))
    img = mx.quant_image(a1)
    buf = img.buf
    again = mx.quant_image(a2, out=img)
    fresh = mx.quant_image(a2)
    c_again = mx.gemm_image(again, packed)
    c_fresh = mx.gemm_image(fresh, packed)
    torch.cuda.synchronize()
    assert again.buf.data_ptr() == buf.data_ptr()
    assert torch.equal(c_again.view(torch.int16), c_fresh.view(torch.int16))
    with pytest.raises(ValueError):
        mx.quant_image(inputs.random_bf16(100, 544, seed=7).cuda(), out=img)


@pytest.mark.parametrize("m,n,k", [(4, 2880, 512), (32, 520, 2080), (33, 256, 512), (64, 384, 2048),
                                   (200, 256, 2048), (1000, 4856, 544), (2044, 512, 2336)])
def test_quant_image_then_gemm_image(m, n, k):
    """A quantized once into the operand layout, multiplied by two different
    weights: both products match the oracle, and for m > 32 (the same plan
    as mxfp4_gemm) they equal mxfp4_gemm bit for bit."""
    a = inputs.random_bf16(m, k, seed=m * 7 + k)
    img = mx.quant_image(a.cuda())
    for seed in (1, 2):
        b = inputs.random_bf16(n, k, seed=n + seed, std=0.3)
        packed, bq, bs = packed_from_oracle(b)
        ldc = n + (8 - n % 8) % 8
        c_full = torch.full((m, ldc), float("nan"), dtype=torch.bfloat16, device="cuda")
        got = mx.gemm_image(img, packed, out=c_full[:, :n])
        torch.cuda.synchronize()
        assert_close_to_ref(got.float().cpu().numpy(), _oracle_full(a, bq, bs), what=f"gemm_image seed {seed}")
        assert torch.isnan(c_full[:, n:].float()).all()
        if m > 32:
            ref = mx.gemm(a.cuda(), packed)
            torch.cuda.synchronize()
            assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def test_persistent_tile_loop_with_ragged_tails():
    """m=1000, n=4856, k=544: 8 x 19 = 152 output tiles of 128 x 256 (at least one
    per SM) run on the CTA-pair kernel as 4 x 19 tiles of 256 x 256; the last
    row tile (104 rows in the odd CTA), the last column tile (248 of 256
    columns, the second weight tile partial) and the last K tile (32 of 256)
    are all ragged."""
    m, n, k = 1000, 4856, 544
    a = inputs.random_bf16(m, k, seed=77)
    b = inputs.random_bf16(n, k, seed=78, std=0.2)
    packed, bq, bs = packed_from_oracle(b)
    got, c_full = _run(a, packed, ldc=n + 8)
    assert_close_to_ref(got, _oracle_full(a, bq, bs), what="persistent")
    assert torch.isnan(c_full[:, n:]).all()


def test_many_row_tiles_but_narrow_n_avoids_the_pair_kernel():
    """m=19456, n=200, k=256: 152 row tiles of 128 but not one full 256-column
    tile, so the planner keeps the one-CTA image kernel (the CTA-pair
    kernel's C box stores need n >= 8 and it wants full 256-column tiles);
    the result matches the oracle."""
    m, n, k = 19456, 200, 256
    a = inputs.random_bf16(m, k, seed=95)
    b = inputs.random_bf16(n, k, seed=96, std=0.2)
    packed, bq, bs = packed_from_oracle(b)
    got, c_full = _run(a, packed, ldc=n + 8)
    assert_close_to_ref(got, _oracle_full(a, bq, bs), what="narrow n, many row tiles")
    assert torch.isnan(c_full[:, n:]).all()


@pytest.mark.parametrize("m,n,k", [(3000, 2304, 288), (4000, 1536, 544), (1100, 4856, 800)])
def test_pair_kernel_later_rounds_and_ragged_edges(m, n, k):
    # More pair tiles than pairs, so each pair walks tiles of several row
    # tiles; a ragged K tail (288), a partial last row tile (4000) and a
    # missing odd row tile (1100).  Full output against the oracle, and equal
    # bit for bit to the same GEMM on a separately made activation image.
    a = inputs.random_bf16(m, k, seed=m + 7 * n + k)
    b = inputs.random_bf16(n, k, seed=n + 3 * k, std=0.5)
    packed, bq, bs = packed_from_oracle(b)
    got, c_full = _run(a, packed, ldc=n + 8)
    assert_close_to_ref(got, _oracle_full(a, bq, bs), what=f"{m}x{n}x{k}")
    assert torch.isnan(c_full[:, n:]).all(), "wrote outside the [m, n] window"
    img = mx.quant_image(a.cuda())
    want = mx.gemm_image(img, packed)
    torch.cuda.synchronize()
    assert torch.equal(c_full[:, :n].view(torch.int16), want.view(torch.int16))


def test_pair_kernel_missing_weight_row_tile():
    """m=1024, n=4700, k=256: 8 x 19 = 152 tiles of 128 x 256 select the CTA-pair
    kernel; the last column tile covers weight rows 4608..4863 but the weights
    end at 4700, so the odd CTA of that tile has no weight row tile at all (it
    copies nothing and writes zero scales for it) and the even CTA's tile is
    ragged (92 of 128 rows)."""
    m, n, k = 1024, 4700, 256
    a = inputs.random_bf16(m, k, seed=93)
    b = inputs.random_bf16(n, k, seed=94, std=0.2)
    packed, bq, bs = packed_from_oracle(b)
    got, c_full = _run(a, packed, ldc=n + 4)
    assert_close_to_ref(got, _oracle_full(a, bq, bs), what="pair kernel, missing weight tile")
    assert torch.isnan(c_full[:, n:]).all()


def test_pair_kernel_more_tiles_than_pairs_and_missing_row_tile():
    """m=1100, n=4856, k=800: 5 x 19 = 95 tiles of 256 x 256 on the CTA pairs,
    so some pairs take two tiles and the ring runs across tiles; the last row
    tile pair has rows 1024-1099 in the even CTA and no activation rows at all
    in the odd one; the last stage holds one and a bit K blocks (K tail 32);
    C's row stride is 4872 elements."""
    m, n, k = 1100, 4856, 800
    a = inputs.random_bf16(m, k, seed=91)
    b = inputs.random_bf16(n, k, seed=92, std=0.2)
    packed, bq, bs = packed_from_oracle(b)
    got, c_full = _run(a, packed, ldc=n + 16)
    assert_close_to_ref(got, _oracle_full(a, bq, bs), what="pair kernel, 95 tiles")
    assert torch.isnan(c_full[:, n:]).all()


@pytest.mark.parametrize("m,n,k", [(16, 2112, 7168), (64, 7168, 2048), (256, 3072, 1536), (4096, 7168, 2048)])
def test_gemm_in_a_captured_cuda_graph(m, n, k):
    """mxfp4_gemm captured into a CUDA graph (for m > 32 the quantization
    kernel and the GEMM as its programmatic dependent) and replayed on new
    contents of the same A buffer gives what the eager call gives."""
    packed, _, _ = packed_from_oracle(inputs.random_bf16(n, k, seed=n + k, std=0.1))
    a = torch.empty((m, k), dtype=torch.bfloat16, device="cuda")
    c = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(mx.workspace_bytes(m, n, k), 16), dtype=torch.uint8, device="cuda")
    a.copy_(inputs.random_bf16(m, k, seed=1))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        mx.gemm(a, packed, out=c, workspace=ws)  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mx.gemm(a, packed, out=c, workspace=ws)
    for seed in (2, 3):
        a.copy_(inputs.random_bf16(m, k, seed=seed))
        g.replay()
        torch.cuda.synchronize()
        want = mx.gemm(a, packed)
        torch.cuda.synchronize()
        assert torch.equal(c.view(torch.int16), want.view(torch.int16)), f"replay with seed {seed}"
    mx.device_status()


@pytest.mark.parametrize("m,n,k", [(1024, 4864, 2560), (1100, 4856, 2016), (4096, 2048, 256), (2048, 4096, 1024)])
def test_pair_kernel_long_k_tails_and_tile_rounds(m, n, k):
    """The CTA-pair plan on long K (2560: ten K blocks, five stages per
    tile), a K tail inside the last stage (2016 = 7.875 K blocks) with a
    missing odd activation row tile and a partial column tile (1100 x 4856),
    more tiles than pairs with the ring running across tiles (4096 x 2048 x
    256: 128 tiles over 76 pairs), and 2048 x 4096 x 1024."""
    a = inputs.random_bf16(m, k, seed=m + n + k)
    b = inputs.random_bf16(n, k, seed=n + 11 * k, std=0.3)
    packed, bq, bs = packed_from_oracle(b)
    got, c_full = _run(a, packed, ldc=n + 8)
    assert_close_to_ref(got, _oracle_full(a, bq, bs), what=f"{m}x{n}x{k}")
    assert torch.isnan(c_full[:, n:]).all(), "wrote outside the [m, n] window"
