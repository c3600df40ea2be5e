"""GPU parity of the whole-layer calls (qg_linear_*): x in, y out, against the
oracle's quantize + GEMM, bit for bit.

The call runs the quantize kernel into a workspace and then the GEMM; for
M <= 16 the decode GEMM is a programmatic dependent of the quantize kernel
(it starts early and waits for the quantize grid before it reads the
activations). Both must give the bits of the oracle, and the same bits as the
separate qg_quantize_act + qg_gemm_* calls.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_quantized_gemm_gb300 as qg
from bit_quantized_gemm_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from bit_quantized_gemm_gb300 import build
    build.build()
    oracle.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def x_dev(x, bits):
    """bf16 activations from their bit patterns, else fp32 values."""
    if bits is not None:
        return to_dev(bits.view(np.int16)).view(torch.bfloat16)
    return to_dev(x.astype(np.float32))


def out_bits(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy().view(np.uint32)


def check_linear(kind, x, bits, weights, N, ldo=None):
    """Run linear_* with bf16 and fp32 outputs; compare outputs and scales with the oracle."""
    M, K = x.shape
    xd = x_dev(x, bits)
    src = bits if bits is not None else x
    oq, os_ = oracle.quantize_act(src)
    gemm = oracle.gemm_w8a8_q8_0 if kind == "q8_0" else oracle.gemm_w4a8_q4k
    y, ob = gemm(oq, os_, weights)
    if kind == "q8_0":
        packed = qg.pack_q8_0(to_dev(weights), N, K)
        fn = qg.linear_w8a8_q8_0
    else:
        packed = qg.pack_q4k(to_dev(weights), N, K)
        fn = qg.linear_w4a8_q4k
    for odt in (torch.bfloat16, torch.float32):
        cols = ldo or N
        full = torch.full((M, cols), 7, dtype=odt, device=DEV)
        out = full[:, :N]
        sc = torch.full((M,), -1.0, dtype=torch.float32, device=DEV)
        fn(xd, packed, N, out=out, scale_out=sc)
        torch.cuda.synchronize()
        qg.check_device_error()
        got = out_bits(out)
        want = ob if odt == torch.bfloat16 else y.view(np.uint32)
        bad = np.argwhere(got != want)
        assert bad.size == 0, (kind, M, K, N, str(odt), bad[:5].tolist())
        assert np.array_equal(sc.cpu().numpy().view(np.uint32), os_.view(np.uint32))
        if ldo:
            # the padding columns of each output row are untouched
            pad = full[:, N:].float().cpu().numpy()
            assert np.all(pad == 7.0)
    return packed


@pytest.mark.parametrize("M,K,N", [(1, 32, 16), (2, 256, 40), (5, 512, 130), (8, 2560, 300),
                                   (9, 96, 64), (16, 1024, 257), (17, 512, 300), (65, 256, 129)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_linear_w8a8_matches_oracle(M, K, N, dtype):
    x, bits = synth.activations(M * 3 + K, M, K, dtype=dtype, outlier_frac=0.01)
    blocks = synth.q8_0_weights(M + K + 7, N, K)
    check_linear("q8_0", x, bits, blocks, N)


@pytest.mark.parametrize("M,K,N", [(1, 256, 16), (3, 512, 40), (8, 1024, 130), (12, 256, 33),
                                   (40, 768, 129)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_linear_w4a8_matches_oracle(M, K, N, dtype):
    x, bits = synth.activations(M * 5 + K, M, K, dtype=dtype, outlier_frac=0.01)
    sblocks = synth.q4k_weights(M + K + 11, N, K)
    check_linear("q4k", x, bits, sblocks, N)


def near_tie_rows(M, K, seed):
    """fp32 rows whose quotients x/s fall within a few ulps of half-integers
    (the quantizer's exact-division branch), a row with a subnormal scale, one
    with a tiny normal scale, and an all-zero row."""
    rng = np.random.default_rng(seed)
    x = np.zeros((M, K), np.float32)
    for m in range(M):
        am = np.float32(rng.uniform(0.5, 4.0))
        s = am / np.float32(127)
        h = rng.integers(-126, 126, size=K).astype(np.float32) + np.float32(0.5)
        v = (h * s).astype(np.float32)
        steps = rng.integers(-3, 4, size=K)
        for i in range(K):
            for _ in range(abs(int(steps[i]))):
                v[i] = np.nextafter(v[i], np.float32(np.inf) if steps[i] > 0 else np.float32(-np.inf))
        v[0] = am
        x[m] = v
    x[M - 1] = x[M - 1] * np.float32(1e-39 / 4.0)   # subnormal scale
    x[M - 2] = x[M - 2] * np.float32(2e-35)        # tiny normal scale
    x[M - 3] = 0.0                                  # s = 0, q = 0
    return x


@pytest.mark.parametrize("kind", ["q8_0", "q4k"])
def test_linear_quantization_near_ties_and_tiny_scales(kind):
    M, K, N = 8, 512, 48
    x = near_tie_rows(M, K, seed=23)
    w = synth.q8_0_weights(5, N, K) if kind == "q8_0" else synth.q4k_weights(5, N, K)
    check_linear(kind, x, None, w, N)


@pytest.mark.parametrize("M", [1, 4, 8, 16])
def test_linear_equals_separate_calls_strided_x_padded_out(M):
    K, N = 1024, 200
    x, bits = synth.activations(M + 41, M, K, dtype="bf16", outlier_frac=0.01)
    # rows of x strided (ldx = K + 64) and outputs padded (ldo = N + 8)
    wide = np.zeros((M, K + 64), np.uint16)
    wide[:, :K] = bits
    xd = to_dev(wide.view(np.int16)).view(torch.bfloat16)[:, :K]
    assert xd.stride(0) == K + 64
    blocks = synth.q8_0_weights(M + 43, N, K)
    packed = qg.pack_q8_0(to_dev(blocks), N, K)
    full = torch.zeros((M, N + 8), dtype=torch.bfloat16, device=DEV)
    qg.linear_w8a8_q8_0(xd, packed, N, out=full[:, :N])
    q, s, _, h = qg.quantize_act(xd, q16=True)
    ref = qg.gemm_w8a8_q8_0(q, h, s, packed, N)
    torch.cuda.synchronize()
    assert np.array_equal(out_bits(full[:, :N]), out_bits(ref))
    assert np.all(full[:, N:].float().cpu().numpy() == 0.0)
    oq, os_ = oracle.quantize_act(bits)
    _, ob = oracle.gemm_w8a8_q8_0(oq, os_, blocks)
    assert np.array_equal(out_bits(ref), ob)


def test_linear_rows_alone_equal_rows_in_batch():
    # a token's output is the same whether it runs alone (decode kernel) or
    # in a batch that takes the prefill kernel
    M, K, N = 96, 2560, 384
    x, bits = synth.activations(77, M, K, dtype="bf16", outlier_frac=0.01)
    blocks = synth.q8_0_weights(78, N, K)
    packed = qg.pack_q8_0(to_dev(blocks), N, K)
    xd = x_dev(x, bits)
    full = out_bits(qg.linear_w8a8_q8_0(xd, packed, N))
    for r in (0, 37, 95):
        one = out_bits(qg.linear_w8a8_q8_0(xd[r:r + 1], packed, N))
        assert np.array_equal(one[0], full[r])
    eight = out_bits(qg.linear_w8a8_q8_0(xd[40:48], packed, N))
    assert np.array_equal(eight, full[40:48])
