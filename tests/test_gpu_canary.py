"""Out-of-bounds write detection without a sanitizer: every output buffer of
the library's calls sits between two guard regions filled with a sentinel
bit pattern, and after each call the guards must be untouched (and the
results still equal the oracle's). Shapes are ragged in M and N so that
every kernel's edge tiles run: decode, tensor-memory prefill (wide and narrow
tiles), 16-row tiles, the quantizer, and the layer call."""
import numpy as np
import pytest
import torch

import oracle
import bit_quantized_gemm_gb300 as qg
from bit_quantized_gemm_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
GUARD = 4096  # elements on each side (keeps 16-byte alignment for every dtype)
SENTINEL = {torch.bfloat16: 0x7FA5, torch.float16: 0x7E5A, torch.float32: 0x7FC0A5A5,
            torch.int8: 0x5A, torch.int32: 0x5A5AA5A5}
INT_VIEW = {torch.bfloat16: torch.int16, torch.float16: torch.int16, torch.float32: torch.int32,
            torch.int8: torch.int8, torch.int32: torch.int32}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from bit_quantized_gemm_gb300 import build
    build.build()
    oracle.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def pattern(dtype):
    """The sentinel as a signed integer of the dtype's width."""
    pat = SENTINEL[dtype]
    bits = {torch.int8: 8, torch.int16: 16, torch.int32: 32}[INT_VIEW[dtype]]
    return pat - (1 << bits) if pat >= 1 << (bits - 1) else pat


def guarded(shape, dtype):
    """(whole buffer, view of `shape` between the guards)"""
    n = int(np.prod(shape))
    buf = torch.empty((GUARD + n + GUARD,), dtype=dtype, device=DEV)
    buf.view(INT_VIEW[dtype]).fill_(pattern(dtype))
    return buf, buf[GUARD:GUARD + n].view(shape)


def guards_intact(buf):
    iv = buf.view(INT_VIEW[buf.dtype]).cpu().numpy()
    pat = pattern(buf.dtype)
    n = iv.size - 2 * GUARD
    return bool(np.all(iv[:GUARD] == pat) and np.all(iv[GUARD + n:] == pat))


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def bits_of(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy().view(np.uint32)


def quantize_guarded(bits, block_sums):
    M, K = bits.shape
    xd = to_dev(bits.view(np.int16)).view(torch.bfloat16)
    qb, q = guarded((M, K), torch.int8)
    sb, s = guarded((M,), torch.float32)
    hb, h = guarded((M, K), torch.float16)
    bb, bs = guarded((M, K // 32), torch.int32) if block_sums else (None, None)
    qg.quantize_act(xd, block_sums=block_sums, q16=True, out=(q, s, bs, h))
    torch.cuda.synchronize()
    for b in (qb, sb, hb, bb):
        if b is not None:
            assert guards_intact(b)
    return q, s, bs, h


@pytest.mark.parametrize("M,K,N,path", [
    (3, 96, 40, "small"), (16, 512, 300, "small"), (17, 512, 300, "large"),
    (129, 1024, 257, "large"), (300, 640, 520, "large"), (2048, 2560, 1000, "large"),
    (2048, 9728, 2560, "auto"),  # wide launch plus the 16-row tail launch
])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_w8a8_writes_stay_inside_their_buffers(M, K, N, path, out_dtype):
    x, bits = synth.activations(M + K + N, M, K, dtype="bf16", outlier_frac=0.01)
    blocks = synth.q8_0_weights(M + N, N, K)
    q, s, _, h = quantize_guarded(bits, block_sums=False)
    packed = qg.pack_q8_0(to_dev(blocks), N, K)
    ob, out = guarded((M, N), out_dtype)
    qg.gemm_w8a8_q8_0(q, h, s, packed, N, out=out, path=path)
    torch.cuda.synchronize()
    qg.check_device_error()
    assert guards_intact(ob)
    rows = np.unique(np.linspace(0, M - 1, num=min(M, 24)).astype(int))
    oq, os_ = oracle.quantize_act(bits[rows])
    y, obits = oracle.gemm_w8a8_q8_0(oq, os_, blocks)
    want = obits if out_dtype == torch.bfloat16 else y.view(np.uint32)
    assert np.array_equal(bits_of(out)[rows], want)


@pytest.mark.parametrize("M,K,N,path", [(5, 512, 40, "small"), (65, 256, 129, "large"),
                                        (200, 768, 300, "large")])
def test_w4a8_writes_stay_inside_their_buffers(M, K, N, path):
    x, bits = synth.activations(M + K, M, K, dtype="bf16", outlier_frac=0.01)
    sblocks = synth.q4k_weights(M + N, N, K)
    q, s, bs, h = quantize_guarded(bits, block_sums=True)
    packed = qg.pack_q4k(to_dev(sblocks), N, K)
    ob, out = guarded((M, N), torch.bfloat16)
    qg.gemm_w4a8_q4k(q, h, s, bs, packed, N, out=out, path=path)
    torch.cuda.synchronize()
    qg.check_device_error()
    assert guards_intact(ob)
    oq, os_ = oracle.quantize_act(bits)
    _, obits = oracle.gemm_w4a8_q4k(oq, os_, sblocks)
    assert np.array_equal(bits_of(out), obits)


@pytest.mark.parametrize("M", [1, 9, 33])
def test_layer_call_writes_stay_inside_its_buffers(M):
    K, N = 512, 130
    x, bits = synth.activations(M + 3, M, K, dtype="bf16", outlier_frac=0.01)
    blocks = synth.q8_0_weights(M + 4, N, K)
    packed = qg.pack_q8_0(to_dev(blocks), N, K)
    xd = to_dev(bits.view(np.int16)).view(torch.bfloat16)
    ob, out = guarded((M, N), torch.bfloat16)
    sb, sc = guarded((M,), torch.float32)
    nbytes = qg.linear_workspace_bytes("q8_0", M, K)
    wb, ws = guarded((nbytes,), torch.int8)
    qg.linear_w8a8_q8_0(xd, packed, N, out=out, scale_out=sc, workspace=ws)
    torch.cuda.synchronize()
    qg.check_device_error()
    assert guards_intact(ob) and guards_intact(sb) and guards_intact(wb)
    oq, os_ = oracle.quantize_act(bits)
    _, obits = oracle.gemm_w8a8_q8_0(oq, os_, blocks)
    assert np.array_equal(bits_of(out), obits)
