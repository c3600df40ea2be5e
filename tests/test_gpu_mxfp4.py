"""GPU parity for MXFP4 weights converted from Q8_0, through the C ABI.

The conversion (qg_pack_mxfp4_q8_0) is checked through what the kernels
compute with it: every output of the GEMM and of the layer call equals the
oracle's (orc_mxfp4_from_q8_0 then orc_gemm_w4a8_mxfp4) bit for bit, on the
decode kernels (dp4a and int8-MMA tiles), the 16-row and the tensor-memory
prefill kernels. Lossy against the original Q8_0 weights by design; the
oracle's CPU tests bound that error.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_quantized_gemm_gb300 as qg
from bit_quantized_gemm_gb300 import synth
from bit_quantized_gemm_gb300._lib import QG_ERANGE, QGError

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


def bf16_dev(bits):
    return to_dev(bits.view(np.int16)).view(torch.bfloat16)


def out_bits(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy().view(np.uint32)


def oracle_out(bits, blocks):
    codes, E = oracle.mxfp4_from_q8_0(blocks)
    oq, os_ = oracle.quantize_act(bits)
    return oracle.gemm_w4a8_mxfp4(oq, os_, codes, E)


@pytest.mark.parametrize("M,K,N", [
    (1, 256, 40), (3, 512, 33), (8, 320, 48), (16, 256, 100), (40, 512, 130), (300, 1024, 260),
])
def test_mxfp4_gemm_and_layer_match_oracle(M, K, N):
    _, bits = synth.activations(M * 7 + K, M, K, dtype="bf16", outlier_frac=0.01)
    blocks = synth.q8_0_weights(N + K, N, K)
    y, ob = oracle_out(bits, blocks)
    packed = qg.pack_mxfp4_q8_0(to_dev(blocks), N, K)
    qg.check_device_error()  # every block scale fits the decode kernels' fp16
    q, s, _, h = qg.quantize_act(bf16_dev(bits), q16=True)
    out = qg.gemm_w4a8_mxfp4(q, h, s, packed, N)
    bad = np.argwhere(out_bits(out) != ob)
    assert bad.size == 0, "first mismatches %s" % bad[:5].tolist()
    out32 = qg.gemm_w4a8_mxfp4(q, h, s, packed, N, out_dtype=torch.float32)
    assert np.array_equal(out_bits(out32), y.view(np.uint32))
    lay = qg.linear_w4a8_mxfp4(bf16_dev(bits), packed, N)
    assert np.array_equal(out_bits(lay), ob)


def test_mxfp4_fixture_blocks_on_gpu():
    """The hand-derived fixture's blocks (ties, saturation, signs, scale,
    zero block, chain order) through the GPU conversion and GEMM."""
    import golden_io
    for case in golden_io.mxfp4_cases():
        blocks, qa = golden_io.mxfp4_case_arrays(case)
        K = qa.shape[1]
        packed = qg.pack_mxfp4_q8_0(to_dev(blocks), 1, K)
        qg.check_device_error()
        q = to_dev(qa)
        s = torch.ones(1, dtype=torch.float32, device=DEV)
        out = qg.gemm_w4a8_mxfp4(q, None, s, packed, 1)
        assert int(out_bits(out)[0, 0]) == case["y"], case["name"]
        if "y32" in case:
            out32 = qg.gemm_w4a8_mxfp4(q, None, s, packed, 1, out_dtype=torch.float32)
            assert int(out_bits(out32)[0, 0]) == case["y32"], case["name"]


def test_mxfp4_decode_full_size():
    """One token through the 5120 -> 17408 projection: every output."""
    M, K, N = 1, 5120, 17408
    _, bits = synth.activations(31, M, K, dtype="bf16", outlier_frac=0.01)
    blocks = synth.q8_0_weights(107, N, K)
    _, ob = oracle_out(bits, blocks)
    packed = qg.pack_mxfp4_q8_0(to_dev(blocks), N, K)
    qg.check_device_error()
    lay = qg.linear_w4a8_mxfp4(bf16_dev(bits), packed, N)
    assert np.array_equal(out_bits(lay), ob)


def test_mxfp4_scale_outside_fp16_is_reported():
    """A block of tiny weights (max |w| = 2^-24) needs X/2 = 2^-27, which the
    decode kernels' fp16 scales cannot hold: the next device-error check
    reports QG_ERANGE, and the one after it is clean again."""
    blocks = np.zeros((2, 1, 34), np.uint8)
    blocks[0, 0, 0:2] = [0x01, 0x00]   # d = 2^-24 (fp16 subnormal)
    blocks[0, 0, 2] = 1
    blocks[1, 0, 0:2] = [0x00, 0x3C]   # d = 1: in range
    blocks[1, 0, 2] = 5
    qg.pack_mxfp4_q8_0(to_dev(blocks), 2, 32)
    with pytest.raises(QGError) as e:
        qg.check_device_error()
    assert e.value.status == QG_ERANGE
    qg.check_device_error()
