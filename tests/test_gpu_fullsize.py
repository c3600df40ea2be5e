"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (AUTO kernel choice), on seeded samples the oracle computes
one by one: whole tensors for the quantizer, and for each GEMM a set of
random rows x all N plus all M x a set of random columns, bit for bit.

Workloads (shapes and value recipes of the 4B/27B-class model projections):
4B prefill M=2048; decode M in {1, 8, 64}; 27B prefill M=8192 with the
batch-invariance runs (rows alone and inside mixed batches); W4A8 Q4_K
M in {1, 64, 4096}.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_quantized_gemm_gb300 as qg
from bit_quantized_gemm_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
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


def bits_of(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def check_sampled(out, oq, os_, weights, kind, n_rows=256, n_cols=256, seed=0):
    """Compare sampled rows (all N) and sampled columns (all M) with the oracle."""
    M, N = out.shape
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, M - 1], rng.choice(M, size=min(n_rows, M), replace=False)]))
    cols = np.unique(np.concatenate([[0, N - 1], rng.choice(N, size=min(n_cols, N), replace=False)]))
    gemm = oracle.gemm_w8a8_q8_0 if kind == "w8a8" else oracle.gemm_w4a8_q4k
    got = bits_of(out)
    _, ob = gemm(oq[rows], os_[rows], weights)
    assert np.array_equal(got[rows], ob), "row sample differs"
    _, oc = gemm(oq, os_, np.ascontiguousarray(weights[cols]))
    assert np.array_equal(got[:, cols], oc), "column sample differs"


def quant_full(name, M, K, seed_offset=0, bsum=False):
    x, bits = synth.config_activations(name, M, K, seed_offset=seed_offset)
    xd = to_dev(bits.view(np.int16)).view(torch.bfloat16)
    q, s, bs, h = qg.quantize_act(xd, block_sums=bsum, q16=True)
    res = oracle.quantize_act(bits, bsum=bsum)
    oq, os_ = res[0], res[1]
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(h.float().cpu().numpy(), oq.astype(np.float32))
    if bsum:
        assert np.array_equal(bs.cpu().numpy(), res[2])
    return (q, s, bs, h), oq, os_


@pytest.mark.parametrize("M,K,N,off", [(2048, 2560, 9728, 0), (2048, 9728, 2560, 1)])
def test_prefill_4b(M, K, N, off):
    (q, s, _, h), oq, os_ = quant_full("prefill_4b_w8a8", M, K, off)
    blocks = synth.config_weights("prefill_4b_w8a8", N, K, seed_offset=off)
    packed = qg.pack_q8_0(to_dev(blocks), N, K)
    out = qg.gemm_w8a8_q8_0(q, h, s, packed, N)
    torch.cuda.synchronize()
    qg.check_device_error()
    check_sampled(out, oq, os_, blocks, "w8a8", seed=M + K)


@pytest.mark.parametrize("K,N", [(5120, 17408), (17408, 5120)])
def test_decode(K, N):
    blocks = synth.config_weights("decode_w8a8", N, K)
    packed = qg.pack_q8_0(to_dev(blocks), N, K)
    for M in (1, 8, 64):
        (q, s, _, h), oq, os_ = quant_full("decode_w8a8", M, K)
        out = qg.gemm_w8a8_q8_0(q, h, s, packed, N)
        torch.cuda.synchronize()
        # all rows of the decode batch are compared in full
        _, ob = oracle.gemm_w8a8_q8_0(oq, os_, blocks)
        assert np.array_equal(bits_of(out), ob), (M, K, N)


@pytest.mark.parametrize("K,N", [(5120, 17408), (17408, 5120)])
def test_prefill_27b_and_batch_invariance(K, N):
    M = 8192
    (q, s, _, h), oq, os_ = quant_full("prefill_27b_w8a8", M, K)
    blocks = synth.config_weights("prefill_27b_w8a8", N, K)
    packed = qg.pack_q8_0(to_dev(blocks), N, K)
    out = qg.gemm_w8a8_q8_0(q, h, s, packed, N)
    torch.cuda.synchronize()
    qg.check_device_error()
    check_sampled(out, oq, os_, blocks, "w8a8", n_rows=128, n_cols=128, seed=K)
    full = bits_of(out)
    # 64 seeded rows alone (decode kernel) and inside mixed batches of 8 and 64
    # rows at random positions equal the same rows of the 8192-row batch
    rng = np.random.default_rng(7)
    probe = rng.choice(M, size=64, replace=False)
    for r in probe[:16]:
        o1 = qg.gemm_w8a8_q8_0(q[r:r + 1], h[r:r + 1], s[r:r + 1], packed, N)
        assert np.array_equal(bits_of(o1)[0], full[r])
    for mb in (8, 64):
        idx = rng.choice(M, size=mb, replace=False)
        idx[: mb // 2] = probe[: mb // 2]
        rng.shuffle(idx)
        ti = torch.from_numpy(idx).to(DEV)
        ob = qg.gemm_w8a8_q8_0(q[ti], h[ti], s[ti], packed, N)
        assert np.array_equal(bits_of(ob), full[idx])


def test_w4a8_q4k():
    K, N = 5120, 17408
    sblocks = synth.config_weights("w4a8_q4k", N, K)
    packed = qg.pack_q4k(to_dev(sblocks), N, K)
    for M in (1, 64, 4096):
        (q, s, bs, h), oq, os_ = quant_full("w4a8_q4k", M, K, bsum=True)
        out = qg.gemm_w4a8_q4k(q, h, s, bs, packed, N)
        torch.cuda.synchronize()
        qg.check_device_error()
        if M <= 64:
            _, ob = oracle.gemm_w4a8_q4k(oq, os_, sblocks)
            assert np.array_equal(bits_of(out), ob), M
        else:
            check_sampled(out, oq, os_, sblocks, "w4a8", n_rows=128, n_cols=128, seed=M)


@pytest.mark.parametrize("M,N,tb", [(24, 5120, 32), (64, 2560, 64), (64, 5120, 64), (40, 5120, 64)])
def test_skinny_long_k_repeated(M, N, tb):
    # 16-row tiles over K = 17408 (272 ring stages per CTA) with many CTAs per
    # SM, three launches in a row: every output of every launch against the
    # oracle (a race in the ring would show as a whole warp's tokens wrong in
    # some CTAs, differently from launch to launch)
    from bit_quantized_gemm_gb300 import _lib
    K = 17408
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms == 152:
        assert _lib.prefill_plan(M, N, sms) == (0, "16-row", tb)
    blocks = synth.config_weights("decode_w8a8", N, K, seed_offset=tb)
    packed = qg.pack_q8_0(to_dev(blocks), N, K)
    (q, s, _, h), oq, os_ = quant_full("decode_w8a8", M, K, seed_offset=tb)
    _, ob = oracle.gemm_w8a8_q8_0(oq, os_, blocks)
    for _ in range(3):
        out = qg.gemm_w8a8_q8_0(q, h, s, packed, N)
        torch.cuda.synchronize()
        qg.check_device_error()
        assert np.array_equal(bits_of(out), ob)


def test_w4a8_q4k_narrow_down_projection():
    # 17408 -> 5120 at 32 and 64 tokens: 40 weight-row tiles of 128, so these
    # run as 16-row tiles (320 per token tile), each walking all 544 sub-blocks;
    # every output compared
    from bit_quantized_gemm_gb300 import _lib
    K, N = 17408, 5120
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert _lib.prefill_tile_q4k(32, N, 152) == ("16-row", 32)
        assert _lib.prefill_tile_q4k(64, N, 152) == ("16-row", 64)
    sblocks = synth.config_weights("w4a8_q4k", N, K)
    packed = qg.pack_q4k(to_dev(sblocks), N, K)
    for M in (32, 64):
        (q, s, bs, h), oq, os_ = quant_full("w4a8_q4k", M, K, bsum=True)
        out = qg.gemm_w4a8_q4k(q, h, s, bs, packed, N)
        torch.cuda.synchronize()
        qg.check_device_error()
        _, ob = oracle.gemm_w4a8_q4k(oq, os_, sblocks)
        assert np.array_equal(bits_of(out), ob), M


def test_tiny_config():
    M, K, N = synth.CONFIGS["tiny_w8a8"]["shapes"][0]
    x, _ = synth.config_activations("tiny_w8a8", M, K)
    blocks = synth.config_weights("tiny_w8a8", N, K)
    q, s, _, h = qg.quantize_act(to_dev(x), q16=True)
    packed = qg.pack_q8_0(to_dev(blocks), N, K)
    out = qg.gemm_w8a8_q8_0(q, h, s, packed, N)
    oq, os_ = oracle.quantize_act(x)
    _, ob = oracle.gemm_w8a8_q8_0(oq, os_, blocks)
    assert np.array_equal(bits_of(out), ob)


def test_launch_plan_of_the_benchmark_step():
    # on 152 SMs the 4B down projection (160 tiles of 256 tokens) runs as one
    # full wave of wide tiles plus a narrow-tile launch; gate/up fills 4 waves
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("plan figures are for 152 SMs")
    assert qg.gemm_launch_count("q8_0", 2048, 2560, 9728) == 1
    assert qg.gemm_launch_count("q8_0", 2048, 9728, 2560) == 2
    assert qg.gemm_launch_count("q8_0", 8192, 5120, 17408) == 1
    assert qg.gemm_launch_count("q4k", 4096, 5120, 17408) == 1
    assert qg.gemm_launch_count("q8_0", 8, 5120, 17408) == 1


@pytest.mark.parametrize("kind,K,N", [("q8_0", 5120, 17408), ("q8_0", 17408, 5120),
                                      ("q4k", 5120, 17408)])
def test_linear_decode_full_size(kind, K, N):
    # the whole layer (x in, y out) at decode sizes (the decode GEMM overlaps
    # the quantize kernel); every output element compared
    name = "decode_w8a8" if kind == "q8_0" else "w4a8_q4k"
    w = synth.config_weights(name, N, K)
    packed = qg.pack_q8_0(to_dev(w), N, K) if kind == "q8_0" else qg.pack_q4k(to_dev(w), N, K)
    fn = qg.linear_w8a8_q8_0 if kind == "q8_0" else qg.linear_w4a8_q4k
    gemm = oracle.gemm_w8a8_q8_0 if kind == "q8_0" else oracle.gemm_w4a8_q4k
    for M in (1, 8, 16):
        x, bits = synth.config_activations(name, M, K)
        xd = to_dev(bits.view(np.int16)).view(torch.bfloat16)
        out = fn(xd, packed, N)
        torch.cuda.synchronize()
        qg.check_device_error()
        oq, os_ = oracle.quantize_act(bits)
        _, ob = gemm(oq, os_, w)
        assert np.array_equal(bits_of(out), ob), (kind, M, K, N)
