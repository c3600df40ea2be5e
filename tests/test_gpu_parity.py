"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle.

Matching rules (the layer's contract): quantized activations, scales and the
per-block int32 sums are bit-exact; outputs are bit-exact too, because every
kernel keeps the oracle's ascending-block, one-FMA-per-block fp32 chain (the
tolerance rule |err| <= 1e-5 * sum|terms| would be the fallback, and is
asserted as well where an fp32 output is compared).
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


def bf16_dev(bits):
    return to_dev(bits.view(np.int16)).view(torch.bfloat16)


def run_quant(x_vals, x_bits, want_bs=True):
    """Quantize on the GPU; returns numpy (q, s, bs, q16) and the device tensors."""
    xd = bf16_dev(x_bits) if x_bits is not None else to_dev(x_vals.astype(np.float32))
    q, s, bs, h = qg.quantize_act(xd, block_sums=want_bs, q16=True)
    torch.cuda.synchronize()
    return (q, s, bs, h)


def oracle_quant(x_vals, x_bits):
    return oracle.quantize_act(x_bits if x_bits is not None else x_vals, bsum=True)


def out_bits(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy().view(np.uint32)


# --------------------------------------------------------------------- quantize
@pytest.mark.parametrize("M,K,dtype,outl,seq", [
    (4, 256, "f32", 0.0, None), (37, 320, "bf16", 0.01, 8), (3, 32, "bf16", 0.0, None),
    (64, 5120, "bf16", 0.0, None), (9, 17408, "bf16", 0.01, None), (5, 24576, "f32", 0.01, None),
    (130, 2560, "bf16", 0.01, 128),
])
def test_quantize_bit_exact(M, K, dtype, outl, seq):
    x, bits = synth.activations(M * 7 + K, M, K, dtype=dtype, outlier_frac=outl, seq_slots=seq,
                                min_len=1 if seq else None)
    q, s, bs, h = run_quant(x, bits)
    oq, os_, obs = oracle_quant(x, bits)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(bs.cpu().numpy(), obs)
    assert np.array_equal(h.float().cpu().numpy(), oq.astype(np.float32))


def test_quantize_golden_ties_and_strided_rows():
    import golden_io
    cases = golden_io.quantize_cases()
    x = np.zeros((len(cases), 32), np.float32)
    for i, c in enumerate(cases):
        for k, v in c["x"].items():
            x[i, k] = v
    # strided rows: ldx = 64
    wide = np.zeros((len(cases), 64), np.float32)
    wide[:, :32] = x
    xd = to_dev(wide)[:, :32]
    q, s, bs, _ = qg.quantize_act(xd, block_sums=True)
    for i, c in enumerate(cases):
        assert s[i].item() == np.float32(c["s"])
        exp = np.zeros(32, np.int8)
        for k, v in c["q"].items():
            exp[k] = v
        assert np.array_equal(q[i].cpu().numpy(), exp)
        assert bs[i, 0].item() == c["bsum"][0]


# --------------------------------------------------------------------- W8A8
def make_w8a8(M, K, N, seed, dtype="bf16", outl=0.0, seq=None):
    x, bits = synth.activations(seed, M, K, dtype=dtype, outlier_frac=outl, seq_slots=seq,
                                min_len=1 if seq else None)
    blocks = synth.q8_0_weights(seed + 100, N, K)
    return x, bits, blocks


def gpu_w8a8(x, bits, blocks, N, path, out_dtype=torch.bfloat16):
    K = x.shape[1]
    q, s, _, h = run_quant(x, bits, want_bs=False)
    packed = qg.pack_q8_0(to_dev(blocks), N, K)
    out = qg.gemm_w8a8_q8_0(q, h, s, packed, N, out_dtype=out_dtype, path=path)
    torch.cuda.synchronize()
    qg.check_device_error()
    return out, (q, h, s, packed)


SHAPES = [(1, 32, 16), (3, 96, 40), (8, 256, 128), (17, 512, 300), (64, 2560, 1000),
          (65, 256, 129), (129, 1024, 257), (300, 640, 520), (513, 96, 130)]


@pytest.mark.parametrize("M,K,N", SHAPES)
@pytest.mark.parametrize("path", ["small", "large"])
def test_w8a8_matches_oracle(M, K, N, path):
    x, bits, blocks = make_w8a8(M, K, N, seed=M + K + N, outl=0.01)
    out, _ = gpu_w8a8(x, bits, blocks, N, path)
    oq, os_ = oracle.quantize_act(bits)
    y, ob = oracle.gemm_w8a8_q8_0(oq, os_, blocks)
    got = out_bits(out)
    bad = np.argwhere(got != ob)
    assert bad.size == 0, "first mismatches %s" % bad[:5].tolist()
    out32, _ = gpu_w8a8(x, bits, blocks, N, path, out_dtype=torch.float32)
    assert np.array_equal(out_bits(out32), y.view(np.uint32))


@pytest.mark.parametrize("M", [1, 3, 9, 20, 200])
def test_longest_k_both_formats(M):
    """K at its upper limit (65536: 2048 blocks, 256 Q4_K super-blocks) on
    every kernel the row count selects (integer decode, int8-MMA decode,
    narrow and 16-row tiles, tensor-memory tiles); W8A8 and W4A8 outputs and
    the layer call against the oracle, every element."""
    K, N = 65536, 40
    x, bits = synth.activations(M + 3, M, K, dtype="bf16", outlier_frac=0.01)
    oq, os_, _ = oracle.quantize_act(bits, bsum=True)
    blocks = synth.q8_0_weights(M + 11, N, K)
    _, ob = oracle.gemm_w8a8_q8_0(oq, os_, blocks)
    out, (q, h, s, packed) = gpu_w8a8(x, bits, blocks, N, "auto")
    assert np.array_equal(out_bits(out), ob)
    lay = qg.linear_w8a8_q8_0(bf16_dev(bits), packed, N)
    assert np.array_equal(out_bits(lay), ob)
    sblocks = synth.q4k_weights(M + 13, N, K)
    _, ob4 = oracle.gemm_w4a8_q4k(oq, os_, sblocks)
    out4, _ = gpu_w4a8(bits, sblocks, N, "auto")
    assert np.array_equal(out_bits(out4), ob4)


@pytest.mark.parametrize("M,K,N,tb", [(32, 9728, 128, 32), (2048, 9728, 128, 64),
                                      (4096, 2560, 128, 128)])
def test_skinny_tiles_every_token_width(M, K, N, tb):
    """The 16-row kernel at each of its token-tile widths (the wave plan
    sends these whole GEMMs to it on 152 SMs), on the 2048 x 9728 x 128 shape
    among them; every output against the oracle."""
    from bit_quantized_gemm_gb300 import _lib
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms == 152:
        assert _lib.prefill_plan(M, N, sms) == (0, "16-row", tb)
    x, bits, blocks = make_w8a8(M, K, N, seed=M + 5 * tb, outl=0.02)
    out, _ = gpu_w8a8(x, bits, blocks, N, "auto")
    oq, os_ = oracle.quantize_act(bits)
    _, ob = oracle.gemm_w8a8_q8_0(oq, os_, blocks)
    bad = np.argwhere(out_bits(out) != ob)
    assert bad.size == 0, "first mismatches %s" % bad[:5].tolist()


def test_w8a8_tiny_config_both_paths():
    M, K, N = synth.CONFIGS["tiny_w8a8"]["shapes"][0]
    x, _ = synth.config_activations("tiny_w8a8", M, K)
    blocks = synth.config_weights("tiny_w8a8", N, K)
    oq, os_ = oracle.quantize_act(x)
    y, ob = oracle.gemm_w8a8_q8_0(oq, os_, blocks)
    for path in ("auto", "small", "large"):
        out, _ = gpu_w8a8(x, None, blocks, N, path)
        assert np.array_equal(out_bits(out), ob)


@pytest.mark.parametrize("path", ["small", "large"])
def test_w8a8_block_sums_exact_adversarial(path):
    """The tensor-core block accumulators must hold the exact integer sums,
    including the extremes +-32*127*127 and full cancellation."""
    M, K, N = 40, 256, 48
    rng = np.random.default_rng(5)
    qa = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    qa[0] = 127
    qa[1] = -127
    qa[2, ::2] = 127
    qa[2, 1::2] = -127
    qw = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
    qw[0] = 127
    qw[1] = -127
    qw[2] = 127
    blocks = np.zeros((N, K // 32, 34), np.uint8)
    blocks[:, :, 0:2] = np.array([0x3C00], np.uint16).view(np.uint8)
    blocks[:, :, 2:] = qw.view(np.uint8).reshape(N, K // 32, 32)
    qd = to_dev(qa)
    hd = qd.to(torch.float16)
    packed = qg.pack_q8_0(to_dev(blocks), N, K)
    isum = qg.debug_block_sums("q8_0", qd, hd, packed, N, path).cpu().numpy()
    ref = oracle.block_sums_q8_0(qa, blocks)
    assert isum[0, 0, 0] == 516128 and isum[1, 0, 0] == -516128
    assert np.array_equal(isum, ref)


@pytest.mark.parametrize("path", ["small", "large"])
def test_w8a8_special_rows(path):
    M, K, N = 70, 256, 64
    x, bits, blocks = make_w8a8(M, K, N, seed=3)
    x = x.copy()
    x[5] = 0.0                      # zero row
    x[6] = 0.0
    x[6, 17] = -2.75                # one-hot row
    x[7] *= 1e-30                   # tiny magnitudes
    blocks = blocks.copy()
    blocks[9, :, 0:2] = 0           # d = 0 row
    out, _ = gpu_w8a8(x, None, blocks, N, path, out_dtype=torch.float32)
    oq, os_ = oracle.quantize_act(x)
    y, _ = oracle.gemm_w8a8_q8_0(oq, os_, blocks)
    assert np.array_equal(out_bits(out), y.view(np.uint32))
    assert np.all(out[5].cpu().numpy().view(np.uint32) == 0)


def test_w8a8_batch_invariance_and_paths():
    """Each row alone (M=1, decode kernel) gives the same bits as inside mixed
    batches on either kernel, at any position, next to zero and outlier rows."""
    K, N = 512, 272
    rng = np.random.default_rng(11)
    xs, bits = synth.activations(77, 300, K, dtype="bf16", outlier_frac=0.01)
    blocks = synth.q8_0_weights(177, N, K)
    packed = qg.pack_q8_0(to_dev(blocks), N, K)
    xd = bf16_dev(bits)
    q, s, _, h = qg.quantize_act(xd, q16=True)
    probe = rng.choice(300, size=12, replace=False)
    alone = {}
    for r in probe:
        o = qg.gemm_w8a8_q8_0(q[r:r + 1], h[r:r + 1], s[r:r + 1], packed, N, path="small")
        alone[r] = out_bits(o)[0]
    for M in (8, 64, 65, 300):
        for path in ("small", "large"):
            idx = torch.from_numpy(rng.permutation(300)[:M])
            for r in probe[:4]:
                idx[rng.integers(0, M)] = int(r)
            qi, si, hi = q[idx.to(DEV)], s[idx.to(DEV)], h[idx.to(DEV)]
            o = out_bits(qg.gemm_w8a8_q8_0(qi, hi, si, packed, N, path=path))
            for j, r in enumerate(idx.tolist()):
                if r in alone:
                    assert np.array_equal(o[j], alone[r]), (M, path, j, r)
    full_s = out_bits(qg.gemm_w8a8_q8_0(q, h, s, packed, N, path="small"))
    full_l = out_bits(qg.gemm_w8a8_q8_0(q, h, s, packed, N, path="large"))
    assert np.array_equal(full_s, full_l)


def test_launch_count_follows_the_wave_plan():
    """qg_gemm_launch_count on this GPU equals the launches of the plan the
    host query gives for its SM count (two when a narrow part follows a wide
    launch)."""
    from bit_quantized_gemm_gb300 import _lib
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for M, K, N in [(8192, 5120, 17408), (8192, 17408, 5120), (2048, 2560, 9728),
                    (2048, 9728, 2560), (64, 5120, 17408), (300, 640, 520), (4096, 5120, 17408)]:
        rows, kind, _ = _lib.prefill_plan(M, N, sms)
        want = 2 if (kind is not None and rows > 0) else 1
        assert qg.gemm_launch_count("q8_0", M, K, N) == want, (M, K, N)
        assert qg.gemm_launch_count("q8_0", M, K, N, path="small") == -(-M // 16)


# --------------------------------------------------------------------- W4A8
def gpu_w4a8(bits, sblocks, N, path, out_dtype=torch.bfloat16):
    K = bits.shape[1]
    q, s, bs, h = qg.quantize_act(bf16_dev(bits), block_sums=True, q16=True)
    packed = qg.pack_q4k(to_dev(sblocks), N, K)
    out = qg.gemm_w4a8_q4k(q, h, s, bs, packed, N, out_dtype=out_dtype, path=path)
    torch.cuda.synchronize()
    qg.check_device_error()
    return out, (q, h, s, bs, packed)


@pytest.mark.parametrize("M,K,N", [(1, 256, 16), (5, 512, 40), (64, 1024, 130), (65, 256, 129),
                                   (200, 768, 300), (300, 2048, 64)])
@pytest.mark.parametrize("path", ["small", "large"])
def test_w4a8_matches_oracle(M, K, N, path):
    x, bits = synth.activations(M + K, M, K, dtype="bf16", outlier_frac=0.01)
    sblocks = synth.q4k_weights(M + K + 100, N, K)
    out, _ = gpu_w4a8(bits, sblocks, N, path)
    oq, os_ = oracle.quantize_act(bits)
    y, ob = oracle.gemm_w4a8_q4k(oq, os_, sblocks)
    got = out_bits(out)
    bad = np.argwhere(got != ob)
    assert bad.size == 0, "first mismatches %s" % bad[:5].tolist()
    out32, _ = gpu_w4a8(bits, sblocks, N, path, out_dtype=torch.float32)
    assert np.array_equal(out_bits(out32), y.view(np.uint32))


@pytest.mark.parametrize("path", ["small", "large"])
def test_w4a8_golden_epilogue_order(path):
    """The hand-derived cases of tests/golden/gemm_q4k_small.txt on both
    kernels: exact value 0, chain result +2^-9 only with the isum term
    before the min term, fused, sub-blocks ascending. Each case row sits
    among seeded rows (rows are independent)."""
    import golden_io
    for case in golden_io.gemm_q4k_cases():
        x, sblocks = golden_io.q4k_case_arrays(case)
        K, N = x.shape[1], sblocks.shape[0]
        _, rnd = synth.activations(K + 5, 3, K, dtype="bf16", outlier_frac=0.01)
        xb = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        bits = np.concatenate([rnd[:1], xb, rnd[1:]], axis=0)
        out, _ = gpu_w4a8(bits, sblocks, N, path, out_dtype=torch.float32)
        got = out.cpu().numpy()
        for n, v in case["y"].items():
            assert got[1, n].view(np.uint32) == np.float32(v).view(np.uint32), (case["name"], got[1, n])
        outb, _ = gpu_w4a8(bits, sblocks, N, path)
        for n, v in case["bf16"].items():
            assert out_bits(outb)[1, n] == v


@pytest.mark.parametrize("path", ["small", "large"])
def test_w4a8_block_sums_exact(path):
    M, K, N = 33, 512, 40
    x, bits = synth.activations(9, M, K, dtype="bf16", outlier_frac=0.05)
    sblocks = synth.q4k_weights(109, N, K)
    q, s, bs, h = qg.quantize_act(bf16_dev(bits), block_sums=True, q16=True)
    packed = qg.pack_q4k(to_dev(sblocks), N, K)
    isum = qg.debug_block_sums("q4k", q, h, packed, N, path).cpu().numpy()
    oq, _ = oracle.quantize_act(bits)
    ri, ra = oracle.block_sums_q4k(oq, sblocks)
    assert np.array_equal(isum, ri)
    assert np.array_equal(bs.cpu().numpy(), ra)


def test_w4a8_256_token_tiles():
    # 700 tokens x 5000 weight rows: on 152 SMs three 256-token tiles per
    # weight-row tile (the last one ragged, and a ragged last weight-row tile),
    # 120 tiles in one wave against 240 as 128-token tiles; every output
    # compared in bf16 and fp32, and rows alone equal the batch's rows
    from bit_quantized_gemm_gb300 import _lib
    M, K, N = 700, 512, 5000
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert _lib.prefill_tile_q4k(M, N, 152) == ("tensor", 256)
    x, bits = synth.activations(71, M, K, dtype="bf16", outlier_frac=0.01)
    sblocks = synth.q4k_weights(171, N, K)
    out, (q, h, s, bs, packed) = gpu_w4a8(bits, sblocks, N, "auto")
    oq, os_ = oracle.quantize_act(bits)
    y, ob = oracle.gemm_w4a8_q4k(oq, os_, sblocks)
    got = out_bits(out)
    bad = np.argwhere(got != ob)
    assert bad.size == 0, "first mismatches %s" % bad[:5].tolist()
    out32, _ = gpu_w4a8(bits, sblocks, N, "auto", out_dtype=torch.float32)
    assert np.array_equal(out_bits(out32), y.view(np.uint32))
    for r in (0, 255, 256, 699):
        o = qg.gemm_w4a8_q4k(q[r:r + 1], h[r:r + 1], s[r:r + 1], bs[r:r + 1], packed, N)
        assert np.array_equal(out_bits(o)[0], got[r])


@pytest.mark.parametrize("M,K,N,tb", [(50, 2048, 1000, 64), (24, 1024, 520, 32), (64, 256, 16, 64)])
def test_w4a8_16_row_tiles(M, K, N, tb):
    # W4A8 GEMMs of at most 64 tokens whose 128-row tiles would fill at most
    # half the SMs run as 16-row tiles (ragged last row tile and token tile);
    # every output against the oracle, and rows alone equal the batch's rows
    from bit_quantized_gemm_gb300 import _lib
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert _lib.prefill_tile_q4k(M, N, 152) == ("16-row", tb)
    x, bits = synth.activations(M + 3 * K, M, K, dtype="bf16", outlier_frac=0.02)
    sblocks = synth.q4k_weights(N + K, N, K)
    out, (q, h, s, bs, packed) = gpu_w4a8(bits, sblocks, N, "auto")
    oq, os_ = oracle.quantize_act(bits)
    y, ob = oracle.gemm_w4a8_q4k(oq, os_, sblocks)
    got = out_bits(out)
    bad = np.argwhere(got != ob)
    assert bad.size == 0, "first mismatches %s" % bad[:5].tolist()
    out32, _ = gpu_w4a8(bits, sblocks, N, "auto", out_dtype=torch.float32)
    assert np.array_equal(out_bits(out32), y.view(np.uint32))
    for r in (0, M - 1):
        o = qg.gemm_w4a8_q4k(q[r:r + 1], h[r:r + 1], s[r:r + 1], bs[r:r + 1], packed, N)
        assert np.array_equal(out_bits(o)[0], got[r])


def test_w4a8_batch_invariance():
    K, N = 512, 96
    xs, bits = synth.activations(31, 150, K, dtype="bf16", outlier_frac=0.01)
    sblocks = synth.q4k_weights(131, N, K)
    full_s, (q, h, s, bs, packed) = gpu_w4a8(bits, sblocks, N, "small")
    full_l, _ = gpu_w4a8(bits, sblocks, N, "large")
    assert np.array_equal(out_bits(full_s), out_bits(full_l))
    for r in (0, 17, 149):
        o = qg.gemm_w4a8_q4k(q[r:r + 1], h[r:r + 1], s[r:r + 1], bs[r:r + 1], packed, N)
        assert np.array_equal(out_bits(o)[0], out_bits(full_l)[r])


def test_quantize_near_ties_and_tiny_scales():
    """Elements whose quotient lands within a few ulps of a half-integer, and
    rows with subnormal scales, take the exact-division branch; all must match
    the oracle bit for bit."""
    rng = np.random.default_rng(17)
    M, K = 64, 512
    x = np.zeros((M, K), np.float32)
    for m in range(M):
        am = np.float32(rng.uniform(0.5, 4.0))
        s = am / np.float32(127)
        h = rng.integers(-126, 126, size=K).astype(np.float32) + np.float32(0.5)
        v = (h * s).astype(np.float32)
        # nudge by -3..3 ulps around each half-integer multiple of s
        steps = rng.integers(-3, 4, size=K)
        v = np.array([np.float32(vi) for vi in v])
        for i in range(K):
            for _ in range(abs(int(steps[i]))):
                v[i] = np.nextafter(v[i], np.float32(np.inf) if steps[i] > 0 else np.float32(-np.inf))
        v[0] = am
        x[m] = v
    x[M - 1] = x[M - 1] * np.float32(1e-39 / 4.0)   # subnormal scale row
    x[M - 2] = x[M - 2] * np.float32(2e-35)        # tiny but normal scale
    q, s, bs, h = run_quant(x, None)
    oq, os_, obs = oracle_quant(x, None)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(bs.cpu().numpy(), obs)
    assert np.array_equal(h.float().cpu().numpy(), oq.astype(np.float32))


def test_bounded_wait_reports_timeout_and_context_survives():
    """Failure detection without a fault: a barrier wait that nothing completes
    gives up after its poll limit, the host reads QG_ETIMEOUT, the word is
    cleared, and the next GEMM still runs and matches the oracle."""
    import time
    from bit_quantized_gemm_gb300 import _lib
    qg.check_device_error()
    t0 = time.time()
    qg.debug_wait_timeout(256)
    with pytest.raises(qg.QGError) as e:
        qg.check_device_error()
    assert e.value.status == _lib.QG_ETIMEOUT
    assert time.time() - t0 < 30
    qg.check_device_error()  # cleared
    M, K, N = 3, 256, 48
    x, bits, blocks = make_w8a8(M, K, N, seed=5)
    out, _ = gpu_w8a8(x, bits, blocks, N, "large")
    oq, os_ = oracle.quantize_act(bits)
    _, ob = oracle.gemm_w8a8_q8_0(oq, os_, blocks)
    assert np.array_equal(out_bits(out), ob)


@pytest.mark.parametrize("M,K,per_row", [(5, 256, True), (37, 2560, False), (16, 17408, True),
                                         (300, 640, False)])
def test_static_quantize_matches_oracle(M, K, per_row):
    """Static (calibrated) scales: saturating int8, block sums and fp16 copy
    bit-exact against the oracle; the W8A8 GEMM on them as well."""
    x, bits = synth.activations(M + K + 3, M, K, dtype="bf16", outlier_frac=0.02)
    rng = np.random.default_rng(M)
    am = np.abs(x).max(axis=1).astype(np.float32)
    # calibrated scales between 0.25x and 1.5x of the row's own absmax/127 (so some rows saturate)
    s = (am / np.float32(127) * rng.uniform(0.25, 1.5, size=M).astype(np.float32)).astype(np.float32)
    s[0] = 0.0
    if not per_row:
        s = s[1:2].copy()
    sd = to_dev(s)
    q, bs, h = qg.quantize_act_static(bf16_dev(bits), sd, block_sums=True, q16=True)
    oq, obs = oracle.quantize_act_static(bits, s, bsum=True)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(bs.cpu().numpy(), obs)
    assert np.array_equal(h.float().cpu().numpy(), oq.astype(np.float32))
    N = 96
    blocks = synth.q8_0_weights(K + 1, N, K)
    srow = s if per_row else np.full(M, s[0], np.float32)
    packed = qg.pack_q8_0(to_dev(blocks), N, K)
    out = qg.gemm_w8a8_q8_0(q, h, to_dev(srow), packed, N)
    _, ob = oracle.gemm_w8a8_q8_0(oq, srow, blocks)
    assert np.array_equal(out_bits(out), ob)


@pytest.mark.parametrize("M,K,N,ldo", [(300, 512, 256, 264), (513, 256, 384, 392),
                                       (300, 512, 256, 259), (2048, 256, 1024, 1032)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_w8a8_padded_output_rows(M, K, N, ldo, out_dtype):
    """Outputs written into rows of pitch ldo > N (bulk tensor stores when the
    pitch is 16-byte aligned, element stores otherwise): the first N columns
    hold the oracle's bits and the padding is left untouched."""
    x, bits, blocks = make_w8a8(M, K, N, seed=M + ldo)
    q, s, _, h = run_quant(x, bits, want_bs=False)
    packed = qg.pack_q8_0(to_dev(blocks), N, K)
    big = torch.full((M, ldo), -7.0, dtype=out_dtype, device=DEV)
    qg.gemm_w8a8_q8_0(q, h, s, packed, N, out=big[:, :N], path="large")
    torch.cuda.synchronize()
    qg.check_device_error()
    oq, os_ = oracle.quantize_act(bits)
    y, ob = oracle.gemm_w8a8_q8_0(oq, os_, blocks)
    want = ob if out_dtype == torch.bfloat16 else y.view(np.uint32)
    assert np.array_equal(out_bits(big[:, :N].contiguous()), want)
    assert bool((big[:, N:] == -7.0).all())


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_w4a8_padded_output_rows(out_dtype):
    M, K, N, ldo = 300, 512, 256, 272
    x, bits = synth.activations(77, M, K, dtype="bf16", outlier_frac=0.01)
    sblocks = synth.q4k_weights(177, N, K)
    q, s, bs, h = qg.quantize_act(bf16_dev(bits), block_sums=True, q16=True)
    packed = qg.pack_q4k(to_dev(sblocks), N, K)
    big = torch.full((M, ldo), -7.0, dtype=out_dtype, device=DEV)
    qg.gemm_w4a8_q4k(q, h, s, bs, packed, N, out=big[:, :N], path="large")
    torch.cuda.synchronize()
    qg.check_device_error()
    oq, os_ = oracle.quantize_act(bits)
    y, ob = oracle.gemm_w4a8_q4k(oq, os_, sblocks)
    want = ob if out_dtype == torch.bfloat16 else y.view(np.uint32)
    assert np.array_equal(out_bits(big[:, :N].contiguous()), want)
    assert bool((big[:, N:] == -7.0).all())


def test_quantize_without_int8_output_and_gemm_from_q16():
    """q = NULL: the quantizer writes only the fp16 copy (plus scales and block
    sums), identical to a full call; the prefill GEMM runs from it alone, and
    the decode kernel, which needs q, is refused."""
    M, K, N = 300, 1024, 256
    x, bits, blocks = make_w8a8(M, K, N, seed=91, outl=0.01)
    q, s, bs, h = qg.quantize_act(bf16_dev(bits), block_sums=True, q16=True)
    q2, s2, bs2, h2 = qg.quantize_act(bf16_dev(bits), block_sums=True, q16=True, int8=False)
    assert q2 is None
    assert torch.equal(s2, s) and torch.equal(bs2, bs) and torch.equal(h2.view(torch.int16), h.view(torch.int16))
    packed = qg.pack_q8_0(to_dev(blocks), N, K)
    out = qg.gemm_w8a8_q8_0(None, h2, s2, packed, N)
    torch.cuda.synchronize()
    oq, os_ = oracle.quantize_act(bits)
    _, ob = oracle.gemm_w8a8_q8_0(oq, os_, blocks)
    assert np.array_equal(out_bits(out), ob)
    with pytest.raises(qg.QGError):
        qg.gemm_w8a8_q8_0(None, h2, s2, packed, N, path="small")
