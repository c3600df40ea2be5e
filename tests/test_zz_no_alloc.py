"""The W8A8 layer call that allocates nothing (qg_linear_w8a8_q8_0_noalloc).

Some callers cannot call cudaMalloc: a host that passes a plug-in only its
input and output buffers through a C interface, or a latency-critical loop
where an allocation (which synchronizes the device) is not acceptable. For
them the library keeps the layer call's scratch (row scales and quantized
activations) in one fixed-size module-scope device array instead of a
caller's workspace. These tests call that entry point through the C ABI and
require the bits of qg_linear_w8a8_q8_0 with a workspace, on consecutive
calls that reuse the shared scratch, and a clean rejection of sizes beyond
the array.

The file is named to run last, so a run that stops at the first failure has
run every other test before it.
"""
import numpy as np
import pytest
import torch

import bit_quantized_gemm_gb300 as qg
from bit_quantized_gemm_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from bit_quantized_gemm_gb300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


def _layer(M, K, N, seed):
    _, bits = synth.activations(seed, M, K, dtype="bf16", outlier_frac=0.01)
    x = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    blocks = torch.from_numpy(synth.q8_0_weights(seed + 100, N, K)).to(DEV)
    return x, qg.pack_q8_0(blocks, N, K)


def test_noalloc_matches_workspace_call_on_consecutive_calls():
    # decode-sized (int8 scratch), prefill-sized (fp16 scratch), then the
    # decode shape again on new rows: each call overwrites what the previous
    # one left in the shared scratch
    cases = [(8, 5120, 1000, 1), (100, 2560, 520, 2), (8, 5120, 1000, 3)]
    packs = {}
    for M, K, N, seed in cases:
        cap = qg.linear_noalloc_scratch_bytes()
        assert qg.linear_workspace_bytes("q8_0", M, K) <= cap
        x, packed = _layer(M, K, N, seed)
        packs[(K, N)] = packed
        s_ref = torch.empty((M,), dtype=torch.float32, device=DEV)
        s_got = torch.full((M,), -1.0, dtype=torch.float32, device=DEV)
        ref = qg.linear_w8a8_q8_0(x, packed, N, scale_out=s_ref)
        got = qg.linear_w8a8_q8_0_noalloc(x, packed, N, scale_out=s_got)
        ref32 = qg.linear_w8a8_q8_0(x, packed, N, out_dtype=torch.float32)
        got32 = qg.linear_w8a8_q8_0_noalloc(x, packed, N, out_dtype=torch.float32)
        torch.cuda.synchronize()
        qg.check_device_error()
        assert np.array_equal(_bits(got), _bits(ref)), (M, K, N)
        assert np.array_equal(got32.cpu().numpy().view(np.uint32),
                              ref32.cpu().numpy().view(np.uint32)), (M, K, N)
        assert np.array_equal(s_got.cpu().numpy().view(np.uint32),
                              s_ref.cpu().numpy().view(np.uint32))


def test_noalloc_rejects_sizes_beyond_the_scratch():
    cap = qg.linear_noalloc_scratch_bytes()
    M, K, N = 1024, 8192, 64
    assert qg.linear_workspace_bytes("q8_0", M, K) > cap
    x, packed = _layer(M, K, N, 4)
    out = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(qg.QGError) as e:
        qg.linear_w8a8_q8_0_noalloc(x, packed, N, out=out)
    assert e.value.status == 1  # QG_EINVAL: rejected on the host
    assert "scratch" in str(e.value)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())  # nothing was launched
