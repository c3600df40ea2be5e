"""Host-side checks of the C ABI (no GPU): the shared library loads, exports
every function include/qgemm.h declares, and rejects bad arguments with the
documented status before touching the GPU."""
import ctypes
import subprocess

import pytest

import bit_quantized_gemm_gb300 as qg
from bit_quantized_gemm_gb300 import _lib
from bit_quantized_gemm_gb300 import build as qbuild

P = ctypes.c_void_p


@pytest.fixture(scope="module")
def L():
    qbuild.build()
    return _lib.load()


def test_exports_every_declared_symbol(L):
    names = _lib.declared_symbols()
    assert len(names) >= 18
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.SO_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        getattr(L, n)


def test_status_strings_and_constants(L):
    for s in range(6):
        assert L.qg_status_string(s).decode().startswith("QG_")
    assert L.qg_version() == 10000
    assert L.qg_small_m_max() == 16


def test_packed_sizes(L):
    # sizes cover the int8 stream, the scales and the fp16 copy
    for N, K in [(1, 32), (17, 96), (128, 256), (9728, 2560)]:
        b = L.qg_q8_0_packed_bytes(N, K)
        assert b % 256 == 0 and b >= N * K * 3 + N * (K // 32) * 6
    for N, K in [(1, 256), (33, 512), (17408, 5120)]:
        b = L.qg_q4k_packed_bytes(N, K)
        assert b % 256 == 0 and b >= N * K * 2 + N * K // 2 + N * (K // 32) * 8
    for N, K in [(0, 32), (4, 0), (4, 48), (4, 65536 + 32), (-1, 32)]:
        assert L.qg_q8_0_packed_bytes(N, K) == 0
    for N, K in [(4, 128), (4, 32), (0, 256)]:
        assert L.qg_q4k_packed_bytes(N, K) == 0


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def _gemm(L, q=FAKE, q16=FAKE, s=FAKE, M=4, K=256, w=FAKE, N=16, out=FAKE, dt=0, ldo=16, path=0):
    return L.qg_gemm_w8a8_q8_0_ex(P(q), P(q16), P(s), M, K, P(w), N, P(out), dt, ldo, path, None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), _lib.QG_EINVAL), (dict(out=0), _lib.QG_EINVAL), (dict(w=0), _lib.QG_EINVAL),
    (dict(M=0), _lib.QG_EINVAL), (dict(N=0), _lib.QG_EINVAL), (dict(K=48), _lib.QG_EINVAL),
    (dict(K=0), _lib.QG_EINVAL), (dict(K=65536 + 32), _lib.QG_EINVAL),
    (dict(ldo=8), _lib.QG_EINVAL), (dict(dt=7), _lib.QG_EINVAL), (dict(path=9), _lib.QG_EINVAL),
    (dict(q=FAKE + 8), _lib.QG_EALIGN), (dict(out=FAKE + 2), _lib.QG_EALIGN),
    (dict(w=FAKE + 16), _lib.QG_EALIGN), (dict(q16=FAKE + 4), _lib.QG_EALIGN),
    (dict(M=17, q16=0), _lib.QG_EINVAL), (dict(M=4, q16=0, path=2), _lib.QG_EINVAL),
    # q may be NULL only when the prefill kernel runs
    (dict(M=17, q=0, path=1), _lib.QG_EINVAL), (dict(M=16, q=0), _lib.QG_EINVAL),
])
def test_gemm_argument_validation(L, kw, status):
    assert _gemm(L, **kw) == status
    assert L.qg_last_error().decode()


def test_q4k_and_quantize_validation(L):
    g = L.qg_gemm_w4a8_q4k_ex
    assert g(P(FAKE), P(FAKE), P(FAKE), None, 4, 256, P(FAKE), 16, P(FAKE), 0, 16, 0, None) == _lib.QG_EINVAL
    assert g(P(FAKE), P(FAKE), P(FAKE), P(FAKE), 4, 288, P(FAKE), 16, P(FAKE), 0, 16, 0, None) == _lib.QG_EINVAL
    assert g(P(FAKE), P(FAKE), P(FAKE), P(FAKE + 8), 4, 256, P(FAKE), 16, P(FAKE), 0, 16, 0, None) == _lib.QG_EALIGN
    qa = L.qg_quantize_act
    assert qa(None, 0, 4, 64, 64, P(FAKE), P(FAKE), None, None, None) == _lib.QG_EINVAL
    assert qa(P(FAKE), 0, 4, 40, 40, P(FAKE), P(FAKE), None, None, None) == _lib.QG_EINVAL
    assert qa(P(FAKE), 0, 4, 64, 32, P(FAKE), P(FAKE), None, None, None) == _lib.QG_EINVAL
    assert qa(P(FAKE), 0, 4, 64, 68, P(FAKE), P(FAKE), None, None, None) == _lib.QG_EALIGN
    assert qa(P(FAKE + 4), 1, 4, 64, 64, P(FAKE), P(FAKE), None, None, None) == _lib.QG_EALIGN
    assert qa(P(FAKE), 5, 4, 64, 64, P(FAKE), P(FAKE), None, None, None) == _lib.QG_EINVAL
    assert qa(P(FAKE), 0, 0, 64, 64, P(FAKE), P(FAKE), None, None, None) == _lib.QG_EINVAL
    # q may be NULL when q16 is written, not both
    assert qa(P(FAKE), 0, 4, 64, 64, None, P(FAKE), None, None, None) == _lib.QG_EINVAL
    assert qa(P(FAKE), 0, 4, 64, 64, None, P(FAKE), None, P(FAKE + 8), None) == _lib.QG_EALIGN
    qs = L.qg_quantize_act_static
    assert qs(P(FAKE), 0, 4, 64, 64, P(FAKE), 1, None, None, None, None) == _lib.QG_EINVAL
    pk = L.qg_pack_q8_0
    assert pk(P(FAKE), 4, 64, P(FAKE + 16), None) == _lib.QG_EALIGN
    assert pk(None, 4, 64, P(FAKE), None) == _lib.QG_EINVAL
    assert L.qg_pack_q4k(P(FAKE), 4, 128, P(FAKE), None) == _lib.QG_EINVAL
    db = L.qg_debug_block_sums_q8_0
    assert db(P(FAKE), P(FAKE), 4096, 4096, P(FAKE), 4096, P(FAKE), 0, None) == _lib.QG_EINVAL


def test_binding_raises_without_gpu_work(L):
    with pytest.raises(qg.QGError):
        _lib._check(_lib.QG_EINVAL)


def test_timeout_probe_validation(L):
    assert L.qg_debug_wait_timeout(0, None) == _lib.QG_EINVAL
    assert L.qg_debug_wait_timeout((1 << 20) + 1, None) == _lib.QG_EINVAL


def test_static_quantize_validation(L):
    qs = L.qg_quantize_act_static
    assert qs(P(FAKE), 0, 4, 64, 64, None, 1, P(FAKE), None, None, None) == _lib.QG_EINVAL
    assert qs(P(FAKE), 0, 4, 64, 64, P(FAKE), 2, P(FAKE), None, None, None) == _lib.QG_EINVAL
    assert qs(P(FAKE), 0, 4, 48, 48, P(FAKE), 1, P(FAKE), None, None, None) == _lib.QG_EINVAL
    assert qs(P(FAKE), 0, 4, 64, 64, P(FAKE), 1, P(FAKE), P(FAKE + 4), None, None) == _lib.QG_EALIGN


def test_gemm_launch_count_host_rules(L):
    # the decode kernel takes up to 16 rows per launch; invalid requests give 0
    assert qg.gemm_launch_count("q8_0", 1, 5120, 17408) == 1
    assert qg.gemm_launch_count("q8_0", 16, 5120, 17408) == 1
    assert qg.gemm_launch_count("q8_0", 40, 5120, 17408, path="small") == 3
    assert qg.gemm_launch_count("q4k", 33, 5120, 17408, path="small") == 3
    assert L.qg_gemm_launch_count(0, 0, 5120, 17408, 0) == 0
    assert L.qg_gemm_launch_count(0, 8, 5100, 17408, 0) == 0      # K not a multiple of 32
    assert L.qg_gemm_launch_count(1, 8, 4096 + 32, 17408, 0) == 0  # K not a multiple of 256
    assert L.qg_gemm_launch_count(2, 8, 5120, 17408, 0) == 0
    assert L.qg_gemm_launch_count(0, 8, 5120, 17408, 7) == 0
