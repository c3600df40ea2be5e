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


def _align(v, a=256):
    return (v + a - 1) // a * a


def test_linear_workspace_layout(L):
    # the documented layout: row scales, then the int8 activations (decode
    # kernel, M <= 16) or their fp16 copy (prefill kernel), then (W4A8) the
    # block sums, each part 256-byte aligned
    for M, K in [(1, 256), (8, 5120), (16, 17408), (17, 256), (2048, 2560), (4096, 5120)]:
        act = M * K if M <= 16 else 2 * M * K
        base = _align(M * 4) + act
        assert L.qg_linear_workspace_bytes(0, M, K) == _align(base)
        assert L.qg_linear_workspace_bytes(1, M, K) == _align(_align(base) + M * (K // 32) * 4)
    assert L.qg_linear_workspace_bytes(2, 9, 256) == 0      # unknown weights kind
    assert L.qg_linear_workspace_bytes(0, 9, 48) == 0       # K not a multiple of 32
    assert L.qg_linear_workspace_bytes(1, 9, 288) == 0      # K not a multiple of 256
    assert L.qg_linear_workspace_bytes(0, 0, 256) == 0
    assert qg.linear_workspace_bytes("q8_0", 17, 256) == L.qg_linear_workspace_bytes(0, 17, 256)


def _linear(L, kind=0, x=FAKE, xdt=0, M=4, K=256, ldx=256, w=FAKE, N=16, out=FAKE, odt=0,
            ldo=16, sc=None, ws=None, wsb=0):
    fn = L.qg_linear_w8a8_q8_0 if kind == 0 else L.qg_linear_w4a8_q4k
    return fn(P(x), xdt, M, K, ldx, P(w), N, P(out), odt, ldo,
              None if sc is None else P(sc), None if ws is None else P(ws), wsb, None)


@pytest.mark.parametrize("kw,status", [
    (dict(x=0), _lib.QG_EINVAL), (dict(w=0), _lib.QG_EINVAL), (dict(out=0), _lib.QG_EINVAL),
    (dict(xdt=3), _lib.QG_EINVAL), (dict(odt=3), _lib.QG_EINVAL), (dict(M=0), _lib.QG_EINVAL),
    (dict(N=0), _lib.QG_EINVAL), (dict(K=48, ldx=48), _lib.QG_EINVAL),
    (dict(kind=1, K=288, ldx=288), _lib.QG_EINVAL), (dict(ldx=128), _lib.QG_EINVAL),
    (dict(ldo=8), _lib.QG_EINVAL),
    (dict(x=FAKE + 8), _lib.QG_EALIGN), (dict(ldx=260), _lib.QG_EALIGN),
    (dict(xdt=1, ldx=258), _lib.QG_EALIGN), (dict(out=FAKE + 2), _lib.QG_EALIGN),
    (dict(w=FAKE + 16), _lib.QG_EALIGN), (dict(sc=FAKE + 2), _lib.QG_EALIGN),
    # a workspace of the reported size is required
    (dict(M=1), _lib.QG_EINVAL), (dict(M=9, ws=FAKE, wsb=1024), _lib.QG_EINVAL),
    (dict(M=17, ws=FAKE + 128, wsb=1 << 20), _lib.QG_EALIGN),
])
def test_linear_argument_validation(L, kw, status):
    assert _linear(L, **kw) == status
    assert L.qg_last_error().decode()


def test_plain_c_client_links_and_runs(L, tmp_path):
    # the boundary is a C ABI: a C program built with gcc against the header
    # and linked to the library runs its host-only checks (no GPU needed)
    import os
    import shutil
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    libdir = os.path.dirname(_lib.SO_PATH)
    exe = str(tmp_path / "abi_host_check")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(root, "include"),
                    os.path.join(here, "c", "abi_host_check.c"), "-L", libdir, "-lqgemm",
                    "-Wl,-rpath," + libdir, "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 failure(s)" in r.stdout
    # the same client as C++: the header's extern "C" block gives unmangled names
    gxx = shutil.which("g++")
    if gxx is not None:
        exe_cc = str(tmp_path / "abi_host_check_cc")
        subprocess.run([gxx, "-x", "c++", "-std=c++17", "-Wall", "-Werror",
                        "-I", os.path.join(root, "include"),
                        os.path.join(here, "c", "abi_host_check.c"), "-x", "none", "-L", libdir,
                        "-lqgemm", "-Wl,-rpath," + libdir, "-o", exe_cc], check=True)
        r = subprocess.run([exe_cc], capture_output=True, text=True)
        assert r.returncode == 0 and "0 failure(s)" in r.stdout, r.stdout + r.stderr


def test_prefill_wave_plan_on_152_sms(L):
    # the plans the benchmark's and the workloads' shapes get on GB300 (152 SMs)
    plan = _lib.prefill_plan
    assert plan(2048, 9728, 152) == (9728, None, 0)        # 4B gate/up: 4 whole waves
    assert plan(2048, 2560, 152) == (2432, "16-row", 64)   # 4B down: 1 wave + 128-row tail
    assert plan(8192, 17408, 152) == (17408, None, 0)      # 27B gate/up
    assert plan(32, 5120, 152) == (0, "16-row", 32)        # narrow prefill: 16-row tiles
    assert plan(64, 17408, 152) == (0, "tensor", 64)       # 64-token tensor-memory tiles
    assert plan(64, 5120, 152) == (0, "16-row", 64)        # 40 row tiles: 16-row tiles, one wave


def test_w4a8_tiles_on_152_sms(L):
    # 256-token tiles where their whole waves, at 1.27 each, beat 128-token
    # ones; 16-row tiles for at most 64 tokens when 128-row tiles fill at most
    # half the SMs
    tile = _lib.prefill_tile_q4k
    assert tile(4096, 17408, 152) == ("tensor", 256)   # 15 waves against 29
    assert tile(4096, 5120, 152) == ("tensor", 256)    # 5 against 9
    assert tile(1024, 5120, 152) == ("tensor", 256)    # 2 against 3
    assert tile(256, 17408, 152) == ("tensor", 256)    # 1 against 2
    assert tile(256, 5120, 152) == ("tensor", 128)     # 40 or 80 tiles: one wave either way
    assert tile(128, 17408, 152) == ("tensor", 128)    # one token tile either way
    assert tile(65, 129, 152) == ("tensor", 128)
    assert tile(700, 5000, 152) == ("tensor", 256)     # the GPU parity case of 256-token tiles
    assert tile(64, 17408, 152) == ("tensor", 64)      # 136 row tiles fill more than half the SMs
    assert tile(32, 17408, 152) == ("tensor", 32)
    assert tile(64, 5120, 152) == ("16-row", 64)       # 40 row tiles
    assert tile(33, 5120, 152) == ("16-row", 64)
    assert tile(32, 5120, 152) == ("16-row", 32)
    assert tile(17, 9728, 152) == ("16-row", 32)       # 76 row tiles: half the SMs
    assert tile(17, 9856, 152) == ("tensor", 32)       # 77
    for M in (17, 40, 64, 65, 100, 300, 1000, 2048, 8192):
        for N in (16, 130, 5120, 17408):
            for sms in (1, 8, 148, 152):
                kind, t = tile(M, N, sms)
                nt = -(-N // 128)
                if M <= 64:
                    assert (kind == "16-row") == (2 * nt <= sms)
                    assert t == (32 if M <= 32 else 64)
                    continue
                assert kind == "tensor" and t in (128, 256)
                w128, w256 = -(-(-(-M // 128) * nt) // sms), -(-(-(-M // 256) * nt) // sms)
                assert (t == 256) == (127 * w256 < 100 * w128)
    with pytest.raises(qg.QGError):
        tile(0, 128, 152)
    with pytest.raises(qg.QGError):
        tile(64, 128, 0)


def test_prefill_wave_plan_invariants(L):
    import random
    rng = random.Random(5)
    for _ in range(400):
        M = rng.choice([17, 33, 64, 100, 256, 300, 1000, 2048, 4096, 8192])
        N = rng.choice([16, 130, 520, 1000, 2560, 5120, 9728, 17408]) + rng.choice([0, 0, 7])
        sms = rng.choice([1, 8, 132, 148, 152, 160])
        rows, kind, tokens = _lib.prefill_plan(M, N, sms)
        assert 0 <= rows <= N
        assert rows == N or rows % 128 == 0        # whole 128-row tiles, or everything
        assert (kind is None) == (rows == N)       # a second launch only for leftover rows
        assert tokens == 0 if kind is None else tokens in (32, 64, 128)
    with pytest.raises(qg.QGError):
        _lib.prefill_plan(0, 128, 152)
    with pytest.raises(qg.QGError):
        _lib.prefill_plan(64, 128, 0)
