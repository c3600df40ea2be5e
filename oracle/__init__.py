"""Plain CPU oracle for the exact int8 / W4A8 quantized linear layer.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this package; the library never does. The
arithmetic lives in ``oracle.c`` (plain C, one fused multiply-add per K block,
built with ``-ffp-contract=off``); this module only compiles it and marshals
numpy arrays through ctypes. It shares no code with the CUDA library.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

_FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
          "-fPIC", "-shared", "-Wall"]


def build(force=False):
    """Compile oracle.c into liboracle.so (gcc, a second or two)."""
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= max(
            os.path.getmtime(src), os.path.getmtime(os.path.join(_HERE, "oracle.h"))):
        return _SO
    tmp = _SO + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", *_FLAGS, src, "-o", tmp, "-lm"])
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_f16_to_f32.restype = ctypes.c_float
        L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
        L.orc_f32_to_bf16.restype = ctypes.c_uint16
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f32.restype = ctypes.c_float
        L.orc_quantize_act.argtypes = [P, I, I64, I64, P, P, P]
        L.orc_quantize_act_static.argtypes = [P, I, I64, I64, P, I64, P, P]
        L.orc_gemm_w8a8_q8_0.argtypes = [P, P, I64, I64, P, I64, P, P]
        L.orc_block_sums_q8_0.argtypes = [P, I64, I64, P, I64, P]
        L.orc_q4k_decode.argtypes = [P, P, P, P, P, P, P]
        L.orc_gemm_w4a8_q4k.argtypes = [P, P, I64, I64, P, I64, P, P]
        L.orc_block_sums_q4k.argtypes = [P, I64, I64, P, I64, P, P]
        L.orc_mxfp4_from_q8_0.argtypes = [P, I64, I64, P, P]
        L.orc_e2m1_value.argtypes = [I]
        L.orc_e2m1_value.restype = ctypes.c_double
        L.orc_gemm_w4a8_mxfp4.argtypes = [P, P, I64, I64, P, P, I64, P, P]
        L.orc_num_threads.restype = I
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    assert a.dtype == dtype, (a.dtype, dtype)
    return a


def num_threads():
    return lib().orc_num_threads()


def f16_to_f32(bits):
    return float(lib().orc_f16_to_f32(int(bits)))


def f32_to_bf16(x):
    return int(lib().orc_f32_to_bf16(float(x)))


def quantize_act(x, bsum=False):
    """x: float32 [M,K] or uint16 bf16 bits [M,K] -> (q int8, s fp32[, bsum int32])."""
    if x.dtype == np.uint16:
        is_bf16 = 1
    else:
        x = x.astype(np.float32, copy=False)
        is_bf16 = 0
    x = np.ascontiguousarray(x)
    M, K = x.shape
    q = np.empty((M, K), np.int8)
    s = np.empty((M,), np.float32)
    bs = np.empty((M, K // 32), np.int32) if bsum else None
    lib().orc_quantize_act(_p(x), is_bf16, M, K, _p(q), _p(s), _p(bs))
    return (q, s, bs) if bsum else (q, s)


def quantize_act_static(x, scale, bsum=False):
    """x: float32 [M,K] or uint16 bf16 bits; scale: float32 [M] (per row) or [1]
    (one for all rows) -> (q int8[, bsum int32])."""
    if x.dtype == np.uint16:
        is_bf16 = 1
    else:
        x = x.astype(np.float32, copy=False)
        is_bf16 = 0
    x = np.ascontiguousarray(x)
    M, K = x.shape
    scale = _c(np.atleast_1d(scale).astype(np.float32), np.float32)
    stride = 0 if scale.shape[0] == 1 else 1
    assert stride == 0 or scale.shape[0] == M
    q = np.empty((M, K), np.int8)
    bs = np.empty((M, K // 32), np.int32) if bsum else None
    lib().orc_quantize_act_static(_p(x), is_bf16, M, K, _p(scale), stride, _p(q), _p(bs))
    return (q, bs) if bsum else q


def gemm_w8a8_q8_0(qa, sa, blocks):
    """qa int8 [M,K], sa fp32 [M], blocks uint8 [N, K/32, 34] -> (y fp32 [M,N], out bf16 bits [M,N])."""
    qa = _c(qa, np.int8)
    sa = _c(sa, np.float32)
    blocks = _c(blocks, np.uint8)
    M, K = qa.shape
    N = blocks.shape[0]
    assert blocks.shape == (N, K // 32, 34)
    y = np.empty((M, N), np.float32)
    out = np.empty((M, N), np.uint16)
    lib().orc_gemm_w8a8_q8_0(_p(qa), _p(sa), M, K, _p(blocks), N, _p(y), _p(out))
    return y, out


def block_sums_q8_0(qa, blocks):
    qa = _c(qa, np.int8)
    blocks = _c(blocks, np.uint8)
    M, K = qa.shape
    N = blocks.shape[0]
    isum = np.empty((M, N, K // 32), np.int32)
    lib().orc_block_sums_q8_0(_p(qa), M, K, _p(blocks), N, _p(isum))
    return isum


def q4k_decode(sb):
    """One 144-byte super-block -> dict of decoded fields and fp64 weights."""
    sb = _c(sb, np.uint8)
    assert sb.shape == (144,)
    w = np.empty(256, np.float64)
    d = ctypes.c_float()
    dmin = ctypes.c_float()
    sc = np.empty(8, np.uint8)
    mn = np.empty(8, np.uint8)
    q = np.empty(256, np.uint8)
    lib().orc_q4k_decode(_p(sb), _p(w), ctypes.byref(d), ctypes.byref(dmin), _p(sc), _p(mn), _p(q))
    return {"w": w, "d": d.value, "dmin": dmin.value, "sc": sc, "m": mn, "q": q}


def gemm_w4a8_q4k(qa, sa, sblocks):
    """qa int8 [M,K], sa fp32 [M], sblocks uint8 [N, K/256, 144] -> (y, out bf16 bits)."""
    qa = _c(qa, np.int8)
    sa = _c(sa, np.float32)
    sblocks = _c(sblocks, np.uint8)
    M, K = qa.shape
    N = sblocks.shape[0]
    assert sblocks.shape == (N, K // 256, 144)
    y = np.empty((M, N), np.float32)
    out = np.empty((M, N), np.uint16)
    lib().orc_gemm_w4a8_q4k(_p(qa), _p(sa), M, K, _p(sblocks), N, _p(y), _p(out))
    return y, out


def block_sums_q4k(qa, sblocks):
    qa = _c(qa, np.int8)
    sblocks = _c(sblocks, np.uint8)
    M, K = qa.shape
    N = sblocks.shape[0]
    isum = np.empty((M, N, K // 32), np.int32)
    asum = np.empty((M, K // 32), np.int32)
    lib().orc_block_sums_q4k(_p(qa), M, K, _p(sblocks), N, _p(isum), _p(asum))
    return isum, asum


def mxfp4_from_q8_0(blocks):
    """Q8_0 blocks uint8 [N, K/32, 34] -> (E2M1 codes uint8 [N, K], exponents uint8 [N, K/32])."""
    blocks = _c(blocks, np.uint8)
    N, B, _ = blocks.shape
    K = B * 32
    codes = np.empty((N, K), np.uint8)
    E = np.empty((N, B), np.uint8)
    lib().orc_mxfp4_from_q8_0(_p(blocks), N, K, _p(codes), _p(E))
    return codes, E


def e2m1_value(code):
    return lib().orc_e2m1_value(int(code))


def gemm_w4a8_mxfp4(qa, sa, codes, E):
    """qa int8 [M,K], sa fp32 [M], codes uint8 [N,K], E uint8 [N,K/32] -> (y fp32, out bf16 bits)."""
    qa = _c(qa, np.int8)
    sa = _c(sa, np.float32)
    codes = _c(codes, np.uint8)
    E = _c(E, np.uint8)
    M, K = qa.shape
    N = codes.shape[0]
    assert codes.shape == (N, K) and E.shape == (N, K // 32)
    y = np.empty((M, N), np.float32)
    out = np.empty((M, N), np.uint16)
    lib().orc_gemm_w4a8_mxfp4(_p(qa), _p(sa), M, K, _p(codes), _p(E), N, _p(y), _p(out))
    return y, out
