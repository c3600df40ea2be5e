"""ctypes binding of libqgemm.so (the C ABI declared in include/qgemm.h).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels. PyTorch tensors provide device memory and the current stream.
If the shared library is missing this module raises -- there is no fallback.
"""
import ctypes
import os
import re

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
SO_PATH = os.path.join(HERE, "libqgemm.so")
HEADER = os.path.join(HERE, "..", "include", "qgemm.h")

QG_OK, QG_EINVAL, QG_EALIGN, QG_EUNSUPPORTED, QG_ECUDA, QG_ETIMEOUT, QG_ERANGE = range(7)
QG_BF16, QG_F32 = 0, 1
QG_PATH_AUTO, QG_PATH_SMALL, QG_PATH_LARGE = 0, 1, 2
PATHS = {"auto": QG_PATH_AUTO, "small": QG_PATH_SMALL, "large": QG_PATH_LARGE}

_lib = None


class QGError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("%s (%s)" % (msg, status))
        self.status = status


def load():
    """Load libqgemm.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(SO_PATH):
        raise RuntimeError("libqgemm.so is not built: run `python -m bit_quantized_gemm_gb300.build` "
                           "(or __graft_entry__.build()); there is no CPU fallback")
    L = ctypes.CDLL(SO_PATH)
    P, I64, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    sigs = {
        "qg_status_string": ([I], ctypes.c_char_p),
        "qg_last_error": ([], ctypes.c_char_p),
        "qg_version": ([], I),
        "qg_small_m_max": ([], I64),
        "qg_check_device_error": ([P], I),
        "qg_quantize_act": ([P, I, I64, I64, I64, P, P, P, P, P], I),
        "qg_quantize_act_static": ([P, I, I64, I64, I64, P, I64, P, P, P, P], I),
        "qg_q8_0_packed_bytes": ([I64, I64], SZ),
        "qg_pack_q8_0": ([P, I64, I64, P, P], I),
        "qg_gemm_w8a8_q8_0": ([P, P, P, I64, I64, P, I64, P, I, I64, P], I),
        "qg_gemm_w8a8_q8_0_ex": ([P, P, P, I64, I64, P, I64, P, I, I64, I, P], I),
        "qg_q4k_packed_bytes": ([I64, I64], SZ),
        "qg_pack_q4k": ([P, I64, I64, P, P], I),
        "qg_gemm_w4a8_q4k": ([P, P, P, P, I64, I64, P, I64, P, I, I64, P], I),
        "qg_gemm_w4a8_q4k_ex": ([P, P, P, P, I64, I64, P, I64, P, I, I64, I, P], I),
        "qg_debug_block_sums_q8_0": ([P, P, I64, I64, P, I64, P, I, P], I),
        "qg_debug_block_sums_q4k": ([P, P, I64, I64, P, I64, P, I, P], I),
        "qg_debug_wait_timeout": ([ctypes.c_uint32, P], I),
        "qg_gemm_launch_count": ([I, I64, I64, I64, I], I),
        "qg_linear_workspace_bytes": ([I, I64, I64], SZ),
        "qg_debug_prefill_plan_q8_0": ([I64, I64, I, P, P, P], I),
        "qg_debug_prefill_tile_q4k": ([I64, I64, I, P, P], I),
        "qg_linear_w8a8_q8_0": ([P, I, I64, I64, I64, P, I64, P, I, I64, P, P, SZ, P], I),
        "qg_linear_w4a8_q4k": ([P, I, I64, I64, I64, P, I64, P, I, I64, P, P, SZ, P], I),
        "qg_linear_w8a8_q8_0_noalloc": ([P, I, I64, I64, I64, P, I64, P, I, I64, P, P], I),
        "qg_mxfp4_packed_bytes": ([I64, I64], SZ),
        "qg_pack_mxfp4_q8_0": ([P, I64, I64, P, P], I),
        "qg_gemm_w4a8_mxfp4": ([P, P, P, I64, I64, P, I64, P, I, I64, P], I),
        "qg_linear_w4a8_mxfp4": ([P, I, I64, I64, I64, P, I64, P, I, I64, P, P, SZ, P], I),
    }
    for name, (args, res) in sigs.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _lib = L
    return L


def declared_symbols():
    """Names of the functions include/qgemm.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qg_[a-z0-9_]+)\s*\(", text)))


def _check(status):
    if status != QG_OK:
        L = load()
        raise QGError(status, L.qg_last_error().decode() or L.qg_status_string(status).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(dt):
    if dt == torch.bfloat16:
        return QG_BF16
    if dt == torch.float32:
        return QG_F32
    raise ValueError("dtype must be torch.bfloat16 or torch.float32")


# ----------------------------------------------------------------------- API
def quantize_act(x, block_sums=False, q16=False, out=None, stream=None, int8=True):
    """x: cuda [M, K] bf16/fp32 (rows may be strided) ->
    (q int8 [M,K] or None, scale fp32 [M], block_sums int32 [M,K/32] or None,
    q16 fp16 [M,K] or None). `out` may supply preallocated (q, scale, block_sums,
    q16); int8=False skips q (the prefill GEMM reads q16 alone)."""
    assert x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    if out is None:
        dev = x.device
        q = torch.empty((M, K), dtype=torch.int8, device=dev) if int8 else None
        s = torch.empty((M,), dtype=torch.float32, device=dev)
        bs = torch.empty((M, K // 32), dtype=torch.int32, device=dev) if block_sums else None
        h = torch.empty((M, K), dtype=torch.float16, device=dev) if q16 else None
    else:
        q, s, bs, h = out
    _check(load().qg_quantize_act(_ptr(x), _dtype_code(x.dtype), M, K, x.stride(0), _ptr(q),
                                  _ptr(s), _ptr(bs), _ptr(h), _stream(stream)))
    return q, s, bs, h


def quantize_act_static(x, scale, block_sums=False, q16=False, out=None, stream=None):
    """x: cuda [M, K] bf16/fp32; scale: cuda fp32 [M] (per row) or [1] (all rows)
    -> (q int8, block_sums or None, q16 or None). Values beyond s*127 saturate."""
    assert x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    stride = 0 if scale.numel() == 1 else 1
    if out is None:
        dev = x.device
        q = torch.empty((M, K), dtype=torch.int8, device=dev)
        bs = torch.empty((M, K // 32), dtype=torch.int32, device=dev) if block_sums else None
        h = torch.empty((M, K), dtype=torch.float16, device=dev) if q16 else None
    else:
        q, bs, h = out
    _check(load().qg_quantize_act_static(_ptr(x), _dtype_code(x.dtype), M, K, x.stride(0),
                                         _ptr(scale), stride, _ptr(q), _ptr(bs), _ptr(h),
                                         _stream(stream)))
    return q, bs, h


def q8_0_packed_bytes(N, K):
    return int(load().qg_q8_0_packed_bytes(N, K))


def q4k_packed_bytes(N, K):
    return int(load().qg_q4k_packed_bytes(N, K))


def pack_q8_0(blocks, N, K, stream=None):
    """blocks: cuda uint8 tensor holding N*K/32 Q8_0 blocks of 34 bytes -> packed uint8 tensor."""
    nbytes = q8_0_packed_bytes(N, K)
    if nbytes == 0:
        raise QGError(QG_EINVAL, "bad N/K for Q8_0")
    packed = torch.empty((nbytes,), dtype=torch.uint8, device=blocks.device)
    _check(load().qg_pack_q8_0(_ptr(blocks), N, K, _ptr(packed), _stream(stream)))
    return packed


def pack_q4k(superblocks, N, K, stream=None):
    nbytes = q4k_packed_bytes(N, K)
    if nbytes == 0:
        raise QGError(QG_EINVAL, "bad N/K for Q4_K")
    packed = torch.empty((nbytes,), dtype=torch.uint8, device=superblocks.device)
    _check(load().qg_pack_q4k(_ptr(superblocks), N, K, _ptr(packed), _stream(stream)))
    return packed


def gemm_w8a8_q8_0(q, q16, scale, packed, N, out=None, out_dtype=torch.bfloat16, path="auto",
                   stream=None):
    """q (may be None when the prefill kernel runs), q16, scale from quantize_act."""
    M, K = (q if q is not None else q16).shape
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=scale.device)
    _check(load().qg_gemm_w8a8_q8_0_ex(_ptr(q), _ptr(q16), _ptr(scale), M, K, _ptr(packed), N,
                                       _ptr(out), _dtype_code(out.dtype), out.stride(0),
                                       PATHS[path], _stream(stream)))
    return out


def gemm_w4a8_q4k(q, q16, scale, block_sums, packed, N, out=None, out_dtype=torch.bfloat16,
                  path="auto", stream=None):
    M, K = (q if q is not None else q16).shape
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=scale.device)
    _check(load().qg_gemm_w4a8_q4k_ex(_ptr(q), _ptr(q16), _ptr(scale), _ptr(block_sums), M, K,
                                      _ptr(packed), N, _ptr(out), _dtype_code(out.dtype),
                                      out.stride(0), PATHS[path], _stream(stream)))
    return out


def debug_block_sums(kind, q, q16, packed, N, path, stream=None):
    """Exact per-block integer sums isum[M][N][K/32] as the chosen kernel computes them."""
    M, K = q.shape
    isum = torch.empty((M, N, K // 32), dtype=torch.int32, device=q.device)
    fn = load().qg_debug_block_sums_q8_0 if kind == "q8_0" else load().qg_debug_block_sums_q4k
    _check(fn(_ptr(q), _ptr(q16), M, K, _ptr(packed), N, _ptr(isum), PATHS[path], _stream(stream)))
    return isum


def debug_wait_timeout(polls, stream=None):
    """Launch one bounded wait that is made to run out (failure-detection test)."""
    _check(load().qg_debug_wait_timeout(polls, _stream(stream)))


def check_device_error(stream=None):
    _check(load().qg_check_device_error(_stream(stream)))


def gemm_launch_count(kind, M, K, N, path="auto"):
    """Kernel launches one GEMM call of these sizes makes (kind "q8_0" or "q4k")."""
    return int(load().qg_gemm_launch_count(0 if kind == "q8_0" else 1, M, K, N, PATHS[path]))


def small_m_max():
    return int(load().qg_small_m_max())


def linear_workspace_bytes(kind, M, K):
    """Workspace bytes a linear_* call of these sizes needs."""
    return int(load().qg_linear_workspace_bytes(0 if kind == "q8_0" else 1, M, K))


def _linear(kind, x, packed, N, out, out_dtype, scale_out, workspace, stream, fn=None):
    assert x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=x.device)
    need = linear_workspace_bytes(kind, M, K)
    if workspace is None and need:
        workspace = torch.empty((need,), dtype=torch.uint8, device=x.device)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if fn is None:
        fn = load().qg_linear_w8a8_q8_0 if kind == "q8_0" else load().qg_linear_w4a8_q4k
    _check(fn(_ptr(x), _dtype_code(x.dtype), M, K, x.stride(0), _ptr(packed), N, _ptr(out),
              _dtype_code(out.dtype), out.stride(0), _ptr(scale_out), _ptr(workspace), nbytes,
              _stream(stream)))
    return out


def linear_w8a8_q8_0(x, packed, N, out=None, out_dtype=torch.bfloat16, scale_out=None,
                     workspace=None, stream=None):
    """The whole layer: x cuda [M, K] bf16/fp32 (rows may be strided) -> out [M, N].
    Quantize, then GEMM, through `workspace` (allocated here when not given);
    for M <= small_m_max() the GEMM overlaps the quantize kernel (programmatic
    dependent launch). scale_out: optional fp32 [M] receiving the row scales."""
    return _linear("q8_0", x, packed, N, out, out_dtype, scale_out, workspace, stream)


def linear_w4a8_q4k(x, packed, N, out=None, out_dtype=torch.bfloat16, scale_out=None,
                    workspace=None, stream=None):
    """As linear_w8a8_q8_0, with Q4_K weights."""
    return _linear("q4k", x, packed, N, out, out_dtype, scale_out, workspace, stream)


def pack_mxfp4_q8_0(blocks, N, K, stream=None):
    """Q8_0 blocks (cuda uint8, N*K/32 x 34 bytes) converted to MXFP4 and packed
    (lossy: see include/qgemm.h). check_device_error() raises QG_ERANGE when a
    block scale does not fit the decode kernels' fp16 scales."""
    nbytes = int(load().qg_mxfp4_packed_bytes(N, K))
    if nbytes == 0:
        raise QGError(QG_EINVAL, "bad N/K for MXFP4")
    packed = torch.empty((nbytes,), dtype=torch.uint8, device=blocks.device)
    _check(load().qg_pack_mxfp4_q8_0(_ptr(blocks), N, K, _ptr(packed), _stream(stream)))
    return packed


def gemm_w4a8_mxfp4(q, q16, scale, packed, N, out=None, out_dtype=torch.bfloat16, stream=None):
    """As gemm_w8a8_q8_0 (AUTO path), on weights from pack_mxfp4_q8_0."""
    M, K = (q if q is not None else q16).shape
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=(q if q is not None else q16).device)
    _check(load().qg_gemm_w4a8_mxfp4(_ptr(q), _ptr(q16), _ptr(scale), M, K, _ptr(packed), N,
                                     _ptr(out), _dtype_code(out.dtype), out.stride(0),
                                     _stream(stream)))
    return out


def linear_w4a8_mxfp4(x, packed, N, out=None, out_dtype=torch.bfloat16, scale_out=None,
                      workspace=None, stream=None):
    """As linear_w8a8_q8_0, on weights from pack_mxfp4_q8_0."""
    return _linear("q8_0", x, packed, N, out, out_dtype, scale_out, workspace, stream,
                   fn=load().qg_linear_w4a8_mxfp4)


def linear_noalloc_scratch_bytes():
    """QG_LINEAR_NOALLOC_SCRATCH_BYTES, read from include/qgemm.h."""
    m = re.search(r"#define\s+QG_LINEAR_NOALLOC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)",
                  open(HEADER).read())
    return int(m.group(1)) << int(m.group(2))


def linear_w8a8_q8_0_noalloc(x, packed, N, out=None, out_dtype=torch.bfloat16, scale_out=None,
                             stream=None):
    """As linear_w8a8_q8_0, with the library's static scratch in place of a
    workspace: the library call allocates nothing (`out` is allocated here
    when not given). Sizes are limited to linear_noalloc_scratch_bytes() of
    scratch; calls that overlap on the GPU share the scratch and race."""
    assert x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=x.device)
    _check(load().qg_linear_w8a8_q8_0_noalloc(
        _ptr(x), _dtype_code(x.dtype), M, K, x.stride(0), _ptr(packed), N, _ptr(out),
        _dtype_code(out.dtype), out.stride(0), _ptr(scale_out), _stream(stream)))
    return out


def prefill_tile_q4k(M, N, sms):
    """The W4A8 GEMM's tiles for M x N on `sms` SMs: ("tensor" / "16-row", token width)."""
    kind = ctypes.c_int()
    tokens = ctypes.c_int()
    _check(load().qg_debug_prefill_tile_q4k(M, N, sms, ctypes.byref(kind), ctypes.byref(tokens)))
    return {1: "tensor", 2: "16-row"}[kind.value], tokens.value


def prefill_plan(M, N, sms):
    """The W8A8 prefill wave plan on `sms` SMs: (rows of the 256-token launch,
    narrow-part kind: None / "tensor" / "16-row", its token-tile width)."""
    rows = ctypes.c_int64()
    kind = ctypes.c_int()
    tokens = ctypes.c_int()
    _check(load().qg_debug_prefill_plan_q8_0(M, N, sms, ctypes.byref(rows), ctypes.byref(kind),
                                             ctypes.byref(tokens)))
    return rows.value, {0: None, 1: "tensor", 2: "16-row"}[kind.value], tokens.value
