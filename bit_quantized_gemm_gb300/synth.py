"""Seeded synthetic inputs for the quantized linear layer.

This module only draws random numbers and encodes them into the storage
formats the layer consumes; it holds none of the layer's own arithmetic
(activation quantization, block sums, scale epilogue). Both the library's
tests/benchmarks and the CPU oracle are fed from here.

Workload recipe (stands in for the 4B/27B-class models' projections of the
StartLux-Prism README, "Supported models and GPUs"; no dataset or weights):
  * activations: standard normal, drawn as float32 by numpy's PCG64, rounded
    to bf16 (round-to-nearest-even) unless fp32 is asked for; optionally 1%
    of the K channels (chosen by the seed, the same for every row) scaled
    x20 ("outlier channels"), optionally right-padded rows (zero rows after
    each sequence's length, one sequence per block of slots);
  * weights: normal with std 0.02, encoded as Q8_0 blocks or Q4_K
    super-blocks by the simple encoders below.

Q8_0 block (34 bytes): fp16 d (little endian), then 32 int8 q; d is the fp16
rounding of absmax/127 over the block and q = clamp(rint(w/d), -127, 127)
(q = 0 when d = 0).

Q4_K super-block (144 bytes, canonical packing of this library):
  bytes 0-1 d (fp16), 2-3 dmin (fp16), 4-15 a 96-bit little-endian string of
  sixteen 6-bit fields (field f at bits [6f, 6f+6): sc_0..sc_7 then
  m_0..m_7), 16-143 nibbles (weight j: low nibble of byte 16+j/2 for even j,
  high nibble for odd j). Weight = d*sc_i*q - dmin*m_i, q in [0, 15].
  Encoder per sub-block i: lo = min(0, min w), hi = max w,
  scale_i = (hi-lo)/15, off_i = -lo; d = fp16(max scale_i / 63),
  dmin = fp16(max off_i / 63); sc_i = clamp(rint(scale_i/d), 0, 63),
  m_i = clamp(rint(off_i/dmin), 0, 63);
  q = clamp(rint((w + dmin*m_i) / (d*sc_i)), 0, 15); a zero denominator gives 0.
"""
import numpy as np
import torch

QBLK = 32
Q8_0_BYTES = 34
Q4K_WEIGHTS = 256
Q4K_BYTES = 144


def _bf16_round(x32):
    """float32 array -> (float32 values rounded to bf16, uint16 bf16 bits)."""
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16).copy()
    vals = t.to(torch.float32).numpy()
    return vals, bits


def activations(seed, M, K, *, dtype="bf16", outlier_frac=0.0, outlier_mult=20.0,
                seq_slots=None, min_len=None):
    """Seeded activation matrix [M, K].

    Returns (values float32 [M,K], bits) where bits is the uint16 bf16 bit
    pattern for dtype="bf16" and None for dtype="f32".
    seq_slots: if given, rows are grouped into sequences of seq_slots rows;
    each sequence keeps its first L rows, L ~ U[min_len, seq_slots], and the
    rest are zero (right padding).
    """
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K), dtype=np.float32)
    if outlier_frac > 0:
        n_out = max(1, int(round(outlier_frac * K)))
        chans = rng.choice(K, size=n_out, replace=False)
        x[:, chans] *= np.float32(outlier_mult)
    if seq_slots:
        lo = min_len if min_len is not None else max(1, seq_slots // 4)
        for s0 in range(0, M, seq_slots):
            L = int(rng.integers(lo, seq_slots + 1))
            x[s0 + L:s0 + seq_slots, :] = 0.0
    if dtype == "bf16":
        return _bf16_round(x)
    if dtype == "f32":
        return x, None
    raise ValueError(dtype)


def normal_weights(seed, N, K, std=0.02):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((N, K), dtype=np.float32) * np.float32(std)


def encode_q8_0(w):
    """float32 [N, K] (K % 32 == 0) -> uint8 [N, K/32, 34] Q8_0 blocks."""
    N, K = w.shape
    assert K % QBLK == 0
    B = K // QBLK
    wb = w.reshape(N, B, QBLK).astype(np.float32)
    absmax = np.abs(wb).max(axis=2)
    d16 = (absmax / np.float32(127.0)).astype(np.float16)
    d32 = d16.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(wb / d32[:, :, None])
    r = np.where(d32[:, :, None] == 0, 0.0, r)
    q = np.clip(r, -127, 127).astype(np.int8)
    out = np.empty((N, B, Q8_0_BYTES), np.uint8)
    out[:, :, 0:2] = d16.view(np.uint8).reshape(N, B, 2)
    out[:, :, 2:] = q.view(np.uint8)
    return out


def q8_0_weights(seed, N, K, std=0.02):
    return encode_q8_0(normal_weights(seed, N, K, std))


def pack_q4k_fields(d16, dmin16, sc, mn, q):
    """Assemble super-blocks from fields.

    d16, dmin16: float16 [N, J]; sc, mn: uint8 [N, J, 8] (< 64);
    q: uint8 [N, J, 256] (< 16) -> uint8 [N, J, 144].
    """
    N, J = d16.shape
    out = np.zeros((N, J, Q4K_BYTES), np.uint8)
    out[:, :, 0:2] = d16.astype(np.float16).view(np.uint8).reshape(N, J, 2)
    out[:, :, 2:4] = dmin16.astype(np.float16).view(np.uint8).reshape(N, J, 2)
    fields = np.concatenate([sc, mn], axis=2).astype(np.uint64)  # [N, J, 16]
    bits = np.zeros((N, J), np.uint64)
    hi = np.zeros((N, J), np.uint64)
    for f in range(16):
        pos = 6 * f
        v = fields[:, :, f] & np.uint64(63)
        if pos + 6 <= 64:
            bits |= v << np.uint64(pos)
        elif pos >= 64:
            hi |= v << np.uint64(pos - 64)
        else:  # straddles bit 64
            bits |= (v << np.uint64(pos)) & np.uint64(0xFFFFFFFFFFFFFFFF)
            hi |= v >> np.uint64(64 - pos)
    for byte in range(12):
        if byte < 8:
            out[:, :, 4 + byte] = ((bits >> np.uint64(8 * byte)) & np.uint64(0xFF)).astype(np.uint8)
        else:
            out[:, :, 4 + byte] = ((hi >> np.uint64(8 * (byte - 8))) & np.uint64(0xFF)).astype(np.uint8)
    qq = q.astype(np.uint8)
    out[:, :, 16:] = (qq[:, :, 0::2] & 0xF) | ((qq[:, :, 1::2] & 0xF) << 4)
    return out


def encode_q4k(w):
    """float32 [N, K] (K % 256 == 0) -> uint8 [N, K/256, 144] Q4_K super-blocks."""
    N, K = w.shape
    assert K % Q4K_WEIGHTS == 0
    J = K // Q4K_WEIGHTS
    ws = w.reshape(N, J, 8, QBLK).astype(np.float32)
    lo = np.minimum(np.float32(0.0), ws.min(axis=3))
    hi = ws.max(axis=3)
    scale = (hi - lo) / np.float32(15.0)
    off = -lo
    d16 = (scale.max(axis=2) / np.float32(63.0)).astype(np.float16)
    dmin16 = (off.max(axis=2) / np.float32(63.0)).astype(np.float16)
    d = d16.astype(np.float32)[:, :, None]
    dmin = dmin16.astype(np.float32)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        sc = np.where(d == 0, 0.0, np.clip(np.rint(scale / d), 0, 63))
        mn = np.where(dmin == 0, 0.0, np.clip(np.rint(off / dmin), 0, 63))
    sc = sc.astype(np.float32)
    mn = mn.astype(np.float32)
    step = (d * sc)[:, :, :, None]
    shift = (dmin * mn)[:, :, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        qf = np.where(step == 0, 0.0, np.clip(np.rint((ws + shift) / step), 0, 15))
    q = qf.astype(np.uint8).reshape(N, J, Q4K_WEIGHTS)
    return pack_q4k_fields(d16, dmin16, sc.astype(np.uint8), mn.astype(np.uint8), q)


def q4k_weights(seed, N, K, std=0.02):
    return encode_q4k(normal_weights(seed, N, K, std))


# The five workloads (shapes and value recipes). Seeds: config i uses seed
# i-1 for activations and i-1+100 for weights (the tiny case's seed 0 is the
# one the workload names).
CONFIGS = {
    "tiny_w8a8": dict(kind="w8a8", shapes=[(4, 256, 128)], act_dtype="f32", outlier=0.0,
                      seed=0),
    "prefill_4b_w8a8": dict(kind="w8a8", shapes=[(2048, 2560, 9728), (2048, 9728, 2560)],
                            act_dtype="bf16", outlier=0.01, seq_slots=128, min_len=32, seed=1),
    "decode_w8a8": dict(kind="w8a8", shapes=[(m, k, n) for m in (1, 8, 64)
                                             for (k, n) in ((5120, 17408), (17408, 5120))],
                        act_dtype="bf16", outlier=0.0, seed=2),
    "prefill_27b_w8a8": dict(kind="w8a8", shapes=[(8192, 5120, 17408), (8192, 17408, 5120)],
                             act_dtype="bf16", outlier=0.01, seed=3),
    "w4a8_q4k": dict(kind="w4a8", shapes=[(m, 5120, 17408) for m in (1, 64, 4096)],
                     act_dtype="bf16", outlier=0.0, seed=4),
}


def config_activations(name, M, K, seed_offset=0):
    c = CONFIGS[name]
    return activations(c["seed"] + seed_offset, M, K, dtype=c["act_dtype"],
                       outlier_frac=c.get("outlier", 0.0),
                       seq_slots=c.get("seq_slots"), min_len=c.get("min_len"))


def config_weights(name, N, K, seed_offset=0):
    c = CONFIGS[name]
    if c["kind"] == "w8a8":
        return q8_0_weights(c["seed"] + 100 + seed_offset, N, K)
    return q4k_weights(c["seed"] + 100 + seed_offset, N, K)
