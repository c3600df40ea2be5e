"""Parsers for the hand-derived text fixtures under tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def fval(v):
    """A decimal number, or an exact fp32 bit pattern written h<hex>."""
    import numpy as np
    if v.startswith("h"):
        return float(np.array([int(v[1:], 16)], np.uint32).view(np.float32)[0])
    return float(v)


def _kv(text, conv):
    out = {}
    for tok in text.split():
        k, v = tok.split("=")
        out[int(k)] = conv(v)
    return out


def quantize_cases(name="quantize_ties.txt"):
    cases, cur = [], None
    for line in _lines(name):
        key, _, rest = line.partition(":") if not line.startswith("row ") else ("row", None, line[4:])
        if key == "row":
            cur = {"name": rest.strip()}
            cases.append(cur)
        elif key == "x":
            cur["x"] = _kv(rest, fval)
        elif key == "s":
            cur["s"] = fval(rest.strip())
        elif key == "q":
            cur["q"] = _kv(rest, int)
        elif key == "bsum":
            cur["bsum"] = _kv(rest, int)
    return cases


def gemm_cases():
    cases, cur = [], None
    for line in _lines("gemm_q8_0_small.txt"):
        if line.startswith("case "):
            cur = {"name": line[5:].strip(), "w": {}, "y": {}, "bf16": {}}
            cases.append(cur)
            continue
        key, _, rest = line.partition(":")
        rest = rest.strip()
        if key == "K":
            cur["K"] = int(rest)
        elif key == "x":
            cur["x"] = _kv(rest, float)
        elif key.startswith("w"):
            dpart, qpart = rest.split(" q=")
            d = [int(h, 16) for h in dpart[2:].split(",")]
            cur["w"][int(key[1:])] = (d, _kv(qpart, int))
        elif key.startswith("y"):
            cur["y"][int(key[1:])] = float(rest)
        elif key.startswith("bf16_"):
            cur["bf16"][int(key[5:])] = int(rest, 16)
    return cases


def q4k_case():
    c = {}
    for line in _lines("q4k_superblock.txt"):
        key, _, rest = line.partition(":")
        rest = rest.strip()
        if key in ("header", "scales", "nibbles8"):
            c[key] = [int(h, 16) for h in rest.split()]
        elif key in ("d", "dmin"):
            c[key] = float(rest)
        elif key in ("sc", "m"):
            c[key] = [int(v) for v in rest.split()]
        elif key == "w":
            c["w"] = _kv(rest, float)
    return c


def _kv_ranges(text, conv):
    """index=value or first-last=value tokens -> {index: value}."""
    out = {}
    for tok in text.split():
        k, v = tok.split("=")
        lo, _, hi = k.partition("-")
        for i in range(int(lo), int(hi or lo) + 1):
            out[i] = conv(v)
    return out


def gemm_q4k_cases():
    """Cases of gemm_q4k_small.txt: K, x, per-row super-block bytes, y, bf16."""
    cases, cur = [], None
    for line in _lines("gemm_q4k_small.txt"):
        if line.startswith("case "):
            cur = {"name": line[5:].strip(), "sb": {}, "y": {}, "bf16": {}}
            cases.append(cur)
            continue
        key, _, rest = line.partition(":")
        rest = rest.strip()
        if key == "K":
            cur["K"] = int(rest)
        elif key == "x":
            cur["x"] = _kv_ranges(rest, float)
        elif key.startswith("sb"):
            cur["sb"][int(key[2:])] = _kv_ranges(rest, lambda h: int(h, 16))
        elif key.startswith("y"):
            cur["y"][int(key[1:])] = float(rest)
        elif key.startswith("bf16_"):
            cur["bf16"][int(key[5:])] = int(rest, 16)
    return cases


def q4k_case_arrays(case):
    """(x fp32 [1, K], sblocks uint8 [N, K/256, 144]) of a gemm_q4k_small.txt case."""
    import numpy as np
    K = case["K"]
    x = np.zeros((1, K), np.float32)
    for k, v in case["x"].items():
        x[0, k] = v
    N = len(case["sb"])
    sb = np.zeros((N, K // 256 * 144), np.uint8)
    for n, bytes_ in case["sb"].items():
        for i, v in bytes_.items():
            sb[n, i] = v
    return x, sb.reshape(N, K // 256, 144)


def mxfp4_cases(name="mxfp4_small.txt"):
    """Cases of mxfp4_small.txt: dicts with d (fp16 bits per block), q, qa,
    codes (index -> value; a plain list means indices 0, 1, ...), E (per
    block), y (bf16 bits) and optionally y32 (fp32 bits)."""
    cases, cur = [], None
    for line in _lines(name):
        key, _, rest = line.partition(" ")
        if key == "case":
            cur = {"name": rest}
            cases.append(cur)
        elif key == "d":
            cur[key] = [int(v, 16) for v in rest.split()]
        elif key in ("y", "y32"):
            cur[key] = int(rest, 16)
        elif key == "E":
            cur[key] = [int(v) for v in rest.split()]
        else:  # q, qa, codes: dense values, or sparse index=value tokens
            toks = rest.split()
            if "=" in toks[0]:
                cur[key] = {int(k): int(v) for k, v in (t.split("=") for t in toks)}
            else:
                cur[key] = {i: int(v) for i, v in enumerate(toks)}
    return cases


def mxfp4_case_arrays(case):
    """The case's Q8_0 row (uint8 [1, K/32, 34]) and int8 activation row [1, K], K = 32 x blocks."""
    import numpy as np
    nb = len(case["d"])
    K = 32 * nb
    blocks = np.zeros((1, nb, 34), np.uint8)
    for b, d in enumerate(case["d"]):
        blocks[0, b, 0] = d & 0xFF
        blocks[0, b, 1] = d >> 8
    for k, v in case["q"].items():
        blocks[0, k // 32, 2 + k % 32] = np.uint8(v & 0xFF)
    qa = np.zeros((1, K), np.int8)
    for k, v in case["qa"].items():
        qa[0, k] = v
    return blocks, qa
