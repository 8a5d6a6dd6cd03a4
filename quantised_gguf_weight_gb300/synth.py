"""Seeded synthetic inputs for the quantised GEMV/GEMM.

This module only draws random numbers and lays them out as GGUF block
records.  It holds none of the dequantise-and-multiply arithmetic: it never
decodes a block, never multiplies a weight and never sums anything.  Both the
CPU oracle (in the tests) and the CUDA path consume what it produces.

Random source: splitmix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), used as a counter-based
generator: value i of stream (seed, stream) is the splitmix64 output mix
applied to key + (i + 1) * golden_gamma.  Normals come from the Box-Muller
transform of two uniform streams.

Block records (the GGUF layouts the weights are stored in):

* Q8_0, 34 bytes: fp16 scale ``d`` then 32 signed 8-bit quants.
* Q4_K, 144 bytes: fp16 ``d``, fp16 ``dmin``, 12 bytes of packed 6-bit
  sub-block scales and mins, 128 bytes of 4-bit quants.

Uniform random bytes in the ``scales`` and ``qs`` fields give every 6-bit
scale/min field a uniform value in [0, 63] and every 4-bit quant a uniform
value in [0, 15], because each field is made of independent random bits; no
packing code is needed to draw them.
"""
from __future__ import annotations

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_STREAM_MULT = 0xD1B54A32D192ED03

Q8_0_DTYPE = np.dtype([("d", "<f2"), ("qs", "i1", (32,))])
Q4_K_DTYPE = np.dtype([("d", "<f2"), ("dmin", "<f2"), ("scales", "u1", (12,)),
                       ("qs", "u1", (128,))])
Q6_K_DTYPE = np.dtype([("ql", "u1", (128,)), ("qh", "u1", (64,)), ("scales", "i1", (16,)), ("d", "<f2")])
assert Q8_0_DTYPE.itemsize == 34 and Q4_K_DTYPE.itemsize == 144 and Q6_K_DTYPE.itemsize == 210

BLOCK = {"q8_0": (32, 34, Q8_0_DTYPE), "q4_k": (256, 144, Q4_K_DTYPE), "q6_k": (256, 210, Q6_K_DTYPE)}


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    k = np.array([(seed * 0x100000001B3 + stream * _STREAM_MULT) & 0xFFFFFFFFFFFFFFFF],
                 dtype=np.uint64)
    return _mix(k + GOLDEN_GAMMA)[0]


def u64(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """n raw 64-bit outputs of stream (seed, stream), counter offset `start`."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        return _mix(_key(seed, stream) + i * GOLDEN_GAMMA)


def uniform(seed: int, stream: int, n: int) -> np.ndarray:
    """Uniform doubles in [0, 1) with 53 random bits."""
    return (u64(seed, stream, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    """Standard normal doubles (Box-Muller, cosine branch)."""
    u1 = uniform(seed, 2 * stream, n)
    u2 = uniform(seed, 2 * stream + 1, n)
    return np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * np.pi * u2)


def randint(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    """Integers uniform in [lo, hi] (inclusive); modulo bias < 2^-50."""
    span = np.uint64(hi - lo + 1)
    return (u64(seed, stream, n) % span).astype(np.int64) + lo


def random_bytes(seed: int, stream: int, n: int) -> np.ndarray:
    return u64(seed, stream, (n + 7) // 8).view(np.uint8)[:n].copy()


def blocks_per_row(fmt: str, K: int) -> int:
    qk = BLOCK[fmt][0]
    return (K + qk - 1) // qk


def row_bytes(fmt: str, K: int) -> int:
    return blocks_per_row(fmt, K) * BLOCK[fmt][1]


def q8_0_weights(rows: int, K: int, seed: int, d_sigma: float = 0.02,
                 stream0: int = 0) -> np.ndarray:
    """Q8_0 tensor [rows][ceil(K/32)] as raw bytes (uint8, flat).

    quants uniform in [-127, 127]; d = fp16(|N(0, d_sigma)| / 127).
    """
    nb = rows * blocks_per_row("q8_0", K)
    rec = np.empty(nb, dtype=Q8_0_DTYPE)
    rec["d"] = (np.abs(normal(seed, stream0 + 0, nb)) * d_sigma / 127.0).astype(np.float16)
    rec["qs"] = randint(seed, stream0 + 1, nb * 32, -127, 127).astype(np.int8).reshape(nb, 32)
    return rec.view(np.uint8).reshape(-1)


def q4_k_weights(rows: int, K: int, seed: int, d_sigma: float = 0.01,
                 dmin_sigma: float = 0.005, stream0: int = 0) -> np.ndarray:
    """Q4_K tensor [rows][ceil(K/256)] as raw bytes (uint8, flat).

    4-bit quants uniform in [0, 15]; 6-bit scales and mins uniform in
    [0, 63]; d = fp16(|N(0, d_sigma)|); dmin = fp16(|N(0, dmin_sigma)|).
    When K is not a multiple of 256 the unused tail of each row's last
    super-block is random too (it must be ignored by every consumer).
    """
    nb = rows * blocks_per_row("q4_k", K)
    rec = np.empty(nb, dtype=Q4_K_DTYPE)
    rec["d"] = (np.abs(normal(seed, stream0 + 0, nb)) * d_sigma).astype(np.float16)
    rec["dmin"] = (np.abs(normal(seed, stream0 + 1, nb)) * dmin_sigma).astype(np.float16)
    rec["scales"] = random_bytes(seed, stream0 + 2, nb * 12).reshape(nb, 12)
    rec["qs"] = random_bytes(seed, stream0 + 3, nb * 128).reshape(nb, 128)
    return rec.view(np.uint8).reshape(-1)


def q6_k_weights(rows: int, K: int, seed: int, d_sigma: float = 1e-4, stream0: int = 0) -> np.ndarray:
    """Q6_K tensor [rows][ceil(K/256)] as raw bytes (uint8, flat).

    ql and qh uniform random bytes (6-bit quants uniform in [0, 63]); int8
    scales uniform in [-127, 127]; d = fp16(|N(0, d_sigma)|).  The unused
    tail of a row's last super-block is random too.
    """
    nb = rows * blocks_per_row("q6_k", K)
    rec = np.empty(nb, dtype=Q6_K_DTYPE)
    rec["ql"] = random_bytes(seed, stream0 + 0, nb * 128).reshape(nb, 128)
    rec["qh"] = random_bytes(seed, stream0 + 1, nb * 64).reshape(nb, 64)
    rec["scales"] = randint(seed, stream0 + 2, nb * 16, -127, 127).astype(np.int8).reshape(nb, 16)
    rec["d"] = (np.abs(normal(seed, stream0 + 3, nb)) * d_sigma).astype(np.float16)
    return rec.view(np.uint8).reshape(-1)


def weights(fmt: str, rows: int, K: int, seed: int, stream0: int = 0) -> np.ndarray:
    if fmt == "q8_0":
        return q8_0_weights(rows, K, seed, stream0=stream0)
    if fmt == "q4_k":
        return q4_k_weights(rows, K, seed, stream0=stream0)
    if fmt == "q6_k":
        return q6_k_weights(rows, K, seed, stream0=stream0)
    raise ValueError(fmt)


def activations(batch: int, K: int, seed: int, stream: int = 100) -> np.ndarray:
    """fp32 activations x[batch][K] ~ N(0, 1)."""
    return normal(seed, stream, batch * K).astype(np.float32).reshape(batch, K)


def small_int_activations(batch: int, K: int, seed: int, lo: int = -8, hi: int = 8,
                          stream: int = 101) -> np.ndarray:
    """fp32 activations holding small integers (exact-arithmetic cases)."""
    return randint(seed, stream, batch * K, lo, hi).astype(np.float32).reshape(batch, K)


def pow2_scaled_blocks(raw: np.ndarray, fmt: str, exps: tuple[int, ...], seed: int) -> np.ndarray:
    """Copy of `raw` whose fp16 d (and dmin) fields are set to 2^e, e drawn from `exps`.

    With power-of-two scales and small-integer activations every partial sum
    of a dot product is exact in fp32, so any summation order gives the same
    bits.
    """
    out = raw.copy()
    rec = out.view(BLOCK[fmt][2])
    n = rec.shape[0]
    e = np.asarray(exps)[randint(seed, 7, n, 0, len(exps) - 1)]
    rec["d"] = np.ldexp(1.0, e).astype(np.float16)
    if fmt == "q4_k":
        e2 = np.asarray(exps)[randint(seed, 8, n, 0, len(exps) - 1)]
        rec["dmin"] = np.ldexp(1.0, e2).astype(np.float16)
    return out


WIDE_RANGE_KINDS = ("group_outlier_2p20", "group_outlier_2p30", "group_tiny_2m30", "outlier_channels",
                    "two_large_per_group", "subnormal", "mixed_subnormal")


def wide_range_activations(batch: int, K: int, seed: int, kind: str, stream: int = 300):
    """fp32 activations x[batch][K] of wide dynamic range, and the columns that hold the large values.

    Every kind starts from N(0, 1) (or a constant 0.3 for group_outlier_2p20)
    and places large or tiny values:

    * group_outlier_2p20: every 32-column group is 0.3 except one column of
      value 2^20 (the column drawn per group);
    * group_outlier_2p30: one column per group is 2^30 times its N(0, 1) value;
    * group_tiny_2m30: one column per group is 2^-30 times its N(0, 1) value;
    * outlier_channels: 8 columns in 8 different groups (the same columns in
      every batch row), each scaled by a factor drawn uniformly from [100, 1000];
    * two_large_per_group: two columns per group are 2^20 times their value;
    * subnormal: every value is N(0, 1) * 2^-140 (fp32 subnormals);
    * mixed_subnormal: even 32-column groups are scaled to subnormals, odd
      groups stay N(0, 1), and one value per odd group is replaced by 2^-130.

    Returns (x, cols): cols[b] is the sorted array of the columns that carry
    the large values in batch row b (empty for the tiny and subnormal kinds).
    """
    if kind not in WIDE_RANGE_KINDS:
        raise ValueError(kind)
    ng = (K + 31) // 32
    x = normal(seed, stream, batch * K).reshape(batch, K)
    cols = []
    for b in range(batch):
        pick_all = randint(seed, stream + 1 + 4 * b, ng, 0, 31) + 32 * np.arange(ng)
        pick = pick_all[pick_all < K]
        big = np.array([], np.int64)
        if kind == "group_outlier_2p20":
            x[b, :] = 0.3
            x[b, pick] = 2.0 ** 20
            big = pick
        elif kind == "group_outlier_2p30":
            x[b, pick] *= 2.0 ** 30
            big = pick
        elif kind == "group_tiny_2m30":
            x[b, pick] *= 2.0 ** -30
        elif kind == "outlier_channels":
            # 8 channels (fewer when K has fewer groups), each in a group of its own
            groups = np.argsort(uniform(seed, stream + 2, ng))[:min(8, ng)]
            ch = np.sort(pick_all[groups])
            ch = ch[ch < K]
            x[b, ch] *= 100.0 + 900.0 * uniform(seed, stream + 3, ch.size)
            big = ch
        elif kind == "two_large_per_group":
            second = randint(seed, stream + 2 + 4 * b, ng, 0, 30) + 32 * np.arange(ng)
            second = np.where(second % 32 >= pick_all % 32, second + 1, second)
            second = second[second < K]
            big = np.unique(np.concatenate([pick, second]))
            x[b, big] *= 2.0 ** 20
        elif kind == "subnormal":
            x[b, :] *= 2.0 ** -140
        elif kind == "mixed_subnormal":
            g = np.arange(K) // 32
            x[b, g % 2 == 0] *= 2.0 ** -140
            odd = pick[(pick // 32) % 2 == 1]
            x[b, odd] = 2.0 ** -130
        cols.append(np.sort(big))
    return x.astype(np.float32), cols
