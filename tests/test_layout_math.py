"""Host checks of the index algebra the prep kernel's operand build relies on
(no GPU).  The kernel addresses token row 8 h8 + l, channels cc and cc + 1, of
every 128-byte-swizzled K-major tile as trow0 ^ (l * 144), and the MN-major
[K e^Gam | V] operand from the same offset; both shortcuts are checked here
against the swizzle's definition (16-byte chunk index XOR (row mod 8) inside a
1024-byte, 8-row atom) for every thread and row.  The integer tf32 rounding is
checked against exact round-to-nearest, ties away from zero (the GPU test
compares it with the conversion instruction)."""
import math

import numpy as np


def sw128_kmajor(r, c):
    """Byte offset of bf16 element (row r, column c < 64) of a K-major tile of
    128-byte rows with the 128-byte swizzle."""
    chunk, within = c // 8, c % 8
    return r * 128 + ((chunk ^ (r % 8)) * 16) + within * 2


def sw128_mnmajor(k, n, sbo):
    """Byte offset of element (k, n) of an MN-major operand: 64 consecutive n
    per 128-byte row, 8 rows (k) per 1024-byte atom, atoms along n 1 KB apart,
    8-row groups along k sbo apart."""
    return (k // 8) * sbo + (n // 64) * 1024 + (k % 8) * 128 + ((((n % 64) // 8) ^ (k % 8)) * 16) + (n % 8) * 2


def yoff_row(I, J, l):
    return 8 * I * (I - 1) + 16 * J + l


def test_token_row_offsets():
    for tid in range(512):
        c0 = 2 * (tid & 63)
        h8, cc, blk = tid >> 6, c0 & 63, c0 >> 6
        G, hf = h8 >> 1, h8 & 1
        trow0 = h8 * 1024 + (((cc >> 3) << 4) | ((cc & 7) << 1))
        for l in range(8):
            i = 8 * h8 + l
            tr = trow0 ^ (l * 144)
            assert sw128_kmajor(i, cc) == tr                      # R, K rows; Q e^Gam image
            assert sw128_kmajor(64 + i, cc) == 8192 + tr          # R, Q rows
            assert sw128_kmajor(96 + i, cc) == 96 * 128 + tr      # Yd
            for I in range(G + 1, 4):                             # Yoff, later row blocks
                assert sw128_kmajor(yoff_row(I, G, 8 * hf + l), cc) == 8 * I * (I - 1) * 128 + tr
            kv = h8 * (4096 - 1024) + blk * 1024 + tr
            assert sw128_mnmajor(i, c0, 4096) == kv               # K e^Gam half
            assert sw128_mnmajor(i, 128 + c0, 4096) == kv + 2048  # V half


def test_tf32_rounding_rule():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(50000) * 10.0 ** rng.integers(-30, 30, 50000)).astype(np.float32)
    ties = np.array([1 + 2 ** -11, -(1 + 2 ** -11), 1 + 3 * 2 ** -11, 2 - 2 ** -12], dtype=np.float32)
    x = np.concatenate([x, ties])
    u = x.view(np.uint32).astype(np.uint64)
    fast = ((u + 0x1000) & 0xFFFFE000).astype(np.uint32).view(np.float32)
    for v, f in zip(x.tolist(), fast.tolist()):
        if v == 0.0:
            assert f == 0.0
            continue
        m, e = math.frexp(abs(v))
        q = max(e - 11, -136)                 # 11 significant bits; subnormal spacing below
        r = math.floor(abs(v) / 2.0 ** q + 0.5) * 2.0 ** q
        assert f == math.copysign(r, v), (v, f)
