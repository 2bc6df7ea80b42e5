"""Reference statement of the repacked int4 weight layout (numpy, no GPU).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU baseline, never by the product path.

The pull request that introduced the Marlin-style int4 GEMM for
`com.microsoft::MatMulNBits` (github.com/justinchuby/onnx-genai pull 960, "What's
landed") describes its repack only as a bijective, column-interleaved reorder of
the nibble-packed weights chosen so that each warp loads contiguous bytes, with
a device repack that must be byte-identical to a host reference. It does not give
the permutation itself, so this library defines its own ("fragment-interleaved")
layout, stated here as an index map from a logical nibble (n, k) of Bq[N][K/2]
(byte k/2 of row n, low nibble for even k) to a (byte, nibble) position of the
repacked buffer, which has the same N*K/2 bytes:

    sub-tile   S  = n // 16                                (16 weight rows)
    k-block    b  = k // 64
    piece      (S, b) starts at byte (S*(K/64) + b)*512, spans 512 bytes
    lane slot  l  = 4*g + (t + g//2) % 4,  g = n % 8,  t = (k % 16) // 4   -> l*16
    word       j  = (k % 64) // 16                         -> j*4 (little-endian u32)
    nibble     p  = 4*(e % 2) + 2*(e // 2) + h,  e = k % 4,  h = (n % 16) // 8
               byte j*4 + p//2 of the lane, high nibble when p is odd

So every 16-row sub-tile is one contiguous span of K/64 pieces, and a run of
consecutive k-blocks of consecutive sub-tiles is a regular 3-D box
(512-byte pieces x k-blocks x sub-tiles) for a tensor-memory-access copy.
N must be a multiple of 16 and K a multiple of 64.

Reading of the layout (what the two GPU consumers rely on; the tests check both
against the PTX ISA's fragment tables):
  * a 16-row x 64-k sub-tile is 512 contiguous bytes; the 16 bytes of the MMA
    fragment owner (g, t) sit in lane slot 4g + (t + g//2) % 4 and hold rows g and
    g+8 at k = 16j + 4t + {0,1,2,3} for j = 0..3. The rotation by g//2 keeps the
    four slots of a row group inside one 64-byte span while spreading the reads of
    a one-row-per-thread consumer (slot 4g + (t + g//2) % 4 for fixed t, g = 0..7)
    over all eight 16-byte bank groups of shared memory;
  * in word j, nibbles (i, i+4) for i = 0,1,2,3 are the element pairs
    (row g, e 0/1), (row g+8, e 0/1), (row g, e 2/3), (row g+8, e 2/3).
"""
from __future__ import annotations

import numpy as np


def check_dims(N: int, K: int) -> None:
    if N <= 0 or K <= 0 or N % 16 or K % 64:
        raise ValueError(f"repacked layout needs N % 16 == 0 and K % 64 == 0 (N={N}, K={K})")


def nibble_position(n, k, N: int, K: int):
    """Vectorised index map: logical nibble (n, k) -> (byte offset, is_high_nibble)."""
    n = np.asarray(n, dtype=np.int64)
    k = np.asarray(k, dtype=np.int64)
    S = n // 16
    b = k // 64
    g = n % 8
    h = (n % 16) // 8
    t = (k % 16) // 4
    j = (k % 64) // 16
    e = k % 4
    lane = 4 * g + (t + g // 2) % 4
    p = 4 * (e % 2) + 2 * (e // 2) + h
    byte = (S * (K // 64) + b) * 512 + lane * 16 + j * 4 + p // 2
    return byte, (p % 2).astype(bool)


def logical_nibbles(bq: np.ndarray, K: int) -> np.ndarray:
    """q[n, k] from the packed input format (byte k/2, low nibble first)."""
    lo = bq & 0x0F
    hi = bq >> 4
    q = np.empty((bq.shape[0], K), dtype=np.uint8)
    q[:, 0::2] = lo
    q[:, 1::2] = hi
    return q


def repack(bq: np.ndarray) -> np.ndarray:
    """Bq [N][K/2] -> repacked bytes (1-D, N*K/2)."""
    N, half_k = bq.shape
    K = 2 * half_k
    check_dims(N, K)
    q = logical_nibbles(bq, K)
    nn, kk = np.meshgrid(np.arange(N), np.arange(K), indexing="ij")
    byte, high = nibble_position(nn, kk, N, K)
    out = np.zeros(N * K // 2, dtype=np.uint8)
    lo_mask = ~high
    # Each byte receives exactly two nibbles (bijection), so plain stores suffice.
    out[byte[lo_mask]] |= q[lo_mask]
    out[byte[high]] |= (q[high] << 4).astype(np.uint8)
    return out


def unpack(rep: np.ndarray, N: int, K: int) -> np.ndarray:
    """Inverse of repack: repacked bytes -> Bq [N][K/2]."""
    check_dims(N, K)
    rep = np.asarray(rep, dtype=np.uint8).reshape(-1)
    if rep.size != N * K // 2:
        raise ValueError("size mismatch")
    nn, kk = np.meshgrid(np.arange(N), np.arange(K), indexing="ij")
    byte, high = nibble_position(nn, kk, N, K)
    vals = rep[byte]
    q = np.where(high, vals >> 4, vals & 0x0F).astype(np.uint8)
    return (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
