"""Pins for the repacked-layout reference (oracle/repack_layout.py), CPU only.

The repack is a permutation of nibbles. Beyond bijectivity and the round trip,
the layout is pinned to what its two GPU consumers need, using the PTX ISA's
published fragment tables rather than the layout formula itself:
  * mma.sync.m16n8k16 (.f16): the A operand fragment of lane (groupID, tig) holds
    a0,a1 = (row groupID, cols 2tig, 2tig+1), a2,a3 = (row groupID+8, same cols),
    a4,a5 = (row groupID, cols 2tig+8, 2tig+9), a6,a7 = (row groupID+8, those cols);
    the B operand holds b0,b1 = (rows 2tig, 2tig+1, col groupID), b2,b3 = (rows
    2tig+8, 2tig+9, col groupID). The kernel fills register i of word j with the
    half2 from nibbles (i, i+4) and loads b0..b3 as four consecutive activations;
    simulating the MMA on those fragments must give the true 16-k dot product.
  * tcgen05 A operand in tensor memory (M = 128, 16-bit types): lane r holds row r,
    32-bit column c holds k = 2c (low half) and 2c+1 (high half). The per-row
    extraction the tensor-core path uses must rebuild each row in that order.
"""
import numpy as np
import pytest

from oracle import repack_layout as RL


def _rand_bq(N, K, seed):
    return np.random.default_rng(seed).integers(0, 256, size=(N, K // 2), dtype=np.uint8)


@pytest.mark.parametrize("N,K", [(16, 64), (128, 64), (144, 128), (400, 192), (256, 256)])
def test_bijection(N, K):
    nn, kk = np.meshgrid(np.arange(N), np.arange(K), indexing="ij")
    byte, high = RL.nibble_position(nn, kk, N, K)
    slot = byte.astype(np.int64) * 2 + high
    assert slot.min() == 0 and slot.max() == N * K - 1
    assert np.unique(slot).size == N * K


@pytest.mark.parametrize("N,K", [(16, 64), (144, 128), (400, 192), (512, 256)])
def test_round_trip_and_histogram(N, K):
    bq = _rand_bq(N, K, N + K)
    rep = RL.repack(bq)
    assert rep.size == bq.size
    np.testing.assert_array_equal(RL.unpack(rep, N, K), bq)
    q = RL.logical_nibbles(bq, K)
    qr = np.concatenate([rep & 0xF, rep >> 4])
    np.testing.assert_array_equal(np.bincount(q.ravel(), minlength=16),
                                  np.bincount(qr.ravel(), minlength=16))


def test_one_hot_nibble_moves_to_one_place():
    N, K = 144, 128
    for (n, k) in [(0, 0), (0, 1), (7, 5), (8, 4), (15, 63), (130, 64), (143, 127)]:
        q = np.zeros((N, K), dtype=np.uint8)
        q[n, k] = 0xA
        bq = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
        rep = RL.repack(bq)
        nz = np.flatnonzero(rep)
        assert nz.size == 1
        assert rep[nz[0]] in (0x0A, 0xA0)


def test_one_row_per_thread_reads_spread_over_bank_groups():
    # For fixed t, the eight row groups g of a sub-tile read eight different
    # 16-byte bank groups (offset mod 128 bytes) of a shared-memory copy.
    for t in range(4):
        groups = {(_slot(g, t) * 16) % 128 for g in range(8)}
        assert len(groups) == 8
    for g in range(8):   # the four slots of one row group stay in one 64-byte span
        assert sorted(_slot(g, t) for t in range(4)) == list(range(4 * g, 4 * g + 4))


@pytest.mark.parametrize("N,K", [(32, 128), (144, 192)])
def test_sub_tile_is_one_contiguous_span(N, K):
    # Rows 16S..16S+15 occupy exactly bytes [S*8K, (S+1)*8K), k-block b of them
    # bytes [S*8K + 512b, S*8K + 512(b+1)).
    for S in range(N // 16):
        for b in range(K // 64):
            nn, kk = np.meshgrid(np.arange(16 * S, 16 * S + 16), np.arange(64 * b, 64 * b + 64), indexing="ij")
            byte, _ = RL.nibble_position(nn, kk, N, K)
            base = S * (K // 64) * 512 + 512 * b
            assert byte.min() == base and byte.max() == base + 511


def test_rejects_unsupported_dims():
    for N, K in [(8, 64), (16, 32), (20, 64)]:
        with pytest.raises(ValueError):
            RL.repack(np.zeros((N, K // 2), dtype=np.uint8))


def _words(rep, N, K, n0, b, s):
    """The 32 lanes x 4 u32 words of the piece of sub-tile (n0 // 16 + s), k-block b."""
    S = n0 // 16 + s
    base = (S * (K // 64) + b) * 512
    return rep[base:base + 512].view("<u4").reshape(32, 4)


def _slot(g, t):
    """Lane slot (16-byte unit of a sub-tile) of the fragment owned by (g, t)."""
    return 4 * g + (t + g // 2) % 4


def _half(word, nib):
    return (int(word) >> (4 * nib)) & 0xF


@pytest.mark.parametrize("N,K", [(144, 128), (256, 64)])
def test_mma_m16n8k16_fragments_compute_true_dot(N, K):
    rng = np.random.default_rng(3)
    bq = _rand_bq(N, K, 4)
    q = RL.logical_nibbles(bq, K).astype(np.int64)
    rep = RL.repack(bq)
    act = rng.integers(-3, 4, size=(8, K)).astype(np.int64)   # 8 tokens, exact ints
    for n0 in range(0, N, 128):
        R = min(128, N - n0)
        for b in range(K // 64):
            for s in range(R // 16):
                w = _words(rep, N, K, n0, b, s)
                for j in range(4):
                    k0 = 64 * b + 16 * j
                    Avirt = np.zeros((16, 16), dtype=np.int64)
                    Bvirt = np.zeros((16, 8), dtype=np.int64)
                    for lane in range(32):
                        gid, tig = lane >> 2, lane & 3
                        word = w[_slot(gid, tig), j]
                        a = [_half(word, i) for i in (0, 4, 1, 5, 2, 6, 3, 7)]  # a0..a7
                        Avirt[gid, 2 * tig], Avirt[gid, 2 * tig + 1] = a[0], a[1]
                        Avirt[gid + 8, 2 * tig], Avirt[gid + 8, 2 * tig + 1] = a[2], a[3]
                        Avirt[gid, 2 * tig + 8], Avirt[gid, 2 * tig + 9] = a[4], a[5]
                        Avirt[gid + 8, 2 * tig + 8], Avirt[gid + 8, 2 * tig + 9] = a[6], a[7]
                        bv = act[gid, k0 + 4 * tig: k0 + 4 * tig + 4]   # b0..b3
                        Bvirt[2 * tig, gid], Bvirt[2 * tig + 1, gid] = bv[0], bv[1]
                        Bvirt[2 * tig + 8, gid], Bvirt[2 * tig + 9, gid] = bv[2], bv[3]
                    D = Avirt @ Bvirt
                    rows = n0 + 16 * s + np.arange(16)
                    truth = q[rows, k0:k0 + 16] @ act[:, k0:k0 + 16].T
                    np.testing.assert_array_equal(D, truth)


@pytest.mark.parametrize("N,K", [(144, 128), (128, 192)])
def test_tmem_row_per_lane_extraction(N, K):
    bq = _rand_bq(N, K, 5)
    q = RL.logical_nibbles(bq, K)
    rep = RL.repack(bq)
    for n0 in range(0, N, 128):
        R = min(128, N - n0)
        for b in range(K // 64):
            for r in range(R):
                s, g, h = r // 16, r % 8, (r % 16) // 8
                w = _words(rep, N, K, n0, b, s)
                cols = np.zeros((32, 2), dtype=np.uint8)      # 32 columns x (lo, hi)
                for t in range(4):
                    for j in range(4):
                        word = w[_slot(g, t), j]
                        cols[8 * j + 2 * t] = (_half(word, h), _half(word, h + 4))
                        cols[8 * j + 2 * t + 1] = (_half(word, h + 2), _half(word, h + 6))
                row_k = cols.reshape(-1)                      # k = 2c + {0, 1}
                np.testing.assert_array_equal(row_k, q[n0 + r, 64 * b:64 * b + 64])
