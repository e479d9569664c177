"""The tiled I2_S weight layout (i2s_tile_weights), restated with numpy from
its definition in include/i2s.h: a test-side description of where each byte
goes, used to check the library's tiling kernel and sizes. It holds none of
the method's arithmetic."""

import numpy as np


def blocks(N, K):
    """(Tn, Tk): row blocks of 128 rows (an even count) and column blocks of
    128 bytes (512 positions)."""
    return 2 * ((N + 255) // 256), (K + 511) // 512


def nbytes(N, K):
    tn, tk = blocks(N, K)
    return tn * tk * 16384 + 32


def tile(packed, N, K):
    """The tiled layout of I2_S bytes `packed` (N*K/4 payload bytes, then the
    32-byte trailer): block (i, j) holds bytes 128j..128j+127 of rows
    128i..128i+127; row rr of a block stores its 16-byte piece c at piece
    position c ^ (rr % 8); zeros past N and K/4; the trailer last."""
    rb = K // 4
    tn, tk = blocks(N, K)
    full = np.zeros((tn * 128, tk * 128), np.uint8)
    full[:N, :rb] = np.asarray(packed[:N * rb]).reshape(N, rb)
    pieces = full.reshape(tn, 128, tk, 8, 16).transpose(0, 2, 1, 3, 4)   # (i, j, rr, c, byte)
    rr = np.arange(128)[:, None]
    c = np.arange(8)[None, :]
    out = np.empty_like(pieces)
    out[:, :, np.broadcast_to(rr, (128, 8)), c ^ (rr & 7), :] = pieces[:, :, np.broadcast_to(rr, (128, 8)),
                                                                       np.broadcast_to(c, (128, 8)), :]
    return np.concatenate([out.reshape(-1), np.asarray(packed[N * rb:N * rb + 32], np.uint8)])
