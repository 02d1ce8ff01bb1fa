"""Views of the library's page-head records in the oracle's plane layout.

The CUDA library stores each page-head (16 tokens of one kv head) as one
record (arrangement documented in include/nvfp4kv.h); the oracle keeps plain
planes: data [pages][Hkv][16][64], scale [pages][Hkv][16][8] for NVFP4 and
[pages][Hkv][16][128] for FP8.  These functions re-arrange GPU output bytes so
the two can be compared byte for byte.  They only move bytes.
"""
import numpy as np

_R = np.arange(8)[:, None, None, None]      # V row (token pair)
_G = np.arange(8)[None, :, None, None]      # group
_J = np.arange(8)[None, None, :, None]      # byte pair index (block)
_W = np.arange(2)[None, None, None, :]      # which byte of the pair


def nvfp4_planes(pool):
    """uint8 [P][H][2304] -> (k_data, k_scale, v_data, v_scale) planes."""
    pool = np.asarray(pool)
    P, H, _ = pool.shape
    k_data = pool[..., :1024].reshape(P, H, 16, 64)
    k_scale = pool[..., 2048:2176].reshape(P, H, 16, 8)
    v_scale = pool[..., 2176:2304].reshape(P, H, 8, 8, 2).transpose(0, 1, 2, 4, 3).reshape(P, H, 16, 8)
    vd = pool[..., 1024:2048].reshape(P, H, 8, 8, 16)             # [row][chunk position][byte]
    pos = (_G + 2 * _R) % 8
    bytes_ = vd[:, :, _R, pos, 2 * _J + _W]                       # [P][H][row][g][j][w]
    codes = np.zeros((P, H, 16, 128), np.uint8)
    ch = np.broadcast_to(16 * _J + _G + 8 * _W, bytes_.shape[2:])
    rows = np.broadcast_to(_R, bytes_.shape[2:])
    codes[:, :, 2 * rows, ch] = bytes_ & 15
    codes[:, :, 2 * rows + 1, ch] = bytes_ >> 4
    v_data = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    return k_data, k_scale, v_data, v_scale


def fp8_planes(pool):
    """uint8 [P][H][4096] -> (k, v) planes [P][H][16][128]."""
    pool = np.asarray(pool)
    P, H, _ = pool.shape
    kr = pool[..., :2048].reshape(P, H, 16, 8, 16)                 # [token][chunk position][byte]
    t = np.arange(16)[:, None]
    c = np.arange(8)[None, :]
    k = kr[:, :, t, (c + t % 2) % 8, :].reshape(P, H, 16, 128)
    vr = pool[..., 2048:].reshape(P, H, 8, 16, 16)                 # [row][chunk position][byte]
    row = np.arange(8)[:, None, None, None]
    cc = np.arange(16)[None, :, None, None]
    i = np.arange(8)[None, None, :, None]
    w = np.arange(2)[None, None, None, :]
    f = (row % 2) + 4 * ((row // 2) % 2)
    vals = vr[:, :, row, (cc + f) % 16, 2 * i + w]                 # [P][H][row][c][i][w]
    v = np.zeros((P, H, 16, 128), np.uint8)
    shp = vals.shape[2:]
    v[:, :, np.broadcast_to(2 * row + w, shp), np.broadcast_to(8 * cc + i, shp)] = vals
    return k, v
