"""The NVFP4 W4A16 weight image of include/moe_gb300.h (GU_IMG / D_IMG of the W4A16 format),
written out for the tests: the converter's bit order (where bits (m, e0, e1, s) of element k of a
canonical 32-bit code word go) and the blocks of 128-row tiles."""
import numpy as np

DST = ((0, 1, 2, 9), (16, 17, 18, 25), (4, 5, 6, 13), (20, 21, 22, 29),
       (10, 11, 12, 19), (26, 27, 28, 3), (14, 7, 8, 15), (30, 23, 24, 31))


def words(codes):
    """Canonical NVFP4 code bytes -> the converter's bit order, word by word (little-endian)."""
    w = np.ascontiguousarray(codes).view("<u4").astype(np.uint64)
    out = np.zeros_like(w)
    for k, dst in enumerate(DST):
        for b, d in enumerate(dst):
            out |= ((w >> np.uint64(4 * k + b)) & np.uint64(1)) << np.uint64(d)
    return out.astype("<u4")


def image(codes, scales, gu):
    """Canonical codes [E, N, K/2] and scales [E, N, K/16] -> the image [E, K/128, N/128, 9216]."""
    E, N, K2 = codes.shape
    K = 2 * K2
    NB, C = N // 128, K // 128
    l = np.arange(128)
    img = np.zeros((E, C, NB, 9216), np.uint8)
    perm = words(codes).view(np.uint8).reshape(E, N, K2)
    for b in range(NB):
        rows = np.where(l < 64, 64 * b + l, N // 2 + 64 * b + l - 64) if gu else 128 * b + l
        for c in range(C):
            pieces = perm[:, rows, 64 * c:64 * c + 64].reshape(E, 128, 4, 16)
            blk = np.zeros((E, 128, 4, 16), np.uint8)
            for p in range(4):
                blk[:, l, p ^ ((l >> 1) & 3)] = pieces[:, :, p]
            img[:, c, b, :8192] = blk.reshape(E, 8192)
            img[:, c, b, 8192:] = scales[:, rows, 8 * c:8 * c + 8].reshape(E, 1024)
    return img
