"""The NVFP4 W4A16 converter bit order of include/moe_gb300.h (GU_IMG / D_IMG of the W4A16
format), written out for the tests: where bits (m, e0, e1, s) of element k of a canonical 32-bit
code word (element k = nibble k) go."""
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
