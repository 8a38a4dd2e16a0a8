"""Vectorised numpy Philox4x32-10 (Salmon et al., SC'11), used only to check
the GPU stream over many counters at once.  Pinned to the published
known-answer vectors in tests/golden/philox4x32_10_kat.txt."""
import numpy as np

_M0, _M1 = np.uint64(0xD2511F53), np.uint64(0xCD9E8D57)
_W0, _W1 = np.uint32(0x9E3779B9), np.uint32(0xBB67AE85)
_MASK = np.uint64(0xFFFFFFFF)


def philox(c0, c1, c2, c3, k0, k1):
    c = [np.asarray(x, dtype=np.uint32).copy() for x in (c0, c1, c2, c3)]
    k0 = np.uint32(k0)
    k1 = np.uint32(k1)
    with np.errstate(over="ignore"):
        for r in range(10):
            pa = _M0 * c[0].astype(np.uint64)
            pb = _M1 * c[2].astype(np.uint64)
            n0 = (pb >> np.uint64(32)).astype(np.uint32) ^ c[1] ^ k0
            n1 = (pb & _MASK).astype(np.uint32)
            n2 = (pa >> np.uint64(32)).astype(np.uint32) ^ c[3] ^ k1
            n3 = (pa & _MASK).astype(np.uint32)
            c = [n0, n1, n2, n3]
            k0 = np.uint32(k0 + _W0)
            k1 = np.uint32(k1 + _W1)
    return np.stack(c, axis=-1)
