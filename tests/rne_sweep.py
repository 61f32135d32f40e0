"""Worker for the exhaustive FP32 -> BF16 sweep (tests/test_oracle_rne_exhaustive.py).

It lives in its own module so that processes started with ``spawn`` can import it.
Each call checks one block of 2**24 consecutive FP32 bit patterns. The oracle's
conversion compares the two neighbouring BF16 values in double precision. The
second formulation here rounds on the bit pattern instead:
- keep the upper 16 bits;
- add one when the dropped 16 bits exceed half a unit in the last place;
- on an exact half, add one only when the kept last bit is odd.

IEEE-754's roundTiesToEven is this rule. For a given sign, BF16 patterns are
ordered like their magnitudes, so the carry into the exponent field gives the next
binade. From the largest finite value the carry gives infinity. A NaN keeps its sign
and its top payload bits and has its quiet bit (0x0040) set.
"""
import numpy as np

import oracle

BLOCK = 1 << 24


def integer_rule(u: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(u, dtype=np.uint32)
    kept = u >> np.uint32(16)
    dropped = u & np.uint32(0xFFFF)
    up = (dropped > np.uint32(0x8000)) | ((dropped == np.uint32(0x8000)) & ((kept & np.uint32(1)) == 1))
    out = kept + up
    exp_ones = (u & np.uint32(0x7F800000)) == np.uint32(0x7F800000)
    nan = exp_ones & ((u & np.uint32(0x7FFFFF)) != 0)
    out[nan] = kept[nan] | np.uint32(0x0040)
    return out.astype(np.uint16)


_bufs = {}


def check_block(k: int):
    """Return (block, mismatches, first mismatching FP32 pattern or -1)."""
    if not _bufs:  # one set of buffers per worker process, reused for every block
        _bufs.update(base=np.arange(BLOCK, dtype=np.uint32), u=np.empty(BLOCK, np.uint32),
                     got=np.empty(BLOCK, np.uint16))
    u, got = _bufs["u"], _bufs["got"]
    np.add(_bufs["base"], np.uint32(k * BLOCK), out=u)
    oracle._load().oracle_f32_to_bf16_array(u.ctypes.data, got.ctypes.data, BLOCK)
    bad = np.flatnonzero(got != integer_rule(u))
    return k, int(bad.size), int(u[bad[0]]) if bad.size else -1
