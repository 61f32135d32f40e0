"""The oracle's FP32 -> BF16 rounding on every one of the 2**32 FP32 bit patterns.

The second formulation is the integer rounding rule in tests/rne_sweep.py. It is
itself pinned here to torch's CPU conversion for every non-NaN pattern of a
block-structured sample, and to a few textbook values. Both formulations must agree
with the oracle on every pattern. The work is spread over processes started with
``spawn``.
"""
import multiprocessing as mp
import os

import numpy as np
import torch

import oracle
import rne_sweep


def test_integer_rule_is_ieee_round_to_nearest_even():
    # Textbook values: ties go to the even neighbour, overflow goes to infinity,
    # and subnormals round within the subnormal grid.
    cases = {0x3F808000: 0x3F80, 0x3F818000: 0x3F82, 0x7F7F8000: 0x7F80, 0x7F7F7FFF: 0x7F7F,
             0x00008000: 0x0000, 0x00018000: 0x0002, 0x007FFFFF: 0x0080, 0x80000001: 0x8000,
             0xFF800000: 0xFF80, 0x7FC00001: 0x7FC0, 0xFF800001: 0xFFC0}
    u = np.array(list(cases), np.uint32)
    assert rne_sweep.integer_rule(u).tolist() == list(cases.values())
    # torch's CPU conversion agrees for every non-NaN pattern whose upper half is
    # any of the 2**16 values and whose lower half is one of the boundary values.
    hi = np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF], np.uint32)
    x = (hi[:, None] | lows[None, :]).reshape(-1)
    x = x[~(((x & 0x7F800000) == 0x7F800000) & ((x & 0x7FFFFF) != 0))]
    t = torch.from_numpy(x.view(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(rne_sweep.integer_rule(x), t)


def test_oracle_rounding_on_every_fp32_pattern():
    oracle.build()
    n_blocks = (1 << 32) // rne_sweep.BLOCK
    procs = max(1, min(16, os.cpu_count() or 1))
    with mp.get_context("spawn").Pool(procs) as pool:
        results = pool.map(rne_sweep.check_block, range(n_blocks), chunksize=1)
    assert len(results) == n_blocks
    bad = [(k, n, first) for k, n, first in results if n]
    assert not bad, [(k, n, hex(first)) for k, n, first in bad[:4]]
