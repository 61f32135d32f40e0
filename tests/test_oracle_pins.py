"""Pins for the CPU oracle: it is checked against what the pages and the
mathematics fix, never against itself or the CUDA path.

* values the pages print ("The unit you wrapped": the Linear(4, 4) shard and
  gradient shards, the 36 / 18 / 9 per-rank counts, the Linear(3, 3) padding;
  the news item's 192 MiB figure);
* brute force: the definitions restated with numpy pad / reshape / hstack and
  byte appends, and torch's own dtype conversions as the cast;
* rounding: a textbook FP32 -> BF16 table, torch's CPU conversion on a large
  structured sample, and an exact-rational (fractions.Fraction) rounding
  reference written by quantum scaling and Python's ties-to-even round();
* invariants (padding slots are zero, total sizes, roundtrip).

Every test here runs without a GPU.  The functions take no fixtures so that
tests/test_oracle_mutants.py can re-run them against deliberately broken
copies of the oracle.
"""
import itertools
import random
from fractions import Fraction

import numpy as np
import torch

import oracle
from oracle import BF16, F32, Param, plan
from fsdp2_gradient_packing_gb300 import workloads as wl
from golden_io import f32_bits, records, sections

NP = {F32: np.uint32, BF16: np.uint16}


# ---------------------------------------------------------------------------
# Independent helpers: torch's conversions, numpy layout restatements.
# ---------------------------------------------------------------------------
def torch_cast(bits: np.ndarray, src: int, dst: int) -> np.ndarray:
    bits = np.ascontiguousarray(bits)
    if src == dst:
        return bits.copy()
    if src == BF16:
        t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
        return t.to(torch.float32).numpy().view(np.uint32).copy()
    t = torch.from_numpy(bits.view(np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def first_appearance(keys):
    seen = []
    for k in keys:
        if k not in seen:
            seen.append(k)
    return seen


def brute_pack(params, W, grads):
    """Pad each flat gradient to a multiple of W, view it as W rows, cast, and
    lay the rows of every parameter of a bucket side by side."""
    outs = []
    for rd in first_appearance([p.reduce_dtype for p in params]):
        blocks = []
        for p, g in zip(params, grads):
            if p.reduce_dtype != rd:
                continue
            c = -(-p.numel // W)
            v = np.pad(torch_cast(g, p.grad_dtype, rd), (0, c * W - p.numel))
            blocks.append(v.reshape(W, c))
        outs.append(np.hstack(blocks).reshape(-1))
    return outs


def brute_copy_in(params, shards):
    """Append each (shard dtype, param dtype) group's cast shards as bytes,
    zero-padding to a 16-byte boundary before each group and at the end.
    Returns the bytes and each parameter's byte position."""
    out = bytearray()
    where = {}
    for pair in first_appearance([(p.shard_dtype, p.param_dtype) for p in params]):
        out += bytes((-len(out)) % 16)
        for k, (p, s) in enumerate(zip(params, shards)):
            if (p.shard_dtype, p.param_dtype) == pair:
                where[k] = len(out)
                out += torch_cast(s, p.shard_dtype, p.param_dtype).tobytes()
    out += bytes((-len(out)) % 16)
    return np.frombuffer(bytes(out), np.uint8).copy(), where


def brute_copy_out(params, W, gathered, where):
    rows = gathered.reshape(W, -1)
    outs = []
    for k, p in enumerate(params):
        c = -(-p.numel // W)
        sz = 4 if p.param_dtype == F32 else 2
        parts = [rows[r, where[k]:where[k] + c * sz].view(NP[p.param_dtype]) for r in range(W)]
        full = np.concatenate(parts) if parts else np.zeros(0, NP[p.param_dtype])
        outs.append(full[:p.numel])
    return outs


def rand_bits(rng, n, dt):
    x = rng.standard_normal(n).astype(np.float32).view(np.uint32)
    return x if dt == F32 else (x >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# Page pins.
# ---------------------------------------------------------------------------
def test_linear4x4_rank0_holds_rows_0_and_1():
    g = sections("linear4x4_w2.txt")
    shard = f32_bits(g["rank0_shard"])
    weight = np.zeros((4, 4), np.float32)
    weight[0] = np.float32(np.array(g["weight_row0"], dtype=np.float64))
    weight[1] = np.float32(np.array(g["weight_row1"], dtype=np.float64))
    weight[2:] = np.random.default_rng(3).standard_normal((2, 4)).astype(np.float32)
    pl = plan([Param(16)], 2)
    assert pl.chunk == [8] and pl.bucket_S == [8]
    buf, = oracle.pack_reduce_scatter(pl, [weight.view(np.uint32).reshape(-1)])
    assert np.array_equal(buf[:8], shard)                     # rank 0 = rows 0-1
    assert np.array_equal(buf[8:], weight[2:].view(np.uint32).reshape(-1))
    # Gathering the unit gives the (4, 4) parameter back on every rank.
    rows = [oracle.allgather_copy_in(pl, [buf[r * 8:(r + 1) * 8]]) for r in range(2)]
    full, = oracle.allgather_copy_out(pl, np.concatenate(rows))
    shape = tuple(int(v) for v in g["summoned_shape"])
    assert np.array_equal(full.reshape(shape), weight.view(np.uint32))


def test_linear4x4_grad_shards():
    g = sections("linear4x4_w2.txt")
    grad = np.zeros((4, 4), np.float32)
    grad[1] = np.float32(1.2830595970)
    pl = plan([Param(16)], 2)
    buf, = oracle.pack_reduce_scatter(pl, [grad.view(np.uint32).reshape(-1)])
    assert np.array_equal(buf[:8], f32_bits(g["rank0_grad_shard"]))
    assert np.array_equal(buf[8:], f32_bits(g["rank1_grad_shard"]))


def test_wrap_policy_per_rank_counts():
    for rec in records("wrap_policy_counts.txt"):
        choice, W, counts = rec[0], int(rec[1]), [int(v) for v in rec[2:]]
        grouping = {"no_policy": "model", "block_units": "block", "linear_units": "linear"}[choice]
        work = wl.tiny_two_blocks(W=W, grouping=grouping)
        assert sum(p.numel for g in work.groups for p in g) == 144
        got = []
        for g in work.groups:
            pl = plan(oracle.params_from_specs(g), W)
            assert len(pl.bucket_S) == 1                      # one reduce dtype
            assert pl.bucket_S[0] == sum(pl.group_elems)      # same count gathered
            got.append(pl.bucket_S[0])
        assert got == counts, (choice, got, counts)


def test_linear3x3_padding():
    d = {r[0]: r[1:] for r in records("linear3x3_w4_padding.txt")}
    n, W = int(d["numel"][0]), int(d["world_size"][0])
    pl = plan([Param(n)], W)
    assert [pl.chunk[0]] * W == [int(v) for v in d["shard"]]
    assert pl.chunk[0] * W == int(d["padded_total"][0])
    grad = (np.arange(1, n + 1, dtype=np.float32)).view(np.uint32)
    buf, = oracle.pack_reduce_scatter(pl, [grad])
    pad = buf[n:]
    assert pad.size == int(d["padding"][0]) and np.all(pad == 0)
    assert np.array_equal(buf[:n], grad)


def test_isolated_pack_avoided_temporary_is_192_mib():
    d = {r[0]: r[1:] for r in records("isolated_pack_test.txt")}
    work = wl.mixed_50m(W=8)
    params = oracle.params_from_specs(work.groups[0])
    n_bf16 = sum(p.numel for p in params if p.grad_dtype == BF16)
    n_all = sum(p.numel for p in params)
    assert n_bf16 == 50_331_648
    assert round(n_all / 1e6, 1) == float(d["elements_millions"][0])
    assert n_bf16 * 4 == int(d["avoided_temporary_mib"][0]) * 2**20   # FP32 copy of the BF16 grads
    pl = plan(params, 8)
    assert pl.bucket_S == [6_292_480] and len(pl.bucket_dtype) == 1
    assert 8 * pl.bucket_S[0] * 4 == 201_359_360


def test_one_bucket_per_reduce_dtype_in_first_appearance_order():
    same = [Param(5, BF16, F32), Param(7, F32, F32), Param(3, BF16, F32)]
    assert plan(same, 4).bucket_dtype == [F32]
    mixed = [Param(5, BF16, BF16), Param(7, F32, F32), Param(3, BF16, BF16)]
    pl = plan(mixed, 4)
    assert pl.bucket_dtype == [BF16, F32]
    assert pl.bucket_of == [0, 1, 0] and pl.bucket_off == [0, 0, 2]
    assert pl.bucket_S == [3, 2]


def test_one_allgather_input_with_groups_by_dtype_pair():
    params = [Param(10, shard_dtype=F32, param_dtype=BF16), Param(3, shard_dtype=F32, param_dtype=F32),
              Param(7, shard_dtype=F32, param_dtype=BF16), Param(1, shard_dtype=BF16, param_dtype=BF16)]
    pl = plan(params, 2)
    assert pl.group_pair == [(F32, BF16), (F32, F32), (BF16, BF16)]
    assert pl.chunk == [5, 2, 4, 1]
    assert pl.group_of == [0, 1, 0, 2] and pl.group_elem_off == [0, 0, 5, 0]
    # group 0: 9 BF16 = 18 B -> group 1 at 32, 2 FP32 = 8 B -> group 2 at 48, 1 BF16 -> 64
    assert pl.group_byte_off == [0, 32, 48] and pl.S_ag == 64


def test_empty_layout_and_empty_parameters():
    pl = plan([], 4)
    assert pl.bucket_dtype == [] and pl.group_pair == [] and pl.S_ag == 0
    assert oracle.pack_reduce_scatter(pl, []) == []
    assert oracle.allgather_copy_in(pl, []).size == 0
    pl = plan([Param(0, BF16, BF16), Param(0)], 3)
    assert pl.chunk == [0, 0] and pl.bucket_S == [0, 0] and pl.S_ag == 0
    bufs = oracle.pack_reduce_scatter(pl, [np.zeros(0, np.uint16), np.zeros(0, np.uint32)])
    assert [b.size for b in bufs] == [0, 0]


def test_world_size_one_is_plain_concatenation():
    rng = np.random.default_rng(11)
    params = [Param(5, BF16, F32), Param(3, F32, F32), Param(4, F32, BF16)]
    grads = [rand_bits(rng, p.numel, p.grad_dtype) for p in params]
    pl = plan(params, 1)
    assert pl.chunk == [5, 3, 4]
    f32buf, bf16buf = oracle.pack_reduce_scatter(pl, grads)
    assert np.array_equal(f32buf, np.concatenate([torch_cast(grads[0], BF16, F32), grads[1]]))
    assert np.array_equal(bf16buf, torch_cast(grads[2], F32, BF16))


# ---------------------------------------------------------------------------
# Brute force on tiny layouts.
# ---------------------------------------------------------------------------
def _pack_case(params, W, seed):
    rng = np.random.default_rng(seed)
    grads = [rand_bits(rng, p.numel, p.grad_dtype) for p in params]
    got = oracle.pack_reduce_scatter(plan(params, W), grads)
    want = brute_pack(params, W, grads)
    assert len(got) == len(want)
    for a, b in zip(got, want):
        assert a.dtype == b.dtype and np.array_equal(a, b), (params, W)


def _gather_case(params, W, seed):
    rng = np.random.default_rng(seed)
    pl = plan(params, W)
    shards = [[rand_bits(rng, c, p.shard_dtype) for p, c in zip(params, pl.chunk)] for _ in range(W)]
    rows = []
    for r in range(W):
        got = oracle.allgather_copy_in(pl, shards[r])
        want, where = brute_copy_in(params, shards[r])
        assert np.array_equal(got, want), (params, W, r)
        rows.append(got)
    gathered = np.concatenate(rows)
    got = oracle.allgather_copy_out(pl, gathered)
    want = brute_copy_out(params, W, gathered, where)
    for a, b in zip(got, want):
        assert np.array_equal(a, b), (params, W)


def test_brute_force_pack_one_and_two_params_exhaustive():
    dts = (F32, BF16)
    for W in range(1, 6):
        for n in range(14):
            for gd, rd in itertools.product(dts, dts):
                _pack_case([Param(n, gd, rd)], W, seed=n * 7 + W)
    k = 0
    for W in range(1, 6):
        for n1, n2 in itertools.product(range(14), range(14)):
            for g1, r1, g2, r2 in itertools.product(dts, dts, dts, dts):
                _pack_case([Param(n1, g1, r1), Param(n2, g2, r2)], W, seed=k)
                k += 1


def test_brute_force_pack_three_params_sampled():
    rnd = random.Random(5)
    dts = (F32, BF16)
    for k in range(1500):
        W = rnd.randint(1, 5)
        params = [Param(rnd.randint(0, 13), rnd.choice(dts), rnd.choice(dts)) for _ in range(3)]
        _pack_case(params, W, seed=10_000 + k)


def test_brute_force_copy_in_out_one_and_two_params_exhaustive():
    dts = (F32, BF16)
    for W in range(1, 6):
        for n in range(14):
            for sd, pd in itertools.product(dts, dts):
                _gather_case([Param(n, shard_dtype=sd, param_dtype=pd)], W, seed=n + 100 * W)
    k = 0
    rnd = random.Random(9)
    for W in range(1, 6):
        for n1, n2 in itertools.product(range(14), range(14)):
            s1, p1, s2, p2 = (rnd.choice(dts) for _ in range(4))
            _gather_case([Param(n1, shard_dtype=s1, param_dtype=p1),
                          Param(n2, shard_dtype=s2, param_dtype=p2)], W, seed=k)
            k += 1


def test_brute_force_copy_in_out_three_params_sampled():
    rnd = random.Random(6)
    dts = (F32, BF16)
    for k in range(600):
        W = rnd.randint(1, 5)
        params = [Param(rnd.randint(0, 13), shard_dtype=rnd.choice(dts), param_dtype=rnd.choice(dts))
                  for _ in range(3)]
        _gather_case(params, W, seed=20_000 + k)


def test_pack_samples_match_whole_pack():
    rng = np.random.default_rng(21)
    params = [Param(37, BF16, F32), Param(5, F32, BF16), Param(64, F32, F32), Param(3, BF16, BF16)]
    grads = [rand_bits(rng, p.numel, p.grad_dtype) for p in params]
    pl = plan(params, 8)
    whole = oracle.pack_reduce_scatter(pl, grads)
    for b, buf in enumerate(whole):
        idx = np.arange(buf.size)
        assert np.array_equal(oracle.pack_samples(pl, grads, b, idx), buf)


# ---------------------------------------------------------------------------
# Invariants.
# ---------------------------------------------------------------------------
def test_padding_slots_are_zero_and_sizes_add_up():
    rnd = random.Random(17)
    dts = (F32, BF16)
    for k in range(300):
        W = rnd.choice([1, 2, 3, 4, 8, 64])
        params = [Param(rnd.randint(0, 200), rnd.choice(dts), rnd.choice(dts)) for _ in range(rnd.randint(1, 5))]
        pl = plan(params, W)
        total = sum(W * S for S in pl.bucket_S)
        n = sum(p.numel for p in params)
        assert total >= n
        assert (total == n) == all(p.numel % W == 0 for p in params)
        # gradients with no zero bits anywhere: every zero in the buffer is padding
        grads = [np.full(p.numel, 0x3F80 if p.grad_dtype == BF16 else 0x3F800000, NP[p.grad_dtype])
                 for p in params]
        bufs = oracle.pack_reduce_scatter(pl, grads)
        assert sum(int(np.count_nonzero(b == 0)) for b in bufs) == total - n


def test_roundtrip_copy_in_then_copy_out_reproduces_parameters():
    rnd = random.Random(23)
    rng = np.random.default_rng(23)
    dts = (F32, BF16)
    for k in range(200):
        W = rnd.choice([1, 2, 3, 4, 8])
        params = [Param(rnd.randint(0, 100), shard_dtype=rnd.choice(dts), param_dtype=rnd.choice(dts))
                  for _ in range(rnd.randint(1, 4))]
        pl = plan(params, W)
        # full parameters whose values are representable in every dtype
        full = [torch_cast(rand_bits(rng, p.numel, BF16), BF16, p.shard_dtype) for p in params]
        rows = []
        for r in range(W):
            shards = []
            for p, c, x in zip(params, pl.chunk, full):
                padded = np.pad(x, (0, c * W - p.numel))
                shards.append(padded.reshape(W, c)[r].copy())
            rows.append(oracle.allgather_copy_in(pl, shards))
        got = oracle.allgather_copy_out(pl, np.concatenate(rows))
        for p, x, y in zip(params, full, got):
            assert np.array_equal(y, torch_cast(x, p.shard_dtype, p.param_dtype))
            assert np.array_equal(torch_cast(y, p.param_dtype, p.shard_dtype), x)


# ---------------------------------------------------------------------------
# Number formats.
# ---------------------------------------------------------------------------
RNE_TABLE = [  # (FP32 bits, BF16 bits): IEEE-754 round to nearest, ties to even
    (0x3F800000, 0x3F80),   # 1.0 exact
    (0x3F808000, 0x3F80),   # 1 + 2^-8: tie, 0x3F80 is even
    (0x3F818000, 0x3F82),   # 1 + 3*2^-8: tie, 0x3F82 is even
    (0x3F808001, 0x3F81),   # just above the tie
    (0x3F807FFF, 0x3F80),   # just below the tie
    (0xBF808000, 0xBF80),   # negative tie
    (0xBF818000, 0xBF82),
    (0x7F7FC99E, 0x7F80),   # 3.4e38 rounds past the largest BF16 to +inf
    (0x7F7FFFFF, 0x7F80),   # FLT_MAX -> +inf
    (0x7F7F8000, 0x7F80),   # tie between BF16 max and 2^128 -> inf (even)
    (0x7F7F7FFF, 0x7F7F),   # below that tie stays finite
    (0xFF7FFFFF, 0xFF80),
    (0x000116C2, 0x0001),   # 1e-40, subnormal: nearest is 0x0001
    (0x00000001, 0x0000),   # smallest subnormal rounds to +0
    (0x80000001, 0x8000),   # ... and to -0 when negative
    (0x00008000, 0x0000),   # tie between 0 and 0x0001 -> even (0)
    (0x00018000, 0x0002),   # tie between 0x0001 and 0x0002 -> even
    (0x00008001, 0x0001),
    (0x007FFFFF, 0x0080),   # largest subnormal rounds up to the smallest normal
    (0x00000000, 0x0000), (0x80000000, 0x8000),
    (0x7F800000, 0x7F80), (0xFF800000, 0xFF80),
]


def test_rne_textbook_table():
    got = oracle.f32_to_bf16(np.array([a for a, _ in RNE_TABLE], np.uint32))
    assert [int(v) for v in got] == [b for _, b in RNE_TABLE]


def test_rne_matches_torch_on_structured_and_random_patterns():
    hi = np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)
    lows = np.array([0x0000, 0x0001, 0x3FFF, 0x4000, 0x7FFF, 0x8000, 0x8001, 0xC000, 0xFFFF], np.uint32)
    x = (hi[:, None] | lows[None, :]).reshape(-1)
    x = np.concatenate([x, np.random.default_rng(31).integers(0, 1 << 32, 1 << 22, dtype=np.uint64).astype(np.uint32)])
    finite = (x & 0x7F800000) != 0x7F800000
    inf = (x & 0x7FFFFFFF) == 0x7F800000
    keep = finite | inf
    assert np.array_equal(oracle.f32_to_bf16(x[keep]), torch_cast(x[keep], F32, BF16))


def _exact_rne(u: int) -> int:
    """Round the exact value of FP32 pattern u to BF16 by scaling to the BF16
    quantum of its binade and rounding with Python's ties-to-even round()."""
    x = Fraction(*np.uint32(u).view(np.float32).item().as_integer_ratio())
    if x == 0:
        return (u >> 16) & 0x8000
    e = max(-126, abs(x).numerator.bit_length() - abs(x).denominator.bit_length())
    while Fraction(2) ** e > abs(x):
        e -= 1
    while Fraction(2) ** (e + 1) <= abs(x):
        e += 1
    e = max(-126, e)
    q = Fraction(2) ** (e - 7)
    y = round(x / q) * q
    if abs(y) >= Fraction(2) ** 128:
        return 0xFF80 if x < 0 else 0x7F80
    f = np.float32(float(y))                # exact: y is a BF16 value
    bits = int(f.view(np.uint32))
    assert bits & 0xFFFF == 0
    if y == 0:
        bits = 0x80000000 if x < 0 else 0
    return bits >> 16


def test_rne_matches_exact_rational_rounding():
    rng = np.random.default_rng(37)
    x = rng.integers(0, 1 << 32, 6000, dtype=np.uint64).astype(np.uint32)
    ties = (x & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    sub = x & np.uint32(0x807FFFFF)                # subnormals
    cases = np.concatenate([x, ties, sub, np.array([a for a, _ in RNE_TABLE], np.uint32)])
    cases = cases[(cases & 0x7F800000) != 0x7F800000]
    got = oracle.f32_to_bf16(cases)
    for u, g in zip(cases.tolist(), got.tolist()):
        assert g == _exact_rne(u), hex(u)


def test_nan_keeps_sign_and_payload_and_is_quiet():
    rng = np.random.default_rng(41)
    mant = rng.integers(1, 1 << 23, 20000, dtype=np.uint64).astype(np.uint32)
    sign = rng.integers(0, 2, 20000, dtype=np.uint64).astype(np.uint32) << np.uint32(31)
    x = sign | np.uint32(0x7F800000) | mant
    got = oracle.f32_to_bf16(x).astype(np.uint32)
    assert np.all((got & 0x7F80) == 0x7F80) and np.all(got & 0x0040)
    assert np.array_equal(got >> 15, x >> 31)
    assert np.array_equal(got & 0x3F, (x >> 16) & 0x3F)


def test_bf16_to_f32_exact_for_every_pattern():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_to_f32(h)
    nan = ((h & 0x7F80) == 0x7F80) & ((h & 0x7F) != 0)
    assert np.array_equal(got[~nan], torch_cast(h[~nan], BF16, F32))
    assert np.array_equal(got[nan], h[nan].astype(np.uint32) << np.uint32(16))


def test_segment_entry_points_compose_to_the_whole_operations():
    rng = np.random.default_rng(43)
    params = [Param(37, BF16, F32, F32, BF16), Param(5, F32, BF16, BF16, BF16), Param(64, F32, F32, F32, F32)]
    W = 4
    pl = plan(params, W)
    grads = [rand_bits(rng, p.numel, p.grad_dtype) for p in params]
    whole = oracle.pack_reduce_scatter(pl, grads)
    parts = [np.full_like(b, 0xAB) for b in whole]
    for r in range(W):
        for p in range(len(params)):
            oracle.pack_segment(pl, grads, parts, r, p)
    assert all(np.array_equal(a, b) for a, b in zip(parts, whole))
    shards = [rand_bits(rng, c, p.shard_dtype) for p, c in zip(params, pl.chunk)]
    row = np.full(pl.S_ag, 0xAB, np.uint8)
    oracle.allgather_copy_in_clear(pl, row)
    for p in range(len(params)):
        oracle.allgather_copy_in_segment(pl, shards, row, p)
    assert np.array_equal(row, oracle.allgather_copy_in(pl, shards))
    gathered = np.concatenate([row] * W)
    full = [np.zeros(p.numel, oracle.DTYPE_NP[p.param_dtype]) for p in params]
    for p in range(len(params)):
        for r in range(W):
            oracle.allgather_copy_out_segment(pl, gathered, full, p, r)
    assert all(np.array_equal(a, b) for a, b in zip(full, oracle.allgather_copy_out(pl, gathered)))


# ---------------------------------------------------------------------------
# Reduce-scatter copy-out: reduced bucket rows -> sharded gradients.
# ---------------------------------------------------------------------------
def brute_rs_copy_out(params, W, rows):
    """Split each bucket row at the cumulative chunk sizes of its parameters
    and cast each piece to the parameter's shard dtype."""
    out = [None] * len(params)
    for b, rd in enumerate(first_appearance([p.reduce_dtype for p in params])):
        members = [k for k, p in enumerate(params) if p.reduce_dtype == rd]
        sizes = [-(-params[k].numel // W) for k in members]
        pieces = np.split(rows[b], np.cumsum(sizes)[:-1]) if members else []
        for k, piece in zip(members, pieces):
            out[k] = torch_cast(piece, rd, params[k].shard_dtype)
    return out


def test_rs_copy_out_gives_the_printed_grad_shards():
    # [Unit], FlatParameter section: with one contributing rank the reduced
    # row is rank 0's packed row, and its sharded gradient is the printed one.
    g = sections("linear4x4_w2.txt")
    grad = np.zeros((4, 4), np.float32)
    grad[1] = np.float32(1.2830595970)
    pl = plan([Param(16)], 2)
    buf, = oracle.pack_reduce_scatter(pl, [grad.view(np.uint32).reshape(-1)])
    shard0, = oracle.reduce_scatter_copy_out(pl, [buf[:8]])
    shard1, = oracle.reduce_scatter_copy_out(pl, [buf[8:]])
    assert np.array_equal(shard0, f32_bits(g["rank0_grad_shard"]))
    assert np.array_equal(shard1, f32_bits(g["rank1_grad_shard"]))


def test_rs_copy_out_brute_force_exhaustive_small():
    dts = (F32, BF16)
    k = 0
    for W in range(1, 5):
        for n1, n2 in itertools.product(range(0, 12, 3), range(0, 12, 2)):
            for g1, r1, s1, r2, s2 in itertools.product(dts, dts, dts, dts, dts):
                params = [Param(n1, g1, r1, s1), Param(n2, F32, r2, s2)]
                pl = plan(params, W)
                rng = np.random.default_rng(k)
                rows = [rand_bits(rng, S, dt) for dt, S in zip(pl.bucket_dtype, pl.bucket_S)]
                got = oracle.reduce_scatter_copy_out(pl, rows)
                want = brute_rs_copy_out(params, W, rows)
                for a, b in zip(got, want):
                    assert a.dtype == b.dtype and np.array_equal(a, b), (params, W)
                k += 1


def test_pack_then_rs_copy_out_returns_each_ranks_chunk():
    # With one contributing rank, row r of the packed buffer is the reduced
    # row, and the sharded gradient is chunk r of the gradient, padded, cast
    # g -> rho -> sigma.
    rnd = random.Random(29)
    rng = np.random.default_rng(29)
    dts = (F32, BF16)
    for k in range(200):
        W = rnd.choice([1, 2, 3, 4, 8])
        params = [Param(rnd.randint(0, 60), rnd.choice(dts), rnd.choice(dts), rnd.choice(dts))
                  for _ in range(rnd.randint(1, 4))]
        pl = plan(params, W)
        grads = [rand_bits(rng, p.numel, p.grad_dtype) for p in params]
        bufs = oracle.pack_reduce_scatter(pl, grads)
        for r in range(W):
            rows = [buf[r * S:(r + 1) * S] for buf, S in zip(bufs, pl.bucket_S)]
            shards = oracle.reduce_scatter_copy_out(pl, rows)
            for p, c, g, got in zip(params, pl.chunk, grads, shards):
                chunk = np.pad(g, (0, c * W - p.numel)).reshape(W, c)[r] if c else g[:0]
                want = torch_cast(torch_cast(chunk, p.grad_dtype, p.reduce_dtype), p.reduce_dtype, p.shard_dtype)
                assert np.array_equal(got, want)


# ---------------------------------------------------------------------------
# Row-chunk mode: pad along dim 0 to a multiple of W rows, split in W row chunks.
# ---------------------------------------------------------------------------
def brute_pack_rows(params, shapes, W, grads):
    """Definition written with 2-D arrays: pad the (d0, row) view of each
    gradient with zero rows to a multiple of W, split it into W row chunks,
    and lay every parameter's chunk r side by side in row r."""
    outs = []
    for rd in first_appearance([p.reduce_dtype for p in params]):
        blocks = []
        for p, (d0, row), g in zip(params, shapes, grads):
            if p.reduce_dtype != rd:
                continue
            v = torch_cast(g, p.grad_dtype, rd).reshape(d0, row)
            rows_per_rank = -(-d0 // W)
            v = np.pad(v, ((0, rows_per_rank * W - d0), (0, 0)))
            blocks.append(v.reshape(W, rows_per_rank * row))
        outs.append(np.hstack(blocks).reshape(-1))
    return outs


def test_row_mode_pack_matches_the_row_definition():
    rnd = random.Random(31)
    dts = (F32, BF16)
    for k in range(400):
        W = rnd.choice([1, 2, 3, 4, 5, 7, 8])
        shapes = [(rnd.randint(0, 11), rnd.randint(1, 6)) for _ in range(rnd.randint(1, 4))]
        params = [Param(d0 * row, rnd.choice(dts), rnd.choice(dts)) for d0, row in shapes]
        pl = plan(params, W, row_elems=[row for _, row in shapes])
        rng = np.random.default_rng(k)
        grads = [rand_bits(rng, p.numel, p.grad_dtype) for p in params]
        got = oracle.pack_reduce_scatter(pl, grads)
        want = brute_pack_rows(params, shapes, W, grads)
        for a, b in zip(got, want):
            assert np.array_equal(a, b), (shapes, W)


def test_row_mode_agrees_with_flattening_when_rows_divide():
    rnd = random.Random(37)
    for k in range(200):
        W = rnd.choice([1, 2, 4, 8])
        shapes = [(W * rnd.randint(0, 5), rnd.randint(1, 9)) for _ in range(rnd.randint(1, 4))]
        params = [Param(d0 * row, BF16, F32, F32, BF16) for d0, row in shapes]
        a = plan(params, W, row_elems=[row for _, row in shapes])
        b = plan(params, W)
        assert a.chunk == b.chunk and a.bucket_S == b.bucket_S and a.S_ag == b.S_ag


def test_row_mode_linear_examples():
    # Linear(4, 4) at W = 2: two rows per rank either way, so the printed
    # shard of rank 0 (rows 0-1) is the same under both readings.
    assert plan([Param(16)], 2, row_elems=[4]).chunk == plan([Param(16)], 2).chunk == [8]
    # Linear(6, 6) at W = 4: ceil(6/4) = 2 rows = 12 elements per rank in row
    # mode, against the flattened 9 that the wrap-policy printout shows.
    assert plan([Param(36)], 4, row_elems=[6]).chunk == [12]
    assert plan([Param(36)], 4).chunk == [9]
    # Linear(3, 3) at W = 4: one row per rank in row mode, 4 rows = 12 slots.
    assert plan([Param(9)], 4, row_elems=[3]).chunk == [3]


# ---------------------------------------------------------------------------
# Emulated reduce-scatter: sum over ranks in rank order, rounded per add.
# ---------------------------------------------------------------------------
def _ers(dt, rows):
    pl = plan([Param(len(rows[0]), dt, dt)], 1)
    return oracle.emulated_reduce_scatter(pl, [[np.asarray(r, NP[dt])] for r in rows])[0]


def f32b(*vals):
    return np.array(vals, np.float32).view(np.uint32)


def test_emulated_rs_textbook_sums():
    # one rank: identity
    x = f32b(1.5, -0.0, 3e-45, 7.0)
    assert np.array_equal(_ers(F32, [x]), x)
    # small integers add exactly in any order
    rng = np.random.default_rng(3)
    ints = rng.integers(-1000, 1000, (8, 50))
    got = _ers(F32, [f32b(*row) for row in ints])
    assert np.array_equal(got.view(np.float32), ints.sum(0).astype(np.float32))
    # order matters, and it is rank order: (1 + 2^24) rounds to 2^24 (tie to
    # even) before -2^24 is added, while 2^24 - 2^24 + 1 = 1
    assert _ers(F32, [f32b(1.0), f32b(2.0**24), f32b(-(2.0**24))]).view(np.float32)[0] == 0.0
    assert _ers(F32, [f32b(2.0**24), f32b(-(2.0**24)), f32b(1.0)]).view(np.float32)[0] == 1.0
    # subnormals are kept: 2 * smallest subnormal
    assert _ers(F32, [np.array([1], np.uint32), np.array([1], np.uint32)])[0] == 2


def test_emulated_rs_nan_sums_are_canonical():
    inf, ninf = 0x7F800000, 0xFF800000
    assert _ers(F32, [np.array([inf], np.uint32), np.array([ninf], np.uint32)])[0] == 0x7FC00000
    payload = 0xFFA12345                       # negative signalling NaN with a payload
    assert _ers(F32, [np.array([payload], np.uint32), np.array([0x3F800000], np.uint32)])[0] == 0x7FC00000
    assert _ers(F32, [np.array([0x3F800000], np.uint32), np.array([payload], np.uint32)])[0] == 0x7FC00000
    assert _ers(F32, [np.array([payload], np.uint32)])[0] == payload   # one rank: no addition
    assert _ers(BF16, [np.array([0x7F80]), np.array([0xFF80])])[0] == 0x7FC0
    assert _ers(BF16, [np.array([0xFFA1]), np.array([0x3F80])])[0] == 0x7FC0
    # -0 survives when nothing is added, and -0 + -0 = -0
    assert _ers(F32, [np.array([0x80000000], np.uint32)])[0] == 0x80000000
    assert _ers(F32, [np.array([0x80000000], np.uint32)] * 2)[0] == 0x80000000


def test_emulated_rs_bf16_rounds_every_partial_sum():
    one, tiny = 0x3F80, 0x3B80                 # 1.0 and 2^-8 in BF16
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even -> 1.0, every time
    assert _ers(BF16, [np.array([one]), np.array([tiny]), np.array([tiny])])[0] == one
    # 2^-8 + 2^-8 = 2^-7 first, then 1 + 2^-7 is exact: 0x3F81
    assert _ers(BF16, [np.array([tiny]), np.array([tiny]), np.array([one])])[0] == 0x3F81


def _bf16_exact_sum(a: int, b: int) -> int:
    """The BF16 pattern nearest to the exact sum of the finite BF16 patterns a
    and b (ties to even): the sum as a Fraction, scaled to the BF16 quantum
    of its binade and rounded with Python's ties-to-even round()."""
    val = lambda u: Fraction(*np.uint32(u << 16).view(np.float32).item().as_integer_ratio())  # noqa: E731
    x = val(a) + val(b)
    if x == 0:                                 # -0 only from -0 + -0
        return 0x8000 if (a & 0x8000) and (b & 0x8000) else 0
    e = abs(x).numerator.bit_length() - abs(x).denominator.bit_length()
    while Fraction(2) ** e > abs(x):
        e -= 1
    while Fraction(2) ** (e + 1) <= abs(x):
        e += 1
    q = Fraction(2) ** (max(-126, e) - 7)
    y = round(x / q) * q
    if abs(y) >= Fraction(2) ** 128:
        return 0xFF80 if x < 0 else 0x7F80
    bits = int(np.float32(float(y)).view(np.uint32))   # exact: y is a BF16 value
    if y == 0:
        bits = 0x80000000 if x < 0 else 0
    return bits >> 16


def test_emulated_rs_bf16_add_is_the_exactly_rounded_sum():
    """Each BF16 addition of the emulated reduce-scatter (binary32 sum, then
    round to nearest even) gives the BF16 value nearest to the exact sum of
    its two operands: binary32 keeps at least 2 x 8 + 1 significant bits, so
    the second rounding never moves a result.  Checked against exact
    rational rounding on random pairs, pairs a half BF16 step apart (ties
    and near-ties), every exponent gap from 0 to 40, subnormals and
    cancellations."""
    rng = np.random.default_rng(71)

    def finite(n):
        u = rng.integers(0, 1 << 16, 4 * n, dtype=np.uint64).astype(np.uint32)
        return u[(u & 0x7F80) != 0x7F80][:n]

    a = finite(3000)
    b = finite(3000)
    # half a BF16 step of a, give or take a few units of the partner's last place
    ea = (a >> 7) & 0xFF
    half = ((np.maximum(ea, 9) - 8) << 7) | rng.integers(0, 4, a.size).astype(np.uint32)
    half |= rng.integers(0, 2, a.size).astype(np.uint32) << 15
    gap = rng.integers(0, 41, a.size).astype(np.uint32)
    shifted = ((np.maximum(ea, gap + 1) - gap) << 7) | (b & 0x807F)
    sub = a & 0x807F                           # subnormals (and zeros)
    cancel = (a ^ 0x8000) + rng.integers(0, 3, a.size).astype(np.uint32)
    cancel = np.where((cancel & 0x7F80) == 0x7F80, a ^ 0x8000, cancel) & 0xFFFF
    A = np.concatenate([a, a, a, sub, a, sub]).astype(np.uint16)
    B = np.concatenate([b, half, shifted, b & 0x807F, cancel, sub[::-1]]).astype(np.uint16)
    got = _ers(BF16, [A, B])
    for x, y, g in zip(A.tolist(), B.tolist(), got.tolist()):
        assert g == _bf16_exact_sum(x, y), (hex(x), hex(y), hex(g))


def test_emulated_rs_matches_sequential_float32_and_pack_composition():
    rng = np.random.default_rng(47)
    params = [Param(37, BF16, F32, F32), Param(20, F32, BF16, BF16), Param(64, F32, F32, BF16)]
    W = 4
    pl = plan(params, W)
    grads = [[rand_bits(rng, p.numel, p.grad_dtype) for p in params] for _ in range(W)]
    # finite inputs only here: numpy keeps a NaN operand's payload, the
    # definition does not
    packed = [oracle.pack_reduce_scatter(pl, grads[q]) for q in range(W)]
    summed = oracle.emulated_reduce_scatter(pl, packed)
    for b, dt in enumerate(pl.bucket_dtype):
        if dt == F32:
            acc = packed[0][b].view(np.float32).copy()
            for q in range(1, W):
                acc = (acc + packed[q][b].view(np.float32)).astype(np.float32)
            assert np.array_equal(summed[b], acc.view(np.uint32))
        else:
            acc = torch_cast(packed[0][b], BF16, F32).view(np.float32)
            for q in range(1, W):
                s = (acc + torch_cast(packed[q][b], BF16, F32).view(np.float32)).astype(np.float32)
                acc = torch_cast(torch_cast(s.view(np.uint32), F32, BF16), BF16, F32).view(np.float32)
            assert np.array_equal(summed[b], torch_cast(acc.view(np.uint32), F32, BF16))
    # rank r's sharded gradients after the emulated reduce-scatter
    for r in range(W):
        rows = [buf[r * S:(r + 1) * S] for buf, S in zip(summed, pl.bucket_S)]
        shards = oracle.reduce_scatter_copy_out(pl, rows)
        assert [s.size for s in shards] == pl.chunk
