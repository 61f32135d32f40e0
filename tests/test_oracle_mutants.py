"""The oracle's pins must catch plausible mistakes in the oracle itself.

Each case below plants one mistake (a dropped term, an off-by-one index, a
wrong comparison, a lost bit) in a temporary copy of ``oracle/fsdp_oracle.c``,
builds it, swaps it in for the real oracle library, and re-runs the pins of
tests/test_oracle_pins.py.  The mutants run in this process, so every one of
them keeps all its memory accesses inside the buffers it is given.  At least one pin must fail for every mutant.
The planner mutants at the end do the same with the oracle's Python planner;
the oracle's wrappers refuse a plan whose offsets do not fit their buffers,
so a broken plan cannot make the C loops write out of bounds.
Everything runs on the CPU; the mistakes are planted in the oracle only.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

MUTANTS = {
    "pack: source index off by one":
        ("int64_t j = (int64_t)r * chunk + i;\n    int64_t d",
         "int64_t j = (int64_t)r * chunk + i + (i > 0);\n    int64_t d"),
    "pack: last real element treated as padding":
        ("if (j < numel)\n      cast_element(grad, grad_dtype, j, buf, rho, d);",
         "if (j + 1 < numel)\n      cast_element(grad, grad_dtype, j, buf, rho, d);"),
    "pack: padding filled with wrapped values":
        ("else\n      store_zero(buf, rho, d);\n  }\n}\n\nvoid oracle_pack_reduce_scatter",
         "else\n      cast_element(grad, grad_dtype, j % numel, buf, rho, d);\n  }\n}\n\nvoid oracle_pack_reduce_scatter"),
    "pack: bucket offset dropped":
        ("(int64_t)r * S_b + bucket_off + i;",
         "(int64_t)r * S_b + i;"),
    "pack: rank stride uses chunk instead of row length":
        ("(int64_t)r * S_b + bucket_off + i;",
         "(int64_t)r * chunk + bucket_off + i;"),
    "rne: ties always round down":
        ("if (d_lo < d_hi) return toward_zero;", "if (d_lo <= d_hi) return toward_zero;"),
    "rne: ties to odd":
        ("return (toward_zero & 1) ? away : toward_zero;", "return (toward_zero & 1) ? toward_zero : away;"),
    "rne: NaN not quieted":
        ("return (uint16_t)((u >> 16) | 0x0040);", "return (uint16_t)(u >> 16);"),
    "rne: subnormal scale wrong":
        ("mag = ldexp((double)f, -126 - 7);", "mag = ldexp((double)f, -127 - 7);"),
    "bf16 decode: exponent bias wrong":
        ("mag = ldexp(128.0 + (double)f, e - 127 - 7);", "mag = ldexp(128.0 + (double)f, e - 126 - 7);"),
    "copy-in: element offset in group dropped":
        ("cast_element(shard, shard_dtype, i, base, param_dtype, group_elem_off + i);",
         "cast_element(shard, shard_dtype, i, base, param_dtype, i);"),
    "copy-in: gap bytes not cleared":
        ("memset(ag_in, 0, (size_t)S_ag);", "memset(ag_in, 0xAB, (size_t)S_ag);"),
    "copy-out: group start dropped":
        ("(int64_t)r * S_ag + group_byte_off + (group_elem_off + i) * sz;",
         "(int64_t)r * S_ag + (group_elem_off + i) * sz;"),
    "copy-out: row stride taken as the chunk":
        ("const uint8_t *from = ag_out + (int64_t)r * S_ag + group_byte_off",
         "const uint8_t *from = ag_out + (int64_t)r * chunk * sz + group_byte_off"),
    "rs copy-out: bucket offset dropped":
        ("cast_element(rows[b], bucket_dtype[b], bucket_off[p] + i, sharded[p], shard_dtype[p], i);",
         "cast_element(rows[b], bucket_dtype[b], i, sharded[p], shard_dtype[p], i);"),
    "rs copy-out: last slot of every chunk skipped":
        ("    for (int64_t i = 0; i < chunk[p]; ++i)\n      cast_element(rows[b], bucket_dtype[b], bucket_off[p] + i",
         "    for (int64_t i = 0; i < chunk[p] - 1; ++i)\n      cast_element(rows[b], bucket_dtype[b], bucket_off[p] + i"),
    "emulated rs: ranks summed in reverse order":
        ("for (int32_t q = 1; q < n_inputs; ++q) acc = add_f32(acc, f32_of_bits(((const uint32_t *)inputs[q])[i]));",
         "for (int32_t q = n_inputs - 1; q >= 1; --q) acc = add_f32(acc, f32_of_bits(((const uint32_t *)inputs[q])[i]));"),
    "emulated rs: bf16 partial sums not rounded":
        ("acc = (sum != sum) ? (uint16_t)0x7FC0 : oracle_f32_to_bf16(bits_of_f32(sum));",
         "acc = (sum != sum) ? (uint16_t)0x7FC0 : (uint16_t)(bits_of_f32(sum) >> 16);"),
    "emulated rs: NaN sums keep a machine payload":
        ("  if (s != s) return f32_of_bits(0x7FC00000u);\n  return s;",
         "  return s;"),
}

PINS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_") and callable(getattr(pins, n))]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name!r} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(lib), str(path), "-lm"],
                   check=True)
    saved = oracle._load()
    oracle._lib = oracle._bind(ctypes.CDLL(os.fspath(lib)))
    failed = []
    try:
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                failed.append(pin.__name__)
                break
    finally:
        oracle._lib = saved
    assert failed, f"no pin caught mutant {name!r}"


# Mistakes planted in the oracle's planner (Python).  A mutated copy of
# oracle.plan is compiled from its source in the oracle module's namespace and
# put in place of the real one, both in the oracle module and where the pins
# imported it by name.
PLAN_MUTANTS = {
    "plan: chunk rounded down":
        ("c = _ceil_div(p.numel, W)", "c = p.numel // W"),
    "plan: row chunk counted in elements, not rows":
        ("c = _ceil_div(p.numel // rows_of, W) * rows_of", "c = _ceil_div(p.numel, W)"),
    "plan: bucket offset counts every earlier parameter":
        ("pl.bucket_off.append(pl.bucket_S[b])", "pl.bucket_off.append(sum(pl.chunk[:-1]))"),
    "plan: buckets keyed by grad dtype":
        ("if p.reduce_dtype not in bucket_index:\n"
         "            bucket_index[p.reduce_dtype] = len(pl.bucket_dtype)\n"
         "            pl.bucket_dtype.append(p.reduce_dtype)\n"
         "            pl.bucket_S.append(0)\n"
         "        b = bucket_index[p.reduce_dtype]",
         "if p.grad_dtype not in bucket_index:\n"
         "            bucket_index[p.grad_dtype] = len(pl.bucket_dtype)\n"
         "            pl.bucket_dtype.append(p.grad_dtype)\n"
         "            pl.bucket_S.append(0)\n"
         "        b = bucket_index[p.grad_dtype]"),
    "plan: group element offset counts every earlier group":
        ("pl.group_elem_off.append(pl.group_elems[g])", "pl.group_elem_off.append(sum(pl.group_elems))"),
    "plan: groups keyed by param dtype only":
        ("pair = (p.shard_dtype, p.param_dtype)", "pair = (p.param_dtype, p.param_dtype)"),
    "plan: group starts not aligned":
        ("start = _align16(end)", "start = end"),
    "plan: all-gather row not rounded up":
        ("pl.S_ag = _align16(end)", "pl.S_ag = end"),
    "plan: group byte size taken as FP32":
        ("end = start + pl.group_elems[g] * DTYPE_SIZE[pi]", "end = start + pl.group_elems[g] * 4"),
}


@pytest.mark.parametrize("name", sorted(PLAN_MUTANTS))
def test_pins_catch_planner_mutant(name):
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(oracle.plan))
    old, new = PLAN_MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name!r} not found exactly once"
    namespace = dict(vars(oracle))
    exec(compile(src.replace(old, new), "<mutant plan>", "exec"), namespace)
    real = oracle.plan
    oracle.plan = pins.plan = namespace["plan"]
    failed = []
    try:
        for pin in PINS:
            try:
                pin()
            except (AssertionError, ValueError):
                failed.append(pin.__name__)
                break
    finally:
        oracle.plan = pins.plan = real
    assert failed, f"no pin caught planner mutant {name!r}"
