"""Seeded synthetic workloads: layouts and input values.

This module is shared by the tests, the benchmark and the CPU oracle's
callers, so it holds none of the packing arithmetic: no chunk sizes, no
offsets, no padding and no FP32 -> BF16 rounding.  It only says which
parameters a fully_shard group has (names, shapes, the four dtypes of the
mixed-precision policy) and draws their values from seeded generators.

Dtypes are the strings ``"f32"`` and ``"bf16"``; each consumer maps them to
its own codes.  Values are raw bit patterns in numpy arrays: ``uint32`` for
FP32 and ``uint16`` for BF16.  BF16 values are drawn as FP32 normals whose low
16 bits are then dropped (the upper half of the FP32 pattern is a valid BF16
value with nearly the same distribution); this is a way to draw inputs, not
the cast the method performs.

Layouts follow the workloads the pages describe:
  * two blocks of two Linear(6, 6) without bias ("The unit you wrapped",
    auto_wrap_policy section);
  * a ~500-parameter transformer-like layout and its all-gather copy-in /
    copy-out ("FSDP2 per-parameter mixed precision" news item, results table);
  * the 50.3M-element mixed BF16 / FP32 pack (same item, the isolated H100
    packing test);
  * an 8-block 1.75B-parameter KDA-style layout (same item, KDA-style test).
"""
from __future__ import annotations

import math
import random
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class ParamSpec:
    name: str
    shape: tuple
    grad_dtype: str = "f32"
    reduce_dtype: str = "f32"
    shard_dtype: str = "f32"
    param_dtype: str = "f32"

    @property
    def numel(self) -> int:
        return int(math.prod(self.shape))


@dataclass(frozen=True)
class Workload:
    name: str
    W: int
    groups: tuple          # tuple of tuples of ParamSpec, one per fully_shard group
    std: float = 1.0
    seed: int = 0

    @property
    def n_params(self) -> int:
        return sum(len(g) for g in self.groups)


# ---------------------------------------------------------------------------
# Layouts
# ---------------------------------------------------------------------------
def tiny_two_blocks(W: int = 4, grouping: str = "linear") -> Workload:
    """Two blocks x two Linear(6, 6), no bias: 144 elements.

    Block 0 has FP32 gradients, block 1 BF16; reduce dtype FP32, shard FP32,
    param dtype BF16.  ``grouping`` picks the fully_shard units: one per Linear
    ("linear", 4 groups), one per block ("block", 2 groups) or one for the whole
    model ("model", 1 group).
    """
    lin = []
    for blk, gd in ((0, "f32"), (1, "bf16")):
        for name in ("a", "b"):
            lin.append(ParamSpec(f"{blk}.{name}.weight", (6, 6), grad_dtype=gd,
                                 reduce_dtype="f32", shard_dtype="f32", param_dtype="bf16"))
    if grouping == "linear":
        groups = tuple((p,) for p in lin)
    elif grouping == "block":
        groups = (tuple(lin[:2]), tuple(lin[2:]))
    elif grouping == "model":
        groups = (tuple(lin),)
    else:
        raise ValueError(grouping)
    return Workload(f"tiny_two_blocks_{grouping}", W, groups, std=1.0, seed=1000)


def transformer_500(W: int = 8, layers: int = 24, homogeneous: bool = False) -> Workload:
    """~500-parameter transformer-like layout, one fully_shard group per layer.

    Each layer: attn_norm[512] FP32, q/k/v/o [512, 512] BF16, mlp_norm[512]
    FP32, gate/up [1408, 512] BF16, down [512, 1408] BF16, and eight FP32
    scalar/vector parameters s0..s7 whose lengths are drawn from U{1..64}.
    Gradients are in the parameter's own dtype; reduce dtype FP32; local
    shards FP32; param dtype BF16 for the matrices and FP32 for the rest
    (``homogeneous``: BF16 for every parameter, one all-gather dtype group).
    """
    rnd = random.Random(2001)
    groups = []
    for layer in range(layers):
        g = [ParamSpec(f"l{layer}.attn_norm", (512,), "f32", "f32", "f32", "f32")]
        for m in ("q", "k", "v", "o"):
            g.append(ParamSpec(f"l{layer}.{m}", (512, 512), "bf16", "f32", "f32", "bf16"))
        g.append(ParamSpec(f"l{layer}.mlp_norm", (512,), "f32", "f32", "f32", "f32"))
        g.append(ParamSpec(f"l{layer}.gate", (1408, 512), "bf16", "f32", "f32", "bf16"))
        g.append(ParamSpec(f"l{layer}.up", (1408, 512), "bf16", "f32", "f32", "bf16"))
        g.append(ParamSpec(f"l{layer}.down", (512, 1408), "bf16", "f32", "f32", "bf16"))
        for s in range(8):
            g.append(ParamSpec(f"l{layer}.s{s}", (rnd.randint(1, 64),), "f32", "f32", "f32", "f32"))
        if homogeneous:
            g = [ParamSpec(p.name, p.shape, p.grad_dtype, p.reduce_dtype, p.shard_dtype, "bf16") for p in g]
        groups.append(tuple(g))
    return Workload(f"transformer500_W{W}" + ("_homogeneous" if homogeneous else ""), W, tuple(groups),
                    std=0.02, seed=1001)


def mixed_50m(W: int = 8, layers: int = 4) -> Workload:
    """The 50.3M-element mixed pack: one fully_shard group.

    4 layers at d=1024: norm1[1024] FP32, q/k/v/o [1024, 1024] BF16,
    norm2[1024] FP32, up [4096, 1024] BF16, down [1024, 4096] BF16
    (50,331,648 BF16 + 8,192 FP32 elements).  Reduce dtype FP32; local shards
    FP32; param dtype BF16 for the matrices, FP32 for the norms.
    """
    g = []
    for layer in range(layers):
        g.append(ParamSpec(f"l{layer}.norm1", (1024,), "f32", "f32", "f32", "f32"))
        for m in ("q", "k", "v", "o"):
            g.append(ParamSpec(f"l{layer}.{m}", (1024, 1024), "bf16", "f32", "f32", "bf16"))
        g.append(ParamSpec(f"l{layer}.norm2", (1024,), "f32", "f32", "f32", "f32"))
        g.append(ParamSpec(f"l{layer}.up", (4096, 1024), "bf16", "f32", "f32", "bf16"))
        g.append(ParamSpec(f"l{layer}.down", (1024, 4096), "bf16", "f32", "f32", "bf16"))
    return Workload(f"mixed50m_W{W}", W, (tuple(g),), std=1.0, seed=1002)


def kda_block(W: int = 8, reduce: str = "f32", blocks: int = 1, d: int = 4096,
              heads: int = 32, ffn: int = 12288, homogeneous: bool = False) -> Workload:
    """KDA-style transformer blocks, one fully_shard group per block.

    Per block: attn_norm[d] FP32, q/k/v/o [d, d] BF16, decay[heads] FP32,
    gate_vec[d] FP32, mlp_norm[d] FP32, w_gate/w_up [ffn, d] BF16,
    w_down [d, ffn] BF16.  Eight blocks at d=4096 hold 1,744,929,024
    parameters.  ``reduce``: "f32" puts everything in one FP32 bucket, "grad"
    gives each parameter the reduce dtype of its gradient (a BF16 and an FP32
    bucket), "bf16" reduces everything in BF16.  Param dtype: BF16 for the
    matrices, FP32 for the small parameters (``homogeneous``: BF16 for all).
    """
    groups = []
    for blk in range(blocks):
        g = []

        def add(name, shape, dt):
            rd = {"f32": "f32", "bf16": "bf16", "grad": dt}[reduce]
            pd = "bf16" if (dt == "bf16" or homogeneous) else "f32"
            g.append(ParamSpec(f"b{blk}.{name}", shape, dt, rd, "f32", pd))

        add("attn_norm", (d,), "f32")
        for m in ("q", "k", "v", "o"):
            add(m, (d, d), "bf16")
        add("decay", (heads,), "f32")
        add("gate_vec", (d,), "f32")
        add("mlp_norm", (d,), "f32")
        add("w_gate", (ffn, d), "bf16")
        add("w_up", (ffn, d), "bf16")
        add("w_down", (d, ffn), "bf16")
        groups.append(tuple(g))
    return Workload(f"kda_W{W}_reduce-{reduce}" + ("_homogeneous" if homogeneous else ""), W, tuple(groups),
                    std=1.0, seed=1004)


# ---------------------------------------------------------------------------
# Values
# ---------------------------------------------------------------------------
def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng([seed, *key])


def normal_bits(n: int, dtype: str, std: float, seed: int, *key: int) -> np.ndarray:
    """n seeded N(0, std) values as raw bits of ``dtype``."""
    x = _rng(seed, *key).standard_normal(n, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    bits = x.view(np.uint32)
    if dtype == "f32":
        return bits
    return (bits >> np.uint32(16)).astype(np.uint16)


def device_random_bytes(nbytes: int, seed: int, *key: int):
    """``nbytes`` uniformly random bytes on the current CUDA device, drawn by
    torch's seeded Philox generator: read as FP32 or BF16 elements, every bit
    pattern is equally likely (NaNs, infinities and subnormals included) and
    the values never repeat with a period that an offset error could hide
    behind.  For inputs of billions of elements, where host generation would
    take minutes; copy the tensor to the host for the oracle."""
    import torch
    state = np.random.SeedSequence([seed, *key]).generate_state(1, np.uint64)[0]
    g = torch.Generator(device="cuda")
    g.manual_seed(int(state))
    return torch.randint(0, 256, (int(nbytes),), dtype=torch.uint8, device="cuda", generator=g)


def device_normal_bits(n: int, dtype: str, std: float, seed: int, *key: int):
    """n seeded N(0, std) values as raw bits of ``dtype`` on the current CUDA
    device (a uint8 tensor of n * element-size bytes), drawn by torch's
    Philox generator.  BF16 values are the upper halves of FP32 draws, as in
    normal_bits.  For timing inputs too large to draw on the host quickly;
    the values differ from normal_bits' (another generator), the
    distribution does not."""
    import torch
    state = np.random.SeedSequence([seed, *key]).generate_state(1, np.uint64)[0]
    g = torch.Generator(device="cuda")
    g.manual_seed(int(state))
    x = torch.randn(int(n), dtype=torch.float32, device="cuda", generator=g)
    if std != 1.0:
        x *= std
    if dtype == "f32":
        return x.view(torch.uint8)
    return (x.view(torch.int32) >> 16).to(torch.int16).view(torch.uint8)


# Special FP32 bit patterns: signed zeros, infinities, NaNs with payloads,
# subnormals, extremes, and values whose low 16 bits sit exactly on, just
# below and just above a BF16 rounding tie.
F32_SPECIALS = np.array([
    0x00000000, 0x80000000, 0x7F800000, 0xFF800000,
    0x7FC00000, 0xFFC00000, 0x7F800001, 0xFF800001, 0x7FBFFFFF, 0x7FFFFFFF, 0xFFFFFFFF,
    0x7F810000, 0x7FA12345,
    0x00000001, 0x80000001, 0x007FFFFF, 0x807FFFFF, 0x00008000, 0x00018000, 0x0000FFFF,
    0x00800000, 0x80800000, 0x7F7FFFFF, 0xFF7FFFFF, 0x7F7F8000, 0x7F7F7FFF, 0x7F7E8000,
    0x3F808000, 0x3F818000, 0x3F807FFF, 0x3F808001, 0xBF808000, 0xBF818000,
    0x3F800000, 0x3F7FFFFF, 0x00FF8000, 0x00FE8000,
], dtype=np.uint32)

BF16_SPECIALS = np.array([
    0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC0, 0x7F81, 0xFFFF, 0x7FFF,
    0x0001, 0x8001, 0x007F, 0x807F, 0x0080, 0x7F7F, 0xFF7F, 0x3F80, 0xBF80,
], dtype=np.uint16)


def inject_specials(bits: np.ndarray, dtype: str, frac: float, seed: int, *key: int,
                    finite: bool = False) -> np.ndarray:
    """Overwrite a seeded fraction of ``bits`` (in place) with special patterns
    (only the finite ones if ``finite``)."""
    n = bits.size
    if n == 0 or frac <= 0:
        return bits
    rng = _rng(seed, 7777, *key)
    k = max(1, int(n * frac))
    pos = rng.choice(n, size=min(k, n), replace=False)
    pool = F32_SPECIALS if dtype == "f32" else BF16_SPECIALS
    if finite:
        exp_mask = np.uint32(0x7F800000) if dtype == "f32" else np.uint16(0x7F80)
        pool = pool[(pool & exp_mask) != exp_mask]
    bits.reshape(-1)[pos] = pool[rng.integers(0, pool.size, size=pos.size)]
    return bits


def grad_values(wl: Workload, group: int, index: int, specials: float = 0.0) -> np.ndarray:
    """Gradient of parameter ``index`` of group ``group``: flat raw bits."""
    p = wl.groups[group][index]
    bits = normal_bits(p.numel, p.grad_dtype, wl.std, wl.seed, group, index, 1)
    if specials:
        inject_specials(bits, p.grad_dtype, specials, wl.seed, group, index, 1)
    return bits


def param_values(wl: Workload, group: int, index: int) -> np.ndarray:
    """Full parameter in its shard dtype: flat raw bits."""
    p = wl.groups[group][index]
    return normal_bits(p.numel, p.shard_dtype, wl.std, wl.seed, group, index, 2)


def shard_values(wl: Workload, group: int, index: int, rank: int, length: int,
                 n_valid: int, specials: float = 0.0) -> np.ndarray:
    """A local shard of ``length`` elements in the shard dtype.

    The caller says how long the shard is and how many leading elements are
    real (the rest are the padding slots, filled with +0).
    """
    p = wl.groups[group][index]
    bits = normal_bits(length, p.shard_dtype, wl.std, wl.seed, group, index, 3, rank)
    if specials:
        inject_specials(bits, p.shard_dtype, specials, wl.seed, group, index, 3, rank)
    bits[max(0, n_valid):] = 0
    return bits


def random_layout(seed: int, max_params: int = 6, max_numel: int = 300,
                  W_choices=(1, 2, 3, 4, 5, 7, 8, 16, 64)) -> Workload:
    """A seeded random single-group layout: random sizes, dtypes and world size."""
    rnd = random.Random(seed)
    W = rnd.choice(W_choices)
    n = rnd.randint(1, max_params)
    dts = ("f32", "bf16")
    g = []
    for i in range(n):
        r = rnd.random()
        if r < 0.1:
            numel = 0
        elif r < 0.4:
            numel = rnd.randint(1, 17)
        else:
            numel = rnd.randint(1, max_numel)
        g.append(ParamSpec(f"p{i}", (numel,), rnd.choice(dts), rnd.choice(dts),
                           rnd.choice(dts), rnd.choice(dts)))
    return Workload(f"random{seed}", W, (tuple(g),), std=1.0, seed=5000 + seed)


def random_layout_2d(seed: int, max_params: int = 5, max_rows: int = 300, max_row: int = 64,
                     W_choices=(1, 2, 3, 5, 6, 7, 8, 16, 64)) -> Workload:
    """A seeded random single-group layout of 1-D and 2-D parameters, for the
    dim-0 row-chunk rule (world sizes that often do not divide d0)."""
    rnd = random.Random(seed)
    W = rnd.choice(W_choices)
    dts = ("f32", "bf16")
    g = []
    for i in range(rnd.randint(1, max_params)):
        d0 = 0 if rnd.random() < 0.08 else rnd.randint(1, max_rows)
        shape = (d0,) if rnd.random() < 0.25 else (d0, rnd.randint(1, max_row))
        g.append(ParamSpec(f"p{i}", shape, rnd.choice(dts), rnd.choice(dts), rnd.choice(dts), rnd.choice(dts)))
    return Workload(f"random2d{seed}", W, (tuple(g),), std=1.0, seed=7000 + seed)
