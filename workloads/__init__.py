"""Seeded synthetic inputs for paged-KV decode attention.

This module only *generates inputs*: lengths, a fragmented physical pool, block
tables, slot mappings and N(0, 1) values.  It holds none of the attention or
append arithmetic, and both the CUDA library's tests and the oracle draw their
inputs from it.

Shapes follow the pages' Llama-7B (32 layers, hidden 4096, MHA) and Llama-70B
(8 KV heads, head_dim 128, GQA) examples.  Five named workloads:

  c1        tiny: 2 sequences, context {37, 50} + 1 appended token, bs 16,
            4 q / 2 kv heads, d 64, fp16, pool of 16 blocks in seeded
            permutation order, scale 1/8
  c2        Llama-7B layer, MHA: 64 sequences, 32/32 heads, d 128, bs 16,
            context uniform in [512, 4096], fp16, shuffled free list
  c3        Llama-70B layer, GQA-8: 32 sequences, 64/8 heads, d 128, bs 16,
            all context 4096, bf16, randomly permuted pool of 8192 blocks
  c4        long context: 8 sequences, 64/8 heads, d 128, bs 16,
            context uniform in [32768, 131072], bf16, shuffled free list
  c5        continuous-batching mix: 256 sequences, 32/8 heads, d 128, bs 16
            (c5_bs32: bs 32), 4 groups of 64 sequences sharing the physical
            blocks of a 2048-token prefix, context = 2048 + suffix with the
            suffix LogNormal(median 1024, sigma 1.0) rounded, >= 1, total
            <= 16384, bf16, shuffled free list

Lengths are ``context_lens`` *after* the step's append (they include the new
token), so the new token's slot is position ``context_len - 1``.

Random draws: structure (lengths, pool order) comes from a CPU
``torch.Generator`` seeded with the workload's seed; values come from a
generator on the target device seeded from the same seed, drawn in fp32 and
rounded to the 16-bit dtype.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field
from typing import Optional

import torch

TORCH_DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Spec:
    name: str
    seed: int
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str
    # ("fixed", (n0, n1, ...)) | ("uniform", lo, hi) | ("const", n)
    # | ("prefix_lognormal", prefix, median, sigma, cap)
    lengths: tuple
    pool: str = "free_list"          # "free_list" | "permutation"
    pool_blocks: Optional[int] = None  # None: exactly the blocks in use (+ slack)
    pool_slack: float = 0.0          # extra unused blocks, as a fraction of those in use
    shared_prefix_groups: int = 0
    max_len_cap: Optional[int] = None  # block-table width = ceil(cap / block_size)
    scale: Optional[float] = None    # None: 1 / sqrt(head_dim)

    def with_(self, **kw) -> "Spec":
        return dataclasses.replace(self, **kw)


SPECS = {
    "c1": Spec("c1", 1, 2, 4, 2, 64, 16, "fp16", ("fixed", (38, 51)), pool="permutation",
               pool_blocks=16, max_len_cap=64, scale=1.0 / 8.0),
    "c2": Spec("c2", 2, 64, 32, 32, 128, 16, "fp16", ("uniform", 512, 4096), pool_slack=0.05,
               max_len_cap=4096),
    "c3": Spec("c3", 3, 32, 64, 8, 128, 16, "bf16", ("const", 4096), pool="permutation",
               max_len_cap=4096),
    "c4": Spec("c4", 4, 8, 64, 8, 128, 16, "bf16", ("uniform", 32768, 131072), pool_slack=0.02,
               max_len_cap=131072),
    "c5": Spec("c5", 5, 256, 32, 8, 128, 16, "bf16", ("prefix_lognormal", 2048, 1024, 1.0, 16384),
               pool_slack=0.05, shared_prefix_groups=4, max_len_cap=16384),
    "c5_bs32": Spec("c5_bs32", 5, 256, 32, 8, 128, 32, "bf16",
                    ("prefix_lognormal", 2048, 1024, 1.0, 16384), pool_slack=0.05,
                    shared_prefix_groups=4, max_len_cap=16384),
}


@dataclass
class Workload:
    spec: Spec
    scale: float
    num_blocks: int
    context_lens: torch.Tensor      # int32 [B], after the append
    block_tables: torch.Tensor      # int32 [B, max_blocks_per_seq], -1 beyond use
    slot_mapping: torch.Tensor      # int64 [B], slot of each sequence's new token
    q: Optional[torch.Tensor]       # [B, H_q, d]
    k_new: Optional[torch.Tensor]   # [B, H_kv, d]
    v_new: Optional[torch.Tensor]   # [B, H_kv, d]
    k_cache: Optional[torch.Tensor]  # [num_blocks, bs, H_kv, d], state before the append
    v_cache: Optional[torch.Tensor]
    shared_blocks: int = 0          # physical blocks referenced by more than one sequence
    # contiguous groups sharing prefix blocks: group_start int32 [G+1],
    # group_prefix_len int32 [G] (a sequence sharing nothing is a group of one)
    group_start: Optional[torch.Tensor] = None
    group_prefix_len: Optional[torch.Tensor] = None
    extra: dict = field(default_factory=dict)

    @property
    def max_group_size(self) -> int:
        return int((self.group_start[1:] - self.group_start[:-1]).max()) if self.group_start is not None else 1

    @property
    def max_prefix_len(self) -> int:
        return int(self.group_prefix_len.max()) if self.group_prefix_len is not None else 0

    @property
    def torch_dtype(self) -> torch.dtype:
        return TORCH_DTYPES[self.spec.dtype]

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max().item()) if self.context_lens.numel() else 0

    def to(self, device) -> "Workload":
        kw = {}
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            kw[f.name] = v.to(device) if isinstance(v, torch.Tensor) else v
        return Workload(**kw)


def _draw_lengths(spec: Spec, g: torch.Generator) -> torch.Tensor:
    kind = spec.lengths[0]
    b = spec.num_seqs
    if kind == "fixed":
        vals = list(spec.lengths[1])
        if len(vals) != b:
            raise ValueError("fixed lengths must list one length per sequence")
        return torch.tensor(vals, dtype=torch.int64)
    if kind == "const":
        return torch.full((b,), int(spec.lengths[1]), dtype=torch.int64)
    if kind == "uniform":
        lo, hi = int(spec.lengths[1]), int(spec.lengths[2])
        return torch.randint(lo, hi + 1, (b,), generator=g, dtype=torch.int64)
    if kind == "prefix_lognormal":
        prefix, median, sigma, cap = spec.lengths[1:]
        suffix = torch.empty(b, dtype=torch.float64).log_normal_(math.log(median), sigma,
                                                                 generator=g)
        suffix = suffix.round().clamp(1, cap - prefix).to(torch.int64)
        return prefix + suffix
    raise ValueError(f"unknown length kind {kind!r}")


def _values(shape, dtype: torch.dtype, device, gen: torch.Generator) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dtype)


def make_workload(name_or_spec, device="cpu", poison: bool = False, with_values: bool = True,
                  **overrides) -> Workload:
    """Builds a seeded workload (see the module docstring).

    ``poison=True`` fills every cache slot that no sequence's context covers
    (tails of last pages, unused pool blocks, and the new tokens' slots before
    the append) with NaN, so that a reader of masked tokens is caught.
    ``with_values=False`` builds the structure only (the value tensors are None).
    """
    spec = SPECS[name_or_spec] if isinstance(name_or_spec, str) else name_or_spec
    if overrides:
        spec = spec.with_(**overrides)
    g = torch.Generator().manual_seed(spec.seed)
    bs = spec.block_size
    lens = _draw_lengths(spec, g)
    b = spec.num_seqs
    pages = [(int(n) + bs - 1) // bs for n in lens]

    # Physical blocks: shared prefix blocks per group first, then each sequence's own.
    prefix_pages = 0
    groups = spec.shared_prefix_groups
    if groups:
        prefix = int(spec.lengths[1])
        if prefix % bs:
            raise ValueError("shared prefix must be block aligned")
        prefix_pages = prefix // bs
        if b % groups:
            raise ValueError("sequences must split evenly into prefix groups")
    in_use = sum(pages) - (b - groups) * prefix_pages if groups else sum(pages)
    if spec.pool_blocks is not None:
        num_blocks = int(spec.pool_blocks)
    else:
        num_blocks = in_use + int(math.ceil(in_use * spec.pool_slack))
    if num_blocks < in_use:
        raise ValueError("pool too small for the sequences' pages")

    # Free list in seeded order; acquiring pops from the front (PageAllocator order).
    free_list = torch.randperm(num_blocks, generator=g).tolist()
    cursor = 0

    def acquire(count: int) -> list[int]:
        nonlocal cursor
        got = free_list[cursor:cursor + count]
        cursor += count
        return got

    cap = spec.max_len_cap if spec.max_len_cap is not None else int(lens.max())
    width = max(1, (cap + bs - 1) // bs)
    if max(pages) > width:
        raise ValueError("a sequence is longer than the block-table width")
    tables = torch.full((b, width), -1, dtype=torch.int32)
    group_prefix = [acquire(prefix_pages) for _ in range(groups)] if groups else []
    for s in range(b):
        own = pages[s]
        row: list[int] = []
        if groups:
            row = list(group_prefix[s // (b // groups)])
            own -= prefix_pages
        row += acquire(own)
        tables[s, :len(row)] = torch.tensor(row, dtype=torch.int32)

    slot = torch.empty(b, dtype=torch.int64)
    for s in range(b):
        pos = int(lens[s]) - 1
        slot[s] = int(tables[s, pos // bs]) * bs + pos % bs

    tdt = TORCH_DTYPES[spec.dtype]
    dev = torch.device(device)
    scale = spec.scale if spec.scale is not None else 1.0 / math.sqrt(spec.head_dim)
    shared = groups * prefix_pages
    if groups:
        per = b // groups
        gstart = torch.arange(0, b + 1, per, dtype=torch.int32)
        gplen = torch.full((groups,), prefix_pages * bs, dtype=torch.int32)
    else:
        gstart = torch.arange(0, b + 1, dtype=torch.int32)
        gplen = torch.zeros(b, dtype=torch.int32)
    gstart, gplen = gstart.to(dev), gplen.to(dev)
    if not with_values:
        return Workload(spec=spec, scale=scale, num_blocks=num_blocks,
                        context_lens=lens.to(torch.int32).to(dev),
                        block_tables=tables.to(dev), slot_mapping=slot.to(dev), q=None,
                        k_new=None, v_new=None, k_cache=None, v_cache=None,
                        shared_blocks=shared, group_start=gstart, group_prefix_len=gplen)
    vg = torch.Generator(device=dev).manual_seed(spec.seed * 7919 + 17)
    h_kv, h_q, d = spec.num_kv_heads, spec.num_q_heads, spec.head_dim
    q = _values((b, h_q, d), tdt, dev, vg)
    k_new = _values((b, h_kv, d), tdt, dev, vg)
    v_new = _values((b, h_kv, d), tdt, dev, vg)
    k_cache = _values((num_blocks, bs, h_kv, d), tdt, dev, vg)
    v_cache = _values((num_blocks, bs, h_kv, d), tdt, dev, vg)

    if poison:
        covered = torch.zeros(num_blocks * bs, dtype=torch.bool)
        for s in range(b):
            n_prev = int(lens[s]) - 1  # tokens already cached before the append
            t = torch.arange(n_prev)
            blk = tables[s, t // bs].to(torch.int64)
            covered[blk * bs + t % bs] = True
        mask = (~covered).view(num_blocks, bs).to(dev)
        k_cache[mask] = float("nan")
        v_cache[mask] = float("nan")

    return Workload(spec=spec, scale=scale, num_blocks=num_blocks,
                    context_lens=lens.to(torch.int32).to(dev), block_tables=tables.to(dev),
                    slot_mapping=slot.to(dev), q=q, k_new=k_new, v_new=v_new,
                    k_cache=k_cache, v_cache=v_cache, shared_blocks=shared,
                    group_start=gstart, group_prefix_len=gplen)


def to_head_major(cache: torch.Tensor) -> torch.Tensor:
    """The same cache in the head-major page layout: [blocks][bs][H_kv][d] ->
    [blocks][H_kv][bs][d] (a permutation of the values, nothing else)."""
    return cache.permute(0, 2, 1, 3).contiguous()


def make_fp8_codes(shape, seed: int, device="cpu", exponents=(1, 10)) -> torch.Tensor:
    """Seeded E4M3 bit patterns (uint8): random sign, exponent field drawn from
    range(*exponents), any fraction; never NaN.  The default gives normal values
    with |value| in [2^-6, 2^3); exponents=(0, 1) gives only subnormal codes
    (and zeros), |value| = fraction * 2^-9."""
    g = torch.Generator().manual_seed(seed * 7919 + 31)
    sign = torch.randint(0, 2, shape, generator=g, dtype=torch.int32) << 7
    expo = torch.randint(exponents[0], exponents[1], shape, generator=g, dtype=torch.int32) << 3
    frac = torch.randint(0, 8, shape, generator=g, dtype=torch.int32)
    return (sign | expo | frac).to(torch.uint8).to(device)


def make_queries(w: Workload, q_len: int, seed: int) -> torch.Tensor:
    """Seeded N(0,1) queries [B, q_len, H_q, d] in the workload's dtype and device
    (several new query tokens per sequence: a prefill chunk or drafted tokens)."""
    s = w.spec
    dev = w.context_lens.device
    g = torch.Generator(device=dev).manual_seed(seed * 7919 + 29)
    return _values((s.num_seqs, q_len, s.num_q_heads, s.head_dim), TORCH_DTYPES[s.dtype], dev, g)


def make_append_case(num_tokens: int, num_blocks: int, block_size: int, num_kv_heads: int,
                     head_dim: int, dtype: str, seed: int, pad_fraction: float = 0.25,
                     device="cpu") -> dict:
    """Random append inputs: distinct slots scattered over the pool, some padded (-1).

    The cache is filled with a sentinel bit pattern (0x7E5A) so untouched bytes
    can be checked afterwards.
    """
    g = torch.Generator().manual_seed(seed)
    total = num_blocks * block_size
    if num_tokens > total:
        raise ValueError("more tokens than slots")
    slots = torch.randperm(total, generator=g)[:num_tokens].to(torch.int64)
    pad = torch.rand(num_tokens, generator=g) < pad_fraction
    slots[pad] = -1
    tdt = TORCH_DTYPES[dtype]
    dev = torch.device(device)
    vg = torch.Generator(device=dev).manual_seed(seed * 7919 + 23)
    k_new = _values((num_tokens, num_kv_heads, head_dim), tdt, dev, vg)
    v_new = _values((num_tokens, num_kv_heads, head_dim), tdt, dev, vg)
    shape = (num_blocks, block_size, num_kv_heads, head_dim)
    k_cache = torch.full(shape, 0x7E5A, dtype=torch.int16, device=dev).view(tdt)
    v_cache = torch.full(shape, 0x7E5A, dtype=torch.int16, device=dev).view(tdt)
    return dict(k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache,
                slot_mapping=slots.to(dev))


def bits(t: torch.Tensor):
    """Raw uint16 bit patterns of a 16-bit tensor, as a numpy array on the host."""
    import numpy as np
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
