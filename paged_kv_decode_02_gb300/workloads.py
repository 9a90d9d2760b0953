"""Seeded synthetic inputs and the host-side block allocator.

This module only draws random numbers and builds block tables; it holds none of the
attention, scatter or quantisation arithmetic. Both the CUDA path (through the tests
and the benchmark) and the CPU oracle are fed from it.

The block allocator follows the block-manager description in "大模型工程（五）：推理
优化核心技法" (chenk.top), section "块管理器：分页如何运作": a pool of physical blocks,
a free list, blocks appended to a request's table as it grows, and refcounted blocks
under copy-on-write (fork adds a reference, free drops one, the block returns to the
pool at zero). Prefix sharing ("分页注意力", same page; section 2.2 of the gsyq.cn page)
is several tables pointing at the same physical blocks.

Workload recipes (names are the shapes they model):

* ``tiny``: batch 4, 8 q heads = 8 KV heads, head_dim 64, block 16, context lengths
  uniform in [1, 64], blocks drawn from a randomly permuted 64-block pool, q/K/V
  bf16 ~ N(0, 1), scale 1/8, seed 0.
* ``7b``: the 7B layer of section 2.1 of the gsyq.cn page: batch 32, 32/32 heads,
  head_dim 128, context 2048 for every request, block 16, pool 1.2x demand, shuffled,
  seed 1.
* ``70b-gqa``: batch 64, 64 q / 8 KV heads, head_dim 128, block 16, context lengths
  log-normal (median 1024, natural-log sigma 1.0) rounded and clipped to
  [128, 32768], pool 1.2x demand, seed 2.
* ``prefix``: batch 256, 32 q / 8 KV heads, head_dim 128, block 16, one shared
  2048-token prefix (128 blocks, refcount 256) plus a private suffix of uniform
  [16, 512] tokens per request, pool 1.2x demand, seed 3.
* ``int8``: batch 128, 32 q / 8 KV heads, head_dim 128, context 8192, block 32
  (``int8-bs16``: block 16), INT8 K/V codes with one fp32 scale per (token, KV head),
  q bf16, seed 4. The codes are drawn directly as rounded N(0, 42.3^2) values clipped
  to [-127, 127] and the scales uniformly from [2.5, 3.5] / 127, the shape that
  symmetric absmax quantisation of N(0, 1) rows with 128 channels produces.
* ``fp8-e5m2`` / ``fp8-e4m3``: the ``int8`` shape with an FP8 cache (the formats of
  "FP8（及 H100/H200 硬件路径）", chenk.top page; E5M2 is the one it names for KV
  caches): codes are N(0, (FP8_MAX/3)^2) values clipped to +-FP8_MAX and rounded to
  the format by PyTorch's float8 cast (FP8_MAX = 57344 or 448), scales uniformly from
  [2.5, 3.5] / FP8_MAX -- again the shape absmax scaling of N(0, 1) rows produces.

* ``spec-70b``: the ``70b-gqa`` shape and lengths with q_len = 6 new tokens per
  request (k = 5 drafted tokens plus the next position, the number of speculative
  tokens in the vLLM example of "推测解码", chenk.top page), for multi-query decode.
  ``spec-70b-q16``: the same with q_len = 16 (128 query rows per KV head).
* ``prefix-int8`` / ``prefix-e5m2`` and ``spec-70b-int8`` / ``spec-70b-e4m3``: the
  ``prefix`` and ``spec-70b`` shapes and lengths over one-byte caches, codes and scales
  drawn as for ``int8`` / ``fp8-*``.
* ``chunk-70b``: a chunk of chunked prefill ("Orca 的迭代级调度", chenk.top page) on the
  ``70b-gqa`` shape: 16 requests whose last 256 tokens are the chunk being prefilled
  (q_len = 256, 2048 query rows per KV head), lengths log-normal (median 1024, sigma 1)
  rounded and clipped to [256, 32768], seed 5.

The tokens appended in the step are the last q_len (1 unless stated) of each
request: ``new_k``/``new_v`` hold them ([B * q_len, Hkv, D], request-major) and
``slot_mapping`` points at their slots (``-1`` for an empty request).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch


class BlockAllocator:
    """Refcounted pool of physical KV blocks with a (shuffled) free list."""

    def __init__(self, num_blocks: int, rng: Optional[np.random.Generator] = None):
        if num_blocks <= 0:
            raise ValueError("num_blocks must be positive")
        self.num_blocks = int(num_blocks)
        order = rng.permutation(self.num_blocks) if rng is not None else np.arange(self.num_blocks)
        # pop() takes from the end: reverse so the first draw is order[0]
        self._free = [int(b) for b in order[::-1]]
        self.refcount = np.zeros(self.num_blocks, dtype=np.int64)

    @property
    def num_free(self) -> int:
        return len(self._free)

    def allocate(self) -> int:
        if not self._free:
            raise MemoryError("KV block pool exhausted")
        b = self._free.pop()
        self.refcount[b] = 1
        return b

    def fork(self, block: int) -> int:
        """Share ``block`` with one more request (copy-on-write reference)."""
        if self.refcount[block] <= 0:
            raise ValueError(f"fork of free block {block}")
        self.refcount[block] += 1
        return block

    def free(self, block: int) -> None:
        """Drop one reference; the block goes back to the pool when none remain."""
        if self.refcount[block] <= 0:
            raise ValueError(f"double free of block {block}")
        self.refcount[block] -= 1
        if self.refcount[block] == 0:
            self._free.append(int(block))


class SequenceBlocks:
    """One request's block table: logical block j -> physical block ``blocks[j]``."""

    def __init__(self, allocator: BlockAllocator, block_size: int):
        self.alloc = allocator
        self.block_size = int(block_size)
        self.blocks: list[int] = []
        self.num_tokens = 0

    def fork_prefix(self, other: "SequenceBlocks", num_tokens: int) -> None:
        """Share the first ``num_tokens`` tokens of ``other`` (whole blocks only)."""
        if num_tokens % self.block_size != 0:
            raise ValueError("a shared prefix must end on a block boundary")
        n = num_tokens // self.block_size
        self.blocks = [self.alloc.fork(b) for b in other.blocks[:n]]
        self.num_tokens = num_tokens

    def fork_all(self, other: "SequenceBlocks") -> None:
        """Share every block of ``other``, a partly filled last block included (a fork
        for parallel sampling or beam search)."""
        self.blocks = [self.alloc.fork(b) for b in other.blocks]
        self.num_tokens = other.num_tokens

    def append_tokens(self, n: int, copies: Optional[list] = None) -> list[int]:
        """Grow by ``n`` tokens, taking a fresh block whenever the last one is full.
        Writing into a partly filled last block that another request still shares
        first moves this request to a private copy (copy-on-write): a fresh block is
        allocated, the pair (shared, fresh) is appended to ``copies`` for the device
        block copy, and the shared block loses this request's reference.
        Returns each new token's slot (physical block * block_size + offset)."""
        slots = []
        for _ in range(n):
            off = self.num_tokens % self.block_size
            if off == 0:
                self.blocks.append(self.alloc.allocate())
            elif self.alloc.refcount[self.blocks[-1]] > 1:
                if copies is None:
                    raise ValueError("a write into a shared block needs a copy list")
                fresh = self.alloc.allocate()
                copies.append((self.blocks[-1], fresh))
                self.alloc.free(self.blocks[-1])
                self.blocks[-1] = fresh
            slots.append(self.blocks[-1] * self.block_size + off)
            self.num_tokens += 1
        return slots

    def swap_out(self) -> list[int]:
        """Evict: return the blocks to copy to host memory (in table order) and drop
        this request's references to them."""
        ids = list(self.blocks)
        for b in ids:
            self.alloc.free(b)
        self.blocks = []
        return ids

    def swap_in(self, num_blocks: int) -> list[int]:
        """Bring an evicted request back: allocate ``num_blocks`` fresh blocks (its new
        table) for the copy from host memory."""
        self.blocks = [self.alloc.allocate() for _ in range(num_blocks)]
        return list(self.blocks)

    def release(self) -> None:
        for b in self.blocks:
            self.alloc.free(b)
        self.blocks = []
        self.num_tokens = 0


@dataclass
class Workload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    kv_dtype: str                      # "bf16", "int8", "fp8_e4m3" or "fp8_e5m2"
    scale: float
    q: torch.Tensor                    # [B, Hq, D] bf16 ([B, q_len, Hq, D] when q_len > 1)
    k_cache: torch.Tensor              # [NB, Hkv, bs, D] bf16, int8 or uint8 (FP8 codes)
    v_cache: torch.Tensor
    block_tables: torch.Tensor         # [B, MBS] int32 (entries past a request's blocks are poison)
    context_lens: torch.Tensor         # [B] int32
    new_k: torch.Tensor                # [B * q_len, Hkv, D] bf16: tokens appended this step
    new_v: torch.Tensor
    slot_mapping: torch.Tensor         # [B * q_len] int64
    k_scale: Optional[torch.Tensor] = None   # [NB, Hkv, bs] fp32 (one-byte caches only)
    v_scale: Optional[torch.Tensor] = None
    refcount: Optional[np.ndarray] = None
    extra: dict = field(default_factory=dict)
    q_len: int = 1                     # new tokens per request (multi-query decode)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def total_tokens(self) -> int:
        return int(self.context_lens.to(torch.int64).sum().item())


def _lognormal_lengths(rng, n, median, sigma, lo, hi):
    x = rng.lognormal(mean=math.log(median), sigma=sigma, size=n)
    return np.clip(np.rint(x), lo, hi).astype(np.int64)


SPECS = {
    "tiny":      dict(B=4,   Hq=8,  Hkv=8,  D=64,  bs=16, seed=0),
    "7b":        dict(B=32,  Hq=32, Hkv=32, D=128, bs=16, seed=1),
    "70b-gqa":   dict(B=64,  Hq=64, Hkv=8,  D=128, bs=16, seed=2),
    "prefix":    dict(B=256, Hq=32, Hkv=8,  D=128, bs=16, seed=3),
    "int8":      dict(B=128, Hq=32, Hkv=8,  D=128, bs=32, seed=4),
    "int8-bs16": dict(B=128, Hq=32, Hkv=8,  D=128, bs=16, seed=4),
    "fp8-e5m2":  dict(B=128, Hq=32, Hkv=8,  D=128, bs=32, seed=4),
    "fp8-e4m3":  dict(B=128, Hq=32, Hkv=8,  D=128, bs=32, seed=4),
    "spec-70b":  dict(B=64,  Hq=64, Hkv=8,  D=128, bs=16, seed=2, q_len=6),
    "spec-70b-q16": dict(B=64, Hq=64, Hkv=8, D=128, bs=16, seed=2, q_len=16),
    "chunk-70b": dict(B=16, Hq=64, Hkv=8, D=128, bs=16, seed=5, q_len=256),
    # one-byte caches under the same shapes (codes and scales drawn as for int8 / fp8-*)
    "prefix-int8": dict(B=256, Hq=32, Hkv=8, D=128, bs=16, seed=3),
    "prefix-e5m2": dict(B=256, Hq=32, Hkv=8, D=128, bs=16, seed=3),
    "spec-70b-int8": dict(B=64, Hq=64, Hkv=8, D=128, bs=16, seed=2, q_len=6),
    "spec-70b-e4m3": dict(B=64, Hq=64, Hkv=8, D=128, bs=16, seed=2, q_len=6),
}

FP8_KV = {"fp8_e4m3": (torch.float8_e4m3fn, 448.0), "fp8_e5m2": (torch.float8_e5m2, 57344.0)}


def _draw_lengths(name, rng, B):
    if name == "tiny":
        return rng.integers(1, 65, size=B).astype(np.int64)
    if name == "7b":
        return np.full(B, 2048, dtype=np.int64)
    if name in ("70b-gqa", "spec-70b", "spec-70b-q16", "spec-70b-int8", "spec-70b-e4m3"):
        return _lognormal_lengths(rng, B, 1024, 1.0, 128, 32768)
    if name == "chunk-70b":
        return _lognormal_lengths(rng, B, 1024, 1.0, 256, 32768)
    if name in ("prefix", "prefix-int8", "prefix-e5m2"):
        return 2048 + rng.integers(16, 513, size=B).astype(np.int64)
    if name.startswith("int8") or name.startswith("fp8"):
        return np.full(B, 8192, dtype=np.int64)
    raise KeyError(name)


def build_tables(lengths, block_size, rng, pool_factor=1.2, num_blocks=None,
                 shared_prefix_tokens=0, poison_pad=7):
    """Allocate blocks for every request and return (tables [B, MBS] int32, slots
    of each request's last token [B] int64, num_blocks, allocator).

    ``shared_prefix_tokens`` > 0 puts that many leading tokens of every request in one
    set of refcounted blocks. Table entries past a request's blocks hold
    ``num_blocks + poison_pad`` (an id no kernel may read).
    """
    lengths = np.asarray(lengths, dtype=np.int64)
    B = len(lengths)
    nblk = [-(-int(L) // block_size) for L in lengths]
    if shared_prefix_tokens:
        pre = shared_prefix_tokens // block_size
        demand = pre + sum(max(n - pre, 0) for n in nblk)
    else:
        demand = sum(nblk)
    if num_blocks is None:
        num_blocks = max(int(math.ceil(pool_factor * demand)), 1)
    alloc = BlockAllocator(num_blocks, rng)
    seqs = []
    proto = None
    if shared_prefix_tokens:
        proto = SequenceBlocks(alloc, block_size)
        proto.append_tokens(shared_prefix_tokens)
    last_slots = np.full(B, -1, dtype=np.int64)
    for s in range(B):
        sb = SequenceBlocks(alloc, block_size)
        L = int(lengths[s])
        if proto is not None and L >= shared_prefix_tokens:
            sb.fork_prefix(proto, shared_prefix_tokens)
        slots = sb.append_tokens(L - sb.num_tokens)
        if L > 0:
            last_slots[s] = slots[-1] if slots else -1
        seqs.append(sb)
    if proto is not None:
        proto.release()   # the prototype's own reference; requests keep theirs
    mbs = max(max((len(sb.blocks) for sb in seqs), default=0), 1)
    tables = np.full((B, mbs), num_blocks + poison_pad, dtype=np.int32)
    for s, sb in enumerate(seqs):
        tables[s, :len(sb.blocks)] = sb.blocks
    return tables, last_slots, num_blocks, alloc


def _randn_bf16(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_workload(name: str, device="cpu", seed: Optional[int] = None,
                  lengths=None, num_seqs=None, num_q_heads=None, num_kv_heads=None,
                  head_dim=None, block_size=None, num_blocks=None,
                  poison_unused=False, kv_dtype=None, prefix_tokens=None,
                  q_len=None) -> Workload:
    """Build a named workload (optionally overriding its sizes) on ``device``.

    ``poison_unused`` fills every cache row that no request's context covers with NaN
    (bf16) or, for INT8, NaN scales, so that a kernel reading one shows up.
    ``prefix_tokens`` (a multiple of the block size) puts that many leading tokens of
    every request in one set of shared, refcounted blocks (2048 for ``prefix``).
    ``q_len`` > 1 gives every request that many new tokens (q [B, q_len, Hq, D]); a
    request's length must then be 0 or at least q_len.
    """
    spec = dict(SPECS[name])
    seed = spec["seed"] if seed is None else seed
    B = num_seqs or spec["B"]
    Hq = num_q_heads or spec["Hq"]
    Hkv = num_kv_heads or spec["Hkv"]
    D = head_dim or spec["D"]
    bs = block_size or spec["bs"]
    n_new = int(q_len if q_len is not None else spec.get("q_len", 1))
    kvt = kv_dtype or ("int8" if name.startswith("int8") or name.endswith("-int8") else
                       "fp8_" + name[4:] if name.startswith("fp8-") else
                       "fp8_" + name[-4:] if name.endswith(("-e4m3", "-e5m2")) else "bf16")
    rng = np.random.default_rng(seed)
    if lengths is None:
        lengths = _draw_lengths(name, rng, B)
    lengths = np.asarray(lengths, dtype=np.int64)
    B = len(lengths)
    if name == "tiny" and num_blocks is None:
        num_blocks = 64
    prefix = (2048 if name.startswith("prefix") else 0) if prefix_tokens is None \
        else int(prefix_tokens)
    tables, last_slots, NB, alloc = build_tables(lengths, bs, rng, num_blocks=num_blocks,
                                                 shared_prefix_tokens=prefix)
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(seed))
    q = _randn_bf16((B, Hq, D) if n_new == 1 else (B, n_new, Hq, D), gen, dev)
    new_k = _randn_bf16((B * n_new, Hkv, D), gen, dev)
    new_v = _randn_bf16((B * n_new, Hkv, D), gen, dev)
    if n_new > 1:
        if np.any((lengths > 0) & (lengths < n_new)):
            raise ValueError("a request holds fewer tokens than its new tokens")
        last_slots = np.full(B * n_new, -1, dtype=np.int64)
        for s in range(B):
            L = int(lengths[s])
            for i in range(n_new if L else 0):
                t = L - n_new + i
                last_slots[s * n_new + i] = int(tables[s, t // bs]) * bs + t % bs
    k_scale = v_scale = None
    if kvt == "bf16":
        k_cache = _randn_bf16((NB, Hkv, bs, D), gen, dev)
        v_cache = _randn_bf16((NB, Hkv, bs, D), gen, dev)
    elif kvt == "int8":
        def codes():
            x = torch.randn((NB, Hkv, bs, D), generator=gen, device=dev) * (127.0 / 3.0)
            return torch.clamp(torch.round(x), -127, 127).to(torch.int8)
        k_cache, v_cache = codes(), codes()
        k_scale = ((2.5 + torch.rand((NB, Hkv, bs), generator=gen, device=dev)) / 127.0).float()
        v_scale = ((2.5 + torch.rand((NB, Hkv, bs), generator=gen, device=dev)) / 127.0).float()
    elif kvt in FP8_KV:
        f8, fmax = FP8_KV[kvt]

        def codes():
            x = torch.randn((NB, Hkv, bs, D), generator=gen, device=dev) * (fmax / 3.0)
            return torch.clamp(x, -fmax, fmax).to(f8).view(torch.uint8)
        k_cache, v_cache = codes(), codes()
        k_scale = ((2.5 + torch.rand((NB, Hkv, bs), generator=gen, device=dev)) / fmax).float()
        v_scale = ((2.5 + torch.rand((NB, Hkv, bs), generator=gen, device=dev)) / fmax).float()
    else:
        raise ValueError(f"unknown kv dtype {kvt}")
    if poison_unused:
        used = np.zeros((NB, bs), dtype=bool)
        for s in range(B):
            L = int(lengths[s])
            for t in range(L):
                used[tables[s, t // bs], t % bs] = True
        unused = torch.from_numpy(~used).to(dev)            # [NB, bs]
        mask = unused[:, None, :].expand(NB, Hkv, bs)
        if kvt == "bf16":
            k_cache[mask] = float("nan")
            v_cache[mask] = float("nan")
        else:
            k_scale[mask] = float("nan")
            v_scale[mask] = float("nan")
    return Workload(
        name=name, num_seqs=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=bs,
        num_blocks=NB, max_blocks_per_seq=tables.shape[1], kv_dtype=kvt,
        scale=1.0 / math.sqrt(D), q=q, k_cache=k_cache, v_cache=v_cache,
        block_tables=torch.from_numpy(tables).to(dev),
        context_lens=torch.from_numpy(lengths.astype(np.int32)).to(dev),
        new_k=new_k, new_v=new_v, slot_mapping=torch.from_numpy(last_slots).to(dev),
        k_scale=k_scale, v_scale=v_scale, refcount=alloc.refcount.copy(),
        extra={"prefix_tokens": prefix}, q_len=n_new)


def host_units(w: Workload, pairs) -> list:
    """Host copies of (sequence, KV head) units of a workload, in the form the CPU
    oracle's process pool takes: each unit holds its sequence's blocks of that KV head
    re-indexed 0..n-1 (bf16 rows as their 16-bit patterns, one-byte codes and their
    scales as stored), the KV head's q rows as float64 [q_len, g, D], the context
    length, and its byte and token counts for throughput accounting (valid KV rows,
    scales, q and out rows, table entries). Only copies: no arithmetic of the method."""
    g = w.group
    bs = w.block_size
    one_byte = w.kv_dtype != "bf16"
    elt = 1 if one_byte else 2
    L_all = w.context_lens.cpu().numpy()
    q = w.q if w.q_len > 1 else w.q[:, None]          # [B, q_len, Hq, D]
    by_seq: dict = {}
    for s, kvh in pairs:
        by_seq.setdefault(int(s), []).append(int(kvh))
    units = {}
    for s, kvhs in by_seq.items():
        L = int(L_all[s])
        n = -(-L // bs)
        blocks = w.block_tables[s, :n].to(torch.int64)
        kc, vc = w.k_cache[blocks], w.v_cache[blocks]
        if not one_byte:
            kc, vc = kc.view(torch.int16), vc.view(torch.int16)
        kc, vc = kc.cpu().numpy(), vc.cpu().numpy()
        if not one_byte:
            kc, vc = kc.view(np.uint16), vc.view(np.uint16)
        if one_byte:
            ks, vs = w.k_scale[blocks].cpu().numpy(), w.v_scale[blocks].cpu().numpy()
        qs = q[s].to(torch.float64).cpu().numpy()    # [q_len, Hq, D]
        for kvh in kvhs:
            u = {"kind": w.kv_dtype, "bs": bs, "L": L, "table": np.arange(n),
                 "k": np.ascontiguousarray(kc[:, kvh:kvh + 1]),
                 "v": np.ascontiguousarray(vc[:, kvh:kvh + 1]),
                 "q": np.ascontiguousarray(qs[:, kvh * g:(kvh + 1) * g]),
                 "scale": float(w.scale), "tokens": L,
                 "bytes": (L * 2 * w.head_dim * elt + (L * 2 * 4 if one_byte else 0) +
                           2 * w.q_len * g * w.head_dim * 2 + 4 * n)}
            if one_byte:
                u["ks"] = np.ascontiguousarray(ks[:, kvh:kvh + 1])
                u["vs"] = np.ascontiguousarray(vs[:, kvh:kvh + 1])
            units[(s, kvh)] = u
    return [units[(int(s), int(kvh))] for s, kvh in pairs]
