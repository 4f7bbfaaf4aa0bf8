"""Seeded synthetic inputs for the attention-sublayer hot path.

This package is shared by the tests, ``bench.py`` and ``__graft_entry__``.
It draws random numbers and lays out the paged cache the way the pages'
scheduler would (block tables, slot numbers, cu_seqlens); it performs none of
the method's arithmetic (no norm, no rotation, no softmax).  Both the CUDA
path and the oracle consume what it produces; neither is imported here.

Workloads follow the shapes of Qwen3-0.6B (hidden 1024, 16 q / 8 kv heads)
and Qwen3-8B (hidden 4096, 32 q / 8 kv heads), head_dim 128, 256-token
blocks, rms eps 1e-6, RoPE base 1e6 ("同一个 Qwen3，两种写法", sec. 2;
"nano-vllm code walkthrough", Block and BlockManager).  Value distributions:
activations, q/k/v and cached K/V ~ N(0, 1); norm weights ~ 1 + N(0, 0.1).

Random streams: every named tensor of a workload draws from its own
``SeedSequence(seed, spawn_key=(crc32(name),))`` so that drawing a subset (for
example only the cache blocks a test reads) never shifts another tensor.
Large tensors are drawn in fixed 4 Mi-element chunks, chunk i from child i of
that stream, so results do not depend on the thread count.
"""
from __future__ import annotations

import math
import os
import zlib
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 256
HEAD_DIM = 128
RMS_EPS = 1e-6
ROPE_BASE = 1e6
MAX_POSITION = 40960

_CHUNK = 1 << 22


# ---------------------------------------------------------------- bf16 bits
def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round-to-nearest-even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    return ((u + (((u >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _stream(seed: int, name: str) -> np.random.SeedSequence:
    return np.random.SeedSequence(seed, spawn_key=(zlib.crc32(name.encode()),))


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def normal_bf16(seed: int, name: str, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """N(mean, std^2) samples rounded to bf16, as uint16 bits of `shape`."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16)
    n_chunks = max(1, math.ceil(n / _CHUNK))
    children = _stream(seed, name).spawn(n_chunks)

    def work(i):
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        g = np.random.Generator(np.random.PCG64(children[i]))
        a = g.standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            a *= np.float32(std)
        if mean != 0.0:
            a += np.float32(mean)
        out[lo:hi] = f32_to_bf16_bits(a)

    if n_chunks == 1:
        work(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(n_chunks)))
    return out.reshape(shape)


def rng(seed: int, name: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(_stream(seed, name)))


# ------------------------------------------------------------ paged layout
def cu_seqlens(lengths) -> np.ndarray:
    """[0, l0, l0+l1, ...] as int32 (the packed-varlen boundary table)."""
    out = np.zeros(len(lengths) + 1, dtype=np.int32)
    np.cumsum(np.asarray(lengths, dtype=np.int64), out=out[1:])
    return out


def carve_block_tables(perm: np.ndarray, capacity_tokens, block_size: int = BLOCK_SIZE):
    """Hand each sequence ceil(capacity/block_size) distinct blocks, taken in
    order from one permutation of the pool; pad rows with -1."""
    need = [max(1, math.ceil(int(c) / block_size)) for c in capacity_tokens]
    mb = max(need) if need else 1
    if sum(need) > perm.size:
        raise ValueError("pool too small for the requested contexts")
    bt = np.full((len(need), mb), -1, dtype=np.int32)
    off = 0
    for b, k in enumerate(need):
        bt[b, :k] = perm[off:off + k]
        off += k
    return bt


def slots_for_positions(block_tables: np.ndarray, seq_ids, positions,
                        block_size: int = BLOCK_SIZE) -> np.ndarray:
    """slot = physical_block * block_size + offset for each (seq, position)."""
    seq_ids = np.asarray(seq_ids, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    blk = block_tables[seq_ids, positions // block_size].astype(np.int64)
    return (blk * block_size + positions % block_size).astype(np.int32)


@dataclass
class PagedPool:
    """K/V pool [num_blocks, block_size, Hkv, d] as bf16 bits.  Only the blocks
    listed in `used` hold N(0,1) data; the others are zero and never read."""
    num_blocks: int
    hkv: int
    k: np.ndarray
    v: np.ndarray
    used: np.ndarray


def make_pool(seed: int, num_blocks: int, used_blocks, hkv: int, d: int = HEAD_DIM,
              block_size: int = BLOCK_SIZE, k_outlier_frac: float = 0.0,
              k_outlier_scale: float = 8.0) -> PagedPool:
    used = np.unique(np.asarray(used_blocks, dtype=np.int64))
    k = np.zeros((num_blocks, block_size, hkv, d), dtype=np.uint16)
    v = np.zeros_like(k)
    shape = (used.size, block_size, hkv, d)
    kd = normal_bf16(seed, "pool.k", shape)
    vd = normal_bf16(seed, "pool.v", shape)
    if k_outlier_frac > 0.0:
        # Scale whole token rows (all Hkv*d elements of a slot) of K.
        g = rng(seed, "pool.k.outliers")
        hit = g.random((used.size, block_size)) < k_outlier_frac
        rows = kd[hit]
        kd[hit] = f32_to_bf16_bits(bf16_bits_to_f32(rows) * np.float32(k_outlier_scale))
    k[used] = kd
    v[used] = vd
    return PagedPool(num_blocks=num_blocks, hkv=hkv, k=k, v=v, used=used)


# -------------------------------------------------------------- workloads
@dataclass
class Shape:
    hidden: int
    hq: int
    hkv: int
    d: int = HEAD_DIM

    @property
    def q_size(self):
        return self.hq * self.d

    @property
    def kv_size(self):
        return self.hkv * self.d

    @property
    def qkv_width(self):
        return self.q_size + 2 * self.kv_size


QWEN3_06B = Shape(hidden=1024, hq=16, hkv=8)
QWEN3_8B = Shape(hidden=4096, hq=32, hkv=8)


@dataclass
class DecodeStep:
    """One decode step of B sequences: every sequence appends one token at
    position ctx-1 and attends over ctx cached tokens (ctx counts the new
    token, which is written before attention)."""
    shape: Shape
    context_lens: np.ndarray     # [B] int32, includes the new token
    positions: np.ndarray        # [B] int64 = context_lens - 1
    block_tables: np.ndarray     # [B, MB] int32
    slot_mapping: np.ndarray     # [B] int32, slot of the new token
    pool: PagedPool
    qkv: np.ndarray              # [B, Q + 2D] bf16 bits (new token's projections)
    x: np.ndarray | None = None  # [B, hidden] bf16 bits (add-RMSNorm input)
    residual: np.ndarray | None = None
    gamma: np.ndarray | None = None
    q_norm_w: np.ndarray | None = None
    k_norm_w: np.ndarray | None = None
    with_norms: bool = False
    name: str = ""


@dataclass
class PrefillBatch:
    """A packed varlen prefill: sequences of `lengths` tokens at positions
    0..len-1, all K/V rows scattered into freshly allocated blocks."""
    shape: Shape
    lengths: np.ndarray          # [B] int64
    cu_seqlens: np.ndarray       # [B+1] int32
    positions: np.ndarray        # [T] int64
    block_tables: np.ndarray     # [B, MB] int32
    slot_mapping: np.ndarray     # [T] int32
    num_blocks: int
    qkv: np.ndarray              # [T, Q + 2D] bf16 bits
    x: np.ndarray                # [T, hidden]
    residual: np.ndarray         # [T, hidden]
    gamma: np.ndarray            # [hidden]
    q_norm_w: np.ndarray         # [d]
    k_norm_w: np.ndarray         # [d]
    name: str = ""
    extra: dict = field(default_factory=dict)


def _norm_weights(seed, shape: Shape, prefix: str):
    return (normal_bf16(seed, prefix + ".gamma", (shape.hidden,), 1.0, 0.1),
            normal_bf16(seed, prefix + ".q_norm", (shape.d,), 1.0, 0.1),
            normal_bf16(seed, prefix + ".k_norm", (shape.d,), 1.0, 0.1))


def make_prefill(seed: int, shape: Shape, lengths, num_blocks: int | None = None,
                 extra_capacity: int = 0, name: str = "prefill") -> PrefillBatch:
    """Prefill batch; each sequence gets blocks for len + extra_capacity tokens
    (room for later decode steps)."""
    lengths = np.asarray(lengths, dtype=np.int64)
    T = int(lengths.sum())
    need = [math.ceil((int(l) + extra_capacity) / BLOCK_SIZE) for l in lengths]
    nb = num_blocks if num_blocks is not None else max(1, sum(need))
    perm = rng(seed, name + ".perm").permutation(nb).astype(np.int32)
    bt = carve_block_tables(perm, [int(l) + extra_capacity for l in lengths])
    seq_ids = np.repeat(np.arange(lengths.size), lengths)
    positions = np.concatenate([np.arange(l, dtype=np.int64) for l in lengths]) if T else \
        np.zeros(0, np.int64)
    slots = slots_for_positions(bt, seq_ids, positions) if T else np.zeros(0, np.int32)
    gamma, qn, kn = _norm_weights(seed, shape, name)
    return PrefillBatch(
        shape=shape, lengths=lengths, cu_seqlens=cu_seqlens(lengths), positions=positions,
        block_tables=bt, slot_mapping=slots, num_blocks=nb,
        qkv=normal_bf16(seed, name + ".qkv", (T, shape.qkv_width)),
        x=normal_bf16(seed, name + ".x", (T, shape.hidden)),
        residual=normal_bf16(seed, name + ".residual", (T, shape.hidden)),
        gamma=gamma, q_norm_w=qn, k_norm_w=kn, name=name)


def make_decode(seed: int, shape: Shape, context_lens, num_blocks: int,
                with_norms: bool, k_outlier_frac: float = 0.0,
                name: str = "decode") -> DecodeStep:
    ctx = np.asarray(context_lens, dtype=np.int32)
    perm = rng(seed, name + ".perm").permutation(num_blocks).astype(np.int32)
    bt = carve_block_tables(perm, ctx)
    used = bt[bt >= 0]
    pool = make_pool(seed, num_blocks, used, shape.hkv, k_outlier_frac=k_outlier_frac)
    B = ctx.size
    positions = ctx.astype(np.int64) - 1
    slots = slots_for_positions(bt, np.arange(B), np.maximum(positions, 0))
    slots[ctx <= 0] = -1
    step = DecodeStep(shape=shape, context_lens=ctx, positions=np.maximum(positions, 0),
                      block_tables=bt, slot_mapping=slots, pool=pool,
                      qkv=normal_bf16(seed, name + ".qkv", (B, shape.qkv_width)),
                      with_norms=with_norms, name=name)
    if with_norms:
        step.x = normal_bf16(seed, name + ".x", (B, shape.hidden))
        step.residual = normal_bf16(seed, name + ".residual", (B, shape.hidden))
        step.gamma, step.q_norm_w, step.k_norm_w = _norm_weights(seed, shape, name)
    return step


# ------------------------------------------------- the five named workloads
def config1(seed: int = 1001):
    """Tiny Qwen3-0.6B-shaped layer: prefill of 37 and 300 tokens into a pool
    of 8 permuted blocks, then 8 decode steps per sequence."""
    shape = QWEN3_06B
    lengths = np.array([37, 300], dtype=np.int64)
    n_steps = 8
    pre = make_prefill(seed, shape, lengths, num_blocks=8, extra_capacity=n_steps,
                       name="cfg1.prefill")
    steps = []
    for s in range(n_steps):
        B = lengths.size
        pos = lengths + s
        ctx = (pos + 1).astype(np.int32)
        slots = slots_for_positions(pre.block_tables, np.arange(B), pos)
        steps.append(dict(
            positions=pos.astype(np.int64), context_lens=ctx, slot_mapping=slots,
            qkv=normal_bf16(seed, f"cfg1.step{s}.qkv", (B, shape.qkv_width)),
            x=normal_bf16(seed, f"cfg1.step{s}.x", (B, shape.hidden)),
            residual=normal_bf16(seed, f"cfg1.step{s}.residual", (B, shape.hidden))))
    return pre, steps


def config2(seed: int = 1002, batch: int = 64, num_blocks: int = 1200):
    """Decode, Qwen3-0.6B heads, B=64, ctx ~ U[512, 4096], pool of 1200."""
    ctx = rng(seed, "cfg2.ctx").integers(512, 4096, size=batch, endpoint=True)
    return make_decode(seed, QWEN3_06B, ctx, num_blocks, with_norms=False, name="cfg2")


def config3(seed: int = 1003, batch: int = 256):
    """Decode, Qwen3-8B, B=256, ctx ~ U[1024, 8192], pool 1.1x the need, with
    add-RMSNorm and QK-Norm+RoPE at position ctx-1."""
    ctx = rng(seed, "cfg3.ctx").integers(1024, 8192, size=batch, endpoint=True)
    need = int(sum(math.ceil(int(c) / BLOCK_SIZE) for c in ctx))
    return make_decode(seed, QWEN3_8B, ctx, math.ceil(1.1 * need), with_norms=True,
                       name="cfg3")


def config4(seed: int = 1004, n_seqs: int = 16):
    """Varlen causal prefill, Qwen3-8B, 16 sequences of U[128, 4096] tokens."""
    lengths = rng(seed, "cfg4.lens").integers(128, 4096, size=n_seqs, endpoint=True)
    return make_prefill(seed, QWEN3_8B, lengths, name="cfg4")


def config5(seed: int = 1005, batch: int = 32, num_blocks: int = 6000):
    """Long-context decode, Qwen3-8B heads, ctx log-uniform in [4096, 40960],
    1% of K token rows scaled x8."""
    u = rng(seed, "cfg5.ctx").uniform(math.log(4096), math.log(40960), size=batch)
    ctx = np.clip(np.floor(np.exp(u)), 4096, 40960).astype(np.int32)
    return make_decode(seed, QWEN3_8B, ctx, num_blocks, with_norms=False,
                       k_outlier_frac=0.01, name="cfg5")


# ------------------------------------------ prefill over the paged cache
@dataclass
class PrefixPrefill:
    """Prefill of `new` tokens per sequence whose first `prefix` tokens are
    already in the paged cache (a prefix-cache hit, or the earlier chunks of a
    chunked prefill).  The pool holds all prefix + new K/V rows of every
    sequence; q holds the new tokens' queries, packed."""
    shape: Shape
    prefix: np.ndarray           # [B] int64, multiples of the block size
    new: np.ndarray              # [B] int64
    cu_seqlens_q: np.ndarray     # [B+1] int32
    cu_seqlens_k: np.ndarray     # [B+1] int32
    block_tables: np.ndarray     # [B, MB] int32
    pool: PagedPool
    q: np.ndarray                # [sum(new), Hq, d] bf16 bits
    name: str = ""


def config_prefix(seed: int = 1006, n_seqs: int = 16):
    """Qwen3-8B heads, 16 sequences with a cached prefix of 256 * U{1..16}
    tokens (prefix caching works in whole blocks) and U[128, 1024] new tokens."""
    g = rng(seed, "pfx.lens")
    prefix = BLOCK_SIZE * g.integers(1, 16, size=n_seqs, endpoint=True).astype(np.int64)
    new = g.integers(128, 1024, size=n_seqs, endpoint=True).astype(np.int64)
    lk = prefix + new
    nb = int(sum(math.ceil(int(L) / BLOCK_SIZE) for L in lk))
    perm = rng(seed, "pfx.perm").permutation(nb).astype(np.int32)
    bt = carve_block_tables(perm, lk)
    pool = make_pool(seed, nb, bt[bt >= 0], QWEN3_8B.hkv)
    q = normal_bf16(seed, "pfx.q", (int(new.sum()), QWEN3_8B.hq, HEAD_DIM))
    return PrefixPrefill(shape=QWEN3_8B, prefix=prefix, new=new, cu_seqlens_q=cu_seqlens(new),
                         cu_seqlens_k=cu_seqlens(lk), block_tables=bt, pool=pool, q=q,
                         name="prefix")


def gather_paged(pool: PagedPool, block_tables: np.ndarray, lengths) -> tuple:
    """The K and V rows of each sequence, in order, packed [sum(lengths), Hkv, d]
    (the contiguous layout of the same keys)."""
    ks, vs = [], []
    for b, L in enumerate(np.asarray(lengths)):
        L = int(L)
        ids = block_tables[b, :math.ceil(L / BLOCK_SIZE)]
        ks.append(pool.k[ids].reshape(-1, pool.hkv, pool.k.shape[-1])[:L])
        vs.append(pool.v[ids].reshape(-1, pool.hkv, pool.v.shape[-1])[:L])
    return np.concatenate(ks), np.concatenate(vs)
