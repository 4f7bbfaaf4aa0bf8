"""GPU parity of paged decode attention (with split-KV and the log-sum-exp
merge) against the fp64 oracle's stitched-sequence definition."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import check_close, dev, dev_i32, err_counter, host

pytestmark = pytest.mark.gpu

import paged_kv_attention_kvcache_gb300 as nv  # noqa: E402

SCALE = 128 ** -0.5


def run_decode(q_bits, pool_k, pool_v, bt, ctx, split=0, q_stride_pad=0, err=None):
    """GPU decode through the binding; returns (out bits, err count)."""
    B, Hq, _ = q_bits.shape
    nb, bs, Hkv, _ = pool_k.shape
    if q_stride_pad:
        qbuf = dev(np.concatenate([q_bits.reshape(B, -1),
                                   np.zeros((B, q_stride_pad), np.uint16)], axis=1))
        q = qbuf[:, :Hq * 128].view(B, Hq, 128)
    else:
        q = dev(q_bits)
    kc = pool_k if isinstance(pool_k, torch.Tensor) else dev(pool_k)
    vc = pool_v if isinstance(pool_v, torch.Tensor) else dev(pool_v)
    o = torch.empty(B, Hq, 128, dtype=torch.bfloat16, device="cuda")
    ws_bytes = nv.nv_decode_attn_workspace_size(B, Hq, Hkv, 128, bt.shape[1], bs, split)
    ws = torch.empty(max(ws_bytes // 4, 1), dtype=torch.float32, device="cuda") if ws_bytes else None
    err = err_counter() if err is None else err
    nv.nv_decode_attn_paged(q, kc, vc, dev_i32(bt), dev_i32(ctx), o, SCALE, workspace=ws,
                            kv_split_tokens=split, err_count=err)
    torch.cuda.synchronize()
    return host(o), int(err.item())


def random_case(seed, B, Hq, Hkv, ctx, bs=256, spare=3, outliers=0.0):
    g = np.random.default_rng(seed)
    ctx = np.asarray(ctx, np.int32)
    need = sum(max(1, math.ceil(int(c) / bs)) for c in ctx)
    nb = need + spare
    perm = g.permutation(nb).astype(np.int32)
    bt = wl.carve_block_tables(perm, ctx, block_size=bs)
    kf = g.standard_normal((nb, bs, Hkv, 128)).astype(np.float32)
    if outliers:
        hit = g.random((nb, bs)) < outliers
        kf[hit] *= 8
    k = wl.f32_to_bf16_bits(kf)
    v = wl.f32_to_bf16_bits(g.standard_normal((nb, bs, Hkv, 128)).astype(np.float32))
    q = wl.f32_to_bf16_bits(g.standard_normal((len(ctx), Hq, 128)).astype(np.float32))
    return q, k, v, bt, ctx


@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 2), (8, 2), (16, 2), (32, 2)])
def test_decode_gqa_groups_and_edge_contexts(hq, hkv):
    ctx = [1, 63, 64, 65, 255, 256, 257, 700]
    q, k, v, bt, ctx = random_case(100 + hq, len(ctx), hq, hkv, ctx)
    got, err = run_decode(q, k, v, bt, ctx)
    assert err == 0
    check_close(got, oracle.paged_decode(q, k, v, bt, ctx, SCALE), f"decode G={hq // hkv}")


@pytest.mark.parametrize("split", [64, 128, 192, 512])
def test_decode_forced_splits_match_oracle(split):
    ctx = [1, 64, 300, 1000, 2049]
    q, k, v, bt, ctx = random_case(200 + split, len(ctx), 8, 2, ctx)
    got, err = run_decode(q, k, v, bt, ctx, split=split)
    assert err == 0
    check_close(got, oracle.paged_decode(q, k, v, bt, ctx, SCALE), f"decode split={split}")


def test_decode_split_count_invariance():
    # Splitting only regroups the sum; what changes is where P is rounded to
    # bf16 (against each split's own running max), which moves outputs by a
    # few 1e-4 at most.  Every split count must also match the oracle.
    ctx = [3000, 1500, 700, 257]
    q, k, v, bt, ctx = random_case(301, len(ctx), 32, 8, ctx)
    ref = oracle.paged_decode(q, k, v, bt, ctx, SCALE)
    outs = []
    for split in (64, 320, 0, 4096):
        got, err = run_decode(q, k, v, bt, ctx, split=split)
        assert err == 0
        check_close(got, ref, f"split={split}")
        outs.append(wl.bf16_bits_to_f32(got).astype(np.float64))
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) <= 2e-3


def test_decode_empty_context_and_token_stride():
    ctx = [0, 5, 0, 129]
    q, k, v, bt, ctx = random_case(302, len(ctx), 8, 2, ctx)
    got, err = run_decode(q, k, v, bt, ctx, q_stride_pad=2 * 2 * 128)
    assert err == 0
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    check_close(got, oracle.paged_decode(q, k, v, bt, ctx, SCALE), "decode ctx=0 / strided q")


def test_decode_nan_in_unused_cache_rows_does_not_leak():
    # Rows past the context in the last block hold NaN bits; they must not
    # reach the output (their probability is zero).
    ctx = [70, 129]
    q, k, v, bt, ctx = random_case(303, len(ctx), 4, 2, ctx)
    for b, L in enumerate(ctx):
        last = bt[b, (int(L) - 1) // 256]
        k[last, int(L) % 256:] = 0x7FC0
        v[last, int(L) % 256:] = 0x7FC0
    got, err = run_decode(q, k, v, bt, ctx)
    assert err == 0
    check_close(got, oracle.paged_decode(q, k, v, bt, ctx, SCALE), "decode with NaN tail")


def _drop_blocks(bt_row, L, bad, bs=256):
    """The block table and context length of the same sequence with the
    blocks at logical indices `bad` removed: what a decode that skips those
    keys attends over.  Only whole blocks, or the last (partial) one, are
    removed, so the remaining keys stay in logical order."""
    n = -(-int(L) // bs)
    keep = [i for i in range(n) if i not in bad]
    gone = sum(min(bs, int(L) - i * bs) for i in bad)
    row = np.full(bt_row.shape, -1, np.int32)
    row[:len(keep)] = bt_row[keep]
    return row, int(L) - gone


@pytest.mark.parametrize("split", [0, 64, 192, 256, 512])
def test_decode_bad_block_id_is_counted_not_faulted(split):
    # Keys of a block id outside the pool are skipped ("nano-vllm code
    # walkthrough", Decode Stage gathers key j from block_tables[b][j / 256]);
    # the output is attention over the keys that remain.  Cases: the last
    # (partial) block bad, the first block bad, a middle block bad, every
    # block bad (zeros), and an untouched sequence.  With 64- and 256-key
    # splits a bad block fills whole splits; with 192 and 512 part of one.
    ctx = [300, 40, 1000, 700, 200, 900]
    bad = {0: [1], 2: [0], 3: [1], 4: [0], 5: [2]}
    q, k, v, bt, ctx = random_case(304, len(ctx), 8, 2, ctx)
    bt = bt.copy()
    for b, blocks in bad.items():
        for i in blocks:
            bt[b, i] = 10_000 if b % 2 == 0 else -7        # past the pool / negative
    got, err = run_decode(q, k, v, bt, ctx, split=split)
    assert err >= len(bad)
    assert err & (1 << 30) == 0
    assert np.all(np.isfinite(wl.bf16_bits_to_f32(got))), "non-finite decode output"
    assert np.all(got[4] == 0), "a sequence with every key skipped returns zeros"
    bt_ref = bt.copy()
    ctx_ref = ctx.copy()
    for b, blocks in bad.items():
        bt_ref[b], ctx_ref[b] = _drop_blocks(bt[b], ctx[b], blocks)
    ref = oracle.paged_decode(q, k, v, bt_ref, ctx_ref, SCALE)
    check_close(got, ref, f"decode with bad block ids, split={split}")


def _planted_case(step: wl.DecodeStep, seed: int):
    """Exact block-table indexing case on a workload's own block tables and
    context lengths.  Query head h of sequence b is a vector u of +-1, and one
    logical key j(b, h) of its kv head holds 32 u: its score (32 * 128 *
    scale = 362) exceeds every other key's by more than 126 binary orders of
    magnitude, so its softmax weight is 1 and every other weight is 0 in
    fp32.  Every V row carries its own logical position, sequence and kv head
    in its first five elements (integers below 256, exact in bf16).  The
    output of (b, h) must then be V at j(b, h), bit for bit: a wrong block,
    offset, tile or split finds another key or another V row."""
    s = step.shape
    B = step.context_lens.size
    G = s.hq // s.hkv
    bs = wl.BLOCK_SIZE
    g = np.random.default_rng(seed)
    ctx = step.context_lens.astype(np.int64)
    bt = step.block_tables
    u = g.choice(np.array([-1.0, 1.0], np.float32), size=(B, s.hq, 128))
    q_bits = wl.f32_to_bf16_bits(u)
    # Planted positions: distinct within each (sequence, kv head); tile,
    # block and split edges first, then random.
    pos = np.empty((B, s.hq), np.int64)
    assert int(ctx.min()) >= G, "one distinct planted key per query head of a group"
    for b in range(B):
        L = int(ctx[b])
        edges = [p for p in (0, L - 1, 63, 64, 255, 256, 1535, 1536, 2047, 2048, 4095, 4096,
                             L // 2) if 0 <= p < L]
        for kvh in range(s.hkv):
            take = []
            start = (b + kvh) % len(edges)
            for i in range(len(edges)):
                p = edges[(start + i) % len(edges)]
                if p not in take and len(take) < G // 2:
                    take.append(p)
            while len(take) < G:
                p = int(g.integers(0, L))
                if p not in take:
                    take.append(p)
            pos[b, kvh * G:(kvh + 1) * G] = take
    k = step.pool.k.copy()
    v = step.pool.v.copy()
    heads = np.arange(s.hq)
    for b in range(B):
        blk = bt[b, pos[b] // bs]
        off = pos[b] % bs
        k[blk, off, heads // G] = wl.f32_to_bf16_bits(32.0 * u[b])
    # V rows: (j & 255, j >> 8, b & 255, kv head, b >> 8) in elements 0..4.
    seq_of = np.full(step.pool.num_blocks, -1, np.int64)
    base = np.zeros(step.pool.num_blocks, np.int64)
    for b in range(B):
        n = -(-int(ctx[b]) // bs)
        seq_of[bt[b, :n]] = b
        base[bt[b, :n]] = np.arange(n) * bs
    used = np.nonzero(seq_of >= 0)[0]
    j = base[used][:, None] + np.arange(bs)[None, :]
    sq = seq_of[used][:, None] + 0 * j
    for kvh in range(s.hkv):
        code = np.stack([j & 255, j >> 8, sq & 255, np.full_like(j, kvh), sq >> 8], axis=-1)
        v[used[:, None], np.arange(bs)[None, :], kvh, :5] = wl.f32_to_bf16_bits(
            code.astype(np.float32))
    want = np.empty((B, s.hq, 128), np.uint16)
    for b in range(B):
        blk = bt[b, pos[b] // bs]
        want[b] = v[blk, pos[b] % bs, heads // G]
    return q_bits, k, v, want


@pytest.mark.parametrize("cfg,splits", [("config3", (0, 64, 192)), ("config5", (0, 256, 1000))])
def test_decode_block_table_indexing_exact(cfg, splits):
    step = getattr(wl, cfg)()
    q_bits, k, v, want = _planted_case(step, 4400 + len(cfg))
    kc, vc = dev(k), dev(v)
    del k, v
    for split in splits:
        got, err = run_decode(q_bits, kc, vc, step.block_tables, step.context_lens, split=split)
        assert err == 0
        bad = np.argwhere(np.any(got != want, axis=-1))
        assert bad.size == 0, (f"{step.name} split={split}: {len(bad)} (seq, head) outputs are "
                               f"not the planted key's V row; first {bad[:5].tolist()}")


def _full_config(step: wl.DecodeStep, split=0):
    """Every (sequence, head) of a configured decode workload against the
    oracle."""
    s = step.shape
    B = step.context_lens.size
    q_bits = step.qkv[:, :s.q_size].reshape(B, s.hq, 128)
    kc, vc = dev(step.pool.k), dev(step.pool.v)
    got, err = run_decode(q_bits, kc, vc, step.block_tables, step.context_lens, split=split)
    assert err == 0
    del kc, vc
    ref = oracle.paged_decode(q_bits, step.pool.k, step.pool.v, step.block_tables,
                              step.context_lens, SCALE)
    return check_close(got, ref, f"{step.name} decode split={split or 'auto'}")


def test_decode_qwen3_06b_batch64_full_size():
    _full_config(wl.config2())


def test_decode_qwen3_8b_batch256_full_size():
    _full_config(wl.config3())


@pytest.mark.parametrize("split", [0, 256])
def test_decode_long_context_split_kv_full_size(split):
    _full_config(wl.config5(), split=split)


def test_decode_longest_context():
    # Contexts of the longest length the model takes, next to a single key.
    ctx = [wl.MAX_POSITION, 1, wl.MAX_POSITION - 1]
    q, k, v, bt, ctx = random_case(306, len(ctx), 32, 8, ctx)
    got, err = run_decode(q, k, v, bt, ctx)
    assert err == 0
    check_close(got, oracle.paged_decode(q, k, v, bt, ctx, SCALE), "decode 40960")


@pytest.mark.parametrize("bs", [64, 128, 512])
@pytest.mark.parametrize("split", [0, 192])
def test_decode_other_block_sizes(bs, split):
    # Block sizes other than the pages' 256 (any multiple of the 64-key tile);
    # a split of 192 keys straddles block boundaries for every one of them.
    ctx = [1, bs - 1, bs, bs + 1, 3 * bs + 17, 1000]
    q, k, v, bt, ctx = random_case(310 + bs + split, len(ctx), 16, 4, ctx, bs=bs)
    got, err = run_decode(q, k, v, bt, ctx, split=split)
    assert err == 0
    check_close(got, oracle.paged_decode(q, k, v, bt, ctx, SCALE), f"decode bs={bs} split={split}")
