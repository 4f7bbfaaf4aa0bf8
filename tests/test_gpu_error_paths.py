"""Device-side range faults the host cannot see are skipped and counted in
err_count, never trapped, and leave the other sequences' results intact (the
ABI's error contract).  Each case plants one bad value among good ones."""
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


def _pool(seed, ctx, hkv, spare=2):
    g = np.random.default_rng(seed)
    nb = int(sum(max(1, math.ceil(int(c) / wl.BLOCK_SIZE)) for c in ctx)) + spare
    bt = wl.carve_block_tables(g.permutation(nb).astype(np.int32), ctx)
    k = wl.f32_to_bf16_bits(g.standard_normal((nb, wl.BLOCK_SIZE, hkv, 128)).astype(np.float32))
    v = wl.f32_to_bf16_bits(g.standard_normal((nb, wl.BLOCK_SIZE, hkv, 128)).astype(np.float32))
    return nb, bt, k, v


def test_decode_context_beyond_the_block_table_is_clamped_and_counted():
    hq, hkv = 8, 2
    ctx_ok = np.array([300, 40, 513], np.int32)
    nb, bt, k, v = _pool(940, ctx_ok, hkv)
    q = wl.normal_bf16(940, "ep.q", (3, hq, 128))
    ctx = ctx_ok.copy()
    ctx[0] = bt.shape[1] * wl.BLOCK_SIZE + 1          # longer than its table can hold
    ctx[1] = -5                                       # negative
    err = err_counter()
    o = torch.empty(3, hq, 128, dtype=torch.bfloat16, device="cuda")
    nv.nv_decode_attn_paged(dev(q), dev(k), dev(v), dev_i32(bt), dev_i32(ctx), o, SCALE,
                            kv_split_tokens=4096, err_count=err)
    torch.cuda.synchronize()
    # Two bad contexts, plus every tile load of the clamped one that reaches the
    # table's -1 padding (counted as bad block ids).
    assert int(err.item()) >= 2
    got = host(o)
    assert np.all(got[1] == 0), "a negative context attends nothing"
    ref = oracle.paged_decode(q[2:], k, v, bt[2:], ctx_ok[2:], SCALE)
    check_close(got[2:], ref, "decode next to bad contexts")


def test_prefill_sequence_with_fewer_keys_than_queries_is_skipped_and_counted():
    hq, hkv = 4, 2
    new = np.array([37, 130, 64])
    keys = new.copy()
    keys[1] = 100                                     # Lk < Lq: malformed
    g = np.random.default_rng(950)
    q = wl.f32_to_bf16_bits(g.standard_normal((int(new.sum()), hq, 128)).astype(np.float32))
    k = wl.f32_to_bf16_bits(g.standard_normal((int(keys.sum()), hkv, 128)).astype(np.float32))
    v = wl.f32_to_bf16_bits(g.standard_normal((int(keys.sum()), hkv, 128)).astype(np.float32))
    cu_q, cu_k = wl.cu_seqlens(new), wl.cu_seqlens(keys)
    o = torch.zeros(int(new.sum()), hq, 128, dtype=torch.bfloat16, device="cuda")
    err = err_counter()
    nv.nv_prefill_attn_varlen(dev(q), dev(k), dev(v), o, dev_i32(cu_q), dev_i32(cu_k),
                              int(new.max()), int(keys.max()), SCALE, err_count=err,
                              sched_counter=torch.zeros(1, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert int(err.item()) >= 1
    got = host(o)
    assert np.all(got[cu_q[1]:cu_q[2]] == 0), "the malformed sequence is left unwritten"
    for b in (0, 2):
        ref = oracle.attention_varlen(q[cu_q[b]:cu_q[b + 1]], k[cu_k[b]:cu_k[b + 1]],
                                      v[cu_k[b]:cu_k[b + 1]], wl.cu_seqlens([new[b]]),
                                      wl.cu_seqlens([keys[b]]), SCALE, True)
        check_close(got[cu_q[b]:cu_q[b + 1]], ref, f"prefill sequence {b} next to a bad one")


def test_paged_prefill_bad_block_id_is_counted_and_reads_zeros():
    hq, hkv = 4, 2
    prefix, new = np.array([300, 0]), np.array([50, 40])
    lk = prefix + new
    nb, bt, kc, vc = _pool(960, lk, hkv)
    bt = bt.copy()
    bt[0, 0] = nb + 7                                 # first block of sequence 0 is outside the pool
    g = np.random.default_rng(961)
    q = wl.f32_to_bf16_bits(g.standard_normal((int(new.sum()), hq, 128)).astype(np.float32))
    cu_q, cu_k = wl.cu_seqlens(new), wl.cu_seqlens(lk)
    o = torch.empty(int(new.sum()), hq, 128, dtype=torch.bfloat16, device="cuda")
    err = err_counter()
    nv.nv_prefill_attn_paged(dev(q), dev(kc), dev(vc), dev_i32(bt), o, dev_i32(cu_q),
                             dev_i32(cu_k), 64, SCALE, err_count=err)
    torch.cuda.synchronize()
    assert int(err.item()) >= 1
    got = host(o)
    # sequence 0 read zeros for its first 256 keys: the oracle with that block zeroed
    used = set(bt[bt >= 0].tolist())
    spare = next(i for i in range(nb) if i not in used)
    kz, vz = kc.copy(), vc.copy()
    bt_z = bt.copy()
    bt_z[0, 0] = spare                                # an unused block, zeroed for the reference
    kz[spare] = 0
    vz[spare] = 0
    ref = oracle.attention_paged_prefill(q, kz, vz, bt_z, cu_q, cu_k, SCALE)
    check_close(got, ref, "paged prefill with a block read as zeros")


def test_prefill_overstated_max_seqlen_is_safe():
    # max_seqlen_q / max_seqlen_k only size the grid: larger values are safe.
    hq, hkv = 4, 2
    lengths = np.array([5, 200, 129])
    T = int(lengths.sum())
    qkv = wl.normal_bf16(970, "ep.qkv", (T, (hq + 2 * hkv) * 128))
    Q, D = hq * 128, hkv * 128
    d_qkv = dev(qkv)
    q = d_qkv[:, :Q].view(T, hq, 128)
    k = d_qkv[:, Q:Q + D].view(T, hkv, 128)
    v = d_qkv[:, Q + D:].view(T, hkv, 128)
    cu = dev_i32(wl.cu_seqlens(lengths))
    o = torch.empty(T, hq, 128, dtype=torch.bfloat16, device="cuda")
    err = err_counter()
    nv.nv_prefill_attn_varlen(q, k, v, o, cu, cu, 4096, 4096, SCALE, err_count=err,
                              sched_counter=torch.zeros(1, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    qb = qkv[:, :Q].reshape(T, hq, 128)
    kb = qkv[:, Q:Q + D].reshape(T, hkv, 128)
    vb = qkv[:, Q + D:].reshape(T, hkv, 128)
    c = wl.cu_seqlens(lengths)
    check_close(host(o), oracle.attention_varlen(qb, kb, vb, c, c, SCALE, True),
                "prefill with overstated max_seqlen")


def test_bounded_wait_gives_up_reports_and_leaves_the_context_usable():
    # A wait on an mbarrier nothing arrives on (the pipelines' own bounded
    # wait) gives up after about a second and sets bit 30 of err_count.
    err = err_counter()
    nv.nv_selftest_wait_timeout(err)
    torch.cuda.synchronize()
    assert int(err.item()) & (1 << 30)
    # Work given the flagged counter is skipped: o keeps its sentinel.
    hq, hkv, lengths = 4, 2, np.array([200, 37])
    T = int(lengths.sum())
    q = wl.normal_bf16(970, "st.q", (T, hq, 128))
    k = wl.normal_bf16(970, "st.k", (T, hkv, 128))
    v = wl.normal_bf16(970, "st.v", (T, hkv, 128))
    cu = wl.cu_seqlens(lengths)
    o = torch.full((T, hq, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    nv.nv_prefill_attn_varlen(dev(q), dev(k), dev(v), o, dev_i32(cu), dev_i32(cu), 200, 200,
                              SCALE, err_count=err)
    torch.cuda.synchronize()
    assert bool(torch.all(o == 7.0))
    # The context is still usable: with a clear counter the same call runs and
    # matches the oracle.
    fresh = err_counter()
    nv.nv_prefill_attn_varlen(dev(q), dev(k), dev(v), o, dev_i32(cu), dev_i32(cu), 200, 200,
                              SCALE, err_count=fresh)
    torch.cuda.synchronize()
    assert int(fresh.item()) == 0
    check_close(host(o), oracle.attention_varlen(q, k, v, cu, cu, SCALE, True),
                "prefill after a reported stall")
