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


def test_decode_bad_block_id_is_counted_not_faulted():
    ctx = [300, 40]
    q, k, v, bt, ctx = random_case(304, len(ctx), 8, 2, ctx)
    bt = bt.copy()
    bt[0, 1] = 10_000                       # beyond the pool: keys 256..299 skipped
    got, err = run_decode(q, k, v, bt, ctx)
    assert err >= 1
    # sequence 1 is unaffected
    ref = oracle.paged_decode(q[1:], k, v, bt[1:], ctx[1:], SCALE)
    check_close(got[1:], ref, "decode unaffected sequence")


def _full_config(step: wl.DecodeStep, n_pairs, seed, split=0):
    s = step.shape
    B = step.context_lens.size
    q_bits = step.qkv[:, :s.q_size].reshape(B, s.hq, 128)
    kc, vc = dev(step.pool.k), dev(step.pool.v)
    got, err = run_decode(q_bits, kc, vc, step.block_tables, step.context_lens, split=split)
    assert err == 0
    g = np.random.default_rng(seed)
    pairs = np.stack([g.integers(0, B, n_pairs), g.integers(0, s.hq, n_pairs)], axis=1)
    ref = oracle.paged_decode(q_bits, step.pool.k, step.pool.v, step.block_tables,
                              step.context_lens, SCALE, pairs=pairs)
    return check_close(got[pairs[:, 0], pairs[:, 1]], ref, step.name)


def test_decode_qwen3_06b_batch64_full_size():
    step = wl.config2()
    _full_config(step, 1024, 402)


def test_decode_qwen3_8b_batch256_full_size():
    step = wl.config3()
    _full_config(step, 256, 403)


@pytest.mark.parametrize("split", [0, 256])
def test_decode_long_context_split_kv_full_size(split):
    step = wl.config5()
    _full_config(step, 96, 405, split=split)


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
