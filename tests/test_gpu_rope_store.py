"""GPU parity of the fused QK-Norm + RoPE + store_kvcache pass.  The oracle
runs the two steps of "Nano-vLLM 源码解读 第17篇", sec. 4 and 5.1, in order:
per-head RMSNorm + rotation in fp64, rounding of q and k to bf16 (the model
dtype), then the slot scatter.  The fused kernel must land within the same
bounds as the two separate kernels, and, because it shares their per-row
arithmetic, give their bits exactly."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import check_cache_rows, check_close, dev, dev_i32, dev_i64, err_counter, host, rope_table

pytestmark = pytest.mark.gpu

import paged_kv_attention_kvcache_gb300 as nv  # noqa: E402


def _inputs(seed, shape, lengths, pad_tokens=0, spare_blocks=2):
    """Packed qkv of a prefill batch, its positions and slots in a fresh pool;
    `pad_tokens` extra rows at the end carry slot -1."""
    g = np.random.default_rng(seed)
    lengths = np.asarray(lengths)
    nb = int(sum(math.ceil(int(L) / wl.BLOCK_SIZE) for L in lengths)) + spare_blocks
    bt = wl.carve_block_tables(g.permutation(nb).astype(np.int32), lengths)
    seq = np.repeat(np.arange(lengths.size), lengths)
    pos = np.concatenate([np.arange(int(L)) for L in lengths]).astype(np.int64)
    slots = wl.slots_for_positions(bt, seq, pos).astype(np.int32)
    T = int(lengths.sum()) + pad_tokens
    qkv = wl.normal_bf16(seed, "rs.qkv", (T, shape.qkv_width))
    pos = np.concatenate([pos, np.zeros(pad_tokens, np.int64)])
    slots = np.concatenate([slots, np.full(pad_tokens, -1, np.int32)])
    qn = wl.normal_bf16(seed, "rs.qn", (128,), 1.0, 0.1)
    kn = wl.normal_bf16(seed, "rs.kn", (128,), 1.0, 0.1)
    kc0 = wl.normal_bf16(seed, "rs.kc", (nb, wl.BLOCK_SIZE, shape.hkv, 128))
    vc0 = wl.normal_bf16(seed, "rs.vc", (nb, wl.BLOCK_SIZE, shape.hkv, 128))
    return qkv, pos, slots, qn, kn, kc0, vc0


def _views(qkv, s):
    T = qkv.shape[0]
    Q, D = s.q_size, s.kv_size
    return (qkv[:, :Q].view(T, s.hq, 128), qkv[:, Q:Q + D].view(T, s.hkv, 128),
            qkv[:, Q + D:].view(T, s.hkv, 128))


def _run_fused(qkv_bits, pos, slots, qn, kn, kc0, vc0, s, write_k):
    table = rope_table()
    qkv, kc, vc = dev(qkv_bits), dev(kc0), dev(vc0)
    q, k, v = _views(qkv, s)
    err = err_counter()
    nv.nv_qknorm_rope_store(q, k, v, dev(qn), dev(kn), table, dev_i64(pos), kc, vc,
                            dev_i32(slots), eps=wl.RMS_EPS, write_k=write_k, err_count=err)
    torch.cuda.synchronize()
    return host(qkv), host(kc), host(vc), int(err.item())


def _run_pair(qkv_bits, pos, slots, qn, kn, kc0, vc0, s):
    table = rope_table()
    qkv, kc, vc = dev(qkv_bits), dev(kc0), dev(vc0)
    q, k, v = _views(qkv, s)
    err = err_counter()
    nv.nv_qknorm_rope(q, k, dev(qn), dev(kn), table, dev_i64(pos), eps=wl.RMS_EPS,
                      err_count=err)
    nv.nv_store_kvcache(k, v, kc, vc, dev_i32(slots), err)
    torch.cuda.synchronize()
    return host(qkv), host(kc), host(vc), int(err.item())


def _oracle(qkv_bits, pos, slots, qn, kn, kc0, vc0, s):
    T, Q, D = qkv_bits.shape[0], s.q_size, s.kv_size
    q_rot = oracle.qknorm_rope(qkv_bits[:, :Q].reshape(T, s.hq, 128), qn, pos)
    k_rot = oracle.qknorm_rope(qkv_bits[:, Q:Q + D].reshape(T, s.hkv, 128), kn, pos)
    kb = oracle.round_to_bf16(k_rot)
    vb = qkv_bits[:, Q + D:].reshape(T, s.hkv, 128)
    kc, vc = kc0.copy(), vc0.copy()
    assert oracle.store_kvcache(kb, vb, kc, vc, slots) == 0
    return q_rot, k_rot, kc, vc


@pytest.mark.parametrize("write_k", [False, True])
def test_fused_rope_store_small_ragged_with_padding(write_k):
    s = wl.QWEN3_06B
    args = _inputs(600, s, [1, 37, 256, 300], pad_tokens=3)
    qkv0 = args[0]
    Q, D = s.q_size, s.kv_size
    got_qkv, got_kc, got_vc, err = _run_fused(*args, s, write_k)
    assert err == 0
    q_rot, k_rot, ref_kc, ref_vc = _oracle(*args, s)
    T = qkv0.shape[0]
    check_close(got_qkv[:, :Q], q_rot.reshape(T, Q), "fused q")
    if write_k:
        check_close(got_qkv[:, Q:Q + D], k_rot.reshape(T, D), "fused k in place")
    else:
        assert np.array_equal(got_qkv[:, Q:Q + D], qkv0[:, Q:Q + D]), "k must stay untouched"
    assert np.array_equal(got_qkv[:, Q + D:], qkv0[:, Q + D:]), "v must stay untouched"
    check_cache_rows(got_kc, ref_kc, "fused k cache")
    assert np.array_equal(got_vc, ref_vc), "v cache must be bit-exact"
    # Same bits as the two separate kernels.
    pair_qkv, pair_kc, pair_vc, perr = _run_pair(*args, s)
    assert perr == 0
    assert np.array_equal(got_qkv[:, :Q], pair_qkv[:, :Q])
    if write_k:
        assert np.array_equal(got_qkv, pair_qkv)
    assert np.array_equal(got_kc, pair_kc) and np.array_equal(got_vc, pair_vc)


def test_fused_rope_store_qwen3_8b_prefill_batch_full_size():
    pre = wl.config4()
    s = pre.shape
    nb = pre.num_blocks
    kc0 = np.zeros((nb, wl.BLOCK_SIZE, s.hkv, 128), np.uint16)
    vc0 = np.zeros_like(kc0)
    args = (pre.qkv, pre.positions, pre.slot_mapping, pre.q_norm_w, pre.k_norm_w, kc0, vc0)
    got_qkv, got_kc, got_vc, err = _run_fused(*args, s, True)
    assert err == 0
    q_rot, k_rot, ref_kc, ref_vc = _oracle(*args, s)
    T, Q, D = pre.qkv.shape[0], s.q_size, s.kv_size
    check_close(got_qkv[:, :Q], q_rot.reshape(T, Q), "8b fused q (every row)")
    check_close(got_qkv[:, Q:Q + D], k_rot.reshape(T, D), "8b fused k (every row)")
    check_cache_rows(got_kc, ref_kc, "8b fused k cache")
    assert np.array_equal(got_vc, ref_vc)


def test_fused_rope_store_counts_bad_slots_and_positions():
    s = wl.QWEN3_06B
    qkv, pos, slots, qn, kn, kc0, vc0 = _inputs(620, s, [40])
    num_slots = kc0.shape[0] * kc0.shape[1]
    slots = slots.copy()
    pos = pos.copy()
    slots[3] = num_slots          # out of range: counted once, nothing cached
    slots[5] = -7                 # negative, not the padding marker
    pos[9] = wl.MAX_POSITION      # out of range: counted per q and k row
    got_qkv, got_kc, got_vc, err = _run_fused(qkv, pos, slots, qn, kn, kc0, vc0, s, False)
    assert err == 2 + (s.hq + s.hkv)
    Q, D = s.q_size, s.kv_size
    assert np.array_equal(got_qkv[9], qkv[9]), "token with a bad position stays untouched"
    # every other token matches the oracle; the bad tokens leave their slots as they were
    good = np.ones(40, bool)
    good[[3, 5, 9]] = False
    q_rot, k_rot, ref_kc, ref_vc = _oracle(qkv[good], pos[good], slots[good], qn, kn, kc0, vc0, s)
    check_close(got_qkv[good, :Q], q_rot.reshape(-1, Q), "q of good tokens")
    # token 9's v row is still copied to its slot (documented)
    ref_vc.reshape(-1, D)[slots[9]] = qkv[9, Q + D:]
    check_cache_rows(got_kc, ref_kc, "k cache with bad tokens")
    assert np.array_equal(got_vc, ref_vc)


def test_bad_tokens_in_late_passes_of_the_grid():
    # A batch of several times the resident grid's rows, so each row group
    # walks many rows; the bad slots and positions sit in late passes and at
    # the very last tokens.  Both the fused pass and the in-place rotation
    # must skip and count exactly those rows and give the same bits elsewhere.
    s = wl.QWEN3_8B
    qkv, pos, slots, qn, kn, kc0, vc0 = _inputs(630, s, [1000, 1500, 700])
    T, Q, D = qkv.shape[0], s.q_size, s.kv_size
    num_slots = kc0.shape[0] * kc0.shape[1]
    slots, pos = slots.copy(), pos.copy()
    slots[2900], slots[T - 1] = num_slots + 5, -3
    pos[3100], pos[T - 2] = -1, wl.MAX_POSITION
    got_qkv, got_kc, got_vc, err = _run_fused(qkv, pos, slots, qn, kn, kc0, vc0, s, True)
    assert err == 2 + 2 * (s.hq + s.hkv)
    for t in (3100, T - 2):
        assert np.array_equal(got_qkv[t], qkv[t]), "token with a bad position stays untouched"
    good = np.ones(T, bool)
    good[[2900, 3100, T - 2, T - 1]] = False
    q_rot, k_rot, ref_kc, ref_vc = _oracle(qkv[good], pos[good], slots[good], qn, kn, kc0, vc0, s)
    check_close(got_qkv[good, :Q], q_rot.reshape(-1, Q), "q of good tokens")
    check_close(got_qkv[good, Q:Q + D], k_rot.reshape(-1, D), "k of good tokens")
    for t in (3100, T - 2):                      # v rows of bad-position tokens are still copied
        ref_vc.reshape(-1, D)[slots[t]] = qkv[t, Q + D:]
    check_cache_rows(got_kc, ref_kc, "k cache with late bad tokens")
    assert np.array_equal(got_vc, ref_vc)

    table = rope_table()
    d_qkv = dev(qkv)
    q, k, _ = _views(d_qkv, s)
    err_t = err_counter()
    nv.nv_qknorm_rope(q, k, dev(qn), dev(kn), table, dev_i64(pos), eps=wl.RMS_EPS,
                      err_count=err_t)
    torch.cuda.synchronize()
    assert int(err_t.item()) == 2 * (s.hq + s.hkv)
    assert np.array_equal(host(d_qkv), got_qkv), "in-place rotation gives the fused pass's bits"
