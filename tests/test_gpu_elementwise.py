"""GPU parity of the HBM-bound ops against the fp64 oracle: store_kvcache (bit
exact), the RoPE table, fused add-RMSNorm and QK-Norm + RoPE, on the small
Qwen3-0.6B layer, the Qwen3-8B decode step and the full 8B prefill batch."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import check_close, dev, dev_i32, dev_i64, err_counter, host, rope_table

pytestmark = pytest.mark.gpu

import paged_kv_attention_kvcache_gb300 as nv  # noqa: E402


@pytest.fixture(scope="module")
def cfg4():
    return wl.config4()


@pytest.fixture(scope="module")
def table():
    return rope_table()


# ------------------------------------------------------------ store_kvcache
def _store_case(batch: wl.PrefillBatch, sentinel: int = 0x7FC1):
    """Store every token's k/v (strided views of the packed qkv buffer) into a
    sentinel-filled cache on both sides; return (gpu_k, gpu_v, ref_k, ref_v)."""
    s = batch.shape
    T, Q, D = batch.qkv.shape[0], s.q_size, s.kv_size
    qkv = dev(batch.qkv)
    k = qkv[:, Q:Q + D].view(T, s.hkv, 128)
    v = qkv[:, Q + D:].view(T, s.hkv, 128)
    shape = (batch.num_blocks, wl.BLOCK_SIZE, s.hkv, 128)
    kc = torch.full(shape, 0, dtype=torch.int16, device="cuda")
    kc.fill_(sentinel)
    kc = kc.view(torch.bfloat16)
    vc = kc.clone()
    err = err_counter()
    nv.nv_store_kvcache(k, v, kc, vc, dev_i32(batch.slot_mapping), err)
    ref_k = np.full(shape, sentinel, np.uint16)
    ref_v = ref_k.copy()
    kb = batch.qkv[:, Q:Q + D].reshape(T, s.hkv, 128)
    vb = batch.qkv[:, Q + D:].reshape(T, s.hkv, 128)
    bad = oracle.store_kvcache(kb, vb, ref_k, ref_v, batch.slot_mapping)
    torch.cuda.synchronize()
    assert bad == 0 and int(err.item()) == 0
    return host(kc), host(vc), ref_k, ref_v


def test_store_kvcache_small_layer_bit_exact():
    pre, _ = wl.config1()
    gk, gv, rk, rv = _store_case(pre)
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)


def test_store_kvcache_full_prefill_bit_exact(cfg4):
    gk, gv, rk, rv = _store_case(cfg4)
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)


def test_store_kvcache_padding_and_bad_slots():
    g = np.random.default_rng(21)
    N, hkv = 9, 8
    key = wl.f32_to_bf16_bits(g.standard_normal((N, hkv, 128)).astype(np.float32))
    val = wl.f32_to_bf16_bits(g.standard_normal((N, hkv, 128)).astype(np.float32))
    slots = np.array([5, -1, 0, 700, 3, -1, -7, 511, 2], np.int32)   # 700, -7 out of range
    shape = (2, 256, hkv, 128)
    kc = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    err = err_counter()
    nv.nv_store_kvcache(dev(key), dev(val), kc, vc, dev_i32(slots), err)
    rk = np.zeros(shape, np.uint16)
    rv = rk.copy()
    bad = oracle.store_kvcache(key, val, rk, rv, slots)
    torch.cuda.synchronize()
    assert int(err.item()) == bad == 2
    assert np.array_equal(host(kc), rk) and np.array_equal(host(vc), rv)
    # empty batch is a no-op
    nv.nv_store_kvcache(dev(key[:0]), dev(val[:0]), kc, vc, dev_i32(slots[:0]), err)
    torch.cuda.synchronize()


# -------------------------------------------------------------- RoPE table
def test_rope_table_matches_exact_angles(table):
    ref = oracle.rope_cos_sin(wl.MAX_POSITION, 128, wl.ROPE_BASE)
    got = table.cpu().numpy().astype(np.float64)
    # only the final fp32 rounding separates the two
    assert np.max(np.abs(got - ref)) <= 2 ** -24


# ------------------------------------------------------------ add-RMSNorm
def _norm_case(x, r, gamma, rows=None):
    T, H = x.shape
    xd, gd = dev(x), dev(gamma)
    rd = None if r is None else dev(r)
    out = torch.empty_like(xd)
    r_out = None if r is None else torch.empty_like(xd)
    nv.nv_add_rmsnorm(xd, rd, gd, out, r_out, eps=wl.RMS_EPS)
    torch.cuda.synchronize()
    sel = slice(None) if rows is None else rows
    y_ref, r_ref = oracle.add_rmsnorm(x[sel], None if r is None else r[sel], gamma, wl.RMS_EPS)
    stats = check_close(host(out)[sel], y_ref, "add_rmsnorm out")
    if r is not None:
        got = host(r_out)[sel]
        want = oracle.round_to_bf16(r_ref)
        # bf16 + bf16 in fp32 is exact unless the exponents differ by more
        # than the fp32 mantissa can bridge; there rounding twice may move
        # the result by one bf16 ulp.
        exact32 = (wl.bf16_bits_to_f32(x[sel]).astype(np.float64) +
                   wl.bf16_bits_to_f32(r[sel]).astype(np.float64)) == \
            (wl.bf16_bits_to_f32(x[sel]) + wl.bf16_bits_to_f32(r[sel])).astype(np.float64)
        assert np.array_equal(got[exact32], want[exact32])
        ulp = np.abs(got.astype(np.int32) - want.astype(np.int32))
        assert ulp.max() <= 1
    return stats


def test_add_rmsnorm_small_layer_with_and_without_residual():
    pre, _ = wl.config1()
    _norm_case(pre.x, pre.residual, pre.gamma)
    _norm_case(pre.x, None, pre.gamma)


def test_add_rmsnorm_decode_step_8b():
    g = np.random.default_rng(22)
    x = wl.f32_to_bf16_bits(g.standard_normal((256, 4096)).astype(np.float32))
    r = wl.f32_to_bf16_bits(g.standard_normal((256, 4096)).astype(np.float32))
    gamma = wl.f32_to_bf16_bits((1 + 0.1 * g.standard_normal(4096)).astype(np.float32))
    _norm_case(x, r, gamma)


def test_add_rmsnorm_strided_rows():
    # Rows that are views into wider buffers (row stride 1024 + 64 elements):
    # each of x, residual, out and residual_out is [T, 1024] with the same
    # stride; the padding between rows must stay untouched.
    g = np.random.default_rng(29)
    T, H, pad = 37, 1024, 64
    x = wl.f32_to_bf16_bits(g.standard_normal((T, H)).astype(np.float32))
    r = wl.f32_to_bf16_bits(g.standard_normal((T, H)).astype(np.float32))
    gamma = wl.f32_to_bf16_bits((1 + 0.1 * g.standard_normal(H)).astype(np.float32))
    fill = np.full((T, pad), 0x3F80, np.uint16)                 # 1.0 in the gaps
    xb, rb = dev(np.concatenate([x, fill], 1)), dev(np.concatenate([r, fill], 1))
    ob = dev(np.concatenate([np.zeros_like(x), fill], 1))
    rob = dev(np.concatenate([np.zeros_like(x), fill], 1))
    nv.nv_add_rmsnorm(xb[:, :H], rb[:, :H], dev(gamma), ob[:, :H], rob[:, :H], eps=wl.RMS_EPS)
    torch.cuda.synchronize()
    y_ref, r_ref = oracle.add_rmsnorm(x, r, gamma, wl.RMS_EPS)
    check_close(host(ob)[:, :H], y_ref, "add_rmsnorm strided out")
    check_close(host(rob)[:, :H], r_ref, "add_rmsnorm strided residual", max_tol=2 ** -8,
                mean_tol=2 ** -9)
    for buf in (ob, rob):
        assert np.all(host(buf)[:, H:] == 0x3F80), "padding between rows was written"


def test_add_rmsnorm_in_place_residual():
    g = np.random.default_rng(23)
    x = wl.f32_to_bf16_bits(g.standard_normal((33, 1024)).astype(np.float32))
    r = wl.f32_to_bf16_bits(g.standard_normal((33, 1024)).astype(np.float32))
    gamma = wl.f32_to_bf16_bits((1 + 0.1 * g.standard_normal(1024)).astype(np.float32))
    xd, rd, gd = dev(x), dev(r), dev(gamma)
    out = torch.empty_like(xd)
    nv.nv_add_rmsnorm(xd, rd, gd, out, rd, eps=wl.RMS_EPS)       # residual updated in place
    torch.cuda.synchronize()
    y_ref, r_ref = oracle.add_rmsnorm(x, r, gamma, wl.RMS_EPS)
    check_close(host(out), y_ref, "in-place out")
    check_close(host(rd), r_ref, "in-place residual", max_tol=2 ** -8, mean_tol=2 ** -9)


def test_add_rmsnorm_full_prefill(cfg4):
    # Every row of the 33,109-token prefill batch at hidden 4096.
    _norm_case(cfg4.x, cfg4.residual, cfg4.gamma)


def test_add_rmsnorm_odd_widths():
    g = np.random.default_rng(25)
    for H in (8, 136, 1032, 16384):
        x = wl.f32_to_bf16_bits(g.standard_normal((3, H)).astype(np.float32))
        r = wl.f32_to_bf16_bits(g.standard_normal((3, H)).astype(np.float32))
        gamma = wl.f32_to_bf16_bits((1 + 0.1 * g.standard_normal(H)).astype(np.float32))
        _norm_case(x, r, gamma)


# ---------------------------------------------------------- QK-Norm + RoPE
def _qknorm_case(qkv_bits, shape: wl.Shape, positions, qn, kn, table, rows=None):
    T = qkv_bits.shape[0]
    Q, D = shape.q_size, shape.kv_size
    qkv = dev(qkv_bits)
    q = qkv[:, :Q].view(T, shape.hq, 128)
    k = qkv[:, Q:Q + D].view(T, shape.hkv, 128)
    err = err_counter()
    nv.nv_qknorm_rope(q, k, dev(qn), dev(kn), table, dev_i64(positions), eps=wl.RMS_EPS,
                      err_count=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = host(qkv)
    sel = slice(None) if rows is None else rows
    src = qkv_bits[sel]
    pos = np.asarray(positions)[sel]
    n = src.shape[0]
    q_ref = oracle.qknorm_rope(src[:, :Q].reshape(n, shape.hq, 128), qn, pos)
    k_ref = oracle.qknorm_rope(src[:, Q:Q + D].reshape(n, shape.hkv, 128), kn, pos)
    g = got[sel]
    check_close(g[:, :Q], q_ref.reshape(n, Q), "q after qknorm+rope")
    check_close(g[:, Q:Q + D], k_ref.reshape(n, D), "k after qknorm+rope")
    assert np.array_equal(g[:, Q + D:], src[:, Q + D:]), "V must be untouched"


def test_qknorm_rope_small_layer(table):
    pre, _ = wl.config1()
    _qknorm_case(pre.qkv, pre.shape, pre.positions, pre.q_norm_w, pre.k_norm_w, table)


def test_qknorm_rope_decode_positions_up_to_max(table):
    g = np.random.default_rng(26)
    shape = wl.QWEN3_8B
    pos = np.concatenate([[0, 1, 40959, 40958], g.integers(0, 40960, 252)]).astype(np.int64)
    qkv = wl.normal_bf16(26, "qk.qkv", (pos.size, shape.qkv_width))
    qn = wl.normal_bf16(26, "qk.qn", (128,), 1.0, 0.1)
    kn = wl.normal_bf16(26, "qk.kn", (128,), 1.0, 0.1)
    _qknorm_case(qkv, shape, pos, qn, kn, table)


def test_qknorm_rope_full_prefill(cfg4, table):
    # Every q and k row of the 33,109-token prefill batch, positions 0..len-1.
    _qknorm_case(cfg4.qkv, cfg4.shape, cfg4.positions, cfg4.q_norm_w, cfg4.k_norm_w, table)


def test_qknorm_rope_bad_position_leaves_row_and_counts(table):
    shape = wl.QWEN3_06B
    qkv_bits = wl.normal_bf16(28, "qk.bad", (3, shape.qkv_width))
    qkv = dev(qkv_bits)
    T, Q, D = 3, shape.q_size, shape.kv_size
    err = err_counter()
    pos = np.array([3, 40960, -1], np.int64)
    qn = wl.normal_bf16(28, "qk.bad.qn", (128,), 1.0, 0.1)
    nv.nv_qknorm_rope(qkv[:, :Q].view(T, 16, 128), qkv[:, Q:Q + D].view(T, 8, 128), dev(qn),
                      dev(qn), table, dev_i64(pos), err_count=err)
    torch.cuda.synchronize()
    got = host(qkv)
    assert int(err.item()) == 2 * (16 + 8)            # one count per (token, head) row
    assert np.array_equal(got[1:], qkv_bits[1:])
    assert not np.array_equal(got[0], qkv_bits[0])
