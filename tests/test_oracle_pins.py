"""Pins for the fp64 oracle: values the pages print, closed forms, invariants
and brute force on tiny inputs.  Nothing here compares the oracle with a copy
of its own formula; each check would fail on a plausible slip in it (a dropped
term, a wrong sign or index, a transposed operand).  CPU only."""
import math

import numpy as np
import pytest

import oracle
import workloads as wl
from conftest import read_golden

B16 = wl.f32_to_bf16_bits
F32 = wl.bf16_bits_to_f32


def bits(a):
    return B16(np.asarray(a, dtype=np.float32))


# ------------------------------------------------------------ bf16 rounding
def test_round_to_bf16_ties_and_specials():
    one = 1.0
    cases = {
        one: 0x3F80,
        one + 2 ** -8: 0x3F80,            # tie between 1 and 1+2^-7: even stays
        one + 3 * 2 ** -8: 0x3F82,        # tie between 1+2^-7 and 1+2^-6: to even
        one + 2 ** -8 + 2 ** -30: 0x3F81,  # just above the tie
        -2.5: 0xC020,
        0.0: 0x0000,
        2.0 ** -133: 0x0001,              # smallest bf16 subnormal
        3.0 * 2.0 ** -134: 0x0002,        # subnormal tie 1.5 quanta -> 2 (even)
        2.0 ** 127 * (2 - 2 ** -7): 0x7F7F,
    }
    got = oracle.round_to_bf16(np.array(list(cases.keys())))
    assert [int(g) for g in got] == list(cases.values())


def test_round_to_bf16_matches_fp32_integer_rounding():
    # Two independent implementations agree on fp32-representable inputs.
    g = np.random.default_rng(0)
    x = (g.standard_normal(200000) * np.exp(g.uniform(-30, 30, 200000))).astype(np.float32)
    assert np.array_equal(oracle.round_to_bf16(x.astype(np.float64)), B16(x))


# ------------------------------------------------------------ store_kvcache
def test_store_kvcache_page_example():
    gold = read_golden("store_kvcache_toy.txt")
    n, hkv, hd, slots = (int(gold[k][0]) for k in ("n_tokens", "kv_heads", "head_dim", "num_slots"))
    D = hkv * hd
    key = (np.arange(n)[:, None] * 10 + np.arange(D)[None, :]).astype(np.float32)
    key = bits(key).reshape(n, hkv, hd)
    value = bits(F32(key) + 100)
    kc = np.zeros((1, slots, hkv, hd), np.uint16)
    vc = np.zeros_like(kc)
    bad = oracle.store_kvcache(key, value, kc, vc, np.array(gold["slot_mapping"], np.int32))
    assert bad == 0
    flat_k = F32(kc).reshape(-1, D)
    for s in range(slots):
        assert flat_k[s].tolist() == gold[f"k_cache_slot{s}"]
    assert F32(vc).reshape(-1, D)[0].tolist() == gold["v_cache_slot0"]


def test_store_scatter_skeleton_example():
    gold = read_golden("scatter_toy.txt")
    n, w = int(gold["n_rows"][0]), int(gold["width"][0])
    src = bits(np.arange(n * w, dtype=np.float32)).reshape(n, 1, w)
    dst_k = np.zeros((1, n, 1, w), np.uint16)
    dst_v = np.zeros_like(dst_k)
    oracle.store_kvcache(src, src, dst_k, dst_v, np.array(gold["slot"], np.int32))
    for r in range(n):
        assert F32(dst_k).reshape(n, w)[r].tolist() == gold[f"dst_row{r}"]
    assert np.array_equal(dst_k, dst_v)


def test_store_out_of_range_slots_skipped_and_counted():
    key = bits(np.ones((3, 1, 4), np.float32))
    kc = np.full((2, 2, 1, 4), 7, np.uint16)
    vc = kc.copy()
    bad = oracle.store_kvcache(key, key, kc, vc, np.array([4, -2, 3], np.int32))
    assert bad == 2
    assert np.all(kc.reshape(4, 4)[:3] == 7)
    assert np.all(F32(kc).reshape(4, 4)[3] == 1.0)


# ------------------------------------------------------------------ RMSNorm
@pytest.mark.parametrize("c", [1.0, -0.75, 3.0, 1e-3])
def test_rmsnorm_constant_vector(c):
    H, eps = 64, 1e-6
    g = np.random.default_rng(1)
    w = bits(1 + 0.1 * g.standard_normal(H))
    x = bits(np.full((2, H), c))
    y, r = oracle.add_rmsnorm(x, None, w, eps)
    cq = float(F32(x)[0, 0])
    expect = F32(w).astype(np.float64) * cq / math.sqrt(cq * cq + eps)
    assert r is None
    np.testing.assert_allclose(y[0], expect, rtol=1e-14, atol=0)
    np.testing.assert_allclose(y[1], expect, rtol=1e-14, atol=0)


def test_rmsnorm_spike_vector_mean_not_sum():
    # x = a*e_k: mean(x^2) = a^2/H, so y_k = w_k * a / sqrt(a^2/H + eps).
    H, eps, a, k = 128, 1e-6, 2.0, 5
    w = bits(np.linspace(0.5, 1.5, H))
    x = np.zeros((1, H), np.float32)
    x[0, k] = a
    y, _ = oracle.add_rmsnorm(bits(x), None, w, eps)
    assert np.count_nonzero(y) == 1
    assert y[0, k] == pytest.approx(float(F32(w)[k]) * a / math.sqrt(a * a / H + eps), rel=1e-14)


def test_add_rmsnorm_residual_cancels_and_doubles():
    g = np.random.default_rng(2)
    H = 256
    x = bits(g.standard_normal((4, H)))
    w = bits(1 + 0.1 * g.standard_normal(H))
    neg = bits(-F32(x))
    y0, r0 = oracle.add_rmsnorm(x, neg, w, 1e-6)        # s = 0 exactly
    assert np.all(r0 == 0) and np.all(y0 == 0)
    y2, r2 = oracle.add_rmsnorm(x, x, w, 1e-6)          # s = 2x exactly
    np.testing.assert_array_equal(r2, 2.0 * F32(x).astype(np.float64))
    y1, _ = oracle.add_rmsnorm(x, None, w, 1e-6)
    # scale invariance up to eps: relative change (3/8) eps / mean(x^2)
    np.testing.assert_allclose(y2, y1, rtol=2e-6, atol=1e-12)


def test_rmsnorm_unit_rms_and_weight_is_elementwise():
    g = np.random.default_rng(3)
    H, eps = 1024, 1e-6
    x = bits(g.standard_normal((8, H)) * 3)
    ones = bits(np.ones(H))
    y, _ = oracle.add_rmsnorm(x, None, ones, eps)
    ms = np.mean(y * y, axis=1)
    np.testing.assert_allclose(ms, 1.0, atol=1e-6)      # mean(y^2) = ms/(ms+eps)
    w = bits(np.linspace(0.25, 2.0, H))
    yw, _ = oracle.add_rmsnorm(x, None, w, eps)
    np.testing.assert_allclose(yw, y * F32(w)[None, :], rtol=1e-14)
    # exact powers of two leave bf16 inputs exact and the output unchanged
    y4, _ = oracle.add_rmsnorm(bits(F32(x) * 4), None, ones, eps)
    np.testing.assert_allclose(y4, y, rtol=2e-6, atol=1e-12)


# --------------------------------------------------------------------- RoPE
def test_rope_table_closed_forms():
    d, base, P = 128, 1e6, 50
    t = oracle.rope_cos_sin(P, d, base)
    assert np.all(t[0, :64] == 1.0) and np.all(t[0, 64:] == 0.0)
    p = np.arange(P)
    np.testing.assert_allclose(t[:, 0], np.cos(p), atol=1e-15)      # inv_freq_0 = 1
    np.testing.assert_allclose(t[:, 64], np.sin(p), atol=1e-15)
    # pair 1 at position 1: angle = base^(-2/128) = 10^(-6/64)
    a1 = 0.8058421877614819
    assert t[1, 1] == pytest.approx(math.cos(a1), abs=1e-15)
    assert t[1, 65] == pytest.approx(math.sin(a1), abs=1e-15)
    # the last pair's frequency is base^(-126/128)
    a63 = 1e6 ** (-126 / 128)
    assert t[7, 63] == pytest.approx(math.cos(7 * a63), abs=1e-15)
    np.testing.assert_allclose(t[:, :64] ** 2 + t[:, 64:] ** 2, 1.0, atol=1e-15)
    # angle linear in position: angle addition from rows 17 and 23 gives row 40
    c = t[17, :64] * t[23, :64] - t[17, 64:] * t[23, 64:]
    s = t[17, 64:] * t[23, :64] + t[17, :64] * t[23, 64:]
    np.testing.assert_allclose(c, t[40, :64], atol=1e-14)
    np.testing.assert_allclose(s, t[40, 64:], atol=1e-14)


def _heads(g, T, nh, d=128, scale=1.0):
    return bits(g.standard_normal((T, nh, d)) * scale)


def test_qknorm_rope_position_zero_is_the_head_rmsnorm():
    g = np.random.default_rng(4)
    x = _heads(g, 5, 16)
    w = bits(1 + 0.1 * g.standard_normal(128))
    y = oracle.qknorm_rope(x, w, np.zeros(5, np.int64))
    n, _ = oracle.add_rmsnorm(x.reshape(-1, 128), None, w, 1e-6)
    np.testing.assert_allclose(y.reshape(-1, 128), n, rtol=1e-13, atol=1e-13)
    assert y.shape == (5, 16, 128)                      # shape kept (sec. 4 example)


def test_qknorm_rope_pairing_and_sign():
    # x = e_0 normalises to sqrt(d)*w_0*e_0; pair (0, 64) rotates by angle p.
    d = 128
    x = np.zeros((3, 1, d), np.float32)
    x[:, 0, 0] = 1.0
    w = bits(np.full(d, 1.0))
    pos = np.array([0, 1, 40959], np.int64)
    y = oracle.qknorm_rope(bits(x), w, pos)
    amp = 1.0 / math.sqrt(1.0 / d + 1e-6)
    for i, p in enumerate(pos):
        nz = np.flatnonzero(np.abs(y[i, 0]) > 1e-12)
        assert set(nz.tolist()) <= {0, 64}
        assert y[i, 0, 0] == pytest.approx(amp * math.cos(p), abs=1e-9)
        assert y[i, 0, 64] == pytest.approx(amp * math.sin(p), abs=1e-9)
    # a second-half input rotates the other way: y1 = -x2 sin, y2 = x2 cos
    x2 = np.zeros((1, 1, d), np.float32)
    x2[0, 0, 64] = 1.0
    y2 = oracle.qknorm_rope(bits(x2), w, np.array([1], np.int64))
    assert y2[0, 0, 0] == pytest.approx(-amp * math.sin(1.0), abs=1e-12)
    assert y2[0, 0, 64] == pytest.approx(amp * math.cos(1.0), abs=1e-12)


def test_qknorm_rope_preserves_pair_norms():
    g = np.random.default_rng(5)
    x = _heads(g, 7, 8)
    w = bits(1 + 0.1 * g.standard_normal(128))
    pos = g.integers(0, 40960, 7)
    y = oracle.qknorm_rope(x, w, pos)
    n = oracle.qknorm_rope(x, w, np.zeros(7, np.int64))
    np.testing.assert_allclose(y[..., :64] ** 2 + y[..., 64:] ** 2,
                               n[..., :64] ** 2 + n[..., 64:] ** 2, rtol=1e-12, atol=1e-12)


def test_rope_scores_depend_on_relative_position_only():
    g = np.random.default_rng(6)
    q = _heads(g, 1, 1)
    k = _heads(g, 1, 1)
    w = bits(np.ones(128))

    def score(m, n):
        qm = oracle.qknorm_rope(q, w, np.array([m], np.int64))
        kn = oracle.qknorm_rope(k, w, np.array([n], np.int64))
        return float(np.sum(qm * kn))

    s = score(10, 3)
    assert score(1010, 1003) == pytest.approx(s, rel=1e-9, abs=1e-9)
    assert score(30007, 30000) == pytest.approx(s, rel=1e-8, abs=1e-8)
    assert abs(score(10, 4) - s) > 1e-3


def test_rope_equals_rotate_half_form():
    # The transformers formulation ("同一个 Qwen3，两种写法", sec. 3.5):
    # y = n * [cos, cos] + rotate_half(n) * [sin, sin], rotate_half(n) = [-n2, n1].
    g = np.random.default_rng(7)
    x = _heads(g, 6, 4)
    w = bits(1 + 0.1 * g.standard_normal(128))
    pos = np.array([0, 1, 2, 100, 4095, 40959], np.int64)
    n = oracle.qknorm_rope(x, w, np.zeros(6, np.int64))
    table = oracle.rope_cos_sin(40960, 128, 1e6)[pos]
    cos_full = np.concatenate([table[:, :64], table[:, :64]], axis=1)[:, None, :]
    sin_full = np.concatenate([table[:, 64:], table[:, 64:]], axis=1)[:, None, :]
    rot = np.concatenate([-n[..., 64:], n[..., :64]], axis=-1)
    expect = n * cos_full + rot * sin_full
    np.testing.assert_allclose(oracle.qknorm_rope(x, w, pos), expect, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- attention
def _single_seq(q, k, v, scale, causal=True):
    T = q.shape[0]
    cu = np.array([0, T], np.int32)
    return oracle.attention_varlen(q, k, v, cu, cu, scale, causal)


def test_attention_page_worked_example():
    gold = read_golden("online_softmax_example.txt")
    s, vals = gold["scores"], gold["values"]
    d, L = 8, len(s)
    q = np.zeros((L, 1, d), np.float32)
    q[:, 0, 0] = 1.0
    k = np.zeros((L, 1, d), np.float32)
    k[:, 0, 0] = s
    v = np.zeros((L, 1, d), np.float32)
    v[:, 0, 0] = vals
    o = _single_seq(bits(q), bits(k), bits(v), scale=1.0)
    half_ulp = 0.5 * 10.0 ** -int(gold["decimals"][0])
    # The last query sees all four keys.
    assert abs(o[L - 1, 0, 0] - gold["output"][0]) <= half_ulp
    assert np.all(o[:, 0, 1:] == 0)
    # The page's intermediate quantities follow from the same scores.
    m = max(s)
    e = np.exp(np.array(s) - m)
    assert m == gold["row_max"][0]
    assert abs(e.sum() - gold["denominator"][0]) <= half_ulp
    np.testing.assert_allclose(e / e.sum(), gold["weights"], atol=half_ulp)
    assert abs(math.exp(3 - 5) - gold["rescale_factor"][0]) <= half_ulp
    eA = np.exp(np.array(s[:2]) - m)
    assert abs(eA.sum() - gold["blocked_denominator_after_A"][0]) <= half_ulp
    assert abs(eA @ np.array(vals[:2]) - gold["blocked_numerator_after_A"][0]) <= half_ulp
    # Causal rows: row 0 sees only key 0, row 1 keys 0..1.
    assert o[0, 0, 0] == pytest.approx(10.0, abs=1e-12)
    e01 = np.exp([1.0, 3.0])
    assert o[1, 0, 0] == pytest.approx((10 * e01[0] + 20 * e01[1]) / e01.sum(), rel=1e-14)


def test_attention_single_key_and_equal_scores():
    g = np.random.default_rng(8)
    d = 128
    q = _heads(g, 1, 2)
    k = _heads(g, 1, 1)
    v = _heads(g, 1, 1)
    o = _single_seq(q, k, v, 128 ** -0.5)
    for h in range(2):
        np.testing.assert_array_equal(o[0, h], F32(v[0, 0]))
    # q = 0: every score equal, output = mean of V (non-causal over 9 keys)
    q0 = np.zeros((9, 1, d), np.uint16)
    k9 = _heads(g, 9, 1)
    v9 = _heads(g, 9, 1)
    o9 = _single_seq(q0, k9, v9, 128 ** -0.5, causal=False)
    np.testing.assert_allclose(o9[:, 0], np.broadcast_to(F32(v9[:, 0]).astype(np.float64).mean(0), (9, d)),
                               rtol=1e-12, atol=1e-12)
    # causal with q = 0: row i is the mean of v_0..v_i; row 0 is v_0
    oc = _single_seq(q0, k9, v9, 128 ** -0.5, causal=True)
    vv = F32(v9[:, 0]).astype(np.float64)
    for i in range(9):
        np.testing.assert_allclose(oc[i, 0], vv[:i + 1].mean(0), rtol=1e-12, atol=1e-12)


def test_attention_scale_is_applied():
    # Two keys with raw dot products 0 and c*sqrt(d): with scale d^-1/2 the
    # weights are 1/(1+e^c) and e^c/(1+e^c).
    d, c = 128, 1.5
    q = np.zeros((2, 1, d), np.float32)
    q[1, 0, 0] = math.sqrt(d) / 4                 # exact in bf16 only for nice d
    k = np.zeros((2, 1, d), np.float32)
    k[1, 0, 0] = 4 * c
    v = np.zeros((2, 1, d), np.float32)
    v[0, 0, 1], v[1, 0, 1] = 1.0, 3.0
    qb = bits(q)
    qv = float(F32(qb)[1, 0, 0])
    o = _single_seq(qb, bits(k), bits(v), d ** -0.5)
    s1 = qv * 4 * c / math.sqrt(d)
    w1 = math.exp(s1) / (1 + math.exp(s1))
    assert o[1, 0, 1] == pytest.approx((1 - w1) * 1.0 + w1 * 3.0, rel=1e-14)
    assert abs(s1 - c) < 0.01


def test_attention_gqa_head_mapping():
    # Distinct constant V per kv head: q head h must return h // (Hq/Hkv).
    g = np.random.default_rng(9)
    T, Hq, Hkv, d = 6, 8, 2, 128
    q = _heads(g, T, Hq)
    k = _heads(g, T, Hkv)
    v = np.zeros((T, Hkv, d), np.float32)
    for kv in range(Hkv):
        v[:, kv, :] = kv + 1
    o = _single_seq(q, k, bits(v), d ** -0.5)
    for h in range(Hq):
        np.testing.assert_allclose(o[:, h, :], h // (Hq // Hkv) + 1, rtol=1e-14)


def test_varlen_mask_matches_page_picture():
    gold = read_golden("varlen_mask_abc.txt")
    lengths = [int(x) for x in gold["lengths"]]
    T = sum(lengths)
    mask = np.array([gold[f"row{i}"] for i in range(T)])
    d = 8
    q = np.zeros((T, 1, d), np.uint16)                 # equal scores everywhere
    k = bits(np.random.default_rng(10).standard_normal((T, 1, d)))
    v = np.zeros((T, 1, d), np.float32)
    v[np.arange(T), 0, np.arange(T)] = 1.0              # one-hot per key token
    cu = wl.cu_seqlens(lengths)
    o = oracle.attention_varlen(q, k, bits(v), cu, cu, 1.0, True)[:, 0, :T]
    np.testing.assert_allclose(o, mask / mask.sum(1, keepdims=True), rtol=1e-14, atol=0)


def test_cu_seqlens_examples():
    gold = read_golden("cu_seqlens_examples.txt")
    for lens, cu in zip(gold["lengths"], gold["cu_seqlens"]):
        assert wl.cu_seqlens([int(x) for x in lens]).tolist() == [int(x) for x in cu]


def test_attention_two_keys_brute_force():
    g = np.random.default_rng(11)
    d = 4
    q = bits(g.standard_normal((2, 1, d)))
    k = bits(g.standard_normal((2, 1, d)))
    v = bits(g.standard_normal((2, 1, d)))
    o = _single_seq(q, k, v, 0.5)
    qf, kf, vf = (F32(a)[:, 0].astype(np.float64) for a in (q, k, v))
    s0 = 0.5 * sum(qf[1, i] * kf[0, i] for i in range(d))
    s1 = 0.5 * sum(qf[1, i] * kf[1, i] for i in range(d))
    e0, e1 = math.exp(s0), math.exp(s1)
    for i in range(d):
        assert o[1, 0, i] == pytest.approx((e0 * vf[0, i] + e1 * vf[1, i]) / (e0 + e1), rel=1e-13)


# ------------------------------------------------------------ paged decode
@pytest.mark.parametrize("hq,hkv", [(4, 4), (4, 2), (8, 2)])
def test_paged_equals_contiguous_with_shuffled_blocks(hq, hkv):
    g = np.random.default_rng(12 + hq + hkv)
    d, bs = 16, 4
    ctx = np.array([1, bs - 1, bs, bs + 1, 3 * bs + 2], np.int32)
    B = ctx.size
    need = [math.ceil(int(c) / bs) for c in ctx]
    nb = sum(need) + 3
    perm = g.permutation(nb).astype(np.int32)
    bt = wl.carve_block_tables(perm, ctx, block_size=bs)
    kc = bits(g.standard_normal((nb, bs, hkv, d)))
    vc = bits(g.standard_normal((nb, bs, hkv, d)))
    q = bits(g.standard_normal((B, hq, d)))
    out = oracle.paged_decode(q, kc, vc, bt, ctx, d ** -0.5)
    # Contiguous reference: gather each sequence's rows in logical order by
    # walking its blocks, pack them, and run the varlen path with one query
    # per sequence aligned to the last key.
    ks, vs = [], []
    for b in range(B):
        for j in range(int(ctx[b])):
            ks.append(kc[bt[b, j // bs], j % bs])
            vs.append(vc[bt[b, j // bs], j % bs])
    kk, vv = np.stack(ks), np.stack(vs)
    cu_q = wl.cu_seqlens([1] * B)
    cu_k = wl.cu_seqlens(ctx)
    ref = oracle.attention_varlen(q, kk, vv, cu_q, cu_k, d ** -0.5, True)
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)
    # A single cached token returns its V.
    np.testing.assert_array_equal(out[0, 0], F32(vc[bt[0, 0], 0, 0]))


def test_paged_decode_empty_context_is_zero_and_pairs_subset():
    g = np.random.default_rng(13)
    d, bs, hkv, hq = 8, 4, 1, 2
    kc = bits(g.standard_normal((3, bs, hkv, d)))
    vc = bits(g.standard_normal((3, bs, hkv, d)))
    bt = np.array([[2, 0], [1, -1]], np.int32)
    ctx = np.array([0, 3], np.int32)
    q = bits(g.standard_normal((2, hq, d)))
    full = oracle.paged_decode(q, kc, vc, bt, ctx, 0.3)
    assert np.all(full[0] == 0)
    sub = oracle.paged_decode(q, kc, vc, bt, ctx, 0.3, pairs=np.array([[1, 1], [1, 0]]))
    np.testing.assert_array_equal(sub, full[1, ::-1])
    with pytest.raises(ValueError):
        oracle.paged_decode(q, kc, vc, np.array([[2, 0], [5, -1]], np.int32), ctx, 0.3)


# ---------------------------------------------- prefill over the paged cache
@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 2)])
def test_paged_prefill_equals_contiguous_bottom_right_causal(hq, hkv):
    # Prefix lengths and new-token counts per sequence; the cache holds all
    # prefix + new keys in shuffled blocks of 4 tokens.
    g = np.random.default_rng(40 + hq)
    d, bs = 16, 4
    prefix = np.array([0, 3, 8, 5])
    new = np.array([5, 1, 4, 7])
    lk = prefix + new
    B = lk.size
    nb = int(sum(math.ceil(int(x) / bs) for x in lk)) + 2
    bt = wl.carve_block_tables(g.permutation(nb).astype(np.int32), lk, block_size=bs)
    kc = bits(g.standard_normal((nb, bs, hkv, d)))
    vc = bits(g.standard_normal((nb, bs, hkv, d)))
    q = bits(g.standard_normal((int(new.sum()), hq, d)))
    cu_q, cu_k = wl.cu_seqlens(new), wl.cu_seqlens(lk)
    out = oracle.attention_paged_prefill(q, kc, vc, bt, cu_q, cu_k, d ** -0.5)
    # contiguous reference: walk each sequence's blocks in logical order
    ks, vs = [], []
    for b in range(B):
        for j in range(int(lk[b])):
            ks.append(kc[bt[b, j // bs], j % bs])
            vs.append(vc[bt[b, j // bs], j % bs])
    ref = oracle.attention_varlen(q, np.stack(ks), np.stack(vs), cu_q, cu_k, d ** -0.5, True)
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)


def test_paged_prefill_single_query_is_paged_decode_and_prefix_mean():
    g = np.random.default_rng(44)
    d, bs, hq, hkv = 8, 4, 4, 2
    lk = np.array([6, 9])
    nb = 6
    bt = wl.carve_block_tables(g.permutation(nb).astype(np.int32), lk, block_size=bs)
    kc = bits(g.standard_normal((nb, bs, hkv, d)))
    vc = bits(g.standard_normal((nb, bs, hkv, d)))
    q = bits(g.standard_normal((2, hq, d)))
    one = wl.cu_seqlens([1, 1])
    pre = oracle.attention_paged_prefill(q, kc, vc, bt, one, wl.cu_seqlens(lk), 0.3)
    dec = oracle.paged_decode(q, kc, vc, bt, lk.astype(np.int32), 0.3)
    np.testing.assert_allclose(pre, dec, rtol=1e-13, atol=1e-13)
    # q = 0: query i of a sequence with prefix P averages keys 0 .. P + i
    q0 = np.zeros((3, hq, d), np.uint16)
    out = oracle.attention_paged_prefill(q0, kc, vc, bt[:1], wl.cu_seqlens([3]),
                                         wl.cu_seqlens([6]), 0.3)
    for i in range(3):
        rows = [vc[bt[0, j // bs], j % bs] for j in range(3 + i + 1)]
        mean = F32(np.stack(rows)).astype(np.float64).mean(0)
        for h in range(hq):
            np.testing.assert_allclose(out[i, h], mean[h // (hq // hkv)], rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- SiluAndMul
def _bits(values):
    return wl.f32_to_bf16_bits(np.asarray(values, dtype=np.float32))


def test_silu_and_mul_gate_first_and_limits():
    # "3.3 Model skeleton and core operators", sec. 4: the first half of the
    # merged projection is the gate, the second the up projection.  A large
    # positive gate passes up through (silu(g) -> g), a large negative one
    # closes it (silu(g) -> 0); swapping the halves changes both results.
    x = _bits([[30.0, 1.0], [-30.0, 5.0], [0.0, 7.0], [1.0, 0.0]])
    out = oracle.silu_and_mul(x)
    assert out.shape == (4, 1)
    assert 0 < 30.0 - out[0, 0] < 30 * math.exp(-30)      # 30 * sigmoid(30) * 1
    assert 0 < -out[1, 0] < 5 * 30 * math.exp(-30)        # gate closed
    assert out[2, 0] == 0.0 and out[3, 0] == 0.0  # silu(0) = 0; up = 0


def test_silu_and_mul_odd_even_identities():
    # silu(g) - silu(-g) = g   and   silu(g) + silu(-g) = g * tanh(g / 2),
    # the second against numpy's tanh: a sign slip in the exponent flips it.
    g = wl.bf16_bits_to_f32(_bits(np.linspace(-9.0, 9.0, 37))).astype(np.float64)
    up = np.ones_like(g)
    pos = oracle.silu_and_mul(_bits(np.stack([g, up], 1)))[:, 0]
    neg = oracle.silu_and_mul(_bits(np.stack([-g, up], 1)))[:, 0]
    assert np.allclose(pos - neg, g, rtol=0, atol=1e-14)
    assert np.allclose(pos + neg, g * np.tanh(g / 2), rtol=0, atol=1e-14)


def test_silu_and_mul_matches_torch_fp64_and_page_toy_shape():
    # The toy MLP of the page: [5, 2I/TP] = [5, 16] in, [5, 8] out.  Values
    # against torch's own silu in fp64 on the CPU (an independent routine).
    torch = pytest.importorskip("torch")
    x = wl.normal_bf16(41, "pin.swiglu", (5, 16), 0.0, 2.0)
    out = oracle.silu_and_mul(x)
    assert out.shape == (5, 8)
    xf = torch.from_numpy(wl.bf16_bits_to_f32(x).astype(np.float64))
    ref = torch.nn.functional.silu(xf[:, :8]) * xf[:, 8:]
    assert np.allclose(out, ref.numpy(), rtol=1e-14, atol=1e-15)
    # up is a plain multiplier
    x2 = x.copy()
    x2[:, 8:] = _bits(2.0 * wl.bf16_bits_to_f32(x[:, 8:]))
    assert np.allclose(oracle.silu_and_mul(x2), 2.0 * out, rtol=1e-15, atol=0)
