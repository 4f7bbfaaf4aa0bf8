"""GPU parity of the tcgen05 varlen causal prefill against the fp64 oracle.
The first case launches a single CTA; later ones span several 128-row tiles
with ragged tails, GQA groups, strided q/k/v views and the full Qwen3-8B
batch, every output element compared."""
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


def sched_counter(dynamic=True):
    """The work counter for the dynamic schedule, deliberately left dirty: the
    call must clear it itself.  None selects the round-robin schedule."""
    return torch.full((1,), 987654, dtype=torch.int32, device="cuda") if dynamic else None


def run_prefill(qkv_bits, lengths, hq, hkv, dynamic=True):
    """Prefill over views of a packed qkv buffer [T, (hq + 2 hkv) * 128]."""
    T = qkv_bits.shape[0]
    Q, D = hq * 128, hkv * 128
    qkv = dev(qkv_bits)
    q = qkv[:, :Q].view(T, hq, 128)
    k = qkv[:, Q:Q + D].view(T, hkv, 128)
    v = qkv[:, Q + D:].view(T, hkv, 128)
    cu = dev_i32(wl.cu_seqlens(lengths))
    o = torch.empty(T, hq, 128, dtype=torch.bfloat16, device="cuda")
    err = err_counter()
    nv.nv_prefill_attn_varlen(q, k, v, o, cu, cu, int(max(lengths)), int(max(lengths)), SCALE,
                              err_count=err, sched_counter=sched_counter(dynamic))
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "pipeline failure flagged"
    return host(o)


def split_qkv(qkv_bits, hq, hkv):
    T = qkv_bits.shape[0]
    Q, D = hq * 128, hkv * 128
    return (qkv_bits[:, :Q].reshape(T, hq, 128), qkv_bits[:, Q:Q + D].reshape(T, hkv, 128),
            qkv_bits[:, Q + D:].reshape(T, hkv, 128))


def case(seed, lengths, hq, hkv, rows=None, dynamic=True):
    T = int(sum(lengths))
    qkv = wl.normal_bf16(seed, "prefill.qkv", (T, (hq + 2 * hkv) * 128))
    got = run_prefill(qkv, lengths, hq, hkv, dynamic)
    q, k, v = split_qkv(qkv, hq, hkv)
    cu = wl.cu_seqlens(lengths)
    ref = oracle.attention_varlen(q, k, v, cu, cu, SCALE, True, rows=rows)
    if rows is None:
        return check_close(got, ref, f"prefill {lengths} {hq}/{hkv}")
    return check_close(got[rows[:, 0], rows[:, 1]], ref, f"prefill rows {hq}/{hkv}")


def test_prefill_single_tile_single_head():
    case(501, [5], 1, 1)


def test_prefill_exact_tiles():
    case(502, [128], 1, 1)
    case(503, [256], 2, 1)


# Work items pair two query heads of a kv head at the same rows when the
# group size is even (4/2, 8/2, 8/1, 16/1) and two adjacent row tiles of one
# head when it is odd (2/2, 6/2, 5/1); both shapes are covered, up to the
# group of 16 the decode supports.
@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 2), (6, 2), (8, 2), (8, 1), (16, 1), (5, 1)])
@pytest.mark.parametrize("dynamic", [True, False])
def test_prefill_ragged_packed_sequences(hq, hkv, dynamic):
    case(510 + hq + 100 * (hkv == 1), [1, 127, 128, 129, 300, 37, 2], hq, hkv, dynamic=dynamic)


def test_prefill_sequences_without_query_rows():
    # A sequence with no new rows (cu_seqlens repeating a value, as when a
    # sequence adds nothing in this step) brings no work item; its neighbours
    # must still match the oracle, under both schedules and over the paged
    # cache (where such a sequence may still own cached keys).
    for dynamic in (True, False):
        case(560, [0, 37, 0, 0, 300, 0, 129], 8, 2, dynamic=dynamic)
    got, ref = _paged_case(561, prefix=[300, 0, 512, 40], new=[0, 37, 0, 129], hq=8, hkv=2)
    check_close(got, ref, "paged prefill next to sequences without new rows")


def test_prefill_more_items_than_ctas_both_schedules_agree():
    # 40 sequences x 8 heads of up to 1000 tokens: several items per CTA under
    # either schedule; both must give the oracle's result on every row.
    g = np.random.default_rng(515)
    lengths = g.integers(1, 1000, 40)
    T = int(lengths.sum())
    qkv = wl.normal_bf16(515, "prefill.qkv", (T, (8 + 2 * 2) * 128))
    q, k, v = split_qkv(qkv, 8, 2)
    cu = wl.cu_seqlens(lengths)
    ref = oracle.attention_varlen(q, k, v, cu, cu, SCALE, True)
    for dynamic in (True, False):
        got = run_prefill(qkv, lengths, 8, 2, dynamic)
        check_close(got, ref, f"prefill many items dynamic={dynamic}")


def test_prefill_small_layer_shape():
    pre, _ = wl.config1()
    s = pre.shape
    got = run_prefill(pre.qkv, pre.lengths, s.hq, s.hkv)
    q, k, v = split_qkv(pre.qkv, s.hq, s.hkv)
    ref = oracle.attention_varlen(q, k, v, pre.cu_seqlens, pre.cu_seqlens, SCALE, True)
    check_close(got, ref, "prefill cfg1")


def test_prefill_qwen3_8b_batch_full_size():
    # The measured prefill batch (16 sequences, 33,109 tokens, Qwen3-8B heads)
    # in the launch the bench times; every (token, head) row compared.
    batch = wl.config4()
    s = batch.shape
    cu = batch.cu_seqlens
    got = run_prefill(batch.qkv, batch.lengths, s.hq, s.hkv)
    q, k, v = split_qkv(batch.qkv, s.hq, s.hkv)
    ref = oracle.attention_varlen(q, k, v, cu, cu, SCALE, True)
    check_close(got, ref, "prefill cfg4 (16 seqs, 33k tokens, 32/8 heads)")


def test_prefill_neighbouring_sequence_nan_rows_do_not_leak():
    # Packed sequences share 128-row key tiles: the last tile of a sequence
    # reads the next sequence's rows, masked.  With NaN in every K and V row
    # of the middle sequence, the other sequences' outputs must still be the
    # oracle's (their masked keys carry probability 0, and 0 * NaN is not 0,
    # so those V rows must be cleared before use).  Both schedules.
    hq, hkv = 8, 2
    lengths = np.array([100, 70, 300, 1, 129])
    T = int(lengths.sum())
    qkv = wl.normal_bf16(535, "prefill.nan", (T, (hq + 2 * hkv) * 128))
    cu = wl.cu_seqlens(lengths)
    qkv[cu[1]:cu[2], hq * 128:] = 0x7FC0          # K and V rows of sequence 1: NaN
    q, k, v = split_qkv(qkv, hq, hkv)
    keep = np.r_[cu[0]:cu[1], cu[2]:cu[5]]
    for dynamic in (True, False):
        got = run_prefill(qkv, lengths, hq, hkv, dynamic)
        ref = oracle.attention_varlen(q, k, v, cu, cu, SCALE, True)
        check_close(got[keep], ref[keep], f"prefill next to NaN rows dynamic={dynamic}")


# ------------------------------------------- keys beyond the queries (prefix)
def test_prefill_contiguous_keys_with_prefix():
    # Each sequence's keys are a prefix followed by its Lq new tokens; query i
    # sees keys <= Lk - Lq + i (causality aligned to the last key).
    hq, hkv = 8, 2
    new = np.array([5, 130, 1, 257])
    prefix = np.array([0, 100, 300, 129])
    lk = new + prefix
    g = np.random.default_rng(530)
    q = wl.f32_to_bf16_bits(g.standard_normal((int(new.sum()), hq, 128)).astype(np.float32))
    k = wl.f32_to_bf16_bits(g.standard_normal((int(lk.sum()), hkv, 128)).astype(np.float32))
    v = wl.f32_to_bf16_bits(g.standard_normal((int(lk.sum()), hkv, 128)).astype(np.float32))
    cu_q, cu_k = wl.cu_seqlens(new), wl.cu_seqlens(lk)
    o = torch.empty(int(new.sum()), hq, 128, dtype=torch.bfloat16, device="cuda")
    err = err_counter()
    nv.nv_prefill_attn_varlen(dev(q), dev(k), dev(v), o, dev_i32(cu_q), dev_i32(cu_k),
                              int(new.max()), int(lk.max()), SCALE, err_count=err,
                              sched_counter=sched_counter())
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.attention_varlen(q, k, v, cu_q, cu_k, SCALE, True)
    check_close(host(o), ref, "prefill with contiguous prefix")


def _paged_case(seed, prefix, new, hq, hkv, nan_tail=True, rows=None, spare=3, dynamic=True,
                bs=wl.BLOCK_SIZE):
    g = np.random.default_rng(seed)
    prefix, new = np.asarray(prefix), np.asarray(new)
    lk = prefix + new
    nb = int(sum(math.ceil(int(x) / bs) for x in lk)) + spare
    bt = wl.carve_block_tables(g.permutation(nb).astype(np.int32), lk, block_size=bs)
    kc = wl.f32_to_bf16_bits(g.standard_normal((nb, bs, hkv, 128)).astype(np.float32))
    vc = wl.f32_to_bf16_bits(g.standard_normal((nb, bs, hkv, 128)).astype(np.float32))
    if nan_tail:
        # rows past each sequence's last key hold NaN bits
        for b, L in enumerate(lk):
            last = bt[b, (int(L) - 1) // bs]
            kc[last, int(L) % bs if L % bs else bs:] = 0x7FC0
            vc[last, int(L) % bs if L % bs else bs:] = 0x7FC0
    q = wl.f32_to_bf16_bits(g.standard_normal((int(new.sum()), hq, 128)).astype(np.float32))
    cu_q, cu_k = wl.cu_seqlens(new), wl.cu_seqlens(lk)
    o = torch.empty(int(new.sum()), hq, 128, dtype=torch.bfloat16, device="cuda")
    err = err_counter()
    nv.nv_prefill_attn_paged(dev(q), dev(kc), dev(vc), dev_i32(bt), o, dev_i32(cu_q),
                             dev_i32(cu_k), int(new.max()), SCALE, err_count=err,
                             sched_counter=sched_counter(dynamic))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.attention_paged_prefill(q, kc, vc, bt, cu_q, cu_k, SCALE, rows=rows)
    got = host(o)
    if rows is not None:
        got = got[rows[:, 0], rows[:, 1]]
    return got, ref


@pytest.mark.parametrize("hq,hkv", [(2, 2), (6, 2), (8, 2), (32, 8)])
def test_prefill_paged_prefix_hit(hq, hkv):
    got, ref = _paged_case(540 + hq, prefix=[0, 37, 256, 300, 511, 1000],
                           new=[5, 1, 128, 200, 129, 300], hq=hq, hkv=hkv)
    check_close(got, ref, f"paged prefill {hq}/{hkv}")


def test_prefill_paged_equals_contiguous_when_no_prefix():
    # With no cached prefix the paged path must agree with the contiguous one.
    got, ref = _paged_case(550, prefix=[0, 0, 0], new=[37, 300, 128], hq=16, hkv=8)
    check_close(got, ref, "paged prefill, no prefix")


def test_prefill_paged_round_robin_schedule():
    got, ref = _paged_case(551, prefix=[0, 37, 256, 300, 511, 1000],
                           new=[5, 1, 128, 200, 129, 300], hq=8, hkv=2, dynamic=False)
    check_close(got, ref, "paged prefill, round-robin")


def test_prefill_paged_chunked_qwen3_8b():
    # Chunked prefill at Qwen3-8B heads: 8 sequences with U[0, 4096] cached
    # tokens and a U[128, 1024] chunk each; every row compared.
    g = np.random.default_rng(560)
    prefix = g.integers(0, 4096, 8, endpoint=True)
    new = g.integers(128, 1024, 8, endpoint=True)
    got, ref = _paged_case(561, prefix, new, 32, 8)
    check_close(got, ref, "chunked prefill 8b")


def test_prefill_longest_context_single_sequence_sampled():
    # One sequence of the longest context the model takes (40960 tokens) at
    # Qwen3-8B heads: 160 query-tile pairs, the heaviest item 320 key tiles.
    L, hq, hkv = wl.MAX_POSITION, 32, 8
    qkv = wl.normal_bf16(570, "prefill.max", (L, (hq + 2 * hkv) * 128))
    g = np.random.default_rng(571)
    toks = np.concatenate([[0, 127, 128, 255, 256, L - 129, L - 128, L - 1], g.integers(0, L, 56)])
    rows = np.stack([toks, g.integers(0, hq, toks.size)], axis=1).astype(np.int64)
    got = run_prefill(qkv, [L], hq, hkv)
    q, k, v = split_qkv(qkv, hq, hkv)
    cu = wl.cu_seqlens([L])
    ref = oracle.attention_varlen(q, k, v, cu, cu, SCALE, True, rows=rows)
    check_close(got[rows[:, 0], rows[:, 1]], ref, "prefill 40960 sampled")


@pytest.mark.parametrize("bs", [128, 512])
def test_prefill_paged_other_block_sizes(bs):
    # Block sizes other than 256 (any multiple of the 128-key tile): tiles
    # then start at every block (128) or every fourth tile starts one (512).
    got, ref = _paged_case(580 + bs, prefix=[0, 37, 256, 300, 640], new=[5, 130, 128, 200, 300],
                           hq=8, hkv=2, bs=bs)
    check_close(got, ref, f"paged prefill bs={bs}")


def test_prefill_paged_prefix_workload_full_size():
    # The measured prefix-hit workload at full size, in the launch the bench
    # times (dynamic queue): 16 sequences, block-aligned cached prefixes of
    # 256..4096 tokens and 128..1024 new ones; every (token, head) row
    # compared.  The contiguous kernel over the same keys gathered from the
    # pool must agree with it bit for bit.
    pre = wl.config_prefix()
    s = pre.shape
    Tq = int(pre.new.sum())
    cu_q, cu_k = pre.cu_seqlens_q, pre.cu_seqlens_k
    o = torch.empty(Tq, s.hq, 128, dtype=torch.bfloat16, device="cuda")
    err = err_counter()
    nv.nv_prefill_attn_paged(dev(pre.q), dev(pre.pool.k), dev(pre.pool.v),
                             dev_i32(pre.block_tables), o, dev_i32(cu_q), dev_i32(cu_k),
                             int(pre.new.max()), SCALE, err_count=err,
                             sched_counter=sched_counter(True))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.attention_paged_prefill(pre.q, pre.pool.k, pre.pool.v, pre.block_tables,
                                         cu_q, cu_k, SCALE)
    got = host(o)
    check_close(got, ref, "prefix-hit workload (16 seqs, 8.8k new over 46k cached)")

    kk, vv = wl.gather_paged(pre.pool, pre.block_tables, pre.prefix + pre.new)
    o2 = torch.empty_like(o)
    nv.nv_prefill_attn_varlen(dev(pre.q), dev(kk), dev(vv), o2, dev_i32(cu_q), dev_i32(cu_k),
                              int(pre.new.max()), int((pre.prefix + pre.new).max()), SCALE,
                              sched_counter=sched_counter(True))
    torch.cuda.synchronize()
    assert np.array_equal(host(o2), got), "paged and contiguous keys give the same bits"
