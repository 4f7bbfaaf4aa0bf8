"""GPU parity of the tcgen05 varlen causal prefill against the fp64 oracle.
The first case launches a single CTA; later ones span several 128-row tiles
with ragged tails, GQA groups, strided q/k/v views and the full Qwen3-8B
batch (sampled rows)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import check_close, dev, dev_i32, err_counter, host

pytestmark = pytest.mark.gpu

import paged_kv_attention_kvcache_gb300 as nv  # noqa: E402

SCALE = 128 ** -0.5


def run_prefill(qkv_bits, lengths, hq, hkv):
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
                              err_count=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "pipeline failure flagged"
    return host(o)


def split_qkv(qkv_bits, hq, hkv):
    T = qkv_bits.shape[0]
    Q, D = hq * 128, hkv * 128
    return (qkv_bits[:, :Q].reshape(T, hq, 128), qkv_bits[:, Q:Q + D].reshape(T, hkv, 128),
            qkv_bits[:, Q + D:].reshape(T, hkv, 128))


def case(seed, lengths, hq, hkv, rows=None):
    T = int(sum(lengths))
    qkv = wl.normal_bf16(seed, "prefill.qkv", (T, (hq + 2 * hkv) * 128))
    got = run_prefill(qkv, lengths, hq, hkv)
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


@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 2), (8, 2)])
def test_prefill_ragged_packed_sequences(hq, hkv):
    case(510 + hq, [1, 127, 128, 129, 300, 37, 2], hq, hkv)


def test_prefill_small_layer_shape():
    pre, _ = wl.config1()
    s = pre.shape
    got = run_prefill(pre.qkv, pre.lengths, s.hq, s.hkv)
    q, k, v = split_qkv(pre.qkv, s.hq, s.hkv)
    ref = oracle.attention_varlen(q, k, v, pre.cu_seqlens, pre.cu_seqlens, SCALE, True)
    check_close(got, ref, "prefill cfg1")


def test_prefill_qwen3_8b_batch_full_size_sampled():
    batch = wl.config4()
    s = batch.shape
    g = np.random.default_rng(520)
    T = batch.qkv.shape[0]
    cu = batch.cu_seqlens
    # first and last rows of every sequence, plus random rows, random heads
    ends = np.concatenate([cu[:-1], cu[1:] - 1])
    toks = np.concatenate([ends, g.integers(0, T, 600)])
    rows = np.stack([toks, g.integers(0, s.hq, toks.size)], axis=1).astype(np.int64)
    got = run_prefill(batch.qkv, batch.lengths, s.hq, s.hkv)
    q, k, v = split_qkv(batch.qkv, s.hq, s.hkv)
    ref = oracle.attention_varlen(q, k, v, cu, cu, SCALE, True, rows=rows)
    check_close(got[rows[:, 0], rows[:, 1]], ref, "prefill cfg4 sampled")
