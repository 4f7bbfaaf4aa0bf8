"""CUDA-graph decode at padded batch sizes ("3.3 Model skeleton and core
operators", sec. 7.1: graph replays pad the decode batch to a fixed size and
padding tokens carry slot -1; "nano-vllm code walkthrough", CUDA graph: one
graph per batch bucket, static addresses).  The whole decode layer -- add-
RMSNorm, QK-Norm + RoPE, store_kvcache, split-KV paged decode -- is captured
once per bucket and replayed with new inputs copied into the static buffers,
either with the separate rotation and store kernels or with the fused
QK-Norm + RoPE + store pass.  Padded rows have context length 0 and slot -1: their output must be zero and
they must never write the cache."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import check_cache_rows, check_close, dev, host, rope_table

pytestmark = pytest.mark.gpu

import paged_kv_attention_kvcache_gb300 as nv  # noqa: E402

SCALE = 128 ** -0.5
SHAPE = wl.QWEN3_06B


def _step_inputs(seed, bucket, n_real, ctx, bt, pos_shift=0):
    """Host inputs of one decode step, padded to `bucket` rows."""
    s = SHAPE
    g = np.random.default_rng(seed)
    qkv = np.zeros((bucket, s.qkv_width), np.uint16)
    qkv[:n_real] = wl.f32_to_bf16_bits(g.standard_normal((n_real, s.qkv_width)).astype(np.float32))
    x = np.zeros((bucket, s.hidden), np.uint16)
    r = np.zeros((bucket, s.hidden), np.uint16)
    x[:n_real] = wl.f32_to_bf16_bits(g.standard_normal((n_real, s.hidden)).astype(np.float32))
    r[:n_real] = wl.f32_to_bf16_bits(g.standard_normal((n_real, s.hidden)).astype(np.float32))
    c = np.zeros(bucket, np.int32)
    c[:n_real] = ctx[:n_real] + pos_shift
    pos = np.maximum(c.astype(np.int64) - 1, 0)
    slots = np.full(bucket, -1, np.int32)
    slots[:n_real] = wl.slots_for_positions(bt, np.arange(n_real), pos[:n_real])
    return dict(qkv=qkv, x=x, r=r, ctx=c, pos=pos, slots=slots)


# Forced 256-key splits exercise the split + merge pair inside the graph; the
# automatic split leaves these short contexts unsplit at buckets 64 and 512
# (one decode kernel) and takes 1024-key splits at bucket 8.
@pytest.mark.parametrize("bucket,n_real,fused,split", [
    (1, 1, False, 256), (8, 5, False, 256), (64, 61, False, 256), (8, 5, True, 256),
    (512, 509, True, 256), (8, 5, False, 0), (64, 61, False, 0), (512, 509, True, 0)])
def test_decode_layer_graph_replay_with_padding(bucket, n_real, fused, split):
    s = SHAPE
    Q, D = s.q_size, s.kv_size
    g = np.random.default_rng(700 + bucket)
    ctx0 = g.integers(200, 1500 if bucket <= 64 else 600, bucket).astype(np.int32)
    cap = ctx0 + 4                                  # room for the replayed steps
    nb = int(sum(math.ceil(int(c) / 256) for c in cap)) + 2
    bt_full = wl.carve_block_tables(g.permutation(nb).astype(np.int32), cap)
    bt = bt_full.copy()
    bt[n_real:] = -1                                # padded rows own no blocks
    pool = wl.make_pool(700 + bucket, nb, bt_full[bt_full >= 0], s.hkv)
    gamma = wl.normal_bf16(701, "g.gamma", (s.hidden,), 1.0, 0.1)
    qn = wl.normal_bf16(701, "g.qn", (128,), 1.0, 0.1)
    kn = wl.normal_bf16(701, "g.kn", (128,), 1.0, 0.1)

    # static device buffers
    table = rope_table()
    kc, vc = dev(pool.k), dev(pool.v)
    d_gamma, d_qn, d_kn = dev(gamma), dev(qn), dev(kn)
    x = torch.zeros(bucket, s.hidden, dtype=torch.bfloat16, device="cuda")
    r = torch.zeros_like(x)
    y = torch.zeros_like(x)
    qkv = torch.zeros(bucket, s.qkv_width, dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(bucket, dtype=torch.int64, device="cuda")
    slots = torch.zeros(bucket, dtype=torch.int32, device="cuda")
    ctx = torch.zeros(bucket, dtype=torch.int32, device="cuda")
    d_bt = torch.from_numpy(bt).cuda()
    o = torch.zeros(bucket, s.hq, 128, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws_b = nv.nv_decode_attn_workspace_size(bucket, s.hq, s.hkv, 128, bt.shape[1], 256, split)
    if split == 0:                                  # what the automatic split chose here
        assert (ws_b > 0) == (bucket == 8)
    ws = torch.empty(max(1, ws_b // 4), dtype=torch.float32, device="cuda")
    q = qkv[:, :Q].view(bucket, s.hq, 128)
    k = qkv[:, Q:Q + D].view(bucket, s.hkv, 128)
    v = qkv[:, Q + D:].view(bucket, s.hkv, 128)

    def layer():
        nv.nv_add_rmsnorm(x, r, d_gamma, y, r, eps=wl.RMS_EPS)
        if fused:
            nv.nv_qknorm_rope_store(q, k, v, d_qn, d_kn, table, pos, kc, vc, slots,
                                    eps=wl.RMS_EPS, err_count=err)
        else:
            nv.nv_qknorm_rope(q, k, d_qn, d_kn, table, pos, eps=wl.RMS_EPS, err_count=err)
            nv.nv_store_kvcache(k, v, kc, vc, slots, err)
        nv.nv_decode_attn_paged(q, kc, vc, d_bt, ctx, o, SCALE, workspace=ws,
                                kv_split_tokens=split, err_count=err)

    def load(inp):
        x.copy_(dev(inp["x"]))
        r.copy_(dev(inp["r"]))
        qkv.copy_(dev(inp["qkv"]))
        pos.copy_(torch.from_numpy(inp["pos"]))
        slots.copy_(torch.from_numpy(inp["slots"]))
        ctx.copy_(torch.from_numpy(inp["ctx"]))

    # The oracle's cache evolves from the same pool, by its own rounded rows only.
    ref_k, ref_v = pool.k.copy(), pool.v.copy()

    def oracle_store(inp):
        q_rot = oracle.qknorm_rope(inp["qkv"][:n_real, :Q].reshape(n_real, s.hq, 128), qn,
                                   inp["pos"][:n_real])
        k_rot = oracle.qknorm_rope(inp["qkv"][:n_real, Q:Q + D].reshape(n_real, s.hkv, 128), kn,
                                   inp["pos"][:n_real])
        qb, kb = oracle.round_to_bf16(q_rot), oracle.round_to_bf16(k_rot)
        vb = inp["qkv"][:n_real, Q + D:].reshape(n_real, s.hkv, 128)
        assert oracle.store_kvcache(kb, vb, ref_k, ref_v, inp["slots"][:n_real]) == 0
        return qb

    # warm up on a side stream (first calls set kernel attributes), then capture
    warm = _step_inputs(710, bucket, n_real, ctx0, bt_full)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        load(warm)
        layer()
    oracle_store(warm)
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer()

    for step in range(3):
        inp = _step_inputs(720 + step, bucket, n_real, ctx0, bt_full, pos_shift=1 + step)
        load(inp)
        graph.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        # oracle chain for the real rows
        y_ref, _ = oracle.add_rmsnorm(inp["x"][:n_real], inp["r"][:n_real], gamma, wl.RMS_EPS)
        check_close(host(y)[:n_real], y_ref, f"graph step {step} norm")
        qb = oracle_store(inp)
        o_ref = oracle.paged_decode(qb, ref_k, ref_v, bt_full[:n_real], inp["ctx"][:n_real], SCALE)
        got = host(o)
        check_close(got[:n_real], o_ref, f"graph step {step} decode")
        assert np.all(got[n_real:] == 0), "padded rows must be zero"
        # padding wrote nothing: the cache equals the oracle's (K up to one ulp
        # where the two roundings of the same value differ)
        gk, gv = host(kc), host(vc)
        assert np.array_equal(gv, ref_v)
        check_cache_rows(gk, ref_k, f"graph step {step} k cache", max_mismatch_frac=1e-3)
