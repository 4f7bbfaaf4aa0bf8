"""Every entry point can be captured into a CUDA graph ("3.3 Model skeleton
and core operators", sec. 7.1 and "nano-vllm code walkthrough", CUDA graph:
the pages replay captured graphs; the ABI only enqueues work on the given
stream).  The calls not covered by the decode-layer graph test are captured
here -- add-RMSNorm, the fused rope+store pass, the varlen prefill (whose work
counter is cleared by a memset node), the paged prefill, SiluAndMul and the
no-alloc decode -- replayed twice, and must give the eager run's bits exactly
(every kernel is deterministic, the dynamic work queue included: each item is
computed by one CTA whichever it is)."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import check_close, dev, dev_i32, dev_i64, host, rope_table

pytestmark = pytest.mark.gpu

import paged_kv_attention_kvcache_gb300 as nv  # noqa: E402

SCALE = 128 ** -0.5


def test_prefill_side_entry_points_replay_from_a_graph():
    s = wl.QWEN3_06B
    g = np.random.default_rng(900)
    lengths = np.array([37, 300, 129, 1])
    T = int(lengths.sum())
    Q, D = s.q_size, s.kv_size
    nb = int(sum(math.ceil(int(L) / wl.BLOCK_SIZE) for L in lengths)) + 2
    bt = wl.carve_block_tables(g.permutation(nb).astype(np.int32), lengths)
    seq = np.repeat(np.arange(lengths.size), lengths)
    pos = np.concatenate([np.arange(int(L)) for L in lengths]).astype(np.int64)
    slots = wl.slots_for_positions(bt, seq, pos).astype(np.int32)
    qkv0 = wl.normal_bf16(901, "gc.qkv", (T, s.qkv_width))
    x0 = wl.normal_bf16(901, "gc.x", (T, s.hidden))
    r0 = wl.normal_bf16(901, "gc.r", (T, s.hidden))
    gamma = wl.normal_bf16(901, "gc.g", (s.hidden,), 1.0, 0.1)
    qn = wl.normal_bf16(901, "gc.qn", (128,), 1.0, 0.1)
    kn = wl.normal_bf16(901, "gc.kn", (128,), 1.0, 0.1)
    gate_up0 = wl.normal_bf16(901, "gc.gu", (T, 2 * 3072))
    cu = wl.cu_seqlens(lengths)

    table = rope_table()
    d_gamma, d_qn, d_kn = dev(gamma), dev(qn), dev(kn)
    d_pos, d_slots, d_cu, d_bt = dev_i64(pos), dev_i32(slots), dev_i32(cu), dev_i32(bt)
    x, r, qkv, gate_up = dev(x0), dev(r0), dev(qkv0), dev(gate_up0)
    y = torch.empty_like(x)
    kc = torch.zeros(nb, wl.BLOCK_SIZE, s.hkv, 128, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    o1 = torch.empty(T, s.hq, 128, dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o1)
    act = torch.empty(T, 3072, dtype=torch.bfloat16, device="cuda")
    sched = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = qkv[:, :Q].view(T, s.hq, 128)
    k = qkv[:, Q:Q + D].view(T, s.hkv, 128)
    v = qkv[:, Q + D:].view(T, s.hkv, 128)
    ml = int(lengths.max())

    def reset():
        x.copy_(dev(x0))
        r.copy_(dev(r0))
        qkv.copy_(dev(qkv0))
        kc.zero_()
        vc.zero_()

    def step():
        nv.nv_add_rmsnorm(x, r, d_gamma, y, r, eps=wl.RMS_EPS)
        nv.nv_qknorm_rope_store(q, k, v, d_qn, d_kn, table, d_pos, kc, vc, d_slots,
                                eps=wl.RMS_EPS, write_k=True)
        nv.nv_prefill_attn_varlen(q, k, v, o1, d_cu, d_cu, ml, ml, SCALE, sched_counter=sched)
        nv.nv_prefill_attn_paged(q, kc, vc, d_bt, o2, d_cu, d_cu, ml, SCALE, sched_counter=sched)
        nv.nv_silu_and_mul(gate_up, act)

    def results():
        torch.cuda.synchronize()
        return [host(t) for t in (y, r, qkv, kc, vc, o1, o2, act)]

    # eager reference run (also warms up every kernel's attributes)
    reset()
    step()
    eager = results()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        reset()
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        reset()
        graph.replay()
        for a, b in zip(results(), eager):
            assert np.array_equal(a, b), "graph replay differs from the eager run"

    # and the replayed attention is the oracle's (rounded q, k as the layer stores them)
    q_rot = oracle.qknorm_rope(qkv0[:, :Q].reshape(T, s.hq, 128), qn, pos)
    k_rot = oracle.qknorm_rope(qkv0[:, Q:Q + D].reshape(T, s.hkv, 128), kn, pos)
    qb, kb = oracle.round_to_bf16(q_rot), oracle.round_to_bf16(k_rot)
    vb = qkv0[:, Q + D:].reshape(T, s.hkv, 128)
    ref = oracle.attention_varlen(qb, kb, vb, cu, cu, SCALE, True)
    check_close(eager[5], ref, "graph-captured prefill")
    # The paged call runs the key-offset kernel (its masked tiles split into
    # visible / partial / invisible chunks), the contiguous one with one
    # cu_seqlens array the plain kernel: both within the oracle's tolerance.
    check_close(eager[6], ref, "graph-captured paged prefill")


def test_noalloc_decode_replays_from_a_graph():
    s = wl.QWEN3_8B
    g = np.random.default_rng(910)
    ctx = np.array([1, 300, 2049, 700], np.int32)
    nb = int(sum(math.ceil(int(c) / wl.BLOCK_SIZE) for c in ctx)) + 2
    bt = wl.carve_block_tables(g.permutation(nb).astype(np.int32), ctx)
    kf = wl.normal_bf16(911, "gc.k", (nb, wl.BLOCK_SIZE, s.hkv, 128))
    vf = wl.normal_bf16(911, "gc.v", (nb, wl.BLOCK_SIZE, s.hkv, 128))
    qb = wl.normal_bf16(911, "gc.q", (ctx.size, s.hq, 128))
    kc, vc, q = dev(kf), dev(vf), dev(qb)
    d_bt, d_ctx = dev_i32(bt), dev_i32(ctx)
    o = torch.empty(ctx.size, s.hq, 128, dtype=torch.bfloat16, device="cuda")
    lib = nv.library()

    def step():
        rc = lib.nv_decode_attn_paged_noalloc(
            q.data_ptr(), s.hq * 128, kc.data_ptr(), vc.data_ptr(), d_bt.data_ptr(), bt.shape[1],
            d_ctx.data_ptr(), o.data_ptr(), ctx.size, s.hq, s.hkv, 128, wl.BLOCK_SIZE, nb, SCALE,
            256, None, torch.cuda.current_stream().cuda_stream)
        assert rc == 0

    step()
    torch.cuda.synchronize()
    eager = host(o)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    o.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(host(o), eager)
    check_close(eager, oracle.paged_decode(qb, kf, vf, bt, ctx, SCALE), "graph-captured decode")
