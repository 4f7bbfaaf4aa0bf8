"""Chained parity of the whole attention-sublayer path: the GPU runs
add-RMSNorm -> QK-Norm + RoPE -> store_kvcache -> attention exactly as one
nano-vllm layer does, and the fp64 oracle runs the same chain on its own.
Where the pages keep a tensor in bf16 (q and k after RoPE, the KV cache) the
oracle rounds its own fp64 value to bf16; no GPU result ever feeds it."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import check_cache_rows, check_close, dev, dev_i32, dev_i64, err_counter, host, rope_table

pytestmark = pytest.mark.gpu

import paged_kv_attention_kvcache_gb300 as nv  # noqa: E402

SCALE = 128 ** -0.5


def test_small_layer_prefill_then_eight_decode_steps():
    pre, steps = wl.config1()
    s = pre.shape
    T, Q, D = pre.qkv.shape[0], s.q_size, s.kv_size
    table = rope_table()
    err = err_counter()
    kc = torch.zeros(pre.num_blocks, wl.BLOCK_SIZE, s.hkv, 128, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    ref_k = np.zeros((pre.num_blocks, wl.BLOCK_SIZE, s.hkv, 128), np.uint16)
    ref_v = np.zeros_like(ref_k)
    gamma, qn, kn = dev(pre.gamma), dev(pre.q_norm_w), dev(pre.k_norm_w)

    def layer_norm(x_bits, r_bits):
        x, r = dev(x_bits), dev(r_bits)
        y = torch.empty_like(x)
        nv.nv_add_rmsnorm(x, r, gamma, y, r, eps=wl.RMS_EPS)   # residual updated in place
        return y, r

    def check_norm(y, r, x_bits, r_bits, what):
        y_ref, r_ref = oracle.add_rmsnorm(x_bits, r_bits, pre.gamma, wl.RMS_EPS)
        check_close(host(y), y_ref, what + " norm")
        check_close(host(r), r_ref, what + " residual", max_tol=2 ** -8, mean_tol=2 ** -9)

    def rope_ref(qkv_bits, positions):
        n = qkv_bits.shape[0]
        q_rot = oracle.qknorm_rope(qkv_bits[:, :Q].reshape(n, s.hq, 128), pre.q_norm_w, positions)
        k_rot = oracle.qknorm_rope(qkv_bits[:, Q:Q + D].reshape(n, s.hkv, 128), pre.k_norm_w,
                                   positions)
        return q_rot, k_rot

    # ---- prefill
    y, r = layer_norm(pre.x, pre.residual)
    qkv = dev(pre.qkv)
    q = qkv[:, :Q].view(T, s.hq, 128)
    k = qkv[:, Q:Q + D].view(T, s.hkv, 128)
    v = qkv[:, Q + D:].view(T, s.hkv, 128)
    nv.nv_qknorm_rope(q, k, qn, kn, table, dev_i64(pre.positions), eps=wl.RMS_EPS, err_count=err)
    nv.nv_store_kvcache(k, v, kc, vc, dev_i32(pre.slot_mapping), err)
    cu = dev_i32(pre.cu_seqlens)
    o = torch.empty(T, s.hq, 128, dtype=torch.bfloat16, device="cuda")
    ml = int(pre.lengths.max())
    sched = torch.zeros(1, dtype=torch.int32, device="cuda")
    nv.nv_prefill_attn_varlen(q, k, v, o, cu, cu, ml, ml, SCALE, err_count=err, sched_counter=sched)
    torch.cuda.synchronize()
    check_norm(y, r, pre.x, pre.residual, "prefill")
    q_rot, k_rot = rope_ref(pre.qkv, pre.positions)
    qb, kb = oracle.round_to_bf16(q_rot), oracle.round_to_bf16(k_rot)
    vb = pre.qkv[:, Q + D:].reshape(T, s.hkv, 128)
    oracle.store_kvcache(kb, vb, ref_k, ref_v, pre.slot_mapping)
    o_ref = oracle.attention_varlen(qb, kb, vb, pre.cu_seqlens, pre.cu_seqlens, SCALE)
    check_close(host(o), o_ref, "prefill attention")
    check_cache_rows(host(kc), ref_k, "prefill k cache")
    assert np.array_equal(host(vc), ref_v), "v cache must be bit-exact"

    # ---- decode steps
    B = pre.lengths.size
    bt = dev_i32(pre.block_tables)
    for i, st in enumerate(steps):
        y, r = layer_norm(st["x"], st["residual"])
        qkv = dev(st["qkv"])
        q = qkv[:, :Q].view(B, s.hq, 128)
        k = qkv[:, Q:Q + D].view(B, s.hkv, 128)
        v = qkv[:, Q + D:].view(B, s.hkv, 128)
        nv.nv_qknorm_rope(q, k, qn, kn, table, dev_i64(st["positions"]), eps=wl.RMS_EPS,
                          err_count=err)
        nv.nv_store_kvcache(k, v, kc, vc, dev_i32(st["slot_mapping"]), err)
        od = torch.empty(B, s.hq, 128, dtype=torch.bfloat16, device="cuda")
        split = 64 if i % 2 else 0            # alternate forced and automatic splits
        ws_b = nv.nv_decode_attn_workspace_size(B, s.hq, s.hkv, 128, pre.block_tables.shape[1],
                                                wl.BLOCK_SIZE, split)
        ws = torch.empty(max(1, ws_b // 4), dtype=torch.float32, device="cuda")
        nv.nv_decode_attn_paged(q, kc, vc, bt, dev_i32(st["context_lens"]), od, SCALE,
                                workspace=ws, kv_split_tokens=split, err_count=err)
        torch.cuda.synchronize()
        check_norm(y, r, st["x"], st["residual"], f"step {i}")
        q_rot, k_rot = rope_ref(st["qkv"], st["positions"])
        qb, kb = oracle.round_to_bf16(q_rot), oracle.round_to_bf16(k_rot)
        vb = st["qkv"][:, Q + D:].reshape(B, s.hkv, 128)
        oracle.store_kvcache(kb, vb, ref_k, ref_v, st["slot_mapping"])
        od_ref = oracle.paged_decode(qb, ref_k, ref_v, pre.block_tables, st["context_lens"], SCALE)
        check_close(host(od), od_ref, f"decode step {i}")
    check_cache_rows(host(kc), ref_k, "final k cache")
    assert np.array_equal(host(vc), ref_v)
    assert int(err.item()) == 0


def test_qwen3_8b_decode_step_full_size():
    step = wl.config3()
    s = step.shape
    B, Q, D = step.context_lens.size, s.q_size, s.kv_size
    table = rope_table()
    err = err_counter()
    x, r = dev(step.x), dev(step.residual)
    y = torch.empty_like(x)
    nv.nv_add_rmsnorm(x, r, dev(step.gamma), y, r, eps=wl.RMS_EPS)
    qkv = dev(step.qkv)
    q = qkv[:, :Q].view(B, s.hq, 128)
    k = qkv[:, Q:Q + D].view(B, s.hkv, 128)
    v = qkv[:, Q + D:].view(B, s.hkv, 128)
    nv.nv_qknorm_rope(q, k, dev(step.q_norm_w), dev(step.k_norm_w), table,
                      dev_i64(step.positions), eps=wl.RMS_EPS, err_count=err)
    kc, vc = dev(step.pool.k), dev(step.pool.v)
    nv.nv_store_kvcache(k, v, kc, vc, dev_i32(step.slot_mapping), err)
    o = torch.empty(B, s.hq, 128, dtype=torch.bfloat16, device="cuda")
    ws_b = nv.nv_decode_attn_workspace_size(B, s.hq, s.hkv, 128, step.block_tables.shape[1],
                                            wl.BLOCK_SIZE, 0)
    ws = torch.empty(max(1, ws_b // 4), dtype=torch.float32, device="cuda")
    nv.nv_decode_attn_paged(q, kc, vc, dev_i32(step.block_tables), dev_i32(step.context_lens), o,
                            SCALE, workspace=ws, err_count=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    y_ref, r_ref = oracle.add_rmsnorm(step.x, step.residual, step.gamma, wl.RMS_EPS)
    check_close(host(y), y_ref, "8b norm")
    check_close(host(r), r_ref, "8b residual", max_tol=2 ** -8, mean_tol=2 ** -9)
    q_rot = oracle.qknorm_rope(step.qkv[:, :Q].reshape(B, s.hq, 128), step.q_norm_w, step.positions)
    k_rot = oracle.qknorm_rope(step.qkv[:, Q:Q + D].reshape(B, s.hkv, 128), step.k_norm_w,
                               step.positions)
    check_close(host(qkv)[:, :Q], q_rot.reshape(B, Q), "8b q rope")
    qb, kb = oracle.round_to_bf16(q_rot), oracle.round_to_bf16(k_rot)
    vb = step.qkv[:, Q + D:].reshape(B, s.hkv, 128)
    # The oracle's cache: the pool with its own rounded new rows written in.
    ref_k, ref_v = step.pool.k, step.pool.v
    assert oracle.store_kvcache(kb, vb, ref_k, ref_v, step.slot_mapping) == 0
    slots = step.slot_mapping.astype(np.int64)
    idx = torch.from_numpy(slots).cuda()
    got_k = host(kc.view(-1, D)[idx])
    got_v = host(vc.view(-1, D)[idx])
    check_cache_rows(got_k, ref_k.reshape(-1, D)[slots], "8b new k rows")
    assert np.array_equal(got_v, ref_v.reshape(-1, D)[slots])
    o_ref = oracle.paged_decode(qb, ref_k, ref_v, step.block_tables, step.context_lens, SCALE)
    check_close(host(o), o_ref, "8b decode layer (B=256, every head)")
