"""Tensors the kernels touch only with ordinary loads and stores may live in
pinned host memory that the device addresses directly (Grace-Blackwell
unified addressing); the kernels then read and write them over the host link.
Each op is run once on device memory and once with those tensors in pinned
host memory, and must give the same bits.  Tensors read through TMA (the KV
caches, the prefill's q, k, v) are refused with NV_EINVAL before anything is
launched."""
import math

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import dev, dev_i32, dev_i64, host, rope_table

pytestmark = pytest.mark.gpu

import paged_kv_attention_kvcache_gb300 as nv  # noqa: E402

SCALE = 128 ** -0.5


def pinned(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
        torch.bfloat16).pin_memory()


def bits(t):
    torch.cuda.synchronize()
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16).copy()


def test_norm_rope_store_swiglu_on_pinned_host_memory():
    s = wl.QWEN3_8B
    T, Q, D = 64, s.q_size, s.kv_size
    g = np.random.default_rng(920)
    x0 = wl.normal_bf16(920, "hm.x", (T, s.hidden))
    r0 = wl.normal_bf16(920, "hm.r", (T, s.hidden))
    gamma = dev(wl.normal_bf16(920, "hm.g", (s.hidden,), 1.0, 0.1))
    qkv0 = wl.normal_bf16(920, "hm.qkv", (T, s.qkv_width))
    qn = dev(wl.normal_bf16(920, "hm.qn", (128,), 1.0, 0.1))
    kn = dev(wl.normal_bf16(920, "hm.kn", (128,), 1.0, 0.1))
    pos = g.integers(0, wl.MAX_POSITION, T).astype(np.int64)
    nb = 4
    slots = g.permutation(nb * wl.BLOCK_SIZE)[:T].astype(np.int32)
    gu0 = wl.normal_bf16(920, "hm.gu", (T, 2 * 12288))
    table = rope_table()

    def run(place):
        x, r, qkv, gu = place(x0), place(r0), place(qkv0), place(gu0)
        y, r_out = torch.empty_like(x), torch.empty_like(x)
        act = torch.empty(T, 12288, dtype=torch.bfloat16, device=x.device)
        if not x.is_cuda:
            y, r_out, act = y.pin_memory(), r_out.pin_memory(), act.pin_memory()
        kc = torch.zeros(nb, wl.BLOCK_SIZE, s.hkv, 128, dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        q = qkv[:, :Q].view(T, s.hq, 128)
        k = qkv[:, Q:Q + D].view(T, s.hkv, 128)
        v = qkv[:, Q + D:].view(T, s.hkv, 128)
        nv.nv_add_rmsnorm(x, r, gamma, y, r_out, eps=wl.RMS_EPS)
        nv.nv_qknorm_rope(q, k, qn, kn, table, dev_i64(pos), eps=wl.RMS_EPS)
        nv.nv_store_kvcache(k, v, kc, vc, dev_i32(slots))
        nv.nv_silu_and_mul(gu, act)
        return [bits(t) for t in (y, r_out, qkv, kc, vc, act)]

    on_device = run(dev)
    on_host = run(pinned)
    for a, b in zip(on_host, on_device):
        assert np.array_equal(a, b)


def test_decode_with_q_and_o_in_pinned_host_memory():
    s = wl.QWEN3_8B
    g = np.random.default_rng(930)
    ctx = np.array([1, 300, 2049, 5000], np.int32)
    nb = int(sum(math.ceil(int(c) / wl.BLOCK_SIZE) for c in ctx)) + 2
    bt = wl.carve_block_tables(g.permutation(nb).astype(np.int32), ctx)
    kc = dev(wl.normal_bf16(930, "hm.k", (nb, wl.BLOCK_SIZE, s.hkv, 128)))
    vc = dev(wl.normal_bf16(930, "hm.v", (nb, wl.BLOCK_SIZE, s.hkv, 128)))
    q0 = wl.normal_bf16(930, "hm.q", (ctx.size, s.hq, 128))
    ws_b = nv.nv_decode_attn_workspace_size(ctx.size, s.hq, s.hkv, 128, bt.shape[1],
                                            wl.BLOCK_SIZE, 256)
    ws = torch.empty(max(1, ws_b // 4), dtype=torch.float32, device="cuda")

    o_dev = torch.empty(ctx.size, s.hq, 128, dtype=torch.bfloat16, device="cuda")
    nv.nv_decode_attn_paged(dev(q0), kc, vc, dev_i32(bt), dev_i32(ctx), o_dev, SCALE,
                            workspace=ws, kv_split_tokens=256)
    o_host = torch.empty(ctx.size, s.hq, 128, dtype=torch.bfloat16).pin_memory()
    bt_host = torch.from_numpy(bt).pin_memory()
    ctx_host = torch.from_numpy(ctx).pin_memory()
    nv.nv_decode_attn_paged(pinned(q0), kc, vc, bt_host, ctx_host, o_host, SCALE,
                            workspace=ws, kv_split_tokens=256)
    assert np.array_equal(bits(o_host), bits(o_dev))


def test_tma_read_tensors_must_be_device_memory():
    s = wl.QWEN3_8B
    ctx = np.array([300], np.int32)
    bt = wl.carve_block_tables(np.arange(2, dtype=np.int32), ctx)
    kc_host = torch.zeros(2, wl.BLOCK_SIZE, s.hkv, 128, dtype=torch.bfloat16).pin_memory()
    vc = torch.zeros(2, wl.BLOCK_SIZE, s.hkv, 128, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(1, s.hq, 128, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    with pytest.raises(nv.NvAttnError) as e:
        nv.nv_decode_attn_paged(q, kc_host, vc, dev_i32(bt), dev_i32(ctx), o, SCALE,
                                kv_split_tokens=4096)            # one split: no workspace
    assert e.value.status == -1
    # the prefill's q read through TMA
    T = 8
    qh = torch.zeros(T, s.hq, 128, dtype=torch.bfloat16).pin_memory()
    kv = torch.zeros(T, s.hkv, 128, dtype=torch.bfloat16, device="cuda")
    cu = dev_i32(wl.cu_seqlens([T]))
    with pytest.raises(nv.NvAttnError) as e:
        nv.nv_prefill_attn_varlen(qh, kv, kv, torch.empty(T, s.hq, 128, dtype=torch.bfloat16,
                                                          device="cuda"), cu, cu, T, T, SCALE)
    assert e.value.status == -1
    torch.cuda.synchronize()
    assert host(o).shape == (1, s.hq, 128)          # nothing was launched; the context is fine
