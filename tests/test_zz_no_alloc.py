"""nv_decode_attn_paged_noalloc: the decode entry point for callers that
cannot allocate device memory (they are handed only their input and output
buffers, e.g. a plugin inside a framework that owns all allocations, or a
serving loop whose free HBM is all committed to the KV cache).  It must give
the same output as nv_decode_attn_paged with a caller-allocated workspace,
call after call, although every call reuses the library's one scratch array.

Called through the C ABI with raw device pointers.  This file is collected
last so that a run stopping at the first failure has run every other test."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import check_close, dev, dev_i32, host

pytestmark = pytest.mark.gpu

NV_EINVAL = -1
NV_EUNSUPPORTED = -2
NV_EWORKSPACE = -4
SCRATCH_BYTES = 16 << 20
SCALE = 128 ** -0.5


@pytest.fixture(scope="module")
def lib():
    from paged_kv_attention_kvcache_gb300 import build as b
    b.build()
    import paged_kv_attention_kvcache_gb300 as nv
    return nv.library()


def _inputs(seed, B, Hq, Hkv, ctx):
    g = np.random.default_rng(seed)
    ctx = np.asarray(ctx, np.int32)
    need = sum(math.ceil(int(c) / 256) for c in ctx)
    nb = need + 2
    bt = wl.carve_block_tables(g.permutation(nb).astype(np.int32), ctx)
    k = wl.f32_to_bf16_bits(g.standard_normal((nb, 256, Hkv, 128)).astype(np.float32))
    v = wl.f32_to_bf16_bits(g.standard_normal((nb, 256, Hkv, 128)).astype(np.float32))
    q = wl.f32_to_bf16_bits(g.standard_normal((B, Hq, 128)).astype(np.float32))
    return dict(q=dev(q), k=dev(k), v=dev(v), bt=dev_i32(bt), ctx=dev_i32(ctx), B=B, Hq=Hq,
                Hkv=Hkv, mb=bt.shape[1], nb=nb, host=(q, k, v, bt, ctx))


def _both(lib, a, split):
    """Run the regular entry point (caller workspace) and the no-alloc one."""
    B, Hq, Hkv = a["B"], a["Hq"], a["Hkv"]
    stream = torch.cuda.current_stream().cuda_stream
    need = lib.nv_decode_attn_workspace_size(B, Hq, Hkv, 128, a["mb"], 256, split)
    assert 0 < need <= SCRATCH_BYTES
    ws = torch.empty(need // 4, dtype=torch.float32, device="cuda")
    o_ref = torch.empty(B, Hq, 128, dtype=torch.bfloat16, device="cuda")
    o_new = torch.full((B, Hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(2, dtype=torch.int32, device="cuda")
    common = (a["q"].data_ptr(), Hq * 128, a["k"].data_ptr(), a["v"].data_ptr(),
              a["bt"].data_ptr(), a["mb"], a["ctx"].data_ptr())
    rc = lib.nv_decode_attn_paged(*common, o_ref.data_ptr(), B, Hq, Hkv, 128, 256, a["nb"],
                                  SCALE, split, ws.data_ptr(), need, err.data_ptr(), stream)
    assert rc == 0
    rc = lib.nv_decode_attn_paged_noalloc(*common, o_new.data_ptr(), B, Hq, Hkv, 128, 256,
                                          a["nb"], SCALE, split, err.data_ptr() + 4, stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert err.tolist() == [0, 0]
    return host(o_ref), host(o_new)


def test_no_alloc_decode_matches_workspace_decode_two_calls_in_a_row(lib):
    # Two different problems back to back: the second call finds the first
    # call's partial results still in the shared scratch array.  Both calls
    # run the same kernels with the same split as the workspace path, so the
    # outputs must be the same bits; each is also checked against the oracle.
    first = _inputs(901, 16, 32, 8, [4096, 300, 2500, 1024, 77, 3000, 4095, 1, 520, 2049,
                                     256, 257, 3500, 900, 4000, 128])
    second = _inputs(902, 8, 16, 8, [5000, 12, 640, 4097, 2300, 1500, 33, 999])
    for a, split in ((first, 256), (second, 512)):
        ref_bits, new_bits = _both(lib, a, split)
        assert np.array_equal(new_bits, ref_bits), f"split={split}: outputs differ"
        q, k, v, bt, ctx = a["host"]
        check_close(new_bits, oracle.paged_decode(q, k, v, bt, ctx, SCALE),
                    f"no-alloc decode split={split}")


def test_no_alloc_decode_rejects_sizes_beyond_its_scratch(lib):
    # Device buffers of a few bytes stand in for the tensors: a call too large
    # for the scratch array is rejected on the host before anything launches.
    B, Hq, Hkv, mb = 256, 32, 8, 160          # 40960-token contexts, 256-key splits
    need = lib.nv_decode_attn_workspace_size(B, Hq, Hkv, 128, mb, 256, 256)
    assert need > SCRATCH_BYTES
    buf = torch.zeros(64, dtype=torch.int32, device="cuda")
    p = buf.data_ptr()
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.nv_decode_attn_paged_noalloc(p, Hq * 128, p, p, p, mb, p, p, B, Hq, Hkv, 128, 256,
                                          1000, SCALE, 256, None, stream)
    assert rc == NV_EWORKSPACE
    # Arguments the regular entry point rejects get its code, not
    # NV_EWORKSPACE, even at sizes beyond the scratch array.
    for hq, hkv, bs, want in ((30, 8, 256, NV_EINVAL), (32, 8, 96, NV_EUNSUPPORTED)):
        rc_new = lib.nv_decode_attn_paged_noalloc(p, hq * 128, p, p, p, mb, p, p, B, hq, hkv,
                                                  128, bs, 1000, SCALE, 256, None, stream)
        rc_ref = lib.nv_decode_attn_paged(p, hq * 128, p, p, p, mb, p, p, B, hq, hkv, 128, bs,
                                          1000, SCALE, 256, None, 0, None, stream)
        assert rc_new == rc_ref == want
    torch.cuda.synchronize()
