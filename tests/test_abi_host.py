"""The C-ABI library builds, loads and exports every symbol the header
declares; bad arguments are rejected on the host with the documented codes
before anything is launched (so these run without a GPU).  Faults are made on
the host only: null pointers, unsupported shapes, misalignment, a workspace
that is too small."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "nv_attn.h")
NV_OK, NV_EINVAL, NV_EUNSUPPORTED, NV_EALIGN, NV_EWORKSPACE = 0, -1, -2, -3, -4


@pytest.fixture(scope="module")
def lib():
    from paged_kv_attention_kvcache_gb300 import build as b
    b.build()
    import paged_kv_attention_kvcache_gb300 as nv
    return nv.library()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_five_ops():
    names = declared_functions()
    for op in ("nv_add_rmsnorm", "nv_qknorm_rope", "nv_store_kvcache", "nv_prefill_attn_varlen",
               "nv_decode_attn_paged"):
        assert op in names


def test_library_exports_every_declared_symbol(lib):
    import paged_kv_attention_kvcache_gb300 as nv
    names = declared_functions()
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(nv.ABI_FUNCTIONS)


def test_status_strings_and_version(lib):
    assert lib.nv_status_string(0) == b"NV_OK"
    for code in (NV_EINVAL, NV_EUNSUPPORTED, NV_EALIGN, NV_EWORKSPACE, -5, -6):
        assert lib.nv_status_string(code).startswith(b"NV_E")
    assert lib.nv_version() >= 100


FAKE = 0x10000          # a 16-byte-aligned non-null address; never dereferenced
MIS = 0x10002           # misaligned


def test_add_rmsnorm_rejects_bad_arguments(lib):
    f = lib.nv_add_rmsnorm
    assert f(None, None, FAKE, FAKE, None, 4, 1024, 1024, 1e-6, None) == NV_EINVAL
    assert f(FAKE, None, FAKE, FAKE, None, -1, 1024, 1024, 1e-6, None) == NV_EINVAL
    assert f(FAKE, None, FAKE, FAKE, None, 4, 1020, 1020, 1e-6, None) == NV_EUNSUPPORTED
    assert f(FAKE, FAKE, FAKE, FAKE, None, 4, 1024, 1024, 1e-6, None) == NV_EINVAL  # no residual_out
    assert f(MIS, None, FAKE, FAKE, None, 4, 1024, 1024, 1e-6, None) == NV_EALIGN
    assert f(FAKE, None, FAKE, FAKE, None, 0, 1024, 1024, 1e-6, None) == NV_OK     # empty: no-op
    assert f(FAKE, None, FAKE, FAKE, None, 4, 1024, 1024, float("nan"), None) == NV_EINVAL
    assert f(FAKE, None, FAKE, FAKE, None, 4, 1024, 1000, 1e-6, None) == NV_EINVAL  # stride < H
    assert f(FAKE, None, FAKE, FAKE, None, 4, 1024, 1028, 1e-6, None) == NV_EALIGN  # stride % 8


def test_qknorm_rope_rejects_bad_arguments(lib):
    f = lib.nv_qknorm_rope
    ok = dict(q=FAKE, qs=6144, k=FAKE, ks=6144, qw=FAKE, kw=FAKE, cs=FAKE, mp=40960, pos=FAKE,
              T=4, Hq=32, Hkv=8, d=128, eps=1e-6)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["q"], a["qs"], a["k"], a["ks"], a["qw"], a["kw"], a["cs"], a["mp"], a["pos"],
                 a["T"], a["Hq"], a["Hkv"], a["d"], a["eps"], None, None)

    assert call(d=64) == NV_EUNSUPPORTED
    assert call(pos=None) == NV_EINVAL
    assert call(qs=100) == NV_EINVAL                 # stride shorter than Hq * d
    assert call(qs=4100) == NV_EALIGN                # stride not a multiple of 8
    assert call(k=MIS) == NV_EALIGN
    assert call(mp=0) == NV_EINVAL
    assert call(T=0) == NV_OK


def test_store_kvcache_rejects_bad_arguments(lib):
    f = lib.nv_store_kvcache
    assert f(FAKE, 1024, FAKE, 1024, FAKE, FAKE, None, 4, 8, 128, 100, None, None) == NV_EINVAL
    assert f(FAKE, 1024, FAKE, 1024, FAKE, FAKE, FAKE, 4, 1, 6, 100, None, None) == NV_EUNSUPPORTED
    assert f(FAKE, 1000, FAKE, 1024, FAKE, FAKE, FAKE, 4, 8, 128, 100, None, None) == NV_EINVAL
    assert f(FAKE, 1032, FAKE, 1028, FAKE, FAKE, FAKE, 4, 8, 128, 100, None, None) == NV_EALIGN
    assert f(FAKE, 1024, FAKE, 1024, MIS, FAKE, FAKE, 4, 8, 128, 100, None, None) == NV_EALIGN
    assert f(FAKE, 1024, FAKE, 1024, FAKE, FAKE, FAKE, 0, 8, 128, 100, None, None) == NV_OK


def test_prefill_rejects_bad_arguments(lib):
    f = lib.nv_prefill_attn_varlen

    def call(Hq=32, Hkv=8, d=128, causal=1, q=FAKE, qs=6144, B=2, scale=0.088, sc=None):
        return f(q, qs, FAKE, 6144, FAKE, 6144, FAKE, FAKE, FAKE, B, 100, 100, 64, 64, Hq, Hkv, d,
                 scale, causal, sc, None, None)

    assert call(Hq=30) == NV_EINVAL                  # Hq % Hkv != 0
    assert call(d=64) == NV_EUNSUPPORTED
    assert call(causal=0) == NV_EUNSUPPORTED
    assert call(q=None) == NV_EINVAL
    assert call(q=MIS) == NV_EALIGN
    assert call(qs=6148) == NV_EALIGN
    assert call(scale=0.0) == NV_EINVAL
    assert call(sc=FAKE + 2) == NV_EALIGN            # work counter must be 4-byte aligned
    assert call(B=0) == NV_OK


def test_decode_rejects_bad_arguments_and_small_workspace(lib):
    f = lib.nv_decode_attn_paged

    def call(Hq=32, Hkv=8, d=128, bs=256, mb=32, ws=None, wsb=0, q=FAKE, B=4, split=0):
        return f(q, 4096, FAKE, FAKE, FAKE, mb, FAKE, FAKE, B, Hq, Hkv, d, bs, 1000, 0.088, split,
                 ws, wsb, None, None)

    assert call(Hq=12) == NV_EINVAL                  # Hq % Hkv != 0
    assert call(Hq=256, Hkv=8) == NV_EUNSUPPORTED    # group of 32 > 16
    assert call(d=96) == NV_EUNSUPPORTED
    assert call(bs=100) == NV_EUNSUPPORTED
    assert call(q=None) == NV_EINVAL
    assert call(q=MIS) == NV_EALIGN
    # A context of 32 blocks with 256-token splits needs a workspace.
    need = lib.nv_decode_attn_workspace_size(4, 32, 8, 128, 32, 256, 256)
    assert need == 4 * 32 * 32 * 129 * 4
    assert call(split=256) == NV_EWORKSPACE
    assert call(split=256, ws=FAKE, wsb=need - 4) == NV_EWORKSPACE
    assert call(split=256, ws=MIS, wsb=need) == NV_EALIGN
    # One split per sequence needs none.
    assert lib.nv_decode_attn_workspace_size(4, 32, 8, 128, 4, 256, 1024) == 0
    assert call(B=0) == NV_OK


def test_decode_automatic_split_choices(lib):
    """The automatic split (kv_split_tokens = 0), read back through the
    workspace query: B * Hq * splits * (128 + 1) floats.  Without a GPU the
    library assumes GB300's 152 SMs."""
    def splits(B, Hq, Hkv, ctx):
        ws = lib.nv_decode_attn_workspace_size(B, Hq, Hkv, 128, ctx // 256, 256, 0)
        assert ws % (B * Hq * 129 * 4) == 0
        return max(1, ws // (B * Hq * 129 * 4))

    # The configured decode sets: 1024-, 2048- and 4096-key splits.
    assert splits(64, 16, 8, 4096) == 4
    assert splits(256, 32, 8, 8192) == 4
    assert splits(32, 32, 8, 40960) == 10
    # Short contexts over at least one (sequence, kv head) pair per SM: unsplit.
    assert splits(64, 32, 8, 1024) == 1
    assert splits(32, 32, 8, 2048) == 1
    # Fewer pairs: 1024-key splits, halved only while the grid has fewer CTAs
    # than half the SMs, and never below 512 keys.
    assert splits(16, 32, 8, 2048) == 2
    assert splits(8, 32, 8, 1024) == 2
    assert splits(8, 32, 8, 512) == 1
    assert splits(1, 32, 8, 8192) == 16
    # A single long sequence fills one wave (2048-key splits); two do not.
    assert splits(1, 32, 8, 40960) == 20
    assert splits(2, 32, 8, 40960) == 40


def test_rope_table_rejects_bad_arguments(lib):
    f = lib.nv_rope_cos_sin_cache
    assert f(FAKE, 16, 127, 1e6, None) == NV_EINVAL
    assert f(FAKE, 16, 128, 0.5, None) == NV_EINVAL
    assert f(None, 16, 128, 1e6, None) == NV_EINVAL
    assert f(None, 0, 128, 1e6, None) == NV_OK


def test_paged_prefill_rejects_bad_arguments(lib):
    f = lib.nv_prefill_attn_paged

    def call(bs=256, d=128, causal=1, bt=FAKE, q=FAKE, Hq=32, Hkv=8, B=2, sc=None):
        return f(q, 4096, FAKE, FAKE, bt, 16, FAKE, FAKE, FAKE, B, 100, 64, Hq, Hkv, d, bs, 1000,
                 0.088, causal, sc, None, None)

    assert call(bs=192) == NV_EUNSUPPORTED          # block must hold whole 128-key tiles
    assert call(d=64) == NV_EUNSUPPORTED
    assert call(causal=0) == NV_EUNSUPPORTED
    assert call(bt=None) == NV_EINVAL
    assert call(Hq=12) == NV_EINVAL
    assert call(q=MIS) == NV_EALIGN
    assert call(sc=FAKE + 1) == NV_EALIGN
    assert call(B=0) == NV_OK


def test_qknorm_rope_store_rejects_bad_arguments(lib):
    f = lib.nv_qknorm_rope_store
    ok = dict(q=FAKE, qs=6144, k=FAKE, ks=6144, v=FAKE, vs=6144, sm=FAKE, kc=FAKE, vc=FAKE,
              ns=1 << 20, T=4, Hq=32, Hkv=8, d=128, wk=0)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["q"], a["qs"], a["k"], a["ks"], a["v"], a["vs"], FAKE, FAKE, FAKE, 40960, FAKE,
                 a["sm"], a["kc"], a["vc"], a["ns"], a["T"], a["Hq"], a["Hkv"], a["d"], 1e-6,
                 a["wk"], None, None)

    assert call(d=64) == NV_EUNSUPPORTED
    assert call(sm=None) == NV_EINVAL
    assert call(vc=None) == NV_EINVAL
    assert call(vs=512) == NV_EINVAL                 # stride shorter than Hkv * d
    assert call(wk=2) == NV_EINVAL
    assert call(ns=-1) == NV_EINVAL
    assert call(kc=MIS) == NV_EALIGN
    assert call(vs=6148) == NV_EALIGN
    assert call(T=0) == NV_OK


def test_silu_and_mul_rejects_bad_arguments(lib):
    f = lib.nv_silu_and_mul
    X, O = 0x100000, 0x900000                         # far apart: no overlap
    assert f(X, 24576, O, 12288, 4, 12280 + 4, None) == NV_EUNSUPPORTED   # I % 8
    assert f(None, 24576, O, 12288, 4, 12288, None) == NV_EINVAL
    assert f(X, 24570, O, 12288, 4, 12288, None) == NV_EINVAL            # stride < 2I
    assert f(X, 24576, O, 12280, 4, 12288, None) == NV_EINVAL            # out stride < I
    assert f(X + 2, 24576, O, 12288, 4, 12288, None) == NV_EALIGN
    assert f(X, 24584 + 4, O, 12288, 4, 12288, None) == NV_EALIGN
    assert f(X, 24576, X + 2 * 12288 * 2, 12288, 4, 12288, None) == NV_EINVAL  # overlap
    assert f(X, 24576, X, 12288, 4, 12288, None) == NV_EINVAL      # same base, other stride
    assert f(X, 24576, O, 12288, 0, 12288, None) == NV_OK
    assert f(X, 24576, O, 12288, -1, 12288, None) == NV_EINVAL


def test_wait_timeout_selftest_rejects_bad_counter(lib):
    # Checked on the host before any launch.
    assert lib.nv_selftest_wait_timeout(None, None) == NV_EINVAL
    assert lib.nv_selftest_wait_timeout(MIS, None) == NV_EINVAL
