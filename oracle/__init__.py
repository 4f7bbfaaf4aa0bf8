"""fp64 CPU oracle for the Qwen3 attention-sublayer hot path.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import this package.  The CUDA library never links, loads or
calls it, and it never calls the CUDA library.

The arithmetic lives in ``nvattn_oracle.c`` (plain C, fp64, OpenMP over
independent rows); this module only compiles it with gcc and marshals numpy
arrays through ctypes.  Each wrapper names the passage of the pages it
follows; the C file carries the definitions.

Every function here is pinned by ``tests/test_oracle_pins.py`` against
values the pages print, closed forms and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvattn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libnvattn_oracle.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int
_F64 = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math: IEEE fp64 semantics)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.orc_num_threads.restype = _I32
            lib.orc_round_to_bf16.argtypes = [_P, _P, _I64]
            lib.orc_add_rmsnorm.argtypes = [_P, _P, _P, _I64, _I64, _F64, _P, _P]
            lib.orc_add_rmsnorm.restype = _I32
            lib.orc_rope_cos_sin.argtypes = [_I64, _I32, _F64, _P]
            lib.orc_rope_cos_sin.restype = _I32
            lib.orc_qknorm_rope.argtypes = [_P, _I64, _I64, _I32, _I32, _P, _P, _F64, _F64, _P]
            lib.orc_qknorm_rope.restype = _I32
            lib.orc_store_kvcache.argtypes = [_P, _I64, _P, _I64, _P, _P, _P, _I64, _I64, _I64]
            lib.orc_store_kvcache.restype = _I64
            lib.orc_silu_and_mul.argtypes = [_P, _I64, _I64, _I64, _P]
            lib.orc_silu_and_mul.restype = _I32
            lib.orc_attention_varlen.argtypes = [_P, _I64, _P, _I64, _P, _I64, _P, _P, _I32,
                                                 _I32, _I32, _I32, _F64, _I32, _P, _I64, _P]
            lib.orc_attention_varlen.restype = _I32
            lib.orc_paged_decode.argtypes = [_P, _I64, _P, _P, _P, _I32, _P, _I32, _I32, _I32,
                                             _I32, _I32, _I64, _F64, _P, _I64, _P]
            lib.orc_paged_decode.restype = _I32
            lib.orc_attention_paged_prefill.argtypes = [_P, _I64, _P, _P, _P, _I32, _P, _P, _I32,
                                                        _I32, _I32, _I32, _I32, _I64, _F64, _P,
                                                        _I64, _P]
            lib.orc_attention_paged_prefill.restype = _I32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 tensors are passed as uint16 bit patterns")
    return a


def num_threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all cores)."""
    return int(_load().orc_num_threads())


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bits, round-to-nearest-even (the model dtype is bf16)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().orc_round_to_bf16(_ptr(x), _ptr(out), x.size)
    return out


def add_rmsnorm(x, residual, weight, eps: float = 1e-6):
    """Residual-add RMSNorm ("3.3 Model skeleton and core operators", sec. 2).

    x, residual: [T, H] bf16 bits (residual may be None: plain RMSNorm);
    weight: [H] bf16 bits.  Returns (y, residual_out) in fp64;
    residual_out is None when residual is None.
    """
    x = _u16(x)
    T, H = x.shape
    r = None if residual is None else _u16(residual)
    w = _u16(weight)
    y = np.empty((T, H), np.float64)
    r_out = None if r is None else np.empty((T, H), np.float64)
    rc = _load().orc_add_rmsnorm(_ptr(x), _ptr(r), _ptr(w), T, H, eps, _ptr(y), _ptr(r_out))
    if rc:
        raise ValueError(f"orc_add_rmsnorm failed: {rc}")
    return y, r_out


def rope_cos_sin(max_position: int, rotary_dim: int, base: float) -> np.ndarray:
    """Exact [max_position, rotary_dim] cos|sin table ("3.3 ...", sec. 3)."""
    out = np.empty((max_position, rotary_dim), np.float64)
    rc = _load().orc_rope_cos_sin(max_position, rotary_dim, base, _ptr(out))
    if rc:
        raise ValueError(f"orc_rope_cos_sin failed: {rc}")
    return out


def qknorm_rope(x, weight, positions, base: float = 1e6, eps: float = 1e-6):
    """Per-head RMSNorm over head_dim, then the half-split rotation.

    x: [T, nheads, d] bf16 bits (a view with any token stride is accepted:
    it is given as the 2-D array [T, row] plus nheads, d via its shape);
    weight: [d] bf16 bits; positions: [T] int64.  Returns [T, nheads, d] fp64.
    """
    x = np.asarray(x)
    if x.ndim != 3:
        raise ValueError("x must be [T, nheads, d]")
    T, nh, d = x.shape
    xc = _u16(x).reshape(T, nh * d)
    w = _u16(weight)
    pos = np.ascontiguousarray(positions, dtype=np.int64)
    out = np.empty((T, nh, d), np.float64)
    rc = _load().orc_qknorm_rope(_ptr(xc), nh * d, T, nh, d, _ptr(w), _ptr(pos), base, eps,
                                 _ptr(out))
    if rc:
        raise ValueError(f"orc_qknorm_rope failed: {rc}")
    return out


def store_kvcache(key, value, k_cache, v_cache, slot_mapping) -> int:
    """Slot scatter ("Nano-vLLM 源码解读 第17篇", sec. 5.1), in place.

    key, value: [N, Hkv, d] bf16 bits; k_cache, v_cache: [nb, bs, Hkv, d]
    bf16 bits (modified in place); slot_mapping: [N] int32.  Returns the
    number of slots outside [0, nb*bs) other than the -1 padding marker.
    """
    key = _u16(key)
    value = _u16(value)
    if not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
        raise ValueError("caches must be contiguous")
    if k_cache.dtype != np.uint16 or v_cache.dtype != np.uint16:
        raise TypeError("caches are bf16 bit patterns")
    N = key.shape[0]
    D = int(np.prod(key.shape[1:])) if N else int(np.prod(k_cache.shape[2:]))
    num_slots = k_cache.shape[0] * k_cache.shape[1]
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int32)
    return int(_load().orc_store_kvcache(_ptr(key), D, _ptr(value), D, _ptr(k_cache),
                                         _ptr(v_cache), _ptr(slots), N, D, num_slots))


def silu_and_mul(x):
    """SwiGLU activation ("3.3 Model skeleton and core operators", sec. 4).

    x: [T, 2I] bf16 bits, gate in the first half, up in the second.  Returns
    silu(gate) * up as [T, I] fp64 (unrounded).
    """
    x = _u16(x)
    if x.ndim != 2 or x.shape[1] % 2:
        raise ValueError("x must be [T, 2I]")
    T, two_i = x.shape
    out = np.empty((T, two_i // 2), dtype=np.float64)
    rc = _load().orc_silu_and_mul(_ptr(x), two_i, T, two_i // 2, _ptr(out))
    if rc:
        raise ValueError("orc_silu_and_mul: bad arguments")
    return out


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool = True,
                     rows=None):
    """Varlen (causal) GQA attention, plain definition.

    q: [Tq, Hq, d], k/v: [Tk, Hkv, d] bf16 bits; cu_seqlens_*: [B+1] int32.
    rows: optional [n, 2] int64 (token, head) pairs.  Returns [Tq, Hq, d]
    or [n, d] fp64.
    """
    q = _u16(q)
    k = _u16(k)
    v = _u16(v)
    Tq, Hq, d = q.shape
    Hkv = k.shape[1]
    cq = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
    ck = np.ascontiguousarray(cu_seqlens_k, dtype=np.int32)
    B = cq.size - 1
    if rows is None:
        out = np.empty((Tq, Hq, d), np.float64)
        rp, n = None, 0
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 2)
        out = np.empty((rows.shape[0], d), np.float64)
        rp, n = rows, rows.shape[0]
    rc = _load().orc_attention_varlen(_ptr(q), Hq * d, _ptr(k), Hkv * d, _ptr(v), Hkv * d,
                                      _ptr(cq), _ptr(ck), B, Hq, Hkv, d, scale,
                                      1 if causal else 0, _ptr(rp), n, _ptr(out))
    if rc:
        raise ValueError(f"orc_attention_varlen failed: {rc}")
    return out


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale: float, pairs=None):
    """Single-query decode over the paged cache ("nano-vllm code walkthrough").

    q: [B, Hq, d] bf16 bits; caches: [nb, bs, Hkv, d] bf16 bits;
    block_tables: [B, MB] int32; context_lens: [B] int32.  pairs: optional
    [n, 2] int64 (b, h).  Returns [B, Hq, d] or [n, d] fp64.
    """
    q = _u16(q)
    B, Hq, d = q.shape
    if k_cache.dtype != np.uint16 or not k_cache.flags.c_contiguous:
        raise TypeError("k_cache must be contiguous bf16 bits")
    if v_cache.dtype != np.uint16 or not v_cache.flags.c_contiguous:
        raise TypeError("v_cache must be contiguous bf16 bits")
    nb, bs, Hkv, d2 = k_cache.shape
    assert d2 == d
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    MB = bt.shape[1] if bt.ndim == 2 else 0
    if pairs is None:
        out = np.empty((B, Hq, d), np.float64)
        pp, n = None, 0
    else:
        pairs = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
        out = np.empty((pairs.shape[0], d), np.float64)
        pp, n = pairs, pairs.shape[0]
    rc = _load().orc_paged_decode(_ptr(q), Hq * d, _ptr(k_cache), _ptr(v_cache), _ptr(bt), MB,
                                  _ptr(ctx), B, Hq, Hkv, d, bs, nb, scale, _ptr(pp), n,
                                  _ptr(out))
    if rc:
        raise ValueError(f"orc_paged_decode failed: {rc}")
    return out


def attention_paged_prefill(q, k_cache, v_cache, block_tables, cu_seqlens_q, cu_seqlens_k,
                            scale: float, rows=None):
    """Prefill over the paged cache (prefix hit / chunked prefill).

    q: [Tq, Hq, d] bf16 bits (the new tokens); caches [nb, bs, Hkv, d] bf16
    bits holding each sequence's Lk keys (prefix + new) through block_tables
    [B, MB] int32; cu_seqlens_q / cu_seqlens_k: [B+1] int32 (Lk >= Lq).
    Query i of a sequence sees keys j <= Lk - Lq + i.  rows: optional [n, 2]
    (token, head).  Returns [Tq, Hq, d] or [n, d] fp64.
    """
    q = _u16(q)
    Tq, Hq, d = q.shape
    for c in (k_cache, v_cache):
        if c.dtype != np.uint16 or not c.flags.c_contiguous:
            raise TypeError("caches must be contiguous bf16 bits")
    nb, bs, Hkv, d2 = k_cache.shape
    assert d2 == d
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cq = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
    ck = np.ascontiguousarray(cu_seqlens_k, dtype=np.int32)
    B = cq.size - 1
    if rows is None:
        out = np.empty((Tq, Hq, d), np.float64)
        rp, n = None, 0
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 2)
        out = np.empty((rows.shape[0], d), np.float64)
        rp, n = rows, rows.shape[0]
    rc = _load().orc_attention_paged_prefill(_ptr(q), Hq * d, _ptr(k_cache), _ptr(v_cache),
                                             _ptr(bt), bt.shape[1], _ptr(cq), _ptr(ck), B, Hq,
                                             Hkv, d, bs, nb, scale, _ptr(rp), n, _ptr(out))
    if rc:
        raise ValueError(f"orc_attention_paged_prefill failed: {rc}")
    return out
