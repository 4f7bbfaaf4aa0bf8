"""Python binding of libnvattn.so, the GB300 attention-sublayer library.

Each function has the name of the C entry point it calls (see
include/nv_attn.h) and only marshals arguments: it reads shapes, strides and
data pointers from torch tensors, passes the current CUDA stream, and raises
``NvAttnError`` on a non-zero status.  Every step of the computation runs in
the library's CUDA kernels; there is no fallback of any kind.  If the shared
library has not been built, importing works but the first call raises.

Layouts (bf16 unless noted; "token stride" may exceed the packed width, so
q/k/v may be column views of one packed qkv buffer):
  q [T, Hq, 128], k/v [T, Hkv, 128]; caches [num_blocks, block_size, Hkv, 128];
  slot_mapping / block_tables / context_lens / cu_seqlens int32; positions
  int64; cos_sin fp32 [max_position, 128].
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB_PATH

__all__ = [
    "NvAttnError", "library", "library_path", "nv_version",
    "nv_rope_cos_sin_cache", "nv_add_rmsnorm", "nv_qknorm_rope", "nv_store_kvcache",
    "nv_qknorm_rope_store", "nv_prefill_attn_varlen", "nv_prefill_attn_paged", "nv_decode_attn_workspace_size",
    "nv_decode_attn_paged", "nv_silu_and_mul", "nv_selftest_wait_timeout", "ABI_FUNCTIONS",
]

ABI_FUNCTIONS = (
    "nv_status_string", "nv_version", "nv_rope_cos_sin_cache", "nv_add_rmsnorm",
    "nv_qknorm_rope", "nv_store_kvcache", "nv_qknorm_rope_store", "nv_prefill_attn_varlen",
    "nv_prefill_attn_paged", "nv_decode_attn_workspace_size", "nv_decode_attn_paged",
    "nv_decode_attn_paged_noalloc", "nv_silu_and_mul", "nv_selftest_wait_timeout",
)

_P, _I64, _I32, _F32, _F64, _SZ = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                   ctypes.c_double, ctypes.c_size_t)
_SIGNATURES = {
    "nv_status_string": ([_I32], ctypes.c_char_p),
    "nv_version": ([], _I32),
    "nv_rope_cos_sin_cache": ([_P, _I32, _I32, _F64, _P], _I32),
    "nv_add_rmsnorm": ([_P, _P, _P, _P, _P, _I64, _I32, _I64, _F32, _P], _I32),
    "nv_qknorm_rope": ([_P, _I64, _P, _I64, _P, _P, _P, _I32, _P, _I64, _I32, _I32, _I32, _F32,
                        _P, _P], _I32),
    "nv_store_kvcache": ([_P, _I64, _P, _I64, _P, _P, _P, _I64, _I32, _I32, _I64, _P, _P], _I32),
    "nv_qknorm_rope_store": ([_P, _I64, _P, _I64, _P, _I64, _P, _P, _P, _I32, _P, _P, _P, _P, _I64,
                              _I64, _I32, _I32, _I32, _F32, _I32, _P, _P], _I32),
    "nv_prefill_attn_varlen": ([_P, _I64, _P, _I64, _P, _I64, _P, _P, _P, _I32, _I64, _I64, _I32,
                                _I32, _I32, _I32, _I32, _F32, _I32, _P, _P, _P], _I32),
    "nv_prefill_attn_paged": ([_P, _I64, _P, _P, _P, _I32, _P, _P, _P, _I32, _I64, _I32, _I32, _I32,
                               _I32, _I32, _I64, _F32, _I32, _P, _P, _P], _I32),
    "nv_silu_and_mul": ([_P, _I64, _P, _I64, _I64, _I32, _P], _I32),
    "nv_selftest_wait_timeout": ([_P, _P], _I32),
    "nv_decode_attn_workspace_size": ([_I32, _I32, _I32, _I32, _I32, _I32, _I32], _SZ),
    "nv_decode_attn_paged": ([_P, _I64, _P, _P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _I32,
                              _I64, _F32, _I32, _P, _SZ, _P, _P], _I32),
    "nv_decode_attn_paged_noalloc": ([_P, _I64, _P, _P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32,
                                      _I32, _I64, _F32, _I32, _P, _P], _I32),
}

_lock = threading.Lock()
_lib = None


class NvAttnError(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = status
        msg = library().nv_status_string(status).decode()
        super().__init__(f"{func} returned {status} ({msg})")


def library_path() -> str:
    return LIB_PATH


def library() -> ctypes.CDLL:
    """The loaded libnvattn.so with argument types set (raw C-ABI access)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ "
                    "as g; g.build()\"` (or paged_kv_attention_kvcache_gb300/build.py)")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def _check(name, status):
    if status != 0:
        raise NvAttnError(name, status)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _heads_view(t, name):
    """[T, H, d] view with contiguous heads and head_dim; returns token stride."""
    if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != t.shape[2]:
        raise ValueError(f"{name} must be [T, H, d] with contiguous heads and head_dim")
    return t.stride(0)


def nv_version() -> int:
    return int(library().nv_version())


def nv_rope_cos_sin_cache(cos_sin: torch.Tensor, base: float = 1e6, stream=None) -> None:
    """Fill cos_sin [max_position, rotary_dim] (fp32) with the RoPE table."""
    assert cos_sin.dtype == torch.float32 and cos_sin.is_contiguous()
    _check("nv_rope_cos_sin_cache", library().nv_rope_cos_sin_cache(
        _ptr(cos_sin), cos_sin.shape[0], cos_sin.shape[1], float(base), _stream(stream)))


def nv_add_rmsnorm(x, residual, weight, out, residual_out=None, eps: float = 1e-6,
                   stream=None) -> None:
    """out = RMSNorm(x + residual) * weight; residual_out = x + residual.

    x, residual, out, residual_out: [T, H] views whose rows share one row
    stride (elements) and whose elements within a row are contiguous."""
    T, H = x.shape
    stride = x.stride(0) if T > 1 else H
    for t in (x, residual, out, residual_out):
        if t is None:
            continue
        if tuple(t.shape) != (T, H) or (H > 1 and t.stride(1) != 1):
            raise ValueError("add_rmsnorm tensors must be [T, H] with contiguous rows")
        if T > 1 and t.stride(0) != stride:
            raise ValueError("add_rmsnorm tensors must share one row stride")
    _check("nv_add_rmsnorm", library().nv_add_rmsnorm(
        _ptr(x), _ptr(residual), _ptr(weight), _ptr(out), _ptr(residual_out), T, H, stride,
        float(eps), _stream(stream)))


def nv_qknorm_rope(q, k, q_norm_weight, k_norm_weight, cos_sin, positions, eps: float = 1e-6,
                   err_count=None, stream=None) -> None:
    """In-place per-head RMSNorm + RoPE of q [T, Hq, 128] and k [T, Hkv, 128]."""
    qs = _heads_view(q, "q")
    ks = _heads_view(k, "k")
    T, Hq, d = q.shape
    _check("nv_qknorm_rope", library().nv_qknorm_rope(
        _ptr(q), qs, _ptr(k), ks, _ptr(q_norm_weight), _ptr(k_norm_weight), _ptr(cos_sin),
        cos_sin.shape[0], _ptr(positions), T, Hq, k.shape[1], d, float(eps), _ptr(err_count),
        _stream(stream)))


def nv_store_kvcache(key, value, k_cache, v_cache, slot_mapping, err_count=None,
                     stream=None) -> None:
    """Scatter key/value [N, Hkv, 128] rows into the caches at slot_mapping."""
    ks = _heads_view(key, "key")
    vs = _heads_view(value, "value")
    N, Hkv, d = key.shape
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    num_slots = k_cache.shape[0] * k_cache.shape[1]
    _check("nv_store_kvcache", library().nv_store_kvcache(
        _ptr(key), ks, _ptr(value), vs, _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), N,
        Hkv, d, num_slots, _ptr(err_count), _stream(stream)))


def nv_qknorm_rope_store(q, k, v, q_norm_weight, k_norm_weight, cos_sin, positions,
                         k_cache, v_cache, slot_mapping, eps: float = 1e-6, write_k: bool = False,
                         err_count=None, stream=None) -> None:
    """QK-Norm + RoPE of q (in place) and k, with k and v written to their
    cache slots in the same pass; k in place too when write_k is set."""
    qs = _heads_view(q, "q")
    ks = _heads_view(k, "k")
    vs = _heads_view(v, "v")
    T, Hq, d = q.shape
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    num_slots = k_cache.shape[0] * k_cache.shape[1]
    _check("nv_qknorm_rope_store", library().nv_qknorm_rope_store(
        _ptr(q), qs, _ptr(k), ks, _ptr(v), vs, _ptr(q_norm_weight), _ptr(k_norm_weight),
        _ptr(cos_sin), cos_sin.shape[0], _ptr(positions), _ptr(slot_mapping), _ptr(k_cache),
        _ptr(v_cache), num_slots, T, Hq, k.shape[1], d, float(eps), int(bool(write_k)),
        _ptr(err_count), _stream(stream)))


def nv_prefill_attn_varlen(q, k, v, o, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                           max_seqlen_k: int, softmax_scale: float, causal: bool = True,
                           err_count=None, stream=None, sched_counter=None) -> None:
    """Varlen causal attention; o [Tq, Hq, 128] contiguous is written.
    sched_counter: optional int32 device tensor (one element) that lets the
    CTAs draw work heaviest first; None gives the round-robin assignment."""
    qs = _heads_view(q, "q")
    ks = _heads_view(k, "k")
    vs = _heads_view(v, "v")
    if not o.is_contiguous():
        raise ValueError("o must be contiguous")
    Tq, Hq, d = q.shape
    B = cu_seqlens_q.shape[0] - 1
    _check("nv_prefill_attn_varlen", library().nv_prefill_attn_varlen(
        _ptr(q), qs, _ptr(k), ks, _ptr(v), vs, _ptr(o), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
        B, Tq, k.shape[0], int(max_seqlen_q), int(max_seqlen_k), Hq, k.shape[1], d,
        float(softmax_scale), 1 if causal else 0, _ptr(sched_counter), _ptr(err_count),
        _stream(stream)))


def nv_prefill_attn_paged(q, k_cache, v_cache, block_tables, o, cu_seqlens_q, cu_seqlens_k,
                          max_seqlen_q: int, softmax_scale: float, causal: bool = True,
                          err_count=None, stream=None, sched_counter=None) -> None:
    """Prefill whose keys (cached prefix + new tokens) are read from the paged
    cache through block_tables; o [Tq, Hq, 128] contiguous is written."""
    qs = _heads_view(q, "q")
    if not o.is_contiguous() or not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("o and the caches must be contiguous")
    Tq, Hq, d = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    B = cu_seqlens_q.shape[0] - 1
    _check("nv_prefill_attn_paged", library().nv_prefill_attn_paged(
        _ptr(q), qs, _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(o), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), B, Tq, int(max_seqlen_q), Hq, Hkv, d,
        bs, nb, float(softmax_scale), 1 if causal else 0, _ptr(sched_counter), _ptr(err_count),
        _stream(stream)))


def nv_decode_attn_workspace_size(B, Hq, Hkv, head_dim, max_blocks_per_seq, block_size,
                                  kv_split_tokens: int = 0) -> int:
    return int(library().nv_decode_attn_workspace_size(B, Hq, Hkv, head_dim, max_blocks_per_seq,
                                                       block_size, kv_split_tokens))


def nv_decode_attn_paged(q, k_cache, v_cache, block_tables, context_lens, o,
                         softmax_scale: float, workspace=None, kv_split_tokens: int = 0,
                         err_count=None, stream=None) -> None:
    """Single-query paged attention; q [B, Hq, 128] (token stride allowed)."""
    qs = _heads_view(q, "q")
    B, Hq, d = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    if not o.is_contiguous():
        raise ValueError("o must be contiguous")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("nv_decode_attn_paged", library().nv_decode_attn_paged(
        _ptr(q), qs, _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), _ptr(o), B, Hq, Hkv, d, bs, nb, float(softmax_scale),
        int(kv_split_tokens), _ptr(workspace), ws_bytes, _ptr(err_count), _stream(stream)))


def nv_selftest_wait_timeout(err_count, stream=None) -> None:
    """One bounded wait that cannot succeed (about a second): sets
    NV_ERR_PIPELINE_FAILURE (bit 30) in err_count, an int32 device tensor."""
    _check("nv_selftest_wait_timeout", library().nv_selftest_wait_timeout(
        _ptr(err_count), _stream(stream)))


def nv_silu_and_mul(x, out, stream=None) -> None:
    """out [T, I] = silu(x[:, :I]) * x[:, I:] for x [T, 2I] (row-strided views
    allowed; out may be x[:, :I] itself)."""
    if x.dim() != 2 or out.dim() != 2 or x.stride(1) != 1 or out.stride(1) != 1:
        raise ValueError("silu_and_mul takes [T, 2I] and [T, I] row-major views")
    T, two_i = x.shape
    if two_i % 2 or tuple(out.shape) != (T, two_i // 2):
        raise ValueError("out must be [T, I] for x [T, 2I]")
    _check("nv_silu_and_mul", library().nv_silu_and_mul(
        _ptr(x), x.stride(0), _ptr(out), out.stride(0), T, two_i // 2, _stream(stream)))
