"""Helpers for the GPU parity tests: device transfer of bf16 bit arrays and the
tolerance check the tests share.

Tolerance (floating-point outputs, bf16): with e_i = |gpu_i - ref_i| /
max(1, |ref_i|) against the fp64 oracle, max e <= 2e-2 and mean e <= 2e-3.
For |ref| <= 1 that is the absolute bound as stated; above 1 it grows with
the value, because rounding the output to bf16 alone already costs up to
2^-9 |ref| (0.031 at |ref| = 16).
"""
import numpy as np
import torch

import workloads as wl

MAX_TOL = 2e-2
MEAN_TOL = 2e-3


def dev(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bits (numpy) -> bf16 CUDA tensor of the same shape."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bits (numpy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def dev_i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def dev_i64(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).cuda()


def err_counter() -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# Every check_close result of the session, in order: (what, stats).  The
# conftest writes them out when NV_PARITY_LOG names a file.
PARITY_LOG = []


def check_close(gpu_bits: np.ndarray, ref: np.ndarray, what: str,
                max_tol: float = MAX_TOL, mean_tol: float = MEAN_TOL) -> dict:
    """Gate on e = |g - r| / max(1, |r|) (max and mean), and report beside it
    the plain absolute error |g - r| (max and mean), the stated metric."""
    g = wl.bf16_bits_to_f32(gpu_bits).astype(np.float64).reshape(ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    absdiff = np.abs(g - ref)
    e = absdiff / np.maximum(1.0, np.abs(ref))
    n = int(e.size)
    stats = dict(n=n,
                 max_err=float(e.max()) if n else 0.0,
                 mean_err=float(e.mean()) if n else 0.0,
                 max_abs=float(absdiff.max()) if n else 0.0,
                 mean_abs=float(absdiff.mean()) if n else 0.0,
                 max_ref=float(np.abs(ref).max()) if n else 0.0)
    PARITY_LOG.append((what, stats))
    print(f"[parity] {what}: n={n} max|err|={stats['max_abs']:.3e} "
          f"mean|err|={stats['mean_abs']:.3e} max e={stats['max_err']:.3e} "
          f"mean e={stats['mean_err']:.3e} max|ref|={stats['max_ref']:.2f}")
    assert stats["max_err"] <= max_tol, f"{what}: max err {stats}"
    assert stats["mean_err"] <= mean_tol, f"{what}: mean err {stats}"
    return stats


def check_close_rows(gpu_bits: np.ndarray, ref_rows, n_rows: int, what: str, chunk: int = 2048,
                     max_tol: float = MAX_TOL, mean_tol: float = MEAN_TOL) -> dict:
    """check_close over every row of a large output, computed in row chunks
    to bound host memory: ref_rows(lo, hi) returns the oracle's rows
    [lo, hi).  The statistics are those of the whole output."""
    n = 0
    acc = dict(max_err=0.0, sum_err=0.0, max_abs=0.0, sum_abs=0.0, max_ref=0.0)
    for lo in range(0, n_rows, chunk):
        hi = min(n_rows, lo + chunk)
        ref = ref_rows(lo, hi)
        g = wl.bf16_bits_to_f32(gpu_bits[lo:hi]).astype(np.float64).reshape(ref.shape)
        assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output in rows {lo}..{hi}"
        absdiff = np.abs(g - ref)
        e = absdiff / np.maximum(1.0, np.abs(ref))
        n += e.size
        acc["max_err"] = max(acc["max_err"], float(e.max()))
        acc["sum_err"] += float(e.sum())
        acc["max_abs"] = max(acc["max_abs"], float(absdiff.max()))
        acc["sum_abs"] += float(absdiff.sum())
        acc["max_ref"] = max(acc["max_ref"], float(np.abs(ref).max()))
    stats = dict(n=n, max_err=acc["max_err"], mean_err=acc["sum_err"] / max(1, n),
                 max_abs=acc["max_abs"], mean_abs=acc["sum_abs"] / max(1, n),
                 max_ref=acc["max_ref"])
    PARITY_LOG.append((what, stats))
    print(f"[parity] {what}: n={n} max|err|={stats['max_abs']:.3e} "
          f"mean|err|={stats['mean_abs']:.3e} max e={stats['max_err']:.3e} "
          f"mean e={stats['mean_err']:.3e} max|ref|={stats['max_ref']:.2f}")
    assert stats["max_err"] <= max_tol, f"{what}: max err {stats}"
    assert stats["mean_err"] <= mean_tol, f"{what}: mean err {stats}"
    return stats


def rope_table(max_position: int = wl.MAX_POSITION, base: float = wl.ROPE_BASE) -> torch.Tensor:
    import paged_kv_attention_kvcache_gb300 as nv
    t = torch.empty(max_position, 128, dtype=torch.float32, device="cuda")
    nv.nv_rope_cos_sin_cache(t, base)
    return t


# K rows reach the cache after the GPU rounds its fp32 rotation to bf16 and
# the oracle rounds its fp64 one.  Away from zero the two differ by at most
# one bf16 ulp (2^-7 |r| bounds it).  Near zero the rotation x*cos - y*sin
# cancels: its fp32 error scales with the terms (|x|, |y| ~ 1 after the
# norm; norm, table and products cost a few 2^-24 each, 1e-6 at worst), not
# with the small result, so an absolute 2^-16 is allowed on top.  A wrong
# sign, index or weight moves values by O(1) and still fails.
CACHE_ABS_TOL = 2.0 ** -16


def check_cache_rows(gpu_bits: np.ndarray, ref_bits: np.ndarray, what: str,
                     max_mismatch_frac: float = 0.01) -> None:
    g = wl.bf16_bits_to_f32(gpu_bits).astype(np.float64)
    r = wl.bf16_bits_to_f32(ref_bits).astype(np.float64)
    diff = np.abs(g - r)
    bad = diff > 2.0 ** -7 * np.abs(r) + CACHE_ABS_TOL
    if bad.any():
        idx = np.argwhere(bad)[:5]
        worst = [(tuple(int(v) for v in i), float(g[tuple(i)]), float(r[tuple(i)])) for i in idx]
        raise AssertionError(f"{what}: {int(bad.sum())} elements beyond one ulp; first {worst}")
    frac = float(np.mean(gpu_bits != ref_bits))
    assert frac < max_mismatch_frac, f"{what}: {frac:.4%} of elements differ by one ulp"
