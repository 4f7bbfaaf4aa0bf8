"""GPU parity of SiluAndMul ("3.3 Model skeleton and core operators", sec. 4)
against the fp64 oracle: the page's toy shape, Qwen3-0.6B and Qwen3-8B
intermediate sizes (3072 and 12288), strided and in-place views, a ragged
tail of vectors that does not fill the last wave, and saturated gates."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import check_close, check_close_rows, dev, host

pytestmark = pytest.mark.gpu

import paged_kv_attention_kvcache_gb300 as nv  # noqa: E402


def _run(x_bits, pad=0):
    T, two_i = x_bits.shape
    buf = np.zeros((T, two_i + pad), np.uint16)
    buf[:, :two_i] = x_bits
    x = dev(buf)[:, :two_i]
    out = torch.empty(T, two_i // 2, dtype=torch.bfloat16, device="cuda")
    nv.nv_silu_and_mul(x, out)
    torch.cuda.synchronize()
    return host(out)


def test_silu_and_mul_page_toy_shape():
    x = wl.normal_bf16(800, "sw.toy", (5, 16), 0.0, 2.0)
    check_close(_run(x), oracle.silu_and_mul(x), "swiglu toy")


@pytest.mark.parametrize("T,I,pad", [(37, 3072, 0), (37, 3072, 16), (1, 8, 0), (513, 1032, 8)])
def test_silu_and_mul_shapes_and_strides(T, I, pad):
    x = wl.normal_bf16(801 + T, "sw.x", (T, 2 * I), 0.0, 2.0)
    check_close(_run(x, pad), oracle.silu_and_mul(x), f"swiglu {T}x{I} pad {pad}")


def test_silu_and_mul_in_place_into_gate_half():
    T, I = 64, 3072
    x_bits = wl.normal_bf16(810, "sw.inplace", (T, 2 * I))
    x = dev(x_bits)
    nv.nv_silu_and_mul(x, x[:, :I])
    torch.cuda.synchronize()
    got = host(x)
    check_close(got[:, :I], oracle.silu_and_mul(x_bits), "swiglu in place")
    assert np.array_equal(got[:, I:], x_bits[:, I:]), "up half must stay untouched"


def test_silu_and_mul_saturated_gates():
    # gates far into both tails: silu -> g above, -> 0 below (no NaN from e^-g)
    g = np.array([-1e4, -200.0, -90.0, -20.0, 0.0, 20.0, 90.0, 200.0, 1e4], np.float32)
    T, I = g.size, 8
    x = np.zeros((T, 2 * I), np.float32)
    x[:, :I] = g[:, None]
    x[:, I:] = 1.5
    xb = wl.f32_to_bf16_bits(x)
    check_close(_run(xb), oracle.silu_and_mul(xb), "swiglu saturated")


def test_silu_and_mul_qwen3_8b_full_size():
    # The MLP activation of the Qwen3-8B prefill batch: ~33k tokens x 2*12288,
    # every output element compared (the oracle runs in row chunks).
    pre = wl.config4()
    T, I = pre.qkv.shape[0], 12288
    x = wl.normal_bf16(820, "sw.8b", (T, 2 * I))
    got = _run(x)
    check_close_rows(got, lambda lo, hi: oracle.silu_and_mul(x[lo:hi]), T,
                     "swiglu 8b (33k tokens x 12288)")
