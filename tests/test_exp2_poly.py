"""The FMA-pipe exponential of the SM-pair extend kernel (host only): its cubic is the minimax fit
that fit_exp2.py derives, and the kernel's steps -- clamp at -127, round-to-nearest through
1.5 * 2^23, cubic in f = x - n, 2^n from exponent bits -- replayed in float32 give 2^x within the
fit's relative error (plus float32 rounding) on [-125, 8], and exactly 0 for -inf and x <= -127."""
import os
import re

import numpy as np

from prefix_shared_kv_gb300 import fit_exp2

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KERNEL = os.path.join(ROOT, "prefix_shared_kv_gb300", "csrc", "extend_pair.cu")


def kernel_coefficients():
    text = open(KERNEL).read()
    return [float(re.search(rf"kExpC{i} = ([0-9.eE+-]+)f;", text).group(1)) for i in range(4)]


def test_kernel_coefficients_are_the_minimax_fit():
    ours = kernel_coefficients()
    fit = fit_exp2.float32_coefficients()
    assert np.allclose(ours, fit, rtol=0, atol=1e-9)
    assert fit_exp2.max_rel_error(ours) < 7.6e-5
    # a lower degree would not do for bf16 P (half an ulp: 2^-9)
    _, e2 = fit_exp2.remez(2)
    assert e2 > 2.0 ** -10


def exp2_steps(x):
    """The kernel's exp2_poly2, step by step, in float32."""
    f32 = np.float32
    x = np.maximum(np.asarray(x, np.float32), f32(-127.0))
    k = f32(12582912.0)
    t = (x + k).astype(np.float32)
    nf = (t - k).astype(np.float32)
    f = (x - nf).astype(np.float32)
    c0, c1, c2, c3 = (f32(c) for c in kernel_coefficients())
    p = ((f * c3 + c2) * f + c1) * f + c0
    e = ((t.view(np.uint32) - np.uint32(0x4B400000) + np.uint32(127)) << np.uint32(23)).astype(
        np.uint32)
    return (p.astype(np.float32) * e.view(np.float32)).astype(np.float32)


def test_reduction_and_cubic_give_two_to_the_x():
    x = np.concatenate([np.linspace(-125.0, 8.0, 2000001, dtype=np.float32),
                        np.arange(-125, 9, dtype=np.float32),
                        np.arange(-125, 8, dtype=np.float32) + np.float32(0.5)])
    y = exp2_steps(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(y / ref - 1.0)) < 7.5e-5 + 4 * 2.0 ** -24
    assert exp2_steps(np.float32(0.0)) == np.float32(fit_exp2.float32_coefficients()[0])


def test_masked_and_underflowing_inputs_give_zero():
    z = exp2_steps(np.array([-np.inf, -1e30, -200.0, -127.0, -126.6], np.float32))
    assert (z == 0.0).all() and not np.signbit(z).any()
