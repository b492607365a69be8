"""The softmax's polynomial base-2 exponential: the committed coefficients are what the Remez
generator produces, and the fp32 evaluation (range reduction + Horner + exponent insertion, as the
attention kernel does it) stays within the stated relative error of 2^x."""
import importlib.util
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "diffusion_transformer_denoiser_gb300", "csrc")


def _gen():
    spec = importlib.util.spec_from_file_location("gen_exp2_poly", os.path.join(CSRC, "gen_exp2_poly.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _header_coeffs():
    text = open(os.path.join(CSRC, "exp2_poly.h")).read()
    return [np.float32(float(v)) for v in re.findall(r"#define MI_EXP2_C\d ([-0-9.e]+)f", text)]


def test_header_matches_generator():
    g = _gen()
    c32 = np.array(g.remez(), dtype=np.float32)
    assert [float(v) for v in c32] == [float(v) for v in _header_coeffs()]


def _kernel_exp2(x):
    """fp32 emulation of exp2_poly2: clamp, rint by the 1.5*2^23 trick, Horner, exponent add."""
    c0, c1, c2, c3 = _header_coeffs()
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(-125.0))
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    n = (t - magic).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = (c3 * f + c2).astype(np.float32)
    p = (p * f + c1).astype(np.float32)
    p = (p * f + c0).astype(np.float32)
    bits = p.view(np.int32).astype(np.int64) + (t.view(np.int32).astype(np.int64) << 23)
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def test_poly_exp2_against_exp2():
    # the softmax feeds exponents in [-125, 8] (the stale max keeps them at most 2^3)
    x = np.concatenate([np.linspace(-125, 8, 2_000_001), np.arange(-125, 9, dtype=np.float64) + 0.5,
                        np.arange(-125, 9, dtype=np.float64)]).astype(np.float32)
    got = _kernel_exp2(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(got - ref) / ref
    assert rel.max() < 1.0e-4          # 2^-13: far below the bf16 rounding of P (2^-9)
    assert np.all(np.isfinite(got)) and np.all(got > 0)


def test_poly_exp2_stated_error():
    g = _gen()
    c32 = np.array(g.remez(), dtype=np.float32)
    assert g.fp32_horner_error(c32) < 8e-5
