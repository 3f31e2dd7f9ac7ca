"""The prefill softmax's FMA-pipe exponential (csrc/exp2_poly.cuh).

CPU: the header's coefficients are the Remez minimax fit that
csrc/fit_exp2_poly.py derives, and the kernel's exact fp32 sequence (sat
clamp, round-down range reduction, Horner cubic, exponent add), emulated
here step by step, stays within 9.0e-5 relative error of 2^x over the
softmax's argument range.  The bound is measured against the bf16 rounding
that P undergoes right after: half an ulp is 2^-9 = 1.95e-3 relative, 21x
larger.  GPU: the kernel's own inline function, through the C ABI, against
the MUFU's ex2.approx on the same scores.
"""
import importlib.util
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_attention_sink_gb300", "csrc")
BOUND = 9.0e-5


def _header_constants():
    text = open(os.path.join(CSRC, "exp2_poly.cuh")).read()
    consts = {}
    for name in ("kC0", "kC1", "kC2", "kC3"):
        m = re.search(rf"constexpr float {name} = (0x[0-9a-fA-F.]+p[-+]?\d+)f;", text)
        assert m, name
        consts[name] = np.float32(float.fromhex(m.group(1)))
    r = re.search(r"constexpr float kRange = ([\d.]+)f;", text)
    return [consts[f"kC{k}"] for k in range(4)], float(r.group(1))


def _fit_module():
    spec = importlib.util.spec_from_file_location("fit_exp2_poly", os.path.join(CSRC, "fit_exp2_poly.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def _fma(a, b, c):
    """fp32 fma: the product of two fp32 values is exact in fp64."""
    return _f32(np.asarray(a, np.float64) * np.asarray(b, np.float64) + np.asarray(c, np.float64))


def emulate(s, scale_log2, m):
    """The device sequence of exp2_poly.cuh, one fp32 rounding per step."""
    c, R = _header_constants()
    M = 12582912.0
    a = _f32(np.float32(scale_log2) * np.float32(1.0 / R))
    b = _fma(np.float32(-m), np.float32(1.0 / R), np.float32(0.5))
    y = _fma(s, a, b)
    y = np.clip(np.nan_to_num(y, nan=0.0), 0.0, 1.0).astype(np.float32)          # .sat
    t = np.floor(y.astype(np.float64) * R + (M - R / 2)).astype(np.float32)       # fma.rm
    u = _f32((M - R / 2) - t.astype(np.float64))                                  # exact
    f = _fma(y, np.float32(R), u)
    p = _fma(_fma(_fma(np.full_like(f, c[3]), f, c[2]), f, c[1]), f, c[0])
    bits = (p.view(np.uint32).astype(np.uint64) + (t.view(np.uint32).astype(np.uint64) << 23)) & 0xFFFFFFFF
    return bits.astype(np.uint32).view(np.float32)


def test_coefficients_are_the_remez_fit():
    (c, _), mod = _header_constants(), _fit_module()
    fit, err = mod.fit(3)
    assert abs(err - 7.478e-5) < 1e-7
    for k in range(4):
        assert np.float32(fit[k]) == c[k], (k, fit[k], c[k])


def test_remez_fit_equioscillates():
    """A minimax fit's error reaches +-E at degree + 2 alternating points."""
    mod = _fit_module()
    coef, err = mod.fit(3)
    g = np.linspace(0.0, 1.0, 400001)
    e = np.polyval(coef[::-1], g) / np.exp2(g) - 1.0
    assert abs(np.abs(e).max() - err) < 1e-9
    # sign changes of the error between its extrema: degree + 1 of them
    assert np.count_nonzero(np.diff(np.sign(e[np.abs(e) > 0.5 * err])) != 0) == 4


@pytest.mark.parametrize("scale_log2,m", [(1.0, 0.0), (0.18033688, 3.7), (0.18033688, -2.5), (0.127516, 40.0)])
def test_emulated_sequence_within_bound(scale_log2, m):
    x = np.linspace(-125.9, 8.5, 2_000_001)
    s = _f32((x + m) / scale_log2)
    got = emulate(s, scale_log2, m).astype(np.float64)
    want = np.exp2(s.astype(np.float64) * np.float64(np.float32(scale_log2)) - m)
    rel = np.abs(got / want - 1.0)
    assert rel.max() <= BOUND, rel.max()
    assert rel.max() < 2.0 ** -9 / 20   # far below bf16's half ulp


def test_emulated_sequence_edge_cases():
    s = np.array([-np.inf, -1e30, -200.0, -126.0, 0.0, 126.0, 300.0, np.inf, np.nan], dtype=np.float32)
    y = emulate(s, 1.0, 0.0).astype(np.float64)
    assert np.all(np.isfinite(y)) and np.all(y >= 0)
    assert np.all(y[:4] <= 2.0 ** -125)                 # at or below the clamp: negligible
    assert abs(y[4] - 1.0) <= BOUND                      # 2^0
    assert np.all(y[5:8] >= 2.0 ** 125)                  # clamped above at 2^126
    assert y[8] <= 2.0 ** -125                           # NaN clamps low


@pytest.mark.gpu
def test_gpu_polynomial_against_mufu():
    import torch
    from paged_kv_attention_sink_gb300 import binding
    for scale_log2, m in [(1.0, 0.0), (0.18033688, 3.7), (0.127516, -1.25)]:
        x = np.linspace(-125.0, 8.5, 1_000_003)
        s = _f32((x + m) / scale_log2)
        sd = torch.from_numpy(s).cuda()
        yp, ym = binding.attn_selftest_exp2(sd, scale_log2, m)
        torch.cuda.synchronize()
        yp = yp.cpu().numpy().astype(np.float64)
        ym = ym.cpu().numpy().astype(np.float64)
        want = np.exp2(s.astype(np.float64) * np.float64(np.float32(scale_log2)) - m)
        assert np.abs(yp / want - 1).max() <= BOUND
        # the MUFU's approximation plus the fp32 rounding of its argument
        # (half an ulp of |x| <= 128 is 2^-18, i.e. 2.6e-6 relative)
        assert np.abs(ym / want - 1).max() <= 4e-6
        assert np.abs(yp / ym - 1).max() <= BOUND + 4e-6
        # the device sequence is the one emulated above, bit for bit or within one fp32 ulp
        ye = emulate(s, scale_log2, m).astype(np.float64)
        assert np.abs(yp / ye - 1).max() <= 2.0 ** -22
    # masked scores and the clamp ends
    s = torch.tensor([-np.inf, -1e30, -300.0, 0.0, 300.0, np.inf], dtype=torch.float32, device="cuda")
    yp, ym = binding.attn_selftest_exp2(s, 1.0, 0.0)
    yp = yp.cpu().numpy().astype(np.float64)
    assert np.all(yp[:3] <= 2.0 ** -125) and np.all(yp[:3] >= 0)
    assert abs(yp[3] - 1.0) <= BOUND
    assert np.all(yp[4:] >= 2.0 ** 125) and np.all(np.isfinite(yp[4:]))
