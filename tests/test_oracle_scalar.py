"""Pins for the oracle's scalar arithmetic: the fp32 exponential / sigmoid
used for the sigmoid router's selection key, and bf16 rounding.

Each check compares against something other than the oracle itself: the
fp64 value of the same function (error bounds), closed forms, limits and
symmetries, or torch's own bf16 conversion.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def ulp32(v):
    v = np.abs(np.asarray(v, dtype=np.float64))
    v32 = v.astype(np.float32)
    return (np.nextafter(v32, np.float32(np.inf)).astype(np.float64) - v32.astype(np.float64))


def test_exp_closed_forms():
    assert oracle.exp_f32(0.0) == np.float32(1.0)
    assert oracle.exp_f32(-0.0) == np.float32(1.0)
    assert oracle.exp_f32(-np.inf) == np.float32(0.0)
    assert oracle.exp_f32(-200.0) == np.float32(0.0)
    # e^(-n ln2) is a power of two to within an ulp
    for n in (1, 2, 10, 50, 100, 126):
        got = float(oracle.exp_f32(np.float32(-n * math.log(2.0))))
        want = math.exp(float(np.float32(-n * math.log(2.0))))
        assert abs(got - want) <= ulp32(want)


def test_exp_accuracy_sweep():
    t = np.concatenate([np.linspace(-87.0, 0.0, 120001, dtype=np.float32),
                        np.random.default_rng(1).uniform(-87, 0, 50000).astype(np.float32)])
    got = oracle.exp_f32_array(t).astype(np.float64)
    want = np.exp(t.astype(np.float64))
    err = np.abs(got - want) / ulp32(want)
    assert err.max() <= 1.0, err.max()
    # a dropped Taylor term or a wrong ln2 tail moves the mean well above this
    assert err.mean() <= 0.35, err.mean()


def test_exp_subnormal_range():
    t = np.linspace(-103.9, -87.5, 20001, dtype=np.float32)
    got = oracle.exp_f32_array(t).astype(np.float64)
    want = np.exp(t.astype(np.float64))
    # results below 2^-126 lose precision gradually: allow one subnormal ulp
    assert np.max(np.abs(got - want)) <= 2.0 ** -149 + 1e-60


def test_sigmoid_closed_forms():
    assert oracle.sigmoid_f32(0.0) == np.float32(0.5)
    assert oracle.sigmoid_f32(-0.0) == np.float32(0.5)
    assert oracle.sigmoid_f32(np.inf) == np.float32(1.0)
    assert oracle.sigmoid_f32(-np.inf) == np.float32(0.0)
    assert oracle.sigmoid_f32(100.0) == np.float32(1.0)
    v = float(oracle.sigmoid_f32(-100.0))
    assert v > 0 and abs(v - math.exp(-100.0)) <= 2.0 ** -149


def test_sigmoid_accuracy_and_shape():
    x = np.concatenate([np.linspace(-80.0, 80.0, 200001, dtype=np.float32),
                        np.random.default_rng(2).standard_normal(100000).astype(np.float32) * 4])
    x = np.sort(x)
    got = oracle.sigmoid_f32_array(x)
    xd = x.astype(np.float64)
    want = 1.0 / (1.0 + np.exp(-xd))
    err = np.abs(got.astype(np.float64) - want) / ulp32(want)
    # e^-|x| carries <= 1 ulp, then one rounding each for 1+e and the
    # division: <= 2.5 ulp in the worst binade position, ~0.4 on average.
    assert err.max() <= 2.5, err.max()
    assert err.mean() <= 0.6, err.mean()
    # monotone non-decreasing
    assert np.all(np.diff(got.astype(np.float64)) >= 0)
    # symmetry sigma(-x) = 1 - sigma(x) for x >= 0 (within 2 ulps of 1)
    pos = x[x >= 0][::50]
    a = oracle.sigmoid_f32_array(pos).astype(np.float64)
    b = oracle.sigmoid_f32_array(-pos).astype(np.float64)
    assert np.max(np.abs(a + b - 1.0)) <= 2 * 2.0 ** -24 + 2.0 ** -24


def test_sigmoid_equals_tanh_form():
    # The pages define sigmoid as 0.5*tanh(0.5x)+0.5; same function in fp64.
    x = np.linspace(-20, 20, 4001, dtype=np.float32)
    got = oracle.sigmoid_f32_array(x).astype(np.float64)
    tanh_form = 0.5 * np.tanh(0.5 * x.astype(np.float64)) + 0.5
    assert np.max(np.abs(got - tanh_form)) <= 2.5 * 2.0 ** -24


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    # add exact ties and values that round up into the next binade
    ties = (np.arange(0, 4096, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    edge = np.array([65504.0, 3.3895314e38, -1.0e-40, 1.0e-45, 0.0, -0.0], dtype=np.float32)
    f = np.concatenate([f, ties, edge])
    got = oracle.f32_to_bf16_bits(f)
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_bf16_widening_is_exact():
    b = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    f = oracle.bf16_bits_to_f32(b)
    want = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    finite = np.isfinite(want)
    assert np.array_equal(f[finite].view(np.uint32), want[finite].view(np.uint32))
