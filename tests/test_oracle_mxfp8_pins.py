"""Pins of the oracle's MXFP8 activation mode (the live-quantisation variant).

The E4M3 element format is pinned against the OCP spec's anchor values and
against PyTorch's float8_e4m3fn (an independent implementation of the same
format); the MX block conversion against closed forms, its error bound and
idempotence; the layer mode against a dense numpy formulation that
quantises x before the gate/up projection and h before the down projection.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_moe_gb300 import inputs

from test_oracle_pins import bf16_f64, dense_decode, expert_of, random_layer, silu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def torch_e4m3_values():
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def torch_e4m3_round(v):
    return torch.from_numpy(np.asarray(v, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


# ------------------------------------------------------------------- E4M3

def test_e4m3_matches_ocp_anchors_and_torch_table():
    with open(os.path.join(GOLDEN, "e4m3_ocp_anchors.txt")) as f:
        rows = [ln.split("#", 1)[0].split() for ln in f]
    anchors = {int(r[0], 16): float(r[1]) for r in rows if r}
    assert len(anchors) == 16
    for code, v in anchors.items():
        got = oracle.e4m3_value(code)
        assert got == v and math.copysign(1.0, got) == math.copysign(1.0, v), hex(code)
    ours = np.array([oracle.e4m3_value(b) for b in range(256)])
    ref = torch_e4m3_values()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.isnan(ours).sum() == 2                      # 0x7F and 0xFF
    fin = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[fin], ref[fin])
    assert np.all(np.diff(ours[:127]) > 0)                # codes 0..126 increase


def test_e4m3_round_matches_torch_inside_the_range():
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(20000) * np.exp2(rng.integers(-14, 9, 20000))).astype(np.float32)
    grid = np.array([oracle.e4m3_value(b) for b in range(0x7F)])
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)     # exact ties
    v = np.concatenate([v, mids, -mids, grid.astype(np.float32)])
    v = v[np.abs(v) < 448]
    ours = np.array([oracle.e4m3_round(float(x)) for x in v], dtype=np.uint8)
    np.testing.assert_array_equal(ours, torch_e4m3_round(v))


def test_e4m3_round_ties_to_even_and_saturates():
    assert oracle.e4m3_round(1.0625) == 0x38               # between 1.0 and 1.125: even mantissa 0
    assert oracle.e4m3_round(1.1875) == 0x3A               # between 1.125 and 1.25: even mantissa 2
    assert oracle.e4m3_round(0.0009765625) == 0x00         # half the smallest subnormal: even 0
    assert oracle.e4m3_round(0.0029296875) == 0x02         # 1.5 quanta: even 2
    for v in (448.0, 460.0, 470.0, 1e6):
        assert oracle.e4m3_round(v) == 0x7E
        assert oracle.e4m3_round(-v) == 0xFE
    assert oracle.e4m3_round(-0.0) == 0x80


# ------------------------------------------------------- MX block conversion

def test_mxfp8_closed_forms():
    grid = np.array([oracle.e4m3_value(b) for b in range(0x7F)])
    rng = np.random.default_rng(4)
    # block 0: values on the E4M3 grid times 2^-20 with max 256 * 2^-20:
    # shared exponent floor(log2(2^-12)) - 8 = -20, every element exact
    b0 = rng.choice(grid[grid <= 256], 32) * rng.choice([-1.0, 1.0], 32)
    b0[5] = 256.0
    b0 = b0 * 2.0 ** -20
    # block 1: max 500 -> exponent 0, 500 clamps to 448
    b1 = np.zeros(32)
    b1[0], b1[1] = 500.0, 3.0
    # block 2: all zero -> exponent -127 (scale byte 0), codes 0
    b2 = np.zeros(32)
    # block 3: max 2^-130 -> exponent clamped to -127; 2^-130 / 2^-127 = 1/8 -> 0x20
    b3 = np.zeros(32)
    b3[31] = 2.0 ** -130
    codes, scales, deq = oracle.mxfp8_quantize(np.concatenate([b0, b1, b2, b3]))
    assert list(scales) == [107, 127, 0, 0]
    np.testing.assert_array_equal(deq[:32], b0)
    assert codes[32] == 0x7E and deq[32] == 448.0 and deq[33] == 3.0
    assert np.all(codes[64:96] == 0) and np.all(deq[64:96] == 0.0)
    assert codes[127] == 0x20 and deq[127] == 2.0 ** -130


def test_mxfp8_error_bound_and_idempotence():
    rng = np.random.default_rng(5)
    v = rng.standard_normal(32 * 64) * np.repeat(np.exp2(rng.integers(-30, 30, 64)), 32)
    codes, scales, deq = oracle.mxfp8_quantize(v)
    X = np.repeat(np.exp2(scales.astype(np.float64) - 127.0), 32)
    amax = np.abs(v.reshape(-1, 32)).max(axis=1)
    assert np.all(np.repeat(amax, 32) / X >= 256) and np.all(np.repeat(amax, 32) / X < 512)
    normal = np.abs(v) / X >= 2.0 ** -6
    err = np.abs(deq - v)
    below = np.abs(v) / X <= 448
    assert np.all(err[normal & below] <= 2.0 ** -4 * np.abs(v[normal & below]))
    assert np.all(err[~normal] <= 2.0 ** -10 * X[~normal])
    c2, s2, d2 = oracle.mxfp8_quantize(deq)
    # re-quantising lands on the same values (a clamped block max may lower its scale)
    np.testing.assert_array_equal(d2, deq)


# -------------------------------------------------------------- layer mode

def dense_mx_layer(x, ids, w, bank):
    xd = bf16_f64(x)
    T, H = xd.shape
    I = bank["w13"].shape[1] // 2
    y = np.zeros((T, H))
    hs = np.zeros((T, ids.shape[1], I))
    for t in range(T):
        xq = oracle.mxfp8_quantize(xd[t])[2]
        for s, e in enumerate(ids[t]):
            W13 = dense_decode(bank["w13"][e], bank["s13"][e])
            W2 = dense_decode(bank["w2"][e], bank["s2"][e])
            h = silu(W13[:I] @ xq) * (W13[I:] @ xq)
            hs[t, s] = h
            y[t] += w[t, s] * (W2 @ oracle.mxfp8_quantize(h)[2])
    return y, hs


def test_mx_layer_matches_dense_formulation():
    x, wr, b, bank = random_layer(T=3, H=64, E=6, k=2, I=64)
    got = oracle.layer_forward(x, wr, b, 2, expert_of(bank), act="mxfp8", want_h=True)
    y, hs = dense_mx_layer(x, got["ids"], got["w"], bank)
    np.testing.assert_allclose(got["h"], hs, rtol=1e-12, atol=1e-12 * np.abs(hs).max())
    np.testing.assert_allclose(got["y"], y, rtol=1e-11, atol=1e-11 * np.abs(y).max())
    exact = oracle.layer_forward(x, wr, b, 2, expert_of(bank))
    assert not np.array_equal(got["y"], exact["y"])      # the mode does change the result


def test_mx_layer_gate_up_is_exact_when_x_is_on_the_mxfp8_grid():
    x, wr, b, bank = random_layer(T=2, H=64, E=4, k=2, I=32)
    xd = bf16_f64(x)
    xq = np.stack([oracle.mxfp8_quantize(r)[2] for r in xd])
    x = inputs.f32_to_bf16_bits(xq.astype(np.float32))       # E4M3 * 2^s is exact in bf16
    assert np.array_equal(bf16_f64(x), xq)
    mx = oracle.layer_forward(x, wr, b, 2, expert_of(bank), act="mxfp8", want_h=True)
    ex = oracle.layer_forward(x, wr, b, 2, expert_of(bank), want_h=True)
    np.testing.assert_array_equal(mx["h"], ex["h"])
    rel = np.abs(mx["y"] - ex["y"]).max() / np.abs(ex["y"]).max()
    assert 0 < rel < 0.1
