"""The fp64 oracle against what the mathematics fixes (CPU only)."""
import math
import os

import numpy as np
import pytest

import pins
import workloads


@pytest.mark.parametrize("name", sorted(pins.ALL_PINS))
def test_pin(oracle_mod, name):
    err = pins.ALL_PINS[name](oracle_mod)
    assert err <= pins.PIN_TOL.get(name, pins.DEFAULT_TOL), (name, err)


def test_softplus_identities(oracle_mod):
    sp = oracle_mod.softplus
    assert sp(0.0) == pytest.approx(math.log(2.0), rel=1e-15)
    for x in np.linspace(-40, 40, 161):
        # softplus(x) - softplus(-x) = x
        assert sp(x) - sp(-x) == pytest.approx(x, abs=1e-13)
        # exp(softplus(x)) - 1 = exp(x)  (softplus is log(1 + e^x))
        if abs(x) < 30:
            assert math.expm1(sp(x)) == pytest.approx(math.exp(x), rel=1e-13)
    # asymptotes
    assert sp(-60.0) == pytest.approx(math.exp(-60.0), rel=1e-13)
    assert sp(60.0) == 60.0
    # derivative is the logistic sigmoid (central difference)
    for x in (-3.0, -0.5, 0.0, 0.7, 4.0):
        hstep = 1e-5
        deriv = (sp(x + hstep) - sp(x - hstep)) / (2 * hstep)
        assert deriv == pytest.approx(1 / (1 + math.exp(-x)), abs=1e-9)


def test_silu_identities(oracle_mod):
    si = oracle_mod.silu
    assert si(0.0) == 0.0
    for z in np.linspace(-30, 30, 121):
        # silu(z) - silu(-z) = z
        assert si(z) - si(-z) == pytest.approx(z, abs=1e-12)
        assert si(z) == pytest.approx(z * 0.5 * (1 + math.tanh(z / 2)), abs=1e-14)
    assert si(-800.0) == 0.0  # no overflow


def test_golden_gated_rnn_halving(oracle_mod):
    """Hand-derived case in tests/golden (see the fixture for its derivation)."""
    path = os.path.join(os.path.dirname(__file__), "golden", "gated_rnn_halving.txt")
    rows = [ln.split("#")[0].split() for ln in open(path) if ln.split("#")[0].strip()]
    kv = {r[0]: r[1:] for r in rows}
    u = np.array([[list(map(float, kv["u"]))]], dtype=np.float32)
    L = u.shape[-1]
    zeros = np.zeros_like(u)
    ones = np.ones_like(u)
    y, hl = oracle_mod.scan_fwd(u, zeros, -np.ones((1, 1), np.float32), ones, ones, z=None)
    ln2 = math.log(2.0)
    expect = [eval(e, {"ln2": ln2}) for e in kv["y"]]
    assert len(expect) == L
    np.testing.assert_allclose(y[0, 0], expect, rtol=1e-15, atol=1e-16)
    assert hl[0, 0, 0] == pytest.approx(expect[-1], rel=1e-15)


def test_bf16_inputs_widen_exactly(oracle_mod):
    c = pins.small_case(seed=21, L=16)
    bits = {k: workloads.f32_to_bf16_bits(c[k]) for k in ("u", "delta", "B", "C", "z")}
    wide = {k: workloads.bf16_bits_to_f32(bits[k]).reshape(c[k].shape) for k in bits}
    ya, ha = oracle_mod.scan_fwd(bits["u"], bits["delta"], c["A"], bits["B"], bits["C"], D=c["D"],
                                 delta_bias=c["delta_bias"], z=bits["z"])
    yb, hb = oracle_mod.scan_fwd(wide["u"], wide["delta"], c["A"], wide["B"], wide["C"], D=c["D"],
                                 delta_bias=c["delta_bias"], z=wide["z"])
    assert np.array_equal(ya, yb) and np.array_equal(ha, hb)


def test_row_subset_matches_full(oracle_mod):
    cfg = workloads.scaled(workloads.CONFIGS["mamba130m"], batch=2, dim=24, seqlen=96)
    full = workloads.scan_inputs(cfg)
    y, hl = oracle_mod.scan_fwd(full["u"].reshape(2, 24, 96), full["delta"].reshape(2, 24, 96),
                                full["A"], full["B"], full["C"], D=full["D"],
                                delta_bias=full["delta_bias"], z=full["z"].reshape(2, 24, 96))
    rows = [0, 5, 23, 24, 47]
    sub = workloads.scan_inputs(cfg, rows=rows)
    assert np.array_equal(sub["u"], full["u"][rows])
    ys, hs = oracle_mod.scan_fwd(sub["u"], sub["delta"], sub["A"], sub["B"], sub["C"], D=sub["D"],
                                 delta_bias=sub["delta_bias"], z=sub["z"], rows=rows, dim=24)
    assert np.array_equal(ys, y.reshape(48, 96)[rows])
    assert np.array_equal(hs, hl.reshape(48, 16)[rows])


def test_threads_do_not_change_results(oracle_mod):
    c = pins.small_case(seed=22, batch=3, dim=5, L=33)
    y1, h1 = oracle_mod.scan_fwd(c["u"], c["delta"], c["A"], c["B"], c["C"], D=c["D"],
                                 delta_bias=c["delta_bias"], z=c["z"], threads=1)
    y4, h4 = oracle_mod.scan_fwd(c["u"], c["delta"], c["A"], c["B"], c["C"], D=c["D"],
                                 delta_bias=c["delta_bias"], z=c["z"], threads=4)
    assert np.array_equal(y1, y4) and np.array_equal(h1, h4)


def test_empty_sequence(oracle_mod):
    c = pins.small_case(seed=23, L=1, with_h0=True)
    e = lambda a: a[..., :0].copy()
    y, hl = oracle_mod.scan_fwd(e(c["u"]), e(c["delta"]), c["A"], e(c["B"]), e(c["C"]),
                                D=c["D"], delta_bias=c["delta_bias"], z=e(c["z"]), h0=c["h0"])
    assert y.shape[-1] == 0
    assert np.array_equal(hl, c["h0"])
