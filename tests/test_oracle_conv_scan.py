"""CPU pins of the oracle's convolution-then-scan composition.

A width-W filter with a single unit tap and no bias or activation is a pure
delay: tap W-1 passes x through unchanged, tap W-2 shifts it one step later
(the step before 0 taken from the initial state). The composition must then
equal the scan oracle run directly on x, or on the shifted x, which pins the
causal alignment of the filter and the hand-over of its initial state."""
import numpy as np

import oracle
import workloads


def _inputs(W, in_dtype="bf16"):
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=2, dim=12, seqlen=40, seed=41,
                           in_dtype=in_dtype)
    inp = workloads.scan_inputs(cfg)
    shp = (cfg.batch, cfg.dim, cfg.seqlen)
    return cfg, inp, shp


def test_unit_last_tap_is_the_plain_scan():
    for W in (2, 3, 4):
        cfg, inp, shp = _inputs(W)
        w = np.zeros((cfg.dim, W), np.float32)
        w[:, W - 1] = 1.0
        x = inp["u"].reshape(shp)
        y, h, u, fs = oracle.conv_scan_fwd(x, w, inp["delta"].reshape(shp), inp["A"], inp["B"],
                                           inp["C"], conv_silu=False, D=inp["D"],
                                           delta_bias=inp["delta_bias"], z=inp["z"].reshape(shp))
        y0, h0 = oracle.scan_fwd(x, inp["delta"].reshape(shp), inp["A"], inp["B"], inp["C"],
                                 D=inp["D"], delta_bias=inp["delta_bias"], z=inp["z"].reshape(shp))
        assert np.array_equal(y, y0) and np.array_equal(h, h0)
        xf = workloads.bf16_bits_to_f32(x).astype(np.float64)
        assert np.array_equal(u, xf)
        assert np.array_equal(fs, xf[:, :, cfg.seqlen - (W - 1):])


def test_unit_previous_tap_delays_by_one_step_with_the_initial_state():
    W = 4
    cfg, inp, shp = _inputs(W, "f32")
    w = np.zeros((cfg.dim, W), np.float32)
    w[:, W - 2] = 1.0
    x = inp["u"].reshape(shp).astype(np.float32)
    init = np.random.default_rng(3).standard_normal((cfg.batch, cfg.dim, W - 1)).astype(np.float32)
    y, h, u, _ = oracle.conv_scan_fwd(x, w, inp["delta"].reshape(shp), inp["A"], inp["B"],
                                      inp["C"], conv_init=init, conv_silu=False,
                                      D=inp["D"], delta_bias=inp["delta_bias"],
                                      z=inp["z"].reshape(shp))
    shifted = np.concatenate([init[:, :, W - 2:W - 1], x[:, :, :-1]], axis=2)
    y0, h0 = oracle.scan_fwd(np.ascontiguousarray(shifted), inp["delta"].reshape(shp), inp["A"],
                             inp["B"], inp["C"], D=inp["D"], delta_bias=inp["delta_bias"],
                             z=inp["z"].reshape(shp))
    assert np.array_equal(u, shifted.astype(np.float64))
    assert np.array_equal(y, y0) and np.array_equal(h, h0)
