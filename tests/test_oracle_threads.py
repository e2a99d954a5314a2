"""The oracle's backward with its rows split over threads equals the
single-threaded run: per-row gradients bit for bit, sums over rows (dA, dB,
dC, dD, ddelta_bias) to fp64 rounding (only their addition order differs)."""
import numpy as np

import oracle
import workloads


def test_threaded_backward_equals_single_thread():
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=3, dim=40, seqlen=64, seed=5)
    inp = workloads.scan_inputs(cfg, with_h0=True)
    shp = (cfg.batch, cfg.dim, cfg.seqlen)
    g = np.random.default_rng(1)
    dy = g.standard_normal(shp)
    dh = g.standard_normal((cfg.batch, cfg.dim, cfg.dstate))
    kw = dict(D=inp["D"], delta_bias=inp["delta_bias"], z=inp["z"].reshape(shp),
              h0=inp["h0"].reshape(cfg.batch, cfg.dim, cfg.dstate), dh_last=dh)
    args = (inp["u"].reshape(shp), inp["delta"].reshape(shp), inp["A"], inp["B"], inp["C"], dy)
    one = oracle.scan_bwd(*args, **kw)
    many = oracle.scan_bwd(*args, threads=7, **kw)
    for k in ("du", "ddelta", "dz", "dh0"):
        assert np.array_equal(one[k], many[k]), k
    for k in ("dA", "dB", "dC", "dD", "ddelta_bias"):
        assert np.allclose(one[k], many[k], rtol=1e-13, atol=1e-13 * np.max(np.abs(one[k]))), k
