"""CPU pins of how the fp64 oracle treats non-finite inputs (the reading the
GPU tests in test_nonfinite_gpu.py compare against).

The recurrence of "Mamba: Linear-Time Sequence Modeling with Selective State
Spaces" (section "Method") makes each state depend on every earlier input of
its row and on B, C of its batch, and on nothing else; so a NaN planted at one
(row, step) must leave earlier steps and all other rows bit-identical to the
clean run, and make every later output of that row NaN. With softplus,
delta = -inf gives dt = 0: the decay is 1 and the input term 0, so that step
leaves the state unchanged.
"""
import numpy as np

import oracle
import workloads


def _cfg():
    return workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=2, dim=8, seqlen=48, seed=93)


def _run(inp, cfg):
    shp = (cfg.batch, cfg.dim, cfg.seqlen)
    y, h = oracle.scan_fwd(inp["u"].reshape(shp), inp["delta"].reshape(shp), inp["A"], inp["B"],
                           inp["C"], D=inp["D"], delta_bias=inp["delta_bias"],
                           z=inp["z"].reshape(shp))
    return y.reshape(cfg.rows, cfg.seqlen), h.reshape(cfg.rows, cfg.dstate)


def _bits(v):
    return workloads.f32_to_bf16_bits(np.array([v], dtype=np.float32))[0]


def test_nan_in_u_poisons_the_rest_of_its_row_only():
    cfg = _cfg()
    clean = workloads.scan_inputs(cfg)
    y0, h0 = _run(clean, cfg)
    bad = workloads.scan_inputs(cfg)
    r, l0 = cfg.dim + 3, 20
    bad["u"][r, l0] = _bits(np.nan)
    y1, h1 = _run(bad, cfg)
    others = np.ones(cfg.rows, bool)
    others[r] = False
    assert np.array_equal(y1[others], y0[others]) and np.array_equal(h1[others], h0[others])
    assert np.array_equal(y1[r, :l0], y0[r, :l0])
    assert np.all(np.isnan(y1[r, l0:])) and np.all(np.isnan(h1[r]))


def test_nan_in_B_poisons_its_batch_from_that_step():
    """B[b, n, l0] = NaN: state n of every row of batch b is NaN from l0 on (the
    other states are untouched), so every later output of that batch is NaN."""
    cfg = _cfg()
    y0, h0 = _run(workloads.scan_inputs(cfg), cfg)
    bad = workloads.scan_inputs(cfg)
    l0 = 31
    bad["B"][1, 4, l0] = _bits(np.nan)
    y1, h1 = _run(bad, cfg)
    b0 = slice(0, cfg.dim)
    b1 = slice(cfg.dim, 2 * cfg.dim)
    assert np.array_equal(y1[b0], y0[b0])
    assert np.array_equal(y1[b1, :l0], y0[b1, :l0])
    assert np.all(np.isnan(y1[b1, l0:]))
    assert np.all(np.isnan(h1[b1, 4]))
    keep = np.arange(cfg.dstate) != 4
    assert np.array_equal(h1[b1][:, keep], h0[b1][:, keep]) and np.array_equal(h1[b0], h0[b0])


def test_negative_infinite_delta_is_a_step_that_changes_nothing():
    cfg = _cfg()
    inp = workloads.scan_inputs(cfg)
    r, l0 = 5, 17
    inp["delta"][r, l0] = _bits(-np.inf)
    y, h = _run(inp, cfg)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(h))
    # the state after step l0 equals the state before it: with u = 0 at l0 the
    # output there is the contraction of the unchanged state, gate applied
    inp2 = workloads.scan_inputs(cfg)
    inp2["delta"][r, l0] = _bits(-np.inf)
    inp2["u"][r, l0] = 0
    y2, _ = _run(inp2, cfg)
    # state entering step l0: the same inputs cut after l0 steps
    cut = lambda x: np.ascontiguousarray(x[..., :l0])
    _, ht = oracle.scan_fwd(cut(inp2["u"][r:r + 1]), cut(inp2["delta"][r:r + 1]), inp2["A"],
                            cut(inp2["B"]), cut(inp2["C"]), D=inp2["D"],
                            delta_bias=inp2["delta_bias"], z=cut(inp2["z"][r:r + 1]),
                            rows=np.array([r]), dim=cfg.dim)
    Cv = workloads.bf16_bits_to_f32(inp2["C"][r // cfg.dim, :, l0]).astype(np.float64)
    z = float(workloads.bf16_bits_to_f32(inp2["z"][r, l0:l0 + 1])[0])
    silu = z / (1.0 + np.exp(-z))
    expect = float(np.dot(Cv, ht[0])) * silu
    assert abs(y2[r, l0] - expect) <= 1e-12 * (1.0 + abs(expect))
