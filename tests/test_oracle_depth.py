"""Pins of the oracle's inner depth loop (CPU only): the projection between
steps against an independent numpy restatement (fp64 product, then
round-to-nearest-even to bf16 written here from the format's definition), and
the loop's wiring against an identity projection."""
import numpy as np

import oracle
import synth

DEPTH_SMALL = synth.Workload("depth-small-2L-d128-h2x64-f160", 2, 128, 2, 64, 160, S=3, T_max=8,
                             pos_lo=0, pos_hi=8)


def _bf16_rne(v: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bits, round to nearest even on the 8-bit significand
    (normal range only, as in these tests)."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)                      # v = m 2^e, |m| in [0.5, 1)
    q = np.round(m * 256.0)                 # numpy rounds halves to even
    r = np.ldexp(q / 256.0, e).astype(np.float32)
    return (r.view(np.uint32) >> 16).astype(np.uint16)


def test_projection_matches_numpy_restatement():
    w = DEPTH_SMALL
    d = w.d_model
    rng = np.random.default_rng(7)
    wp = _bf16_rne(rng.normal(0, 1 / np.sqrt(d), (d, d)))
    y = _bf16_rne(rng.normal(0, 1, (5, d)))
    got = oracle.proj(w, wp, y)
    ref = _bf16_rne(synth.bf16_bits_to_f32(y).astype(np.float64) @ synth.bf16_bits_to_f32(wp).astype(np.float64).T)
    assert np.array_equal(got, ref)


def test_depth_loop_with_identity_projection_chains_outputs_into_inputs():
    w = DEPTH_SMALL
    d, n, steps = w.d_model, 2, 5
    W = synth.weights_host(w)
    eye = np.zeros((d, d), dtype=np.uint16)
    eye[np.arange(d), np.arange(d)] = 0x3F80   # bf16 1.0
    x0 = synth.x_bf16(w, n)
    ys, ye, xs = oracle.depth_loop(w, W, eye, x0, steps)
    assert np.array_equal(xs[0], x0)
    for k in range(1, steps):
        assert np.array_equal(xs[k], ys[k - 1])     # W_p = I: x_k = y_{k-1} exactly
    # the same chain by hand: fresh cache, step k at depth position k
    L, H, T, D = w.n_layers, w.n_heads, w.T_max, w.head_dim
    kv = np.full((L, 2, n, H, T, D), 0x7F, dtype=np.uint8)
    sc = np.full((L, 2, n, H, T), np.nan, dtype=np.float32)
    x = x0
    for k in range(steps):
        y, _, _ = oracle.step(w, W, kv, sc, np.full(n, k, dtype=np.int32), x)
        assert np.array_equal(y, ys[k])
        x = y


def test_depth_loop_sessions_are_independent():
    w = DEPTH_SMALL
    W = synth.weights_host(w)
    wp = synth.proj_host(w)
    x0 = synth.x_bf16(w, 3)
    ys, _, _ = oracle.depth_loop(w, W, wp, x0, 4)
    ys1, _, _ = oracle.depth_loop(w, W, wp, x0[1:2], 4)
    assert np.array_equal(ys[:, 1:2], ys1)
