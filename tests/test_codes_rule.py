"""The end-to-end code rule of the GPU tests (gpu_case.codes_vs_oracle),
checked on the CPU with the oracle alone: rows moved by a known amount and
requantised pass it, with many codes moved; a code moved off a rounding
boundary, or by two steps, on rows that agree exactly, fails it."""
import numpy as np
import pytest

import oracle
import synth
from gpu_case import codes_vs_oracle


@pytest.fixture(scope="module")
def tiny_step():
    w = synth.TINY
    W = synth.weights_host(w)
    pos = synth.positions(w)
    x = synth.x_bf16(w)
    sess = list(range(w.S))
    kv, sc = oracle.prefill_history(w, sess, pos, poison=True)
    _, _, kv_new = oracle.step(w, W, kv, sc, pos, x[sess], want_kv_new=True)
    return pos, kv, sc, kv_new


def test_requantised_nearby_rows_pass(tiny_step):
    pos, kv, sc, kv_new = tiny_step
    rng = np.random.default_rng(0)
    moved = 0
    for j in range(len(pos)):
        P = int(pos[j])
        pre = kv_new[:, :, j].astype(np.float32)
        amax = np.max(np.abs(pre), axis=-1, keepdims=True)
        g_pre = (pre + rng.normal(0, 3e-4, pre.shape) * amax).astype(np.float32)
        g_codes, _ = oracle.quantize_rows(np.ascontiguousarray(g_pre))
        moved += codes_vs_oracle(g_codes, g_pre, kv[:, :, j, :, P], sc[:, :, j, :, P], kv_new[:, :, j])
    assert moved > 0


@pytest.mark.parametrize("step", [1, 2])
def test_a_moved_code_on_exact_rows_fails(tiny_step, step):
    pos, kv, sc, kv_new = tiny_step
    P = int(pos[0])
    bad = kv[:, :, 0, :, P].copy()
    c = int(bad[1, 0, 2, 7])
    m = c & 0x7F
    bad[1, 0, 2, 7] = (c & 0x80) | (m + step if m + step <= 0x7E else m - step)
    exact = kv_new[:, :, 0].astype(np.float64)
    with pytest.raises(AssertionError):
        codes_vs_oracle(bad, exact, kv[:, :, 0, :, P], sc[:, :, 0, :, P], exact)
