"""Pins of the oracle's whole step (CPU only).

Closed forms (zero weights give y = x; a one-hot input writes a known K row),
invariants (batch invariance, slots beyond pos never read), and an
independent PyTorch fp64 restatement on small shapes.
"""
import numpy as np
import pytest

import oracle
import synth
import torch_ref

SMALL = synth.Workload("small-2L-d128-h2x64-f160", 2, 128, 2, 64, 160, S=3, T_max=16, pos_lo=0, pos_hi=16)


def _inputs(w, S=None, poison=True):
    S = w.S if S is None else S
    pos = synth.positions(w, S)
    x = synth.x_bf16(w, S)
    kv, sc = oracle.prefill_history(w, list(range(S)), pos, poison=poison)
    return pos, x, kv, sc


@pytest.mark.parametrize("w", [SMALL, synth.TINY])
def test_step_matches_independent_torch_restatement(w):
    W = synth.weights_host(w)
    pos, x, kv, sc = _inputs(w)
    kv2, sc2 = kv.copy(), sc.copy()
    y, y_exact, _ = oracle.step(w, W, kv, sc, pos, x)
    ref = torch_ref.step(w, W, kv2, sc2, pos, x)
    assert np.allclose(y_exact, ref, rtol=1e-9, atol=1e-9)
    assert np.array_equal(kv, kv2)
    assert np.array_equal(np.nan_to_num(sc, nan=-1.0), np.nan_to_num(sc2, nan=-1.0))


def test_step_zero_projections_return_x_and_write_zero_rows():
    w = SMALL
    W = synth.weights_host(w)
    lay = synth.layer_layout(w)
    for l in range(w.n_layers):
        b = l * lay["layer"]
        for name, n in (("wqkv", 3 * w.HD * w.d_model), ("wo", w.d_model * w.HD),
                        ("wgu", 2 * w.ffn * w.d_model), ("wdown", w.d_model * w.ffn)):
            W[b + lay[name]: b + lay[name] + n] = 0
    pos, x, kv, sc = _inputs(w)
    y, _, _ = oracle.step(w, W, kv, sc, pos, x)
    assert np.array_equal(y, x)
    for j, P in enumerate(pos):
        assert np.all(kv[:, :, j, :, P, :] == 0) and np.all(sc[:, :, j, :, P] == 0)


def test_step_one_hot_input_writes_known_key_row():
    # x = c e_j: RMSNorm with gain 1 gives xn = bf16(c / sqrt(c^2/d + eps)) e_j,
    # so k = Wk[:, j] * xn_j, rotated at pos and quantised per head.
    w = SMALL
    W = synth.weights_host(w)
    lay = synth.layer_layout(w)
    d, HD, H, D = w.d_model, w.HD, w.n_heads, w.head_dim
    j, c, P = 37, 2.0, 5
    x = np.zeros((1, d), dtype=np.uint16)
    x[0, j] = 0x4000  # bf16 2.0
    pos = np.array([P], dtype=np.int32)
    kv, sc = oracle.prefill_history(w, [0], pos)
    oracle.step(w, W, kv, sc, pos, x)
    L = oracle.lib()
    xn = L.oracle_bf16_round(c / np.sqrt(c * c / d + w.rms_eps))
    Wq = synth.bf16_bits_to_f32(W[lay["wqkv"]: lay["wqkv"] + 3 * HD * d]).astype(np.float64).reshape(3 * HD, d)
    for h in range(H):
        k = Wq[HD + h * D: HD + (h + 1) * D, j] * xn
        v = Wq[2 * HD + h * D: 2 * HD + (h + 1) * D, j] * xn
        k = oracle.rope(k, P)
        ck, sk = oracle.quantize_rows(k.astype(np.float32)[None])
        cv, sv = oracle.quantize_rows(v.astype(np.float32)[None])
        assert np.array_equal(kv[0, 0, 0, h, P], ck[0]) and sc[0, 0, 0, h, P] == sk[0]
        assert np.array_equal(kv[0, 1, 0, h, P], cv[0]) and sc[0, 1, 0, h, P] == sv[0]


def test_step_batch_invariance():
    w = SMALL
    W = synth.weights_host(w)
    pos, x, kv, sc = _inputs(w)
    y_all, e_all, _ = oracle.step(w, W, kv, sc, pos, x)
    for j in range(w.S):
        p1, x1 = pos[j:j + 1].copy(), x[j:j + 1].copy()
        kv1, sc1 = oracle.prefill_history(w, [j], p1)
        y1, e1, _ = oracle.step(w, W, kv1, sc1, p1, x1)
        assert np.array_equal(y1[0], y_all[j]) and np.array_equal(e1[0], e_all[j])
        assert np.array_equal(kv1[:, :, 0], kv[:, :, j])


def test_step_never_reads_slots_beyond_position():
    w = SMALL
    W = synth.weights_host(w)
    pos, x, kv, sc = _inputs(w, poison=True)
    _, _, kvz, scz = _inputs(w, poison=False)
    y1, e1, _ = oracle.step(w, W, kv, sc, pos, x)
    y2, e2, _ = oracle.step(w, W, kvz, scz, pos, x)
    assert np.all(np.isfinite(e1))
    assert np.array_equal(e1, e2)


def test_rounded_and_pure_fp64_variants_agree_closely():
    w = SMALL
    W = synth.weights_host(w)
    pos, x, kv, sc = _inputs(w)
    _, e1, _ = oracle.step(w, W, kv.copy(), sc.copy(), pos, x, round_acts=True)
    _, e2, _ = oracle.step(w, W, kv.copy(), sc.copy(), pos, x, round_acts=False)
    assert np.max(np.abs(e1 - e2)) / np.max(np.abs(e2)) < 2e-2


def test_step_rejects_out_of_range_position():
    w = SMALL
    W = synth.weights_host(w)
    pos, x, kv, sc = _inputs(w)
    bad = pos.copy()
    bad[1] = w.T_max
    with pytest.raises(ValueError):
        oracle.step(w, W, kv, sc, bad, x)


def test_empty_slot_passes_x_through_and_leaves_the_others_alone():
    # A negative position marks a place of the fixed-shape batch with no
    # session in it: y = x bit for bit, its cache untouched, and the other
    # sessions' results and cache writes equal to a batch without that place.
    w = synth.TINY
    W = synth.weights_host(w)
    pos, x, kv, sc = _inputs(w)
    pos = pos.copy()
    pos[1] = -1
    kv, sc = oracle.prefill_history(w, list(range(w.S)), pos, poison=True)
    kv0, sc0 = kv.copy(), sc.copy()
    y, y_exact, kv_new = oracle.step(w, W, kv, sc, pos, x, want_kv_new=True)
    assert np.array_equal(y[1], x[1])
    assert np.array_equal(y_exact[1], synth.bf16_bits_to_f32(x[1]).astype(np.float64))
    assert np.array_equal(kv[:, :, 1], kv0[:, :, 1])
    assert np.array_equal(sc[:, :, 1].view(np.uint32), sc0[:, :, 1].view(np.uint32))
    assert np.all(np.isnan(kv_new[:, :, 1]))
    keep = [0, 2, 3]
    kv2, sc2 = oracle.prefill_history(w, keep, pos[keep], poison=True)
    y2, _, _ = oracle.step(w, W, kv2, sc2, pos[keep], x[keep])
    assert np.array_equal(y[keep], y2)
    assert np.array_equal(kv[:, :, keep], kv2)
    assert np.array_equal(sc[:, :, keep].view(np.uint32), sc2.view(np.uint32))


def test_position_at_t_max_is_refused():
    w = synth.TINY
    W = synth.weights_host(w)
    pos, x, kv, sc = _inputs(w)
    pos = pos.copy()
    pos[2] = w.T_max
    with pytest.raises(ValueError):
        oracle.step(w, W, kv, sc, pos, x)
