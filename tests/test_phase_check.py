"""CPU pins of the phase-by-phase checker (tests/phase_check.py) used by the
GPU tests: records of a frame built with the oracle's own functions pass it,
and a record with one phase moved by 1% anywhere fails it."""
import numpy as np
import pytest

import oracle
import phase_check as pc
import synth


def _decoder_records(w, W, pos, x_bits, kv, sc):
    """One session's frame through the oracle's functions, every phase's
    input and output kept in the dump-record layout (fp32), the appended
    K/V written into kv / sc [L][2][H][T][D]."""
    d, HD, F, H, D = w.d_model, w.HD, w.ffn, w.n_heads, w.head_dim
    sec = pc.Sections(d, HD, F)
    lay = synth.layer_layout(w)
    recs = np.zeros((w.n_layers, sec.R), dtype=np.float32)
    r = synth.bf16_bits_to_f32(x_bits).astype(np.float64)
    for l in range(w.n_layers):
        b = l * lay["layer"]
        rec = recs[l]
        rec[sec.IN:sec.IN + d] = r
        xn = pc.bf16_round(oracle.rmsnorm(r, W[b + lay["g_attn"]: b + lay["g_attn"] + d], w.rms_eps))
        rec[sec.XN1:sec.XN1 + d] = xn
        qkv = oracle.matvec(W[b + lay["wqkv"]: b + lay["wqkv"] + 3 * HD * d].reshape(3 * HD, d), xn)
        rec[sec.PROJ:sec.PROJ + 3 * HD] = qkv
        for h in range(H):
            k = oracle.rope(qkv[HD + h * D: HD + (h + 1) * D], pos, w.rope_base)
            v = qkv[2 * HD + h * D: 2 * HD + (h + 1) * D]
            for which, row in ((0, k), (1, v)):
                c, s_ = oracle.quantize_rows(row.astype(np.float32)[None, :])
                kv[l, which, h, pos] = c[0]
                sc[l, which, h, pos] = s_[0]
        att = pc.bf16_round(pc._attention(w, qkv[:HD], pos, kv[l, 0], sc[l, 0], kv[l, 1], sc[l, 1]))
        rec[sec.MIX:sec.MIX + HD] = att
        r = r + oracle.matvec(W[b + lay["wo"]: b + lay["wo"] + d * HD].reshape(d, HD), att)
        rec[sec.MID:sec.MID + d] = r
        xn2 = pc.bf16_round(oracle.rmsnorm(r, W[b + lay["g_mlp"]: b + lay["g_mlp"] + d], w.rms_eps))
        rec[sec.XN2:sec.XN2 + d] = xn2
        gu = oracle.matvec(W[b + lay["wgu"]: b + lay["wgu"] + 2 * F * d].reshape(2 * F, d), xn2)
        u = pc.bf16_round(pc.silu(gu[:F]) * gu[F:])
        rec[sec.U:sec.U + F] = u
        r = r + oracle.matvec(W[b + lay["wdown"]: b + lay["wdown"] + d * F].reshape(d, F), u)
        rec[sec.OUT:sec.OUT + d] = r
        # the next layer reads the fp32 residual, as the GPU does
        r = rec[sec.OUT:sec.OUT + d].astype(np.float64)
    y = synth.f32_to_bf16_bits(pc.bf16_round(r).astype(np.float32))
    return recs, y


@pytest.fixture(scope="module")
def frame():
    w = synth.TINY
    W = synth.weights_host(w)
    pos = synth.positions(w, w.S)
    x = synth.x_bf16(w, w.S)
    kv, sc = oracle.prefill_history(w, [0], pos[:1], poison=True)
    kv1, sc1 = np.ascontiguousarray(kv[:, :, 0]), np.ascontiguousarray(sc[:, :, 0])
    recs, y = _decoder_records(w, W, int(pos[0]), x[0], kv1, sc1)
    return w, W, int(pos[0]), x[0], kv1, sc1, recs, y


def _check(frame, recs):
    w, W, pos, x, kv, sc, _, y = frame
    worst = {}
    pc.check_decoder_frame(w, W, recs, pos, kv, sc, x, y, worst)
    return worst


def test_oracle_records_pass_both_criteria(frame):
    worst = _check(frame, frame[6])
    assert all(v <= 1.0 for v in worst.values()), worst
    assert {"norm", "qkv", "attn", "o", "norm2", "gu", "down", "y"} <= set(worst)


@pytest.mark.parametrize("section,phase", [("PROJ", "qkv"), ("MIX", "attn"), ("U", "gu"), ("XN2", "norm2")])
def test_one_percent_off_in_one_phase_fails(frame, section, phase):
    w = frame[0]
    sec = pc.Sections(w.d_model, w.HD, w.ffn)
    recs = frame[6].copy()
    lo = getattr(sec, section)
    l = 1
    row = recs[l, lo:lo + 64]
    j = int(np.argmax(np.abs(row)))
    recs[l, lo + j] *= 1.01          # one element of one phase of one layer, 1% off
    worst = _check(frame, recs)
    assert worst[phase + "/tight"] > 1.0, worst


def test_a_dropped_residual_term_fails(frame):
    w = frame[0]
    sec = pc.Sections(w.d_model, w.HD, w.ffn)
    recs = frame[6].copy()
    # the residual after O recorded without the attention half's contribution
    recs[0, sec.MID:sec.MID + w.d_model] = recs[0, sec.IN:sec.IN + w.d_model]
    worst = _check(frame, recs)
    assert worst["o"] > 1.0
