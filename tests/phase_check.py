"""Phase-by-phase checks of one session's step against the oracle's own
functions, fed with the GPU's inputs to that phase (the activation-dump
testing hook records every phase's input and output).  Because each phase is
checked on its own inputs, no one-ulp flip of an earlier bf16 rounding can
cascade into the comparison: every phase of every layer is held to the
stated element-wise bound |got - ref| <= 1e-3 + 2e-2 |ref| at any depth and
width.  Test infrastructure only."""
from __future__ import annotations

import numpy as np

import oracle
import synth

ATOL, RTOL = 1e-3, 2e-2


def bf16_round(a) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 (ties to even), once."""
    u = np.ascontiguousarray(a, dtype=np.float64).view(np.uint64)
    u = (u + np.uint64((1 << 44) - 1) + ((u >> np.uint64(45)) & np.uint64(1))) & ~np.uint64((1 << 45) - 1)
    return u.view(np.float64)


def silu(g):
    return g / (1.0 + np.exp(-g))


def ratio(got, ref) -> float:
    """Worst |got - ref| / (atol + rtol |ref|) over the elements (<= 1 passes)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape and np.all(np.isfinite(got)), (got.shape, ref.shape)
    return float(np.max(np.abs(got - ref) / (ATOL + RTOL * np.abs(ref))))


# The tight criterion: a phase's fp32 output within 2e-5 of the row's largest
# reference value of the fp64 reference (fp32 accumulation against fp64), a
# bf16 output within one bf16 step (2^-8 relative) of the unrounded
# reference plus the same floor.  A phase off by 1% anywhere fails it.
TIGHT_FLOOR = 2e-5


def tight(got, u, rounded: bool) -> float:
    got = np.asarray(got, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    bound = TIGHT_FLOOR * np.max(np.abs(u)) + (2.0 ** -8 * np.abs(u) if rounded else 0.0) + 1e-30
    return float(np.max(np.abs(got - u) / bound))


def note(worst, name, got, u, rounded):
    """Record phase `name`: got against the reference u (fp64, before the
    bf16 rounding when the phase rounds), under both criteria."""
    ref = bf16_round(u) if rounded else np.asarray(u, dtype=np.float64)
    worst[name] = max(worst.get(name, 0.0), ratio(got, ref))
    worst[name + "/tight"] = max(worst.get(name + "/tight", 0.0), tight(got, u, rounded))


class Sections:
    """Offsets of a dump record's sections (see wave_debug_dump_acts)."""

    def __init__(self, d, HD, F=0, in_rows=0, d_inner=0):
        n1, n2 = max(3 * HD, in_rows), max(HD, d_inner)
        self.IN, self.XN1, self.PROJ = 0, d, 2 * d
        self.MIX = 2 * d + n1
        self.MID = self.MIX + n2
        self.XN2 = self.MID + d
        self.U = self.XN2 + d
        self.OUT = self.U + F
        self.R = self.OUT + d


def _attention(w, q_all, pos, kc, ks, vc, vs):
    """Attention of every head (fp64, before the bf16 rounding), q before
    RoPE (fp64 [H*D]); kc/vc [H][T][D] codes and ks/vs [H][T] scales as the
    GPU read them."""
    H, D = w.n_heads, w.head_dim
    out = np.empty(H * D)
    for h in range(H):
        q = oracle.rope(q_all[h * D:(h + 1) * D], pos, w.rope_base)
        out[h * D:(h + 1) * D] = oracle.attention_head(q, kc[h, :pos + 1], ks[h, :pos + 1], vc[h, :pos + 1],
                                                       vs[h, :pos + 1], pos)
    return out


def attention_block(w, sec, rec, g, wqkv, wo, pos, kc, ks, vc, vs, worst, tag):
    """norm -> QKV -> attention -> O of one layer's record; updates worst."""
    d, HD = w.d_model, w.n_heads * w.head_dim
    r_in = rec[sec.IN:sec.IN + d].astype(np.float64)
    xn = rec[sec.XN1:sec.XN1 + d].astype(np.float64)
    note(worst, tag + "norm", xn, oracle.rmsnorm(r_in, g, w.rms_eps), True)
    qkv = rec[sec.PROJ:sec.PROJ + 3 * HD].astype(np.float64)
    note(worst, tag + "qkv", qkv, oracle.matvec(wqkv, xn), False)
    att = rec[sec.MIX:sec.MIX + HD].astype(np.float64)
    note(worst, tag + "attn", att, _attention(w, qkv[:HD], pos, kc, ks, vc, vs), True)
    return r_in + oracle.matvec(wo, att)


def decoder_layer(w, W, l, rec, pos, kc, ks, vc, vs, next_in, worst):
    """Every phase of decoder layer l for one session.  rec: the layer's
    record; kc/ks/vc/vs: the layer's history [H][T][D] / [H][T] as read
    (slot pos holds the appended K/V); next_in: the output residual the
    next phase saw (the next layer's input, fp32) or None for the last
    layer.  Returns the reference output residual (fp64)."""
    d, HD, F = w.d_model, w.HD, w.ffn
    sec = Sections(d, HD, F)
    lay = synth.layer_layout(w)
    b = l * lay["layer"]
    g1 = W[b + lay["g_attn"]: b + lay["g_attn"] + d]
    wqkv = W[b + lay["wqkv"]: b + lay["wqkv"] + 3 * HD * d].reshape(3 * HD, d)
    wo = W[b + lay["wo"]: b + lay["wo"] + d * HD].reshape(d, HD)
    g2 = W[b + lay["g_mlp"]: b + lay["g_mlp"] + d]
    wgu = W[b + lay["wgu"]: b + lay["wgu"] + 2 * F * d].reshape(2 * F, d)
    wdown = W[b + lay["wdown"]: b + lay["wdown"] + d * F].reshape(d, F)
    mid_ref = attention_block(w, sec, rec, g1, wqkv, wo, pos, kc, ks, vc, vs, worst, "")
    mid = rec[sec.MID:sec.MID + d].astype(np.float64)
    note(worst, "o", mid, mid_ref, False)
    xn2 = rec[sec.XN2:sec.XN2 + d].astype(np.float64)
    note(worst, "norm2", xn2, oracle.rmsnorm(mid, g2, w.rms_eps), True)
    gu = oracle.matvec(wgu, xn2)
    u = rec[sec.U:sec.U + F].astype(np.float64)
    note(worst, "gu", u, silu(gu[:F]) * gu[F:], True)
    out_ref = mid + oracle.matvec(wdown, u)
    if next_in is not None:
        note(worst, "down", next_in, out_ref, False)
    return out_ref


def check_decoder_frame(w, W, recs, pos, kv, sc, x_bits, y_bits, worst):
    """All layers of one session's frame: recs [L][R]; kv [L][2][H][T][D],
    sc [L][2][H][T] the history as read (appended slot included); x_bits /
    y_bits the session's input and output rows."""
    L, d = w.n_layers, w.d_model
    sec = Sections(d, w.HD, w.ffn)
    # the first layer's input is x itself, and every later layer's input is
    # the previous layer's recorded output, bit for bit
    assert np.array_equal(recs[0, :d], synth.bf16_bits_to_f32(x_bits))
    for l in range(1, L):
        assert np.array_equal(recs[l, :d], recs[l - 1, sec.OUT:sec.OUT + d])
    for l in range(L):
        nxt = recs[l + 1, :d].astype(np.float64) if l + 1 < L else None
        out_ref = decoder_layer(w, W, l, recs[l], int(pos), kv[l, 0], sc[l, 0], kv[l, 1], sc[l, 1], nxt, worst)
    note(worst, "y", synth.bf16_bits_to_f32(y_bits), out_ref, True)


def check_hybrid_frame(w, blob, recs, pos, kv, sc, state_old, state_new, x_bits, y_bits, worst):
    """All layers of one session's hybrid frame: recs [L][R]; kv / sc the
    attention blocks' history [La][2][H][T][D] as read; state_old /
    state_new [Lm][Hs][P][N] before and after the frame."""
    L, d, e = w.n_layers, w.d_model, w.attn_every
    HD, di = w.HD, w.d_inner
    sec = Sections(d, HD, 0, w.in_rows, di)
    lay = synth.hybrid_layout(w)
    assert np.array_equal(recs[0, :d], synth.bf16_bits_to_f32(x_bits))
    for l in range(1, L):
        assert np.array_equal(recs[l, :d], recs[l - 1, sec.MID:sec.MID + d])
    for l in range(L):
        b = synth.hybrid_layer_offset(w, l)
        g = blob[b:b + d]
        nxt = recs[l + 1, :d].astype(np.float64) if l + 1 < L else None
        if w.is_attn(l):
            a = lay["attn"]
            la = l // e
            wqkv = blob[b + a["wqkv"]: b + a["wqkv"] + 3 * HD * d].reshape(3 * HD, d)
            wo = blob[b + a["wo"]: b + a["wo"] + d * HD].reshape(d, HD)
            out_ref = attention_block(w, sec, recs[l], g, wqkv, wo, int(pos), kv[la, 0], sc[la, 0], kv[la, 1],
                                      sc[la, 1], worst, "a_")
            key = "a_o"
        else:
            m = lay["mamba"]
            lm = l - l // e
            w_in = blob[b + m["w_in"]: b + m["w_in"] + w.in_rows * d].reshape(w.in_rows, d)
            w_out = blob[b + m["w_out"]: b + m["w_out"] + d * di].reshape(d, di)
            prm = blob[b + m["a_log"]: b + m["a_log"] + 3 * w.ssm_heads]
            r_in = recs[l, sec.IN:sec.IN + d].astype(np.float64)
            xn = recs[l, sec.XN1:sec.XN1 + d].astype(np.float64)
            note(worst, "s_norm", xn, oracle.rmsnorm(r_in, g, w.rms_eps), True)
            zx = recs[l, sec.PROJ:sec.PROJ + w.in_rows].astype(np.float64)
            note(worst, "s_in", zx, oracle.matvec(w_in, xn), False)
            st = np.ascontiguousarray(state_old[lm], dtype=np.float32).copy()
            gated = oracle.ssm_update(w, zx, prm[:w.ssm_heads], prm[w.ssm_heads:2 * w.ssm_heads],
                                      prm[2 * w.ssm_heads:], st)
            note(worst, "s_state", state_new[lm], st, False)
            mix = recs[l, sec.MIX:sec.MIX + di].astype(np.float64)
            note(worst, "s_mix", mix, gated, True)
            out_ref = r_in + oracle.matvec(w_out, mix)
            key = "s_out"
        if nxt is not None:
            note(worst, key, nxt, out_ref, False)
    note(worst, "y", synth.bf16_bits_to_f32(y_bits), out_ref, True)
