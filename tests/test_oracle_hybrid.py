"""Pins of the oracle's hybrid recurrent step (CPU only).

Closed forms of the selective-state mixer (A -> -inf leaves only the new
input; dt -> 0 leaves the state untouched), the attention layers against the
already-pinned decoder step (a hybrid whose Mamba blocks add nothing equals
the decoder with its MLPs zeroed), batch invariance and the empty slot."""
import numpy as np

import oracle
import synth

W = synth.HYBRID_SMALL


def _bf16(v):
    return synth.f32_to_bf16_bits(np.asarray(v, dtype=np.float32))


def _mixer_inputs(seed=3):
    w = W
    rng = np.random.default_rng(seed)
    d, Hs = w.d_model, w.ssm_heads
    w_in = _bf16(rng.normal(0, 0.05, (w.in_rows, d)))
    xn = synth.bf16_bits_to_f32(_bf16(rng.normal(0, 1, d))).astype(np.float64)
    state = rng.normal(0, 1, (Hs, w.ssm_head_dim, w.ssm_state)).astype(np.float32)
    return w_in, xn, state


def _split(w, w_in, xn):
    zx = synth.bf16_bits_to_f32(w_in).astype(np.float64) @ xn
    di, N, Hs = w.d_inner, w.ssm_state, w.ssm_heads
    return zx[:di], zx[di:2 * di], zx[2 * di:2 * di + N], zx[2 * di + N:2 * di + 2 * N], zx[2 * di + 2 * N:]


def test_mixer_with_infinitely_fast_decay_keeps_only_the_new_input():
    w = W
    w_in, xn, state = _mixer_inputs()
    Hs, P = w.ssm_heads, w.ssm_head_dim
    a_log = _bf16(np.full(Hs, 30.0))            # A = -exp(30): exp(dt A) == 0
    dt_bias = _bf16(np.zeros(Hs))
    d_skip = _bf16(np.linspace(-1, 1, Hs))
    st = state.copy()
    out = oracle.ssm_mixer(w, w_in, a_log, dt_bias, d_skip, xn, st)
    z, x, B, C, dtr = _split(w, w_in, xn)
    for h in range(Hs):
        dt = np.log1p(np.exp(dtr[h])) if dtr[h] <= 0 else dtr[h] + np.log1p(np.exp(-dtr[h]))
        Dh = float(synth.bf16_bits_to_f32(d_skip[h:h + 1])[0])
        for p in range(P):
            xp = x[h * P + p]
            hn = (dt * B * xp).astype(np.float32)          # the new state is the input term alone
            assert np.array_equal(st[h, p], hn)
            y = np.dot(C, hn.astype(np.float64)) + Dh * xp
            zz = z[h * P + p]
            assert np.isclose(out[h * P + p], y * zz / (1 + np.exp(-zz)), rtol=1e-12, atol=1e-12)


def test_mixer_with_vanishing_step_leaves_the_state_alone():
    w = W
    w_in, xn, state = _mixer_inputs(4)
    Hs, P = w.ssm_heads, w.ssm_head_dim
    a_log = _bf16(np.zeros(Hs))
    dt_bias = _bf16(np.full(Hs, -120.0))        # dt = softplus(-120 + .) ~ 1e-52
    d_skip = _bf16(np.ones(Hs))
    st = state.copy()
    out = oracle.ssm_mixer(w, w_in, a_log, dt_bias, d_skip, xn, st)
    assert np.array_equal(st, state)
    z, x, B, C, dtr = _split(w, w_in, xn)
    for h in range(Hs):
        for p in range(P):
            y = np.dot(C, state[h, p].astype(np.float64)) + x[h * P + p]
            zz = z[h * P + p]
            assert np.isclose(out[h * P + p], y * zz / (1 + np.exp(-zz)), rtol=1e-12, atol=1e-12)


def test_attention_layers_equal_the_decoder_with_mlps_zeroed():
    # Mamba blocks with W_out = 0 add nothing to the residual, so the hybrid
    # reduces to its attention blocks; a decoder with the same attention
    # weights and zero MLP weights computes the same frame.
    w = W
    blob = synth.hybrid_weights_host(w)
    lay = synth.hybrid_layout(w)
    m = lay["mamba"]
    for l in range(w.n_layers):
        if not w.is_attn(l):
            b = synth.hybrid_layer_offset(w, l) + m["w_out"]
            blob[b: b + w.d_model * w.d_inner] = 0
    aw = w.attention_view()
    dec = synth.Workload("dec", w.n_attn, w.d_model, w.n_heads, w.head_dim, 64, S=w.S, T_max=w.T_max,
                         pos_lo=w.pos_lo, pos_hi=w.pos_hi)
    dl = synth.layer_layout(dec)
    dblob = np.zeros(synth.weight_elems(dec), dtype=np.uint16)
    a = lay["attn"]
    for la in range(w.n_attn):
        src = synth.hybrid_layer_offset(w, la * w.attn_every + w.attn_every - 1)
        dst = la * dl["layer"]
        dblob[dst + dl["g_attn"]: dst + dl["g_attn"] + w.d_model] = blob[src: src + w.d_model]
        dblob[dst + dl["wqkv"]: dst + dl["wo"] + w.d_model * w.HD] = blob[src + a["wqkv"]: src + a["size"]]
        dblob[dst + dl["g_mlp"]: dst + dl["g_mlp"] + w.d_model] = 0x3F80
    pos = synth.positions(aw, w.S)
    x = synth.x_bf16(aw, w.S)
    kv, sc, st = oracle.hybrid_prefill(w, list(range(w.S)), pos)
    kv2, sc2 = kv.copy(), sc.copy()
    y, ye = oracle.hybrid_step(w, blob, kv, sc, st, pos, x)
    y2, ye2, _ = oracle.step(dec, dblob, kv2, sc2, pos, x)
    assert np.array_equal(y, y2)
    assert np.array_equal(kv, kv2)


def test_sessions_are_independent_and_an_empty_slot_passes_through():
    w = W
    blob = synth.hybrid_weights_host(w)
    aw = w.attention_view()
    pos = synth.positions(aw, w.S).copy()
    pos[2] = -1
    x = synth.x_bf16(aw, w.S)
    kv, sc, st = oracle.hybrid_prefill(w, list(range(w.S)), pos)
    st0 = st.copy()
    y, _ = oracle.hybrid_step(w, blob, kv, sc, st, pos, x)
    assert np.array_equal(y[2], x[2])
    assert np.array_equal(st[:, 2], st0[:, 2])
    keep = [0, 1, 3, 4]
    kv1, sc1, st1 = oracle.hybrid_prefill(w, keep, pos[keep])
    y1, _ = oracle.hybrid_step(w, blob, kv1, sc1, st1, pos[keep], x[keep])
    assert np.array_equal(y[keep], y1)
    assert np.array_equal(st[:, keep], st1)
