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


def _blob_with_live_parameters(w, seed=11):
    """The synthetic blob with every selective-state block's dt_bias and D
    drawn away from their defaults (0 and 1), so that each enters the
    frame with a non-trivial value; W_out and A_log as generated."""
    blob = synth.hybrid_weights_host(w)
    lay = synth.hybrid_layout(w)["mamba"]
    rng = np.random.default_rng(seed)
    for l in range(w.n_layers):
        if w.is_attn(l):
            continue
        b = synth.hybrid_layer_offset(w, l)
        blob[b + lay["dt_bias"]: b + lay["dt_bias"] + w.ssm_heads] = _bf16(rng.normal(0, 0.7, w.ssm_heads))
        blob[b + lay["d_skip"]: b + lay["d_skip"] + w.ssm_heads] = _bf16(rng.normal(1, 0.5, w.ssm_heads))
    return blob


def test_hybrid_step_matches_independent_torch_restatement():
    # every block at work: non-zero W_out, A_log ~ N(0, 1), dt_bias and D
    # away from their defaults; the restatement has its own layout arithmetic,
    # softplus, state update and FP8 codec (PyTorch's float8_e4m3fn)
    import torch_ref
    w = W
    blob = _blob_with_live_parameters(w)
    aw = w.attention_view()
    pos = synth.positions(aw, w.S).copy()
    pos[3] = -1  # an empty slot too
    x = synth.x_bf16(aw, w.S)
    kv, sc, st = oracle.hybrid_prefill(w, list(range(w.S)), pos)
    kv2, sc2, st2 = kv.copy(), sc.copy(), st.copy()
    _, ye = oracle.hybrid_step(w, blob, kv, sc, st, pos, x)
    ref = torch_ref.hybrid_step(w, blob, kv2, sc2, st2, pos, x)
    assert np.allclose(ye, ref, rtol=1e-9, atol=1e-9), float(np.max(np.abs(ye - ref)))
    assert np.array_equal(kv, kv2)
    assert np.array_equal(np.nan_to_num(sc, nan=-1.0), np.nan_to_num(sc2, nan=-1.0))
    assert np.allclose(st, st2, rtol=2.0 ** -22, atol=0), float(np.max(np.abs(st - st2)))


def test_selective_state_blocks_carry_weight_in_the_pinned_frame():
    # the comparison above is not vacuous: dropping every selective-state
    # block's output (W_out = 0) or its state (zeros) moves y far beyond the
    # restatement's agreement
    w = W
    blob = _blob_with_live_parameters(w)
    aw = w.attention_view()
    pos = synth.positions(aw, w.S)
    x = synth.x_bf16(aw, w.S)
    kv, sc, st = oracle.hybrid_prefill(w, list(range(w.S)), pos)
    _, ye = oracle.hybrid_step(w, blob, kv.copy(), sc.copy(), st.copy(), pos, x)
    cut = blob.copy()
    m = synth.hybrid_layout(w)["mamba"]
    for l in range(w.n_layers):
        if not w.is_attn(l):
            b = synth.hybrid_layer_offset(w, l) + m["w_out"]
            cut[b: b + w.d_model * w.d_inner] = 0
    _, ye_cut = oracle.hybrid_step(w, cut, kv.copy(), sc.copy(), st.copy(), pos, x)
    _, ye_zero = oracle.hybrid_step(w, blob, kv.copy(), sc.copy(), np.zeros_like(st), pos, x)
    scale = np.max(np.abs(ye))
    assert np.max(np.abs(ye - ye_cut)) > 1e-2 * scale
    assert np.max(np.abs(ye - ye_zero)) > 1e-2 * scale
