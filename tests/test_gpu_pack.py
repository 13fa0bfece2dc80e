"""GPU: wave_pack_weights / wave_hybrid_pack_weights against a numpy
restatement of the packed layout (include/wave.h): every projection matrix
as 128-row x 64-input blocks, tile-major then block-major, zero beyond the
matrix, gate/up tiles pairing 64 gate rows with the 64 matching up rows;
vectors copied.  Bit for bit, on shapes with ragged rows and inputs."""
import numpy as np
import pytest
import torch

import frame_step_decode_gb300 as fsd
import synth

pytestmark = pytest.mark.gpu


def _pack(W, rows, gu_F=0):
    """W [N][K] (bf16 bits) -> packed blocks, rows: the tile row count (128,
    or 64 per half for gate/up)."""
    N, K = W.shape
    ku = -(-K // 128)
    if gu_F:
        tiles = -(-gu_F // 64)
        full = np.zeros((tiles * 128, ku * 128), dtype=np.uint16)
        for t in range(tiles):
            g = W[t * 64: min(gu_F, t * 64 + 64)]
            u = W[gu_F + t * 64: gu_F + min(gu_F, t * 64 + 64)]
            full[t * 128: t * 128 + g.shape[0], :K] = g
            full[t * 128 + 64: t * 128 + 64 + u.shape[0], :K] = u
    else:
        tiles = -(-N // 128)
        full = np.zeros((tiles * 128, ku * 128), dtype=np.uint16)
        full[:N, :K] = W
    return full.reshape(tiles, 128, 2 * ku, 64).transpose(0, 2, 1, 3).reshape(-1)


def _packed_decoder(w, blob):
    lay = synth.layer_layout(w)
    d, HD, F = w.d_model, w.HD, w.ffn
    out = []
    for l in range(w.n_layers):
        b = l * lay["layer"]
        m = lambda name, n, k: blob[b + lay[name]: b + lay[name] + n * k].reshape(n, k)
        out += [blob[b + lay["g_attn"]: b + lay["g_attn"] + d], _pack(m("wqkv", 3 * HD, d), 128),
                _pack(m("wo", d, HD), 128), blob[b + lay["g_mlp"]: b + lay["g_mlp"] + d],
                _pack(m("wgu", 2 * F, d), 64, gu_F=F), _pack(m("wdown", d, F), 128)]
    return np.concatenate(out)


# ragged in every dimension the packing pads: F = 1376 (gate/up tiles,
# down inputs), 3HD = 384 + HD = 128 (a QKV tile exactly), d = 320
RAGGED = synth.Workload("ragged-2L-d320-h1x128-f1376", 2, 320, 1, 128, 1376, S=3, T_max=64, pos_lo=0, pos_hi=64)


@pytest.mark.parametrize("w", [synth.TINY, synth.MID, RAGGED], ids=["tiny", "mid", "ragged"])
def test_pack_weights_matches_the_layout(w):
    cfg = fsd.WaveConfig.of(w)
    blob = synth.weights_host(w)
    src = torch.from_numpy(blob.view(np.int16)).to("cuda").view(torch.bfloat16)
    dst = torch.full((fsd.packed_weights_bytes(cfg) // 2,), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    fsd.pack_weights(cfg, src, dst)
    torch.cuda.synchronize()
    got = dst.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = _packed_decoder(w, blob)
    assert got.size == ref.size
    assert np.array_equal(got, ref)


def test_hybrid_pack_weights_matches_the_layout():
    w = synth.HYBRID_SMALL
    cfg = fsd.WaveHybridConfig.of(w)
    blob = synth.hybrid_weights_host(w)
    src = torch.from_numpy(blob.view(np.int16)).to("cuda").view(torch.bfloat16)
    dst = torch.zeros(fsd.hybrid_packed_weights_bytes(cfg) // 2, dtype=torch.bfloat16, device="cuda")
    fsd.hybrid_pack_weights(cfg, src, dst)
    torch.cuda.synchronize()
    got = dst.view(torch.int16).cpu().numpy().view(np.uint16)
    lay = synth.hybrid_layout(w)
    d, di, HD, Hs = w.d_model, w.d_inner, w.HD, w.ssm_heads
    parts = []
    for l in range(w.n_layers):
        b = synth.hybrid_layer_offset(w, l)
        parts.append(blob[b:b + d])
        if w.is_attn(l):
            a = lay["attn"]
            parts += [_pack(blob[b + a["wqkv"]: b + a["wqkv"] + 3 * HD * d].reshape(3 * HD, d), 128),
                      _pack(blob[b + a["wo"]: b + a["wo"] + d * HD].reshape(d, HD), 128)]
        else:
            m = lay["mamba"]
            small = np.zeros((3 * Hs + 7) // 8 * 8, dtype=np.uint16)
            small[:3 * Hs] = blob[b + m["a_log"]: b + m["a_log"] + 3 * Hs]
            parts += [_pack(blob[b + m["w_in"]: b + m["w_in"] + w.in_rows * d].reshape(w.in_rows, d), 128),
                      _pack(blob[b + m["w_out"]: b + m["w_out"] + d * di].reshape(d, di), 128), small]
    ref = np.concatenate(parts)
    assert got.size == ref.size
    # the padding after A_log, dt_bias, D is never written: compare the rest
    mask = np.ones(ref.size, dtype=bool)
    o = 0
    for l in range(w.n_layers):
        if w.is_attn(l):
            o += d + _pack(np.zeros((3 * HD, d), np.uint16), 128).size + _pack(np.zeros((d, HD), np.uint16), 128).size
        else:
            o += d + _pack(np.zeros((w.in_rows, d), np.uint16), 128).size + _pack(np.zeros((d, di), np.uint16), 128).size
            n_small = (3 * Hs + 7) // 8 * 8
            mask[o + 3 * Hs: o + n_small] = False
            o += n_small
    assert np.array_equal(got[mask], ref[mask])


def test_ragged_shape_step_matches_oracle():
    # the step on the padded packing of a ragged shape, against the oracle
    from gpu_case import DeviceCase, oracle_reference, y_close
    case = DeviceCase(RAGGED)
    wave = fsd.Wave(case.cfg, case.S_max, RAGGED.T_max)
    try:
        case.step(wave)
        assert wave.status() == fsd.WAVE_OK
        _, y_exact, _, _, _ = oracle_reference(RAGGED, range(case.S), case.pos_h, case.x_h)
        ok, worst = y_close(case.y_bits(), y_exact)
        assert ok, worst
    finally:
        wave.close()
