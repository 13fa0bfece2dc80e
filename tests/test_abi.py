"""CPU: the step library builds, loads, and exports every symbol that
include/wave.h declares (no compute call: there may be no GPU here)."""
import os
import re

import pytest

import frame_step_decode_gb300 as fsd
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    with open(os.path.join(ROOT, "include", "wave.h")) as f:
        txt = f.read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(wave_[a-z_0-9]+)\s*\(", txt)))


def test_library_exports_every_declared_symbol():
    L = fsd.lib()
    names = declared_symbols()
    assert len(names) >= 13
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(fsd.EXPORTS)


def test_weight_layout_matches_the_generator_layout():
    import synth
    for w in (synth.TINY, synth.SEVEN_B, synth.MID):
        cfg = fsd.WaveConfig.of(w)
        lay = synth.layer_layout(w)
        assert fsd.weights_bytes(cfg) == 2 * synth.weight_elems(w)
        for which, name in enumerate(("g_attn", "wqkv", "wo", "g_mlp", "wgu", "wdown")):
            assert fsd.weight_offset(cfg, 1, which) == 2 * (lay["layer"] + lay[name])
    assert fsd.weights_bytes(fsd.WaveConfig.of(synth.SEVEN_B)) == 12_952_535_040


def test_strerror_and_bad_layout_queries():
    assert fsd.strerror(fsd.WAVE_ETIMEOUT) == "a device-side wait timed out"
    bad = fsd.WaveConfig(2, 256, 4, 96, 688, 1e-5, 1e4)
    assert fsd.weights_bytes(bad) == 0
    assert fsd.weight_offset(bad, 0, 0) == (1 << 64) - 1


@pytest.mark.parametrize("w", [synth.HYBRID_SMALL, synth.HYBRID])
def test_hybrid_blob_layout_matches_the_generator(w):
    cfg = fsd.WaveHybridConfig.of(w)
    assert fsd.hybrid_weights_bytes(cfg) == 2 * synth.hybrid_weight_elems(w)
    for l in range(w.n_layers + 1):
        assert fsd.hybrid_layer_offset(cfg, l) == 2 * synth.hybrid_layer_offset(w, l)
    bad = fsd.WaveHybridConfig.of(w)
    bad.ssm_state = 64
    assert fsd.hybrid_weights_bytes(bad) == 0
    # the per-head parameters are staged in shared memory: at most 1024 heads
    many = fsd.WaveHybridConfig.of(w)
    many.ssm_heads = 1028
    assert fsd.hybrid_weights_bytes(many) == 0
    many.ssm_heads = 1024
    assert fsd.hybrid_weights_bytes(many) > 0


def test_packed_blob_sizes():
    # every projection matrix padded to 128-row tiles (gate/up: 64-row
    # halves) and 128-input units, vectors as they are
    def up(a, b):
        return -(-a // b) * b
    for w in (synth.TINY, synth.SEVEN_B, synth.MID, synth.DEPTH):
        d, HD, F = w.d_model, w.HD, w.ffn
        per_layer = (2 * d + up(3 * HD, 128) * up(d, 128) + up(d, 128) * up(HD, 128)
                     + up(F, 64) * 2 * up(d, 128) + up(d, 128) * up(F, 128))
        assert fsd.packed_weights_bytes(fsd.WaveConfig.of(w)) == 2 * w.n_layers * per_layer
    assert fsd.packed_weights_bytes(fsd.WaveConfig.of(synth.SEVEN_B)) == fsd.weights_bytes(fsd.WaveConfig.of(synth.SEVEN_B))
    h = synth.HYBRID
    d, di, HD, Hs = h.d_model, h.d_inner, h.HD, h.ssm_heads
    mamba = d + up(h.in_rows, 128) * up(d, 128) + up(d, 128) * up(di, 128) + up(3 * Hs, 8)
    attn = d + up(3 * HD, 128) * up(d, 128) + up(d, 128) * up(HD, 128)
    groups = h.n_layers // h.attn_every
    assert fsd.hybrid_packed_weights_bytes(fsd.WaveHybridConfig.of(h)) == 2 * groups * ((h.attn_every - 1) * mamba + attn)
