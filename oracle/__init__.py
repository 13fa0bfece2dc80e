"""CPU oracle of the frame-locked batched decode step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
path (``frame_step_decode_gb300``) never does.

``oracle.c`` is a plain fp64 restatement of the step (see its header for the
passages it follows and the readings it takes); this module loads it with
ctypes and adds the input plumbing: building an FP8 history with the oracle's
own quantiser from the shared seeded generator (``synth``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(HERE, "liboracle.so")
_lib = None


class OracleCfg(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("d_model", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int), ("rms_eps", ctypes.c_float),
                ("rope_base", ctypes.c_float)]


def build() -> None:
    """Compile liboracle.so with gcc (fp64, OpenMP, no FMA contraction)."""
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
           os.path.join(HERE, "oracle.c"), "-o", _SO, "-lm"]
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if p.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + p.stdout.decode())


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_SO):
            build()
        L = ctypes.CDLL(_SO)
        vp, i32, i64, f32, f64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                  ctypes.c_double)
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_double.restype = f64
        L.oracle_double_to_bf16.argtypes = [f64]
        L.oracle_double_to_bf16.restype = ctypes.c_uint16
        L.oracle_bf16_round.argtypes = [f64]
        L.oracle_bf16_round.restype = f64
        L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_decode.restype = f64
        L.oracle_e4m3_encode.argtypes = [f32]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e4m3_encode_many.argtypes = [vp, i64, vp]
        L.oracle_quantize_row.argtypes = [vp, i32, vp, vp]
        L.oracle_quantize_rows.argtypes = [vp, i64, i32, vp, vp]
        L.oracle_rmsnorm.argtypes = [vp, vp, i32, f64, vp]
        L.oracle_matvec.argtypes = [vp, i32, i32, vp, vp]
        L.oracle_rope.argtypes = [vp, i32, i32, f64]
        L.oracle_attention_head.argtypes = [vp, vp, vp, vp, vp, i32, i32, vp]
        L.oracle_silu.argtypes = [f64]
        L.oracle_silu.restype = f64
        L.oracle_hybrid_step.argtypes = [ctypes.POINTER(OracleHybridCfg), i32, vp, i32, vp, vp, vp, vp, vp,
                                         vp, vp]
        L.oracle_hybrid_step.restype = i32
        L.oracle_ssm_mixer.argtypes = [ctypes.POINTER(OracleHybridCfg), vp, vp, vp, vp, vp, vp, vp]
        L.oracle_ssm_mixer.restype = None
        L.oracle_ssm_update.argtypes = [ctypes.POINTER(OracleHybridCfg), vp, vp, vp, vp, vp, vp]
        L.oracle_ssm_update.restype = None
        L.oracle_hybrid_layer_offset.argtypes = [ctypes.POINTER(OracleHybridCfg), i32]
        L.oracle_hybrid_layer_offset.restype = i64
        L.oracle_proj.argtypes = [vp, i32, i32, vp, vp]
        L.oracle_proj.restype = None
        L.oracle_step.argtypes = [ctypes.POINTER(OracleCfg), i32, vp, i32, vp, vp, vp, vp, vp, vp,
                                  i32, vp]
        L.oracle_step.restype = i32
        _lib = L
    return _lib


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ----------------------------------------------------------------- wrappers
def e4m3_decode_all() -> np.ndarray:
    L = lib()
    return np.array([L.oracle_e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32).ravel()
    out = np.empty(v.size, dtype=np.uint8)
    lib().oracle_e4m3_encode_many(_p(v), v.size, _p(out))
    return out


def quantize_rows(v: np.ndarray):
    """FP8 quantiser over the last axis: (codes uint8, scales float32)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    D = v.shape[-1]
    rows = v.size // D
    codes = np.empty(v.shape, dtype=np.uint8)
    scales = np.empty(v.shape[:-1], dtype=np.float32)
    lib().oracle_quantize_rows(_p(v), rows, D, _p(codes), _p(scales))
    return codes, scales


def rmsnorm(r: np.ndarray, g_bf16: np.ndarray, eps: float) -> np.ndarray:
    r = np.ascontiguousarray(r, dtype=np.float64)
    g = np.ascontiguousarray(g_bf16, dtype=np.uint16)
    out = np.empty_like(r)
    lib().oracle_rmsnorm(_p(r), _p(g), r.size, eps, _p(out))
    return out


def matvec(W_bf16: np.ndarray, x: np.ndarray) -> np.ndarray:
    W = np.ascontiguousarray(W_bf16, dtype=np.uint16)
    x = np.ascontiguousarray(x, dtype=np.float64)
    N, K = W.shape
    y = np.empty(N, dtype=np.float64)
    lib().oracle_matvec(_p(W), N, K, _p(x), _p(y))
    return y


def rope(v: np.ndarray, pos: int, base: float = 10000.0) -> np.ndarray:
    v = np.array(v, dtype=np.float64)
    lib().oracle_rope(_p(v), v.size, pos, base)
    return v


def attention_head(q, kc, ks, vc, vs, pos: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float64)
    kc = np.ascontiguousarray(kc, dtype=np.uint8)
    vc = np.ascontiguousarray(vc, dtype=np.uint8)
    ks = np.ascontiguousarray(ks, dtype=np.float32)
    vs = np.ascontiguousarray(vs, dtype=np.float32)
    D = q.size
    o = np.empty(D, dtype=np.float64)
    lib().oracle_attention_head(_p(q), _p(kc), _p(ks), _p(vc), _p(vs), pos, D, _p(o))
    return o


class OracleHybridCfg(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("d_model", ctypes.c_int), ("attn_every", ctypes.c_int),
                ("n_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ssm_heads", ctypes.c_int),
                ("ssm_head_dim", ctypes.c_int), ("ssm_state", ctypes.c_int), ("rms_eps", ctypes.c_float),
                ("rope_base", ctypes.c_float)]


def hybrid_cfg_of(w) -> OracleHybridCfg:
    return OracleHybridCfg(w.n_layers, w.d_model, w.attn_every, w.n_heads, w.head_dim, w.ssm_heads,
                           w.ssm_head_dim, w.ssm_state, w.rms_eps, w.rope_base)


def cfg_of(w) -> OracleCfg:
    return OracleCfg(w.n_layers, w.d_model, w.n_heads, w.head_dim, w.ffn, w.rms_eps, w.rope_base)


def step(w, weights: np.ndarray, kv: np.ndarray, kv_scales: np.ndarray, pos: np.ndarray,
         x: np.ndarray, round_acts: bool = True, want_kv_new: bool = False):
    """Run one frame for the sessions held in kv/kv_scales/pos/x (all n of them).

    kv [L][2][n][H][T_max][D] uint8 and kv_scales [L][2][n][H][T_max] float32
    are updated in place at slot pos[s].  A negative pos[s] is an empty slot:
    y[s] = x[s] and its cache is left alone.  Returns (y bf16 bits [n][d],
    y_exact fp64 [n][d], kv_new fp32 [L][2][n][H][D] or None).
    """
    n = pos.size
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    assert kv.flags["C_CONTIGUOUS"] and kv_scales.flags["C_CONTIGUOUS"]
    y = np.empty((n, w.d_model), dtype=np.uint16)
    y_exact = np.empty((n, w.d_model), dtype=np.float64)
    kv_new = (np.empty((w.n_layers, 2, n, w.n_heads, w.head_dim), dtype=np.float32)
              if want_kv_new else None)
    c = cfg_of(w)
    rc = lib().oracle_step(ctypes.byref(c), w.T_max, _p(weights), n, _p(kv), _p(kv_scales),
                           _p(pos), _p(x), _p(y), _p(y_exact), int(round_acts),
                           _p(kv_new) if kv_new is not None else None)
    if rc != 0:
        raise ValueError(f"oracle_step: position of session {-rc - 1} at or beyond T_max")
    return y, y_exact, kv_new


def prefill_history(w, sessions, pos, poison: bool = True):
    """FP8 history for the given sessions, built by the oracle's quantiser.

    Slots t < pos[j] of session sessions[j] hold the shared generator's raw
    N(0, 1) values quantised per (layer, K|V, head, token); slots >= pos[j]
    hold NaN codes (0x7F) and NaN scales when poison is set, zeros otherwise.
    Returns kv [L][2][n][H][T_max][D] uint8 and scales [L][2][n][H][T_max].
    """
    import synth
    n = len(sessions)
    L, H, T, D = w.n_layers, w.n_heads, w.T_max, w.head_dim
    kv = np.empty((L, 2, n, H, T, D), dtype=np.uint8)
    sc = np.empty((L, 2, n, H, T), dtype=np.float32)
    for l in range(L):
        for which in range(2):
            for j, s in enumerate(sessions):
                P = max(int(pos[j]), 0)  # an empty slot (negative position) has no history
                raw = synth.kv_raw_host(w, l, which, int(s), 1, P)
                codes, scales = quantize_rows(raw)
                kv[l, which, j] = codes[0]
                sc[l, which, j] = scales[0]
                if poison:
                    kv[l, which, j, :, P:, :] = 0x7F
                    sc[l, which, j, :, P:] = np.nan
    return kv, sc


def proj(w, wp: np.ndarray, y: np.ndarray) -> np.ndarray:
    """x_next = bf16(W_p y) per row (fp64 accumulation), bf16 bits [n][d]."""
    y = np.ascontiguousarray(y, dtype=np.uint16)
    wp = np.ascontiguousarray(wp, dtype=np.uint16)
    out = np.empty_like(y)
    lib().oracle_proj(_p(wp), w.d_model, y.shape[0], _p(y), _p(out))
    return out


def depth_loop(w, weights: np.ndarray, wp: np.ndarray, x0: np.ndarray, steps: int):
    """The inner depth loop for n sessions: step k at depth position k over a
    fresh depth cache (every slot it reads was written earlier in the loop),
    x_0 = x0 and x_k = bf16(W_p y_{k-1}).  Returns (y bits [steps][n][d],
    y_exact fp64 [steps][n][d], x bits [steps][n][d])."""
    n = x0.shape[0]
    L, H, T, D = w.n_layers, w.n_heads, w.T_max, w.head_dim
    kv = np.full((L, 2, n, H, T, D), 0x7F, dtype=np.uint8)   # NaN codes: never read before written
    sc = np.full((L, 2, n, H, T), np.nan, dtype=np.float32)
    ys = np.empty((steps, n, w.d_model), dtype=np.uint16)
    ye = np.empty((steps, n, w.d_model), dtype=np.float64)
    xs = np.empty((steps, n, w.d_model), dtype=np.uint16)
    x = np.ascontiguousarray(x0, dtype=np.uint16)
    for k in range(steps):
        xs[k] = x
        y, y_exact, _ = step(w, weights, kv, sc, np.full(n, k, dtype=np.int32), x)
        ys[k], ye[k] = y, y_exact
        x = proj(w, wp, y)
    return ys, ye, xs


def hybrid_prefill(w, sessions, pos, poison: bool = True):
    """The hybrid step's state for the listed sessions: the attention layers'
    FP8 history (as prefill_history, over the attention layers alone) and
    the Mamba layers' fp32 state from the shared generator.  Returns (kv,
    scales, state [Lm][n][Hs][P][N])."""
    import synth
    kv, sc = prefill_history(w.attention_view(), sessions, np.maximum(np.asarray(pos), 0), poison=poison)
    n = len(sessions)
    st = np.empty((w.n_mamba, n, w.ssm_heads, w.ssm_head_dim, w.ssm_state), dtype=np.float32)
    for lm in range(w.n_mamba):
        for j, s in enumerate(sessions):
            st[lm, j] = synth.hybrid_state_host(w, lm, int(s), 1)[0]
    return kv, sc, st


def hybrid_step(w, weights: np.ndarray, kv: np.ndarray, kv_scales: np.ndarray, state: np.ndarray,
                pos: np.ndarray, x: np.ndarray):
    """One frame of the hybrid model for n sessions (see oracle.c): kv,
    kv_scales and state are updated in place.  Returns (y bits, y_exact)."""
    n = pos.size
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    assert kv.flags["C_CONTIGUOUS"] and kv_scales.flags["C_CONTIGUOUS"] and state.flags["C_CONTIGUOUS"]
    y = np.empty((n, w.d_model), dtype=np.uint16)
    y_exact = np.empty((n, w.d_model), dtype=np.float64)
    c = hybrid_cfg_of(w)
    rc = lib().oracle_hybrid_step(ctypes.byref(c), w.T_max, _p(weights), n, _p(kv), _p(kv_scales), _p(state),
                                  _p(pos), _p(x), _p(y), _p(y_exact))
    if rc != 0:
        raise ValueError(f"oracle_hybrid_step: position of session {-rc - 1} at or beyond T_max")
    return y, y_exact


def ssm_mixer(w, w_in: np.ndarray, a_log: np.ndarray, dt_bias: np.ndarray, d_skip: np.ndarray,
              xn: np.ndarray, state: np.ndarray) -> np.ndarray:
    """One Mamba2-style mixer for one session (see oracle.c): xn fp64 [d],
    state fp32 [Hs][P][N] updated in place; returns the gated output
    (unrounded) [d_i]."""
    c = hybrid_cfg_of(w)
    out = np.empty(w.d_inner, dtype=np.float64)
    xn = np.ascontiguousarray(xn, dtype=np.float64)
    lib().oracle_ssm_mixer(ctypes.byref(c), _p(np.ascontiguousarray(w_in)), _p(np.ascontiguousarray(a_log)),
                           _p(np.ascontiguousarray(dt_bias)), _p(np.ascontiguousarray(d_skip)), _p(xn),
                           _p(state), _p(out))
    return out


def ssm_update(w, zx: np.ndarray, a_log: np.ndarray, dt_bias: np.ndarray, d_skip: np.ndarray,
               state: np.ndarray) -> np.ndarray:
    """The state update and gated output of one Mamba2-style block for one
    session from its in-projection output zx (fp64 [in_rows]): state fp32
    [Hs][P][N] updated in place; returns the gated output (unrounded) [d_i]."""
    c = hybrid_cfg_of(w)
    out = np.empty(w.d_inner, dtype=np.float64)
    zx = np.ascontiguousarray(zx, dtype=np.float64)
    assert state.flags["C_CONTIGUOUS"] and state.dtype == np.float32
    lib().oracle_ssm_update(ctypes.byref(c), _p(zx), _p(np.ascontiguousarray(a_log)),
                            _p(np.ascontiguousarray(dt_bias)), _p(np.ascontiguousarray(d_skip)), _p(state),
                            _p(out))
    return out
