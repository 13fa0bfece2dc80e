"""Seeded synthetic inputs for the frame-locked batched decode step.

Serves both the CUDA library's tests/bench and the CPU oracle.  It holds none
of the step's arithmetic: it draws weights, activations, positions and the raw
fp32 values of a prefilled K/V history.  Each side turns those raw values into
FP8 codes with its own quantiser.

The generator is defined in ``synth.c`` (host) and ``synth_gpu.cu`` (device
twin); ``normal_ref``/``word_ref`` below restate it in numpy for small counts
so the compiled versions can be checked against it.

The pages measure on private recordings and checkpoints, so these seeded
draws stand in for them: weights ~N(0, 0.02) in bf16, RMSNorm gains 1.0,
x ~N(0, 1) in bf16, positions uniform in the workload's range, and a K/V
history of N(0, 1) values (Irwin-Hall(12) - 6 approximations of N(0, 1)).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field, replace

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SO = os.path.join(HERE, "libsynth.so")
_GPU_SO = os.path.join(HERE, "libsynth_gpu.so")

SEED_WEIGHTS, SEED_X, SEED_POS, SEED_KV = 1, 2, 3, 4
STREAM_X, STREAM_POS, STREAM_PROJ = 1, 2, 3
WEIGHT_STREAM_BASE, KV_STREAM_BASE = 1000, 2000
M_WQKV, M_WO, M_WGU, M_WDOWN, M_WIN, M_WOUT, M_ALOG = 1, 2, 4, 5, 6, 7, 8
SEED_STATE = 5
WEIGHT_STD = 0.02

_G = 0x9E3779B97F4A7C15
_MASK = (1 << 64) - 1


# ---------------------------------------------------------------- workloads
@dataclass(frozen=True)
class Workload:
    """Shapes and input recipe of one step configuration."""
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    head_dim: int
    ffn: int
    S: int
    T_max: int
    pos_lo: int
    pos_hi: int
    rms_eps: float = 1e-5
    rope_base: float = 10000.0
    extra: dict = field(default_factory=dict, compare=False)

    @property
    def HD(self) -> int:
        return self.n_heads * self.head_dim

    def with_S(self, S: int) -> "Workload":
        return replace(self, S=S)


TINY = Workload("tiny-2L-d256-h4x64-f688", 2, 256, 4, 64, 688, S=4, T_max=64, pos_lo=1, pos_hi=64)
SEVEN_B = Workload("7b-class-32L-d4096-h32x128-f11008", 32, 4096, 32, 128, 11008,
                   S=80, T_max=3000, pos_lo=0, pos_hi=3000)
SWEEP_S = (1, 8, 16, 32, 48, 56, 64, 80, 96, 128)
# Parity shape that spans several GEMM tiles, several attention chunks and
# ragged tails in every dimension (S, F, positions).
MID = Workload("mid-3L-d512-h4x128-f1376", 3, 512, 4, 128, 1376, S=19, T_max=320, pos_lo=0, pos_hi=320)
DEPTH = Workload("depth-6L-d1024-h16x64-f2816", 6, 1024, 16, 64, 2816, S=80, T_max=8, pos_lo=0, pos_hi=8,
                 extra={"depth_steps": 8})


@dataclass(frozen=True)
class HybridWorkload:
    """Shapes and input recipe of the hybrid recurrent step: every
    attn_every-th layer an attention block, the others Mamba2-style
    selective-state blocks (no MLP layers)."""
    name: str
    n_layers: int
    d_model: int
    attn_every: int
    n_heads: int
    head_dim: int
    ssm_heads: int
    ssm_head_dim: int
    ssm_state: int
    S: int
    T_max: int
    pos_lo: int
    pos_hi: int
    rms_eps: float = 1e-5
    rope_base: float = 10000.0

    @property
    def HD(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def d_inner(self) -> int:
        return self.ssm_heads * self.ssm_head_dim

    @property
    def in_rows(self) -> int:
        return 2 * self.d_inner + 2 * self.ssm_state + self.ssm_heads

    @property
    def n_attn(self) -> int:
        return self.n_layers // self.attn_every

    @property
    def n_mamba(self) -> int:
        return self.n_layers - self.n_attn

    def is_attn(self, l: int) -> bool:
        return l % self.attn_every == self.attn_every - 1

    def attention_view(self) -> Workload:
        """The attention layers alone, as a Workload (their K/V history is
        drawn and quantised exactly like the decoder step's)."""
        return Workload(self.name + "-attn", self.n_attn, self.d_model, self.n_heads, self.head_dim, 0,
                        S=self.S, T_max=self.T_max, pos_lo=self.pos_lo, pos_hi=self.pos_hi,
                        rms_eps=self.rms_eps, rope_base=self.rope_base)


HYBRID = HybridWorkload("hybrid-48L-d4096-attn6-h32x128-ssm64x64x128", 48, 4096, 6, 32, 128, 64, 64, 128,
                        S=56, T_max=1500, pos_lo=0, pos_hi=1500)
# Parity shape: two groups of three layers (two Mamba blocks, one attention
# block), ragged S, several state heads.
HYBRID_SMALL = HybridWorkload("hybrid-6L-d256-attn3-h4x64-ssm4x64x128", 6, 256, 3, 4, 64, 4, 64, 128,
                              S=5, T_max=64, pos_lo=0, pos_hi=64)


def hybrid_layout(w: HybridWorkload) -> dict:
    """Element counts of one layer of each kind and the offsets inside them.

    Mamba block: g[d], W_in[in_rows][d] (z, x, B, C, dt rows), W_out[d][d_i],
    A_log[Hs], dt_bias[Hs], D[Hs] (padded to a multiple of 8 elements).
    Attention block: g[d], Wqkv[3HD][d],
    Wo[d][HD].  Group of attn_every layers: (attn_every - 1) Mamba blocks,
    then one attention block."""
    d, di, Hs, HD = w.d_model, w.d_inner, w.ssm_heads, w.HD
    m = {"g": 0, "w_in": d, "w_out": d + w.in_rows * d}
    m["a_log"] = m["w_out"] + d * di
    m["dt_bias"] = m["a_log"] + Hs
    m["d_skip"] = m["dt_bias"] + Hs
    m["size"] = m["a_log"] + (3 * Hs + 7) // 8 * 8   # parameter block padded to 16 bytes
    a = {"g": 0, "wqkv": d, "wo": d + 3 * HD * d}
    a["size"] = a["wo"] + d * HD
    return {"mamba": m, "attn": a}


def hybrid_layer_offset(w: HybridWorkload, l: int) -> int:
    lay = hybrid_layout(w)
    M, A, e = lay["mamba"]["size"], lay["attn"]["size"], w.attn_every
    return (l // e) * ((e - 1) * M + A) + (l % e) * M


def hybrid_weight_elems(w: HybridWorkload) -> int:
    return hybrid_layer_offset(w, w.n_layers)


# ------------------------------------------------------- weight blob layout
def layer_layout(w: Workload) -> dict:
    """Element offsets inside one layer of the bf16 weight blob.

    Order: g_attn[d], Wqkv[3*H*D][d] (q rows, k rows, v rows), Wo[d][H*D],
    g_mlp[d], Wgu[2*F][d] (gate rows, then up rows), Wdown[d][F].
    Every matrix is stored [out][in], the in-dimension contiguous.
    """
    d, HD, F = w.d_model, w.HD, w.ffn
    off = {}
    o = 0
    for name, n in (("g_attn", d), ("wqkv", 3 * HD * d), ("wo", d * HD), ("g_mlp", d),
                    ("wgu", 2 * F * d), ("wdown", d * F)):
        off[name] = o
        o += n
    off["layer"] = o
    return off


def weight_elems(w: Workload) -> int:
    return layer_layout(w)["layer"] * w.n_layers


# ------------------------------------------------------------ numpy restatement
def word_ref(seed: int, stream: int, n: np.ndarray) -> np.ndarray:
    """word(key(seed, stream), n) for an array of counters (numpy, uint64)."""
    with np.errstate(over="ignore"):
        key = _mix_np(np.uint64((seed * 0xD1B54A32D192ED03 + (stream + 1) * _G) & _MASK))
        z = key + (np.asarray(n, dtype=np.uint64) + np.uint64(1)) * np.uint64(_G)
        return _mix_np(z)


def _mix_np(z):
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def normal_ref(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Irwin-Hall(12) - 6 values, numpy restatement of synth.c (fp32)."""
    i = np.arange(start, start + count, dtype=np.uint64)
    total = np.zeros(count, dtype=np.int64)
    for j in range(4):
        w = word_ref(seed, stream, np.uint64(4) * i + np.uint64(j))
        for sh in (0, 20, 40):
            total += ((w >> np.uint64(sh)) & np.uint64(0xFFFFF)).astype(np.int64)
    return ((total - 6 * 1048576).astype(np.float32) * np.float32(1.0 / 1048576.0))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bit patterns (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ------------------------------------------------------------ compiled host side
_lib = None


def build(verbose: bool = False) -> None:
    """Compile libsynth.so (gcc) and libsynth_gpu.so (nvcc, sm_103a)."""
    cmds = [
        ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
         os.path.join(HERE, "synth.c"), "-o", _HOST_SO],
        ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
         "-shared", "-Xcompiler", "-fPIC", os.path.join(HERE, "synth_gpu.cu"), "-o", _GPU_SO],
    ]
    procs = [subprocess.Popen(c, stdout=subprocess.PIPE, stderr=subprocess.STDOUT) for c in cmds]
    for c, p in zip(cmds, procs):
        out, _ = p.communicate()
        if p.returncode != 0:
            raise RuntimeError(f"synth build failed: {' '.join(c)}\n{out.decode()}")
        if verbose and out:
            print(out.decode())


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_HOST_SO):
            build()
        L = ctypes.CDLL(_HOST_SO)
        u64, i64, i32, f32, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32,
                                  ctypes.c_float, ctypes.c_void_p)
        L.synth_key.argtypes = [u64, u64]
        L.synth_key.restype = u64
        L.synth_word.argtypes = [u64, u64, u64]
        L.synth_word.restype = u64
        L.synth_normal_f32.argtypes = [u64, u64, u64, i64, vp]
        L.synth_normal_bf16.argtypes = [u64, u64, u64, i64, f32, vp]
        L.synth_uniform_int.argtypes = [u64, u64, u64, i64, i32, i32, vp]
        L.synth_fill_bf16.argtypes = [i64, f32, vp]
        L.synth_kv_slab_f32.argtypes = [u64, u64, i32, i32, i32, i32, i32, i32, i64, vp]
        _lib = L
    return _lib


def normal_f32(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.float32)
    lib().synth_normal_f32(seed, stream, start, count, out.ctypes.data)
    return out


def normal_bf16(seed: int, stream: int, start: int, count: int, scale: float) -> np.ndarray:
    out = np.empty(count, dtype=np.uint16)
    lib().synth_normal_bf16(seed, stream, start, count, scale, out.ctypes.data)
    return out


def positions(w: Workload, S: int | None = None) -> np.ndarray:
    """pos[s], s < S: the first S draws of one stream (nested across S)."""
    S = w.S if S is None else S
    out = np.empty(S, dtype=np.int32)
    lib().synth_uniform_int(SEED_POS, STREAM_POS, 0, S, w.pos_lo, w.pos_hi, out.ctypes.data)
    return out


def x_bf16(w: Workload, S: int | None = None) -> np.ndarray:
    """x[S][d] as bf16 bit patterns, x ~ N(0, 1)."""
    S = w.S if S is None else S
    return normal_bf16(SEED_X, STREAM_X, 0, S * w.d_model, 1.0).reshape(S, w.d_model)


def proj_std(w: Workload) -> float:
    """Scale of the depth loop's projection W_p: N(0, 1/d), so that W_p y keeps
    the scale of y (1/sqrt(d) is a power of two for the d used here)."""
    return 1.0 / float(np.sqrt(w.d_model))


def proj_host(w: Workload) -> np.ndarray:
    """W_p [d][d] as bf16 bit patterns (row = output)."""
    d = w.d_model
    return normal_bf16(SEED_WEIGHTS, STREAM_PROJ, 0, d * d, proj_std(w)).reshape(d, d)


def weights_host(w: Workload) -> np.ndarray:
    """The whole bf16 weight blob (uint16 bit patterns) on the host."""
    lay = layer_layout(w)
    blob = np.empty(weight_elems(w), dtype=np.uint16)
    L = lib()
    d, HD, F = w.d_model, w.HD, w.ffn
    for l in range(w.n_layers):
        base = l * lay["layer"]
        for name, n in (("g_attn", d), ("g_mlp", d)):
            L.synth_fill_bf16(n, 1.0, blob[base + lay[name]:].ctypes.data)
        for name, m, n in (("wqkv", M_WQKV, 3 * HD * d), ("wo", M_WO, d * HD),
                           ("wgu", M_WGU, 2 * F * d), ("wdown", M_WDOWN, d * F)):
            L.synth_normal_bf16(SEED_WEIGHTS, WEIGHT_STREAM_BASE + 16 * l + m, 0, n, WEIGHT_STD,
                                blob[base + lay[name]:].ctypes.data)
    return blob


def hybrid_weights_host(w: HybridWorkload) -> np.ndarray:
    """The hybrid model's bf16 blob: matrices ~N(0, 0.02), gains 1.0,
    A_log ~N(0, 1) (A = -exp(A_log)), dt_bias 0, D 1.0."""
    lay = hybrid_layout(w)
    blob = np.empty(hybrid_weight_elems(w), dtype=np.uint16)
    L = lib()
    d, di, HD = w.d_model, w.d_inner, w.HD
    for l in range(w.n_layers):
        base = hybrid_layer_offset(w, l)
        L.synth_fill_bf16(d, 1.0, blob[base:].ctypes.data)
        if w.is_attn(l):
            a = lay["attn"]
            for name, m, n in (("wqkv", M_WQKV, 3 * HD * d), ("wo", M_WO, d * HD)):
                L.synth_normal_bf16(SEED_WEIGHTS, WEIGHT_STREAM_BASE + 16 * l + m, 0, n, WEIGHT_STD,
                                    blob[base + a[name]:].ctypes.data)
        else:
            m_ = lay["mamba"]
            for name, m, n in (("w_in", M_WIN, w.in_rows * d), ("w_out", M_WOUT, d * di)):
                L.synth_normal_bf16(SEED_WEIGHTS, WEIGHT_STREAM_BASE + 16 * l + m, 0, n, WEIGHT_STD,
                                    blob[base + m_[name]:].ctypes.data)
            L.synth_normal_bf16(SEED_WEIGHTS, WEIGHT_STREAM_BASE + 16 * l + M_ALOG, 0, w.ssm_heads, 1.0,
                                blob[base + m_["a_log"]:].ctypes.data)
            L.synth_fill_bf16(w.ssm_heads, 0.0, blob[base + m_["dt_bias"]:].ctypes.data)
            L.synth_fill_bf16(w.ssm_heads, 1.0, blob[base + m_["d_skip"]:].ctypes.data)
    return blob


def hybrid_state_host(w: HybridWorkload, lm: int, s0: int, ns: int) -> np.ndarray:
    """Initial fp32 state of Mamba layer lm for sessions s0..s0+ns-1:
    [ns][Hs][P][N] ~N(0, 1)."""
    blk = w.ssm_heads * w.ssm_head_dim * w.ssm_state
    return normal_f32(SEED_STATE, lm, s0 * blk, ns * blk).reshape(ns, w.ssm_heads, w.ssm_head_dim,
                                                                 w.ssm_state)


def kv_raw_host(w: Workload, layer: int, which: int, s0: int, ns: int, t_count: int,
                out_T: int | None = None) -> np.ndarray:
    """Raw fp32 history values [ns][H][out_T][D] for slots t < t_count."""
    out_T = w.T_max if out_T is None else out_T
    out = np.zeros((ns, w.n_heads, out_T, w.head_dim), dtype=np.float32)
    lib().synth_kv_slab_f32(SEED_KV, KV_STREAM_BASE + 2 * layer + which, s0, ns, w.n_heads,
                            w.T_max, t_count, w.head_dim, out_T, out.ctypes.data)
    return out


# ------------------------------------------------------------ device twin
_glib = None


def gpu_lib():
    """ctypes handle of the device twin (libsynth_gpu.so)."""
    global _glib
    if _glib is None:
        if not os.path.exists(_GPU_SO):
            raise RuntimeError("libsynth_gpu.so is not built; run __graft_entry__.build()")
        L = ctypes.CDLL(_GPU_SO)
        u64, i64, i32, f32, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32,
                                  ctypes.c_float, ctypes.c_void_p)
        L.synth_gpu_normal_bf16.argtypes = [u64, u64, u64, i64, f32, vp, vp]
        L.synth_gpu_normal_f32.argtypes = [u64, u64, u64, i64, vp, vp]
        L.synth_gpu_kv_slab_f32.argtypes = [u64, u64, i32, i32, i32, i32, i32, i32, i64, vp, vp]
        for f in (L.synth_gpu_normal_bf16, L.synth_gpu_normal_f32, L.synth_gpu_kv_slab_f32):
            f.restype = ctypes.c_int
        _glib = L
    return _glib


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"{what} failed with CUDA error {rc}")


def weights_device(w: Workload, blob, stream_ptr: int) -> None:
    """Fill a device bf16 blob (a torch tensor of weight_elems(w) bf16) in place."""
    lay = layer_layout(w)
    G = gpu_lib()
    d, HD, F = w.d_model, w.HD, w.ffn
    out_ptr = blob.data_ptr()
    for l in range(w.n_layers):
        base = l * lay["layer"]
        for name in ("g_attn", "g_mlp"):
            blob[base + lay[name]: base + lay[name] + d].fill_(1.0)
        for name, m, n in (("wqkv", M_WQKV, 3 * HD * d), ("wo", M_WO, d * HD),
                           ("wgu", M_WGU, 2 * F * d), ("wdown", M_WDOWN, d * F)):
            _check(G.synth_gpu_normal_bf16(SEED_WEIGHTS, WEIGHT_STREAM_BASE + 16 * l + m, 0, n,
                                           WEIGHT_STD, out_ptr + 2 * (base + lay[name]),
                                           stream_ptr), "synth_gpu_normal_bf16")


def kv_raw_device(w: Workload, layer: int, which: int, s0: int, ns: int, t_count: int,
                  out_ptr: int, out_T: int, stream_ptr: int) -> None:
    """Device twin of kv_raw_host: writes [ns][H][out_T][D] fp32 for t < t_count."""
    _check(gpu_lib().synth_gpu_kv_slab_f32(SEED_KV, KV_STREAM_BASE + 2 * layer + which, s0, ns,
                                           w.n_heads, w.T_max, t_count, w.head_dim, out_T,
                                           out_ptr, stream_ptr), "synth_gpu_kv_slab_f32")


def x_device(w: Workload, S: int, out_ptr: int, stream_ptr: int) -> None:
    _check(gpu_lib().synth_gpu_normal_bf16(SEED_X, STREAM_X, 0, S * w.d_model, 1.0, out_ptr,
                                           stream_ptr), "synth_gpu_normal_bf16")


def proj_device(w: Workload, out_ptr: int, stream_ptr: int) -> None:
    """Device twin of proj_host (d*d bf16 at out_ptr)."""
    d = w.d_model
    _check(gpu_lib().synth_gpu_normal_bf16(SEED_WEIGHTS, STREAM_PROJ, 0, d * d, proj_std(w), out_ptr,
                                           stream_ptr), "synth_gpu_normal_bf16")


def hybrid_weights_device(w: HybridWorkload, blob, stream_ptr: int) -> None:
    """Device twin of hybrid_weights_host (a torch bf16 tensor of
    hybrid_weight_elems(w) elements, filled in place)."""
    lay = hybrid_layout(w)
    G = gpu_lib()
    d, di, HD = w.d_model, w.d_inner, w.HD
    out_ptr = blob.data_ptr()
    for l in range(w.n_layers):
        base = hybrid_layer_offset(w, l)
        blob[base: base + d].fill_(1.0)
        if w.is_attn(l):
            a = lay["attn"]
            for name, m, n in (("wqkv", M_WQKV, 3 * HD * d), ("wo", M_WO, d * HD)):
                _check(G.synth_gpu_normal_bf16(SEED_WEIGHTS, WEIGHT_STREAM_BASE + 16 * l + m, 0, n, WEIGHT_STD,
                                               out_ptr + 2 * (base + a[name]), stream_ptr), "synth_gpu_normal_bf16")
        else:
            m_ = lay["mamba"]
            for name, m, n in (("w_in", M_WIN, w.in_rows * d), ("w_out", M_WOUT, d * di)):
                _check(G.synth_gpu_normal_bf16(SEED_WEIGHTS, WEIGHT_STREAM_BASE + 16 * l + m, 0, n, WEIGHT_STD,
                                               out_ptr + 2 * (base + m_[name]), stream_ptr), "synth_gpu_normal_bf16")
            _check(G.synth_gpu_normal_bf16(SEED_WEIGHTS, WEIGHT_STREAM_BASE + 16 * l + M_ALOG, 0, w.ssm_heads, 1.0,
                                           out_ptr + 2 * (base + m_["a_log"]), stream_ptr), "synth_gpu_normal_bf16")
            blob[base + m_["dt_bias"]: base + m_["dt_bias"] + w.ssm_heads].fill_(0.0)
            blob[base + m_["d_skip"]: base + m_["d_skip"] + w.ssm_heads].fill_(1.0)


def hybrid_state_device(w: HybridWorkload, lm: int, s0: int, ns: int, out_ptr: int, stream_ptr: int) -> None:
    """Device twin of hybrid_state_host: [ns][Hs][P][N] fp32 at out_ptr."""
    blk = w.ssm_heads * w.ssm_head_dim * w.ssm_state
    _check(gpu_lib().synth_gpu_normal_f32(SEED_STATE, lm, s0 * blk, ns * blk, out_ptr, stream_ptr),
           "synth_gpu_normal_f32")
