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
M_WQKV, M_WO, M_WGU, M_WDOWN = 1, 2, 4, 5
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
