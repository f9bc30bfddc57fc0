"""Seeded synthetic inputs for the packed 2D-RoPE varlen attention path.

This module is shared by the FP64 oracle tests and by the CUDA path's tests and
benchmark.  It holds none of the attention method's arithmetic: it draws the
packing specs of each workload and the bf16 Q/K/V/dO tensors from a
counter-based generator (splitmix64 finaliser + Box-Muller, defined in
``synth.c``).  ``_np_*`` restate the same generator in numpy for small sizes so
a test can check the C build bit for bit.

Workloads (the pages' workload shapes; the pages' own data are proprietary):
  tiny            3 samples (5, 4x6), (7, 8x8), (3, 2x16); 2 heads x 64
  single_1024     (256, 64x64); 24 heads x 128; forward only
  mixed_50k       latent grids from {32x32, 48x64, 64x48, 64x64, 40x96, 96x40},
                  text U[32, 512], appended until the next sample would exceed
                  50,000 tokens; 24 x 128; forward + backward
  cfg_2048        (512, 128x128) conditional and (64, 128x128) unconditional
                  branch of one 2048^2 image; 24 x 128; forward only
  extreme_aspect  (t, 32x128), (t, 128x32), (t, 128x128), then (t, 64x64)
                  fillers up to 50,000 tokens, t ~ U[64, 512]; 24 x 128;
                  Q/K/V = bf16(s * N(0,1)) with s ~ U(0.5, 2) per tensor and head;
                  forward + backward
  edit_tiny       editing pack (text, source grid, target grid):
                  (5, 2x3, 2x3), (3, 4x2, 3x3), (0, 1x1, 1x1); 2 heads x 64
  edit_50k        editing pack: one latent grid per sample from the mixed set,
                  used for both the source and the target image, text U[32, 512],
                  appended until the next sample would exceed 50,000 tokens;
                  24 x 128; forward + backward
Editing specs are (text_len, Hs, Ws, Ht, Wt) and the sample is [text; source;
target].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libsynth.so")

# stream ids of the generator
STREAM_SPECS = 1
STREAM_Q, STREAM_K, STREAM_V, STREAM_DO = 2, 3, 4, 5
STREAM_SCALE_Q, STREAM_SCALE_K, STREAM_SCALE_V = 12, 13, 14

MASK64 = (1 << 64) - 1


def build(force: bool = False) -> str:
    """Compile synth.c into _build/libsynth.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-D_DEFAULT_SOURCE", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        u64, i64 = ctypes.c_uint64, ctypes.c_int64
        p = ctypes.c_void_p
        _lib.synth_draws.argtypes = [u64, u64, i64, p]
        _lib.synth_randint.argtypes = [u64, u64, i64, i64, i64, p]
        _lib.synth_uniform.argtypes = [u64, u64, i64, p]
        _lib.synth_normal_bf16.argtypes = [u64, u64, i64, p, i64, i64, p]
        _lib.synth_normal_f64.argtypes = [u64, u64, i64, p]
        for f in (_lib.synth_draws, _lib.synth_randint, _lib.synth_uniform,
                  _lib.synth_normal_bf16, _lib.synth_normal_f64):
            f.restype = None
    return _lib


# ----------------------------------------------------------------- C-backed draws
def draws(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    lib().synth_draws(seed & MASK64, stream, n, out.ctypes.data)
    return out


def randint(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int64)
    lib().synth_randint(seed & MASK64, stream, n, lo, hi, out.ctypes.data)
    return out


def uniform(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    lib().synth_uniform(seed & MASK64, stream, n, out.ctypes.data)
    return out


def normal_f64(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    lib().synth_normal_f64(seed & MASK64, stream, n, out.ctypes.data)
    return out


def normal_bf16_bits(seed: int, stream: int, shape, head_scale=None) -> np.ndarray:
    """uint16 bf16 bit patterns of bf16(s * N(0,1)), C order, given shape.

    ``head_scale`` (length ``shape[1]``) scales element [t, a, e] by head_scale[a]."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    if head_scale is not None:
        hs = np.ascontiguousarray(head_scale, dtype=np.float64)
        assert len(shape) == 3 and hs.shape == (shape[1],)
        lib().synth_normal_bf16(seed & MASK64, stream, n, hs.ctypes.data, shape[1], shape[2],
                                out.ctypes.data)
    else:
        lib().synth_normal_bf16(seed & MASK64, stream, n, None, 1, 1, out.ctypes.data)
    return out.reshape(shape)


# --------------------------------------------- numpy restatement (small n only)
def _np_mix64(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64)
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(0xBF58476D1CE4E5B9)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(0x94D049BB133111EB)
    z = z ^ (z >> np.uint64(31))
    return z


def _np_draws(seed: int, stream: int, n: int) -> np.ndarray:
    with np.errstate(over="ignore"):
        s = _np_mix64(np.array([stream], dtype=np.uint64) + np.uint64(0x632BE59BD9B4E019))
        base = _np_mix64(np.array([seed & MASK64], dtype=np.uint64) ^ s)
        i = np.arange(1, n + 1, dtype=np.uint64)
        return _np_mix64(base + i * np.uint64(0x9E3779B97F4A7C15))


def _np_normal_bf16_bits(seed: int, stream: int, n: int) -> np.ndarray:
    d = _np_draws(seed, stream, n + (n & 1))
    u = (d >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    u1, u2 = u[0::2], u[1::2]
    rad = np.sqrt(-2.0 * np.log(1.0 - u1))
    z = np.empty(len(u), dtype=np.float64)
    z[0::2] = rad * np.cos(2.0 * np.pi * u2)
    z[1::2] = rad * np.sin(2.0 * np.pi * u2)
    f = z[:n].astype(np.float32).view(np.uint32)
    return ((f + np.uint32(0x7FFF) + ((f >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


# ------------------------------------------------------------------- workloads
MIXED_GRIDS = [(32, 32), (48, 64), (64, 48), (64, 64), (40, 96), (96, 40)]
TOKEN_BUDGET = 50_000


@dataclass
class Workload:
    name: str
    specs: list  # [(text_len, H_lat, W_lat)]
    heads: int
    head_dim: int
    seed: int
    backward: bool
    head_scale: bool = False
    note: str = ""

    @property
    def edit(self) -> bool:
        """Editing pack: specs are (text_len, Hs, Ws, Ht, Wt)."""
        return bool(self.specs) and len(self.specs[0]) == 5

    @property
    def lengths(self):
        return [s[0] + s[1] * s[2] + (s[3] * s[4] if len(s) == 5 else 0) for s in self.specs]

    @property
    def total(self):
        return sum(self.lengths)

    @property
    def max_len(self):
        return max(self.lengths) if self.specs else 0

    def flops_fwd(self) -> float:
        """4 * sum(L_i^2) * d * h: the two within-sample GEMMs S = Q'K'^T and O = PV."""
        return 4.0 * sum(L * L for L in self.lengths) * self.head_dim * self.heads

    def flops_bwd(self) -> float:
        return 2.5 * self.flops_fwd()


def tiny(seed: int = 0) -> Workload:
    return Workload("tiny", [(5, 4, 6), (7, 8, 8), (3, 2, 16)], 2, 64, seed, True)


def single_1024(seed: int = 0) -> Workload:
    return Workload("single_1024", [(256, 64, 64)], 24, 128, seed, False)


def mixed_50k(seed: int = 0, budget: int = TOKEN_BUDGET) -> Workload:
    specs, total, k = [], 0, 0
    while True:
        g = int(randint(seed, STREAM_SPECS, k + 1, 0, len(MIXED_GRIDS) - 1)[k])
        t = int(randint(seed, STREAM_SPECS + 100, k + 1, 32, 512)[k])
        H, W = MIXED_GRIDS[g]
        L = t + H * W
        if total + L > budget:
            break
        specs.append((t, H, W))
        total += L
        k += 1
    return Workload("mixed_50k", specs, 24, 128, seed, True)


def cfg_2048(seed: int = 0) -> Workload:
    return Workload("cfg_2048", [(512, 128, 128), (64, 128, 128)], 24, 128, seed, False)


def extreme_aspect(seed: int = 0, budget: int = TOKEN_BUDGET) -> Workload:
    texts = randint(seed, STREAM_SPECS + 200, 64, 64, 512)
    specs, total = [], 0
    fixed = [(32, 128), (128, 32), (128, 128)]
    k = 0
    while True:
        H, W = fixed[k] if k < len(fixed) else (64, 64)
        t = int(texts[k])
        L = t + H * W
        if total + L > budget:
            break
        specs.append((t, H, W))
        total += L
        k += 1
    return Workload("extreme_aspect", specs, 24, 128, seed, True, head_scale=True)


def edit_tiny(seed: int = 0) -> Workload:
    return Workload("edit_tiny", [(5, 2, 3, 2, 3), (3, 4, 2, 3, 3), (0, 1, 1, 1, 1)], 2, 64, seed,
                    True)


def edit_50k(seed: int = 0, budget: int = TOKEN_BUDGET) -> Workload:
    specs, total, k = [], 0, 0
    while True:
        g = int(randint(seed, STREAM_SPECS + 300, k + 1, 0, len(MIXED_GRIDS) - 1)[k])
        t = int(randint(seed, STREAM_SPECS + 400, k + 1, 32, 512)[k])
        H, W = MIXED_GRIDS[g]
        L = t + 2 * H * W
        if total + L > budget:
            break
        specs.append((t, H, W, H, W))
        total += L
        k += 1
    return Workload("edit_50k", specs, 24, 128, seed, True)


WORKLOADS = {f.__name__: f for f in (tiny, single_1024, mixed_50k, cfg_2048, extreme_aspect,
                                     edit_tiny, edit_50k)}


def workload(name: str, seed: int = 0, budget: int | None = None) -> Workload:
    """A named workload; `budget` overrides the 50,000-token budget of the two
    budget-packed workloads (used for smaller profiling captures)."""
    if budget is not None and name in ("mixed_50k", "extreme_aspect", "edit_50k"):
        return WORKLOADS[name](seed, budget=budget)
    return WORKLOADS[name](seed)


def head_scales(wl: Workload, stream: int) -> np.ndarray | None:
    if not wl.head_scale:
        return None
    return 0.5 + 1.5 * uniform(wl.seed, stream, wl.heads)


def make_inputs(wl: Workload, with_do: bool | None = None):
    """bf16 bit patterns (numpy uint16, [T, heads, head_dim]) of q, k, v and dO."""
    shape = (wl.total, wl.heads, wl.head_dim)
    q = normal_bf16_bits(wl.seed, STREAM_Q, shape, head_scales(wl, STREAM_SCALE_Q))
    k = normal_bf16_bits(wl.seed, STREAM_K, shape, head_scales(wl, STREAM_SCALE_K))
    v = normal_bf16_bits(wl.seed, STREAM_V, shape, head_scales(wl, STREAM_SCALE_V))
    if with_do is None:
        with_do = wl.backward
    do = normal_bf16_bits(wl.seed, STREAM_DO, shape) if with_do else None
    return q, k, v, do


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact conversion of bf16 bit patterns to float64."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bits_to_torch(bits: np.ndarray):
    import torch
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)


def torch_to_bits(t) -> np.ndarray:
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
