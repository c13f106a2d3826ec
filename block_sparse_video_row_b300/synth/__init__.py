"""Seeded synthetic workloads for frame-aligned block-sparse attention.

This module is shared by the fp64 oracle and the CUDA path and holds none of
the method's arithmetic: it only draws input tensors (bf16 Q, K, V) and builds
the frame-granular block masks of the workloads the pages describe (a video
super-resolution transformer attending over a window of neighbouring frames,
"HeyGen x Google Cloud: Bringing Avatar IV to TPUs", section on shrinking the
block to 16; the shapes are the 720p / 1080p latent chunks of that pipeline).

Random numbers: counter-based SplitMix64 -> Box-Muller (fp64) -> fp32 -> bf16,
implemented once in ``gen.c``.  bf16 tensors are returned as ``numpy.uint16``
arrays holding the raw bf16 bits.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Callable, Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libbsvsynth.so")

TAG_Q, TAG_K, TAG_V, TAG_Z, TAG_OUTLIER = 1, 2, 3, 4, 5


def build(force: bool = False) -> str:
    """Compile gen.c into libbsvsynth.so next to this file (gcc, pthreads)."""
    src = os.path.join(_HERE, "gen.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-o", _LIB_PATH, src, "-lm", "-lpthread"])
    return _LIB_PATH


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.synth_stream_key.restype = ctypes.c_uint64
        lib.synth_stream_key.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]
        lib.synth_splitmix64_at.restype = ctypes.c_uint64
        lib.synth_splitmix64_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_tensor_bf16.restype = None
        lib.synth_tensor_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_int32]
        lib.synth_stream_f64.restype = None
        lib.synth_stream_f64.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                         ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p]
        _lib = lib
    return _lib


def _nthreads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1))


def stream_key(seed: int, tag: int, b: int, h: int) -> int:
    return int(_load().synth_stream_key(seed, tag, b, h))


def splitmix64_at(key: int, i: int) -> int:
    return int(_load().synth_splitmix64_at(key, i))


def stream_f64(seed: int, tag: int, b: int, h: int, n: int, uniform: bool = False) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().synth_stream_f64(seed, tag, b, h, n, 2 if uniform else 1, out.ctypes.data)
    return out


def tensor_bf16(seed: int, tag: int, B: int, H: int, L: int, D: int,
                row_scale: Optional[np.ndarray] = None) -> np.ndarray:
    """[B,H,L,D] bf16 bits (uint16) of N(0,1) draws, times row_scale[B,H,L] if given."""
    out = np.empty((B, H, L, D), dtype=np.uint16)
    rs = None
    if row_scale is not None:
        rs = np.ascontiguousarray(row_scale, dtype=np.float64).reshape(B, H, L)
    _load().synth_tensor_bf16(seed, tag, B, H, L, D, None if rs is None else rs.ctypes.data,
                              out.ctypes.data, _nthreads())
    return out


def bf16_bits_to_f64(x: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to fp64 (bf16 -> fp32 is a 16-bit shift)."""
    return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bits, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


# ----------------------------------------------------------------------------------------------
# block masks (frame granularity)


def window_mask(nb: int, w: int, first_frame_global: bool = False) -> np.ndarray:
    """uint8 [nb, nb]; entry [f, g] = 1 when query frame f reads key frame g.

    f reads g when |f - g| <= w; with ``first_frame_global`` every query frame
    also reads frame 0 (a column-global first frame; frame 0 itself reads only
    its own window)."""
    f = np.arange(nb)[:, None]
    g = np.arange(nb)[None, :]
    m = np.abs(f - g) <= w
    if first_frame_global:
        m = m | (g == 0)
    return m.astype(np.uint8)


def dense_mask(nb: int) -> np.ndarray:
    return np.ones((nb, nb), dtype=np.uint8)


def mixed_head_masks(nb: int, H: int) -> np.ndarray:
    """uint8 [H, nb, nb], one mask per head: head h follows rule h % 4 -- window +-1 plus
    a global first frame, window +-2, its own frame only, every frame."""
    rules = (window_mask(nb, 1, True), window_mask(nb, 2), window_mask(nb, 0), dense_mask(nb))
    return np.stack([rules[h % 4] for h in range(H)])


# ----------------------------------------------------------------------------------------------
# the workloads


@dataclass(frozen=True)
class Workload:
    """A problem shape.  ``frames`` key/value frames; the queries are the last
    ``q_frames`` of them (0: all, self-attention over the chunk).  With
    q_frames < frames this is a streamed chunk whose queries read earlier context
    frames as well as the chunk: the mask is the last q_frames rows of the
    frames x frames mask, and Q is the last q_frames frames of the full-window
    query tensor (so its rows equal the matching rows of the self-attention
    problem over all frames)."""
    name: str
    B: int
    H: int
    D: int
    frames: int
    tokens_per_frame: int
    mask: Callable[[int], np.ndarray]
    keys: str = "normal"      # "normal" or "lognormal_outliers"
    seed: int = 0
    q_frames: int = 0

    @property
    def nq(self) -> int:
        return self.q_frames or self.frames

    @property
    def L(self) -> int:
        """Query rows per head."""
        return self.nq * self.tokens_per_frame

    @property
    def L_kv(self) -> int:
        return self.frames * self.tokens_per_frame

    @property
    def block(self) -> int:
        return self.tokens_per_frame

    @property
    def nb(self) -> int:
        """Query frames."""
        return self.nq

    @property
    def nb_kv(self) -> int:
        return self.frames

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / np.sqrt(self.D)))

    def block_mask(self) -> np.ndarray:
        """uint8 [nq, frames]: the last nq rows of the frames x frames mask ([H, nq, frames]
        for a workload with one mask per head)."""
        m = self.mask(self.frames)
        if m.ndim == 3 and m.shape[0] != self.H:  # fewer or more heads than the masks were made for
            m = np.stack([m[h % m.shape[0]] for h in range(self.H)])
        return np.ascontiguousarray(m[..., self.frames - self.nq:, :])


WORKLOADS: Dict[str, Workload] = {
    # 4 frames x 48 tokens, each frame reads frames f-1..f+1
    "tiny": Workload("tiny", 1, 2, 64, 4, 48, lambda nb: window_mask(nb, 1)),
    # 8 frames x 400 tokens, window +-2 frames plus frame 0 for every query frame
    "small": Workload("small", 1, 8, 128, 8, 400, lambda nb: window_mask(nb, 2, True)),
    # 720p latent chunk: 13 frames x 3600 tokens (45x80 patches), window +-1 plus frame 0
    "720p": Workload("720p", 1, 24, 128, 13, 3600, lambda nb: window_mask(nb, 1, True)),
    # 1080p latent chunk: 13 frames x 8160 tokens (68x120 patches), window +-1
    "1080p": Workload("1080p", 1, 24, 128, 13, 8160, lambda nb: window_mask(nb, 1)),
    # same shape, every frame reads every frame (a dense reference point)
    "1080p_dense": Workload("1080p_dense", 1, 24, 128, 13, 8160, dense_mask),
    # 720p shape with keys whose per-token norms are log-normal (sigma 1.5) and 1% outliers at 8x
    "stress": Workload("stress", 1, 24, 128, 13, 3600, lambda nb: window_mask(nb, 1, True),
                       keys="lognormal_outliers"),
    # a streamed chunk: 3 query frames of 400 tokens reading 5 context frames plus the chunk
    # (window +-2 plus frame 0 over the 8 frames)
    "stream_small": Workload("stream_small", 1, 8, 128, 8, 400, lambda nb: window_mask(nb, 2, True),
                             q_frames=3),
    # a streamed 720p chunk: 4 query frames of 3600 tokens reading 9 context frames plus the chunk
    # (window +-1 plus frame 0 over the 13 frames)
    "stream": Workload("stream", 1, 24, 128, 13, 3600, lambda nb: window_mask(nb, 1, True), q_frames=4),
    # one mask per head (rules cycling over the heads: window +-1 plus frame 0, window +-2,
    # own frame, every frame) at the small shape, as a streamed chunk, and at 720p
    "small_heads": Workload("small_heads", 1, 8, 128, 8, 400, lambda nb: mixed_head_masks(nb, 8)),
    "stream_heads": Workload("stream_heads", 1, 8, 128, 8, 400, lambda nb: mixed_head_masks(nb, 8), q_frames=3),
    "720p_heads": Workload("720p_heads", 1, 24, 128, 13, 3600, lambda nb: mixed_head_masks(nb, 24)),
}


def key_row_scale(seed: int, B: int, H: int, L: int, sigma: float = 1.5,
                  outlier_frac: float = 0.01, outlier_mult: float = 8.0) -> np.ndarray:
    """Per-token key multipliers [B,H,L] for the loose-bound stress workload.

    Token j of head (b,h) is scaled by exp(sigma * z_j), z_j ~ N(0,1); exactly
    floor(outlier_frac * L) tokens per head, picked by a seeded partial
    Fisher-Yates shuffle, are further multiplied by outlier_mult."""
    n_out = int(np.floor(outlier_frac * L))
    out = np.empty((B, H, L), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            z = stream_f64(seed, TAG_Z, b, h, L)
            s = np.exp(sigma * z)
            u = stream_f64(seed, TAG_OUTLIER, b, h, max(n_out, 1), uniform=True)
            perm = np.arange(L)
            for i in range(n_out):
                j = i + int(np.floor(u[i] * (L - i)))
                perm[i], perm[j] = perm[j], perm[i]
            s[perm[:n_out]] *= outlier_mult
            out[b, h] = s
    return out


def make_qkv(w: Workload):
    """(q [B,H,L,D], k [B,H,L_kv,D], v [B,H,L_kv,D]) as uint16 bf16 bits; q holds the last
    L rows of the full-window query tensor."""
    q = tensor_bf16(w.seed, TAG_Q, w.B, w.H, w.L_kv, w.D)
    if w.L != w.L_kv:
        q = np.ascontiguousarray(q[:, :, w.L_kv - w.L:, :])
    rs = key_row_scale(w.seed, w.B, w.H, w.L_kv) if w.keys == "lognormal_outliers" else None
    k = tensor_bf16(w.seed, TAG_K, w.B, w.H, w.L_kv, w.D, rs)
    v = tensor_bf16(w.seed, TAG_V, w.B, w.H, w.L_kv, w.D)
    return q, k, v


def useful_flop(w_or_B, H=None, D=None, block=None, mask=None) -> float:
    """4 * sum over allowed (q-block, kv-block) pairs of block^2 * D * H * B (a per-head
    mask [H, nq, nkv] already counts its pairs over the heads)."""
    if isinstance(w_or_B, Workload):
        w = w_or_B
        B, H, D, block, mask = w.B, w.H, w.D, w.block, w.block_mask()
    else:
        B = w_or_B
    heads = 1 if np.ndim(mask) == 3 else H
    return 4.0 * float(np.count_nonzero(mask)) * block * block * D * heads * B
