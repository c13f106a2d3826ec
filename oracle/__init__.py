"""fp64 CPU oracle for frame-aligned block-sparse attention -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may import this package.  The CUDA library never calls it,
and it shares no code with the CUDA path (the one shared module is the seeded
input generator, which holds none of the method's arithmetic).

The arithmetic lives in ``oracle.c`` (plain C, fp64, compiled with gcc and
``-ffp-contract=off``); this file only compiles it and marshals numpy arrays.
Every function states the passage it follows; see the header of ``oracle.c``.

Pins (tests/test_oracle.py, CPU only): brute-force dense attention with an
explicit -inf mask, torch's fp64 scaled_dot_product_attention on an all-ones
mask, closed forms (q = 0, equal keys, constant values, one dominant key,
permutation inside a block, two-key softmax), the Cauchy-Schwarz invariant,
shift invariance of the softmax (bound shift vs max shift), and the fp32 norm
recipe against fp64 norms and exact special cases.  Per-head masks ([H, nbq,
nbkv]) are the same routines run head by head, pinned by brute force per head.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "oracle.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-o", _LIB_PATH, src, "-lm", "-lpthread"])
    return _LIB_PATH


_lib = None
_P = ctypes.c_void_p


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i32, i64, f32, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double
        lib.orc_allowed_csr.restype = i32
        lib.orc_allowed_csr.argtypes = [i32, i32, _P, _P, _P]
        lib.orc_attention.restype = None
        lib.orc_attention.argtypes = [i32, i32, i64, i64, i32, i32, _P, _P, _P, _P, f64, i64, _P, _P, _P, _P, _P,
                                      i32]
        lib.orc_row_norms_f64.restype = None
        lib.orc_row_norms_f64.argtypes = [i64, i32, _P, _P]
        lib.orc_row_bounds_f64.restype = None
        lib.orc_row_bounds_f64.argtypes = [i32, i64, i64, i32, _P, f64, _P, _P, _P]
        lib.orc_row_norms_f32.restype = None
        lib.orc_row_norms_f32.argtypes = [i64, i32, _P, _P]
        lib.orc_block_max_f32.restype = None
        lib.orc_block_max_f32.argtypes = [i32, i32, i32, _P, _P]
        lib.orc_row_bounds_f32.restype = None
        lib.orc_row_bounds_f32.argtypes = [i32, i64, i32, i32, _P, f32, _P, _P, _P]
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "bf16 tensors are passed as uint16 bit patterns"
    return a


def n_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def allowed_csr(mask: np.ndarray):
    """(row_ptr[nbq+1], col_idx[nnz]) of the allowed key blocks of each query block, ascending."""
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    nbq, nbkv = m.shape
    row_ptr = np.zeros(nbq + 1, dtype=np.int32)
    col_idx = np.zeros(max(nbq * nbkv, 1), dtype=np.int32)
    nnz = _load().orc_allowed_csr(nbq, nbkv, _ptr(m), _ptr(row_ptr), _ptr(col_idx))
    return row_ptr, col_idx[:nnz].copy()


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, mask: np.ndarray, block: int, scale: float,
              rows: Optional[np.ndarray] = None, shift: Optional[np.ndarray] = None,
              nthreads: Optional[int] = None):
    """fp64 masked softmax attention.

    q: uint16 bf16 bits [B,H,Lq,D]; k, v: [B,H,Lkv,D]; mask [Lq/block, Lkv/block].
    rows: global query row ids into B*H*Lq (None = all).
    Returns (O [nrows, D] fp64, LSE [nrows], l [nrows]) where l = sum_j exp(S_ij - shift_i)
    (shift = row max when ``shift`` is None)."""
    if np.ndim(mask) == 3:
        return _attention_per_head(q, k, v, np.asarray(mask), block, scale, rows, shift, nthreads)
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, H, Lq, D = q.shape
    Lkv = k.shape[2]
    assert k.shape == (B, H, Lkv, D) and v.shape == k.shape and Lq % block == 0 and Lkv % block == 0
    m = np.ascontiguousarray(mask, dtype=np.uint8)
    assert m.shape == (Lq // block, Lkv // block)
    nrows = B * H * Lq if rows is None else len(rows)
    rws = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    sh = None if shift is None else np.ascontiguousarray(shift, dtype=np.float64)
    if sh is not None:
        assert sh.shape == (nrows,)
    out = np.empty((nrows, D), dtype=np.float64)
    lse = np.empty(nrows, dtype=np.float64)
    lsum = np.empty(nrows, dtype=np.float64)
    _load().orc_attention(B, H, Lq, Lkv, D, block, _ptr(m), _ptr(q), _ptr(k), _ptr(v), float(scale), nrows,
                          _ptr(rws), _ptr(sh), _ptr(out), _ptr(lse), _ptr(lsum),
                          nthreads or n_threads())
    return out, lse, lsum


def _attention_per_head(q, k, v, mask, block, scale, rows, shift, nthreads):
    """One mask per head (mask [H, nbq, nbkv]): the heads are independent attentions, so
    head h is the plain masked attention of its own slice of Q, K, V under mask[h]."""
    B, H, Lq, D = q.shape
    assert mask.shape[0] == H
    grow = np.arange(B * H * Lq, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    bh, i = grow // Lq, grow % Lq
    b, h = bh // H, bh % H
    out = np.empty((len(grow), D), dtype=np.float64)
    lse = np.empty(len(grow), dtype=np.float64)
    lsum = np.empty(len(grow), dtype=np.float64)
    for hh in range(H):
        sel = np.nonzero(h == hh)[0]
        if len(sel) == 0:
            continue
        o_h, lse_h, l_h = attention(q[:, hh:hh + 1], k[:, hh:hh + 1], v[:, hh:hh + 1], mask[hh], block, scale,
                                    rows=b[sel] * Lq + i[sel], shift=None if shift is None else shift[sel],
                                    nthreads=nthreads)
        out[sel], lse[sel], lsum[sel] = o_h, lse_h, l_h
    return out, lse, lsum


def row_norms_f64(x: np.ndarray) -> np.ndarray:
    x = _u16(x)
    D = x.shape[-1]
    out = np.empty(x.shape[:-1], dtype=np.float64)
    _load().orc_row_norms_f64(x.size // D, D, _ptr(x), _ptr(out))
    return out


def row_bounds_f64(qnorm: np.ndarray, knorm: np.ndarray, mask: np.ndarray, block: int, scale: float):
    """M_i = scale * |q_i| * max_{j allowed} |k_j| in fp64; qnorm [B,H,Lq], knorm [B,H,Lkv]
    (mask [H, nbq, nbkv]: head h under mask[h])."""
    if np.ndim(mask) == 3:
        return np.concatenate([row_bounds_f64(qnorm[:, h:h + 1], knorm[:, h:h + 1], mask[h], block, scale)
                               for h in range(np.shape(qnorm)[1])], axis=1)
    qn = np.ascontiguousarray(qnorm, dtype=np.float64)
    kn = np.ascontiguousarray(knorm, dtype=np.float64)
    B, H, Lq = qn.shape
    out = np.empty_like(qn)
    _load().orc_row_bounds_f64(B * H, Lq, kn.shape[2], block, _ptr(np.ascontiguousarray(mask, dtype=np.uint8)),
                               float(scale), _ptr(qn), _ptr(kn), _ptr(out))
    return out


def row_norms_f32(x: np.ndarray) -> np.ndarray:
    """Canonical fp32 row norms (16 chunks, fmaf in order, xor-tree, sqrtf)."""
    x = _u16(x)
    D = x.shape[-1]
    assert D % 16 == 0
    out = np.empty(x.shape[:-1], dtype=np.float32)
    _load().orc_row_norms_f32(x.size // D, D, _ptr(x), _ptr(out))
    return out


def block_max_f32(knorm: np.ndarray, block: int) -> np.ndarray:
    kn = np.ascontiguousarray(knorm, dtype=np.float32)
    B, H, L = kn.shape
    nb = L // block
    out = np.empty((B, H, nb), dtype=np.float32)
    _load().orc_block_max_f32(B * H, nb, block, _ptr(kn), _ptr(out))
    return out


def row_bounds_f32(qnorm: np.ndarray, kmax: np.ndarray, mask: np.ndarray, block: int, scale: float):
    """fl(fl(scale * qnorm_i) * max over the allowed key blocks of kmax) (mask [H, nbq, nbkv]: head h under mask[h])."""
    if np.ndim(mask) == 3:
        return np.concatenate([row_bounds_f32(qnorm[:, h:h + 1], kmax[:, h:h + 1], mask[h], block, scale)
                               for h in range(np.shape(qnorm)[1])], axis=1)
    qn = np.ascontiguousarray(qnorm, dtype=np.float32)
    km = np.ascontiguousarray(kmax, dtype=np.float32)
    B, H, Lq = qn.shape
    out = np.empty_like(qn)
    _load().orc_row_bounds_f32(B * H, Lq, km.shape[2], block, _ptr(np.ascontiguousarray(mask, dtype=np.uint8)),
                               np.float32(scale), _ptr(qn), _ptr(km), _ptr(out))
    return out


def metadata_f32(q: np.ndarray, k: np.ndarray, mask: np.ndarray, block: int, scale: float):
    """(qnorm [B,H,Lq], kmax [B,H,nbkv], rowbound [B,H,Lq]) with the canonical fp32 recipe."""
    qn = row_norms_f32(q)
    kn = row_norms_f32(k)
    km = block_max_f32(kn, block)
    return qn, km, row_bounds_f32(qn, km, mask, block, scale)
