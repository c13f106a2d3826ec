"""Python binding of libbsattn.so (the C ABI in include/bsattn.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  The functions keep the C names (``bsattn_create_layout``,
``bsattn_row_bounds``, ``bsattn_forward``, ``bsattn_destroy``, ...).  Tensors
may be ``torch.Tensor`` (their ``data_ptr()`` is passed) or raw integer device
pointers; streams may be ``torch.cuda.Stream`` or raw ``cudaStream_t`` ints.
PyTorch is used only for device memory and streams.

There is no fallback: if the compiled library is missing this module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbsattn.so")

BSATTN_OK = 0
BSATTN_ERR_INVALID_ARG = 1
BSATTN_ERR_UNALIGNED_BLOCK = 2
BSATTN_ERR_UNSUPPORTED = 3
BSATTN_ERR_CUDA = 4
BSATTN_ERR_OOM = 5
BSATTN_ERR_TIMEOUT = 6
BSATTN_ERR_DEVICE = 7
BSATTN_ERR_INDEX = 8

BSATTN_BOUND = 0
BSATTN_ONLINE_MAX = 1
BSATTN_NO_FALLBACK = 2
BSATTN_BOUND_ONLY = 4
BSATTN_DEBUG_STALL = 0x100
BSATTN_DEBUG_CHECKS = 0x200
BSATTN_DEBUG_PLANT_INDEX = 0x400
BSATTN_ELIGIBLE_BOUND = 64.0
BSATTN_PLAN_ONLY = 0x10
BSATTN_MASK_PER_HEAD = 0x20

EXPORTED = ("bsattn_create_layout", "bsattn_create_layout_rect", "bsattn_row_bounds",
            "bsattn_row_bounds_from_norms", "bsattn_forward", "bsattn_destroy",
            "bsattn_status_string", "bsattn_query_stats", "bsattn_query_eligibility", "bsattn_layout_info",
            "bsattn_layout_export", "bsattn_layout_schedule",
            "bsattn_forward_noalloc", "bsattn_noalloc_query", "bsattn_forward_host")


class LayoutInfo(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("D", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("nb", ctypes.c_int32), ("L", ctypes.c_int64),
                ("nnz_blocks", ctypes.c_int32), ("kv_tile", ctypes.c_int32), ("key_tiles", ctypes.c_int32),
                ("q_tiles_per_block", ctypes.c_int32), ("n_units", ctypes.c_int32),
                ("mma_rows", ctypes.c_int64), ("useful_flop", ctypes.c_double), ("L_kv", ctypes.c_int64),
                ("nb_kv", ctypes.c_int32), ("mask_heads", ctypes.c_int32), ("n_segments", ctypes.c_int32),
                ("tail_units", ctypes.c_int32)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class BsattnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


_lib = None


def load(path: Optional[str] = None):
    """Load (once) and return the ctypes handle of libbsattn.so."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libbsattn.so not built ({p}); run block_sparse_video_row_b300._build.build()")
    lib = ctypes.CDLL(p)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.bsattn_create_layout.restype = i32
    lib.bsattn_create_layout.argtypes = [ctypes.POINTER(vp), i32, i32, i64, i32, i32, vp, i32]
    lib.bsattn_create_layout_rect.restype = i32
    lib.bsattn_create_layout_rect.argtypes = [ctypes.POINTER(vp), i32, i32, i64, i64, i32, i32, vp, i32]
    lib.bsattn_row_bounds.restype = i32
    lib.bsattn_row_bounds.argtypes = [vp, vp, vp, f32, vp, vp, vp, vp]
    lib.bsattn_row_bounds_from_norms.restype = i32
    lib.bsattn_row_bounds_from_norms.argtypes = [vp, vp, vp, f32, vp, vp, vp]
    lib.bsattn_forward.restype = i32
    lib.bsattn_forward.argtypes = [vp, vp, vp, vp, vp, f32, vp, vp, i32, vp]
    lib.bsattn_destroy.restype = None
    lib.bsattn_destroy.argtypes = [vp]
    lib.bsattn_status_string.restype = ctypes.c_char_p
    lib.bsattn_status_string.argtypes = [i32]
    lib.bsattn_query_stats.restype = i32
    lib.bsattn_query_stats.argtypes = [vp, ctypes.POINTER(i64), ctypes.POINTER(i64), ctypes.POINTER(i32), vp]
    lib.bsattn_query_eligibility.restype = i32
    lib.bsattn_query_eligibility.argtypes = [vp, ctypes.POINTER(i64), ctypes.POINTER(i64), vp]
    lib.bsattn_layout_info.restype = i32
    lib.bsattn_layout_info.argtypes = [vp, ctypes.POINTER(LayoutInfo)]
    lib.bsattn_forward_noalloc.restype = i32
    lib.bsattn_forward_noalloc.argtypes = [vp, vp, vp, vp, i32, i32, i64, i32, i32, vp, f32, vp, vp, i32, vp]
    lib.bsattn_noalloc_query.restype = i32
    lib.bsattn_noalloc_query.argtypes = [ctypes.POINTER(i64), ctypes.POINTER(i64), ctypes.POINTER(i32), vp]
    lib.bsattn_forward_host.restype = i32
    lib.bsattn_forward_host.argtypes = [vp, vp, vp, vp, vp, f32, vp, i32, i32, vp]
    lib.bsattn_layout_schedule.restype = i32
    lib.bsattn_layout_schedule.argtypes = [vp, i32, vp, ctypes.POINTER(i32)]
    lib.bsattn_layout_export.restype = i32
    lib.bsattn_layout_export.argtypes = [vp, vp, vp, vp, vp, vp]
    _lib = lib
    return lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    if isinstance(x, np.ndarray):
        return int(x.ctypes.data)
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _check_arg(name: str, x, numel: int, itemsize: int, on_device: bool) -> None:
    """A torch tensor or numpy array given for a C-ABI pointer must be contiguous and hold
    exactly `numel` elements of `itemsize` bytes on the side the call reads it from (the
    current CUDA device, or host memory): the library sees only the pointer, so a wrong
    size or a host pointer in a kernel would read out of bounds.  Integer pointers and
    None pass unchecked."""
    if x is None or isinstance(x, int):
        return
    if hasattr(x, "data_ptr"):  # torch.Tensor
        if not x.is_contiguous():
            raise ValueError(f"{name}: tensor must be contiguous")
        import torch
        ok = x.dtype == torch.float32 if itemsize == 4 else x.dtype in (torch.bfloat16, torch.int16, torch.uint16)
        if not ok:
            raise TypeError(f"{name}: expected {'bf16 (or its 16-bit pattern)' if itemsize == 2 else 'fp32'} "
                            f"elements, got {x.dtype}")
        if x.numel() != numel:
            raise ValueError(f"{name}: {x.numel()} elements, expected {numel}")
        if on_device:
            if not x.is_cuda or x.device.index != torch.cuda.current_device():
                raise TypeError(f"{name}: must be a tensor on the current CUDA device (got {x.device})")
        elif x.is_cuda:
            raise TypeError(f"{name}: must be a host tensor")
        return
    if isinstance(x, np.ndarray):
        if on_device:
            raise TypeError(f"{name}: a numpy array is host memory; this call takes device pointers")
        if not x.flags.c_contiguous:
            raise ValueError(f"{name}: array must be C-contiguous")
        if x.itemsize != itemsize or (itemsize == 4 and x.dtype.kind != "f"):
            raise TypeError(f"{name}: expected {'bf16 bits (2-byte)' if itemsize == 2 else 'float32'} elements")
        if x.size != numel:
            raise ValueError(f"{name}: {x.size} elements, expected {numel}")
        return
    raise TypeError(f"{name}: cannot pass {type(x)} as a pointer")


def _check_io(lay: "Layout", on_device: bool, q=None, k=None, v=None, o=None, rows=(), kmax=None) -> None:
    i = lay.info
    BH = i.B * i.H
    for name, x in (("q", q), ("o", o)):
        _check_arg(name, x, BH * i.L * i.D, 2, on_device)
    for name, x in (("k", k), ("v", v)):
        _check_arg(name, x, BH * i.L_kv * i.D, 2, on_device)
    for name, x in rows:
        _check_arg(name, x, BH * i.L, 4, on_device)
    _check_arg("kmax", kmax, BH * i.nb_kv, 4, on_device)


def _stream(s) -> Optional[int]:
    if s is None:
        try:
            import torch
            if torch.cuda.is_available():
                return int(torch.cuda.current_stream().cuda_stream)
        except Exception:
            pass
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def status_string(status: int) -> str:
    return load().bsattn_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != BSATTN_OK:
        raise BsattnError(status, what)


class Layout:
    """Owns a bsattn_layout_t; freed by destroy() or when garbage collected."""

    def __init__(self, handle: int, mask: np.ndarray):
        self.handle = handle
        self.mask = mask
        self.info = bsattn_layout_info(self)

    def destroy(self):
        if self.handle:
            load().bsattn_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.destroy()


def bsattn_create_layout(B: int, H: int, L: int, D: int, block_size: int, block_mask, flags: int = 0,
                         raise_on_error: bool = True, L_kv: Optional[int] = None):
    """Returns a Layout (or, with raise_on_error=False, the pair (status, Layout or None)).
    L_kv (key tokens, default L) other than L builds a streamed-chunk layout through
    bsattn_create_layout_rect; block_mask is then [L / block_size, L_kv / block_size].
    A 3-D block_mask [H, nb, nb_kv] gives each head its own mask (BSATTN_MASK_PER_HEAD)."""
    m = np.ascontiguousarray(np.asarray(block_mask), dtype=np.uint8)
    if m.ndim == 3:
        if m.shape[0] != H:
            raise ValueError(f"a per-head block_mask needs {H} masks, got {m.shape[0]}")
        flags |= BSATTN_MASK_PER_HEAD
    h = ctypes.c_void_p()
    if L_kv is None or L_kv == L:
        st = load().bsattn_create_layout(ctypes.byref(h), B, H, L, D, block_size, m.ctypes.data, flags)
        what = "bsattn_create_layout"
    else:
        st = load().bsattn_create_layout_rect(ctypes.byref(h), B, H, L, L_kv, D, block_size, m.ctypes.data, flags)
        what = "bsattn_create_layout_rect"
    if not raise_on_error:
        return st, (Layout(h.value, m) if st == BSATTN_OK else None)
    _check(st, what)
    return Layout(h.value, m)


def bsattn_create_layout_rect(B: int, H: int, L: int, L_kv: int, D: int, block_size: int, block_mask,
                              flags: int = 0, raise_on_error: bool = True):
    """A streamed-chunk layout: L query tokens reading L_kv key tokens."""
    return bsattn_create_layout(B, H, L, D, block_size, block_mask, flags, raise_on_error, L_kv=L_kv)


def bsattn_row_bounds(lay: Layout, q, k, scale: float, qnorm, kmax, rowbound, stream=None,
                      raise_on_error: bool = True) -> int:
    if lay.handle:
        _check_io(lay, True, q=q, k=k, rows=(("qnorm", qnorm), ("rowbound", rowbound)), kmax=kmax)
    st = load().bsattn_row_bounds(lay.handle, _ptr(q), _ptr(k), float(scale), _ptr(qnorm), _ptr(kmax),
                                  _ptr(rowbound), _stream(stream))
    if raise_on_error:
        _check(st, "bsattn_row_bounds")
    return st


def bsattn_row_bounds_from_norms(lay: Layout, qnorm, knorm, scale: float, kmax, rowbound, stream=None,
                                 raise_on_error: bool = True) -> int:
    if lay.handle:
        i = lay.info
        _check_io(lay, True, rows=(("qnorm", qnorm), ("rowbound", rowbound)), kmax=kmax)
        _check_arg("knorm", knorm, i.B * i.H * i.L_kv, 4, True)
    st = load().bsattn_row_bounds_from_norms(lay.handle, _ptr(qnorm), _ptr(knorm), float(scale), _ptr(kmax),
                                             _ptr(rowbound), _stream(stream))
    if raise_on_error:
        _check(st, "bsattn_row_bounds_from_norms")
    return st


def bsattn_forward(lay: Layout, q, k, v, o, scale: float, rowbound, lse=None, flags: int = 0, stream=None,
                   raise_on_error: bool = True) -> int:
    if lay.handle:
        _check_io(lay, True, q=q, k=k, v=v, o=o, rows=(("rowbound", rowbound), ("lse", lse)))
    st = load().bsattn_forward(lay.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), float(scale), _ptr(rowbound),
                               _ptr(lse), flags, _stream(stream))
    if raise_on_error:
        _check(st, "bsattn_forward")
    return st


def bsattn_forward_noalloc(q, k, v, o, B: int, H: int, L: int, D: int, block_size: int, block_mask,
                           scale: float, rowbound, lse=None, flags: int = 0, stream=None,
                           raise_on_error: bool = True) -> int:
    """The forward without a layout, for callers that may not allocate device memory
    (see bsattn_forward_noalloc in include/bsattn.h)."""
    m = np.ascontiguousarray(np.asarray(block_mask), dtype=np.uint8)
    if m.ndim == 3:
        if m.shape[0] != H:
            raise ValueError(f"a per-head block_mask needs {H} masks, got {m.shape[0]}")
        flags |= BSATTN_MASK_PER_HEAD
    n = B * H * L
    for name, x in (("q", q), ("k", k), ("v", v), ("o", o)):
        _check_arg(name, x, n * D, 2, True)
    for name, x in (("rowbound", rowbound), ("lse", lse)):
        _check_arg(name, x, n, 4, True)
    st = load().bsattn_forward_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, L, D, block_size, m.ctypes.data,
                                       float(scale), _ptr(rowbound), _ptr(lse), flags, _stream(stream))
    if raise_on_error:
        _check(st, "bsattn_forward_noalloc")
    return st


def bsattn_forward_host(lay: Layout, q, k, v, o, scale: float, lse=None, flags: int = 0,
                        pairs_per_chunk: int = 0, stream=None) -> None:
    """Row bounds + forward for host tensors (pinned CPU torch tensors or numpy arrays): copies,
    kernels and copy-out pipelined per chunk of (batch, head) pairs; synchronise `stream` before
    reading o."""
    _check_io(lay, False, q=q, k=k, v=v, o=o, rows=(("lse", lse),))
    _check(load().bsattn_forward_host(lay.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(o), float(scale), _ptr(lse),
                                      flags, pairs_per_chunk, _stream(stream)), "bsattn_forward_host")


def bsattn_destroy(lay: Layout) -> None:
    lay.destroy()


def bsattn_status_string(status: int) -> str:
    return status_string(status)


def bsattn_query_stats(lay: Layout, stream=None):
    """(fallback_rows, fallback_units, device_status); synchronises the stream."""
    rows, units, dev = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
    _check(load().bsattn_query_stats(lay.handle, ctypes.byref(rows), ctypes.byref(units), ctypes.byref(dev),
                                     _stream(stream)), "bsattn_query_stats")
    return rows.value, units.value, dev.value


def bsattn_query_eligibility(lay: Layout, stream=None):
    """(bound_units, online_units) of the last forward's eligibility check; synchronises the stream."""
    b, o = ctypes.c_int64(), ctypes.c_int64()
    _check(load().bsattn_query_eligibility(lay.handle, ctypes.byref(b), ctypes.byref(o), _stream(stream)),
           "bsattn_query_eligibility")
    return b.value, o.value


def bsattn_noalloc_query(stream=None):
    """(fallback_rows, fallback_units, device_status) of the last bsattn_forward_noalloc on the
    current device; synchronises the stream and allocates nothing."""
    rows, units, dev = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
    _check(load().bsattn_noalloc_query(ctypes.byref(rows), ctypes.byref(units), ctypes.byref(dev), _stream(stream)),
           "bsattn_noalloc_query")
    return rows.value, units.value, dev.value


def bsattn_layout_info(lay: Layout) -> LayoutInfo:
    info = LayoutInfo()
    _check(load().bsattn_layout_info(lay.handle, ctypes.byref(info)), "bsattn_layout_info")
    return info


def bsattn_layout_schedule(lay: Layout, grid: int) -> np.ndarray:
    """int32 [n_slots, 4]: slot k * grid + c is CTA c's k-th unit (empty slots are zeros)."""
    n = ctypes.c_int32()
    _check(load().bsattn_layout_schedule(lay.handle, grid, None, ctypes.byref(n)), "bsattn_layout_schedule")
    out = np.zeros((n.value, 4), dtype=np.int32)
    _check(load().bsattn_layout_schedule(lay.handle, grid, out.ctypes.data, ctypes.byref(n)),
           "bsattn_layout_schedule")
    return out


def bsattn_layout_export(lay: Layout, with_tiles: bool = False):
    """(row_ptr [mask_heads*nb+1], col_idx [nnz], units [n_units, 4]) as int32 numpy arrays; with_tiles
    adds (tile_ptr [n_segments+1], tiles [key_tiles, 2]).  Segment m*nb + qb is query block qb of
    mask m (m = 0 for a shared mask, the head for per-head masks); segments from mask_heads*nb on are
    packed-tail tiles, whose tiles' width words carry the allowed row groups in bits 16.."""
    i = lay.info
    nseg = max(1, i.mask_heads) * i.nb  # (mask, query block) segments
    row_ptr = np.zeros(nseg + 1, np.int32)
    col_idx = np.zeros(max(i.nnz_blocks, 1), np.int32)
    units = np.zeros((i.n_units, 4), np.int32)
    tile_ptr = np.zeros(max(i.n_segments, nseg) + 1, np.int32)
    tiles = np.zeros((max(i.key_tiles, 1), 2), np.int32)
    _check(load().bsattn_layout_export(lay.handle, row_ptr.ctypes.data, col_idx.ctypes.data, units.ctypes.data,
                                       tile_ptr.ctypes.data, tiles.ctypes.data), "bsattn_layout_export")
    out = (row_ptr, col_idx[:i.nnz_blocks].copy(), units)
    if with_tiles:
        out += (tile_ptr, tiles[:i.key_tiles].copy())
    return out


# ------------------------------------------------------------------------------------------------
# convenience: one call for bounds + forward on torch tensors


def attention(q, k, v, block_mask, block_size: int, scale: Optional[float] = None, flags: int = 0,
              return_lse: bool = False, layout: Optional[Layout] = None, stream=None):
    """O = block-sparse attention of bf16 [B,H,L,D] CUDA tensors (allocates O, metadata and LSE with torch)."""
    import torch
    B, H, L, D = q.shape
    L_kv = k.shape[2]
    if scale is None:
        scale = float(np.float32(1.0 / np.sqrt(D)))
    lay = layout or bsattn_create_layout(B, H, L, D, block_size, block_mask, L_kv=L_kv)
    nb = L_kv // block_size
    dev = q.device
    o = torch.empty_like(q)
    qnorm = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    kmax = torch.empty((B, H, nb), dtype=torch.float32, device=dev)
    rowbound = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=dev) if return_lse else None
    if not (flags & BSATTN_ONLINE_MAX):
        bsattn_row_bounds(lay, q, k, scale, qnorm, kmax, rowbound, stream)
    bsattn_forward(lay, q, k, v, o, scale, rowbound, lse, flags, stream)
    return (o, lse) if return_lse else o
