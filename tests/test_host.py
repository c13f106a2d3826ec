"""Host-side logic of the C ABI, on CPU: exported symbols, the plan, argument checks.

No compute call is made here (there may be no GPU): plan-only layouts are inspected
and every error path that returns before touching a device is exercised.
"""
import os
import re

import numpy as np
import pytest

import oracle
from block_sparse_video_row_b300 import _build, bsattn, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return bsattn.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "bsattn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bsattn_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert set(declared) == set(bsattn.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name


def check_tiles(mask, bs, tile_ptr, tiles):
    """Key tiles of each query frame: exactly its allowed keys, in order; widths a multiple
    of 16 and at most 128; a tile never spans a masked frame; within a run of consecutive
    allowed frames every tile but the last is 128 keys."""
    nb, nbkv = mask.shape
    for qb in range(nb):
        t = tiles[tile_ptr[qb]:tile_ptr[qb + 1]]
        keys = np.concatenate([np.arange(s, s + w) for s, w in t]) if len(t) else np.zeros(0, int)
        allowed = np.concatenate([np.arange(kb * bs, (kb + 1) * bs) for kb in range(nbkv) if mask[qb, kb]]
                                 ) if mask[qb].any() else np.zeros(0, int)
        assert np.array_equal(keys, allowed)
        assert np.all(t[:, 1] % 16 == 0) and np.all((t[:, 1] >= 16) & (t[:, 1] <= 128))
        for (s, w), nxt in zip(t, list(t[1:]) + [None]):
            if nxt is not None and nxt[0] == s + w:   # same run continues
                assert w == 128


def check_units(masks, bs, H, units, tile_ptr, tiles, BH):
    """Every (sequence, frame, query tile) exactly once.  A unit is 1 or 2 query tiles of one
    frame, or a packed tile of frame tails (b*H+h, first frame, segment, -n): the last query
    tile of frames qb0 .. qb0+n-1, reading the key tiles of its segment.  Those are cut at frame
    edges, cover exactly the key frames any of its frames reads, and carry in bits 16.. of the
    width the frames (row groups) allowed to read them.  Packing happens only for frames with an
    odd number of query tiles and a tail of at most 64 rows, and only when cheaper than the
    frames' own tail units."""
    nb, nbkv = masks.shape[1], masks.shape[2]
    nqt = -(-bs // 128)
    tail_rows = bs - (nqt - 1) * 128
    seen = np.zeros((BH, nb, nqt), np.int32)
    for bh, qb, z, w in units:
        if w > 0:
            assert w in (1, 2) and z % 2 == 0 and z + w <= nqt
            seen[bh, qb, z:z + w] += 1
            continue
        n = -w
        assert nqt % 2 == 1 and 2 * tail_rows <= 128 and 2 <= n <= min(8, 128 // tail_rows)
        m = masks[bh % H] if len(masks) > 1 else masks[0]
        seen[bh, qb:qb + n, nqt - 1] += 1
        assert z >= len(masks) * nb
        t = tiles[tile_ptr[z]:tile_ptr[z + 1]]
        width, groups = t[:, 1] & 0xFFFF, t[:, 1] >> 16
        frames = t[:, 0] // bs
        assert np.all(frames == (t[:, 0] + width - 1) // bs)        # within one frame
        union = sorted({kb for g in range(n) for kb in range(nbkv) if m[qb + g, kb]})
        assert list(np.unique(frames)) == union
        for kb in union:                                            # each frame whole, in order
            sel = t[frames == kb]
            keys = np.concatenate([np.arange(a, a + (b & 0xFFFF)) for a, b in sel])
            assert np.array_equal(keys, np.arange(kb * bs, (kb + 1) * bs))
        for (a, _), gbits, kb in zip(t, groups, frames):
            assert gbits == sum(1 << g for g in range(n) if m[qb + g, kb])
        own = sum(tile_ptr[qb + g + 1] - tile_ptr[qb + g] for g in range(n)) if len(masks) == 1 else None
        if own is not None:
            assert len(t) < own                                     # cheaper than n own tail units
    assert np.all(seen == 1)


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_plan_matches_oracle(lib, name):
    w = synth.WORKLOADS[name]
    mask = w.block_mask()
    masks = mask if mask.ndim == 3 else mask[None]  # per-head plans: segment m * nb + qb is mask m
    lay = bsattn.bsattn_create_layout(w.B, w.H, w.L, w.D, w.block, mask, bsattn.BSATTN_PLAN_ONLY, L_kv=w.L_kv)
    info = lay.info
    assert info.mask_heads == len(masks)
    row_ptr, col_idx, units, tile_ptr, tiles = bsattn.bsattn_layout_export(lay, with_tiles=True)
    orp, oci = [0], []
    for m in masks:
        rp, ci = oracle.allowed_csr(m)
        orp += list(rp[1:] + orp[-1])
        oci += list(ci)
    assert np.array_equal(row_ptr, orp) and np.array_equal(col_idx, oci)
    assert info.nnz_blocks == len(oci) and info.nb == w.nb
    assert info.L == w.L and info.L_kv == w.L_kv and info.nb_kv == w.nb_kv
    assert info.kv_tile == 128 and info.key_tiles == len(tiles)
    for mi, m in enumerate(masks):
        seg = tile_ptr[mi * w.nb:(mi + 1) * w.nb + 1]
        check_tiles(m, w.block, seg, tiles)
    nqt = -(-w.block // 128)
    assert info.q_tiles_per_block == nqt
    assert abs(info.useful_flop - synth.useful_flop(w)) == 0
    check_units(masks, w.block, w.H, units, tile_ptr, tiles, w.B * w.H)
    # plan order: (head, frame, first query tile), a packed tail after its last frame's units
    last = np.where(units[:, 3] < 0, units[:, 1] - units[:, 3] - 1, units[:, 1])
    pos = np.where(units[:, 3] < 0, nqt, units[:, 2])
    key = (units[:, 0].astype(np.int64) * w.nb + last) * (nqt + 1) + pos
    assert np.all(np.diff(key) > 0)
    lay.destroy()


def _unit_cost(units, tile_ptr, H, nb, per_head):
    # the documented model: 100 per key tile for a unit of two query tiles, 83 for one, plus 150
    # a packed tail (w < 0) reads the tiles of its own segment z, as one query tile
    segment = np.where(units[:, 3] < 0, units[:, 2], (units[:, 0] % H if per_head else 0) * nb + units[:, 1])
    ntile = np.diff(tile_ptr)[segment]
    return ntile * np.where(units[:, 3] == 2, 100, 83) + 150


@pytest.mark.parametrize("name,grid", [("720p", 148), ("stream", 148), ("small", 148), ("small", 7),
                                       ("720p_heads", 148), ("1080p", 148), ("tiny", 148)])
def test_schedule_deals_every_unit_once_head_major_then_by_cost(lib, name, grid):
    w = synth.WORKLOADS[name]
    mask = w.block_mask()
    lay = bsattn.bsattn_create_layout(w.B, w.H, w.L, w.D, w.block, mask, bsattn.BSATTN_PLAN_ONLY, L_kv=w.L_kv)
    _, _, units, tile_ptr, _ = bsattn.bsattn_layout_export(lay, with_tiles=True)
    n = len(units)
    g = min(grid, n)
    slots = bsattn.bsattn_layout_schedule(lay, g)
    assert len(slots) % g == 0
    real = slots[:, 3] != 0
    assert np.all(slots[~real] == 0)
    # every unit exactly once
    got = sorted(map(tuple, slots[real]))
    assert got == sorted(map(tuple, units))
    # the order the units were dealt in: plan order, then the last 4 * grid units by cost
    cost_of = {tuple(u): c for u, c in zip(units, _unit_cost(units, tile_ptr, w.H, w.nb, mask.ndim == 3))}
    n_tail = min(n, 4 * g)
    head = [tuple(u) for u in units[:n - n_tail]]
    tail = sorted((tuple(u) for u in units[n - n_tail:]), key=lambda u: -cost_of[u])  # stable
    # replay the least-loaded deal (ties: lowest CTA) and compare slot by slot
    import heapq
    heap = [(0, c) for c in range(g)]
    per = [[] for _ in range(g)]
    for u in head + tail:
        load, c = heapq.heappop(heap)
        per[c].append(u)
        heapq.heappush(heap, (load + cost_of[u], c))
    K = max(len(x) for x in per)
    assert len(slots) == K * g
    for kk in range(K):
        for c in range(g):
            want = per[c][kk] if kk < len(per[c]) else (0, 0, 0, 0)
            assert tuple(slots[kk * g + c]) == want
    # balance: the most loaded CTA is within one unit of the mean load
    loads = [sum(cost_of[u] for u in x) for x in per]
    assert max(loads) <= sum(loads) / g + max(cost_of.values())
    lay.destroy()


def test_plan_edge_shapes(lib):
    # single frame of 16 tokens; a frame that reads nothing; ragged 128-row tiles
    for (L, bs) in [(16, 16), (48, 16), (400, 400), (1040, 208), (272, 272)]:
        nb = L // bs
        mask = np.ones((nb, nb), np.uint8)
        if nb > 1:
            mask[1, :] = 0
        lay = bsattn.bsattn_create_layout(2, 3, L, 64, bs, mask, bsattn.BSATTN_PLAN_ONLY)
        _, _, units, tile_ptr, tiles = bsattn.bsattn_layout_export(lay, with_tiles=True)
        check_tiles(mask, bs, tile_ptr, tiles)
        assert len(units) == lay.info.n_units == 6 * nb * ((-(-bs // 128) + 1) // 2)


@pytest.mark.parametrize("args,status", [
    ((1, 1, 192, 64, 40), bsattn.BSATTN_ERR_UNALIGNED_BLOCK),     # block not a multiple of 16
    ((1, 1, 200, 64, 48), bsattn.BSATTN_ERR_UNALIGNED_BLOCK),     # L not a multiple of block
    ((1, 1, 192, 96, 48), bsattn.BSATTN_ERR_UNSUPPORTED),         # head dim 96
    ((0, 1, 192, 64, 48), bsattn.BSATTN_ERR_INVALID_ARG),         # B = 0
    ((1, 1, 192, 64, 0), bsattn.BSATTN_ERR_INVALID_ARG),          # block 0
    ((1, 1, 16 * 5000, 64, 16), bsattn.BSATTN_ERR_UNSUPPORTED),   # too many frames
    ((40000, 64, 1024, 64, 16 * 64), bsattn.BSATTN_ERR_UNSUPPORTED),  # B*H*L beyond int32
])
def test_create_rejects_bad_arguments(lib, args, status):
    B, H, L, D, bs = args
    nb = max(L // bs, 1) if bs else 1
    mask = np.ones((min(nb, 5000), min(nb, 5000)), np.uint8)
    st, lay = bsattn.bsattn_create_layout(B, H, L, D, bs, mask, bsattn.BSATTN_PLAN_ONLY, raise_on_error=False)
    assert st == status and lay is None


def test_rect_create_checks_the_key_side(lib):
    mask = np.ones((2, 5), np.uint8)
    st, lay = bsattn.bsattn_create_layout(1, 1, 32, 64, 16, mask, bsattn.BSATTN_PLAN_ONLY, raise_on_error=False,
                                          L_kv=88)  # 88 keys: not a multiple of the block
    assert st == bsattn.BSATTN_ERR_UNALIGNED_BLOCK and lay is None
    st, lay = bsattn.bsattn_create_layout(1, 1, 96, 64, 16, np.ones((6, 5), np.uint8), bsattn.BSATTN_PLAN_ONLY,
                                          raise_on_error=False, L_kv=80)  # more query than key tokens
    assert st == bsattn.BSATTN_ERR_UNSUPPORTED and lay is None
    lay = bsattn.bsattn_create_layout(1, 1, 32, 64, 16, mask, bsattn.BSATTN_PLAN_ONLY, L_kv=80)
    assert (lay.info.nb, lay.info.nb_kv, lay.info.L, lay.info.L_kv) == (2, 5, 32, 80)
    assert lay.info.nnz_blocks == 10
    lay.destroy()


def test_create_rejects_null_mask_and_bad_flags(lib):
    import ctypes
    h = ctypes.c_void_p()
    assert lib.bsattn_create_layout(ctypes.byref(h), 1, 1, 192, 64, 48, None, 0) == bsattn.BSATTN_ERR_INVALID_ARG
    assert h.value is None
    m = np.ones((4, 4), np.uint8)
    assert lib.bsattn_create_layout(ctypes.byref(h), 1, 1, 192, 64, 48, m.ctypes.data, 0x4) == \
        bsattn.BSATTN_ERR_INVALID_ARG
    assert lib.bsattn_create_layout(None, 1, 1, 192, 64, 48, m.ctypes.data, 0) == bsattn.BSATTN_ERR_INVALID_ARG


def test_plan_only_layout_refuses_device_calls(lib):
    lay = bsattn.bsattn_create_layout(1, 2, 192, 64, 48, synth.window_mask(4, 1), bsattn.BSATTN_PLAN_ONLY)
    fake = 1 << 20  # never dereferenced: the plan-only check comes first
    assert bsattn.bsattn_row_bounds(lay, fake, fake, 0.125, fake, fake, fake, 0, raise_on_error=False) == \
        bsattn.BSATTN_ERR_INVALID_ARG
    assert bsattn.bsattn_forward(lay, fake, fake, fake, fake, 0.125, fake, None, 0, 0, raise_on_error=False) == \
        bsattn.BSATTN_ERR_INVALID_ARG
    assert bsattn.bsattn_row_bounds_from_norms(lay, fake, fake, 0.125, fake, fake, 0, raise_on_error=False) == \
        bsattn.BSATTN_ERR_INVALID_ARG
    lay.destroy()
    lib.bsattn_destroy(None)  # NULL is ignored


def test_new_entry_points_reject_bad_arguments(lib):
    import ctypes
    lay = bsattn.bsattn_create_layout(1, 2, 192, 64, 48, synth.window_mask(4, 1), bsattn.BSATTN_PLAN_ONLY)
    n = ctypes.c_int32()
    # the schedule needs a grid of at least one CTA and somewhere to put the slot count
    assert lib.bsattn_layout_schedule(lay.handle, 0, None, ctypes.byref(n)) == bsattn.BSATTN_ERR_INVALID_ARG
    assert lib.bsattn_layout_schedule(lay.handle, 4, None, None) == bsattn.BSATTN_ERR_INVALID_ARG
    assert lib.bsattn_layout_schedule(None, 4, None, ctypes.byref(n)) == bsattn.BSATTN_ERR_INVALID_ARG
    assert lib.bsattn_layout_schedule(lay.handle, 3, None, ctypes.byref(n)) == bsattn.BSATTN_OK
    assert n.value % 3 == 0 and n.value >= lay.info.n_units
    # eligibility counts need a device layout
    b, o = ctypes.c_int64(), ctypes.c_int64()
    assert lib.bsattn_query_eligibility(lay.handle, ctypes.byref(b), ctypes.byref(o), None) == \
        bsattn.BSATTN_ERR_INVALID_ARG
    lay.destroy()


def test_noalloc_entry_points_without_a_gpu_report_an_error(lib):
    import ctypes
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rows, units, dev = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
    st = lib.bsattn_noalloc_query(ctypes.byref(rows), ctypes.byref(units), ctypes.byref(dev), None)
    assert st in (bsattn.BSATTN_ERR_DEVICE, bsattn.BSATTN_ERR_CUDA)
    fake = 1 << 20  # never dereferenced: the device look-up fails first
    st = bsattn.bsattn_forward_noalloc(fake, fake, fake, fake, 1, 2, 192, 64, 48, synth.window_mask(4, 1), 0.125,
                                       fake, None, 0, raise_on_error=False)
    assert st in (bsattn.BSATTN_ERR_DEVICE, bsattn.BSATTN_ERR_CUDA)


def test_status_strings(lib):
    for st in range(9):
        assert isinstance(bsattn.status_string(st), str) and bsattn.status_string(st)
    assert bsattn.status_string(99) == "unknown status"


def test_device_layout_without_gpu_reports_an_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, lay = bsattn.bsattn_create_layout(1, 2, 192, 64, 48, synth.window_mask(4, 1), 0, raise_on_error=False)
    assert st in (bsattn.BSATTN_ERR_DEVICE, bsattn.BSATTN_ERR_CUDA) and lay is None


def test_binding_checks_tensor_arguments(lib):
    # The C ABI sees only pointers, so the binding checks torch / numpy arguments first:
    # a host tensor where device memory is read, a wrong element type, a strided view or
    # a wrong element count is refused before any call into the library.
    import torch
    lay = bsattn.bsattn_create_layout(1, 2, 192, 64, 48, synth.window_mask(4, 1), bsattn.BSATTN_PLAN_ONLY)
    q = torch.zeros(1, 2, 192, 64, dtype=torch.bfloat16)
    rb = torch.zeros(1, 2, 192)
    with pytest.raises(TypeError, match="CUDA device"):
        bsattn.bsattn_forward(lay, q, q, q, q, 0.125, rb)
    with pytest.raises(TypeError, match="bf16"):
        bsattn.bsattn_forward(lay, q.float(), q, q, q, 0.125, rb)
    with pytest.raises(ValueError, match="contiguous"):
        bsattn.bsattn_forward(lay, q.transpose(2, 3), q, q, q, 0.125, rb)
    with pytest.raises(TypeError, match="fp32"):
        bsattn.bsattn_row_bounds(lay, 1 << 20, 1 << 20, 0.125, rb.double(), 1 << 20, 1 << 20)
    with pytest.raises(ValueError, match="elements"):
        bsattn.bsattn_forward_host(lay, q, q, q, q[:, :1], 0.125)
    with pytest.raises(TypeError, match="host"):
        bsattn.bsattn_forward_noalloc(np.zeros(q.shape, np.uint16), 1 << 20, 1 << 20, 1 << 20, 1, 2, 192, 64, 48,
                                      synth.window_mask(4, 1), 0.125, 1 << 20)
    # right sizes on the host pass the binding; the library then refuses the plan-only layout
    with pytest.raises(bsattn.BsattnError):
        bsattn.bsattn_forward_host(lay, q, q, q, torch.empty_like(q), 0.125)
    lay.destroy()


C_CLIENT = r"""
#include <stdio.h>
#include <stdlib.h>
#include "bsattn.h"

/* A plain C client of the library: plan a 4-frame window mask on the host only and
   read the plan back.  Every declared entry point is referenced, so the link step
   also checks that the library exports them with C linkage. */
int main(void) {
    void *volatile refs[] = {
        (void *)bsattn_create_layout, (void *)bsattn_create_layout_rect, (void *)bsattn_row_bounds,
        (void *)bsattn_forward, (void *)bsattn_forward_host, (void *)bsattn_forward_noalloc,
        (void *)bsattn_destroy, (void *)bsattn_status_string, (void *)bsattn_query_stats,
        (void *)bsattn_layout_info, (void *)bsattn_layout_export};
    uint8_t mask[16];
    int i, j;
    for (i = 0; i < 4; ++i)
        for (j = 0; j < 4; ++j) mask[4 * i + j] = (uint8_t)(i - j <= 1 && j - i <= 1);
    bsattn_layout_t lay = NULL;
    bsattn_status st = bsattn_create_layout(&lay, 1, 2, 192, 64, 48, mask, BSATTN_PLAN_ONLY);
    if (st != BSATTN_OK) { printf("create: %s\n", bsattn_status_string(st)); return 1; }
    bsattn_layout_info_t info;
    if (bsattn_layout_info(lay, &info) != BSATTN_OK) return 2;
    int32_t *row_ptr = malloc(sizeof(int32_t) * (size_t)(info.nb + 1));
    int32_t *col_idx = malloc(sizeof(int32_t) * (size_t)info.nnz_blocks);
    int32_t *units = malloc(sizeof(int32_t) * 4 * (size_t)info.n_units);
    if (bsattn_layout_export(lay, row_ptr, col_idx, units, NULL, NULL) != BSATTN_OK) return 3;
    printf("nb=%d nnz=%d units=%d row_ptr_last=%d refs=%d\n", info.nb, info.nnz_blocks, info.n_units,
           row_ptr[info.nb], (int)(sizeof(refs) / sizeof(refs[0])));
    bsattn_destroy(lay);
    free(row_ptr); free(col_idx); free(units);
    return 0;
}
"""


def test_header_is_plain_c_and_a_c_client_links_and_runs(lib, tmp_path):
    # include/bsattn.h compiles as C11 with warnings as errors, and a C program using it
    # links against the in-tree library and plans a layout on the host.
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(_build.LIB)
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(exe), "-L", libdir, "-lbsattn", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.strip() == "nb=4 nnz=10 units=8 row_ptr_last=10 refs=11"


def test_plan_matches_oracle_on_random_masks(lib):
    # Random shapes and masks (shared, streamed and per head, some rows empty): the plan's
    # CSR equals the oracle's per mask, and the key tiles cover exactly the allowed keys.
    rng = np.random.default_rng(2024)
    for trial in range(60):
        bs = int(rng.choice([16, 48, 128, 144, 272, 400]))
        nbkv = int(rng.integers(1, 9))
        nb = int(rng.integers(1, nbkv + 1))
        H = int(rng.integers(1, 5))
        per_head = bool(rng.integers(0, 2))
        shape = (H, nb, nbkv) if per_head else (nb, nbkv)
        mask = (rng.random(shape) < rng.uniform(0.1, 0.9)).astype(np.uint8)
        lay = bsattn.bsattn_create_layout(2, H, nb * bs, 64, bs, mask, bsattn.BSATTN_PLAN_ONLY, L_kv=nbkv * bs)
        row_ptr, col_idx, units, tile_ptr, tiles = bsattn.bsattn_layout_export(lay, with_tiles=True)
        masks = mask if per_head else mask[None]
        assert lay.info.mask_heads == len(masks)
        orp, oci = [0], []
        for m in masks:
            rp, ci = oracle.allowed_csr(m)
            orp += list(rp[1:] + orp[-1])
            oci += list(ci)
        assert np.array_equal(row_ptr, orp) and np.array_equal(col_idx, oci), trial
        for mi, m in enumerate(masks):
            check_tiles(m, bs, tile_ptr[mi * nb:(mi + 1) * nb + 1], tiles)
        check_units(masks, bs, H, units, tile_ptr, tiles, 2 * H)
        lay.destroy()


def test_binding_constants_match_the_header():
    # Every BSATTN_* enum value and numeric #define in include/bsattn.h has the same value in
    # the Python binding (no drift between the C ABI and its binding).
    src = open(os.path.join(ROOT, "include", "bsattn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    vals = {}
    for name, v in re.findall(r"\b(BSATTN_[A-Z_]+)\s*=\s*(0x[0-9A-Fa-f]+|\d+)", src):
        vals[name] = int(v, 0)
    for name, v in re.findall(r"#define\s+(BSATTN_[A-Z_]+)\s+([0-9.]+)f?\b", src):
        vals[name] = float(v)
    assert len(vals) > 15
    for name, v in vals.items():
        if name.startswith("BSATTN_MAX_") or name == "BSATTN_NOALLOC_SCRATCH_BYTES":
            continue
        assert hasattr(bsattn, name), name
        assert getattr(bsattn, name) == v, (name, getattr(bsattn, name), v)
