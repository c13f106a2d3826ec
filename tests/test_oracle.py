"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test fixes the oracle to mathematics or an independent route: brute-force
dense attention with an explicit -inf mask (numpy), torch's fp64
scaled_dot_product_attention, closed forms, the Cauchy-Schwarz invariant, the
shift invariance of softmax that the method relies on, exact special cases of
the fp32 norm recipe, and the hand-counted workload sizes in tests/golden.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from block_sparse_video_row_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "workloads.json")


def _f64(x):
    return synth.bf16_bits_to_f64(x)


def _rand_qkv(B, H, L, D, seed=7):
    q = synth.tensor_bf16(seed, synth.TAG_Q, B, H, L, D)
    k = synth.tensor_bf16(seed, synth.TAG_K, B, H, L, D)
    v = synth.tensor_bf16(seed, synth.TAG_V, B, H, L, D)
    return q, k, v


def _brute_dense(q, k, v, mask, bs, scale):
    """Dense route: full S = scale Q K^T over every key, element mask from the block mask
    (q [B,H,Lq,D], k and v [B,H,Lkv,D], mask [Lq/bs, Lkv/bs])."""
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    B, H, L, D = qf.shape
    Lkv = kf.shape[2]
    allowed = mask.astype(bool)[(np.arange(L) // bs)[:, None], (np.arange(Lkv) // bs)[None, :]]  # [Lq, Lkv]
    O = np.zeros((B, H, L, D))
    LSE = np.full((B, H, L), -np.inf)
    for b in range(B):
        for h in range(H):
            S = scale * (qf[b, h] @ kf[b, h].T)
            S = np.where(allowed, S, -np.inf)
            mu = S.max(axis=1, keepdims=True)
            has = np.isfinite(mu[:, 0])
            mu = np.where(np.isfinite(mu), mu, 0.0)
            P = np.exp(S - mu)
            l = P.sum(axis=1, keepdims=True)
            O[b, h] = np.where(has[:, None], (P @ vf[b, h]) / np.where(l > 0, l, 1.0), 0.0)
            LSE[b, h] = np.where(has, mu[:, 0] + np.log(np.where(l[:, 0] > 0, l[:, 0], 1.0)), -np.inf)
    return O.reshape(-1, D), LSE.reshape(-1)


# ------------------------------------------------------------------------------------------------
# attention values


@pytest.mark.parametrize("name", ["tiny"])
def test_brute_force_dense_tiny(name):
    w = synth.WORKLOADS[name]
    q, k, v = synth.make_qkv(w)
    O, lse, _ = oracle.attention(q, k, v, w.block_mask(), w.block, w.scale)
    Ob, lseb = _brute_dense(q, k, v, w.block_mask(), w.block, w.scale)
    assert np.max(np.abs(O - Ob)) <= 1e-12
    assert np.max(np.abs(lse - lseb)) <= 1e-12


def test_brute_force_streamed_chunk():
    # queries of a 3-frame chunk reading 4 context frames plus the chunk (7 key frames), with a
    # rectangular mask that is not a slice of any symmetric rule, and one query frame reading nothing
    B, H, D, bs, nq, nkv = 2, 2, 64, 16, 3, 7
    mask = np.zeros((nq, nkv), np.uint8)
    mask[0, [0, 3, 4]] = 1
    mask[1, [0, 1, 5, 6]] = 1
    q = synth.tensor_bf16(11, synth.TAG_Q, B, H, nq * bs, D)
    k = synth.tensor_bf16(11, synth.TAG_K, B, H, nkv * bs, D)
    v = synth.tensor_bf16(11, synth.TAG_V, B, H, nkv * bs, D)
    scale = float(np.float32(1 / 8))
    O, lse, _ = oracle.attention(q, k, v, mask, bs, scale)
    Ob, lseb = _brute_dense(q, k, v, mask, bs, scale)
    assert np.max(np.abs(O - Ob)) <= 1e-12
    fin = np.isfinite(lseb)
    assert np.array_equal(np.isfinite(lse), fin) and np.max(np.abs(lse[fin] - lseb[fin])) <= 1e-12
    # the frame that reads nothing: O = 0
    rows = (np.arange(B * H * nq * bs) % (nq * bs)) // bs == 2
    assert np.all(O[rows] == 0)


def test_streamed_chunk_equals_last_rows_of_the_full_window():
    # a chunk's queries are the last query rows of the self-attention problem over all frames, and
    # its mask the last rows of that problem's mask: the outputs must be the same rows
    w = synth.WORKLOADS["stream_small"]
    wf = synth.Workload("full", w.B, w.H, w.D, w.frames, w.block, w.mask, w.keys, w.seed)
    q, k, v = synth.make_qkv(w)
    qf, kf, vf = synth.make_qkv(wf)
    assert np.array_equal(k, kf) and np.array_equal(q, qf[:, :, w.L_kv - w.L:])
    rows = np.array([0, 57, 399, 400, 1199], dtype=np.int64)
    O, lse, _ = oracle.attention(q, k, v, w.block_mask(), w.block, w.scale, rows=rows)
    Of, lsef, _ = oracle.attention(qf, kf, vf, wf.block_mask(), w.block, w.scale, rows=rows + (w.L_kv - w.L))
    assert np.array_equal(O, Of) and np.array_equal(lse, lsef)


def test_sdpa_streamed_all_ones():
    # every chunk query reads every key: torch's fp64 scaled_dot_product_attention with Lq != Lkv
    B, H, D, bs, nq, nkv = 1, 2, 64, 16, 2, 5
    q = synth.tensor_bf16(5, synth.TAG_Q, B, H, nq * bs, D)
    k = synth.tensor_bf16(5, synth.TAG_K, B, H, nkv * bs, D)
    v = synth.tensor_bf16(5, synth.TAG_V, B, H, nkv * bs, D)
    scale = 0.125
    O, _, _ = oracle.attention(q, k, v, np.ones((nq, nkv), np.uint8), bs, scale)
    t = [torch.from_numpy(_f64(x)) for x in (q, k, v)]
    ref = torch.nn.functional.scaled_dot_product_attention(*t, scale=scale).numpy().reshape(-1, D)
    assert np.max(np.abs(O - ref)) <= 1e-12


def test_streamed_metadata_bounds_and_cauchy_schwarz():
    # rectangular metadata: fp32 recipe against fp64 norms; every unmasked logit below its bound
    B, H, D, bs, nq, nkv = 1, 2, 64, 16, 2, 5
    mask = synth.window_mask(nkv, 1, True)[nkv - nq:]
    q = synth.tensor_bf16(9, synth.TAG_Q, B, H, nq * bs, D)
    k = synth.tensor_bf16(9, synth.TAG_K, B, H, nkv * bs, D)
    qn, km, rb = oracle.metadata_f32(q, k, mask, bs, 0.125)
    assert km.shape == (B, H, nkv) and rb.shape == (B, H, nq * bs)
    M = oracle.row_bounds_f64(oracle.row_norms_f64(q), oracle.row_norms_f64(k), mask, bs, 0.125)
    assert np.max(np.abs(rb - M) / M) <= 2.0 ** -20
    qf, kf = _f64(q), _f64(k)
    for h in range(H):
        S = 0.125 * qf[0, h] @ kf[0, h].T
        allowed = mask.astype(bool)[(np.arange(nq * bs) // bs)[:, None], (np.arange(nkv * bs) // bs)[None, :]]
        assert np.all(S[allowed] <= np.broadcast_to(M[0, h][:, None], S.shape)[allowed])


def test_brute_force_asymmetric_mask():
    # first frame global is not symmetric: a transposed mask would fail here
    B, H, D, nb, bs = 1, 2, 64, 8, 16
    mask = synth.window_mask(nb, 2, True)
    assert not np.array_equal(mask, mask.T)
    q, k, v = _rand_qkv(B, H, nb * bs, D)
    scale = float(np.float32(1 / 8))
    O, lse, _ = oracle.attention(q, k, v, mask, bs, scale)
    Ob, lseb = _brute_dense(q, k, v, mask, bs, scale)
    assert np.max(np.abs(O - Ob)) <= 1e-12
    assert np.max(np.abs(lse - lseb)) <= 1e-12
    Ot, _, _ = oracle.attention(q, k, v, mask.T.copy(), bs, scale)
    assert np.max(np.abs(Ot - Ob)) > 1e-3


def test_random_masks_with_empty_rows():
    rng = np.random.default_rng(3)
    B, H, D, nb, bs = 2, 2, 64, 6, 16
    q, k, v = _rand_qkv(B, H, nb * bs, D, seed=11)
    for _ in range(3):
        mask = (rng.random((nb, nb)) < 0.4).astype(np.uint8)
        mask[2, :] = 0  # a query block that reads nothing
        O, lse, l = oracle.attention(q, k, v, mask, bs, 0.125)
        Ob, lseb = _brute_dense(q, k, v, mask, bs, 0.125)
        assert np.max(np.abs(O - Ob)) <= 1e-12
        fin = np.isfinite(lseb)
        assert np.array_equal(fin, np.isfinite(lse))
        assert np.max(np.abs(lse[fin] - lseb[fin])) <= 1e-12
        # empty rows: O = 0, LSE = -inf, l = 0
        rows = (np.arange(B * H * nb * bs) % (nb * bs)) // bs == 2
        assert np.all(O[rows] == 0) and np.all(np.isneginf(lse[rows])) and np.all(l[rows] == 0)


@pytest.mark.parametrize("dense", [True, False])
def test_torch_sdpa_fp64(dense):
    B, H, D, nb, bs = 1, 3, 128, 5, 32
    L = nb * bs
    q, k, v = _rand_qkv(B, H, L, D, seed=5)
    mask = synth.dense_mask(nb) if dense else synth.window_mask(nb, 1, True)
    scale = float(np.float32(1 / math.sqrt(D)))
    O, _, _ = oracle.attention(q, k, v, mask, bs, scale)
    blk = torch.arange(L) // bs
    m = torch.from_numpy(mask.astype(bool))[blk[:, None], blk[None, :]]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(_f64(q)), torch.from_numpy(_f64(k)), torch.from_numpy(_f64(v)),
        attn_mask=m, scale=scale)
    assert np.max(np.abs(O - ref.numpy().reshape(-1, D))) <= 1e-12


def test_closed_forms():
    B, H, D, nb, bs = 1, 2, 64, 4, 16
    L = nb * bs
    mask = synth.window_mask(nb, 1, True)
    q, k, v = _rand_qkv(B, H, L, D, seed=9)
    vf = _f64(v)
    blk = np.arange(L) // bs
    allowed = mask.astype(bool)[blk[:, None], blk[None, :]]

    # q_i = 0: every allowed key gets weight 1/n -> mean of allowed v_j
    qz = q.copy()
    qz[0, 1, 20] = 0
    O, _, _ = oracle.attention(qz, k, v, mask, bs, 0.125)
    want = vf[0, 1][allowed[20]].mean(axis=0)
    assert np.max(np.abs(O[L + 20] - want)) <= 1e-14

    # all keys equal: the same mean for every row
    ke = np.broadcast_to(k[:, :, :1, :], k.shape).copy()
    O, _, _ = oracle.attention(q, ke, v, mask, bs, 0.125)
    for i in (0, 17, 40, 63):
        assert np.max(np.abs(O[i] - vf[0, 0][allowed[i]].mean(axis=0))) <= 1e-13

    # constant values: O = c
    c = synth.f32_to_bf16_bits(np.array([1.5], np.float32))[0]
    vc = np.full_like(v, c)
    O, _, _ = oracle.attention(q, k, vc, mask, bs, 0.125)
    assert np.max(np.abs(O - 1.5)) <= 1e-14

    # one dominant key: k_j = 64 * q_i (exact in bf16) -> O_i ~ v_j
    kd = k.copy()
    i, j = 37, 5  # row 37 is in block 2, which reads block 0 (global first frame)
    assert allowed[i, j]
    kd[0, 0, j] = synth.f32_to_bf16_bits(_f64(q[0, 0, i]).astype(np.float32) * 64)
    O, _, _ = oracle.attention(q, kd, v, mask, bs, 0.125)
    assert np.max(np.abs(O[i] - vf[0, 0, j])) <= 1e-6

    # permuting keys (with their values) inside a block leaves O unchanged
    perm = np.arange(L)
    rng = np.random.default_rng(1)
    for b0 in range(nb):
        perm[b0 * bs:(b0 + 1) * bs] = b0 * bs + rng.permutation(bs)
    O1, _, _ = oracle.attention(q, k, v, mask, bs, 0.125)
    O2, _, _ = oracle.attention(q, k[:, :, perm], v[:, :, perm], mask, bs, 0.125)
    assert np.max(np.abs(O1 - O2)) <= 1e-13


def test_two_key_softmax():
    # one token per block, two blocks, both read: S = (0, s) for query e_0
    D = 16
    one = synth.f32_to_bf16_bits(np.array([1.0], np.float32))[0]
    q = np.zeros((1, 1, 2, D), np.uint16)
    k = np.zeros_like(q)
    v = np.zeros_like(q)
    q[0, 0, 0, 0] = one
    k[0, 0, 1, 0] = one              # k_0 = 0, k_1 = e_0
    v[0, 0, 0, 1] = one              # v_0 = e_1, v_1 = 4 e_2
    v[0, 0, 1, 2] = synth.f32_to_bf16_bits(np.array([4.0], np.float32))[0]
    s = float(np.float32(math.log(3.0)))
    O, lse, _ = oracle.attention(q, k, v, np.ones((2, 2), np.uint8), 1, s)
    p1 = math.exp(s) / (1 + math.exp(s))
    assert abs(O[0, 1] - (1 - p1)) <= 1e-15 and abs(O[0, 2] - 4 * p1) <= 1e-15
    assert abs(lse[0] - math.log(1 + math.exp(s))) <= 1e-15


# ------------------------------------------------------------------------------------------------
# the bound


def test_cauchy_schwarz_invariant_and_shift_invariance():
    w = synth.WORKLOADS["tiny"]
    q, k, v = synth.make_qkv(w)
    mask, bs, scale = w.block_mask(), w.block, w.scale
    qn, kn = oracle.row_norms_f64(q), oracle.row_norms_f64(k)
    M = oracle.row_bounds_f64(qn, kn, mask, bs, scale)
    _, _, m32 = oracle.metadata_f32(q, k, mask, bs, scale)
    qf, kf = _f64(q), _f64(k)
    L = w.L
    blk = np.arange(L) // bs
    allowed = mask.astype(bool)[blk[:, None], blk[None, :]]
    for b in range(w.B):
        for h in range(w.H):
            S = scale * (qf[b, h] @ kf[b, h].T)
            S = np.where(allowed, S, -np.inf)
            assert np.all(S <= M[b, h][:, None] * (1 + 1e-12))
            assert np.all(S <= m32[b, h][:, None].astype(np.float64) * (1 + 2.0 ** -20))
    # softmax with the bound as its shift equals softmax with the max shift
    O_max, lse_max, _ = oracle.attention(q, k, v, mask, bs, scale)
    O_cs, lse_cs, l_cs = oracle.attention(q, k, v, mask, bs, scale, shift=M.reshape(-1))
    assert np.max(np.abs(O_cs - O_max)) <= 1e-12
    assert np.max(np.abs(lse_cs - lse_max)) <= 1e-12
    # l under the bound shift is exp(LSE - M) <= n_allowed
    assert np.max(np.abs(np.log(l_cs) - (lse_max - M.reshape(-1)))) <= 1e-12


def test_bound_shift_underflow_case_is_detectable():
    # a key scaled to ~1e4 makes the bound far above every logit of rows that read it
    w = synth.WORKLOADS["tiny"]
    q, k, v = synth.make_qkv(w)
    k = k.copy()
    big = _f64(k[0, 0, 3]) * 1.0e4
    k[0, 0, 3] = synth.f32_to_bf16_bits(big.astype(np.float32))
    mask, bs, scale = w.block_mask(), w.block, w.scale
    _, lse, _ = oracle.attention(q, k, v, mask, bs, scale)
    _, _, m32 = oracle.metadata_f32(q, k, mask, bs, scale)
    gap = m32.reshape(-1).astype(np.float64) - lse       # -ln(l under the bound shift)
    reads0 = (np.arange(w.B * w.H * w.L) // w.L == 0) & ((np.arange(w.B * w.H * w.L) % w.L) // bs <= 1)
    assert np.all(gap[reads0] > 100.0)                   # flagged: l < 2^-64
    assert np.all(gap[~reads0] < 30.0)                   # untouched rows keep l >> 2^-64


# ------------------------------------------------------------------------------------------------
# the fp32 norm recipe


def _bits(vals, D):
    x = np.zeros((1, D), np.float32)
    for i, val in vals:
        x[0, i] = val
    return synth.f32_to_bf16_bits(x)


@pytest.mark.parametrize("D", [16, 64, 128])
def test_norm_recipe_exact_cases(D):
    assert oracle.row_norms_f32(_bits([], D))[0] == 0.0
    ones = synth.f32_to_bf16_bits(np.ones((1, D), np.float32))
    assert oracle.row_norms_f32(ones)[0] == np.sqrt(np.float32(D))
    for x in (3.0, -0.75, 2.0 ** 60, 2.0 ** -70):
        assert oracle.row_norms_f32(_bits([(D // 2 + 1, x)], D))[0] == np.float32(abs(x))
    assert np.isinf(oracle.row_norms_f32(_bits([(0, 2.0 ** 64)], D))[0])


@pytest.mark.parametrize("D,w_exact", [(16, 2 ** 24 + 14), (64, 2 ** 24 + 60), (128, 2 ** 24 + 120)])
def test_norm_recipe_order(D, w_exact):
    # x_0 = 4096 and every other element 1: within chunk 0 each +1 is lost (ties to even at 2^24);
    # the other 15 chunks hold (D/16) each and meet chunk 0 through the 8-4-2-1 tree, which keeps them.
    # Hand count: D=16 -> 2^24 + 14, D=64 -> 2^24 + 60, D=128 -> 2^24 + 120 (a plain sequential sum
    # would stay at 2^24, the exact sum is 2^24 + D - 1).
    x = np.ones((1, D), np.float32)
    x[0, 0] = 4096.0
    n = oracle.row_norms_f32(synth.f32_to_bf16_bits(x))[0]
    assert n == np.sqrt(np.float32(w_exact))
    assert n != np.sqrt(np.float32(2 ** 24))


def test_norm_recipe_vs_fp64_and_bounds():
    w = synth.WORKLOADS["small"]
    q, k, _ = synth.make_qkv(w)
    mask, bs, scale = w.block_mask(), w.block, w.scale
    qn32, km32, rb32 = oracle.metadata_f32(q, k, mask, bs, scale)
    qn64, kn64 = oracle.row_norms_f64(q), oracle.row_norms_f64(k)
    assert np.max(np.abs(qn32 / qn64 - 1)) <= 2.0 ** -20
    km64 = kn64.reshape(w.B, w.H, w.nb, bs).max(axis=-1)
    assert np.max(np.abs(km32 / km64 - 1)) <= 2.0 ** -20
    M = oracle.row_bounds_f64(qn64, kn64, mask, bs, scale)
    assert np.max(np.abs(rb32 / M - 1)) <= 2.0 ** -20
    # kmax is a max of norms: exact, and equal to one of them
    kn32 = oracle.row_norms_f32(k).reshape(w.B, w.H, w.nb, bs)
    assert np.array_equal(km32, kn32.max(axis=-1))


# ------------------------------------------------------------------------------------------------
# workload sizes and the allowed-block sets


def test_workload_sizes_golden():
    g = json.load(open(GOLDEN))["workloads"]
    for name, w in synth.WORKLOADS.items():
        mask = w.block_mask()
        masks = mask if mask.ndim == 3 else mask[None]  # one mask per head, or one for all
        csrs = [oracle.allowed_csr(m) for m in masks]
        assert sum(len(c) for _, c in csrs) == g[name]["nnz"], name
        if mask.ndim == 3:
            assert len(masks) == w.H
        assert (w.B, w.H, w.D, w.frames, w.block) == (g[name]["B"], g[name]["H"], g[name]["D"],
                                                       g[name]["frames"], g[name]["block"])
        assert w.nq == g[name].get("q_frames", g[name]["frames"])
        assert synth.useful_flop(w) == g[name]["useful_flop"]
        # ascending within each query block
        for row_ptr, col_idx in csrs:
            for qb in range(w.nb):
                s = col_idx[row_ptr[qb]:row_ptr[qb + 1]]
                assert np.all(np.diff(s) > 0)


def _golden_allowed(g, w, h):
    """The hand-typed allowed key frames of each query frame under head h's mask."""
    if "allowed" in g:
        return g["allowed"]
    return g["allowed_by_rule"][str(h % 4)]


def test_allowed_csr_per_query_block_golden():
    # The allowed-block sets of every workload, typed by hand from the mask rules
    # ("HeyGen Avatar IV on Trillium TPU" deep-dive, section 把 block 縮到 16: the mask
    # decides per frame block which key frames a query frame reads).  The first-frame-
    # global masks are not symmetric, so a transposed reading of the mask, a row_ptr
    # shifted by one block or a dropped block fails here.
    g = json.load(open(GOLDEN))["workloads"]
    for name, w in synth.WORKLOADS.items():
        mask = w.block_mask()
        masks = mask if mask.ndim == 3 else mask[None]
        for h, m in enumerate(masks):
            want = _golden_allowed(g[name], w, h)
            assert len(want) == w.nq, name
            row_ptr, col_idx = oracle.allowed_csr(m)
            assert list(row_ptr) == list(np.cumsum([0] + [len(a) for a in want])), (name, h)
            for qb, a in enumerate(want):
                assert list(col_idx[row_ptr[qb]:row_ptr[qb + 1]]) == a, (name, h, qb)


def test_allowed_csr_rectangular_by_hand():
    # 3 query blocks reading 4 key blocks; the CSR written out by hand.
    m = np.array([[1, 0, 0, 1],
                  [0, 0, 0, 0],
                  [0, 1, 1, 1]], np.uint8)
    row_ptr, col_idx = oracle.allowed_csr(m)
    assert list(row_ptr) == [0, 2, 2, 5]
    assert list(col_idx) == [0, 3, 1, 2, 3]


def test_generator_matches_splitmix64_definition():
    # published SplitMix64 outputs for state 1234567
    assert [synth.splitmix64_at(1234567, i) for i in range(3)] == [
        6457827717110365317, 3203168211198807973, 9817491932198370423]
    # fp32 -> bf16 round-to-nearest-even on ties
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -7], np.float32)
    assert list(synth.bf16_bits_to_f64(synth.f32_to_bf16_bits(x))) == [1.0, 1 + 2 ** -6, 1 + 2 ** -7]
    q = _f64(synth.tensor_bf16(0, synth.TAG_Q, 1, 2, 4096, 64))
    assert abs(q.mean()) < 0.01 and abs(q.std() - 1) < 0.01


# ------------------------------------------------------------------------------------------------
# one block mask per head


def _per_head_masks(nb, rng):
    m0 = synth.window_mask(nb, 1)
    m1 = (rng.random((nb, nb)) < 0.5).astype(np.uint8)
    m1[1, :] = 0  # a query block that reads nothing under this head's mask
    m2 = np.ones((nb, nb), np.uint8)
    return np.stack([m0, m1, m2])


def test_per_head_masks_brute_force():
    # Each head under its own mask: the dense route builds head h's element mask from
    # mask[h] (numpy, independent of the oracle's slicing); all rows and sampled rows.
    rng = np.random.default_rng(5)
    B, H, D, nb, bs = 2, 3, 64, 5, 16
    L = nb * bs
    masks = _per_head_masks(nb, rng)
    q, k, v = _rand_qkv(B, H, L, D, seed=13)
    scale = 0.125
    O, lse, _ = oracle.attention(q, k, v, masks, bs, scale)
    Ob = np.zeros((B, H, L, D))
    lseb = np.zeros((B, H, L))
    for h in range(H):
        o_h, l_h = _brute_dense(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], masks[h], bs, scale)
        Ob[:, h] = o_h.reshape(B, L, D)
        lseb[:, h] = l_h.reshape(B, L)
    Ob, lseb = Ob.reshape(-1, D), lseb.reshape(-1)
    assert np.max(np.abs(O - Ob)) <= 1e-12
    fin = np.isfinite(lseb)
    assert np.array_equal(fin, np.isfinite(lse)) and np.max(np.abs(lse[fin] - lseb[fin])) <= 1e-12
    # head 1's empty query block: O = 0 there, other heads' rows of that block are not empty
    rows = np.arange(B * H * L)
    empty = ((rows // L) % H == 1) & ((rows % L) // bs == 1)
    assert np.all(O[empty] == 0) and np.all(np.isneginf(lse[empty]))
    assert np.all(np.isfinite(lse[~empty]))
    # the sampled-row route gives the same rows
    pick = rng.choice(B * H * L, 37, replace=False)
    Os, lses, _ = oracle.attention(q, k, v, masks, bs, scale, rows=pick)
    assert np.array_equal(Os, O[pick]) and np.array_equal(lses, lse[pick])


def test_per_head_masks_equal_masks_match_the_shared_mask():
    w = synth.WORKLOADS["tiny"]
    q, k, v = synth.make_qkv(w)
    m = w.block_mask()
    O1, lse1, l1 = oracle.attention(q, k, v, m, w.block, w.scale)
    O2, lse2, l2 = oracle.attention(q, k, v, np.stack([m] * w.H), w.block, w.scale)
    assert np.array_equal(O1, O2) and np.array_equal(lse1, lse2) and np.array_equal(l1, l2)
    _, _, rb1 = oracle.metadata_f32(q, k, m, w.block, w.scale)
    _, _, rb2 = oracle.metadata_f32(q, k, np.stack([m] * w.H), w.block, w.scale)
    assert np.array_equal(rb1.view(np.uint32), rb2.view(np.uint32))


def test_per_head_row_bounds_by_hand():
    # M_i = scale * |q_i| * max over head h's allowed key blocks of |k_j|, computed here with
    # numpy from the definition; every allowed logit of the head lies below it.
    rng = np.random.default_rng(9)
    B, H, D, nb, bs = 1, 3, 64, 5, 16
    L = nb * bs
    masks = _per_head_masks(nb, rng)
    q, k, _ = _rand_qkv(B, H, L, D, seed=17)
    qf, kf = _f64(q), _f64(k)
    qn, kn = np.sqrt((qf ** 2).sum(-1)), np.sqrt((kf ** 2).sum(-1))
    M = oracle.row_bounds_f64(qn, kn, masks, bs, 0.125)
    for h in range(H):
        kblk = kn[0, h].reshape(nb, bs).max(axis=1)
        for i in range(L):
            allowed = np.nonzero(masks[h, i // bs])[0]
            want = 0.125 * qn[0, h, i] * (kblk[allowed].max() if len(allowed) else 0.0)
            assert M[0, h, i] == pytest.approx(want, rel=1e-15, abs=0.0)
            if len(allowed):
                keys = np.concatenate([np.arange(kb * bs, kb * bs + bs) for kb in allowed])
                assert np.all(0.125 * (kf[0, h, keys] @ qf[0, h, i]) <= M[0, h, i] * (1 + 1e-12))
