"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (bf16 output of an fp32-accumulated, bf16-operand attention):
  O:          max |O_gpu - O_oracle| <= 2e-2 and mean <= 2e-3
  LSE:        |LSE_gpu - LSE_oracle| <= 5e-3 + D * 2^-24 * m_i per row (m_i the row bound: the
              fp32 dot-product error of the logits, which matters only for huge logits)
  metadata:   qnorm, kmax, rowbound bit-identical to the oracle's fp32 recipe
Small shapes are compared on every row; the 720p / 1080p / stress shapes on
sampled rows that the oracle computes one by one (first, last, tile-edge and
random rows of each frame), with the metadata checked on every row.
"""
import numpy as np
import pytest

import oracle
from block_sparse_video_row_b300 import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 5e-3


@pytest.fixture(scope="module")
def ba():
    from block_sparse_video_row_b300 import _build, bsattn
    _build.build()
    bsattn.load()
    return bsattn


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()


def _host_bf16(t):
    return synth.bf16_bits_to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16))


def run_gpu(ba, q, k, v, mask, bs, scale, flags=0, want_meta=True, lay=None):
    B, H, L, D = q.shape
    L_kv = k.shape[2]
    nb = L_kv // bs  # key blocks (kmax)
    own = lay is None
    if own:
        lay = ba.bsattn_create_layout(B, H, L, D, bs, mask, L_kv=L_kv)
    dq, dk, dv = _dev(q), _dev(k), _dev(v)
    o = torch.full_like(dq, float("nan"))
    qn = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    km = torch.empty((B, H, nb), dtype=torch.float32, device="cuda")
    rb = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    ba.bsattn_row_bounds(lay, dq, dk, scale, qn, km, rb)
    ba.bsattn_forward(lay, dq, dk, dv, o, scale, rb, lse, flags)
    rows, units, status = ba.bsattn_query_stats(lay)
    bound_units, online_units = ba.bsattn_query_eligibility(lay)
    torch.cuda.synchronize()
    out = dict(o=_host_bf16(o).reshape(-1, D), lse=lse.cpu().numpy().reshape(-1), fb_rows=rows, fb_units=units,
               status=status, o_raw=o, bound_units=bound_units, online_units=online_units)
    if want_meta:
        out.update(qnorm=qn.cpu().numpy(), kmax=km.cpu().numpy(), rowbound=rb.cpu().numpy())
    if own:
        lay.destroy()
    return out


def sample_rows(B, H, L, bs, heads=None, per_frame_random=2, seed=0):
    rng = np.random.default_rng(seed)
    nb = L // bs
    rows = []
    for bh in (range(B * H) if heads is None else heads):
        for f in range(nb):
            base = bh * L + f * bs
            cand = {0, bs - 1, min(127, bs - 1), min(128, bs - 1), (bs - 1) // 128 * 128}
            cand |= set(rng.integers(0, bs, per_frame_random).tolist())
            rows += [base + c for c in sorted(cand)]
    return np.array(rows, dtype=np.int64)


def check_o(got, want, what=""):
    err = np.abs(got - want)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert err.max() <= O_MAX, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"{what}: mean abs err {err.mean():.3e}"


def check_meta(res, q, k, mask, bs, scale):
    qn, km, rb = oracle.metadata_f32(q, k, mask, bs, scale)
    assert np.array_equal(res["qnorm"].view(np.uint32), qn.view(np.uint32))
    assert np.array_equal(res["kmax"].view(np.uint32), km.view(np.uint32))
    assert np.array_equal(res["rowbound"].view(np.uint32), rb.view(np.uint32))
    return rb


def lse_tolerance(D, rowbound):
    """LSE_MAX plus the fp32 error of the logits themselves: an fp32 dot product of length D is
    exact to D * 2^-24 * sum_d |q_d k_d| <= D * 2^-24 * |q| |k| (Cauchy-Schwarz), i.e. to
    D * 2^-24 * m_i nats after the scale, m_i being the row's bound.  The second term is ~1e-4
    for N(0,1) rows and matters only for rows with logits of thousands."""
    return LSE_MAX + D * 2.0 ** -24 * np.abs(rowbound)


def full_case(ba, q, k, v, mask, bs, scale, flags=0, what=""):
    res = run_gpu(ba, q, k, v, mask, bs, scale, flags)
    rb = check_meta(res, q, k, mask, bs, scale).reshape(-1).astype(np.float64)
    O, lse, _ = oracle.attention(q, k, v, mask, bs, scale)
    check_o(res["o"], O, what)
    fin = np.isfinite(lse)
    assert np.array_equal(np.isfinite(res["lse"]), fin)
    if fin.any():
        err = np.abs(res["lse"][fin] - lse[fin])
        assert np.all(err <= lse_tolerance(q.shape[-1], rb[fin])), f"{what}: LSE err {err.max():.3e}"
    assert res["status"] == 0
    return res


# ------------------------------------------------------------------------------------------------


@pytest.mark.parametrize("name", ["tiny", "small", "stream_small", "small_heads", "stream_heads"])
def test_workload_full(ba, name):
    w = synth.WORKLOADS[name]
    q, k, v = synth.make_qkv(w)
    res = full_case(ba, q, k, v, w.block_mask(), w.block, w.scale, what=name)
    assert res["fb_rows"] == 0 and res["fb_units"] == 0


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B,H,frames,bs,mask_kind", [
    (1, 1, 1, 16, "dense"),         # one frame of 16 tokens: 16-row query tile, 16-key tile
    (2, 3, 3, 48, "window"),        # partial query tile, several batches
    (1, 2, 4, 128, "window_first"),  # exactly one query tile per frame, key tile 128
    (1, 2, 3, 256, "dense"),        # two full query tiles per frame (one unit of 2 tiles)
    (1, 2, 3, 272, "window"),       # 3 query tiles (unit of 2 + unit of 1, 16-row tail), key tile 272/17=16
    (1, 2, 5, 208, "empty_row"),    # a frame that reads nothing: O = 0, LSE = -inf
])
def test_edge_shapes(ba, D, B, H, frames, bs, mask_kind):
    L = frames * bs
    if mask_kind == "dense":
        mask = synth.dense_mask(frames)
    elif mask_kind == "window":
        mask = synth.window_mask(frames, 1)
    elif mask_kind == "window_first":
        mask = synth.window_mask(frames, 1, True)
    else:
        mask = synth.window_mask(frames, 1, True)
        mask[2, :] = 0
    q = synth.tensor_bf16(3, synth.TAG_Q, B, H, L, D)
    k = synth.tensor_bf16(3, synth.TAG_K, B, H, L, D)
    v = synth.tensor_bf16(3, synth.TAG_V, B, H, L, D)
    scale = float(np.float32(1 / np.sqrt(D)))
    res = full_case(ba, q, k, v, mask, bs, scale, what=f"{B}x{H}x{frames}x{bs} D{D} {mask_kind}")
    if mask_kind == "empty_row":
        rows = (np.arange(B * H * L) % L) // bs == 2
        assert np.all(res["o"][rows] == 0) and np.all(np.isneginf(res["lse"][rows]))


# online max everywhere; bound without the rerun; bound for every row (no eligibility switch),
# with and without the rerun
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B,H,nq,nkv,bs", [
    (2, 3, 1, 3, 48),     # one query frame reading three key frames; partial query tile
    (1, 2, 2, 2, 16),     # L_kv == L through the rectangular entry point
    (1, 2, 3, 9, 272),    # three query tiles per frame, 16-row tail, irregular mask
])
def test_streamed_edge_shapes(ba, D, B, H, nq, nkv, bs):
    rng = np.random.default_rng(nq * 100 + nkv)
    mask = (rng.random((nq, nkv)) < 0.6).astype(np.uint8)
    mask[:, 0] = 1                       # every query frame reads at least the first key frame
    mask[np.arange(nq), nkv - nq + np.arange(nq)] = 1  # and its own frame
    q = synth.tensor_bf16(4, synth.TAG_Q, B, H, nq * bs, D)
    k = synth.tensor_bf16(4, synth.TAG_K, B, H, nkv * bs, D)
    v = synth.tensor_bf16(4, synth.TAG_V, B, H, nkv * bs, D)
    scale = float(np.float32(1 / np.sqrt(D)))
    full_case(ba, q, k, v, mask, bs, scale, what=f"stream {B}x{H} {nq}/{nkv}x{bs} D{D}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B,H,nq,nkv,bs", [
    (2, 3, 3, 3, 48),     # self-attention, several batches (head h of every batch reads mask h)
    (1, 4, 2, 5, 272),    # streamed chunk, three query tiles per frame, 16-row tail
])
def test_per_head_edge_shapes(ba, D, B, H, nq, nkv, bs):
    # One random mask per head, one head with a query frame that reads nothing: every
    # row against the oracle, metadata bit-exact.
    rng = np.random.default_rng(H * 10 + nkv)
    masks = (rng.random((H, nq, nkv)) < 0.5).astype(np.uint8)
    masks[:, np.arange(nq), nkv - nq + np.arange(nq)] = 1  # every frame reads its own frame ...
    masks[1, 0, :] = 0                                     # ... except frame 0 under head 1's mask
    q = synth.tensor_bf16(6, synth.TAG_Q, B, H, nq * bs, D)
    k = synth.tensor_bf16(6, synth.TAG_K, B, H, nkv * bs, D)
    v = synth.tensor_bf16(6, synth.TAG_V, B, H, nkv * bs, D)
    scale = float(np.float32(1 / np.sqrt(D)))
    res = full_case(ba, q, k, v, masks, bs, scale, what=f"per-head {B}x{H} {nq}/{nkv}x{bs} D{D}")
    L = nq * bs
    rows = np.arange(B * H * L)
    empty = ((rows // L) % H == 1) & ((rows % L) // bs == 0)
    assert np.all(res["o"][empty] == 0) and np.all(np.isneginf(res["lse"][empty]))


@pytest.mark.parametrize("seed", range(8))
def test_random_shapes(ba, seed):
    # Random small problems: head dim, batch, heads, frame size (a multiple of 16), query
    # and key frame counts, and a random mask (shared or one per head, streamed or not);
    # every row against the oracle, metadata bit-exact.
    rng = np.random.default_rng(1000 + seed)
    D = int(rng.choice([64, 128]))
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
    bs = 16 * int(rng.integers(1, 20))
    nkv = int(rng.integers(1, 7))
    nq = nkv if rng.random() < 0.5 else int(rng.integers(1, nkv + 1))
    shape = (H, nq, nkv) if rng.random() < 0.5 else (nq, nkv)
    mask = (rng.random(shape) < 0.6).astype(np.uint8)
    q = synth.tensor_bf16(2000 + seed, synth.TAG_Q, B, H, nq * bs, D)
    k = synth.tensor_bf16(2000 + seed, synth.TAG_K, B, H, nkv * bs, D)
    v = synth.tensor_bf16(2000 + seed, synth.TAG_V, B, H, nkv * bs, D)
    scale = float(np.float32(1 / np.sqrt(D)))
    full_case(ba, q, k, v, mask, bs, scale, what=f"random {seed}: D{D} {B}x{H} {nq}/{nkv}x{bs} mask{shape}")


@pytest.mark.parametrize("seed", range(6))
def test_random_loose_keys_route_and_guard(ba, seed):
    # Random small problems as above, with a few keys made 10^0.5 .. 10^4 times longer, so
    # that some units fail the eligibility check (routed online), some bound rows underflow
    # (flagged and rerun) and the rest stay on the bound path.  Every row against the
    # oracle; the online-unit count exactly as the oracle's fp32 bounds predict (any row of
    # the unit above 64 nats); the flagged rows inside the guard's must/may band.
    rng = np.random.default_rng(3000 + seed)
    D = int(rng.choice([64, 128]))
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
    bs = 16 * int(rng.integers(1, 26))
    nkv = int(rng.integers(1, 6))
    nq = nkv if rng.random() < 0.5 else int(rng.integers(1, nkv + 1))
    shape = (H, nq, nkv) if rng.random() < 0.5 else (nq, nkv)
    mask = (rng.random(shape) < 0.7).astype(np.uint8)
    q = synth.tensor_bf16(4000 + seed, synth.TAG_Q, B, H, nq * bs, D)
    k = synth.tensor_bf16(4000 + seed, synth.TAG_K, B, H, nkv * bs, D).copy()
    v = synth.tensor_bf16(4000 + seed, synth.TAG_V, B, H, nkv * bs, D)
    for _ in range(int(rng.integers(1, 4))):
        b, h, j = int(rng.integers(0, B)), int(rng.integers(0, H)), int(rng.integers(0, nkv * bs))
        f = 10.0 ** rng.uniform(0.5, 4.0)
        k[b, h, j] = synth.f32_to_bf16_bits((synth.bf16_bits_to_f64(k[b, h, j]) * f).astype(np.float32))
    scale = float(np.float32(1 / np.sqrt(D)))
    what = f"loose {seed}: D{D} {B}x{H} {nq}/{nkv}x{bs} mask{shape}"
    res = full_case(ba, q, k, v, mask, bs, scale, what=what)
    unit_of_row, n_units = _row_units(ba, q, k, mask, bs)
    must, may, _, online = _predicted_flags(q, k, v, mask, bs, scale, eligible=64.0, unit_of_row=unit_of_row)
    want_online = len(np.unique(unit_of_row[online]))
    assert res["online_units"] == want_online, what
    assert res["bound_units"] == n_units - want_online, what
    assert must <= res["fb_rows"] <= may, what


@pytest.mark.parametrize("flags", [1, 2, 4, 6])
def test_variants_small(ba, flags):
    w = synth.WORKLOADS["small"]
    q, k, v = synth.make_qkv(w)
    full_case(ba, q, k, v, w.block_mask(), w.block, w.scale, flags=flags, what=f"small flags={flags}")


@pytest.mark.parametrize("flags", [1, 4])
def test_variants_per_head(ba, flags):
    # the online-max kernel and the bound-only path on one mask per head
    w = synth.WORKLOADS["stream_heads"]
    q, k, v = synth.make_qkv(w)
    full_case(ba, q, k, v, w.block_mask(), w.block, w.scale, flags=flags, what=f"stream_heads flags={flags}")


def _scaled_key(w, factor):
    q, k, v = synth.make_qkv(w)
    k = k.copy()
    k[0, 0, 3] = synth.f32_to_bf16_bits((synth.bf16_bits_to_f64(k[0, 0, 3]) * factor).astype(np.float32))
    return q, k, v


def _row_units(ba, q, k, mask, bs):
    """(unit index of every query row, number of units) from the layout's plan: 1 or 2 query tiles
    of one frame, or a packed tile of the tails of several frames (b*H+h, first frame, segment, -n)."""
    B, H, L, D = q.shape
    lay = ba.bsattn_create_layout(B, H, L, D, bs, mask, ba.BSATTN_PLAN_ONLY, L_kv=k.shape[2])
    _, _, units, _, _ = ba.bsattn_layout_export(lay, with_tiles=True)
    lay.destroy()
    r0 = (-(-bs // 128) - 1) * 128
    out = np.full(B * H * L, -1, np.int64)
    for i, (bh, qb, z, w) in enumerate(units):
        if w > 0:
            a = bh * L + qb * bs + z * 128
            out[a:min(bh * L + (qb + 1) * bs, a + w * 128)] = i
        else:
            for g in range(-w):
                a = bh * L + (qb + g) * bs + r0
                out[a:a + bs - r0] = i
    assert np.all(out >= 0)
    return out, len(units)


def _predicted_flags(q, k, v, mask, bs, scale, eligible=np.inf, unit_of_row=None):
    """(must, may) counts of guard-flagged rows: a row is a bound row when every row of its work
    unit has a bound <= eligible (units from unit_of_row; default: query tiles 2c and 2c + 1 of a
    frame, i.e. frame rows 256c .. 256c + 255); a bound row must be flagged when ln l < ln 2^-65
    and may be when ln l < ln 2^-63, l being the bound-shifted denominator."""
    B, H, L, D = q.shape
    _, lse, _ = oracle.attention(q, k, v, mask, bs, scale)
    _, _, m32 = oracle.metadata_f32(q, k, mask, bs, scale)
    m = m32.reshape(-1).astype(np.float64)
    log_l = lse - m
    r = np.arange(B * H * L)
    pos = r % L
    units_per_block = (bs + 255) // 256
    group = (((r // L) * (L // bs) + pos // bs) * units_per_block + (pos % bs) // 256
             if unit_of_row is None else unit_of_row)
    online = np.zeros(B * H * L, dtype=bool)
    for g in np.unique(group):
        sel = group == g
        online[sel] = np.any(m[sel] > eligible)
    fin = np.isfinite(log_l)
    must = int(np.sum(~online & fin & (log_l < np.log(2.0 ** -65))))
    may = int(np.sum(~online & fin & (log_l < np.log(2.0 ** -63))))
    return must, may, log_l, online


def test_guard_forced_and_zero_queries(ba):
    # one key 1e4 times longer: rows that read it have a bound far above their best logit
    w = synth.WORKLOADS["tiny"]
    q, k, v = _scaled_key(w, 1e4)
    q = q.copy()
    q[0, 1, 100:110] = 0  # zero query rows: P = 1 for every allowed key, never flagged
    mask, bs, scale = w.block_mask(), w.block, w.scale
    res = full_case(ba, q, k, v, mask, bs, scale, flags=4, what="guard")  # bound for every row
    # rows of head 0 in frames 0 and 1 read the huge key: the bound is far too loose there
    _, lse, _ = oracle.attention(q, k, v, mask, bs, scale)
    _, _, m32 = oracle.metadata_f32(q, k, mask, bs, scale)
    log_l = lse - m32.reshape(-1).astype(np.float64)       # ln of the bound-shifted denominator
    must = int(np.sum(log_l < np.log(2.0 ** -65)))
    may = int(np.sum(log_l < np.log(2.0 ** -63)))
    assert must <= res["fb_rows"] <= may and must > 0
    assert res["fb_units"] >= 1
    # without the rerun those rows are not trusted, the others still match
    res2 = run_gpu(ba, q, k, v, mask, bs, scale, flags=6, want_meta=False)
    ok_rows = log_l > np.log(2.0 ** -63)
    O, _, _ = oracle.attention(q, k, v, mask, bs, scale)
    check_o(res2["o"][ok_rows], O[ok_rows], "guard, unflagged rows")


def test_eligibility_check_sends_loose_units_online(ba):
    # Default mode on the same inputs: the work units holding a row whose bound is above the
    # eligibility limit go to the online-max launch, whole, before any bound softmax runs, so the
    # guard flags nothing; the check's counts are exactly the units the oracle's bounds predict.
    w = synth.WORKLOADS["tiny"]
    q, k, v = _scaled_key(w, 1e4)
    mask, bs, scale = w.block_mask(), w.block, w.scale
    must, may, _, online = _predicted_flags(q, k, v, mask, bs, scale, eligible=64.0)
    assert online.any() and must == may == 0
    res = full_case(ba, q, k, v, mask, bs, scale, flags=0, what="eligibility check")
    assert res["fb_rows"] == 0 and res["fb_units"] == 0
    n_units = w.B * w.H * w.nb * ((bs + 255) // 256)
    r = np.arange(w.B * w.H * w.L)
    unit_of_row = ((r // w.L) * w.nb + (r % w.L) // bs) * ((bs + 255) // 256) + (r % bs) // 256
    want_online = len(np.unique(unit_of_row[online]))
    assert res["online_units"] == want_online and res["bound_units"] == n_units - want_online


def test_eligibility_check_on_a_streamed_chunk_with_per_head_masks(ba):
    # One key of head 1 (rule 1: window +-2) in frame 5 made 1e4 times longer: every query
    # frame of the chunk (5, 6, 7) reads frame 5 under head 1's mask, so all of head 1's units
    # fail the check and no other unit does; the whole chunk still matches the oracle.
    w = synth.WORKLOADS["stream_heads"]
    q, k, v = synth.make_qkv(w)
    k = k.copy()
    k[0, 1, 5 * w.block + 100] = synth.f32_to_bf16_bits(
        (synth.bf16_bits_to_f64(k[0, 1, 5 * w.block + 100]) * 1e4).astype(np.float32))
    mask = w.block_mask()
    res = full_case(ba, q, k, v, mask, w.block, w.scale, what="streamed per-head eligibility")
    units_per_frame = (w.block + 255) // 256
    assert res["online_units"] == w.nq * units_per_frame
    assert res["bound_units"] == (w.B * w.H - 1) * w.nq * units_per_frame
    assert res["fb_rows"] == 0


def test_guard_fires_on_eligible_rows(ba):
    # A key 5x longer puts the bounds of the rows that read it between 22 and 64 nats (57 at most):
    # they stay on the bound path (eligible), and those whose best logit lies > 44 nats below the
    # bound are flagged and rerun; the predicted count follows the work units the eligibility check routes.
    w = synth.WORKLOADS["tiny"]
    q, k, v = _scaled_key(w, 5.0)
    mask, bs, scale = w.block_mask(), w.block, w.scale
    must, may, log_l, online = _predicted_flags(q, k, v, mask, bs, scale, eligible=64.0)
    assert must > 0 and not online.any()
    res = full_case(ba, q, k, v, mask, bs, scale, flags=0, what="guard on eligible rows")
    assert must <= res["fb_rows"] <= may and res["fb_units"] >= 1


def test_streamed_chunk_equals_last_rows_of_the_full_window(ba):
    # the chunk's queries are the last query rows of the full-window problem and its mask the
    # last mask rows, and every row's key tiles are the same: the GPU rows must be identical
    w = synth.WORKLOADS["stream_small"]
    wf = synth.Workload("full", w.B, w.H, w.D, w.frames, w.block, w.mask, w.keys, w.seed)
    q, k, v = synth.make_qkv(w)
    qf, _, _ = synth.make_qkv(wf)
    chunk = run_gpu(ba, q, k, v, w.block_mask(), w.block, w.scale)
    full = run_gpu(ba, qf, k, v, wf.block_mask(), w.block, w.scale)
    tail = full["o_raw"][:, :, w.L_kv - w.L:]
    assert torch.equal(chunk["o_raw"].view(torch.int16), tail.contiguous().view(torch.int16))
    assert np.array_equal(chunk["kmax"].view(np.uint32), full["kmax"].view(np.uint32))
    assert np.array_equal(chunk["rowbound"].view(np.uint32),
                          full["rowbound"][:, :, w.L_kv - w.L:].view(np.uint32))


def test_per_head_plan_with_equal_masks_equals_the_shared_plan(ba):
    # One mask per head, every head given the shared mask: the same key tiles for every
    # row, so the per-head plan reproduces the shared plan's output bit for bit.
    w = synth.WORKLOADS["small"]
    q, k, v = synth.make_qkv(w)
    mask = w.block_mask()
    shared = run_gpu(ba, q, k, v, mask, w.block, w.scale, want_meta=True)
    per_head = run_gpu(ba, q, k, v, np.stack([mask] * w.H), w.block, w.scale, want_meta=True)
    assert torch.equal(shared["o_raw"].view(torch.int16), per_head["o_raw"].view(torch.int16))
    assert np.array_equal(shared["rowbound"].view(np.uint32), per_head["rowbound"].view(np.uint32))
    assert per_head["status"] == 0


def test_deterministic(ba):
    w = synth.WORKLOADS["small"]
    q, k, v = synth.make_qkv(w)
    a = run_gpu(ba, q, k, v, w.block_mask(), w.block, w.scale, want_meta=False)
    b = run_gpu(ba, q, k, v, w.block_mask(), w.block, w.scale, want_meta=False)
    assert torch.equal(a["o_raw"].view(torch.int16), b["o_raw"].view(torch.int16))


@pytest.mark.parametrize("name,heads", [("720p", [0, 7, 23]), ("stress", [0, 11]), ("1080p", [5]),
                                        ("stream", [0, 13]), ("720p_heads", [0, 1, 2, 3, 22])])
def test_workload_sampled(ba, name, heads):
    w = synth.WORKLOADS[name]
    q, k, v = synth.make_qkv(w)
    mask = w.block_mask()
    res = run_gpu(ba, q, k, v, mask, w.block, w.scale)
    rb = check_meta(res, q, k, mask, w.block, w.scale).reshape(-1).astype(np.float64)
    rows = sample_rows(w.B, w.H, w.L, w.block, heads=heads)
    O, lse, _ = oracle.attention(q, k, v, mask, w.block, w.scale, rows=rows)
    check_o(res["o"][rows], O, name)
    tol = lse_tolerance(w.D, rb[rows])
    assert np.all(np.abs(res["lse"][rows] - lse) <= tol)
    assert np.all(np.isfinite(res["o"]))
    assert res["fb_rows"] == 0  # stress: loose units go to the online launch before any bound softmax
    assert res["status"] == 0
    if name != "stress":
        assert res["online_units"] == 0  # N(0,1) data: every unit is eligible
    else:
        assert res["online_units"] > 0
    if name == "stress":
        # the bound path for every row: the guard flags the loose rows and the rerun fixes them
        res2 = run_gpu(ba, q, k, v, mask, w.block, w.scale, flags=4, want_meta=False)
        check_o(res2["o"][rows], O, name + " bound only")
        assert np.all(np.abs(res2["lse"][rows] - lse) <= tol)
        assert res2["fb_rows"] > 0 and res2["fb_units"] > 0 and res2["status"] == 0


def test_dense_1080p_sampled(ba):
    w = synth.WORKLOADS["1080p_dense"]
    q, k, v = synth.make_qkv(w)
    mask = w.block_mask()
    res = run_gpu(ba, q, k, v, mask, w.block, w.scale, want_meta=False)
    rows = sample_rows(w.B, w.H, w.L, w.block, heads=[3], per_frame_random=0)[::3]
    O, _, _ = oracle.attention(q, k, v, mask, w.block, w.scale, rows=rows)
    check_o(res["o"][rows], O, "1080p dense")


def _pinned(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).pin_memory()


@pytest.mark.parametrize("name,pairs,flags", [("small", 3, 0), ("small", 0, 1), ("tiny", 1, 4),
                                              ("stream_small", 3, 0), ("small_heads", 3, 0),
                                              ("stream_heads", 0, 0)])
def test_host_path_equals_device_path(ba, name, pairs, flags):
    # bsattn_forward_host (pinned host tensors, chunked copies and kernels on three streams)
    # against bsattn_forward on device copies: the same kernels per row, so identical bits.
    # small with 3 pairs per chunk runs chunks of 3, 3 and 2 heads (two chunk layouts).
    w = synth.WORKLOADS[name]
    q, k, v = synth.make_qkv(w)
    if name == "tiny":  # a loose key, so the guard flags rows (bound softmax for every row)
        q, k, v = _scaled_key(w, 1e4)
    mask = w.block_mask()
    lay = ba.bsattn_create_layout(w.B, w.H, w.L, w.D, w.block, mask, L_kv=w.L_kv)
    dev = run_gpu(ba, q, k, v, mask, w.block, w.scale, flags, want_meta=False, lay=lay)
    hq, hk, hv = _pinned(q), _pinned(k), _pinned(v)
    ho = torch.full_like(hq, float("nan")).pin_memory()
    hl = torch.full((w.B, w.H, w.L), float("nan"), dtype=torch.float32).pin_memory()
    for _ in range(2):  # the second call reuses the staging and streams
        ba.bsattn_forward_host(lay, hq, hk, hv, ho, w.scale, hl, flags, pairs)
        torch.cuda.synchronize()
        rows, units, status = ba.bsattn_query_stats(lay)
        assert torch.equal(ho.view(torch.int16), dev["o_raw"].cpu().view(torch.int16))
        assert np.array_equal(hl.numpy().reshape(-1).view(np.uint32), dev["lse"].view(np.uint32))
        assert (rows, units, status) == (dev["fb_rows"], dev["fb_units"], 0)
    if name == "tiny":
        assert rows > 0
    lay.destroy()


@pytest.mark.parametrize("pairs", [1, 2])
def test_host_path_with_packed_tails(ba, pairs):
    # Frames with 16-row tails and one mask per head through the host-tensor path: each
    # chunk's layout packs its heads' tails as the whole layout does, so the output is the
    # device path's bit for bit, and the eligibility counts of the chunks add up to its counts.
    q, k, v, mask, bs, scale = _tails_case(128, True, loose=True)
    B, H, L, D = q.shape
    lay = ba.bsattn_create_layout(B, H, L, D, bs, mask)
    assert lay.info.tail_units > 0
    dev = run_gpu(ba, q, k, v, mask, bs, scale, 0, want_meta=False, lay=lay)
    hq, hk, hv = _pinned(q), _pinned(k), _pinned(v)
    ho = torch.full_like(hq, float("nan")).pin_memory()
    ba.bsattn_forward_host(lay, hq, hk, hv, ho, scale, None, 0, pairs)
    torch.cuda.synchronize()
    assert torch.equal(ho.view(torch.int16), dev["o_raw"].cpu().view(torch.int16))
    assert ba.bsattn_query_eligibility(lay) == (dev["bound_units"], dev["online_units"])
    assert dev["online_units"] > 0
    lay.destroy()


def test_bounded_wait_runs_out_and_the_context_stays_usable(ba, monkeypatch):
    # BSATTN_DEBUG_STALL withholds the first unit's query tiles in every CTA: the MMA
    # issuers' waits run out after the layout's 200 ms limit, the CTA aborts (copies in
    # flight drained, TMEM freed) and the kernel returns; the status word says so.
    w = synth.WORKLOADS["small"]
    q, k, v = synth.make_qkv(w)
    mask = w.block_mask()
    monkeypatch.setenv("BSATTN_TIMEOUT_MS", "200")
    lay = ba.bsattn_create_layout(w.B, w.H, w.L, w.D, w.block, mask)  # reads the limit
    monkeypatch.delenv("BSATTN_TIMEOUT_MS")
    res = run_gpu(ba, q, k, v, mask, w.block, w.scale, flags=ba.BSATTN_DEBUG_STALL, want_meta=False, lay=lay)
    assert res["status"] == ba.BSATTN_ERR_TIMEOUT
    lay.destroy()
    # the same process and context still compute correct results
    full_case(ba, q, k, v, mask, w.block, w.scale, what="after a timeout")


def _mid_case():
    # 192 work units (8 heads x 6 frames x 4 pairs of query tiles): more than one per CTA
    B, H, nf, bs, D = 1, 8, 6, 1024, 128
    L = nf * bs
    q = synth.tensor_bf16(31, synth.TAG_Q, B, H, L, D)
    k = synth.tensor_bf16(31, synth.TAG_K, B, H, L, D)
    v = synth.tensor_bf16(31, synth.TAG_V, B, H, L, D)
    return q, k, v, synth.window_mask(nf, 1), bs, 1.0 / np.sqrt(D)


def _tails_case(D=128, per_head=False, loose=False):
    # 9 frames of 272 tokens (two full query tiles and a 16-row tail): the tails of up to 8
    # consecutive frames share one packed query tile
    B, H, nf, bs = 1, 3, 9, 272
    L = nf * bs
    q = synth.tensor_bf16(77, synth.TAG_Q, B, H, L, D)
    k = synth.tensor_bf16(77, synth.TAG_K, B, H, L, D)
    v = synth.tensor_bf16(77, synth.TAG_V, B, H, L, D)
    if loose:  # a key of head 1 in frame 4, 1e4 times longer: the units that read frame 4 go online
        k = k.copy()
        k[0, 1, 4 * bs + 7] = synth.f32_to_bf16_bits((synth.bf16_bits_to_f64(k[0, 1, 4 * bs + 7]) * 1e4)
                                                     .astype(np.float32))
    mask = (np.stack([synth.window_mask(nf, 1, True), synth.window_mask(nf, 2), synth.dense_mask(nf)])
            if per_head else synth.window_mask(nf, 1, True))
    return q, k, v, mask, bs, float(np.float32(1 / np.sqrt(D)))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("per_head", [False, True])
@pytest.mark.parametrize("flags", [0, 1, 4])
def test_packed_tails_full(ba, D, per_head, flags):
    # Frames whose last query tile holds 16 rows: their tails are packed into shared query
    # tiles that read the union of the frames' key frames, each row only its own frames.
    # Every row against the oracle (bound path, online kernel, bound softmax for every row).
    q, k, v, mask, bs, scale = _tails_case(D, per_head)
    B, H, L, _ = q.shape
    lay = ba.bsattn_create_layout(B, H, L, D, bs, mask, ba.BSATTN_PLAN_ONLY)
    assert lay.info.tail_units > 0
    lay.destroy()
    res = full_case(ba, q, k, v, mask, bs, scale, flags=flags, what=f"packed tails D{D} per_head={per_head}")
    assert res["fb_rows"] == 0


def test_packed_tails_with_a_loose_key(ba):
    # The loose key sends the units that read its frame, packed tails included, to the online
    # launch: every row against the oracle, the online units as the oracle's bounds predict.
    q, k, v, mask, bs, scale = _tails_case(128, True, loose=True)
    res = full_case(ba, q, k, v, mask, bs, scale, what="packed tails, loose key")
    unit_of_row, n_units = _row_units(ba, q, k, mask, bs)
    must, may, _, online = _predicted_flags(q, k, v, mask, bs, scale, eligible=64.0, unit_of_row=unit_of_row)
    want_online = len(np.unique(unit_of_row[online]))
    assert want_online > 0 and res["online_units"] == want_online
    assert res["bound_units"] == n_units - want_online and must <= res["fb_rows"] <= may


@pytest.mark.parametrize("name", ["tiny", "small", "stream_small", "small_heads", "mid", "tails"])
def test_device_checks_accept_valid_plans_and_change_nothing(ba, name):
    # BSATTN_DEBUG_CHECKS on a valid plan: no unit rejected (status stays ok) and the
    # output is bit-identical to the unchecked launch.
    if name == "mid":
        q, k, v, mask, bs, scale = _mid_case()
    elif name == "tails":
        q, k, v, mask, bs, scale = _tails_case(128, True)
    else:
        w = synth.WORKLOADS[name]
        q, k, v = synth.make_qkv(w)
        mask, bs, scale = w.block_mask(), w.block, w.scale
    plain = run_gpu(ba, q, k, v, mask, bs, scale, 0, want_meta=False)
    checked = run_gpu(ba, q, k, v, mask, bs, scale, ba.BSATTN_DEBUG_CHECKS, want_meta=False)
    assert plain["status"] == 0 and checked["status"] == 0
    assert torch.equal(plain["o_raw"].view(torch.int16), checked["o_raw"].view(torch.int16))


def test_device_checks_reject_a_planted_key_tile(ba):
    # Testing flag: the checks see the first key tile of every CTA's first work unit as
    # starting past the last key.  Every role skips those units (their rows keep the NaN
    # the output was filled with, whole query tiles at a time), the other units match the
    # oracle, no rerun touches the skipped ones, and the layout reports the index status.
    q, k, v, mask, bs, scale = _mid_case()
    B, H, L, D = q.shape
    res = run_gpu(ba, q, k, v, mask, bs, scale, ba.BSATTN_DEBUG_CHECKS | ba.BSATTN_DEBUG_PLANT_INDEX,
                  want_meta=False)
    assert res["status"] == ba.BSATTN_ERR_INDEX
    assert res["fb_rows"] == 0
    skipped = np.isnan(res["o"]).all(axis=1)
    assert np.array_equal(skipped, np.isnan(res["o"]).any(axis=1))
    tiles = skipped.reshape(B * H, L // bs, bs // 128, 128)
    assert np.all(tiles.all(axis=3) == tiles.any(axis=3)), "a query tile was skipped in part"
    n_tiles_skipped = int(tiles.all(axis=3).sum())
    grid = min(B * H * (L // bs) * (bs // 256), torch.cuda.get_device_properties(0).multi_processor_count)
    assert 0 < n_tiles_skipped <= 2 * grid
    assert n_tiles_skipped < tiles.shape[0] * tiles.shape[1] * tiles.shape[2]
    O, _, _ = oracle.attention(q, k, v, mask, bs, scale)
    check_o(res["o"][~skipped], O[~skipped], "units the checks let through")


def test_cuda_graph_capture_and_replay(ba):
    # A whole step (row bounds + forward with its memset, bound kernel and rerun launch)
    # captured once in a CUDA graph and replayed on new inputs copied into the same buffers:
    # the replays reproduce plain launches bit for bit.
    w = synth.WORKLOADS["small"]
    lay = ba.bsattn_create_layout(w.B, w.H, w.L, w.D, w.block, w.block_mask())
    q, k, v = synth.make_qkv(w)
    dq, dk, dv = _dev(q), _dev(k), _dev(v)
    o = torch.empty_like(dq)
    qn = torch.empty((w.B, w.H, w.L), dtype=torch.float32, device="cuda")
    km = torch.empty((w.B, w.H, w.nb_kv), dtype=torch.float32, device="cuda")
    rb = torch.empty((w.B, w.H, w.L), dtype=torch.float32, device="cuda")

    def step():
        ba.bsattn_row_bounds(lay, dq, dk, w.scale, qn, km, rb)
        ba.bsattn_forward(lay, dq, dk, dv, o, w.scale, rb, None, ba.BSATTN_BOUND)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for seed in (21, 22):
        q2 = synth.tensor_bf16(seed, synth.TAG_Q, w.B, w.H, w.L, w.D)
        k2 = synth.tensor_bf16(seed, synth.TAG_K, w.B, w.H, w.L, w.D)
        v2 = synth.tensor_bf16(seed, synth.TAG_V, w.B, w.H, w.L, w.D)
        dq.copy_(_dev(q2)); dk.copy_(_dev(k2)); dv.copy_(_dev(v2))
        g.replay()
        torch.cuda.synchronize()
        replayed = o.clone()
        step()
        torch.cuda.synchronize()
        assert torch.equal(replayed.view(torch.int16), o.view(torch.int16))
        O, _, _ = oracle.attention(q2, k2, v2, w.block_mask(), w.block, w.scale)
        check_o(_host_bf16(replayed).reshape(-1, w.D), O, f"graph replay seed {seed}")
    _, _, status = ba.bsattn_query_stats(lay)
    assert status == 0
    lay.destroy()


# ------------------------------------------------------------------------------------------------
# row bounds from norms supplied by the caller's producer kernel


@pytest.mark.parametrize("name", ["tiny", "small", "stream_small", "small_heads"])
def test_row_bounds_from_norms_bit_exact(ba, name):
    # The norm table of the deep-dive (section 拿掉 softmax 的序列相依) handed in by a
    # producer: given the oracle's own per-token norms, kmax and rowbound are the oracle's
    # bit for bit, and the forward with that bound equals the forward after
    # bsattn_row_bounds bit for bit.  Arbitrary positive norms (not the norms of Q and K)
    # are checked against the oracle's block maximum and row bound as well.
    w = synth.WORKLOADS[name]
    q, k, v = synth.make_qkv(w)
    mask = w.block_mask()
    B, H, L, D = q.shape
    L_kv = k.shape[2]
    nbkv = L_kv // w.block
    lay = ba.bsattn_create_layout(B, H, L, D, w.block, mask, L_kv=L_kv)
    qn_o, km_o, rb_o = oracle.metadata_f32(q, k, mask, w.block, w.scale)
    kn_o = oracle.row_norms_f32(k)
    dqn = torch.from_numpy(qn_o).cuda()
    dkn = torch.from_numpy(kn_o).cuda()
    km = torch.full((B, H, nbkv), float("nan"), dtype=torch.float32, device="cuda")
    rb = torch.full((B, H, L), float("nan"), dtype=torch.float32, device="cuda")
    ba.bsattn_row_bounds_from_norms(lay, dqn, dkn, w.scale, km, rb)
    torch.cuda.synchronize()
    assert np.array_equal(km.cpu().numpy().view(np.uint32), km_o.view(np.uint32))
    assert np.array_equal(rb.cpu().numpy().view(np.uint32), rb_o.view(np.uint32))

    res = run_gpu(ba, q, k, v, mask, w.block, w.scale, lay=lay)
    dq, dk, dv = _dev(q), _dev(k), _dev(v)
    o = torch.full_like(dq, float("nan"))
    ba.bsattn_forward(lay, dq, dk, dv, o, w.scale, rb, None, 0)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), res["o_raw"].view(torch.int16))

    rng = np.random.default_rng(3)
    qn_r = (rng.random((B, H, L)) * 20).astype(np.float32)
    kn_r = (rng.random((B, H, L_kv)) * 20).astype(np.float32)
    kn_r[0, 0, : w.block] = 0.0  # a key block whose norms are all zero
    km_want = oracle.block_max_f32(kn_r, w.block)
    rb_want = oracle.row_bounds_f32(qn_r, km_want, mask, w.block, w.scale)
    ba.bsattn_row_bounds_from_norms(lay, torch.from_numpy(qn_r).cuda(), torch.from_numpy(kn_r).cuda(), w.scale,
                                    km, rb)
    torch.cuda.synchronize()
    assert np.array_equal(km.cpu().numpy().view(np.uint32), km_want.view(np.uint32))
    assert np.array_equal(rb.cpu().numpy().view(np.uint32), rb_want.view(np.uint32))
    lay.destroy()


def test_row_bounds_from_norms_720p(ba):
    # full size: the bound from the oracle's norms equals bsattn_row_bounds' bit for bit
    w = synth.WORKLOADS["720p"]
    q, k, v = synth.make_qkv(w)
    B, H, L, D = q.shape
    lay = ba.bsattn_create_layout(B, H, L, D, w.block, w.block_mask())
    dq, dk = _dev(q), _dev(k)
    qn = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    km = torch.empty((B, H, w.nb), dtype=torch.float32, device="cuda")
    rb = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    ba.bsattn_row_bounds(lay, dq, dk, w.scale, qn, km, rb)
    dkn = torch.from_numpy(oracle.row_norms_f32(k)).cuda()
    km2, rb2 = torch.empty_like(km), torch.empty_like(rb)
    ba.bsattn_row_bounds_from_norms(lay, qn, dkn, w.scale, km2, rb2)
    torch.cuda.synchronize()
    assert torch.equal(km.view(torch.int32), km2.view(torch.int32))
    assert torch.equal(rb.view(torch.int32), rb2.view(torch.int32))
    lay.destroy()


def test_ulysses_head_groups_on_one_gpu_equal_the_whole_attention(ba, monkeypatch):
    # The head-group pipeline of ulysses.py with one rank (NCCL, the exchanges are copies):
    # each group's attention runs through the C ABI on its heads' slice of the per-head masks,
    # and the result equals one forward over all heads bit for bit (every unit computes the
    # same rows in the same order, whatever the grid and schedule).
    import torch.distributed as dist
    from block_sparse_video_row_b300 import ulysses
    monkeypatch.setenv("NCCL_NVLS_ENABLE", "0")
    monkeypatch.setenv("MASTER_ADDR", "127.0.0.1")
    monkeypatch.setenv("MASTER_PORT", "29637")
    w = synth.WORKLOADS["small_heads"]
    q, k, v = synth.make_qkv(w)
    dq, dk, dv = _dev(q), _dev(k), _dev(v)
    mask = w.block_mask()
    whole = ba.attention(dq, dk, dv, mask, w.block, w.scale)
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        got = ulysses.ulysses_attention(dq, dk, dv, ulysses.bsattn_group_attend(mask, w.block, w.scale), groups=4)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    assert torch.equal(got.view(torch.int16), whole.view(torch.int16))
