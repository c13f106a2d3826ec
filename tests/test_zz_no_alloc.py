"""bsattn_forward_noalloc: the forward for callers that may not allocate device memory.

A plugin whose host framework owns all device memory, or a streaming loop that
cannot take cudaMalloc's implicit synchronisation, cannot create a layout (that
allocates the work plan and the guard workspace on the device).  The no-alloc
entry point keeps those in a fixed device array inside the library.  It runs the
same kernels on the same schedule as the layout-based bsattn_forward, so here its
output must equal bsattn_forward's bit for bit, and the fp64 oracle's within the
tolerance of the other GPU tests, on several calls in a row through the C ABI.
The loose-key case is run twice in a row: its guard flags units in the shared
array, so the second call must start from cleared flags and counters, or the
flagged units would not be rerun and the output would differ.  This file is
collected last on purpose.
"""
import warnings

import numpy as np
import pytest

import oracle
from block_sparse_video_row_b300 import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN = 2e-2, 2e-3


@pytest.fixture(scope="module")
def ba():
    from block_sparse_video_row_b300 import _build, bsattn
    _build.build()
    bsattn.load()
    return bsattn


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()


def _f64(t):
    return synth.bf16_bits_to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16))


def _case(name, loose_key=False):
    w = synth.WORKLOADS[name]
    q, k, v = synth.make_qkv(w)
    if loose_key:  # one key 1e4 times longer: the bound underflows for the rows that read it
        k = k.copy()
        k[0, 0, 3] = synth.f32_to_bf16_bits((synth.bf16_bits_to_f64(k[0, 0, 3]) * 1e4).astype(np.float32))
    return w, q, k, v


def _both(ba, w, q, k, v, flags):
    """(layout output, no-alloc output, layout stats, no-alloc stats) on the same inputs."""
    mask = w.block_mask()
    dq, dk, dv = _dev(q), _dev(k), _dev(v)
    lay = ba.bsattn_create_layout(w.B, w.H, w.L, w.D, w.block, mask)
    qn = torch.empty((w.B, w.H, w.L), dtype=torch.float32, device="cuda")
    km = torch.empty((w.B, w.H, w.nb), dtype=torch.float32, device="cuda")
    rb = torch.empty((w.B, w.H, w.L), dtype=torch.float32, device="cuda")
    ba.bsattn_row_bounds(lay, dq, dk, w.scale, qn, km, rb)
    o_ref = torch.full_like(dq, float("nan"))
    ba.bsattn_forward(lay, dq, dk, dv, o_ref, w.scale, rb, None, flags)
    stats_ref = ba.bsattn_query_stats(lay)
    o_na = torch.full_like(dq, float("nan"))
    ba.bsattn_forward_noalloc(dq, dk, dv, o_na, w.B, w.H, w.L, w.D, w.block, mask, w.scale, rb, None,
                              flags)
    stats_na = ba.bsattn_noalloc_query()
    lay.destroy()
    return o_ref, o_na, stats_ref, stats_na


def _check(ba, name, flags, loose_key=False):
    w, q, k, v = _case(name, loose_key)
    o_ref, o_na, st_ref, st_na = _both(ba, w, q, k, v, flags)
    assert st_ref[2] == 0 and st_na == st_ref  # same guard counts, status ok
    assert torch.equal(o_na.view(torch.int16), o_ref.view(torch.int16))  # same kernels, same schedule
    want, _, _ = oracle.attention(q, k, v, w.block_mask(), w.block, w.scale)
    got = _f64(o_na).reshape(-1, w.D)
    err = np.abs(got - want)
    assert np.all(np.isfinite(got)) and err.max() <= O_MAX and err.mean() <= O_MEAN
    return st_na


def test_noalloc_matches_forward_on_calls_in_a_row(ba):
    # calls 1 and 2: rows that need the online-max rerun (the bound softmax for every row,
    # so the guard fires instead of the eligibility switch); the same units are flagged
    # both times, which needs the flags of call 1 cleared before call 2
    first = _check(ba, "tiny", ba.BSATTN_BOUND_ONLY, loose_key=True)
    assert first[0] > 0 and first[1] > 0
    second = _check(ba, "tiny", ba.BSATTN_BOUND_ONLY, loose_key=True)
    assert second == first
    # call 3: a larger problem with nothing to rerun
    assert _check(ba, "small", ba.BSATTN_BOUND)[:2] == (0, 0)


def test_noalloc_with_one_mask_per_head(ba):
    assert _check(ba, "small_heads", ba.BSATTN_BOUND)[:2] == (0, 0)


def test_noalloc_reports_a_wait_that_ran_out(ba, monkeypatch):
    # The testing flag keeps the first work unit of every CTA from getting its query tiles,
    # so the kernel's bounded waits run out after BSATTN_TIMEOUT_MS and it returns; the
    # no-alloc query reports the timeout, and the next call works and reports ok.
    monkeypatch.setenv("BSATTN_TIMEOUT_MS", "200")
    w, q, k, v = _case("tiny")
    dq, dk, dv = _dev(q), _dev(k), _dev(v)
    o = torch.empty_like(dq)
    rb = torch.zeros((w.B, w.H, w.L), dtype=torch.float32, device="cuda")  # any bound works for the stall
    ba.bsattn_forward_noalloc(dq, dk, dv, o, w.B, w.H, w.L, w.D, w.block, w.block_mask(), w.scale, rb, None,
                              ba.BSATTN_DEBUG_STALL)
    assert ba.bsattn_noalloc_query()[2] == ba.BSATTN_ERR_TIMEOUT
    monkeypatch.delenv("BSATTN_TIMEOUT_MS")
    assert _check(ba, "tiny", ba.BSATTN_BOUND)[2] == 0


def test_noalloc_rejects_plans_beyond_its_array(ba):
    # 512 heads of the 720p shape: ~100k work units, more than the 1 MiB array holds.
    # The check comes before any device work, so the pointers are never dereferenced.
    fake = 1 << 20
    mask = synth.window_mask(13, 1, True)
    st = ba.bsattn_forward_noalloc(fake, fake, fake, fake, 1, 512, 13 * 3600, 128, 3600, mask, 0.088, fake, None,
                                   0, raise_on_error=False)
    assert st == ba.BSATTN_ERR_UNSUPPORTED


def test_noalloc_refuses_stream_capture(ba):
    # Its plan copy reads a host buffer that is gone once the call returns, so a captured
    # graph would replay a copy from freed memory: the call refuses a capturing stream
    # before any work (nothing is captured).
    w = synth.WORKLOADS["tiny"]
    q, k, v = synth.make_qkv(w)
    dq, dk, dv = _dev(q), _dev(k), _dev(v)
    o = torch.empty_like(dq)
    rb = torch.ones((w.B, w.H, w.L), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with warnings.catch_warnings():
        warnings.simplefilter("ignore")  # torch notes that the captured graph is empty, as intended
        with torch.cuda.graph(g):
            st = ba.bsattn_forward_noalloc(dq, dk, dv, o, w.B, w.H, w.L, w.D, w.block, w.block_mask(), w.scale,
                                           rb, None, 0, raise_on_error=False)
    assert st == ba.BSATTN_ERR_UNSUPPORTED
