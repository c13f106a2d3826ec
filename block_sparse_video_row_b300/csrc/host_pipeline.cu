// bsattn_forward_host: row bounds and forward for Q, K, V and O held in host
// memory.  The (batch, head) pairs are cut into chunks of G consecutive pairs
// (contiguous in the [B, H, L, D] layout); chunk c runs
//     host -> device copies of its Q, K, V          on the copy-in stream,
//     row bounds + forward (+ rerun)                 on the compute stream,
//     device -> host copy of its O (and LSE)         on the copy-out stream,
// with two sets of device staging buffers, so the copies of one chunk overlap the
// kernels of its neighbours.  Events order each buffer's reuse: chunk c's copy-in
// waits for chunk c-2's compute (the inputs it overwrites), and chunk c's compute
// waits for chunk c-2's copy-out (the output it overwrites).  The call is ordered
// after earlier work on the caller's stream, and the caller's stream waits for
// its last copy-out.  Every chunk is an ordinary forward on a layout of shape
// (1, G, L, D) with the same mask (with one mask per head: the masks of the
// chunk's heads), so the results are those of bsattn_forward.
#include <algorithm>
#include <cmath>
#include <new>
#include <vector>

#include "bsattn.h"
#include "internal.h"
#include "layout.h"

namespace bsv {

struct HostPipe {
    int32_t G = 0, G_last = 0;             // pairs per chunk; pairs of the last chunk
    std::vector<bsattn_layout_t> chunk;    // the layout each chunk runs on
    std::vector<bsattn_layout_t> owned;    // the distinct chunk layouts
    cudaStream_t s_in = nullptr, s_cmp = nullptr, s_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_done = nullptr;
    cudaEvent_t ev_in[2] = {}, ev_cmp[2] = {}, ev_out[2] = {};
    uint16_t *dq[2] = {}, *dk[2] = {}, *dv[2] = {}, *dO[2] = {};
    float *qn[2] = {}, *km[2] = {}, *rb[2] = {}, *lse[2] = {};
};

void host_pipe_destroy(HostPipe *hp) {
    if (!hp) return;
    for (cudaStream_t s : {hp->s_in, hp->s_cmp, hp->s_out})
        if (s) cudaStreamSynchronize(s);
    for (int b = 0; b < 2; ++b) {
        for (void *p : {static_cast<void *>(hp->dq[b]), static_cast<void *>(hp->dk[b]),
                        static_cast<void *>(hp->dv[b]), static_cast<void *>(hp->dO[b]),
                        static_cast<void *>(hp->qn[b]), static_cast<void *>(hp->km[b]),
                        static_cast<void *>(hp->rb[b]), static_cast<void *>(hp->lse[b])})
            if (p) cudaFree(p);
        for (cudaEvent_t e : {hp->ev_in[b], hp->ev_cmp[b], hp->ev_out[b]})
            if (e) cudaEventDestroy(e);
    }
    if (hp->ev_start) cudaEventDestroy(hp->ev_start);
    if (hp->ev_done) cudaEventDestroy(hp->ev_done);
    for (cudaStream_t s : {hp->s_in, hp->s_cmp, hp->s_out})
        if (s) cudaStreamDestroy(s);
    for (bsattn_layout_t sub : hp->owned) bsattn_destroy(sub);
    delete hp;
}

namespace {

// Adds a chunk's counters into the layout's workspace (slots 0: status bits, 4: units
// rerun, 5: rows flagged, 6: units routed online, 7: units left bound), so
// bsattn_query_stats and bsattn_query_eligibility report the whole call.
__global__ void fold_stats_kernel(const int32_t *src, int32_t *dst) {
    dst[0] |= src[0];
    for (int i = 4; i < 8; ++i) dst[i] += src[i];  // guard and eligibility counters
}

bsattn_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return BSATTN_OK;
    return e == cudaErrorMemoryAllocation ? BSATTN_ERR_OOM : BSATTN_ERR_CUDA;
}

// Staging, streams, events and the chunk layouts for G pairs per chunk.
bsattn_status host_pipe_create(const bsattn_layout_s &lay, int32_t G, HostPipe **out) {
    HostPipe *hp = new (std::nothrow) HostPipe;
    if (!hp) return BSATTN_ERR_OOM;
    const int32_t BH = lay.B * lay.H;
    hp->G = G;
    hp->G_last = BH - (BH - 1) / G * G;
    // The masks, rebuilt from the plan: [mask_heads][nb][nbkv].
    const size_t per_mask = static_cast<size_t>(lay.nb) * lay.nbkv;
    std::vector<uint8_t> mask;
    try {
        mask.assign(static_cast<size_t>(lay.mask_heads) * per_mask, 0);
    } catch (const std::bad_alloc &) {
        host_pipe_destroy(hp);
        return BSATTN_ERR_OOM;
    }
    for (int32_t sg = 0; sg < lay.mask_heads * lay.nb; ++sg)
        for (int32_t e = lay.row_ptr[sg]; e < lay.row_ptr[sg + 1]; ++e)
            mask[static_cast<size_t>(sg) * lay.nbkv + lay.col_idx[e]] = 1;
    // Chunk c holds pairs c*G .. c*G + g - 1; pair p is head p % H.  With a shared mask
    // every chunk of g pairs runs on the same layout; with one mask per head, chunks
    // whose first head and size agree do.
    const int32_t nc = (BH + G - 1) / G;
    std::vector<std::pair<int64_t, bsattn_layout_t>> made;
    std::vector<uint8_t> sub_mask;
    bsattn_status st = BSATTN_OK;
    try {
        hp->chunk.reserve(static_cast<size_t>(nc));
        hp->owned.reserve(static_cast<size_t>(nc));
        made.reserve(static_cast<size_t>(nc));
        sub_mask.reserve(static_cast<size_t>(G) * per_mask * (lay.mask_heads > 1 ? 1 : 0));
    } catch (const std::bad_alloc &) {
        host_pipe_destroy(hp);
        return BSATTN_ERR_OOM;
    }
    for (int32_t c = 0; c < nc && st == BSATTN_OK; ++c) {
        const int32_t g = c == nc - 1 ? hp->G_last : G;
        const int32_t h0 = lay.mask_heads > 1 ? static_cast<int32_t>((static_cast<int64_t>(c) * G) % lay.H) : 0;
        const int64_t key = static_cast<int64_t>(h0) * (BH + 1) + g;
        bsattn_layout_t sub = nullptr;
        for (const auto &m : made)
            if (m.first == key) sub = m.second;
        if (!sub) {
            const uint8_t *mk = mask.data();
            int32_t fl = 0;
            if (lay.mask_heads > 1) {
                sub_mask.resize(static_cast<size_t>(g) * per_mask);
                for (int32_t i = 0; i < g; ++i)
                    std::copy_n(mask.data() + static_cast<size_t>((h0 + i) % lay.H) * per_mask, per_mask,
                                sub_mask.data() + static_cast<size_t>(i) * per_mask);
                mk = sub_mask.data();
                fl = BSATTN_MASK_PER_HEAD;
            }
            st = bsattn_create_layout_rect(&sub, 1, g, lay.L, lay.Lkv, lay.D, lay.bs, mk, fl);
            if (st != BSATTN_OK) break;
            made.push_back({key, sub});
            hp->owned.push_back(sub);
        }
        hp->chunk.push_back(sub);
    }
    if (st != BSATTN_OK) {
        host_pipe_destroy(hp);
        return st;
    }
    const size_t q_elems = static_cast<size_t>(G) * lay.L * lay.D;    // Q, O
    const size_t kv_elems = static_cast<size_t>(G) * lay.Lkv * lay.D; // K, V
    const size_t rows = static_cast<size_t>(G) * lay.L;
    cudaError_t e = cudaSuccess;
    for (cudaStream_t *s : {&hp->s_in, &hp->s_cmp, &hp->s_out})
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
    for (cudaEvent_t *ev : {&hp->ev_start, &hp->ev_done})
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
        for (cudaEvent_t *ev : {&hp->ev_in[b], &hp->ev_cmp[b], &hp->ev_out[b]})
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        for (uint16_t **p : {&hp->dq[b], &hp->dO[b]})
            if (e == cudaSuccess) e = cudaMalloc(p, q_elems * 2);
        for (uint16_t **p : {&hp->dk[b], &hp->dv[b]})
            if (e == cudaSuccess) e = cudaMalloc(p, kv_elems * 2);
        for (float **p : {&hp->qn[b], &hp->rb[b], &hp->lse[b]})
            if (e == cudaSuccess) e = cudaMalloc(p, rows * 4);
        if (e == cudaSuccess) e = cudaMalloc(&hp->km[b], static_cast<size_t>(G) * lay.nbkv * 4);
    }
    if (e != cudaSuccess) {
        host_pipe_destroy(hp);
        return from_cuda(e);
    }
    *out = hp;
    return BSATTN_OK;
}

}  // namespace
}  // namespace bsv

extern "C" bsattn_status bsattn_forward_host(bsattn_layout_t lay, const void *q, const void *k, const void *v,
                                             void *o, float scale, float *lse, int32_t flags,
                                             int32_t pairs_per_chunk, bsattn_stream_t stream) {
    if (!lay || lay->plan_only) return BSATTN_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != lay->device) return BSATTN_ERR_INVALID_ARG;
    if (!q || !k || !v || !o || pairs_per_chunk < 0) return BSATTN_ERR_INVALID_ARG;
    if ((flags & ~(BSATTN_ONLINE_MAX | BSATTN_NO_FALLBACK | BSATTN_BOUND_ONLY | BSATTN_DEBUG_CHECKS)) != 0)
        return BSATTN_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return BSATTN_ERR_INVALID_ARG;
    const int32_t BH = lay->B * lay->H;
    // About twelve chunks: the copies of one chunk overlap the kernels of its neighbours,
    // and the first copy-in and last copy-out, which nothing overlaps, stay short (at 720p,
    // two pairs per chunk measured 1.3% faster than three and 3.4% faster than six).
    const int32_t G = pairs_per_chunk > 0 ? std::min(pairs_per_chunk, BH) : std::max(1, (BH + 11) / 12);
    if (lay->host && lay->host->G != G) {
        bsv::host_pipe_destroy(lay->host);
        lay->host = nullptr;
    }
    if (!lay->host) {
        const bsattn_status st = bsv::host_pipe_create(*lay, G, &lay->host);
        if (st != BSATTN_OK) return st;
    }
    bsv::HostPipe &hp = *lay->host;
    const bool online = (flags & BSATTN_ONLINE_MAX) != 0;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const int32_t nc = (BH + G - 1) / G;
    const size_t pair_q = static_cast<size_t>(lay->L) * lay->D;     // elements of one pair's Q or O
    const size_t pair_kv = static_cast<size_t>(lay->Lkv) * lay->D;  // elements of one pair's K or V

    cudaError_t e = cudaEventRecord(hp.ev_start, cs);
    for (cudaStream_t s : {hp.s_in, hp.s_cmp, hp.s_out})
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hp.ev_start, 0);
    // the call's guard counters accumulate in the layout's workspace
    if (e == cudaSuccess) e = cudaMemsetAsync(lay->d_ws + 4, 0, 4 * sizeof(int32_t), hp.s_cmp);
    for (int32_t c = 0; c < nc && e == cudaSuccess; ++c) {
        const int b = c & 1;
        const int32_t g = c == nc - 1 ? hp.G_last : G;
        bsattn_layout_t sub = hp.chunk[c];
        const size_t off_q = static_cast<size_t>(c) * G * pair_q, off_kv = static_cast<size_t>(c) * G * pair_kv;
        const size_t bytes_q = static_cast<size_t>(g) * pair_q * 2, bytes_kv = static_cast<size_t>(g) * pair_kv * 2;
        const size_t rows = static_cast<size_t>(g) * lay->L;
        // copy in (buffer b is free once chunk c-2's kernels are done with it)
        if (c >= 2) e = cudaStreamWaitEvent(hp.s_in, hp.ev_cmp[b], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(hp.dq[b], static_cast<const uint16_t *>(q) + off_q, bytes_q, cudaMemcpyHostToDevice,
                                hp.s_in);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(hp.dk[b], static_cast<const uint16_t *>(k) + off_kv, bytes_kv,
                                cudaMemcpyHostToDevice, hp.s_in);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(hp.dv[b], static_cast<const uint16_t *>(v) + off_kv, bytes_kv,
                                cudaMemcpyHostToDevice, hp.s_in);
        if (e == cudaSuccess) e = cudaEventRecord(hp.ev_in[b], hp.s_in);
        // compute (the output buffer is free once chunk c-2's copy-out is done)
        if (e == cudaSuccess) e = cudaStreamWaitEvent(hp.s_cmp, hp.ev_in[b], 0);
        if (e == cudaSuccess && c >= 2) e = cudaStreamWaitEvent(hp.s_cmp, hp.ev_out[b], 0);
        if (e != cudaSuccess) break;
        bsattn_stream_t sc = reinterpret_cast<bsattn_stream_t>(hp.s_cmp);
        bsattn_status st = BSATTN_OK;
        if (!online) st = bsattn_row_bounds(sub, hp.dq[b], hp.dk[b], scale, hp.qn[b], hp.km[b], hp.rb[b], sc);
        if (st == BSATTN_OK)
            st = bsattn_forward(sub, hp.dq[b], hp.dk[b], hp.dv[b], hp.dO[b], scale, online ? nullptr : hp.rb[b],
                                lse ? hp.lse[b] : nullptr, flags, sc);
        if (st != BSATTN_OK) return st;
        bsv::fold_stats_kernel<<<1, 1, 0, hp.s_cmp>>>(sub->d_ws, lay->d_ws);
        e = cudaGetLastError();
        if (e == cudaSuccess) e = cudaEventRecord(hp.ev_cmp[b], hp.s_cmp);
        // copy out
        if (e == cudaSuccess) e = cudaStreamWaitEvent(hp.s_out, hp.ev_cmp[b], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<uint16_t *>(o) + off_q, hp.dO[b], bytes_q, cudaMemcpyDeviceToHost,
                                hp.s_out);
        if (e == cudaSuccess && lse)
            e = cudaMemcpyAsync(lse + static_cast<size_t>(c) * G * lay->L, hp.lse[b], rows * 4,
                                cudaMemcpyDeviceToHost, hp.s_out);
        if (e == cudaSuccess) e = cudaEventRecord(hp.ev_out[b], hp.s_out);
    }
    // every copy-out waited for its chunk's kernels, which waited for its copy-in
    if (e == cudaSuccess) e = cudaEventRecord(hp.ev_done, hp.s_out);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, hp.ev_done, 0);
    return bsv::from_cuda(e);
}
