// bsattn_forward_noalloc: the attention forward for callers that may not allocate
// device memory.
//
// Some callers cannot call cudaMalloc: a plugin whose host framework owns every
// byte of device memory through its own fixed arena, or a streaming loop that
// must not take cudaMalloc's implicit device synchronisation in the middle of a
// chunk.  bsattn_create_layout allocates a few device buffers (the work plan and
// the underflow-guard workspace), so such a caller cannot use bsattn_forward.
// This entry point runs the same kernels with those buffers placed in one
// fixed, file-scope device array instead.
//
// The array is kNoallocScratchBytes (1 MiB) of device memory that every GPU which
// loads this library keeps until the process exits.  All calls share it and it
// keeps the contents of the last call; each call rewrites what must start at
// zero (status word, counters, per-unit flags) together with the plan.  Calls
// whose work overlaps on the GPU (different streams, or different host threads
// without ordering) race on the array.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "bsattn.h"
#include "internal.h"
#include "layout.h"

namespace {

constexpr size_t kNoallocScratchBytes = BSATTN_NOALLOC_SCRATCH_BYTES;

// The scratch array.  In host code `g_scratch` names a host-side stand-in, not a
// device address: its address must come from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
struct DeviceState {
    bool ready = false;
    unsigned char *scratch = nullptr;  // device address of g_scratch on this device
    int num_sms = 0;
};
DeviceState g_devices[kMaxDevices];
std::mutex g_mutex;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Once per device, with that device current: check it, fetch the device address of
// the scratch array and the SM count.
bsattn_status device_setup(int dev, DeviceState **out) {
    if (dev < 0 || dev >= kMaxDevices) return BSATTN_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState &d = g_devices[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return BSATTN_ERR_DEVICE;
        if (major != 10 || minor != 3) return BSATTN_ERR_DEVICE;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return BSATTN_ERR_CUDA;
        d.scratch = static_cast<unsigned char *>(p);
        d.num_sms = sms;
        d.ready = true;
    }
    *out = &d;
    return BSATTN_OK;
}

// Device state of the current device (set-up on first use), or an error.
bsattn_status current_device(DeviceState **ds) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return BSATTN_ERR_DEVICE;
    return device_setup(dev, ds);
}

}  // namespace

extern "C" bsattn_status bsattn_forward_noalloc(const void *q, const void *k, const void *v, void *o, int32_t B,
                                                int32_t H, int64_t L, int32_t D, int32_t block_size,
                                                const uint8_t *block_mask, float scale, const float *rowbound,
                                                float *lse, int32_t flags, bsattn_stream_t stream) {
    if ((flags & ~(BSATTN_ONLINE_MAX | BSATTN_NO_FALLBACK | BSATTN_BOUND_ONLY | BSATTN_MASK_PER_HEAD |
                   BSATTN_DEBUG_STALL)) != 0)
        return BSATTN_ERR_INVALID_ARG;
    const bool online = (flags & BSATTN_ONLINE_MAX) != 0;
    if (!q || !k || !v || !o || (!online && !rowbound)) return BSATTN_ERR_INVALID_ARG;
    const auto mis16 = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15u) != 0; };
    if (mis16(q) || mis16(k) || mis16(v) || mis16(o)) return BSATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(rowbound) & 3) || (reinterpret_cast<uintptr_t>(lse) & 3))
        return BSATTN_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return BSATTN_ERR_INVALID_ARG;
    // The plan is copied from a host buffer that lives only during this call, so a
    // graph captured from it would read freed memory at replay.
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &capture) != cudaSuccess)
        return BSATTN_ERR_CUDA;
    if (capture != cudaStreamCaptureStatusNone) return BSATTN_ERR_UNSUPPORTED;

    // The work plan, built on the host only (the plan-only layout touches no device),
    // and dealt to one persistent CTA per SM by the same cost model as a device layout,
    // so the kernels see the same slots as bsattn_forward's.
    DeviceState *ds = nullptr;
    bsattn_status st = current_device(&ds);
    if (st != BSATTN_OK) return st;
    bsattn_layout_t plan = nullptr;
    st = bsattn_create_layout(&plan, B, H, L, D, block_size, block_mask,
                              BSATTN_PLAN_ONLY | (flags & BSATTN_MASK_PER_HEAD));
    if (st != BSATTN_OK) return st;
    bsattn_layout_info_t info;
    bsattn_layout_info(plan, &info);
    const int grid = std::max(1, std::min(info.n_units, ds->num_sms));
    std::vector<int32_t> slots;
    int32_t n_slots = 0;
    try {
        n_slots = bsv::schedule_units(*plan, grid, slots);
    } catch (const std::bad_alloc &) {
        bsattn_destroy(plan);
        return BSATTN_ERR_OOM;
    }
    const size_t n = static_cast<size_t>(n_slots);
    const size_t ntiles = static_cast<size_t>(info.key_tiles > 0 ? info.key_tiles : 1);

    // Scratch layout: guard workspace (8 header ints: status, -, -, -, fallback count,
    // fallback rows, units routed online, units left bound; then per slot a guard flag,
    // the fallback list and the route), the slots, the key-tile table.  Sizes beyond the
    // array are rejected here, before any device work.
    const size_t off_units = align256((bsv::kWsHeaderInts + 3 * n) * 4);
    const size_t off_tileptr = align256(off_units + 16 * n);
    const size_t off_tiles = align256(off_tileptr + 4 * (static_cast<size_t>(info.n_segments) + 1));
    const size_t total = off_tiles + 8 * ntiles;
    if (total > kNoallocScratchBytes) {
        bsattn_destroy(plan);
        return BSATTN_ERR_UNSUPPORTED;
    }
    std::vector<unsigned char> host;
    try {
        host.assign(total, 0);
    } catch (const std::bad_alloc &) {
        bsattn_destroy(plan);
        return BSATTN_ERR_OOM;
    }
    std::memcpy(host.data() + off_units, slots.data(), slots.size() * 4);
    bsattn_layout_export(plan, nullptr, nullptr, nullptr, reinterpret_cast<int32_t *>(host.data() + off_tileptr),
                         reinterpret_cast<int32_t *>(host.data() + off_tiles));

    CUtensorMap tq, tk, tv;
    if (!bsv::encode_layout_maps(plan, q, k, v, &tq, &tk, &tv)) {
        bsattn_destroy(plan);
        return BSATTN_ERR_CUDA;
    }
    cudaError_t e = info.D == 128 ? bsv::configure_attention_d128() : bsv::configure_attention_d64();
    bsattn_destroy(plan);
    if (e != cudaSuccess) return BSATTN_ERR_CUDA;

    // One stream-ordered copy writes the plan and zeroes the workspace (the host
    // buffer may be released on return: a pageable-source copy is staged first).
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned char *base = ds->scratch;
    e = cudaMemcpyAsync(base, host.data(), total, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return BSATTN_ERR_CUDA;

    int32_t *ws = reinterpret_cast<int32_t *>(base);
    bsv::AttnParams p;
    p.units = reinterpret_cast<const int4 *>(base + off_units);
    p.n_units = n_slots;
    p.tile_ptr = reinterpret_cast<const int32_t *>(base + off_tileptr);
    p.tiles = reinterpret_cast<const int2 *>(base + off_tiles);
    p.n_tiles = info.key_tiles;
    p.n_seg = info.n_segments;
    p.q = q;
    p.bh = info.B * info.H;
    p.heads = info.H;
    p.mask_heads = info.mask_heads;
    p.rowbound = rowbound;
    p.o = static_cast<uint16_t *>(o);
    p.lse = lse;
    p.ws = bsv::workspace_at(ws, n_slots);
    p.L = L;
    p.Lkv = L;
    p.block = block_size;
    p.nb = info.nb;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.elig_m = (flags & BSATTN_BOUND_ONLY) ? INFINITY : BSATTN_ELIGIBLE_BOUND;
    p.debug_stall = (flags & BSATTN_DEBUG_STALL) ? 1 : 0;
    p.checks = 0;
    p.debug_plant = 0;
    uint64_t ms = 4000;
    if (const char *env = std::getenv("BSATTN_TIMEOUT_MS")) {
        const long long val = std::atoll(env);
        if (val > 0) ms = static_cast<uint64_t>(val);
    }
    p.timeout_ns = ms * 1000000ull;
    auto launch = [&](bool on) {
        return info.D == 128 ? bsv::launch_attention_d128(tq, tk, tv, p, on, grid, s)
                             : bsv::launch_attention_d64(tq, tk, tv, p, on, grid, s);
    };
    if (online) {
        p.mode = bsv::kModeOnlineAll;
        return launch(true) == cudaSuccess ? BSATTN_OK : BSATTN_ERR_CUDA;
    }
    if (bsv::launch_route(p, s) != cudaSuccess) return BSATTN_ERR_CUDA;
    p.mode = bsv::kModeBound;
    if (launch(false) != cudaSuccess) return BSATTN_ERR_CUDA;
    if (flags & BSATTN_NO_FALLBACK) return BSATTN_OK;
    p.mode = bsv::kModeFallback;
    p.debug_stall = 0;
    return launch(true) == cudaSuccess ? BSATTN_OK : BSATTN_ERR_CUDA;
}

extern "C" bsattn_status bsattn_noalloc_query(int64_t *fallback_rows, int64_t *fallback_units,
                                              int32_t *device_status, bsattn_stream_t stream) {
    DeviceState *ds = nullptr;
    bsattn_status st = current_device(&ds);
    if (st != BSATTN_OK) return st;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return BSATTN_ERR_CUDA;
    int32_t h[8];
    if (cudaMemcpy(h, ds->scratch, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return BSATTN_ERR_CUDA;
    if (fallback_units) *fallback_units = h[4];
    if (fallback_rows) *fallback_rows = h[5];
    if (device_status)
        *device_status = (h[0] & bsv::kStatusTimeout) ? BSATTN_ERR_TIMEOUT
                         : (h[0] & bsv::kStatusIndex) ? BSATTN_ERR_INDEX
                                                       : BSATTN_OK;
    return BSATTN_OK;
}
