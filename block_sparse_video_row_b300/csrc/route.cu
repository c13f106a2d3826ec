// Eligibility of each work unit for the bound softmax, decided before the attention
// launches.  The deep-dive ("HeyGen Avatar IV on Trillium TPU", section
// 拿掉 softmax 的序列相依) checks per head whether the Cauchy-Schwarz bound is tight
// enough to serve as the softmax shift and sends the heads that fail to the online
// softmax.  Here the check is per work unit (one or two 128-row query tiles of one
// frame): a unit whose rows all have m_i <= elig_m stays with the bound-softmax
// launch, and a unit with a larger bound goes, whole, to the online-max launch that
// follows it on the same stream.  Neither kernel then carries the other's loop.
//
// One warp per schedule slot reads the bounds of the slot's rows (at most 256 floats; a
// packed tile of frame tails reads the tail rows of each of its frames).
// Every slot's guard flag is cleared here too, so the forward needs no memset of the
// per-slot arrays.  A slot whose unit fields are out of range is left to the bound
// launch, whose device checks (when on) reject and report it.
#include "internal.h"
#include "ptx.cuh"

namespace bsv {

constexpr int kRouteThreads = 256;

__global__ void __launch_bounds__(kRouteThreads) route_kernel(const AttnParams p) {
    grid_dep_launch_next();  // the bound launch may start launching (it waits for this kernel)
    const int64_t slot = (static_cast<int64_t>(blockIdx.x) * kRouteThreads + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (slot >= p.n_units) return;  // whole warps leave together
    const int4 U = p.units[slot];
    bool online = false;
    if (U.w > 0) {
        const bool valid = U.w <= 2 && U.x >= 0 && U.x < p.bh && U.y >= 0 && U.y < p.nb && U.z >= 0 &&
                           (static_cast<int64_t>(U.z) + U.w - 1) * kQTile < p.block;
        if (valid) {
            const int64_t base = static_cast<int64_t>(U.x) * p.L + static_cast<int64_t>(U.y) * p.block;
            for (int t = 0; t < U.w; ++t) {
                const int r0 = (U.z + t) * kQTile;
                const int nrows = min(kQTile, p.block - r0);
                for (int r = lane; r < nrows; r += 32) online |= __ldg(p.rowbound + base + r0 + r) > p.elig_m;
            }
        }
    } else if (U.w < 0) {
        // packed tails: the tail rows of frames U.y .. U.y - U.w - 1
        const bool valid = U.w >= -kMaxTailGroup && U.x >= 0 && U.x < p.bh && U.y >= 0 && U.y - U.w <= p.nb;
        if (valid) {
            const int r0 = tail_row0(p.block), nrows = tail_rows(p.block);
            for (int g = 0; g < -U.w; ++g) {
                const int64_t base = static_cast<int64_t>(U.x) * p.L + static_cast<int64_t>(U.y + g) * p.block + r0;
                for (int r = lane; r < nrows; r += 32) online |= __ldg(p.rowbound + base + r) > p.elig_m;
            }
        }
    }
    online = __any_sync(0xFFFFFFFFu, online);
    if (lane == 0) {
        p.ws.slot_online[slot] = online ? 1 : 0;
        p.ws.unit_flag[slot] = 0;
        if (U.w != 0) atomicAdd(online ? p.ws.n_online : p.ws.n_bound, 1);
    }
}

cudaError_t launch_route(const AttnParams &p, cudaStream_t s) {
    const int64_t warps_per_cta = kRouteThreads / 32;
    const int64_t grid = (static_cast<int64_t>(p.n_units) + warps_per_cta - 1) / warps_per_cta;
    route_kernel<<<static_cast<unsigned>(grid > 0 ? grid : 1), kRouteThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace bsv
