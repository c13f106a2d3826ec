// The layout object behind bsattn_layout_t (shared by the C-ABI translation units).
#pragma once

#include <cstdint>
#include <vector>

#include "internal.h"

struct bsattn_layout_s;

namespace bsv {
struct HostPipe;                   // staging and streams of bsattn_forward_host (host_pipeline.cu)
void host_pipe_destroy(HostPipe *hp);
constexpr int kWsHeader = kWsHeaderInts;  // int32 workspace header: [0] status, [4] fb_count,
                                         // [5] fb_rows, [6] n_online, [7] n_bound
// The per-CTA schedule for a grid of G persistent CTAs: the units, in the layout's
// cost order, each given to the least-loaded CTA; slot k * G + c holds CTA c's k-th
// unit (4 int32 each), and empty slots are (0, 0, 0, 0), a unit of no query tiles
// that every role skips.  Returns the number of slots (a multiple of G).
int32_t schedule_units(const bsattn_layout_s &lay, int32_t G, std::vector<int32_t> &slots);
}  // namespace bsv

struct bsattn_layout_s {
    int32_t B = 0, H = 0, D = 0, bs = 0, nb = 0;  // nb: query blocks
    int64_t L = 0;                                // query tokens per sequence
    int32_t nbkv = 0;                             // key blocks
    int64_t Lkv = 0;                              // key tokens per sequence
    int32_t mask_heads = 1;                       // block masks: 1 (shared) or H (one per head)
    bool plan_only = false;
    std::vector<int32_t> row_ptr, col_idx, units;
    std::vector<int32_t> tile_ptr, tiles;  // tiles: (first key within the head, width) pairs
    int32_t kv_tile = 0, qt_per_block = 0, n_units = 0;
    int32_t n_segments = 0;  // segments of tile_ptr: masks * nb, then one per packed tail tile
    int32_t tail_units = 0;  // units that are packed tails of several frames
    std::vector<int64_t> unit_cost;  // cost model of each unit of `units`
    int32_t grid = 0, n_slots = 0;   // persistent CTAs and scheduled slots (device layouts)
    int64_t mma_rows = 0;
    double useful_flop = 0.0;
    int device = -1, num_sms = 0;
    int32_t *d_row_ptr = nullptr, *d_col_idx = nullptr, *d_tile_ptr = nullptr;
    int2 *d_tiles = nullptr;
    int4 *d_units = nullptr;
    int32_t *d_ws = nullptr;
    bsv::Workspace ws{};
    uint64_t timeout_ns = 0;
    bsv::HostPipe *host = nullptr;  // created by the first bsattn_forward_host call
};
