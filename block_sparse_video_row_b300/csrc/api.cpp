// The C ABI of libbsattn.so: argument checks, the host plan (allowed key blocks,
// key tile, work list), device buffers, TMA tensor maps and kernel launches.
// The operation and its conventions are documented in include/bsattn.h.
#include "bsattn.h"

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "internal.h"
#include "layout.h"

namespace {

constexpr int kWsHeader = bsv::kWsHeader;

bsattn_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return BSATTN_OK;
    return e == cudaErrorMemoryAllocation ? BSATTN_ERR_OOM : BSATTN_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

void build_plan(bsattn_layout_s &lay, const uint8_t *mask) {
    const int32_t nb = lay.nb;
    const int32_t nbkv = lay.nbkv;
    const int32_t nseg = lay.mask_heads * nb;  // (mask, query block) segments
    lay.row_ptr.assign(static_cast<size_t>(nseg) + 1, 0);
    lay.col_idx.clear();
    for (int32_t sg = 0; sg < nseg; ++sg) {
        for (int32_t kb = 0; kb < nbkv; ++kb)
            if (mask[static_cast<int64_t>(sg) * nbkv + kb]) lay.col_idx.push_back(kb);
        lay.row_ptr[sg + 1] = static_cast<int32_t>(lay.col_idx.size());
    }
    // Key tiles: the allowed key blocks of a query block, grouped into runs of
    // consecutive frames (contiguous keys, all allowed), each run cut into tiles of
    // kKvTile keys and one last tile of the remaining keys.  Frames are multiples of
    // 16 tokens, so every width is a multiple of 16: an exactly sized MMA, with no
    // element mask and no padding, and no tile reaches into a masked frame.
    lay.kv_tile = bsv::kKvTile;
    lay.qt_per_block = (lay.bs + bsv::kQTile - 1) / bsv::kQTile;
    lay.tile_ptr.assign(static_cast<size_t>(nseg) + 1, 0);
    lay.tiles.clear();
    for (int32_t sg = 0; sg < nseg; ++sg) {
        int32_t e = lay.row_ptr[sg];
        const int32_t e1 = lay.row_ptr[sg + 1];
        while (e < e1) {
            int32_t run_end = e + 1;
            while (run_end < e1 && lay.col_idx[run_end] == lay.col_idx[run_end - 1] + 1) ++run_end;
            const int64_t k0 = static_cast<int64_t>(lay.col_idx[e]) * lay.bs;
            const int64_t k1 = static_cast<int64_t>(lay.col_idx[run_end - 1] + 1) * lay.bs;
            for (int64_t k = k0; k < k1; k += bsv::kKvTile) {
                lay.tiles.push_back(static_cast<int32_t>(k));
                lay.tiles.push_back(static_cast<int32_t>(std::min<int64_t>(bsv::kKvTile, k1 - k)));
            }
            e = run_end;
        }
        lay.tile_ptr[sg + 1] = static_cast<int32_t>(lay.tiles.size() / 2);
    }

    // Tail groups.  A frame of an odd number of query tiles whose last tile holds at most
    // half a tile of rows (a 3600-token frame: 28 full tiles and 16 rows) leaves that tail
    // as a unit of its own, which costs a whole tile's pass over the frame's key tiles for
    // a few rows.  The tails of consecutive frames are packed into one query tile instead
    // (row group g = frame qb0 + g, rows [g * tail_rows, (g + 1) * tail_rows)), as long as
    // each added frame costs fewer key tiles than its own unit would: the packed tile reads
    // every key frame any of its frames reads, cut into tiles at frame edges so that each
    // key tile belongs to one frame, and each tile carries the set of row groups allowed to
    // read it (bits 16.. of its width word); the kernel gives the other rows a shift of
    // -inf for that tile, so their P is exactly 0.  No element mask is needed: a row reads
    // whole key frames or nothing, as in every other unit.
    const int32_t qt = lay.qt_per_block;
    const int32_t tail_row0 = (qt - 1) * bsv::kQTile;
    const int32_t tail_rows = lay.bs - tail_row0;
    const bool grouping = qt % 2 == 1 && 2 * tail_rows <= bsv::kQTile;
    const int32_t max_group = grouping ? std::min(bsv::kMaxTailGroup, bsv::kQTile / tail_rows) : 1;
    const int64_t tiles_per_frame = (lay.bs + bsv::kKvTile - 1) / bsv::kKvTile;
    struct Group {
        int32_t qb0, n, seg;
    };
    std::vector<std::vector<Group>> groups(static_cast<size_t>(lay.mask_heads));
    std::vector<int32_t> in_group(static_cast<size_t>(nseg), 0);  // frame's tail is in a packed tile
    int32_t n_seg_all = nseg;
    for (int32_t m = 0; m < lay.mask_heads && grouping; ++m) {
        int32_t qb = 0;
        while (qb < nb) {
            const int32_t s0 = m * nb + qb;
            if (lay.row_ptr[s0 + 1] == lay.row_ptr[s0]) {  // reads nothing: its own unit writes zeros
                ++qb;
                continue;
            }
            std::vector<uint8_t> uni(static_cast<size_t>(nbkv), 0);
            for (int32_t e = lay.row_ptr[s0]; e < lay.row_ptr[s0 + 1]; ++e) uni[lay.col_idx[e]] = 1;
            int64_t n_uni = lay.row_ptr[s0 + 1] - lay.row_ptr[s0];      // key frames of the union
            int64_t own_sum = lay.tile_ptr[s0 + 1] - lay.tile_ptr[s0];  // the members' own tail units
            int32_t n = 1;
            while (n < max_group && qb + n < nb) {
                const int32_t s1 = m * nb + qb + n;
                if (lay.row_ptr[s1 + 1] == lay.row_ptr[s1]) break;
                int64_t added = 0;
                for (int32_t e = lay.row_ptr[s1]; e < lay.row_ptr[s1 + 1]; ++e) added += uni[lay.col_idx[e]] ? 0 : 1;
                const int64_t own = lay.tile_ptr[s1 + 1] - lay.tile_ptr[s1];
                // the packed tile (frame-cut tiles of the union) must stay cheaper than the
                // members' own tail units together
                if ((n_uni + added) * tiles_per_frame >= own_sum + own) break;
                for (int32_t e = lay.row_ptr[s1]; e < lay.row_ptr[s1 + 1]; ++e) uni[lay.col_idx[e]] = 1;
                n_uni += added;
                own_sum += own;
                ++n;
            }
            if (n >= 2) {
                const int32_t seg = n_seg_all++;
                for (int32_t kb = 0; kb < nbkv; ++kb) {
                    if (!uni[kb]) continue;
                    int32_t rows = 0;  // row groups allowed to read key frame kb
                    for (int32_t g = 0; g < n; ++g)
                        if (mask[static_cast<int64_t>(m * nb + qb + g) * nbkv + kb]) rows |= 1 << g;
                    const int64_t k0 = static_cast<int64_t>(kb) * lay.bs, k1 = k0 + lay.bs;
                    for (int64_t k = k0; k < k1; k += bsv::kKvTile) {
                        lay.tiles.push_back(static_cast<int32_t>(k));
                        lay.tiles.push_back(static_cast<int32_t>(std::min<int64_t>(bsv::kKvTile, k1 - k)) |
                                            (rows << 16));
                    }
                }
                lay.tile_ptr.push_back(static_cast<int32_t>(lay.tiles.size() / 2));
                groups[m].push_back({qb, n, seg});
                for (int32_t g = 0; g < n; ++g) in_group[m * nb + qb + g] = 1;
            }
            qb += n;
        }
    }
    lay.n_segments = n_seg_all;
    lay.tail_units = 0;

    // Cost model (in hundredths of a two-tile key tile): a unit of two query tiles takes
    // 100 per key tile; a unit of one tile (a frame's lone tail, or packed tails) 83,
    // because its softmax cannot overlap another tile's MMAs; plus 150 per unit (query
    // loads, epilogue).  Units are listed in (head, frame, tile) order, a packed tile
    // after the last frame of its group; schedule_units orders and deals them.
    const int32_t BH = lay.B * lay.H;
    std::vector<int32_t> &U = lay.units;
    U.clear();
    lay.unit_cost.clear();
    U.reserve(static_cast<size_t>(BH) * nb * ((qt + 1) / 2) * 4);
    int64_t mma_tiles = 0, allowed_pairs = 0;  // over the B * H sequences
    auto push = [&](int32_t x, int32_t y, int32_t z, int32_t w, int64_t cost, int64_t tiles_through_mma) {
        U.push_back(x);
        U.push_back(y);
        U.push_back(z);
        U.push_back(w);
        lay.unit_cost.push_back(cost);
        mma_tiles += tiles_through_mma;
    };
    for (int32_t bh = 0; bh < BH; ++bh) {
        const int32_t m = lay.mask_heads > 1 ? bh % lay.H : 0;
        size_t next_group = 0;
        for (int32_t qb = 0; qb < nb; ++qb) {
            const int sg = bsv::plan_segment(lay.mask_heads, lay.H, nb, bh, qb);
            const int64_t ntile = lay.tile_ptr[sg + 1] - lay.tile_ptr[sg];
            allowed_pairs += lay.row_ptr[sg + 1] - lay.row_ptr[sg];
            const int64_t reads = ntile > 0 ? 1 : 0;
            for (int32_t qt0 = 0; qt0 < qt; qt0 += 2) {
                const int32_t nt = std::min(2, qt - qt0);
                if (nt == 1 && in_group[m * nb + qb]) continue;  // its tail rides in a packed tile
                push(bh, qb, qt0, nt, ntile * (nt == 2 ? 100 : 83) + 150, reads * nt);
            }
            if (next_group < groups[m].size()) {
                const Group &gr = groups[m][next_group];
                if (qb == gr.qb0 + gr.n - 1) {
                    const int64_t gt = lay.tile_ptr[gr.seg + 1] - lay.tile_ptr[gr.seg];
                    push(bh, gr.qb0, gr.seg, -gr.n, gt * 83 + 150, 1);
                    ++lay.tail_units;
                    ++next_group;
                }
            }
        }
    }
    lay.n_units = static_cast<int32_t>(lay.unit_cost.size());
    lay.mma_rows = mma_tiles * bsv::kQTile;
    lay.useful_flop =
        4.0 * static_cast<double>(allowed_pairs) * static_cast<double>(lay.bs) * static_cast<double>(lay.bs) * lay.D;
}

// cuTensorMapEncodeTiled, fetched from the driver once (no link-time libcuda dependency).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Q (and O) viewed as [B*H*nb frames][block rows][D]: a 128-row box that starts
// inside a frame and runs past its end reads zeros there (never the next frame).
bool encode_q_map(CUtensorMap *m, const bsattn_layout_s &lay, const void *ptr) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(lay.D), static_cast<cuuint64_t>(lay.bs),
                                static_cast<cuuint64_t>(lay.B) * lay.H * lay.nb};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(lay.D) * 2,
                                   static_cast<cuuint64_t>(lay.D) * 2 * lay.bs};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(bsv::kQTile), 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K and V viewed as [B*H*L_kv rows][D].  A box of kv_tile rows starts at a key tile; when the
// tile is the narrower last one of a run, the rows past it are loaded but never used.
bool encode_kv_map(CUtensorMap *m, const bsattn_layout_s &lay, const void *ptr) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(lay.D),
                                static_cast<cuuint64_t>(lay.B) * lay.H * static_cast<cuuint64_t>(lay.Lkv)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(lay.D) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(lay.kv_tile)};
    const cuuint32_t es[2] = {1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

void free_device(bsattn_layout_s *lay) {
    if (lay->d_row_ptr) cudaFree(lay->d_row_ptr);
    if (lay->d_col_idx) cudaFree(lay->d_col_idx);
    if (lay->d_units) cudaFree(lay->d_units);
    if (lay->d_tile_ptr) cudaFree(lay->d_tile_ptr);
    if (lay->d_tiles) cudaFree(lay->d_tiles);
    if (lay->d_ws) cudaFree(lay->d_ws);
    lay->d_row_ptr = lay->d_col_idx = lay->d_tile_ptr = nullptr;
    lay->d_tiles = nullptr;
    lay->d_units = nullptr;
    lay->d_ws = nullptr;
}

bsattn_status setup_device(bsattn_layout_s &lay) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BSATTN_ERR_DEVICE;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return BSATTN_ERR_DEVICE;
    if (prop.major != 10 || prop.minor != 3) return BSATTN_ERR_DEVICE;  // built for sm_103a only
    if (!encode_fn()) return BSATTN_ERR_CUDA;
    lay.device = dev;
    lay.num_sms = prop.multiProcessorCount;

    cudaError_t e = lay.D == 128 ? bsv::configure_attention_d128() : bsv::configure_attention_d64();
    if (e != cudaSuccess) return from_cuda(e);

    const size_t nnz = std::max<size_t>(lay.col_idx.size(), 1);
    const size_t ntiles = std::max<size_t>(lay.tiles.size() / 2, 1);
    lay.grid = std::max(1, std::min(lay.n_units, lay.num_sms));
    std::vector<int32_t> slots;
    try {
        lay.n_slots = bsv::schedule_units(lay, lay.grid, slots);
    } catch (const std::bad_alloc &) {
        return BSATTN_ERR_OOM;
    }
    const size_t ws_ints = kWsHeader + 3 * static_cast<size_t>(lay.n_slots);
    if ((e = cudaMalloc(&lay.d_row_ptr, lay.row_ptr.size() * 4)) != cudaSuccess ||
        (e = cudaMalloc(&lay.d_col_idx, nnz * 4)) != cudaSuccess ||
        (e = cudaMalloc(&lay.d_tile_ptr, lay.tile_ptr.size() * 4)) != cudaSuccess ||
        (e = cudaMalloc(&lay.d_tiles, ntiles * sizeof(int2))) != cudaSuccess ||
        (e = cudaMalloc(&lay.d_units, static_cast<size_t>(lay.n_slots) * sizeof(int4))) != cudaSuccess ||
        (e = cudaMalloc(&lay.d_ws, ws_ints * 4)) != cudaSuccess) {
        free_device(&lay);
        return from_cuda(e);
    }
    if ((e = cudaMemcpy(lay.d_row_ptr, lay.row_ptr.data(), lay.row_ptr.size() * 4, cudaMemcpyHostToDevice)) !=
            cudaSuccess ||
        (!lay.col_idx.empty() &&
         (e = cudaMemcpy(lay.d_col_idx, lay.col_idx.data(), lay.col_idx.size() * 4, cudaMemcpyHostToDevice)) !=
             cudaSuccess) ||
        (e = cudaMemcpy(lay.d_units, slots.data(), slots.size() * 4, cudaMemcpyHostToDevice)) !=
            cudaSuccess ||
        (e = cudaMemcpy(lay.d_tile_ptr, lay.tile_ptr.data(), lay.tile_ptr.size() * 4, cudaMemcpyHostToDevice)) !=
            cudaSuccess ||
        (!lay.tiles.empty() &&
         (e = cudaMemcpy(lay.d_tiles, lay.tiles.data(), lay.tiles.size() * 4, cudaMemcpyHostToDevice)) !=
             cudaSuccess) ||
        (e = cudaMemset(lay.d_ws, 0, ws_ints * 4)) != cudaSuccess) {
        free_device(&lay);
        return from_cuda(e);
    }
    lay.ws = bsv::workspace_at(lay.d_ws, lay.n_slots);

    uint64_t ms = 4000;
    if (const char *env = std::getenv("BSATTN_TIMEOUT_MS")) {
        const long long v = std::atoll(env);
        if (v > 0) ms = static_cast<uint64_t>(v);
    }
    lay.timeout_ns = ms * 1000000ull;
    return BSATTN_OK;
}

// Parameters of the bound kernels for a layout (Q and K pointers left null).
bsv::BoundsParams bounds_params(const bsattn_layout_s &lay, float scale, float *qnorm, float *kmax, float *rowbound) {
    bsv::BoundsParams p;
    p.q = nullptr;
    p.k = nullptr;
    p.qnorm = qnorm;
    p.kmax_bits = reinterpret_cast<uint32_t *>(kmax);
    p.rowbound = rowbound;
    p.row_ptr = lay.d_row_ptr;
    p.col_idx = lay.d_col_idx;
    p.L = lay.L;
    p.Lkv = lay.Lkv;
    p.block = lay.bs;
    p.nb = lay.nb;
    p.nbkv = lay.nbkv;
    p.BH = lay.B * lay.H;
    p.heads = lay.H;
    p.mask_heads = lay.mask_heads;
    p.chunks_per_block = (lay.bs + bsv::bounds_chunk_rows() - 1) / bsv::bounds_chunk_rows();
    p.scale = scale;
    return p;
}

bsattn_status check_runnable(const bsattn_layout_s *lay) {
    if (!lay || lay->plan_only) return BSATTN_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != lay->device) return BSATTN_ERR_INVALID_ARG;
    return BSATTN_OK;
}

}  // namespace

namespace bsv {
// Units of the schedule's cost-sorted tail, in waves of G (one unit per CTA).
constexpr int32_t kTailWaves = 4;

int32_t schedule_units(const bsattn_layout_s &lay, int32_t G, std::vector<int32_t> &slots) {
    G = std::max(1, G);
    // Deal order: the plan's (head, frame, tile) order, so that the CTAs running at any
    // one time work on one or two heads and find each K/V tile in L2 after its first read
    // (a head's K and V take 1.8 MB per 3600-token frame); then the last kTailWaves * G
    // units by cost, largest first (ties keep plan order), so small units fill the end
    // and the CTAs finish together.
    const int32_t n = lay.n_units;
    std::vector<int32_t> order(static_cast<size_t>(n));
    for (int32_t u = 0; u < n; ++u) order[u] = u;
    const int64_t tail = std::min<int64_t>(n, static_cast<int64_t>(kTailWaves) * G);
    std::stable_sort(order.begin() + (n - tail), order.end(),
                     [&](int32_t a, int32_t b) { return lay.unit_cost[a] > lay.unit_cost[b]; });
    std::vector<std::vector<int32_t>> per(static_cast<size_t>(G));
    std::vector<int64_t> load(static_cast<size_t>(G), 0);
    // least-loaded CTA first (ties: lowest index), units in cost order
    typedef std::pair<int64_t, int32_t> Entry;
    std::vector<Entry> heap;
    for (int32_t c = 0; c < G; ++c) heap.push_back({0, c});
    auto cmp = [](const Entry &a, const Entry &b) { return a.first != b.first ? a.first > b.first : a.second > b.second; };
    std::make_heap(heap.begin(), heap.end(), cmp);
    for (int32_t u : order) {
        std::pop_heap(heap.begin(), heap.end(), cmp);
        Entry &e = heap.back();
        per[e.second].push_back(u);
        e.first += lay.unit_cost[u];
        std::push_heap(heap.begin(), heap.end(), cmp);
    }
    size_t K = 0;
    for (const auto &v : per) K = std::max(K, v.size());
    slots.assign(K * G * 4, 0);
    for (size_t k = 0; k < K; ++k)
        for (int32_t c = 0; c < G; ++c)
            if (k < per[c].size())
                for (int f = 0; f < 4; ++f) slots[(k * G + c) * 4 + f] = lay.units[4 * per[c][k] + f];
    return static_cast<int32_t>(K * G);
}

bool encode_o_store_map(CUtensorMap *m, const AttnParams &p, int D) {
    if (!encode_fn()) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(p.block),
                                static_cast<cuuint64_t>(p.bh) * static_cast<cuuint64_t>(p.nb)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(D) * 2 * p.block};
    const cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.o, dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                       CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_q_tail_map(CUtensorMap *m, const AttnParams &p, int D) {
    if (!encode_fn()) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(p.block),
                                static_cast<cuuint64_t>(p.bh) * static_cast<cuuint64_t>(p.nb)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(D) * 2 * p.block};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(tail_rows(p.block)), 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(p.q), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_layout_maps(const bsattn_layout_s *lay, const void *q, const void *k, const void *v, CUtensorMap *tq,
                        CUtensorMap *tk, CUtensorMap *tv) {
    return encode_fn() && encode_q_map(tq, *lay, q) && encode_kv_map(tk, *lay, k) && encode_kv_map(tv, *lay, v);
}
}  // namespace bsv

extern "C" {

bsattn_status bsattn_create_layout(bsattn_layout_t *out, int32_t B, int32_t H, int64_t L, int32_t D,
                                   int32_t block_size, const uint8_t *block_mask, int32_t flags) {
    return bsattn_create_layout_rect(out, B, H, L, L, D, block_size, block_mask, flags);
}

bsattn_status bsattn_create_layout_rect(bsattn_layout_t *out, int32_t B, int32_t H, int64_t L, int64_t L_kv,
                                        int32_t D, int32_t block_size, const uint8_t *block_mask, int32_t flags) {
    if (!out) return BSATTN_ERR_INVALID_ARG;
    *out = nullptr;
    if (!block_mask || B < 1 || H < 1 || L < 1 || L_kv < 1 || block_size < 1) return BSATTN_ERR_INVALID_ARG;
    if ((flags & ~(BSATTN_PLAN_ONLY | BSATTN_MASK_PER_HEAD)) != 0) return BSATTN_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return BSATTN_ERR_UNSUPPORTED;
    if (block_size % 16 != 0 || L % block_size != 0 || L_kv % block_size != 0) return BSATTN_ERR_UNALIGNED_BLOCK;
    const int64_t nb = L / block_size, nbkv = L_kv / block_size;
    if (nb > BSATTN_MAX_NB || nbkv > BSATTN_MAX_NB) return BSATTN_ERR_UNSUPPORTED;
    if (L_kv < L) return BSATTN_ERR_UNSUPPORTED;  // a chunk reads at least its own frames' worth of keys
    if (static_cast<int64_t>(B) * H * std::max(L, L_kv) > BSATTN_MAX_ROWS) return BSATTN_ERR_UNSUPPORTED;

    bsattn_layout_s *lay = new (std::nothrow) bsattn_layout_s;
    if (!lay) return BSATTN_ERR_OOM;
    try {
        lay->B = B;
        lay->H = H;
        lay->L = L;
        lay->Lkv = L_kv;
        lay->D = D;
        lay->bs = block_size;
        lay->nb = static_cast<int32_t>(nb);
        lay->nbkv = static_cast<int32_t>(nbkv);
        lay->mask_heads = (flags & BSATTN_MASK_PER_HEAD) ? H : 1;
        lay->plan_only = (flags & BSATTN_PLAN_ONLY) != 0;
        build_plan(*lay, block_mask);
    } catch (const std::bad_alloc &) {
        delete lay;
        return BSATTN_ERR_OOM;
    }
    if (!lay->plan_only) {
        const bsattn_status st = setup_device(*lay);
        if (st != BSATTN_OK) {
            delete lay;
            return st;
        }
    }
    *out = lay;
    return BSATTN_OK;
}

bsattn_status bsattn_row_bounds(bsattn_layout_t lay, const void *q, const void *k, float scale, float *qnorm,
                                float *kmax, float *rowbound, bsattn_stream_t stream) {
    bsattn_status st = check_runnable(lay);
    if (st != BSATTN_OK) return st;
    if (!q || !k || !qnorm || !kmax || !rowbound) return BSATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned4(qnorm) || !aligned4(kmax) || !aligned4(rowbound))
        return BSATTN_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return BSATTN_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    bsv::BoundsParams p = bounds_params(*lay, scale, qnorm, kmax, rowbound);
    p.q = static_cast<const uint16_t *>(q);
    p.k = static_cast<const uint16_t *>(k);
    cudaError_t e = cudaMemsetAsync(kmax, 0, static_cast<size_t>(p.BH) * lay->nbkv * 4, s);
    if (e == cudaSuccess) e = bsv::launch_norms(p, lay->D, s);
    if (e == cudaSuccess) e = bsv::launch_rowbound(p, s);
    return from_cuda(e);
}

bsattn_status bsattn_row_bounds_from_norms(bsattn_layout_t lay, const float *qnorm, const float *knorm, float scale,
                                           float *kmax, float *rowbound, bsattn_stream_t stream) {
    bsattn_status st = check_runnable(lay);
    if (st != BSATTN_OK) return st;
    if (!qnorm || !knorm || !kmax || !rowbound) return BSATTN_ERR_INVALID_ARG;
    if (!aligned4(qnorm) || !aligned4(knorm) || !aligned4(kmax) || !aligned4(rowbound)) return BSATTN_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return BSATTN_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the row-bound kernel only reads qnorm
    bsv::BoundsParams p = bounds_params(*lay, scale, const_cast<float *>(qnorm), kmax, rowbound);
    cudaError_t e = cudaMemsetAsync(kmax, 0, static_cast<size_t>(p.BH) * lay->nbkv * 4, s);
    if (e == cudaSuccess) e = bsv::launch_kmax_from_norms(p, knorm, s);
    if (e == cudaSuccess) e = bsv::launch_rowbound(p, s);
    return from_cuda(e);
}

bsattn_status bsattn_forward(bsattn_layout_t lay, const void *q, const void *k, const void *v, void *o,
                             float scale, const float *rowbound, float *lse, int32_t flags,
                             bsattn_stream_t stream) {
    bsattn_status st = check_runnable(lay);
    if (st != BSATTN_OK) return st;
    if ((flags & ~(BSATTN_ONLINE_MAX | BSATTN_NO_FALLBACK | BSATTN_BOUND_ONLY | BSATTN_DEBUG_STALL |
                   BSATTN_DEBUG_CHECKS | BSATTN_DEBUG_PLANT_INDEX)) != 0)
        return BSATTN_ERR_INVALID_ARG;
    if ((flags & BSATTN_DEBUG_PLANT_INDEX) && !(flags & BSATTN_DEBUG_CHECKS)) return BSATTN_ERR_INVALID_ARG;
    const bool online = (flags & BSATTN_ONLINE_MAX) != 0;
    if (!q || !k || !v || !o || (!online && !rowbound)) return BSATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return BSATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(rowbound) & 3) || (reinterpret_cast<uintptr_t>(lse) & 3))
        return BSATTN_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return BSATTN_ERR_INVALID_ARG;

    CUtensorMap tq, tk, tv;
    if (!encode_q_map(&tq, *lay, q) || !encode_kv_map(&tk, *lay, k) || !encode_kv_map(&tv, *lay, v))
        return BSATTN_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // per-call counters of the workspace header: fb_count, fb_rows, n_online, n_bound
    cudaError_t e = cudaMemsetAsync(lay->d_ws + 4, 0, (kWsHeader - 4) * 4, s);
    if (e != cudaSuccess) return from_cuda(e);

    bsv::AttnParams p;
    p.units = lay->d_units;
    p.n_units = lay->n_slots;
    p.tile_ptr = lay->d_tile_ptr;
    p.tiles = lay->d_tiles;
    p.n_tiles = static_cast<int32_t>(lay->tiles.size() / 2);
    p.n_seg = lay->n_segments;
    p.q = q;
    p.bh = lay->B * lay->H;
    p.heads = lay->H;
    p.mask_heads = lay->mask_heads;
    p.rowbound = rowbound;
    p.o = static_cast<uint16_t *>(o);
    p.lse = lse;
    p.ws = lay->ws;
    p.L = lay->L;
    p.Lkv = lay->Lkv;
    p.block = lay->bs;
    p.nb = lay->nb;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.elig_m = (flags & BSATTN_BOUND_ONLY) ? INFINITY : BSATTN_ELIGIBLE_BOUND;
    p.debug_stall = (flags & BSATTN_DEBUG_STALL) ? 1 : 0;
    p.checks = (flags & BSATTN_DEBUG_CHECKS) ? 1 : 0;
    p.debug_plant = (flags & BSATTN_DEBUG_PLANT_INDEX) ? 1 : 0;
    p.timeout_ns = lay->timeout_ns;
    const int grid = lay->grid;  // the width the schedule was built for
    auto launch = [&](bool on) {
        return lay->D == 128 ? bsv::launch_attention_d128(tq, tk, tv, p, on, grid, s)
                             : bsv::launch_attention_d64(tq, tk, tv, p, on, grid, s);
    };
    if (online) {
        p.mode = bsv::kModeOnlineAll;
        return from_cuda(launch(true));
    }
    // the eligibility check of every unit, then the bound launch over the eligible ones
    // and the online launch over the others and the guard's fallback list
    e = bsv::launch_route(p, s);
    if (e != cudaSuccess) return from_cuda(e);
    p.mode = bsv::kModeBound;
    e = launch(false);
    if (e != cudaSuccess) return from_cuda(e);
    if (flags & BSATTN_NO_FALLBACK) return BSATTN_OK;
    p.mode = bsv::kModeFallback;
    p.debug_stall = 0;
    p.debug_plant = 0;
    return from_cuda(launch(true));
}

void bsattn_destroy(bsattn_layout_t lay) {
    if (!lay) return;
    if (!lay->plan_only) {
        int cur = -1;
        cudaGetDevice(&cur);
        if (cur != lay->device) cudaSetDevice(lay->device);
        bsv::host_pipe_destroy(lay->host);
        lay->host = nullptr;
        free_device(lay);
        if (cur != lay->device && cur >= 0) cudaSetDevice(cur);
    }
    delete lay;
}

const char *bsattn_status_string(bsattn_status st) {
    switch (st) {
        case BSATTN_OK: return "ok";
        case BSATTN_ERR_INVALID_ARG: return "invalid argument";
        case BSATTN_ERR_UNALIGNED_BLOCK: return "block size not a multiple of 16, or L not a multiple of it";
        case BSATTN_ERR_UNSUPPORTED: return "unsupported size or head dim";
        case BSATTN_ERR_CUDA: return "CUDA error";
        case BSATTN_ERR_OOM: return "out of device memory";
        case BSATTN_ERR_TIMEOUT: return "a bounded device wait ran out";
        case BSATTN_ERR_DEVICE: return "no usable sm_103 device";
        case BSATTN_ERR_INDEX: return "the device checks found a work unit or key tile out of range";
    }
    return "unknown status";
}

bsattn_status bsattn_query_stats(bsattn_layout_t lay, int64_t *fallback_rows, int64_t *fallback_units,
                                 int32_t *device_status, bsattn_stream_t stream) {
    bsattn_status st = check_runnable(lay);
    if (st != BSATTN_OK) return st;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return from_cuda(e);
    int32_t h[kWsHeader];
    e = cudaMemcpy(h, lay->d_ws, sizeof h, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return from_cuda(e);
    if (fallback_units) *fallback_units = h[4];
    if (fallback_rows) *fallback_rows = h[5];
    if (device_status)
        *device_status = (h[0] & bsv::kStatusTimeout) ? BSATTN_ERR_TIMEOUT
                         : (h[0] & bsv::kStatusIndex) ? BSATTN_ERR_INDEX
                                                       : BSATTN_OK;
    return BSATTN_OK;
}

bsattn_status bsattn_query_eligibility(bsattn_layout_t lay, int64_t *bound_units, int64_t *online_units,
                                      bsattn_stream_t stream) {
    bsattn_status st = check_runnable(lay);
    if (st != BSATTN_OK) return st;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return from_cuda(e);
    int32_t h[kWsHeader];
    e = cudaMemcpy(h, lay->d_ws, sizeof h, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return from_cuda(e);
    if (online_units) *online_units = h[6];
    if (bound_units) *bound_units = h[7];
    return BSATTN_OK;
}

bsattn_status bsattn_layout_info(bsattn_layout_t lay, bsattn_layout_info_t *info) {
    if (!lay || !info) return BSATTN_ERR_INVALID_ARG;
    info->B = lay->B;
    info->H = lay->H;
    info->D = lay->D;
    info->block_size = lay->bs;
    info->nb = lay->nb;
    info->L = lay->L;
    info->nnz_blocks = static_cast<int32_t>(lay->col_idx.size());
    info->kv_tile = lay->kv_tile;
    info->key_tiles = static_cast<int32_t>(lay->tiles.size() / 2);
    info->q_tiles_per_block = lay->qt_per_block;
    info->n_units = lay->n_units;
    info->mma_rows = lay->mma_rows;
    info->useful_flop = lay->useful_flop;
    info->L_kv = lay->Lkv;
    info->nb_kv = lay->nbkv;
    info->mask_heads = lay->mask_heads;
    info->n_segments = lay->n_segments;
    info->tail_units = lay->tail_units;
    return BSATTN_OK;
}

bsattn_status bsattn_layout_schedule(bsattn_layout_t lay, int32_t grid, int32_t *slots, int32_t *n_slots) {
    if (!lay || !n_slots || grid < 1) return BSATTN_ERR_INVALID_ARG;
    std::vector<int32_t> v;
    try {
        *n_slots = bsv::schedule_units(*lay, grid, v);
    } catch (const std::bad_alloc &) {
        return BSATTN_ERR_OOM;
    }
    if (slots && !v.empty()) std::memcpy(slots, v.data(), v.size() * 4);
    return BSATTN_OK;
}

bsattn_status bsattn_layout_export(bsattn_layout_t lay, int32_t *row_ptr, int32_t *col_idx, int32_t *units,
                                   int32_t *tile_ptr, int32_t *tiles) {
    if (!lay) return BSATTN_ERR_INVALID_ARG;
    if (tile_ptr) std::memcpy(tile_ptr, lay->tile_ptr.data(), lay->tile_ptr.size() * 4);
    if (tiles && !lay->tiles.empty()) std::memcpy(tiles, lay->tiles.data(), lay->tiles.size() * 4);
    if (row_ptr) std::memcpy(row_ptr, lay->row_ptr.data(), lay->row_ptr.size() * 4);
    if (col_idx && !lay->col_idx.empty()) std::memcpy(col_idx, lay->col_idx.data(), lay->col_idx.size() * 4);
    if (units && !lay->units.empty()) std::memcpy(units, lay->units.data(), lay->units.size() * 4);
    return BSATTN_OK;
}

}  // extern "C"
