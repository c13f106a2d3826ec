// Internal interfaces between the C-ABI host code (api.cpp) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

struct bsattn_layout_s;

namespace bsv {

constexpr int kQTile = 128;           // query rows per tile (the MMA M dimension)
constexpr int kKvTile = 128;          // keys per full key tile (TMEM: 2 S + 2 O accumulators of 128 columns)
constexpr int kMaxTailGroup = 8;      // frames whose tails share one packed query tile (mask bits 16..23)
constexpr int kAttnThreads = 384;     // 12 warps: TMA, MMA, 2 idle, 2 softmax warpgroups
constexpr int kLaunchRegs = 168;      // registers per thread at launch (65536 / 384, rounded down to 8)
constexpr int kRegsLow = 72;          // TMA / MMA warpgroup after setmaxnreg.dec
constexpr int kRegsHigh = 208;        // softmax warpgroups after setmaxnreg.inc
static_assert(128 * kRegsLow + 256 * kRegsHigh <= kAttnThreads * kLaunchRegs, "register split");
constexpr float kGuardTau = 5.421010862427522e-20f;  // 2^-64: smallest denominator trusted
constexpr int kStatusTimeout = 1;     // bits in the device status word: a bounded wait ran out,
constexpr int kStatusIndex = 2;       // the device checks rejected a work unit

// Device-side workspace of a layout (one allocation): an 8-int header, then three
// arrays of one int per schedule slot.  The header's counters are zeroed per forward
// (the status word only at create); the route kernel rewrites the per-slot arrays.
struct Workspace {
    int32_t *fb_count;     // [4] units appended to the fallback list
    int32_t *fb_rows;      // [5] rows flagged by the guard
    int32_t *status;       // [0] device status bits (kStatus*)
    int32_t *n_online;     // [6] units routed to the online-max launch (eligibility check)
    int32_t *n_bound;      // [7] units left to the bound-softmax launch
    int32_t *unit_flag;    // per slot: already appended to the fallback list
    int32_t *fb_list;      // slot indices to rerun
    int32_t *slot_online;  // per slot: 1 = a row of the unit is above the eligibility limit
};

// Workspace views over ws_ints = kWsHeaderInts + 3 * n_slots ints at d.
constexpr int kWsHeaderInts = 8;
inline Workspace workspace_at(int32_t *d, int32_t n_slots) {
    Workspace w;
    w.status = d + 0;
    w.fb_count = d + 4;
    w.fb_rows = d + 5;
    w.n_online = d + 6;
    w.n_bound = d + 7;
    w.unit_flag = d + kWsHeaderInts;
    w.fb_list = d + kWsHeaderInts + n_slots;
    w.slot_online = d + kWsHeaderInts + 2 * static_cast<int64_t>(n_slots);
    return w;
}

enum AttnMode : int32_t {
    kModeBound = 0,     // bound softmax over the slots the route kernel left bound, guard on
    kModeOnlineAll = 1, // online max over every unit
    kModeFallback = 2   // online max over the slots routed online, then the units listed in
                        // fb_list[0 .. *fb_count) by the bound launch's guard
};

struct AttnParams {
    const int4 *units;        // (b*H + h, qb, first q tile, tiles in unit: 1 or 2), or for packed
                              // tails (b*H + h, first frame, segment, -frames)
    int32_t n_units;
    const int32_t *tile_ptr;  // key tiles of segment s: tiles[tile_ptr[s] .. tile_ptr[s+1])
    const int2 *tiles;        // (first key within the head, width: a multiple of 16, <= kKvTile,
                              //  | row groups allowed << 16 for the tiles of a packed-tail segment)
    int32_t n_tiles;          // entries of tiles
    int32_t n_seg;            // segments (entries of tile_ptr minus one)
    const void *q;            // Q (bf16): the packed-tail loads use their own tensor map
    int32_t bh;               // B * H
    int32_t heads;            // H
    int32_t mask_heads;       // block masks: 1 (shared by all heads) or H (mask h for head h)
    const float *rowbound;    // [B*H*L]
    uint16_t *o;              // [B*H*L, D] bf16 bits
    float *lse;               // [B*H*L] or null
    Workspace ws;
    int64_t L;                // query tokens per sequence (Q, O rows per head)
    int64_t Lkv;              // key tokens per sequence (K, V rows per head)
    int32_t block;            // tokens per frame block
    int32_t nb;               // query blocks
    float scale_log2;         // scale * log2(e)
    float elig_m;             // route kernel: a unit with a larger row bound goes to the online launch
    int32_t mode;
    int32_t debug_stall;      // testing: skip the first unit's query-tile loads (waits run out)
    int32_t checks;           // device-side index checks of every unit before use
    int32_t debug_plant;      // testing, with checks: the first unit's first key tile reads as out of range
    uint64_t timeout_ns;
};

struct BoundsParams {
    const uint16_t *q, *k;
    float *qnorm;
    uint32_t *kmax_bits;      // fp32 bits, zeroed before the norms launch
    float *rowbound;
    const int32_t *row_ptr, *col_idx;
    int64_t L, Lkv;           // query / key tokens per sequence
    int32_t block, nb, nbkv, BH;
    int32_t heads, mask_heads; // H; block masks: 1 (shared) or H (mask h for head h)
    int32_t chunks_per_block; // row chunks per frame block
    float scale;
};

// Width and allowed row groups of a key tile.
__host__ __device__ __forceinline__ int tile_width(int2 t) { return t.y & 0xFFFF; }
__host__ __device__ __forceinline__ int tile_row_groups(int2 t) { return static_cast<int>(static_cast<uint32_t>(t.y) >> 16); }

// Rows of a frame's last query tile, and its first row, for frames of `block` tokens.
__host__ __device__ __forceinline__ int tail_row0(int block) { return (block - 1) / kQTile * kQTile; }
__host__ __device__ __forceinline__ int tail_rows(int block) { return block - tail_row0(block); }

// Segment of the plan's tables (row_ptr, tile_ptr) for query block qb of sequence bh
// (= b * H + h): mask m = h of a per-head plan (0 for a shared mask), segment m * nb + qb.
__host__ __device__ __forceinline__ int plan_segment(int mask_heads, int heads, int nb, int64_t bh, int qb) {
    return (mask_heads > 1 ? static_cast<int>(bh % heads) * nb : 0) + qb;
}

// TMA map for the epilogue's O stores (built per launch from p.o): 3-D (D, block rows,
// B*H*nb frames), box 32 columns x 32 rows, 64-byte swizzle.  False if the driver entry
// point is missing or the driver rejects the map.
bool encode_o_store_map(CUtensorMap *m, const AttnParams &p, int D);
// TMA map for the Q loads of packed tails (built per launch from p.q): the frame layout of Q
// with a box of tail_rows(block) rows, so each frame's tail lands in its own row group.
bool encode_q_tail_map(CUtensorMap *m, const AttnParams &p, int D);

// Launchers (return the launch error, if any).
// The eligibility check of every schedule slot before the forward's two launches: a
// unit with a row bound above p.elig_m is routed to the online-max launch; also
// clears the per-slot guard flags and counts n_online / n_bound (zeroed before).
// Launch a kernel that may start while the kernel before it on the stream is still running
// (programmatic dependent launch).  Every such kernel executes grid_dep_wait() before it reads
// or writes anything the previous kernel touches; launched after a memset or a copy, or on a
// device without the feature, it is ordered as an ordinary launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_after_kernel(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                                cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

cudaError_t launch_route(const AttnParams &p, cudaStream_t s);
cudaError_t launch_norms(const BoundsParams &p, int D, cudaStream_t s);
cudaError_t launch_rowbound(const BoundsParams &p, cudaStream_t s);
// kmax[bh, kb] from caller-supplied key norms knorm [B*H*L_kv] (p.q, p.k unused).
cudaError_t launch_kmax_from_norms(const BoundsParams &p, const float *knorm, cudaStream_t s);
int bounds_chunk_rows();

// Attention kernel for head dim D; grid = n_ctas persistent CTAs.
cudaError_t launch_attention_d64(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                                 const AttnParams &p, bool online, int n_ctas, cudaStream_t s);
cudaError_t launch_attention_d128(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                                  const AttnParams &p, bool online, int n_ctas, cudaStream_t s);
// Check the register count of both variants for head dim D and raise their dynamic
// shared-memory limit (an error if the compiled register count does not match the
// register split the kernel performs).
cudaError_t configure_attention_d64();
cudaError_t configure_attention_d128();

// TMA tensor maps of Q (3-D, frame-local boxes) and K, V (2-D) for a layout's shape;
// works for plan-only layouts too.  False if the driver entry point is missing or
// the driver rejects a map.
bool encode_layout_maps(const bsattn_layout_s *lay, const void *q, const void *k, const void *v, CUtensorMap *tq,
                        CUtensorMap *tk, CUtensorMap *tv);

}  // namespace bsv
