// Frame-aligned block-sparse attention forward on sm_103a: a persistent,
// warp-specialised kernel with TMA-fed tcgen05 MMAs accumulating in TMEM.
//
// The method ("HeyGen Avatar IV on Trillium TPU" deep-dive, sections
// 把 block 縮到 16 and 拿掉 softmax 的序列相依; "How is HeyGen optimizing AI video
// on Google Cloud TPUs", section "Innovating Beyond Serial Dependencies"):
//   * query and key blocks are whole frames, a multiple of 16 tokens; the mask
//     says which key frames a query frame reads.  The allowed frames of a query
//     frame form runs of consecutive frames; each run is cut into key tiles of
//     128 keys plus one last tile of the remaining keys, itself a multiple of
//     16, so every tile is an exactly sized MMA (N = its width): no element
//     mask, no padding, and no tile reaches into a masked frame;
//   * the softmax shift of row i is its Cauchy-Schwarz bound m_i (precomputed),
//     so P = exp(scale*S - m_i) needs no running max and no rescaling of the
//     accumulator: every key tile is independent.
//
// One CTA per SM processes work units: a unit is one or two 128-row query tiles
// of the same frame (they share every K/V tile), looping over the frame's key
// tiles (under its head's own mask when the layout has one mask per head, found
// through plan_segment).  The host deals the units to the CTAs (slot k * gridDim + c is CTA c's
// k-th unit; empty slots have no query tiles and are skipped).  Query rows index
// Q and O over L tokens per head, keys index K and V over L_kv >= L (a streamed
// chunk reads context frames before its own).
//   warp 0      TMA producer: Q tiles, then a ring of STAGES K and V tiles.
//   warps 1, 2  MMA issuers (one thread each), one per query tile t = warp - 1:
//               S_t = Q_t K^T (A, B from smem) and O_t += P_t V (A = P_t from
//               TMEM, B = V from smem).  Two issuers keep one tile's MMAs from
//               queueing behind the other tile's issue loop.
//   warps 4-11  softmax and epilogue.  Warp w reads TMEM lanes 32*(w%4).. (its
//               rows) and column half h = (w-4)/4 of the key tile, so all eight
//               warps work on one query tile at a time: tile 0's softmax runs
//               while the tensor cores run tile 1's MMAs, and vice versa.  In
//               the epilogue each warp stages its 32 rows x 32 columns of O in
//               shared memory and one lane stores them with a TMA tensor store,
//               clipped at the frame edge by the Q/O frame layout.
// TMEM (512 columns): S_0/P_0 at column 0, S_1/P_1 at 128, O_0 at 256, O_1 at 384.
// P (bf16, two per 32-bit column) of key half h overwrites the first 32 of that
// half's 64 S columns: keys 64h + 2c, 64h + 2c + 1 sit in column 64h + c.
//
// Issuer t issues, per key tile j, PV_t(j) then S_t(j+1).  PV_t(j) comes in two
// parts: the k-steps of each half's first 32 keys once every softmax warp has
// stored that P (p_full), the rest with S_t(j+1) once all of P is stored
// (p_rest), so the first part overlaps the end of the softmax.  tcgen05 MMAs
// from one thread complete in issue order, so the commit that signals S_t(j+1)
// also guarantees that PV_t(j) has finished: O_t is stable whenever its softmax
// holds S_t (the online variant rescales it then).  Each K/V stage is released by
// both issuers (a tile absent from a unit still takes part, without MMAs).
//
// Every wait is bounded (a wall-clock limit, mbarriers only: no named barrier
// inside the loops); on expiry the CTA raises a shared abort flag and a device
// status bit, lets in-flight copies and MMAs land, frees its TMEM and returns.
#pragma once

#include "internal.h"
#include "ptx.cuh"

namespace bsv {

template <int D>
struct AttnCfg {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int N = kKvTile;                 // keys per full tile
    static constexpr int DH = D / 64;                 // 64-column (128-byte) halves of a row
    static constexpr int HALF_Q = kQTile * 128;       // bytes of one half of a Q tile
    static constexpr int Q_TILE = DH * HALF_Q;
    static constexpr int HALF_KV = N * 128;
    static constexpr int KV_TILE = DH * HALF_KV;
    static constexpr int SMEM_CAP = 232448;           // 227 KB per CTA
    static constexpr int BAR_BYTES = 512;             // mbarriers, TMEM slot, abort flag
    static constexpr int XCHG_BYTES = 2 * 2 * kQTile * 4;  // row exchange: [parity][half][row] fp32
    static constexpr int OST_BYTES = 8 * 2048;                       // O staging: 2 KB per softmax warp
    static constexpr int RESERVED = 1024 + BAR_BYTES + XCHG_BYTES + 1024 + OST_BYTES;  // + alignment slack
    static constexpr int STAGES_FIT = (SMEM_CAP - RESERVED - 2 * Q_TILE) / (2 * KV_TILE);
    static constexpr int STAGES = STAGES_FIT > 4 ? 4 : STAGES_FIT;
    static_assert(STAGES >= 2, "shared memory");
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = 2 * Q_TILE;
    static constexpr int OFF_V = OFF_K + STAGES * KV_TILE;
    static constexpr int OFF_BAR = OFF_V + STAGES * KV_TILE;
    static constexpr int OFF_XCHG = OFF_BAR + BAR_BYTES;
    static constexpr int OFF_OST = (OFF_XCHG + XCHG_BYTES + 1023) / 1024 * 1024;
    static constexpr int SMEM_USED = OFF_OST + OST_BYTES + 1024;
    // Above half of the SM's shared memory, so one CTA (and one TMEM owner) per SM.
    static constexpr int SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
    static_assert(SMEM <= SMEM_CAP, "shared memory");
    static constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 384;
    // QK^T descriptor without its N field (set per tile from the tile's width).
    static constexpr uint32_t IDESC_QK0 = idesc_bf16_f32(kQTile, 16, false, false) & ~(0x3Fu << 17);
    static constexpr uint32_t IDESC_PV = idesc_bf16_f32(kQTile, D, false, true);
};

// Barrier block layout (uint64 slots).
struct Bars {
    uint64_t *q_full, *q_empty, *s_full, *p_full, *p_rest, *o_full, *drain, *xbar;
    uint64_t *k_full, *k_empty, *v_full, *v_empty;
    uint32_t *tmem_slot;
    volatile int *abort;
    float *xchg;  // [2 parity][2 half][kQTile rows]
};

constexpr int kSoftmaxWarps = 8;
constexpr int kIssuers = 2;

template <int STAGES>
__device__ __forceinline__ Bars carve_bars(uint8_t *base, uint8_t *xchg) {
    uint64_t *b = reinterpret_cast<uint64_t *>(base);
    Bars r;
    r.q_full = b + 0;
    r.q_empty = b + 2;
    r.s_full = b + 4;
    r.p_full = b + 6;
    r.o_full = b + 8;
    r.drain = b + 10;
    r.xbar = b + 12;  // one per TMEM lane quarter
    r.p_rest = b + 16;
    r.k_full = b + 18;
    r.k_empty = r.k_full + STAGES;
    r.v_full = r.k_empty + STAGES;
    r.v_empty = r.v_full + STAGES;
    r.tmem_slot = reinterpret_cast<uint32_t *>(r.v_empty + STAGES);
    r.abort = reinterpret_cast<volatile int *>(r.tmem_slot + 1);
    r.xchg = reinterpret_cast<float *>(xchg);
    return r;
}

// Sequence position i of this launch -> schedule slot.  The fallback launch first walks
// the schedule (positions below `base`, where base = n_units when the route kernel sent
// units to it, else 0), then the guard's fallback list.
__device__ __forceinline__ int unit_index(const AttnParams &p, int i, int base) {
    return (p.mode == kModeFallback && i >= base) ? p.ws.fb_list[i - base] : i;
}

// Whether schedule position i is this launch's work: the bound launch takes the slots
// the route kernel left bound, the fallback launch the ones it routed online (and every
// fallback-list entry); the online-max-everywhere launch takes all.
__device__ __forceinline__ bool slot_for_launch(const AttnParams &p, int i, int base) {
    if (p.mode == kModeBound) return p.ws.slot_online[i] == 0;
    if (p.mode == kModeFallback && i < base) return p.ws.slot_online[i] != 0;
    return true;
}

// The work unit of slot i, checked (device checks on): false when the slot, the unit
// (head, query block, each query tile starting inside the frame), its key-tile range
// or any key tile it reads (16-aligned start, width 16..kKvTile, inside the head's
// L_kv keys) is out of range.  Reads only what the checks before it allowed.
__device__ __forceinline__ bool fetch_unit_checked(const AttnParams &p, int i, int base, int &u, int4 &U,
                                                   bool report) {
    bool ok = i >= 0 && (p.mode == kModeFallback ? i - base < p.n_units : i < p.n_units);
    if (ok) {
        u = unit_index(p, i, base);
        ok = u >= 0 && u < p.n_units;
    }
    if (ok) {
        U = p.units[u];
        ok = U.w >= -kMaxTailGroup && U.w <= 2 && U.w != -1;
        if (ok && U.w != 0) {
            if (U.w > 0)
                ok = U.x >= 0 && U.x < p.bh && U.y >= 0 && U.y < p.nb && U.z >= 0 &&
                     (static_cast<int64_t>(U.z) + U.w - 1) * kQTile < p.block;
            else  // packed tails: frames U.y .. U.y - U.w - 1, segment U.z past the (mask, frame) ones
                ok = U.x >= 0 && U.x < p.bh && U.y >= 0 && U.y - U.w <= p.nb &&
                     U.z >= p.mask_heads * p.nb && U.z < p.n_seg && -U.w * tail_rows(p.block) <= kQTile;
            if (ok) {
                const int sg = U.w > 0 ? plan_segment(p.mask_heads, p.heads, p.nb, U.x, U.y) : U.z;
                const int a = p.tile_ptr[sg], b = p.tile_ptr[sg + 1];
                ok = a >= 0 && a <= b && b <= p.n_tiles;
                for (int t = a; ok && t < b; ++t) {
                    int2 T = p.tiles[t];
                    // testing only: the CTA's first unit sees its first key tile past the last key
                    if (p.debug_plant && t == a && i == static_cast<int>(blockIdx.x)) T.x = static_cast<int>(p.Lkv);
                    const int tw = tile_width(T);
                    ok = T.x >= 0 && (T.x & 15) == 0 && tw >= 16 && tw <= kKvTile && (tw & 15) == 0 &&
                         static_cast<int64_t>(T.x) + tw <= p.Lkv &&
                         (U.w > 0 ? tile_row_groups(T) == 0 : tile_row_groups(T) < (1 << -U.w));
                }
            }
        }
    }
    if (!ok) {
        u = 0;
        U = make_int4(0, 0, 0, 0);
        if (report) atomicOr(p.ws.status, kStatusIndex);
    }
    return ok;
}

// The work unit at sequence position i of this launch.  False for a slot that is not
// this launch's work (slot_for_launch) and, with device checks on, for a unit the
// checks reject; the caller skips it.  Every role calls this with the same i, so all
// roles skip the same units; only the caller with `report` records the status bit.
__device__ __forceinline__ bool fetch_unit(const AttnParams &p, int i, int base, int &u, int4 &U, bool report) {
    // (slot_for_launch reads slot_online[i] only where i < n_units: the loops of every
    // role run i < n_units in the bound launch, and i < base = n_units for the schedule
    // part of the fallback launch)
    if (!slot_for_launch(p, i, base)) return false;
    if (p.checks) return fetch_unit_checked(p, i, base, u, U, report);
    u = unit_index(p, i, base);
    U = p.units[u];
    return true;
}

// Wait that ignores the abort flag: used only to let already-issued copies/MMAs land.
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity, uint64_t timeout_ns) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(a, parity)) {
        if (globaltimer_ns() - t0 > timeout_ns) break;
    }
}

// All 384 threads of the CTA (each warp converged) meet here.
__device__ __forceinline__ void cta_barrier() {
    __syncwarp();
    asm volatile("bar.sync 1, %0;" ::"n"(kAttnThreads) : "memory");
}

// ----------------------------------------------------------------------------------------------
// softmax of one column half of an S tile (one row per thread), P written back to TMEM as bf16

// Two logits -> two probabilities: P = 2^(S*c1 - m2) with c1 = scale*log2(e) and
// m2 = the row shift in log2 units; returns them as packed bf16 and adds the
// rounded values (the ones the P.V product uses) to the accumulators l0, l1.
__device__ __forceinline__ uint32_t softmax_pair(uint32_t s0, uint32_t s1, uint64_t c1x2, uint64_t nm2x2,
                                                 float &l0, float &l1) {
    float x0, x1;
    f2_split(f2_fma(f2_from_bits(s0, s1), c1x2, nm2x2), x0, x1);
    const uint32_t pk = pack_bf16x2(ex2_approx(x0), ex2_approx(x1));
    add_bf16x2_to(pk, l0, l1);
    return pk;
}

// S columns [tS, tS + w), w a multiple of 16 and at most 64, in buf: two TMEM loads of
// 32 columns, the second in flight while the first is converted -- or, with PRE, S is
// already in buf (loaded by load_half_max on the running-max path).  P of the first 32
// keys goes to columns [tS, tS + 16) and of the next 32 to [tS + 16, tS + 32): both
// were loaded by then, and a load in flight reads columns >= tS + 32.  mid() runs once
// the first group's P is stored (its P.V MMAs may then start), whatever w is.
template <bool PRE, typename Mid>
__device__ __forceinline__ void softmax_half(uint32_t tS, int w, uint64_t c1x2, uint64_t nm2x2, float (&l)[4],
                                             uint32_t (&buf)[2][32], Mid &&mid) {
    if (w <= 0) {
        mid();
        return;
    }
    if (!PRE) {
        if (w >= 32)
            tmem_ld32(tS, buf[0]);
        else
            tmem_ld16_into32(tS, buf[0]);
    }
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        if (32 * g < w) {
            const bool full = w - 32 * g >= 32;
            if (!PRE) {
                tmem_wait_ld();
                reg_fence32(buf[g]);
            }
            if (!PRE && g == 0 && w > 32) {
                if (w >= 64)
                    tmem_ld32(tS + 32, buf[1]);
                else
                    tmem_ld16_into32(tS + 32, buf[1]);
            }
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                pk[e] = softmax_pair(buf[g][2 * e], buf[g][2 * e + 1], c1x2, nm2x2, l[2 * (e & 1)],
                                     l[2 * (e & 1) + 1]);
            if (full) {
#pragma unroll
                for (int e = 8; e < 16; ++e)
                    pk[e] = softmax_pair(buf[g][2 * e], buf[g][2 * e + 1], c1x2, nm2x2, l[2 * (e & 1)],
                                         l[2 * (e & 1) + 1]);
                tmem_st16(tS + 16 * g, pk);
            } else {
                uint32_t hh[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) hh[e] = pk[e];
                tmem_st8(tS + 16 * g, hh);
            }
        }
        if (g == 0) mid();
    }
}

// For the running-max path: S columns [tS, tS + w) loaded once into buf (both groups
// of 32, the second possibly of 16) and their maximum returned (raw logits; -inf if
// w == 0); softmax_half<true> then converts the same registers.
__device__ __forceinline__ float load_half_max(uint32_t tS, int w, uint32_t (&buf)[2][32]) {
    float mx = -INFINITY;
    if (w <= 0) return mx;
    if (w >= 32)
        tmem_ld32(tS, buf[0]);
    else
        tmem_ld16_into32(tS, buf[0]);
    if (w >= 64)
        tmem_ld32(tS + 32, buf[1]);
    else if (w > 32)
        tmem_ld16_into32(tS + 32, buf[1]);
    tmem_wait_ld();
    reg_fence32(buf[0]);
    if (w > 32) reg_fence32(buf[1]);
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        if (32 * g < w) {
#pragma unroll
            for (int e = 0; e < 16; ++e) mx = fmaxf(mx, __uint_as_float(buf[g][e]));
            if (w - 32 * g >= 32) {
#pragma unroll
                for (int e = 16; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(buf[g][e]));
            }
        }
    }
    return mx;
}

// Multiply NC fp32 columns of one row of the O accumulator by alpha (warp-collective).
template <int NC>
__device__ __forceinline__ void rescale_o_cols(uint32_t tO, float alpha) {
    const uint64_t a2 = f2_make(alpha, alpha);
#pragma unroll
    for (int c = 0; c < NC / 32; ++c) {
        uint32_t a[32];
        tmem_ld32(tO + c * 32, a);
        tmem_wait_ld();
        reg_fence32(a);
        uint32_t r0[16], r1[16];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float x0, x1;
            f2_split(f2_mul(f2_from_bits(a[2 * e], a[2 * e + 1]), a2), x0, x1);
            r0[2 * e] = __float_as_uint(x0);
            r0[2 * e + 1] = __float_as_uint(x1);
            f2_split(f2_mul(f2_from_bits(a[16 + 2 * e], a[16 + 2 * e + 1]), a2), x0, x1);
            r1[2 * e] = __float_as_uint(x0);
            r1[2 * e + 1] = __float_as_uint(x1);
        }
        tmem_st16(tO + c * 32, r0);
        tmem_st16(tO + c * 32 + 16, r1);
    }
    tmem_wait_st();
}

// The two warps that own the same rows (same TMEM lane quarter q, column halves 0 and
// 1) swap one fp32 value per row through shared memory.  The slot alternates with the
// parity of the exchange count, which both warps advance together; a warp can reach
// exchange n + 2 only after its partner has arrived at n + 1, i.e. after the partner
// has read slot n.  Returns false if the bounded wait gave up.
__device__ __forceinline__ bool pair_exchange(const Bars &bar, int q, int h, int r, uint32_t &uses, float mine,
                                              float &other, int *status, uint64_t tmo) {
    const uint32_t par = uses & 1;
    float *slot = bar.xchg + par * (2 * kQTile);
    slot[h * kQTile + r] = mine;
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar.xbar + q);
    bool ok = mbar_wait(bar.xbar + q, par, bar.abort, status, kStatusTimeout, tmo);
    ok = __all_sync(0xFFFFFFFFu, ok);
    ++uses;
    other = slot[(1 - h) * kQTile + r];
    return ok;
}

// ----------------------------------------------------------------------------------------------

template <int D, bool ONLINE>
__global__ void __launch_bounds__(kAttnThreads, 1)
    bsattn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                      const __grid_constant__ CUtensorMap tm_qt, const AttnParams p) {
    using C = AttnCfg<D>;
    // Launched as soon as the kernel before it on the stream (the eligibility check, or the bound
    // launch for the online one) lets it: wait for that kernel's results before reading anything.
    grid_dep_wait();
    grid_dep_launch_next();
    // Positions of this launch: the bound launch walks the schedule unless the route kernel
    // sent every unit online; the fallback launch walks the schedule when it sent some
    // (base = n_units), then the guard's fallback list.
    int n_seq = p.n_units, base = 0;
    if (p.mode == kModeBound) {
        if (*reinterpret_cast<volatile int32_t *>(p.ws.n_bound) == 0) n_seq = 0;
    } else if (p.mode == kModeFallback) {
        base = *reinterpret_cast<volatile int32_t *>(p.ws.n_online) > 0 ? p.n_units : 0;
        n_seq = base + *reinterpret_cast<volatile int32_t *>(p.ws.fb_count);
    }
    if (static_cast<int>(blockIdx.x) >= n_seq) return;  // nothing to do: exit before any TMEM allocation

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars bar = carve_bars<C::STAGES>(smem + C::OFF_BAR, smem + C::OFF_XCHG);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar.q_full + t, 1);
            mbar_init(bar.q_empty + t, 1);
            mbar_init(bar.s_full + t, 1);
            mbar_init(bar.p_full + t, kSoftmaxWarps);
            mbar_init(bar.p_rest + t, kSoftmaxWarps);
            mbar_init(bar.o_full + t, 1);
            mbar_init(bar.drain + t, 1);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) mbar_init(bar.xbar + q, 2);
#pragma unroll
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(bar.k_full + s, 1);
            mbar_init(bar.k_empty + s, kIssuers);
            mbar_init(bar.v_full + s, 1);
            mbar_init(bar.v_empty + s, kIssuers);
        }
        *bar.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(bar.tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *bar.tmem_slot;
    int *status = p.ws.status;
    const uint64_t tmo = p.timeout_ns;

    // Registers move from the TMA/MMA warpgroup to the two softmax warpgroups.  The
    // CTA launches with kLaunchRegs per thread (checked on the host before any launch)
    // and 128 * kRegsLow + 256 * kRegsHigh <= 384 * kLaunchRegs.  Each role keeps its
    // own branch to the end, where all threads meet at a named barrier.
    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------------------ TMA producer
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            const uint64_t pol_kv = policy_evict_last();
            const uint64_t pol_q = policy_evict_first();
            uint32_t q_uses0 = 0, q_uses1 = 0;
            uint32_t g = 0;           // key tiles started by this CTA
            uint32_t gk = 0, gv = 0;  // K / V copies issued
            bool ok = true;
            for (int i = blockIdx.x; i < n_seq && ok; i += gridDim.x) {
                int u;
                int4 U;
                if (!fetch_unit(p, i, base, u, U, true)) continue;  // not this launch's, or rejected by the checks
                if (U.w == 0) continue;  // an empty schedule slot
                const bool tail = U.w < 0;
                const int sg = tail ? U.z : plan_segment(p.mask_heads, p.heads, p.nb, U.x, U.y);
                const int t0 = p.tile_ptr[sg], nkv = p.tile_ptr[sg + 1] - t0;
                if (nkv == 0) continue;  // reads nothing
                // testing only: the first unit's query tiles are never loaded, so the
                // issuers' bounded waits run out and the CTA aborts and returns
                const int n_q = (p.debug_stall && i == static_cast<int>(blockIdx.x)) ? 0 : (tail ? 1 : U.w);
                for (int t = 0; t < n_q && ok; ++t) {
                    uint32_t &qu = t ? q_uses1 : q_uses0;
                    ok = mbar_wait(bar.q_empty + t, (qu & 1) ^ 1, bar.abort, status, kStatusTimeout, tmo);
                    if (!ok) break;
                    ++qu;
                    if (tail) {
                        // packed tails: row group g holds the tail rows of frame U.y + g; rows past
                        // the last group keep stale data, which the softmax gives P = 0
                        const int tr = tail_rows(p.block);
                        mbar_arrive_expect_tx(bar.q_full, -U.w * tr * 128 * C::DH);
                        for (int gq = 0; gq < -U.w; ++gq)
#pragma unroll
                            for (int h = 0; h < C::DH; ++h)
                                tma_load_3d(smem + C::OFF_Q + h * C::HALF_Q + gq * tr * 128, &tm_qt, h * 64,
                                            tail_row0(p.block), U.x * p.nb + U.y + gq, bar.q_full, pol_q);
                    } else {
                        mbar_arrive_expect_tx(bar.q_full + t, C::Q_TILE);
#pragma unroll
                        for (int h = 0; h < C::DH; ++h)
                            tma_load_3d(smem + C::OFF_Q + t * C::Q_TILE + h * C::HALF_Q, &tm_q, h * 64,
                                        (U.z + t) * kQTile, U.x * p.nb + U.y, bar.q_full + t, pol_q);
                    }
                }
                for (int j = 0; j < nkv && ok; ++j, ++g) {
                    const int row = static_cast<int>(static_cast<int64_t>(U.x) * p.Lkv) + p.tiles[t0 + j].x;
                    const int s = static_cast<int>(g % C::STAGES);
                    const uint32_t ph = (g / C::STAGES) & 1;
                    ok = mbar_wait(bar.k_empty + s, ph ^ 1, bar.abort, status, kStatusTimeout, tmo);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar.k_full + s, C::KV_TILE);
#pragma unroll
                    for (int h = 0; h < C::DH; ++h)
                        tma_load_2d(smem + C::OFF_K + s * C::KV_TILE + h * C::HALF_KV, &tm_k, h * 64, row,
                                    bar.k_full + s, pol_kv);
                    ++gk;
                    ok = mbar_wait(bar.v_empty + s, ph ^ 1, bar.abort, status, kStatusTimeout, tmo);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar.v_full + s, C::KV_TILE);
#pragma unroll
                    for (int h = 0; h < C::DH; ++h)
                        tma_load_2d(smem + C::OFF_V + s * C::KV_TILE + h * C::HALF_KV, &tm_v, h * 64, row,
                                    bar.v_full + s, pol_kv);
                    ++gv;
                }
            }
            if (!ok) {
                // Let every copy already issued land before the CTA's shared memory goes away.
                if (q_uses0) mbar_drain(bar.q_full + 0, (q_uses0 - 1) & 1, tmo);
                if (q_uses1) mbar_drain(bar.q_full + 1, (q_uses1 - 1) & 1, tmo);
                for (uint32_t x = (gk > C::STAGES ? gk - C::STAGES : 0); x < gk; ++x)
                    mbar_drain(bar.k_full + x % C::STAGES, (x / C::STAGES) & 1, tmo);
                for (uint32_t x = (gv > C::STAGES ? gv - C::STAGES : 0); x < gv; ++x)
                    mbar_drain(bar.v_full + x % C::STAGES, (x / C::STAGES) & 1, tmo);
            }
        } else if ((warp == 1 || warp == 2) && lane == 0) {
            // ------------------------------------------------------------ MMA issuer of query tile t
            const int t = warp - 1;
            const uint32_t dS = tmem + (t ? C::COL_S1 : C::COL_S0);
            const uint32_t dO = tmem + (t ? C::COL_O1 : C::COL_O0);
            // Descriptors of the first stage; a byte offset X adds X >> 4 to the start
            // address field (shared addresses stay below 2^18, so the field never carries).
            const uint64_t q_desc = smem_desc_sw128(smem_u32(smem + C::OFF_Q + t * C::Q_TILE), 16, 1024);
            const uint64_t k_desc = smem_desc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);
            const uint64_t v_desc = smem_desc_sw128(smem_u32(smem + C::OFF_V), C::HALF_KV, 1024);
            // S_t = Q_t K^T over the first w keys of stage s (N = w in the instruction).
            auto issue_qk = [&](int s, int w) {
                const uint32_t idesc = C::IDESC_QK0 | (static_cast<uint32_t>(w >> 3) << 17);
                const uint64_t kd = k_desc + static_cast<uint64_t>((s * C::KV_TILE) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t qo = ((kk >> 2) * C::HALF_Q + (kk & 3) * 32) >> 4;
                    const uint32_t ko = ((kk >> 2) * C::HALF_KV + (kk & 3) * 32) >> 4;
                    mma_ss(dS, q_desc + qo, kd + ko, idesc, kk > 0 ? 1u : 0u);
                }
            };
            // O_t += P_t V over the first w keys (K = w, in steps of 16); the P of keys
            // 16kk .. 16kk+15 sits in S columns 64*(kk/4) + 8*(kk%4) .. +8.  part 0 issues
            // the k-steps of each half's first 32 keys (kk % 4 < 2), part 1 the rest.
            auto issue_pv = [&](int s, int w, bool acc, int part) {
                const uint64_t vd = v_desc + static_cast<uint64_t>((s * C::KV_TILE) >> 4);
#pragma unroll
                for (int kk = 0; kk < kKvTile / 16; ++kk) {
                    if (((kk >> 1) & 1) == part && 16 * kk < w)
                        mma_ts(dO, dS + 64 * (kk >> 2) + 8 * (kk & 3), vd + ((kk * 16 * 128) >> 4), C::IDESC_PV,
                               (acc || part > 0 || kk > 0) ? 1u : 0u);
                }
            };
            uint32_t q_uses = 0, p_uses = 0;
            uint32_t g = 0;
            bool ok = true;
            for (int i = blockIdx.x; i < n_seq && ok; i += gridDim.x) {
                int u;
                int4 U;
                if (!fetch_unit(p, i, base, u, U, false)) continue;  // not this launch's, or rejected by the checks
                if (U.w == 0) continue;  // an empty schedule slot
                const int sg = U.w < 0 ? U.z : plan_segment(p.mask_heads, p.heads, p.nb, U.x, U.y);
                const int t0 = p.tile_ptr[sg], nkv = p.tile_ptr[sg + 1] - t0;
                if (nkv == 0) continue;  // reads nothing
                if (t >= (U.w < 0 ? 1 : U.w)) {
                    // This query tile is absent from the unit: release each stage without MMAs,
                    // after its copy has landed (so the arrival counts toward the right phase).
                    for (int j = 0; j < nkv && ok; ++j) {
                        const uint32_t gj = g + j;
                        const int sj = static_cast<int>(gj % C::STAGES);
                        const uint32_t ph = (gj / C::STAGES) & 1;
                        ok = mbar_wait(bar.k_full + sj, ph, bar.abort, status, kStatusTimeout, tmo);
                        if (!ok) break;
                        mbar_arrive(bar.k_empty + sj);
                        ok = mbar_wait(bar.v_full + sj, ph, bar.abort, status, kStatusTimeout, tmo);
                        if (!ok) break;
                        mbar_arrive(bar.v_empty + sj);
                    }
                    g += nkv;
                    continue;
                }
                ok = mbar_wait(bar.q_full + t, q_uses & 1, bar.abort, status, kStatusTimeout, tmo);
                ++q_uses;
                if (!ok) break;
                int w_next = tile_width(p.tiles[t0]);
                {
                    const int s0 = static_cast<int>(g % C::STAGES);
                    ok = mbar_wait(bar.k_full + s0, (g / C::STAGES) & 1, bar.abort, status, kStatusTimeout, tmo);
                    if (!ok) break;
                    tc_fence_after();
                    issue_qk(s0, w_next);
                    mma_commit(bar.s_full + t);
                    if (nkv == 1) mma_commit(bar.q_empty + t);
                    mma_commit(bar.k_empty + s0);
                }
                for (int j = 0; j < nkv && ok; ++j) {
                    const uint32_t gj = g + j, gn = g + j + 1;
                    const int sj = static_cast<int>(gj % C::STAGES), sn = static_cast<int>(gn % C::STAGES);
                    const bool more = j + 1 < nkv;
                    const int wj = w_next;
                    if (more) w_next = tile_width(p.tiles[t0 + j + 1]);
                    ok = mbar_wait(bar.v_full + sj, (gj / C::STAGES) & 1, bar.abort, status, kStatusTimeout, tmo);
                    if (ok && more)
                        ok = mbar_wait(bar.k_full + sn, (gn / C::STAGES) & 1, bar.abort, status, kStatusTimeout,
                                       tmo);
                    if (ok) ok = mbar_wait(bar.p_full + t, p_uses & 1, bar.abort, status, kStatusTimeout, tmo);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv(sj, wj, j > 0, 0);
                    ok = mbar_wait(bar.p_rest + t, p_uses & 1, bar.abort, status, kStatusTimeout, tmo);
                    if (!ok) break;
                    ++p_uses;
                    tc_fence_after();
                    issue_pv(sj, wj, j > 0, 1);
                    if (more) {
                        issue_qk(sn, w_next);
                        mma_commit(bar.s_full + t);
                        if (j + 2 == nkv) mma_commit(bar.q_empty + t);
                    } else {
                        mma_commit(bar.o_full + t);
                    }
                    mma_commit(bar.v_empty + sj);
                    if (more) mma_commit(bar.k_empty + sn);
                }
                g += nkv;
            }
            // Every MMA issued must complete before TMEM is freed.
            mma_commit(bar.drain + t);
            mbar_drain(bar.drain + t, 0, tmo);
        }
        tc_fence_before();
        cta_barrier();
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem, 512);
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
        // ---------------------------------------------------------------- softmax + epilogue
        constexpr int DC = D / 2;        // O columns of one half
        const int q = warp & 3;          // TMEM lane quarter: rows 32q .. 32q+31
        const int h = (warp - 4) >> 2;   // key / O column half
        const int r = q * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t tS0 = tmem + lane_base + C::COL_S0 + 64 * h;
        const uint32_t tS1 = tmem + lane_base + C::COL_S1 + 64 * h;
        const uint32_t tO0 = tmem + lane_base + C::COL_O0 + DC * h;
        const uint32_t tO1 = tmem + lane_base + C::COL_O1 + DC * h;
        const float c1 = p.scale_log2;
        const uint64_t c1x2 = f2_make(c1, c1);
        uint8_t *ost = smem + C::OFF_OST + (warp - 4) * 2048;  // this warp's O staging (32 rows x 64 B)
        bool ost_busy = false;
        uint32_t s_uses0 = 0, s_uses1 = 0, o_uses0 = 0, o_uses1 = 0, x_uses = 0;
        bool ok = true;
        for (int i = blockIdx.x; i < n_seq && ok; i += gridDim.x) {
            int u;
            int4 U;
            if (!fetch_unit(p, i, base, u, U, false)) continue;  // not this launch's, or rejected by the checks
            if (U.w == 0) continue;  // an empty schedule slot
            const bool tail = U.w < 0;
            const int nt = tail ? 1 : U.w;
            const int sg = tail ? U.z : plan_segment(p.mask_heads, p.heads, p.nb, U.x, U.y);
            const int t0 = p.tile_ptr[sg], nkv = p.tile_ptr[sg + 1] - t0;
            // This thread's row of tile 0.  Packed tails: row r is in row group r / tail_rows,
            // the tail of frame U.y + group; rowbit marks its group in the key tiles' masks
            // (rows past the last group match no mask and keep P = 0 on every tile).
            int64_t row0;
            bool valid0, valid1;
            uint32_t rowbit = 0;
            if (tail) {
                const int tr = tail_rows(p.block), grp = r / tr;
                valid0 = grp < -U.w;
                valid1 = false;
                rowbit = valid0 ? 1u << grp : 0u;
                row0 = static_cast<int64_t>(U.x) * p.L + static_cast<int64_t>(U.y + grp) * p.block + tail_row0(p.block) +
                       (r - grp * tr);
            } else {
                row0 = static_cast<int64_t>(U.x) * p.L + static_cast<int64_t>(U.y) * p.block +
                       static_cast<int64_t>(U.z) * kQTile + r;
                valid0 = r < min(kQTile, p.block - U.z * kQTile);
                valid1 = nt > 1 && r < min(kQTile, p.block - (U.z + 1) * kQTile);
            }
            if (nkv == 0) {  // the frame reads no key block: O = 0, LSE = -inf
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (t < nt && (t ? valid1 : valid0)) {
                        const int64_t grow = row0 + t * kQTile;
                        uint4 *dst = reinterpret_cast<uint4 *>(p.o + grow * D + DC * h);
#pragma unroll
                        for (int c = 0; c < DC / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
                        if (p.lse && h == 0) p.lse[grow] = -INFINITY;
                    }
                }
                continue;
            }
            // mrow: the bound m_i (natural units) on the bound path; the running max (log2
            // units) on the online path.  The route kernel sent every unit with a row above
            // the eligibility limit to the online launch, so each kernel has one path.
            float mrow0, mrow1;
            if constexpr (ONLINE) {
                mrow0 = mrow1 = -INFINITY;
            } else {
                mrow0 = valid0 ? p.rowbound[row0] : 0.0f;
                mrow1 = valid1 ? p.rowbound[row0 + kQTile] : 0.0f;
            }
            uint64_t nm0 = f2_make(-mrow0 * 1.4426950408889634f, -mrow0 * 1.4426950408889634f);
            uint64_t nm1 = f2_make(-mrow1 * 1.4426950408889634f, -mrow1 * 1.4426950408889634f);
            // row-sum accumulators: key 4i + k of a half goes to lt[k]
            float lt0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, lt1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            const uint64_t ninf2 = f2_make(-INFINITY, -INFINITY);
            for (int j = 0; j < nkv && ok; ++j) {
                const int2 T = p.tiles[t0 + j];
                const int w = tile_width(T);
                const int wh = max(0, min(64, w - 64 * h));
                // packed tails: a row whose frame may not read this key tile gets a shift of -inf
                // for it (P = 0, and no effect on its running max)
                const bool allowed = !tail || (static_cast<uint32_t>(tile_row_groups(T)) & rowbit) != 0;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (t >= nt) break;
                    uint32_t &su = t ? s_uses1 : s_uses0;
                    ok = mbar_wait(bar.s_full + t, su & 1, bar.abort, status, kStatusTimeout, tmo);
                    ok = __all_sync(0xFFFFFFFFu, ok);
                    if (!ok) break;
                    ++su;
                    tc_fence_after();
                    const uint32_t tS = t ? tS1 : tS0;
                    float(&lt)[4] = t ? lt1 : lt0;
                    uint64_t &nm = t ? nm1 : nm0;
                    // S of this half: loaded here for the running max (and kept for P), or by
                    // softmax_half on the bound path.
                    uint32_t sbuf[2][32];
                    if constexpr (ONLINE) {
                        float &mrow = t ? mrow1 : mrow0;
                        float other;
                        float mine = load_half_max(tS, wh, sbuf) * c1;  // warp-collective load
                        if (!allowed) mine = -INFINITY;
                        ok = pair_exchange(bar, q, h, r, x_uses, mine, other, status, tmo);
                        if (!ok) break;
                        const float mx = fmaxf(mine, other);
                        if (j == 0) {
                            mrow = mx;
                        } else {
                            // Rescale only when the max grew by more than 2^8: a stale max
                            // keeps P <= 2^8, exact in fp32 and bf16.
                            const bool need = mx > mrow + 8.0f;
                            if (__any_sync(0xFFFFFFFFu, need)) {
                                const float alpha = need ? ex2_approx(mrow - mx) : 1.0f;
                                if (need) mrow = mx;
#pragma unroll
                                for (int k = 0; k < 4; ++k) lt[k] *= alpha;
                                rescale_o_cols<DC>(t ? tO1 : tO0, alpha);
                            }
                        }
                        nm = f2_make(-mrow, -mrow);
                    }
                    // p_full[t]: the P of every warp's first 32 keys is stored (P.V k-steps 0, 1,
                    // 4, 5 may start); p_rest[t]: all of it is.
                    const auto handoff = [&]() {
                        tmem_wait_st();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar.p_full + t);
                    };
                    softmax_half<ONLINE>(tS, wh, c1x2, allowed ? nm : ninf2, lt, sbuf, handoff);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar.p_rest + t);
                }
            }
            if (!ok) break;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (t >= nt) break;
                uint32_t &ou = t ? o_uses1 : o_uses0;
                ok = mbar_wait(bar.o_full + t, ou & 1, bar.abort, status, kStatusTimeout, tmo);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) break;
                ++ou;
                tc_fence_after();
                const float(&lt)[4] = t ? lt1 : lt0;
                const float mine = (lt[0] + lt[1]) + (lt[2] + lt[3]);
                float other;
                ok = pair_exchange(bar, q, h, r, x_uses, mine, other, status, tmo);
                if (!ok) break;
                const float l = h == 0 ? mine + other : other + mine;  // half 0 + half 1, in that order
                const float inv = l > 0.0f ? 1.0f / l : 0.0f;
                const uint64_t inv2 = f2_make(inv, inv);
                const bool valid = t ? valid1 : valid0;
                const int64_t grow = row0 + t * kQTile;
                const uint32_t tO = t ? tO1 : tO0;
                // O rows of this warp go out as 32-row boxes of a 3-D (D, frame rows, frames) map:
                // a box running past the frame's last row is clipped there, one starting past it
                // is not issued.  y0: the box's first row in the frame.
                const int y0 = (U.z + t) * kQTile + q * 32;
#pragma unroll
                for (int c = 0; c < DC / 32; ++c) {
                    uint32_t a[32];
                    tmem_ld32(tO + c * 32, a);
                    tmem_wait_ld();
                    reg_fence32(a);
                    uint32_t wv[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float x0, x1;
                        f2_split(f2_mul(f2_from_bits(a[2 * e], a[2 * e + 1]), inv2), x0, x1);
                        wv[e] = pack_bf16x2(x0, x1);
                    }
                    if (tail) {  // packed tails: this warp's rows lie in several frames
                        if (valid) {
                            uint4 *dst = reinterpret_cast<uint4 *>(p.o + grow * D + DC * h + 32 * c);
                            dst[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                            dst[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
                            dst[2] = make_uint4(wv[8], wv[9], wv[10], wv[11]);
                            dst[3] = make_uint4(wv[12], wv[13], wv[14], wv[15]);
                        }
                        continue;
                    }
                    if (ost_busy) {  // the previous store must have read the staging buffer
                        if (lane == 0) bulk_wait_read0();
                        __syncwarp();
                    }
                    // row = lane, 64 B per row, 16-byte chunk k at (k ^ ((row >> 1) & 3)) (64-byte swizzle)
                    uint8_t *rowp = ost + lane * 64;
                    const int sw = (lane >> 1) & 3;
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        *reinterpret_cast<uint4 *>(rowp + ((k ^ sw) << 4)) =
                            make_uint4(wv[4 * k], wv[4 * k + 1], wv[4 * k + 2], wv[4 * k + 3]);
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0 && y0 < p.block) {
                        tma_store_3d(&tm_o, DC * h + 32 * c, y0, U.x * p.nb + U.y, ost);
                        bulk_commit();
                    }
                    ost_busy = true;
                }
                if (h == 0) {
                    const float mrow = t ? mrow1 : mrow0;
                    if (valid && p.lse) {
                        if constexpr (ONLINE)
                            p.lse[grow] = (mrow + log2f(l)) * 0.6931471805599453f;
                        else
                            p.lse[grow] = mrow + logf(l);
                    }
                    if constexpr (!ONLINE) {
                        if (p.mode == kModeBound) {
                            // Underflow guard: a denominator below 2^-64 (or not finite) means the
                            // bound was too loose for exp to resolve this row; rerun its unit with
                            // the online max.
                            const bool bad = valid && !(l >= kGuardTau && l <= 3.402823466e38f);
                            const unsigned ballot = __ballot_sync(0xFFFFFFFFu, bad);
                            if (ballot && lane == 0) {
                                atomicAdd(p.ws.fb_rows, __popc(ballot));
                                if (atomicExch(p.ws.unit_flag + u, 1) == 0) {
                                    const int pos = atomicAdd(p.ws.fb_count, 1);
                                    p.ws.fb_list[pos] = u;
                                }
                            }
                        }
                    }
                }
            }
        }
        if (lane == 0) bulk_wait0();  // the last stores are complete (and their staging read)
        __syncwarp();
        tc_fence_before();
        cta_barrier();
    }
}

template <int D, bool ONLINE>
cudaError_t launch_fwd_instance(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                                const AttnParams &p, int n_ctas, cudaStream_t s) {
    CUtensorMap to, tqt;
    if (!encode_o_store_map(&to, p, D) || !encode_q_tail_map(&tqt, p, D)) return cudaErrorInvalidValue;
    return launch_after_kernel(bsattn_fwd_kernel<D, ONLINE>, static_cast<unsigned>(n_ctas), kAttnThreads,
                               AttnCfg<D>::SMEM, s, tq, tk, tv, to, tqt, p);
}

// The register split in the kernel is valid only if it launches with exactly
// kLaunchRegs registers per thread; refuse to configure (and so to run) otherwise.
template <int D, bool ONLINE>
cudaError_t configure_one() {
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, bsattn_fwd_kernel<D, ONLINE>);
    if (e != cudaSuccess) return e;
    if ((a.numRegs + 7) / 8 * 8 != kLaunchRegs) return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(bsattn_fwd_kernel<D, ONLINE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                AttnCfg<D>::SMEM);
}

template <int D>
cudaError_t configure_instance() {
    cudaError_t e = configure_one<D, false>();
    return e != cudaSuccess ? e : configure_one<D, true>();
}

}  // namespace bsv
