// Cauchy-Schwarz row bounds: the small table of precomputed norms that lets
// every query row know the largest logit it can reach before its softmax
// starts ("HeyGen Avatar IV on Trillium TPU" deep-dive, section
// 拿掉 softmax 的序列相依 / remove softmax's serial dependency;
// "Optimizing HeyGen's Avatar IV diffusion model for Google Cloud TPUs",
// section "How it works": an upper bound derived from vector norms).
//
//   qnorm[r]        = |q_r|
//   kmax[bh, kb]    = max over keys j of block kb of |k_j|
//   rowbound[r]     = (scale * qnorm[r]) * max over allowed kb of kmax[bh, kb]
//
// Norm rounding order (fixed, so results are reproducible bit for bit): the D
// elements of a row split into 16 contiguous chunks of D/16, one per lane of a
// 16-lane group; each lane accumulates fmaf(x, x, s) over its chunk in order;
// the 16 partial sums meet through an xor butterfly at distances 8, 4, 2, 1;
// then a correctly rounded square root.
//
// HBM-bound: Q and K are each read once with 16-byte (D=128) or 8-byte (D=64)
// coalesced loads; a 16-lane group covers one row, a warp two rows.  Q has L rows
// per head and K L_kv (more than L for a streamed chunk reading context frames).
#include "internal.h"
#include "ptx.cuh"

namespace bsv {

constexpr int kNormThreads = 256;
constexpr int kChunkRows = 256;  // rows of one frame block handled by one CTA

template <int PER>
__device__ __forceinline__ void load_chunk(const uint16_t *p, uint32_t (&w)[PER / 2]) {
    if constexpr (PER == 8) {
        const uint4 x = __ldg(reinterpret_cast<const uint4 *>(p));
        w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
    } else {
        const uint2 x = __ldg(reinterpret_cast<const uint2 *>(p));
        w[0] = x.x; w[1] = x.y;
    }
}

template <int PER>
__device__ __forceinline__ float chunk_sumsq(const uint32_t (&w)[PER / 2]) {
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < PER / 2; ++i) {
        const float a = __uint_as_float(w[i] << 16);          // element 2i (low half)
        const float b = __uint_as_float(w[i] & 0xFFFF0000u);  // element 2i+1
        s = __fmaf_rn(a, a, s);
        s = __fmaf_rn(b, b, s);
    }
    return s;
}

__device__ __forceinline__ float tree16(float s, unsigned mask) {
    s = __fadd_rn(s, __shfl_xor_sync(mask, s, 8));
    s = __fadd_rn(s, __shfl_xor_sync(mask, s, 4));
    s = __fadd_rn(s, __shfl_xor_sync(mask, s, 2));
    s = __fadd_rn(s, __shfl_xor_sync(mask, s, 1));
    return s;
}

// One CTA per row chunk of one key block kb: it folds the chunk's key norms into
// kmax[b, h, kb] and, when query block kb exists (kb < nb; a streamed chunk has
// fewer query than key blocks), writes the norms of the same rows of Q.
template <int D>
__global__ void __launch_bounds__(kNormThreads) norms_kernel(const BoundsParams p) {
    grid_dep_launch_next();  // the row-bound kernel may start launching
    constexpr int PER = D / 16;
    const int cpb = p.chunks_per_block;
    const int chunk = static_cast<int>(blockIdx.x % cpb);
    const int64_t seg = blockIdx.x / cpb;  // (b*H + h) * nbkv + kb
    const int kb = static_cast<int>(seg % p.nbkv);
    const int64_t bh = seg / p.nbkv;
    const bool has_q = kb < p.nb;
    const int64_t in_blk = static_cast<int64_t>(kb) * p.block + static_cast<int64_t>(chunk) * kChunkRows;
    const int64_t krow0 = bh * p.Lkv + in_blk;
    const int64_t qrow0 = bh * p.L + in_blk;
    const int nrows = min(kChunkRows, p.block - chunk * kChunkRows);  // a multiple of 16
    const int lane16 = threadIdx.x & 15;
    const int grp = threadIdx.x >> 4;
    const unsigned gmask = 0xFFFFu << (threadIdx.x & 16);

    float kmax = 0.0f;
    constexpr int U = 4;  // rows per group in flight
    for (int r = grp; r < nrows; r += 16 * U) {
        uint32_t wq[U][PER / 2], wk[U][PER / 2];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (r + 16 * u < nrows) {
                const int64_t off = static_cast<int64_t>(r + 16 * u) * D + lane16 * PER;
                if (has_q) load_chunk<PER>(p.q + qrow0 * D + off, wq[u]);
                load_chunk<PER>(p.k + krow0 * D + off, wk[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (r + 16 * u < nrows) {
                if (has_q) {
                    const float qn = __fsqrt_rn(tree16(chunk_sumsq<PER>(wq[u]), gmask));
                    if (lane16 == 0) p.qnorm[qrow0 + r + 16 * u] = qn;
                }
                const float kn = __fsqrt_rn(tree16(chunk_sumsq<PER>(wk[u]), gmask));
                kmax = kn > kmax ? kn : kmax;
            }
        }
    }
    // CTA max of the key norms, then one atomic per CTA (norms are >= 0, so the
    // unsigned order of the fp32 bit patterns is the numeric order).
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(0xFFFFFFFFu, kmax, off);
        kmax = o > kmax ? o : kmax;
    }
    __shared__ float warp_max[kNormThreads / 32];
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = kmax;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = warp_max[0];
#pragma unroll
        for (int w = 1; w < kNormThreads / 32; ++w) m = warp_max[w] > m ? warp_max[w] : m;
        atomicMax(p.kmax_bits + seg, __float_as_uint(m));
    }
}

__global__ void __launch_bounds__(kNormThreads) rowbound_kernel(const BoundsParams p) {
    grid_dep_wait();  // the norms and kmax of the kernel before are complete
    const int cpb = p.chunks_per_block;
    const int chunk = static_cast<int>(blockIdx.x % cpb);
    const int64_t seg = blockIdx.x / cpb;  // (b*H + h) * nb + qb
    const int qb = static_cast<int>(seg % p.nb);
    const int64_t bh = seg / p.nb;
    __shared__ float kB;
    if (threadIdx.x == 0) {
        const int sg = plan_segment(p.mask_heads, p.heads, p.nb, bh, qb);
        float m = 0.0f;
        for (int e = p.row_ptr[sg]; e < p.row_ptr[sg + 1]; ++e) {
            const float x = __uint_as_float(p.kmax_bits[bh * p.nbkv + p.col_idx[e]]);
            m = x > m ? x : m;
        }
        kB = m;
    }
    __syncthreads();
    const int nrows = min(kChunkRows, p.block - chunk * kChunkRows);
    if (static_cast<int>(threadIdx.x) < nrows) {
        const int64_t row = bh * p.L + static_cast<int64_t>(qb) * p.block +
                            static_cast<int64_t>(chunk) * kChunkRows + threadIdx.x;
        p.rowbound[row] = __fmul_rn(__fmul_rn(p.scale, p.qnorm[row]), kB);
    }
}

// kmax from per-token key norms that the caller's producer already wrote (its QK-norm
// or projection epilogue), so K is not read again: one CTA per row chunk of one key
// block, one norm per thread, one atomic max per CTA.  Negative and NaN entries lose
// every comparison against the running maximum, which starts at 0.
__global__ void __launch_bounds__(kNormThreads) kmax_from_norms_kernel(const BoundsParams p, const float *knorm) {
    grid_dep_launch_next();  // the row-bound kernel may start launching
    const int cpb = p.chunks_per_block;
    const int chunk = static_cast<int>(blockIdx.x % cpb);
    const int64_t seg = blockIdx.x / cpb;  // (b*H + h) * nbkv + kb
    const int kb = static_cast<int>(seg % p.nbkv);
    const int64_t bh = seg / p.nbkv;
    const int nrows = min(kChunkRows, p.block - chunk * kChunkRows);
    float m = 0.0f;
    if (static_cast<int>(threadIdx.x) < nrows) {
        const float x = __ldg(knorm + bh * p.Lkv + static_cast<int64_t>(kb) * p.block +
                              static_cast<int64_t>(chunk) * kChunkRows + threadIdx.x);
        m = x > m ? x : m;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(0xFFFFFFFFu, m, off);
        m = o > m ? o : m;
    }
    __shared__ float warp_max[kNormThreads / 32];
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float r = warp_max[0];
#pragma unroll
        for (int w = 1; w < kNormThreads / 32; ++w) r = warp_max[w] > r ? warp_max[w] : r;
        atomicMax(p.kmax_bits + seg, __float_as_uint(r));
    }
}

cudaError_t launch_kmax_from_norms(const BoundsParams &p, const float *knorm, cudaStream_t s) {
    const int64_t grid = static_cast<int64_t>(p.BH) * p.nbkv * p.chunks_per_block;
    kmax_from_norms_kernel<<<static_cast<unsigned>(grid), kNormThreads, 0, s>>>(p, knorm);
    return cudaGetLastError();
}

cudaError_t launch_norms(const BoundsParams &p, int D, cudaStream_t s) {
    const int64_t grid = static_cast<int64_t>(p.BH) * p.nbkv * p.chunks_per_block;  // nb <= nbkv
    if (D == 128)
        norms_kernel<128><<<static_cast<unsigned>(grid), kNormThreads, 0, s>>>(p);
    else
        norms_kernel<64><<<static_cast<unsigned>(grid), kNormThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_rowbound(const BoundsParams &p, cudaStream_t s) {
    const int64_t grid = static_cast<int64_t>(p.BH) * p.nb * p.chunks_per_block;
    return launch_after_kernel(rowbound_kernel, static_cast<unsigned>(grid), kNormThreads, 0, s, p);
}

int bounds_chunk_rows() { return kChunkRows; }

}  // namespace bsv
