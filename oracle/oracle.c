/*
 * oracle.c -- plain, slow, fp64 CPU oracle for frame-aligned block-sparse
 * attention.  TEST INFRASTRUCTURE ONLY: it is linked by nothing but the tests,
 * the bench's CPU-baseline leg and the smoke check.  It shares no code, header
 * or table with the CUDA library.
 *
 * Sources (web pages about HeyGen's Avatar IV port to Trillium TPUs):
 *   [deep-dive]   "HeyGen Avatar IV on Trillium TPU" deep-dive (vatt-ghern.pages.dev), sections
 *                 "把 block 縮到 16" (shrink the block to 16) and
 *                 "拿掉 softmax 的序列相依" (remove softmax's serial dependency);
 *   [bytechap]    "Optimizing HeyGen's Avatar IV diffusion model for Google Cloud TPUs", section
 *                 "How it works";
 *   [cloudcurated] "How is HeyGen optimizing AI video on Google Cloud TPUs", section
 *                 "Innovating Beyond Serial Dependencies".
 *
 * What the method computes, read from those sections:
 *   - attention whose block mask, at frame granularity, says which key/value
 *     blocks each query block reads; blocks coincide with frame edges, so no
 *     element-level predicate exists ([deep-dive] shrink the block to 16;
 *     [bytechap] How it works);
 *   - a softmax whose shift is a per-row upper bound on the logits, made from
 *     the query norm times the largest key norm (Cauchy-Schwarz), so no running
 *     max is needed ([deep-dive] remove softmax's serial dependency;
 *     [cloudcurated] Innovating Beyond Serial Dependencies).
 * Softmax is shift-invariant, so the method reaches exactly (up to rounding)
 * masked softmax attention.  The oracle is that definition written out, with
 * the textbook max shift, in fp64 (orc_attention with shift == NULL).
 *
 * Conventions: q is bf16 bit patterns (uint16) laid out [B,H,Lq,D], k and v
 * [B,H,Lkv,D]; Lq = nbq * bs, Lkv = nbkv * bs; query row i of head (b,h) lies in
 * block i / bs, key j in block j / bs.  mask is uint8 [nbq, nbkv] row-major,
 * mask[qb*nbkv + kb] != 0 means query block qb reads key block kb; one mask
 * serves every batch and head.  Self-attention over one chunk is Lq = Lkv; a
 * streamed chunk whose queries read earlier context frames as well as the chunk
 * ("HeyGen Avatar IV on Trillium TPU" deep-dive, opening section: the output is
 * streamed chunk by chunk) has Lkv > Lq.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static inline double bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* ----------------------------------------------------------------------------
 * The allowed key blocks of each query block, A(qb) = { kb : mask[qb,kb] != 0 },
 * in ascending kb order, as CSR (row_ptr[nb+1], col_idx[nnz]).  Returns nnz.
 * ([deep-dive] shrink the block to 16: the mask is decided per block.)
 */
int32_t orc_allowed_csr(int32_t nbq, int32_t nbkv, const uint8_t *mask, int32_t *row_ptr, int32_t *col_idx) {
    int32_t nnz = 0;
    row_ptr[0] = 0;
    for (int32_t qb = 0; qb < nbq; ++qb) {
        for (int32_t kb = 0; kb < nbkv; ++kb)
            if (mask[(int64_t)qb * nbkv + kb]) col_idx[nnz++] = kb;
        row_ptr[qb + 1] = nnz;
    }
    return nnz;
}

/* ----------------------------------------------------------------------------
 * Masked softmax attention in fp64, for a list of query rows.
 *
 *   S_ij  = scale * sum_d q_id k_jd           for keys j whose block is allowed
 *   c_i   = shift_i if given, else max_j S_ij (the textbook max shift)
 *   l_i   = sum_j exp(S_ij - c_i)
 *   O_i   = sum_j exp(S_ij - c_i) v_j / l_i
 *   LSE_i = c_i + ln l_i
 * A row with no allowed key gets O_i = 0, LSE_i = -inf, l_i = 0.
 *
 * rows: global query row ids r = (b*H + h)*Lq + i (NULL: all B*H*Lq rows, in order).
 * shift: per listed row (NULL: max shift).  Given the Cauchy-Schwarz bound as
 * the shift this is the method's own formulation ([deep-dive] remove softmax's
 * serial dependency); both give the same O up to rounding.
 * out: nrows x D; lse, lsum: nrows (nullable).
 */
typedef struct {
    int32_t H, D, bs, nbkv;
    int64_t Lq, Lkv;
    const uint8_t *mask;
    const uint16_t *q, *k, *v;
    double scale;
    const int64_t *rows;
    const double *shift;
    double *out, *lse, *lsum;
    int64_t r0, r1;
} attn_job_t;

static void attn_rows(const attn_job_t *J) {
    const int32_t D = J->D, bs = J->bs, nbkv = J->nbkv;
    const int64_t Lq = J->Lq, Lkv = J->Lkv;
    double *S = (double *)malloc(sizeof(double) * (size_t)(Lkv > 0 ? Lkv : 1));
    int64_t *key = (int64_t *)malloc(sizeof(int64_t) * (size_t)(Lkv > 0 ? Lkv : 1));
    double *qv = (double *)malloc(sizeof(double) * (size_t)D);
    double *acc = (double *)malloc(sizeof(double) * (size_t)D);
    for (int64_t r = J->r0; r < J->r1; ++r) {
        const int64_t row = J->rows ? J->rows[r] : r;
        const int64_t bh = row / Lq, i = row % Lq;
        const int32_t qb = (int32_t)(i / bs);
        for (int32_t d = 0; d < D; ++d) qv[d] = bf16_to_f64(J->q[row * D + d]);

        int64_t n = 0;
        for (int32_t kb = 0; kb < nbkv; ++kb) {
            if (!J->mask[(int64_t)qb * nbkv + kb]) continue;
            for (int64_t j = (int64_t)kb * bs; j < (int64_t)(kb + 1) * bs; ++j) {
                const uint16_t *kj = J->k + (bh * Lkv + j) * D;
                double dot = 0.0;
                for (int32_t d = 0; d < D; ++d) dot += qv[d] * bf16_to_f64(kj[d]);
                S[n] = J->scale * dot;
                key[n] = j;
                ++n;
            }
        }
        double *o = J->out + r * D;
        if (n == 0) {
            for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
            if (J->lse) J->lse[r] = -INFINITY;
            if (J->lsum) J->lsum[r] = 0.0;
            continue;
        }
        double c;
        if (J->shift) {
            c = J->shift[r];
        } else {
            c = S[0];
            for (int64_t t = 1; t < n; ++t) c = S[t] > c ? S[t] : c;
        }
        double l = 0.0;
        for (int32_t d = 0; d < D; ++d) acc[d] = 0.0;
        for (int64_t t = 0; t < n; ++t) {
            const double p = exp(S[t] - c);
            l += p;
            const uint16_t *vj = J->v + (bh * Lkv + key[t]) * D;
            for (int32_t d = 0; d < D; ++d) acc[d] += p * bf16_to_f64(vj[d]);
        }
        for (int32_t d = 0; d < D; ++d) o[d] = acc[d] / l;
        if (J->lse) J->lse[r] = c + log(l);
        if (J->lsum) J->lsum[r] = l;
    }
    free(S);
    free(key);
    free(qv);
    free(acc);
}

static void *attn_thread(void *arg) { attn_rows((const attn_job_t *)arg); return NULL; }

void orc_attention(int32_t B, int32_t H, int64_t Lq, int64_t Lkv, int32_t D, int32_t bs, const uint8_t *mask,
                   const uint16_t *q, const uint16_t *k, const uint16_t *v, double scale,
                   int64_t nrows, const int64_t *rows, const double *shift,
                   double *out, double *lse, double *lsum, int32_t nthreads) {
    attn_job_t base;
    memset(&base, 0, sizeof base);
    base.H = H; base.D = D; base.bs = bs; base.nbkv = (int32_t)(Lkv / bs); base.Lq = Lq; base.Lkv = Lkv;
    base.mask = mask; base.q = q; base.k = k; base.v = v; base.scale = scale;
    base.rows = rows; base.shift = shift; base.out = out; base.lse = lse; base.lsum = lsum;
    if (!rows) nrows = (int64_t)B * H * Lq;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if (nthreads > nrows) nthreads = (int32_t)(nrows > 0 ? nrows : 1);
    pthread_t th[512];
    attn_job_t jobs[512];
    int ok[512];
    const int64_t chunk = (nrows + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].r0 = (int64_t)t * chunk;
        jobs[t].r1 = jobs[t].r0 + chunk < nrows ? jobs[t].r0 + chunk : nrows;
        if (jobs[t].r0 > jobs[t].r1) jobs[t].r0 = jobs[t].r1;
        ok[t] = pthread_create(&th[t], NULL, attn_thread, &jobs[t]) == 0;
        if (!ok[t]) attn_rows(&jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        if (ok[t]) pthread_join(th[t], NULL);
}

/* ----------------------------------------------------------------------------
 * Norms and the Cauchy-Schwarz row bound ([deep-dive] remove softmax's serial
 * dependency: a small set of precomputed norms gives each row its bound, the
 * query's own norm times the largest key norm; [bytechap] How it works: an
 * upper bound derived from vector norms).
 *
 * fp64 form: |x| exactly rounded from an fp64 sum of squares, and
 *   M_i = scale * |q_i| * max_{j allowed for i} |k_j|.
 */
void orc_row_norms_f64(int64_t nrows, int32_t D, const uint16_t *x, double *out) {
    for (int64_t r = 0; r < nrows; ++r) {
        double s = 0.0;
        for (int32_t d = 0; d < D; ++d) {
            const double e = bf16_to_f64(x[r * D + d]);
            s += e * e;
        }
        out[r] = sqrt(s);
    }
}

void orc_row_bounds_f64(int32_t BH, int64_t Lq, int64_t Lkv, int32_t bs, const uint8_t *mask, double scale,
                        const double *qnorm, const double *knorm, double *bound) {
    const int32_t nbkv = (int32_t)(Lkv / bs);
    for (int32_t bh = 0; bh < BH; ++bh)
        for (int64_t i = 0; i < Lq; ++i) {
            const int32_t qb = (int32_t)(i / bs);
            double kmax = 0.0;
            int any = 0;
            for (int32_t kb = 0; kb < nbkv; ++kb) {
                if (!mask[(int64_t)qb * nbkv + kb]) continue;
                for (int64_t j = (int64_t)kb * bs; j < (int64_t)(kb + 1) * bs; ++j) {
                    const double kn = knorm[(int64_t)bh * Lkv + j];
                    if (!any || kn > kmax) kmax = kn;
                    any = 1;
                }
            }
            bound[(int64_t)bh * Lq + i] = scale * qnorm[(int64_t)bh * Lq + i] * kmax;
        }
}

/*
 * fp32 metadata with one fixed rounding order, so that any implementation
 * following the same order gets the same bits (the pages fix no precision for
 * the norm table; this order is the build's reading):
 *   - split the D elements of a row into 16 contiguous chunks of D/16;
 *   - per chunk c, s_c = fmaf(x, x, s_c) over its elements in order, from 0;
 *   - t_c = s_c + s_{c+8} (c < 8), u_c = t_c + t_{c+4} (c < 4),
 *     v_c = u_c + u_{c+2} (c < 2), w = v_0 + v_1;
 *   - norm = sqrtf(w) (correctly rounded).
 *   kmax[b,h,kb]  = max of the norms of the keys of block kb (exact);
 *   kB[b,h,qb]    = max of kmax[b,h,kb] over the allowed kb (exact);
 *   rowbound_i    = (scale * qnorm_i) * kB[b,h,qb(i)], each product rounded to fp32.
 * Compiled with -ffp-contract=off so the only fused operation is the explicit fmaf.
 */
void orc_row_norms_f32(int64_t nrows, int32_t D, const uint16_t *x, float *out) {
    const int32_t per = D / 16;
    for (int64_t r = 0; r < nrows; ++r) {
        float s[16];
        for (int c = 0; c < 16; ++c) {
            float a = 0.0f;
            for (int32_t e = 0; e < per; ++e) {
                const float xe = (float)bf16_to_f64(x[r * D + c * per + e]);
                a = fmaf(xe, xe, a);
            }
            s[c] = a;
        }
        float t[8], u[4], v[2];
        for (int c = 0; c < 8; ++c) t[c] = s[c] + s[c + 8];
        for (int c = 0; c < 4; ++c) u[c] = t[c] + t[c + 4];
        for (int c = 0; c < 2; ++c) v[c] = u[c] + u[c + 2];
        out[r] = sqrtf(v[0] + v[1]);
    }
}

void orc_block_max_f32(int32_t BH, int32_t nb, int32_t bs, const float *knorm, float *kmax) {
    for (int32_t bh = 0; bh < BH; ++bh)
        for (int32_t kb = 0; kb < nb; ++kb) {
            const float *p = knorm + ((int64_t)bh * nb + kb) * bs;
            float m = p[0];
            for (int32_t j = 1; j < bs; ++j) m = p[j] > m ? p[j] : m;
            kmax[(int64_t)bh * nb + kb] = m;
        }
}

void orc_row_bounds_f32(int32_t BH, int64_t Lq, int32_t nbkv, int32_t bs, const uint8_t *mask, float scale,
                        const float *qnorm, const float *kmax, float *rowbound) {
    const int32_t nbq = (int32_t)(Lq / bs);
    for (int32_t bh = 0; bh < BH; ++bh)
        for (int32_t qb = 0; qb < nbq; ++qb) {
            float kB = 0.0f;
            for (int32_t kb = 0; kb < nbkv; ++kb)
                if (mask[(int64_t)qb * nbkv + kb]) {
                    const float m = kmax[(int64_t)bh * nbkv + kb];
                    kB = m > kB ? m : kB;
                }
            for (int64_t i = (int64_t)qb * bs; i < (int64_t)(qb + 1) * bs; ++i) {
                const float a = scale * qnorm[(int64_t)bh * Lq + i];
                rowbound[(int64_t)bh * Lq + i] = a * kB;
            }
        }
}
