/*
 * Engram conditional memory -- CPU ORACLE for the hash-gather and context-aware-gate hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg load this library.  The product path (the CUDA
 * library under engram_conditional_memory_gb300/) never calls it, links it or
 * shares any code, header, table or constant with it.
 *
 * Everything here is a plain scalar loop written straight from the definitions,
 * one token at a time, with fp64 accumulation.  Nothing is blocked, fused,
 * vectorised or reordered beyond what the definition states.  Sources:
 *
 *   [T34]  TileLang tutorial, ch. 34 "TileKernels: Engram and mHC"
 *            sec. 1.2  the four parts of Engram (compression P: V->V', multi-head
 *                      multiply-XOR hashing into prime-sized tables, the
 *                      context-aware gate alpha = sigmoid(RMSNorm(h)^T RMSNorm(k)/sqrt(d)),
 *                      output alpha * v)
 *            sec. 2.1  tensors and the data flow fused_weight -> gate_fwd -> gate_bwd
 *                      -> grad_w_reduce; the saved dot / alpha / rstd_x / rstd_k
 *            sec. 2.3  addressing: (max_n - 1) * heads rows per token, exclusive
 *                      prefix-sum offsets into one concatenated table
 *            sec. 3.1  the weighted-RMSNorm identity that allows w_h (*) w_k folding
 *            sec. 4.2  backward chain rule of the gate
 *            sec. 4.3  the weight-gradient reduction: sum the partials, then
 *                      grad_w_h += S * w_k and grad_w_k += S * w_h
 *   [T13]  TileLang tutorial, ch. 13 "elementwise / norm / RoPE", sec. 5.4:
 *          the RMS mean divides by the true length d.
 *
 *   NEXT-1 (the multi-branch production gate of the TileKernels release): T34 sec. 2.1
 *   (x [T, hc, d], kv [T, hc+1, d], the signed-sqrt + clamp activation, out = x + alpha v),
 *   sec. 3.2 (forward) and sec. 4.2 (backward, including the zero-gradient clamp branch).
 *   NEXT-4 (the Engram Sinkhorn of the TileKernels release): T34 sec. 5.3 -- momentum update,
 *   the row step with its column partial sums, the ordered reduction, finalize.
 *   NEXT-2 (the short convolution after the gate): T34 sec. 1.2 item 4 -- Y = SiLU(Conv1D(
 *   RMSNorm(V~))) + V~, H <- H + Y, kernel size 4, dilation the largest N-gram order.
 *
 * Readings where the pages leave a step open (each one is also listed in the
 * design notes):
 *   - the exact hash: h = XOR_{j<n} (uint64) id'[t-j] * M[n,k,j] (mod 2^64),
 *     idx = h mod p[n,k] with unsigned 64-bit modulo; j = 0 is the current token,
 *     positions before the sequence start contribute the pad id 0;
 *   - the gate uses the plain sigmoid of the paper's Eq. 4 (no signed square root)
 *     and outputs alpha * v (no residual);
 *   - eps sits inside the root: rstd = 1 / sqrt(mean(x^2) + eps).
 *
 * Pins (every function is checked against something other than itself, in the
 * CPU test suite): closed-form hash cases with special multipliers and tiny
 * primes, sequence resets, brute-force invariants; gathered rows against a table
 * whose rows encode their own index; the gate against torch's rms_norm +
 * sigmoid in fp64, the k = 0 and h = +-k closed forms and the fused/unfused
 * identity; the backward against torch autograd and central finite differences
 * (both forms of the gate, the multi-branch one also through its clamp branch);
 * the reduction against constant partials with closed-form sums.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define EO_F32 0
#define EO_BF16 1

#define EO_OK 0
#define EO_ERR_ARG 1
#define EO_ERR_INDEX 2

/* Element i of a row-major tensor stored as fp32 or as raw bfloat16 bits, exactly widened to double. */
static double eo_load(const void *base, int dtype, int64_t i)
{
    if (dtype == EO_F32)
        return (double)((const float *)base)[i];
    uint32_t u = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double eo_sigmoid(double z)
{
    if (z >= 0.0)
        return 1.0 / (1.0 + exp(-z));
    double e = exp(z);
    return e / (1.0 + e);
}

/* ------------------------------------------------------------------------- */
/* A0-A1: compression and the multi-head N-gram hash  [T34 sec. 1.2, 2.3]      */
/* ------------------------------------------------------------------------- */

/*
 * For each token t in [t_begin, t_end) and each table (n, k), n = min_order ..
 * min_order + num_orders - 1, k = 0 .. heads - 1, in that order (table index
 * (n - min_order) * heads + k):
 *     id'(q) = compress_map[token_ids[q]]  (identity if compress_map is NULL),
 *              or the pad id 0 when q lies before the start of t's sequence;
 *     h = 0;  for j = 0 .. n-1:  h ^= id'(t - j) * M[table][j]   (mod 2^64)
 *     idx = h mod primes[table]
 * out_idx is [(t_end - t_begin), tables].  multipliers is [tables][mult_stride].
 * seq_offsets holds num_seqs + 1 boundaries (0 = first, T = last).
 */
int eo_hash_indices(const int32_t *token_ids, int64_t T,
                    const int64_t *seq_offsets, int32_t num_seqs,
                    const int32_t *compress_map, int32_t vocab,
                    int32_t min_order, int32_t num_orders, int32_t heads,
                    const uint64_t *multipliers, int32_t mult_stride,
                    const uint64_t *primes,
                    int64_t t_begin, int64_t t_end, int64_t *out_idx)
{
    const int32_t tables = num_orders * heads;
    if (!token_ids || !seq_offsets || !multipliers || !primes || !out_idx)
        return EO_ERR_ARG;
    if (num_seqs < 1 || min_order < 1 || num_orders < 1 || heads < 1)
        return EO_ERR_ARG;
    if (mult_stride < min_order + num_orders - 1 || t_begin < 0 || t_end > T || t_begin > t_end)
        return EO_ERR_ARG;
    if (seq_offsets[0] != 0 || seq_offsets[num_seqs] != T)
        return EO_ERR_ARG;
    for (int32_t tb = 0; tb < tables; ++tb)
        if (primes[tb] == 0)
            return EO_ERR_ARG;

    for (int64_t t = t_begin; t < t_end; ++t) {
        /* The sequence holding t: the one with seq_offsets[s] <= t < seq_offsets[s+1]. */
        int64_t start = -1;
        for (int32_t s = 0; s < num_seqs; ++s)
            if (seq_offsets[s] <= t && t < seq_offsets[s + 1])
                start = seq_offsets[s];
        if (start < 0)
            return EO_ERR_ARG;

        for (int32_t ni = 0; ni < num_orders; ++ni) {
            const int32_t n = min_order + ni;
            for (int32_t k = 0; k < heads; ++k) {
                const int32_t tb = ni * heads + k;
                uint64_t h = 0;
                for (int32_t j = 0; j < n; ++j) {
                    const int64_t q = t - j;
                    uint64_t id = 0; /* pad id before the sequence start */
                    if (q >= start) {
                        const int32_t raw = token_ids[q];
                        if (raw < 0 || raw >= vocab)
                            return EO_ERR_INDEX;
                        id = (uint64_t)(compress_map ? compress_map[raw] : raw);
                    }
                    h ^= id * multipliers[(int64_t)tb * mult_stride + j];
                }
                out_idx[(t - t_begin) * tables + tb] = (int64_t)(h % primes[tb]);
            }
        }
    }
    return EO_OK;
}

/* ------------------------------------------------------------------------- */
/* A2: the gather from the concatenated table  [T34 sec. 2.3]                 */
/* ------------------------------------------------------------------------- */

/*
 * All tables E_{n,k} live in one [sum(primes), row] table; table tb starts at
 * the exclusive prefix sum of primes[0..tb-1].  For each token t < ntok and
 * table tb the output row (t, tb) is a byte copy of table row
 * offset[tb] + idx[t][tb].  out is [ntok, tables, row_bytes] bytes, i.e. the
 * concatenation e_t in table order.
 */
int eo_gather_rows(const void *table, int64_t table_rows, int32_t row_bytes,
                   const uint64_t *primes, int32_t tables,
                   const int64_t *idx, int64_t ntok, void *out)
{
    if (!table || !primes || !idx || !out || row_bytes <= 0 || tables <= 0)
        return EO_ERR_ARG;
    for (int64_t t = 0; t < ntok; ++t) {
        uint64_t offset = 0;
        for (int32_t tb = 0; tb < tables; ++tb) {
            const int64_t i = idx[t * tables + tb];
            if (i < 0 || (uint64_t)i >= primes[tb])
                return EO_ERR_INDEX;
            const uint64_t row = offset + (uint64_t)i;
            if (row >= (uint64_t)table_rows)
                return EO_ERR_INDEX;
            memcpy((char *)out + (t * tables + tb) * (int64_t)row_bytes,
                   (const char *)table + (int64_t)row * row_bytes, (size_t)row_bytes);
            offset += primes[tb];
        }
    }
    return EO_OK;
}

/* ------------------------------------------------------------------------- */
/* B0: the weight fold  [T34 sec. 3.1]                                         */
/* ------------------------------------------------------------------------- */

/* w[i] = w_h[i] * w_k[i] in fp64 (the GPU path rounds it to fp32). */
int eo_fuse_weight(const float *w_h, const float *w_k, int32_t d, double *w)
{
    if (!w_h || !w_k || !w || d <= 0)
        return EO_ERR_ARG;
    for (int32_t i = 0; i < d; ++i)
        w[i] = (double)w_h[i] * (double)w_k[i];
    return EO_OK;
}

/* ------------------------------------------------------------------------- */
/* B1: the context-aware gate, forward  [T34 sec. 1.2 item 3, 2.1, 3.1]        */
/* ------------------------------------------------------------------------- */

/* Statistics of one token: rstd of h and of k, the fused-weight dot product, and z. */
struct eo_token_stats {
    double rh, rk, dot, z_unfused, z_fused, alpha;
};

static void eo_token_forward(const void *h, const void *k, int dtype, const float *w_h, const float *w_k,
                             int64_t t, int32_t d, double eps, struct eo_token_stats *st)
{
    const int64_t base = t * (int64_t)d;
    double sh = 0.0, sk = 0.0;
    for (int32_t i = 0; i < d; ++i) {
        const double x = eo_load(h, dtype, base + i);
        const double y = eo_load(k, dtype, base + i);
        sh += x * x;
        sk += y * y;
    }
    /* RMSNorm scale: 1 / sqrt(mean(x^2) + eps), mean over the true length d. */
    st->rh = 1.0 / sqrt(sh / (double)d + eps);
    st->rk = 1.0 / sqrt(sk / (double)d + eps);

    /* Paper form: normalise both vectors with their own RMSNorm weights, then take
     * the inner product scaled by 1/sqrt(d). */
    double acc = 0.0;
    for (int32_t i = 0; i < d; ++i) {
        const double nh = eo_load(h, dtype, base + i) * st->rh * (double)w_h[i];
        const double nk = eo_load(k, dtype, base + i) * st->rk * (double)w_k[i];
        acc += nh * nk;
    }
    st->z_unfused = acc / sqrt((double)d);

    /* The saved statistic: dot = sum_i h_i * (w_h,i * w_k,i) * k_i, and the z it gives. */
    double dot = 0.0;
    for (int32_t i = 0; i < d; ++i)
        dot += eo_load(h, dtype, base + i) * ((double)w_h[i] * (double)w_k[i]) * eo_load(k, dtype, base + i);
    st->dot = dot;
    st->z_fused = st->rh * st->rk * dot / sqrt((double)d);

    st->alpha = eo_sigmoid(st->z_unfused);
}

/*
 * For t in [t_begin, t_end):  alpha_t = sigmoid(RMSNorm(h_t; w_h) . RMSNorm(k_t; w_k) / sqrt(d)),
 * out_t = alpha_t * v_t, plus the saved statistics rstd_h, rstd_k and dot.
 * Row-major inputs [T, d]; outputs are indexed from t_begin.  z_fused (nullable)
 * receives rstd_h * rstd_k * dot / sqrt(d), which must equal the paper-form z.
 */
int eo_gate_fwd(const void *h, const void *k, const void *v, int dtype,
                const float *w_h, const float *w_k, int64_t T, int32_t d, double eps,
                int64_t t_begin, int64_t t_end,
                double *out, double *alpha, double *rstd_h, double *rstd_k, double *dot, double *z_fused)
{
    if (!h || !k || !v || !w_h || !w_k || !out || !alpha || !rstd_h || !rstd_k || !dot)
        return EO_ERR_ARG;
    if ((dtype != EO_F32 && dtype != EO_BF16) || d <= 0 || t_begin < 0 || t_end > T || t_begin > t_end)
        return EO_ERR_ARG;
    for (int64_t t = t_begin; t < t_end; ++t) {
        struct eo_token_stats st;
        eo_token_forward(h, k, dtype, w_h, w_k, t, d, eps, &st);
        const int64_t o = t - t_begin;
        alpha[o] = st.alpha;
        rstd_h[o] = st.rh;
        rstd_k[o] = st.rk;
        dot[o] = st.dot;
        if (z_fused)
            z_fused[o] = st.z_fused;
        for (int32_t i = 0; i < d; ++i)
            out[o * d + i] = st.alpha * eo_load(v, dtype, t * (int64_t)d + i);
    }
    return EO_OK;
}

/* ------------------------------------------------------------------------- */
/* B2: the gate backward  [T34 sec. 4.1, 4.2]                                  */
/* ------------------------------------------------------------------------- */

/*
 * Given the upstream gradient g = dL/dout for t in [t_begin, t_end), with
 * w_i = w_h,i * w_k,i and s = 1/sqrt(d):
 *     dv_t    = alpha_t * g_t
 *     dalpha  = sum_i g_i v_i
 *     c_t     = dalpha * alpha (1 - alpha) * s * rh * rk            (= dL/d dot)
 *     dh_t,i  = c_t * (w_i k_i - dot * rh^2 * h_i / d)
 *     dk_t,i  = c_t * (w_i h_i - dot * rk^2 * k_i / d)
 *     dweight_i = sum_t c_t h_t,i k_t,i                             (= dL/dw_i)
 * The forward statistics are recomputed here in fp64 from h and k.
 * dweight [d] is overwritten with the sum over [t_begin, t_end) in token order.
 * dweight_abs (nullable) receives sum_t |c_t h_t,i k_t,i|, the magnitude scale
 * that an fp32 accumulation of dweight is compared against.
 */
int eo_gate_bwd(const void *g, const void *h, const void *k, const void *v, int dtype,
                const float *w_h, const float *w_k, int64_t T, int32_t d, double eps,
                int64_t t_begin, int64_t t_end,
                double *dh, double *dk, double *dv, double *dweight, double *dweight_abs)
{
    if (!g || !h || !k || !v || !w_h || !w_k || !dh || !dk || !dv || !dweight)
        return EO_ERR_ARG;
    if ((dtype != EO_F32 && dtype != EO_BF16) || d <= 0 || t_begin < 0 || t_end > T || t_begin > t_end)
        return EO_ERR_ARG;
    const double s = 1.0 / sqrt((double)d);
    for (int32_t i = 0; i < d; ++i) {
        dweight[i] = 0.0;
        if (dweight_abs)
            dweight_abs[i] = 0.0;
    }
    for (int64_t t = t_begin; t < t_end; ++t) {
        struct eo_token_stats st;
        eo_token_forward(h, k, dtype, w_h, w_k, t, d, eps, &st);
        const int64_t base = t * (int64_t)d;
        const int64_t o = (t - t_begin) * (int64_t)d;

        double dalpha = 0.0;
        for (int32_t i = 0; i < d; ++i)
            dalpha += eo_load(g, dtype, base + i) * eo_load(v, dtype, base + i);
        const double c = dalpha * st.alpha * (1.0 - st.alpha) * s * st.rh * st.rk;

        for (int32_t i = 0; i < d; ++i) {
            const double hi = eo_load(h, dtype, base + i);
            const double ki = eo_load(k, dtype, base + i);
            const double wi = (double)w_h[i] * (double)w_k[i];
            dv[o + i] = st.alpha * eo_load(g, dtype, base + i);
            dh[o + i] = c * (wi * ki - st.dot * st.rh * st.rh * hi / (double)d);
            dk[o + i] = c * (wi * hi - st.dot * st.rk * st.rk * ki / (double)d);
            dweight[i] += c * hi * ki;
            if (dweight_abs)
                dweight_abs[i] += fabs(c * hi * ki);
        }
    }
    return EO_OK;
}

/* ------------------------------------------------------------------------- */
/* B3: the weight-gradient reduction  [T34 sec. 4.3, 4.4]                      */
/* ------------------------------------------------------------------------- */

/*
 * S_i = sum_{p<P} partial[p][i] (fp64, p ascending).  When w_h and w_k are given,
 * inc_h = S (*) w_k and inc_k = S (*) w_h are the increments that the reduction
 * adds to the accumulated fp32 parameter gradients of w_h and w_k.
 */
int eo_grad_w_reduce(const float *partial, int32_t P, int32_t d,
                     const float *w_h, const float *w_k, double *S, double *inc_h, double *inc_k)
{
    if (!partial || !S || P < 0 || d <= 0)
        return EO_ERR_ARG;
    for (int32_t i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int32_t p = 0; p < P; ++p)
            acc += (double)partial[(int64_t)p * d + i];
        S[i] = acc;
        if (w_h && w_k && inc_h && inc_k) {
            inc_h[i] = acc * (double)w_k[i];
            inc_k[i] = acc * (double)w_h[i];
        }
    }
    return EO_OK;
}

/* ------------------------------------------------------------------------- */
/* NEXT-1: the multi-branch gate of the TileKernels release  [T34 sec. 2.1, 3.2, 4.2] */
/* ------------------------------------------------------------------------- */

/*
 * hc branches share one value.  x is [T, hc, d]; kv is [T, hc+1, d] with rows 0..hc-1 the
 * branch keys and row hc the shared value; w_h and w_k are [hc, d].  For branch h of token t,
 * with s = 1/sqrt(d) and the clamp value c:
 *     rstd_x = 1/sqrt(sum_i x^2/d + eps),   rstd_k likewise over the key row,
 *     dot    = sum_i x_i (w_h,i w_k,i) k_i,
 *     z      = s * rstd_x * rstd_k * dot            (the paper form's pre-activation)
 *     gate   = sigmoid(sign(z) * sqrt(max(|z|, c)))  (sign(0) taken as +, as copysign(., +0) gives)
 *     out    = x + gate * v.
 * Here too the paper form is evaluated: both RMSNorms with their own weights, then the scaled
 * inner product; the saved dot is the fused-weight sum.  Outputs are indexed from t_begin.
 */
static void eo_branch_forward(const void *x, const void *kv, int dtype, const float *w_h, const float *w_k,
                              int64_t t, int32_t hc, int32_t h, int32_t d, double eps, double clamp,
                              double *rx, double *rk, double *dot, double *z_out, double *gate)
{
    const int64_t xb = (t * hc + h) * (int64_t)d;
    const int64_t kb = (t * (hc + 1) + h) * (int64_t)d;
    const float *wh = w_h + (int64_t)h * d, *wk = w_k + (int64_t)h * d;
    double sx = 0.0, sk = 0.0;
    for (int32_t i = 0; i < d; ++i) {
        const double a = eo_load(x, dtype, xb + i), b = eo_load(kv, dtype, kb + i);
        sx += a * a;
        sk += b * b;
    }
    *rx = 1.0 / sqrt(sx / (double)d + eps);
    *rk = 1.0 / sqrt(sk / (double)d + eps);
    double acc = 0.0, dt = 0.0;
    for (int32_t i = 0; i < d; ++i) {
        const double a = eo_load(x, dtype, xb + i), b = eo_load(kv, dtype, kb + i);
        acc += (a * (*rx) * (double)wh[i]) * (b * (*rk) * (double)wk[i]);
        dt += a * ((double)wh[i] * (double)wk[i]) * b;
    }
    const double z = acc / sqrt((double)d);
    const double m = fabs(z) > clamp ? fabs(z) : clamp;
    const double sgn = signbit(z) ? -1.0 : 1.0;
    *dot = dt;
    *z_out = z;
    *gate = eo_sigmoid(sgn * sqrt(m));
}

int eo_gate_hc_fwd(const void *x, const void *kv, int dtype, const float *w_h, const float *w_k,
                   int64_t T, int32_t hc, int32_t d, double eps, double clamp, int64_t t_begin, int64_t t_end,
                   double *out, double *gate, double *rstd_x, double *rstd_k, double *dot)
{
    if (!x || !kv || !w_h || !w_k || !out || !gate || !rstd_x || !rstd_k || !dot)
        return EO_ERR_ARG;
    if ((dtype != EO_F32 && dtype != EO_BF16) || hc < 1 || d <= 0 || t_begin < 0 || t_end > T || t_begin > t_end)
        return EO_ERR_ARG;
    for (int64_t t = t_begin; t < t_end; ++t) {
        const int64_t vb = (t * (hc + 1) + hc) * (int64_t)d;
        for (int32_t h = 0; h < hc; ++h) {
            double rx, rk, dt, z, g;
            eo_branch_forward(x, kv, dtype, w_h, w_k, t, hc, h, d, eps, clamp, &rx, &rk, &dt, &z, &g);
            const int64_t o = (t - t_begin) * hc + h;
            gate[o] = g;
            rstd_x[o] = rx;
            rstd_k[o] = rk;
            dot[o] = dt;
            const int64_t xb = (t * hc + h) * (int64_t)d;
            for (int32_t i = 0; i < d; ++i)
                out[o * d + i] = eo_load(x, dtype, xb + i) + g * eo_load(kv, dtype, vb + i);
        }
    }
    return EO_OK;
}

/*
 * Backward of eo_gate_hc_fwd for tokens [t_begin, t_end), g = dL/dout [T, hc, d]:
 *     dgate_h = sum_i g_h,i v_i
 *     c_h     = 0 when |z_h| < c (the clamp holds the activation constant there), else
 *               dgate_h * gate_h (1 - gate_h) / (2 sqrt|z_h|) * s * rstd_x * rstd_k   (= dL/d dot_h)
 *     dx_h    = g_h + c_h (w_h (*) w_k * k_h - dot_h rstd_x^2 x_h / d)
 *     dk_h    = c_h (w_h (*) w_k * x_h - dot_h rstd_k^2 k_h / d)
 *     dv      = sum_h gate_h g_h
 *     dweight[h, i] = sum_t c_h x_h,i k_h,i   ([hc, d], token order), dweight_abs the sum of |terms|.
 * dx is [n, hc, d], dkv is [n, hc+1, d] (row hc = dv).
 */
int eo_gate_hc_bwd(const void *g, const void *x, const void *kv, int dtype, const float *w_h, const float *w_k,
                   int64_t T, int32_t hc, int32_t d, double eps, double clamp, int64_t t_begin, int64_t t_end,
                   double *dx, double *dkv, double *dweight, double *dweight_abs)
{
    if (!g || !x || !kv || !w_h || !w_k || !dx || !dkv || !dweight)
        return EO_ERR_ARG;
    if ((dtype != EO_F32 && dtype != EO_BF16) || hc < 1 || d <= 0 || t_begin < 0 || t_end > T || t_begin > t_end)
        return EO_ERR_ARG;
    const double s = 1.0 / sqrt((double)d);
    for (int64_t i = 0; i < (int64_t)hc * d; ++i) {
        dweight[i] = 0.0;
        if (dweight_abs)
            dweight_abs[i] = 0.0;
    }
    for (int64_t t = t_begin; t < t_end; ++t) {
        const int64_t vb = (t * (hc + 1) + hc) * (int64_t)d;
        const int64_t o = t - t_begin;
        double *dv = dkv + (o * (hc + 1) + hc) * (int64_t)d;
        for (int32_t i = 0; i < d; ++i)
            dv[i] = 0.0;
        for (int32_t h = 0; h < hc; ++h) {
            double rx, rk, dt, z, gt;
            eo_branch_forward(x, kv, dtype, w_h, w_k, t, hc, h, d, eps, clamp, &rx, &rk, &dt, &z, &gt);
            const int64_t xb = (t * hc + h) * (int64_t)d;
            const int64_t kb = (t * (hc + 1) + h) * (int64_t)d;
            double dgate = 0.0;
            for (int32_t i = 0; i < d; ++i)
                dgate += eo_load(g, dtype, xb + i) * eo_load(kv, dtype, vb + i);
            double c = 0.0;
            if (!(fabs(z) < clamp))
                c = dgate * gt * (1.0 - gt) / (2.0 * sqrt(fabs(z))) * s * rx * rk;
            double *dxr = dx + (o * hc + h) * (int64_t)d;
            double *dkr = dkv + (o * (hc + 1) + h) * (int64_t)d;
            for (int32_t i = 0; i < d; ++i) {
                const double xi = eo_load(x, dtype, xb + i), ki = eo_load(kv, dtype, kb + i);
                const double gi = eo_load(g, dtype, xb + i);
                const double wi = (double)w_h[(int64_t)h * d + i] * (double)w_k[(int64_t)h * d + i];
                dxr[i] = gi + c * (wi * ki - dt * rx * rx * xi / (double)d);
                dkr[i] = c * (wi * xi - dt * rk * rk * ki / (double)d);
                dv[i] += gt * gi;
                dweight[(int64_t)h * d + i] += c * xi * ki;
                if (dweight_abs)
                    dweight_abs[(int64_t)h * d + i] += fabs(c * xi * ki);
            }
        }
    }
    return EO_OK;
}

/* ------------------------------------------------------------------------- */
/* NEXT-4: the Engram Sinkhorn (row / column L2 scaling)  [T34 sec. 5.3]      */
/* ------------------------------------------------------------------------- */

/*
 * Momentum update (the momentum form of T34 sec. 5.3 step 1; the exact update is this
 * library's reading): m <- beta1 * m + g;  input = nesterov ? g + beta1 * m : m.
 * grad is fp32 or bf16 [n], momentum_in fp32 [n]; outputs are fp64 [n].
 */
int eo_sinkhorn_momentum(const void *grad, int dtype, const float *momentum_in, int64_t n, double beta1,
                         int nesterov, double *momentum_out, double *input_out)
{
    if (!grad || !momentum_in || !momentum_out || !input_out || n < 0 || (dtype != EO_F32 && dtype != EO_BF16))
        return EO_ERR_ARG;
    for (int64_t i = 0; i < n; ++i) {
        const double g = eo_load(grad, dtype, i);
        const double m = beta1 * (double)momentum_in[i] + g;
        momentum_out[i] = m;
        input_out[i] = nesterov ? g + beta1 * m : m;
    }
    return EO_OK;
}

/*
 * The row step (T34 sec. 5.3 step 2), for rows [r_begin, r_end) of a [rows, head_dim] matrix:
 *     x          = row_scale[r] * matrix[r, :] (*) col_scale
 *     row_norm   = ||x||_2
 *     row_scale' = row_scale[r] / (row_norm + eps)
 *     col_sumsq += (x / (row_norm + eps))^2         (column-wise, rows in ascending order)
 * Outputs indexed from r_begin (row_norm, row_scale_out [n]); col_sumsq [head_dim] is overwritten.
 */
int eo_sinkhorn_step(const float *matrix, const float *row_scale, const float *col_scale, int64_t rows,
                     int32_t head_dim, double eps, int64_t r_begin, int64_t r_end,
                     double *row_norm, double *row_scale_out, double *col_sumsq)
{
    if (!matrix || !row_scale || !col_scale || !row_norm || !row_scale_out || !col_sumsq)
        return EO_ERR_ARG;
    if (head_dim <= 0 || r_begin < 0 || r_end > rows || r_begin > r_end)
        return EO_ERR_ARG;
    for (int32_t c = 0; c < head_dim; ++c)
        col_sumsq[c] = 0.0;
    for (int64_t r = r_begin; r < r_end; ++r) {
        double ss = 0.0;
        for (int32_t c = 0; c < head_dim; ++c) {
            const double x = (double)row_scale[r] * (double)matrix[r * head_dim + c] * (double)col_scale[c];
            ss += x * x;
        }
        const double nrm = sqrt(ss);
        const double inv = 1.0 / (nrm + eps);
        row_norm[r - r_begin] = nrm;
        row_scale_out[r - r_begin] = (double)row_scale[r] * inv;
        for (int32_t c = 0; c < head_dim; ++c) {
            const double x = (double)row_scale[r] * (double)matrix[r * head_dim + c] * (double)col_scale[c] * inv;
            col_sumsq[c] += x * x;
        }
    }
    return EO_OK;
}

/*
 * The column step that the caller of T34's step_reduce performs: the reduced column sums of squares
 * give the column L2 norms, and col_scale' = col_scale / (sqrt(col_sumsq) + eps).
 */
int eo_sinkhorn_col_update(const double *col_sumsq, const float *col_scale, int32_t head_dim, double eps,
                           double *col_scale_out)
{
    if (!col_sumsq || !col_scale || !col_scale_out || head_dim <= 0)
        return EO_ERR_ARG;
    for (int32_t c = 0; c < head_dim; ++c)
        col_scale_out[c] = (double)col_scale[c] / (sqrt(col_sumsq[c]) + eps);
    return EO_OK;
}

/*
 * Finalize (T34 sec. 5.3 step 4): out[r, :] = alpha * x / (||x||_2 + eps), x = row_scale[r] * matrix[r, :]
 * (*) col_scale.  out is [rows, head_dim] fp64.
 */
int eo_sinkhorn_finalize(const float *matrix, const float *row_scale, const float *col_scale, int64_t rows,
                         int32_t head_dim, double eps, double alpha, double *out)
{
    if (!matrix || !row_scale || !col_scale || !out || head_dim <= 0 || rows < 0)
        return EO_ERR_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int32_t c = 0; c < head_dim; ++c) {
            const double x = (double)row_scale[r] * (double)matrix[r * head_dim + c] * (double)col_scale[c];
            ss += x * x;
        }
        const double f = alpha / (sqrt(ss) + eps);
        for (int32_t c = 0; c < head_dim; ++c)
            out[r * head_dim + c] =
                (double)row_scale[r] * (double)matrix[r * head_dim + c] * (double)col_scale[c] * f;
    }
    return EO_OK;
}

/* ------------------------------------------------------------------------- */
/* NEXT-2: the short convolution + SiLU + residual after the gate  [T34 sec. 1.2 item 4] */
/* ------------------------------------------------------------------------- */

/*
 * The pages give only Y = SiLU(Conv1D(RMSNorm(V~))) + V~ and H <- H + Y, with kernel size w = 4
 * and the dilation equal to the largest N-gram order (the step is not in the TileKernels release).
 * Readings (listed in the design notes):
 *   - V~ [T, d] is the gate's output sequence alpha_t v_t; RMSNorm has a learnable weight
 *     norm_w [d] and eps inside the root, like the gate's norms;
 *   - Conv1D is depthwise (one w-tap filter per channel, conv_w [d][w], optional bias [d]) and
 *     causal within each sequence: tap i multiplies the token (w - 1 - i) * dilation steps back, so
 *     tap w - 1 is the current token (torch's conv1d layout with (w - 1) * dilation left padding);
 *     positions before the sequence start are zero;
 *   - out = H + SiLU(c) + V~ (H nullable: then out = Y).
 */

static int eo_seq_of(const int64_t *offs, int32_t num_seqs, int64_t t)
{
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) { /* largest s with offs[s] <= t */
        const int mid = (lo + hi + 1) / 2;
        if (offs[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

static double eo_conv_rstd(const void *v, int dtype, int64_t t, int32_t d, double eps)
{
    double ss = 0.0;
    for (int32_t j = 0; j < d; ++j) {
        const double x = eo_load(v, dtype, t * (int64_t)d + j);
        ss += x * x;
    }
    return 1.0 / sqrt(ss / (double)d + eps);
}

/*
 * rstd of the tokens [lo, hi) around the range a call works on, computed once per token (the
 * same value the definition gives at every use; nothing is reordered).
 */
typedef struct {
    int64_t lo, hi;
    double *r;
} eo_rstd_cache;

static int eo_rstd_cache_fill(eo_rstd_cache *rc, const void *v, int dtype, int64_t T, int32_t d, double eps,
                              int64_t lo, int64_t hi)
{
    rc->lo = lo < 0 ? 0 : lo;
    rc->hi = hi > T ? T : hi;
    rc->r = (double *)malloc(sizeof(double) * (size_t)(rc->hi > rc->lo ? rc->hi - rc->lo : 1));
    if (!rc->r) return EO_ERR_ARG;
    for (int64_t t = rc->lo; t < rc->hi; ++t)
        rc->r[t - rc->lo] = eo_conv_rstd(v, dtype, t, d, eps);
    return EO_OK;
}

/* u[t', j] = V~[t', j] * rstd(t') * norm_w[j] when t' lies in [seq_start, T), else 0. */
static double eo_conv_u(const void *v, int dtype, const float *norm_w, const eo_rstd_cache *rc, int64_t tp,
                        int64_t seq_start, int32_t d, int32_t j)
{
    if (tp < seq_start) return 0.0;
    return eo_load(v, dtype, tp * (int64_t)d + j) * rc->r[tp - rc->lo] * (double)norm_w[j];
}

/* c[t, j] = bias[j] + sum_i conv_w[j][i] * u[t - (w - 1 - i) * dilation, j] */
static double eo_conv_c(const void *v, int dtype, const float *norm_w, const float *conv_w, const float *bias,
                        const eo_rstd_cache *rc, int64_t t, int64_t seq_start, int32_t d, int32_t w, int32_t dil,
                        int32_t j)
{
    double c = bias ? (double)bias[j] : 0.0;
    for (int32_t i = 0; i < w; ++i)
        c += (double)conv_w[(int64_t)j * w + i] *
             eo_conv_u(v, dtype, norm_w, rc, t - (int64_t)(w - 1 - i) * dil, seq_start, d, j);
    return c;
}

static int eo_conv_args(const void *v, int dtype, const float *norm_w, const float *conv_w,
                        const int64_t *offs, int32_t num_seqs, int64_t T, int32_t d, int32_t w, int32_t dil,
                        int64_t t_begin, int64_t t_end)
{
    if (!v || !norm_w || !conv_w || !offs || num_seqs < 1 || d <= 0 || w < 1 || dil < 1)
        return EO_ERR_ARG;
    if ((dtype != EO_F32 && dtype != EO_BF16) || t_begin < 0 || t_end > T || t_begin > t_end)
        return EO_ERR_ARG;
    if (offs[0] != 0 || offs[num_seqs] != T)
        return EO_ERR_ARG;
    for (int32_t s = 0; s < num_seqs; ++s)
        if (offs[s + 1] < offs[s]) return EO_ERR_ARG;
    return EO_OK;
}

/*
 * Forward for tokens [t_begin, t_end): out = H + SiLU(c) + V~ (rows indexed from t_begin, fp64),
 * c (nullable) the convolution output, rstd (nullable) [n] the RMSNorm statistic of V~.
 */
int eo_short_conv_fwd(const void *v, const void *h, int dtype, const float *norm_w, const float *conv_w,
                      const float *bias, const int64_t *offs, int32_t num_seqs, int64_t T, int32_t d, int32_t w,
                      int32_t dil, double eps, int64_t t_begin, int64_t t_end, double *out, double *c_out,
                      double *rstd)
{
    if (eo_conv_args(v, dtype, norm_w, conv_w, offs, num_seqs, T, d, w, dil, t_begin, t_end) != EO_OK || !out)
        return EO_ERR_ARG;
    eo_rstd_cache rc;
    if (eo_rstd_cache_fill(&rc, v, dtype, T, d, eps, t_begin - (int64_t)(w - 1) * dil, t_end) != EO_OK)
        return EO_ERR_ARG;
    for (int64_t t = t_begin; t < t_end; ++t) {
        const int64_t s0 = offs[eo_seq_of(offs, num_seqs, t)];
        if (rstd) rstd[t - t_begin] = rc.r[t - rc.lo];
        for (int32_t j = 0; j < d; ++j) {
            const double c = eo_conv_c(v, dtype, norm_w, conv_w, bias, &rc, t, s0, d, w, dil, j);
            const double y = c * eo_sigmoid(c) + eo_load(v, dtype, t * (int64_t)d + j);
            out[(t - t_begin) * d + j] = (h ? eo_load(h, dtype, t * (int64_t)d + j) : 0.0) + y;
            if (c_out) c_out[(t - t_begin) * d + j] = c;
        }
    }
    free(rc.r);
    return EO_OK;
}

/* dL/dc at (t, j) given dout = g: g * SiLU'(c), SiLU'(c) = s (1 + c (1 - s)), s = sigmoid(c). */
static double eo_conv_dc(const void *g, const void *v, int dtype, const float *norm_w, const float *conv_w,
                         const float *bias, const eo_rstd_cache *rc, int64_t t, int64_t seq_start, int32_t d,
                         int32_t w, int32_t dil, int32_t j)
{
    const double c = eo_conv_c(v, dtype, norm_w, conv_w, bias, rc, t, seq_start, d, w, dil, j);
    const double s = eo_sigmoid(c);
    return eo_load(g, dtype, t * (int64_t)d + j) * s * (1.0 + c * (1.0 - s));
}

/*
 * Backward for tokens [t_begin, t_end), given g = dL/dout [T, d] (dL/dH = g, not returned):
 *     du[t, j]  = sum_i conv_w[j][i] * dc[t + (w - 1 - i) * dil, j]   (same sequence only)
 *     s[t]      = sum_j norm_w[j] du[t, j] V~[t, j]
 *     dV~[t, j] = g[t, j] + rstd(t) norm_w[j] du[t, j] - rstd(t)^3 V~[t, j] s[t] / d
 * and, accumulated over the range (zeroed first):
 *     dconv_w[j][i] += dc[t, j] * u[t - (w - 1 - i) * dil, j]
 *     dbias[j]      += dc[t, j]
 *     dnorm_w[j]    += du[t, j] * V~[t, j] * rstd(t)
 * dv is [n, d] from t_begin.  The *_abs outputs (nullable) are the same sums over |terms|, for
 * tolerances: dv_abs[t, j] = |g| + |rstd norm_w du| + |rstd^3 V~ s / d|.
 */
int eo_short_conv_bwd(const void *g, const void *v, int dtype, const float *norm_w, const float *conv_w,
                      const float *bias, const int64_t *offs, int32_t num_seqs, int64_t T, int32_t d, int32_t w,
                      int32_t dil, double eps, int64_t t_begin, int64_t t_end, double *dv, double *dconv_w,
                      double *dbias, double *dnorm_w, double *dv_abs, double *dconv_w_abs, double *dbias_abs,
                      double *dnorm_w_abs)
{
    if (eo_conv_args(v, dtype, norm_w, conv_w, offs, num_seqs, T, d, w, dil, t_begin, t_end) != EO_OK || !g ||
        !dv || !dconv_w || !dbias || !dnorm_w)
        return EO_ERR_ARG;
    for (int64_t k = 0; k < (int64_t)d * w; ++k) {
        dconv_w[k] = 0.0;
        if (dconv_w_abs) dconv_w_abs[k] = 0.0;
    }
    for (int32_t j = 0; j < d; ++j) {
        dbias[j] = dnorm_w[j] = 0.0;
        if (dbias_abs) dbias_abs[j] = 0.0;
        if (dnorm_w_abs) dnorm_w_abs[j] = 0.0;
    }
    eo_rstd_cache rc;
    if (eo_rstd_cache_fill(&rc, v, dtype, T, d, eps, t_begin - (int64_t)(w - 1) * dil,
                           t_end + (int64_t)(w - 1) * dil) != EO_OK)
        return EO_ERR_ARG;
    for (int64_t t = t_begin; t < t_end; ++t) {
        const int sq = eo_seq_of(offs, num_seqs, t);
        const int64_t s0 = offs[sq], s1 = offs[sq + 1];
        const double r = rc.r[t - rc.lo];
        double *row = dv + (t - t_begin) * d;
        double s = 0.0, s_abs = 0.0;
        for (int32_t j = 0; j < d; ++j) {
            /* du from the taps that read token t: tokens t + (w - 1 - i) * dil of the same sequence */
            double du = 0.0;
            for (int32_t i = 0; i < w; ++i) {
                const int64_t tf = t + (int64_t)(w - 1 - i) * dil;
                if (tf < s1)
                    du += (double)conv_w[(int64_t)j * w + i] *
                          eo_conv_dc(g, v, dtype, norm_w, conv_w, bias, &rc, tf, s0, d, w, dil, j);
            }
            const double x = eo_load(v, dtype, t * (int64_t)d + j);
            row[j] = du; /* kept here until s is known */
            s += (double)norm_w[j] * du * x;
            s_abs += fabs((double)norm_w[j] * du * x);
            dnorm_w[j] += du * x * r;
            if (dnorm_w_abs) dnorm_w_abs[j] += fabs(du * x * r);
            /* weight gradients of the taps at token t */
            const double dc = eo_conv_dc(g, v, dtype, norm_w, conv_w, bias, &rc, t, s0, d, w, dil, j);
            dbias[j] += dc;
            if (dbias_abs) dbias_abs[j] += fabs(dc);
            for (int32_t i = 0; i < w; ++i) {
                const double u = eo_conv_u(v, dtype, norm_w, &rc, t - (int64_t)(w - 1 - i) * dil, s0, d, j);
                dconv_w[(int64_t)j * w + i] += dc * u;
                if (dconv_w_abs) dconv_w_abs[(int64_t)j * w + i] += fabs(dc * u);
            }
        }
        for (int32_t j = 0; j < d; ++j) {
            const double du = row[j];
            const double x = eo_load(v, dtype, t * (int64_t)d + j);
            const double gj = eo_load(g, dtype, t * (int64_t)d + j);
            row[j] = gj + r * (double)norm_w[j] * du - r * r * r * x * s / (double)d;
            if (dv_abs)
                dv_abs[(t - t_begin) * d + j] =
                    fabs(gj) + fabs(r * (double)norm_w[j] * du) + fabs(r * r * r * x) * s_abs / (double)d;
        }
    }
    free(rc.r);
    return EO_OK;
}
