/*
 * engram.h -- C ABI of the GB300 (sm_103a) Engram conditional-memory hot path.
 *
 * The library implements the data-parallel hot path of Engram's conditional
 * memory as hand-written CUDA kernels:
 *
 *   A  the deterministic multi-head N-gram hash over compressed token ids and the
 *      gather of rows from prime-sized embedding tables  (engram_hash_gather);
 *   B  the context-aware gate: weight fold (engram_fuse_weight), forward
 *      (engram_gate_fwd), backward (engram_gate_bwd) and the deterministic
 *      cross-block weight-gradient reduction (engram_grad_w_reduce).
 *
 * Sources (the TileLang tutorial, ch. 34 "TileKernels: Engram and mHC"):
 *   sec. 1.2  the method: compression P: V -> V', K hash heads per N-gram order into
 *             prime-sized tables E_{n,k}, the gate
 *             alpha_t = sigmoid(RMSNorm(h_t)^T RMSNorm(k_t) / sqrt(d)), output alpha_t v_t;
 *   sec. 2.1  the operator chain fused_weight -> gate_fwd -> gate_bwd -> grad_w_reduce
 *             and the saved per-token statistics;
 *   sec. 2.3  addressing: (max_n - 1) * heads rows per token, one concatenated table
 *             indexed through exclusive prefix-sum offsets;
 *   sec. 3.1  the fold w_fused = w_h (*) w_k that turns two RMSNorms and a dot
 *             product into one pass over h and k;
 *   sec. 4.1-4.4  backward, per-block partial weight gradients, the separate
 *             reduction kernel with accumulate (main_grad) semantics.
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers of the current CUDA device, owned by
 *     the caller.  The library never allocates, frees or keeps them.
 *   - Per-token tensors may be NULL when the token count is 0 (an empty tensor
 *     has no storage); dw_partial may be NULL when P is 0.
 *   - Tensors are dense, row-major, and start on a 16-byte boundary; rows of
 *     [T, d] tensors are d elements long (so d * element size must be a
 *     multiple of 16 bytes).
 *   - Every call is asynchronous on `stream` (NULL = the legacy default
 *     stream) and never synchronises, except engram_read_error_word (also
 *     exported as engram_get_error) and engram_device_status, which say so.
 *   - Host-side argument checks run before anything is launched; a call that
 *     returns an error other than ENGRAM_ERR_CUDA has launched nothing.
 *   - Thread safety: calls from several host threads are safe; the text behind
 *     engram_last_error_string() is per thread.
 *   - The kernels contain no unbounded wait: a pipeline wait that exceeds about
 *     two seconds gives up, sets ENGRAM_DEVERR_TIMEOUT in the library's device
 *     status word and returns.
 *   - Per-device state is looked up on a device's first call and cached for the
 *     life of the process: the address of the library's status word and of the
 *     allocation-free entry point's array, and kernel attributes.  A
 *     cudaDeviceReset of a device the library has run on leaves those addresses
 *     stale, so the library must not be called on that device after such a reset.
 */
#ifndef ENGRAM_GB300_H
#define ENGRAM_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA stream type (cudaStream_t) without including the CUDA headers. */
typedef struct CUstream_st *engram_stream_t;

#define ENGRAM_ABI_VERSION 1

/* Largest number of hash tables (orders x heads) and largest N-gram order. */
#define ENGRAM_MAX_TABLES 32
#define ENGRAM_MAX_ORDER 8
/* Largest gate row, in bytes (d * element size): 8192 bf16 or 4096 fp32 elements. */
#define ENGRAM_MAX_ROW_BYTES 16384

typedef enum {
    ENGRAM_F32 = 0,  /* IEEE binary32 */
    ENGRAM_BF16 = 1  /* bfloat16; results are rounded to nearest even */
} engram_dtype;

typedef enum {
    ENGRAM_OK = 0,
    ENGRAM_ERR_NULL = 1,   /* a required pointer is NULL */
    ENGRAM_ERR_SHAPE = 2,  /* a size is negative, zero where it may not be, or too large */
    ENGRAM_ERR_DTYPE = 3,  /* unknown dtype, or a dtype the entry point does not take */
    ENGRAM_ERR_ALIGN = 4,  /* a tensor or a row does not start on a 16-byte boundary */
    ENGRAM_ERR_CUDA = 5,   /* a CUDA runtime call failed; see engram_last_error_string() */
    ENGRAM_ERR_INDEX = 6,  /* engram_read_error_word found a device-side error bit */
    ENGRAM_ERR_DEVICE = 7  /* a pointer is not device memory of the current device */
} engram_status;

/* Bits of a device error word (engram_hash_gather's err_word, engram_device_status). */
#define ENGRAM_DEVERR_TOKEN_ID 0x1u    /* a raw token id outside [0, vocab): hashed as the pad id 0 */
#define ENGRAM_DEVERR_COMPRESSED 0x2u  /* a compressed id outside [0, vocab_c): hashed as 0 */
#define ENGRAM_DEVERR_SEQ_OFFSETS 0x4u /* seq_offsets not 0 = o_0 <= o_1 <= ... <= o_S = T */
#define ENGRAM_DEVERR_TIMEOUT 0x8u     /* a bounded in-kernel wait gave up (should never happen) */

/* ------------------------------------------------------------------------- */
/* Library information and errors                                            */
/* ------------------------------------------------------------------------- */

/* ENGRAM_ABI_VERSION of the loaded library. */
int32_t engram_abi_version(void);

/* Static text for a status code. */
const char *engram_status_string(engram_status status);

/* Text of the last ENGRAM_ERR_CUDA (or other error) raised on the calling thread; "" if none. */
const char *engram_last_error_string(void);

/*
 * Device-pointer checks.  level 1 (default) asks the CUDA runtime whether every
 * tensor pointer is device memory of the current device (ENGRAM_ERR_DEVICE
 * otherwise); level 0 skips that query and keeps only the host-side checks.
 * Returns the previous level.  Process-wide.
 */
int32_t engram_set_validation(int32_t level);

/*
 * Caps the number of CTAs each kernel launch uses (0 = no cap, the default:
 * grids are sized from the SM count).  For sharing the GPU with concurrent work
 * on other streams.  Results do not depend on it: every partition of the work
 * is fixed by the problem sizes alone.  Returns the previous cap.  Process-wide.
 */
int32_t engram_set_max_ctas(int32_t max_ctas);

/*
 * Programmatic dependent launch for the step's kernels (hash gather, weight fold, gate forward,
 * gate backward, weight-gradient reduction): with it on (the default), each is launched with the
 * programmatic-stream-serialization attribute, so its launch overlaps the previous kernel's exit, and
 * waits in-kernel for that kernel's completion before touching memory; results are identical either
 * way.  Returns the previous setting.  Process-wide.
 */
int32_t engram_set_pdl(int32_t on);

/*
 * The multi-branch gate (engram_gate_hc_fwd / _bwd) runs a whole token of hc branches in one
 * kernel when its rows fit twice in shared memory.  When they do not, a cluster of two CTAs (or
 * four, two per SM) shares each token, each holding its part of every row and the CTAs exchanging
 * their parts' sums through distributed shared memory (rows a multiple of 32 / 64 bytes).  Only
 * when that does not fit either does it run branch by branch on strided views (plus one kernel for
 * the shared value's gradient).  on = 1 forces the branch-by-branch form at every size, on = 2 / 4
 * the cluster form over 2 / 4 CTAs wherever its parts fit, on = 0 (or any other value) restores the
 * choice above; for testing: results agree with the oracle in every form, though not bit for bit
 * with each other (the sums' thread layouts differ).  Returns the previous setting.  Process-wide.
 */
int32_t engram_set_hc_split(int32_t on);

/*
 * Copies a device error word to *host_out.  SYNCHRONISES `stream` first.
 * Returns ENGRAM_ERR_INDEX when any bit is set, ENGRAM_OK otherwise.
 */
engram_status engram_read_error_word(const uint32_t *err_word, engram_stream_t stream, uint32_t *host_out);

/* The same call under a second name (identical arguments, behaviour and return codes). */
engram_status engram_get_error(const uint32_t *err_word, engram_stream_t stream, uint32_t *host_out);

/*
 * The library's own device status word of the current device (ENGRAM_DEVERR_* bits
 * OR-ed by every kernel, e.g. ENGRAM_DEVERR_TIMEOUT).  SYNCHRONISES the device.
 * clear != 0 resets it to 0 after reading.
 */
engram_status engram_device_status(uint32_t *host_out, int32_t clear);

/*
 * Failure-detection self-check (no counterpart in the pages): launches one CTA that waits, with
 * the same bounded wait the pipelines use, on an mbarrier nothing completes.  It gives up after
 * limit_us microseconds (1 .. 2,000,000) and sets ENGRAM_DEVERR_TIMEOUT in the device status word,
 * as a stalled pipeline would; the context stays usable.  Nothing faults, traps or hangs.
 */
engram_status engram_check_wait_timeout(uint32_t limit_us, engram_stream_t stream);

/* ------------------------------------------------------------------------- */
/* A0-A2: compression, multi-head N-gram hash and gather  (ch. 34 sec. 1.2 item 2, sec. 2.3) */
/* ------------------------------------------------------------------------- */

/*
 * Fixed hash hyper-parameters (host memory; read during the call only).
 *
 * Tables are numbered in (order ascending, head ascending) order:
 * table = (n - min_order) * heads + k for n in [min_order, min_order + num_orders),
 * k in [0, heads).  tables = num_orders * heads <= ENGRAM_MAX_TABLES.
 * multipliers is [tables][mult_stride] (mult_stride >= max order), primes is
 * [tables]; primes are the row counts p_{n,k} of the tables, each in [1, 2^31).
 * They need not be prime, but the method's collision behaviour assumes it.
 */
typedef struct {
    int32_t min_order;           /* smallest N-gram order n (>= 1; the method uses 2) */
    int32_t num_orders;          /* number of orders (>= 1); max order <= ENGRAM_MAX_ORDER */
    int32_t heads;               /* K hash heads per order (>= 1) */
    int32_t mult_stride;         /* row length of `multipliers` */
    const uint64_t *multipliers; /* HOST [tables][mult_stride]; entry j < n multiplies id'[t - j] */
    const uint64_t *primes;      /* HOST [tables] */
} engram_hash_spec;

typedef struct {
    const int32_t *token_ids;    /* [T] raw ids in [0, vocab) */
    int64_t T;                   /* number of tokens (>= 0) */
    const int64_t *seq_offsets;  /* [num_seqs + 1] boundaries 0 = o_0 <= ... <= o_S = T (cu_seqlens) */
    int32_t num_seqs;            /* >= 1 */
    const int32_t *compress_map; /* [vocab] -> [0, vocab_c), the compression P; NULL = identity */
    int32_t vocab;               /* raw vocabulary size (>= 1) */
    int32_t vocab_c;             /* compressed vocabulary size (>= 1; = vocab when compress_map is NULL) */
    const void *table;           /* [table_rows, row_dim] concatenated E_{n,k}, table order */
    int64_t table_rows;          /* >= sum(primes) */
    int32_t row_dim;             /* elements per row; row_dim * element size a multiple of 16 bytes,
                                    and tables * row bytes (one token's e_t row) at most 64 KB */
    engram_dtype dtype;          /* element type of table and out_rows (bit copies either way) */
    int32_t *out_indices;        /* [T, tables] local index idx_{n,k}(t) in [0, p); NULL = not written */
    void *out_rows;              /* [T, tables * row_dim] e_t = concatenated rows; NULL = not written */
    uint32_t *err_word;          /* device word, OR-ed with ENGRAM_DEVERR_* bits; NULL = not reported */
} engram_hash_gather_args;

/*
 * For every token t (in the sequence s with o_s <= t < o_{s+1}) and table (n, k):
 *     id'(q) = compress_map[token_ids[q]] for o_s <= q, else the pad id 0;
 *     h      = XOR over j < n of  (uint64) id'(t - j) * multipliers[table][j]   (mod 2^64);
 *     idx    = h mod primes[table]   (unsigned 64-bit);
 *     row    = (exclusive prefix sum of primes before `table`) + idx;
 *     out_rows[t, table * row_dim : (table + 1) * row_dim] = table[row, :]   (bit copy).
 * The pages name only a "lightweight multiplicative-XOR hash"; this exact form
 * is the library's reading (ch. 34 sec. 1.2 item 2).  Indices depend only on the
 * ids, so results are bit-identical across runs and devices (sec. 2.3).
 * Bad ids are reported through err_word and hashed as 0; no read leaves the table.
 */
engram_status engram_hash_gather(const engram_hash_spec *spec, const engram_hash_gather_args *args,
                                 engram_stream_t stream);

/*
 * The same computation with the table in HOST memory (the Engram paper's offload of the tables,
 * possible because a token's rows follow from its ids alone; ch. 34 sec. 2.3).  args->table must
 * be page-locked and mapped into the device's address space (cudaHostAlloc, or cudaHostRegister
 * with cudaHostRegisterMapped; torch's pin_memory() qualifies): anything else returns
 * ENGRAM_ERR_DEVICE.  Every other pointer is device memory as above.  Rows cross the host link
 * with ordinary loads, so the call's speed is set by that link, not by HBM.
 */
engram_status engram_hash_gather_host(const engram_hash_spec *spec, const engram_hash_gather_args *args,
                                      engram_stream_t stream);

/* ------------------------------------------------------------------------- */
/* B0: weight fold  (ch. 34 sec. 3.1, sec. 4.1)                               */
/* ------------------------------------------------------------------------- */

/*
 * w_fused[i] = w_h[i] * w_k[i], computed and stored in fp32, for i < d.
 * w_h and w_k are the RMSNorm weights of the hidden state and of the key, in
 * `dtype` (fp32 or bf16, both widened exactly to fp32).  Run once per weight update.
 */
engram_status engram_fuse_weight(const void *w_h, const void *w_k, engram_dtype dtype, float *w_fused,
                                 int32_t d, engram_stream_t stream);

/* ------------------------------------------------------------------------- */
/* B1: gate forward  (ch. 34 sec. 1.2 item 3, sec. 2.1, sec. 3.1-3.2)          */
/* ------------------------------------------------------------------------- */

/*
 * For each token t < T, with rows h_t, k_t, v_t of length d in `dtype` and
 * s = 1/sqrt(d):
 *     rstd_h = 1/sqrt(sum_i h_i^2 / d + eps),  rstd_k likewise,
 *     dot    = sum_i h_i * w_fused_i * k_i,
 *     alpha  = sigmoid(s * rstd_h * rstd_k * dot),
 *     out_t  = alpha * v_t     (in `dtype`, rounded to nearest even for bf16).
 * All arithmetic is fp32.  alpha, rstd_h, rstd_k and dot are [T] fp32 and are
 * saved for the backward; each may be NULL (inference needs none of them).
 * out may not alias h, k or v.
 */
engram_status engram_gate_fwd(const void *h, const void *k, const void *v, engram_dtype dtype,
                              const float *w_fused, int64_t T, int32_t d, float eps,
                              void *out, float *alpha, float *rstd_h, float *rstd_k, float *dot,
                              engram_stream_t stream);

/*
 * engram_gate_fwd with the fold of engram_fuse_weight done in the forward's weight preload (ch. 34
 * sec. 3.1): w_h and w_k [d] in w_dtype (fp32 or bf16) replace w_fused, every CTA forms its slice
 * of w_h (*) w_k in fp32 exactly as engram_fuse_weight rounds it, and w_fused_out [d] fp32
 * (nullable) receives that fold for the backward.  Outputs are bitwise those of engram_fuse_weight
 * followed by engram_gate_fwd; one launch instead of two, for the first forward after a weight
 * update.  T = 0 writes only w_fused_out.  w_h, w_k, w_fused_out 16-byte aligned device memory.
 */
engram_status engram_gate_fwd_fold(const void *h, const void *k, const void *v, engram_dtype dtype,
                                   const void *w_h, const void *w_k, engram_dtype w_dtype, int64_t T, int32_t d,
                                   float eps, void *out, float *alpha, float *rstd_h, float *rstd_k, float *dot,
                                   float *w_fused_out, engram_stream_t stream);

/*
 * engram_gate_fwd, plus the RMS statistic of every output row as stored (after its rounding to
 * `dtype`), for the RMSNorm that reads the gate's output next (the short convolution, ch. 34
 * sec. 1.2 item 4):
 *     out_rstd[t] = 1/sqrt(sum_i out_t,i^2 / d + out_eps)      (out_rstd [T] fp32, not NULL)
 * The sum adds each thread's squares in element order, a 32-lane butterfly per warp, then the
 * warps in order: it depends on d only.  The other outputs are bitwise those of engram_gate_fwd.
 * engram_short_conv_fwd_given_rstd takes out_rstd in place of its own statistic pass.
 */
engram_status engram_gate_fwd_rms(const void *h, const void *k, const void *v, engram_dtype dtype,
                                  const float *w_fused, int64_t T, int32_t d, float eps,
                                  void *out, float *alpha, float *rstd_h, float *rstd_k, float *dot,
                                  float *out_rstd, float out_eps, engram_stream_t stream);

/* ------------------------------------------------------------------------- */
/* B2: gate backward  (ch. 34 sec. 4.1-4.2)                                   */
/* ------------------------------------------------------------------------- */

/*
 * The recommended number of weight-gradient partials P for (T, d).  A function
 * of T and d only (never of the GPU), so the partials and the reduced gradient
 * are bitwise reproducible on any device.  Host only.
 */
engram_status engram_gate_bwd_num_partials(int64_t T, int32_t d, int32_t *P);

/*
 * Given dout = dL/dout [T, d] and the forward's saved alpha, rstd_h, rstd_k,
 * dot [T] (fp32), with w = w_fused and s = 1/sqrt(d), for each token:
 *     dv     = alpha * dout
 *     dalpha = sum_i dout_i v_i
 *     c      = dalpha * alpha * (1 - alpha) * s * rstd_h * rstd_k
 *     dh_i   = c * (w_i k_i - dot * rstd_h^2 * h_i / d)
 *     dk_i   = c * (w_i h_i - dot * rstd_k^2 * k_i / d)
 * and the weight-gradient partials
 *     dw_partial[p, i] = sum over t in [p*C, min(T, (p+1)*C)) of c_t h_t,i k_t,i,
 * C = ceil(T / P), tokens summed in ascending order (a partial with no token is 0).
 * dh, dk, dv are [T, d] in `dtype`; dw_partial is [P, d] fp32, P >= 1.
 * Outputs may not alias inputs.
 */
engram_status engram_gate_bwd(const void *dout, const void *h, const void *k, const void *v, engram_dtype dtype,
                              const float *w_fused, const float *alpha, const float *rstd_h,
                              const float *rstd_k, const float *dot, int64_t T, int32_t d,
                              void *dh, void *dk, void *dv, float *dw_partial, int32_t P,
                              engram_stream_t stream);

/*
 * engram_gate_bwd for gradient accumulation over micro-batches (ch. 34 sec. 4.3-4.4: the
 * partials feed one reduction, whose result accumulates like a main_grad buffer).  Arguments,
 * layouts and checks are those of engram_gate_bwd; dh, dk, dv are written the same way, but each
 * partial row is added to instead of overwritten:
 *     dw_partial[p, i] = dw_partial[p, i] + c_t h_t,i k_t,i + ... over t in [p*C, min(T, (p+1)*C))
 * in ascending token order, starting from the row's current value (a partial with no token keeps
 * its row).  Calls in stream order on one [P, d] array, the first of them engram_gate_bwd, so
 * give bitwise reproducible partials; one engram_grad_w_reduce over those P rows then reduces
 * every micro-batch at once.  P must be the same in every call on the array.
 */
engram_status engram_gate_bwd_accumulate(const void *dout, const void *h, const void *k, const void *v,
                                         engram_dtype dtype, const float *w_fused, const float *alpha,
                                         const float *rstd_h, const float *rstd_k, const float *dot, int64_t T,
                                         int32_t d, void *dh, void *dk, void *dv, float *dw_partial, int32_t P,
                                         engram_stream_t stream);

/* ------------------------------------------------------------------------- */
/* B3: weight-gradient reduction  (ch. 34 sec. 4.3-4.4; determinism: the DSL article's
 *     "partitioned writes plus one ordered reduction instead of atomics")      */
/* ------------------------------------------------------------------------- */

/*
 * S = sum over p < P of dw_partial[p, :] in a fixed order that depends on P only
 * (bitwise reproducible).  dweight_fused (nullable) receives S.  When the four
 * weight pointers are given (all or none):
 *     grad_w_h += S * w_k,   grad_w_k += S * w_h     (accumulate, like a main_grad buffer)
 * w_h, w_k, grad_w_h, grad_w_k are [d] fp32.  At least one output must be given.
 */
engram_status engram_grad_w_reduce(const float *dw_partial, int32_t P, int32_t d, float *dweight_fused,
                                   const float *w_h, const float *w_k, float *grad_w_h, float *grad_w_k,
                                   engram_stream_t stream);

/* ------------------------------------------------------------------------- */
/* The multi-branch gate of the TileKernels release  (ch. 34 sec. 2.1, 3.2, 4.2) */
/* ------------------------------------------------------------------------- */

/*
 * hc branches (hc = 1, 2 or 4; the release fixes 4) share one value row.  x is [T, hc, d],
 * kv is [T, hc+1, d] (rows 0..hc-1 the branch keys, row hc the shared value), w_fused is
 * [hc, d] fp32 (engram_fuse_weight over hc*d elements).  For branch h of token t, s = 1/sqrt(d):
 *     rstd_x = 1/sqrt(sum_i x_i^2 / d + eps),  rstd_k likewise over the key row,
 *     dot    = sum_i x_i w_fused[h, i] k_i,     z = s * rstd_x * rstd_k * dot,
 *     gate   = sigmoid(sign(z) * sqrt(max(|z|, clamp_value)))   (sign(+0) = +),
 *     out    = x + gate * v.
 * gate, rstd_x, rstd_k, dot are [T, hc] fp32, each nullable.  out may equal x (in-place
 * writing) only when no statistic is saved: a backward needs the original x, so that
 * combination is refused (ENGRAM_ERR_SHAPE).  Rows up to ENGRAM_MAX_ROW_BYTES: a token whose
 * (2 hc + 1) rows fit twice in shared memory, with d at most 4096 bf16 / 2048 fp32 elements for
 * hc = 4 (twice / four times that for hc = 2 / 1), runs in one CTA; a larger one (d = 7168 bf16
 * at hc = 4, the release's width, among them) in a cluster of two CTAs that each hold half of
 * every row (engram_set_hc_split).
 */
engram_status engram_gate_hc_fwd(const void *x, const void *kv, engram_dtype dtype, const float *w_fused,
                                 int64_t T, int32_t hc, int32_t d, float eps, float clamp_value, void *out,
                                 float *gate, float *rstd_x, float *rstd_k, float *dot, engram_stream_t stream);

/*
 * Backward of engram_gate_hc_fwd given dout = dL/dout [T, hc, d] and the saved statistics:
 *     dgate_h = sum_i dout_h,i v_i
 *     c_h     = 0 where |z_h| < clamp_value (the clamp holds the gate constant), else
 *               dgate_h gate_h (1 - gate_h) / (2 sqrt|z_h|) * s rstd_x rstd_k      (= dL/d dot_h)
 *     dx_h    = dout_h + c_h (w_h k_h - dot_h rstd_x^2 x_h / d)
 *     dk_h    = c_h (w_h x_h - dot_h rstd_k^2 k_h / d)
 *     dv      = sum_h gate_h dout_h
 * dx is [T, hc, d]; dkv is [T, hc+1, d] (row hc = dv).  dw_partial is [P, hc, d] fp32 with
 * partial p the sum of c_h x_h k_h over tokens [p*C, min(T, (p+1)*C)), C = ceil(T / P) --
 * reduce it with engram_grad_w_reduce over hc*d columns.
 * In-place writing: dx may be dout or x, and dkv may be kv (the same pointer, the same layout);
 * any other overlap between dx, dkv and the inputs is refused (ENGRAM_ERR_SHAPE).  The branch-by-
 * branch form (see engram_set_hc_split) takes dx over dout or dkv over kv, but not both in one
 * call: the value row's gradient reads dout and the branch kernels read the value row, so that
 * pair is refused there (ENGRAM_ERR_SHAPE) and served by the other two forms.
 */
engram_status engram_gate_hc_bwd(const void *dout, const void *x, const void *kv, engram_dtype dtype,
                                 const float *w_fused, const float *gate, const float *rstd_x,
                                 const float *rstd_k, const float *dot, int64_t T, int32_t hc, int32_t d,
                                 float clamp_value, void *dx, void *dkv, float *dw_partial, int32_t P,
                                 engram_stream_t stream);

/* ------------------------------------------------------------------------- */
/* The short convolution after the gate  (ch. 34 sec. 1.2 item 4)             */
/* ------------------------------------------------------------------------- */

/*
 * Y = SiLU(Conv1D(RMSNorm(V~))) + V~ and H <- H + Y, for V~ = the gate's output sequence [T, d].
 * With u = V~ * rstd * norm_w, rstd = 1/sqrt(sum_j V~_j^2 / d + eps), per token t and channel c:
 *     conv[t, c] = bias[c] + sum_{i < width} conv_w[c, i] * u[t - (width - 1 - i) * dilation, c]
 * where u is 0 before the start of t's sequence (sequences from seq_offsets, cu_seqlens style:
 * [num_seqs + 1] int64, 0 first, T last, non-decreasing), and
 *     out[t, c] = h[t, c] + SiLU(conv[t, c]) + V~[t, c]        (h nullable: then without it).
 * conv_w is [d, width] fp32 (torch's depthwise [d, 1, width] layout; tap width - 1 is the current
 * token), norm_w [d] and bias [d] (nullable) fp32.  width 1..4, dilation >= 1 (the pages: 4 and
 * the largest N-gram order).  rstd [T] fp32 is required: it is written and is the backward's
 * saved statistic.  v, h, out are [T, d] in `dtype`, rows a multiple of 16 bytes, d <= 8192,
 * 16-byte aligned; out may equal h (in place) but not v.
 */
engram_status engram_short_conv_fwd(const void *v, const void *h, engram_dtype dtype, const float *norm_w,
                                    const float *conv_w, const float *bias, const int64_t *seq_offsets,
                                    int32_t num_seqs, int64_t T, int32_t d, int32_t width, int32_t dilation,
                                    float eps, void *out, float *rstd, engram_stream_t stream);

/*
 * engram_short_conv_fwd with rstd [T] given (read, not written): the statistic of V~ that
 * engram_gate_fwd_rms produced with V~, so that V~ is read once here instead of twice.  The same
 * conditions on the other arguments; the eps of the RMSNorm is the one rstd was made with.
 */
engram_status engram_short_conv_fwd_given_rstd(const void *v, const void *h, engram_dtype dtype,
                                               const float *norm_w, const float *conv_w, const float *bias,
                                               const int64_t *seq_offsets, int32_t num_seqs, int64_t T,
                                               int32_t d, int32_t width, int32_t dilation, const float *rstd,
                                               void *out, engram_stream_t stream);

/*
 * Weight-gradient partials of engram_short_conv_bwd: P = ceil(T / L) * dilation with
 * L = max(256, ceil(T / 256)) tokens per time chunk; one partial per (chunk, residue class of
 * t mod dilation).  Depends on T and dilation only.  Host only.
 */
engram_status engram_short_conv_num_partials(int64_t T, int32_t dilation, int32_t *P);

/*
 * Backward of engram_short_conv_fwd given dout = dL/dout [T, d] and its saved rstd; dL/dh = dout
 * (not written).  With dc = dout * SiLU'(conv) and, within each sequence,
 *     du[t, c] = sum_i conv_w[c, i] * dc[t + (width - 1 - i) * dilation, c],
 *     s[t]     = sum_c norm_w[c] du[t, c] V~[t, c],
 *     dv[t, c] = dout[t, c] + rstd norm_w[c] du[t, c] - rstd^3 V~[t, c] s[t] / d,
 * dv [T, d] in `dtype` (not aliasing v or dout) and dw_partial [P, width + 2, d] fp32 with
 * P = engram_short_conv_num_partials(T, dilation).  With u' = V~ rstd and A_i = the sum, over the
 * outputs t of work item (chunk, class) in ascending time order, of dc[t] u'[t - (width-1-i) dilation]:
 * row i (0..width-1) holds norm_w * A_i, row width the sum of dc, and row width + 1
 * sum_i conv_w[c, i] A_i (ascending i; summed over a sequence that is sum_t du V~ rstd, the chain
 * rule grouped the other way).  The convolution is recomputed with the norm weight folded into the
 * taps (conv_w[c, i] * norm_w[c], rounded once) and du carried as norm_w du.  Reduce the partials
 * with engram_short_conv_grad_reduce.  s sums, in this order: a thread's four channels as
 * (c0 + c2) + (c1 + c3); a warp's 32 threads (128 channels) as a butterfly pairing lanes 16, 8, 4,
 * 2, 1 apart; a 512-channel block's four warp sums as (w_0 + w_1) + (w_2 + w_3); then the
 * C = ceil(d / 512) block sums b_k pairwise: b_k + b_(k+8) first when C > 8, then
 * ((b_0 + b_1) + (b_2 + b_3)) + ((b_4 + b_5) + (b_6 + b_7)), absent blocks adding zero.  One pass
 * over dout and V~ on thread-block clusters of ceil(d / 512) CTAs; dout, v, dv and dw_partial
 * 16-byte aligned.
 */
engram_status engram_short_conv_bwd(const void *dout, const void *v, engram_dtype dtype, const float *norm_w,
                                    const float *conv_w, const float *bias, const float *rstd,
                                    const int64_t *seq_offsets, int32_t num_seqs, int64_t T, int32_t d,
                                    int32_t width, int32_t dilation, void *dv, float *dw_partial, int32_t P,
                                    engram_stream_t stream);

/*
 * dconv_w [d, width], dbias [d] (nullable) and dnorm_w [d] = the sums of the P partial rows of
 * engram_short_conv_bwd, in a fixed order that depends on P only (128 groups of ceil(P / 128) consecutive partials, each summed in ascending order; runs of 16
 * consecutive group sums, each in ascending order; then the 8 run sums in ascending order).
 * P = 0 writes zeros.  dw_partial 16-byte aligned; d a multiple of 4.
 */
engram_status engram_short_conv_grad_reduce(const float *dw_partial, int32_t P, int32_t width, int32_t d,
                                            float *dconv_w, float *dbias, float *dnorm_w, engram_stream_t stream);

/* ------------------------------------------------------------------------- */
/* The Engram Sinkhorn of the TileKernels release: row / column L2 scaling of a  */
/* [rows, head_dim] fp32 matrix  (ch. 34 sec. 5.3, the Engram version's four     */
/* kernels)                                                                      */
/* ------------------------------------------------------------------------- */

/*
 * Momentum update, in place on momentum [n] fp32, with grad [n] fp32 or bf16:
 *     m = beta1 * m + g;   sinkhorn_input = nesterov ? g + beta1 * m : m     (fp32 [n]).
 * The pages name the arguments (grad, momentum, beta1, nesterov) and the fp32 result, not the
 * update itself; this is the plain heavy-ball / Nesterov form.  sinkhorn_input may not alias
 * momentum.  All three pointers 16-byte aligned device memory; n == 0 is a no-op.
 */
engram_status engram_sinkhorn_momentum_update(const void *grad, engram_dtype dtype, float *momentum,
                                              float *sinkhorn_input, int64_t n, float beta1, int32_t nesterov,
                                              engram_stream_t stream);

/*
 * The number of column partials the library recommends for `rows` rows: about 16 or more rows
 * per partial and at most 1024 partials.  It depends on rows only, so the partials and their
 * reduction are bitwise reproducible on any device.  Host only.
 */
engram_status engram_sinkhorn_num_partials(int64_t rows, int32_t head_dim, int32_t *P);

/*
 * The row step over matrix [rows, head_dim] fp32 (row-major), row_scale [rows] and
 * col_scale [head_dim] fp32.  For each row r, with x = row_scale[r] * matrix[r, :] (*) col_scale:
 *     row_norm[r]  = ||x||_2                                  (row_norm nullable)
 *     row_scale[r] = row_scale[r] / (row_norm[r] + eps)       (in place)
 * and the column partials
 *     col_sumsq_partial[p, c] = sum over r in [p*C, min(rows, (p+1)*C)) of (x_c / (row_norm[r] + eps))^2,
 * C = ceil(rows / P), a partial with no row 0.  Summation order (fixed by rows and P only, so the
 * result is bitwise reproducible on any device): the rows at even offsets from p*C in ascending
 * order, the rows at odd offsets in ascending order, then the first sum plus the second.
 * col_sumsq_partial is [P, head_dim] fp32, P >= 1.  head_dim a multiple of 4 and at most 8192;
 * matrix, col_scale and col_sumsq_partial 16-byte aligned.  Outputs may not alias the matrix or col_scale.
 */
engram_status engram_sinkhorn_step(const float *matrix, float *row_scale, const float *col_scale, int64_t rows,
                                   int32_t head_dim, float eps, float *row_norm, float *col_sumsq_partial,
                                   int32_t P, engram_stream_t stream);

/*
 * col_sumsq[c] = sum over p < P of col_sumsq_partial[p, c] in a fixed order that depends on P
 * only (128 groups of ceil(P / 128) consecutive partials, each summed in ascending order; runs of 16
 * consecutive group sums, each in ascending order; then the 8 run sums in ascending order).  col_sumsq [head_dim] is nullable; when col_scale [head_dim] is
 * given, the column step of the alternating iteration is applied in place:
 *     col_scale[c] = col_scale[c] / (sqrt(col_sumsq[c]) + eps).
 * At least one of the two outputs must be given.  16-byte aligned device pointers.
 */
engram_status engram_sinkhorn_step_reduce(const float *col_sumsq_partial, int32_t P, int32_t head_dim,
                                          float *col_sumsq, float *col_scale, float eps, engram_stream_t stream);

/*
 * out[r, :] = alpha * x / (||x||_2 + eps), x = row_scale[r] * matrix[r, :] (*) col_scale:
 * out [rows, head_dim] fp32, not aliasing matrix.  Shape rules as for engram_sinkhorn_step;
 * rows == 0 is a no-op.
 */
engram_status engram_sinkhorn_finalize(const float *matrix, const float *row_scale, const float *col_scale,
                                       int64_t rows, int32_t head_dim, float eps, float alpha, float *out,
                                       engram_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Allocation-free backward + reduction                                       */
/* ------------------------------------------------------------------------- */

/* Bytes of weight-gradient partials that engram_gate_bwd_reduce_noalloc holds (16 MiB). */
#define ENGRAM_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * The paper has no counterpart to this entry point; it exists for callers that
 * cannot allocate device memory.  Examples: a program that has handed all device
 * memory to a framework's caching allocator or to an arena reserved at start-up,
 * where a raw cudaMalloc would fail or fragment that pool; and a serving loop that
 * forbids allocation once it runs, because cudaMalloc and cudaFree can synchronise
 * the device and stall every stream.
 *
 * It computes what engram_gate_bwd followed by engram_grad_w_reduce compute, with
 * P = engram_gate_bwd_num_partials(T, d): the same dh, dk, dv, dweight_fused
 * (nullable) and, when the four weight pointers are given, the same
 * accumulation into grad_w_h and grad_w_k.  Arguments have the meaning, layout
 * and ownership they have there; the caller still provides every input and
 * output.  Only the [P, d] fp32 partials move: they live in one array of
 * ENGRAM_NOALLOC_SCRATCH_BYTES that the library keeps on each device that
 * loads it, until the process exits.  The call allocates and frees nothing.
 *
 * Limits and rules:
 *   - Sizes whose partials need more than ENGRAM_NOALLOC_SCRATCH_BYTES
 *     (P * d * 4 bytes; e.g. T >= 9361 at d = 7168) are rejected with
 *     ENGRAM_ERR_SHAPE and a message; use engram_gate_bwd with a buffer then.
 *   - The first call on a device looks up the array's device address on that
 *     device (cudaGetSymbolAddress) and caches it: make that first call, with the
 *     device current, before any stream capture on it.  The cached address does
 *     not survive a cudaDeviceReset of that device: do not call this entry point
 *     (or any other of the library) on a device after resetting it.
 *   - All calls share the one array, which keeps whatever the last call left
 *     there.  Each call overwrites every partial row it reads, so nothing has to
 *     be cleared between calls, but calls that overlap on the GPU (other
 *     streams, other host threads) race on it: order them on one stream or
 *     synchronise between them.
 */
engram_status engram_gate_bwd_reduce_noalloc(const void *dout, const void *h, const void *k, const void *v,
                                             engram_dtype dtype, const float *w_fused, const float *alpha,
                                             const float *rstd_h, const float *rstd_k, const float *dot,
                                             int64_t T, int32_t d, void *dh, void *dk, void *dv,
                                             float *dweight_fused, const float *w_h, const float *w_k,
                                             float *grad_w_h, float *grad_w_k, engram_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ENGRAM_GB300_H */
