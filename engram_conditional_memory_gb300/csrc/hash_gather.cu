// A0 compression, A1 multi-head N-gram hash, A2 gather from the concatenated table.
//
// TileLang tutorial, ch. 34 "TileKernels: Engram and mHC":
//   sec. 1.2 item 1  tokenizer compression P: V -> V' (a surjection onto canonical ids);
//   sec. 1.2 item 2  K heads per N-gram order, each a multiplicative-XOR hash into a
//                    prime-sized table E_{n,k};
//   sec. 2.3         indices depend only on token ids; (max_n - 1) * heads rows per
//                    token whatever the table size; one concatenated table addressed
//                    through exclusive prefix-sum offsets.
// Hash form (the library's reading of "multiplicative-XOR"):
//   h = XOR_{j<n} (uint64) id'(t - j) * M[table][j]  (mod 2^64),  idx = h mod p[table],
//   id'(q) = pad id 0 for q before the start of t's sequence.
//
// Kernel layout: a persistent CTA walks tiles of kTile consecutive tokens, software-pipelined
// so that the next tile's hashing overlaps the current tile's row loads:
//   1. the compressed ids of the tile plus its (max_order - 1)-token look-back window and
//      every token's sequence start (a binary search in the sequence offsets, which are
//      staged in shared memory once per CTA when they fit) go to shared memory;
//   2. the tile's kTile x tables hashes are computed, one per thread, into a shared table
//      of row numbers (and the optional index output);
//   3. the tile's rows are gathered with 16-byte loads -- 8 consecutive threads per 128-byte
//      row, so each row is read as whole 32-byte sectors -- and written as one contiguous
//      block (the tile's e_t rows are adjacent).
// Steps 1-2 of tile i+1 run while the loads of step 3 of tile i are in flight.
#include <algorithm>

#include "engram_internal.cuh"

namespace engram {

constexpr int kTile = 32;            // tokens per tile
constexpr int kHashThreads = 256;    // threads per CTA
constexpr int kBatch = 16;           // 16-byte vectors in flight per thread
constexpr int kSmemSeqs = 4096;      // sequence offsets staged in shared memory up to this count

struct HashGatherParams {
    const int32_t *ids;
    const int64_t *seq_offsets;
    const int32_t *cmap;
    const uint8_t *table;
    uint8_t *out_rows;
    int32_t *out_idx;
    uint32_t *err_word;
    uint32_t *status;
    int64_t T;
    int32_t num_seqs;
    int32_t vocab;
    int32_t vocab_c;
    int32_t tables;
    int32_t max_order;
    uint32_t row_bytes;
    int8_t order[ENGRAM_MAX_TABLES];
    uint64_t prime[ENGRAM_MAX_TABLES];
    int64_t row_off[ENGRAM_MAX_TABLES];
    uint64_t mult[ENGRAM_MAX_TABLES][ENGRAM_MAX_ORDER];
};

// Start of the sequence holding token t: the last o_s <= t (upper bound search over
// offs[0..num_seqs]), clamped into [0, t] so that malformed offsets can never send a read
// out of range.
__device__ __forceinline__ int64_t sequence_start(const int64_t *offs, int32_t num_seqs, int64_t t) {
    int lo = 0, hi = num_seqs;  // invariant: answer in [lo, hi)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (offs[mid] <= t) lo = mid;
        else hi = mid;
    }
    int64_t s = offs[lo];
    if (s > t) s = t;
    if (s < 0) s = 0;
    return s;
}

struct TileState {
    int32_t cid[2][kTile + ENGRAM_MAX_ORDER];
    int64_t start[2][kTile];
    int64_t rows[2][kTile][ENGRAM_MAX_TABLES];
};

// Step 1 for tile `tile` into buffer `b`: compressed ids of positions t0 - back .. t0 + ntok - 1
// and the sequence start of each token.
__device__ __forceinline__ void tile_ids(const HashGatherParams &p, const int64_t *offs, TileState &st, int b,
                                         int64_t tile, int tid) {
    const int back = p.max_order - 1;
    const int64_t t0 = tile * kTile;
    const int ntok = static_cast<int>(p.T - t0 < kTile ? p.T - t0 : kTile);
    if (tid < ntok + back) {
        const int64_t q = t0 - back + tid;
        int32_t id = 0;
        if (q >= 0) {
            const int32_t raw = __ldg(p.ids + q);
            if (raw < 0 || raw >= p.vocab) {
                report(p.status, p.err_word, ENGRAM_DEVERR_TOKEN_ID);
            } else {
                id = p.cmap ? __ldg(p.cmap + raw) : raw;
                if (id < 0 || id >= p.vocab_c) {
                    report(p.status, p.err_word, ENGRAM_DEVERR_COMPRESSED);
                    id = 0;
                }
            }
        }
        st.cid[b][tid] = id;
    }
    if (tid >= kHashThreads - kTile) {
        const int i = tid - (kHashThreads - kTile);
        if (i < ntok) st.start[b][i] = sequence_start(offs, p.num_seqs, t0 + i);
    }
}

// Step 2 for tile `tile` from buffer `b`: one hash per (token, table).
__device__ __forceinline__ void tile_hash(const HashGatherParams &p, TileState &st, int b, int64_t tile, int tid) {
    const int back = p.max_order - 1;
    const int64_t t0 = tile * kTile;
    const int ntok = static_cast<int>(p.T - t0 < kTile ? p.T - t0 : kTile);
    for (int e = tid; e < ntok * p.tables; e += kHashThreads) {
        const int i = e / p.tables;
        const int tb = e - i * p.tables;
        const int64_t t = t0 + i;
        const int n = p.order[tb];
        uint64_t h = 0;
        for (int j = 0; j < n; ++j) {
            const uint64_t id = (t - j >= st.start[b][i]) ? static_cast<uint64_t>(st.cid[b][i + back - j]) : 0ull;
            h ^= id * p.mult[tb][j];
        }
        const uint64_t idx = h % p.prime[tb];
        st.rows[b][i][tb] = p.row_off[tb] + static_cast<int64_t>(idx);
        if (p.out_idx) p.out_idx[t * p.tables + tb] = static_cast<int32_t>(idx);
    }
}

__global__ void __launch_bounds__(kHashThreads, 2) hash_gather_kernel(const __grid_constant__ HashGatherParams p) {
    extern __shared__ __align__(16) int64_t smem_offs[];  // [num_seqs + 1] when staged
    __shared__ TileState st;

    const int tid = threadIdx.x;
    const int64_t ntiles = (p.T + kTile - 1) / kTile;
    const uint32_t vpr = p.row_bytes / 16;                       // 16-byte vectors per table row
    const uint32_t vpt = vpr * static_cast<uint32_t>(p.tables);  // per token (one e_t row)

    // Sequence offsets: staged in shared memory when they fit; one CTA also checks that
    // 0 = o_0 <= o_1 <= ... <= o_S = T.
    const bool staged = p.num_seqs + 1 <= kSmemSeqs;
    const int64_t *offs = p.seq_offsets;
    if (staged) {
        for (int s = tid; s <= p.num_seqs; s += kHashThreads) smem_offs[s] = p.seq_offsets[s];
        offs = smem_offs;
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int s = tid; s <= p.num_seqs; s += kHashThreads) {
            const int64_t o = offs[s];
            bool bad = (s == 0 && o != 0) || (s == p.num_seqs && o != p.T) || o < 0 || o > p.T;
            if (s > 0 && offs[s - 1] > o) bad = true;
            if (bad) report(p.status, p.err_word, ENGRAM_DEVERR_SEQ_OFFSETS);
        }
    }

    int64_t tile = blockIdx.x;
    int b = 0;
    if (tile < ntiles) {
        tile_ids(p, offs, st, 0, tile, tid);
        __syncthreads();
        tile_hash(p, st, 0, tile, tid);
    }
    __syncthreads();

    for (; tile < ntiles; tile += gridDim.x, b ^= 1) {
        const int64_t t0 = tile * kTile;
        const int ntok = static_cast<int>(p.T - t0 < kTile ? p.T - t0 : kTile);
        const int64_t next = tile + gridDim.x;
        const uint32_t total = p.out_rows ? static_cast<uint32_t>(ntok) * vpt : 0u;
        uint8_t *dst = p.out_rows + static_cast<size_t>(t0) * vpt * 16;

        // 3a. first batch of this tile's row loads (vector e = token e / vpt, table (e % vpt) / vpr)
        uint4 buf[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const uint32_t e = k * kHashThreads + tid;
            if (e < total) {
                const uint32_t i = e / vpt;
                const uint32_t r = e - i * vpt;
                const uint32_t tb = r / vpr;
                const uint32_t piece = r - tb * vpr;
                const uint8_t *src = p.table + static_cast<size_t>(st.rows[b][i][tb]) * p.row_bytes + piece * 16;
                buf[k] = __ldg(reinterpret_cast<const uint4 *>(src));
            }
        }
        // 1-2 of the next tile while those loads are in flight
        if (next < ntiles) tile_ids(p, offs, st, b ^ 1, next, tid);
        __syncthreads();
        if (next < ntiles) tile_hash(p, st, b ^ 1, next, tid);
        // 3b. store the first batch, then any further batches of this tile
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const uint32_t e = k * kHashThreads + tid;
            if (e < total) st_global_v4(dst + static_cast<size_t>(e) * 16, buf[k]);
        }
        for (uint32_t base = kHashThreads * kBatch; base < total; base += kHashThreads * kBatch) {
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const uint32_t e = base + k * kHashThreads + tid;
                if (e < total) {
                    const uint32_t i = e / vpt;
                    const uint32_t r = e - i * vpt;
                    const uint32_t tb = r / vpr;
                    const uint32_t piece = r - tb * vpr;
                    const uint8_t *src =
                        p.table + static_cast<size_t>(st.rows[b][i][tb]) * p.row_bytes + piece * 16;
                    buf[k] = __ldg(reinterpret_cast<const uint4 *>(src));
                }
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const uint32_t e = base + k * kHashThreads + tid;
                if (e < total) st_global_v4(dst + static_cast<size_t>(e) * 16, buf[k]);
            }
        }
        __syncthreads();  // buffer b is rewritten two tiles from now; b ^ 1 is complete
    }
}

}  // namespace engram

using namespace engram;

extern "C" engram_status engram_hash_gather(const engram_hash_spec *spec, const engram_hash_gather_args *a,
                                            engram_stream_t stream) {
    if (!spec || !a) return fail(ENGRAM_ERR_NULL, "engram_hash_gather: NULL argument");
    if (!spec->multipliers || !spec->primes) return fail(ENGRAM_ERR_NULL, "engram_hash_gather: NULL spec array");
    // token_ids and the outputs may be NULL only when there is no token.
    if ((!a->token_ids && a->T > 0) || !a->seq_offsets || !a->table)
        return fail(ENGRAM_ERR_NULL, "engram_hash_gather: NULL token_ids, seq_offsets or table");
    if (!a->out_rows && !a->out_indices && a->T > 0) return fail(ENGRAM_ERR_NULL, "engram_hash_gather: no output");
    const int64_t tables64 = static_cast<int64_t>(spec->num_orders) * spec->heads;
    const int max_order = spec->min_order + spec->num_orders - 1;
    if (spec->min_order < 1 || spec->num_orders < 1 || spec->heads < 1 || tables64 > ENGRAM_MAX_TABLES ||
        max_order > ENGRAM_MAX_ORDER || spec->mult_stride < max_order)
        return fail(ENGRAM_ERR_SHAPE, "engram_hash_gather: orders %d+%d, heads %d, stride %d", spec->min_order,
                    spec->num_orders, spec->heads, spec->mult_stride);
    const int tables = static_cast<int>(tables64);
    if (a->T < 0 || a->num_seqs < 1 || a->vocab < 1 || a->vocab_c < 1 || a->row_dim < 1 || a->table_rows < 0)
        return fail(ENGRAM_ERR_SHAPE, "engram_hash_gather: T %lld, num_seqs %d, vocab %d/%d, row_dim %d",
                    (long long)a->T, a->num_seqs, a->vocab, a->vocab_c, a->row_dim);
    if (!a->compress_map && a->vocab_c < a->vocab)
        return fail(ENGRAM_ERR_SHAPE, "engram_hash_gather: identity map needs vocab_c >= vocab");
    const int es = dtype_size(a->dtype);
    if (es == 0) return fail(ENGRAM_ERR_DTYPE, "engram_hash_gather: dtype %d", (int)a->dtype);
    const int64_t row_bytes = static_cast<int64_t>(a->row_dim) * es;
    if (row_bytes % 16 != 0) return fail(ENGRAM_ERR_ALIGN, "engram_hash_gather: row of %lld bytes", (long long)row_bytes);
    if (row_bytes * tables > (1 << 20)) return fail(ENGRAM_ERR_SHAPE, "engram_hash_gather: e_t row too long");
    if (!aligned16(a->table) || (a->out_rows && !aligned16(a->out_rows)) || !aligned16(a->seq_offsets))
        return fail(ENGRAM_ERR_ALIGN, "engram_hash_gather: table, out_rows or seq_offsets not 16-byte aligned");

    HashGatherParams p{};
    int64_t sum = 0;
    for (int tb = 0; tb < tables; ++tb) {
        const uint64_t pr = spec->primes[tb];
        if (pr == 0 || pr >= (1ull << 31)) return fail(ENGRAM_ERR_SHAPE, "engram_hash_gather: primes[%d] = %llu", tb,
                                                      (unsigned long long)pr);
        p.prime[tb] = pr;
        p.row_off[tb] = sum;
        sum += static_cast<int64_t>(pr);
        p.order[tb] = static_cast<int8_t>(spec->min_order + tb / spec->heads);
        for (int j = 0; j < ENGRAM_MAX_ORDER; ++j)
            p.mult[tb][j] = j < p.order[tb] ? spec->multipliers[static_cast<int64_t>(tb) * spec->mult_stride + j] : 0;
    }
    if (sum > a->table_rows)
        return fail(ENGRAM_ERR_SHAPE, "engram_hash_gather: sum(primes) = %lld > table_rows = %lld", (long long)sum,
                    (long long)a->table_rows);

    DeviceInfo dev;
    engram_status st = current_device(&dev);
    if (st != ENGRAM_OK) return st;
    const void *ptrs[] = {a->token_ids, a->seq_offsets, a->compress_map, a->table, a->out_indices, a->out_rows,
                          a->err_word};
    const char *names[] = {"token_ids", "seq_offsets", "compress_map", "table", "out_indices", "out_rows",
                           "err_word"};
    for (int i = 0; i < 7; ++i)
        if ((st = check_device_ptr(ptrs[i], dev.device, names[i])) != ENGRAM_OK) return st;

    p.ids = a->token_ids;
    p.seq_offsets = a->seq_offsets;
    p.cmap = a->compress_map;
    p.table = static_cast<const uint8_t *>(a->table);
    p.out_rows = static_cast<uint8_t *>(a->out_rows);
    p.out_idx = a->out_indices;
    p.err_word = a->err_word;
    p.status = dev.status_word;
    p.T = a->T;
    p.num_seqs = a->num_seqs;
    p.vocab = a->vocab;
    p.vocab_c = a->compress_map ? a->vocab_c : a->vocab;
    p.tables = tables;
    p.max_order = max_order;
    p.row_bytes = static_cast<uint32_t>(row_bytes);

    // Persistent grid: as many CTAs as fit on the device at once (>= 1: T = 0 still checks the offsets).
    const int dyn = a->num_seqs + 1 <= kSmemSeqs ? (a->num_seqs + 1) * static_cast<int>(sizeof(int64_t)) : 0;
    if ((st = set_smem(reinterpret_cast<const void *>(hash_gather_kernel), dyn)) != ENGRAM_OK) return st;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, hash_gather_kernel, kHashThreads, dyn);
    if (e != cudaSuccess) return fail(ENGRAM_ERR_CUDA, "engram_hash_gather occupancy: %s", cudaGetErrorString(e));
    const int64_t ntiles = (a->T + kTile - 1) / kTile;
    int64_t grid = static_cast<int64_t>(dev.num_sms) * std::max(per_sm, 1);
    if (grid > ntiles) grid = ntiles;
    grid = cap_grid(grid);
    hash_gather_kernel<<<static_cast<unsigned>(grid), kHashThreads, dyn, reinterpret_cast<cudaStream_t>(stream)>>>(p);
    return check_launch("engram_hash_gather");
}
