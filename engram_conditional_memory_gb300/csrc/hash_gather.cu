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
// Kernel layout for a table in device memory:
//   hash_gather_kernel (rows wanted): a persistent CTA walks tiles of consecutive tokens (~32 KB of
//      e_t rows, at most kTileMax tokens).  Its hash warp computes each tile's row numbers (lane =
//      token: the compressed window, the pad id 0 before the sequence's start found by a binary
//      search in the sequence offsets, every table's hash) into a ring of shared-memory slots, up to
//      kRowRing tiles ahead; its copy threads fetch every table row of a tile by one bulk
//      asynchronous copy (TMA, 1-D) into a double-buffered shared tile in e_t order, completing on
//      the tile's mbarrier, and when all have landed one thread stores the whole tile -- its e_t rows
//      are adjacent in the output -- with a single bulk copy.  The hashing of later tiles overlaps
//      the copies of the current one;
//   hash_index_kernel (the index output alone): one thread per token.
// Random 128-byte rows are where this beats 16-byte loads from every thread: the copy engine keeps
// far more rows in flight per SM than the load units can (measured: 53 us against 70 us for the
// 65,536-token, 16-table gather on GB300).  With a table in host memory, hash_gather_host_kernel
// keeps the tile hashing (tile_ids, tile_hash) and loads the rows over the host link.
#include <algorithm>

#include "engram_internal.cuh"

namespace engram {

constexpr int kTileMax = 32;           // tokens per tile at most
constexpr int kHashThreads = 256;      // copy threads of a gather CTA (all of a host-table CTA)
constexpr int kTileBytes = 32 * 1024;  // target bytes of e_t rows per tile
constexpr int kIndexThreads = 128;     // hash_index_kernel: one thread per token
constexpr int kSmemSeqs = 4096;        // sequence offsets staged in shared memory up to this count
constexpr int kMaxEtBytes = 64 * 1024; // largest e_t row (tables x row bytes) the kernel takes

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
    int32_t tile_tokens;   // tokens per tile (1..kTileMax)
    int32_t staged_seqs;   // 1 when the offsets are staged in shared memory
    int8_t order[ENGRAM_MAX_TABLES];
    uint64_t prime[ENGRAM_MAX_TABLES];
    uint64_t prime_inv[ENGRAM_MAX_TABLES];  // floor((2^64 - 1) / prime): Barrett reduction
    int64_t row_off[ENGRAM_MAX_TABLES];
    uint64_t mult[ENGRAM_MAX_TABLES][ENGRAM_MAX_ORDER];
};

// Dynamic shared memory of a host-table CTA (hash_gather_host_kernel, which passes row_bytes 0: its
// rows go through registers, not tiles), laid out by the host and the kernel alike.
struct HashSmemLayout {
    uint32_t tiles;    // 2 tiles of e_t rows (tile_tokens x tables x row_bytes each), 128-byte aligned
    uint32_t rows;     // int64 [2][tile_tokens][tables] row numbers
    uint32_t offs;     // int64 [num_seqs + 1] staged offsets (or empty)
    uint32_t bars;     // 2 mbarriers
    uint32_t total;
};

__host__ __device__ inline HashSmemLayout hash_smem_layout(int tile_tokens, int tables, uint32_t row_bytes,
                                                          int staged_entries) {
    HashSmemLayout L;
    const uint32_t tile = static_cast<uint32_t>(tile_tokens) * tables * row_bytes;
    L.tiles = 0;
    L.rows = 2 * tile;
    L.offs = L.rows + 2u * tile_tokens * tables * 8u;
    L.bars = L.offs + static_cast<uint32_t>(staged_entries) * 8u;
    L.total = L.bars + 16u;
    return L;
}

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

// h mod p by Barrett reduction (P. Barrett, 1986) with inv = floor((2^64 - 1) / p): the quotient
// estimate q = floor(h inv / 2^64) lies in [floor(h / p) - 2, floor(h / p)], so h - q p is below 3p
// and at most two subtractions make it exact -- the same value as the % operator.
__device__ __forceinline__ uint64_t mod_prime(uint64_t h, uint64_t p, uint64_t inv) {
    uint64_t r = h - __umul64hi(h, inv) * p;
    if (r >= p) r -= p;
    if (r >= p) r -= p;
    return r;
}

struct TileIds {
    int32_t cid[2][kTileMax + ENGRAM_MAX_ORDER];
    int64_t start[2][kTileMax];
};

// Step 1 for tile `tile` into buffer `b`: compressed ids of positions t0 - back .. t0 + ntok - 1
// and the sequence start of each token.
__device__ __forceinline__ void tile_ids(const HashGatherParams &p, const int64_t *offs, TileIds &st, int b,
                                         int64_t tile, int tid) {
    const int back = p.max_order - 1;
    const int64_t t0 = tile * p.tile_tokens;
    const int ntok = static_cast<int>(p.T - t0 < p.tile_tokens ? p.T - t0 : p.tile_tokens);
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
    if (tid >= kHashThreads - kTileMax) {
        const int i = tid - (kHashThreads - kTileMax);
        if (i < ntok) st.start[b][i] = sequence_start(offs, p.num_seqs, t0 + i);
    }
}

// Step 2 for tile `tile` from buffer `b`: one hash per (token, table) into rows[b].
__device__ __forceinline__ void tile_hash(const HashGatherParams &p, const TileIds &st, int64_t *rows, int b,
                                          int64_t tile, int tid) {
    const int back = p.max_order - 1;
    const int64_t t0 = tile * p.tile_tokens;
    const int ntok = static_cast<int>(p.T - t0 < p.tile_tokens ? p.T - t0 : p.tile_tokens);
    int64_t *r = rows + static_cast<size_t>(b) * p.tile_tokens * p.tables;
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
        const uint64_t idx = mod_prime(h, p.prime[tb], p.prime_inv[tb]);
        r[e] = p.row_off[tb] + static_cast<int64_t>(idx);
        if (p.out_idx) p.out_idx[t * p.tables + tb] = static_cast<int32_t>(idx);
    }
}

__device__ __forceinline__ void bulk_store_commit(void *dst_gmem, const void *src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst_gmem),
                 "r"(smem_addr(src_smem)), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until no committed bulk store still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Index of a token in table tb: the multiply-XOR hash of its compressed window, reduced mod the prime.
// The multipliers of a table beyond its order are zero (set so on the host), so every table runs
// the kernel-wide max_order terms and the extra ones add nothing; compressed ids are below 2^31, so
// each product is a 32 x 64-bit multiply.
__device__ __forceinline__ uint64_t table_index(const HashGatherParams &p, const uint32_t (&cid)[ENGRAM_MAX_ORDER],
                                                int tb) {
    uint64_t h = 0;
#pragma unroll
    for (int j = 0; j < ENGRAM_MAX_ORDER; ++j) {
        if (j >= p.max_order) break;
        h ^= static_cast<uint64_t>(cid[j]) * p.mult[tb][j];
    }
    return mod_prime(h, p.prime[tb], p.prime_inv[tb]);
}

// Steps 1-2 for token t: its compressed window (the pad id 0 before its sequence's start) and the
// index of tables tb_first, tb_first + tb_step, ..., the tables in one order on every lane so that a
// warp reads each table's constants once; the absolute row numbers row_off[table] + index go to
// dst[table] when dst is given, the indices to the optional index output.  An invalid id is
// reported by the token that holds it.
__device__ __forceinline__ void token_rows(const HashGatherParams &p, const int64_t *offs, int64_t t, int64_t *dst,
                                           int tb_first = 0, int tb_step = 1) {
    const int64_t s0 = sequence_start(offs, p.num_seqs, t);
    uint32_t cid[ENGRAM_MAX_ORDER];
#pragma unroll
    for (int j = 0; j < ENGRAM_MAX_ORDER; ++j) {
        cid[j] = 0;
        const int64_t q = t - j;
        if (j < p.max_order && q >= s0) {
            const int32_t raw = __ldg(p.ids + q);
            if (raw < 0 || raw >= p.vocab) {
                if (j == 0) report(p.status, p.err_word, ENGRAM_DEVERR_TOKEN_ID);
            } else {
                const int32_t id = p.cmap ? __ldg(p.cmap + raw) : raw;
                if (id < 0 || id >= p.vocab_c) {
                    if (j == 0) report(p.status, p.err_word, ENGRAM_DEVERR_COMPRESSED);
                } else {
                    cid[j] = static_cast<uint32_t>(id);
                }
            }
        }
    }
#pragma unroll 4
    for (int tb = tb_first; tb < p.tables; tb += tb_step) {
        const uint64_t idx = table_index(p, cid, tb);
        if (dst) dst[tb] = p.row_off[tb] + static_cast<int64_t>(idx);
        if (p.out_idx) p.out_idx[t * p.tables + tb] = static_cast<int32_t>(idx);
    }
}

// Checks, in block 0, that 0 = o_0 <= o_1 <= ... <= o_S = T.
__device__ __forceinline__ void check_offsets(const HashGatherParams &p, const int64_t *offs) {
    if (blockIdx.x != 0) return;
    for (int s = threadIdx.x; s <= p.num_seqs; s += blockDim.x) {
        const int64_t o = offs[s];
        bool bad = (s == 0 && o != 0) || (s == p.num_seqs && o != p.T) || o < 0 || o > p.T;
        if (s > 0 && offs[s - 1] > o) bad = true;
        if (bad) report(p.status, p.err_word, ENGRAM_DEVERR_SEQ_OFFSETS);
    }
}

// Steps 1-2 alone, for the index output without rows: one thread per token.
__global__ void __launch_bounds__(kIndexThreads) hash_index_kernel(const __grid_constant__ HashGatherParams p) {
    pdl_wait();  // the previous kernel's writes are complete and visible
    extern __shared__ __align__(16) int64_t so[];
    const int64_t *offs = p.seq_offsets;
    if (p.staged_seqs) {  // the sequence offsets in shared memory when they fit
        for (int s = threadIdx.x; s <= p.num_seqs; s += blockDim.x) so[s] = p.seq_offsets[s];
        offs = so;
        __syncthreads();
    }
    check_offsets(p, offs);
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < p.T;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x)
        token_rows(p, offs, t, nullptr);
}

// ---- steps 1-3 in one persistent kernel: a hash warp and the copy threads

constexpr int kRowRing = 4;                        // tiles of row numbers the hash warp may run ahead
constexpr int kGatherThreads = kHashThreads + 32;  // the copy threads, then the hash warp
constexpr int kGatherSeqs = 512;                   // sequence offsets staged in shared memory up to this count

// Dynamic shared memory of hash_gather_kernel, laid out by the host and the kernel alike.
struct GatherSmemLayout {
    uint32_t tiles;    // 2 tiles of e_t rows (tile_tokens x tables x row_bytes each)
    uint32_t rows;     // int64 [kRowRing][tile_tokens][tables] row numbers
    uint32_t offs;     // int64 [num_seqs + 1] staged offsets (or empty)
    uint32_t bars;     // mbarriers: 2 tiles landed, kRowRing row numbers ready, kRowRing row numbers read
    uint32_t total;
};

__host__ __device__ inline GatherSmemLayout gather_smem_layout(int tile_tokens, int tables, uint32_t row_bytes,
                                                              int staged_entries) {
    GatherSmemLayout L;
    const uint32_t tile = static_cast<uint32_t>(tile_tokens) * tables * row_bytes;
    L.tiles = 0;
    L.rows = 2 * tile;
    L.offs = L.rows + static_cast<uint32_t>(kRowRing) * tile_tokens * tables * 8u;
    L.bars = L.offs + static_cast<uint32_t>(staged_entries) * 8u;
    L.total = L.bars + (2u + 2u * kRowRing) * 8u;
    return L;
}

// Named barrier 1 over the copy threads alone (the hash warp never takes part): true on every
// copy thread when `v` holds on any.
__device__ __forceinline__ bool copy_threads_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "n"(kHashThreads)
        : "memory");
    return r != 0;
}

// Steps 1-3.  A persistent CTA walks tiles of consecutive tokens (tile, tile + gridDim.x, ...).
//   The hash warp (lane = token of the tile, token_rows) writes each tile's absolute row numbers
//   into a ring of kRowRing slots, up to kRowRing tiles ahead, and marks the slot ready.
//   The copy threads take a tile's row numbers, fetch every table row with one bulk asynchronous
//   copy (TMA, 1-D) into a double-buffered shared tile in e_t order, completing on the tile's
//   mbarrier, release the slot, and one thread stores the landed tile's adjacent e_t rows with a
//   single bulk copy.
// So the hashing runs beside the copies instead of before them.  All waits are bounded.
__global__ void __launch_bounds__(kGatherThreads) hash_gather_kernel(const __grid_constant__ HashGatherParams p) {
    pdl_wait();  // the previous kernel's writes are complete and visible
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int staged = p.staged_seqs ? p.num_seqs + 1 : 0;
    const GatherSmemLayout L = gather_smem_layout(p.tile_tokens, p.tables, p.row_bytes, staged);
    uint8_t *tiles = smem + L.tiles;
    int64_t *rows = reinterpret_cast<int64_t *>(smem + L.rows);
    int64_t *so = reinterpret_cast<int64_t *>(smem + L.offs);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L.bars);  // [2] a tile's rows have landed
    uint64_t *rows_full = bar + 2;                                  // [kRowRing] a slot's row numbers are ready
    uint64_t *rows_empty = rows_full + kRowRing;                    // [kRowRing] a slot's row numbers were read
    const int64_t ntiles = (p.T + p.tile_tokens - 1) / p.tile_tokens;
    const uint32_t et_bytes = static_cast<uint32_t>(p.tables) * p.row_bytes;  // one token's e_t row
    const uint32_t tile_bytes = static_cast<uint32_t>(p.tile_tokens) * et_bytes;
    const int slot_words = p.tile_tokens * p.tables;
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        for (int i = 0; i < kRowRing; ++i) {
            mbar_init(&rows_full[i], 1);
            mbar_init(&rows_empty[i], kHashThreads);
        }
        mbar_init_fence();
    }
    const int64_t *offs = p.seq_offsets;
    if (p.staged_seqs) {
        for (int s = tid; s <= p.num_seqs; s += blockDim.x) so[s] = p.seq_offsets[s];
        offs = so;
    }
    __syncthreads();
    check_offsets(p, offs);

    if (tid >= kHashThreads) {
        // ---- the hash warp, from the CTA's second tile on
        const int lane = tid - kHashThreads;
        int k = 1;
        for (int64_t tile = blockIdx.x + gridDim.x; tile < ntiles; tile += gridDim.x, ++k) {
            const int slot = k & (kRowRing - 1);
            if (k >= kRowRing) {  // the slot's previous tile was read by every copy thread
                bool ok = true;
                if (lane == 0) ok = mbar_wait_sleep(&rows_empty[slot], static_cast<uint32_t>((k / kRowRing - 1) & 1));
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    if (lane == 0) report(p.status, p.err_word, ENGRAM_DEVERR_TIMEOUT);
                    break;
                }
            }
            const int64_t t0 = tile * p.tile_tokens;
            const int ntok = static_cast<int>(p.T - t0 < p.tile_tokens ? p.T - t0 : p.tile_tokens);
            if (lane < ntok) token_rows(p, offs, t0 + lane, rows + static_cast<size_t>(slot) * slot_words + lane * p.tables);
            __syncwarp();  // every lane's row numbers before the release
            if (lane == 0) mbar_arrive(&rows_full[slot]);
        }
        return;
    }

    // ---- the copy threads: tile k's copies are issued before tile k - 1 is waited for and stored, so
    // two tiles are in flight
    bool failed = false;
    int k = 0;
    int pend_k = -1;         // (thread 0) the tile issued last and not yet stored: its iteration,
    int64_t pend_t0 = 0;     // first token
    int pend_ntok = 0;       // and tokens
    // (thread 0) waits until tile kk has landed in buffer kk & 1 and stores it; false on a timeout
    auto land_and_store = [&](int kk, int64_t t0, int ntok) {
        const int bb = kk & 1;
        const uint32_t parity = static_cast<uint32_t>((kk >> 1) & 1);
        if (!mbar_wait(&bar[bb], parity)) {
            report(p.status, p.err_word, ENGRAM_DEVERR_TIMEOUT);
            // the copies into this CTA's shared memory may still be in flight: wait once more
            if (!mbar_wait(&bar[bb], parity)) report(p.status, p.err_word, ENGRAM_DEVERR_TIMEOUT);
            return false;
        }
        bulk_store_commit(p.out_rows + static_cast<size_t>(t0) * et_bytes, tiles + static_cast<size_t>(bb) * tile_bytes,
                          static_cast<uint32_t>(ntok) * et_bytes);
        return true;
    };
    if (blockIdx.x < ntiles) {
        // the CTA's first tile is hashed by the copy warps themselves, so that its copies start
        // after two tables' hashes instead of all of them: warp w takes tables w, w + 8, ...
        const int warp = tid >> 5, lane = tid & 31;
        const int64_t t0 = static_cast<int64_t>(blockIdx.x) * p.tile_tokens;
        const int ntok = static_cast<int>(p.T - t0 < p.tile_tokens ? p.T - t0 : p.tile_tokens);
        if (lane < ntok) token_rows(p, offs, t0 + lane, rows + lane * p.tables, warp, kHashThreads / 32);
        copy_threads_any(false);  // every copy warp's row numbers are in slot 0
        if (tid == 0) mbar_arrive(&rows_full[0]);
    }
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k) {
        const int b = k & 1, slot = k & (kRowRing - 1);
        const int64_t t0 = tile * p.tile_tokens;
        const int ntok = static_cast<int>(p.T - t0 < p.tile_tokens ? p.T - t0 : p.tile_tokens);
        uint8_t *tl = tiles + static_cast<size_t>(b) * tile_bytes;
        const int ncopies = ntok * p.tables;

        const bool got = mbar_wait_sleep(&rows_full[slot], static_cast<uint32_t>((k / kRowRing) & 1));
        // buffer b held tile k - 2, whose store was issued in the previous iteration: once that store
        // has read it, refill it
        if (tid == 0) {
            bulk_wait_read_all();
            if (got) mbar_arrive_expect_tx(&bar[b], static_cast<uint32_t>(ncopies) * p.row_bytes);
        }
        if (copy_threads_any(!got)) {
            if (tid == 0) report(p.status, p.err_word, ENGRAM_DEVERR_TIMEOUT);
            failed = true;
            break;
        }
        const int64_t *r = rows + static_cast<size_t>(slot) * slot_words;
        for (int e = tid; e < ncopies; e += kHashThreads)
            bulk_load_plain(tl + static_cast<size_t>(e) * p.row_bytes,
                            p.table + static_cast<size_t>(r[e]) * p.row_bytes, p.row_bytes, &bar[b]);
        mbar_arrive(&rows_empty[slot]);  // this thread has read its row numbers from the slot

        if (tid == 0) {
            if (pend_k >= 0 && !land_and_store(pend_k, pend_t0, pend_ntok)) failed = true;
            pend_k = k, pend_t0 = t0, pend_ntok = ntok;
        }
        if (copy_threads_any(failed)) break;
    }
    if (tid == 0) {
        // the last tile (after a failure: only wait for its copies)
        if (pend_k >= 0) {
            if (failed) {
                const uint32_t parity = static_cast<uint32_t>((pend_k >> 1) & 1);
                if (!mbar_wait(&bar[pend_k & 1], parity)) report(p.status, p.err_word, ENGRAM_DEVERR_TIMEOUT);
            } else {
                land_and_store(pend_k, pend_t0, pend_ntok);
            }
        }
        bulk_wait_all();  // every store has completed before the CTA's shared memory goes away
    }
}

// The same hash + gather with the table in page-locked host memory (NEXT-3: the paper's offload
// of the tables to host memory, possible because the rows a token needs follow from its ids
// alone).  Rows cross the host link with plain 16-byte loads through the table's device-mapped
// address -- 8 threads per 128-byte row, kBatch vectors in flight per thread -- issued before the
// next tile is hashed so that the link's latency overlaps the hashing; each tile's e_t rows are
// then written to device memory in one contiguous block.
constexpr int kBatch = 16;

__global__ void __launch_bounds__(kHashThreads, 2) hash_gather_host_kernel(const __grid_constant__ HashGatherParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ TileIds st;

    const int tid = threadIdx.x;
    const int staged_entries = p.staged_seqs ? p.num_seqs + 1 : 0;
    const HashSmemLayout L = hash_smem_layout(p.tile_tokens, p.tables, 0u, staged_entries);  // no tiles
    int64_t *rows = reinterpret_cast<int64_t *>(smem + L.rows);
    const int64_t ntiles = (p.T + p.tile_tokens - 1) / p.tile_tokens;
    const uint32_t vpr = p.row_bytes / 16;                       // 16-byte vectors per table row
    const uint32_t vpt = vpr * static_cast<uint32_t>(p.tables);  // per token (one e_t row)

    const int64_t *offs = p.seq_offsets;
    if (p.staged_seqs) {
        int64_t *so = reinterpret_cast<int64_t *>(smem + L.offs);
        for (int s = tid; s <= p.num_seqs; s += kHashThreads) so[s] = p.seq_offsets[s];
        offs = so;
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
    if (tile < ntiles) {
        tile_ids(p, offs, st, 0, tile, tid);
        __syncthreads();
        tile_hash(p, st, rows, 0, tile, tid);
    }
    __syncthreads();

    for (int b = 0; tile < ntiles; tile += gridDim.x, b ^= 1) {
        const int64_t t0 = tile * p.tile_tokens;
        const int ntok = static_cast<int>(p.T - t0 < p.tile_tokens ? p.T - t0 : p.tile_tokens);
        const int64_t next = tile + gridDim.x;
        const uint32_t total = p.out_rows ? static_cast<uint32_t>(ntok) * vpt : 0u;
        uint8_t *dst = p.out_rows + static_cast<size_t>(t0) * vpt * 16;
        const int64_t *r = rows + static_cast<size_t>(b) * p.tile_tokens * p.tables;

        for (uint32_t base = 0; base < total || base == 0; base += kHashThreads * kBatch) {
            uint4 buf[kBatch];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const uint32_t e = base + k * kHashThreads + tid;
                if (e < total) {
                    const uint32_t i = e / vpt;
                    const uint32_t rr = e - i * vpt;
                    const uint32_t tb = rr / vpr;
                    const uint32_t piece = rr - tb * vpr;
                    buf[k] = *reinterpret_cast<const uint4 *>(
                        p.table + static_cast<size_t>(r[i * p.tables + tb]) * p.row_bytes + piece * 16);
                }
            }
            if (base == 0) {  // hash the next tile while the first batch crosses the link
                if (next < ntiles) tile_ids(p, offs, st, b ^ 1, next, tid);
                __syncthreads();
                if (next < ntiles) tile_hash(p, st, rows, b ^ 1, next, tid);
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const uint32_t e = base + k * kHashThreads + tid;
                if (e < total) st_global_v4(dst + static_cast<size_t>(e) * 16, buf[k]);
            }
            if (total == 0) break;
        }
        __syncthreads();  // rows[b] is rewritten two tiles from now; rows[b ^ 1] is complete
    }
}

}  // namespace engram

using namespace engram;

namespace {

// Host-side checks and kernel parameters shared by both entry points.  `host_table` selects a
// page-locked host table (whose device-mapped address replaces a->table in the parameters).
engram_status prepare_hash_gather(const engram_hash_spec *spec, const engram_hash_gather_args *a, bool host_table,
                                  HashGatherParams *pp, DeviceInfo *devp) {
    HashGatherParams &p = *pp;
    DeviceInfo &dev = *devp;
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
    if (row_bytes * tables > kMaxEtBytes)
        return fail(ENGRAM_ERR_SHAPE, "engram_hash_gather: e_t row of %lld bytes exceeds %d", (long long)(row_bytes * tables),
                    kMaxEtBytes);
    if (!aligned16(a->table) || (a->out_rows && !aligned16(a->out_rows)) || !aligned16(a->seq_offsets))
        return fail(ENGRAM_ERR_ALIGN, "engram_hash_gather: table, out_rows or seq_offsets not 16-byte aligned");

    p = HashGatherParams{};
    int64_t sum = 0;
    for (int tb = 0; tb < tables; ++tb) {
        const uint64_t pr = spec->primes[tb];
        if (pr == 0 || pr >= (1ull << 31)) return fail(ENGRAM_ERR_SHAPE, "engram_hash_gather: primes[%d] = %llu", tb,
                                                      (unsigned long long)pr);
        p.prime[tb] = pr;
        p.prime_inv[tb] = ~0ull / pr;
        p.row_off[tb] = sum;
        sum += static_cast<int64_t>(pr);
        p.order[tb] = static_cast<int8_t>(spec->min_order + tb / spec->heads);
        for (int j = 0; j < ENGRAM_MAX_ORDER; ++j)
            p.mult[tb][j] = j < p.order[tb] ? spec->multipliers[static_cast<int64_t>(tb) * spec->mult_stride + j] : 0;
    }
    if (sum > a->table_rows)
        return fail(ENGRAM_ERR_SHAPE, "engram_hash_gather: sum(primes) = %lld > table_rows = %lld", (long long)sum,
                    (long long)a->table_rows);

    engram_status st = current_device(&dev);
    if (st != ENGRAM_OK) return st;
    const void *ptrs[] = {a->token_ids, a->seq_offsets, a->compress_map, host_table ? nullptr : a->table,
                          a->out_indices, a->out_rows, a->err_word};
    const char *names[] = {"token_ids", "seq_offsets", "compress_map", "table", "out_indices", "out_rows",
                           "err_word"};
    for (int i = 0; i < 7; ++i)
        if ((st = check_device_ptr(ptrs[i], dev.device, names[i])) != ENGRAM_OK) return st;
    const void *table = a->table;
    if (host_table) {
        // Only page-locked host memory registered with CUDA is read (checked at every validation
        // level: pageable memory must never reach the kernel); then its device-side address.
        cudaPointerAttributes attr;
        cudaError_t e = cudaPointerGetAttributes(&attr, a->table);
        if (e != cudaSuccess || attr.type != cudaMemoryTypeHost) {
            cudaGetLastError();
            return fail(ENGRAM_ERR_DEVICE, "engram_hash_gather_host: table is not page-locked host memory");
        }
        void *dptr = nullptr;
        e = cudaHostGetDevicePointer(&dptr, const_cast<void *>(a->table), 0);
        if (e != cudaSuccess || !dptr) {
            cudaGetLastError();
            return fail(ENGRAM_ERR_DEVICE, "engram_hash_gather_host: table is not page-locked, mapped host memory (%s)",
                        cudaGetErrorString(e));
        }
        table = dptr;
    }

    p.ids = a->token_ids;
    p.seq_offsets = a->seq_offsets;
    p.cmap = a->compress_map;
    p.table = static_cast<const uint8_t *>(table);
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

    return ENGRAM_OK;
}

}  // namespace

extern "C" engram_status engram_hash_gather(const engram_hash_spec *spec, const engram_hash_gather_args *a,
                                            engram_stream_t stream) {
    HashGatherParams p;
    DeviceInfo dev;
    engram_status st = prepare_hash_gather(spec, a, false, &p, &dev);
    if (st != ENGRAM_OK) return st;
    const int tables = p.tables;
    const int64_t row_bytes = p.row_bytes;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!p.out_rows) {
        // the index output alone: one thread per token (>= 1 block: T = 0 still checks the offsets)
        const int64_t iblocks =
            std::max<int64_t>(1, std::min<int64_t>((a->T + kIndexThreads - 1) / kIndexThreads, 16LL * dev.num_sms));
        p.staged_seqs = a->num_seqs + 1 <= kSmemSeqs ? 1 : 0;
        const int ismem = p.staged_seqs ? (a->num_seqs + 1) * 8 : 0;
        if ((st = set_smem(reinterpret_cast<const void *>(hash_index_kernel), ismem)) != ENGRAM_OK) return st;
        cudaError_t le =
            launch_kernel(hash_index_kernel, dim3(static_cast<unsigned>(iblocks)), dim3(kIndexThreads), ismem, s, p);
        if (le != cudaSuccess) return fail(ENGRAM_ERR_CUDA, "engram_hash_gather launch: %s", cudaGetErrorString(le));
        return check_launch("engram_hash_gather");
    }
    // tiles of ~kTileBytes of e_t rows; persistent grid of as many CTAs as fit at once (>= 1 block:
    // T = 0 still checks the offsets)
    const int et_bytes = static_cast<int>(row_bytes) * tables;
    p.tile_tokens = std::min(kTileMax, std::max(1, kTileBytes / et_bytes));
    p.staged_seqs = a->num_seqs + 1 <= kGatherSeqs ? 1 : 0;
    const GatherSmemLayout L = gather_smem_layout(p.tile_tokens, tables, p.row_bytes, p.staged_seqs ? a->num_seqs + 1 : 0);
    const int dyn = static_cast<int>(L.total);
    if (dyn > dev.smem_optin) return fail(ENGRAM_ERR_SHAPE, "engram_hash_gather: %d bytes of shared memory needed", dyn);
    if ((st = set_smem(reinterpret_cast<const void *>(hash_gather_kernel), dyn)) != ENGRAM_OK) return st;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, hash_gather_kernel, kGatherThreads, dyn);
    if (e != cudaSuccess) return fail(ENGRAM_ERR_CUDA, "engram_hash_gather occupancy: %s", cudaGetErrorString(e));
    const int64_t ntiles = (a->T + p.tile_tokens - 1) / p.tile_tokens;
    int64_t grid = static_cast<int64_t>(dev.num_sms) * std::max(per_sm, 1);
    if (grid > ntiles) grid = ntiles;
    grid = cap_grid(std::max<int64_t>(grid, 1));
    cudaError_t le = launch_kernel(hash_gather_kernel, dim3(static_cast<unsigned>(grid)), dim3(kGatherThreads), dyn, s, p);
    if (le != cudaSuccess) return fail(ENGRAM_ERR_CUDA, "engram_hash_gather launch: %s", cudaGetErrorString(le));
    return check_launch("engram_hash_gather");
}

extern "C" engram_status engram_hash_gather_host(const engram_hash_spec *spec, const engram_hash_gather_args *a,
                                                 engram_stream_t stream) {
    HashGatherParams p;
    DeviceInfo dev;
    engram_status st = prepare_hash_gather(spec, a, true, &p, &dev);
    if (st != ENGRAM_OK) return st;
    // Tiles of kTileMax tokens (the e_t rows go through registers, not shared memory); persistent grid.
    p.tile_tokens = kTileMax;
    p.staged_seqs = a->num_seqs + 1 <= kSmemSeqs ? 1 : 0;
    const HashSmemLayout L = hash_smem_layout(p.tile_tokens, p.tables, 0u, p.staged_seqs ? a->num_seqs + 1 : 0);
    const int dyn = static_cast<int>(L.total);
    if ((st = set_smem(reinterpret_cast<const void *>(hash_gather_host_kernel), dyn)) != ENGRAM_OK) return st;
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, hash_gather_host_kernel, kHashThreads, dyn);
    if (e != cudaSuccess) return fail(ENGRAM_ERR_CUDA, "engram_hash_gather_host occupancy: %s", cudaGetErrorString(e));
    const int64_t ntiles = (a->T + p.tile_tokens - 1) / p.tile_tokens;
    int64_t grid = static_cast<int64_t>(dev.num_sms) * std::max(per_sm, 1);
    if (grid > ntiles) grid = ntiles;
    grid = cap_grid(grid);
    hash_gather_host_kernel<<<static_cast<unsigned>(grid), kHashThreads, dyn,
                              reinterpret_cast<cudaStream_t>(stream)>>>(p);
    return check_launch("engram_hash_gather_host");
}
