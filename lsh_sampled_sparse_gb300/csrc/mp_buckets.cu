// Bucketed hash tables in HBM: the retrieval structure of "MagicPIG: LSH Sampling for Efficient
// LLM Generation" (system co-design item 3: the query's codes are looked up in L prebuilt hash
// tables) and of "MagicPIG: don't pick the tallest" (section 6: every table stores a pointer to
// every key; a query scans about L n / 2^K entries).
//
// Layout per (sequence, KV head), in 32-bit words: offsets [L][2^K + 1], then members [L][n],
// then the build's scratch [L][kBucketRanges][2^K];
// members[t][offsets[t][c] .. offsets[t][c + 1]) are the keys whose table-t code is c. The order
// of keys inside a bucket is not fixed (buckets are sets); everything that reads them only counts.
//
// Build, one kernel: a cluster of R CTAs per (table, sequence x KV head), each CTA one key range
// (R = 1, 2, 4 or 8, so that a range holds about 12 blocks: short contexts take fewer, longer
// ranges and pay the per-range histogram work fewer times). A CTA stages its range's plane rows,
// decodes the codes of min(4, floor(32 / K)) 32-key words per warp bit transpose, counts them in
// a shared-memory histogram (the count's old value is the key's rank among the range's keys of
// that code), reads the other ranges' histograms through distributed shared memory to get the
// table's offsets and its own write base per code, sorts its keys by code in shared memory and
// writes them out in runs, so a bucket's part from one range is one contiguous store. Ranges too
// large for shared memory (very long contexts) take three kernels instead: per-range counts to
// the scratch words, one CTA per table scanning them into offsets and write bases, and a scatter
// with one shared atomic per key; the scratch [kBucketRanges][2^K] per table after the members
// serves them.
// Lookup: one warp per (query row, table) reads the query's bucket and sets each key's bit in
// two saturating bitmaps, ge1 (>= 1 table) and ge2 (>= 2 tables), stored in
// the selection-word layout of the dense scan ([row][block][32 words]).
#include <cooperative_groups.h>

#include "mp_internal.cuh"

namespace mp {
namespace {

constexpr int kBuildThreads = 256;
constexpr int kLookupWarps = 8;       // tables per lookup CTA, one warp each
constexpr int kLookupUnroll = 4;      // bucket entries a lookup lane loads before its atomics
constexpr int kStageBlocks = 4;       // 1024-key blocks whose plane rows a build CTA stages at once
constexpr size_t kClusterBuildSmem = 200 * 1024;   // dynamic shared memory of a cluster-build CTA
constexpr int kClusterThreads = 512;  // threads of a cluster-build CTA
constexpr int kMaxClusterRanges = 8;  // CTAs (key ranges) of a cluster-build table, at most
constexpr int kClusterRangeBlocks = 12;   // blocks a cluster-build range aims at
constexpr int kWordsAtOnce = 2;       // bit transposes a cluster-build warp runs together
constexpr int kStageRow = kWordsPerBlock + 1;   // staged plane row stride (words): lanes reading
                                                // word w of planes 0..K-1 hit distinct banks

// words per (sequence, KV head): offsets, members, then the build's per-range counts / bases
__host__ __device__ __forceinline__ size_t bucket_words(int n, int K, int L) {
    const size_t nb = static_cast<size_t>(1) << K;
    return static_cast<size_t>(L) * ((nb + 1) + static_cast<size_t>(n) + kBucketRanges * nb);
}

// Walk the keys of key range `range` of table t: stage kStageBlocks blocks' plane rows at a
// time (row stride kStageRow); then each warp takes 32-key words: lane p < K holds plane p's
// word, and one 32x32 bit transpose leaves in lane j the K-bit code of the word's key j.
// f(key, code) is called by the lane of every key (keys past n are skipped).
template <typename F>
__device__ __forceinline__ void for_range_keys(const uint32_t* codes, int bh, int t, int range,
                                              int n, int K, int L, int nblk, int cblk,
                                              uint32_t* stage,
                                              F&& f) {
    const int C = K * L, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b0 = (nblk * range) / kBucketRanges, b1 = (nblk * (range + 1)) / kBucketRanges;
    const int rowsz = K * kWordsPerBlock, srow = K * kStageRow;
    for (int blk = b0; blk < b1; blk += kStageBlocks) {
        const int nbk = min(kStageBlocks, b1 - blk);
        __syncthreads();                          // the previous stage is consumed
        for (int i = tid; i < nbk * rowsz; i += kBuildThreads) {
            const int kb = i / rowsz, w = i % rowsz;
            stage[kb * srow + (w / kWordsPerBlock) * kStageRow + w % kWordsPerBlock] =
                __ldcs(codes + (static_cast<size_t>(bh) * cblk + blk + kb) * C * kWordsPerBlock +
                       static_cast<size_t>(t) * rowsz + w);
        }
        __syncthreads();
        for (int wi = warp; wi < nbk * kWordsPerBlock; wi += kBuildThreads / 32) {
            const int kb = wi / kWordsPerBlock, w = wi % kWordsPerBlock;
            const uint32_t x = lane < K ? stage[kb * srow + lane * kStageRow + w] : 0u;
            const uint32_t code = warp_transpose32(x, lane);
            const int key = (blk + kb) * kKeysPerBlock + w * 32 + lane;
            if (key < n) f(key, code);
        }
    }
}

// 1. per key range: its count of every code -> scratch[t][range][c]
__global__ void __launch_bounds__(kBuildThreads)
    bucket_count_kernel(const uint32_t* codes, int n, int K, int L, int nblk, int cblk,
                        uint32_t* buckets) {
    extern __shared__ __align__(16) uint32_t sm[];
    const int nb = 1 << K, range = blockIdx.x, t = blockIdx.y, bh = blockIdx.z;
    uint32_t* hist = sm;
    uint32_t* stage = sm + nb;
    for (int c = threadIdx.x; c < nb; c += kBuildThreads) hist[c] = 0u;
    for_range_keys(codes, bh, t, range, n, K, L, nblk, cblk, stage,
                   [&](int, uint32_t c) { atomicAdd(&hist[c], 1u); });
    __syncthreads();
    uint32_t* scratch = buckets + static_cast<size_t>(bh) * bucket_words(n, K, L) +
                        static_cast<size_t>(L) * ((nb + 1) + static_cast<size_t>(n)) +
                        (static_cast<size_t>(t) * kBucketRanges + range) * nb;
    for (int c = threadIdx.x; c < nb; c += kBuildThreads) scratch[c] = hist[c];
}

// 2. per table: offsets = exclusive scan over codes of the total counts; each range's count is
//    replaced by its write base: offsets[c] + the counts of the lower ranges for code c
__global__ void __launch_bounds__(kBuildThreads)
    bucket_scan_kernel(int n, int K, int L, uint32_t* buckets) {
    __shared__ uint32_t wsum[kBuildThreads / 32];
    const int nb = 1 << K, t = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    uint32_t* base = buckets + static_cast<size_t>(bh) * bucket_words(n, K, L);
    uint32_t* offsets = base + static_cast<size_t>(t) * (nb + 1);
    uint32_t* scratch = base + static_cast<size_t>(L) * ((nb + 1) + static_cast<size_t>(n)) +
                        static_cast<size_t>(t) * kBucketRanges * nb;
    const int per = (nb + kBuildThreads - 1) / kBuildThreads;
    const int c0 = min(nb, tid * per), c1 = min(nb, c0 + per);
    uint32_t run = 0u;
    for (int c = c0; c < c1; ++c)
        for (int r = 0; r < kBucketRanges; ++r) run += scratch[r * nb + c];
    uint32_t incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    uint32_t acc = incl - run;
    for (int w = 0; w < warp; ++w) acc += wsum[w];
    for (int c = c0; c < c1; ++c) {
        offsets[c] = acc;
        for (int r = 0; r < kBucketRanges; ++r) {
            const uint32_t cnt = scratch[r * nb + c];
            scratch[r * nb + c] = acc;
            acc += cnt;
        }
    }
    if (tid == kBuildThreads - 1) offsets[nb] = acc;
}

// 3. per key range: every key to its bucket, from the range's base (cursors in shared memory)
__global__ void __launch_bounds__(kBuildThreads)
    bucket_scatter_kernel(const uint32_t* codes, int n, int K, int L, int nblk, int cblk,
                          uint32_t* buckets) {
    extern __shared__ __align__(16) uint32_t sm[];
    const int nb = 1 << K, range = blockIdx.x, t = blockIdx.y, bh = blockIdx.z;
    uint32_t* cursor = sm;
    uint32_t* stage = sm + nb;
    uint32_t* base = buckets + static_cast<size_t>(bh) * bucket_words(n, K, L);
    const uint32_t* scratch = base + static_cast<size_t>(L) * ((nb + 1) + static_cast<size_t>(n)) +
                              (static_cast<size_t>(t) * kBucketRanges + range) * nb;
    uint32_t* members = base + static_cast<size_t>(L) * (nb + 1) + static_cast<size_t>(t) * n;
    for (int c = threadIdx.x; c < nb; c += kBuildThreads) cursor[c] = scratch[c];
    for_range_keys(codes, bh, t, range, n, K, L, nblk, cblk, stage, [&](int key, uint32_t c) {
        members[atomicAdd(&cursor[c], 1u)] = static_cast<uint32_t>(key);
    });
}

// warp_transpose32 of U independent words, interleaved so that their shuffles overlap
template <int U>
__device__ __forceinline__ void warp_transpose32_x(uint32_t (&x)[U], int lane) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {                // s = 16, 8: whole bytes, one byte permute
        const int s = 16 >> i;
        const bool up = (lane & s) != 0;
        const uint32_t sel = i == 0 ? (up ? 0x3276u : 0x5410u) : (up ? 0x3715u : 0x6240u);
        uint32_t y[U];
#pragma unroll
        for (int u = 0; u < U; ++u) y[u] = __shfl_xor_sync(0xffffffffu, x[u], s);
#pragma unroll
        for (int u = 0; u < U; ++u) x[u] = __byte_perm(x[u], y[u], sel);
    }
    const uint32_t low[3] = {0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const int s = 4 >> i;
        const bool up = (lane & s) != 0;
        const uint32_t keep = up ? ~low[i] : low[i];
        uint32_t y[U];
#pragma unroll
        for (int u = 0; u < U; ++u) y[u] = __shfl_xor_sync(0xffffffffu, x[u], s);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t r = __funnelshift_l(y[u], y[u], up ? 32 - s : s);
            x[u] = (x[u] & keep) | (r & ~keep);
        }
    }
}

// Codes of staged 32-key words, P words per transposed 32x32 bit block (P K <= 32): lane
// l < P K loads plane l % K of word w + l / K, so after the transpose bits [q K, q K + K) of
// lane j are the code of key j of word w + q. Transposes u = 0 .. U-1 take words
// w0 + u P .. w0 + u P + P - 1 (words at or past nw give 0). Plane rows are kStageRow words
// apart, blocks srow words apart.
template <int U, int P>
__device__ __forceinline__ void staged_codes(const uint32_t* stage, int w0, int nw, int K,
                                             int srow, int lane, uint32_t (&x)[U]) {
    const int dw = lane / K, pl = lane - dw * K;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int wi = w0 + u * P + dw;
        x[u] = (dw < P && wi < nw)
                   ? stage[(wi / kWordsPerBlock) * srow + pl * kStageRow + wi % kWordsPerBlock]
                   : 0u;
    }
    warp_transpose32_x<U>(x, lane);
}

// Pass 1 of the cluster build for P words per transpose: every key's code, and its rank among
// the range's keys of that code (the histogram count before its own), as (code << 16) | rank.
// The U P atomics of a round are issued back to back.
template <int U, int P, int T>
__device__ __forceinline__ void count_codes(const uint32_t* stage, int nw, int m, int K, int srow,
                                            uint32_t* hist, uint32_t* crank) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t cmask = (1u << K) - 1u;
    for (int w0 = warp * U * P; w0 < nw; w0 += (T / 32) * U * P) {
        uint32_t x[U];
        staged_codes<U, P>(stage, w0, nw, K, srow, lane, x);
        uint32_t c[U][P], rk[U][P];
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int q = 0; q < P; ++q) {
                c[u][q] = (x[u] >> (q * K)) & cmask;
                rk[u][q] = (w0 + u * P + q) * 32 + lane < m ? atomicAdd(&hist[c[u][q]], 1u) : 0u;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int q = 0; q < P; ++q) {
                const int i = (w0 + u * P + q) * 32 + lane;
                if (i < m) crank[i] = (c[u][q] << 16) | rk[u][q];
            }
        }
    }
}

// In-place exclusive prefix sum of v[0, nb) by the whole CTA of T threads; wsum holds T / 32
// words. Ends with a barrier.
template <int T>
__device__ void block_exclusive_scan(uint32_t* v, int nb, uint32_t* wsum) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (nb + T - 1) / T;
    const int c0 = min(nb, tid * per), c1 = min(nb, c0 + per);
    uint32_t run = 0u;
    for (int c = c0; c < c1; ++c) run += v[c];
    uint32_t incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    uint32_t acc = incl - run;
    for (int w = 0; w < warp; ++w) acc += wsum[w];
    for (int c = c0; c < c1; ++c) {
        const uint32_t x = v[c];
        v[c] = acc;
        acc += x;
    }
    __syncthreads();
}

// Shared memory of the cluster build for ranges of at most `rb` blocks, in bytes: three code
// arrays, then per key the (code, rank) word and the sorted (code, key) word; the staged plane
// rows share the sorted words' space (they are dead once every key has its code and rank).
__host__ __device__ __forceinline__ size_t cluster_build_smem(int rb, int K) {
    const size_t nb = static_cast<size_t>(1) << K;
    const size_t keys = static_cast<size_t>(rb) * kKeysPerBlock;
    const size_t stage = static_cast<size_t>(rb) * K * kStageRow;
    return (3 * nb + keys + (stage > keys ? stage : keys)) * 4;
}

// One CTA per key range, a cluster of R CTAs per table (grid x = R; the cluster size is set at
// launch). Each warp runs kWordsAtOnce bit transposes at a time (each decoding
// min(4, floor(32 / K)) words) so that their shuffles and shared atomics overlap.
template <int R>
__global__ void __launch_bounds__(kClusterThreads)
    bucket_build_cluster_kernel(const uint32_t* codes, int n, int K, int L, int nblk, int cblk,
                                uint32_t* buckets) {
    namespace cg = cooperative_groups;
    constexpr int T = kClusterThreads, U = kWordsAtOnce;
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ __align__(16) uint32_t sm[];
    __shared__ uint32_t wsum[T / 32];
    const int nb = 1 << K, r = static_cast<int>(cluster.block_rank()), t = blockIdx.y,
              bh = blockIdx.z;
    const int tid = threadIdx.x;
    const int rb = (nblk + R - 1) / R;
    const int b0 = (nblk * r) / R, b1 = (nblk * (r + 1)) / R;
    const int nbk = b1 - b0, nw = nbk * kWordsPerBlock, k0 = b0 * kKeysPerBlock;
    const int m = max(0, min(n, b1 * kKeysPerBlock) - k0);        // keys of this range
    const int C = K * L, srow = K * kStageRow;
    uint32_t* hist = sm;                   // [nb] this range's count of each code
    uint32_t* total = sm + nb;             // [nb] the table's count, then its offsets
    uint32_t* delta = sm + 2 * nb;         // [nb] lower ranges' count, then output - sorted pos
    uint32_t* crank = sm + 3 * nb;         // [rb * 1024] (code << 16) | rank, by key
    uint32_t* ent = crank + static_cast<size_t>(rb) * kKeysPerBlock;   // sorted (code << 16) | key
    uint32_t* stage = ent;                 // [rb][K][kStageRow] the range's plane rows (pass 1)

    for (int c = tid; c < nb; c += T) hist[c] = 0u;
    {   // plane rows as 16-byte loads: row j = kb * K + p is staged at j * kStageRow
        const int per = K * (kWordsPerBlock / 4);
        const uint32_t* src = codes + (static_cast<size_t>(bh) * cblk + b0) * C * kWordsPerBlock +
                              static_cast<size_t>(t) * K * kWordsPerBlock;
        for (int j = tid; j < nbk * per; j += T) {
            const int kb = j / per, q = j - kb * per;        // q: plane * 8 + 16-byte chunk
            const uint4 v = __ldcs(reinterpret_cast<const uint4*>(
                src + static_cast<size_t>(kb) * C * kWordsPerBlock) + q);
            uint32_t* d = stage + (kb * K + (q >> 3)) * kStageRow + (q & 7) * 4;
            d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
        }
    }
    __syncthreads();
    // pass 1: count; the count before the key's own is its rank within (range, code). One
    // transpose decodes min(4, floor(32 / K)) words (three at K = 10).
    if (K == 0) {
        for (int i = tid; i < m; i += T) crank[i] = atomicAdd(&hist[0], 1u);
    } else if (K <= 8) {
        count_codes<U, 4, T>(stage, nw, m, K, srow, hist, crank);
    } else if (K <= 10) {
        count_codes<U, 3, T>(stage, nw, m, K, srow, hist, crank);
    } else if (K <= 16) {
        count_codes<U, 2, T>(stage, nw, m, K, srow, hist, crank);
    } else {
        count_codes<U, 1, T>(stage, nw, m, K, srow, hist, crank);
    }
    cluster.sync();                        // every range's histogram is complete
    for (int c = tid; c < nb; c += T) {
        uint32_t v[R];
#pragma unroll
        for (int q = 0; q < R; ++q) v[q] = cluster.map_shared_rank(hist, q)[c];
        uint32_t tot = 0u, pre = 0u;
#pragma unroll
        for (int q = 0; q < R; ++q) {
            pre += q < r ? v[q] : 0u;
            tot += v[q];
        }
        total[c] = tot;
        delta[c] = pre;
    }
    cluster.sync();                        // no peer reads this CTA's histogram any more
    block_exclusive_scan<T>(total, nb, wsum);                 // the table's offsets
    uint32_t* base = buckets + static_cast<size_t>(bh) * bucket_words(n, K, L);
    if (r == 0) {
        uint32_t* offsets = base + static_cast<size_t>(t) * (nb + 1);
        for (int c = tid; c < nb; c += T) offsets[c] = total[c];
        if (tid == 0) offsets[nb] = static_cast<uint32_t>(n);
    }
    for (int c = tid; c < nb; c += T) delta[c] += total[c];   // this range's base
    block_exclusive_scan<T>(hist, nb, wsum);                  // sorted start of each code
    for (int c = tid; c < nb; c += T) delta[c] -= hist[c];
    // pass 2: sort the range's keys by code in shared memory (the stage is dead)
    for (int i0 = tid; i0 < m; i0 += T * U) {         // loads first, U keys a thread at once
        uint32_t e[U], dst[U];
#pragma unroll
        for (int u = 0; u < U; ++u) e[u] = i0 + u * T < m ? crank[i0 + u * T] : 0u;
#pragma unroll
        for (int u = 0; u < U; ++u) dst[u] = hist[e[u] >> 16] + (e[u] & 0xffffu);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (i0 + u * T < m) ent[dst[u]] = (e[u] & 0xffff0000u) | static_cast<uint32_t>(i0 + u * T);
    }
    __syncthreads();
    // pass 3: sorted position p of code c goes to members[p + delta[c]]
    uint32_t* members = base + static_cast<size_t>(L) * (nb + 1) + static_cast<size_t>(t) * n;
    for (int p0 = tid; p0 < m; p0 += T * U) {
        uint32_t e[U], dl[U];
#pragma unroll
        for (int u = 0; u < U; ++u) e[u] = p0 + u * T < m ? ent[p0 + u * T] : 0u;
#pragma unroll
        for (int u = 0; u < U; ++u) dl[u] = delta[e[u] >> 16];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (p0 + u * T < m)
                members[p0 + u * T + dl[u]] = static_cast<uint32_t>(k0) + (e[u] & 0xffffu);
    }
}

// the K-bit code of table t in a row of query bits
__device__ __forceinline__ uint32_t query_code(const uint32_t* qb, int K, int t) {
    if (K == 0) return 0u;
    const int bit = t * K, w = bit >> 5, s = bit & 31;
    uint64_t v = qb[w];
    if (s + K > 32) v |= static_cast<uint64_t>(qb[w + 1]) << 32;
    return static_cast<uint32_t>((v >> s) & ((1ull << K) - 1ull));
}

// One warp per (query row, table): the query's bucket in that table, kLookupUnroll entries a lane
// loaded before their atomics are issued, so that a warp waits about three memory round trips.
__global__ void __launch_bounds__(kLookupWarps * 32)
    bucket_lookup_kernel(const uint32_t* buckets, const uint32_t* qbits, int qwords, int Hq,
                         int Hkv, int n, int K, int L, int nblk, uint32_t* ge1, uint32_t* ge2,
                         int* status) {
    allow_dependents();
    constexpr int U = kLookupUnroll;
    const int row = blockIdx.y, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kLookupWarps + (threadIdx.x >> 5);
    if (t >= L) return;
    const int G = Hq / Hkv, b = row / Hq, h = row % Hq;
    const int bh = b * Hkv + h / G;
    const int nb = 1 << K;
    const uint32_t* base = buckets + static_cast<size_t>(bh) * bucket_words(n, K, L);
    const uint32_t c = query_code(qbits + static_cast<size_t>(row) * qwords, K, t);
    const uint32_t* off = base + static_cast<size_t>(t) * (nb + 1);
    // a table built by mp_build_buckets has lo <= hi <= n and members below n; the range and
    // the members are clamped to that all the same (the buckets are the caller's memory), and
    // the MP_CHECKS build reports a table that needed it
    uint32_t lo = __ldg(off + c), hi = __ldg(off + c + 1);
    if (lane == 0) {
        mp_check(status, hi, static_cast<long long>(n) + 1, kSiteBucketRange);
        mp_check(status, lo, static_cast<long long>(hi) + 1, kSiteBucketRange);
    }
    hi = min(hi, static_cast<uint32_t>(n));
    lo = min(lo, hi);
    const uint32_t* mem = base + static_cast<size_t>(L) * (nb + 1) + static_cast<size_t>(t) * n;
    uint32_t* g1 = ge1 + static_cast<size_t>(row) * nblk * kWordsPerBlock;
    uint32_t* g2 = ge2 + static_cast<size_t>(row) * nblk * kWordsPerBlock;
    for (uint32_t i0 = lo + lane; i0 < hi; i0 += 32u * U) {
        uint32_t key[U], old[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            key[u] = i0 + 32u * u < hi ? __ldg(mem + i0 + 32u * u) : ~0u;
            if (key[u] != ~0u && !mp_check(status, key[u], n, kSiteBucketKey)) key[u] = ~0u;
            if (key[u] >= static_cast<uint32_t>(n)) key[u] = ~0u;
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            old[u] = key[u] != ~0u ? atomicOr(g1 + (key[u] >> 5), 1u << (key[u] & 31u)) : 0u;
        // saturating count: the second table to hit the key sees its first bit set
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t bit = 1u << (key[u] & 31u);
            if (key[u] != ~0u && (old[u] & bit)) atomicOr(g2 + (key[u] >> 5), bit);
        }
    }
}

}  // namespace

size_t bucket_table_bytes(int B, int Hkv, int n, int K, int L) {
    if (B < 1 || Hkv < 1 || n < 1 || K < 0 || K > kMaxBucketBits || L < 1) return 0;
    return static_cast<size_t>(B) * Hkv * bucket_words(n, K, L) * 4;
}

// Ranges per table for the cluster build: about kClusterRangeBlocks blocks each, 1 to 8.
int cluster_ranges(int nblk) {
    int R = 1;
    while (R < kMaxClusterRanges && nblk > R * kClusterRangeBlocks) R *= 2;
    return R;
}

cudaError_t launch_bucket_build(const uint32_t* codes, int B, int Hkv, int cblk, int n, int K,
                                int L, uint32_t* buckets, cudaStream_t st) {
    const int nblk = (n + kKeysPerBlock - 1) / kKeysPerBlock;
    const int R = cluster_ranges(nblk);
    const int rb = (nblk + R - 1) / R;
    const size_t csmem = cluster_build_smem(rb, K);
    if (csmem <= kClusterBuildSmem && rb * kKeysPerBlock <= 65536) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(R, L, B * Hkv);        // the ranges of one table run side by side
        cfg.blockDim = dim3(kClusterThreads);
        cfg.dynamicSmemBytes = csmem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = R;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        switch (R) {
            case 1: return cudaLaunchKernelEx(&cfg, bucket_build_cluster_kernel<1>, codes, n, K,
                                              L, nblk, cblk, buckets);
            case 2: return cudaLaunchKernelEx(&cfg, bucket_build_cluster_kernel<2>, codes, n, K,
                                              L, nblk, cblk, buckets);
            case 4: return cudaLaunchKernelEx(&cfg, bucket_build_cluster_kernel<4>, codes, n, K,
                                              L, nblk, cblk, buckets);
            default: return cudaLaunchKernelEx(&cfg, bucket_build_cluster_kernel<8>, codes, n, K,
                                               L, nblk, cblk, buckets);
        }
    }
    const dim3 ranges(kBucketRanges, L, B * Hkv);
    const size_t smem = (static_cast<size_t>(1) << K) * 4 +
                        static_cast<size_t>(kStageBlocks) * K * kStageRow * 4;
    bucket_count_kernel<<<ranges, kBuildThreads, smem, st>>>(codes, n, K, L, nblk, cblk, buckets);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bucket_scan_kernel<<<dim3(L, B * Hkv), kBuildThreads, 0, st>>>(n, K, L, buckets);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bucket_scatter_kernel<<<ranges, kBuildThreads, smem, st>>>(codes, n, K, L, nblk, cblk,
                                                               buckets);
    return cudaGetLastError();
}

cudaError_t launch_bucket_lookup(const uint32_t* buckets, const uint32_t* qbits,
                                 const DecodeShape& s, uint32_t* ge1, uint32_t* ge2,
                                 cudaStream_t st) {
    const size_t bytes = static_cast<size_t>(s.B) * s.Hq * s.nblk * kWordsPerBlock * 4;
    // one memset when the two bitmaps are neighbours (the decode workspace carves them so)
    uint32_t* lo_map = ge1 < ge2 ? ge1 : ge2;
    uint32_t* hi_map = ge1 < ge2 ? ge2 : ge1;
    const size_t gap = static_cast<size_t>(reinterpret_cast<uint8_t*>(hi_map) -
                                           reinterpret_cast<uint8_t*>(lo_map));
    cudaError_t e;
    if (gap >= bytes && gap <= bytes + 256) {
        e = cudaMemsetAsync(lo_map, 0, gap + bytes, st);
    } else {
        e = cudaMemsetAsync(ge1, 0, bytes, st);
        if (e == cudaSuccess) e = cudaMemsetAsync(ge2, 0, bytes, st);
    }
    if (e != cudaSuccess) return e;
    const dim3 grid((s.L + kLookupWarps - 1) / kLookupWarps, s.B * s.Hq);
    bucket_lookup_kernel<<<grid, kLookupWarps * 32, 0, st>>>(buckets, qbits, s.qwords, s.Hq,
                                                             s.Hkv, s.n_indexed, s.K, s.L, s.nblk,
                                                             ge1, ge2, device_status_ptr());
    return cudaGetLastError();
}

cudaError_t prepare_buckets() {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, bucket_count_kernel);
    if (e != cudaSuccess) return e;
    if ((e = cudaFuncGetAttributes(&fa, bucket_scan_kernel)) != cudaSuccess) return e;
    if ((e = cudaFuncGetAttributes(&fa, bucket_scatter_kernel)) != cudaSuccess) return e;
    for (auto fn : {bucket_build_cluster_kernel<1>, bucket_build_cluster_kernel<2>,
                    bucket_build_cluster_kernel<4>, bucket_build_cluster_kernel<8>})
        if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(kClusterBuildSmem))) != cudaSuccess)
            return e;
    return cudaFuncGetAttributes(&fa, bucket_lookup_kernel);
}

}  // namespace mp
