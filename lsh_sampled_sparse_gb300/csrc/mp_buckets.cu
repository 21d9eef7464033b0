// Bucketed hash tables in HBM: the retrieval structure of "MagicPIG: LSH Sampling for Efficient
// LLM Generation" (system co-design item 3: the query's codes are looked up in L prebuilt hash
// tables) and of "MagicPIG: don't pick the tallest" (section 6: every table stores a pointer to
// every key; a query scans about L n / 2^K entries).
//
// Layout per (sequence, KV head), in 32-bit words: offsets [L][2^K + 1], then members [L][n];
// members[t][offsets[t][c] .. offsets[t][c + 1]) are the keys whose table-t code is c. The order
// of keys inside a bucket is not fixed (buckets are sets); everything that reads them only counts.
//
// Build: one CTA per (table, sequence x KV head) reads that table's K plane rows of every
// 1024-key block twice: the first pass counts codes in a shared-memory histogram, an exclusive
// scan turns the counts into offsets, the second pass places each key at its bucket's cursor.
// Lookup: one CTA per (query row, chunk of tables) reads the query's bucket in each table and
// sets the key's bit in two saturating bitmaps, ge1 (>= 1 table) and ge2 (>= 2 tables), stored in
// the selection-word layout of the dense scan ([row][block][32 words]).
#include "mp_internal.cuh"

namespace mp {
namespace {

constexpr int kBuildThreads = 256;
constexpr int kLookupThreads = 256;
constexpr int kLookupTables = 8;      // tables per lookup CTA

__device__ __forceinline__ size_t bucket_words(int n, int K, int L) {
    return static_cast<size_t>(L) * ((1u << K) + 1 + static_cast<size_t>(n));
}

// code of key `i` of the staged block (plane p of the table is the 32-word row planes[p])
__device__ __forceinline__ uint32_t key_code(const uint32_t* planes, int K, int i) {
    const int w = i >> 5, b = i & 31;
    uint32_t c = 0u;
    for (int p = 0; p < K; ++p) c |= ((planes[p * kWordsPerBlock + w] >> b) & 1u) << p;
    return c;
}

__global__ void __launch_bounds__(kBuildThreads)
    bucket_build_kernel(const uint32_t* codes, int n, int K, int L, int nblk, uint32_t* buckets) {
    extern __shared__ __align__(16) uint32_t sm[];
    const int nb = 1 << K;
    uint32_t* hist = sm;                          // [2^K] counts, then cursors
    uint32_t* planes = sm + nb;                   // [K][32] one block's plane rows of this table
    __shared__ uint32_t wsum[kBuildThreads / 32];
    const int t = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x, lane = tid & 31,
              warp = tid >> 5;
    const int C = K * L;
    uint32_t* base = buckets + static_cast<size_t>(bh) * bucket_words(n, K, L);
    uint32_t* offsets = base + static_cast<size_t>(t) * (nb + 1);
    uint32_t* members = base + static_cast<size_t>(L) * (nb + 1) + static_cast<size_t>(t) * n;
    for (int c = tid; c < nb; c += kBuildThreads) hist[c] = 0u;

    for (int pass = 0; pass < 2; ++pass) {
        for (int blk = 0; blk < nblk; ++blk) {
            __syncthreads();                      // previous block's planes fully consumed
            const uint32_t* rows = codes + (static_cast<size_t>(bh) * nblk + blk) * C * kWordsPerBlock +
                                   static_cast<size_t>(t) * K * kWordsPerBlock;
            for (int i = tid; i < K * kWordsPerBlock; i += kBuildThreads) planes[i] = __ldcs(rows + i);
            __syncthreads();
            for (int i = tid; i < kKeysPerBlock; i += kBuildThreads) {
                const int key = blk * kKeysPerBlock + i;
                if (key >= n) break;
                const uint32_t c = key_code(planes, K, i);
                if (pass == 0) {
                    atomicAdd(&hist[c], 1u);
                } else {
                    const uint32_t pos = atomicAdd(&hist[c], 1u);
                    members[pos] = static_cast<uint32_t>(key);
                }
            }
        }
        if (pass == 1) break;
        // exclusive scan of the counts: thread tid owns a contiguous run of buckets
        __syncthreads();
        const int per = (nb + kBuildThreads - 1) / kBuildThreads;
        const int c0 = min(nb, tid * per), c1 = min(nb, c0 + per);
        uint32_t run = 0u;
        for (int c = c0; c < c1; ++c) run += hist[c];
        uint32_t incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        uint32_t before = 0u;
        for (int w = 0; w < warp; ++w) before += wsum[w];
        uint32_t acc = before + incl - run;
        for (int c = c0; c < c1; ++c) {
            const uint32_t cnt = hist[c];
            offsets[c] = acc;
            hist[c] = acc;                        // cursor for the second pass
            acc += cnt;
        }
        if (tid == kBuildThreads - 1) offsets[nb] = acc;
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

__global__ void __launch_bounds__(kLookupThreads)
    bucket_lookup_kernel(const uint32_t* buckets, const uint32_t* qbits, int qwords, int Hq,
                         int Hkv, int n, int K, int L, int nblk, uint32_t* ge1, uint32_t* ge2) {
    const int row = blockIdx.y, tid = threadIdx.x;
    const int G = Hq / Hkv, b = row / Hq, h = row % Hq;
    const int bh = b * Hkv + h / G;
    const int nb = 1 << K;
    const uint32_t* base = buckets + static_cast<size_t>(bh) * bucket_words(n, K, L);
    const uint32_t* qb = qbits + static_cast<size_t>(row) * qwords;
    uint32_t* g1 = ge1 + static_cast<size_t>(row) * nblk * kWordsPerBlock;
    uint32_t* g2 = ge2 + static_cast<size_t>(row) * nblk * kWordsPerBlock;
    const int t0 = blockIdx.x * kLookupTables, t1 = min(L, t0 + kLookupTables);
    for (int t = t0; t < t1; ++t) {
        const uint32_t c = query_code(qb, K, t);
        const uint32_t* off = base + static_cast<size_t>(t) * (nb + 1);
        const uint32_t lo = __ldg(off + c), hi = __ldg(off + c + 1);
        const uint32_t* mem = base + static_cast<size_t>(L) * (nb + 1) + static_cast<size_t>(t) * n;
        for (uint32_t i = lo + tid; i < hi; i += kLookupThreads) {
            const uint32_t key = __ldg(mem + i);
            const uint32_t bit = 1u << (key & 31u);
            // saturating count: the second table to hit the key sees its first bit set
            if (atomicOr(g1 + (key >> 5), bit) & bit) atomicOr(g2 + (key >> 5), bit);
        }
    }
}

}  // namespace

size_t bucket_table_bytes(int B, int Hkv, int n, int K, int L) {
    if (B < 1 || Hkv < 1 || n < 1 || K < 0 || K > kMaxBucketBits || L < 1) return 0;
    return static_cast<size_t>(B) * Hkv * static_cast<size_t>(L) *
           ((static_cast<size_t>(1) << K) + 1 + static_cast<size_t>(n)) * 4;
}

cudaError_t launch_bucket_build(const uint32_t* codes, int B, int Hkv, int n, int K, int L,
                                uint32_t* buckets, cudaStream_t st) {
    const int nblk = (n + kKeysPerBlock - 1) / kKeysPerBlock;
    const size_t smem = (static_cast<size_t>(1) << K) * 4 + static_cast<size_t>(K) * kWordsPerBlock * 4;
    bucket_build_kernel<<<dim3(L, B * Hkv), kBuildThreads, smem, st>>>(codes, n, K, L, nblk,
                                                                       buckets);
    return cudaGetLastError();
}

cudaError_t launch_bucket_lookup(const uint32_t* buckets, const uint32_t* qbits,
                                 const DecodeShape& s, uint32_t* ge1, uint32_t* ge2,
                                 cudaStream_t st) {
    const size_t words = static_cast<size_t>(s.B) * s.Hq * s.nblk * kWordsPerBlock;
    cudaError_t e = cudaMemsetAsync(ge1, 0, words * 4, st);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(ge2, 0, words * 4, st);
    if (e != cudaSuccess) return e;
    const dim3 grid((s.L + kLookupTables - 1) / kLookupTables, s.B * s.Hq);
    bucket_lookup_kernel<<<grid, kLookupThreads, 0, st>>>(buckets, qbits, s.qwords, s.Hq, s.Hkv,
                                                          s.n, s.K, s.L, s.nblk, ge1, ge2);
    return cudaGetLastError();
}

cudaError_t prepare_buckets() {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, bucket_build_kernel);
    if (e != cudaSuccess) return e;
    return cudaFuncGetAttributes(&fa, bucket_lookup_kernel);
}

}  // namespace mp
