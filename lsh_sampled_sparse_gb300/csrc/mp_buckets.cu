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
// Build, three kernels over (table, sequence x KV head) split into kBucketRanges key ranges:
// each range counts its codes (shared-memory histogram), one CTA per table turns the counts into
// offsets and per-range write bases (an exclusive scan over codes, ranges in order within a
// code), and each range places its keys at its bases. The ranges of one table run side by side,
// so the table's members array (n words) stays in L2 while it fills. The counts and bases live
// in kBucketRanges * 2^K scratch words per table after the members.
// Lookup: one CTA per (query row, chunk of tables) reads the query's bucket in each table and
// sets the key's bit in two saturating bitmaps, ge1 (>= 1 table) and ge2 (>= 2 tables), stored in
// the selection-word layout of the dense scan ([row][block][32 words]).
#include "mp_internal.cuh"

namespace mp {
namespace {

constexpr int kBuildThreads = 256;
constexpr int kLookupThreads = 256;
constexpr int kLookupTables = 8;      // tables per lookup CTA
constexpr int kStageBlocks = 4;       // 1024-key blocks whose plane rows a build CTA stages at once
constexpr int kStageRow = kWordsPerBlock + 1;   // staged plane row stride (words): lanes reading
                                                // word w of planes 0..K-1 hit distinct banks

// words per (sequence, KV head): offsets, members, then the build's per-range counts / bases
__host__ __device__ __forceinline__ size_t bucket_words(int n, int K, int L) {
    const size_t nb = static_cast<size_t>(1) << K;
    return static_cast<size_t>(L) * ((nb + 1) + static_cast<size_t>(n) + kBucketRanges * nb);
}

// Walk the keys of key range `range` of table t: stage kStageBlocks blocks' plane rows at a
// time (row stride kStageRow); then each warp takes 32-key words: lane p < K holds plane p's word, and one 32x32 bit
// transpose leaves in lane j the K-bit code of the word's key j. f(key, code) is called by the
// lane of every key (keys past n are skipped).
template <typename F>
__device__ __forceinline__ void for_range_keys(const uint32_t* codes, int bh, int t, int range,
                                              int n, int K, int L, int nblk, uint32_t* stage,
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
                __ldcs(codes + (static_cast<size_t>(bh) * nblk + blk + kb) * C * kWordsPerBlock +
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
    bucket_count_kernel(const uint32_t* codes, int n, int K, int L, int nblk, uint32_t* buckets) {
    extern __shared__ __align__(16) uint32_t sm[];
    const int nb = 1 << K, range = blockIdx.x, t = blockIdx.y, bh = blockIdx.z;
    uint32_t* hist = sm;
    uint32_t* stage = sm + nb;
    for (int c = threadIdx.x; c < nb; c += kBuildThreads) hist[c] = 0u;
    for_range_keys(codes, bh, t, range, n, K, L, nblk, stage,
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
    bucket_scatter_kernel(const uint32_t* codes, int n, int K, int L, int nblk, uint32_t* buckets) {
    extern __shared__ __align__(16) uint32_t sm[];
    const int nb = 1 << K, range = blockIdx.x, t = blockIdx.y, bh = blockIdx.z;
    uint32_t* cursor = sm;
    uint32_t* stage = sm + nb;
    uint32_t* base = buckets + static_cast<size_t>(bh) * bucket_words(n, K, L);
    const uint32_t* scratch = base + static_cast<size_t>(L) * ((nb + 1) + static_cast<size_t>(n)) +
                              (static_cast<size_t>(t) * kBucketRanges + range) * nb;
    uint32_t* members = base + static_cast<size_t>(L) * (nb + 1) + static_cast<size_t>(t) * n;
    for (int c = threadIdx.x; c < nb; c += kBuildThreads) cursor[c] = scratch[c];
    for_range_keys(codes, bh, t, range, n, K, L, nblk, stage, [&](int key, uint32_t c) {
        members[atomicAdd(&cursor[c], 1u)] = static_cast<uint32_t>(key);
    });
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
    return static_cast<size_t>(B) * Hkv * bucket_words(n, K, L) * 4;
}

cudaError_t launch_bucket_build(const uint32_t* codes, int B, int Hkv, int n, int K, int L,
                                uint32_t* buckets, cudaStream_t st) {
    const int nblk = (n + kKeysPerBlock - 1) / kKeysPerBlock;
    const size_t smem = (static_cast<size_t>(1) << K) * 4 +
                        static_cast<size_t>(kStageBlocks) * K * kStageRow * 4;
    const dim3 ranges(kBucketRanges, L, B * Hkv);   // the ranges of one table run side by side
    bucket_count_kernel<<<ranges, kBuildThreads, smem, st>>>(codes, n, K, L, nblk, buckets);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bucket_scan_kernel<<<dim3(L, B * Hkv), kBuildThreads, 0, st>>>(n, K, L, buckets);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bucket_scatter_kernel<<<ranges, kBuildThreads, smem, st>>>(codes, n, K, L, nblk, buckets);
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
    cudaError_t e = cudaFuncGetAttributes(&fa, bucket_count_kernel);
    if (e != cudaSuccess) return e;
    if ((e = cudaFuncGetAttributes(&fa, bucket_scan_kernel)) != cudaSuccess) return e;
    if ((e = cudaFuncGetAttributes(&fa, bucket_scatter_kernel)) != cudaSuccess) return e;
    return cudaFuncGetAttributes(&fa, bucket_lookup_kernel);
}

}  // namespace mp
