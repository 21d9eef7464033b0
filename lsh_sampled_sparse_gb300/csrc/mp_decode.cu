// Decode step: query encoding; a scan kernel that streams the packed codes of a block of 1024
// keys and selects the keys colliding with the query in >= 2 tables; an attend kernel that
// gathers only those K/V rows and folds them with importance weights into partial softmaxes,
// the last CTA of each query row merging the partials by log-sum-exp.
//
// The method is Algorithm 1 of "MagicPIG: LSH Sampling for Efficient LLM Generation" (method
// details, algorithm execution), with the inclusion probability of the hash-function-choice
// section and the exact sink/local set ("static cache") of the system co-design section, whose
// "recursive attention" merge of partial outputs is the log-sum-exp merge done here.
#include <algorithm>
#include <type_traits>

#include "mp_internal.cuh"

namespace mp {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCombinePitch = 132;                  // floats per (warp, head) partial: o, m, l
constexpr int kAttendBlocks = kAttendBlockGroup;
constexpr int kAWarps = 4;                          // attend CTA: 4 warps, 8 half-warps on rows
static_assert(kAttendBlocks <= kAWarps, "one warp lists each block of an attend CTA");
constexpr int kAThreads = 32 * kAWarps;
constexpr int kMergeRegs = 8;                       // partials a merging warp holds in registers
static_assert(kAThreads == kD && 4 * 32 == kD,
              "the attend merge: a thread per output dim; a merging lane holds 4 dims");
constexpr int kRingDepth = 5;                       // tables in flight per warp in the async scan
constexpr int kRingMinK = 8, kRingMaxK = 11;        // K range the async scan handles
constexpr int kLuIntervals = kLogUTableIntervals;   // log u tables: cosine grid intervals

// ------------------------------------------------------------------------------------------------
// Query encoding: qbit_j = [w_j . q > 0] (the query is not centred), |q| and q.mu for the cosine.
// One warp per query row, one lane per hyperplane of a 32-plane word. Besides the packed bits it
// writes the per-plane XOR masks the scan uses (0 where the query bit is 1, ~0 where it is 0),
// laid out [sequence x KV head][plane][head of the group] so a scan CTA copies its group's masks
// in one contiguous piece.
// ------------------------------------------------------------------------------------------------
constexpr int kQRows = 8;       // query rows per CTA (one per warp)

struct QArgs {
    const void* q;
    const void* W;
    const float* centre;
    uint32_t* qbits;
    uint32_t* qmask;
    float4* qstat;
    unsigned* counters;
    float* logu_tab;                             // filled by the extra row of CTAs
    int* status;                                 // index checks of the MP_CHECKS build
    int q_bf16, w_bf16, BHq, Hq, G, C, cpad, qwords, n_counters, K, L, qrow_ctas;
};

__global__ void __launch_bounds__(kThreads) qencode_kernel(const QArgs a) {
    __shared__ float Qs[kQRows][kD];
    __shared__ float Ws[kD][32];                 // this word's 32 hyperplane columns
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    allow_dependents();                          // the scan may start streaming codes meanwhile
    if (blockIdx.y == a.qrow_ctas) {
        // the extra row of CTAs: the attend kernel's table of log u over the cosine
        for (int seg = blockIdx.x; seg < kLogUSegments; seg += gridDim.x)
            log_inclusion_segment(seg, a.K, a.L, &Ws[0][0], a.logu_tab);
        return;
    }
    const int wd = blockIdx.x, r0 = blockIdx.y * kQRows;
    const int nq = min(kQRows, a.BHq - r0);
    const int row = r0 + warp;
    const int Hkv = a.Hq / a.G;
    // the CTAs of word 0 also compute |q| and q.mu: the centre is loaded with the other inputs
    float mu4[kD / 32] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (blockIdx.x == 0 && warp < nq) {
        const int b = row / a.Hq, g = (row % a.Hq) / a.G;
        const float* mu = a.centre + (static_cast<size_t>(b) * Hkv + g) * kD;
#pragma unroll
        for (int k = 0; k < kD / 32; ++k) mu4[k] = mu[lane + 32 * k];
    }
    {
        // all loads first, then the stores: the loop bodies must not wait for each other
        constexpr int kQPer = kQRows * kD / kThreads, kWPer = kD * 32 / kThreads;
        float qv[kQPer], wv[kWPer];
#pragma unroll
        for (int k = 0; k < kQPer; ++k) {
            const int idx = tid + k * kThreads;
            qv[k] = idx < nq * kD ? load_elem(a.q, a.q_bf16, static_cast<size_t>(r0) * kD + idx)
                                  : 0.0f;
        }
#pragma unroll
        for (int k = 0; k < kWPer; ++k) {
            const int idx = tid + k * kThreads, e = idx >> 5, j = wd * 32 + (idx & 31);
            wv[k] = j < a.C ? load_elem(a.W, a.w_bf16, static_cast<size_t>(e) * a.C + j) : 0.0f;
        }
#pragma unroll
        for (int k = 0; k < kQPer; ++k) {
            const int idx = tid + k * kThreads;
            Qs[idx / kD][idx % kD] = qv[k];
        }
#pragma unroll
        for (int k = 0; k < kWPer; ++k) {
            const int idx = tid + k * kThreads;
            Ws[idx >> 5][idx & 31] = wv[k];
        }
    }
    __syncthreads();
    if (warp < nq && a.C > 0) {
        const int j = wd * 32 + lane;
        // four interleaved partial sums over the 128 dimensions (a short dependency chain)
        float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 8
        for (int e = 0; e < kD; e += 4) {
#pragma unroll
            for (int i = 0; i < 4; ++i) s4[i] = fmaf(Ws[e + i][lane], Qs[warp][e + i], s4[i]);
        }
        const float s = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        const bool bit = j < a.C && s > 0.0f;
        const uint32_t word = __ballot_sync(0xffffffffu, bit);
        const long long qbi = static_cast<long long>(row) * a.qwords + wd;
        if (lane == 0 && mp_check(a.status, qbi, static_cast<long long>(a.BHq) * a.qwords,
                                  kSiteQencodeStore))
            a.qbits[qbi] = word;
        const int b = row / a.Hq, h = row % a.Hq;
        const size_t bg = static_cast<size_t>(b) * Hkv + h / a.G;
        const long long qmi = (static_cast<long long>(bg) * a.cpad + j) * a.G + (h % a.G);
        if (j < a.cpad &&
            mp_check(a.status, qmi, static_cast<long long>(a.BHq) * a.cpad, kSiteQencodeStore))
            a.qmask[qmi] = bit ? 0u : 0xffffffffu;
    }
    if (blockIdx.x == 0) {
        if (warp < nq) {
            float nn = 0.0f, qm = 0.0f;
#pragma unroll
            for (int k = 0; k < kD / 32; ++k) {
                const float x = Qs[warp][lane + 32 * k];
                nn = fmaf(x, x, nn);
                qm = fmaf(x, mu4[k], qm);
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                nn += __shfl_xor_sync(0xffffffffu, nn, o);
                qm += __shfl_xor_sync(0xffffffffu, qm, o);
            }
            if (lane == 0 && mp_check(a.status, row, a.BHq, kSiteQencodeStore))
                a.qstat[row] = make_float4(sqrtf(nn), qm, 0.0f, 0.0f);
        }
        if (blockIdx.y == 0)
            for (int i = tid; i < a.n_counters; i += kThreads) a.counters[i] = 0u;
    }
}

// ------------------------------------------------------------------------------------------------
// Collide -> select, one CTA per (1024-key block, sequence x KV head); the gather + attend +
// merge kernel follows as a programmatic dependent
// ------------------------------------------------------------------------------------------------
struct CArgs {
    const uint32_t* codes;
    const uint32_t* qmask;
    uint32_t* selmask;
    int n, nblk, Hq, Hkv, K, L, C, cpad, n_sink, n_local;
    int cblk;                                    // code blocks per head in memory
    int blk0;                                    // first block scanned (grid x + blk0)
    int* status;                                 // index checks of the MP_CHECKS build
};

// Attend CTA shared memory: [work][selection words][prefix counts][row keys][cbuf][misc]. The
// work region holds kAttendRows row slots of staged K/V rows; cbuf joins the warps' partials.
constexpr int kAttendRows = 64;                      // row slots in an attend CTA's stage
constexpr int kRowKeys = 256;                        // selected keys listed once per attend CTA
struct AttendSmem {
    size_t work, total;
};
inline AttendSmem attend_smem(int nsp, size_t kv_elem) {
    (void)nsp;
    AttendSmem m;
    m.work = static_cast<size_t>(kAttendRows) * 2 * kD * kv_elem;
    m.total = m.work + static_cast<size_t>(kAThreads) * 4 + (kAThreads + 4) * 4 +
              static_cast<size_t>(kRowKeys) * 4 + static_cast<size_t>(kAWarps) * kCombinePitch * 4 +
              32;
    return m;
}

template <int G>
size_t collide_smem_bytes(int cpad, int K) {
    // with the ring, each warp's counters go into its own ring once it has drained
    static_assert(kRingDepth * kRingMinK >= 2 * 8, "a drained ring holds its warp's counters");
    const size_t area = (K >= kRingMinK && K <= kRingMaxK)
                            ? static_cast<size_t>(kWarps) * kRingDepth * K * kWordsPerBlock * 4
                            : static_cast<size_t>(kWarps) * 2 * G * 32 * 4;
    return static_cast<size_t>(cpad) * G * 4 + area;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
// The same copy with an L2 eviction-priority policy (from l2_evict_first) for data read once
__device__ __forceinline__ void cp_async16_hint(void* dst, const void* src, uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src), "l"(policy)
                 : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    return policy;
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
}

template <int G>
__device__ __forceinline__ void load_qneg(const uint32_t* p, uint32_t (&v)[G]) {
    if constexpr (G % 4 == 0) {
#pragma unroll
        for (int h = 0; h < G; h += 4) {
            const uint4 t = *reinterpret_cast<const uint4*>(p + h);
            v[h] = t.x;
            v[h + 1] = t.y;
            v[h + 2] = t.z;
            v[h + 3] = t.w;
        }
    } else if constexpr (G == 2) {
        const uint2 t = *reinterpret_cast<const uint2*>(p);
        v[0] = t.x;
        v[1] = t.y;
    } else {
#pragma unroll
        for (int h = 0; h < G; ++h) v[h] = p[h];
    }
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_pending() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Phase 1 for a compile-time K with the plane rows streamed through a per-warp shared-memory
// ring: table t + kRingDepth - 1 is copied (cp.async, 16 B per lane) while table t is reduced,
// so each warp keeps kRingDepth tables (kRingDepth * K * 128 bytes) in flight without holding
// them in registers. cb points at the block's first plane row (no lane offset). The codes are
// read once per decode step: their copies carry the L2 evict-first policy.
template <int K>
__device__ __forceinline__ void ring_issue(const uint32_t* cb, uint32_t* ring, int t, int slot,
                                           int lane, uint64_t policy) {
    constexpr int kSlot = K * kWordsPerBlock;      // words per table
    constexpr int kPieces = K * 8;                 // 16-byte pieces per table
    const uint32_t* src = cb + static_cast<size_t>(t) * kSlot;
    uint32_t* dst = ring + slot * kSlot;
#pragma unroll
    for (int pc = lane; pc < kPieces; pc += 32) cp_async16_hint(dst + 4 * pc, src + 4 * pc, policy);
}
// The ring's first kRingDepth - 1 tables, one commit group each. The codes are an input of the
// call, not something the query encoding writes, so the scan issues these before it waits.
template <int K>
__device__ __forceinline__ void ring_fill(const uint32_t* cb, uint32_t* ring, int t0, int t1,
                                          int lane) {
    const uint64_t policy = l2_evict_first();
#pragma unroll
    for (int d = 0; d < kRingDepth - 1; ++d) {
        if (t0 + d < t1) ring_issue<K>(cb, ring, t0 + d, d, lane, policy);
        cp_async_commit();
    }
}
// The ring after ring_fill (its groups may have been followed by other, completed ones).
template <int G, int K>
__device__ __forceinline__ void scan_tables_async(const uint32_t* cb, uint32_t* ring,
                                                  const uint32_t* qneg, int t0, int t1, int lane,
                                                  uint32_t (&ge1)[G], uint32_t (&ge2)[G]) {
    constexpr int kSlot = K * kWordsPerBlock;
    const uint64_t policy = l2_evict_first();
    int slot = 0;
    for (int t = t0; t < t1; ++t) {
        const int nt = t + kRingDepth - 1;
        if (nt < t1) ring_issue<K>(cb, ring, nt, (slot + kRingDepth - 1) % kRingDepth, lane, policy);
        cp_async_commit();
        cp_async_wait_pending<kRingDepth - 1>();   // this lane's pieces of table t have landed
        __syncwarp();                              // ... and every other lane's
        const uint32_t* planes = ring + slot * kSlot + lane;
        uint32_t acc[G];
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h] = 0xffffffffu;
#pragma unroll
        for (int b = 0; b < K; ++b) {
            const uint32_t x = planes[b * kWordsPerBlock];
            uint32_t qn[G];
            load_qneg<G>(qneg + (t * K + b) * G, qn);
#pragma unroll
            for (int h = 0; h < G; ++h) acc[h] &= x ^ qn[h];
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            ge2[h] |= ge1[h] & acc[h];
            ge1[h] |= acc[h];
        }
        __syncwarp();                              // the slot is refilled next iteration
        slot = (slot + 1) % kRingDepth;
    }
    cp_async_wait_pending<0>();
}

// Phase 1 for any K: the planes of [t0, t1) as one stream, 16 loads in flight.
template <int G>
__device__ __forceinline__ void scan_tables_any(const uint32_t* cb, const uint32_t* qneg, int K,
                                                int t0, int t1, uint32_t (&ge1)[G],
                                                uint32_t (&ge2)[G]) {
    uint32_t acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = 0xffffffffu;
    const int jend = t1 * K;
    int bb = 0;
    for (int j = t0 * K; j < jend; j += 16) {
        uint32_t x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            x[i] = (j + i < jend) ? __ldcs(cb + static_cast<size_t>(j + i) * kWordsPerBlock) : 0u;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (j + i < jend) {
                uint32_t qn[G];
                load_qneg<G>(qneg + (j + i) * G, qn);
#pragma unroll
                for (int h = 0; h < G; ++h) acc[h] &= x[i] ^ qn[h];
                if (++bb == K) {
                    bb = 0;
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        ge2[h] |= ge1[h] & acc[h];
                        ge1[h] |= acc[h];
                        acc[h] = 0xffffffffu;
                    }
                }
            }
        }
    }
}

struct AArgs {
    const uint32_t* selmask;
    const float4* qstat;
    const void* q;
    const float* centre;
    const void* keys;
    const void* values;
    float* pm;
    float* pl;
    float* po;
    unsigned* counters;
    float* out;
    const float* logu_tab;                       // log u over the cosine (SimHash: per call)
    int table_only;                              // cross-polytope: the table at every cosine
    int q_bf16, n, nblk, nsb, Hq, Hkv, G, K, L, n_sink, n_local;
    int ncap;                                    // K/V rows per head in memory
    int* status;                                 // index checks of the MP_CHECKS build
    const float* radius;                         // MIPS variant: longest centred key per head
    float scale;
    int work_bytes;                              // bytes of the row stage region
};

// The scan of one (1024-key block, sequence x KV head) for its GQA group of G query heads,
// run by all kThreads threads of a CTA: before the query masks exist, start this warp's first
// tables of codes (an input of the call) into the ring for the ring's K, else into L2; wait for
// the query encoding, then let the next kernel be scheduled; copy the group's query masks into
// shared memory; per 32-key word (lane) and table, match = AND_b (plane ^ qmask), kept as
// bit-sliced saturating counters ge1 = (>= 1 match), ge2 = (>= 2 matches); the warps split the L
// tables and their counters combine in a fixed order. Threads tid < G * 32 return the selection
// word w = tid % 32 of head tid / 32, S = ge2 & valid & not T, in *sel and the block's T word in
// *tmask. Shared memory: qneg [cpad][G], then per warp either its ring [kRingDepth][K][32]
// (K in the ring's range; the warp's counters [2][G][32] go into its own ring once drained) or
// its counters alone; warp w's counters start at gebuf + w * gstride. The CTA is past a barrier
// on return.
template <int G>
__device__ __forceinline__ void scan_block(const CArgs& a, int blk, int bg, uint32_t* qneg,
                                           uint32_t* gebuf, int gstride, uint32_t* ring,
                                           uint32_t* sel,
                                           uint32_t* tmask) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    allow_dependents();
    const int t0 = (a.L * warp) / kWarps, t1 = (a.L * (warp + 1)) / kWarps;
    const uint32_t* cb0 =
        a.codes + (static_cast<size_t>(bg) * a.cblk + blk) * a.C * kWordsPerBlock;
    switch (a.K) {
        case 8: ring_fill<8>(cb0, ring, t0, t1, lane); break;
        case 9: ring_fill<9>(cb0, ring, t0, t1, lane); break;
        case 10: ring_fill<10>(cb0, ring, t0, t1, lane); break;
        case 11: ring_fill<11>(cb0, ring, t0, t1, lane); break;
        default: {
            const uint32_t* first = cb0 + static_cast<size_t>(t0) * a.K * kWordsPerBlock;
            const int rows = min(kRingDepth * a.K, (t1 - t0) * a.K);
            for (int r = lane; r < rows; r += 32)
                asm volatile("prefetch.global.L2 [%0];"
                             ::"l"(first + static_cast<size_t>(r) * kWordsPerBlock));
        }
    }
    wait_for_predecessor();

    // ---- the group's query masks (one contiguous piece)
    {
        const uint4* src = reinterpret_cast<const uint4*>(a.qmask +
                                                          static_cast<size_t>(bg) * a.cpad * G);
        const int n16 = a.cpad * G / 4;
        for (int i = tid; i < n16; i += kThreads) cp_async16(qneg + 4 * i, src + i);
    }
    cp_async_wait_all();
    __syncthreads();

    uint32_t ge1[G], ge2[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        ge1[h] = 0u;
        ge2[h] = 0u;
    }
    switch (a.K) {
        case 0:
#pragma unroll
            for (int h = 0; h < G; ++h) {
                ge1[h] = (t1 - t0 >= 1) ? 0xffffffffu : 0u;
                ge2[h] = (t1 - t0 >= 2) ? 0xffffffffu : 0u;
            }
            break;
        case 8: scan_tables_async<G, 8>(cb0, ring, qneg, t0, t1, lane, ge1, ge2); break;
        case 9: scan_tables_async<G, 9>(cb0, ring, qneg, t0, t1, lane, ge1, ge2); break;
        case 10: scan_tables_async<G, 10>(cb0, ring, qneg, t0, t1, lane, ge1, ge2); break;
        case 11: scan_tables_async<G, 11>(cb0, ring, qneg, t0, t1, lane, ge1, ge2); break;
        default: scan_tables_any<G>(cb0 + lane, qneg, a.K, t0, t1, ge1, ge2); break;
    }
    uint32_t* mine = gebuf + warp * gstride;     // this warp's ring, drained (or its own slot)
#pragma unroll
    for (int h = 0; h < G; ++h) {
        mine[(0 * G + h) * 32 + lane] = ge1[h];
        mine[(1 * G + h) * 32 + lane] = ge2[h];
    }
    __syncthreads();
    if (tid < G * 32) {
        const int h = tid >> 5, w = lane;
        uint32_t g1 = 0u, g2 = 0u;
#pragma unroll
        for (int ww = 0; ww < kWarps; ++ww) {
            const uint32_t a1 = gebuf[ww * gstride + (0 * G + h) * 32 + w];
            const uint32_t a2 = gebuf[ww * gstride + (1 * G + h) * 32 + w];
            g2 |= a2 | (g1 & a1);
            g1 |= a1;
        }
        const int key0 = blk * kKeysPerBlock + w * 32;
        const uint32_t valid = bits_below(a.n - key0);
        const uint32_t tm =
            (bits_below(a.n_sink - key0) | ~bits_below(a.n - a.n_local - key0)) & valid;
        *sel = g2 & valid & ~tm;
        *tmask = tm;
    }
}

// Collide + select: per (1024-key block, sequence x KV head) the selection words
// S_h = [>= 2 of L tables match] & valid & not T, for every query head h of the group.
template <int G>
__global__ void __launch_bounds__(kThreads, 3) collide_kernel(const CArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int blk = blockIdx.x + a.blk0, bg = blockIdx.y;
    if (!mp_check(a.status, static_cast<long long>(bg) * a.cblk + blk,
                  static_cast<long long>(gridDim.y) * a.cblk, kSiteScanCodes) ||
        !mp_check(a.status, blk, a.nblk, kSiteScanCodes))
        return;                                  // the whole CTA: the condition is uniform
    const int b = bg / a.Hkv, g = bg % a.Hkv;
    const int row0 = b * a.Hq + g * G;          // first query row of this KV head's group
    uint32_t* qneg = reinterpret_cast<uint32_t*>(smem);                    // [cpad][G]
    uint32_t* area = qneg + static_cast<size_t>(a.cpad) * G;
    const bool ringed = a.K >= kRingMinK && a.K <= kRingMaxK;
    const int rstride = kRingDepth * a.K * kWordsPerBlock;                 // ring words per warp
    uint32_t* ring = area + static_cast<size_t>(warp) * rstride;          // [8][depth][K][32]
    uint32_t s = 0u, tm = 0u;
    scan_block<G>(a, blk, bg, qneg, area, ringed ? rstride : 2 * G * 32, ring, &s, &tm);
    if (threadIdx.x < G * 32) {
        const int h = threadIdx.x >> 5, w = threadIdx.x & 31;
        const long long si = (static_cast<long long>(row0 + h) * a.nblk + blk) * 32 + w;
        if (mp_check(a.status, si, static_cast<long long>(gridDim.y) * G * a.nblk * 32,
                     kSiteScanSelect))
            a.selmask[si] = s;
    }
}

// The 8 consecutive elements [8 hl, 8 hl + 8) of a staged K or V row as floats.
__device__ __forceinline__ void load8(const uint8_t* p, const __nv_bfloat16*, float (&f)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}
__device__ __forceinline__ void load8(const uint8_t* p, const float*, float (&f)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 16);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__device__ __forceinline__ unsigned atomic_add_acq_rel_gpu(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(v)
                 : "memory");
    return old;
}

// Gather + weight + attend for one query head. CTA sb < nsb takes the sampled keys S_h of
// kAttendBlocks consecutive 1024-key blocks (ascending, from the selection words); CTA nsb takes
// the exact set T = [0, n_sink) u [n - n_local, n) with log u = 0, so that the 68 sink/local rows
// do not pile onto the CTA of the last blocks. Each CTA folds its rows into one partial softmax;
// the last CTA of each query row merges the row's nsb + 1 partials by log-sum-exp.
// Each warp copies and folds its own rows (row e goes to half-warp e mod 8) in a pipeline of
// groups of four rows per half-warp through two sets of row slots in shared memory: the group
// after next is copied (cp.async) into a group's slots as soon as that group is folded.
template <typename KV>
__global__ void __launch_bounds__(kAThreads, 6) attend_kernel(const AArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sb = blockIdx.x, row = blockIdx.y;
    const int b = row / a.Hq, h = row % a.Hq;
    const int bg = b * a.Hkv + h / a.G;
    const bool exact = sb == a.nsb;              // this CTA takes T
    const int nsp = a.nsb + 1;                   // partials per query row

    constexpr int kRowBytes = 2 * kD * static_cast<int>(sizeof(KV));     // K then V
    constexpr int kPieces = kRowBytes / 16;
    constexpr int kWords = kAttendBlocks * 32;                            // selection words
    static_assert(kWords == kAThreads, "one selection word per thread");
    uint8_t* stage = smem;                                    // [kAttendRows] K/V row slots
    uint32_t* wsel = reinterpret_cast<uint32_t*>(smem + a.work_bytes);      // [kWords]
    int* wpre = reinterpret_cast<int*>(wsel + kWords);                      // [kWords + 4]
    int* rowkey = wpre + kWords + 4;                                        // [kRowKeys]
    float* cbuf = reinterpret_cast<float*>(rowkey + kRowKeys);              // [4][kCombinePitch]
    int* misc = reinterpret_cast<int*>(cbuf + kAWarps * kCombinePitch);     // [8]

    const int half = lane >> 4, hl = lane & 15;
    const unsigned hmask = 0xffffu << (lane & 16);
    float q8[8], mu8[8];                         // inputs of the call: readable right away
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        q8[i] = load_elem(a.q, a.q_bf16, static_cast<size_t>(row) * kD + 8 * hl + i);
        mu8[i] = a.centre[static_cast<size_t>(bg) * kD + 8 * hl + i];
    }
    wait_for_predecessor();                      // selection words, query norms
    const float4 st = a.qstat[row];
    const float qn = st.x, qmu = st.y;
    const float rad = a.radius ? a.radius[bg] : 0.0f;   // MIPS: cos = q.(k - mu) / (|q| r)

    // ---- the rows of this CTA: T by arithmetic, or the selected keys of its blocks, found
    //      through the selection words and their prefix counts (no list is materialised)
    const int t_a = min(a.n_sink, a.n), t_b = max(a.n - a.n_local, t_a);
    const int blk0 = sb * kAttendBlocks;
    int nsel;
    if (exact) {
        nsel = t_a + (a.n - t_b);
    } else {
        const int nb = min(kAttendBlocks, a.nblk - blk0);
        uint32_t U = 0u;
        if (warp < nb) {
            // the scan already masked its words; selection words from elsewhere (the bucketed
            // lookup's >= 2 bitmap) need valid & not T here
            const int blk = blk0 + warp;
            const int key0 = blk * kKeysPerBlock + lane * 32;
            const uint32_t valid = bits_below(a.n - key0);
            const uint32_t tmask =
                (bits_below(a.n_sink - key0) | ~bits_below(a.n - a.n_local - key0)) & valid;
            const long long wi = (static_cast<long long>(row) * a.nblk + blk) * 32 + lane;
            if (mp_check(a.status, wi, static_cast<long long>(gridDim.y) * a.nblk * 32,
                         kSiteAttendSelect))
                U = a.selmask[wi] & valid & ~tmask;
        }
        wsel[tid] = U;
        const int c = __popc(U);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) misc[warp] = incl;
        __syncthreads();
        int before = 0;
        for (int w = 0; w < warp; ++w) before += misc[w];
        wpre[tid] = before + incl - c;
        if (tid == kAThreads - 1) wpre[kWords] = before + incl;
        __syncthreads();
        nsel = wpre[kWords];
    }
    // key of entry i: T by arithmetic; else the word holding it (the last with wpre <= i) and its
    // (i - wpre)-th set bit
    auto key_of = [&](int i) -> int {
        if (exact) return i < t_a ? i : t_b + (i - t_a);
        int lo = 0, hi = kWords - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (wpre[mid] <= i) lo = mid;
            else hi = mid - 1;
        }
        const int bit = static_cast<int>(__fns(wsel[lo], 0, i - wpre[lo] + 1));
        return (blk0 + (lo >> 5)) * kKeysPerBlock + (lo & 31) * 32 + bit;
    };

    // ---- the rows: each warp copies the rows it folds (cp.async) in groups and folds each
    //      group as it lands (a warp whose rows land early computes while others still wait);
    //      a half-warp folds its rows of a group together: partial q.k and |k - mu|^2 over the
    //      lane's 8 dimensions, one reduce-scatter so that a few lanes hold each row's sums,
    //      the log-weight s - log u lane-parallel (log u from the per-call table or its closed
    //      form, the cross-polytope table, or 0 for T), one online-softmax step
    float m = -INFINITY, l = 0.0f, o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = 0.0f;
    const uint8_t* Kg = reinterpret_cast<const uint8_t*>(a.keys) +
                        static_cast<size_t>(bg) * a.ncap * kD * sizeof(KV);
    const uint8_t* Vg = reinterpret_cast<const uint8_t*>(a.values) +
                        static_cast<size_t>(bg) * a.ncap * kD * sizeof(KV);
    const bool weighted = !exact && a.K > 0;
    const int hw = 2 * warp + half;
    constexpr int kHalves = 2 * kAWarps;
    // One online-softmax step of this half-warp over its rows ent + kHalves j, j < cnt <= NB: the
    // partial sums of NB rows are reduce-scattered so that lanes j LPR .. j LPR + LPR - 1 hold row
    // j's (LPR = 16 / NB), the log-weight is computed lane-parallel, V is folded in.
    auto fold = [&](int ent, int cnt, auto nb_tag) {
        constexpr int NB = decltype(nb_tag)::value;
        constexpr int LPR = 16 / NB;
        if (cnt <= 0) return;
        float pd[NB], pk[NB];
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            const int r = j < cnt ? ent + j * kHalves : ent;
            float kf[8];
            load8(stage + r * kRowBytes + 8 * hl * sizeof(KV), static_cast<const KV*>(nullptr), kf);
            float d = 0.0f, k2 = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float x = kf[i] - mu8[i];
                k2 = fmaf(x, x, k2);
                d = fmaf(q8[i], kf[i], d);
            }
            pd[j] = d;
            pk[j] = k2;
        }
        // each level keeps half the rows and adds the partner's copy of them
#pragma unroll
        for (int lv = 0; (8 >> lv) >= LPR; ++lv) {
            const int off = 8 >> lv, nk = (NB / 2) >> lv;
            const bool up = (hl & off) != 0;
#pragma unroll
            for (int i = 0; i < nk; ++i) {
                const float sd = up ? pd[i] : pd[i + nk];
                const float sk = up ? pk[i] : pk[i + nk];
                const float rd = __shfl_xor_sync(hmask, sd, off);
                const float rk = __shfl_xor_sync(hmask, sk, off);
                pd[i] = (up ? pd[i + nk] : pd[i]) + rd;
                pk[i] = (up ? pk[i + nk] : pk[i]) + rk;
            }
        }
        float dot = pd[0], kb2 = pk[0];
#pragma unroll
        for (int sh = LPR / 2; sh; sh >>= 1) {
            dot += __shfl_xor_sync(hmask, dot, sh);
            kb2 += __shfl_xor_sync(hmask, kb2, sh);
        }
        const int jl = hl / LPR;
        float logit = -INFINITY;
        if (jl < cnt) {
            float lw = 0.0f;
            if (weighted) {
                const float den = qn * (a.radius ? rad : sqrtf(kb2));
                float cs = den > 0.0f ? (dot - qmu) / den : 0.0f;
                cs = fminf(1.0f, fmaxf(-1.0f, cs));
                if (a.table_only) {                      // cross-polytope: p has no closed form
                    const float tt = (cs + 1.0f) * (0.5f * kLuIntervals);
                    const int ti = min(static_cast<int>(tt), kLuIntervals - 1);
                    const float g0 = __ldg(a.logu_tab + ti), g1 = __ldg(a.logu_tab + ti + 1);
                    lw = fmaf(tt - static_cast<float>(ti), g1 - g0, g0);
                } else {
                    lw = log_inclusion_at(cs, a.logu_tab, a.K, a.L);
                }
            }
            logit = dot * a.scale - lw;
        }
        float bm = logit;
#pragma unroll
        for (int sh = 8; sh; sh >>= 1) bm = fmaxf(bm, __shfl_xor_sync(hmask, bm, sh));
        const float mn = fmaxf(m, bm);
        const float corr = __expf(m - mn);
        const float wgt = jl < cnt ? __expf(logit - mn) : 0.0f;
        float ws = (hl % LPR) ? 0.0f : wgt;                    // each row counted once
#pragma unroll
        for (int sh = 8; sh; sh >>= 1) ws += __shfl_xor_sync(hmask, ws, sh);
        l = fmaf(l, corr, ws);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] *= corr;
        const int src0 = lane & 16;
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            const float wj = __shfl_sync(hmask, wgt, src0 + LPR * j);
            if (j < cnt) {
                float vf[8];
                load8(stage + (ent + j * kHalves) * kRowBytes + (kD + 8 * hl) * sizeof(KV),
                      static_cast<const KV*>(nullptr), vf);
#pragma unroll
                for (int i = 0; i < 8; ++i) o[i] = fmaf(wj, vf[i], o[i]);
            }
        }
        m = mn;
    };
    static_assert(kAttendRows == 8 * kHalves, "the stage gives each half-warp 8 row slots");
    // the keys of the first kRowKeys entries, listed once (later ones are found on demand)
    for (int i = tid; i < min(nsel, kRowKeys); i += kAThreads) rowkey[i] = key_of(i);
    __syncthreads();
    // Group k of a warp: entries hw + 8 (4 k + j), j < 4, of its two half-warps, in the slots
    // hw + 8 (4 (k & 1) + j); group k + 2 reuses group k's slots once group k is folded.
    const int lo_hw = 2 * warp;                  // the warp's first half-warp has its most rows
    const int ngroups = nsel > lo_hw ? ((nsel - lo_hw + kHalves - 1) / kHalves + 3) / 4 : 0;
    const int my_rows = nsel > hw ? (nsel - hw + kHalves - 1) / kHalves : 0;
    auto issue = [&](int k) {                    // one row (K then V) per instruction
        if (k < ngroups) {
            for (int jj = 0; jj < 8; ++jj) {
                const int e = lo_hw + (jj & 1) + kHalves * (4 * k + (jj >> 1));
                if (e >= nsel) continue;
                const int r = lo_hw + (jj & 1) + kHalves * (4 * (k & 1) + (jj >> 1));
                const size_t key = static_cast<size_t>(e < kRowKeys ? rowkey[e] : key_of(e));
                if (!mp_check(a.status, static_cast<long long>(key), min(a.n, a.ncap),
                              kSiteAttendRow))
                    continue;
                for (int pc = lane; pc < kPieces; pc += 32) {
                    const uint8_t* src = (pc < kPieces / 2 ? Kg : Vg) + key * kD * sizeof(KV) +
                                         16 * (pc % (kPieces / 2));
                    cp_async16(stage + r * kRowBytes + 16 * pc, src);
                }
            }
        }
        cp_async_commit();                       // one group per call, empty or not
    };
    issue(0);
    issue(1);
    for (int k = 0; k < ngroups; ++k) {
        cp_async_wait_pending<1>();              // group k has landed (group k + 1 may not have)
        __syncwarp();
        fold(hw + kHalves * 4 * (k & 1), min(4, max(0, my_rows - 4 * k)),
             std::integral_constant<int, 4>());
        __syncwarp();                            // every lane is done with group k's slots
        issue(k + 2);
    }
    cp_async_wait_pending<0>();

    // ---- merge the two half-warps, then the warps (fixed order)
    {
        const float mo = __shfl_xor_sync(0xffffffffu, m, 16);
        const float lo = __shfl_xor_sync(0xffffffffu, l, 16);
        const float mn = fmaxf(m, mo);
        const float sa = mn == -INFINITY ? 0.0f : __expf(m - mn);
        const float sb2 = mn == -INFINITY ? 0.0f : __expf(mo - mn);
        l = l * sa + lo * sb2;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float oo = __shfl_xor_sync(0xffffffffu, o[i], 16);
            o[i] = o[i] * sa + oo * sb2;
        }
        m = mn;
        float* dst = cbuf + warp * kCombinePitch;
        if (half == 0) {
            reinterpret_cast<float4*>(dst)[2 * hl] = make_float4(o[0], o[1], o[2], o[3]);
            reinterpret_cast<float4*>(dst)[2 * hl + 1] = make_float4(o[4], o[5], o[6], o[7]);
        }
        if (lane == 0) {
            dst[128] = m;
            dst[129] = l;
        }
    }
    __syncthreads();
    const size_t prow = static_cast<size_t>(row) * nsp + sb;
    if (tid < kD && mp_check(a.status, static_cast<long long>(prow),
                             static_cast<long long>(gridDim.y) * nsp, kSiteAttendPartial)) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAWarps; ++w) M = fmaxf(M, cbuf[w * kCombinePitch + 128]);
        float Ls = 0.0f, Os = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kAWarps; ++w) {
                const float* rr = cbuf + w * kCombinePitch;
                const float s = __expf(rr[128] - M);
                Ls += s * rr[129];
                Os += s * rr[tid];
            }
        }
        a.po[prow * kD + tid] = Os;
        if (tid == 0) {
            a.pm[prow] = M;
            a.pl[prow] = Ls;
        }
    }

    // ---- the last CTA of this query row merges the row's partials: the barrier orders every
    //      thread's partial writes before thread 0's release-acquire increment
    __syncthreads();
    if (tid == 0)
        misc[4] = (atomic_add_acq_rel_gpu(a.counters + row, 1u) == static_cast<unsigned>(nsp - 1));
    __syncthreads();
    if (!misc[4]) return;

    // ---- merge: warp w folds the row's partials j = w, w + 4, w + 8, ... in ascending order,
    //      lane l dims 4l..4l+3; a pass loads kMergeRegs partials per warp into registers at once
    //      (one round trip covers 4 * kMergeRegs partials) and rescales a running maximum. The
    //      four warps' (m, l, o) are then joined through shared memory in warp order.
    const size_t rb = static_cast<size_t>(row) * nsp;
    float mw = -INFINITY, lw = 0.0f;
    float4 ow = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int j0 = warp; j0 < nsp; j0 += kAWarps * kMergeRegs) {
        float pmj[kMergeRegs], plj[kMergeRegs];
        float4 poj[kMergeRegs];
#pragma unroll
        for (int c = 0; c < kMergeRegs; ++c) {
            const int j = j0 + kAWarps * c;
            pmj[c] = -INFINITY;
            plj[c] = 0.0f;
            poj[c] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (j < nsp) {
                pmj[c] = __ldcg(a.pm + rb + j);
                plj[c] = __ldcg(a.pl + rb + j);
                poj[c] = __ldcg(reinterpret_cast<const float4*>(a.po + (rb + j) * kD) + lane);
            }
        }
        float mn = mw;
#pragma unroll
        for (int c = 0; c < kMergeRegs; ++c) mn = fmaxf(mn, pmj[c]);
        if (mn != -INFINITY) {
            const float sa = expf(mw - mn);      // 0 while nothing is folded (mw = -inf)
            lw *= sa;
            ow = make_float4(ow.x * sa, ow.y * sa, ow.z * sa, ow.w * sa);
#pragma unroll
            for (int c = 0; c < kMergeRegs; ++c) {
                const float sj = expf(pmj[c] - mn);   // 0 for an empty partial (m = -inf)
                lw = fmaf(sj, plj[c], lw);
                ow = make_float4(fmaf(sj, poj[c].x, ow.x), fmaf(sj, poj[c].y, ow.y),
                                 fmaf(sj, poj[c].z, ow.z), fmaf(sj, poj[c].w, ow.w));
            }
            mw = mn;
        }
    }
    {
        float* dst = cbuf + warp * kCombinePitch;
        reinterpret_cast<float4*>(dst)[lane] = ow;
        if (lane == 0) {
            dst[128] = mw;
            dst[129] = lw;
        }
    }
    __syncthreads();
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAWarps; ++w) M = fmaxf(M, cbuf[w * kCombinePitch + 128]);
    float Ls = 0.0f, Os = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kAWarps; ++w) {
            const float* rr = cbuf + w * kCombinePitch;
            const float sw = expf(rr[128] - M);
            Ls = fmaf(sw, rr[129], Ls);
            Os = fmaf(sw, rr[tid], Os);
        }
    }
    // a query with a NaN or infinite element has no defined output: NaN, not a silent zero
    if (mp_check(a.status, row, gridDim.y, kSiteAttendPartial))
        a.out[static_cast<size_t>(row) * kD + tid] =
            isfinite(qn) ? (Ls > 0.0f ? Os / Ls : 0.0f) : __int_as_float(0x7fc00000);
    if (tid == 0) a.counters[row] = 0u;
}

// Inspection: log u at given cosines exactly as the attend kernel evaluates it for SimHash codes
// (the per-call table, here rebuilt in shared memory, and the closed form where it is not used).
__global__ void log_inclusion_kernel(const float* cosines, int count, int K, int L, float* out) {
    __shared__ float tab[kLuIntervals + 1];      // the table the query encoding fills per call
    __shared__ float buf[2 * kLogUSegment + 3];
    for (int seg = 0; seg < kLogUSegments; ++seg) log_inclusion_segment(seg, K, L, buf, tab);
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < count) out[i] = log_inclusion_at(cosines[i], tab, K, L);
}

typedef void (*KernelFn)(const CArgs);

KernelFn pick_collide(int G) {
    switch (G) {
        case 1: return collide_kernel<1>;
        case 2: return collide_kernel<2>;
        case 4: return collide_kernel<4>;
        case 8: return collide_kernel<8>;
        default: return nullptr;
    }
}

typedef void (*AttendFn)(const AArgs);

AttendFn pick_attend(bool kv_bf16) {
    return kv_bf16 ? attend_kernel<__nv_bfloat16> : attend_kernel<float>;
}

size_t collide_smem_for(int G, int cpad, int K) {
    switch (G) {
        case 1: return collide_smem_bytes<1>(cpad, K);
        case 2: return collide_smem_bytes<2>(cpad, K);
        case 4: return collide_smem_bytes<4>(cpad, K);
        case 8: return collide_smem_bytes<8>(cpad, K);
        default: return 0;
    }
}

size_t attend_smem_for(int nblk, bool kv_bf16) {
    return attend_smem(attend_partials(nblk), kv_bf16 ? 2 : 4).total;
}

constexpr size_t kMaxSmem = 232448;   // 227 KB opt-in per CTA

}  // namespace

bool decode_supported(const DecodeShape& s, bool kv_bf16) {
    const int G = s.Hq / s.Hkv;
    if (!pick_collide(G)) return false;
    return collide_smem_for(G, s.cpad, s.K) <= kMaxSmem &&
           attend_smem_for(s.nblk, kv_bf16) <= kMaxSmem;
}

cudaError_t prepare_decode() {
    const int Gs[4] = {1, 2, 4, 8};
    for (int i = 0; i < 4; ++i) {
        cudaError_t e = cudaFuncSetAttribute(pick_collide(Gs[i]),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kMaxSmem));
        if (e != cudaSuccess) return e;
    }
    for (int bf = 0; bf < 2; ++bf) {
        cudaError_t e = cudaFuncSetAttribute(pick_attend(bf != 0),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kMaxSmem));
        if (e != cudaSuccess) return e;
    }
    // one shared-memory carve-out (the largest) for every kernel of a decode step: an SM still
    // running CTAs of one kernel can then take CTAs of the next without first draining to
    // reconfigure its L1 / shared-memory split
    const void* fns[] = {reinterpret_cast<const void*>(qencode_kernel),
                         reinterpret_cast<const void*>(pick_collide(1)),
                         reinterpret_cast<const void*>(pick_collide(2)),
                         reinterpret_cast<const void*>(pick_collide(4)),
                         reinterpret_cast<const void*>(pick_collide(8)),
                         reinterpret_cast<const void*>(pick_attend(false)),
                         reinterpret_cast<const void*>(pick_attend(true))};
    for (const void* f : fns) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
    }
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, log_inclusion_kernel);
    if (e != cudaSuccess) return e;
    return cudaFuncGetAttributes(&fa, qencode_kernel);
}

cudaError_t launch_log_inclusion(const float* cosines, int count, int K, int L, float* out,
                                 cudaStream_t st) {
    if (count <= 0) return cudaSuccess;
    log_inclusion_kernel<<<(count + 255) / 256, 256, 0, st>>>(cosines, count, K, L, out);
    return cudaGetLastError();
}

cudaError_t launch_qencode(const void* q, bool q_bf16, const float* centre, const void* W,
                           bool w_bf16, const DecodeShape& s, const DecodeScratch& ws,
                           cudaStream_t st) {
    QArgs qa;
    qa.q = q;
    qa.W = W;
    qa.centre = centre;
    qa.qbits = ws.qbits;
    qa.qmask = ws.qmask;
    qa.qstat = ws.qstat;
    qa.counters = ws.counters;
    qa.q_bf16 = q_bf16;
    qa.w_bf16 = w_bf16;
    qa.BHq = s.B * s.Hq;
    qa.Hq = s.Hq;
    qa.G = s.Hq / s.Hkv;
    qa.C = s.C;
    qa.cpad = s.cpad;
    qa.qwords = s.qwords;
    qa.n_counters = ws.n_counters;
    qa.logu_tab = ws.logu_tab;
    qa.status = device_status_ptr();
    qa.K = s.K;
    qa.L = s.L;
    qa.qrow_ctas = (qa.BHq + kQRows - 1) / kQRows;
    const dim3 qgrid(s.qwords > 0 ? s.qwords : 1, qa.qrow_ctas + 1);
    qencode_kernel<<<qgrid, kThreads, 0, st>>>(qa);
    return cudaGetLastError();
}

namespace {
CArgs scan_args(const uint32_t* codes, const DecodeShape& s, const DecodeScratch& ws, int blk0) {
    CArgs ca;
    ca.codes = codes;
    ca.qmask = ws.qmask;
    ca.selmask = ws.selmask;
    ca.n = s.n;
    ca.nblk = s.nblk;
    ca.Hq = s.Hq;
    ca.Hkv = s.Hkv;
    ca.K = s.K;
    ca.L = s.L;
    ca.C = s.C;
    ca.cpad = s.cpad;
    ca.n_sink = s.n_sink;
    ca.n_local = s.n_local;
    ca.cblk = s.cblk;
    ca.blk0 = blk0;
    ca.status = device_status_ptr();
    return ca;
}

}  // namespace

cudaError_t launch_collide(const void* q, bool q_bf16, const uint32_t* codes,
                           const float* centre, const void* keys, const void* values,
                           bool kv_bf16, const DecodeShape& s, float* out,
                           const DecodeScratch& ws, cudaStream_t st, int blk0) {
    const int G = s.Hq / s.Hkv;
    const CArgs ca = scan_args(codes, s, ws, blk0);
    KernelFn scan = pick_collide(G);
    const size_t smem_scan = collide_smem_for(G, s.cpad, s.K);
    if (!scan || smem_scan > kMaxSmem || attend_smem_for(s.nblk, kv_bf16) > kMaxSmem)
        return cudaErrorNotSupported;
    if (blk0 < 0 || blk0 > s.nblk) return cudaErrorInvalidValue;
    if (blk0 < s.nblk) {
        const cudaError_t e = launch_dependent(scan, dim3(s.nblk - blk0, s.B * s.Hkv),
                                               dim3(kThreads), smem_scan, st, ca);
        if (e != cudaSuccess) return e;
    }
    return launch_attend(q, q_bf16, centre, keys, values, kv_bf16, s, out, ws, st);
}

cudaError_t launch_attend(const void* q, bool q_bf16, const float* centre, const void* keys,
                          const void* values, bool kv_bf16, const DecodeShape& s, float* out,
                          const DecodeScratch& ws, cudaStream_t st) {
    const int G = s.Hq / s.Hkv;
    AttendFn attend = pick_attend(kv_bf16);
    const size_t smem_att = attend_smem_for(s.nblk, kv_bf16);
    if (smem_att > kMaxSmem) return cudaErrorNotSupported;
    AArgs aa;
    aa.selmask = ws.selmask;
    aa.qstat = ws.qstat;
    aa.q = q;
    aa.centre = centre;
    aa.keys = keys;
    aa.values = values;
    aa.pm = ws.pm;
    aa.pl = ws.pl;
    aa.po = ws.po;
    aa.counters = ws.counters;
    aa.out = out;
    aa.logu_tab = s.logu_ext ? s.logu_ext : ws.logu_tab;
    aa.table_only = s.logu_ext != nullptr;     // cross-polytope: p has no closed form
    aa.q_bf16 = q_bf16;
    aa.n = s.n;
    aa.nblk = s.nblk;
    aa.nsb = (s.nblk + kAttendBlocks - 1) / kAttendBlocks;
    aa.Hq = s.Hq;
    aa.Hkv = s.Hkv;
    aa.G = G;
    aa.K = s.K;
    aa.L = s.L;
    aa.n_sink = s.n_sink;
    aa.n_local = s.n_local;
    aa.ncap = s.ncap;
    aa.status = device_status_ptr();
    aa.radius = s.radius;
    aa.scale = s.scale;
    {
        const AttendSmem m = attend_smem(attend_partials(s.nblk), kv_bf16 ? 2 : 4);
        aa.work_bytes = static_cast<int>(m.work);
    }
    return launch_dependent(attend, dim3(aa.nsb + 1, s.B * s.Hq), dim3(kAThreads), smem_att, st,
                            aa);
}

}  // namespace mp
