// Decode step: query encoding; a scan kernel that streams the packed codes of a block of 1024
// keys and selects the keys colliding with the query in >= 2 tables; an attend kernel that
// gathers only those K/V rows and folds them with importance weights into partial softmaxes,
// the last CTA of each query row merging the partials by log-sum-exp.
//
// The method is Algorithm 1 of "MagicPIG: LSH Sampling for Efficient LLM Generation" (method
// details, algorithm execution), with the inclusion probability of the hash-function-choice
// section and the exact sink/local set ("static cache") of the system co-design section, whose
// "recursive attention" merge of partial outputs is the log-sum-exp merge done here.
#include "mp_internal.cuh"

namespace mp {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr float kLogFltMin = -87.336544750553102f;   // log(FLT_MIN)
constexpr float kPi = 3.14159265358979323846f;
constexpr int kCombinePitch = 132;                  // floats per (warp, head) partial: o, m, l
constexpr int kAttendBlocks = kAttendBlockGroup;
constexpr int kAWarps = 4;                          // attend CTA: 4 warps, 8 half-warps on rows
static_assert(kAttendBlocks <= kAWarps, "one warp lists each block of an attend CTA");
constexpr int kAThreads = 32 * kAWarps;
constexpr int kRing = 4;                            // rows in flight per lane (cp.async ring)
static_assert(kAThreads == kD, "the attend merge gives one thread to each of the 128 output dims");
constexpr int kRingDepth = 4;                       // tables in flight per warp in the async scan
constexpr int kRingMinK = 8, kRingMaxK = 11;        // K range the async scan handles
constexpr int kLuIntervals = kLogUTableIntervals;   // log u table: cosine grid on [-1, 1]

// 1 / (j + 1) for the binomial-tail series below
__constant__ float c_inv_next[66] = {
    1.0f / 1, 1.0f / 2, 1.0f / 3, 1.0f / 4, 1.0f / 5, 1.0f / 6, 1.0f / 7, 1.0f / 8, 1.0f / 9,
    1.0f / 10, 1.0f / 11, 1.0f / 12, 1.0f / 13, 1.0f / 14, 1.0f / 15, 1.0f / 16, 1.0f / 17,
    1.0f / 18, 1.0f / 19, 1.0f / 20, 1.0f / 21, 1.0f / 22, 1.0f / 23, 1.0f / 24, 1.0f / 25,
    1.0f / 26, 1.0f / 27, 1.0f / 28, 1.0f / 29, 1.0f / 30, 1.0f / 31, 1.0f / 32, 1.0f / 33,
    1.0f / 34, 1.0f / 35, 1.0f / 36, 1.0f / 37, 1.0f / 38, 1.0f / 39, 1.0f / 40, 1.0f / 41,
    1.0f / 42, 1.0f / 43, 1.0f / 44, 1.0f / 45, 1.0f / 46, 1.0f / 47, 1.0f / 48, 1.0f / 49,
    1.0f / 50, 1.0f / 51, 1.0f / 52, 1.0f / 53, 1.0f / 54, 1.0f / 55, 1.0f / 56, 1.0f / 57,
    1.0f / 58, 1.0f / 59, 1.0f / 60, 1.0f / 61, 1.0f / 62, 1.0f / 63, 1.0f / 64, 1.0f / 65,
    1.0f / 66};

// log u(p) = log P[Binomial(L, p^K) >= 2] in fp32, two branches: directly when L p^K >= 1/2,
// else as log t_2 + log(1 + sum_{j>=3} t_j / t_2) with t_j the binomial terms; p <= 0 clamps to
// log(FLT_MIN). log C(L, 2) comes in as log_c2, the series ratios (L - j) / (j + 1) use a
// reciprocal table (at most 64 terms: below L p^K = 1/2 they shrink at least threefold per step),
// log p and exp use the fast hardware approximations (errors far below the 1e-3 output
// tolerance); log1p(-x) stays exact because (L - 2) multiplies it.
__device__ __forceinline__ float log_inclusion_fast(float p, int K, int L, float log_c2) {
    if (L < 2) return -INFINITY;
    if (K == 0) return 0.0f;                       // p^0 = 1 and L >= 2: u = 1
    if (!(p > 0.0f)) return kLogFltMin;
    const float lx = static_cast<float>(K) * __logf(p);
    const float x = __expf(lx);
    const float Lf = static_cast<float>(L);
    if (x >= 1.0f) return 0.0f;
    const float l1 = log1pf(-x);
    if (Lf * x >= 0.5f) {
        const float u = 1.0f - __expf(Lf * l1) - Lf * x * __expf((Lf - 1.0f) * l1);
        return __logf(fmaxf(u, 1.17549435e-38f));
    }
    const float r = __fdividef(x, 1.0f - x);
    float term = 1.0f, tot = 1.0f;
    const int jmax = min(L, 65);
    for (int j = 2; j < jmax; ++j) {
        term *= (Lf - static_cast<float>(j)) * c_inv_next[j] * r;
        tot += term;
        if (term < 1e-9f * tot) break;
    }
    return log_c2 + 2.0f * lx + (Lf - 2.0f) * l1 + __logf(tot);
}

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
    float* logu_tab;
    int q_bf16, w_bf16, BHq, Hq, G, C, cpad, qwords, n_counters, K, L, qrow_ctas;
};

__global__ void __launch_bounds__(kThreads) qencode_kernel(const QArgs a) {
    __shared__ float Qs[kQRows][kD];
    __shared__ float Ws[kD][32];                 // this word's 32 hyperplane columns
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    allow_dependents();                          // the scan may start streaming codes meanwhile
    if (blockIdx.y == a.qrow_ctas) {
        // the extra row of CTAs fills the log u table on the cosine grid c_i = -1 + 2 i / N
        for (int i = blockIdx.x * kThreads + tid; i <= kLuIntervals; i += gridDim.x * kThreads) {
            const float c = fminf(1.0f, -1.0f + 2.0f * static_cast<float>(i) / kLuIntervals);
            a.logu_tab[i] = log_inclusion_ref(1.0f - acosf(c) / kPi, a.K, a.L);
        }
        return;
    }
    const int wd = blockIdx.x, r0 = blockIdx.y * kQRows;
    const int nq = min(kQRows, a.BHq - r0);
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
    const int row = r0 + warp;
    const int Hkv = a.Hq / a.G;
    if (warp < nq && a.C > 0) {
        const int j = wd * 32 + lane;
        float s = 0.0f;
#pragma unroll 16
        for (int e = 0; e < kD; ++e) s = fmaf(Ws[e][lane], Qs[warp][e], s);
        const bool bit = j < a.C && s > 0.0f;
        const uint32_t word = __ballot_sync(0xffffffffu, bit);
        if (lane == 0) a.qbits[static_cast<size_t>(row) * a.qwords + wd] = word;
        const int b = row / a.Hq, h = row % a.Hq;
        const size_t bg = static_cast<size_t>(b) * Hkv + h / a.G;
        if (j < a.cpad)
            a.qmask[(bg * a.cpad + j) * a.G + (h % a.G)] = bit ? 0u : 0xffffffffu;
    }
    if (blockIdx.x == 0) {
        if (warp < nq) {
            const int b = row / a.Hq, h = row % a.Hq, g = h / a.G;
            const float* mu = a.centre + (static_cast<size_t>(b) * Hkv + g) * kD;
            float nn = 0.0f, qm = 0.0f;
            for (int e = lane; e < kD; e += 32) {
                const float x = Qs[warp][e];
                nn = fmaf(x, x, nn);
                qm = fmaf(x, mu[e], qm);
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                nn += __shfl_xor_sync(0xffffffffu, nn, o);
                qm += __shfl_xor_sync(0xffffffffu, qm, o);
            }
            if (lane == 0) a.qstat[row] = make_float4(sqrtf(nn), qm, 0.0f, 0.0f);
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
};

// Attend CTA shared memory: [work][cbuf][misc]. The work region holds the CTA's row list, and in
// the merging CTA up to `merge_cap` staged partial outputs (all of them unless that exceeds
// 48 KB; the merge then runs in rounds).
struct AttendSmem {
    size_t work, total;
    int merge_cap;
};
// Bytes of the per-lane row ring for K/V elements of kv_elem bytes: kRing slots of a K and a V
// fragment (16 bytes per bf16 fragment, 32 per fp32 one) for each of the CTA's lanes.
__host__ __device__ constexpr size_t attend_ring_bytes(size_t kv_elem) {
    return static_cast<size_t>(kRing) * 2 * kv_elem * 8 * kAThreads;
}

inline AttendSmem attend_smem(int nsp, size_t kv_elem) {
    constexpr size_t kList = static_cast<size_t>(kAttendBlocks) * kKeysPerBlock * 4;
    constexpr size_t kRow = static_cast<size_t>(kD) * 4;
    size_t work = static_cast<size_t>(nsp) * kRow;
    if (work > 48 * 1024) work = 48 * 1024;
    if (work < kList) work = kList;
    AttendSmem m;
    m.work = work;
    m.merge_cap = static_cast<int>(work / kRow);
    m.total = work + static_cast<size_t>(kAWarps) * kCombinePitch * 4 + 64 +
              attend_ring_bytes(kv_elem);
    return m;
}

template <int G>
size_t collide_smem_bytes(int cpad, int K) {
    const size_t ring = (K >= kRingMinK && K <= kRingMaxK)
                            ? static_cast<size_t>(kWarps) * kRingDepth * K * kWordsPerBlock * 4
                            : 0;
    return static_cast<size_t>(cpad) * G * 4 + static_cast<size_t>(kWarps) * 2 * G * 32 * 4 + ring;
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
    const float* logu_tab;
    int q_bf16, n, nblk, nsb, Hq, Hkv, G, K, L, n_sink, n_local;
    int ncap;                                    // K/V rows per head in memory
    const float* radius;                         // MIPS variant: longest centred key per head
    int table_only;                              // log u from the table at every cosine
    float scale, log_c2;
    int merge_cap;                               // partials staged per merge round
    int work_bytes;                              // bytes of the list / merge stage region
};

// Collide + select: per (1024-key block, sequence x KV head) the selection words
// S_h = [>= 2 of L tables match] & valid & not T, for every query head h of the group.
template <int G>
__global__ void __launch_bounds__(kThreads, 3) collide_kernel(const CArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int blk = blockIdx.x + a.blk0, bg = blockIdx.y;
    const int b = bg / a.Hkv, g = bg % a.Hkv;
    const int row0 = b * a.Hq + g * G;          // first query row of this KV head's group
    uint32_t* qneg = reinterpret_cast<uint32_t*>(smem);                    // [cpad][G]
    uint32_t* gebuf = qneg + static_cast<size_t>(a.cpad) * G;              // [8][2][G][32]
    uint32_t* ring = gebuf + kWarps * 2 * G * 32 +                         // [8][depth][K][32]
                     static_cast<size_t>(warp) * kRingDepth * a.K * kWordsPerBlock;

    // ---- before the query masks exist: let the attend kernel be scheduled (it waits for this
    //      kernel's completion itself), and start this warp's first tables of codes (an input
    //      of the call): into the ring for the ring's K, else into L2
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

    // ---- prologue: the group's query masks (one contiguous piece)
    {
        const uint4* src = reinterpret_cast<const uint4*>(a.qmask +
                                                          static_cast<size_t>(bg) * a.cpad * G);
        const int n16 = a.cpad * G / 4;
        for (int i = tid; i < n16; i += kThreads) cp_async16(qneg + 4 * i, src + i);
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- phase 1: per 32-key word (lane), per table, match = AND_b (plane ^ qmask); keep
    //      bit-sliced saturating counters ge1 = (>= 1 match), ge2 = (>= 2 matches)
    uint32_t ge1[G], ge2[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        ge1[h] = 0u;
        ge2[h] = 0u;
    }
    {
        const uint32_t* cb = cb0 + lane;
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
            default: scan_tables_any<G>(cb, qneg, a.K, t0, t1, ge1, ge2); break;
        }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
        gebuf[((warp * 2 + 0) * G + h) * 32 + lane] = ge1[h];
        gebuf[((warp * 2 + 1) * G + h) * 32 + lane] = ge2[h];
    }
    __syncthreads();
    if (tid < G * 32) {
        const int h = tid >> 5, w = lane;
        uint32_t g1 = 0u, g2 = 0u;
#pragma unroll
        for (int ww = 0; ww < kWarps; ++ww) {
            const uint32_t a1 = gebuf[((ww * 2 + 0) * G + h) * 32 + w];
            const uint32_t a2 = gebuf[((ww * 2 + 1) * G + h) * 32 + w];
            g2 |= a2 | (g1 & a1);
            g1 |= a1;
        }
        const int key0 = blk * kKeysPerBlock + w * 32;
        const uint32_t valid = bits_below(a.n - key0);
        const uint32_t tm =
            (bits_below(a.n_sink - key0) | ~bits_below(a.n - a.n_local - key0)) & valid;
        const uint32_t s = g2 & valid & ~tm;
        a.selmask[(static_cast<size_t>(row0 + h) * a.nblk + blk) * 32 + w] = s;
    }
    __syncthreads();
}

// A K or V row fragment: the 8 elements [8 hl, 8 hl + 8) a lane of a half-warp holds
template <typename KV>
struct RowFrag;
template <>
struct RowFrag<__nv_bfloat16> {
    uint4 k, v;
    __device__ __forceinline__ void from_pieces(const uint4 (&p)[2]) { k = p[0]; v = p[1]; }
    __device__ __forceinline__ void unpack(float (&kf)[8], float (&vf)[8]) const {
        const uint32_t kw[4] = {k.x, k.y, k.z, k.w}, vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kw[i]));
            const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vw[i]));
            kf[2 * i] = a.x;
            kf[2 * i + 1] = a.y;
            vf[2 * i] = b.x;
            vf[2 * i + 1] = b.y;
        }
    }
};
template <>
struct RowFrag<float> {
    float4 k0, k1, v0, v1;
    __device__ __forceinline__ void from_pieces(const uint4 (&p)[4]) {
        k0 = *reinterpret_cast<const float4*>(&p[0]);
        k1 = *reinterpret_cast<const float4*>(&p[1]);
        v0 = *reinterpret_cast<const float4*>(&p[2]);
        v1 = *reinterpret_cast<const float4*>(&p[3]);
    }
    __device__ __forceinline__ void unpack(float (&kf)[8], float (&vf)[8]) const {
        kf[0] = k0.x; kf[1] = k0.y; kf[2] = k0.z; kf[3] = k0.w;
        kf[4] = k1.x; kf[5] = k1.y; kf[6] = k1.z; kf[7] = k1.w;
        vf[0] = v0.x; vf[1] = v0.y; vf[2] = v0.z; vf[3] = v0.w;
        vf[4] = v1.x; vf[5] = v1.y; vf[6] = v1.z; vf[7] = v1.w;
    }
};

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
// Each half-warp takes every eighth row; each lane streams its own pieces of the rows (16 bytes
// of a bf16 K row and of its V row) through a private ring of kRing slots in shared memory with
// cp.async, so kRing rows per lane are in flight while the current one is reduced.
template <typename KV>
__global__ void __launch_bounds__(kAThreads, 6) attend_kernel(const AArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sb = blockIdx.x, row = blockIdx.y;
    const int b = row / a.Hq, h = row % a.Hq;
    const int bg = b * a.Hkv + h / a.G;
    const bool exact = sb == a.nsb;              // this CTA takes T
    const int nsp = a.nsb + 1;                   // partials per query row

    int* lidx = reinterpret_cast<int*>(smem);
    float* cbuf = reinterpret_cast<float*>(smem + a.work_bytes);
    int* misc = reinterpret_cast<int*>(cbuf + kAWarps * kCombinePitch);  // [0..3] counts, [4]

    const int half = lane >> 4, hl = lane & 15;
    float q8[8], mu8[8];                         // inputs of the call: readable right away
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        q8[i] = load_elem(a.q, a.q_bf16, static_cast<size_t>(row) * kD + 8 * hl + i);
        mu8[i] = a.centre[static_cast<size_t>(bg) * kD + 8 * hl + i];
    }
    wait_for_predecessor();                      // selection words, query norms, log u table
    const float4 st = a.qstat[row];
    const float qn = st.x, qmu = st.y;
    const float rad = a.radius ? a.radius[bg] : 0.0f;   // MIPS: cos = q.(k - mu) / (|q| r)

    // ---- the rows of this CTA: T by arithmetic, or the selected keys of its blocks by a list
    const int t_a = min(a.n_sink, a.n), t_b = max(a.n - a.n_local, t_a);
    int nsel;
    if (exact) {
        nsel = t_a + (a.n - t_b);
    } else {
        const int blk0 = sb * kAttendBlocks;
        const int nb = min(kAttendBlocks, a.nblk - blk0);
        uint32_t U = 0u;
        int key0 = 0, excl = 0;
        if (warp < nb) {
            const int blk = blk0 + warp;
            key0 = blk * kKeysPerBlock + lane * 32;
            {
                // the scan already masked its words; selection words from elsewhere (the
                // bucketed lookup's >= 2 bitmap) need valid & not T here
                const uint32_t valid = bits_below(a.n - key0);
                const uint32_t tmask =
                    (bits_below(a.n_sink - key0) | ~bits_below(a.n - a.n_local - key0)) & valid;
                U = a.selmask[(static_cast<size_t>(row) * a.nblk + blk) * 32 + lane] & valid & ~tmask;
            }
            const int c = __popc(U);
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            excl = incl - c;
            if (lane == 31) misc[warp] = incl;
        }
        __syncthreads();
        int base = 0;
        nsel = 0;
        for (int w = 0; w < nb; ++w) {
            if (w < warp) base += misc[w];
            nsel += misc[w];
        }
        if (warp < nb) {
            int pos = base + excl;
            uint32_t bits = U;
            while (bits) {
                const int bit = __ffs(bits) - 1;
                bits &= bits - 1;
                lidx[pos++] = key0 + bit;
            }
        }
        __syncthreads();
    }
    auto key_of = [&](int r) { return exact ? (r < t_a ? r : t_b + (r - t_a)) : lidx[r]; };

    // ---- rows: half-warp hw takes entries hw, hw + 8, ...; each lane streams its own 16-byte
    //      pieces of the rows through a private cp.async ring of kRing slots in shared memory
    float m = -INFINITY, l = 0.0f, o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = 0.0f;
    constexpr int kPieces = static_cast<int>(sizeof(KV)) / 2;     // 16-byte pieces per fragment
    const uint8_t* Kb = reinterpret_cast<const uint8_t*>(a.keys) +
                        (static_cast<size_t>(bg) * a.ncap * kD + 8 * hl) * sizeof(KV);
    const uint8_t* Vb = reinterpret_cast<const uint8_t*>(a.values) +
                        (static_cast<size_t>(bg) * a.ncap * kD + 8 * hl) * sizeof(KV);
    uint4* ring = reinterpret_cast<uint4*>(smem + a.work_bytes + kAWarps * kCombinePitch * 4 + 64);
    const bool weighted = !exact && a.K > 0;
    const int hw = 2 * warp + half;
    auto issue = [&](int k) {                    // entry hw + 8 k into slot k % kRing
        const int r = hw + 2 * kAWarps * k;
        if (r < nsel) {
            const size_t off = static_cast<size_t>(key_of(r)) * kD * sizeof(KV);
            const int slot = k % kRing;
#pragma unroll
            for (int c = 0; c < kPieces; ++c) {
                cp_async16(ring + ((slot * 2 + 0) * kPieces + c) * kAThreads + tid, Kb + off + 16 * c);
                cp_async16(ring + ((slot * 2 + 1) * kPieces + c) * kAThreads + tid, Vb + off + 16 * c);
            }
        }
        cp_async_commit();
    };
    const int nk = (nsel - 2 * warp + 2 * kAWarps - 1) / (2 * kAWarps);   // the warp's iterations
#pragma unroll
    for (int k = 0; k < kRing; ++k) issue(k);
    for (int k = 0; k < nk; ++k) {
        cp_async_wait_pending<kRing - 1>();
        const bool live = hw + 2 * kAWarps * k < nsel;
        const int slot = k % kRing;
        RowFrag<KV> f;
        {
            uint4 kv[2 * kPieces];
#pragma unroll
            for (int c = 0; c < kPieces; ++c) {
                kv[c] = ring[((slot * 2 + 0) * kPieces + c) * kAThreads + tid];
                kv[kPieces + c] = ring[((slot * 2 + 1) * kPieces + c) * kAThreads + tid];
            }
            f.from_pieces(kv);
        }
        float kf[8], vf[8];
        f.unpack(kf, vf);
        issue(k + kRing);                        // the slot's pieces are in registers now
        float kb2 = 0.0f, dot = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float dk = kf[i] - mu8[i];
            kb2 = fmaf(dk, dk, kb2);
            dot = fmaf(q8[i], kf[i], dot);
        }
#pragma unroll
        for (int sh = 8; sh; sh >>= 1) {
            kb2 += __shfl_xor_sync(0xffffffffu, kb2, sh);
            dot += __shfl_xor_sync(0xffffffffu, dot, sh);
        }
        if (live) {
            float lw = 0.0f;
            if (weighted) {
                const float den = qn * (a.radius ? rad : sqrtf(kb2));
                float cs = den > 0.0f ? __fdividef(dot - qmu, den) : 0.0f;
                cs = fminf(1.0f, fmaxf(-1.0f, cs));
                if (a.table_only || (cs > -0.9f && cs < 0.999f)) {
                    const float tt = (cs + 1.0f) * (0.5f * kLuIntervals);
                    const int i = min(static_cast<int>(tt), kLuIntervals - 1);
                    const float g0 = __ldg(a.logu_tab + i), g1 = __ldg(a.logu_tab + i + 1);
                    lw = fmaf(tt - static_cast<float>(i), g1 - g0, g0);
                } else {
                    lw = log_inclusion_fast(1.0f - acosf(cs) * (1.0f / kPi), a.K, a.L, a.log_c2);
                }
            }
            const float logit = dot * a.scale - lw;
            const float mn = fmaxf(m, logit);
            const float corr = __expf(m - mn);
            const float pw = __expf(logit - mn);
            l = l * corr + pw;
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = fmaf(o[i], corr, pw * vf[i]);
            m = mn;
        }
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
    if (tid < kD) {
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

    // ---- merge: the partial outputs are staged in shared memory (the row list's space) with
    //      cp.async, issued before the maximum is known; m and l of the partials are loaded
    //      meanwhile and sc[j] = exp(m_j - M) kept in cbuf. Rounds of kMergeCap partials.
    const int kMergeCap = a.merge_cap;
    float* stage = reinterpret_cast<float*>(smem);
    float* red = cbuf;                            // [0, 8): reductions
    float* sc = cbuf + 8;                         // scales, kMergeCap at a time
    const size_t rb = static_cast<size_t>(row) * nsp;
    auto stage_round = [&](int j0) {
        const int cnt = min(kMergeCap, nsp - j0);
        const float* src = a.po + (rb + j0) * kD;
        for (int i = tid; i < cnt * (kD / 4); i += kAThreads) cp_async16(stage + 4 * i, src + 4 * i);
        cp_async_commit();
    };
    stage_round(0);
    // thread j < nsp keeps (m_j, l_j) of the first round from this one round trip
    float pm0 = -INFINITY, pl0 = 0.0f;
    if (tid < nsp) {
        pm0 = __ldcg(a.pm + rb + tid);
        pl0 = __ldcg(a.pl + rb + tid);
    }
    float mx = pm0;
    for (int j = tid + kAThreads; j < nsp; j += kAThreads) mx = fmaxf(mx, __ldcg(a.pm + rb + j));
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAWarps; ++w) M = fmaxf(M, red[w]);
    float ls = 0.0f, Os = 0.0f;
    for (int j0 = 0; j0 < nsp; j0 += kMergeCap) {
        const int cnt = min(kMergeCap, nsp - j0);
        if (tid < cnt) {
            const float pmj = j0 == 0 ? pm0 : __ldcg(a.pm + rb + j0 + tid);
            const float plj = j0 == 0 ? pl0 : __ldcg(a.pl + rb + j0 + tid);
            const float sj = M == -INFINITY ? 0.0f : expf(pmj - M);
            sc[tid] = sj;
            ls = fmaf(sj, plj, ls);
        }
        cp_async_wait_pending<0>();
        __syncthreads();                         // staged rows and scales visible to all
#pragma unroll 8
        for (int j = 0; j < cnt; ++j) Os = fmaf(sc[j], stage[j * kD + tid], Os);
        __syncthreads();                         // stage and scales are refilled next round
        if (j0 + kMergeCap < nsp) stage_round(j0 + kMergeCap);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
    if (lane == 0) red[4 + warp] = ls;
    __syncthreads();
    float Ls = 0.0f;
#pragma unroll
    for (int w = 0; w < kAWarps; ++w) Ls += red[4 + w];
    a.out[static_cast<size_t>(row) * kD + tid] = Ls > 0.0f ? Os / Ls : 0.0f;
    if (tid == 0) a.counters[row] = 0u;
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

// launch `kern` so that it may be scheduled while the previous kernel in the stream finishes
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
    cudaFuncAttributes fa;
    return cudaFuncGetAttributes(&fa, qencode_kernel);
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
    qa.n_counters = s.B * s.Hq;
    qa.logu_tab = ws.logu_tab;
    qa.K = s.K;
    qa.L = s.L;
    qa.qrow_ctas = (qa.BHq + kQRows - 1) / kQRows;
    const dim3 qgrid(s.qwords > 0 ? s.qwords : 1, qa.qrow_ctas + 1);
    qencode_kernel<<<qgrid, kThreads, 0, st>>>(qa);
    return cudaGetLastError();
}

cudaError_t launch_collide(const void* q, bool q_bf16, const uint32_t* codes,
                           const float* centre, const void* keys, const void* values,
                           bool kv_bf16, const DecodeShape& s, float* out,
                           const DecodeScratch& ws, cudaStream_t st, int blk0) {
    const int G = s.Hq / s.Hkv;
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
    aa.table_only = s.logu_ext != nullptr;     // no closed form for p: the table everywhere
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
    aa.radius = s.radius;
    aa.scale = s.scale;
    aa.log_c2 = s.L >= 2 ? logf(0.5f * static_cast<float>(s.L) * static_cast<float>(s.L - 1)) : 0.0f;
    {
        const AttendSmem m = attend_smem(attend_partials(s.nblk), kv_bf16 ? 2 : 4);
        aa.merge_cap = m.merge_cap;
        aa.work_bytes = static_cast<int>(m.work);
    }
    return launch_dependent(attend, dim3(aa.nsb + 1, s.B * s.Hq), dim3(kAThreads), smem_att, st,
                            aa);
}

}  // namespace mp
