// Internal declarations shared by the translation units of libmagicpig.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "magicpig.h"

namespace mp {

constexpr int kKeysPerBlock = MP_KEYS_PER_BLOCK;   // keys per bit-sliced code block
constexpr int kWordsPerBlock = kKeysPerBlock / 32;  // uint32 words per plane row
constexpr int kD = 128;                             // the only head dimension supported
constexpr int kAttendBlockGroup = 4;                // 1024-key blocks per attend CTA
constexpr int kLogUTableIntervals = 4096;           // log u tables over the cosine: intervals
constexpr int kMaxBucketBits = 12;                  // bucketed tables: at most 2^12 buckets a table
constexpr int kBucketRanges = 8;                    // key ranges a table's bucket build is split into
constexpr int kAppendMaxKeys = 64;                  // mp_encode_keys ranges up to this run on CUDA cores

// Partial softmax states per query row: one per group of kAttendBlockGroup blocks (sampled
// keys) plus one for the exact sink/local set.
inline int attend_partials(int nblk) { return (nblk + kAttendBlockGroup - 1) / kAttendBlockGroup + 1; }

// Device status word values (mp_status codes): kernels raise MP_ERR_TIMEOUT (a bounded wait gave
// up) and, in the MP_CHECKS build, MP_ERR_BOUNDS. The word after it keeps the site of the first
// failed index check.
int* device_status_ptr();          // address of this device's status word (nullptr on error)

#ifndef MP_CHECKS
#define MP_CHECKS 0
#endif
// Sites of the index checks (the number mp_debug_check_report returns).
enum CheckSite : int {
    kSiteQencodeStore = 1,       // query bits / masks / norms written by the query encoding
    kSiteScanCodes = 2,          // the code block a scan CTA streams
    kSiteScanSelect = 3,         // the selection words a scan CTA writes
    kSiteAttendRow = 4,          // a K/V row the attend kernel copies (key < n)
    kSiteAttendPartial = 5,      // a partial softmax state or an output row it writes
    kSiteAttendSelect = 6,       // the selection words it reads
    kSiteBucketRange = 7,        // a bucket's [offset, next offset) outside the table's n keys
    kSiteBucketKey = 8,          // a bucket member outside [0, n)
    kSiteEncodeCodes = 9,        // the code words an encoder CTA writes
};

// Index check of the MP_CHECKS build (the memory checker's stand-in): there an index outside
// [0, limit) raises MP_ERR_BOUNDS in the status word, keeps `site` beside it if it is the first,
// and returns false so that the caller skips the access; nothing traps. In the product build it
// is true and compiles away.
__device__ __forceinline__ bool mp_check(int* status, long long idx, long long limit, int site) {
#if MP_CHECKS
    if (idx >= 0 && idx < limit) return true;
    if (status && atomicCAS(status, 0, static_cast<int>(MP_ERR_BOUNDS)) == 0)
        atomicExch(status + 1, site);
    return false;
#else
    (void)status;
    (void)idx;
    (void)limit;
    (void)site;
    return true;
#endif
}
int device_sm_count();

// Scratch carved out of the decode workspace (all pointers 256-byte aligned).
struct DecodeScratch {
    uint32_t* qbits;     // [B*Hq][qwords] query sign bits
    uint32_t* qmask;     // [B*Hkv][cpad][G] per-plane XOR masks (0 where the query bit is 1)
    float4* qstat;       // [B*Hq] {|q|, q.mu, 0, 0}
    float* pm;           // [B*Hq][nsp] max logit of each attend CTA's partial softmax
    float* pl;           // [B*Hq][nsp] its sum of weights
    float* po;           // [B*Hq][nsp][128] its weighted value sum
    unsigned* counters;  // [B*Hq] attend CTAs finished, for the last one's merge
    int n_counters;      // counters the query encoding resets
    uint32_t* selmask;   // [B*Hq][nblk][32] selection words, written by the scan kernel
    uint32_t* sel_ge1;   // [B*Hq][nblk][32] keys hit by >= 1 table (bucketed lookup only)
    float* logu_tab;     // [kLogUTableIntervals + 1] log_inclusion_segment's table, filled per call
};

struct DecodeShape {
    int B, Hq, Hkv, n, d, K, L, C, qwords, nblk, n_sink, n_local;
    int cpad;            // C rounded up to a multiple of 4 (16-byte rows of query masks)
    int ncap;            // K/V rows per (sequence, KV head) in memory (>= n)
    int cblk;            // code blocks per (sequence, KV head) in memory: ceil(ncap / 1024)
    int n_indexed;       // keys in the bucketed tables (<= n)
    float scale;
    const float* radius; // MIPS variant: [B*Hkv] longest centred key; nullptr otherwise
    bool cp;             // cross-polytope variant: byte codes, qwords = ceil(L / 4) words of codes
    const float* logu_ext;   // cross-polytope: the caller's log u table (nullptr otherwise)
};

size_t decode_scratch_bytes(const DecodeShape& s, bool debug);
// Shapes, parameters, dtypes, pointers and alignment of a decode call, everything but the
// workspace (the checks of mp_decode_attention); fills *s on success.
mp_status validate_decode(const void* q, mp_dtype q_dtype, const uint32_t* codes,
                          const float* centre, const void* W, mp_dtype w_dtype, const void* keys,
                          const void* values, mp_dtype kv_dtype, int B, int Hq, int Hkv, int n,
                          int d, const mp_params* prm, const float* out, DecodeShape* s);
DecodeScratch carve_decode_scratch(void* ws, const DecodeShape& s, bool debug);

// ---- launchers (each returns the launch error, cudaSuccess otherwise) -------------------------
cudaError_t launch_key_mean(const void* keys, bool bf16, int BH, int ncap, int n, float* centre,
                            float* partial, int nsplit, cudaStream_t st);
int key_mean_splits(int BH, int n);

// Encode whole 1024-key blocks [blk0, blk1) of every head of a cache laid out for ncap keys
// per head (keys >= ncap read as zero).
// With norms (|k_i - mu| per key, [B*Hkv][ncap]) and radius ([B*Hkv]): the MIPS variant, W with
// d + 1 rows. With argmax: the cross-polytope codes (bytes), W = G [L][d][d], K = d (a table is
// d hyperplanes).
cudaError_t launch_encode_tc(const void* keys, const float* centre, const void* W, int B,
                             int Hkv, int ncap, int blk0, int blk1, int K, int L,
                             uint32_t* codes, int* status, cudaStream_t st,
                             const float* norms = nullptr, const float* radius = nullptr,
                             bool argmax = false);
cudaError_t launch_encode_simt(const void* keys, bool keys_bf16, const float* centre,
                               const void* W, bool w_bf16, int B, int Hkv, int ncap, int blk0,
                               int blk1, int K, int L, uint32_t* codes, cudaStream_t st);
// Encode keys [n0, n1) (a short range) into their words, keeping the other keys' bits.
cudaError_t launch_encode_append(const void* keys, bool keys_bf16, const float* centre,
                                 const void* W, bool w_bf16, int B, int Hkv, int ncap, int n0,
                                 int n1, int K, int L, uint32_t* codes, cudaStream_t st);

// query sign bits, |q| and q.mu into the scratch; also resets the merge counters
cudaError_t launch_qencode(const void* q, bool q_bf16, const float* centre, const void* W,
                           bool w_bf16, const DecodeShape& s, const DecodeScratch& ws,
                           cudaStream_t st);
// The code scan over blocks [blk0, nblk) (selection words of those blocks; every block when
// blk0 == 0), then the attend kernel over every block. cudaErrorNotSupported if it cannot fit a
// CTA
cudaError_t launch_collide(const void* q, bool q_bf16, const uint32_t* codes,
                           const float* centre, const void* keys, const void* values,
                           bool kv_bf16, const DecodeShape& s, float* out,
                           const DecodeScratch& ws, cudaStream_t st, int blk0 = 0);
bool decode_supported(const DecodeShape& s, bool kv_bf16);
// the attend kernel alone, on selection words already in ws.selmask (masked with valid & not T)
cudaError_t launch_attend(const void* q, bool q_bf16, const float* centre, const void* keys,
                          const void* values, bool kv_bf16, const DecodeShape& s, float* out,
                          const DecodeScratch& ws, cudaStream_t st);

// ---- bucketed hash tables (mp_buckets.cu) ------------------------------------------------------
size_t bucket_table_bytes(int B, int Hkv, int n, int K, int L);   // 0 if unsupported
// tables of keys [0, n) of codes laid out for cblk blocks per head
cudaError_t launch_bucket_build(const uint32_t* codes, int B, int Hkv, int cblk, int n, int K,
                                int L, uint32_t* buckets, cudaStream_t st);
// ge1 / ge2 bitmaps of the query rows' bucket hits (tables of s.n_indexed keys), in the
// selection-word layout
cudaError_t launch_bucket_lookup(const uint32_t* buckets, const uint32_t* qbits,
                                 const DecodeShape& s, uint32_t* ge1, uint32_t* ge2,
                                 cudaStream_t st);
cudaError_t prepare_buckets();

// ascending indices of the selection words' keys, masked with the valid keys and not T
cudaError_t launch_compact_selection(const uint32_t* selmask, int rows, int n, int nblk,
                                     int n_sink, int n_local, int32_t* sel_idx,
                                     int32_t* sel_count, cudaStream_t st);
// log u at count cosines, as the decode kernels evaluate it (log_inclusion_cos)
cudaError_t launch_log_inclusion(const float* cosines, int count, int K, int L, float* out,
                                 cudaStream_t st);
// one bounded wait on an mbarrier that nothing completes (the failure path's test hook)
cudaError_t launch_wait_expiry(unsigned long long limit_ns, int* status, cudaStream_t st);
cudaError_t launch_collision_counts(const uint32_t* codes, const uint32_t* qbits,
                                    const DecodeShape& s, uint8_t* cnt, cudaStream_t st);
cudaError_t launch_codes_unpack(const uint32_t* codes, int BH, int n, int K, int L,
                                uint32_t* out, cudaStream_t st);

// Force-load every kernel of the library (so that nothing loads lazily inside a stream capture)
// and raise the dynamic shared-memory limits once per device.
cudaError_t prepare_encode_tc();
cudaError_t prepare_decode();
cudaError_t prepare_misc();
cudaError_t prepare_append();
cudaError_t prepare_mips();
cudaError_t prepare_cross_polytope();

// ---- cross-polytope variant (mp_cross_polytope.cu) ----------------------------------------------
size_t cp_codes_bytes(int B, int Hkv, int n, int L);
// log u over kLogUTableIntervals + 1 cosines on [-1, 1] for the cross-polytope p (one hash a table)
cudaError_t launch_cp_logu_table(int K, int L, float* table, cudaStream_t st);
// codes of keys [n0, n1): bytes [B*Hkv][ceil(ncap/1024)][L][1024]; G [L][d][d]
cudaError_t launch_encode_cp(const void* keys, bool keys_bf16, const float* centre, const void* G,
                             bool g_bf16, int B, int Hkv, int ncap, int n0, int n1, int L,
                             uint8_t* codes, cudaStream_t st);
// query codes (bytes in ws.qbits), |q|, q.mu, and the merge counters
cudaError_t launch_qencode_cp(const void* q, bool q_bf16, const float* centre, const void* G,
                              bool g_bf16, const DecodeShape& s, const DecodeScratch& ws,
                              cudaStream_t st);
// the byte-code scan over blocks [blk0, nblk), then the attend kernel over every block
cudaError_t launch_collide_cp(const void* q, bool q_bf16, const uint8_t* codes,
                              const float* centre, const void* keys, const void* values,
                              bool kv_bf16, const DecodeShape& s, float* out,
                              const DecodeScratch& ws, cudaStream_t st, int blk0 = 0);

// ---- MIPS -> cosine variant (mp_mips.cu) -------------------------------------------------------
// radius[bh] = max over keys [0, n) of |k - mu| (radius may be null), and with norms
// ([BH][ncap]) |k_i - mu| of keys [k0, k1) as well (k0 = 0, k1 = n when only the radius is asked)
cudaError_t launch_key_radius(const void* keys, bool keys_bf16, const float* centre, int BH,
                              int ncap, int n, float* radius, cudaStream_t st,
                              float* norms = nullptr, int k0 = 0, int k1 = -1);
// codes of keys [n0, n1) from the keys extended by sqrt(r^2 - |k - mu|^2), W with d + 1 rows
cudaError_t launch_encode_mips(const void* keys, bool keys_bf16, const float* centre,
                               const void* W, bool w_bf16, const float* radius, int B, int Hkv,
                               int ncap, int n0, int n1, int K, int L, uint32_t* codes,
                               cudaStream_t st);

// Launch `kern` as a programmatic dependent of the previous kernel in the stream.
template <typename Arg>
cudaError_t launch_dependent(void (*kern)(Arg), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, const Arg& arg) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, arg);
}

// ---- small device helpers ---------------------------------------------------------------------
__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ float load_elem(const void* p, bool bf16, size_t i) {
    return bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i])
                : reinterpret_cast<const float*>(p)[i];
}

// 32x32 bit-matrix transpose across a warp: on entry bit b of lane r is element (r, b); on exit
// bit r of lane b is that element. Each stage swaps the off-diagonal s x s blocks.
// Lanes without bit s of their index keep the positions b with (b & s) == 0 and take the
// partner's such bits moved up by s; lanes with bit s keep the others and take the partner's
// moved down by s. For s = 16 and 8 the blocks are whole bytes and one byte permute of the lane's
// and the partner's word does both; for s = 4, 2, 1 a rotation does both moves (the bits it
// wraps around are masked off) and a three-input logic op merges. Every stage has one shuffle.
__device__ __forceinline__ uint32_t warp_transpose32(uint32_t x, int lane) {
    {
        const uint32_t y = __shfl_xor_sync(0xffffffffu, x, 16);
        x = __byte_perm(x, y, (lane & 16) ? 0x3276 : 0x5410);   // [y2 y3 x2 x3] / [x0 x1 y0 y1]
    }
    {
        const uint32_t y = __shfl_xor_sync(0xffffffffu, x, 8);
        x = __byte_perm(x, y, (lane & 8) ? 0x3715 : 0x6240);    // [y1 x1 y3 x3] / [x0 y0 x2 y2]
    }
    const uint32_t low[3] = {0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const int s = 4 >> i;
        const bool up = (lane & s) != 0;
        const uint32_t keep = up ? ~low[i] : low[i];
        const uint32_t y = __shfl_xor_sync(0xffffffffu, x, s);
        const uint32_t r = __funnelshift_l(y, y, up ? 32 - s : s);   // rotate left
        x = (x & keep) | (r & ~keep);
    }
    return x;
}

// Programmatic dependent launch: the next kernel in the stream may be scheduled once every CTA
// of this one has started; a kernel launched that way waits for its predecessor's completion
// (and memory) before it touches anything the predecessor writes.
__device__ __forceinline__ void allow_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_for_predecessor() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// log u(p) = log P[Binomial(L, p^K) >= 2] in fp32: the inclusion probability u = 1 - (1-p^K)^L -
// L p^K (1-p^K)^(L-1) of the hash-function-choice section of "LSH Sampling...", in the log domain
// ("don't pick the tallest", section 5, asks for stable probability arithmetic). With x = p^K and
// lambda = L x: for lambda >= 0.05 directly, u = -expm1(L log1p(-x)) - lambda e^{(L-1) log1p(-x)}
// (the two terms cancel to lambda^2 / 2 at worst, a factor 40 at lambda = 0.05, so u keeps about
// 20 correct bits); below, log t_2 + log1p(sum_{j>=3} t_j / t_2) with t_j the binomial terms, whose
// ratios t_{j+1} / t_j = (L - j) / (j + 1) * x / (1 - x) are then below 0.02: seven terms leave a
// remainder under 1e-13. p <= 0 (a key that cannot collide) clamps to log(FLT_MIN); L < 2 gives
// -inf (no key can collide in two tables); K = 0 gives 0 (every key collides in every table).
__device__ inline float log_inclusion_p(float p, int K, int L) {
    if (L < 2) return -INFINITY;
    if (K == 0) return 0.0f;
    if (!(p > 0.0f)) return -87.336544750553102f;   // log(FLT_MIN)
    const float lx = static_cast<float>(K) * logf(p);
    const float x = expf(lx);
    const float Lf = static_cast<float>(L);
    if (x >= 1.0f) return 0.0f;
    const float l1 = log1pf(-x);
    const float lam = Lf * x;
    if (lam >= 0.05f) {
        const float u = -expm1f(Lf * l1) - lam * expf((Lf - 1.0f) * l1);
        return logf(fmaxf(u, 1.17549435e-38f));
    }
    const float r = x / (1.0f - x);
    float term = 1.0f, sum = 0.0f;
#pragma unroll
    for (int j = 2; j < 9; ++j) {
        if (j >= L) break;
        term *= (Lf - static_cast<float>(j)) * (1.0f / static_cast<float>(j + 1)) * r;
        sum += term;
    }
    return logf(0.5f * Lf * (Lf - 1.0f)) + 2.0f * lx + (Lf - 2.0f) * l1 + log1pf(sum);
}

// log u at the cosine c of q and k - mu. SimHash's bit agreement is p = 1 - arccos(c) / pi
// ("LSH Sampling...", background, LSH basics), evaluated as arccos(-c) / pi: the same number,
// without the cancellation of 1 - (1 - small) as c approaches -1.
__device__ inline float log_inclusion_cos(float c, int K, int L) {
    return log_inclusion_p(acosf(-c) * 0.318309886183790672f, K, L);
}

// The attend kernel's log u for SimHash keys: linear interpolation in a per-call table of the
// closed form at the cosines -1 + 2 i / N (N = kLogUTableIntervals), on every interval where the
// chord stays within kLogUTableTol of the closed form; the closed form itself elsewhere.
// Linear interpolation errs most near an interval's midpoint, by about h^2 |f''| / 8, so the gap
// there measures it. Where log u bends sharply (the cosine near +-1, or many bits and few
// tables) the gap is larger and those intervals keep the closed form.
constexpr float kLogUTableTol = 2e-5f;

__device__ __forceinline__ float log_inclusion_grid(float i, int K, int L) {
    return log_inclusion_cos(fminf(1.0f, -1.0f + 2.0f * i / kLogUTableIntervals), K, L);
}

__device__ __forceinline__ bool log_inclusion_chord_ok(float fa, float fb, float fm) {
    return fabsf(fm - 0.5f * (fa + fb)) <= kLogUTableTol;   // false for NaN or inf - inf
}

// Entries [seg * kLogUSegment, (seg + 1) * kLogUSegment) (those <= N) of the table: entry i is
// log u at the cosine -1 + 2 i / N, or NaN when an interval it bounds is not interpolated (every
// cosine of such an interval then takes the closed form). The closed form is evaluated once per
// grid point and interval midpoint of the segment (and its two neighbours) into buf, shared
// memory of at least 2 * kLogUSegment + 3 floats. Called by every thread of the block.
constexpr int kLogUSegment = 128;
__device__ inline void log_inclusion_segment(int seg, int K, int L, float* buf, float* tab) {
    const int i0 = seg * kLogUSegment;
    float* fg = buf;                             // grid points i0 - 1 .. i0 + kLogUSegment
    float* fm = buf + kLogUSegment + 2;          // midpoints of intervals i0 - 1 .. i0 + kLogUSegment - 1
    for (int k = threadIdx.x; k < 2 * kLogUSegment + 3; k += blockDim.x) {
        if (k < kLogUSegment + 2) {
            const int i = i0 - 1 + k;
            fg[k] = i >= 0 && i <= kLogUTableIntervals
                        ? log_inclusion_grid(static_cast<float>(i), K, L) : 0.0f;
        } else {
            const int j = i0 - 1 + (k - (kLogUSegment + 2));
            fm[k - (kLogUSegment + 2)] = j >= 0 && j < kLogUTableIntervals
                        ? log_inclusion_grid(static_cast<float>(j) + 0.5f, K, L) : 0.0f;
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < kLogUSegment; t += blockDim.x) {
        const int i = i0 + t;
        if (i > kLogUTableIntervals) break;
        float e = fg[t + 1];
        if (i >= 1 && !log_inclusion_chord_ok(fg[t], fg[t + 1], fm[t])) e = __int_as_float(0x7fc00000);
        if (i < kLogUTableIntervals && !log_inclusion_chord_ok(fg[t + 1], fg[t + 2], fm[t + 1]))
            e = __int_as_float(0x7fc00000);
        tab[i] = e;
    }
    __syncthreads();                             // buf is refilled by the next segment
}
constexpr int kLogUSegments = kLogUTableIntervals / kLogUSegment + 1;

// tab: the table above, in global or shared memory (plain loads).
__device__ __forceinline__ float log_inclusion_at(float c, const float* tab, int K, int L) {
    if (c > -1.0f && c < 1.0f) {
        const float tt = (c + 1.0f) * (0.5f * kLogUTableIntervals);
        const int i = min(static_cast<int>(tt), kLogUTableIntervals - 1);
        const float g0 = tab[i], g1 = tab[i + 1];
        const float lw = fmaf(tt - static_cast<float>(i), g1 - g0, g0);
        if (lw == lw) return lw;                 // NaN: an interval kept for the closed form
    }
    return log_inclusion_cos(c, K, L);
}

// ---- mbarriers and the bounded wait every spin in this library goes through -----------------
constexpr unsigned long long kWaitLimitNs = 4000000000ull;   // 4 s: far beyond any real wait

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait: false on timeout (status raised, abort flag set) or when another role aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0u) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicExch(status, (int)MP_ERR_TIMEOUT);
                return false;
            }
        }
    }
}
// bits of a 32-key word whose offset within the word is below x (x may be out of [0, 32])
__device__ __forceinline__ uint32_t bits_below(int x) {
    return x <= 0 ? 0u : (x >= 32 ? 0xffffffffu : ((1u << x) - 1u));
}

}  // namespace mp
