// Key encoding on the tcgen05 tensor cores: codes = [W^T (k - mu) > 0], bit-sliced.
//
// The SimHash projection of every cached key on K*L hyperplanes ("MagicPIG: LSH Sampling for
// Efficient LLM Generation", background, LSH basics: Sign(w^T x); method details, hash-function
// choice; system co-design item 2: the random projection is a dense GEMM kept on the GPU) is
// the one dense contraction of the path: [keys x 128] x [128 x K*L].
//
// With bf16 keys and a bf16 W every product is exact in fp32, so the MMA computes w_j . k_i
// with fp32 accumulation; the centre enters as the per-(head, plane) constant c_j = w_j . mu
// and the sign test is [w_j . k_i > c_j], i.e. [w_j . (k_i - mu) > 0]. The constant is folded
// into the contraction as one more K=16 step: its A slice is [1, 1, 1, 0, ...] in every row and
// its B slice holds c_j split exactly into three bf16 terms (c = hi + mid + lo to 2^-24 of c), so
// that step sets the accumulator to c_j and the eight K=16 steps over the key dimensions add
// k_i . (-w_j). The result is c_j - w_j . k_i and its sign bit is the code bit.
//
// Structure (one CTA per SM, persistent over a contiguous range of 1024-key blocks, and one
// 256-hyperplane chunk of W held in shared memory for the CTA's whole life):
//   warp 0   TMA producer: 128-key x 128-dim bf16 tiles, 128-byte swizzle, 3-stage ring (2 for
//            the MIPS variant, whose producer warp also writes each tile's key slice)
//   warp 1   TMEM allocator and single-thread MMA issuer: M=128, N<=256, K=16 x (1 + 8) per
//            tile, double-buffered fp32 accumulators (2 x 256 TMEM columns)
//   warps 2-17 epilogue: tcgen05.ld the accumulator; per key (lane) gather its sign bits into
//            a 32-bit word for 32 hyperplanes (funnel shifts and FP32 sums), transpose the
//            32x32 bit block across the warp with 5 shuffle stages so that each lane holds one
//            hyperplane's 32-key word, stage a block's words in shared memory, then write each
//            plane row (128 bytes) of the block with coalesced stores. When the head changes
//            they also write the new c_j slice (three head slots, so that a slot is rewritten
//            only after the MMAs of the head that used it have completed).
// Every mbarrier wait is bounded; on expiry the CTA records MP_ERR_TIMEOUT in the device status
// word, stops issuing work, and still releases its TMEM before returning.
#include <cuda.h>

#include "mp_internal.cuh"

namespace mp {
namespace {

constexpr int kTileM = 128;            // keys per MMA tile (TMEM lanes)
constexpr int kChunkN = 256;           // hyperplanes per CTA (MMA N, TMEM columns per buffer)
// 16 epilogue warps + 2 = 18 warps: some SM sub-partition holds 5 of them, and its 16K
// registers cap the kernel at 96 registers per thread (ptxas picks that from the launch bound).
constexpr int kEpiWarps = 16;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kStageBytes = kTileM * kD * 2;      // 32 KB: two 64-column swizzled halves
constexpr uint32_t kHalfBytes = kTileM * 128;          // 16 KB: 128 rows x 128 bytes
constexpr uint32_t kBBytes = kChunkN * kD * 2;         // 64 KB
constexpr uint32_t kBHalfBytes = kChunkN * 128;        // 32 KB
constexpr int kStgPitch = kWordsPerBlock * 8 + 1;      // 257: staging row pitch (words)

// Centre region: 256 rows x 128 bytes, 128-byte swizzle, four K=16 slices per row: slices 0-2
// hold the c_j terms of three heads (B operand, rows = hyperplanes), slice 3 of rows 0-127 the
// constant [1, 1, 1, 0, ...] (A operand, rows = keys).
constexpr uint32_t kCBytes = kChunkN * 128;            // 32 KB
constexpr int kCSlots = 3;
constexpr int kOnesSlice = 3;
static_assert(kStgPitch == 257, "staging pitch");

constexpr int kSign = 0, kMips = 1, kArgmax = 2;         // epilogue modes of the encoder

// Shared memory of an encoder CTA: the A-tile ring, the -W chunk (B), the centre region, for
// the MIPS variant its key slices, the word staging, barriers and the MIPS row of W. The MIPS
// variant's key slices ([1, 1, 1, a_hi, a_mid, a_lo, 0, ...] per key: the extra coordinate a_i
// enters the contraction beside the centre) take one K=16 slice per ring stage of a 128-row,
// 128-byte-swizzled region; they fit beside a 2-stage ring.
template <int kMode>
struct EncLayout {
    static constexpr int kStages = kMode == kMips ? 2 : 3;            // A-tile ring depth
    static constexpr uint32_t kOffA = 0;
    static constexpr uint32_t kOffB = kOffA + kStages * kStageBytes;
    static constexpr uint32_t kOffC = kOffB + kBBytes;
    static constexpr uint32_t kOffKs = kOffC + kCBytes;               // MIPS key slices
    static constexpr uint32_t kKsBytes = kMode == kMips ? kTileM * 128 : 0;
    static constexpr uint32_t kOffStg = kOffKs + kKsBytes;
    static constexpr uint32_t kOffBars = kOffStg + kWordsPerBlock * kStgPitch * 4;
    static constexpr uint32_t kOffMisc = kOffBars + 128;
    static constexpr uint32_t kOffWd = kOffMisc + 16;               // MIPS: W[d][j0 + r]
    static constexpr uint32_t kSmemBytes = kOffWd + kChunkN * 4 + 1024;   // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kOffC % 1024 == 0 && kOffKs % 1024 == 0,
                  "swizzled operands start on 1024-byte boundaries");
    static_assert(kMode != kMips || kStages <= 4, "a key slice per ring stage");
};
constexpr uint32_t kXchOff = 2 * kKeysPerBlock;          // argmax: exchange area after the codes
static_assert(kXchOff + 2 * 2 * 2 * kTileM * 8 <= kWordsPerBlock * kStgPitch * 4,
              "the argmax staging fits the word staging area");

struct EncodeArgs {
    const float* centre;            // [BH][128]
    const __nv_bfloat16* W;         // [128][C]
    uint32_t* codes;
    int* status;
    int C, nchunk, nblk, n, units, parts;
    int blk0;                       // first block encoded; a unit's block is blk0 + u % nblk
    int cblk;                       // code blocks per head in memory (the codes' head stride)
    // MIPS variant only: |k_i - mu| per key [BH][n] and r per head [BH]
    const float* norms;
    const float* radius;
};

// ---- PTX wrappers -----------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address >> 4
    d |= static_cast<uint64_t>(1) << 16;                    // leading offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;            // stride offset: 8 rows x 128 B
    d |= static_cast<uint64_t>(1) << 46;                    // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                    // 128-byte swizzle
    return d;
}
// Instruction descriptor, kind::f16: D f32, A and B bf16, both K-major, M x N.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
          "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
          "=r"(v[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void epi_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
}
// the four epilogue warps of one 64-column group (named barriers 2 .. 5)
__device__ __forceinline__ void group_sync(int cg) {
    asm volatile("bar.sync %0, 128;" ::"r"(2 + cg) : "memory");
}
// 1.0 if the fp32 accumulator (as bits) is negative, else 0.0: -2^126 x, saturated to [0, 1]
// (denormals flush to zero), on the FP32 pipe
__device__ __forceinline__ float neg_as_one(uint32_t v) {
    float r;
    asm("mul.rn.ftz.sat.f32 %0, %1, 0fFE800000;" : "=f"(r) : "f"(__uint_as_float(v)));
    return r;
}
// Bit c of the result = [accumulator column c < 0] (c_c - w_c . k, so the bit is
// [w_c . k > c_c]) for c in 0..31, one byte per chain of 8 columns. Funnel shifts move the sign
// bits in; they run on the integer pipe at half rate. kFpBytes of the bytes (from byte 0) are
// summed on the FP32 pipe instead, as 2^23 + sum_c 2^c [acc_c < 0], whose low mantissa bits are
// the byte (exact: small integers). For the SimHash epilogue, which has no other
// FP32 work, one FP byte of four balanced the two pipes best (0, 1, 2 and 3 measured); the MIPS
// variant's extra coordinate enters the contraction, so its epilogue is the same. The two forms
// differ only for an accumulator of -0 or a negative denormal, i.e. an exact or sub-2^-126 tie,
// where either bit lies within the near-tie band.
template <int kFpBytes>
__device__ __forceinline__ uint32_t pack_signs(const uint32_t (&v)[32]) {
    uint32_t x[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (k < kFpBytes) {
            // pairs, quads, then the byte (a tree: four dependent steps instead of eight)
            float p[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                p[c] = fmaf(neg_as_one(v[8 * k + 2 * c + 1]), 2.0f, neg_as_one(v[8 * k + 2 * c]));
            const float q0 = fmaf(p[1], 4.0f, p[0]), q1 = fmaf(p[3], 4.0f, p[2]);
            x[k] = __float_as_uint(fmaf(q1, 16.0f, q0) + 8388608.0f);   // + 2^23
        } else {
            x[k] = 0u;
#pragma unroll
            for (int c = 7; c >= 0; --c) x[k] = __funnelshift_l(v[8 * k + c], x[k], 1);
        }
    }
    return __byte_perm(__byte_perm(x[0], x[1], 0x0040), __byte_perm(x[2], x[3], 0x0040), 0x5410);
}
// kMode: kSign, the SimHash codes; kMips, the MIPS -> cosine variant, whose keys carry an extra
// coordinate a_i = sqrt(max(0, r^2 - |k_i - mu|^2)) on a (d + 1)-th row of W: the producer warp
// writes each tile's key slice [1, 1, 1, a_hi, a_mid, a_lo, 0, ...] (a_i split exactly into three
// bf16 terms, from the norms it loads two tiles ahead) and the centre's B slice carries
// [c_hi, c_mid, c_lo, -W[d][j] x 3], so the first K=16 step puts c_j - W[d][j] a_i into the
// accumulator and the epilogue is the SimHash one;
// kArgmax, the cross-polytope codes: W is G [L][d][d] (hyperplane j = row j % d of G_{j / d}), a
// chunk holds two tables, and the epilogue keeps, per key and table, the first index of the
// largest |accumulator| (two warps cover a table's 128 columns and meet in shared memory), then
// writes one code byte per (table, key).
template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    encode_tc_kernel(const __grid_constant__ CUtensorMap kmap, const EncodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    using Lay = EncLayout<kMode>;
    constexpr int kStages = Lay::kStages;
    uint8_t* sA = smem + Lay::kOffA;
    uint8_t* sB = smem + Lay::kOffB;
    uint32_t* stg = reinterpret_cast<uint32_t*>(smem + Lay::kOffStg);
    uint8_t* sC = smem + Lay::kOffC;
    uint8_t* sK = smem + Lay::kOffKs;            // MIPS: the key slices
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kOffBars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kOffMisc + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chunk = blockIdx.x % a.nchunk;
    const int part = blockIdx.x / a.nchunk;
    const int j0 = chunk * kChunkN;
    const int Nc = min(kChunkN, a.C - j0);          // real hyperplanes in this chunk
    const int Nmma = (Nc + 15) & ~15;               // MMA N (multiple of 16)
    const int u_begin = static_cast<int>((static_cast<long long>(a.units) * part) / a.parts);
    const int u_end = static_cast<int>((static_cast<long long>(a.units) * (part + 1)) / a.parts);

    const uint32_t bar_full = smem_u32(bars);            // [kStages]
    const uint32_t bar_empty = bar_full + 8 * kStages;   // [kStages]
    const uint32_t bar_tfull = bar_empty + 8 * kStages;  // [2]
    const uint32_t bar_tempty = bar_tfull + 16;          // [2]

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            // MIPS: the stage is full once its TMA bytes and its key slice are in place
            mbar_init(bar_full + 8 * s, kMode == kMips ? 2 : 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar_tfull + 8 * s, 1);
            mbar_init(bar_tempty + 8 * s, kEpiWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // -W chunk -> shared memory as the B operand: row r = hyperplane j0 + r, K-major, swizzled
    // (negating a bf16 is exact). Batches of 16 loads per thread are in flight at once.
    {
        constexpr int kElems = kChunkN * kD, kBatch = 16;
        for (int base = 0; base < kElems; base += kThreads * kBatch) {
            __nv_bfloat16 w[kBatch];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int idx = base + k * kThreads + tid;
                const int r = idx % kChunkN, e = idx / kChunkN;
                w[k] = __float2bfloat16(0.0f);
                if (idx < kElems && r < Nc)
                    w[k] = __hneg(kMode == kArgmax ? a.W[static_cast<size_t>(j0 + r) * kD + e]
                                                   : a.W[static_cast<size_t>(e) * a.C + j0 + r]);
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int idx = base + k * kThreads + tid;
                const int r = idx % kChunkN, e = idx / kChunkN;
                const uint32_t off = (e >> 6) * kBHalfBytes + r * 128 +
                                     ((((e & 63) >> 3) ^ (r & 7)) << 4) + ((e & 7) << 1);
                if (idx < kElems) *reinterpret_cast<__nv_bfloat16*>(sB + off) = w[k];
            }
        }
    }
    // centre region: zero, then [1, 1, 1, 0, 0, 0, 0, 0] in the first 16 bytes of slice 3, rows
    // 0-127 (the rest of the slice stays 0)
    for (int i = tid; i < static_cast<int>(kCBytes / 16); i += kThreads)
        reinterpret_cast<uint4*>(sC)[i] = make_uint4(0u, 0u, 0u, 0u);
    if constexpr (kMode == kMips) {
        for (int i = tid; i < static_cast<int>(Lay::kKsBytes / 16); i += kThreads)
            reinterpret_cast<uint4*>(sK)[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    if (tid < kTileM) {
        const uint32_t one2 = 0x3F803F80u;   // two bf16 1.0
        *reinterpret_cast<uint4*>(sC + tid * 128 + (((2 * kOnesSlice) ^ (tid & 7)) << 4)) =
            make_uint4(one2, 0x00003F80u, 0u, 0u);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(2 * kChunkN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        // (MIPS: the whole warp; besides the loads it writes each tile's key slice, from the
        // keys' norms and the head's radius, which it loads two tiles ahead)
        if (kMode == kMips || lane == 0) {
            int it = 0;
            bool ok = true;
            // MIPS prefetch: norms of this lane's keys (rows lane + 32 i) and the radius, for the
            // next tile (nk1, r1) and the one after (nk2, r2); `ahead` is the tile after those
            float nk1[4] = {0.0f, 0.0f, 0.0f, 0.0f}, nk2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            float r1 = 0.0f, r2 = 0.0f;
            int ahead_u = u_begin, ahead_t = 0;
            auto load_ahead = [&](float (&nk)[4], float& r) {
                if (ahead_u >= u_end) return;
                const int bg_ = ahead_u / a.nblk, blk_ = ahead_u % a.nblk;
                const int key0 = (a.blk0 + blk_) * kKeysPerBlock + ahead_t * kTileM;
                r = __ldg(a.radius + bg_);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int key = key0 + lane + 32 * i;
                    nk[i] = key < a.n ? __ldg(a.norms + static_cast<size_t>(bg_) * a.n + key) : r;
                }
                const int rows_ = min(kKeysPerBlock, a.n - (a.blk0 + blk_) * kKeysPerBlock);
                if (++ahead_t == (rows_ + kTileM - 1) / kTileM) {
                    ahead_t = 0;
                    ++ahead_u;
                }
            };
            if constexpr (kMode == kMips) {
                load_ahead(nk1, r1);
                load_ahead(nk2, r2);
            }
            for (int u = u_begin; u < u_end && ok; ++u) {
                const int bg = u / a.nblk, blk = u % a.nblk;
                const int rows = min(kKeysPerBlock, a.n - (a.blk0 + blk) * kKeysPerBlock);
                const int ntile = (rows + kTileM - 1) / kTileM;
                for (int t = 0; t < ntile; ++t, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    bool got = mbar_wait(bar_empty + 8 * s, ph ^ 1, abort_flag, a.status);
                    if constexpr (kMode == kMips) got = __all_sync(0xffffffffu, got);
                    if (!got) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        mbar_arrive_expect_tx(bar_full + 8 * s, kStageBytes);
                        const uint32_t dst = smem_u32(sA + s * kStageBytes);
                        const int row0 = (a.blk0 + blk) * kKeysPerBlock + t * kTileM;
                        tma_load_3d(dst, &kmap, bar_full + 8 * s, 0, row0, bg);
                        tma_load_3d(dst + kHalfBytes, &kmap, bar_full + 8 * s, 64, row0, bg);
                    }
                    if constexpr (kMode == kMips) {
                        // key row `row` of slice s: [1, 1, 1, a_hi, a_mid, a_lo, 0, 0] in its
                        // first 16 bytes, a = sqrt(max(0, r^2 - |k - mu|^2)) split exactly into
                        // three bf16 terms (the rest of the slice stays 0)
                        float nk[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            nk[i] = nk1[i];
                            nk1[i] = nk2[i];
                        }
                        const float r = r1;
                        r1 = r2;
                        load_ahead(nk2, r2);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int row = lane + 32 * i;
                            const float ae = sqrtf(fmaxf(0.0f, fmaf(r, r, -nk[i] * nk[i])));
                            const __nv_bfloat16 hi = __float2bfloat16_rn(ae);
                            const float rem = ae - __bfloat162float(hi);
                            const __nv_bfloat16 mid = __float2bfloat16_rn(rem);
                            const __nv_bfloat16 lo =
                                __float2bfloat16_rn(rem - __bfloat162float(mid));
                            const uint32_t bhi = __bfloat16_as_ushort(hi);
                            const uint32_t bmid = __bfloat16_as_ushort(mid);
                            const uint32_t blo = __bfloat16_as_ushort(lo);
                            uint8_t* dst = sK + row * 128 + (((2 * s) ^ (row & 7)) << 4);
                            *reinterpret_cast<uint4*>(dst) =
                                make_uint4(0x3F803F80u, 0x3F80u | (bhi << 16), bmid | (blo << 16), 0u);
                        }
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar_full + 8 * s);
                    }
                }
            }
            if (!ok && lane == 0) {
                // drain: let loads already issued land before the CTA can exit (bounded)
                for (int k = 1; k <= kStages && it - k >= 0; ++k) {
                    const int i2 = it - k;
                    volatile int never = 0;
                    mbar_wait(bar_full + 8 * (i2 % kStages), (i2 / kStages) & 1, &never, a.status);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = make_idesc(kTileM, Nmma);
            const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB), c_base = smem_u32(sC);
            int it = 0;
            bool ok = true;
            for (int u = u_begin; u < u_end && ok; ++u) {
                const int blk = u % a.nblk;
                const uint32_t c_slice = static_cast<uint32_t>((u / a.nblk) % kCSlots) * 32;
                const int rows = min(kKeysPerBlock, a.n - (a.blk0 + blk) * kKeysPerBlock);
                const int ntile = (rows + kTileM - 1) / kTileM;
                for (int t = 0; t < ntile; ++t, ++it) {
                    const int s = it % kStages;
                    const int ab = it & 1;
                    if (!mbar_wait(bar_full + 8 * s, (it / kStages) & 1, abort_flag, a.status) ||
                        !mbar_wait(bar_tempty + 8 * ab, (it >> 1) & 1, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + ab * kChunkN;
                    // D = 1 . c (three bf16 terms) (MIPS: - w_d . a too, from the stage's key
                    // slice), then D += k . (-w) over the 128 dimensions
                    const uint32_t a_first = kMode == kMips
                                                 ? smem_u32(sK) + static_cast<uint32_t>(s) * 32
                                                 : c_base + kOnesSlice * 32;
                    tc_mma(d_tmem, sw128_desc(a_first), sw128_desc(c_base + c_slice), idesc, 0u);
#pragma unroll
                    for (int k = 0; k < kD / 16; ++k) {
                        const uint32_t koff = (k >> 2) * kHalfBytes + (k & 3) * 32;
                        const uint32_t kboff = (k >> 2) * kBHalfBytes + (k & 3) * 32;
                        tc_mma(d_tmem, sw128_desc(a_base + s * kStageBytes + koff),
                               sw128_desc(b_base + kboff), idesc, 1u);
                    }
                    tc_commit(bar_empty + 8 * s);
                    tc_commit(bar_tfull + 8 * ab);
                }
            }
        }
    } else {
        // ---------------- epilogue ----------------
        const int ew = warp - 2;                 // 0..15
        const int quad = warp & 3;               // TMEM lane quadrant this warp may read
        const int colA = (ew >> 2) * 64;         // this warp's two 32-column groups start here
        const int et = tid - 64;                 // 0..511
        const uint32_t tquad = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
        bool aborted = false;
        float* sWd = reinterpret_cast<float*>(smem + Lay::kOffWd);
        if constexpr (kMode == kMips) {
            if (et < kChunkN)
                sWd[et] = et < Nc ? __bfloat162float(a.W[static_cast<size_t>(kD) * a.C + j0 + et])
                                  : 0.0f;
            epi_sync();
        }
        // c_j = w_j . mu of head h, as three bf16 terms, into centre slot h % 3 (thread et
        // writes hyperplane row et). The MMAs that read the slot last (head h - 3) are complete:
        // this runs for the tile two ahead of the one being drained, and heads never decrease.
        int c_head = -1;
        auto ensure_c = [&](int h) {
            if (h == c_head) return;
            c_head = h;
            if (et < kChunkN) {
                float c = 0.0f;
                if (et < Nc) {
                    const float* mu = a.centre + static_cast<size_t>(h) * kD;
                    for (int e = 0; e < kD; ++e) {
                        const uint32_t off = (e >> 6) * kBHalfBytes + et * 128 +
                                             ((((e & 63) >> 3) ^ (et & 7)) << 4) + ((e & 7) << 1);
                        c = fmaf(-__bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sB + off)),
                                 __ldg(mu + e), c);
                    }
                }
                c += 0.0f;                       // never -0: the sign bit must mean c - w.k < 0
                const __nv_bfloat16 hi = __float2bfloat16_rn(c);
                const float r1 = c - __bfloat162float(hi);
                const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
                const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
                const uint32_t w01 = static_cast<uint32_t>(__bfloat16_as_ushort(hi)) |
                                     (static_cast<uint32_t>(__bfloat16_as_ushort(mid)) << 16);
                uint32_t w2 = __bfloat16_as_ushort(lo), w3 = 0u;
                if constexpr (kMode == kMips) {
                    // -W[d][j] against the key slice's three terms of a (a bf16 value: exact)
                    const uint32_t nw = __bfloat16_as_ushort(__float2bfloat16_rn(-sWd[et]));
                    w2 |= nw << 16;
                    w3 = nw | (nw << 16);
                }
                const int slot = h % kCSlots;
                *reinterpret_cast<uint4*>(sC + et * 128 + (((2 * slot) ^ (et & 7)) << 4)) =
                    make_uint4(w01, w2, w3, 0u);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
        };
        auto tiles_in_block = [&](int blk) {
            const int rows = min(kKeysPerBlock, a.n - (a.blk0 + blk) * kKeysPerBlock);
            return (rows + kTileM - 1) / kTileM;
        };
        // The next tile whose centre slot has to be ready (two ahead of the one being drained),
        // tracked incrementally: unit fu = (fbg, fblk), tile ft of fnt.
        int fu = u_begin, ft = 0, fbg = u_begin / a.nblk, fblk = u_begin % a.nblk;
        int fnt = tiles_in_block(fblk);
        auto fill_next = [&]() {
            if (fu >= u_end) return;
            ensure_c(fbg);
            if (++ft == fnt) {
                ft = 0;
                ++fu;
                if (++fblk == a.nblk) {
                    fblk = 0;
                    ++fbg;
                }
                fnt = tiles_in_block(fblk);
            }
        };
        // one unit's staged words -> its Nc plane rows in global memory (coalesced rows); for
        // the argmax codes, its Nc / d table rows of 1024 code bytes
        uint8_t* stg_bytes = reinterpret_cast<uint8_t*>(stg);
        auto store_unit = [&](int bg, int blk) {
            const bool in_range =
                mp_check(a.status, static_cast<long long>(bg) * a.cblk + a.blk0 + blk,
                         static_cast<long long>(a.units / a.nblk) * a.cblk, kSiteEncodeCodes);
            if constexpr (kMode == kArgmax) {
                epi_sync();
                if (!aborted && in_range) {
                    const int ntab = Nc / kD, L = a.C / kD;
                    uint8_t* dst = reinterpret_cast<uint8_t*>(a.codes) +
                                   ((static_cast<size_t>(bg) * a.cblk + a.blk0 + blk) * L + j0 / kD) *
                                       kKeysPerBlock;
                    if (et < ntab * (kKeysPerBlock / 4))
                        reinterpret_cast<uint32_t*>(dst)[et] =
                            reinterpret_cast<const uint32_t*>(stg_bytes)[et];
                }
                epi_sync();
            } else {
                // the staged words of planes colA .. colA + 63 come from the four warps of this
                // column group alone, so those four store them, between barriers of their own
                group_sync(ew >> 2);
                if (!aborted && in_range) {
                    uint32_t* dst = a.codes + (static_cast<size_t>(bg) * a.cblk + a.blk0 + blk) *
                                                  static_cast<size_t>(a.C) * kWordsPerBlock +
                                    static_cast<size_t>(j0) * kWordsPerBlock;
                    // four rows per warp instruction: lane l takes words 4 (l % 8) .. + 3 of
                    // row r0 + l / 8 (bank (w + r) mod 32: distinct across the warp)
                    const int rl = lane >> 3, c4 = (lane & 7) * 4;
                    const int rend = min(Nc, colA + 64);
                    for (int r0 = colA + 4 * (ew & 3); r0 < rend; r0 += 16) {
                        const int r = r0 + rl;
                        if (r < rend) {
                            uint4 v;
                            v.x = stg[(c4 + 0) * kStgPitch + r];
                            v.y = stg[(c4 + 1) * kStgPitch + r];
                            v.z = stg[(c4 + 2) * kStgPitch + r];
                            v.w = stg[(c4 + 3) * kStgPitch + r];
                            *reinterpret_cast<uint4*>(dst + r * kWordsPerBlock + c4) = v;
                        }
                    }
                }
                group_sync(ew >> 2);
            }
        };
        for (int ab = 0; ab < 2; ++ab) {
            fill_next();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_tempty + 8 * ab);
        }
        int it = 0;
        int bg = u_begin / a.nblk, blk = u_begin % a.nblk;
        for (int u = u_begin; u < u_end; ++u) {
            const int ntile = tiles_in_block(blk);
            for (int t = 0; t < ntile; ++t, ++it) {
                const int ab = it & 1;
                if (!aborted) {
                    const bool got = mbar_wait(bar_tfull + 8 * ab, (it >> 1) & 1, abort_flag,
                                               a.status);
                    aborted = !__all_sync(0xffffffffu, got);   // keep the warp uniform
                }
                // sign bits of this warp's two 32-column groups into registers (one TMEM wait
                // per group keeps 32 accumulator registers live) ...
                uint32_t x[2] = {0u, 0u};
                float best64 = -1.0f;        // argmax: this lane's key over this warp's 64 columns
                int code64 = 0;
                if (!aborted) {
                    tc_fence_after();
                    const uint32_t trow = tquad + ab * kChunkN;
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
                        if (colA + 32 * g < Nc) {
                            uint32_t v[32];
                            tmem_ld32(trow + colA + 32 * g, v);
                            tmem_ld_wait();
                            if constexpr (kMode == kArgmax) {
                                // y = -accumulator; first index of the largest |y| of the group:
                                // the leading accumulator and its column, compared by magnitude
                                // (one compare and two selects per element), the code
                                // 2 i + [accumulator > 0] formed once from the winner
                                float bv = 0.0f;
                                int bi = 0;
#pragma unroll
                                for (int c = 0; c < 32; ++c) {
                                    const float ac = __uint_as_float(v[c]);
                                    if (fabsf(ac) > fabsf(bv)) {
                                        bv = ac;
                                        bi = c;
                                    }
                                }
                                const float bst = fabsf(bv);
                                const int cd = 2 * ((colA & (kD - 1)) + 32 * g + bi) + (bv > 0.0f ? 1 : 0);
                                if (g == 0 || bst > best64) {
                                    best64 = bst;
                                    code64 = cd;
                                }
                            } else {
                                x[g] = pack_signs<1>(v);
                            }
                        }
                    }
                }
                // ... which frees the accumulator buffer for the tile two ahead at once
                fill_next();
                tc_fence_before();
                __syncwarp();
                if (lane == 0 && !aborted) mbar_arrive(bar_tempty + 8 * ab);
                if constexpr (kMode == kArgmax) {
                    // the two halves of a table meet: (|y|, code) per (table, half, key row) in
                    // the exchange area (two parities, so a tile's reads never race the next
                    // tile's writes), then the lower half picks and stages the code byte
                    const int tab = colA / kD, half = (colA / 64) & 1, row = quad * 32 + lane;
                    float2* xch = reinterpret_cast<float2*>(stg_bytes + kXchOff) +
                                  (it & 1) * (2 * 2 * kTileM);
                    if (!aborted && colA < Nc)
                        xch[(tab * 2 + half) * kTileM + row] =
                            make_float2(best64, __int_as_float(code64));
                    epi_sync();
                    if (!aborted && colA < Nc && half == 0) {
                        const float2 o = xch[(tab * 2 + 1) * kTileM + row];
                        const int code = o.x > best64 ? __float_as_int(o.y) : code64;
                        stg_bytes[tab * kKeysPerBlock + t * kTileM + row] = static_cast<uint8_t>(code);
                    }
                } else if (!aborted) {
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
                        const int col = colA + 32 * g;
                        if (col < Nc) {
                            const uint32_t y = warp_transpose32(x[g], lane);
                            if (col + lane < Nc) stg[(t * 4 + quad) * kStgPitch + col + lane] = y;
                        }
                    }
                }
            }
            // the block's rows go out once its last tile is staged (its accumulator already
            // released, so the MMA keeps running meanwhile); kept out of the tile loop, whose
            // body then stays free of the store's registers and barriers
            store_unit(bg, blk);
            if (++blk == a.nblk) {
                blk = 0;
                ++bg;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(2 * kChunkN)
                     : "memory");
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// The failure path's test hook: one thread waits, with the encoder's bounded wait, on an
// mbarrier whose phase nothing completes (no arrival, no copy, no MMA), so the wait gives up
// after limit_ns and raises MP_ERR_TIMEOUT in the status word, as a stalled encoder would.
__global__ void wait_expiry_kernel(unsigned long long limit_ns, int* status) {
    __shared__ __align__(8) uint64_t bar_storage;
    __shared__ int abort_flag;
    const uint32_t bar = static_cast<uint32_t>(__cvta_generic_to_shared(&bar_storage));
    abort_flag = 0;
    mbar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_wait(bar, 0, &abort_flag, status, limit_ns);
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

}  // namespace

cudaError_t launch_wait_expiry(unsigned long long limit_ns, int* status, cudaStream_t st) {
    wait_expiry_kernel<<<1, 1, 0, st>>>(limit_ns, status);
    return cudaGetLastError();
}

cudaError_t prepare_encode_tc() {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, wait_expiry_kernel) != cudaSuccess) return cudaErrorNotSupported;
    const struct {
        void (*fn)(const CUtensorMap, const EncodeArgs);
        uint32_t smem;
    } kernels[] = {{encode_tc_kernel<kSign>, EncLayout<kSign>::kSmemBytes},
                   {encode_tc_kernel<kMips>, EncLayout<kMips>::kSmemBytes},
                   {encode_tc_kernel<kArgmax>, EncLayout<kArgmax>::kSmemBytes}};
    for (const auto& k : kernels) {
        const cudaError_t e = cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(k.smem));
        if (e != cudaSuccess) return e;
    }
    return encode_tiled_fn() ? cudaSuccess : cudaErrorNotSupported;
}

cudaError_t launch_encode_tc(const void* keys, const float* centre, const void* W, int B,
                             int Hkv, int ncap, int blk0, int blk1, int K, int L,
                             uint32_t* codes, int* status, cudaStream_t st, const float* norms,
                             const float* radius, bool argmax) {
    const int C = K * L;
    if (C == 0 || blk1 <= blk0) return cudaSuccess;
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap map;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(ncap),
                                static_cast<cuuint64_t>(B) * Hkv};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2,
                                   static_cast<cuuint64_t>(ncap) * kD * 2};
    const cuuint32_t box[3] = {64, kTileM, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(keys), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    EncodeArgs a;
    a.centre = centre;
    a.W = reinterpret_cast<const __nv_bfloat16*>(W);
    a.codes = codes;
    a.status = status;
    a.C = C;
    a.nchunk = (C + kChunkN - 1) / kChunkN;
    a.nblk = blk1 - blk0;
    a.n = ncap;
    a.blk0 = blk0;
    a.cblk = (ncap + kKeysPerBlock - 1) / kKeysPerBlock;
    a.norms = norms;
    a.radius = radius;
    a.units = B * Hkv * a.nblk;
    int parts = device_sm_count() / a.nchunk;
    if (parts < 1) parts = 1;
    if (parts > a.units) parts = a.units;
    a.parts = parts;
    if (argmax)
        encode_tc_kernel<kArgmax><<<a.nchunk * parts, kThreads, EncLayout<kArgmax>::kSmemBytes,
                                    st>>>(map, a);
    else if (norms)
        encode_tc_kernel<kMips><<<a.nchunk * parts, kThreads, EncLayout<kMips>::kSmemBytes,
                                  st>>>(map, a);
    else
        encode_tc_kernel<kSign><<<a.nchunk * parts, kThreads, EncLayout<kSign>::kSmemBytes,
                                  st>>>(map, a);
    return cudaGetLastError();
}

}  // namespace mp
