// Key centre, the fp32 CUDA-core encoder, and the inspection kernels (selection lists,
// collision counts, unpacked codes).
#include <algorithm>

#include "mp_internal.cuh"

namespace mp {
namespace {

// ------------------------------------------------------------------------------------------------
// Centre: mu = (1/n) sum_i k_i per head ("LSH Sampling...", method details, data preprocessing
// and centering). Fixed partition into row ranges, fixed reduction order: run-to-run identical.
// ------------------------------------------------------------------------------------------------
constexpr int kMeanMaxRows = 1024;   // rows per partial sum for long contexts
constexpr int kMeanMinRows = 64;     // ... and at least this many for short ones
constexpr int kMeanCtas = 608;       // row ranges wanted in all (four per SM of a GB300)
constexpr int kMeanThreads = 256;

// One CTA per (row range, head): the range's column sums into `partial`; the last CTA of a head
// to finish (release-acquire counter) adds the head's partials in range order and writes mu.
template <typename T>
__global__ void __launch_bounds__(kMeanThreads)
    key_mean_kernel(const T* keys, int ncap, int n, int rows, int nsplit, float* partial,
                    unsigned* counters, float* centre) {
    // thread -> (column group of 16 bytes, row phase); rows stride by the number of row phases
    constexpr int kPer = 16 / sizeof(T);                 // elements per 16-byte load
    constexpr int kGroups = kD / kPer;                   // column groups per row
    constexpr int kPhases = kMeanThreads / kGroups;      // rows read in parallel
    __shared__ float red[kPhases][kD + 4];
    __shared__ int last;
    const int bh = blockIdx.y, split = blockIdx.x, tid = threadIdx.x;
    const int cg = tid % kGroups, ph = tid / kGroups;
    const int r0 = split * rows, r1 = min(n, r0 + rows);
    const T* base = keys + static_cast<size_t>(bh) * ncap * kD + cg * kPer;
    float acc[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] = 0.0f;
#pragma unroll 8
    for (int r = r0 + ph; r < r1; r += kPhases) {
        const uint4 raw = __ldcs(reinterpret_cast<const uint4*>(base + static_cast<size_t>(r) * kD));
        const T* v = reinterpret_cast<const T*>(&raw);
#pragma unroll
        for (int i = 0; i < kPer; ++i) acc[i] += to_float(v[i]);
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) red[ph][cg * kPer + i] = acc[i];
    __syncthreads();
    if (tid < kD) {
        float s = 0.0f;
        for (int p = 0; p < kPhases; ++p) s += red[p][tid];
        partial[(static_cast<size_t>(bh) * nsplit + split) * kD + tid] = s;
    }
    __syncthreads();
    if (tid == 0) {
        unsigned old;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                     : "=r"(old)
                     : "l"(counters + bh)
                     : "memory");
        last = old == static_cast<unsigned>(nsplit - 1);
    }
    __syncthreads();
    if (!last) return;
    // the head's partials: thread t sums columns 4 (t % 32) .. + 3 of the ranges k = t / 32,
    // t / 32 + 8, ... in order (16-byte loads, all of a thread's in flight at once), then the
    // 8 slices add up in order: a fixed order, and one memory round trip for the partials
    static_assert(kMeanThreads == 256 && kPhases >= 8, "8 slices of 32 four-column groups");
    const int c4 = tid & 31, slice = tid >> 5;
    const float4* ph4 = reinterpret_cast<const float4*>(partial + static_cast<size_t>(bh) * nsplit * kD) + c4;
    float4 acc4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    constexpr int kBatch = 16;
    for (int k0 = slice; k0 < nsplit; k0 += 8 * kBatch) {
        float4 v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int k = k0 + 8 * j;
            v[j] = k < nsplit ? __ldcg(ph4 + static_cast<size_t>(k) * (kD / 4))
                              : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            acc4.x += v[j].x;
            acc4.y += v[j].y;
            acc4.z += v[j].z;
            acc4.w += v[j].w;
        }
    }
    red[slice][4 * c4 + 0] = acc4.x;
    red[slice][4 * c4 + 1] = acc4.y;
    red[slice][4 * c4 + 2] = acc4.z;
    red[slice][4 * c4 + 3] = acc4.w;
    __syncthreads();
    if (tid < kD) {
        float t = 0.0f;
#pragma unroll
        for (int q = 0; q < 8; ++q) t += red[q][tid];
        centre[static_cast<size_t>(bh) * kD + tid] = t / static_cast<float>(n);
    }
    if (tid == 0) counters[bh] = 0u;
}

// ------------------------------------------------------------------------------------------------
// fp32 CUDA-core encoder for dtype pairs the tensor-core path does not take (fp32 keys or W):
// bit_{i,j} = [sum_e W[e][j] (k_i[e] - mu[e]) > 0] in fp32, one key per thread, a warp's 32 keys
// form one word per hyperplane through a ballot. Whole 1024-key blocks from blk0 on (keys at or
// past ncap read as zero). Grid z splits the hyperplanes when there are few keys, so that short
// contexts still fill the GPU; every sum is the same sequence of fmaf over e either way.
// ------------------------------------------------------------------------------------------------
constexpr int kSimtKeys = 64;      // keys per CTA (2 words)
constexpr int kSimtPlanes = 16;    // hyperplanes per pass

__global__ void __launch_bounds__(kSimtKeys)
    encode_simt_kernel(const void* keys, int keys_bf16, const float* centre, const void* W,
                       int w_bf16, int ncap, int C, int cblk, int blk0, uint32_t* codes) {
    __shared__ float kbar[kSimtKeys][kD + 1];
    __shared__ float Wsm[kD][kSimtPlanes];
    const int bh = blockIdx.y, tile = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
    const int warp = tid >> 5;
    const int i0 = blk0 * kKeysPerBlock + tile * kSimtKeys;
    for (int idx = tid; idx < kSimtKeys * kD; idx += kSimtKeys) {
        const int r = idx / kD, e = idx % kD, i = i0 + r;
        float v = 0.0f;
        if (i < ncap)
            v = load_elem(keys, keys_bf16, (static_cast<size_t>(bh) * ncap + i) * kD + e) -
                centre[static_cast<size_t>(bh) * kD + e];
        kbar[r][e] = v;
    }
    const int blk = i0 / kKeysPerBlock;
    const int word = (i0 % kKeysPerBlock) / 32 + warp;
    uint32_t* dst = codes + (static_cast<size_t>(bh) * cblk + blk) * static_cast<size_t>(C) *
                                kWordsPerBlock + word;
    const int passes = (C + kSimtPlanes - 1) / kSimtPlanes;
    const int per = (passes + gridDim.z - 1) / gridDim.z;          // passes of this CTA
    const int j_lo = blockIdx.z * per * kSimtPlanes;
    const int j_hi = min(C, j_lo + per * kSimtPlanes);
    for (int j0 = j_lo; j0 < j_hi; j0 += kSimtPlanes) {
        __syncthreads();
        for (int idx = tid; idx < kD * kSimtPlanes; idx += kSimtKeys) {
            const int e = idx / kSimtPlanes, c = idx % kSimtPlanes, j = j0 + c;
            Wsm[e][c] = j < C ? load_elem(W, w_bf16, static_cast<size_t>(e) * C + j) : 0.0f;
        }
        __syncthreads();
        float P[kSimtPlanes];
#pragma unroll
        for (int c = 0; c < kSimtPlanes; ++c) P[c] = 0.0f;
        for (int e = 0; e < kD; ++e) {
            const float x = kbar[tid][e];
#pragma unroll
            for (int c = 0; c < kSimtPlanes; ++c) P[c] = fmaf(Wsm[e][c], x, P[c]);
        }
        uint32_t mine = 0;
#pragma unroll
        for (int c = 0; c < kSimtPlanes; ++c) {
            const uint32_t bal = __ballot_sync(0xffffffffu, P[c] > 0.0f);
            if (lane == c) mine = bal;
        }
        if (lane < kSimtPlanes && j0 + lane < C)
            dst[static_cast<size_t>(j0 + lane) * kWordsPerBlock] = mine;
    }
}

// ------------------------------------------------------------------------------------------------
// Inspection kernels
// ------------------------------------------------------------------------------------------------
// Per query row: ascending indices of the selected keys from the per-block selection words.
__global__ void compact_selection_kernel(const uint32_t* selmask, int n, int nblk, int n_sink,
                                         int n_local, int32_t* sel_idx, int32_t* sel_count) {
    const int row = blockIdx.x, lane = threadIdx.x;
    const uint32_t* m = selmask + static_cast<size_t>(row) * nblk * 32;
    int32_t* out = sel_idx + static_cast<size_t>(row) * n;
    int pos = 0;
    for (int blk = 0; blk < nblk; ++blk) {
        // the scan's words exclude T already; the bucketed lookup's do not
        const int key0 = blk * kKeysPerBlock + lane * 32;
        const uint32_t valid = bits_below(n - key0);
        const uint32_t tm = (bits_below(n_sink - key0) | ~bits_below(n - n_local - key0)) & valid;
        const uint32_t w = m[blk * 32 + lane] & valid & ~tm;
        const int c = __popc(w);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        int p = pos + incl - c;
        uint32_t bits = w;
        while (bits) {
            const int bit = __ffs(bits) - 1;
            bits &= bits - 1;
            out[p++] = blk * kKeysPerBlock + lane * 32 + bit;
        }
        pos += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) sel_count[row] = pos;
}

// Exact collision counts, one thread per (key, query row), straight from the definition.
__global__ void collision_counts_kernel(const uint32_t* codes, const uint32_t* qbits, int n,
                                        int nblk, int Hq, int G, int K, int L, int qwords,
                                        uint8_t* cnt) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int row = blockIdx.y;
    if (i >= n) return;
    const int b = row / Hq, h = row % Hq, bh = b * (Hq / G) + h / G;
    const int C = K * L;
    const uint32_t* cb = codes + (static_cast<size_t>(bh) * nblk + i / kKeysPerBlock) *
                                     static_cast<size_t>(C) * kWordsPerBlock +
                         (i % kKeysPerBlock) / 32;
    const uint32_t* qb = qbits + static_cast<size_t>(row) * qwords;
    int c = 0;
    for (int t = 0; t < L; ++t) {
        bool eq = true;
        for (int bb = 0; bb < K; ++bb) {
            const int j = t * K + bb;
            const uint32_t kbit = (cb[static_cast<size_t>(j) * kWordsPerBlock] >> (i & 31)) & 1u;
            const uint32_t qbit = (qb[j >> 5] >> (j & 31)) & 1u;
            eq = eq && (kbit == qbit);
        }
        c += eq ? 1 : 0;
    }
    cnt[static_cast<size_t>(row) * n + i] = static_cast<uint8_t>(c > 255 ? 255 : c);
}

__global__ void codes_unpack_kernel(const uint32_t* codes, int n, int nblk, int K, int L,
                                    uint32_t* out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int bh = blockIdx.y;
    if (i >= n) return;
    const int C = K * L;
    const uint32_t* cb = codes + (static_cast<size_t>(bh) * nblk + i / kKeysPerBlock) *
                                     static_cast<size_t>(C) * kWordsPerBlock +
                         (i % kKeysPerBlock) / 32;
    for (int t = 0; t < L; ++t) {
        uint32_t code = 0;
        for (int bb = 0; bb < K; ++bb) {
            const int j = t * K + bb;
            code |= ((cb[static_cast<size_t>(j) * kWordsPerBlock] >> (i & 31)) & 1u) << bb;
        }
        out[(static_cast<size_t>(bh) * n + i) * L + t] = code;
    }
}

}  // namespace

// Rows per range: 1024, halved (down to 64) while the BH heads would give fewer than kMeanCtas
// ranges, so that short contexts spread over the GPU too. A function of (BH, n) only: the
// workspace size and the launch agree.
int key_mean_rows(int BH, int n) {
    int rows = kMeanMaxRows;
    while (rows > kMeanMinRows &&
           static_cast<long long>(BH) * ((n + rows - 1) / rows) < kMeanCtas)
        rows /= 2;
    return rows;
}
int key_mean_splits(int BH, int n) {
    const int rows = key_mean_rows(BH, n);
    return (n + rows - 1) / rows;
}

cudaError_t launch_key_mean(const void* keys, bool bf16, int BH, int ncap, int n, float* centre,
                            float* partial, int nsplit, cudaStream_t st) {
    // the per-head counters follow the partial sums in the workspace; they start at zero
    unsigned* counters = reinterpret_cast<unsigned*>(partial + static_cast<size_t>(BH) * nsplit * kD);
    cudaError_t e = cudaMemsetAsync(counters, 0, static_cast<size_t>(BH) * sizeof(unsigned), st);
    if (e != cudaSuccess) return e;
    const dim3 grid(nsplit, BH);
    const int rows = key_mean_rows(BH, n);
    if (nsplit != key_mean_splits(BH, n)) return cudaErrorInvalidValue;
    if (bf16)
        key_mean_kernel<__nv_bfloat16><<<grid, kMeanThreads, 0, st>>>(
            reinterpret_cast<const __nv_bfloat16*>(keys), ncap, n, rows, nsplit, partial,
            counters, centre);
    else
        key_mean_kernel<float><<<grid, kMeanThreads, 0, st>>>(
            reinterpret_cast<const float*>(keys), ncap, n, rows, nsplit, partial, counters,
            centre);
    return cudaGetLastError();
}

cudaError_t launch_encode_simt(const void* keys, bool keys_bf16, const float* centre,
                               const void* W, bool w_bf16, int B, int Hkv, int ncap, int blk0,
                               int blk1, int K, int L, uint32_t* codes, cudaStream_t st) {
    const int C = K * L;
    if (C == 0 || blk1 <= blk0) return cudaSuccess;
    const int cblk = (ncap + kKeysPerBlock - 1) / kKeysPerBlock;
    const int tiles = (blk1 - blk0) * (kKeysPerBlock / kSimtKeys) * B * Hkv;
    // hyperplane parts: enough CTAs for about four per SM, at most one part per pass
    const int passes = (C + kSimtPlanes - 1) / kSimtPlanes;
    const int want = (4 * device_sm_count() + tiles - 1) / tiles;
    const int parts = std::max(1, std::min(passes, want));
    const dim3 grid((blk1 - blk0) * (kKeysPerBlock / kSimtKeys), B * Hkv, parts);
    encode_simt_kernel<<<grid, kSimtKeys, 0, st>>>(keys, keys_bf16, centre, W, w_bf16, ncap, C,
                                                    cblk, blk0, codes);
    return cudaGetLastError();
}

cudaError_t launch_compact_selection(const uint32_t* selmask, int rows, int n, int nblk,
                                     int n_sink, int n_local, int32_t* sel_idx,
                                     int32_t* sel_count, cudaStream_t st) {
    compact_selection_kernel<<<rows, 32, 0, st>>>(selmask, n, nblk, n_sink, n_local, sel_idx,
                                                  sel_count);
    return cudaGetLastError();
}

cudaError_t launch_collision_counts(const uint32_t* codes, const uint32_t* qbits,
                                    const DecodeShape& s, uint8_t* cnt, cudaStream_t st) {
    const dim3 grid((s.n + 255) / 256, s.B * s.Hq);
    collision_counts_kernel<<<grid, 256, 0, st>>>(codes, qbits, s.n, s.cblk, s.Hq, s.Hq / s.Hkv,
                                                  s.K, s.L, s.qwords, cnt);
    return cudaGetLastError();
}

cudaError_t launch_codes_unpack(const uint32_t* codes, int BH, int n, int K, int L,
                                uint32_t* out, cudaStream_t st) {
    const int nblk = (n + kKeysPerBlock - 1) / kKeysPerBlock;
    const dim3 grid((n + 255) / 256, BH);
    codes_unpack_kernel<<<grid, 256, 0, st>>>(codes, n, nblk, K, L, out);
    return cudaGetLastError();
}

cudaError_t prepare_misc() {
    cudaFuncAttributes fa;
    cudaError_t e;
    if ((e = cudaFuncGetAttributes(&fa, key_mean_kernel<float>)) != cudaSuccess) return e;
    if ((e = cudaFuncGetAttributes(&fa, key_mean_kernel<__nv_bfloat16>)) != cudaSuccess) return e;
    if ((e = cudaFuncGetAttributes(&fa, encode_simt_kernel)) != cudaSuccess) return e;
    if ((e = cudaFuncGetAttributes(&fa, compact_selection_kernel)) != cudaSuccess) return e;
    if ((e = cudaFuncGetAttributes(&fa, collision_counts_kernel)) != cudaSuccess) return e;
    return cudaFuncGetAttributes(&fa, codes_unpack_kernel);
}

}  // namespace mp
