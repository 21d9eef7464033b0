// MIPS -> cosine variant of the key encoding ("MagicPIG: LSH Sampling for Efficient LLM
// Generation", method details, variance reduction with LSH): with r the largest key length, the
// query is extended by a 0 and each key by sqrt(r^2 - |k|^2), so every extended key has length r
// and the collision probability of the extended pair grows with the inner product q.k (its
// cosine is q.k / (|q| r)). The keys extended are the centred ones, k - mu, since the centring
// step comes before the tables are built. W carries a (d + 1)-th row for the extra coordinate;
// the query's bits use the first d rows (its extra coordinate is 0), so query encoding is
// unchanged.
#include "mp_internal.cuh"

namespace mp {
namespace {

constexpr int kRadiusRows = 1024;      // keys per radius CTA
constexpr int kRadiusThreads = 256;
constexpr int kMipsKeys = 64;          // keys per encoding CTA (two 32-key words)
constexpr int kMipsPlanes = 16;        // hyperplanes per pass

constexpr int kRadiusRowsAtOnce = 4;   // key rows a half-warp has in flight

// the 8 elements [8 hl, 8 hl + 8) of key row `row` minus the centre, squared and summed
__device__ __forceinline__ float row_part_sq(const void* keys, int keys_bf16, size_t row, int hl,
                                             const float (&mu)[8]) {
    float f[8];
    if (keys_bf16) {
        const uint4 v = *reinterpret_cast<const uint4*>(
            reinterpret_cast<const __nv_bfloat16*>(keys) + row * kD + 8 * hl);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    } else {
        const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(keys) +
                                                          row * kD + 8 * hl);
        const float4 a = p[0], b = p[1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float x = f[i] - mu[i];
        s = fmaf(x, x, s);
    }
    return s;
}

// |k_i - mu| of keys [k0, k1): a half-warp per key row (16 lanes x 16-byte loads of a bf16 row,
// two for fp32; kRadiusRowsAtOnce rows in flight), lane hl elements 8 hl .. 8 hl + 7. With
// radius: its maximum into radius[bh] (the maximum of non-negative floats through their ordered
// bit patterns); with norms: each row's into norms[bh][i].
__global__ void __launch_bounds__(kRadiusThreads)
    key_radius_kernel(const void* keys, int keys_bf16, const float* centre, int ncap, int k0,
                      int k1, float* radius, float* norms) {
    constexpr int U = kRadiusRowsAtOnce;
    constexpr int kHalves = kRadiusThreads / 16;
    const int bh = blockIdx.y, lane = threadIdx.x & 31, hw = threadIdx.x >> 4, hl = lane & 15;
    const unsigned hmask = 0xffffu << (lane & 16);
    const int r0 = k0 + blockIdx.x * kRadiusRows, r1 = min(k1, r0 + kRadiusRows);
    float mu[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mu[i] = centre[static_cast<size_t>(bh) * kD + 8 * hl + i];
    float best = 0.0f;
    for (int rb = r0 + hw * U; rb < r1; rb += kHalves * U) {
        float s[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int r = min(rb + u, r1 - 1);            // past r1: a repeat of the last row
            s[u] = row_part_sq(keys, keys_bf16, static_cast<size_t>(bh) * ncap + r, hl, mu);
        }
#pragma unroll
        for (int o = 8; o; o >>= 1)
#pragma unroll
            for (int u = 0; u < U; ++u) s[u] += __shfl_xor_sync(hmask, s[u], o);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float nr = sqrtf(s[u]);
            best = fmaxf(best, nr);
            if (norms && hl == u && rb + u < r1) norms[static_cast<size_t>(bh) * ncap + rb + u] = nr;
        }
    }
    best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, 16));
    if (radius && lane == 0)
        atomicMax(reinterpret_cast<unsigned*>(radius + bh), __float_as_uint(best));
}

// Codes of keys [n0, n1) from the extended centred keys: one key per thread, a warp's 32 keys
// form one word per hyperplane through a ballot; only the range's bits of a word change (each
// (plane, word) has one writer). bit = [sum_e W[e][j] (k[e] - mu[e]) + W[d][j] a > 0] with
// a = sqrt(max(0, r^2 - |k - mu|^2)), in fp32.
__global__ void __launch_bounds__(kMipsKeys)
    encode_mips_kernel(const void* keys, int keys_bf16, const float* centre, const void* W,
                       int w_bf16, const float* radius, int ncap, int n0, int n1, int C,
                       int cblk, uint32_t* codes) {
    __shared__ float kbar[kMipsKeys][kD + 1];
    __shared__ float Wsm[kD + 1][kMipsPlanes];
    const int bh = blockIdx.y, tid = threadIdx.x, lane = tid & 31;
    const int i0 = (n0 / kMipsKeys + blockIdx.x) * kMipsKeys;
    for (int idx = tid; idx < kMipsKeys * kD; idx += kMipsKeys) {
        const int r = idx / kD, e = idx % kD, i = i0 + r;
        float v = 0.0f;
        if (i < ncap)
            v = load_elem(keys, keys_bf16, (static_cast<size_t>(bh) * ncap + i) * kD + e) -
                centre[static_cast<size_t>(bh) * kD + e];
        kbar[r][e] = v;
    }
    __syncthreads();
    float nn = 0.0f;
    for (int e = 0; e < kD; ++e) nn = fmaf(kbar[tid][e], kbar[tid][e], nn);
    const float rr = radius[bh];
    const float extra = sqrtf(fmaxf(0.0f, fmaf(rr, rr, -nn)));
    const int key = i0 + tid;
    const uint32_t keep = __ballot_sync(0xffffffffu, key >= n0 && key < n1);   // range bits
    const int w = key / 32;
    uint32_t* dst = codes + (static_cast<size_t>(bh) * cblk + w / kWordsPerBlock) *
                                static_cast<size_t>(C) * kWordsPerBlock + w % kWordsPerBlock;
    for (int j0 = 0; j0 < C; j0 += kMipsPlanes) {
        __syncthreads();
        for (int idx = tid; idx < (kD + 1) * kMipsPlanes; idx += kMipsKeys) {
            const int e = idx / kMipsPlanes, c = idx % kMipsPlanes, j = j0 + c;
            Wsm[e][c] = j < C ? load_elem(W, w_bf16, static_cast<size_t>(e) * C + j) : 0.0f;
        }
        __syncthreads();
        float P[kMipsPlanes];
#pragma unroll
        for (int c = 0; c < kMipsPlanes; ++c) P[c] = 0.0f;
        for (int e = 0; e < kD; ++e) {
            const float x = kbar[tid][e];
#pragma unroll
            for (int c = 0; c < kMipsPlanes; ++c) P[c] = fmaf(Wsm[e][c], x, P[c]);
        }
        uint32_t mine = 0;
#pragma unroll
        for (int c = 0; c < kMipsPlanes; ++c) {
            const uint32_t bal = __ballot_sync(0xffffffffu, fmaf(Wsm[kD][c], extra, P[c]) > 0.0f);
            if (lane == c) mine = bal;
        }
        if (keep != 0u && lane < kMipsPlanes && j0 + lane < C) {
            uint32_t* p = dst + static_cast<size_t>(j0 + lane) * kWordsPerBlock;
            *p = keep == 0xffffffffu ? mine : ((*p & ~keep) | (mine & keep));
        }
    }
}

}  // namespace

cudaError_t launch_key_radius(const void* keys, bool keys_bf16, const float* centre, int BH,
                              int ncap, int n, float* radius, cudaStream_t st, float* norms,
                              int k0, int k1) {
    if (k1 < 0) k1 = n;
    if (radius) {
        const cudaError_t e = cudaMemsetAsync(radius, 0, static_cast<size_t>(BH) * sizeof(float),
                                              st);
        if (e != cudaSuccess) return e;
    }
    if (k1 <= k0) return cudaSuccess;
    const dim3 grid((k1 - k0 + kRadiusRows - 1) / kRadiusRows, BH);
    key_radius_kernel<<<grid, kRadiusThreads, 0, st>>>(keys, keys_bf16, centre, ncap, k0, k1,
                                                       radius, norms);
    return cudaGetLastError();
}

cudaError_t launch_encode_mips(const void* keys, bool keys_bf16, const float* centre,
                               const void* W, bool w_bf16, const float* radius, int B, int Hkv,
                               int ncap, int n0, int n1, int K, int L, uint32_t* codes,
                               cudaStream_t st) {
    const int C = K * L;
    if (C == 0 || n1 <= n0) return cudaSuccess;
    const int cblk = (ncap + kKeysPerBlock - 1) / kKeysPerBlock;
    const int tiles = (n1 - 1) / kMipsKeys - n0 / kMipsKeys + 1;
    const dim3 grid(tiles, B * Hkv);
    encode_mips_kernel<<<grid, kMipsKeys, 0, st>>>(keys, keys_bf16, centre, W, w_bf16, radius,
                                                   ncap, n0, n1, C, cblk, codes);
    return cudaGetLastError();
}

cudaError_t prepare_mips() {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, key_radius_kernel);
    if (e != cudaSuccess) return e;
    return cudaFuncGetAttributes(&fa, encode_mips_kernel);
}

}  // namespace mp
