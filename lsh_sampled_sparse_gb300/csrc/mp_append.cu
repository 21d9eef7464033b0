// Incremental append of decode tokens: the codes of a short range of keys [n0, n1), written into
// the 32-key words they share with keys already encoded (whose bits are kept).
//
// The pages compute the centre and build the tables once, before decoding ("MagicPIG: LSH
// Sampling for Efficient LLM Generation", method details, data preprocessing and centering), and
// are silent on tokens generated afterwards; each new key is encoded here with the centre of the
// build, bit_{i,j} = [w_j . (k_i - mu) > 0], the same definition as the build.
#include "mp_internal.cuh"

namespace mp {
namespace {

constexpr int kAppendWarps = 4;                                // >= the words a range touches
static_assert(kAppendWarps >= (kAppendMaxKeys + 31) / 32 + 1, "a warp per touched word");
constexpr int kAppendThreads = kAppendWarps * 32;
constexpr int kStageBatch = 16;                                // loads a thread issues at once
constexpr int kAppendPlanes = 32;                              // hyperplanes per CTA (one a lane)
constexpr int kAppendKeysAtOnce = 4;                           // independent sums a lane carries

// One CTA per (chunk of 32 hyperplanes, head). The chunk of W and the range's centred keys are
// staged in shared memory, kStageBatch loads in flight per thread; warp w then takes the range's
// w-th 32-key word, lane j hyperplane j0 + j, and rewrites that word's bits of the range only (each
// (plane, word) has one owner, so a plain read-modify-write). Each sum runs over e in order,
// fmaf(W[e][j], k[e] - mu[e], acc): the arithmetic of the CUDA-core block encoder.
__global__ void __launch_bounds__(kAppendThreads)
    encode_append_kernel(const void* keys, int keys_bf16, const float* centre, const void* W,
                         int w_bf16, int ncap, int n0, int n1, int C, int cblk, uint32_t* codes) {
    extern __shared__ __align__(16) float sm[];
    float* Ws = sm;                                   // [kD][kAppendPlanes]
    float* kbar = sm + kD * kAppendPlanes;            // [n1 - n0][kD]
    const int bh = blockIdx.y, j0 = blockIdx.x * kAppendPlanes, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int m = n1 - n0;
    for (int base = 0; base < kD * kAppendPlanes; base += kAppendThreads * kStageBatch) {
        float v[kStageBatch];
#pragma unroll
        for (int u = 0; u < kStageBatch; ++u) {
            const int idx = base + u * kAppendThreads + tid;
            const int e = idx / kAppendPlanes, j = j0 + idx % kAppendPlanes;
            v[u] = idx < kD * kAppendPlanes && j < C
                       ? load_elem(W, w_bf16, static_cast<size_t>(e) * C + j) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < kStageBatch; ++u) {
            const int idx = base + u * kAppendThreads + tid;
            if (idx < kD * kAppendPlanes) Ws[idx] = v[u];
        }
    }
    for (int base = 0; base < m * kD; base += kAppendThreads * kStageBatch) {
        float v[kStageBatch];
#pragma unroll
        for (int u = 0; u < kStageBatch; ++u) {
            const int idx = base + u * kAppendThreads + tid;
            v[u] = idx < m * kD
                       ? load_elem(keys, keys_bf16,
                                   (static_cast<size_t>(bh) * ncap + n0 + idx / kD) * kD + idx % kD) -
                             centre[static_cast<size_t>(bh) * kD + idx % kD]
                       : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < kStageBatch; ++u) {
            const int idx = base + u * kAppendThreads + tid;
            if (idx < m * kD) kbar[idx] = v[u];
        }
    }
    __syncthreads();
    const int w = n0 / 32 + warp;                     // absolute 32-key word
    const int k0 = max(n0, w * 32), k1 = min(n1, w * 32 + 32);
    const int j = j0 + lane;
    if (k0 >= k1 || j >= C) return;
    uint32_t bits = 0u;
    for (int r0 = k0; r0 < k1; r0 += kAppendKeysAtOnce) {
        const float* kr[kAppendKeysAtOnce];
        float P[kAppendKeysAtOnce];
#pragma unroll
        for (int u = 0; u < kAppendKeysAtOnce; ++u) {
            kr[u] = kbar + static_cast<size_t>(min(r0 + u, k1 - 1) - n0) * kD;   // past k1: a repeat
            P[u] = 0.0f;
        }
#pragma unroll 4
        for (int e = 0; e < kD; ++e) {
            const float wv = Ws[e * kAppendPlanes + lane];
#pragma unroll
            for (int u = 0; u < kAppendKeysAtOnce; ++u) P[u] = fmaf(wv, kr[u][e], P[u]);
        }
#pragma unroll
        for (int u = 0; u < kAppendKeysAtOnce; ++u)
            if (r0 + u < k1 && P[u] > 0.0f) bits |= 1u << ((r0 + u) & 31);
    }
    const uint32_t range = bits_below(k1 - w * 32) & ~bits_below(k0 - w * 32);
    uint32_t* dst = codes + ((static_cast<size_t>(bh) * cblk + w / kWordsPerBlock) * C + j) *
                                kWordsPerBlock + w % kWordsPerBlock;
    *dst = (*dst & ~range) | bits;
}

}  // namespace

cudaError_t launch_encode_append(const void* keys, bool keys_bf16, const float* centre,
                                 const void* W, bool w_bf16, int B, int Hkv, int ncap, int n0,
                                 int n1, int K, int L, uint32_t* codes, cudaStream_t st) {
    const int C = K * L;
    if (C == 0 || n1 <= n0) return cudaSuccess;
    if (n1 - n0 > kAppendMaxKeys) return cudaErrorInvalidValue;
    const int cblk = (ncap + kKeysPerBlock - 1) / kKeysPerBlock;
    const size_t smem = (static_cast<size_t>(kD) * kAppendPlanes +
                         static_cast<size_t>(n1 - n0) * kD) * sizeof(float);
    const dim3 grid((C + kAppendPlanes - 1) / kAppendPlanes, B * Hkv);
    encode_append_kernel<<<grid, kAppendThreads, smem, st>>>(keys, keys_bf16, centre, W, w_bf16,
                                                            ncap, n0, n1, C, cblk, codes);
    return cudaGetLastError();
}

cudaError_t prepare_append() {
    cudaFuncAttributes fa;
    return cudaFuncGetAttributes(&fa, encode_append_kernel);
}

}  // namespace mp
