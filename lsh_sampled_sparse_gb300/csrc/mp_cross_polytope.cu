// Cross-polytope hashing, the hash the pages name as the way to shrink the tables ("MagicPIG: LSH
// Sampling for Efficient LLM Generation", conclusion: future work). A table hashes a vector x to
// the signed index of the largest |coordinate| of G_t x, G_t a d x d matrix of i.i.d. N(0, 1)
// entries: code = 2 i + (1 if (G_t x)_i < 0), one byte for d = 128. One hash per table (K = 1);
// keys are centred first and the query is not, as for SimHash.
//
// Codes: bytes [B*Hkv][blocks][L][1024]: per 1024-key block, one 1 KB row per table.
// Collision probability of two vectors at cosine rho, for Gaussian G (the coordinate pairs are
// i.i.d. standard bivariate normal with correlation rho):
//   p(rho) = 2d * int_{a>0} int_{b>0} phi_rho(a, b) F_rho(a, b)^(d-1) da db,
//   F_rho(a, b) = P[|X| < a, |Y| < b] = int_{-a}^{a} phi(t) [Phi((b - rho t)/s) - Phi((-b - rho t)/s)] dt,
// s = sqrt(1 - rho^2), by Gauss-Legendre quadrature on [0, 8] (96 nodes, 192 above |rho| = 0.95);
// above rho = 0.99 the density is too narrow for the quadrature and p runs linearly to p(1) = 1.
// The table of log u over the cosine that the attend kernel interpolates is built from it once
// (mp_cp_logu_table); the decode then runs the same attend kernel on that table.
#include <math.h>

#include "mp_internal.cuh"

namespace mp {

namespace {

constexpr int kCpKeys = 256;         // keys per encoding CTA, one per thread
constexpr int kCpOut = 16;           // projections a thread accumulates at once
constexpr int kCpThreads = 256;      // collide CTA
constexpr int kCpWarps = kCpThreads / 32;
constexpr int kCpQThreads = 128;     // query CTA: one thread per projection
constexpr int kCpQRows = 4;          // query rows per query CTA (<= the CTA's warps)
constexpr int kCpTableThreads = 256;
constexpr int kGlMax = 192;          // Gauss-Legendre nodes, at most
constexpr double kCpRhoMax = 0.99;

__device__ double g_gl_x[2][kGlMax];   // nodes on [-1, 1] for 96 and for 192 points
__device__ double g_gl_w[2][kGlMax];

// ---- keys -------------------------------------------------------------------------------------
// One CTA per (256-key tile, head): the centred keys in shared memory, then per table the
// transposed G_t (Gt[e][j]); each thread runs its key through the 128 projections, 16 at a time,
// keeping the first index of the largest |y| (the order an exact tie resolves to).
__global__ void __launch_bounds__(kCpKeys)
    encode_cp_kernel(const void* keys, int keys_bf16, const float* centre, const void* G,
                     int g_bf16, int ncap, int n0, int n1, int L, int cblk, uint8_t* codes) {
    extern __shared__ __align__(16) float sm[];
    float* Gt = sm;                               // [kD][kD]: Gt[e * kD + j] = G_t[j][e]
    float* kbar = sm + kD * kD;                   // [kCpKeys][kD + 1]
    const int bh = blockIdx.y, tid = threadIdx.x;
    const int i0 = (n0 / kCpKeys + blockIdx.x) * kCpKeys;
    for (int idx = tid; idx < kCpKeys * kD; idx += kCpKeys) {
        const int r = idx / kD, e = idx % kD, i = i0 + r;
        float v = 0.0f;
        if (i < ncap)
            v = load_elem(keys, keys_bf16, (static_cast<size_t>(bh) * ncap + i) * kD + e) -
                centre[static_cast<size_t>(bh) * kD + e];
        kbar[r * (kD + 1) + e] = v;
    }
    const int key = i0 + tid;
    const bool mine = key >= n0 && key < n1;     // n1 <= ncap: the byte exists
    uint8_t* dst = codes + (static_cast<size_t>(bh) * cblk + (mine ? key / kKeysPerBlock : 0)) *
                               L * kKeysPerBlock + key % kKeysPerBlock;
    for (int t = 0; t < L; ++t) {
        __syncthreads();                          // the previous table's Gt is consumed
        for (int idx = tid; idx < kD * kD; idx += kCpKeys) {
            const int j = idx / kD, e = idx % kD;   // coalesced along e in G
            Gt[e * kD + j] = load_elem(G, g_bf16, (static_cast<size_t>(t) * kD + j) * kD + e);
        }
        __syncthreads();
        float best = -1.0f;
        int code = 0;
        for (int j0 = 0; j0 < kD; j0 += kCpOut) {
            float y[kCpOut];
#pragma unroll
            for (int c = 0; c < kCpOut; ++c) y[c] = 0.0f;
            for (int e = 0; e < kD; ++e) {
                const float x = kbar[tid * (kD + 1) + e];
                const float4* g4 = reinterpret_cast<const float4*>(Gt + e * kD + j0);
#pragma unroll
                for (int c4 = 0; c4 < kCpOut / 4; ++c4) {
                    const float4 g = g4[c4];
                    y[4 * c4 + 0] = fmaf(g.x, x, y[4 * c4 + 0]);
                    y[4 * c4 + 1] = fmaf(g.y, x, y[4 * c4 + 1]);
                    y[4 * c4 + 2] = fmaf(g.z, x, y[4 * c4 + 2]);
                    y[4 * c4 + 3] = fmaf(g.w, x, y[4 * c4 + 3]);
                }
            }
#pragma unroll
            for (int c = 0; c < kCpOut; ++c) {
                const float ay = fabsf(y[c]);
                if (ay > best) {
                    best = ay;
                    code = 2 * (j0 + c) + (y[c] < 0.0f ? 1 : 0);
                }
            }
        }
        if (mine) dst[static_cast<size_t>(t) * kKeysPerBlock] = static_cast<uint8_t>(code);
    }
}

// ---- queries ----------------------------------------------------------------------------------
struct CpQArgs {
    const void* q;
    const void* G;
    const float* centre;
    uint8_t* qcodes;          // [rows][qbytes]
    float4* qstat;            // [rows] {|q|, q.mu}
    unsigned* counters;       // [rows], reset here
    int q_bf16, g_bf16, Hq, G_heads, L, qbytes, rows;
};

// One CTA per (table, group of kCpQRows query rows): G_t is staged in shared memory (rows padded
// to 129 floats) with coalesced loads; thread j computes (G_t q)_j for each row of the group, and
// per row the CTA keeps the first index of the largest |y|. The CTAs of table 0 also write |q|
// and q.mu and reset the merge counters of their rows.
__global__ void __launch_bounds__(kCpQThreads) qencode_cp_kernel(const CpQArgs a) {
    extern __shared__ __align__(16) float qsm[];
    float* Gs = qsm;                              // [kD][kD + 1]
    float* qs = qsm + kD * (kD + 1);              // [kCpQRows][kD]
    __shared__ float wbest[kCpQRows][kCpQThreads / 32];
    __shared__ int wcode[kCpQRows][kCpQThreads / 32];
    allow_dependents();                           // the scan may start meanwhile
    const int t = blockIdx.x, r0 = blockIdx.y * kCpQRows, j = threadIdx.x;
    const int lane = j & 31, warp = j >> 5;
    const int nr = min(kCpQRows, a.rows - r0);
    for (int idx = j; idx < kD * kD; idx += kCpQThreads)
        Gs[(idx / kD) * (kD + 1) + idx % kD] =
            load_elem(a.G, a.g_bf16, static_cast<size_t>(t) * kD * kD + idx);
    for (int idx = j; idx < kCpQRows * kD; idx += kCpQThreads)
        qs[idx] = idx < nr * kD ? load_elem(a.q, a.q_bf16, static_cast<size_t>(r0) * kD + idx)
                                : 0.0f;
    __syncthreads();
    float y[kCpQRows];
#pragma unroll
    for (int r = 0; r < kCpQRows; ++r) y[r] = 0.0f;
    for (int e = 0; e < kD; ++e) {
        const float g = Gs[j * (kD + 1) + e];
#pragma unroll
        for (int r = 0; r < kCpQRows; ++r) y[r] = fmaf(g, qs[r * kD + e], y[r]);
    }
#pragma unroll
    for (int r = 0; r < kCpQRows; ++r) {
        float best = fabsf(y[r]);
        int code = 2 * j + (y[r] < 0.0f ? 1 : 0);
#pragma unroll
        for (int o = 16; o; o >>= 1) {            // larger |y| wins, the smaller index on a tie
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int oc = __shfl_xor_sync(0xffffffffu, code, o);
            if (ob > best || (ob == best && oc < code)) {
                best = ob;
                code = oc;
            }
        }
        if (lane == 0) {
            wbest[r][warp] = best;
            wcode[r][warp] = code;
        }
    }
    __syncthreads();
    if (j < nr) {
        float b = wbest[j][0];
        int c = wcode[j][0];
        for (int w = 1; w < kCpQThreads / 32; ++w)
            if (wbest[j][w] > b || (wbest[j][w] == b && wcode[j][w] < c)) {
                b = wbest[j][w];
                c = wcode[j][w];
            }
        a.qcodes[static_cast<size_t>(r0 + j) * a.qbytes + t] = static_cast<uint8_t>(c);
    }
    if (t == 0 && warp < nr) {                    // warp r: |q| and q.mu of row r0 + r
        const int row = r0 + warp;
        const int b = row / a.Hq, h = row % a.Hq, Hkv = a.Hq / a.G_heads;
        const float* mu = a.centre + (static_cast<size_t>(b) * Hkv + h / a.G_heads) * kD;
        float nn = 0.0f, qm = 0.0f;
        for (int e = lane; e < kD; e += 32) {
            const float x = qs[warp * kD + e];
            nn = fmaf(x, x, nn);
            qm = fmaf(x, mu[e], qm);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            nn += __shfl_xor_sync(0xffffffffu, nn, o);
            qm += __shfl_xor_sync(0xffffffffu, qm, o);
        }
        if (lane == 0) {
            a.qstat[row] = make_float4(sqrtf(nn), qm, 0.0f, 0.0f);
            a.counters[row] = 0u;
        }
    }
}

// ---- collide + select -------------------------------------------------------------------------
struct CpCArgs {
    const uint8_t* codes;
    const uint8_t* qcodes;
    uint32_t* selmask;
    int n, nblk, cblk, blk0, Hq, Hkv, L, qbytes, n_sink, n_local;
};

// The 4 match bits of the bytes of a __vcmpeq4 result (0xff where equal), in bits 0-3.
__device__ __forceinline__ uint32_t byte_matches(uint32_t eq) {
    return ((eq & 0x01010101u) * 0x10204080u) >> 28;
}

// Per (1024-key block, sequence x KV head): warps split the tables, lane w takes keys
// [32 w, 32 w + 32) of the block (32 code bytes); per table and query head of the group a
// 32-bit match mask feeds the saturating counters (>= 1, >= 2); the warps' counters combine in a
// fixed order into S_h = [>= 2 tables] & valid & not T.
template <int G>
__global__ void __launch_bounds__(kCpThreads) collide_cp_kernel(const CpCArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint32_t* gebuf = reinterpret_cast<uint32_t*>(smem);                     // [8][2][G][32]
    uint8_t* qc = smem + kCpWarps * 2 * G * 32 * 4;                         // [G][L]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int blk = blockIdx.x + a.blk0, bg = blockIdx.y;
    const int b = bg / a.Hkv, g = bg % a.Hkv;
    const int row0 = b * a.Hq + g * G;
    allow_dependents();
    const uint8_t* base = a.codes + (static_cast<size_t>(bg) * a.cblk + blk) * a.L * kKeysPerBlock +
                          lane * 32;
    const int t0 = (a.L * warp) / kCpWarps, t1 = (a.L * (warp + 1)) / kCpWarps;
    // the codes are an input of the call: pull this warp's tables into L2 before the wait
    if ((lane & 3) == 0)
        for (int t = t0; t < t1; ++t)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(base + static_cast<size_t>(t) * kKeysPerBlock));
    wait_for_predecessor();                      // the query codes of this call
    for (int i = tid; i < G * a.L; i += kCpThreads)
        qc[i] = a.qcodes[static_cast<size_t>(row0 + i / a.L) * a.qbytes + i % a.L];
    __syncthreads();
    uint32_t ge1[G], ge2[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        ge1[h] = 0u;
        ge2[h] = 0u;
    }
    for (int t = t0; t < t1; ++t) {
        const uint4* p = reinterpret_cast<const uint4*>(base + static_cast<size_t>(t) * kKeysPerBlock);
        const uint4 c0 = __ldcs(p), c1 = __ldcs(p + 1);
        const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const uint32_t qq = static_cast<uint32_t>(qc[h * a.L + t]) * 0x01010101u;
            uint32_t m = 0u;
#pragma unroll
            for (int k = 0; k < 8; ++k) m |= byte_matches(__vcmpeq4(w[k], qq)) << (4 * k);
            ge2[h] |= ge1[h] & m;
            ge1[h] |= m;
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
        for (int ww = 0; ww < kCpWarps; ++ww) {
            const uint32_t a1 = gebuf[((ww * 2 + 0) * G + h) * 32 + w];
            const uint32_t a2 = gebuf[((ww * 2 + 1) * G + h) * 32 + w];
            g2 |= a2 | (g1 & a1);
            g1 |= a1;
        }
        const int key0 = blk * kKeysPerBlock + w * 32;
        const uint32_t valid = bits_below(a.n - key0);
        const uint32_t tm =
            (bits_below(a.n_sink - key0) | ~bits_below(a.n - a.n_local - key0)) & valid;
        a.selmask[(static_cast<size_t>(row0 + h) * a.nblk + blk) * 32 + w] = g2 & valid & ~tm;
    }
}

// ---- the log u table --------------------------------------------------------------------------
// p(rho) by the quadrature of the file comment; 4096 intervals of the cosine on [-1, 1] as the
// attend kernel expects, one CTA per entry, fp32 integrands summed in fp64.
__device__ double cp_quadrature(double rho, int set, int n, double* red) {
    const double s = sqrt(1.0 - rho * rho);
    const float rf = static_cast<float>(rho), inv_s = static_cast<float>(1.0 / s);
    double acc = 0.0;
    for (int pair = threadIdx.x; pair < n * n; pair += kCpTableThreads) {
        const int ia = pair / n, ib = pair % n;
        const double xa = (g_gl_x[set][ia] + 1.0) * 4.0, wa = g_gl_w[set][ia] * 4.0;
        const double xb = (g_gl_x[set][ib] + 1.0) * 4.0, wb = g_gl_w[set][ib] * 4.0;
        // F(a, b) = sum_k w_k a phi(t_k) [Phi((b - rho t)/s) - Phi((-b - rho t)/s)], t = a x_k
        float F = 0.0f;
        const float af = static_cast<float>(xa), bf = static_cast<float>(xb);
        for (int k = 0; k < n; ++k) {
            const float tk = static_cast<float>(g_gl_x[set][k]) * af;
            const float wk = static_cast<float>(g_gl_w[set][k]) * af;
            const float ph = 0.3989422804014327f * __expf(-0.5f * tk * tk);
            F += wk * ph * (normcdff((bf - rf * tk) * inv_s) - normcdff((-bf - rf * tk) * inv_s));
        }
        F = fminf(fmaxf(F, 0.0f), 1.0f);
        const double q = (xa * xa - 2.0 * rho * xa * xb + xb * xb) / (2.0 * s * s);
        const double dens = exp(-q) / (2.0 * 3.14159265358979323846 * s);
        acc += wa * wb * dens * pow(static_cast<double>(F), kD - 1);
    }
    red[threadIdx.x] = acc;
    __syncthreads();
    for (int o = kCpTableThreads / 2; o; o >>= 1) {
        if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
        __syncthreads();
    }
    const double p = 2.0 * kD * red[0];
    __syncthreads();
    return p;
}

__global__ void __launch_bounds__(kCpTableThreads) cp_logu_table_kernel(int K, int L, float* table) {
    __shared__ double red[kCpTableThreads];
    const int i = blockIdx.x;
    const double c = i >= kLogUTableIntervals ? 1.0 : -1.0 + 2.0 * i / kLogUTableIntervals;
    double p;
    if (c >= 1.0) {
        p = 1.0;
    } else if (c <= -1.0) {
        p = 0.0;
    } else if (c > kCpRhoMax) {
        const double p0 = cp_quadrature(kCpRhoMax, 1, 192, red);
        p = p0 + (1.0 - p0) * (c - kCpRhoMax) / (1.0 - kCpRhoMax);
    } else if (fabs(c) > 0.95) {
        p = cp_quadrature(c, 1, 192, red);
    } else {
        p = cp_quadrature(c, 0, 96, red);
    }
    if (threadIdx.x == 0) table[i] = log_inclusion_p(static_cast<float>(p), K, L);
}

// Gauss-Legendre nodes and weights on [-1, 1] by Newton's method on P_n (host, double).
void gauss_legendre(int n, double* x, double* w) {
    for (int i = 0; i < n; ++i) {
        double z = cos(3.14159265358979323846 * (i + 0.75) / (n + 0.5));
        double dp = 1.0;
        for (int it = 0; it < 100; ++it) {
            double p0 = 1.0, p1 = z;
            for (int k = 2; k <= n; ++k) {
                const double pk = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p0) / k;
                p0 = p1;
                p1 = pk;
            }
            dp = n * (z * p1 - p0) / (z * z - 1.0);
            const double dz = p1 / dp;
            z -= dz;
            if (fabs(dz) < 1e-15) break;
        }
        x[i] = z;
        w[i] = 2.0 / ((1.0 - z * z) * dp * dp);
    }
}

template <int G>
size_t collide_cp_smem(int L) {
    return static_cast<size_t>(kCpWarps) * 2 * G * 32 * 4 + static_cast<size_t>(G) * L;
}

typedef void (*CpCollideFn)(const CpCArgs);
CpCollideFn pick_collide_cp(int G, size_t* smem, int L) {
    switch (G) {
        case 1: *smem = collide_cp_smem<1>(L); return collide_cp_kernel<1>;
        case 2: *smem = collide_cp_smem<2>(L); return collide_cp_kernel<2>;
        case 4: *smem = collide_cp_smem<4>(L); return collide_cp_kernel<4>;
        case 8: *smem = collide_cp_smem<8>(L); return collide_cp_kernel<8>;
        default: return nullptr;
    }
}

}  // namespace

size_t cp_codes_bytes(int B, int Hkv, int n, int L) {
    if (B < 1 || Hkv < 1 || n < 1 || L < 1) return 0;
    const size_t nblk = (static_cast<size_t>(n) + kKeysPerBlock - 1) / kKeysPerBlock;
    return static_cast<size_t>(B) * Hkv * nblk * L * kKeysPerBlock;
}

struct GaussLegendreSets {
    double x[2][kGlMax], w[2][kGlMax];
    GaussLegendreSets() {
        gauss_legendre(96, x[0], w[0]);
        gauss_legendre(192, x[1], w[1]);
    }
};

cudaError_t launch_cp_logu_table(int K, int L, float* table, cudaStream_t st) {
    static const GaussLegendreSets gl;            // built once, thread-safe (a function static)
    cudaError_t e = cudaMemcpyToSymbolAsync(g_gl_x, gl.x, sizeof(gl.x), 0, cudaMemcpyHostToDevice,
                                            st);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbolAsync(g_gl_w, gl.w, sizeof(gl.w), 0, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return e;
    cp_logu_table_kernel<<<kLogUTableIntervals + 1, kCpTableThreads, 0, st>>>(K, L, table);
    return cudaGetLastError();
}

cudaError_t launch_encode_cp(const void* keys, bool keys_bf16, const float* centre, const void* G,
                             bool g_bf16, int B, int Hkv, int ncap, int n0, int n1, int L,
                             uint8_t* codes, cudaStream_t st) {
    if (n1 <= n0) return cudaSuccess;
    const int cblk = (ncap + kKeysPerBlock - 1) / kKeysPerBlock;
    const int tiles = (n1 - 1) / kCpKeys - n0 / kCpKeys + 1;
    const size_t smem = (static_cast<size_t>(kD) * kD + static_cast<size_t>(kCpKeys) * (kD + 1)) *
                        sizeof(float);
    encode_cp_kernel<<<dim3(tiles, B * Hkv), kCpKeys, smem, st>>>(
        keys, keys_bf16, centre, G, g_bf16, ncap, n0, n1, L, cblk, codes);
    return cudaGetLastError();
}

cudaError_t launch_qencode_cp(const void* q, bool q_bf16, const float* centre, const void* G,
                              bool g_bf16, const DecodeShape& s, const DecodeScratch& ws,
                              cudaStream_t st) {
    CpQArgs a;
    a.q = q;
    a.G = G;
    a.centre = centre;
    a.qcodes = reinterpret_cast<uint8_t*>(ws.qbits);
    a.qstat = ws.qstat;
    a.counters = ws.counters;
    a.q_bf16 = q_bf16;
    a.g_bf16 = g_bf16;
    a.Hq = s.Hq;
    a.G_heads = s.Hq / s.Hkv;
    a.L = s.L;
    a.qbytes = s.qwords * 4;
    a.rows = s.B * s.Hq;
    const size_t smem = (static_cast<size_t>(kD) * (kD + 1) + static_cast<size_t>(kCpQRows) * kD) *
                        sizeof(float);
    qencode_cp_kernel<<<dim3(s.L, (a.rows + kCpQRows - 1) / kCpQRows), kCpQThreads, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_collide_cp(const void* q, bool q_bf16, const uint8_t* codes,
                              const float* centre, const void* keys, const void* values,
                              bool kv_bf16, const DecodeShape& s, float* out,
                              const DecodeScratch& ws, cudaStream_t st, int blk0) {
    size_t smem = 0;
    CpCollideFn fn = pick_collide_cp(s.Hq / s.Hkv, &smem, s.L);
    if (!fn || smem > 48 * 1024) return cudaErrorNotSupported;
    CpCArgs a;
    a.codes = codes;
    a.qcodes = reinterpret_cast<const uint8_t*>(ws.qbits);
    a.selmask = ws.selmask;
    a.n = s.n;
    a.nblk = s.nblk;
    a.cblk = s.cblk;
    a.blk0 = blk0;
    a.Hq = s.Hq;
    a.Hkv = s.Hkv;
    a.L = s.L;
    a.qbytes = s.qwords * 4;
    a.n_sink = s.n_sink;
    a.n_local = s.n_local;
    if (blk0 < s.nblk) {
        const cudaError_t e = launch_dependent(fn, dim3(s.nblk - blk0, s.B * s.Hkv),
                                               dim3(kCpThreads), smem, st, a);
        if (e != cudaSuccess) return e;
    }
    return launch_attend(q, q_bf16, centre, keys, values, kv_bf16, s, out, ws, st);
}

cudaError_t prepare_cross_polytope() {
    cudaError_t e = cudaFuncSetAttribute(encode_cp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>((static_cast<size_t>(kD) * kD +
                                                           static_cast<size_t>(kCpKeys) * (kD + 1)) *
                                                          sizeof(float)));
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncSetAttribute(qencode_cp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>((static_cast<size_t>(kD) * (kD + 1) +
                                                    static_cast<size_t>(kCpQRows) * kD) *
                                                   sizeof(float)))) != cudaSuccess)
        return e;
    if ((e = cudaFuncGetAttributes(&fa, cp_logu_table_kernel)) != cudaSuccess) return e;
    for (int G : {1, 2, 4, 8}) {
        size_t sm = 0;
        if ((e = cudaFuncGetAttributes(&fa, pick_collide_cp(G, &sm, 1))) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace mp
