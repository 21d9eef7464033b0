// Decode step: query encoding, then one fused kernel that streams the packed codes of a block
// of 1024 keys, selects the keys colliding with the query in >= 2 tables, gathers only those
// K/V rows, and folds them with importance weights into a partial softmax; the last block of
// each KV head merges the partials by log-sum-exp.
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
constexpr int kTFlag = 1 << 15;                     // list entry belongs to the exact set T
constexpr int kCombinePitch = 132;                  // floats per (warp, head) partial: o, m, l

// ------------------------------------------------------------------------------------------------
// Query encoding: qbit_j = [w_j . q > 0] (the query is not centred), |q| and q.mu for the cosine
// ------------------------------------------------------------------------------------------------
constexpr int kQPlanes = 64;    // hyperplanes per CTA
constexpr int kQRows = 32;      // query rows per CTA

struct QArgs {
    const void* q;
    const void* W;
    const float* centre;
    uint32_t* qbits;
    float4* qstat;
    unsigned* counters;
    int q_bf16, w_bf16, BHq, Hq, G, C, qwords, n_counters;
};

__global__ void __launch_bounds__(kThreads) qencode_kernel(const QArgs a) {
    __shared__ float Ws[kD][kQPlanes];
    __shared__ float Qs[kQRows][kD];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int j0 = blockIdx.x * kQPlanes, r0 = blockIdx.y * kQRows;
    const int nq = min(kQRows, a.BHq - r0);
    for (int idx = tid; idx < kD * kQPlanes; idx += kThreads) {
        const int e = idx / kQPlanes, c = idx % kQPlanes, j = j0 + c;
        Ws[e][c] = j < a.C ? load_elem(a.W, a.w_bf16, static_cast<size_t>(e) * a.C + j) : 0.0f;
    }
    for (int idx = tid; idx < nq * kD; idx += kThreads)
        Qs[idx / kD][idx % kD] = load_elem(a.q, a.q_bf16, static_cast<size_t>(r0) * kD + idx);
    __syncthreads();
    for (int pr = warp; pr < nq * 2; pr += kWarps) {
        const int qi = pr >> 1, wd = pr & 1, c = wd * 32 + lane, j = j0 + c;
        float s = 0.0f;
#pragma unroll 16
        for (int e = 0; e < kD; ++e) s = fmaf(Ws[e][c], Qs[qi][e], s);
        const uint32_t word = __ballot_sync(0xffffffffu, j < a.C && s > 0.0f);
        const int wi = (j0 >> 5) + wd;
        if (lane == 0 && wi < a.qwords)
            a.qbits[static_cast<size_t>(r0 + qi) * a.qwords + wi] = word;
    }
    if (blockIdx.x == 0) {
        const int Hkv = a.Hq / a.G;
        for (int qi = warp; qi < nq; qi += kWarps) {
            const int row = r0 + qi, b = row / a.Hq, h = row % a.Hq, g = h / a.G;
            const float* mu = a.centre + (static_cast<size_t>(b) * Hkv + g) * kD;
            float nn = 0.0f, qm = 0.0f;
            for (int e = lane; e < kD; e += 32) {
                const float x = Qs[qi][e];
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
// log u(p) = log P[Binomial(L, p^K) >= 2], stable in fp32: directly when L p^K >= 1/2, else as
// t_2 (1 + sum_{j>=3} t_j / t_2) with t_j the binomial terms. p <= 0 clamps to log(FLT_MIN).
// ------------------------------------------------------------------------------------------------
__device__ float log_inclusion(float p, int K, int L) {
    if (L < 2) return -INFINITY;
    float x, lx;
    if (K == 0) {
        x = 1.0f;
        lx = 0.0f;
    } else {
        if (!(p > 0.0f)) return kLogFltMin;
        lx = static_cast<float>(K) * logf(p);
        x = expf(lx);
    }
    const float Lf = static_cast<float>(L);
    if (Lf * x >= 0.5f) {
        if (x >= 1.0f) return 0.0f;
        const float l1 = log1pf(-x);
        const float u = 1.0f - expf(Lf * l1) - Lf * x * expf((Lf - 1.0f) * l1);
        return logf(fmaxf(u, 1.17549435e-38f));
    }
    const float l1 = log1pf(-x);
    const float r = x / (1.0f - x);
    float term = 1.0f, tot = 1.0f;
    for (int j = 2; j < L; ++j) {
        term *= static_cast<float>(L - j) / static_cast<float>(j + 1) * r;
        tot += term;
        if (term < 1e-9f * tot) break;
    }
    return logf(0.5f * Lf * (Lf - 1.0f)) + 2.0f * lx + (Lf - 2.0f) * l1 + logf(tot);
}

// ------------------------------------------------------------------------------------------------
// Fused collide -> select -> gather -> attend, one CTA per (1024-key block, sequence x KV head)
// ------------------------------------------------------------------------------------------------
struct CArgs {
    const uint32_t* codes;
    const uint32_t* qbits;
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
    uint32_t* selmask;
    int q_bf16, n, nblk, Hq, Hkv, K, L, C, qwords, n_sink, n_local;
    float scale;
};

template <typename KV>
__host__ __device__ constexpr int stage_rows() {
    return sizeof(KV) == 2 ? 64 : 32;   // 32 KB of K+V rows either way
}

__host__ __device__ constexpr size_t align16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

template <int G, typename KV>
__host__ __device__ size_t region_bytes(int C) {
    const size_t a = static_cast<size_t>(C) * G * 4;
    const size_t b = static_cast<size_t>(kWarps) * G * kCombinePitch * 4;
    return align16(a > b ? a : b);
}

template <int G, typename KV>
size_t collide_smem_bytes(int C) {
    return region_bytes<G, KV>(C) + 2 * align16(stage_rows<KV>() * kD * sizeof(KV)) +
           align16(G * kD * 4) + kD * 4 + align16(G * 32 * 4) + kKeysPerBlock * 4 +
           kKeysPerBlock * 2 + 16;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
    const uint2 raw = *reinterpret_cast<const uint2*>(p);
    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
    const float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
    return make_float4(a.x, a.y, b.x, b.y);
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

template <int G, typename KV>
__global__ void __launch_bounds__(kThreads) collide_attend_kernel(const CArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int CH = stage_rows<KV>();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int blk = blockIdx.x, bg = blockIdx.y;
    const int b = bg / a.Hkv, g = bg % a.Hkv;
    const int row0 = b * a.Hq + g * G;          // first query row of this KV head's group

    size_t off = 0;
    uint32_t* region = reinterpret_cast<uint32_t*>(smem + off);
    off += region_bytes<G, KV>(a.C);
    KV* stK = reinterpret_cast<KV*>(smem + off);
    off += align16(CH * kD * sizeof(KV));
    KV* stV = reinterpret_cast<KV*>(smem + off);
    off += align16(CH * kD * sizeof(KV));
    float* qf = reinterpret_cast<float*>(smem + off);
    off += align16(G * kD * 4);
    float* muf = reinterpret_cast<float*>(smem + off);
    off += kD * 4;
    uint32_t* sel = reinterpret_cast<uint32_t*>(smem + off);
    off += align16(G * 32 * 4);
    int* lidx = reinterpret_cast<int*>(smem + off);
    off += kKeysPerBlock * 4;
    uint16_t* lhm = reinterpret_cast<uint16_t*>(smem + off);
    off += kKeysPerBlock * 2;
    int* misc = reinterpret_cast<int*>(smem + off);
    uint32_t* qneg = region;                                  // phase 1: [C][G] match masks
    uint32_t* gebuf = reinterpret_cast<uint32_t*>(stK);       // phase 1 -> 2: warp counters
    float* cbuf = reinterpret_cast<float*>(region);           // end: [warp][G][132] partials

    // ---- prologue: query bits as XOR masks (0 where the query bit is 1), q and mu as floats
    for (int j = tid; j < a.C; j += kThreads) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const uint32_t w = a.qbits[static_cast<size_t>(row0 + h) * a.qwords + (j >> 5)];
            qneg[j * G + h] = ((w >> (j & 31)) & 1u) ? 0u : 0xffffffffu;
        }
    }
    for (int idx = tid; idx < G * kD; idx += kThreads)
        qf[idx] = load_elem(a.q, a.q_bf16, static_cast<size_t>(row0) * kD + idx);
    if (tid < kD) muf[tid] = a.centre[static_cast<size_t>(bg) * kD + tid];
    __syncthreads();

    // ---- phase 1: per 32-key word (lane), per table, match = AND_b (plane ^ qmask); keep
    //      bit-sliced saturating counters ge1 = (>= 1 match), ge2 = (>= 2 matches)
    uint32_t ge1[G], ge2[G];
    {
        const int t0 = (a.L * warp) / kWarps, t1 = (a.L * (warp + 1)) / kWarps;
        if (a.K == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                ge1[h] = (t1 - t0 >= 1) ? 0xffffffffu : 0u;
                ge2[h] = (t1 - t0 >= 2) ? 0xffffffffu : 0u;
            }
        } else {
            uint32_t acc[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                acc[h] = 0xffffffffu;
                ge1[h] = 0u;
                ge2[h] = 0u;
            }
            const uint32_t* cb = a.codes +
                                 (static_cast<size_t>(bg) * a.nblk + blk) * a.C * kWordsPerBlock +
                                 lane;
            const int jend = t1 * a.K;
            int bb = 0;
            for (int j = t0 * a.K; j < jend; j += 16) {
                uint32_t x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    x[i] = (j + i < jend) ? __ldcs(cb + static_cast<size_t>(j + i) * kWordsPerBlock)
                                          : 0u;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    if (j + i < jend) {
                        uint32_t qn[G];
                        load_qneg<G>(qneg + (j + i) * G, qn);
#pragma unroll
                        for (int h = 0; h < G; ++h) acc[h] &= x[i] ^ qn[h];
                        if (++bb == a.K) {
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
        sel[h * 32 + w] = s;
        if (a.selmask) a.selmask[(static_cast<size_t>(row0 + h) * a.nblk + blk) * 32 + w] = s;
    }
    __syncthreads();

    // ---- compaction: ascending list of the block's keys in S_h (any h) or in T
    if (warp == 0) {
        const int key0 = blk * kKeysPerBlock + lane * 32;
        const uint32_t valid = bits_below(a.n - key0);
        const uint32_t tm =
            (bits_below(a.n_sink - key0) | ~bits_below(a.n - a.n_local - key0)) & valid;
        uint32_t s[G];
        uint32_t U = tm;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            s[h] = sel[h * 32 + lane];
            U |= s[h];
        }
        const int c = __popc(U);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        int pos = incl - c;
        uint32_t bits = U;
        while (bits) {
            const int bit = __ffs(bits) - 1;
            bits &= bits - 1;
            int hm;
            if ((tm >> bit) & 1u) {
                hm = kTFlag | ((1 << G) - 1);
            } else {
                hm = 0;
#pragma unroll
                for (int h = 0; h < G; ++h) hm |= static_cast<int>((s[h] >> bit) & 1u) << h;
            }
            lidx[pos] = key0 + bit;
            lhm[pos] = static_cast<uint16_t>(hm);
            ++pos;
        }
        if (lane == 31) misc[0] = incl;
    }
    __syncthreads();
    const int nsel = misc[0];

    // ---- phase 2: gather the listed K/V rows, weight, online softmax per head
    float m[G], l[G];
    float4 o[G];
    float qn[G], qmu[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.0f;
        o[h] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        const float4 st = a.qstat[row0 + h];
        qn[h] = st.x;
        qmu[h] = st.y;
    }
    const float4 mu4 = reinterpret_cast<const float4*>(muf)[lane];
    const KV* Kb = reinterpret_cast<const KV*>(a.keys) + static_cast<size_t>(bg) * a.n * kD;
    const KV* Vb = reinterpret_cast<const KV*>(a.values) + static_cast<size_t>(bg) * a.n * kD;
    constexpr int P = kD * static_cast<int>(sizeof(KV)) / 16;   // 16-byte pieces per row
    for (int c0 = 0; c0 < nsel; c0 += CH) {
        const int nrow = min(CH, nsel - c0);
        for (int pc = tid; pc < nrow * 2 * P; pc += kThreads) {
            const int r = pc / (2 * P), rem = pc % (2 * P), arr = rem / P, piece = rem % P;
            const KV* src = (arr ? Vb : Kb) + static_cast<size_t>(lidx[c0 + r]) * kD;
            KV* dst = (arr ? stV : stK) + r * kD;
            cp_async16(reinterpret_cast<uint8_t*>(dst) + piece * 16,
                       reinterpret_cast<const uint8_t*>(src) + piece * 16);
        }
        cp_async_wait_all();
        __syncthreads();
        for (int r = warp; r < nrow; r += kWarps) {
            const float4 kf = load4(stK + r * kD + 4 * lane);
            const float4 vf = load4(stV + r * kD + 4 * lane);
            const float dx = kf.x - mu4.x, dy = kf.y - mu4.y, dz = kf.z - mu4.z, dw = kf.w - mu4.w;
            float kb2 = dx * dx + dy * dy + dz * dz + dw * dw;
            float dot[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float4 q4 = reinterpret_cast<const float4*>(qf)[h * 32 + lane];
                dot[h] = q4.x * kf.x + q4.y * kf.y + q4.z * kf.z + q4.w * kf.w;
            }
#pragma unroll
            for (int sh = 16; sh; sh >>= 1) {
                kb2 += __shfl_xor_sync(0xffffffffu, kb2, sh);
#pragma unroll
                for (int h = 0; h < G; ++h) dot[h] += __shfl_xor_sync(0xffffffffu, dot[h], sh);
            }
            const int hm = lhm[c0 + r];
            const float kbn = sqrtf(kb2);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                if (!((hm >> h) & 1)) continue;
                float lw = 0.0f;
                if (!(hm & kTFlag)) {
                    const float den = qn[h] * kbn;
                    float cs = den > 0.0f ? (dot[h] - qmu[h]) / den : 0.0f;
                    cs = fminf(1.0f, fmaxf(-1.0f, cs));
                    lw = log_inclusion(1.0f - acosf(cs) / kPi, a.K, a.L);
                }
                const float logit = dot[h] * a.scale - lw;
                const float mn = fmaxf(m[h], logit);
                const float corr = expf(m[h] - mn);
                const float pw = expf(logit - mn);
                l[h] = l[h] * corr + pw;
                o[h].x = o[h].x * corr + pw * vf.x;
                o[h].y = o[h].y * corr + pw * vf.y;
                o[h].z = o[h].z * corr + pw * vf.z;
                o[h].w = o[h].w * corr + pw * vf.w;
                m[h] = mn;
            }
        }
        __syncthreads();
    }

    // ---- merge the warps' partials into this block's partial (fixed order)
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float* dst = cbuf + (warp * G + h) * kCombinePitch;
        reinterpret_cast<float4*>(dst)[lane] = o[h];
        if (lane == 0) {
            dst[128] = m[h];
            dst[129] = l[h];
        }
    }
    __syncthreads();
    for (int x = tid; x < G * kD; x += kThreads) {
        const int h = x / kD, e = x % kD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, cbuf[(w * G + h) * kCombinePitch + 128]);
        float Ls = 0.0f, Os = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float* r = cbuf + (w * G + h) * kCombinePitch;
                const float s = expf(r[128] - M);
                Ls += s * r[129];
                Os += s * r[e];
            }
        }
        const size_t prow = static_cast<size_t>(row0 + h) * a.nblk + blk;
        a.po[prow * kD + e] = Os;
        if (e == 0) {
            a.pm[prow] = M;
            a.pl[prow] = Ls;
        }
    }

    // ---- the last block of this (sequence, KV head) merges all blocks' partials
    __threadfence();
    __syncthreads();
    if (tid == 0) misc[1] = (atomicAdd(a.counters + bg, 1u) == static_cast<unsigned>(a.nblk - 1));
    __syncthreads();
    if (!misc[1]) return;
    __threadfence();
    for (int x = tid; x < G * kD; x += kThreads) {
        const int h = x / kD, e = x % kD;
        const size_t base = static_cast<size_t>(row0 + h) * a.nblk;
        float M = -INFINITY;
        for (int j = 0; j < a.nblk; ++j) M = fmaxf(M, __ldcg(a.pm + base + j));
        float res = 0.0f;
        if (M != -INFINITY) {
            float Ls = 0.0f, Os = 0.0f;
            for (int j = 0; j < a.nblk; ++j) {
                const float s = expf(__ldcg(a.pm + base + j) - M);
                Ls += s * __ldcg(a.pl + base + j);
                Os += s * __ldcg(a.po + (base + j) * kD + e);
            }
            res = Os / Ls;
        }
        a.out[static_cast<size_t>(row0 + h) * kD + e] = res;
    }
    if (tid == 0) a.counters[bg] = 0u;
}

typedef void (*CollideFn)(const CArgs);

CollideFn pick(int G, bool kv_bf16) {
    switch (G) {
        case 1: return kv_bf16 ? collide_attend_kernel<1, __nv_bfloat16> : collide_attend_kernel<1, float>;
        case 2: return kv_bf16 ? collide_attend_kernel<2, __nv_bfloat16> : collide_attend_kernel<2, float>;
        case 4: return kv_bf16 ? collide_attend_kernel<4, __nv_bfloat16> : collide_attend_kernel<4, float>;
        case 8: return kv_bf16 ? collide_attend_kernel<8, __nv_bfloat16> : collide_attend_kernel<8, float>;
        default: return nullptr;
    }
}

size_t smem_for(int G, bool kv_bf16, int C) {
    switch (G) {
        case 1: return kv_bf16 ? collide_smem_bytes<1, __nv_bfloat16>(C) : collide_smem_bytes<1, float>(C);
        case 2: return kv_bf16 ? collide_smem_bytes<2, __nv_bfloat16>(C) : collide_smem_bytes<2, float>(C);
        case 4: return kv_bf16 ? collide_smem_bytes<4, __nv_bfloat16>(C) : collide_smem_bytes<4, float>(C);
        case 8: return kv_bf16 ? collide_smem_bytes<8, __nv_bfloat16>(C) : collide_smem_bytes<8, float>(C);
        default: return 0;
    }
}

constexpr size_t kMaxSmem = 232448;   // 227 KB opt-in per CTA

}  // namespace

bool decode_supported(const DecodeShape& s, bool kv_bf16) {
    const int G = s.Hq / s.Hkv;
    if (!pick(G, kv_bf16)) return false;
    return smem_for(G, kv_bf16, s.C) <= kMaxSmem;
}

cudaError_t prepare_decode() {
    const int Gs[4] = {1, 2, 4, 8};
    for (int i = 0; i < 4; ++i)
        for (int bf = 0; bf < 2; ++bf) {
            cudaError_t e = cudaFuncSetAttribute(pick(Gs[i], bf != 0),
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
    qa.qstat = ws.qstat;
    qa.counters = ws.counters;
    qa.q_bf16 = q_bf16;
    qa.w_bf16 = w_bf16;
    qa.BHq = s.B * s.Hq;
    qa.Hq = s.Hq;
    qa.G = s.Hq / s.Hkv;
    qa.C = s.C;
    qa.qwords = s.qwords;
    qa.n_counters = s.B * s.Hkv;
    const int gx = (s.C + kQPlanes - 1) / kQPlanes;
    const dim3 qgrid(gx > 0 ? gx : 1, (qa.BHq + kQRows - 1) / kQRows);
    qencode_kernel<<<qgrid, kThreads, 0, st>>>(qa);
    return cudaGetLastError();
}

cudaError_t launch_collide(const void* q, bool q_bf16, const uint32_t* codes,
                           const float* centre, const void* keys, const void* values,
                           bool kv_bf16, const DecodeShape& s, float* out,
                           const DecodeScratch& ws, cudaStream_t st) {
    const int G = s.Hq / s.Hkv;
    CArgs ca;
    ca.codes = codes;
    ca.qbits = ws.qbits;
    ca.qstat = ws.qstat;
    ca.q = q;
    ca.centre = centre;
    ca.keys = keys;
    ca.values = values;
    ca.pm = ws.pm;
    ca.pl = ws.pl;
    ca.po = ws.po;
    ca.counters = ws.counters;
    ca.out = out;
    ca.selmask = ws.selmask;
    ca.q_bf16 = q_bf16;
    ca.n = s.n;
    ca.nblk = s.nblk;
    ca.Hq = s.Hq;
    ca.Hkv = s.Hkv;
    ca.K = s.K;
    ca.L = s.L;
    ca.C = s.C;
    ca.qwords = s.qwords;
    ca.n_sink = s.n_sink;
    ca.n_local = s.n_local;
    ca.scale = s.scale;
    CollideFn fn = pick(G, kv_bf16);
    const size_t smem = smem_for(G, kv_bf16, s.C);
    if (!fn || smem > kMaxSmem) return cudaErrorNotSupported;
    fn<<<dim3(s.nblk, s.B * s.Hkv), kThreads, smem, st>>>(ca);
    return cudaGetLastError();
}

}  // namespace mp
