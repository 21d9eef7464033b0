// Host side of the C ABI declared in include/magicpig.h: argument checks (before any launch),
// workspace layout, kernel selection, and the device status word.
#include <math.h>

#include <algorithm>

#include <mutex>

#include "mp_internal.cuh"

namespace mp {

// One status word per device; kernels with bounded waits raise MP_ERR_TIMEOUT here, the index
// checks of the MP_CHECKS build MP_ERR_BOUNDS (with the first failed site in the second word).
__device__ int g_device_status[2];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mutex;
int* g_status_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
bool g_prepared[kMaxDevices] = {};

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

// First use on a device: resolve the status word's address, read the SM count, load every
// kernel and raise shared-memory limits, so that later calls (possibly inside a stream
// capture) only launch.
bool ensure_prepared() {
    const int dev = current_device();
    if (dev < 0) return false;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_prepared[dev]) return true;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return false;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    if (prepare_misc() != cudaSuccess || prepare_decode() != cudaSuccess ||
        prepare_buckets() != cudaSuccess || prepare_append() != cudaSuccess ||
        prepare_mips() != cudaSuccess || prepare_cross_polytope() != cudaSuccess)
        return false;
    prepare_encode_tc();   // failure only disables the tensor-core encoder
    cudaGetLastError();
    g_status_ptr[dev] = static_cast<int*>(p);
    g_sm_count[dev] = sms;
    g_prepared[dev] = true;
    return true;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool valid_dtype(mp_dtype t) { return t == MP_F32 || t == MP_BF16; }

bool fill_shape(int B, int Hq, int Hkv, int n, int d, const mp_params* prm, DecodeShape* s) {
    if (!prm) return false;
    if (B < 1 || Hq < 1 || Hkv < 1 || n < 1 || d < 1) return false;
    if (Hq % Hkv) return false;
    if (prm->K < 0 || prm->K > 32 || prm->L < 1 || prm->n_sink < 0 || prm->n_local < 0 ||
        (prm->flags & ~(MP_FLAG_MIPS | MP_FLAG_CROSS_POLYTOPE)) != 0u || !(prm->scale >= 0.0f))
        return false;
    // cross-polytope: one hash per table, the caller's log u table, not with the MIPS variant
    const bool cp = (prm->flags & MP_FLAG_CROSS_POLYTOPE) != 0u;
    if (cp && (prm->K != 1 || (prm->flags & MP_FLAG_MIPS) != 0u || !prm->logu_table ||
               (reinterpret_cast<uintptr_t>(prm->logu_table) & 3u)))
        return false;
    if (!cp && prm->logu_table) return false;
    // the MIPS variant needs the radii; without the flag there must be none
    if (((prm->flags & MP_FLAG_MIPS) != 0u) != (prm->radius != nullptr)) return false;
    if (prm->radius && (reinterpret_cast<uintptr_t>(prm->radius) & 3u)) return false;
    if (static_cast<long long>(prm->K) * prm->L > (1 << 20)) return false;
    if (prm->n_capacity < 0 || (prm->n_capacity > 0 && prm->n_capacity < n)) return false;
    if (prm->n_indexed < 0 || prm->n_indexed > n) return false;
    s->B = B;
    s->Hq = Hq;
    s->Hkv = Hkv;
    s->n = n;
    s->d = d;
    s->K = prm->K;
    s->L = prm->L;
    s->C = prm->K * prm->L;
    s->qwords = cp ? (prm->L + 3) / 4 : (s->C + 31) / 32;   // bits, or code bytes
    s->cpad = (s->C + 3) & ~3;
    s->nblk = (n + kKeysPerBlock - 1) / kKeysPerBlock;
    s->ncap = prm->n_capacity > 0 ? prm->n_capacity : n;
    s->cblk = (s->ncap + kKeysPerBlock - 1) / kKeysPerBlock;
    s->n_indexed = prm->n_indexed > 0 ? prm->n_indexed : n;
    s->radius = prm->radius;
    s->cp = cp;
    s->logu_ext = prm->logu_table;
    s->n_sink = prm->n_sink;
    s->n_local = prm->n_local;
    s->scale = prm->scale > 0.0f ? prm->scale : 1.0f / sqrtf(static_cast<float>(d));
    return true;
}

mp_status to_status(cudaError_t e) { return e == cudaSuccess ? MP_OK : MP_ERR_CUDA; }
}  // namespace

int* device_status_ptr() {
    const int dev = current_device();
    return dev < 0 ? nullptr : g_status_ptr[dev];
}
int device_sm_count() {
    const int dev = current_device();
    return dev < 0 || g_sm_count[dev] <= 0 ? 148 : g_sm_count[dev];
}

// Decode workspace, in order (each piece 256-byte aligned): query bits, query masks, query
// norms, the attend kernel's partials, merge counters, selection words, the bucketed lookup's
// >= 1 bitmap, the table of log u over the cosine.
namespace {
struct ScratchSizes {
    size_t qbits, qmask, qstat, pml, po, counters, sel, tab;
    int n_counters;
};
ScratchSizes scratch_sizes(const DecodeShape& s) {
    const size_t rows = static_cast<size_t>(s.B) * s.Hq;
    const size_t nsp = attend_partials(s.nblk);
    ScratchSizes z;
    z.qbits = align256(rows * s.qwords * 4);
    z.qmask = align256(rows * s.cpad * 4);
    z.qstat = align256(rows * 16);
    z.pml = align256(rows * nsp * 4);
    z.po = align256(rows * nsp * kD * 4);
    z.n_counters = static_cast<int>(rows);
    z.counters = align256(static_cast<size_t>(z.n_counters) * 4);
    z.sel = align256(rows * s.nblk * 32 * 4);
    z.tab = align256((kLogUTableIntervals + 1) * 4);
    return z;
}
}  // namespace

size_t decode_scratch_bytes(const DecodeShape& s, bool debug) {
    const ScratchSizes z = scratch_sizes(s);
    (void)debug;                                         // the debug path needs nothing more
    return z.qbits + z.qmask + z.qstat + 2 * z.pml + z.po + z.counters + 2 * z.sel + z.tab;
}

DecodeScratch carve_decode_scratch(void* ws, const DecodeShape& s, bool debug) {
    const ScratchSizes z = scratch_sizes(s);
    uint8_t* p = static_cast<uint8_t*>(ws);
    DecodeScratch d;
    d.qbits = reinterpret_cast<uint32_t*>(p);
    p += z.qbits;
    d.qmask = reinterpret_cast<uint32_t*>(p);
    p += z.qmask;
    d.qstat = reinterpret_cast<float4*>(p);
    p += z.qstat;
    d.pm = reinterpret_cast<float*>(p);
    p += z.pml;
    d.pl = reinterpret_cast<float*>(p);
    p += z.pml;
    d.po = reinterpret_cast<float*>(p);
    p += z.po;
    d.counters = reinterpret_cast<unsigned*>(p);
    d.n_counters = z.n_counters;
    p += z.counters;
    d.selmask = reinterpret_cast<uint32_t*>(p);
    p += z.sel;
    d.sel_ge1 = reinterpret_cast<uint32_t*>(p);
    p += z.sel;
    d.logu_tab = reinterpret_cast<float*>(p);
    (void)debug;
    return d;
}

// The query encoding and the scan + attend of the decode, for the SimHash codes or the
// cross-polytope ones.
cudaError_t query_encode(const void* q, bool q_bf16, const float* centre, const void* W,
                         bool w_bf16, const DecodeShape& s, const DecodeScratch& ws,
                         cudaStream_t st) {
    return s.cp ? launch_qencode_cp(q, q_bf16, centre, W, w_bf16, s, ws, st)
                : launch_qencode(q, q_bf16, centre, W, w_bf16, s, ws, st);
}

cudaError_t scan_and_attend(const void* q, bool q_bf16, const uint32_t* codes,
                            const float* centre, const void* keys, const void* values,
                            bool kv_bf16, const DecodeShape& s, float* out,
                            const DecodeScratch& ws, cudaStream_t st, int blk0 = 0) {
    return s.cp ? launch_collide_cp(q, q_bf16, reinterpret_cast<const uint8_t*>(codes), centre,
                                    keys, values, kv_bf16, s, out, ws, st, blk0)
                : launch_collide(q, q_bf16, codes, centre, keys, values, kv_bf16, s, out, ws, st,
                                 blk0);
}

}  // namespace mp

using namespace mp;

namespace mp {
mp_status validate_decode(const void* q, mp_dtype q_dtype, const uint32_t* codes,
                          const float* centre, const void* W, mp_dtype w_dtype, const void* keys,
                          const void* values, mp_dtype kv_dtype, int B, int Hq, int Hkv, int n,
                          int d, const mp_params* prm, const float* out, DecodeShape* s) {
    if (!fill_shape(B, Hq, Hkv, n, d, prm, s)) return MP_ERR_INVALID_ARG;
    if (!valid_dtype(q_dtype) || !valid_dtype(w_dtype) || !valid_dtype(kv_dtype))
        return MP_ERR_INVALID_ARG;
    if (!q || !centre || !keys || !values || !out) return MP_ERR_INVALID_ARG;
    if (s->C > 0 && (!codes || !W)) return MP_ERR_INVALID_ARG;
    if (!aligned(keys, 16) || !aligned(values, 16) || !aligned(out, 4) ||
        !aligned(centre, 16) || !aligned(q, q_dtype == MP_BF16 ? 2 : 4) ||
        (codes && !aligned(codes, 16)))
        return MP_ERR_INVALID_ARG;
    if (d != kD) return MP_ERR_UNSUPPORTED;
    if (!decode_supported(*s, kv_dtype == MP_BF16)) return MP_ERR_UNSUPPORTED;
    return MP_OK;
}
}  // namespace mp

static mp_status check_decode(const void* q, mp_dtype q_dtype, const uint32_t* codes,
                              const float* centre, const void* W, mp_dtype w_dtype,
                              const void* keys, const void* values, mp_dtype kv_dtype, int B,
                              int Hq, int Hkv, int n, int d, const mp_params* prm, float* out,
                              void* workspace, size_t ws_bytes, bool debug, DecodeShape* s) {
    const mp_status st = validate_decode(q, q_dtype, codes, centre, W, w_dtype, keys, values,
                                         kv_dtype, B, Hq, Hkv, n, d, prm, out, s);
    if (st != MP_OK) return st;
    if (!workspace || !aligned(workspace, 256)) return MP_ERR_INVALID_ARG;
    if (ws_bytes < decode_scratch_bytes(*s, debug)) return MP_ERR_WORKSPACE;
    return MP_OK;
}

extern "C" {

const char* mp_status_string(mp_status s) {
    switch (s) {
        case MP_OK: return "MP_OK";
        case MP_ERR_INVALID_ARG: return "MP_ERR_INVALID_ARG";
        case MP_ERR_UNSUPPORTED: return "MP_ERR_UNSUPPORTED";
        case MP_ERR_CUDA: return "MP_ERR_CUDA";
        case MP_ERR_TIMEOUT: return "MP_ERR_TIMEOUT";
        case MP_ERR_WORKSPACE: return "MP_ERR_WORKSPACE";
        case MP_ERR_BOUNDS: return "MP_ERR_BOUNDS";
        default: return "MP_UNKNOWN_STATUS";
    }
}

int mp_abi_version(void) { return MP_ABI_VERSION; }

size_t mp_codes_bytes(int B, int Hkv, int n, int K, int L) {
    if (B < 1 || Hkv < 1 || n < 1 || K < 0 || L < 1) return 0;
    const size_t nblk = (static_cast<size_t>(n) + kKeysPerBlock - 1) / kKeysPerBlock;
    return static_cast<size_t>(B) * Hkv * nblk * static_cast<size_t>(K) * L * kWordsPerBlock * 4;
}

size_t mp_key_mean_workspace_bytes(int B, int Hkv, int n, int d) {
    if (B < 1 || Hkv < 1 || n < 1 || d != kD) return 0;
    // partial column sums per row range, then one counter per head
    return align256(static_cast<size_t>(B) * Hkv * key_mean_splits(B * Hkv, n) * kD * 4 +
                    static_cast<size_t>(B) * Hkv * 4);
}

mp_status mp_key_mean(const void* keys, mp_dtype key_dtype, int B, int Hkv, int n, int d,
                      float* centre, void* workspace, size_t ws_bytes, cudaStream_t stream) {
    return mp_key_mean_cap(keys, key_dtype, B, Hkv, n, n, d, centre, workspace, ws_bytes, stream);
}

mp_status mp_key_mean_cap(const void* keys, mp_dtype key_dtype, int B, int Hkv, int n_capacity,
                          int n, int d, float* centre, void* workspace, size_t ws_bytes,
                          cudaStream_t stream) {
    if (!keys || !centre || !workspace || !valid_dtype(key_dtype)) return MP_ERR_INVALID_ARG;
    if (B < 1 || Hkv < 1 || n < 1 || d < 1 || n_capacity < n) return MP_ERR_INVALID_ARG;
    if (d != kD) return MP_ERR_UNSUPPORTED;
    if (!aligned(keys, 16) || !aligned(centre, 4) || !aligned(workspace, 256))
        return MP_ERR_INVALID_ARG;
    if (ws_bytes < mp_key_mean_workspace_bytes(B, Hkv, n, d)) return MP_ERR_WORKSPACE;
    if (!ensure_prepared()) return MP_ERR_CUDA;
    return to_status(launch_key_mean(keys, key_dtype == MP_BF16, B * Hkv, n_capacity, n, centre,
                                     static_cast<float*>(workspace), key_mean_splits(B * Hkv, n),
                                     stream));
}

mp_status mp_build_tables(const void* keys, mp_dtype key_dtype, const float* centre,
                          const void* W, mp_dtype w_dtype, int B, int Hkv, int n, int d, int K,
                          int L, uint32_t* codes, cudaStream_t stream) {
    if (n < 1) return MP_ERR_INVALID_ARG;
    return mp_encode_keys(keys, key_dtype, centre, W, w_dtype, B, Hkv, n, 0, n, d, K, L, codes,
                          stream);
}

mp_status mp_encode_keys(const void* keys, mp_dtype key_dtype, const float* centre,
                         const void* W, mp_dtype w_dtype, int B, int Hkv, int n_capacity,
                         int n_begin, int n_end, int d, int K, int L, uint32_t* codes,
                         cudaStream_t stream) {
    if (B < 1 || Hkv < 1 || n_capacity < 1 || d < 1 || K < 0 || K > 32 || L < 1)
        return MP_ERR_INVALID_ARG;
    if (n_begin < 0 || n_end > n_capacity || n_begin > n_end) return MP_ERR_INVALID_ARG;
    if (!valid_dtype(key_dtype) || !valid_dtype(w_dtype)) return MP_ERR_INVALID_ARG;
    if (d != kD) return MP_ERR_UNSUPPORTED;
    if (static_cast<long long>(K) * L > (1 << 20)) return MP_ERR_INVALID_ARG;
    if (K == 0 || n_begin == n_end) return MP_OK;   // nothing to encode
    if (!keys || !centre || !W || !codes) return MP_ERR_INVALID_ARG;
    if (!aligned(keys, 16) || !aligned(codes, 16) || !aligned(centre, 4) ||
        !aligned(W, w_dtype == MP_BF16 ? 2 : 4))
        return MP_ERR_INVALID_ARG;
    if (!ensure_prepared()) return MP_ERR_CUDA;
    const bool kbf = key_dtype == MP_BF16, wbf = w_dtype == MP_BF16;
    if (n_end - n_begin <= kAppendMaxKeys)
        return to_status(launch_encode_append(keys, kbf, centre, W, wbf, B, Hkv, n_capacity,
                                              n_begin, n_end, K, L, codes, stream));
    const int blk0 = n_begin / kKeysPerBlock;
    const int blk1 = (n_end + kKeysPerBlock - 1) / kKeysPerBlock;
    if (kbf && wbf) {
        const cudaError_t e = launch_encode_tc(keys, centre, W, B, Hkv, n_capacity, blk0, blk1,
                                               K, L, codes, device_status_ptr(), stream);
        if (e != cudaErrorNotSupported) return to_status(e);
        cudaGetLastError();
    }
    return to_status(launch_encode_simt(keys, kbf, centre, W, wbf, B, Hkv, n_capacity, blk0,
                                        blk1, K, L, codes, stream));
}

mp_status mp_key_radius(const void* keys, mp_dtype key_dtype, const float* centre, int B,
                        int Hkv, int n_capacity, int n, int d, float* radius,
                        cudaStream_t stream) {
    if (!keys || !centre || !radius || !valid_dtype(key_dtype)) return MP_ERR_INVALID_ARG;
    if (B < 1 || Hkv < 1 || n < 1 || d < 1 || n_capacity < n) return MP_ERR_INVALID_ARG;
    if (d != kD) return MP_ERR_UNSUPPORTED;
    if (!aligned(keys, 16) || !aligned(centre, 4) || !aligned(radius, 4))
        return MP_ERR_INVALID_ARG;
    if (!ensure_prepared()) return MP_ERR_CUDA;
    return to_status(launch_key_radius(keys, key_dtype == MP_BF16, centre, B * Hkv, n_capacity,
                                       n, radius, stream));
}

mp_status mp_encode_keys_mips(const void* keys, mp_dtype key_dtype, const float* centre,
                              const void* W_aug, mp_dtype w_dtype, const float* radius, int B,
                              int Hkv, int n_capacity, int n_begin, int n_end, int d, int K,
                              int L, uint32_t* codes, float* norms_scratch,
                              cudaStream_t stream) {
    if (B < 1 || Hkv < 1 || n_capacity < 1 || d < 1 || K < 0 || K > 32 || L < 1)
        return MP_ERR_INVALID_ARG;
    if (n_begin < 0 || n_end > n_capacity || n_begin > n_end) return MP_ERR_INVALID_ARG;
    if (!valid_dtype(key_dtype) || !valid_dtype(w_dtype)) return MP_ERR_INVALID_ARG;
    if (d != kD) return MP_ERR_UNSUPPORTED;
    if (static_cast<long long>(K) * L > (1 << 20)) return MP_ERR_INVALID_ARG;
    if (K == 0 || n_begin == n_end) return MP_OK;
    if (!keys || !centre || !W_aug || !radius || !codes) return MP_ERR_INVALID_ARG;
    if (!aligned(keys, 16) || !aligned(codes, 16) || !aligned(centre, 4) ||
        !aligned(radius, 4) || !aligned(W_aug, w_dtype == MP_BF16 ? 2 : 4) ||
        !aligned(norms_scratch, 4))
        return MP_ERR_INVALID_ARG;
    if (!ensure_prepared()) return MP_ERR_CUDA;
    if (norms_scratch && key_dtype == MP_BF16 && w_dtype == MP_BF16 &&
        n_end - n_begin > kAppendMaxKeys) {
        // whole blocks on the tensor cores: the norms of every key of those blocks first
        const int blk0 = n_begin / kKeysPerBlock;
        const int blk1 = (n_end + kKeysPerBlock - 1) / kKeysPerBlock;
        cudaError_t e = launch_key_radius(keys, true, centre, B * Hkv, n_capacity, n_end, nullptr,
                                          stream, norms_scratch, blk0 * kKeysPerBlock,
                                          std::min(blk1 * kKeysPerBlock, n_capacity));
        if (e != cudaSuccess) return MP_ERR_CUDA;
        e = launch_encode_tc(keys, centre, W_aug, B, Hkv, n_capacity, blk0, blk1, K, L, codes,
                             device_status_ptr(), stream, norms_scratch, radius);
        if (e != cudaErrorNotSupported) return to_status(e);
        cudaGetLastError();
    }
    return to_status(launch_encode_mips(keys, key_dtype == MP_BF16, centre, W_aug,
                                        w_dtype == MP_BF16, radius, B, Hkv, n_capacity, n_begin,
                                        n_end, K, L, codes, stream));
}

size_t mp_cp_codes_bytes(int B, int Hkv, int n, int L) { return cp_codes_bytes(B, Hkv, n, L); }

mp_status mp_cp_logu_table(int K, int L, int d, float* table, cudaStream_t stream) {
    if (K < 1 || L < 1 || !table || !aligned(table, 4)) return MP_ERR_INVALID_ARG;
    if (d != kD) return MP_ERR_UNSUPPORTED;
    if (!ensure_prepared()) return MP_ERR_CUDA;
    return to_status(launch_cp_logu_table(K, L, table, stream));
}

mp_status mp_encode_keys_cp(const void* keys, mp_dtype key_dtype, const float* centre,
                            const void* G, mp_dtype g_dtype, int B, int Hkv, int n_capacity,
                            int n_begin, int n_end, int d, int L, uint8_t* codes,
                            cudaStream_t stream) {
    if (B < 1 || Hkv < 1 || n_capacity < 1 || d < 1 || L < 1) return MP_ERR_INVALID_ARG;
    if (n_begin < 0 || n_end > n_capacity || n_begin > n_end) return MP_ERR_INVALID_ARG;
    if (!valid_dtype(key_dtype) || !valid_dtype(g_dtype)) return MP_ERR_INVALID_ARG;
    if (d != kD) return MP_ERR_UNSUPPORTED;
    if (n_begin == n_end) return MP_OK;
    if (!keys || !centre || !G || !codes) return MP_ERR_INVALID_ARG;
    if (!aligned(keys, 16) || !aligned(codes, 16) || !aligned(centre, 4) ||
        !aligned(G, g_dtype == MP_BF16 ? 2 : 4))
        return MP_ERR_INVALID_ARG;
    if (!ensure_prepared()) return MP_ERR_CUDA;
    if (key_dtype == MP_BF16 && g_dtype == MP_BF16 && n_end - n_begin > kAppendMaxKeys) {
        // whole 1024-key blocks on the tensor cores (a table is d hyperplanes of the encoder)
        const int blk0 = n_begin / kKeysPerBlock;
        const int blk1 = (n_end + kKeysPerBlock - 1) / kKeysPerBlock;
        const cudaError_t e = launch_encode_tc(keys, centre, G, B, Hkv, n_capacity, blk0, blk1, kD,
                                               L, reinterpret_cast<uint32_t*>(codes),
                                               device_status_ptr(), stream, nullptr, nullptr, true);
        if (e != cudaErrorNotSupported) return to_status(e);
        cudaGetLastError();
    }
    return to_status(launch_encode_cp(keys, key_dtype == MP_BF16, centre, G, g_dtype == MP_BF16,
                                      B, Hkv, n_capacity, n_begin, n_end, L, codes, stream));
}

size_t mp_decode_workspace_bytes(int B, int Hq, int Hkv, int n, int d, const mp_params* prm) {
    DecodeShape s;
    if (!fill_shape(B, Hq, Hkv, n, d, prm, &s)) return 0;
    return decode_scratch_bytes(s, false);
}

size_t mp_debug_workspace_bytes(int B, int Hq, int Hkv, int n, int d, const mp_params* prm) {
    DecodeShape s;
    if (!fill_shape(B, Hq, Hkv, n, d, prm, &s)) return 0;
    return decode_scratch_bytes(s, true);
}

mp_status mp_decode_attention(const void* q, mp_dtype q_dtype, const uint32_t* codes,
                              const float* centre, const void* W, mp_dtype w_dtype,
                              const void* keys, const void* values, mp_dtype kv_dtype, int B,
                              int Hq, int Hkv, int n, int d, const mp_params* prm, float* out,
                              void* workspace, size_t ws_bytes, cudaStream_t stream) {
    DecodeShape s;
    const mp_status st = check_decode(q, q_dtype, codes, centre, W, w_dtype, keys, values,
                                      kv_dtype, B, Hq, Hkv, n, d, prm, out, workspace, ws_bytes,
                                      false, &s);
    if (st != MP_OK) return st;
    if (!ensure_prepared()) return MP_ERR_CUDA;
    const DecodeScratch ws = carve_decode_scratch(workspace, s, false);
    cudaError_t e = query_encode(q, q_dtype == MP_BF16, centre, W, w_dtype == MP_BF16, s, ws,
                                 stream);
    if (e != cudaSuccess) return MP_ERR_CUDA;
    return to_status(scan_and_attend(q, q_dtype == MP_BF16, codes, centre, keys, values,
                                     kv_dtype == MP_BF16, s, out, ws, stream));
}

mp_status mp_encode_query(const void* q, mp_dtype q_dtype, const float* centre, const void* W,
                          mp_dtype w_dtype, int B, int Hq, int Hkv, int n, int d,
                          const mp_params* prm, void* workspace, size_t ws_bytes,
                          cudaStream_t stream) {
    DecodeShape s;
    if (!fill_shape(B, Hq, Hkv, n, d, prm, &s)) return MP_ERR_INVALID_ARG;
    if (!valid_dtype(q_dtype) || !valid_dtype(w_dtype)) return MP_ERR_INVALID_ARG;
    if (!q || !centre || !workspace || (s.C > 0 && !W)) return MP_ERR_INVALID_ARG;
    if (!aligned(q, q_dtype == MP_BF16 ? 2 : 4) || !aligned(centre, 16) ||
        !aligned(workspace, 256))
        return MP_ERR_INVALID_ARG;
    if (d != kD) return MP_ERR_UNSUPPORTED;
    if (ws_bytes < decode_scratch_bytes(s, false)) return MP_ERR_WORKSPACE;
    if (!ensure_prepared()) return MP_ERR_CUDA;
    const DecodeScratch ws = carve_decode_scratch(workspace, s, false);
    return to_status(query_encode(q, q_dtype == MP_BF16, centre, W, w_dtype == MP_BF16, s, ws,
                                  stream));
}

mp_status mp_sampled_attention(const void* q, mp_dtype q_dtype, const uint32_t* codes,
                               const float* centre, const void* keys, const void* values,
                               mp_dtype kv_dtype, int B, int Hq, int Hkv, int n, int d,
                               const mp_params* prm, float* out, void* workspace,
                               size_t ws_bytes, cudaStream_t stream) {
    DecodeShape s;
    // W is only read by the query encoding; q stands in for it in the shared checks
    const mp_status st = check_decode(q, q_dtype, codes, centre, q, MP_F32, keys, values,
                                      kv_dtype, B, Hq, Hkv, n, d, prm, out, workspace, ws_bytes,
                                      false, &s);
    if (st != MP_OK) return st;
    if (!ensure_prepared()) return MP_ERR_CUDA;
    const DecodeScratch ws = carve_decode_scratch(workspace, s, false);
    return to_status(scan_and_attend(q, q_dtype == MP_BF16, codes, centre, keys, values,
                                     kv_dtype == MP_BF16, s, out, ws, stream));
}

size_t mp_buckets_bytes(int B, int Hkv, int n, int K, int L) {
    return bucket_table_bytes(B, Hkv, n, K, L);
}

mp_status mp_build_buckets(const uint32_t* codes, int B, int Hkv, int n, int K, int L,
                           uint32_t* buckets, cudaStream_t stream) {
    return mp_build_buckets_cap(codes, B, Hkv, n, n, K, L, buckets, stream);
}

mp_status mp_build_buckets_cap(const uint32_t* codes, int B, int Hkv, int n_capacity, int n,
                               int K, int L, uint32_t* buckets, cudaStream_t stream) {
    if (B < 1 || Hkv < 1 || n < 1 || n_capacity < n || K < 0 || K > 32 || L < 1)
        return MP_ERR_INVALID_ARG;
    if (K > kMaxBucketBits) return MP_ERR_UNSUPPORTED;
    if (!buckets || (K > 0 && !codes)) return MP_ERR_INVALID_ARG;
    if ((codes && !aligned(codes, 16)) || !aligned(buckets, 4)) return MP_ERR_INVALID_ARG;
    if (!ensure_prepared()) return MP_ERR_CUDA;
    const int cblk = (n_capacity + kKeysPerBlock - 1) / kKeysPerBlock;
    return to_status(launch_bucket_build(codes, B, Hkv, cblk, n, K, L, buckets, stream));
}

mp_status mp_sampled_attention_buckets(const void* q, mp_dtype q_dtype, const uint32_t* buckets,
                                       const uint32_t* codes, const float* centre,
                                       const void* keys, const void* values, mp_dtype kv_dtype,
                                       int B, int Hq, int Hkv, int n, int d,
                                       const mp_params* prm, float* out, void* workspace,
                                       size_t ws_bytes, cudaStream_t stream) {
    if (!buckets) return MP_ERR_INVALID_ARG;
    DecodeShape s;
    // the buckets stand in for the codes, q for W, in the shared checks
    const mp_status st = check_decode(q, q_dtype, buckets, centre, q, MP_F32, keys, values,
                                      kv_dtype, B, Hq, Hkv, n, d, prm, out, workspace, ws_bytes,
                                      false, &s);
    if (st != MP_OK) return st;
    if (s.K > kMaxBucketBits || s.cp) return MP_ERR_UNSUPPORTED;
    // keys appended since the tables were built come from a scan of their code blocks
    const bool tail = s.n_indexed < s.n && s.C > 0;
    if (tail && (!codes || !aligned(codes, 16))) return MP_ERR_INVALID_ARG;
    if (!ensure_prepared()) return MP_ERR_CUDA;
    const DecodeScratch ws = carve_decode_scratch(workspace, s, false);
    cudaError_t e = launch_bucket_lookup(buckets, ws.qbits, s, ws.sel_ge1, ws.selmask, stream);
    if (e != cudaSuccess) return MP_ERR_CUDA;
    if (tail)
        return to_status(scan_and_attend(q, q_dtype == MP_BF16, codes, centre, keys, values,
                                         kv_dtype == MP_BF16, s, out, ws, stream,
                                         s.n_indexed / kKeysPerBlock));
    return to_status(launch_attend(q, q_dtype == MP_BF16, centre, keys, values,
                                   kv_dtype == MP_BF16, s, out, ws, stream));
}

mp_status mp_debug_select(const void* q, mp_dtype q_dtype, const uint32_t* codes,
                          const float* centre, const void* W, mp_dtype w_dtype, const void* keys,
                          const void* values, mp_dtype kv_dtype, int B, int Hq, int Hkv, int n,
                          int d, const mp_params* prm, float* out, uint32_t* q_bits,
                          int32_t* sel_idx, int32_t* sel_count, uint8_t* cnt, void* workspace,
                          size_t ws_bytes, cudaStream_t stream) {
    DecodeShape s;
    const mp_status st = check_decode(q, q_dtype, codes, centre, W, w_dtype, keys, values,
                                      kv_dtype, B, Hq, Hkv, n, d, prm, out, workspace, ws_bytes,
                                      true, &s);
    if (st != MP_OK) return st;
    if (!sel_idx || !sel_count || (s.qwords > 0 && !q_bits)) return MP_ERR_INVALID_ARG;
    if (s.cp && cnt) return MP_ERR_UNSUPPORTED;   // counts are for the SimHash codes only
    if (!ensure_prepared()) return MP_ERR_CUDA;
    DecodeScratch ws = carve_decode_scratch(workspace, s, true);
    if (s.qwords > 0) ws.qbits = q_bits;
    cudaError_t e = query_encode(q, q_dtype == MP_BF16, centre, W, w_dtype == MP_BF16, s, ws,
                                 stream);
    if (e != cudaSuccess) return MP_ERR_CUDA;
    e = scan_and_attend(q, q_dtype == MP_BF16, codes, centre, keys, values, kv_dtype == MP_BF16, s,
                        out, ws, stream);
    if (e != cudaSuccess) return MP_ERR_CUDA;
    e = launch_compact_selection(ws.selmask, s.B * s.Hq, s.n, s.nblk, s.n_sink, s.n_local,
                                 sel_idx, sel_count, stream);
    if (e != cudaSuccess) return MP_ERR_CUDA;
    if (cnt) {
        if (s.C == 0) {
            // no hyperplanes: every table agrees for every key
            const size_t total = static_cast<size_t>(s.B) * s.Hq * s.n;
            e = cudaMemsetAsync(cnt, s.L > 255 ? 255 : s.L, total, stream);
        } else {
            e = launch_collision_counts(codes, ws.qbits, s, cnt, stream);
        }
        if (e != cudaSuccess) return MP_ERR_CUDA;
    }
    return MP_OK;
}

mp_status mp_debug_select_buckets(const void* q, mp_dtype q_dtype, const uint32_t* buckets,
                                  const uint32_t* codes, const float* centre, const void* W,
                                  mp_dtype w_dtype, const void* keys, const void* values,
                                  mp_dtype kv_dtype, int B, int Hq, int Hkv, int n, int d,
                                  const mp_params* prm, float* out, uint32_t* q_bits,
                                  int32_t* sel_idx, int32_t* sel_count, void* workspace,
                                  size_t ws_bytes, cudaStream_t stream) {
    if (!buckets) return MP_ERR_INVALID_ARG;
    DecodeShape s;
    // the buckets stand in for the codes in the shared checks (the codes are checked below)
    const mp_status st = check_decode(q, q_dtype, buckets, centre, W, w_dtype, keys, values,
                                      kv_dtype, B, Hq, Hkv, n, d, prm, out, workspace, ws_bytes,
                                      true, &s);
    if (st != MP_OK) return st;
    if (s.K > kMaxBucketBits || s.cp) return MP_ERR_UNSUPPORTED;
    if (!sel_idx || !sel_count || (s.qwords > 0 && !q_bits)) return MP_ERR_INVALID_ARG;
    const bool tail = s.n_indexed < s.n && s.C > 0;
    if (tail && (!codes || !aligned(codes, 16))) return MP_ERR_INVALID_ARG;
    if (!ensure_prepared()) return MP_ERR_CUDA;
    DecodeScratch ws = carve_decode_scratch(workspace, s, true);
    if (s.qwords > 0) ws.qbits = q_bits;
    cudaError_t e = query_encode(q, q_dtype == MP_BF16, centre, W, w_dtype == MP_BF16, s, ws,
                                 stream);
    if (e != cudaSuccess) return MP_ERR_CUDA;
    e = launch_bucket_lookup(buckets, ws.qbits, s, ws.sel_ge1, ws.selmask, stream);
    if (e != cudaSuccess) return MP_ERR_CUDA;
    // the same kernels as mp_sampled_attention_buckets
    if (tail)
        e = scan_and_attend(q, q_dtype == MP_BF16, codes, centre, keys, values,
                            kv_dtype == MP_BF16, s, out, ws, stream, s.n_indexed / kKeysPerBlock);
    else
        e = launch_attend(q, q_dtype == MP_BF16, centre, keys, values, kv_dtype == MP_BF16, s,
                          out, ws, stream);
    if (e != cudaSuccess) return MP_ERR_CUDA;
    return to_status(launch_compact_selection(ws.selmask, s.B * s.Hq, s.n, s.nblk, s.n_sink,
                                              s.n_local, sel_idx, sel_count, stream));
}

mp_status mp_debug_log_inclusion(const float* cosines, int count, int K, int L, float* out,
                                 cudaStream_t stream) {
    if (count < 0 || K < 0 || K > 32 || L < 1) return MP_ERR_INVALID_ARG;
    if (count > 0 && (!cosines || !out || !aligned(cosines, 4) || !aligned(out, 4)))
        return MP_ERR_INVALID_ARG;
    if (!ensure_prepared()) return MP_ERR_CUDA;
    return to_status(launch_log_inclusion(cosines, count, K, L, out, stream));
}

mp_status mp_debug_wait_expiry(int limit_us, cudaStream_t stream) {
    if (limit_us < 1 || limit_us > 100000) return MP_ERR_INVALID_ARG;
    if (!ensure_prepared()) return MP_ERR_CUDA;
    int* status = device_status_ptr();
    if (!status) return MP_ERR_CUDA;
    return to_status(launch_wait_expiry(1000ull * static_cast<unsigned>(limit_us), status, stream));
}

mp_status mp_codes_unpack(const uint32_t* codes, int B, int Hkv, int n, int K, int L,
                          uint32_t* table_codes, cudaStream_t stream) {
    if (B < 1 || Hkv < 1 || n < 1 || K < 0 || K > 32 || L < 1 || !table_codes)
        return MP_ERR_INVALID_ARG;
    if (K > 0 && !codes) return MP_ERR_INVALID_ARG;
    if (!ensure_prepared()) return MP_ERR_CUDA;
    if (K == 0)
        return to_status(cudaMemsetAsync(table_codes, 0,
                                         static_cast<size_t>(B) * Hkv * n * L * 4, stream));
    return to_status(launch_codes_unpack(codes, B * Hkv, n, K, L, table_codes, stream));
}

mp_status mp_device_status(int* status) {
    if (!status) return MP_ERR_INVALID_ARG;
    if (!ensure_prepared()) return MP_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return MP_ERR_CUDA;
    int v[2] = {0, 0};
    if (cudaMemcpyFromSymbol(v, g_device_status, sizeof(v)) != cudaSuccess) return MP_ERR_CUDA;
    const int zero[2] = {0, 0};
    if (cudaMemcpyToSymbol(g_device_status, zero, sizeof(zero)) != cudaSuccess) return MP_ERR_CUDA;
    *status = v[0];
    return MP_OK;
}

mp_status mp_debug_check_report(int* enabled, int* site) {
    if (!enabled || !site) return MP_ERR_INVALID_ARG;
    if (!ensure_prepared()) return MP_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return MP_ERR_CUDA;
    int v[2] = {0, 0};
    if (cudaMemcpyFromSymbol(v, g_device_status, sizeof(v)) != cudaSuccess) return MP_ERR_CUDA;
    *enabled = MP_CHECKS;
    *site = v[0] == MP_ERR_BOUNDS ? v[1] : 0;
    return MP_OK;
}

}  // extern "C"
