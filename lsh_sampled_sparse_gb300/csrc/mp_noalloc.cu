// mp_decode_attention_noalloc: the decode step for callers that cannot allocate device memory.
//
// Some callers are not allowed to allocate: they run inside a framework or runtime that owns
// every byte of device memory through its own pool and forbids cudaMalloc from plugins, or in a
// latency-critical loop where an allocation (which may synchronise the device) is not
// acceptable, or simply hold no handle to an allocator when they call this library. This entry
// point runs the same two kernels as mp_decode_attention, but its scratch (query bits, per-block
// partial softmax states, merge counters) lives in the fixed array below instead of a
// caller-provided workspace. Nothing here calls cudaMalloc, cudaFree or any allocating routine.
//
// The array is MP_NOALLOC_SCRATCH_BYTES large and stays resident on every GPU that loads the
// library until the process exits. Shapes whose scratch would not fit are rejected with
// MP_ERR_WORKSPACE before anything is launched. All calls on a device share the one array and
// it keeps whatever the last call left: the merge counters, the only part that must start at
// zero, are reset by the query-encoding kernel at the start of every call, and everything else
// is written before it is read. Calls whose kernels overlap on the GPU (different streams, or
// different host threads without ordering) race on the array and must be serialised by the
// caller.
#include <mutex>

#include "mp_internal.cuh"

namespace mp {
namespace {

constexpr size_t kScratchBytes = MP_NOALLOC_SCRATCH_BYTES;

// The scratch itself. In host code its name is only a stand-in for the symbol, not a device
// address; the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Per-device set-up on the first call with that device current: resolve the array's device
// address and load/configure the decode kernels. Returns nullptr if either fails.
void* scratch_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        if (prepare_misc() != cudaSuccess || prepare_decode() != cudaSuccess) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace
}  // namespace mp

extern "C" mp_status mp_decode_attention_noalloc(
    const void* q, mp_dtype q_dtype, const uint32_t* codes, const float* centre, const void* W,
    mp_dtype w_dtype, const void* keys, const void* values, mp_dtype kv_dtype, int B, int Hq,
    int Hkv, int n, int d, const mp_params* prm, float* out, cudaStream_t stream) {
    using namespace mp;
    // the same checks as mp_decode_attention, on the same shape description
    DecodeShape s;
    const mp_status st = validate_decode(q, q_dtype, codes, centre, W, w_dtype, keys, values,
                                         kv_dtype, B, Hq, Hkv, n, d, prm, out, &s);
    if (st != MP_OK) return st;
    if (s.cp) return MP_ERR_UNSUPPORTED;   // its query encoding and scan are not wired here
    const size_t need = decode_scratch_bytes(s, false);
    if (need > kScratchBytes) return MP_ERR_WORKSPACE;   // larger than the built-in scratch
    void* base = scratch_address();
    if (!base) return MP_ERR_CUDA;
    const DecodeScratch ws = carve_decode_scratch(base, s, false);
    cudaError_t e = launch_qencode(q, q_dtype == MP_BF16, centre, W, w_dtype == MP_BF16, s, ws,
                                   stream);
    if (e != cudaSuccess) return MP_ERR_CUDA;
    e = launch_collide(q, q_dtype == MP_BF16, codes, centre, keys, values, kv_dtype == MP_BF16, s,
                       out, ws, stream);
    return e == cudaSuccess ? MP_OK : MP_ERR_CUDA;
}
