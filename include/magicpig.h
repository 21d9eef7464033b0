/*
 * magicpig.h -- C ABI of libmagicpig, LSH-sampled decode attention on one GB300 (sm_103a).
 *
 * The method is MagicPIG's ("MagicPIG: LSH Sampling for Efficient LLM Generation", method
 * details; "MagicPIG: don't pick the tallest", section 5): keys are centred and SimHash-encoded
 * into L tables of K bits; a decode query keeps the keys whose code equals its own in at least
 * two tables, weights each kept key by its closed-form inclusion probability u, and merges that
 * self-normalised importance-sampled attention with exact attention over the sink and local
 * tokens. Everything stays in device memory; every step runs in this library's CUDA kernels.
 *
 * Conventions for every entry point below:
 *   - Pointers to tensors are DEVICE pointers owned by the caller. Nothing here allocates device
 *     memory; scratch comes from a caller-provided workspace whose size a *_workspace_bytes
 *     function returns. Workspace pointers must be 256-byte aligned.
 *   - Tensors are contiguous, row-major:
 *       keys, values  [B][Hkv][n_cap][d]   (MP_BF16 or MP_F32); n_cap = n unless a call takes
 *                                          a capacity (mp_params.n_capacity, or an n_capacity
 *                                          argument): a cache allocated for n_cap tokens per
 *                                          head of which the first n are in use
 *       q             [B][Hq][d]           (MP_BF16 or MP_F32)
 *       out           [B][Hq][d]           float32
 *       centre        [B][Hkv][d]          float32  (mu, the mean key of each head)
 *       W             [d][K*L]             (MP_BF16 or MP_F32); column j = t*K + b is bit b
 *                                          (least significant first) of table t. One W serves
 *                                          every head and layer.
 *   - GQA: query head h reads KV head h / (Hq / Hkv); Hq must be a multiple of Hkv.
 *   - d must be 128. 0 <= K <= 32 and 1 <= L; K == 0 is the degenerate case where every key
 *     collides in every table (u = 1 when L >= 2).
 *   - Packed codes ("codes") are bit-sliced in blocks of 1024 keys: for head (b, g) and block
 *     blk = i / 1024, plane j (= t*K + b) is a row of 32 uint32 words, and bit (i % 32) of word
 *     (i % 1024) / 32 holds the sign bit of key i for hyperplane j. Layout:
 *       codes[((b*Hkv + g)*nblk + blk)*(K*L) + j][w],   nblk = ceil(n_cap / 1024).
 *     Bits of positions i >= n (padding, or capacity not yet in use) are unspecified.
 *   - Calls are asynchronous on `stream`: argument checks run on the host and return an error
 *     before anything is launched; device-side problems (a bounded wait that gave up) set a
 *     device status word that mp_device_status() reads.
 *   - No global mutable state besides that status word; calls on different streams may run
 *     concurrently if their buffers do not overlap.
 */
#ifndef MAGICPIG_H
#define MAGICPIG_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MP_API __attribute__((visibility("default")))
#else
#define MP_API
#endif

#define MP_ABI_VERSION 6
#define MP_KEYS_PER_BLOCK 1024

typedef enum {
    MP_OK = 0,
    MP_ERR_INVALID_ARG = 1,   /* bad shape, null pointer, misalignment, inconsistent sizes */
    MP_ERR_UNSUPPORTED = 2,   /* a valid request the library does not implement (e.g. d != 128) */
    MP_ERR_CUDA = 3,          /* a CUDA runtime call failed; cudaGetLastError() has the cause */
    MP_ERR_TIMEOUT = 4,       /* a device-side bounded wait gave up (see mp_device_status) */
    MP_ERR_WORKSPACE = 5,     /* the workspace passed is smaller than *_workspace_bytes */
    MP_ERR_BOUNDS = 6         /* an index check of the MP_CHECKS build failed (see
                                 mp_debug_check_report); never raised by the product build */
} mp_status;

typedef enum { MP_F32 = 0, MP_BF16 = 1 } mp_dtype;

/* Decode parameters. K, L: LSH bits per table and tables ("LSH Sampling...", method details,
 * hash-function choice). n_sink, n_local: the exact set T = {0..n_sink-1} u {n-n_local..n-1},
 * attended with u = 1 and never sampled (Algorithm 1's static cache; "don't pick the tallest",
 * section 5). scale: score scale, 0 means 1/sqrt(d). flags: 0, MP_FLAG_MIPS or
 * MP_FLAG_CROSS_POLYTOPE.
 * n_capacity: tokens per head the keys, values and codes are laid out for (0 means n; else
 * n_capacity >= n). A decode cache that grows by appending (mp_encode_keys) keeps one
 * n_capacity for its lifetime and passes the current length as n.
 * n_indexed: keys [0, n_indexed) of each head are in the bucketed tables (0 means n; else
 * n_indexed <= n); only mp_sampled_attention_buckets reads it.
 * radius: with MP_FLAG_MIPS, [B][Hkv] float32 device array from mp_key_radius (the longest
 * centred key of each head); NULL otherwise.
 * logu_table: with MP_FLAG_CROSS_POLYTOPE, the MP_LOGU_TABLE_ENTRIES floats of mp_cp_logu_table
 * for this K and L; NULL otherwise. */
typedef struct {
    int K;
    int L;
    int n_sink;
    int n_local;
    float scale;
    unsigned flags;
    int n_capacity;
    int n_indexed;
    const float* radius;
    const float* logu_table;
} mp_params;

/* MIPS -> cosine variant ("LSH Sampling...", method details, variance reduction with LSH): the
 * query is extended by a 0 and each centred key k - mu by sqrt(r^2 - |k - mu|^2), r the longest
 * centred key, so the collision probability grows with the inner product: p_i = 1 -
 * arccos(q.(k_i - mu) / (|q| r)) / pi replaces the cosine of q and k_i - mu. W then has d + 1
 * rows ([d + 1][K*L]; the query uses the first d), the codes come from mp_encode_keys_mips, and
 * every decode call of the variant sets this flag and mp_params.radius. */
#define MP_FLAG_MIPS 1u

/* Cross-polytope variant (the hash "LSH Sampling..." names in its conclusion as the way to shrink
 * the tables): table t hashes x to the signed index of the largest |coordinate| of G_t x, G_t a
 * d x d matrix of i.i.d. N(0, 1) entries, code = 2 i + (1 if negative), one byte (d = 128); keys
 * are centred, the query is not; one hash per table (K must be 1). W is then G: [L][d][d], row j
 * of G_t at (t * d + j) * d. Codes are bytes [B][Hkv][ceil(n_cap/1024)][L][1024] (mp_cp_codes_bytes,
 * written by mp_encode_keys_cp). p_i is the collision probability of two vectors at the cosine
 * of q and k_i - mu for Gaussian G, p(rho) = 2d int int_{a,b>0} phi_rho(a,b) P[|X|<a, |Y|<b]^(d-1),
 * which has no closed form: the decode reads log u from mp_params.logu_table, built once by
 * mp_cp_logu_table (Gauss-Legendre quadrature; above rho = 0.99 p runs linearly to p(1) = 1).
 * Not with the MIPS variant, the bucketed tables or mp_decode_attention_noalloc
 * (MP_ERR_UNSUPPORTED there), and mp_debug_select gives no collision counts for it. */
#define MP_FLAG_CROSS_POLYTOPE 2u
#define MP_LOGU_TABLE_ENTRIES 4097

/* Human-readable name of a status code (static storage). */
MP_API const char* mp_status_string(mp_status s);

/* MP_ABI_VERSION of the loaded library. */
MP_API int mp_abi_version(void);

/* Bytes of packed codes for B*Hkv heads of n keys: B*Hkv*ceil(n/1024)*K*L*128. */
MP_API size_t mp_codes_bytes(int B, int Hkv, int n, int K, int L);

/* Workspace bytes mp_key_mean needs: fixed-order partial sums plus one counter per head (the
 * call clears the counters itself; the workspace needs no initial contents). */
MP_API size_t mp_key_mean_workspace_bytes(int B, int Hkv, int n, int d);

/* Centre of the cached keys: centre[b][g][:] = (1/n) sum_i keys[b][g][i][:], float32
 * accumulation in a fixed order (run-to-run identical).
 * ("LSH Sampling...", method details, data preprocessing and centering: keys are centred before
 * the tables are built; "don't pick the tallest", section 5.)
 * One kernel: each CTA sums a range of rows (1024, halved down to 64 while the B*Hkv heads
 * would have fewer than 608 ranges, a function of B*Hkv and n only), the last CTA of a head adds
 * the ranges in order. Errors: MP_ERR_INVALID_ARG for n < 1, null pointers; MP_ERR_WORKSPACE if
 * ws_bytes is short. */
MP_API mp_status mp_key_mean(const void* keys, mp_dtype key_dtype, int B, int Hkv, int n, int d,
                             float* centre, void* workspace, size_t ws_bytes,
                             cudaStream_t stream);

/* mp_key_mean over the first n keys of a cache laid out for n_capacity tokens per head
 * (n <= n_capacity); the workspace is mp_key_mean_workspace_bytes(B, Hkv, n, d). */
MP_API mp_status mp_key_mean_cap(const void* keys, mp_dtype key_dtype, int B, int Hkv,
                                 int n_capacity, int n, int d, float* centre, void* workspace,
                                 size_t ws_bytes, cudaStream_t stream);

/* Build the hash tables of one layer: centre each key, project it on the K*L hyperplanes of W,
 * keep the sign (bit = 1 iff w_j.(k_i - mu) > 0), pack into the bit-sliced codes above.
 * ("LSH Sampling...", background, LSH basics: Sign(w^T x); method details, hash-function choice
 * and system co-design item 2: the random projection runs on the GPU.)
 * bf16 keys with a bf16 W run on the tcgen05 tensor cores (exact products, fp32 accumulation);
 * other dtype pairs use an fp32 CUDA-core kernel.
 * codes: mp_codes_bytes(B, Hkv, n, K, L) bytes, 16-byte aligned; may be NULL when K == 0.
 * Errors: MP_ERR_INVALID_ARG (shapes, null, misalignment), MP_ERR_UNSUPPORTED (d != 128). */
MP_API mp_status mp_build_tables(const void* keys, mp_dtype key_dtype, const float* centre,
                                 const void* W, mp_dtype w_dtype, int B, int Hkv, int n, int d,
                                 int K, int L, uint32_t* codes, cudaStream_t stream);

/* Encode keys [n_begin, n_end) of every head of a cache laid out for n_capacity tokens per head
 * into codes laid out for n_capacity (mp_codes_bytes(B, Hkv, n_capacity, K, L) bytes), with a
 * given centre. This is the incremental append of decode tokens: after a build over the prompt
 * (mp_key_mean_cap + mp_encode_keys(0, n)), each new token's key is written to the cache at
 * position n and encoded with mp_encode_keys(n, n + 1); the next decode passes n + 1. The local
 * window of T slides with n, so the key that leaves it joins the sampled keys with the code it
 * got when it was appended. The centre stays the one of the build: the pages compute it once,
 * before the tables are built ("LSH Sampling...", method details, data preprocessing and
 * centering) and say nothing of updates; codes and the weights p_i both use the centre the
 * caller passes, so any fixed centre gives a consistent sampler, and refreshing it means a
 * rebuild (mp_key_mean_cap, then mp_encode_keys over [0, n)).
 * Bits of keys outside [n_begin, n_end) that share a 32-key word with the range are kept. Short
 * ranges (up to 64 keys) run on CUDA cores; longer ones re-encode whole 1024-key blocks (bf16
 * keys and W: tensor cores), which rewrites the blocks' other keys with their own codes again.
 * Errors: MP_ERR_INVALID_ARG (shapes, n_begin < 0, n_end > n_capacity, n_begin > n_end, null,
 * misalignment), MP_ERR_UNSUPPORTED (d != 128). An empty range does nothing. */
MP_API mp_status mp_encode_keys(const void* keys, mp_dtype key_dtype, const float* centre,
                                const void* W, mp_dtype w_dtype, int B, int Hkv, int n_capacity,
                                int n_begin, int n_end, int d, int K, int L, uint32_t* codes,
                                cudaStream_t stream);

/* Workspace bytes mp_decode_attention (and its two halves below) need for these shapes;
 * 0 if the shapes or parameters are invalid. */
MP_API size_t mp_decode_workspace_bytes(int B, int Hq, int Hkv, int n, int d,
                                        const mp_params* prm);

/* One decode step of LSH-sampled attention for B*Hq query rows (Algorithm 1 of "LSH
 * Sampling...", method details, algorithm execution):
 *   q_code = Encode(q, W)                              (q is not centred)
 *   cnt_i  = #{t : code_t(k_i) == code_t(q)}           from the packed codes
 *   S      = {i not in T : cnt_i >= 2}
 *   p_i    = 1 - arccos(q.(k_i - mu) / (|q| |k_i - mu|)) / pi
 *   u_i    = 1 - (1 - p_i^K)^L - L p_i^K (1 - p_i^K)^(L-1)
 *   out    = softmax([s_S - log u_S, s_T]) . [V_S, V_T],   s = scale * q.k_i  (raw keys)
 * log u is a closed form, evaluated in fp32 in the log domain: directly when L p^K >= 0.05, else
 * as the binomial tail series from its second term. The query encoding tabulates it per call at
 * the 4097 cosines -1 + 2 i / 4096; a selected key takes the linear interpolation of that table
 * wherever the chord of its interval lies within 2e-5 of the closed form at the interval's
 * midpoint, and the closed form itself elsewhere (mp_debug_log_inclusion returns exactly this
 * evaluation). The softmax over S and T is computed in pieces of 1024 keys and
 * merged by log-sum-exp (the "recursive attention" merge of the system co-design section). If S
 * and T are both empty the output row is zero. Zero-length q or k - mu gives cosine 0 (p = 1/2).
 * A query row with a NaN or infinite element gets a NaN output row; the other rows are unaffected
 * and the status word is not raised.
 * Errors: MP_ERR_INVALID_ARG (shapes, null, Hq % Hkv, n_sink/n_local < 0, flags other than
 *         MP_FLAG_MIPS or MP_FLAG_CROSS_POLYTOPE, or a flag without its radius / log u table),
 *         MP_ERR_UNSUPPORTED (d != 128, Hq/Hkv not in {1, 2, 4, 8}, or K*L*(Hq/Hkv) so
 *         large that a CTA's query masks no longer fit in shared memory),
 *         MP_ERR_WORKSPACE (ws_bytes < mp_decode_workspace_bytes). */
MP_API mp_status mp_decode_attention(const void* q, mp_dtype q_dtype, const uint32_t* codes,
                                     const float* centre, const void* W, mp_dtype w_dtype,
                                     const void* keys, const void* values, mp_dtype kv_dtype,
                                     int B, int Hq, int Hkv, int n, int d, const mp_params* prm,
                                     float* out, void* workspace, size_t ws_bytes,
                                     cudaStream_t stream);

/* The two halves of mp_decode_attention, for callers that schedule or time them apart. Both
 * take the same workspace; mp_sampled_attention reads what mp_encode_query wrote there for the
 * same q, centre and shapes, so the two must run in that order on the same stream.
 *
 * mp_encode_query: q_code = Encode(q, W), plus |q| and q.mu (Algorithm 1's first step).
 * mp_sampled_attention: collision counts, S, gather of K_S and V_S, importance weights, and the
 * merged softmax with the exact set T (Algorithm 1's remaining steps).
 * Errors as mp_decode_attention. */
MP_API mp_status mp_encode_query(const void* q, mp_dtype q_dtype, const float* centre,
                                 const void* W, mp_dtype w_dtype, int B, int Hq, int Hkv, int n,
                                 int d, const mp_params* prm, void* workspace, size_t ws_bytes,
                                 cudaStream_t stream);
MP_API mp_status mp_sampled_attention(const void* q, mp_dtype q_dtype, const uint32_t* codes,
                                      const float* centre, const void* keys, const void* values,
                                      mp_dtype kv_dtype, int B, int Hq, int Hkv, int n, int d,
                                      const mp_params* prm, float* out, void* workspace,
                                      size_t ws_bytes, cudaStream_t stream);

/* ---- Bucketed hash tables ---------------------------------------------------------------------
 * The retrieval structure of the pages: per table, the keys of each K-bit code ("LSH Sampling...",
 * system co-design item 3: the query's codes are looked up in L prebuilt hash tables; "don't pick
 * the tallest", section 6: every table stores a pointer to every key, and a query scans about
 * L n / 2^K entries). Layout per (sequence, KV head), 32-bit words: offsets[L][2^K + 1], then
 * members[L][n], then the build's scratch [L][8][2^K]; members[t][offsets[t][c] .. offsets[t][c+1])
 * are the keys with code c in table t. The order inside a bucket is not fixed (a bucket is a set).
 * mp_buckets_bytes: bytes for B*Hkv such tables (L (2^K + 1 + n + 8 * 2^K) words each); 0 if
 * K > 12 or the shapes are invalid. */
MP_API size_t mp_buckets_bytes(int B, int Hkv, int n, int K, int L);

/* Build the bucketed tables from the packed codes of mp_build_tables (same B, Hkv, n, K, L).
 * buckets: caller-owned device memory of mp_buckets_bytes bytes, 4-byte aligned; codes may be
 * NULL when K == 0. Errors: MP_ERR_INVALID_ARG (shapes, null, misalignment), MP_ERR_UNSUPPORTED
 * (K > 12). */
MP_API mp_status mp_build_buckets(const uint32_t* codes, int B, int Hkv, int n, int K, int L,
                                  uint32_t* buckets, cudaStream_t stream);

/* MIPS variant: radius[b][g] = max over keys [0, n) of |k_i - mu| (float32, [B][Hkv], written
 * by this call; fp32 arithmetic). The keys are laid out for n_capacity tokens per head.
 * Errors: MP_ERR_INVALID_ARG (shapes, null, misalignment), MP_ERR_UNSUPPORTED (d != 128). */
MP_API mp_status mp_key_radius(const void* keys, mp_dtype key_dtype, const float* centre,
                               int B, int Hkv, int n_capacity, int n, int d, float* radius,
                               cudaStream_t stream);

/* MIPS variant of mp_encode_keys: codes of keys [n_begin, n_end) from the extended centred keys,
 * bit = [sum_e W[e][j] (k[e] - mu[e]) + W[d][j] sqrt(max(0, r^2 - |k - mu|^2)) > 0].
 * W_aug: [d + 1][K*L]; radius from mp_key_radius (a key longer than r, appended after r was
 * taken, gets 0 in the extra coordinate).
 * norms_scratch: NULL, or caller-owned device memory of B*Hkv*n_capacity floats. With it, bf16
 * keys and W and more than 64 keys, whole 1024-key blocks are re-encoded on the tensor cores
 * (the centred part and the extra coordinate, split exactly into three bf16 terms, both by MMA;
 * the norms of the blocks' keys are written to the scratch first). Otherwise fp32 CUDA cores encode the range
 * itself, keeping the other keys' bits of the words it touches.
 * Errors as mp_encode_keys; MP_ERR_INVALID_ARG also for a NULL radius. */
MP_API mp_status mp_encode_keys_mips(const void* keys, mp_dtype key_dtype, const float* centre,
                                     const void* W_aug, mp_dtype w_dtype, const float* radius,
                                     int B, int Hkv, int n_capacity, int n_begin, int n_end,
                                     int d, int K, int L, uint32_t* codes, float* norms_scratch,
                                     cudaStream_t stream);

/* Cross-polytope variant: bytes of codes for B*Hkv heads of n keys and L tables,
 * B*Hkv*ceil(n/1024)*L*1024; 0 for invalid shapes. */
MP_API size_t mp_cp_codes_bytes(int B, int Hkv, int n, int L);

/* Cross-polytope variant: log u at the MP_LOGU_TABLE_ENTRIES cosines -1 + 2 i / 4096, i.e.
 * log P[Binomial(L, p^K) >= 2] with p the cross-polytope collision probability (d = 128),
 * into the caller's float32 device array `table`, for mp_params.logu_table. One kernel of a few
 * milliseconds; build it once per (K, L). Errors: MP_ERR_INVALID_ARG (K, L < 1, null,
 * misalignment), MP_ERR_UNSUPPORTED (d != 128). */
MP_API mp_status mp_cp_logu_table(int K, int L, int d, float* table, cudaStream_t stream);

/* Cross-polytope variant: codes of keys [n_begin, n_end) of a cache laid out for n_capacity
 * tokens per head, G [L][d][d] (MP_F32 or MP_BF16), ties to the smaller index. With bf16 keys and
 * G and more than 64 keys, whole 1024-key blocks are re-encoded on the tensor cores (the
 * encoder's projections, an argmax instead of the signs); otherwise fp32 CUDA cores encode the
 * range itself and leave other keys' bytes untouched (appends).
 * codes: mp_cp_codes_bytes(B, Hkv, n_capacity, L) bytes, 16-byte aligned.
 * Errors: MP_ERR_INVALID_ARG (shapes, range, null, misalignment), MP_ERR_UNSUPPORTED (d != 128). */
MP_API mp_status mp_encode_keys_cp(const void* keys, mp_dtype key_dtype, const float* centre,
                                   const void* G, mp_dtype g_dtype, int B, int Hkv,
                                   int n_capacity, int n_begin, int n_end, int d, int L,
                                   uint8_t* codes, cudaStream_t stream);

/* mp_build_buckets over keys [0, n) of codes laid out for n_capacity tokens per head (the
 * appendable cache of mp_encode_keys); buckets is mp_buckets_bytes(B, Hkv, n, K, L) bytes. A
 * decode then passes n_indexed = n in mp_params while its own n grows. */
MP_API mp_status mp_build_buckets_cap(const uint32_t* codes, int B, int Hkv, int n_capacity,
                                      int n, int K, int L, uint32_t* buckets,
                                      cudaStream_t stream);

/* mp_sampled_attention with the bucketed tables instead of a scan of the packed codes: each
 * query row reads its bucket in every table and keeps the keys hit by >= 2 tables (the same S as
 * the scan, bit for bit), then the same gather, importance weights and merged softmax. Needs the
 * query encoding of mp_encode_query in the workspace first, like mp_sampled_attention.
 * The tables cover keys [0, prm->n_indexed); keys appended since (up to n) are found by the code
 * scan over the 1024-key blocks from n_indexed / 1024 on, which replaces the lookup's result in
 * those blocks. So codes must be passed too (NULL only when n_indexed == n and n is a multiple
 * of 1024, or K == 0) and the tables must have been built for n_indexed keys.
 * buckets: 16-byte aligned. Errors as mp_sampled_attention; MP_ERR_UNSUPPORTED also for K > 12. */
MP_API mp_status mp_sampled_attention_buckets(const void* q, mp_dtype q_dtype,
                                              const uint32_t* buckets, const uint32_t* codes,
                                              const float* centre,
                                              const void* keys, const void* values,
                                              mp_dtype kv_dtype, int B, int Hq, int Hkv, int n,
                                              int d, const mp_params* prm, float* out,
                                              void* workspace, size_t ws_bytes,
                                              cudaStream_t stream);

/* Workspace bytes mp_debug_select needs. */
MP_API size_t mp_debug_workspace_bytes(int B, int Hq, int Hkv, int n, int d,
                                       const mp_params* prm);

/* mp_decode_attention plus what it decided, for checking against a reference:
 *   q_bits    [B][Hq][ceil(K*L/32)] uint32: bit j%32 of word j/32 is the query's sign bit j
 *   sel_idx   [B][Hq][n] int32: ascending indices of S (the sampled set, T excluded), the first
 *             sel_count[b][h] entries are valid
 *   sel_count [B][Hq] int32
 *   cnt       [B][Hq][n] uint8 collision counts (saturating at 255), or NULL to skip
 * The selection comes from the same kernel mp_decode_attention runs; cnt from a separate
 * counting kernel. Errors as mp_decode_attention. */
MP_API mp_status mp_debug_select(const void* q, mp_dtype q_dtype, const uint32_t* codes,
                                 const float* centre, const void* W, mp_dtype w_dtype,
                                 const void* keys, const void* values, mp_dtype kv_dtype, int B,
                                 int Hq, int Hkv, int n, int d, const mp_params* prm, float* out,
                                 uint32_t* q_bits, int32_t* sel_idx, int32_t* sel_count,
                                 uint8_t* cnt, void* workspace, size_t ws_bytes,
                                 cudaStream_t stream);

/* mp_sampled_attention_buckets plus what it decided, for checking the bucketed retrieval against
 * a reference: the query encoding of mp_encode_query (its sign bits into q_bits), the bucket lookup
 * (and the scan of keys appended since the tables were built), the same attend kernel, and the
 * sampled sets S (T excluded, ascending) into sel_idx / sel_count, laid out as in mp_debug_select.
 * The workspace is mp_debug_workspace_bytes. Errors as mp_sampled_attention_buckets. */
MP_API mp_status mp_debug_select_buckets(const void* q, mp_dtype q_dtype, const uint32_t* buckets,
                                         const uint32_t* codes, const float* centre,
                                         const void* W, mp_dtype w_dtype, const void* keys,
                                         const void* values, mp_dtype kv_dtype, int B, int Hq,
                                         int Hkv, int n, int d, const mp_params* prm, float* out,
                                         uint32_t* q_bits, int32_t* sel_idx, int32_t* sel_count,
                                         void* workspace, size_t ws_bytes, cudaStream_t stream);

/* log u at each of `count` cosines c (float32 device arrays cosines -> out), evaluated as the
 * decode kernels evaluate it for every selected key of the SimHash codes (the per-call table and
 * the closed form where the table is not used, as mp_decode_attention describes): p = 1 -
 * arccos(c) / pi, u = P[Binomial(L, p^K) >= 2] ("LSH Sampling...", method details, the u_i formula),
 * in fp32 in the log domain; p = 0 gives log(FLT_MIN), L = 1 gives -inf. For checking that
 * evaluation against a reference. Errors: MP_ERR_INVALID_ARG (count < 0, K outside [0, 32],
 * L < 1, null or misaligned arrays). */
MP_API mp_status mp_debug_log_inclusion(const float* cosines, int count, int K, int L, float* out,
                                        cudaStream_t stream);

/* Test hook of the failure path: one thread waits, with the bounded wait the tensor-core encoder
 * uses on its pipeline barriers, on an mbarrier that nothing completes (no arrival, copy or MMA is
 * issued), gives up after limit_us microseconds (1 to 100000) and records MP_ERR_TIMEOUT in the
 * device status word, as a stalled encoder would; mp_device_status then returns it once.
 * The paper has no counterpart. Errors: MP_ERR_INVALID_ARG (limit out of range). */
MP_API mp_status mp_debug_wait_expiry(int limit_us, cudaStream_t stream);

/* Unpack codes into one integer per (key, table): table_codes[b][g][i][t] = code_t(k_i) =
 * sum_b bit_{i, t*K+b} << b. Requires K <= 32. */
MP_API mp_status mp_codes_unpack(const uint32_t* codes, int B, int Hkv, int n, int K, int L,
                                 uint32_t* table_codes, cudaStream_t stream);

/* Size of the fixed scratch array mp_decode_attention_noalloc uses (8 MiB). */
#define MP_NOALLOC_SCRATCH_BYTES (8u << 20)

/* mp_decode_attention for callers that cannot allocate device memory. The paper has no
 * counterpart; this entry point exists for callers such as plugins of a runtime that owns all
 * device memory through its own pool, or latency-critical loops where an allocation (which may
 * synchronise the device) is not allowed, or code that holds no allocator at all. It takes the
 * same inputs and output as mp_decode_attention, without a workspace: its scratch is a fixed
 * array of MP_NOALLOC_SCRATCH_BYTES inside the library, resident on every GPU that loads the
 * library until the process exits. It never allocates or frees memory.
 *   - The first call on a device (with that device current) resolves the array's address and
 *     loads the decode kernels; make that first call before any stream capture.
 *   - Shapes that need more scratch than the array holds (mp_decode_workspace_bytes() above
 *     MP_NOALLOC_SCRATCH_BYTES) are rejected with MP_ERR_WORKSPACE before anything is launched.
 *   - Every call on a device shares the one array. The merge counters are reset at the start of
 *     each call and the rest is written before it is read, so sequential calls are independent;
 *     calls whose kernels overlap on the GPU (other streams, unordered threads) race on it.
 * Other errors as mp_decode_attention. */
MP_API mp_status mp_decode_attention_noalloc(const void* q, mp_dtype q_dtype,
                                             const uint32_t* codes, const float* centre,
                                             const void* W, mp_dtype w_dtype, const void* keys,
                                             const void* values, mp_dtype kv_dtype, int B, int Hq,
                                             int Hkv, int n, int d, const mp_params* prm,
                                             float* out, cudaStream_t stream);

/* Synchronise the current device, return its status word (MP_OK, MP_ERR_TIMEOUT, or in the
 * MP_CHECKS build MP_ERR_BOUNDS) through *status and reset it, with the check site beside it, to
 * MP_OK. Returns MP_ERR_CUDA if the device cannot be reached. */
MP_API mp_status mp_device_status(int* status);

/* The MP_CHECKS build (the library compiled with -DMP_CHECKS=1, libmagicpig_checks.so): every
 * kernel of the decode path, the bucketed lookup and the tensor-core encoder check the indices of
 * their global accesses (code blocks, selection words, K/V rows, partial states, bucket ranges
 * and members, code words written) and skip an access that is out of range instead of making
 * it, raising MP_ERR_BOUNDS in the status word. A stand-in for a memory checker: the paper has
 * no counterpart. Synchronises the device and returns through *enabled 1 in that build, 0 in the
 * product build, and through *site the site of the first failed check since the status word was
 * last reset (0 if none): 1 query encoding stores, 2 scanned code block, 3 selection words
 * written, 4 K/V row copied, 5 partial state or output written, 6 selection words read,
 * 7 bucket range beyond the table's keys, 8 bucket member beyond n_indexed, 9 code words written
 * by the encoder. Neither word is reset. Errors: MP_ERR_INVALID_ARG (null), MP_ERR_CUDA. */
MP_API mp_status mp_debug_check_report(int* enabled, int* site);

#ifdef __cplusplus
}
#endif
#endif /* MAGICPIG_H */
