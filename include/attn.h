/*
 * attn.h -- C ABI of libattn: scaled-dot-product attention for LLM decode,
 * prefill and vision-tower inference on one NVIDIA GB300 (sm_103a).
 *
 * Every call is asynchronous on the caller's CUDA stream and allocates no
 * device memory: the caller owns every buffer it passes.  Pointers named
 * "device" must be device (or managed) addresses of the current CUDA device.
 * "stream" is a cudaStream_t (CUstream) handle; NULL is the legacy default
 * stream.  On a non-OK status nothing has been launched (argument errors are
 * detected on the host before any launch) and attn_last_error() describes the
 * problem.
 *
 * Notation: B batch, Hq query heads, Hkv kv heads (Hq % Hkv == 0, G = Hq/Hkv),
 * D head_dim, L_b = kv_len[b], S prefill length, P page size, W window.
 *
 * What is computed (for each sequence/prompt b, query head h, query i):
 *   g = h / G;  s_j = scale * (q_i . k_j[g]);  s_j = c*tanh(s_j/c) if c > 0;
 *   o_i = sum_j softmax_j(s) v_j[g] over the kept keys j, in fp32 with f16 I/O.
 * Sources: doppler src/gpu/kernels/attention.js (createAttentionUniformBuffer:
 * numHeads, numKVHeads, headDim, kvLen, seqLen, scale, causal, attnSoftcap
 * and slidingWindow (0 turns either off), pageSize, kvLayout
 * contiguous/ring/paged; executeAttention: the per-call kvLen buffer and page
 * table; executeAttentionTiered / executeAttentionTieredQuant: the hot and
 * cold tiers), doppler src/inference/pipelines/text/attention/run.js
 * (runLayerAttentionGPU: the decode query sits at position kvLen-1, the
 * sliding-window clamp, scale = 1/sqrt(query_pre_attn_scalar)), and rullama
 * src/backend/dispatch/attention.rs (vision_attention_chained: bidirectional
 * attention over [n_patches, n_heads, head_dim] tensors).
 */
#ifndef LIBATTN_ATTN_H
#define LIBATTN_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_EINVAL = 1,        /* invalid argument (null pointer, bad size, bad count) */
    ATTN_EUNSUPPORTED = 2,  /* valid but not supported (head_dim, page size, ...) */
    ATTN_ECUDA = 3,         /* a CUDA runtime/driver call failed */
    ATTN_EBOUNDS = 4,       /* device data out of range (attn_decode_validate) */
    ATTN_ETIMEOUT = 5       /* a kernel abandoned a pipeline wait (attn_device_status) */
} attn_status;

typedef enum {
    ATTN_KV_F16 = 0,        /* K/V cache elements are IEEE binary16 */
    ATTN_KV_INT8 = 1        /* K/V cache elements are int8 codes with per-(token, kv-head)
                               f16 scales: value = code * scale (attention.js,
                               executeAttentionTieredQuant: int8 K/V with separate
                               K and V scale buffers) */
} attn_kv_dtype;

/* Element type of decode queries and outputs (attn_decode_ex, attn_decode_tiered). */
typedef enum {
    ATTN_F16 = 0,           /* IEEE binary16 */
    ATTN_F32 = 1            /* IEEE binary32 (attention.js: the int8 tier takes f32 Q only;
                               outputDtype f16 or f32 per variant) */
} attn_dtype;

/* Library version, e.g. "libattn 0.1.0 sm_103a". */
const char* attn_version(void);

/* Message for the last non-OK status returned on this host thread. */
const char* attn_last_error(void);

/*
 * Bytes of scratch memory attn_decode needs for these sizes.  max_kv is the
 * largest kv_len any sequence may have in the call; split_keys as in
 * attn_decode (0 = automatic).  Returns 0 for invalid sizes.
 */
size_t attn_decode_workspace_size(int batch, int n_heads, int n_kv_heads, int head_dim,
                                  int max_kv, int split_keys);

/*
 * attn_decode -- split-KV flash-decode: one new query token per sequence
 * attends to that sequence's KV cache.
 *
 *  q           device, f16 [B, Hq, D] (row-major), the new tokens' queries.
 *  k_cache,    device.  Contiguous layout (page_table == NULL):
 *  v_cache       [B, max_kv, Hkv, D]; token t of sequence b at [b, t].
 *                Paged layout: a pool [n_pages, P, Hkv, D]; token t of
 *                sequence b at [page_table[b, t / P], t % P].
 *                Elements f16 (ATTN_KV_F16) or int8 codes (ATTN_KV_INT8).
 *  kv_len      device, int32 [B]: L_b, the number of cached tokens including
 *                the new one (the query's position is L_b - 1, so the causal
 *                mask keeps every cached token).  Values are clamped to the
 *                layout's capacity; L_b <= 0 yields a zero output row and
 *                lse = -inf.  attn_decode_validate checks them.
 *  page_table  device, int32 [B, max_pages_per_seq], or NULL for contiguous.
 *                Entries past ceil(L_b / P) are never read.
 *  page_size   P: a power of two in [1, 1024] (>= 8 for int8 caches).
 *  n_pages     pages in the pool (paged layout only).
 *  max_kv      contiguous: tokens per sequence in the cache (capacity; a
 *                multiple of 8 for int8 caches).  Paged: an upper bound on
 *                L_b (<= max_pages_per_seq * P), used to size the split plan.
 *  k_scales,   device f16, int8 caches only (else NULL).  Contiguous:
 *  v_scales      [B, Hkv, max_kv]; paged: [n_pages, Hkv, P].
 *  window      W > 0 keeps only the W most recent tokens (positions
 *                L_b - W .. L_b - 1, run.js sliding-window clamp); 0 = off.
 *  softcap     c > 0 applies s -> c * tanh(s / c) after scaling; 0 = off.
 *  scale       the logit scale, e.g. 1/sqrt(D) or 1/sqrt(query_pre_attn_scalar).
 *  split_keys  keys per split (a multiple of 16), or 0 for automatic.  The
 *                result does not depend on it beyond fp32 rounding.  With 0, a
 *                call whose sequences keep at most 512 keys (max_kv, or the
 *                window), with G * D <= 1024 and a small cache in all (at most
 *                2^22 to 2^24 (sequence, kv head, key, dim) elements by head
 *                dim and dtype), runs in one launch without splits or the
 *                combine pass and leaves the workspace untouched.
 *  out         device, f16 [B, Hq, D].
 *  lse_out     device, f32 [B, Hq] or NULL: log-sum-exp of the kept scaled
 *                logits (natural log).
 *  workspace   device scratch of workspace_bytes >= attn_decode_workspace_size(
 *                B, Hq, Hkv, D, max_kv, split_keys); contents need no
 *                initialisation and are overwritten.
 *  D must be 64, 128 or 256; G = Hq / Hkv any positive integer.
 *  The same split plan and arithmetic order are used for both layouts, so a
 *  paged cache holding the same values as a contiguous one gives bit-identical
 *  results.
 */
attn_status attn_decode(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* kv_len, const int32_t* page_table,
                        int page_size, int max_pages_per_seq, int n_pages, int max_kv,
                        const void* k_scales, const void* v_scales, attn_kv_dtype kv_dtype,
                        int batch, int n_heads, int n_kv_heads, int head_dim,
                        int window, float softcap, float scale, int split_keys,
                        void* out, float* lse_out,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_decode_ring -- attn_decode over a ring (rolling-buffer) KV cache, the
 * layout a sliding-window model keeps: each sequence owns ring_size slots and
 * token t is written to slot t % ring_size, overwriting token t - ring_size.
 * (Sliding-window attention, rolling buffer cache; the window of W tokens
 * needs no more than W slots.)
 *
 *  k_ring,     device, [B, ring_size, Hkv, D] f16 or int8 codes; token t of
 *  v_ring        sequence b at [b, t % ring_size].
 *  seq_len     device, int32 [B]: L_b, the LOGICAL number of tokens the
 *                sequence has seen, including the new one (any value; not
 *                clamped to ring_size).  The query's position is L_b - 1.
 *                L_b <= 0 yields a zero output row and lse = -inf.
 *  ring_size   slots per sequence: a positive multiple of 16, so no 16-token
 *                tile wraps round the ring.  ATTN_EUNSUPPORTED otherwise.
 *  k_scales,   int8 caches only: [B, Hkv, ring_size], slot-indexed like the
 *  v_scales      codes.
 *  window      W > 0 keeps the W most recent tokens; the ring itself keeps
 *                at most ring_size, so the kept keys are the last
 *                min(L_b, ring_size, W or ring_size) tokens.
 *  workspace   >= attn_decode_workspace_size(B, Hq, Hkv, D, ring_size,
 *                split_keys).
 *  The other arguments are those of attn_decode.  Slots that hold no kept
 *  token (not yet written, or older than the window) are never used for the
 *  result, whatever they contain.  A ring whose slots hold the same values as
 *  a contiguous cache's last kept tokens gives the result of attn_decode on
 *  that cache with the window min(ring_size, W), up to fp32 rounding order.
 */
attn_status attn_decode_ring(const void* q, const void* k_ring, const void* v_ring,
                             const int32_t* seq_len, int ring_size,
                             const void* k_scales, const void* v_scales, attn_kv_dtype kv_dtype,
                             int batch, int n_heads, int n_kv_heads, int head_dim,
                             int window, float softcap, float scale, int split_keys,
                             void* out, float* lse_out,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_decode_ex -- attn_decode with every cache layout and the query and
 * output element types as arguments.
 *
 *  q, q_dtype      device [B, Hq, D] of ATTN_F16 or ATTN_F32.  How far f32
 *                    queries keep their precision depends on the cache:
 *                    f16 caches with D 64/128 (tensor-core kernel) multiply two
 *                    f16 terms hi + lo (hi = f16(q), lo = f16(q - hi), together
 *                    within 2^-22 |q|) into one accumulator; f16 caches with
 *                    D 256 or pages of fewer than 16 tokens read q as f32.
 *                    int8 caches round every query (f16 or f32) to 16-bit fixed
 *                    point with one scale per (sequence, head), 1/32767 of that
 *                    head's largest |q| (error at most max|q| / 65534 per
 *                    element), so that q.k is an exact integer dot product of
 *                    the codes: there f32 queries are no more precise than
 *                    that rounding.
 *  ring_size       > 0 selects the ring layout of attn_decode_ring (kv_len is
 *                    then the logical length, page_table must be NULL and max_kv
 *                    is ignored); 0 selects attn_decode's contiguous or paged
 *                    layout.
 *  out, out_dtype  device [B, Hq, D] of ATTN_F16 (rounded to nearest even) or
 *                    ATTN_F32.
 *  The other arguments, the workspace (attn_decode_workspace_size with max_kv,
 *  or ring_size for a ring) and the errors are attn_decode's.  With f16 q and
 *  f16 out the result is attn_decode's bit for bit; f32 out holds the same
 *  values before their rounding to f16.
 */
attn_status attn_decode_ex(const void* q, attn_dtype q_dtype,
                           const void* k_cache, const void* v_cache,
                           const int32_t* kv_len, const int32_t* page_table,
                           int page_size, int max_pages_per_seq, int n_pages, int max_kv, int ring_size,
                           const void* k_scales, const void* v_scales, attn_kv_dtype kv_dtype,
                           int batch, int n_heads, int n_kv_heads, int head_dim,
                           int window, float softcap, float scale, int split_keys,
                           void* out, attn_dtype out_dtype, float* lse_out,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_decode_tiered -- decode over two tiers of one sequence's cache in one
 * call: a cold tier (the older tokens: contiguous or paged, f16 or int8 with
 * scales) and a hot tier (the newest tokens: an f16 ring).  (doppler
 * attention.js executeAttentionTiered / executeAttentionTieredQuant: coldLen,
 * hotLen, hotWindow, hotStart, coldPageTable, coldPageSize, coldLayout paged
 * or contiguous, hotLayout ring.)
 *
 *  cold_*      the cold tier exactly as attn_decode takes a cache:
 *                cold_k/cold_v, cold_k_scales/cold_v_scales (int8 only),
 *                cold_dtype, cold_len (kv_len: cold tokens of each sequence,
 *                clamped to the capacity), cold_page_table (NULL for
 *                contiguous [B, cold_max_kv, Hkv, D]), cold_page_size,
 *                cold_max_pages_per_seq, cold_n_pages, cold_max_kv (contiguous
 *                capacity, or paged bound).  Same rules and errors.
 *  hot_k,      device f16 [B, hot_ring, Hkv, D]: hot token i of sequence b in
 *  hot_v         slot (hot_start[b] + i) mod hot_ring.
 *  hot_len     device int32 [B]: hot tokens of each sequence (<= 0: none).
 *                The ring holds the newest hot_ring of them; older ones are
 *                gone.
 *  hot_start   device int32 [B]: slot of hot token 0 (any integer; taken
 *                modulo hot_ring).
 *  hot_ring    slots per sequence, a positive multiple of 16
 *                (ATTN_EUNSUPPORTED otherwise).
 *  Positions: cold token j at j, hot token i at cold_len + i; the query is the
 *  newest token, at cold_len + hot_len - 1.  window W > 0 keeps the keys whose
 *  position is within W of the query (it may end inside either tier); 0 = off.
 *  q_dtype,    the element types of q and out, as in attn_decode_ex (the
 *  out_dtype     int8 tier of the pages takes f32 q).
 *  The other arguments are those of attn_decode; out and lse_out receive one
 *  softmax over the kept keys of both tiers.  A sequence with no kept key gets
 *  a zero row and lse = -inf.
 *  workspace   >= attn_decode_tiered_workspace_size(B, Hq, Hkv, D,
 *                cold_max_kv, hot_ring, split_keys) bytes, 256-byte aligned.
 *  Three kernels run on the stream: the cold tier's split kernel, the hot
 *  tier's, and one log-sum-exp combine over both.
 */
size_t attn_decode_tiered_workspace_size(int batch, int n_heads, int n_kv_heads, int head_dim,
                                         int cold_max_kv, int hot_ring, int split_keys);
attn_status attn_decode_tiered(const void* q, attn_dtype q_dtype,
                               const void* cold_k, const void* cold_v,
                               const void* cold_k_scales, const void* cold_v_scales,
                               attn_kv_dtype cold_dtype, const int32_t* cold_len,
                               const int32_t* cold_page_table, int cold_page_size,
                               int cold_max_pages_per_seq, int cold_n_pages, int cold_max_kv,
                               const void* hot_k, const void* hot_v,
                               const int32_t* hot_len, const int32_t* hot_start, int hot_ring,
                               int batch, int n_heads, int n_kv_heads, int head_dim,
                               int window, float softcap, float scale, int split_keys,
                               void* out, attn_dtype out_dtype, float* lse_out,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_decode_noalloc -- attn_decode for callers that cannot allocate device
 * memory, so cannot supply a workspace: for example a plugin running inside
 * an engine that owns all device memory and offers it no allocator, or a
 * latency-critical decode loop that must never call cudaMalloc (a call that
 * can synchronise the whole device).  The source pages have no counterpart of
 * this entry point; it is an addition of this library.
 *
 * Arguments and results are those of attn_decode without workspace and
 * workspace_bytes.  The split partials go to a fixed 16 MiB device array
 * compiled into the library; every GPU that loads the library holds that
 * array until the process exits.  Sizes whose attn_decode_workspace_size
 * exceeds 16 MiB are rejected with ATTN_EUNSUPPORTED (a larger split_keys
 * lowers the need).  The calls themselves allocate nothing, but the array is
 * reserved when the library's device module loads: at context creation with
 * eager module loading, else (lazy loading, the default) inside the first
 * call of the library on that device, which may synchronise the device.
 * Make one warm-up call at initialisation, outside stream capture and
 * latency-critical loops.  Every call looks the array's device address up
 * (cudaGetSymbolAddress, no allocation once loaded), so a cudaDeviceReset
 * between calls is safe.  All calls share the one array and no part of it
 * needs to start at zero; calls whose kernels overlap on the GPU (different
 * streams without ordering) race on it, so order them on one stream.
 */
attn_status attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* kv_len, const int32_t* page_table,
                                int page_size, int max_pages_per_seq, int n_pages, int max_kv,
                                const void* k_scales, const void* v_scales, attn_kv_dtype kv_dtype,
                                int batch, int n_heads, int n_kv_heads, int head_dim,
                                int window, float softcap, float scale, int split_keys,
                                void* out, float* lse_out, void* stream);

/*
 * attn_prefill -- tiled prefill / vision attention of S tokens over themselves
 * on the tensor cores (tcgen05 + TMEM, operands staged by TMA).
 *
 *  q     device f16 [S, Hq, D];  k, v  device f16 [S, Hkv, D]  (token-major,
 *        heads interleaved: the q/k/v layout vision_attention_chained shares
 *        with text attention).
 *  causal  nonzero: query i keeps keys j <= i (text prefill); 0: bidirectional
 *          (vision tower).
 *  window  W > 0: causal keeps i - W < j <= i; bidirectional keeps |i - j| < W.
 *  softcap, scale  as in attn_decode.
 *  out   device f16 [S, Hq, D].   lse_out  device f32 [S, Hq] or NULL.
 *  D must be 64, 128 or 256; seq_len at most 65535 * 128.  Base addresses
 *  must be 16-byte aligned.
 */
attn_status attn_prefill(const void* q, const void* k, const void* v,
                         int seq_len, int n_heads, int n_kv_heads, int head_dim,
                         int causal, int window, float softcap, float scale,
                         void* out, float* lse_out, void* stream);

/*
 * attn_prefill_paged -- chunked prefill / multi-token decode: each sequence
 * appends a chunk of new tokens to its paged KV cache and the chunk's queries
 * attend causally to every cached token up to their own position
 * (doppler attention.js, createAttentionUniformBuffer: seqLen new tokens at
 * startPos over kvLen keys with the paged layout's page table and pageSize;
 * attn_decode is the one-token case).  Same tensor-core kernel as
 * attn_prefill, with K/V read through the page table.
 *
 *  q         device f16 [total_q, Hq, D]: sequence b's new tokens are the rows
 *            q_start[b] .. q_start[b+1]-1 (packed, sequences in order).
 *  k_cache, v_cache  device f16 page pool [n_pages, P, Hkv, D].  The chunk's
 *            own K/V must already be written: they are the last q_len of the
 *            sequence's kv_len tokens.
 *  q_start   device i32 [B+1], non-decreasing, q_start[0] = 0, q_start[B] = total_q.
 *  kv_len    device i32 [B]: cached tokens of each sequence, chunk included.
 *            Query i of sequence b (q_len = q_start[b+1] - q_start[b]) sits at
 *            position kv_len[b] - q_len + i and keeps keys j <= position
 *            (and position - j < window when window > 0).  Keys at or above
 *            max_pages_per_seq * P are clamped away (as in attn_decode); a
 *            query at a negative position keeps no key: out = 0, lse = -inf.
 *  page_table  device i32 [B, max_pages_per_seq]: logical token t of sequence b
 *            is row t % P of page page_table[b][t / P].  A page id in use that
 *            lies outside [0, n_pages) is never read (its keys read as zeros)
 *            and is reported through attn_device_status (ATTN_EBOUNDS).
 *  page_size P: a power of two >= 8.
 *  total_q   rows of q; max_q: an upper bound of q_len over the sequences
 *            (sizes the launch; a chunk longer than max_q is cut at max_q rows).
 *  softcap, scale  as in attn_decode.
 *  out       device f16 [total_q, Hq, D]; lse_out device f32 [total_q, Hq] or NULL.
 *  D must be 64, 128 or 256; base addresses 16-byte aligned.  Asynchronous on
 *  `stream`; the host reads none of the device arrays.
 */
attn_status attn_prefill_paged(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* q_start, const int32_t* kv_len, const int32_t* page_table,
                               int page_size, int max_pages_per_seq, int n_pages,
                               int batch, int total_q, int max_q,
                               int n_heads, int n_kv_heads, int head_dim,
                               int window, float softcap, float scale,
                               void* out, float* lse_out, void* stream);

/*
 * attn_decode_validate -- synchronous check of the device-side decode inputs:
 * every kv_len[b] in [1, capacity] and every page id a sequence uses in
 * [0, n_pages).  Launches one small kernel on stream and waits for it.
 * Returns ATTN_OK, ATTN_EBOUNDS (bad page id or length > capacity; *bad_seq
 * receives the first offending sequence if bad_seq != NULL) or ATTN_EINVAL
 * (kv_len <= 0).  Not needed on the fast path: attn_decode never reads outside
 * its buffers on such data (lengths are clamped to the capacity, a page id
 * outside [0, n_pages) is replaced by page 0 and reported through
 * attn_device_status), it only gives meaningless rows for those sequences.
 */
attn_status attn_decode_validate(const int32_t* kv_len, const int32_t* page_table,
                                 int batch, int page_size, int max_pages_per_seq,
                                 int n_pages, int max_kv, int* bad_seq, void* stream);

/*
 * attn_device_status -- synchronises stream, then reads and clears the
 * library's device error word.  Returns ATTN_ETIMEOUT if a kernel abandoned a
 * pipeline wait (its output is then invalid), ATTN_EBOUNDS if attn_decode met
 * a page id outside the pool, else ATTN_OK.
 */
attn_status attn_device_status(void* stream);

/*
 * attn_testing_set_waits -- testing hook for the failure path of the kernels'
 * bounded waits; not for production use.  (The source pages have no
 * counterpart: their WebGPU host code throws on errors and has no device-side
 * waits.)  Every pipeline wait of the kernels (a tile's copy, a tensor-core
 * result, a free buffer) gives up after a time limit, records a code in the
 * library's device error word, raises the CTA's abort flag so that every role
 * leaves its loop, waits (with the full limit) for its own copies and
 * tensor-core work already in flight, frees its tensor memory and returns.
 *
 *  wait_limit_ns     the time limit of pipeline waits in ns; 0 restores the
 *                      default (4 s).  Waits for work already in flight keep
 *                      the default.
 *  stall_first_tile  1: from now on every CTA of the prefill and tensor-core
 *                      decode kernels holds back the signal that its first
 *                      S tile is ready, and the CUDA-core decode kernel issues
 *                      no copy, so one pipeline wait of every CTA runs out:
 *                      the call's output is invalid and attn_device_status
 *                      then returns ATTN_ETIMEOUT.  0: normal operation.
 *  The settings apply to the current device and to every later launch; the
 *  call is synchronous.  Returns ATTN_EINVAL for another stall value.
 */
attn_status attn_testing_set_waits(unsigned long long wait_limit_ns, int stall_first_tile);

#ifdef __cplusplus
}
#endif

#endif /* LIBATTN_ATTN_H */
