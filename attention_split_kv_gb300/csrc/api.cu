// api.cu -- the C ABI of libattn: host-side argument checks, split planning,
// TMA tensor-map encoding and kernel launches.  No call allocates device
// memory; every check that can be made on the host is made before anything
// is launched.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "attn.h"
#include "attn_internal.h"

namespace attn {

namespace {
thread_local char g_msg[512] = "";

// The library's device error word: kernels that abandon a pipeline wait
// record a code here (see ptx.cuh); attn_device_status reads and clears it.
__device__ int g_device_error = 0;

// Result words of attn_decode_validate.
__device__ int g_validate_code = 0;
__device__ int g_validate_seq = 0x7fffffff;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices] = {};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn get_encode() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return g_encode;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

__global__ void validate_kernel(const int32_t* kv_len, const int32_t* page_table, int B, int P, int max_pages,
                                int n_pages, int cap) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int L = kv_len[b];
    int code = 0;
    if (L <= 0) code = ATTN_EINVAL;
    else if (L > cap) code = ATTN_EBOUNDS;
    else if (page_table) {
        const int np = (L + P - 1) / P;
        for (int i = 0; i < np; ++i) {
            const int pg = page_table[(size_t)b * max_pages + i];
            if (pg < 0 || pg >= n_pages) { code = ATTN_EBOUNDS; break; }
        }
    }
    if (code) {
        atomicMin(&g_validate_seq, b);
        atomicMax(&g_validate_code, code);
    }
}
}  // namespace

attn_status set_error(attn_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return st;
}

bool trace_enabled() {
    static const bool on = [] {
        const char* e = std::getenv("ATTN_TRACE");
        return e != nullptr && e[0] != '\0' && std::strcmp(e, "0") != 0;
    }();
    return on;
}

void trace(const char* fmt, ...) {
    if (!trace_enabled()) return;
    char line[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(line, sizeof(line), fmt, ap);
    va_end(ap);
    std::fprintf(stderr, "[libattn] %s\n", line);
}

// Looked up on every call rather than cached: after cudaDeviceReset (or any
// teardown and re-creation of the context) the module reloads at another
// address.  Once the module is loaded the lookup is a host-side table read.
int* device_error_word() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    return static_cast<int*>(p);
}

int sm_count() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDevices) return 148;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sms[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_sms[dev] = n > 0 ? n : 148;
    }
    return g_sms[dev];
}

attn_status encode_tmap_plain(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int rank,
                              const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return set_error(ATTN_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t d[5], s[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) s[i] = strides_bytes[i];
    }
    CUresult r = enc(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, s, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(ATTN_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return ATTN_OK;
}

attn_status encode_tmap_sw128(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int rank,
                              const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return set_error(ATTN_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t d[5], s[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) s[i] = strides_bytes[i];
    }
    CUresult r = enc(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, s, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(ATTN_ECUDA, "cuTensorMapEncodeTiled (swizzled) failed (%d)", (int)r);
    return ATTN_OK;
}

attn_status encode_tmap_3d_f16_sw128(CUtensorMap* map, const void* base, int D, int H, int S, int box_rows) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return set_error(ATTN_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t d[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S};
    cuuint64_t s[2] = {(cuuint64_t)D * 2, (cuuint64_t)D * 2 * H};
    cuuint32_t bx[3] = {64u, 1u, (cuuint32_t)box_rows};
    cuuint32_t es[3] = {1u, 1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), d, s, bx, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(ATTN_ECUDA, "cuTensorMapEncodeTiled (swizzled) failed (%d)", (int)r);
    return ATTN_OK;
}

}  // namespace attn

using namespace attn;

extern "C" {

const char* attn_version(void) { return "libattn 0.1.0 sm_103a"; }

const char* attn_last_error(void) { return g_msg; }

size_t attn_decode_workspace_size(int batch, int n_heads, int n_kv_heads, int head_dim, int max_kv, int split_keys) {
    DecodePlan plan;
    if (batch > kDecodeMaxBatch) return 0;
    if (!make_decode_plan(batch, n_heads, n_kv_heads, head_dim, max_kv, split_keys, &plan)) return 0;
    return plan.bytes;
}

// Host checks and launch description of one decode cache (everything but the
// workspace); ring > 0 selects the ring layout.
static attn_status decode_prepare(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_len,
                                  const int32_t* page_table, int page_size, int max_pages_per_seq, int n_pages,
                                  int max_kv, const void* k_scales, const void* v_scales, attn_kv_dtype kv_dtype,
                                  int batch, int n_heads, int n_kv_heads, int head_dim, int window, float softcap,
                                  float scale, int split_keys, void* out, float* lse_out, void* stream, int ring,
                                  attn_dtype q_dtype, attn_dtype out_dtype, DecodeLaunch* Lp, DecodePlan* plan_p) {
    if ((q_dtype != ATTN_F16 && q_dtype != ATTN_F32) || (out_dtype != ATTN_F16 && out_dtype != ATTN_F32))
        return set_error(ATTN_EINVAL, "attn_decode: q_dtype and out_dtype must be ATTN_F16 or ATTN_F32");
    if (!q || !k_cache || !v_cache || !kv_len || !out)
        return set_error(ATTN_EINVAL, "attn_decode: q, k_cache, v_cache, kv_len and out must be non-null");
    if (batch <= 0 || n_heads <= 0 || n_kv_heads <= 0)
        return set_error(ATTN_EINVAL, "attn_decode: batch, n_heads and n_kv_heads must be positive");
    if (n_heads % n_kv_heads != 0)
        return set_error(ATTN_EINVAL, "attn_decode: n_heads (%d) must be a multiple of n_kv_heads (%d)", n_heads,
                         n_kv_heads);
    if (batch > kDecodeMaxBatch)
        return set_error(ATTN_EUNSUPPORTED, "attn_decode: batch %d exceeds %d", batch, kDecodeMaxBatch);
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return set_error(ATTN_EUNSUPPORTED, "attn_decode: head_dim %d not supported (64, 128, 256)", head_dim);
    if (kv_dtype != ATTN_KV_F16 && kv_dtype != ATTN_KV_INT8)
        return set_error(ATTN_EINVAL, "attn_decode: unknown kv_dtype %d", (int)kv_dtype);
    const bool int8 = kv_dtype == ATTN_KV_INT8;
    if (int8 && (!k_scales || !v_scales))
        return set_error(ATTN_EINVAL, "attn_decode: int8 caches need k_scales and v_scales");
    if (window < 0) return set_error(ATTN_EINVAL, "attn_decode: window must be >= 0 (0 = off)");
    if (!(softcap >= 0.f) || !std::isfinite(softcap))
        return set_error(ATTN_EINVAL, "attn_decode: softcap must be finite and >= 0 (0 = off)");
    if (!std::isfinite(scale)) return set_error(ATTN_EINVAL, "attn_decode: scale must be finite");
    if (max_kv <= 0) return set_error(ATTN_EINVAL, "attn_decode: max_kv must be positive");
    if (split_keys < 0 || split_keys % 16 != 0)
        return set_error(ATTN_EINVAL, "attn_decode: split_keys must be 0 or a positive multiple of 16");
    if (page_table) {
        if (!pow2(page_size) || page_size > 1024)
            return set_error(ATTN_EUNSUPPORTED, "attn_decode: page_size %d must be a power of two <= 1024", page_size);
        if (int8 && page_size < 8)
            return set_error(ATTN_EUNSUPPORTED, "attn_decode: int8 caches need page_size >= 8");
        if (max_pages_per_seq <= 0 || n_pages <= 0)
            return set_error(ATTN_EINVAL, "attn_decode: max_pages_per_seq and n_pages must be positive");
    } else if (int8 && max_kv % 8 != 0) {
        return set_error(ATTN_EUNSUPPORTED, "attn_decode: contiguous int8 caches need max_kv %% 8 == 0");
    }
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        (int8 && (!aligned(k_scales, 16) || !aligned(v_scales, 16))))
        return set_error(ATTN_EINVAL, "attn_decode: q, caches, scales and out must be 16-byte aligned");
    DecodePlan& plan = *plan_p;
    if (!make_decode_plan(batch, n_heads, n_kv_heads, head_dim, max_kv, split_keys, &plan))
        return set_error(ATTN_EINVAL, "attn_decode: invalid sizes for the split plan");
    DecodeLaunch& L = *Lp;
    L.q = q;
    L.k = k_cache;
    L.v = v_cache;
    L.k_scales = k_scales;
    L.v_scales = v_scales;
    L.kv_len = kv_len;
    L.page_table = page_table;
    L.page_size = page_size;
    L.max_pages = max_pages_per_seq;
    L.n_pages = n_pages;
    L.max_kv = max_kv;
    L.int8 = int8;
    L.B = batch;
    L.Hq = n_heads;
    L.Hkv = n_kv_heads;
    L.D = head_dim;
    // a ring keeps at most `ring` logical tokens: the window is never wider
    L.window = ring > 0 ? ((window > 0 && window < ring) ? window : ring) : window;
    L.ring = ring;
    L.softcap = softcap;
    L.scale = scale;
    L.split_keys = split_keys;
    L.out = out;
    L.lse = lse_out;
    L.q_f32 = q_dtype == ATTN_F32;
    L.out_f32 = out_dtype == ATTN_F32;
    L.stream = static_cast<cudaStream_t>(stream);
    return ATTN_OK;
}

static attn_status check_workspace(const char* fn, void* workspace, size_t workspace_bytes, size_t need) {
    if (!workspace || workspace_bytes < need)
        return set_error(ATTN_EINVAL, "%s: workspace of %zu bytes needed, %zu given", fn, need,
                         workspace ? workspace_bytes : (size_t)0);
    if (!aligned(workspace, 256)) return set_error(ATTN_EINVAL, "%s: workspace must be 256-byte aligned", fn);
    return ATTN_OK;
}

// attn_decode and attn_decode_ring: ring > 0 selects the ring cache
static attn_status decode_entry(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_len,
                                const int32_t* page_table, int page_size, int max_pages_per_seq, int n_pages,
                                int max_kv, const void* k_scales, const void* v_scales, attn_kv_dtype kv_dtype,
                                int batch, int n_heads, int n_kv_heads, int head_dim, int window, float softcap,
                                float scale, int split_keys, void* out, float* lse_out, void* workspace,
                                size_t workspace_bytes, void* stream, int ring, attn_dtype q_dtype = ATTN_F16,
                                attn_dtype out_dtype = ATTN_F16) {
    DecodeLaunch L;
    DecodePlan plan;
    attn_status st = decode_prepare(q, k_cache, v_cache, kv_len, page_table, page_size, max_pages_per_seq, n_pages,
                                    max_kv, k_scales, v_scales, kv_dtype, batch, n_heads, n_kv_heads, head_dim,
                                    window, softcap, scale, split_keys, out, lse_out, stream, ring, q_dtype,
                                    out_dtype, &L, &plan);
    if (st != ATTN_OK) return st;
    if ((st = check_workspace("attn_decode", workspace, workspace_bytes, plan.bytes)) != ATTN_OK) return st;
    int* err = device_error_word();
    if (!err) return set_error(ATTN_ECUDA, "attn_decode: no CUDA device / error word");
    L.workspace = workspace;
    L.workspace_bytes = workspace_bytes;
    L.err_word = err;
    return launch_decode(L, plan);
}

// The two plans of a tiered decode and the workspace they share: the cold
// tier's partials first, the hot ring's from the next 256-byte boundary.
static bool tiered_plans(int batch, int n_heads, int n_kv_heads, int head_dim, int cold_max_kv, int hot_ring,
                         int split_keys, DecodePlan* cold, DecodePlan* hot, size_t* hot_off, size_t* bytes) {
    if (batch <= 0 || batch > kDecodeMaxBatch || hot_ring < 16 || hot_ring % 16 != 0) return false;
    if (!make_decode_plan(batch, n_heads, n_kv_heads, head_dim, cold_max_kv, split_keys, cold)) return false;
    if (!make_decode_plan(batch, n_heads, n_kv_heads, head_dim, hot_ring, split_keys, hot)) return false;
    *hot_off = (cold->bytes + 255) / 256 * 256;
    *bytes = *hot_off + hot->bytes;
    return true;
}

size_t attn_decode_tiered_workspace_size(int batch, int n_heads, int n_kv_heads, int head_dim, int cold_max_kv,
                                         int hot_ring, int split_keys) {
    DecodePlan c, h;
    size_t off = 0, bytes = 0;
    if (!tiered_plans(batch, n_heads, n_kv_heads, head_dim, cold_max_kv, hot_ring, split_keys, &c, &h, &off, &bytes))
        return 0;
    return bytes;
}

attn_status attn_decode_tiered(const void* q, attn_dtype q_dtype, const void* cold_k, const void* cold_v,
                               const void* cold_k_scales,
                               const void* cold_v_scales, attn_kv_dtype cold_dtype, const int32_t* cold_len,
                               const int32_t* cold_page_table, int cold_page_size, int cold_max_pages_per_seq,
                               int cold_n_pages, int cold_max_kv, const void* hot_k, const void* hot_v,
                               const int32_t* hot_len, const int32_t* hot_start, int hot_ring, int batch,
                               int n_heads, int n_kv_heads, int head_dim, int window, float softcap, float scale,
                               int split_keys, void* out, attn_dtype out_dtype, float* lse_out, void* workspace,
                               size_t workspace_bytes, void* stream) {
    if (!hot_k || !hot_v || !hot_len || !hot_start)
        return set_error(ATTN_EINVAL, "attn_decode_tiered: hot_k, hot_v, hot_len and hot_start must be non-null");
    if (hot_ring < 16 || hot_ring % 16 != 0)
        return set_error(ATTN_EUNSUPPORTED, "attn_decode_tiered: hot_ring %d must be a positive multiple of 16",
                         hot_ring);
    DecodeLaunch Lc, Lh;
    DecodePlan pc, ph;
    attn_status st = decode_prepare(q, cold_k, cold_v, cold_len, cold_page_table, cold_page_size,
                                    cold_max_pages_per_seq, cold_n_pages, cold_max_kv, cold_k_scales, cold_v_scales,
                                    cold_dtype, batch, n_heads, n_kv_heads, head_dim, window, softcap, scale,
                                    split_keys, out, lse_out, stream, 0, q_dtype, out_dtype, &Lc, &pc);
    if (st != ATTN_OK) return st;
    st = decode_prepare(q, hot_k, hot_v, hot_len, nullptr, 0, 0, 0, hot_ring, nullptr, nullptr, ATTN_KV_F16, batch,
                        n_heads, n_kv_heads, head_dim, window, softcap, scale, split_keys, out, lse_out, stream,
                        hot_ring, q_dtype, out_dtype, &Lh, &ph);
    if (st != ATTN_OK) return st;
    size_t hot_off = 0, bytes = 0;
    if (!tiered_plans(batch, n_heads, n_kv_heads, head_dim, cold_max_kv, hot_ring, split_keys, &pc, &ph, &hot_off,
                      &bytes))
        return set_error(ATTN_EINVAL, "attn_decode_tiered: invalid sizes for the split plans");
    if ((st = check_workspace("attn_decode_tiered", workspace, workspace_bytes, bytes)) != ATTN_OK) return st;
    int* err = device_error_word();
    if (!err) return set_error(ATTN_ECUDA, "attn_decode_tiered: no CUDA device / error word");
    // the window counts positions over both tiers (tier_range): the raw value
    Lc.tier = 1;
    Lc.hot_len = hot_len;
    Lc.window = window;
    Lh.tier = 2;
    Lh.hot_len = hot_len;
    Lh.hot_start = hot_start;
    Lh.window = window;
    Lc.workspace = workspace;
    Lc.workspace_bytes = hot_off;
    Lh.workspace = static_cast<uint8_t*>(workspace) + hot_off;
    Lh.workspace_bytes = bytes - hot_off;
    Lc.err_word = Lh.err_word = err;
    return launch_decode_tiered(Lc, pc, Lh, ph);
}

attn_status attn_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_len,
                        const int32_t* page_table, int page_size, int max_pages_per_seq, int n_pages, int max_kv,
                        const void* k_scales, const void* v_scales, attn_kv_dtype kv_dtype, int batch, int n_heads,
                        int n_kv_heads, int head_dim, int window, float softcap, float scale, int split_keys,
                        void* out, float* lse_out, void* workspace, size_t workspace_bytes, void* stream) {
    return decode_entry(q, k_cache, v_cache, kv_len, page_table, page_size, max_pages_per_seq, n_pages, max_kv,
                        k_scales, v_scales, kv_dtype, batch, n_heads, n_kv_heads, head_dim, window, softcap, scale,
                        split_keys, out, lse_out, workspace, workspace_bytes, stream, 0);
}

attn_status attn_decode_ex(const void* q, attn_dtype q_dtype, const void* k_cache, const void* v_cache,
                           const int32_t* kv_len, const int32_t* page_table, int page_size, int max_pages_per_seq,
                           int n_pages, int max_kv, int ring_size, const void* k_scales, const void* v_scales,
                           attn_kv_dtype kv_dtype, int batch, int n_heads, int n_kv_heads, int head_dim, int window,
                           float softcap, float scale, int split_keys, void* out, attn_dtype out_dtype,
                           float* lse_out, void* workspace, size_t workspace_bytes, void* stream) {
    if (ring_size != 0) {
        if (ring_size < 16 || ring_size % 16 != 0)
            return set_error(ATTN_EUNSUPPORTED, "attn_decode_ex: ring_size %d must be a positive multiple of 16",
                             ring_size);
        if (page_table) return set_error(ATTN_EINVAL, "attn_decode_ex: a ring cache takes no page table");
        max_kv = ring_size;
    }
    return decode_entry(q, k_cache, v_cache, kv_len, page_table, page_size, max_pages_per_seq, n_pages, max_kv,
                        k_scales, v_scales, kv_dtype, batch, n_heads, n_kv_heads, head_dim, window, softcap, scale,
                        split_keys, out, lse_out, workspace, workspace_bytes, stream, ring_size, q_dtype, out_dtype);
}

attn_status attn_decode_ring(const void* q, const void* k_ring, const void* v_ring, const int32_t* seq_len,
                             int ring_size, const void* k_scales, const void* v_scales, attn_kv_dtype kv_dtype,
                             int batch, int n_heads, int n_kv_heads, int head_dim, int window, float softcap,
                             float scale, int split_keys, void* out, float* lse_out, void* workspace,
                             size_t workspace_bytes, void* stream) {
    if (ring_size < 16 || ring_size % 16 != 0)
        return set_error(ATTN_EUNSUPPORTED, "attn_decode_ring: ring_size %d must be a positive multiple of 16",
                         ring_size);
    return decode_entry(q, k_ring, v_ring, seq_len, nullptr, 0, 0, 0, ring_size, k_scales, v_scales, kv_dtype,
                        batch, n_heads, n_kv_heads, head_dim, window, softcap, scale, split_keys, out, lse_out,
                        workspace, workspace_bytes, stream, ring_size);
}

attn_status attn_prefill(const void* q, const void* k, const void* v, int seq_len, int n_heads, int n_kv_heads,
                         int head_dim, int causal, int window, float softcap, float scale, void* out, float* lse_out,
                         void* stream) {
    if (!q || !k || !v || !out) return set_error(ATTN_EINVAL, "attn_prefill: q, k, v and out must be non-null");
    if (seq_len < 0 || n_heads <= 0 || n_kv_heads <= 0)
        return set_error(ATTN_EINVAL, "attn_prefill: seq_len >= 0 and positive head counts required");
    if (n_heads % n_kv_heads != 0)
        return set_error(ATTN_EINVAL, "attn_prefill: n_heads (%d) must be a multiple of n_kv_heads (%d)", n_heads,
                         n_kv_heads);
    if (n_heads > 65535) return set_error(ATTN_EUNSUPPORTED, "attn_prefill: n_heads above 65535");
    if ((seq_len + 127) / 128 > 65535)
        return set_error(ATTN_EUNSUPPORTED, "attn_prefill: seq_len above %d", 65535 * 128);
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return set_error(ATTN_EUNSUPPORTED, "attn_prefill: head_dim %d not supported (64, 128, 256)", head_dim);
    if (window < 0) return set_error(ATTN_EINVAL, "attn_prefill: window must be >= 0 (0 = off)");
    if (!(softcap >= 0.f) || !std::isfinite(softcap))
        return set_error(ATTN_EINVAL, "attn_prefill: softcap must be finite and >= 0 (0 = off)");
    if (!std::isfinite(scale)) return set_error(ATTN_EINVAL, "attn_prefill: scale must be finite");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
        return set_error(ATTN_EINVAL, "attn_prefill: q, k, v and out must be 16-byte aligned");
    if (seq_len == 0) return ATTN_OK;
    int* err = device_error_word();
    if (!err) return set_error(ATTN_ECUDA, "attn_prefill: no CUDA device / error word");
    PrefillLaunch L;
    L.q = q;
    L.k = k;
    L.v = v;
    L.out = out;
    L.lse = lse_out;
    L.S = seq_len;
    L.Hq = n_heads;
    L.Hkv = n_kv_heads;
    L.D = head_dim;
    L.causal = causal != 0;
    L.window = window;
    L.softcap = softcap;
    L.scale = scale;
    L.err_word = err;
    L.stream = static_cast<cudaStream_t>(stream);
    return launch_prefill(L);
}

attn_status attn_prefill_paged(const void* q, const void* k_cache, const void* v_cache, const int32_t* q_start,
                               const int32_t* kv_len, const int32_t* page_table, int page_size,
                               int max_pages_per_seq, int n_pages, int batch, int total_q, int max_q, int n_heads,
                               int n_kv_heads, int head_dim, int window, float softcap, float scale, void* out,
                               float* lse_out, void* stream) {
    if (!q || !k_cache || !v_cache || !q_start || !kv_len || !page_table || !out)
        return set_error(ATTN_EINVAL, "attn_prefill_paged: q, caches, q_start, kv_len, page_table and out must be "
                                      "non-null");
    if (batch <= 0 || n_heads <= 0 || n_kv_heads <= 0 || total_q < 0 || max_q < 0)
        return set_error(ATTN_EINVAL, "attn_prefill_paged: positive batch and head counts, total_q/max_q >= 0 "
                                      "required");
    if (n_heads % n_kv_heads != 0)
        return set_error(ATTN_EINVAL, "attn_prefill_paged: n_heads (%d) must be a multiple of n_kv_heads (%d)",
                         n_heads, n_kv_heads);
    if (n_heads > 65535 || batch > 65535)
        return set_error(ATTN_EUNSUPPORTED, "attn_prefill_paged: n_heads and batch must be at most 65535");
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return set_error(ATTN_EUNSUPPORTED, "attn_prefill_paged: head_dim %d not supported (64, 128, 256)",
                         head_dim);
    if (page_size < 8 || (page_size & (page_size - 1)) != 0)
        return set_error(ATTN_EUNSUPPORTED, "attn_prefill_paged: page_size %d must be a power of two >= 8",
                         page_size);
    if (max_pages_per_seq <= 0 || n_pages <= 0)
        return set_error(ATTN_EINVAL, "attn_prefill_paged: max_pages_per_seq and n_pages must be positive");
    if (window < 0) return set_error(ATTN_EINVAL, "attn_prefill_paged: window must be >= 0 (0 = off)");
    if (!(softcap >= 0.f) || !std::isfinite(softcap))
        return set_error(ATTN_EINVAL, "attn_prefill_paged: softcap must be finite and >= 0 (0 = off)");
    if (!std::isfinite(scale)) return set_error(ATTN_EINVAL, "attn_prefill_paged: scale must be finite");
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
        return set_error(ATTN_EINVAL, "attn_prefill_paged: q, caches and out must be 16-byte aligned");
    if (total_q == 0 || max_q == 0) return ATTN_OK;
    int* err = device_error_word();
    if (!err) return set_error(ATTN_ECUDA, "attn_prefill_paged: no CUDA device / error word");
    PrefillLaunch L;
    L.q = q;
    L.k = k_cache;
    L.v = v_cache;
    L.out = out;
    L.lse = lse_out;
    L.S = 0;
    L.Hq = n_heads;
    L.Hkv = n_kv_heads;
    L.D = head_dim;
    L.causal = 1;
    L.window = window;
    L.softcap = softcap;
    L.scale = scale;
    L.err_word = err;
    L.stream = static_cast<cudaStream_t>(stream);
    L.paged = 1;
    L.q_start = q_start;
    L.kv_len = kv_len;
    L.page_table = page_table;
    L.page_size = page_size;
    L.max_pages = max_pages_per_seq;
    L.n_pages = n_pages;
    L.B = batch;
    L.total_q = total_q;
    L.max_q = max_q;
    return launch_prefill(L);
}

attn_status attn_decode_validate(const int32_t* kv_len, const int32_t* page_table, int batch, int page_size,
                                 int max_pages_per_seq, int n_pages, int max_kv, int* bad_seq, void* stream) {
    if (!kv_len || batch <= 0 || max_kv <= 0)
        return set_error(ATTN_EINVAL, "attn_decode_validate: kv_len, batch > 0 and max_kv > 0 required");
    if (page_table && (!pow2(page_size) || max_pages_per_seq <= 0 || n_pages <= 0))
        return set_error(ATTN_EINVAL, "attn_decode_validate: bad paged-layout sizes");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int zero = 0, big = 0x7fffffff;
    int cap = max_kv;
    if (page_table && (long)max_pages_per_seq * page_size < cap) cap = max_pages_per_seq * page_size;
    if (cudaMemcpyToSymbolAsync(g_validate_code, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_validate_seq, &big, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return set_error(ATTN_ECUDA, "attn_decode_validate: reset failed");
    validate_kernel<<<(batch + 127) / 128, 128, 0, s>>>(kv_len, page_table, batch, page_size, max_pages_per_seq,
                                                      n_pages, cap);
    int code = 0, seq = 0;
    if (cudaMemcpyFromSymbolAsync(&code, g_validate_code, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyFromSymbolAsync(&seq, g_validate_seq, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return set_error(ATTN_ECUDA, "attn_decode_validate: %s", cudaGetErrorString(cudaGetLastError()));
    if (code == 0) return ATTN_OK;
    if (bad_seq) *bad_seq = seq;
    return set_error((attn_status)code, "attn_decode_validate: sequence %d has %s", seq,
                     code == ATTN_EINVAL ? "kv_len <= 0" : "kv_len above capacity or a page id out of range");
}

attn_status attn_testing_set_waits(unsigned long long wait_limit_ns, int stall_first_tile) {
    if (stall_first_tile != 0 && stall_first_tile != 1)
        return set_error(ATTN_EINVAL, "attn_testing_set_waits: stall_first_tile must be 0 or 1");
    const unsigned long long limit = wait_limit_ns ? wait_limit_ns : 4000000000ull;
    attn_status st = set_test_controls_prefill(limit, stall_first_tile);
    if (st == ATTN_OK) st = set_test_controls_decode(limit, stall_first_tile);
    return st;
}

attn_status attn_device_status(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int v = 0;
    const int zero = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess)
        return set_error(ATTN_ECUDA, "attn_device_status: %s", cudaGetErrorString(cudaGetLastError()));
    if (v == kErrBadPage)
        return set_error(ATTN_EBOUNDS, "attn_decode read a page id outside the pool (page 0 was used instead)");
    if (v) return set_error(ATTN_ETIMEOUT, "a kernel abandoned a pipeline wait (code %d)", v);
    return ATTN_OK;
}

}  // extern "C"
