// decode_direct.cu -- one-launch decode of small calls.
//
// Same problem as the split kernels of decode.cu (doppler
// src/gpu/kernels/attention.js: executeAttention's decode variants; run.js
// runLayerAttentionGPU: the query at position kvLen-1 and the sliding-window
// clamp; executeAttentionTieredQuant's int8 codes with separate K and V
// scales).  When every sequence keeps only a few hundred keys, splitting buys
// nothing: the split kernel's pipeline start-up, its partials and the combine
// launch are most of such a call.  Here one CTA takes one (sequence, kv head)
// pair with the G query heads that read it and computes the exact softmax in
// shared memory, in one launch and without the workspace:
//   1. q of the G heads, times the logit factor, into shared memory;
//   2. each thread takes whole keys: it asks L2 for the key's V row, reads
//      its K row (and int8 scales), forms the G scores (capped when a softcap
//      is set) and keeps them in shared memory;
//   3. one warp per head: row max, exponentials, row sum;
//   4. each warp takes KS keys at a time (D/E lanes a key, E dims a lane) and
//      accumulates p * V for the G heads; the key groups of a warp are added
//      with shuffles, the 8 warps in shared memory, and the sums divided by
//      the row sum.
// Scores, weights and sums are fp32 (p is not rounded to f16), so the result
// agrees with the split path to within the rounding of either.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "attn_internal.h"
#include "decode_range.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kDirectMaxKeys = 512;      // kept keys per sequence this kernel takes
constexpr int kDirectMaxGD = 1024;       // G * D: query heads per kv head times head dim
constexpr int kDirectThreads = 256;
constexpr int kDirectWarps = kDirectThreads / 32;
constexpr int kDirectMaxG = kDirectMaxGD / 64;
// Above these sizes the split path streams the cache faster than one CTA per
// (sequence, kv head) does (measured on GB300): (sequence, kv head, key, dim)
// elements in the call at most 2^24 for D = 64, 2^23 for f16 D = 128, 2^22
// otherwise; int8 caches also at most 2^15 (key, dim) elements per sequence,
// where the CUDA-core split kernel is quicker still.
constexpr long direct_max_elems(int D, bool int8) {
    return D == 64 ? (1L << 24) : (D == 128 && !int8) ? (1L << 23) : (1L << 22);
}
constexpr long kDirectMaxSeqElemsI8 = 1L << 15;
constexpr float kLog2e = 1.4426950408889634f;

struct DirectArgs {
    const void* q;            // f16 or f32 [B, Hq, D]
    const void* k;            // f16 or int8 codes: contiguous [B, rows, Hkv, D] or pool [n_pages, P, Hkv, D]
    const void* v;
    const __half* k_scales;   // int8: [B, Hkv, rows] or [n_pages, Hkv, P]
    const __half* v_scales;
    const int32_t* kv_len;
    const int32_t* page_table;
    void* out;                // f16 or f32 [B, Hq, D]
    float* lse;               // [B, Hq] or null
    int Hq, Hkv, G;
    int cap_eff, window, ring;
    int rows;                 // contiguous: token rows per sequence (max_kv, or the ring size)
    int paged, P, logP, max_pages, n_pages;
    int q_f32, out_f32;
    float qscale;             // multiplies q: scale*log2e (no cap) or scale/c (cap)
    float cap_log2;           // c*log2e, 0 when the cap is off
    int* err;
};

// Shared memory of one CTA (floats unless noted): q [G][D]; per key its row's
// element offset (int64) and its int8 V scale; m and l of each head; then the
// scores [G][kDirectMaxKeys], reused after step 4 for the warps' partial
// outputs [8][G][D].
constexpr int direct_union_floats(int G, int D) {
    return G * kDirectMaxKeys > kDirectWarps * G * D ? G * kDirectMaxKeys : kDirectWarps * G * D;
}
constexpr size_t direct_smem_bytes(int G, int D) {
    return (size_t)G * D * 4 + (size_t)kDirectMaxKeys * 8 + (size_t)kDirectMaxKeys * 4 + 2 * kDirectMaxG * 4 +
           (size_t)direct_union_floats(G, D) * 4;
}
static_assert(direct_smem_bytes(kDirectMaxGD / 64, 64) <= 48 * 1024 &&
                  direct_smem_bytes(kDirectMaxGD / 128, 128) <= 48 * 1024 &&
                  direct_smem_bytes(kDirectMaxGD / 256, 256) <= 48 * 1024,
              "direct decode fits the default shared-memory limit");

// int8 code j (0..3) of a 32-bit word, as a float
__device__ __forceinline__ float code_of(uint32_t w, int j) { return (float)((int)(w << (24 - 8 * j)) >> 24); }

// E consecutive values (element offset off) of a K/V row, f16 or int8 codes,
// as floats
template <int E, bool I8>
__device__ __forceinline__ void load_vals(const void* base, long long off, float (&f)[E]) {
    if constexpr (I8) {
        const int8_t* p = static_cast<const int8_t*>(base) + off;
        if constexpr (E == 8) {
            const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                f[j] = code_of(w.x, j);
                f[4 + j] = code_of(w.y, j);
            }
        } else {
            static_assert(E == 4, "4 or 8 values");
            const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(p));
#pragma unroll
            for (int j = 0; j < 4; ++j) f[j] = code_of(w, j);
        }
    } else {
        const __half* p = static_cast<const __half*>(base) + off;
        if constexpr (E == 8) {
            const uint4 w = __ldg(reinterpret_cast<const uint4*>(p));
            const __half2* h = reinterpret_cast<const __half2*>(&w);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 x = __half22float2(h[e]);
                f[2 * e] = x.x;
                f[2 * e + 1] = x.y;
            }
        } else {
            static_assert(E == 4, "4 or 8 values");
            const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
            const __half2* h = reinterpret_cast<const __half2*>(&w);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float2 x = __half22float2(h[e]);
                f[2 * e] = x.x;
                f[2 * e + 1] = x.y;
            }
        }
    }
}

// GM: the query heads per kv head this instantiation holds in registers
// (G <= GM; the launch picks the smallest power of two).
template <int D, bool I8, int GM>
__global__ void __launch_bounds__(kDirectThreads) decode_direct_kernel(const DirectArgs A) {
    constexpr int E = (GM * 8 <= 64) ? 8 : 4;   // dims per lane in step 4
    constexpr int LPK = D / E;                  // lanes per key in step 4
    constexpr int KS = 32 / LPK;                // keys per warp step
    static_assert(LPK <= 32 && KS * LPK == 32, "step-4 lane layout");
    extern __shared__ __align__(16) unsigned char dsm[];
    const int G = A.G;
    float* qs = reinterpret_cast<float*>(dsm);
    long long* roff = reinterpret_cast<long long*>(qs + G * D);
    float* vsc = reinterpret_cast<float*>(roff + kDirectMaxKeys);
    float* mh = vsc + kDirectMaxKeys;
    float* lh = mh + kDirectMaxG;
    float* sc = lh + kDirectMaxG;   // scores / weights, then the partial outputs
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x / A.Hkv, g = blockIdx.x - b * A.Hkv;
    const int h0 = g * G;

    int start, end;
    seq_range(__ldg(&A.kv_len[b]), A.cap_eff, A.window, start, end);
    // the host sends only calls whose sequences keep at most kDirectMaxKeys keys
    const int n = min(end - start, kDirectMaxKeys);

    // 1. q of the group, scaled
    const size_t qbase = ((size_t)b * A.Hq + h0) * D;
    for (int i = tid; i < G * D; i += kDirectThreads) {
        const float x = A.q_f32 ? __ldg(static_cast<const float*>(A.q) + qbase + i)
                                : __half2float(static_cast<const __half*>(A.q)[qbase + i]);
        qs[i] = x * A.qscale;
    }
    __syncthreads();

    // 2. scores: thread i takes keys i, i+256
#pragma unroll 2
    for (int i = tid; i < n; i += kDirectThreads) {
        const int t = start + i;
        long long row, srow;   // token row of the [rows, Hkv, D] view; scale index
        if (A.paged) {
            int page = __ldg(&A.page_table[(size_t)b * A.max_pages + (t >> A.logP)]);
            if (page < 0 || page >= A.n_pages) {
                // a page id outside the pool: read page 0 instead and report it
                atomicExch(A.err, kErrBadPage);
                page = 0;
            }
            const int pr = t & (A.P - 1);
            row = (long long)page * A.P + pr;
            srow = ((long long)page * A.Hkv + g) * A.P + pr;
        } else {
            const int r = A.ring > 0 ? t % A.ring : t;
            row = (long long)b * A.rows + r;
            srow = ((long long)b * A.Hkv + g) * A.rows + r;
        }
        const long long off = (row * A.Hkv + g) * D;
        roff[i] = off;
        constexpr int RB = D * (I8 ? 1 : 2);   // bytes of a V row
        const char* vrow = static_cast<const char*>(A.v) + off * (I8 ? 1 : 2);
#pragma unroll
        for (int c = 0; c < RB; c += 128) prefetch_l2(vrow + c);
        float s[GM];
#pragma unroll
        for (int h = 0; h < GM; ++h) s[h] = 0.f;
#pragma unroll
        for (int c = 0; c < D; c += 64) {   // 64 dims at a time: 8 loads of 8 values in flight
            float f[8][8];
#pragma unroll
            for (int j = 0; j < 8; ++j) load_vals<8, I8>(A.k, off + c + 8 * j, f[j]);
#pragma unroll
            for (int h = 0; h < GM; ++h) {
                if (h < G) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 qa = *reinterpret_cast<const float4*>(&qs[h * D + c + 8 * j]);
                        const float4 qb = *reinterpret_cast<const float4*>(&qs[h * D + c + 8 * j + 4]);
                        s[h] += qa.x * f[j][0] + qa.y * f[j][1] + qa.z * f[j][2] + qa.w * f[j][3] +
                                qb.x * f[j][4] + qb.y * f[j][5] + qb.z * f[j][6] + qb.w * f[j][7];
                    }
                }
            }
        }
        float ks = 1.f;
        if constexpr (I8) {
            ks = __half2float(A.k_scales[srow]);
            vsc[i] = __half2float(A.v_scales[srow]);
        }
#pragma unroll
        for (int h = 0; h < GM; ++h) {
            if (h < G) {
                float x = s[h] * ks;
                if (A.cap_log2 > 0.f) x = A.cap_log2 * tanh_abs_accurate(x);
                sc[h * kDirectMaxKeys + i] = x;   // log2-domain logit
            }
        }
    }
    __syncthreads();

    // 3. softmax of each head: max, weights 2^(s - m), sum
    for (int h = warp; h < G; h += kDirectWarps) {
        float* srow = sc + h * kDirectMaxKeys;
        float m = -INFINITY;
        for (int i = lane; i < n; i += 32) m = fmaxf(m, srow[i]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.f;
        if (m > -INFINITY) {
            for (int i = lane; i < n; i += 32) {
                const float p = ex2_approx(srow[i] - m);
                srow[i] = p;
                l += p;
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            mh[h] = m;
            lh[h] = l;
        }
    }
    __syncthreads();

    // 4. p * V: key group kg of warp w takes keys (w * KS + kg) + 8 * KS * step;
    // lane dl of the group owns dims dl*E .. dl*E+E-1
    const int kg = lane / LPK, dl = lane - kg * LPK;
    float acc[GM][E];
#pragma unroll
    for (int h = 0; h < GM; ++h)
#pragma unroll
        for (int j = 0; j < E; ++j) acc[h][j] = 0.f;
#pragma unroll 4
    for (int i = warp * KS + kg; i < n; i += kDirectWarps * KS) {
        float v[E];
        load_vals<E, I8>(A.v, roff[i] + dl * E, v);
        const float vs = I8 ? vsc[i] : 1.f;
#pragma unroll
        for (int h = 0; h < GM; ++h) {
            if (h < G) {
                const float p = sc[h * kDirectMaxKeys + i] * vs;
#pragma unroll
                for (int j = 0; j < E; ++j) acc[h][j] += p * v[j];
            }
        }
    }
#pragma unroll
    for (int o = LPK; o < 32; o <<= 1)
#pragma unroll
        for (int h = 0; h < GM; ++h)
#pragma unroll
            for (int j = 0; j < E; ++j) acc[h][j] += __shfl_xor_sync(0xffffffffu, acc[h][j], o);
    __syncthreads();   // every warp is done with the weights: reuse their space
    float* part = sc;  // [8][G][D]
    if (kg == 0) {
#pragma unroll
        for (int h = 0; h < GM; ++h)
            if (h < G) {
#pragma unroll
                for (int j = 0; j < E; ++j) part[(warp * G + h) * D + dl * E + j] = acc[h][j];
            }
    }
    __syncthreads();
    const size_t obase = ((size_t)b * A.Hq + h0) * D;
    for (int i = tid; i < G * D; i += kDirectThreads) {
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < kDirectWarps; ++w) o += part[w * G * D + i];
        const float l = lh[i / D];
        o = l > 0.f ? o / l : 0.f;
        if (A.out_f32)
            static_cast<float*>(A.out)[obase + i] = o;
        else
            static_cast<__half*>(A.out)[obase + i] = __float2half_rn(o);
    }
    if (A.lse && tid < G) {
        const float l = lh[tid];
        A.lse[(size_t)b * A.Hq + h0 + tid] = l > 0.f ? (mh[tid] + __log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
}

// Most keys a sequence of the call can keep: the bound the kernel relies on.
int kept_keys_bound(const DecodeLaunch& L) {
    if (L.ring > 0) return L.window;   // clamped to the ring by the entry point
    return (L.window > 0 && L.window < L.max_kv) ? L.window : L.max_kv;
}

template <int D, bool I8, int GM>
attn_status launch_direct_t(const DecodeLaunch& L) {
    const bool paged = L.page_table != nullptr;
    const int cap_layout = paged ? L.max_pages * L.page_size : L.max_kv;
    DirectArgs a;
    a.q = L.q;
    a.k = L.k;
    a.v = L.v;
    a.k_scales = static_cast<const __half*>(L.k_scales);
    a.v_scales = static_cast<const __half*>(L.v_scales);
    a.kv_len = L.kv_len;
    a.page_table = L.page_table;
    a.out = L.out;
    a.lse = L.lse;
    a.Hq = L.Hq;
    a.Hkv = L.Hkv;
    a.G = L.Hq / L.Hkv;
    a.cap_eff = L.ring > 0 ? (1 << 30) : (cap_layout < L.max_kv ? cap_layout : L.max_kv);
    a.window = L.window;
    a.ring = L.ring;
    a.rows = L.max_kv;
    a.paged = paged;
    a.P = paged ? L.page_size : 0;
    a.logP = 0;
    while (paged && (1 << a.logP) < L.page_size) ++a.logP;
    a.max_pages = L.max_pages;
    a.n_pages = paged ? L.n_pages : 0;
    a.q_f32 = L.q_f32;
    a.out_f32 = L.out_f32;
    const bool capped = L.softcap > 0.f;
    a.qscale = capped ? L.scale / L.softcap : L.scale * kLog2e;
    a.cap_log2 = capped ? L.softcap * kLog2e : 0.f;
    a.err = L.err_word;
    const size_t smem = direct_smem_bytes(a.G, D);
    const int grid = L.B * L.Hkv;
    if (trace_enabled())
        trace("decode_direct_kernel<D=%d,int8=%d,GM=%d> grid=%d block=%d smem=%zu B=%d Hq=%d Hkv=%d layout=%s "
              "max_keys=%d (one CTA per (sequence, kv head), no split, no combine)",
              D, (int)I8, GM, grid, kDirectThreads, smem, L.B, L.Hq, L.Hkv,
              paged ? "paged" : L.ring > 0 ? "ring" : "contiguous", kept_keys_bound(L));
    decode_direct_kernel<D, I8, GM><<<grid, kDirectThreads, smem, L.stream>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(ATTN_ECUDA, "direct decode launch failed: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

template <int D, bool I8>
attn_status launch_direct_g(const DecodeLaunch& L) {
    const int G = L.Hq / L.Hkv;   // <= kDirectMaxGD / D (direct_decode_fits)
    if (G <= 1) return launch_direct_t<D, I8, 1>(L);
    if (G <= 2) return launch_direct_t<D, I8, 2>(L);
    if (G <= 4) return launch_direct_t<D, I8, 4>(L);
    if constexpr (D <= 128) {
        if (G <= 8) return launch_direct_t<D, I8, 8>(L);
    }
    if constexpr (D == 64) return launch_direct_t<D, I8, 16>(L);
    return set_error(ATTN_EUNSUPPORTED, "direct decode: %d query heads per kv head at head_dim %d", G, D);
}

}  // namespace

bool direct_decode_fits(const DecodeLaunch& L) {
    const long n = kept_keys_bound(L);
    const long ctas = (long)L.B * L.Hkv;
    return L.split_keys == 0 && L.tier == 0 && n <= kDirectMaxKeys && (L.Hq / L.Hkv) * L.D <= kDirectMaxGD &&
           ctas * n * L.D <= direct_max_elems(L.D, L.int8) && (!L.int8 || n * L.D <= kDirectMaxSeqElemsI8);
}

attn_status launch_direct(const DecodeLaunch& L) {
    switch (L.D) {
        case 64: return L.int8 ? launch_direct_g<64, true>(L) : launch_direct_g<64, false>(L);
        case 128: return L.int8 ? launch_direct_g<128, true>(L) : launch_direct_g<128, false>(L);
        case 256: return L.int8 ? launch_direct_g<256, true>(L) : launch_direct_g<256, false>(L);
        default: return set_error(ATTN_EUNSUPPORTED, "head_dim %d not supported (64, 128, 256)", L.D);
    }
}

}  // namespace attn
