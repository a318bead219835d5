// decode.cu -- split-KV flash-decode over an f16 or int8 KV cache
// (contiguous or paged), with GQA, sliding window, softcap, online softmax
// and a log-sum-exp combine pass.
//
// Problem (doppler src/gpu/kernels/attention.js: executeAttention's decode
// variants with the per-call kvLen buffer and the paged layout's page table
// and pageSize; executeAttentionTieredQuant's int8 K/V with separate scale
// buffers; doppler run.js runLayerAttentionGPU: decode query at position
// kvLen-1 and the sliding-window clamp).  The pages' decode kernels give one
// workgroup per head and reduce with subgroup max/add; here the KV range of
// each (sequence, kv head, head group) is cut into fixed-size splits so the
// whole GPU streams the cache:
//
//   decode_split_kernel   persistent, one CTA per SM.  A producer warp streams
//                         16-token K/V tiles (plus int8 scales) into a ring
//                         of shared-memory slots with TMA, following the page
//                         table; 7 consumer warps each take whole tiles and
//                         keep an online softmax per query head.  Inside a
//                         warp, 8 (or 16) lanes share one key: each lane holds
//                         D/8 dims of all GH query heads of the group in
//                         registers, so a K row is read once for the GH heads
//                         (GQA: q-head h reads kv-head h / G).  Partial dots
//                         are reduce-scattered across the key's lanes with
//                         warp shuffles; int8 codes become floats in registers
//                         and the per-token scales are applied once per key.
//                         At the end of a split the 7 warps merge their
//                         (max, sum, o) states in shared memory and the split
//                         writes (lse, o / l) to the workspace.
//   decode_combine_kernel merges the splits of each (sequence, head) with the
//                         log-sum-exp rule and writes f16 output (+ lse).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int T = 16;                     // keys per tile (one ring slot)
constexpr int NCW = 7;                    // consumer warps (+1 producer: 256 threads, 255 registers each)
constexpr int kDecThreads = (NCW + 1) * 32;
constexpr int kSmemBudget = 226 * 1024;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;

template <int D, bool I8, int GH>
struct DecCfg {
    static constexpr int ESZ = I8 ? 1 : 2;
    static constexpr int RB = D * ESZ;                       // bytes of one K/V row
    static constexpr int LPK = (D == 256) ? 16 : 8;          // lanes sharing one key
    static constexpr int LOG_LPK = (LPK == 16) ? 4 : 3;
    static constexpr int KPS = 32 / LPK;                     // keys per warp step
    static constexpr int NSTEP = T / KPS;
    static constexpr int E = D / LPK;                        // elements per lane
    static constexpr int VB = (RB / LPK) < 16 ? (RB / LPK) : 16;   // bytes per vector load
    static constexpr int EV = VB / ESZ;                      // elements per vector
    static constexpr int NV = E / EV;                        // vectors per lane per row
    static constexpr int LOG_GH = (GH == 4) ? 2 : (GH == 2) ? 1 : 0;
    static constexpr int SCALE_BYTES = I8 ? 256 : 0;         // per tensor per slot
    static constexpr int SLOT = 2 * T * RB + 2 * SCALE_BYTES;
    static constexpr int OFF_PREFIX = 0;
    static constexpr int PREFIX_BYTES = ((kDecodeMaxBatch + 1) * 4 + 127) / 128 * 128;
    static constexpr int OFF_MERGE = OFF_PREFIX + PREFIX_BYTES;
    static constexpr int MERGE_BYTES = (NCW * GH * (D + 2) * 4 + 127) / 128 * 128;
    static constexpr int OFF_MISC = OFF_MERGE + MERGE_BYTES;   // scan scratch (32 ints) + abort flag
    static constexpr int MISC_BYTES = 256;
    static constexpr int OFF_BARS = OFF_MISC + MISC_BYTES;
    static constexpr int NSLOT_RAW = (kSmemBudget - OFF_BARS - 2 * 32 * 8 - 1024) / SLOT;
    static constexpr int NSLOT = NSLOT_RAW > 32 ? 32 : NSLOT_RAW;
    static constexpr int OFF_RING = ((OFF_BARS + 2 * NSLOT * 8) + 1023) / 1024 * 1024;
    static constexpr int SMEM_USED = OFF_RING + NSLOT * SLOT;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;
    static_assert(NSLOT >= 10, "ring too small");
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
    static_assert(E % EV == 0 && E % 2 == 0, "lane layout");
};

struct DecArgs {
    const __half* q;
    const int32_t* kv_len;
    const int32_t* page_table;
    int32_t* ws_prefix;
    float* ws_lse;
    float* ws_o;
    int B, Hq, Hkv, G, HG, split, cap_eff, window, P, R, max_pages, n_pages, paged;
    float qscale;      // multiplies q: scale*log2e (no cap) or scale/c (cap)
    float cap_log2;    // c*log2e, 0 when the cap is off
    int* err;
};

// Range of kept keys of a sequence: [start, end).  The decode query sits at
// position L-1, so the causal mask keeps everything below L; a window keeps
// the W most recent tokens (run.js: kvLen = min(kvLen, W), kvStart = L - kvLen).
__device__ __forceinline__ void seq_range(int L, int cap_eff, int W, int& start, int& end) {
    L = min(max(L, 0), cap_eff);
    start = (W > 0) ? max(0, L - W) : 0;
    end = L;
}
// Splits of a sequence: aligned to the tile so that tiles start on multiples
// of 16 keys (and so on page boundaries for pages of >= 16 tokens).
__device__ __forceinline__ int seq_splits(int start, int end, int split) {
    if (end <= start) return 0;
    const int a = (start / T) * T;
    return (end - a + split - 1) / split;
}

struct Item {
    int b, g, hg, ks, ke, start, ntile;
};

__device__ __forceinline__ Item decode_item(int it, const int* pref, const DecArgs& A) {
    int lo = 0, hi = A.B;   // largest b with pref[b] <= it
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pref[mid] <= it) lo = mid; else hi = mid;
    }
    Item r;
    r.b = lo;
    int start, end;
    seq_range(__ldg(&A.kv_len[lo]), A.cap_eff, A.window, start, end);
    const int ns = seq_splits(start, end, A.split);
    const int rem = it - pref[lo];
    const int gh = rem / ns, s = rem - gh * ns;
    r.g = gh / A.HG;
    r.hg = gh - r.g * A.HG;
    const int a = (start / T) * T;
    r.ks = a + s * A.split;
    r.ke = min(r.ks + A.split, end);
    r.start = start;
    r.ntile = (r.ke - r.ks + T - 1) / T;
    return r;
}

// Exclusive prefix over sequences of their work-item counts (block-wide scan).
__device__ void build_prefix(const DecArgs& A, int* pref, int* scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    int carry = 0;
    for (int base = 0; base < A.B; base += blockDim.x) {
        const int b = base + threadIdx.x;
        int v = 0;
        if (b < A.B) {
            int start, end;
            seq_range(__ldg(&A.kv_len[b]), A.cap_eff, A.window, start, end);
            v = A.Hkv * A.HG * seq_splits(start, end, A.split);
        }
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) scratch[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = lane < nw ? scratch[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            scratch[lane] = w;
        }
        __syncthreads();
        const int woff = warp > 0 ? scratch[warp - 1] : 0;
        if (b < A.B) pref[b] = carry + woff + x - v;
        carry += scratch[nw - 1];
        __syncthreads();
    }
    if (threadIdx.x == 0) pref[A.B] = carry;
    __syncthreads();
}

// ---- packed fp32 helpers (sm_100 family f32x2 instructions)
__device__ __forceinline__ uint64_t pk(float2 a) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a.x), "f"(a.y));
    return r;
}
__device__ __forceinline__ float2 upk(uint64_t r) {
    float2 a;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a.x), "=f"(a.y) : "l"(r));
    return a;
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(pk(a)), "l"(pk(b)), "l"(pk(c)));
    return upk(d);
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk(a)), "l"(pk(b)));
    return upk(d);
}

// One lane's slice of a K or V row -> E floats (as E/2 pairs).
template <int D, bool I8, int GH>
__device__ __forceinline__ void load_row_slice(const uint8_t* row, int c, float2 (&x)[DecCfg<D, I8, GH>::E / 2]) {
    using C = DecCfg<D, I8, GH>;
#pragma unroll
    for (int v = 0; v < C::NV; ++v) {
        const uint8_t* src = row + (v * C::LPK + c) * C::VB;
        if constexpr (!I8) {
            static_assert(C::VB == 16, "f16 rows are read 16 bytes at a time");
            const uint4 w = *reinterpret_cast<const uint4*>(src);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                __half2 h2 = *reinterpret_cast<const __half2*>(&ws[i]);
                x[v * 4 + i] = __half22float2(h2);
            }
        } else {
            // int8 code u -> float: bytes biased to unsigned, placed in the low
            // mantissa bits of 2^23, then the bias 2^23 + 128 is subtracted.
            constexpr int NW = C::VB / 4;
            uint32_t ws[NW];
            if constexpr (NW == 4) {
                const uint4 w = *reinterpret_cast<const uint4*>(src);
                ws[0] = w.x; ws[1] = w.y; ws[2] = w.z; ws[3] = w.w;
            } else {
                const uint2 w = *reinterpret_cast<const uint2*>(src);
                ws[0] = w.x; ws[1] = w.y;
            }
            const float2 bias = make_float2(-8388736.0f, -8388736.0f);
#pragma unroll
            for (int i = 0; i < NW; ++i) {
                const uint32_t u = ws[i] ^ 0x80808080u;
                const float2 lo = make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540u)),
                                              __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541u)));
                const float2 hi = make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7542u)),
                                              __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7543u)));
                x[(v * C::EV) / 2 + 2 * i] = fadd2(lo, bias);
                x[(v * C::EV) / 2 + 2 * i + 1] = fadd2(hi, bias);
            }
        }
    }
}

template <int D, bool I8, int GH>
__global__ void __launch_bounds__(kDecThreads, 1)
decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_ks, const __grid_constant__ CUtensorMap tm_vs,
                    const DecArgs A) {
    using C = DecCfg<D, I8, GH>;
    constexpr int NSLOT = C::NSLOT, LPK = C::LPK, E = C::E;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int* pref = reinterpret_cast<int*>(smem + C::OFF_PREFIX);
    float* mb = reinterpret_cast<float*>(smem + C::OFF_MERGE);
    int* scratch = reinterpret_cast<int*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 128);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
    const uint32_t ring = smem_u32(smem + C::OFF_RING);
    auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
    auto empty_bar = [&](int s) { return smem_u32(&bars[NSLOT + s]); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    build_prefix(A, pref, scratch);   // ends with __syncthreads
    const int total = pref[A.B];
    if (blockIdx.x == 0) {
        for (int b = threadIdx.x; b <= A.B; b += blockDim.x) A.ws_prefix[b] = pref[b];
    }

    if (warp == NCW) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            if (I8) {
                tma_prefetch_desc(&tm_ks);
                tma_prefetch_desc(&tm_vs);
            }
        }
        const int NB = T / A.R;          // boxes per tile per tensor
        uint32_t gt = 0;
        int cache_b = -1, cache_base = -1, pid = -1;
        bool ok = true;
        for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
            const Item I = decode_item(it, pref, A);
            int start, end;
            seq_range(__ldg(&A.kv_len[I.b]), A.cap_eff, A.window, start, end);
            for (int i = 0; i < I.ntile; ++i, ++gt) {
                const int t0 = I.ks + i * T;
                const int slot = gt % NSLOT;
                int pi0 = 0, cb = 0;
                if (A.paged) {
                    pi0 = t0 / A.P;
                    cb = pi0 & ~31;
                    if (I.b != cache_b || cb != cache_base) {
                        const int idx = cb + lane;
                        pid = idx < A.max_pages ? __ldg(&A.page_table[(size_t)I.b * A.max_pages + idx]) : -1;
                        cache_b = I.b;
                        cache_base = cb;
                    }
                }
                int good = 1;
                if (lane == 0 && gt >= (uint32_t)NSLOT)
                    good = mbar_wait(empty_bar(slot), ((gt / NSLOT) - 1) & 1, abort_flag, A.err, kErrTimeoutSlot);
                good = __shfl_sync(0xffffffffu, good, 0);
                if (!good) { ok = false; break; }
                const uint32_t sb = ring + slot * C::SLOT;
                const int row0 = (A.paged && A.P >= T) ? (t0 % A.P) : (A.paged ? 0 : t0);
                uint32_t bytes = 0;
                // count the boxes first (lane 0 arms the barrier before any copy lands)
                int nbox = 0;
                if (!A.paged) {
                    nbox = 1;
                } else {
                    for (int r = 0; r < NB; ++r)
                        if ((pi0 + r) * A.P < end) nbox = r + 1;
                }
                bytes = nbox * A.R * (2 * C::RB + (I8 ? 4 : 0));
                if (lane == 0) mbar_arrive_expect_tx(full_bar(slot), bytes);
                for (int r = 0; r < nbox; ++r) {
                    int page = I.b;
                    if (A.paged) {
                        page = __shfl_sync(0xffffffffu, pid, pi0 + r - cb);
                        if (page < 0 || page >= A.n_pages) {
                            // a page id outside the pool: read page 0 instead and report it
                            if (lane == 0) atomicExch(A.err, kErrBadPage);
                            page = 0;
                        }
                    }
                    if (lane == 0) {
                        const int rr = row0;
                        tma_load_4d(sb + r * A.R * C::RB, &tm_k, full_bar(slot), 0, I.g, rr, page);
                        tma_load_4d(sb + T * C::RB + r * A.R * C::RB, &tm_v, full_bar(slot), 0, I.g, rr, page);
                        if (I8) {
                            tma_load_3d(sb + 2 * T * C::RB + r * 128, &tm_ks, full_bar(slot), rr, I.g, page);
                            tma_load_3d(sb + 2 * T * C::RB + C::SCALE_BYTES + r * 128, &tm_vs, full_bar(slot), rr,
                                        I.g, page);
                        }
                    }
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) {
            // let copies in flight land before shared memory is released
            volatile int never = 0;
            const uint32_t first = gt > (uint32_t)NSLOT ? gt - NSLOT : 0;
            for (uint32_t x = first; x < gt; ++x)
                mbar_wait(full_bar(x % NSLOT), (x / NSLOT) & 1, &never, A.err, kErrTimeoutLoad);
        }
    } else {
        // ---------------------------------------------------------------- consumers
        const int c = lane & (LPK - 1);          // position inside the key's lane group
        const int kk = lane >> C::LOG_LPK;       // key of the step handled by this group
        const int grp = lane & ~(LPK - 1);
        // reduce-scatter bookkeeping: slot s of this lane holds head s ^ rot
        int rot = 0;
#pragma unroll
        for (int k = 0; k < C::LOG_GH; ++k) rot |= ((c >> (C::LOG_LPK - 1 - k)) & 1) << (C::LOG_GH - 1 - k);
        int src_lane[GH];   // a lane of this group holding head h after the scatter
#pragma unroll
        for (int h = 0; h < GH; ++h) {
            int cl = 0;
#pragma unroll
            for (int k = 0; k < C::LOG_GH; ++k) cl |= ((h >> (C::LOG_GH - 1 - k)) & 1) << (C::LOG_LPK - 1 - k);
            src_lane[h] = grp | cl;
        }
        uint32_t gt_base = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < total; it += gridDim.x) {
            const Item I = decode_item(it, pref, A);
            // queries of the GH heads, pre-scaled, in this lane's dims and slot order
            float2 q2[GH][E / 2];
#pragma unroll
            for (int s = 0; s < GH; ++s) {
                const int head = I.g * A.G + I.hg * GH + (s ^ rot);
                const __half* qrow = A.q + ((size_t)I.b * A.Hq + head) * D;
#pragma unroll
                for (int v = 0; v < C::NV; ++v)
#pragma unroll
                    for (int e = 0; e < C::EV; e += 2) {
                        const int dim = (v * LPK + c) * C::EV + e;
                        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(qrow + dim));
                        q2[s][(v * C::EV + e) / 2] = make_float2(f.x * A.qscale, f.y * A.qscale);
                    }
            }
            float2 o2[GH][E / 2];
#pragma unroll
            for (int h = 0; h < GH; ++h)
#pragma unroll
                for (int j = 0; j < E / 2; ++j) o2[h][j] = make_float2(0.f, 0.f);
            float m = -INFINITY, l = 0.f;

            for (int i = warp; i < I.ntile; i += NCW) {
                const uint32_t gt = gt_base + i;
                const int slot = gt % NSLOT;
                bool got = ok && mbar_wait(full_bar(slot), (gt / NSLOT) & 1, abort_flag, A.err, kErrTimeoutLoad);
                got = __all_sync(0xffffffffu, got);   // keep the warp converged for the shuffles below
                if (!got) { ok = false; continue; }
                const int t0 = I.ks + i * T;
                const int v_lo = max(I.start - t0, 0);
                const int v_hi = min(I.ke - t0, T);
                const uint8_t* kt = smem + C::OFF_RING + slot * C::SLOT;
                const uint8_t* vt = kt + T * C::RB;
                const __half* kst = reinterpret_cast<const __half*>(kt + 2 * T * C::RB);
                const __half* vst = reinterpret_cast<const __half*>(kt + 2 * T * C::RB + C::SCALE_BYTES);

                float tsc[C::NSTEP];
#pragma unroll
                for (int st = 0; st < C::NSTEP; ++st) {
                    const int key = st * C::KPS + kk;
                    float2 kx[E / 2];
                    load_row_slice<D, I8, GH>(kt + key * C::RB, c, kx);
                    float acc[GH];
#pragma unroll
                    for (int s = 0; s < GH; ++s) {
                        float2 a = make_float2(0.f, 0.f);
#pragma unroll
                        for (int j = 0; j < E / 2; ++j) a = ffma2(q2[s][j], kx[j], a);
                        acc[s] = a.x + a.y;
                    }
                    // reduce-scatter: after it, slot 0 holds the full dot of head `rot`
#pragma unroll
                    for (int k = 0; k < C::LOG_GH; ++k) {
                        const int half = GH >> (k + 1);
                        const int dist = LPK >> (k + 1);
#pragma unroll
                        for (int s = 0; s < half; ++s) acc[s] += __shfl_xor_sync(0xffffffffu, acc[s + half], dist);
                    }
#pragma unroll
                    for (int dist = LPK >> (C::LOG_GH + 1); dist >= 1; dist >>= 1)
                        acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], dist);
                    float t = acc[0];
                    if (I8) t *= __half2float(kst[(key / A.R) * 64 + (key % A.R)]);
                    if (A.cap_log2 > 0.f) t = A.cap_log2 * tanh_abs_accurate(t);
                    tsc[st] = (key >= v_lo && key < v_hi) ? t : -INFINITY;
                }
                // tile max of this lane's head, across the key groups
                float tmax = -INFINITY;
#pragma unroll
                for (int st = 0; st < C::NSTEP; ++st) tmax = fmaxf(tmax, tsc[st]);
#pragma unroll
                for (int dist = LPK; dist < 32; dist <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, dist));
                const bool need = tmax > m + kRescaleThreshold || (m == -INFINITY && tmax > -INFINITY);
                if (__any_sync(0xffffffffu, need)) {
                    const float m_new = need ? fmaxf(tmax, m) : m;
                    const float alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - m_new);
#pragma unroll
                    for (int h = 0; h < GH; ++h) {
                        const float ah = __shfl_sync(0xffffffffu, alpha, src_lane[h]);
#pragma unroll
                        for (int j = 0; j < E / 2; ++j) o2[h][j] = make_float2(o2[h][j].x * ah, o2[h][j].y * ah);
                    }
                    l *= alpha;
                    m = m_new;
                }
                const float m_off = (m == -INFINITY) ? 0.f : m;
                float pv[C::NSTEP];
#pragma unroll
                for (int st = 0; st < C::NSTEP; ++st) {
                    const float p = ex2_approx(tsc[st] - m_off);
                    l += p;
                    pv[st] = p;
                    if (I8) {
                        const int key = st * C::KPS + kk;
                        const bool valid = key >= v_lo && key < v_hi;
                        pv[st] = valid ? p * __half2float(vst[(key / A.R) * 64 + (key % A.R)]) : 0.f;
                    }
                }
#pragma unroll
                for (int st = 0; st < C::NSTEP; ++st) {
                    const int key = st * C::KPS + kk;
                    float pg[GH];
#pragma unroll
                    for (int h = 0; h < GH; ++h) pg[h] = __shfl_sync(0xffffffffu, pv[st], src_lane[h]);
                    if (key >= v_lo && key < v_hi) {
                        float2 vx[E / 2];
                        load_row_slice<D, I8, GH>(vt + key * C::RB, c, vx);
#pragma unroll
                        for (int h = 0; h < GH; ++h) {
                            const float2 pp = make_float2(pg[h], pg[h]);
#pragma unroll
                            for (int j = 0; j < E / 2; ++j) o2[h][j] = ffma2(pp, vx[j], o2[h][j]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(slot));
            }
            gt_base += I.ntile;

            // ---- merge: lanes of a key group -> group 0, then warps via shared memory
#pragma unroll
            for (int dist = LPK; dist < 32; dist <<= 1) {
#pragma unroll
                for (int h = 0; h < GH; ++h)
#pragma unroll
                    for (int j = 0; j < E / 2; ++j) {
                        o2[h][j].x += __shfl_xor_sync(0xffffffffu, o2[h][j].x, dist);
                        o2[h][j].y += __shfl_xor_sync(0xffffffffu, o2[h][j].y, dist);
                    }
                l += __shfl_xor_sync(0xffffffffu, l, dist);
            }
            float* mb_m = mb;                         // [NCW][GH]
            float* mb_l = mb + NCW * GH;              // [NCW][GH]
            float* mb_o = mb + 2 * NCW * GH;          // [NCW][GH][D]
            if (lane < LPK) {
#pragma unroll
                for (int h = 0; h < GH; ++h)
#pragma unroll
                    for (int v = 0; v < C::NV; ++v)
#pragma unroll
                        for (int e = 0; e < C::EV; e += 2) {
                            const int dim = (v * LPK + c) * C::EV + e;
                            *reinterpret_cast<float2*>(&mb_o[(warp * GH + h) * D + dim]) = o2[h][(v * C::EV + e) / 2];
                        }
                if ((c & ((LPK >> C::LOG_GH) - 1)) == 0) {   // one writer per head
                    mb_m[warp * GH + rot] = m;
                    mb_l[warp * GH + rot] = l;
                }
            }
            named_bar_sync(1, NCW * 32);
            for (int idx = threadIdx.x; idx < GH * D; idx += NCW * 32) {
                const int h = idx / D, d = idx - h * D;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < NCW; ++w) M = fmaxf(M, mb_m[w * GH + h]);
                float wsum = 0.f, acc = 0.f;
                if (M > -INFINITY) {
#pragma unroll
                    for (int w = 0; w < NCW; ++w) {
                        const float mw = mb_m[w * GH + h];
                        if (mw > -INFINITY) {
                            const float f = ex2_approx(mw - M);
                            wsum += mb_l[w * GH + h] * f;
                            acc += mb_o[(w * GH + h) * D + d] * f;
                        }
                    }
                }
                const size_t row = (size_t)it * GH + h;
                A.ws_o[row * D + d] = wsum > 0.f ? acc / wsum : 0.f;
                if (d == 0) A.ws_lse[row] = wsum > 0.f ? M + __log2f(wsum) : -INFINITY;
            }
            named_bar_sync(1, NCW * 32);
        }
    }
}

// One warp per (sequence, query head): log-sum-exp merge of the splits.
template <int D>
__global__ void __launch_bounds__(128)
decode_combine_kernel(const int32_t* __restrict__ kv_len, const int32_t* __restrict__ ws_prefix,
                      const float* __restrict__ ws_lse, const float* __restrict__ ws_o, __half* __restrict__ out,
                      float* __restrict__ lse_out, int B, int Hq, int Hkv, int G, int GH, int HG, int split,
                      int cap_eff, int window) {
    constexpr int DPL = D / 32;   // dims per lane
    const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= B * Hq) return;
    const int b = gw / Hq, h = gw - b * Hq;
    const int g = h / G, r = h - g * G, hg = r / GH, hs = r - hg * GH;
    int start, end;
    seq_range(kv_len[b], cap_eff, window, start, end);
    const int ns = seq_splits(start, end, split);
    const int item0 = ws_prefix[b] + (g * HG + hg) * ns;
    float M = -INFINITY;
    for (int s = lane; s < ns; s += 32) M = fmaxf(M, ws_lse[(size_t)(item0 + s) * GH + hs]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
    float wsum = 0.f;
    if (M > -INFINITY) {
        for (int s = 0; s < ns; ++s) {
            const size_t row = (size_t)(item0 + s) * GH + hs;
            const float ls = ws_lse[row];
            if (ls == -INFINITY) continue;
            const float w = ex2_approx(ls - M);
            wsum += w;
            const float* src = ws_o + row * D + lane * DPL;
#pragma unroll
            for (int i = 0; i < DPL; ++i) acc[i] += w * src[i];
        }
    }
    const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
    __half* dst = out + ((size_t)b * Hq + h) * D + lane * DPL;
#pragma unroll
    for (int i = 0; i < DPL; i += 2) *reinterpret_cast<__half2*>(dst + i) = __floats2half2_rn(acc[i] * inv, acc[i + 1] * inv);
    if (lse_out && lane == 0)
        lse_out[(size_t)b * Hq + h] = wsum > 0.f ? (M + __log2f(wsum)) * 0.6931471805599453f : -INFINITY;
}

template <int D, bool I8, int GH>
attn_status launch_decode_t(const DecodeLaunch& L, const DecodePlan& plan) {
    using C = DecCfg<D, I8, GH>;
    const int esz = I8 ? 1 : 2;
    const CUtensorMapDataType kvt = I8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const bool paged = L.page_table != nullptr;
    const int R = paged ? (L.page_size < T ? L.page_size : T) : T;
    CUtensorMap tk, tv, tks, tvs;
    attn_status st;
    {
        uint64_t dims[4], strides[3];
        uint32_t box[4] = {(uint32_t)D, 1u, (uint32_t)R, 1u};
        dims[0] = D;
        dims[1] = L.Hkv;
        dims[2] = paged ? L.page_size : L.max_kv;
        dims[3] = paged ? L.n_pages : L.B;
        strides[0] = (uint64_t)D * esz;
        strides[1] = strides[0] * L.Hkv;
        strides[2] = strides[1] * dims[2];
        if ((st = encode_tmap_plain(&tk, L.k, kvt, 4, dims, strides, box)) != ATTN_OK) return st;
        if ((st = encode_tmap_plain(&tv, L.v, kvt, 4, dims, strides, box)) != ATTN_OK) return st;
    }
    if (I8) {
        uint64_t dims[3], strides[2];
        uint32_t box[3] = {(uint32_t)R, 1u, 1u};
        dims[0] = paged ? L.page_size : L.max_kv;
        dims[1] = L.Hkv;
        dims[2] = paged ? L.n_pages : L.B;
        strides[0] = dims[0] * 2;
        strides[1] = strides[0] * L.Hkv;
        if ((st = encode_tmap_plain(&tks, L.k_scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, dims, strides, box)) != ATTN_OK)
            return st;
        if ((st = encode_tmap_plain(&tvs, L.v_scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, dims, strides, box)) != ATTN_OK)
            return st;
    } else {
        tks = tk;   // unused
        tvs = tk;
    }
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(decode_split_kernel<D, I8, GH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM_ALLOC) != cudaSuccess)
            return set_error(ATTN_ECUDA, "cudaFuncSetAttribute(decode smem) failed");
        attr_set[dev] = true;
    }
    const int cap_layout = paged ? L.max_pages * L.page_size : L.max_kv;
    DecArgs a;
    a.q = static_cast<const __half*>(L.q);
    a.kv_len = L.kv_len;
    a.page_table = L.page_table;
    uint8_t* ws = static_cast<uint8_t*>(L.workspace);
    a.ws_prefix = reinterpret_cast<int32_t*>(ws);
    a.ws_lse = reinterpret_cast<float*>(ws + plan.off_lse);
    a.ws_o = reinterpret_cast<float*>(ws + plan.off_o);
    a.B = L.B;
    a.Hq = L.Hq;
    a.Hkv = L.Hkv;
    a.G = L.Hq / L.Hkv;
    a.HG = plan.HG;
    a.split = plan.split;
    a.cap_eff = cap_layout < L.max_kv ? cap_layout : L.max_kv;
    a.window = L.window;
    a.P = paged ? L.page_size : 0;
    a.R = R;
    a.max_pages = L.max_pages;
    a.n_pages = paged ? L.n_pages : 0;
    a.paged = paged;
    const bool capped = L.softcap > 0.f;
    a.qscale = capped ? L.scale / L.softcap : L.scale * kLog2e;
    a.cap_log2 = capped ? L.softcap * kLog2e : 0.f;
    a.err = L.err_word;
    long grid = sm_count();
    if (plan.max_items < grid) grid = plan.max_items;
    if (grid < 1) grid = 1;
    decode_split_kernel<D, I8, GH><<<(unsigned)grid, kDecThreads, C::SMEM_ALLOC, L.stream>>>(tk, tv, tks, tvs, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(ATTN_ECUDA, "decode split launch failed: %s", cudaGetErrorString(e));
    const int nwarps = L.B * L.Hq;
    decode_combine_kernel<D><<<(nwarps + 3) / 4, 128, 0, L.stream>>>(
        L.kv_len, a.ws_prefix, a.ws_lse, a.ws_o, static_cast<__half*>(L.out), L.lse, L.B, L.Hq, L.Hkv, a.G, GH,
        plan.HG, plan.split, a.cap_eff, L.window);
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(ATTN_ECUDA, "decode combine launch failed: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

template <int D, bool I8>
attn_status launch_decode_gh(const DecodeLaunch& L, const DecodePlan& plan) {
    switch (plan.GH) {
        case 4: return launch_decode_t<D, I8, 4>(L, plan);
        case 2: return launch_decode_t<D, I8, 2>(L, plan);
        default: return launch_decode_t<D, I8, 1>(L, plan);
    }
}

}  // namespace

bool make_decode_plan(int B, int Hq, int Hkv, int D, int max_kv, int split_keys, DecodePlan* plan) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_kv <= 0 || split_keys < 0) return false;
    if (D != 64 && D != 128 && D != 256) return false;
    const int G = Hq / Hkv;
    plan->GH = (G % 4 == 0) ? 4 : (G % 2 == 0) ? 2 : 1;
    plan->HG = G / plan->GH;
    const long units = (long)B * Hkv * plan->HG;
    int split = split_keys;
    if (split == 0) {
        // aim at ~2048 work items for the longest sequences
        long want = (units * (long)max_kv + 2047) / 2048;
        long p = 256;
        while (p < want && p < 4096) p <<= 1;
        split = (int)p;
    }
    if (split % T != 0) return false;
    plan->split = split;
    // +1 split: tile alignment of a window start can add one partial split
    plan->max_items = units * ((max_kv + split - 1) / split + 1);
    size_t off = ((size_t)(B + 1) * 4 + 255) / 256 * 256;
    plan->off_lse = off;
    off += ((size_t)plan->max_items * plan->GH * 4 + 255) / 256 * 256;
    plan->off_o = off;
    off += (size_t)plan->max_items * plan->GH * D * 4;
    plan->bytes = off;
    return true;
}

attn_status launch_decode(const DecodeLaunch& L, const DecodePlan& plan) {
    switch (L.D) {
        case 64: return L.int8 ? launch_decode_gh<64, true>(L, plan) : launch_decode_gh<64, false>(L, plan);
        case 128: return L.int8 ? launch_decode_gh<128, true>(L, plan) : launch_decode_gh<128, false>(L, plan);
        case 256: return L.int8 ? launch_decode_gh<256, true>(L, plan) : launch_decode_gh<256, false>(L, plan);
        default: return set_error(ATTN_EUNSUPPORTED, "head_dim %d not supported (64, 128, 256)", L.D);
    }
}

}  // namespace attn

// ----------------------------------------------------------------------------
// attn_decode_noalloc: attn_decode with its scratch memory taken from a fixed
// array compiled into this library instead of from the caller.
//
// Some callers cannot hand the library a workspace: code hosted inside an
// engine that owns every byte of device memory and exposes no allocator to
// its plugins, or a latency-critical decode loop that must never call
// cudaMalloc (which can synchronise the whole device).  For them the split
// partials live in `g_decode_scratch`, a file-scope device array of
// kNoAllocScratchBytes that every GPU loading this library keeps until the
// process exits.
//
// The array's name means nothing to host code (it is a host-side shadow, not
// a device address), so the device address is looked up once per device with
// cudaGetSymbolAddress while that device is current, and passed to the
// kernels like any workspace pointer.  That lookup happens inside the first
// call on each device; make that first call before any stream capture.
// Nothing in the scratch needs to start at zero: every byte the kernels read
// is written earlier in the same call.  All calls share the one array, so two
// calls whose kernels overlap on the GPU (different streams, no ordering)
// race on it; order such calls on one stream.
// ----------------------------------------------------------------------------
namespace attn {
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB per device
}  // namespace attn

static __device__ __align__(256) unsigned char g_decode_scratch[attn::kNoAllocScratchBytes];

namespace attn {
namespace {
std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};

// Device address of g_decode_scratch on the current device (looked up once).
attn_status scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error(ATTN_ECUDA, "attn_decode_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return set_error(ATTN_EUNSUPPORTED, "attn_decode_noalloc: device index %d above 63", dev);
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess || p == nullptr)
            return set_error(ATTN_ECUDA, "attn_decode_noalloc: cudaGetSymbolAddress(scratch): %s",
                             cudaGetErrorString(e));
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return ATTN_OK;
}
}  // namespace
}  // namespace attn

extern "C" attn_status attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                           const int32_t* kv_len, const int32_t* page_table, int page_size,
                                           int max_pages_per_seq, int n_pages, int max_kv, const void* k_scales,
                                           const void* v_scales, attn_kv_dtype kv_dtype, int batch, int n_heads,
                                           int n_kv_heads, int head_dim, int window, float softcap, float scale,
                                           int split_keys, void* out, float* lse_out, void* stream) {
    const size_t need = attn_decode_workspace_size(batch, n_heads, n_kv_heads, head_dim, max_kv, split_keys);
    if (need > attn::kNoAllocScratchBytes)
        return attn::set_error(ATTN_EUNSUPPORTED,
                               "attn_decode_noalloc: these sizes need %zu bytes of scratch, above the library's "
                               "fixed %zu (use attn_decode with a caller workspace, or a larger split_keys)",
                               need, attn::kNoAllocScratchBytes);
    void* scratch = nullptr;
    if (need > 0) {   // invalid sizes (need == 0) are reported by attn_decode below
        const attn_status st = attn::scratch_for_current_device(&scratch);
        if (st != ATTN_OK) return st;
    }
    return attn_decode(q, k_cache, v_cache, kv_len, page_table, page_size, max_pages_per_seq, n_pages, max_kv,
                       k_scales, v_scales, kv_dtype, batch, n_heads, n_kv_heads, head_dim, window, softcap, scale,
                       split_keys, out, lse_out, scratch, scratch ? attn::kNoAllocScratchBytes : 0, stream);
}
