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
// each sequence is cut into fixed-size splits so the whole GPU streams the
// cache:
//
//   decode_split_kernel   persistent, one CTA per SM: 8 consumer warps (and,
//                         for int8, a producer warp).  A work item
//                         is (sequence, head block, split): a head block is up
//                         to 8 (kv head, query-head group) units and warp w
//                         owns unit w for the whole split.  Tiles of 16 tokens
//                         (8 for D=256) of every kv head of the block are one
//                         TMA box per tensor (per page when paged): tens of KB
//                         contiguous in the cache, so a handful of copies keep
//                         HBM busy.  The producer warp (f16: warp 0's lane 0,
//                         between its own tiles) issues those copies ahead
//                         into a ring of shared-memory slots (full/empty
//                         mbarriers).  Inside a warp,
//                         8 (16 for D=256) lanes share one key: each lane
//                         holds D/8 dims of the GH query heads of its unit in
//                         registers, so a K row is read once for GH heads
//                         (GQA: q-head h reads kv-head h / G).  Partial dots
//                         are reduce-scattered across the key's lanes with
//                         warp shuffles; int8 codes become floats in registers
//                         and per-token scales apply once per key.  At the end
//                         of a split each warp writes (lse, o / l) of its unit.
//   decode_combine_kernel merges the splits of each (sequence, head) with the
//                         log-sum-exp rule and writes f16 output (+ lse).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "attn_internal.h"
#include "decode_range.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int NW = 8;                     // consumer warps per CTA = units per head block
constexpr int kSmemBudget = 226 * 1024;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;

template <int D, bool I8, int GH>
struct DecCfg {
    // int8: a ninth warp issues the copies, so that no consumer interleaves them
    // with its own tiles (9 warps are allocated registers as 12: 168 a thread).
    // f16 (more registers a lane) keeps the copies on consumer warp 0.
    static constexpr int NPROD = I8 ? 1 : 0;
    static constexpr int THREADS = (NW + NPROD) * 32;
    static constexpr int PROD = NPROD ? NW : 0;          // the warp that issues the copies
    static constexpr int ESZ = I8 ? 1 : 2;
    static constexpr int RB = D * ESZ;                       // bytes of one K/V row
    static constexpr int LPK = (D == 256) ? 16 : 8;          // lanes sharing one key
    static constexpr int LOG_LPK = (LPK == 16) ? 4 : 3;
    static constexpr int KPS = 32 / LPK;                     // keys per warp step
    static constexpr int T = (D == 256) ? 8 : 16;            // tokens per tile
    static constexpr int NSTEP = T / KPS;
    static constexpr int E = D / LPK;                        // elements per lane
    static constexpr int VB = (RB / LPK) < 16 ? (RB / LPK) : 16;   // bytes per vector load
    static constexpr int EV = VB / ESZ;                      // elements per vector
    static constexpr int NV = E / EV;                        // vectors per lane per row
    static constexpr int LOG_GH = (GH == 4) ? 2 : (GH == 2) ? 1 : 0;
    static constexpr int KV_BYTES = T * NW * RB;             // one K (or V) tile, up to 8 kv heads
    static constexpr int SC_BYTES = I8 ? 256 : 0;            // one K (or V) scale tile
    static constexpr int SLOT = 2 * KV_BYTES + 2 * SC_BYTES;
    static constexpr int OFF_PREFIX = 0;
    static constexpr int PREFIX_BYTES = ((kDecodeMaxBatch + 1) * 4 + 127) / 128 * 128;
    static constexpr int OFF_MISC = OFF_PREFIX + PREFIX_BYTES;   // scan scratch (32 ints) + abort flag
    static constexpr int MISC_BYTES = 256;
    static constexpr int OFF_BARS = OFF_MISC + MISC_BYTES;
    static constexpr int NSLOT_RAW = (kSmemBudget - OFF_BARS - 2 * 8 * 8 - 1024) / SLOT;
    static constexpr int NSLOT = NSLOT_RAW > 8 ? 8 : NSLOT_RAW;
    static constexpr int OFF_RING = ((OFF_BARS + 2 * NSLOT * 8) + 1023) / 1024 * 1024;
    static constexpr int SMEM_USED = OFF_RING + NSLOT * SLOT;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;
    static_assert(NSLOT >= 3, "ring too small");
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
    static_assert(E % EV == 0 && E % 2 == 0, "lane layout");
    static_assert(NSTEP * KPS == T, "tile layout");
};

struct DecArgs {
    const __half* q;
    const float* q32;  // f32 queries (then q is unused by the CUDA-core kernel)
    const int32_t* kv_len;
    const int32_t* page_table;
    int32_t* ws_prefix;
    float* ws_lse;
    float* ws_o;
    // balanced tensor-core kernel only: tile prefix over sequences and the
    // per-CTA fix-up partials (see decode_tc.cuh)
    int32_t* ws_tpref;
    int32_t* ws_fix_meta;
    float* ws_fix_lse;
    float* ws_fix_o;
    int B, Hq, Hkv, G, HG, U, n_hb, nh_box, split, cap_eff, window, P, R, max_pages, n_pages, paged;
    int ring;          // > 0: contiguous ring cache, logical token t in row t % ring
    int logR;          // log2(R): rows per box are a power of two (a tile or a page)
    int logP;          // log2(P) (paged)
    // tiered decode: kTierCold reads kv_len = cold lengths (window counted from the
    // newest hot token), kTierHot the hot ring (hot_len, hot_start); kTierPlain alone
    int tier;
    const int32_t* hot_len;
    const int32_t* hot_start;
    float qscale;      // multiplies q: scale*log2e (no cap) or scale/c (cap)
    float cap_log2;    // c*log2e, 0 when the cap is off
    int* err;
};

enum : int { kTierPlain = 0, kTierCold = 1, kTierHot = 2 };

// Kept keys [start, end) of sequence b in the index space of the call's cache
// (logical tokens; for the hot ring, hot token i is index hot_start + i, read
// from slot index % ring).  Tiered decode (attention.js executeAttentionTiered):
// the cold tier's tokens sit at positions 0 .. cold_len-1 and the hot tier's at
// cold_len + i, the query at cold_len + hot_len - 1; a window W keeps positions
// within W of the query, and the ring holds only its newest `ring` hot tokens.
// T is DecArgs or a combine tier (same field names).
template <class T>
__device__ __forceinline__ void tier_range(const T& A, int b, int& start, int& end) {
    if (A.tier == kTierPlain) {
        seq_range(__ldg(&A.kv_len[b]), A.cap_eff, A.window, start, end);
        return;
    }
    const int hl = max(__ldg(&A.hot_len[b]), 0);
    if (A.tier == kTierCold) {
        const int L = min(max(__ldg(&A.kv_len[b]), 0), A.cap_eff);
        start = A.window > 0 ? max(0, L - max(A.window - hl, 0)) : 0;
        end = L;
    } else {
        int hs = __ldg(&A.hot_start[b]) % A.ring;
        if (hs < 0) hs += A.ring;
        int keep = min(hl, A.ring);
        if (A.window > 0) keep = min(keep, A.window);
        end = hs + hl;
        start = end - keep;
    }
}

// Splits of a sequence: aligned to 16 tokens so that tiles start on multiples
// of the tile (and so on page boundaries for pages of >= 16 tokens).
__device__ __forceinline__ int seq_splits(int start, int end, int split) {
    if (end <= start) return 0;
    const int a = (start / 16) * 16;
    return (end - a + split - 1) / split;
}

struct Item {
    int b, hb, ks, ke, start, end, ntile;
};

template <int T>
__device__ __forceinline__ Item decode_item(int it, const int* pref, const DecArgs& A) {
    int lo = 0, hi = A.B;   // largest b with pref[b] <= it
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pref[mid] <= it) lo = mid; else hi = mid;
    }
    Item r;
    r.b = lo;
    tier_range(A, lo, r.start, r.end);
    const int ns = seq_splits(r.start, r.end, A.split);
    const int rem = it - pref[lo];
    r.hb = rem / ns;
    const int s = rem - r.hb * ns;
    r.ks = (r.start / 16) * 16 + s * A.split;
    r.ke = min(r.ks + A.split, r.end);
    r.ntile = (r.ke - r.ks + T - 1) / T;
    return r;
}

// Exclusive prefix over sequences of count(start, end) (block-wide scan).
template <typename F>
__device__ void build_prefix_of(const DecArgs& A, int* pref, int* scratch, F count) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    int carry = 0;
    for (int base = 0; base < A.B; base += blockDim.x) {
        const int b = base + threadIdx.x;
        int v = 0;
        if (b < A.B) {
            int start, end;
            tier_range(A, b, start, end);
            v = count(start, end);
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

// Work items (sequence, head block, split) per sequence.
__device__ void build_prefix(const DecArgs& A, int* pref, int* scratch) {
    build_prefix_of(A, pref, scratch, [&](int start, int end) { return A.n_hb * seq_splits(start, end, A.split); });
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
            constexpr int NWD = C::VB / 4;
            uint32_t ws[NWD];
            if constexpr (NWD == 4) {
                const uint4 w = *reinterpret_cast<const uint4*>(src);
                ws[0] = w.x; ws[1] = w.y; ws[2] = w.z; ws[3] = w.w;
            } else {
                const uint2 w = *reinterpret_cast<const uint2*>(src);
                ws[0] = w.x; ws[1] = w.y;
            }
            const float2 bias = make_float2(-8388736.0f, -8388736.0f);
#pragma unroll
            for (int i = 0; i < NWD; ++i) {
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
__global__ void __launch_bounds__(DecCfg<D, I8, GH>::THREADS, 1)
decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_ks, const __grid_constant__ CUtensorMap tm_vs,
                    const DecArgs A) {
    using C = DecCfg<D, I8, GH>;
    constexpr int NSLOT = C::NSLOT, LPK = C::LPK, E = C::E, T = C::T;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int* pref = reinterpret_cast<int*>(smem + C::OFF_PREFIX);
    int* scratch = reinterpret_cast<int*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 128);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
    const uint32_t ring = smem_u32(smem + C::OFF_RING);
    auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
    auto empty_bar = [&](int s) { return smem_u32(&bars[NSLOT + s]); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t kv_policy = l2_policy_evict_first();   // the cache is read once
    if (threadIdx.x == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), NW);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    build_prefix(A, pref, scratch);   // ends with __syncthreads
    const int total = pref[A.B];
    if (blockIdx.x == 0) {
        for (int b = threadIdx.x; b <= A.B; b += blockDim.x) A.ws_prefix[b] = pref[b];
    }
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        if (I8) {
            tma_prefetch_desc(&tm_ks);
            tma_prefetch_desc(&tm_vs);
        }
    }

    // ------------------------------------------------------------------ producer state (warp NW)
    // Tiles are issued in the order the CTA consumes them; `issued` counts
    // them, (p_it, p_i) is the next tile to issue.
    uint32_t issued = 0;
    int p_it = blockIdx.x, p_i = 0;
    Item p_item;
    if (warp == C::PROD && p_it < total) p_item = decode_item<T>(p_it, pref, A);
    int cache_b = -1, cache_base = -1, pid = -1;
    const int NB = T / A.R;                                   // boxes per tile per tensor
    const uint32_t box_kv = A.R * A.nh_box * C::RB;           // bytes of one K (or V) box
    const uint32_t box_sc = A.R * A.nh_box * 2;               // bytes of one scale box
    const uint32_t sbb = (box_sc + 127) / 128 * 128;          // scale boxes start 128-byte aligned
    bool ok = true;

    // testing hook: issue nothing, so that the consumers' wait for the first
    // tile runs out (the failure path, without a fault)
    const bool stall = stall_first_tile();
    // Issue tiles until `target` (a consumption count) is covered.  Whole producer warp.
    auto produce_until = [&](uint32_t target) {
        while (ok && !stall && issued <= target && p_it < total) {
            const int t0 = p_item.ks + p_i * T;
            const int slot = issued % NSLOT;
            const int g0 = (p_item.hb * NW) / A.HG;
            int pi0 = 0, cb = 0;
            if (A.paged) {
                pi0 = t0 / A.P;
                cb = pi0 & ~31;
                if (p_item.b != cache_b || cb != cache_base) {
                    const int idx = cb + lane;
                    pid = idx < A.max_pages ? __ldg(&A.page_table[(size_t)p_item.b * A.max_pages + idx]) : -1;
                    cache_b = p_item.b;
                    cache_base = cb;
                }
            }
            int good = 1;
            if (lane == 0 && issued >= (uint32_t)NSLOT)
                good = mbar_wait(empty_bar(slot), ((issued / NSLOT) - 1) & 1, abort_flag, A.err, kErrTimeoutSlot);
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) { ok = false; break; }
            const uint32_t sb = ring + slot * C::SLOT;
            int nbox = 1;
            if (A.paged) {
                nbox = 0;
                for (int r = 0; r < NB; ++r)
                    if ((pi0 + r) * A.P < p_item.end) nbox = r + 1;
            }
            const uint32_t bytes = nbox * (2 * box_kv + (I8 ? 2 * box_sc : 0));
            if (lane == 0) mbar_arrive_expect_tx(full_bar(slot), bytes);
            for (int r = 0; r < nbox; ++r) {
                int page = p_item.b, row = t0;
                if (A.paged) {
                    page = __shfl_sync(0xffffffffu, pid, pi0 + r - cb);
                    if (page < 0 || page >= A.n_pages) {
                        // a page id outside the pool: read page 0 instead and report it
                        if (lane == 0) atomicExch(A.err, kErrBadPage);
                        page = 0;
                    }
                    row = (A.P >= T) ? (t0 % A.P) : 0;
                } else if (A.ring > 0) {
                    row = t0 % A.ring;   // 16-token tiles never wrap: ring % 16 == 0
                }
                if (lane == 0) {
                    tma_load_4d_hint(sb + r * box_kv, &tm_k, full_bar(slot), 0, g0, row, page, kv_policy);
                    tma_load_4d_hint(sb + C::KV_BYTES + r * box_kv, &tm_v, full_bar(slot), 0, g0, row, page,
                                     kv_policy);
                    if (I8) {
                        tma_load_3d_hint(sb + 2 * C::KV_BYTES + r * sbb, &tm_ks, full_bar(slot), row, g0, page,
                                         kv_policy);
                        tma_load_3d_hint(sb + 2 * C::KV_BYTES + C::SC_BYTES + r * sbb, &tm_vs, full_bar(slot), row,
                                         g0, page, kv_policy);
                    }
                }
            }
            __syncwarp();
            ++issued;
            if (++p_i == p_item.ntile) {
                p_i = 0;
                p_it += gridDim.x;
                if (p_it < total) p_item = decode_item<T>(p_it, pref, A);
            }
        }
    };

    // ------------------------------------------------------------------ consumers (all warps)
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
    if (C::NPROD && warp == C::PROD) {
        // the producer warp runs ahead of the consumers by up to the whole ring,
        // each slot reused once all NW consumer warps have released it
        produce_until(0xffffffffu);
    }
    uint32_t gcons = 0;
    for (int it = blockIdx.x; warp < NW && it < total; it += gridDim.x) {
        const Item I = decode_item<T>(it, pref, A);
        const int u = I.hb * NW + warp;
        const bool active = u < A.U;
        const int g = active ? u / A.HG : 0;
        const int hg = active ? u - g * A.HG : 0;
        const int hl = g - (I.hb * NW) / A.HG;   // this unit's kv head inside the tile
        float2 q2[GH][E / 2];
        // int8 caches: q in 16-bit fixed point with one scale per head, so the
        // dot with the raw int8 codes is exact integer arithmetic (dp2a); the
        // only approximation is q's rounding to 1/32767 of its largest value
        uint32_t qi[GH][E / 2];
        float inv_qs[GH];
        if (active) {
#pragma unroll
            for (int s = 0; s < GH; ++s) {
                const int head = g * A.G + hg * GH + (s ^ rot);
                const size_t qoff = ((size_t)I.b * A.Hq + head) * D;
#pragma unroll
                for (int v = 0; v < C::NV; ++v)
#pragma unroll
                    for (int e = 0; e < C::EV; e += 2) {
                        const int dim = (v * LPK + c) * C::EV + e;
                        const float2 f = A.q32 ? *reinterpret_cast<const float2*>(A.q32 + qoff + dim)
                                               : __half22float2(*reinterpret_cast<const __half2*>(A.q + qoff + dim));
                        q2[s][(v * C::EV + e) / 2] = make_float2(f.x * A.qscale, f.y * A.qscale);
                    }
            }
            if constexpr (I8) {
                // per-head max |q| over the D dims held by the key's lanes; the
                // partner at xor distance d holds this slot's head in slot s ^ rb(d)
                float mq[GH];
#pragma unroll
                for (int s = 0; s < GH; ++s) {
                    mq[s] = 0.f;
#pragma unroll
                    for (int j = 0; j < E / 2; ++j) mq[s] = fmaxf(mq[s], fmaxf(fabsf(q2[s][j].x), fabsf(q2[s][j].y)));
                }
#pragma unroll
                for (int k = 0; k < C::LOG_LPK; ++k) {
                    const int d = LPK >> (k + 1);
                    const int rb = k < C::LOG_GH ? (GH >> (k + 1)) : 0;
                    float other[GH];
#pragma unroll
                    for (int s = 0; s < GH; ++s) other[s] = __shfl_xor_sync(0xffffffffu, mq[s ^ rb], d);
#pragma unroll
                    for (int s = 0; s < GH; ++s) mq[s] = fmaxf(mq[s], other[s]);
                }
#pragma unroll
                for (int s = 0; s < GH; ++s) {
                    const float qs = mq[s] > 0.f ? 32767.0f / mq[s] : 0.f;
                    inv_qs[s] = mq[s] > 0.f ? mq[s] / 32767.0f : 0.f;
#pragma unroll
                    for (int j = 0; j < E / 2; ++j) {
                        const int lo = __float2int_rn(q2[s][j].x * qs), hi = __float2int_rn(q2[s][j].y * qs);
                        qi[s][j] = (static_cast<uint32_t>(lo) & 0xFFFFu) | (static_cast<uint32_t>(hi) << 16);
                    }
                }
            }
        }
        float2 o2[GH][E / 2];
#pragma unroll
        for (int h = 0; h < GH; ++h)
#pragma unroll
            for (int j = 0; j < E / 2; ++j) o2[h][j] = make_float2(0.f, 0.f);
        float m = -INFINITY, l = 0.f;

        for (int i = 0; i < I.ntile; ++i, ++gcons) {
            if (!C::NPROD && warp == 0) produce_until(gcons + NSLOT - 1);
            const int slot = gcons % NSLOT;
            bool got = ok && mbar_wait(full_bar(slot), (gcons / NSLOT) & 1, abort_flag, A.err, kErrTimeoutLoad);
            got = __all_sync(0xffffffffu, got);   // keep the warp converged for the shuffles below
            if (!got) { ok = false; continue; }
            if (active) {
                const int t0 = I.ks + i * T;
                const int v_lo = max(I.start - t0, 0);
                const int v_hi = min(I.ke - t0, T);
                const uint8_t* kt = smem + C::OFF_RING + slot * C::SLOT;
                const uint8_t* vt = kt + C::KV_BYTES;
                const __half* kst = reinterpret_cast<const __half*>(kt + 2 * C::KV_BYTES);
                const __half* vst = reinterpret_cast<const __half*>(kt + 2 * C::KV_BYTES + C::SC_BYTES);
                const int sc_off = hl * A.R;   // this head's scales inside a scale box (elements)

                float tsc[C::NSTEP];
#pragma unroll
                for (int st = 0; st < C::NSTEP; ++st) {
                    const int key = st * C::KPS + kk;
                    float t;
                    if constexpr (I8) {
                        // exact int32 dots of the int8 codes with the fixed-point q (dp2a)
                        const uint8_t* krow = kt + (key * A.nh_box + hl) * C::RB;
                        // two accumulators per head (lo and hi halves of each word): chains of
                        // NV * VB / 4 dependent dp2a instead of twice that
                        int acc[GH], acc_hi[GH];
#pragma unroll
                        for (int s = 0; s < GH; ++s) acc[s] = acc_hi[s] = 0;
#pragma unroll
                        for (int v = 0; v < C::NV; ++v) {
                            uint32_t w[C::VB / 4];
                            if constexpr (C::VB == 16) {
                                const uint4 x = *reinterpret_cast<const uint4*>(krow + (v * LPK + c) * C::VB);
                                w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
                            } else {
                                const uint2 x = *reinterpret_cast<const uint2*>(krow + (v * LPK + c) * C::VB);
                                w[0] = x.x; w[1] = x.y;
                            }
#pragma unroll
                            for (int i = 0; i < C::VB / 4; ++i)
#pragma unroll
                                for (int s = 0; s < GH; ++s) {
                                    const int j = (v * C::EV) / 2 + 2 * i;
                                    asm("dp2a.lo.s32.s32 %0, %1, %2, %0;" : "+r"(acc[s]) : "r"(qi[s][j]), "r"(w[i]));
                                    asm("dp2a.hi.s32.s32 %0, %1, %2, %0;" : "+r"(acc_hi[s]) : "r"(qi[s][j + 1]), "r"(w[i]));
                                }
                        }
#pragma unroll
                        for (int s = 0; s < GH; ++s) acc[s] += acc_hi[s];
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
                        t = static_cast<float>(acc[0]) * inv_qs[0] *
                            __half2float(kst[(key >> A.logR) * (sbb / 2) + sc_off + (key & (A.R - 1))]);
                    } else {
                        float2 kx[E / 2];
                        load_row_slice<D, I8, GH>(kt + (key * A.nh_box + hl) * C::RB, c, kx);
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
                        t = acc[0];
                    }
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
                        pv[st] = valid ? p * __half2float(vst[(key >> A.logR) * (sbb / 2) + sc_off + (key & (A.R - 1))]) : 0.f;
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
                        load_row_slice<D, I8, GH>(vt + (key * A.nh_box + hl) * C::RB, c, vx);
#pragma unroll
                        for (int h = 0; h < GH; ++h) {
                            const float2 pp = make_float2(pg[h], pg[h]);
#pragma unroll
                            for (int j = 0; j < E / 2; ++j) o2[h][j] = ffma2(pp, vx[j], o2[h][j]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(slot));
        }
        if (!active) continue;

        // ---- end of the split: key groups -> group 0, then (lse, o / l) of each head
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
        const size_t prow = ((size_t)it * NW + warp) * GH;   // this unit's partial rows
#pragma unroll
        for (int h = 0; h < GH; ++h) {
            const float lh = __shfl_sync(0xffffffffu, l, src_lane[h]);
            const float mh = __shfl_sync(0xffffffffu, m, src_lane[h]);
            const float inv = lh > 0.f ? 1.0f / lh : 0.f;
            if (lane < LPK) {
#pragma unroll
                for (int v = 0; v < C::NV; ++v)
#pragma unroll
                    for (int e = 0; e < C::EV; e += 2) {
                        const int dim = (v * LPK + c) * C::EV + e;
                        const float2 ov = o2[h][(v * C::EV + e) / 2];
                        *reinterpret_cast<float2*>(&A.ws_o[(prow + h) * D + dim]) = make_float2(ov.x * inv, ov.y * inv);
                    }
            }
            if (lane == 0) A.ws_lse[prow + h] = lh > 0.f ? mh + __log2f(lh) : -INFINITY;
        }
    }
    // this CTA's partials are written: the combine pass may be scheduled (it
    // still waits for the whole grid to finish)
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
    if (warp == C::PROD && !ok && lane == 0) {
        // let copies in flight land before shared memory is released
        const uint32_t first = issued > (uint32_t)NSLOT ? issued - NSLOT : 0;
        for (uint32_t x = first; x < issued; ++x)
            mbar_wait_drain(full_bar(x % NSLOT), (x / NSLOT) & 1, A.err, kErrTimeoutLoad);
    }
}

#include "decode_tc.cuh"

// One tier of the combine: where a split kernel left its partials, and the
// range arguments that say which items it wrote.
struct CombTier {
    const int32_t* kv_len;
    const int32_t* hot_len;
    const int32_t* hot_start;
    int tier, cap_eff, window, ring, split, n_fix;
    const int32_t* ws_prefix;
    const float* ws_lse;
    const float* ws_o;
    const int32_t* fix_meta;
    const float* fix_lse;
    const float* fix_o;
};
template <int NT>
struct CombTiers {
    CombTier t[NT];
};

// One warp per (sequence, query head): log-sum-exp merge of the splits of
// every tier (one tier for a plain decode; cold and hot for a tiered decode).
// RB: partial rows read per batch (all loads in flight together): 16 for the
// CUDA-core kernel's partials (many splits per row, no fix-up slots), 8 otherwise.
template <int D, int NT, typename OutT, int RB>
__global__ void __launch_bounds__(128)
decode_combine_kernel(const CombTiers<NT> T, OutT* __restrict__ out, float* __restrict__ lse_out, int B, int Hq,
                      int G, int GH, int HG, int n_hb) {
    constexpr int DPL = D / 32;   // dims per lane
    // launched as a programmatic dependent of the split kernel: wait until that
    // grid has finished and its partials are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= B * Hq) return;
    const int b = gw / Hq, h = gw - b * Hq;
    const int g = h / G, r = h - g * G, hg = r / GH, hs = r - hg * GH;
    const int u = g * HG + hg, hb = u / NW, w = u - hb * NW;
    const int fid = b * n_hb + hb;     // fix-up slots written for this (sequence, head block)
    // per tier: the lse of the first KR*32 splits and every fix-up tag, as
    // independent loads kept in registers (both passes below use them)
    constexpr int KR = 4, KF = kDecodeMaxFix / 32;
    int ns[NT] = {}, item0[NT] = {};
    float lsr[NT][KR];
    bool mine[NT][KF];
    float fls[NT][KF];
    auto lrow = [&](int ti, int sp) { return ((size_t)(item0[ti] + sp) * NW + w) * GH + hs; };
    float M = -INFINITY;
#pragma unroll
    for (int ti = 0; ti < NT; ++ti) {
        const CombTier& t = T.t[ti];
        int start, end;
        tier_range(t, b, start, end);
        ns[ti] = seq_splits(start, end, t.split);
        item0[ti] = t.ws_prefix[b] + hb * ns[ti];
#pragma unroll
        for (int k = 0; k < KR; ++k)
            lsr[ti][k] = (k * 32 + lane < ns[ti]) ? t.ws_lse[lrow(ti, k * 32 + lane)] : -INFINITY;
#pragma unroll
        for (int q = 0; q < KF; ++q) mine[ti][q] = (q * 32 + lane < t.n_fix) && t.fix_meta[q * 32 + lane] == fid;
#pragma unroll
        for (int q = 0; q < KF; ++q)
            fls[ti][q] = mine[ti][q] ? t.fix_lse[((size_t)(q * 32 + lane) * NW + w) * GH + hs] : -INFINITY;
#pragma unroll
        for (int k = 0; k < KR; ++k) M = fmaxf(M, lsr[ti][k]);
        for (int sp = KR * 32 + lane; sp < ns[ti]; sp += 32) M = fmaxf(M, t.ws_lse[lrow(ti, sp)]);
#pragma unroll
        for (int q = 0; q < KF; ++q) M = fmaxf(M, fls[ti][q]);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float acc[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
    float wl_sum = 0.f;   // this lane's share of the weight sum
    // DPL floats of a partial row (this lane's dims)
    auto load_row = [&](const float* o_rows, size_t row, float (&v)[DPL]) {
        const float* src = o_rows + row * D + lane * DPL;
        if constexpr (DPL % 4 == 0) {
#pragma unroll
            for (int i = 0; i < DPL; i += 4) {
                const float4 x = *reinterpret_cast<const float4*>(src + i);
                v[i] = x.x; v[i + 1] = x.y; v[i + 2] = x.z; v[i + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < DPL; i += 2) {
                const float2 x = *reinterpret_cast<const float2*>(src + i);
                v[i] = x.x; v[i + 1] = x.y;
            }
        }
    };
    // acc += wt * v, as a select: rows whose lse is -inf were never written and
    // may hold anything, so their (zero) weight must not multiply them
    auto accumulate = [&](float wt, const float (&v)[DPL]) {
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] += (wt != 0.f) ? wt * v[i] : 0.f;
    };
    auto weight = [&](float ls) { return (ls == -INFINITY) ? 0.f : ex2_approx(ls - M); };
    if (M > -INFINITY) {
#pragma unroll
        for (int ti = 0; ti < NT; ++ti) {
            const CombTier& t = T.t[ti];
            // 32 splits at a time: lane l holds the weight of split base+l, then the
            // warp reads the partial rows RB at a time, all loads in flight together
            for (int base = 0; base < ns[ti]; base += 32) {
                const int k32 = base / 32;
                float ls = -INFINITY;
#pragma unroll
                for (int k = 0; k < KR; ++k)
                    if (k == k32) ls = lsr[ti][k];
                if (k32 >= KR && base + lane < ns[ti]) ls = t.ws_lse[lrow(ti, base + lane)];
                const float wl = weight(ls);
                wl_sum += wl;
                // the splits with weight (the rest were merged into another row or saw
                // no key), read RB at a time with all loads in flight together
                unsigned mk = __ballot_sync(0xffffffffu, wl != 0.f);
                while (mk) {
                    float v[RB][DPL];
                    float wt[RB];
                    const int k_first = __ffs(mk) - 1;
#pragma unroll
                    for (int q = 0; q < RB; ++q) {
                        int k = k_first;
                        wt[q] = 0.f;
                        if (mk) {
                            k = __ffs(mk) - 1;
                            mk &= mk - 1;
                            wt[q] = __shfl_sync(0xffffffffu, wl, k);
                        }
                        load_row(t.ws_o, lrow(ti, base + k), v[q]);
                    }
#pragma unroll
                    for (int q = 0; q < RB; ++q) accumulate(wt[q], v[q]);
                }
            }
            // the fix-up slots of this (sequence, head block)
#pragma unroll
            for (int q = 0; q < KF; ++q) {
                const float wl = weight(fls[ti][q]);
                wl_sum += wl;
                unsigned m = __ballot_sync(0xffffffffu, mine[ti][q]);
                while (m) {
                    const int k = __ffs(m) - 1;
                    m &= m - 1;
                    const float wt = __shfl_sync(0xffffffffu, wl, k);
                    if (wt != 0.f) {
                        float v[DPL];
                        load_row(t.fix_o, ((size_t)(q * 32 + k) * NW + w) * GH + hs, v);
                        accumulate(wt, v);
                    }
                }
            }
        }
    }
    float wsum = wl_sum;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
    OutT* dst = out + ((size_t)b * Hq + h) * D + lane * DPL;
#pragma unroll
    for (int i = 0; i < DPL; i += 2) {
        if constexpr (sizeof(OutT) == 4)
            *reinterpret_cast<float2*>(dst + i) = make_float2(acc[i] * inv, acc[i + 1] * inv);
        else
            *reinterpret_cast<__half2*>(dst + i) = __floats2half2_rn(acc[i] * inv, acc[i + 1] * inv);
    }
    if (lse_out && lane == 0)
        lse_out[(size_t)b * Hq + h] = wsum > 0.f ? (M + __log2f(wsum)) * 0.6931471805599453f : -INFINITY;
}

// Kernel arguments shared by both split kernels.
DecArgs make_dec_args(const DecodeLaunch& L, const DecodePlan& plan, int R) {
    const bool paged = L.page_table != nullptr;
    const int cap_layout = paged ? L.max_pages * L.page_size : L.max_kv;
    DecArgs a;
    a.q = L.q_f32 ? nullptr : static_cast<const __half*>(L.q);
    a.q32 = L.q_f32 ? static_cast<const float*>(L.q) : nullptr;
    a.kv_len = L.kv_len;
    a.page_table = L.page_table;
    uint8_t* ws = static_cast<uint8_t*>(L.workspace);
    a.ws_prefix = reinterpret_cast<int32_t*>(ws);
    a.ws_lse = reinterpret_cast<float*>(ws + plan.off_lse);
    a.ws_o = reinterpret_cast<float*>(ws + plan.off_o);
    a.ws_tpref = reinterpret_cast<int32_t*>(ws + plan.off_tpref);
    a.ws_fix_meta = reinterpret_cast<int32_t*>(ws + plan.off_fix_meta);
    a.ws_fix_lse = reinterpret_cast<float*>(ws + plan.off_fix_lse);
    a.ws_fix_o = reinterpret_cast<float*>(ws + plan.off_fix_o);
    a.B = L.B;
    a.Hq = L.Hq;
    a.Hkv = L.Hkv;
    a.G = L.Hq / L.Hkv;
    a.HG = plan.HG;
    a.U = L.Hkv * plan.HG;
    a.n_hb = plan.n_hb;
    a.nh_box = plan.nh_box;
    a.split = plan.split;
    // a ring holds the newest `ring` tokens of sequences of any length: no clamp
    a.cap_eff = L.ring > 0 ? (1 << 30) : (cap_layout < L.max_kv ? cap_layout : L.max_kv);
    a.ring = L.ring;
    a.tier = L.tier;
    a.hot_len = L.hot_len;
    a.hot_start = L.hot_start;
    a.window = L.window;
    a.P = paged ? L.page_size : 0;
    a.R = R;
    a.logR = 0;
    while ((1 << a.logR) < R) ++a.logR;
    a.logP = 0;
    while (paged && (1 << a.logP) < L.page_size) ++a.logP;
    a.max_pages = L.max_pages;
    a.n_pages = paged ? L.n_pages : 0;
    a.paged = paged;
    const bool capped = L.softcap > 0.f;
    a.qscale = capped ? L.scale / L.softcap : L.scale * kLog2e;
    a.cap_log2 = capped ? L.softcap * kLog2e : 0.f;
    a.err = L.err_word;
    return a;
}

// What a split kernel launch leaves for the combine: its arguments and the
// fix-up slots it wrote (its grid for the balanced tensor-core kernel, 0 for
// the item-per-CTA kernel).
struct SplitOut {
    DecArgs a;
    int n_fix;
};

CombTier comb_tier(const SplitOut& so) {
    const DecArgs& a = so.a;
    CombTier t;
    t.kv_len = a.kv_len;
    t.hot_len = a.hot_len;
    t.hot_start = a.hot_start;
    t.tier = a.tier;
    t.cap_eff = a.cap_eff;
    t.window = a.window;
    t.ring = a.ring;
    t.split = a.split;
    t.n_fix = so.n_fix;
    t.ws_prefix = a.ws_prefix;
    t.ws_lse = a.ws_lse;
    t.ws_o = a.ws_o;
    t.fix_meta = a.ws_fix_meta;
    t.fix_lse = a.ws_fix_lse;
    t.fix_o = a.ws_fix_o;
    return t;
}

// The combine is a programmatic dependent launch: its CTAs may be scheduled
// while the split kernel's last CTAs finish (hiding the launch latency) and
// wait in griddepcontrol.wait for that grid to complete.  (A tiered decode's
// cold split kernel finished before its hot split kernel started: plain stream
// order.)
template <int D, int NT>
attn_status launch_combine(const DecodeLaunch& L, const DecodePlan& plan, const CombTiers<NT>& T) {
    const int nwarps = L.B * L.Hq;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((nwarps + 3) / 4);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (trace_enabled())
        trace("decode_combine_kernel<D=%d,tiers=%d,out=%s> grid=%u block=128 (one warp per (sequence, head); "
              "programmatic dependent launch)", D, NT, L.out_f32 ? "f32" : "f16", cfg.gridDim.x);
    // the CUDA-core kernel's partials (no fix-up slots) come many splits to a row
    cudaError_t e;
    auto go = [&](auto kernel, auto* out) {
        return cudaLaunchKernelEx(&cfg, kernel, T, out, L.lse, L.B, L.Hq, L.Hq / L.Hkv, plan.GH, plan.HG, plan.n_hb);
    };
    float* o32 = static_cast<float*>(L.out);
    __half* o16 = static_cast<__half*>(L.out);
    if constexpr (NT == 1 && D <= 128) {
        const bool wide = T.t[0].n_fix == 0;
        if (L.out_f32)
            e = wide ? go(decode_combine_kernel<D, NT, float, 16>, o32) : go(decode_combine_kernel<D, NT, float, 8>, o32);
        else
            e = wide ? go(decode_combine_kernel<D, NT, __half, 16>, o16) : go(decode_combine_kernel<D, NT, __half, 8>, o16);
    } else {
        e = L.out_f32 ? go(decode_combine_kernel<D, NT, float, 8>, o32) : go(decode_combine_kernel<D, NT, __half, 8>, o16);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(ATTN_ECUDA, "decode combine launch failed: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

template <int NT>
attn_status launch_combine_d(const DecodeLaunch& L, const DecodePlan& plan, const CombTiers<NT>& T) {
    switch (L.D) {
        case 64: return launch_combine<64, NT>(L, plan, T);
        case 128: return launch_combine<128, NT>(L, plan, T);
        default: return launch_combine<256, NT>(L, plan, T);
    }
}

int decode_grid(const DecodePlan& plan) {
    long grid = sm_count();
    if (plan.max_items < grid) grid = plan.max_items;
    return grid < 1 ? 1 : (int)grid;
}

// Tensor-core split kernel: f16 caches with head_dim 64/128; boxes of R rows x
// NH heads.  Q2: f32 queries (split into f16 hi and lo terms by the kernel as it
// loads them).
template <int D, int NH, bool Q2>
attn_status launch_decode_tc(const DecodeLaunch& L, const DecodePlan& plan, SplitOut* so) {
    using C = tcdec::Cfg<D, Q2>;
    const bool paged = L.page_table != nullptr;
    // rows per box: 16, or the page size when pages are shorter (R * NH >= 8)
    const int R = paged && L.page_size < 16 ? L.page_size : 16;
    CUtensorMap tk, tv;
    attn_status st;
    const int q_rows = L.Hq < tcdec::QROWS ? L.Hq : tcdec::QROWS;
    {
        // [pages or B][rows][Hkv][D]: boxes of (64 dims, NH heads, R rows, 1), 128-byte swizzle
        uint64_t dims[4], strides[3];
        const uint32_t box[4] = {64u, (uint32_t)NH, (uint32_t)R, 1u};
        dims[0] = D;
        dims[1] = L.Hkv;
        dims[2] = paged ? L.page_size : L.max_kv;
        dims[3] = paged ? L.n_pages : L.B;
        strides[0] = (uint64_t)D * 2;
        strides[1] = strides[0] * L.Hkv;
        strides[2] = strides[1] * dims[2];
        if ((st = encode_tmap_sw128(&tk, L.k, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, dims, strides, box)) != ATTN_OK)
            return st;
        if ((st = encode_tmap_sw128(&tv, L.v, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, dims, strides, box)) != ATTN_OK)
            return st;
    }
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(tcdec::decode_tc_kernel<D, NH, Q2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM_ALLOC) != cudaSuccess)
            return set_error(ATTN_ECUDA, "cudaFuncSetAttribute(decode tc smem) failed");
        attr_set[dev] = true;
    }
    const DecArgs a = make_dec_args(L, plan, R);
    // balanced: every CTA takes an equal share of the tiles (see decode_tc.cuh)
    const int grid = sm_count() < plan.n_fix ? sm_count() : plan.n_fix;
    if (trace_enabled())
        trace("decode_tc_kernel<D=%d,NH=%d,f32q=%d> grid=%d block=%d smem=%u B=%d Hq=%d Hkv=%d layout=%s "
              "tier=%d split=%d head_blocks=%d units=%d max_items=%ld tile_tokens=%d ring_slots=%d+%d "
              "(tiles balanced over the CTAs)",
              D, NH, (int)Q2, grid, tcdec::kThreads, C::SMEM_ALLOC, L.B, L.Hq, L.Hkv,
              paged ? "paged" : L.ring > 0 ? "ring" : "contiguous", L.tier, plan.split, plan.n_hb, a.U,
              plan.max_items, tcdec::TR / NH, C::NK, C::NV);
    tcdec::decode_tc_kernel<D, NH, Q2><<<grid, tcdec::kThreads, C::SMEM_ALLOC, L.stream>>>(tk, tv, a, q_rows);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(ATTN_ECUDA, "decode tc launch failed: %s", cudaGetErrorString(e));
    so->a = a;
    so->n_fix = grid;
    return ATTN_OK;
}

template <int D, bool I8, int GH>
attn_status launch_decode_t(const DecodeLaunch& L, const DecodePlan& plan, SplitOut* so) {
    using C = DecCfg<D, I8, GH>;
    const int esz = I8 ? 1 : 2;
    const CUtensorMapDataType kvt = I8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const bool paged = L.page_table != nullptr;
    if constexpr (!I8 && D != 256) {
        // both contractions on the tensor cores where the boxes allow it: a
        // box covers at most Hkv heads and 16 rows of one page; with pages
        // shorter than 16 tokens each box of P rows must start 1024-byte aligned
        // (P * NH >= 8); batches of up to 2048
        int nh = 1;
        while (nh < plan.nh_box) nh <<= 1;
        const bool boxes_ok = !paged || L.page_size % 16 == 0 || L.page_size * nh >= 8;
        if (boxes_ok && nh <= L.Hkv && L.B <= tcdec::kMaxBatch) {
            switch (nh) {
                case 1: return L.q_f32 ? launch_decode_tc<D, 1, true>(L, plan, so) : launch_decode_tc<D, 1, false>(L, plan, so);
                case 2: return L.q_f32 ? launch_decode_tc<D, 2, true>(L, plan, so) : launch_decode_tc<D, 2, false>(L, plan, so);
                case 4: return L.q_f32 ? launch_decode_tc<D, 4, true>(L, plan, so) : launch_decode_tc<D, 4, false>(L, plan, so);
                default: return L.q_f32 ? launch_decode_tc<D, 8, true>(L, plan, so) : launch_decode_tc<D, 8, false>(L, plan, so);
            }
        }
    }
    const int R = paged ? (L.page_size < C::T ? L.page_size : C::T) : C::T;
    CUtensorMap tk, tv, tks, tvs;
    attn_status st;
    {
        // [pages or B][rows][Hkv][D]: boxes of (D, nh_box heads, R rows, 1)
        uint64_t dims[4], strides[3];
        uint32_t box[4] = {(uint32_t)D, (uint32_t)plan.nh_box, (uint32_t)R, 1u};
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
        // [pages or B][Hkv][rows]: boxes of (R rows, nh_box heads, 1)
        uint64_t dims[3], strides[2];
        uint32_t box[3] = {(uint32_t)R, (uint32_t)plan.nh_box, 1u};
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
    const DecArgs a = make_dec_args(L, plan, R);
    if (trace_enabled())
        trace("decode_split_kernel<D=%d,int8=%d,GH=%d> grid=%d block=%d smem=%d B=%d Hq=%d Hkv=%d layout=%s tier=%d "
              "split=%d head_blocks=%d box_heads=%d box_rows=%d max_items=%ld ring_slots=%d "
              "(items round-robin over the CTAs)",
              D, (int)I8, GH, decode_grid(plan), C::THREADS, C::SMEM_ALLOC, L.B, L.Hq, L.Hkv,
              paged ? "paged" : L.ring > 0 ? "ring" : "contiguous", L.tier, plan.split, plan.n_hb, plan.nh_box, R,
              plan.max_items, C::NSLOT);
    decode_split_kernel<D, I8, GH><<<decode_grid(plan), C::THREADS, C::SMEM_ALLOC, L.stream>>>(tk, tv, tks, tvs, a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(ATTN_ECUDA, "decode split launch failed: %s", cudaGetErrorString(e));
    so->a = a;
    so->n_fix = 0;
    return ATTN_OK;
}

template <int D, bool I8>
attn_status launch_decode_gh(const DecodeLaunch& L, const DecodePlan& plan, SplitOut* so) {
    switch (plan.GH) {
        case 4: return launch_decode_t<D, I8, 4>(L, plan, so);
        case 2: return launch_decode_t<D, I8, 2>(L, plan, so);
        default: return launch_decode_t<D, I8, 1>(L, plan, so);
    }
}

// The split kernel for one cache (either kernel; see launch_decode_t).
attn_status launch_split(const DecodeLaunch& L, const DecodePlan& plan, SplitOut* so) {
    switch (L.D) {
        case 64: return L.int8 ? launch_decode_gh<64, true>(L, plan, so) : launch_decode_gh<64, false>(L, plan, so);
        case 128: return L.int8 ? launch_decode_gh<128, true>(L, plan, so) : launch_decode_gh<128, false>(L, plan, so);
        case 256: return L.int8 ? launch_decode_gh<256, true>(L, plan, so) : launch_decode_gh<256, false>(L, plan, so);
        default: return set_error(ATTN_EUNSUPPORTED, "head_dim %d not supported (64, 128, 256)", L.D);
    }
}

}  // namespace

bool make_decode_plan(int B, int Hq, int Hkv, int D, int max_kv, int split_keys, DecodePlan* plan) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_kv <= 0 || split_keys < 0) return false;
    if (D != 64 && D != 128 && D != 256) return false;
    const int G = Hq / Hkv;
    plan->GH = (G % 4 == 0) ? 4 : (G % 2 == 0) ? 2 : 1;
    plan->HG = G / plan->GH;
    const int U = Hkv * plan->HG;                  // (kv head, head group) units
    plan->n_hb = (U + NW - 1) / NW;                // head blocks of up to 8 units
    int nh = 1;
    for (int hb = 0; hb < plan->n_hb; ++hb) {
        const int u0 = hb * NW, u1 = (u0 + NW < U ? u0 + NW : U) - 1;
        const int span = u1 / plan->HG - u0 / plan->HG + 1;
        if (span > nh) nh = span;
    }
    plan->nh_box = nh;                             // kv heads one TMA box covers
    const long units = (long)B * plan->n_hb;
    int split = split_keys;
    if (split == 0) {
        // aim at ~1024 work items of (sequence, head block, split) for the longest sequences
        long want = (units * (long)max_kv + 1023) / 1024;
        long p = 64;
        while (p < want && p < 8192) p <<= 1;
        split = (int)p;
    }
    if (split % 16 != 0) return false;
    plan->split = split;
    // +1 split: aligning a window start down to the tile can add one partial split
    plan->max_items = units * ((max_kv + split - 1) / split + 1);
    // fix-up slots: the balanced kernel launches at most this many CTAs
    plan->n_fix = plan->max_items < kDecodeMaxFix ? (int)plan->max_items : kDecodeMaxFix;
    const size_t rows = (size_t)plan->max_items * NW * plan->GH;   // (item, warp, head) partial rows
    const size_t frows = (size_t)plan->n_fix * NW * plan->GH;      // (CTA, warp, head) fix-up rows
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    size_t off = up((size_t)(B + 1) * 4);                          // item prefix
    plan->off_tpref = off;
    off += up((size_t)(B + 1) * 4);
    plan->off_fix_meta = off;
    off += up((size_t)plan->n_fix * 4);
    plan->off_lse = off;
    off += up(rows * 4);
    plan->off_fix_lse = off;
    off += up(frows * 4);
    plan->off_o = off;
    off += up(rows * D * 4);
    plan->off_fix_o = off;
    off += up(frows * D * 4);
    plan->bytes = off;
    return true;
}

attn_status launch_decode(const DecodeLaunch& L, const DecodePlan& plan) {
    if (direct_decode_fits(L)) return launch_direct(L);
    SplitOut so;
    attn_status st = launch_split(L, plan, &so);
    if (st != ATTN_OK) return st;
    CombTiers<1> T;
    T.t[0] = comb_tier(so);
    return launch_combine_d<1>(L, plan, T);
}

// Tiered decode: the cold tier's split kernel, then the hot ring's, then one
// combine over the partials of both (the two launches share out, lse and the
// stream; each has its own plan and part of the workspace).
attn_status launch_decode_tiered(const DecodeLaunch& cold, const DecodePlan& cold_plan, const DecodeLaunch& hot,
                                 const DecodePlan& hot_plan) {
    SplitOut sc, sh;
    attn_status st = launch_split(cold, cold_plan, &sc);
    if (st != ATTN_OK) return st;
    if ((st = launch_split(hot, hot_plan, &sh)) != ATTN_OK) return st;
    CombTiers<2> T;
    T.t[0] = comb_tier(sc);
    T.t[1] = comb_tier(sh);
    return launch_combine_d<2>(cold, cold_plan, T);
}

// Sets this translation unit's test controls (see ptx.cuh).
attn_status set_test_controls_decode(unsigned long long wait_limit_ns, int stall) {
    if (cudaMemcpyToSymbol(g_wait_limit_ns, &wait_limit_ns, sizeof(wait_limit_ns)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_stall_first_tile, &stall, sizeof(stall)) != cudaSuccess)
        return set_error(ATTN_ECUDA, "test controls (decode): %s", cudaGetErrorString(cudaGetLastError()));
    return ATTN_OK;
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
// a device address), so every call looks the device address up with
// cudaGetSymbolAddress on the current device and passes it to the kernels
// like any workspace pointer.  The lookup is not cached: after cudaDeviceReset
// the module reloads at another address.  The first call on a device loads
// the module (lazy loading), which reserves the array; make that first call
// at initialisation, before any stream capture or latency-critical loop.
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
// Device address of g_decode_scratch on the current device.
attn_status scratch_for_current_device(void** out) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr)
        return set_error(ATTN_ECUDA, "attn_decode_noalloc: cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    *out = p;
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
