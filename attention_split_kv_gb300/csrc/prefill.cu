// prefill.cu -- tiled causal / bidirectional attention (text prefill and the
// vision tower) on the sm_103a tensor cores.
//
// Problem (doppler src/gpu/kernels/attention.js, the prefill tiers of
// selectAttentionTier / executeAttention; rullama src/backend/dispatch/
// attention.rs, vision_attention_chained and its flash variants): for every
// query token i and head h, softmax over the kept keys j of
// scale * q_i . k_j (optionally soft-capped), applied to v_j.  The pages'
// kernels tile K/V through workgroup-shared memory and run an online softmax
// with 1-16 queries per workgroup; here a CTA owns a 128-query tile and the
// two contractions run on tcgen05:
//
//   S_j  = Q K_j^T     128 x BN, f32 in TMEM    (tcgen05.mma, Q and K in smem)
//   P_j  = exp2(S_j * scale*log2e - m)         (4 softmax warps, 1 row/thread),
//                      f16 written back to TMEM with tcgen05.st
//   O   += P_j V_j     128 x D,  f32 in TMEM    (tcgen05.mma, P from TMEM,
//                                               V in smem as the MN-major operand)
//
// Roles: warps 0-3 softmax + epilogue (thread t owns query row t = TMEM lane
// t), warp 4 TMA producer of Q and K, warp 5 TMEM allocator + MMA issuer, warp
// 6 TMA producer of V (D=64/128 add an idle warp 7 to complete the second
// warpgroup for setmaxnreg; D=256 has 8 softmax warps, so these are 8-10).
// The MMA warp issues S_{j+1} before waiting for P_j, so QK^T of the next tile
// overlaps the softmax of the current one.  O is rescaled lazily: only when a
// row's running max grows by more than 8 (log2 units), so P <= 2^8 stays
// exact in f16 range and the final O / l is unchanged.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int BM = 128;                 // queries per CTA (TMEM lanes)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

// Softmax modes (compile-time): positive scale without a cap works on raw
// accumulators; otherwise logits are scaled (and capped) first.
enum : int { kModeRaw = 0, kModeScaled = 1, kModeCapped = 2 };

constexpr int BN_OF(int D) { return (D == 128) ? 64 : 128; }

template <int D>
struct PrefillCfg {
    static constexpr int NCH = D / 64;                   // 64-element (128-byte) chunks of D
    // D=64/128 run two CTAs per SM (256 TMEM columns each) so that two softmax
    // warpgroups share every SM; D=256 runs one CTA per SM.
    static constexpr int CTAS_PER_SM = (D <= 128) ? 2 : 1;
    // D=64/128: two full warpgroups, so that setmaxnreg can move registers
    // from the producer/MMA warpgroup (warps 4-7, two of them idle) to the
    // softmax warpgroup: 2 CTAs x 256 threads x 128 registers at launch, then
    // 128 x 200 + 128 x 56 per CTA.  D=256 (one CTA per SM) runs two softmax
    // warpgroups that split each row's keys in halves (so every SMSP has two
    // softmax warps), then the producer, MMA and V-producer warps: 11 warps.
    static constexpr int NSM = (D == 256) ? 8 : 4;       // softmax warps
    static constexpr int THREADS = (D <= 128) ? 256 : (NSM + 3) * 32;
    static constexpr int PROD_WARP = NSM, MMA_WARP = NSM + 1, PROD_V_WARP = NSM + 2;
    static constexpr int CW = BN_OF(D) / (NSM / 4);      // S columns per softmax thread
    static constexpr int REG_SOFTMAX = 200, REG_OTHER = 56;
    static_assert(THREADS != 256 || (REG_SOFTMAX + REG_OTHER) * 128 * CTAS_PER_SM == 65536, "register split");
    static constexpr int BN = BN_OF(D);                  // keys per tile
    // S and P buffers in TMEM: one of each (D=64: S 128 + O 64 + P 64; D=128
    // with 64-key tiles: S 64 + O 128 + P 32; D=256 with 128-key tiles: S 128 +
    // O 256 + P 64 of 512): the softmax frees S as soon as its row is in
    // registers, so the next QK^T still overlaps the exponentials.
    static constexpr int NBUF = 1;
    // K/V ring depths: K is consumed a whole softmax earlier than V, so it gets
    // the deeper ring where shared memory allows (two D=128 CTAs per SM leave
    // room for two of each; D=256's 64 KB Q, K and V tiles leave one of each:
    // its QK^T then runs N = 128 MMAs, at the tensor peak, instead of N = 64)
    static constexpr int KST = (D == 64) ? 3 : (D == 128) ? 2 : 1;
    static constexpr int VST = (D == 256) ? 1 : 2;
    static constexpr int STAGES = KST > VST ? KST : VST;  // barrier array size
    static constexpr uint32_t Q_BYTES = NCH * BM * 128;
    static constexpr uint32_t KV_CHUNK = BN * 128;       // one 64-column box of a K or V tile
    static constexpr uint32_t KV_BYTES = NCH * KV_CHUNK; // one K (or V) tile
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + KST * KV_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_V + VST * KV_BYTES;
    // barriers: q_full, k_full[S], v_full[S], k_empty[S], v_empty[S], s_full[2], p_full[2], pv_done[2],
    // teardown, s_free.  K stages are released after their QK^T MMA and V stages after
    // their PV MMA, so the next K tiles load while the softmax still runs.
    // then, for split rows, x_full[4 quarters][2 parities]: the two halves of a
    // row exchange their partial maxima through TMEM columns COL_X..
    static constexpr int N_BARS = 1 + 4 * STAGES + 6 + 1 + 1 + 8;
    static constexpr uint32_t OFF_MISC = OFF_BAR + N_BARS * 8;
    static constexpr uint32_t SMEM_USED = OFF_MISC + 16;
    static constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;   // slack for 1024-byte alignment
    // TMEM columns: S buffers, O, P buffers (f16 pairs per column)
    static constexpr uint32_t COL_O = NBUF * BN;
    static constexpr uint32_t COL_P = COL_O + D;
    static constexpr uint32_t P_COLS = BN / 2;
    static constexpr uint32_t TMEM_COLS = (CTAS_PER_SM == 2) ? 256 : 512;
    static constexpr uint32_t COL_X = COL_P + NBUF * P_COLS;   // split rows: 4 max slots + 2 sum slots
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
    static_assert(COL_P + NBUF * P_COLS + (NSM == 8 ? 6 : 0) <= TMEM_COLS, "TMEM budget");
    static_assert(NSM == 4 || CTAS_PER_SM == 1, "split rows need one CTA per SM");
    // at most CTAS_PER_SM CTAs fit in an SM's 228 KB (1 KB reserved per CTA),
    // and together they never ask for more than the SM's 512 TMEM columns, so
    // no tcgen05.alloc waits on another CTA
    static_assert(CTAS_PER_SM * (SMEM_ALLOC + 1024) <= 233472, "CTAs per SM fit");
    static_assert((CTAS_PER_SM + 1) * (SMEM_ALLOC + 1024) > 233472, "no extra CTA per SM");
    static_assert(CTAS_PER_SM * TMEM_COLS <= 512, "TMEM per SM");
};

// A row whose exponentials against the running max sum to at most this (2 to the
// lazy-rescale threshold) keeps them: no tile max needed.
constexpr float kFastSumLimit = 256.0f;

// Per-warpgroup register budgets (all four warps of a warpgroup execute these).
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Max of a row of N logits with eight independent partial maxima (short
// dependency chains) and three-input max instructions.
template <int N>
__device__ __forceinline__ float row_max(const float (&t)[N]) {
    static_assert(N % 8 == 0 && N >= 16, "row length");
    float a[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) a[k] = t[k];
    int i = 8;
#pragma unroll
    for (; i + 16 <= N; i += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k) a[k] = max3(a[k], t[i + k], t[i + 8 + k]);
#pragma unroll
    for (; i < N; i += 8)
#pragma unroll
        for (int k = 0; k < 8; ++k) a[k] = fmaxf(a[k], t[i + k]);
    return fmaxf(max3(a[0], a[1], a[2]), max3(a[3], a[4], fmaxf(a[5], max3(a[6], a[7], a[0]))));
}

struct PrefillArgs {
    __half* out;
    float* lse;
    int S, Hq, Hkv, causal, window;
    float softcap, scale;
    int* err;
    // paged chunks only: sequence b's queries are packed rows q_start[b] ..
    // q_start[b+1]-1 at positions kv_len[b] - q_len + i over its kv_len[b] cached
    // keys, read through the page table in boxes of box_rows rows
    const int32_t* q_start;
    const int32_t* kv_len;
    const int32_t* page_table;
    int P, log2P, max_pages, n_pages, box_rows;
    int B, max_qt;     // sequences, query tiles of the longest chunk
    int lpt;           // 1: a 1-D grid walks (sequence, query tile) pairs longest first
    int total_q;       // rows of q/out (S for contiguous prefill)
};

// Chunks with at most this many (sequence, query tile) pairs are launched
// longest first: every CTA ranks all pairs by their key tiles.
constexpr int kLptMaxPairs = 128;

template <int D, int MODE, bool PAGED>
__global__ void __launch_bounds__(PrefillCfg<D>::THREADS, PrefillCfg<D>::CTAS_PER_SM)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const PrefillArgs args) {
    using C = PrefillCfg<D>;
    constexpr int BN = C::BN, NCH = C::NCH, STAGES = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    const int B_QFULL = 0;
    const int B_KFULL = 1, B_VFULL = 1 + STAGES, B_KEMPTY = 1 + 2 * STAGES, B_VEMPTY = 1 + 3 * STAGES;
    const int B_SFULL = 1 + 4 * STAGES, B_PFULL = B_SFULL + 2, B_PVDONE = B_SFULL + 4;
    const int B_TEARDOWN = B_SFULL + 6;
    const int B_SFREE = B_SFULL + 7;     // softmax has S in registers (single S buffer only)
    const int B_XFULL = B_SFULL + 8;     // split rows: [quarter][parity], 64 arrivals each
    constexpr int NBUF = C::NBUF;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Geometry.  Queries i in [0, n_q) of one sequence sit at positions pos0 + i
    // over keys [0, L); contiguous prefill has one sequence of S tokens with
    // positions 0 .. S-1, a paged chunk the last n_q of its sequence's tokens.
    const int W = args.window;
    // key tiles [jt0, jt0 + count) kept by queries q0 .. q_last at positions pos0 + i over L keys
    auto key_tiles = [&](int L_, int pos0_, int q0_, int q_last_, int& jt0_) {
        int hi_ = args.causal ? min(L_, pos0_ + q_last_ + 1) : L_;
        if (!args.causal && W > 0) hi_ = min(L_, q_last_ + W);
        const int lo_ = W > 0 ? max(0, pos0_ + q0_ - W + 1) : 0;
        jt0_ = lo_ / BN;
        return hi_ > lo_ ? (hi_ + BN - 1) / BN - jt0_ : 0;
    };
    // contiguous prefill: heads fastest (x), query tiles (y), so that the longest
    // causal tiles of every head launch first; paged chunks set these below
    int n_q = args.S, L = args.S, pos0 = 0, q_base = 0, b = 0, qt = 0, h = blockIdx.x;
    if constexpr (PAGED) {
        auto chunk_of = [&](int bb, int& qs, int& nq, int& Lb, int& p0) {
            qs = args.q_start[bb];
            nq = args.q_start[bb + 1] - qs;
            const int kvl = args.kv_len[bb];
            Lb = min(max(kvl, 0), args.max_pages * args.P);
            p0 = kvl - nq;
        };
        if (args.lpt) {
            // longest first across sequences: CTA x takes head x % Hq of the
            // (x / Hq)-th (sequence, query tile) pair, pairs ranked by the key
            // tiles of their sequence's longest query tile, then by their own
            // (ties by index).  The last wave holds the shortest CTAs, and the
            // query tiles of one sequence (which read the same pages) run next
            // to each other, so those pages come from DRAM about once.  The
            // scratch sits where Q lands, before any copy is issued.
            int* wk = reinterpret_cast<int*>(smem + C::OFF_Q);
            int* wseq = wk + kLptMaxPairs;
            int* sel = wseq + kLptMaxPairs;
            const int n_pairs = args.B * args.max_qt;
            if (threadIdx.x < n_pairs) {
                const int bb = threadIdx.x / args.max_qt, t = threadIdx.x % args.max_qt;
                int qs, nq, Lb, p0, j0, w = -1, ws = -1;   // -1: no queries, ranked last
                chunk_of(bb, qs, nq, Lb, p0);
                if (t * BM < nq) {
                    w = key_tiles(Lb, p0, t * BM, min(t * BM + BM - 1, nq - 1), j0);
                    const int tl = (nq - 1) / BM;
                    ws = key_tiles(Lb, p0, tl * BM, nq - 1, j0);
                }
                wk[threadIdx.x] = w;
                wseq[threadIdx.x] = ws;
            }
            __syncthreads();
            const int want = static_cast<int>(blockIdx.x) / args.Hq;
            if (threadIdx.x < n_pairs) {
                const int me = wk[threadIdx.x], ms = wseq[threadIdx.x];
                int rank = 0;
                for (int j = 0; j < n_pairs; ++j) {
                    const int o = wk[j], os = wseq[j];
                    rank += (os > ms || (os == ms && (o > me || (o == me && j < static_cast<int>(threadIdx.x))))) ? 1
                                                                                                                : 0;
                }
                if (rank == want) *sel = threadIdx.x;   // ranks are a permutation: one writer
            }
            __syncthreads();
            const int pair = *sel;
            b = pair / args.max_qt;
            qt = pair % args.max_qt;
            h = static_cast<int>(blockIdx.x) % args.Hq;
        } else {
            b = blockIdx.z;
            h = blockIdx.y;
            qt = static_cast<int>(gridDim.x - 1 - blockIdx.x);
        }
        chunk_of(b, q_base, n_q, L, pos0);
    }
    const int n_qt = (n_q + BM - 1) / BM;
    // causal tiles late in the sequence carry the most keys: launch them first
    if constexpr (!PAGED) qt = args.causal ? (n_qt - 1 - static_cast<int>(blockIdx.y)) : static_cast<int>(blockIdx.y);
    if (PAGED && qt >= n_qt) return;   // a shorter chunk: no queries for this CTA
    const int g = h / (args.Hq / args.Hkv);
    const int q0 = qt * BM;
    const int q_last = min(q0 + BM - 1, n_q - 1);
    int jt0;
    const int n_tiles = key_tiles(L, pos0, q0, q_last, jt0);

    if (threadIdx.x == 0) {
        mbar_init(bar(B_QFULL), 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(B_KFULL + s), 1);
            mbar_init(bar(B_VFULL + s), 1);
            mbar_init(bar(B_KEMPTY + s), 1);
            mbar_init(bar(B_VEMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_SFULL + b), 1);
            mbar_init(bar(B_PFULL + b), C::NSM * 32);
            mbar_init(bar(B_PVDONE + b), 1);
        }
        mbar_init(bar(B_TEARDOWN), 1);
        mbar_init(bar(B_SFREE), C::NSM * 32);
        for (int x = 0; x < 8; ++x) mbar_init(bar(B_XFULL + x), 64);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == C::MMA_WARP) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp >= C::NSM) {
        // (setmaxnreg is executed by all four warps of a warpgroup)
        if constexpr (C::THREADS == 256) setmaxnreg_dec<C::REG_OTHER>();
        if (warp == C::PROD_WARP || warp == C::PROD_V_WARP) {
            // ------------------------------------------------------------ TMA producers
            // One warp loads Q and the K tiles, another the V tiles, so that neither
            // waits behind the other's waits.  Contiguous: lane 0 of each.  Paged:
            // lanes 0-15 of each, lane i the box of the tile's i-th page (R rows; one
            // box inside a page when pages are longer than the tile), so the boxes of a
            // tile are issued in parallel; lane 0 waits for the stage and posts the
            // byte count.
            const int grp_lane = PAGED ? lane : 0;
            if (PAGED ? lane < 16 : lane == 0) {
                const bool is_k = warp == C::PROD_WARP;
                const bool leader = grp_lane == 0;
                const unsigned gmask = 0x0000ffffu;
                const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
                const uint32_t off = is_k ? C::OFF_K : C::OFF_V;
                const int b_full = is_k ? B_KFULL : B_VFULL, b_empty = is_k ? B_KEMPTY : B_VEMPTY;
                const int NST = is_k ? C::KST : C::VST;
                if (leader) tma_prefetch_desc(tm);
                if (is_k && leader) {
                    tma_prefetch_desc(&tm_q);
                    mbar_arrive_expect_tx(bar(B_QFULL), C::Q_BYTES);
                    for (int c = 0; c < NCH; ++c)
                        tma_load_3d(sbase + C::OFF_Q + c * (BM * 128), &tm_q, bar(B_QFULL), c * 64, h, q_base + q0);
                }
                int issued = 0;
                const int R = PAGED ? args.box_rows : BN;
                const bool has_box = grp_lane * R < BN;   // pages of >= 8 tokens: at most 16 boxes
                // the page id of this lane's box in tile j+1 is loaded right after tile j's
                // copies are issued, so its latency hides behind the wait for a free stage
                int pg = 0;
                auto fetch_page = [&](int j) {
                    const int kk = (jt0 + j) * BN + grp_lane * R;
                    pg = (has_box && j < n_tiles && kk < L)
                             ? __ldg(&args.page_table[(size_t)b * args.max_pages + (kk >> args.log2P)]) : 0;
                };
                if constexpr (PAGED) fetch_page(0);
                for (int j = 0; j < n_tiles; ++j) {
                    const int st = j % NST;
                    if (j >= NST) {
                        int ok = 1;
                        if (leader) ok = mbar_wait(bar(b_empty + st), ((j / NST) - 1) & 1, abort_flag, args.err,
                                                   kErrTimeoutSlot);
                        if constexpr (PAGED) ok = __shfl_sync(gmask, ok, 0);
                        if (!ok) break;
                    }
                    const int key0 = (jt0 + j) * BN;
                    if (leader) mbar_arrive_expect_tx(bar(b_full + st), C::KV_BYTES);
                    if constexpr (PAGED) {
                        __syncwarp(gmask);
                        // boxes past the cached keys get the page coordinate n_pages, past
                        // the pool, so the copy fills zeros instead of reading anything
                        if (has_box) {
                            const int kk = key0 + grp_lane * R;
                            int page = args.n_pages, row = 0;
                            if (kk < L) {
                                if (pg >= 0 && pg < args.n_pages) page = pg;
                                else atomicExch(args.err, kErrBadPage);   // never read: reported
                                row = kk & (args.P - 1);
                            }
                            for (int c = 0; c < NCH; ++c)
                                tma_load_4d(sbase + off + st * C::KV_BYTES + c * C::KV_CHUNK + grp_lane * R * 128,
                                            tm, bar(b_full + st), c * 64, g, row, page);
                        }
                        fetch_page(j + 1);
                    } else {
                        for (int c = 0; c < NCH; ++c)
                            tma_load_3d(sbase + off + st * C::KV_BYTES + c * C::KV_CHUNK, tm, bar(b_full + st), c * 64,
                                        g, key0);
                    }
                    issued = j + 1;
                }
                if (leader && *abort_flag) {
                    // let copies already in flight land before the CTA's shared memory goes away
                    // (the stage's byte count covers every lane's boxes)
                    if (is_k) mbar_wait_drain(bar(B_QFULL), 0, args.err, kErrTimeoutLoad);
                    for (int j = max(0, issued - NST); j < issued; ++j)
                        mbar_wait_drain(bar(b_full + (j % NST)), (j / NST) & 1, args.err, kErrTimeoutLoad);
                }
            }
        } else if (warp == C::MMA_WARP) {
            // ------------------------------------------------------------ MMA issuer
            if (lane == 0) {
                constexpr uint32_t idesc_s = idesc_f16_f32(BM, BN, false);
                constexpr uint32_t idesc_o = idesc_f16_f32(BM, D, true);
                bool ok = mbar_wait(bar(B_QFULL), 0, abort_flag, args.err, kErrTimeoutLoad);
                // testing hook: hold back the signal of the first S tile, so that the
                // softmax's wait for it runs out (the failure path, without a fault)
                const bool stall = stall_first_tile();
                // base descriptors, built once: each MMA's operands are a constant
                // offset from them (this thread shares its issue slots with softmax warps)
                const uint64_t q_desc = smem_desc_sw128(sbase + C::OFF_Q, 16, 1024);
                const uint64_t k_desc = smem_desc_sw128(sbase + C::OFF_K, 16, 1024);
                const uint64_t v_desc = smem_desc_sw128(sbase + C::OFF_V, C::KV_CHUNK, 1024);
                auto issue_s = [&](int j) {
                    const int st = j % C::KST;
                    const uint32_t d_tmem = tmem + (j % NBUF) * BN;
                    const uint64_t kd = desc_advance(k_desc, st * C::KV_BYTES);
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t a = desc_advance(q_desc, c * (BM * 128) + kk * 32);
                            const uint64_t b = desc_advance(kd, c * C::KV_CHUNK + kk * 32);
                            tc_mma_f16_ss(d_tmem, a, b, idesc_s, (c | kk) != 0);
                        }
                    }
                    if (!(stall && j == 0)) tc_commit(bar(B_SFULL + (j % NBUF)));
                    tc_commit(bar(B_KEMPTY + st));
                };
                if (ok && n_tiles > 0) {
                    ok = mbar_wait(bar(B_KFULL + 0), 0, abort_flag, args.err, kErrTimeoutLoad);
                    if (ok) {
                        tc_fence_after();
                        issue_s(0);
                    }
                }
                for (int j = 0; ok && j < n_tiles; ++j) {
                    if (j + 1 < n_tiles) {
                        const int st1 = (j + 1) % C::KST;
                        // a single S buffer is overwritten only once the softmax holds S_j in registers
                        if (NBUF == 1 &&
                            !mbar_wait(bar(B_SFREE), j & 1, abort_flag, args.err, kErrTimeoutSoftmax)) break;
                        if (!mbar_wait(bar(B_KFULL + st1), ((j + 1) / C::KST) & 1, abort_flag, args.err, kErrTimeoutLoad)) break;
                        tc_fence_after();
                        issue_s(j + 1);
                    }
                    if (!mbar_wait(bar(B_PFULL + (j % NBUF)), (j / NBUF) & 1, abort_flag, args.err, kErrTimeoutSoftmax)) break;
                    const int st = j % C::VST;
                    if (!mbar_wait(bar(B_VFULL + st), (j / C::VST) & 1, abort_flag, args.err, kErrTimeoutLoad)) break;
                    tc_fence_after();
                    const uint32_t p_tmem = tmem + C::COL_P + (j % NBUF) * C::P_COLS;
                    const uint64_t vd = desc_advance(v_desc, st * C::KV_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        // 16 keys per MMA: 8 TMEM columns of P, 16 rows of V (2048 bytes)
                        tc_mma_f16_ts(tmem + C::COL_O, p_tmem + kk * 8, desc_advance(vd, kk * 16 * 128), idesc_o,
                                      (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(bar(B_PVDONE + (j % NBUF)));
                    tc_commit(bar(B_VEMPTY + st));
                }
                // all issued MMAs must retire before TMEM is released
                tc_commit(bar(B_TEARDOWN));
                mbar_wait_drain(bar(B_TEARDOWN), 0, args.err, kErrTimeoutMma);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        if constexpr (C::THREADS == 256) setmaxnreg_inc<C::REG_SOFTMAX>();
        // split rows (D=256): warps w and w+4 share the TMEM lanes of quarter w%4
        // and take the first / second half of each tile's keys and of O's columns
        constexpr bool SPLIT = C::NSM == 8;
        constexpr int CW = C::CW;              // S columns of this thread
        constexpr int OW = D / (C::NSM / 4);   // O columns of this thread
        const int quarter = warp & 3;
        const int ch = SPLIT ? (warp >> 2) : 0;
        const int row = quarter * 32 + lane;   // 0..127 == TMEM lane
        const int qi = q0 + row;             // query index within the sequence
        const int pos = pos0 + qi;           // its position among the keys
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        // split rows: hand this thread's value to the other half of its row and
        // take that half's (through TMEM column slot `col`), on the quarter's
        // exchange barrier of parity k & 1; false if the wait gave up
        auto exchange = [&](float mine, uint32_t col, int k, float& other) -> bool {
            tc_st_32x32b_x1(lane_base + C::COL_X + col + ch, __float_as_uint(mine));
            tc_wait_st();
            tc_fence_before();
            const int xb = B_XFULL + quarter * 2 + (k & 1);
            mbar_arrive(bar(xb));
            if (!mbar_wait(bar(xb), (k >> 1) & 1, abort_flag, args.err, kErrTimeoutSoftmax)) return false;
            tc_fence_after();
            other = __uint_as_float(tc_ld_32x32b_x1(lane_base + C::COL_X + col + (ch ^ 1)));
            tc_wait_ld();
            return true;
        };
        const float scale_log2 = args.scale * kLog2e;
        const float cap_log2 = args.softcap * kLog2e;
        const float inv_cap_scale = MODE == kModeCapped ? args.scale / args.softcap : 0.f;
        float m_used = -INFINITY;   // running max actually used as the exponent offset (log2 units)
        float l_sum = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles && ok; ++j) {
            if (!mbar_wait(bar(B_SFULL + (j % NBUF)), (j / NBUF) & 1, abort_flag, args.err, kErrTimeoutMma)) { ok = false; break; }
            tc_fence_after();
            float t[CW];
            {
                uint32_t r[CW];
#pragma unroll
                for (int c = 0; c < CW / 32; ++c)
                    tc_ld_32x32b_x32(lane_base + (j % NBUF) * BN + ch * CW + c * 32,
                                     *reinterpret_cast<uint32_t(*)[32]>(r + c * 32));
                tc_wait_ld();
#pragma unroll
                for (int i = 0; i < CW; ++i) t[i] = __uint_as_float(r[i]);
            }
            const int key0 = (jt0 + j) * BN;
            const int key_last = key0 + BN - 1;
            bool full = key_last < L;
            if (args.causal) full = full && key_last <= pos;
            if (W > 0) full = full && (pos - key0 < W) && (args.causal || key_last - pos < W);
            // logits in log2 units (the raw mode keeps accumulators and scales in the exponent)
            if constexpr (MODE == kModeCapped) {
                // c*tanh(s/c) in log2 units: x times the even Taylor polynomial of
                // tanh(x)/x through x^6, its coefficients pre-multiplied by c*log2e, on the
                // FMA pipe (the dropped x^9 term is below 8.4e-8 for |x| <= 1/4); a warp
                // with any element outside that range recomputes its tile with the
                // exp/reciprocal form
                const float2 ics = make_float2(inv_cap_scale, inv_cap_scale);
                const float k1 = cap_log2 * (-1.0f / 3.0f), k2 = cap_log2 * (2.0f / 15.0f),
                            k3 = cap_log2 * (-17.0f / 315.0f);
                const float2 c0 = make_float2(cap_log2, cap_log2), c1 = make_float2(k1, k1),
                             c2 = make_float2(k2, k2), c3 = make_float2(k3, k3);
                float ax = 0.f;   // largest |x| of this thread's elements
#pragma unroll
                for (int i = 0; i < CW; i += 2) {
                    const float2 x = fmul2(make_float2(t[i], t[i + 1]), ics);
                    ax = fmaxf(ax, fmaxf(fabsf(x.x), fabsf(x.y)));
                    const float2 y = fmul2(x, x);
                    float2 q = ffma2(y, c3, c2);
                    q = ffma2(q, y, c1);
                    q = ffma2(q, y, c0);
                    const float2 r = fmul2(x, q);
                    t[i] = r.x;
                    t[i + 1] = r.y;
                }
                if (__any_sync(0xffffffffu, !(ax <= 0.25f))) {
                    uint32_t r[CW];
#pragma unroll
                    for (int c = 0; c < CW / 32; ++c)
                        tc_ld_32x32b_x32(lane_base + (j % NBUF) * BN + ch * CW + c * 32,
                                         *reinterpret_cast<uint32_t(*)[32]>(r + c * 32));
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < CW; ++i)
                        t[i] = cap_log2 * tanh_abs_accurate(__uint_as_float(r[i]) * inv_cap_scale);
                }
            } else if constexpr (MODE == kModeScaled) {
#pragma unroll
                for (int i = 0; i < CW; ++i) t[i] *= scale_log2;
            }
            if constexpr (NBUF == 1) {
                // S_j is in registers: the MMA warp may write S_{j+1}
                tc_fence_before();
                mbar_arrive(bar(B_SFREE));
            }
            if (!full) {
#pragma unroll
                for (int i = 0; i < CW; ++i) {
                    const int kj = key0 + ch * CW + i;
                    bool keep = kj < L;
                    if (args.causal) keep = keep && kj <= pos;
                    if (W > 0) {
                        int dist = pos - kj;
                        if (!args.causal && dist < 0) dist = -dist;
                        keep = keep && dist < W;
                    }
                    if (!keep) t[i] = -INFINITY;
                }
            }
            // P buffer j % NBUF is free once PV_{j-NBUF} has retired
            auto p_free = [&]() -> bool {
                return j < NBUF || mbar_wait(bar(B_PVDONE + (j % NBUF)), ((j - NBUF) / NBUF) & 1, abort_flag,
                                             args.err, kErrTimeoutMma);
            };
            const float2 sl2 = make_float2(scale_log2, scale_log2);
            const uint32_t p_addr = lane_base + C::COL_P + (j % NBUF) * C::P_COLS + ch * (CW / 2);
            // p = 2^(t*scale - m_off) (or 2^(t - m_off)) in packed f32x2 arithmetic, rounded to
            // f16 and stored to TMEM 32 elements at a time; returns the row's sum of the
            // ROUNDED p, the values the PV product multiplies, so that the output is a
            // convex combination of V rows (one dominant key gives its V row exactly)
            auto exps = [&](float m_off) -> float {
                float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // independent partial sums
                const float2 nm2 = make_float2(-m_off, -m_off);
#pragma unroll
                for (int c = 0; c < CW / 32; ++c) {
                    uint32_t packed[16];
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float2 ti = make_float2(t[c * 32 + i], t[c * 32 + i + 1]);
                        const float2 x = MODE == kModeRaw ? ffma2(ti, sl2, nm2) : fadd2(ti, nm2);
                        const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                        const __half2 hp = __floats2half2_rn(p.x, p.y);
                        packed[i / 2] = *reinterpret_cast<const uint32_t*>(&hp);
                        const int a = (i / 2) & 3;
                        ls[2 * a] = add_f16_lo(ls[2 * a], packed[i / 2]);
                        ls[2 * a + 1] = add_f16_hi(ls[2 * a + 1], packed[i / 2]);
                    }
                    tc_st_32x32b_x16(p_addr + c * 16, packed);
                }
                return ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
            };
            // Optimistic pass (D=128, whole rows): exponentials against the running max,
            // without the tile's max.  A row whose p sum to at most 2^8 has every p <= 2^8,
            // the bound the lazy rescale keeps; a warp with any other row (or a NaN) redoes
            // the tile below with the tile's max, overwriting P.  (Measured slower for
            // D=64, whose 128-key tiles keep the max computation off the critical path.)
            bool fast = false;
            if constexpr (!SPLIT && D == 128) {
                if (__all_sync(0xffffffffu, m_used != -INFINITY)) {
                    if (!p_free()) { ok = false; break; }
                    const float lsum = exps(m_used);
                    if (!__any_sync(0xffffffffu, !(lsum <= kFastSumLimit))) {
                        l_sum += lsum;
                        fast = true;
                    }
                }
            }
            bool rescale = false;
            float alpha_o = 1.f;
            if (!fast) {
                float mx = row_max(t);
                if constexpr (SPLIT) {
                    float other;
                    if (!exchange(mx, 2 * (j & 1), j, other)) { ok = false; break; }
                    mx = fmaxf(mx, other);
                }
                const float m_tile = MODE == kModeRaw ? mx * scale_log2 : mx;
                const bool need = m_tile > m_used + kRescaleThreshold || (m_used == -INFINITY && m_tile > -INFINITY);
                // the warp rescales O (below, once t[] is no longer live) if any of its rows moved its max
                rescale = __any_sync(0xffffffffu, need) && j > 0;
                if (need) {
                    const float m_new = fmaxf(m_tile, m_used);
                    const float alpha = (m_used == -INFINITY) ? 0.f : ex2_approx(m_used - m_new);
                    alpha_o = alpha;
                    l_sum *= alpha;
                    m_used = m_new;
                }
                const float m_off = (m_used == -INFINITY) ? 0.f : m_used;
                if (!p_free()) { ok = false; break; }
                l_sum += exps(m_off);
            }
            if (rescale) {
                // O must not be in flight while it is rescaled (PV_j waits for p_full below)
                if (NBUF > 1 &&
                    !mbar_wait(bar(B_PVDONE + ((j - 1) % NBUF)), ((j - 1) / NBUF) & 1, abort_flag, args.err, kErrTimeoutMma)) { ok = false; break; }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < OW / 32; ++c) {
                    uint32_t r[32];
                    tc_ld_32x32b_x32(lane_base + C::COL_O + ch * OW + c * 32, r);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha_o);
                    tc_st_32x32b_x32(lane_base + C::COL_O + ch * OW + c * 32, r);
                }
            }
            if constexpr (PAGED) {
                if (key0 + BN > L) {
                    // keys past the cache: zero their V rows, since the cache may hold
                    // anything there and P = 0 must not meet a NaN
                    const int stv = j % C::VST;
                    if (!mbar_wait(bar(B_VFULL + stv), (j / C::VST) & 1, abort_flag, args.err, kErrTimeoutLoad)) {
                        ok = false;
                        break;
                    }
                    const int r0 = max(L - key0, 0);
                    const int per_chunk = (BN - r0) * 8;          // 16-byte units per chunk
                    uint8_t* vt = smem + C::OFF_V + stv * C::KV_BYTES;
                    for (int u = ch * BM + row; u < NCH * per_chunk; u += C::NSM * 32) {
                        const int c = u / per_chunk, rem = u - c * per_chunk;
                        *reinterpret_cast<uint4*>(vt + c * C::KV_CHUNK + (r0 + rem / 8) * 128 + (rem % 8) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
            }
            tc_wait_st();
            tc_fence_before();
            mbar_arrive(bar(B_PFULL + (j % NBUF)));
        }
        // ------------------------------------------------------------ epilogue
        if (ok && n_tiles > 0) {
            const int jl = n_tiles - 1;
            ok = mbar_wait(bar(B_PVDONE + (jl % NBUF)), (jl / NBUF) & 1, abort_flag, args.err, kErrTimeoutMma);
        }
        if constexpr (SPLIT) {
            // the row sum is the two halves' sums
            float other = 0.f;
            if (ok) ok = exchange(l_sum, 4, n_tiles, other);
            l_sum += other;
        }
        // D=256: whole tiles leave through shared memory and tiled bulk stores (rows past
        // S are clipped by the tensor map).  Row by row, each thread's 256 bytes per
        // 128 columns would go out as 16-byte pieces 4 KB apart, one L2 sector per lane
        // and store; D=64/128 have a quarter or half of that and keep the direct stores,
        // which let the CTA retire without waiting for a bulk copy.  A chunk's last,
        // partial tile is stored row by row, since the rows after it belong to the next
        // sequence.  The staging area is Q's: every MMA has retired.
        bool via_tma = D == 256;
        if constexpr (PAGED) via_tma = via_tma && q0 + BM <= n_q && q_base >= 0 && q_base + q0 + BM <= args.total_q;
        uint8_t* stage = smem + C::OFF_Q;
        if (ok) {
            tc_fence_after();
            const float inv_l = l_sum > 0.f ? 1.0f / l_sum : 0.f;
            // a row of this chunk, inside q/out even if q_start disagrees with total_q
            const bool row_ok = qi < n_q && q_base + qi >= 0 && q_base + qi < args.total_q;
            __half* orow = args.out + (static_cast<size_t>(q_base + qi) * args.Hq + h) * D;
#pragma unroll 1
            for (int c = 0; c < OW / 32; ++c) {
                float o[32];
                if (n_tiles > 0) {
                    uint32_t r[32];
                    tc_ld_32x32b_x32(lane_base + C::COL_O + ch * OW + c * 32, r);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(r[i]) * inv_l;
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0.f;   // no key at all: O was never written
                }
                uint32_t hv[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const __half2 p2 = __floats2half2_rn(o[2 * i], o[2 * i + 1]);
                    hv[i] = *reinterpret_cast<const uint32_t*>(&p2);
                }
                if (via_tma) {
                    // columns col0 .. col0+31 of this row: 16-byte units u0 .. u0+3 of its
                    // 128-byte line in chunk col0 / 64, at the 128-byte swizzle's positions
                    const int col0 = ch * OW + c * 32;
                    uint8_t* line = stage + (col0 >> 6) * (BM * 128) + row * 128;
                    const int u0 = (col0 & 63) >> 3;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        *reinterpret_cast<uint4*>(line + (((u0 + i) ^ (row & 7)) << 4)) =
                            make_uint4(hv[4 * i], hv[4 * i + 1], hv[4 * i + 2], hv[4 * i + 3]);
                } else if (row_ok) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + ch * OW + c * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(hv[4 * i], hv[4 * i + 1], hv[4 * i + 2], hv[4 * i + 3]);
                }
            }
            if (args.lse && row_ok && ch == 0) {
                args.lse[static_cast<size_t>(q_base + qi) * args.Hq + h] =
                    l_sum > 0.f ? (m_used + __log2f(l_sum)) * 0.6931471805599453f : -INFINITY;
            }
        }
        if (via_tma) {
            // every softmax thread's staged lines are visible to the bulk copy, then
            // one thread stores the tile and waits until its reads of shared memory are done
            fence_proxy_async_smem();
            named_bar_sync(1, C::NSM * 32);
            if (threadIdx.x == 0 && ok) {
#pragma unroll
                for (int c = 0; c < NCH; ++c) tma_store_3d(&tm_o, smem_u32(stage + c * (BM * 128)), c * 64, h, q_base + q0);
                tma_store_commit();
                tma_store_wait_read();
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == C::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D, int MODE, bool PAGED>
attn_status launch_prefill_dm(const PrefillLaunch& L) {
    using C = PrefillCfg<D>;
    CUtensorMap tq, tk, tv, to;
    attn_status st;
    int box_rows = C::BN;
    if (!PAGED) {
        // 3-D maps over [S, H, D] f16: dims (D, H, S), 64-element x rows boxes, 128-byte swizzle
        if ((st = encode_tmap_3d_f16_sw128(&tq, L.q, D, L.Hq, L.S, BM)) != ATTN_OK) return st;
        if ((st = encode_tmap_3d_f16_sw128(&to, L.out, D, L.Hq, L.S, BM)) != ATTN_OK) return st;
        if ((st = encode_tmap_3d_f16_sw128(&tk, L.k, D, L.Hkv, L.S, C::BN)) != ATTN_OK) return st;
        if ((st = encode_tmap_3d_f16_sw128(&tv, L.v, D, L.Hkv, L.S, C::BN)) != ATTN_OK) return st;
    } else {
        // q [total_q, Hq, D] as above; the pool [n_pages, P, Hkv, D] as (D, Hkv, P, n_pages)
        // with boxes of (64, 1 head, min(P, tile keys) rows, 1 page)
        if ((st = encode_tmap_3d_f16_sw128(&tq, L.q, D, L.Hq, L.total_q, BM)) != ATTN_OK) return st;
        if ((st = encode_tmap_3d_f16_sw128(&to, L.out, D, L.Hq, L.total_q, BM)) != ATTN_OK) return st;
        box_rows = L.page_size < C::BN ? L.page_size : C::BN;
        const uint64_t dims[4] = {(uint64_t)D, (uint64_t)L.Hkv, (uint64_t)L.page_size, (uint64_t)L.n_pages};
        const uint64_t strides[3] = {(uint64_t)D * 2, (uint64_t)D * 2 * L.Hkv,
                                     (uint64_t)D * 2 * L.Hkv * L.page_size};
        const uint32_t box[4] = {64u, 1u, (uint32_t)box_rows, 1u};
        if ((st = encode_tmap_sw128(&tk, L.k, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, dims, strides, box)) != ATTN_OK)
            return st;
        if ((st = encode_tmap_sw128(&tv, L.v, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, dims, strides, box)) != ATTN_OK)
            return st;
    }
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(prefill_tc_kernel<D, MODE, PAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM_ALLOC) != cudaSuccess)
            return set_error(ATTN_ECUDA, "cudaFuncSetAttribute(prefill smem) failed");
        attr_set[dev] = true;
    }
    PrefillArgs a;
    a.out = static_cast<__half*>(L.out);
    a.lse = L.lse;
    a.S = L.S;
    a.Hq = L.Hq;
    a.Hkv = L.Hkv;
    a.causal = L.causal;
    a.window = L.window;
    a.softcap = L.softcap;
    a.scale = L.scale;
    a.err = L.err_word;
    a.q_start = L.q_start;
    a.kv_len = L.kv_len;
    a.page_table = L.page_table;
    a.P = L.page_size;
    a.log2P = 0;
    while ((1 << a.log2P) < L.page_size) ++a.log2P;
    a.max_pages = L.max_pages;
    a.n_pages = L.n_pages;
    a.box_rows = box_rows;
    a.total_q = PAGED ? L.total_q : L.S;
    a.B = L.B;
    a.max_qt = PAGED ? (L.max_q + BM - 1) / BM : 0;
    const int n_pairs = L.B * a.max_qt;
    a.lpt = PAGED && n_pairs <= kLptMaxPairs;
    // contiguous: heads fastest, then query tiles (longest first when causal)
    const dim3 grid = !PAGED ? dim3(L.Hq, (L.S + BM - 1) / BM)
                      : a.lpt ? dim3(n_pairs * L.Hq) : dim3(a.max_qt, L.Hq, L.B);
    if (trace_enabled())
        trace("prefill_tc_kernel<D=%d,mode=%s,paged=%d> grid=(%u,%u,%u) block=%d smem=%u tmem_cols=%u "
              "ctas_per_sm=%d key_tile=%d S=%d Hq=%d Hkv=%d causal=%d window=%d softcap=%g scale=%g%s",
              D, MODE == kModeRaw ? "raw" : MODE == kModeScaled ? "scaled" : "capped", (int)PAGED, grid.x, grid.y,
              grid.z, C::THREADS, C::SMEM_ALLOC, C::TMEM_COLS, C::CTAS_PER_SM, C::BN, PAGED ? L.total_q : L.S,
              L.Hq, L.Hkv, L.causal, L.window, L.softcap, L.scale,
              PAGED ? (a.lpt ? " order=heads fastest, sequences longest first, their query tiles together" : " order=(tile,head,seq)")
                    : L.causal ? " order=heads fastest, longest query tiles first" : " order=heads fastest");
    prefill_tc_kernel<D, MODE, PAGED><<<grid, C::THREADS, C::SMEM_ALLOC, L.stream>>>(tq, tk, tv, to, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(ATTN_ECUDA, "prefill launch failed: %s", cudaGetErrorString(e));
    return ATTN_OK;
}

template <int D, bool PAGED>
attn_status launch_prefill_d(const PrefillLaunch& L) {
    if (L.softcap > 0.f) return launch_prefill_dm<D, kModeCapped, PAGED>(L);
    if (L.scale > 0.f) return launch_prefill_dm<D, kModeRaw, PAGED>(L);
    return launch_prefill_dm<D, kModeScaled, PAGED>(L);
}

template <bool PAGED>
attn_status launch_prefill_p(const PrefillLaunch& L) {
    switch (L.D) {
        case 64: return launch_prefill_d<64, PAGED>(L);
        case 128: return launch_prefill_d<128, PAGED>(L);
        case 256: return launch_prefill_d<256, PAGED>(L);
        default: return set_error(ATTN_EUNSUPPORTED, "head_dim %d not supported (64, 128, 256)", L.D);
    }
}

}  // namespace

attn_status launch_prefill(const PrefillLaunch& L) {
    return L.paged ? launch_prefill_p<true>(L) : launch_prefill_p<false>(L);
}

// Sets this translation unit's test controls (see ptx.cuh).
attn_status set_test_controls_prefill(unsigned long long wait_limit_ns, int stall) {
    if (cudaMemcpyToSymbol(g_wait_limit_ns, &wait_limit_ns, sizeof(wait_limit_ns)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_stall_first_tile, &stall, sizeof(stall)) != cudaSuccess)
        return set_error(ATTN_ECUDA, "test controls (prefill): %s", cudaGetErrorString(cudaGetLastError()));
    return ATTN_OK;
}

}  // namespace attn
