// decode_tc.cuh -- split-KV decode with both contractions on the tcgen05
// tensor cores (f16 caches, head_dim 64 or 128, contiguous or paged with
// pages of a multiple of 16 tokens).  Included by decode.cu, whose work-item
// enumeration (sequence, head block, split), partial-row workspace and
// log-sum-exp combine pass it shares; only the per-split kernel differs.
//
// Same computation as decode_split_kernel (doppler attention.js, the decode
// variants of executeAttention): for each query head h of kv head g, softmax
// over the kept keys of scale * q_h . k_j applied to v_j, here accumulated per
// split with an online softmax and merged across splits by the combine pass.
//
// A work item covers the up-to-32 query heads of one head block.  Each TMA
// box holds 16 tokens x NH kv heads x 64 dims of K (or V) with the 128-byte
// swizzle, so NBX = 8 / NH boxes of consecutive 16-token groups stack into a
// 128-row operand whose row m is (token m / NH, kv head m % NH):
//
//   S   = Q' K^T   M=128, N=128 rows of the tile, K=D; f32 in TMEM.  Q' is the
//                  A operand in TMEM: lane 32w + r holds query row r of the
//                  block for every lane quadrant w, so each quadrant holds the
//                  whole S of the block
//   P   = exp2(S * scale * log2 e - m)  softmax warp w owns quadrant w and, of
//                  the tile's 128 rows, the 32 rows 32w..32w+31: one thread
//                  per query head keeps the entries of its own kv head (every
//                  NH-th row), runs its own online softmax over them, and
//                  writes them as f16 into its lane's P words 16w..16w+15
//                  (the rest of its P row stays zero)
//   O  += P V      M=128, N=D, K=128 (P from TMEM, V in shared memory as the
//                  MN-major operand): lane 32w + r sums quadrant w's rows only,
//                  so each quadrant accumulates its own partial O
//
// At the end of a run the four quadrant partials (m_w, l_w, O_w) of each head
// are merged by log-sum-exp through shared memory, in a fixed order.  The MMA
// does no more work than one quadrant would (M=128 is its smallest useful
// shape), and four warps share each tile's softmax with no per-tile exchange.
// Roles (192 threads): warps 0-3 softmax, Q' loads and the per-run epilogue;
// warp 4 TMA producers (lane 0: K, lane 1: V); warp 5 TMEM allocator + MMA
// issuer, which issues whichever of the next QK^T and the next PV is ready.
// Shared memory holds little besides the K and V rings (three tiles each for
// D=128), which keep enough copies in flight to cover HBM latency.  S has one
// TMEM buffer, released as soon as the softmax holds its quarter in
// registers, so the next QK^T overlaps the exponentials; O has two, and the
// epilogue of a run runs after the first tile of the next one, so no MMA
// waits for it.  Keys outside the split (window start, sequence end, boxes
// never loaded) are masked in the softmax, and their V rows are zeroed in
// shared memory before the PV product so that stale or unwritten cache
// contents never reach it.

namespace tcdec {

constexpr int kSoftmaxWarps = 4;
constexpr int kThreads = (kSoftmaxWarps + 2) * 32;   // softmax warps, producer warp, MMA warp
constexpr int kProdWarp = kSoftmaxWarps, kMmaWarp = kSoftmaxWarps + 1;
constexpr int TR = 128;                       // rows of the K/V operand per MMA tile
constexpr int QROWS = 32;                     // query rows of a head block (NW units x up to 4 heads)
constexpr int kMaxBatch = 2048;               // sequences per call (two prefixes live in shared memory)

// Q2: f32 queries, held as two f16 terms (q = hi + lo to 2^-22 relative) in
// two TMEM regions; every QK^T step runs a second MMA on the lo terms into the
// same accumulator.
template <int D, bool Q2 = false>
struct Cfg {
    static constexpr int NCH = D / 64;                         // 64-dim (128-byte) chunks
    static constexpr uint32_t CHUNK = TR * 128;                // one chunk of a K or V tile
    static constexpr uint32_t KV_BYTES = NCH * CHUNK;          // one K (or V) tile
    // the run epilogue: quadrants 1-3 hand warp 0 their scaled partial O in
    // chunks of 32 columns ([3][32 columns][32 rows] f32), and every quadrant
    // its (m, l) per head ([2 parities][4][32] float2)
    static constexpr uint32_t XCH = 3 * 32 * 32 * 4;
    static constexpr uint32_t OFF_X = 0;
    static constexpr uint32_t OFF_ML = OFF_X + XCH;
    static constexpr uint32_t OFF_RING = (OFF_ML + 2 * 4 * 32 * 8 + 1023) / 1024 * 1024;
    static constexpr uint32_t PREFIX_ONE = ((kMaxBatch + 1) * 4 + 127) / 128 * 128;
    static constexpr uint32_t PREFIX_BYTES = 2 * PREFIX_ONE;   // item prefix, tile prefix
    // Separate K and V rings: a K tile is released once its QK^T has run, a V
    // tile only once its PV has run (after the softmax), so V gets the deeper
    // ring when the tiles are odd in number.
    static constexpr int NTILE_RAW = (int)((226u * 1024u - OFF_RING - PREFIX_BYTES - 1024u - 512u) / KV_BYTES);
    static constexpr int NV = ((NTILE_RAW + 1) / 2) > 6 ? 6 : (NTILE_RAW + 1) / 2;   // V ring slots
    static constexpr int NK = (NTILE_RAW - NV) > 6 ? 6 : NTILE_RAW - NV;            // K ring slots
    static constexpr uint32_t OFF_VRING = OFF_RING + NK * KV_BYTES;
    static constexpr uint32_t OFF_BARS = OFF_VRING + NV * KV_BYTES;
    // barriers: k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], q_full, s_full,
    // s_free, p_full, pv_done[2], o_free[2], teardown, ml_full, x_full, x_free
    static constexpr int N_BARS = 2 * NK + 2 * NV + 14;
    static constexpr uint32_t OFF_PREFIX = OFF_BARS + N_BARS * 8;
    static constexpr uint32_t OFF_MISC = OFF_PREFIX + PREFIX_BYTES;   // scan scratch, abort flag, TMEM base
    static constexpr uint32_t SMEM_USED = OFF_MISC + 256;
    static constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
    // TMEM columns: S (128), P (64: 128 f16 keys), O[NOB] (D each), Q' (D/2 per
    // f16 term).  f32 queries with D=128 keep one O buffer to fit.
    static constexpr int NOB = (Q2 && D == 128) ? 1 : 2;
    static constexpr uint32_t COL_S = 0, COL_P = 128, COL_O = 192;
    static constexpr uint32_t COL_Q = COL_O + NOB * D;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(COL_Q + (Q2 ? 2 : 1) * (D / 2) <= TMEM_COLS, "TMEM budget");
    static_assert(NK >= 2 && NV >= 2, "rings too small");
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

// the NH candidates c[0..NH) -> c[sel] with a select tree on the bits of sel
template <int NH>
__device__ __forceinline__ float pick(const uint32_t* c, int sel) {
    if constexpr (NH == 1) {
        return __uint_as_float(c[0]);
    } else if constexpr (NH == 2) {
        return __uint_as_float((sel & 1) ? c[1] : c[0]);
    } else if constexpr (NH == 4) {
        const uint32_t a0 = (sel & 1) ? c[1] : c[0], a1 = (sel & 1) ? c[3] : c[2];
        return __uint_as_float((sel & 2) ? a1 : a0);
    } else {
        const uint32_t a0 = (sel & 1) ? c[1] : c[0], a1 = (sel & 1) ? c[3] : c[2];
        const uint32_t a2 = (sel & 1) ? c[5] : c[4], a3 = (sel & 1) ? c[7] : c[6];
        const uint32_t b0 = (sel & 2) ? a1 : a0, b1 = (sel & 2) ? a3 : a2;
        return __uint_as_float((sel & 4) ? b1 : b0);
    }
}

// Work split.  The MMA tiles of a launch are numbered sequence by sequence,
// head block by head block: (b, hb) has Tb tiles of TT tokens from the first
// kept key rounded down to 16.  CTA c takes tiles [c*NT/G, (c+1)*NT/G) of the
// NT in total, so every CTA streams the same amount of cache whatever the
// sequence lengths.  Consecutive tiles of one (b, hb) form a run with one
// online softmax.  A run that starts where a split of the item enumeration
// starts writes its partial into that item's row and -inf lse into the rows
// of the items that start inside it; only a CTA's first run can start inside
// an item, and it writes a fix-up slot of its own, tagged with (b, hb), which
// the combine pass merges with the item rows.
struct TileCur {
    int x, x_end;          // current tile, end of this CTA's range
    int b, hb, t, Tb;      // sequence, head block, tile within (b, hb), tiles per (b, hb)
    int a, start, end;     // first token of tile 0 (16-aligned), kept keys [start, end)
    int run;               // index of the current run within this CTA
    bool first, last;      // first / last tile of its run
};

template <int TT>
__device__ __forceinline__ void tcur_locate(TileCur& c, const int* tpref, const DecArgs& A) {
    int lo = 0, hi = A.B;   // largest b with tpref[b] <= x: a sequence with tiles
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tpref[mid] <= c.x) lo = mid; else hi = mid;
    }
    c.b = lo;
    tier_range(A, lo, c.start, c.end);
    c.a = (c.start / 16) * 16;
    c.Tb = (tpref[lo + 1] - tpref[lo]) / A.n_hb;
    const int rel = c.x - tpref[lo];
    c.hb = rel / c.Tb;
    c.t = rel - c.hb * c.Tb;
}
template <int TT>
__device__ __forceinline__ void tcur_mark_last(TileCur& c) {
    c.last = (c.t + 1 == c.Tb) || (c.x + 1 == c.x_end);
}
template <int TT>
__device__ __forceinline__ void tcur_start(TileCur& c, const int* tpref, const DecArgs& A) {
    const long long nt = tpref[A.B];
    c.x = (int)((long long)blockIdx.x * nt / gridDim.x);
    c.x_end = (int)((long long)(blockIdx.x + 1) * nt / gridDim.x);
    c.run = 0;
    c.first = true;
    if (c.x < c.x_end) {
        tcur_locate<TT>(c, tpref, A);
        tcur_mark_last<TT>(c);
    }
}
template <int TT>
__device__ __forceinline__ void tcur_next(TileCur& c, const int* tpref, const DecArgs& A) {
    if (++c.x >= c.x_end) return;
    c.first = false;
    if (++c.t == c.Tb) {
        ++c.run;
        c.first = true;
        c.t = 0;
        if (++c.hb == A.n_hb) tcur_locate<TT>(c, tpref, A);
    }
    tcur_mark_last<TT>(c);
}

template <int D, int NH, bool Q2>
__global__ void __launch_bounds__(kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v, const DecArgs A,
                 const int q_rows) {
    using C = Cfg<D, Q2>;
    constexpr int NCH = C::NCH, NK = C::NK, NV = C::NV, NOB = C::NOB;
    constexpr int TT = TR / NH;                 // tokens per MMA tile
    constexpr int TQ = TT / kSoftmaxWarps;      // tokens of a tile in one quadrant
    constexpr int NXC = D / 32;                 // 32-column chunks of O merged per run
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
    int* pref = reinterpret_cast<int*>(smem + C::OFF_PREFIX);     // item prefix over sequences
    int* tpref = reinterpret_cast<int*>(smem + C::OFF_PREFIX + C::PREFIX_ONE);   // tile prefix over sequences
    int* scratch = reinterpret_cast<int*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 128);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC + 132);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    const int B_KFULL = 0, B_KEMPTY = NK, B_VFULL = 2 * NK, B_VEMPTY = 2 * NK + NV, B_QFULL = 2 * NK + 2 * NV,
              B_SFULL = B_QFULL + 1, B_SFREE = B_SFULL + 1, B_PFULL = B_SFREE + 1, B_PVDONE = B_PFULL + 1,
              B_OFREE = B_PVDONE + 2, B_TEARDOWN = B_OFREE + 2, B_MLFULL = B_TEARDOWN + 1, B_XFULL = B_MLFULL + 1,
              B_XFREE = B_XFULL + 1;
    constexpr int NSMT = kSoftmaxWarps * 32;    // softmax threads

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t kv_policy = l2_policy_evict_first();   // the cache is read once
    if (threadIdx.x == 0) {
        for (int s = 0; s < NK; ++s) {
            mbar_init(bar(B_KFULL + s), 1);
            mbar_init(bar(B_KEMPTY + s), 1);
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(bar(B_VFULL + s), 1);
            mbar_init(bar(B_VEMPTY + s), 1);
        }
        mbar_init(bar(B_QFULL), NSMT);
        mbar_init(bar(B_SFULL), 1);
        mbar_init(bar(B_SFREE), NSMT);
        mbar_init(bar(B_PFULL), NSMT);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_PVDONE + b), 1);
            mbar_init(bar(B_OFREE + b), NSMT);
        }
        mbar_init(bar(B_TEARDOWN), 1);
        mbar_init(bar(B_MLFULL), NSMT);
        mbar_init(bar(B_XFULL), NSMT - 32);     // quadrants 1-3
        mbar_init(bar(B_XFREE), 32);            // warp 0
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    build_prefix(A, pref, scratch);   // ends with __syncthreads
    build_prefix_of(A, tpref, scratch, [&](int start, int end) {
        return end > start ? A.n_hb * ((end - (start / 16) * 16 + TT - 1) / TT) : 0;
    });
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    if (blockIdx.x == 0) {
        for (int b = threadIdx.x; b <= A.B; b += blockDim.x) A.ws_prefix[b] = pref[b];
    }
    const int GH = A.G / A.HG;                  // query heads per unit
    const int QB = NW * GH;                     // query rows of a head block

    if (warp == kProdWarp) {
        // ------------------------------------------------------------ TMA producers
        // lane 0 loads the K tiles, lane 1 the V tiles; each waits only for its own ring
        if (lane < 2) {
            const bool is_k = lane == 0;
            const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
            const int NS = is_k ? NK : NV;
            const int b_full = is_k ? B_KFULL : B_VFULL, b_empty = is_k ? B_KEMPTY : B_VEMPTY;
            const uint32_t ring = sbase + (is_k ? C::OFF_RING : C::OFF_VRING);
            tma_prefetch_desc(tm);
            TileCur c;
            tcur_start<TT>(c, tpref, A);
            uint32_t j = 0;
            bool ok = true;
            for (; c.x < c.x_end; tcur_next<TT>(c, tpref, A), ++j) {
                const int slot = j % NS;
                if (j >= (uint32_t)NS &&
                    !mbar_wait(bar(b_empty + slot), ((j / NS) - 1) & 1, abort_flag, A.err, kErrTimeoutSlot)) {
                    ok = false;
                    break;
                }
                const int g0 = (c.hb * NW) / A.HG;
                const int t0 = c.a + c.t * TT;
                // boxes of R rows (16, or the page size when pages are shorter, with
                // R * NH >= 8 so that every box starts 1024-byte aligned, as the
                // 128-byte swizzle requires); boxes wholly past the end are skipped
                const int R = A.R;
                const int nbox = (min(TT, c.end - t0) + R - 1) / R;
                mbar_arrive_expect_tx(bar(b_full + slot), nbox * NCH * R * NH * 128);
                for (int bx = 0; bx < nbox; ++bx) {
                    const int tk = t0 + bx * R;
                    int page = c.b, row = A.ring > 0 ? tk % A.ring : tk;   // ring: slot t % ring (ring % 16 == 0)
                    if (A.paged) {
                        page = __ldg(&A.page_table[(size_t)c.b * A.max_pages + (tk >> A.logP)]);
                        if (page < 0 || page >= A.n_pages) {
                            // a page id outside the pool: read page 0 instead and report it
                            atomicExch(A.err, kErrBadPage);
                            page = 0;
                        }
                        row = tk & (A.P - 1);
                    }
#pragma unroll
                    for (int ch = 0; ch < NCH; ++ch)
                        tma_load_4d_hint(ring + slot * C::KV_BYTES + ch * C::CHUNK + bx * R * NH * 128, tm,
                                         bar(b_full + slot), ch * 64, g0, row, page, kv_policy);
                }
            }
            if (!ok) {
                // let copies in flight land before shared memory is released
                const uint32_t first = j > (uint32_t)NS ? j - NS : 0;
                for (uint32_t x = first; x < j; ++x)
                    mbar_wait_drain(bar(b_full + (x % NS)), (x / NS) & 1, A.err, kErrTimeoutLoad);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // One thread issues whichever is ready first: the next QK^T (its run's Q'
        // in TMEM, the single S buffer released by the softmax, its K tile) or
        // the next PV (its P written, its V tile, and for the first PV of a run
        // its O buffer read out by the epilogue of the run that used it before).
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_f16_f32(128, TR, false);
            constexpr uint32_t idesc_o = idesc_f16_f32(128, D, true);
            TileCur cs, cp;                   // next S to issue, next PV to issue
            tcur_start<TT>(cs, tpref, A);
            tcur_start<TT>(cp, tpref, A);
            uint32_t js = 0, jp = 0;          // S and PV issued
            // testing hook: hold back the signal of the first S tile, so that the
            // softmax's wait for it runs out (the failure path, without a fault)
            const bool stall = stall_first_tile();
            const uint64_t limit = *static_cast<volatile unsigned long long*>(&g_wait_limit_ns);
            uint64_t t_idle = globaltimer();
            // base descriptors, built once: each MMA's operand is a constant offset
            // from them (this thread shares its issue slots with a softmax warp)
            const uint64_t k_desc = smem_desc_sw128(sbase + C::OFF_RING, 16, 1024);
            const uint64_t v_desc = smem_desc_sw128(sbase + C::OFF_VRING, C::CHUNK, 1024);
            for (uint32_t spin = 0; cs.x < cs.x_end || cp.x < cp.x_end; ++spin) {
                bool progress = false;
                if (cs.x < cs.x_end) {
                    const int slot = js % NK;
                    if ((!cs.first || mbar_test_wait(bar(B_QFULL), cs.run & 1)) &&
                        (js == 0 || mbar_test_wait(bar(B_SFREE), (js - 1) & 1)) &&
                        mbar_test_wait(bar(B_KFULL + slot), (js / NK) & 1)) {
                        tc_fence_after();
                        const uint64_t kd = desc_advance(k_desc, slot * C::KV_BYTES);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint64_t b = desc_advance(kd, (kk >> 2) * C::CHUNK + (kk & 3) * 32);
                            tc_mma_f16_ts(tmem + C::COL_S, tmem + C::COL_Q + kk * 8, b, idesc_s, kk != 0);
                            if constexpr (Q2)
                                tc_mma_f16_ts(tmem + C::COL_S, tmem + C::COL_Q + D / 2 + kk * 8, b, idesc_s, 1u);
                        }
                        if (!(stall && js == 0)) tc_commit(bar(B_SFULL));
                        tc_commit(bar(B_KEMPTY + slot));
                        ++js;
                        tcur_next<TT>(cs, tpref, A);
                        progress = true;
                    }
                }
                if (jp < js) {
                    const int slot = jp % NV;
                    const int ob = cp.run % NOB;
                    if (mbar_test_wait(bar(B_PFULL), jp & 1) &&
                        (!cp.first || cp.run < NOB || mbar_test_wait(bar(B_OFREE + ob), ((cp.run / NOB) - 1) & 1)) &&
                        mbar_test_wait(bar(B_VFULL + slot), (jp / NV) & 1)) {
                        tc_fence_after();
                        const uint64_t vd = desc_advance(v_desc, slot * C::KV_BYTES);
#pragma unroll
                        for (int kk = 0; kk < TR / 16; ++kk) {
                            // 16 rows per MMA: 8 TMEM columns of P, 16 rows of V (2048 bytes)
                            const uint64_t b = desc_advance(vd, kk * 16 * 128);
                            tc_mma_f16_ts(tmem + C::COL_O + ob * D, tmem + C::COL_P + kk * 8, b, idesc_o,
                                          (!cp.first || kk > 0) ? 1u : 0u);
                        }
                        tc_commit(bar(B_PVDONE + (jp & 1)));
                        tc_commit(bar(B_VEMPTY + slot));
                        ++jp;
                        tcur_next<TT>(cp, tpref, A);
                        progress = true;
                    }
                }
                if (progress) {
                    spin = 0;
                } else if ((spin & 31u) == 31u) {
                    if (*abort_flag) break;
                    const uint64_t now = globaltimer();
                    if (spin == 31u) t_idle = now;
                    else if (now - t_idle > limit) {
                        *abort_flag = 1;
                        atomicExch(A.err, kErrTimeoutSoftmax);
                        break;
                    }
                }
            }
            // all issued MMAs must retire before TMEM is released
            tc_commit(bar(B_TEARDOWN));
            mbar_wait_drain(bar(B_TEARDOWN), 0, A.err, kErrTimeoutMma);
        }
    } else {
        // ------------------------------------------------------------ softmax (warps 0-3)
        const int qd = warp;                        // TMEM lane quadrant = tile rows 32*qd .. +31
        const int r = lane;                         // query row of the head block
        const int wu = r / GH, hs = r - wu * GH;    // unit of the head block, head inside it
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(qd * 32) << 16);
        float2* ml = reinterpret_cast<float2*>(smem + C::OFF_ML);       // [2][4][32] (m, l)
        float* xb = reinterpret_cast<float*>(smem + C::OFF_X);           // [3][32 cols][32 rows]

        // this lane's P row starts at zero; a tile only ever writes its own
        // quadrant's 16 words, so the rest of the row stays zero
        {
            uint32_t z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0u;
            tc_st_32x32b_x32(lane_base + C::COL_P, z);
            tc_st_32x32b_x32(lane_base + C::COL_P + 32, z);
        }
        // Q' of a run: query row r of head block hb of sequence b (zeros past the
        // block's rows or the heads), written to this lane's Q' columns: f16 pairs
        // in the A-operand layout (Q2: the hi terms, then the lo terms)
        auto q_row = [&](int b, int hb) -> bool {
            const int head = hb * QB + r;
            const bool valid = r < q_rows && r < QB && head < A.Hq;
            const size_t qoff = ((size_t)b * A.Hq + head) * D;
#pragma unroll 1
            for (int cc = 0; cc < D / 64; ++cc) {
                uint32_t hi[32];
                if constexpr (!Q2) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint4 w = valid ? __ldg(reinterpret_cast<const uint4*>(A.q + qoff + cc * 64) + i)
                                              : make_uint4(0u, 0u, 0u, 0u);
                        hi[4 * i] = w.x;
                        hi[4 * i + 1] = w.y;
                        hi[4 * i + 2] = w.z;
                        hi[4 * i + 3] = w.w;
                    }
                    tc_st_32x32b_x32(lane_base + C::COL_Q + cc * 32, hi);
                } else {
                    uint32_t lo[32];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float4 x = valid ? __ldg(reinterpret_cast<const float4*>(A.q32 + qoff + cc * 64) + i)
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
                        const __half2 h0 = __floats2half2_rn(x.x, x.y), h1 = __floats2half2_rn(x.z, x.w);
                        const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
                        const __half2 l0 = __floats2half2_rn(x.x - f0.x, x.y - f0.y);
                        const __half2 l1 = __floats2half2_rn(x.z - f1.x, x.w - f1.y);
                        hi[2 * i] = *reinterpret_cast<const uint32_t*>(&h0);
                        hi[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&h1);
                        lo[2 * i] = *reinterpret_cast<const uint32_t*>(&l0);
                        lo[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&l1);
                    }
                    tc_st_32x32b_x32(lane_base + C::COL_Q + cc * 32, hi);
                    tc_st_32x32b_x32(lane_base + C::COL_Q + D / 2 + cc * 32, lo);
                }
            }
            tc_wait_st();
            tc_fence_before();
            mbar_arrive(bar(B_QFULL));
            return true;
        };
        // the first tile of the run after the one that contains tile c (none: b = -1)
        auto next_run = [&](const TileCur& c, int& nb, int& nhb) {
            TileCur n = c;
            n.x = c.x + (c.Tb - c.t);
            nb = -1;
            if (n.x < c.x_end) {
                tcur_locate<TT>(n, tpref, A);
                nb = n.b;
                nhb = n.hb;
            }
        };

        TileCur c;
        tcur_start<TT>(c, tpref, A);
        // the fix-up tag of this CTA: (b, hb) if its first run starts inside a split
        if (qd == 0 && lane == 0) {
            int tag = -1;
            if (c.x < c.x_end && (c.t * TT) % A.split != 0) tag = c.b * A.n_hb + c.hb;
            A.ws_fix_meta[blockIdx.x] = tag;
        }
        if (c.x < c.x_end) q_row(c.b, c.hb);       // the first run's Q'
        bool ok = true;

        // a run's epilogue, run one tile late: the four quadrant partials of this
        // thread's query head merged by log-sum-exp (weights 2^(m_w - M) in a fixed
        // order), then (lse, o / l) into the item row (or the fix-up slot) and -inf
        // into the rows of the items that start inside the run
        struct Pending {
            bool on, act;
            int b, hb, t_first, t_last, ob, ns;
            uint32_t j_last;
            float m, l;
        } pend;
        pend.on = false;
        uint32_t n_epi = 0;                         // epilogues run so far (barrier parities)
        auto epilogue = [&]() -> bool {
            if (!mbar_wait(bar(B_PVDONE + (pend.j_last & 1)), (pend.j_last >> 1) & 1, abort_flag, A.err, kErrTimeoutMma))
                return false;
            tc_fence_after();
            const uint32_t e = n_epi++;
            ml[((e & 1) * kSoftmaxWarps + qd) * 32 + r] = make_float2(pend.m, pend.l);
            mbar_arrive(bar(B_MLFULL));
            if (!mbar_wait(bar(B_MLFULL), e & 1, abort_flag, A.err, kErrTimeoutSoftmax)) return false;
            float mq[kSoftmaxWarps], lq[kSoftmaxWarps];
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kSoftmaxWarps; ++w) {
                const float2 v = ml[((e & 1) * kSoftmaxWarps + w) * 32 + r];
                mq[w] = v.x;
                lq[w] = v.y;
                M = fmaxf(M, v.x);
            }
            float L = 0.f, wmine = 0.f;
#pragma unroll
            for (int w = 0; w < kSoftmaxWarps; ++w) {
                const float a = lq[w] > 0.f ? ex2_approx(mq[w] - M) : 0.f;
                L += a * lq[w];
                if (w == qd) wmine = a;
            }
            const float f = L > 0.f ? wmine / L : 0.f;     // this quadrant's factor on O_w
            const int f0 = pend.t_first * TT;          // first token of the run, from the sequence's tile 0
            const int item0 = pref[pend.b] + pend.hb * pend.ns;
            float* o_dst = nullptr;
            float* l_dst = nullptr;
            if (qd == 0) {
                if (f0 % A.split == 0) {
                    const size_t prow = ((size_t)(item0 + f0 / A.split) * NW + wu) * GH + hs;
                    o_dst = A.ws_o + prow * D;
                    l_dst = A.ws_lse + prow;
                } else {
                    const size_t prow = ((size_t)blockIdx.x * NW + wu) * GH + hs;
                    o_dst = A.ws_fix_o + prow * D;
                    l_dst = A.ws_fix_lse + prow;
                }
            }
#pragma unroll 1
            for (int q = 0; q < NXC; ++q) {
                const uint32_t u = e * NXC + q;        // uses of the exchange buffer so far
                uint32_t o[32];
                tc_ld_32x32b_x32(lane_base + C::COL_O + pend.ob * D + q * 32, o);
                tc_wait_ld();
                if (qd != 0) {
                    // quadrants 1-3: hand f_w * O_w to warp 0 ([column][row]: conflict-free)
                    if (u > 0 && !mbar_wait(bar(B_XFREE), (u - 1) & 1, abort_flag, A.err, kErrTimeoutSoftmax))
                        return false;
                    float* dst = xb + (qd - 1) * 32 * 32;
#pragma unroll
                    for (int i = 0; i < 32; ++i) dst[i * 32 + r] = f != 0.f ? __uint_as_float(o[i]) * f : 0.f;
                    mbar_arrive(bar(B_XFULL));
                } else {
                    float acc[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[i] = f != 0.f ? __uint_as_float(o[i]) * f : 0.f;
                    if (!mbar_wait(bar(B_XFULL), u & 1, abort_flag, A.err, kErrTimeoutSoftmax)) return false;
#pragma unroll
                    for (int w = 0; w < 3; ++w)
#pragma unroll
                        for (int i = 0; i < 32; ++i) acc[i] += xb[(w * 32 + i) * 32 + r];
                    mbar_arrive(bar(B_XFREE));
                    if (pend.act) {
                        float4* dst4 = reinterpret_cast<float4*>(o_dst + q * 32);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst4[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
                    }
                }
            }
            if (qd == 0 && pend.act) {
                *l_dst = L > 0.f ? M + __log2f(L) : -INFINITY;
                const int s_hi = min(((pend.t_last + 1) * TT - 1) / A.split, pend.ns - 1);
                for (int sp = f0 / A.split + 1; sp <= s_hi; ++sp)
                    A.ws_lse[((size_t)(item0 + sp) * NW + wu) * GH + hs] = -INFINITY;
            }
            tc_fence_before();
            mbar_arrive(bar(B_OFREE + pend.ob));
            pend.on = false;
            return true;
        };

        uint32_t j = 0;
        bool act = false;
        int gl = 0, t_first = 0;
        float m_used = -INFINITY, l_sum = 0.f;
        for (; ok && c.x < c.x_end; tcur_next<TT>(c, tpref, A), ++j) {
            if (c.first) {
                const int u = c.hb * NW + wu;
                act = wu < NW && r < QB && u < A.U;
                gl = act ? u / A.HG - (c.hb * NW) / A.HG : 0;   // kv head inside the tile (row % NH)
                t_first = c.t;
                m_used = -INFINITY;
                l_sum = 0.f;
                // bring the next run's query row into L2 now: it is loaded at this run's end
                int nb, nhb;
                next_run(c, nb, nhb);
                const int head = nhb * QB + r;
                if (nb >= 0 && r < q_rows && r < QB && head < A.Hq) {
                    const char* row = Q2 ? reinterpret_cast<const char*>(A.q32 + ((size_t)nb * A.Hq + head) * D)
                                         : reinterpret_cast<const char*>(A.q + ((size_t)nb * A.Hq + head) * D);
#pragma unroll
                    for (int o = 0; o < D * (Q2 ? 4 : 2); o += 128) prefetch_l2(row + o);
                }
            }
            const int ob = c.run % NOB;
            if (!mbar_wait(bar(B_SFULL), j & 1, abort_flag, A.err, kErrTimeoutMma)) { ok = false; break; }
            tc_fence_after();
            float s[TQ];
            {
                uint32_t v[32];
                tc_ld_32x32b_x32(lane_base + C::COL_S + qd * 32, v);
                tc_wait_ld();
                tc_fence_before();
                mbar_arrive(bar(B_SFREE));         // S is in registers: the next QK^T may run
#pragma unroll
                for (int t = 0; t < TQ; ++t) s[t] = pick<NH>(v + t * NH, gl);
            }
            if (c.last) {
                // the run's last QK^T has run, so Q' may be replaced: the next run's
                // query rows (the MMA waits for them before its first QK^T)
                int nb, nhb;
                next_run(c, nb, nhb);
                if (nb >= 0) q_row(nb, nhb);
            }

            // this quadrant's tokens of the tile: tok0 .. tok0 + TQ - 1
            const int t0 = c.a + c.t * TT;
            const int tok0 = qd * TQ;
            const int v_lo = max(c.start - t0, 0);
            const int v_hi = min(c.end - t0, TT);
            float mx = -INFINITY;
#pragma unroll
            for (int t = 0; t < TQ; ++t) {
                float x = s[t] * A.qscale;
                if (A.cap_log2 > 0.f) x = A.cap_log2 * tanh_abs_accurate(x);
                x = (act && tok0 + t >= v_lo && tok0 + t < v_hi) ? x : -INFINITY;
                s[t] = x;
                mx = fmaxf(mx, x);
            }
            const bool need = mx > m_used + kRescaleThreshold || (m_used == -INFINITY && mx > -INFINITY);
            const bool rescale = __any_sync(0xffffffffu, need) && !c.first;
            float alpha = 1.f;
            if (need) {
                const float m_new = fmaxf(mx, m_used);
                alpha = (m_used == -INFINITY) ? 0.f : ex2_approx(m_used - m_new);
                l_sum *= alpha;
                m_used = m_new;
            }
            const float m_off = (m_used == -INFINITY) ? 0.f : m_used;
            // this quadrant's 16 words of the P row (32 f16 entries, tile rows
            // 32*qd .. +31); the row sum is taken over the rounded values the PV
            // product multiplies (a convex combination of V rows)
            uint32_t pw[16];
            float ls0 = 0.f, ls1 = 0.f;
            if constexpr (NH == 1) {
#pragma unroll
                for (int t = 0; t < TQ; t += 2) {
                    const float p0 = ex2_approx(s[t] - m_off), p1 = ex2_approx(s[t + 1] - m_off);
                    const __half2 h2 = __floats2half2_rn(p0, p1);
                    const uint32_t w = *reinterpret_cast<const uint32_t*>(&h2);
                    ls0 = add_f16_lo(ls0, w);
                    ls1 = add_f16_hi(ls1, w);
                    pw[t / 2] = act ? w : 0u;
                }
            } else {
                const int hp = gl >> 1;
#pragma unroll
                for (int t = 0; t < TQ; ++t) {
                    const float p = ex2_approx(s[t] - m_off);
                    const uint32_t h = __half_as_ushort(__float2half_rn(p));
                    if (t & 1) ls1 = add_f16_lo(ls1, h); else ls0 = add_f16_lo(ls0, h);
                    const uint32_t word = act ? ((gl & 1) ? (h << 16) : h) : 0u;
#pragma unroll
                    for (int w = 0; w < NH / 2; ++w) pw[t * (NH / 2) + w] = (w == hp) ? word : 0u;
                }
            }
            l_sum += ls0 + ls1;
            // the single P buffer and O: PV_{j-1} must have retired
            if (j >= 1) {
                if (!mbar_wait(bar(B_PVDONE + ((j - 1) & 1)), ((j - 1) >> 1) & 1, abort_flag, A.err, kErrTimeoutMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            if (rescale) {
                // this quadrant's rows of O
#pragma unroll 1
                for (int q = 0; q < D / 32; ++q) {
                    uint32_t o[32];
                    tc_ld_32x32b_x32(lane_base + C::COL_O + ob * D + q * 32, o);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tc_st_32x32b_x32(lane_base + C::COL_O + ob * D + q * 32, o);
                }
            }
            tc_st_32x32b_x16(lane_base + C::COL_P + qd * 16, pw);
            // zero the V rows of this quadrant's masked tokens (all NH heads, every
            // chunk), once the tile's copy has landed: P is zero there, and stale or
            // unwritten cache rows must not meet it
            const int z_lo = tok0, z_lo_end = min(v_lo, tok0 + TQ);
            const int z_hi = max(v_hi, tok0), z_hi_end = tok0 + TQ;
            if (z_lo < z_lo_end || z_hi < z_hi_end) {
                if (!mbar_wait(bar(B_VFULL + (j % NV)), (j / NV) & 1, abort_flag, A.err, kErrTimeoutLoad)) { ok = false; break; }
                uint8_t* vt = smem + C::OFF_VRING + (j % NV) * C::KV_BYTES;
#pragma unroll 1
                for (int ch = 0; ch < NCH; ++ch) {
                    uint8_t* cb = vt + ch * C::CHUNK;
                    for (int o = z_lo * NH * 128 + lane * 16; o < z_lo_end * NH * 128; o += 32 * 16)
                        *reinterpret_cast<uint4*>(cb + o) = make_uint4(0u, 0u, 0u, 0u);
                    for (int o = z_hi * NH * 128 + lane * 16; o < z_hi_end * NH * 128; o += 32 * 16)
                        *reinterpret_cast<uint4*>(cb + o) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            tc_wait_st();
            tc_fence_before();
            mbar_arrive(bar(B_PFULL));
            // the previous run's epilogue, now that this run's first P is out
            if (pend.on && !epilogue()) { ok = false; break; }
            if (c.last) {
                pend.on = true;
                pend.act = act;
                pend.b = c.b;
                pend.hb = c.hb;
                pend.t_first = t_first;
                pend.t_last = c.t;
                pend.ob = ob;
                pend.ns = seq_splits(c.start, c.end, A.split);
                pend.j_last = j;
                pend.m = m_used;
                pend.l = l_sum;
            }
        }
        if (ok && pend.on) epilogue();
    }
    tc_fence_before();
    __syncthreads();
    // this CTA's partials are written: the combine pass may be scheduled (it
    // still waits for the whole grid to finish)
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace tcdec
