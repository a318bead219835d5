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
//   S   = Q' K^T   M=128 (rows 0-31: the block's query heads, loaded by TMA
//                  from q), N=128 rows of the tile, K=D; f32 in TMEM
//   P   = exp2(S * scale * log2 e - m)  one thread of warp 0 per query head:
//                  it keeps the entries of its own kv head (every NH-th
//                  column), zeros the rest, and writes the row to TMEM as f16
//   O  += P V      M=128, N=D, K=128 (P from TMEM, V in shared memory as the
//                  MN-major operand): P is zero off its kv head, so each
//                  query head only sums its own head's values
//
// Rows 32-127 of S/P/O are never read.  Roles (96 threads): warp 0 softmax +
// per-split epilogue, warp 1 TMA producers (lane 0: Q' and K, lane 1: V),
// warp 2 TMEM allocator + MMA issuer.  S has one TMEM buffer, released as soon
// as the softmax holds its row in registers, so the next QK^T still overlaps
// the exponentials; P and O have two, and the epilogue of a split runs after
// the first tile of the next one, so no MMA waits for it.
// Keys outside the split (window start, sequence end, boxes never loaded) are
// masked in the softmax, and their V rows are zeroed in shared memory before
// the PV product so that stale or unwritten cache contents never reach it.

namespace tcdec {

constexpr int kThreads = 96;
constexpr int TR = 128;                       // rows of the K/V operand per MMA tile
constexpr int QROWS = 32;                     // query rows written (NW units x up to 4 heads)
constexpr int kMaxBatch = 2048;               // sequences per call (two prefixes live in shared memory)

// Q2: f32 queries, held as two f16 terms (q = hi + lo to 2^-22 relative): a
// Q' chunk keeps hi in rows 0-31 and lo in rows 32-63, and every QK^T step
// runs a second MMA on the lo rows into the same accumulator.
template <int D, bool Q2 = false>
struct Cfg {
    static constexpr int NCH = D / 64;                         // 64-dim (128-byte) chunks
    static constexpr uint32_t CHUNK = TR * 128;                // one chunk of a K or V tile
    static constexpr uint32_t KV_BYTES = NCH * CHUNK;          // one K (or V) tile
    static constexpr uint32_t Q_LO = QROWS * 128;              // offset of the lo rows in a chunk
    static constexpr uint32_t QCH = (Q2 ? 2 : 1) * QROWS * 128;   // one chunk of Q' (32 or 64 rows)
    static constexpr uint32_t QBUF = NCH * QCH;
    static constexpr uint32_t OFF_Q = 0;                       // two Q' buffers
    static constexpr uint32_t OFF_RING = 2 * QBUF;             // the MMA reads 128 rows from a Q'
    // chunk; rows 32-127 run on into the rings (never used), so the K ring must
    // hold at least 96 more rows of 128 bytes after the last Q' chunk.
    // Separate K and V rings: a K tile is released once its QK^T has run, a V
    // tile once its PV has run, so K loads run further ahead.
    static constexpr int NTILE_RAW = (int)((226u * 1024u - OFF_RING - 1024u - 4096u) / KV_BYTES);
    static constexpr int NK = (NTILE_RAW / 2) > 6 ? 6 : NTILE_RAW / 2;   // K ring slots
    static constexpr int NV = NK;                                      // V ring slots
    static constexpr uint32_t OFF_VRING = OFF_RING + NK * KV_BYTES;
    static constexpr uint32_t OFF_BARS = OFF_VRING + NV * KV_BYTES;
    // barriers: k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], q_full[2], q_empty[2],
    // s_full, s_free, p_full[2], pv_done[2], o_free[2], teardown
    static constexpr int N_BARS = 2 * NK + 2 * NV + 15;
    static constexpr uint32_t OFF_PREFIX = OFF_BARS + N_BARS * 8;
    static constexpr uint32_t PREFIX_ONE = ((kMaxBatch + 1) * 4 + 127) / 128 * 128;
    static constexpr uint32_t PREFIX_BYTES = 2 * PREFIX_ONE;        // item prefix, tile prefix
    static constexpr uint32_t OFF_MISC = OFF_PREFIX + PREFIX_BYTES;   // scan scratch, abort flag, TMEM base
    static constexpr uint32_t SMEM_USED = OFF_MISC + 256;
    static constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
    // TMEM columns: S (128), P[2] (64 each: 128 f16 keys), O[2] (D each)
    static constexpr uint32_t COL_S = 0, COL_P = 128, COL_O = 256;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(COL_O + 2 * D <= TMEM_COLS, "TMEM budget");
    static_assert(NK >= 2 && NV >= 2, "rings too small");
    static_assert(NK * KV_BYTES >= 3 * QCH, "Q' overrun stays inside the K ring");
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
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const DecArgs A, const int q_rows) {
    using C = Cfg<D, Q2>;
    constexpr int NCH = C::NCH, NK = C::NK, NV = C::NV;
    constexpr int NBX = 8 / NH;                 // 16-token boxes per MMA tile
    constexpr int TT = TR / NH;                 // tokens per MMA tile
    constexpr uint32_t BOXB = 16 * NH * 128;    // bytes of one box (one chunk)
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
              B_QEMPTY = B_QFULL + 2, B_SFULL = B_QEMPTY + 2, B_SFREE = B_SFULL + 1, B_PFULL = B_SFREE + 1,
              B_PVDONE = B_PFULL + 2, B_OFREE = B_PVDONE + 2, B_TEARDOWN = B_OFREE + 2;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NK; ++s) {
            mbar_init(bar(B_KFULL + s), 1);
            mbar_init(bar(B_KEMPTY + s), 1);
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(bar(B_VFULL + s), 1);
            mbar_init(bar(B_VEMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_QFULL + b), 1);
            mbar_init(bar(B_QEMPTY + b), 1);
            mbar_init(bar(B_PFULL + b), 32);
            mbar_init(bar(B_PVDONE + b), 1);
            mbar_init(bar(B_OFREE + b), 32);
        }
        mbar_init(bar(B_SFULL), 1);
        mbar_init(bar(B_SFREE), 32);
        mbar_init(bar(B_TEARDOWN), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 2) {
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

    if (warp == 1) {
        // ------------------------------------------------------------ TMA producers
        // lane 0 loads Q' (once per run) and the K tiles, lane 1 the V tiles;
        // each waits only for its own buffers
        if (lane < 2) {
            const bool is_k = lane == 0;
            const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
            const int NS = is_k ? NK : NV;
            const int b_full = is_k ? B_KFULL : B_VFULL, b_empty = is_k ? B_KEMPTY : B_VEMPTY;
            const uint32_t ring = sbase + (is_k ? C::OFF_RING : C::OFF_VRING);
            tma_prefetch_desc(tm);
            if (is_k) tma_prefetch_desc(&tm_q);
            TileCur c;
            tcur_start<TT>(c, tpref, A);
            uint32_t j = 0;
            int q_last[2] = {-1, -1};   // last run whose Q' was loaded into each buffer
            bool ok = true;
            for (; c.x < c.x_end; tcur_next<TT>(c, tpref, A), ++j) {
                if (is_k && c.first) {
                    // Q' of this run: query heads hb*QB .. +q_rows of sequence b
                    const int qb = c.run & 1;
                    if (c.run >= 2 &&
                        !mbar_wait(bar(B_QEMPTY + qb), ((c.run >> 1) - 1) & 1, abort_flag, A.err, kErrTimeoutSlot)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(B_QFULL + qb), (Q2 ? 2 : 1) * NCH * q_rows * 128);
                    q_last[qb] = c.run;
#pragma unroll
                    for (int ch = 0; ch < NCH; ++ch) {
                        tma_load_3d(sbase + C::OFF_Q + qb * C::QBUF + ch * C::QCH, &tm_q, bar(B_QFULL + qb), ch * 64,
                                    c.hb * QB, c.b);
                        // Q2: the lo terms sit B "sequences" further on in the same map
                        if constexpr (Q2)
                            tma_load_3d(sbase + C::OFF_Q + qb * C::QBUF + ch * C::QCH + C::Q_LO, &tm_q,
                                        bar(B_QFULL + qb), ch * 64, c.hb * QB, c.b + A.B);
                    }
                }
                const int slot = j % NS;
                if (j >= (uint32_t)NS &&
                    !mbar_wait(bar(b_empty + slot), ((j / NS) - 1) & 1, abort_flag, A.err, kErrTimeoutSlot)) {
                    ok = false;
                    break;
                }
                const int g0 = (c.hb * NW) / A.HG;
                const int t0 = c.a + c.t * TT;
                const int nbox = min(NBX, (c.end - t0 + 15) / 16);
                mbar_arrive_expect_tx(bar(b_full + slot), nbox * NCH * BOXB);
                for (int bx = 0; bx < nbox; ++bx) {
                    const int tk = t0 + bx * 16;
                    int page = c.b, row = A.ring > 0 ? tk % A.ring : tk;   // ring: slot t % ring (ring % 16 == 0)
                    if (A.paged) {
                        page = __ldg(&A.page_table[(size_t)c.b * A.max_pages + tk / A.P]);
                        if (page < 0 || page >= A.n_pages) {
                            // a page id outside the pool: read page 0 instead and report it
                            atomicExch(A.err, kErrBadPage);
                            page = 0;
                        }
                        row = tk % A.P;
                    }
#pragma unroll
                    for (int ch = 0; ch < NCH; ++ch)
                        tma_load_4d(ring + slot * C::KV_BYTES + ch * C::CHUNK + bx * BOXB, tm, bar(b_full + slot),
                                    ch * 64, g0, row, page);
                }
            }
            if (!ok) {
                // let copies in flight land before shared memory is released
                const uint32_t first = j > (uint32_t)NS ? j - NS : 0;
                for (uint32_t x = first; x < j; ++x)
                    mbar_wait_drain(bar(b_full + (x % NS)), (x / NS) & 1, A.err, kErrTimeoutLoad);
                for (int qb = 0; qb < 2; ++qb)
                    if (q_last[qb] >= 0) mbar_wait_drain(bar(B_QFULL + qb), (q_last[qb] >> 1) & 1, A.err, kErrTimeoutLoad);
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_f16_f32(128, TR, false);
            constexpr uint32_t idesc_o = idesc_f16_f32(128, D, true);
            TileCur cs, cp;                   // next S to issue, next PV to issue
            tcur_start<TT>(cs, tpref, A);
            tcur_start<TT>(cp, tpref, A);
            uint32_t js = 0;                  // tiles whose S has been issued
            bool ok = true;
            // testing hook: hold back the signal of the first S tile, so that the
            // softmax's wait for it runs out (the failure path, without a fault)
            const bool stall = stall_first_tile();
            // S_js: Q' of its run (buffer run & 1) times the K tile of ring slot js
            auto issue_s = [&]() -> bool {
                const int slot = js % NK;
                if (cs.first &&
                    !mbar_wait(bar(B_QFULL + (cs.run & 1)), (cs.run >> 1) & 1, abort_flag, A.err, kErrTimeoutLoad))
                    return false;
                // the single S buffer: the softmax has tile js-1 in registers
                if (js > 0 && !mbar_wait(bar(B_SFREE), (js - 1) & 1, abort_flag, A.err, kErrTimeoutSoftmax)) return false;
                if (!mbar_wait(bar(B_KFULL + slot), (js / NK) & 1, abort_flag, A.err, kErrTimeoutLoad)) return false;
                tc_fence_after();
                const uint32_t qb = sbase + C::OFF_Q + (cs.run & 1) * C::QBUF;
                const uint32_t kb = sbase + C::OFF_RING + slot * C::KV_BYTES;
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t a = smem_desc_sw128(qb + ch * C::QCH + kk * 32, 16, 1024);
                        const uint64_t b = smem_desc_sw128(kb + ch * C::CHUNK + kk * 32, 16, 1024);
                        tc_mma_f16_ss(tmem + C::COL_S, a, b, idesc_s, (ch | kk) != 0);
                        if constexpr (Q2) {
                            const uint64_t a_lo = smem_desc_sw128(qb + ch * C::QCH + C::Q_LO + kk * 32, 16, 1024);
                            tc_mma_f16_ss(tmem + C::COL_S, a_lo, b, idesc_s, 1u);
                        }
                    }
                if (!(stall && js == 0)) tc_commit(bar(B_SFULL));
                tc_commit(bar(B_KEMPTY + slot));
                if (cs.last) tc_commit(bar(B_QEMPTY + (cs.run & 1)));   // last S of the run
                ++js;
                tcur_next<TT>(cs, tpref, A);
                return true;
            };
            if (cs.x < cs.x_end) ok = issue_s();
            for (uint32_t j = 0; ok && cp.x < cp.x_end; ++j, tcur_next<TT>(cp, tpref, A)) {
                // S_{j+1} first (it waits for the softmax to hold S_j), so QK^T of
                // the next tile overlaps the exponentials of this one
                if (cs.x < cs.x_end && !(ok = issue_s())) break;
                if (!mbar_wait(bar(B_PFULL + (j & 1)), (j >> 1) & 1, abort_flag, A.err, kErrTimeoutSoftmax)) break;
                const int ob = cp.run & 1;
                // the first PV of a run overwrites its O buffer: the epilogue of the
                // run that used it before must have read it
                if (cp.first && cp.run >= 2 &&
                    !mbar_wait(bar(B_OFREE + ob), ((cp.run >> 1) - 1) & 1, abort_flag, A.err, kErrTimeoutSoftmax))
                    break;
                const int slot = j % NV;
                if (!mbar_wait(bar(B_VFULL + slot), (j / NV) & 1, abort_flag, A.err, kErrTimeoutLoad)) break;
                tc_fence_after();
                const uint32_t vb = sbase + C::OFF_VRING + slot * C::KV_BYTES;
                const uint32_t p_tmem = tmem + C::COL_P + (j & 1) * 64;
#pragma unroll
                for (int kk = 0; kk < TR / 16; ++kk) {
                    // 16 rows per MMA: 8 TMEM columns of P, 16 rows of V (2048 bytes)
                    const uint64_t b = smem_desc_sw128(vb + kk * 16 * 128, C::CHUNK, 1024);
                    tc_mma_f16_ts(tmem + C::COL_O + ob * D, p_tmem + kk * 8, b, idesc_o, (!cp.first || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar(B_PVDONE + (j & 1)));
                tc_commit(bar(B_VEMPTY + slot));
            }
            // all issued MMAs must retire before TMEM is released
            tc_commit(bar(B_TEARDOWN));
            mbar_wait_drain(bar(B_TEARDOWN), 0, A.err, kErrTimeoutMma);
        }
    } else {
        // ------------------------------------------------------------ softmax (warp 0)
        const int r = lane;                         // query row = TMEM lane
        const int wu = r / GH, hs = r - wu * GH;    // unit of the head block, head inside it
        const uint32_t lane_base = tmem;            // warp 0: TMEM lanes 0-31

        TileCur c;
        tcur_start<TT>(c, tpref, A);
        // the fix-up tag of this CTA: (b, hb) if its first run starts inside a split
        if (lane == 0) {
            int tag = -1;
            if (c.x < c.x_end && (c.t * TT) % A.split != 0) tag = c.b * A.n_hb + c.hb;
            A.ws_fix_meta[blockIdx.x] = tag;
        }

        // a run's epilogue, run one tile late: (lse, o / l) of this thread's query
        // head into the item row (or the fix-up slot), -inf into the rows of the
        // items that start inside the run
        struct Pending {
            bool on, act;
            int b, hb, t_first, t_last, ob, ns;
            uint32_t j_last;
            float m, l;
        } pend;
        pend.on = false;
        auto epilogue = [&]() -> bool {
            if (!mbar_wait(bar(B_PVDONE + (pend.j_last & 1)), (pend.j_last >> 1) & 1, abort_flag, A.err, kErrTimeoutMma))
                return false;
            tc_fence_after();
            const float inv = pend.l > 0.f ? 1.0f / pend.l : 0.f;
            const int f = pend.t_first * TT;          // first token of the run, from the sequence's tile 0
            const int item0 = pref[pend.b] + pend.hb * pend.ns;
            float* o_dst;
            float* l_dst;
            if (f % A.split == 0) {
                const size_t prow = ((size_t)(item0 + f / A.split) * NW + wu) * GH + hs;
                o_dst = A.ws_o + prow * D;
                l_dst = A.ws_lse + prow;
            } else {
                const size_t prow = ((size_t)blockIdx.x * NW + wu) * GH + hs;
                o_dst = A.ws_fix_o + prow * D;
                l_dst = A.ws_fix_lse + prow;
            }
#pragma unroll 1
            for (int q = 0; q < D / 32; ++q) {
                uint32_t o[32];
                tc_ld_32x32b_x32(lane_base + C::COL_O + pend.ob * D + q * 32, o);
                tc_wait_ld();
                if (pend.act) {
                    float4* dst = reinterpret_cast<float4*>(o_dst + q * 32);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                             __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
                }
            }
            if (pend.act) {
                *l_dst = pend.l > 0.f ? pend.m + __log2f(pend.l) : -INFINITY;
                const int s_hi = min(((pend.t_last + 1) * TT - 1) / A.split, pend.ns - 1);
                for (int sp = f / A.split + 1; sp <= s_hi; ++sp)
                    A.ws_lse[((size_t)(item0 + sp) * NW + wu) * GH + hs] = -INFINITY;
            }
            tc_fence_before();
            mbar_arrive(bar(B_OFREE + pend.ob));
            pend.on = false;
            return true;
        };

        uint32_t j = 0;
        bool ok = true;
        bool act = false;
        int gl = 0, t_first = 0;
        float m_used = -INFINITY, l_sum = 0.f;
        for (; c.x < c.x_end; tcur_next<TT>(c, tpref, A), ++j) {
            if (c.first) {
                const int u = c.hb * NW + wu;
                act = wu < NW && r < QB && u < A.U;
                gl = act ? u / A.HG - (c.hb * NW) / A.HG : 0;   // kv head inside the tile (row % NH)
                t_first = c.t;
                m_used = -INFINITY;
                l_sum = 0.f;
            }
            const int ob = c.run & 1;
            if (!mbar_wait(bar(B_SFULL), j & 1, abort_flag, A.err, kErrTimeoutMma)) { ok = false; break; }
            tc_fence_after();
            float s[TT];
            {
                uint32_t v[TR];
#pragma unroll
                for (int q = 0; q < TR / 32; ++q)
                    tc_ld_32x32b_x32(lane_base + C::COL_S + q * 32, *reinterpret_cast<uint32_t(*)[32]>(v + q * 32));
                tc_wait_ld();
                tc_fence_before();
                mbar_arrive(bar(B_SFREE));         // S is in registers: the next QK^T may run
#pragma unroll
                for (int t = 0; t < TT; ++t) s[t] = pick<NH>(v + t * NH, gl);
            }
            const int t0 = c.a + c.t * TT;
            const int v_lo = max(c.start - t0, 0);
            const int v_hi = min(c.end - t0, TT);
            float mx = -INFINITY;
#pragma unroll
            for (int t = 0; t < TT; ++t) {
                float x = s[t] * A.qscale;
                if (A.cap_log2 > 0.f) x = A.cap_log2 * tanh_abs_accurate(x);
                x = (act && t >= v_lo && t < v_hi) ? x : -INFINITY;
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
            // the P row: 128 f16 entries.  The row sum is taken over the rounded
            // values the PV product multiplies (a convex combination of V rows)
            uint32_t pw[64];
            float ls0 = 0.f, ls1 = 0.f;
            if constexpr (NH == 1) {
#pragma unroll
                for (int t = 0; t < TT; t += 2) {
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
                for (int t = 0; t < TT; ++t) {
                    const float p = ex2_approx(s[t] - m_off);
                    const uint32_t h = __half_as_ushort(__float2half_rn(p));
                    if (t & 1) ls1 = add_f16_lo(ls1, h); else ls0 = add_f16_lo(ls0, h);
                    const uint32_t word = act ? ((gl & 1) ? (h << 16) : h) : 0u;
#pragma unroll
                    for (int w = 0; w < NH / 2; ++w) pw[t * (NH / 2) + w] = (w == hp) ? word : 0u;
                }
            }
            l_sum += ls0 + ls1;
            if (rescale) {
                // O must not be in flight while it is rescaled
                if (!mbar_wait(bar(B_PVDONE + ((j - 1) & 1)), ((j - 1) >> 1) & 1, abort_flag, A.err, kErrTimeoutMma)) { ok = false; break; }
                tc_fence_after();
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
            // P buffer j & 1 was last read by PV_{j-2}
            if (j >= 2 && !mbar_wait(bar(B_PVDONE + (j & 1)), ((j - 2) >> 1) & 1, abort_flag, A.err, kErrTimeoutMma)) { ok = false; break; }
            tc_st_32x32b_x32(lane_base + C::COL_P + (j & 1) * 64, *reinterpret_cast<const uint32_t(*)[32]>(pw));
            tc_st_32x32b_x32(lane_base + C::COL_P + (j & 1) * 64 + 32, *reinterpret_cast<const uint32_t(*)[32]>(pw + 32));
            if (v_lo > 0 || v_hi < TT) {
                // zero the V rows of masked tokens (all NH heads, every chunk), once
                // the tile's copy has landed
                if (!mbar_wait(bar(B_VFULL + (j % NV)), (j / NV) & 1, abort_flag, A.err, kErrTimeoutLoad)) { ok = false; break; }
                uint8_t* vt = smem + C::OFF_VRING + (j % NV) * C::KV_BYTES;
                const int lo_end = v_lo * NH * 128, hi_beg = v_hi * NH * 128;
#pragma unroll 1
                for (int ch = 0; ch < NCH; ++ch) {
                    uint8_t* cb = vt + ch * C::CHUNK;
                    for (int o = lane * 16; o < lo_end; o += 32 * 16) *reinterpret_cast<uint4*>(cb + o) = make_uint4(0u, 0u, 0u, 0u);
                    for (int o = hi_beg + lane * 16; o < (int)C::CHUNK; o += 32 * 16)
                        *reinterpret_cast<uint4*>(cb + o) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            tc_wait_st();
            tc_fence_before();
            mbar_arrive(bar(B_PFULL + (j & 1)));
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
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace tcdec
