// draft_pos.cu - spec_draft_block for batches larger than one fixed-point launch: the
// chain walked position by position on the tcgen05 tensor cores.
//
// Defines: "Speculative Decoding Part 2" (VESSL AI), DSpark section, bias equation
// z_j = l_j + W_1[x_{j-1}] W_2, with x_j the argmax (T=0) or the inverse-CDF draw
// (T=1) of softmax(z_j); the "SpecOPD" summary, "how it works": many anchors of many
// references drafted at once.  The results are spec_draft_block's (draft_common.cuh).
//
// The fixed-point kernel keeps every row's A operand in shared memory, so one launch
// takes at most 256 rows, and each of its passes reads the drafter rows again.  For a
// large batch this path walks the positions in order instead: position j needs only
// x_{j-1}, so each position reads its drafter rows once and the weights once for every
// request.  Per position, two kernels:
//   draft_pos_tiles_kernel  one CTA per SM over a contiguous range of 256-entry tiles,
//     18 warps:
//     warp 0   TMA producer: the tile's Wt rows as r/64 boxes [256 entries x 64 k]
//              (128-byte swizzle) into a ring of 32 KB stages, resident while every
//              M tile of 128 requests passes; per (tile, M tile) the M tile's gathered
//              U rows (the A operand, r/64 boxes [128 requests x 64 k]) into a ring of
//              16 KB stages (and, for logits rows not 32-byte aligned, an L2 prefetch of
//              its drafter logits over the tile);
//     warp 1   tcgen05.mma (M = 128 requests, N = 256 entries, K = 16, bf16 in, f32
//              accumulate) into two 256-column TMEM accumulators, one per epilogue group;
//     warps 2-17  epilogue, two groups of 8 warps; group g takes the M tiles mt = g
//              (mod 2); warp w of a group reads TMEM lane quadrant w % 4 and one 128-entry
//              half of the tile.  A thread owns one request's row: it loads the
//              logits two 32-entry chunks ahead (a 32-byte sector per load when the
//              rows are 32-byte aligned), adds them,
//              folds the half-tile's 128 biased logits into the row's record for that
//              128-entry tile, and into its running record over the CTA's tiles.
//   draft_pos_draw_kernel   a CTA of 4 warps per request merges the records and takes
//     x_j: the argmax, or the T=1 draw (the CTA range, then the 128-entry tile, then
//     that tile's biased logits recomputed on CUDA cores and scanned), writes the
//     outputs and U[x_j], the next position's A row.
#include "draft_common.cuh"
#include "tc_common.cuh"

namespace spec {

constexpr int kPosK = 64;                        // k per 128-byte swizzle block
constexpr int kPosN = 256;                       // vocabulary entries per tile (MMA N)
constexpr int kPosWBlock = kPosN * kPosK * 2;    // 32 KB: one Wt box [256 entries x 64 k]
constexpr int kPosABlock = 128 * kPosK * 2;      // 16 KB: one U box [128 requests x 64 k]
constexpr int kPosWStages = 5;                   // a whole tile (r/64 <= 4 boxes) and one more
constexpr int kPosAStages = 3;
constexpr int kPosEpi = 16;                      // epilogue warps: two groups of 8
constexpr int kPosThreads = 32 * (2 + kPosEpi);
constexpr int kPosMaxB = 1024;                   // requests per launch: 8 M tiles, 4 per group
constexpr int kPosMaxMT = kPosMaxB / 128 / 2;    // running records per epilogue thread
constexpr int kPosMaxCtas = 256;
constexpr uint32_t kPosIdesc = idesc_bf16_f32(128, kPosN);
constexpr uint32_t kPosTmemCols = 2 * kPosN;     // two 256-column accumulators
static_assert(kPosN == 2 * kDraftTile, "a tile is two record tiles");

// What the position kernels need beyond DraftParams (whose tile_rec / cta_rec point at
// this path's records: tile_rec [B][n_tiles], cta_rec [B][nC][2], one per tile half).
struct PosExtra {
    int j;               // position of this launch (1-based)
    int nC;              // CTAs of the tiles kernel
    int n_t2;            // 256-entry tiles
    int32_t* xprev;      // [B] x_{j-1} (-1: the request has ended)
    bf16_t* ug;          // [B][r] U[x_{j-1}] (zero rows for ended requests)
};

// 256-entry tiles [pos_t2_begin(c), pos_t2_begin(c + 1)) belong to CTA c.
__device__ __forceinline__ int pos_t2_begin(int c, int nC, int n_t2) { return (int)(((long)c * n_t2) / nC); }

__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" :: "l"(map), "r"(x), "r"(y)
                 : "memory");
}

// L32: the logits rows are 32-byte aligned (loaded a sector at a time)
template <int TT, bool L32>
__global__ void __launch_bounds__(kPosThreads, 1)
    draft_pos_tiles_kernel(const __grid_constant__ DraftParams p, const __grid_constant__ PosExtra e,
                           const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap umap,
                           const __grid_constant__ CUtensorMap lmap) {
    extern __shared__ uint8_t pos_raw[];
    uint8_t* base = pos_raw + ((1024u - (smem_u32(pos_raw) & 1023u)) & 1023u);
    uint8_t* s_w = base;                                          // [kPosWStages][32 KB]
    uint8_t* s_a = s_w + (size_t)kPosWStages * kPosWBlock;         // [kPosAStages][16 KB]
    __shared__ __align__(8) uint64_t s_wfull[kPosWStages], s_wempty[kPosWStages];
    __shared__ __align__(8) uint64_t s_afull[kPosAStages], s_aempty[kPosAStages];
    __shared__ __align__(8) uint64_t s_tfull[2], s_tempty[2], s_drain;
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const int KB = p.r / kPosK;
    const int nM = (p.B + 127) / 128;
    const int tb = pos_t2_begin(c, e.nC, e.n_t2), te = pos_t2_begin(c + 1, e.nC, e.n_t2);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPosWStages; ++s) { mbar_init(&s_wfull[s], 1); mbar_init(&s_wempty[s], 1); }
        for (int s = 0; s < kPosAStages; ++s) { mbar_init(&s_afull[s], 1); mbar_init(&s_aempty[s], 1); }
        for (int s = 0; s < 2; ++s) { mbar_init(&s_tfull[s], 1); mbar_init(&s_tempty[s], kPosEpi / 2); }
        mbar_init(&s_drain, 1);
        s_fail = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&s_tmem, kPosTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    uint32_t iw = 0, ia = 0;   // producer: Wt stages and U stages issued

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();   // Wt is streamed once per position
            // the first tile's weights depend on nothing: requested before the wait for
            // the previous position's draw, which writes the U rows
            for (int kb = 0; kb < KB; ++kb) {
                mbar_arrive_expect_tx(&s_wfull[kb], kPosWBlock);
                tma_load_2d_hint(s_w + (size_t)kb * kPosWBlock, &wmap, kb * kPosK, tb * kPosN, &s_wfull[kb], pol);
            }
            iw = (uint32_t)KB;
            pdl_wait_primary();
            bool ok = true;
            for (int T = tb; T < te && ok; ++T) {
                if (T > tb)
                    for (int kb = 0; kb < KB && ok; ++kb) {
                        const uint32_t s = iw % kPosWStages, ph = (iw / kPosWStages) & 1u;
                        ok = mbar_wait(&s_wempty[s], ph ^ 1u, p.status, kWaitLimitNs);
                        if (!ok) break;
                        mbar_arrive_expect_tx(&s_wfull[s], kPosWBlock);
                        tma_load_2d_hint(s_w + (size_t)s * kPosWBlock, &wmap, kb * kPosK, T * kPosN, &s_wfull[s], pol);
                        ++iw;
                    }
                for (int mt = 0; mt < nM && ok; ++mt) {
                    // with 16-byte loads the epilogue reads this M tile's logits over the
                    // tile from L2; its 32-byte loads ran faster without the prefetch
                    if constexpr (!L32) {
                        tma_prefetch_2d(&lmap, T * kPosN, mt * 128);
                        tma_prefetch_2d(&lmap, T * kPosN + 128, mt * 128);
                    }
                    for (int kb = 0; kb < KB && ok; ++kb) {
                        const uint32_t s = ia % kPosAStages, ph = (ia / kPosAStages) & 1u;
                        ok = mbar_wait(&s_aempty[s], ph ^ 1u, p.status, kWaitLimitNs);
                        if (!ok) break;
                        mbar_arrive_expect_tx(&s_afull[s], kPosABlock);
                        tma_load_2d(s_a + (size_t)s * kPosABlock, &umap, kb * kPosK, mt * 128, &s_afull[s]);
                        ++ia;
                    }
                }
            }
            if (!ok) s_fail = 1;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t mw = 0, ma = 0, jt[2] = {0u, 0u};
            bool ok = true;
            for (int T = tb; T < te && ok && !*(volatile int*)&s_fail; ++T) {
                for (int mt = 0; mt < nM && ok; ++mt) {
                    const int buf = mt & 1;
                    ok = mbar_wait(&s_tempty[buf], (jt[buf] & 1u) ^ 1u, p.status, kWaitLimitNs);
                    if (!ok) break;
                    tc_fence_after();
                    for (int kb = 0; kb < KB && ok; ++kb) {
                        const uint32_t ws = (mw + kb) % kPosWStages;
                        if (mt == 0) {
                            ok = mbar_wait(&s_wfull[ws], ((mw + kb) / kPosWStages) & 1u, p.status, kWaitLimitNs);
                            if (!ok) break;
                        }
                        const uint32_t as = ma % kPosAStages;
                        ok = mbar_wait(&s_afull[as], (ma / kPosAStages) & 1u, p.status, kWaitLimitNs);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t a0 = smem_u32(s_a + (size_t)as * kPosABlock);
                        const uint32_t w0 = smem_u32(s_w + (size_t)ws * kPosWBlock);
#pragma unroll
                        for (int kk = 0; kk < kPosK / 16; ++kk)
                            umma_f16(tmem + buf * kPosN, sw128_desc(a0 + kk * 32), sw128_desc(w0 + kk * 32), kPosIdesc,
                                     (kb | kk) != 0 ? 1u : 0u);
                        umma_commit(&s_aempty[as]);
                        ++ma;
                    }
                    if (!ok) break;
                    umma_commit(&s_tfull[buf]);
                    ++jt[buf];
                }
                if (!ok) break;
                // the tile's weight stages are free once every M tile's MMAs complete
                for (int kb = 0; kb < KB; ++kb) umma_commit(&s_wempty[(mw + kb) % kPosWStages]);
                mw += (uint32_t)KB;
            }
            if (!ok) s_fail = 1;
        }
    } else {
        const int ew = warp - 2;          // epilogue warp 0..15
        const int g = ew >> 3;            // its group: M tiles mt = g (mod 2), TMEM buffer g
        const int q = warp & 3;           // its TMEM lane quadrant: requests 32 q .. +31 of an M tile
        const int h = (ew >> 2) & 1;      // its half of a tile: entries 128 h .. +127
        const bf16_t* L = static_cast<const bf16_t*>(p.logits);
        pdl_wait_primary();               // x_{j-1}; the previous draw's reads of the records
        RowAcc run[kPosMaxMT];            // per M tile of the group: the row's record over the CTA's tiles
        unsigned live = 0u;
#pragma unroll
        for (int i = 0; i < kPosMaxMT; ++i) {
            run[i] = rowacc_empty();
            const int row = (g + 2 * i) * 128 + 32 * q + lane;
            if (g + 2 * i < nM && row < p.B && __ldcg(&e.xprev[row]) >= 0) live |= 1u << i;
        }
        uint32_t k = 0;                   // the group's tiles consumed
        bool ok = true;
        uint4 w0[LWords<bf16_t>::N], w1[LWords<bf16_t>::N];
        auto pair_row = [&](int i) { return (g + 2 * i) * 128 + 32 * q + lane; };
        auto pair_lrow = [&](int i) {
            const int row = pair_row(i);
            return L + ((size_t)(row < p.B ? row : 0) * p.gamma + (e.j - 1)) * p.V;
        };
        // the first pair's first two chunks
        if (tb < te && ((live & 1u) != 0u) && 2 * tb + h < p.n_tiles) {
            load_l32<bf16_t, L32>(pair_lrow(0), (long)(2 * tb + h) * kDraftTile, p.V, w0);
            load_l32<bf16_t, L32>(pair_lrow(0), (long)(2 * tb + h) * kDraftTile + 32, p.V, w1);
        }
        for (int T = tb; T < te && ok; ++T) {
            const int t = 2 * T + h;      // the 128-entry tile of this half
            const long v0 = (long)t * kDraftTile;
#pragma unroll
            for (int i = 0; i < kPosMaxMT; ++i) {
                const int mt = g + 2 * i;
                if (mt >= nM) break;      // warp-uniform
                const int row = pair_row(i);
                const bool lv = ((live >> i) & 1u) && t < p.n_tiles;
                const bf16_t* lrow = pair_lrow(i);
                // the group's next pair: (T, mt + 2), else (T + 1, g)
                const bool nxt_same = g + 2 * (i + 1) < nM && i + 1 < kPosMaxMT;
                const int ni = nxt_same ? i + 1 : 0;
                const int nT = nxt_same ? T : T + 1;
                const bool nlv = nT < te && ((live >> ni) & 1u) && 2 * nT + h < p.n_tiles;
                const bf16_t* nlrow = pair_lrow(ni);
                const long nv0 = (long)(2 * nT + h) * kDraftTile;
                ok = __all_sync(0xffffffffu, mbar_wait(&s_tfull[g], k & 1u, p.status, kWaitLimitNs));
                if (!ok) break;
                tc_fence_after();
                const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(g * kPosN + h * kDraftTile);
                RowAcc rec = rowacc_empty();
                float z[32];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    tmem_ld32(ta + 32 * ch, z);
                    if (lv) {
                        if (ch & 1) add_l32<bf16_t>(w1, z);
                        else add_l32<bf16_t>(w0, z);
                        if (ch == 0) load_l32<bf16_t, L32>(lrow, v0 + 64, p.V, w0);
                        if (ch == 1) load_l32<bf16_t, L32>(lrow, v0 + 96, p.V, w1);
                    }
                    if (ch == 2 && nlv) load_l32<bf16_t, L32>(nlrow, nv0, p.V, w0);
                    if (ch == 3 && nlv) load_l32<bf16_t, L32>(nlrow, nv0 + 32, p.V, w1);
                    if (lv) {
                        const float run_mx = fmaxf(run[i].mx, rec.mx);
                        rec = rowacc_merge(rec, record32(z, (int)(v0 + 32 * ch), run_mx, TT == 0));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive1(&s_tempty[g]);
                ++k;
                if (lv) {
                    if (TT == 1) p.tile_rec[(size_t)row * p.n_tiles + t] = rowacc_pack(rec);
                    run[i] = rowacc_merge(run[i], rec);
                }
            }
        }
        if (!ok) {
            s_fail = 1;
        } else {
            // one record per (request, CTA, tile half)
#pragma unroll
            for (int i = 0; i < kPosMaxMT; ++i) {
                const int row = (g + 2 * i) * 128 + 32 * q + lane;
                if (g + 2 * i < nM && row < p.B) p.cta_rec[((size_t)row * e.nC + c) * 2 + h] = rowacc_pack(run[i]);
            }
        }
    }

    // every MMA has completed before TMEM is released, and no copy still writes this
    // CTA's shared memory when it exits (stages requested and never consumed, after an
    // error)
    __syncthreads();
    if (threadIdx.x == 32) {
        umma_commit(&s_drain);
        mbar_wait(&s_drain, 0u, p.status, kWaitLimitNs);
    }
    if (threadIdx.x == 0) {
        const uint32_t nw = iw < (uint32_t)kPosWStages ? iw : (uint32_t)kPosWStages;
        for (uint32_t i = iw - nw; i < iw; ++i)
            mbar_wait(&s_wfull[i % kPosWStages], (i / kPosWStages) & 1u, p.status, kWaitLimitNs);
        const uint32_t na = ia < (uint32_t)kPosAStages ? ia : (uint32_t)kPosAStages;
        for (uint32_t i = ia - na; i < ia; ++i)
            mbar_wait(&s_afull[i % kPosAStages], (i / kPosAStages) & 1u, p.status, kWaitLimitNs);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kPosTmemCols);
    }
}

// x_0 and its U row for position 1: one warp per request.
__global__ void draft_pos_gather_kernel(const __grid_constant__ DraftParams p, const __grid_constant__ PosExtra e) {
    const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (b >= p.B) return;
    const int a = p.anchor[b];
    const bool ok = a >= 0 && a < p.V;
    if (lane == 0) e.xprev[b] = ok ? a : -1;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const bf16_t*>(p.U) + (size_t)(ok ? a : 0) * p.r);
    uint4* dst = reinterpret_cast<uint4*>(e.ug + (size_t)b * p.r);
    for (int w = lane; w < p.r / 8; w += 32) dst[w] = ok ? __ldg(src + w) : make_uint4(0u, 0u, 0u, 0u);
}

// One CTA of 4 warps per request: x_j and its outputs; x_j and U[x_j] for the next
// position.  128-thread CTAs let 8 or more fit on an SM, so a batch of 1024 requests runs
// in one wave.  One wave of loads brings CTA c's two half records to thread c % 128 (two
// CTAs per thread); a block merge gives the row's maximum and sum.  At T=1 a block scan of
// the CTAs' weights (in index order, the first 128 CTAs then the rest) finds the CTA
// range where the CDF crosses u * Z; every warp then finds the 128-entry tile within that
// range from the tile records (the same loads, so the same decision), computes 32 of its
// biased logits on CUDA cores (lane l takes the rank slice [8l, 8l + 8) of each entry),
// and warp 0 scans them.
constexpr int kPosDrawWarps = 4;
constexpr int kPosDrawThreads = 32 * kPosDrawWarps;
static_assert(kPosMaxCtas <= 2 * kPosDrawThreads, "two CTA record pairs per thread");

template <int TT>
__global__ void __launch_bounds__(kPosDrawThreads, 8)
    draft_pos_draw_kernel(const __grid_constant__ DraftParams p, const __grid_constant__ PosExtra e) {
    constexpr int EPW = kDraftTile / kPosDrawWarps;   // entries of the tile per warp
    __shared__ float s_z[kDraftTile];
    __shared__ float4 s_red[kPosDrawWarps];
    __shared__ float s_wsum[kPosDrawWarps];
    __shared__ int s_first, s_last, s_x;
    __shared__ float s_tl;
    pdl_launch_dependents();   // the next position's tiles kernel may request its weights
    const int b = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t out = (size_t)b * p.gamma + (e.j - 1);
    const int xp = __ldcg(&e.xprev[b]);
    const bf16_t* U = static_cast<const bf16_t*>(p.U);
    const bf16_t* Wt = static_cast<const bf16_t*>(p.Wt);
    auto finish = [&](int x, float conf, float qx, unsigned flag) {   // thread 0
        p.tokens_out[out] = x;
        p.conf_out[out] = conf;
        if (p.qtok_out) p.qtok_out[out] = qx;
        e.xprev[b] = x;
        if (flag) atomicOr(p.status, flag);
        if (e.j == p.gamma && b == 0 && p.passes_out) atomicMax(p.passes_out, p.gamma);
    };
    if (xp < 0) {   // the anchor is out of range (position 1), or the request ended earlier
        if (tid == 0) finish(-1, NAN, NAN, e.j == 1 ? SPEC_DEV_TOKEN : 0u);
        return;
    }
    // one wave of loads: CTAs tid and tid + 128's two half records, the U row of x_{j-1}
    const float4* recs = p.cta_rec + (size_t)b * e.nC * 2;
    const int ca = tid, cb = tid + kPosDrawThreads;
    RowAcc ra0 = rowacc_empty(), ra1 = rowacc_empty(), rb0 = rowacc_empty(), rb1 = rowacc_empty();
    if (ca < e.nC) {
        ra0 = rowacc_unpack(__ldcg(&recs[2 * ca]));
        ra1 = rowacc_unpack(__ldcg(&recs[2 * ca + 1]));
    }
    if (cb < e.nC) {
        rb0 = rowacc_unpack(__ldcg(&recs[2 * cb]));
        rb1 = rowacc_unpack(__ldcg(&recs[2 * cb + 1]));
    }
    const bool has = lane < (p.r >> 3);
    uint4 uw = make_uint4(0u, 0u, 0u, 0u);
    if (TT == 1 && has) uw = __ldg(reinterpret_cast<const uint4*>(U + (size_t)xp * p.r) + lane);
    const float u = TT == 1 ? philox_uniform(p.seeds[b], (uint64_t)(p.b_base + b), (uint64_t)e.j, 0) : 0.0f;
    // the row's record
    {
        const RowAcc w = warp_rowacc(rowacc_merge(rowacc_merge(ra0, ra1), rowacc_merge(rb0, rb1)));
        if (lane == 0) s_red[warp] = rowacc_pack(w);
    }
    if (tid == 0) { s_first = e.nC; s_last = -1; }
    __syncthreads();
    RowAcc acc = rowacc_empty();
#pragma unroll
    for (int w = 0; w < kPosDrawWarps; ++w) acc = rowacc_merge(acc, rowacc_unpack(s_red[w]));
    if (acc.bad || acc.mx == -INFINITY) {   // no distribution: the request ends here
        if (tid == 0) finish(-1, NAN, NAN, SPEC_DEV_NONFINITE);
        return;
    }
    const float M2 = acc.mx * kLog2e;
    const float S = acc.s;
    const float conf = ex2(fmaf(acc.mx, kLog2e, -M2)) / S;
    int x = acc.idx;
    float qx = conf;
    if constexpr (TT == 1) {
        const float thr = u * S;
        auto weight = [&](const RowAcc& r) { return r.mx == -INFINITY ? 0.0f : r.s * ex2(r.mx * kLog2e - M2); };
        // level 1: the CTA ranges' weights in index order, a block scan over the first 128
        // CTAs, then over the rest on top of their total
        const float wa = ca < e.nC ? weight(ra0) + weight(ra1) : 0.0f;
        const float wb = cb < e.nC ? weight(rb0) + weight(rb1) : 0.0f;
        float ia = warp_inclusive_scan(wa), ib = warp_inclusive_scan(wb);
        if (lane == 31) s_wsum[warp] = ia;
        __syncthreads();
        float tot_a = 0.0f;
#pragma unroll
        for (int w2 = 0; w2 < kPosDrawWarps; ++w2) {
            const float v = s_wsum[w2];
            if (w2 < warp) ia += v;
            tot_a += v;
        }
        __syncthreads();   // s_wsum is rewritten
        if (lane == 31) s_wsum[warp] = ib;
        __syncthreads();
        ib += tot_a;
        for (int w2 = 0; w2 < warp; ++w2) ib += s_wsum[w2];
        if (ca < e.nC && ia > thr) atomicMin(&s_first, ca);
        if (cb < e.nC && ib > thr) atomicMin(&s_first, cb);
        if (ca < e.nC && wa > 0.0f) atomicMax(&s_last, ca);
        if (cb < e.nC && wb > 0.0f) atomicMax(&s_last, cb);
        __syncthreads();
        const int first = s_first;
        if (ca == first) s_tl = thr - (ia - wa);
        if (cb == first) s_tl = thr - (ib - wb);
        __syncthreads();
        const bool crossed = first < e.nC;
        const int cta = crossed ? first : max(0, s_last);
        float tl = crossed ? s_tl : INFINITY;
        // level 2: the CTA's 128-entry tiles (every warp alike)
        const int tb = 2 * pos_t2_begin(cta, e.nC, e.n_t2);
        const int te = min(2 * pos_t2_begin(cta + 1, e.nC, e.n_t2), p.n_tiles);
        int tile = -1, last_tile = te - 1;
        float carry = 0.0f;
        for (int t0 = tb; t0 < te && tile < 0; t0 += 32) {
            const int t = t0 + lane;
            const float wt = t < te ? weight(rowacc_unpack(__ldcg(&p.tile_rec[(size_t)b * p.n_tiles + t]))) : 0.0f;
            const float inc = warp_inclusive_scan(wt) + carry;
            const unsigned hit = __ballot_sync(0xffffffffu, t < te && inc > tl);
            if (hit) {
                const int Lt = __ffs(hit) - 1;
                tile = t0 + Lt;
                tl -= __shfl_sync(0xffffffffu, inc - wt, Lt);
            }
            const unsigned pos = __ballot_sync(0xffffffffu, t < te && wt > 0.0f);
            if (pos) last_tile = t0 + 31 - __clz(pos);
            carry = __shfl_sync(0xffffffffu, inc, 31);
        }
        if (tile < 0) { tile = last_tile; tl = INFINITY; }
        tile = max(0, min(tile, p.n_tiles - 1));
        // level 3: this warp's EPW biased logits of the tile: its Wt rows (contiguous)
        // requested into L2 at once, then taken kZBatch at a time
        float uu[8];
        {
            const uint32_t a[4] = {uw.x, uw.y, uw.z, uw.w};
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {
                uu[2 * k2] = __uint_as_float(a[k2] << 16);
                uu[2 * k2 + 1] = __uint_as_float(a[k2] & 0xffff0000u);
            }
        }
        const bf16_t* lrow = static_cast<const bf16_t*>(p.logits) + out * p.V;
        const long e0 = (long)tile * kDraftTile + warp * EPW;
        const long e1 = e0 + EPW < p.V ? e0 + EPW : p.V;
        if (lane == 0 && e1 > e0) bulk_prefetch_l2(Wt + (size_t)e0 * p.r, (unsigned)((e1 - e0) * p.r * 2));
        const float zl = (lane < EPW && e0 + lane < p.V) ? load_one(lrow + e0 + lane) : 0.0f;
#pragma unroll 1
        for (int hb = 0; hb < EPW / kZBatch; ++hb) {
            uint4 wr[kZBatch];
#pragma unroll
            for (int qq = 0; qq < kZBatch; ++qq) {
                const long v = e0 + hb * kZBatch + qq;
                wr[qq] = make_uint4(0u, 0u, 0u, 0u);
                if (has && v < p.V) wr[qq] = __ldg(reinterpret_cast<const uint4*>(Wt + (size_t)v * p.r) + lane);
            }
#pragma unroll
            for (int qq = 0; qq < kZBatch; ++qq) {
                const uint32_t a[4] = {wr[qq].x, wr[qq].y, wr[qq].z, wr[qq].w};
                float part = 0.0f;
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2) {
                    part = fmaf(uu[2 * k2], __uint_as_float(a[k2] << 16), part);
                    part = fmaf(uu[2 * k2 + 1], __uint_as_float(a[k2] & 0xffff0000u), part);
                }
                part = warp_sum(part);
                const int qi = hb * kZBatch + qq;
                const float zq = __shfl_sync(0xffffffffu, zl, qi);
                if (lane == 0) s_z[warp * EPW + qi] = e0 + qi < p.V ? zq + part : -INFINITY;
            }
        }
        __syncthreads();
        if (warp == 0) {
            float z[4];
            long v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[i] = (long)tile * kDraftTile + 32 * i + lane;
                z[i] = v[i] < p.V ? s_z[32 * i + lane] : -INFINITY;
            }
            int found = -1;
            float zf = 0.0f;
            draw_scan_tile(z, v, p.V, M2, tl, tile, found, zf);
            x = found;
            qx = wexp(zf, M2) / S;
            if (lane == 0) s_x = x;
        }
        __syncthreads();
        x = s_x;
    }
    if (tid == 0) finish(x, conf, qx, x < 0 ? SPEC_DEV_NONFINITE : 0u);
    // the next position's A row
    if (warp == 0 && e.j < p.gamma) {
        const uint4* src = reinterpret_cast<const uint4*>(U + (size_t)(x >= 0 ? x : 0) * p.r);
        uint4* dst = reinterpret_cast<uint4*>(e.ug + (size_t)b * p.r);
        for (int w = lane; w < p.r / 8; w += 32) dst[w] = x >= 0 ? __ldg(src + w) : make_uint4(0u, 0u, 0u, 0u);
    }
}

// ----------------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------------
static size_t pos_align(size_t x) { return (x + 255) / 256 * 256; }

// [header | tile records | CTA records | x_{j-1} | U rows] for a slice of requests.
size_t draft_pos_workspace_bytes(int B, int V, int r) {
    const size_t S = (size_t)(B < kPosMaxB ? B : kPosMaxB);
    const size_t n_tiles = ((size_t)V + kDraftTile - 1) / kDraftTile;
    size_t off = kWsHeaderBytes;
    off = pos_align(off + sizeof(float4) * S * n_tiles);
    off = pos_align(off + sizeof(float4) * S * kPosMaxCtas * 2);
    off = pos_align(off + sizeof(int32_t) * S);
    off = pos_align(off + sizeof(bf16_t) * S * (size_t)r);
    return off;
}

bool draft_pos_supported(const DraftParams& p) {
    return (long)p.B * p.gamma > 256 && p.ldt == SPEC_BF16 && p.wdt == SPEC_BF16 && p.r >= kPosK && p.r <= 256 &&
           p.r % kPosK == 0 && p.V % 8 == 0 && p.qlogits_out == nullptr && encode_tiled() != nullptr;
}

template <int TT>
static cudaError_t pos_launch_slice(const DraftParams& q, PosExtra e, cudaStream_t stream) {
    const int KB = q.r / kPosK;
    (void)KB;
    const size_t smem = 1024 + (size_t)kPosWStages * kPosWBlock + (size_t)kPosAStages * kPosABlock;
    // 32-byte loads of the logits when every row of every position starts on 32 bytes
    const bool l32 = (reinterpret_cast<uintptr_t>(q.logits) & 31u) == 0 && ((size_t)q.V * 2) % 32 == 0;
    auto tiles = l32 ? draft_pos_tiles_kernel<TT, true> : draft_pos_tiles_kernel<TT, false>;
    cudaError_t err = cudaFuncSetAttribute(tiles, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    CUtensorMap wmap, umap;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)q.r, (cuuint64_t)q.V};
        const cuuint64_t strides[1] = {(cuuint64_t)q.r * 2};
        const cuuint32_t box[2] = {(cuuint32_t)kPosK, (cuuint32_t)kPosN};
        const cuuint32_t estr[2] = {1, 1};
        if (encode_tiled()(&wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q.Wt), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)q.r, (cuuint64_t)q.B};
        const cuuint64_t strides[1] = {(cuuint64_t)q.r * 2};
        const cuuint32_t box[2] = {(cuuint32_t)kPosK, 128u};
        const cuuint32_t estr[2] = {1, 1};
        if (encode_tiled()(&umap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, e.ug, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    draft_pos_gather_kernel<<<(q.B + 7) / 8, 256, 0, stream>>>(q, e);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    for (int j = 1; j <= q.gamma; ++j) {
        e.j = j;
        // the logits of position j, [B rows][V] with a row stride of gamma * V entries, for
        // the L2 prefetches ([128 requests x 128 entries] boxes)
        CUtensorMap lmap;
        const cuuint64_t dims[2] = {(cuuint64_t)q.V, (cuuint64_t)q.B};
        const cuuint64_t strides[1] = {(cuuint64_t)q.gamma * q.V * 2};
        const cuuint32_t box[2] = {128u, 128u};
        const cuuint32_t estr[2] = {1, 1};
        void* lbase = const_cast<bf16_t*>(static_cast<const bf16_t*>(q.logits) + (size_t)(j - 1) * q.V);
        if (encode_tiled()(&lmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lbase, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        // the tiles kernel as a programmatic dependent of the previous draw: its first
        // weights are requested before it waits for the U rows
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)e.nC);
        cfg.blockDim = dim3(kPosThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        err = cudaLaunchKernelEx(&cfg, tiles, q, e, wmap, umap, lmap);
        if (err != cudaSuccess) return err;
        draft_pos_draw_kernel<TT><<<q.B, kPosDrawThreads, 0, stream>>>(q, e);
        err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

// The batch in slices of at most kPosMaxB requests (the Philox request index stays the
// request's index in the whole batch), each slice's records in the same workspace.
cudaError_t draft_pos_launch(const DraftParams& p, void* ws, cudaStream_t stream) {
    char* w = static_cast<char*>(ws);
    DraftParams q = p;
    q.status = &reinterpret_cast<WsHeader*>(w)->status;
    q.n_tiles = (int)(((size_t)p.V + kDraftTile - 1) / kDraftTile);
    const size_t S = (size_t)(p.B < kPosMaxB ? p.B : kPosMaxB);
    size_t off = kWsHeaderBytes;
    q.tile_rec = reinterpret_cast<float4*>(w + off);
    off = pos_align(off + sizeof(float4) * S * q.n_tiles);
    q.cta_rec = reinterpret_cast<float4*>(w + off);
    off = pos_align(off + sizeof(float4) * S * kPosMaxCtas * 2);
    PosExtra e;
    e.xprev = reinterpret_cast<int32_t*>(w + off);
    off = pos_align(off + sizeof(int32_t) * S);
    e.ug = reinterpret_cast<bf16_t*>(w + off);
    e.n_t2 = (p.V + kPosN - 1) / kPosN;
    int nC = device_sm_count();   // one CTA per SM (TMEM and shared memory sized for it)
    if (nC > kPosMaxCtas) nC = kPosMaxCtas;
    if (nC > e.n_t2) nC = e.n_t2;
    e.nC = nC;
    e.j = 0;
    if (p.passes_out) {
        const cudaError_t err = cudaMemsetAsync(p.passes_out, 0, sizeof(int32_t), stream);
        if (err != cudaSuccess) return err;
    }
    const size_t lsize = 2;
    for (int b0 = 0; b0 < p.B; b0 += kPosMaxB) {
        const size_t rows = (size_t)b0 * p.gamma;
        q.B = p.B - b0 < kPosMaxB ? p.B - b0 : kPosMaxB;
        q.b_base = p.b_base + b0;
        q.logits = static_cast<const char*>(p.logits) + rows * p.V * lsize;
        q.anchor = p.anchor + b0;
        q.seeds = p.seeds ? p.seeds + b0 : nullptr;
        q.tokens_out = p.tokens_out + rows;
        q.conf_out = p.conf_out + rows;
        q.qtok_out = p.qtok_out ? p.qtok_out + rows : nullptr;
        const cudaError_t err = p.temperature == 0 ? pos_launch_slice<0>(q, e, stream) : pos_launch_slice<1>(q, e, stream);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace spec
