// draft_tc.cu - DSpark block draft, Markov bias on the tcgen05 tensor cores.
//
// Defines: "Speculative Decoding Part 2" (VESSL AI), DSpark section, bias equation
// B(x_{k-1}, .) = W_1[x_{k-1}] W_2; the fixed-point pass loop, finalize and chain
// semantics are those of draft_common.cuh (shared with the CUDA-core kernel).
//
// One biased pass computes, for every row n = (request, position) and every vocabulary
// entry v, z[n, v] = l[n, v] + sum_k U[x_prev(n), k] Wt[v, k]: a GEMM with M = rows
// (B*gamma <= 256, padded to 128 or 256), N = V, K = r.  W is the big operand (r*V
// bf16, 127 MB at r = 256, V = 248,320) and is read once per pass; the rows are few,
// so the tensor cores only keep the contraction off the critical path of the stream.
//
// Per CTA (one per SM, persistent, contiguous tile range), 18 warps:
//   warp 0      TMA producer: Wt tiles [128 entries x 64 k] (128-byte swizzle) into a
//               ring of 16 KB stages, completion counted on mbarriers;
//   warp 1      allocates TMEM and issues tcgen05.mma (M=128, N=128, K=16, bf16 in,
//               f32 accumulate) from one thread, committing to the ring's "empty"
//               barriers and, per tile, to a "TMEM full" barrier; two TMEM buffers;
//   warps 2-17  epilogue.  Warp w may read TMEM lanes 32*(w%4)..+31 only, so the 16
//               warps form four groups per lane quadrant, each group splitting the
//               tile's 128 columns (32 columns per warp with one 128-row M tile, 64
//               with two).  A thread owns one row: it pulls its columns with
//               tcgen05.ld, adds the drafter logits (fetched one tile ahead) and folds
//               max / sum-exp / argmax into its row's running record; the column
//               slices are merged through shared memory.  Rows are laid out
//               round-robin over the lane quadrants so a handful of rows still keeps
//               every group busy.
// The A operand (the gathered rows U[x_prev(n)]) is written to shared memory in the
// same K-major 128-byte-swizzled layout once per pass.  Pass 0 (no bias yet) and the
// finalize run on CUDA cores with every warp.
#include "draft_common.cuh"
#include "tc_common.cuh"

namespace spec {

constexpr int kTcN = 128;                    // vocabulary entries per tile (MMA N)
constexpr int kTcK = 64;                     // k per 128-byte swizzle block
constexpr int kTcBlock = 128 * kTcK * 2;     // 16 KB: 128 rows x 64 k of bf16
static_assert(kTcN == kDraftTile, "tile width shared with the CUDA-core phases");

constexpr uint32_t kTcIdesc = idesc_bf16_f32(128, kTcN);

__device__ __forceinline__ void umma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t accumulate) {
    umma_f16(d, a, b, kTcIdesc, accumulate);
}

// Rows are spread over the TMEM lane quadrants so that every epilogue group has rows
// when there are few: row n sits at MMA row 128*mt + 32*q + l with (mt, q) = the
// quadrant slot n mod (4*MT) and lane l = n / (4*MT).
__device__ __forceinline__ int mma_row(int n, int MT) {
    const int slot = n % (4 * MT), l = n / (4 * MT);
    return (slot >> 2) * 128 + (slot & 3) * 32 + l;
}
__device__ __forceinline__ int row_of(int mt, int q, int l, int MT) { return l * (4 * MT) + mt * 4 + q; }

constexpr int kTcWarps = 18;                 // producer, MMA, 16 epilogue warps
// TMEM accumulator buffers: all 512 columns, so the MMA runs up to NB-1 tiles ahead
// of the epilogue (4 with one 128-row M tile, 2 with two)
template <int MT> struct TcBufs { static constexpr int N = MT == 1 ? 4 : 2; };
// Wt ring stages of 16 KB: a compile-time count, so the single-thread producer and MMA
// loops index the ring without integer division (deeper rings did not stream faster
// with one M tile: the extra copies only queue behind the first ones).  With two M
// tiles at T=1 the ring holds one whole tile (4 stages at r = 256).
template <int MT, int TT> struct TcStages { static constexpr int N = MT == 1 ? 6 : (TT == 1 ? 4 : 3); };
constexpr int kTcThreads = 32 * kTcWarps;

struct TcShared {
    uint8_t* a;          // MT * KB blocks (gathered U rows)
    uint8_t* b;          // S blocks (Wt tiles)
    float4* slice_rec;   // [4 groups][4 quadrants][32 lanes] running records
    float4* tile_rec;    // [2][4][4][32] per-tile slice records (T=1)
    uint64_t* full;      // [S]
    uint64_t* empty;     // [S]
    uint64_t* tfull;     // [NB]
    uint64_t* tempty;    // [NB]
    uint64_t* drain;     // [1]
};

// The tensor-core tile phase of one biased pass.  Pipeline counters persist across
// passes in the registers of the thread that owns each role.
template <int MT, typename LT, int TT>
__device__ bool tc_tile_phase(const DraftParams& p, const CUtensorMap* tmap, const int32_t* prev, const int32_t* anc,
                              float4* rec_out, const TcShared& sh, uint32_t tmem, uint32_t& it_p, uint32_t& it_m,
                              uint32_t& jt_m, uint32_t& jt_e, uint32_t& pre_issued, unsigned long long* keys,
                              const uint8_t* act) {
    constexpr int NB = TcBufs<MT>::N;
    constexpr int EW = 4 / MT;                 // column slices per quadrant and M tile
    constexpr int CPW = kTcN / EW;             // columns per epilogue warp (32 * MT)
    constexpr int NCH = CPW / 32;              // 32-column chunks per warp (MT)
    constexpr int LW = LWords<LT>::N;          // 16-byte words per chunk of logits
    const int R = p.B * p.gamma;
    const int KB = p.r / kTcK;
    const int CPR = p.r / 8;                  // 16-byte chunks per U row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bf16_t* U = static_cast<const bf16_t*>(p.U);
    __shared__ int s_fail;
    // T=1 from the second biased pass on: only the rows flagged in act are recomputed
    auto live = [&](int n) { return TT == 1 && act != nullptr ? act[n] != 0 : true; };

    const int tb = tile_begin(blockIdx.x, gridDim.x, p.n_tiles), te = tile_begin(blockIdx.x + 1, gridDim.x, p.n_tiles);
    // the epilogue's first tile of logits depends on no token: requested before the gather,
    // so the two round trips overlap
    uint4 lw[NCH][LW];
    if (warp >= 2) {
        const int q = warp & 3, g4 = (warp - 2) >> 2;
        const int g = row_of(g4 / EW, q, lane, MT);
        if (g < R && live(g) && tb < te) {
            const LT* lrow = static_cast<const LT*>(p.logits) + (size_t)g * p.V;
#pragma unroll
            for (int c = 0; c < NCH; ++c) load_l32<LT>(lrow, (long)tb * kTcN + (g4 % EW) * CPW + 32 * c, p.V, lw[c]);
        }
    }
    // gather A = U[x_prev(n)] for the padded rows, 128-byte swizzled, K-major
    if (threadIdx.x == 0) s_fail = 0;
    __shared__ int s_xp[TT == 1 ? 256 : 1];   // T=1: x_prev of every row (R <= 256)
    if constexpr (TT == 1) {
        // the rows' previous tokens come from global memory: read them all at once,
        // then keep GU of a thread's 16-byte U words in flight
        for (int n = threadIdx.x; n < R; n += blockDim.x) s_xp[n] = live(n) ? prev_token(p, prev, n, anc) : -1;
        __syncthreads();
        constexpr int GU = 8;
        const int total = MT * 128 * CPR;
        for (int i0 = threadIdx.x; i0 < total; i0 += GU * blockDim.x) {
            uint4 v[GU];
#pragma unroll
            for (int u = 0; u < GU; ++u) {
                const int idx = i0 + u * (int)blockDim.x;
                v[u] = make_uint4(0u, 0u, 0u, 0u);
                if (idx < total) {
                    const int n = idx / CPR, kc = idx - n * CPR;
                    const int x = n < R ? s_xp[n] : -1;
                    if (x >= 0 && x < p.V) v[u] = __ldg(reinterpret_cast<const uint4*>(U + (size_t)x * p.r) + kc);
                }
            }
#pragma unroll
            for (int u = 0; u < GU; ++u) {
                const int idx = i0 + u * (int)blockDim.x;
                if (idx < total) {
                    const int n = idx / CPR, kc = idx - n * CPR;
                    const int pos = mma_row(n, MT);
                    const int kb = kc >> 3, c = kc & 7, mt = pos >> 7, nl = pos & 127;
                    *reinterpret_cast<uint4*>(sh.a + (size_t)(mt * KB + kb) * kTcBlock + nl * 128 + ((c ^ (nl & 7)) << 4)) =
                        v[u];
                }
            }
        }
    } else
    for (int idx = threadIdx.x; idx < MT * 128 * CPR; idx += blockDim.x) {
        const int n = idx / CPR, kc = idx - n * CPR;
        const int pos = mma_row(n, MT);
        const int kb = kc >> 3, c = kc & 7, mt = pos >> 7, nl = pos & 127;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (n < R && live(n)) {
            const int x = prev_token(p, prev, n, anc);
            if (x >= 0 && x < p.V) v = __ldg(reinterpret_cast<const uint4*>(U + (size_t)x * p.r) + kc);
        }
        *reinterpret_cast<uint4*>(sh.a + (size_t)(mt * KB + kb) * kTcBlock + nl * 128 + ((c ^ (nl & 7)) << 4)) = v;
    }
    fence_proxy_async_smem();
    __syncthreads();

    constexpr int S = TcStages<MT, TT>::N;
    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();   // Wt is streamed once per pass
            uint32_t skip = pre_issued;   // stages of this pass already in flight
            pre_issued = 0;
            for (int t = tb; t < te && !*(volatile int*)&s_fail; ++t) {
                for (int kb = 0; kb < KB; ++kb) {
                    if (skip > 0) { --skip; continue; }
                    const uint32_t s = it_p % S, ph = (it_p / S) & 1u;
                    if (!mbar_wait(&sh.empty[s], ph ^ 1u, p.status, kWaitLimitNs)) { s_fail = 1; break; }
                    mbar_arrive_expect_tx(&sh.full[s], kTcBlock);
                    tma_load_2d_hint(sh.b + (size_t)s * kTcBlock, tmap, kb * kTcK, t * kTcN, &sh.full[s], pol);
                    ++it_p;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            for (int t = tb; t < te && !*(volatile int*)&s_fail; ++t) {
                const uint32_t buf = jt_m % NB, jph = (jt_m / NB) & 1u;
                if (!mbar_wait(&sh.tempty[buf], jph ^ 1u, p.status, kWaitLimitNs)) { s_fail = 1; break; }
                tc_fence_after();
                for (int kb = 0; kb < KB; ++kb) {
                    const uint32_t s = it_m % S, ph = (it_m / S) & 1u;
                    if (!mbar_wait(&sh.full[s], ph, p.status, kWaitLimitNs)) { s_fail = 1; break; }
                    tc_fence_after();
                    const uint32_t b0 = smem_u32(sh.b + (size_t)s * kTcBlock);
#pragma unroll
                    for (int kk = 0; kk < kTcK / 16; ++kk) {
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            const uint32_t a0 = smem_u32(sh.a + (size_t)(mt * KB + kb) * kTcBlock);
                            umma_bf16(tmem + (buf * MT + mt) * kTcN, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32),
                                      (kb | kk) != 0 ? 1u : 0u);
                        }
                    }
                    umma_commit(&sh.empty[s]);
                    ++it_m;
                }
                umma_commit(&sh.tfull[buf]);
                ++jt_m;
            }
        }
    } else {
        // epilogue: group g4 = (w-2)/4 of lane quadrant q = w%4 holds column slice cs
        // of M tile mt; thread = one row
        const int q = warp & 3, g4 = (warp - 2) >> 2;
        const int mt = g4 / EW, cs = g4 % EW;
        const int g = row_of(mt, q, lane, MT);
        const bool group_rows = row_of(mt, q, 0, MT) < R;
        const bool mine = g < R && live(g);
        int prev_ok = 1;
        if (mine) {
            const int x = TT == 1 ? s_xp[g] : prev_token(p, prev, g, anc);
            prev_ok = (x >= 0 && x < p.V) ? 1 : 0;
        }
        const LT* lrow = static_cast<const LT*>(p.logits) + (size_t)(mine ? g : 0) * p.V;
        const bool write_z = p.qlogits_out != nullptr;
        constexpr bool keep_tiles = TT == 1;
        constexpr bool want_idx = TT == 0;
        const int col0 = cs * CPW;
        RowAcc run = rowacc_empty();
        // logits of this warp's columns of tile t, chunk c of tile t+1 requested as soon
        // as chunk c of tile t is consumed
        for (int t = tb; t < te; ++t) {
            const uint32_t buf = jt_e % NB, jph = (jt_e / NB) & 1u;
            const long v0 = (long)t * kTcN + col0;
            if (!mbar_wait(&sh.tfull[buf], jph, p.status, kWaitLimitNs)) { s_fail = 1; break; }
            tc_fence_after();
            RowAcc tacc = rowacc_empty();
            if (group_rows) {
                const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (buf * MT + mt) * kTcN + col0;
                const bool full = v0 + CPW <= p.V;
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    float z[32];
                    tmem_ld32(taddr + 32 * c, z);
                    if (mine) {
                        add_l32<LT>(lw[c], z);
                        if (t + 1 < te) load_l32<LT>(lrow, v0 + kTcN + 32 * c, p.V, lw[c]);
                        if (!full) {
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (v0 + 32 * c + e >= p.V) z[e] = -INFINITY;
                        }
                        tacc = rowacc_merge(tacc, record32(z, (int)(v0 + 32 * c), fmaxf(run.mx, tacc.mx), want_idx));
                        if (write_z) {
                            float* dst = p.qlogits_out + (size_t)g * p.V + v0 + 32 * c;
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                if (v0 + 32 * c + 4 * i + 4 <= p.V)
                                    *reinterpret_cast<float4*>(dst + 4 * i) =
                                        make_float4(z[4 * i], z[4 * i + 1], z[4 * i + 2], z[4 * i + 3]);
                        }
                    }
                }
                if (mine && !prev_ok) tacc.bad = 2;
                run = rowacc_merge(run, tacc);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive1(&sh.tempty[buf]);
            const uint32_t tsl = jt_e & 1u;   // two record slots suffice: a named barrier per tile
            ++jt_e;
            if (keep_tiles && group_rows) {
                // T=1: merge the column slices of the tile in slice order
                float4* slot = sh.tile_rec + (size_t)(tsl * 16 + g4 * 4 + q) * 32;
                slot[lane] = rowacc_pack(tacc);
                named_barrier(1 + mt * 4 + q, 32 * EW);
                if (cs == 0 && mine) {
                    RowAcc m = rowacc_empty();
                    for (int k = 0; k < EW; ++k)
                        m = rowacc_merge(m, rowacc_unpack(sh.tile_rec[(size_t)(tsl * 16 + (mt * EW + k) * 4 + q) * 32 + lane]));
                    p.tile_rec[(size_t)g * p.n_tiles + t] = rowacc_pack(m);
                }
            }
        }
        if (mine && !prev_ok) run.bad = 2;
        sh.slice_rec[(size_t)(g4 * 4 + q) * 32 + lane] = rowacc_pack(run);
    }
    __syncthreads();
    // the CTA's record per row: its column slices merged in slice order
    if (warp >= 2) {
        const int q = warp & 3, g4 = (warp - 2) >> 2;
        const int mt = g4 / EW, cs = g4 % EW;
        const int g = row_of(mt, q, lane, MT);
        if (cs == 0 && g < R && live(g)) {
            RowAcc m = rowacc_empty();
            for (int k = 0; k < EW; ++k)
                m = rowacc_merge(m, rowacc_unpack(sh.slice_rec[(size_t)((mt * EW + k) * 4 + q) * 32 + lane]));
            rec_out[(size_t)g * gridDim.x + blockIdx.x] = rowacc_pack(m);
            if (keys) red_max_u64(&keys[(size_t)g * kKeyStride], rec_key(m));
        }
    }
    return *(volatile int*)&s_fail == 0;
}

// TT = the temperature (0 or 1): each kernel holds only its own temperature's code.
template <int MT, typename LT, int TT>
__global__ void __launch_bounds__(kTcThreads, 1)
    draft_tc_kernel(const __grid_constant__ DraftParams p, const __grid_constant__ CUtensorMap tmap) {
    extern __shared__ uint8_t s_raw[];
    uint8_t* base = s_raw + ((1024u - (smem_u32(s_raw) & 1023u)) & 1023u);
    const int KB = p.r / kTcK;
    const int nw = blockDim.x >> 5;
    // shared layout: A | Wt ring (S stages) | slice records | [T=1: tile records |
    // the draw groups' tile logits] | mbarriers | TMEM address | tokens | anchors.  T=0
    // needs neither T=1 region.
    TcShared sh;
    constexpr int S = TcStages<MT, TT>::N;
    sh.a = base;
    sh.b = base + (size_t)MT * KB * kTcBlock;
    sh.slice_rec = reinterpret_cast<float4*>(sh.b + (size_t)S * kTcBlock);
    constexpr bool t1 = TT == 1;
    sh.tile_rec = t1 ? sh.slice_rec + 16 * 32 : nullptr;
    float* s_uw_all = reinterpret_cast<float*>(sh.slice_rec + (t1 ? 3 : 1) * 16 * 32);
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_uw_all + (t1 ? (size_t)kDraftTile * (nw / kDrawWarps) : 0));
    sh.full = bars;
    sh.empty = bars + S;
    constexpr int NB = TcBufs<MT>::N;
    sh.tfull = bars + 2 * S;
    sh.tempty = bars + 2 * S + NB;
    sh.drain = bars + 2 * S + 2 * NB;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 2 * S + 2 * NB + 1);
    const int R = p.B * p.gamma;
    int32_t* s_tok = reinterpret_cast<int32_t*>(s_tmem + 4);   // [2][B*gamma] (T=0)
    int32_t* s_anc = s_tok + 2 * R;                             // [B] anchors
    float* s_mx = reinterpret_cast<float*>(s_anc + p.B);        // [B*gamma] row maxima (T=0)
    const int warp = threadIdx.x >> 5;
    constexpr uint32_t tmem_cols = 512u;

    pdl_launch_dependents();   // a following verify may stream its target rows meanwhile
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) { mbar_init(&sh.full[s], 1); mbar_init(&sh.empty[s], 1); }
        for (int b = 0; b < NB; ++b) { mbar_init(&sh.tfull[b], 1); mbar_init(&sh.tempty[b], kTcWarps - 2); }
        mbar_init(sh.drain, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(s_tmem, tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    uint32_t it_p = 0, it_m = 0, jt_m = 0, jt_e = 0, pre_issued = 0;
    __shared__ uint32_t s_pre;
    if (warp == nw - 1) {
        // the last warp has no pass-0 row unless there are more rows than warps.  It
        // requests the first biased pass's first Wt stages, which depend on no token, so
        // they land while pass 0 streams the logits; the producer (thread 0) takes the
        // count over after the next barrier.  It also loads the anchors, first needed
        // after pass 0 and its barrier.
        if ((threadIdx.x & 31) == 0) {
            const int tb = tile_begin(blockIdx.x, gridDim.x, p.n_tiles);
            const int te = tile_begin(blockIdx.x + 1, gridDim.x, p.n_tiles);
            const uint32_t total = (uint32_t)(te - tb) * (uint32_t)KB;
            const uint32_t n = total < (uint32_t)S ? total : (uint32_t)S;
            const uint64_t pol = l2_evict_first_policy();
            for (uint32_t i = 0; i < n; ++i) {
                mbar_arrive_expect_tx(&sh.full[i], kTcBlock);
                tma_load_2d_hint(sh.b + (size_t)i * kTcBlock, &tmap, (int)(i % KB) * kTcK, (tb + (int)(i / KB)) * kTcN,
                                 &sh.full[i], pol);
            }
            s_pre = n;
        }
        for (int b = threadIdx.x & 31; b < p.B; b += 32) s_anc[b] = p.anchor[b];
    }
    const unsigned nb = gridDim.x;
    GridBarrier gb = grid_barrier_init(p.barrier);
    __shared__ int s_last_out;   // this CTA was the last to leave (thread 0 sets it)
    bool exited = false;         // the exit count is taken
    bool ok = true;
    int pass = 0;
    // T=0 argmax keys: pass j folds into buffer j % 3, read after its barrier; the buffer
    // of pass j + 1 was last read before barrier j - 1, so CTA 0 clears it at the start
    // of pass j (j >= 2; all three are zero at launch, and the last CTA to leave
    // clears them again)
    auto key_buf = [&](int pass_) { return p.keys + (size_t)(pass_ % 3) * R * kKeyStride; };
    if constexpr (TT == 0) {
        // T=0: every CTA takes every row's token from the folded keys, so a pass needs
        // one grid barrier; only the last pass's confidences are merged, by the row
        // owners.  Records alternate between two buffers so no CTA overwrites what an
        // owner still reads.
        int32_t* tok[2] = {s_tok, s_tok + R};
        tile_phase_stream0_t0<LT>(p, p.cta_rec, false, key_buf(0));
        if (!grid_barrier(gb, nb, p.status)) ok = false;
        if (threadIdx.x == 0) { pre_issued = s_pre; it_p = s_pre; }
        if (ok) finalize_keys_t0(p, key_buf(0), nullptr, tok[0], s_mx, false);
        for (pass = 1; ok; ++pass) {
            if (pass >= 2 && blockIdx.x == 0)
                for (int r = threadIdx.x; r < R; r += blockDim.x) key_buf(pass + 1)[(size_t)r * kKeyStride] = 0ull;
            float4* rec = (pass & 1) ? p.cta_rec2 : p.cta_rec;
            if (!tc_tile_phase<MT, LT, TT>(p, &tmap, tok[(pass + 1) & 1], s_anc, rec, sh, tmem, it_p, it_m, jt_m, jt_e,
                                       pre_issued, key_buf(pass), nullptr)) {
                ok = false;
                break;
            }
            if (!grid_barrier(gb, nb, p.status)) { ok = false; break; }
            const bool changed = finalize_keys_t0(p, key_buf(pass), tok[(pass + 1) & 1], tok[pass & 1], s_mx, true);
            if (!changed || pass == p.gamma) {
                // no barrier and no key read follow: count this CTA out now, so the
                // count's round trip overlaps the owners' work
                if (threadIdx.x == 0) s_last_out = grid_barrier_exit(gb, nb) ? 1 : 0;
                exited = true;
                owner_outputs_t0(p, rec, tok[pass & 1], s_mx, s_anc);
                break;
            }
        }
    } else {
        // Row j of pass k draws from the fixed uniform of its position given x_{j-1} of
        // pass k-1 alone, so from pass 2 on a row whose predecessor kept its token keeps
        // its own token, confidence and probability: only the rows whose predecessor
        // changed in the last pass are recomputed (s_act, one flag per row, in the room
        // T=0 keeps its tokens in).  Every CTA reads the same two token buffers, which
        // no CTA writes before the next grid barrier, so all take the same flags.
        uint8_t* s_act = reinterpret_cast<uint8_t*>(s_tok);
        for (;; ++pass) {
            const bool use_bias = pass > 0;
            const int32_t* prev = p.tokbuf + ((pass + 1) & 1) * (size_t)R;
            int32_t* cur = p.tokbuf + (pass & 1) * (size_t)R;
            if (blockIdx.x == 0 && threadIdx.x == 0) p.changed[pass + 1] = 0u;
            const uint8_t* act = nullptr;
            if (pass >= 2) {
                int n_act = 0;
                for (int r0 = 0; r0 < R; r0 += blockDim.x) {
                    const int row = r0 + threadIdx.x;
                    bool a = false;
                    if (row < R && row % p.gamma != 0) a = __ldcg(&prev[row - 1]) != __ldcg(&cur[row - 1]);
                    if (row < R) s_act[row] = a ? 1 : 0;
                    n_act += __syncthreads_count(a);
                }
                if (n_act == 0) break;   // the pass would change no row: the chain is final
                act = s_act;
            }
            if (use_bias) {
                if (!tc_tile_phase<MT, LT, TT>(p, &tmap, prev, s_anc, p.cta_rec, sh, tmem, it_p, it_m, jt_m, jt_e,
                                           pre_issued, nullptr, act)) {
                    ok = false;
                    break;
                }
            } else {
                tile_phase_stream0_t1<LT>(p);
            }
            if (!grid_barrier(gb, nb, p.status)) { ok = false; break; }
            if (pass == 0 && threadIdx.x == 0) { pre_issued = s_pre; it_p = s_pre; }
            if (use_bias) finalize_rows_t1g<LT>(p, pass, prev, cur, gridDim.x, s_uw_all, act);
            else finalize_rows<LT, bf16_t>(p, pass, use_bias, prev, cur, gridDim.x, nullptr);   // no bias: no U row
            if (!grid_barrier(gb, nb, p.status)) { ok = false; break; }
            if (pass >= 1 && __ldcg(&p.changed[pass]) == 0u) break;
            if (pass == p.gamma) break;
        }
    }

    // every MMA this CTA issued has completed before TMEM is released, and no TMA copy
    // still writes this CTA's shared memory when it exits (stages requested ahead and
    // never consumed, after an error)
    __syncthreads();
    if (threadIdx.x == 32) {
        umma_commit(sh.drain);
        mbar_wait(sh.drain, 0u, p.status, kWaitLimitNs);
    }
    if (threadIdx.x == 0) {
        if (it_p == 0) it_p = s_pre;   // stopped before taking the requested stages over
        const uint32_t n = it_p < (uint32_t)S ? it_p : (uint32_t)S;
        for (uint32_t i = it_p - n; i < it_p; ++i)
            mbar_wait(&sh.full[i % S], (i / S) & 1u, p.status, kWaitLimitNs);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
    if (!exited && threadIdx.x == 0) s_last_out = (ok && grid_barrier_exit(gb, nb)) ? 1 : 0;
    __syncthreads();
    if (s_last_out && TT == 0)
        for (int i = threadIdx.x; i < 3 * R; i += blockDim.x) p.keys[(size_t)i * kKeyStride] = 0ull;
    if (!ok || blockIdx.x != 0) return;
    if (TT != 0) chain_fixup(p);   // T=0 owners applied the chain rule already
    if (threadIdx.x == 0 && p.passes_out) {
        if (p.passes_max) atomicMax(p.passes_out, pass);
        else *p.passes_out = pass;
    }
}

// ----------------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------------
bool draft_tc_supported(const DraftParams& p) {
    const int R = p.B * p.gamma;
    return p.r >= kTcK && p.r <= 256 && p.r % kTcK == 0 && p.wdt == SPEC_BF16 && R <= 256 && p.vec_l &&
           encode_tiled() != nullptr;
}

constexpr size_t kTcSmemBudget = 227 * 1024;   // dynamic shared memory per CTA

template <int MT, typename LT, int TT>
static cudaError_t launch_tc(const DraftParams& p, cudaStream_t stream) {
    const int threads = kTcThreads;
    const int KB = p.r / kTcK;
    constexpr bool t1 = TT == 1;
    constexpr int S = TcStages<MT, TT>::N;
    const size_t smem = 1024 + (size_t)MT * KB * kTcBlock + (size_t)S * kTcBlock +
                        sizeof(float4) * (t1 ? 3 : 1) * 16 * 32 +
                        (t1 ? sizeof(float) * kDraftTile * (kTcWarps / kDrawWarps) : 0) +
                        sizeof(uint64_t) * (2 * S + 2 * TcBufs<MT>::N + 1) + 16 +
                        sizeof(int32_t) * (2 * (size_t)p.B * p.gamma + p.B) + sizeof(float) * (size_t)p.B * p.gamma;
    if (smem > kTcSmemBudget) return cudaErrorInvalidConfiguration;
    auto kern = draft_tc_kernel<MT, LT, TT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    int grid = device_sm_count();   // one CTA per SM (TMEM and shared memory sized for it)
    if (grid > p.n_tiles) grid = p.n_tiles;

    CUtensorMap tmap;
    const cuuint64_t dims[2] = {(cuuint64_t)p.r, (cuuint64_t)p.V};
    const cuuint64_t strides[1] = {(cuuint64_t)p.r * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kTcK, (cuuint32_t)kTcN};
    const cuuint32_t estr[2] = {1, 1};
    if (encode_tiled()(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.Wt), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    DraftParams args = p;
    void* kargs[] = {&args, &tmap};
    return cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(threads), kargs, smem, stream);
}

cudaError_t draft_launch_tc(const DraftParams& p, cudaStream_t stream) {
    const int R = p.B * p.gamma;
    const bool lb = p.ldt == SPEC_BF16;
    if (p.temperature == 0) {
        if (R <= 128) return lb ? launch_tc<1, bf16_t, 0>(p, stream) : launch_tc<1, float, 0>(p, stream);
        return lb ? launch_tc<2, bf16_t, 0>(p, stream) : launch_tc<2, float, 0>(p, stream);
    }
    if (R <= 128) return lb ? launch_tc<1, bf16_t, 1>(p, stream) : launch_tc<1, float, 1>(p, stream);
    return lb ? launch_tc<2, bf16_t, 1>(p, stream) : launch_tc<2, float, 1>(p, stream);
}

}  // namespace spec
