// draft_topk.cu - the DSpark block draft at T=1 with top-k / top-p filtered draws
// (spec_draft_block_topk).
//
// Defines: "Speculative Decoding Part 2" (VESSL AI), DSpark section, bias equation: the
// chain x_j = draw(l_j + W_1[x_{j-1}] W_2); "DSpine card numbers and public file
// headers" (aiwithghost.com), section on raising the temperature: sampling at T=1 with
// top_p 0.95 and top_k 20.  The filter is spec_verify_topk's reading; the draw is the
// inverse CDF of the filtered row in vocabulary-index order with u = Philox(seed_b; b,
// j, 0); the confidence stays 1/Z of the unfiltered row; q_j(x_j) is the filtered
// probability of the drawn token.
//
// A filtered draw needs the biased row's k largest entries, so the chain is walked
// position by position: per position j, two kernels.
//   draft_topk_tiles_kernel  CTA c owns a contiguous range of 128-entry vocabulary tiles
//                            (one CTA per SM).  The tiles' Wt rows stream through a
//                            two-stage ring of bulk copies, so the next tile lands while
//                            the current one is used.  For 32 requests at a time it
//                            gathers U[x_{j-1}] into shared memory; per tile it forms the
//                            128 x 32 bias block with bf16 tensor-core MMAs (float32
//                            accumulate) and adds the drafter logits.  Each request's z
//                            values are folded into base-2 softmax statistics (one record
//                            per request and CTA), the tile's largest key (value, lowest
//                            index) is recorded, and z itself is written out (float32).
//   draft_topk_pick_kernel   one CTA per request: merges the statistics (c_j = 1/Z).  The
//                            row's k largest entries lie in the k tiles with the largest
//                            maxima: no other tile holds an entry at or above the k-th
//                            largest tile maximum T, which is itself at or below the row's
//                            k-th largest entry.  So the k largest tile maxima are selected,
//                            those tiles' z values re-read, the entries at or above T
//                            ranked, and the k largest filtered and drawn.  It writes the
//                            outputs and x_j for position j+1.
// The weights are read once per position for every 32 requests.  From position 2 on, the
// tiles kernel is a programmatic dependent of the previous pick: its first weight copies
// are issued before it waits for x_{j-1}.
#include <mma.h>

#include "spec_device.cuh"
#include "internal.h"
#include "tc_common.cuh"
#include "topk_common.cuh"

namespace spec {

constexpr int kDtThreads = 512;               // tiles kernel: 16 warps
constexpr int kDpThreads = 256;               // pick kernel
constexpr int kDpWarps = kDpThreads / 32;
constexpr int kDtChunk = 32;                  // requests per gathered U block
constexpr int kDtTile = 128;                  // vocabulary entries per tile
constexpr int kDtMaxCtas = 512;               // CTA ranges (workspace sizing)
constexpr int kDtRecMax = 4 * kDtMaxCtas;     // statistics records per request (CTA, or CTA and quadrant)
constexpr int kDtCandCap = 4096;              // candidates of the pick kernel
constexpr int kDtLdz = kDtTile + 4;           // bias block row (floats)
constexpr int kDpPer = kDtCandCap / kDpThreads;   // candidates per pick thread
constexpr int kDpRecPer = kDtRecMax / kDpThreads;  // statistics records per pick thread
static_assert(SPEC_MAX_V_DRAFT_TOPK / kDtTile <= kDtCandCap, "every tile maximum fits the candidate buffer");
static_assert(SPEC_MAX_TOP_K * kDtTile <= kDtCandCap, "the k best tiles' entries fit the candidate buffer");

struct DraftTopkParams {
    const void* logits;        // [B, gamma, V]
    int ldt;
    const int32_t* anchor;     // [B]
    const bf16_t* U;           // [V, r] (r = 0: no bias)
    const bf16_t* Wt;          // [V, r]
    int r, B, gamma, V, k, j;  // j: the position of this launch (1-based)
    double top_p;
    const uint64_t* seeds;
    int32_t* tokens_out;       // [B, gamma]
    float* conf_out;
    float* qtok_out;           // nullable
    int nC;                    // CTA ranges of the tiles kernel
    int nrec;                  // statistics records per request (nC, or 4 nC on the tensor-core path)
    int n_tiles;
    long ldzb;                 // row stride of zbuf: V rounded up to a multiple of 4
    bool vec;                  // logits rows 16-byte aligned with V % 4 == 0 (4-entry loads)
    bool lbulk;                // logits rows a multiple of 16 bytes: tiles copied with the weights
    unsigned* status;
    int32_t* xprev;            // [B] x_{j-1} for j >= 2 (-1: the request has ended)
    float2* stats;             // [B * kDtRecMax] (m2, s) per record
    unsigned* bad;             // [B * kDtRecMax]
    unsigned long long* tmax;  // [B * n_tiles] each tile's largest key (zero between positions)
    float* zbuf;               // [B][ldzb] the biased logits z_j
};

__device__ __forceinline__ int dt_prev(const DraftTopkParams& p, int b) {
    const int x = p.j == 1 ? p.anchor[b] : p.xprev[b];
    return (x >= 0 && x < p.V) ? x : -1;
}

// Four consecutive drafter logits from entry v (-inf past V).
template <typename LT>
__device__ __forceinline__ void load4(const LT* row, long v, int V, bool vec, float (&x)[4]) {
    if (vec && v + 4 <= V) {
        if constexpr (sizeof(LT) == 2) {
            const uint2 w = __ldg(reinterpret_cast<const uint2*>(row + v));
            x[0] = __uint_as_float(w.x << 16);
            x[1] = __uint_as_float(w.x & 0xffff0000u);
            x[2] = __uint_as_float(w.y << 16);
            x[3] = __uint_as_float(w.y & 0xffff0000u);
        } else {
            const float4 w = __ldg(reinterpret_cast<const float4*>(row + v));
            x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = v + e < V ? load_one(row + v + e) : -INFINITY;
    }
}

// One logit from shared memory as float.
__device__ __forceinline__ float load_one_smem(const float* q) { return *q; }
__device__ __forceinline__ float load_one_smem(const bf16_t* q) {
    return __uint_as_float((uint32_t)*reinterpret_cast<const unsigned short*>(q) << 16);
}

template <typename LT>
__global__ void __launch_bounds__(kDtThreads, 1) draft_topk_tiles_kernel(DraftTopkParams p) {
    using namespace nvcuda;
    extern __shared__ __align__(128) uint8_t dt_smem[];
    __shared__ __align__(8) uint64_t s_full[2];
    const int r = p.r;
    const int ldw = r + 8;   // padded Wt / U rows (bf16): 16-byte multiples, no bank conflicts
    const bool lbulk = p.lbulk;
    // ring stage: the tile's Wt rows [128][ldw], then the chunk's logits [32][128]
    const size_t wbytes = r > 0 ? (size_t)kDtTile * ldw * sizeof(bf16_t) : 0;
    const size_t stage = wbytes + (lbulk ? (size_t)kDtChunk * kDtTile * sizeof(LT) : 0);
    bf16_t* s_u = reinterpret_cast<bf16_t*>(dt_smem + 2 * stage);                        // [32][ldw]
    float* s_z = reinterpret_cast<float*>(s_u + (size_t)kDtChunk * ldw);                 // [2][32][kDtLdz]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c = blockIdx.x;
    const int tb = (int)(((long)c * p.n_tiles) / p.nC), te = (int)(((long)(c + 1) * p.n_tiles) / p.nC);
    const int nt = te - tb;
    const int nchunks = (p.B + kDtChunk - 1) / kDtChunk;
    const bool ring = r > 0 || lbulk;
    const long total = ring ? (long)nchunks * nt : 0;   // ring items: (chunk, tile) in order

    // ring item i: tile tb + i % nt of chunk i / nt into stage i % 2 (issued by warp 0): the
    // tile's Wt rows and the chunk's drafter logits over the tile
    auto issue = [&](long i) {
        const long v0 = (long)(tb + (int)(i % nt)) * kDtTile;
        const int nv = (int)min((long)kDtTile, (long)p.V - v0);
        const int b0 = (int)(i / nt) * kDtChunk, nb = min(kDtChunk, p.B - b0);
        uint8_t* dst = dt_smem + (size_t)(i & 1) * stage;
        const unsigned bytes = (unsigned)(r > 0 ? nv * r * 2 : 0) + (unsigned)(lbulk ? nb * nv * (int)sizeof(LT) : 0);
        if (lane == 0) mbar_arrive_expect_tx(&s_full[i & 1], bytes);
        __syncwarp();
        if (r > 0)
            for (int q = lane; q < nv; q += 32)
                bulk_g2s(dst + (size_t)q * ldw * sizeof(bf16_t), p.Wt + (size_t)(v0 + q) * r, (unsigned)(r * 2),
                         &s_full[i & 1]);
        if (lbulk)
            for (int q = lane; q < nb; q += 32)
                bulk_g2s(dst + wbytes + (size_t)q * kDtTile * sizeof(LT),
                         static_cast<const LT*>(p.logits) + ((size_t)(b0 + q) * p.gamma + (p.j - 1)) * p.V + v0,
                         (unsigned)(nv * (int)sizeof(LT)), &s_full[i & 1]);
    };
    if (threadIdx.x == 0) {
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    long issued = 0;
    if (warp == 0)
        for (; issued < 2 && issued < total; ++issued) issue(issued);   // independent of x_{j-1}
    pdl_wait_primary();   // x_{j-1}, and the previous position's reads of this workspace

    long i = 0;           // ring items consumed
    bool abort = false;
    for (int ch = 0; ch < nchunks && !abort; ++ch) {
        const int b0 = ch * kDtChunk, nb = min(kDtChunk, p.B - b0);
        // U[x_{j-1}] of the chunk's requests (zero rows for ended requests and padding)
        if (r > 0) {
            const int wpr = r / 8;   // 16-byte words per row
            for (int q = threadIdx.x; q < kDtChunk * wpr; q += blockDim.x) {
                const int rb = q / wpr, w = q - rb * wpr;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (rb < nb) {
                    const int x = dt_prev(p, b0 + rb);
                    if (x >= 0) v = __ldg(reinterpret_cast<const uint4*>(p.U + (size_t)x * r) + w);
                }
                *reinterpret_cast<uint4*>(s_u + (size_t)rb * ldw + w * 8) = v;
            }
        }
        // this warp's two requests of the chunk: running statistics
        float m2[2], sacc[2];
        int bad[2], live[2];
        const LT* lrow[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int rb = warp * 2 + h, b = b0 + rb;
            m2[h] = -INFINITY;
            sacc[h] = 0.0f;
            bad[h] = 0;
            live[h] = (rb < nb && dt_prev(p, b) >= 0) ? 1 : 0;
            lrow[h] = static_cast<const LT*>(p.logits) + ((size_t)b * p.gamma + (p.j - 1)) * p.V;
        }
        __syncthreads();

        for (int t = tb; t < te; ++t) {
            const long v0 = (long)t * kDtTile;
            float* sz = s_z + (size_t)(i & 1) * kDtChunk * kDtLdz;
            const uint8_t* st = dt_smem + (size_t)(i & 1) * stage;
            bool ok = true;
            if (ring) ok = mbar_wait(&s_full[i & 1], (unsigned)((i >> 1) & 1), p.status, kWaitLimitNs);
            // this warp's two requests' logits over the tile (lane l: entries v0 + 4l .. +3),
            // taken before the stage is released
            float lv[2][4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (!live[h]) continue;
                if (lbulk) {
                    const LT* sl = reinterpret_cast<const LT*>(st + wbytes) + (size_t)(warp * 2 + h) * kDtTile + 4 * lane;
                    if constexpr (sizeof(LT) == 2) {
                        const uint2 w = *reinterpret_cast<const uint2*>(sl);
                        lv[h][0] = __uint_as_float(w.x << 16);
                        lv[h][1] = __uint_as_float(w.x & 0xffff0000u);
                        lv[h][2] = __uint_as_float(w.y << 16);
                        lv[h][3] = __uint_as_float(w.y & 0xffff0000u);
                    } else {
                        const float4 w = *reinterpret_cast<const float4*>(sl);
                        lv[h][0] = w.x; lv[h][1] = w.y; lv[h][2] = w.z; lv[h][3] = w.w;
                    }
                } else {
                    load4<LT>(lrow[h], v0 + 4 * lane, p.V, p.vec, lv[h]);
                }
            }
            if (ring) {
                // bias block: warp w takes vocabulary rows 16 (w % 8) .. and requests 16 (w / 8) ..
                if (ok && r > 0) {
                    wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::row_major> fa;
                    wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::col_major> fb;
                    wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc;
                    wmma::fill_fragment(acc, 0.0f);
                    const __nv_bfloat16* A = reinterpret_cast<const __nv_bfloat16*>(st) + (size_t)(16 * (warp & 7)) * ldw;
                    const __nv_bfloat16* Bm = reinterpret_cast<const __nv_bfloat16*>(s_u) + (size_t)(16 * (warp >> 3)) * ldw;
                    for (int kk = 0; kk < r; kk += 16) {
                        wmma::load_matrix_sync(fa, A + kk, ldw);
                        wmma::load_matrix_sync(fb, Bm + kk, ldw);
                        wmma::mma_sync(acc, fa, fb, acc);
                    }
                    // element (v, b) goes to sz[b * kDtLdz + v]
                    wmma::store_matrix_sync(sz + (size_t)(16 * (warp >> 3)) * kDtLdz + 16 * (warp & 7), acc, kDtLdz,
                                            wmma::mem_col_major);
                }
                if (__syncthreads_or(!ok)) { abort = true; break; }
                // stage i % 2 is free: refill it with item i + 2
                if (warp == 0 && issued < total && issued == i + 2) {
                    fence_proxy_async_smem();
                    issue(issued);
                    ++issued;
                }
                ++i;
            }
            // fold the tile for this warp's two requests: lane l holds entries v0 + 4l .. +3
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (!live[h]) continue;   // warp-uniform
                const int rb = warp * 2 + h, b = b0 + rb;
                const long vb = v0 + 4 * lane;
                float z[4] = {lv[h][0], lv[h][1], lv[h][2], lv[h][3]};
                if (r > 0) {
                    const float4 bz = *reinterpret_cast<const float4*>(sz + (size_t)rb * kDtLdz + 4 * lane);
                    z[0] += bz.x; z[1] += bz.y; z[2] += bz.z; z[3] += bz.w;
                }
                int lbad = 0;
                float lmax = -INFINITY;
                unsigned long long kmax = 0ull;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (vb + e < p.V) {
                        if (bad_logit(z[e])) lbad = 1;
                        lmax = fmaxf(lmax, z[e]);
                        const unsigned long long kk = argmax_key(z[e], (uint32_t)(vb + e));
                        kmax = kk > kmax ? kk : kmax;
                    } else {
                        z[e] = -INFINITY;
                    }
                }
                bad[h] |= warp_or(lbad);
                if (bad[h]) continue;
                const float lm2 = lmax * kLog2e;
                if (lm2 > m2[h]) {
                    sacc[h] *= ex2(m2[h] - lm2);
                    m2[h] = lm2;
                }
                if (m2[h] != -INFINITY) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) sacc[h] += wexp(z[e], m2[h]);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const unsigned long long k2 = shfl_u64(kmax, lane ^ o);
                    kmax = k2 > kmax ? k2 : kmax;
                }
                if (lane == 0) p.tmax[(size_t)b * p.n_tiles + t] = kmax;
                if (vb < p.V)
                    *reinterpret_cast<float4*>(p.zbuf + (size_t)b * p.ldzb + vb) = make_float4(z[0], z[1], z[2], z[3]);
            }
        }
        if (abort) break;

        // one record per (request, CTA)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int rb = warp * 2 + h, b = b0 + rb;
            if (rb >= nb) continue;   // warp-uniform
            const size_t rec = (size_t)b * kDtRecMax + c;
            const float M = warp_max(m2[h]);
            float s = (m2[h] != -INFINITY && M != -INFINITY) ? sacc[h] * ex2(m2[h] - M) : 0.0f;
            s = warp_sum(s);
            if (lane == 0) {
                p.stats[rec] = make_float2(M, s);
                p.bad[rec] = bad[h] ? 1u : 0u;
            }
        }
        __syncthreads();   // s_u is rewritten by the next chunk
    }
    if (abort && threadIdx.x == 0)   // copies still in flight land before the CTA leaves (bounded)
        for (long q = i; q < issued; ++q) mbar_wait(&s_full[q & 1], (unsigned)((q >> 1) & 1), p.status, kWaitLimitNs);
}

// ----------------------------------------------------------------------------------
// The tiles kernel on the tcgen05 tensor cores (bf16 weights, r a multiple of 64, logits
// rows a multiple of 16 bytes).  Per CTA (one per SM), 18 warps:
//   warp 0      TMA producer: per tile, its Wt rows as r / 64 boxes [128 entries x 64 k]
//               (128-byte swizzle) into a ring of 16 KB stages, and the chunk's drafter
//               logits over the tile as one box [32 requests x 128 entries] into a ring
//               of its own;
//   warp 1      allocates TMEM and issues tcgen05.mma (M = 128 entries, N = 32 requests,
//               K = 16, bf16 in, f32 accumulate) from one thread into two 32-column
//               accumulators, so the next tile's MMAs run while the epilogue reads this
//               one;
//   warps 2-17  epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 (one entry per
//               thread) and 8 of the 32 request columns; per request it adds the
//               logits, folds the softmax statistics, writes z, and folds the tile's
//               largest key into tmax with one atomicMax per warp.
// The B operand, U[x_{j-1}] of the chunk's 32 requests, is written by the epilogue warps
// in the same K-major 128-byte-swizzled layout, double-buffered across chunks.  No
// block-wide barrier runs after the set-up: every wait is a bounded mbarrier wait.
// ----------------------------------------------------------------------------------
constexpr int kDkK = 64;                                 // k per 128-byte swizzle block
constexpr int kDkWBlock = kDtTile * kDkK * 2;            // 16 KB: one Wt box
constexpr int kDkUBlock = kDtChunk * kDkK * 2;           // 4 KB: one U block
// Wt ring stages of 16 KB (two tiles at r = 256; 9 or 10 stages streamed slower: the
// extra copies only queue behind the first ones)
template <typename LT> struct DkStages { static constexpr int N = 8; };
constexpr int kDkLStages = 3;                            // logits ring
constexpr int kDkEpi = 16;                               // epilogue warps
constexpr int kDkThreads = 32 * (2 + kDkEpi);
constexpr uint32_t kDkIdesc = idesc_bf16_f32(kDtTile, kDtChunk);
constexpr uint32_t kDkTmemCols = 2 * kDtChunk;           // two accumulators of 32 columns

template <typename LT>
__global__ void __launch_bounds__(kDkThreads, 1)
    draft_topk_tc_kernel(const __grid_constant__ DraftTopkParams p, const __grid_constant__ CUtensorMap wmap,
                         const __grid_constant__ CUtensorMap lmap) {
    extern __shared__ uint8_t dk_raw[];
    uint8_t* base = dk_raw + ((1024u - (smem_u32(dk_raw) & 1023u)) & 1023u);
    constexpr int kDkStages = DkStages<LT>::N;
    constexpr int LBYTES = kDtChunk * kDtTile * (int)sizeof(LT);
    const int KB = p.r / kDkK;
    uint8_t* s_w = base;                                          // [kDkStages][16 KB]
    uint8_t* s_u = s_w + (size_t)kDkStages * kDkWBlock;           // [2][KB][4 KB]
    uint8_t* s_l = s_u + (size_t)2 * KB * kDkUBlock;              // [kDkLStages][LBYTES]
    __shared__ __align__(8) uint64_t s_full[kDkStages], s_empty[kDkStages];
    __shared__ __align__(8) uint64_t s_lfull[kDkLStages], s_lempty[kDkLStages];
    __shared__ __align__(8) uint64_t s_tfull[2], s_tempty[2], s_ufull[2], s_drain;
    __shared__ uint32_t s_tmem;
    __shared__ int s_fail;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const int tb = (int)(((long)c * p.n_tiles) / p.nC), te = (int)(((long)(c + 1) * p.n_tiles) / p.nC);
    const int nchunks = (p.B + kDtChunk - 1) / kDtChunk;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kDkStages; ++s) { mbar_init(&s_full[s], 1); mbar_init(&s_empty[s], 1); }
        for (int s = 0; s < kDkLStages; ++s) { mbar_init(&s_lfull[s], 1); mbar_init(&s_lempty[s], kDkEpi); }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&s_tfull[s], 1);
            mbar_init(&s_tempty[s], kDkEpi);
            mbar_init(&s_ufull[s], kDkEpi);
        }
        mbar_init(&s_drain, 1);
        s_fail = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&s_tmem, kDkTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    uint32_t iw = 0, il = 0;   // producer: Wt stages and logits stages issued

    if (warp == 0) {
        // neither the weights nor the logits depend on the previous kernel: no wait
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();   // Wt and the logits are streamed once
            for (int ch = 0; ch < nchunks && !*(volatile int*)&s_fail; ++ch)
                for (int t = tb; t < te; ++t) {
                    bool ok = true;
                    for (int kb = 0; kb < KB && ok; ++kb) {
                        const uint32_t s = iw % kDkStages, ph = (iw / kDkStages) & 1u;
                        ok = mbar_wait(&s_empty[s], ph ^ 1u, p.status, kWaitLimitNs);
                        if (!ok) break;
                        mbar_arrive_expect_tx(&s_full[s], kDkWBlock);
                        tma_load_2d_hint(s_w + (size_t)s * kDkWBlock, &wmap, kb * kDkK, t * kDtTile, &s_full[s], pol);
                        ++iw;
                    }
                    if (ok) {
                        const uint32_t s = il % kDkLStages, ph = (il / kDkLStages) & 1u;
                        ok = mbar_wait(&s_lempty[s], ph ^ 1u, p.status, kWaitLimitNs);
                        if (ok) {
                            mbar_arrive_expect_tx(&s_lfull[s], LBYTES);
                            tma_load_2d_hint(s_l + (size_t)s * LBYTES, &lmap, t * kDtTile, ch * kDtChunk, &s_lfull[s], pol);
                            ++il;
                        }
                    }
                    if (!ok) { s_fail = 1; break; }
                }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t im = 0, jt = 0;
            for (int ch = 0; ch < nchunks && !*(volatile int*)&s_fail; ++ch) {
                if (!mbar_wait(&s_ufull[ch & 1], (unsigned)((ch >> 1) & 1), p.status, kWaitLimitNs)) { s_fail = 1; break; }
                tc_fence_after();
                const uint32_t u0 = smem_u32(s_u + (size_t)(ch & 1) * KB * kDkUBlock);
                bool ok = true;
                for (int t = tb; t < te && ok; ++t) {
                    const uint32_t buf = jt & 1u, jph = (jt >> 1) & 1u;
                    ok = mbar_wait(&s_tempty[buf], jph ^ 1u, p.status, kWaitLimitNs);
                    if (!ok) break;
                    tc_fence_after();
                    for (int kb = 0; kb < KB; ++kb) {
                        const uint32_t s = im % kDkStages, ph = (im / kDkStages) & 1u;
                        ok = mbar_wait(&s_full[s], ph, p.status, kWaitLimitNs);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t w0 = smem_u32(s_w + (size_t)s * kDkWBlock);
#pragma unroll
                        for (int kk = 0; kk < kDkK / 16; ++kk)
                            umma_f16(tmem + buf * kDtChunk, sw128_desc(w0 + kk * 32),
                                     sw128_desc(u0 + kb * kDkUBlock + kk * 32), kDkIdesc, (kb | kk) != 0 ? 1u : 0u);
                        umma_commit(&s_empty[s]);
                        ++im;
                    }
                    if (!ok) break;
                    umma_commit(&s_tfull[buf]);
                    ++jt;
                }
                if (!ok) { s_fail = 1; break; }
            }
        }
    } else {
        const int e = warp - 2;        // epilogue warp 0..15
        const int q = warp & 3;        // its TMEM lane quadrant: entries 32 q .. +31 of a tile
        const int g = e >> 2;          // its requests: 8 g .. 8 g + 7 of the chunk
        const int CPR = p.r / 8;       // 16-byte chunks per U row
        pdl_wait_primary();            // x_{j-1}; the previous pick's reads of z and tmax
        uint32_t je = 0, ie = 0;       // tiles and logits stages consumed
        for (int ch = 0; ch < nchunks; ++ch) {
            const int b0 = ch * kDtChunk, nb = min(kDtChunk, p.B - b0);
            // B operand: U[x_{j-1}] of the chunk's requests (zero rows for ended requests and
            // padding), 128-byte swizzled, K-major, into buffer ch % 2 (its previous user,
            // chunk ch - 2, finished its MMAs before this warp saw chunk ch - 1's tiles)
            uint8_t* ub = s_u + (size_t)(ch & 1) * KB * kDkUBlock;
            for (int idx = (int)threadIdx.x - 64; idx < kDtChunk * CPR; idx += 32 * kDkEpi) {
                const int n = idx / CPR, kc = idx - n * CPR;
                const int kb = kc >> 3, cc = kc & 7;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (n < nb) {
                    const int x = dt_prev(p, b0 + n);
                    if (x >= 0) v = __ldg(reinterpret_cast<const uint4*>(p.U + (size_t)x * p.r) + kc);
                }
                *reinterpret_cast<uint4*>(ub + (size_t)kb * kDkUBlock + n * 128 + ((cc ^ (n & 7)) << 4)) = v;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive1(&s_ufull[ch & 1]);

            // this warp's 8 requests: warp-uniform running maximum (base 2), per-lane sums
            float m2[8], sl[8];
            unsigned live = 0u, badm = 0u;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                m2[i] = -INFINITY;
                sl[i] = 0.0f;
                const int rb = 8 * g + i;
                if (rb < nb && dt_prev(p, b0 + rb) >= 0) live |= 1u << i;
            }
            bool ok = true;
            for (int t = tb; t < te; ++t) {
                const uint32_t buf = je & 1u, jph = (je >> 1) & 1u;
                ok = __all_sync(0xffffffffu, mbar_wait(&s_tfull[buf], jph, p.status, kWaitLimitNs));
                if (!ok) break;
                tc_fence_after();
                float bias[8];
                tmem_ld8(tmem + ((uint32_t)(32 * q) << 16) + buf * kDtChunk + 8 * g, bias);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive1(&s_tempty[buf]);
                ++je;
                const uint32_t ls = ie % kDkLStages, lph = (ie / kDkLStages) & 1u;
                ok = __all_sync(0xffffffffu, mbar_wait(&s_lfull[ls], lph, p.status, kWaitLimitNs));
                if (!ok) break;
                const LT* lt = reinterpret_cast<const LT*>(s_l + (size_t)ls * LBYTES);
                const int vl = 32 * q + lane;   // this thread's entry of the tile
                float z[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) z[i] = load_one_smem(lt + (8 * g + i) * kDtTile + vl) + bias[i];
                __syncwarp();
                if (lane == 0) mbar_arrive1(&s_lempty[ls]);
                ++ie;
                const long v = (long)t * kDtTile + vl;
                const bool in = v < p.V;
                if (!in) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) z[i] = -INFINITY;
                }
                // a NaN or +inf entry ends its request (one OR over the warp for all 8)
                unsigned bl = 0u;
#pragma unroll
                for (int i = 0; i < 8; ++i) bl |= bad_logit(z[i]) ? 1u << i : 0u;
                badm |= __reduce_or_sync(0xffffffffu, bl) & live;
                // the quadrant's 8 maxima at once: at the xor-16, -8 and -4 steps each lane
                // keeps half of its values, so lanes 4r .. 4r+3 end with request r's
                float h4[4], h2[2], h1;
                {
                    const bool up = (lane & 16) != 0;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float give = up ? z[j] : z[j + 4], keep = up ? z[j + 4] : z[j];
                        h4[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, give, 16));
                    }
                }
                {
                    const bool up = (lane & 8) != 0;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const float give = up ? h4[j] : h4[j + 2], keep = up ? h4[j + 2] : h4[j];
                        h2[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, give, 8));
                    }
                }
                {
                    const bool up = (lane & 4) != 0;
                    const float give = up ? h2[0] : h2[1], keep = up ? h2[1] : h2[0];
                    h1 = fmaxf(keep, __shfl_xor_sync(0xffffffffu, give, 4));
                }
                h1 = fmaxf(h1, __shfl_xor_sync(0xffffffffu, h1, 2));
                h1 = fmaxf(h1, __shfl_xor_sync(0xffffffffu, h1, 1));
                const int ri = lane >> 2;   // the request whose maximum this lane holds
                unsigned my_hit = 0u;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (!((live >> i) & 1u) || ((badm >> i) & 1u)) continue;   // warp-uniform
                    const int b = b0 + 8 * g + i;
                    const float m = __shfl_sync(0xffffffffu, h1, 4 * i);
                    // the lowest index of the maximum: the tile's key, folded below by lane 4i
                    const unsigned hit = __ballot_sync(0xffffffffu, in && z[i] == m);
                    if (ri == i) my_hit = hit;
                    const float tm2 = m * kLog2e;
                    if (tm2 > m2[i]) {
                        sl[i] *= ex2(m2[i] - tm2);
                        m2[i] = tm2;
                    }
                    if (in) {
                        if (m2[i] != -INFINITY) sl[i] += wexp(z[i], m2[i]);
                        p.zbuf[(size_t)b * p.ldzb + v] = z[i];
                    }
                }
                // the tile keys of the live requests: one atomic instruction, lanes 4i
                if ((lane & 3) == 0 && my_hit != 0u && ((live >> ri) & 1u) && !((badm >> ri) & 1u))
                    atomicMax(&p.tmax[(size_t)(b0 + 8 * g + ri) * p.n_tiles + t],
                              argmax_key(h1, (uint32_t)((long)t * kDtTile + 32 * q + __ffs(my_hit) - 1)));
            }
            if (!ok) { s_fail = 1; break; }
            // one record per (request, CTA, quadrant)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int rb = 8 * g + i;
                if (rb >= nb) continue;   // warp-uniform
                const float S = warp_sum(sl[i]);
                if (lane == 0) {
                    const size_t rec = (size_t)(b0 + rb) * kDtRecMax + (size_t)c * 4 + q;
                    p.stats[rec] = make_float2(m2[i], S);
                    p.bad[rec] = ((badm >> i) & 1u) ? 1u : 0u;
                }
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
        const uint32_t nw = iw < (uint32_t)kDkStages ? iw : (uint32_t)kDkStages;
        for (uint32_t i = iw - nw; i < iw; ++i) mbar_wait(&s_full[i % kDkStages], (i / kDkStages) & 1u, p.status, kWaitLimitNs);
        const uint32_t nl = il < (uint32_t)kDkLStages ? il : (uint32_t)kDkLStages;
        for (uint32_t i = il - nl; i < il; ++i) mbar_wait(&s_lfull[i % kDkLStages], (i / kDkLStages) & 1u, p.status, kWaitLimitNs);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kDkTmemCols);
    }
}

// The CTA's k-th largest of the keys held one per thread (k <= 32), by a per-warp sort
// and a rank across the warps' sorted lists; 0 if the CTA holds fewer than k non-zero keys.
// Every thread returns the same value.
__device__ unsigned long long dp_block_kth(unsigned long long key, int k, unsigned long long* s_buf) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // bitonic sort of the warp's keys, descending
#pragma unroll
    for (int kk = 2; kk <= 32; kk <<= 1)
#pragma unroll
        for (int jj = kk >> 1; jj > 0; jj >>= 1) {
            const unsigned long long o = shfl_u64(key, lane ^ jj);
            const bool take_max = ((lane & kk) == 0) == ((lane & jj) == 0);
            key = take_max ? (o > key ? o : key) : (o < key ? o : key);
        }
    s_buf[threadIdx.x] = key;
    __syncthreads();
    __shared__ unsigned long long s_kth;
    if (threadIdx.x == 0) s_kth = 0ull;
    __syncthreads();
    if (lane < k && key != 0ull) {
        int rank = lane;
        for (int w = 0; w < kDpWarps; ++w) {
            if (w == warp) continue;
            const unsigned long long* a = s_buf + w * 32;
            int lo = 0, hi = k;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (a[mid] > key) lo = mid + 1;
                else hi = mid;
            }
            rank += lo;
        }
        if (rank == k - 1) s_kth = key;
    }
    __syncthreads();
    const unsigned long long r = s_kth;
    __syncthreads();   // s_buf and s_kth may be reused
    return r;
}

// The n keys of s_c ranked: those among the k largest go to s_top[rank] (s_top zeroed
// first, so fewer than k keys leave zeros).  Keys are distinct.
__device__ void dp_top_k(const unsigned long long* s_c, int n, int k, unsigned long long* s_top) {
    if (threadIdx.x < kTopkMax) s_top[threadIdx.x] = 0ull;
    __syncthreads();
    for (int q = threadIdx.x; q < n; q += blockDim.x) {
        const unsigned long long key = s_c[q];
        int rank = 0;
        for (int i = 0; i < n && rank < k; ++i) rank += s_c[i] > key ? 1 : 0;
        if (rank < k) s_top[rank] = key;
    }
    __syncthreads();
}

// One CTA per request: merge the CTA records, select, filter, draw x_j.
__global__ void __launch_bounds__(kDpThreads) draft_topk_pick_kernel(DraftTopkParams p) {
    __shared__ unsigned long long s_cand[kDtCandCap];
    __shared__ unsigned long long s_top[kTopkMax];
    __shared__ FRow s_row;
    __shared__ float s_red[kDpWarps];
    __shared__ int s_badw[kDpWarps];
    __shared__ unsigned long long s_sort[kDpThreads];
    __shared__ int s_cnt;
    pdl_launch_dependents();   // the next position's tiles kernel may start its weight copies
    const int b = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const size_t out = (size_t)b * p.gamma + (p.j - 1);
    const int k = p.k;
    auto end_request = [&](unsigned flag) {   // no distribution at this position: -1 from here on
        if (threadIdx.x == 0) {
            p.tokens_out[out] = -1;
            p.conf_out[out] = NAN;
            if (p.qtok_out) p.qtok_out[out] = NAN;
            p.xprev[b] = -1;
            if (flag) atomicOr(p.status, flag);
        }
    };
    // one wave of loads: this request's tile maxima (returned to zero for the next
    // position, whose tensor-core tiles kernel folds them by atomicMax), its statistics
    // records and its previous token, all held in registers
    unsigned long long* tm = p.tmax + (size_t)b * p.n_tiles;
    unsigned long long kr[kDpPer];
    unsigned long long lmax = 0ull;
#pragma unroll
    for (int u = 0; u < kDpPer; ++u) {
        const int t = (int)threadIdx.x + u * kDpThreads;
        kr[u] = t < p.n_tiles ? __ldcg(&tm[t]) : 0ull;
    }
    float2 st[kDpRecPer];
    unsigned bd = 0u;
#pragma unroll
    for (int u = 0; u < kDpRecPer; ++u) {
        const int c = (int)threadIdx.x + u * kDpThreads;
        const size_t rec = (size_t)b * kDtRecMax + c;
        st[u] = c < p.nrec ? __ldcg(&p.stats[rec]) : make_float2(-INFINITY, 0.0f);
        bd |= c < p.nrec ? __ldcg(&p.bad[rec]) : 0u;
    }
    const int xp = dt_prev(p, b);
    // the draw's uniform depends on no data: warp 0 takes it while the loads are in flight
    const float u_draw = warp == 0 ? philox_uniform(p.seeds[b], (uint64_t)b, (uint64_t)p.j, 0) : 0.0f;
#pragma unroll
    for (int u = 0; u < kDpPer; ++u) {
        const int t = (int)threadIdx.x + u * kDpThreads;
        lmax = kr[u] > lmax ? kr[u] : lmax;
        if (t < p.n_tiles) tm[t] = 0ull;
    }
    if (xp < 0) {   // ended earlier (or the anchor is out of range)
        end_request((p.j == 1 && (p.anchor[b] < 0 || p.anchor[b] >= p.V)) ? SPEC_DEV_TOKEN : 0u);
        return;
    }
    // statistics: the maximum (NaN or a bad record ends the row), then the rescaled sums
    float M = -INFINITY;
    int lbad = bd != 0u ? 1 : 0;
#pragma unroll
    for (int u = 0; u < kDpRecPer; ++u) {
        if (isnan(st[u].x)) lbad = 1;
        M = fmaxf(M, st[u].x);
    }
    M = warp_max(M);
    lbad = warp_or(lbad);
    if (lane == 0) { s_red[warp] = M; s_badw[warp] = lbad; }
    if (threadIdx.x == 0) s_cnt = 0;
    __syncthreads();
    M = -INFINITY;
    int bad_row = 0;
    for (int w = 0; w < kDpWarps; ++w) {
        M = fmaxf(M, s_red[w]);
        bad_row |= s_badw[w];
    }
    if (bad_row || M == -INFINITY) {
        end_request(SPEC_DEV_NONFINITE);
        return;
    }
    float S = 0.0f;
#pragma unroll
    for (int u = 0; u < kDpRecPer; ++u)
        if (st[u].x != -INFINITY) S += st[u].y * ex2(st[u].x - M);
    S = warp_sum(S);
    __syncthreads();   // s_red is rewritten
    if (lane == 0) s_red[warp] = S;
    // 1. a bound at or below the k-th largest tile maximum: the k-th largest of the
    //    threads' maxima (distinct tile maxima)
    const unsigned long long t_lo = dp_block_kth(lmax, k, s_sort);
    // 2. the tile maxima at or above it (at most n_tiles <= kDtCandCap), and the k largest
#pragma unroll
    for (int u = 0; u < kDpPer; ++u)
        if (kr[u] != 0ull && kr[u] >= t_lo) s_cand[atomicAdd(&s_cnt, 1)] = kr[u];
    __syncthreads();
    dp_top_k(s_cand, s_cnt, k, s_top);
    // 3. the entries of those tiles at or above the smallest of them, T
    unsigned long long T = 0ull;
    int ntop = 0;
    for (int q = 0; q < k; ++q)
        if (s_top[q] != 0ull) { T = s_top[q]; ntop = q + 1; }
    if (ntop < k) T = 0ull;   // fewer than k tiles: every entry of them
    __syncthreads();
    if (threadIdx.x == 0) s_cnt = 0;
    __syncthreads();
    const float* zr = p.zbuf + (size_t)b * p.ldzb;
    float zv[kDpPer];
#pragma unroll
    for (int u = 0; u < kDpPer; ++u) {   // one wave of loads
        const int q = (int)threadIdx.x + u * kDpThreads;
        const long v = q < ntop * kDtTile ? (long)(key_index(s_top[q / kDtTile]) / kDtTile) * kDtTile + (q % kDtTile) : p.V;
        zv[u] = v < p.V ? __ldcg(&zr[v]) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kDpPer; ++u) {
        const int q = (int)threadIdx.x + u * kDpThreads;
        const long v = q < ntop * kDtTile ? (long)(key_index(s_top[q / kDtTile]) / kDtTile) * kDtTile + (q % kDtTile) : p.V;
        if (v < p.V) {
            const unsigned long long kv = argmax_key(zv[u], (uint32_t)v);
            if (kv >= T) s_cand[atomicAdd(&s_cnt, 1)] = kv;
        }
    }
    __syncthreads();
    dp_top_k(s_cand, s_cnt, k, s_top);
    if (warp != 0) return;
    filter_row(s_top, k, p.top_p, s_row);
    __syncwarp();
    if (s_row.n == 0) {   // no finite entry
        end_request(SPEC_DEV_NONFINITE);
        return;
    }
    float Z = 0.0f;   // the unfiltered row's normaliser (base-2 sums against M)
    for (int w = 0; w < kDpWarps; ++w) Z += s_red[w];
    const float u = u_draw;
    int near = 0;
    const int il = lane < s_row.n ? s_row.idx[lane] : -1;
    const int x = warp_draw(il, lane < s_row.n ? s_row.pf[lane] : 0.0f, u, near);
    const float qx = frow_prob(s_row, x);
    if (lane == 0) {
        p.tokens_out[out] = x;
        p.conf_out[out] = 1.0f / Z;
        if (p.qtok_out) p.qtok_out[out] = qx;
        p.xprev[b] = x;
        // the next position gathers U[x_j]: bring the row into L2 now
        if (p.r > 0 && p.j < p.gamma && x >= 0) bulk_prefetch_l2(p.U + (size_t)x * p.r, (unsigned)(p.r * 2));
    }
}

// ----------------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------------
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static size_t dt_ldzb(int V) { return ((size_t)V + 3) / 4 * 4; }

// The tensor-core tiles kernel and the picks, position by position.  The weights' map is
// [V rows][r] (boxes of 128 rows x 64 k, 128-byte swizzle); the logits' map for position
// j is [B rows][V] with a row stride of gamma * V entries (boxes of 32 rows x 128
// entries), so one copy brings a chunk's logits over a tile.
template <typename LT>
static cudaError_t launch_topk_tc(DraftTopkParams p, const DraftTopkLaunch& a, cudaStream_t stream) {
    const int KB = p.r / kDkK;
    const size_t lbytes = (size_t)kDtChunk * kDtTile * sizeof(LT);
    const size_t smem = 1024 + (size_t)DkStages<LT>::N * kDkWBlock + (size_t)2 * KB * kDkUBlock + (size_t)kDkLStages * lbytes;
    auto kern = draft_topk_tc_kernel<LT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int grid = device_sm_count();   // one CTA per SM (TMEM and shared memory sized for it)
    if (grid > kDtMaxCtas) grid = kDtMaxCtas;
    if (grid > p.n_tiles) grid = p.n_tiles;
    p.nC = grid;
    p.nrec = 4 * grid;

    CUtensorMap wmap;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)p.r, (cuuint64_t)p.V};
        const cuuint64_t strides[1] = {(cuuint64_t)p.r * 2};
        const cuuint32_t box[2] = {(cuuint32_t)kDkK, (cuuint32_t)kDtTile};
        const cuuint32_t estr[2] = {1, 1};
        if (encode_tiled()(&wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<bf16_t*>(p.Wt), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    for (int j = 1; j <= a.gamma; ++j) {
        p.j = j;
        CUtensorMap lmap;
        const cuuint64_t dims[2] = {(cuuint64_t)p.V, (cuuint64_t)p.B};
        const cuuint64_t strides[1] = {(cuuint64_t)p.gamma * p.V * sizeof(LT)};
        const cuuint32_t box[2] = {(cuuint32_t)kDtTile, (cuuint32_t)kDtChunk};
        const cuuint32_t estr[2] = {1, 1};
        void* lbase = const_cast<LT*>(static_cast<const LT*>(p.logits) + (size_t)(j - 1) * p.V);
        if (encode_tiled()(&lmap, sizeof(LT) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                           lbase, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        // from position 2 on, the tiles kernel is a programmatic dependent of the previous
        // pick (its copies and MMAs need nothing from it; its epilogue waits)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(kDkThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        // position 1 follows the caller's work on the stream (which may write the logits
        // or the weights), so it starts only once that work has finished; later positions
        // follow this library's own pick kernel
        cfg.numAttrs = j > 1 ? 1 : 0;
        e = cudaLaunchKernelEx(&cfg, kern, p, wmap, lmap);
        if (e != cudaSuccess) return e;
        draft_topk_pick_kernel<<<a.B, kDpThreads, 0, stream>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

size_t draft_topk_workspace_bytes(int B, int V) {
    const size_t n = (size_t)B * kDtRecMax;
    const size_t n_tiles = ((size_t)V + kDtTile - 1) / kDtTile;
    size_t off = kWsHeaderBytes;
    off = align_up(off + sizeof(int32_t) * (size_t)B, 256);                    // xprev
    off = align_up(off + sizeof(float2) * n, 256);                             // stats
    off = align_up(off + sizeof(unsigned) * n, 256);                           // bad
    off = align_up(off + sizeof(unsigned long long) * (size_t)B * n_tiles, 256);   // tmax
    off = align_up(off + sizeof(float) * (size_t)B * dt_ldzb(V), 256);        // zbuf
    return off;
}

cudaError_t draft_topk_launch(const DraftTopkLaunch& a, void* ws, cudaStream_t stream) {
    DraftTopkParams p;
    memset(&p, 0, sizeof(p));
    p.logits = a.logits;
    p.ldt = a.ldt;
    p.anchor = a.anchor;
    p.U = static_cast<const bf16_t*>(a.U);
    p.Wt = static_cast<const bf16_t*>(a.Wt);
    p.r = a.r;
    p.B = a.B;
    p.gamma = a.gamma;
    p.V = a.V;
    p.k = a.k;
    p.top_p = a.top_p;
    p.seeds = a.seeds;
    p.tokens_out = a.tokens_out;
    p.conf_out = a.conf_out;
    p.qtok_out = a.qtok_out;
    p.n_tiles = (a.V + kDtTile - 1) / kDtTile;
    p.ldzb = (long)dt_ldzb(a.V);
    p.vec = a.V % 4 == 0 && (reinterpret_cast<uintptr_t>(a.logits) & 15u) == 0;
    const size_t esize = a.ldt == SPEC_BF16 ? 2 : 4;
    p.lbulk = ((size_t)a.V * esize) % 16 == 0 && (reinterpret_cast<uintptr_t>(a.logits) & 15u) == 0;
    char* w = static_cast<char*>(ws);
    p.status = &reinterpret_cast<WsHeader*>(w)->status;
    const size_t n = (size_t)a.B * kDtRecMax;
    size_t off = kWsHeaderBytes;
    p.xprev = reinterpret_cast<int32_t*>(w + off);
    off = align_up(off + sizeof(int32_t) * (size_t)a.B, 256);
    p.stats = reinterpret_cast<float2*>(w + off);
    off = align_up(off + sizeof(float2) * n, 256);
    p.bad = reinterpret_cast<unsigned*>(w + off);
    off = align_up(off + sizeof(unsigned) * n, 256);
    p.tmax = reinterpret_cast<unsigned long long*>(w + off);
    off = align_up(off + sizeof(unsigned long long) * (size_t)a.B * p.n_tiles, 256);
    p.zbuf = reinterpret_cast<float*>(w + off);

    if (a.r >= kDkK && a.r % kDkK == 0 && a.r <= 256 && p.lbulk && encode_tiled() != nullptr)
        return a.ldt == SPEC_BF16 ? launch_topk_tc<bf16_t>(p, a, stream) : launch_topk_tc<float>(p, a, stream);

    const int ldw = a.r + 8;
    const size_t stage = (a.r > 0 ? (size_t)kDtTile * ldw * sizeof(bf16_t) : 0) +
                         (p.lbulk ? (size_t)kDtChunk * kDtTile * esize : 0);
    const size_t smem = 2 * stage + (size_t)kDtChunk * ldw * sizeof(bf16_t) + (size_t)2 * kDtChunk * kDtLdz * sizeof(float);
    void (*kt)(DraftTopkParams) = a.ldt == SPEC_BF16 ? draft_topk_tiles_kernel<bf16_t> : draft_topk_tiles_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(kt, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kt, kDtThreads, smem) != cudaSuccess || occ < 1) occ = 1;
    int nC = device_sm_count() * occ;
    if (nC > kDtMaxCtas) nC = kDtMaxCtas;
    if (nC > p.n_tiles) nC = p.n_tiles;
    p.nC = nC;
    p.nrec = nC;
    for (int j = 1; j <= a.gamma; ++j) {
        p.j = j;
        // from position 2 on, the tiles kernel is a programmatic dependent of the previous
        // pick (its weight copies are issued before it waits)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)nC);
        cfg.blockDim = dim3(kDtThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        // position 1 follows the caller's work on the stream (which may write the logits
        // or the weights), so it starts only once that work has finished; later positions
        // follow this library's own pick kernel
        cfg.numAttrs = j > 1 ? 1 : 0;
        e = cudaLaunchKernelEx(&cfg, kt, p);
        if (e != cudaSuccess) return e;
        draft_topk_pick_kernel<<<a.B, kDpThreads, 0, stream>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace spec
