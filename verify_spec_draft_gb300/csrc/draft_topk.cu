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
//   draft_topk_tiles_kernel  CTA c owns a contiguous range of 128-entry vocabulary tiles.
//                            For 32 requests at a time it gathers U[x_{j-1}] into shared
//                            memory; per tile it stages the tile's Wt rows, forms the
//                            128 x 32 bias block with bf16 tensor-core MMAs (float32
//                            accumulate), adds the drafter logits, and folds each
//                            request's z values into base-2 softmax statistics and a
//                            warp-sorted list of its k largest keys (entries below the
//                            list's threshold are skipped).  One record per (request,
//                            CTA).
//   draft_topk_pick_kernel   one CTA per request: merges the statistics (c_j = 1/Z),
//                            takes the row's k largest keys from the CTAs' lists (only
//                            keys at or above the largest CTA k-th key can qualify),
//                            filters, draws, writes the outputs and x_j for position j+1.
// The weights are read once per position (per 32 requests).
#include <mma.h>

#include "spec_device.cuh"
#include "internal.h"
#include "topk_common.cuh"

namespace spec {

constexpr int kDtThreads = 256;
constexpr int kDtWarps = kDtThreads / 32;
constexpr int kDtChunk = 32;        // requests per gathered U block
constexpr int kDtTile = 128;        // vocabulary entries per tile
constexpr int kDtMaxCtas = 512;     // CTA ranges (workspace sizing)
constexpr int kDtCandCap = 4096;    // merge buffer of the pick kernel

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
    int n_tiles;
    unsigned* status;
    int32_t* xprev;            // [B] x_{j-1} for j >= 2 (-1: the request has ended)
    float2* stats;             // [B * kDtMaxCtas] (m2, s) per CTA range
    unsigned* bad;             // [B * kDtMaxCtas]
    unsigned long long* keys;  // [B * kDtMaxCtas * kTopkMax]
};

__device__ __forceinline__ int dt_prev(const DraftTopkParams& p, int b) {
    const int x = p.j == 1 ? p.anchor[b] : p.xprev[b];
    return (x >= 0 && x < p.V) ? x : -1;
}

template <typename LT>
__global__ void __launch_bounds__(kDtThreads) draft_topk_tiles_kernel(DraftTopkParams p) {
    using namespace nvcuda;
    extern __shared__ __align__(128) uint8_t dt_smem[];
    const int r = p.r;
    const int ldw = r + 8;                      // padded rows (bf16), a multiple of 8
    constexpr int ldz = kDtTile + 4;            // z block [32 requests][ldz] float
    bf16_t* s_w = reinterpret_cast<bf16_t*>(dt_smem);                        // [128][ldw]
    bf16_t* s_u = s_w + (size_t)kDtTile * ldw;                                // [32][ldw]
    float* s_z = reinterpret_cast<float*>(s_u + (size_t)kDtChunk * ldw);      // [32][ldz]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c = blockIdx.x;
    const int tb = (int)(((long)c * p.n_tiles) / p.nC), te = (int)(((long)(c + 1) * p.n_tiles) / p.nC);
    const int k = p.k;

    for (int b0 = 0; b0 < p.B; b0 += kDtChunk) {
        const int nb = min(kDtChunk, p.B - b0);
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
        // this warp's four requests of the chunk: running statistics and top-k lists
        unsigned long long mine[4], kth[4], thr[4];
        float thr_v[4], m2[4], sacc[4];
        int bad[4], live[4];
        const LT* lrow[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rb = warp * 4 + i, b = b0 + rb;
            mine[i] = kth[i] = thr[i] = 0ull;
            thr_v[i] = -INFINITY;
            m2[i] = -INFINITY;
            sacc[i] = 0.0f;
            bad[i] = 0;
            live[i] = (rb < nb && dt_prev(p, b) >= 0) ? 1 : 0;
            lrow[i] = static_cast<const LT*>(p.logits) + ((size_t)b * p.gamma + (p.j - 1)) * p.V;
        }
        __syncthreads();

        for (int t = tb; t < te; ++t) {
            const long v0 = (long)t * kDtTile;
            if (r > 0) {
                // the tile's Wt rows (contiguous in memory; zero past V)
                const int wpr = r / 8;
                const int nv = (int)min((long)kDtTile, (long)p.V - v0);
                const uint4* src = reinterpret_cast<const uint4*>(p.Wt + (size_t)v0 * r);
                for (int q = threadIdx.x; q < kDtTile * wpr; q += blockDim.x) {
                    const int rv = q / wpr, w = q - rv * wpr;
                    const uint4 v = rv < nv ? __ldg(src + (size_t)rv * wpr + w) : make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(s_w + (size_t)rv * ldw + w * 8) = v;
                }
                __syncthreads();
                // bias block: rows v of this warp's 16, columns the 32 requests
                wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::row_major> fa;
                wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::col_major> fb;
                wmma::fragment<wmma::accumulator, 16, 16, 16, float> acc0, acc1;
                wmma::fill_fragment(acc0, 0.0f);
                wmma::fill_fragment(acc1, 0.0f);
                const __nv_bfloat16* A = reinterpret_cast<const __nv_bfloat16*>(s_w) + (size_t)(16 * warp) * ldw;
                const __nv_bfloat16* Bm = reinterpret_cast<const __nv_bfloat16*>(s_u);
                for (int kk = 0; kk < r; kk += 16) {
                    wmma::load_matrix_sync(fa, A + kk, ldw);
                    wmma::load_matrix_sync(fb, Bm + kk, ldw);
                    wmma::mma_sync(acc0, fa, fb, acc0);
                    wmma::load_matrix_sync(fb, Bm + (size_t)16 * ldw + kk, ldw);
                    wmma::mma_sync(acc1, fa, fb, acc1);
                }
                // element (v, b) goes to s_z[b * ldz + v]
                wmma::store_matrix_sync(s_z + 16 * warp, acc0, ldz, wmma::mem_col_major);
                wmma::store_matrix_sync(s_z + (size_t)16 * ldz + 16 * warp, acc1, ldz, wmma::mem_col_major);
                __syncthreads();
            }
            // fold the tile's z values of this warp's requests
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (!live[i]) continue;   // warp-uniform
                const int rb = warp * 4 + i;
                float z[4];
                bool in[4];
                float lmax = -INFINITY;
                int lbad = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const long v = v0 + 32 * q + lane;
                    in[q] = v < p.V;
                    z[q] = in[q] ? load_one(lrow[i] + v) + (r > 0 ? s_z[(size_t)rb * ldz + 32 * q + lane] : 0.0f)
                                 : -INFINITY;
                    if (in[q] && bad_logit(z[q])) lbad = 1;
                    lmax = fmaxf(lmax, z[q]);
                }
                bad[i] |= warp_or(lbad);
                if (bad[i]) continue;
                // statistics: per-lane running maximum (base 2) and rescaled sum
                const float lm2 = lmax * kLog2e;
                if (lm2 > m2[i]) {
                    sacc[i] *= ex2(m2[i] - lm2);
                    m2[i] = lm2;
                }
                if (m2[i] != -INFINITY) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) sacc[i] += wexp(z[q], m2[i]);
                }
                // first tile of the range: start the threshold at the k-th largest lane maximum
                if (t == tb) {
                    float lm = lmax;
#pragma unroll
                    for (int kk2 = 2; kk2 <= 32; kk2 <<= 1)
#pragma unroll
                        for (int jj = kk2 >> 1; jj > 0; jj >>= 1) {
                            const float o = __shfl_xor_sync(0xffffffffu, lm, jj);
                            const bool take_max = ((lane & kk2) == 0) != ((lane & jj) == 0);
                            lm = take_max ? fmaxf(lm, o) : fminf(lm, o);
                        }
                    const float seed = __shfl_sync(0xffffffffu, lm, 32 - k);   // ascending: the k-th largest
                    thr_v[i] = fmaxf(thr_v[i], seed);
                }
                // candidates at or above the threshold, inserted one by one (warp-uniform)
                const float cut = thr_v[i];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    unsigned hot = __ballot_sync(0xffffffffu, in[q] && z[q] >= cut);
                    while (hot) {
                        const int src = __ffs(hot) - 1;
                        hot &= hot - 1;
                        const float zv = __shfl_sync(0xffffffffu, z[q], src);
                        const unsigned long long key = argmax_key(zv, (uint32_t)(v0 + 32 * q + src));
                        if (key > thr[i]) {
                            list_insert(mine[i], key, k, kth[i]);
                            if (kth[i] > thr[i]) {
                                thr[i] = kth[i];
                                thr_v[i] = fmaxf(thr_v[i], key_value(kth[i]));
                            }
                        }
                    }
                }
            }
            if (r > 0) __syncthreads();   // s_w and s_z are rewritten for the next tile
        }

        // one record per (request, CTA)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rb = warp * 4 + i, b = b0 + rb;
            if (rb >= nb) continue;   // warp-uniform
            const size_t rec = (size_t)b * kDtMaxCtas + c;
            const float M = warp_max(m2[i]);
            float s = (m2[i] != -INFINITY && M != -INFINITY) ? sacc[i] * ex2(m2[i] - M) : 0.0f;
            s = warp_sum(s);
            if (lane == 0) {
                p.stats[rec] = make_float2(M, s);
                p.bad[rec] = bad[i] ? 1u : 0u;
            }
            p.keys[rec * kTopkMax + lane] = (live[i] && !bad[i] && lane < k) ? mine[i] : 0ull;
        }
        __syncthreads();   // s_u is rewritten by the next chunk
    }
}

// One CTA per request: merge the CTA records, filter, draw x_j.
__global__ void __launch_bounds__(kDtThreads) draft_topk_pick_kernel(DraftTopkParams p) {
    __shared__ unsigned long long s_cand[kDtCandCap];
    __shared__ unsigned long long s_top[kTopkMax];
    __shared__ FRow s_row;
    __shared__ float s_red[kDtWarps];
    __shared__ unsigned long long s_red64[kDtWarps];
    __shared__ int s_cnt, s_bad;
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
    const int xp = dt_prev(p, b);
    if (xp < 0) {   // ended earlier (or the anchor is out of range)
        end_request((p.j == 1 && (p.anchor[b] < 0 || p.anchor[b] >= p.V)) ? SPEC_DEV_TOKEN : 0u);
        return;
    }
    // statistics: the maximum (NaN or a bad record ends the row), then the rescaled sums
    if (threadIdx.x == 0) { s_cnt = 0; s_bad = 0; }
    __syncthreads();
    float M = -INFINITY;
    unsigned long long T = 0ull;
    for (int c = threadIdx.x; c < p.nC; c += blockDim.x) {
        const size_t rec = (size_t)b * kDtMaxCtas + c;
        const float2 st = __ldcg(&p.stats[rec]);
        if (__ldcg(&p.bad[rec]) || isnan(st.x)) s_bad = 1;
        M = fmaxf(M, st.x);
        const unsigned long long kk = __ldcg(&p.keys[rec * kTopkMax + (k - 1)]);
        T = kk > T ? kk : T;
    }
    M = warp_max(M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long t2 = shfl_u64(T, lane ^ o);
        T = t2 > T ? t2 : T;
    }
    if (lane == 0) { s_red[warp] = M; s_red64[warp] = T; }
    __syncthreads();
    M = -INFINITY;
    T = 0ull;
    for (int w = 0; w < kDtWarps; ++w) {
        M = fmaxf(M, s_red[w]);
        T = s_red64[w] > T ? s_red64[w] : T;
    }
    __syncthreads();
    if (s_bad || M == -INFINITY) {
        end_request(SPEC_DEV_NONFINITE);
        return;
    }
    float S = 0.0f;
    for (int c = threadIdx.x; c < p.nC; c += blockDim.x) {
        const float2 st = __ldcg(&p.stats[(size_t)b * kDtMaxCtas + c]);
        if (st.x != -INFINITY) S += st.y * ex2(st.x - M);
    }
    S = warp_sum(S);
    if (lane == 0) s_red[warp] = S;
    // candidates: keys at or above the largest CTA k-th key (every CTA list is sorted)
    for (int c = threadIdx.x; c < p.nC; c += blockDim.x) {
        const unsigned long long* kl = p.keys + ((size_t)b * kDtMaxCtas + c) * kTopkMax;
        for (int i = 0; i < k; ++i) {
            const unsigned long long kv = __ldcg(&kl[i]);
            if (kv == 0ull || kv < T) break;
            const int pos = atomicAdd(&s_cnt, 1);
            if (pos < kDtCandCap) s_cand[pos] = kv;
        }
    }
    __syncthreads();
    S = 0.0f;
    for (int w = 0; w < kDtWarps; ++w) S += s_red[w];
    const int cnt = min(s_cnt, kDtCandCap);
    if (warp != 0) return;
    // the k largest candidates (k rounds of a warp maximum), descending
    unsigned long long prev_best = ~0ull;
    for (int rr = 0; rr < k; ++rr) {
        unsigned long long best = 0ull;
        for (int i = lane; i < cnt; i += 32) {
            const unsigned long long kv = s_cand[i];
            if (kv < prev_best && kv > best) best = kv;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long t2 = shfl_u64(best, lane ^ o);
            best = t2 > best ? t2 : best;
        }
        if (lane == 0) s_top[rr] = best;
        prev_best = best;
        if (best == 0ull) {
            for (int q = rr + 1 + lane; q < k; q += 32) s_top[q] = 0ull;
            break;
        }
    }
    __syncwarp();
    filter_row(s_top, k, p.top_p, s_row);
    __syncwarp();
    if (s_row.n == 0) {   // no finite entry
        end_request(SPEC_DEV_NONFINITE);
        return;
    }
    const float u = philox_uniform(p.seeds[b], (uint64_t)b, (uint64_t)p.j, 0);
    int near = 0;
    const int il = lane < s_row.n ? s_row.idx[lane] : -1;
    const int x = warp_draw(il, lane < s_row.n ? s_row.pf[lane] : 0.0f, u, near);
    const float qx = frow_prob(s_row, x);
    if (lane == 0) {
        p.tokens_out[out] = x;
        p.conf_out[out] = 1.0f / S;
        if (p.qtok_out) p.qtok_out[out] = qx;
        p.xprev[b] = x;
    }
}

// ----------------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------------
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t draft_topk_workspace_bytes(int B) {
    const size_t n = (size_t)B * kDtMaxCtas;
    size_t off = kWsHeaderBytes;
    off = align_up(off + sizeof(int32_t) * (size_t)B, 256);
    off = align_up(off + sizeof(float2) * n, 256);
    off = align_up(off + sizeof(unsigned) * n, 256);
    off = align_up(off + sizeof(unsigned long long) * n * kTopkMax, 256);
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
    char* w = static_cast<char*>(ws);
    p.status = &reinterpret_cast<WsHeader*>(w)->status;
    const size_t n = (size_t)a.B * kDtMaxCtas;
    size_t off = kWsHeaderBytes;
    p.xprev = reinterpret_cast<int32_t*>(w + off);
    off = align_up(off + sizeof(int32_t) * (size_t)a.B, 256);
    p.stats = reinterpret_cast<float2*>(w + off);
    off = align_up(off + sizeof(float2) * n, 256);
    p.bad = reinterpret_cast<unsigned*>(w + off);
    off = align_up(off + sizeof(unsigned) * n, 256);
    p.keys = reinterpret_cast<unsigned long long*>(w + off);

    p.n_tiles = (a.V + kDtTile - 1) / kDtTile;
    int nC = 2 * device_sm_count();
    if (nC > kDtMaxCtas) nC = kDtMaxCtas;
    if (nC > p.n_tiles) nC = p.n_tiles;
    p.nC = nC;
    const int ldw = a.r + 8;
    const size_t smem = a.r > 0 ? (size_t)(kDtTile + kDtChunk) * ldw * sizeof(bf16_t) +
                                      (size_t)kDtChunk * (kDtTile + 4) * sizeof(float)
                                : 0;
    void (*kt)(DraftTopkParams) = a.ldt == SPEC_BF16 ? draft_topk_tiles_kernel<bf16_t> : draft_topk_tiles_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(kt, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    for (int j = 1; j <= a.gamma; ++j) {
        p.j = j;
        kt<<<nC, kDtThreads, smem, stream>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        draft_topk_pick_kernel<<<a.B, kDtThreads, 0, stream>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace spec
