// verify_topk.cu - T=1 verification against top-k / top-p filtered rows
// (spec_verify_topk).
//
// Defines: "DSpine card numbers and public file headers" (aiwithghost.com), section on
// raising the temperature - sampling at T=1 with top_p 0.95 and top_k 20; the rejection
// rule is spec_verify's ("Solar Open2 DSpark", sections 1 and 6; "Speculative Decoding
// Part 2", blockwise decoding section), applied to the filtered rows.
//
// Reading (the page names only the setting): a row's filtered distribution keeps its k
// largest logits (ties to the lowest index), renormalised over them; then the shortest
// prefix, in descending order, whose running sum reaches top_p; renormalised again.  Only
// a row's top k entries matter, so no row-wide softmax is needed:
//
//   topk_rows_kernel   one CTA per row (target and draft rows in one grid) streams it
//                      (HBM-bound).  Each warp keeps the 32 largest 64-bit keys it has
//                      seen (ordered value high, inverted index low: a larger key is a
//                      larger value or, on a tie, a lower index) as a sorted list spread
//                      over its lanes.  A lane looks inside its 8-entry groups only when a
//                      group's packed maximum reaches the threshold, the larger of the
//                      warp's k-th key and the CTA's best published k-th key (no entry
//                      below it can be among the row's k largest); the threshold starts
//                      at the k-th largest lane maximum of the first item.  The entries
//                      above it go to a per-warp buffer (one prefix over the lanes) and are
//                      inserted one by one.  NaN or +inf marks the row bad (it has no
//                      distribution).  The CTA's k largest are ranked out of the lists.
//   topk_accept_kernel one CTA per request.  Each warp filters rows from their key lists
//                      (one candidate per lane, float32; the cut-off is taken again in
//                      float64 when a running sum lies within 1e-5 of top_p), then warp 0
//                      runs the accept tests (Philox stream 1) and the residual or bonus
//                      draw over at most k candidates in index order (streams 2, 3).
#include "spec_device.cuh"
#include "internal.h"
#include "chunk_rows.cuh"
#include "topk_common.cuh"

namespace spec {

constexpr int kTopkThreads = 256;
constexpr int kTopkWarps = kTopkThreads / 32;

// Candidates a warp found in one item, waiting for insertion into its list.
constexpr int kCandCap = 128;

// Entry q (in decode_words order) of a thread's words, decoded on its own.
template <typename T, int NW>
__device__ __forceinline__ float word_entry(const uint4 (&w)[NW], int q) {
    if constexpr (sizeof(T) == 2) {
        const uint4 v = w[q >> 3];
        const int h = (q & 7) >> 1;
        const uint32_t a = h == 0 ? v.x : (h == 1 ? v.y : (h == 2 ? v.z : v.w));
        return (q & 1) ? __uint_as_float(a & 0xffff0000u) : __uint_as_float(a << 16);
    } else {
        const uint4 v = w[q >> 2];
        const int h = q & 3;
        return __uint_as_float(h == 0 ? v.x : (h == 1 ? v.y : (h == 2 ? v.z : v.w)));
    }
}

// The row at `rowp` (V entries); its k largest keys go to keys[row * kTopkMax + i] in
// descending order (0 where the row has fewer entries), its bad flag to bad_out[row].
template <typename T>
__device__ __forceinline__ void topk_row(const T* rowp, long V, int k, bool vec, int row, unsigned long long* keys,
                                         unsigned* bad_out) {
    constexpr int NW = Words<T>::N;
    __shared__ unsigned long long s_thr;                       // best k-th key a warp has published
    __shared__ unsigned long long s_all[kTopkThreads];         // the warps' lists, for the final ranking
    __shared__ unsigned long long s_cand[kTopkWarps][kCandCap];
    __shared__ int s_bad;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nch = (int)((V + kVerifyChunk - 1) / kVerifyChunk);
    if (threadIdx.x == 0) { s_thr = 0ull; s_bad = 0; }
    __syncthreads();

    unsigned long long mine = 0ull;   // this lane's slot of the warp's sorted list
    unsigned long long kth = 0ull;    // the warp's k-th key (0 while the list is short)
    unsigned long long thr = 0ull;    // the key to beat: the larger of kth and the CTA's best
    float thr_v = -INFINITY;          // value threshold: entries below it are skipped
    int bad = 0;
    uint4 cur[NW], nxt[NW];
    load_words_il<T, NW>(cur, rowp, V, il_seg(0), vec);
    for (int c = 0; c < nch; ++c) {
        if (c + 1 < nch) load_words_il<T, NW>(nxt, rowp, V, il_seg(c + 1), vec);
        if (c == 0) {
            // seed: the k-th largest of the 32 lane maxima (each an entry of this item)
            float lm = chunk_max_nan<T, NW>(cur);
            if (isnan(lm) || lm == INFINITY) bad = 1;
#pragma unroll
            for (int kk = 2; kk <= 32; kk <<= 1)   // bitonic sort of the lane maxima, ascending
#pragma unroll
                for (int j = kk >> 1; j > 0; j >>= 1) {
                    const float o = __shfl_xor_sync(0xffffffffu, lm, j);
                    const bool take_max = ((lane & kk) == 0) != ((lane & j) == 0);
                    lm = take_max ? fmaxf(lm, o) : fminf(lm, o);
                }
            const float seed = __shfl_sync(0xffffffffu, lm, 32 - k);   // the k-th largest
            thr_v = isnan(seed) ? -INFINITY : seed;
        }
        // the CTA's best k-th key, read once and broadcast: every lane of the warp must see
        // the same threshold (the insertions below are warp-collective), and other warps
        // raise s_thr concurrently
        unsigned long long st_l = 0ull;
        if (lane == 0) st_l = *(volatile unsigned long long*)&s_thr;
        const unsigned long long shared_thr = shfl_u64(st_l, 0);
        if (shared_thr > thr) {
            thr = shared_thr;
            thr_v = fmaxf(thr_v, key_value(shared_thr));
        }
        // this lane's entries at or above the threshold (their keys), counted first; entry
        // q of the lane is vocabulary index ebase + (q / 8) * 256 + q % 8 (V < 2^31)
        const int ebase = (int)il_seg(c) + lane * 8;
        const int vi = (int)V;
        int ncand = 0;
        float gmax[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if constexpr (sizeof(T) == 2) gmax[j] = u4_max_nan<2>(cur[j]);
            else gmax[j] = f_max_nan(u4_max_nan<4>(cur[2 * j]), u4_max_nan<4>(cur[2 * j + 1]));
            if (isnan(gmax[j]) || gmax[j] == INFINITY) bad = 1;
        }
        const bool any_hot = !bad && (gmax[0] >= thr_v || gmax[1] >= thr_v || gmax[2] >= thr_v || gmax[3] >= thr_v);
        if (__any_sync(0xffffffffu, any_hot)) {
            const float cut = thr_v;   // the entries taken this item: fixed while they are buffered
            if (any_hot) {
#pragma unroll
                for (int q = 0; q < kEPT; ++q)
                    ncand += (word_entry<T, NW>(cur, q) >= cut && ebase + (q >> 3) * 256 + (q & 7) < vi) ? 1 : 0;
            }
            // write them to the warp's buffer (an exclusive prefix over lanes); rounds of at
            // most kCandCap, each followed by the insertions
            int before = 0, total = 0;
            {
                int incl = ncand;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                before = incl - ncand;
                total = __shfl_sync(0xffffffffu, incl, 31);
            }
            for (int r0 = 0; r0 < total; r0 += kCandCap) {
                int pos = before - r0;
                if (any_hot && ncand > 0) {
#pragma unroll
                    for (int q = 0; q < kEPT; ++q) {
                        const int e = ebase + (q >> 3) * 256 + (q & 7);
                        const float xq = word_entry<T, NW>(cur, q);
                        if (xq >= cut && e < vi) {
                            if (pos >= 0 && pos < kCandCap) s_cand[warp][pos] = argmax_key(xq, (uint32_t)e);
                            ++pos;
                        }
                    }
                }
                __syncwarp();
                const int nr = min(kCandCap, total - r0);
                for (int i = 0; i < nr; ++i) {   // warp-uniform
                    const unsigned long long key = s_cand[warp][i];
                    if (key > thr) {
                        list_insert(mine, key, k, kth);
                        if (kth > thr) {
                            thr = kth;
                            thr_v = fmaxf(thr_v, key_value(kth));
                        }
                    }
                }
                __syncwarp();
            }
            // publish the warp's k-th key
            if (lane == 0 && kth > *(volatile unsigned long long*)&s_thr) atomicMax(&s_thr, kth);
        }
#pragma unroll
        for (int i = 0; i < NW; ++i) cur[i] = nxt[i];
    }
    if (bad) s_bad = 1;
    __syncthreads();
    bad = s_bad;
    // the row's k largest: only a warp's first k keys can be among them; rank each of
    // those among all of them (keys are distinct, the index being part of them, except
    // the empty key 0)
    const bool lane_k = lane < k;
    s_all[threadIdx.x] = lane_k ? mine : 0ull;
    __syncthreads();
    unsigned long long* out = keys + (size_t)row * kTopkMax;
    if (threadIdx.x < kTopkMax) out[threadIdx.x] = 0ull;
    __syncthreads();
    if (!bad && lane_k && mine != 0ull) {
        int rank = 0;
        for (int w = 0; w < kTopkWarps; ++w)
            for (int i = 0; i < k; ++i) rank += s_all[w * 32 + i] > mine ? 1 : 0;
        if (rank < k) out[rank] = mine;
    }
    if (threadIdx.x == 0) bad_out[row] = bad ? 1u : 0u;
}

// All rows of a request batch in one grid: target rows 0 .. nT-1, then draft rows.
template <typename TT, typename DT>
__global__ void __launch_bounds__(kTopkThreads) topk_rows_kernel(TopkParams p, bool vt, bool vd) {
    const int row = blockIdx.x;
    const int nT = p.B * (p.gamma + 1);
    if (row < nT)
        topk_row<TT>(static_cast<const TT*>(p.target) + (size_t)row * p.V, p.V, p.k, vt, row, p.keys, p.bad);
    else
        topk_row<DT>(static_cast<const DT*>(p.draft) + (size_t)(row - nT) * p.V, p.V, p.k, vd, row, p.keys, p.bad);
}

// ----------------------------------------------------------------------------------
// Accept and draw: one CTA per request
// ----------------------------------------------------------------------------------
__global__ void __launch_bounds__(kTopkThreads) topk_accept_kernel(TopkParams p) {
    const int b = blockIdx.x;
    const int G = p.gamma;
    const int nT = p.B * (G + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    extern __shared__ __align__(16) unsigned char s_dyn[];
    FRow* rows = reinterpret_cast<FRow*>(s_dyn);   // [2G+1]: target rows 0..G, then draft rows
    __shared__ int s_ok;
    if (threadIdx.x == 0) s_ok = 1;
    __syncthreads();
    for (int i = threadIdx.x; i < G; i += blockDim.x) {
        const int x = p.tokens[(size_t)b * G + i];
        if (x < 0 || x >= p.V) s_ok = 0;
    }
    for (int r = warp; r < 2 * G + 1; r += kTopkWarps) {
        const size_t gr = r <= G ? (size_t)b * (G + 1) + r : (size_t)nT + (size_t)b * G + (r - G - 1);
        if (p.bad[gr]) {
            if (lane == 0) { rows[r].n = 0; s_ok = 0; }
            continue;
        }
        filter_row(p.keys + gr * kTopkMax, p.k, p.top_p, rows[r]);
        __syncwarp();
        if (lane == 0 && rows[r].n == 0) s_ok = 0;
    }
    __syncthreads();
    if (warp != 0) return;
    int32_t* com = p.committed_out + (size_t)b * (G + 1);
    if (!s_ok) {
        for (int i = lane; i <= G; i += 32) com[i] = -1;
        if (lane == 0) {
            p.n_out[b] = -1;
            p.bonus_out[b] = -1;
            if (p.near_out) p.near_out[b] = 0;
            atomicOr(p.status, SPEC_DEV_TOKEN);
        }
        return;
    }
    const uint64_t seed = p.seeds[b];
    int near = 0;
    for (int j = 1; j <= G; ++j) {
        const FRow& P = rows[j - 1];
        const FRow& Q = rows[G + j];
        const int x = p.tokens[(size_t)b * G + j - 1];
        const float px = frow_prob(P, x), qx = frow_prob(Q, x);
        const float u = philox_uniform(seed, (uint64_t)b, (uint64_t)j, 1);
        if (fabsf(u * qx - px) < 1e-6f * qx) near = 1;
        if (u * qx < px) {   // accepted (q = 0 accepts iff p > 0)
            if (lane == 0) com[j - 1] = x;
            continue;
        }
        // the residual max(0, p - q) on the filtered p's candidates (from p if all zero)
        const int il = lane < P.n ? P.idx[lane] : -1;
        const float pl = lane < P.n ? P.pf[lane] : 0.0f;
        const float ql = il >= 0 ? frow_prob_lane(Q, il) : 0.0f;
        float rl = fmaxf(0.0f, pl - ql);
        if (!(warp_sum(rl) > 0.0f)) rl = pl;
        const float u2 = philox_uniform(seed, (uint64_t)b, (uint64_t)j, 2);
        const int y = warp_draw(il, rl, u2, near);
        for (int i = j - 1 + lane; i <= G; i += 32) com[i] = i == j - 1 ? y : -1;
        if (lane == 0) {
            p.n_out[b] = j - 1;
            p.bonus_out[b] = y;
            if (p.near_out) p.near_out[b] = near;
        }
        return;
    }
    const FRow& P = rows[G];
    const int il = lane < P.n ? P.idx[lane] : -1;
    const float u3 = philox_uniform(seed, (uint64_t)b, (uint64_t)(G + 1), 3);
    const int y = warp_draw(il, lane < P.n ? P.pf[lane] : 0.0f, u3, near);
    if (lane == 0) {
        com[G] = y;
        p.n_out[b] = G;
        p.bonus_out[b] = y;
        if (p.near_out) p.near_out[b] = near;
    }
}

size_t verify_topk_workspace_bytes(int B, int gamma) {
    const size_t rows = (size_t)B * (2 * gamma + 1);
    return kWsHeaderBytes + rows * kTopkMax * sizeof(unsigned long long) + rows * sizeof(unsigned);
}

template <typename TT, typename DT>
static cudaError_t launch_rows(const TopkParams& p, bool vt, bool vd, cudaStream_t stream) {
    const long rows = (long)p.B * (2 * p.gamma + 1);
    topk_rows_kernel<TT, DT><<<(unsigned)rows, kTopkThreads, 0, stream>>>(p, vt, vd);
    return cudaGetLastError();
}

cudaError_t verify_topk_launch(TopkParams& p, void* ws, cudaStream_t stream) {
    char* w = static_cast<char*>(ws);
    p.status = &reinterpret_cast<WsHeader*>(w)->status;
    const size_t rows = (size_t)p.B * (2 * p.gamma + 1);
    p.keys = reinterpret_cast<unsigned long long*>(w + kWsHeaderBytes);
    p.bad = reinterpret_cast<unsigned*>(w + kWsHeaderBytes + rows * kTopkMax * sizeof(unsigned long long));
    const bool vt = ((size_t)p.V * (p.tdt == SPEC_BF16 ? 2 : 4)) % 16 == 0;
    const bool vd = ((size_t)p.V * (p.ddt == SPEC_BF16 ? 2 : 4)) % 16 == 0;
    cudaError_t e;
    if (p.tdt == SPEC_BF16 && p.ddt == SPEC_BF16) e = launch_rows<bf16_t, bf16_t>(p, vt, vd, stream);
    else if (p.tdt == SPEC_BF16) e = launch_rows<bf16_t, float>(p, vt, vd, stream);
    else if (p.ddt == SPEC_BF16) e = launch_rows<float, bf16_t>(p, vt, vd, stream);
    else e = launch_rows<float, float>(p, vt, vd, stream);
    if (e != cudaSuccess) return e;
    const size_t smem = (size_t)(2 * p.gamma + 1) * sizeof(FRow);
    e = cudaFuncSetAttribute(topk_accept_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    topk_accept_kernel<<<p.B, kTopkThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace spec
