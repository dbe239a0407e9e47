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
//   topk_rows_kernel   persistent CTAs stream the rows (target and draft rows in one
//                      grid), each row in at most 6 pieces on consecutive CTAs; the CTA
//                      that finishes a row's last piece merges the pieces.  Each warp keeps the 32 largest 64-bit keys it has
//                      seen (ordered value high, inverted index low: a larger key is a
//                      larger value or, on a tie, a lower index) as a sorted list spread
//                      over its lanes.  A lane looks inside its 8-entry groups only when a
//                      group's packed maximum reaches the threshold, the largest of the
//                      warp's k-th key, the CTA's best published bound and the best bound
//                      any CTA sharing the row has published through global memory (no
//                      entry below it can be among the row's k largest); the threshold starts
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

// Resident CTAs per SM the row kernel is built for: 4 with bf16 rows (two 64-byte item
// buffers per thread fit in 64 registers), 2 when either row type is float32.
template <typename TT, typename DT> struct TopkOcc {
    static constexpr int N = sizeof(TT) == 2 && sizeof(DT) == 2 ? 4 : 2;
};

// A relaxed load of the row's published bound (other CTAs raise it with atomicMax).
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// The CTA whose item range [c*I/G, (c+1)*I/G) holds item i.
__device__ __forceinline__ long topk_cta_of(long i, long I, long G) { return ((i + 1) * G - 1) / I; }

// Lane `e` (< 8) of the warp: entry e of lane L's 8-entry group j of the current item.
template <typename T, int NW>
__device__ __forceinline__ float group_entry(const uint4 (&w)[NW], int j, int L, int e) {
    if constexpr (sizeof(T) == 2) {
        const unsigned a0 = __shfl_sync(0xffffffffu, w[j].x, L), a1 = __shfl_sync(0xffffffffu, w[j].y, L);
        const unsigned a2 = __shfl_sync(0xffffffffu, w[j].z, L), a3 = __shfl_sync(0xffffffffu, w[j].w, L);
        const int h = (e >> 1) & 3;
        const unsigned a = h == 0 ? a0 : (h == 1 ? a1 : (h == 2 ? a2 : a3));
        return (e & 1) ? __uint_as_float(a & 0xffff0000u) : __uint_as_float(a << 16);
    } else {
        const uint4 lo = w[2 * j], hi = w[2 * j + 1];
        const unsigned b0 = __shfl_sync(0xffffffffu, lo.x, L), b1 = __shfl_sync(0xffffffffu, lo.y, L);
        const unsigned b2 = __shfl_sync(0xffffffffu, lo.z, L), b3 = __shfl_sync(0xffffffffu, lo.w, L);
        const unsigned b4 = __shfl_sync(0xffffffffu, hi.x, L), b5 = __shfl_sync(0xffffffffu, hi.y, L);
        const unsigned b6 = __shfl_sync(0xffffffffu, hi.z, L), b7 = __shfl_sync(0xffffffffu, hi.w, L);
        const int h = e & 7;
        const unsigned a = h < 4 ? (h == 0 ? b0 : (h == 1 ? b1 : (h == 2 ? b2 : b3)))
                                 : (h == 4 ? b4 : (h == 5 ? b5 : (h == 6 ? b6 : b7)));
        return __uint_as_float(a);
    }
}

// Keys of the descending list a[0..n) (distinct, 0 = empty) greater than `key`.
__device__ __forceinline__ int count_above(const unsigned long long* a, int n, unsigned long long key) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] > key) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// Chunks [c0, c1) of the row at `rowp` (global row `row`), streamed by the CTA: each warp
// takes its 1024-entry segment of every chunk and keeps the k largest keys it has seen
// as a sorted list over its lanes.  The piece's k largest go to slot `slot` of the row;
// the CTA that finishes the row's last piece (of `npieces`) merges them into keys[row].
template <typename T>
__device__ __forceinline__ void topk_piece(const TopkParams& p, const T* rowp, long V, bool vec, int c0, int c1,
                                           long row, int slot, int npieces) {
    constexpr int NW = Words<T>::N;
    __shared__ unsigned long long s_thr;                 // a key at or below the piece's k-th largest
    __shared__ unsigned long long s_mth[kTopkWarps];     // each warp's m-th largest key so far
    __shared__ float s_seed[kTopkWarps];                 // each warp's m-th largest lane maximum
    __shared__ unsigned long long s_all[kTopkThreads];   // the warps' lists, then the pieces' lists
    __shared__ int s_bad, s_last;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int k = p.k;
    const int m = (k + kTopkWarps - 1) / kTopkWarps;   // m keys from each of the 8 warps make k
    __syncthreads();   // the previous piece's readers of s_thr and s_all are done
    if (threadIdx.x == 0) { s_thr = 0ull; s_bad = 0; }
    if (threadIdx.x < kTopkWarps) s_mth[threadIdx.x] = 0ull;

    unsigned long long mine = 0ull;   // this lane's slot of the warp's sorted list
    unsigned long long kth = 0ull;    // the warp's k-th key (0 while the list is short)
    unsigned long long thr = 0ull;    // the key to beat: the larger of kth and the CTA's best
    float thr_v = -INFINITY;          // value threshold: entries below it are skipped
    int bad = 0;
    const int vi = (int)V;            // V < 2^31
    uint4 cur[NW], nxt[NW];
    load_words_il<T, NW>(cur, rowp, V, il_seg(c0), vec);
    unsigned long long mth = 0ull;   // the warp's m-th key, as last published
    // the row's bound from every piece (lane 0): requested one chunk ahead of its use,
    // and raised by this warp when its own bound passes it
    unsigned long long gthr = lane == 0 ? ld_relaxed_u64(&p.row_thr[row]) : 0ull;
    for (int c = c0; c < c1; ++c) {
        if (c + 1 < c1) {
            const long sg = il_seg(c + 1);
            if (vec && sg + 1024 <= V) load_words_il_full<T, NW>(nxt, rowp, sg);   // the whole segment in the row
            else load_words_il<T, NW>(nxt, rowp, V, sg, vec);
        }
        float g[4];   // the maxima of this lane's four 8-entry groups (NaN if any is NaN)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if constexpr (sizeof(T) == 2) g[j] = u4_max_nan<2>(cur[j]);
            else g[j] = f_max_nan(u4_max_nan<4>(cur[2 * j]), u4_max_nan<4>(cur[2 * j + 1]));
        }
        float lm = f_max_nan(f_max_nan(g[0], g[1]), f_max_nan(g[2], g[3]));
        if (isnan(lm) || lm == INFINITY) bad = 1;
        if (c == c0) {
            // seed: the k-th largest of the 32 lane maxima (each an entry of this item)
            float sm = lm;
#pragma unroll
            for (int kk = 2; kk <= 32; kk <<= 1)   // bitonic sort of the lane maxima, ascending
#pragma unroll
                for (int j = kk >> 1; j > 0; j >>= 1) {
                    const float o = __shfl_xor_sync(0xffffffffu, sm, j);
                    const bool take_max = ((lane & kk) == 0) != ((lane & j) == 0);
                    sm = take_max ? fmaxf(sm, o) : fminf(sm, o);
                }
            // a value with k entries of the item at or above it: this warp's k-th largest
            // lane maximum, or the smallest of the warps' m-th largest (m from each warp)
            const float own = __shfl_sync(0xffffffffu, sm, 32 - k);
            const float mw = __shfl_sync(0xffffffffu, sm, 32 - m);
            if (lane == 0) s_seed[warp] = mw;
            __syncthreads();
            float cta = s_seed[0];
#pragma unroll
            for (int w = 1; w < kTopkWarps; ++w) cta = fminf(cta, s_seed[w]);
            const float seed = fmaxf(own, cta);
            thr_v = isnan(seed) ? -INFINITY : seed;
        }
        // the CTA's best k-th key, read once and broadcast: every lane must see the same
        // threshold (the insertions below are warp-collective)
        unsigned long long st_l = 0ull;
        if (lane == 0) {
            st_l = *(volatile unsigned long long*)&s_thr;
            st_l = gthr > st_l ? gthr : st_l;
            gthr = ld_relaxed_u64(&p.row_thr[row]);   // for the next chunk
        }
        const unsigned long long shared_thr = shfl_u64(st_l, 0);
        if (shared_thr > thr) {
            thr = shared_thr;
            thr_v = fmaxf(thr_v, key_value(shared_thr));
        }
        if (__any_sync(0xffffffffu, !bad && lm >= thr_v)) {
            const int seg = (int)il_seg(c);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                // the lanes whose group j reaches the threshold, one group at a time: lanes
                // 0..7 take its entries, and the keys above the threshold are inserted
                unsigned hm = __ballot_sync(0xffffffffu, !bad && g[j] >= thr_v);
                while (hm) {
                    const int L = __ffs(hm) - 1;
                    hm &= hm - 1u;
                    const float x = group_entry<T, NW>(cur, j, L, lane);
                    const int e = seg + (j * 32 + L) * 8 + (lane & 7);
                    const unsigned long long key = argmax_key(x, (uint32_t)e);
                    unsigned cm = __ballot_sync(0xffffffffu, lane < 8 && e < vi && x >= thr_v && key > thr);
                    while (cm) {   // warp-uniform
                        const int s = __ffs(cm) - 1;
                        cm &= cm - 1u;
                        const unsigned long long ks = shfl_u64(key, s);
                        if (ks > thr) {
                            list_insert(mine, ks, k, kth);
                            if (kth > thr) {
                                thr = kth;
                                thr_v = fmaxf(thr_v, key_value(kth));
                            }
                        }
                    }
                }
            }
            // publish the warp's k-th key, and its m-th: the smallest of the warps' m-th
            // keys has at least k keys at or above it (each value stays valid: a list's
            // j-th key never falls)
            const unsigned long long mt = shfl_u64(mine, m - 1);
            if (lane == 0) {
                unsigned long long bound = kth;
                if (mt != mth) {
                    *(volatile unsigned long long*)&s_mth[warp] = mt;
                    unsigned long long lo = mt;
#pragma unroll
                    for (int w = 0; w < kTopkWarps; ++w) {
                        const unsigned long long v = *(volatile unsigned long long*)&s_mth[w];
                        lo = v < lo ? v : lo;
                    }
                    bound = lo > bound ? lo : bound;
                }
                if (bound > *(volatile unsigned long long*)&s_thr) atomicMax(&s_thr, bound);
                if (bound > gthr) atomicMax(&p.row_thr[row], bound);   // every piece of the row may use it
            }
            mth = mt;
        }
#pragma unroll
        for (int i = 0; i < NW; ++i) cur[i] = nxt[i];
    }
    if (bad) s_bad = 1;
    // the piece's k largest: only a warp's first k keys can be among them; rank each of
    // those among all of them (keys are distinct, the index being part of them, except
    // the empty key 0)
    const bool lane_k = lane < k;
    s_all[threadIdx.x] = lane_k ? mine : 0ull;
    __syncthreads();
    const size_t ps = (size_t)row * kTopkPieces + slot;
    unsigned long long* out = p.part + ps * kTopkMax;
    if (threadIdx.x < kTopkMax) out[threadIdx.x] = 0ull;
    __syncthreads();
    if (!s_bad && lane_k && mine != 0ull) {
        int rank = lane;   // the keys of this warp's list above this one
        for (int w = 0; w < kTopkWarps; ++w)
            if (w != warp) rank += count_above(s_all + w * 32, k, mine);
        if (rank < k) out[rank] = mine;
    }
    if (threadIdx.x == 0) p.part_bad[ps] = s_bad ? 1u : 0u;

    // the last piece of the row to finish merges the pieces' lists
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(&p.row_done[row], 1u) == (unsigned)npieces - 1u ? 1 : 0;
        if (s_last) __threadfence();
    }
    __syncthreads();
    if (!s_last) return;
    unsigned long long* kout = p.keys + (size_t)row * kTopkMax;
    const int q = threadIdx.x;   // kTopkThreads == kTopkPieces * kTopkMax
    const unsigned long long key =
        q / kTopkMax < npieces && q % kTopkMax < k ? __ldcg(&p.part[(size_t)row * kTopkPieces * kTopkMax + q]) : 0ull;
    const int pbad = q < npieces ? (int)__ldcg(&p.part_bad[(size_t)row * kTopkPieces + q]) : 0;
    s_all[q] = key;
    if (q < kTopkMax) kout[q] = 0ull;
    const int rowbad = __syncthreads_or(pbad);
    if (!rowbad && key != 0ull) {
        int rank = q % kTopkMax;   // the keys of this piece's list above this one
        for (int w = 0; w < npieces; ++w)
            if (w != q / kTopkMax) rank += count_above(s_all + w * kTopkMax, k, key);
        if (rank < k) kout[rank] = key;
    }
    if (q == 0) {
        p.bad[row] = rowbad ? 1u : 0u;
        p.row_done[row] = 0u;
        p.row_thr[row] = 0ull;   // every other piece of the row has finished reading it
    }
}

// Items (row, chunk of 8192 entries) of the target rows 0 .. nT-1, then of the draft
// rows; CTA c streams items [c*I/G, (c+1)*I/G), at least a quarter of a row, so that a
// row is split over at most 6 CTAs.
template <typename T>
__device__ __forceinline__ void topk_range(const TopkParams& p, const T* base, bool vec, long a, long b, long row0,
                                           long nch, long I) {
    const long G = gridDim.x;
    for (long it = a; it < b;) {
        const long row = it / nch;
        const long end = b < (row + 1) * nch ? b : (row + 1) * nch;
        const long cf = topk_cta_of(row * nch, I, G), cl = topk_cta_of((row + 1) * nch - 1, I, G);
        topk_piece<T>(p, base + (size_t)(row - row0) * p.V, p.V, vec, (int)(it - row * nch), (int)(end - row * nch),
                      row, (int)(blockIdx.x - cf), (int)(cl - cf + 1));
        it = end;
    }
}

template <typename TT, typename DT>
__global__ void __launch_bounds__(kTopkThreads, TopkOcc<TT, DT>::N) topk_rows_kernel(TopkParams p, bool vt, bool vd) {
    static_assert(kTopkThreads == kTopkPieces * kTopkMax, "merge layout");
    const long nch = ((long)p.V + kVerifyChunk - 1) / kVerifyChunk;
    const long nT = (long)p.B * (p.gamma + 1);
    const long I = (long)p.B * (2 * p.gamma + 1) * nch;
    const long G = gridDim.x;
    const long i0 = (long)blockIdx.x * I / G, i1 = ((long)blockIdx.x + 1) * I / G;
    const long tend = nT * nch;
    if (i0 < tend) topk_range<TT>(p, static_cast<const TT*>(p.target), vt, i0, i1 < tend ? i1 : tend, 0, nch, I);
    if (i1 > tend) topk_range<DT>(p, static_cast<const DT*>(p.draft), vd, i0 > tend ? i0 : tend, i1, nT, nch, I);
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

static size_t topk_align(size_t x) { return (x + 255) / 256 * 256; }

size_t verify_topk_workspace_bytes(int B, int gamma) {
    const size_t rows = (size_t)B * (2 * gamma + 1);
    size_t off = kWsHeaderBytes;
    off = topk_align(off + rows * kTopkMax * sizeof(unsigned long long));                 // keys
    off = topk_align(off + rows * sizeof(unsigned));                                      // bad
    off = topk_align(off + rows * kTopkPieces * kTopkMax * sizeof(unsigned long long));   // part
    off = topk_align(off + rows * kTopkPieces * sizeof(unsigned));                        // part_bad
    off = topk_align(off + rows * sizeof(unsigned));                                      // row_done
    return topk_align(off + rows * sizeof(unsigned long long));                           // row_thr
}

template <typename TT, typename DT>
static cudaError_t launch_rows(const TopkParams& p, bool vt, bool vd, cudaStream_t stream) {
    void (*k)(TopkParams, bool, bool) = topk_rows_kernel<TT, DT>;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kTopkThreads, 0) != cudaSuccess || occ < 1) occ = 1;
    const long nch = ((long)p.V + kVerifyChunk - 1) / kVerifyChunk;
    const long I = (long)p.B * (2 * p.gamma + 1) * nch;
    const long per_min = (nch + 3) / 4;   // a CTA takes at least a quarter of a row
    long grid = (long)device_sm_count() * occ;
    if (grid > I / per_min) grid = I / per_min;
    if (grid < 1) grid = 1;
    k<<<(unsigned)grid, kTopkThreads, 0, stream>>>(p, vt, vd);
    return cudaGetLastError();
}

cudaError_t verify_topk_launch(TopkParams& p, void* ws, cudaStream_t stream) {
    char* w = static_cast<char*>(ws);
    p.status = &reinterpret_cast<WsHeader*>(w)->status;
    const size_t rows = (size_t)p.B * (2 * p.gamma + 1);
    size_t off = kWsHeaderBytes;
    p.keys = reinterpret_cast<unsigned long long*>(w + off);
    off = topk_align(off + rows * kTopkMax * sizeof(unsigned long long));
    p.bad = reinterpret_cast<unsigned*>(w + off);
    off = topk_align(off + rows * sizeof(unsigned));
    p.part = reinterpret_cast<unsigned long long*>(w + off);
    off = topk_align(off + rows * kTopkPieces * kTopkMax * sizeof(unsigned long long));
    p.part_bad = reinterpret_cast<unsigned*>(w + off);
    off = topk_align(off + rows * kTopkPieces * sizeof(unsigned));
    p.row_done = reinterpret_cast<unsigned*>(w + off);
    off = topk_align(off + rows * sizeof(unsigned));
    p.row_thr = reinterpret_cast<unsigned long long*>(w + off);
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
