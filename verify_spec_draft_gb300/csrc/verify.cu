// verify.cu - target verification of a draft block (spec_verify).
//
// Defines: "Solar Open2 DSpark" (sionic.ai), sections 1 and 6 - one target forward
// over gamma+1 positions checks the drafts and commits the agreeing prefix;
// "Speculative Decoding Part 2" (VESSL AI), blockwise decoding section - the longest
// matching prefix is accepted.  T=1 is standard rejection sampling with a residual or
// bonus draw (the pages' overlap 1 - TV is its acceptance probability).
//
// Design (HBM-bound; every row streamed once):
//   Work items are (row, 8192-entry chunk); a persistent grid walks them with the next
//   item's 16-byte loads in flight while the current one is reduced (register double
//   buffering), each thread holding 32 contiguous entries.
//   T=0  one kernel.  Each warp folds its entries into a 64-bit argmax key (value,
//        lowest index) and merges it with one atomicMax per row.  The last CTA to
//        finish ("last CTA done" counter, no waiting) scans every request's prefix,
//        one warp per request, and writes the outputs.
//   T=1  one cooperative kernel in four phases separated by bounded grid barriers:
//        (1) base-2 softmax statistics of every target and draft row, one partial per
//        1024-entry warp segment; (2) per request, merge its rows in order while the
//        request's uniforms are drawn, run the gamma accept tests in parallel, record
//        the row to sample from; (3) re-read that row pair (residual) or row (bonus)
//        for its weight per segment in vocabulary order; (4) one CTA per request
//        locates the segment holding u * sum and the entry inside it.  No counters or
//        fences in the streaming phase.
#include "spec_device.cuh"
#include "internal.h"
#include "chunk_rows.cuh"

namespace spec {

enum { MODE_DONE = 0, MODE_RESID = 1, MODE_BONUS = 2 };

__device__ __forceinline__ long thread_base(int c) {
    return (long)c * kVerifyChunk + (long)threadIdx.x * kEPT;
}

// ----------------------------------------------------------------------------------
// T = 0
// ----------------------------------------------------------------------------------
// T=0 runs 256-thread CTAs on 8192-entry items, as many CTAs as fit.
constexpr int kT0Threads = 256;
constexpr int kT0Warps = kT0Threads / 32;
constexpr int kT0Chunk = kT0Threads * kEPT;

__device__ __forceinline__ long t0_base(int c) { return (long)c * kT0Chunk + (long)threadIdx.x * kEPT; }

template <typename TT>
__global__ void __launch_bounds__(kT0Threads) verify_t0_kernel(VerifyParams p) {
    // Launched with programmatic stream serialization, this grid may start before the
    // previous kernel on the stream has finished.  Standalone, that kernel may be the
    // producer of the target rows or the tokens, so wait for it before reading anything;
    // as the dependent of the library's own draft kernel, only the tokens come from it
    // (waited for before the final scan).
    if (!p.after_own_draft) pdl_wait_primary();
    const TT* target = static_cast<const TT*>(p.target);
    const long V = p.V;
    const unsigned nch = (unsigned)((V + kT0Chunk - 1) / kT0Chunk);
    const long items = (long)p.B * (p.gamma + 1) * nch;
    const bool vec = p.vec_t != 0;
    constexpr int NW = Words<TT>::N;
    uint4 cur[NW], nxt[NW];
    __shared__ unsigned long long s_key[2][kT0Warps];
    int par = 0;

    long it = blockIdx.x;
    auto split = [&](long i, int& row, int& c) {   // 32-bit division where the index fits
        if (i <= 0xffffffffL) { row = (int)((unsigned)i / nch); c = (int)((unsigned)i - (unsigned)row * nch); }
        else { row = (int)(i / nch); c = (int)(i - (long)row * nch); }
    };
    if (it < items) {
        int row, c;
        split(it, row, c);
        load_words<TT, NW>(cur, target + (size_t)row * V, V, t0_base(c), vec);
    }
    for (; it < items; it += gridDim.x) {
        const long nx = it + gridDim.x;
        if (nx < items) {
            int rn, cn;
            split(nx, rn, cn);
            load_words<TT, NW>(nxt, target + (size_t)rn * V, V, t0_base(cn), vec);
        }
        int row, c;
        split(it, row, c);
        // NaN-propagating max of the 32 entries (-inf pads the row end), then the
        // warp max; only lanes holding it look for their lowest index
        const float lm = chunk_max_nan<TT, NW>(cur);
        const float m = warp_max_nan(lm);
        const int bad = (isnan(m) || m == INFINITY) ? 1 : 0;
        int idx = 0x7fffffff;
        if (!bad && lm == m) {
            const int k = first_equal<TT, NW>(cur, m);
            if (k >= 0) idx = (int)(t0_base(c) + k);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) idx = min(idx, __shfl_xor_sync(0xffffffffu, idx, o));
        // one atomic per CTA and item: warps post their keys, thread 0 folds them
        // (slots alternate with the item parity, so one barrier per item suffices)
        if ((threadIdx.x & 31) == 0)
            s_key[par][threadIdx.x >> 5] = bad ? ~0ull : argmax_key(m, (uint32_t)idx);
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned long long k = 0ull;
            int anybad = 0;
            for (int w = 0; w < kT0Warps; ++w) {
                const unsigned long long kw = s_key[par][w];
                if (kw == ~0ull) anybad = 1;
                else k = kw > k ? kw : k;
            }
            if (anybad) atomicOr(&p.rowbad[row], 1u);
            else atomicMax(&p.keys[row], k);
        }
        par ^= 1;
#pragma unroll
        for (int i = 0; i < NW; ++i) cur[i] = nxt[i];
    }

    if (!last_block_done(&p.done[0], gridDim.x)) return;
    if (p.after_own_draft) pdl_wait_primary();   // the draft tokens come from the kernel this one overlaps

    // prefix scan: one warp per request, one lane per row
    const int G = p.gamma;
    const int lane = threadIdx.x & 31;
    for (int b = threadIdx.x >> 5; b < p.B; b += kT0Warps) {
        unsigned long long k3[3] = {0ull, 0ull, 0ull};
        int tok3[3] = {0, 0, 0};
        unsigned bad_row = 0, bad_tok = 0, mism[3] = {0u, 0u, 0u};
#pragma unroll
        for (int h = 0; h < 3; ++h) {
            const int i = lane + 32 * h;
            bool rb = false, tb = false, mm = false;
            if (i <= G) {
                const int row = b * (G + 1) + i;
                k3[h] = __ldcg(&p.keys[row]);
                rb = __ldcg(&p.rowbad[row]) != 0u || key_value(k3[h]) == -INFINITY;
                p.keys[row] = 0ull;
                p.rowbad[row] = 0u;
                if (i < G) {
                    tok3[h] = p.tokens[(size_t)b * G + i];
                    tb = tok3[h] < 0 || tok3[h] >= p.V;
                    mm = tok3[h] != (int)key_index(k3[h]);
                }
            }
            bad_row |= __ballot_sync(0xffffffffu, rb);
            bad_tok |= __ballot_sync(0xffffffffu, tb);
            mism[h] = __ballot_sync(0xffffffffu, mm);
        }
        int n = G;
        for (int h = 2; h >= 0; --h)
            if (mism[h]) n = 32 * h + __ffs(mism[h]) - 1;
        const unsigned long long kn =
            __shfl_sync(0xffffffffu, n < 32 ? k3[0] : (n < 64 ? k3[1] : k3[2]), n & 31);
        const int y = (int)key_index(kn);
        int32_t* com = p.committed_out + (size_t)b * (G + 1);
        const bool invalid = bad_row || bad_tok;
#pragma unroll
        for (int h = 0; h < 3; ++h) {
            const int i = lane + 32 * h;
            if (i <= G) com[i] = invalid ? -1 : (i < n ? tok3[h] : (i == n ? y : -1));
        }
        if (lane == 0) {
            if (invalid) atomicOr(p.status, (bad_tok ? SPEC_DEV_TOKEN : 0u) | (bad_row ? SPEC_DEV_NONFINITE : 0u));
            p.n_out[b] = invalid ? -1 : n;
            p.bonus_out[b] = invalid ? -1 : y;
            if (p.near_out) p.near_out[b] = 0;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) p.done[0] = 0u;
}

// ----------------------------------------------------------------------------------
// T = 1: one cooperative kernel, four phases separated by bounded grid barriers
//   1  base-2 softmax statistics of every target and draft row, one partial per
//      (row, chunk, warp): (m2, s) with s = sum 2^(x log2e - m2), m2 = NaN if bad
//   2  one CTA per request: merge its rows, run the gamma accept tests, record the
//      row to draw from (residual at the first rejection, or the bonus row)
//   3  weights of those rows per (request, chunk, warp), in vocabulary order
//   4  one CTA per request: locate the 1024-entry segment holding u * sum, then the
//      entry inside it
// ----------------------------------------------------------------------------------
struct Item1 { int b, lr, c; };   // local rows 0..G target, G+1..2G draft
__device__ __forceinline__ Item1 item1(const VerifyParams& p, long it) {
    const unsigned per_req = (unsigned)(2 * p.gamma + 1) * (unsigned)p.nchunk;   // < 2^21
    Item1 r;
    unsigned rem;
    if (it <= 0xffffffffL) {   // 32-bit division where the index fits
        const unsigned u = (unsigned)it;
        r.b = (int)(u / per_req);
        rem = u - (unsigned)r.b * per_req;
    } else {
        r.b = (int)(it / (long)per_req);
        rem = (unsigned)(it - (long)r.b * per_req);
    }
    r.lr = (int)(rem / (unsigned)p.nchunk);
    r.c = (int)(rem - (unsigned)r.lr * (unsigned)p.nchunk);
    return r;
}

template <typename TT, typename DT, int NW>
__device__ __forceinline__ void load_item1(const VerifyParams& p, long it, uint4 (&w)[NW]) {
    const Item1 q = item1(p, it);
    const int G = p.gamma;
    if (q.lr <= G)
        load_words<TT, NW>(w, static_cast<const TT*>(p.target) + ((size_t)q.b * (G + 1) + q.lr) * p.V, p.V,
                           thread_base(q.c), p.vec_t != 0);
    else
        load_words<DT, NW>(w, static_cast<const DT*>(p.draft) + ((size_t)q.b * G + (q.lr - G - 1)) * p.V, p.V,
                           thread_base(q.c), p.vec_d != 0);
}

template <typename T, int NW>
__device__ __forceinline__ float2 warp_partial(const uint4 (&w)[NW]) {
    const float m = warp_max_nan(chunk_max_nan<T, NW>(w));
    if (isnan(m) || m == INFINITY) return make_float2(NAN, 0.0f);
    if (m == -INFINITY) return make_float2(-INFINITY, 0.0f);
    const float m2 = m * kLog2e;
    float x[kEPT];
    decode_words<T, NW>(w, x);
    float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
    for (int e = 0; e < kEPT; e += 2) { s0 += wexp(x[e], m2); s1 += wexp(x[e + 1], m2); }
    return make_float2(m2, warp_sum(s0 + s1));
}

template <typename TT, typename DT>
__device__ __forceinline__ void phase_stats(const VerifyParams& p) {
    const long items = (long)(2 * p.gamma + 1) * p.nchunk * p.B;
    constexpr int NW = Words<TT>::N > Words<DT>::N ? Words<TT>::N : Words<DT>::N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint4 cur[NW], nxt[NW];
    long it = blockIdx.x;
    if (it < items) load_item1<TT, DT, NW>(p, it, cur);
    for (; it < items; it += gridDim.x) {
        const long nx = it + gridDim.x;
        if (nx < items) load_item1<TT, DT, NW>(p, nx, nxt);
        const Item1 q = item1(p, it);
        const float2 st = (q.lr <= p.gamma) ? warp_partial<TT, NW>(cur) : warp_partial<DT, NW>(cur);
        if (lane == 0) {
            const size_t rowid = (size_t)q.b * (2 * p.gamma + 1) + q.lr;
            p.stats[(rowid * p.nchunk + q.c) * kWarps + warp] = st;
        }
#pragma unroll
        for (int i = 0; i < NW; ++i) cur[i] = nxt[i];
    }
}

// Phase 1 with the rows staged by bulk copies (rows 16-byte aligned): each CTA keeps
// S chunk copies in flight in a shared-memory ring, one mbarrier per stage; the 8
// warps reduce their 1024-entry segments of a stage into the same per-(row, chunk,
// warp) partials as phase_stats, then thread 0 refills the stage with the CTA's item
// S further on.  Bytes in flight per SM no longer depend on registers.
constexpr int kV1StagesBf16 = 4;   // 16 KB stages; with float32 rows, 2 stages of 32 KB
constexpr unsigned long long kV1WaitNs = kWaitLimitNs;
// ring layout: full and empty mbarriers, the staged items' (b, row, chunk, entries),
// then the stages (128-byte aligned)
constexpr int kV1RingOffset = 256;
static_assert(2 * 8 * kV1StagesBf16 + 16 * kV1StagesBf16 <= kV1RingOffset, "ring header");


template <typename TT, typename DT>
__device__ __forceinline__ void issue_item1(const VerifyParams& p, long it, uint8_t* dst, uint64_t* bar,
                                            int4* slot, uint64_t pol) {
    const Item1 q = item1(p, it);
    const int G = p.gamma;
    const long e0 = (long)q.c * kVerifyChunk;
    const long n = (long)p.V - e0 < kVerifyChunk ? (long)p.V - e0 : kVerifyChunk;
    const void* src;
    unsigned bytes;
    if (q.lr <= G) {
        src = static_cast<const TT*>(p.target) + ((size_t)q.b * (G + 1) + q.lr) * p.V + e0;
        bytes = (unsigned)(n * (long)sizeof(TT));
    } else {
        src = static_cast<const DT*>(p.draft) + ((size_t)q.b * G + (q.lr - G - 1)) * p.V + e0;
        bytes = (unsigned)(n * (long)sizeof(DT));
    }
    *slot = make_int4(q.b, q.lr, q.c, (int)n);   // published to the consumers by the barrier phase
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s_hint(dst, src, bytes, bar, pol);   // each chunk is read once here
}

// This warp's 1024-entry segment of a staged chunk as 32 entries per lane (lane-
// interleaved 16-byte words, so a warp's shared loads hit distinct banks), -inf past
// the `nvalid` entries the chunk holds.
template <typename T, int NW>
__device__ __forceinline__ void stage_words(const uint8_t* stage, int warp, int lane, int nvalid, uint4 (&w)[NW]) {
    constexpr int EPV = 16 / (int)sizeof(T);
    constexpr int WPS = 1024 / EPV;   // 16-byte words per warp segment
    const uint4* seg = reinterpret_cast<const uint4*>(stage) + (size_t)warp * WPS;
    const uint32_t ninf = sizeof(T) == 2 ? 0xff80ff80u : 0xff800000u;
#pragma unroll
    for (int j = 0; j < Words<T>::N; ++j) {
        const int u = j * 32 + lane;
        w[j] = (warp * 1024 + u * EPV + EPV <= nvalid) ? seg[u] : make_uint4(ninf, ninf, ninf, ninf);
    }
}

template <typename TT, typename DT>
__device__ __forceinline__ void phase_stats_staged(const VerifyParams& p, uint8_t* ring, uint64_t* full,
                                                   uint64_t* empty, int4* s_item, int S, size_t stage_bytes) {

    const long items = (long)(2 * p.gamma + 1) * p.nchunk * p.B;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long mine = items > (long)blockIdx.x ? (items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const uint64_t pol = l2_evict_first_policy();
    if (threadIdx.x == 0)
        for (long k = 0; k < S && k < mine; ++k)
            issue_item1<TT, DT>(p, blockIdx.x + k * gridDim.x, ring + (size_t)k * stage_bytes, &full[k], &s_item[k],
                                pol);
    for (long k = 0; k < mine; ++k) {
        const int s = (int)(k % S);
        if (threadIdx.x == 0 && k >= 1 && k - 1 + S < mine) {
            // refill the stage of item k-1 with item k-1+S once every warp has left it
            const int sp = (int)((k - 1) % S);
            mbar_wait(&empty[sp], (unsigned)(((k - 1) / S) & 1), p.status, kV1WaitNs);
            fence_proxy_async_smem();
            issue_item1<TT, DT>(p, blockIdx.x + (k - 1 + S) * gridDim.x, ring + (size_t)sp * stage_bytes, &full[sp],
                                &s_item[sp], pol);
        }
        const uint8_t* stage = ring + (size_t)s * stage_bytes;
        mbar_wait(&full[s], (unsigned)((k / S) & 1), p.status, kV1WaitNs);
        const int4 qi = s_item[s];
        const Item1 q{qi.x, qi.y, qi.z};
        const int nvalid = qi.w;
        float2 st;
        if (q.lr <= p.gamma) {
            uint4 w[Words<TT>::N];
            stage_words<TT>(stage, warp, lane, nvalid, w);
            st = warp_partial<TT, Words<TT>::N>(w);
        } else {
            uint4 w[Words<DT>::N];
            stage_words<DT>(stage, warp, lane, nvalid, w);
            st = warp_partial<DT, Words<DT>::N>(w);
        }
        __syncwarp();
        if (lane == 0) {
            const size_t rowid = (size_t)q.b * (2 * p.gamma + 1) + q.lr;
            p.stats[(rowid * p.nchunk + q.c) * kWarps + warp] = st;
            mbar_arrive1(&empty[s]);   // this warp is done with stage s
        }
    }
    // no copy may still be landing in this CTA's shared memory when it leaves the phase:
    // thread 0 waits (bounded) on the phase of the last item issued into each stage
    // (already complete, unless a wait above ran out)
    if (threadIdx.x == 0)
        for (int s = 0; s < S && s < mine; ++s) {
            const long last = s + (mine - 1 - s) / S * S;
            mbar_wait(&full[s], (unsigned)((last / S) & 1), p.status, kV1WaitNs);
        }
}

// What the accept test of request b reads besides the row statistics: its draft tokens
// and the target and draft logits at them, loaded by the CTA that tests request b
// right after its streaming phase, so the two dependent round trips overlap the wait
// at the grid barrier (threads 64.., one per position); and the request's uniforms,
// which depend on no data: drawn at kernel start (threads 32..32+2G) while the first
// copies are in flight.  u[j] is the accept test of position j+1 (stream 1), u[G+j]
// the residual draw at position j+1 (stream 2), u[2G] the bonus draw (stream 3).
struct AcceptInputs {
    int tok[SPEC_MAX_GAMMA];
    float lt[SPEC_MAX_GAMMA], ld[SPEC_MAX_GAMMA];
    float u[2 * SPEC_MAX_GAMMA + 1];
};
__device__ __forceinline__ void accept_uniforms(const VerifyParams& p, int b, AcceptInputs& ai) {
    const int G = p.gamma;
    const int t = (int)threadIdx.x - 32;
    if (t < 0 || t > 2 * G) return;
    const int pos = t < G ? t + 1 : (t < 2 * G ? t - G + 1 : G + 1);
    const int stream = t < G ? 1 : (t < 2 * G ? 2 : 3);
    ai.u[t] = philox_uniform(p.seeds[b], (uint64_t)b, (uint64_t)pos, (uint64_t)stream);
}
template <typename TT, typename DT>
__device__ __forceinline__ void load_accept_inputs(const VerifyParams& p, int b, AcceptInputs& ai) {
    const int G = p.gamma;
    const int j = (int)threadIdx.x - 64;
    if (j < 0 || j >= G) return;
    const int t = p.tokens[(size_t)b * G + j];
    ai.tok[j] = t;
    if (t >= 0 && t < p.V) {
        ai.lt[j] = to_float(static_cast<const TT*>(p.target)[((size_t)b * (G + 1) + j) * p.V + t]);
        ai.ld[j] = to_float(static_cast<const DT*>(p.draft)[((size_t)b * G + j) * p.V + t]);
    }
}

template <typename TT, typename DT>
__device__ __noinline__ void accept_phase(const VerifyParams& p, int b, const AcceptInputs* pre) {
    const TT* target = static_cast<const TT*>(p.target);
    const DT* draft = static_cast<const DT*>(p.draft);
    const int G = p.gamma;
    const int nr = 2 * G + 1;
    __shared__ float s_m2[2 * SPEC_MAX_GAMMA + 1], s_s[2 * SPEC_MAX_GAMMA + 1];
    __shared__ int s_badrow, s_badtok;
    __shared__ int s_acc[SPEC_MAX_GAMMA], s_near[SPEC_MAX_GAMMA];
    // the request's uniforms (as AcceptInputs::u), drawn here unless `pre` has them
    __shared__ float s_u[2 * SPEC_MAX_GAMMA + 1];
    __shared__ int s_k;
    const float* U = pre ? pre->u : s_u;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) { s_badrow = 0; s_badtok = 0; }
    __syncthreads();

    // each row's partials: the maximum first, then every partial's sum rescaled to it
    // (independent exponentials, no chain of pairwise merges); a warp takes two rows
    // with all their loads in flight.  NaN in a partial marks a row without a
    // distribution.
    const int np = p.nchunk * p.parts;
    for (int lr0 = warp; lr0 < nr; lr0 += 2 * kWarps) {
        float2 v[2][8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int lr = lr0 + h * kWarps;
            const size_t rowid = (size_t)b * nr + (lr < nr ? lr : 0);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = lane + 32 * u;
                v[h][u] = (lr < nr && i < np) ? __ldcg(&p.stats[rowid * np + i]) : make_float2(-INFINITY, 0.0f);
            }
        }
        // without `pre`, the Philox draws are computed while the loads are in flight
        // (threads 0..2G lie in warps below nr, which all run this first iteration)
        if (!pre && lr0 == warp && (int)threadIdx.x < nr) {
            const int t = threadIdx.x;
            const int pos = t < G ? t + 1 : (t < 2 * G ? t - G + 1 : G + 1);
            const int stream = t < G ? 1 : (t < 2 * G ? 2 : 3);
            s_u[t] = philox_uniform(p.seeds[b], (uint64_t)b, (uint64_t)pos, (uint64_t)stream);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int lr = lr0 + h * kWarps;
            const size_t rowid = (size_t)b * nr + (lr < nr ? lr : 0);
            float M = -INFINITY;
            int bad = 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (isnan(v[h][u].x)) bad = 1;
                else M = fmaxf(M, v[h][u].x);
            }
            for (int i = lane + 256; i < np; i += 32) {
                const float2 w = __ldcg(&p.stats[rowid * np + i]);
                if (isnan(w.x)) bad = 1;
                else M = fmaxf(M, w.x);
            }
            M = warp_max(M);
            float sum = 0.0f;
            if (M != -INFINITY) {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (!isnan(v[h][u].x) && v[h][u].x != -INFINITY) sum += v[h][u].y * ex2(v[h][u].x - M);
                for (int i = lane + 256; i < np; i += 32) {
                    const float2 w = __ldcg(&p.stats[rowid * np + i]);
                    if (!isnan(w.x) && w.x != -INFINITY) sum += w.y * ex2(w.x - M);
                }
            }
            sum = warp_sum(sum);
            bad = warp_or(bad);
            if (lane == 0 && lr < nr) {
                s_m2[lr] = M;
                s_s[lr] = sum;
                if (bad || M == -INFINITY) atomicOr(&s_badrow, 1);
            }
        }
    }
    __syncthreads();

    // the gamma accept tests, one thread each; p and q of the drafted token with the
    // accurate exp2 (the decision is compared against exact arithmetic)
    for (int j = threadIdx.x; j < G; j += blockDim.x) {
        const int t = pre ? pre->tok[j] : p.tokens[(size_t)b * G + j];
        int acc = 0, near = 0;
        if (t < 0 || t >= p.V) {
            atomicOr(&s_badtok, 1);
        } else {
            const float lp = pre ? pre->lt[j] : to_float(target[((size_t)b * (G + 1) + j) * p.V + t]);
            const float lq = pre ? pre->ld[j] : to_float(draft[((size_t)b * G + j) * p.V + t]);
            const float pj = exp2f(fmaf(lp, kLog2e, -s_m2[j])) / s_s[j];
            const float qj = exp2f(fmaf(lq, kLog2e, -s_m2[G + 1 + j])) / s_s[G + 1 + j];
            const float u = U[j];
            acc = (u * qj < pj) ? 1 : 0;
            near = (fabsf(u * qj - pj) < kNearTie * qj) ? 1 : 0;
        }
        s_acc[j] = acc;
        s_near[j] = near;
    }
    __syncthreads();

    // the outcome (thread 0): k accepted, or -1 for a request without a valid row or
    // token; then the committed tokens, one thread per position (position k gets the
    // draw later)
    if (threadIdx.x == 0) {
        int4 st0 = make_int4(MODE_DONE, -1, 0, 0);
        int4 st1 = make_int4(0, 0, 0, 0);
        int k = -1;
        if (s_badrow || s_badtok) {
            atomicOr(p.status, (s_badtok ? SPEC_DEV_TOKEN : 0u) | (s_badrow ? SPEC_DEV_NONFINITE : 0u));
            p.n_out[b] = -1;
            p.bonus_out[b] = -1;
            if (p.near_out) p.near_out[b] = 0;
        } else {
            int near = 0;
            k = 0;
            while (k < G && s_acc[k]) { near |= s_near[k]; ++k; }
            if (k < G) near |= s_near[k];
            if (k < G) {   // rejected at position k+1: target row k and draft row k
                st0 = make_int4(MODE_RESID, k, near, __float_as_int(U[G + k]));
                st1 = make_int4(__float_as_int(s_m2[k]), __float_as_int(s_s[k]),
                                __float_as_int(s_m2[G + 1 + k]), __float_as_int(s_s[G + 1 + k]));
            } else {       // all accepted: bonus from target row gamma
                st0 = make_int4(MODE_BONUS, G, near, __float_as_int(U[2 * G]));
                st1 = make_int4(__float_as_int(s_m2[G]), __float_as_int(s_s[G]), 0, 0);
            }
        }
        p.state[2 * b] = st0;
        p.state[2 * b + 1] = st1;
        s_k = k;
    }
    __syncthreads();
    const int k = s_k;
    int32_t* com = p.committed_out + (size_t)b * (G + 1);
    for (int i = threadIdx.x; i <= G; i += blockDim.x) {
        if (k < 0 || i > k) com[i] = -1;
        else if (i < k) com[i] = pre ? pre->tok[i] : p.tokens[(size_t)b * G + i];
    }
    __syncthreads();
}

struct DrawRow {   // what the accept phase recorded for a request
    int mode, n, near;
    float u;       // the draw's uniform
    float m2p, sp, m2q, sq;
};
__device__ __forceinline__ DrawRow draw_row(const VerifyParams& p, int b) {
    const int4 a = __ldcg(&p.state[2 * b]);
    const int4 c = __ldcg(&p.state[2 * b + 1]);
    return DrawRow{a.x, a.y, a.z, __int_as_float(a.w),
                   __int_as_float(c.x), __int_as_float(c.y), __int_as_float(c.z), __int_as_float(c.w)};
}

// Weights of 32 entries, summed in order: wr = max(0, p - q) (residual mode only) and
// wp = p, with p = 2^(l log2e - m2p) / sp and q = 2^(d log2e - m2q) / sq.  The draw
// recomputes the entries of one segment with this same per-entry arithmetic.
template <typename TT, typename DT, int NW>
__device__ __forceinline__ void weight_sums(const DrawRow& d, const uint4 (&wt)[NW], const uint4 (&wd)[NW],
                                            float& sr, float& sp) {
    float lt[kEPT];
    decode_words<TT, NW>(wt, lt);
    const float ip = 1.0f / d.sp;
    sr = 0.0f;
    sp = 0.0f;
    if (d.mode == MODE_RESID) {
        float ld[kEPT];
        decode_words<DT, NW>(wd, ld);
        const float iq = 1.0f / d.sq;
#pragma unroll
        for (int e = 0; e < kEPT; ++e) {
            const float pv = wexp(lt[e], d.m2p) * ip;
            const float qv = wexp(ld[e], d.m2q) * iq;
            sp += pv;
            sr += fmaxf(0.0f, pv - qv);
        }
    } else {
#pragma unroll
        for (int e = 0; e < kEPT; ++e) sp += wexp(lt[e], d.m2p) * ip;
    }
}

template <typename TT, typename DT, int NW>
__device__ __forceinline__ void load_draw(const VerifyParams& p, int b, long base, const DrawRow& d,
                                          uint4 (&wt)[NW], uint4 (&wd)[NW]) {
    const int G = p.gamma;
    load_words<TT, NW>(wt, static_cast<const TT*>(p.target) + ((size_t)b * (G + 1) + d.n) * p.V, p.V, base,
                       p.vec_t != 0);
    if (d.mode == MODE_RESID)
        load_words<DT, NW>(wd, static_cast<const DT*>(p.draft) + ((size_t)b * G + d.n) * p.V, p.V, base,
                           p.vec_d != 0);
}

template <typename TT, typename DT>
__device__ __forceinline__ void phase_weights(const VerifyParams& p) {
    const long items = (long)p.B * p.nchunk;
    constexpr int NW = Words<TT>::N > Words<DT>::N ? Words<TT>::N : Words<DT>::N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint4 ct[NW], cd[NW], nt[NW], nd[NW];
    DrawRow dc{MODE_DONE, 0, 0, 0.f, 0.f, 0.f, 0.f, 0.f}, dn = dc;
    // items = B * nchunk < 2^31 (B <= 65535, nchunk <= 8192): 32-bit index math
    const unsigned nch = (unsigned)p.nchunk;
    unsigned it = blockIdx.x;
    if ((long)it < items) {
        const int b = (int)(it / nch);
        dc = draw_row(p, b);
        if (dc.mode != MODE_DONE) load_draw<TT, DT, NW>(p, b, thread_base((int)(it - (unsigned)b * nch)), dc, ct, cd);
    }
    for (; (long)it < items; it += gridDim.x) {
        const unsigned nx = it + gridDim.x;
        if ((long)nx < items) {
            const int bn = (int)(nx / nch);
            dn = draw_row(p, bn);
            if (dn.mode != MODE_DONE)
                load_draw<TT, DT, NW>(p, bn, thread_base((int)(nx - (unsigned)bn * nch)), dn, nt, nd);
        }
        if (dc.mode != MODE_DONE) {
            const int b = (int)(it / nch);
            const int c = (int)(it - (unsigned)b * nch);
            float sr, sp;
            weight_sums<TT, DT, NW>(dc, ct, cd, sr, sp);
            const float ir = warp_inclusive_scan(sr), ip = warp_inclusive_scan(sp);
            if (lane == 31) p.ksums[((size_t)b * p.nchunk + c) * kWarps + warp] = make_float2(ir, ip);
        }
        dc = dn;
#pragma unroll
        for (int i = 0; i < NW; ++i) { ct[i] = nt[i]; cd[i] = nd[i]; }
    }
}

// Phase 3 with the rows staged by bulk copies (rows 16-byte aligned): CTA c's items
// c, c + G, ... (request b, chunk c) go through slots of the phase-1 ring, one chunk
// of the target row and one of the draft row per slot (two slots of bf16 rows), all
// slots requested at once; the request states of the first items are loaded together.
// The barriers are initialised again for this phase (phase 1 has no copy or arrival
// pending on them).  Same per-entry arithmetic as phase_weights; each lane sums its
// segment's 8-entry groups lane-interleaved (stage_groups).
template <typename TT, typename DT>
__device__ __forceinline__ void phase_weights_staged(const VerifyParams& p, uint8_t* ring, uint64_t* full,
                                                     uint64_t* empty, int4* s_info) {
    constexpr size_t kT = (size_t)kVerifyChunk * sizeof(TT), kD = (size_t)kVerifyChunk * sizeof(DT);
    constexpr int NS = (int)(((size_t)kV1StagesBf16 * kVerifyChunk * 2) / (kT + kD));   // slots, >= 1
    constexpr int NW = Words<TT>::N > Words<DT>::N ? Words<TT>::N : Words<DT>::N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.gamma;
    const unsigned nch = (unsigned)p.nchunk;
    const unsigned items = (unsigned)p.B * nch;   // < 2^31 (B <= 65535, nchunk <= 8192)
    const unsigned mine = items > blockIdx.x ? (items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], kWarps); }
        fence_mbar_init();
    }
    __syncthreads();
    // item k of this CTA into slot s (thread 0)
    auto issue = [&](unsigned k, int s, const DrawRow& d) {
        const unsigned it = blockIdx.x + k * gridDim.x;
        const int b = (int)(it / nch), c = (int)(it - (unsigned)b * nch);
        const long e0 = (long)c * kVerifyChunk;
        const int nvalid = (int)((long)p.V - e0 < kVerifyChunk ? (long)p.V - e0 : kVerifyChunk);
        s_info[2 * s] = make_int4(b, c, d.mode, nvalid);
        s_info[2 * s + 1] = make_int4(__float_as_int(d.m2p), __float_as_int(d.sp), __float_as_int(d.m2q),
                                      __float_as_int(d.sq));
        uint64_t* bar = &full[s];
        if (d.mode == MODE_DONE) { mbar_arrive1(bar); return; }
        uint8_t* dst = ring + (size_t)s * (kT + kD);
        const unsigned bt = (unsigned)nvalid * (unsigned)sizeof(TT);
        const unsigned bd = d.mode == MODE_RESID ? (unsigned)nvalid * (unsigned)sizeof(DT) : 0u;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, bt + bd);
        bulk_g2s(dst, static_cast<const TT*>(p.target) + ((size_t)b * (G + 1) + d.n) * p.V + e0, bt, bar);
        if (bd) bulk_g2s(dst + kT, static_cast<const DT*>(p.draft) + ((size_t)b * G + d.n) * p.V + e0, bd, bar);
    };
    if (threadIdx.x == 0) {
        DrawRow d0[NS];
#pragma unroll
        for (int j = 0; j < NS; ++j)
            if ((unsigned)j < mine) d0[j] = draw_row(p, (int)((blockIdx.x + j * gridDim.x) / nch));
#pragma unroll
        for (int j = 0; j < NS; ++j)
            if ((unsigned)j < mine) issue((unsigned)j, j, d0[j]);
    }
    for (unsigned k = 0; k < mine; ++k) {
        const int s = (int)(k % NS);
        if (threadIdx.x == 0 && k >= 1 && k - 1 + NS < mine) {
            // refill the slot of item k-1 once every warp has left it
            const int sp = (int)((k - 1) % NS);
            const unsigned kn = k - 1 + NS;
            const DrawRow dn = draw_row(p, (int)((blockIdx.x + kn * gridDim.x) / nch));
            mbar_wait(&empty[sp], ((k - 1) / NS) & 1u, p.status, kV1WaitNs);
            issue(kn, sp, dn);
        }
        if (!mbar_wait(&full[s], (k / NS) & 1u, p.status, kV1WaitNs)) break;
        const int4 i0 = s_info[2 * s], i1 = s_info[2 * s + 1];
        if (i0.z != MODE_DONE) {
            DrawRow d{i0.z, 0, 0, 0.0f, __int_as_float(i1.x), __int_as_float(i1.y), __int_as_float(i1.z),
                      __int_as_float(i1.w)};
            const uint8_t* st = ring + (size_t)s * (kT + kD);
            uint4 wt[NW], wd[NW];
            stage_groups<TT>(st, warp, lane, i0.w, wt);
            if (d.mode == MODE_RESID) stage_groups<DT>(st + kT, warp, lane, i0.w, wd);
            float sr, sp;
            weight_sums<TT, DT, NW>(d, wt, wd, sr, sp);
            const float ir = warp_inclusive_scan(sr), ip = warp_inclusive_scan(sp);
            if (lane == 31) p.ksums[((size_t)i0.x * p.nchunk + i0.y) * kWarps + warp] = make_float2(ir, ip);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive1(&empty[s]);
    }
    if (threadIdx.x == 0)   // as in phase 1: no copy in flight when the CTA leaves
        for (int s = 0; s < NS && (unsigned)s < mine; ++s) {
            const unsigned last = s + (mine - 1 - s) / NS * NS;
            mbar_wait(&full[s], (last / NS) & 1u, p.status, kV1WaitNs);
        }
}

// Inclusive prefix over the CTA's threads, in thread order, and the total.  `buf`
// holds one float per warp.
__device__ __forceinline__ float block_inclusive_scan(float x, float* buf, float& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float wi = warp_inclusive_scan(x);
    if (lane == 31) buf[warp] = wi;
    __syncthreads();
    float off = 0.0f, tot = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const float v = buf[w];
        if (w < warp) off += v;
        tot += v;
    }
    __syncthreads();   // buf is reused by the next scan
    total = tot;
    return off + wi;
}

// Four consecutive entries of a row from element v, -inf past its end.
__device__ __forceinline__ void load4(const bf16_t* row, long v, long V, bool vec_ok, float (&o)[4]) {
    if (vec_ok && v + 4 <= V) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(row + v));
        o[0] = __uint_as_float(w.x << 16); o[1] = __uint_as_float(w.x & 0xffff0000u);
        o[2] = __uint_as_float(w.y << 16); o[3] = __uint_as_float(w.y & 0xffff0000u);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] = (v + e < V) ? load_one(row + v + e) : -INFINITY;
    }
}
__device__ __forceinline__ void load4(const float* row, long v, long V, bool vec_ok, float (&o)[4]) {
    if (vec_ok && v + 4 <= V) {
        const float4 w = __ldg(reinterpret_cast<const float4*>(row + v));
        o[0] = w.x; o[1] = w.y; o[2] = w.z; o[3] = w.w;
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] = (v + e < V) ? load_one(row + v + e) : -INFINITY;
    }
}

// One CTA draws the token of request b.  Segments are the weights pass's 1024-entry
// (chunk c, warp w) sums; thread t holds segments [t K, t K + K) in order, so the
// prefix over threads is the prefix over segments.  The thread whose range passes
// t = u * W finds the segment and the remainder tl; the segment's entries (four per
// thread) get the weights pass's arithmetic again, and the first entry whose running
// sum passes tl is drawn.
template <typename TT, typename DT>
__device__ __noinline__ void draw_block(const VerifyParams& p, int b) {
    __shared__ float s_scan[kWarps];
    __shared__ int s_sel, s_seg, s_tok, s_near;
    __shared__ float s_tl;
    const int tid = threadIdx.x;
    const int G = p.gamma;
    const int nseg = p.nchunk * kWarps;
    const float2* ks = p.ksums + (size_t)b * nseg;
    const int K = (nseg + kThreads - 1) / kThreads;
    const int s0 = min(nseg, tid * K), s1 = min(nseg, s0 + K);
    // the thread's first segment sums, requested together with the request's state
    constexpr int KR = 4;
    float2 kv[KR];
#pragma unroll
    for (int u = 0; u < KR; ++u) kv[u] = (s0 + u < s1) ? __ldcg(&ks[s0 + u]) : make_float2(0.0f, 0.0f);
    auto kseg = [&](int i) -> float2 {
        const int u = i - s0;
        return u == 0 ? kv[0] : (u == 1 ? kv[1] : (u == 2 ? kv[2] : (u == 3 ? kv[3] : __ldcg(&ks[i]))));
    };
    const DrawRow d = draw_row(p, b);
    if (d.mode == MODE_DONE) return;   // the same for every thread
    float sr = 0.0f, sp = 0.0f;
#pragma unroll
    for (int u = 0; u < KR; ++u) { sr += kv[u].x; sp += kv[u].y; }
    for (int i = s0 + KR; i < s1; ++i) { const float2 v = __ldcg(&ks[i]); sr += v.x; sp += v.y; }
    float Wr, Wp;
    const float ir = block_inclusive_scan(sr, s_scan, Wr);
    const float ip = block_inclusive_scan(sp, s_scan, Wp);
    const bool ur = (d.mode == MODE_RESID) && (Wr > 0.0f);
    const float W = ur ? Wr : Wp;
    const float incl = ur ? ir : ip, mine = ur ? sr : sp;
    const float t = d.u * W;

    // the segment: first thread whose inclusive prefix passes t
    if (tid == 0) { s_sel = kThreads; s_seg = -1; s_tl = INFINITY; }
    __syncthreads();
    if (incl > t) atomicMin(&s_sel, tid);
    __syncthreads();
    const int T = s_sel;
    if (T < kThreads) {
        if (tid == T) {
            float run = incl - mine;
            int sg = -1;
            float tt = INFINITY;
            for (int i = s0; i < s1; ++i) {
                const float2 v = kseg(i);
                const float w = ur ? v.x : v.y;
                if (run + w > t) { sg = i; tt = t - run; break; }
                run += w;
            }
            s_seg = sg < 0 ? s1 - 1 : sg;
            s_tl = tt;
        }
    } else {   // u * W rounded up to W: the last segment with positive weight
        int last = -1;
        for (int i = s0; i < s1; ++i) {
            const float2 v = kseg(i);
            if ((ur ? v.x : v.y) > 0.0f) last = i;
        }
        if (last >= 0) atomicMax(&s_seg, last);
    }
    __syncthreads();
    const int seg = max(0, min(s_seg, nseg - 1));
    const float tl = s_tl;

    // the entry: four per thread, in vocabulary order
    const long base = (long)(seg / kWarps) * kVerifyChunk + (long)(seg % kWarps) * 1024 + (long)tid * 4;
    float lt[4], w[4];
    load4(static_cast<const TT*>(p.target) + ((size_t)b * (G + 1) + d.n) * p.V, base, p.V, p.vec_t != 0, lt);
    const float ipv = 1.0f / d.sp;
    if (ur) {
        float ld[4];
        load4(static_cast<const DT*>(p.draft) + ((size_t)b * G + d.n) * p.V, base, p.V, p.vec_d != 0, ld);
        const float iq = 1.0f / d.sq;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float pv = wexp(lt[e], d.m2p) * ipv;
            const float qv = wexp(ld[e], d.m2q) * iq;
            w[e] = fmaxf(0.0f, pv - qv);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = wexp(lt[e], d.m2p) * ipv;
    }
    const float mysum = (w[0] + w[1]) + (w[2] + w[3]);
    float segtot;
    const float inc = block_inclusive_scan(mysum, s_scan, segtot);
    const float ex = inc - mysum;
    if (tid == 0) { s_sel = kThreads; s_tok = -1; s_near = 0; }
    __syncthreads();
    if (ex <= tl && inc > tl) atomicMin(&s_sel, tid);
    __syncthreads();
    if (tid == s_sel) {
        float run = ex;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (run + w[e] > tl && w[e] > 0.0f) {
                s_tok = (int)(base + e);
                const float tol = kNearTie * W;
                s_near = ((run > 0.0f && fabsf(tl - run) < tol) || fabsf(run + w[e] - tl) < tol) ? 1 : 0;
                break;
            }
            run += w[e];
        }
    }
    __syncthreads();
    if (s_tok < 0) {   // rounding left no crossing: last entry of positive weight in the segment
        int last = -1;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (w[e] > 0.0f && base + e < p.V) last = (int)(base + e);
        if (last >= 0) atomicMax(&s_tok, last);
        __syncthreads();
    }
    if (tid == 0) {
        p.committed_out[(size_t)b * (G + 1) + d.n] = s_tok;
        p.bonus_out[b] = s_tok;
        p.n_out[b] = d.n;
        if (p.near_out) p.near_out[b] = d.near | s_near;
    }
    __syncthreads();   // shared state is reused by the CTA's next request
}

template <typename TT, typename DT>
__global__ void __launch_bounds__(kThreads, 2) verify_t1_kernel(VerifyParams p) {
    const unsigned nb = gridDim.x;
    __shared__ AcceptInputs s_ai;
    if ((int)blockIdx.x < p.B) accept_uniforms(p, blockIdx.x, s_ai);
    if (p.vec_t && p.vec_d) {
        extern __shared__ __align__(128) uint8_t v1_smem[];
        constexpr bool wide = sizeof(TT) == 4 || sizeof(DT) == 4;
        constexpr int S = wide ? kV1StagesBf16 / 2 : kV1StagesBf16;
        constexpr size_t stage_bytes = (size_t)kVerifyChunk * (wide ? 4 : 2);
        uint64_t* full = reinterpret_cast<uint64_t*>(v1_smem);
        uint64_t* empty = full + kV1StagesBf16;
        int4* s_item = reinterpret_cast<int4*>(v1_smem + 2 * 8 * kV1StagesBf16);
        uint8_t* ring = v1_smem + kV1RingOffset;
        if (threadIdx.x == 0) {
            for (int i = 0; i < S; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], kWarps); }
            fence_mbar_init();
        }
        __syncthreads();
        phase_stats_staged<TT, DT>(p, ring, full, empty, s_item, S, stage_bytes);
    } else {
        phase_stats<TT, DT>(p);
    }
    if ((int)blockIdx.x < p.B) load_accept_inputs<TT, DT>(p, blockIdx.x, s_ai);
    GridBarrier gb = grid_barrier_init(p.barrier);
    if (!grid_barrier(gb, nb, p.status)) return;
    for (int b = blockIdx.x; b < p.B; b += gridDim.x) accept_phase<TT, DT>(p, b, b == (int)blockIdx.x ? &s_ai : nullptr);
    if (!grid_barrier(gb, nb, p.status)) return;
    if (p.vec_t && p.vec_d) {
        extern __shared__ __align__(128) uint8_t v3_smem[];
        phase_weights_staged<TT, DT>(p, v3_smem + kV1RingOffset, reinterpret_cast<uint64_t*>(v3_smem),
                                     reinterpret_cast<uint64_t*>(v3_smem) + kV1StagesBf16,
                                     reinterpret_cast<int4*>(v3_smem + 2 * 8 * kV1StagesBf16));
    } else {
        phase_weights<TT, DT>(p);
    }
    if (!grid_barrier(gb, nb, p.status)) return;
    grid_barrier_exit(gb, nb);
    for (int b = blockIdx.x; b < p.B; b += gridDim.x) draw_block<TT, DT>(p, b);
}

// ----------------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------------
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t verify_workspace_bytes(int B, int gamma, int V) {
    const size_t nchunk = ((size_t)V + kVerifyChunk - 1) / kVerifyChunk;
    const size_t nr = 2 * (size_t)gamma + 1;
    size_t off = kWsHeaderBytes;
    off = align_up(off + sizeof(unsigned long long) * (size_t)B * (gamma + 1), 256);
    off = align_up(off + sizeof(unsigned) * (size_t)B * (gamma + 1), 256);
    off = align_up(off + sizeof(float2) * (size_t)B * nr * nchunk * kWarps, 256);
    off = align_up(off + sizeof(int4) * 2 * (size_t)B, 256);
    off = align_up(off + sizeof(float2) * (size_t)B * nchunk * kWarps, 256);
    return off;
}

void verify_bind_workspace(VerifyParams& p, void* ws) {
    char* w = static_cast<char*>(ws);
    WsHeader* h = reinterpret_cast<WsHeader*>(w);
    p.status = &h->status;
    p.done = h->done;
    p.barrier = &h->barrier[0][0];
    const size_t nchunk = ((size_t)p.V + kVerifyChunk - 1) / kVerifyChunk;
    const size_t nr = 2 * (size_t)p.gamma + 1;
    size_t off = kWsHeaderBytes;
    p.keys = reinterpret_cast<unsigned long long*>(w + off);
    off = align_up(off + sizeof(unsigned long long) * (size_t)p.B * (p.gamma + 1), 256);
    p.rowbad = reinterpret_cast<unsigned*>(w + off);
    off = align_up(off + sizeof(unsigned) * (size_t)p.B * (p.gamma + 1), 256);
    p.stats = reinterpret_cast<float2*>(w + off);
    off = align_up(off + sizeof(float2) * (size_t)p.B * nr * nchunk * kWarps, 256);
    p.state = reinterpret_cast<int4*>(w + off);
    off = align_up(off + sizeof(int4) * 2 * (size_t)p.B, 256);
    p.ksums = reinterpret_cast<float2*>(w + off);
}

template <typename TT, typename DT>
static cudaError_t launch_t1(const VerifyParams& p, cudaStream_t stream) {
    auto kern = verify_t1_kernel<TT, DT>;
    // the bulk-copy ring of phases 1 and 3 (rows 16-byte aligned): 64 KB per CTA, two per
    // SM (128 KB in flight per SM streamed faster than 192 KB)
    const size_t smem = (p.vec_t && p.vec_d) ? kV1RingOffset + (size_t)kV1StagesBf16 * kVerifyChunk * 2 : 0;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const long items = (long)p.B * (2 * p.gamma + 1) * p.nchunk;
    long grid = (long)device_sm_count() * occ;
    if (grid > items) grid = items;
    VerifyParams args = p;
    args.parts = kWarps;
    void* kargs[] = {&args};
    return cudaLaunchCooperativeKernel((const void*)kern, dim3((unsigned)grid), dim3(kThreads), kargs, smem, stream);
}

cudaError_t verify_launch(const VerifyParams& p, cudaStream_t stream) {
    if (p.temperature == 0) {
        const long items = (long)p.B * (p.gamma + 1) * (((long)p.V + kT0Chunk - 1) / kT0Chunk);
        // launched as a programmatic dependent: its launch and set-up overlap the end
        // of the kernel before it; after the library's own draft kernel, the target-row
        // pass overlaps it too and only the final scan waits (after_own_draft)
        void (*k)(VerifyParams) = p.tdt == SPEC_BF16 ? verify_t0_kernel<bf16_t> : verify_t0_kernel<float>;
        cudaLaunchConfig_t cfg = {};
        int occ = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kT0Threads, 0) != cudaSuccess || occ < 1) occ = 1;
        const long cap = (long)device_sm_count() * occ;
        cfg.gridDim = dim3((unsigned)(items < cap ? (items > 0 ? items : 1) : cap));
        cfg.blockDim = dim3(kT0Threads);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        VerifyParams args = p;
        return cudaLaunchKernelEx(&cfg, k, args);
    }
    if (p.tdt == SPEC_BF16 && p.ddt == SPEC_BF16) return launch_t1<bf16_t, bf16_t>(p, stream);
    if (p.tdt == SPEC_BF16 && p.ddt == SPEC_F32) return launch_t1<bf16_t, float>(p, stream);
    if (p.tdt == SPEC_F32 && p.ddt == SPEC_BF16) return launch_t1<float, bf16_t>(p, stream);
    return launch_t1<float, float>(p, stream);
}

}  // namespace spec
