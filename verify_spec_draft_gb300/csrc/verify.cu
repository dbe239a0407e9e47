// verify.cu - target verification of a draft block (spec_verify).
//
// Defines: "Solar Open2 DSpark" (sionic.ai), sections 1 and 6 - one target forward
// over gamma+1 positions checks the drafts and commits the agreeing prefix;
// "Speculative Decoding Part 2" (VESSL AI), blockwise decoding section - the longest
// matching prefix is accepted.  T=1 is standard rejection sampling with a residual or
// bonus draw (the pages' overlap 1 - TV is its acceptance probability).
//
// Design (HBM-bound; one pass over every row):
//   T=0  one kernel.  Work items are (row, 8192-element chunk); each CTA reduces a
//        chunk to a 64-bit argmax key (value, lowest index) and merges it with one
//        atomicMax.  The last CTA to finish ("last CTA done" counter, no waiting)
//        scans every request's prefix and writes the outputs.
//   T=1  two kernels.  (1) Softmax statistics (max, sum exp) of every target and
//        draft row per chunk; the CTA that completes a request's last chunk merges
//        that request's rows in chunk order, runs the gamma accept tests in
//        parallel, and records the row to sample from.  (2) For each request one
//        row pair (residual) or one row (bonus) is re-read in chunks to get its
//        weight per chunk in vocabulary order; the CTA completing a request finds
//        the chunk holding u * sum and scans inside it.
#include "spec_device.cuh"
#include "internal.h"

namespace spec {

constexpr int kEPT = kVerifyChunk / kThreads;   // 32 contiguous elements per thread

enum { MODE_DONE = 0, MODE_RESID = 1, MODE_BONUS = 2 };

// Loads this thread's 32 contiguous elements of chunk `c` of a row (-inf past V).
template <typename T>
__device__ __forceinline__ void load_chunk(const T* row, long V, int c, bool vec_ok, float (&x)[kEPT]) {
    constexpr int N = VecTraits<T>::N;
    const long base = (long)c * kVerifyChunk + (long)threadIdx.x * kEPT;
#pragma unroll
    for (int g = 0; g < kEPT / N; ++g) {
        float v[N];
        load_group<T, N>(row, base + g * N, V, vec_ok, v);
#pragma unroll
        for (int e = 0; e < N; ++e) x[g * N + e] = v[e];
    }
}

__device__ __forceinline__ long thread_base(int c) {
    return (long)c * kVerifyChunk + (long)threadIdx.x * kEPT;
}

// ----------------------------------------------------------------------------------
// T = 0
// ----------------------------------------------------------------------------------
template <typename TT>
__global__ void __launch_bounds__(kThreads) verify_t0_kernel(VerifyParams p) {
    const TT* target = static_cast<const TT*>(p.target);
    const long V = p.V;
    const int rows = p.B * (p.gamma + 1);
    const long items = (long)rows * p.nchunk;
    __shared__ unsigned long long s_key[kWarps];
    __shared__ int s_bad[kWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    for (long it = blockIdx.x; it < items; it += gridDim.x) {
        const int row = (int)(it / p.nchunk);
        const int c = (int)(it - (long)row * p.nchunk);
        float x[kEPT];
        load_chunk<TT>(target + (size_t)row * V, V, c, p.vec_t != 0, x);
        const long base = thread_base(c);
        unsigned long long key = 0ull;
        int bad = 0;
#pragma unroll
        for (int e = 0; e < kEPT; ++e) {
            if (base + e < V) {
                bad |= bad_logit(x[e]) ? 1 : 0;
                const unsigned long long k = argmax_key(x[e], (uint32_t)(base + e));
                key = k > key ? k : key;
            }
        }
        key = warp_max_u64(key);
        bad = warp_or(bad);
        if (lane == 0) { s_key[warp] = key; s_bad[warp] = bad; }
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned long long k = s_key[0];
            int b = s_bad[0];
            for (int w = 1; w < kWarps; ++w) { k = s_key[w] > k ? s_key[w] : k; b |= s_bad[w]; }
            atomicMax(&p.keys[row], k);
            if (b) atomicOr(&p.rowbad[row], 1u);
        }
        __syncthreads();
    }

    if (!last_block_done(&p.done[0], gridDim.x)) return;

    // Prefix scan, one thread per request; resets the keys for the next call.
    const int G = p.gamma;
    for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
        bool bad_row = false, bad_tok = false;
        int n = -1, y = -1;
        for (int i = 0; i <= G; ++i) {
            const int row = b * (G + 1) + i;
            const unsigned long long k = __ldcg(&p.keys[row]);
            const unsigned rb = __ldcg(&p.rowbad[row]);
            p.keys[row] = 0ull;
            p.rowbad[row] = 0u;
            if (rb || key_value(k) == -INFINITY) bad_row = true;
            const int am = (int)key_index(k);
            if (i < G) {
                const int t = p.tokens[(size_t)b * G + i];
                if (t < 0 || t >= p.V) bad_tok = true;
                if (n < 0 && t != am) { n = i; y = am; }
            } else if (n < 0) {
                n = G; y = am;
            }
        }
        int32_t* com = p.committed_out + (size_t)b * (G + 1);
        if (bad_row || bad_tok) {
            atomicOr(p.status, (bad_tok ? SPEC_DEV_TOKEN : 0u) | (bad_row ? SPEC_DEV_NONFINITE : 0u));
            p.n_out[b] = -1;
            p.bonus_out[b] = -1;
            for (int i = 0; i <= G; ++i) com[i] = -1;
        } else {
            p.n_out[b] = n;
            p.bonus_out[b] = y;
            for (int i = 0; i < n; ++i) com[i] = p.tokens[(size_t)b * G + i];
            com[n] = y;
            for (int i = n + 1; i <= G; ++i) com[i] = -1;
        }
        if (p.near_out) p.near_out[b] = 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) p.done[0] = 0u;
}

// ----------------------------------------------------------------------------------
// T = 1, kernel 1: row statistics + per-request accept tests
// ----------------------------------------------------------------------------------

// Softmax statistics of this thread's elements (two passes over registers), then of
// the CTA (fixed order).  Result valid in thread 0.
__device__ __forceinline__ Stat block_stat(const float (&x)[kEPT], long base, long V, int& bad, Stat* s_stat) {
    float m = -INFINITY;
#pragma unroll
    for (int e = 0; e < kEPT; ++e) {
        if (base + e < V) { bad |= bad_logit(x[e]) ? 1 : 0; m = fmaxf(m, x[e]); }
    }
    float s = 0.0f;
    if (m != -INFINITY) {
#pragma unroll
        for (int e = 0; e < kEPT; ++e) s += expf(x[e] - m);   // -inf past V gives 0
    }
    Stat st = warp_stat(Stat{m, s});
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) s_stat[warp] = st;
    __syncthreads();
    Stat r = s_stat[0];
    if (threadIdx.x == 0) {
        for (int w = 1; w < kWarps; ++w) r = stat_merge(r, s_stat[w]);
    }
    return r;
}

template <typename TT, typename DT>
__device__ void accept_phase(const VerifyParams& p, int b) {
    const TT* target = static_cast<const TT*>(p.target);
    const DT* draft = static_cast<const DT*>(p.draft);
    const int G = p.gamma;
    const int nr = 2 * G + 1;                 // local rows: 0..G target, G+1..2G draft
    __shared__ float s_m[2 * SPEC_MAX_GAMMA + 1], s_Z[2 * SPEC_MAX_GAMMA + 1];
    __shared__ int s_badrow;
    __shared__ int s_acc[SPEC_MAX_GAMMA], s_near[SPEC_MAX_GAMMA], s_badtok;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) { s_badrow = 0; s_badtok = 0; }
    __syncthreads();

    // merge each row's chunk statistics in chunk order (lane-strided, fixed tree)
    for (int lr = warp; lr < nr; lr += kWarps) {
        const size_t rowid = (size_t)b * nr + lr;
        Stat acc = stat_empty();
        for (int c = lane; c < p.nchunk; c += 32) {
            const float2 st = __ldcg(&p.stats[rowid * p.nchunk + c]);
            acc = stat_merge(acc, Stat{st.x, st.y});
        }
        acc = warp_stat(acc);
        if (lane == 0) {
            s_m[lr] = acc.m;
            s_Z[lr] = acc.s;
            const unsigned rb = __ldcg(&p.rowbad[rowid]);
            p.rowbad[rowid] = 0u;
            if (rb || acc.m == -INFINITY) atomicOr(&s_badrow, 1);
        }
    }
    __syncthreads();

    // the gamma accept tests, one thread each
    const uint64_t seed = p.seeds[b];
    for (int j = threadIdx.x; j < G; j += blockDim.x) {
        const int t = p.tokens[(size_t)b * G + j];
        int acc = 0, near = 0;
        if (t < 0 || t >= p.V) {
            atomicOr(&s_badtok, 1);
        } else {
            const float lp = to_float(target[((size_t)b * (G + 1) + j) * p.V + t]);
            const float lq = to_float(draft[((size_t)b * G + j) * p.V + t]);
            const float pj = expf(lp - s_m[j]) / s_Z[j];
            const float qj = expf(lq - s_m[G + 1 + j]) / s_Z[G + 1 + j];
            const float u = philox_uniform(seed, (uint64_t)b, (uint64_t)(j + 1), 1);
            acc = (u * qj < pj) ? 1 : 0;
            near = (fabsf(u * qj - pj) < kNearTie * qj) ? 1 : 0;
        }
        s_acc[j] = acc;
        s_near[j] = near;
    }
    __syncthreads();

    if (threadIdx.x == 0) {
        int32_t* com = p.committed_out + (size_t)b * (G + 1);
        int4 st0 = make_int4(MODE_DONE, -1, 0, 0);
        int4 st1 = make_int4(0, 0, 0, 0);
        if (s_badrow || s_badtok) {
            atomicOr(p.status, (s_badtok ? SPEC_DEV_TOKEN : 0u) | (s_badrow ? SPEC_DEV_NONFINITE : 0u));
            p.n_out[b] = -1;
            p.bonus_out[b] = -1;
            for (int i = 0; i <= G; ++i) com[i] = -1;
            if (p.near_out) p.near_out[b] = 0;
        } else {
            int k = 0, near = 0;
            while (k < G && s_acc[k]) { near |= s_near[k]; ++k; }
            if (k < G) near |= s_near[k];
            for (int i = 0; i < k; ++i) com[i] = p.tokens[(size_t)b * G + i];
            for (int i = k + 1; i <= G; ++i) com[i] = -1;
            if (k < G) {   // rejected at position k+1: target row k and draft row k
                st0 = make_int4(MODE_RESID, k, near, 0);
                st1 = make_int4(__float_as_int(s_m[k]), __float_as_int(s_Z[k]),
                                __float_as_int(s_m[G + 1 + k]), __float_as_int(s_Z[G + 1 + k]));
            } else {       // all accepted: bonus from target row gamma
                st0 = make_int4(MODE_BONUS, G, near, 0);
                st1 = make_int4(__float_as_int(s_m[G]), __float_as_int(s_Z[G]), 0, 0);
            }
        }
        p.state[2 * b] = st0;
        p.state[2 * b + 1] = st1;
    }
    __syncthreads();
}

template <typename TT, typename DT>
__global__ void __launch_bounds__(kThreads) verify_t1_stats_kernel(VerifyParams p) {
    const TT* target = static_cast<const TT*>(p.target);
    const DT* draft = static_cast<const DT*>(p.draft);
    const long V = p.V;
    const int G = p.gamma;
    const int nr = 2 * G + 1;
    const long per_req = (long)nr * p.nchunk;
    const long items = per_req * p.B;
    __shared__ Stat s_stat[kWarps];
    __shared__ int s_badw[kWarps];
    __shared__ int s_last;

    for (long it = blockIdx.x; it < items; it += gridDim.x) {
        const int b = (int)(it / per_req);
        const long rem = it - (long)b * per_req;
        const int lr = (int)(rem / p.nchunk);
        const int c = (int)(rem - (long)lr * p.nchunk);
        float x[kEPT];
        if (lr <= G) load_chunk<TT>(target + ((size_t)b * (G + 1) + lr) * V, V, c, p.vec_t != 0, x);
        else load_chunk<DT>(draft + ((size_t)b * G + (lr - G - 1)) * V, V, c, p.vec_d != 0, x);
        int bad = 0;
        const Stat st = block_stat(x, thread_base(c), V, bad, s_stat);
        bad = warp_or(bad);
        if ((threadIdx.x & 31) == 0) s_badw[threadIdx.x >> 5] = bad;
        __syncthreads();
        if (threadIdx.x == 0) {
            const size_t rowid = (size_t)b * nr + lr;
            p.stats[rowid * p.nchunk + c] = make_float2(st.m, st.s);
            int bb = 0;
            for (int w = 0; w < kWarps; ++w) bb |= s_badw[w];
            if (bb) atomicOr(&p.rowbad[rowid], 1u);
            __threadfence();
            const unsigned prev = atomicAdd(&p.done1[b], 1u);
            s_last = (prev == (unsigned)per_req - 1u) ? 1 : 0;
            if (s_last) { __threadfence(); p.done1[b] = 0u; }
        }
        __syncthreads();
        if (s_last) accept_phase<TT, DT>(p, b);
    }
}

// ----------------------------------------------------------------------------------
// T = 1, kernel 2: residual / bonus draw
// ----------------------------------------------------------------------------------

// Weights of this thread's 32 elements of chunk c: w = max(0, p - q) (residual) and
// p, with p = exp(l - mp) / Zp, q = exp(d - mq) / Zq.  Identical arithmetic in the
// chunk-sum pass and in the final scan, so the per-thread sums agree bit for bit.
template <typename TT, typename DT>
__device__ __forceinline__ void chunk_weights(const VerifyParams& p, int b, int mode, int n, int c,
                                              float mp, float Zp, float mq, float Zq,
                                              float (&wr)[kEPT], float (&wp)[kEPT]) {
    const TT* target = static_cast<const TT*>(p.target);
    const DT* draft = static_cast<const DT*>(p.draft);
    const long V = p.V;
    const int G = p.gamma;
    float lt[kEPT];
    load_chunk<TT>(target + ((size_t)b * (G + 1) + n) * V, V, c, p.vec_t != 0, lt);
    if (mode == MODE_RESID) {
        float ld[kEPT];
        load_chunk<DT>(draft + ((size_t)b * G + n) * V, V, c, p.vec_d != 0, ld);
#pragma unroll
        for (int e = 0; e < kEPT; ++e) {
            const float pv = expf(lt[e] - mp) / Zp;
            const float qv = expf(ld[e] - mq) / Zq;
            wp[e] = pv;
            wr[e] = fmaxf(0.0f, pv - qv);
        }
    } else {
#pragma unroll
        for (int e = 0; e < kEPT; ++e) {
            wp[e] = expf(lt[e] - mp) / Zp;
            wr[e] = 0.0f;
        }
    }
}

// Block-wide exclusive scan of one float per thread (fixed order).  Returns the
// exclusive prefix of this thread; *total receives the block total.
__device__ __forceinline__ float block_exclusive_scan(float x, float* s_warp, float* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float incl = warp_inclusive_scan(x);
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const float w = lane < kWarps ? s_warp[lane] : 0.0f;
        const float wi = warp_inclusive_scan(w);
        if (lane < kWarps) s_warp[kWarps + lane] = wi - w;    // exclusive warp offsets
        if (lane == kWarps - 1) s_warp[2 * kWarps] = wi;
    }
    __syncthreads();
    const float ex = s_warp[kWarps + warp] + (incl - x);
    *total = s_warp[2 * kWarps];
    __syncthreads();
    return ex;
}

template <typename TT, typename DT>
__device__ void sample_phase(const VerifyParams& p, int b, int4 st0, int4 st1) {
    const int G = p.gamma;
    const int mode = st0.x, n = st0.y;
    const float mp = __int_as_float(st1.x), Zp = __int_as_float(st1.y);
    const float mq = __int_as_float(st1.z), Zq = __int_as_float(st1.w);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __shared__ float s_scan[2 * kWarps + 1];
    __shared__ int s_chunk, s_use_resid, s_tok, s_near;
    __shared__ float s_tloc, s_W;

    // totals and the chunk that holds the threshold (warp 0, contiguous segments)
    if (warp == 0) {
        const int K = (p.nchunk + 31) / 32;
        const int c0 = lane * K, c1 = min(p.nchunk, c0 + K);
        float sr = 0.0f, sp = 0.0f;
        for (int c = c0; c < c1; ++c) {
            const float2 ks = __ldcg(&p.ksums[(size_t)b * p.nchunk + c]);
            sr += ks.x;
            sp += ks.y;
        }
        const float ir = warp_inclusive_scan(sr), ip = warp_inclusive_scan(sp);
        const float Wr = __shfl_sync(0xffffffffu, ir, 31), Wp = __shfl_sync(0xffffffffu, ip, 31);
        const int use_resid = (mode == MODE_RESID) && (Wr > 0.0f);
        const float W = use_resid ? Wr : Wp;
        const float incl = use_resid ? ir : ip;
        const float mine = use_resid ? sr : sp;
        const float u = (mode == MODE_RESID) ? philox_uniform(p.seeds[b], (uint64_t)b, (uint64_t)(n + 1), 2)
                                             : philox_uniform(p.seeds[b], (uint64_t)b, (uint64_t)(G + 1), 3);
        const float t = u * W;
        const unsigned cross = __ballot_sync(0xffffffffu, incl > t);
        int chunk = -1;
        float tloc = 0.0f;
        if (cross) {
            const int L = __ffs(cross) - 1;
            if (lane == L) {
                float run = incl - mine;
                for (int c = c0; c < c1; ++c) {
                    const float2 ks = __ldcg(&p.ksums[(size_t)b * p.nchunk + c]);
                    const float w = use_resid ? ks.x : ks.y;
                    if (run + w > t) { chunk = c; tloc = t - run; break; }
                    run += w;
                }
                if (chunk < 0) {   // rounding: the segment's walk fell short
                    chunk = c1 - 1;
                    tloc = INFINITY;
                }
            }
            chunk = __shfl_sync(0xffffffffu, chunk, L);
            tloc = __shfl_sync(0xffffffffu, tloc, L);
        } else {
            // u * W rounded up to W: take the last chunk with positive weight
            int last = -1;
            for (int c = c0; c < c1; ++c) {
                const float2 ks = __ldcg(&p.ksums[(size_t)b * p.nchunk + c]);
                if ((use_resid ? ks.x : ks.y) > 0.0f) last = c;
            }
            const unsigned has = __ballot_sync(0xffffffffu, last >= 0);
            chunk = has ? __shfl_sync(0xffffffffu, last, 31 - __clz(has)) : 0;
            tloc = INFINITY;
        }
        chunk = max(0, min(chunk, p.nchunk - 1));
        if (lane == 0) { s_chunk = chunk; s_tloc = tloc; s_use_resid = use_resid; s_W = W; }
    }
    __syncthreads();

    // scan inside the chunk
    const int c = s_chunk;
    float wr[kEPT], wp[kEPT];
    chunk_weights<TT, DT>(p, b, mode, n, c, mp, Zp, mq, Zq, wr, wp);
    const bool ur = s_use_resid != 0;
    float mysum = 0.0f;
#pragma unroll
    for (int e = 0; e < kEPT; ++e) mysum += ur ? wr[e] : wp[e];
    float total;
    const float ex = block_exclusive_scan(mysum, s_scan, &total);
    const float tl = s_tloc;
    const long base = thread_base(c);
    // the thread whose range crosses tl scans its elements
    int tok = -1;
    float near_lo = 0.0f, near_hi = 0.0f;
    if (ex <= tl && ex + mysum > tl) {
        float run = ex;
        for (int e = 0; e < kEPT; ++e) {
            const float w = ur ? wr[e] : wp[e];
            if (run + w > tl && w > 0.0f) { tok = (int)(base + e); near_lo = run; near_hi = run + w; break; }
            run += w;
        }
    }
    if (threadIdx.x == 0) { s_tok = -1; s_near = 0; }
    __syncthreads();
    if (tok >= 0) atomicMax(&s_tok, tok);   // at most one thread crosses; max is safe
    __syncthreads();
    if (s_tok < 0) {
        // rounding left no crossing: the last element of positive weight in the chunk
        int last = -1;
        for (int e = 0; e < kEPT; ++e)
            if ((ur ? wr[e] : wp[e]) > 0.0f && base + e < p.V) last = (int)(base + e);
        if (last >= 0) atomicMax(&s_tok, last);
        __syncthreads();
    }
    if (tok >= 0) {
        const float tol = kNearTie * s_W;
        if ((near_lo > 0.0f && fabsf(tl - near_lo) < tol) || fabsf(near_hi - tl) < tol) s_near = 1;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const int y = s_tok;
        p.committed_out[(size_t)b * (G + 1) + n] = y;
        p.bonus_out[b] = y;
        p.n_out[b] = n;
        if (p.near_out) p.near_out[b] = st0.z | s_near;
    }
    __syncthreads();
}

template <typename TT, typename DT>
__global__ void __launch_bounds__(kThreads) verify_t1_sample_kernel(VerifyParams p) {
    const long items = (long)p.B * p.nchunk;
    __shared__ float s_red[2][2 * kWarps + 1];
    __shared__ int s_last;
    for (long it = blockIdx.x; it < items; it += gridDim.x) {
        const int b = (int)(it / p.nchunk);
        const int c = (int)(it - (long)b * p.nchunk);
        const int4 st0 = __ldcg(&p.state[2 * b]);
        if (st0.x == MODE_DONE) continue;
        const int4 st1 = __ldcg(&p.state[2 * b + 1]);
        float wr[kEPT], wp[kEPT];
        chunk_weights<TT, DT>(p, b, st0.x, st0.y, c, __int_as_float(st1.x), __int_as_float(st1.y),
                              __int_as_float(st1.z), __int_as_float(st1.w), wr, wp);
        float sr = 0.0f, sp = 0.0f;
#pragma unroll
        for (int e = 0; e < kEPT; ++e) { sr += wr[e]; sp += wp[e]; }
        // chunk totals with exactly the association of the final in-chunk scan
        float tr, tp;
        block_exclusive_scan(sr, s_red[0], &tr);
        block_exclusive_scan(sp, s_red[1], &tp);
        if (threadIdx.x == 0) {
            p.ksums[(size_t)b * p.nchunk + c] = make_float2(tr, tp);
            __threadfence();
            const unsigned prev = atomicAdd(&p.done2[b], 1u);
            s_last = (prev == (unsigned)p.nchunk - 1u) ? 1 : 0;
            if (s_last) { __threadfence(); p.done2[b] = 0u; }
        }
        __syncthreads();
        if (s_last) sample_phase<TT, DT>(p, b, st0, st1);
    }
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
    off = align_up(off + sizeof(unsigned) * (size_t)B * nr, 256);
    off = align_up(off + sizeof(float2) * (size_t)B * nr * nchunk, 256);
    off = align_up(off + sizeof(unsigned) * (size_t)B, 256);
    off = align_up(off + sizeof(unsigned) * (size_t)B, 256);
    off = align_up(off + sizeof(int4) * 2 * (size_t)B, 256);
    off = align_up(off + sizeof(float2) * (size_t)B * nchunk, 256);
    return off;
}

void verify_bind_workspace(VerifyParams& p, void* ws) {
    char* w = static_cast<char*>(ws);
    WsHeader* h = reinterpret_cast<WsHeader*>(w);
    p.status = &h->status;
    p.done = h->done;
    const size_t nchunk = ((size_t)p.V + kVerifyChunk - 1) / kVerifyChunk;
    const size_t nr = 2 * (size_t)p.gamma + 1;
    size_t off = kWsHeaderBytes;
    p.keys = reinterpret_cast<unsigned long long*>(w + off);
    off = align_up(off + sizeof(unsigned long long) * (size_t)p.B * (p.gamma + 1), 256);
    p.rowbad = reinterpret_cast<unsigned*>(w + off);
    off = align_up(off + sizeof(unsigned) * (size_t)p.B * nr, 256);
    p.stats = reinterpret_cast<float2*>(w + off);
    off = align_up(off + sizeof(float2) * (size_t)p.B * nr * nchunk, 256);
    p.done1 = reinterpret_cast<unsigned*>(w + off);
    off = align_up(off + sizeof(unsigned) * (size_t)p.B, 256);
    p.done2 = reinterpret_cast<unsigned*>(w + off);
    off = align_up(off + sizeof(unsigned) * (size_t)p.B, 256);
    p.state = reinterpret_cast<int4*>(w + off);
    off = align_up(off + sizeof(int4) * 2 * (size_t)p.B, 256);
    p.ksums = reinterpret_cast<float2*>(w + off);
}

template <typename TT, typename DT>
static cudaError_t launch_t1(const VerifyParams& p, cudaStream_t stream) {
    const int sms = device_sm_count();
    const long items1 = (long)p.B * (2 * p.gamma + 1) * p.nchunk;
    const int grid1 = (int)(items1 < (long)sms * 8 ? items1 : (long)sms * 8);
    verify_t1_stats_kernel<TT, DT><<<grid1, kThreads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long items2 = (long)p.B * p.nchunk;
    const int grid2 = (int)(items2 < (long)sms * 8 ? items2 : (long)sms * 8);
    verify_t1_sample_kernel<TT, DT><<<grid2, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t verify_launch(const VerifyParams& p, cudaStream_t stream) {
    const int sms = device_sm_count();
    if (p.temperature == 0) {
        const long items = (long)p.B * (p.gamma + 1) * p.nchunk;
        const int grid = (int)(items < (long)sms * 8 ? items : (long)sms * 8);
        if (p.tdt == SPEC_BF16) verify_t0_kernel<bf16_t><<<grid, kThreads, 0, stream>>>(p);
        else verify_t0_kernel<float><<<grid, kThreads, 0, stream>>>(p);
        return cudaGetLastError();
    }
    if (p.tdt == SPEC_BF16 && p.ddt == SPEC_BF16) return launch_t1<bf16_t, bf16_t>(p, stream);
    if (p.tdt == SPEC_BF16 && p.ddt == SPEC_F32) return launch_t1<bf16_t, float>(p, stream);
    if (p.tdt == SPEC_F32 && p.ddt == SPEC_BF16) return launch_t1<float, bf16_t>(p, stream);
    return launch_t1<float, float>(p, stream);
}

}  // namespace spec
