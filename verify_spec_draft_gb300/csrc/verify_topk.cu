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
//   topk_rows_kernel   one CTA per row streams it; every thread keeps its k largest
//                      64-bit keys (ordered value high, inverted index low, so a larger
//                      key is a larger value or, on a tie, a lower index) in registers,
//                      inserting only keys above its current k-th; the CTA then takes its
//                      k largest by k rounds of a block maximum over the threads' heads.
//                      NaN or +inf in the row flags it.
//   topk_accept_kernel one thread per request: the filtered rows from the key lists in
//                      float64, the accept tests (Philox stream 1), and the residual or
//                      bonus draw over at most k candidates in index order (streams 2, 3).
#include "spec_device.cuh"
#include "internal.h"

namespace spec {

constexpr int kTopkThreads = 256;

__device__ __forceinline__ void topk_insert(unsigned long long (&L)[kTopkMax], unsigned long long key, int k,
                                            unsigned long long& thr) {
#pragma unroll
    for (int i = 0; i < kTopkMax; ++i) {
        if (key > L[i]) {
            const unsigned long long t = L[i];
            L[i] = key;
            key = t;
        }
    }
#pragma unroll
    for (int i = 0; i < kTopkMax; ++i)
        if (i == k - 1) thr = L[i];
}

template <typename T>
__device__ __forceinline__ void topk_take(float x, long idx, unsigned long long (&L)[kTopkMax], int k,
                                          unsigned long long& thr, int& bad) {
    bad |= bad_logit(x) ? 1 : 0;
    const unsigned long long key = argmax_key(x, (uint32_t)idx);
    if (key > thr) topk_insert(L, key, k, thr);
}

// Rows row0 .. row0 + gridDim.x - 1 of `src` ([rows, V]); the CTA's k keys go to
// keys[(out0 + blockIdx.x) * kTopkMax + i] (0 where the row has fewer entries).
template <typename T>
__global__ void __launch_bounds__(kTopkThreads) topk_rows_kernel(const T* src, long V, int k, bool vec,
                                                                 unsigned long long* keys, unsigned* bad_out,
                                                                 int out0) {
    extern __shared__ __align__(16) unsigned long long s_list[];   // [threads][k]
    __shared__ unsigned long long s_wmax[kTopkThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const T* row = src + (size_t)blockIdx.x * V;
    unsigned long long L[kTopkMax];
#pragma unroll
    for (int i = 0; i < kTopkMax; ++i) L[i] = 0ull;
    unsigned long long thr = 0ull;
    int bad = 0;
    if (vec) {
        constexpr int N = VecTraits<T>::N;
        const long nw = V / N;
        for (long w = tid; w < nw; w += blockDim.x) {
            float x[N];
            load_vec(row + w * N, x);
#pragma unroll
            for (int e = 0; e < N; ++e) topk_take<T>(x[e], w * N + e, L, k, thr, bad);
        }
    } else {
        for (long v = tid; v < V; v += blockDim.x) topk_take<T>(load_one(row + v), v, L, k, thr, bad);
    }
    for (int i = 0; i < k; ++i) {
        unsigned long long w = 0ull;
#pragma unroll
        for (int q = 0; q < kTopkMax; ++q)
            if (q == i) w = L[q];
        s_list[(size_t)tid * k + i] = w;
    }
    bad = __syncthreads_or(bad);
    // k rounds: the largest remaining head over the block; its thread moves on (keys
    // are distinct, the index being part of them, except the empty key 0)
    int pos = 0;
    unsigned long long* out = keys + (size_t)(out0 + blockIdx.x) * kTopkMax;
    for (int r = 0; r < k; ++r) {
        const unsigned long long head = pos < k ? s_list[(size_t)tid * k + pos] : 0ull;
        unsigned long long m = head;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long t = __shfl_xor_sync(0xffffffffu, m, o);
            m = t > m ? t : m;
        }
        if (lane == 0) s_wmax[warp] = m;
        __syncthreads();
        unsigned long long best = 0ull;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) best = s_wmax[w] > best ? s_wmax[w] : best;
        if (best != 0ull && head == best) ++pos;
        if (tid == 0) out[r] = best;
        __syncthreads();
    }
    if (tid == 0) bad_out[out0 + blockIdx.x] = bad ? 1u : 0u;
}

// A filtered row from its key list: kept entries (index, weight) in descending order of
// value, weights normalised to sum 1.  Returns the number kept, 0 for no distribution.
__device__ int topk_filter(const unsigned long long* keys, int k, double top_p, int (&idx)[kTopkMax],
                           double (&w)[kTopkMax]) {
    int n = 0;
    double m = 0.0, S = 0.0;
    for (int i = 0; i < k; ++i) {
        const unsigned long long key = keys[i];
        if (key == 0ull) break;
        const float v = key_value(key);
        if (i == 0) {
            if (!(v > -INFINITY)) return 0;   // no finite entry
            m = (double)v;
        }
        idx[n] = (int)key_index(key);
        w[n] = exp((double)v - m);
        S += w[n];
        ++n;
    }
    double run = 0.0, Z = 0.0;
    int kept = 0;
    for (int i = 0; i < n; ++i) {
        run += w[i] / S;
        Z += w[i];
        ++kept;
        if (run >= top_p) break;
    }
    for (int i = 0; i < kept; ++i) w[i] /= Z;
    return kept;
}

__device__ __forceinline__ double topk_prob(const int (&idx)[kTopkMax], const double (&w)[kTopkMax], int n, int x) {
    for (int i = 0; i < n; ++i)
        if (idx[i] == x) return w[i];
    return 0.0;
}

// Inverse-CDF draw over (index, weight) candidates in index order: the smallest index
// whose running weight passes u * total, else the last of positive weight; `near` when
// the threshold lies within 1e-6 of the total from a boundary between two positive
// entries.
__device__ int topk_draw(int (&idx)[kTopkMax], double (&w)[kTopkMax], int n, double u, int& near) {
    for (int i = 1; i < n; ++i) {   // insertion sort by index
        const int ki = idx[i];
        const double kw = w[i];
        int j = i - 1;
        while (j >= 0 && idx[j] > ki) { idx[j + 1] = idx[j]; w[j + 1] = w[j]; --j; }
        idx[j + 1] = ki;
        w[j + 1] = kw;
    }
    double Z = 0.0;
    for (int i = 0; i < n; ++i) Z += w[i];
    const double t = u * Z;
    double C = 0.0, Cprev = 0.0;
    int v = -1, last = -1;
    for (int i = 0; i < n; ++i) {
        if (w[i] > 0.0) last = i;
        Cprev = C;
        C += w[i];
        if (v < 0 && C > t) {
            v = i;
            bool later = false;
            for (int q = i + 1; q < n; ++q) later |= w[q] > 0.0;
            if (fabs(C - t) < 1e-6 * Z && later) near = 1;
            if (Cprev > 0.0 && fabs(Cprev - t) < 1e-6 * Z) near = 1;
        }
    }
    if (v < 0) v = last;
    return v < 0 ? -1 : idx[v];
}

__global__ void topk_accept_kernel(TopkParams p) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= p.B) return;
    const int G = p.gamma;
    const int nT = p.B * (G + 1);
    int32_t* com = p.committed_out + (size_t)b * (G + 1);
    bool ok = true;
    for (int j = 0; j < G; ++j) {
        const int x = p.tokens[(size_t)b * G + j];
        ok &= x >= 0 && x < p.V;
    }
    for (int i = 0; i <= G; ++i) ok &= p.bad[b * (G + 1) + i] == 0u;
    for (int i = 0; i < G; ++i) ok &= p.bad[nT + b * G + i] == 0u;
    int idx_p[kTopkMax], idx_q[kTopkMax];
    double wp[kTopkMax], wq[kTopkMax];
    if (ok) {   // every row the request reads has a distribution
        for (int i = 0; i <= G && ok; ++i)
            ok = topk_filter(p.keys + (size_t)(b * (G + 1) + i) * kTopkMax, p.k, p.top_p, idx_p, wp) > 0;
        for (int i = 0; i < G && ok; ++i)
            ok = topk_filter(p.keys + (size_t)(nT + b * G + i) * kTopkMax, p.k, p.top_p, idx_q, wq) > 0;
    }
    if (!ok) {
        p.n_out[b] = -1;
        p.bonus_out[b] = -1;
        for (int i = 0; i <= G; ++i) com[i] = -1;
        if (p.near_out) p.near_out[b] = 0;
        atomicOr(p.status, SPEC_DEV_TOKEN);
        return;
    }
    const uint64_t seed = p.seeds[b];
    int near = 0;
    for (int j = 1; j <= G; ++j) {
        const int np = topk_filter(p.keys + (size_t)(b * (G + 1) + j - 1) * kTopkMax, p.k, p.top_p, idx_p, wp);
        const int nq = topk_filter(p.keys + (size_t)(nT + b * G + j - 1) * kTopkMax, p.k, p.top_p, idx_q, wq);
        const int x = p.tokens[(size_t)b * G + j - 1];
        const double px = topk_prob(idx_p, wp, np, x), qx = topk_prob(idx_q, wq, nq, x);
        const double u = (double)philox_uniform(seed, (uint64_t)b, (uint64_t)j, 1);
        if (fabs(u * qx - px) < 1e-6 * qx) near = 1;
        if (u * qx < px) {   // accepted (q = 0 accepts iff p > 0)
            com[j - 1] = x;
            continue;
        }
        // residual max(0, p - q): positive only on the filtered p's entries
        double r[kTopkMax];
        double rs = 0.0;
        for (int i = 0; i < np; ++i) {
            r[i] = wp[i] - topk_prob(idx_q, wq, nq, idx_p[i]);
            r[i] = r[i] > 0.0 ? r[i] : 0.0;
            rs += r[i];
        }
        if (!(rs > 0.0))
            for (int i = 0; i < np; ++i) r[i] = wp[i];
        const double u2 = (double)philox_uniform(seed, (uint64_t)b, (uint64_t)j, 2);
        const int y = topk_draw(idx_p, r, np, u2, near);
        com[j - 1] = y;
        for (int i = j; i <= G; ++i) com[i] = -1;
        p.n_out[b] = j - 1;
        p.bonus_out[b] = y;
        if (p.near_out) p.near_out[b] = near;
        return;
    }
    const int np = topk_filter(p.keys + (size_t)(b * (G + 1) + G) * kTopkMax, p.k, p.top_p, idx_p, wp);
    const double u3 = (double)philox_uniform(seed, (uint64_t)b, (uint64_t)(G + 1), 3);
    const int y = topk_draw(idx_p, wp, np, u3, near);
    com[G] = y;
    p.n_out[b] = G;
    p.bonus_out[b] = y;
    if (p.near_out) p.near_out[b] = near;
}

size_t verify_topk_workspace_bytes(int B, int gamma) {
    const size_t rows = (size_t)B * (2 * gamma + 1);
    return kWsHeaderBytes + rows * kTopkMax * sizeof(unsigned long long) + rows * sizeof(unsigned);
}

template <typename T>
static cudaError_t launch_rows(const void* src, int rows, long V, int k, bool vec, unsigned long long* keys,
                               unsigned* bad, int out0, cudaStream_t stream) {
    const size_t smem = (size_t)kTopkThreads * k * sizeof(unsigned long long);
    cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    topk_rows_kernel<T><<<rows, kTopkThreads, smem, stream>>>(static_cast<const T*>(src), V, k, vec, keys, bad, out0);
    return cudaGetLastError();
}

cudaError_t verify_topk_launch(TopkParams& p, void* ws, cudaStream_t stream) {
    char* w = static_cast<char*>(ws);
    p.status = &reinterpret_cast<WsHeader*>(w)->status;
    const size_t rows = (size_t)p.B * (2 * p.gamma + 1);
    p.keys = reinterpret_cast<unsigned long long*>(w + kWsHeaderBytes);
    p.bad = reinterpret_cast<unsigned*>(w + kWsHeaderBytes + rows * kTopkMax * sizeof(unsigned long long));
    const int nT = p.B * (p.gamma + 1), nD = p.B * p.gamma;
    const bool vt = ((size_t)p.V * (p.tdt == SPEC_BF16 ? 2 : 4)) % 16 == 0;
    const bool vd = ((size_t)p.V * (p.ddt == SPEC_BF16 ? 2 : 4)) % 16 == 0;
    cudaError_t e = p.tdt == SPEC_BF16
                        ? launch_rows<bf16_t>(p.target, nT, p.V, p.k, vt, p.keys, p.bad, 0, stream)
                        : launch_rows<float>(p.target, nT, p.V, p.k, vt, p.keys, p.bad, 0, stream);
    if (e != cudaSuccess) return e;
    e = p.ddt == SPEC_BF16 ? launch_rows<bf16_t>(p.draft, nD, p.V, p.k, vd, p.keys, p.bad, nT, stream)
                           : launch_rows<float>(p.draft, nD, p.V, p.k, vd, p.keys, p.bad, nT, stream);
    if (e != cudaSuccess) return e;
    topk_accept_kernel<<<(p.B + 63) / 64, 64, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace spec
