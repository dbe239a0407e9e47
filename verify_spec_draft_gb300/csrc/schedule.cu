// schedule.cu - the verify budget across a batch (spec_verify_budget).
//
// Defines: "Speculative Decoding Part 2: the evolution of drafter architectures" (VESSL
// AI), DSpark section, the paragraphs after the bias equation: per position, the
// confidence is the probability that it passes given that every earlier position
// passed; a scheduler multiplies these into expected lengths, gives the verification
// budget to the positions with the highest pass probability across all requests of
// the batch, and maximises throughput against a measured hardware curve.
//
// Reading (the pages give no formula): P[b, j] = prod_{i<=j} clamp(c[b, i], 0, 1), NaN
// read as 0; candidates ordered by P descending, ties by flat index b * gamma + j
// ascending (the first k hold a prefix of every request, since P never grows with j);
// E(k) = B + sum of the first k P; k* = argmax_{k <= K} E(k) / t[k] (smallest k on
// ties, non-positive or NaN t[k] excluded), or K without a curve; gamma_b = request
// b's count among the first k*.
//
// One CTA holds everything in shared memory (at most SPEC_MAX_BUDGET_CANDIDATES
// candidates): the confidences loaded in one coalesced pass, products in float64 in
// position order, a bitonic sort of (P, index) pairs on P's bit pattern (P >= 0, so
// the unsigned order of its bits is its order; no float64 compare on this GPU's slow
// FP64 pipe), a blocked float64 prefix scan, the objective per k, a block argmax,
// counts.
#include <float.h>
#include <limits.h>

#include "spec_device.cuh"
#include "internal.h"

namespace spec {

constexpr int kSchedThreads = 1024;

__device__ __forceinline__ bool sched_precedes(unsigned long long pa, int ia, unsigned long long pb, int ib) {
    return pa > pb || (pa == pb && ia < ib);
}

__global__ void __launch_bounds__(kSchedThreads) verify_budget_kernel(const float* conf, int B, int G, int K,
                                                                      const float* cost, int32_t* gamma_out,
                                                                      float* expected_out) {
    extern __shared__ __align__(16) unsigned char s_raw[];
    const int N = B * G;
    int M = 1;
    while (M < N) M <<= 1;
    double* sp = reinterpret_cast<double*>(s_raw);   // [M] c, then P (sorted), then prefix sums
    unsigned long long* sb = reinterpret_cast<unsigned long long*>(s_raw);   // the same words as bits
    int* si = reinterpret_cast<int*>(sp + M);         // [M] flat candidate indices
    int* scount = si + M;                             // [B] positions per request
    __shared__ double s_part[kSchedThreads / 32];
    __shared__ double s_bobj[kSchedThreads / 32];
    __shared__ int s_bk[kSchedThreads / 32];
    __shared__ int s_kstar;
    __shared__ unsigned long long s_xk[2][kSchedThreads];   // the register sort's exchange buffers
    __shared__ int s_xi[2][kSchedThreads];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nt = blockDim.x;

    // the clamped confidences, every thread one coalesced load at a time
    for (int i = tid; i < N; i += nt) {
        const float c = conf[i];
        sp[i] = (double)(c > 0.0f ? fminf(c, 1.0f) : 0.0f);   // NaN, -0 and below: +0
        si[i] = i;
    }
    for (int i = N + tid; i < M; i += nt) { sb[i] = 0ull; si[i] = INT_MAX; }   // padding: P = 0, sorts last
    __syncthreads();
    // pass products, one request per thread, in position order
    for (int b = tid; b < B; b += nt) {
        double run = 1.0;
        for (int j = 0; j < G; ++j) {
            run *= sp[b * G + j];
            sp[b * G + j] = run;
        }
        scount[b] = 0;
    }
    __syncthreads();

    // bitonic sort into candidate order (P descending, index ascending)
    if (M <= nt) {
        // one candidate per thread, in registers: partners closer than a warp are reached
        // by shuffles, farther ones through a shared array (two buffers, so one barrier a
        // step)
        unsigned long long pk = tid < M ? sb[tid] : 0ull;
        int ik = tid < M ? si[tid] : INT_MAX;
        int buf = 0;
        for (int size = 2; size <= M; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                unsigned long long po;
                int io;
                if (stride < 32) {
                    po = ((unsigned long long)__shfl_xor_sync(0xffffffffu, (unsigned)(pk >> 32), stride) << 32) |
                         (unsigned)__shfl_xor_sync(0xffffffffu, (unsigned)pk, stride);
                    io = __shfl_xor_sync(0xffffffffu, ik, stride);
                } else {
                    s_xk[buf][tid] = pk;
                    s_xi[buf][tid] = ik;
                    __syncthreads();
                    po = s_xk[buf][tid ^ stride];
                    io = s_xi[buf][tid ^ stride];
                    buf ^= 1;
                }
                // the lower position of a pair keeps the preceding candidate in an ascending
                // run (up), the other one in a descending run
                const bool up = (tid & size) == 0;
                const bool lower = (tid & stride) == 0;
                const bool other_first = sched_precedes(po, io, pk, ik);
                if (tid < M && (lower == up ? other_first : !other_first)) { pk = po; ik = io; }
            }
        }
        __syncthreads();   // every read of the shared exchange buffers and of sb / si is done
        if (tid < M) { sb[tid] = pk; si[tid] = ik; }
    } else {
        for (int size = 2; size <= M; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int i = tid; i < M; i += nt) {
                    const int l = i ^ stride;
                    if (l > i) {
                        const bool up = (i & size) == 0;
                        const unsigned long long pi_ = sb[i], pl = sb[l];
                        const int ii = si[i], il = si[l];
                        const bool swap = up ? sched_precedes(pl, il, pi_, ii) : sched_precedes(pi_, ii, pl, il);
                        if (swap) { sb[i] = pl; sb[l] = pi_; si[i] = il; si[l] = ii; }
                    }
                }
                __syncthreads();
            }
        }
    }
    __syncthreads();

    // inclusive prefix sums of the sorted P over the first N (each thread a run of R).
    // This GPU's float64 pipe is slow, so only warps holding candidates add, and the
    // warps' offsets come from one shuffle scan of their totals by warp 0.
    const int R = (M + nt - 1) / nt;
    const int r0 = tid * R, r1 = min(N, r0 + R);
    const bool wlive = warp * 32 * R < N;   // this warp's runs hold candidates
    double local = 0.0, excl = 0.0;
    if (wlive) {
        for (int i = r0; i < r1; ++i) local += sp[i];
        double inc = local;   // thread-level inclusive scan of the run totals
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        excl = __shfl_up_sync(0xffffffffu, inc, 1);
        if (lane == 0) excl = 0.0;
        if (lane == 31) s_part[warp] = inc;
    } else if (lane == 0) {
        s_part[warp] = 0.0;
    }
    __syncthreads();
    if (warp == 0) {   // exclusive scan of the warp totals
        const double tot = lane < nt / 32 ? s_part[lane] : 0.0;
        double inc = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        double ex = __shfl_up_sync(0xffffffffu, inc, 1);
        if (lane == 0) ex = 0.0;
        __syncwarp();
        if (lane < nt / 32) s_part[lane] = ex;
    }
    __syncthreads();
    if (wlive) {
        double run = s_part[warp] + excl;   // exclusive prefix of this thread's run
        for (int i = r0; i < r1; ++i) { run += sp[i]; sp[i] = run; }
    }
    __syncthreads();

    // k*: the best E(k) / t[k] over k = 0..K (smallest k on ties), or K
    if (cost == nullptr) {
        if (tid == 0) s_kstar = K;
    } else {
        // only the warps that hold some k take part (k = tid, tid + nt, ...)
        const int nwk = min(nt / 32, K / 32 + 1);
        if (warp < nwk) {
            double best = -DBL_MAX;
            int bk = INT_MAX;
            for (int k = tid; k <= K; k += nt) {
                const float t = cost[k];
                if (!(t > 0.0f) || isinf(t)) continue;
                const double E = (double)B + (k > 0 ? sp[k - 1] : 0.0);
                const double obj = E / (double)t;
                if (obj > best || (obj == best && k < bk)) { best = obj; bk = k; }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const double ob = __shfl_xor_sync(0xffffffffu, best, o);
                const int kb = __shfl_xor_sync(0xffffffffu, bk, o);
                if (ob > best || (ob == best && kb < bk)) { best = ob; bk = kb; }
            }
            if (lane == 0) { s_bobj[warp] = best; s_bk[warp] = bk; }
        }
        __syncthreads();
        if (tid == 0) {
            double b0 = -DBL_MAX;
            int k0 = INT_MAX;
            for (int w = 0; w < nwk; ++w)
                if (s_bobj[w] > b0 || (s_bobj[w] == b0 && s_bk[w] < k0)) { b0 = s_bobj[w]; k0 = s_bk[w]; }
            s_kstar = k0 == INT_MAX ? 0 : k0;   // no usable cost entry: verify nothing
        }
    }
    __syncthreads();
    const int ks = s_kstar;

    // positions per request among the first k* candidates
    for (int i = tid; i < ks; i += nt) atomicAdd(&scount[si[i] / G], 1);
    __syncthreads();
    for (int b = tid; b < B; b += nt) gamma_out[b] = scount[b];
    if (tid == 0 && expected_out) *expected_out = (float)((double)B + (ks > 0 ? sp[ks - 1] : 0.0));
}

size_t verify_budget_smem(int B, int gamma) {
    int M = 1;
    while (M < B * gamma) M <<= 1;
    return (size_t)M * (sizeof(double) + sizeof(int)) + (size_t)B * sizeof(int);
}

cudaError_t verify_budget_launch(const float* conf, int B, int gamma, int budget, const float* cost,
                                 int32_t* gamma_out, float* expected_out, cudaStream_t stream) {
    const size_t smem = verify_budget_smem(B, gamma);
    cudaError_t e = cudaFuncSetAttribute(verify_budget_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    verify_budget_kernel<<<1, kSchedThreads, smem, stream>>>(conf, B, gamma, budget, cost, gamma_out, expected_out);
    return cudaGetLastError();
}

}  // namespace spec
