// e2etv.cu - SpecOPD E2E-TV surrogate and its gradient (spec_e2etv).
//
// Defines: "SpecOPD" paper summary (onedev.kr), section "how to use it" - per-position
// overlap of q and p equal to 1 - TV, loss maximising the mean prefix-survival
// product over branches and positions, gradient through the draft probabilities and
// the prefix products with sampled tokens and target held fixed; "Speculative
// Decoding Part 2" (VESSL AI), DSpark section - alpha = 1 - D_TV.
//
// Every row needs three sweeps: (1) max / sum-exp of p and q, (2) a = sum min(p, q)
// and s = sum_{q<p} q, which need (1)'s normalisers, (3) the gradient, which needs
// kappa and so every a of the branch.  A branch (Wb row pairs) is handled by a
// GROUP of CTAs; each CTA stages its column slice of all 2*Wb rows in shared memory
// once, so HBM sees each logit read once and each gradient written once (6 bytes
// per entry), and the sweeps run from shared memory.  Groups move through branches
// independently; inside a group two bounded barriers (after sweeps 1 and 2) exchange
// per-CTA partials through global memory.  The grid is one cooperative launch with
// several CTAs per SM, so one CTA's barrier wait overlaps another's sweeps.
//
// Exponentials use the log-sum-exp form p_v = exp(l_v - LSE_p); the test q_v < p_v
// is taken on logits, d_v - LSE_q < l_v - LSE_p, and min(p, q) = exp(min(...)).
#include "spec_device.cuh"
#include "internal.h"

namespace spec {

constexpr int kE2Smem = 110 * 1024;   // staging budget per CTA (2 CTAs per SM)

// Reads the 8 elements at columns k..k+7 of a row as float: one 16-byte load from
// shared or global memory on the vector path, else scalar loads with -inf past ncol.
template <bool STAGED, bool VEC>
__device__ __forceinline__ void load8(const bf16_t* row, int k, int ncol, float (&o)[8]) {
    if (!VEC) {
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = (k + e < ncol) ? load_one(row + k + e) : -INFINITY;
        return;
    }
    const bf16_t* p = row + k;
    uint4 v;
    if (STAGED) {
        const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    } else {
        asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    }
    o[0] = __uint_as_float(v.x << 16); o[1] = __uint_as_float(v.x & 0xffff0000u);
    o[2] = __uint_as_float(v.y << 16); o[3] = __uint_as_float(v.y & 0xffff0000u);
    o[4] = __uint_as_float(v.z << 16); o[5] = __uint_as_float(v.z & 0xffff0000u);
    o[6] = __uint_as_float(v.w << 16); o[7] = __uint_as_float(v.w & 0xffff0000u);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const uint32_t a = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t b = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return a | (b << 16);
}

// Row access for one branch: staged rows live in shared memory (row stride `cols`),
// unstaged rows are read from global memory (row stride V).  Columns are relative to
// the CTA's first column c0; `ncol` is a multiple of 8 on the vector path.
struct Rows {
    const bf16_t* tgt;   // row 0 of the target slice
    const bf16_t* drf;   // row 0 of the draft slice
    size_t stride;
};

template <bool STAGED, bool VEC>
__device__ __forceinline__ void sweep_stats(const Rows& rw, int i, bool is_draft, int ncol, Stat& out, int& bad) {
    const int lane = threadIdx.x & 31;
    const bf16_t* row = (is_draft ? rw.drf : rw.tgt) + (size_t)i * rw.stride;
    float m = -INFINITY;
    for (int k = lane * 8; k < ncol; k += 256) {
        float x[8];
        load8<STAGED, VEC>(row, k, ncol, x);
#pragma unroll
        for (int e = 0; e < 8; ++e) { bad |= bad_logit(x[e]) ? 1 : 0; m = fmaxf(m, x[e]); }
    }
    m = warp_max(m);
    float s = 0.0f;
    if (m != -INFINITY) {
        for (int k = lane * 8; k < ncol; k += 256) {
            float x[8];
            load8<STAGED, VEC>(row, k, ncol, x);
#pragma unroll
            for (int e = 0; e < 8; ++e) s += expf(x[e] - m);
        }
    }
    out = Stat{m, warp_sum(s)};
}

template <bool STAGED, bool VEC>
__device__ __forceinline__ void sweep_overlap(const Rows& rw, int i, int ncol, float lse_p, float lse_q,
                                              float& a, float& s) {
    const int lane = threadIdx.x & 31;
    const bf16_t* tr = rw.tgt + (size_t)i * rw.stride;
    const bf16_t* dr = rw.drf + (size_t)i * rw.stride;
    float sa = 0.0f, ss = 0.0f;
    for (int k = lane * 8; k < ncol; k += 256) {
        float l[8], d[8];
        load8<STAGED, VEC>(tr, k, ncol, l);
        load8<STAGED, VEC>(dr, k, ncol, d);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float lp = l[e] - lse_p, lq = d[e] - lse_q;
            const float mn = expf(fminf(lp, lq));
            sa += mn;
            ss += (lq < lp) ? mn : 0.0f;
        }
    }
    a = warp_sum(sa);
    s = warp_sum(ss);
}

template <bool STAGED, bool VEC>
__global__ void __launch_bounds__(kThreads) e2etv_kernel(E2etvParams p) {
    extern __shared__ uint4 s_dyn[];
    bf16_t* s_rows = reinterpret_cast<bf16_t*>(s_dyn);
    const int Wb = p.Wb, nr = 2 * Wb;
    const int g = blockIdx.x / p.group_size;
    const int gi = blockIdx.x - g * p.group_size;
    const long V = p.V;
    const long c0 = (long)gi * p.cols;
    const int ncol = (int)max(0L, min(V, c0 + p.cols) - c0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ float s_lse[2 * SPEC_MAX_GAMMA];
    __shared__ float s_a[SPEC_MAX_GAMMA], s_s[SPEC_MAX_GAMMA], s_kappa[SPEC_MAX_GAMMA];
    __shared__ int s_bad;
    unsigned* bar = p.barriers + (size_t)g * 64;
    float2* part = p.partials + (size_t)g * 2 * p.group_size * nr;
    const double inv_total = 1.0 / ((double)p.n_branches * Wb);
    const bool active = g < p.n_groups;

    for (int n = g; active && n < p.n_branches; n += p.n_groups) {
        const bf16_t* gt = p.target + (size_t)n * Wb * V + c0;
        const bf16_t* gd = p.draft + (size_t)n * Wb * V + c0;
        Rows rw;
        if (STAGED) {
            // stage the slice of the 2*Wb rows (16-byte vector copies)
            const int nv = ncol / 8;
            for (int idx = threadIdx.x; idx < nr * nv; idx += blockDim.x) {
                const int i = idx / nv, k = (idx - i * nv) * 8;
                const bf16_t* src = (i < Wb ? gt : gd) + (size_t)(i % Wb) * V + k;
                uint4 v;
                asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(src));
                *reinterpret_cast<uint4*>(s_rows + (size_t)i * p.cols + k) = v;
            }
            __syncthreads();
            rw.tgt = s_rows;
            rw.drf = s_rows + (size_t)Wb * p.cols;
            rw.stride = p.cols;
        } else {
            rw.tgt = gt;
            rw.drf = gd;
            rw.stride = V;
        }

        // sweep 1: per-row max and sum-exp of this CTA's slice
        for (int i = warp; i < nr; i += kWarps) {
            Stat st;
            int bad = 0;
            sweep_stats<STAGED, VEC>(rw, i % Wb, i >= Wb, ncol, st, bad);
            bad = warp_or(bad);
            if (lane == 0) {
                part[(size_t)gi * nr + i] = make_float2(st.m, st.s);
                if (bad) atomicOr(&p.branch_bad[n], 1u);
            }
        }
        if (!block_barrier(bar, p.group_size, p.status)) return;

        // merge the group's partials in CTA order: LSE of every row
        for (int i = warp; i < nr; i += kWarps) {
            Stat acc = stat_empty();
            for (int c = lane; c < p.group_size; c += 32) {
                const float2 v = __ldcg(&part[(size_t)c * nr + i]);
                acc = stat_merge(acc, Stat{v.x, v.y});
            }
            acc = warp_stat(acc);
            if (lane == 0) s_lse[i] = (acc.m == -INFINITY) ? NAN : acc.m + logf(acc.s);
        }
        if (threadIdx.x == 0) s_bad = (__ldcg(&p.branch_bad[n]) != 0u) ? 1 : 0;
        __syncthreads();
        if (threadIdx.x < nr && isnan(s_lse[threadIdx.x])) s_bad = 1;
        __syncthreads();
        const bool bad_branch = s_bad != 0;

        // sweep 2: overlap a and s of every row pair
        float2* part2 = part + (size_t)p.group_size * nr;
        if (!bad_branch) {
            for (int i = warp; i < Wb; i += kWarps) {
                float a, s;
                sweep_overlap<STAGED, VEC>(rw, i, ncol, s_lse[i], s_lse[Wb + i], a, s);
                if (lane == 0) part2[(size_t)gi * Wb + i] = make_float2(a, s);
            }
        }
        if (!block_barrier(bar, p.group_size, p.status)) return;

        if (!bad_branch) {
            for (int i = warp; i < Wb; i += kWarps) {
                float a = 0.0f, s = 0.0f;
                for (int c = lane; c < p.group_size; c += 32) {
                    const float2 v = __ldcg(&part2[(size_t)c * Wb + i]);
                    a += v.x;
                    s += v.y;
                }
                a = warp_sum(a);
                s = warp_sum(s);
                if (lane == 0) { s_a[i] = a; s_s[i] = s; }
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                // kappa_i = P_{i-1} * T_i / (N*Wb), T_i = 1 + a_{i+1} T_{i+1}, T_last = 1
                float T = 1.0f;
                for (int i = Wb - 1; i >= 0; --i) {
                    s_kappa[i] = T;
                    if (i > 0) T = 1.0f + s_a[i] * T;
                }
                float P = 1.0f, sum_s = 0.0f;
                for (int i = 0; i < Wb; ++i) {
                    s_kappa[i] = (float)((double)(P * s_kappa[i]) * inv_total);
                    P *= s_a[i];
                    sum_s += P;
                    if (gi == 0) {
                        p.a_out[(size_t)n * Wb + i] = s_a[i];
                        p.surv_out[(size_t)n * Wb + i] = P;
                    }
                }
                if (gi == 0) p.branch_sum[n] = sum_s;
            }
            __syncthreads();
        } else if (threadIdx.x == 0 && gi == 0) {
            for (int i = 0; i < Wb; ++i) {
                p.a_out[(size_t)n * Wb + i] = NAN;
                p.surv_out[(size_t)n * Wb + i] = NAN;
            }
            p.branch_sum[n] = NAN;
        }

        // sweep 3: gradient of the loss w.r.t. the draft logits, rounded once to bf16
        {
            const int ng = (ncol + 7) / 8;
            for (int idx = threadIdx.x; idx < Wb * ng; idx += blockDim.x) {
                const int i = idx / ng, k = (idx - i * ng) * 8;
                float gv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if (!bad_branch) {
                    float l[8], d[8];
                    load8<STAGED, VEC>(rw.tgt + (size_t)i * rw.stride, k, ncol, l);
                    load8<STAGED, VEC>(rw.drf + (size_t)i * rw.stride, k, ncol, d);
                    const float lse_p = s_lse[i], lse_q = s_lse[Wb + i];
                    const float kap = -s_kappa[i], si = s_s[i];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float lq = d[e] - lse_q;
                        const float q = expf(lq);
                        const float ind = (lq < l[e] - lse_p) ? 1.0f : 0.0f;
                        gv[e] = kap * q * (ind - si);
                    }
                }
                uint16_t* dst = p.grad_out + ((size_t)n * Wb + i) * V + c0 + k;
                if (VEC) {
                    const uint4 out = make_uint4(pack_bf16x2(gv[0], gv[1]), pack_bf16x2(gv[2], gv[3]),
                                                 pack_bf16x2(gv[4], gv[5]), pack_bf16x2(gv[6], gv[7]));
                    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                                 :: "l"(dst), "r"(out.x), "r"(out.y), "r"(out.z), "r"(out.w) : "memory");
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (k + e < ncol) dst[e] = __bfloat16_as_ushort(__float2bfloat16_rn(gv[e]));
                }
            }
        }
        __syncthreads();   // the next branch overwrites the staged rows
    }

    // loss = 1 - mean S, summed over branches in order by the last CTA to finish
    if (!last_block_done(p.done, gridDim.x)) return;
    if (warp == 0) {
        const int N = p.n_branches;
        const int K = (N + 31) / 32;
        float sum = 0.0f;
        int bad = 0;
        for (int n = lane * K; n < min(N, lane * K + K); ++n) {
            sum += __ldcg(&p.branch_sum[n]);
            bad |= (__ldcg(&p.branch_bad[n]) != 0u) ? 1 : 0;
            p.branch_bad[n] = 0u;
        }
        const float tot = __shfl_sync(0xffffffffu, warp_inclusive_scan(sum), 31);
        bad = warp_or(bad);
        if (lane == 0) {
            *p.loss_out = (float)(1.0 - (double)tot * inv_total);
            if (bad || isnan(tot)) { *p.loss_out = NAN; atomicOr(p.status, SPEC_DEV_NONFINITE); }
            *p.done = 0u;
        }
    }
}

// ----------------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------------
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Upper bound on the grid: 152 SMs x 2 CTAs plus headroom for other parts.
constexpr int kE2MaxGrid = 1024;

size_t e2etv_workspace_bytes(int n_branches, int Wb, int V) {
    (void)V;
    size_t off = kWsHeaderBytes;
    off = align_up(off + sizeof(float2) * 2 * (size_t)kE2MaxGrid * 2 * Wb, 256);
    off = align_up(off + sizeof(float) * (size_t)n_branches, 256);
    off = align_up(off + sizeof(unsigned) * (size_t)n_branches, 256);
    return off;
}

template <bool STAGED, bool VEC>
static cudaError_t launch_typed(E2etvParams& p, size_t smem, int grid, cudaStream_t stream) {
    auto kern = e2etv_kernel<STAGED, VEC>;
    if (smem > 0) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    E2etvParams args = p;
    void* kargs[] = {&args};
    return cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(kThreads), kargs, smem, stream);
}

template <bool STAGED, bool VEC>
static int occupancy(size_t smem) {
    auto kern = e2etv_kernel<STAGED, VEC>;
    if (smem > 0 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return 0;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem) != cudaSuccess) return 0;
    return occ;
}

cudaError_t e2etv_launch(E2etvParams& p, void* ws, cudaStream_t stream) {
    char* w = static_cast<char*>(ws);
    WsHeader* h = reinterpret_cast<WsHeader*>(w);
    p.status = &h->status;
    p.done = &h->done[0];
    p.barriers = &h->barrier[0][0];
    size_t off = kWsHeaderBytes;
    p.partials = reinterpret_cast<float2*>(w + off);
    off = align_up(off + sizeof(float2) * 2 * (size_t)kE2MaxGrid * 2 * p.Wb, 256);
    p.branch_sum = reinterpret_cast<float*>(w + off);
    off = align_up(off + sizeof(float) * (size_t)p.n_branches, 256);
    p.branch_bad = reinterpret_cast<unsigned*>(w + off);

    const int sms = device_sm_count();
    // Plan: up to four groups; a staged plan needs every CTA's slice of the 2*Wb rows
    // within the shared-memory budget, which sets the smallest group.
    for (int per_sm = 2; per_sm >= 1; --per_sm) {
        int grid = sms * per_sm;
        if (grid > kE2MaxGrid) grid = kE2MaxGrid;
        bool staged = false;
        int n_groups = 0, group_size = 0;
        const long budget = per_sm == 2 ? kE2Smem : 2 * kE2Smem;
        const long cols_max = (budget / (4L * p.Wb)) / 8 * 8;
        if (p.vec_ok && cols_max >= 64) {
            const long need = (p.V + cols_max - 1) / cols_max;
            if (need <= grid) {
                n_groups = (int)(grid / need);
                if (n_groups > 4) n_groups = 4;
                if (n_groups > p.n_branches) n_groups = p.n_branches;
                group_size = grid / n_groups;
                staged = true;
            }
        }
        if (!staged) {
            n_groups = p.n_branches < 4 ? p.n_branches : 4;
            group_size = grid / n_groups;
        }
        long cols = (p.V + group_size - 1) / group_size;
        cols = (cols + 7) / 8 * 8;
        const size_t smem = staged ? (size_t)2 * p.Wb * cols * sizeof(uint16_t) : 0;
        int occ;
        if (staged) occ = occupancy<true, true>(smem);
        else if (p.vec_ok) occ = occupancy<false, true>(0);
        else occ = occupancy<false, false>(0);
        if (occ < per_sm) continue;
        p.n_groups = n_groups;
        p.group_size = group_size;
        p.cols = (int)cols;
        grid = n_groups * group_size;
        if (staged) return launch_typed<true, true>(p, smem, grid, stream);
        if (p.vec_ok) return launch_typed<false, true>(p, 0, grid, stream);
        return launch_typed<false, false>(p, 0, grid, stream);
    }
    return cudaErrorInvalidConfiguration;
}

}  // namespace spec
