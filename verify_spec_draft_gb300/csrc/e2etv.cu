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
// GROUP of CTAs, each on a column slice of its 2*Wb rows.  Groups move through
// branches independently; inside a group two bounded barriers (after sweeps 1 and 2)
// exchange per-CTA partials through global memory.  Sweep 2 keeps the q < p test as
// one bit per entry, so the target rows are free after it.
//
// Two plans.  Rows 16-byte aligned, many branches: the sweeps read the rows from
// global memory, sweep 1 from DRAM and sweeps 2 and 3 about half from L2, each lane
// keeping several 16-byte words in flight; about two dozen groups of a few dozen CTAs (four
// per SM) keep that many branches in flight, so one group's barrier waits overlap
// other groups' sweeps.  Otherwise: each CTA stages its slice of all 2*Wb rows in
// shared memory with TMA bulk copies (the next branch's target rows are fetched while
// the group waits at the second barrier, its draft rows once sweep 3 is done), at most
// four groups.  Either way HBM sees each logit read once and each gradient written
// once (6 bytes per entry).
//
// Arithmetic is base 2 on FFMA-scaled logits: p_v = 2^(l_v log2e - LSE2_p), LSE2 the
// log2 of the row normaliser; q_v < p_v is decided on the exponents; min(p, q) =
// 2^(min of the exponents).  Each exponential is one FFMA and one MUFU ex2; the row
// maximum uses packed bf16x2 max with NaN propagation, which also flags invalid rows.
#include <cuda_bf16.h>

#include "spec_device.cuh"
#include "internal.h"

namespace spec {

constexpr int kE2Smem = 110 * 1024;   // staging budget per CTA at two CTAs per SM

// ---------------------------------------------------------------------------------
// 8-entry groups: one 16-byte word of bf16 from shared (staged) or global memory.
// ---------------------------------------------------------------------------------
template <bool STAGED>
__device__ __forceinline__ uint4 ld16(const bf16_t* p) {
    uint4 v;
    if (STAGED) {
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_u32(p)));
    } else {
        v = __ldg(reinterpret_cast<const uint4*>(p));
    }
    return v;
}
// Global rows with an L2 eviction policy: a row read again by a later sweep is kept
// (evict_last), a row at its last read goes first (evict_first), so that the rows of
// the branches in flight stay in L2 while finished rows leave it.
__device__ __forceinline__ uint64_t l2_policy_keep() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_policy_last_use() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
template <bool STAGED>
__device__ __forceinline__ uint4 ld16p(const bf16_t* p, uint64_t pol) {
    if (STAGED) return ld16<true>(p);
    uint4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ float lo_bf(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Scalar path (V not a multiple of 8): the same 8-entry group with -inf past ncol.
__device__ __forceinline__ uint4 ld16_scalar(const bf16_t* row, int k, int ncol) {
    uint32_t h[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        h[e] = (k + e < ncol) ? (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(row) + k + e) : 0xff80u;
    return make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
}

template <bool STAGED, bool VEC>
__device__ __forceinline__ uint4 group8(const bf16_t* row, int k, int ncol) {
    if (VEC) return ld16<STAGED>(row + k);
    return ld16_scalar(row, k, ncol);
}

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Two floats rounded to nearest-even bf16, lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Rows of one branch: staged in shared memory (stride cols) or read from global.
struct Rows {
    const bf16_t* tgt;
    const bf16_t* drf;
    size_t stride;
};

// Sweep 1 for one row slice: (m2, s) with s = sum 2^(x log2e - m2), m2 = max*log2e;
// bad if the slice holds NaN or +inf.
template <bool STAGED, bool VEC>
__device__ __forceinline__ void sweep_stats(const bf16_t* row, int ncol, Stat2& out, int& bad) {
    const int lane = threadIdx.x & 31;
    uint32_t mx2 = 0xff80ff80u;   // (-inf, -inf)
    for (int k = lane * 8; k < ncol; k += 256) {
        const uint4 w = group8<STAGED, VEC>(row, k, ncol);
        mx2 = bmax2(mx2, bmax2(bmax2(w.x, w.y), bmax2(w.z, w.w)));
    }
    float m = fmaxf(lo_bf(mx2), hi_bf(mx2));
    if (isnan(lo_bf(mx2)) || isnan(hi_bf(mx2))) m = NAN;
    // warp max with NaN propagation
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float y = __shfl_xor_sync(0xffffffffu, m, o);
        m = (isnan(m) || isnan(y)) ? NAN : fmaxf(m, y);
    }
    bad = (isnan(m) || m == INFINITY) ? 1 : 0;
    float s0 = 0.0f, s1 = 0.0f;
    const float m2 = m * kLog2e;
    if (!bad && m != -INFINITY) {
        for (int k = lane * 8; k < ncol; k += 256) {
            const uint4 w = group8<STAGED, VEC>(row, k, ncol);
            s0 += ex2(fmaf(lo_bf(w.x), kLog2e, -m2)) + ex2(fmaf(hi_bf(w.x), kLog2e, -m2));
            s1 += ex2(fmaf(lo_bf(w.y), kLog2e, -m2)) + ex2(fmaf(hi_bf(w.y), kLog2e, -m2));
            s0 += ex2(fmaf(lo_bf(w.z), kLog2e, -m2)) + ex2(fmaf(hi_bf(w.z), kLog2e, -m2));
            s1 += ex2(fmaf(lo_bf(w.w), kLog2e, -m2)) + ex2(fmaf(hi_bf(w.w), kLog2e, -m2));
        }
    }
    out = Stat2{(bad || m == -INFINITY) ? -INFINITY : m2, warp_sum(s0 + s1)};
}

// Sweep 2 for one row pair: a = sum min(p, q), s = sum_{q<p} q; the q < p bits of
// each 8-entry group go to mask[k/8].
template <bool STAGED, bool VEC>
__device__ __forceinline__ void sweep_overlap(const bf16_t* tr, const bf16_t* dr, int ncol, float lse_p,
                                              float lse_q, uint8_t* mask, float& a, float& s) {
    const int lane = threadIdx.x & 31;
    float sa = 0.0f, ss = 0.0f;
    for (int k = lane * 8; k < ncol; k += 256) {
        const uint4 wl = group8<STAGED, VEC>(tr, k, ncol);
        const uint4 wd = group8<STAGED, VEC>(dr, k, ncol);
        const uint32_t l4[4] = {wl.x, wl.y, wl.z, wl.w};
        const uint32_t d4[4] = {wd.x, wd.y, wd.z, wd.w};
        uint32_t bits = 0;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const float lp0 = fmaf(lo_bf(l4[h]), kLog2e, -lse_p), lq0 = fmaf(lo_bf(d4[h]), kLog2e, -lse_q);
            const float lp1 = fmaf(hi_bf(l4[h]), kLog2e, -lse_p), lq1 = fmaf(hi_bf(d4[h]), kLog2e, -lse_q);
            const float m0 = ex2(fminf(lp0, lq0)), m1 = ex2(fminf(lp1, lq1));
            sa += m0 + m1;
            if (lq0 < lp0) { ss += m0; bits |= 1u << (2 * h); }
            if (lq1 < lp1) { ss += m1; bits |= 2u << (2 * h); }
        }
        mask[k >> 3] = (uint8_t)bits;
    }
    a = warp_sum(sa);
    s = warp_sum(ss);
}

// Batched variants of the two reductions for 16-byte aligned slices, staged or in
// global memory: each lane keeps B of its 16-byte words in flight at once (instead of
// one load, then its arithmetic, then the next load), and sums go to independent
// accumulators.  Same results up to the order of float additions.
template <int B, bool STAGED>
__device__ __forceinline__ void slice_stats(const bf16_t* row, int ncol, Stat2& out, int& bad, uint64_t pol) {
    // one pass: each lane keeps a running maximum m2 (base 2) and rescales its sums
    // when a batch raises it; the lanes' (m2, s) are merged at the end
    const int lane = threadIdx.x & 31;
    const uint32_t ninf = 0xff80ff80u;
    float m2 = -INFINITY;
    f2x acc0 = f2_pack(0.0f, 0.0f), acc1 = acc0;
    int lbad = 0;
    for (int k0 = lane * 8; k0 < ncol; k0 += 256 * B) {
        uint4 w[B];
        if ((k0 - lane * 8) + 256 * B <= ncol) {   // the warp's whole batch lies in the slice
#pragma unroll
            for (int g = 0; g < B; ++g) w[g] = ld16p<STAGED>(row + k0 + 256 * g, pol);
        } else {
#pragma unroll
            for (int g = 0; g < B; ++g) {
                const int k = k0 + 256 * g;
                w[g] = k < ncol ? ld16p<STAGED>(row + k, pol) : make_uint4(ninf, ninf, ninf, ninf);
            }
        }
        uint32_t mx2 = ninf;
#pragma unroll
        for (int g = 0; g < B; ++g) mx2 = bmax2(mx2, bmax2(bmax2(w[g].x, w[g].y), bmax2(w[g].z, w[g].w)));
        const float bl = lo_bf(mx2), bh = hi_bf(mx2);
        const float bm = fmaxf(bl, bh);
        if (isnan(bl) || isnan(bh) || bm == INFINITY) lbad = 1;
        if (lbad || bm == -INFINITY) continue;   // a batch of -inf adds nothing
        const float bm2 = bm * kLog2e;
        if (bm2 > m2) {
            const float r = ex2(m2 - bm2);          // 0 when m2 was -inf
            const f2x rr = f2_pack(r, r);
            acc0 = f2_mul(acc0, rr);
            acc1 = f2_mul(acc1, rr);
            m2 = bm2;
        }
        // -inf entries contribute 2^-inf = 0; both halves of a word in one packed FMA
        const f2x cl = f2_pack(kLog2e, kLog2e), cm = f2_pack(-m2, -m2);
#pragma unroll
        for (int g = 0; g < B; ++g) {
            acc0 = f2_add(acc0, f2_ex2(f2_fma(bf2_widen(w[g].x), cl, cm)));
            acc1 = f2_add(acc1, f2_ex2(f2_fma(bf2_widen(w[g].y), cl, cm)));
            acc0 = f2_add(acc0, f2_ex2(f2_fma(bf2_widen(w[g].z), cl, cm)));
            acc1 = f2_add(acc1, f2_ex2(f2_fma(bf2_widen(w[g].w), cl, cm)));
        }
    }
    bad = warp_or(lbad);
    const float M = warp_max(m2);
    float s = 0.0f;
    const float2 a0 = f2_unpack(acc0), a1 = f2_unpack(acc1);
    if (!bad && M != -INFINITY && m2 != -INFINITY) s = ((a0.x + a0.y) + (a1.x + a1.y)) * ex2(m2 - M);
    s = warp_sum(s);
    out = Stat2{(bad || M == -INFINITY) ? -INFINITY : M, s};
}

template <int B, bool STAGED>
__device__ __forceinline__ void slice_overlap(const bf16_t* tr, const bf16_t* dr, int ncol, float lse_p, float lse_q,
                                              uint8_t* mask, float& a, float& s, uint64_t pol_t, uint64_t pol_d) {
    const int lane = threadIdx.x & 31;
    const uint32_t ninf = 0xff80ff80u;
    f2x sa = f2_pack(0.0f, 0.0f), ss = sa;
    const f2x cl = f2_pack(kLog2e, kLog2e), cp = f2_pack(-lse_p, -lse_p), cq = f2_pack(-lse_q, -lse_q);
    for (int k0 = lane * 8; k0 < ncol; k0 += 256 * B) {
        uint4 wl[B], wd[B];
        const bool full = (k0 - lane * 8) + 256 * B <= ncol;   // the warp's whole batch lies in the slice
        if (full) {
#pragma unroll
            for (int g = 0; g < B; ++g) {
                wl[g] = ld16p<STAGED>(tr + k0 + 256 * g, pol_t);
                wd[g] = ld16p<STAGED>(dr + k0 + 256 * g, pol_d);
            }
        } else {
#pragma unroll
            for (int g = 0; g < B; ++g) {
                const int k = k0 + 256 * g;
                const bool in = k < ncol;
                wl[g] = in ? ld16p<STAGED>(tr + k, pol_t) : make_uint4(ninf, ninf, ninf, ninf);
                wd[g] = in ? ld16p<STAGED>(dr + k, pol_d) : make_uint4(ninf, ninf, ninf, ninf);
            }
        }
#pragma unroll
        for (int g = 0; g < B; ++g) {
            const uint32_t l4[4] = {wl[g].x, wl[g].y, wl[g].z, wl[g].w};
            const uint32_t d4[4] = {wd[g].x, wd[g].y, wd[g].z, wd[g].w};
            uint32_t bits = 0;
#pragma unroll
            for (int h = 0; h < 4; ++h) {   // exponents of both halves of a word in one packed FMA
                const float2 P = f2_unpack(f2_fma(bf2_widen(l4[h]), cl, cp));
                const float2 Q = f2_unpack(f2_fma(bf2_widen(d4[h]), cl, cq));
                const float m0 = ex2(fminf(P.x, Q.x)), m1 = ex2(fminf(P.y, Q.y));
                const bool b0 = Q.x < P.x, b1 = Q.y < P.y;
                sa = f2_add(sa, f2_pack(m0, m1));
                ss = f2_add(ss, f2_pack(b0 ? m0 : 0.0f, b1 ? m1 : 0.0f));
                bits |= (b0 ? 1u : 0u) << (2 * h);
                bits |= (b1 ? 2u : 0u) << (2 * h);
            }
            const int k = k0 + 256 * g;
            if (full || k < ncol) mask[k >> 3] = (uint8_t)bits;
        }
    }
    const float2 A = f2_unpack(sa), Sx = f2_unpack(ss);
    a = warp_sum(A.x + A.y);
    s = warp_sum(Sx.x + Sx.y);
}

template <bool STAGED, bool VEC>
__global__ void __launch_bounds__(kThreads, STAGED ? 2 : 4) e2etv_kernel(E2etvParams p) {
    extern __shared__ __align__(128) uint8_t s_dyn[];
    const int Wb = p.Wb, nr = 2 * Wb;
    const int g = blockIdx.x / p.group_size;
    const int gi = blockIdx.x - g * p.group_size;
    const long V = p.V;
    const long c0 = (long)gi * p.cols;
    const int ncol = (int)max(0L, min(V, c0 + p.cols) - c0);
    const int ngroups8 = (p.cols + 7) / 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // shared layout: [STAGED: target rows | draft rows] | q<p bits, one byte per 8 entries
    bf16_t* s_tgt = reinterpret_cast<bf16_t*>(s_dyn);
    bf16_t* s_drf = s_tgt + (STAGED ? (size_t)Wb * p.cols : 0);
    uint8_t* s_mask = reinterpret_cast<uint8_t*>(s_drf + (STAGED ? (size_t)Wb * p.cols : 0));
    __shared__ float s_lse[2 * SPEC_MAX_GAMMA];
    __shared__ float s_a[SPEC_MAX_GAMMA], s_s[SPEC_MAX_GAMMA], s_c1[SPEC_MAX_GAMMA], s_c0[SPEC_MAX_GAMMA];
    // per row, the gradient coefficients of a word's two entries for each pair of their
    // q<p bits: entry (lo, hi) takes kappa (s - 1) where its bit is set, kappa s elsewhere
    __shared__ f2x s_ctab[SPEC_MAX_GAMMA][4];
    __shared__ int s_bad;
    __shared__ __align__(8) uint64_t s_bar[2];   // [0] target rows, [1] draft rows
    // the group's barrier: a monotonic arrival count (slot word 0), as for the draft's
    // grid barrier; the last CTA of the launch resets every group's count
    GridBarrier gbar = grid_barrier_init(p.barriers + (size_t)g * 64);
    float2* part = p.partials + (size_t)g * 2 * p.group_size * nr;
    float2* part2 = part + (size_t)p.group_size * nr;
    const double inv_total = 1.0 / ((double)p.total_branches * Wb);
    const unsigned bytes = (unsigned)ncol * 2u;
    unsigned ph_t = 0, ph_d = 0;
    const uint64_t pol_keep = STAGED ? 0ull : l2_policy_keep();
    const uint64_t pol_last = STAGED ? 0ull : l2_policy_last_use();

    // TMA bulk loads of one half (target or draft rows) of branch n's slice
    auto issue = [&](int n, int half) {
        if (!STAGED || ncol == 0 || n >= p.n_branches) return;
        const bf16_t* src = (half == 0 ? p.target : p.draft) + (size_t)n * Wb * V + c0;
        bf16_t* dst = half == 0 ? s_tgt : s_drf;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&s_bar[half], bytes * (unsigned)Wb);
        for (int i = 0; i < Wb; ++i) bulk_g2s(dst + (size_t)i * p.cols, src + (size_t)i * V, bytes, &s_bar[half]);
    };

    if (STAGED) {
        if (threadIdx.x == 0) {
            mbar_init(&s_bar[0], 1);
            mbar_init(&s_bar[1], 1);
            fence_mbar_init();
        }
        __syncthreads();
        if (threadIdx.x == 0) { issue(g, 0); issue(g, 1); }
    }

    for (int n = g; n < p.n_branches; n += p.n_groups) {
        Rows rw;
        if (STAGED) {
            if (ncol > 0) {
                if (!mbar_wait(&s_bar[0], ph_t, p.status, kWaitLimitNs) ||
                    !mbar_wait(&s_bar[1], ph_d, p.status, kWaitLimitNs)) {
                    mbar_wait(&s_bar[0], ph_t, p.status, kWaitLimitNs);   // let copies in flight land
                    mbar_wait(&s_bar[1], ph_d, p.status, kWaitLimitNs);
                    return;
                }
                ph_t ^= 1u;
                ph_d ^= 1u;
            }
            rw.tgt = s_tgt;
            rw.drf = s_drf;
            rw.stride = p.cols;
        } else {
            rw.tgt = p.target + (size_t)n * Wb * V + c0;
            rw.drf = p.draft + (size_t)n * Wb * V + c0;
            rw.stride = V;
        }

        // sweep 1: per-row max and sum-exp of this CTA's slice
        for (int i = warp; i < nr; i += kWarps) {
            Stat2 st;
            int bad = 0;
            if (VEC)
                slice_stats<8, STAGED>((i < Wb ? rw.tgt : rw.drf) + (size_t)(i % Wb) * rw.stride, ncol, st, bad, pol_keep);
            else sweep_stats<STAGED, VEC>((i < Wb ? rw.tgt : rw.drf) + (size_t)(i % Wb) * rw.stride, ncol, st, bad);
            if (lane == 0) {
                part[(size_t)gi * nr + i] = make_float2(st.m2, st.s);
                if (bad) atomicOr(&p.branch_bad[n], 1u);
            }
        }
        if (!grid_barrier(gbar, p.group_size, p.status)) return;

        // the group's partials of every row: LSE2 = log2 of the sum over CTAs of
        // s * 2^(m2 - M) with M the largest m2, plus M.  A warp takes two rows with all
        // their loads in flight (up to 128 CTAs per group; more are read in a loop).
        for (int i0 = warp; i0 < nr; i0 += 2 * kWarps) {
            float2 v[2][4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = i0 + h * kWarps;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c = lane + 32 * u;
                    v[h][u] = (i < nr && c < p.group_size) ? __ldcg(&part[(size_t)c * nr + i])
                                                            : make_float2(-INFINITY, 0.0f);
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = i0 + h * kWarps;
                float M = -INFINITY;
#pragma unroll
                for (int u = 0; u < 4; ++u) M = fmaxf(M, v[h][u].x);
                for (int c = lane + 128; c < p.group_size && i < nr; c += 32) M = fmaxf(M, __ldcg(&part[(size_t)c * nr + i]).x);
                M = warp_max(M);
                float sum = 0.0f;
                if (M != -INFINITY) {
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (v[h][u].x != -INFINITY) sum += v[h][u].y * ex2(v[h][u].x - M);
                    for (int c = lane + 128; c < p.group_size && i < nr; c += 32) {
                        const float2 w = __ldcg(&part[(size_t)c * nr + i]);
                        if (w.x != -INFINITY) sum += w.y * ex2(w.x - M);
                    }
                }
                sum = warp_sum(sum);
                if (lane == 0 && i < nr) s_lse[i] = (M == -INFINITY) ? NAN : M + log2f(sum);
            }
        }
        if (threadIdx.x == 0) s_bad = (__ldcg(&p.branch_bad[n]) != 0u) ? 1 : 0;
        __syncthreads();
        if (threadIdx.x < nr && isnan(s_lse[threadIdx.x])) s_bad = 1;
        __syncthreads();
        const bool bad_branch = s_bad != 0;

        // sweep 2: overlap a and s of every row pair, q<p bits to shared memory
        if (!bad_branch) {
            for (int i = warp; i < Wb; i += kWarps) {
                float a, s;
                if (VEC)
                    slice_overlap<4, STAGED>(rw.tgt + (size_t)i * rw.stride, rw.drf + (size_t)i * rw.stride, ncol, s_lse[i],
                                     s_lse[Wb + i], s_mask + (size_t)i * ngroups8, a, s, pol_last, pol_keep);
                else
                    sweep_overlap<STAGED, VEC>(rw.tgt + (size_t)i * rw.stride, rw.drf + (size_t)i * rw.stride, ncol,
                                               s_lse[i], s_lse[Wb + i], s_mask + (size_t)i * ngroups8, a, s);
                if (lane == 0) part2[(size_t)gi * Wb + i] = make_float2(a, s);
            }
        }
        __syncthreads();                                   // target rows no longer read
        if (threadIdx.x == 0) issue(n + p.n_groups, 0);
        if (!grid_barrier(gbar, p.group_size, p.status)) return;

        if (!bad_branch) {
            for (int i = warp; i < Wb; i += kWarps) {
                float a = 0.0f, s = 0.0f;
                float2 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c = lane + 32 * u;
                    v[u] = c < p.group_size ? __ldcg(&part2[(size_t)c * Wb + i]) : make_float2(0.0f, 0.0f);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) { a += v[u].x; s += v[u].y; }
                for (int c = lane + 128; c < p.group_size; c += 32) {
                    const float2 w = __ldcg(&part2[(size_t)c * Wb + i]);
                    a += w.x;
                    s += w.y;
                }
                a = warp_sum(a);
                s = warp_sum(s);
                if (lane == 0) { s_a[i] = a; s_s[i] = s; }
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                // kappa_i = P_{i-1} * T_i / (N*Wb), T_i = 1 + a_{i+1} T_{i+1}, T_last = 1;
                // grad = q * kappa (s - 1) where q < p, q * kappa s elsewhere
                float T = 1.0f;
                for (int i = Wb - 1; i >= 0; --i) {
                    s_c1[i] = T;
                    if (i > 0) T = 1.0f + s_a[i] * T;
                }
                float P = 1.0f, sum_s = 0.0f;
                for (int i = 0; i < Wb; ++i) {
                    const float kap = (float)((double)(P * s_c1[i]) * inv_total);
                    s_c1[i] = kap * (s_s[i] - 1.0f);
                    s_c0[i] = kap * s_s[i];
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
            if ((int)threadIdx.x < 4 * Wb) {
                const int i = threadIdx.x >> 2, m = threadIdx.x & 3;
                s_ctab[i][m] = f2_pack((m & 1) ? s_c1[i] : s_c0[i], (m & 2) ? s_c1[i] : s_c0[i]);
            }
            __syncthreads();
        } else if (threadIdx.x == 0 && gi == 0) {
            for (int i = 0; i < Wb; ++i) {
                p.a_out[(size_t)n * Wb + i] = NAN;
                p.surv_out[(size_t)n * Wb + i] = NAN;
            }
            p.branch_sum[n] = NAN;
        }

        // sweep 3: gradient w.r.t. the draft logits, rounded once to bf16.  A warp item is
        // 32*U consecutive 8-entry groups of one row (a lane takes U of them, 32 groups
        // apart, with all their loads in flight); the warps step through the items of the
        // slice's Wb rows, so a row's constants and addresses are set once per item.
        {
            constexpr int U = (!STAGED && VEC) ? 4 : 1;
            const int ng = (ncol + 7) / 8;
            const int parts = (ng + 32 * U - 1) / (32 * U);
            const int total = Wb * parts;
            const f2x cl = f2_pack(kLog2e, kLog2e);
            int i = 0, pt = warp;
            if (parts > 0)
                while (pt >= parts) { pt -= parts; ++i; }
            for (int item = warp; item < total; item += kWarps) {
                const bf16_t* src = rw.drf + (size_t)i * rw.stride;
                uint16_t* dst = p.grad_out + ((size_t)n * Wb + i) * V + c0;
                const int g0 = pt * 32 * U + lane;
                uint4 wdu[U];
                const bool full = (pt + 1) * 32 * U <= ng;   // the whole item lies in the slice
                if (full && !bad_branch) {
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int gq = g0 + 32 * u;
                        wdu[u] = VEC ? ld16p<STAGED>(src + (size_t)gq * 8, pol_last) : group8<STAGED, VEC>(src, gq * 8, ncol);
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int gq = g0 + 32 * u;
                        wdu[u] = make_uint4(0u, 0u, 0u, 0u);
                        if (gq < ng && !bad_branch)
                            wdu[u] = VEC ? ld16p<STAGED>(src + (size_t)gq * 8, pol_last) : group8<STAGED, VEC>(src, gq * 8, ncol);
                    }
                }
                const uint8_t* mrow = s_mask + (size_t)i * ngroups8;
                const f2x* ctab = s_ctab[i];
                const float nl = -s_lse[Wb + i];
                const f2x cq = f2_pack(nl, nl);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int gq = g0 + 32 * u;
                    if (full || gq < ng) {
                        const int k = gq * 8;
                        uint4 out = make_uint4(0u, 0u, 0u, 0u);
                        if (!bad_branch) {
                            const uint4 wd = wdu[u];
                            const uint32_t bits = mrow[gq];
                            const uint32_t d4[4] = {wd.x, wd.y, wd.z, wd.w};
                            uint32_t o4[4];
#pragma unroll
                            for (int h = 0; h < 4; ++h) {   // both halves of a word in packed FMA/MUL
                                const f2x q = f2_ex2(f2_fma(bf2_widen(d4[h]), cl, cq));
                                const f2x c = ctab[(bits >> (2 * h)) & 3u];
                                const float2 g = f2_unpack(f2_mul(q, c));
                                o4[h] = pack_bf16x2(g.x, g.y);
                            }
                            out = make_uint4(o4[0], o4[1], o4[2], o4[3]);
                        }
                        uint16_t* d = dst + k;
                        if (VEC) {
                            asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                                         :: "l"(d), "r"(out.x), "r"(out.y), "r"(out.z), "r"(out.w) : "memory");
                        } else {
                            const uint32_t o4[4] = {out.x, out.y, out.z, out.w};
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                if (k + e < ncol) d[e] = (uint16_t)((o4[e >> 1] >> (16 * (e & 1))) & 0xffffu);
                        }
                    }
                }
                pt += kWarps;
                while (pt >= parts) { pt -= parts; ++i; }
            }
        }
        __syncthreads();                                   // draft rows no longer read
        if (threadIdx.x == 0) issue(n + p.n_groups, 1);
    }

    // loss = 1 - mean S, summed over branches in order by the last CTA to finish
    if (!last_block_done(p.done, gridDim.x)) return;
    for (int i = threadIdx.x; i < p.n_groups; i += blockDim.x) p.barriers[(size_t)i * 64] = 0u;
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
            const double M = (double)tot * inv_total;   // this call's part of the mean survival
            *p.loss_out = (float)(p.share_out ? M : 1.0 - M);
            if (bad || isnan(tot)) { *p.loss_out = NAN; atomicOr(p.status, SPEC_DEV_NONFINITE); }
            *p.done = 0u;
        }
    }
}

// ----------------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------------
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int kE2MaxGrid = 1024;
constexpr int kE2MaxPerSm = 6;                         // CTAs per SM of the unstaged plan
// Branch bytes in flight of the unstaged plan: 24 groups for 7-row branches at
// V = 248,320 (6.95 MB each); of 15 to 27 groups measured, 19 to 27 ran within 4 % of
// each other and fewer ran slower.  A branch's target rows are dead after its sweep 2 and its draft
// rows after sweep 3 (both then read evict-first), so the live rows in L2 (129 MB)
// are fewer than this.
constexpr size_t kE2InFlightBytes = (size_t)160 << 20;
constexpr int kE2MaxGroups = 64;                       // one barrier slot per group

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
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    E2etvParams args = p;
    void* kargs[] = {&args};
    return cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(kThreads), kargs, smem, stream);
}

template <bool STAGED, bool VEC>
static int occupancy(size_t smem) {
    auto kern = e2etv_kernel<STAGED, VEC>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
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
    // Rows 16-byte aligned: rows read from global memory (sweep 1 from DRAM, sweeps 2
    // and 3 about half from L2), kE2InFlightBytes of branches in flight (a branch is 2*Wb
    // rows of V bf16 values), each on a group of CTAs, as many CTAs per SM as fit (up
    // to kE2MaxPerSm).  With fewer than eight such groups the plan below is used.
    if (p.vec_ok) {
        int per_sm = occupancy<false, true>(16384);
        if (per_sm > kE2MaxPerSm) per_sm = kE2MaxPerSm;
        int grid = sms * per_sm;
        if (grid > kE2MaxGrid) grid = kE2MaxGrid;
        const size_t branch_bytes = (size_t)2 * p.Wb * (size_t)p.V * sizeof(uint16_t);
        long n_groups = (long)(kE2InFlightBytes / branch_bytes);
        n_groups = n_groups < p.n_branches ? n_groups : p.n_branches;
        n_groups = n_groups < kE2MaxGroups ? n_groups : kE2MaxGroups;
        n_groups = n_groups < grid ? n_groups : grid;
        if (per_sm >= 1 && n_groups >= 8) {
            const int group_size = grid / (int)n_groups;
            long cols = (p.V + group_size - 1) / group_size;
            cols = (cols + 7) / 8 * 8;
            const size_t mask_bytes = align_up((size_t)p.Wb * (size_t)(cols / 8), 16);
            if (occupancy<false, true>(mask_bytes) >= per_sm) {
                p.n_groups = (int)n_groups;
                p.group_size = group_size;
                p.cols = (int)cols;
                return launch_typed<false, true>(p, mask_bytes, (int)n_groups * group_size, stream);
            }
        }
    }
    // Plan: up to four groups.  A staged plan needs every CTA's slice of the 2*Wb rows
    // (plus its q<p bits) within the shared-memory budget, which sets the smallest group.
    for (int per_sm = 2; per_sm >= 1; --per_sm) {
        int grid = sms * per_sm;
        if (grid > kE2MaxGrid) grid = kE2MaxGrid;
        bool staged = false;
        int n_groups = 0, group_size = 0;
        const long budget = per_sm == 2 ? kE2Smem : 2 * kE2Smem;
        const long cols_max = ((budget - 64) * 8 / (32L * p.Wb + p.Wb)) / 8 * 8;
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
        const size_t mask_bytes = align_up((size_t)p.Wb * (size_t)(cols / 8), 16);
        const size_t smem = (staged ? (size_t)2 * p.Wb * cols * sizeof(uint16_t) : 0) + mask_bytes;
        int occ;
        if (staged) occ = occupancy<true, true>(smem);
        else if (p.vec_ok) occ = occupancy<false, true>(smem);
        else occ = occupancy<false, false>(smem);
        if (occ < per_sm) continue;
        p.n_groups = n_groups;
        p.group_size = group_size;
        p.cols = (int)cols;
        grid = n_groups * group_size;
        if (staged) return launch_typed<true, true>(p, smem, grid, stream);
        if (p.vec_ok) return launch_typed<false, true>(p, smem, grid, stream);
        return launch_typed<false, false>(p, smem, grid, stream);
    }
    return cudaErrorInvalidConfiguration;
}

}  // namespace spec
