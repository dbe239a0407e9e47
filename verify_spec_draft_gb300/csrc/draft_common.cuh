// draft_common.cuh - fixed-point pass loop and per-row finalize shared by the draft
// kernels (CUDA-core bias in draft.cu, tcgen05 bias in draft_tc.cu).
//
// The chain x_j = choose(l_j + U[x_{j-1}] W_2) ("Speculative Decoding Part 2", VESSL
// AI, DSpark section, bias equation) is solved as a fixed point: pass k recomputes
// every position from the previous pass's tokens; pass 0 is the unbiased guess.  A
// pass is [tile phase] -> barrier -> [finalize] -> barrier.
//
// Tile phase contract: CTA c owns the contiguous vocabulary tiles
// [tile_begin(c), tile_begin(c+1)) and, for every row, writes one record merging those
// tiles (RowRec: max z, sum 2^(z log2e - fl(max log2e)), argmax, bad flag) to
// p.cta_rec[row * gridDim.x + c]; at T=1 it also writes one record per tile to
// p.tile_rec[row * n_tiles + t] (the inverse CDF locates its draw inside a tile).
// A row whose previous token is invalid is recorded with bad = 2.
#pragma once

#include "spec_device.cuh"
#include "internal.h"

namespace spec {

__device__ __forceinline__ int tile_begin(int c, int nblk, int n_tiles) {
    return (int)(((long)c * n_tiles) / nblk);
}

struct RowAcc {
    float mx;      // max z (-inf when empty)
    float s;       // sum 2^(z log2e - fl(mx log2e))
    int idx;       // lowest index attaining mx
    int bad;
};

__device__ __forceinline__ RowAcc rowacc_empty() { return RowAcc{-INFINITY, 0.0f, 0x7fffffff, 0}; }

__device__ __forceinline__ RowAcc rowacc_merge(RowAcc a, RowAcc b) {
    RowAcc r;
    r.bad = a.bad | b.bad;
    if (b.mx == -INFINITY) { r.mx = a.mx; r.s = a.s; r.idx = a.idx; return r; }
    if (a.mx == -INFINITY) { r.mx = b.mx; r.s = b.s; r.idx = b.idx; return r; }
    r.mx = fmaxf(a.mx, b.mx);
    const float m2 = r.mx * kLog2e;
    r.s = a.s * ex2(a.mx * kLog2e - m2) + b.s * ex2(b.mx * kLog2e - m2);
    r.idx = (a.mx == b.mx) ? min(a.idx, b.idx) : (a.mx > b.mx ? a.idx : b.idx);
    return r;
}

__device__ __forceinline__ float4 rowacc_pack(RowAcc a) {
    return make_float4(a.mx, a.s, __int_as_float(a.idx), __int_as_float(a.bad));
}
__device__ __forceinline__ RowAcc rowacc_unpack(float4 v) {
    return RowAcc{v.x, v.y, __float_as_int(v.z), __float_as_int(v.w)};
}

__device__ __forceinline__ RowAcc warp_rowacc(RowAcc a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        RowAcc b;
        b.mx = __shfl_xor_sync(0xffffffffu, a.mx, o);
        b.s = __shfl_xor_sync(0xffffffffu, a.s, o);
        b.idx = __shfl_xor_sync(0xffffffffu, a.idx, o);
        b.bad = __shfl_xor_sync(0xffffffffu, a.bad, o);
        a = rowacc_merge(a, b);
    }
    return a;
}

// Record of a set of entries held one per lane-slot (four per lane), -inf = absent.
__device__ __forceinline__ RowAcc warp_rowacc_of(const float (&z)[4], const long (&v)[4], long V) {
    float m = -INFINITY;
    int bad = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (v[i] < V) { bad |= bad_logit(z[i]) ? 1 : 0; m = fmaxf(m, z[i]); }
    m = warp_max(m);
    bad = warp_or(bad);
    int idx = 0x7fffffff;
    float s = 0.0f;
    if (m != -INFINITY) {
        const float m2 = m * kLog2e;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (v[i] < V) {
                s += wexp(z[i], m2);
                if (z[i] == m) idx = min(idx, (int)v[i]);
            }
        }
    }
    s = warp_sum(s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) idx = min(idx, __shfl_xor_sync(0xffffffffu, idx, o));
    return RowAcc{m, s, idx, bad};
}

__device__ __forceinline__ int prev_token(const DraftParams& p, const int32_t* prev, int row) {
    const int j = row % p.gamma;
    return j == 0 ? p.anchor[row / p.gamma] : __ldcg(&prev[row - 1]);
}

// z for the four entries v = tile*128 + 32*i + lane of one row, computed on CUDA
// cores: l + sum_k u[k] Wt[v, k] in float32, k ascending.
template <typename WT>
__device__ __forceinline__ float bias_dot(const float* __restrict__ u, const WT* __restrict__ wrow, int r,
                                          bool vec_w) {
    constexpr int N = VecTraits<WT>::N;
    float acc = 0.0f;
    if (vec_w) {
        for (int k = 0; k < r; k += N) {
            float w[N];
            load_vec(wrow + k, w);
#pragma unroll
            for (int e = 0; e < N; ++e) acc = fmaf(u[k + e], w[e], acc);
        }
    } else {
        for (int k = 0; k < r; ++k) acc = fmaf(u[k], load_one(wrow + k), acc);
    }
    return acc;
}

template <typename LT, typename WT>
__device__ __forceinline__ void row_tile_z(const DraftParams& p, int row, int tile, bool use_bias,
                                           const float* u, float (&z)[4], long (&v)[4]) {
    const LT* lrow = static_cast<const LT*>(p.logits) + (size_t)row * p.V;
    const WT* Wt = static_cast<const WT*>(p.Wt);
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[i] = (long)tile * kDraftTile + 32 * i + lane;
        if (v[i] < p.V) {
            float zi = load_one(lrow + v[i]);
            if (use_bias) zi += bias_dot<WT>(u, Wt + (size_t)v[i] * p.r, p.r, p.vec_w != 0);
            z[i] = zi;
        } else {
            z[i] = -INFINITY;
        }
    }
}

// One warp per row: merge the CTA records, choose x_j, write the outputs, flag a
// change against the previous pass.  `s_uw` is this warp's r-float scratch.
template <typename LT, typename WT>
__device__ void finalize_rows(const DraftParams& p, int pass, bool use_bias, const int32_t* prev, int32_t* cur,
                              int nblk_tile, float* s_uw) {
    const int R = p.B * p.gamma;
    const int lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    const int gw = blockIdx.x * nw + (threadIdx.x >> 5);
    const int TW = gridDim.x * nw;
    const WT* U = static_cast<const WT*>(p.U);
    for (int row = gw; row < R; row += TW) {
        const int b = row / p.gamma, j = row % p.gamma;
        const float4* recs = p.cta_rec + (size_t)row * nblk_tile;
        RowAcc acc = rowacc_empty();
#pragma unroll 4
        for (int c = lane; c < nblk_tile; c += 32) acc = rowacc_merge(acc, rowacc_unpack(__ldcg(&recs[c])));
        acc = warp_rowacc(acc);
        const bool valid = !acc.bad && acc.mx != -INFINITY;
        const float M2 = acc.mx * kLog2e;
        const float S = acc.s;     // sum of 2^(z log2e - M2) over the row
        int x = -1;
        float qx = NAN, conf = NAN;
        if (valid) {
            const float wmax = ex2(fmaf(acc.mx, kLog2e, -M2));   // weight of the max entry
            conf = wmax / S;
            if (p.temperature == 0) {
                x = acc.idx;
                qx = conf;
            } else {
                const float u = philox_uniform(p.seeds[b], (uint64_t)b, (uint64_t)(j + 1), 0);
                const float thr = u * S;
                // level 1: CTA ranges, contiguous segments per lane
                const int Kc = (nblk_tile + 31) / 32;
                const int c0 = lane * Kc, c1 = min(nblk_tile, c0 + Kc);
                float seg = 0.0f;
                for (int c = c0; c < c1; ++c) {
                    const RowAcc r = rowacc_unpack(__ldcg(&recs[c]));
                    if (r.mx != -INFINITY) seg += r.s * ex2(r.mx * kLog2e - M2);
                }
                const float incl = warp_inclusive_scan(seg);
                unsigned cross = __ballot_sync(0xffffffffu, incl > thr);
                int cta = -1;
                float tl = INFINITY;
                if (cross) {
                    const int L = __ffs(cross) - 1;
                    if (lane == L) {
                        float run = incl - seg;
                        for (int c = c0; c < c1; ++c) {
                            const RowAcc r = rowacc_unpack(__ldcg(&recs[c]));
                            const float w = (r.mx == -INFINITY) ? 0.0f : r.s * ex2(r.mx * kLog2e - M2);
                            if (run + w > thr) { cta = c; tl = thr - run; break; }
                            run += w;
                        }
                        if (cta < 0) cta = c1 - 1;
                    }
                    cta = __shfl_sync(0xffffffffu, cta, L);
                    tl = __shfl_sync(0xffffffffu, tl, L);
                } else {
                    int last = -1;
                    for (int c = c0; c < c1; ++c) {
                        const RowAcc r = rowacc_unpack(__ldcg(&recs[c]));
                        if (r.mx != -INFINITY && r.s > 0.0f) last = c;
                    }
                    const unsigned has = __ballot_sync(0xffffffffu, last >= 0);
                    cta = has ? __shfl_sync(0xffffffffu, last, 31 - __clz(has)) : 0;
                }
                cta = max(0, min(cta, nblk_tile - 1));
                // level 2: the tiles of that CTA (at most 32 per pass of the warp)
                const int tb = tile_begin(cta, nblk_tile, p.n_tiles), te = tile_begin(cta + 1, nblk_tile, p.n_tiles);
                int tile = -1, last_tile = te - 1;
                float carry = 0.0f;
                for (int t0 = tb; t0 < te && tile < 0; t0 += 32) {
                    const int t = t0 + lane;
                    float w = 0.0f;
                    if (t < te) {
                        const RowAcc r = rowacc_unpack(__ldcg(&p.tile_rec[(size_t)row * p.n_tiles + t]));
                        w = (r.mx == -INFINITY) ? 0.0f : r.s * ex2(r.mx * kLog2e - M2);
                    }
                    const float inc = warp_inclusive_scan(w) + carry;
                    const unsigned hit = __ballot_sync(0xffffffffu, t < te && inc > tl);
                    if (hit) {
                        const int L = __ffs(hit) - 1;
                        tile = t0 + L;
                        const float before = __shfl_sync(0xffffffffu, inc - w, L);
                        tl -= before;
                    }
                    const unsigned pos = __ballot_sync(0xffffffffu, t < te && w > 0.0f);
                    if (pos) last_tile = t0 + 31 - __clz(pos);
                    carry = __shfl_sync(0xffffffffu, inc, 31);
                }
                if (tile < 0) { tile = last_tile; tl = INFINITY; }
                tile = max(0, min(tile, p.n_tiles - 1));
                // level 3: recompute the tile's z on CUDA cores and scan it
                if (use_bias) {
                    const int xp = prev_token(p, prev, row);
                    for (int k = lane; k < p.r; k += 32) s_uw[k] = load_one(U + (size_t)xp * p.r + k);
                    __syncwarp();
                }
                float z[4];
                long v[4];
                row_tile_z<LT, WT>(p, row, tile, use_bias, s_uw, z, v);
                float car = 0.0f, zf = 0.0f, zl = 0.0f;
                int found = -1, last_pos = -1;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float w = (v[i] < p.V) ? wexp(z[i], M2) : 0.0f;
                    const float inc = warp_inclusive_scan(w) + car;
                    const unsigned hit = __ballot_sync(0xffffffffu, w > 0.0f && inc > tl);
                    if (found < 0 && hit) {
                        const int L = __ffs(hit) - 1;
                        found = tile * kDraftTile + 32 * i + L;
                        zf = __shfl_sync(0xffffffffu, z[i], L);
                    }
                    const unsigned pos = __ballot_sync(0xffffffffu, w > 0.0f);
                    if (pos) {
                        const int L = 31 - __clz(pos);
                        last_pos = tile * kDraftTile + 32 * i + L;
                        zl = __shfl_sync(0xffffffffu, z[i], L);
                    }
                    car = __shfl_sync(0xffffffffu, inc, 31);
                }
                if (found < 0) { found = last_pos; zf = zl; }
                x = found;
                qx = wexp(zf, M2) / S;
                __syncwarp();
            }
        }
        if (lane == 0) {
            p.tokens_out[row] = x;
            p.conf_out[row] = conf;
            if (p.qtok_out) p.qtok_out[row] = qx;
            cur[row] = x;
            if (pass > 0 && __ldcg(&prev[row]) != x) atomicOr(&p.changed[pass], 1u);
        }
    }
}

// CUDA-core tile phase: z = l + U[x_prev] . Wt[v] in float32, one warp per row, four
// entries per lane per tile; the CTA's contiguous tile range folded into one record
// per row (and one per tile at T=1).
template <typename LT, typename WT>
__device__ void tile_phase_cc(const DraftParams& p, bool use_bias, const int32_t* prev, float* s_uw) {
    const int R = p.B * p.gamma;
    const int lane = threadIdx.x & 31;
    const WT* U = static_cast<const WT*>(p.U);
    const bool write_z = p.qlogits_out != nullptr && (use_bias || p.r == 0);
    const bool keep_tiles = p.temperature == 1;
    const int tb = tile_begin(blockIdx.x, gridDim.x, p.n_tiles), te = tile_begin(blockIdx.x + 1, gridDim.x, p.n_tiles);
    for (int row = threadIdx.x >> 5; row < R; row += (int)(blockDim.x >> 5)) {
        int prev_ok = 1;
        if (use_bias) {
            const int xp = prev_token(p, prev, row);
            prev_ok = (xp >= 0 && xp < p.V) ? 1 : 0;
            for (int k = lane; k < p.r; k += 32) s_uw[k] = prev_ok ? load_one(U + (size_t)xp * p.r + k) : 0.0f;
            __syncwarp();
        }
        RowAcc acc = rowacc_empty();
        for (int t = tb; t < te; ++t) {
            float z[4];
            long v[4];
            row_tile_z<LT, WT>(p, row, t, use_bias, s_uw, z, v);
            RowAcc tr = warp_rowacc_of(z, v, p.V);
            if (!prev_ok) tr.bad = 2;
            if (keep_tiles && lane == 0) p.tile_rec[(size_t)row * p.n_tiles + t] = rowacc_pack(tr);
            acc = rowacc_merge(acc, tr);
            if (write_z) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (v[i] < p.V) p.qlogits_out[(size_t)row * p.V + v[i]] = z[i];
            }
        }
        if (lane == 0) p.cta_rec[(size_t)row * gridDim.x + blockIdx.x] = rowacc_pack(acc);
        __syncwarp();
    }
}

// Chain validity after the last pass (CTA 0): an anchor outside [0, V) or an invalid
// position voids the rest of the request; sets the status flags.
__device__ __forceinline__ void chain_fixup(const DraftParams& p) {
    for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
        const int a = p.anchor[b];
        bool dead = (a < 0 || a >= p.V);
        unsigned flag = dead ? SPEC_DEV_TOKEN : 0u;
        for (int j = 0; j < p.gamma; ++j) {
            const size_t row = (size_t)b * p.gamma + j;
            if (!dead && __ldcg(&p.tokens_out[row]) < 0) { dead = true; flag |= SPEC_DEV_NONFINITE; }
            if (dead) {
                p.tokens_out[row] = -1;
                p.conf_out[row] = NAN;
                if (p.qtok_out) p.qtok_out[row] = NAN;
            }
        }
        if (flag) atomicOr(p.status, flag);
    }
}

}  // namespace spec
