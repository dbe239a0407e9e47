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

__device__ __forceinline__ float fmax_nan_f(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// Drafter logits of 32 consecutive entries (v0 a multiple of 32, rows 16-byte aligned,
// V a multiple of the vector width): LW 16-byte words, -inf past V.
template <typename LT> struct LWords { static constexpr int N = 32 * (int)sizeof(LT) / 16; };

// L32: the row's bytes are 32-byte aligned and V is a multiple of 32 bytes' worth of
// entries, so the words come two at a time, one 32-byte load (a whole sector) each.  A
// thread reads along its own row, so an L2 miss fetches the row's whole 256-byte block
// (`L2::256B`), which the thread's next loads then find in L2.
template <typename LT, bool L32 = false>
__device__ __forceinline__ void load_l32(const LT* row, long v0, long V, uint4 (&w)[LWords<LT>::N]) {
    constexpr int N = LWords<LT>::N, EPV = 32 / N;
    const uint32_t ninf = sizeof(LT) == 2 ? 0xff80ff80u : 0xff800000u;
    if constexpr (L32) {
#pragma unroll
        for (int i = 0; i < N; i += 2) {
            const long v = v0 + EPV * i;
            if (v + 2 * EPV <= V) {
                asm volatile("ld.global.nc.L2::256B.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                             : "=r"(w[i].x), "=r"(w[i].y), "=r"(w[i].z), "=r"(w[i].w), "=r"(w[i + 1].x),
                               "=r"(w[i + 1].y), "=r"(w[i + 1].z), "=r"(w[i + 1].w)
                             : "l"(row + v));
            } else {
                w[i] = make_uint4(ninf, ninf, ninf, ninf);
                w[i + 1] = w[i];
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const long v = v0 + EPV * i;
            w[i] = (v + EPV <= V) ? __ldg(reinterpret_cast<const uint4*>(row + v)) : make_uint4(ninf, ninf, ninf, ninf);
        }
    }
}
// z[e] += logit e, in place, two entries per float32x2 add (each half rounds as the
// scalar add would)
__device__ __forceinline__ void add_pair(float& z0, float& z1, f2x l) {
    const float2 r = f2_unpack(f2_add(f2_pack(z0, z1), l));
    z0 = r.x;
    z1 = r.y;
}
template <typename LT>
__device__ __forceinline__ void add_l32(const uint4 (&w)[LWords<LT>::N], float (&z)[32]) {
    if (sizeof(LT) == 2) {
#pragma unroll
        for (int i = 0; i < LWords<LT>::N; ++i) {
            const uint32_t a[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) add_pair(z[(8 * i + 2 * k) & 31], z[(8 * i + 2 * k + 1) & 31], bf2_widen(a[k]));
        }
    } else {
#pragma unroll
        for (int i = 0; i < LWords<LT>::N; ++i) {
            add_pair(z[(4 * i) & 31], z[(4 * i + 1) & 31], f2_pack(__uint_as_float(w[i].x), __uint_as_float(w[i].y)));
            add_pair(z[(4 * i + 2) & 31], z[(4 * i + 3) & 31], f2_pack(__uint_as_float(w[i].z), __uint_as_float(w[i].w)));
        }
    }
}

// Record of 32 consecutive entries of one row held by one thread.  The lowest index
// of the maximum is needed only when this chunk raises the running maximum `run_mx`
// (entries are visited in increasing order, so on a tie the earlier index stands);
// `want_idx` is false when no argmax is used (T=1).
// The maximum is a tree of NaN-propagating maxima (exact in any order); the sum keeps
// the even and the odd entries in the two halves of a float32x2 accumulator, each in
// increasing order, and adds the halves at the end.
__device__ __forceinline__ RowAcc record32(const float (&z)[32], int v0, float run_mx, bool want_idx) {
    float t[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) t[e] = fmax_nan_f(z[2 * e], z[2 * e + 1]);
#pragma unroll
    for (int w = 8; w > 0; w >>= 1)
#pragma unroll
        for (int e = 0; e < w; ++e) t[e] = fmax_nan_f(t[e], t[e + w]);
    const float m = t[0];
    RowAcc r;
    r.bad = (isnan(m) || m == INFINITY) ? 1 : 0;
    r.mx = r.bad ? -INFINITY : m;
    r.s = 0.0f;
    r.idx = 0x7fffffff;
    if (!r.bad && m != -INFINITY) {
        const float m2 = m * kLog2e;
        const f2x k2 = f2_pack(kLog2e, kLog2e), nm2 = f2_pack(-m2, -m2);
        f2x acc = f2_pack(0.0f, 0.0f);
#pragma unroll
        for (int e = 0; e < 32; e += 2) acc = f2_add(acc, f2_ex2(f2_fma(f2_pack(z[e], z[e + 1]), k2, nm2)));
        const float2 s2 = f2_unpack(acc);
        r.s = s2.x + s2.y;
        if (want_idx && m > run_mx) {
#pragma unroll
            for (int e = 31; e >= 0; --e)
                if (z[e] == m) r.idx = v0 + e;
        }
    }
    return r;
}

// 64-bit argmax key of a row record: the ordered maximum in the high word, the
// inverted index in the low word, so the largest key is the largest value at its
// lowest index, as rowacc_merge decides; all ones for a row without a distribution.
// The CTAs' keys of a row are folded with a relaxed red.max (the grid barrier that
// follows orders them), one key per 128-byte line.
constexpr int kKeyStride = 16;
__device__ __forceinline__ unsigned long long rec_key(const RowAcc& a) {
    return a.bad ? ~0ull : argmax_key(a.mx, (uint32_t)a.idx);
}
__device__ __forceinline__ void red_max_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
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

// x_{j-1} of a row: the anchor at j = 0, else the previous pass's token of the row
// before (in shared or global memory; read with a relaxed load so a token another CTA
// wrote is seen).
__device__ __forceinline__ int prev_token(const DraftParams& p, const int32_t* prev, int row, const int32_t* anc) {
    const int j = row % p.gamma;
    return j == 0 ? anc[row / p.gamma] : ld_relaxed_i32(&prev[row - 1]);
}
__device__ __forceinline__ int prev_token(const DraftParams& p, const int32_t* prev, int row) {
    return prev_token(p, prev, row, p.anchor);
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

// The bias of one tile's 128 entries for bf16 weight rows of r <= 256 values in whole
// 16-byte words: lane l takes the rank slice [8l, 8l + 8) of every entry, so each
// entry's Wt row is one coalesced warp load, kZBatch rows are in flight at once, and
// the lanes' partial dot products are summed across the warp (the same bits in every
// lane).  Lane l ends with the bias of entries 32i + l.
constexpr int kZBatch = 8;
__device__ __forceinline__ void tile_bias_bf16(const DraftParams& p, int tile, const float* u, float (&zb)[4]) {
    const bf16_t* Wt = static_cast<const bf16_t*>(p.Wt);
    const int lane = threadIdx.x & 31;
    const bool has = lane < (p.r >> 3);
    {   // the tile's Wt rows are contiguous: one bulk request into L2 ahead of the loads
        const long v0 = (long)tile * kDraftTile;
        const long v1 = v0 + kDraftTile < p.V ? v0 + kDraftTile : p.V;
        if (lane == 0 && v1 > v0) bulk_prefetch_l2(Wt + (size_t)v0 * p.r, (unsigned)((v1 - v0) * p.r * 2));
    }
    float uu[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) uu[e] = has ? u[lane * 8 + e] : 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float mine = 0.0f;
#pragma unroll 1
        for (int h = 0; h < 32 / kZBatch; ++h) {
            const long base = (long)tile * kDraftTile + 32 * i + h * kZBatch;
            uint4 w[kZBatch];
#pragma unroll
            for (int q = 0; q < kZBatch; ++q) {
                w[q] = make_uint4(0u, 0u, 0u, 0u);
                if (has && base + q < p.V)
                    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(w[q].x), "=r"(w[q].y), "=r"(w[q].z), "=r"(w[q].w)
                                 : "l"(Wt + (size_t)(base + q) * p.r + lane * 8));
            }
#pragma unroll
            for (int q = 0; q < kZBatch; ++q) {
                const uint32_t a[4] = {w[q].x, w[q].y, w[q].z, w[q].w};
                float part = 0.0f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    part = fmaf(uu[2 * k], __uint_as_float(a[k] << 16), part);
                    part = fmaf(uu[2 * k + 1], __uint_as_float(a[k] & 0xffff0000u), part);
                }
                part = warp_sum(part);
                if (lane == h * kZBatch + q) mine = part;
            }
        }
        zb[i] = mine;
    }
}

template <typename LT, typename WT>
__device__ __forceinline__ void row_tile_z(const DraftParams& p, int row, int tile, bool use_bias,
                                           const float* u, float (&z)[4], long (&v)[4]) {
    const LT* lrow = static_cast<const LT*>(p.logits) + (size_t)row * p.V;
    const WT* Wt = static_cast<const WT*>(p.Wt);
    const int lane = threadIdx.x & 31;
    if (sizeof(WT) == 2 && use_bias && p.vec_w && (p.r & 7) == 0 && p.r <= 256) {
        float zb[4];
        tile_bias_bf16(p, tile, u, zb);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[i] = (long)tile * kDraftTile + 32 * i + lane;
            z[i] = v[i] < p.V ? load_one(lrow + v[i]) + zb[i] : -INFINITY;
        }
        return;
    }
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

// The T=1 draw's first two levels for one row (one warp; every lane gets the result):
// the CTA range in which the row's CDF (the CTA records' weights, in index order)
// crosses thr, then the tile of that range, and what is left of thr at that tile's
// start (INFINITY when rounding leaves no crossing, with the last tile of weight).
__device__ __forceinline__ void draw_locate(const DraftParams& p, const float4* recs, int row, int nblk_tile,
                                            float M2, float thr, int& tile_out, float& tl_out) {
    const int lane = threadIdx.x & 31;
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
        // lane L's segment (Kc <= 32 records), one record per lane, scanned in one go
        const int L = __ffs(cross) - 1;
        const float before = __shfl_sync(0xffffffffu, incl - seg, L);
        const int s0 = L * Kc, s1 = min(nblk_tile, s0 + Kc);
        const int c = s0 + lane;
        float w = 0.0f;
        if (c < s1) {
            const RowAcc r = rowacc_unpack(__ldcg(&recs[c]));
            if (r.mx != -INFINITY) w = r.s * ex2(r.mx * kLog2e - M2);
        }
        const float inc = warp_inclusive_scan(w) + before;
        const unsigned hit = __ballot_sync(0xffffffffu, c < s1 && w > 0.0f && inc > thr);
        if (hit) {
            const int H = __ffs(hit) - 1;
            cta = s0 + H;
            tl = thr - __shfl_sync(0xffffffffu, inc - w, H);
        } else {
            cta = s1 - 1;
        }
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
    tile_out = tile;
    tl_out = tl;
}

// The draw's last level: the tile's entries in index order (lane l holds entries
// 32i + l as z[i]); returns the entry where the running weight passes tl, or the last
// entry of positive weight, and its z.
__device__ __forceinline__ void draw_scan_tile(const float (&z)[4], const long (&v)[4], long V, float M2, float tl,
                                               int tile, int& found_out, float& zf_out) {
    float car = 0.0f, zf = 0.0f, zl = 0.0f;
    int found = -1, last_pos = -1;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float w = (v[i] < V) ? wexp(z[i], M2) : 0.0f;
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
    found_out = found;
    zf_out = zf;
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
                const float u = philox_uniform(p.seeds[b], (uint64_t)(p.b_base + b), (uint64_t)(j + 1), 0);
                const float thr = u * S;
                int tile = 0;
                float tl = INFINITY;
                draw_locate(p, recs, row, nblk_tile, M2, thr, tile, tl);
                // level 3: recompute the tile's z on CUDA cores and scan it
                if (use_bias) {
                    const int xp = prev_token(p, prev, row);
                    for (int k = lane; k < p.r; k += 32) s_uw[k] = load_one(U + (size_t)xp * p.r + k);
                    __syncwarp();
                }
                float z[4];
                long v[4];
                row_tile_z<LT, WT>(p, row, tile, use_bias, s_uw, z, v);
                int found = -1;
                float zf = 0.0f;
                draw_scan_tile(z, v, p.V, M2, tl, tile, found, zf);
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

// T=1 draws after a biased pass with bf16 weight rows of whole 16-byte words (r <= 256):
// a group of kDrawWarps warps per row.  Every warp of the group merges the row's
// records and locates the tile itself (the same loads, so the same decisions); each
// then computes kDraftTile / kDrawWarps of the tile's biased logits (the rank split
// over its lanes) into the group's kDraftTile floats of `s_z`, and after a named
// barrier the group's first warp scans them.  Rows go to CTAs first (row r to CTA
// r % gridDim.x), so every SM takes a share of the rows.  Warps beyond the last whole
// group take no part.
constexpr int kDrawWarps = 8;
constexpr int kDrawBarrier = 9;   // named barrier of group g: kDrawBarrier + g
__device__ __forceinline__ void draw_group_sync(int grp) {
    asm volatile("bar.sync %0, %1;" :: "r"(kDrawBarrier + grp), "r"(32 * kDrawWarps) : "memory");
}

template <typename LT>
__device__ void finalize_rows_t1g(const DraftParams& p, int pass, const int32_t* prev, int32_t* cur, int nblk_tile,
                                  float* s_z, const uint8_t* act = nullptr) {
    constexpr int EPW = kDraftTile / kDrawWarps;   // entries of the tile per warp
    const int R = p.B * p.gamma;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ngrp = (blockDim.x >> 5) / kDrawWarps;
    const int grp = warp / kDrawWarps, gw = warp % kDrawWarps;
    if (grp >= ngrp) return;
    float* z_s = s_z + (size_t)grp * kDraftTile;
    const bf16_t* U = static_cast<const bf16_t*>(p.U);
    const bf16_t* Wt = static_cast<const bf16_t*>(p.Wt);
    const bool has = lane < (p.r >> 3);
    for (int row = grp * gridDim.x + blockIdx.x; row < R; row += gridDim.x * ngrp) {
        if (act != nullptr && !act[row]) {
            // the row's predecessor kept its token: so does the row (its outputs stand)
            if (gw == 0 && lane == 0) cur[row] = __ldcg(&prev[row]);
            continue;
        }
        const int b = row / p.gamma, j = row % p.gamma;
        const float4* recs = p.cta_rec + (size_t)row * nblk_tile;
        const LT* lrow = static_cast<const LT*>(p.logits) + (size_t)row * p.V;
        // x_{j-1}'s U row is requested first: its two dependent loads overlap the record
        // merge and the search
        const int xp = prev_token(p, prev, row);
        uint4 uw = make_uint4(0u, 0u, 0u, 0u);
        if (has && xp >= 0 && xp < p.V)   // a valid row always has a valid previous token
            uw = __ldg(reinterpret_cast<const uint4*>(U + (size_t)xp * p.r) + lane);
        RowAcc acc = rowacc_empty();
#pragma unroll 4
        for (int c = lane; c < nblk_tile; c += 32) acc = rowacc_merge(acc, rowacc_unpack(__ldcg(&recs[c])));
        acc = warp_rowacc(acc);
        const bool valid = !acc.bad && acc.mx != -INFINITY;
        const float M2 = acc.mx * kLog2e;
        const float S = acc.s;
        int tile = 0;
        float tl = INFINITY;
        if (valid) {
            const float u = philox_uniform(p.seeds[b], (uint64_t)(p.b_base + b), (uint64_t)(j + 1), 0);
            draw_locate(p, recs, row, nblk_tile, M2, u * S, tile, tl);
            const long e0 = (long)tile * kDraftTile + gw * EPW;
            const long e1 = e0 + EPW < p.V ? e0 + EPW : p.V;
            if (lane == 0 && e1 > e0) bulk_prefetch_l2(Wt + (size_t)e0 * p.r, (unsigned)((e1 - e0) * p.r * 2));
            float uu[8];
            {
                const uint32_t a[4] = {uw.x, uw.y, uw.z, uw.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    uu[2 * k] = __uint_as_float(a[k] << 16);
                    uu[2 * k + 1] = __uint_as_float(a[k] & 0xffff0000u);
                }
            }
#pragma unroll 1
            for (int h = 0; h < EPW / kZBatch; ++h) {
                const long base = e0 + h * kZBatch;
                uint4 w[kZBatch];
#pragma unroll
                for (int q = 0; q < kZBatch; ++q) {
                    w[q] = make_uint4(0u, 0u, 0u, 0u);
                    if (has && base + q < p.V)
                        asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                                     : "=r"(w[q].x), "=r"(w[q].y), "=r"(w[q].z), "=r"(w[q].w)
                                     : "l"(Wt + (size_t)(base + q) * p.r + lane * 8));
                }
                float zl = 0.0f;
                if (lane < kZBatch && base + lane < p.V) zl = load_one(lrow + base + lane);
#pragma unroll
                for (int q = 0; q < kZBatch; ++q) {
                    const uint32_t a[4] = {w[q].x, w[q].y, w[q].z, w[q].w};
                    float part = 0.0f;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        part = fmaf(uu[2 * k], __uint_as_float(a[k] << 16), part);
                        part = fmaf(uu[2 * k + 1], __uint_as_float(a[k] & 0xffff0000u), part);
                    }
                    part = warp_sum(part);
                    if (lane == q) z_s[gw * EPW + h * kZBatch + q] = base + q < p.V ? zl + part : -INFINITY;
                }
            }
        }
        draw_group_sync(grp);
        if (gw == 0) {
            int x = -1;
            float qx = NAN, conf = NAN;
            if (valid) {
                conf = ex2(fmaf(acc.mx, kLog2e, -M2)) / S;
                float z[4];
                long v[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[i] = (long)tile * kDraftTile + 32 * i + lane;
                    z[i] = v[i] < p.V ? z_s[32 * i + lane] : -INFINITY;
                }
                int found = -1;
                float zf = 0.0f;
                draw_scan_tile(z, v, p.V, M2, tl, tile, found, zf);
                x = found;
                qx = wexp(zf, M2) / S;
            }
            if (lane == 0) {
                p.tokens_out[row] = x;
                p.conf_out[row] = conf;
                if (p.qtok_out) p.qtok_out[row] = qx;
                cur[row] = x;
                if (pass > 0 && __ldcg(&prev[row]) != x) atomicOr(&p.changed[pass], 1u);
            }
        }
        draw_group_sync(grp);   // the group's z_s is free for its next row
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

// Pass 0 at T=0: only the argmax of the unbiased rows is used when a biased pass
// follows (need_s false), so each lane keeps a running (max, lowest index) and, if
// need_s, a running sum rescaled when the max grows; one warp reduction per row.
template <typename LT>
__device__ void tile_phase_stream0_t0(const DraftParams& p, float4* rec_out, bool need_s, unsigned long long* keys) {
    constexpr int EPL = 16 / (int)sizeof(LT);
    constexpr int UNIT = 32 * EPL;
    const int R = p.B * p.gamma;
    const int lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    const int tb = tile_begin(blockIdx.x, gridDim.x, p.n_tiles), te = tile_begin(blockIdx.x + 1, gridDim.x, p.n_tiles);
    const long e_begin = (long)tb * kDraftTile, e_end = (long)te * kDraftTile;
    const int upr = (int)((e_end - e_begin + UNIT - 1) / UNIT);
    for (int row = threadIdx.x >> 5; row < R; row += nw) {
        const LT* lrow = static_cast<const LT*>(p.logits) + (size_t)row * p.V;
        float m = -INFINITY, s = 0.0f, mall = -INFINITY;
        int idx = 0x7fffffff, bad = 0;
        for (int u0 = 0; u0 < upr; u0 += 8) {
            uint4 w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const long e0 = e_begin + (long)(u0 + k) * UNIT + (long)lane * EPL;
                w[k] = (u0 + k < upr && e0 < e_end && e0 + EPL <= p.V)
                           ? __ldg(reinterpret_cast<const uint4*>(lrow + e0))
                           : (sizeof(LT) == 2 ? make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u)
                                              : make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u));
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const long e0 = e_begin + (long)(u0 + k) * UNIT + (long)lane * EPL;
                if (!need_s) {
                    // argmax only: one packed NaN-propagating maximum per word; the
                    // entries are looked at only when the word raises the lane's maximum
                    // (a lane visits its words in increasing index order, so on a tie
                    // the earlier index stands)
                    const float m8 = u4_max_nan<(int)sizeof(LT)>(w[k]);
                    mall = f_max_nan(mall, m8);
                    if (m8 > m) {
                        m = m8;
                        if (sizeof(LT) == 2) {
                            const uint32_t a[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
                            for (int h = 3; h >= 0; --h) {
                                if (__uint_as_float(a[h] & 0xffff0000u) == m8) idx = (int)(e0 + 2 * h + 1);
                                if (__uint_as_float(a[h] << 16) == m8) idx = (int)(e0 + 2 * h);
                            }
                        } else {
                            const uint32_t a[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
                            for (int h = 3; h >= 0; --h)
                                if (__uint_as_float(a[h]) == m8) idx = (int)(e0 + h);
                        }
                    }
                    continue;
                }
                float x[EPL];
                if (sizeof(LT) == 2) {
                    const uint32_t a[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        x[(2 * h) % EPL] = __uint_as_float(a[h] << 16);
                        x[(2 * h + 1) % EPL] = __uint_as_float(a[h] & 0xffff0000u);
                    }
                } else {
                    x[0] = __uint_as_float(w[k].x);
                    x[1 % EPL] = __uint_as_float(w[k].y);
                    x[2 % EPL] = __uint_as_float(w[k].z);
                    x[3 % EPL] = __uint_as_float(w[k].w);
                }
                float m8 = x[0];
#pragma unroll
                for (int e = 1; e < EPL; ++e) m8 = fmaxf(m8, x[e]);
#pragma unroll
                for (int e = 0; e < EPL; ++e) bad |= bad_logit(x[e]) ? 1 : 0;
                if (m8 > m) {
                    if (need_s && m != -INFINITY) s *= ex2(m * kLog2e - m8 * kLog2e);
                    m = m8;
#pragma unroll
                    for (int e = EPL - 1; e >= 0; --e)
                        if (x[e] == m8) idx = (int)(e0 + e);
                } else if (m8 == m && m != -INFINITY) {
#pragma unroll
                    for (int e = EPL - 1; e >= 0; --e)
                        if (x[e] == m8) idx = min(idx, (int)(e0 + e));
                }
                if (need_s && m != -INFINITY) {
                    const float m2 = m * kLog2e;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) s += wexp(x[e], m2);
                }
            }
        }
        if (!need_s) bad = (isnan(mall) || mall == INFINITY) ? 1 : 0;
        RowAcc a{bad ? -INFINITY : m, need_s ? s : 0.0f, idx, bad};
        a = warp_rowacc(a);
        if (lane == 0) {
            rec_out[(size_t)row * gridDim.x + blockIdx.x] = rowacc_pack(a);
            if (keys) red_max_u64(&keys[(size_t)row * kKeyStride], rec_key(a));
        }
    }
}

// The entries of one 16-byte word of logits as float32.
template <typename LT>
__device__ __forceinline__ void unpack_word(const uint4& w, float (&x)[16 / sizeof(LT)]) {
    if constexpr (sizeof(LT) == 2) {
        const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[2 * k] = __uint_as_float(a[k] << 16);
            x[2 * k + 1] = __uint_as_float(a[k] & 0xffff0000u);
        }
    } else {
        x[0] = __uint_as_float(w.x);
        x[1] = __uint_as_float(w.y);
        x[2] = __uint_as_float(w.z);
        x[3] = __uint_as_float(w.w);
    }
}

// Pass 0 at T=1 (unbiased rows) on rows of whole 16-byte words: the per-(row, tile)
// records of the draw and one record per (row, CTA); no argmax is kept, since T=1
// draws.  A warp holds one row's slice of this CTA's tile range in registers (at most
// kS1Units units of 32 words, one word per lane: 256 bf16 or 128 float32 entries).  The
// slice maximum takes a packed NaN-propagating maximum per word (a NaN or +inf entry
// shows as a NaN or +inf maximum) and one warp reduction; each tile's sum against it
// takes the exponent arguments and sums two entries at a time (float32x2), then a
// reduction over the tile's lanes.  Records carry the slice maximum as their reference.
// Each warp requests its rows' slices into L2 kS1Ahead rows ahead of their loads.
constexpr int kS1Units = 8;
constexpr int kS1Ahead = 3;
template <typename LT>
__device__ bool stream0_t1_rows(const DraftParams& p) {
    constexpr int EPL = 16 / (int)sizeof(LT);          // entries per lane per unit
    constexpr int UNIT = 32 * EPL;                     // entries per unit
    constexpr int TPU = UNIT / kDraftTile;             // tiles per unit (1 or 2)
    constexpr int LPT = 32 / TPU;                      // lanes per tile
    const int R = p.B * p.gamma;
    const int lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    const int tb = tile_begin(blockIdx.x, gridDim.x, p.n_tiles), te = tile_begin(blockIdx.x + 1, gridDim.x, p.n_tiles);
    const long e_begin = (long)tb * kDraftTile, e_end = (long)te * kDraftTile;
    const int upr = (int)((e_end - e_begin + UNIT - 1) / UNIT);
    if (upr > kS1Units) return false;
    const uint4 ninf = sizeof(LT) == 2 ? make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u)
                                       : make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
    const LT* L = static_cast<const LT*>(p.logits);
    const long e_stop = e_end < p.V ? e_end : p.V;
    const unsigned slice_bytes = e_stop > e_begin ? (unsigned)((e_stop - e_begin) * (long)sizeof(LT)) : 0u;
    auto prefetch_row = [&](int r) {
        if (lane == 0 && r < R && slice_bytes > 0) bulk_prefetch_l2(L + (size_t)r * p.V + e_begin, slice_bytes);
    };
#pragma unroll
    for (int a = 0; a < kS1Ahead; ++a) prefetch_row((int)(threadIdx.x >> 5) + a * nw);
    const f2x k2 = f2_pack(kLog2e, kLog2e);
    for (int row = (int)(threadIdx.x >> 5); row < R; row += nw) {
        prefetch_row(row + kS1Ahead * nw);
        const LT* lrow = L + (size_t)row * p.V;
        uint4 w[kS1Units];
#pragma unroll
        for (int u = 0; u < kS1Units; ++u) {
            const long e0 = e_begin + (long)u * UNIT + (long)lane * EPL;
            w[u] = ninf;
            if (u < upr && e0 < e_end && e0 + EPL <= p.V) w[u] = __ldg(reinterpret_cast<const uint4*>(lrow + e0));
        }
        float m = u4_max_nan<sizeof(LT)>(w[0]);
#pragma unroll
        for (int u = 1; u < kS1Units; ++u) m = f_max_nan(m, u4_max_nan<sizeof(LT)>(w[u]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = f_max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
        const int bad = bad_logit(m) ? 1 : 0;
        const bool live = !bad && m != -INFINITY;
        const float m2 = m * kLog2e;
        const f2x nm2 = f2_pack(-m2, -m2);
        float tot = 0.0f;
#pragma unroll
        for (int u = 0; u < kS1Units; ++u) {
            if (u >= upr) break;
            float sum = 0.0f;
            if (live) {   // -inf entries add 0
                const uint32_t a[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
                f2x acc = f2_pack(0.0f, 0.0f);
                if constexpr (sizeof(LT) == 2) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc = f2_add(acc, f2_ex2(f2_fma(bf2_widen(a[q]), k2, nm2)));
                } else {
#pragma unroll
                    for (int q = 0; q < 2; ++q)
                        acc = f2_add(acc, f2_ex2(f2_fma(f2_pack(__uint_as_float(a[2 * q]), __uint_as_float(a[2 * q + 1])),
                                                        k2, nm2)));
                }
                const float2 s2 = f2_unpack(acc);
                sum = s2.x + s2.y;
            }
#pragma unroll
            for (int o = LPT >> 1; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            tot += sum;
            if ((lane & (LPT - 1)) == 0) {
                const int t = tb + u * TPU + lane / LPT;
                if (t < te)
                    p.tile_rec[(size_t)row * p.n_tiles + t] =
                        rowacc_pack(RowAcc{live ? m : -INFINITY, live ? sum : 0.0f, 0x7fffffff, bad});
            }
        }
        if (TPU == 2) tot += __shfl_xor_sync(0xffffffffu, tot, 16);
        if (lane == 0)
            p.cta_rec[(size_t)row * gridDim.x + blockIdx.x] =
                rowacc_pack(RowAcc{live ? m : -INFINITY, live ? tot : 0.0f, 0x7fffffff, bad});
    }
    return true;
}

// Pass 0 at T=1 for slices longer than kS1Units units: each warp streams its rows'
// slices of the CTA's tile range as one flat sequence of units (32 words, one per lane: 256 bf16 or 128 float32 entries, so two
// tiles or one), with D units' loads in flight per lane in a register ring that runs
// across row boundaries.  A unit folds on its own: each tile's maximum comes from its
// own lanes (a NaN or +inf entry shows as a NaN or +inf maximum), then the tile's sum
// against it.  The tile's first lane writes the tile record and merges it into the
// row's slice record.  Rows are also requested into L2 a few rows ahead.
template <typename LT>
__device__ void stream0_t1_ring(const DraftParams& p) {
    constexpr int EPL = 16 / (int)sizeof(LT);          // entries per lane per unit
    constexpr int UNIT = 32 * EPL;                     // entries per unit
    constexpr int TPU = UNIT / kDraftTile;             // tiles per unit (1 or 2)
    constexpr int LPT = 32 / TPU;                      // lanes per tile
    constexpr int D = 8;                               // units in flight per lane
    const int R = p.B * p.gamma;
    const int lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    const int w0 = (int)(threadIdx.x >> 5);
    const int tb = tile_begin(blockIdx.x, gridDim.x, p.n_tiles), te = tile_begin(blockIdx.x + 1, gridDim.x, p.n_tiles);
    const long e_begin = (long)tb * kDraftTile, e_end = (long)te * kDraftTile;
    const int upr = (int)((e_end - e_begin + UNIT - 1) / UNIT);   // units per row
    if (upr == 0) {   // an empty tile range: empty records
        if (lane == 0)
            for (int row = w0; row < R; row += nw)
                p.cta_rec[(size_t)row * gridDim.x + blockIdx.x] = rowacc_pack(rowacc_empty());
        return;
    }
    const LT* L = static_cast<const LT*>(p.logits);
    const long e_stop = e_end < p.V ? e_end : p.V;
    const unsigned slice_bytes = e_stop > e_begin ? (unsigned)((e_stop - e_begin) * (long)sizeof(LT)) : 0u;
    auto prefetch_row = [&](int r) {
        if (lane == 0 && r < R && slice_bytes > 0) bulk_prefetch_l2(L + (size_t)r * p.V + e_begin, slice_bytes);
    };
#pragma unroll
    for (int a = 0; a < kS1Ahead; ++a) prefetch_row(w0 + a * nw);
    const uint4 ninf = sizeof(LT) == 2 ? make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u)
                                       : make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
    // load cursor (row, unit); rows past R load nothing
    int lrow = w0, lu = 0;
    auto load_next = [&]() -> uint4 {
        uint4 v = ninf;
        const long e0 = e_begin + (long)lu * UNIT + (long)lane * EPL;
        if (lrow < R && e0 < e_end && e0 + EPL <= p.V)
            v = __ldg(reinterpret_cast<const uint4*>(L + (size_t)lrow * p.V + e0));
        if (++lu == upr) {
            lu = 0;
            lrow += nw;
            prefetch_row(lrow + (kS1Ahead - 1) * nw);
        }
        return v;
    };
    const int my_rows = w0 < R ? (R - w0 + nw - 1) / nw : 0;
    const int Nu = my_rows * upr;
    uint4 ring[D];
#pragma unroll
    for (int s = 0; s < D; ++s) ring[s] = load_next();
    int crow = w0, cu = 0;   // consume cursor
    RowAcc acc = rowacc_empty();
    for (int u0 = 0; u0 < Nu; u0 += D) {
#pragma unroll
        for (int s = 0; s < D; ++s) {
            if (u0 + s < Nu) {
                const uint4 w = ring[s];
                ring[s] = load_next();
                float m = u4_max_nan<sizeof(LT)>(w);
#pragma unroll
                for (int o = LPT >> 1; o > 0; o >>= 1) m = f_max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
                const bool bad = bad_logit(m);
                const bool live = !bad && m != -INFINITY;
                float sum = 0.0f;
                if (live) {
                    float x[EPL];
                    unpack_word<LT>(w, x);
                    const float m2 = m * kLog2e;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) sum += wexp(x[e], m2);   // -inf entries add 0
                }
#pragma unroll
                for (int o = LPT >> 1; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                const int t = tb + cu * TPU + lane / LPT;
                if ((lane & (LPT - 1)) == 0 && t < te) {
                    const RowAcc tr{live ? m : -INFINITY, live ? sum : 0.0f, 0x7fffffff, bad ? 1 : 0};
                    p.tile_rec[(size_t)crow * p.n_tiles + t] = rowacc_pack(tr);
                    acc = rowacc_merge(acc, tr);
                }
                if (++cu == upr) {
                    if (TPU == 2) {   // the second tile's lanes hold the odd tiles' part
                        RowAcc o;
                        o.mx = __shfl_sync(0xffffffffu, acc.mx, LPT % 32);
                        o.s = __shfl_sync(0xffffffffu, acc.s, LPT % 32);
                        o.idx = 0x7fffffff;
                        o.bad = __shfl_sync(0xffffffffu, acc.bad, LPT % 32);
                        acc = rowacc_merge(acc, o);
                    }
                    if (lane == 0) p.cta_rec[(size_t)crow * gridDim.x + blockIdx.x] = rowacc_pack(acc);
                    acc = rowacc_empty();
                    cu = 0;
                    crow += nw;
                }
            }
        }
    }
}

// Pass 0 at T=1: the per-row form where a slice fits the registers, else the ring.
template <typename LT>
__device__ void tile_phase_stream0_t1(const DraftParams& p) {
    if (!stream0_t1_rows<LT>(p)) stream0_t1_ring<LT>(p);
}

// T=0 tokens from the folded argmax keys, in every CTA (one load per row): into the
// shared array `cur`, and the row maxima into `cur_mx`; returns whether any token
// differs from `prev` (the same in every CTA).
__device__ __forceinline__ bool finalize_keys_t0(const DraftParams& p, const unsigned long long* keys,
                                                 const int32_t* prev, int32_t* cur, float* cur_mx, bool compare) {
    const int R = p.B * p.gamma;
    for (int row = threadIdx.x; row < R; row += blockDim.x) {
        const unsigned long long k = __ldcg(&keys[(size_t)row * kKeyStride]);
        const bool valid = k != ~0ull && key_value(k) != -INFINITY;
        cur[row] = valid ? (int32_t)key_index(k) : -1;
        cur_mx[row] = valid ? key_value(k) : -INFINITY;
    }
    __syncthreads();
    int diff = 0;
    if (compare)
        for (int row = threadIdx.x; row < R; row += blockDim.x) diff |= (cur[row] != prev[row]) ? 1 : 0;
    return __syncthreads_or(diff) != 0;
}

// After the last T=0 pass: the CTA owning a row (row % gridDim.x) computes its
// confidence 1 / sum 2^(z log2e - m2) from the CTA records, each record's sum rescaled
// to the row maximum from the keys (m2 = max log2e), independent exponentials summed
// per warp and then over warps in order; the whole CTA takes the owned rows two at a
// time with all records requested at once.  Then it writes the outputs, applying the
// chain rule (an invalid anchor or position voids the rest of the request).  `cur` and
// `cur_mx` hold every row's token and maximum.
__device__ __forceinline__ void owner_outputs_t0(const DraftParams& p, const float4* recs_all, const int32_t* cur,
                                                 const float* cur_mx, const int32_t* anc) {
    const int R = p.B * p.gamma;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    const int nblk = gridDim.x;
    const int nown = R > (int)blockIdx.x ? (R - 1 - (int)blockIdx.x) / nblk + 1 : 0;
    __shared__ float s_part[2][32];
    for (int k0 = 0; k0 < nown; k0 += 2) {
        float part[2] = {0.0f, 0.0f};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (k0 + h >= nown) continue;
            const int row = blockIdx.x + (k0 + h) * nblk;
            if (cur[row] < 0) continue;
            const float m2 = cur_mx[row] * kLog2e;
            for (int c = threadIdx.x; c < nblk; c += blockDim.x) {
                const RowAcc a = rowacc_unpack(__ldcg(&recs_all[(size_t)row * nblk + c]));
                if (a.mx != -INFINITY) part[h] += a.s * ex2(a.mx * kLog2e - m2);
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float w = warp_sum(part[h]);
            if (lane == 0) s_part[h][warp] = w;
        }
        __syncthreads();
        if (threadIdx.x < 2 && k0 + (int)threadIdx.x < nown) {
            const int row = blockIdx.x + (k0 + (int)threadIdx.x) * nblk;
            float S = 0.0f;
            for (int w = 0; w < nw; ++w) S += s_part[threadIdx.x][w];
            const float mx = cur_mx[row];
            p.conf_out[row] = cur[row] >= 0 ? ex2(fmaf(mx, kLog2e, -mx * kLog2e)) / S : NAN;
        }
        __syncthreads();
    }
    for (int row = blockIdx.x + nblk * (int)threadIdx.x; row < R; row += nblk * (int)blockDim.x) {
        const int b = row / p.gamma, j = row % p.gamma;
        const int a = anc[b];
        bool dead = (a < 0 || a >= p.V);
        int first_dead = dead ? 0 : -1;
        for (int k = 0; k <= j && !dead; ++k)
            if (cur[b * p.gamma + k] < 0) { dead = true; first_dead = k; }
        if (dead) {
            p.tokens_out[row] = -1;
            p.conf_out[row] = NAN;
            if (p.qtok_out) p.qtok_out[row] = NAN;
            if (first_dead == j) atomicOr(p.status, (a < 0 || a >= p.V) ? SPEC_DEV_TOKEN : SPEC_DEV_NONFINITE);
        } else {
            p.tokens_out[row] = cur[row];
            if (p.qtok_out) p.qtok_out[row] = p.conf_out[row];
        }
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
