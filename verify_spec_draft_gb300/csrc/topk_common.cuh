// topk_common.cuh - top-k / top-p pieces shared by the filtered verification and the
// filtered draft.
//
// Keys are 64-bit: the ordered float value in the high word, the inverted index in the
// low word, so a larger key is a larger value or, on a tie, a lower index (as for an
// argmax).  A warp keeps up to 32 keys as a list sorted in descending order, lane i
// holding the (i+1)-th largest.  A filtered row (reading of the DSpine card's setting:
// the top_k largest logits renormalised, then the shortest prefix in descending order
// whose running sum reaches top_p, renormalised again) is built from its top-k keys,
// one candidate per lane, in float32, with the cut-off taken again in float64 when a
// running sum lies within 1e-5 of top_p.  Draws are the inverse CDF in vocabulary-index
// order.
#pragma once

#include "spec_device.cuh"
#include "internal.h"

namespace spec {

constexpr int kTopkWarpsMax = 32;   // warps of a CTA that may call warp_draw

__device__ __forceinline__ unsigned long long shfl_u64(unsigned long long v, int src) {
    const unsigned lo = __shfl_sync(0xffffffffu, (unsigned)v, src);
    const unsigned hi = __shfl_sync(0xffffffffu, (unsigned)(v >> 32), src);
    return ((unsigned long long)hi << 32) | lo;
}
__device__ __forceinline__ unsigned long long shfl_up_u64(unsigned long long v) {
    const unsigned lo = __shfl_up_sync(0xffffffffu, (unsigned)v, 1);
    const unsigned hi = __shfl_up_sync(0xffffffffu, (unsigned)(v >> 32), 1);
    return ((unsigned long long)hi << 32) | lo;
}

// The warp's list: lane i holds its (i+1)-th largest key (0 = empty).  Inserts `key`
// (warp-uniform, smaller than at most k - 1 list keys) and updates `kth`, the list's
// k-th key.
__device__ __forceinline__ void list_insert(unsigned long long& mine, unsigned long long key, int k,
                                            unsigned long long& kth) {
    const int lane = threadIdx.x & 31;
    const int pos = __popc(__ballot_sync(0xffffffffu, mine > key));   // list keys above it: a prefix
    const unsigned long long up = shfl_up_u64(mine);
    if (lane == pos) mine = key;
    else if (lane > pos) mine = up;
    kth = shfl_u64(mine, k - 1);
}

struct FRow {                 // a filtered row: candidates in descending order of value
    int idx[kTopkMax];
    float pf[kTopkMax];       // filtered probability (0 past n)
    int n;                    // kept candidates; 0 for a row without a distribution
};

// Warp: filter the row whose key list is `kl` (k keys, descending, 0 = none).
static __device__ void filter_row(const unsigned long long* kl, int k, double top_p, FRow& r) {
    const int lane = threadIdx.x & 31;
    const unsigned long long key = lane < k ? kl[lane] : 0ull;
    const bool valid = key != 0ull;
    const float v = valid ? key_value(key) : -INFINITY;
    const float m = __shfl_sync(0xffffffffu, v, 0);
    if (!(m > -INFINITY)) {   // no finite entry
        if (lane == 0) r.n = 0;
        return;
    }
    const float w = valid ? ex2(fmaf(v, kLog2e, -m * kLog2e)) : 0.0f;
    const float S = warp_sum(w);
    const float cw = warp_inclusive_scan(w);
    const float run = cw / S;
    const unsigned reach = __ballot_sync(0xffffffffu, valid && (double)run >= top_p);
    const unsigned close = __ballot_sync(0xffffffffu, valid && fabs((double)run - top_p) < 1e-5);
    const int nvalid = __popc(__ballot_sync(0xffffffffu, valid));
    int n_keep = reach ? __ffs(reach) : nvalid;
    if (close) {   // the cut-off is close: take it again in float64
        const double w64 = valid ? exp((double)v - (double)m) : 0.0;
        double S64 = w64, run64 = w64;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) S64 += __shfl_xor_sync(0xffffffffu, S64, o);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, run64, o);
            if (lane >= o) run64 += y;
        }
        const unsigned reach64 = __ballot_sync(0xffffffffu, valid && run64 / S64 >= top_p);
        n_keep = reach64 ? __ffs(reach64) : nvalid;
    }
    const float Z = __shfl_sync(0xffffffffu, cw, n_keep - 1);
    r.idx[lane] = valid ? (int)key_index(key) : -1;
    r.pf[lane] = lane < n_keep ? w / Z : 0.0f;
    if (lane == 0) r.n = n_keep;
}

// Warp: the filtered probability of token x in row r (0 if not kept).
__device__ __forceinline__ float frow_prob(const FRow& r, int x) {
    const int lane = threadIdx.x & 31;
    const unsigned hit = __ballot_sync(0xffffffffu, lane < r.n && r.idx[lane] == x);
    return hit ? r.pf[__ffs(hit) - 1] : 0.0f;
}

// Per lane: the filtered probability of this lane's token x in row r (0 if not kept).
__device__ __forceinline__ float frow_prob_lane(const FRow& r, int x) {
    float v = 0.0f;
    for (int i = 0; i < r.n; ++i)
        if (r.idx[i] == x) v = r.pf[i];
    return v;
}

// Warp: inverse-CDF draw over lane weights wl (candidate index il, -1 for none) in
// vocabulary-index order: the smallest index whose running weight passes u * total, else
// the last of positive weight; `near` as in the other draws (1e-6 of the total).
static __device__ int warp_draw(int il, float wl, float u, int& near) {
    const int lane = threadIdx.x & 31;
    // order of each candidate by index (candidates are distinct; none sort last)
    const int key = il < 0 ? 0x7fffffff : il;
    int rank = 0;
    for (int j = 0; j < 32; ++j) {
        const int o = __shfl_sync(0xffffffffu, key, j);
        rank += (o < key || (o == key && j < lane)) ? 1 : 0;
    }
    __shared__ float s_w[kTopkWarpsMax][32];
    __shared__ int s_i[kTopkWarpsMax][32];
    const int warp = threadIdx.x >> 5;
    s_w[warp][rank] = il < 0 ? 0.0f : wl;
    s_i[warp][rank] = il;
    __syncwarp();
    const float ow = s_w[warp][lane];
    const int oi = s_i[warp][lane];
    const float C = warp_inclusive_scan(ow);
    const float Z = __shfl_sync(0xffffffffu, C, 31);
    const float t = u * Z;
    const float Cprev = C - ow;
    const unsigned cross = __ballot_sync(0xffffffffu, oi >= 0 && C > t);
    const unsigned pos = __ballot_sync(0xffffffffu, oi >= 0 && ow > 0.0f);
    int v;
    if (cross) v = __ffs(cross) - 1;
    else v = pos ? 31 - __clz(pos) : -1;
    if (v >= 0 && cross) {
        const float Cv = __shfl_sync(0xffffffffu, C, v);
        const float Cp = __shfl_sync(0xffffffffu, Cprev, v);
        const bool later = (pos >> v) > 1u;
        if ((fabsf(Cv - t) < 1e-6f * Z && later) || (Cp > 0.0f && fabsf(Cp - t) < 1e-6f * Z)) near = 1;
    }
    const int y = v < 0 ? -1 : __shfl_sync(0xffffffffu, oi, v);
    __syncwarp();
    return y;
}

}  // namespace spec
