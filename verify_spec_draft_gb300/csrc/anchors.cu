// anchors.cu - the SpecOPD anchor-branch plan (spec_branch_plan).
//
// Defines: "SpecOPD" paper summary (onedev.kr), section "how it works" - n anchors
// picked at random on a reference response, one branch of W drafted tokens from
// each, the branches independent of one another; section "how it differs" - the
// branches packed into one proposal tree, every node seeing its own reference prefix
// and its own branch's history through a parent map, with its semantic position (not
// its packing order) as its rotary position.
//
// Reading (the pages give no formula): the anchors of reference r are n distinct
// positions of 0..L_r-1, the n smallest (key, position) where the key of position i
// is word0 >> 40 of Philox4x64-10 with key (seed, 0) and counter (r, i, 4, 0); they
// are listed in ascending position.  Branch k, step t = 1..W, is packed as node
// L_r + k*W + t-1 (the trunk holds nodes 0..L_r-1), with parent a_k for t = 1 and
// the node before otherwise, and semantic position a_k + t.
//
// One CTA per reference.  The (key, position) words of every position go to shared
// memory as key << 16 | position (positions < 2^16: unique words in (key, position)
// order); a radix select, most significant 8-bit digit first, finds the n-th smallest
// word; the picks are marked in a bitmap over the positions, and each bitmap word's
// picks are written in ascending position at the popcount of the words before it.
#include "spec_device.cuh"
#include "internal.h"

namespace spec {

constexpr int kPlanThreads = 1024;
constexpr uint64_t kPlanStream = 4;   // Philox stream of the anchor choice
constexpr int kPlanDigits = 5;        // 8-bit digits of a 40-bit word
static_assert(SPEC_MAX_TRUNK <= 65536, "positions fit the word's low 16 bits");
static_assert(SPEC_MAX_TRUNK <= 32 * kPlanThreads, "one bitmap word per thread");

__device__ __forceinline__ int plan_block_exclusive_scan(int v, int* s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < (int)(blockDim.x >> 5) ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        s_warp[lane] = w;   // inclusive prefix over the warps
    }
    __syncthreads();
    const int before = warp > 0 ? s_warp[warp - 1] : 0;
    return before + incl - v;
}

__global__ void __launch_bounds__(kPlanThreads) branch_plan_kernel(BranchPlanParams p) {
    extern __shared__ __align__(16) unsigned long long s_key[];   // [Lmax]
    __shared__ int s_hist[256];
    __shared__ int s_warp[32];
    __shared__ unsigned long long s_prefix;
    __shared__ int s_need;
    const int r = blockIdx.x;
    const int n = p.n_anchors, W = p.W;
    const int L = p.lengths[r];
    int32_t* anchors = p.anchors_out + (size_t)r * n;
    int32_t* atok = p.anchor_tok_out + (size_t)r * n;
    int32_t* parent = p.parent_out + (size_t)r * n * W;
    int32_t* position = p.position_out + (size_t)r * n * W;
    if (L < n || L > p.Lmax || L < 1) {   // no anchors for this reference
        for (int i = threadIdx.x; i < n; i += blockDim.x) { anchors[i] = -1; atok[i] = -1; }
        for (int i = threadIdx.x; i < n * W; i += blockDim.x) { parent[i] = -1; position[i] = -1; }
        if (threadIdx.x == 0) atomicOr(p.status, SPEC_DEV_TOKEN);
        return;
    }
    uint32_t* s_bits = reinterpret_cast<uint32_t*>(s_key + p.Lmax);   // [ceil(Lmax / 32)]
    int32_t* s_anc = reinterpret_cast<int32_t*>(s_bits + (p.Lmax + 31) / 32);   // [n]
    const int nwords = (L + 31) / 32;
    for (int i = threadIdx.x; i < L; i += blockDim.x)
        s_key[i] = ((philox_word0(p.seed, (uint64_t)r, (uint64_t)i, kPlanStream) >> 40) << 16) | (unsigned)i;
    for (int i = threadIdx.x; i < nwords; i += blockDim.x) s_bits[i] = 0u;
    if (threadIdx.x == 0) { s_prefix = 0ull; s_need = n; }
    // radix select: after the pass of digit d the high digits of the n-th smallest word
    // are known, and s_need counts how many words with those high digits come up to it
    for (int d = kPlanDigits - 1; d >= 0; --d) {
        const int shift = 8 * d;
        for (int i = threadIdx.x; i < 256; i += blockDim.x) s_hist[i] = 0;
        __syncthreads();
        const unsigned long long hi = s_prefix >> (shift + 8);
        for (int i = threadIdx.x; i < L; i += blockDim.x) {
            const unsigned long long w = s_key[i];
            if ((w >> (shift + 8)) == hi) atomicAdd(&s_hist[(int)((w >> shift) & 255u)], 1);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // lane l takes bins 8l .. 8l+7; the digit is where the running count reaches s_need
            const int lane = threadIdx.x;
            int c[8], tot = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) { c[k] = s_hist[8 * lane + k]; tot += c[k]; }
            int incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            const int need = s_need;
            int run = incl - tot;
            const bool mine = run < need && need <= incl;
            if (mine) {
                int k = 0;
                while (run + c[k] < need) run += c[k++];
                s_prefix |= (unsigned long long)(8 * lane + k) << shift;
                s_need = need - run;
            }
        }
        __syncthreads();
    }
    // the n smallest words are those up to the n-th; mark their positions
    const unsigned long long nth = s_prefix;
    for (int i = threadIdx.x; i < L; i += blockDim.x)
        if (s_key[i] <= nth) atomicOr(&s_bits[i >> 5], 1u << (i & 31));
    __syncthreads();
    // each bitmap word's picks at the popcount of the words before it, ascending (one
    // bitmap word per thread)
    {
        const int wi = threadIdx.x;
        const uint32_t bits = wi < nwords ? s_bits[wi] : 0u;
        int at = plan_block_exclusive_scan(__popc(bits), s_warp);
        for (uint32_t m = bits; m; m &= m - 1) s_anc[at++] = wi * 32 + __ffs(m) - 1;
        __syncthreads();
    }
    for (int k = threadIdx.x; k < n; k += blockDim.x) {
        const int a = s_anc[k];
        anchors[k] = a;
        atok[k] = p.trunk[(size_t)r * p.Lmax + a];
    }
    for (int i = threadIdx.x; i < n * W; i += blockDim.x) {
        const int k = i / W, t = i - k * W + 1;
        const int a = s_anc[k];
        parent[i] = t == 1 ? a : L + i - 1;
        position[i] = a + t;
    }
}

size_t branch_plan_smem(int Lmax) {
    return sizeof(unsigned long long) * (size_t)Lmax + sizeof(uint32_t) * (size_t)((Lmax + 31) / 32) +
           sizeof(int32_t) * (size_t)Lmax;
}

cudaError_t branch_plan_launch(const BranchPlanParams& p, cudaStream_t stream) {
    const size_t smem = branch_plan_smem(p.Lmax);
    cudaError_t e = cudaFuncSetAttribute(branch_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    branch_plan_kernel<<<p.n_refs, kPlanThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace spec
