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
// One CTA per reference: the 64-bit (key, position) words of every position in
// shared memory, one bitonic sort, the first n positions sorted again, the outputs
// written with coalesced stores.  The work is a few microseconds per reference.
#include "spec_device.cuh"
#include "internal.h"

namespace spec {

constexpr int kPlanThreads = 1024;
constexpr uint64_t kPlanStream = 4;   // Philox stream of the anchor choice

// Ascending bitonic sort of M (a power of two) 64-bit words in shared memory.
__device__ __forceinline__ void plan_sort(unsigned long long* s, int M) {
    for (int size = 2; size <= M; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < M; i += blockDim.x) {
                const int l = i ^ stride;
                if (l > i) {
                    const bool up = (i & size) == 0;
                    const unsigned long long a = s[i], b = s[l];
                    if (up ? (a > b) : (a < b)) { s[i] = b; s[l] = a; }
                }
            }
            __syncthreads();
        }
    }
}

__global__ void __launch_bounds__(kPlanThreads) branch_plan_kernel(BranchPlanParams p) {
    extern __shared__ __align__(16) unsigned long long s_key[];
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
    int M = 1;
    while (M < L) M <<= 1;
    for (int i = threadIdx.x; i < M; i += blockDim.x) {
        unsigned long long w = ~0ull;   // padding sorts last
        if (i < L) w = ((philox_word0(p.seed, (uint64_t)r, (uint64_t)i, kPlanStream) >> 40) << 32) | (unsigned)i;
        s_key[i] = w;
    }
    __syncthreads();
    plan_sort(s_key, M);
    // the first n positions, in ascending order
    int Mn = 1;
    while (Mn < n) Mn <<= 1;
    unsigned long long pos[(16384 + kPlanThreads - 1) / kPlanThreads];   // this thread's picks
    int c = 0;
    for (int i = threadIdx.x; i < Mn; i += blockDim.x) pos[c++] = i < n ? (s_key[i] & 0xffffffffull) : ~0ull;
    __syncthreads();
    c = 0;
    for (int i = threadIdx.x; i < Mn; i += blockDim.x) s_key[i] = pos[c++];
    __syncthreads();
    plan_sort(s_key, Mn);
    const int32_t* trunk = p.trunk + (size_t)r * p.Lmax;
    for (int k = threadIdx.x; k < n; k += blockDim.x) {
        const int a = (int)s_key[k];
        anchors[k] = a;
        atok[k] = trunk[a];
    }
    for (int i = threadIdx.x; i < n * W; i += blockDim.x) {
        const int k = i / W, t = i - k * W + 1;
        const int a = (int)s_key[k];
        parent[i] = t == 1 ? a : L + i - 1;
        position[i] = a + t;
    }
}

size_t branch_plan_smem(int Lmax) {
    int M = 1;
    while (M < Lmax) M <<= 1;
    return (size_t)M * sizeof(unsigned long long);
}

cudaError_t branch_plan_launch(const BranchPlanParams& p, cudaStream_t stream) {
    const size_t smem = branch_plan_smem(p.Lmax);
    cudaError_t e = cudaFuncSetAttribute(branch_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    branch_plan_kernel<<<p.n_refs, kPlanThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace spec
