// tree.cu - EAGLE-2 draft trees: path-product selection and T=0 verification
// (spec_tree_select, spec_tree_verify).
//
// Defines: "Speculative Decoding Part 2: the evolution of drafter architectures" (VESSL
// AI), EAGLE section - EAGLE-2 scores each branch of a dynamic draft tree by the
// product of the confidences from the root, so a parent scores at least as high as its
// children and keeping the highest-scored nodes keeps their parents; "Solar Open2
// DSpark" (sionic.ai), sections 1 and 6 - verification commits the longest prefix that
// agrees with the target, here along the tree's paths.
//
// Selection: one CTA per tree.  Scores are float64 products taken level by level
// (score[i] = conf[i] * score[parent[i]] once the parent's is known), the same single
// multiply per node as the definition, so the scores are bit-identical to a sequential
// pass.  The m largest are found by ranking every node against every other on the
// scores' bit patterns (non-negative doubles order as unsigned integers), ties to the
// lower index.
//
// Verification (T=0): HBM-bound.  A persistent grid streams the root row and every kept
// node's row in 8192-entry items (the items of dropped nodes are compacted away, 256 at
// a time), two items of loads in flight per thread (32-byte loads where the rows start
// on 32 bytes, 16-byte ones otherwise).  Each warp folds its
// 1024-entry segment of an item into the row's 64-bit argmax key (value, lowest index)
// with one atomicMax, so warps never wait for one another.  The last CTA to finish then
// marks, for every node in parallel, whether its token is the argmax of its parent's row
// (keeping the lowest such child per parent), and one thread per tree follows those
// marks from the root.
#include "spec_device.cuh"
#include "internal.h"
#include "chunk_rows.cuh"

namespace spec {

// ----------------------------------------------------------------------------------
// Selection
// ----------------------------------------------------------------------------------
constexpr int kSelThreads = 1024;

__global__ void __launch_bounds__(kSelThreads) tree_select_kernel(TreeSelectParams p) {
    const int t = blockIdx.x;
    const int n = p.n_nodes;
    __shared__ double s_score[SPEC_MAX_TREE_NODES];
    __shared__ float s_conf[SPEC_MAX_TREE_NODES];
    __shared__ int s_parent[SPEC_MAX_TREE_NODES];
    __shared__ int s_keep[SPEC_MAX_TREE_NODES];
    __shared__ int s_bad;
    const int32_t* par = p.parent + (size_t)t * n;
    const float* conf = p.conf + (size_t)t * n;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int pa = par[i];
        float c = conf[i];
        c = isnan(c) ? 0.0f : fminf(fmaxf(c, 0.0f), 1.0f);   // NaN reads as 0, clamped to [0, 1]
        s_parent[i] = pa;
        s_conf[i] = c;
        s_score[i] = -1.0;                                    // not yet known
        if (pa < -1 || pa >= i) s_bad = 1;
    }
    __syncthreads();
    if (s_bad) {   // parents not in topological order: no scores, no selection
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            if (p.score_out) p.score_out[(size_t)t * n + i] = __longlong_as_double(0x7ff8000000000000ll);
            p.keep_out[(size_t)t * n + i] = 0;
        }
        if (p.selected_out)
            for (int j = threadIdx.x; j < p.m; j += blockDim.x) p.selected_out[(size_t)t * p.m + j] = -1;
        return;
    }
    // level by level: a node whose parent's score is known takes its own (a concurrent
    // reader of a score sees either "not yet known" or its final value)
    for (;;) {
        int progressed = 0;
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            if (s_score[i] >= 0.0) continue;
            const int pa = s_parent[i];
            if (pa < 0) { s_score[i] = (double)s_conf[i]; progressed = 1; }
            else {
                const double sp = s_score[pa];
                if (sp >= 0.0) { s_score[i] = (double)s_conf[i] * sp; progressed = 1; }
            }
        }
        if (!__syncthreads_or(progressed)) break;
    }
    // rank of node i: nodes with a larger score, or an equal score and a lower index
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const unsigned long long si = (unsigned long long)__double_as_longlong(s_score[i]);
        int rank = 0;
        for (int j = 0; j < n; ++j) {
            const unsigned long long sj = (unsigned long long)__double_as_longlong(s_score[j]);
            rank += (sj > si || (sj == si && j < i)) ? 1 : 0;
        }
        const int keep = rank < p.m ? 1 : 0;
        s_keep[i] = keep;
        p.keep_out[(size_t)t * n + i] = keep;
        if (p.score_out) p.score_out[(size_t)t * n + i] = s_score[i];
    }
    __syncthreads();
    if (p.selected_out) {   // the kept nodes in index order, then -1
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            if (!s_keep[i]) continue;
            int pos = 0;
            for (int j = 0; j < i; ++j) pos += s_keep[j];
            p.selected_out[(size_t)t * p.m + pos] = i;
        }
        const int kept = p.m < n ? p.m : n;
        for (int j = kept + (int)threadIdx.x; j < p.m; j += blockDim.x) p.selected_out[(size_t)t * p.m + j] = -1;
    }
}

cudaError_t tree_select_launch(const TreeSelectParams& p, cudaStream_t stream) {
    tree_select_kernel<<<p.n_trees, kSelThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------------
// Verification (T=0)
// ----------------------------------------------------------------------------------
constexpr int kTvThreads = 256;
constexpr int kTvWarps = kTvThreads / 32;
constexpr int kTvChunk = kTvThreads * kEPT;   // 8192 entries per item
#ifndef TV_DEPTH_BF16
#define TV_DEPTH_BF16 2
#endif

// The row of item `it` (rows are tree-major: tree t, then its root row and node rows)
// and its chunk; false when the row belongs to a node that is not kept.
__device__ __forceinline__ bool tv_item(const TreeVerifyParams& p, long it, unsigned nch, long& row, int& c) {
    row = it / (long)nch;
    c = (int)(it - row * (long)nch);
    const int rpt = p.n_nodes + 1;
    const int t = (int)(row / rpt);
    const int node = (int)(row - (long)t * rpt) - 1;
    return node < 0 || !p.keep || p.keep[(size_t)t * p.n_nodes + node] != 0;
}

// One warp's 1024 entries of an item (group- or sector-interleaved): fold them into the row's
// argmax key (or its bad flag) with one atomic per warp, so warps never wait for one
// another.  Only the lanes holding the maximum look for its lowest index.
template <typename TT, int NW, bool L32>
__device__ __forceinline__ void tv_fold(const TreeVerifyParams& p, const uint4 (&w)[NW], long row, int c) {
    const float lm = chunk_max_nan<TT, NW>(w);
    const float m = warp_max_nan(lm);
    const int bad = (isnan(m) || m == INFINITY) ? 1 : 0;
    int idx = 0x7fffffff;
    if (!bad && lm == m) {
        const int k = first_equal<TT, NW>(w, m);
        if (k >= 0) idx = (int)(L32 ? il32_entry<TT>(il_seg(c), k) : il_entry(il_seg(c), k));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) idx = min(idx, __shfl_xor_sync(0xffffffffu, idx, o));
    if ((threadIdx.x & 31) == 0) {
        if (bad) atomicOr(&p.rowbad[row], 1u);
        else atomicMax(&p.keys[row], argmax_key(m, (uint32_t)idx));
    }
}

// D items of loads in flight per thread (the one being reduced included).
template <typename TT> struct TvDepth { static constexpr int D = sizeof(TT) == 2 ? TV_DEPTH_BF16 : 2; };

// L32: the target rows start on 32 bytes and hold whole 32-byte groups, so the chunks
// are read in the sector-interleaved layout, one 32-byte load per group.
template <typename TT, bool L32>
__global__ void __launch_bounds__(kTvThreads) tree_verify_kernel(TreeVerifyParams p) {
    const TT* target = static_cast<const TT*>(p.target);
    const long V = p.V;
    const unsigned nch = (unsigned)((V + kTvChunk - 1) / kTvChunk);
    const int n = p.n_nodes, rpt = n + 1;
    const long items = (long)p.n_trees * rpt * nch;
    const bool vec = p.vec_t != 0;
    constexpr int NW = Words<TT>::N;
    constexpr int D = TvDepth<TT>::D;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ int s_row[kTvThreads];   // the CTA's kept items of the current batch: row
    __shared__ int s_c[kTvThreads];     // and chunk
    __shared__ int s_wc[kTvWarps];
    const long mine = items > (long)blockIdx.x ? (items - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    for (long k0 = 0; k0 < mine; k0 += kTvThreads) {
        // the next 256 items of this CTA, with those of dropped rows removed: each thread
        // resolves one item, then a block compaction keeps their order
        int cnt;
        {
            const long k = k0 + threadIdx.x;
            const long it = (long)blockIdx.x + k * (long)gridDim.x;
            long row;
            int c;
            const bool kept = k < mine && tv_item(p, it, nch, row, c);
            const unsigned bal = __ballot_sync(0xffffffffu, kept);
            if (lane == 0) s_wc[warp] = __popc(bal);
            __syncthreads();
            int off = 0;
            cnt = 0;
#pragma unroll
            for (int w = 0; w < kTvWarps; ++w) {
                const int v = s_wc[w];
                off += w < warp ? v : 0;
                cnt += v;
            }
            if (kept) {
                const int at = off + __popc(bal & ((1u << lane) - 1u));
                s_row[at] = (int)row;
                s_c[at] = c;
            }
            __syncthreads();
        }
        // stream the batch with D items of loads in flight per thread
        uint4 buf[D][NW];
        int rows[D], cs[D];
#pragma unroll
        for (int d = 0; d < D - 1; ++d)
            if (d < cnt) {
                rows[d] = s_row[d];
                cs[d] = s_c[d];
                if constexpr (L32) load_words_il32<TT, NW>(buf[d], target + (size_t)rows[d] * V, V, il_seg(cs[d]));
                else load_words_il<TT, NW>(buf[d], target + (size_t)rows[d] * V, V, il_seg(cs[d]), vec);
            }
        for (int j0 = 0; j0 < cnt; j0 += D) {
#pragma unroll
            for (int d = 0; d < D; ++d) {
                const int j = j0 + d;
                const int jn = j + D - 1, dn = (d + D - 1) % D;
                if (jn < cnt) {
                    rows[dn] = s_row[jn];
                    cs[dn] = s_c[jn];
                    if constexpr (L32)
                        load_words_il32<TT, NW>(buf[dn], target + (size_t)rows[dn] * V, V, il_seg(cs[dn]));
                    else load_words_il<TT, NW>(buf[dn], target + (size_t)rows[dn] * V, V, il_seg(cs[dn]), vec);
                }
                if (j < cnt) tv_fold<TT, NW, L32>(p, buf[d], rows[d], cs[d]);
            }
        }
        __syncthreads();   // s_row and s_c are rewritten by the next batch
    }

    if (!last_block_done(&p.done[0], gridDim.x)) return;

    // 1. every kept node whose token is the argmax of its parent's row: the lowest such
    //    child of each parent, as first[parent + 1] = n - child (0: none); a parent
    //    outside [-1, child) marks the tree invalid
    const long total = (long)p.n_trees * n;
    for (long q = threadIdx.x; q < total; q += blockDim.x) {
        const int t = (int)(q / n), i = (int)(q - (long)t * n);
        const int pa = p.parent[q];
        if (pa < -1 || pa >= i) { atomicOr(&p.treebad[t], 1u); continue; }
        if (p.keep && p.keep[q] == 0) continue;
        const unsigned long long k = __ldcg(&p.keys[(size_t)t * rpt + pa + 1]);
        if (p.token[q] == (int32_t)key_index(k)) atomicMax(&p.first[(size_t)t * rpt + pa + 1], (unsigned)(n - i));
    }
    __syncthreads();

    // 2. one thread per tree follows the marks from the root; every row on the way must
    //    hold a distribution
    for (int t = threadIdx.x; t < p.n_trees; t += blockDim.x) {
        const size_t r0 = (size_t)t * rpt;
        int32_t* path = p.path_out + (size_t)t * n;
        int32_t* com = p.committed_out + (size_t)t * rpt;
        unsigned fl = __ldcg(&p.treebad[t]) ? SPEC_DEV_TOKEN : 0u;
        int cur_node = -1, L = 0;
        while (!fl) {
            const size_t r = r0 + cur_node + 1;
            if (__ldcg(&p.rowbad[r]) != 0u || key_value(__ldcg(&p.keys[r])) == -INFINITY) {
                fl = SPEC_DEV_NONFINITE;
                break;
            }
            const unsigned f = __ldcg(&p.first[r]);
            if (f == 0u) break;
            const int child = n - (int)f;
            path[L] = child;
            com[L] = p.token[(size_t)t * n + child];
            ++L;
            cur_node = child;
        }
        if (fl) {
            atomicOr(p.status, fl);
            for (int j = 0; j < n; ++j) path[j] = -1;
            for (int j = 0; j <= n; ++j) com[j] = -1;
            p.n_out[t] = -1;
            p.bonus_out[t] = -1;
        } else {
            const int y = (int)key_index(__ldcg(&p.keys[r0 + cur_node + 1]));
            com[L] = y;
            for (int j = L; j < n; ++j) path[j] = -1;
            for (int j = L + 1; j <= n; ++j) com[j] = -1;
            p.n_out[t] = L;
            p.bonus_out[t] = y;
        }
    }
    __syncthreads();

    // 3. leave the workspace zeroed for the next call
    const long rows = (long)p.n_trees * rpt;
    for (long r = threadIdx.x; r < rows; r += blockDim.x) {
        p.keys[r] = 0ull;
        p.rowbad[r] = 0u;
        p.first[r] = 0u;
    }
    for (int t = threadIdx.x; t < p.n_trees; t += blockDim.x) p.treebad[t] = 0u;
    if (threadIdx.x == 0) p.done[0] = 0u;
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t tree_verify_workspace_bytes(int n_trees, int n_nodes) {
    const size_t rows = (size_t)n_trees * (n_nodes + 1);
    size_t off = kWsHeaderBytes;
    off = align_up(off + sizeof(unsigned long long) * rows, 256);   // keys
    off = align_up(off + sizeof(unsigned) * rows, 256);             // rowbad
    off = align_up(off + sizeof(unsigned) * rows, 256);             // first
    off = align_up(off + sizeof(unsigned) * (size_t)n_trees, 256);  // treebad
    return off;
}

cudaError_t tree_verify_launch(TreeVerifyParams& p, void* ws, cudaStream_t stream) {
    char* w = static_cast<char*>(ws);
    WsHeader* h = reinterpret_cast<WsHeader*>(w);
    p.status = &h->status;
    p.done = h->done;
    const size_t rows = (size_t)p.n_trees * (p.n_nodes + 1);
    size_t off = kWsHeaderBytes;
    p.keys = reinterpret_cast<unsigned long long*>(w + off);
    off = align_up(off + sizeof(unsigned long long) * rows, 256);
    p.rowbad = reinterpret_cast<unsigned*>(w + off);
    off = align_up(off + sizeof(unsigned) * rows, 256);
    p.first = reinterpret_cast<unsigned*>(w + off);
    off = align_up(off + sizeof(unsigned) * rows, 256);
    p.treebad = reinterpret_cast<unsigned*>(w + off);

    // rows that start on 32 bytes and hold whole 32-byte groups: the sector layout
    const size_t esize = p.tdt == SPEC_BF16 ? 2 : 4;
    const bool l32 = p.vec_t && (reinterpret_cast<uintptr_t>(p.target) & 31u) == 0 && ((size_t)p.V * esize) % 32 == 0;
    void (*k)(TreeVerifyParams) =
        p.tdt == SPEC_BF16 ? (l32 ? tree_verify_kernel<bf16_t, true> : tree_verify_kernel<bf16_t, false>)
                           : (l32 ? tree_verify_kernel<float, true> : tree_verify_kernel<float, false>);
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kTvThreads, 0) != cudaSuccess || occ < 1) occ = 1;
    const long nch = ((long)p.V + kTvChunk - 1) / kTvChunk;
    const long items = (long)rows * nch;
    const long cap = (long)device_sm_count() * occ;
    const long grid = items < cap ? items : cap;
    k<<<(unsigned)(grid > 0 ? grid : 1), kTvThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace spec
