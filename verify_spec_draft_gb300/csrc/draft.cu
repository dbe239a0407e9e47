// draft.cu - DSpark block draft with the rank-r Markov logit bias (spec_draft_block),
// bias on CUDA cores; the tcgen05 tensor-core variant is draft_tc.cu.
//
// Defines: "Speculative Decoding Part 2" (VESSL AI), DSpark section, bias equation
// B(x_{k-1}, .) = W_1[x_{k-1}] W_2 added to each position's logits; "Solar Open2
// DSpark" (sionic.ai), section 2 (Markov correction + per-position confidence).
//
// The chain x_j = choose(l_j + U[x_{j-1}] W_2) is sequential in j.  Instead of gamma
// dependent V-wide steps (gamma reads of W), the kernel solves it as a fixed point
// (Jacobi iteration): from a guess x^(k-1) it recomputes every position at once,
// x^(k)_j = choose(l_j + U[x^(k-1)_{j-1}] W_2), until x^(k) = x^(k-1).  Each step is a
// deterministic function of the previous token (the T=1 uniform of position j is
// fixed), so the fixed point is unique and equals the sequential chain; pass k fixes
// at least positions 1..k, so at most gamma passes run, and one pass reads W once.
// The initial guess is the unbiased choice of each position (pass 0), which a small
// bias rarely changes, so one biased pass usually confirms it.
//
// One cooperative persistent launch runs every pass (draft_common.cuh).  This file's
// tile phase computes z = l + U[x_prev] . Wt[v] in float32 on CUDA cores: one warp
// per row, four entries per lane per 128-entry tile, the CTA's contiguous tile range
// folded into one record per row.  It serves float32 weights and shapes the
// tensor-core path does not take.
#include "draft_common.cuh"

namespace spec {

template <typename LT, typename WT>
__global__ void __launch_bounds__(kThreads) draft_kernel(DraftParams p) {
    extern __shared__ float s_dyn[];
    float* s_uw = s_dyn + (size_t)(threadIdx.x >> 5) * (p.r > 0 ? p.r : 1);   // [kWarps][r]
    const bool biased = p.r > 0;
    const unsigned nb = gridDim.x;
    const int R = p.B * p.gamma;
    pdl_launch_dependents();   // a following verify may stream its target rows meanwhile
    GridBarrier gb = grid_barrier_init(p.barrier);
    int pass = 0;
    for (;; ++pass) {
        const bool use_bias = biased && pass > 0;
        const int32_t* prev = p.tokbuf + ((pass + 1) & 1) * (size_t)R;
        int32_t* cur = p.tokbuf + (pass & 1) * (size_t)R;
        if (blockIdx.x == 0 && threadIdx.x == 0) p.changed[pass + 1] = 0u;
        if (!use_bias && p.vec_l && p.temperature == 0) tile_phase_stream0_t0<LT>(p, p.cta_rec, !biased, nullptr);
        else if (!use_bias && p.vec_l) {
            tile_phase_stream0_t1<LT>(p);
        }
        else tile_phase_cc<LT, WT>(p, use_bias, prev, s_uw);
        if (!grid_barrier(gb, nb, p.status)) return;
        finalize_rows<LT, WT>(p, pass, use_bias, prev, cur, gridDim.x, s_uw);
        if (!grid_barrier(gb, nb, p.status)) return;
        if (!biased) break;
        if (pass >= 1 && __ldcg(&p.changed[pass]) == 0u) break;
        if (pass == p.gamma) break;
    }
    grid_barrier_exit(gb, nb);
    if (blockIdx.x != 0) return;
    chain_fixup(p);
    if (threadIdx.x == 0 && p.passes_out) {
        if (p.passes_max) atomicMax(p.passes_out, biased ? pass : 0);
        else *p.passes_out = biased ? pass : 0;
    }
}

// ----------------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------------
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr int kDraftMaxGrid = 1024;

size_t draft_workspace_bytes(int B, int gamma, int V, int r) {
    (void)r;
    const size_t R = (size_t)B * gamma;
    const size_t n_tiles = ((size_t)V + kDraftTile - 1) / kDraftTile;
    size_t off = kWsHeaderBytes;
    off = align_up(off + sizeof(float4) * R * n_tiles, 256);        // tile records
    off = align_up(off + sizeof(float4) * R * kDraftMaxGrid, 256);  // CTA records
    off = align_up(off + sizeof(float4) * R * kDraftMaxGrid, 256);  // second buffer
    off = align_up(off + sizeof(int32_t) * 2 * R, 256);
    off = align_up(off + sizeof(unsigned) * (gamma + 2), 256);
    off = align_up(off + sizeof(unsigned long long) * 3 * R * kKeyStride, 256);   // argmax keys
    return off;
}

// spec_draft_verify's workspace: the draft's, then a verify workspace.
static size_t dv_verify_offset(int B, int gamma, int V, int r) {
    return align_up(draft_workspace_bytes(B, gamma, V, r), 256);
}
size_t draft_verify_workspace_bytes(int B, int gamma, int V, int r) {
    return dv_verify_offset(B, gamma, V, r) + verify_workspace_bytes(B, gamma, V);
}
void* draft_verify_verify_ws(void* ws, int B, int gamma, int V, int r) {
    return static_cast<char*>(ws) + dv_verify_offset(B, gamma, V, r);
}

void draft_bind_workspace(DraftParams& p, void* ws) {
    char* w = static_cast<char*>(ws);
    WsHeader* h = reinterpret_cast<WsHeader*>(w);
    p.status = &h->status;
    p.barrier = &h->barrier[0][0];
    const size_t R = (size_t)p.B * p.gamma;
    p.n_tiles = (int)(((size_t)p.V + kDraftTile - 1) / kDraftTile);
    size_t off = kWsHeaderBytes;
    p.tile_rec = reinterpret_cast<float4*>(w + off);
    off = align_up(off + sizeof(float4) * R * p.n_tiles, 256);
    p.cta_rec = reinterpret_cast<float4*>(w + off);
    off = align_up(off + sizeof(float4) * R * kDraftMaxGrid, 256);
    p.cta_rec2 = reinterpret_cast<float4*>(w + off);
    off = align_up(off + sizeof(float4) * R * kDraftMaxGrid, 256);
    p.tokbuf = reinterpret_cast<int32_t*>(w + off);
    off = align_up(off + sizeof(int32_t) * 2 * R, 256);
    p.changed = reinterpret_cast<unsigned*>(w + off);
    off = align_up(off + sizeof(unsigned) * (p.gamma + 2), 256);
    p.keys = reinterpret_cast<unsigned long long*>(w + off);
}

template <typename LT, typename WT>
static cudaError_t launch_typed(const DraftParams& p, cudaStream_t stream) {
    const size_t smem = sizeof(float) * (size_t)kWarps * (p.r > 0 ? p.r : 1);
    auto kern = draft_kernel<LT, WT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const int sms = device_sm_count();
    int grid = sms * (occ < 2 ? occ : 2);
    if (grid > kDraftMaxGrid) grid = kDraftMaxGrid;
    if (grid > p.n_tiles) grid = p.n_tiles > 0 ? p.n_tiles : 1;
    DraftParams args = p;
    void* kargs[] = {&args};
    return cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(kThreads), kargs, smem, stream);
}

cudaError_t draft_launch_cc(const DraftParams& p, cudaStream_t stream) {
    const bool lb = p.ldt == SPEC_BF16;
    const bool wb = p.r == 0 ? lb : (p.wdt == SPEC_BF16);
    if (lb && wb) return launch_typed<bf16_t, bf16_t>(p, stream);
    if (lb && !wb) return launch_typed<bf16_t, float>(p, stream);
    if (!lb && wb) return launch_typed<float, bf16_t>(p, stream);
    return launch_typed<float, float>(p, stream);
}

bool draft_tc_supported(const DraftParams& p);
cudaError_t draft_launch_tc(const DraftParams& p, cudaStream_t stream);

// bf16 weights with r a multiple of 64 (<= 256) and at most 256 rows take the tcgen05
// kernel; everything else the CUDA-core kernel.
cudaError_t draft_launch(const DraftParams& p, cudaStream_t stream) {
    if (draft_tc_supported(p)) return draft_launch_tc(p, stream);
    return draft_launch_cc(p, stream);
}

// A batch larger than one launch takes (256 rows on the tcgen05 kernel, kDraftMaxRows
// on the CUDA-core kernel) runs as consecutive launches over slices of whole requests
// on the same stream, reusing one slice's workspace: the requests are independent,
// and b_base keeps each draw's Philox request index the one of the whole batch.
int draft_requests_per_launch(const DraftParams& p) {
    DraftParams q = p;
    q.B = 256 / p.gamma > 0 ? 256 / p.gamma : 1;
    const int per = draft_tc_supported(q) ? q.B : (kDraftMaxRows / p.gamma > 0 ? kDraftMaxRows / p.gamma : 1);
    return p.B < per ? p.B : per;
}

cudaError_t draft_launch_batched(const DraftParams& p, cudaStream_t stream) {
    const int per = draft_requests_per_launch(p);
    if (per >= p.B) return draft_launch(p, stream);
    DraftParams q = p;
    if (p.passes_out) {
        cudaError_t e = cudaMemsetAsync(p.passes_out, 0, sizeof(int32_t), stream);
        if (e != cudaSuccess) return e;
        q.passes_max = 1;
    }
    const size_t lsize = p.ldt == SPEC_BF16 ? 2 : 4;
    for (int b0 = 0; b0 < p.B; b0 += per) {
        const size_t rows = (size_t)b0 * p.gamma;
        q.B = p.B - b0 < per ? p.B - b0 : per;
        q.b_base = p.b_base + b0;
        q.logits = static_cast<const char*>(p.logits) + rows * p.V * lsize;
        q.anchor = p.anchor + b0;
        q.seeds = p.seeds ? p.seeds + b0 : nullptr;
        q.tokens_out = p.tokens_out + rows;
        q.conf_out = p.conf_out + rows;
        q.qtok_out = p.qtok_out ? p.qtok_out + rows : nullptr;
        q.qlogits_out = p.qlogits_out ? p.qlogits_out + rows * p.V : nullptr;
        cudaError_t e = draft_launch(q, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace spec
