// abi.cu - the C ABI (include/spec.h): argument checks, workspace layout, launches.
//
// Every check that can fail is done here, on the host, before anything is enqueued;
// conditions only the device can see go to the workspace status word.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "spec.h"
#include "internal.h"
#include "spec_device.cuh"

namespace spec {

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    static int cache[128] = {0};
    if (dev >= 0 && dev < 128 && cache[dev] > 0) return cache[dev];
    int n = 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    if (dev >= 0 && dev < 128) cache[dev] = n;
    return n;
}

static thread_local int g_last_cuda_error = 0;   // per host thread, like errno

static spec_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return SPEC_OK;
    g_last_cuda_error = (int)e;
    return SPEC_ERR_CUDA;
}

spec_status record_cuda_error(cudaError_t e) { return cuda_status(e); }

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool dtype_ok(int d) { return d == SPEC_F32 || d == SPEC_BF16; }
static size_t dtype_size(int d) { return d == SPEC_F32 ? 4 : 2; }

}  // namespace spec

using namespace spec;

extern "C" {

size_t spec_workspace_bytes(spec_op op, int B, int gamma, int V, int r) {
    if (op == SPEC_OP_DRAFT_TOPK) {
        if (B < 1 || B > 65535 || V < 1 || V > SPEC_MAX_V_DRAFT_TOPK) return 0;
        return draft_topk_workspace_bytes(B, V);
    }
    if (op == SPEC_OP_TREE_VERIFY) {   // gamma is the number of nodes per tree
        if (B < 1 || B > 65535 || gamma < 0 || gamma > SPEC_MAX_TREE_NODES || V < 1 || V > SPEC_MAX_V) return 0;
        return tree_verify_workspace_bytes(B, gamma);
    }
    if (B < 1 || gamma < 1 || gamma > SPEC_MAX_GAMMA || V < 1 || V > SPEC_MAX_V) return 0;
    switch (op) {
        case SPEC_OP_DRAFT:
            // one launch's slice of requests at most (see spec_draft_block)
            if (r < 0 || r > SPEC_MAX_RANK || (long)B * gamma > SPEC_MAX_DRAFT_ROWS) return 0;
            {
                const size_t fp = draft_workspace_bytes(B < kDraftMaxRows / gamma ? B : kDraftMaxRows / gamma, gamma, V, r);
                // a batch of more than 256 rows may take the position-by-position path
                const size_t pos = (long)B * gamma > 256 ? draft_pos_workspace_bytes(B, V, r) : 0;
                return fp > pos ? fp : pos;
            }
        case SPEC_OP_VERIFY:
            if (B > 65535) return 0;
            return verify_workspace_bytes(B, gamma, V);
        case SPEC_OP_DRAFT_VERIFY:
            if (r < 0 || r > SPEC_MAX_RANK || (long)B * gamma > 4096) return 0;
            return draft_verify_workspace_bytes(B, gamma, V, r);
        case SPEC_OP_VERIFY_TOPK:
            if (B > 65535) return 0;
            return verify_topk_workspace_bytes(B, gamma);
        case SPEC_OP_BRANCH_PLAN:
            return kWsHeaderBytes;   // the status word only
        case SPEC_OP_E2ETV:
            if ((long)B * gamma > (1L << 24)) return 0;
            return e2etv_workspace_bytes(B, gamma, V);
        default:
            return 0;
    }
}

spec_status spec_workspace_init(void* workspace, size_t bytes, spec_stream_t stream) {
    if (!workspace || bytes < kWsHeaderBytes) return SPEC_ERR_WORKSPACE;
    return cuda_status(cudaMemsetAsync(workspace, 0, bytes, (cudaStream_t)stream));
}

spec_status spec_get_device_status(const void* workspace, spec_stream_t stream, uint32_t* flags_out) {
    if (!workspace) return SPEC_ERR_WORKSPACE;
    uint32_t flags = 0;
    if (cuda_status(cudaMemcpyAsync(&flags, workspace, sizeof(flags), cudaMemcpyDeviceToHost, (cudaStream_t)stream)))
        return SPEC_ERR_CUDA;
    if (cuda_status(cudaStreamSynchronize((cudaStream_t)stream))) return SPEC_ERR_CUDA;
    if (flags_out) *flags_out = flags;
    if (flags & SPEC_DEV_TIMEOUT) return SPEC_ERR_TIMEOUT;
    if (flags & SPEC_DEV_TOKEN) return SPEC_ERR_TOKEN;
    if (flags & SPEC_DEV_NONFINITE) return SPEC_ERR_NONFINITE;
    return SPEC_OK;
}

const char* spec_status_string(spec_status s) {
    switch (s) {
        case SPEC_OK: return "ok";
        case SPEC_ERR_INVALID_ARG: return "invalid argument (null pointer, temperature, op code)";
        case SPEC_ERR_SHAPE: return "size outside the supported range";
        case SPEC_ERR_DTYPE: return "unknown dtype";
        case SPEC_ERR_ALIGN: return "base pointer not 16-byte aligned";
        case SPEC_ERR_CUDA: return "CUDA runtime error";
        case SPEC_ERR_TIMEOUT: return "a bounded device wait ran out";
        case SPEC_ERR_NONFINITE: return "a row holds NaN/+inf or no finite entry";
        case SPEC_ERR_TOKEN: return "a token outside [0, V)";
        case SPEC_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

int spec_last_cuda_error(void) { return g_last_cuda_error; }

const char* spec_last_cuda_error_string(void) {
    return g_last_cuda_error ? cudaGetErrorString((cudaError_t)g_last_cuda_error) : "no CUDA error";
}

spec_status spec_draft_block(const void* draft_logits, spec_dtype logits_dtype, const int32_t* anchor,
                             const void* U, const void* Wt, spec_dtype w_dtype, int r, int B, int gamma, int V,
                             int temperature, const uint64_t* seeds, int32_t* tokens_out, float* conf_out,
                             float* qtok_out, float* qlogits_out, int32_t* passes_out, void* workspace,
                             size_t workspace_bytes, spec_stream_t stream) {
    if (!dtype_ok(logits_dtype) || (r > 0 && !dtype_ok(w_dtype))) return SPEC_ERR_DTYPE;
    if (B < 1 || gamma < 1 || gamma > SPEC_MAX_GAMMA || V < 1 || V > SPEC_MAX_V || r < 0 || r > SPEC_MAX_RANK ||
        (long)B * gamma > SPEC_MAX_DRAFT_ROWS)
        return SPEC_ERR_SHAPE;
    if (temperature != 0 && temperature != 1) return SPEC_ERR_INVALID_ARG;
    if (!draft_logits || !anchor || !tokens_out || !conf_out) return SPEC_ERR_INVALID_ARG;
    if (r > 0 && (!U || !Wt)) return SPEC_ERR_INVALID_ARG;
    if (temperature == 1 && !seeds) return SPEC_ERR_INVALID_ARG;
    if (!aligned16(draft_logits) || (r > 0 && (!aligned16(U) || !aligned16(Wt))) ||
        (qlogits_out && !aligned16(qlogits_out)))
        return SPEC_ERR_ALIGN;

    DraftParams p;
    memset(&p, 0, sizeof(p));
    p.logits = draft_logits;
    p.ldt = logits_dtype;
    p.anchor = anchor;
    p.U = U;
    p.Wt = Wt;
    p.wdt = r > 0 ? w_dtype : logits_dtype;
    p.r = r;
    p.B = B;
    p.gamma = gamma;
    p.V = V;
    p.temperature = temperature;
    p.seeds = seeds;
    p.tokens_out = tokens_out;
    p.conf_out = conf_out;
    p.qtok_out = qtok_out;
    p.qlogits_out = qlogits_out;
    p.passes_out = passes_out;
    p.vec_l = ((size_t)V * dtype_size(logits_dtype)) % 16 == 0;
    p.vec_w = r > 0 && ((size_t)r * dtype_size(w_dtype)) % 16 == 0;
    // a batch of more than 256 rows with bf16 logits and weights and r a multiple of 64
    // walks the chain position by position, reading each row and the weights once per
    // position
    if (draft_pos_supported(p)) {
        if (!workspace || workspace_bytes < draft_pos_workspace_bytes(B, V, r)) return SPEC_ERR_WORKSPACE;
        return cuda_status(draft_pos_launch(p, workspace, (cudaStream_t)stream));
    }
    // otherwise a batch larger than one launch runs as consecutive launches over slices
    // of requests, each with the workspace of one slice
    const int per = draft_requests_per_launch(p);
    const size_t need = draft_workspace_bytes(per, gamma, V, r);
    if (!workspace || workspace_bytes < need) return SPEC_ERR_WORKSPACE;
    DraftParams bound = p;
    bound.B = per;
    draft_bind_workspace(bound, workspace);
    bound.B = B;
    return cuda_status(draft_launch_batched(bound, (cudaStream_t)stream));
}

spec_status spec_verify(const void* target_logits, spec_dtype target_dtype, const void* draft_logits,
                        spec_dtype draft_dtype, const int32_t* draft_tokens, int B, int gamma, int V, int temperature,
                        const uint64_t* seeds, int32_t* n_accepted_out, int32_t* committed_out, int32_t* bonus_out,
                        int32_t* near_tie_out, void* workspace, size_t workspace_bytes, spec_stream_t stream) {
    if (!dtype_ok(target_dtype) || (temperature == 1 && !dtype_ok(draft_dtype))) return SPEC_ERR_DTYPE;
    if (B < 1 || B > 65535 || gamma < 1 || gamma > SPEC_MAX_GAMMA || V < 1 || V > SPEC_MAX_V) return SPEC_ERR_SHAPE;
    if (temperature != 0 && temperature != 1) return SPEC_ERR_INVALID_ARG;
    if (!target_logits || !draft_tokens || !n_accepted_out || !committed_out || !bonus_out)
        return SPEC_ERR_INVALID_ARG;
    if (temperature == 1 && (!draft_logits || !seeds)) return SPEC_ERR_INVALID_ARG;
    if (!aligned16(target_logits) || (temperature == 1 && !aligned16(draft_logits))) return SPEC_ERR_ALIGN;
    const size_t need = verify_workspace_bytes(B, gamma, V);
    if (!workspace || workspace_bytes < need) return SPEC_ERR_WORKSPACE;

    VerifyParams p;
    memset(&p, 0, sizeof(p));
    p.target = target_logits;
    p.draft = temperature == 1 ? draft_logits : nullptr;
    p.tdt = target_dtype;
    p.ddt = temperature == 1 ? draft_dtype : target_dtype;
    p.tokens = draft_tokens;
    p.seeds = seeds;
    p.B = B;
    p.gamma = gamma;
    p.V = V;
    p.temperature = temperature;
    p.nchunk = (V + kVerifyChunk - 1) / kVerifyChunk;
    p.vec_t = ((size_t)V * dtype_size(target_dtype)) % 16 == 0;
    p.vec_d = temperature == 1 && ((size_t)V * dtype_size(draft_dtype)) % 16 == 0;
    p.n_out = n_accepted_out;
    p.committed_out = committed_out;
    p.bonus_out = bonus_out;
    p.near_out = near_tie_out;
    verify_bind_workspace(p, workspace);
    return cuda_status(verify_launch(p, (cudaStream_t)stream));
}

spec_status spec_draft_verify(const void* draft_logits, spec_dtype logits_dtype, const int32_t* anchor,
                              const void* U, const void* Wt, spec_dtype w_dtype, int r, int B, int gamma, int V,
                              const void* target_logits, spec_dtype target_dtype, int32_t* tokens_out,
                              float* conf_out, float* qtok_out, int32_t* passes_out, int32_t* n_accepted_out,
                              int32_t* committed_out, int32_t* bonus_out, void* workspace, size_t workspace_bytes,
                              spec_stream_t stream) {
    if (!dtype_ok(logits_dtype) || !dtype_ok(target_dtype) || (r > 0 && !dtype_ok(w_dtype))) return SPEC_ERR_DTYPE;
    if (B < 1 || gamma < 1 || gamma > SPEC_MAX_GAMMA || V < 1 || V > SPEC_MAX_V || r < 0 || r > SPEC_MAX_RANK ||
        (long)B * gamma > 4096)
        return SPEC_ERR_SHAPE;
    if (!draft_logits || !anchor || !tokens_out || !conf_out || !target_logits || !n_accepted_out || !committed_out ||
        !bonus_out)
        return SPEC_ERR_INVALID_ARG;
    if (r > 0 && (!U || !Wt)) return SPEC_ERR_INVALID_ARG;
    if (!aligned16(draft_logits) || !aligned16(target_logits) || (r > 0 && (!aligned16(U) || !aligned16(Wt))))
        return SPEC_ERR_ALIGN;
    const size_t need = draft_verify_workspace_bytes(B, gamma, V, r);
    if (!workspace || workspace_bytes < need) return SPEC_ERR_WORKSPACE;

    DraftParams p;
    memset(&p, 0, sizeof(p));
    p.logits = draft_logits;
    p.ldt = logits_dtype;
    p.anchor = anchor;
    p.U = U;
    p.Wt = Wt;
    p.wdt = r > 0 ? w_dtype : logits_dtype;
    p.r = r;
    p.B = B;
    p.gamma = gamma;
    p.V = V;
    p.temperature = 0;
    p.tokens_out = tokens_out;
    p.conf_out = conf_out;
    p.qtok_out = qtok_out;
    p.passes_out = passes_out;
    p.vec_l = ((size_t)V * dtype_size(logits_dtype)) % 16 == 0;
    p.vec_w = r > 0 && ((size_t)r * dtype_size(w_dtype)) % 16 == 0;
    draft_bind_workspace(p, workspace);
    const bool vec_t = ((size_t)V * dtype_size(target_dtype)) % 16 == 0;
    // the draft kernel, then verify T=0 as its programmatic dependent (its target-row
    // pass may start while the draft finishes); verify writes its flags into this
    // workspace's status word
    spec_status st = cuda_status(draft_launch(p, (cudaStream_t)stream));
    if (st != SPEC_OK) return st;
    VerifyParams v;
    memset(&v, 0, sizeof(v));
    v.target = target_logits;
    v.tdt = target_dtype;
    v.ddt = target_dtype;
    v.tokens = tokens_out;
    v.B = B;
    v.gamma = gamma;
    v.V = V;
    v.temperature = 0;
    v.nchunk = (V + kVerifyChunk - 1) / kVerifyChunk;
    v.vec_t = vec_t;
    v.n_out = n_accepted_out;
    v.committed_out = committed_out;
    v.bonus_out = bonus_out;
    v.after_own_draft = 1;
    verify_bind_workspace(v, draft_verify_verify_ws(workspace, B, gamma, V, r));
    v.status = p.status;
    return cuda_status(verify_launch(v, (cudaStream_t)stream));
}

spec_status spec_draft_block_topk(const void* draft_logits, spec_dtype logits_dtype, const int32_t* anchor,
                                  const void* U, const void* Wt, spec_dtype w_dtype, int r, int B, int gamma, int V,
                                  int top_k, double top_p, const uint64_t* seeds, int32_t* tokens_out,
                                  float* conf_out, float* qtok_out, void* workspace, size_t workspace_bytes,
                                  spec_stream_t stream) {
    if (!dtype_ok(logits_dtype) || (r > 0 && w_dtype != SPEC_BF16)) return SPEC_ERR_DTYPE;
    if (B < 1 || B > 65535 || gamma < 1 || gamma > SPEC_MAX_GAMMA || V < 1 || V > SPEC_MAX_V_DRAFT_TOPK || r < 0 ||
        r > SPEC_MAX_RANK || (r % 16) != 0 || top_k < 1 || top_k > SPEC_MAX_TOP_K)
        return SPEC_ERR_SHAPE;
    if (!(top_p > 0.0 && top_p <= 1.0)) return SPEC_ERR_INVALID_ARG;
    if (!draft_logits || !anchor || !seeds || !tokens_out || !conf_out) return SPEC_ERR_INVALID_ARG;
    if (r > 0 && (!U || !Wt)) return SPEC_ERR_INVALID_ARG;
    if (!aligned16(draft_logits) || (r > 0 && (!aligned16(U) || !aligned16(Wt)))) return SPEC_ERR_ALIGN;
    if (!workspace || workspace_bytes < draft_topk_workspace_bytes(B, V)) return SPEC_ERR_WORKSPACE;
    DraftTopkLaunch d;
    memset(&d, 0, sizeof(d));
    d.logits = draft_logits;
    d.ldt = logits_dtype;
    d.anchor = anchor;
    d.U = r > 0 ? U : nullptr;
    d.Wt = r > 0 ? Wt : nullptr;
    d.r = r;
    d.B = B;
    d.gamma = gamma;
    d.V = V;
    d.k = top_k;
    d.top_p = top_p;
    d.seeds = seeds;
    d.tokens_out = tokens_out;
    d.conf_out = conf_out;
    d.qtok_out = qtok_out;
    return cuda_status(draft_topk_launch(d, workspace, (cudaStream_t)stream));
}

spec_status spec_tree_select(const int32_t* parent, const float* conf, int n_trees, int n_nodes, int m,
                             double* score_out, int32_t* keep_out, int32_t* selected_out, spec_stream_t stream) {
    if (n_trees < 1 || n_trees > 65535 || n_nodes < 1 || n_nodes > SPEC_MAX_TREE_NODES || m < 0)
        return SPEC_ERR_SHAPE;
    if (!parent || !conf || !keep_out) return SPEC_ERR_INVALID_ARG;
    TreeSelectParams p;
    memset(&p, 0, sizeof(p));
    p.parent = parent;
    p.conf = conf;
    p.n_trees = n_trees;
    p.n_nodes = n_nodes;
    p.m = m;
    p.score_out = score_out;
    p.keep_out = keep_out;
    p.selected_out = selected_out;
    return cuda_status(tree_select_launch(p, (cudaStream_t)stream));
}

spec_status spec_tree_verify(const void* target_logits, spec_dtype target_dtype, const int32_t* parent,
                             const int32_t* token, const int32_t* keep, int n_trees, int n_nodes, int V,
                             int32_t* n_accepted_out, int32_t* path_out, int32_t* committed_out, int32_t* bonus_out,
                             void* workspace, size_t workspace_bytes, spec_stream_t stream) {
    if (!dtype_ok(target_dtype)) return SPEC_ERR_DTYPE;
    if (n_trees < 1 || n_trees > 65535 || n_nodes < 0 || n_nodes > SPEC_MAX_TREE_NODES || V < 1 || V > SPEC_MAX_V)
        return SPEC_ERR_SHAPE;
    if (!target_logits || !n_accepted_out || !committed_out || !bonus_out) return SPEC_ERR_INVALID_ARG;
    if (n_nodes > 0 && (!parent || !token || !path_out)) return SPEC_ERR_INVALID_ARG;
    if (!aligned16(target_logits)) return SPEC_ERR_ALIGN;
    const size_t need = tree_verify_workspace_bytes(n_trees, n_nodes);
    if (!workspace || workspace_bytes < need) return SPEC_ERR_WORKSPACE;
    TreeVerifyParams p;
    memset(&p, 0, sizeof(p));
    p.target = target_logits;
    p.tdt = target_dtype;
    p.parent = parent;
    p.token = token;
    p.keep = n_nodes > 0 ? keep : nullptr;
    p.n_trees = n_trees;
    p.n_nodes = n_nodes;
    p.V = V;
    p.vec_t = ((size_t)V * dtype_size(target_dtype)) % 16 == 0;
    p.n_out = n_accepted_out;
    p.path_out = path_out;
    p.committed_out = committed_out;
    p.bonus_out = bonus_out;
    return cuda_status(tree_verify_launch(p, workspace, (cudaStream_t)stream));
}

spec_status spec_e2etv(const uint16_t* target_logits, const uint16_t* draft_logits, int n_branches, int Wb, int V,
                       float* a_out, float* surv_out, float* loss_out, uint16_t* grad_out, void* workspace,
                       size_t workspace_bytes, spec_stream_t stream) {
    if (n_branches < 1 || Wb < 1 || Wb > SPEC_MAX_GAMMA || V < 1 || V > SPEC_MAX_V ||
        (long)n_branches * Wb > (1L << 24))
        return SPEC_ERR_SHAPE;
    if (!target_logits || !draft_logits || !a_out || !surv_out || !loss_out || !grad_out)
        return SPEC_ERR_INVALID_ARG;
    if (!aligned16(target_logits) || !aligned16(draft_logits) || !aligned16(grad_out)) return SPEC_ERR_ALIGN;
    const size_t need = e2etv_workspace_bytes(n_branches, Wb, V);
    if (!workspace || workspace_bytes < need) return SPEC_ERR_WORKSPACE;

    E2etvParams p;
    memset(&p, 0, sizeof(p));
    p.target = target_logits;
    p.draft = draft_logits;
    p.n_branches = n_branches;
    p.Wb = Wb;
    p.V = V;
    p.vec_ok = (V % 8) == 0;
    p.a_out = a_out;
    p.surv_out = surv_out;
    p.loss_out = loss_out;
    p.grad_out = grad_out;
    p.total_branches = n_branches;
    p.share_out = 0;
    return cuda_status(e2etv_launch(p, workspace, (cudaStream_t)stream));
}

spec_status spec_e2etv_shard(const uint16_t* target_logits, const uint16_t* draft_logits, int n_branches, int Wb,
                             int V, int total_branches, float* a_out, float* surv_out, float* msum_out,
                             uint16_t* grad_out, void* workspace, size_t workspace_bytes, spec_stream_t stream) {
    if (n_branches < 1 || Wb < 1 || Wb > SPEC_MAX_GAMMA || V < 1 || V > SPEC_MAX_V ||
        (long)n_branches * Wb > (1L << 24) || total_branches < n_branches)
        return SPEC_ERR_SHAPE;
    if (!target_logits || !draft_logits || !a_out || !surv_out || !msum_out || !grad_out)
        return SPEC_ERR_INVALID_ARG;
    if (!aligned16(target_logits) || !aligned16(draft_logits) || !aligned16(grad_out)) return SPEC_ERR_ALIGN;
    const size_t need = e2etv_workspace_bytes(n_branches, Wb, V);
    if (!workspace || workspace_bytes < need) return SPEC_ERR_WORKSPACE;

    E2etvParams p;
    memset(&p, 0, sizeof(p));
    p.target = target_logits;
    p.draft = draft_logits;
    p.n_branches = n_branches;
    p.Wb = Wb;
    p.V = V;
    p.vec_ok = (V % 8) == 0;
    p.a_out = a_out;
    p.surv_out = surv_out;
    p.loss_out = msum_out;
    p.grad_out = grad_out;
    p.total_branches = total_branches;
    p.share_out = 1;
    return cuda_status(e2etv_launch(p, workspace, (cudaStream_t)stream));
}

spec_status spec_verify_budget(const float* conf, int B, int gamma, int budget, const float* cost_us,
                               int32_t* gamma_out, float* expected_out, spec_stream_t stream) {
    if (!conf || !gamma_out) return SPEC_ERR_INVALID_ARG;
    if (B < 1 || gamma < 1 || gamma > SPEC_MAX_GAMMA || (long)B * gamma > SPEC_MAX_BUDGET_CANDIDATES)
        return SPEC_ERR_SHAPE;
    if (budget < 0 || (long)budget > (long)B * gamma) return SPEC_ERR_SHAPE;
    return cuda_status(verify_budget_launch(conf, B, gamma, budget, cost_us, gamma_out, expected_out,
                                            (cudaStream_t)stream));
}

spec_status spec_branch_plan(const int32_t* trunk_tokens, const int32_t* lengths, int n_refs, int Lmax,
                             int n_anchors, int W, uint64_t seed, int32_t* anchors_out, int32_t* anchor_tok_out,
                             int32_t* parent_out, int32_t* position_out, void* workspace, size_t workspace_bytes,
                             spec_stream_t stream) {
    if (!trunk_tokens || !lengths || !anchors_out || !anchor_tok_out || !parent_out || !position_out)
        return SPEC_ERR_INVALID_ARG;
    if (n_refs < 1 || n_refs > 65535 || Lmax < 1 || Lmax > SPEC_MAX_TRUNK || n_anchors < 1 || n_anchors > Lmax ||
        W < 1 || W > SPEC_MAX_GAMMA)
        return SPEC_ERR_SHAPE;
    if (!workspace || workspace_bytes < kWsHeaderBytes) return SPEC_ERR_WORKSPACE;
    BranchPlanParams p;
    memset(&p, 0, sizeof(p));
    p.trunk = trunk_tokens;
    p.lengths = lengths;
    p.n_refs = n_refs;
    p.Lmax = Lmax;
    p.n_anchors = n_anchors;
    p.W = W;
    p.seed = seed;
    p.anchors_out = anchors_out;
    p.anchor_tok_out = anchor_tok_out;
    p.parent_out = parent_out;
    p.position_out = position_out;
    p.status = &reinterpret_cast<WsHeader*>(workspace)->status;
    return cuda_status(branch_plan_launch(p, (cudaStream_t)stream));
}

spec_status spec_verify_topk(const void* target_logits, spec_dtype target_dtype, const void* draft_logits,
                             spec_dtype draft_dtype, const int32_t* draft_tokens, int B, int gamma, int V, int top_k,
                             double top_p, const uint64_t* seeds, int32_t* n_accepted_out, int32_t* committed_out,
                             int32_t* bonus_out, int32_t* near_tie_out, void* workspace, size_t workspace_bytes,
                             spec_stream_t stream) {
    if (!dtype_ok(target_dtype) || !dtype_ok(draft_dtype)) return SPEC_ERR_DTYPE;
    if (B < 1 || B > 65535 || gamma < 1 || gamma > SPEC_MAX_GAMMA || V < 1 || V > SPEC_MAX_V || top_k < 1 ||
        top_k > SPEC_MAX_TOP_K)
        return SPEC_ERR_SHAPE;
    if (!(top_p > 0.0 && top_p <= 1.0)) return SPEC_ERR_INVALID_ARG;
    if (!target_logits || !draft_logits || !draft_tokens || !seeds || !n_accepted_out || !committed_out ||
        !bonus_out)
        return SPEC_ERR_INVALID_ARG;
    if (!aligned16(target_logits) || !aligned16(draft_logits)) return SPEC_ERR_ALIGN;
    if (!workspace || workspace_bytes < verify_topk_workspace_bytes(B, gamma)) return SPEC_ERR_WORKSPACE;
    TopkParams p;
    memset(&p, 0, sizeof(p));
    p.target = target_logits;
    p.draft = draft_logits;
    p.tdt = target_dtype;
    p.ddt = draft_dtype;
    p.tokens = draft_tokens;
    p.seeds = seeds;
    p.B = B;
    p.gamma = gamma;
    p.V = V;
    p.k = top_k;
    p.top_p = top_p;
    p.n_out = n_accepted_out;
    p.committed_out = committed_out;
    p.bonus_out = bonus_out;
    p.near_out = near_tie_out;
    return cuda_status(verify_topk_launch(p, workspace, (cudaStream_t)stream));
}

}  // extern "C"
