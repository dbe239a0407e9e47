// internal.h - launch interfaces between the C ABI layer (abi.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "spec.h"

namespace spec {

// Streaming work granularity of the verify kernels: elements per work item and per
// thread (256 threads x 32 contiguous elements).
constexpr int kVerifyChunk = 8192;

struct VerifyParams {
    const void* target;        // [B, gamma+1, V]
    const void* draft;         // [B, gamma, V] (T=1)
    int tdt, ddt;              // spec_dtype of target / draft
    const int32_t* tokens;     // [B, gamma]
    const uint64_t* seeds;     // [B]
    int B, gamma, V, temperature;
    int nchunk;                // ceil(V / kVerifyChunk)
    int vec_t, vec_d;          // rows 16-byte aligned (vector loads allowed)
    int after_own_draft;       // T=0: launched as the programmatic dependent of the
                               // library's own draft kernel (spec_draft_verify), whose
                               // start already followed every producer of the target
                               // rows; otherwise the kernel waits for the previous
                               // kernel on the stream before it reads anything
    int32_t* n_out;
    int32_t* committed_out;
    int32_t* bonus_out;
    int32_t* near_out;         // nullable
    // workspace regions
    unsigned* status;
    unsigned* done;            // header done[] counters
    unsigned* barrier;         // grid barrier slot (T=1)
    unsigned long long* keys;  // [B*(gamma+1)] argmax keys (T=0)
    unsigned* rowbad;          // [B*(gamma+1)] (T=0)
    float2* stats;             // [B*(2*gamma+1)*nchunk*parts] (m2, s) partials (T=1)
    int parts;                 // partials per (row, chunk): 8 warp segments, or 1 merged
    int4* state;               // [B*2]: mode, n, near, pad | m2p, sp, m2q, sq (float bits)
    float2* ksums;             // [B*nchunk*8] (residual sum, p sum) per warp segment
};

size_t verify_workspace_bytes(int B, int gamma, int V);
void verify_bind_workspace(VerifyParams& p, void* ws);
cudaError_t verify_launch(const VerifyParams& p, cudaStream_t stream);

struct DraftParams {
    const void* logits;        // [B, gamma, V]
    int ldt;                   // spec_dtype
    const int32_t* anchor;     // [B]
    const void* U;             // [V, r]
    const void* Wt;            // [V, r]
    int wdt;
    int r, B, gamma, V, temperature;
    const uint64_t* seeds;
    int32_t* tokens_out;
    float* conf_out;
    float* qtok_out;           // nullable
    float* qlogits_out;        // nullable
    int32_t* passes_out;       // nullable
    int passes_max;            // 1: fold passes_out with atomicMax (a batch run as several launches)
    int b_base;                // batch index of request 0 (the Philox counter's request index)
    int vec_l;                 // logits rows 16-byte aligned
    int vec_w;                 // weight rows 16-byte aligned
    int n_tiles;               // ceil(V / kDraftTile)
    // workspace regions
    unsigned* status;
    unsigned* barrier;         // one barrier slot
    float4* tile_rec;          // [R * n_tiles] per-tile records (T=1): max, sum, argmax, bad
    float4* cta_rec;           // [R * grid] per-(row, CTA) records
    float4* cta_rec2;          // [R * grid] second buffer (passes alternate at T=0)
    int32_t* tokbuf;           // [2 * R] fixed-point iterates
    unsigned* changed;         // [gamma + 2]
    unsigned long long* keys;  // [3][R] argmax keys, one per 128-byte line (T=0, tcgen05); zero between launches
};

constexpr int kDraftTile = 128;   // vocabulary entries per tile

size_t draft_workspace_bytes(int B, int gamma, int V, int r);
void draft_bind_workspace(DraftParams& p, void* ws);
cudaError_t draft_launch(const DraftParams& p, cudaStream_t stream);
// spec_draft_block: requests per launch, and the batch as consecutive launches over
// slices of that many requests (workspace bound for one slice)
int draft_requests_per_launch(const DraftParams& p);
cudaError_t draft_launch_batched(const DraftParams& p, cudaStream_t stream);
// a batch larger than one fixed-point launch, walked position by position on the
// tensor cores (bf16 logits and weights, r a multiple of 64): its own workspace layout
bool draft_pos_supported(const DraftParams& p);
size_t draft_pos_workspace_bytes(int B, int V, int r);
cudaError_t draft_pos_launch(const DraftParams& p, void* ws, cudaStream_t stream);
constexpr int kDraftMaxRows = 4096;   // rows (requests x gamma) of one launch

// spec_draft_verify: [draft workspace | verify workspace]
size_t draft_verify_workspace_bytes(int B, int gamma, int V, int r);
void* draft_verify_verify_ws(void* ws, int B, int gamma, int V, int r);
bool draft_tc_supported(const DraftParams& p);

struct E2etvParams {
    const uint16_t* target;    // bf16 [R, V]
    const uint16_t* draft;     // bf16 [R, V]
    int n_branches, Wb, V;
    int vec_ok;                // V % 8 == 0 (rows 16-byte aligned)
    float* a_out;
    float* surv_out;
    float* loss_out;           // 1 - M, or M alone (share_out) for one shard of a batch
    uint16_t* grad_out;
    int total_branches;        // branches of the whole batch (the mean's count)
    int share_out;
    // layout chosen at launch
    int n_groups;              // groups of CTAs, each processing one branch at a time
    int group_size;            // CTAs per group
    int cols;                  // columns per CTA (multiple of 8)
    // workspace regions
    unsigned* status;
    unsigned* barriers;        // n_groups barrier slots (stride 64 words)
    unsigned* done;
    float2* partials;          // [n_groups][2][group_size][2*Wb]
    float* branch_sum;         // [n_branches]
    unsigned* branch_bad;      // [n_branches]
};

size_t e2etv_workspace_bytes(int n_branches, int Wb, int V);
cudaError_t e2etv_launch(E2etvParams& p, void* ws, cudaStream_t stream);

constexpr int kTopkMax = 32;   // largest top_k of spec_verify_topk
struct TopkParams {
    const void* target;        // [B, gamma+1, V]
    const void* draft;         // [B, gamma, V]
    int tdt, ddt;
    const int32_t* tokens;     // [B, gamma]
    const uint64_t* seeds;     // [B]
    int B, gamma, V, k;
    double top_p;
    int32_t* n_out;
    int32_t* committed_out;
    int32_t* bonus_out;
    int32_t* near_out;         // nullable
    unsigned* status;
    unsigned long long* keys;  // [B*(2*gamma+1)][kTopkMax] each row's largest keys
    unsigned* bad;             // [B*(2*gamma+1)] NaN or +inf in the row
    unsigned long long* part;  // [rows][kTopkPieces][kTopkMax] the pieces' largest keys
    unsigned* part_bad;        // [rows][kTopkPieces]
    unsigned* row_done;        // [rows] pieces finished (returned to 0 by the merge)
    unsigned long long* row_thr;   // [rows] the best bound any piece has published (0 after the merge)
};
constexpr int kTopkPieces = 8;   // most CTAs that share one row of spec_verify_topk
size_t verify_topk_workspace_bytes(int B, int gamma);
cudaError_t verify_topk_launch(TopkParams& p, void* ws, cudaStream_t stream);

// spec_draft_block_topk: the T=1 chain with filtered draws, position by position.
struct DraftTopkLaunch {
    const void* logits;        // [B, gamma, V]
    int ldt;
    const int32_t* anchor;     // [B]
    const void* U;             // bf16 [V, r] (r = 0: no bias)
    const void* Wt;            // bf16 [V, r]
    int r, B, gamma, V, k;
    double top_p;
    const uint64_t* seeds;     // [B]
    int32_t* tokens_out;       // [B, gamma]
    float* conf_out;           // [B, gamma]
    float* qtok_out;           // [B, gamma] (nullable)
};
size_t draft_topk_workspace_bytes(int B, int V);
cudaError_t draft_topk_launch(const DraftTopkLaunch& a, void* ws, cudaStream_t stream);

struct BranchPlanParams {
    const int32_t* trunk;      // [n_refs, Lmax] token ids
    const int32_t* lengths;    // [n_refs]
    int n_refs, Lmax, n_anchors, W;
    uint64_t seed;
    int32_t* anchors_out;      // [n_refs, n_anchors]
    int32_t* anchor_tok_out;   // [n_refs, n_anchors]
    int32_t* parent_out;       // [n_refs, n_anchors * W]
    int32_t* position_out;     // [n_refs, n_anchors * W]
    unsigned* status;
};
cudaError_t branch_plan_launch(const BranchPlanParams& p, cudaStream_t stream);

struct TreeSelectParams {
    const int32_t* parent;     // [n_trees, n_nodes]
    const float* conf;         // [n_trees, n_nodes]
    int n_trees, n_nodes, m;
    double* score_out;         // [n_trees, n_nodes] (nullable)
    int32_t* keep_out;         // [n_trees, n_nodes]
    int32_t* selected_out;     // [n_trees, m] (nullable)
};
cudaError_t tree_select_launch(const TreeSelectParams& p, cudaStream_t stream);

struct TreeVerifyParams {
    const void* target;        // [n_trees, n_nodes + 1, V]: root row, then node rows
    int tdt;
    const int32_t* parent;     // [n_trees, n_nodes]
    const int32_t* token;      // [n_trees, n_nodes]
    const int32_t* keep;       // [n_trees, n_nodes] (nullable: every node kept)
    int n_trees, n_nodes, V;
    int vec_t;                 // rows 16-byte aligned
    int32_t* n_out;            // [n_trees]
    int32_t* path_out;         // [n_trees, n_nodes]
    int32_t* committed_out;    // [n_trees, n_nodes + 1]
    int32_t* bonus_out;        // [n_trees]
    // workspace regions
    unsigned* status;
    unsigned* done;
    unsigned long long* keys;  // [n_trees * (n_nodes + 1)] argmax keys
    unsigned* rowbad;          // [n_trees * (n_nodes + 1)]
    unsigned* first;           // [n_trees * (n_nodes + 1)] n - (lowest matching child) per parent
    unsigned* treebad;         // [n_trees] parents out of order
};
size_t tree_verify_workspace_bytes(int n_trees, int n_nodes);
cudaError_t tree_verify_launch(TreeVerifyParams& p, void* ws, cudaStream_t stream);

int device_sm_count();

cudaError_t verify_budget_launch(const float* conf, int B, int gamma, int budget, const float* cost,
                                 int32_t* gamma_out, float* expected_out, cudaStream_t stream);

// Keeps e as the calling thread's last CUDA error (spec_last_cuda_error) and
// returns SPEC_ERR_CUDA, or SPEC_OK for cudaSuccess.
spec_status record_cuda_error(cudaError_t e);

}  // namespace spec
