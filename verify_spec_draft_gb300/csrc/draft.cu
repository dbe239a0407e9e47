// draft.cu - DSpark block draft with the rank-r Markov logit bias (spec_draft_block).
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
// The initial guess is the unbiased choice of each position (pass 0), which the
// small bias rarely changes, so one biased pass usually confirms it.
//
// One cooperative persistent launch runs every pass; phases are separated by a
// bounded grid barrier:  [tile phase: per (row, 128-wide vocabulary tile) softmax
// statistics and argmax of z]  ->  barrier  ->  [finalize: one warp per row merges
// the tiles in vocabulary order, picks x_j (argmax, or inverse CDF locating the tile
// then the entry), writes outputs, flags a change]  ->  barrier  ->  next pass.
//
// This file computes the bias on CUDA cores in float32 (used for float32 weights and
// as the general path); draft_tc.cu holds the tcgen05 tensor-core tile phase.
#include "spec_device.cuh"
#include "internal.h"

namespace spec {

constexpr int kRowBlock = 32;   // rows whose U[x_{j-1}] is cached in shared memory

// dot(u, Wt[v, :]) in float32, k ascending (the same order everywhere).
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

__device__ __forceinline__ int prev_token(const DraftParams& p, const int32_t* prev, int row) {
    const int j = row % p.gamma;
    return j == 0 ? p.anchor[row / p.gamma] : __ldcg(&prev[row - 1]);
}

// z for the four entries v = tile*128 + lane + 32*i of one row.
template <typename LT, typename WT>
__device__ __forceinline__ void row_tile_z(const DraftParams& p, int row, int tile, bool use_bias,
                                           const float* u, float (&z)[4]) {
    const LT* lrow = static_cast<const LT*>(p.logits) + (size_t)row * p.V;
    const WT* Wt = static_cast<const WT*>(p.Wt);
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const long v = (long)tile * kDraftTile + lane + 32 * i;
        if (v < p.V) {
            float zi = load_one(lrow + v);
            if (use_bias) zi += bias_dot<WT>(u, Wt + (size_t)v * p.r, p.r, p.vec_w != 0);
            z[i] = zi;
        } else {
            z[i] = -INFINITY;
        }
    }
}

template <typename LT, typename WT>
__device__ void tile_phase(const DraftParams& p, bool use_bias, const int32_t* prev, float* s_u, int* s_ok) {
    const int R = p.B * p.gamma;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const WT* U = static_cast<const WT*>(p.U);
    const bool write_z = p.qlogits_out != nullptr && (use_bias || p.r == 0);
    for (int rb0 = 0; rb0 < R; rb0 += kRowBlock) {
        const int rb1 = min(R, rb0 + kRowBlock);
        if (use_bias) {
            __syncthreads();
            for (int i = threadIdx.x; i < (rb1 - rb0); i += blockDim.x) {
                const int x = prev_token(p, prev, rb0 + i);
                s_ok[i] = (x >= 0 && x < p.V) ? 1 : 0;
            }
            __syncthreads();
            for (int idx = threadIdx.x; idx < (rb1 - rb0) * p.r; idx += blockDim.x) {
                const int i = idx / p.r, k = idx - i * p.r;
                float val = 0.0f;
                if (s_ok[i]) val = load_one(U + (size_t)prev_token(p, prev, rb0 + i) * p.r + k);
                s_u[i * p.r + k] = val;
            }
            __syncthreads();
        }
        for (int tile = blockIdx.x; tile < p.n_tiles; tile += gridDim.x) {
            for (int row = rb0 + warp; row < rb1; row += kWarps) {
                float z[4];
                row_tile_z<LT, WT>(p, row, tile, use_bias, s_u + (size_t)(row - rb0) * p.r, z);
                int bad = 0;
                unsigned long long key = 0ull;
                float m = -INFINITY;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const long v = (long)tile * kDraftTile + lane + 32 * i;
                    if (v < p.V) {
                        bad |= bad_logit(z[i]) ? 1 : 0;
                        const unsigned long long k = argmax_key(z[i], (uint32_t)v);
                        key = k > key ? k : key;
                        m = fmaxf(m, z[i]);
                    }
                }
                m = warp_max(m);
                float s = 0.0f;
                if (m != -INFINITY) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) s += expf(z[i] - m);
                }
                s = warp_sum(s);
                key = warp_max_u64(key);
                bad = warp_or(bad);
                if (use_bias && !s_ok[row - rb0]) bad = 2;
                if (lane == 0)
                    p.tile_stats[(size_t)row * p.n_tiles + tile] =
                        make_float4(m, s, __int_as_float((int)key_index(key)), (float)bad);
                if (write_z) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const long v = (long)tile * kDraftTile + lane + 32 * i;
                        if (v < p.V) p.qlogits_out[(size_t)row * p.V + v] = z[i];
                    }
                }
            }
        }
    }
}

template <typename LT, typename WT>
__device__ void finalize_phase(const DraftParams& p, int pass, bool use_bias, const int32_t* prev,
                               int32_t* cur, float* s_u_warp) {
    const int R = p.B * p.gamma;
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int TW = gridDim.x * kWarps;
    const int K = (p.n_tiles + 31) / 32;
    const WT* U = static_cast<const WT*>(p.U);
    for (int row = gw; row < R; row += TW) {
        const int b = row / p.gamma, j = row % p.gamma;
        const size_t base = (size_t)row * p.n_tiles;
        const int t0 = lane * K, t1 = min(p.n_tiles, t0 + K);
        Stat seg = stat_empty();
        unsigned long long key = 0ull;
        int bad = 0;
        for (int t = t0; t < t1; ++t) {
            const float4 ts = __ldcg(&p.tile_stats[base + t]);
            seg = stat_merge(seg, Stat{ts.x, ts.y});
            const unsigned long long k = argmax_key(ts.x, (uint32_t)__float_as_int(ts.z));
            key = (ts.x != -INFINITY && k > key) ? k : key;
            bad |= (ts.w != 0.0f) ? 1 : 0;
        }
        const Stat rs = warp_stat(seg);
        key = warp_max_u64(key);
        bad = warp_or(bad);
        const float m = rs.m, Z = rs.s;
        int x = -1;
        float qx = NAN;
        const bool valid = !bad && m != -INFINITY;
        if (valid && p.temperature == 0) {
            x = (int)key_index(key);
            qx = 1.0f / Z;
        } else if (valid) {
            const float u = philox_uniform(p.seeds[b], (uint64_t)b, (uint64_t)(j + 1), 0);
            const float thr = u * Z;
            // lane segments rescaled to the row maximum, scanned in vocabulary order
            const float sl = (seg.m == -INFINITY) ? 0.0f : seg.s * expf(seg.m - m);
            const float incl = warp_inclusive_scan(sl);
            const unsigned cross = __ballot_sync(0xffffffffu, incl > thr);
            int tile = -1;
            float tloc = INFINITY;
            if (cross) {
                const int L = __ffs(cross) - 1;
                if (lane == L) {
                    float run = incl - sl;
                    for (int t = t0; t < t1; ++t) {
                        const float4 ts = __ldcg(&p.tile_stats[base + t]);
                        const float w = (ts.x == -INFINITY) ? 0.0f : ts.y * expf(ts.x - m);
                        if (run + w > thr) { tile = t; tloc = thr - run; break; }
                        run += w;
                    }
                    if (tile < 0) { tile = t1 - 1; tloc = INFINITY; }
                }
                tile = __shfl_sync(0xffffffffu, tile, L);
                tloc = __shfl_sync(0xffffffffu, tloc, L);
            } else {
                int last = -1;
                for (int t = t0; t < t1; ++t) {
                    const float4 ts = __ldcg(&p.tile_stats[base + t]);
                    if (ts.x != -INFINITY && ts.y > 0.0f) last = t;
                }
                const unsigned has = __ballot_sync(0xffffffffu, last >= 0);
                tile = has ? __shfl_sync(0xffffffffu, last, 31 - __clz(has)) : 0;
            }
            tile = max(0, min(tile, p.n_tiles - 1));
            // recompute the tile's z with the tile phase's own arithmetic and scan it
            if (use_bias) {
                const int xp = prev_token(p, prev, row);
                for (int k = lane; k < p.r; k += 32) s_u_warp[k] = load_one(U + (size_t)xp * p.r + k);
                __syncwarp();
            }
            float z[4];
            row_tile_z<LT, WT>(p, row, tile, use_bias, s_u_warp, z);
            float carry = 0.0f;
            int found = -1, last_pos = -1;
            float zfound = 0.0f, zlast = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float w = expf(z[i] - m);
                const float inc = warp_inclusive_scan(w) + carry;
                const unsigned hit = __ballot_sync(0xffffffffu, w > 0.0f && inc > tloc);
                if (found < 0 && hit) {
                    const int L = __ffs(hit) - 1;
                    found = tile * kDraftTile + 32 * i + L;
                    zfound = __shfl_sync(0xffffffffu, z[i], L);
                }
                const unsigned pos = __ballot_sync(0xffffffffu, w > 0.0f);
                if (pos) {
                    const int L = 31 - __clz(pos);
                    last_pos = tile * kDraftTile + 32 * i + L;
                    zlast = __shfl_sync(0xffffffffu, z[i], L);
                }
                carry = __shfl_sync(0xffffffffu, inc, 31);
            }
            if (found < 0) { found = last_pos; zfound = zlast; }
            x = found;
            qx = expf(zfound - m) / Z;
            __syncwarp();
        }
        if (lane == 0) {
            p.tokens_out[row] = x;
            p.conf_out[row] = valid ? 1.0f / Z : NAN;
            if (p.qtok_out) p.qtok_out[row] = valid ? qx : NAN;
            cur[row] = x;
            if (pass > 0 && __ldcg(&prev[row]) != x) atomicOr(&p.changed[pass], 1u);
        }
    }
}

template <typename LT, typename WT>
__global__ void __launch_bounds__(kThreads) draft_kernel(DraftParams p) {
    extern __shared__ float s_dyn[];
    float* s_u = s_dyn;                                       // [kRowBlock * r]
    float* s_uw = s_dyn + (size_t)kRowBlock * p.r;            // [kWarps * r]
    __shared__ int s_ok[kRowBlock];
    const bool biased = p.r > 0;
    const unsigned nb = gridDim.x;
    int pass = 0;
    for (;; ++pass) {
        const bool use_bias = biased && pass > 0;
        const int32_t* prev = p.tokbuf + ((pass + 1) & 1) * (size_t)(p.B * p.gamma);
        int32_t* cur = p.tokbuf + (pass & 1) * (size_t)(p.B * p.gamma);
        if (blockIdx.x == 0 && threadIdx.x == 0) p.changed[pass + 1] = 0u;
        tile_phase<LT, WT>(p, use_bias, prev, s_u, s_ok);
        if (!block_barrier(p.barrier, nb, p.status)) return;
        finalize_phase<LT, WT>(p, pass, use_bias, prev, cur, s_uw + (size_t)(threadIdx.x >> 5) * (p.r > 0 ? p.r : 1));
        if (!block_barrier(p.barrier, nb, p.status)) return;
        if (!biased) break;
        if (pass >= 1 && __ldcg(&p.changed[pass]) == 0u) break;
        if (pass == p.gamma) break;
    }
    if (blockIdx.x != 0) return;
    // chain validity: an anchor outside [0, V) or an invalid position voids the rest
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
    if (threadIdx.x == 0 && p.passes_out) *p.passes_out = biased ? pass : 0;
}

// ----------------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------------
static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t draft_workspace_bytes(int B, int gamma, int V, int r) {
    (void)r;
    const size_t R = (size_t)B * gamma;
    const size_t n_tiles = ((size_t)V + kDraftTile - 1) / kDraftTile;
    size_t off = kWsHeaderBytes;
    off = align_up(off + sizeof(float4) * R * n_tiles, 256);
    off = align_up(off + sizeof(int32_t) * 2 * R, 256);
    off = align_up(off + sizeof(unsigned) * (gamma + 2), 256);
    return off;
}

void draft_bind_workspace(DraftParams& p, void* ws) {
    char* w = static_cast<char*>(ws);
    WsHeader* h = reinterpret_cast<WsHeader*>(w);
    p.status = &h->status;
    p.barrier = &h->barrier[0][0];
    const size_t R = (size_t)p.B * p.gamma;
    p.n_tiles = (int)(((size_t)p.V + kDraftTile - 1) / kDraftTile);
    size_t off = kWsHeaderBytes;
    p.tile_stats = reinterpret_cast<float4*>(w + off);
    off = align_up(off + sizeof(float4) * R * p.n_tiles, 256);
    p.tokbuf = reinterpret_cast<int32_t*>(w + off);
    off = align_up(off + sizeof(int32_t) * 2 * R, 256);
    p.changed = reinterpret_cast<unsigned*>(w + off);
}

template <typename LT, typename WT>
static cudaError_t launch_typed(const DraftParams& p, cudaStream_t stream) {
    const size_t smem = sizeof(float) * ((size_t)kRowBlock + kWarps) * (p.r > 0 ? p.r : 1);
    auto kern = draft_kernel<LT, WT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const int sms = device_sm_count();
    int grid = sms * (occ < 2 ? occ : 2);
    if (grid > p.n_tiles) grid = p.n_tiles > 0 ? p.n_tiles : 1;
    DraftParams args = p;
    void* kargs[] = {&args};
    return cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(kThreads), kargs, smem, stream);
}

cudaError_t draft_launch(const DraftParams& p, cudaStream_t stream) {
    const bool lb = p.ldt == SPEC_BF16;
    const bool wb = p.r == 0 ? lb : (p.wdt == SPEC_BF16);
    if (lb && wb) return launch_typed<bf16_t, bf16_t>(p, stream);
    if (lb && !wb) return launch_typed<bf16_t, float>(p, stream);
    if (!lb && wb) return launch_typed<float, bf16_t>(p, stream);
    return launch_typed<float, float>(p, stream);
}

}  // namespace spec
