// spec_device.cuh - device helpers shared by the draft, verify and E2E-TV kernels.
//
// Row loads (128-bit, read-only, L1 no-allocate), Philox4x64-10, order-preserving
// argmax keys, softmax statistics and their merge, warp reductions, and the bounded
// grid/group barrier used by the persistent kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <math.h>

#include "spec.h"

namespace spec {

constexpr int kThreads = 256;               // threads per CTA for the streaming kernels
constexpr int kWarps = kThreads / 32;
constexpr float kNearTie = 1e-6f;           // relative window of a near-tie draw
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // bounded waits: 1 s

// ---------------------------------------------------------------------------------
// Element loads.  bf16 is carried as raw uint16 words; widening to float32 is exact.
// ---------------------------------------------------------------------------------
typedef uint16_t bf16_t;

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(bf16_t x) { return __uint_as_float(((uint32_t)x) << 16); }

template <typename T> struct VecTraits;
template <> struct VecTraits<float> { static constexpr int N = 4; };
template <> struct VecTraits<bf16_t> { static constexpr int N = 8; };

// One 16-byte read-only streaming load of N elements, widened to float.
__device__ __forceinline__ void load_vec(const float* p, float (&o)[4]) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
}
__device__ __forceinline__ void load_vec(const bf16_t* p, float (&o)[8]) {
    uint32_t a, b, c, d;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "l"(p));
    o[0] = __uint_as_float(a << 16); o[1] = __uint_as_float(a & 0xffff0000u);
    o[2] = __uint_as_float(b << 16); o[3] = __uint_as_float(b & 0xffff0000u);
    o[4] = __uint_as_float(c << 16); o[5] = __uint_as_float(c & 0xffff0000u);
    o[6] = __uint_as_float(d << 16); o[7] = __uint_as_float(d & 0xffff0000u);
}

__device__ __forceinline__ float load_one(const float* p) { return __ldg(p); }
__device__ __forceinline__ float load_one(const bf16_t* p) {
    return to_float((bf16_t)__ldg(reinterpret_cast<const unsigned short*>(p)));
}

// A valid logit is finite or -inf; NaN and +inf are not.
__device__ __forceinline__ bool bad_logit(float x) { return !(x < INFINITY); }

// Larger of two floats, NaN when either is NaN.
__device__ __forceinline__ float f_max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
// Maximum of the entries of one 16-byte word of logits (8 bf16 or 4 float32), NaN
// when any entry is NaN: one reduction both finds the maximum and flags a NaN, and a
// +inf entry shows as a maximum of +inf.
template <int ELT_BYTES>
__device__ __forceinline__ float u4_max_nan(const uint4& w) {
    if (ELT_BYTES == 2) {
        uint32_t a, b, c;
        asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(w.x), "r"(w.y));
        asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(b) : "r"(w.z), "r"(w.w));
        asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(c) : "r"(a), "r"(b));
        return f_max_nan(__uint_as_float(c << 16), __uint_as_float(c & 0xffff0000u));
    }
    return f_max_nan(f_max_nan(__uint_as_float(w.x), __uint_as_float(w.y)),
                     f_max_nan(__uint_as_float(w.z), __uint_as_float(w.w)));
}

// ---------------------------------------------------------------------------------
// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, SC'11, section 3.2, table 2).
// ---------------------------------------------------------------------------------
// First output word for key (seed, 0) and counter (b, j, stream, 0).
__device__ __forceinline__ uint64_t philox_word0(uint64_t seed, uint64_t b, uint64_t j, uint64_t stream) {
    const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
    uint64_t c0 = b, c1 = j, c2 = stream, c3 = 0;
    uint64_t k0 = seed, k1 = 0;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) { k0 += W0; k1 += W1; }
        const uint64_t hi0 = __umul64hi(M0, c0), lo0 = M0 * c0;
        const uint64_t hi1 = __umul64hi(M1, c2), lo1 = M1 * c2;
        const uint64_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    }
    return c0;
}
__device__ __forceinline__ float philox_uniform(uint64_t seed, uint64_t b, uint64_t j, uint64_t stream) {
    return (float)(philox_word0(seed, b, j, stream) >> 40) * 0x1p-24f;   // 24-bit uniform, exact in float32
}

// ---------------------------------------------------------------------------------
// Argmax keys: a 64-bit integer whose maximum is the largest value and, among equal
// values, the lowest index.  -0.0 is folded into +0.0 so the two compare equal.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t float_order(float f) {
    if (f == 0.0f) f = 0.0f;
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float order_float(uint32_t o) {
    const uint32_t b = (o & 0x80000000u) ? (o & 0x7fffffffu) : ~o;
    return __uint_as_float(b);
}
__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx) {
    return ((unsigned long long)float_order(v) << 32) | (unsigned long long)(~idx);
}
__device__ __forceinline__ uint32_t key_index(unsigned long long k) { return ~(uint32_t)(k & 0xffffffffu); }
__device__ __forceinline__ float key_value(unsigned long long k) { return order_float((uint32_t)(k >> 32)); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float y = __shfl_xor_sync(0xffffffffu, x, o);
        x = ((threadIdx.x & o) == 0) ? x + y : y + x;
    }
    return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ int warp_or(int x) { return __any_sync(0xffffffffu, x) ? 1 : 0; }

// Inclusive prefix sum over the lanes of a warp (fixed association order).
__device__ __forceinline__ float warp_inclusive_scan(float x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x = y + x;
    }
    return x;
}

// ---------------------------------------------------------------------------------
// Base-2 softmax statistics for the streaming loops.  A row's weights are
// w_v = 2^(x_v*log2e - m2) for a reference m2 (in practice fl(max*log2e)); the
// product x*log2e is formed exactly inside one FFMA, so each weight costs one FFMA and
// one MUFU ex2.  Merging two partials rescales by 2^(m2_a - m2) with the same m2_a
// the partial was summed against, so the rounding of m2_a cancels; only per-operation
// rounding remains.  Normalised quantities (p_v = w_v / sum w) equal exp(x_v - m)/Z
// up to float32 rounding and the 1.3e-8 relative error of log2e in float32.
// ---------------------------------------------------------------------------------
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Pairs of floats held as one 64-bit register pair, and this architecture's float32x2
// arithmetic: one instruction rounds both halves exactly as the scalar instruction would.
typedef unsigned long long f2x;
__device__ __forceinline__ f2x f2_pack(float lo, float hi) {
    f2x r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 f2_unpack(f2x v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ f2x f2_fma(f2x a, f2x b, f2x c) {
    f2x r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ f2x f2_add(f2x a, f2x b) {
    f2x r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2x f2_mul(f2x a, f2x b) {
    f2x r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
// The two bf16 values of a 32-bit word, widened (exactly) into a pair.
__device__ __forceinline__ f2x bf2_widen(uint32_t w) {
    return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// (2^x, 2^y) of a pair
__device__ __forceinline__ f2x f2_ex2(f2x v) {
    const float2 a = f2_unpack(v);
    return f2_pack(ex2(a.x), ex2(a.y));
}

// 2^(x*log2e - m2)
__device__ __forceinline__ float wexp(float x, float m2) { return ex2(fmaf(x, kLog2e, -m2)); }

struct Stat2 { float m2; float s; };   // s = sum 2^(x*log2e - m2); empty: (-inf, 0)

// ---------------------------------------------------------------------------------
// Memory-model helpers and the bounded barrier.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void red_add_release(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// Grid barrier on a monotonic arrival counter (slot[0]): barrier k of a launch is
// complete once the counter reaches k * nblocks.  An arrival is a fire-and-forget
// release reduction, so a barrier costs one poll round trip after the last arrival,
// and nothing is read at kernel entry.  The counter must be 0 at launch: every CTA
// calls grid_barrier_exit after its last barrier, and the last one to do so resets
// the counter and the exit count (slot[32]); by then no CTA is still waiting.  After
// a timeout the counters are left as they are (the workspace must be re-zeroed).
struct GridBarrier {
    unsigned* count;
    unsigned* exits;
    unsigned target;
};
__device__ __forceinline__ GridBarrier grid_barrier_init(unsigned* slot) {
    return GridBarrier{slot, slot + 32, 0u};
}
__device__ __forceinline__ bool grid_barrier(GridBarrier& gb, unsigned nblocks, unsigned* status) {
    __shared__ int s_ok;
    __syncthreads();
    gb.target += nblocks;
    if (threadIdx.x == 0) {
        red_add_release(gb.count, 1u);
        bool ok = true;
        const unsigned long long t0 = global_timer_ns();
        unsigned spins = 0;
        while ((int)(ld_acquire(gb.count) - gb.target) < 0) {
            if (((++spins) & 255u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) {
                atomicOr(status, SPEC_DEV_TIMEOUT);
                ok = false;
                break;
            }
        }
        s_ok = ok ? 1 : 0;
    }
    __syncthreads();
    return s_ok != 0;
}
// Returns true in thread 0 of the last CTA to leave.
__device__ __forceinline__ bool grid_barrier_exit(const GridBarrier& gb, unsigned nblocks) {
    if (threadIdx.x == 0 && atom_add_acq_rel(gb.exits, 1u) == nblocks - 1u) {
        atomicExch(gb.count, 0u);
        atomicExch(gb.exits, 0u);
        return true;
    }
    return false;
}

__device__ __forceinline__ int ld_relaxed_i32(const int32_t* p) {
    int v;
    asm volatile("ld.relaxed.gpu.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// "Last CTA done" test: every CTA calls it once after its writes; exactly one CTA
// (the last) gets true, after which it sees every other CTA's writes.  The counter
// is left for that CTA to reset.  No waiting is involved.
__device__ __forceinline__ bool last_block_done(unsigned* counter, unsigned expected) {
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(counter, 1u);
        s_last = (prev == expected - 1u) ? 1 : 0;
        if (s_last) __threadfence();
    }
    __syncthreads();
    return s_last != 0;
}

// ---------------------------------------------------------------------------------
// mbarrier + TMA bulk copies (global -> shared), with a bounded wait.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive1(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// Bulk prefetch of `bytes` (multiple of 16, 16-byte aligned) from global memory into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(src), "r"(bytes) : "memory");
}
// 1-D bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
// An L2 policy that evicts first the lines it brings in, for operands streamed once: after
// a large write has left L2 full of dirty lines, the stream then takes the place of its
// own earlier lines instead of forcing those lines out (a write-back each).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// bulk_g2s with an L2 cache policy
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, unsigned bytes, uint64_t* bar, uint64_t pol) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
                 :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// Wait for phase `parity` of the barrier to complete, for at most `limit_ns`.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, unsigned* status,
                                          unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, SPEC_DEV_TIMEOUT);
            return false;
        }
    }
    return true;
}

// ---------------------------------------------------------------------------------
// Programmatic dependent launch.  A kernel that produces what the next one reads last
// lets the next one start early; the dependent waits only where it needs the data.
// Both are no-ops for launches without the programmatic-serialization attribute.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Workspace header (32 KiB at the start of every workspace).
struct WsHeader {
    unsigned status;             // SPEC_DEV_* flags, sticky
    unsigned pad0[31];
    unsigned done[32];           // last-CTA counters of single-kernel phases
    unsigned barrier[64][64];    // barrier slots: [i][0] count, [i][32] generation or exit count
};
static_assert(sizeof(WsHeader) <= 32768, "workspace header exceeds 32 KiB");
constexpr size_t kWsHeaderBytes = 32768;

}  // namespace spec
