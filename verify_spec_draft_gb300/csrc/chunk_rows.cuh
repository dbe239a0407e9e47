// chunk_rows.cuh - per-thread chunks of logit rows for the streaming kernels.
//
// A work item is 8192 consecutive entries of one row, 32 contiguous entries per thread
// of a 256-thread CTA, loaded as 16-byte words (-inf past the row end) and reduced with
// a NaN-propagating maximum (packed bf16x2 for bf16 rows), so that one reduction gives
// the maximum and flags a NaN.
#pragma once

#include "spec_device.cuh"
#include "internal.h"

namespace spec {

constexpr int kEPT = kVerifyChunk / kThreads;   // 32 contiguous entries per thread
static_assert(kEPT == 32, "chunk layout");

// ----------------------------------------------------------------------------------
// Raw chunk loads: this thread's 32 entries as 16-byte words, -inf past the row end.
// ----------------------------------------------------------------------------------
template <typename T> struct Words { static constexpr int N = kEPT * (int)sizeof(T) / 16; };

__device__ __forceinline__ uint4 partial_words(const float* row, long e0, long V) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) w[e] = (e0 + e < V) ? __float_as_uint(__ldg(row + e0 + e)) : 0xff800000u;
    return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ uint4 partial_words(const bf16_t* row, long e0, long V) {
    uint32_t h[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        h[e] = (e0 + e < V) ? (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(row) + e0 + e) : 0xff80u;
    return make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
}

// Two 16-byte words at p (32-byte aligned) in one load: a whole 32-byte sector.  The
// rows read this way are read once, so their lines are the first L2 evicts
// (evict_first): the stream then replaces its own clean lines instead of writing back
// whatever dirty lines L2 held before it.  The policy asm has no side effects, so the
// compiler creates it once per loop, not per load.
__device__ __forceinline__ void ld_sector(const void* p, uint4& a, uint4& b) {
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    asm volatile("ld.global.nc.L2::cache_hint.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                 : "l"(p), "l"(pol));
}

template <typename T, int NW>
__device__ __forceinline__ void load_words(uint4 (&w)[NW], const T* row, long V, long base, bool vec_ok) {
    constexpr int EPV = 16 / (int)sizeof(T);
#pragma unroll
    for (int i = 0; i < Words<T>::N; ++i) {
        const long e0 = base + (long)i * EPV;
        if (vec_ok && e0 + EPV <= V) w[i] = __ldg(reinterpret_cast<const uint4*>(row + e0));
        else w[i] = partial_words(row, e0, V);
    }
}

// The same 32 entries per thread in the group-interleaved layout: lane l of warp w holds
// the 8-entry groups j * 32 + l (j < 4) of the warp's 1024-entry segment of chunk c,
// seg = c * 8192 + w * 1024; a group is one 16-byte word of bf16 or two of float32.
// Decoded entry k (decode_words) is entry seg + ((k / 8) * 32 + l) * 8 + k % 8 for either
// type, so rows of different types pair up entry by entry, and each load instruction
// of a warp reads 512 contiguous bytes (bf16; float32 rows take two instructions per
// 1 KB).
__device__ __forceinline__ long il_seg(int c) {
    return (long)c * kVerifyChunk + (long)(threadIdx.x >> 5) * 1024;
}
__device__ __forceinline__ long il_entry(long seg, int k) {
    return seg + (long)((k >> 3) * 32 + (int)(threadIdx.x & 31)) * 8 + (k & 7);
}
template <typename T, int NW>
__device__ __forceinline__ void load_words_il(uint4 (&w)[NW], const T* row, long V, long seg, bool vec_ok) {
    constexpr int EPV = 16 / (int)sizeof(T);
    constexpr int WPG = 8 / EPV;   // 16-byte words per 8-entry group
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int h = 0; h < WPG; ++h) {
            const long e0 = il_entry(seg, 8 * j) + h * EPV;
            if (vec_ok && e0 + EPV <= V) w[j * WPG + h] = __ldg(reinterpret_cast<const uint4*>(row + e0));
            else w[j * WPG + h] = partial_words(row, e0, V);
        }
    }
}

// The same for a segment that lies wholly in the row (vec_ok, seg + 1024 <= V).
template <typename T, int NW>
__device__ __forceinline__ void load_words_il_full(uint4 (&w)[NW], const T* row, long seg) {
    constexpr int EPV = 16 / (int)sizeof(T);
    constexpr int WPG = 8 / EPV;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int h = 0; h < WPG; ++h)
            w[j * WPG + h] = __ldg(reinterpret_cast<const uint4*>(row + il_entry(seg, 8 * j) + h * EPV));
}

// The sector-interleaved layout, for rows that start on 32 bytes: lane l of warp w holds
// the 32-byte groups j * 32 + l (j < NW / 2) of the warp's 1024-entry segment, 16 bf16
// or 8 float32 entries each, one load per group, so each load instruction of a warp
// reads 1 KB contiguous.  Decoded entry k is entry seg + ((k / E) * 32 + l) * E + k % E
// with E = 32 / sizeof(T); for float32 rows this is the group-interleaved layout.
template <typename T>
__device__ __forceinline__ long il32_entry(long seg, int k) {
    constexpr int E = 32 / (int)sizeof(T);
    return seg + (long)((k / E) * 32 + (int)(threadIdx.x & 31)) * E + (k % E);
}
template <typename T, int NW>
__device__ __forceinline__ void load_words_il32(uint4 (&w)[NW], const T* row, long V, long seg) {
    constexpr int E = 32 / (int)sizeof(T);
    const uint32_t ninf = sizeof(T) == 2 ? 0xff80ff80u : 0xff800000u;
#pragma unroll
    for (int j = 0; j < NW / 2; ++j) {
        const long e0 = il32_entry<T>(seg, j * E);
        if (e0 + E <= V) {
            ld_sector(row + e0, w[2 * j], w[2 * j + 1]);
        } else {   // the row's last group: whole words up to V (V is a multiple of E here)
            w[2 * j] = make_uint4(ninf, ninf, ninf, ninf);
            w[2 * j + 1] = w[2 * j];
        }
    }
}

// This warp's 1024-entry segment of a chunk staged in shared memory, in the
// group-interleaved layout: lane L holds groups j * 32 + L (j < 4), one 16-byte word each
// in bf16, two in float32, so that entry k of decode_words is the same vocabulary entry
// for either type.  -inf past the `nvalid` entries the chunk holds (checked per word).
template <typename T, int NW>
__device__ __forceinline__ void stage_groups(const uint8_t* stage, int warp, int lane, int nvalid, uint4 (&w)[NW]) {
    constexpr int WPG = (int)sizeof(T) / 2;   // 16-byte words per 8-entry group
    constexpr int EPV = 16 / (int)sizeof(T);
    const uint4* seg = reinterpret_cast<const uint4*>(stage) + (size_t)warp * (1024 / 8) * WPG;
    const uint32_t ninf = sizeof(T) == 2 ? 0xff80ff80u : 0xff800000u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int g = j * 32 + lane;
#pragma unroll
        for (int h = 0; h < WPG; ++h) {
            const bool in = warp * 1024 + g * 8 + h * EPV + EPV <= nvalid;
            w[j * WPG + h] = in ? seg[g * WPG + h] : make_uint4(ninf, ninf, ninf, ninf);
        }
    }
}

template <typename T, int NW>
__device__ __forceinline__ void decode_words(const uint4 (&w)[NW], float (&x)[kEPT]) {
    if (sizeof(T) == 2) {
#pragma unroll
        for (int i = 0; i < kEPT / 8; ++i) {
            const uint32_t a[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                x[8 * i + 2 * k] = __uint_as_float(a[k] << 16);
                x[8 * i + 2 * k + 1] = __uint_as_float(a[k] & 0xffff0000u);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < kEPT / 4; ++i) {
            x[4 * i] = __uint_as_float(w[i].x);
            x[4 * i + 1] = __uint_as_float(w[i].y);
            x[4 * i + 2] = __uint_as_float(w[i].z);
            x[4 * i + 3] = __uint_as_float(w[i].w);
        }
    }
}

__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// Max of this thread's 32 entries, NaN if any is NaN (bf16: packed pairs).
template <typename T, int NW>
__device__ __forceinline__ float chunk_max_nan(const uint4 (&w)[NW]) {
    if (sizeof(T) == 2) {
        uint32_t m = bmax2_nan(bmax2_nan(w[0].x, w[0].y), bmax2_nan(w[0].z, w[0].w));
#pragma unroll
        for (int i = 1; i < kEPT / 8; ++i)
            m = bmax2_nan(m, bmax2_nan(bmax2_nan(w[i].x, w[i].y), bmax2_nan(w[i].z, w[i].w)));
        return fmax_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    }
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kEPT / 4; ++i)
        m = fmax_nan(fmax_nan(m, fmax_nan(__uint_as_float(w[i].x), __uint_as_float(w[i].y))),
                     fmax_nan(__uint_as_float(w[i].z), __uint_as_float(w[i].w)));
    return m;
}
// The decode-order position (0..31) of the first of this thread's entries equal to m,
// or -1: the first 8-entry group whose maximum is m, then the first entry of that group
// (decode order is index order within a thread's group and across its groups, in both
// the contiguous and the group-interleaved layout).  For a lane whose entries hold the
// warp's maximum, this replaces decoding and comparing all 32 entries.
template <typename T, int NW>
__device__ __forceinline__ int first_equal(const uint4 (&w)[NW], float m) {
    constexpr int WPG = NW / 4;   // 16-byte words per 8-entry group: 1 (bf16) or 2 (float32)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float gm;
        if constexpr (sizeof(T) == 2) gm = u4_max_nan<2>(w[j]);
        else gm = f_max_nan(u4_max_nan<4>(w[WPG * j]), u4_max_nan<4>(w[WPG * j + 1]));
        if (gm == m) {
            float x[8];
            if constexpr (sizeof(T) == 2) {
                const uint32_t a[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    x[2 * k] = __uint_as_float(a[k] << 16);
                    x[2 * k + 1] = __uint_as_float(a[k] & 0xffff0000u);
                }
            } else {
                const uint4 lo = w[WPG * j], hi = w[WPG * j + 1];
                x[0] = __uint_as_float(lo.x); x[1] = __uint_as_float(lo.y);
                x[2] = __uint_as_float(lo.z); x[3] = __uint_as_float(lo.w);
                x[4] = __uint_as_float(hi.x); x[5] = __uint_as_float(hi.y);
                x[6] = __uint_as_float(hi.z); x[7] = __uint_as_float(hi.w);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (x[e] == m) return 8 * j + e;
        }
    }
    return -1;
}

__device__ __forceinline__ float warp_max_nan(float m) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmax_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
    return m;
}

}  // namespace spec
