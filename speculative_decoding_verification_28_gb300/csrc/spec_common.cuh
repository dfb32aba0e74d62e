// spec_common.cuh -- device helpers shared by the library's kernels:
// workspace layout, storage-type loads, the argmax ordering key, and inline
// PTX for mbarriers and 1-D bulk (TMA) copies on sm_103a.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "specverify.h"

namespace spec {

// ---------------------------------------------------------------------------
// sizes
// ---------------------------------------------------------------------------
constexpr int kThreads = 256;          // threads of the row-streaming kernels
constexpr int kMinChunk = 4096;        // smallest vocabulary chunk of a verify work unit
#ifndef SPEC_TARGET_UNITS
#define SPEC_TARGET_UNITS 2432
#endif
constexpr int kTargetUnits = SPEC_TARGET_UNITS;  // the best of a sweep over 608 .. 19456 units
constexpr int kDrawChunk = 8192;       // elements per CTA of the draw sums kernel (one 1024-element segment per warp)
constexpr int kMaxRows = SPEC_MAX_K + 1;
constexpr int kStopBase = 1024;        // stop row j is stored as kStopBase - j

// Split of each logits row into work units: about kTargetUnits units over the
// whole batch (four waves of four 256-thread CTAs per SM), each at least
// kMinChunk elements, lengths a multiple of 64 elements (16-byte aligned
// starts whenever the row start is).
struct Split {
    int C;    // chunks per row
    int len;  // elements per chunk (the last one may be shorter)
};
__host__ __device__ inline Split verify_split(int B, int k, int V)
{
    const long long rows = (long long)(B > 0 ? B : 1) * (k + 1);
    long long c = (kTargetUnits + rows - 1) / rows;
    long long cmax = V / kMinChunk;
    if (cmax < 1)
        cmax = 1;
    if (c > cmax)
        c = cmax;
    if (c < 1)
        c = 1;
    int len = (int)((V + c - 1) / c);
    len = (len + 63) & ~63;
    Split sp;
    sp.len = len;
    sp.C = (V + len - 1) / len;
    return sp;
}
__host__ __device__ inline int verify_chunks(int B, int k, int V) { return verify_split(B, k, V).C; }
__host__ __device__ inline int draw_chunks(int V) { return (V + kDrawChunk - 1) / kDrawChunk; }
constexpr int kDrawSeg = 1024;  // elements per draw segment: one warp's sums, the pick's final scan
__host__ __device__ inline int draw_segs(int V) { return (V + kDrawSeg - 1) / kDrawSeg; }

// ---------------------------------------------------------------------------
// workspace layout (byte offsets; every array 256-byte aligned)
//   [realign region: depends on B]
//   [counter region: depends on B; zero between calls]
//   [verify scratch: depends on B, k, V]
// ---------------------------------------------------------------------------
struct Layout {
    // realignment plan
    size_t order, delta, src_pad, run, seq_src, seq_dst, misc;
    // counters that every verify call leaves at zero
    size_t zero_begin, seq_cnt, stop_enc, row_cnt, zero_end;
    // verify scratch
    size_t row_tok, row_ms, row_flag, row_cut, part, draw_row, rpart, rtot;
    size_t total;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline Layout make_layout(int B, int k, int V)
{
    Layout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align256(o + bytes);
        return at;
    };
    const size_t b = (size_t)(B > 0 ? B : 0);
    const size_t rows = b * (size_t)(k + 1);
    const size_t C = (size_t)verify_chunks(B, k, V > 0 ? V : 1);
    L.order = take(b * 4);
    L.delta = take(b * 4);
    L.src_pad = take(b * 4);
    L.run = take(b * 4);
    L.seq_src = take(b * 4);
    L.seq_dst = take(b * 4);
    L.misc = take(64);
    L.zero_begin = o;
    L.seq_cnt = take(b * 4);
    L.stop_enc = take(b * 4);
    L.row_cnt = take(b * kMaxRows * 4);  // sized for the largest k
    L.zero_end = o;
    L.row_tok = take(rows * 4);
    L.row_ms = take(rows * 8);
    L.row_flag = take(rows * 4);
    L.row_cut = take(rows * 4);
    L.part = take(rows * C * 16);
    L.draw_row = take(b * 4);
    L.rpart = take(b * (size_t)draw_segs(V > 0 ? V : 1) * 8);  // two floats per draw segment
    L.rtot = take(b * 8);
    L.total = o;
    return L;
}

// misc slots of the realignment plan
enum { MISC_NMOVING = 0, MISC_WORK = 1, MISC_WIDTH = 2, MISC_ERR = 3, MISC_TOTAL_ROWS = 4 };

template <typename T>
__host__ __device__ inline T *ws_at(void *ws, size_t off)
{
    return reinterpret_cast<T *>(reinterpret_cast<char *>(ws) + off);
}

// ---------------------------------------------------------------------------
// storage types
// ---------------------------------------------------------------------------
template <typename T>
struct Storage;
template <>
struct Storage<float> {
    static constexpr int kVec = 4;  // elements per 16-byte vector
    __device__ static float at(const float *p, int64_t i) { return __ldg(p + i); }
    __device__ static void unpack(const uint4 &u, float (&f)[4])
    {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    }
};
template <>
struct Storage<__nv_bfloat16> {
    static constexpr int kVec = 8;
    __device__ static float at(const __nv_bfloat16 *p, int64_t i)
    {
        const unsigned short h = __ldg(reinterpret_cast<const unsigned short *>(p) + i);
        return __uint_as_float((uint32_t)h << 16);
    }
    __device__ static void unpack(const uint4 &u, float (&f)[8])
    {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
};
template <>
struct Storage<__half> {
    static constexpr int kVec = 8;
    __device__ static float at(const __half *p, int64_t i) { return __half2float(__ldg(p + i)); }
    __device__ static void unpack(const uint4 &u, float (&f)[8])
    {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h;
            memcpy(&h, &w[i], 4);
            const float2 t = __half22float2(h);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
};

// 16-byte streaming load that does not allocate in L1 (each logit is read once)
__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ int ld_relaxed(const int *p)
{
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Ordering key for "largest value, lowest index on ties, NaN above all":
// a larger key is a better candidate.  +0 and -0 compare equal.
__device__ __forceinline__ uint64_t argmax_key(float v, uint32_t idx)
{
    uint32_t ord;
    if (v != v) {
        ord = 0xFFFFFFFFu;
    } else {
        uint32_t b = (v == 0.0f) ? 0u : __float_as_uint(v);
        ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    }
    return ((uint64_t)ord << 32) | (uint64_t)(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ uint32_t key_index(uint64_t key) { return 0xFFFFFFFFu - (uint32_t)key; }

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int m)
{
    uint32_t lo = (uint32_t)v, hi = (uint32_t)(v >> 32);
    lo = __shfl_xor_sync(0xFFFFFFFFu, lo, m);
    hi = __shfl_xor_sync(0xFFFFFFFFu, hi, m);
    return ((uint64_t)hi << 32) | lo;
}

}  // namespace spec
