// verify_common.cuh -- work decomposition shared by the greedy and the
// stochastic verification kernels.
//
// One CTA handles one unit (sequence b, row j, vocabulary chunk c).  Units are
// numbered row-major over j first: all row-0 units of every sequence, then all
// row-1 units, ...  Verification only needs rows up to the first stop of a
// sequence (first rejection, EOS, budget, or the bonus row): the proposals
// after a rejection were drafted after a token that is not kept, so their
// rows decide nothing ("Chapter 10 Speculative Decoding (Code Walkthrough)",
// §4.2).  So each unit first looks at the earliest stop row already known for
// its sequence and skips its reads when that row lies before it.  The known
// stop can only move earlier, and a row is evaluated only if no earlier stop
// was known when its finaliser ran, which guarantees that every row up to the
// true first stop was fully read.  Nothing waits on anything: a unit whose
// earlier rows are still in flight simply reads its chunk.
//
// Completion is counted: the last CTA of a row (atomic counter) combines the
// row's chunk partials, and the last row of a sequence runs the first-stop
// scan with one warp ballot.  Every counter is returned to zero by the CTA
// that consumed it, so the workspace is clean after every call.
#pragma once

#include "spec_common.cuh"
#include "spec_launch.h"

namespace spec {

struct Unit {
    int b, j, c, row;  // row = b * (k + 1) + j
    int kb;            // proposals of sequence b
    int rem;           // output budget of sequence b
    bool needed;       // row j can matter at all (j <= k_b and j < budget)
};

__device__ __forceinline__ Unit decode_unit(const VerifyArgs &a)
{
    Unit u;
    const int bid = blockIdx.x;
    const int jb = bid / a.C;
    u.c = bid - jb * a.C;
    u.b = jb % a.B;
    u.j = jb / a.B;
    u.row = u.b * (a.k + 1) + u.j;
    int kb = a.draft_len ? a.draft_len[u.b] : a.k;
    u.kb = kb < 0 ? 0 : (kb > a.k ? a.k : kb);
    u.rem = a.remaining ? a.remaining[u.b] : 0x7FFFFFFF;
    u.needed = (u.j <= u.kb) && (u.j < u.rem);
    return u;
}

// true when a stop earlier than row j is already recorded for sequence b
__device__ __forceinline__ bool stopped_before(const int *stop_enc, int b, int j)
{
    const int enc = ld_relaxed(stop_enc + b);
    return enc > 0 && (kStopBase - enc) < j;
}

// 2^x by the SFU instruction ex2.approx.ftz.f32 (relative error about
// 2^-22; results below 2^-126 flush to zero, negligible in a softmax sum).
// e^x is computed as 2^(x log2 e) with the scale folded into one FFMA.
__device__ __forceinline__ float exp2_sfu(float x)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Maxima that propagate NaN (PTX max.NaN): a vector's maximum is NaN when
// any element is NaN, so one comparison per 16-byte vector finds both a new
// largest value and a NaN.
__device__ __forceinline__ float max_nan(float a, float b)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t max_nan_f16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.NaN.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// maximum (NaN-propagating) of the elements of one 16-byte vector, as fp32
template <typename T>
__device__ __forceinline__ float vec_max(const uint4 &u);
template <>
__device__ __forceinline__ float vec_max<float>(const uint4 &u)
{
    return max_nan(max_nan(__uint_as_float(u.x), __uint_as_float(u.y)),
                   max_nan(__uint_as_float(u.z), __uint_as_float(u.w)));
}
template <>
__device__ __forceinline__ float vec_max<__nv_bfloat16>(const uint4 &u)
{
    const uint32_t m = max_nan_bf16x2(max_nan_bf16x2(u.x, u.y), max_nan_bf16x2(u.z, u.w));
    return max_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}
template <>
__device__ __forceinline__ float vec_max<__half>(const uint4 &u)
{
    const uint32_t m = max_nan_f16x2(max_nan_f16x2(u.x, u.y), max_nan_f16x2(u.z, u.w));
    __half2 h;
    memcpy(&h, &m, 4);
    const float2 f = __half22float2(h);
    return max_nan(f.x, f.y);
}

// NaN-propagating element-wise maximum of two 16-byte vectors (32-bit words
// holding one fp32 or two bf16 / fp16 values)
template <typename T>
__device__ __forceinline__ uint32_t max_word(uint32_t a, uint32_t b);
template <>
__device__ __forceinline__ uint32_t max_word<float>(uint32_t a, uint32_t b)
{
    return __float_as_uint(max_nan(__uint_as_float(a), __uint_as_float(b)));
}
template <>
__device__ __forceinline__ uint32_t max_word<__nv_bfloat16>(uint32_t a, uint32_t b)
{
    return max_nan_bf16x2(a, b);
}
template <>
__device__ __forceinline__ uint32_t max_word<__half>(uint32_t a, uint32_t b)
{
    return max_nan_f16x2(a, b);
}
template <typename T>
__device__ __forceinline__ uint4 max_vec(const uint4 &a, const uint4 &b)
{
    return make_uint4(max_word<T>(a.x, b.x), max_word<T>(a.y, b.y), max_word<T>(a.z, b.z), max_word<T>(a.w, b.w));
}

constexpr float kLog2e = 1.4426950408889634f;  // log2(e): e^x = 2^(x log2 e)

// Per-warp re-check, between load batches, that the unit's row is still
// needed: once a stop before row j is recorded for the sequence, the row will
// never be evaluated (the record only moves earlier), so the warp can drop
// the rest of its chunk.  Lane 0 reads the word; the decision is warp-uniform.
// The read is split in two so that it can travel with a batch of loads:
// load() issues it (lane 0; the other lanes return 0), stopped() decides on
// its value one batch later, when it has long arrived.  A decision on a word
// read one batch earlier only drops a chunk later, never one that is needed.
struct StopProbe {
    const int *stop_enc;
    int b, j;
    __device__ __forceinline__ int load() const
    {
        return ((threadIdx.x & 31) == 0) ? ld_relaxed(stop_enc + b) : 0;
    }
    __device__ __forceinline__ bool stopped(int enc) const
    {
        const int e = __shfl_sync(0xFFFFFFFFu, enc, 0);
        return e > 0 && (kStopBase - e) < j;
    }
};

// Block-wide max of a u64 key for thread 0 only: warp shuffles, one
// shared-memory exchange, one barrier (the other threads' results are
// meaningless).
__device__ __forceinline__ uint64_t block_max_u64_to0(uint64_t key, uint64_t *s_red)
{
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        const uint64_t o = shfl_xor_u64(key, m);
        key = o > key ? o : key;
    }
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0)
        s_red[w] = key;
    __syncthreads();
    if (threadIdx.x < 32) {
        key = (l < (int)(blockDim.x >> 5)) ? s_red[l] : 0;
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) {
            const uint64_t o = shfl_xor_u64(key, m);
            key = o > key ? o : key;
        }
    }
    return key;
}

// Block-wide max of a u64 key (all threads get the result).
__device__ __forceinline__ uint64_t block_max_u64(uint64_t key, uint64_t *s_red)
{
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        const uint64_t o = shfl_xor_u64(key, m);
        key = o > key ? o : key;
    }
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0)
        s_red[w] = key;
    __syncthreads();
    key = (l < (int)(blockDim.x >> 5)) ? s_red[l] : 0;
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        const uint64_t o = shfl_xor_u64(key, m);
        key = o > key ? o : key;
    }
    __syncthreads();
    return key;
}

// Chunk [lo, hi) of a row as an aligned 16-byte vector body plus scalar head
// and tail.  `row` points at element 0 of the row.
template <typename T>
struct ChunkSplit {
    int head_end;  // elements lo .. head_end-1 are scalar
    int nvec;      // 16-byte vectors starting at head_end
    int tail_beg;  // elements tail_beg .. hi-1 are scalar
    __device__ ChunkSplit(const T *row, int lo, int hi)
    {
        constexpr int VEC = Storage<T>::kVec;
        const uintptr_t addr = reinterpret_cast<uintptr_t>(row + lo);
        int head = (int)(((16u - (uint32_t)(addr & 15u)) & 15u) / sizeof(T));
        if ((addr & (sizeof(T) - 1)) != 0)  // not even element-aligned: all scalar
            head = hi - lo;
        if (head > hi - lo)
            head = hi - lo;
        head_end = lo + head;
        nvec = (hi - head_end) / VEC;
        tail_beg = head_end + nvec * VEC;
    }
};

}  // namespace spec
