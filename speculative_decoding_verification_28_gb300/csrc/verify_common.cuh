// verify_common.cuh -- work decomposition shared by the greedy and the
// stochastic verification kernels.
//
// One CTA handles one unit (sequence b, row j, vocabulary chunk c).  Units are
// numbered row-major over j first: all row-0 units of every sequence, then all
// row-1 units, ...  Verification only needs rows up to the first stop of a
// sequence (first rejection, EOS, budget, or the bonus row): "remaining
// proposals were predicted under the wrong prefix; discard them and the later
// verification rows" ("Chapter 10 Speculative Decoding (Code Walkthrough)",
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
    u.c = bid % a.C;
    const int jb = bid / a.C;
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
