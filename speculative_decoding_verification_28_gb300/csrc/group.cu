// group.cu -- same-length grouping over a pool of ragged sequences (EXSPEC,
// "Correctness Forensics for Batch Speculative Decoding", §3.2: keep
// sequences ragged and batch sequences of identical current length so that
// realignment is bypassed).  The pages give no algorithm; the policy is this
// library's: L* = most frequent active length (ties to the smaller), members of
// length L* by ascending index (at most B), then other active sequences by
// ascending (|len - L*|, index); -1 beyond the active count.
// One CTA: bitonic sort of (length, index) keys, run lengths by binary
// search, best run by a max-reduction, second sort for the fill.  Pools of
// up to 1024 sequences keep one key per thread in a register: compare-exchange
// stages with strides below 32 go through warp shuffles, the wider ones
// through shared memory with one barrier each (15 of the network's 55
// stages); larger pools sort in shared memory.
#include "spec_common.cuh"
#include "spec_launch.h"

namespace spec {

constexpr int kGroupThreads = 1024;

__device__ void bitonic_sort_asc(uint64_t *k, int P)
{
    for (int size = 2; size <= P; size <<= 1)
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < P; i += kGroupThreads) {
                const int j = i ^ stride;
                if (j > i) {
                    const bool asc = (i & size) == 0;
                    const uint64_t x = k[i], y = k[j];
                    if (asc ? (x > y) : (x < y)) {
                        k[i] = y;
                        k[j] = x;
                    }
                }
            }
            __syncthreads();
        }
}

__global__ void __launch_bounds__(kGroupThreads)
    group_kernel(int N, const int32_t *len, const uint8_t *active, int B, int32_t *out_idx,
                 int32_t *out_count_equal, int32_t *out_group_len)
{
    __shared__ uint64_t key[SPEC_MAX_GROUP_N];
    __shared__ unsigned long long s_best;
    __shared__ int s_nact;
    const uint64_t NONE = ~0ull;
    int P = 1;
    while (P < N)
        P <<= 1;
    if (threadIdx.x == 0) {
        s_best = 0;
        s_nact = 0;
    }
    // (length ^ sign bit, index): unsigned order of the key = signed order of length
    for (int i = threadIdx.x; i < P; i += kGroupThreads) {
        uint64_t kk = NONE;
        if (i < N && (!active || active[i]))
            kk = ((uint64_t)((uint32_t)len[i] ^ 0x80000000u) << 32) | (uint32_t)i;
        key[i] = kk;
    }
    __syncthreads();
    bitonic_sort_asc(key, P);
    // active count = first NONE position
    for (int i = threadIdx.x; i < P; i += kGroupThreads)
        if (key[i] != NONE && (i + 1 == P || key[i + 1] == NONE))
            s_nact = i + 1;
    __syncthreads();
    const int nact = s_nact;
    // each run start: its length by binary search for the first larger length
    for (int i = threadIdx.x; i < nact; i += kGroupThreads) {
        const uint32_t li = (uint32_t)(key[i] >> 32);
        if (i > 0 && (uint32_t)(key[i - 1] >> 32) == li)
            continue;
        int lo = i, hi = nact;  // first index with length > li
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if ((uint32_t)(key[mid] >> 32) > li)
                hi = mid;
            else
                lo = mid + 1;
        }
        const unsigned long long cand =
            ((unsigned long long)(lo - i) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)i);
        atomicMax(&s_best, cand);
    }
    __syncthreads();
    const unsigned long long best = s_best;
    const int start = nact > 0 ? (int)(0xFFFFFFFFu - (uint32_t)best) : 0;
    const int cnt = nact > 0 ? (int)(best >> 32) : 0;
    const int ce = cnt < B ? cnt : B;
    const uint32_t lstar_u = nact > 0 ? (uint32_t)(key[start] >> 32) : 0u;
    const int lstar = (int)(lstar_u ^ 0x80000000u);
    for (int s = threadIdx.x; s < ce; s += kGroupThreads)
        out_idx[s] = (int)(uint32_t)key[start + s];
    __syncthreads();
    // fill: other active sequences by (|len - L*|, index); new keys are built
    // in registers, then written after every thread has read the old ones
    constexpr int kPer = SPEC_MAX_GROUP_N / kGroupThreads;
    uint64_t nk[kPer];
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
        const int i = threadIdx.x + r * kGroupThreads;
        uint64_t kk = NONE;
        if (i < nact && !(i >= start && i < start + ce)) {
            const int li = (int)((uint32_t)(key[i] >> 32) ^ 0x80000000u);
            const long long dist = (long long)li - lstar;
            const uint32_t ad = (uint32_t)(dist < 0 ? -dist : dist);
            kk = ((uint64_t)ad << 32) | (uint32_t)key[i];
        }
        nk[r] = kk;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
        const int i = threadIdx.x + r * kGroupThreads;
        if (i < P)
            key[i] = nk[r];
    }
    __syncthreads();
    bitonic_sort_asc(key, P);
    for (int s = ce + threadIdx.x; s < B; s += kGroupThreads) {
        const int r = s - ce;
        out_idx[s] = (r < P && key[r] != NONE) ? (int)(uint32_t)key[r] : -1;
    }
    if (threadIdx.x == 0) {
        *out_count_equal = ce;
        *out_group_len = nact > 0 ? lstar : -1;
    }
}

// Bitonic network over the 1024 keys held one per thread (thread i ends with
// the i-th smallest).  buf: 2 x 1024 keys of shared memory, alternated so that
// one barrier per shared-memory stage suffices.
__device__ uint64_t bitonic_sort_reg(uint64_t x, uint64_t *buf)
{
    const int i = threadIdx.x;
    int flip = 0;
    for (int size = 2; size <= kGroupThreads; size <<= 1)
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            uint64_t y;
            if (stride >= 32) {
                uint64_t *b = buf + flip * kGroupThreads;
                b[i] = x;
                __syncthreads();
                y = b[i ^ stride];
                flip ^= 1;
            } else {
                y = shfl_xor_u64(x, stride);
            }
            const bool asc = (i & size) == 0, lower = (i & stride) == 0;
            x = (lower == asc) ? (x < y ? x : y) : (x > y ? x : y);
        }
    return x;
}

// N <= kGroupThreads: the same policy with one key per thread
__global__ void __launch_bounds__(kGroupThreads)
    group_kernel_reg(int N, const int32_t *len, const uint8_t *active, int B, int32_t *out_idx,
                     int32_t *out_count_equal, int32_t *out_group_len)
{
    __shared__ uint64_t buf[2 * kGroupThreads];
    __shared__ unsigned long long s_best;
    const uint64_t NONE = ~0ull;
    const int i = threadIdx.x;
    if (i == 0)
        s_best = 0;
    uint64_t x = NONE;
    if (i < N && (!active || active[i]))
        x = ((uint64_t)((uint32_t)len[i] ^ 0x80000000u) << 32) | (uint32_t)i;
    x = bitonic_sort_reg(x, buf);
    const int nact = __syncthreads_count(x != NONE);  // the sorted keys: the active ones first
    uint64_t *key = buf;  // the sorted keys, for neighbours and the binary search
    key[i] = x;
    __syncthreads();
    if (i < nact) {
        const uint32_t li = (uint32_t)(x >> 32);
        if (i == 0 || (uint32_t)(key[i - 1] >> 32) != li) {  // a run starts here
            int lo = i, hi = nact;  // first position with a larger length
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if ((uint32_t)(key[mid] >> 32) > li)
                    hi = mid;
                else
                    lo = mid + 1;
            }
            atomicMax(&s_best, ((unsigned long long)(lo - i) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)i));
        }
    }
    __syncthreads();
    const unsigned long long best = s_best;
    const int start = nact > 0 ? (int)(0xFFFFFFFFu - (uint32_t)best) : 0;
    const int cnt = nact > 0 ? (int)(best >> 32) : 0;
    const int ce = cnt < B ? cnt : B;
    const int lstar = nact > 0 ? (int)((uint32_t)(key[start] >> 32) ^ 0x80000000u) : 0;
    if (i < ce)
        out_idx[i] = (int)(uint32_t)key[start + i];
    // fill: the other active sequences by (|len - L*|, index)
    uint64_t x2 = NONE;
    if (i < nact && !(i >= start && i < start + ce)) {
        const long long dist = (long long)(int)((uint32_t)(x >> 32) ^ 0x80000000u) - lstar;
        x2 = ((uint64_t)(uint32_t)(dist < 0 ? -dist : dist) << 32) | (uint32_t)x;
    }
    __syncthreads();  // every read of key[] (buf) is done before the second sort reuses it
    x2 = bitonic_sort_reg(x2, buf);
    if (ce + i < B)
        out_idx[ce + i] = x2 != NONE ? (int)(uint32_t)x2 : -1;
    for (int s = kGroupThreads + ce + i; s < B; s += kGroupThreads)  // B beyond the pool: -1
        out_idx[s] = -1;
    if (i == 0) {
        *out_count_equal = ce;
        *out_group_len = nact > 0 ? lstar : -1;
    }
}

cudaError_t launch_group(int N, const int32_t *len, const uint8_t *active, int B, int32_t *out_idx,
                         int32_t *out_count_equal, int32_t *out_group_len, cudaStream_t st)
{
    if (N <= kGroupThreads)
        group_kernel_reg<<<1, kGroupThreads, 0, st>>>(N, len, active, B, out_idx, out_count_equal, out_group_len);
    else
        group_kernel<<<1, kGroupThreads, 0, st>>>(N, len, active, B, out_idx, out_count_equal, out_group_len);
    return cudaGetLastError();
}

}  // namespace spec
