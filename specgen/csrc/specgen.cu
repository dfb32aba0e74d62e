// specgen.cu -- synthetic KV contents on the GPU (input generation only).
//
// f(seq, tok, pos, l, c, h, d) = ((splitmix64(splitmix64(key1) ^ key2) >> 56)
// - 128) / 128, key1 = seq << 36 | tok << 16 | pos, key2 = l << 20 | c << 19 |
// h << 10 | d, with Vigna's splitmix64 output function -- the same published
// definition as specgen/np_gen.py, restated here for the device.
//
// kv layout [L, 2, B, H, S, D]; storage: 0 = fp32, 1 = bf16, 2 = fp16.  The
// values are multiples of 1/128 in [-1, 1), exact in all three types.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t splitmix64(uint64_t x)
{
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t row_hash(uint32_t seq, uint32_t tok, uint32_t pos)
{
    return splitmix64(((uint64_t)seq << 36) | ((uint64_t)tok << 16) | (uint64_t)pos);
}

__device__ __forceinline__ float kv_value(uint64_t h1, uint32_t l, uint32_t c, uint32_t h, uint32_t d)
{
    const uint64_t key2 = ((uint64_t)l << 20) | ((uint64_t)c << 19) | ((uint64_t)h << 10) | d;
    const int top = (int)(splitmix64(h1 ^ key2) >> 56);
    return (float)(top - 128) / 128.0f;
}

__device__ __forceinline__ void store(void *kv, int elt, size_t i, float v)
{
    if (elt == 0)
        reinterpret_cast<float *>(kv)[i] = v;
    else if (elt == 1)
        reinterpret_cast<__nv_bfloat16 *>(kv)[i] = __float2bfloat16(v);
    else
        reinterpret_cast<__half *>(kv)[i] = __float2half(v);
}

__device__ __forceinline__ float load(const void *kv, int elt, size_t i)
{
    if (elt == 0)
        return reinterpret_cast<const float *>(kv)[i];
    if (elt == 1)
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(kv)[i]);
    return __half2float(reinterpret_cast<const __half *>(kv)[i]);
}

struct Shape {
    int L, B, H, S, D;
};

// one warp per (l, c, b, h, s) row
__global__ void fill_kernel(void *kv, int elt, Shape sh, const int32_t *tokens, const int32_t *pad,
                            const int32_t *nvalid, int junk)
{
    const long long rows = (long long)sh.L * 2 * sh.B * sh.H * sh.S;
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        long long x = r;
        const int s = (int)(x % sh.S);
        x /= sh.S;
        const int h = (int)(x % sh.H);
        x /= sh.H;
        const int b = (int)(x % sh.B);
        x /= sh.B;
        const int c = (int)(x % 2);
        const int l = (int)(x / 2);
        const int p = s - pad[b];
        uint64_t h1;
        if (p >= 0 && p < nvalid[b])
            h1 = row_hash((uint32_t)b, (uint32_t)tokens[(size_t)b * sh.S + p], (uint32_t)p);
        else if (junk)
            h1 = row_hash((uint32_t)b, 999000u + (uint32_t)s, 0u);
        else
            continue;
        const size_t base = (size_t)r * sh.D;
        for (int d = lane; d < sh.D; d += 32)
            store(kv, elt, base + d, kv_value(h1, l, c, h, d));
    }
}

// the synthetic forward's KV write for the k+1 query slots W-1 .. W+k1-2
// (W from the host, or read on the device from W_dev when it is given)
__global__ void write_query_kernel(void *kv, int elt, Shape sh, const int32_t *qtok, int k1, const int32_t *pos,
                                   int W_host, const int32_t *W_dev)
{
    const int W = W_dev ? *W_dev : W_host;
    const long long rows = (long long)sh.L * 2 * sh.B * sh.H * k1;
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        long long x = r;
        const int j = (int)(x % k1);
        x /= k1;
        const int h = (int)(x % sh.H);
        x /= sh.H;
        const int b = (int)(x % sh.B);
        x /= sh.B;
        const int c = (int)(x % 2);
        const int l = (int)(x / 2);
        const int slot = W - 1 + j;
        if (slot < 0 || slot >= sh.S)
            continue;
        const uint64_t h1 = row_hash((uint32_t)b, (uint32_t)qtok[(size_t)b * k1 + j],
                                     (uint32_t)pos[(size_t)b * sh.S + slot]);
        const size_t base = ((((size_t)(l * 2 + c) * sh.B + b) * sh.H + h) * sh.S + slot) * sh.D;
        for (int d = lane; d < sh.D; d += 32)
            store(kv, elt, base + d, kv_value(h1, l, c, h, d));
    }
}

// the forward's KV write on a ragged pool [L, 2, N, H, S, D]: batch row b is
// pool sequence seq[b] and its k1 query slots start at base[b]; in a pool the
// position of a slot is its index
__global__ void write_query_pool_kernel(void *kv, int elt, Shape sh, const int32_t *qtok, int k1, int B,
                                        const int32_t *seq, const int32_t *base)
{
    const long long rows = (long long)sh.L * 2 * B * sh.H * k1;
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        long long x = r;
        const int j = (int)(x % k1);
        x /= k1;
        const int h = (int)(x % sh.H);
        x /= sh.H;
        const int b = (int)(x % B);
        x /= B;
        const int c = (int)(x % 2);
        const int l = (int)(x / 2);
        const int n = seq[b], slot = base[b] + j;
        if (n < 0 || n >= sh.B || slot < 0 || slot >= sh.S)
            continue;
        const uint64_t h1 = row_hash((uint32_t)n, (uint32_t)qtok[(size_t)b * k1 + j], (uint32_t)slot);
        const size_t at = ((((size_t)(l * 2 + c) * sh.B + n) * sh.H + h) * sh.S + slot) * sh.D;
        for (int d = lane; d < sh.D; d += 32)
            store(kv, elt, at + d, kv_value(h1, l, c, h, d));
    }
}

// invariant I2 over the whole cache: slot pad'_b + p holds f(b, tok_p, p) for
// every p < len'_b - 1; counts the elements that differ
__global__ void check_kernel(const void *kv, int elt, Shape sh, const int32_t *tokens, const int32_t *pad_new,
                             const int32_t *len_new, unsigned long long *bad)
{
    const long long rows = (long long)sh.L * 2 * sh.B * sh.H * sh.S;
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    unsigned long long miss = 0;
    for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        long long x = r;
        const int s = (int)(x % sh.S);
        x /= sh.S;
        const int h = (int)(x % sh.H);
        x /= sh.H;
        const int b = (int)(x % sh.B);
        x /= sh.B;
        const int c = (int)(x % 2);
        const int l = (int)(x / 2);
        const int p = s - pad_new[b];
        if (p < 0 || p >= len_new[b] - 1)
            continue;
        const uint64_t h1 = row_hash((uint32_t)b, (uint32_t)tokens[(size_t)b * sh.S + p], (uint32_t)p);
        const size_t base = (size_t)r * sh.D;
        for (int d = lane; d < sh.D; d += 32)
            miss += load(kv, elt, base + d) != kv_value(h1, l, c, h, d);
    }
    for (int m = 16; m > 0; m >>= 1)
        miss += __shfl_xor_sync(0xFFFFFFFFu, miss, m);
    if (lane == 0 && miss)
        atomicAdd(bad, miss);
}

unsigned grid_for(long long rows)
{
    long long blocks = (rows + 7) / 8;  // 8 warps per block
    if (blocks > 152LL * 64)
        blocks = 152LL * 64;
    return (unsigned)(blocks > 0 ? blocks : 1);
}

}  // namespace

extern "C" {

int specgen_kv_fill(void *kv, int elt, int L, int B, int H, int S, int D, const int32_t *tokens,
                    const int32_t *pad, const int32_t *nvalid, int junk, void *stream)
{
    Shape sh{L, B, H, S, D};
    fill_kernel<<<grid_for((long long)L * 2 * B * H * S), 256, 0, (cudaStream_t)stream>>>(kv, elt, sh, tokens, pad,
                                                                                         nvalid, junk);
    return (int)cudaGetLastError();
}

int specgen_kv_write_query(void *kv, int elt, int L, int B, int H, int S, int D, const int32_t *qtok, int k1,
                           const int32_t *pos, int W, void *stream)
{
    Shape sh{L, B, H, S, D};
    write_query_kernel<<<grid_for((long long)L * 2 * B * H * k1), 256, 0, (cudaStream_t)stream>>>(kv, elt, sh, qtok,
                                                                                                 k1, pos, W, nullptr);
    return (int)cudaGetLastError();
}

// as specgen_kv_write_query, with the width read on the device (no host
// round trip between a round and the next forward)
int specgen_kv_write_query_dev(void *kv, int elt, int L, int B, int H, int S, int D, const int32_t *qtok, int k1,
                               const int32_t *pos, const int32_t *W_dev, void *stream)
{
    Shape sh{L, B, H, S, D};
    write_query_kernel<<<grid_for((long long)L * 2 * B * H * k1), 256, 0, (cudaStream_t)stream>>>(kv, elt, sh, qtok,
                                                                                                 k1, pos, 0, W_dev);
    return (int)cudaGetLastError();
}

int specgen_kv_write_query_pool(void *kv, int elt, int L, int N, int H, int S, int D, const int32_t *qtok, int k1,
                                int B, const int32_t *seq, const int32_t *base, void *stream)
{
    Shape sh{L, N, H, S, D};
    write_query_pool_kernel<<<grid_for((long long)L * 2 * B * H * k1), 256, 0, (cudaStream_t)stream>>>(
        kv, elt, sh, qtok, k1, B, seq, base);
    return (int)cudaGetLastError();
}

int specgen_kv_check(const void *kv, int elt, int L, int B, int H, int S, int D, const int32_t *tokens,
                     const int32_t *pad_new, const int32_t *len_new, unsigned long long *bad, void *stream)
{
    Shape sh{L, B, H, S, D};
    check_kernel<<<grid_for((long long)L * 2 * B * H * S), 256, 0, (cudaStream_t)stream>>>(kv, elt, sh, tokens,
                                                                                          pad_new, len_new, bad);
    return (int)cudaGetLastError();
}

}  // extern "C"
