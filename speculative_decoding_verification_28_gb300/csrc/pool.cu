// pool.cu -- the ragged pool of EXSPEC ("Correctness Forensics for Batch
// Speculative Decoding", §3.2: keep sequences ragged, batch same-length
// sequences so realignment is bypassed, fall back to unpad-append-repad).
//
// Pool cache pool[L, 2, N, H, S, D]: sequence n left-aligned at slot 0, so its
// position IDs are its slot indices and a group of equal lengths is already
// rectangular.  Three operations:
//   commit : pool_len[idx[b]] += n_emit[b] after a round on a group -- the
//            rollback of rejected tokens in this variable-length layout ([CF]
//            §2) is that length update: their KV rows lie past the new length;
//   repad  : pool -> left-padded batch (the chosen sequences' rows
//            0 .. len - 2 at slot W - len, W the longest), for a fallback round;
//   unpad  : batch -> pool (rows pad .. pad + len - 2 back to slot 0) after it;
//            with n_emit the lengths are len + n_emit, straight from the batch a
//            round has extended (no realignment needed before unpadding).
// repad / unpad are out-of-place copies of every slab's run, done by the same
// bulk-copy engine as the realignment shift.  Roofline: HBM-bound,
// 2 * (len - 1) * D * elt bytes per slab.
#include "bulk_copy.cuh"
#include "spec_common.cuh"
#include "spec_launch.h"

namespace spec {

constexpr int kPoolPlanThreads = 1024;
constexpr int kMaxPool = 65536;  // duplicate check: one bit per pool sequence in shared memory

struct PoolPlan {
    int *order, *dst_off, *src_off, *rows, *seq_src, *seq_dst, *misc;
};
__device__ __forceinline__ PoolPlan pool_plan(void *ws, int B)
{
    const Layout lay = make_layout(B, 0, 1);
    return PoolPlan{ws_at<int>(ws, lay.order),   ws_at<int>(ws, lay.delta),   ws_at<int>(ws, lay.src_pad),
                    ws_at<int>(ws, lay.run),     ws_at<int>(ws, lay.seq_src), ws_at<int>(ws, lay.seq_dst),
                    ws_at<int>(ws, lay.misc)};
}

// marks idx[b] in a shared bitmap; false if out of range or already marked
__device__ __forceinline__ bool mark_index(uint32_t *bits, int n, int N)
{
    if (n < 0 || n >= N)
        return false;
    const uint32_t bit = 1u << (n & 31);
    return (atomicOr(bits + (n >> 5), bit) & bit) == 0;
}

__global__ void __launch_bounds__(kPoolPlanThreads) pool_plan_kernel(PoolArgs a)
{
    __shared__ uint32_t s_bits[kMaxPool / 32];
    __shared__ int s_bad, s_W;
    dep_release();  // the copy kernel may be scheduled; it waits for this grid
    const PoolPlan pp = pool_plan(a.ws, a.B);
    const int t = threadIdx.x, nt = blockDim.x;
    for (int i = t; i < (a.N + 31) / 32; i += nt)
        s_bits[i] = 0;
    if (t == 0) {
        s_bad = 0;
        s_W = 0;
    }
    __syncthreads();
    for (int b = t; b < a.B; b += nt) {
        const int n = a.idx[b];
        bool ok = mark_index(s_bits, n, a.N);
        if (ok && a.repad) {
            const int l = a.pool_len[n];
            ok = l >= 1 && l <= a.S;
            if (ok)
                atomicMax(&s_W, l);
        } else if (ok) {
            const int e = a.n_emit ? a.n_emit[b] : 0;
            const long long l = (long long)a.len[b] + e;
            const int p = a.pad[b];
            ok = e >= 0 && l >= 1 && p >= 0 && p + l - 1 <= a.S;
        }
        if (!ok)
            atomicOr(&s_bad, 1);
    }
    __syncthreads();
    if (s_bad) {
        if (t == 0) {
            pp.misc[MISC_NMOVING] = 0;
            *a.err = SPEC_REALIGN_LAYOUT;
        }
        return;
    }
    const int W = s_W;
    for (int b = t; b < a.B; b += nt) {
        const int n = a.idx[b];
        if (a.repad) {
            const int l = a.pool_len[n];
            pp.seq_src[b] = n;
            pp.src_off[b] = 0;
            pp.seq_dst[b] = b;
            pp.dst_off[b] = W - l;
            pp.rows[b] = l - 1;
            a.len_out[b] = l;
            a.pad_out[b] = W - l;
        } else {
            const int l = a.len[b] + (a.n_emit ? a.n_emit[b] : 0);
            pp.seq_src[b] = b;
            pp.src_off[b] = a.pad[b];
            pp.seq_dst[b] = n;
            pp.dst_off[b] = 0;
            pp.rows[b] = l - 1;
            a.pool_len_out[n] = l;
        }
    }
    __syncthreads();
    if (t == 0) {  // the rows to copy, in batch order
        int c = 0;
        for (int b = 0; b < a.B; ++b)
            if (pp.rows[b] > 0)
                pp.order[c++] = b;
        pp.misc[MISC_NMOVING] = c;
        pp.misc[MISC_WORK] = 0;
        if (a.repad)
            *a.width_out = W;
        *a.err = SPEC_REALIGN_OK;
    }
}

// every slab's run of every listed sequence, source and destination in
// different buffers (any tile order is safe)
struct PoolSource {
    const PoolArgs *a;
    PoolPlan pp;
    long long n_items, item;
    RunTiles cur;
    __device__ bool open(long long it)
    {
        if (it >= n_items)
            return false;
        const int sps = a->L * 2 * a->H;
        const long long row_bytes = (long long)a->D * a->elt_bytes;
        const long long slab_bytes = row_bytes * a->S;
        const int r = (int)(it / sps), within = (int)(it % sps);
        const int b = pp.order[r];
        const int h = within % a->H, lc = within / a->H;
        const int src_seqs = a->repad ? a->N : a->B, dst_seqs = a->repad ? a->B : a->N;
        const char *s = reinterpret_cast<const char *>(a->src) +
                        (((long long)lc * src_seqs + pp.seq_src[b]) * a->H + h) * slab_bytes;
        char *d = reinterpret_cast<char *>(a->dst) + (((long long)lc * dst_seqs + pp.seq_dst[b]) * a->H + h) * slab_bytes;
        cur.src = s + (long long)pp.src_off[b] * row_bytes;
        cur.dst = d + (long long)pp.dst_off[b] * row_bytes;
        cur.nbytes = (long long)pp.rows[b] * row_bytes;
        cur.done = 0;
        cur.desc = 0;
        return true;
    }
    __device__ bool next(const char *&s, char *&d, uint32_t &bytes)
    {
        while (!cur.next(s, d, bytes)) {
            if (!open(item))
                return false;
            item = atomicAdd(pp.misc + MISC_WORK, 1);
        }
        return true;
    }
};

__global__ void __launch_bounds__(32) pool_copy_bulk_kernel(PoolArgs a)
{
    extern __shared__ __align__(128) unsigned char stage_mem[];
    __shared__ __align__(8) uint64_t full[kBulkStages];
    if (threadIdx.x != 0)
        return;
    dep_wait();
    PoolSource src;
    src.a = &a;
    src.pp = pool_plan(a.ws, a.B);
    const int n = src.pp.misc[MISC_NMOVING];
    if (n <= 0)
        return;
    src.n_items = (long long)n * a.L * 2 * a.H;
    src.cur = RunTiles{nullptr, nullptr, 0, 0, 0};
    src.item = atomicAdd(src.pp.misc + MISC_WORK, 1);
    if (!bulk_copy_pipeline(src, stage_mem, full))
        *a.err = SPEC_REALIGN_TIMEOUT;
}

// rows that are not 16-byte multiples: one CTA per slab, element copies
template <typename E>
__global__ void __launch_bounds__(256) pool_copy_plain_kernel(PoolArgs a)
{
    dep_wait();
    const PoolPlan pp = pool_plan(a.ws, a.B);
    const int n = pp.misc[MISC_NMOVING];
    const int sps = a.L * 2 * a.H;
    const long long it = blockIdx.x;
    if (it >= (long long)n * sps)
        return;
    const int r = (int)(it / sps), within = (int)(it % sps);
    const int b = pp.order[r];
    const int h = within % a.H, lc = within / a.H;
    const int src_seqs = a.repad ? a.N : a.B, dst_seqs = a.repad ? a.B : a.N;
    const E *s = reinterpret_cast<const E *>(a.src) +
                 ((((long long)lc * src_seqs + pp.seq_src[b]) * a.H + h) * a.S + pp.src_off[b]) * a.D;
    E *d = reinterpret_cast<E *>(a.dst) + ((((long long)lc * dst_seqs + pp.seq_dst[b]) * a.H + h) * a.S + pp.dst_off[b]) *
                                              a.D;
    const long long cnt = (long long)pp.rows[b] * a.D;
    for (long long i = threadIdx.x; i < cnt; i += blockDim.x)
        d[i] = s[i];
}

static int g_pool_sm[64];
static bool g_pool_smem_set[64];

cudaError_t launch_pool_copy(const PoolArgs &a, cudaStream_t st)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const int slot = dev & 63;
    if (g_pool_sm[slot] == 0) {
        e = cudaDeviceGetAttribute(&g_pool_sm[slot], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
    }
    int threads = ((a.B + 31) / 32) * 32;
    threads = threads < 32 ? 32 : (threads > kPoolPlanThreads ? kPoolPlanThreads : threads);
    pool_plan_kernel<<<1, threads, 0, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const long long row_bytes = (long long)a.D * a.elt_bytes;
    const bool bulk = row_bytes % 16 == 0 && reinterpret_cast<uintptr_t>(a.src) % 16 == 0 &&
                      reinterpret_cast<uintptr_t>(a.dst) % 16 == 0;
    if (bulk) {
        if (!g_pool_smem_set[slot]) {
            e = cudaFuncSetAttribute(pool_copy_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kBulkSmem);
            if (e != cudaSuccess)
                return e;
            g_pool_smem_set[slot] = true;
        }
        cfg.gridDim = dim3(g_pool_sm[slot]);
        cfg.blockDim = dim3(32);
        cfg.dynamicSmemBytes = kBulkSmem;
        e = cudaLaunchKernelEx(&cfg, pool_copy_bulk_kernel, a);
    } else {
        cfg.gridDim = dim3((unsigned)((long long)a.B * a.L * 2 * a.H));
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = 0;
        e = a.elt_bytes == 4 ? cudaLaunchKernelEx(&cfg, pool_copy_plain_kernel<uint32_t>, a)
                             : cudaLaunchKernelEx(&cfg, pool_copy_plain_kernel<uint16_t>, a);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

// pool_len[idx[b]] += n_emit[b]; every index checked (range, repeats), every
// count (>= 0) and every new length (<= S) before anything is written
__global__ void __launch_bounds__(kPoolPlanThreads)
    commit_ragged_kernel(int N, int32_t *pool_len, int B, const int32_t *idx, const int32_t *n_emit, int S, int32_t *err)
{
    __shared__ uint32_t s_bits[kMaxPool / 32];
    __shared__ int s_bad, s_cap;
    const int t = threadIdx.x, nt = blockDim.x;
    for (int i = t; i < (N + 31) / 32; i += nt)
        s_bits[i] = 0;
    if (t == 0) {
        s_bad = 0;
        s_cap = 0;
    }
    __syncthreads();
    for (int b = t; b < B; b += nt) {
        const int n = idx[b];
        if (!mark_index(s_bits, n, N) || n_emit[b] < 0)
            atomicOr(&s_bad, 1);
        else if ((long long)pool_len[n] + n_emit[b] > S)
            atomicOr(&s_cap, 1);
    }
    __syncthreads();
    if (s_bad || s_cap) {
        if (t == 0)
            *err = s_bad ? SPEC_REALIGN_LAYOUT : SPEC_REALIGN_CAPACITY;
        return;
    }
    for (int b = t; b < B; b += nt)
        pool_len[idx[b]] += n_emit[b];
    if (t == 0)
        *err = SPEC_REALIGN_OK;
}

cudaError_t launch_commit_ragged(int N, int32_t *pool_len, int B, const int32_t *idx, const int32_t *n_emit, int S,
                                 int32_t *err, cudaStream_t st)
{
    int threads = ((B + 31) / 32) * 32;
    threads = threads < 32 ? 32 : (threads > kPoolPlanThreads ? kPoolPlanThreads : threads);
    commit_ragged_kernel<<<1, threads, 0, st>>>(N, pool_len, B, idx, n_emit, S, err);
    return cudaGetLastError();
}

}  // namespace spec
