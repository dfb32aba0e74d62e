// realign.cu -- ragged-to-rectangular realignment of a contiguous
// left-padded KV cache after a speculative round ("unpad-append-repad",
// "Correctness Forensics for Batch Speculative Decoding", §3.2 and App. B:
// relocate retained entries, drop rejected ones, keep the target-computed
// entries of accepted tokens, repad).
//
// plan  (1 CTA): checks rectangular alignment of the input, computes
//       len' = len + n, W' = max len', pad' = W' - len', the shift
//       delta = pad' - pad and the run of len' - 1 rows to move, and lists the
//       sequences that move, longest run first (so the long slabs start early
//       and the tail of the shift is short).
// shift (persistent, one thread per CTA drives the bulk-copy engine): each
//       (layer, K/V, sequence, head) slab of a moving sequence, in every cache
//       the call realigns (e.g. target and draft, by the one plan), is an in-place
//       memmove of run * D * elt contiguous bytes by delta rows.  Tiles are
//       staged global -> shared -> global with cp.async.bulk; they are taken
//       from the end the run moves towards (descending for delta > 0), so a
//       tile's destination overlaps only its own source and sources already
//       loaded.  Loads run up to kStages - 1 tiles ahead of the stores; the
//       stores are issued strictly in tile order after each tile's load has
//       completed on its mbarrier.
// Roofline: HBM-bound, 2 * run * D * elt bytes per moving slab.
#include "bulk_copy.cuh"
#include "spec_common.cuh"
#include "spec_launch.h"

namespace spec {

constexpr int kPlanThreads = 1024;
constexpr int kSortMax = 2048;  // longest-first ordering up to this batch size

struct PlanView {
    int *order, *delta, *src_pad, *run, *misc;
};

__device__ __forceinline__ PlanView plan_view(void *ws, int B)
{
    const Layout lay = make_layout(B, 0, 1);
    return PlanView{ws_at<int>(ws, lay.order), ws_at<int>(ws, lay.delta), ws_at<int>(ws, lay.src_pad),
                    ws_at<int>(ws, lay.run), ws_at<int>(ws, lay.misc)};
}

__global__ void __launch_bounds__(kPlanThreads) realign_plan_kernel(RealignArgs a)
{
    __shared__ uint64_t s_key[kSortMax];
    __shared__ int s_bad2, s_bad3, s_minpad, s_maxlen, s_count, s_rows;
    // the shift kernel may be scheduled now; it waits for this grid's results
    dep_release();
    const PlanView pv = plan_view(a.ws, a.B);
    const int t = threadIdx.x;
    const int nt = blockDim.x;
    if (t == 0) {
        s_bad2 = 0;
        s_bad3 = 0;
        s_minpad = 0x7FFFFFFF;
        s_maxlen = 0;
        s_count = 0;
        s_rows = 0;
    }
    __syncthreads();
    const int W = a.pad[0] + a.len[0];
    int bad2 = 0, bad3 = 0, minpad = 0x7FFFFFFF, maxlen = 0;
    for (int b = t; b < a.B; b += nt) {
        const int l = a.len[b], p = a.pad[b], n = a.n_emit[b];
        if (l < 1 || p < 0 || p + l != W)
            bad2 = 1;
        if (n < 0 || (long long)W + n - 1 > a.S)
            bad3 = 1;
        minpad = min(minpad, p);
        if (n >= 0)
            maxlen = max(maxlen, l + n);
    }
    if (bad2)
        atomicOr(&s_bad2, 1);
    if (bad3)
        atomicOr(&s_bad3, 1);
    atomicMin(&s_minpad, minpad);
    atomicMax(&s_maxlen, maxlen);
    __syncthreads();
    int err = SPEC_REALIGN_OK;
    if (s_bad2 || s_minpad != 0)
        err = SPEC_REALIGN_LAYOUT;
    else if (s_bad3)
        err = SPEC_REALIGN_EMIT;
    else if (s_maxlen > a.S)
        err = SPEC_REALIGN_CAPACITY;
    const int Wn = s_maxlen;
    if (err != SPEC_REALIGN_OK) {
        if (t == 0) {
            pv.misc[MISC_NMOVING] = 0;
            pv.misc[MISC_ERR] = err;
            *a.err = err;
        }
        return;
    }
    // per-sequence shift; inputs are read before any output is written
    // (len_new / pad_new may alias len / pad)
    int rows = 0;
    for (int b = t; b < a.B; b += nt) {
        const int l = a.len[b], p = a.pad[b], n = a.n_emit[b];
        const int ln = l + n, pn = Wn - ln;
        const int d = pn - p;
        const int run = (d != 0 && ln - 1 > 0) ? ln - 1 : 0;
        pv.delta[b] = d;
        pv.src_pad[b] = p;
        pv.run[b] = run;
        rows += run;
    }
    atomicAdd(&s_rows, rows);
    __syncthreads();
    for (int b = t; b < a.B; b += nt) {
        const int pn = pv.src_pad[b] + pv.delta[b];
        a.pad_new[b] = pn;
        a.len_new[b] = Wn - pn;
    }
    // moving sequences, longest run first (ties: lower index first)
    if (a.B <= kSortMax) {
        int P = 1;
        while (P < a.B)
            P <<= 1;
        for (int i = t; i < P; i += nt) {
            uint64_t key = 0;
            if (i < a.B && pv.run[i] > 0)
                key = ((uint64_t)pv.run[i] << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)i);
            s_key[i] = key;
        }
        __syncthreads();
        for (int size = 2; size <= P; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int i = t; i < P; i += nt) {
                    const int jx = i ^ stride;
                    if (jx > i) {
                        const bool desc = (i & size) == 0;
                        const uint64_t x = s_key[i], y = s_key[jx];
                        if (desc ? (x < y) : (x > y)) {
                            s_key[i] = y;
                            s_key[jx] = x;
                        }
                    }
                }
                __syncthreads();
            }
        }
        for (int i = t; i < a.B; i += nt) {
            const uint64_t key = s_key[i];
            if (key != 0) {
                pv.order[i] = (int)(0xFFFFFFFFu - (uint32_t)key);
                atomicAdd(&s_count, 1);
            }
        }
    } else {
        // large batches: stable compaction in index order
        if (t == 0) {
            int c = 0;
            for (int b = 0; b < a.B; ++b)
                if (pv.run[b] > 0)
                    pv.order[c++] = b;
            s_count = c;
        }
    }
    __syncthreads();
    if (t == 0) {
        pv.misc[MISC_NMOVING] = s_count;
        pv.misc[MISC_WORK] = 0;
        pv.misc[MISC_WIDTH] = Wn;
        pv.misc[MISC_ERR] = 0;
        pv.misc[MISC_TOTAL_ROWS] = s_rows;
        *a.width_new = Wn;
        *a.err = SPEC_REALIGN_OK;
    }
}

// ---------------------------------------------------------------------------
// bulk-copy shift
// ---------------------------------------------------------------------------
constexpr int kShiftSmem = kBulkSmem;

// the moving slabs of every bulk cache, fetched longest-first from a shared
// counter; each slab's run is tiled from the end it moves towards
struct ShiftSource {
    const RealignArgs *a;
    PlanView pv;
    int n_moving;
    long long n_items, item;
    RunTiles cur;
    __device__ bool open(long long it)
    {
        if (it >= n_items)
            return false;
        int c = 0;
        for (; c < a->n_caches; ++c) {
            if (!(a->bulk_mask & (1u << c)))
                continue;
            const long long cnt = (long long)n_moving * a->cache[c].L * 2 * a->cache[c].H;
            if (it < cnt)
                break;
            it -= cnt;
        }
        const CacheDesc &cd = a->cache[c];
        const int sps = cd.L * 2 * cd.H;  // slabs per sequence
        const long long row_bytes = (long long)cd.D * cd.elt_bytes;
        const long long slab_bytes = row_bytes * a->S;
        const int r = (int)(it / sps), within = (int)(it % sps);
        const int b = pv.order[r];
        const int h = within % cd.H, lc = within / cd.H;  // lc = l * 2 + k/v
        char *slab = reinterpret_cast<char *>(cd.kv) + (((long long)lc * a->B + b) * cd.H + h) * slab_bytes;
        const int d = pv.delta[b];
        cur.src = slab + (long long)pv.src_pad[b] * row_bytes;
        cur.dst = slab + (long long)(pv.src_pad[b] + d) * row_bytes;
        cur.nbytes = (long long)pv.run[b] * row_bytes;
        cur.done = 0;
        cur.desc = d > 0;
        return true;
    }
    __device__ bool next(const char *&s, char *&d, uint32_t &bytes)
    {
        while (!cur.next(s, d, bytes)) {
            if (!open(item))
                return false;
            item = atomicAdd(pv.misc + MISC_WORK, 1);  // the item after, fetched ahead
        }
        return true;
    }
};

__global__ void __launch_bounds__(32) kv_shift_bulk_kernel(RealignArgs a)
{
    extern __shared__ __align__(128) unsigned char stage_mem[];
    __shared__ __align__(8) uint64_t full[kBulkStages];
    if (threadIdx.x != 0)
        return;
    dep_wait();     // the plan kernel's results are complete and visible
    dep_release();  // a following position/mask rebuild may run alongside
    ShiftSource src;
    src.a = &a;
    src.pv = plan_view(a.ws, a.B);
    src.n_moving = src.pv.misc[MISC_NMOVING];
    if (src.n_moving <= 0)
        return;
    src.n_items = 0;
    for (int c = 0; c < a.n_caches; ++c)
        if (a.bulk_mask & (1u << c))
            src.n_items += (long long)src.n_moving * a.cache[c].L * 2 * a.cache[c].H;
    src.cur = RunTiles{nullptr, nullptr, 0, 0, 0};
    src.item = atomicAdd(src.pv.misc + MISC_WORK, 1);
    if (!bulk_copy_pipeline(src, stage_mem, full))
        *a.err = SPEC_REALIGN_TIMEOUT;
}

// Plain path for rows that are not a multiple of 16 bytes (or an unaligned
// cache): one CTA per slab, tiles staged in registers, element granularity.
template <typename E>
__global__ void __launch_bounds__(256) kv_shift_plain_kernel(RealignArgs a)
{
    dep_wait();
    dep_release();
    const PlanView pv = plan_view(a.ws, a.B);
    const int n_moving = pv.misc[MISC_NMOVING];
    const CacheDesc &cd = a.cache[a.plain_cache];
    const int sps = cd.L * 2 * cd.H;
    const long long it = blockIdx.x;
    if (it >= (long long)n_moving * sps)
        return;
    const int r = (int)(it / sps), within = (int)(it % sps);
    const int b = pv.order[r];
    const int h = within % cd.H, lc = within / cd.H;
    const long long slab = ((long long)lc * a.B + b) * cd.H + h;
    E *base = reinterpret_cast<E *>(cd.kv) + slab * (long long)a.S * cd.D;
    const int d = pv.delta[b];
    const long long n = (long long)pv.run[b] * cd.D;
    E *src = base + (long long)pv.src_pad[b] * cd.D;
    E *dst = src + (long long)d * cd.D;
    constexpr int kPer = 4, kT = 256 * kPer;
    for (long long done = 0; done < n; done += kT) {
        const long long take = (n - done) < kT ? (n - done) : kT;
        const long long lo = d > 0 ? n - done - take : done;
        E v[kPer];
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            const long long i = lo + threadIdx.x + e * 256;
            if (i < lo + take)
                v[e] = src[i];
        }
        __syncthreads();  // the whole tile is read before any of it is written
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            const long long i = lo + threadIdx.x + e * 256;
            if (i < lo + take)
                dst[i] = v[e];
        }
        __syncthreads();
    }
}

static int g_sm_count[64];
static bool g_smem_set[64];

cudaError_t launch_realign(const RealignArgs &a, cudaStream_t st)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const int slot = dev & 63;
    if (g_sm_count[slot] == 0) {
        e = cudaDeviceGetAttribute(&g_sm_count[slot], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
    }
    int plan_threads = ((a.B + 31) / 32) * 32;
    plan_threads = plan_threads < 32 ? 32 : (plan_threads > kPlanThreads ? kPlanThreads : plan_threads);
    realign_plan_kernel<<<1, plan_threads, 0, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    // the shift is launched programmatically: it becomes resident while the
    // plan runs and waits for it on the device
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    RealignArgs la = a;
    la.bulk_mask = 0;
    for (int c = 0; c < a.n_caches; ++c) {
        const long long row_bytes = (long long)a.cache[c].D * a.cache[c].elt_bytes;
        if (row_bytes % 16 == 0 && reinterpret_cast<uintptr_t>(a.cache[c].kv) % 16 == 0)
            la.bulk_mask |= 1u << c;
    }
    if (la.bulk_mask) {
        if (!g_smem_set[slot]) {
            e = cudaFuncSetAttribute(kv_shift_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kShiftSmem);
            if (e != cudaSuccess)
                return e;
            g_smem_set[slot] = true;
        }
        cfg.gridDim = dim3(g_sm_count[slot]);
        cfg.blockDim = dim3(32);
        cfg.dynamicSmemBytes = kShiftSmem;
        e = cudaLaunchKernelEx(&cfg, kv_shift_bulk_kernel, la);
        if (e != cudaSuccess)
            return e;
    }
    // caches whose rows are not 16-byte multiples (or that are unaligned)
    for (int c = 0; c < a.n_caches; ++c) {
        if (la.bulk_mask & (1u << c))
            continue;
        RealignArgs pa = la;
        pa.plain_cache = c;
        const long long blocks = (long long)a.B * a.cache[c].L * 2 * a.cache[c].H;
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = 0;
        if (a.cache[c].elt_bytes == 4)
            e = cudaLaunchKernelEx(&cfg, kv_shift_plain_kernel<uint32_t>, pa);
        else
            e = cudaLaunchKernelEx(&cfg, kv_shift_plain_kernel<uint16_t>, pa);
        if (e != cudaSuccess)
            return e;
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace spec
