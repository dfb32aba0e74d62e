// verify_greedy.cu -- greedy verification of one speculative round.
//
// Definition ("Chapter 10 Speculative Decoding (Code Walkthrough)", §4.1
// greedy_commit; "Design Document -- speculative-decoding-real", "Standard
// Greedy Algorithm" steps 4-6): the argmax of target row j is committed;
// the round stops after a mismatch with proposal j (the argmax is then the
// correction), after EOS, or at the output budget; after full acceptance the
// argmax of row k_b is the bonus, from the target ("Correctness Forensics for
// Batch Speculative Decoding", App. D).
//
// Roofline: HBM-bound stream of the needed rows, V * sizeof(T) bytes per row;
// one compare per element.  See verify_common.cuh for the decomposition.
#include "verify_common.cuh"

namespace spec {

// Threads per CTA of the greedy kernel: 128 measured as fast as 256 or
// faster on every workload (twice the CTAs per SM over the same units).
constexpr int kGreedyThreads = 128;

// Argmax key of chunk [lo, hi) of one row.  Per 16-byte vector: its
// NaN-propagating maximum (3 packed max instructions for 8 bf16 values); the
// elements are looked at one by one only when that maximum beats the running
// best, which happens O(log n) times per thread.  A chunk holding a NaN is
// recomputed exactly (NaN counts as larger than every number; first NaN wins).
// y: the row's proposal (-1: none).  As soon as this thread block has seen
// a finite element strictly above x[y] anywhere in its chunk, the row's
// argmax cannot be y: the row rejects, and its stop is posted at once
// (atomicMax(stop_word, stop_val)) so that later rows of the sequence can be
// skipped before the row is finalised.  (A NaN anywhere would be the argmax,
// which is not y either; x[y] NaN or y outside [0, V): no early test.)
template <typename T>
__device__ uint64_t chunk_argmax(const T *row, int V, int lo, int hi, uint64_t *s_red, const StopProbe &probe, int y,
                                 int *stop_word, int stop_val)
{
    constexpr int VEC = Storage<T>::kVec;
    constexpr int UNROLL = 8;  // 16-byte loads in flight per thread
    const ChunkSplit<T> cs(row, lo, hi);
    float best = -INFINITY;
    uint32_t bidx = 0xFFFFFFFFu;
    uint32_t first = 0xFFFFFFFFu;  // first element this thread saw
    bool nan = false;

    auto see = [&](float x, uint32_t i) {
        first = first == 0xFFFFFFFFu ? i : first;
        if (x > best) {
            best = x;
            bidx = i;
        }
        nan |= (x != x);
    };

    const int t = threadIdx.x;
    if (lo + t < cs.head_end)
        see(Storage<T>::at(row, lo + t), lo + t);
    const T *body = row + cs.head_end;
    if (t < cs.nvec)
        first = first == 0xFFFFFFFFu ? (uint32_t)(cs.head_end + t * VEC) : first;
    bool signalled = y < 0 || y >= V;  // warp-uniform
    float xy = INFINITY;
    int enc = 0;  // the stop word, read with the previous batch
    for (int base = 0; base < cs.nvec; base += UNROLL * kGreedyThreads) {  // warp-uniform trip count
        if (base > 0 && probe.stopped(enc))
            break;
        const int i = base + t;
        uint4 r[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int vi = i + u * kGreedyThreads;
            if (vi < cs.nvec)
                r[u] = ld_stream16(body + (size_t)vi * VEC);
        }
        enc = probe.load();  // in flight with the batch
        if (base == 0 && !signalled)
            xy = Storage<T>::at(row, y);  // after the batch's loads are in flight
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int vi = i + u * kGreedyThreads;
            if (vi < cs.nvec) {
                const float vm = vec_max<T>(r[u]);
                nan |= (vm != vm);
                if (vm > best) {  // a new maximum: its first position in the vector
                    float f[VEC];
                    Storage<T>::unpack(r[u], f);
                    int e = 0;
#pragma unroll
                    for (int q = VEC - 1; q >= 0; --q)
                        e = (f[q] == vm) ? q : e;
                    best = vm;
                    bidx = (uint32_t)(cs.head_end + vi * VEC + e);
                }
            }
        }
        if (!signalled && __any_sync(0xFFFFFFFFu, best > xy)) {
            if ((t & 31) == 0)
                atomicMax(stop_word, stop_val);
            signalled = true;
        }
    }
    if (cs.tail_beg + t < hi)
        see(Storage<T>::at(row, cs.tail_beg + t), cs.tail_beg + t);

    uint64_t key = 0;
    if (first != 0xFFFFFFFFu)
        key = bidx != 0xFFFFFFFFu ? argmax_key(best, bidx) : argmax_key(-INFINITY, first);
    if (__syncthreads_or(nan)) {  // rare: a NaN somewhere in the chunk
        key = 0;
        for (int i = lo + t; i < hi; i += kGreedyThreads) {
            const uint64_t kk = argmax_key(Storage<T>::at(row, i), (uint32_t)i);
            key = kk > key ? kk : key;
        }
    }
    return block_max_u64_to0(key, s_red);  // meaningful in thread 0
}

template <typename T>
__global__ void __launch_bounds__(kGreedyThreads) verify_greedy_kernel(VerifyArgs a)
{
    __shared__ uint64_t s_red[kGreedyThreads / 32];
    __shared__ int s_skip, s_last;  // written once each: no read/write race between them
    int *stop_enc = a.stop_enc, *row_cnt = a.row_cnt, *seq_cnt = a.seq_cnt, *row_tok = a.row_tok;
    uint64_t *part = static_cast<uint64_t *>(a.part);

    const Unit u = decode_unit(a);
    const int y = u.j < u.kb ? a.draft[(size_t)u.b * a.k + u.j] : -1;  // used after the first batch is issued
    if (threadIdx.x == 0)
        s_skip = (!u.needed || stopped_before(stop_enc, u.b, u.j)) ? 1 : 0;
    __syncthreads();
    if (!s_skip) {
        const T *row = reinterpret_cast<const T *>(a.logits) + (size_t)u.row * a.V;
        const int lo = u.c * a.chunk;
        const int hi = min(a.V, lo + a.chunk);
        const uint64_t key = chunk_argmax<T>(row, a.V, lo, hi, s_red, StopProbe{stop_enc, u.b, u.j}, y,
                                             stop_enc + u.b, kStopBase - u.j);
        if (threadIdx.x == 0)
            part[((size_t)u.row * a.C + u.c) * 2] = key;
    }
    // arrival on the row counter; the last CTA of the row finalises it
    if (threadIdx.x == 0) {
        if (a.C > 1) {
            __threadfence();
            s_last = (atomicAdd(row_cnt + u.row, 1) == a.C - 1) ? 1 : 0;
        } else {
            s_last = 1;  // a single-chunk row is finalised by its only CTA
        }
    }
    __syncthreads();
    if (!s_last || threadIdx.x >= 32)
        return;
    __threadfence();
    const int lane = threadIdx.x;
    // one reading of the stop word decides for the whole warp
    int eval = 0;
    if (lane == 0)
        eval = (u.needed && !stopped_before(stop_enc, u.b, u.j)) ? 1 : 0;
    eval = __shfl_sync(0xFFFFFFFFu, eval, 0);
    if (eval) {
        uint64_t key = 0;
        for (int c = lane; c < a.C; c += 32) {
            const uint64_t kk = part[((size_t)u.row * a.C + c) * 2];
            key = kk > key ? kk : key;
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) {
            const uint64_t o = shfl_xor_u64(key, m);
            key = o > key ? o : key;
        }
        if (lane == 0) {
            const int t = (int)key_index(key);
            row_tok[u.row] = t;
            bool stop;
            if (u.j < u.kb) {
                const int d = a.draft[(size_t)u.b * a.k + u.j];
                stop = (t != d) || (a.eos >= 0 && t == a.eos) || (u.j + 1 == u.rem);
            } else {
                stop = true;  // the bonus row ends the round
            }
            if (stop)
                atomicMax(stop_enc + u.b, kStopBase - u.j);
        }
    }
    int last_row = 0;
    if (lane == 0) {
        row_cnt[u.row] = 0;
        __threadfence();
        last_row = (atomicAdd(seq_cnt + u.b, 1) == a.k) ? 1 : 0;
    }
    last_row = __shfl_sync(0xFFFFFFFFu, last_row, 0);
    if (!last_row)
        return;
    __threadfence();

    // sequence finaliser: first-stop scan over rows 0..k with one ballot
    const int b = u.b, kb = u.kb, rem = u.rem, j = lane;
    int t = -1, d = -1;
    bool stop = false;
    if (j <= a.k && rem > 0) {
        t = row_tok[b * (a.k + 1) + j];
        if (j < kb) {
            d = a.draft[(size_t)b * a.k + j];
            stop = (t != d) || (a.eos >= 0 && t == a.eos) || (j + 1 == rem);
        } else {
            stop = (j == kb);
        }
    }
    const unsigned mask = __ballot_sync(0xFFFFFFFFu, stop);
    const int js = mask ? __ffs(mask) - 1 : -1;  // -1: nothing to commit
    const int t_js = __shfl_sync(0xFFFFFFFFu, t, js < 0 ? 0 : js);
    const int d_js = __shfl_sync(0xFFFFFFFFu, d, js < 0 ? 0 : js);
    if (j <= a.k)
        a.out_tokens[(size_t)b * (a.k + 1) + j] = (j <= js) ? t : -1;
    if (lane == 0) {
        a.n_emit[b] = js + 1;
        a.n_accept[b] = js < 0 ? 0 : ((js < kb && t_js == d_js) ? js + 1 : js);
        seq_cnt[b] = 0;
        stop_enc[b] = 0;
    }
}

void resolve_verify_args(VerifyArgs &a)
{
    const Split sp = verify_split(a.B, a.k, a.V);
    a.C = sp.C;
    a.chunk = sp.len;
    const Layout lay = make_layout(a.B, a.k, a.V);
    a.stop_enc = ws_at<int>(a.ws, lay.stop_enc);
    a.row_cnt = ws_at<int>(a.ws, lay.row_cnt);
    a.seq_cnt = ws_at<int>(a.ws, lay.seq_cnt);
    a.row_tok = ws_at<int>(a.ws, lay.row_tok);
    a.draw_row = ws_at<int>(a.ws, lay.draw_row);
    a.row_ms = ws_at<float2>(a.ws, lay.row_ms);
    a.row_flag = ws_at<uint32_t>(a.ws, lay.row_flag);
    a.row_cut = ws_at<float>(a.ws, lay.row_cut);
    a.part = ws_at<void>(a.ws, lay.part);
    a.rpart = ws_at<float>(a.ws, lay.rpart);
    a.rtot = ws_at<double>(a.ws, lay.rtot);
}

cudaError_t launch_verify_greedy(const VerifyArgs &args, spec_dtype dt, cudaStream_t st)
{
    VerifyArgs a = args;
    resolve_verify_args(a);
    const unsigned grid = (unsigned)(a.B * (a.k + 1) * a.C);
    switch (dt) {
    case SPEC_F32:
        verify_greedy_kernel<float><<<grid, kGreedyThreads, 0, st>>>(a);
        break;
    case SPEC_BF16:
        verify_greedy_kernel<__nv_bfloat16><<<grid, kGreedyThreads, 0, st>>>(a);
        break;
    case SPEC_F16:
        verify_greedy_kernel<__half><<<grid, kGreedyThreads, 0, st>>>(a);
        break;
    default:
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace spec
