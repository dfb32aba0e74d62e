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

// Argmax key of chunk [lo, hi) of one row: fast float compare per element,
// exact key recomputation for the (rare) chunk that holds a NaN.
template <typename T>
__device__ uint64_t chunk_argmax(const T *row, int lo, int hi, uint64_t *s_red)
{
    constexpr int VEC = Storage<T>::kVec;
    const ChunkSplit<T> cs(row, lo, hi);
    float best = -INFINITY;
    uint32_t bidx = 0xFFFFFFFFu;
    uint32_t first = 0xFFFFFFFFu;  // first element this thread saw
    bool nan = false;

    auto see = [&](float x, uint32_t i) {
        first = first == 0xFFFFFFFFu ? i : first;
        const bool gt = x > best;
        best = gt ? x : best;
        bidx = gt ? i : bidx;
        nan |= (x != x);
    };

    const int t = threadIdx.x;
    if (lo + t < cs.head_end)
        see(Storage<T>::at(row, lo + t), lo + t);
    const T *body = row + cs.head_end;
    for (int i = t; i < cs.nvec; i += 4 * kThreads) {
        uint4 r[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int vi = i + u * kThreads;
            if (vi < cs.nvec)
                r[u] = ld_stream16(body + (size_t)vi * VEC);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int vi = i + u * kThreads;
            if (vi < cs.nvec) {
                float f[VEC];
                Storage<T>::unpack(r[u], f);
                const uint32_t i0 = (uint32_t)(cs.head_end + vi * VEC);
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    see(f[e], i0 + e);
            }
        }
    }
    if (cs.tail_beg + t < hi)
        see(Storage<T>::at(row, cs.tail_beg + t), cs.tail_beg + t);

    uint64_t key = 0;
    if (first != 0xFFFFFFFFu)
        key = bidx != 0xFFFFFFFFu ? argmax_key(best, bidx) : argmax_key(-INFINITY, first);
    if (__syncthreads_or(nan)) {
        // exact path: NaN counts as larger than every number, first NaN wins
        key = 0;
        for (int i = lo + t; i < hi; i += kThreads) {
            const uint64_t kk = argmax_key(Storage<T>::at(row, i), (uint32_t)i);
            key = kk > key ? kk : key;
        }
    }
    return block_max_u64(key, s_red);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) verify_greedy_kernel(VerifyArgs a)
{
    __shared__ uint64_t s_red[kThreads / 32];
    __shared__ int s_flag;
    const Layout lay = make_layout(a.B, a.k, a.V);
    int *stop_enc = ws_at<int>(a.ws, lay.stop_enc);
    int *row_cnt = ws_at<int>(a.ws, lay.row_cnt);
    int *seq_cnt = ws_at<int>(a.ws, lay.seq_cnt);
    int *row_tok = ws_at<int>(a.ws, lay.row_tok);
    uint64_t *part = ws_at<uint64_t>(a.ws, lay.part);

    const Unit u = decode_unit(a);
    if (threadIdx.x == 0)
        s_flag = (!u.needed || stopped_before(stop_enc, u.b, u.j)) ? 1 : 0;
    __syncthreads();
    if (!s_flag) {
        const T *row = reinterpret_cast<const T *>(a.logits) + (size_t)u.row * a.V;
        const int lo = u.c * kChunk;
        const int hi = min(a.V, lo + kChunk);
        const uint64_t key = chunk_argmax<T>(row, lo, hi, s_red);
        if (threadIdx.x == 0)
            part[((size_t)u.row * a.C + u.c) * 2] = key;
    }
    // arrival on the row counter; the last CTA of the row finalises it
    if (threadIdx.x == 0) {
        __threadfence();
        s_flag = (atomicAdd(row_cnt + u.row, 1) == a.C - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!s_flag || threadIdx.x >= 32)
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

cudaError_t launch_verify_greedy(const VerifyArgs &a, spec_dtype dt, cudaStream_t st)
{
    const unsigned grid = (unsigned)(a.B * (a.k + 1) * a.C);
    switch (dt) {
    case SPEC_F32:
        verify_greedy_kernel<float><<<grid, kThreads, 0, st>>>(a);
        break;
    case SPEC_BF16:
        verify_greedy_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(a);
        break;
    case SPEC_F16:
        verify_greedy_kernel<__half><<<grid, kThreads, 0, st>>>(a);
        break;
    default:
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace spec
