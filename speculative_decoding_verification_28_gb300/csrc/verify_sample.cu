// verify_sample.cu -- stochastic verification of one speculative round.
//
// Definition ("Chapter 10 Speculative Decoding (Code Walkthrough)", §5.1;
// "Speculative decoding: proposals and verified output", "The mechanism"
// steps 2-4 and "Acceptance and rejection correction"):
//   p_j = softmax(x_j / T); proposal y accepted iff u_j < p_j(y) / q_j(y);
//   first rejection -> correction drawn from normalised max(0, p_j - q_j);
//   full acceptance -> bonus drawn from p_{k_b} (the target).
//
// Three kernels, stream-ordered:
//   stats  : per (b, j, chunk) online max / sum-of-exp of x/T (lazy rows, as
//            in the greedy kernel); the row's last CTA gathers x[y] and q[y],
//            runs the ratio test; the sequence's last row runs the first-stop
//            ballot scan and decides which row (if any) is drawn from;
//   draw   : per (b, chunk) of the drawn row, one pass over p (and q) that
//            sums the residual and p; the row's last CTA picks the mode,
//            finds the chunk holding u * total from the chunk prefix sums and
//            scans that one chunk (now in L2) for the inverse-CDF index;
//   resid  : optional, writes the normalised distribution of the draw.
// Roofline: HBM-bound; stats reads V * sizeof(T) per needed row; draw reads
// V * (sizeof(T) + 4) for one row per drawing sequence.
#include <float.h>

#include "verify_common.cuh"

namespace spec {

struct RowStats {
    float m, s;
};

// ---------------------------------------------------------------------------
// stats kernel
// ---------------------------------------------------------------------------
template <typename T>
__device__ void chunk_softmax_stats(const T *row, int lo, int hi, float inv_temp, bool unit, float &m_out,
                                    float &s_out, bool &bad_out, float *s_f, int *s_i)
{
    constexpr int VEC = Storage<T>::kVec;
    const ChunkSplit<T> cs(row, lo, hi);
    float m = -INFINITY, s = 0.0f;
    bool bad = false;
    auto add_vec = [&](const float *z, int n) {
        float vmax = -INFINITY;
        for (int e = 0; e < n; ++e) {
            vmax = fmaxf(vmax, z[e]);
            bad |= !(fabsf(z[e]) <= FLT_MAX);
        }
        if (vmax > m) {
            s = (m > -INFINITY) ? s * expf(m - vmax) : 0.0f;
            m = vmax;
        }
        if (m > -INFINITY)
            for (int e = 0; e < n; ++e)
                s += expf(z[e] - m);
    };
    const int t = threadIdx.x;
    if (lo + t < cs.head_end) {
        float z = Storage<T>::at(row, lo + t);
        z = unit ? z : z * inv_temp;
        add_vec(&z, 1);
    }
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
                if (!unit) {
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        f[e] *= inv_temp;
                }
                add_vec(f, VEC);
            }
        }
    }
    if (cs.tail_beg + t < hi) {
        float z = Storage<T>::at(row, cs.tail_beg + t);
        z = unit ? z : z * inv_temp;
        add_vec(&z, 1);
    }
    // block combine: max, then rescaled sum
    const int w = t >> 5, l = t & 31;
    float mm = m;
#pragma unroll
    for (int k = 16; k > 0; k >>= 1)
        mm = fmaxf(mm, __shfl_xor_sync(0xFFFFFFFFu, mm, k));
    if (l == 0)
        s_f[w] = mm;
    __syncthreads();
    float mb = -INFINITY;
    for (int i = 0; i < kThreads / 32; ++i)
        mb = fmaxf(mb, s_f[i]);
    float ss = (m > -INFINITY) ? s * expf(m - mb) : 0.0f;
#pragma unroll
    for (int k = 16; k > 0; k >>= 1)
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, k);
    const int any_bad = __syncthreads_or(bad);
    if (l == 0)
        s_f[kThreads / 32 + w] = ss;
    __syncthreads();
    float sb = 0.0f;
    for (int i = 0; i < kThreads / 32; ++i)
        sb += s_f[kThreads / 32 + i];
    m_out = mb;
    s_out = sb;
    bad_out = any_bad != 0;
    (void)s_i;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) verify_stats_kernel(VerifyArgs a)
{
    __shared__ float s_f[2 * kThreads / 32];
    __shared__ int s_flag;
    const Layout lay = make_layout(a.B, a.k, a.V);
    int *stop_enc = ws_at<int>(a.ws, lay.stop_enc);
    int *row_cnt = ws_at<int>(a.ws, lay.row_cnt);
    int *seq_cnt = ws_at<int>(a.ws, lay.seq_cnt);
    int *row_acc = ws_at<int>(a.ws, lay.row_tok);
    RowStats *row_ms = ws_at<RowStats>(a.ws, lay.row_ms);
    uint32_t *row_flag = ws_at<uint32_t>(a.ws, lay.row_flag);
    float4 *part = ws_at<float4>(a.ws, lay.part);
    int *draw_row = ws_at<int>(a.ws, lay.draw_row);

    const Unit u = decode_unit(a);
    const T *row = reinterpret_cast<const T *>(a.logits) + (size_t)u.row * a.V;
    if (threadIdx.x == 0)
        s_flag = (!u.needed || stopped_before(stop_enc, u.b, u.j)) ? 1 : 0;
    __syncthreads();
    if (!s_flag) {
        const int lo = u.c * kChunk;
        const int hi = min(a.V, lo + kChunk);
        float m, s;
        bool bad;
        chunk_softmax_stats<T>(row, lo, hi, a.inv_temp, a.unit_temp != 0, m, s, bad, s_f, nullptr);
        if (threadIdx.x == 0)
            part[(size_t)u.row * a.C + u.c] = make_float4(m, s, bad ? 1.0f : 0.0f, 0.0f);
    }
    if (threadIdx.x == 0) {
        __threadfence();
        s_flag = (atomicAdd(row_cnt + u.row, 1) == a.C - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!s_flag || threadIdx.x >= 32)
        return;
    __threadfence();
    const int lane = threadIdx.x;
    int eval = 0;
    if (lane == 0)
        eval = (u.needed && !stopped_before(stop_enc, u.b, u.j)) ? 1 : 0;
    eval = __shfl_sync(0xFFFFFFFFu, eval, 0);
    if (eval) {
        // merge the chunk statistics of the row
        float m = -INFINITY;
        for (int c = lane; c < a.C; c += 32)
            m = fmaxf(m, part[(size_t)u.row * a.C + c].x);
#pragma unroll
        for (int k = 16; k > 0; k >>= 1)
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, k));
        float s = 0.0f, bad = 0.0f;
        for (int c = lane; c < a.C; c += 32) {
            const float4 p = part[(size_t)u.row * a.C + c];
            if (p.x > -INFINITY)
                s += p.y * expf(p.x - m);
            bad = fmaxf(bad, p.z);
        }
#pragma unroll
        for (int k = 16; k > 0; k >>= 1) {
            s += __shfl_xor_sync(0xFFFFFFFFu, s, k);
            bad = fmaxf(bad, __shfl_xor_sync(0xFFFFFFFFu, bad, k));
        }
        if (lane == 0) {
            uint32_t fl = (bad > 0.0f || !(s <= FLT_MAX) || !(s > 0.0f)) ? SPEC_FLAG_NONFINITE : 0u;
            int acc = 0;
            bool stop;
            if (u.j < u.kb) {
                const int y = a.draft[(size_t)u.b * a.k + u.j];
                if (y < 0 || y >= a.V) {
                    fl |= SPEC_FLAG_BAD_TOKEN;
                } else {
                    float zy = Storage<T>::at(row, y);
                    zy = a.unit_temp ? zy : zy * a.inv_temp;
                    const float py = expf(zy - m) / s;
                    const float qy = a.q[((size_t)u.b * a.k + u.j) * a.V + y];
                    if (qy == 0.0f)
                        fl |= SPEC_FLAG_Q_ZERO;
                    const float ratio = py / qy;
                    acc = (a.u[(size_t)u.b * (a.k + 1) + u.j] < ratio) ? 1 : 0;
                    stop = false;
                }
                stop = !acc || (a.eos >= 0 && y == a.eos) || (u.j + 1 == u.rem);
            } else {
                stop = true;  // the bonus row ends the round
            }
            row_acc[u.row] = acc;
            row_ms[u.row] = RowStats{m, s};
            row_flag[u.row] = fl;
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

    // sequence finaliser: first stop by ballot, commit the accepted prefix,
    // hand the draw (correction or bonus) to the draw kernel
    const int b = u.b, kb = u.kb, rem = u.rem, j = lane;
    int acc = 0, d = -1;
    uint32_t fl = 0;
    bool stop = false;
    if (j <= a.k && rem > 0) {
        acc = row_acc[b * (a.k + 1) + j];
        fl = row_flag[b * (a.k + 1) + j];
        if (j < kb) {
            d = a.draft[(size_t)b * a.k + j];
            stop = !acc || (a.eos >= 0 && d == a.eos) || (j + 1 == rem);
        } else {
            stop = (j == kb);
        }
    }
    const unsigned mask = __ballot_sync(0xFFFFFFFFu, stop);
    const int js = mask ? __ffs(mask) - 1 : -1;
    const int acc_js = __shfl_sync(0xFFFFFFFFu, acc, js < 0 ? 0 : js);
    const bool accepted_stop = js >= 0 && js < kb && acc_js;  // EOS / budget on an accepted proposal
    uint32_t seq_fl = (j <= js) ? fl : 0u;
#pragma unroll
    for (int k = 16; k > 0; k >>= 1)
        seq_fl |= __shfl_xor_sync(0xFFFFFFFFu, seq_fl, k);
    if (j <= a.k) {
        int tok = -1;
        if (j < js || (j == js && accepted_stop))
            tok = d;
        a.out_tokens[(size_t)b * (a.k + 1) + j] = tok;
    }
    if (lane == 0) {
        a.n_emit[b] = js + 1;
        a.n_accept[b] = js < 0 ? 0 : (accepted_stop ? js + 1 : js);
        draw_row[b] = (js >= 0 && !accepted_stop) ? js : -1;
        if (a.flags)
            a.flags[b] = seq_fl;
        seq_cnt[b] = 0;
        stop_enc[b] = 0;
    }
}

// ---------------------------------------------------------------------------
// draw kernel: inverse CDF of the residual (or of p) for one row per sequence
// ---------------------------------------------------------------------------
template <typename T>
struct DrawRow {
    const T *x;       // target logits row
    const float *q;   // draft row (residual mode) or nullptr
    float m, s, it;   // row max / sum of the scaled logits, 1/T
    bool unit;
    __device__ float p(int v) const
    {
        float z = Storage<T>::at(x, v);
        z = unit ? z : z * it;
        return expf(z - m) / s;
    }
    // weight of index v; residual mode needs q
    __device__ float w(int v, bool residual) const
    {
        const float pv = p(v);
        return residual ? fmaxf(pv - __ldg(q + v), 0.0f) : pv;
    }
};

template <typename T>
__device__ DrawRow<T> draw_row_of(const VerifyArgs &a, int b, int r, int kb)
{
    const Layout lay = make_layout(a.B, a.k, a.V);
    const RowStats ms = ws_at<RowStats>(a.ws, lay.row_ms)[b * (a.k + 1) + r];
    DrawRow<T> d;
    d.x = reinterpret_cast<const T *>(a.logits) + ((size_t)b * (a.k + 1) + r) * a.V;
    d.q = (r < kb) ? a.q + ((size_t)b * a.k + r) * a.V : nullptr;
    d.m = ms.m;
    d.s = ms.s;
    d.it = a.inv_temp;
    d.unit = a.unit_temp != 0;
    return d;
}

__device__ __forceinline__ float block_sum(float v, float *s_f)
{
#pragma unroll
    for (int k = 16; k > 0; k >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, k);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0)
        s_f[w] = v;
    __syncthreads();
    float t = 0.0f;
    for (int i = 0; i < kThreads / 32; ++i)
        t += s_f[i];
    return t;
}

template <typename T>
__global__ void __launch_bounds__(kThreads) verify_draw_kernel(VerifyArgs a)
{
    __shared__ float s_f[kThreads / 32];
    __shared__ double s_d[kThreads / 32];
    __shared__ int s_flag, s_pick, s_lastpos;
    __shared__ double s_base;
    __shared__ int s_chunk;
    const Layout lay = make_layout(a.B, a.k, a.V);
    const int b = blockIdx.x / a.C, c = blockIdx.x % a.C;
    const int r = ws_at<int>(a.ws, lay.draw_row)[b];
    if (r < 0)
        return;
    int kb = a.draft_len ? a.draft_len[b] : a.k;
    kb = kb < 0 ? 0 : (kb > a.k ? a.k : kb);
    const bool residual = r < kb;
    const DrawRow<T> dr = draw_row_of<T>(a, b, r, kb);
    float *rpart = ws_at<float>(a.ws, lay.rpart);
    int *res_cnt = ws_at<int>(a.ws, lay.res_cnt);
    double *rtot = ws_at<double>(a.ws, lay.rtot);

    // pass over this chunk: sum of the residual and sum of p
    const int lo = c * kChunk, hi = min(a.V, lo + kChunk);
    float sr = 0.0f, sp = 0.0f;
    for (int v = lo + threadIdx.x; v < hi; v += kThreads) {
        const float pv = dr.p(v);
        sp += pv;
        if (residual)
            sr += fmaxf(pv - __ldg(dr.q + v), 0.0f);
    }
    sr = block_sum(sr, s_f);
    sp = block_sum(sp, s_f);
    if (threadIdx.x == 0) {
        rpart[((size_t)b * a.C + c) * 2 + 0] = sr;
        rpart[((size_t)b * a.C + c) * 2 + 1] = sp;
        __threadfence();
        s_flag = (atomicAdd(res_cnt + b, 1) == a.C - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!s_flag)
        return;
    __threadfence();

    // last CTA of the row: choose the weights, find the chunk, scan it
    bool use_res = false;
    if (threadIdx.x == 0) {
        double R = 0.0, P = 0.0;
        for (int i = 0; i < a.C; ++i) {
            R += (double)rpart[((size_t)b * a.C + i) * 2 + 0];
            P += (double)rpart[((size_t)b * a.C + i) * 2 + 1];
        }
        use_res = residual && R > 0.0;
        const int sel = use_res ? 0 : 1;
        const double W = use_res ? R : P;
        const double target = (double)a.u[(size_t)b * (a.k + 1) + a.k] * W;
        double acc = 0.0;
        int cs = -1, lastpos = -1;
        for (int i = 0; i < a.C; ++i) {
            const double pc = (double)rpart[((size_t)b * a.C + i) * 2 + sel];
            if (pc > 0.0)
                lastpos = i;
            if (cs < 0 && acc + pc > target) {
                cs = i;
                s_base = acc;
            }
            acc += pc;
        }
        if (cs < 0) {  // rounding left u * W at or past the total: last positive chunk
            cs = lastpos >= 0 ? lastpos : a.C - 1;
            s_base = -1.0;  // take the last positive index of that chunk
        }
        s_chunk = cs;
        s_pick = 0x7FFFFFFF;
        s_lastpos = -1;
        rtot[b] = use_res ? W : -W;  // sign records the mode for the residual writer
        if (residual && !use_res && a.flags)
            a.flags[b] |= SPEC_FLAG_ZERO_RESIDUAL;
        res_cnt[b] = 0;
        s_d[0] = target;
    }
    __syncthreads();
    use_res = rtot[b] > 0.0;
    const double target = s_d[0];
    const double base = s_base;
    const int cs = s_chunk;
    __syncthreads();
    // each thread owns a contiguous segment of the chunk
    const int clo = cs * kChunk, chi = min(a.V, clo + kChunk);
    const int per = (chi - clo + kThreads - 1) / kThreads;
    const int slo = clo + threadIdx.x * per, shi = min(chi, slo + per);
    float seg = 0.0f;
    int seg_last = -1;
    for (int v = slo; v < shi; ++v) {
        const float wv = dr.w(v, use_res);
        seg += wv;
        if (wv > 0.0f)
            seg_last = v;
    }
    // exclusive scan of the segment sums (fp64)
    double incl = (double)seg;
    const int l = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int k = 1; k < 32; k <<= 1) {
        const double o = __shfl_up_sync(0xFFFFFFFFu, incl, k);
        if (l >= k)
            incl += o;
    }
    if (l == 31)
        s_d[wid] = incl;
    __syncthreads();
    double warp_off = 0.0;
    for (int i = 0; i < wid; ++i)
        warp_off += s_d[i];
    double run = base + warp_off + incl - (double)seg;
    if (base >= 0.0) {
        for (int v = slo; v < shi; ++v) {
            run += (double)dr.w(v, use_res);
            if (run > target) {
                atomicMin(&s_pick, v);
                break;
            }
        }
    }
    if (seg_last >= 0)
        atomicMax(&s_lastpos, seg_last);
    __syncthreads();
    if (threadIdx.x == 0) {
        int tok = s_pick;
        if (tok == 0x7FFFFFFF)
            tok = s_lastpos >= 0 ? s_lastpos : chi - 1;
        a.out_tokens[(size_t)b * (a.k + 1) + r] = tok;
    }
}

// optional: the normalised distribution of each sequence's draw
template <typename T>
__global__ void __launch_bounds__(kThreads) verify_residual_kernel(VerifyArgs a)
{
    const Layout lay = make_layout(a.B, a.k, a.V);
    const int b = blockIdx.x / a.C, c = blockIdx.x % a.C;
    const int r = ws_at<int>(a.ws, lay.draw_row)[b];
    if (r < 0)
        return;
    int kb = a.draft_len ? a.draft_len[b] : a.k;
    kb = kb < 0 ? 0 : (kb > a.k ? a.k : kb);
    const DrawRow<T> dr = draw_row_of<T>(a, b, r, kb);
    const double W = ws_at<double>(a.ws, lay.rtot)[b];
    const bool use_res = W > 0.0;
    const float inv = (float)(1.0 / (use_res ? W : -W));
    const int lo = c * kChunk, hi = min(a.V, lo + kChunk);
    float *out = a.out_residual + (size_t)b * a.V;
    for (int v = lo + threadIdx.x; v < hi; v += kThreads)
        out[v] = dr.w(v, use_res) * inv;
}

template <typename T>
static cudaError_t launch_sample_t(const VerifyArgs &a, cudaStream_t st)
{
    const unsigned g1 = (unsigned)(a.B * (a.k + 1) * a.C);
    const unsigned g2 = (unsigned)(a.B * a.C);
    verify_stats_kernel<T><<<g1, kThreads, 0, st>>>(a);
    verify_draw_kernel<T><<<g2, kThreads, 0, st>>>(a);
    if (a.out_residual)
        verify_residual_kernel<T><<<g2, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_verify_sample(const VerifyArgs &a, spec_dtype dt, cudaStream_t st)
{
    switch (dt) {
    case SPEC_F32:
        return launch_sample_t<float>(a, st);
    case SPEC_BF16:
        return launch_sample_t<__nv_bfloat16>(a, st);
    case SPEC_F16:
        return launch_sample_t<__half>(a, st);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace spec
