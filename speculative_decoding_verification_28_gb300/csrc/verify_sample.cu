// verify_sample.cu -- stochastic verification of one speculative round.
//
// Definition ("Chapter 10 Speculative Decoding (Code Walkthrough)", §5.1;
// "Speculative decoding: proposals and verified output", "The mechanism"
// steps 2-4 and "Acceptance and rejection correction"):
//   p_j = softmax(x_j / T); proposal y accepted iff u_j < p_j(y) / q_j(y);
//   first rejection -> correction drawn from normalised max(0, p_j - q_j);
//   full acceptance -> bonus drawn from p_{k_b} (the target).
//
// Arithmetic: p_v = 2^(x_v * c - m) / s with c = log2(e) / T, m the row
// maximum of x * c and s = sum of 2^(x * c - m) -- the same softmax in base
// 2, so each element costs one FFMA and one ex2.approx.  A -inf logit is a masked
// token (probability 0); NaN / +inf, or a row without a finite logit, flags
// the row as undefined.
//
// Three kernels, stream-ordered:
//   stats  : per (b, j, chunk) max / sum of 2^(x c - m) (lazy rows, as in the
//            greedy kernel; 8 loads in flight per thread, one packed maximum
//            and one rescale test per batch of vectors); the row's last CTA
//            gathers x[y] and q[y] and runs the ratio test; the sequence's
//            last row runs the first-stop ballot and decides which row (if
//            any) is drawn from.  With top-k / top-p the filter kernel of
//            verify_filter.cuh takes this place (one CTA per row, and the
//            row's cut goes to the draw kernel);
//   draw   : per (b, chunk) of the drawn row, one vectorised pass summing the
//            residual and p; the row's last CTA picks the mode, finds the chunk
//            holding u * total from the chunk sums, stages that chunk's weights
//            in shared memory and scans them for the inverse-CDF index; it is
//            launched programmatically and waits for the first kernel on the
//            device;
//   resid  : optional, writes the normalised distribution of the draw.
// Roofline: HBM-bound; stats reads V * sizeof(T) per needed row; draw reads
// V * (sizeof(T) + 4) for one row per drawing sequence.
#include <float.h>

#include <type_traits>

#include "bulk_copy.cuh"
#include "sample_final.cuh"

namespace spec {


// ---------------------------------------------------------------------------
// stats kernel
// ---------------------------------------------------------------------------
// kRaw: also the unscaled maximum of the logits (to xmax_out of warp 0;
// s_f then needs 4 * NT / 32 floats); NT = threads of the block
template <typename T, bool kRaw, int NT = kThreads>
__device__ void chunk_softmax_stats(const T *row, int lo, int hi, float c, float &m_out, float &s_out,
                                    bool &bad_out, float *s_f, const StopProbe &probe, float *xmax_out)
{
    constexpr int VEC = Storage<T>::kVec;
    const ChunkSplit<T> cs(row, lo, hi);
    float m = -INFINITY, s = 0.0f, xr = -INFINITY;
    bool bad = false;
    // one element (head / tail)
    auto add1 = [&](float x) {
        if (kRaw)
            xr = max_nan(xr, x);
        const float z = x * c;
        bad |= !(z < INFINITY);  // NaN or +inf; -inf is a masked token
        if (z > m) {
            s = (m > -INFINITY) ? s * exp2f(m - z) : 0.0f;
            m = z;
        }
        if (m > -INFINITY)
            s += exp2_sfu(fmaf(x, c, -m));
    };
    const int t = threadIdx.x;
    if (lo + t < cs.head_end)
        add1(Storage<T>::at(row, lo + t));
    const T *body = row + cs.head_end;
    // Full batches (every thread has all its vectors in range): one packed
    // maximum over the batch, one NaN / +inf test and one rescale test per
    // batch, and a lazy reference: sums are kept relative to `m`, which is
    // moved only when the batch maximum exceeds it by more than 8 (terms up
    // to 2^8 lose nothing in fp32); `mt` tracks the exact maximum and the sum
    // is brought to it once at the end.  Four partial sums break the add
    // chain.  What remains after the full batches takes the guarded loop.
    float mt = m;                              // the head element, if any, is already in (m, s)
    float sa[4] = {s, 0.0f, 0.0f, 0.0f};
    int base = 0;
    bool dropped = false;
    // one full batch of NB vectors per thread starting at vector `base`
    auto batch = [&](auto nb) {
        constexpr int NB = decltype(nb)::value;
        uint4 r[NB];
#pragma unroll
        for (int u = 0; u < NB; ++u)
            r[u] = ld_stream16(body + (size_t)(base + t + u * NT) * VEC);
        uint4 mx = r[0];
#pragma unroll
        for (int u = 1; u < NB; ++u)
            mx = max_vec<T>(mx, r[u]);
        const float vraw = vec_max<T>(mx);
        if (kRaw)
            xr = max_nan(xr, vraw);
        const float vm = vraw * c;  // c > 0: the maximum commutes with the scale
        bad |= !(vm < INFINITY);    // NaN or +inf in the batch
        mt = fmaxf(mt, vm);
        if (vm > m + 8.0f || m == -INFINITY) {
            const float scale = (m > -INFINITY) ? exp2f(m - vm) : 0.0f;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                sa[q] *= scale;
            m = vm;
        }
        if (m > -INFINITY) {
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                float f[VEC];
                Storage<T>::unpack(r[u], f);
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    sa[e & 3] += exp2_sfu(fmaf(f[e], c, -m));
            }
        }
    };
    // full batches of 8 vectors (128 bytes in flight per thread)
    for (; base + 8 * NT <= cs.nvec; base += 8 * NT) {  // warp-uniform trip count
        if (base > 0 && probe.dropped()) {
            dropped = true;
            break;
        }
        batch(std::integral_constant<int, 8>());
    }
    s = (sa[0] + sa[1]) + (sa[2] + sa[3]);
    if (m > -INFINITY && mt > m) {  // bring the sum to the exact maximum
        s *= exp2f(m - mt);
        m = mt;
    }
    // the rest (fewer than 8 vectors per thread): one guarded round, all of
    // its loads in flight together
    constexpr int GU = 8;
    for (; !dropped && base < cs.nvec; base += GU * NT) {
        if (base > 0 && probe.dropped())
            break;
        const int i = base + t;
        uint4 r[GU];
#pragma unroll
        for (int u = 0; u < GU; ++u) {
            const int vi = i + u * NT;
            if (vi < cs.nvec)
                r[u] = ld_stream16(body + (size_t)vi * VEC);
        }
#pragma unroll
        for (int u = 0; u < GU; ++u) {
            const int vi = i + u * NT;
            if (vi < cs.nvec) {
                const float vraw = vec_max<T>(r[u]);
                if (kRaw)
                    xr = max_nan(xr, vraw);
                const float vm = vraw * c;  // c > 0: the maximum commutes with the scale
                bad |= !(vm < INFINITY);                // NaN or +inf in the vector
                if (vm > m) {
                    s = (m > -INFINITY) ? s * exp2f(m - vm) : 0.0f;
                    m = vm;
                }
                if (m > -INFINITY) {
                    float f[VEC];
                    Storage<T>::unpack(r[u], f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        s += exp2_sfu(fmaf(f[e], c, -m));
                }
            }
        }
    }
    if (cs.tail_beg + t < hi)
        add1(Storage<T>::at(row, cs.tail_beg + t));
    // combine for thread 0: (max, rescaled sum) merged within each warp by
    // shuffles, then across warps by warp 0 after one barrier
    const int w = t >> 5, l = t & 31;
    auto merge = [](float &ma, float &sa, float mb, float sb) {
        const float mx = fmaxf(ma, mb);
        const float a = (ma > -INFINITY) ? sa * exp2f(ma - mx) : 0.0f;
        const float b = (mb > -INFINITY) ? sb * exp2f(mb - mx) : 0.0f;
        ma = mx;
        sa = a + b;
    };
#pragma unroll
    for (int k = 16; k > 0; k >>= 1)
        merge(m, s, __shfl_xor_sync(0xFFFFFFFFu, m, k), __shfl_xor_sync(0xFFFFFFFFu, s, k));
    const bool wbad = __any_sync(0xFFFFFFFFu, bad);
    if (kRaw) {
#pragma unroll
        for (int k = 16; k > 0; k >>= 1)
            xr = max_nan(xr, __shfl_xor_sync(0xFFFFFFFFu, xr, k));
    }
    if (l == 0) {
        s_f[w] = m;
        s_f[NT / 32 + w] = wbad ? -s : s;  // the sign carries the warp's flag (s >= 0)
        s_f[2 * (NT / 32) + w] = wbad ? 1.0f : 0.0f;
        if (kRaw)
            s_f[3 * (NT / 32) + w] = xr;
    }
    __syncthreads();
    if (t < 32) {
        float mm = (l < NT / 32) ? s_f[l] : -INFINITY;
        float ss = (l < NT / 32) ? fabsf(s_f[NT / 32 + l]) : 0.0f;
        const bool bb = (l < NT / 32) && s_f[2 * (NT / 32) + l] > 0.0f;
#pragma unroll
        for (int k = 16; k > 0; k >>= 1)
            merge(mm, ss, __shfl_xor_sync(0xFFFFFFFFu, mm, k), __shfl_xor_sync(0xFFFFFFFFu, ss, k));
        m_out = mm;
        s_out = ss;
        bad_out = __any_sync(0xFFFFFFFFu, bb);
        if (kRaw) {
            float xx = (l < NT / 32) ? s_f[3 * (NT / 32) + l] : -INFINITY;
#pragma unroll
            for (int k = 16; k > 0; k >>= 1)
                xx = max_nan(xx, __shfl_xor_sync(0xFFFFFFFFu, xx, k));
            *xmax_out = xx;
        }
    }
}

// (max, sum) of two base-2 softmax partials
__device__ __forceinline__ void merge_ms(float &ma, float &sa, float mb, float sb)
{
    const float mx = fmaxf(ma, mb);
    const float x = (ma > -INFINITY) ? sa * exp2f(ma - mx) : 0.0f;
    const float y = (mb > -INFINITY) ? sb * exp2f(mb - mx) : 0.0f;
    ma = mx;
    sa = x + y;
}

// One lane, after the last unit of row u.row was counted: unless an earlier
// stop is known, merges the row's chunk partials (read through L2: other
// CTAs wrote them) and runs the ratio test; resets the row's counter.  y is
// the row's proposal (row_proposal), loaded by the caller ahead of time.
// The stop word, the partials and the test's inputs are loaded together.
template <typename T>
__device__ void stats_row_finish(const VerifyArgs &a, const Unit &u, int y)
{
    if (u.needed) {
        const bool stopped = stopped_before(a.stop_enc, u.b, u.j);
        const T *row = reinterpret_cast<const T *>(a.logits) + (size_t)u.row * a.V;
        const RowInputs in = row_inputs<T>(a, u, row, y);
        const float4 *part = static_cast<const float4 *>(a.part) + (size_t)u.row * a.C;
        float m = -INFINITY, s = 0.0f;
        bool bad = false;
#pragma unroll 8
        for (int cc = 0; cc < a.C; ++cc) {
            const float4 p = __ldcg(part + cc);
            merge_ms(m, s, p.x, p.y);
            bad |= p.z > 0.0f;
        }
        if (!stopped)
            row_decide(a, u, in, m, s, -INFINITY, bad);
    }
    a.row_cnt[u.row] = 0;
}

// One lane, after unit u's chunk statistics (m, s, bad: the base-2 maximum,
// the sum relative to it and the non-finite flag; m = -inf and s = 0 for a
// chunk that was not read): stores the partial and counts it; the row's last
// unit finishes the row and counts it for the sequence.  True when that was
// the sequence's last row.  The row's proposal is loaded before the counter
// round trip, in case this unit is the last.
template <typename T>
__device__ bool stats_unit_count(const VerifyArgs &a, const Unit &u, float m_c, float s_c, bool bad_c)
{
    const int y = u.needed ? row_proposal(a, u) : -1;
    static_cast<float4 *>(a.part)[(size_t)u.row * a.C + u.c] = make_float4(m_c, s_c, bad_c ? 1.0f : 0.0f, 0.0f);
    if (a.C > 1) {
        __threadfence();
        if (atomicAdd(a.row_cnt + u.row, 1) != a.C - 1)
            return false;
        __threadfence();
    }
    stats_row_finish<T>(a, u, y);
    return sample_seq_count(a, u.b);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) verify_stats_kernel(VerifyArgs a)
{
    __shared__ float s_f[3 * kThreads / 32];
    __shared__ int s_skip;
    const float c = scale_of(a);
    const Unit u = decode_unit(a);
    const T *row = reinterpret_cast<const T *>(a.logits) + (size_t)u.row * a.V;
    if (threadIdx.x == 0)
        s_skip = (!u.needed || stopped_before(a.stop_enc, u.b, u.j)) ? 1 : 0;
    __syncthreads();
    float m = -INFINITY, s = 0.0f;
    bool bad = false;
    if (!s_skip) {
        const int lo = u.c * a.chunk;
        const int hi = min(a.V, lo + a.chunk);
        chunk_softmax_stats<T, false>(row, lo, hi, c, m, s, bad, s_f, StopProbe{a.stop_enc, u.b, u.j}, nullptr);
    }
    if (threadIdx.x < 32) {
        int seq_last = 0;
        if (threadIdx.x == 0)
            seq_last = stats_unit_count<T>(a, u, m, s, bad) ? 1 : 0;
        if (__shfl_sync(0xFFFFFFFFu, seq_last, 0))
            sample_seq_outputs(a, u.b, u.kb, u.rem);
    }
}

}  // namespace spec

#include "verify_filter.cuh"

namespace spec {

// ---------------------------------------------------------------------------
// draw kernel: inverse CDF of the residual (or of p) for one row per sequence
// ---------------------------------------------------------------------------
template <typename T>
struct DrawRow {
    const T *x;      // target logits row
    const float *q;  // draft row (residual mode) or nullptr
    float m, inv_s, c;  // base-2 row maximum, 1 / kept sum, scale log2(e)/T
    float cut;          // smallest kept logit (-inf: no top-k / top-p)
    __device__ float p(float x_v) const { return (x_v >= cut) ? exp2_sfu(fmaf(x_v, c, -m)) * inv_s : 0.0f; }
    __device__ float pv(int v) const { return p(Storage<T>::at(x, v)); }
    // weight of index v; residual mode needs q
    __device__ float w(int v, bool residual) const
    {
        const float p_v = pv(v);
        return residual ? fmaxf(p_v - __ldg(q + v), 0.0f) : p_v;
    }
};

template <typename T>
__device__ DrawRow<T> draw_row_of(const VerifyArgs &a, int b, int r, int kb)
{
    const RowStats ms = reinterpret_cast<const RowStats *>(a.row_ms)[b * (a.k + 1) + r];
    DrawRow<T> d;
    d.x = reinterpret_cast<const T *>(a.logits) + ((size_t)b * (a.k + 1) + r) * a.V;
    d.q = (r < kb) ? a.q + ((size_t)b * a.k + r) * a.V : nullptr;
    d.m = ms.m;
    d.inv_s = 1.0f / ms.s;
    d.c = scale_of(a);
    d.cut = a.filtered ? a.row_cut[b * (a.k + 1) + r] : -INFINITY;
    return d;
}

// two block sums for thread 0: warp shuffles, one barrier, warp 0 finishes
__device__ __forceinline__ void block_sum2_to0(float &a, float &b, float *s_f)
{
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) {
        a += __shfl_xor_sync(0xFFFFFFFFu, a, k);
        b += __shfl_xor_sync(0xFFFFFFFFu, b, k);
    }
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) {
        s_f[w] = a;
        s_f[kThreads / 32 + w] = b;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        a = (l < kThreads / 32) ? s_f[l] : 0.0f;
        b = (l < kThreads / 32) ? s_f[kThreads / 32 + l] : 0.0f;
#pragma unroll
        for (int k = 16; k > 0; k >>= 1) {
            a += __shfl_xor_sync(0xFFFFFFFFu, a, k);
            b += __shfl_xor_sync(0xFFFFFFFFu, b, k);
        }
    }
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

// sums of max(0, p - q) and of p over elements [lo, hi) of the drawn row:
// 16-byte loads of the logits and of q where both rows allow it
template <typename T>
__device__ void draw_chunk_sums(const DrawRow<T> &dr, bool residual, int lo, int hi, float &sr, float &sp)
{
    constexpr int VEC = Storage<T>::kVec;
    const bool vec_ok = ((reinterpret_cast<uintptr_t>(dr.x + lo) & 15) == 0) &&
                        (!residual || (reinterpret_cast<uintptr_t>(dr.q + lo) & 15) == 0);
    int v0 = lo;
    if (vec_ok) {
        constexpr int UNROLL = 4;
        constexpr int QV = VEC / 4;  // 16-byte q vectors per logits vector
        const int nvec = (hi - lo) / VEC;
        for (int i = threadIdx.x; i < nvec; i += UNROLL * kThreads) {
            uint4 r[UNROLL], qq[UNROLL][QV];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int vi = i + u * kThreads;
                if (vi < nvec) {
                    r[u] = ld_stream16(dr.x + lo + (size_t)vi * VEC);
                    if (residual) {
#pragma unroll
                        for (int h = 0; h < QV; ++h)
                            qq[u][h] = ld_stream16(dr.q + lo + (size_t)vi * VEC + 4 * h);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int vi = i + u * kThreads;
                if (vi < nvec) {
                    float f[VEC];
                    Storage<T>::unpack(r[u], f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const float p = dr.p(f[e]);
                        sp += p;
                        if (residual) {
                            const uint4 &w4 = qq[u][e / 4];
                            const uint32_t qb = (e & 3) == 0 ? w4.x : (e & 3) == 1 ? w4.y : (e & 3) == 2 ? w4.z : w4.w;
                            sr += fmaxf(p - __uint_as_float(qb), 0.0f);
                        }
                    }
                }
            }
        }
        v0 = lo + nvec * VEC;
    }
    for (int v = v0 + threadIdx.x; v < hi; v += kThreads) {
        const float p = dr.pv(v);
        sp += p;
        if (residual)
            sr += fmaxf(p - __ldg(dr.q + v), 0.0f);
    }
}

constexpr int kSeg = kDrawChunk / kThreads;  // contiguous elements per thread in the final scan
constexpr int kPadded = kDrawChunk + kDrawChunk / 32;

template <typename T>
__global__ void __launch_bounds__(kThreads) verify_draw_kernel(VerifyArgs a)
{
    __shared__ float s_w[kPadded];  // weights of the chosen chunk, one pad word per 32
    __shared__ float s_f[2 * kThreads / 32];
    __shared__ double s_d[kThreads / 32];
    __shared__ int s_flag, s_pick, s_lastpos, s_chunk, s_use_res;
    __shared__ double s_base, s_target;
    dep_wait();  // launched programmatically: the stats grid's results are complete
    const int Cd = draw_chunks(a.V);
    const int b = blockIdx.x / Cd, c = blockIdx.x % Cd;
    const int r = a.draw_row[b];
    if (r < 0)
        return;
    int kb = a.draft_len ? a.draft_len[b] : a.k;
    kb = kb < 0 ? 0 : (kb > a.k ? a.k : kb);
    const bool residual = r < kb;
    const DrawRow<T> dr = draw_row_of<T>(a, b, r, kb);
    float *rpart = a.rpart;
    int *res_cnt = a.res_cnt;
    double *rtot = a.rtot;

    // one pass over this chunk: sum of the residual and sum of p
    const int lo = c * kDrawChunk, hi = min(a.V, lo + kDrawChunk);
    float sr = 0.0f, sp = 0.0f;
    draw_chunk_sums<T>(dr, residual, lo, hi, sr, sp);
    block_sum2_to0(sr, sp, s_f);
    if (threadIdx.x == 0) {
        rpart[((size_t)b * Cd + c) * 2 + 0] = sr;
        rpart[((size_t)b * Cd + c) * 2 + 1] = sp;
        __threadfence();
        s_flag = (atomicAdd(res_cnt + b, 1) == Cd - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!s_flag)
        return;
    __threadfence();

    // last CTA of the row: choose the weights, find the chunk, scan it.
    // Warp 0 loads the chunk sums in parallel (32 chunks per pass) and scans
    // them in fp64 with shuffles; a ballot finds the chunk holding u * total.
    if (threadIdx.x < 32) {
        const int l = threadIdx.x;
        double R = 0.0, P = 0.0;
        for (int i0 = 0; i0 < Cd; i0 += 32) {
            const int i = i0 + l;
            if (i < Cd) {
                R += (double)rpart[((size_t)b * Cd + i) * 2 + 0];
                P += (double)rpart[((size_t)b * Cd + i) * 2 + 1];
            }
        }
#pragma unroll
        for (int k = 16; k > 0; k >>= 1) {
            R += __shfl_xor_sync(0xFFFFFFFFu, R, k);
            P += __shfl_xor_sync(0xFFFFFFFFu, P, k);
        }
        const bool use_res = residual && R > 0.0;
        const int sel = use_res ? 0 : 1;
        const double W = use_res ? R : P;
        const double target = (double)a.u[(size_t)b * (a.k + 1) + a.k] * W;
        double before = 0.0;  // sum of the chunks of earlier passes
        int cs = -1, lastpos = -1;
        double cs_base = 0.0;
        for (int i0 = 0; i0 < Cd && cs < 0; i0 += 32) {
            const int i = i0 + l;
            const double pc = (i < Cd) ? (double)rpart[((size_t)b * Cd + i) * 2 + sel] : 0.0;
            double incl = pc;
#pragma unroll
            for (int k = 1; k < 32; k <<= 1) {
                const double o = __shfl_up_sync(0xFFFFFFFFu, incl, k);
                if (l >= k)
                    incl += o;
            }
            const unsigned pos = __ballot_sync(0xFFFFFFFFu, pc > 0.0);
            if (pos)
                lastpos = i0 + 31 - __clz((int)pos);
            const unsigned hit = __ballot_sync(0xFFFFFFFFu, i < Cd && before + incl > target);
            if (hit) {
                const int f = __ffs(hit) - 1;
                cs = i0 + f;
                cs_base = before + __shfl_sync(0xFFFFFFFFu, incl - pc, f);
            }
            before += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (l == 0) {
            if (cs < 0) {  // rounding left u * W at or past the total: last positive chunk
                cs = lastpos >= 0 ? lastpos : Cd - 1;
                cs_base = -1.0;  // take the last positive index of that chunk
            }
            s_base = cs_base;
            s_chunk = cs;
            s_use_res = use_res ? 1 : 0;
            s_target = target;
            s_pick = 0x7FFFFFFF;
            s_lastpos = -1;
            rtot[b] = use_res ? W : -W;  // sign records the mode for the residual writer
            if (residual && !use_res && a.flags)
                a.flags[b] |= SPEC_FLAG_ZERO_RESIDUAL;
            res_cnt[b] = 0;
        }
    }
    __syncthreads();
    const bool use_res = s_use_res != 0;
    const double target = s_target, base = s_base;
    const int clo = s_chunk * kDrawChunk, n = min(a.V, clo + kDrawChunk) - clo;
    // stage the chunk's weights: every thread issues all of its 16-byte loads
    // (logits and q) before using any, then writes weights to shared memory
    {
        constexpr int VEC = Storage<T>::kVec;
        constexpr int NV = kDrawChunk / VEC / kThreads;  // vectors per thread
        const bool vec_ok = (n == kDrawChunk) && ((reinterpret_cast<uintptr_t>(dr.x + clo) & 15) == 0) &&
                            (!use_res || (reinterpret_cast<uintptr_t>(dr.q + clo) & 15) == 0);
        if (vec_ok) {
            constexpr int NH = NV / 2;  // two halves keep the register count down
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
            uint4 xr[NH], qr[NH][VEC / 4];
#pragma unroll
            for (int v = 0; v < NH; ++v) {
                const int i = (threadIdx.x + (half * NH + v) * kThreads) * VEC;
                xr[v] = ld_stream16(dr.x + clo + i);
                if (use_res) {
#pragma unroll
                    for (int h = 0; h < VEC / 4; ++h)
                        qr[v][h] = ld_stream16(dr.q + clo + i + 4 * h);
                }
            }
#pragma unroll
            for (int v = 0; v < NH; ++v) {
                const int i = (threadIdx.x + (half * NH + v) * kThreads) * VEC;
                float f[VEC];
                Storage<T>::unpack(xr[v], f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float p = dr.p(f[e]);
                    float wv = p;
                    if (use_res) {
                        const uint4 &w4 = qr[v][e / 4];
                        const uint32_t qb = (e & 3) == 0 ? w4.x : (e & 3) == 1 ? w4.y : (e & 3) == 2 ? w4.z : w4.w;
                        wv = fmaxf(p - __uint_as_float(qb), 0.0f);
                    }
                    s_w[(i + e) + ((i + e) >> 5)] = wv;
                }
            }
            }
        } else {
            for (int i = threadIdx.x; i < n; i += kThreads)
                s_w[i + (i >> 5)] = dr.w(clo + i, use_res);
        }
    }
    __syncthreads();
    const int slo = threadIdx.x * kSeg, shi = min(n, slo + kSeg);
    float seg = 0.0f;
    int seg_last = -1;
    for (int i = slo; i < shi; ++i) {
        const float wv = s_w[i + (i >> 5)];
        seg += wv;
        if (wv > 0.0f)
            seg_last = clo + i;
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
    // the segment holding the target: its start offset in fp64, the walk
    // within it in fp32 against the remaining distance
    const double seg_start = base + warp_off + incl - (double)seg;
    if (base >= 0.0 && seg_start + (double)seg > target) {
        const float rem = (float)(target - seg_start);
        float run = 0.0f;
        for (int i = slo; i < shi; ++i) {
            run += s_w[i + (i >> 5)];
            if (run > rem) {
                atomicMin(&s_pick, clo + i);
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
            tok = s_lastpos >= 0 ? s_lastpos : clo + n - 1;
        a.out_tokens[(size_t)b * (a.k + 1) + r] = tok;
    }
}

// optional: the normalised distribution of each sequence's draw
template <typename T>
__global__ void __launch_bounds__(kThreads) verify_residual_kernel(VerifyArgs a)
{
    const int Cd = draw_chunks(a.V);
    const int b = blockIdx.x / Cd, c = blockIdx.x % Cd;
    const int r = a.draw_row[b];
    if (r < 0)
        return;
    int kb = a.draft_len ? a.draft_len[b] : a.k;
    kb = kb < 0 ? 0 : (kb > a.k ? a.k : kb);
    const DrawRow<T> dr = draw_row_of<T>(a, b, r, kb);
    const double W = a.rtot[b];
    const bool use_res = W > 0.0 && r < kb;  // the bonus row has no draft row
    const float inv = (float)(1.0 / (use_res ? W : -W));
    const int lo = c * kDrawChunk, hi = min(a.V, lo + kDrawChunk);
    float *out = a.out_residual + (size_t)b * a.V;
    for (int v = lo + threadIdx.x; v < hi; v += kThreads)
        out[v] = dr.w(v, use_res) * inv;
}

template <typename T>
static cudaError_t launch_sample_t(const VerifyArgs &args, cudaStream_t st)
{
    VerifyArgs a = args;
    resolve_verify_args(a);
    const unsigned g2 = (unsigned)(a.B * draw_chunks(a.V));
    if (a.filtered) {
        const cudaError_t ef = launch_filter_rows<T>(a, st);
        if (ef != cudaSuccess)
            return ef;
    } else {
        verify_stats_kernel<T><<<a.B * (a.k + 1) * a.C, kThreads, 0, st>>>(a);
    }
    // the draw kernel becomes resident while the stats kernel drains and
    // waits for it on the device (griddepcontrol.wait)
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g2);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, verify_draw_kernel<T>, a);
    if (e != cudaSuccess)
        return e;
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
