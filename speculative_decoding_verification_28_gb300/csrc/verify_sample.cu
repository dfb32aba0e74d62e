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
// Four kernels, stream-ordered:
//   stats  : per (b, j, chunk) max / sum of 2^(x c - m) (lazy rows, as in the
//            greedy kernel; 8 loads in flight per thread, one packed maximum
//            and one rescale test per batch of vectors, the last batch padded
//            with -inf, two elements per paired fp32 instruction; 128-thread
//            CTAs when a chunk is short); the row's last CTA gathers x[y] and
//            q[y] and runs the ratio test; the sequence's last row runs the
//            first-stop ballot and decides which row (if any) is drawn from.
//            With top-k / top-p the filter kernel of verify_filter.cuh takes
//            this place (one CTA per row, and the row's cut goes to the draw
//            kernels);
//   sums   : per (b, 1024-element segment) of the drawn row, one warp sums
//            the residual and p in a vectorised pass;
//   pick   : one warp per drawing sequence picks the mode, finds the segment
//            holding u * total from the segment sums, loads that segment
//            into registers and scans it for the inverse-CDF index: prefix
//            sums over segments and lanes in exact 64-bit fixed point, the
//            walk within a lane in fp32.  Sums and pick are launched
//            programmatically and wait for the kernel before them on the
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
// -inf in every element of a 16-byte vector (padding past a chunk's end)
template <typename T>
__device__ __forceinline__ uint4 neg_inf_vec();
template <>
__device__ __forceinline__ uint4 neg_inf_vec<float>()
{
    return make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
}
template <>
__device__ __forceinline__ uint4 neg_inf_vec<__nv_bfloat16>()
{
    return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
}
template <>
__device__ __forceinline__ uint4 neg_inf_vec<__half>()
{
    return make_uint4(0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u);
}

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
    // chain.  What remains after the full batches is one guarded batch.
    float mt = m;  // the head element, if any, is already in (m, s)
    // partial sums (0, 1) and (2, 3) as pairs: element e of a vector goes to
    // partial sum e mod 4; paired fp32 instructions (FFMA2 / FADD2 / FMUL2,
    // each lane rounded to nearest) do two elements at a time
    float2 sa[2] = {make_float2(s, 0.0f), make_float2(0.0f, 0.0f)};
    int base = 0;
    bool dropped = false;
    int enc = 0;  // the stop word, read with the previous full batch
    // one batch of NB vectors per thread starting at vector `base`; guarded
    // (the last, partial batch): vectors past the chunk's end read as -inf
    auto batch = [&](auto nb, auto guard) {
        constexpr int NB = decltype(nb)::value;
        constexpr bool kGuard = decltype(guard)::value;
        uint4 r[NB];
#pragma unroll
        for (int u = 0; u < NB; ++u) {
            const int vi = base + t + u * NT;
            r[u] = (!kGuard || vi < cs.nvec) ? ld_stream16(body + (size_t)vi * VEC) : neg_inf_vec<T>();
        }
        if (!kGuard)
            enc = probe.load();  // in flight with the batch
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
            sa[0] = __fmul2_rn(sa[0], make_float2(scale, scale));
            sa[1] = __fmul2_rn(sa[1], make_float2(scale, scale));
            m = vm;
        }
        if (m > -INFINITY) {
            const float2 c2 = make_float2(c, c), nm2 = make_float2(-m, -m);
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                float f[VEC];
                Storage<T>::unpack(r[u], f);
#pragma unroll
                for (int e = 0; e < VEC; e += 2) {
                    const float2 z = __ffma2_rn(make_float2(f[e], f[e + 1]), c2, nm2);
                    sa[(e >> 1) & 1] = __fadd2_rn(sa[(e >> 1) & 1], make_float2(exp2_sfu(z.x), exp2_sfu(z.y)));
                }
            }
        }
    };
    // full batches of 8 vectors (128 bytes in flight per thread)
    for (; base + 8 * NT <= cs.nvec; base += 8 * NT) {  // warp-uniform trip count
        if (base > 0 && probe.stopped(enc)) {
            dropped = true;
            break;
        }
        batch(std::integral_constant<int, 8>(), std::false_type());
    }
    // the rest (fewer than 8 vectors per thread): one guarded batch, with the
    // same single packed maximum and lazy rescale test
    if (!dropped && base < cs.nvec && (base == 0 || !probe.stopped(enc)))
        batch(std::integral_constant<int, 8>(), std::true_type());
    s = (sa[0].x + sa[0].y) + (sa[1].x + sa[1].y);
    if (m > -INFINITY && mt > m) {  // bring the sum to the exact maximum
        s *= exp2f(m - mt);
        m = mt;
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

// NT threads per CTA: 128 when a unit would give 256 threads at most one
// batch of 8 vectors each (twice the CTAs per SM, two batches per thread),
// else kThreads
template <typename T, int NT>
__global__ void __launch_bounds__(NT) verify_stats_kernel(VerifyArgs a)
{
    __shared__ float s_f[3 * NT / 32];
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
        chunk_softmax_stats<T, false, NT>(row, lo, hi, c, m, s, bad, s_f, StopProbe{a.stop_enc, u.b, u.j}, nullptr);
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

// Segments: the drawn row is cut into segments of kDrawSeg elements; a warp
// of the sums kernel sums one segment, and the pick scans one segment.
constexpr int kSegPerLane = kDrawSeg / 32;  // contiguous elements per lane in the pick
static_assert(kDrawChunk == kDrawSeg * (kThreads / 32), "a sums CTA covers one segment per warp");

__device__ __forceinline__ bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// q bits of element e (0 .. VEC-1) of a 16-byte logits vector, from its VEC/4 q vectors
__device__ __forceinline__ float q_elem(const uint4 *qq, int e)
{
    const uint4 &w4 = qq[e / 4];
    const uint32_t qb = (e & 3) == 0 ? w4.x : (e & 3) == 1 ? w4.y : (e & 3) == 2 ? w4.z : w4.w;
    return __uint_as_float(qb);
}

// One warp: sums of max(0, p - q) and of p over elements [lo, hi) of the
// drawn row, for every lane.  A full aligned segment is read with 16-byte
// loads, lane l taking vectors l, l + 32, ... (all of a batch in flight).
template <typename T>
__device__ void draw_segment_sums(const DrawRow<T> &dr, bool residual, int lo, int hi, float &sr, float &sp)
{
    constexpr int VEC = Storage<T>::kVec;
    constexpr int QV = VEC / 4;                 // 16-byte q vectors per logits vector
    constexpr int NV = kDrawSeg / VEC / 32;     // logits vectors per lane: 4 (16-bit types) or 8 (fp32)
    constexpr int NB = NV > 4 ? 4 : NV;         // vectors per batch
    const int l = threadIdx.x & 31;
    sr = 0.0f;
    sp = 0.0f;
    if (hi - lo == kDrawSeg && aligned16(dr.x + lo) && (!residual || aligned16(dr.q + lo))) {
        // two elements per paired fp32 instruction (FFMA2 / FMUL2 / FADD2):
        // p as DrawRow::p computes it, sums in two lanes each
        const float2 c2 = make_float2(dr.c, dr.c), nm2 = make_float2(-dr.m, -dr.m);
        const float2 is2 = make_float2(dr.inv_s, dr.inv_s), neg1 = make_float2(-1.0f, -1.0f);
        float2 sp2 = make_float2(0.0f, 0.0f), sr2 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int b0 = 0; b0 < NV; b0 += NB) {
            uint4 r[NB], qq[NB][QV];
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                const int vi = (b0 + u) * 32 + l;
                r[u] = ld_stream16(dr.x + lo + (size_t)vi * VEC);
                if (residual) {
#pragma unroll
                    for (int h = 0; h < QV; ++h)
                        qq[u][h] = ld_stream16(dr.q + lo + (size_t)vi * VEC + 4 * h);
                }
            }
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                float f[VEC];
                Storage<T>::unpack(r[u], f);
#pragma unroll
                for (int e = 0; e < VEC; e += 2) {
                    const float2 z = __ffma2_rn(make_float2(f[e], f[e + 1]), c2, nm2);
                    float2 p = __fmul2_rn(make_float2(exp2_sfu(z.x), exp2_sfu(z.y)), is2);
                    p.x = f[e] >= dr.cut ? p.x : 0.0f;
                    p.y = f[e + 1] >= dr.cut ? p.y : 0.0f;
                    sp2 = __fadd2_rn(sp2, p);
                    if (residual) {
                        const float2 d = __ffma2_rn(make_float2(q_elem(qq[u], e), q_elem(qq[u], e + 1)), neg1, p);
                        sr2 = __fadd2_rn(sr2, make_float2(fmaxf(d.x, 0.0f), fmaxf(d.y, 0.0f)));
                    }
                }
            }
        }
        sp = sp2.x + sp2.y;
        sr = sr2.x + sr2.y;
    } else {
        for (int v = lo + l; v < hi; v += 32) {
            const float p = dr.pv(v);
            sp += p;
            if (residual)
                sr += fmaxf(p - __ldg(dr.q + v), 0.0f);
        }
    }
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) {
        sr += __shfl_xor_sync(0xFFFFFFFFu, sr, k);
        sp += __shfl_xor_sync(0xFFFFFFFFu, sp, k);
    }
}

// draw, pass 1: per (b, segment) of the drawn row, the sums of the residual
// and of p, one warp per segment.  Launched programmatically behind the
// statistics kernel; no barrier, no counter: a warp retires once its sums
// are out.
template <typename T>
__global__ void __launch_bounds__(kThreads) verify_draw_sums_kernel(VerifyArgs a)
{
    dep_wait();  // the statistics grid's results are complete
    const int Cd = draw_chunks(a.V), Ns = draw_segs(a.V);
    const int b = blockIdx.x / Cd, c = blockIdx.x % Cd;
    const int r = a.draw_row[b];
    if (r < 0)
        return;
    const int sg = c * (kThreads / 32) + (threadIdx.x >> 5);
    if (sg >= Ns)
        return;  // warps past the end of the row
    int kb = a.draft_len ? a.draft_len[b] : a.k;
    kb = kb < 0 ? 0 : (kb > a.k ? a.k : kb);
    const bool residual = r < kb;
    const DrawRow<T> dr = draw_row_of<T>(a, b, r, kb);
    const int lo = sg * kDrawSeg, hi = min(a.V, lo + kDrawSeg);
    float sr, sp;
    draw_segment_sums<T>(dr, residual, lo, hi, sr, sp);
    if ((threadIdx.x & 31) == 0) {
        a.rpart[((size_t)b * Ns + sg) * 2 + 0] = sr;
        a.rpart[((size_t)b * Ns + sg) * 2 + 1] = sp;
    }
}

// x * 2^60 as an unsigned integer, truncated (the fixed point of the pick:
// weights are probabilities, below 2).  0 for x <= 0 and for x below 2^-60;
// x >= 2, inf and NaN (rows already flagged non-finite) saturate at 2^62.
// Integer operations only: FP64 is slow on this part.
__device__ __forceinline__ unsigned long long fixed60(float x)
{
    const uint32_t bits = __float_as_uint(x);
    if ((int32_t)bits <= 0)
        return 0ull;                               // +-0, negatives, negative NaN
    const int sh = (int)(bits >> 23) - 127 + 37;  // x = mant * 2^(e - 23), x * 2^60 = mant * 2^(e + 37)
    const unsigned long long mant = (bits & 0x7FFFFFu) | 0x800000u;
    if (sh >= 38)
        return 1ull << 62;
    if (sh >= 0)
        return mant << sh;
    return sh <= -24 ? 0ull : (mant >> -sh);
}

constexpr int kPickSegs = 8;   // segment sums per lane and block: a block covers 256 segments (V <= 262144)
constexpr int kPickWarps = 2;  // sequences per CTA of the pick kernel

// draw, pass 2: one warp per drawing sequence (kPickWarps per CTA), launched
// programmatically behind the sums.  The weights are the residual when it has
// positive mass, else p (the bonus row always draws from p).  Prefix sums
// over segments and lanes are exact unsigned 64-bit fixed point (fixed60), so
// the target u * total (u * 2^64 times the total, high half) lies in exactly
// one segment.
// Segment sums are read a block of 256 at a time, lane l holding segments
// 8 l .. 8 l + 7 of the block, in the same round as the sequence's draw row,
// budget and uniform; a prefix over the lanes finds the lane, the lane finds
// the segment.  That segment is loaded with lane l holding its elements
// 32 l .. 32 l + 31 in registers; the lanes' fp32 sums, in fixed point, give
// an exact prefix that finds the lane, and the lane walks its 32 weights in
// fp32 against the remaining distance.  The pick is the first index whose
// cumulative weight exceeds the target.  The segment sums come from the sums
// kernel's fp32 arithmetic and the lane weights are re-summed here, so at
// the last few ulps the two can disagree: if the lane's walk ends short of
// the target, the lane's last index of positive weight is taken, and if no
// lane of the segment holds the target, the segment's.
template <typename T>
__global__ void __launch_bounds__(kPickWarps * 32) verify_draw_pick_kernel(VerifyArgs a)
{
    typedef unsigned long long u64;
    dep_wait();  // the sums grid's results are complete
    const int l = threadIdx.x & 31;
    const int b = blockIdx.x * kPickWarps + (threadIdx.x >> 5);
    if (b >= a.B)
        return;
    const int Ns = draw_segs(a.V);
    const float *rs = a.rpart + (size_t)b * Ns * 2;
    // one round: the draw row, the budget, the uniform, the first block of segment sums
    const int r = a.draw_row[b];
    int kb = a.draft_len ? a.draft_len[b] : a.k;
    const float uu = a.u[(size_t)b * (a.k + 1) + a.k];
    float bR[kPickSegs], bP[kPickSegs];
    auto load_block = [&](int s0) {
#pragma unroll
        for (int j = 0; j < kPickSegs; ++j) {
            const int i = s0 + l * kPickSegs + j;
            bR[j] = i < Ns ? __ldcg(rs + 2 * i) : 0.0f;
            bP[j] = i < Ns ? __ldcg(rs + 2 * i + 1) : 0.0f;
        }
    };
    load_block(0);
    if (r < 0)
        return;
    kb = kb < 0 ? 0 : (kb > a.k ? a.k : kb);
    const bool residual = r < kb;
    const DrawRow<T> dr = draw_row_of<T>(a, b, r, kb);
    constexpr int kBlock = 32 * kPickSegs;

    // totals
    u64 R = 0, P = 0;
    for (int s0 = 0; s0 < Ns; s0 += kBlock) {
        if (s0 > 0)
            load_block(s0);
#pragma unroll
        for (int j = 0; j < kPickSegs; ++j) {
            R += fixed60(bR[j]);
            P += fixed60(bP[j]);
        }
    }
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) {
        R += __shfl_xor_sync(0xFFFFFFFFu, R, k);
        P += __shfl_xor_sync(0xFFFFFFFFu, P, k);
    }
    const bool use_res = residual && R > 0;
    const u64 W = use_res ? R : P;
    const u64 target = __umul64hi(fixed60(uu) << 4, W);  // u in [0, 1): u * 2^64 fits; target < W when W > 0
    if (l == 0) {
        const double Wd = (double)W * 0x1p-60;
        a.rtot[b] = use_res ? Wd : -Wd;  // sign records the mode for the residual writer
        if (residual && !use_res && a.flags)
            a.flags[b] |= SPEC_FLAG_ZERO_RESIDUAL;
    }

    // the segment holding the target
    u64 before = 0, cs_base = 0;
    int cs = -1;
    for (int s0 = 0; s0 < Ns && cs < 0 && W > 0; s0 += kBlock) {
        if (s0 > 0 || Ns > kBlock)
            load_block(s0);  // block 0 is still in registers when it is the only one
        u64 f[kPickSegs], tot = 0;
#pragma unroll
        for (int j = 0; j < kPickSegs; ++j) {
            f[j] = fixed60(use_res ? bR[j] : bP[j]);
            tot += f[j];
        }
        u64 incl = tot;
#pragma unroll
        for (int k = 1; k < 32; k <<= 1) {
            const u64 o = __shfl_up_sync(0xFFFFFFFFu, incl, k);
            if (l >= k)
                incl += o;
        }
        const u64 lo_l = before + incl - tot;
        int my = -1;
        u64 my_base = 0;
        if (lo_l <= target && target - lo_l < tot) {
            u64 run = lo_l;
#pragma unroll
            for (int j = 0; j < kPickSegs; ++j) {
                if (my < 0 && target - run < f[j]) {
                    my = s0 + l * kPickSegs + j;
                    my_base = run;
                }
                run += f[j];
            }
        }
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, my >= 0);
        if (hit) {
            const int h = __ffs(hit) - 1;
            cs = __shfl_sync(0xFFFFFFFFu, my, h);
            cs_base = __shfl_sync(0xFFFFFFFFu, my_base, h);
        }
        before += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    const bool take_last = cs < 0;  // no positive weight at all (W = 0)
    if (take_last)
        cs = Ns - 1;

    // the segment's weights, 32 contiguous ones per lane
    const int slo = cs * kDrawSeg, shi = min(a.V, slo + kDrawSeg);
    const int e0 = slo + l * kSegPerLane;
    float w[kSegPerLane];
    constexpr int VEC = Storage<T>::kVec;
    if (shi - slo == kDrawSeg && aligned16(dr.x + slo) && (!use_res || aligned16(dr.q + slo))) {
        uint4 xr[kSegPerLane / VEC], qr[kSegPerLane / 4];
#pragma unroll
        for (int v = 0; v < kSegPerLane / VEC; ++v)
            xr[v] = ld_stream16(dr.x + e0 + v * VEC);
        if (use_res) {
#pragma unroll
            for (int v = 0; v < kSegPerLane / 4; ++v)
                qr[v] = ld_stream16(dr.q + e0 + v * 4);
        }
#pragma unroll
        for (int v = 0; v < kSegPerLane / VEC; ++v) {
            float f[VEC];
            Storage<T>::unpack(xr[v], f);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const float p = dr.p(f[e]);
                w[v * VEC + e] = use_res ? fmaxf(p - q_elem(qr + (v * VEC) / 4, e), 0.0f) : p;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < kSegPerLane; ++i)
            w[i] = (e0 + i < shi) ? dr.w(e0 + i, use_res) : 0.0f;
    }
    // lane sums in fp32 (four partial sums), their prefix exact in fixed point
    float ls[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    int lane_last = -1;
#pragma unroll
    for (int i = 0; i < kSegPerLane; ++i) {
        ls[i & 3] += w[i];
        if (w[i] > 0.0f)
            lane_last = e0 + i;
    }
    const u64 lane_sum = fixed60((ls[0] + ls[1]) + (ls[2] + ls[3]));
    u64 incl = lane_sum;
#pragma unroll
    for (int k = 1; k < 32; k <<= 1) {
        const u64 o = __shfl_up_sync(0xFFFFFFFFu, incl, k);
        if (l >= k)
            incl += o;
    }
    const u64 start = cs_base + incl - lane_sum;
    int cand = 0x7FFFFFFF;
    if (!take_last && start <= target && target - start < lane_sum) {
        // the lane's walk in fp32 against the remaining distance
        const float rem = (float)(target - start) * 0x1p-60f;
        float run = 0.0f;
#pragma unroll
        for (int i = 0; i < kSegPerLane; ++i) {
            run += w[i];
            if (cand == 0x7FFFFFFF && run > rem && w[i] > 0.0f)
                cand = e0 + i;
        }
        if (cand == 0x7FFFFFFF)
            cand = lane_last;  // rounding: the lane's own last positive weight
    }
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) {
        cand = min(cand, __shfl_xor_sync(0xFFFFFFFFu, cand, k));
        lane_last = max(lane_last, __shfl_xor_sync(0xFFFFFFFFu, lane_last, k));
    }
    if (l == 0) {
        const int tok = cand != 0x7FFFFFFF ? cand : (lane_last >= 0 ? lane_last : shi - 1);
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
        const long long vec_per_unit = (long long)a.chunk * (long long)sizeof(T) / 16;
        if (vec_per_unit <= 8LL * kThreads)
            verify_stats_kernel<T, 128><<<a.B * (a.k + 1) * a.C, 128, 0, st>>>(a);
        else
            verify_stats_kernel<T, kThreads><<<a.B * (a.k + 1) * a.C, kThreads, 0, st>>>(a);
    }
    // the two draw kernels become resident while the kernel before each
    // drains, and wait for it on the device (griddepcontrol.wait)
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g2);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, verify_draw_sums_kernel<T>, a);
    if (e != cudaSuccess)
        return e;
    cfg.gridDim = dim3((unsigned)((a.B + kPickWarps - 1) / kPickWarps));
    cfg.blockDim = dim3(kPickWarps * 32);
    e = cudaLaunchKernelEx(&cfg, verify_draw_pick_kernel<T>, a);
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
