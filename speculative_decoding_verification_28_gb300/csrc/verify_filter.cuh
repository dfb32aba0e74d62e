// verify_filter.cuh -- top-k / top-p on the target rows of stochastic
// verification (included by verify_sample.cu, which owns the launch).
//
// The ratio test, the residual and the bonus use the distribution the target
// samples from ("Chapter 10 Speculative Decoding (Code Walkthrough)", §5.1:
// with temperature, top-k or top-p the processed probabilities are kept;
// "Speculative decoding: proposals and verified output", "The mechanism"
// step 1).  Definitions (temperature, then top-k, then top-p):
//   top-k, 0 < k < V: keep x >= the k-th largest logit (ties kept);
//   top-p, top_p < 1: among those, keep v iff the mass of strictly larger
//     logits is below top_p times their total (ties kept; the largest value
//     always kept);
//   p = softmax(x / T) renormalised over the kept tokens.
// The top-p boundary is decided on exact integer sums of fixed-point weights
// Q = floor(2^40 * 2^t), t = (x - x_max) * log2(e) / T, computed to about
// 2e-9 relative (DecScale, dec_weight below): x - x_max exactly (TwoSum),
// t as a float-float product with log2(e)/T held as a float pair, 2^t as
// 2^n * 2^(k/64) * 2^r (Tang's table-driven method: 64 float-float table
// entries, |r| <= 1/128 plus the low part of t, 2^r - 1 from its degree-4
// Taylor polynomial), and the floor taken from the float pair in integers
// (within one unit of 2^-40).  The kept set then differs from the one the
// real masses give only where the true mass above a value lies within ~4e-9
// of top_p times the total (plus V * 2^-39 for the floors, in units of the
// top mass).  Integer sums do not
// depend on the order of summation, so the decision is reproducible; the
// kept token probabilities use the same ex2-based softmax as the unfiltered
// path.
//
// Two kernels, one CTA per target row each (rows j-major, skipped once an
// earlier stop of the sequence is known, as in the statistics kernel).
// 16-bit rows of at least kTabMinV logits take the table form further down
// (a count per bit pattern, one weight per distinct value).  Every other row
// takes the radix form: 1024, 512 or 256 threads by the number of rows
// (launch_filter_rows).  Its pass 1 reads the row from
// HBM: its maximum when the row is filtered (the kept sum then comes from the
// Q masses), else the softmax statistics.  The cuts are radix selections on
// an order-preserving 32-bit key of the logit, 11-bit digits (two levels for
// 16-bit logits, whose keys carry at most 22 significant bits; three for
// fp32): each level is one more pass over the row (now in L2) building
// per-digit counts and Q masses in shared memory (32-bit atomics on three
// parts of each mass), then a block scan from the top digit finds the digit
// holding the k-th largest key (counts) or the top-p boundary (masses).
// Roofline: HBM reads V * sizeof(T) per needed row; the radix form's later
// passes are L2 reads, a fixed-point weight per logit and shared-memory
// atomics, which make it instruction-bound; the table form is bound by its
// one shared atomic per logit and by the selection's latency.
#pragma once

#include <type_traits>

#include "sample_final.cuh"

namespace spec {

constexpr int kFBins = 2048;

// Counts and Q masses per digit.  A mass is kept as three 32-bit parts
// (Q = lo + mid 2^14 + hi 2^28): 32-bit shared-memory atomics are native,
// 64-bit adds are not, and the parts' sums stay exact for rows of at most
// 2^18 logits.
struct FilterHist {
    unsigned int cnt[kFBins];
    unsigned int mlo[kFBins], mmid[kFBins], mhi[kFBins];
    __device__ unsigned long long mass(int i) const
    {
        return (unsigned long long)mlo[i] + ((unsigned long long)mmid[i] << 14) +
               ((unsigned long long)mhi[i] << 28);
    }
};

struct FilterSel {
    int bin;                       // selected digit
    unsigned int cnt_above;        // count of the digits above it (this level)
    unsigned long long mass_above; // Q mass of the digits above it (this level)
    unsigned long long athr;       // ceil(top_p * total Q mass) (set at the first top-p level)
    int low_thread;                // last thread holding a non-empty digit
};

// order-preserving key of a logit; -0 and +0 share one key
__device__ __forceinline__ uint32_t order_key(float f)
{
    uint32_t u = __float_as_uint(f);
    if (f == 0.0f)
        u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// digit layout: level 0 = key bits 31..21, level 1 = bits 20..10, level 2 =
// bits 9..0
__device__ __forceinline__ int lvl_shift(int l) { return l == 0 ? 21 : (l == 1 ? 10 : 0); }
__device__ __forceinline__ int lvl_bins(int l) { return l == 2 ? 1024 : 2048; }
template <typename T>
struct KeyLevels {
    static constexpr int kLevels = 2;  // 16-bit logits: keys carry <= 22 significant bits
};
template <>
struct KeyLevels<float> {
    static constexpr int kLevels = 3;
};

// The decision scale log2(e) / T as a float pair (hi + lo, ~48 bits) and
// the shared-memory copy of the table 2^(k/64).
struct DecScale {
    float hi, lo;
    const float2 *tab;
};

// 2^(k/64), k = 0..63, as float pairs hi + lo: hi = 2^(k/64) rounded to fp32,
// lo = the rest rounded to fp32 (the table of Tang's table-driven exponential;
// the pair is within 2^-48 of 2^(k/64) relative)
static __constant__ float2 kExp2Tab64[64] = {
    {0x1p+0f, 0.0f}, {0x1.02c9a4p+0f, -0x1.887fap-28f}, {0x1.059b0ep+0f, -0x1.9d4f52p-25f}, {0x1.087452p+0f, -0x1.e2990ep-26f},
    {0x1.0b5586p+0f, 0x1.9f3122p-25f}, {0x1.0e3ec4p+0f, -0x1.a585ccp-25f}, {0x1.11301ep+0f, -0x1.fdb496p-25f}, {0x1.1429aap+0f, 0x1.d525bcp-25f},
    {0x1.172b84p+0f, -0x1.c15742p-27f}, {0x1.1a35bep+0f, 0x1.6df96ep-25f}, {0x1.1d4874p+0f, -0x1.d2e8cap-25f}, {0x1.2063b8p+0f, 0x1.0c519ap-25f},
    {0x1.2387a6p+0f, 0x1.ceac48p-25f}, {0x1.26b456p+0f, 0x1.789f38p-26f}, {0x1.29e9ep+0f, -0x1.5c0424p-25f}, {0x1.2d285ap+0f, 0x1.b900c2p-26f},
    {0x1.306fep+0f, 0x1.4636e2p-25f}, {0x1.33c08cp+0f, -0x1.b37d2p-25f}, {0x1.371a74p+0f, -0x1.18aac6p-25f}, {0x1.3a7db4p+0f, -0x1.634c02p-25f},
    {0x1.3dea64p+0f, 0x1.824684p-25f}, {0x1.4160a2p+0f, 0x1.f72e2ap-28f}, {0x1.44e086p+0f, 0x1.8624b4p-30f}, {0x1.486a2cp+0f, -0x1.47d866p-25f},
    {0x1.4bfdaep+0f, -0x1.593abcp-25f}, {0x1.4f9b28p+0f, -0x1.2c5a6cp-25f}, {0x1.5342b6p+0f, -0x1.2c561p-25f}, {0x1.56f474p+0f, -0x1.295b04p-25f},
    {0x1.5ab07ep+0f, -0x1.5bd5ecp-27f}, {0x1.5e76f2p+0f, -0x1.4a5bd6p-25f}, {0x1.6247ecp+0f, -0x1.f8b55p-25f}, {0x1.662388p+0f, 0x1.2a9112p-27f},
    {0x1.6a09e6p+0f, 0x1.9fcef4p-26f}, {0x1.6dfb24p+0f, -0x1.cd72e8p-27f}, {0x1.71f75ep+0f, 0x1.1d8beep-25f}, {0x1.75feb6p+0f, -0x1.37b306p-25f},
    {0x1.7a1148p+0f, -0x1.829fdp-25f}, {0x1.7e2f34p+0f, -0x1.261634p-25f}, {0x1.82589ap+0f, -0x1.accc7cp-26f}, {0x1.868d9ap+0f, -0x1.2edb44p-26f},
    {0x1.8ace54p+0f, 0x1.15506ep-27f}, {0x1.8f1aeap+0f, -0x1.baa232p-26f}, {0x1.93737cp+0f, -0x1.e64744p-25f}, {0x1.97d82ap+0f, -0x1.0d8d84p-31f},
    {0x1.9c4918p+0f, 0x1.51f848p-27f}, {0x1.a0c668p+0f, -0x1.2886a6p-26f}, {0x1.a5503cp+0f, -0x1.b83b54p-25f}, {0x1.a9e6b6p+0f, -0x1.50c048p-25f},
    {0x1.ae89fap+0f, -0x1.a94b14p-26f}, {0x1.b33a2cp+0f, -0x1.ec3a82p-26f}, {0x1.b7f77p+0f, -0x1.a09438p-25f}, {0x1.bcc1eap+0f, -0x1.f687c6p-25f},
    {0x1.c199bep+0f, -0x1.3d56b2p-27f}, {0x1.c67f12p+0f, 0x1.cafa2ap-25f}, {0x1.cb720ep+0f, -0x1.8837ccp-27f}, {0x1.d072d4p+0f, 0x1.40f13p-25f},
    {0x1.d5818ep+0f, -0x1.822dbcp-27f}, {0x1.da9e6p+0f, 0x1.ed9942p-27f}, {0x1.dfc974p+0f, -0x1.908c94p-25f}, {0x1.e502eep+0f, 0x1.e2cffep-26f},
    {0x1.ea4afap+0f, 0x1.52486cp-27f}, {0x1.efa1bep+0f, 0x1.cc2b44p-25f}, {0x1.f50766p+0f, -0x1.246ebp-26f}, {0x1.fa7c18p+0f, 0x1.9e90d8p-28f},
};

// all threads, before the first barrier of the kernel: the table into shared
// memory (the weight's lookup index differs across a warp's lanes)
__device__ __forceinline__ void dec_table_init(float2 *tab)
{
    for (int i = threadIdx.x; i < 64; i += blockDim.x)
        tab[i] = kExp2Tab64[i];
}

// 2^r - 1 for |r| <= 1/128 + 2^-18: Taylor coefficients (ln 2)^n / n!, n = 1..4
// (the degree-5 term is below 4e-14)
__device__ __forceinline__ float exp2m1_small(float r)
{
    float q = __fmaf_rn(0x1.3b2ab6p-7f, r, 0x1.c6b08ep-5f);
    q = __fmaf_rn(q, r, 0x1.ebfbe0p-3f);
    q = __fmaf_rn(q, r, 0x1.62e430p-1f);
    return __fmul_rn(q, r);
}

// The Q weight from p + tl (the high and low parts of t <= 0): 2^t = 2^n *
// 2^(k/64) * 2^r with j = rint(64 p), n = floor(j / 64), k = j mod 64 and
// r = (p - j/64) + tl (p - j/64 is exact); w = T_hi + w_lo with
// w_lo = T_hi * (2^r - 1) + T_lo (|w_lo| < 2^-6), and Q = floor(w * 2^(n+40))
// from Z = w * 2^47 in integers: T_hi in [1, 2) is its 24-bit significand
// m_h times 2^-23, and w_lo * 2^47 = A * 2^24 + B with A = floor(w_lo * 2^23)
// and 0 <= B < 2^24, both exact fp32 values converted by 32-bit conversions
// (B rounds only when |w_lo| < 2^-23, by less than one unit of 2^-47); then
// Q = Z >> (7 - n), within one unit of the exact floor.
__device__ __forceinline__ unsigned long long dec_q(float p, float tl, const float2 *tab)
{
    if (!(p >= -64.0f))  // 2^t < 2^-64: Q = 0 (also -inf and NaN)
        return 0ull;
    const float j = rintf(__fmul_rn(p, 64.0f));
    const float r = __fadd_rn(__fmaf_rn(j, -0.015625f, p), tl);
    const float q = exp2m1_small(r);
    const int ji = (int)j;
    const float2 T = tab[ji & 63];
    const float wl = __fmaf_rn(T.x, q, T.y);
    const float a = floorf(__fmul_rn(wl, 0x1p23f));
    const float b = __fmaf_rn(-a, 0x1p24f, __fmul_rn(wl, 0x1p47f));
    const uint32_t mh_a = ((__float_as_uint(T.x) & 0x7FFFFFu) | 0x800000u) + (uint32_t)(int)a;
    const unsigned long long Z = ((unsigned long long)mh_a << 24) + (unsigned long long)(uint32_t)b;
    const int sh = 7 - (ji >> 6);  // 7 .. 71
    return sh < 64 ? (Z >> sh) : 0ull;
}

// Q weight of a logit x against the row maximum xmax (x <= xmax)
__device__ __forceinline__ unsigned long long dec_weight(float x, float xmax, const DecScale &dw)
{
    // d = dh + dl = x - xmax exactly (TwoSum)
    const float dh = __fsub_rn(x, xmax);
    const float bb = __fsub_rn(dh, x);
    const float dl = __fadd_rn(__fsub_rn(x, __fsub_rn(dh, bb)), __fsub_rn(-xmax, bb));
    // t = p + tl = d * (hi + lo) to ~2^-46 relative
    const float p = __fmul_rn(dh, dw.hi);
    const float e = __fmaf_rn(dh, dw.hi, -p);  // the product's rounding error, exactly
    const float tl = __fmaf_rn(dh, dw.lo, __fmaf_rn(dl, dw.hi, e));
    return dec_q(p, tl, dw.tab);
}

// dec_weight of two logits, the float steps paired (FADD2 / FMUL2 / FFMA2;
// each lane rounded as the scalar form, so the results are dec_weight's)
__device__ __forceinline__ void dec_weight2(float x0, float x1, float xmax, const DecScale &dw,
                                            unsigned long long &q0, unsigned long long &q1)
{
    const float2 x = make_float2(x0, x1), nm = make_float2(-xmax, -xmax);
    const float2 dh = __fadd2_rn(x, nm);
    const float2 bb = __fadd2_rn(dh, make_float2(-x0, -x1));
    const float2 t1 = __fadd2_rn(dh, make_float2(-bb.x, -bb.y));
    const float2 dl = __fadd2_rn(__fadd2_rn(x, make_float2(-t1.x, -t1.y)), __fadd2_rn(nm, make_float2(-bb.x, -bb.y)));
    const float2 p = __fmul2_rn(dh, make_float2(dw.hi, dw.hi));
    const float2 e = __ffma2_rn(dh, make_float2(dw.hi, dw.hi), make_float2(-p.x, -p.y));
    const float2 tl = __ffma2_rn(dh, make_float2(dw.lo, dw.lo), __ffma2_rn(dl, make_float2(dw.hi, dw.hi), e));
    q0 = dec_q(p.x, tl.x, dw.tab);
    q1 = dec_q(p.y, tl.y, dw.tab);
}

// f(x) for every logit of the row: 16-byte vectors, scalar head and tail
template <typename T, int NT, typename F>
__device__ __forceinline__ void row_for_each(const T *row, int V, F &f)
{
    constexpr int VEC = Storage<T>::kVec;
    constexpr int UNROLL = 4;
    const ChunkSplit<T> cs(row, 0, V);
    const int t = threadIdx.x;
    for (int v = t; v < cs.head_end; v += NT)
        f(Storage<T>::at(row, v));
    const T *body = row + cs.head_end;
    for (int base = 0; base < cs.nvec; base += UNROLL * NT) {
        uint4 r[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int vi = base + t + u * NT;
            if (vi < cs.nvec)
                r[u] = ld_stream16(body + (size_t)vi * VEC);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int vi = base + t + u * NT;
            if (vi < cs.nvec) {
                float e[VEC];
                Storage<T>::unpack(r[u], e);
#pragma unroll
                for (int q = 0; q < VEC; ++q)
                    f(e[q]);
            }
        }
    }
    for (int v = cs.tail_beg + t; v < V; v += NT)
        f(Storage<T>::at(row, v));
}

// f2(x0, x1) for the element pairs of every 16-byte vector of the row, f(x)
// for the scalar head and tail
template <typename T, int NT, typename F, typename F2>
__device__ __forceinline__ void row_for_each_pair(const T *row, int V, F &f, F2 &f2)
{
    constexpr int VEC = Storage<T>::kVec;
    constexpr int UNROLL = 4;
    const ChunkSplit<T> cs(row, 0, V);
    const int t = threadIdx.x;
    for (int v = t; v < cs.head_end; v += NT)
        f(Storage<T>::at(row, v));
    const T *body = row + cs.head_end;
    for (int base = 0; base < cs.nvec; base += UNROLL * NT) {
        uint4 r[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int vi = base + t + u * NT;
            if (vi < cs.nvec)
                r[u] = ld_stream16(body + (size_t)vi * VEC);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int vi = base + t + u * NT;
            if (vi < cs.nvec) {
                float e[VEC];
                Storage<T>::unpack(r[u], e);
#pragma unroll
                for (int q = 0; q < VEC; q += 2)
                    f2(e[q], e[q + 1]);
            }
        }
    }
    for (int v = cs.tail_beg + t; v < V; v += NT)
        f(Storage<T>::at(row, v));
}

template <int NT>
__device__ __forceinline__ void hist_clear(FilterHist &h, int nb)
{
    for (int i = threadIdx.x; i < nb; i += NT) {
        h.cnt[i] = 0u;
        h.mlo[i] = h.mmid[i] = h.mhi[i] = 0u;
    }
}

// Counts (and Q masses) per digit of level l over the logits whose key is
// >= lo_key and whose higher digits equal `prefix`.
template <typename T, bool kMass, int NT>
__device__ void hist_pass(const T *row, int V, int l, uint32_t prefix, uint32_t lo_key, float xmax,
                          const DecScale &dw, FilterHist &h)
{
    const int sh = lvl_shift(l), msk = lvl_bins(l) - 1;
    const int shp = (l == 0) ? 0 : lvl_shift(l - 1);
    auto add = [&](float x) {
        const uint32_t key = order_key(x);
        if (key < lo_key || (l > 0 && (key >> shp) != prefix))
            return;
        const int dg = (int)((key >> sh) & (uint32_t)msk);
        atomicAdd(&h.cnt[dg], 1u);
        if (kMass) {
            const unsigned long long q = dec_weight(x, xmax, dw);
            atomicAdd(&h.mlo[dg], (unsigned int)(q & 0x3FFFull));
            atomicAdd(&h.mmid[dg], (unsigned int)((q >> 14) & 0x3FFFull));
            atomicAdd(&h.mhi[dg], (unsigned int)(q >> 28));
        }
    };
    // Level 0: every logit at or above lo_key is in, so weights go two at a
    // time -- in the 256-thread form; the 512- and 1024-thread forms are held
    // to 64 registers, where the pairs' extra live values cost more than they
    // save.
    if constexpr (kMass && NT <= 256) {
        if (l != 0) {
            row_for_each<T, NT>(row, V, add);
            return;
        }
        auto add2 = [&](float x0, float x1) {
            const uint32_t k0 = order_key(x0), k1 = order_key(x1);
            unsigned long long q0, q1;
            dec_weight2(x0, x1, xmax, dw, q0, q1);
            if (k0 >= lo_key) {
                const int dg = (int)(k0 >> sh);
                atomicAdd(&h.cnt[dg], 1u);
                atomicAdd(&h.mlo[dg], (unsigned int)(q0 & 0x3FFFull));
                atomicAdd(&h.mmid[dg], (unsigned int)((q0 >> 14) & 0x3FFFull));
                atomicAdd(&h.mhi[dg], (unsigned int)(q0 >> 28));
            }
            if (k1 >= lo_key) {
                const int dg = (int)(k1 >> sh);
                atomicAdd(&h.cnt[dg], 1u);
                atomicAdd(&h.mlo[dg], (unsigned int)(q1 & 0x3FFFull));
                atomicAdd(&h.mmid[dg], (unsigned int)((q1 >> 14) & 0x3FFFull));
                atomicAdd(&h.mhi[dg], (unsigned int)(q1 >> 28));
            }
        };
        row_for_each_pair<T, NT>(row, V, add, add2);
    } else {
        row_for_each<T, NT>(row, V, add);
    }
}

// ceil(tp * M) for an fp32 0 <= tp < 1 and M < 2^63, exactly, in integers:
// tp = m * 2^-s with a 24-bit m and s >= 24, so the product is m * M / 2^s
// with m * M a 128-bit integer.  The top-p test "mass above < tp * M" is
// then "mass above < ceil(tp * M)" for integer masses.
__device__ __forceinline__ unsigned long long ceil_mul_frac(float tp, unsigned long long M)
{
    const uint32_t b = __float_as_uint(tp);
    const uint32_t e = (b >> 23) & 0xFFu;
    const unsigned long long m = (unsigned long long)((b & 0x7FFFFFu) | (e ? 0x800000u : 0u));
    if ((b >> 31) || m == 0ull || M == 0ull)
        return 0ull;                           // tp <= 0
    const int sh = e ? 150 - (int)e : 149;     // tp = m * 2^-sh, sh >= 24 for tp < 1
    const unsigned long long lo = m * M, hi = __umul64hi(m, M);
    if (sh >= 128)
        return 1ull;                           // 0 < tp * M < 1
    unsigned long long q;
    bool rem;
    if (sh < 64) {
        q = (lo >> sh) | (hi << (64 - sh));
        rem = (lo & ((1ull << sh) - 1ull)) != 0ull;
    } else {
        q = sh == 64 ? hi : hi >> (sh - 64);
        rem = lo != 0ull || (sh > 64 && (hi & ((1ull << (sh - 64)) - 1ull)) != 0ull);
    }
    return q + (rem ? 1ull : 0ull);
}

// First digit from the top whose inclusive cumulative count reaches `need`
// (counts), or the first non-empty digit from the top with
// base + cumulative mass >= ceil(top_p * total) (masses; the threshold is
// formed at the first level).  With masses and no such digit, the lowest non-empty one.
// Thread t owns digits nb-1-tP .. nb-P-tP (P = nb / NT), scanned in
// descending order.  Ends with a barrier; the result is in `sel`.
template <bool kMass, int NT>
__device__ void hist_select(const FilterHist &h, int nb, unsigned int need, unsigned long long base, float top_p,
                            bool first_level, FilterSel &sel, unsigned int *s_wc, unsigned long long *s_wm)
{
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int P = nb / NT, top = nb - 1 - t * P;
    unsigned int lc = 0;
    unsigned long long lm = 0;
    for (int i = 0; i < P; ++i) {
        lc += h.cnt[top - i];
        lm += h.mass(top - i);
    }
    unsigned int ic = lc;
    unsigned long long im = lm;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned int oc = __shfl_up_sync(0xFFFFFFFFu, ic, o);
        const unsigned long long om = __shfl_up_sync(0xFFFFFFFFu, im, o);
        if (lane >= o) {
            ic += oc;
            im += om;
        }
    }
    if (lane == 31) {
        s_wc[w] = ic;
        s_wm[w] = im;
    }
    if (t == 0) {
        sel.bin = -1;
        sel.low_thread = -1;
    }
    __syncthreads();
    unsigned int cb = ic - lc;
    unsigned long long mb = im - lm, total = 0;
    for (int i = 0; i < NT / 32; ++i) {
        if (i < w) {
            cb += s_wc[i];
            mb += s_wm[i];
        }
        total += s_wm[i];
    }
    unsigned long long athr = 0ull;
    if (kMass)
        athr = first_level ? ceil_mul_frac(top_p, total) : sel.athr;
    const bool earlier = kMass ? (cb > 0u && base + mb >= athr) : (cb >= need);
    if (!earlier) {
        unsigned int cc = cb;
        unsigned long long mm = mb;
        for (int i = 0; i < P; ++i) {
            const int bin = top - i;
            const unsigned int c1 = h.cnt[bin];
            const unsigned long long m1 = h.mass(bin);
            const bool hit = kMass ? (c1 > 0u && base + mm + m1 >= athr) : (cc + c1 >= need);
            if (hit) {
                sel.bin = bin;
                sel.cnt_above = cc;
                sel.mass_above = mm;
                break;
            }
            cc += c1;
            mm += m1;
        }
    }
    if (kMass && lc > 0u)
        atomicMax(&sel.low_thread, t);
    __syncthreads();
    if (kMass) {
        if (sel.bin < 0 && t == sel.low_thread) {
            unsigned int cc = cb;
            unsigned long long mm = mb;
            int lowest = -1;
            unsigned int c_at = 0;
            unsigned long long m_at = 0;
            for (int i = 0; i < P; ++i) {
                const int bin = top - i;
                if (h.cnt[bin] > 0u) {
                    lowest = bin;
                    c_at = cc;
                    m_at = mm;
                }
                cc += h.cnt[bin];
                mm += h.mass(bin);
            }
            sel.bin = lowest;
            sel.cnt_above = c_at;
            sel.mass_above = m_at;
        }
        if (first_level && t == 0)
            sel.athr = athr;
        __syncthreads();
    }
}

// Maximum of a whole row (NaN-propagating: a NaN anywhere gives NaN) for
// every thread of the block; 8 loads in flight per thread.  s_f: NT / 32
// floats of scratch.
template <typename T, int NT>
__device__ float row_max_pass(const T *row, int V, float *s_f)
{
    constexpr int VEC = Storage<T>::kVec;
    constexpr int U = 8;
    const ChunkSplit<T> cs(row, 0, V);
    const int t = threadIdx.x;
    float mx = -INFINITY;
    for (int v = t; v < cs.head_end; v += NT)
        mx = max_nan(mx, Storage<T>::at(row, v));
    const T *body = row + cs.head_end;
    for (int base = 0; base < cs.nvec; base += U * NT) {
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int vi = base + t + u * NT;
            if (vi < cs.nvec)
                r[u] = ld_stream16(body + (size_t)vi * VEC);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int vi = base + t + u * NT;
            if (vi < cs.nvec)
                mx = max_nan(mx, vec_max<T>(r[u]));
        }
    }
    for (int v = cs.tail_beg + t; v < V; v += NT)
        mx = max_nan(mx, Storage<T>::at(row, v));
#pragma unroll
    for (int k = 16; k > 0; k >>= 1)
        mx = max_nan(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, k));
    if ((t & 31) == 0)
        s_f[t >> 5] = mx;
    __syncthreads();
    float r = -INFINITY;
    for (int i = 0; i < NT / 32; ++i)
        r = max_nan(r, s_f[i]);
    __syncthreads();
    return r;
}

// Radix selection of a filtered row's cut (all NT threads; ends with a
// barrier): the k-th largest logit, then the top-p boundary among the logits
// at or above it.  Returns the smallest kept logit; kept_mass: the Q mass of
// the kept logits.
template <typename T, int NT>
__device__ __forceinline__ float radix_cut(const T *row, int V, float xmax, const DecScale &dw, int tk, float tp, bool use_k,
                                           bool use_p, FilterHist &h, FilterSel &sel, unsigned int *s_wc,
                                           unsigned long long *s_wm, unsigned long long &kept_mass)
{
    constexpr int L = KeyLevels<T>::kLevels;
    uint32_t K = 0u;
    kept_mass = 0ull;
    if (use_k) {
        uint32_t prefix = 0u;
        unsigned int need = (unsigned int)tk;
        unsigned long long above = 0ull;
        for (int l = 0; l < L; ++l) {
            const int nb = lvl_bins(l);
            hist_clear<NT>(h, nb);
            __syncthreads();
            if (use_p)
                hist_pass<T, false, NT>(row, V, l, prefix, 0u, xmax, dw, h);
            else
                hist_pass<T, true, NT>(row, V, l, prefix, 0u, xmax, dw, h);
            __syncthreads();
            hist_select<false, NT>(h, nb, need, 0ull, 0.0f, false, sel, s_wc, s_wm);
            const int bin = sel.bin < 0 ? 0 : sel.bin;  // a digit is always found
            need -= sel.cnt_above;
            above += sel.mass_above;
            if (l == L - 1)
                kept_mass = above + h.mass(bin);
            prefix = (l == 0) ? (uint32_t)bin : ((prefix << (lvl_shift(l - 1) - lvl_shift(l))) | (uint32_t)bin);
            __syncthreads();
        }
        K = prefix << lvl_shift(L - 1);
    }
    if (use_p) {
        uint32_t prefix = 0u;
        unsigned long long A = 0ull;
        for (int l = 0; l < L; ++l) {
            const int nb = lvl_bins(l);
            hist_clear<NT>(h, nb);
            __syncthreads();
            hist_pass<T, true, NT>(row, V, l, prefix, K, xmax, dw, h);
            __syncthreads();
            hist_select<true, NT>(h, nb, 0u, A, tp, l == 0, sel, s_wc, s_wm);
            const int bin = sel.bin < 0 ? 0 : sel.bin;  // a digit is always found
            A += sel.mass_above;
            if (l == L - 1)
                kept_mass = A + h.mass(bin);
            prefix = (l == 0) ? (uint32_t)bin : ((prefix << (lvl_shift(l - 1) - lvl_shift(l))) | (uint32_t)bin);
            __syncthreads();
        }
        K = prefix << lvl_shift(L - 1);
    }
    const uint32_t low = (1u << lvl_shift(L - 1)) - 1u;  // key bits below the last digit
    return key_value(K | ((K & 0x80000000u) ? 0u : low));
}

template <typename T, int NT>
__global__ void __launch_bounds__(NT, NT >= 1024 ? 1 : (NT >= 512 ? 2 : 3)) verify_filter_kernel(VerifyArgs a)
{
    __shared__ FilterHist h;
    __shared__ float s_f[4 * NT / 32];
    __shared__ unsigned int s_wc[NT / 32];
    __shared__ unsigned long long s_wm[NT / 32];
    __shared__ FilterSel sel;
    __shared__ float s_m, s_s, s_xmax;
    __shared__ int s_bad, s_skip;
    __shared__ float2 s_e2[64];
    const float c = scale_of(a);
    const Unit u = decode_unit(a);
    const T *row = reinterpret_cast<const T *>(a.logits) + (size_t)u.row * a.V;
    const int t = threadIdx.x;
    if (t == 0)
        s_skip = (!u.needed || stopped_before(a.stop_enc, u.b, u.j)) ? 1 : 0;
    dec_table_init(s_e2);
    __syncthreads();
    const DecScale dw{a.dec_hi, a.dec_lo, s_e2};
    float cut = -INFINITY, s_kept = 0.0f;
    if (!s_skip) {
        const int tk = a.top_k ? a.top_k[u.b] : 0;
        const float tp = a.top_p ? a.top_p[u.b] : 1.0f;
        const bool use_k = tk > 0 && tk < a.V, use_p = tp < 1.0f;
        if (use_k || use_p) {
            // the kept sum comes from the fixed-point masses: pass 1 needs only
            // the maximum (a NaN or +inf gives a non-finite maximum; so does a
            // row of -inf only)
            const float xm = row_max_pass<T, NT>(row, a.V, s_f);
            if (t == 0) {
                s_xmax = xm;
                s_m = xm * c;
                s_s = 0.0f;
                s_bad = (xm > -INFINITY && xm < INFINITY) ? 0 : 1;
                s_skip = stopped_before(a.stop_enc, u.b, u.j) ? 1 : 0;
            }
        } else {
            float m, s;
            bool bad;
            chunk_softmax_stats<T, true, NT>(row, 0, a.V, c, m, s, bad, s_f, StopProbe{a.stop_enc, u.b, u.j},
                                             &s_xmax);
            if (t == 0) {
                s_m = m;
                s_s = s;
                s_bad = (bad || !(s > 0.0f) || !(s <= FLT_MAX)) ? 1 : 0;
                s_skip = stopped_before(a.stop_enc, u.b, u.j) ? 1 : 0;
            }
        }
        __syncthreads();
        s_kept = s_s;
        if (!s_skip && !s_bad && (use_k || use_p)) {
            unsigned long long kept_mass;
            cut = radix_cut<T, NT>(row, a.V, s_xmax, dw, tk, tp, use_k, use_p, h, sel, s_wc, s_wm, kept_mass);
            s_kept = (float)((double)kept_mass * 0x1p-40);
        }
    }
    if (t >= 32)
        return;
    int eval = 0;
    if (t == 0)
        eval = (u.needed && !stopped_before(a.stop_enc, u.b, u.j)) ? 1 : 0;
    if (eval)
        sample_row_decide<T>(a, u, row, s_m, s_kept, cut, s_bad != 0);
    sample_seq_finish(a, u, __shfl_sync(0xFFFFFFFFu, eval, 0) != 0);
}

// ---------------------------------------------------------------------------
// 16-bit logits (bf16 / fp16): the cut from a table of value counts.
//
// A 16-bit logit takes at most 65536 values, so one pass over the row counts
// each bit pattern (16-bit counters, two per shared word; one shared atomic
// per logit) and the rest works on the table: the row maximum is its highest
// non-empty value, and the Q mass of a value is its count times the value's
// weight dec_weight(x, x_max) -- the same weights and the same exact
// integer sums as the radix selection, with one weight per distinct value
// instead of one per logit per pass.  A block scan in descending value order
// gives the k-th largest value and the top-p boundary; the thread range that
// holds either one is then walked by one warp.  A counter that wraps (more
// than 65535 equal logits) shows as a total count below V; the row then
// takes the radix selection, on the same shared memory.
// ---------------------------------------------------------------------------
constexpr int kTabThreads = 1024;
constexpr int kTabWords = 32768;  // 65536 16-bit counters
constexpr int kTabMinV = 32768;   // rows at least this long take the table form
constexpr int kTabSmem = kTabWords * 4;

template <typename T>
struct Tab16;
template <>
struct Tab16<__nv_bfloat16> {
    static constexpr uint32_t kPinfKey = 0xFF80u, kNinfKey = 0x007Fu;  // order keys of +inf and -inf
    __device__ static float value(uint32_t h) { return __uint_as_float(h << 16); }
};
template <>
struct Tab16<__half> {
    static constexpr uint32_t kPinfKey = 0xFC00u, kNinfKey = 0x03FFu;
    __device__ static float value(uint32_t h) { return __half2float(__ushort_as_half((unsigned short)h)); }
};

// order key of a 16-bit pattern and back (-0 has its own key, 0x7FFF, below
// +0's 0x8000; the table merges -0 into +0 before any key is formed)
__device__ __forceinline__ uint32_t pat_key(uint32_t h) { return (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u); }
__device__ __forceinline__ uint32_t key_pat(uint32_t k) { return (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu); }

// Thread t owns the 64 keys 65535 - 64 t (rank 0) down to 65472 - 64 t (rank
// 63): non-negative patterns 0x7FFF - 64 t - r for t < 512, negative ones
// 64 t + r above; either way the 32 table words from tab_base(t).
__device__ __forceinline__ uint32_t rank_pat(int t, int r)
{
    return t < 512 ? 0x7FFFu - 64u * (uint32_t)t - (uint32_t)r : 64u * (uint32_t)t + (uint32_t)r;
}
__device__ __forceinline__ int tab_base(int t) { return t < 512 ? 0x3FE0 - 32 * t : 32 * t; }
__device__ __forceinline__ uint32_t tab_half(uint32_t x, uint32_t h) { return (h & 1u) ? (x >> 16) : (x & 0xFFFFu); }

// Element-wise minimum of two 16-byte vectors of 16-bit floats (NaN is not
// propagated: a NaN anywhere already makes the row's maximum NaN).
template <typename T>
__device__ __forceinline__ uint32_t min_word16(uint32_t a, uint32_t b);
template <>
__device__ __forceinline__ uint32_t min_word16<__nv_bfloat16>(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
template <>
__device__ __forceinline__ uint32_t min_word16<__half>(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("min.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
template <typename T>
__device__ __forceinline__ float word_lo(uint32_t w)
{
    if constexpr (std::is_same<T, __nv_bfloat16>::value)
        return __uint_as_float(w << 16);
    else
        return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
}
template <typename T>
__device__ __forceinline__ float word_hi(uint32_t w)
{
    if constexpr (std::is_same<T, __nv_bfloat16>::value)
        return __uint_as_float(w & 0xFFFF0000u);
    else
        return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}

// all threads: counts every logit of the row into the table (cleared
// before), and finds the row's maximum (NaN-propagating: a NaN anywhere
// gives NaN) and minimum on the way: warp w's go to s_mx[w] / s_mn[w]
// (the caller's barrier publishes them)
template <typename T>
__device__ __forceinline__ void tab_count(const T *row, int V, unsigned int *tab, float *s_mx, float *s_mn)
{
    constexpr int NT = kTabThreads;
    const ChunkSplit<T> cs(row, 0, V);
    const int t = threadIdx.x;
    float mx = -INFINITY, mn = INFINITY;
    auto add = [&](uint32_t h) { atomicAdd(tab + (h >> 1), (h & 1u) ? 0x10000u : 1u); };
    auto add1 = [&](unsigned short h) {
        add(h);
        const float v = word_lo<T>(h);
        mx = max_nan(mx, v);
        mn = fminf(mn, v);
    };
    for (int v = t; v < cs.head_end; v += NT)
        add1(__ldg(reinterpret_cast<const unsigned short *>(row) + v));
    const T *body = row + cs.head_end;
    constexpr int U = 8;  // 128 KB of loads in flight per CTA (one CTA per SM)
    bool any = false;
    uint32_t wmx = 0u, wmn = 0u;  // running packed maximum / minimum of the vectors
    for (int base = 0; base < cs.nvec; base += U * NT) {
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int vi = base + t + u * NT;
            if (vi < cs.nvec)
                r[u] = ld_stream16(body + (size_t)vi * 8);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int vi = base + t + u * NT;
            if (vi < cs.nvec) {
                const uint32_t w[4] = {r[u].x, r[u].y, r[u].z, r[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    add(w[e] & 0xFFFFu);
                    add(w[e] >> 16);
                }
                const uint32_t vx = max_word<T>(max_word<T>(r[u].x, r[u].y), max_word<T>(r[u].z, r[u].w));
                const uint32_t vn =
                    min_word16<T>(min_word16<T>(r[u].x, r[u].y), min_word16<T>(r[u].z, r[u].w));
                wmx = any ? max_word<T>(wmx, vx) : vx;
                wmn = any ? min_word16<T>(wmn, vn) : vn;
                any = true;
            }
        }
    }
    for (int v = cs.tail_beg + t; v < V; v += NT)
        add1(__ldg(reinterpret_cast<const unsigned short *>(row) + v));
    if (any) {
        mx = max_nan(mx, max_nan(word_lo<T>(wmx), word_hi<T>(wmx)));
        mn = fminf(mn, fminf(word_lo<T>(wmn), word_hi<T>(wmn)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mx = max_nan(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
    }
    if ((t & 31) == 0) {
        s_mx[t >> 5] = mx;
        s_mn[t >> 5] = mn;
    }
}

// Block-wide exclusive prefix (thread order) of a count and a mass, with
// both totals; ends with a barrier.  s_wc, s_wm: one slot per warp and the
// total (warp 0 turns the warp totals into their exclusive prefix by
// shuffles).
__device__ __forceinline__ void tab_scan(uint32_t c, unsigned long long m, uint32_t &c_ex, unsigned long long &m_ex,
                                         uint32_t &c_tot, unsigned long long &m_tot, unsigned int *s_wc,
                                         unsigned long long *s_wm)
{
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    uint32_t ic = c;
    unsigned long long im = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t oc = __shfl_up_sync(0xFFFFFFFFu, ic, o);
        const unsigned long long om = __shfl_up_sync(0xFFFFFFFFu, im, o);
        if (lane >= o) {
            ic += oc;
            im += om;
        }
    }
    __syncthreads();  // earlier readers of s_wc / s_wm are done
    if (lane == 31) {
        s_wc[w] = ic;
        s_wm[w] = im;
    }
    __syncthreads();
    static_assert(kTabThreads == 1024, "one warp total per lane of warp 0");
    if (w == 0) {  // inclusive prefix of the 32 warp totals, stored exclusive
        uint32_t wc = s_wc[lane];
        unsigned long long wm = s_wm[lane];
        const uint32_t wc0 = wc;
        const unsigned long long wm0 = wm;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t oc = __shfl_up_sync(0xFFFFFFFFu, wc, o);
            const unsigned long long om = __shfl_up_sync(0xFFFFFFFFu, wm, o);
            if (lane >= o) {
                wc += oc;
                wm += om;
            }
        }
        __syncwarp();
        s_wc[lane] = wc - wc0;
        s_wm[lane] = wm - wm0;
        if (lane == 31) {  // the block totals
            s_wc[32] = wc;
            s_wm[32] = wm;
        }
    }
    __syncthreads();
    c_ex = ic - c + s_wc[w];
    m_ex = im - m + s_wm[w];
    c_tot = s_wc[32];
    m_tot = s_wm[32];
}

// Warp 0 (all lanes): walks the 64 keys of thread tc in descending order,
// lane l taking ranks 2 l and 2 l + 1 (one table word).  Keys below kk count
// as empty.  Finds the first non-empty key where the running count from the
// top (c0 + counts) reaches `need` (kCount) or the running mass (m0 +
// masses) reaches the threshold `athr`; writes that key and the running mass
// at it to *key_out / *mass_out (untouched when there is none).
template <typename T, bool kCount>
__device__ __forceinline__ void tab_walk(const unsigned int *tab, int tc, uint32_t kk, float xmax, const DecScale &dw,
                                         uint32_t c0, uint32_t need, unsigned long long m0, unsigned long long athr,
                                         int *key_out, unsigned long long *mass_out)
{
    const int lane = threadIdx.x & 31;
    const uint32_t ha = rank_pat(tc, 2 * lane), hb = rank_pat(tc, 2 * lane + 1);
    const uint32_t x = tab[ha >> 1];
    const uint32_t ka = pat_key(ha), kb = pat_key(hb);
    const uint32_t na = ka >= kk ? tab_half(x, ha) : 0u, nb = kb >= kk ? tab_half(x, hb) : 0u;
    // an empty key's weight is not needed: x_max stands in (no inf or NaN)
    const float va = na ? Tab16<T>::value(ha) : xmax, vb = nb ? Tab16<T>::value(hb) : xmax;
    unsigned long long qa, qb;
    dec_weight2(va, vb, xmax, dw, qa, qb);
    const unsigned long long ma = (unsigned long long)na * qa, mb = (unsigned long long)nb * qb;
    uint32_t ic = na + nb;
    unsigned long long im = ma + mb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t oc = __shfl_up_sync(0xFFFFFFFFu, ic, o);
        const unsigned long long om = __shfl_up_sync(0xFFFFFFFFu, im, o);
        if (lane >= o) {
            ic += oc;
            im += om;
        }
    }
    const uint32_t ce = c0 + ic - (na + nb);
    const unsigned long long me = m0 + im - (ma + mb);
    bool hit_a, hit_b;
    if (kCount) {
        hit_a = na > 0u && ce + na >= need;
        hit_b = nb > 0u && ce + na + nb >= need;
    } else {
        hit_a = na > 0u && me + ma >= athr;
        hit_b = nb > 0u && me + ma + mb >= athr;
    }
    const unsigned hits = __ballot_sync(0xFFFFFFFFu, hit_a || hit_b);
    if (hits && lane == __ffs(hits) - 1) {
        *key_out = (int)(hit_a ? ka : kb);
        *mass_out = hit_a ? me + ma : me + ma + mb;
    }
}

// 16-bit pattern of a value of the row (exact: the value came from one)
template <typename T>
__device__ __forceinline__ uint32_t pat_of(float v)
{
    if constexpr (std::is_same<T, __nv_bfloat16>::value)
        return __float_as_uint(v) >> 16;
    else
        return (uint32_t)__half_as_ushort(__float2half_rn(v));
}

// Table selection (all threads, after tab_count and a barrier).  Returns
// false when the table is unusable (a wrapped counter: the caller runs the
// radix selection); else the row's maximum, its non-finite flag and, when
// the row is filtered and finite, the cut and the kept Q mass.  xmax / xmin:
// the row's maximum (NaN-propagating) and minimum from tab_count.  s_i: 9
// ints, s_u: 5 u64, s_cl / s_ml: kTabThreads u32 / u64 of shared scratch
// (every slot written once per row).
template <typename T>
__device__ bool tab_select(unsigned int *tab, int V, float xmax, float xmin, const DecScale &dw, int tk, float tp,
                           bool use_k, bool use_p, bool &bad_out, float &cut_out, unsigned long long &kept_out,
                           unsigned int *s_wc, unsigned long long *s_wm, int *s_i, unsigned long long *s_u,
                           unsigned int *s_cl, unsigned long long *s_ml)
{
    const int t = threadIdx.x, lane = t & 31;
    s_cl[t] = 0u;  // the merged pass writes the slots of non-empty blocks only
    s_ml[t] = 0ull;
    if (t == 0) {  // -0 (pattern 0x8000) joins +0 (pattern 0)
        const uint32_t nz = tab[0x4000] & 0xFFFFu, pz = tab[0] & 0xFFFFu;
        s_i[0] = (nz + pz > 0xFFFFu) ? 1 : 0;  // would wrap
        tab[0x4000] -= nz;
        tab[0] += nz;
        s_i[3] = -1;  // thread holding the k-th largest key
        s_i[5] = -1;  // the k-th largest key
        s_i[7] = -1;  // thread holding the top-p boundary
        s_i[8] = -1;  // the top-p boundary key
    }
    // +inf or a NaN anywhere, or nothing above -inf
    bad_out = !(xmax > -INFINITY && xmax < INFINITY);
    __syncthreads();
    if (bad_out)
        return s_i[0] == 0;  // a wrap is not checked here: the row is undefined either way
    if (xmax == 0.0f)
        xmax = 0.0f;  // -0 counts as +0 (its key)
    if (xmin == 0.0f)
        xmin = 0.0f;
    const uint32_t kmin = pat_key(pat_of<T>(xmin));
    // one pass: each thread range's count and Q mass, two values per word
    // with paired weights.  The non-empty words form a band of values, which
    // in the threads' own ranges would load a few warps only; so the table's
    // 1024 blocks of 32 words (block b = the range of one thread) are dealt
    // out by warp -- warp w takes blocks w, w + 32, ... -- each lane one word
    // of the block, and the block's sums go to its owner's slots (no atomics:
    // each block has one warp).  A first sweep of ballots marks the
    // non-empty blocks; only those are visited.
    {
        const int w = t >> 5;
        uint32_t busy = 0u;  // bit i: block w + 32 i holds a count (independent loads)
#pragma unroll 8
        for (int i = 0; i < 32; ++i)
            busy |= (__ballot_sync(0xFFFFFFFFu, tab[32u * (uint32_t)(w + 32 * i) + (uint32_t)lane] != 0u) != 0u ? 1u : 0u)
                    << i;
        while (busy) {
            const int i = __ffs(busy) - 1;
            busy &= busy - 1u;
            const int blk = w + 32 * i;  // words 32 blk .. 32 blk + 31
            const uint32_t word = 32u * (uint32_t)blk + (uint32_t)lane;
            const uint32_t x = tab[word];
            unsigned long long m = 0;
            if (x != 0u) {
                const uint32_t h = 2u * word;
                const float v0 = (x & 0xFFFFu) ? Tab16<T>::value(h) : xmax,
                            v1 = (x >> 16) ? Tab16<T>::value(h + 1u) : xmax;
                unsigned long long q0, q1;
                dec_weight2(v0, v1, xmax, dw, q0, q1);
                m = (unsigned long long)(x & 0xFFFFu) * q0 + (unsigned long long)(x >> 16) * q1;
            }
            const uint32_t c = __reduce_add_sync(0xFFFFFFFFu, (x & 0xFFFFu) + (x >> 16));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                m += __shfl_xor_sync(0xFFFFFFFFu, m, o);
            if (lane == 0) {  // the owner of block blk (tab_base inverted)
                const int own = blk < 512 ? 511 - blk : blk;
                s_cl[own] = c;
                s_ml[own] = m;
            }
        }
    }
    __syncthreads();
    const uint32_t cl = s_cl[t];
    const unsigned long long ml = s_ml[t];
    uint32_t c_ex, c_tot;
    unsigned long long m_ex, m_tot;
    tab_scan(cl, ml, c_ex, m_ex, c_tot, m_tot, s_wc, s_wm);
    if (s_i[0] || c_tot != (uint32_t)V)
        return false;  // a counter wrapped (or would have)
    // top-k: the key where the count from the top reaches tk (ties kept)
    uint32_t kk = 0u;                  // lowest key top-k keeps
    unsigned long long tot_p = m_tot;  // Q mass of the logits top-k keeps
    int tck = 1024;                    // thread holding kk
    if (use_k) {
        const uint32_t need = (uint32_t)tk;
        if (c_ex < need && need <= c_ex + cl) {  // exactly one thread
            s_i[3] = t;
            s_i[4] = (int)c_ex;
            s_u[2] = m_ex;
        }
        __syncthreads();
        tck = s_i[3];
        if (t < 32)
            tab_walk<T, true>(tab, tck, 0u, xmax, dw, (uint32_t)s_i[4], need, s_u[2], 0ull, s_i + 5, s_u);
        __syncthreads();
        kk = (uint32_t)s_i[5];
        tot_p = s_u[0];
    }
    if (!use_p) {
        cut_out = Tab16<T>::value(key_pat(kk));
        kept_out = tot_p;
        return true;
    }
    // top-p among the keys >= kk: the first non-empty key from the top at
    // which mass above + its mass >= ceil(tp * tot_p).  The running mass only
    // grows, so that key lies in the one thread whose kept range holds a key,
    // has its mass above below the threshold (or nothing non-empty above) and
    // reaches it within the range.
    const unsigned long long athr = ceil_mul_frac(tp, tot_p);
    if (t <= tck) {
        const uint32_t cl_r = (t == tck) ? 1u : cl;  // thread tck keeps kk at least
        const unsigned long long ml_r = (t == tck) ? tot_p - m_ex : ml;
        if (cl_r > 0u && (c_ex == 0u || m_ex < athr) && m_ex + ml_r >= athr) {
            s_i[7] = t;
            s_u[3] = m_ex;
        }
    }
    __syncthreads();
    const int tcp = s_i[7];
    if (tcp >= 0 && t < 32)
        tab_walk<T, false>(tab, tcp, kk, xmax, dw, 0u, 0u, s_u[3], athr, s_i + 8, s_u + 1);
    __syncthreads();
    if (s_i[8] < 0) {  // no key reached the bound: the lowest key kept
        cut_out = Tab16<T>::value(key_pat(use_k ? kk : kmin));
        kept_out = tot_p;
    } else {
        cut_out = Tab16<T>::value(key_pat((uint32_t)s_i[8]));
        kept_out = s_u[1];
    }
    return true;
}

// One CTA of kTabThreads per target row of 16-bit logits, V >= kTabMinV;
// dynamic shared memory: kTabSmem bytes (the table, or the radix
// histograms when a counter wrapped)
template <typename T>
__global__ void __launch_bounds__(kTabThreads, 1) verify_filter_tab_kernel(VerifyArgs a)
{
    constexpr int NT = kTabThreads;
    extern __shared__ __align__(16) unsigned int tab[];
    __shared__ float s_f[4 * NT / 32];
    __shared__ unsigned int s_wc[NT / 32 + 1];
    __shared__ unsigned long long s_wm[NT / 32 + 1];
    __shared__ FilterSel sel;
    __shared__ int s_i[9];
    __shared__ unsigned long long s_u[5];
    __shared__ unsigned int s_cl[kTabThreads];
    __shared__ unsigned long long s_ml[kTabThreads];
    __shared__ float s_m, s_s, s_xmax, s_cut;
    __shared__ int s_bad, s_skip;
    __shared__ float2 s_e2[64];
    const float c = scale_of(a);
    const Unit u = decode_unit(a);
    const T *row = reinterpret_cast<const T *>(a.logits) + (size_t)u.row * a.V;
    const int t = threadIdx.x;
    // thread 0 carries the row's ratio-test inputs: the proposal now, the
    // rest once the count pass is done, so that both load rounds are off
    // the row's end
    int y_in = -1;
    RowInputs in{-1, 0.0f, 1.0f, 0.0f};
    if (t == 0) {
        s_skip = (!u.needed || stopped_before(a.stop_enc, u.b, u.j)) ? 1 : 0;
        s_cut = -INFINITY;
        y_in = row_proposal(a, u);
    }
    dec_table_init(s_e2);
    __syncthreads();
    const DecScale dw{a.dec_hi, a.dec_lo, s_e2};
    if (!s_skip) {
        const int tk = a.top_k ? a.top_k[u.b] : 0;
        const float tp = a.top_p ? a.top_p[u.b] : 1.0f;
        const bool use_k = tk > 0 && tk < a.V, use_p = tp < 1.0f;
        if (use_k || use_p) {
            for (int i = t; i < kTabWords / 4; i += NT)
                reinterpret_cast<uint4 *>(tab)[i] = make_uint4(0u, 0u, 0u, 0u);  // 8 stores per thread
            __syncthreads();
            tab_count<T>(row, a.V, tab, s_f, s_f + NT / 32);
            if (t == 0) {
                s_skip = stopped_before(a.stop_enc, u.b, u.j) ? 1 : 0;
                in = row_inputs<T>(a, u, row, y_in);
            }
            __syncthreads();
            if (!s_skip) {
                // the warps' extremes, reduced by every warp (one per lane)
                float xmax = s_f[t & 31], xmin = s_f[NT / 32 + (t & 31)], cutv;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    xmax = max_nan(xmax, __shfl_xor_sync(0xFFFFFFFFu, xmax, o));
                    xmin = fminf(xmin, __shfl_xor_sync(0xFFFFFFFFu, xmin, o));
                }
                bool bad;
                unsigned long long kept;
                // block-uniform result (it derives from shared values only)
                if (tab_select<T>(tab, a.V, xmax, xmin, dw, tk, tp, use_k, use_p, bad, cutv, kept, s_wc, s_wm,
                                  s_i, s_u, s_cl, s_ml)) {
                    if (t == 0) {
                        s_m = xmax * c;
                        s_bad = bad ? 1 : 0;
                        s_s = bad ? 0.0f : (float)((double)kept * 0x1p-40);
                        s_cut = bad ? -INFINITY : cutv;
                    }
                } else {  // a counter wrapped: the radix selection on the same memory
                    __syncthreads();
                    const float xm = row_max_pass<T, NT>(row, a.V, s_f);
                    const bool badm = !(xm > -INFINITY && xm < INFINITY);
                    float cr = -INFINITY;
                    unsigned long long km = 0ull;
                    if (!badm)
                        cr = radix_cut<T, NT>(row, a.V, xm, dw, tk, tp, use_k, use_p,
                                              *reinterpret_cast<FilterHist *>(tab), sel, s_wc, s_wm, km);
                    if (t == 0) {
                        s_m = xm * c;
                        s_bad = badm ? 1 : 0;
                        s_s = (float)((double)km * 0x1p-40);
                        s_cut = cr;
                    }
                }
            }
        } else {
            float m, s;
            bool bad;
            chunk_softmax_stats<T, true, NT>(row, 0, a.V, c, m, s, bad, s_f, StopProbe{a.stop_enc, u.b, u.j},
                                             &s_xmax);
            if (t == 0) {
                s_m = m;
                s_s = s;
                s_bad = (bad || !(s > 0.0f) || !(s <= FLT_MAX)) ? 1 : 0;
                s_skip = stopped_before(a.stop_enc, u.b, u.j) ? 1 : 0;
            }
        }
        __syncthreads();
    }
    if (t >= 32)
        return;
    int eval = 0;
    if (t == 0)
        eval = (u.needed && !stopped_before(a.stop_enc, u.b, u.j)) ? 1 : 0;
    if (eval) {
        if (in.y != y_in)  // the unfiltered path: the rest of the inputs now
            in = row_inputs<T>(a, u, row, y_in);
        row_decide(a, u, in, s_m, s_s, s_cut, s_bad != 0);
    }
    sample_seq_finish(a, u, __shfl_sync(0xFFFFFFFFu, eval, 0) != 0);
}

// Block size by the number of rows (one CTA per row): a row per SM at most
// -> 1024 threads; two rows per SM at most -> 512 for top-p alone (two CTAs
// fit on an SM, so every row runs in the first wave; measured faster), 1024
// with top-k (its count-only passes are issue-bound: two CTAs sharing an SM
// gain nothing over a second wave); more rows -> 256.
template <typename T>
cudaError_t launch_filter_rows(const VerifyArgs &args, cudaStream_t st)
{
    static int sm_count[64];
    VerifyArgs f = args;
    f.C = 1;  // one CTA per row
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (sm_count[dev & 63] == 0) {
        e = cudaDeviceGetAttribute(&sm_count[dev & 63], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
    }
    const unsigned rows = (unsigned)(f.B * (f.k + 1)), sms = (unsigned)sm_count[dev & 63];
    if constexpr (sizeof(T) == 2) {
        if (f.V >= kTabMinV) {
            static bool attr_set[64];
            if (!attr_set[dev & 63]) {
                e = cudaFuncSetAttribute(verify_filter_tab_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kTabSmem);
                if (e != cudaSuccess)
                    return e;
                attr_set[dev & 63] = true;
            }
            verify_filter_tab_kernel<T><<<rows, kTabThreads, kTabSmem, st>>>(f);
            return cudaGetLastError();
        }
    }
    if (rows <= sms)
        verify_filter_kernel<T, 1024><<<rows, 1024, 0, st>>>(f);
    else if (rows <= 2u * sms && f.top_k == nullptr)
        verify_filter_kernel<T, 512><<<rows, 512, 0, st>>>(f);
    else if (rows <= 2u * sms)
        verify_filter_kernel<T, 1024><<<rows, 1024, 0, st>>>(f);
    else
        verify_filter_kernel<T, kThreads><<<rows, kThreads, 0, st>>>(f);
    return cudaGetLastError();
}

}  // namespace spec
