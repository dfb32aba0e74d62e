// sample_final.cuh -- the end of a stochastic verification row and of a
// sequence, shared by the plain statistics kernel (softmax of the whole
// vocabulary) and the filtered one (top-k / top-p).
//
// Row: proposal y of row j is accepted iff u_j < p_j(y) / q_j(y), with p_j the
// distribution the target samples from ("Chapter 10 Speculative Decoding (Code
// Walkthrough)", §5.1: after temperature, top-k or top-p, the processed
// probabilities).  A token below the row's cut (top-k / top-p) has p = 0.
// Sequence: the first stop by one warp ballot; the accepted prefix is
// committed and the draw (correction or bonus) handed to the draw kernel.
#pragma once

#include <float.h>

#include "verify_common.cuh"

namespace spec {

struct RowStats {
    float m, s;  // base-2 row maximum of x * c and sum of 2^(x c - m) over the kept tokens
};

__device__ __forceinline__ float scale_of(const VerifyArgs &a) { return a.unit_temp ? kLog2e : a.inv_temp * kLog2e; }

// The loaded inputs of one row's ratio test.
struct RowInputs {
    int y;        // the proposal (-1: none, the bonus row or a stopped budget)
    float xy;     // its target logit
    float qy;     // its draft probability
    float u;      // the row's uniform
};

// One lane: the draft token of row u.row (first load round).
__device__ __forceinline__ int row_proposal(const VerifyArgs &a, const Unit &u)
{
    return (u.j < u.kb) ? a.draft[(size_t)u.b * a.k + u.j] : -1;
}

// One lane: the rest of the row's inputs, given its proposal y (second round).
template <typename T>
__device__ __forceinline__ RowInputs row_inputs(const VerifyArgs &a, const Unit &u, const T *row, int y)
{
    RowInputs in{y, 0.0f, 1.0f, 0.0f};
    if (u.j < u.kb && y >= 0 && y < a.V) {
        in.xy = Storage<T>::at(row, y);
        in.qy = a.q[((size_t)u.b * a.k + u.j) * a.V + y];
        in.u = a.u[(size_t)u.b * (a.k + 1) + u.j];
    }
    return in;
}

// One lane: ratio test of row u.row from its loaded inputs, and its results.
// m, s: the row's base-2 maximum and kept sum; cut: the smallest kept logit
// (-inf: all kept); bad: the row's softmax is undefined.
__device__ __forceinline__ void row_decide(const VerifyArgs &a, const Unit &u, const RowInputs &in, float m, float s,
                                           float cut, bool bad)
{
    const float c = scale_of(a);
    uint32_t fl = (bad || !(s <= FLT_MAX) || !(s > 0.0f)) ? SPEC_FLAG_NONFINITE : 0u;
    int acc = 0;
    bool stop;
    if (u.j < u.kb) {
        const int y = in.y;
        if (y < 0 || y >= a.V) {
            fl |= SPEC_FLAG_BAD_TOKEN;
        } else {
            const float py = (in.xy >= cut) ? exp2f(fmaf(in.xy, c, -m)) / s : 0.0f;
            if (in.qy == 0.0f)
                fl |= SPEC_FLAG_Q_ZERO;
            acc = (in.u < py / in.qy) ? 1 : 0;
        }
        stop = !acc || (a.eos >= 0 && y == a.eos) || (u.j + 1 == u.rem);
    } else {
        stop = true;  // the bonus row ends the round
    }
    a.row_tok[u.row] = acc;
    reinterpret_cast<RowStats *>(a.row_ms)[u.row] = RowStats{m, s};
    a.row_flag[u.row] = fl;
    if (a.filtered)
        a.row_cut[u.row] = cut;
    if (stop)
        atomicMax(a.stop_enc + u.b, kStopBase - u.j);
}

// One lane: loads the row's inputs and runs the ratio test.
template <typename T>
__device__ void sample_row_decide(const VerifyArgs &a, const Unit &u, const T *row, float m, float s, float cut,
                                  bool bad)
{
    row_decide(a, u, row_inputs<T>(a, u, row, row_proposal(a, u)), m, s, cut, bad);
}

// One lane, after row u.row's results are stored: counts the row for its
// sequence; true for the sequence's last row (whose warp then writes the
// outputs with sample_seq_outputs).  wrote: the row stored results (a row
// that did not -- one past its sequence's stop -- has nothing to publish
// before the count, and its results are never read).
__device__ __forceinline__ bool sample_seq_count(const VerifyArgs &a, int b, bool wrote = true)
{
    if (wrote)
        __threadfence();
    return atomicAdd(a.seq_cnt + b, 1) == a.k;
}

// One warp (all 32 lanes), after every row of sequence b was counted: the
// first stop by one ballot (lane j = row j), the accepted prefix committed,
// the draw (correction or bonus) handed to the draw kernel, the sequence's
// counters reset.  Row results written by other CTAs are read through L2.
__device__ __forceinline__ void sample_seq_outputs(const VerifyArgs &a, int b, int kb, int rem)
{
    __threadfence();
    const int lane = threadIdx.x & 31;
    const int j = lane;
    int acc = 0, d = -1;
    uint32_t fl = 0;
    bool stop = false;
    if (j <= a.k && rem > 0) {
        acc = __ldcg(a.row_tok + b * (a.k + 1) + j);
        fl = __ldcg(a.row_flag + b * (a.k + 1) + j);
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
        a.draw_row[b] = (js >= 0 && !accepted_stop) ? js : -1;
        if (a.flags)
            a.flags[b] = seq_fl;
        a.seq_cnt[b] = 0;
        a.stop_enc[b] = 0;
    }
}

// Warp 0 (all 32 lanes) after a row of sequence u.b is done: counts the row;
// the sequence's last row writes the outputs.  wrote: as sample_seq_count.
__device__ __forceinline__ void sample_seq_finish(const VerifyArgs &a, const Unit &u, bool wrote = true)
{
    int last_row = 0;
    if ((threadIdx.x & 31) == 0)
        last_row = sample_seq_count(a, u.b, wrote) ? 1 : 0;
    if (__shfl_sync(0xFFFFFFFFu, last_row, 0))
        sample_seq_outputs(a, u.b, u.kb, u.rem);
}

}  // namespace spec
