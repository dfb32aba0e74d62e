// spec_launch.h -- host-side launchers of the library's kernels (internal;
// the public ABI is include/specverify.h, implemented in api.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "specverify.h"

namespace spec {

struct VerifyArgs {
    const void *logits;
    int B, k, V, C;
    int chunk;  // elements per work unit (set by the launcher)
    const int32_t *draft;
    const int32_t *draft_len;
    int32_t eos;
    const int32_t *remaining;
    int32_t *out_tokens;
    int32_t *n_accept;
    int32_t *n_emit;
    void *ws;
    // workspace arrays, resolved on the host by the launcher from ws
    int *stop_enc, *row_cnt, *seq_cnt, *row_tok, *draw_row;
    float2 *row_ms;
    uint32_t *row_flag;
    void *part;
    float *rpart;
    double *rtot;
    // stochastic verification only
    float inv_temp;
    int unit_temp;
    const float *q;
    const float *u;
    float *out_residual;
    uint32_t *flags;
    // top-k / top-p (filtered = 0: neither, the plain statistics kernel runs)
    int filtered;
    const int32_t *top_k;  // [B] or null
    const float *top_p;    // [B] or null
    float dec_hi, dec_lo;  // log2(e) / T as a float pair: the scale of the top-p decision weights
    float *row_cut;        // workspace: smallest kept logit per row
};

// fills C, chunk and the workspace pointers of `a` from B, k, V and ws
void resolve_verify_args(VerifyArgs &a);
cudaError_t launch_verify_greedy(const VerifyArgs &a, spec_dtype dt, cudaStream_t st);
cudaError_t launch_verify_sample(const VerifyArgs &a, spec_dtype dt, cudaStream_t st);

// one KV cache [L, 2, B, H, S, D] moved by a realignment plan
struct CacheDesc {
    void *kv;
    int elt_bytes, L, H, D;
};

struct RealignArgs {
    CacheDesc cache[SPEC_MAX_CACHES];
    int n_caches;
    int B, S;
    const int32_t *len, *pad, *n_emit;
    int32_t *len_new, *pad_new, *width_new, *err;
    void *ws;
    unsigned bulk_mask;  // caches moved by the bulk-copy kernel (set by the launcher)
    int plain_cache;     // the cache a plain-path launch moves (set by the launcher)
};
cudaError_t launch_realign(const RealignArgs &a, cudaStream_t st);

// ragged pool (EXSPEC): move runs between a pool [L,2,N,H,S,D] and a
// left-padded batch [L,2,B,H,S,D]
struct PoolArgs {
    const void *src;  // pool (repad) or batch (unpad)
    void *dst;        // batch (repad) or pool (unpad)
    int elt_bytes, L, N, B, H, S, D;
    int repad;        // 1: pool -> batch, 0: batch -> pool
    const int32_t *idx;       // [B] pool index of each batch row
    const int32_t *pool_len;  // repad: [N] lengths in the pool
    const int32_t *len, *pad; // unpad: [B] batch lengths and paddings
    const int32_t *n_emit;    // unpad: [B] commits added to len, or null
    int32_t *len_out, *pad_out, *width_out;  // repad outputs
    int32_t *pool_len_out;    // unpad: [N] lengths written back
    int32_t *err;
    void *ws;
};
cudaError_t launch_pool_copy(const PoolArgs &a, cudaStream_t st);
cudaError_t launch_commit_ragged(int N, int32_t *pool_len, int B, const int32_t *idx, const int32_t *n_emit, int S,
                                 int32_t *err, cudaStream_t st);

cudaError_t launch_pos_mask(int B, int S, const int32_t *pad_old, const int32_t *pad_new, int32_t *pos,
                            uint8_t *mask, cudaStream_t st);

cudaError_t launch_group(int N, const int32_t *len, const uint8_t *active, int B, int32_t *out_idx,
                         int32_t *out_count_equal, int32_t *out_group_len, cudaStream_t st);

}  // namespace spec
