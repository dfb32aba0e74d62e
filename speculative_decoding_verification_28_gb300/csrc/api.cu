// api.cu -- the extern "C" entry points of include/specverify.h: host-side
// argument checks (nothing is launched on an error) and kernel launches.
#include <limits.h>

#include "spec_common.cuh"
#include "spec_launch.h"

using namespace spec;

namespace {

bool dtype_ok(int dt) { return dt == SPEC_F32 || dt == SPEC_BF16 || dt == SPEC_F16; }
int dtype_bytes(int dt) { return dt == SPEC_F32 ? 4 : 2; }
bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_workspace(void *ws, size_t have, size_t need)
{
    if (need == 0)
        return SPEC_OK;
    if (!ws || have < need || !aligned(ws, 256))
        return SPEC_EWORKSPACE;
    return SPEC_OK;
}

int launched(cudaError_t e) { return e == cudaSuccess ? SPEC_OK : SPEC_ECUDA; }

int check_verify_common(const void *logits, int dt, int B, int k, int V, const int32_t *draft, const int32_t *draft_len,
                        const int32_t *remaining,
                        const int32_t *out_tokens, const int32_t *n_accept, const int32_t *n_emit)
{
    if (B < 0 || k < 0 || k > SPEC_MAX_K || V < 1)
        return SPEC_EINVAL;
    if (!dtype_ok(dt))
        return SPEC_EDTYPE;
    if (B == 0)
        return SPEC_OK;
    if (!logits || (k > 0 && !draft) || !out_tokens || !n_accept || !n_emit)
        return SPEC_EINVAL;
    const long long units = (long long)B * (k + 1) * verify_chunks(B, k, V);
    if (units > INT_MAX)
        return SPEC_EINVAL;
    if (!aligned(logits, dtype_bytes(dt)) || !aligned(out_tokens, 4) || !aligned(n_accept, 4) ||
        !aligned(n_emit, 4) || (draft && !aligned(draft, 4)) || (draft_len && !aligned(draft_len, 4)) ||
        (remaining && !aligned(remaining, 4)))
        return SPEC_EALIGN;
    return SPEC_OK;
}

// ---- verification: checks and arguments ----------------------------------
int check_greedy(const void *logits, int dt, int B, int k, int V, const int32_t *draft, const int32_t *draft_len,
                 const int32_t *remaining, const int32_t *out_tokens,
                 const int32_t *n_accept, const int32_t *n_emit, void *workspace, size_t workspace_bytes)
{
    const int rc = check_verify_common(logits, dt, B, k, V, draft, draft_len, remaining, out_tokens, n_accept, n_emit);
    if (rc != SPEC_OK || B == 0)
        return rc;
    return check_workspace(workspace, workspace_bytes, spec_workspace_bytes(B, k, V));
}

int check_sample(const void *logits, int dt, float temperature, const int32_t *top_k, const float *top_p,
                 const float *draft_probs, const int32_t *draft, const float *uniforms, int B, int k, int V,
                 const int32_t *draft_len, const int32_t *remaining,
                 const int32_t *out_tokens, const int32_t *n_accept, const int32_t *n_emit,
                 const float *out_residual, const uint32_t *flags, void *workspace, size_t workspace_bytes)
{
    const int rc = check_verify_common(logits, dt, B, k, V, draft, draft_len, remaining, out_tokens, n_accept, n_emit);
    if (rc != SPEC_OK || B == 0)
        return rc;
    if (!(temperature > 0.0f) || !(temperature <= 3.0e38f) || !uniforms || (k > 0 && !draft_probs))
        return SPEC_EINVAL;
    if ((top_k || top_p) && V > SPEC_MAX_FILTER_V)
        return SPEC_EINVAL;
    if (!aligned(uniforms, 4) || (draft_probs && !aligned(draft_probs, 4)) ||
        (out_residual && !aligned(out_residual, 4)) || (flags && !aligned(flags, 4)) ||
        (top_k && !aligned(top_k, 4)) || (top_p && !aligned(top_p, 4)))
        return SPEC_EALIGN;
    return check_workspace(workspace, workspace_bytes, spec_workspace_bytes(B, k, V));
}

VerifyArgs verify_args(const void *logits, int B, int k, int V, const int32_t *draft, const int32_t *draft_len,
                       int32_t eos_id, const int32_t *remaining, int32_t *out_tokens, int32_t *n_accept,
                       int32_t *n_emit, void *workspace)
{
    VerifyArgs a{};
    a.logits = logits;
    a.B = B;
    a.k = k;
    a.V = V;
    a.draft = draft;
    a.draft_len = draft_len;
    a.eos = eos_id;
    a.remaining = remaining;
    a.out_tokens = out_tokens;
    a.n_accept = n_accept;
    a.n_emit = n_emit;
    a.ws = workspace;
    return a;
}

VerifyArgs sample_args(const void *logits, float temperature, const int32_t *top_k, const float *top_p,
                       const float *draft_probs, const int32_t *draft, const float *uniforms, int B, int k, int V,
                       const int32_t *draft_len, int32_t eos_id, const int32_t *remaining, int32_t *out_tokens,
                       int32_t *n_accept, int32_t *n_emit, float *out_residual, uint32_t *flags, void *workspace)
{
    VerifyArgs a = verify_args(logits, B, k, V, draft, draft_len, eos_id, remaining, out_tokens, n_accept, n_emit,
                               workspace);
    a.inv_temp = 1.0f / temperature;
    a.unit_temp = temperature == 1.0f ? 1 : 0;
    a.q = draft_probs;
    a.u = uniforms;
    a.out_residual = out_residual;
    a.flags = flags;
    a.filtered = (top_k || top_p) ? 1 : 0;
    a.top_k = top_k;
    a.top_p = top_p;
    const double dec = 1.44269504088896340736 / (double)temperature;
    a.dec_hi = (float)dec;
    a.dec_lo = (float)(dec - (double)a.dec_hi);
    return a;
}

int run_sample(const void *logits, spec_dtype dt, float temperature, const int32_t *top_k, const float *top_p,
               const float *draft_probs, const int32_t *draft, const float *uniforms, int B, int k, int V,
               const int32_t *draft_len, int32_t eos_id, const int32_t *remaining, int32_t *out_tokens,
               int32_t *n_accept, int32_t *n_emit, float *out_residual, uint32_t *flags, void *workspace,
               size_t workspace_bytes, void *cuda_stream)
{
    const int rc = check_sample(logits, dt, temperature, top_k, top_p, draft_probs, draft, uniforms, B, k, V,
                                draft_len, remaining, out_tokens, n_accept, n_emit, out_residual, flags, workspace,
                                workspace_bytes);
    if (rc != SPEC_OK || B == 0)
        return rc;
    return launched(launch_verify_sample(sample_args(logits, temperature, top_k, top_p, draft_probs, draft, uniforms, B,
                                                     k, V, draft_len, eos_id, remaining, out_tokens, n_accept,
                                                     n_emit, out_residual, flags, workspace),
                                         dt, (cudaStream_t)cuda_stream));
}

}  // namespace

extern "C" {

size_t spec_workspace_bytes(int B, int k, int V)
{
    if (B <= 0)
        return 0;
    k = k < 0 ? 0 : (k > SPEC_MAX_K ? SPEC_MAX_K : k);
    V = V < 1 ? 1 : V;
    return make_layout(B, k, V).total;
}

int spec_workspace_init(void *workspace, size_t bytes, void *cuda_stream)
{
    if (bytes == 0)
        return SPEC_OK;
    if (!workspace)
        return SPEC_EWORKSPACE;
    return launched(cudaMemsetAsync(workspace, 0, bytes, (cudaStream_t)cuda_stream));
}

const char *spec_status_str(int status)
{
    switch (status) {
    case SPEC_OK:
        return "ok";
    case SPEC_EINVAL:
        return "invalid argument (null pointer, negative size or k out of range)";
    case SPEC_EDTYPE:
        return "unknown spec_dtype";
    case SPEC_EWORKSPACE:
        return "workspace missing, misaligned (256 B) or smaller than spec_workspace_bytes()";
    case SPEC_ECUDA:
        return "a CUDA launch failed";
    case SPEC_EALIGN:
        return "a pointer lacks the alignment of its element type";
    case SPEC_ESCRATCH:
        return "sizes need more scratch than the library's built-in SPEC_STATIC_SCRATCH_BYTES";
    default:
        return "unknown status";
    }
}

int spec_verify_greedy(const void *target_logits, spec_dtype dt, int B, int k, int V,
                       const int32_t *draft_tokens, const int32_t *draft_len, int32_t eos_id,
                       const int32_t *remaining, int32_t *out_tokens, int32_t *n_accept, int32_t *n_emit,
                       void *workspace, size_t workspace_bytes, void *cuda_stream)
{
    const int rc = check_greedy(target_logits, dt, B, k, V, draft_tokens, draft_len, remaining, out_tokens, n_accept,
                                n_emit, workspace, workspace_bytes);
    if (rc != SPEC_OK || B == 0)
        return rc;
    return launched(launch_verify_greedy(verify_args(target_logits, B, k, V, draft_tokens, draft_len, eos_id, remaining,
                                                     out_tokens, n_accept, n_emit, workspace),
                                         dt, (cudaStream_t)cuda_stream));
}

int spec_verify_sample(const void *target_logits, spec_dtype dt, float temperature, const float *draft_probs,
                       const int32_t *draft_tokens, const float *uniforms, int B, int k, int V,
                       const int32_t *draft_len, int32_t eos_id, const int32_t *remaining, int32_t *out_tokens,
                       int32_t *n_accept, int32_t *n_emit, float *out_residual, uint32_t *flags,
                       void *workspace, size_t workspace_bytes, void *cuda_stream)
{
    return run_sample(target_logits, dt, temperature, nullptr, nullptr, draft_probs, draft_tokens, uniforms,
                              B, k, V, draft_len, eos_id, remaining, out_tokens, n_accept, n_emit, out_residual,
                              flags, workspace, workspace_bytes, cuda_stream);
}

int spec_verify_sample_filtered(const void *target_logits, spec_dtype dt, float temperature, const int32_t *top_k,
                                const float *top_p, const float *draft_probs, const int32_t *draft_tokens,
                                const float *uniforms, int B, int k, int V, const int32_t *draft_len,
                                int32_t eos_id, const int32_t *remaining, int32_t *out_tokens, int32_t *n_accept,
                                int32_t *n_emit, float *out_residual, uint32_t *flags, void *workspace,
                                size_t workspace_bytes, void *cuda_stream)
{
    return run_sample(target_logits, dt, temperature, top_k, top_p, draft_probs, draft_tokens, uniforms, B,
                              k, V, draft_len, eos_id, remaining, out_tokens, n_accept, n_emit, out_residual, flags,
                              workspace, workspace_bytes, cuda_stream);
}

}  // extern "C"

namespace {

// argument checks of a realignment over `caches` (nothing launched)
int check_realign(const spec_kv_cache *caches, int n_caches, int B, int S, const int32_t *len, const int32_t *pad,
                  const int32_t *n_emit, const int32_t *len_new, const int32_t *pad_new, const int32_t *width_new,
                  const int32_t *err, void *workspace, size_t workspace_bytes)
{
    if (!caches || n_caches < 1 || n_caches > SPEC_MAX_CACHES || B < 0 || S < 1)
        return SPEC_EINVAL;
    for (int c = 0; c < n_caches; ++c) {
        const spec_kv_cache &kc = caches[c];
        if (kc.L < 1 || kc.H < 1 || kc.D < 1)
            return SPEC_EINVAL;
        if (!dtype_ok(kc.dt))
            return SPEC_EDTYPE;
        if ((long long)B * kc.L * 2 * kc.H > INT_MAX)
            return SPEC_EINVAL;
    }
    if (B == 0)
        return SPEC_OK;
    if (!len || !pad || !n_emit || !len_new || !pad_new || !width_new || !err)
        return SPEC_EINVAL;
    for (int c = 0; c < n_caches; ++c)
        if (!caches[c].kv)
            return SPEC_EINVAL;
    for (int c = 0; c < n_caches; ++c)
        if (!aligned(caches[c].kv, dtype_bytes(caches[c].dt)))
            return SPEC_EALIGN;
    if (!aligned(len, 4) || !aligned(pad, 4) || !aligned(n_emit, 4) || !aligned(len_new, 4) || !aligned(pad_new, 4) ||
        !aligned(width_new, 4) || !aligned(err, 4))
        return SPEC_EALIGN;
    return check_workspace(workspace, workspace_bytes, spec_workspace_bytes(B, 0, 1));
}

cudaError_t start_realign(const spec_kv_cache *caches, int n_caches, int B, int S, const int32_t *len,
                          const int32_t *pad, const int32_t *n_emit, int32_t *len_new, int32_t *pad_new,
                          int32_t *width_new, int32_t *err, void *workspace, cudaStream_t st)
{
    RealignArgs a{};
    for (int c = 0; c < n_caches; ++c)
        a.cache[c] = CacheDesc{caches[c].kv, dtype_bytes(caches[c].dt), caches[c].L, caches[c].H, caches[c].D};
    a.n_caches = n_caches;
    a.B = B;
    a.S = S;
    a.len = len;
    a.pad = pad;
    a.n_emit = n_emit;
    a.len_new = len_new;
    a.pad_new = pad_new;
    a.width_new = width_new;
    a.err = err;
    a.ws = workspace;
    return launch_realign(a, st);
}

int check_pos_mask(int B, int S, const int32_t *pad_old, const int32_t *pad_new, const int32_t *pos,
                   const uint8_t *mask)
{
    if (B < 0 || S < 0 || B > 65535)
        return SPEC_EINVAL;
    if (B == 0 || S == 0)
        return SPEC_OK;
    if (!pad_new || !pos || !mask || (pad_old && pad_old == pad_new))
        return SPEC_EINVAL;
    if (!aligned(pad_new, 4) || !aligned(pos, 4) || (pad_old && !aligned(pad_old, 4)))
        return SPEC_EALIGN;
    return SPEC_OK;
}

}  // namespace

extern "C" {

int spec_realign_kv_multi(const spec_kv_cache *caches, int n_caches, int B, int S, const int32_t *len,
                          const int32_t *pad, const int32_t *n_emit, int32_t *len_new, int32_t *pad_new,
                          int32_t *width_new, int32_t *err, void *workspace, size_t workspace_bytes,
                          void *cuda_stream)
{
    const int rc = check_realign(caches, n_caches, B, S, len, pad, n_emit, len_new, pad_new, width_new, err,
                                 workspace, workspace_bytes);
    if (rc != SPEC_OK || B == 0)
        return rc;
    return launched(start_realign(caches, n_caches, B, S, len, pad, n_emit, len_new, pad_new, width_new, err,
                                  workspace, (cudaStream_t)cuda_stream));
}

int spec_realign_kv(void *kv, spec_dtype dt, int L, int B, int H, int S, int D, const int32_t *len,
                    const int32_t *pad, const int32_t *n_emit, int32_t *len_new, int32_t *pad_new,
                    int32_t *width_new, int32_t *err, void *workspace, size_t workspace_bytes, void *cuda_stream)
{
    if (B < 0 || L < 1 || H < 1 || S < 1 || D < 1)
        return SPEC_EINVAL;
    if (!dtype_ok(dt))
        return SPEC_EDTYPE;
    if (B == 0)
        return SPEC_OK;
    if (!kv)
        return SPEC_EINVAL;
    const spec_kv_cache one = {kv, dt, L, H, D};
    return spec_realign_kv_multi(&one, 1, B, S, len, pad, n_emit, len_new, pad_new, width_new, err, workspace,
                                 workspace_bytes, cuda_stream);
}

int spec_rebuild_pos_mask(int B, int S, const int32_t *pad_old, const int32_t *pad_new, int32_t *pos,
                          uint8_t *mask, void *cuda_stream)
{
    const int rc = check_pos_mask(B, S, pad_old, pad_new, pos, mask);
    if (rc != SPEC_OK || B == 0 || S == 0)
        return rc;
    return launched(launch_pos_mask(B, S, pad_old, pad_new, pos, mask, (cudaStream_t)cuda_stream));
}

int spec_group_by_length(int N, const int32_t *len, const uint8_t *active, int B, int32_t *out_idx,
                         int32_t *out_count_equal, int32_t *out_group_len, void *cuda_stream)
{
    if (N < 0 || N > SPEC_MAX_GROUP_N || B < 0)
        return SPEC_EINVAL;
    if ((N > 0 && !len) || (B > 0 && !out_idx) || !out_count_equal || !out_group_len)
        return SPEC_EINVAL;
    if ((len && !aligned(len, 4)) || (out_idx && !aligned(out_idx, 4)) || !aligned(out_count_equal, 4) ||
        !aligned(out_group_len, 4))
        return SPEC_EALIGN;
    return launched(
        launch_group(N, len, active, B, out_idx, out_count_equal, out_group_len, (cudaStream_t)cuda_stream));
}

int spec_commit_ragged(int N, int32_t *pool_len, int B, const int32_t *idx, const int32_t *n_emit, int S, int32_t *err,
                       void *cuda_stream)
{
    if (N < 0 || N > SPEC_MAX_POOL || B < 0 || S < 1)
        return SPEC_EINVAL;
    if (B == 0)
        return SPEC_OK;
    if (!pool_len || !idx || !n_emit || !err)
        return SPEC_EINVAL;
    if (!aligned(pool_len, 4) || !aligned(idx, 4) || !aligned(n_emit, 4) || !aligned(err, 4))
        return SPEC_EALIGN;
    return launched(launch_commit_ragged(N, pool_len, B, idx, n_emit, S, err, (cudaStream_t)cuda_stream));
}

static int pool_common(const void *src, const void *dst, int dt, int L, int N, int B, int H, int S, int D,
                       const int32_t *idx, const int32_t *err, void *workspace, size_t workspace_bytes)
{
    if (L < 1 || N < 0 || N > SPEC_MAX_POOL || B < 0 || H < 1 || S < 1 || D < 1)
        return SPEC_EINVAL;
    if (!dtype_ok(dt))
        return SPEC_EDTYPE;
    if (B == 0)
        return SPEC_OK;
    if (!src || !dst || !idx || !err)
        return SPEC_EINVAL;
    if ((long long)(B > N ? B : N) * L * 2 * H > INT_MAX)
        return SPEC_EINVAL;
    if (!aligned(src, dtype_bytes(dt)) || !aligned(dst, dtype_bytes(dt)) || !aligned(idx, 4) || !aligned(err, 4))
        return SPEC_EALIGN;
    return check_workspace(workspace, workspace_bytes, spec_workspace_bytes(B, 0, 1));
}

int spec_repad_gather(const void *pool, void *batch, spec_dtype dt, int L, int N, int B, int H, int S, int D,
                      const int32_t *idx, const int32_t *pool_len, int32_t *len_out, int32_t *pad_out,
                      int32_t *width_out, int32_t *err, void *workspace, size_t workspace_bytes, void *cuda_stream)
{
    int rc = pool_common(pool, batch, dt, L, N, B, H, S, D, idx, err, workspace, workspace_bytes);
    if (rc != SPEC_OK || B == 0)
        return rc;
    if (!pool_len || !len_out || !pad_out || !width_out)
        return SPEC_EINVAL;
    if (!aligned(pool_len, 4) || !aligned(len_out, 4) || !aligned(pad_out, 4) || !aligned(width_out, 4))
        return SPEC_EALIGN;
    PoolArgs a{};
    a.src = pool;
    a.dst = batch;
    a.elt_bytes = dtype_bytes(dt);
    a.L = L;
    a.N = N;
    a.B = B;
    a.H = H;
    a.S = S;
    a.D = D;
    a.repad = 1;
    a.idx = idx;
    a.pool_len = pool_len;
    a.len_out = len_out;
    a.pad_out = pad_out;
    a.width_out = width_out;
    a.err = err;
    a.ws = workspace;
    return launched(launch_pool_copy(a, (cudaStream_t)cuda_stream));
}

int spec_unpad_scatter(const void *batch, void *pool, spec_dtype dt, int L, int N, int B, int H, int S, int D,
                       const int32_t *idx, const int32_t *len, const int32_t *pad, const int32_t *n_emit,
                       int32_t *pool_len, int32_t *err, void *workspace, size_t workspace_bytes, void *cuda_stream)
{
    int rc = pool_common(batch, pool, dt, L, N, B, H, S, D, idx, err, workspace, workspace_bytes);
    if (rc != SPEC_OK || B == 0)
        return rc;
    if (!len || !pad || !pool_len)
        return SPEC_EINVAL;
    if (!aligned(len, 4) || !aligned(pad, 4) || !aligned(pool_len, 4) || (n_emit && !aligned(n_emit, 4)))
        return SPEC_EALIGN;
    PoolArgs a{};
    a.src = batch;
    a.dst = pool;
    a.elt_bytes = dtype_bytes(dt);
    a.L = L;
    a.N = N;
    a.B = B;
    a.H = H;
    a.S = S;
    a.D = D;
    a.repad = 0;
    a.idx = idx;
    a.len = len;
    a.pad = pad;
    a.n_emit = n_emit;
    a.pool_len_out = pool_len;
    a.err = err;
    a.ws = workspace;
    return launched(launch_pool_copy(a, (cudaStream_t)cuda_stream));
}

// ---- one whole round ------------------------------------------------------
// verify, realign every cache by one plan, rebuild positions and mask: every
// argument is checked before the first launch; the launches follow one
// another on the stream (the realignment reads n_emit on the device).
int spec_round_greedy(const void *target_logits, spec_dtype dt, int B, int k, int V, const int32_t *draft_tokens,
                      const int32_t *draft_len, int32_t eos_id, const int32_t *remaining, const spec_kv_cache *caches,
                      int n_caches, int S, const int32_t *len, const int32_t *pad, int32_t *pos, uint8_t *mask,
                      int32_t *out_tokens, int32_t *n_accept, int32_t *n_emit, int32_t *len_new, int32_t *pad_new,
                      int32_t *width_new, int32_t *err, void *workspace, size_t workspace_bytes, void *cuda_stream)
{
    int rc = check_greedy(target_logits, dt, B, k, V, draft_tokens, draft_len, remaining, out_tokens, n_accept, n_emit,
                          workspace, workspace_bytes);
    if (rc == SPEC_OK)
        rc = check_realign(caches, n_caches, B, S, len, pad, n_emit, len_new, pad_new, width_new, err, workspace,
                           workspace_bytes);
    if (rc == SPEC_OK)
        rc = check_pos_mask(B, S, pad, pad_new, pos, mask);
    if (rc != SPEC_OK || B == 0)
        return rc;
    const cudaStream_t st = (cudaStream_t)cuda_stream;
    cudaError_t e = launch_verify_greedy(verify_args(target_logits, B, k, V, draft_tokens, draft_len, eos_id,
                                                     remaining, out_tokens, n_accept, n_emit, workspace),
                                         dt, st);
    if (e == cudaSuccess)
        e = start_realign(caches, n_caches, B, S, len, pad, n_emit, len_new, pad_new, width_new, err, workspace, st);
    if (e == cudaSuccess)
        e = launch_pos_mask(B, S, pad, pad_new, pos, mask, st);
    return launched(e);
}

int spec_round_sample(const void *target_logits, spec_dtype dt, float temperature, const int32_t *top_k,
                      const float *top_p, const float *draft_probs, const int32_t *draft_tokens,
                      const float *uniforms, int B, int k, int V, const int32_t *draft_len, int32_t eos_id,
                      const int32_t *remaining, const spec_kv_cache *caches, int n_caches, int S, const int32_t *len,
                      const int32_t *pad, int32_t *pos, uint8_t *mask, int32_t *out_tokens, int32_t *n_accept,
                      int32_t *n_emit, float *out_residual, uint32_t *flags, int32_t *len_new, int32_t *pad_new,
                      int32_t *width_new, int32_t *err, void *workspace, size_t workspace_bytes, void *cuda_stream)
{
    int rc = check_sample(target_logits, dt, temperature, top_k, top_p, draft_probs, draft_tokens, uniforms, B, k, V,
                          draft_len, remaining, out_tokens, n_accept, n_emit, out_residual, flags, workspace,
                          workspace_bytes);
    if (rc == SPEC_OK)
        rc = check_realign(caches, n_caches, B, S, len, pad, n_emit, len_new, pad_new, width_new, err, workspace,
                           workspace_bytes);
    if (rc == SPEC_OK)
        rc = check_pos_mask(B, S, pad, pad_new, pos, mask);
    if (rc != SPEC_OK || B == 0)
        return rc;
    const cudaStream_t st = (cudaStream_t)cuda_stream;
    cudaError_t e = launch_verify_sample(sample_args(target_logits, temperature, top_k, top_p, draft_probs, draft_tokens,
                                                     uniforms, B, k, V, draft_len, eos_id, remaining, out_tokens,
                                                     n_accept, n_emit, out_residual, flags, workspace),
                                         dt, st);
    if (e == cudaSuccess)
        e = start_realign(caches, n_caches, B, S, len, pad, n_emit, len_new, pad_new, width_new, err, workspace, st);
    if (e == cudaSuccess)
        e = launch_pos_mask(B, S, pad, pad_new, pos, mask, st);
    return launched(e);
}

}  // extern "C"
