// verify_static.cu -- spec_verify_greedy_static: greedy verification with
// its scratch in a device array built into the library, for callers that
// cannot allocate device memory when they call in (see specverify.h).
//
// The array lives for as long as the library is loaded, on every device that
// loads it.  Host code only ever sees a host-side stand-in for its name; the
// device address is looked up once per device with cudaGetSymbolAddress and
// cached.  Calls share the array: the counter region is cleared on the
// caller's stream before each launch, everything else is written before it
// is read by the same call.
#include <mutex>

#include "spec_common.cuh"
#include "spec_launch.h"

using namespace spec;

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[SPEC_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];
std::mutex g_setup_mutex;

// device address of the scratch on the current device (looked up once); a
// stream of another device is refused: the clear and the launch would run
// there against this device's array
int scratch_on_current_device(cudaStream_t st, void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return SPEC_ECUDA;
    if (st != nullptr && st != cudaStreamLegacy && st != cudaStreamPerThread) {
        int sdev = -1;
        if (cudaStreamGetDevice(st, &sdev) != cudaSuccess)
            return SPEC_ECUDA;
        if (sdev != dev)
            return SPEC_EINVAL;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p)
            return SPEC_ECUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SPEC_OK;
}

bool aligned_to(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int spec_verify_greedy_static(const void *target_logits, spec_dtype dt, int B, int k, int V,
                                         const int32_t *draft_tokens, const int32_t *draft_len, int32_t eos_id,
                                         const int32_t *remaining, int32_t *out_tokens, int32_t *n_accept,
                                         int32_t *n_emit, void *cuda_stream)
{
    if (B < 0 || k < 0 || k > SPEC_MAX_K || V < 1)
        return SPEC_EINVAL;
    if (dt != SPEC_F32 && dt != SPEC_BF16 && dt != SPEC_F16)
        return SPEC_EDTYPE;
    if (B == 0)
        return SPEC_OK;
    if (!target_logits || (k > 0 && !draft_tokens) || !out_tokens || !n_accept || !n_emit)
        return SPEC_EINVAL;
    if ((long long)B * (k + 1) * verify_chunks(B, k, V) > 0x7FFFFFFFLL)
        return SPEC_EINVAL;
    if (!aligned_to(target_logits, dt == SPEC_F32 ? 4 : 2) || !aligned_to(out_tokens, 4) ||
        !aligned_to(n_accept, 4) || !aligned_to(n_emit, 4) || (draft_tokens && !aligned_to(draft_tokens, 4)) ||
        (draft_len && !aligned_to(draft_len, 4)) || (remaining && !aligned_to(remaining, 4)))
        return SPEC_EALIGN;
    const Layout lay = make_layout(B, k, V);
    if (lay.total > SPEC_STATIC_SCRATCH_BYTES)
        return SPEC_ESCRATCH;
    cudaStream_t st = (cudaStream_t)cuda_stream;
    void *scratch = nullptr;
    const int rc = scratch_on_current_device(st, &scratch);
    if (rc != SPEC_OK)
        return rc;
    if (cudaMemsetAsync(static_cast<char *>(scratch) + lay.zero_begin, 0, lay.zero_end - lay.zero_begin, st) !=
        cudaSuccess)
        return SPEC_ECUDA;
    VerifyArgs a{};
    a.logits = target_logits;
    a.B = B;
    a.k = k;
    a.V = V;
    a.draft = draft_tokens;
    a.draft_len = draft_len;
    a.eos = eos_id;
    a.remaining = remaining;
    a.out_tokens = out_tokens;
    a.n_accept = n_accept;
    a.n_emit = n_emit;
    a.ws = scratch;
    return launch_verify_greedy(a, dt, st) == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}
