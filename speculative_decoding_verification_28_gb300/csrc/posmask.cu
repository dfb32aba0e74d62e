// posmask.cu -- position IDs and attention mask recomputed from the new
// padding after realignment, in one pass ("Correctness Forensics for Batch
// Speculative Decoding", App. B: position IDs are restored by recomputing them
// from the attention mask after repadding).
//   mask[b, s] = s >= pad'_b;   pos[b, s] = s - pad'_b there, 0 in the padding
// (cumsum(mask) - 1 clamped at 0).  Rows whose padding did not change are
// skipped.  Roofline: write-only, 5 bytes per slot of a changed row.
//
// Ordering.  The kernel is launched programmatically, so after a
// realignment it runs alongside the KV shift.  Two rules keep that safe:
//  * it reads pad_new, which the plan kernel wrote.  The shift lets its
//    dependents launch only after its own griddepcontrol.wait has returned
//    (the plan grid complete, its writes performed), so this kernel never
//    starts before those writes.
//  * every CTA ends with griddepcontrol.wait, so this grid cannot complete
//    before the grid it follows (the shift) has completed and its writes
//    are visible.  Work the caller enqueues after the round -- the next
//    forward reading the cache, a copy of the error word the shift may set
//    -- follows this grid in ordinary stream order, hence the shift too.
#include "bulk_copy.cuh"
#include "spec_common.cuh"
#include "spec_launch.h"

namespace spec {

constexpr int kPmThreads = 256;
constexpr int kPmSlots = 8;  // slots per thread on the vector path

__device__ __forceinline__ void pos_mask_row(int S, int pn, int32_t *prow, uint8_t *mrow, int vec)
{
    if (vec) {
        const int s0 = (blockIdx.x * kPmThreads + threadIdx.x) * kPmSlots;
        if (s0 >= S)
            return;
        int p[kPmSlots];
        uint32_t m[2] = {0, 0};
#pragma unroll
        for (int e = 0; e < kPmSlots; ++e) {
            const int s = s0 + e;
            const bool in = s >= pn;
            p[e] = in ? s - pn : 0;
            m[e >> 2] |= (in ? 1u : 0u) << (8 * (e & 3));
        }
        *reinterpret_cast<int4 *>(prow + s0) = make_int4(p[0], p[1], p[2], p[3]);
        *reinterpret_cast<int4 *>(prow + s0 + 4) = make_int4(p[4], p[5], p[6], p[7]);
        *reinterpret_cast<uint2 *>(mrow + s0) = make_uint2(m[0], m[1]);
    } else {
        for (int s = blockIdx.x * kPmThreads + threadIdx.x; s < S; s += gridDim.x * kPmThreads) {
            const bool in = s >= pn;
            prow[s] = in ? s - pn : 0;
            mrow[s] = in ? 1 : 0;
        }
    }
}

__global__ void __launch_bounds__(kPmThreads)
    pos_mask_kernel(int B, int S, const int32_t *pad_old, const int32_t *pad_new, int32_t *pos, uint8_t *mask,
                    int vec)
{
    const int b = blockIdx.y;
    const int pn = pad_new[b];
    if (!(pad_old && pad_old[b] == pn))
        pos_mask_row(S, pn, pos + (size_t)b * S, mask + (size_t)b * S, vec);
    // no CTA completes before the grid this one follows has completed
    if (threadIdx.x == 0)
        dep_wait();
}

cudaError_t launch_pos_mask(int B, int S, const int32_t *pad_old, const int32_t *pad_new, int32_t *pos,
                            uint8_t *mask, cudaStream_t st)
{
    const bool vec = (S % kPmSlots == 0) && (reinterpret_cast<uintptr_t>(pos) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(mask) % 8 == 0);
    const int per_block = vec ? kPmThreads * kPmSlots : kPmThreads * 4;
    // Launched programmatically: it may start while the previous kernel on
    // the stream finishes, once that kernel allows it.  The library's KV shift
    // allows it only after the plan that wrote pad_new is complete, and it
    // never touches pos or mask; a kernel that does not release dependents
    // early (any other kernel) completes first, as in an ordinary launch.
    // Either way the grid's final griddepcontrol.wait keeps it from completing
    // before that kernel.
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((S + per_block - 1) / per_block), (unsigned)B);
    cfg.blockDim = dim3(kPmThreads);
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, pos_mask_kernel, B, S, pad_old, pad_new, pos, mask, vec ? 1 : 0);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace spec
