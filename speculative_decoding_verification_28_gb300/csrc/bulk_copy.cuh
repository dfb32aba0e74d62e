// bulk_copy.cuh -- inline PTX for mbarriers and 1-D bulk copies
// (cp.async.bulk, the non-tensor TMA path) on sm_103a, used by the KV shift
// and the pool copies.
#pragma once

#include <stdint.h>

namespace spec {

// ---------------------------------------------------------------------------
// mbarrier + 1-D bulk copy (cp.async.bulk) wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// one bounded probe of the barrier phase; true once phase `parity` completed
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000000;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// global -> shared bulk copy completing on an mbarrier
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// shared -> global bulk copy tracked by bulk async-groups
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src_smem, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_addr(src_smem)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------------------
// A copy engine on one thread: runs of bytes staged global -> shared ->
// global through kBulkStages stages of kBulkTile bytes.  Loads run up to
// kBulkStages - 1 tiles ahead of the stores; each store is issued after its
// tile's load completed on the stage's mbarrier, strictly in tile order, and
// a stage is reloaded only after the store that read it has finished reading.
// The tile source decides the order, so an in-place move that takes its tiles
// from the end the run moves towards never overwrites bytes not yet loaded.
// ---------------------------------------------------------------------------
constexpr int kBulkStages = 4;
constexpr int kBulkTile = 48 * 1024;  // bytes per stage
constexpr int kBulkSmem = kBulkStages * kBulkTile;
constexpr int kBulkWaitLimit = 4000;  // probes of up to ~1 ms each before giving up

// tiles of one contiguous run: ascending, or descending (from the top) when
// `desc` (an in-place move towards higher addresses)
struct RunTiles {
    const char *src;
    char *dst;
    long long nbytes, done;
    int desc;
    __device__ bool next(const char *&s, char *&d, uint32_t &bytes)
    {
        if (done >= nbytes)
            return false;
        long long take = nbytes - done;
        if (take > kBulkTile)
            take = kBulkTile;
        const long long lo = desc ? nbytes - done - take : done;
        s = src + lo;
        d = dst + lo;
        bytes = (uint32_t)take;
        done += take;
        return true;
    }
};

template <int N>
__device__ __forceinline__ void bulk_wait_read_upto(int newer)
{
    if constexpr (N > 0) {
        if (newer >= N) {
            bulk_wait_read<N>();
            return;
        }
        bulk_wait_read_upto<N - 1>(newer);
    } else {
        bulk_wait_read<0>();
    }
}

// Copies every tile `source.next(src, dst, bytes)` yields (16-byte aligned
// addresses and sizes).  One thread.  Returns false when a bounded wait gave
// up (after waiting, bounded, for the copies still in flight).
template <class Source>
__device__ bool bulk_copy_pipeline(Source &source, unsigned char *stage_mem, uint64_t *full)
{
    for (int s = 0; s < kBulkStages; ++s)
        mbar_init(&full[s], 1);
    fence_mbar_init();
    char *dst_of[kBulkStages];
    uint32_t bytes_of[kBulkStages];
    uint32_t parity = 0;
    long long issued = 0, done = 0;
    bool more = true, failed = false;
    while (true) {
        while (more && issued - done < kBulkStages - 1) {
            const char *src;
            char *dst;
            uint32_t bytes;
            if (!source.next(src, dst, bytes)) {
                more = false;
                break;
            }
            const int s = (int)(issued % kBulkStages);
            if (issued >= kBulkStages)
                bulk_wait_read_upto<kBulkStages - 1>((int)(done - 1 - (issued - kBulkStages)));
            mbar_arrive_expect_tx(&full[s], bytes);
            bulk_g2s(stage_mem + (size_t)s * kBulkTile, src, bytes, &full[s]);
            dst_of[s] = dst;
            bytes_of[s] = bytes;
            ++issued;
        }
        if (done == issued)
            break;
        const int s = (int)(done % kBulkStages);
        const uint32_t par = (parity >> s) & 1u;
        int probes = 0;
        while (!mbar_try_wait(&full[s], par)) {
            if (++probes >= kBulkWaitLimit) {
                failed = true;
                break;
            }
        }
        if (failed)
            break;
        parity ^= 1u << s;
        bulk_s2g(dst_of[s], stage_mem + (size_t)s * kBulkTile, bytes_of[s]);
        bulk_commit();
        ++done;
    }
    if (failed) {  // wait (bounded) for the loads still in flight
        for (long long i = done; i < issued; ++i) {
            const int s = (int)(i % kBulkStages);
            const uint32_t par = (parity >> s) & 1u;
            for (int p = 0; p < kBulkWaitLimit && !mbar_try_wait(&full[s], par); ++p) {
            }
            parity ^= 1u << s;
        }
    }
    bulk_wait_all();
    return !failed;
}

// Programmatic dependent launch (griddepcontrol, sm_90+).  `dep_wait` blocks
// until the grids this one depends on have completed and their memory is
// visible (a no-op when the launch was not programmatic); `dep_release` lets
// the next programmatically launched grid start once every CTA of this grid
// has executed it or exited.
__device__ __forceinline__ void dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void dep_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace spec
