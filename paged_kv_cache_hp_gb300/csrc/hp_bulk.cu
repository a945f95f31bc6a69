// hp_bulk.cu -- the TMA bulk-copy engine for pure data movement (gather, append and the
// per-lane layout) when every row is a multiple of 16 bytes and both bases are 16-byte
// aligned (the alignment cp.async.bulk requires).
//
// One CTA per SM owns a contiguous range of copy units (see hp_copy.cu for the units).
// Inside the CTA the work is split by role.  Resolver warps turn units into a
// double-buffered descriptor ring in shared memory (sequence by binary search over the
// unit prefix, block-table entry, source/destination offsets, bytes) and hand each batch
// over through a "full" mbarrier; they refill a buffer once the "empty" mbarrier says it
// has been consumed.  The bytes stream through a ring of shared-memory stages,
// cp.async.bulk global->shared (completion counted on the stage's mbarrier) then
// cp.async.bulk shared->global from the same stage, in one of two ways (measured on
// GB300):
//   8 KiB x 24 stages (units of 64 KiB and more): one producer thread issues both the
//               loads and the stores, keeping up to 23 loads in flight and reusing a
//               stage once all but the newest store have read shared memory;
//   16 KiB x 12 stages (units of 16-64 KiB): a loader thread (warp 0) and a storer
//               thread (warp 1).  The loader waits for a free stage, records the chunk's
//               destination and size with it and issues the load; the storer waits for
//               each stage in turn to be loaded, issues its store, and hands a stage back
//               through its "free" mbarrier once all but the newest kStoresInFlight = 8
//               stores have read shared memory, so up to 8 stores and 4 loads are in
//               flight.  After the last chunk the loader hands the storer a zero-byte
//               chunk to end on.
// (Split roles lose on 8 KiB chunks -- the storer's per-chunk wait caps the stores in
// flight -- and a single thread loses on 16-32 KiB chunks.  On the 16-64 KiB units, 16 KiB
// x 12 with 8 stores in flight beat 32 KiB x 6 with 3 (0.97 -> 0.995 of the copy
// bandwidth on 2 KiB rows, and a little better with shared prefix pages); 32 KiB x 6 with
// 4 stores reached 1.01 on the first and lost 3% on the second; 7, 9 or 10 stores of
// 16 KiB, or 5 of 32 KiB, were slower on one or both.)  Every wait is bounded (about
// 2 s of %globaltimer); a wait that runs out stores HP_ERR_TIMEOUT in *d_status, stops
// issuing and lets the loads in flight land (again bounded) before the CTA's shared
// memory goes.
#include <cuda_runtime.h>

#include <algorithm>

#include "hp_internal.cuh"
#include "hp_resolve.cuh"
#include "hp_tma.cuh"

namespace hp {
namespace {

using namespace tma;

#ifndef HP_BULK_STORE_EVICT_FIRST
#define HP_BULK_STORE_EVICT_FIRST 0
#endif

constexpr int kResolvers = 96;         // resolver threads (warps 1-3, or 2-4 with split roles)
constexpr int kBatch = 256;            // units per descriptor buffer

struct Desc {
    unsigned long long src[2][kBatch];
    unsigned long long dst[2][kBatch];
    unsigned long long bytes[2][kBatch];
};

// The ring holds kStages stages of kStage bytes (192 KiB either way): 8 KiB stages
// suit copy units of 64 KiB and more, 16 KiB stages units of 16-64 KiB (measured).
// STALL: the HP_TEST_STALL variant (a separate instantiation, so the copy path carries
// no test check in its per-chunk loop).
template <uint32_t kStage> __host__ __device__ constexpr int threads_for()
{
    return kStage >= 16384 ? 160 : 128;
}

template <int MODE, typename IndexT, uint32_t kStage, int kStages, bool STALL = false>
__global__ void __launch_bounds__(threads_for<kStage>(), 1) bulk_kernel(const CopyArgs a)
{
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) unsigned long long loaded_bar[kStages], free_bar[kStages];
    __shared__ __align__(8) unsigned long long full_bar[2], empty_bar[2];
    __shared__ Desc desc;
    __shared__ unsigned long long chunk_dst[kStages];
    __shared__ uint32_t chunk_bytes[kStages];

    // split roles (loader and storer threads) for 16 KiB stages, one producer for 8 KiB
    constexpr bool kSplit = kStage >= 16384;
    constexpr int kFirstResolver = kSplit ? 64 : 32;
    static_assert(threads_for<kStage>() - kFirstResolver == kResolvers, "96 resolvers");
    // split roles: stores left reading shared memory before their stages are handed back;
    // fewer than kStages, so the loader always has a stage it can wait for without a cycle
    constexpr int kStoresInFlight = 8;
    static_assert(kStoresInFlight < kStages, "a free stage must not wait on a later load");
    uint64_t total;
    if (MODE == kGather || MODE == kAppend) {
        pdl_wait();  // the plan (and table check) before this launch must be complete
        if (a.hdr->verdict != kVerdictOk) return;  // the plan rejected the batch
        total = a.hdr->total_units;
    } else {
        total = a.lane_units;
    }
    const uint64_t G = gridDim.x, b = blockIdx.x;
    const uint64_t per = total / G, rem = total % G;
    const uint64_t lo = b * per + umin(b, rem);
    const uint64_t hi = lo + per + (b < rem ? 1 : 0);
    if (lo >= hi) return;
    const uint64_t nbatches = (hi - lo + kBatch - 1) / kBatch;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&loaded_bar[i]), 1);
            if (kSplit) mbar_init(smem_u32(&free_bar[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&full_bar[i]), kResolvers);
            mbar_init(smem_u32(&empty_bar[i]), 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (threadIdx.x >= kFirstResolver) {
        // ---------------------------------------------------------------- resolvers
        const int r = threadIdx.x - kFirstResolver;
        for (uint64_t bt = 0; bt < nbatches; ++bt) {
            const int buf = (int)(bt & 1);
            if (bt >= 2 && !mbar_wait(smem_u32(&empty_bar[buf]), (uint32_t)((bt / 2 - 1) & 1)))
                return;  // the loader stopped (it has reported why)
            const uint64_t base = lo + bt * kBatch;
            for (int i = r; i < kBatch; i += kResolvers) {
                const uint64_t u = base + i;
                if (u < hi) {
                    const Unit un = resolve<MODE, IndexT>(a, u);
                    desc.src[buf][i] = un.src;
                    desc.dst[buf][i] = un.dst;
                    desc.bytes[buf][i] = (unsigned long long)un.rows * a.row_bytes;
                }
            }
            mbar_arrive(smem_u32(&full_bar[buf]));
        }
        return;
    }
    const uint32_t ring0 = smem_u32(ring);
    if constexpr (kSplit) {
        if (threadIdx.x == 32) {
            // ------------------------------------------------------------------- storer
            // Chunk c sits in stage c % kStages, loaded in round c / kStages.  After the store
            // of chunk c is issued, the wait for all but the newest kStoresInFlight stores
            // to have read shared memory frees the stage of chunk c - kStoresInFlight.
            unsigned long long policy = 0;
#if HP_BULK_STORE_EVICT_FIRST
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
#endif
            uint64_t c = 0;
            bool ok = true;
            while (true) {
                const uint32_t st = (uint32_t)(c % kStages);
                if (!mbar_wait(smem_u32(&loaded_bar[st]), (uint32_t)((c / kStages) & 1))) {
                    ok = false;
                    break;
                }
                const uint32_t bytes = chunk_bytes[st];
                if (bytes == 0) break;  // the loader's end mark
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                bulk_store(a.dst + chunk_dst[st], ring0 + st * kStage, bytes, policy);
                if (c >= kStoresInFlight) {
                    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kStoresInFlight) : "memory");
                    mbar_arrive(smem_u32(&free_bar[(c - kStoresInFlight) % kStages]));
                }
                ++c;
            }
            if (!ok) report(a.d_status, HP_ERR_TIMEOUT);
            // free the stages of the last stores once they have read shared memory
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            for (uint64_t k = c > kStoresInFlight ? c - kStoresInFlight : 0; k < c; ++k)
                mbar_arrive(smem_u32(&free_bar[k % kStages]));
            asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
            return;
        }
        if (threadIdx.x != 0) return;

        // --------------------------------------------------------------------- loader
        // Chunk L goes to stage L % kStages once the store of chunk L - kStages has freed it
        // (free phase L / kStages - 1).  A batch's descriptor buffer is handed back as soon
        // as its last load is issued.
        uint64_t L = 0;     // chunks issued so far
        uint64_t lb = 0;    // batch of the load cursor
        uint32_t li = 0;    // unit of the load cursor within its batch
        uint64_t loff = 0;  // byte offset of the load cursor within that unit
        bool have = false;  // descriptors of batch lb observed
        bool ok = true;
        while (lb < nbatches) {
            const int buf = (int)(lb & 1);
            if (!have) {
                if (!mbar_wait(smem_u32(&full_bar[buf]), (uint32_t)((lb / 2) & 1))) {
                    ok = false;
                    break;
                }
                have = true;
                li = 0;
                loff = 0;
            }
            if (li == umin(kBatch, hi - lo - lb * kBatch)) {
                mbar_arrive(smem_u32(&empty_bar[buf]));  // buffer free for batch lb + 2
                ++lb;
                have = false;
                continue;
            }
            const unsigned long long nbytes = desc.bytes[buf][li];
            if (loff >= nbytes) {
                ++li;
                loff = 0;
                continue;
            }
            const uint32_t bytes = (uint32_t)umin(kStage, nbytes - loff);
            const uint32_t st = (uint32_t)(L % kStages);
            if (L >= kStages &&
                !mbar_wait(smem_u32(&free_bar[st]), (uint32_t)((L / kStages - 1) & 1))) {
                ok = false;
                break;
            }
            chunk_dst[st] = desc.dst[buf][li] + loff;
            chunk_bytes[st] = bytes;
            const uint32_t bar = smem_u32(&loaded_bar[st]);
            mbar_expect_tx(bar, bytes);
            if (!STALL || L != 0)  // HP_TEST_STALL: the first load is never issued
                bulk_load(ring0 + st * kStage, a.src + desc.src[buf][li] + loff, bytes, bar);
            ++L;
            loff += bytes;
        }
        if (ok) {
            // the end mark: a zero-byte chunk in the next stage, once that stage is free
            const uint32_t st = (uint32_t)(L % kStages);
            if (L >= kStages &&
                !mbar_wait(smem_u32(&free_bar[st]), (uint32_t)((L / kStages - 1) & 1)))
                ok = false;
            else {
                chunk_bytes[st] = 0;
                mbar_arrive(smem_u32(&loaded_bar[st]));
            }
        }
        if (!ok) {
            report(a.d_status, HP_ERR_TIMEOUT);
            // let this side's loads in flight land before the CTA's shared memory goes: the
            // last kStages chunks issued (each wait bounded)
            for (uint64_t k = L > kStages ? L - kStages : 0; k < L; ++k)
                mbar_wait(smem_u32(&loaded_bar[k % kStages]), (uint32_t)((k / kStages) & 1));
        }
    } else {
        if (threadIdx.x != 0) return;

        // -------------------------------------------------------------------- producer
        // Loads walk the units of batch lb (descriptors in buffer lb & 1); each load records
        // its destination and size with its stage, so stores need no descriptors.  A
        // batch's buffer is handed back as soon as its last load is issued.
        uint64_t L = 0, S = 0;   // chunks loaded / stored so far
        uint64_t lb = 0;         // batch of the load cursor
        uint32_t li = 0;         // unit of the load cursor within its batch
        uint64_t loff = 0;       // byte offset of the load cursor within that unit
        bool have = false;       // descriptors of batch lb observed
        bool ok = true;
        unsigned long long policy = 0;
#if HP_BULK_STORE_EVICT_FIRST
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
#endif
        while (true) {
            while (lb < nbatches && L - S < kStages - 1) {
                const int buf = (int)(lb & 1);
                if (!have) {
                    const uint32_t fb = smem_u32(&full_bar[buf]);
                    const uint32_t par = (uint32_t)((lb / 2) & 1);
                    // block only when nothing else can progress (no chunk left to store)
                    if (!(S == L ? mbar_wait(fb, par) : mbar_try_wait(fb, par))) {
                        if (S == L) ok = false;
                        break;
                    }
                    have = true;
                    li = 0;
                    loff = 0;
                }
                if (li == umin(kBatch, hi - lo - lb * kBatch)) {
                    mbar_arrive(smem_u32(&empty_bar[buf]));  // buffer free for batch lb + 2
                    ++lb;
                    have = false;
                    continue;
                }
                const unsigned long long nbytes = desc.bytes[buf][li];
                if (loff >= nbytes) {
                    ++li;
                    loff = 0;
                    continue;
                }
                const uint32_t bytes = (uint32_t)umin(kStage, nbytes - loff);
                const uint32_t st = (uint32_t)(L % kStages);
                // chunk L - kStages used this stage; its store is at least one group old
                if (L >= kStages) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                chunk_dst[st] = desc.dst[buf][li] + loff;
                chunk_bytes[st] = bytes;
                const uint32_t bar = smem_u32(&loaded_bar[st]);
                mbar_expect_tx(bar, bytes);
                if (!STALL || L != 0)  // HP_TEST_STALL: the first load is never issued
                    bulk_load(ring0 + st * kStage, a.src + desc.src[buf][li] + loff, bytes, bar);
                ++L;
                loff += bytes;
            }
            if (!ok) break;
            if (S == L) {
                if (lb >= nbatches) break;  // everything loaded and stored
                continue;                   // blocks on the next batch's descriptors above
            }
            const uint32_t st = (uint32_t)(S % kStages);
            if (!mbar_wait(smem_u32(&loaded_bar[st]), (uint32_t)((S / kStages) & 1))) {
                ok = false;
                break;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            bulk_store(a.dst + chunk_dst[st], ring0 + st * kStage, chunk_bytes[st], policy);
            ++S;
        }
        if (!ok) {
            report(a.d_status, HP_ERR_TIMEOUT);
            // let every load in flight land before the CTA's shared memory goes (each wait
            // bounded; a stage that never completes costs one more wait limit)
            for (; S < L; ++S)
                mbar_wait(smem_u32(&loaded_bar[S % kStages]), (uint32_t)((S / kStages) & 1));
        }
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
}

template <int MODE, typename IndexT, uint32_t kStage, int kStages, bool STALL = false>
int launch_t(const CopyArgs& a, cudaStream_t st)
{
    auto kern = bulk_kernel<MODE, IndexT, kStage, kStages, STALL>;
    const int smem = kStages * kStage;
    int dev = 0;
    const int sms = current_sms(&dev);
    if (sms == 0 ||
        !allow_dynamic_smem<bulk_kernel<MODE, IndexT, kStage, kStages, STALL>>(dev, smem))
        return HP_ERR_CUDA;
    uint64_t grid = (uint64_t)sms;
    if (host_counted(MODE)) grid = std::min<uint64_t>(grid, a.lane_units);
    if (grid == 0) return HP_OK;
    if (host_counted(MODE)) {
        kern<<<(unsigned)grid, threads_for<kStage>(), smem, st>>>(a);
        return cudaGetLastError() == cudaSuccess ? HP_OK : HP_ERR_CUDA;
    }
    return launch_dependent(kern, (unsigned)grid, threads_for<kStage>(), (size_t)smem, st, a) ==
                   cudaSuccess
               ? HP_OK
               : HP_ERR_CUDA;
}

template <int MODE, typename IndexT>
int launch_ring(const CopyArgs& a, int big_stages, cudaStream_t st)
{
    if constexpr (MODE == kGather) {
        if (a.test_stall)
            return big_stages ? launch_t<MODE, IndexT, 16384, 12, true>(a, st)
                              : launch_t<MODE, IndexT, 8192, 24, true>(a, st);
    }
    return big_stages ? launch_t<MODE, IndexT, 16384, 12>(a, st)
                      : launch_t<MODE, IndexT, 8192, 24>(a, st);
}

}  // namespace

int launch_bulk(CopyMode mode, int index_u64, const CopyArgs& a, int big_stages, void* stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (mode) {
    case kGather:
        return index_u64 ? launch_ring<kGather, unsigned long long>(a, big_stages, st)
                         : launch_ring<kGather, unsigned int>(a, big_stages, st);
    case kAppend:
        return index_u64 ? launch_ring<kAppend, unsigned long long>(a, big_stages, st)
                         : launch_ring<kAppend, unsigned int>(a, big_stages, st);
    case kLaneGather:
        return launch_ring<kLaneGather, unsigned long long>(a, big_stages, st);
    case kLaneAppend:
        return launch_ring<kLaneAppend, unsigned long long>(a, big_stages, st);
    case kCopyPages:
        return index_u64 ? launch_ring<kCopyPages, unsigned long long>(a, big_stages, st)
                         : launch_ring<kCopyPages, unsigned int>(a, big_stages, st);
    default:
        return HP_ERR_ARG;
    }
}

}  // namespace hp
