// hp_writer.cu -- writer-side kernels: zeroing the slots no sequence reads before the cache
// crosses a trust or tenant boundary ("Block-Paged Layout -- Hurray Format Specification",
// Partial trailing page: a writer should zero the unused slots past a sequence's count).
//
// After the plan has validated the descriptor:
//   live_kernel  one thread per block-table entry k: its sequence s (binary search over
//                seq_ptr), its logical page j = k - seq_ptr[s], and the tokens of s that
//                page holds, min(page_size, len_s - j*page_size) or 0; atomicMax into a
//                per-page count, so a page shared by several sequences keeps what the
//                longest of them uses (Prefix Sharing).
//   zero_kernel  one warp per entry: the first entry naming a page claims it (bit 31 of
//                its count) and zeroes the page's slots from that count to the end.
// Pages no slice names are never touched.
#include <cuda_runtime.h>

#include "hp_internal.cuh"

namespace hp {
namespace {

constexpr unsigned kClaimed = 0x80000000u;

template <typename IndexT>
__global__ void __launch_bounds__(256) live_kernel(const PlanArgs a, unsigned* live)
{
    pdl_wait();  // the plan and the table check before this launch are complete
    if (a.ws.hdr->verdict != kVerdictOk) return;
    const IndexT* sp = static_cast<const IndexT*>(a.seq_ptr);
    const IndexT* lens = static_cast<const IndexT*>(a.lens);
    const IndexT* table = static_cast<const IndexT*>(a.table);
    const uint64_t P = a.page_size;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t k = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; k < a.table_len;
         k += stride) {
        uint64_t lo = 0, hi = a.num_seqs;  // sp[lo] <= k < sp[hi] (validated invariants)
        while (hi - lo > 1) {
            const uint64_t mid = (lo + hi) >> 1;
            if ((uint64_t)sp[mid] <= k) lo = mid;
            else hi = mid;
        }
        const uint64_t j = k - (uint64_t)sp[lo];
        const uint64_t len = lens[lo];
        const uint64_t used = len > j * P ? (len - j * P < P ? len - j * P : P) : 0;
        atomicMax(live + (uint64_t)table[k], (unsigned)used);
    }
}

template <typename IndexT>
__global__ void __launch_bounds__(256) zero_kernel(const PlanArgs a, unsigned* live,
                                                   uint64_t row_bytes, char* pool)
{
    pdl_wait();  // every count is final
    if (a.ws.hdr->verdict != kVerdictOk) return;
    const IndexT* table = static_cast<const IndexT*>(a.table);
    const uint64_t P = a.page_size;
    const unsigned lane = threadIdx.x & 31;
    const uint64_t warps = (uint64_t)gridDim.x * (blockDim.x / 32);
    const bool wide = row_bytes % 16 == 0;
    for (uint64_t k = (uint64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
         k < a.table_len; k += warps) {
        const uint64_t page = table[k];
        unsigned old = 0;
        if (lane == 0) old = atomicOr(live + page, kClaimed);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old & kClaimed) continue;  // another entry of this page zeroes it
        const uint64_t from = (page * P + (old & ~kClaimed)) * row_bytes;
        const uint64_t to = (page + 1) * P * row_bytes;
        if (wide) {
            uint4* d = reinterpret_cast<uint4*>(pool + from);
            const uint64_t n = (to - from) / 16;
            for (uint64_t v = lane; v < n; v += 32) d[v] = make_uint4(0, 0, 0, 0);
        } else {
            for (uint64_t b = from + lane; b < to; b += 32) pool[b] = 0;
        }
    }
}

template <typename IndexT>
int launch_t(const PlanArgs& a, unsigned* live, uint64_t row_bytes, void* pool,
             cudaStream_t st)
{
    int dev = 0;
    const int sms = current_sms(&dev);
    if (sms == 0) return HP_ERR_CUDA;
    const uint64_t cap = (uint64_t)sms * 8;
    uint64_t g1 = (a.table_len + 255) / 256, g2 = (a.table_len + 7) / 8;
    g1 = g1 < cap ? g1 : cap;
    g2 = g2 < cap ? g2 : cap;
    if (launch_dependent(live_kernel<IndexT>, (unsigned)g1, 256, 0, st, a, live) != cudaSuccess)
        return HP_ERR_CUDA;
    if (launch_dependent(zero_kernel<IndexT>, (unsigned)g2, 256, 0, st, a, live, row_bytes,
                         static_cast<char*>(pool)) != cudaSuccess)
        return HP_ERR_CUDA;
    return HP_OK;
}

}  // namespace

int launch_zero_tails(int index_u64, const PlanArgs& a, unsigned* live, uint64_t row_bytes,
                      void* pool, void* stream)
{
    if (a.table_len == 0) return HP_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return index_u64 ? launch_t<unsigned long long>(a, live, row_bytes, pool, st)
                     : launch_t<unsigned int>(a, live, row_bytes, pool, st);
}

}  // namespace hp
