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
//   zero_kernel  one thread per entry: the first entry naming a page claims it (bit 31
//                of its count); the warp then zeroes, page by page, the slots from the
//                count to the end of each page its lanes claimed that has any.
// Pages no slice names are never touched.
//
// The decode-step append ("Block-Paged Layout -- Hurray Format Specification", Element
// Lookup used as a store: row i of sequence s goes to token len_s + i), for appends of
// less than a page per sequence on average:
//   append_rows_kernel  one warp per sequence, no unit search (after the plan's verdict
//                when the descriptor is validated, with no plan at all when it is
//                permissive): its new rows are
//                rows new_ptr[s] .. new_ptr[s+1] of the input and token len_s + i lives in
//                slot (len_s + i) mod P of page block_table[seq_ptr[s] + (len_s + i) / P].
//                The row loads go out together with the block-table lookup.  A row whose
//                logical page lies outside the slice or the table is skipped with
//                HP_ERR_LEN, one naming a page outside the pool with HP_ERR_PAGE_ID; a
//                sequence whose new_ptr pair runs backwards or past total_new (possible
//                only without a plan) is skipped whole with HP_ERR_NEW_PTR_ORDER or
//                HP_ERR_NEW_PTR_END, so no input row past total_new is read.
#include <cuda_runtime.h>

#include "hp_internal.cuh"
#include "hp_resolve.cuh"

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
    // one entry per lane: the first entry naming a page claims it; the warp then zeroes
    // the tails of the pages its lanes claimed that have unused slots, one page at a time
    for (uint64_t base = ((uint64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5)) * 32;
         base < a.table_len; base += warps * 32) {
        const uint64_t k = base + lane;
        uint64_t page = 0;
        unsigned old = kClaimed;
        if (k < a.table_len) {
            page = table[k];
            old = atomicOr(live + page, kClaimed);
        }
        unsigned todo = __ballot_sync(0xffffffffu, !(old & kClaimed) && old < P);
        while (todo) {
            const int src = __ffs(todo) - 1;
            todo &= todo - 1;
            const uint64_t pg = __shfl_sync(0xffffffffu, page, src);
            const unsigned used = __shfl_sync(0xffffffffu, old, src);
            const uint64_t from = (pg * P + used) * row_bytes;
            const uint64_t to = (pg + 1) * P * row_bytes;
            if (wide) {
                uint4* d = reinterpret_cast<uint4*>(pool + from);
                const uint64_t n = (to - from) / 16;
                for (uint64_t v = lane; v < n; v += 32) d[v] = make_uint4(0, 0, 0, 0);
            } else {
                for (uint64_t x = from + lane; x < to; x += 32) pool[x] = 0;
            }
        }
    }
}

template <int VEC> struct VecOf;
template <> struct VecOf<16> { using T = uint4; };
template <> struct VecOf<8> { using T = uint2; };
template <> struct VecOf<4> { using T = unsigned int; };
template <> struct VecOf<2> { using T = unsigned short; };
template <> struct VecOf<1> { using T = unsigned char; };

template <typename IndexT, int VEC>
__global__ void __launch_bounds__(256) append_rows_kernel(const CopyArgs a)
{
    using T = typename VecOf<VEC>::T;
    constexpr int kHeld = 4;  // vectors per lane held for one row (rows up to 2 KiB at VEC 16)
    const IndexT* np = static_cast<const IndexT*>(a.new_ptr);
    const IndexT* lens = static_cast<const IndexT*>(a.lens);
    const IndexT* sp = static_cast<const IndexT*>(a.seq_ptr);
    const IndexT* table = static_cast<const IndexT*>(a.table);
    const unsigned lane = threadIdx.x & 31;
    if (a.hdr) {  // after a plan: wait for its verdict, write nothing unless it is OK
        pdl_wait();
        if (a.hdr->verdict != kVerdictOk) return;
    }
    const uint64_t P = a.page_size, nv = a.row_bytes / VEC;
    const uint64_t warps = (uint64_t)gridDim.x * (blockDim.x / 32);
    for (uint64_t s = (uint64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
         s < a.num_seqs; s += warps) {
        const uint64_t r0 = np[s], r1 = np[s + 1], len = lens[s];
        const uint64_t lo = sp[s], hi = sp[s + 1];
        if (r1 < r0 || r1 > a.total_new) {  // permissive only: a plan's verdict rules it out
            report(a.d_status, r1 < r0 ? HP_ERR_NEW_PTR_ORDER : HP_ERR_NEW_PTR_END);
            continue;  // no row of the input outside [0, total_new) is read
        }
        for (uint64_t i = 0; i < r1 - r0; ++i) {
            const T* src = reinterpret_cast<const T*>(a.src + (r0 + i) * a.row_bytes);
            T held[kHeld];  // the row's first vectors, loaded before the table lookup lands
#pragma unroll
            for (int k = 0; k < kHeld; ++k) {
                const uint64_t v = lane + 32 * k;
                if (v < nv) held[k] = __ldg(src + v);
            }
            const uint64_t t = len + i, j = t / P;
            if (lo > hi || j >= hi - lo || lo + j >= a.table_len) {
                report(a.d_status, HP_ERR_LEN);
                continue;
            }
            const uint64_t phys = table[lo + j];
            if (phys >= a.num_pages) {
                report(a.d_status, HP_ERR_PAGE_ID);
                continue;
            }
            T* dst = reinterpret_cast<T*>(a.dst + (phys * P + (t - j * P)) * a.row_bytes);
#pragma unroll
            for (int k = 0; k < kHeld; ++k) {
                const uint64_t v = lane + 32 * k;
                if (v < nv) dst[v] = held[k];
            }
            for (uint64_t v = lane + 32 * kHeld; v < nv; v += 32) dst[v] = __ldg(src + v);
        }
    }
}

template <typename IndexT, int VEC>
int launch_rows(const CopyArgs& a, cudaStream_t st)
{
    int dev = 0;
    const int sms = current_sms(&dev);
    if (sms == 0) return HP_ERR_CUDA;
    uint64_t grid = (a.num_seqs + 7) / 8;
    const uint64_t cap = (uint64_t)sms * 8;
    grid = grid < cap ? grid : cap;
    if (a.hdr)  // a dependent of the plan and the table check
        return launch_dependent(append_rows_kernel<IndexT, VEC>, (unsigned)grid, 256, 0, st, a) ==
                       cudaSuccess
                   ? HP_OK
                   : HP_ERR_CUDA;
    append_rows_kernel<IndexT, VEC><<<(unsigned)grid, 256, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? HP_OK : HP_ERR_CUDA;
}

template <typename IndexT>
int launch_rows_v(const CopyArgs& a, int vec, cudaStream_t st)
{
    switch (vec) {
    case 16: return launch_rows<IndexT, 16>(a, st);
    case 8: return launch_rows<IndexT, 8>(a, st);
    case 4: return launch_rows<IndexT, 4>(a, st);
    case 2: return launch_rows<IndexT, 2>(a, st);
    default: return launch_rows<IndexT, 1>(a, st);
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
    uint64_t g1 = (a.table_len + 255) / 256, g2 = (a.table_len + 255) / 256;
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

int launch_append_rows(int index_u64, const CopyArgs& a, int vec, void* stream)
{
    if (a.num_seqs == 0) return HP_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return index_u64 ? launch_rows_v<unsigned long long>(a, vec, st)
                     : launch_rows_v<unsigned int>(a, vec, st);
}

int launch_zero_tails(int index_u64, const PlanArgs& a, unsigned* live, uint64_t row_bytes,
                      void* pool, void* stream)
{
    if (a.table_len == 0) return HP_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return index_u64 ? launch_t<unsigned long long>(a, live, row_bytes, pool, st)
                     : launch_t<unsigned int>(a, live, row_bytes, pool, st);
}

}  // namespace hp
