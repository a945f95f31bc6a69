// hp_resolve.cuh -- device-side mapping of a copy unit to its source, destination and
// row count, shared by the two copy engines (hp_copy.cu, hp_bulk.cu).
//
// "Block-Paged Layout -- Hurray Format Specification", Element Lookup: token t of
// sequence s lives in slot t mod page_size of page block_table[seq_ptr[s] + t/page_size];
// a unit is the run of a sequence's rows inside one page.  "Keep token order across cache
// pages", row_start: row p of lane l sits at ((T[p/P]*lanes + l)*P + p%P)*width.
#pragma once

#include <cstdint>

#include "hp_internal.cuh"

namespace hp {

__device__ __forceinline__ uint64_t umin(uint64_t a, uint64_t b) { return a < b ? a : b; }
__device__ __forceinline__ uint64_t umax(uint64_t a, uint64_t b) { return a > b ? a : b; }

__device__ __forceinline__ void report(int* d_status, int code)
{
    if (d_status) atomicCAS(d_status, HP_OK, code);
}

// Largest s in [0, S) with units_off[s] <= u, given units_off[0] <= u < units_off[S].
__device__ __forceinline__ uint64_t find_seq(const unsigned long long* units_off, uint64_t S,
                                             uint64_t u)
{
    uint64_t lo = 0, hi = S;
    while (hi - lo > 1) {
        const uint64_t mid = (lo + hi) >> 1;
        if (units_off[mid] <= u) lo = mid;
        else hi = mid;
    }
    return lo;
}

struct Unit {
    unsigned long long src, dst, scale;  // byte offsets into src/dst; first scale index
    unsigned rows;                       // 0 = nothing to copy
};

// The slice checks a permissive reader still needs before reading block_table:
// the logical page must lie in the sequence's slice and in the table, and the page
// it names in the pool.  Returns the physical page, or ~0 after reporting.
template <typename IndexT>
__device__ __forceinline__ unsigned long long slice_page(const CopyArgs& a, uint64_t s,
                                                         uint64_t j)
{
    const IndexT* sp = static_cast<const IndexT*>(a.seq_ptr);
    const unsigned long long lo = sp[s], hi = sp[s + 1];
    if (lo > hi || j >= hi - lo || lo + j >= a.table_len) {
        report(a.d_status, HP_ERR_LEN);
        return ~0ull;
    }
    const unsigned long long phys = static_cast<const IndexT*>(a.table)[lo + j];
    if (phys >= a.num_pages) {
        report(a.d_status, HP_ERR_PAGE_ID);
        return ~0ull;
    }
    return phys;
}

template <int MODE, typename IndexT>
__device__ __forceinline__ Unit resolve(const CopyArgs& a, uint64_t u)
{
    Unit r{0, 0, 0, 0};
    const uint64_t P = a.page_size;
    if (MODE == kGather || MODE == kDequant) {
        const uint64_t s = find_seq(a.units_off, a.num_seqs, u);
        const uint64_t j = u - a.units_off[s];
        const uint64_t len = static_cast<const IndexT*>(a.lens)[s];
        const uint64_t t0 = j * P;
        const unsigned long long phys = slice_page<IndexT>(a, s, j);
        if (phys == ~0ull) return r;
        r.rows = (unsigned)umin(P, len - t0);
        r.src = phys * P * a.row_bytes;
        const uint64_t out_row = MODE == kDequant ? a.row_elems * 2 : a.row_bytes;
        r.dst = (a.rows_off[s] + t0) * out_row;
        r.scale = phys * P;
    } else if (MODE == kAppend) {
        const uint64_t s = find_seq(a.units_off, a.num_seqs, u);
        const uint64_t k = u - a.units_off[s];
        const uint64_t start = static_cast<const IndexT*>(a.lens)[s];
        const uint64_t n0 = static_cast<const IndexT*>(a.new_ptr)[s];
        const uint64_t n1 = static_cast<const IndexT*>(a.new_ptr)[s + 1];
        const uint64_t end = start + (n1 - n0);
        const uint64_t j = start / P + k;
        const uint64_t t0 = umax(start, j * P);
        const uint64_t t1 = umin(end, (j + 1) * P);
        const unsigned long long phys = slice_page<IndexT>(a, s, j);
        if (phys == ~0ull) return r;
        r.rows = (unsigned)(t1 - t0);
        r.src = (n0 + (t0 - start)) * a.row_bytes;
        r.dst = (phys * P + t0 % P) * a.row_bytes;
    } else if (MODE == kCopyPages) {
        const unsigned long long from = static_cast<const IndexT*>(a.src_pages)[u];
        const unsigned long long to = static_cast<const IndexT*>(a.dst_pages)[u];
        if (from >= a.num_pages || to >= a.num_pages) {
            report(a.d_status, HP_ERR_PAGE_ID);
            return r;
        }
        r.rows = 1;  // one "row" of page_bytes
        r.src = from * a.row_bytes;
        r.dst = to * a.row_bytes;
    } else {
        const uint64_t A = a.lane_pages;
        const uint64_t lane = u / A, q = a.lane_first_page + u % A;
        const unsigned long long phys = static_cast<const unsigned long long*>(a.table)[q];
        if (phys >= a.num_pages) {
            report(a.d_status, HP_ERR_PHYSICAL_PAGE);
            return r;
        }
        const uint64_t n = a.lane_n;
        if (MODE == kLaneGather) {
            const uint64_t t0 = q * P;
            r.rows = (unsigned)umin(P, n - t0);
            r.src = (phys * a.lanes + lane) * P * a.row_bytes;
            r.dst = (lane * n + t0) * a.row_bytes;
        } else {
            const uint64_t m = a.lane_m;
            const uint64_t t0 = umax(n, q * P);
            const uint64_t t1 = umin(n + m, (q + 1) * P);
            r.rows = (unsigned)(t1 - t0);
            r.src = (lane * m + (t0 - n)) * a.row_bytes;
            r.dst = ((phys * a.lanes + lane) * P + t0 % P) * a.row_bytes;
        }
    }
    return r;
}

}  // namespace hp
