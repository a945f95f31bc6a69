// hp_plan.cu -- the plan step of the block-paged path: descriptor validation on the
// device and the ragged prefix sums that place each sequence's rows and copy units.
//
// "Block-Paged Layout -- Hurray Format Specification", sections Storage Invariants
// (invariants (1)-(3)), Logical Shape (total_tokens is the sum of the per-sequence
// token counts) and Partial trailing page (a reader stops at a sequence's count).
//
// Two kernels, launched in stream order:
//   plan_kernel   one CTA of 1024 threads walks seq_ptr / seq_lens (/ new_ptr) in
//                 chunks of 1024 sequences: saturating block scans of the token
//                 counts and of the per-sequence unit counts, the O(num_seqs) rules,
//                 and a plain store of the verdict key into the workspace header.
//   table_kernel  grid-stride pass over block_table for invariant (3); a CTA that
//                 finds a bad entry lowers the verdict with atomicMin.
// The smallest verdict key is the first failing rule (in the order of hp_status) at
// its first failing index, whichever thread found it.
#include <cuda_runtime.h>

#include "hp_internal.cuh"

namespace hp {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kWarps = kPlanThreads / 32;

__device__ __forceinline__ unsigned long long sat_add(unsigned long long a, unsigned long long b)
{
    unsigned long long c = a + b;
    return c < a ? ~0ull : c;
}

// Exclusive block scan of two counters at once with saturating addition (which is
// associative: it is min(a + b, 2^64 - 1) over the naturals).  Returns the
// exclusive prefixes; *tot receives the block totals.
__device__ __forceinline__ void block_scan2(unsigned long long v0, unsigned long long v1,
                                            unsigned long long& ex0, unsigned long long& ex1,
                                            unsigned long long& tot0, unsigned long long& tot1)
{
    __shared__ unsigned long long w0[kWarps], w1[kWarps];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    unsigned long long i0 = v0, i1 = v1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        unsigned long long n0 = __shfl_up_sync(0xffffffffu, i0, o);
        unsigned long long n1 = __shfl_up_sync(0xffffffffu, i1, o);
        if (lane >= o) {
            i0 = sat_add(n0, i0);
            i1 = sat_add(n1, i1);
        }
    }
    unsigned long long e0 = __shfl_up_sync(0xffffffffu, i0, 1);
    unsigned long long e1 = __shfl_up_sync(0xffffffffu, i1, 1);
    if (lane == 0) e0 = e1 = 0;
    if (lane == 31) {
        w0[wid] = i0;
        w1[wid] = i1;
    }
    __syncthreads();
    if (wid == 0) {
        unsigned long long a0 = w0[lane], a1 = w1[lane];  // kWarps == 32
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            unsigned long long n0 = __shfl_up_sync(0xffffffffu, a0, o);
            unsigned long long n1 = __shfl_up_sync(0xffffffffu, a1, o);
            if (lane >= o) {
                a0 = sat_add(n0, a0);
                a1 = sat_add(n1, a1);
            }
        }
        w0[lane] = a0;
        w1[lane] = a1;
    }
    __syncthreads();
    unsigned long long p0 = wid ? w0[wid - 1] : 0, p1 = wid ? w1[wid - 1] : 0;
    ex0 = sat_add(p0, e0);
    ex1 = sat_add(p1, e1);
    tot0 = w0[kWarps - 1];
    tot1 = w1[kWarps - 1];
    __syncthreads();  // w0/w1 are reused by the next call
}

// a*b > c with a 128-bit product and a 65-bit c = c_hi*2^64 + c_lo.
__device__ __forceinline__ bool gt_sum(unsigned long long c_lo, unsigned c_carry,
                                      unsigned long long a, unsigned long long b)
{
    // returns (c_carry:c_lo) > a*b
    unsigned long long lo = a * b, hi = __umul64hi(a, b);
    if (c_carry != hi) return c_carry > hi;
    return c_lo > lo;
}

template <typename IndexT, int MODE>
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a)
{
    const IndexT* sp = static_cast<const IndexT*>(a.seq_ptr);
    const IndexT* lens = static_cast<const IndexT*>(a.lens);
    const IndexT* np = static_cast<const IndexT*>(a.new_ptr);
    const uint64_t S = a.num_seqs, P = a.page_size;

    __shared__ unsigned long long s_key;
    __shared__ int s_fault;
    __shared__ unsigned long long s_carry_rows, s_carry_units;
    pdl_trigger();  // let the table check start scanning now
    if (threadIdx.x == 0) {
        s_key = kVerdictOk;
        s_fault = HP_OK;
        s_carry_rows = 0;
        s_carry_units = 0;
    }
    __syncthreads();

    for (uint64_t base = 0; base < S; base += kPlanThreads) {
        const uint64_t s = base + threadIdx.x;
        unsigned long long rows = 0, units = 0;
        if (s < S) {
            const unsigned long long lo = sp[s], hi = sp[s + 1], len = lens[s];
            if (MODE == kPlanGather || MODE == kPlanAttention) {
                rows = len;
                units = len / P + (len % P != 0);
                if (a.strict) {
                    if (lo > hi)
                        atomicMin(&s_key, verdict_key(kRankSeqPtrOrder, s));
                    else if (units > hi - lo)
                        atomicMin(&s_key, verdict_key(kRankLen, s));
                }
                if (MODE == kPlanAttention)  // tokens -> steps of step_tokens tokens
                    units = len / a.step_tokens + (len % a.step_tokens != 0);
            } else {
                const unsigned long long n0 = np[s], n1 = np[s + 1];
                const bool ok_new = n0 <= n1 && n1 <= a.total_new;
                const unsigned long long n_new = ok_new ? n1 - n0 : 0;
                const unsigned long long end = len + n_new;
                const unsigned carry = end < len;
                rows = n_new;
                if (n_new > 0 && !carry)
                    units = (end - 1) / P - len / P + 1;
                if (a.strict) {
                    if (lo > hi) atomicMin(&s_key, verdict_key(kRankSeqPtrOrder, s));
                    if (n0 > n1) atomicMin(&s_key, verdict_key(kRankNewPtrOrder, s));
                    if (lo <= hi && gt_sum(end, carry, hi - lo, P))
                        atomicMin(&s_key, verdict_key(kRankCapacity, s));
                } else if (!ok_new) {
                    atomicCAS(&s_fault, HP_OK, n0 > n1 ? HP_ERR_NEW_PTR_ORDER : HP_ERR_NEW_PTR_END);
                } else if (carry) {
                    atomicCAS(&s_fault, HP_OK, HP_ERR_CAPACITY);
                }
            }
        }
        unsigned long long ex_rows, ex_units, tot_rows, tot_units;
        block_scan2(rows, units, ex_rows, ex_units, tot_rows, tot_units);
        const unsigned long long cr = s_carry_rows, cu = s_carry_units;
        if (s < S) {
            a.ws.rows_off[s] = sat_add(cr, ex_rows);
            a.ws.units_off[s] = sat_add(cu, ex_units);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            s_carry_rows = sat_add(cr, tot_rows);
            s_carry_units = sat_add(cu, tot_units);
        }
        __syncthreads();
    }

    if (threadIdx.x == 0) {
        unsigned long long key = s_key;
        const unsigned long long total_rows = s_carry_rows, total_units = s_carry_units;
        if (a.strict) {
            if (sp[0] != 0) key = min(key, verdict_key(kRankSeqPtrStart, 0));
            if ((unsigned long long)sp[S] != a.table_len)
                key = min(key, verdict_key(kRankSeqPtrEnd, S));
            if (MODE == kPlanAppend) {
                if (np[0] != 0) key = min(key, verdict_key(kRankNewPtrStart, 0));
                if ((unsigned long long)np[S] != a.total_new)
                    key = min(key, verdict_key(kRankNewPtrEnd, S));
            }
        }
        if (MODE == kPlanGather && a.check_out &&
            (total_rows == ~0ull || total_rows != a.out_tokens))
            key = min(key, verdict_key(kRankOutSize, 0));
        a.ws.rows_off[S] = total_rows;
        a.ws.units_off[S] = total_units;
        a.ws.hdr->total_rows = total_rows;
        a.ws.hdr->total_units = total_units;
        a.ws.hdr->verdict = key;
        if (a.d_status) *a.d_status = key != kVerdictOk ? key_status(key) : s_fault;
    }
}

// Invariant (3): every block-table entry names a page of the pool.
template <typename IndexT>
__global__ void __launch_bounds__(256) table_kernel(const IndexT* __restrict__ table,
                                                    uint64_t n, uint64_t num_pages,
                                                    WsHeader* hdr, int* d_status)
{
    unsigned long long first = ~0ull;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t k = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += stride) {
        if ((unsigned long long)__ldg(table + k) >= num_pages) {
            first = k;  // k only grows: this thread's first bad entry
            break;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
    __shared__ unsigned long long s_first;
    if (threadIdx.x == 0) s_first = ~0ull;
    __syncthreads();
    if ((threadIdx.x & 31) == 0 && first != ~0ull) atomicMin(&s_first, first);
    __syncthreads();
    pdl_trigger();  // the copy may be scheduled; it waits for this grid to finish
    pdl_wait();     // the plan's verdict store must land before it is lowered
    if (threadIdx.x == 0 && s_first != ~0ull) {
        const unsigned long long key = verdict_key(kRankPageId, s_first);
        const unsigned long long old = atomicMin(&hdr->verdict, key);
        // every key of this rule maps to the same status code, so concurrent
        // stores from several CTAs agree
        if (key < old && d_status) *d_status = HP_ERR_PAGE_ID;
    }
}

// ---------------------------------------------------------- block-table forms
// A padded table [batch, max_blocks] with token counts (the form an attention kernel
// takes, "Visualize PagedAttention block layout", How the attention kernel uses the block
// table) versus the CSR slices of the block-paged descriptor.  Sequence s uses the first
// ceil(len_s / page_size) entries of its row.

template <typename IndexT>
__global__ void __launch_bounds__(kPlanThreads) padded_scan_kernel(
    const IndexT* lens, uint64_t batch, uint64_t max_blocks, uint64_t P, uint64_t cap,
    WsHeader* hdr, unsigned long long* prefix, int* d_status)
{
    pdl_trigger();
    __shared__ unsigned long long s_key, s_carry;
    if (threadIdx.x == 0) {
        s_key = kVerdictOk;
        s_carry = 0;
    }
    __syncthreads();
    for (uint64_t base = 0; base < batch; base += kPlanThreads) {
        const uint64_t s = base + threadIdx.x;
        unsigned long long need = 0;
        if (s < batch) {
            const unsigned long long len = lens[s];
            need = len / P + (len % P != 0);
            if (need > max_blocks) atomicMin(&s_key, verdict_key(kRankLen, s));
        }
        unsigned long long ex, ex2, tot, tot2;
        block_scan2(need, 0, ex, ex2, tot, tot2);
        const unsigned long long c = s_carry;
        if (s < batch) prefix[s] = sat_add(c, ex);
        __syncthreads();
        if (threadIdx.x == 0) s_carry = sat_add(c, tot);
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        unsigned long long key = s_key;
        const unsigned long long total = s_carry;
        if (total > cap) key = min(key, verdict_key(kRankOutSize, 0));
        prefix[batch] = total;
        hdr->total_units = total;
        hdr->verdict = key;
        if (d_status) *d_status = key_status(key);
    }
}

template <typename IndexT>
__global__ void __launch_bounds__(256) padded_fill_kernel(
    const IndexT* padded, uint64_t batch, uint64_t max_blocks, const WsHeader* hdr,
    const unsigned long long* prefix, IndexT* table_out, IndexT* seq_ptr_out)
{
    pdl_wait();
    if (hdr->verdict != kVerdictOk) return;
    if (blockIdx.x == 0 && threadIdx.x == 0) seq_ptr_out[batch] = (IndexT)prefix[batch];
    const unsigned lane = threadIdx.x & 31;
    const uint64_t warps = (uint64_t)gridDim.x * (blockDim.x / 32);
    for (uint64_t s = (uint64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); s < batch;
         s += warps) {
        const unsigned long long at = prefix[s], need = prefix[s + 1] - at;
        if (lane == 0) seq_ptr_out[s] = (IndexT)at;
        for (uint64_t j = lane; j < need; j += 32) table_out[at + j] = padded[s * max_blocks + j];
    }
}

template <typename IndexT>
__global__ void __launch_bounds__(kPlanThreads) csr_check_kernel(
    const IndexT* seq_ptr, uint64_t batch, uint64_t max_blocks, uint64_t table_len,
    WsHeader* hdr, int* d_status)
{
    pdl_trigger();
    __shared__ unsigned long long s_key;
    if (threadIdx.x == 0) s_key = kVerdictOk;
    __syncthreads();
    for (uint64_t s = threadIdx.x; s < batch; s += kPlanThreads) {
        const unsigned long long lo = seq_ptr[s], hi = seq_ptr[s + 1];
        if (hi < lo || hi > table_len || hi - lo > max_blocks)
            atomicMin(&s_key, verdict_key(kRankLen, s));
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        hdr->verdict = s_key;
        if (d_status) *d_status = key_status(s_key);
    }
}

template <typename IndexT>
__global__ void __launch_bounds__(256) csr_fill_kernel(
    const IndexT* table, const IndexT* seq_ptr, uint64_t batch, uint64_t max_blocks,
    unsigned long long pad, const WsHeader* hdr, IndexT* padded_out)
{
    pdl_wait();
    if (hdr->verdict != kVerdictOk) return;
    const uint64_t n = batch * max_blocks, stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint64_t s = i / max_blocks, j = i - s * max_blocks;
        const unsigned long long lo = seq_ptr[s], cnt = seq_ptr[s + 1] - lo;
        padded_out[i] = j < cnt ? table[lo + j] : (IndexT)pad;
    }
}

template <typename IndexT>
int launch_tables_t(const TableArgs& t, cudaStream_t st)
{
    int dev = 0;
    const int sms = current_sms(&dev);
    if (sms == 0) return HP_ERR_CUDA;
    const uint64_t cap = (uint64_t)sms * 8;
    WsHeader* hdr = static_cast<WsHeader*>(t.workspace);
    unsigned long long* prefix =
        reinterpret_cast<unsigned long long*>(static_cast<char*>(t.workspace) + kWsHeaderBytes);
    if (t.to_csr) {
        padded_scan_kernel<IndexT><<<1, kPlanThreads, 0, st>>>(
            static_cast<const IndexT*>(t.lens), t.batch, t.max_blocks, t.page_size, t.cap, hdr,
            prefix, t.d_status);
        if (cudaGetLastError() != cudaSuccess) return HP_ERR_CUDA;
        uint64_t g = (t.batch + 7) / 8;
        g = g == 0 ? 1 : (g < cap ? g : cap);
        return launch_dependent(padded_fill_kernel<IndexT>, (unsigned)g, 256, 0, st,
                                static_cast<const IndexT*>(t.in), t.batch, t.max_blocks,
                                (const WsHeader*)hdr, (const unsigned long long*)prefix,
                                static_cast<IndexT*>(t.out), static_cast<IndexT*>(t.out2)) ==
                       cudaSuccess
                   ? HP_OK
                   : HP_ERR_CUDA;
    }
    csr_check_kernel<IndexT><<<1, kPlanThreads, 0, st>>>(
        static_cast<const IndexT*>(t.seq_ptr), t.batch, t.max_blocks, t.table_len, hdr,
        t.d_status);
    if (cudaGetLastError() != cudaSuccess) return HP_ERR_CUDA;
    const uint64_t n = t.batch * t.max_blocks;
    if (n == 0) return HP_OK;
    uint64_t g = (n + 255) / 256;
    g = g < cap ? g : cap;
    return launch_dependent(csr_fill_kernel<IndexT>, (unsigned)g, 256, 0, st,
                            static_cast<const IndexT*>(t.in), static_cast<const IndexT*>(t.seq_ptr),
                            t.batch, t.max_blocks, (unsigned long long)t.pad, (const WsHeader*)hdr,
                            static_cast<IndexT*>(t.out)) == cudaSuccess
               ? HP_OK
               : HP_ERR_CUDA;
}

template <typename IndexT>
int launch_plan_t(PlanMode mode, const PlanArgs& a, cudaStream_t st)
{
    if (mode == kPlanGather)
        plan_kernel<IndexT, kPlanGather><<<1, kPlanThreads, 0, st>>>(a);
    else if (mode == kPlanAppend)
        plan_kernel<IndexT, kPlanAppend><<<1, kPlanThreads, 0, st>>>(a);
    else
        plan_kernel<IndexT, kPlanAttention><<<1, kPlanThreads, 0, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return HP_ERR_CUDA;
    if (a.strict && a.table_len > 0) {
        int dev = 0;
        const int sms = current_sms(&dev);
        if (sms == 0) return HP_ERR_CUDA;
        uint64_t blocks = (a.table_len + 255) / 256;
        const uint64_t cap = (uint64_t)sms * 8;
        if (blocks > cap) blocks = cap;
        if (launch_dependent(table_kernel<IndexT>, (unsigned)blocks, 256, 0, st,
                             static_cast<const IndexT*>(a.table), a.table_len, a.num_pages,
                             a.ws.hdr, a.d_status) != cudaSuccess)
            return HP_ERR_CUDA;
    }
    return HP_OK;
}

}  // namespace

int launch_tables(int index_u64, const TableArgs& t, void* stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return index_u64 ? launch_tables_t<unsigned long long>(t, st)
                     : launch_tables_t<unsigned int>(t, st);
}

int launch_plan(PlanMode mode, int index_u64, const PlanArgs& a, void* stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return index_u64 ? launch_plan_t<unsigned long long>(mode, a, st)
                     : launch_plan_t<unsigned int>(mode, a, st);
}

}  // namespace hp
