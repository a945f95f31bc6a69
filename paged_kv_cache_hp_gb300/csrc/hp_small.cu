// hp_small.cu -- the validated gather of a small batch in one launch.
//
// "Block-Paged Layout -- Hurray Format Specification": Storage Invariants (1)-(3), the
// token-count rule and Logical Shape decide the verdict; the Element Lookup moves the
// rows.  For a batch of at most kMaxSeqs sequences and kMaxTable block-table entries the
// plan, the table check and the copy of the regular path (three chained kernels) fold
// into one: every CTA repeats the plan's scans and rules and the table check on its own
// (a few thousand index entries from L2), so every CTA reaches the same verdict without a
// barrier across the grid; CTA 0 publishes it (status word and workspace, as the plan
// would), and all CTAs copy only when it is OK, one copy unit (a sequence's rows in one
// page) per warp.  Verdicts follow the regular path's rule order exactly: the smallest
// (rule rank, index) key over the O(num_seqs) rules, invariant (3) and the output size.
#include <cuda_runtime.h>

#include <algorithm>

#include "hp_internal.cuh"
#include "hp_small.cuh"

namespace hp {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
static_assert(kMaxSeqs <= kThreads, "one thread per sequence");

__device__ __forceinline__ unsigned long long sat_add(unsigned long long a, unsigned long long b)
{
    const unsigned long long c = a + b;
    return c < a ? ~0ull : c;
}

template <int VEC> struct VecOf;
template <> struct VecOf<16> { using T = uint4; };
template <> struct VecOf<8> { using T = uint2; };
template <> struct VecOf<4> { using T = unsigned int; };
template <> struct VecOf<2> { using T = unsigned short; };
template <> struct VecOf<1> { using T = unsigned char; };

template <typename IndexT, int VEC>
__global__ void __launch_bounds__(kThreads) small_gather_kernel(const SmallGatherArgs a)
{
    using T = typename VecOf<VEC>::T;
    __shared__ unsigned long long s_rows[kMaxSeqs + 1], s_units[kMaxSeqs + 1];
    __shared__ unsigned long long s_w0[kWarps], s_w1[kWarps];
    __shared__ unsigned long long s_key;
    const IndexT* sp = static_cast<const IndexT*>(a.seq_ptr);
    const IndexT* lens = static_cast<const IndexT*>(a.lens);
    const IndexT* table = static_cast<const IndexT*>(a.table);
    const unsigned tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const uint64_t S = a.num_seqs, P = a.page_size;
    if (tid == 0) s_key = kVerdictOk;
    __syncthreads();

    // the plan's per-sequence counts and rules (thread s takes sequence s)
    unsigned long long rows = 0, units = 0;
    if (tid < S) {
        const unsigned long long lo = sp[tid], hi = sp[tid + 1], len = lens[tid];
        rows = len;
        units = len / P + (len % P != 0);
        if (lo > hi)
            atomicMin(&s_key, verdict_key(kRankSeqPtrOrder, tid));
        else if (units > hi - lo)
            atomicMin(&s_key, verdict_key(kRankLen, tid));
    }
    // saturating exclusive scans of rows and units (warp shuffles, then across warps)
    unsigned long long r = rows, q = units;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long nr = __shfl_up_sync(0xffffffffu, r, o);
        const unsigned long long nq = __shfl_up_sync(0xffffffffu, q, o);
        if ((int)lane >= o) {
            r = sat_add(nr, r);
            q = sat_add(nq, q);
        }
    }
    if (lane == 31) {
        s_w0[wid] = r;
        s_w1[wid] = q;
    }
    __syncthreads();
    if (wid == 0) {
        unsigned long long x = s_w0[lane], y = s_w1[lane];  // kWarps == 32
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long nx = __shfl_up_sync(0xffffffffu, x, o);
            const unsigned long long ny = __shfl_up_sync(0xffffffffu, y, o);
            if ((int)lane >= o) {
                x = sat_add(nx, x);
                y = sat_add(ny, y);
            }
        }
        s_w0[lane] = x;
        s_w1[lane] = y;
    }
    __syncthreads();
    const unsigned long long pr = wid ? s_w0[wid - 1] : 0, pq = wid ? s_w1[wid - 1] : 0;
    // exclusive prefix: the warps before, plus the previous lane's inclusive value
    unsigned long long er = __shfl_up_sync(0xffffffffu, r, 1);
    unsigned long long eq = __shfl_up_sync(0xffffffffu, q, 1);
    if (lane == 0) er = eq = 0;
    if (tid < S) {
        s_rows[tid] = sat_add(pr, er);
        s_units[tid] = sat_add(pq, eq);
    }
    if (tid == 0) {
        s_rows[S] = s_w0[kWarps - 1];
        s_units[S] = s_w1[kWarps - 1];
    }
    // invariant (3): this thread's first bad block-table entry
    unsigned long long bad = ~0ull;
    for (uint64_t k = tid; k < a.table_len; k += kThreads)
        if ((unsigned long long)table[k] >= a.num_pages) {
            bad = k;
            break;
        }
    if (bad != ~0ull) atomicMin(&s_key, verdict_key(kRankPageId, bad));
    __syncthreads();
    if (tid == 0) {
        unsigned long long key = s_key;
        if (sp[0] != 0) key = min(key, verdict_key(kRankSeqPtrStart, 0));
        if ((unsigned long long)sp[S] != a.table_len) key = min(key, verdict_key(kRankSeqPtrEnd, S));
        const unsigned long long total_rows = s_rows[S];
        if (total_rows == ~0ull || total_rows != a.out_tokens)
            key = min(key, verdict_key(kRankOutSize, 0));
        s_key = key;
    }
    __syncthreads();
    const unsigned long long key = s_key;
    if (blockIdx.x == 0) {  // publish as the plan and the table check would
        for (uint64_t s = tid; s <= S; s += kThreads) {
            a.ws.rows_off[s] = s_rows[s];
            a.ws.units_off[s] = s_units[s];
        }
        if (tid == 0) {
            a.ws.hdr->verdict = key;
            a.ws.hdr->total_rows = s_rows[S];
            a.ws.hdr->total_units = s_units[S];
            if (a.d_status) *a.d_status = key_status(key);
        }
    }
    if (key != kVerdictOk) return;

    // the copy: unit u (sequence s, its j-th page) per warp
    const uint64_t total = s_units[S];
    const uint64_t nw = (uint64_t)gridDim.x * kWarps;
    for (uint64_t u = (uint64_t)blockIdx.x * kWarps + wid; u < total; u += nw) {
        uint64_t lo = 0, hi = S;  // s_units[lo] <= u < s_units[hi]
        while (hi - lo > 1) {
            const uint64_t mid = (lo + hi) >> 1;
            if (s_units[mid] <= u) lo = mid;
            else hi = mid;
        }
        const uint64_t s = lo, j = u - s_units[s], t0 = j * P;
        const uint64_t len = lens[s], n = (len - t0 < P ? len - t0 : P) * a.row_bytes / VEC;
        const uint64_t phys = table[(uint64_t)sp[s] + j];
        const T* src = reinterpret_cast<const T*>(a.pool + phys * P * a.row_bytes);
        T* dst = reinterpret_cast<T*>(a.out + (s_rows[s] + t0) * a.row_bytes);
        for (uint64_t v = lane; v < n; v += 32 * 4) {
            T x[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (v + 32 * k < n) x[k] = __ldg(src + v + 32 * k);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (v + 32 * k < n) dst[v + 32 * k] = x[k];
        }
    }
}

template <typename IndexT, int VEC>
int launch_v(const SmallGatherArgs& a, cudaStream_t st)
{
    int dev = 0;
    const int sms = current_sms(&dev);
    if (sms == 0) return HP_ERR_CUDA;
    // about four units per warp, at most two CTAs per SM
    const uint64_t want = (a.table_len + 4 * kWarps - 1) / (4 * kWarps);
    const uint64_t grid = std::max<uint64_t>(1, std::min<uint64_t>(want, 2ull * sms));
    small_gather_kernel<IndexT, VEC><<<(unsigned)grid, kThreads, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? HP_OK : HP_ERR_CUDA;
}

template <typename IndexT>
int launch_i(const SmallGatherArgs& a, int vec, cudaStream_t st)
{
    switch (vec) {
    case 16: return launch_v<IndexT, 16>(a, st);
    case 8: return launch_v<IndexT, 8>(a, st);
    case 4: return launch_v<IndexT, 4>(a, st);
    case 2: return launch_v<IndexT, 2>(a, st);
    default: return launch_v<IndexT, 1>(a, st);
    }
}

}  // namespace

int launch_small_gather(int index_u64, const SmallGatherArgs& a, int vec, void* stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return index_u64 ? launch_i<unsigned long long>(a, vec, st)
                     : launch_i<unsigned int>(a, vec, st);
}

}  // namespace hp
