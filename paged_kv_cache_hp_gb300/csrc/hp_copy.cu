// hp_copy.cu -- the copy step: one persistent engine for every data-movement mode.
//
// The pool is [num_pages, page_size, H, D] ("Block-Paged Layout -- Hurray Format
// Specification", Element Lookup; the vLLM [num_blocks, block_size, num_kv_heads,
// head_dim] mapping of its Framework Compliance section), so the valid rows of one
// page of one sequence are a single contiguous run of rows*H*D elements, and so are
// that sequence's rows of the logical [total_tokens, H, D] output.  A gather is
// therefore a batch of independent contiguous copies of at most page_size rows: the
// "units" of this engine.
//
//   gather / dequant   unit = (sequence s, logical page j): rows [jP, min(len,(j+1)P))
//   append             unit = (sequence s, page the new rows touch)
//   lane gather/append unit = (lane, logical page) of the [N, B, H_kv, P, d] layout of
//                      "Keep token order across cache pages" (row_start)
//
// Grid: one wave of CTAs (SM count x resident CTAs per SM), each owning a contiguous
// range of units, so work is balanced to within one unit per CTA.  A CTA resolves up
// to 256 units at a time -- thread k maps unit u0+k to its sequence by binary search
// over the unit prefix, reads the block-table entry and stages (source offset,
// destination offset, rows) in shared memory -- then all 256 threads copy the staged
// units one after another with 16-byte vector loads and stores, eight in flight per
// thread.  Only a sequence's valid rows are read; the undefined tail of a partial
// last page is never touched.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "hp_internal.cuh"
#include "hp_resolve.cuh"

namespace hp {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;

template <int VEC> struct Vec;
template <> struct Vec<16> { using T = uint4; };
template <> struct Vec<8> { using T = uint2; };
template <> struct Vec<4> { using T = unsigned int; };
template <> struct Vec<2> { using T = unsigned short; };
template <> struct Vec<1> { using T = unsigned char; };

// Streaming loads (read-only path, no L1 allocation) and evict-first stores: every
// byte is touched once.
template <typename T>
__device__ __forceinline__ T ld_stream(const T* p) { return __ldg(p); }
template <>
__device__ __forceinline__ uint4 ld_stream<uint4>(const uint4* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
template <typename T>
__device__ __forceinline__ void st_stream(T* p, T v) { *p = v; }
template <>
__device__ __forceinline__ void st_stream<uint4>(uint4* p, uint4 v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// All threads of the CTA copy `n` vectors.
template <int VEC>
__device__ __forceinline__ void copy_run(const char* __restrict__ src, char* __restrict__ dst,
                                         uint64_t n)
{
    using T = typename Vec<VEC>::T;
    const T* s = reinterpret_cast<const T*>(src);
    T* d = reinterpret_cast<T*>(dst);
    for (uint64_t v0 = threadIdx.x; v0 < n; v0 += (uint64_t)kThreads * kUnroll) {
        T r[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const uint64_t v = v0 + (uint64_t)k * kThreads;
            if (v < n) r[k] = ld_stream(s + v);
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const uint64_t v = v0 + (uint64_t)k * kThreads;
            if (v < n) st_stream(d + v, r[k]);
        }
    }
}

// The bfloat16 nearest to the exact product q*s (ties to even).  The binary32
// product p = RN(q*s) rounds to the same bfloat16 as the exact value unless p is
// itself a bfloat16 midpoint (low 16 bits 0x8000): every midpoint is a binary32
// number, so a closer one cannot lie between q*s and p.  At a midpoint the sign of
// the exact residual q*s - p, which one fused multiply-add returns (the
// "TwoProduct" error-free transformation of Ogita, Rump and Oishi, "Accurate sum
// and dot product", 2005), decides the direction.
__device__ __forceinline__ unsigned dq_bf16(float q, float s)
{
    const float p = __fmul_rn(q, s);
    unsigned r = __bfloat16_as_ushort(__float2bfloat16_rn(p));
    const unsigned b = __float_as_uint(p);
    if ((b & 0xFFFFu) == 0x8000u && (b & 0x7F800000u) != 0x7F800000u) {
        const float e = __fmaf_rn(q, s, -p);
        if (e != 0.0f) r = (b >> 16) + (((e > 0.0f) == (p > 0.0f)) ? 1u : 0u);
    }
    return r;
}

__device__ __forceinline__ unsigned dq_pair(unsigned w, int k, float s)
{
    const float lo = (float)(signed char)(w >> (16 * k));
    const float hi = (float)(signed char)(w >> (16 * k + 8));
    return dq_bf16(lo, s) | (dq_bf16(hi, s) << 16);
}

// int8 rows -> bfloat16 rows, 16 elements per vector; rows of `vpr` vectors.
__device__ __forceinline__ void dequant_run16(const char* __restrict__ src, char* __restrict__ dst,
                                              const float* __restrict__ scales, uint32_t n,
                                              uint32_t vpr)
{
    const uint4* s = reinterpret_cast<const uint4*>(src);
    uint4* d = reinterpret_cast<uint4*>(dst);
    for (uint32_t v0 = threadIdx.x; v0 < n; v0 += kThreads * kUnroll) {
        uint4 q[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const uint32_t v = v0 + k * kThreads;
            if (v < n) q[k] = ld_stream(s + v);
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const uint32_t v = v0 + k * kThreads;
            if (v < n) {
                const float sc = __ldg(scales + v / vpr);
                uint4 o0, o1;
                o0.x = dq_pair(q[k].x, 0, sc);
                o0.y = dq_pair(q[k].x, 1, sc);
                o0.z = dq_pair(q[k].y, 0, sc);
                o0.w = dq_pair(q[k].y, 1, sc);
                o1.x = dq_pair(q[k].z, 0, sc);
                o1.y = dq_pair(q[k].z, 1, sc);
                o1.z = dq_pair(q[k].w, 0, sc);
                o1.w = dq_pair(q[k].w, 1, sc);
                st_stream(d + 2 * v, o0);
                st_stream(d + 2 * v + 1, o1);
            }
        }
    }
}

// Element-wise fallback for rows whose length is not a multiple of 16 elements.
__device__ __forceinline__ void dequant_run1(const char* __restrict__ src, char* __restrict__ dst,
                                             const float* __restrict__ scales, uint64_t n,
                                             uint64_t row_elems)
{
    const signed char* s = reinterpret_cast<const signed char*>(src);
    unsigned short* d = reinterpret_cast<unsigned short*>(dst);
    for (uint64_t e = threadIdx.x; e < n; e += kThreads)
        d[e] = (unsigned short)dq_bf16((float)s[e], __ldg(scales + e / row_elems));
}

template <int MODE, typename IndexT, int VEC>
__global__ void __launch_bounds__(kThreads) copy_kernel(const CopyArgs a)
{
    __shared__ unsigned long long s_src[kThreads], s_dst[kThreads], s_scale[kThreads];
    __shared__ unsigned s_rows[kThreads];

    uint64_t total;
    if (MODE == kGather || MODE == kDequant || MODE == kAppend) {
        if (a.hdr->verdict != kVerdictOk) return;  // the plan rejected the batch
        total = a.hdr->total_units;
    } else {
        total = a.lane_units;
    }
    const uint64_t G = gridDim.x, b = blockIdx.x;
    const uint64_t per = total / G, rem = total % G;
    const uint64_t lo = b * per + umin(b, rem);
    const uint64_t hi = lo + per + (b < rem ? 1 : 0);

    for (uint64_t u0 = lo; u0 < hi; u0 += kThreads) {
        const uint64_t u = u0 + threadIdx.x;
        if (u < hi) {
            const Unit r = resolve<MODE, IndexT>(a, u);
            s_src[threadIdx.x] = r.src;
            s_dst[threadIdx.x] = r.dst;
            s_scale[threadIdx.x] = r.scale;
            s_rows[threadIdx.x] = r.rows;
        }
        __syncthreads();
        const int nb = (int)umin(kThreads, hi - u0);
        for (int i = 0; i < nb; ++i) {
            const unsigned rows = s_rows[i];
            if (rows == 0) continue;
            if (MODE == kDequant) {
                if (VEC == 16)
                    dequant_run16(a.src + s_src[i], a.dst + s_dst[i], a.scales + s_scale[i],
                                  (uint32_t)(rows * a.row_elems / 16),
                                  (uint32_t)(a.row_elems / 16));
                else
                    dequant_run1(a.src + s_src[i], a.dst + s_dst[i], a.scales + s_scale[i],
                                 rows * a.row_elems, a.row_elems);
            } else {
                copy_run<VEC>(a.src + s_src[i], a.dst + s_dst[i], rows * a.row_bytes / VEC);
            }
        }
        __syncthreads();
    }
}

template <int MODE, typename IndexT, int VEC>
int launch_t(const CopyArgs& a, cudaStream_t st)
{
    auto kern = copy_kernel<MODE, IndexT, VEC>;
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, 0) != cudaSuccess)
        return HP_ERR_CUDA;
    uint64_t grid = (uint64_t)sms * (uint64_t)std::max(per_sm, 1);
    if (MODE == kLaneGather || MODE == kLaneAppend) grid = std::min<uint64_t>(grid, a.lane_units);
    if (grid == 0) return HP_OK;
    kern<<<(unsigned)grid, kThreads, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? HP_OK : HP_ERR_CUDA;
}

template <int MODE, typename IndexT>
int launch_vec(const CopyArgs& a, int vec, cudaStream_t st)
{
    if (MODE == kDequant) return vec == 16 ? launch_t<MODE, IndexT, 16>(a, st)
                                           : launch_t<MODE, IndexT, 1>(a, st);
    switch (vec) {
    case 16: return launch_t<MODE, IndexT, 16>(a, st);
    case 8: return launch_t<MODE, IndexT, 8>(a, st);
    case 4: return launch_t<MODE, IndexT, 4>(a, st);
    case 2: return launch_t<MODE, IndexT, 2>(a, st);
    default: return launch_t<MODE, IndexT, 1>(a, st);
    }
}

}  // namespace

int launch_copy(CopyMode mode, int index_u64, const CopyArgs& a, int vec, void* stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
#ifndef HP_COPY_ENGINE_LDG
    if (vec == 16 && mode != kDequant) return launch_bulk(mode, index_u64, a, stream);
#endif
    switch (mode) {
    case kGather:
        return index_u64 ? launch_vec<kGather, unsigned long long>(a, vec, st)
                         : launch_vec<kGather, unsigned int>(a, vec, st);
    case kDequant:
        return index_u64 ? launch_vec<kDequant, unsigned long long>(a, vec, st)
                         : launch_vec<kDequant, unsigned int>(a, vec, st);
    case kAppend:
        return index_u64 ? launch_vec<kAppend, unsigned long long>(a, vec, st)
                         : launch_vec<kAppend, unsigned int>(a, vec, st);
    case kLaneGather:
        return launch_vec<kLaneGather, unsigned long long>(a, vec, st);
    case kLaneAppend:
        return launch_vec<kLaneAppend, unsigned long long>(a, vec, st);
    }
    return HP_ERR_ARG;
}

}  // namespace hp
