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

#include "hp_dequant.cuh"
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

// One warp copies `n` vectors (units small enough that a CTA-wide copy would leave
// most of each thread's unrolled loads unused).
template <int VEC>
__device__ __forceinline__ void copy_run_warp(const char* __restrict__ src, char* __restrict__ dst,
                                              uint64_t n)
{
    using T = typename Vec<VEC>::T;
    const T* s = reinterpret_cast<const T*>(src);
    T* d = reinterpret_cast<T*>(dst);
    const unsigned lane = threadIdx.x & 31;
    for (uint64_t v0 = lane; v0 < n; v0 += 32 * kUnroll) {
        T r[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const uint64_t v = v0 + (uint64_t)k * 32;
            if (v < n) r[k] = ld_stream(s + v);
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const uint64_t v = v0 + (uint64_t)k * 32;
            if (v < n) st_stream(d + v, r[k]);
        }
    }
}

__device__ __forceinline__ uint2 ld_stream8(const uint2* p)
{
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p));
    return v;
}

// 8-byte loads in flight per thread, by measurement on GB300 (a 2.5 GB pool, fraction of
// the copy bandwidth): per slot 0.85 / 0.90 / 0.81 at 16 / 12 / 24; per head 0.83 at 8,
// 0.86 at 12; per head_dim 0.84 at 8, 0.79 at 6 and 12.  With the packed conversion at 3
// CTAs per SM (the 13 GB pool): per slot 0.949 / 0.945 / 0.897 at 10 / 12 / 16, per slot
// affine 0.936 / 0.929 / 0.902, per tensor 0.918 / 0.923 / 0.903.  Fewer loads leave too
// little in flight; more cost registers and resident CTAs.
#ifndef HP_DQ_UNROLL
#define HP_DQ_UNROLL 10
#endif
#ifndef HP_DQ_UNROLL_DIM
#define HP_DQ_UNROLL_DIM 8
#endif
constexpr int kDqUnroll = HP_DQ_UNROLL;
constexpr int kDqUnrollDim = HP_DQ_UNROLL_DIM;  // per-head_dim scales and zero points
#ifndef HP_DQ_DIM_HOIST
#define HP_DQ_DIM_HOIST 0
#endif
// Per-head_dim scales and zero points held in registers cost 16 live values per thread
// (101 registers, 2 CTAs per SM); read per group from L1 instead the kernel keeps 4 CTAs
// per SM and its loads in flight (0.76 -> 0.83 of the copy bandwidth on a 2.5 GB pool).
constexpr bool kDqDimHoist = HP_DQ_DIM_HOIST;

// 8-bit rows -> bfloat16 rows, 8 elements per thread step.  `n8` groups of 8; the row of
// group v within the unit is v / (row_elems/8) and, for per-channel schemes, its head is
// (v mod row_elems/8) / (head_dim/8) (both by invariant-divisor multiplication).
// `slot0` is the unit's first page-slot index (per-block-affine parameters).
template <int Q>
__device__ __forceinline__ void dequant_run8(const CopyArgs& a, const char* __restrict__ src,
                                             char* __restrict__ dst, uint64_t slot0, uint32_t n8)
{
    constexpr int kScheme = Q >> 1;
    constexpr bool kZp = Q & 1;
    const bool sgn = a.q_signed != 0;
    const float* __restrict__ scales = a.scales;
    const unsigned char* __restrict__ zps = a.q_zp;
    float s_t = 0.0f, z_t = 0.0f;  // per-tensor parameters, loaded once
    if (kScheme == kQTensor) {
        s_t = __ldg(scales);
        if (kZp) z_t = code_to_f32(__ldg(zps), sgn);
    }
    // Per head, when the groups of a row divide the CTA's width (q_fixed) every group a
    // thread handles sits at the same place in its row, so its scale and zero point are
    // loaded once here.
    float sc_f[8], zc_f[8];
    const bool fixed = (kScheme == kQHead || (kScheme == kQDim && kDqDimHoist)) && a.q_fixed;
    if (fixed) {
        const uint32_t g = threadIdx.x & (a.q_gpr - 1);
        const uint32_t h = div_invariant(g, a.q_hd_m, a.q_hd_l);
        if (kScheme == kQHead) {
            const float s1 = __ldg(scales + h);
            const float z1 = kZp ? code_to_f32(__ldg(zps + h), sgn) : 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                sc_f[e] = s1;
                zc_f[e] = z1;
            }
        } else {
            const uint32_t d0 = (g - h * a.q_gph) * 8;
            const float4 lo = __ldg(reinterpret_cast<const float4*>(scales + d0));
            const float4 hi = __ldg(reinterpret_cast<const float4*>(scales + d0 + 4));
            sc_f[0] = lo.x; sc_f[1] = lo.y; sc_f[2] = lo.z; sc_f[3] = lo.w;
            sc_f[4] = hi.x; sc_f[5] = hi.y; sc_f[6] = hi.z; sc_f[7] = hi.w;
            if (kZp) codes_to_f32(__ldg(reinterpret_cast<const uint2*>(zps + d0)), sgn, zc_f);
            else {
#pragma unroll
                for (int e = 0; e < 8; ++e) zc_f[e] = 0.0f;
            }
        }
    }
    // per slot with zero points (per-block-affine) keeps 8 in flight: 0.953 of the copy
    // bandwidth against 0.940 at 10 (two alternating passes on GB300, 13 GB pool)
    constexpr int kU = kScheme == kQDim ? kDqUnrollDim : (kScheme == kQSlot && kZp) ? 8 : kDqUnroll;
    const uint2* s = reinterpret_cast<const uint2*>(src);
    uint4* d = reinterpret_cast<uint4*>(dst);
    // per slot: when a row's groups divide the CTA width, the row of group v0 + k * kThreads
    // is the row of v0 plus k * (kThreads / groups per row), one division per pass
    const uint32_t rstep = kScheme == kQSlot && kThreads % a.q_gpr == 0 ? kThreads / a.q_gpr : 0;
    for (uint32_t v0 = threadIdx.x; v0 < n8; v0 += kThreads * kU) {
        const uint32_t r0 = rstep ? div_invariant(v0, a.div_m, a.div_l) : 0;
        uint2 q[kU];
#pragma unroll
        for (int k = 0; k < kU; ++k) {
            const uint32_t v = v0 + k * kThreads;
            if (v < n8) q[k] = ld_stream8(s + v);
        }
#pragma unroll
        for (int k = 0; k < kU; ++k) {
            const uint32_t v = v0 + k * kThreads;
            if (v >= n8) continue;
            float sc[8], zc[8];
            if (kScheme == kQSlot || kScheme == kQTensor) {
                float s1 = s_t, z1 = z_t;
                if (kScheme == kQSlot) {
                    const uint64_t i =
                        slot0 + (rstep ? r0 + k * rstep : div_invariant(v, a.div_m, a.div_l));
                    s1 = __ldg(scales + i);
                    if (kZp) z1 = code_to_f32(__ldg(zps + i), sgn);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    sc[e] = s1;
                    zc[e] = z1;
                }
            } else if (fixed) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    sc[e] = sc_f[e];
                    zc[e] = zc_f[e];
                }
            } else {
                const uint32_t r = div_invariant(v, a.div_m, a.div_l);
                const uint32_t g = v - r * a.q_gpr;          // group within the row
                const uint32_t h = div_invariant(g, a.q_hd_m, a.q_hd_l);
                if (kScheme == kQHead) {
                    const float s1 = __ldg(scales + h);
                    const float z1 = kZp ? code_to_f32(__ldg(zps + h), sgn) : 0.0f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        sc[e] = s1;
                        zc[e] = z1;
                    }
                } else {
                    const uint32_t d0 = (g - h * a.q_gph) * 8;  // first feature of the group
                    const float4 lo = __ldg(reinterpret_cast<const float4*>(scales + d0));
                    const float4 hi = __ldg(reinterpret_cast<const float4*>(scales + d0 + 4));
                    sc[0] = lo.x; sc[1] = lo.y; sc[2] = lo.z; sc[3] = lo.w;
                    sc[4] = hi.x; sc[5] = hi.y; sc[6] = hi.z; sc[7] = hi.w;
                    if (kZp) codes_to_f32(__ldg(reinterpret_cast<const uint2*>(zps + d0)), sgn, zc);
                }
            }
            if (!kZp) {
#pragma unroll
                for (int e = 0; e < 8; ++e) zc[e] = 0.0f;
            }
            st_stream(d + v, dequant8(q[k], sgn, zc, sc));
        }
    }
}

// Element-wise fallback for rows (or, per channel, heads) that do not split into groups
// of 8 elements.
template <int Q>
__device__ __forceinline__ void dequant_run1(const CopyArgs& a, const char* __restrict__ src,
                                             char* __restrict__ dst, uint64_t slot0, uint64_t n)
{
    constexpr int kScheme = Q >> 1;
    constexpr bool kZp = Q & 1;
    const bool sgn = a.q_signed != 0;
    const unsigned char* s = reinterpret_cast<const unsigned char*>(src);
    unsigned short* d = reinterpret_cast<unsigned short*>(dst);
    for (uint64_t e = threadIdx.x; e < n; e += kThreads) {
        const uint64_t r = e / a.row_elems, c = e - r * a.row_elems;
        uint64_t i = 0;
        if (kScheme == kQSlot) i = slot0 + r;
        else if (kScheme == kQHead) i = c / a.q_head_dim;
        else if (kScheme == kQDim) i = c % a.q_head_dim;
        float f = code_to_f32(s[e], sgn);
        if (kZp) f -= code_to_f32(__ldg(a.q_zp + i), sgn);
        d[e] = (unsigned short)dq_bf16(f, __ldg(a.scales + i));
    }
}

template <int MODE, typename IndexT, int VEC, bool WARP_UNITS, int Q = 0>
__global__ void __launch_bounds__(kThreads) copy_kernel(const CopyArgs a)
{
    __shared__ unsigned long long s_src[kThreads], s_dst[kThreads], s_scale[kThreads];
    __shared__ unsigned s_rows[kThreads];

    uint64_t total;
    if (MODE == kGather || MODE == kDequant || MODE == kAppend) {
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

    if constexpr (WARP_UNITS) {
        // Each warp resolves 32 units at a time (one per lane) and copies them one after
        // the other, descriptors handed over by shuffle: no CTA-wide barrier, so one
        // warp's resolution overlaps the other warps' copies.
        const unsigned lane = threadIdx.x & 31;
        for (uint64_t w0 = lo + (threadIdx.x >> 5) * 32; w0 < hi; w0 += kThreads) {
            Unit r{0, 0, 0, 0};
            if (w0 + lane < hi) r = resolve<MODE, IndexT>(a, w0 + lane);
            const int nb = (int)umin(32, hi - w0);
            for (int i = 0; i < nb; ++i) {
                const unsigned rows = __shfl_sync(0xffffffffu, r.rows, i);
                if (rows == 0) continue;
                const unsigned long long us = __shfl_sync(0xffffffffu, r.src, i);
                const unsigned long long ud = __shfl_sync(0xffffffffu, r.dst, i);
                copy_run_warp<VEC>(a.src + us, a.dst + ud, rows * a.row_bytes / VEC);
            }
        }
    } else {
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
                        dequant_run8<Q>(a, a.src + s_src[i], a.dst + s_dst[i], s_scale[i],
                                        (uint32_t)(rows * a.row_elems / 8));
                    else
                        dequant_run1<Q>(a, a.src + s_src[i], a.dst + s_dst[i], s_scale[i],
                                        rows * a.row_elems);
                } else {
                    copy_run<VEC>(a.src + s_src[i], a.dst + s_dst[i], rows * a.row_bytes / VEC);
                }
            }
            __syncthreads();
        }
    }
}

template <int MODE, typename IndexT, int VEC, bool WARP_UNITS, int Q = 0>
int launch_t(const CopyArgs& a, cudaStream_t st)
{
    auto kern = copy_kernel<MODE, IndexT, VEC, WARP_UNITS, Q>;
    int dev = 0;
    const int sms = current_sms(&dev);
    const int per_sm =
        sms ? resident_ctas<copy_kernel<MODE, IndexT, VEC, WARP_UNITS, Q>>(dev, kThreads, 0) : 0;
    if (sms == 0 || per_sm == 0) return HP_ERR_CUDA;
    // dequantising gathers: at most 3 CTAs per SM except per head_dim, whose scales and zero
    // points are read per group (measured on GB300: per slot 0.891 -> 0.945 of the copy
    // bandwidth with 3 instead of 4, per head 0.896 -> 0.935, per slot affine 0.886 -> 0.929,
    // per tensor unchanged; per head_dim 0.901 with 4, 0.827 with 3)
    const bool cap3 = MODE == kDequant && (Q >> 1) != kQDim;
    uint64_t grid = (uint64_t)sms * (uint64_t)(cap3 ? std::min(per_sm, 3) : per_sm);
    if (host_counted(MODE)) grid = std::min<uint64_t>(grid, a.lane_units);
    if (grid == 0) return HP_OK;
    if (host_counted(MODE)) {
        kern<<<(unsigned)grid, kThreads, 0, st>>>(a);
        return cudaGetLastError() == cudaSuccess ? HP_OK : HP_ERR_CUDA;
    }
    return launch_dependent(kern, (unsigned)grid, kThreads, 0, st, a) == cudaSuccess ? HP_OK
                                                                                    : HP_ERR_CUDA;
}

template <int MODE, typename IndexT, bool W>
int launch_vec_w(const CopyArgs& a, int vec, cudaStream_t st)
{
    switch (vec) {
    case 16: return launch_t<MODE, IndexT, 16, W>(a, st);
    case 8: return launch_t<MODE, IndexT, 8, W>(a, st);
    case 4: return launch_t<MODE, IndexT, 4, W>(a, st);
    case 2: return launch_t<MODE, IndexT, 2, W>(a, st);
    default: return launch_t<MODE, IndexT, 1, W>(a, st);
    }
}

// Units of at most 8 KiB go one per warp; larger ones are copied by the whole CTA.
template <int MODE, typename IndexT>
int launch_vec(const CopyArgs& a, int vec, cudaStream_t st)
{
    if constexpr (MODE == kDequant) {
        switch (a.q_kind) {
#define HP_DQ(q)                                                                        \
    case q:                                                                             \
        return vec == 16 ? launch_t<MODE, IndexT, 16, false, q>(a, st)                  \
                         : launch_t<MODE, IndexT, 1, false, q>(a, st);
            HP_DQ(0) HP_DQ(1) HP_DQ(2) HP_DQ(3) HP_DQ(4) HP_DQ(5) HP_DQ(6) HP_DQ(7)
#undef HP_DQ
        default: return HP_ERR_ARG;
        }
    } else {
        return a.unit_bytes <= 8192 ? launch_vec_w<MODE, IndexT, true>(a, vec, st)
                                    : launch_vec_w<MODE, IndexT, false>(a, vec, st);
    }
}

}  // namespace

int launch_copy(CopyMode mode, int index_u64, const CopyArgs& a, int vec, void* stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Engine by copy-unit size (measured on GB300): the TMA ring with 8 KiB stages for
    // units of 64 KiB and more, with 16 KiB stages for 16-64 KiB, registers below.
#ifndef HP_BULK_MIN_UNIT
#define HP_BULK_MIN_UNIT 16384
#endif
#ifndef HP_BULK_BIG_STAGES_BELOW
#define HP_BULK_BIG_STAGES_BELOW 65536
#endif
#ifndef HP_COPY_ENGINE_LDG
    if (vec == 16 && mode != kDequant && a.unit_bytes >= HP_BULK_MIN_UNIT)
        return launch_bulk(mode, index_u64, a, a.unit_bytes < HP_BULK_BIG_STAGES_BELOW ? 1 : 0,
                           stream);
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
    case kCopyPages:
        return index_u64 ? launch_vec<kCopyPages, unsigned long long>(a, vec, st)
                         : launch_vec<kCopyPages, unsigned int>(a, vec, st);
    }
    return HP_ERR_ARG;
}

}  // namespace hp
