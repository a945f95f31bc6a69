// hp_attention.cu -- decode attention that reads K and V straight through the block table.
//
// "Visualize PagedAttention block layout", How the attention kernel uses the block table:
// the attention kernel iterates over a sequence's blocks, loading each block's keys and
// values through the table.  Here: for sequence s and query head qh (K/V head
// g = qh / G, G = Hq / H_kv), score_t = scale * q . K(s,t,g) for t < len_s, softmax over t,
// out = sum_t weight_t V(s,t,g); every K(s,t,g) / V(s,t,g) row is the Element Lookup of
// "Block-Paged Layout -- Hurray Format Specification".
//
// Decode attention reads every key and value once for about 2G flops per byte, so it is
// bound by HBM, not by arithmetic: it runs on the CUDA cores.
//   attn_kernel     one CTA per (sequence, chunk of chunk_pages pages, group of <= 8 K/V
//                   heads); warp w takes K/V head 8*group + w, so a CTA reads each token's
//                   rows of those heads as one contiguous run.  Lane l owns dims
//                   [l*E, l*E+E) (E = D/32).  Tokens go 32/G at a time: the 32 (token,
//                   head) partial dot products are summed across the warp with a
//                   transposed butterfly (31 shuffles, lane l ends with pair l), then an
//                   online softmax per head updates the running max, sum and the lane's
//                   E dims of each head's weighted value sum.  Each chunk leaves
//                   (max, sum, acc[D]) per query head in the workspace.
//   combine_kernel  one warp per (sequence, query head) merges its chunks' partials.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "hp_internal.cuh"
#include "hp_resolve.cuh"

namespace hp {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

template <int E> struct Pack;
template <> struct Pack<2> { using T = unsigned int; };
template <> struct Pack<4> { using T = uint2; };
template <> struct Pack<8> { using T = uint4; };

template <bool BF16>
__device__ __forceinline__ float to_f32(unsigned short v)
{
    if (BF16) return __uint_as_float((unsigned)v << 16);
    return __half2float(__ushort_as_half(v));
}

template <bool BF16, int E>
__device__ __forceinline__ void unpack(const typename Pack<E>::T& raw, float f[E])
{
    const unsigned short* h = reinterpret_cast<const unsigned short*>(&raw);
#pragma unroll
    for (int k = 0; k < E; ++k) f[k] = to_f32<BF16>(h[k]);
}

// E consecutive 16-bit elements at p (E*2 bytes, aligned) as floats.
template <bool BF16, int E>
__device__ __forceinline__ void load_row(const unsigned short* p, float f[E])
{
    typename Pack<E>::T raw = __ldg(reinterpret_cast<const typename Pack<E>::T*>(p));
    const unsigned short* h = reinterpret_cast<const unsigned short*>(&raw);
#pragma unroll
    for (int k = 0; k < E; ++k) f[k] = to_f32<BF16>(h[k]);
}

template <typename IndexT, bool BF16, int G, int E>
__global__ void __launch_bounds__(kThreads, 2) attn_kernel(const AttnArgs a)
{
    // TS tokens per step: their TS*G (token, head) dot products fill NP <= 32 slots, and the
    // step's raw K and V rows take TS*E registers (at most 64).
    constexpr int TS = (32 / G) < (64 / E) ? (32 / G) : (64 / E);
    constexpr int NP = TS * G;  // partial dot products per step
    constexpr int R = 32 / NP;  // lanes holding the same reduced partial
    pdl_wait();                 // the plan before this launch is complete
    if (a.hdr->verdict != kVerdictOk) return;
    const unsigned warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t items = a.hdr->total_units * a.hgroups;
    const IndexT* table = static_cast<const IndexT*>(a.table);
    const IndexT* sp = static_cast<const IndexT*>(a.seq_ptr);
    const IndexT* lens = static_cast<const IndexT*>(a.lens);
    const unsigned short* K = static_cast<const unsigned short*>(a.k_pool);
    const unsigned short* V = static_cast<const unsigned short*>(a.v_pool);
    const unsigned short* Q = static_cast<const unsigned short*>(a.q);
    const uint64_t P = a.page_size, D = a.D;
    // the reduced partial lane l holds: token j / G, head j % G of the step
    const unsigned j = lane / R, my_tok = j / G, my_head = j % G;

    for (uint64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const uint64_t u = it / a.hgroups;
        const uint32_t g = (uint32_t)(it - u * a.hgroups) * kWarps + warp;
        if (g >= a.Hkv) continue;  // whole warp; no block-wide barrier below
        const uint64_t s = find_seq(a.units_off, a.num_seqs, u);
        const uint64_t c = u - a.units_off[s];
        const uint64_t len = lens[s];
        const uint64_t t_begin = c * a.chunk_pages * P;
        const uint64_t t_end = umin(len, t_begin + a.chunk_pages * P);
        const uint64_t tab0 = sp[s];

        float qv[G][E];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            load_row<BF16, E>(Q + ((s * a.Hq + (uint64_t)g * G + h) * D + lane * E), qv[h]);
#pragma unroll
            for (int k = 0; k < E; ++k) qv[h][k] *= a.scale;
        }
        float m[G], l[G], acc[G][E];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m[h] = -INFINITY;
            l[h] = 0.0f;
#pragma unroll
            for (int k = 0; k < E; ++k) acc[h][k] = 0.0f;
        }

        // the chunk's page IDs, one per lane (a chunk has at most 32 pages)
        const uint64_t n_pg = (t_end - t_begin + P - 1) / P;
        const unsigned long long my_page =
            lane < n_pg ? (unsigned long long)table[tab0 + c * a.chunk_pages + lane] : 0ull;

        for (uint64_t t0 = t_begin; t0 < t_end; t0 += TS) {
            // every K and V row of the step is requested before any arithmetic
            typename Pack<E>::T kraw[TS], vraw[TS];
#pragma unroll
            for (int i = 0; i < TS; ++i) {
                const uint64_t t = t0 + i;
                if (t < t_end) {  // uniform across the warp
                    const unsigned long long page =
                        __shfl_sync(0xffffffffu, my_page, (int)((t - t_begin) / P));
                    const uint64_t row = ((page * P + t % P) * a.Hkv + g) * D + lane * E;
                    kraw[i] = __ldg(reinterpret_cast<const typename Pack<E>::T*>(K + row));
                    vraw[i] = __ldg(reinterpret_cast<const typename Pack<E>::T*>(V + row));
                } else {
                    kraw[i] = typename Pack<E>::T{};
                    vraw[i] = typename Pack<E>::T{};
                }
            }
            float part[NP];  // (token i, head h) at i*G + h
#pragma unroll
            for (int i = 0; i < TS; ++i) {
                float kf[E];
                unpack<BF16, E>(kraw[i], kf);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float d = 0.0f;
#pragma unroll
                    for (int k = 0; k < E; ++k) d = fmaf(qv[h][k], kf[k], d);
                    part[i * G + h] = d;
                }
            }
            // transposed butterfly over the top log2(NP) lane bits: lane l keeps slot l / R
            // summed over those bits; a plain butterfly over the low bits finishes the sum.
#pragma unroll
            for (int o = 16, n = NP; n > 1; o >>= 1, n >>= 1) {
                const bool upper = lane & o;
#pragma unroll
                for (int k = 0; k < n / 2; ++k) {
                    const float send = upper ? part[k] : part[k + n / 2];
                    const float keep = upper ? part[k + n / 2] : part[k];
                    part[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
#pragma unroll
            for (int o = R / 2; o >= 1; o >>= 1) part[0] += __shfl_xor_sync(0xffffffffu, part[0], o);
            const float sc = (t0 + my_tok < t_end) ? part[0] : -INFINITY;
            // per-head step maximum: lanes of one head differ only in the token bits (>= R*G)
            float bm = sc;
#pragma unroll
            for (int o = R * G; o < 32; o <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
            float mnew[G], corr[G], my_m = 0.0f;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                mnew[h] = fmaxf(m[h], __shfl_sync(0xffffffffu, bm, h * R));
                corr[h] = expf(m[h] - mnew[h]);  // 0 on the first step (m = -inf)
                if ((int)my_head == h) my_m = mnew[h];
            }
            const float p = expf(sc - my_m);  // 0 for tokens past the chunk
            float ps = p;
#pragma unroll
            for (int o = R * G; o < 32; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                l[h] = l[h] * corr[h] + __shfl_sync(0xffffffffu, ps, h * R);
                m[h] = mnew[h];
#pragma unroll
                for (int k = 0; k < E; ++k) acc[h][k] *= corr[h];
            }
#pragma unroll
            for (int i = 0; i < TS; ++i) {
                float vf[E];
                unpack<BF16, E>(vraw[i], vf);  // zero rows past the chunk: weight 0
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float w = __shfl_sync(0xffffffffu, p, (i * G + h) * R);
#pragma unroll
                    for (int k = 0; k < E; ++k) acc[h][k] = fmaf(w, vf[k], acc[h][k]);
                }
            }
        }
        float* out = a.partials + (u * a.Hq + (uint64_t)g * G) * (D + 2);
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float* o = out + h * (D + 2);
            if (lane == 0) {
                o[0] = m[h];
                o[1] = l[h];
            }
#pragma unroll
            for (int k = 0; k < E; ++k) o[2 + lane * E + k] = acc[h][k];
        }
    }
}

// One warp per (sequence, query head): merge the chunks' (max, sum, acc) partials.
__global__ void __launch_bounds__(256) combine_kernel(const AttnArgs a)
{
    pdl_wait();
    if (a.hdr->verdict != kVerdictOk) return;
    const unsigned lane = threadIdx.x & 31;
    const uint64_t pairs = a.num_seqs * a.Hq, D = a.D;
    const uint64_t warps = (uint64_t)gridDim.x * (blockDim.x / 32);
    for (uint64_t w = (uint64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); w < pairs;
         w += warps) {
        const uint64_t s = w / a.Hq, qh = w - s * a.Hq;
        const uint64_t c0 = a.units_off[s], c1 = a.units_off[s + 1];
        float* out = a.out + w * D;
        float M = -INFINITY;
        for (uint64_t c = c0; c < c1; ++c) M = fmaxf(M, a.partials[(c * a.Hq + qh) * (D + 2)]);
        float L = 0.0f;
        for (uint64_t c = c0; c < c1; ++c) {
            const float* pc = a.partials + (c * a.Hq + qh) * (D + 2);
            L += pc[1] * expf(pc[0] - M);
        }
        for (uint64_t d = lane; d < D; d += 32) {
            float acc = 0.0f;
            for (uint64_t c = c0; c < c1; ++c) {
                const float* pc = a.partials + (c * a.Hq + qh) * (D + 2);
                acc = fmaf(pc[2 + d], expf(pc[0] - M), acc);
            }
            out[d] = c1 > c0 ? acc / L : 0.0f;
        }
    }
}

template <typename IndexT, bool BF16, int G, int E>
int launch_g(const AttnArgs& a, cudaStream_t st)
{
    int dev = 0;
    const int sms = current_sms(&dev);
    if (sms == 0) return HP_ERR_CUDA;
    const int per_sm = resident_ctas<attn_kernel<IndexT, BF16, G, E>>(dev, kThreads, 0);
    if (per_sm == 0) return HP_ERR_CUDA;
    if (launch_dependent(attn_kernel<IndexT, BF16, G, E>, (unsigned)(sms * per_sm), kThreads, 0,
                         st, a) != cudaSuccess)
        return HP_ERR_CUDA;
    uint64_t g2 = (a.num_seqs * a.Hq + 7) / 8;
    const uint64_t cap = (uint64_t)sms * 8;
    g2 = g2 == 0 ? 1 : (g2 < cap ? g2 : cap);
    return launch_dependent(combine_kernel, (unsigned)g2, 256, 0, st, a) == cudaSuccess
               ? HP_OK
               : HP_ERR_CUDA;
}

template <typename IndexT, bool BF16, int E>
int launch_e(const AttnArgs& a, cudaStream_t st)
{
    switch (a.G) {
    case 1: return launch_g<IndexT, BF16, 1, E>(a, st);
    case 2: return launch_g<IndexT, BF16, 2, E>(a, st);
    case 4: return launch_g<IndexT, BF16, 4, E>(a, st);
    case 8: return launch_g<IndexT, BF16, 8, E>(a, st);
    default: return HP_ERR_ARG;
    }
}

template <typename IndexT, bool BF16>
int launch_b(const AttnArgs& a, cudaStream_t st)
{
    switch (a.D) {
    case 64: return launch_e<IndexT, BF16, 2>(a, st);
    case 128: return launch_e<IndexT, BF16, 4>(a, st);
    case 256: return launch_e<IndexT, BF16, 8>(a, st);
    default: return HP_ERR_ARG;
    }
}

}  // namespace

int launch_attention(int index_u64, const AttnArgs& a, void* stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (index_u64)
        return a.elem_bf16 ? launch_b<unsigned long long, true>(a, st)
                           : launch_b<unsigned long long, false>(a, st);
    return a.elem_bf16 ? launch_b<unsigned int, true>(a, st) : launch_b<unsigned int, false>(a, st);
}

}  // namespace hp
