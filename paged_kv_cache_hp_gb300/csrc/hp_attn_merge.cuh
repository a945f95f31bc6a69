// hp_attn_merge.cuh -- pieces shared by the two decode-attention kernels (hp_attention.cu
// on the CUDA cores, hp_attn_tc.cu on the tensor cores): the base-2 exponential and the
// merge of a sequence's segment records into its normalised result.  Scores, maxima and
// weight sums are in log2 units.
#pragma once

#include <cstdint>

#include "hp_attn.cuh"

namespace hp {

__device__ __forceinline__ float exp2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// E floats of a record written earlier in this launch by another warp (L2, not L1).
template <int E>
__device__ __forceinline__ void load_dims(const float* p, float (&x)[E])
{
    if constexpr (E == 2) {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(p));
        x[0] = v.x;
        x[1] = v.y;
    } else {
#pragma unroll
        for (int k = 0; k < E / 4; ++k) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(p) + k);
            x[4 * k] = v.x;
            x[4 * k + 1] = v.y;
            x[4 * k + 2] = v.z;
            x[4 * k + 3] = v.w;
        }
    }
}

// Merges the nr segment records of one (sequence, K/V head) -- record j's query head hh
// at row row0 + j * H_kv * G + hh -- into the G normalised results at out + hh * D (the
// lane's E dims).  The maxima and weight sums first: lane l takes head l % G of records
// l / G, l / G + 32 / G, ... with a running (max, sum), and the lanes of a head merge
// theirs pairwise; then the weighted accumulators, CH records at a time.  PAIR: the
// record's D = 128 dims are two 64-dim K/V heads side by side (head_dim 64 taken two heads
// at a time), query head hh belongs to the first for hh < G / 2 and to the second after
// it, and only its own head's 64 dims are written, to out + hh * 64 (out then carries no
// lane offset).
template <int G, int E, bool PAIR = false>
__device__ __forceinline__ void merge_segments(const AttnArgs& a, uint64_t row0, uint64_t nr,
                                            float* out, unsigned lane)
{
    constexpr int CH = G >= 8 ? 1 : 8 / G;  // records per pass of the accumulator loop
    const float2* ml = reinterpret_cast<const float2*>(a.part_ml);
    const uint64_t stride = (uint64_t)a.Hkv * G, D = a.D;
    float mx = -INFINITY, sm = 0.0f;
    for (uint64_t j = lane / G; j < nr; j += 32 / G) {
        const float2 x = __ldcg(ml + row0 + j * stride + lane % G);  // x.x finite
        const float mn = fmaxf(mx, x.x);
        sm = sm * exp2_approx(mx - mn) + x.y * exp2_approx(x.x - mn);
        mx = mn;
    }
#pragma unroll
    for (int o = G; o < 32; o <<= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, mx, o);
        const float os = __shfl_xor_sync(0xffffffffu, sm, o);
        const float mn = fmaxf(mx, om);
        if (mn != -INFINITY) {
            sm = sm * exp2_approx(mx - mn) + os * exp2_approx(om - mn);
            mx = mn;
        }
    }
    float M[G], acc[G][E];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        M[hh] = __shfl_sync(0xffffffffu, mx, hh);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[hh][e] = 0.0f;
    }
    const float L = sm;  // lane hh < G holds head hh's sum
    for (uint64_t j = 0; j < nr; j += CH) {
        float x[CH][G][E], w[CH][G];
#pragma unroll
        for (int c = 0; c < CH; ++c)
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const uint64_t row = row0 + (j + c < nr ? j + c : j) * stride + hh;
                load_dims<E>(a.part_acc + row * D + lane * E, x[c][hh]);
                w[c][hh] = j + c < nr ? __ldcg(ml + row).x : -INFINITY;
            }
#pragma unroll
        for (int c = 0; c < CH; ++c)
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const float wt = exp2_approx(w[c][hh] - M[hh]);  // 0 past the last record
#pragma unroll
                for (int e = 0; e < E; ++e) acc[hh][e] = fmaf(wt, x[c][hh][e], acc[hh][e]);
            }
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        const float inv = 1.0f / __shfl_sync(0xffffffffu, L, hh);
        float* o = out + hh * D;
        if (PAIR) {
            const unsigned d0 = lane * E, half = (unsigned)(2 * hh / G);
            if ((d0 >> 6) != half) continue;
            o = out + hh * 64 + (d0 & 63);
        }
#pragma unroll
        for (int e = 0; e < E; e += 2)
            *reinterpret_cast<float2*>(o + e) = make_float2(acc[hh][e] * inv, acc[hh][e + 1] * inv);
    }
}

}  // namespace hp
