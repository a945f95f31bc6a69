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
//   attn_kernel     a step is TS tokens of one sequence for one K/V head.  The plan
//                   counts each sequence's steps; CTA b owns an equal share of the
//                   (sequence, step) space for every K/V head, split into R sub-ranges
//                   (R = 8 / H_kv when H_kv < 8, else 1), and warp w takes head w mod H_kv
//                   (or heads w, w+8, ...) of sub-range w / H_kv.  So the warps of a CTA
//                   read the heads of the same tokens together, and every warp runs the
//                   same number of steps whatever the sequence lengths.  A warp streams
//                   each sequence segment of its range into a ring of kStages shared-memory
//                   stages with cp.async (a step's K rows, then its V rows; the pages come
//                   from a window of 32 page IDs held one per lane), so the loads of the
//                   next steps are in flight while it computes.  Lane l owns dims
//                   [l*E, l*E+E) (E = D/32).  The TS*G (token, query head) partial dot
//                   products of a step are summed across the warp with a transposed
//                   butterfly (one shuffle per product), then an online softmax per query
//                   head updates the lane's E dims of the weighted value sum; the running
//                   maxima move (and the sums are rescaled) only on steps where some score
//                   exceeds its head's, and each lane keeps its share of its head's weight
//                   sum.  A warp that covers a whole sequence writes its normalised
//                   result.  Otherwise each segment leaves (max, sum, acc[D]) per query
//                   head as record (s + v) * H_kv + g, v the warp's worker index, and
//                   counts itself done for (s, g); the warp that finishes the last
//                   segment merges the records into the result, so no second kernel and
//                   no pass over the sequences follow.
// Records: acc [records, G, D] and (max, sum) [records, G] in the workspace after the
// plan, then one count per (sequence, K/V head): zeroed by the plan, and set back to zero
// by the warp that merges, so planned calls can follow one another on one workspace.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "hp_attn.cuh"
#include "hp_attn_merge.cuh"
#include "hp_internal.cuh"
#include "hp_resolve.cuh"

namespace hp {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;  // per-warp ring of shared-memory stages

template <int E> struct Pack;
template <> struct Pack<2> { using T = unsigned int; };
template <> struct Pack<4> { using T = uint2; };
template <> struct Pack<8> { using T = uint4; };

// Geometry of one step for G query heads per K/V head and E = D/32 dims per lane.
template <int G, int E> struct Step {
    // TS tokens per step: their TS*G (token, head) dot products fill NP <= 32 slots and a
    // stage (the step's K rows, then its V rows) is at most 4 KiB.
    static constexpr int TS = (32 / G) < (32 / E) ? (32 / G) : (32 / E);
    static constexpr int NP = TS * G;        // partial dot products per step
    static constexpr int R = 32 / NP;        // lanes holding the same reduced partial
    static constexpr int ROW = 64 * E;       // bytes of one head's K or V row
    static constexpr int PIECES = ROW / 16;  // 16-byte pieces of a row
    static constexpr int LT = 32 / TS;       // lanes copying one token's rows
    static constexpr int NPC = PIECES / LT;  // pieces of each row a lane copies
    static constexpr int STAGE = 2 * TS * ROW;
    static constexpr int WBUF = 32 * 8;      // the step's weights, each stored twice
    static constexpr int WARP_SMEM = kStages * STAGE + WBUF;
};

template <int G, int E>
constexpr int smem_bytes() { return kWarps * Step<G, E>::WARP_SMEM; }

// Two fp32 values in one 64-bit register pair, for the packed f32x2 arithmetic.
using f2 = unsigned long long;
__device__ __forceinline__ f2 pack2(float lo, float hi)
{
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(f2 v, float& lo, float& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c)
{
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b)
{
    f2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// A 32-bit word of two 16-bit elements as an f2 (element 0 low).
template <bool BF16>
__device__ __forceinline__ f2 widen2(unsigned w)
{
    if (BF16) return pack2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
    return pack2(f.x, f.y);
}

template <bool BF16, int E>
__device__ __forceinline__ void widen_row(const typename Pack<E>::T& raw, f2 v[E / 2])
{
    const unsigned* w = reinterpret_cast<const unsigned*>(&raw);
#pragma unroll
    for (int k = 0; k < E / 2; ++k) v[k] = widen2<BF16>(w[k]);
}

// 16 bytes global -> shared, L2 only; src_bytes 0 stores zeros and reads nothing.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes)
{
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// Request one step's rows: tokens t0 .. t0+TS-1 of the sequence (len tokens), K rows then
// V rows of head g.  The pages come from the window of 32 page IDs whose first slot is
// token wbeg (lane j holds the window's page j; the step lies inside the window).  Lane l copies token
// l / LT: pieces l % LT + LT*m of both rows, so the LT lanes of a token read LT*16
// contiguous bytes per instruction.  Tokens at or past len become zero rows.
template <typename IndexT, int G, int E>
__device__ __forceinline__ void issue_step(const AttnArgs& a, unsigned char* stage, uint64_t t0,
                                           uint64_t len, uint64_t wbeg, IndexT my_page,
                                           uint32_t g, unsigned lane)
{
    using S = Step<G, E>;
    const char* K = static_cast<const char*>(a.k_pool);
    const char* V = static_cast<const char*>(a.v_pool);
    const unsigned i = lane / S::LT, jp = lane % S::LT;
    const uint64_t x = t0 + i;
    const bool live = x < len;
    // offset from the window's first slot: below 32 pages (< 2^31) for a live token
    const uint32_t rel = (uint32_t)(x - wbeg);
    const uint32_t pi = div_invariant(rel, a.p_m, a.p_l);
    const IndexT page = __shfl_sync(0xffffffffu, my_page, (int)(pi & 31));
    const uint64_t slot_row = (uint64_t)page * a.page_size + (rel - pi * (uint32_t)a.page_size);
    const uint64_t off = (slot_row * a.Hkv + g) * S::ROW + jp * 16;
    const char* ks = live ? K + off : K;
    const char* vs = live ? V + off : K;
    const uint32_t n = live ? 16u : 0u;
    unsigned char* kd = stage + i * S::ROW + jp * 16;
#pragma unroll
    for (int m = 0; m < S::NPC; ++m) {
        cp_async16(kd + m * S::LT * 16, ks + m * S::LT * 16, n);
        cp_async16(kd + S::TS * S::ROW + m * S::LT * 16, vs + m * S::LT * 16, n);
    }
}

// G = 8 query heads at D >= 128 keep 64 to 128 fp32 query and accumulator values per
// lane: those variants run one CTA per SM with the registers they need instead of spilling.
template <typename IndexT, bool BF16, int G, int E>
__global__ void __launch_bounds__(kThreads, (G == 8 && E >= 4) ? 1 : 2) attn_kernel(const AttnArgs a)
{
    using S = Step<G, E>;
    constexpr int TS = S::TS, NP = S::NP, R_ = S::R;
    using RowT = typename Pack<E>::T;
    extern __shared__ __align__(16) unsigned char smem[];
    pdl_wait();  // the plan before this launch is complete
    if (a.hdr->verdict != kVerdictOk) return;
    const unsigned warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a sequence without tokens has no step: one warp of the grid writes its zeros
    for (uint64_t s = (uint64_t)blockIdx.x * kWarps + warp; s < a.num_seqs;
         s += (uint64_t)gridDim.x * kWarps)
        if (a.units_off[s] == a.units_off[s + 1]) {
            float4* o = reinterpret_cast<float4*>(a.out + s * a.Hq * a.D);
            for (uint64_t i = lane; i < a.Hq * a.D / 4; i += 32) o[i] = make_float4(0, 0, 0, 0);
        }
    unsigned char* ring = smem + warp * S::WARP_SMEM;
    f2* wbuf = reinterpret_cast<f2*>(ring + kStages * S::STAGE);
    const unsigned short* Q = static_cast<const unsigned short*>(a.q);
    const uint64_t D = a.D;
    // After the reduction lane l holds slot lx = l / R_ (R_ lanes per slot): token lx / G,
    // head lx % G of the step.  Before it, lane l keeps slot k ^ lx at array position k, so every level of
    // the transposed butterfly keeps the low half and sends the high half: position k
    // reads K row (k / G) ^ lt with query head (k % G) ^ lh.
    const unsigned lx = lane / R_, my_tok = lx / G, my_head = lx % G;
    const unsigned lt = my_tok, lh = my_head;
    uint32_t roff[TS];  // byte offset in a stage of the K row position i reads
#pragma unroll
    for (int i = 0; i < TS; ++i) roff[i] = (i ^ lt) * S::ROW + lane * (2 * E);
    const float qscale = a.scale * 1.4426950408889634f;  // scores in log2 units

    const uint64_t S_steps = a.hdr->total_units;  // steps of all sequences, one head
    const uint64_t Lw = (S_steps + a.workers - 1) / a.workers;
    const uint32_t R = a.R;                                 // step ranges per CTA
    const uint32_t r = a.Hkv >= kWarps ? 0 : warp / a.Hkv;  // this warp's sub-range
    if (r >= R || S_steps == 0) return;  // whole warp; no block-wide barrier in this kernel
    const uint64_t v = (uint64_t)blockIdx.x * R + r;       // worker index
    const uint64_t beg = umin(v * Lw, S_steps), end = umin(beg + Lw, S_steps);
    if (beg >= end) return;
    const IndexT* table = static_cast<const IndexT*>(a.table);
    const IndexT* spp = static_cast<const IndexT*>(a.seq_ptr);
    const IndexT* lensp = static_cast<const IndexT*>(a.lens);
    const uint64_t P = a.page_size;
    f2 qp[G][E / 2];   // position h holds query head h ^ lh, scaled
    float m[G];        // each head's running maximum (the same in every lane)
    f2 acc[G][E / 2];  // the lane's dims of each head's weighted value sum
    const uint64_t s_first = find_seq(a.units_off, a.num_seqs, beg);
    for (uint32_t g = a.Hkv >= kWarps ? warp : warp % a.Hkv; g < a.Hkv;
         g += a.Hkv >= kWarps ? kWarps : a.Hkv) {
        // A segment's count of (sequence, head) -- and, for its last segment, the merge --
        // waits until the next segment's first loads are in flight.
        uint64_t pend = ~0ull;  // the sequence of the record waiting to be counted
        auto settle = [&]() {
            if (pend == ~0ull) return;
            __threadfence();  // the record is visible before the count moves
            __syncwarp();
            unsigned done = 0;
            if (lane == 0) done = atomicAdd(a.seg_done + pend * a.Hkv + g, 1u);
            done = __shfl_sync(0xffffffffu, done, 0);
            const uint64_t so = a.units_off[pend], ns = a.units_off[pend + 1] - so;
            const uint64_t f = so / Lw, nr = (so + ns - 1) / Lw - f + 1;
            if (done + 1 == nr) {
                __threadfence();  // every other segment's record is visible
                merge_segments<G, E>(a, ((pend + f) * a.Hkv + g) * G, nr,
                                     a.out + (pend * a.Hq + (uint64_t)g * G) * D + lane * E,
                                     lane);
                // back to zero for the next call on this workspace (no other warp of
                // this launch touches the count any more)
                if (lane == 0) a.seg_done[pend * a.Hkv + g] = 0u;
            }
            pend = ~0ull;
        };
        uint64_t s = s_first;
        for (uint64_t pos = beg; pos < end;) {
            while (a.units_off[s + 1] <= pos) ++s;  // skips sequences without steps
            const uint64_t so = a.units_off[s];
            const uint64_t k0 = pos - so, k1 = umin(a.units_off[s + 1], end) - so;
            pos = so + k1;
            const uint64_t len = lensp[s], tab0 = spp[s];
            // the window of 32 page IDs the issuing steps read from: logical pages
            // pw0 .. pw0+31, tokens [wbeg, wend)
            const uint64_t tab1 = spp[s + 1];
            uint64_t pw0 = k0 * TS / P, wbeg = pw0 * P, wend = wbeg + 32 * P;
            IndexT my_page = tab0 + pw0 + lane < tab1 ? table[tab0 + pw0 + lane] : IndexT(0);
            auto issue = [&](uint64_t k, unsigned char* stage) {
                const uint64_t t0 = k * TS;
                if (umin(t0 + TS, len) > wend) {  // move the window to this step's first page
                    pw0 = t0 / P;
                    wbeg = pw0 * P;
                    wend = wbeg + 32 * P;
                    my_page = tab0 + pw0 + lane < tab1 ? table[tab0 + pw0 + lane] : IndexT(0);
                }
                issue_step<IndexT, G, E>(a, stage, t0, len, wbeg, my_page, g, lane);
            };
#pragma unroll
            for (int j = 0; j < kStages - 1; ++j) {
                if (k0 + j < k1) issue(k0 + j, ring + j * S::STAGE);
                cp_async_commit();
            }
            settle();  // the previous segment's count, behind this one's first loads
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const RowT raw = __ldg(reinterpret_cast<const RowT*>(
                    Q + ((s * a.Hq + (uint64_t)g * G + (hh ^ lh)) * D + lane * E)));
                widen_row<BF16, E>(raw, qp[hh]);
#pragma unroll
                for (int e = 0; e < E / 2; ++e) qp[hh][e] = mul2(qp[hh][e], pack2(qscale, qscale));
                m[hh] = -INFINITY;
#pragma unroll
                for (int e = 0; e < E / 2; ++e) acc[hh][e] = 0ull;
            }
            float my_m = -INFINITY, lp = 0.0f;  // this lane's head: running max, weight sum

            uint32_t slot = 0;
            for (uint64_t k = k0; k < k1; ++k) {
                const uint64_t kn = k + kStages - 1;
                if (kn < k1)
                    issue(kn, ring + (slot == 0 ? kStages - 1 : slot - 1) * S::STAGE);
                cp_async_commit();
                cp_async_wait<kStages - 1>();  // this lane's pieces of step k have landed
                __syncwarp();                  // and every other lane's
                const unsigned char* st = ring + slot * S::STAGE;
                if (++slot == kStages) slot = 0;

                float part[NP];
#pragma unroll
                for (int i = 0; i < TS; ++i) {
                    f2 kv[E / 2];
                    widen_row<BF16, E>(*reinterpret_cast<const RowT*>(st + roff[i]), kv);
#pragma unroll
                    for (int hh = 0; hh < G; ++hh) {
                        f2 d = mul2(qp[hh][0], kv[0]);
#pragma unroll
                        for (int e = 1; e < E / 2; ++e) d = fma2(qp[hh][e], kv[e], d);
                        float d0, d1;
                        unpack2(d, d0, d1);
                        part[i * G + hh] = d0 + d1;
                    }
                }
                // transposed butterfly: every level keeps the low half and sends the high half
#pragma unroll
                for (int o = 16, n = NP; n > 1; o >>= 1, n >>= 1) {
#pragma unroll
                    for (int e = 0; e < n / 2; ++e)
                        part[e] += __shfl_xor_sync(0xffffffffu, part[e + n / 2], o);
                }
#pragma unroll
                for (int o = R_ / 2; o >= 1; o >>= 1) part[0] += __shfl_xor_sync(0xffffffffu, part[0], o);
                const float sc = (k * TS + my_tok < len) ? part[0] : -INFINITY;
                // Online softmax.  The running maxima change only when some score exceeds
                // its head's: then (always on a segment's first step) the step maximum
                // per head moves m and rescales the sums; otherwise the step skips it.
                if (__any_sync(0xffffffffu, sc > my_m)) {
                    // per-head step maximum: lanes of one head differ in the token bits
                    float bm = sc;
#pragma unroll
                    for (int o = R_ * G; o < 32; o <<= 1)
                        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
#pragma unroll
                    for (int hh = 0; hh < G; ++hh) {
                        const float mnew = fmaxf(m[hh], __shfl_sync(0xffffffffu, bm, hh * R_));
                        const float corr = exp2_approx(m[hh] - mnew);  // 0 when m = -inf
                        m[hh] = mnew;
                        const f2 c2 = pack2(corr, corr);
#pragma unroll
                        for (int e = 0; e < E / 2; ++e) acc[hh][e] = mul2(acc[hh][e], c2);
                        if ((int)my_head == hh) {
                            lp *= corr;
                            my_m = mnew;
                        }
                    }
                }
                const float p = exp2_approx(sc - my_m);  // 0 for tokens past the sequence
                lp += p;  // this lane's share of its head's weight sum
                if (lane % R_ == 0) wbuf[lx] = pack2(p, p);
                __syncwarp();  // the weights are in wbuf
#pragma unroll
                for (int i = 0; i < TS; ++i) {
                    f2 vv[E / 2];  // rows past the sequence are zeros with weight 0
                    widen_row<BF16, E>(
                        *reinterpret_cast<const RowT*>(st + (TS + i) * S::ROW + lane * (2 * E)), vv);
#pragma unroll
                    for (int hh = 0; hh < G; ++hh) {
                        const f2 w = wbuf[i * G + hh];
#pragma unroll
                        for (int e = 0; e < E / 2; ++e) acc[hh][e] = fma2(w, vv[e], acc[hh][e]);
                    }
                }
                __syncwarp();  // the stage and wbuf are rewritten by later steps
            }
            // each head's weight sum from its lanes' shares (lanes of one head differ in
            // the token bits; the low bits are copies)
#pragma unroll
            for (int o = R_ * G; o < 32; o <<= 1) lp += __shfl_xor_sync(0xffffffffu, lp, o);
            // the sequence's steps met workers f .. f + nr - 1 (equal shares of Lw steps)
            const uint64_t ns = a.units_off[s + 1] - so;
            const uint64_t f = so / Lw, nr = (so + ns - 1) / Lw - f + 1;
            float* out = a.out + (s * a.Hq + (uint64_t)g * G) * D + lane * E;
            if (nr == 1) {  // the whole sequence: its result, normalised
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const float inv = 1.0f / __shfl_sync(0xffffffffu, lp, hh * R_);
                    f2* o = reinterpret_cast<f2*>(out + hh * D);
#pragma unroll
                    for (int e = 0; e < E / 2; ++e) o[e] = mul2(acc[hh][e], pack2(inv, inv));
                }
                continue;
            }
            // one segment of several: its record now, its count later (settle); the warp
            // that finishes the last one merges them all
            const uint64_t row0 = ((s + v) * a.Hkv + g) * G;
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const float lh = __shfl_sync(0xffffffffu, lp, hh * R_);
                if (lane == 0)
                    reinterpret_cast<float2*>(a.part_ml)[row0 + hh] = make_float2(m[hh], lh);
                f2* o = reinterpret_cast<f2*>(a.part_acc + (row0 + hh) * D + lane * E);
#pragma unroll
                for (int e = 0; e < E / 2; ++e) o[e] = acc[hh][e];
            }
            pend = s;
        }
        settle();
    }
}

template <typename IndexT, bool BF16, int G, int E>
int launch_g(const AttnArgs& a, cudaStream_t st)
{
    constexpr int smem = smem_bytes<G, E>();
    int dev = 0;
    const int sms = current_sms(&dev);
    if (sms == 0) return HP_ERR_CUDA;
    if (!allow_dynamic_smem<attn_kernel<IndexT, BF16, G, E>>(dev, smem)) return HP_ERR_CUDA;
    const int per_sm = resident_ctas<attn_kernel<IndexT, BF16, G, E>>(dev, kThreads, smem);
    if (per_sm == 0) return HP_ERR_CUDA;
    AttnArgs b = a;
    const uint64_t ctas = std::min<uint64_t>((uint64_t)sms * per_sm, HP_ATTN_MAX_CTAS);
    b.workers = ctas * b.R;
    return launch_dependent(attn_kernel<IndexT, BF16, G, E>, (unsigned)ctas, kThreads, smem, st,
                            b) == cudaSuccess
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
