// hp_attn_tc.cu -- decode attention through the block table on the tensor cores (tcgen05),
// for head_dim 128 and pages of 8-128 slots.
//
// The same computation as hp_attention.cu ("Visualize PagedAttention block layout", How the
// attention kernel uses the block table; K(s,t,g) and V(s,t,g) read through the Element
// Lookup of "Block-Paged Layout -- Hurray Format Specification"): for sequence s and query
// head qh (K/V head g = qh / G), score_t = scale * q . K(s,t,g) over t < len_s, softmax over
// t, out = sum_t weight_t V(s,t,g).  The work is split the same way -- steps balanced over
// workers, segments, records merged by the last segment's finisher -- with a step of 128
// tokens of one K/V head, and the two contractions of a step on the tensor cores:
//   S [128 tokens x 16]  = K [128 x 128 dims] . Q^T        (the G query heads, padded to 16)
//   O^T [128 dims x 16]  = V^T [128 dims x 128 tokens] . P^T
// One CTA per SM, six roles, each running ahead as far as its buffers allow:
//   warps 0, 7  TMA: per step, the K (warp 0) and V (warp 7) rows of the step's pages (one
//               head's 128 dims of P tokens per box, two 64-dim boxes per page, 128-byte
//               swizzled by the tensor map) into rings of 3 stages of 32 KiB, counted on
//               "k_full"/"v_full"; a K stage comes back once S has read it, a V stage once
//               O has;
//   warp 1      tcgen05.mma issue of S (one thread): step j into TMEM buffer j % 2 as soon
//               as its K stage and the segment's Q are in, committed to "s_full";
//   warp 6      tcgen05.mma issue of O (one thread): step j from its V stage and weights,
//               committed to "o_full";
//   warps 2-5   softmax and accumulation, one thread per TMEM lane: a step's scores (lane =
//               token), masked past the sequence, the running maximum per query head (a
//               cross-warp maximum through shared memory), the weights written as bfloat16
//               (or half) pairs hi + lo = p (so P.V keeps about 16 significant bits where a
//               single 16-bit P would keep 8), then the previous step's O (lane = dim) folded
//               into fp32 registers with the usual online-softmax rescaling.
// Rows of V past the sequence (an unfilled last page, or pages a step does not have) are
// zeroed in shared memory before their weights (zero) are handed over, so no stale or
// undefined value reaches the product.  Every wait is bounded (about 2 s); a wait that runs
// out reports HP_ERR_TIMEOUT, and every role then leaves its loop; the loads and the matrix
// operations already issued are waited for (bounded) before the TMEM is freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "hp_attn.cuh"
#include "hp_attn_merge.cuh"
#include "hp_internal.cuh"
#include "hp_resolve.cuh"
#include "hp_tma.cuh"

namespace hp {
namespace {

using namespace tma;

constexpr int kTok = 128;           // tokens per step
constexpr int kD = 128;             // head_dim
constexpr int kN = 16;              // query-head columns of the MMAs (G padded)
constexpr int kKV = 3;              // K/V stages
constexpr uint32_t kHalf = kTok * 128;       // one 64-dim half of a K or V tile (16 KiB)
constexpr uint32_t kTile = 2 * kHalf;        // one K or V tile (32 KiB)
constexpr uint32_t kPBuf = 2 * kN * 128;     // one P operand: 16 rows x 128 tokens (4 KiB)
constexpr uint32_t kQBuf = 2 * kN * 128;     // one Q operand: 16 rows x 128 dims (4 KiB)
constexpr int kThreadsTc = 8 * 32;
constexpr int kSoftmax = 128;       // warps 2-5
constexpr uint32_t kTmemCols = 64;  // S x 2 buffers, O x 2 buffers

// shared memory: K ring, V ring, then P (2 steps x hi/lo), then Q (2 segments)
constexpr uint32_t kOffP = kKV * 2 * kTile;
constexpr uint32_t kOffQ = kOffP + 2 * 2 * kPBuf;
constexpr uint32_t kSmemTc = kOffQ + 2 * kQBuf + 1024;  // + room to align the base to 1 KiB

__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = (uint64_t)((addr & 0x3FFFF) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version of tcgen05
    d |= (uint64_t)2 << 61;  // 128-byte swizzle
    return d;
}

// kind::f16 instruction descriptor: fp32 accumulator, A and B both bf16 (or both f16),
// A K-major (S) or M-major (O^T), B K-major, N = 16, M = 128.
__host__ __device__ constexpr uint32_t mma_idesc(bool bf16, bool a_mn_major)
{
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((a_mn_major ? 1u : 0u) << 15) | ((uint32_t)(kN >> 3) << 17) | ((128u >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem, uint64_t ad, uint64_t bd, uint32_t idesc,
                                        uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
                 "l"(ad), "l"(bd), "r"(idesc), "r"(accumulate)
                 : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                       uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                       uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// Byte offset of element (row r, column c) of a 128-byte-swizzled K-major operand whose
// 8-row groups are 1024 bytes apart, c < 64 (one 128-byte row).
__device__ __forceinline__ uint32_t sw128_off(uint32_t r, uint32_t c)
{
    return (r >> 3) * 1024 + (r & 7) * 128 + ((((c * 2) >> 4) ^ (r & 7)) << 4) + ((c * 2) & 15);
}

__device__ __forceinline__ void named_sync(int id, int n)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// true in every one of the n threads at named barrier `id` iff v is true in all of them: the
// softmax threads take every decision to stop together, so none is left at a barrier
__device__ __forceinline__ bool named_and(int id, int n, bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
                 "barrier.cta.red.and.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)v), "r"(id), "r"(n)
                 : "memory");
    return r != 0;
}

// The segments of a worker's step range, in the order every role walks them: for each K/V
// head g, the sequences whose steps meet [beg, end).
struct SegWalk {
    const unsigned long long* units_off;
    uint64_t num_seqs, beg, end, s_first;
    uint32_t Hkv;
    uint32_t g = 0;
    uint64_t s = 0, pos = 0;
    bool started = false;
    // next segment: head g, sequence s, steps k0 .. k1 - 1 of it; false at the end
    __device__ bool next(uint32_t& og, uint64_t& os, uint64_t& k0, uint64_t& k1)
    {
        if (!started) {
            started = true;
            g = 0;
            s = s_first;
            pos = beg;
        }
        while (g < Hkv) {
            if (pos < end) {
                while (units_off[s + 1] <= pos) ++s;  // skips sequences without steps
                const uint64_t so = units_off[s];
                k0 = pos - so;
                k1 = umin(units_off[s + 1], end) - so;
                pos = so + k1;
                og = g;
                os = s;
                return true;
            }
            ++g;
            s = s_first;
            pos = beg;
        }
        return false;
    }
};

template <typename IndexT, bool BF16, int G>
__global__ void __launch_bounds__(kThreadsTc, 1)
    attn_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmq)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) unsigned long long k_full[kKV], v_full[kKV], k_free[kKV], v_free[kKV];
    __shared__ __align__(8) unsigned long long s_full[2], s_free[2], p_full[2], o_full[2],
        o_free[2], q_full[2], q_free[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ float red[4][kN];
    __shared__ unsigned merge_done;

    pdl_wait();  // the plan before this launch is complete
    if (a.hdr->verdict != kVerdictOk) return;
    const unsigned warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a sequence without tokens has no step: the grid writes its zeros
    for (uint64_t s = (uint64_t)blockIdx.x * 8 + warp; s < a.num_seqs; s += (uint64_t)gridDim.x * 8)
        if (a.units_off[s] == a.units_off[s + 1]) {
            float4* o = reinterpret_cast<float4*>(a.out + s * a.Hq * a.D);
            for (uint64_t i = lane; i < a.Hq * a.D / 4; i += 32) o[i] = make_float4(0, 0, 0, 0);
        }
    const uint64_t S_steps = a.hdr->total_units;  // steps of all sequences, one head
    const uint64_t Lw = (S_steps + a.workers - 1) / a.workers;
    const uint64_t v = blockIdx.x;  // worker index (one per CTA)
    const uint64_t beg = umin(v * Lw, S_steps), end = umin(beg + Lw, S_steps);
    if (beg >= end) return;  // the whole CTA, before any barrier or TMEM

    // the swizzled operands assume 1024-byte-aligned tiles: align the base explicitly
    const uint32_t sm0 = (smem_u32(smem_raw) + 1023u) & ~1023u;
    unsigned char* smem = smem_raw + (sm0 - smem_u32(smem_raw));
    if (threadIdx.x == 0) {
        for (int i = 0; i < kKV; ++i) {
            mbar_init(smem_u32(&k_full[i]), 1);
            mbar_init(smem_u32(&v_full[i]), 1);
            mbar_init(smem_u32(&k_free[i]), 1);
            mbar_init(smem_u32(&v_free[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s_full[i]), 1);
            mbar_init(smem_u32(&s_free[i]), kSoftmax);
            mbar_init(smem_u32(&p_full[i]), kSoftmax);
            mbar_init(smem_u32(&o_full[i]), 1);
            mbar_init(smem_u32(&o_free[i]), kSoftmax);
            mbar_init(smem_u32(&q_full[i]), 1);
            mbar_init(smem_u32(&q_free[i]), 1);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // the P operands' padding rows (query heads G..15) stay zero for the whole launch
    for (uint32_t i = threadIdx.x; i < 2 * 2 * kPBuf / 16; i += kThreadsTc)
        *reinterpret_cast<uint4*>(smem + kOffP + i * 16) = make_uint4(0, 0, 0, 0);
    for (uint32_t i = threadIdx.x; i < 2 * kQBuf / 16; i += kThreadsTc)
        *reinterpret_cast<uint4*>(smem + kOffQ + i * 16) = make_uint4(0, 0, 0, 0);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = tmem_base;
    const IndexT* table = static_cast<const IndexT*>(a.table);
    const IndexT* spp = static_cast<const IndexT*>(a.seq_ptr);
    const IndexT* lensp = static_cast<const IndexT*>(a.lens);
    const uint32_t P = (uint32_t)a.page_size;
    const uint32_t ppt = kTok / P;  // pages per step
    SegWalk walk{a.units_off, a.num_seqs, beg, end, find_seq(a.units_off, a.num_seqs, beg),
                 a.Hkv};
    auto failed = [&](bool ok) {
        if (!ok) {
            abort_flag = 1;
            report(a.d_status, HP_ERR_TIMEOUT);
        }
        return !ok || *(volatile int*)&abort_flag;
    };

    if (warp == 0 || warp == 7) {
        // ---------------------------------------------------- TMA: K (warp 0), V (warp 7)
        const bool is_k = warp == 0;
        const CUtensorMap* map = is_k ? &tmk : &tmv;
        unsigned long long* full = is_k ? k_full : v_full;
        unsigned long long* freed = is_k ? k_free : v_free;
        const uint32_t base = sm0 + (is_k ? 0u : kKV * kTile);
        uint64_t j = 0, seg = 0;  // steps and segments issued
        uint32_t g;
        uint64_t s, k0, k1;
        bool stop = false;
        while (!stop && walk.next(g, s, k0, k1)) {
            const uint64_t len = lensp[s], tab0 = spp[s];
            if (is_k) {
                // the segment's G query rows, both 64-dim halves, into Q buffer seg % 2 once
                // the S of segment seg - 2 have read it (rows G..15 stay zero)
                int ok = 1;
                if (lane == 0) {
                    ok = seg < 2 || mbar_wait(smem_u32(&q_free[seg % 2]), (uint32_t)((seg / 2 - 1) & 1));
                    if (ok) {
                        const uint32_t qb = sm0 + kOffQ + (uint32_t)(seg % 2) * kQBuf;
                        const int row = (int)(s * a.Hq + (uint64_t)g * G);
                        mbar_expect_tx(smem_u32(&q_full[seg % 2]), 2 * G * 128);
                        tma_2d(qb, &tmq, 0, row, smem_u32(&q_full[seg % 2]));
                        tma_2d(qb + 2048, &tmq, 64, row, smem_u32(&q_full[seg % 2]));
                    }
                }
                if (failed(__shfl_sync(0xffffffffu, ok, 0) != 0)) break;
                ++seg;
            }
            for (uint64_t k = k0; k < k1; ++k, ++j) {
                const uint32_t st = (uint32_t)(j % kKV);
                // lane i < ppt: the step's page i, if any of its slots holds a live token
                // (its ID read before the wait for the stage)
                const uint64_t t0 = k * kTok + (uint64_t)lane * P;
                const bool live = lane < ppt && t0 < len;
                const unsigned long long phys = live ? (unsigned long long)table[tab0 + t0 / P] : 0ull;
                const uint32_t npages = __popc(__ballot_sync(0xffffffffu, live));
                int ok = 1;
                if (lane == 0 && j >= kKV)
                    ok = mbar_wait(smem_u32(&freed[st]), (uint32_t)((j / kKV - 1) & 1));
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (failed(ok != 0)) {
                    stop = true;
                    break;
                }
                if (lane == 0) mbar_expect_tx(smem_u32(&full[st]), npages * P * 256);
                __syncwarp();
                if (live) {
                    const uint32_t dst = base + st * kTile + lane * P * 128;
                    const int row = (int)(phys * P);
                    tma_3d(dst, map, 0, (int)g, row, smem_u32(&full[st]));
                    tma_3d(dst + kHalf, map, 64, (int)g, row, smem_u32(&full[st]));
                }
            }
        }
        // the loads of the last stages land before the CTA's shared memory goes
        if (lane == 0) {
            for (uint64_t x = j > kKV ? j - kKV : 0; x < j; ++x)
                mbar_wait(smem_u32(&full[x % kKV]), (uint32_t)((x / kKV) & 1));
            if (is_k)
                for (uint64_t x = seg > 2 ? seg - 2 : 0; x < seg; ++x)
                    mbar_wait(smem_u32(&q_full[x % 2]), (uint32_t)((x / 2) & 1));
        }
    } else if (warp == 1) {
        // --------------------------------------------------- S = K . Q^T (one thread issues)
        const uint32_t id_s = mma_idesc(BF16, false);
        uint64_t j = 0, seg = 0;
        uint32_t g;
        uint64_t s, k0, k1;
        bool stop = false;
        while (!stop && walk.next(g, s, k0, k1)) {
            for (uint64_t k = k0; k < k1; ++k, ++j) {
                int ok = 1;
                if (lane == 0) {
                    ok = mbar_wait(smem_u32(&k_full[j % kKV]), (uint32_t)((j / kKV) & 1)) &&
                         (k != k0 || mbar_wait(smem_u32(&q_full[seg % 2]), (uint32_t)((seg / 2) & 1))) &&
                         (j < 2 || mbar_wait(smem_u32(&s_free[j % 2]), (uint32_t)((j / 2 - 1) & 1)));
                    if (ok) {
                        fence_after();
                        const uint32_t kst = sm0 + (uint32_t)(j % kKV) * kTile;
                        const uint32_t qb = sm0 + kOffQ + (uint32_t)(seg % 2) * kQBuf;
                        const uint32_t d = tmem + (uint32_t)(j % 2) * kN;
                        for (uint32_t h = 0; h < 2; ++h)
                            for (uint32_t kk = 0; kk < 4; ++kk)
                                mma_f16(d, sw128_desc(kst + h * kHalf + kk * 32, 16, 1024),
                                        sw128_desc(qb + h * 2048 + kk * 32, 16, 1024), id_s,
                                        h | kk);
                        mma_commit(smem_u32(&s_full[j % 2]));
                        mma_commit(smem_u32(&k_free[j % kKV]));  // K of this step is read
                        if (k + 1 == k1) mma_commit(smem_u32(&q_free[seg % 2]));  // and Q
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (failed(ok != 0)) {
                    stop = true;
                    break;
                }
            }
            ++seg;
        }
        // every S issued has completed before the TMEM goes
        if (lane == 0 && j >= 1) mbar_wait(smem_u32(&s_full[(j - 1) % 2]), (uint32_t)(((j - 1) / 2) & 1));
    } else if (warp == 6) {
        // ------------------------------------------- O^T = V^T . P^T (one thread issues)
        const uint32_t id_o = mma_idesc(BF16, true);
        uint64_t j = 0;
        uint32_t g;
        uint64_t s, k0, k1;
        bool stop = false;
        while (!stop && walk.next(g, s, k0, k1)) {
            for (uint64_t k = k0; k < k1; ++k, ++j) {
                int ok = 1;
                if (lane == 0) {
                    ok = mbar_wait(smem_u32(&p_full[j % 2]), (uint32_t)((j / 2) & 1)) &&
                         mbar_wait(smem_u32(&v_full[j % kKV]), (uint32_t)((j / kKV) & 1)) &&
                         (j < 2 || mbar_wait(smem_u32(&o_free[j % 2]), (uint32_t)((j / 2 - 1) & 1)));
                    if (ok) {
                        fence_after();
                        const uint32_t vst = sm0 + kKV * kTile + (uint32_t)(j % kKV) * kTile;
                        const uint32_t pb = sm0 + kOffP + (uint32_t)(j % 2) * 2 * kPBuf;
                        const uint32_t d = tmem + 32 + (uint32_t)(j % 2) * kN;
                        for (uint32_t kk = 0; kk < kTok / 16; ++kk) {
                            const uint64_t ad = sw128_desc(vst + kk * 2048, kHalf, 1024);
                            for (uint32_t part = 0; part < 2; ++part) {  // weights hi, then lo
                                const uint32_t pa = pb + part * kPBuf + (kk >> 2) * 2048 + (kk & 3) * 32;
                                mma_f16(d, ad, sw128_desc(pa, 16, 1024), id_o, kk | part);
                            }
                        }
                        mma_commit(smem_u32(&o_full[j % 2]));
                        mma_commit(smem_u32(&v_free[j % kKV]));  // V of this step is read
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (failed(ok != 0)) {
                    stop = true;
                    break;
                }
            }
        }
        // every O issued has completed before the TMEM goes
        if (lane == 0 && j >= 1) mbar_wait(smem_u32(&o_full[(j - 1) % 2]), (uint32_t)(((j - 1) / 2) & 1));
    } else {
        // ------------------------------------------------------- softmax, accumulation
        const uint32_t t = threadIdx.x - 64;          // 0..127
        const uint32_t q4 = warp & 3;                  // this warp's TMEM lane quarter
        const uint32_t my = q4 * 32 + lane;            // TMEM lane: token (S) or dim (O)
        const uint32_t lane_addr = (q4 * 32) << 16;
        const float qscale = a.scale * 1.4426950408889634f;  // scores in log2 units
        uint64_t j = 0, seg = 0;
        uint32_t g;
        uint64_t s, k0, k1;
        // a wait of every softmax thread, decided together; on a timeout the launch stops
        auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
            const bool ok = named_and(2, kSoftmax, mbar_wait(bar, parity));
            if (!ok && t == 0) {
                abort_flag = 1;
                report(a.d_status, HP_ERR_TIMEOUT);
            }
            return ok;
        };
        bool stop = false;
        float acc[G];
        while (!stop && walk.next(g, s, k0, k1)) {
            const uint64_t len = lensp[s];
            float m[G], m_acc[G];  // running maxima: of the scores, and of acc
#pragma unroll
            for (int h = 0; h < G; ++h) {
                m[h] = -INFINITY;
                m_acc[h] = -INFINITY;
                acc[h] = 0.0f;
            }
            float lp[G];  // this thread's share of each head's weight sum
#pragma unroll
            for (int h = 0; h < G; ++h) lp[h] = 0.0f;
            // folds O of step jj (weights relative to mj) into acc
            auto fold = [&](uint64_t jj, const float (&mj)[G]) -> bool {
                if (!wait_all(smem_u32(&o_full[jj % 2]), (uint32_t)((jj / 2) & 1))) return false;
                fence_after();
                float o[16];
                tmem_ld16(tmem + lane_addr + 32 + (uint32_t)(jj % 2) * kN, o);
                fence_before();
                mbar_arrive(smem_u32(&o_free[jj % 2]));
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float c = exp2_approx(m_acc[h] - mj[h]);  // 0 while acc is empty
                    acc[h] = acc[h] * c + o[h];
                    m_acc[h] = mj[h];
                }
                return true;
            };
            float m_prev[G];
            for (uint64_t k = k0; k < k1; ++k, ++j) {
                if (!wait_all(smem_u32(&s_full[j % 2]), (uint32_t)((j / 2) & 1))) {
                    stop = true;
                    break;
                }
                fence_after();
                float sc[16];
                tmem_ld16(tmem + lane_addr + (uint32_t)(j % 2) * kN, sc);
                fence_before();
                mbar_arrive(smem_u32(&s_free[j % 2]));
                const uint64_t tok = k * kTok + my;
                const bool valid = tok < len;
                float mx[G];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    sc[h] = valid ? sc[h] * qscale : -INFINITY;
                    float x = sc[h];
#pragma unroll
                    for (int o2 = 16; o2 >= 1; o2 >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o2));
                    mx[h] = x;
                }
#pragma unroll
                for (int h = 0; h < G; ++h)
                    if (lane == (unsigned)h) red[q4][h] = mx[h];  // every lane holds the maxima
                named_sync(1, kSoftmax);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    m_prev[h] = m[h];
                    m[h] = fmaxf(m[h], fmaxf(fmaxf(red[0][h], red[1][h]), fmaxf(red[2][h], red[3][h])));
                }
                named_sync(1, kSoftmax);  // red is rewritten next step
                // weights relative to the new maxima, as hi + lo pairs of 16-bit values
                unsigned char* pb = smem + kOffP + (uint32_t)(j % 2) * 2 * kPBuf;
                const uint32_t pcol = my & 63, patom = (my >> 6) * 2048;
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float p = exp2_approx(sc[h] - m[h]);  // 0 past the sequence
                    lp[h] = lp[h] * exp2_approx(m_prev[h] - m[h]) + p;
                    unsigned short hi, lo;
                    if (BF16) {
                        const __nv_bfloat16 bh = __float2bfloat16_rn(p);
                        hi = __bfloat16_as_ushort(bh);
                        lo = __bfloat16_as_ushort(__float2bfloat16_rn(p - __bfloat162float(bh)));
                    } else {
                        const __half hh = __float2half_rn(p);
                        hi = __half_as_ushort(hh);
                        lo = __half_as_ushort(__float2half_rn(p - __half2float(hh)));
                    }
                    const uint32_t off = patom + sw128_off((uint32_t)h, pcol);
                    *reinterpret_cast<unsigned short*>(pb + off) = hi;
                    *reinterpret_cast<unsigned short*>(pb + kPBuf + off) = lo;
                }
                // rows of V past the sequence become zeros (their weights are zero, and a
                // stale or undefined value must not reach the product)
                if ((k + 1) * kTok > len) {  // the same in every softmax thread
                    if (!wait_all(smem_u32(&v_full[j % kKV]), (uint32_t)((j / kKV) & 1))) {
                        stop = true;
                        break;
                    }
                    // rows r0 .. 127 of both halves, 16-byte pieces spread over the threads
                    // (consecutive threads, consecutive pieces of a row)
                    const uint32_t r0 = (uint32_t)(len - k * kTok);
                    unsigned char* vst = smem + (kKV + (uint32_t)(j % kKV)) * kTile;
                    for (uint32_t x = t; x < (kTok - r0) * 16; x += kSoftmax) {
                        const uint32_t row = r0 + (x >> 4), piece = x & 15;
                        *reinterpret_cast<uint4*>(vst + (piece >> 3) * kHalf + row * 128 +
                                                  (piece & 7) * 16) = make_uint4(0, 0, 0, 0);
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive(smem_u32(&p_full[j % 2]));
                // the previous step's O, now that this step's weights are handed over
                if (k > k0 && !fold(j - 1, m_prev)) {
                    stop = true;
                    break;
                }
            }
            if (stop || !fold(j - 1, m)) break;
            // each head's weight sum over the 128 threads
            float l[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float x = lp[h];
#pragma unroll
                for (int o2 = 16; o2 >= 1; o2 >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o2);
                if (lane == 0) red[q4][h] = x;
            }
            named_sync(1, kSoftmax);
#pragma unroll
            for (int h = 0; h < G; ++h) l[h] = red[0][h] + red[1][h] + red[2][h] + red[3][h];
            named_sync(1, kSoftmax);
            const uint64_t so = a.units_off[s], ns = a.units_off[s + 1] - so;
            const uint64_t f = so / Lw, nr = (so + ns - 1) / Lw - f + 1;
            float* out = a.out + (s * a.Hq + (uint64_t)g * G) * kD + my;
            if (nr == 1) {  // the whole sequence: its normalised result
#pragma unroll
                for (int h = 0; h < G; ++h) out[h * kD] = acc[h] / l[h];
            } else {
                const uint64_t row0 = ((s + v) * a.Hkv + g) * G;
#pragma unroll
                for (int h = 0; h < G; ++h) a.part_acc[(row0 + h) * kD + my] = acc[h];
                if (t == 0) {
#pragma unroll
                    for (int h = 0; h < G; ++h)
                        reinterpret_cast<float2*>(a.part_ml)[row0 + h] = make_float2(m[h], l[h]);
                }
                __threadfence();  // the record is visible before the count moves
                named_sync(1, kSoftmax);
                if (t == 0) {
                    const unsigned done = atomicAdd(a.seg_done + s * a.Hkv + g, 1u);
                    merge_done = done + 1 == nr;
                }
                named_sync(1, kSoftmax);
                if (merge_done && t < 32) {  // the last segment: merge them all (one warp)
                    __threadfence();
                    merge_segments<G, kD / 32>(a, ((s + f) * a.Hkv + g) * G, nr,
                                               a.out + (s * a.Hq + (uint64_t)g * G) * kD + lane * (kD / 32),
                                               lane);
                    if (lane == 0) a.seg_done[s * a.Hkv + g] = 0u;
                }
                named_sync(1, kSoftmax);  // merge_done is rewritten by the next segment
            }
            ++seg;
        }
    }
    // every role is done; the TMEM goes back (the MMA warp waited for its operations)
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

// cuTensorMapEncodeTiled through the runtime's driver entry point, looked up once.
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn()
{
    static EncodeFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (EncodeFn) nullptr;
        return reinterpret_cast<EncodeFn>(p);
    }();
    return fn;
}

// A pool [num_pages * P tokens, H_kv, 128] as a 3-d tensor: boxes of 64 dims x 1 head x P
// tokens, 128-byte swizzled.
bool pool_map(CUtensorMap* m, const void* pool, const AttnArgs& a, bool bf16)
{
    EncodeFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {kD, a.Hkv, a.num_pages * a.page_size};
    const cuuint64_t strides[2] = {kD * 2, (cuuint64_t)a.Hkv * kD * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)a.page_size};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
              const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The queries [num_seqs * Hq rows, 128] as a 2-d tensor: boxes of 64 dims x G rows (the
// query heads of one K/V head), 128-byte swizzled.
bool query_map(CUtensorMap* m, const AttnArgs& a, bool bf16)
{
    EncodeFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {kD, a.num_seqs * a.Hq};
    const cuuint64_t strides[1] = {kD * 2};
    const cuuint32_t box[2] = {64, a.G};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
              const_cast<void*>(a.q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename IndexT, bool BF16, int G>
int launch_g(const AttnArgs& a, cudaStream_t st)
{
    CUtensorMap mk, mv, mq;
    if (!pool_map(&mk, a.k_pool, a, BF16) || !pool_map(&mv, a.v_pool, a, BF16) ||
        !query_map(&mq, a, BF16))
        return HP_ERR_CUDA;
    int dev = 0;
    const int sms = current_sms(&dev);
    if (sms == 0 || !allow_dynamic_smem<attn_tc_kernel<IndexT, BF16, G>>(dev, (int)kSmemTc))
        return HP_ERR_CUDA;
    AttnArgs b = a;
    b.workers = (uint64_t)sms;
    return launch_dependent(attn_tc_kernel<IndexT, BF16, G>, (unsigned)sms, kThreadsTc,
                            (size_t)kSmemTc, st, b, mk, mv, mq) == cudaSuccess
               ? HP_OK
               : HP_ERR_CUDA;
}

template <typename IndexT, bool BF16>
int launch_b(const AttnArgs& a, cudaStream_t st)
{
    switch (a.G) {
    case 1: return launch_g<IndexT, BF16, 1>(a, st);
    case 2: return launch_g<IndexT, BF16, 2>(a, st);
    case 4: return launch_g<IndexT, BF16, 4>(a, st);
    case 8: return launch_g<IndexT, BF16, 8>(a, st);
    default: return HP_ERR_ARG;
    }
}

}  // namespace

#ifndef HP_ATTN_TC
#define HP_ATTN_TC 1
#endif

bool attention_tc_fits(uint64_t head_dim, uint64_t page_size, uint64_t num_pages, bool host_memory)
{
    return HP_ATTN_TC && !host_memory && head_dim == kD &&
           (page_size == 8 || page_size == 16 || page_size == 32 || page_size == 64 ||
            page_size == 128) &&
           num_pages * page_size < (1ull << 31);
}


uint64_t attention_tc_step_tokens() { return kTok; }

int launch_attention_tc(int index_u64, const AttnArgs& a, void* stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (index_u64)
        return a.elem_bf16 ? launch_b<unsigned long long, true>(a, st)
                           : launch_b<unsigned long long, false>(a, st);
    return a.elem_bf16 ? launch_b<unsigned int, true>(a, st) : launch_b<unsigned int, false>(a, st);
}

}  // namespace hp
