// hp_attn_tc.cu -- decode attention through the block table on the tensor cores (tcgen05),
// for head_dim 128 (and head_dim 64 taken two K/V heads at a time, see below).
//
// The same computation as hp_attention.cu ("Visualize PagedAttention block layout", How the
// attention kernel uses the block table; K(s,t,g) and V(s,t,g) read through the Element
// Lookup of "Block-Paged Layout -- Hurray Format Specification"): for sequence s and query
// head qh (K/V head g = qh / G), score_t = scale * q . K(s,t,g) over t < len_s, softmax over
// t, out = sum_t weight_t V(s,t,g).  The work is split the same way -- steps balanced over
// workers, one record per segment of a sequence, the records merged by the last segment's
// finisher -- with a step of TS = 128 / H_kv tokens of a sequence and ALL its K/V heads: the
// 128 rows of the step's tiles are (head, token) pairs, h * TS + t.  So a step reads whole
// pages (all heads of its tokens, contiguous in the pool) and a worker's range holds few
// segments.  The two contractions of a step run on the tensor cores (kind::f16, fp32
// accumulators in TMEM):
//   S [128 rows x 32] = K [128 rows x 128 dims] . Q^T     Q: the sequence's Hq <= 32 query
//                                                         heads (padded to 32); row h * TS + t
//                                                         keeps the G columns of head h
//   O_h^T [128 dims x 16] = V_h^T [128 dims x TS] . P_h^T for each K/V head h: its TS rows of
//                                                         V and its weights (G rows, padded)
// One CTA per SM, six roles, each running ahead as far as its buffers allow:
//   warps 0, 7  TMA: per step, the K (warp 0) and V (warp 7) rows of the step's pages, one
//               box per (head, page): 64 dims x 1 head x P tokens, 128-byte swizzled by the
//               tensor map, two per (head, page) for the two 64-dim halves, into rings of 3
//               stages of 32 KiB counted on "k_full"/"v_full"; warp 0 also brings each
//               segment's queries (one box per half); a K stage comes back once S has read
//               it, a V stage once O has;
//   warp 1      tcgen05.mma issue of S (one thread, 8 products of K = 16), committed to
//               "s_full";
//   warp 6      tcgen05.mma issue of the H_kv O products (one thread, 8 slices of 16 rows,
//               twice each: hi and lo weights), committed to "o_full"; both issuers run
//               unrolled code with the descriptors precomputed, because a product of M = 128
//               and N <= 64 keeps the tensor pipe only about 45 cycles (measured on GB300),
//               less than a loop that rebuilds descriptors takes to issue it;
//   warps 2-5   softmax and accumulation, one thread per TMEM lane: a step's scores (lane =
//               row = (head, token)), masked past the sequence, weighed against each query
//               head's reference maximum -- which moves (a shuffle reduction over the head's
//               rows, a factor for the sums and the accumulators) only when some score exceeds
//               it by more than 2^kTau: lazy rescaling --, the weights written as 16-bit pairs
//               hi + lo = p (so P.V keeps about 16 significant bits where one 16-bit P would
//               keep 8), then the previous step's O (lane = dim) folded into fp32 registers,
//               rescaled only after the steps whose references moved.
// Rows of V past the sequence (an unfilled last page, or pages a step does not have) are
// zeroed in shared memory before their weights (zero) are handed over, so no stale or
// undefined value reaches the product.  Every wait is bounded (about 2 s); a wait that runs
// out reports HP_ERR_TIMEOUT, every role leaves its loop (the softmax threads decide it
// together at their one barrier per step, so none is left at a barrier), and the loads and
// matrix operations already issued are waited for (bounded) before the TMEM is freed.
//
// One launch takes up to 8 K/V heads and 32 query heads of 128 dims.  The host runs more as
// groups of K/V heads, one launch each on the same plan: the tensor maps then cover the
// group's slice of each pool row and of each sequence's queries (full-row strides), and the
// output pointer and its sequence stride (TcShape::hq_row) do the same.  Head_dim 64 runs as
// pairs of K/V heads (TcShape::pair): two adjacent 64-dim heads are one 128-dim row, each
// query is zero-padded to 128 dims in its own head's half (qpad_kernel), so its score is its
// 64-dim one, and each query head keeps only its head's 64 dims of the value sums.
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

constexpr int kRows = 128;          // rows of a step's tiles: H_kv heads x TS tokens
constexpr int kD = 128;             // head_dim
constexpr int kNS = 32;             // S columns: the query heads, padded
constexpr int kNO = 16;             // O columns of one K/V head: its G query heads, padded
constexpr int kMaxHkv = 8;
constexpr int kKV = 3;              // K/V stages
constexpr uint32_t kHalf = kRows * 128;      // one 64-dim half of a K or V tile (16 KiB)
constexpr uint32_t kTile = 2 * kHalf;        // one K or V tile (32 KiB)
constexpr uint32_t kPBuf = 2 * kNO * 128;    // one P operand: 16 rows x 128 (head, token) cols
constexpr uint32_t kQBuf = 2 * kNS * 128;    // one Q operand: 32 rows x 128 dims (8 KiB)
constexpr int kThreadsTc = 8 * 32;
constexpr int kSoftmax = 128;       // warps 2-5
constexpr uint32_t kTmemCols = 512; // S x 2 (64 columns), O x 2 (up to 2 x 8 x 16)
constexpr uint32_t kOCol = 2 * kNS; // first O column
constexpr float kTau = 8.0f;        // log2 units a score may exceed its head's reference by

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
// A K-major (S) or M-major (O^T), B K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t mma_idesc(bool bf16, bool a_mn_major, uint32_t n)
{
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((a_mn_major ? 1u : 0u) << 15) | ((n >> 3) << 17) | ((128u >> 4) << 24);
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

// tcgen05.ld of N consecutive TMEM columns of this thread's lane (32x32b shape) into r,
// not yet waited for; the column is a multiple of N
template <int N> __device__ __forceinline__ void tmem_issue(uint32_t taddr, uint32_t* r);

template <> __device__ __forceinline__ void tmem_issue<1>(uint32_t taddr, uint32_t* r)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];"
                 : "=r"(r[0])
                 : "r"(taddr));
}

template <> __device__ __forceinline__ void tmem_issue<2>(uint32_t taddr, uint32_t* r)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1])
                 : "r"(taddr));
}

template <> __device__ __forceinline__ void tmem_issue<4>(uint32_t taddr, uint32_t* r)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
}

template <> __device__ __forceinline__ void tmem_issue<8>(uint32_t taddr, uint32_t* r)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

template <> __device__ __forceinline__ void tmem_issue<16>(uint32_t taddr, uint32_t* r)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
}

// waits for this thread's TMEM loads; the registers they fill are operands of the wait, so
// no use of them is scheduled above it
template <int N> __device__ __forceinline__ void tmem_wait(uint32_t (&r)[N]);

template <> __device__ __forceinline__ void tmem_wait<1>(uint32_t (&r)[1])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0])::"memory");
}

template <> __device__ __forceinline__ void tmem_wait<2>(uint32_t (&r)[2])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1])::"memory");
}

template <> __device__ __forceinline__ void tmem_wait<4>(uint32_t (&r)[4])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3])::"memory");
}

template <> __device__ __forceinline__ void tmem_wait<8>(uint32_t (&r)[8])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7])::"memory");
}

template <> __device__ __forceinline__ void tmem_wait<16>(uint32_t (&r)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])::"memory");
}

template <> __device__ __forceinline__ void tmem_wait<32>(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])::"memory");
}

// N consecutive TMEM columns of this thread's lane, waited for
template <int N> __device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&v)[N])
{
    uint32_t r[N];
    tmem_issue<N>(taddr, r);
    tmem_wait<N>(r);
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = __uint_as_float(r[i]);
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

// true in every one of the n threads at named barrier `id` iff v is true in all (and) / in
// any (or) of them; the softmax threads take every decision to stop together, so none is
// left at a barrier
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
__device__ __forceinline__ bool named_or(int id, int n, bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
                 "barrier.cta.red.or.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)v), "r"(id), "r"(n)
                 : "memory");
    return r != 0;
}

// The segments of a worker's step range, in the order every role walks them: the sequences
// whose steps meet [beg, end).
struct SegWalk {
    const unsigned long long* units_off;
    uint64_t beg, end, s;
    uint64_t pos = ~0ull;
    // next segment: sequence s, steps k0 .. k1 - 1 of it; false at the end
    __device__ bool next(uint64_t& os, uint64_t& k0, uint64_t& k1)
    {
        if (pos == ~0ull) pos = beg;
        if (pos >= end) return false;
        while (units_off[s + 1] <= pos) ++s;  // skips sequences without steps
        const uint64_t so = units_off[s];
        k0 = pos - so;
        k1 = umin(units_off[s + 1], end) - so;
        pos = so + k1;
        os = s;
        return true;
    }
};

__device__ __forceinline__ unsigned long long table_at(const void* table, bool u64, uint64_t i)
{
    return u64 ? (unsigned long long)static_cast<const unsigned long long*>(table)[i]
               : (unsigned long long)static_cast<const unsigned int*>(table)[i];
}

// Run-time shape of a launch, beside AttnArgs.
struct TcShape {
    uint32_t hkv;   // K/V heads: 1, 2, 4 or 8
    uint32_t ts;    // tokens per step: 128 / hkv
    uint32_t lts;   // log2(ts)
    uint32_t pps;   // pages per step: ts / page_size
    uint32_t idx64; // index type: uint64 (1) or uint32 (0)
    uint32_t bf16;  // element type: bf16 (1) or f16 (0)
    uint32_t stall; // HP_TEST_STALL: the K loader arms its first step but never issues it
    uint32_t pair;  // head_dim 64 as pairs of K/V heads: 64 output dims per query head
    uint32_t hq_row;  // query heads per sequence in out (this launch's group: a.Hq of them)
};

template <int G>
__global__ void __launch_bounds__(kThreadsTc, 1)
    attn_tc_kernel(const AttnArgs a, const TcShape sh, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmq)
{
    constexpr int kHeads = (kMaxHkv * G < kNS ? kMaxHkv * G : kNS) / G;  // K/V heads at most
    constexpr int kAcc = kHeads * G;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) unsigned long long k_full[kKV], v_full[kKV], k_free[kKV], v_free[kKV];
    __shared__ __align__(8) unsigned long long s_full[2], s_free[2], p_full[2], o_full[2],
        o_free[2], q_full[2], q_free[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ float corr_s[2][kNS];  // per step parity: each query head's rescale factor
    __shared__ float red_s[4][8];     // per-warp maxima or sums when a head's rows span warps
    __shared__ float ml_s[2][kNS];    // a segment's maxima and weight sums per query head
    __shared__ float inv_s[kNS];      // and the reciprocals of those sums
    __shared__ unsigned merge_done;
    __shared__ int fail_s[2];         // softmax waits that ran out, by step parity

    pdl_wait();  // the plan before this launch is complete
    if (a.hdr->verdict != kVerdictOk) return;
    const unsigned warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t outD = sh.pair ? 64 : kD;  // output dims per query head
    // a sequence without tokens has no step: the grid writes its zeros
    for (uint64_t s = (uint64_t)blockIdx.x * 8 + warp; s < a.num_seqs; s += (uint64_t)gridDim.x * 8)
        if (a.units_off[s] == a.units_off[s + 1]) {
            float4* o = reinterpret_cast<float4*>(a.out + s * sh.hq_row * outD);
            for (uint64_t i = lane; i < a.Hq * outD / 4; i += 32) o[i] = make_float4(0, 0, 0, 0);
        }
    const uint64_t S_steps = a.hdr->total_units;  // steps of all sequences (all heads each)
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
        fail_s[0] = fail_s[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // padding rows stay zero for the whole launch: P rows G..15, Q rows Hq..31
    for (uint32_t i = threadIdx.x; i < (2 * 2 * kPBuf + 2 * kQBuf) / 16; i += kThreadsTc)
        *reinterpret_cast<uint4*>(smem + kOffP + i * 16) = make_uint4(0, 0, 0, 0);
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
    const uint32_t P = (uint32_t)a.page_size, TS = sh.ts, HKV = sh.hkv, PPS = sh.pps;
    const bool u64 = sh.idx64 != 0, bf16 = sh.bf16 != 0;
    SegWalk walk{a.units_off, beg, end, find_seq(a.units_off, a.num_seqs, beg)};
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
        const uint32_t lh = lane / PPS, li = lane % PPS;  // this lane's (head, page of the step)
        const bool active = lane < HKV * PPS;
        uint64_t j = 0, seg = 0;  // steps and segments issued
        uint64_t s, k0, k1;
        bool stop = false;
        while (!stop && walk.next(s, k0, k1)) {
            const uint64_t len = table_at(a.lens, u64, s), tab0 = table_at(a.seq_ptr, u64, s);
            if (is_k) {
                // the sequence's query heads, both 64-dim halves, into Q buffer seg % 2 once
                // the S of segment seg - 2 have read it (rows Hq..31 stay zero)
                int ok = 1;
                if (lane == 0) {
                    ok = seg < 2 || mbar_wait(smem_u32(&q_free[seg % 2]), (uint32_t)((seg / 2 - 1) & 1));
                    if (ok) {
                        const uint32_t qb = sm0 + kOffQ + (uint32_t)(seg % 2) * kQBuf;
                        mbar_expect_tx(smem_u32(&q_full[seg % 2]), 2 * a.Hq * 128);
                        tma_3d(qb, &tmq, 0, 0, (int)s, smem_u32(&q_full[seg % 2]));
                        tma_3d(qb + kNS * 128, &tmq, 64, 0, (int)s, smem_u32(&q_full[seg % 2]));
                    }
                }
                if (failed(__shfl_sync(0xffffffffu, ok, 0) != 0)) break;
                ++seg;
            }
            for (uint64_t k = k0; k < k1; ++k, ++j) {
                const uint32_t st = (uint32_t)(j % kKV);
                // the lane's page (its ID read before the wait for the stage), if any of its
                // slots holds a live token
                const uint64_t t0 = k * TS + (uint64_t)li * P;
                const bool live = active && t0 < len;
                const unsigned long long phys = live ? table_at(a.table, u64, tab0 + k * PPS + li) : 0ull;
                const uint32_t nlive = __popc(__ballot_sync(0xffffffffu, live));
                int ok = 1;
                if (lane == 0 && j >= kKV)
                    ok = mbar_wait(smem_u32(&freed[st]), (uint32_t)((j / kKV - 1) & 1));
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (failed(ok != 0)) {
                    stop = true;
                    break;
                }
                if (lane == 0) mbar_expect_tx(smem_u32(&full[st]), nlive * P * 256);
                __syncwarp();
                if (live && !(is_k && sh.stall && j == 0)) {
                    const uint32_t dst = base + st * kTile + (lh * TS + li * P) * 128;
                    const int row = (int)(phys * P);
                    tma_3d(dst, map, 0, (int)lh, row, smem_u32(&full[st]));
                    tma_3d(dst + kHalf, map, 64, (int)lh, row, smem_u32(&full[st]));
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
        const uint32_t id_s = mma_idesc(bf16, false, kNS);
        // descriptors of K stage 0 and Q buffer 0; the others differ only in the start
        // address field (addresses >> 4, below 2^14 for all of shared memory)
        const uint64_t kd0 = sw128_desc(sm0, 16, 1024), qd0 = sw128_desc(sm0 + kOffQ, 16, 1024);
        uint64_t j = 0, seg = 0;
        uint64_t s, k0, k1;
        bool stop = false;
        while (!stop && walk.next(s, k0, k1)) {
            for (uint64_t k = k0; k < k1; ++k, ++j) {
                int ok = 1;
                if (lane == 0) {
                    ok = mbar_wait(smem_u32(&k_full[j % kKV]), (uint32_t)((j / kKV) & 1)) &&
                         (k != k0 || mbar_wait(smem_u32(&q_full[seg % 2]), (uint32_t)((seg / 2) & 1))) &&
                         (j < 2 || mbar_wait(smem_u32(&s_free[j % 2]), (uint32_t)((j / 2 - 1) & 1)));
                    if (ok) {
                        fence_after();
                        const uint64_t kd = kd0 + (((uint32_t)(j % kKV) * kTile) >> 4);
                        const uint64_t qd = qd0 + (((uint32_t)(seg % 2) * kQBuf) >> 4);
                        const uint32_t d = tmem + (uint32_t)(j % 2) * kNS;
                        // 8 products of 16 dims: 64-dim half h, 32-byte slice kk of its rows
#pragma unroll
                        for (uint32_t u = 0; u < 8; ++u) {
                            const uint32_t h = u >> 2, kk = u & 3;
                            mma_f16(d, kd + ((h * kHalf + kk * 32) >> 4),
                                    qd + ((h * kNS * 128 + kk * 32) >> 4), id_s, u);
                        }
                        mma_commit(smem_u32(&s_full[j % 2]));
                        mma_commit(smem_u32(&k_free[j % kKV]));  // K of this step is read
                        if (k + 1 == k1) mma_commit(smem_u32(&q_free[seg % 2]));  // and Q
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (failed(ok != 0)) {
                    j += ok != 0;  // issued before another role stopped: waited for below
                    stop = true;
                    break;
                }
            }
            ++seg;
        }
        // every S issued has completed before the TMEM goes
        if (lane == 0 && j >= 1) mbar_wait(smem_u32(&s_full[(j - 1) % 2]), (uint32_t)(((j - 1) / 2) & 1));
    } else if (warp == 6) {
        // ------------------------------ O_h^T = V_h^T . P_h^T for every head (one thread issues)
        const uint32_t id_o = mma_idesc(bf16, true, kNO);
        // descriptors of V stage 0 and P buffer 0 (as for S: only the start address moves)
        const uint64_t vd0 = sw128_desc(sm0 + kKV * kTile, kHalf, 1024);
        const uint64_t pd0 = sw128_desc(sm0 + kOffP, 16, 1024);
        uint64_t j = 0;
        uint64_t s, k0, k1;
        bool stop = false;
        while (!stop && walk.next(s, k0, k1)) {
            for (uint64_t k = k0; k < k1; ++k, ++j) {
                int ok = 1;
                if (lane == 0) {
                    ok = mbar_wait(smem_u32(&p_full[j % 2]), (uint32_t)((j / 2) & 1)) &&
                         mbar_wait(smem_u32(&v_full[j % kKV]), (uint32_t)((j / kKV) & 1)) &&
                         (j < 2 || mbar_wait(smem_u32(&o_free[j % 2]), (uint32_t)((j / 2 - 1) & 1)));
                    if (ok) {
                        fence_after();
                        const uint64_t vd = vd0 + (((uint32_t)(j % kKV) * kTile) >> 4);
                        const uint64_t pd = pd0 + (((uint32_t)(j % 2) * 2 * kPBuf) >> 4);
                        const uint32_t ob = tmem + kOCol + (uint32_t)(j % 2) * HKV * kNO;
                        // 8 slices of 16 rows (V rows, P columns), each in its head's O: the
                        // weights' hi part, then their lo part
#pragma unroll
                        for (uint32_t u = 0; u < 8; ++u) {
                            const uint32_t row = u * 16, h = row >> sh.lts;
                            const uint64_t ad = vd + ((row * 128) >> 4);
                            const uint64_t bd = pd + (((row >> 6) * 2048 + (row & 63) * 2) >> 4);
                            mma_f16(ob + h * kNO, ad, bd, id_o, (row & (TS - 1)) != 0);
                            mma_f16(ob + h * kNO, ad, bd + (kPBuf >> 4), id_o, 1u);
                        }
                        mma_commit(smem_u32(&o_full[j % 2]));
                        mma_commit(smem_u32(&v_free[j % kKV]));  // V of this step is read
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (failed(ok != 0)) {
                    j += ok != 0;  // issued before another role stopped: waited for below
                    stop = true;
                    break;
                }
            }
        }
        // every O issued has completed before the TMEM goes
        if (lane == 0 && j >= 1) mbar_wait(smem_u32(&o_full[(j - 1) % 2]), (uint32_t)(((j - 1) / 2) & 1));
    } else {
        // ------------------------------------------------------- softmax, accumulation
        const uint32_t t = threadIdx.x - 64;        // 0..127
        const uint32_t q4 = warp & 3;                // this warp's TMEM lane quarter
        const uint32_t my = q4 * 32 + lane;          // TMEM lane: row (S, P) or dim (O)
        const uint32_t rh = my >> sh.lts, rt = my & (TS - 1);  // the row's head and token
        const uint32_t lane_addr = (q4 * 32) << 16;
        const uint32_t span = TS < 32 ? TS : 32;     // lanes of a warp holding one head's rows
        const uint32_t hw = TS > 32 ? TS / 32 : 1;   // warps holding one head's rows
        const float qscale = a.scale * 1.4426950408889634f;  // scores in log2 units
        // The softmax threads wait each on its own, and stop together: a wait that runs out
        // marks fail_s[w % 2] for the window w it falls in -- window w runs from the step
        // barrier of step w - 1 to that of step w -- and after the step barrier of step w
        // every thread reads the same mark (nothing writes it until the next window).  A
        // thread whose wait ran out carries on to that barrier with values it discards.
        bool ok_w = true;  // this thread's waits since the last step barrier
        auto wait_one = [&](uint32_t bar, uint32_t parity, uint64_t w) {
            if (!mbar_wait(bar, parity)) {
                fail_s[w % 2] = 1;
                abort_flag = 1;
                report(a.d_status, HP_ERR_TIMEOUT);
                ok_w = false;
            }
        };
        // x[g] over the rows of this thread's head: the warp's lanes of the head by shuffles,
        // then (rows spanning warps) the head's warps through red_s
        auto head_reduce = [&](float (&x)[G], bool is_max) {
#pragma unroll
            for (int g = 0; g < G; ++g)
                for (uint32_t o2 = 1; o2 < span; o2 <<= 1) {
                    const float y = __shfl_xor_sync(0xffffffffu, x[g], o2);
                    x[g] = is_max ? fmaxf(x[g], y) : x[g] + y;
                }
            if (hw > 1) {
                if (lane == 0)
#pragma unroll
                    for (int g = 0; g < G; ++g) red_s[q4][g] = x[g];
                named_sync(1, kSoftmax);
                const uint32_t w0 = (rh * TS) >> 5;  // first TMEM quarter of the head
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float r = red_s[w0][g];
                    for (uint32_t w2 = 1; w2 < hw; ++w2)
                        r = is_max ? fmaxf(r, red_s[w0 + w2][g]) : r + red_s[w0 + w2][g];
                    x[g] = r;
                }
                named_sync(1, kSoftmax);  // red_s is rewritten next time
            }
        };
        float acc[kAcc];
        // folds O of step jj into acc, each query head rescaled by its factor of step jj
        // (every factor is 1 when no maximum rose in that step)
        auto fold = [&](uint64_t jj, bool rescale, uint64_t w) {
            wait_one(smem_u32(&o_full[jj % 2]), (uint32_t)((jj / 2) & 1), w);
            fence_after();
            const uint32_t ob = tmem + lane_addr + kOCol + (uint32_t)(jj % 2) * HKV * kNO;
            uint32_t o[kAcc];  // every head's G columns, loaded together, one wait
#pragma unroll
            for (int i = 0; i < kAcc; ++i) o[i] = 0u;
#pragma unroll
            for (int hh = 0; hh < kHeads; ++hh)
                if ((uint32_t)hh < HKV) tmem_issue<G>(ob + hh * kNO, o + hh * G);
            tmem_wait<kAcc>(o);
#pragma unroll
            for (int i = 0; i < kAcc; ++i) {
                const float c = rescale ? corr_s[jj % 2][i] : 1.0f;  // (i < Hq when it counts)
                acc[i] = acc[i] * c + __uint_as_float(o[i]);
            }
            fence_before();
            mbar_arrive(smem_u32(&o_free[jj % 2]));
        };
        uint64_t j = 0;
        uint64_t s, k0, k1;
        bool stop = false;
        while (!stop && walk.next(s, k0, k1)) {
            const uint64_t len = table_at(a.lens, u64, s);
            float m_run[G], lp[G];  // this row's head: running maxima, this row's weight sums
#pragma unroll
            for (int g = 0; g < G; ++g) {
                m_run[g] = -INFINITY;
                lp[g] = 0.0f;
            }
#pragma unroll
            for (int i = 0; i < kAcc; ++i) acc[i] = 0.0f;
            bool up_prev = false;
            for (uint64_t k = k0; k < k1; ++k, ++j) {
                wait_one(smem_u32(&s_full[j % 2]), (uint32_t)((j / 2) & 1), j);
                fence_after();
                // the G score columns of this row's head: a warp holds the rows of one head,
                // or (16-token steps) of two, whose 2G columns it loads together
                float x[G], mx[G];
                const uint32_t sbase = tmem + lane_addr + (uint32_t)(j % 2) * kNS;
                if (TS == 16) {
                    float sc[2 * G];
                    tmem_ld<2 * G>(sbase + q4 * 2 * G, sc);
#pragma unroll
                    for (int g = 0; g < G; ++g) x[g] = lane < 16 ? sc[g] : sc[G + g];
                } else {
                    tmem_ld<G>(sbase + rh * G, x);
                }
                fence_before();
                mbar_arrive(smem_u32(&s_free[j % 2]));
                const bool valid = k * TS + rt < len;
                // Lazy rescaling: each query head's weights are exp2(x - m_ref) against a
                // reference m_ref that moves only when some score exceeds it by more than
                // kTau (weights stay below 2^kTau, well inside the fp32 sums and the two
                // 16-bit parts) -- on a head's first step, and rarely after.  The step
                // barrier is the vote; only when it passes are the heads' maxima reduced and
                // the factors that rescale the sums and (at the next fold) the accumulators
                // formed.
                bool need = false;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    x[g] = valid ? x[g] * qscale : -INFINITY;
                    need |= x[g] > m_run[g] + kTau;  // (m_run -inf: any valid score)
                }
                // the step barrier: whether any reference must move, and whether any wait
                // of this window ran out
                need = named_or(3, kSoftmax, need);
                ok_w = true;
                if (*(volatile int*)&fail_s[j % 2]) {
                    stop = true;
                    break;
                }
                if (need) {  // the same in every softmax thread
#pragma unroll
                    for (int g = 0; g < G; ++g) mx[g] = x[g];
                    head_reduce(mx, true);  // the step's maximum of each query head of rh
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float mn = fmaxf(m_run[g], mx[g]);
                        const float c = exp2_approx(m_run[g] - mn);  // 0 while nothing is summed
                        lp[g] *= c;
                        if (rt == 0) corr_s[j % 2][rh * G + g] = c;
                        m_run[g] = mn;
                    }
                }
                unsigned char* pb = smem + kOffP + (uint32_t)(j % 2) * 2 * kPBuf;
                const uint32_t pcol = my & 63, patom = (my >> 6) * 2048;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float p = exp2_approx(x[g] - m_run[g]);  // 0 past the sequence
                    lp[g] += p;
                    unsigned short hi, lo;
                    if (bf16) {
                        const __nv_bfloat16 bh = __float2bfloat16_rn(p);
                        hi = __bfloat16_as_ushort(bh);
                        lo = __bfloat16_as_ushort(__float2bfloat16_rn(p - __bfloat162float(bh)));
                    } else {
                        const __half hh = __float2half_rn(p);
                        hi = __half_as_ushort(hh);
                        lo = __half_as_ushort(__float2half_rn(p - __half2float(hh)));
                    }
                    const uint32_t off = patom + sw128_off((uint32_t)g, pcol);
                    *reinterpret_cast<unsigned short*>(pb + off) = hi;
                    *reinterpret_cast<unsigned short*>(pb + kPBuf + off) = lo;
                }
                // rows of V past the sequence become zeros (their weights are zero, and a
                // stale or undefined value must not reach the product)
                if ((k + 1) * TS > len) {  // the same in every softmax thread
                    wait_one(smem_u32(&v_full[j % kKV]), (uint32_t)((j / kKV) & 1), j + 1);
                    if (!valid) {
                        unsigned char* vrow = smem + (kKV + (uint32_t)(j % kKV)) * kTile + my * 128;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            *reinterpret_cast<uint4*>(vrow + i * 16) = make_uint4(0, 0, 0, 0);
                            *reinterpret_cast<uint4*>(vrow + kHalf + i * 16) = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive(smem_u32(&p_full[j % 2]));
                // the previous step's O, now that this step's weights are handed over (the
                // factors of step j - 1 were written before this step's barrier)
                if (k > k0) fold(j - 1, up_prev, j + 1);
                up_prev = need;
            }
            if (stop) break;
            fold(j - 1, up_prev, j);
            if (!named_and(2, kSoftmax, ok_w)) break;  // the segment's last waits
            // each query head's weight sum over its rows, and its maximum, per head leader
            head_reduce(lp, false);
            if (rt == 0)
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    ml_s[0][rh * G + g] = m_run[g];
                    ml_s[1][rh * G + g] = lp[g];
                    inv_s[rh * G + g] = 1.0f / lp[g];  // one division per query head
                }
            named_sync(1, kSoftmax);
            const uint64_t so = a.units_off[s], ns = a.units_off[s + 1] - so;
            const uint64_t f = so / Lw, nr = (so + ns - 1) / Lw - f + 1;
            if (nr == 1) {  // the whole sequence: its normalised result, thread = dim
                if (sh.pair) {  // query head i keeps the 64 dims of its own K/V head
                    float* out = a.out + s * sh.hq_row * 64 + (my & 63);
#pragma unroll
                    for (int i = 0; i < kAcc; ++i)
                        if ((uint32_t)i < a.Hq && (my >> 6) == (uint32_t)((2 * (i % G)) / G))
                            out[(uint64_t)i * 64] = acc[i] * inv_s[i];
                } else {
                    float* out = a.out + s * sh.hq_row * kD + my;
#pragma unroll
                    for (int i = 0; i < kAcc; ++i)
                        if ((uint32_t)i < a.Hq) out[(uint64_t)i * kD] = acc[i] * inv_s[i];
                }
            } else {
                const uint64_t row0 = (s + v) * a.Hq;  // record rows of all query heads
#pragma unroll
                for (int i = 0; i < kAcc; ++i)
                    if ((uint32_t)i < a.Hq) a.part_acc[(row0 + i) * kD + my] = acc[i];
                if (t < a.Hq)
                    reinterpret_cast<float2*>(a.part_ml)[row0 + t] = make_float2(ml_s[0][t], ml_s[1][t]);
                __threadfence();  // the record is visible before the count moves
                named_sync(1, kSoftmax);
                if (t == 0) {
                    const unsigned done = atomicAdd(a.seg_done + s * a.Hkv, 1u);
                    merge_done = done + 1 == nr;
                }
                named_sync(1, kSoftmax);
                if (merge_done) {  // the last segment: merge every head's records, a warp each
                    __threadfence();
                    for (uint32_t hh = t >> 5; hh < HKV; hh += 4) {
                        const uint64_t r0 = ((s + f) * a.Hkv + hh) * G;
                        if (sh.pair)
                            merge_segments<G, kD / 32, true>(
                                a, r0, nr, a.out + (s * sh.hq_row + (uint64_t)hh * G) * 64, lane);
                        else
                            merge_segments<G, kD / 32>(
                                a, r0, nr,
                                a.out + (s * sh.hq_row + (uint64_t)hh * G) * kD + lane * (kD / 32),
                                lane);
                    }
                    if (t == 0) a.seg_done[s * a.Hkv] = 0u;
                }
            }
            named_sync(1, kSoftmax);  // ml_s and merge_done are rewritten by the next segment
        }
    }
    // every role is done; the TMEM goes back (the issuers waited for their operations)
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

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

// A pool [num_pages * P tokens, H_kv, 128] as a 3-d tensor (this launch's H_kv heads of the
// Hkv_row in each token's row): boxes of 64 dims x 1 head x P tokens, 128-byte swizzled.
bool pool_map(CUtensorMap* m, const void* pool, const AttnArgs& a, bool bf16)
{
    EncodeFn fn = encode_fn();
    if (!fn) return false;
    const uint64_t row = a.Hkv_row ? a.Hkv_row : a.Hkv;
    const cuuint64_t dims[3] = {kD, a.Hkv, a.num_pages * a.page_size};
    const cuuint64_t strides[2] = {kD * 2, (cuuint64_t)row * kD * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)a.page_size};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
              const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The queries [num_seqs, Hq, 128] as a 3-d tensor (this launch's Hq query heads of the
// Hq_row of each sequence): boxes of 64 dims x Hq heads x 1 sequence, 128-byte swizzled.
bool query_map(CUtensorMap* m, const AttnArgs& a, bool bf16)
{
    EncodeFn fn = encode_fn();
    if (!fn) return false;
    const uint64_t row = a.Hq_row ? a.Hq_row : a.Hq;
    const cuuint64_t dims[3] = {kD, a.Hq, a.num_seqs};
    const cuuint64_t strides[2] = {kD * 2, (cuuint64_t)row * kD * 2};
    const cuuint32_t box[3] = {64, a.Hq, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
              const_cast<void*>(a.q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


template <int G>
int launch_g(const AttnArgs& a, const TcShape& sh, cudaStream_t st)
{
    CUtensorMap mk, mv, mq;
    const bool bf16 = sh.bf16 != 0;
    if (!pool_map(&mk, a.k_pool, a, bf16) || !pool_map(&mv, a.v_pool, a, bf16) ||
        !query_map(&mq, a, bf16))
        return HP_ERR_CUDA;
    int dev = 0;
    const int sms = current_sms(&dev);
    if (sms == 0 || !allow_dynamic_smem<attn_tc_kernel<G>>(dev, (int)kSmemTc)) return HP_ERR_CUDA;
    AttnArgs b = a;
    b.workers = (uint64_t)sms;
    return launch_dependent(attn_tc_kernel<G>, (unsigned)sms, kThreadsTc, (size_t)kSmemTc, st, b,
                            sh, mk, mv, mq) == cudaSuccess
               ? HP_OK
               : HP_ERR_CUDA;
}

uint32_t log2_exact(uint32_t x)
{
    uint32_t l = 0;
    while ((1u << l) < x) ++l;
    return l;
}

}  // namespace

#ifndef HP_ATTN_TC
#define HP_ATTN_TC 1
#endif

bool attention_tc_fits(uint64_t head_dim, uint64_t page_size, uint64_t num_pages, bool host_memory,
                       uint64_t num_kv_heads, uint64_t num_q_heads)
{
    const uint64_t hkv = num_kv_heads;
    if (!HP_ATTN_TC || host_memory || head_dim != kD) return false;
    if (hkv != 1 && hkv != 2 && hkv != 4 && hkv != 8) return false;
    if (num_q_heads > (uint64_t)kNS || num_q_heads % hkv != 0) return false;
    const uint64_t g = num_q_heads / hkv;
    if (g != 1 && g != 2 && g != 4 && g != 8) return false;
    // a step's pages tile its TS = 128 / H_kv tokens exactly
    const uint64_t ts = kRows / hkv;
    return page_size >= 8 && page_size <= ts && (page_size & (page_size - 1)) == 0 &&
           num_pages * page_size < (1ull << 31);
}

uint64_t attention_tc_step_tokens(uint64_t num_kv_heads) { return kRows / num_kv_heads; }

namespace {

// One 16-byte vector (8 elements) of the padded queries per thread, grid-stride.
__global__ void qpad_kernel(const uint4* __restrict__ q, uint4* __restrict__ qpad, uint64_t nvec,
                            uint32_t Hq, uint32_t G)
{
    for (uint64_t v = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec;
         v += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t row = v >> 4;          // (sequence, query head): 16 vectors of 128 dims
        const uint32_t part = (uint32_t)(v & 15), qh = (uint32_t)(row % Hq);
        const uint32_t half = (qh / G) & 1u;  // the K/V head's place in its pair
        qpad[v] = (part >> 3) == half ? q[row * 8 + (part & 7)] : make_uint4(0, 0, 0, 0);
    }
}

}  // namespace

int launch_attention_qpad(const void* q, void* qpad, uint64_t num_seqs, uint32_t Hq, uint32_t G,
                          void* stream)
{
    const uint64_t nvec = num_seqs * Hq * 16;
    if (nvec == 0) return HP_OK;
    int dev = 0;
    const int sms = current_sms(&dev);
    if (sms == 0) return HP_ERR_CUDA;
    const uint64_t grid = std::min<uint64_t>((nvec + 255) / 256, (uint64_t)sms * 8);
    qpad_kernel<<<(unsigned)grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(q), static_cast<uint4*>(qpad), nvec, Hq, G);
    return cudaGetLastError() == cudaSuccess ? HP_OK : HP_ERR_CUDA;
}

int launch_attention_tc(int index_u64, const AttnArgs& a, void* stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    TcShape sh;
    sh.hkv = a.Hkv;
    sh.ts = kRows / a.Hkv;
    sh.lts = log2_exact(sh.ts);
    sh.pps = sh.ts / (uint32_t)a.page_size;
    sh.idx64 = index_u64 != 0;
    sh.bf16 = a.elem_bf16 != 0;
    sh.stall = a.test_stall != 0;
    sh.pair = a.pair != 0;
    sh.hq_row = a.Hq_row ? a.Hq_row : a.Hq;
    switch (a.G) {
    case 1: return launch_g<1>(a, sh, st);
    case 2: return launch_g<2>(a, sh, st);
    case 4: return launch_g<4>(a, sh, st);
    case 8: return launch_g<8>(a, sh, st);
    default: return HP_ERR_ARG;
    }
}

}  // namespace hp
