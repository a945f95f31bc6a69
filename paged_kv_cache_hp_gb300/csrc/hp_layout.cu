// hp_layout.cu -- layout conversions at the boundary of the block-paged format.
//
// "Block-Paged Layout -- Hurray Format Specification", Framework Compliance: the portable
// layout is [num_blocks, block_size, num_kv_heads, head_dim]; a producer that stores its
// cache in a kernel-internal layout such as [num_blocks, num_kv_heads, head_dim/x,
// block_size, x] must transpose before emitting a descriptor.  (x = 1 is the
// [num_blocks, num_kv_heads, head_dim, block_size] value-cache form.)
//
// Unit of work: one (block, head).  In the internal layout a unit is one contiguous run
// of block_size*head_dim elements ([head_dim/x, block_size, x]); in the interchange layout
// it is block_size rows of head_dim elements, one per slot, num_kv_heads*head_dim apart.
// A CTA stages whole units (up to 32 KiB of them at a time) in shared memory, so both the
// global reads and the global writes are contiguous vector accesses; only the
// shared-memory side is permuted.  When an x-chunk is one 16-byte vector and block_size
// is a multiple of 8, chunk (dx, t) of a unit sits at position dx*bs + (t ^ (dx & 7)):
// eight lanes reading one slot's row (dx = 0..7, same t) and eight lanes reading
// consecutive slots of one chunk row (same dx) then both touch eight different 16-byte
// bank groups, where the plain order puts the first eight on one.
#include <cuda_runtime.h>

#include <algorithm>

#include "hp_internal.cuh"

namespace hp {
namespace {

constexpr int kThreads = 256;

template <int VEC> struct VecT;
template <> struct VecT<16> { using T = uint4; };
template <> struct VecT<8> { using T = uint2; };
template <> struct VecT<4> { using T = unsigned int; };
template <> struct VecT<2> { using T = unsigned short; };
template <> struct VecT<1> { using T = unsigned char; };

struct TransposeArgs {
    const char* src;
    char* dst;
    uint64_t units;          // num_blocks * num_heads
    uint32_t bs, H;          // block_size, num_heads
    uint32_t cb;             // bytes of one x-chunk (x * element bytes)
    uint32_t rowb;           // bytes of one head row (head_dim * element bytes)
    uint32_t vpr;            // VEC-vectors per head row
    uint32_t vpr_m, vpr_l;   // divide by vpr
    uint32_t cb_m, cb_l;     // divide by cb
    uint32_t nv, nv_m, nv_l; // VEC-vectors per unit, divide by nv
    uint32_t per_tile;       // units staged together (their bytes fit the tile)
    uint32_t bs_m, bs_l;     // divide by bs (swizzled layout)
    uint32_t H_m, H_l;       // divide by H
};

// Offset in a staged unit ([D/x, bs, x] order) of byte `byte` of slot t's row.
template <bool SWZ>
__device__ __forceinline__ uint32_t tile_offset(const TransposeArgs& a, uint32_t t, uint32_t byte)
{
    const uint32_t dx = div_invariant(byte, a.cb_m, a.cb_l);  // which x-chunk
    if (SWZ) return (dx * a.bs + (t ^ (dx & 7))) * 16;       // cb == 16: byte is dx * 16
    return (dx * a.bs + t) * a.cb + (byte - dx * a.cb);
}

// Offset in a staged unit of its linear 16-byte chunk p (= dx * bs + t).
template <bool SWZ>
__device__ __forceinline__ uint32_t linear_offset(const TransposeArgs& a, uint32_t p)
{
    if (!SWZ) return p * 16;
    return (p ^ (div_invariant(p, a.bs_m, a.bs_l) & 7)) * 16;
}

// Up to per_tile consecutive units (u = block * H + head) are staged at once (up to
// 32 KiB); each thread moves its vectors in batches of kBatch, every load of a batch
// issued before the first use.  The interchange-side address of staged vector i: unit
// k = i / nv, slot t and byte offset within the slot's row from the rest; the unit's
// block and head come from the tile's first unit by a 32-bit step (no 64-bit division
// per vector).
constexpr int kBatch = 8;

template <int VEC>
__device__ __forceinline__ uint64_t interchange_offset(const TransposeArgs& a, uint64_t b0,
                                                       uint32_t h0, uint32_t i, uint32_t& k,
                                                       uint32_t& t, uint32_t& byte)
{
    k = div_invariant(i, a.nv_m, a.nv_l);
    const uint32_t iv = i - k * a.nv;
    t = div_invariant(iv, a.vpr_m, a.vpr_l);
    byte = (iv - t * a.vpr) * VEC;
    uint32_t h = h0 + k;
    const uint32_t db = div_invariant(h, a.H_m, a.H_l);
    h -= db * a.H;
    return (((b0 + db) * a.bs + t) * a.H + h) * a.rowb + byte;
}

template <int VEC, bool TO_INTERCHANGE, bool SWZ>
__global__ void __launch_bounds__(kThreads) transpose_kernel(const TransposeArgs a)
{
    static_assert(!SWZ || VEC == 16, "the swizzled layout moves 16-byte chunks");
    using T = typename VecT<VEC>::T;
    extern __shared__ __align__(16) unsigned char tile[];
    const uint32_t U = a.bs * a.rowb;  // bytes of a unit
    for (uint64_t u0 = (uint64_t)blockIdx.x * a.per_tile; u0 < a.units;
         u0 += (uint64_t)gridDim.x * a.per_tile) {
        const uint32_t k_units = (uint32_t)(a.units - u0 < a.per_tile ? a.units - u0 : a.per_tile);
        const uint32_t n = k_units * a.nv;
        const uint64_t b0 = u0 / a.H;
        const uint32_t h0 = (uint32_t)(u0 - b0 * a.H);
        // phase 1: global -> tile
        for (uint32_t base = 0; base < n; base += kThreads * kBatch) {
            T r[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const uint32_t i = base + threadIdx.x + j * kThreads;
                if (i < n) {
                    if (TO_INTERCHANGE) {  // internal units u0.. are contiguous
                        r[j] = __ldg(reinterpret_cast<const T*>(a.src + u0 * U) + i);
                    } else {
                        uint32_t k, t, byte;
                        r[j] = __ldg(reinterpret_cast<const T*>(
                            a.src + interchange_offset<VEC>(a, b0, h0, i, k, t, byte)));
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const uint32_t i = base + threadIdx.x + j * kThreads;
                if (i < n) {
                    const uint32_t k = div_invariant(i, a.nv_m, a.nv_l);
                    uint32_t off;
                    if (TO_INTERCHANGE) {
                        off = SWZ ? linear_offset<true>(a, i - k * a.nv) : (i - k * a.nv) * VEC;
                    } else {
                        const uint32_t iv = i - k * a.nv;
                        const uint32_t t = div_invariant(iv, a.vpr_m, a.vpr_l);
                        off = tile_offset<SWZ>(a, t, (iv - t * a.vpr) * VEC);
                    }
                    *reinterpret_cast<T*>(tile + k * U + off) = r[j];
                }
            }
        }
        __syncthreads();
        // phase 2: tile -> global
        for (uint32_t base = 0; base < n; base += kThreads * kBatch) {
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const uint32_t i = base + threadIdx.x + j * kThreads;
                if (i < n) {
                    const uint32_t k = div_invariant(i, a.nv_m, a.nv_l);
                    if (TO_INTERCHANGE) {
                        uint32_t kk, t, byte;
                        const uint64_t g = interchange_offset<VEC>(a, b0, h0, i, kk, t, byte);
                        *reinterpret_cast<T*>(a.dst + g) =
                            *reinterpret_cast<const T*>(tile + k * U + tile_offset<SWZ>(a, t, byte));
                    } else {
                        const uint32_t off =
                            SWZ ? linear_offset<true>(a, i - k * a.nv) : (i - k * a.nv) * VEC;
                        reinterpret_cast<T*>(a.dst + u0 * U)[i] =
                            *reinterpret_cast<const T*>(tile + k * U + off);
                    }
                }
            }
        }
        __syncthreads();  // the tile is reused by the next units
    }
}

template <int VEC, bool TO, bool SWZ = false>
int launch_t(const TransposeArgs& a, uint32_t smem, cudaStream_t st)
{
    auto kern = transpose_kernel<VEC, TO, SWZ>;
    int dev = 0;
    const int sms = current_sms(&dev);
    if (sms == 0) return HP_ERR_CUDA;
    const int per_sm = resident_ctas<transpose_kernel<VEC, TO, SWZ>>(dev, kThreads, smem);
    if (per_sm == 0) return HP_ERR_CUDA;
    const uint64_t tiles = (a.units + a.per_tile - 1) / a.per_tile;
    const uint64_t grid = std::min<uint64_t>(tiles, (uint64_t)sms * per_sm);
    if (grid == 0) return HP_OK;
    kern<<<(unsigned)grid, kThreads, smem, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? HP_OK : HP_ERR_CUDA;
}

}  // namespace

int launch_transpose(const void* src, void* dst, uint64_t nb, uint64_t bs, uint64_t H,
                     uint64_t D, uint64_t x, uint64_t es, bool to_interchange, void* stream)
{
    TransposeArgs a{};
    a.src = static_cast<const char*>(src);
    a.dst = static_cast<char*>(dst);
    a.units = nb * H;
    a.bs = (uint32_t)bs;
    a.H = (uint32_t)H;
    a.cb = (uint32_t)(x * es);
    a.rowb = (uint32_t)(D * es);
    // widest vector dividing the chunk, the row and both bases
    const uintptr_t m = a.cb | a.rowb | reinterpret_cast<uintptr_t>(src) |
                        reinterpret_cast<uintptr_t>(dst);
    int vec = 1;
    for (int v = 16; v > 1; v >>= 1)
        if (m % v == 0) {
            vec = v;
            break;
        }
    a.vpr = a.rowb / vec;
    invariant_divisor(a.vpr, &a.vpr_m, &a.vpr_l);
    invariant_divisor(a.cb, &a.cb_m, &a.cb_l);
    const uint32_t U = a.bs * a.rowb;
    a.nv = U / vec;
    invariant_divisor(a.nv, &a.nv_m, &a.nv_l);
    a.per_tile = U >= 32768 ? 1 : 32768 / U;
    invariant_divisor(a.H, &a.H_m, &a.H_l);
    const uint32_t smem = a.per_tile * U;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (vec == 16 && a.cb == 16 && bs % 8 == 0) {
        invariant_divisor(a.bs, &a.bs_m, &a.bs_l);
        return to_interchange ? launch_t<16, true, true>(a, smem, st)
                              : launch_t<16, false, true>(a, smem, st);
    }
#define HP_TR(v)                                                                        \
    case v:                                                                             \
        return to_interchange ? launch_t<v, true>(a, smem, st) : launch_t<v, false>(a, smem, st);
    switch (vec) {
        HP_TR(16) HP_TR(8) HP_TR(4) HP_TR(2)
    default:
        return to_interchange ? launch_t<1, true>(a, smem, st) : launch_t<1, false>(a, smem, st);
    }
#undef HP_TR
}

}  // namespace hp
