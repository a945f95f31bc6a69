// hp_internal.cuh -- shared declarations of the libhp CUDA sources (not installed).
//
// Workspace layout (device, 256-byte aligned, hp_workspace_bytes() bytes):
//   [0, 64)          WsHeader: verdict key, totals
//   [256, 256+A)     rows_off[S+1]  exclusive prefix of the token counts (first output
//                    row of each sequence), A = round_up(8*(S+1), 256)
//   [256+A, 256+2A)  units_off[S+1] exclusive prefix of each sequence's copy units
//                    (page spans of a gather, pages touched by an append)
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "hp.h"

namespace hp {

// Rule ranks: the order in which the checks of a descriptor apply.  A verdict
// key is (rank << 58) | index; the smallest key is the first failing rule at
// its first failing index.  kVerdictOk means no rule failed.
enum Rank : unsigned {
    kRankSeqPtrStart = 1,
    kRankSeqPtrOrder = 2,
    kRankSeqPtrEnd = 3,
    kRankPageId = 4,
    kRankLen = 5,
    kRankNewPtrStart = 6,
    kRankNewPtrOrder = 7,
    kRankNewPtrEnd = 8,
    kRankCapacity = 9,
    kRankOutSize = 10,
};
constexpr unsigned long long kVerdictOk = ~0ull;
constexpr unsigned long long kIndexMask = (1ull << 58) - 1;

__host__ __device__ inline unsigned long long verdict_key(unsigned rank, unsigned long long index)
{
    return ((unsigned long long)rank << 58) | (index < kIndexMask ? index : kIndexMask);
}

__host__ __device__ inline int rank_status(unsigned rank)
{
    switch (rank) {
    case kRankSeqPtrStart: return HP_ERR_SEQ_PTR_START;
    case kRankSeqPtrOrder: return HP_ERR_SEQ_PTR_ORDER;
    case kRankSeqPtrEnd: return HP_ERR_SEQ_PTR_END;
    case kRankPageId: return HP_ERR_PAGE_ID;
    case kRankLen: return HP_ERR_LEN;
    case kRankNewPtrStart: return HP_ERR_NEW_PTR_START;
    case kRankNewPtrOrder: return HP_ERR_NEW_PTR_ORDER;
    case kRankNewPtrEnd: return HP_ERR_NEW_PTR_END;
    case kRankCapacity: return HP_ERR_CAPACITY;
    case kRankOutSize: return HP_ERR_OUT_SIZE;
    default: return HP_OK;
    }
}

__host__ __device__ inline int key_status(unsigned long long key)
{
    return key == kVerdictOk ? HP_OK : rank_status((unsigned)(key >> 58));
}

struct WsHeader {
    unsigned long long verdict;      // smallest failing key, kVerdictOk if none
    unsigned long long total_rows;   // sum of token counts (gather)
    unsigned long long total_units;  // units_off[S]
    unsigned long long pad[5];
};

constexpr uint64_t kWsHeaderBytes = 256;

inline uint64_t round_up_256(uint64_t x) { return (x + 255) & ~255ull; }

struct WsView {
    WsHeader* hdr;
    unsigned long long* rows_off;
    unsigned long long* units_off;
};

inline WsView ws_view(void* ws, uint64_t num_seqs)
{
    char* base = static_cast<char*>(ws);
    uint64_t a = round_up_256(8 * (num_seqs + 1));
    return WsView{reinterpret_cast<WsHeader*>(base),
                  reinterpret_cast<unsigned long long*>(base + kWsHeaderBytes),
                  reinterpret_cast<unsigned long long*>(base + kWsHeaderBytes + a)};
}

// ------------------------------------------------------------------ plan step
enum PlanMode { kPlanGather = 0, kPlanAppend = 1, kPlanAttention = 2 };

struct PlanArgs {
    const void* seq_ptr;
    const void* lens;
    const void* new_ptr;      // append only
    const void* table;
    uint64_t num_seqs, page_size, table_len, num_pages;
    uint64_t out_tokens;      // gather: expected total rows
    uint64_t total_new;       // append: expected new_ptr[S]
    uint64_t step_tokens;     // attention: tokens per step (its units are steps)
    int strict;               // check the storage invariants
    int check_out;            // gather: compare the total with out_tokens
    int* d_status;
    WsView ws;
};

// Launches the plan (and, when strict, the block-table check) on `stream`.
int launch_plan(PlanMode mode, int index_u64, const PlanArgs& a, void* stream);

// Block-table forms (hp_plan.cu): padded [batch, max_blocks] + counts <-> CSR slices.
struct TableArgs {
    bool to_csr;
    const void* in;        // padded (to_csr) or CSR table
    const void* lens;      // to_csr: token counts
    const void* seq_ptr;   // from CSR: offsets
    void* out;             // CSR table (to_csr) or padded
    void* out2;            // to_csr: seq_ptr out
    uint64_t batch, max_blocks, page_size, cap, table_len, pad;
    void* workspace;       // header + batch+1 prefix entries
    int* d_status;
};
int launch_tables(int index_u64, const TableArgs& t, void* stream);

// Layout transpose (hp_layout.cu) between [nb, H, D/x, bs, x] and [nb, bs, H, D].
int launch_transpose(const void* src, void* dst, uint64_t nb, uint64_t bs, uint64_t H,
                     uint64_t D, uint64_t x, uint64_t es, bool to_interchange, void* stream);

// Writer side (hp_writer.cu): after a plan on `stream`, the per-page live counts and the
// zeroing of the slots past them.
int launch_zero_tails(int index_u64, const PlanArgs& a, unsigned* live, uint64_t row_bytes,
                      void* pool, void* stream);

// ------------------------------------------------------------------ copy step
enum CopyMode {
    kGather = 0,
    kDequant = 1,
    kAppend = 2,
    kLaneGather = 3,
    kLaneAppend = 4,
    kCopyPages = 5,  // whole pages src_pages[u] -> dst_pages[u] (host-known count)
};

// Modes whose unit count the host passes (no plan in front of the copy).
__host__ __device__ constexpr bool host_counted(int mode)
{
    return mode == kLaneGather || mode == kLaneAppend || mode == kCopyPages;
}

struct CopyArgs {
    // block-paged descriptor data
    const void* seq_ptr;
    const void* lens;
    const void* new_ptr;
    const void* table;
    const float* scales;
    uint64_t num_seqs, page_size, table_len, num_pages;
    uint64_t total_new;
    const WsHeader* hdr;
    const unsigned long long* rows_off;
    const unsigned long long* units_off;
    // per-lane layout (lane_units is also the pair count of kCopyPages)
    uint64_t lanes, lane_n, lane_m, lane_units, lane_first_page, lane_pages;
    const void* src_pages;    // kCopyPages
    const void* dst_pages;
    // data movement
    const char* src;          // gather: pool; append: new rows
    char* dst;                // gather: out; append: pool
    uint64_t row_bytes;       // bytes of one source row
    uint64_t row_elems;       // elements of one row (dequant)
    uint64_t unit_bytes;      // largest unit: page_size rows of row_bytes
    uint32_t div_m, div_l;    // dequant: divide a group index by row_elems/8
    // dequant scheme: q_kind = scheme * 2 + (zero points present), scheme 0 per page slot,
    // 1 per tensor, 2 per head (axis 1), 3 per feature (axis 2)
    int q_kind;
    int q_signed;             // codes are int8 (1) or uint8 (0)
    const unsigned char* q_zp;  // zero points, one byte each, or NULL
    uint32_t q_gpr, q_gph;    // groups of 8 per row, per head
    uint32_t q_hd_m, q_hd_l;  // divide a group-in-row index by q_gph
    uint64_t q_head_dim;
    int q_fixed;              // per channel: q_gpr divides the CTA width (a power of two)
    int test_stall;           // HP_TEST_STALL: the TMA engine never issues its first load
    int* d_status;
};

int launch_copy(CopyMode mode, int index_u64, const CopyArgs& a, int vec, void* stream);

// The permissive decode-step append (hp_writer.cu): one warp per sequence, no plan.
int launch_append_rows(int index_u64, const CopyArgs& a, int vec, void* stream);

// The TMA bulk engine (hp_bulk.cu): pure copies whose rows and bases are 16-byte aligned.
// big_stages selects 16 KiB ring stages with split roles (else 8 KiB, one producer).
int launch_bulk(CopyMode mode, int index_u64, const CopyArgs& a, int big_stages, void* stream);

// ------------------------------------------------------- per-device launch facts
// Looked up on first use on each device and kept for the process: the launch path then
// costs no runtime queries (a decode step's latency is mostly launch overhead).
constexpr int kMaxDevices = 256;

// SM count of the current device (0 if it cannot be read); *dev receives the ordinal.
inline int current_sms(int* dev)
{
    static std::atomic<int> cache[kMaxDevices];
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return 0;
    int v = cache[*dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess)
            return 0;
        cache[*dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

// Resident CTAs per SM of `kernel` on `dev` (one cache per kernel).
template <auto kernel>
inline int resident_ctas(int dev, int threads, size_t smem)
{
    static std::atomic<int> cache[kMaxDevices];
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kernel, threads, smem) != cudaSuccess)
            return 0;
        if (v < 1) v = 1;
        cache[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

// Raises `kernel`'s dynamic shared-memory limit on `dev` once.
template <auto kernel>
inline bool allow_dynamic_smem(int dev, int bytes)
{
    static std::atomic<int> done[kMaxDevices];
    if (done[dev].load(std::memory_order_acquire)) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
        return false;
    done[dev].store(1, std::memory_order_release);
    return true;
}

// Quotient n / d for an invariant divisor d <= 2^31 from a multiply-high and shifts:
// m = floor(2^32 (2^l - d) / d) + 1 with l = ceil(log2 d), computed on the host
// (Granlund and Montgomery, "Division by invariant integers using multiplication",
// PLDI 1994, round-up method).
__device__ __forceinline__ uint32_t div_invariant(uint32_t n, uint32_t m, uint32_t l)
{
    if (l == 0) return n;
    const uint32_t t1 = __umulhi(m, n);
    return (t1 + ((n - t1) >> 1)) >> (l - 1);
}

// Host side of div_invariant: (m, l) for the divisor g (1 <= g <= 2^31).
inline void invariant_divisor(uint64_t g, uint32_t* m, uint32_t* l)
{
    uint32_t ll = 0;
    while ((1ull << ll) < g) ++ll;  // ceil(log2 g)
    *l = ll;
    *m = (uint32_t)(((((unsigned __int128)1) << 32) * ((((unsigned __int128)1) << ll) - g)) / g + 1);
}

// ------------------------------------------------------- dependent launches
// The plan, the block-table check and the copy go into the stream back to back.  The
// check and the copy are launched as programmatic dependents of the kernel before
// them, so their CTAs are scheduled while it finishes; each waits (griddepcontrol.wait)
// before it touches anything that kernel writes, and writes nothing before that wait.
// The plan itself is launched normally: it overwrites the workspace a previous copy
// may still be reading.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename Kernel, typename... Args>
inline cudaError_t launch_dependent(Kernel kernel, unsigned grid, unsigned block, size_t smem,
                                    cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace hp
