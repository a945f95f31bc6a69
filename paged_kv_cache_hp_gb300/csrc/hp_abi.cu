// hp_abi.cu -- the extern "C" entry points of libhp.so (declared in include/hp.h):
// host-side argument checks, then the plan and copy launches on the caller's stream.
//
// The structural checks follow "Block-Paged Layout -- Hurray Format Specification":
// Description (rank 3), Logical Shape (paged_axis 0), Sharding (no shard descriptor),
// Additional Descriptor Fields (index type 0x00 / 0x01; uint32 addresses at most
// 0xFFFFFFFF pages), Scale-buffer size (num_pages * page_size scales), Alignment
// (64 bytes) and Storage Invariants (4) (the pool's byte size).  The lane checks follow
// the constructor of "Keep token order across cache pages" (PagedKvLayout::new).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <vector>

#include "hp_attn.cuh"
#include "hp_internal.cuh"
#include "hp_small.cuh"

#define HP_API extern "C" __attribute__((visibility("default")))

namespace {

using u64 = uint64_t;
using u128 = unsigned __int128;

u64 elem_bytes(uint32_t dtype)
{
    switch (dtype) {
    case HP_F32: return 4;
    case HP_F16: return 2;
    case HP_BF16: return 2;
    case HP_I8: return 1;
    case HP_U8: return 1;
    case HP_F64: return 8;
    default: return 0;
    }
}

bool misaligned(const void* p, u64 a) { return reinterpret_cast<uintptr_t>(p) % a != 0; }

int check_desc(const hp_paged_desc* d)
{
    if (!d) return HP_ERR_NULL;
    if (d->rank != 3) return HP_ERR_RANK;
    if (d->paged_axis != 0) return HP_ERR_PAGED_AXIS;
    if (d->has_shard) return HP_ERR_SHARD;
    if (d->index_type != HP_IDX_U32 && d->index_type != HP_IDX_U64) return HP_ERR_INDEX_TYPE;
    if (d->index_type == HP_IDX_U32 && (d->num_pages > (1ull << 32) || d->table_len > 0xFFFFFFFFull))
        return HP_ERR_INDEX_TYPE;
    const u64 es = elem_bytes(d->dtype);
    if (!es) return HP_ERR_DTYPE;
    if (!d->page_size || !d->num_heads || !d->head_dim) return HP_ERR_ZERO_DIM;
    const bool quant = d->flags & HP_HAS_QUANT;
    if (quant && (!d->scales || (u128)d->scales_len != (u128)d->num_pages * d->page_size))
        return HP_ERR_SCALES;
    if ((d->num_pages && !d->page_pool) || !d->seq_ptr || (d->num_seqs && !d->seq_lens) ||
        (d->table_len && !d->block_table))
        return HP_ERR_NULL;
    if (misaligned(d->page_pool, 64) || misaligned(d->block_table, 64) ||
        misaligned(d->seq_ptr, 64) || misaligned(d->seq_lens, 64) ||
        (quant && misaligned(d->scales, 64)))
        return HP_ERR_ALIGN;
    u128 bytes = (u128)d->num_pages * d->page_size;
    bytes *= d->num_heads;
    if (bytes >> 64) return HP_ERR_OVERFLOW;
    bytes *= d->head_dim;
    if (bytes >> 64) return HP_ERR_OVERFLOW;
    bytes *= es;
    if (bytes >> 64) return HP_ERR_OVERFLOW;
    return HP_OK;
}

u64 row_bytes_of(const hp_paged_desc* d)
{
    return d->num_heads * d->head_dim * elem_bytes(d->dtype);
}

int ws_bytes(const hp_paged_desc* d, u64* out)
{
    if (d->num_seqs >= (1ull << 58)) return HP_ERR_OVERFLOW;
    *out = hp::kWsHeaderBytes + 2 * hp::round_up_256(8 * (d->num_seqs + 1));
    return HP_OK;
}

int check_ws(const hp_paged_desc* d, const void* ws, u64 have)
{
    u64 need = 0;
    int rc = ws_bytes(d, &need);
    if (rc) return rc;
    if (!ws || misaligned(ws, 256) || have < need) return HP_ERR_WORKSPACE;
    return HP_OK;
}

// Widest power-of-two vector (<= 16 bytes) that divides the row and both bases.
int pick_vec(u64 row_bytes, const void* a, const void* b)
{
    const uintptr_t m = static_cast<uintptr_t>(row_bytes) | reinterpret_cast<uintptr_t>(a) |
                        reinterpret_cast<uintptr_t>(b);
    for (int v = 16; v > 1; v >>= 1)
        if (m % v == 0) return v;
    return 1;
}

hp::PlanArgs plan_args(const hp_paged_desc* d, void* ws, int* d_status)
{
    hp::PlanArgs a{};
    a.seq_ptr = d->seq_ptr;
    a.lens = d->seq_lens;
    a.table = d->block_table;
    a.num_seqs = d->num_seqs;
    a.page_size = d->page_size;
    a.table_len = d->table_len;
    a.num_pages = d->num_pages;
    a.strict = !(d->flags & HP_PERMISSIVE);
    a.d_status = d_status;
    a.ws = hp::ws_view(ws, d->num_seqs);
    return a;
}

hp::CopyArgs copy_args(const hp_paged_desc* d, const void* ws, int* d_status)
{
    hp::CopyArgs a{};
    a.seq_ptr = d->seq_ptr;
    a.lens = d->seq_lens;
    a.table = d->block_table;
    a.scales = d->scales;
    a.num_seqs = d->num_seqs;
    a.page_size = d->page_size;
    a.table_len = d->table_len;
    a.num_pages = d->num_pages;
    const hp::WsView v = hp::ws_view(const_cast<void*>(ws), d->num_seqs);
    a.hdr = v.hdr;
    a.rows_off = v.rows_off;
    a.units_off = v.units_off;
    a.row_bytes = row_bytes_of(d);
    a.row_elems = d->num_heads * d->head_dim;
    a.unit_bytes = d->page_size * a.row_bytes;
    a.test_stall = (d->flags & HP_TEST_STALL) != 0;
    a.d_status = d_status;
    return a;
}

// HP_HOST_MEMORY: the caller's buffers may be page-locked host memory (e.g. Grace memory
// holding an offloaded pool).  Kernels reach it with ordinary loads and stores over the
// host link; the TMA copy engine is kept to device memory, so such an operation takes the
// register engine.  The caller declares it; no runtime query runs per call.
inline bool host_memory(uint32_t flags) { return (flags & HP_HOST_MEMORY) != 0; }

// Units of at most 8 KiB keep an operation on the register engine (one warp per unit).
constexpr u64 kRegisterEngineUnit = 8192;

int sync_verdict(const void* ws, u64* first_bad, void* stream)
{
    unsigned long long key = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&key, &static_cast<const hp::WsHeader*>(ws)->verdict, sizeof(key),
                        cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return HP_ERR_CUDA;
    if (first_bad) *first_bad = key == hp::kVerdictOk ? 0 : (key & hp::kIndexMask);
    return hp::key_status(key);
}

// [HF] Per-scheme composition, for hp_gather_dequant_q, in the order hp.h lists.
int check_quant(const hp_paged_desc* d, const hp_quant_desc* q)
{
    if (!q) return HP_ERR_NULL;
    if (d->dtype != HP_I8 && d->dtype != HP_U8) return HP_ERR_DTYPE;
    u64 want;
    if (q->scheme_tag == HP_QUANT_PER_TENSOR) {
        want = 1;
    } else if (q->scheme_tag == HP_QUANT_PER_CHANNEL) {
        if (q->axis == 1) want = d->num_heads;
        else if (q->axis == 2) want = d->head_dim;
        else return HP_ERR_QUANT_SCHEME;
    } else if (q->scheme_tag == HP_QUANT_PER_BLOCK_AFFINE) {
        if (q->axis != 0 || q->block_size != d->page_size) return HP_ERR_QUANT_BLOCK;
        const u128 n = (u128)d->num_pages * d->page_size;
        if (n >> 64) return HP_ERR_SCALES;
        want = (u64)n;
    } else {
        return HP_ERR_QUANT_SCHEME;
    }
    if (q->count != want) return HP_ERR_SCALES;
    if (!q->scales) return HP_ERR_NULL;
    if (misaligned(q->scales, 64) || misaligned(q->zero_points, 64)) return HP_ERR_ALIGN;
    return HP_OK;
}

// The copy step of a gather; `dequant` selects the dequantising forms, with the
// parameters of `quant` or (quant == NULL) the descriptor's per-slot scales.
int gather_planned(const hp_paged_desc* d, void* out, const void* ws, int* d_status,
                   void* stream, bool dequant, const hp_quant_desc* quant = nullptr)
{
    int rc = check_desc(d);
    if (rc) return rc;
    if (dequant && quant) {
        rc = check_quant(d, quant);
        if (rc) return rc;
    } else if (dequant) {
        if (d->dtype != HP_I8) return HP_ERR_DTYPE;
        if (!(d->flags & HP_HAS_QUANT)) return HP_ERR_SCALES;
    }
    if (!ws || misaligned(ws, 256)) return HP_ERR_WORKSPACE;
    if (d->num_seqs == 0) return HP_OK;
    if (!out) return HP_ERR_NULL;
    hp::CopyArgs a = copy_args(d, ws, d_status);
    a.src = static_cast<const char*>(d->page_pool);
    a.dst = static_cast<char*>(out);
    int vec;
    if (dequant) {
        int scheme = 0;  // per page slot
        if (quant) {
            a.scales = quant->scales;
            a.q_zp = static_cast<const unsigned char*>(quant->zero_points);
            if (quant->scheme_tag == HP_QUANT_PER_TENSOR) scheme = 1;
            else if (quant->scheme_tag == HP_QUANT_PER_CHANNEL) scheme = quant->axis == 1 ? 2 : 3;
        }
        a.q_kind = scheme * 2 + (a.q_zp != nullptr);
        a.q_signed = d->dtype == HP_I8;
        a.q_head_dim = d->head_dim;
        // groups of 8 elements per thread when rows (and, per channel, heads) split into
        // them and a unit's groups fit 32-bit indices; element by element otherwise
        const u64 g = a.row_elems / 8;
        const bool per_channel = scheme >= 2;
        const bool v8 = a.row_elems % 8 == 0 && !misaligned(out, 16) && g <= (1ull << 31) &&
                        (u128)d->page_size * g < ((u128)1 << 32) &&
                        (!per_channel || d->head_dim % 8 == 0);
        if (v8) {
            hp::invariant_divisor(g, &a.div_m, &a.div_l);
            a.q_gpr = (uint32_t)g;
            if (per_channel) {
                a.q_gph = (uint32_t)(d->head_dim / 8);
                hp::invariant_divisor(a.q_gph, &a.q_hd_m, &a.q_hd_l);
                a.q_fixed = 256 % g == 0;  // the copy kernel's CTA width
            }
        }
        vec = v8 ? 16 : 1;
        return hp::launch_copy(hp::kDequant, d->index_type == HP_IDX_U64, a, vec, stream);
    }
    vec = pick_vec(a.row_bytes, d->page_pool, out);
    if (host_memory(d->flags)) a.unit_bytes = std::min<u64>(a.unit_bytes, kRegisterEngineUnit);
    return hp::launch_copy(hp::kGather, d->index_type == HP_IDX_U64, a, vec, stream);
}

// The descriptor a scheme-driven dequantising gather validates: its quantisation
// parameters come from the hp_quant_desc, so the descriptor's own flag is dropped.
hp_paged_desc without_quant_flag(const hp_paged_desc* d)
{
    hp_paged_desc c = *d;
    c.flags &= ~HP_HAS_QUANT;
    return c;
}

int plan_gather(const hp_paged_desc* d, u64 out_tokens, void* ws, u64 wsb, int* d_status,
                void* stream, bool check_out)
{
    int rc = check_ws(d, ws, wsb);
    if (rc) return rc;
    if (check_out) {
        // a dequantising gather writes 2-byte elements from 1-byte codes
        const u64 es = elem_bytes(d->dtype) < 2 ? 2 : elem_bytes(d->dtype);
        const u128 out_bytes = (u128)out_tokens * d->num_heads * d->head_dim * es;
        if (out_bytes >> 64) return HP_ERR_OUT_SIZE;
    }
    hp::PlanArgs a = plan_args(d, ws, d_status);
    a.out_tokens = out_tokens;
    a.check_out = check_out;
    return hp::launch_plan(hp::kPlanGather, d->index_type == HP_IDX_U64, a, stream);
}

int plan_append(const hp_paged_desc* d, const void* new_ptr, u64 total_new, void* ws, u64 wsb,
                int* d_status, void* stream)
{
    int rc = check_ws(d, ws, wsb);
    if (rc) return rc;
    if (!new_ptr) return HP_ERR_NULL;
    if (misaligned(new_ptr, d->index_type == HP_IDX_U64 ? 8 : 4)) return HP_ERR_ALIGN;
    if ((u128)total_new * row_bytes_of(d) >> 64) return HP_ERR_OVERFLOW;
    hp::PlanArgs a = plan_args(d, ws, d_status);
    a.new_ptr = new_ptr;
    a.total_new = total_new;
    return hp::launch_plan(hp::kPlanAppend, d->index_type == HP_IDX_U64, a, stream);
}

int append_planned(const hp_paged_desc* d, const void* new_rows, const void* new_ptr,
                   u64 total_new, const void* ws, int* d_status, void* stream)
{
    if (!ws || misaligned(ws, 256)) return HP_ERR_WORKSPACE;
    if (d->num_seqs == 0) return HP_OK;
    if (!new_ptr) return HP_ERR_NULL;
    hp::CopyArgs a = copy_args(d, ws, d_status);
    a.new_ptr = new_ptr;
    a.total_new = total_new;
    if ((u128)total_new < (u128)d->num_seqs * d->page_size) {
        // decode-sized: one warp per sequence after the plan's verdict, no unit search
        a.src = static_cast<const char*>(new_rows);
        a.dst = static_cast<char*>(const_cast<void*>(d->page_pool));
        if (!a.src) a.src = reinterpret_cast<const char*>(d->page_pool);  // never read
        return hp::launch_append_rows(d->index_type == HP_IDX_U64, a,
                                      pick_vec(a.row_bytes, a.src, d->page_pool), stream);
    }
    // a unit is at most one page of rows, and on average total_new / num_seqs rows
    const u64 avg_rows = total_new / d->num_seqs + (total_new % d->num_seqs != 0);
    if (avg_rows < d->page_size) a.unit_bytes = avg_rows * a.row_bytes;
    a.src = static_cast<const char*>(new_rows);
    a.dst = static_cast<char*>(const_cast<void*>(d->page_pool));
    if (!a.src) a.src = reinterpret_cast<const char*>(d->page_pool);  // no rows: never read
    const int vec = pick_vec(a.row_bytes, a.src, d->page_pool);
    if (host_memory(d->flags)) a.unit_bytes = std::min<u64>(a.unit_bytes, kRegisterEngineUnit);
    return hp::launch_copy(hp::kAppend, d->index_type == HP_IDX_U64, a, vec, stream);
}

// Lane-layout argument checks shared by gather and append.
int check_lane(const void* pool, const uint64_t* table, u64 capacity, u64 page_tokens, u64 batch,
               u64 kv_heads, u64 width, uint32_t dtype, u64* pages, u64* row_bytes)
{
    const u64 es = elem_bytes(dtype);
    if (!es) return HP_ERR_DTYPE;
    if (capacity == 0) return HP_ERR_ZERO_CAPACITY;
    if (page_tokens == 0) return HP_ERR_ZERO_PAGE_SIZE;
    if (!batch || !kv_heads || !width) return HP_ERR_ZERO_DIM;
    const u64 n_pages = capacity / page_tokens + (capacity % page_tokens != 0);
    u128 total = (u128)n_pages * page_tokens;
    if (total >> 64) return HP_ERR_LANE_OVERFLOW;
    total *= batch;
    if (total >> 64) return HP_ERR_LANE_OVERFLOW;
    total *= kv_heads;
    if (total >> 64) return HP_ERR_LANE_OVERFLOW;
    total *= width;
    if (total >> 64) return HP_ERR_LANE_OVERFLOW;
    total *= es;
    if (total >> 64) return HP_ERR_LANE_OVERFLOW;
    if (!pool || !table) return HP_ERR_NULL;
    if (misaligned(table, 8)) return HP_ERR_ALIGN;
    *pages = n_pages;
    *row_bytes = width * es;
    return HP_OK;
}

int reset_status(int* d_status, void* stream)
{
    if (!d_status) return HP_OK;
    return cudaMemsetAsync(d_status, 0, sizeof(int), static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? HP_OK
               : HP_ERR_CUDA;
}

}  // namespace

// ============================================================================ API

HP_API const char* hp_status_string(int s)
{
    switch (s) {
#define HP_NAME(c) \
    case c: return #c;
        HP_NAME(HP_OK)
        HP_NAME(HP_ERR_RANK)
        HP_NAME(HP_ERR_PAGED_AXIS)
        HP_NAME(HP_ERR_SHARD)
        HP_NAME(HP_ERR_INDEX_TYPE)
        HP_NAME(HP_ERR_DTYPE)
        HP_NAME(HP_ERR_ZERO_DIM)
        HP_NAME(HP_ERR_SCALES)
        HP_NAME(HP_ERR_NULL)
        HP_NAME(HP_ERR_ALIGN)
        HP_NAME(HP_ERR_OVERFLOW)
        HP_NAME(HP_ERR_SEQ_PTR_START)
        HP_NAME(HP_ERR_SEQ_PTR_ORDER)
        HP_NAME(HP_ERR_SEQ_PTR_END)
        HP_NAME(HP_ERR_PAGE_ID)
        HP_NAME(HP_ERR_LEN)
        HP_NAME(HP_ERR_NEW_PTR_START)
        HP_NAME(HP_ERR_NEW_PTR_ORDER)
        HP_NAME(HP_ERR_NEW_PTR_END)
        HP_NAME(HP_ERR_CAPACITY)
        HP_NAME(HP_ERR_OUT_SIZE)
        HP_NAME(HP_ERR_ZERO_CAPACITY)
        HP_NAME(HP_ERR_ZERO_PAGE_SIZE)
        HP_NAME(HP_ERR_LANE_OVERFLOW)
        HP_NAME(HP_ERR_PAGE_COUNT)
        HP_NAME(HP_ERR_PHYSICAL_PAGE)
        HP_NAME(HP_ERR_ALIASED_PAGE)
        HP_NAME(HP_ERR_LENGTH)
        HP_NAME(HP_ERR_ALLOCATION_FAILED)
        HP_NAME(HP_ERR_WORKSPACE)
        HP_NAME(HP_ERR_ARG)
        HP_NAME(HP_ERR_CUDA)
        HP_NAME(HP_ERR_TIMEOUT)
        HP_NAME(HP_ERR_NOALLOC_LIMIT)
        HP_NAME(HP_ERR_QUANT_SCHEME)
        HP_NAME(HP_ERR_QUANT_BLOCK)
#undef HP_NAME
    default: return "HP_ERR_UNKNOWN";
    }
}

HP_API int hp_workspace_bytes(const hp_paged_desc* desc, uint64_t* bytes)
{
    if (!desc || !bytes) return HP_ERR_NULL;
    return ws_bytes(desc, bytes);
}

HP_API int hp_validate(const hp_paged_desc* desc, void* workspace, uint64_t workspace_bytes,
                       uint64_t* first_bad, void* stream)
{
    if (first_bad) *first_bad = 0;
    int rc = check_desc(desc);
    if (rc) return rc;
    if (desc->flags & HP_PERMISSIVE) return HP_OK;
    rc = plan_gather(desc, 0, workspace, workspace_bytes, nullptr, stream, false);
    if (rc) return rc;
    return sync_verdict(workspace, first_bad, stream);
}

HP_API int hp_plan(const hp_paged_desc* desc, uint64_t out_tokens, void* workspace,
                   uint64_t workspace_bytes, int* d_status, void* stream)
{
    int rc = check_desc(desc);
    if (rc) return rc;
    return plan_gather(desc, out_tokens, workspace, workspace_bytes, d_status, stream, true);
}

HP_API int hp_gather_planned(const hp_paged_desc* desc, void* out, const void* workspace,
                             int* d_status, void* stream)
{
    return gather_planned(desc, out, workspace, d_status, stream, false);
}

HP_API int hp_gather(const hp_paged_desc* desc, void* out, uint64_t out_tokens, void* workspace,
                     uint64_t workspace_bytes, int* d_status, void* stream)
{
    int rc = check_desc(desc);
    if (rc) return rc;
    if (out_tokens && !out) return HP_ERR_NULL;
    const hp_paged_desc* d = desc;
    if (!(d->flags & (HP_PERMISSIVE | HP_TEST_STALL)) && d->num_seqs <= hp::kMaxSeqs &&
        d->table_len <= hp::kMaxTable &&
        (u128)d->table_len * d->page_size * row_bytes_of(d) <= hp::kMaxBytes) {
        // a small validated batch: plan, table check and copy in one launch
        rc = check_ws(d, workspace, workspace_bytes);
        if (rc) return rc;
        if (((u128)out_tokens * row_bytes_of(d)) >> 64) return HP_ERR_OUT_SIZE;
        hp::SmallGatherArgs a{};
        a.seq_ptr = d->seq_ptr;
        a.lens = d->seq_lens;
        a.table = d->block_table;
        a.pool = static_cast<const char*>(d->page_pool);
        a.out = static_cast<char*>(out);
        a.num_seqs = d->num_seqs;
        a.page_size = d->page_size;
        a.table_len = d->table_len;
        a.num_pages = d->num_pages;
        a.row_bytes = row_bytes_of(d);
        a.out_tokens = out_tokens;
        a.ws = hp::ws_view(workspace, d->num_seqs);
        a.d_status = d_status;
        if (!a.pool) a.pool = static_cast<const char*>(out);  // no pages: never read
        if (!a.out) a.out = static_cast<char*>(const_cast<void*>(d->page_pool));  // no rows
        return hp::launch_small_gather(d->index_type == HP_IDX_U64, a,
                                       pick_vec(a.row_bytes, d->page_pool, out), stream);
    }
    rc = plan_gather(desc, out_tokens, workspace, workspace_bytes, d_status, stream, true);
    if (rc) return rc;
    return gather_planned(desc, out, workspace, d_status, stream, false);
}

HP_API int hp_gather_dequant_planned(const hp_paged_desc* desc, void* out_bf16,
                                     const void* workspace, int* d_status, void* stream)
{
    return gather_planned(desc, out_bf16, workspace, d_status, stream, true);
}

HP_API int hp_gather_dequant(const hp_paged_desc* desc, void* out_bf16, uint64_t out_tokens,
                             void* workspace, uint64_t workspace_bytes, int* d_status,
                             void* stream)
{
    int rc = check_desc(desc);
    if (rc) return rc;
    if (desc->dtype != HP_I8) return HP_ERR_DTYPE;
    if (!(desc->flags & HP_HAS_QUANT)) return HP_ERR_SCALES;
    if (out_tokens && !out_bf16) return HP_ERR_NULL;
    rc = plan_gather(desc, out_tokens, workspace, workspace_bytes, d_status, stream, true);
    if (rc) return rc;
    return gather_planned(desc, out_bf16, workspace, d_status, stream, true);
}

HP_API int hp_gather_dequant_q(const hp_paged_desc* desc, const hp_quant_desc* quant,
                               void* out_bf16, uint64_t out_tokens, void* workspace,
                               uint64_t workspace_bytes, int* d_status, void* stream)
{
    if (!desc) return HP_ERR_NULL;
    const hp_paged_desc d = without_quant_flag(desc);
    int rc = check_desc(&d);
    if (rc) return rc;
    rc = check_quant(&d, quant);
    if (rc) return rc;
    if (out_tokens && !out_bf16) return HP_ERR_NULL;
    rc = plan_gather(&d, out_tokens, workspace, workspace_bytes, d_status, stream, true);
    if (rc) return rc;
    return gather_planned(&d, out_bf16, workspace, d_status, stream, true, quant);
}

HP_API int hp_gather_dequant_q_planned(const hp_paged_desc* desc, const hp_quant_desc* quant,
                                       void* out_bf16, const void* workspace, int* d_status,
                                       void* stream)
{
    if (!desc) return HP_ERR_NULL;
    const hp_paged_desc d = without_quant_flag(desc);
    return gather_planned(&d, out_bf16, workspace, d_status, stream, true, quant);
}

HP_API int hp_append_plan(const hp_paged_desc* desc, const void* new_ptr, uint64_t total_new,
                          void* workspace, uint64_t workspace_bytes, int* d_status, void* stream)
{
    int rc = check_desc(desc);
    if (rc) return rc;
    return plan_append(desc, new_ptr, total_new, workspace, workspace_bytes, d_status, stream);
}

HP_API int hp_scatter_append_planned(const hp_paged_desc* desc, const void* new_rows,
                                     const void* new_ptr, uint64_t total_new,
                                     const void* workspace, int* d_status, void* stream)
{
    int rc = check_desc(desc);
    if (rc) return rc;
    return append_planned(desc, new_rows, new_ptr, total_new, workspace, d_status, stream);
}

HP_API int hp_scatter_append(const hp_paged_desc* desc, const void* new_rows, const void* new_ptr,
                             uint64_t total_new, void* workspace, uint64_t workspace_bytes,
                             int* d_status, void* stream)
{
    int rc = check_desc(desc);
    if (rc) return rc;
    if (total_new && !new_rows) return HP_ERR_NULL;
    if ((desc->flags & HP_PERMISSIVE) && desc->num_seqs &&
        (u128)total_new < (u128)desc->num_seqs * desc->page_size) {
        // decode-sized and vouched for: one warp per sequence, no plan, no table check
        rc = check_ws(desc, workspace, workspace_bytes);
        if (rc) return rc;
        if (!new_ptr) return HP_ERR_NULL;
        if (misaligned(new_ptr, desc->index_type == HP_IDX_U64 ? 8 : 4)) return HP_ERR_ALIGN;
        if ((u128)total_new * row_bytes_of(desc) >> 64) return HP_ERR_OVERFLOW;
        rc = reset_status(d_status, stream);
        if (rc) return rc;
        hp::CopyArgs a = copy_args(desc, workspace, d_status);
        a.hdr = nullptr;  // no plan to wait for
        a.new_ptr = new_ptr;
        a.total_new = total_new;  // bounds the rows read: new_ptr is not validated
        a.src = static_cast<const char*>(new_rows);
        a.dst = static_cast<char*>(const_cast<void*>(desc->page_pool));
        if (!a.src) a.src = reinterpret_cast<const char*>(desc->page_pool);  // never read
        return hp::launch_append_rows(desc->index_type == HP_IDX_U64, a,
                                      pick_vec(a.row_bytes, a.src, desc->page_pool), stream);
    }
    rc = plan_append(desc, new_ptr, total_new, workspace, workspace_bytes, d_status, stream);
    if (rc) return rc;
    return append_planned(desc, new_rows, new_ptr, total_new, workspace, d_status, stream);
}

HP_API int hp_validate_append(const hp_paged_desc* desc, const void* new_ptr, uint64_t total_new,
                              void* workspace, uint64_t workspace_bytes, uint64_t* first_bad,
                              void* stream)
{
    if (first_bad) *first_bad = 0;
    int rc = check_desc(desc);
    if (rc) return rc;
    if (desc->flags & HP_PERMISSIVE) return HP_OK;
    rc = plan_append(desc, new_ptr, total_new, workspace, workspace_bytes, nullptr, stream);
    if (rc) return rc;
    return sync_verdict(workspace, first_bad, stream);
}

HP_API int hp_copy_pages(void* page_pool, uint64_t num_pages, uint64_t page_bytes,
                         uint32_t index_type, const void* src_pages, const void* dst_pages,
                         uint64_t num_pairs, uint32_t flags, int* d_status, void* stream)
{
    if (index_type != HP_IDX_U32 && index_type != HP_IDX_U64) return HP_ERR_INDEX_TYPE;
    if (page_bytes == 0) return HP_ERR_ZERO_DIM;
    if (((u128)num_pages * page_bytes) >> 64) return HP_ERR_OVERFLOW;
    if (num_pairs && (!page_pool || !src_pages || !dst_pages)) return HP_ERR_NULL;
    if (misaligned(page_pool, 64) ||
        misaligned(src_pages, index_type == HP_IDX_U64 ? 8 : 4) ||
        misaligned(dst_pages, index_type == HP_IDX_U64 ? 8 : 4))
        return HP_ERR_ALIGN;
    int rc = reset_status(d_status, stream);
    if (rc || num_pairs == 0) return rc;
    hp::CopyArgs a{};
    a.num_pages = num_pages;
    a.src_pages = src_pages;
    a.dst_pages = dst_pages;
    a.lane_units = num_pairs;
    a.src = static_cast<const char*>(page_pool);
    a.dst = static_cast<char*>(page_pool);
    a.row_bytes = page_bytes;
    a.unit_bytes = host_memory(flags) ? std::min<u64>(page_bytes, kRegisterEngineUnit)
                                      : page_bytes;
    a.d_status = d_status;
    return hp::launch_copy(hp::kCopyPages, index_type == HP_IDX_U64, a,
                           pick_vec(page_bytes, page_pool, page_pool), stream);
}

HP_API int hp_zero_tails_scratch_bytes(const hp_paged_desc* desc, uint64_t* bytes)
{
    if (!desc || !bytes) return HP_ERR_NULL;
    if (desc->num_pages > (1ull << 61)) return HP_ERR_OVERFLOW;
    *bytes = 4 * desc->num_pages;
    return HP_OK;
}

HP_API int hp_zero_tails(const hp_paged_desc* desc, void* workspace, uint64_t workspace_bytes,
                         void* scratch, uint64_t scratch_bytes, int* d_status, void* stream)
{
    if (!desc) return HP_ERR_NULL;
    hp_paged_desc d = *desc;
    d.flags &= ~HP_PERMISSIVE;  // never zero through an unvalidated descriptor
    int rc = check_desc(&d);
    if (rc) return rc;
    if (d.page_size >= (1ull << 31)) return HP_ERR_ARG;  // counts keep bit 31 free
    if (!scratch || misaligned(scratch, 4) || scratch_bytes < 4 * d.num_pages)
        return HP_ERR_WORKSPACE;
    rc = check_ws(&d, workspace, workspace_bytes);
    if (rc) return rc;
    if (d.num_pages &&
        cudaMemsetAsync(scratch, 0, 4 * d.num_pages, static_cast<cudaStream_t>(stream)) !=
            cudaSuccess)
        return HP_ERR_CUDA;
    rc = plan_gather(&d, 0, workspace, workspace_bytes, d_status, stream, false);
    if (rc) return rc;
    hp::PlanArgs a = plan_args(&d, workspace, d_status);
    return hp::launch_zero_tails(d.index_type == HP_IDX_U64, a, static_cast<unsigned*>(scratch),
                                 row_bytes_of(&d), const_cast<void*>(d.page_pool), stream);
}

namespace {

// Decode attention: a step is TS tokens of one sequence for one K/V head, TS = min(32/G,
// 32/E) with E = head_dim/32 (the kernel's register budget); R step ranges per CTA.
u64 attn_step_tokens(u64 G, u64 D)
{
    const u64 E = D / 32;
    return (32 / G) < (32 / E) ? 32 / G : 32 / E;
}
uint32_t attn_ranges_per_cta(u64 Hkv) { return Hkv < 8 ? (uint32_t)(8 / Hkv) : 1u; }

// Head_dim 64 reaches the tensor-core kernel as pairs of K/V heads: two adjacent 64-dim
// heads are one 128-dim row of the pool, and each query, zero-padded to 128 dims in its own
// head's half, scores only its head's keys.  So an even K/V head count, and G <= 4 (the
// pairs have 2G query heads each).  Measured on GB300, 32 sequences of 1K-32K tokens: 8 K/V
// heads of G = 4 0.896 of the copy bandwidth in pairs against 0.704 on the CUDA cores, 16
// of G = 2 0.961 against 0.770.
bool attn_pairs(const hp_paged_desc* d, u64 G)
{
    return d->head_dim == 64 && d->num_heads % 2 == 0 && G <= 4;
}
// The K/V heads as the tensor-core kernel sees them, their query heads per head, and the
// heads of one launch: at most 8, with at most 32 query heads (larger counts run as groups
// of K/V heads, one launch each).
u64 attn_tc_heads(const hp_paged_desc* d, u64 G) { return attn_pairs(d, G) ? d->num_heads / 2 : d->num_heads; }
u64 attn_tc_g(const hp_paged_desc* d, u64 G) { return attn_pairs(d, G) ? 2 * G : G; }
u64 attn_tc_group(const hp_paged_desc* d, u64 G)
{
    u64 hg = attn_tc_heads(d, G);
    while (hg > 1 && (hg > 8 || hg * attn_tc_g(d, G) > 32)) hg /= 2;
    return hg;
}

// The tensor-core kernel serves head_dim 128 (and 64 in pairs) on device-memory pools with
// power-of-two K/V head counts, in launches of at most 8 K/V heads and 32 query heads, pages
// of 8 .. 128 / H_kv slots (H_kv of one launch; its steps are 128 (head, token) rows); by
// default head_dim 128 with G = 8 always (the CUDA-core kernel reaches 0.32-0.50 of the copy
// bandwidth there, the tensor-core one 0.53-0.90, and small batches are faster too), every
// other shape in at most two launches and only on batches with at least
// HP_ATTN_TC_MIN_STEPS such steps per SM (a quarter as many for long sequences).  The plan and the planned call decide alike, from
// the descriptor and the query heads alone.
bool attn_on_tensor_cores(const hp_paged_desc* d, u64 G)
{
    const u64 hkv = attn_tc_heads(d, G), hg = attn_tc_group(d, G);
    const u64 dim = attn_pairs(d, G) ? 128 : d->head_dim;
    if (hkv % hg || !hp::attention_tc_fits(dim, d->page_size, d->num_pages,
                                           (d->flags & HP_HOST_MEMORY) != 0, hg,
                                           hg * attn_tc_g(d, G)) ||
        (d->flags & HP_ATTN_CUDA_CORES) || d->num_seqs >= (1ull << 31))
        return false;  // (a sequence is a 32-bit tensor coordinate of the queries)
    if ((d->flags & HP_ATTN_TENSOR_CORES) || (G == 8 && !attn_pairs(d, G))) return true;
    // more than two launches cost more than they save unless G = 8 (measured: 32 K/V heads
    // of G = 2 in 4 groups 0.855 of the copy bandwidth against 0.895 on the CUDA cores)
    if (hkv / hg > 2) return false;
    int dev = 0;
    const int sms = hp::current_sms(&dev);
    if (sms == 0) return false;
    // HP_ATTN_TC_MIN_STEPS steps per SM, or a quarter of that when the sequences average
    // HP_ATTN_TC_LONG_TOKENS of capacity or more (measured on GB300, 32 sequences of 1K-32K
    // tokens: 4 K/V heads of G = 4, 103 steps per SM, 0.896 of the copy bandwidth on the
    // tensor cores against 0.808; 1 K/V head of G = 4, 26 per SM, 0.592 against 0.438;
    // head_dim 64 in pairs, 8 K/V heads of G = 4, 103 per SM, 0.858 against 0.687; but 256
    // sequences of 64-512 tokens, 31 per SM, 80 us against 76 on the CUDA cores)
    const u128 steps = (u128)d->table_len * d->page_size * hkv / 128;
    const u128 cap = d->num_seqs ? (u128)d->table_len * d->page_size / d->num_seqs : 0;
    const u128 min_steps =
        cap >= HP_ATTN_TC_LONG_TOKENS ? HP_ATTN_TC_MIN_STEPS / 4 : HP_ATTN_TC_MIN_STEPS;
    return steps >= min_steps * (u128)sms;
}

// Floats of one segment record's value sums: head_dim, or 128 for head_dim 64 (a record of
// the tensor-core kernel then holds a pair of heads).
u64 attn_record_dim(const hp_paged_desc* d) { return d->head_dim == 64 ? 128 : d->head_dim; }

// Segment records a batch can leave: worker v (of at most HP_ATTN_MAX_CTAS * R) writes
// record (s + v) * H_kv + g for each sequence s and head g it meets.
u64 attn_records(const hp_paged_desc* d)
{
    return (d->num_seqs + (u64)HP_ATTN_MAX_CTAS * attn_ranges_per_cta(d->num_heads)) * d->num_heads;
}

int attention_ws(const hp_paged_desc* d, uint32_t hq, u64* bytes)
{
    u64 plan = 0;
    int rc = ws_bytes(d, &plan);
    if (rc) return rc;
    const u128 part = (u128)attn_records(d) * (hq / d->num_heads) * (attn_record_dim(d) + 2) * 4;
    const u128 counts = (u128)d->num_seqs * d->num_heads * 4;
    // head_dim 64: the queries padded to 128 dims for the tensor-core kernel, 256-aligned
    const u128 qpad = d->head_dim == 64 ? (u128)d->num_seqs * hq * 256 + 256 : 0;
    if ((part + plan + counts + qpad) >> 64) return HP_ERR_OVERFLOW;
    *bytes = plan + (u64)part + (u64)counts + (u64)qpad;
    return HP_OK;
}

}  // namespace

HP_API int hp_attention_decode_workspace_bytes(const hp_paged_desc* k_desc, uint32_t num_q_heads,
                                               uint64_t* bytes)
{
    if (!k_desc || !bytes) return HP_ERR_NULL;
    return attention_ws(k_desc, num_q_heads, bytes);
}

namespace {

// Host checks shared by the attention entry points, on a strict copy of the descriptor:
// an attention reader always validates (it cannot skip rows it could not read).
struct AttnPrep {
    hp_paged_desc d;
    u64 G;
    char* part;          // the records, after the plan's workspace
    unsigned* seg_done;  // one count per (sequence, K/V head), after the records
    void* qpad;          // head_dim 64: the padded queries, after the counts (256-aligned)
};

int attention_prepare(const hp_paged_desc* k_desc, uint32_t num_q_heads, const void* workspace,
                      uint64_t workspace_bytes, AttnPrep* p)
{
    if (!k_desc) return HP_ERR_NULL;
    p->d = *k_desc;
    p->d.flags &= ~HP_PERMISSIVE;
    const hp_paged_desc* d = &p->d;
    int rc = check_desc(d);
    if (rc) return rc;
    if (d->dtype != HP_F16 && d->dtype != HP_BF16) return HP_ERR_DTYPE;
    if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256) return HP_ERR_ARG;
    if (num_q_heads == 0 || num_q_heads % d->num_heads) return HP_ERR_ARG;
    p->G = num_q_heads / d->num_heads;
    if (p->G != 1 && p->G != 2 && p->G != 4 && p->G != 8) return HP_ERR_ARG;
    if (d->page_size > (1u << 26)) return HP_ERR_ARG;  // offsets in a 32-page window fit 32 bits
    u64 need = 0;
    rc = attention_ws(d, num_q_heads, &need);
    if (rc) return rc;
    if (!workspace || misaligned(workspace, 256) || workspace_bytes < need) return HP_ERR_WORKSPACE;
    u64 plan_bytes = 0;
    ws_bytes(d, &plan_bytes);
    p->part = static_cast<char*>(const_cast<void*>(workspace)) + plan_bytes;
    p->seg_done =
        reinterpret_cast<unsigned*>(p->part + attn_records(d) * p->G * (attn_record_dim(d) + 2) * 4);
    const uintptr_t end = reinterpret_cast<uintptr_t>(p->seg_done + d->num_seqs * d->num_heads);
    p->qpad = reinterpret_cast<void*>((end + 255) & ~uintptr_t(255));
    return HP_OK;
}

}  // namespace

HP_API int hp_attention_plan(const hp_paged_desc* k_desc, uint32_t num_q_heads, void* workspace,
                             uint64_t workspace_bytes, int* d_status, void* stream)
{
    AttnPrep p;
    int rc = attention_prepare(k_desc, num_q_heads, workspace, workspace_bytes, &p);
    if (rc) return rc;
    const hp_paged_desc* d = &p.d;
    if (d->num_seqs && cudaMemsetAsync(p.seg_done, 0, 4 * d->num_seqs * d->num_heads,
                                       static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return HP_ERR_CUDA;
    hp::PlanArgs pa = plan_args(d, workspace, d_status);
    pa.step_tokens = attn_on_tensor_cores(d, p.G)
                         ? hp::attention_tc_step_tokens(attn_tc_group(d, p.G))
                         : attn_step_tokens(p.G, d->head_dim);
    return hp::launch_plan(hp::kPlanAttention, d->index_type == HP_IDX_U64, pa, stream);
}

HP_API int hp_attention_decode_planned(const hp_paged_desc* k_desc, const void* v_pool,
                                       const void* q, uint32_t num_q_heads, float scale,
                                       float* out, const void* workspace,
                                       uint64_t workspace_bytes, int* d_status, void* stream)
{
    AttnPrep p;
    int rc = attention_prepare(k_desc, num_q_heads, workspace, workspace_bytes, &p);
    if (rc) return rc;
    const hp_paged_desc* d = &p.d;
    if (d->num_seqs && (!q || !out)) return HP_ERR_NULL;
    if (d->num_pages && !v_pool) return HP_ERR_NULL;
    if (misaligned(v_pool, 64) || misaligned(q, 16) || misaligned(out, 16)) return HP_ERR_ALIGN;
    if (d->num_seqs == 0) return HP_OK;
    const hp::WsView ws = hp::ws_view(const_cast<void*>(workspace), d->num_seqs);
    hp::AttnArgs a{};
    a.k_pool = d->page_pool;
    a.v_pool = v_pool;
    a.q = q;
    a.table = d->block_table;
    a.seq_ptr = d->seq_ptr;
    a.lens = d->seq_lens;
    a.num_seqs = d->num_seqs;
    a.page_size = d->page_size;
    a.num_pages = d->num_pages;
    a.table_len = d->table_len;
    a.Hkv = (uint32_t)d->num_heads;
    a.Hq = num_q_heads;
    a.D = (uint32_t)d->head_dim;
    a.G = (uint32_t)p.G;
    hp::invariant_divisor(d->page_size, &a.p_m, &a.p_l);
    a.R = attn_ranges_per_cta(d->num_heads);
    a.scale = scale;
    a.hdr = ws.hdr;
    a.units_off = ws.units_off;
    a.part_acc = reinterpret_cast<float*>(p.part);
    a.part_ml = a.part_acc + attn_records(d) * p.G * attn_record_dim(d);
    a.seg_done = p.seg_done;
    a.out = out;
    a.elem_bf16 = d->dtype == HP_BF16;
    a.test_stall = (d->flags & HP_TEST_STALL) != 0;
    a.d_status = d_status;
    if (attn_on_tensor_cores(d, p.G)) {
        if (attn_pairs(d, p.G)) {
            // pairs of 64-dim heads as 128-dim heads: padded queries, half the heads, twice G
            rc = hp::launch_attention_qpad(q, p.qpad, d->num_seqs, num_q_heads, (uint32_t)p.G, stream);
            if (rc) return rc;
            a.q = p.qpad;
            a.Hkv = (uint32_t)(d->num_heads / 2);
            a.G = (uint32_t)(2 * p.G);
            a.D = 128;
            a.pair = 1;
        }
        // groups of K/V heads with at most 32 query heads, one launch each: the pool rows
        // and the query and output rows keep their full strides, the pointers move to the
        // group's first head (256 bytes of K or V per head; 128-dim queries; outD floats)
        const uint32_t hg = (uint32_t)attn_tc_group(d, p.G), groups = a.Hkv / hg;
        const uint64_t outD = a.pair ? 64 : 128;
        hp::AttnArgs ag = a;
        ag.Hkv_row = a.Hkv;
        ag.Hq_row = a.Hq;
        ag.Hkv = hg;
        ag.Hq = hg * a.G;
        for (uint32_t grp = 0; grp < groups; ++grp) {
            ag.k_pool = static_cast<const char*>(a.k_pool) + (u64)grp * hg * 256;
            ag.v_pool = static_cast<const char*>(a.v_pool) + (u64)grp * hg * 256;
            ag.q = static_cast<const char*>(a.q) + (u64)grp * ag.Hq * 256;
            ag.out = a.out + (u64)grp * ag.Hq * outD;
            rc = hp::launch_attention_tc(d->index_type == HP_IDX_U64, ag, stream);
            if (rc) return rc;
        }
        return HP_OK;
    }
    return hp::launch_attention(d->index_type == HP_IDX_U64, a, stream);
}

HP_API int hp_attention_decode(const hp_paged_desc* k_desc, const void* v_pool, const void* q,
                               uint32_t num_q_heads, float scale, float* out, void* workspace,
                               uint64_t workspace_bytes, int* d_status, void* stream)
{
    AttnPrep p;
    int rc = attention_prepare(k_desc, num_q_heads, workspace, workspace_bytes, &p);
    if (rc) return rc;
    const hp_paged_desc* d = &p.d;
    // every host check of the launch before anything is enqueued
    if (d->num_seqs && (!q || !out)) return HP_ERR_NULL;
    if (d->num_pages && !v_pool) return HP_ERR_NULL;
    if (misaligned(v_pool, 64) || misaligned(q, 16) || misaligned(out, 16)) return HP_ERR_ALIGN;
    rc = hp_attention_plan(k_desc, num_q_heads, workspace, workspace_bytes, d_status, stream);
    if (rc) return rc;
    return hp_attention_decode_planned(k_desc, v_pool, q, num_q_heads, scale, out, workspace,
                                       workspace_bytes, d_status, stream);
}

namespace {

int transpose(const void* src, void* dst, uint64_t nb, uint64_t bs, uint64_t H, uint64_t D,
              uint64_t x, uint32_t dtype, bool to_interchange, void* stream)
{
    const u64 es = elem_bytes(dtype);
    if (!es) return HP_ERR_DTYPE;
    if (!bs || !H || !D || !x) return HP_ERR_ZERO_DIM;
    if (D % x) return HP_ERR_ARG;
    if ((u128)bs * D * es > 48 * 1024) return HP_ERR_ARG;
    if (H >= (1ull << 31)) return HP_ERR_ARG;  // heads are counted in 32 bits on the device
    const u128 total = (u128)nb * bs * H * D * es;
    if (total >> 64) return HP_ERR_OVERFLOW;
    if (nb == 0) return HP_OK;
    if (!src || !dst) return HP_ERR_NULL;
    return hp::launch_transpose(src, dst, nb, bs, H, D, x, es, to_interchange, stream);
}

u64 table_ws_bytes(u64 batch) { return hp::kWsHeaderBytes + hp::round_up_256(8 * (batch + 1)); }

}  // namespace

HP_API int hp_from_kernel_layout(const void* src, void* dst, uint64_t num_blocks,
                                 uint64_t block_size, uint64_t num_heads, uint64_t head_dim,
                                 uint64_t x, uint32_t dtype, void* stream)
{
    return transpose(src, dst, num_blocks, block_size, num_heads, head_dim, x, dtype, true, stream);
}

HP_API int hp_to_kernel_layout(const void* src, void* dst, uint64_t num_blocks,
                               uint64_t block_size, uint64_t num_heads, uint64_t head_dim,
                               uint64_t x, uint32_t dtype, void* stream)
{
    return transpose(src, dst, num_blocks, block_size, num_heads, head_dim, x, dtype, false,
                     stream);
}

HP_API int hp_table_workspace_bytes(uint64_t batch, uint64_t* bytes)
{
    if (!bytes) return HP_ERR_NULL;
    if (batch >= (1ull << 58)) return HP_ERR_OVERFLOW;
    *bytes = table_ws_bytes(batch);
    return HP_OK;
}

HP_API int hp_padded_to_csr(const void* padded, const void* lens, uint64_t batch,
                            uint64_t max_blocks, uint64_t page_size, uint32_t index_type,
                            void* table_out, uint64_t table_cap, void* seq_ptr_out,
                            void* workspace, uint64_t workspace_bytes, int* d_status,
                            void* stream)
{
    if (index_type != HP_IDX_U32 && index_type != HP_IDX_U64) return HP_ERR_INDEX_TYPE;
    if (!page_size) return HP_ERR_ZERO_PAGE_SIZE;
    if (batch >= (1ull << 58) || ((u128)batch * max_blocks) >> 64) return HP_ERR_OVERFLOW;
    if (!seq_ptr_out || (batch && (!lens || (max_blocks && !padded))) || (table_cap && !table_out))
        return HP_ERR_NULL;
    if (!workspace || misaligned(workspace, 256) || workspace_bytes < table_ws_bytes(batch))
        return HP_ERR_WORKSPACE;
    hp::TableArgs t{};
    t.to_csr = true;
    t.in = padded;
    t.lens = lens;
    t.out = table_out;
    t.out2 = seq_ptr_out;
    t.batch = batch;
    t.max_blocks = max_blocks;
    t.page_size = page_size;
    t.cap = table_cap;
    t.workspace = workspace;
    t.d_status = d_status;
    return hp::launch_tables(index_type == HP_IDX_U64, t, stream);
}

HP_API int hp_csr_to_padded(const void* table, uint64_t table_len, const void* seq_ptr,
                            uint64_t batch, uint64_t max_blocks, uint64_t pad,
                            uint32_t index_type, void* padded_out, void* workspace,
                            uint64_t workspace_bytes, int* d_status, void* stream)
{
    if (index_type != HP_IDX_U32 && index_type != HP_IDX_U64) return HP_ERR_INDEX_TYPE;
    if (index_type == HP_IDX_U32 && pad > 0xFFFFFFFFull) return HP_ERR_ARG;
    if (batch >= (1ull << 58) || ((u128)batch * max_blocks) >> 64) return HP_ERR_OVERFLOW;
    if (!seq_ptr || (table_len && !table) || (batch && max_blocks && !padded_out))
        return HP_ERR_NULL;
    if (!workspace || misaligned(workspace, 256) || workspace_bytes < table_ws_bytes(batch))
        return HP_ERR_WORKSPACE;
    hp::TableArgs t{};
    t.to_csr = false;
    t.in = table;
    t.seq_ptr = seq_ptr;
    t.out = padded_out;
    t.batch = batch;
    t.max_blocks = max_blocks;
    t.table_len = table_len;
    t.pad = pad;
    t.workspace = workspace;
    t.d_status = d_status;
    return hp::launch_tables(index_type == HP_IDX_U64, t, stream);
}

HP_API int hp_lane_validate(uint64_t capacity, uint64_t page_tokens, const uint64_t* table,
                            uint64_t table_len, uint64_t* detail)
{
    uint64_t scratch[2];
    uint64_t* det = detail ? detail : scratch;
    det[0] = det[1] = 0;
    if (capacity == 0) return HP_ERR_ZERO_CAPACITY;
    if (page_tokens == 0) return HP_ERR_ZERO_PAGE_SIZE;
    const u64 pages = capacity / page_tokens + (capacity % page_tokens != 0);
    if (((u128)pages * page_tokens) >> 64) return HP_ERR_LANE_OVERFLOW;
    if (table_len != pages) {
        det[0] = pages;
        det[1] = table_len;
        return HP_ERR_PAGE_COUNT;
    }
    if (pages && !table) return HP_ERR_NULL;
    std::vector<unsigned char> seen;
    try {
        seen.assign(pages, 0);
    } catch (...) {
        return HP_ERR_ALLOCATION_FAILED;
    }
    for (u64 q = 0; q < pages; ++q) {
        const u64 p = table[q];
        if (p >= pages) {
            det[0] = q;
            det[1] = p;
            return HP_ERR_PHYSICAL_PAGE;
        }
        if (seen[p]) {
            det[0] = p;
            return HP_ERR_ALIASED_PAGE;
        }
        seen[p] = 1;
    }
    return HP_OK;
}

HP_API int hp_lane_gather(const void* pool, const uint64_t* table, uint64_t capacity,
                          uint64_t page_tokens, uint64_t batch, uint64_t kv_heads, uint64_t width,
                          uint32_t dtype, uint64_t n, void* out, uint32_t flags, int* d_status,
                          void* stream)
{
    u64 pages = 0, rb = 0;
    int rc = check_lane(pool, table, capacity, page_tokens, batch, kv_heads, width, dtype, &pages,
                        &rb);
    if (rc) return rc;
    if (n > capacity) return HP_ERR_LENGTH;
    if (n && !out) return HP_ERR_NULL;
    rc = reset_status(d_status, stream);
    if (rc || n == 0) return rc;
    hp::CopyArgs a{};
    a.table = table;
    a.num_pages = pages;
    a.page_size = page_tokens;
    a.lanes = batch * kv_heads;
    a.lane_n = n;
    a.lane_pages = n / page_tokens + (n % page_tokens != 0);
    a.lane_first_page = 0;
    a.lane_units = a.lanes * a.lane_pages;
    a.src = static_cast<const char*>(pool);
    a.dst = static_cast<char*>(out);
    a.row_bytes = rb;
    a.unit_bytes = page_tokens * rb;
    if (host_memory(flags)) a.unit_bytes = std::min<u64>(a.unit_bytes, kRegisterEngineUnit);
    a.d_status = d_status;
    return hp::launch_copy(hp::kLaneGather, 1, a, pick_vec(rb, pool, out), stream);
}

HP_API int hp_lane_append(void* pool, const uint64_t* table, uint64_t capacity,
                          uint64_t page_tokens, uint64_t batch, uint64_t kv_heads, uint64_t width,
                          uint32_t dtype, uint64_t n, uint64_t m, const void* new_rows,
                          uint32_t flags, int* d_status, void* stream)
{
    u64 pages = 0, rb = 0;
    int rc = check_lane(pool, table, capacity, page_tokens, batch, kv_heads, width, dtype, &pages,
                        &rb);
    if (rc) return rc;
    if (n > capacity || m > capacity - n) return HP_ERR_LENGTH;
    if (m && !new_rows) return HP_ERR_NULL;
    rc = reset_status(d_status, stream);
    if (rc || m == 0) return rc;
    hp::CopyArgs a{};
    a.table = table;
    a.num_pages = pages;
    a.page_size = page_tokens;
    a.lanes = batch * kv_heads;
    a.lane_n = n;
    a.lane_m = m;
    a.lane_first_page = n / page_tokens;
    a.lane_pages = (n + m - 1) / page_tokens - n / page_tokens + 1;
    a.lane_units = a.lanes * a.lane_pages;
    a.src = static_cast<const char*>(new_rows);
    a.dst = static_cast<char*>(pool);
    a.row_bytes = rb;
    a.unit_bytes = page_tokens * rb;
    if (host_memory(flags)) a.unit_bytes = std::min<u64>(a.unit_bytes, kRegisterEngineUnit);
    a.d_status = d_status;
    return hp::launch_copy(hp::kLaneAppend, 1, a, pick_vec(rb, new_rows, pool), stream);
}
