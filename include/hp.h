/*
 * hp.h -- C ABI of the block-paged KV-cache library (libhp.so) for GB300 (sm_103a).
 *
 * The library implements the data path of the block-paged layout defined in
 * "Block-Paged Layout -- Hurray Format Specification" (cited below as [HF]), of the
 * per-lane page layout in "Keep token order across cache pages"
 * (practical-ch20-paged-kv-layout, cited as [CH]) and of the block-table reader and
 * copy-on-write of "Visualize PagedAttention block layout" (cited as [VA]):
 *
 *   - a planner/validator for a block-paged descriptor,
 *   - a gather of a ragged batch into the logical [total_tokens, H, D] tensor,
 *   - the inverse scatter that appends new K/V rows into their pages,
 *   - a dequantising gather of an 8-bit pool with per-page-slot fp32 scales, and
 *     under the other schemes of [HF] Per-scheme composition (per tensor, per
 *     channel, per block, with or without zero points),
 *   - gather and append for the [N, B, H_kv, P, d] per-lane layout,
 *   - the writer side: a batched page copy (copy-on-write) and the zeroing of the
 *     slots no sequence reads,
 *   - decode attention that reads K and V through the block table,
 *   - conversions between a kernel-internal cache layout and the interchange layout,
 *     and between a padded block table and the descriptor's slices.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All functions return an int status: HP_OK (0) or a negative hp_status code.
 *   hp_status_string() names it.  Nothing aborts or prints.
 * - Pointers named d_* or described as "device" point to GPU memory of the
 *   current CUDA device; pointers described as "host" point to CPU memory.
 *   The page pool and the output of the gathers (dequantising ones included), the
 *   pool and new rows of the appends, the pool of hp_copy_pages, the buffers of the
 *   lane operations and the K and V pools of decode attention may instead be
 *   page-locked host memory (from the CUDA host allocator or cudaHostRegister,
 *   mapped): those operations then read and write it in place over the host link.
 *   The caller says so with HP_HOST_MEMORY (the copies then take the register
 *   engine); the library never asks the runtime where a pointer lives.  Index
 *   buffers, workspaces, status words and the other operations' buffers are device
 *   memory.
 *   The caller owns every buffer.  The library allocates no device memory; the
 *   only state it keeps between calls is a per-device cache of launch facts (SM
 *   count, resident CTAs per kernel), filled on first use.  It is safe to call from
 *   several host threads on different streams.
 * - `stream` is a cudaStream_t passed as void*; NULL means the legacy default
 *   stream.  Functions marked ASYNC only enqueue work on `stream` and return
 *   once it is enqueued; functions marked SYNC wait for their own work.
 * - Errors the host can see (bad descriptor fields, null or misaligned
 *   pointers, a short workspace) are returned before anything is enqueued and
 *   leave every output untouched.  Errors that depend on device-resident data
 *   (seq_ptr, block_table, token counts) are found on the device: the ASYNC
 *   operations then write nothing to their outputs and store the status code
 *   in *d_status (an optional caller-owned device int).  When d_status is
 *   non-NULL the operation first stores HP_OK there, then the first error
 *   found, if any.  In permissive mode (HP_PERMISSIVE) the storage invariants
 *   are not validated; a row whose lookup would leave its slice, the table or
 *   the pool is then skipped (its output row is left as it was) and one of the
 *   codes of the skipped rows is stored in *d_status.  No device code traps,
 *   asserts or waits on another agent.
 * - Launch errors reported by the CUDA runtime map to HP_ERR_CUDA.
 */
#ifndef HP_H
#define HP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ status */
typedef enum hp_status {
    HP_OK = 0,
    /* structural descriptor checks, always made on the host, in this order */
    HP_ERR_RANK = -1,           /* [HF] Description: rank is not 3                          */
    HP_ERR_PAGED_AXIS = -2,     /* [HF] Logical Shape, invariant (6): paged_axis is not 0    */
    HP_ERR_SHARD = -3,          /* [HF] Sharding: a shard descriptor is attached              */
    HP_ERR_INDEX_TYPE = -4,     /* [HF] Additional Descriptor Fields: index type not 0x00/0x01,
                                   or uint32 with more than 2^32 pages / 2^32-1 table entries */
    HP_ERR_DTYPE = -5,          /* unknown element type (or not int8 for a dequantising gather) */
    HP_ERR_ZERO_DIM = -6,       /* page_size, num_heads or head_dim is 0                      */
    HP_ERR_SCALES = -7,         /* [HF] Scale-buffer size: HP_HAS_QUANT without
                                   num_pages*page_size fp32 scales                            */
    HP_ERR_NULL = -8,           /* a required buffer pointer is NULL                          */
    HP_ERR_ALIGN = -9,          /* [HF] Alignment: a descriptor buffer is not 64-byte aligned  */
    HP_ERR_OVERFLOW = -10,      /* [HF] invariant (4): the pool's byte size exceeds 2^64      */
    /* storage invariants, checked on the device, in this order */
    HP_ERR_SEQ_PTR_START = -11, /* [HF] invariant (1): seq_ptr[0] != 0                        */
    HP_ERR_SEQ_PTR_ORDER = -12, /* [HF] invariant (2): seq_ptr[s] > seq_ptr[s+1]               */
    HP_ERR_SEQ_PTR_END = -13,   /* [HF] invariant (1): seq_ptr[num_seqs] != table_len          */
    HP_ERR_PAGE_ID = -14,       /* [HF] invariant (3): block_table[k] >= num_pages             */
    HP_ERR_LEN = -15,           /* [HF] Partial trailing page: seq_lens[s] exceeds the slots of
                                   the sequence's slice, (seq_ptr[s+1]-seq_ptr[s])*page_size   */
    /* append checks, after the storage invariants */
    HP_ERR_NEW_PTR_START = -16, /* new_ptr[0] != 0                                            */
    HP_ERR_NEW_PTR_ORDER = -17, /* new_ptr[s] > new_ptr[s+1]                                  */
    HP_ERR_NEW_PTR_END = -18,   /* new_ptr[num_seqs] != total_new                             */
    HP_ERR_CAPACITY = -19,      /* seq_lens[s] + new rows exceed the slice's slots            */
    /* argument checks */
    HP_ERR_OUT_SIZE = -20,      /* out_tokens != sum of seq_lens (or the sum exceeds 2^64)     */
    /* per-lane layout, [CH] PagedKvLayout::new and the live length */
    HP_ERR_ZERO_CAPACITY = -21,
    HP_ERR_ZERO_PAGE_SIZE = -22,
    HP_ERR_LANE_OVERFLOW = -23, /* ceil(C/P)*P or a buffer size exceeds 2^64                  */
    HP_ERR_PAGE_COUNT = -24,    /* table length != ceil(C/P)                                  */
    HP_ERR_PHYSICAL_PAGE = -25, /* a table entry >= ceil(C/P)                                 */
    HP_ERR_ALIASED_PAGE = -26,  /* a table entry repeats                                      */
    HP_ERR_LENGTH = -27,        /* live length (plus appended rows) exceeds the capacity      */
    HP_ERR_ALLOCATION_FAILED = -28, /* host scratch for the lane table check unavailable     */
    /* library */
    HP_ERR_WORKSPACE = -29,     /* workspace NULL, misaligned (256 B) or smaller than required */
    HP_ERR_ARG = -30,           /* another argument is invalid (see the function)            */
    HP_ERR_CUDA = -31,          /* the CUDA runtime rejected a launch or a copy               */
    HP_ERR_TIMEOUT = -32,       /* a kernel's bounded wait for its own asynchronous copies ran
                                   out (about 2 s); its output is incomplete                   */
    HP_ERR_NOALLOC_LIMIT = -33, /* hp_gather_noalloc: more than HP_NOALLOC_MAX_SEQS sequences */
    HP_ERR_QUANT_SCHEME = -34,  /* unknown scheme tag, or per-channel on an axis other than
                                   1 (num_heads) or 2 (head_dim)                             */
    HP_ERR_QUANT_BLOCK = -35    /* [HF] Per-scheme composition: per-block-affine whose axis is
                                   not 0 or whose block_size is not page_size                */
} hp_status;

/* Name of a status code ("HP_OK", "HP_ERR_RANK", ...); "HP_ERR_UNKNOWN" otherwise. */
const char* hp_status_string(int status);

/* --------------------------------------------------------------- descriptor */
typedef enum hp_dtype {     /* element type of the page pool */
    HP_F32 = 0, HP_F16 = 1, HP_BF16 = 2, HP_I8 = 3, HP_U8 = 4, HP_F64 = 5
} hp_dtype;

typedef enum hp_index_type { /* [HF] block_table_index_type; also the type of seq_ptr,
                                seq_lens and an append's new_ptr */
    HP_IDX_U32 = 0x00, HP_IDX_U64 = 0x01
} hp_index_type;

#define HP_PERMISSIVE 0x1u /* [HF] Storage Invariants: a reader in permissive mode does not
                              reject descriptors that violate invariants (1)-(3)          */
#define HP_HAS_QUANT 0x2u  /* [HF] Buffer Table: quantisation parameters present          */
/* Memory placement (no counterpart in the pages, which describe device buffers): the page
 * pool, the output or the new rows of the call may lie in page-locked host memory that
 * the GPU reaches directly (cudaHostAlloc'd or cudaHostRegister'ed memory, e.g. a pool
 * offloaded to Grace memory).  The copy then runs on the register engine, with ordinary
 * loads and stores over the host link.  Without the flag every buffer must be device
 * memory: the library asks the runtime nothing about a pointer, and its TMA engine is for
 * device memory only.  In the descriptor's `flags`, and in the `flags` argument of
 * hp_copy_pages, hp_lane_gather and hp_lane_append. */
#define HP_HOST_MEMORY 0x4u
/* Decode attention's kernel (no counterpart in the pages).  By default the library picks
 * the tensor-core kernel when the shape allows it -- head_dim 128, or 64 in pairs of K/V
 * heads (see hp_attention_decode); a power-of-two number of K/V heads; G = num_q_heads /
 * num_heads in {1, 2, 4, 8}; pages of a power of two from 8 to 128 / h slots, h the K/V
 * heads of one launch (at most 8, with at most 32 query heads; more K/V heads run as groups
 * of h, one launch each); device memory -- and either G = 8 at head_dim 128, or the batch
 * takes at most two launches and has at least HP_ATTN_TC_MIN_STEPS steps of 128 (head,
 * token) rows per SM (table_len * page_size * num_heads / 128 / SMs, pairs counting as
 * heads for head_dim 64), a quarter of that when its sequences average
 * HP_ATTN_TC_LONG_TOKENS slots of capacity (table_len * page_size / num_seqs) or more.
 * Otherwise the CUDA-core kernel.  (Measured on GB300: the tensor-core kernel is the faster on batches
 * of that size and at G = 8, the CUDA-core one on batches of few, short sequences.)
 * HP_ATTN_TENSOR_CORES asks for the tensor-core kernel wherever the shape allows it,
 * HP_ATTN_CUDA_CORES for the CUDA-core kernel always.  The plan and the planned calls that
 * follow it must carry the same flags. */
#define HP_ATTN_TENSOR_CORES 0x8u
#define HP_ATTN_CUDA_CORES 0x10u
#define HP_ATTN_TC_MIN_STEPS 32
#define HP_ATTN_TC_LONG_TOKENS 2048
/* Test hook for the bounded waits (no counterpart in the pages): the TMA copy engine sets
 * up the first load of each of its CTAs but never issues it, so the wait for it runs out
 * (after about 2 s), the call stores HP_ERR_TIMEOUT in *d_status and returns without
 * copying the rest.  Only a gather that takes the TMA engine (16-byte rows and bases,
 * copy units of 16 KiB or more, a batch too large for the one-launch path) sees it, and
 * decode attention on the tensor cores, whose K loaders arm their first step's loads
 * without issuing them (every role's waits then run out, the call stores HP_ERR_TIMEOUT
 * and the output is undefined); never set it outside tests. */
#define HP_TEST_STALL 0x100u

/*
 * A block-paged descriptor ([HF] Buffer Table, Additional Descriptor Fields):
 * one batch of one {kv_role, layer_index}, a static snapshot.
 *
 *   page_pool    device, [num_pages, page_size, num_heads, head_dim] elements of
 *                `dtype`, row-major; num_pages*page_size*num_heads*head_dim*width
 *                bytes ([HF] invariant (4)).  Written only by hp_scatter_append and
 *                hp_zero_tails (hp_copy_pages takes its pool as an argument of its own).
 *   block_table  device, table_len entries of the index type: physical page IDs,
 *                the per-sequence slices concatenated.  May be NULL iff
 *                table_len == 0 ([HF] Buffer Table, empty batch).
 *   seq_ptr      device, num_seqs+1 entries: sequence s owns block_table
 *                [seq_ptr[s], seq_ptr[s+1]) ([HF] Description, CSR-style).
 *   seq_lens     device, num_seqs entries: the token count of each sequence (the
 *                count that bounds a reader, [HF] Partial trailing page).  May be
 *                NULL iff num_seqs == 0.
 *   scales       device, scales_len fp32 per-page-slot scales, required iff
 *                flags has HP_HAS_QUANT; scales_len must be num_pages*page_size
 *                ([HF] Per-page-slot parameters, Scale-buffer size).
 *
 * Every present buffer must be 64-byte aligned ([HF] Alignment).
 * rank must be 3, paged_axis 0 and has_shard 0 ([HF] Description, Logical
 * Shape, Sharding).  Aliased page IDs (prefix sharing) are allowed and never
 * checked ([HF] Prefix Sharing).
 */
typedef struct hp_paged_desc {
    uint32_t rank;
    uint32_t paged_axis;
    uint32_t has_shard;
    uint32_t flags;        /* HP_PERMISSIVE | HP_HAS_QUANT | HP_HOST_MEMORY
                              (| HP_TEST_STALL in tests) */
    uint32_t dtype;        /* hp_dtype */
    uint32_t index_type;   /* hp_index_type */
    uint64_t num_pages;
    uint64_t page_size;
    uint64_t num_heads;
    uint64_t head_dim;
    uint64_t num_seqs;
    uint64_t table_len;
    uint64_t scales_len;
    const void* page_pool;
    const void* block_table;
    const void* seq_ptr;
    const void* seq_lens;
    const float* scales;
} hp_paged_desc;

/* ----------------------------------------------------------------- planning */
/*
 * Bytes of device workspace the planned operations need for `desc`
 * (256 + 2 * 256-rounded 8*(num_seqs+1)).  Host only; no GPU work.
 * The workspace must be 256-byte aligned.  Returns HP_ERR_NULL if an argument
 * is NULL, HP_ERR_OVERFLOW if the size does not fit in 64 bits.
 */
int hp_workspace_bytes(const hp_paged_desc* desc, uint64_t* bytes);

/*
 * SYNC.  Validate a block-paged descriptor the way a conforming reader does
 * ([HF] Storage Invariants): the structural checks on the host, then -- unless
 * HP_PERMISSIVE -- invariants (1)-(3) and the token-count rule on the device
 * (one pass over seq_ptr/seq_lens and one over block_table), with the first
 * failing rule in the order of hp_status and, within it, the first failing
 * index.  Returns that rule's code (HP_OK if none) and stores the index in
 * *first_bad (host, may be NULL; 0 for structural errors).  Uses `workspace`
 * (hp_workspace_bytes) as scratch.  Waits for `stream`.
 */
int hp_validate(const hp_paged_desc* desc, void* workspace, uint64_t workspace_bytes,
                uint64_t* first_bad, void* stream);

/*
 * ASYNC.  Plan a gather: validate as hp_validate does (without waiting), check
 * that out_tokens equals the sum of seq_lens ([HF] Logical Shape: total_tokens
 * is that sum), and store in `workspace` the exclusive prefix sums of the token
 * counts (each sequence's first output row) and of ceil(seq_lens[s]/page_size)
 * (each sequence's first page span).  hp_gather_planned and
 * hp_gather_dequant_planned consume the workspace, in stream order.
 */
int hp_plan(const hp_paged_desc* desc, uint64_t out_tokens, void* workspace,
            uint64_t workspace_bytes, int* d_status, void* stream);

/* ------------------------------------------------------------------- gather */
/*
 * ASYNC.  Gather the ragged batch into `out` (device, out_tokens rows of
 * num_heads*head_dim elements of desc->dtype, row-major): row tok_off[s]+t holds
 * token t of sequence s for t < seq_lens[s], element (h, d) of it being
 * page_pool[((phys*page_size + t % page_size)*num_heads + h)*head_dim + d] with
 * phys = block_table[seq_ptr[s] + t / page_size] ([HF] Element Lookup).
 * Elements are copied as bytes.  No slot past a sequence's token count is read
 * ([HF] Partial trailing page).  Equivalent to hp_plan then hp_gather_planned
 * (same verdicts, same workspace contents); a validated batch of at most 1024
 * sequences, 8192 table entries and 8 MiB of pages runs as a single kernel.
 * `out` must be 16-byte aligned for the vector path (any alignment works).
 */
int hp_gather(const hp_paged_desc* desc, void* out, uint64_t out_tokens, void* workspace,
              uint64_t workspace_bytes, int* d_status, void* stream);

/* ASYNC.  The copy step of hp_gather, for a workspace hp_plan filled earlier on the same
 * stream with the same descriptor -- or one that differs only in page_pool (the plan
 * reads no page, so one plan serves the pools of every layer that shares the table,
 * offsets and counts).  Does nothing if that plan failed. */
int hp_gather_planned(const hp_paged_desc* desc, void* out, const void* workspace,
                      int* d_status, void* stream);

/*
 * ASYNC.  Dequantising gather of an int8 pool (desc->dtype == HP_I8, flags with
 * HP_HAS_QUANT): like hp_gather, but element (h, d) of token t of sequence s is
 * the bfloat16 nearest (ties to even) to the exact product
 * value * scales[phys*page_size + t % page_size] ([HF] Element Lookup, quantized
 * case; Per-page-slot parameters; a symmetric scheme, no zero point).
 * `out_bf16` (device) holds out_tokens rows of num_heads*head_dim bfloat16.
 */
int hp_gather_dequant(const hp_paged_desc* desc, void* out_bf16, uint64_t out_tokens,
                      void* workspace, uint64_t workspace_bytes, int* d_status, void* stream);

/* ASYNC.  The copy step of hp_gather_dequant, after hp_plan on the same stream. */
int hp_gather_dequant_planned(const hp_paged_desc* desc, void* out_bf16, const void* workspace,
                              int* d_status, void* stream);

/* ------------------------------------------------------ quantization schemes */
/*
 * [HF] Quantization Compatibility, Per-scheme composition: how a quantization scheme
 * composes with the paged structure.
 *   HP_QUANT_PER_TENSOR (0x01)        one scale (and zero point) for the whole tensor;
 *   HP_QUANT_PER_CHANNEL (0x02)       one per channel along axis 1 (num_heads) or 2
 *                                     (head_dim), independent of the pages; axis 0 is
 *                                     rejected (a writer must not quantize the paged axis
 *                                     per channel);
 *   HP_QUANT_PER_BLOCK_AFFINE (0x03)  only with axis 0 and block_size == page_size, where
 *                                     its blocks are the page slots: scale of page p, slot i
 *                                     at p*page_size + i ([HF] Per-page-slot parameters);
 *                                     any other axis or block size is rejected.
 * The value of element (s, t, h, d) is the bfloat16 nearest (ties to even) to the exact
 * (q - zero_point) * scale, where q is the pool element the Element Lookup names and the
 * scale and zero point are the entries the scheme assigns it; zero_points == NULL is the
 * symmetric case (zero point 0).  The affine form (q - zero_point) * scale is this
 * library's reading of the scheme bodies, which the specification keeps in a separate
 * document.
 */
typedef enum hp_quant_scheme {
    HP_QUANT_PER_TENSOR = 0x01,
    HP_QUANT_PER_CHANNEL = 0x02,
    HP_QUANT_PER_BLOCK_AFFINE = 0x03
} hp_quant_scheme;

typedef struct hp_quant_desc {
    uint32_t scheme_tag;      /* hp_quant_scheme */
    uint32_t axis;            /* per-channel: 1 or 2; per-block-affine: must be 0 */
    uint64_t block_size;      /* per-block-affine: must equal page_size */
    uint64_t count;           /* entries in scales (and zero_points): 1, num_heads or
                                 head_dim, or num_pages*page_size ([HF] Scale-buffer size) */
    const float* scales;      /* device, fp32, 64-byte aligned */
    const void* zero_points;  /* device, `count` entries of the pool's element type (int8 or
                                 uint8), 64-byte aligned; NULL for a symmetric scheme */
} hp_quant_desc;

/*
 * ASYNC.  Dequantising gather under an explicit scheme.  desc->dtype must be HP_I8 or
 * HP_U8; the parameters come from `quant` (desc->flags' HP_HAS_QUANT, desc->scales and
 * desc->scales_len are not used).  Host checks, in order: quant NULL (HP_ERR_NULL),
 * element type (HP_ERR_DTYPE), scheme tag and per-channel axis (HP_ERR_QUANT_SCHEME),
 * per-block-affine axis and block size (HP_ERR_QUANT_BLOCK), count (HP_ERR_SCALES),
 * NULL scales (HP_ERR_NULL), alignment (HP_ERR_ALIGN); then as hp_gather_dequant.
 * `out_bf16` holds out_tokens rows of num_heads*head_dim bfloat16.
 */
int hp_gather_dequant_q(const hp_paged_desc* desc, const hp_quant_desc* quant, void* out_bf16,
                        uint64_t out_tokens, void* workspace, uint64_t workspace_bytes,
                        int* d_status, void* stream);

/* ASYNC.  The copy step of hp_gather_dequant_q, after hp_plan on the same stream. */
int hp_gather_dequant_q_planned(const hp_paged_desc* desc, const hp_quant_desc* quant,
                                void* out_bf16, const void* workspace, int* d_status,
                                void* stream);

/* ------------------------------------------------------------------- append */
/*
 * ASYNC.  Append new K (or V) rows to their sequences: new row new_ptr[s]+i of
 * `new_rows` (device, total_new rows of num_heads*head_dim elements of
 * desc->dtype) becomes token t = seq_lens[s] + i of sequence s, written to the
 * pool slot the Element Lookup names for t ([HF] Element Lookup, used as a
 * store).  desc->seq_lens holds the counts BEFORE the append; the library does
 * not update them.  new_ptr (device, num_seqs+1 entries of the index type) is a
 * CSR offset array over the new rows.  Validation (device, unless permissive):
 * the storage invariants, then new_ptr[0] = 0, non-decreasing,
 * new_ptr[num_seqs] = total_new, then seq_lens[s] + rows of s <= the slice's
 * slots.  Rows whose targets alias (two sequences naming one page and slot)
 * land in an unspecified order.  `new_rows` must be 16-byte aligned for the
 * vector path.  With HP_PERMISSIVE the caller vouches for the descriptor: nothing is
 * validated up front, a row whose logical page lies outside its slice or the table is
 * skipped with HP_ERR_LEN in *d_status, one naming a page outside the pool with
 * HP_ERR_PAGE_ID; a sequence whose pair new_ptr[s] .. new_ptr[s+1] runs backwards or
 * ends past total_new appends nothing (HP_ERR_NEW_PTR_ORDER / HP_ERR_NEW_PTR_END), so
 * no row outside the total_new rows of `new_rows` is ever read, in either mode.  An
 * append of fewer than num_seqs*page_size rows (a decode step)
 * runs as one kernel with one warp per sequence (after the plan when validated).
 */
int hp_scatter_append(const hp_paged_desc* desc, const void* new_rows, const void* new_ptr,
                      uint64_t total_new, void* workspace, uint64_t workspace_bytes,
                      int* d_status, void* stream);

/* ASYNC.  The validation and planning step of hp_scatter_append. */
int hp_append_plan(const hp_paged_desc* desc, const void* new_ptr, uint64_t total_new,
                   void* workspace, uint64_t workspace_bytes, int* d_status, void* stream);

/* ASYNC.  The copy step of hp_scatter_append, after hp_append_plan (with the same
 * new_ptr and total_new, and a descriptor that differs at most in page_pool) on the same
 * stream; one plan serves every layer's pool.  Does nothing if that plan failed. */
int hp_scatter_append_planned(const hp_paged_desc* desc, const void* new_rows,
                              const void* new_ptr, uint64_t total_new, const void* workspace,
                              int* d_status, void* stream);

/* SYNC.  The verdict hp_append_plan reaches, returned like hp_validate's. */
int hp_validate_append(const hp_paged_desc* desc, const void* new_ptr, uint64_t total_new,
                       void* workspace, uint64_t workspace_bytes, uint64_t* first_bad,
                       void* stream);

/* ---------------------------------------------------------------- writer side */
/*
 * ASYNC.  Copy-on-write page copy ([VA] "Copy-on-write for beam search and prefix
 * sharing": a shared block is copied when one request is about to modify it).  For every
 * i < num_pairs, page dst_pages[i] of `page_pool` (device, num_pages pages of page_bytes
 * bytes) becomes a byte copy of page src_pages[i].  src_pages and dst_pages are device
 * arrays of num_pairs entries of `index_type` (HP_IDX_U32 / HP_IDX_U64).  A pair naming a
 * page >= num_pages copies nothing and stores HP_ERR_PAGE_ID in *d_status.  Destination
 * pages must differ from each other and from every source page (the result is otherwise
 * unspecified).  page_pool must be 64-byte aligned.  flags: 0, or HP_HOST_MEMORY when
 * page_pool is page-locked host memory.
 */
int hp_copy_pages(void* page_pool, uint64_t num_pages, uint64_t page_bytes, uint32_t index_type,
                  const void* src_pages, const void* dst_pages, uint64_t num_pairs,
                  uint32_t flags, int* d_status, void* stream);

/* Bytes of scratch hp_zero_tails needs for `desc`: one 32-bit word per page. */
int hp_zero_tails_scratch_bytes(const hp_paged_desc* desc, uint64_t* bytes);

/*
 * ASYNC.  The writer's duty of [HF] Partial trailing page before the cache crosses a trust
 * or tenant boundary: zero the slots no sequence of the batch reads.  For every page the
 * slices name, the slots past the largest count any referencing sequence keeps in it are
 * set to zero bytes (a page shared by several sequences keeps what the longest of them
 * uses, [HF] Prefix Sharing); pages no slice names are not touched.  The descriptor is
 * always validated as hp_validate does (HP_PERMISSIVE is ignored here: zeroing through an
 * invalid descriptor could destroy live rows); on a violation nothing is written and the
 * rule's code goes to *d_status.  `workspace` is the plan's (hp_workspace_bytes);
 * `scratch` (device, 4-byte aligned) holds hp_zero_tails_scratch_bytes bytes.  Writes the
 * page pool.
 */
int hp_zero_tails(const hp_paged_desc* desc, void* workspace, uint64_t workspace_bytes,
                  void* scratch, uint64_t scratch_bytes, int* d_status, void* stream);

/* ---------------------------------------------------------- decode attention */
/*
 * Bytes of device workspace hp_attention_decode needs: the plan's (hp_workspace_bytes)
 * plus fp32 records (max, sum and head_dim accumulators per query head; 128 accumulators
 * for head_dim 64) for up to (num_seqs + HP_ATTN_MAX_CTAS * R) * num_heads sequence
 * segments, R = 8 / num_heads when num_heads < 8, else 1, plus a 4-byte count per
 * (sequence, K/V head), plus for head_dim 64 the queries padded to 128 dims (256 bytes per
 * query head, 256-aligned).  It depends only on the descriptor's num_seqs, num_heads and
 * head_dim, and on num_q_heads.
 */
#define HP_ATTN_MAX_CTAS 512
int hp_attention_decode_workspace_bytes(const hp_paged_desc* k_desc, uint32_t num_q_heads,
                                        uint64_t* bytes);

/*
 * ASYNC.  Decode attention over the block-paged cache -- the consumer of the block table
 * in [VA] "How the attention kernel uses the block table".  For every sequence s and query
 * head qh (of num_q_heads; K/V head g = qh / (num_q_heads / num_heads), grouped-query
 * sharing): score_t = scale * sum_d q[s, qh, d] * K(s, t, g, d) for t < seq_lens[s],
 * weights = softmax over t, out[s, qh, d] = sum_t weight_t * V(s, t, g, d), where K comes
 * from k_desc's pool and V from `v_pool` (same geometry, table, offsets and counts), both
 * read through the Element Lookup ([HF]).  q (device, [num_seqs, num_q_heads, head_dim])
 * has the pool's element type (HP_F16 or HP_BF16); out (device, fp32, same shape) gets 0
 * for a sequence with no tokens.  Arithmetic is fp32.  Supported: head_dim 64, 128 or
 * 256, num_q_heads / num_heads in {1, 2, 4, 8}, page_size <= 2^26 (HP_ERR_ARG otherwise).
 * With head_dim 128, a power-of-two number of K/V heads (more than 8, or more than 32
 * query heads, in groups of K/V heads, one launch each), pages of 8 to 128 / h slots (h the
 * K/V heads of one launch) and both pools in device memory the scores and the weighted value
 * sums may run on the tensor cores (products of the 16-bit inputs accumulated in fp32; the
 * weights as two 16-bit parts, so the result stays within about 2^-16 of max|V| of the
 * fp32 one); so may head_dim 64 with an even, power-of-two number of K/V heads and
 * num_q_heads / num_heads <= 4, taken as pairs of K/V heads (two adjacent 64-dim heads as
 * one 128-dim row, each query zero-padded to 128 dims in its own head's half; h then counts
 * pairs); otherwise on the CUDA cores in fp32 --
 * see HP_ATTN_TENSOR_CORES for the choice.  K and V pools in page-locked host memory need
 * HP_HOST_MEMORY in k_desc's flags (they are then read in place over the host link by the
 * CUDA-core kernel).
 * The descriptor is always validated as hp_plan validates a strict one: HP_PERMISSIVE
 * is ignored, because an attention reader cannot skip the rows it could not read -- a
 * descriptor that fails a rule gets that rule's code in *d_status and no output.
 */
int hp_attention_decode(const hp_paged_desc* k_desc, const void* v_pool, const void* q,
                        uint32_t num_q_heads, float scale, float* out, void* workspace,
                        uint64_t workspace_bytes, int* d_status, void* stream);

/*
 * The two halves of hp_attention_decode, for a block table shared by several calls (the
 * layers of one decode step read their K/V pools through the same table, offsets and
 * counts).  ASYNC hp_attention_plan validates k_desc (always; see above), stores each
 * sequence's step counts in `workspace` and zeroes its segment counts.  ASYNC
 * hp_attention_decode_planned then runs the attention kernel alone; any number of
 * planned calls may follow one plan on the same stream, each with its own K pool (the
 * descriptor's page_pool), V pool, q, scale and out, provided the descriptor's table,
 * offsets, counts and geometry and num_q_heads are those of the plan.  A planned call
 * after a plan that failed writes nothing.  The host checks of hp_attention_decode
 * apply to both; neither stores HP_OK over an earlier error in *d_status.
 */
int hp_attention_plan(const hp_paged_desc* k_desc, uint32_t num_q_heads, void* workspace,
                      uint64_t workspace_bytes, int* d_status, void* stream);
int hp_attention_decode_planned(const hp_paged_desc* k_desc, const void* v_pool, const void* q,
                                uint32_t num_q_heads, float scale, float* out,
                                const void* workspace, uint64_t workspace_bytes, int* d_status,
                                void* stream);

/* --------------------------------------------------------- layout conversions */
/*
 * ASYNC.  [HF] Framework Compliance: a producer whose cache sits in a kernel-internal
 * layout must transpose it to the interchange layout before emitting a descriptor.
 * hp_from_kernel_layout reads `src` as [num_blocks, num_heads, head_dim/x, block_size, x]
 * (the older key-cache reshape; x = 1 gives [num_blocks, num_heads, head_dim, block_size])
 * and writes `dst` as [num_blocks, block_size, num_heads, head_dim]: element (b, t, h, d)
 * of dst is element (b, h, d/x, t, d mod x) of src.  hp_to_kernel_layout is the inverse.
 * Elements of `dtype` are copied as bytes; src and dst are device buffers that must not
 * overlap.  x must divide head_dim (HP_ERR_ARG); block_size*head_dim*width must not exceed
 * 48 KiB (one (block, head) unit is staged in shared memory; HP_ERR_ARG beyond), and
 * num_heads must be below 2^31 (HP_ERR_ARG).
 */
int hp_from_kernel_layout(const void* src, void* dst, uint64_t num_blocks, uint64_t block_size,
                          uint64_t num_heads, uint64_t head_dim, uint64_t x, uint32_t dtype,
                          void* stream);
int hp_to_kernel_layout(const void* src, void* dst, uint64_t num_blocks, uint64_t block_size,
                        uint64_t num_heads, uint64_t head_dim, uint64_t x, uint32_t dtype,
                        void* stream);

/* Device workspace (256-byte aligned) the table conversions need for `batch` sequences. */
int hp_table_workspace_bytes(uint64_t batch, uint64_t* bytes);

/*
 * ASYNC.  A padded block table [batch, max_blocks] with per-sequence token counts -- the
 * form of [VA] "How the attention kernel uses the block table" -- to the CSR slices of a
 * block-paged descriptor ([HF] Description): sequence s keeps the first
 * ceil(lens[s] / page_size) entries of its row.  `padded`, `lens` (batch entries) and the
 * outputs `table_out` (table_cap entries) and `seq_ptr_out` (batch+1 entries) are device
 * arrays of `index_type`.  On the device: a sequence needing more than max_blocks pages
 * stores HP_ERR_LEN, more than table_cap entries in all HP_ERR_OUT_SIZE; then nothing is
 * written.
 */
int hp_padded_to_csr(const void* padded, const void* lens, uint64_t batch, uint64_t max_blocks,
                     uint64_t page_size, uint32_t index_type, void* table_out,
                     uint64_t table_cap, void* seq_ptr_out, void* workspace,
                     uint64_t workspace_bytes, int* d_status, void* stream);

/*
 * ASYNC.  The inverse: row s of `padded_out` ([batch, max_blocks]) holds the slice
 * table[seq_ptr[s] .. seq_ptr[s+1]) followed by `pad`.  A slice that is reversed, ends
 * past table_len or is longer than max_blocks stores HP_ERR_LEN (nothing written).
 */
int hp_csr_to_padded(const void* table, uint64_t table_len, const void* seq_ptr, uint64_t batch,
                     uint64_t max_blocks, uint64_t pad, uint32_t index_type, void* padded_out,
                     void* workspace, uint64_t workspace_bytes, int* d_status, void* stream);

/* ------------------------------------------------------------ per-lane layout */
/*
 * Host only.  The checks of [CH] PagedKvLayout::new for a layout of logical
 * capacity `capacity` with `page_tokens` positions per page and page table
 * `table` (host, table_len entries): zero capacity, zero page size, an
 * overflowing ceil(C/P)*P, table_len != ceil(C/P), an entry >= ceil(C/P), a
 * repeated entry -- in that order, first failing entry first.  detail (host,
 * 2 entries, may be NULL) receives (expected, actual) for HP_ERR_PAGE_COUNT,
 * (logical page, physical page) for HP_ERR_PHYSICAL_PAGE, (physical page, 0)
 * for HP_ERR_ALIASED_PAGE.  A table that passes is a permutation of
 * 0..ceil(C/P)-1.
 */
int hp_lane_validate(uint64_t capacity, uint64_t page_tokens, const uint64_t* table,
                     uint64_t table_len, uint64_t* detail);

/*
 * ASYNC.  Logical snapshot of the per-lane layout ([CH] "Include the batch,
 * shared head and feature"): `pool` (device) is [N, B, H_kv, P, d] elements of
 * `dtype` with N = ceil(capacity/page_tokens), P = page_tokens, B = batch,
 * H_kv = kv_heads, d = width; `table` (device, N uint64 entries) maps logical
 * page q to physical page table[q].  `out` (device) receives [B, H_kv, n, d]:
 * element (b, h, p, f) = pool scalar ((table[p/P]*B*H_kv + b*H_kv + h)*P +
 * p%P)*d + f, for the n live positions p < n.  Requires n <= capacity
 * (HP_ERR_LENGTH).  The table is not validated here (hp_lane_validate does
 * that once); an entry >= N skips its rows and stores HP_ERR_PHYSICAL_PAGE in
 * *d_status.  flags: 0, or HP_HOST_MEMORY when pool or out is page-locked host memory.
 */
int hp_lane_gather(const void* pool, const uint64_t* table, uint64_t capacity,
                   uint64_t page_tokens, uint64_t batch, uint64_t kv_heads, uint64_t width,
                   uint32_t dtype, uint64_t n, void* out, uint32_t flags, int* d_status,
                   void* stream);

/*
 * ASYNC.  Append m rows per lane at positions n..n+m-1 (a decode step appends
 * one): element (b, h, i, f) of `new_rows` (device, [B, H_kv, m, d]) is written
 * to pool scalar ((table[p/P]*B*H_kv + b*H_kv + h)*P + p%P)*d + f with p = n+i.
 * Requires n + m <= capacity (HP_ERR_LENGTH, nothing written).  flags: 0, or
 * HP_HOST_MEMORY when pool or new_rows is page-locked host memory.
 */
int hp_lane_append(void* pool, const uint64_t* table, uint64_t capacity, uint64_t page_tokens,
                   uint64_t batch, uint64_t kv_heads, uint64_t width, uint32_t dtype,
                   uint64_t n, uint64_t m, const void* new_rows, uint32_t flags, int* d_status,
                   void* stream);

/* ---------------------------------------------------- no-allocation variant */
/*
 * ASYNC.  hp_gather without a caller-provided workspace.  (The pages have no counterpart:
 * this is a convenience of this library.)
 *
 * Who needs it: callers that cannot allocate device memory -- a plugin inside a framework
 * that owns the device's memory budget and gives its plugins buffers but no allocator, or
 * a latency-critical loop that must not call cudaMalloc/cudaFree (they can block, and
 * cudaFree synchronises the device).  Inputs and output are as for hp_gather; the plan's
 * workspace lives instead in one fixed array of device memory inside the library,
 * sized for HP_NOALLOC_MAX_SEQS sequences (about 257 KiB).  Every device that loads the
 * library holds that array until the process exits.  This function allocates nothing.
 *
 * - num_seqs > HP_NOALLOC_MAX_SEQS returns HP_ERR_NOALLOC_LIMIT before anything else is
 *   checked; use hp_gather with your own workspace for larger batches.
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, which may also load the library's device code on that
 *   device) and keeps it for the life of the process; make that first call before any
 *   stream capture.  Because the address is kept, resetting a device
 *   (cudaDeviceReset) after its first call is not supported: the device code may load
 *   elsewhere in the new context, and later calls would write through the stale address.
 * - All calls on a device share the one array.  Two calls whose work overlaps on the
 *   GPU (different streams, or different host threads, without ordering between them)
 *   race on it and may produce wrong output; order them, e.g. on one stream.  A call
 *   does not depend on what an earlier call left in the array.
 */
#define HP_NOALLOC_MAX_SEQS 16384
int hp_gather_noalloc(const hp_paged_desc* desc, void* out, uint64_t out_tokens,
                      int* d_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* HP_H */
