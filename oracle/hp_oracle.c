/*
 * hp_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU restatement of what the block-paged
 * KV-cache hot path computes.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this file's library; the product
 * path never does.  It shares no code, header, table or constant with the
 * CUDA library: it has its own descriptor struct and its own rule codes.
 *
 * Sources (each function names the passage it follows):
 *   [HF]  "Block-Paged Layout -- Hurray Format Specification"
 *   [CH]  "Keep token order across cache pages" (practical-ch20-paged-kv-layout)
 *
 * Every function below is pinned by a test against values the pages print,
 * closed forms, or brute force (see tests/test_oracle_pins.py and
 * tests/test_oracle_bruteforce.py).  Nothing here is blocked, fused or
 * reordered beyond what the passage states.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -shared -fPIC (no fast-math: the
 * dequantising lookup relies on IEEE double arithmetic).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- codes -- */
/* The oracle's own rule codes.  Tests compare them with the library's codes
 * by NAME (or_code_name), never by number. */
enum {
    OR_OK = 0,
    /* structural checks, evaluated in this order */
    OR_RANK = 1,          /* [HF] Description: rank must be 3               */
    OR_PAGED_AXIS,        /* [HF] Logical Shape / invariant (6)              */
    OR_SHARD,             /* [HF] Sharding: shard descriptor must be rejected */
    OR_INDEX_TYPE,        /* [HF] Additional Descriptor Fields: 0x00 / 0x01  */
    OR_DTYPE,             /* element type not one this reader knows          */
    OR_ZERO_DIM,          /* page_size, num_heads or head_dim is zero        */
    OR_SCALES,            /* [HF] Scale-buffer size: num_pages*page_size     */
    OR_NULL,              /* a required buffer is absent                     */
    OR_ALIGN,             /* [HF] Alignment: at least 64 bytes               */
    OR_OVERFLOW,          /* [HF] invariant (4): pool byte size must exist   */
    /* storage invariants, evaluated in this order */
    OR_SEQ_PTR_START,     /* [HF] invariant (1): seq_ptr[0] = 0              */
    OR_SEQ_PTR_ORDER,     /* [HF] invariant (2): non-decreasing              */
    OR_SEQ_PTR_END,       /* [HF] invariant (1): seq_ptr[S] = table length   */
    OR_PAGE_ID,           /* [HF] invariant (3): 0 <= block_table[k] < pages */
    OR_LEN,               /* token count must fit in the sequence's slice    */
    /* append-only checks */
    OR_NEW_PTR_START,
    OR_NEW_PTR_ORDER,
    OR_NEW_PTR_END,
    OR_CAPACITY,
    /* gather argument */
    OR_OUT_SIZE,
    /* per-lane layout ([CH] PagedKvLayout::new and payload) */
    OR_ZERO_CAPACITY,
    OR_ZERO_PAGE_SIZE,
    OR_LANE_OVERFLOW,
    OR_PAGE_COUNT,
    OR_PHYSICAL_PAGE,
    OR_ALIASED_PAGE,
    OR_LENGTH,
    OR_ALLOCATION_FAILED,
    /* quantization schemes ([HF] Per-scheme composition) */
    OR_QUANT_SCHEME,
    OR_QUANT_BLOCK,
    OR_NCODES
};

static const char* const or_names[OR_NCODES] = {
    "OK", "RANK", "PAGED_AXIS", "SHARD", "INDEX_TYPE", "DTYPE", "ZERO_DIM",
    "SCALES", "NULL", "ALIGN", "OVERFLOW", "SEQ_PTR_START", "SEQ_PTR_ORDER",
    "SEQ_PTR_END", "PAGE_ID", "LEN", "NEW_PTR_START", "NEW_PTR_ORDER",
    "NEW_PTR_END", "CAPACITY", "OUT_SIZE", "ZERO_CAPACITY", "ZERO_PAGE_SIZE",
    "LANE_OVERFLOW", "PAGE_COUNT", "PHYSICAL_PAGE", "ALIASED_PAGE", "LENGTH",
    "ALLOCATION_FAILED", "QUANT_SCHEME", "QUANT_BLOCK"};

const char* or_code_name(int code)
{
    if (code < 0 || code >= OR_NCODES) return "UNKNOWN";
    return or_names[code];
}

/* Element types the oracle knows, with their byte widths. */
enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_I8 = 3, OR_U8 = 4, OR_F64 = 5 };

uint64_t or_elem_size(uint32_t dtype)
{
    switch (dtype) {
    case OR_F32: return 4;
    case OR_F16: return 2;
    case OR_BF16: return 2;
    case OR_I8: return 1;
    case OR_U8: return 1;
    case OR_F64: return 8;
    default: return 0;
    }
}

/* ----------------------------------------------------------- descriptor -- */
/* [HF] Buffer Table / Additional Descriptor Fields: buffers 0-2 are page_pool,
 * block_table and seq_ptr; buffers 3+ carry quantisation parameters.  The
 * per-sequence token count is carried beside them (seq_lens), in the index
 * type of block_table. */
typedef struct or_desc {
    uint32_t rank, paged_axis, has_shard, flags, dtype, index_type;
    uint64_t num_pages, page_size, num_heads, head_dim, num_seqs, table_len,
        scales_len;
    void* page_pool;          /* host copy: [num_pages, page_size, H, D]     */
    const void* block_table;  /* host copy: table_len entries                */
    const void* seq_ptr;      /* host copy: num_seqs + 1 entries             */
    const void* seq_lens;     /* host copy: num_seqs entries                 */
    const float* scales;      /* host copy: num_pages * page_size entries    */
    /* the buffer addresses a reader sees (checked for presence/alignment) */
    uint64_t addr_pool, addr_table, addr_seq_ptr, addr_lens, addr_scales;
} or_desc;

#define OR_PERMISSIVE 1u
#define OR_HAS_QUANT 2u

/* Read entry i of an index buffer (uint32 when index_type = 0x00, uint64
 * when 0x01; [HF] Additional Descriptor Fields). */
static uint64_t ix(const or_desc* d, const void* buf, uint64_t i)
{
    if (d->index_type == 0) return ((const uint32_t*)buf)[i];
    return ((const uint64_t*)buf)[i];
}

/* -------------------------------------------------------------- checks -- */
/* Structural checks, in a fixed order: [HF] Description (rank 3), Logical
 * Shape (paged_axis 0), Sharding (no shard descriptor), Additional
 * Descriptor Fields (index type 0x00/0x01; a uint32 table addresses at most
 * 0xFFFFFFFF pages), Scale-buffer size, Alignment (64 bytes), invariant (4)
 * (the pool's byte size num_pages*page_size*H*D*width must exist). */
static int structural(const or_desc* d)
{
    if (d->rank != 3) return OR_RANK;
    if (d->paged_axis != 0) return OR_PAGED_AXIS;
    if (d->has_shard) return OR_SHARD;
    if (d->index_type > 1) return OR_INDEX_TYPE;
    if (d->index_type == 0 &&
        (d->num_pages > 0x100000000ull || d->table_len > 0xFFFFFFFFull))
        return OR_INDEX_TYPE;
    if (or_elem_size(d->dtype) == 0) return OR_DTYPE;
    if (d->page_size == 0 || d->num_heads == 0 || d->head_dim == 0) return OR_ZERO_DIM;
    if (d->flags & OR_HAS_QUANT) {
        unsigned __int128 want = (unsigned __int128)d->num_pages * d->page_size;
        if (d->addr_scales == 0 || (unsigned __int128)d->scales_len != want) return OR_SCALES;
    }
    if ((d->num_pages > 0 && d->addr_pool == 0) || d->addr_seq_ptr == 0 ||
        (d->num_seqs > 0 && d->addr_lens == 0) ||
        (d->table_len > 0 && d->addr_table == 0))
        return OR_NULL;
    if (d->addr_pool % 64 || d->addr_table % 64 || d->addr_seq_ptr % 64 ||
        d->addr_lens % 64 || ((d->flags & OR_HAS_QUANT) && d->addr_scales % 64))
        return OR_ALIGN;
    unsigned __int128 bytes = (unsigned __int128)d->num_pages * d->page_size;
    bytes *= d->num_heads;
    if (bytes >> 64) return OR_OVERFLOW;
    bytes *= d->head_dim;
    if (bytes >> 64) return OR_OVERFLOW;
    bytes *= or_elem_size(d->dtype);
    if (bytes >> 64) return OR_OVERFLOW;
    return OR_OK;
}

/* Storage invariants (1)-(3) of [HF] Storage Invariants, then the token-count
 * rule: a sequence's token count must fit in the pages its slice names,
 * len_s <= (seq_ptr[s+1]-seq_ptr[s]) * page_size ([HF] Partial trailing page:
 * a reader must not read past the count bounded by seq_ptr).  First failing
 * rule wins; within a rule the first failing index wins. */
static int invariants(const or_desc* d, uint64_t* first)
{
    const uint64_t S = d->num_seqs;
    if (ix(d, d->seq_ptr, 0) != 0) { *first = 0; return OR_SEQ_PTR_START; }
    for (uint64_t s = 0; s < S; ++s)
        if (ix(d, d->seq_ptr, s) > ix(d, d->seq_ptr, s + 1)) { *first = s; return OR_SEQ_PTR_ORDER; }
    if (ix(d, d->seq_ptr, S) != d->table_len) { *first = S; return OR_SEQ_PTR_END; }
    for (uint64_t k = 0; k < d->table_len; ++k)
        if (ix(d, d->block_table, k) >= d->num_pages) { *first = k; return OR_PAGE_ID; }
    for (uint64_t s = 0; s < S; ++s) {
        uint64_t slice = ix(d, d->seq_ptr, s + 1) - ix(d, d->seq_ptr, s);
        unsigned __int128 room = (unsigned __int128)slice * d->page_size;
        if ((unsigned __int128)ix(d, d->seq_lens, s) > room) { *first = s; return OR_LEN; }
    }
    return OR_OK;
}

/* Reader validation ([HF] Storage Invariants): the structural checks always;
 * invariants (1)-(3) and the token-count rule unless permissive.  Aliased page
 * IDs are never checked ([HF] Prefix Sharing). */
int or_validate(const or_desc* d, uint64_t* first)
{
    *first = 0;
    int c = structural(d);
    if (c != OR_OK) return c;
    if (d->flags & OR_PERMISSIVE) return OR_OK;
    return invariants(d, first);
}

/* Total logical tokens = sum of per-sequence token counts ([HF] Logical Shape).
 * Returns 0 and sets *ok = 0 when the sum does not fit in 64 bits. */
uint64_t or_total_tokens(const or_desc* d, int* ok)
{
    unsigned __int128 sum = 0;
    for (uint64_t s = 0; s < d->num_seqs; ++s) sum += ix(d, d->seq_lens, s);
    *ok = (sum >> 64) == 0;
    return (uint64_t)sum;
}

/* --------------------------------------------------------- element lookup */
/* [HF] Element Lookup, step by step.  Returns 0 and the flat pool index on
 * success.  Returns a rule code when the lookup leaves its slice, the table or
 * the pool (only reachable in permissive mode, where those are not validated
 * beforehand): the element is then not read. */
static int lookup_flat(const or_desc* d, uint64_t s, uint64_t t, uint64_t h,
                       uint64_t dd, uint64_t* flat, uint64_t* phys_out,
                       uint64_t* off_out)
{
    const uint64_t P = d->page_size;
    uint64_t page_in_seq = t / P;                 /* integer division */
    uint64_t offset_in_page = t % P;
    uint64_t lo = ix(d, d->seq_ptr, s), hi = ix(d, d->seq_ptr, s + 1);
    if (hi < lo || page_in_seq >= hi - lo) return OR_LEN;
    if (lo + page_in_seq >= d->table_len) return OR_LEN;
    uint64_t phys_page = ix(d, d->block_table, lo + page_in_seq);
    if (phys_page >= d->num_pages) return OR_PAGE_ID;
    *flat = ((phys_page * P + offset_in_page) * d->num_heads + h) * d->head_dim + dd;
    if (phys_out) *phys_out = phys_page;
    if (off_out) *off_out = offset_in_page;
    return OR_OK;
}

/* The value at (s, t, h, d), copied byte for byte into *value (element width
 * bytes).  Returns 0, or the rule code that stopped the lookup. */
int or_lookup(const or_desc* d, uint64_t s, uint64_t t, uint64_t h, uint64_t dd,
              void* value)
{
    uint64_t flat;
    int c = lookup_flat(d, s, t, h, dd, &flat, 0, 0);
    if (c != OR_OK) return c;
    const uint64_t es = or_elem_size(d->dtype);
    memcpy(value, (const unsigned char*)d->page_pool + flat * es, es);
    return OR_OK;
}

/* Gather the ragged batch into the logical [total_tokens, H, D] tensor: the
 * rows of sequence s follow those of sequences 0..s-1 in order ([HF] Logical
 * Shape), and every element is the Element Lookup's value, copied as bytes.
 * Only t < len_s is visited ([HF] Partial trailing page).  A lookup that
 * fails (permissive mode only) leaves its output row untouched; such rows are
 * marked 0 in row_written (optional) and the first failure's code is
 * returned. */
int or_gather(const or_desc* d, void* out, unsigned char* row_written)
{
    const uint64_t es = or_elem_size(d->dtype);
    const uint64_t H = d->num_heads, D = d->head_dim;
    int first_fault = OR_OK;
    uint64_t row = 0; /* running sum of the counts of sequences before s */
    for (uint64_t s = 0; s < d->num_seqs; ++s) {
        const uint64_t len = ix(d, d->seq_lens, s);
        for (uint64_t t = 0; t < len; ++t, ++row) {
            uint64_t flat;
            int c = lookup_flat(d, s, t, 0, 0, &flat, 0, 0);
            if (row_written) row_written[row] = (c == OR_OK);
            if (c != OR_OK) {
                if (first_fault == OR_OK) first_fault = c;
                continue;
            }
            for (uint64_t h = 0; h < H; ++h)
                for (uint64_t dd = 0; dd < D; ++dd) {
                    lookup_flat(d, s, t, h, dd, &flat, 0, 0);
                    memcpy((unsigned char*)out + ((row * H + h) * D + dd) * es,
                           (const unsigned char*)d->page_pool + flat * es, es);
                }
        }
    }
    return first_fault;
}

/* ------------------------------------------------------------- dequant -- */
/* Round a double to the nearest bfloat16, ties to even, from the IEEE 754
 * definition of the binary16-brain format (8 significant bits, the exponent
 * range of binary32, subnormals down to 2^-133).  Returns the 16-bit code. */
uint16_t or_bf16_rne(double x)
{
    if (isnan(x)) return signbit(x) ? 0xFFC0 : 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isinf(a)) return sign | 0x7F80;
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                /* a = m * 2^e, 0.5 <= m < 1 */
    int qexp = e - 8;            /* quantum of an 8-bit significand */
    if (qexp < -133) qexp = -133; /* subnormal quantum */
    double r = ldexp(a, -qexp);  /* exact: scaling by a power of two */
    double n = rint(r);          /* default rounding: nearest, ties to even */
    double v = ldexp(n, qexp);
    if (v >= ldexp(1.0, 128)) return sign | 0x7F80; /* beyond the format */
    float f = (float)v;          /* exact: v has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    return sign | (uint16_t)(bits >> 16);
}

/* [HF] Element Lookup, quantized case, with [HF] Per-page-slot parameters:
 * the int8 value at (s,t,h,d) times scales[phys_page*page_size +
 * offset_in_page], a symmetric scheme (no zero point).  The product is formed
 * exactly in double (an 8-bit integer times a 24-bit significand fits in 53
 * bits) and rounded once to bfloat16. */
int or_lookup_dequant(const or_desc* d, uint64_t s, uint64_t t, uint64_t h,
                      uint64_t dd, uint16_t* value)
{
    uint64_t flat, phys, off;
    int c = lookup_flat(d, s, t, h, dd, &flat, &phys, &off);
    if (c != OR_OK) return c;
    int8_t q = ((const int8_t*)d->page_pool)[flat];
    double scale = d->scales[phys * d->page_size + off];
    *value = or_bf16_rne((double)q * scale);
    return OR_OK;
}

/* Dequantising gather: or_gather with each element replaced by its
 * dequantised bfloat16 value. */
int or_gather_dequant(const or_desc* d, uint16_t* out, unsigned char* row_written)
{
    const uint64_t H = d->num_heads, D = d->head_dim;
    int first_fault = OR_OK;
    uint64_t row = 0;
    for (uint64_t s = 0; s < d->num_seqs; ++s) {
        const uint64_t len = ix(d, d->seq_lens, s);
        for (uint64_t t = 0; t < len; ++t, ++row) {
            uint16_t v;
            int c = or_lookup_dequant(d, s, t, 0, 0, &v);
            if (row_written) row_written[row] = (c == OR_OK);
            if (c != OR_OK) {
                if (first_fault == OR_OK) first_fault = c;
                continue;
            }
            for (uint64_t h = 0; h < H; ++h)
                for (uint64_t dd = 0; dd < D; ++dd) {
                    or_lookup_dequant(d, s, t, h, dd, &v);
                    out[(row * H + h) * D + dd] = v;
                }
        }
    }
    return first_fault;
}

/* ------------------------------------------------- quantization schemes -- */
/* [HF] Quantization Compatibility, Per-scheme composition.  A scheme tag with its axis
 * and block size, the scale count, fp32 scales and optional zero points of the pool's
 * element type (host copies), and the addresses a reader sees. */
typedef struct or_quant {
    uint32_t scheme_tag, axis;
    uint64_t block_size, count;
    const float* scales;
    const void* zero_points; /* NULL: symmetric, zero point 0 */
    uint64_t addr_scales, addr_zero_points;
} or_quant;

enum { OR_PER_TENSOR = 0x01, OR_PER_CHANNEL = 0x02, OR_PER_BLOCK_AFFINE = 0x03 };

/* The checks on a scheme, in this order: the pool holds 8-bit integers; the tag is one
 * of 0x01, 0x02, 0x03; a per-channel axis is 1 (num_heads) or 2 (head_dim) -- the paged
 * axis must not be quantized per channel; a per-block-affine scheme has axis 0 and
 * block_size == page_size (a reader must reject it otherwise); the count is what the
 * scheme needs (1; num_heads or head_dim; num_pages*page_size per [HF] Scale-buffer
 * size); scales are present; both buffers are 64-byte aligned ([HF] Alignment). */
int or_validate_quant(const or_desc* d, const or_quant* q)
{
    if (d->dtype != OR_I8 && d->dtype != OR_U8) return OR_DTYPE;
    uint64_t want;
    if (q->scheme_tag == OR_PER_TENSOR) {
        want = 1;
    } else if (q->scheme_tag == OR_PER_CHANNEL) {
        if (q->axis == 1) want = d->num_heads;
        else if (q->axis == 2) want = d->head_dim;
        else return OR_QUANT_SCHEME;
    } else if (q->scheme_tag == OR_PER_BLOCK_AFFINE) {
        if (q->axis != 0 || q->block_size != d->page_size) return OR_QUANT_BLOCK;
        unsigned __int128 n = (unsigned __int128)d->num_pages * d->page_size;
        if (n >> 64) return OR_SCALES;
        want = (uint64_t)n;
    } else {
        return OR_QUANT_SCHEME;
    }
    if (q->count != want) return OR_SCALES;
    if (q->addr_scales == 0) return OR_NULL;
    if (q->addr_scales % 64 || q->addr_zero_points % 64) return OR_ALIGN;
    return OR_OK;
}

/* [HF] Element Lookup, quantized case, under a scheme: the pool element q at (s,t,h,d),
 * the parameter entry the scheme assigns it (0; h or d; phys_page*page_size +
 * offset_in_page), and the bfloat16 nearest the exact (q - zero_point) * scale -- formed
 * in double, exact for 8-bit integers and a 24-bit significand, rounded once. */
int or_lookup_dequant_q(const or_desc* d, const or_quant* q, uint64_t s, uint64_t t,
                        uint64_t h, uint64_t dd, uint16_t* value)
{
    uint64_t flat, phys, off;
    int c = lookup_flat(d, s, t, h, dd, &flat, &phys, &off);
    if (c != OR_OK) return c;
    uint64_t k;
    if (q->scheme_tag == OR_PER_TENSOR) k = 0;
    else if (q->scheme_tag == OR_PER_CHANNEL) k = q->axis == 1 ? h : dd;
    else k = phys * d->page_size + off;
    double qv, zp = 0.0;
    if (d->dtype == OR_I8) {
        qv = ((const int8_t*)d->page_pool)[flat];
        if (q->zero_points) zp = ((const int8_t*)q->zero_points)[k];
    } else {
        qv = ((const uint8_t*)d->page_pool)[flat];
        if (q->zero_points) zp = ((const uint8_t*)q->zero_points)[k];
    }
    *value = or_bf16_rne((qv - zp) * (double)q->scales[k]);
    return OR_OK;
}

/* The dequantising gather under a scheme: or_gather with each element replaced by
 * or_lookup_dequant_q's value. */
int or_gather_dequant_q(const or_desc* d, const or_quant* q, uint16_t* out,
                        unsigned char* row_written)
{
    const uint64_t H = d->num_heads, D = d->head_dim;
    int first_fault = OR_OK;
    uint64_t row = 0;
    for (uint64_t s = 0; s < d->num_seqs; ++s) {
        const uint64_t len = ix(d, d->seq_lens, s);
        for (uint64_t t = 0; t < len; ++t, ++row) {
            uint16_t v;
            int c = or_lookup_dequant_q(d, q, s, t, 0, 0, &v);
            if (row_written) row_written[row] = (c == OR_OK);
            if (c != OR_OK) {
                if (first_fault == OR_OK) first_fault = c;
                continue;
            }
            for (uint64_t h = 0; h < H; ++h)
                for (uint64_t dd = 0; dd < D; ++dd) {
                    or_lookup_dequant_q(d, q, s, t, h, dd, &v);
                    out[(row * H + h) * D + dd] = v;
                }
        }
    }
    return first_fault;
}

/* --------------------------------------------------------------- append -- */
/* Validation for an append: the structural checks; then, unless permissive,
 * invariants (1)-(3) ([HF] Storage Invariants); then the CSR offsets of the
 * new rows (new_ptr[0] = 0, non-decreasing, new_ptr[S] = total_new); then the
 * capacity rule: the count before the append plus the new rows must fit in the
 * slice's pages, len_s + n_s <= slice_s * page_size. */
int or_validate_append(const or_desc* d, const void* new_ptr, uint64_t total_new,
                       uint64_t* first)
{
    *first = 0;
    int c = structural(d);
    if (c != OR_OK) return c;
    if (d->flags & OR_PERMISSIVE) return OR_OK;
    const uint64_t S = d->num_seqs;
    if (ix(d, d->seq_ptr, 0) != 0) { *first = 0; return OR_SEQ_PTR_START; }
    for (uint64_t s = 0; s < S; ++s)
        if (ix(d, d->seq_ptr, s) > ix(d, d->seq_ptr, s + 1)) { *first = s; return OR_SEQ_PTR_ORDER; }
    if (ix(d, d->seq_ptr, S) != d->table_len) { *first = S; return OR_SEQ_PTR_END; }
    for (uint64_t k = 0; k < d->table_len; ++k)
        if (ix(d, d->block_table, k) >= d->num_pages) { *first = k; return OR_PAGE_ID; }
    if (ix(d, new_ptr, 0) != 0) { *first = 0; return OR_NEW_PTR_START; }
    for (uint64_t s = 0; s < S; ++s)
        if (ix(d, new_ptr, s) > ix(d, new_ptr, s + 1)) { *first = s; return OR_NEW_PTR_ORDER; }
    if (ix(d, new_ptr, S) != total_new) { *first = S; return OR_NEW_PTR_END; }
    for (uint64_t s = 0; s < S; ++s) {
        uint64_t slice = ix(d, d->seq_ptr, s + 1) - ix(d, d->seq_ptr, s);
        unsigned __int128 room = (unsigned __int128)slice * d->page_size;
        unsigned __int128 want = (unsigned __int128)ix(d, d->seq_lens, s) +
                                 (ix(d, new_ptr, s + 1) - ix(d, new_ptr, s));
        if (want > room) { *first = s; return OR_CAPACITY; }
    }
    return OR_OK;
}

/* Append the new rows of every sequence: row i of sequence s (new row
 * new_ptr[s]+i of the [total_new, H, D] input) goes to token
 * t = seq_lens[s] + i, written through the same Element Lookup as the gather
 * ([HF] Element Lookup, applied as a store).  Sequences are visited in
 * increasing s, rows in increasing i.  A lookup that fails (permissive mode
 * only) writes nothing for that row.  The input holds total_new rows and no row
 * outside it is read: a sequence whose pair new_ptr[s] .. new_ptr[s+1] runs
 * backwards (NEW_PTR_ORDER) or past total_new (NEW_PTR_END) contributes no rows
 * (permissive mode only; a validated append has neither).  The first failure's
 * code is returned. */
int or_scatter_append(const or_desc* d, const void* new_rows, const void* new_ptr,
                      uint64_t total_new)
{
    const uint64_t es = or_elem_size(d->dtype);
    const uint64_t H = d->num_heads, D = d->head_dim;
    int first_fault = OR_OK;
    for (uint64_t s = 0; s < d->num_seqs; ++s) {
        const uint64_t base = ix(d, new_ptr, s), end = ix(d, new_ptr, s + 1);
        if (end < base || end > total_new) {
            if (first_fault == OR_OK) first_fault = end < base ? OR_NEW_PTR_ORDER : OR_NEW_PTR_END;
            continue;
        }
        for (uint64_t i = 0; i < end - base; ++i) {
            const uint64_t t = ix(d, d->seq_lens, s) + i;
            uint64_t flat;
            int c = lookup_flat(d, s, t, 0, 0, &flat, 0, 0);
            if (c != OR_OK) {
                if (first_fault == OR_OK) first_fault = c;
                continue;
            }
            for (uint64_t h = 0; h < H; ++h)
                for (uint64_t dd = 0; dd < D; ++dd) {
                    lookup_flat(d, s, t, h, dd, &flat, 0, 0);
                    memcpy((unsigned char*)d->page_pool + flat * es,
                           (const unsigned char*)new_rows + (((base + i) * H + h) * D + dd) * es,
                           es);
                }
        }
    }
    return first_fault;
}

/* ----------------------------------------------------------- writer side -- */
/* [VA] "Copy-on-write for beam search and prefix sharing": a shared block is copied
 * when one request needs to modify it.  For each pair i, physical page dst[i] becomes a
 * byte copy of page src[i] (all page_size rows); pages are page_bytes long.  Page IDs
 * are in the index type of the descriptor.  A pair naming a page >= num_pages copies
 * nothing; the first such pair's code (PAGE_ID) is returned. */
int or_copy_pages(void* pool, uint64_t num_pages, uint64_t page_bytes, uint32_t index_type,
                  const void* src, const void* dst, uint64_t pairs)
{
    int first_fault = OR_OK;
    for (uint64_t i = 0; i < pairs; ++i) {
        uint64_t a = index_type == 0 ? ((const uint32_t*)src)[i] : ((const uint64_t*)src)[i];
        uint64_t b = index_type == 0 ? ((const uint32_t*)dst)[i] : ((const uint64_t*)dst)[i];
        if (a >= num_pages || b >= num_pages) {
            if (first_fault == OR_OK) first_fault = OR_PAGE_ID;
            continue;
        }
        memmove((unsigned char*)pool + b * page_bytes, (const unsigned char*)pool + a * page_bytes,
                page_bytes);
    }
    return first_fault;
}

/* [HF] Partial trailing page: a writer should zero the slots past a sequence's valid
 * token count when the cache crosses a trust boundary.  Slots are zeroed only where no
 * sequence of the batch reads them: for each page the slices name, the number of leading
 * slots that hold a valid token of some sequence referencing it is found first (a shared
 * page keeps what its longest user needs -- [HF] Prefix Sharing), then the rest of that
 * page is set to zero bytes.  Pages no slice names are left alone.  The descriptor must
 * be valid (or_validate); `live` is caller scratch of num_pages entries. */
void or_zero_tails(const or_desc* d, uint64_t* live)
{
    const uint64_t P = d->page_size;
    const uint64_t row_bytes = d->num_heads * d->head_dim * or_elem_size(d->dtype);
    unsigned char* referenced = (unsigned char*)calloc(d->num_pages ? d->num_pages : 1, 1);
    for (uint64_t p = 0; p < d->num_pages; ++p) live[p] = 0;
    for (uint64_t s = 0; s < d->num_seqs; ++s) {
        const uint64_t lo = ix(d, d->seq_ptr, s), hi = ix(d, d->seq_ptr, s + 1);
        const uint64_t len = ix(d, d->seq_lens, s);
        for (uint64_t j = 0; j < hi - lo; ++j) {
            const uint64_t page = ix(d, d->block_table, lo + j);
            uint64_t used = len > j * P ? len - j * P : 0; /* tokens of s in this page */
            if (used > P) used = P;
            if (used > live[page]) live[page] = used;
            referenced[page] = 1;
        }
    }
    for (uint64_t p = 0; p < d->num_pages; ++p)
        if (referenced[p])
            memset((unsigned char*)d->page_pool + (p * P + live[p]) * row_bytes, 0,
                   (P - live[p]) * row_bytes);
    free(referenced);
}

/* ---------------------------------------------------- decode attention -- */
/* binary16 and bfloat16 values as doubles, from the IEEE 754 definitions (binary16: 1
 * sign, 5 exponent bits biased by 15, 10 fraction bits; bfloat16: the upper half of a
 * binary32). */
double or_f16_to_double(uint16_t h)
{
    const int sign = h >> 15, e = (h >> 10) & 0x1F, f = h & 0x3FF;
    double v;
    if (e == 0) v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    else if (e == 31) v = f ? NAN : INFINITY;
    else v = ldexp(1.0 + f / 1024.0, e - 15);
    return sign ? -v : v;
}

double or_bf16_to_double(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

static double elem_value(uint32_t dtype, const void* base, uint64_t i)
{
    switch (dtype) {
    case OR_F16: return or_f16_to_double(((const uint16_t*)base)[i]);
    case OR_BF16: return or_bf16_to_double(((const uint16_t*)base)[i]);
    case OR_F32: return ((const float*)base)[i];
    default: return ((const double*)base)[i];
    }
}

/* Decode attention over a block-paged K/V cache ([VA] "How the attention kernel uses the
 * block table"; [HF] Element Lookup for every key and value): for sequence s and query
 * head qh, kv head g = qh / (Hq / H_kv) (consecutive query heads share a K/V head, as in
 * grouped-query attention); score_t = scale * sum_d q[s,qh,d] * K(s,t,g,d) for t < len_s;
 * weights = softmax(scores) (the maximum subtracted before exp); out[s,qh,d] =
 * sum_t weight_t * V(s,t,g,d).  K comes through the descriptor's pool, V through v_pool
 * with the same table, offsets and counts; q is [num_seqs, Hq, D] of the pool's element
 * type; everything is computed in double.  A sequence with no tokens gets zeros. */
void or_attention_decode(const or_desc* d, const void* v_pool, const void* q, uint64_t Hq,
                         double scale, double* out)
{
    const uint64_t H = d->num_heads, D = d->head_dim, G = Hq / H;
    or_desc vd = *d;
    vd.page_pool = (void*)v_pool;
    for (uint64_t s = 0; s < d->num_seqs; ++s) {
        const uint64_t len = ix(d, d->seq_lens, s);
        double* scores = (double*)malloc((len ? len : 1) * sizeof(double));
        for (uint64_t qh = 0; qh < Hq; ++qh) {
            const uint64_t g = qh / G;
            double* o = out + (s * Hq + qh) * D;
            for (uint64_t dd = 0; dd < D; ++dd) o[dd] = 0.0;
            if (len == 0) continue;
            double mx = -INFINITY;
            for (uint64_t t = 0; t < len; ++t) {
                double acc = 0.0;
                for (uint64_t dd = 0; dd < D; ++dd) {
                    uint64_t flat;
                    lookup_flat(d, s, t, g, dd, &flat, 0, 0);
                    acc += elem_value(d->dtype, q, (s * Hq + qh) * D + dd) *
                           elem_value(d->dtype, d->page_pool, flat);
                }
                scores[t] = scale * acc;
                if (scores[t] > mx) mx = scores[t];
            }
            double sum = 0.0;
            for (uint64_t t = 0; t < len; ++t) {
                scores[t] = exp(scores[t] - mx);
                sum += scores[t];
            }
            for (uint64_t t = 0; t < len; ++t)
                for (uint64_t dd = 0; dd < D; ++dd) {
                    uint64_t flat;
                    lookup_flat(&vd, s, t, g, dd, &flat, 0, 0);
                    o[dd] += scores[t] / sum * elem_value(d->dtype, v_pool, flat);
                }
        }
        free(scores);
    }
}

/* ------------------------------------------------- layout conversions -- */
/* [HF] Framework Compliance: a producer whose cache sits in a kernel-internal layout
 * [num_blocks, num_heads, head_dim/x, block_size, x] must transpose it to the interchange
 * layout [num_blocks, block_size, num_heads, head_dim] before emitting a descriptor.
 * Element (b, t, h, d) of the interchange array is element (b, h, d/x, t, d mod x) of the
 * internal one; elements are es bytes, copied as bytes.  x must divide head_dim. */
static uint64_t internal_index(uint64_t b, uint64_t t, uint64_t h, uint64_t d, uint64_t bs,
                               uint64_t H, uint64_t D, uint64_t x)
{
    return (((b * H + h) * (D / x) + d / x) * bs + t) * x + d % x;
}

void or_from_kernel_layout(const void* src, void* dst, uint64_t nb, uint64_t bs, uint64_t H,
                           uint64_t D, uint64_t x, uint64_t es)
{
    for (uint64_t b = 0; b < nb; ++b)
        for (uint64_t t = 0; t < bs; ++t)
            for (uint64_t h = 0; h < H; ++h)
                for (uint64_t d = 0; d < D; ++d)
                    memcpy((unsigned char*)dst + (((b * bs + t) * H + h) * D + d) * es,
                           (const unsigned char*)src + internal_index(b, t, h, d, bs, H, D, x) * es,
                           es);
}

/* The inverse: interchange [num_blocks, block_size, num_heads, head_dim] to the
 * kernel-internal layout. */
void or_to_kernel_layout(const void* src, void* dst, uint64_t nb, uint64_t bs, uint64_t H,
                         uint64_t D, uint64_t x, uint64_t es)
{
    for (uint64_t b = 0; b < nb; ++b)
        for (uint64_t t = 0; t < bs; ++t)
            for (uint64_t h = 0; h < H; ++h)
                for (uint64_t d = 0; d < D; ++d)
                    memcpy((unsigned char*)dst + internal_index(b, t, h, d, bs, H, D, x) * es,
                           (const unsigned char*)src + (((b * bs + t) * H + h) * D + d) * es,
                           es);
}

/* [VA] "How the attention kernel uses the block table": an attention kernel may take a
 * padded table [batch, max_num_blocks] with per-sequence valid-token counts; the
 * block-paged descriptor carries the same slices CSR-style ([HF] Description).  A
 * sequence of len tokens uses its row's first ceil(len / page_size) entries.
 * padded -> CSR: returns LEN (first bad s in *first) when a sequence needs more than
 * max_blocks pages, OUT_SIZE when the entries exceed table_cap. */
static uint64_t ix_t(uint32_t it, const void* buf, uint64_t i)
{
    return it == 0 ? ((const uint32_t*)buf)[i] : ((const uint64_t*)buf)[i];
}

static void put_t(uint32_t it, void* buf, uint64_t i, uint64_t v)
{
    if (it == 0) ((uint32_t*)buf)[i] = (uint32_t)v;
    else ((uint64_t*)buf)[i] = v;
}

int or_padded_to_csr(const void* padded, const void* lens, uint64_t batch, uint64_t max_blocks,
                     uint64_t page_size, uint32_t it, void* table_out, uint64_t table_cap,
                     void* seq_ptr_out, uint64_t* first)
{
    *first = 0;
    uint64_t total = 0;
    for (uint64_t s = 0; s < batch; ++s) {
        const uint64_t len = ix_t(it, lens, s);
        const uint64_t need = len / page_size + (len % page_size != 0);
        if (need > max_blocks) { *first = s; return OR_LEN; }
        total += need;
    }
    if (total > table_cap) return OR_OUT_SIZE;
    uint64_t k = 0;
    put_t(it, seq_ptr_out, 0, 0);
    for (uint64_t s = 0; s < batch; ++s) {
        const uint64_t len = ix_t(it, lens, s);
        const uint64_t need = len / page_size + (len % page_size != 0);
        for (uint64_t j = 0; j < need; ++j) put_t(it, table_out, k++, ix_t(it, padded, s * max_blocks + j));
        put_t(it, seq_ptr_out, s + 1, k);
    }
    return OR_OK;
}

/* CSR -> padded: row s holds slice s (block_table[seq_ptr[s] .. seq_ptr[s+1])) followed
 * by `pad`; LEN (first s) when a slice is longer than max_blocks. */
int or_csr_to_padded(const void* table, const void* seq_ptr, uint64_t batch, uint64_t max_blocks,
                     uint64_t pad, uint32_t it, void* padded_out, uint64_t* first)
{
    *first = 0;
    for (uint64_t s = 0; s < batch; ++s)
        if (ix_t(it, seq_ptr, s + 1) - ix_t(it, seq_ptr, s) > max_blocks) { *first = s; return OR_LEN; }
    for (uint64_t s = 0; s < batch; ++s) {
        const uint64_t lo = ix_t(it, seq_ptr, s), n = ix_t(it, seq_ptr, s + 1) - lo;
        for (uint64_t j = 0; j < max_blocks; ++j)
            put_t(it, padded_out, s * max_blocks + j, j < n ? ix_t(it, table, lo + j) : pad);
    }
    return OR_OK;
}

/* ------------------------------------------------------- per-lane layout -- */
/* [CH] "Locate a row without changing its logical meaning", PagedKvLayout::new:
 * zero capacity, zero page size, an overflowing rounded capacity, a table whose
 * length is not ceil(C/P), an out-of-range physical page and a repeated
 * physical page are rejected, in that order; the first failing entry wins.
 * detail[0..1] receive (expected, actual) for PAGE_COUNT, (logical page,
 * physical page) for PHYSICAL_PAGE and (physical page, 0) for ALIASED_PAGE. */
int or_lane_new(uint64_t capacity, uint64_t page_tokens, const uint64_t* table,
                uint64_t table_len, uint64_t* detail)
{
    detail[0] = detail[1] = 0;
    if (capacity == 0) return OR_ZERO_CAPACITY;
    if (page_tokens == 0) return OR_ZERO_PAGE_SIZE;
    uint64_t pages = capacity / page_tokens + (capacity % page_tokens != 0);
    unsigned __int128 physical_tokens = (unsigned __int128)pages * page_tokens;
    if (physical_tokens >> 64) return OR_LANE_OVERFLOW;
    if (table_len != pages) {
        detail[0] = pages;
        detail[1] = table_len;
        return OR_PAGE_COUNT;
    }
    unsigned char* used = (unsigned char*)calloc(pages ? pages : 1, 1);
    if (!used) return OR_ALLOCATION_FAILED;
    int code = OR_OK;
    for (uint64_t logical_page = 0; logical_page < pages; ++logical_page) {
        uint64_t physical_page = table[logical_page];
        if (physical_page >= pages) {
            detail[0] = logical_page;
            detail[1] = physical_page;
            code = OR_PHYSICAL_PAGE;
            break;
        }
        if (used[physical_page]) {
            detail[0] = physical_page;
            code = OR_ALIASED_PAGE;
            break;
        }
        used[physical_page] = 1;
    }
    free(used);
    return code;
}

/* [CH] PagedKvLayout::address: position -> (logical page, physical page,
 * offset in page); "None" (return 1) when the position is at or past the
 * capacity. */
int or_lane_address(uint64_t capacity, uint64_t page_tokens, const uint64_t* table,
                    uint64_t position, uint64_t* out3)
{
    if (position >= capacity) return 1;
    uint64_t logical_page = position / page_tokens;
    out3[0] = logical_page;
    out3[1] = table[logical_page];
    out3[2] = position % page_tokens;
    return 0;
}

/* [CH] PagedKvLayout::row_start: first scalar of the row of `lane` (one of
 * `lanes`) at `position`, ((physical_page*lanes + lane)*P + offset)*width.
 * The caller has checked lane, width and the position. */
uint64_t or_lane_row_start(uint64_t capacity, uint64_t page_tokens,
                           const uint64_t* table, uint64_t lane, uint64_t lanes,
                           uint64_t width, uint64_t position)
{
    uint64_t a[3];
    or_lane_address(capacity, page_tokens, table, position, a);
    return ((a[1] * lanes + lane) * page_tokens + a[2]) * width;
}

/* [CH] "Include the batch, shared head and feature", physical_row_start: the
 * lane of (batch, head) is batch*heads + head over batch_size*heads lanes.
 * With no table (table == NULL) the contiguous layout (lane*C + p)*width
 * applies.  Returns 1 ("None") when batch, head or position is out of range. */
int or_lane_physical_row_start(uint64_t capacity, uint64_t page_tokens,
                               const uint64_t* table, uint64_t batch_size,
                               uint64_t heads, uint64_t width, uint64_t batch,
                               uint64_t head, uint64_t position, uint64_t* out)
{
    if (batch >= batch_size || head >= heads || position >= capacity) return 1;
    uint64_t lane = batch * heads + head;
    if (table == 0) {
        *out = (lane * capacity + position) * width;
        return 0;
    }
    *out = or_lane_row_start(capacity, page_tokens, table, lane, batch_size * heads,
                             width, position);
    return 0;
}

/* [CH] "Include the batch, shared head and feature": the logical snapshot
 * [B, H_kv, n, d] holds the filled rows p < n of every lane in logical order;
 * element (b, h, p, f) is physical scalar row_start(b*H_kv+h, p) + f of the
 * [N, B, H_kv, P, d] array.  Elements are copied as bytes. */
void or_lane_gather(const void* pool, uint64_t capacity, uint64_t page_tokens,
                    const uint64_t* table, uint64_t batch_size, uint64_t heads,
                    uint64_t width, uint64_t es, uint64_t n, void* out)
{
    for (uint64_t b = 0; b < batch_size; ++b)
        for (uint64_t h = 0; h < heads; ++h)
            for (uint64_t p = 0; p < n; ++p) {
                uint64_t start;
                or_lane_physical_row_start(capacity, page_tokens, table, batch_size,
                                           heads, width, b, h, p, &start);
                for (uint64_t f = 0; f < width; ++f)
                    memcpy((unsigned char*)out + (((b * heads + h) * n + p) * width + f) * es,
                           (const unsigned char*)pool + (start + f) * es, es);
            }
}

/* Append m rows per lane at positions n..n+m-1 (the decode step appends one):
 * element (b, h, i, f) of the [B, H_kv, m, d] input goes to physical scalar
 * row_start(b*H_kv+h, n+i) + f.  Returns LENGTH when n + m exceeds the
 * capacity (nothing written). */
int or_lane_append(void* pool, uint64_t capacity, uint64_t page_tokens,
                   const uint64_t* table, uint64_t batch_size, uint64_t heads,
                   uint64_t width, uint64_t es, uint64_t n, uint64_t m,
                   const void* new_rows)
{
    if (n > capacity || m > capacity - n) return OR_LENGTH;
    for (uint64_t b = 0; b < batch_size; ++b)
        for (uint64_t h = 0; h < heads; ++h)
            for (uint64_t i = 0; i < m; ++i) {
                uint64_t start;
                or_lane_physical_row_start(capacity, page_tokens, table, batch_size,
                                           heads, width, b, h, n + i, &start);
                for (uint64_t f = 0; f < width; ++f)
                    memcpy((unsigned char*)pool + (start + f) * es,
                           (const unsigned char*)new_rows +
                               (((b * heads + h) * m + i) * width + f) * es,
                           es);
            }
    return OR_OK;
}

/* [CH] "Count live rows and two kinds of unused payload", payload():
 * U = 2*B*H_kv*d K+V scalar slots per token position; A = ceil(n/P) active
 * pages; allocated = U*physical_tokens, live = U*n, unused = allocated - live,
 * tail = U*(A*P - n), inactive = U*(physical_tokens - A*P); bytes are slots
 * times 8 (f64).  out[12] = reserved_pages, active_pages, then the allocated,
 * live, unused, tail and inactive slot counts, then the same five as bytes --
 * the order in which PagedKvPayload lists its fields.  Returns LENGTH when n > C and
 * LANE_OVERFLOW when a product does not fit in 64 bits. */
int or_payload(uint64_t capacity, uint64_t page_tokens, uint64_t length,
               uint64_t batch, uint64_t kv_heads, uint64_t width, uint64_t* out)
{
    if (length > capacity) return OR_LENGTH;
    uint64_t pages = capacity / page_tokens + (capacity % page_tokens != 0);
    unsigned __int128 physical_tokens = (unsigned __int128)pages * page_tokens;
    unsigned __int128 per_position = (unsigned __int128)2 * batch;
    per_position *= kv_heads;
    if (per_position >> 64) return OR_LANE_OVERFLOW;
    per_position *= width;
    if (per_position >> 64) return OR_LANE_OVERFLOW;
    uint64_t active_pages = length / page_tokens + (length % page_tokens != 0);
    unsigned __int128 active_positions = (unsigned __int128)active_pages * page_tokens;
    unsigned __int128 v[5];
    v[0] = per_position * physical_tokens;                    /* allocated */
    v[1] = per_position * length;                             /* live */
    v[2] = v[0] - v[1];                                       /* unused */
    v[3] = per_position * (active_positions - length);        /* tail */
    v[4] = per_position * (physical_tokens - active_positions); /* inactive */
    out[0] = pages;
    out[1] = active_pages;
    for (int i = 0; i < 5; ++i) {
        if (v[i] >> 64) return OR_LANE_OVERFLOW;
        if ((v[i] * 8) >> 64) return OR_LANE_OVERFLOW;
        out[2 + i] = (uint64_t)v[i];
        out[7 + i] = (uint64_t)(v[i] * 8);
    }
    return OR_OK;
}
