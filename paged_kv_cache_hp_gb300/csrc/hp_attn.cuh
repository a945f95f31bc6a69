// hp_attn.cuh -- the launch interface of decode attention (hp_attention.cu), kept apart
// from hp_internal.cuh so that the copy engines' sources do not depend on it.
#pragma once

#include <cstdint>

#include "hp_internal.cuh"

namespace hp {

// Decode attention (hp_attention.cu), after a kPlanAttention plan on the same stream.
struct AttnArgs {
    const void* k_pool;
    const void* v_pool;
    const void* q;            // [num_seqs, Hq, D]
    const void* table;
    const void* seq_ptr;
    const void* lens;
    uint64_t num_seqs, page_size, num_pages, table_len;
    uint32_t Hkv, Hq, D, G;   // G = Hq / Hkv query heads per K/V head
    uint32_t p_m, p_l;        // div_invariant constants of page_size
    uint32_t R;               // workers per CTA: step ranges a CTA splits among its warps
    uint64_t workers;         // CTAs * R
    float scale;
    const WsHeader* hdr;
    const unsigned long long* units_off;  // steps per sequence, prefix
    float* part_acc;          // [records, G, D]: each segment's weighted value sums
    float* part_ml;           // [records, G, 2]: its score maximum and weight sum
    unsigned* seg_done;       // [num_seqs, Hkv]: segments finished; zero at launch and
                              // again when the launch ends
    float* out;               // [num_seqs, Hq, D] fp32
    int elem_bf16;            // element type: bf16 (1) or f16 (0)
    int test_stall;           // HP_TEST_STALL: the tensor-core kernel never issues its
                              // first K load
    int pair;                 // tensor cores, head_dim 64 taken as pairs of K/V heads: Hkv,
                              // G and D describe the pairs (D = 128), q the padded queries,
                              // out keeps 64 dims per query head
    uint32_t Hkv_row;         // tensor cores, one group of K/V heads per launch: the heads of
                              // a pool row (k_pool, v_pool point at the group's first head);
                              // 0 = Hkv
    uint32_t Hq_row;          // and the query heads of a sequence in q and out (both point at
                              // the group's first query head); 0 = Hq
    int* d_status;
};
int launch_attention(int index_u64, const AttnArgs& a, void* stream);

// Decode attention on the tensor cores (hp_attn_tc.cu): head_dim 128, K and V in device
// memory, H_kv in {1, 2, 4, 8} K/V heads, G in {1, 2, 4, 8} query heads per K/V head with
// at most 32 query heads, pages of 8 .. 128 / H_kv slots (a power of two); a step is
// attention_tc_step_tokens(H_kv) = 128 / H_kv tokens of a sequence and all its K/V heads.
// Head_dim 64 runs as pairs of K/V heads (AttnArgs::pair): the queries are first written,
// zero-padded to 128 dims in their head's half, by launch_attention_qpad.  More than 32 query
// heads run as groups of K/V heads, one launch each (AttnArgs::Hkv_row, Hq_row).
bool attention_tc_fits(uint64_t head_dim, uint64_t page_size, uint64_t num_pages, bool host_memory,
                       uint64_t num_kv_heads, uint64_t num_q_heads);
uint64_t attention_tc_step_tokens(uint64_t num_kv_heads);
int launch_attention_tc(int index_u64, const AttnArgs& a, void* stream);
// q [num_seqs, Hq, 64] (16-bit) -> qpad [num_seqs, Hq, 128]: query head qh (K/V head
// qh / G) in dims 64 * ((qh / G) % 2) .. + 64, zeros in the other half.
int launch_attention_qpad(const void* q, void* qpad, uint64_t num_seqs, uint32_t Hq, uint32_t G,
                          void* stream);


}  // namespace hp
