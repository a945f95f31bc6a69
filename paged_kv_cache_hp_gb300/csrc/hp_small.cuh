// hp_small.cuh -- the launch interface of the one-launch gather of a small validated batch
// (hp_small.cu).
#pragma once

#include <cstdint>

#include "hp_internal.cuh"

namespace hp {

// Limits of the one-launch path: every CTA rescans this much index data.
constexpr uint64_t kMaxSeqs = 1024;
constexpr uint64_t kMaxTable = 8192;
constexpr uint64_t kMaxBytes = 8ull << 20;  // table_len * page_size * row bytes

struct SmallGatherArgs {
    const void* seq_ptr;
    const void* lens;
    const void* table;
    const char* pool;
    char* out;
    uint64_t num_seqs, page_size, table_len, num_pages, row_bytes;
    uint64_t out_tokens;  // the expected total rows
    WsView ws;            // the plan's workspace, filled as the plan would
    int* d_status;
};

int launch_small_gather(int index_u64, const SmallGatherArgs& a, int vec, void* stream);

}  // namespace hp
