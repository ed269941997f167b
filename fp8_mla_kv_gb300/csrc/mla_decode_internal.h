// Internal interface between the decode entry points and the 64-head kernel.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace mla_host {

// A validated decode call (device pointers; layouts as in the C header).
struct DecodeCall {
    const void* q;              // bf16 [T, H, d_qk]
    const uint8_t* cache;       // packed rows
    const int32_t* topk;        // [T, W] slots, or sequence positions when page_size > 0
    void* out;                  // bf16 [T, H, 512]
    float* lse;                 // [T, H]
    float* ws_o;                // [T, nsplit, H, 512] normalised partials (nsplit > 1)
    float* ws_lse;              // [T, nsplit, H]
    int* err;                   // device error word
    int64_t num_slots;
    int64_t row_bytes;          // 656, or 528 (NoPE rows without a tail)
    const int32_t* block_table; // [n_seq, bt_pages] (page_size > 0)
    const int32_t* token_seq;   // [T] or null
    int bt_pages, n_seq, page_size;
    int T, H, d_qk, W, nsplit;
    // split by positions (split_len each) or, when rank_chunk > 0, by present entries
    int split_len, rank_chunk;
    float sm_scale_log2;        // sm_scale * log2(e)
};

// Splits of each token's list for the 64-head kernel (H a multiple of 64).
int choose_nsplit_h64(int T, int H, int W, int sms);
int rank_chunk_h64(int W, int nsplit);
// Launches the 64-head kernel (PDL-serialised behind the previous kernel on the
// stream); the caller launches the split merge when nsplit > 1.
int launch_decode_h64(const DecodeCall& c, cudaStream_t stream);

}  // namespace mla_host
