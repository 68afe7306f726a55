// pa_internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// Records a message for pa_last_error() and returns `st`.
pa_status fail(pa_status st, const char* fmt, ...);
// Maps a CUDA error to PA_ERR_CUDA with the call site in the message.
pa_status cuda_fail(cudaError_t e, const char* what);
void count_launch();
// Limit of the main in-kernel waits for launches made now (pa_set_wait_limit_ns; default 1 s).
uint64_t wait_limit_ns();

// ----------------------------------------------------------------------------- cache ops

pa_status launch_reshape_and_cache(const void* k, const void* v, void* pool, const int64_t* slot_mapping, int T,
                                   int NB, int B, int H_kv, int D, int* dev_err, cudaStream_t stream);
pa_status launch_write_contiguous(const void* k, const void* v, void* k_buf, void* v_buf, const int32_t* req_ids,
                                  const int32_t* positions, int T, int N_max, int S, int H_kv, int D, int* dev_err,
                                  cudaStream_t stream);
pa_status launch_swap_blocks(void* dst, int NB_dst, const void* src, int NB_src, const int64_t* pairs, int n,
                             int64_t blk_bytes, int* dev_err, cudaStream_t stream);
pa_status launch_update_tables(int32_t* tables, int N, int MB, const int32_t* updates, int n, int* dev_err,
                               cudaStream_t stream);
pa_status launch_copy_blocks(void* pool, const int64_t* pairs, int n, int NB, int B, int H_kv, int D, int* dev_err,
                             cudaStream_t stream);

// ----------------------------------------------------------------------------- decode

constexpr int kStageTok = 32;         // tokens of one KV head per pipeline stage
constexpr int kMaxGroup = 8;          // query heads per KV head (mma N = 8)
constexpr int kDefaultPartition = 512;
constexpr int kUnpartitioned = 1 << 30;

struct WorkspaceLayout {
    size_t header;     // int[4]: record count, spare
    size_t nparts;     // int[N]: partitions per sequence (0 for an invalid one)
    size_t records;    // int4[N * P * H_kv]
    size_t part_m2;    // float[N * H_q * P]
    size_t part_l;     // float[N * H_q * P]
    size_t part_acc;   // float[N * H_q * P * D]
    size_t total;
    int P;             // partitions per sequence (stride)
    int PT;            // tokens per partition (kUnpartitioned when off)
};

// Returns false for invalid arguments.
bool workspace_layout(int N, int H_q, int H_kv, int D, int max_ctx, int partition_tokens, WorkspaceLayout* out);

struct DecodeArgs {
    void* out;
    int out_dtype;         // pa_dtype
    const void* q;
    int kv_dtype;          // pa_dtype
    // paged source
    const void* pool;
    const int32_t* tables;
    int B, MB, NB;
    // contiguous source
    const void* k_buf;
    const void* v_buf;
    const int32_t* req_ids;
    int N_max, S_max;
    bool paged;
    const int32_t* ctx_lens;
    int N, H_q, H_kv, D, max_ctx;
    float scale;
    int partition_tokens;
    void* workspace;
    size_t ws_bytes;
    int* dev_err;
    void* const* attend_events;
    cudaStream_t stream;
};

pa_status launch_decode(const DecodeArgs& a);

struct PrefillArgs {
    void* out;
    int out_dtype;
    const void* q;
    const void* pool;
    const int32_t* tables;
    const int32_t* ctx_lens;
    const int32_t* q_start;
    int N, T, H_q, H_kv, D, B, MB, NB, max_q_len;
    float scale;
    int kv_dtype;
    void* workspace;  // nullable: V staging area for bf16 caches
    size_t ws_bytes;
    int* dev_err;
    cudaStream_t stream;
};

struct PrefillWorkspace {
    int S_pad;     // keys per staged (sequence, KV head) row: MB * B rounded up to the 128-key tile
    size_t split;  // offset of the per-(sequence, KV head) marks (after the staged V)
    size_t total;
};

// Returns false for invalid arguments.
bool prefill_workspace_layout(int N, int H_kv, int D, int B, int MB, PrefillWorkspace* out);
pa_status launch_prefill(const PrefillArgs& a);

pa_status launch_partition_reduce(void* out, int out_dtype, const float* m2, const float* l, const float* acc,
                                  const int32_t* nparts, int rows_per_seq, int R, int P, int D, bool skip_single,
                                  int* dev_err, cudaStream_t stream);
bool pdl_enabled();

}  // namespace pa
