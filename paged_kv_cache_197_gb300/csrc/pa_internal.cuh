// Internal declarations shared by the translation units of the library.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// ---------------------------------------------------------------- host errors
// Records a message for pa_last_error_string() and returns `status`.
pa_status fail(pa_status status, const char *fmt, ...);
// Turns the result of the launches just made into a status.
pa_status check_launch(const char *what);

// ------------------------------------------------------------- decode planning
// Split of each sequence's context into partitions processed by separate CTAs
// and combined by a log-sum-exp merge.
struct DecodePlan {
    int part_tokens;    // tokens per partition (multiple of the block size)
    int max_parts;      // partitions of the longest allowed context
    int head_chunks;    // ceil(G / 8): query heads of one kv head are taken 8 at a time
    size_t ws_acc_off;  // byte offsets of the partial outputs and the (max, sum) pairs
    size_t ws_ml_off;
    size_t ws_bytes;    // 0 when max_parts == 1
    bool single;        // split contexts on the single-buffered kernel (three CTAs per SM)
};

// allow_single: false where the launch keeps the double-buffered kernel (the own tokens
// of a shared-prefix call).
DecodePlan plan_decode(int S, int Hq, int Hkv, int D, int bs, int kv_dtype, int max_context_len,
                       bool allow_single = true);

// Parameters of the decode and merge kernels.
struct DecodeArgs {
    uint16_t *out;
    const uint16_t *q;
    const void *k_cache;
    const void *v_cache;
    const float *k_scale;
    const float *v_scale;
    const int32_t *block_tables;
    const int32_t *context_lens;
    float *ws_acc;  // [S][Hq][max_parts][D]
    float *ws_ml;   // [S][Hq][max_parts][2]
    int *err_flag;
    int M, S, Hq, Hkv, G, N;
    int head_chunks, part_tokens, max_parts;
    int max_context_len;  // host bound; longer contexts are clamped and flagged
    float scale_log2;  // softmax scale times log2(e)
    const int32_t *start_tokens;  // nullable [S]: tokens to skip (a shared prefix)
    int partials_only;            // write partial results even for a single partition
    int single;                   // decode on the single-buffered kernel (DecodePlan::single)
    // Rows mode (multi-token attention of narrow chunks): non-null [S + 1] row ranges
    // of T query rows.  A CTA takes rows_per_cta consecutive new tokens of a sequence
    // (grid x is partition x token group); token i of sequence s (row query_start[s] +
    // i) attends the first ctx - L + i + 1 tokens, and q, out and the partials
    // [T][Hq][max_parts] are indexed by that row.
    const int32_t *query_start;
    int T, Lq, rows_per_cta;
};

// Shared-prefix decode: groups of consecutive sequences whose block tables start with
// the same prefix blocks.
struct PrefixArgs {
    const int32_t *group_start;   // [n_groups + 1]: group g = sequences [start[g], start[g+1])
    const int32_t *group_prefix;  // [n_groups]: shared prefix tokens (multiple of bs)
    int n_groups, max_group_size, max_prefix;
    int32_t *seq_start;           // [S] workspace: prefix tokens each sequence skips
    int32_t *seq_group;           // [S] workspace: its group, or -1
    float *pacc;                  // [S][Hq][PP][D] prefix partials
    float *pml;                   // [S][Hq][PP][2]
    int PP;                       // prefix chunks of the longest prefix
    int CB;                       // blocks of 128 query columns per kv head
    int chunk;                    // prefix tokens per partial (prefix_chunk_tokens)
};

// Prefix tokens per grouped partial: 256 on the tcgen05 path (bf16, head_dim 128),
// else 128 (the mma.sync grouped kernel stages one chunk in shared memory).
int prefix_chunk_tokens(int kv_dtype, int D);
int prefix_cols_per_cta();
cudaError_t launch_decode_shared_prefix(const DecodeArgs &a, const PrefixArgs &p, int D, int bs, int kv_dtype,
                                        cudaStream_t stream);

// Multi-token attention: the newest L_s tokens of each sequence attend the cache.
struct MultiArgs {
    uint16_t *out;                 // [T][Hq][D] bf16
    const uint16_t *q;             // [T][Hq][D] bf16
    const void *k_cache, *v_cache;
    const float *k_scale, *v_scale;  // int8 / fp8 caches: [N][Hkv][bs]
    const int32_t *block_tables, *context_lens;
    const int32_t *query_start;    // [S + 1]: rows of sequence s
    float *ws_acc, *ws_ml;         // [T][Hq][max_parts][D], [T][Hq][max_parts][2]
    int *err_flag;
    int M, S, T, Hq, Hkv, G, N;
    int g_shift;                   // log2(G) when G is a power of two, else -1
    int CB;                        // blocks of 128 (token, head) columns per kv head
    int part_tokens, max_parts;    // context partitions (multiple of 64 tokens)
    int max_context_len, max_query_len;
    float scale_log2;
    // Group mode (the tcgen05 kernel only; shared-prefix decode): non-null [S] prefix
    // lengths of S groups whose members are the query rows query_start[g] ..
    // query_start[g + 1] - 1 of the decode queries [T][Hq][D]; every member attends
    // all of its group's prefix through the first member's block table, no causal
    // mask, and every column leaves a partial (no direct output).  seq_group [T]: a
    // member whose entry is not g is left out.
    const int32_t *group_prefix;
    const int32_t *seq_group;
};

int multi_cols_per_cta();
cudaError_t launch_multi_token(const MultiArgs &a, int D, int bs, int kv_dtype, cudaStream_t stream);
// The log-sum-exp merge of multi-token partials (a programmatic dependent launch).
cudaError_t launch_multi_merge(const MultiArgs &a, int D, int bs, cudaStream_t stream);
// Whether a multi-token call runs on the decode kernel in rows mode (a CTA per one or
// two new tokens, a kv head's token groups side by side so they share K/V through
// L2); plan and launch both follow it.
bool multi_per_token_eligible(int D, int kv_dtype, int G, int max_query_len);
// The decode kernel alone in rows mode, 8-bit caches (a programmatic dependent
// launch); the caller launches the merge.  decode_rows_per_cta: the new tokens one
// CTA takes for a call of max_query_len new tokens per sequence.
int decode_rows_per_cta(int max_query_len);
// CTAs per SM of the single-buffered decode kernel (its launch bounds) for a cache type.
int decode_single_ctas_per_sm(int kv_dtype);
cudaError_t launch_decode_rows(const DecodeArgs &a, int D, int bs, int kv_dtype, cudaStream_t stream);
// Whether multi-token attention of this shape runs on the tcgen05 kernel (8-bit caches
// after the dequantising pass below) rather than the mma.sync one; plan and launch both
// follow it.
bool multi_tc_eligible(int D, int kv_dtype, int G, int max_query_len);
cudaError_t launch_multi_tc(const MultiArgs &a, int bs, cudaStream_t stream);  // bf16 caches
// The tcgen05 kernel in group mode (the caller merges the partials).
cudaError_t launch_multi_tc_groups(const MultiArgs &a, int bs, cudaStream_t stream);
int multi_tc_rows();  // (token or member, head) columns per CTA of the tcgen05 kernel
// 8-bit caches, prefill-shaped calls: the attended blocks dequantised into a bf16 pool
// of `cap` blocks, sequences packed back to back (offsets off[S + 1]), and the table
// [S][Mq] of pool slots, all in the workspace.
cudaError_t launch_dequant_blocks(const MultiArgs &a, int bs, int kv_dtype, int Mq, uint16_t *kq, uint16_t *vq,
                                  int32_t *tab, int32_t *off, int64_t cap, cudaStream_t stream);

// Launch `kernel` as a programmatic dependent of the kernel before it on `stream`: it
// may be scheduled while that kernel drains, and must execute griddepcontrol.wait
// before it reads or writes anything that kernel may touch.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args &&...args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// ------------------------------------------------------------------ launchers
// Each returns the CUDA error of its launch (cudaSuccess when nothing was launched).
cudaError_t launch_reshape_and_cache(const uint16_t *key, const uint16_t *value, uint16_t *k_cache,
                                     uint16_t *v_cache, const int64_t *slot_mapping, int T,
                                     int Hkv, int D, int bs, int N, int *err_flag,
                                     cudaStream_t stream);
cudaError_t launch_quantize_kv(const uint16_t *key, const uint16_t *value, int8_t *k_cache,
                               int8_t *v_cache, float *k_scale, float *v_scale,
                               const int64_t *slot_mapping, int T, int Hkv, int D, int bs, int N,
                               int *err_flag, cudaStream_t stream);
cudaError_t launch_quantize_kv_fp8(const uint16_t *key, const uint16_t *value, uint8_t *k_cache,
                                   uint8_t *v_cache, float *k_scale, float *v_scale,
                                   const int64_t *slot_mapping, int T, int Hkv, int D, int bs,
                                   int N, int *err_flag, cudaStream_t stream);
cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, float *k_scale, float *v_scale,
                               const int64_t *block_mapping, int n, size_t block_bytes,
                               int scale_elems_per_block, cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs &args, int D, int bs, int kv_dtype,
                          cudaStream_t stream);

}  // namespace pa
