/*
 * pa.h -- C ABI of the paged KV-cache decode library (GB300, sm_103a).
 *
 * The library implements the decode hot path of paged attention over a
 * block-paged KV cache:
 *   - the KV cache is cut into fixed-size physical blocks of 16 or 32 tokens and a
 *     per-sequence block table maps logical blocks to physical ones
 *     (gotburnout.io "PagedAttention & Gestion du KV-Cache", section 2 block-table
 *     figure; ia-vox-magazine KV-cache article, "PagedAttention : la revolution de
 *     l'allocation memoire"; deeplearn.tn KV-cache article, "Le Paged Attention");
 *   - each decode step appends the new token's key and value to its sequence's
 *     cache (blog.fabienvernieres.com "Cache KV en production", "Un cache par
 *     requete, une memoire commune") and attends from the new token's query over
 *     the cached keys and values (same page, opening section; deeplearn.tn, "Le
 *     compromis fondamental de l'inference": only the new query is needed);
 *   - sequences sharing a prefix point at the same physical blocks and a block is
 *     copied only when a sequence starts writing its own tokens (gotburnout.io,
 *     section 3.01 "Partage de prefixes (Prefix Caching / Copy-on-Write)");
 *   - an optional int8 cache with a scale recomputed for every token
 *     (ia-vox-magazine, "Quantization du KV cache").
 *
 * Conventions for every call:
 *   - Tensors are dense, row-major, and 16-byte aligned.  Device pointers are
 *     owned by the caller; the library allocates nothing and keeps no pointer
 *     after a call returns.
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).  A call returns after its kernels are queued.
 *   - pa_bf16 is a raw bfloat16 bit pattern.
 *   - Cache layout, K and V alike: [N blocks][Hkv][bs][D]; int8 scales:
 *     [N][Hkv][bs] fp32, one per (token slot, kv head).
 *   - Query head h reads kv head h / (Hq / Hkv) (grouped-query attention).
 *   - Arguments are checked on the host before anything is queued; a failed
 *     check returns a status other than PA_OK and queues nothing.  Values that
 *     live in device memory (slots, block ids, context lengths) are checked by
 *     the kernels: an offending entry is skipped (its rows are neither read nor
 *     written) and a PA_FLAG_* bit is OR-ed into *err_flag when err_flag is not
 *     NULL.  The caller reads err_flag after synchronising.
 *   - pa_last_error_string() describes the last failure of the calling thread.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t pa_bf16;

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad alignment, shape mismatch */
    PA_ERR_UNSUPPORTED = 2, /* head_dim, block size or kv dtype not compiled in */
    PA_ERR_OUT_OF_RANGE = 3, /* a host-visible index (block id, length) out of range */
    PA_ERR_CUDA = 4,         /* a CUDA launch failed; see pa_last_error_string() */
    PA_ERR_NO_SPACE = 5      /* the block pool cannot hold the request (pa_blocks.h) */
} pa_status;

enum { PA_KV_BF16 = 0, PA_KV_INT8 = 1, PA_KV_FP8 = 2 };

/* Bits OR-ed into *err_flag by the kernels. */
enum {
    PA_FLAG_SLOT_OUT_OF_RANGE = 1,    /* slot_mapping[t] >= N * bs: token not written   */
    PA_FLAG_BLOCK_OUT_OF_RANGE = 2,   /* block_tables entry outside [0, N): block skipped */
    PA_FLAG_CONTEXT_OUT_OF_RANGE = 4, /* context_lens[s] < 0, > M * bs or > max_context_len:
                                         clamped to the valid range                        */
    PA_FLAG_PREFIX_MISMATCH = 8,      /* pa_decode_shared_prefix: a group or member did not
                                         meet the prefix preconditions and was decoded on
                                         its own (the result is still correct)            */
    PA_FLAG_QUERY_OUT_OF_RANGE = 16,  /* pa_multi_token_attention: query offsets of a
                                         sequence outside [0, T], decreasing, longer than
                                         its context or than max_query_len: its rows are
                                         not written                                      */
    PA_FLAG_TIMEOUT = 32,             /* a kernel's bounded wait for its own copies or
                                         tensor-core products gave up, or its shared
                                         memory could not be laid out (the affected
                                         outputs are not written); not expected in normal
                                         operation                                        */
    PA_FLAG_FP16_RANGE = 64,          /* pa_decode_shared_prefix: an 8-bit row of a shared
                                         prefix, staged as fp16 code x scale, has a scale
                                         whose largest code leaves fp16's range (scale >
                                         65504 / 127 for int8, > 65504 / 448 for fp8): the
                                         outputs that attend it are not finite            */
    PA_FLAG_WORKSPACE_SHORT = 128     /* pa_multi_token_attention, 8-bit cache, prefill-
                                         shaped call: the workspace's dequantised pool could
                                         not hold every attended block; the blocks beyond
                                         it were read as zeros (PA_FLAG_BLOCK_OUT_OF_RANGE
                                         may be raised for them as well)                  */
};

/* Version of this ABI (bumped on any signature change). */
int pa_version(void);

/* Static text for a status code. */
const char *pa_status_string(pa_status status);

/* Message of the last failed call on this thread ("" when none). */
const char *pa_last_error_string(void);

/*
 * Append (reshape_and_cache): write the key and value rows of T new tokens into
 * their slots of a bf16 cache.
 *   key, value      [T][Hkv][D] bf16, device.
 *   k_cache,v_cache [N][Hkv][bs][D] bf16, device; row (slot / bs, h, slot % bs)
 *                   receives key[t][h] (resp. value[t][h]).
 *   slot_mapping    [T] int64, device: slot = physical block * bs + offset, i.e.
 *                   block_table[p / bs] * bs + p % bs for logical position p
 *                   (gotburnout.io block-table figure).  A negative slot marks a
 *                   padding token and is skipped.  slot >= N * bs: skipped and
 *                   PA_FLAG_SLOT_OUT_OF_RANGE raised.
 *   D in {64, 128}, bs in {16, 32}.  T == 0 is a no-op.
 * Two tokens with the same slot in one call race; the caller must not do that.
 */
pa_status pa_reshape_and_cache(const pa_bf16 *key, const pa_bf16 *value, pa_bf16 *k_cache,
                               pa_bf16 *v_cache, const int64_t *slot_mapping, int T, int Hkv,
                               int D, int bs, int N, int *err_flag, void *stream);

/*
 * Quantise-and-append into an int8 cache with a dynamic per-(token, kv head)
 * scale (ia-vox-magazine, "Quantization du KV cache": the scale is recomputed for
 * every token; 8 bits halve the cache).  For each new token t and kv head h,
 * separately for the key row and the value row x[0..D):
 *   absmax = max_d |x_d|;  scale = absmax / 127 (IEEE fp32 division), or 1 if
 *   absmax == 0;  code_d = clamp(rint(x_d / scale), -127, 127) (IEEE division,
 *   round half to even).  Dequantised value: code * scale.
 *   key, value        [T][Hkv][D] bf16, device.
 *   k_cache, v_cache  [N][Hkv][bs][D] int8, device.
 *   k_scale, v_scale  [N][Hkv][bs] fp32, device.
 *   slot_mapping etc. as in pa_reshape_and_cache.
 * Results are bit-identical to the CPU statement of the same rule for finite
 * inputs; non-finite inputs give unspecified codes.
 */
pa_status pa_quantize_kv(const pa_bf16 *key, const pa_bf16 *value, int8_t *k_cache,
                         int8_t *v_cache, float *k_scale, float *v_scale,
                         const int64_t *slot_mapping, int T, int Hkv, int D, int bs, int N,
                         int *err_flag, void *stream);

/*
 * Quantise-and-append into an fp8 (e4m3) cache with a dynamic per-(token, kv head)
 * scale: the same rule as pa_quantize_kv with scale = absmax / 448 (1 if absmax is
 * 0) and code = e4m3(x / scale) (IEEE fp32 division; round to nearest, ties to the
 * even mantissa, saturating at +-448).  The pages recommend fp8 KV caches on recent
 * GPUs (ia-vox-magazine, "Quantization du KV cache"; blog.fabienvernieres.com,
 * "Reduire le poids par token").  Caches hold raw e4m3 bytes, [N][Hkv][bs][D];
 * scales [N][Hkv][bs] fp32.  Bit-identical to the CPU statement of the rule for
 * finite inputs.
 */
pa_status pa_quantize_kv_fp8(const pa_bf16 *key, const pa_bf16 *value, uint8_t *k_cache,
                             uint8_t *v_cache, float *k_scale, float *v_scale,
                             const int64_t *slot_mapping, int T, int Hkv, int D, int bs, int N,
                             int *err_flag, void *stream);

/*
 * Copy-on-write block copy (gotburnout.io section 3.01): for each pair
 * (src, dst) copy the whole physical block src onto block dst, in the K cache and
 * in the V cache, and, when k_scale / v_scale are given, the block's scales.
 *   k_cache, v_cache   device, N blocks of block_bytes bytes each.
 *   k_scale, v_scale   device, N blocks of scale_elems_per_block fp32 each, or both
 *                      NULL (then scale_elems_per_block must be 0).
 *   block_mapping      HOST array [n][2] int64 of (src, dst) physical block ids.
 *                      It is read during the call and may be freed right after.
 *   block_bytes        multiple of 16.
 * Pairs are validated on the host: every id in [0, N) (else PA_ERR_OUT_OF_RANGE),
 * destinations pairwise distinct and no destination also a source (else
 * PA_ERR_INVALID_ARG), because the result would otherwise depend on copy order.
 */
pa_status pa_copy_blocks(void *k_cache, void *v_cache, float *k_scale, float *v_scale,
                         const int64_t *block_mapping, int n, int N, size_t block_bytes,
                         int scale_elems_per_block, void *stream);

/*
 * Bytes of device workspace pa_decode needs for these arguments (0 when the
 * contexts are short enough to need no split).  Pass the same values to
 * pa_decode.  Returns 0 for invalid arguments as well; pa_decode reports those.
 */
size_t pa_decode_workspace_size(int S, int Hq, int Hkv, int D, int bs, int kv_dtype,
                                int max_context_len);

/*
 * Paged decode attention (deeplearn.tn, "Le compromis fondamental de
 * l'inference"; blog.fabienvernieres.com, opening section): for every sequence s
 * and query head h
 *   out[s][h] = sum_t softmax_t(scale * q[s][h] . K_s[t]) V_s[t],  t < context_lens[s],
 * where K_s[t], V_s[t] are read from physical block block_tables[s][t / bs] at
 * offset t % bs, kv head h / (Hq / Hkv); int8 and fp8 entries are value * scale.  A
 * sequence with context length 0 gets an all-zero output.
 *   out             [S][Hq][D] bf16, device (written).
 *   query           [S][Hq][D] bf16, device.
 *   k_cache,v_cache [N][Hkv][bs][D], bf16 (kv_dtype PA_KV_BF16), int8 (PA_KV_INT8)
 *                   or e4m3 bytes (PA_KV_FP8).
 *   k_scale,v_scale [N][Hkv][bs] fp32 for int8 and fp8; ignored (may be NULL) for bf16.
 *   block_tables    [S][M] int32, device; entries past a sequence's last block are
 *                   never read.
 *   context_lens    [S] int32, device.
 *   max_context_len host upper bound of context_lens (0 <= it <= M * bs); longer
 *                   contexts are clamped to it and flagged.
 *   workspace       device scratch of at least pa_decode_workspace_size(...) bytes
 *                   (may be NULL when that size is 0); its contents are not
 *                   preserved.  Calls sharing a workspace must be stream-ordered.
 *   err_flag        nullable device int (see PA_FLAG_*).
 * Accumulation is fp32 (softmax statistics, dot products, weighted sums); the
 * result is rounded once to bf16.  D in {64, 128}, bs in {16, 32}.
 */
pa_status pa_decode(pa_bf16 *out, const pa_bf16 *query, const void *k_cache,
                    const void *v_cache, const float *k_scale, const float *v_scale,
                    int kv_dtype, const int32_t *block_tables, int M,
                    const int32_t *context_lens, int S, int Hq, int Hkv, int D, int bs, int N,
                    float scale, int max_context_len, void *workspace, size_t workspace_bytes,
                    int *err_flag, void *stream);

/*
 * Prefix-aware paged decode.  Same results as pa_decode (same arguments, same
 * tolerance), for a batch in which groups of consecutive sequences share a prefix:
 * the same physical blocks at the head of every member's block table, as prefix
 * caching and branching produce (ia-vox-magazine, "PagedAttention : la revolution de
 * l'allocation memoire": a shared 2000-token prompt is stored once; gotburnout.io,
 * sections 3.01 and 3.02).  Each shared block is read from HBM once per kv head for
 * the whole group instead of once per member.
 *   group_start       device [n_groups + 1] int32, non-decreasing: group g is
 *                     sequences [group_start[g], group_start[g + 1]).  Sequences in
 *                     no group are decoded as by pa_decode.
 *   group_prefix_len  device [n_groups] int32: shared prefix tokens of group g, a
 *                     positive multiple of bs, at most max_prefix_len; every member's
 *                     first group_prefix_len / bs table entries equal the first
 *                     member's, and every member's context is at least that long.
 *                     A group or member that fails these checks is decoded on its
 *                     own and PA_FLAG_PREFIX_MISMATCH is raised.
 *   max_group_size    host bound of the group sizes; max_prefix_len host bound of the
 *                     prefixes (multiple of bs, <= max_context_len).
 *   workspace         pa_decode_shared_prefix_workspace_size(...) bytes; contents
 *                     not preserved.
 * bf16, int8 and fp8 caches (k_scale, v_scale as for pa_decode).  With an 8-bit cache
 * the shared prefix is staged as fp16 code x scale and attended with fp16 products
 * (values within fp16's range); the members' own tokens go through pa_decode's exact
 * path.
 */
size_t pa_decode_shared_prefix_workspace_size(int S, int Hq, int Hkv, int D, int bs, int kv_dtype,
                                              int max_context_len, int max_group_size,
                                              int max_prefix_len);

pa_status pa_decode_shared_prefix(pa_bf16 *out, const pa_bf16 *query, const void *k_cache,
                                  const void *v_cache, const float *k_scale, const float *v_scale,
                                  int kv_dtype, const int32_t *block_tables, int M,
                                  const int32_t *context_lens, int S, int Hq, int Hkv, int D, int bs,
                                  int N, float scale, int max_context_len,
                                  const int32_t *group_start, const int32_t *group_prefix_len,
                                  int n_groups, int max_group_size, int max_prefix_len,
                                  void *workspace, size_t workspace_bytes, int *err_flag,
                                  void *stream);

/*
 * Multi-token paged attention: several new tokens per sequence attend the paged
 * cache in one call -- a chunk of a long prompt (chunked prefill) or the draft
 * tokens a large model verifies in one pass (speculative decoding): deeplearn.tn,
 * "Les leviers d'optimisation en production"; the gaiatechstar.com discussion, reply
 * on chunked prefill.  The new tokens' K and V must already be in the cache
 * (pa_reshape_and_cache with one slot per new token).
 *   query           [T][Hq][D] bf16, device: sequence s owns rows
 *                   query_start[s] .. query_start[s + 1] - 1, its L_s newest tokens in
 *                   order (varlen packing; rows of no sequence are not written).
 *   query_start     [S + 1] int32, device.
 *   context_lens    [S] int32, device: tokens in the cache including the L_s new ones.
 *   out             [T][Hq][D] bf16, device.
 *   New token i of sequence s sits at position p = context_lens[s] - L_s + i and
 *   attends positions 0 .. p (causal inside the chunk; L_s = 1 is pa_decode):
 *     out[row][h] = sum_{t <= p} softmax_t(scale * q[row][h] . k_t) v_t,
 *   k_t, v_t read through block_tables[s] from kv head h / (Hq / Hkv).
 *   max_query_len   host bound of every L_s (sizes the grid and the workspace); a
 *                   sequence with a larger L_s, offsets outside [0, T], a negative L_s or
 *                   L_s > context_lens[s] is skipped with PA_FLAG_QUERY_OUT_OF_RANGE.
 *   workspace       pa_multi_token_workspace_size(...) bytes (NULL when that is 0);
 *                   contents not preserved.
 * bf16, int8 and fp8 caches (k_scale, v_scale required for the last two); other
 * arguments as pa_decode.  With head_dim 128 and max_query_len * Hq / Hkv >= 64
 * (prefill-shaped calls), 8-bit entries of the attended blocks are first dequantised
 * into the workspace's pool as bf16 (code x scale, rounded once) and the products are bf16
 * with fp32 accumulation, as for a bf16 cache.  Otherwise the codes are converted to
 * exact fp16 values (in registers for chunks of at most 8 new tokens, through shared
 * memory for longer ones) and the query rows to fp16 scaled by a power of two; the
 * products are fp16 with fp32 accumulation, the key scale multiplies the score and the
 * value scale the softmax weight in fp32 (no range limit).
 */
size_t pa_multi_token_workspace_size(int S, int T, int Hq, int Hkv, int D, int bs, int kv_dtype,
                                     int max_context_len, int max_query_len);

/*
 * The same for a batch whose context lengths add up to at most total_context_tokens
 * (a host-side bound the caller's scheduler knows).  For prefill-shaped calls on an
 * 8-bit cache the workspace holds a bf16 pool of the attended blocks, sequences packed
 * back to back: pa_multi_token_workspace_size sizes it for every sequence at
 * max_context_len (S x ceil(max_context_len / bs) blocks), this call for the tokens
 * the batch holds (ceil(total / bs) + S blocks).  pa_multi_token_attention takes a
 * workspace of any size from the smaller of the two: its pool holds as many blocks
 * as the rest of the workspace has room for; attended blocks beyond that are read as
 * zeros and PA_FLAG_WORKSPACE_SHORT is raised.  Returns 0 for invalid arguments.
 */
size_t pa_multi_token_workspace_size_for_tokens(int S, int T, int Hq, int Hkv, int D, int bs, int kv_dtype,
                                                int max_context_len, int max_query_len,
                                                int64_t total_context_tokens);

pa_status pa_multi_token_attention(pa_bf16 *out, const pa_bf16 *query, const void *k_cache,
                                   const void *v_cache, const float *k_scale,
                                   const float *v_scale, int kv_dtype,
                                   const int32_t *block_tables, int M,
                                   const int32_t *context_lens, const int32_t *query_start,
                                   int S, int T, int Hq, int Hkv, int D, int bs, int N,
                                   float scale, int max_context_len, int max_query_len,
                                   void *workspace, size_t workspace_bytes, int *err_flag,
                                   void *stream);

/*
 * Paged decode without any allocation: the same computation, arguments and
 * results as pa_decode, for callers that cannot allocate device memory and so
 * cannot provide pa_decode's workspace (a host application that owns every
 * allocation, a fixed memory budget, or capture code that may not allocate).
 * The source pages have no counterpart: this is a packaging of pa_decode.
 *
 * The split-K scratch lives in a fixed array inside the library, of
 * PA_NOALLOC_SCRATCH_BYTES bytes per GPU; every GPU that loads the library holds
 * it until the process exits.  Sizes whose scratch (pa_decode_workspace_size)
 * exceeds it are rejected with PA_ERR_UNSUPPORTED before anything is queued; use
 * pa_decode with a caller-owned workspace for those.  The call allocates nothing
 * and calls no allocating CUDA or library routine.
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and remembers it; make that first call before any stream
 * capture.  The remembered address belongs to the device's primary context: after
 * cudaDeviceReset on that device it is stale, so do not call this entry point
 * again in a process that reset the device.  All calls on a device share the one array, so calls that overlap on
 * the GPU (on different streams, or from different threads without ordering) race
 * and may corrupt each other's results; order them on one stream.  Nothing in the
 * array needs to start at zero: each call writes every partial result it reads.
 */
#define PA_NOALLOC_SCRATCH_BYTES (16u << 20)

pa_status pa_decode_noalloc(pa_bf16 *out, const pa_bf16 *query, const void *k_cache,
                            const void *v_cache, const float *k_scale, const float *v_scale,
                            int kv_dtype, const int32_t *block_tables, int M,
                            const int32_t *context_lens, int S, int Hq, int Hkv, int D, int bs,
                            int N, float scale, int max_context_len, int *err_flag,
                            void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
