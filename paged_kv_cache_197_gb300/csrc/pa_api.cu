// C-ABI entry points: host-side argument checks, planning and kernel launches.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "pa_internal.cuh"

namespace pa {

static thread_local char g_last_error[512] = "";

pa_status fail(pa_status status, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return status;
}

pa_status check_launch(const char *what) {
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess)
        return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(err));
    return PA_OK;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Split of long contexts: each CTA handles one partition of one (sequence, kv head,
// query-head chunk) unit.  A CTA pays a pipeline ramp-up (its first tiles' latency,
// worth about 64 tokens of streaming) and a partial result per head, so long
// partitions are cheaper; but the grid must hold at least three waves of CTAs
// (2 resident per SM), and a last wave that is mostly empty wastes the difference.
// Each candidate length is scored by (fraction of the last wave in use) x
// (length / (length + 64)) for the longest context, and the best is taken.
// When the units alone give six waves and contexts are at most 4096 tokens there is
// no split at all (no merge launch).  Measured on GB300 for Llama-2-13B-shaped decode:
// 512-token partitions 6.15 TB/s, one 2048-token partition 6.55 TB/s; Llama-3-70B-
// shaped: 1024 -> 5.67, 768 -> 5.71.
constexpr int kPartChoices[] = {4096, 3072, 2048, 1536, 1024, 768, 512, 384, 256};
constexpr int kRampTokens = 64;
constexpr double kSingleRampTokens = 512.0;  // the single-buffered kernel's (see plan_decode)
constexpr int kCtasPerSm = 2;

static int device_sms() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();  // no device here: plan for GB300's 152 SMs
        return 152;
    }
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 152;
        }
        cached[dev] = n;
    }
    return cached[dev];
}

DecodePlan plan_decode(int S, int Hq, int Hkv, int D, int bs, int kv_dtype, int max_context_len,
                       bool allow_single) {
    (void)bs;
    DecodePlan p{};
    const int G = Hq / Hkv;
    p.head_chunks = (G + 7) / 8;
    const int64_t units = (int64_t)S * Hkv * p.head_chunks;
    const double slots = (double)device_sms() * kCtasPerSm;
    p.part_tokens = kPartChoices[sizeof(kPartChoices) / sizeof(int) - 1];
    double best = -1.0;
    if ((double)units >= 6.0 * slots && max_context_len <= 4096) {
        // enough units of bounded length to keep every SM busy: no split, no merge
        p.part_tokens = std::max(max_context_len, 1);
        best = 1.0;
    }
    for (int cand : kPartChoices) {
        if (best >= 1.0) break;
        const int64_t parts = std::max<int64_t>(1, (max_context_len + cand - 1) / cand);
        const double waves = (double)(units * parts) / slots;
        if (waves < 3.0) continue;
        const double fill = waves / std::ceil(waves);
        const double len = (double)std::min(cand, std::max(max_context_len, 1));
        const double score = fill * len / (len + kRampTokens);
        if (score > best + 1e-9) {
            best = score;
            p.part_tokens = cand;
        }
    }
    p.max_parts = std::max(1, (max_context_len + p.part_tokens - 1) / p.part_tokens);
    p.single = false;
    if (allow_single && p.max_parts > 1 && kv_dtype != PA_KV_FP8) {
        // Split contexts of bf16 and int8 caches: the single-buffered kernel, four (bf16)
        // or three (int8) CTAs per SM.  Its CTAs expose each tile's load latency and rely on the other warps,
        // so fewer, longer partitions pay: n balanced partitions of the longest context
        // (as in the multi-token plan) scored by (last-wave fill) x len / (len + 512)
        // with at least 1.5 waves.  Measured on GB300, 70B-shaped decode (8 layers,
        // four CTAs per SM, 608 slots): 1152-token partitions (1.84 waves) 106.6 us,
        // 768 (2.9) 108.8, 1344 111.9, 512 114.1, 640 115.4, 1024 (2.1 waves) 121.3 --
        // the order of the score.
        p.single = true;
        const double slots3 = (double)device_sms() * decode_single_ctas_per_sm(kv_dtype);
        const int ctx = std::max(max_context_len, 1);
        double best = -1.0;
        int best_len = p.part_tokens;
        for (int n = 1; n <= (ctx + 255) / 256; ++n) {
            const int cand = std::min(4096, std::max(256, (int)align_up((size_t)((ctx + n - 1) / n), 64)));
            const int parts = (ctx + cand - 1) / cand;
            if (parts != n) continue;  // the same length as a smaller n
            const double waves = (double)(units * parts) / slots3;
            if (waves < 1.5 && cand != 256) continue;
            const double len = (double)std::min(cand, ctx);
            const double score = waves / std::ceil(waves) * len / (len + kSingleRampTokens);
            if (score > best + 1e-9) {
                best = score;
                best_len = cand;
            }
        }
        p.part_tokens = best_len;
        p.max_parts = std::max(1, (max_context_len + p.part_tokens - 1) / p.part_tokens);
        if (p.max_parts == 1) p.single = false;
    }
    if (p.max_parts == 1) {
        p.ws_acc_off = p.ws_ml_off = p.ws_bytes = 0;
        return p;
    }
    const size_t rows = (size_t)S * Hq * p.max_parts;
    p.ws_acc_off = 0;
    p.ws_ml_off = align_up(rows * D * sizeof(float), 256);
    p.ws_bytes = align_up(p.ws_ml_off + rows * 2 * sizeof(float), 256);
    return p;
}

}  // namespace pa

using namespace pa;

extern "C" {

int pa_version(void) { return 1; }

const char *pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported configuration";
        case PA_ERR_OUT_OF_RANGE: return "index out of range";
        case PA_ERR_CUDA: return "CUDA error";
        case PA_ERR_NO_SPACE: return "block pool exhausted";
    }
    return "unknown status";
}

const char *pa_last_error_string(void) { return g_last_error; }

static pa_status check_cache_shape(const char *fn, int Hkv, int D, int bs, int N) {
    if (Hkv <= 0 || N <= 0)
        return fail(PA_ERR_INVALID_ARG, "%s: Hkv (%d) and N (%d) must be positive", fn, Hkv, N);
    if (D != 64 && D != 128)
        return fail(PA_ERR_UNSUPPORTED, "%s: head_dim %d not supported (64 or 128)", fn, D);
    if (bs != 16 && bs != 32)
        return fail(PA_ERR_UNSUPPORTED, "%s: block size %d not supported (16 or 32)", fn, bs);
    if ((int64_t)N * bs > (int64_t)1 << 40)
        return fail(PA_ERR_INVALID_ARG, "%s: pool too large", fn);
    return PA_OK;
}

pa_status pa_reshape_and_cache(const pa_bf16 *key, const pa_bf16 *value, pa_bf16 *k_cache,
                               pa_bf16 *v_cache, const int64_t *slot_mapping, int T, int Hkv,
                               int D, int bs, int N, int *err_flag, void *stream) {
    const char *fn = "pa_reshape_and_cache";
    g_last_error[0] = 0;
    if (T < 0) return fail(PA_ERR_INVALID_ARG, "%s: T = %d is negative", fn, T);
    pa_status st = check_cache_shape(fn, Hkv, D, bs, N);
    if (st != PA_OK) return st;
    if (T == 0) return PA_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping)
        return fail(PA_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", fn);
    if ((int64_t)T * Hkv * D > ((int64_t)1 << 40))
        return fail(PA_ERR_INVALID_ARG, "%s: too many tokens", fn);
    launch_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, T, Hkv, D, bs, N,
                             err_flag, (cudaStream_t)stream);
    return check_launch(fn);
}

pa_status pa_quantize_kv(const pa_bf16 *key, const pa_bf16 *value, int8_t *k_cache,
                         int8_t *v_cache, float *k_scale, float *v_scale,
                         const int64_t *slot_mapping, int T, int Hkv, int D, int bs, int N,
                         int *err_flag, void *stream) {
    const char *fn = "pa_quantize_kv";
    g_last_error[0] = 0;
    if (T < 0) return fail(PA_ERR_INVALID_ARG, "%s: T = %d is negative", fn, T);
    pa_status st = check_cache_shape(fn, Hkv, D, bs, N);
    if (st != PA_OK) return st;
    if (T == 0) return PA_OK;
    if (!key || !value || !k_cache || !v_cache || !k_scale || !v_scale || !slot_mapping)
        return fail(PA_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(k_scale) || !aligned16(v_scale))
        return fail(PA_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", fn);
    launch_quantize_kv(key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, T, Hkv, D,
                       bs, N, err_flag, (cudaStream_t)stream);
    return check_launch(fn);
}

pa_status pa_quantize_kv_fp8(const pa_bf16 *key, const pa_bf16 *value, uint8_t *k_cache,
                             uint8_t *v_cache, float *k_scale, float *v_scale,
                             const int64_t *slot_mapping, int T, int Hkv, int D, int bs, int N,
                             int *err_flag, void *stream) {
    const char *fn = "pa_quantize_kv_fp8";
    g_last_error[0] = 0;
    if (T < 0) return fail(PA_ERR_INVALID_ARG, "%s: T = %d is negative", fn, T);
    pa_status st = check_cache_shape(fn, Hkv, D, bs, N);
    if (st != PA_OK) return st;
    if (T == 0) return PA_OK;
    if (!key || !value || !k_cache || !v_cache || !k_scale || !v_scale || !slot_mapping)
        return fail(PA_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(k_scale) || !aligned16(v_scale))
        return fail(PA_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", fn);
    launch_quantize_kv_fp8(key, value, k_cache, v_cache, k_scale, v_scale, slot_mapping, T, Hkv, D,
                           bs, N, err_flag, (cudaStream_t)stream);
    return check_launch(fn);
}

pa_status pa_copy_blocks(void *k_cache, void *v_cache, float *k_scale, float *v_scale,
                         const int64_t *block_mapping, int n, int N, size_t block_bytes,
                         int scale_elems_per_block, void *stream) {
    const char *fn = "pa_copy_blocks";
    g_last_error[0] = 0;
    if (n < 0 || N <= 0) return fail(PA_ERR_INVALID_ARG, "%s: n = %d, N = %d", fn, n, N);
    if (n == 0) return PA_OK;
    if (!k_cache || !v_cache || !block_mapping)
        return fail(PA_ERR_INVALID_ARG, "%s: null pointer", fn);
    if ((k_scale == nullptr) != (v_scale == nullptr))
        return fail(PA_ERR_INVALID_ARG, "%s: give both scale arrays or neither", fn);
    if ((k_scale == nullptr) != (scale_elems_per_block == 0) || scale_elems_per_block < 0)
        return fail(PA_ERR_INVALID_ARG, "%s: scale_elems_per_block = %d does not match the scale arrays",
                    fn, scale_elems_per_block);
    if (block_bytes == 0 || block_bytes % 16 != 0)
        return fail(PA_ERR_INVALID_ARG, "%s: block_bytes = %zu must be a positive multiple of 16", fn,
                    block_bytes);
    if (!aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "%s: caches must be 16-byte aligned", fn);
    std::vector<int64_t> dst(n), src(n);
    for (int i = 0; i < n; ++i) {
        src[i] = block_mapping[2 * i];
        dst[i] = block_mapping[2 * i + 1];
        if (src[i] < 0 || src[i] >= N || dst[i] < 0 || dst[i] >= N)
            return fail(PA_ERR_OUT_OF_RANGE, "%s: pair %d (%lld -> %lld) outside [0, %d)", fn, i,
                        (long long)src[i], (long long)dst[i], N);
    }
    std::vector<int64_t> ds(dst), ss(src);
    std::sort(ds.begin(), ds.end());
    std::sort(ss.begin(), ss.end());
    for (int i = 1; i < n; ++i)
        if (ds[i] == ds[i - 1])
            return fail(PA_ERR_INVALID_ARG, "%s: block %lld is the destination of two pairs", fn,
                        (long long)ds[i]);
    for (int i = 0; i < n; ++i)
        if (std::binary_search(ss.begin(), ss.end(), dst[i]))
            return fail(PA_ERR_INVALID_ARG, "%s: block %lld is both a source and a destination", fn,
                        (long long)dst[i]);
    launch_copy_blocks(k_cache, v_cache, k_scale, v_scale, block_mapping, n, block_bytes,
                       scale_elems_per_block, (cudaStream_t)stream);
    return check_launch(fn);
}

static pa_status check_decode_shape(const char *fn, int S, int Hq, int Hkv, int D, int bs,
                                    int kv_dtype, int max_context_len) {
    if (S < 0 || Hq <= 0 || Hkv <= 0)
        return fail(PA_ERR_INVALID_ARG, "%s: S = %d, Hq = %d, Hkv = %d", fn, S, Hq, Hkv);
    if (Hq % Hkv != 0)
        return fail(PA_ERR_INVALID_ARG, "%s: Hq (%d) must be a multiple of Hkv (%d)", fn, Hq, Hkv);
    if (D != 64 && D != 128)
        return fail(PA_ERR_UNSUPPORTED, "%s: head_dim %d not supported (64 or 128)", fn, D);
    if (bs != 16 && bs != 32)
        return fail(PA_ERR_UNSUPPORTED, "%s: block size %d not supported (16 or 32)", fn, bs);
    if (kv_dtype != PA_KV_BF16 && kv_dtype != PA_KV_INT8 && kv_dtype != PA_KV_FP8)
        return fail(PA_ERR_UNSUPPORTED, "%s: kv dtype %d not supported", fn, kv_dtype);
    if (max_context_len < 0)
        return fail(PA_ERR_INVALID_ARG, "%s: max_context_len = %d", fn, max_context_len);
    if (S > 65535)
        return fail(PA_ERR_UNSUPPORTED, "%s: at most 65535 sequences per call (got %d)", fn, S);
    if ((int64_t)Hkv * ((Hq / Hkv + 7) / 8) > 65535)
        return fail(PA_ERR_UNSUPPORTED, "%s: too many heads", fn);
    return PA_OK;
}

size_t pa_decode_workspace_size(int S, int Hq, int Hkv, int D, int bs, int kv_dtype,
                                int max_context_len) {
    if (check_decode_shape("pa_decode_workspace_size", S, Hq, Hkv, D, bs, kv_dtype,
                           max_context_len) != PA_OK)
        return 0;
    return plan_decode(S, Hq, Hkv, D, bs, kv_dtype, max_context_len).ws_bytes;
}

pa_status pa_decode(pa_bf16 *out, const pa_bf16 *query, const void *k_cache,
                    const void *v_cache, const float *k_scale, const float *v_scale,
                    int kv_dtype, const int32_t *block_tables, int M,
                    const int32_t *context_lens, int S, int Hq, int Hkv, int D, int bs, int N,
                    float scale, int max_context_len, void *workspace, size_t workspace_bytes,
                    int *err_flag, void *stream) {
    const char *fn = "pa_decode";
    g_last_error[0] = 0;
    pa_status st = check_decode_shape(fn, S, Hq, Hkv, D, bs, kv_dtype, max_context_len);
    if (st != PA_OK) return st;
    if (S == 0) return PA_OK;
    if (N <= 0 || M <= 0)
        return fail(PA_ERR_INVALID_ARG, "%s: N = %d, M = %d must be positive", fn, N, M);
    if ((int64_t)max_context_len > (int64_t)M * bs)
        return fail(PA_ERR_OUT_OF_RANGE, "%s: max_context_len %d exceeds M * bs = %lld", fn,
                    max_context_len, (long long)M * bs);
    if (!out || !query || !k_cache || !v_cache || !block_tables || !context_lens)
        return fail(PA_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (kv_dtype != PA_KV_BF16 && (!k_scale || !v_scale))
        return fail(PA_ERR_INVALID_ARG, "%s: int8 / fp8 caches need k_scale and v_scale", fn);
    if (kv_dtype != PA_KV_BF16 && (!aligned16(k_scale) || !aligned16(v_scale)))
        return fail(PA_ERR_INVALID_ARG, "%s: scales must be 16-byte aligned", fn);
    if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", fn);
    if (!(scale == scale) || scale == __builtin_inff() || scale == -__builtin_inff())
        return fail(PA_ERR_INVALID_ARG, "%s: scale must be finite", fn);
    const DecodePlan plan = plan_decode(S, Hq, Hkv, D, bs, kv_dtype, max_context_len);
    if (plan.ws_bytes > 0) {
        if (!workspace || workspace_bytes < plan.ws_bytes)
            return fail(PA_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed, %zu given", fn,
                        plan.ws_bytes, workspace ? workspace_bytes : (size_t)0);
        if (!aligned16(workspace))
            return fail(PA_ERR_INVALID_ARG, "%s: workspace must be 16-byte aligned", fn);
    }
    DecodeArgs a{};
    a.out = out;
    a.q = query;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.ws_acc = plan.ws_bytes ? (float *)((char *)workspace + plan.ws_acc_off) : nullptr;
    a.ws_ml = plan.ws_bytes ? (float *)((char *)workspace + plan.ws_ml_off) : nullptr;
    a.err_flag = err_flag;
    a.M = M;
    a.S = S;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.N = N;
    a.head_chunks = plan.head_chunks;
    a.part_tokens = plan.part_tokens;
    a.max_parts = plan.max_parts;
    a.single = plan.single;
    a.max_context_len = max_context_len;
    a.scale_log2 = scale * 1.4426950408889634f;
    launch_decode(a, D, bs, kv_dtype, (cudaStream_t)stream);
    return check_launch(fn);
}

constexpr int kShortOwnTokens = 1024;

// Workspace of the shared-prefix decode: per-sequence start and group, prefix
// partials per 128-token chunk, own-token partials per partition.
struct PrefixPlan {
    DecodePlan own;
    int PP, CB, MP, chunk;
    size_t start_off, group_off, pacc_off, pml_off, acc_off, ml_off, bytes;
};

static PrefixPlan plan_prefix(int S, int Hq, int Hkv, int D, int bs, int kv_dtype, int max_context_len,
                              int max_group_size, int max_prefix_len) {
    PrefixPlan p{};
    // the own tokens of a member of a group with the longest prefix number at most
    // max_context_len - max_prefix_len: partitions are sized for that length; longer
    // own ranges (shorter prefixes, sequences in no group) just take more partitions
    const int own_len = std::max(1, max_context_len - max_prefix_len);
    p.own = plan_decode(S, Hq, Hkv, D, bs, kv_dtype, own_len, false);
    // short own ranges run next to the grouped prefix kernel, which fills the GPU as
    // well: one partition each (one partial per head for the merge) beats splitting
    // them further (measured: 512-token ranges 48.8 us in one, 52.9 us in 256-token
    // partitions, 59.0 us in 128-token ones)
    if (own_len <= kShortOwnTokens) p.own.part_tokens = own_len;
    p.own.part_tokens = (int)align_up((size_t)p.own.part_tokens, 64);  // whole tiles and blocks
    p.MP = std::max(1, (max_context_len + p.own.part_tokens - 1) / p.own.part_tokens);
    const int chunk = prefix_chunk_tokens(kv_dtype, D);
    p.chunk = chunk;
    p.PP = (max_prefix_len + chunk - 1) / chunk;
    p.CB = std::max(1, (max_group_size * (Hq / Hkv) + prefix_cols_per_cta() - 1) / prefix_cols_per_cta());
    const size_t rows_pre = (size_t)S * Hq * p.PP, rows_own = (size_t)S * Hq * p.MP;
    p.start_off = 0;
    p.group_off = align_up((size_t)S * sizeof(int32_t), 256);
    p.pacc_off = align_up(p.group_off + (size_t)S * sizeof(int32_t), 256);
    p.pml_off = align_up(p.pacc_off + rows_pre * D * sizeof(float), 256);
    p.acc_off = align_up(p.pml_off + rows_pre * 2 * sizeof(float), 256);
    p.ml_off = align_up(p.acc_off + rows_own * D * sizeof(float), 256);
    p.bytes = align_up(p.ml_off + rows_own * 2 * sizeof(float), 256);
    return p;
}

static pa_status check_prefix_args(const char *fn, int S, int Hq, int Hkv, int D, int bs, int kv_dtype,
                                   int max_context_len, int n_groups, int max_group_size,
                                   int max_prefix_len) {
    pa_status st = check_decode_shape(fn, S, Hq, Hkv, D, bs, kv_dtype, max_context_len);
    if (st != PA_OK) return st;
    if (n_groups < 0 || n_groups > 65535)
        return fail(PA_ERR_INVALID_ARG, "%s: n_groups = %d", fn, n_groups);
    if (max_prefix_len < 0 || max_prefix_len % bs != 0 || max_prefix_len > max_context_len)
        return fail(PA_ERR_INVALID_ARG, "%s: max_prefix_len = %d must be a multiple of %d within max_context_len",
                    fn, max_prefix_len, bs);
    if (max_group_size < 1 || max_group_size > S)
        return fail(PA_ERR_INVALID_ARG, "%s: max_group_size = %d", fn, max_group_size);
    const int64_t cb = ((int64_t)max_group_size * (Hq / Hkv) + prefix_cols_per_cta() - 1) / prefix_cols_per_cta();
    if ((int64_t)Hkv * cb > 65535) return fail(PA_ERR_UNSUPPORTED, "%s: groups too large", fn);
    return PA_OK;
}

size_t pa_decode_shared_prefix_workspace_size(int S, int Hq, int Hkv, int D, int bs, int kv_dtype,
                                              int max_context_len, int max_group_size,
                                              int max_prefix_len) {
    if (check_prefix_args("pa_decode_shared_prefix_workspace_size", S, Hq, Hkv, D, bs, kv_dtype,
                          max_context_len, 0, max_group_size, max_prefix_len) != PA_OK)
        return 0;
    return plan_prefix(S, Hq, Hkv, D, bs, kv_dtype, max_context_len, max_group_size, max_prefix_len).bytes;
}

pa_status pa_decode_shared_prefix(pa_bf16 *out, const pa_bf16 *query, const void *k_cache,
                                  const void *v_cache, const float *k_scale, const float *v_scale,
                                  int kv_dtype, const int32_t *block_tables, int M,
                                  const int32_t *context_lens, int S, int Hq, int Hkv, int D, int bs,
                                  int N, float scale, int max_context_len,
                                  const int32_t *group_start, const int32_t *group_prefix_len,
                                  int n_groups, int max_group_size, int max_prefix_len,
                                  void *workspace, size_t workspace_bytes, int *err_flag,
                                  void *stream) {
    const char *fn = "pa_decode_shared_prefix";
    g_last_error[0] = 0;
    if (S == 0) return PA_OK;
    pa_status st = check_prefix_args(fn, S, Hq, Hkv, D, bs, kv_dtype, max_context_len, n_groups,
                                      max_group_size, max_prefix_len);
    if (st != PA_OK) return st;
    if (N <= 0 || M <= 0)
        return fail(PA_ERR_INVALID_ARG, "%s: N = %d, M = %d must be positive", fn, N, M);
    if ((int64_t)max_context_len > (int64_t)M * bs)
        return fail(PA_ERR_OUT_OF_RANGE, "%s: max_context_len %d exceeds M * bs = %lld", fn,
                    max_context_len, (long long)M * bs);
    if (!out || !query || !k_cache || !v_cache || !block_tables || !context_lens)
        return fail(PA_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (n_groups > 0 && (!group_start || !group_prefix_len))
        return fail(PA_ERR_INVALID_ARG, "%s: group arrays missing", fn);
    if (kv_dtype != PA_KV_BF16 && (!k_scale || !v_scale || !aligned16(k_scale) || !aligned16(v_scale)))
        return fail(PA_ERR_INVALID_ARG, "%s: an int8 or fp8 cache needs 16-byte aligned k_scale and v_scale", fn);
    if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", fn);
    if (!(scale == scale) || scale == __builtin_inff() || scale == -__builtin_inff())
        return fail(PA_ERR_INVALID_ARG, "%s: scale must be finite", fn);
    const PrefixPlan plan = plan_prefix(S, Hq, Hkv, D, bs, kv_dtype, max_context_len, max_group_size,
                                        max_prefix_len);
    if (!workspace || workspace_bytes < plan.bytes)
        return fail(PA_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed, %zu given", fn, plan.bytes,
                    workspace ? workspace_bytes : (size_t)0);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(PA_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", fn);
    char *ws = static_cast<char *>(workspace);
    DecodeArgs a{};
    a.out = out;
    a.q = query;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.ws_acc = (float *)(ws + plan.acc_off);
    a.ws_ml = (float *)(ws + plan.ml_off);
    a.err_flag = err_flag;
    a.M = M;
    a.S = S;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.N = N;
    a.head_chunks = plan.own.head_chunks;
    a.part_tokens = plan.own.part_tokens;
    a.max_parts = plan.MP;
    a.max_context_len = max_context_len;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.start_tokens = (const int32_t *)(ws + plan.start_off);
    a.partials_only = 1;
    PrefixArgs p{};
    p.group_start = group_start;
    p.group_prefix = group_prefix_len;
    p.n_groups = n_groups;
    p.max_group_size = max_group_size;
    p.max_prefix = max_prefix_len;
    p.seq_start = (int32_t *)(ws + plan.start_off);
    p.seq_group = (int32_t *)(ws + plan.group_off);
    p.pacc = (float *)(ws + plan.pacc_off);
    p.pml = (float *)(ws + plan.pml_off);
    p.PP = plan.PP;
    p.CB = plan.CB;
    p.chunk = plan.chunk;
    launch_decode_shared_prefix(a, p, D, bs, kv_dtype, (cudaStream_t)stream);
    return check_launch(fn);
}

// Multi-token attention plan: CTAs of 128 (token, head) columns per kv head; the
// context is split into partitions (multiples of 64 tokens, at most 4096) when the
// columns alone do not fill 4 waves of 2 CTAs per SM.
struct MultiPlan {
    int CB, part_tokens, max_parts;
    size_t acc_off, ml_off, bytes;
    // 8-bit caches on the tcgen05 kernel: the dequantised pool (Mq = ceil(max context /
    // bs) table entries per sequence; Mq = 0: none): the table [S][Mq] and the sequences'
    // pool offsets [S + 1] at tab_off and off_off, then K and V pools of pool_blocks
    // blocks of block_bytes each from kq_off
    int Mq;
    size_t tab_off, off_off, kq_off, block_bytes;
    int64_t pool_blocks;
};

// Fixed cost of one multi-token CTA (q fragments or the tensor-memory setup, the join
// of token slices, the writes, the partial rows the merge reads) in tokens of
// streaming: larger than the decode kernel's.  Measured on GB300 with balanced
// partitions, where the score at 256 tokens nearly tied two lengths the longer one
// was faster: 70B-shaped 4-token verification 5 x 1600 tokens 129.2 us against
// 7 x 1152 132.7 us; 64 x 3000-token contexts with 16 columns 2 x 1536 148.9 us
// against 4 x 768 157.0 us.
constexpr double kMultiRampTokens = 512.0;

// pool_blocks_hint: blocks the dequantised pool must hold (an upper bound of the blocks
// the sequences attend), or -1 for the largest need, S * Mq.
static MultiPlan plan_multi(int S, int T, int Hq, int Hkv, int D, int bs, int kv_dtype, int max_context_len,
                            int max_query_len, int64_t pool_blocks_hint = -1) {
    MultiPlan p{};
    const int G = Hq / Hkv;
    p.CB = std::max(1, (int)(((int64_t)max_query_len * G + multi_cols_per_cta() - 1) / multi_cols_per_cta()));
    const bool tc = multi_tc_eligible(D, kv_dtype, G, max_query_len);
    // CTAs per context partition: the decode kernel in rows mode takes one or two new
    // tokens and up to 8 query heads each
    const bool per_token = !tc && multi_per_token_eligible(D, kv_dtype, G, max_query_len);
    const int rows = decode_rows_per_cta(max_query_len);
    const int64_t units = per_token ? (int64_t)S * Hkv * ((G + 7) / 8) * ((max_query_len + rows - 1) / rows)
                                    : (int64_t)S * Hkv * p.CB;
    const double slots = (double)device_sms() * 2;  // both kernels keep two CTAs per SM
    const int ctx = std::max(max_context_len, 1);
    p.part_tokens = 256;
    if (tc && (int64_t)max_query_len * G >= 64) {
        // chunks of half a tile of columns and more (compute-heavy): whole contexts
        // (partials and their merge cost more than a ragged last wave), unless the CTAs
        // would fill less than half the slots, then about one wave; narrower chunks
        // (streaming-bound) are planned like the mma.sync kernel's
        p.part_tokens = (int)align_up((size_t)ctx, 64);
        if ((double)units < slots / 2) {
            const int64_t want = (int64_t)std::ceil(slots / (double)units);
            p.part_tokens = std::max(512, (int)align_up((size_t)((ctx + want - 1) / want), 128));
        }
    } else if ((double)units >= 4.0 * slots && ctx <= 4096) {
        p.part_tokens = (int)align_up((size_t)ctx, 64);
    } else {
        // n balanced partitions of the longest context (each a multiple of 64 tokens,
        // so the last one is not a ragged remainder), n chosen by the same score as the
        // decode plan's.  Against the former choice among 4096, 2048, ..., 256 tokens,
        // measured on GB300: 70B-shaped 4-token verification 1024 -> 1600 tokens
        // 134.2 -> 129.2 us (fp8 cache 259.8 -> 245.3), 64 x 3000-token contexts with
        // 16 columns 2048 -> 1536 156.5 -> 148.9 us, 16 x 6000 with 8 columns 1024 -> 896
        // 90.3 -> 85.9 us
        double best = -1.0;
        const int nmax = (ctx + 255) / 256;
        for (int n = 1; n <= nmax; ++n) {
            const int cand = std::min(4096, std::max(256, (int)align_up((size_t)((ctx + n - 1) / n), 64)));
            const int64_t parts = (ctx + cand - 1) / cand;
            if (parts != n) continue;  // the same length as a smaller n
            const double waves = (double)(units * parts) / slots;
            if (waves < 2.0 && cand != 256) continue;
            const double fill = waves / std::ceil(waves);
            const double len = (double)std::min(cand, ctx);
            const double score = fill * len / (len + kMultiRampTokens);
            if (score > best + 1e-9) {
                best = score;
                p.part_tokens = cand;
            }
        }
    }
    p.max_parts = (ctx + p.part_tokens - 1) / p.part_tokens;
    size_t end = 0;
    if (p.max_parts > 1) {
        const size_t rows = (size_t)T * Hq * p.max_parts;
        // the partial rows come first: the merge reads them with 16-byte vector loads,
        // so their offset must stay a multiple of 16 (checked at launch)
        p.acc_off = 0;
        p.ml_off = align_up(rows * D * sizeof(float), 256);
        end = align_up(p.ml_off + rows * 2 * sizeof(float), 256);
    }
    if (tc && kv_dtype != PA_KV_BF16) {
        p.Mq = (ctx + bs - 1) / bs;
        p.tab_off = end;
        p.off_off = align_up(p.tab_off + (size_t)S * p.Mq * sizeof(int32_t), 256);
        p.kq_off = align_up(p.off_off + (size_t)(S + 1) * sizeof(int32_t), 256);
        p.block_bytes = (size_t)Hkv * bs * D * 2;  // a multiple of 256
        const int64_t most = (int64_t)S * p.Mq;
        p.pool_blocks = pool_blocks_hint < 0 ? most : std::min(most, std::max<int64_t>(pool_blocks_hint, 1));
        end = p.kq_off + 2 * (size_t)p.pool_blocks * p.block_bytes;
    }
    p.bytes = end;
    return p;
}

static pa_status check_multi_args(const char *fn, int S, int T, int Hq, int Hkv, int D, int bs,
                                  int kv_dtype, int max_context_len, int max_query_len) {
    pa_status st = check_decode_shape(fn, S, Hq, Hkv, D, bs, kv_dtype, max_context_len);
    if (st != PA_OK) return st;
    if (T < 0) return fail(PA_ERR_INVALID_ARG, "%s: T = %d", fn, T);
    if (max_query_len < 1 || max_query_len > max_context_len || max_query_len > T)
        return fail(PA_ERR_INVALID_ARG, "%s: max_query_len = %d (1 .. min(T, max_context_len))", fn,
                    max_query_len);
    const int64_t cb = ((int64_t)max_query_len * (Hq / Hkv) + multi_cols_per_cta() - 1) / multi_cols_per_cta();
    if ((int64_t)Hkv * cb > 65535 || ((int64_t)max_query_len * Hq + 3) / 4 > 0x7fffffffLL)
        return fail(PA_ERR_UNSUPPORTED, "%s: too many new tokens per sequence", fn);
    return PA_OK;
}

size_t pa_multi_token_workspace_size(int S, int T, int Hq, int Hkv, int D, int bs, int kv_dtype,
                                     int max_context_len, int max_query_len) {
    if (check_multi_args("pa_multi_token_workspace_size", S, T, Hq, Hkv, D, bs, kv_dtype,
                         max_context_len, max_query_len) != PA_OK)
        return 0;
    return plan_multi(S, T, Hq, Hkv, D, bs, kv_dtype, max_context_len, max_query_len).bytes;
}

size_t pa_multi_token_workspace_size_for_tokens(int S, int T, int Hq, int Hkv, int D, int bs, int kv_dtype,
                                                int max_context_len, int max_query_len,
                                                int64_t total_context_tokens) {
    if (check_multi_args("pa_multi_token_workspace_size_for_tokens", S, T, Hq, Hkv, D, bs, kv_dtype,
                         max_context_len, max_query_len) != PA_OK ||
        total_context_tokens < 0)
        return 0;
    // sum_s ceil(ctx_s / bs) <= sum_s ctx_s / bs + S
    const int64_t blocks = (total_context_tokens + bs - 1) / bs + S;
    return plan_multi(S, T, Hq, Hkv, D, bs, kv_dtype, max_context_len, max_query_len, blocks).bytes;
}

pa_status pa_multi_token_attention(pa_bf16 *out, const pa_bf16 *query, const void *k_cache,
                                   const void *v_cache, const float *k_scale,
                                   const float *v_scale, int kv_dtype,
                                   const int32_t *block_tables, int M,
                                   const int32_t *context_lens, const int32_t *query_start,
                                   int S, int T, int Hq, int Hkv, int D, int bs, int N,
                                   float scale, int max_context_len, int max_query_len,
                                   void *workspace, size_t workspace_bytes, int *err_flag,
                                   void *stream) {
    const char *fn = "pa_multi_token_attention";
    g_last_error[0] = 0;
    if (S == 0 || T == 0) return PA_OK;
    pa_status st = check_multi_args(fn, S, T, Hq, Hkv, D, bs, kv_dtype, max_context_len, max_query_len);
    if (st != PA_OK) return st;
    if (N <= 0 || M <= 0)
        return fail(PA_ERR_INVALID_ARG, "%s: N = %d, M = %d must be positive", fn, N, M);
    if ((int64_t)max_context_len > (int64_t)M * bs)
        return fail(PA_ERR_OUT_OF_RANGE, "%s: max_context_len %d exceeds M * bs = %lld", fn,
                    max_context_len, (long long)M * bs);
    if (!out || !query || !k_cache || !v_cache || !block_tables || !context_lens || !query_start)
        return fail(PA_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (kv_dtype != PA_KV_BF16 && (!k_scale || !v_scale))
        return fail(PA_ERR_INVALID_ARG, "%s: an int8 or fp8 cache needs k_scale and v_scale", fn);
    if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "%s: tensors must be 16-byte aligned", fn);
    if (!(scale == scale) || scale == __builtin_inff() || scale == -__builtin_inff())
        return fail(PA_ERR_INVALID_ARG, "%s: scale must be finite", fn);
    const MultiPlan plan = plan_multi(S, T, Hq, Hkv, D, bs, kv_dtype, max_context_len, max_query_len);
    // the dequantised pool holds as many blocks as the workspace leaves room for, at
    // least one (pa_multi_token_workspace_size_for_tokens sizes it for the attended ones)
    const size_t need = plan.Mq > 0 ? plan.kq_off + 2 * plan.block_bytes : plan.bytes;
    if (need && (!workspace || workspace_bytes < need))
        return fail(PA_ERR_INVALID_ARG, "%s: workspace of %zu bytes needed, %zu given", fn, need,
                    workspace ? workspace_bytes : (size_t)0);
    if (plan.bytes && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(PA_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", fn);
    if (plan.max_parts > 1 && (plan.acc_off % 16 != 0 || plan.ml_off % 16 != 0))
        return fail(PA_ERR_INVALID_ARG, "%s: internal workspace layout is not 16-byte aligned", fn);
    MultiArgs a{};
    a.out = out;
    a.q = query;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.query_start = query_start;
    a.ws_acc = plan.max_parts > 1 ? (float *)((char *)workspace + plan.acc_off) : nullptr;
    a.ws_ml = plan.max_parts > 1 ? (float *)((char *)workspace + plan.ml_off) : nullptr;
    a.err_flag = err_flag;
    a.M = M;
    a.S = S;
    a.T = T;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.g_shift = (a.G & (a.G - 1)) == 0 ? __builtin_ctz((unsigned)a.G) : -1;
    a.N = N;
    a.CB = plan.CB;
    a.part_tokens = plan.part_tokens;
    a.max_parts = plan.max_parts;
    a.max_context_len = max_context_len;
    a.max_query_len = max_query_len;
    a.scale_log2 = scale * 1.4426950408889634f;
    if (plan.Mq > 0) {
        // 8-bit cache, prefill-shaped: dequantise the attended blocks once, then the bf16
        // kernel reads them through the identity table
        const int64_t cap = std::min<int64_t>((int64_t)S * plan.Mq,
                                              (int64_t)((workspace_bytes - plan.kq_off) / (2 * plan.block_bytes)));
        uint16_t *kq = (uint16_t *)((char *)workspace + plan.kq_off);
        uint16_t *vq = (uint16_t *)((char *)workspace + plan.kq_off + (size_t)cap * plan.block_bytes);
        int32_t *tab = (int32_t *)((char *)workspace + plan.tab_off);
        int32_t *off = (int32_t *)((char *)workspace + plan.off_off);
        launch_dequant_blocks(a, bs, kv_dtype, plan.Mq, kq, vq, tab, off, cap, (cudaStream_t)stream);
        MultiArgs b = a;
        b.k_cache = kq;
        b.v_cache = vq;
        b.k_scale = b.v_scale = nullptr;
        b.block_tables = tab;
        b.M = plan.Mq;
        b.N = (int)cap;
        launch_multi_token(b, D, bs, PA_KV_BF16, (cudaStream_t)stream);
    } else {
        launch_multi_token(a, D, bs, kv_dtype, (cudaStream_t)stream);
    }
    return check_launch(fn);
}

}  // extern "C"
