// Multi-token paged attention: several new tokens of a sequence attend the paged
// cache in one pass -- a chunk of a long prompt (chunked prefill) or the draft tokens
// a large model verifies at once (speculative decoding); deeplearn.tn, "Les leviers
// d'optimisation en production", and the gaiatechstar.com discussion's reply on
// chunked prefill.  New token i of sequence s sits at position ctx - L + i and
// attends every cached token up to and including its own position (causal inside
// the chunk); with L = 1 this is the decode step.
//
// Work unit ("column"): one (new token, query head) pair.  The columns of a sequence
// and kv head share that kv head's K and V, so a CTA takes up to 128 of them and
// streams the sequence's K and V once for all: 64-token chunks staged in shared
// memory by cp.async, double-buffered.  The columns are the rows (M) of the
// tensor-core products, FlashAttention-2 style: a warp owns 16 columns and, per
// chunk, computes S = Q K^T over its share of the chunk's tokens (Q fragments from
// shared memory, K by ldmatrix), one online-softmax step in the exp2 domain with each
// row's max over the 4 lanes that hold it and each column masked at its own
// position, then O += P V with P's accumulators reused as the A operand.  Warps are
// (column group, token slice) pairs: with 5..8 groups a warp takes whole chunks;
// with up to four groups (draft tokens) two warps split each chunk of a group (32
// tokens each: narrower slices cost more per token than the idle warps they would
// employ), and the slices are joined by log-sum-exp in shared memory before a column
// is written.
// Long contexts are split into partitions (grid x); a column whose visible tokens
// span one partition is finished in place, the others leave (max, sum, output)
// partials that a second kernel joins by log-sum-exp.
#include <cuda_bf16.h>
#include <math.h>

#include <atomic>
#include <type_traits>

#include "pa_internal.cuh"
#include "pa_mma.cuh"

namespace pa {
namespace {

using namespace tiled;


constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kColsPerWarp = 16;                   // two mma n-tiles of 8 columns
constexpr int kColsPerCta = kWarps * kColsPerWarp;  // 128
constexpr int kChunk = 64;                         // tokens per shared-memory stage
constexpr int kMaxPartBlocks = 4096 / 16;          // block ids of one partition
constexpr int kPerTokenMaxQuery = 8;               // longest chunk served one CTA per token

__device__ __forceinline__ void raise_flag(int *err_flag, int bit) {
    if (err_flag) atomicOr(err_flag, bit);
}

// The sequence's context, new-token count and first query row, checked: a context
// outside [0, min(M * bs, max_context_len)] is clamped (CONTEXT flag); query offsets
// outside [0, T], a negative count, more new tokens than context or than
// max_query_len leave the sequence out (QUERY flag, its rows are not written).
struct SeqView {
    int ctx, L, row0, base;
    bool ok;
};

template <int BS>
__device__ __forceinline__ SeqView seq_view(const MultiArgs &a, int s, bool report) {
    SeqView v;
    int ctx = a.context_lens[s];
    const int lim = min(a.M * BS, a.max_context_len);
    if (ctx < 0 || ctx > lim) {
        if (report) raise_flag(a.err_flag, PA_FLAG_CONTEXT_OUT_OF_RANGE);
        ctx = ctx < 0 ? 0 : lim;
    }
    const int r0 = a.query_start[s], r1 = a.query_start[s + 1];
    v.ctx = ctx;
    v.row0 = r0;
    v.L = r1 - r0;
    v.ok = r0 >= 0 && r1 <= a.T && v.L >= 0 && v.L <= ctx && v.L <= a.max_query_len;
    if (!v.ok && report) raise_flag(a.err_flag, PA_FLAG_QUERY_OUT_OF_RANGE);
    v.base = ctx - v.L;
    return v;
}

// Column c of a kv head is new token c / G, query head c % G: a shift and a mask when
// G is a power of two (g_shift >= 0), else a division.
__device__ __forceinline__ int col_token(const MultiArgs &a, int c) {
    return a.g_shift >= 0 ? c >> a.g_shift : c / a.G;
}
__device__ __forceinline__ int col_head(const MultiArgs &a, int c) {
    return a.g_shift >= 0 ? c & (a.G - 1) : c % a.G;
}

template <int D>
__host__ __device__ constexpr int multi_smem_bytes() {
    // K and V stages, then the query rows; the slice join reuses the stages
    return 4 * kChunk * (2 * D + 16) + kColsPerCta * (2 * D + 16);
}

// 8-bit caches: raw codes of a chunk (K then V) as copied from the cache
template <int D>
__host__ __device__ constexpr int raw_chunk_bytes() {
    return 2 * kChunk * D;
}

// 8-bit caches: one fp16 K and V stage, the query rows, two raw chunks
template <int D>
__host__ __device__ constexpr int multi_smem_bytes_q() {
    return 2 * kChunk * (2 * D + 16) + kColsPerCta * (2 * D + 16) + 2 * raw_chunk_bytes<D>();
}
static_assert(kWarps * kColsPerWarp * (128 + 4) * 4 <= 2 * kChunk * (2 * 128 + 16) + kColsPerCta * (2 * 128 + 16),
              "the join fits the stage and query rows");
static_assert(kWarps * kColsPerWarp * (128 + 4) * 4 <= 4 * kChunk * (2 * 128 + 16), "join fits the stages");

// One online-softmax step of a warp over NTW 8-token n-tiles of a staged chunk:
// S = Q K^T (rows = the warp's 16 columns), mask, running max and sum, O += P V.
template <int D, int NTW>
__device__ __forceinline__ void attend_tokens(float (&o)[D / 8][4], float (&m)[2], float (&l)[2],
                                              uint32_t qaddr, uint32_t kb, uint32_t vb, int tok0,
                                              bool full, const int (&lim)[2], float scale_log2, int t) {
    constexpr int RS = 2 * D + 16;
    constexpr int KC = D / 16;
    constexpr int DT = D / 8;
    float sc[NTW][4];
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int kc = 0; kc < KC; ++kc) {
        uint32_t qa[4];
        ldsm_x4(qa, qaddr + kc * 32);
#pragma unroll
        for (int np = 0; np < NTW / 2; ++np) {
            uint32_t kb4[4];
            ldsm_x4(kb4, kb + np * 16 * RS + kc * 32);
            mma16816(sc[2 * np], qa, kb4[0], kb4[1]);
            mma16816(sc[2 * np + 1], qa, kb4[2], kb4[3]);
        }
    }
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float x = sc[nt][c] * scale_log2;
            if (!full) {
                const int tok = tok0 + nt * 8 + 2 * t + (c & 1);
                x = tok <= lim[c >> 1] ? x : -INFINITY;
            }
            sc[nt][c] = x;
            mx[c >> 1] = fmaxf(mx[c >> 1], x);
        }
    float base[2], alpha[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
        const float mnew = fmaxf(m[h], mx[h]);
        base[h] = mnew == -INFINITY ? 0.f : mnew;
        alpha[h] = ex2(m[h] - base[h]);
        m[h] = mnew;
        l[h] *= alpha[h];
    }
    // the running maxima settle after a few steps: rescale only when one moved
    if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) {
            o[dt][0] *= alpha[0];
            o[dt][1] *= alpha[0];
            o[dt][2] *= alpha[1];
            o[dt][3] *= alpha[1];
        }
    }
#pragma unroll
    for (int kk = 0; kk < NTW / 2; ++kk) {
        float p[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                p[u][c] = ex2(sc[2 * kk + u][c] - base[c >> 1]);
                l[c >> 1] += p[u][c];
            }
        const uint32_t pa[4] = {bf16x2(p[0][0], p[0][1]), bf16x2(p[0][2], p[0][3]),
                                bf16x2(p[1][0], p[1][1]), bf16x2(p[1][2], p[1][3])};
#pragma unroll
        for (int dp = 0; dp < DT / 2; ++dp) {
            uint32_t vb4[4];
            ldsm_x4_trans(vb4, vb + kk * 16 * RS + dp * 32);
            mma16816(o[2 * dp], pa, vb4[0], vb4[1]);
            mma16816(o[2 * dp + 1], pa, vb4[2], vb4[3]);
        }
    }
}

// The step of attend_tokens for 8-bit caches.  K and V rows are the exact codes as
// fp16; the query rows fp16 scaled by a power of two per row (rs[h] = softmax scale x
// 2^-sig of row gq + 8h); ksc / vsc the staged tokens' key and value scales.  A score
// is (q . code) x rs x key scale, in fp32.  The value scale multiplies the softmax
// weight fed to the fp16 product, in units of 2^ve (ve: the exponent of the largest
// value scale this warp has seen, O rescaled when it grows), so weight x scale stays
// below 1; the running sum takes the weights alone.  No value leaves fp16's range
// whatever the scales.
template <int D, int NTW>
__device__ __forceinline__ void attend_tokens_q(float (&o)[D / 8][4], float (&m)[2], float (&l)[2], int &ve,
                                                uint32_t qaddr, uint32_t kb, uint32_t vb, const float *ksc,
                                                const float *vsc, int tok0, bool full, const int (&lim)[2],
                                                const float (&rs)[2], int t) {
    constexpr int RS = 2 * D + 16;
    constexpr int KC = D / 16;
    constexpr int DT = D / 8;
    const int lane = threadIdx.x & 31;
    float sc[NTW][4];
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int kc = 0; kc < KC; ++kc) {
        uint32_t qa[4];
        ldsm_x4(qa, qaddr + kc * 32);
#pragma unroll
        for (int np = 0; np < NTW / 2; ++np) {
            uint32_t kb4[4];
            ldsm_x4(kb4, kb + np * 16 * RS + kc * 32);
            mma16816_f16(sc[2 * np], qa, kb4[0], kb4[1]);
            mma16816_f16(sc[2 * np + 1], qa, kb4[2], kb4[3]);
        }
    }
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int j = nt * 8 + 2 * t + (c & 1);  // token of the slice
            float x = sc[nt][c] * rs[c >> 1] * ksc[j];
            if (!full) x = tok0 + j <= lim[c >> 1] ? x : -INFINITY;
            sc[nt][c] = x;
            mx[c >> 1] = fmaxf(mx[c >> 1], x);
        }
    float base[2], alpha[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
        const float mnew = fmaxf(m[h], mx[h]);
        base[h] = mnew == -INFINITY ? 0.f : mnew;
        alpha[h] = ex2(m[h] - base[h]);
        m[h] = mnew;
        l[h] *= alpha[h];
    }
    // the largest value scale of the slice's tokens: O in units of 2^ve
    float vmax = 0.f;
    for (int j = lane; j < NTW * 8; j += 32) vmax = fmaxf(vmax, vsc[j]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
    float grow = 1.f;
    if (vmax > 0.f) {
        const int e = exponent_above(vmax);
        if (e > ve) {
            grow = ve < -200 ? 0.f : ldexpf(1.f, ve - e);
            ve = e;
        }
    }
    if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f || grow != 1.f)) {
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) {
            o[dt][0] *= alpha[0] * grow;
            o[dt][1] *= alpha[0] * grow;
            o[dt][2] *= alpha[1] * grow;
            o[dt][3] *= alpha[1] * grow;
        }
    }
    const float vmul = ldexpf(1.f, -ve);
#pragma unroll
    for (int kk = 0; kk < NTW / 2; ++kk) {
        float p[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int j = (2 * kk + u) * 8 + 2 * t + (c & 1);
                const float w = ex2(sc[2 * kk + u][c] - base[c >> 1]);
                l[c >> 1] += w;
                p[u][c] = w * (vsc[j] * vmul);
            }
        const uint32_t pa[4] = {f16x2(p[0][0], p[0][1]), f16x2(p[0][2], p[0][3]),
                                f16x2(p[1][0], p[1][1]), f16x2(p[1][2], p[1][3])};
#pragma unroll
        for (int dp = 0; dp < DT / 2; ++dp) {
            uint32_t vb4[4];
            ldsm_x4_trans(vb4, vb + kk * 16 * RS + dp * 32);
            mma16816_f16(o[2 * dp], pa, vb4[0], vb4[1]);
            mma16816_f16(o[2 * dp + 1], pa, vb4[2], vb4[3]);
        }
    }
}

template <typename KV, int D, int BS>
__global__ void __launch_bounds__(kThreads, 2) paged_multi_kernel(const __grid_constant__ MultiArgs a) {
    constexpr bool QUANT = sizeof(KV) == 1;  // int8 / fp8 cache: exact fp16 codes, fp32 scales, fp16 products
    constexpr int ROW = D * 2;          // bytes of one token row (bf16)
    constexpr int RS = ROW + 16;        // padded shared-memory row stride
    constexpr int STAGE = kChunk * RS;  // one K (or V) stage
    constexpr int CPR = ROW / 16;       // 16-byte pieces per row
    constexpr int DT = D / 8;           // 8-wide d-tiles of O
    constexpr int PER = D / 32;         // values per lane in the join
    extern __shared__ __align__(128) unsigned char smem[];  // K0 K1 V0 V1 Q (8-bit: K V Q raw0 raw1)
    __shared__ int s_blk[kMaxPartBlocks];
    __shared__ float s_ml[kWarps][kColsPerWarp][2];  // each warp's (max, sum) per row
    // 8-bit caches: each query row's softmax scale x 2^-sig (its fp16 copy is scaled
    // by 2^sig), and the staged chunk's key and value scales
    __shared__ float s_qs[QUANT ? kColsPerCta : 1];
    __shared__ float s_sc[QUANT ? 2 * kChunk : 1];

    const int part = blockIdx.x;
    const int kvh = blockIdx.y / a.CB, cb = blockIdx.y % a.CB;
    const int s = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, t = lane & 3;

    const SeqView v = seq_view<BS>(a, s, part == 0 && blockIdx.y == 0 && tid == 0);
    if (!v.ok) return;
    const int ncols = v.L * a.G;
    const int col0 = cb * kColsPerCta;
    if (col0 >= ncols) return;
    // the CTA's last column sees the most tokens
    const int cta_lim = v.base + col_token(a, min(ncols, col0 + kColsPerCta) - 1);  // inclusive
    const int tok_begin = part * a.part_tokens;
    const int tok_end = min(tok_begin + a.part_tokens, cta_lim + 1);
    if (tok_begin >= tok_end) return;
    const int blk0 = tok_begin / BS;  // partitions start on a block boundary
    const int nblk = (tok_end - tok_begin + BS - 1) / BS;
    for (int i = tid; i < nblk; i += kThreads) {
        int b = a.block_tables[(int64_t)s * a.M + blk0 + i];
        if (b < 0 || b >= a.N) {
            if (cb == 0) raise_flag(a.err_flag, PA_FLAG_BLOCK_OUT_OF_RANGE);
            b = -1;  // read as zeros
        }
        s_blk[i] = b;
    }
    unsigned char *ks = smem, *vs = smem + (QUANT ? 1 : 2) * STAGE, *qs = smem + (QUANT ? 2 : 4) * STAGE;
    unsigned char *raw = qs + kColsPerCta * RS;  // 8-bit caches only
    // the CTA's query rows, one per column (zeros past the last column)
    if constexpr (!QUANT) {
        for (int i = tid; i < kColsPerCta * CPR; i += kThreads) {
            const int r = i / CPR, pc = i % CPR;
            const int c = col0 + r;
            const void *src = a.q;
            uint32_t bytes = 0;
            if (c < ncols) {
                const int64_t row = v.row0 + col_token(a, c);
                src = reinterpret_cast<const char *>(a.q + (row * a.Hq + kvh * a.G + col_head(a, c)) * D) + pc * 16;
                bytes = 16;
            }
            cp_async16(smem_u32(qs + r * RS + pc * 16), src, bytes);
        }
    } else {
        // as fp16 scaled by 2^sig per row, sig putting the row's largest |q| in
        // [2^13, 2^14); the CPR threads of a row are consecutive lanes of one warp
        for (int i = tid; i < kColsPerCta * CPR; i += kThreads) {
            const int r = i / CPR, pc = i % CPR;
            const int c = col0 + r;
            uint4 raw = make_uint4(0u, 0u, 0u, 0u);
            if (c < ncols) {
                const int64_t row = v.row0 + col_token(a, c);
                raw = __ldg(reinterpret_cast<const uint4 *>(a.q + (row * a.Hq + kvh * a.G + col_head(a, c)) * D) + pc);
            }
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
            float f[8], amax = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                f[2 * e] = __uint_as_float(w[e] << 16);
                f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
                amax = fmaxf(amax, fmaxf(fabsf(f[2 * e]), fabsf(f[2 * e + 1])));
            }
#pragma unroll
            for (int off = CPR / 2; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            const int sig = amax > 0.f ? min(100, max(-100, 14 - exponent_above(amax))) : 0;
            const float up = ldexpf(1.f, sig);
            uint4 h;
            h.x = f16x2(f[0] * up, f[1] * up);
            h.y = f16x2(f[2] * up, f[3] * up);
            h.z = f16x2(f[4] * up, f[5] * up);
            h.w = f16x2(f[6] * up, f[7] * up);
            *reinterpret_cast<uint4 *>(qs + r * RS + pc * 16) = h;
            if (pc == 0) s_qs[r] = a.scale_log2 * ldexpf(1.f, -sig);
        }
    }

    // warps = (group of 16 columns, token slice)
    const int ncg = (min(ncols - col0, kColsPerCta) + kColsPerWarp - 1) / kColsPerWarp;
    const int P2 = ncg <= 1 ? 1 : ncg <= 2 ? 2 : ncg <= 4 ? 4 : 8;
    const int slices = min(2, kWarps / P2);  // a slice keeps >= 32 tokens per step
    const int grp = warp % P2, slice = warp / P2;
    const bool active = grp < ncg && slice < slices;
    const int width = kChunk / slices;  // tokens of a chunk per slice
    const int wcol0 = col0 + grp * kColsPerWarp;
    // rows gq and gq + 8: last visible position, clamped to the partition (-1: none)
    int lim[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int c = wcol0 + gq + 8 * h;
        lim[h] = (active && c < ncols) ? min(v.base + col_token(a, c), tok_end - 1) : -1;
    }
    const int warp_hi = (active && wcol0 < ncols) ? min(v.base + col_token(a, min(ncols, wcol0 + kColsPerWarp) - 1), tok_end - 1) : -1;
    const int warp_lo = (active && wcol0 < ncols) ? min(v.base + col_token(a, wcol0), tok_end - 1) : -1;
    __syncthreads();  // s_blk

    // staging (bf16): thread tid always copies 16-byte piece pc of rows pr, pr + RPP, ...
    // of a chunk, for K and for V; a (block, kv head) is BS contiguous rows in the cache
    constexpr int RPP = kThreads / CPR;
    constexpr int PASSES = kChunk / RPP;
    const int pc = tid % CPR, pr = tid / CPR;
    const int64_t block_stride = (int64_t)a.Hkv * BS * ROW;
    const char *kbase_g = static_cast<const char *>(a.k_cache) + (int64_t)kvh * BS * ROW + pc * 16;
    const char *vbase_g = static_cast<const char *>(a.v_cache) + (int64_t)kvh * BS * ROW + pc * 16;
    const uint32_t kdst0 = smem_u32(ks) + pr * RS + pc * 16, vdst0 = smem_u32(vs) + pr * RS + pc * 16;
    auto stage_chunk = [&](int j, int buf) {
        const int c0 = tok_begin + j * kChunk;
#pragma unroll
        for (int k = 0; k < PASSES; ++k) {
            const int tok = c0 + pr + k * RPP;
            const char *ksrc = kbase_g, *vsrc = vbase_g;
            uint32_t bytes = 0;
            if (tok < tok_end) {
                const int b = s_blk[tok / BS - blk0];
                if (b >= 0) {
                    const int64_t off = b * block_stride + (tok % BS) * ROW;
                    ksrc += off;
                    vsrc += off;
                    bytes = 16;
                }
            }
            const uint32_t doff = buf * STAGE + k * RPP * RS;
            cp_async16(kdst0 + doff, ksrc, bytes);
            cp_async16(vdst0 + doff, vsrc, bytes);
        }
        cp_async_commit();
    };

    float o[DT][4];
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    int ve = -1000;  // 8-bit caches: O is kept in units of 2^ve (no value scale seen yet)
    // ldmatrix lane addresses: Q as A (rows = columns), K as B (rows = tokens), V as
    // B transposed (rows = tokens), the last two at the slice's first token
    const uint32_t qaddr = smem_u32(qs) + (grp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * RS + (lane >> 4) * 16;
    const uint32_t krow = (slice * width + (lane & 7) + ((lane >> 4) << 3)) * RS + ((lane >> 3) & 1) * 16;
    const uint32_t vrow = (slice * width + (lane & 7) + (((lane >> 3) & 1) << 3)) * RS + (lane >> 4) * 16;

    const int nchunks = (tok_end - tok_begin + kChunk - 1) / kChunk;
    float rs[2] = {0.f, 0.f};  // 8-bit caches: the rows' softmax scale x 2^-sig
    auto attend_chunk = [&](int j) {
        const int tok0 = tok_begin + j * kChunk + slice * width;
        if (tok0 <= warp_hi) {  // warp-uniform (inactive warps have warp_hi = -1)
            const int buf = QUANT ? 0 : (j & 1);
            const uint32_t kb = smem_u32(ks + buf * STAGE) + krow;
            const uint32_t vb = smem_u32(vs + buf * STAGE) + vrow;
            const bool full = tok0 + width - 1 <= warp_lo;  // every row sees all: no mask
            if constexpr (QUANT) {
                const float *ksc = s_sc + slice * width, *vsc = s_sc + kChunk + slice * width;
                if (slices == 1)
                    attend_tokens_q<D, 8>(o, m, l, ve, qaddr, kb, vb, ksc, vsc, tok0, full, lim, rs, t);
                else
                    attend_tokens_q<D, 4>(o, m, l, ve, qaddr, kb, vb, ksc, vsc, tok0, full, lim, rs, t);
            } else {
                if (slices == 1)
                    attend_tokens<D, 8>(o, m, l, qaddr, kb, vb, tok0, full, lim, a.scale_log2, t);
                else
                    attend_tokens<D, 4>(o, m, l, qaddr, kb, vb, tok0, full, lim, a.scale_log2, t);
            }
        }
    };
    if constexpr (!QUANT) {
        stage_chunk(0, 0);  // first group: the query rows and chunk 0
        for (int j = 0; j < nchunks; ++j) {
            if (j + 1 < nchunks) {
                stage_chunk(j + 1, (j + 1) & 1);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            attend_chunk(j);
            __syncthreads();  // this buffer is refilled two chunks later
        }
    } else {
        // 8-bit caches: the next chunk's codes are copied raw (cp.async) into the other
        // of two raw buffers, and its rows' scales loaded into registers, while the
        // current chunk is computed; each thread then converts the pieces it copied
        // itself (its own completed copies need no barrier) to exact fp16 codes in the
        // single K and V stage, and the rows' scales go beside them.
        constexpr int QPR = D / 16;                  // 16-code pieces per row
        constexpr int NPT = kChunk * QPR / kThreads;  // pieces per thread and chunk
        const char *kc8 = static_cast<const char *>(a.k_cache), *vc8 = static_cast<const char *>(a.v_cache);
        float ksr[NPT], vsr[NPT];
        auto issue_raw = [&](int j, int b) {
            const int c0 = tok_begin + j * kChunk;
            unsigned char *rb = raw + b * raw_chunk_bytes<D>();
#pragma unroll
            for (int k = 0; k < NPT; ++k) {
                const int i = tid + k * kThreads, r = i / QPR, qc = i % QPR;
                const int tok = c0 + r;
                const char *ksrc = kc8, *vsrc = vc8;
                uint32_t bytes = 0;
                ksr[k] = vsr[k] = 0.f;
                if (tok < tok_end) {
                    const int blk = s_blk[tok / BS - blk0];
                    if (blk >= 0) {
                        const int64_t row = ((int64_t)blk * a.Hkv + kvh) * BS + tok % BS;
                        ksrc += row * D + qc * 16;
                        vsrc += row * D + qc * 16;
                        ksr[k] = __ldg(a.k_scale + row);
                        vsr[k] = __ldg(a.v_scale + row);
                        bytes = 16;
                    }
                }
                cp_async16(smem_u32(rb + r * D + qc * 16), ksrc, bytes);
                cp_async16(smem_u32(rb + kChunk * D + r * D + qc * 16), vsrc, bytes);
            }
            cp_async_commit();
        };
        auto convert_raw = [&](int b) {
            const unsigned char *rb = raw + b * raw_chunk_bytes<D>();
#pragma unroll
            for (int k = 0; k < NPT; ++k) {
                const int i = tid + k * kThreads, r = i / QPR, qc = i % QPR;
                uint4 lo, hi;
                codes_to_f16_exact<KV>(*reinterpret_cast<const uint4 *>(rb + r * D + qc * 16), lo, hi);
                uint4 *kd = reinterpret_cast<uint4 *>(ks + r * RS + qc * 32);
                kd[0] = lo;
                kd[1] = hi;
                codes_to_f16_exact<KV>(*reinterpret_cast<const uint4 *>(rb + kChunk * D + r * D + qc * 16), lo, hi);
                uint4 *vd = reinterpret_cast<uint4 *>(vs + r * RS + qc * 32);
                vd[0] = lo;
                vd[1] = hi;
                if (qc == 0) {  // rows past the partition or of a skipped block: scale 0
                    s_sc[r] = ksr[k];
                    s_sc[kChunk + r] = vsr[k];
                }
            }
        };
        issue_raw(0, 0);
        cp_async_wait<0>();
        convert_raw(0);
        __syncthreads();  // query rows, row scales, chunk 0
        rs[0] = s_qs[grp * 16 + gq];
        rs[1] = s_qs[grp * 16 + gq + 8];
        for (int j = 0; j < nchunks; ++j) {
            if (j + 1 < nchunks) issue_raw(j + 1, (j + 1) & 1);
            attend_chunk(j);
            __syncthreads();  // the stage is free
            if (j + 1 < nchunks) {
                cp_async_wait<0>();
                convert_raw((j + 1) & 1);
            }
            __syncthreads();  // chunk j + 1 staged
        }
    }
    // the merge grid may launch now (it still waits for this grid before reading)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

#pragma unroll
    for (int h = 0; h < 2; ++h) {
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
    }
    if constexpr (QUANT) {  // O back from units of 2^ve
        const float f = ve < -200 ? 1.f : ldexpf(1.f, ve);
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) {
            o[dt][0] *= f;
            o[dt][1] *= f;
            o[dt][2] *= f;
            o[dt][3] *= f;
        }
    }
    if (slices > 1) {
        // leave each warp's state in shared memory (the stages are free: every warp
        // passed the loop's last barrier), rows [column][d]
        float *so = reinterpret_cast<float *>(smem) + warp * kColsPerWarp * (D + 4);
#pragma unroll
        for (int dt = 0; dt < DT; ++dt)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                *reinterpret_cast<float2 *>(so + (gq + 8 * h) * (D + 4) + dt * 8 + 2 * t) =
                    make_float2(o[dt][2 * h], o[dt][2 * h + 1]);
        if (t == 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                s_ml[warp][gq + 8 * h][0] = m[h];
                s_ml[warp][gq + 8 * h][1] = l[h];
            }
        }
        __syncthreads();
        // one warp per column (round robin): join the slices, then finish the column
        // (one partition) or leave a partial
#pragma unroll 1
        for (int cc = warp; cc < ncg * kColsPerWarp; cc += kWarps) {
            const int c = col0 + cc;
            if (c >= ncols) break;
            const int lim_c = v.base + col_token(a, c);
            if (tok_begin > lim_c) continue;  // this partition holds nothing the column sees
            const int g = cc / kColsPerWarp, r = cc % kColsPerWarp;
            float mv = -INFINITY;
            for (int sl = 0; sl < slices; ++sl) mv = fmaxf(mv, s_ml[sl * P2 + g][r][0]);
            const float mb = mv == -INFINITY ? 0.f : mv;
            float acc[PER];
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[e] = 0.f;
            float lv = 0.f;
            for (int sl = 0; sl < slices; ++sl) {
                const int w = sl * P2 + g;
                const float f = ex2(s_ml[w][r][0] - mb);
                lv += f * s_ml[w][r][1];
                const float *src = reinterpret_cast<const float *>(smem) + (w * kColsPerWarp + r) * (D + 4) + lane * PER;
#pragma unroll
                for (int e = 0; e < PER; ++e) acc[e] += f * src[e];
            }
            const int64_t pair = (int64_t)(v.row0 + col_token(a, c)) * a.Hq + kvh * a.G + col_head(a, c);
            if (lim_c < a.part_tokens) {
                const float inv = lv > 0.f ? 1.f / lv : 0.f;
                uint16_t *dst = a.out + pair * D + lane * PER;
                if constexpr (PER == 4)
                    *reinterpret_cast<uint2 *>(dst) = make_uint2(bf16x2(acc[0] * inv, acc[1] * inv), bf16x2(acc[2] * inv, acc[3] * inv));
                else
                    *reinterpret_cast<uint32_t *>(dst) = bf16x2(acc[0] * inv, acc[1] * inv);
            } else {
                const int64_t prow = pair * a.max_parts + part;
                float *dst = a.ws_acc + prow * D + lane * PER;
                if constexpr (PER == 4)
                    *reinterpret_cast<float4 *>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                else
                    *reinterpret_cast<float2 *>(dst) = make_float2(acc[0], acc[1]);
                if (lane == 0) *reinterpret_cast<float2 *>(a.ws_ml + prow * 2) = make_float2(mv, lv);
            }
        }
        return;
    }
    // one slice: each warp finishes its own rows
    if (!active || wcol0 >= ncols) return;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int c = wcol0 + gq + 8 * h;
        if (c >= ncols) continue;
        const int lim_c = v.base + col_token(a, c);
        if (tok_begin > lim_c) continue;
        const int64_t pair = (int64_t)(v.row0 + col_token(a, c)) * a.Hq + kvh * a.G + col_head(a, c);
        if (lim_c < a.part_tokens) {
            const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
            uint16_t *dst = a.out + pair * D + 2 * t;
#pragma unroll
            for (int dt = 0; dt < DT; ++dt)
                *reinterpret_cast<uint32_t *>(dst + dt * 8) = bf16x2(o[dt][2 * h] * inv, o[dt][2 * h + 1] * inv);
        } else {
            const int64_t prow = pair * a.max_parts + part;
            float *dst = a.ws_acc + prow * D + 2 * t;
#pragma unroll
            for (int dt = 0; dt < DT; ++dt)
                *reinterpret_cast<float2 *>(dst + dt * 8) = make_float2(o[dt][2 * h], o[dt][2 * h + 1]);
            if (t == 0) *reinterpret_cast<float2 *>(a.ws_ml + prow * 2) = make_float2(m[h], l[h]);
        }
    }
}

// Log-sum-exp merge of a column's partitions: out = sum_p 2^(m_p - M) acc_p /
// sum_p 2^(m_p - M) l_p, M = max_p m_p.  One warp per (new token, query head) of a
// sequence (grid y); launched as a programmatic dependent of the attention kernel.
// The workspace is 256-byte aligned and a partial row is D floats, so a lane's slice
// of PER floats is a 16-byte (D 128) or 8-byte (D 64) aligned vector.
template <int D, int BS>
__global__ void __launch_bounds__(128) merge_multi_kernel(const __grid_constant__ MultiArgs a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr int PER = D / 32;
    const int lane = threadIdx.x & 31;
    const int s = blockIdx.y;
    const int jidx = blockIdx.x * 4 + (threadIdx.x >> 5);
    const SeqView v = seq_view<BS>(a, s, false);
    if (!v.ok) return;
    const int i = jidx / a.Hq, h = jidx % a.Hq;
    if (i >= v.L) return;
    const int nparts = (v.base + i) / a.part_tokens + 1;
    if (nparts <= 1) return;  // finished by the attention kernel
    const int64_t row0 = ((int64_t)(v.row0 + i) * a.Hq + h) * a.max_parts;
    float mmax = -INFINITY;
    for (int p = lane; p < nparts; p += 32) mmax = fmaxf(mmax, a.ws_ml[(row0 + p) * 2]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
    const float mbase = mmax == -INFINITY ? 0.f : mmax;
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    float lsum = 0.f;
    for (int p0 = 0; p0 < nparts; p0 += 32) {
        float f = 0.f;
        if (p0 + lane < nparts) {
            const float2 ml = *reinterpret_cast<const float2 *>(a.ws_ml + (row0 + p0 + lane) * 2);
            f = ex2(ml.x - mbase);
            lsum += f * ml.y;
        }
        const int cnt = min(32, nparts - p0);
        // vector loads of whole lane slices, eight partitions' rows in flight at once
#pragma unroll 8
        for (int q = 0; q < cnt; ++q) {
            const float fq = __shfl_sync(0xffffffffu, f, q);
            const float *src = a.ws_acc + (row0 + p0 + q) * D + lane * PER;
            if constexpr (PER == 4) {
                const float4 x = *reinterpret_cast<const float4 *>(src);
                acc[0] += fq * x.x;
                acc[1] += fq * x.y;
                acc[2] += fq * x.z;
                acc[3] += fq * x.w;
            } else {
                const float2 x = *reinterpret_cast<const float2 *>(src);
                acc[0] += fq * x.x;
                acc[1] += fq * x.y;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    uint16_t *dst = a.out + ((int64_t)(v.row0 + i) * a.Hq + h) * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; e += 2) *reinterpret_cast<uint32_t *>(dst + e) = bf16x2(acc[e] * inv, acc[e + 1] * inv);
}

template <typename KV, int D, int BS>
cudaError_t launch_multi_typed(const MultiArgs &a, cudaStream_t stream) {
    constexpr int SMEM = sizeof(KV) == 1 ? multi_smem_bytes_q<D>() : multi_smem_bytes<D>();
    static std::atomic<bool> configured[64];  // per device: the shared-memory attribute is set
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(paged_multi_kernel<KV, D, BS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        configured[dev].store(true, std::memory_order_release);
    }
    dim3 grid(a.max_parts, a.Hkv * a.CB, a.S);
    paged_multi_kernel<KV, D, BS><<<grid, kThreads, SMEM, stream>>>(a);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess || a.max_parts == 1) return err;
    return launch_multi_merge(a, D, BS, stream);
}

template <int D, int BS>
cudaError_t launch_merge_typed(const MultiArgs &a, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.max_query_len * a.Hq + 3) / 4), a.S);
    cfg.blockDim = dim3(128);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_multi_kernel<D, BS>, a);
}

}  // namespace

int multi_cols_per_cta() { return kColsPerCta; }

cudaError_t launch_multi_merge(const MultiArgs &a, int D, int bs, cudaStream_t stream) {
    if (D == 128) return bs == 16 ? launch_merge_typed<128, 16>(a, stream) : launch_merge_typed<128, 32>(a, stream);
    return bs == 16 ? launch_merge_typed<64, 16>(a, stream) : launch_merge_typed<64, 32>(a, stream);
}

template <typename KV>
cudaError_t launch_multi_kv(const MultiArgs &a, int D, int bs, cudaStream_t stream) {
    if (D == 128)
        return bs == 16 ? launch_multi_typed<KV, 128, 16>(a, stream) : launch_multi_typed<KV, 128, 32>(a, stream);
    return bs == 16 ? launch_multi_typed<KV, 64, 16>(a, stream) : launch_multi_typed<KV, 64, 32>(a, stream);
}

bool multi_per_token_eligible(int D, int kv_dtype, int G, int max_query_len) {
    (void)D;
    (void)G;
    // draft verification with an 8-bit cache: the decode kernel keeps the codes in
    // registers and converts each tile once per CTA, where the mma.sync kernel converts
    // through shared memory between barriers (measured on GB300 with an fp8 cache,
    // 70B-shaped 4-token verification: 263 us on the mma.sync kernel)
    return (kv_dtype == PA_KV_INT8 || kv_dtype == PA_KV_FP8) && max_query_len <= kPerTokenMaxQuery;
}

// Per-token mode of the decode kernel: the multi-token arguments as decode arguments,
// then the multi-token merge over the same [T][Hq][max_parts] partials.
static cudaError_t launch_multi_per_token(const MultiArgs &m, int D, int bs, int kv_dtype, cudaStream_t stream) {
    DecodeArgs a{};
    a.out = m.out;
    a.q = m.q;
    a.k_cache = m.k_cache;
    a.v_cache = m.v_cache;
    a.k_scale = m.k_scale;
    a.v_scale = m.v_scale;
    a.block_tables = m.block_tables;
    a.context_lens = m.context_lens;
    a.ws_acc = m.ws_acc;
    a.ws_ml = m.ws_ml;
    a.err_flag = m.err_flag;
    a.M = m.M;
    a.S = m.S;
    a.Hq = m.Hq;
    a.Hkv = m.Hkv;
    a.G = m.G;
    a.N = m.N;
    a.head_chunks = (m.G + 7) / 8;
    a.part_tokens = m.part_tokens;
    a.max_parts = m.max_parts;
    a.max_context_len = m.max_context_len;
    a.scale_log2 = m.scale_log2;
    a.query_start = m.query_start;
    a.T = m.T;
    a.Lq = m.max_query_len;
    a.rows_per_cta = decode_rows_per_cta(m.max_query_len);
    cudaError_t err = launch_decode_rows(a, D, bs, kv_dtype, stream);
    if (err != cudaSuccess || m.max_parts == 1) return err;
    return launch_multi_merge(m, D, bs, stream);
}

cudaError_t launch_multi_token(const MultiArgs &a, int D, int bs, int kv_dtype, cudaStream_t stream) {
    if (kv_dtype == PA_KV_BF16 && multi_tc_eligible(D, kv_dtype, a.G, a.max_query_len)) return launch_multi_tc(a, bs, stream);
    if (!multi_tc_eligible(D, kv_dtype, a.G, a.max_query_len) &&
        multi_per_token_eligible(D, kv_dtype, a.G, a.max_query_len))
        return launch_multi_per_token(a, D, bs, kv_dtype, stream);
    if (kv_dtype == PA_KV_INT8) return launch_multi_kv<int8_t>(a, D, bs, stream);
    if (kv_dtype == PA_KV_FP8) return launch_multi_kv<e4m3_tag>(a, D, bs, stream);
    return launch_multi_kv<uint16_t>(a, D, bs, stream);
}

}  // namespace pa
