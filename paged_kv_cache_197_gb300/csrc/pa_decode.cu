// Paged decode attention for GB300 (sm_103a).
//
// What is computed (deeplearn.tn KV-cache article, "Le compromis fondamental de
// l'inference"; blog.fabienvernieres.com "Cache KV en production", opening
// section): for every sequence s and query head h, the new token's query attends
// over the sequence's cached keys and values,
//   out[s][h] = sum_t softmax_t(scale * q . K[t]) V[t],
// with K[t], V[t] gathered from physical block block_tables[s][t / bs] at offset
// t % bs (gotburnout.io "PagedAttention & Gestion du KV-Cache", section 2
// block-table figure) from kv head h / G.
//
// Design (decode is bound by HBM bandwidth; every K/V byte is read once):
//   * One CTA of 4 warps per (sequence, kv head, group of <= 8 query heads,
//     partition of 256 to 4096 tokens, chosen on the host).  Warps take the partition's tiles round-robin and
//     each keeps its own online-softmax state; the CTA merges its warps in shared
//     memory.  Longer contexts are split over several CTAs whose partial results
//     (unnormalised output, running max, running sum) a second kernel, launched as a
//     programmatic dependent, merges by log-sum-exp.
//   * A tile is 16 tokens (bf16) or a whole block (int8) of one kv head: one
//     contiguous run of bytes in the [N][Hkv][bs][D] cache.  Each lane loads its
//     share with 16-byte loads straight into registers, in the layout the tensor-
//     core fragments need, so no shared-memory staging is required and every
//     32-byte sector fetched is fully used.  The next tile's loads are issued
//     before the current tile is consumed.
//   * q.K^T and P.V of the query-head group run on the tensor cores
//     (mma.sync m16n8k16, bf16 in, fp32 accumulate): S[16 tokens x 8 heads] =
//     K_tile . q^T, then O^T[D x 8 heads] += V^T . P^T.  The head dimension order
//     inside a lane is permuted consistently for q and K (a dot product does not
//     depend on it), which turns each lane's K loads into whole 16-byte vectors.
//     P leaves the first product as a C fragment and enters the second as a B
//     fragment after one movmatrix transpose per 8x8 quarter.
//   * int8 entries are turned into exact bf16 integers with integer ops; the key
//     scale multiplies the score, the value scale multiplies the softmax weight.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <type_traits>

#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxPartBlocks = 256;  // 4096-token partitions of 16-token blocks
constexpr int kHeadsPerCta = 8;
constexpr int kMergeInRegs = 16;  // partitions whose partial rows the merge loads at once
constexpr float kRescaleLog2 = 8.0f;  // running-max slack before O is rescaled (log2 units)

// ------------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ void ldg16(uint32_t *w, const void *p) {
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
        : "l"(p));
}

__device__ __forceinline__ void ldg8(uint32_t *w, const void *p) {
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "l"(p));
}

template <int NB>
__device__ __forceinline__ void ldg_bytes(uint32_t *w, const char *p) {
    static_assert(NB % 8 == 0, "8-byte granules");
    if constexpr (NB % 16 == 0) {
#pragma unroll
        for (int i = 0; i < NB / 16; ++i) ldg16(w + 4 * i, p + 16 * i);
    } else {
        ldg8(w, p);
    }
}

// D = A . B + D, A 16x16 bf16 (row), B 16x8 bf16 (col), D 16x8 fp32.
__device__ __forceinline__ void mma_bf16(float *c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A . B + D, A 16x16 fp16 (row), B 16x8 fp16 (col), D 16x8 fp32.
__device__ __forceinline__ void mma_f16(float *c, uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose an 8x8 matrix of 16-bit values held one row pair per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// int8 -> fp16, biased.  The fp16 bit pattern 0x64XX is 1024 + XX for XX in
// [0, 255]; with XX = x + 128 (the int8 byte with its top bit flipped) the value is
// 1152 + x, exactly.  The tensor-core products take these biased values and the bias
// is taken out of their fp32 results instead: a score loses kInt8Bias * sum_d q_d
// (fixed per head), an output element kInt8Bias * sum_t p_t over the fp16 weights
// fed to the product -- one subtraction per result rather than one per converted
// pair.
constexpr float kInt8Bias = 1152.0f;

// The four int8 values of word w (one K row) as the biased fp16 pairs (w0, w1), (w2, w3).
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    lo = __byte_perm(u, 0x64646464u, 0x4140);
    hi = __byte_perm(u, 0x64646464u, 0x4342);
}

// Byte 0 and byte 2 of t hold int8 values a and b (bytes 1 and 3 are ignored): the
// biased fp16 pair (a, b).  One logic op flips the top bits and writes the 0x64 bytes.
__device__ __forceinline__ uint32_t i8pair_to_f16x2(uint32_t t) {
    const uint32_t m = 0x00ff00ffu, c = 0x64806480u;
    return (m & (t ^ c)) | (~m & c);
}

// fp8 (e4m3) cache entries: every e4m3 value is exactly an fp16 value, and the
// hardware converts a pair with one instruction (low byte -> low half).
struct e4m3_t {
    uint8_t bits;
};

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t pair16) {
    uint32_t out;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
        : "=r"(out)
        : "r"(pair16));
    return out;
}

// The four 8-bit entries of word w (one K row, d = 4t .. 4t+3 of a 16-wide step) as
// the fp16 pairs (w0, w1), (w2, w3).
template <typename KV>
__device__ __forceinline__ void k8x4_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi) {
    if constexpr (sizeof(KV) == 1 && !std::is_same<KV, e4m3_t>::value) {
        i8x4_to_f16(w, lo, hi);
    } else {
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
            : "=r"(lo), "=r"(hi)
            : "r"(w));
    }
}

// The fp16 pair (A.byte j, B.byte j): entry j of two V rows (two tokens).
template <typename KV>
__device__ __forceinline__ uint32_t v8_pair_to_f16(uint32_t A, uint32_t B, uint32_t j) {
    if constexpr (std::is_same<KV, e4m3_t>::value)
        return e4m3x2_to_f16x2(__byte_perm(A, B, j | ((4u + j) << 4)));
    else
        return i8pair_to_f16x2(__byte_perm(A, B, j | ((4u + j) << 8)));
}

// Exponent e with |x| < 2^e for a finite, positive x (normal range).
__device__ __forceinline__ int exponent_above(float x) {
    return (int)((__float_as_uint(x) >> 23) & 0xffu) - 126;
}

__device__ __forceinline__ void raise_flag(int *err_flag, int bit) {
    if (err_flag) atomicOr(err_flag, bit);
}

// Context length after the range checks: negative -> 0, beyond the table or the
// planned maximum -> clamped.
__device__ __forceinline__ int checked_context(const DecodeArgs &a, int s, int bs, bool report) {
    int ctx = a.context_lens[s];
    const int lim = min(a.M * bs, a.max_context_len);
    if (ctx < 0 || ctx > lim) {
        if (report) raise_flag(a.err_flag, PA_FLAG_CONTEXT_OUT_OF_RANGE);
        ctx = ctx < 0 ? 0 : lim;
    }
    return ctx;
}

// ---------------------------------------------------------------- tile geometry
template <typename KV, int D, int TILE>
struct Geo {
    static constexpr int ELEM = sizeof(KV);
    static constexpr int ROW_BYTES = D * ELEM;     // one token of one kv head
    static constexpr int K_ROWS = TILE / 8;        // K rows per lane: tokens g + 8r
    static constexpr int K_CHUNKS = ROW_BYTES / 64;  // 16-byte chunks per K row per lane
    static constexpr int K_WORDS = K_CHUNKS * 4;
    static constexpr int V_TOKS = TILE / 4;        // V rows per lane
    static constexpr int V_BYTES = ROW_BYTES / 8;  // bytes of one V row per lane
    static constexpr int V_WORDS = V_BYTES / 4;
    static constexpr int KSTEPS = D / 16;          // k-steps of the score product
    static constexpr int MT = D / 16;              // d tiles of the output product
    static constexpr int SUB = TILE / 16;          // 16-token sub-tiles
    static constexpr int QW = D / 8;               // q words per lane
    // int8 entries enter the products biased by kInt8Bias (fp8 ones are exact)
    static constexpr bool BIASED = std::is_same<KV, int8_t>::value;
    static_assert(K_CHUNKS >= 1 && V_BYTES >= 8, "unsupported head_dim / dtype");
};

template <class GEO>
struct Tile {
    uint32_t k[GEO::K_ROWS][GEO::K_WORDS];
    uint32_t v[GEO::V_TOKS][GEO::V_WORDS];
    float ks, vs;  // int8: scales of token `lane` of the tile
    int nvalid;    // tokens of the partition from the tile's first on (>= TILE: all valid)
};

// V row j of a lane: sub-tile j / 4, token 2t, 2t+1, 2t+8 or 2t+9 of it.
__device__ __forceinline__ int v_token(int j, int t) {
    const int jj = j & 3;
    return 16 * (j >> 2) + 2 * t + (jj & 1) + ((jj >> 1) << 3);
}

template <typename KV, int D, int BS, int TILE>
__device__ __forceinline__ void load_tile(Tile<Geo<KV, D, TILE>> &R, const DecodeArgs &a,
                                          const int *s_blk, int blk_begin, int tok_begin,
                                          int tok_end, int i, int kvh, int g, int t, int lane) {
    using G_ = Geo<KV, D, TILE>;
    const int tok0 = tok_begin + i * TILE;
    int blk = s_blk[tok0 / BS - blk_begin];
    R.nvalid = tok_end - tok0;  // may exceed TILE: tokens of the partition from this tile on
    if (blk < 0) {  // flagged when the table was read: the tile is skipped
        R.nvalid = 0;
        blk = 0;
    }
    const int off = tok0 % BS;
    const int64_t row0 = ((int64_t)blk * a.Hkv + kvh) * BS + off;
    const char *kb = static_cast<const char *>(a.k_cache) + row0 * G_::ROW_BYTES;
    const char *vb = static_cast<const char *>(a.v_cache) + row0 * G_::ROW_BYTES;
#pragma unroll
    for (int r = 0; r < G_::K_ROWS; ++r)
#pragma unroll
        for (int c = 0; c < G_::K_CHUNKS; ++c)
            ldg16(&R.k[r][4 * c], kb + (g + 8 * r) * G_::ROW_BYTES + c * 64 + t * 16);
#pragma unroll
    for (int j = 0; j < G_::V_TOKS; ++j) {
        const char *row = vb + v_token(j, t) * G_::ROW_BYTES;
        if constexpr (G_::ELEM == 2) {
            // two runs of D/16 values: d in [h*D/2 + g*D/16, +D/16), h = 0, 1
            ldg_bytes<G_::V_BYTES / 2>(&R.v[j][0], row + g * (G_::V_BYTES / 2));
            ldg_bytes<G_::V_BYTES / 2>(&R.v[j][G_::V_WORDS / 2],
                                       row + G_::ROW_BYTES / 2 + g * (G_::V_BYTES / 2));
        } else {
            // one run of D/8 values: d in [g*D/8, +D/8)
            ldg_bytes<G_::V_BYTES>(&R.v[j][0], row + g * G_::V_BYTES);
        }
    }
    if constexpr (G_::ELEM == 1) {
        const int64_t srow = row0 + (lane < TILE ? lane : 0);
        R.ks = __ldg(a.k_scale + srow);
        R.vs = __ldg(a.v_scale + srow);
    }
}

// Head-dim index of the e-th value a lane holds of a K row (and of q): lane quad t
// owns 16-byte chunks c*64 + t*16 of each K row.
template <int ELEM>
__device__ __forceinline__ int k_dim(int e, int t) {
    constexpr int PER = 16 / ELEM;  // values per 16-byte chunk
    return (e / PER) * (64 / ELEM) + t * PER + e % PER;
}

// Head-dim index held in row g (h = 0) or g + 8 (h = 1) of output d-tile mt.
template <int ELEM, int D>
__device__ __forceinline__ int out_dim(int mt, int g, int h) {
    if constexpr (ELEM == 2)
        return h * (D / 2) + g * (D / 16) + mt;
    else
        return g * (D / 8) + 2 * mt + h;
}

// One warp's online-softmax state for NC column sets.  A column set is the CTA's
// query heads for one query token: decode has one, a CTA serving several new tokens
// of a multi-token call one per token.
template <typename KV, int D, int TILE, int NC>
struct WarpState {
    float o[NC][D / 16][4];  // O^T fragments: [set][d tile][c0..c3]
    float m[NC][2];          // running max of heads 2t, 2t+1 (log2 units)
    float l[NC][2];          // running sum, partial over this lane's tokens
    int ve;                  // 8-bit: O is kept in units of 2^ve (ve >= exponent of every value scale so far)
    float ps[NC][2];         // int8: sum of the fp16 weights fed to the value product, heads 2t, 2t+1
};

// Consume one tile for NC column sets.  Set c sees the tile's first R.nvalid - cut[c]
// tokens (its own causal limit); every K and V entry is converted once and feeds the
// products of all sets.
template <typename KV, int D, int TILE, int NC>
__device__ __forceinline__ void consume_tile(WarpState<KV, D, TILE, NC> &st, Tile<Geo<KV, D, TILE>> &R,
                                             const uint32_t (&qw)[NC][Geo<KV, D, TILE>::QW],
                                             const float (&qb)[NC][2], const float (&scale_log2)[NC],
                                             const int (&cut)[NC], int g, int t) {
    using G_ = Geo<KV, D, TILE>;
    // ---- scores S[token][head] for the tile's 16-token sub-tiles
    float sc[NC][G_::SUB][4];
#pragma unroll
    for (int s = 0; s < G_::SUB; ++s) {
#pragma unroll
        for (int c = 0; c < NC; ++c) sc[c][s][0] = sc[c][s][1] = sc[c][s][2] = sc[c][s][3] = 0.0f;
#pragma unroll
        for (int kc = 0; kc < G_::KSTEPS; ++kc) {
            uint32_t a0, a1, a2, a3;
            if constexpr (G_::ELEM == 2) {
                a0 = R.k[2 * s][2 * kc];
                a2 = R.k[2 * s][2 * kc + 1];
                a1 = R.k[2 * s + 1][2 * kc];
                a3 = R.k[2 * s + 1][2 * kc + 1];
#pragma unroll
                for (int c = 0; c < NC; ++c) mma_bf16(sc[c][s], a0, a1, a2, a3, qw[c][2 * kc], qw[c][2 * kc + 1]);
            } else {
                k8x4_to_f16<KV>(R.k[2 * s][kc], a0, a2);
                k8x4_to_f16<KV>(R.k[2 * s + 1][kc], a1, a3);
#pragma unroll
                for (int c = 0; c < NC; ++c) mma_f16(sc[c][s], a0, a1, a2, a3, qw[c][2 * kc], qw[c][2 * kc + 1]);
            }
        }
    }
    // ---- online softmax over the tile (log2 domain), per column set
    float ksc[G_::SUB][2];  // 8-bit: key scales of tokens g and g + 8 of each sub-tile
    if constexpr (G_::ELEM == 1) {
#pragma unroll
        for (int s = 0; s < G_::SUB; ++s) {
            ksc[s][0] = __shfl_sync(0xffffffffu, R.ks, 16 * s + g);
            ksc[s][1] = __shfl_sync(0xffffffffu, R.ks, 16 * s + g + 8);
        }
    }
    float x[NC][G_::SUB][4];
    float base[NC][2];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const int lim = R.nvalid - cut[c];
        // one multiplier per (sub-tile, token row): the softmax scale, times the key
        // scale for an 8-bit cache; int8: the bias comes off in the same fused step
        float kk[G_::SUB][2], qk[G_::SUB][2][2];
#pragma unroll
        for (int s = 0; s < G_::SUB; ++s)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                kk[s][h] = G_::ELEM == 1 ? scale_log2[c] * ksc[s][h] : scale_log2[c];
                if constexpr (G_::BIASED) {
                    qk[s][h][0] = qb[c][0] * kk[s][h];
                    qk[s][h][1] = qb[c][1] * kk[s][h];
                }
            }
#pragma unroll
        for (int s = 0; s < G_::SUB; ++s)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                x[c][s][e] = G_::BIASED ? fmaf(sc[c][s][e], kk[s][e >> 1], -qk[s][e >> 1][e & 1])
                                        : sc[c][s][e] * kk[s][e >> 1];
        if (lim < TILE) {  // a tile the set sees only in part (uniform across the warp)
#pragma unroll
            for (int s = 0; s < G_::SUB; ++s)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (16 * s + g + 8 * (e >> 1) >= lim) x[c][s][e] = -INFINITY;
        }
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int s = 0; s < G_::SUB; ++s)
#pragma unroll
            for (int e = 0; e < 4; ++e) mx[e & 1] = fmaxf(mx[e & 1], x[c][s][e]);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 4));
            mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 8));
            mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 16));
        }
        float alpha[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            // the running max moves only when the tile's max exceeds it by more than
            // kRescaleLog2 (weights then stay below 2^kRescaleLog2: fine in fp32, and in
            // fp16 for the 8-bit products, whose weights carry value scales below 1)
            const float mnew = mx[j] > st.m[c][j] + kRescaleLog2 ? mx[j] : st.m[c][j];
            base[c][j] = mnew == -INFINITY ? 0.0f : mnew;
            alpha[j] = fast_exp2(st.m[c][j] - base[c][j]);
            st.m[c][j] = mnew;
        }
        if (__any_sync(0xffffffffu, alpha[0] != 1.0f || alpha[1] != 1.0f)) {
#pragma unroll
            for (int mt = 0; mt < G_::MT; ++mt) {
                st.o[c][mt][0] *= alpha[0];
                st.o[c][mt][1] *= alpha[1];
                st.o[c][mt][2] *= alpha[0];
                st.o[c][mt][3] *= alpha[1];
            }
            st.l[c][0] *= alpha[0];
            st.l[c][1] *= alpha[1];
            if constexpr (G_::BIASED) {
                st.ps[c][0] *= alpha[0];
                st.ps[c][1] *= alpha[1];
            }
        }
    }
    // 8-bit: keep the weights p * v_scale below 1 in fp16 by working in units of 2^ve,
    // ve the exponent of the largest value scale seen so far (O rescaled when it grows)
    float vmul = 1.0f;
    if constexpr (G_::ELEM == 1) {
        const float vl = (int)(threadIdx.x & 31) < R.nvalid ? R.vs : 0.0f;
        // only a tile holding a value scale of a higher exponent raises ve (one vote
        // instead of a reduction in the common case)
        if (__any_sync(0xffffffffu, vl > 0.0f && exponent_above(vl) > st.ve)) {
            float vmax = vl;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
            const int e = exponent_above(vmax);
            {
                const float f = st.ve < -200 ? 0.0f : ldexpf(1.0f, st.ve - e);
#pragma unroll
                for (int c = 0; c < NC; ++c) {
#pragma unroll
                    for (int mt = 0; mt < G_::MT; ++mt) {
                        st.o[c][mt][0] *= f;
                        st.o[c][mt][1] *= f;
                        st.o[c][mt][2] *= f;
                        st.o[c][mt][3] *= f;
                    }
                    if constexpr (G_::BIASED) {
                        st.ps[c][0] *= f;
                        st.ps[c][1] *= f;
                    }
                }
                st.ve = e;
            }
        }
        vmul = ldexpf(1.0f, -st.ve);
    }
    // ---- values: zero rows past the context (they may hold any bit pattern)
    if (R.nvalid < TILE) {
#pragma unroll
        for (int j = 0; j < G_::V_TOKS; ++j)
            if (v_token(j, t) >= R.nvalid)
#pragma unroll
                for (int w = 0; w < G_::V_WORDS; ++w) R.v[j][w] = 0u;
    }
#pragma unroll
    for (int s = 0; s < G_::SUB; ++s) {
        float vsc[2];  // 8-bit: value scales of tokens g and g + 8 of the sub-tile, in units of 2^ve
        if constexpr (G_::ELEM == 1) {
            vsc[0] = __shfl_sync(0xffffffffu, R.vs, 16 * s + g) * vmul;
            vsc[1] = __shfl_sync(0xffffffffu, R.vs, 16 * s + g + 8) * vmul;
        }
        // P[head][token] of each set as the B operand: transpose the [token][head] quarters
        uint32_t b0[NC], b1[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const int lim = R.nvalid - cut[c];
            float p[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                p[e] = fast_exp2(x[c][s][e] - base[c][e & 1]);
                st.l[c][e & 1] += p[e];
                if constexpr (G_::ELEM == 1) p[e] *= vsc[e >> 1];
            }
            if constexpr (G_::ELEM == 1) {
                // tokens the set does not see: a zero weight (their scales may be NaN)
                if (lim < TILE) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (16 * s + g + 8 * (e >> 1) >= lim) p[e] = 0.0f;
                }
            }
            if constexpr (G_::ELEM == 2) {
                b0[c] = movmatrix_trans(pack_bf16x2(p[0], p[1]));
                b1[c] = movmatrix_trans(pack_bf16x2(p[2], p[3]));
            } else {
                const uint32_t w0 = pack_f16x2(p[0], p[1]), w1 = pack_f16x2(p[2], p[3]);
                if constexpr (G_::BIASED) {  // the weights exactly as the product sees them
                    const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&w0));
                    const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&w1));
                    st.ps[c][0] += f0.x + f1.x;
                    st.ps[c][1] += f0.y + f1.y;
                }
                b0[c] = movmatrix_trans(w0);
                b1[c] = movmatrix_trans(w1);
            }
        }
        const int j0 = 4 * s;  // V rows 2t, 2t+1, 2t+8, 2t+9 of this sub-tile
#pragma unroll
        for (int mt = 0; mt < G_::MT; ++mt) {
            uint32_t a0, a1, a2, a3;
            if constexpr (G_::ELEM == 2) {
                constexpr int HW = G_::V_WORDS / 2;
                const int w = mt >> 1;
                const uint32_t sel = (mt & 1) ? 0x7632u : 0x5410u;
                a0 = __byte_perm(R.v[j0][w], R.v[j0 + 1][w], sel);
                a1 = __byte_perm(R.v[j0][HW + w], R.v[j0 + 1][HW + w], sel);
                a2 = __byte_perm(R.v[j0 + 2][w], R.v[j0 + 3][w], sel);
                a3 = __byte_perm(R.v[j0 + 2][HW + w], R.v[j0 + 3][HW + w], sel);
            } else {
                const int w = mt >> 1;
                const uint32_t b = 2u * (mt & 1);
                a0 = v8_pair_to_f16<KV>(R.v[j0][w], R.v[j0 + 1][w], b);
                a1 = v8_pair_to_f16<KV>(R.v[j0][w], R.v[j0 + 1][w], b + 1u);
                a2 = v8_pair_to_f16<KV>(R.v[j0 + 2][w], R.v[j0 + 3][w], b);
                a3 = v8_pair_to_f16<KV>(R.v[j0 + 2][w], R.v[j0 + 3][w], b + 1u);
            }
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                if constexpr (G_::ELEM == 2)
                    mma_bf16(st.o[c][mt], a0, a1, a2, a3, b0[c], b1[c]);
                else
                    mma_f16(st.o[c][mt], a0, a1, a2, a3, b0[c], b1[c]);
            }
        }
    }
}

// NT == 0: decode, one query row per sequence (grid x = partition).  NT >= 1: rows
// mode of a multi-token call, NT consecutive new tokens of a sequence per CTA (grid x =
// partition x token groups), each token a column set with its own causal limit.
// SINGLE (decode only): one tile register set per warp instead of two (the next
// tile is not prefetched), three or four CTAs per SM: twelve or sixteen warps per SM
// keep loads in flight where eight double-buffered ones did.
template <typename KV, int D, int BS, int TILE, int NT, bool SINGLE>
__device__ __forceinline__ void decode_body(const DecodeArgs &a) {
    using G_ = Geo<KV, D, TILE>;
    constexpr bool ROWS = NT > 0;
    constexpr int NC = ROWS ? NT : 1;
    static_assert(BS % TILE == 0, "a tile lies inside one block");
    __shared__ int s_blk[kMaxPartBlocks];
    __shared__ float s_m[kWarps][kHeadsPerCta];
    __shared__ float s_l[kWarps][kHeadsPerCta];
    __shared__ __align__(16) float s_o[kWarps][kHeadsPerCta][D];

    const int groups = ROWS ? (a.Lq + NC - 1) / NC : 1;
    const int part = ROWS ? blockIdx.x / groups : blockIdx.x;
    const int kvh = blockIdx.y / a.head_chunks;
    const int chunk = blockIdx.y % a.head_chunks;
    const int s = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;

    // everything this kernel reads may come from the kernel before it on the stream
    // (a programmatic dependent launch): wait for that grid before any load
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const bool reporter = blockIdx.x == 0 && blockIdx.y == 0 && tid == 0;
    int ctx = checked_context(a, s, BS, reporter);
    int row0 = s;  // q / out row of column set 0 (set c: row0 + c)
    int nt = 1;    // column sets in use
    if constexpr (ROWS) {
        // new tokens i0 .. i0 + nt - 1 of sequence s: rows [r0, r1) of the call, token i
        // attends the first ctx - L + i + 1 tokens
        const int i0 = (blockIdx.x - part * groups) * NC;
        const int r0 = a.query_start[s], r1 = a.query_start[s + 1], L = r1 - r0;
        if (!(r0 >= 0 && r1 <= a.T && L >= 0 && L <= ctx && L <= a.Lq)) {
            if (reporter) raise_flag(a.err_flag, PA_FLAG_QUERY_OUT_OF_RANGE);
            return;
        }
        if (i0 >= L) return;
        nt = min(NC, L - i0);
        ctx = ctx - L + i0 + nt;  // the last set's limit
        row0 = r0 + i0;
    }
    // tokens before `start` (a shared prefix, attended by the grouped prefix kernel)
    // are skipped; start is a multiple of the block size
    const int start = (!ROWS && a.start_tokens) ? min(a.start_tokens[s], ctx) : 0;
    const int nparts = max(1, (ctx - start + a.part_tokens - 1) / a.part_tokens);
    if (part >= nparts) return;
    const int tok_begin = start + part * a.part_tokens;
    const int tok_end = min(ctx, tok_begin + a.part_tokens);
    const int blk_begin = tok_begin / BS;
    const int nblk = max(0, (tok_end - tok_begin + BS - 1) / BS);
    const int h0 = kvh * a.G + chunk * kHeadsPerCta;
    const int nh = min(kHeadsPerCta, a.G - chunk * kHeadsPerCta);
    // tokens of the partition that set c does not see (its limit is nt - 1 - c below
    // the last set's); sets past nt see none
    int cut[NC];
    if constexpr (ROWS) {
#pragma unroll
        for (int c = 0; c < NC; ++c)
            cut[c] = c < nt ? tok_end - min(ctx - (nt - 1 - c), tok_begin + a.part_tokens) : (1 << 30);
    } else {
        cut[0] = 0;
    }

    for (int i = tid; i < nblk; i += kThreads) {
        int b = a.block_tables[(int64_t)s * a.M + blk_begin + i];
        if (b < 0 || b >= a.N) {
            if (chunk == 0) raise_flag(a.err_flag, PA_FLAG_BLOCK_OUT_OF_RANGE);
            b = -1;
        }
        s_blk[i] = b;
    }

    // q fragments: lane (g, t) holds head g's values at the K-row positions it owns
    uint32_t qw[NC][G_::QW];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        if (g < nh && c < nt) {
            const char *qrow = reinterpret_cast<const char *>(a.q + ((int64_t)(row0 + c) * a.Hq + h0 + g) * D);
#pragma unroll
            for (int k = 0; k < G_::K_CHUNKS; ++k)
                ldg_bytes<32 / G_::ELEM>(&qw[c][k * (8 / G_::ELEM)],
                                         qrow + 2 * k_dim<G_::ELEM>(k * (16 / G_::ELEM), t));
        } else {
#pragma unroll
            for (int i = 0; i < G_::QW; ++i) qw[c][i] = 0u;
        }
    }
    float scale_log2[NC];
    float qb[NC][2];  // int8: score bias per score column
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        scale_log2[c] = a.scale_log2;
        qb[c][0] = qb[c][1] = 0.0f;
        if constexpr (G_::ELEM == 1) {
            // fp16 q for the 8-bit products: scaled by 2^sig so the largest |q| of the
            // set's heads lands in [2^13, 2^14); the scores are scaled back by 2^-sig
            float qmax = 0.0f;
#pragma unroll
            for (int i = 0; i < G_::QW; ++i)
                qmax = fmaxf(qmax, fmaxf(fabsf(__uint_as_float(qw[c][i] << 16)),
                                         fabsf(__uint_as_float(qw[c][i] & 0xffff0000u))));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, o));
            const int sig = qmax > 0.0f ? min(100, max(-100, 14 - exponent_above(qmax))) : 0;
            const float up = ldexpf(1.0f, sig);
#pragma unroll
            for (int i = 0; i < G_::QW; ++i)
                qw[c][i] = pack_f16x2(__uint_as_float(qw[c][i] << 16) * up,
                                      __uint_as_float(qw[c][i] & 0xffff0000u) * up);
            scale_log2[c] *= ldexpf(1.0f, -sig);
            if constexpr (G_::BIASED) {
                // kInt8Bias * sum_d q_d of the fp16 q fed to the score product, for the
                // heads of this lane's score columns (2t, 2t+1; head g sits in lanes 4g..)
                float sum = 0.0f;
#pragma unroll
                for (int i = 0; i < G_::QW; ++i) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&qw[c][i]));
                    sum += f.x + f.y;
                }
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                qb[c][0] = kInt8Bias * __shfl_sync(0xffffffffu, sum, 8 * t);
                qb[c][1] = kInt8Bias * __shfl_sync(0xffffffffu, sum, 8 * t + 4);
            }
        }
    }
    __syncthreads();

    WarpState<KV, D, TILE, NC> st;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
#pragma unroll
        for (int mt = 0; mt < G_::MT; ++mt) st.o[c][mt][0] = st.o[c][mt][1] = st.o[c][mt][2] = st.o[c][mt][3] = 0.f;
        st.m[c][0] = st.m[c][1] = -INFINITY;
        st.l[c][0] = st.l[c][1] = 0.0f;
        st.ps[c][0] = st.ps[c][1] = 0.0f;
    }
    st.ve = -1000;  // no value scale seen yet

    const int ntiles = (tok_end - tok_begin + TILE - 1) / TILE;
    if constexpr (SINGLE) {
        Tile<G_> A;
        for (int i = warp; i < ntiles; i += kWarps) {
            load_tile<KV, D, BS, TILE>(A, a, s_blk, blk_begin, tok_begin, tok_end, i, kvh, g, t, lane);
            consume_tile<KV, D, TILE, NC>(st, A, qw, qb, scale_log2, cut, g, t);
        }
    } else {
        Tile<G_> A, B;
        int i = warp;
        if (i < ntiles) load_tile<KV, D, BS, TILE>(A, a, s_blk, blk_begin, tok_begin, tok_end, i, kvh, g, t, lane);
        while (i < ntiles) {
            if (i + kWarps < ntiles)
                load_tile<KV, D, BS, TILE>(B, a, s_blk, blk_begin, tok_begin, tok_end, i + kWarps, kvh, g, t, lane);
            consume_tile<KV, D, TILE, NC>(st, A, qw, qb, scale_log2, cut, g, t);
            i += kWarps;
            if (i >= ntiles) break;
            if (i + kWarps < ntiles)
                load_tile<KV, D, BS, TILE>(A, a, s_blk, blk_begin, tok_begin, tok_end, i + kWarps, kvh, g, t, lane);
            consume_tile<KV, D, TILE, NC>(st, B, qw, qb, scale_log2, cut, g, t);
            i += kWarps;
        }
    }

    // the dependent merge grid may launch once every CTA got here (it still waits for
    // this grid to finish before reading)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const float oscale = (G_::ELEM == 1 && st.ve > -200) ? ldexpf(1.0f, st.ve) : 1.0f;
    constexpr int DPT = D / 16;  // output values per thread: 16 threads per head
    const int hj = tid >> 4;
    const int d0 = (tid & 15) * DPT;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        if (c >= nt) break;  // uniform across the CTA
        if (c > 0) __syncthreads();  // the previous set's reads of shared memory are done
        // ---- per-warp totals, then merge the CTA's warps through shared memory
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            st.l[c][j] += __shfl_xor_sync(0xffffffffu, st.l[c][j], 4);
            st.l[c][j] += __shfl_xor_sync(0xffffffffu, st.l[c][j], 8);
            st.l[c][j] += __shfl_xor_sync(0xffffffffu, st.l[c][j], 16);
        }
        if (g == 0) {
            s_m[warp][2 * t] = st.m[c][0];
            s_m[warp][2 * t + 1] = st.m[c][1];
            s_l[warp][2 * t] = st.l[c][0];
            s_l[warp][2 * t + 1] = st.l[c][1];
        }
        float obias[2] = {0.0f, 0.0f};  // int8: kInt8Bias * the weights summed over all tokens
        if constexpr (G_::BIASED) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float v = st.ps[c][j];
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                obias[j] = kInt8Bias * v;
            }
        }
#pragma unroll
        for (int mt = 0; mt < G_::MT; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                s_o[warp][2 * t + (e & 1)][out_dim<G_::ELEM, D>(mt, g, e >> 1)] =
                    (st.o[c][mt][e] - obias[e & 1]) * oscale;
        __syncthreads();

        // set c's partitions: those of its own limit (the last set's for decode)
        const int nparts_c = ROWS ? max(1, (ctx - (nt - 1 - c) + a.part_tokens - 1) / a.part_tokens) : nparts;
        if (hj < nh && part < nparts_c) {
            float mmax = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) mmax = fmaxf(mmax, s_m[w][hj]);
            const float mbase = mmax == -INFINITY ? 0.0f : mmax;
            float acc[DPT];
#pragma unroll
            for (int e = 0; e < DPT; ++e) acc[e] = 0.0f;
            float lsum = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float f = fast_exp2(s_m[w][hj] - mbase);
                lsum += f * s_l[w][hj];
#pragma unroll
                for (int e = 0; e < DPT; ++e) acc[e] += f * s_o[w][hj][d0 + e];
            }
            const int h = h0 + hj;
            const int64_t row = row0 + c;
            if (nparts_c == 1 && !a.partials_only) {
                const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
                uint32_t packed[DPT / 2];
#pragma unroll
                for (int e = 0; e < DPT / 2; ++e) packed[e] = pack_bf16x2(acc[2 * e] * inv, acc[2 * e + 1] * inv);
                uint16_t *dst = a.out + (row * a.Hq + h) * D + d0;
                if constexpr (DPT == 8)
                    *reinterpret_cast<uint4 *>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                else
                    *reinterpret_cast<uint2 *>(dst) = make_uint2(packed[0], packed[1]);
            } else {
                const int64_t prow = (row * a.Hq + h) * a.max_parts + part;
                float *dst = a.ws_acc + prow * D + d0;
#pragma unroll
                for (int e = 0; e < DPT; e += 4)
                    *reinterpret_cast<float4 *>(dst + e) = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
                if ((tid & 15) == 0) *reinterpret_cast<float2 *>(a.ws_ml + prow * 2) = make_float2(mmax, lsum);
            }
        }
    }
}

template <typename KV, int D, int BS, int TILE, int NT>
__global__ void __launch_bounds__(kThreads) paged_decode_kernel(const DecodeArgs a) {
    decode_body<KV, D, BS, TILE, NT, false>(a);
}

// bf16 (16-token tiles) fits 128 registers: four CTAs per SM; int8 (32-token tiles)
// three (decode_single_ctas_per_sm, which the partition plan counts).
template <typename KV, int D, int BS, int TILE>
__global__ void __launch_bounds__(kThreads, sizeof(KV) == 2 ? 4 : 3) paged_decode_single_kernel(const DecodeArgs a) {
    decode_body<KV, D, BS, TILE, 0, true>(a);
}

// Log-sum-exp merge of the partitions of each (sequence, query head):
// out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p, M = max_p m_p.
// One warp per (sequence, head): lane p holds partition p's (max, sum), 32 partitions
// at a time, so the maximum and the weights come from shuffles, and every
// partition's partial row is loaded independently of the others (no chain of
// dependent loads).  Launched as a programmatic dependent of the decode kernel: its
// launch overlaps the decode tail and it waits for the decode results here.
template <int D, int BS>
__global__ void __launch_bounds__(128) merge_partitions_kernel(const __grid_constant__ DecodeArgs a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the next kernel on the stream may launch now (it waits for this grid to finish
    // before it reads anything)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int PER = D / 32;  // output values per lane
    const int lane = threadIdx.x & 31;
    const int64_t pair = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);  // s * Hq + h
    if (pair >= (int64_t)a.S * a.Hq) return;
    const int s = (int)(pair / a.Hq);
    const int64_t row0 = pair * a.max_parts;
    if (a.max_parts <= kMergeInRegs) {
        // every partition's (max, sum) and this lane's slice of every partial row are
        // loaded at once, with the context length: one round trip; rows of partitions
        // past the context are loaded but never used (they may hold anything)
        const int ctx_raw = a.context_lens[s];
        float2 ml = make_float2(-INFINITY, 0.0f);
        if (lane < a.max_parts) ml = *reinterpret_cast<const float2 *>(a.ws_ml + (row0 + lane) * 2);
        float v[kMergeInRegs][PER];
#pragma unroll
        for (int q = 0; q < kMergeInRegs; ++q) {
            if (q < a.max_parts) {
                const float *src = a.ws_acc + (row0 + q) * D + lane * PER;
                if constexpr (PER == 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(src);
                    v[q][0] = x.x;
                    v[q][1] = x.y;
                    v[q][2] = x.z;
                    v[q][3] = x.w;
                } else {
                    const float2 x = *reinterpret_cast<const float2 *>(src);
                    v[q][0] = x.x;
                    v[q][1] = x.y;
                }
            }
        }
        const int lim = min(a.M * BS, a.max_context_len);
        const int ctx = ctx_raw < 0 ? 0 : min(ctx_raw, lim);
        const int nparts = (ctx + a.part_tokens - 1) / a.part_tokens;
        if (nparts <= 1) return;  // the decode kernel wrote the output itself
        const bool mine = lane < nparts;
        float mmax = mine ? ml.x : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
        const float mbase = mmax == -INFINITY ? 0.0f : mmax;
        const float f = mine ? fast_exp2(ml.x - mbase) : 0.0f;
        float lsum = mine ? f * ml.y : 0.0f;
        float acc[PER];
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] = 0.0f;
#pragma unroll
        for (int q = 0; q < kMergeInRegs; ++q) {
            const float fq = __shfl_sync(0xffffffffu, f, q);
            if (q < nparts) {
#pragma unroll
                for (int e = 0; e < PER; ++e) acc[e] += fq * v[q][e];
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
        const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
        uint16_t *dst = a.out + pair * D + lane * PER;
        if constexpr (PER == 4)
            *reinterpret_cast<uint2 *>(dst) =
                make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv));
        else
            *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        return;
    }
    const int ctx = checked_context(a, s, BS, false);
    const int nparts = (ctx + a.part_tokens - 1) / a.part_tokens;
    if (nparts <= 1) return;  // the decode kernel wrote the output itself
    float mmax = -INFINITY;
    for (int p = lane; p < nparts; p += 32) mmax = fmaxf(mmax, a.ws_ml[(row0 + p) * 2]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
    const float mbase = mmax == -INFINITY ? 0.0f : mmax;
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.0f;
    float lsum = 0.0f;
    for (int p0 = 0; p0 < nparts; p0 += 32) {
        float f = 0.0f;
        if (p0 + lane < nparts) {
            const float2 ml = *reinterpret_cast<const float2 *>(a.ws_ml + (row0 + p0 + lane) * 2);
            f = fast_exp2(ml.x - mbase);
            lsum += f * ml.y;
        }
        const int cnt = min(32, nparts - p0);
#pragma unroll 4
        for (int q = 0; q < cnt; ++q) {
            const float fq = __shfl_sync(0xffffffffu, f, q);
            const float *src = a.ws_acc + (row0 + p0 + q) * D + lane * PER;
            if constexpr (PER == 4) {
                const float4 v = *reinterpret_cast<const float4 *>(src);
                acc[0] += fq * v.x;
                acc[1] += fq * v.y;
                acc[2] += fq * v.z;
                acc[3] += fq * v.w;
            } else {
                const float2 v = *reinterpret_cast<const float2 *>(src);
                acc[0] += fq * v.x;
                acc[1] += fq * v.y;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
    uint16_t *dst = a.out + pair * D + lane * PER;
    if constexpr (PER == 4)
        *reinterpret_cast<uint2 *>(dst) =
            make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv));
    else
        *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
}

template <typename KV, int D, int BS, int TILE>
cudaError_t launch_typed(const DecodeArgs &a, cudaStream_t stream) {
    // a programmatic dependent of the kernel before it on the stream (an append, the
    // previous layer's merge): it launches while that kernel drains and waits for it
    // before reading
    dim3 grid(a.max_parts, a.Hkv * a.head_chunks, a.S);
    // The plan's choice (DecodePlan::single): split contexts of bf16 and int8 caches on
    // the single-buffered kernel at four (bf16) or three CTAs per SM; unsplit contexts, fp8 caches and
    // the own tokens of a shared-prefix call on the double-buffered one at two.
    // Measured on GB300 (decode call, us, double -> single, same partitions): 70B-shaped
    // bf16 114.1 -> 111.8, int8 522.2 -> 513.7; fp8 513.0 -> 527.2, 13B-shaped bf16 (no
    // split) 215.8 -> 220.4, shared-prompt call 42.2 -> 43.5.
    constexpr bool kSingleOk = !std::is_same<KV, e4m3_t>::value;
    cudaError_t err;
    if constexpr (kSingleOk) {
        if (a.single && !a.start_tokens)
            err = launch_dependent(paged_decode_single_kernel<KV, D, BS, TILE>, grid, dim3(kThreads), 0, stream, a);
        else
            err = launch_dependent(paged_decode_kernel<KV, D, BS, TILE, 0>, grid, dim3(kThreads), 0, stream, a);
    } else {
        err = launch_dependent(paged_decode_kernel<KV, D, BS, TILE, 0>, grid, dim3(kThreads), 0, stream, a);
    }
    if (err != cudaSuccess || a.max_parts == 1 || a.partials_only) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(((int64_t)a.S * a.Hq + 3) / 4));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_partitions_kernel<D, BS>, a);
}

template <typename KV, int D>
cudaError_t launch_bs(const DecodeArgs &a, int bs, cudaStream_t stream) {
    constexpr bool ONE_BYTE = sizeof(KV) == 1;  // int8 and fp8: a tile is a whole 32-token block
    if (bs == 16) return launch_typed<KV, D, 16, 16>(a, stream);
    return launch_typed<KV, D, 32, ONE_BYTE ? 32 : 16>(a, stream);
}

// Rows mode: NT new tokens per CTA, the token groups of one partition consecutive CTAs
// (they read the same K/V tiles, so all but the first hit L2).  Several tokens per CTA
// use 16-token tiles (registers for their column sets).
template <typename KV, int D, int NT>
cudaError_t launch_rows_nt(const DecodeArgs &a, int bs, cudaStream_t stream) {
    constexpr int T32 = (sizeof(KV) == 1 && NT == 1) ? 32 : 16;
    const dim3 grid((unsigned)(a.max_parts * ((a.Lq + NT - 1) / NT)), a.Hkv * a.head_chunks, a.S);
    if (bs == 16)
        return launch_dependent(paged_decode_kernel<KV, D, 16, 16, NT>, grid, dim3(kThreads), 0, stream, a);
    return launch_dependent(paged_decode_kernel<KV, D, 32, T32, NT>, grid, dim3(kThreads), 0, stream, a);
}

template <typename KV, int D>
cudaError_t launch_rows_bs(const DecodeArgs &a, int bs, cudaStream_t stream) {
    if (a.rows_per_cta == 2) return launch_rows_nt<KV, D, 2>(a, bs, stream);
    return launch_rows_nt<KV, D, 1>(a, bs, stream);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, int D, int bs, int kv_dtype, cudaStream_t stream) {
    static_assert(kMaxPartBlocks * 16 >= 4096, "partition block list fits in shared memory");
    if (kv_dtype == PA_KV_BF16)
        return D == 128 ? launch_bs<uint16_t, 128>(a, bs, stream) : launch_bs<uint16_t, 64>(a, bs, stream);
    if (kv_dtype == PA_KV_FP8)
        return D == 128 ? launch_bs<e4m3_t, 128>(a, bs, stream) : launch_bs<e4m3_t, 64>(a, bs, stream);
    return D == 128 ? launch_bs<int8_t, 128>(a, bs, stream) : launch_bs<int8_t, 64>(a, bs, stream);
}

int decode_rows_per_cta(int max_query_len) { return max_query_len >= 2 ? 2 : 1; }

int decode_single_ctas_per_sm(int kv_dtype) { return kv_dtype == PA_KV_BF16 ? 4 : 3; }

cudaError_t launch_decode_rows(const DecodeArgs &a, int D, int bs, int kv_dtype, cudaStream_t stream) {
    if (!a.query_start || a.Lq <= 0 || a.start_tokens || a.partials_only || kv_dtype == PA_KV_BF16 ||
        (a.rows_per_cta != 1 && a.rows_per_cta != 2))
        return cudaErrorInvalidValue;
    if (kv_dtype == PA_KV_FP8)
        return D == 128 ? launch_rows_bs<e4m3_t, 128>(a, bs, stream) : launch_rows_bs<e4m3_t, 64>(a, bs, stream);
    return D == 128 ? launch_rows_bs<int8_t, 128>(a, bs, stream) : launch_rows_bs<int8_t, 64>(a, bs, stream);
}

}  // namespace pa
