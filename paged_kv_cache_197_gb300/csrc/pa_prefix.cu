// Prefix-aware paged decode: a prefix shared by a group of sequences (the same
// physical blocks at the head of every member's block table) is read once per kv
// head for the whole group instead of once per sequence.
//
// The pages: requests sharing a system prompt or a document point at the same
// physical pages and store them once (ia-vox-magazine, "PagedAttention : la
// revolution de l'allocation memoire"; gotburnout.io "PagedAttention & Gestion du
// KV-Cache", section 3.01); branches of one request share their context (section
// 3.02).  The result is the same paged attention as pa_decode: for every member,
// softmax over all its tokens, prefix and own.
//
// Four launches (the second on a side stream of the library's, overlapping the third):
//   1. setup (a warp per sequence): its group and the number of prefix tokens to
//      skip; a member whose table does not repeat the group's prefix blocks, or whose
//      context is shorter than the prefix, is flagged and decoded on its own;
//   2. grouped prefix kernel: CTA = (128-token chunk of the prefix, kv head, block of
//      128 query columns, group).  The chunk's K and V rows are staged once in shared
//      memory (cp.async, rows padded so ldmatrix hits 32 banks) and each of 8 warps
//      multiplies them against 16 query columns -- (member, query head) pairs of
//      the group -- on the tensor cores, leaving one partial (max, sum, output) per
//      column and chunk;
//   3. the ordinary decode kernel over each sequence's own tokens (start offset =
//      its prefix), writing partials;
//   4. a merge per (sequence, head) of the prefix partials and the own-token
//      partials by log-sum-exp.
#include <cuda_bf16.h>
#include <math.h>

#include <atomic>
#include <map>
#include <mutex>
#include <type_traits>
#include <utility>

#include "pa_internal.cuh"
#include "pa_mma.cuh"

namespace pa {
namespace {

using namespace tiled;

constexpr int kPrefixChunk = 128;   // prefix tokens per CTA of the grouped kernel
constexpr int kPrefixChunkTc = 256;  // prefix tokens per CTA on the tcgen05 path
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kColsPerWarp = 16;    // two mma n-tiles of 8 query columns
constexpr int kColsPerCta = kWarps * kColsPerWarp;

__device__ __forceinline__ void raise_flag(int *err_flag, int bit) {
    if (err_flag) atomicOr(err_flag, bit);
}

__device__ __forceinline__ int checked_ctx(const DecodeArgs &a, int s, int bs) {
    const int ctx = a.context_lens[s];
    const int lim = min(a.M * bs, a.max_context_len);
    return ctx < 0 ? 0 : (ctx > lim ? lim : ctx);
}

// ------------------------------------------------------------------ 1. setup
// The group of sequence s: the last g < n_groups with group_start[g] <= s, if
// s < group_start[g + 1] (with non-decreasing offsets, the one group holding s), else -1.
__device__ __forceinline__ int find_group(const PrefixArgs &p, int s) {
    int lo = 0, hi = p.n_groups;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (p.group_start[mid] <= s) lo = mid + 1;
        else hi = mid;
    }
    const int g = lo - 1;
    return (g >= 0 && s < p.group_start[g + 1]) ? g : -1;
}

constexpr int kSetupOffsets = 128;  // group offsets a warp holds in registers (4 per lane)
constexpr int kSetupEntries = 128;  // table entries a warp compares per pass (4 per lane)

// The same search over offsets held by the warp: lane l has off[k] = group_start[l + 32k].
__device__ __forceinline__ int find_group_warp(const int (&off)[4], int n_groups, int s, int lane) {
    int g = -1;
#pragma unroll
    for (int k = 3; k >= 0; --k) {
        const unsigned m = __ballot_sync(0xffffffffu, lane + 32 * k < n_groups && off[k] <= s);
        if (g < 0 && m) g = 32 * k + 31 - __clz(m);
    }
    if (g < 0) return -1;
    const int k1 = (g + 1) >> 5;
    const int mine = k1 == 0 ? off[0] : k1 == 1 ? off[1] : k1 == 2 ? off[2] : off[3];
    const int next = __shfl_sync(0xffffffffu, mine, (g + 1) & 31);
    return s < next ? g : -1;
}

// One warp per sequence: seq_group[s] = its group (or -1), seq_start[s] = the group's
// prefix tokens (or 0).  A member joins its group only if the group is well formed,
// the group's first member lands in the same group and holds the prefix, and its
// table repeats the first member's prefix blocks, all of them inside the pool; a
// member joined to g thus implies that the first member is joined to g too.  With up
// to 127 groups and 128 prefix blocks the warp needs two batches of dependent loads.
__global__ void __launch_bounds__(256) prefix_setup_kernel(const __grid_constant__ DecodeArgs a,
                                                           const __grid_constant__ PrefixArgs p, int bs) {
    const int lane = threadIdx.x & 31;
    const int s = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (s >= a.S) return;
    const int32_t *row = a.block_tables + (int64_t)s * a.M;
    // first batch of loads: the group offsets, this sequence's length and first table entries
    int off[4], mine[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = lane + 32 * k;
        off[k] = (p.n_groups < kSetupOffsets && i <= p.n_groups) ? p.group_start[i] : 0;
        mine[k] = i < a.M ? row[i] : -1;
    }
    const int ctx_s = checked_ctx(a, s, bs);
    const bool small = p.n_groups < kSetupOffsets;
    const int g = small ? find_group_warp(off, p.n_groups, s, lane) : find_group(p, s);
    int grp = -1, start = 0;
    if (g >= 0) {
        int lo, hi;
        if (small) {
            const int k0 = g >> 5, k1 = (g + 1) >> 5;
            lo = __shfl_sync(0xffffffffu, k0 == 0 ? off[0] : k0 == 1 ? off[1] : k0 == 2 ? off[2] : off[3], g & 31);
            hi = __shfl_sync(0xffffffffu, k1 == 0 ? off[0] : k1 == 1 ? off[1] : k1 == 2 ? off[2] : off[3], (g + 1) & 31);
        } else {
            lo = p.group_start[g];
            hi = p.group_start[g + 1];
        }
        const bool lo_ok = lo >= 0 && lo < hi && hi <= a.S;
        // second batch of loads: the prefix length, the first member's length and table entries
        const int plen = p.group_prefix[g];
        const int32_t *lead = a.block_tables + (int64_t)(lo_ok ? lo : s) * a.M;
        int theirs[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) theirs[k] = lane + 32 * k < a.M ? lead[lane + 32 * k] : -1;
        const int ctx_lo = lo_ok ? checked_ctx(a, lo, bs) : 0;
        const int glead = lo_ok ? (small ? find_group_warp(off, p.n_groups, lo, lane) : find_group(p, lo)) : -1;
        bool ok = lo_ok && plen > 0 && plen % bs == 0 && plen <= p.max_prefix &&
                  hi - lo <= p.max_group_size && ctx_lo >= plen && ctx_s >= plen && glead == g;
        if (ok) {
            const int nb = plen / bs;
            bool same = true;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (lane + 32 * k < nb) same = same && mine[k] == theirs[k] && theirs[k] >= 0 && theirs[k] < a.N;
            for (int j = kSetupEntries + lane; j < nb; j += 32) {  // longer prefixes
                const int b = lead[j];
                same = same && row[j] == b && b >= 0 && b < a.N;
            }
            ok = __all_sync(0xffffffffu, same);
        }
        if (ok) {
            grp = g;
            start = plen;
        } else if (lane == 0) {
            raise_flag(a.err_flag, PA_FLAG_PREFIX_MISMATCH);  // decoded on its own
        }
    }
    if (lane == 0) {
        p.seq_group[s] = grp;
        p.seq_start[s] = start;
    }
}

// ---------------------------------------------------- 2. grouped prefix kernel
template <typename KV, int D, int BS>
__global__ void __launch_bounds__(kThreads) grouped_prefix_kernel(const __grid_constant__ DecodeArgs a,
                                                                  const __grid_constant__ PrefixArgs p) {
    // 8-bit caches: rows staged as fp16 code x scale, q as fp16 scaled by a power of two
    // per column, fp16 products
    constexpr bool QUANT = sizeof(KV) == 1;
    constexpr int ROW = D * 2;        // bytes of one staged token row (bf16 or fp16)
    constexpr int RS = ROW + 16;      // padded shared-memory row stride
    constexpr int KC = D / 16;        // k-steps of the score product
    constexpr int MT = D / 16;        // d tiles of the output product
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ks = smem;                        // [kPrefixChunk][RS]
    unsigned char *vs = smem + kPrefixChunk * RS;    // [kPrefixChunk][RS]
    __shared__ int s_blk[kPrefixChunk / 16];

    const int chunk = blockIdx.x;
    const int g = blockIdx.z;
    const int cb = blockIdx.y % p.CB, kvh = blockIdx.y / p.CB;
    const int lo = p.group_start[g], hi = p.group_start[g + 1];
    const int plen = p.group_prefix[g];
    // a group whose first member did not join it has no member at all
    if (lo < 0 || hi > a.S || lo >= hi || p.seq_group[lo] != g) return;
    const int tok0 = chunk * kPrefixChunk;
    if (tok0 >= plen) return;
    const int ntok = min(kPrefixChunk, plen - tok0);
    const int ncols = (hi - lo) * a.G;
    const int col0 = cb * kColsPerCta;
    if (col0 >= ncols) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, t = lane & 3;

    // the chunk's blocks, from the first member's table (every member repeats them)
    if (tid < (ntok + BS - 1) / BS) s_blk[tid] = a.block_tables[(int64_t)lo * a.M + tok0 / BS + tid];
    __syncthreads();
    // stage the chunk's K and V rows; rows past the prefix are zero-filled
    if constexpr (!QUANT) {
        constexpr int CPR = ROW / 16;  // 16-byte chunks per row
        for (int i = tid; i < 2 * kPrefixChunk * CPR; i += kThreads) {
            const int isv = i >= kPrefixChunk * CPR;
            const int rem = isv ? i - kPrefixChunk * CPR : i;
            const int r = rem / CPR, c = rem % CPR;
            const void *src = a.k_cache;
            uint32_t bytes = 0;
            if (r < ntok) {
                const int blk = s_blk[r / BS];
                const int64_t row = ((int64_t)blk * a.Hkv + kvh) * BS + (tok0 + r) % BS;
                src = static_cast<const char *>(isv ? a.v_cache : a.k_cache) + row * ROW + c * 16;
                bytes = 16;
            }
            cp_async16(smem_u32((isv ? vs : ks) + r * RS + c * 16), src, bytes);
        }
        cp_async_wait_all();
    } else {
        // sixteen codes and the row's scale per piece, all loads issued before the
        // conversions
        constexpr int QPR = D / 16;                        // 16-code pieces per row
        constexpr int NPT = kPrefixChunk * QPR / kThreads;  // pieces per thread
        uint4 kr[NPT], vr[NPT];
        float ksr[NPT], vsr[NPT];
#pragma unroll
        for (int k = 0; k < NPT; ++k) {
            const int i = tid + k * kThreads, r = i / QPR, qc = i % QPR;
            kr[k] = vr[k] = make_uint4(0u, 0u, 0u, 0u);
            ksr[k] = vsr[k] = 0.f;
            if (r < ntok) {
                const int blk = s_blk[r / BS];
                const int64_t row = ((int64_t)blk * a.Hkv + kvh) * BS + (tok0 + r) % BS;
                kr[k] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const char *>(a.k_cache) + row * D) + qc);
                vr[k] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const char *>(a.v_cache) + row * D) + qc);
                ksr[k] = __ldg(a.k_scale + row);
                vsr[k] = __ldg(a.v_scale + row);
            }
        }
        bool over = false;  // a row whose code x scale leaves fp16's range
#pragma unroll
        for (int k = 0; k < NPT; ++k) over |= fmaxf(ksr[k], vsr[k]) > max_f16_scale<KV>();
        if (over) raise_flag(a.err_flag, PA_FLAG_FP16_RANGE);
#pragma unroll
        for (int k = 0; k < NPT; ++k) {
            const int i = tid + k * kThreads, r = i / QPR, qc = i % QPR;
            uint4 lo, hi;
            codes_to_f16<KV>(kr[k], ksr[k], lo, hi);
            reinterpret_cast<uint4 *>(ks + r * RS + qc * 32)[0] = lo;
            reinterpret_cast<uint4 *>(ks + r * RS + qc * 32)[1] = hi;
            codes_to_f16<KV>(vr[k], vsr[k], lo, hi);
            reinterpret_cast<uint4 *>(vs + r * RS + qc * 32)[0] = lo;
            reinterpret_cast<uint4 *>(vs + r * RS + qc * 32)[1] = hi;
        }
    }
    __syncthreads();

    // this warp's 16 query columns (member, head) -> B fragments of q
    uint32_t qf[2][KC][2];
    float csc[2][2];  // score scale of this lane's score columns 2t, 2t + 1 per n-tile
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int c = col0 + warp * kColsPerWarp + nt * 8 + gq;
        if (c < ncols && p.seq_group[lo + c / a.G] == g) {
            const int s = lo + c / a.G, h = kvh * a.G + c % a.G;
            const uint16_t *qrow = a.q + ((int64_t)s * a.Hq + h) * D;
#pragma unroll
            for (int kc = 0; kc < KC; ++kc) {
                qf[nt][kc][0] = __ldg(reinterpret_cast<const uint32_t *>(qrow + kc * 16 + 2 * t));
                qf[nt][kc][1] = __ldg(reinterpret_cast<const uint32_t *>(qrow + kc * 16 + 8 + 2 * t));
            }
        } else {
#pragma unroll
            for (int kc = 0; kc < KC; ++kc) qf[nt][kc][0] = qf[nt][kc][1] = 0u;
        }
        float colscale = a.scale_log2;  // of column nt * 8 + gq
        if constexpr (QUANT) {
            // fp16 q scaled by 2^sig, sig putting the column's largest |q| (spread over
            // the 4 lanes of the quad) in [2^13, 2^14)
            float amax = 0.f;
#pragma unroll
            for (int kc = 0; kc < KC; ++kc)
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    amax = fmaxf(amax, fabsf(__uint_as_float(qf[nt][kc][w] << 16)));
                    amax = fmaxf(amax, fabsf(__uint_as_float(qf[nt][kc][w] & 0xffff0000u)));
                }
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const int sig = amax > 0.f ? min(100, max(-100, 14 - exponent_above(amax))) : 0;
            const float up = ldexpf(1.f, sig);
#pragma unroll
            for (int kc = 0; kc < KC; ++kc)
#pragma unroll
                for (int w = 0; w < 2; ++w)
                    qf[nt][kc][w] = f16x2(__uint_as_float(qf[nt][kc][w] << 16) * up,
                                          __uint_as_float(qf[nt][kc][w] & 0xffff0000u) * up);
            colscale = a.scale_log2 * ldexpf(1.f, -sig);
        }
        // score column 2t + j is held (as column gq) by lanes 4 (2t + j) .. + 3
        csc[nt][0] = __shfl_sync(0xffffffffu, colscale, 8 * t);
        csc[nt][1] = __shfl_sync(0xffffffffu, colscale, 8 * t + 4);
    }
    if (col0 + warp * kColsPerWarp >= ncols) return;  // nothing for this warp (no more barriers)

    float o[2][MT][4];
    float m[2][2], l[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
        m[nt][0] = m[nt][1] = -INFINITY;
        l[nt][0] = l[nt][1] = 0.f;
    }
    const uint32_t kbase = smem_u32(ks), vbase = smem_u32(vs);
    for (int tile = 0; tile * 16 < ntok; ++tile) {
        const int nvalid = min(16, ntok - tile * 16);
        // scores S[token][column] for both n-tiles
        float sc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
        {
            const int row = tile * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const uint32_t rb = kbase + row * RS + (lane >> 4) * 16;
#pragma unroll
            for (int kc = 0; kc < KC; ++kc) {
                uint32_t af[4];
                ldsm_x4(af, rb + kc * 32);
                if constexpr (QUANT) {
                    mma16816_f16(sc[0], af, qf[0][kc][0], qf[0][kc][1]);
                    mma16816_f16(sc[1], af, qf[1][kc][0], qf[1][kc][1]);
                } else {
                    mma16816(sc[0], af, qf[0][kc][0], qf[0][kc][1]);
                    mma16816(sc[1], af, qf[1][kc][0], qf[1][kc][1]);
                }
            }
        }
        uint32_t pb[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            float x[4], mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int tok = gq + 8 * (c >> 1);
                x[c] = tok < nvalid ? sc[nt][c] * csc[nt][c & 1] : -INFINITY;
                mx[c & 1] = fmaxf(mx[c & 1], x[c]);
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 4));
                mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 8));
                mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 16));
            }
            float base[2], alpha[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float mnew = fmaxf(m[nt][j], mx[j]);
                base[j] = mnew == -INFINITY ? 0.f : mnew;
                alpha[j] = ex2(m[nt][j] - base[j]);
                m[nt][j] = mnew;
                l[nt][j] *= alpha[j];
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                o[nt][mt][0] *= alpha[0];
                o[nt][mt][1] *= alpha[1];
                o[nt][mt][2] *= alpha[0];
                o[nt][mt][3] *= alpha[1];
            }
            float pr[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                pr[c] = ex2(x[c] - base[c & 1]);
                l[nt][c & 1] += pr[c];
            }
            if constexpr (QUANT) {
                pb[nt][0] = movmatrix_t(f16x2(pr[0], pr[1]));
                pb[nt][1] = movmatrix_t(f16x2(pr[2], pr[3]));
            } else {
                pb[nt][0] = movmatrix_t(bf16x2(pr[0], pr[1]));
                pb[nt][1] = movmatrix_t(bf16x2(pr[2], pr[3]));
            }
        }
        // O^T += V^T P^T; the V fragments serve both n-tiles (rows past the prefix are 0)
        {
            const int row = tile * 16 + (lane & 7) + (lane >> 4) * 8;
            const uint32_t rb = vbase + row * RS + ((lane >> 3) & 1) * 16;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t af[4];
                ldsm_x4_trans(af, rb + mt * 32);
                if constexpr (QUANT) {
                    mma16816_f16(o[0][mt], af, pb[0][0], pb[0][1]);
                    mma16816_f16(o[1][mt], af, pb[1][0], pb[1][1]);
                } else {
                    mma16816(o[0][mt], af, pb[0][0], pb[0][1]);
                    mma16816(o[1][mt], af, pb[1][0], pb[1][1]);
                }
            }
        }
    }
    // partials of this chunk: (max, sum) and unnormalised output per column
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            l[nt][j] += __shfl_xor_sync(0xffffffffu, l[nt][j], 4);
            l[nt][j] += __shfl_xor_sync(0xffffffffu, l[nt][j], 8);
            l[nt][j] += __shfl_xor_sync(0xffffffffu, l[nt][j], 16);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int c = col0 + warp * kColsPerWarp + nt * 8 + 2 * t + j;
            if (c >= ncols) continue;
            const int s = lo + c / a.G, h = kvh * a.G + c % a.G;
            if (p.seq_group[s] != g) continue;  // decoded on its own (or by another group)
            const int64_t row = ((int64_t)s * a.Hq + h) * p.PP + chunk;
            float *dst = p.pacc + row * D;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                dst[mt * 16 + gq] = o[nt][mt][j];
                dst[mt * 16 + gq + 8] = o[nt][mt][2 + j];
            }
            if (gq == 0) *reinterpret_cast<float2 *>(p.pml + row * 2) = make_float2(m[nt][j], l[nt][j]);
        }
    }
}

// ------------------------------------------------------------------ 4. merge
// One warp per (sequence, head): the prefix chunks of its group (if any) and the
// partitions of its own tokens, joined by log-sum-exp:
// out = sum_i 2^(m_i - M) acc_i / sum_i 2^(m_i - M) l_i, M = max_i m_i.
template <int PER>
struct Vec;
template <>
struct Vec<4> {
    static __device__ __forceinline__ void load(float (&v)[4], const float *p) {
        const float4 x = __ldg(reinterpret_cast<const float4 *>(p));
        v[0] = x.x, v[1] = x.y, v[2] = x.z, v[3] = x.w;
    }
};
template <>
struct Vec<2> {
    static __device__ __forceinline__ void load(float (&v)[2], const float *p) {
        const float2 x = __ldg(reinterpret_cast<const float2 *>(p));
        v[0] = x.x, v[1] = x.y;
    }
};

template <int D, int BS>
__global__ void __launch_bounds__(128) merge_prefix_kernel(const __grid_constant__ DecodeArgs a,
                                                           const __grid_constant__ PrefixArgs p) {
    constexpr int PER = D / 32;
    const int lane = threadIdx.x & 31;
    const int64_t pair = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (pair >= (int64_t)a.S * a.Hq) return;
    const int s = (int)(pair / a.Hq);
    const int ctx = checked_ctx(a, s, BS);
    const int start = min(p.seq_start[s], ctx);
    const int nown = max(1, (ctx - start + a.part_tokens - 1) / a.part_tokens);
    const int npre = p.seq_group[s] >= 0 ? (start + p.chunk - 1) / p.chunk : 0;
    const int64_t own0 = pair * a.max_parts, pre0 = pair * p.PP;
    const int n = npre + nown;
    auto row_of = [&](int i, const float *&acc, const float *&ml) {
        if (i < npre) {
            acc = p.pacc + (pre0 + i) * D;
            ml = p.pml + (pre0 + i) * 2;
        } else {
            acc = a.ws_acc + (own0 + i - npre) * D;
            ml = a.ws_ml + (own0 + i - npre) * 2;
        }
    };
    // lane i holds partial i's (max, sum), 32 partials at a time; the first rows are
    // requested together with them
    constexpr int INFL = 8;  // partial rows in flight per lane
    float v[INFL][PER];
    auto fetch = [&](int base) {
#pragma unroll
        for (int u = 0; u < INFL; ++u) {
            if (base + u < n) {
                const float *r, *ml;
                row_of(base + u, r, ml);
                Vec<PER>::load(v[u], r + lane * PER);
            }
        }
    };
    fetch(0);
    float mmax = -INFINITY;
    for (int i = lane; i < n; i += 32) {
        const float *acc, *ml;
        row_of(i, acc, ml);
        mmax = fmaxf(mmax, __ldg(ml));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
    const float mbase = mmax == -INFINITY ? 0.0f : mmax;
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    float lsum = 0.f;
    float f = 0.f;
    for (int base = 0; base < n; base += INFL) {
        if ((base & 31) == 0) {  // weights of the next 32 partials
            f = 0.f;
            if (base + lane < n) {
                const float *r, *ml;
                row_of(base + lane, r, ml);
                const float2 w = __ldg(reinterpret_cast<const float2 *>(ml));
                f = ex2(w.x - mbase);
                lsum += f * w.y;
            }
        }
#pragma unroll
        for (int u = 0; u < INFL; ++u) {
            const float fq = __shfl_sync(0xffffffffu, f, (base + u) & 31);
            if (base + u < n) {
#pragma unroll
                for (int e = 0; e < PER; ++e) acc[e] += fq * v[u][e];
            }
        }
        if (base + INFL < n) fetch(base + INFL);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    uint16_t *dst = a.out + pair * D + lane * PER;
    if constexpr (PER == 4)
        *reinterpret_cast<uint2 *>(dst) = make_uint2(bf16x2(acc[0] * inv, acc[1] * inv), bf16x2(acc[2] * inv, acc[3] * inv));
    else
        *reinterpret_cast<uint32_t *>(dst) = bf16x2(acc[0] * inv, acc[1] * inv);
}

// The grouped prefix kernel does not depend on the own-token decode, so it runs on a
// second stream of the library's, forked from and joined back to the caller's stream
// with events (both captured as graph edges when the caller's stream is capturing).
// Each (device, caller stream) pair gets its own side stream and events, created on
// first use and kept until the process exits, so unrelated callers on different
// streams never wait for each other.  Calls on one caller stream are ordered by that
// stream; enqueueing on the same caller stream from several host threads at once is
// not supported (as for any stream-ordered work).
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

cudaError_t side_stream(int dev, cudaStream_t caller, SideStream *&out) {
    static std::mutex mu;  // guards the map only
    static std::map<std::pair<int, cudaStream_t>, SideStream> sides;
    std::lock_guard<std::mutex> lock(mu);
    SideStream &ss = sides[{dev, caller}];
    if (!ss.stream) {
        cudaError_t e = cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            sides.erase({dev, caller});
            return e;
        }
    }
    out = &ss;  // std::map nodes never move
    return cudaSuccess;
}

// bf16 caches with head_dim 128: each group's prefix on the tcgen05 kernel in group mode
// (the members' (query head) columns as its rows, 128-token partitions as its chunks),
// leaving the same partials as the grouped kernel.
template <int BS>
cudaError_t launch_prefix_tc(const DecodeArgs &a, const PrefixArgs &p, cudaStream_t stream) {
    // p.CB counts blocks of kColsPerCta columns; the tcgen05 kernel takes as many per CTA
    if (multi_tc_rows() != kColsPerCta) return cudaErrorInvalidValue;
    MultiArgs m{};
    m.out = a.out;
    m.q = a.q;
    m.k_cache = a.k_cache;
    m.v_cache = a.v_cache;
    m.block_tables = a.block_tables;
    m.context_lens = a.context_lens;
    m.query_start = p.group_start;
    m.ws_acc = p.pacc;
    m.ws_ml = p.pml;
    m.err_flag = a.err_flag;
    m.M = a.M;
    m.S = p.n_groups;
    m.T = a.S;
    m.Hq = a.Hq;
    m.Hkv = a.Hkv;
    m.G = a.G;
    m.N = a.N;
    m.g_shift = (a.G & (a.G - 1)) == 0 ? __builtin_ctz((unsigned)a.G) : -1;
    m.CB = p.CB;
    m.part_tokens = p.chunk;
    m.max_parts = p.PP;
    m.max_context_len = p.max_prefix;
    m.max_query_len = p.max_group_size;
    m.scale_log2 = a.scale_log2;
    m.group_prefix = p.group_prefix;
    m.seq_group = p.seq_group;
    return launch_multi_tc_groups(m, BS, stream);
}

template <typename KV, int D, int BS>
cudaError_t launch_prefix_typed(const DecodeArgs &a, const PrefixArgs &p, int kv_dtype, cudaStream_t stream) {
    constexpr int SMEM = 2 * kPrefixChunk * (D * 2 + 16);
    static std::atomic<bool> configured[64];  // per device: the shared-memory attribute is set
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(grouped_prefix_kernel<KV, D, BS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        configured[dev].store(true, std::memory_order_release);
    }
    SideStream *ss = nullptr;
    cudaError_t err = side_stream(dev, stream, ss);
    if (err != cudaSuccess) return err;
    prefix_setup_kernel<<<(unsigned)((a.S + 7) / 8), 256, 0, stream>>>(a, p, BS);
    const bool grouped = p.n_groups > 0 && p.PP > 0;
    if (grouped) {
        if ((err = cudaEventRecord(ss->fork, stream)) != cudaSuccess) return err;
        if ((err = cudaStreamWaitEvent(ss->stream, ss->fork, 0)) != cudaSuccess) return err;
        if constexpr (std::is_same<KV, uint16_t>::value && D == 128) {
            err = launch_prefix_tc<BS>(a, p, ss->stream);
        } else if (p.chunk != kPrefixChunk) {
            err = cudaErrorInvalidValue;
        } else {
            dim3 grid(p.PP, a.Hkv * p.CB, p.n_groups);
            grouped_prefix_kernel<KV, D, BS><<<grid, kThreads, SMEM, ss->stream>>>(a, p);
            err = cudaGetLastError();
        }
        const cudaError_t e = cudaEventRecord(ss->join, ss->stream);  // recorded even on error
        if (err == cudaSuccess) err = e;
        if (err != cudaSuccess) return err;
    }
    err = launch_decode(a, D, BS, kv_dtype, stream);  // own tokens, partials only
    if (grouped) {
        const cudaError_t e = cudaStreamWaitEvent(stream, ss->join, 0);  // join even on error
        if (err == cudaSuccess) err = e;
    }
    if (err != cudaSuccess) return err;
    merge_prefix_kernel<D, BS><<<(unsigned)(((int64_t)a.S * a.Hq + 3) / 4), 128, 0, stream>>>(a, p);
    return cudaGetLastError();
}

}  // namespace

int prefix_chunk_tokens(int kv_dtype, int D) {
    // the tcgen05 path's CTA pays a longer prologue (tensor memory, barriers, Q staged in
    // tensor memory) than the grouped kernel's: measured on the shared-prompt workload,
    // 256-token partials 42.5 us per call against 44.2 with 128 and 44.7 with 512
    return kv_dtype == PA_KV_BF16 && D == 128 ? kPrefixChunkTc : kPrefixChunk;
}
int prefix_cols_per_cta() { return kColsPerCta; }

template <typename KV>
cudaError_t launch_prefix_kv(const DecodeArgs &a, const PrefixArgs &p, int D, int bs, int kv_dtype,
                             cudaStream_t stream) {
    if (D == 128)
        return bs == 16 ? launch_prefix_typed<KV, 128, 16>(a, p, kv_dtype, stream)
                        : launch_prefix_typed<KV, 128, 32>(a, p, kv_dtype, stream);
    return bs == 16 ? launch_prefix_typed<KV, 64, 16>(a, p, kv_dtype, stream)
                    : launch_prefix_typed<KV, 64, 32>(a, p, kv_dtype, stream);
}

cudaError_t launch_decode_shared_prefix(const DecodeArgs &a, const PrefixArgs &p, int D, int bs, int kv_dtype,
                                        cudaStream_t stream) {
    if (kv_dtype == PA_KV_INT8) return launch_prefix_kv<int8_t>(a, p, D, bs, kv_dtype, stream);
    if (kv_dtype == PA_KV_FP8) return launch_prefix_kv<e4m3_tag>(a, p, D, bs, kv_dtype, stream);
    return launch_prefix_kv<uint16_t>(a, p, D, bs, kv_dtype, stream);
}

}  // namespace pa
