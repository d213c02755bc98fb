// Multi-token paged attention on the fifth-generation tensor cores (tcgen05) with
// head_dim 128, when a kv head of a sequence has at least 16 (new token, query head)
// columns: prefill chunks and draft verification on bf16 caches, prefill chunks on
// 8-bit ones.
//
// What is computed is the same as the mma.sync kernel in pa_multi.cu (deeplearn.tn,
// "Les leviers d'optimisation en production": a chunk of new tokens attends the
// paged cache, each token up to its own position).  One CTA takes 128 columns of one
// (sequence, kv head, context partition) and streams the partition in 64-token
// tiles; two CTAs share an SM (113 KB of shared memory and 256 tensor-memory columns
// each), so one's softmax overlaps the other's products.  Its seven warps have fixed
// roles, coupled only through mbarriers:
//   * warp 4 copies K tiles, warp 5 V tiles, into three stages each by TMA: per cache
//     block, two boxes of 64 dims x block-size rows with the 128-byte swizzle, so a
//     staged tile is the K-major layout the tensor core reads (the block ids come
//     from the table, one lane per block; entries outside the pool and blocks past
//     the partition are copied from past the end of the pool, i.e. as zeros);
//   * warp 6 issues, from one lane, S_t = Q K_t^T (M 128 columns x N 64 tokens,
//     K 128 dims; Q from tensor memory, where the row threads put it, K from the
//     staged tile) and commits it to the barriers that free the K stage and wake the
//     row warps; row thread 0 issues O += P_t V_t (N 128 dims, K 64 tokens; P from
//     shared memory, V read as an MN-major operand from the same staged tile) as soon
//     as every row's P is in (no hand-off through warp 6, whose next S may be waiting
//     for its K tile) and commits it to the barriers that free the V stage and P;
//   * warps 0-3 own one row each (tensor-memory lane = thread): they read the row's
//     scores, mask tokens past its position, keep a running max (raised only when a
//     tile's max exceeds it by more than 2^8 in the exp2 domain; O is then rescaled in
//     tensor memory) and sum, write P in bf16 to shared memory in the swizzled K-major
//     layout, and finally write the output row or its (max, sum, output) partial for
//     the merge kernel shared with the mma.sync path; a warp whose 32 rows are all
//     padding (narrow chunks) only keeps step with the barriers.
// Tensor memory: S in columns 0-63, Q (bf16 pairs) 64-127, O 128-255.
// Every wait is bounded (PA_FLAG_TIMEOUT when one gives up; the outputs are then not
// written).
// 8-bit caches take this kernel for prefill-shaped chunks (64 columns and more) after a
// pass that dequantises the blocks each sequence attends, once, into a bf16 pool in
// the workspace (dequant_blocks_kernel below): converting inside this kernel would
// repeat the work in every column block of a kv head.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <atomic>
#include <type_traits>

#include "pa_internal.cuh"
#include "pa_stages.h"

namespace pa {
namespace {

// Narrower chunks (decode-like steps) stay on the mma.sync kernel; from 16 (token, head)
// columns per kv head up the staged K/V serve enough rows to pay for the idle ones.
constexpr int kTcMinCols = 16;
constexpr int kTcRows = 128;  // columns per CTA: the M of both products
constexpr int kTcTile = 64;  // cached tokens per tile: N of S, K of P V
constexpr int kTcD = 128;
constexpr int kTcTileBytes = kTcTile * kTcD * 2;
constexpr int kTcAtom = kTcTile * 128;  // one 64-dim half of a K/V tile: kTcTile rows of 128 B
constexpr int kQAtom = kTcRows * 128;   // one 64-element half of Q or P: 128 rows of 128 B
constexpr int kPBytes = kTcRows * kTcTile * 2;
constexpr int kTcStages = 3;  // K and V tiles in flight per CTA
constexpr int kOffK = 0, kOffV = kOffK + kTcStages * kTcTileBytes, kOffP = kOffV + kTcStages * kTcTileBytes;
// tensor memory columns: S (single buffer), Q (bf16 pairs), O
constexpr uint32_t kTmemS = 0, kTmemQ = 64, kTmemO = 128;
// K x3, V x3, P, then the barriers inside the 1 KB kept for alignment: 113 KB, so two
// CTAs fit an SM
constexpr int kTcSmem = kOffP + kPBytes + 1024;
constexpr float kTcRescaleLog2 = 8.0f;
constexpr unsigned long long kTcWaitNs = 2000000000ull;

__device__ __forceinline__ uint32_t tc_smem(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long tc_now() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void tc_raise(int *err_flag, int bit) {
    if (err_flag) atomicOr(err_flag, bit);
}

__device__ __forceinline__ void mbar_init(uint32_t bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Wait for the phase with the given parity to complete; false after kTcWaitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    unsigned long long t0 = 0;
    for (int it = 0;; ++it) {
        uint32_t done;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if (it == 0)
            t0 = tc_now();
        else if (tc_now() - t0 > kTcWaitNs)
            return false;
    }
}

__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle: start, leading and stride byte
// offsets (16-byte units), descriptor version 1, layout type 2.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, A K-major,
// B K-major (b_mn = 0) or MN-major (1), N and M.
__host__ __device__ constexpr uint32_t bf16_idesc(int M, int N, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// The same with A (M x 16 bf16) read from tensor memory: lane = row, column c holding
// elements 2c (low half) and 2c + 1.
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of the calling thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
        "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
        "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float tc_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t tc_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Byte offset of the 16-byte chunk ch (8 bf16 values, ch in [0, 16)) of row r in a
// 128-row, 128-element K-major tile with 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_chunk(int r, int ch) {
    return (ch >> 3) * kQAtom + (r >> 3) * 1024 + (r & 7) * 128 + (((ch & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ void mbar_init_n(uint32_t bar, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(n) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Roles: warps 0-3 own the 128 rows (scores, softmax, P, epilogue); warp 4 copies K
// tiles, warp 5 V tiles, warp 6 issues the tensor-core products (one lane each).
constexpr int kTcSoftmaxWarps = 4;
constexpr int kTcWarps = 7;
constexpr int kTcAllThreads = kTcWarps * 32;

// Sixteen 8-bit codes as sixteen exact bf16 values (the caller applies the scales): e4m3 through the hardware conversion to fp16 (every e4m3 value is an fp16
// and a bf16 value); int8 through the fp16 pattern 0x64XX = 1024 + XX with XX = x + 128,
// less 1152 (exact), then fp16 -> fp32 -> bf16 (exact for |x| <= 127).
template <typename KV>
__device__ __forceinline__ void codes_to_bf16(const uint4 &c, uint4 &lo, uint4 &hi) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t h[2];
        if constexpr (std::is_same<KV, int8_t>::value) {
            const uint32_t u = w[i] ^ 0x80808080u;
            const __half2 bias = __half2half2(__ushort_as_half(0x6480));  // 1152
            const uint32_t b0 = __byte_perm(u, 0x64646464u, 0x4140), b1 = __byte_perm(u, 0x64646464u, 0x4342);
            const __half2 h0 = __hsub2(*reinterpret_cast<const __half2 *>(&b0), bias);
            const __half2 h1 = __hsub2(*reinterpret_cast<const __half2 *>(&b1), bias);
            h[0] = *reinterpret_cast<const uint32_t *>(&h0);
            h[1] = *reinterpret_cast<const uint32_t *>(&h1);
        } else {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const uint32_t pair = (w[i] >> (16 * k)) & 0xffffu;
                asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
                    : "=r"(h[k])
                    : "r"(pair));
            }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h[k]));
            out[2 * i + k] = tc_bf16x2(f.x, f.y);
        }
    }
    lo = make_uint4(out[0], out[1], out[2], out[3]);
    hi = make_uint4(out[4], out[5], out[6], out[7]);
}

struct TcShared {
    uint64_t kfull[kTcStages], vfull[kTcStages];  // tile landed (TMA transaction count)
    uint64_t kfree[kTcStages], vfree[kTcStages];  // stage consumed by S_t / by P V_t
    uint64_t sfull, sfree;        // S_t in tensor memory / read by all 128 rows
    uint64_t pfull, odone;        // P_t written by all rows / P V_t done
    uint64_t qready;              // Q in tensor memory (all 128 rows)
    uint64_t drain;               // every product issued so far is done (abort path only)
    uint64_t drain_rows;          // the same for the P V products row thread 0 issued
    uint32_t taddr;
    int abort;
};

template <int BS>
__global__ void __launch_bounds__(kTcAllThreads, 2)
multi_tc_kernel(const __grid_constant__ MultiArgs a, const __grid_constant__ CUtensorMap kmap,
                const __grid_constant__ CUtensorMap vmap) {
    extern __shared__ __align__(1024) unsigned char dsm[];
    unsigned char *base = dsm + ((1024 - (tc_smem(dsm) & 1023)) & 1023);
    // the barriers follow the tiles, inside the 1 KB kept for alignment
    if ((size_t)(base - dsm) + kOffP + kPBytes + sizeof(TcShared) > (size_t)kTcSmem) {
        if (threadIdx.x == 0) tc_raise(a.err_flag, PA_FLAG_TIMEOUT);
        return;
    }
    TcShared &sh = *reinterpret_cast<TcShared *>(base + kOffP + kPBytes);
    unsigned char *Ps = base + kOffP;
    const uint32_t p_s = tc_smem(Ps);

    const int part = blockIdx.x;
    const int kvh = blockIdx.y / a.CB, cb = blockIdx.y % a.CB;
    const int s = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- the sequence, the CTA's columns and its token range (as in pa_multi.cu); in
    // group mode blockIdx.z is a group, its members the rows and its prefix the context
    const bool grouped = a.group_prefix != nullptr;
    const int lim_ctx = min(a.M * BS, a.max_context_len);
    const bool report = part == 0 && blockIdx.y == 0 && tid == 0 && !grouped;
    const int r0 = a.query_start[s], r1 = a.query_start[s + 1];
    const int L = r1 - r0;
    int ctx;
    if (grouped) {
        // groups the setup pass rejected (their first member is not in them) and
        // prefixes past the planned maximum have nothing to attend here
        ctx = a.group_prefix[s];
        if (!(r0 >= 0 && r1 <= a.T && L >= 1 && L <= a.max_query_len && ctx >= 0 && ctx <= lim_ctx &&
              a.seq_group[r0] == s))
            return;
    } else {
        ctx = a.context_lens[s];
        if (ctx < 0 || ctx > lim_ctx) {
            if (report) tc_raise(a.err_flag, PA_FLAG_CONTEXT_OUT_OF_RANGE);
            ctx = ctx < 0 ? 0 : lim_ctx;
        }
        if (!(r0 >= 0 && r1 <= a.T && L >= 0 && L <= ctx && L <= a.max_query_len)) {
            if (report) tc_raise(a.err_flag, PA_FLAG_QUERY_OUT_OF_RANGE);
            return;
        }
    }
    const int qbase = ctx - L;
    const int ncols = L * a.G;
    const int col0 = cb * kTcRows;
    if (col0 >= ncols) return;
    const int trow = grouped ? r0 : s;  // the block table read (a group: its first member's)
    auto ctok = [&](int c) { return a.g_shift >= 0 ? c >> a.g_shift : c / a.G; };
    auto chead = [&](int c) { return a.g_shift >= 0 ? c & (a.G - 1) : c % a.G; };
    // last token column c sees: its own position, or the whole prefix of a group
    auto col_lim = [&](int c) { return grouped ? ctx - 1 : qbase + ctok(c); };
    const int cta_lim = col_lim(min(ncols, col0 + kTcRows) - 1);
    const int tok_begin = part * a.part_tokens;
    const int tok_end = min(tok_begin + a.part_tokens, cta_lim + 1);
    if (tok_begin >= tok_end) return;
    const int blk0 = tok_begin / BS;
    const int nblk = (tok_end - tok_begin + BS - 1) / BS;
    const int ntile = (tok_end - tok_begin + kTcTile - 1) / kTcTile;

    // ---- rows: thread tid < 128 owns column col0 + tid
    const bool row_thread = warp < kTcSoftmaxWarps;
    const int c = col0 + tid;
    const bool col = row_thread && c < ncols;  // a real (token or member, head) column
    int64_t pair = 0;
    if (col) pair = (int64_t)(r0 + ctok(c)) * a.Hq + kvh * a.G + chead(c);
    // a group's member left out by the setup pass computes (its query row exists) but
    // writes nothing
    const bool has = col && (!grouped || a.seq_group[r0 + ctok(c)] == s);
    const int lim = has ? col_lim(c) : -1;  // last visible token
    const int lim_p = min(lim, tok_end - 1);     // ... inside this partition
    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < kTcStages; ++i) {
            mbar_init(tc_smem(&sh.kfull[i]));
            mbar_init(tc_smem(&sh.vfull[i]));
            mbar_init(tc_smem(&sh.kfree[i]));
            mbar_init(tc_smem(&sh.vfree[i]));
        }
        mbar_init(tc_smem(&sh.sfull));
        mbar_init_n(tc_smem(&sh.sfree), kTcRows);
        mbar_init_n(tc_smem(&sh.pfull), kTcRows);
        mbar_init_n(tc_smem(&sh.qready), kTcRows);
        mbar_init(tc_smem(&sh.odone));
        mbar_init(tc_smem(&sh.drain));
        mbar_init(tc_smem(&sh.drain_rows));
        sh.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(tc_smem(&sh.taddr))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.taddr;
    const uint32_t t_o = tmem + kTmemO;
    // the row's query into tensor memory (lane = row), as bf16 pairs: the A operand of S
    if (row_thread) {
        const uint4 *src = reinterpret_cast<const uint4 *>(a.q + pair * kTcD);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float w[32];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint4 x = make_uint4(0u, 0u, 0u, 0u);
                if (col) x = __ldg(src + 8 * h + i);
                w[4 * i] = __uint_as_float(x.x);
                w[4 * i + 1] = __uint_as_float(x.y);
                w[4 * i + 2] = __uint_as_float(x.z);
                w[4 * i + 3] = __uint_as_float(x.w);
            }
            tmem_st32(tmem + ((uint32_t)(warp * 32) << 16) + kTmemQ + 32 * h, w);
        }
        tmem_wait_st();
        // the product warp waits for this before the first S; the copy warps start
        // fetching K and V meanwhile
        tc_fence_before();
        mbar_arrive(tc_smem(&sh.qready));
    }

    if (warp == 4 || warp == 5) {
        // ---- copies: K (warp 4) or V (warp 5) tiles into their three stages; the whole
        // warp follows the loop (waits), lane 0 issues
        const bool is_k = warp == 4;
        const CUtensorMap *map = is_k ? &kmap : &vmap;
        const int oob_row = a.N * a.Hkv * BS;  // a row past the pool: the copy fills zeros
        int issued = 0;
#pragma unroll 1
        for (int t = 0; t < ntile; ++t) {
            const int st = t % kTcStages, use = t / kTcStages;
            // lane i < kTcTile / BS reads the table entry of the tile's block i; entries
            // outside [0, N) are flagged (once, by the K copies of the first column
            // block) and read as zeros, like blocks past the partition
            int y = oob_row;
            const int idx = t * (kTcTile / BS) + lane;
            if (lane < kTcTile / BS && idx < nblk) {
                const int b = __ldg(a.block_tables + (int64_t)trow * a.M + blk0 + idx);
                if (b >= 0 && b < a.N)
                    y = (b * a.Hkv + kvh) * BS;
                else if (is_k && cb == 0)
                    tc_raise(a.err_flag, PA_FLAG_BLOCK_OUT_OF_RANGE);
            }
            bool ok = true;
            if (use > 0) ok = mbar_wait(tc_smem(is_k ? &sh.kfree[st] : &sh.vfree[st]), (use - 1) & 1);
            if (__any_sync(0xffffffffu, !ok || sh.abort != 0)) {
                if (lane == 0 && !ok) atomicOr(&sh.abort, 1);
                break;
            }
            if (lane == 0) mbar_expect(tc_smem(is_k ? &sh.kfull[st] : &sh.vfull[st]), kTcTileBytes);
            __syncwarp();
            const uint32_t bar = tc_smem(is_k ? &sh.kfull[st] : &sh.vfull[st]);
            const uint32_t dst = tc_smem(base + (is_k ? kOffK : kOffV) + st * kTcTileBytes);
#pragma unroll
            for (int i = 0; i < kTcTile / BS; ++i) {
                const int yi = __shfl_sync(0xffffffffu, y, i);
                if (lane == 0) {
                    tma_load(dst + (i * BS / 8) * 1024, map, 0, yi, bar);
                    tma_load(dst + kTcAtom + (i * BS / 8) * 1024, map, 64, yi, bar);
                }
            }
            __syncwarp();
            issued = t + 1;
        }
        if (issued < ntile || sh.abort != 0) {
            // stopping early: the copies already issued may still be landing in this
            // block's shared memory; wait (bounded) for the last fill of every stage
#pragma unroll 1
            for (int st = 0; st < kTcStages; ++st) {
                const StageFill f = last_fill(issued, kTcStages, st);
                if (f.any) mbar_wait(tc_smem(is_k ? &sh.kfull[st] : &sh.vfull[st]), f.parity);
            }
        }
    } else if (warp == 6) {
        // ---- the score products S_0, S_1, ... (P V is issued by row thread 0): the
        // whole warp waits, lane 0 issues
        auto issue_s = [&](int t) -> bool {
            const int st = t % kTcStages;
            bool ok = mbar_wait(tc_smem(&sh.kfull[st]), (t / kTcStages) & 1);
            if (ok && t >= 1) ok = mbar_wait(tc_smem(&sh.sfree), (t - 1) & 1);
            if (!__all_sync(0xffffffffu, ok)) return false;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t kb = tc_smem(base + kOffK + st * kTcTileBytes);
#pragma unroll
                for (int kk = 0; kk < kTcD / 16; ++kk) {
                    const uint32_t w = (kk & 3) * 32;
                    umma_ts(tmem + kTmemS, tmem + kTmemQ + kk * 8, sw128_desc(kb + (kk >> 2) * kTcAtom + w, 16, 1024),
                            bf16_idesc(128, kTcTile, 0), kk > 0);
                }
                umma_commit(tc_smem(&sh.sfull));
                umma_commit(tc_smem(&sh.kfree[st]));
            }
            __syncwarp();
            return true;
        };
        bool ok = __all_sync(0xffffffffu, mbar_wait(tc_smem(&sh.qready), 0));
        if (ok) {
            tc_fence_after();
            ok = issue_s(0);
        }
#pragma unroll 1
        for (int t = 1; ok && t < ntile; ++t) {
            ok = issue_s(t);
            if (!__all_sync(0xffffffffu, ok && sh.abort == 0)) {
                ok = false;
                break;
            }
        }
        if (!ok) {
            // stopping early: let every product already issued finish before tensor
            // memory is released (one more commit tracks all of them; bounded wait)
            if (lane == 0) {
                atomicOr(&sh.abort, 1);
                umma_commit(tc_smem(&sh.drain));
            }
            __syncwarp();
            mbar_wait(tc_smem(&sh.drain), 0);
        }
    } else {
        // ---- rows: scores, online softmax, P, output
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        int pv_issued = 0;  // row thread 0: P V products issued
        // A row warp none of whose 32 columns is real (a chunk of fewer than 97 columns
        // per kv head, e.g. draft verification) keeps only its part of the barrier
        // protocol -- it arrives on sfree and pfull in step, after the waits that keep
        // each arrival in its phase, and zeroes its share of the last tile's stale V
        // rows -- instead of reading S and writing P for rows no one reads.  Group mode
        // keeps every warp busy: there the prefix runs beside the own-token decode, and
        // a faster prefix only takes bandwidth from it.
        const bool idle_warp = !grouped && col0 + warp * 32 >= ncols;
#pragma unroll 1
        for (int j = 0; idle_warp && j < ntile; ++j) {
            const int st = j % kTcStages;
            ok = mbar_wait(tc_smem(&sh.sfull), j & 1);
            if (__any_sync(0xffffffffu, !ok || sh.abort != 0)) { ok = false; break; }
            mbar_arrive(tc_smem(&sh.sfree));
            if (j > 0) {
                ok = mbar_wait(tc_smem(&sh.odone), (j - 1) & 1);
                if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
            }
            const int k0 = tok_begin + j * kTcTile;
            const int r_lo = tok_end - k0;
            if (j == ntile - 1 && r_lo < kTcTile && tok_end % BS != 0) {
                ok = mbar_wait(tc_smem(&sh.vfull[st]), (j / kTcStages) & 1);
                if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
                const int r_hi = min(kTcTile, (tok_end + BS - 1) / BS * BS - k0);
                unsigned char *vst = base + kOffV + st * kTcTileBytes;
                for (int i = tid; i < (r_hi - r_lo) * 16; i += kTcRows) {
                    const int r = r_lo + i / 16, ch = i % 16;
                    *reinterpret_cast<uint4 *>(vst + (ch >> 3) * kTcAtom + (r >> 3) * 1024 + (r & 7) * 128 +
                                               (((ch & 7) ^ (r & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            mbar_arrive(tc_smem(&sh.pfull));
        }
#pragma unroll 1
        for (int j = 0; !idle_warp && j < ntile; ++j) {
            const int st = j % kTcStages;
            ok = mbar_wait(tc_smem(&sh.sfull), j & 1);
            if (__any_sync(0xffffffffu, !ok || sh.abort != 0)) { ok = false; break; }
            tc_fence_after();
            float sv[kTcTile];
#pragma unroll
            for (int q = 0; q < kTcTile / 32; ++q) tmem_ld32(tmem + lane_off + kTmemS + 32 * q, sv + 32 * q);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(tc_smem(&sh.sfree));

            // masked row max, eight independent chains
            const int k0 = tok_begin + j * kTcTile;
            if (k0 + kTcTile - 1 > lim_p) {
#pragma unroll
                for (int k = 0; k < kTcTile; ++k)
                    if (k0 + k > lim_p) sv[k] = -INFINITY;
            }
            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = sv[i];
#pragma unroll
            for (int k = 8; k < kTcTile; ++k) mx[k & 7] = fmaxf(mx[k & 7], sv[k]);
            const float mt_s =
                fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) *
                a.scale_log2;

            // the previous product is done: O is stable and P may be rewritten
            if (j > 0) {
                ok = mbar_wait(tc_smem(&sh.odone), (j - 1) & 1);
                if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
                tc_fence_after();
            }
            // the running max moves only when the tile's max exceeds it by more than
            // 2^8 in the exp2 domain; then the row's sum and output are rescaled
            // (tensor-memory accesses are warp-wide: the warp's other rows take 1)
            float f = 1.f;
            bool resc = false;
            if (mt_s > m_run + kTcRescaleLog2) {
                if (m_run != -INFINITY) {
                    f = tc_exp2(m_run - mt_s);
                    l_run *= f;
                    resc = true;
                }
                m_run = mt_s;
            }
            if (__any_sync(0xffffffffu, resc)) {
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    float ov[32];
                    tmem_ld32(t_o + lane_off + 32 * q, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] *= f;
                    tmem_st32(t_o + lane_off + 32 * q, ov);
                }
                tmem_wait_st();
            }
            const float mb = m_run == -INFINITY ? 0.f : m_run;
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ch = 0; ch < kTcTile / 8; ++ch) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p0 = tc_exp2(fmaf(sv[8 * ch + 2 * e], a.scale_log2, -mb));
                    const float p1 = tc_exp2(fmaf(sv[8 * ch + 2 * e + 1], a.scale_log2, -mb));
                    ls[e] += p0 + p1;
                    w[e] = tc_bf16x2(p0, p1);
                }
                *reinterpret_cast<uint4 *>(Ps + sw128_chunk(tid, ch)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            // the last tile's rows past the partition in a partly used block may hold
            // anything (a zero weight times a NaN is a NaN): zero them in the V stage
            const int r_lo = tok_end - k0;
            if (j == ntile - 1 && r_lo < kTcTile && tok_end % BS != 0) {
                ok = mbar_wait(tc_smem(&sh.vfull[st]), (j / kTcStages) & 1);
                if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
                const int r_hi = min(kTcTile, (tok_end + BS - 1) / BS * BS - k0);
                unsigned char *vst = base + kOffV + st * kTcTileBytes;
                for (int i = tid; i < (r_hi - r_lo) * 16; i += kTcRows) {
                    const int r = r_lo + i / 16, ch = i % 16;
                    *reinterpret_cast<uint4 *>(vst + (ch >> 3) * kTcAtom + (r >> 3) * 1024 + (r & 7) * 128 +
                                               (((ch & 7) ^ (r & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // P visible to the tensor core
            tc_fence_before();
            mbar_arrive(tc_smem(&sh.pfull));
            if (tid == 0) {
                // P V_j from here: once every row's P is in and V_j has landed
                const bool pv_ok = mbar_wait(tc_smem(&sh.pfull), j & 1) &&
                                   mbar_wait(tc_smem(&sh.vfull[st]), (j / kTcStages) & 1);
                if (pv_ok) {
                    tc_fence_after();
                    const uint32_t vb = tc_smem(base + kOffV + st * kTcTileBytes);
#pragma unroll
                    for (int kk = 0; kk < kTcTile / 16; ++kk)
                        umma(t_o, sw128_desc(p_s + (kk >> 2) * kQAtom + (kk & 3) * 32, 16, 1024),
                             sw128_desc(vb + kk * 2048, kTcAtom, 1024), bf16_idesc(128, 128, 1), (j > 0 || kk > 0));
                    umma_commit(tc_smem(&sh.odone));
                    umma_commit(tc_smem(&sh.vfree[st]));
                    ++pv_issued;
                } else {
                    atomicOr(&sh.abort, 1);
                }
            }
            __syncwarp();
        }
        if (ok) ok = mbar_wait(tc_smem(&sh.odone), (ntile - 1) & 1);
        if (!ok) atomicOr(&sh.abort, 1);
        if (tid == 0 && pv_issued > 0 && !ok) {
            // stopping early: the products this thread issued finish before tensor memory
            // is released (bounded wait)
            umma_commit(tc_smem(&sh.drain_rows));
            mbar_wait(tc_smem(&sh.drain_rows), 0);
        }
        tc_fence_after();
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        if (__all_sync(0xffffffffu, ok) && !idle_warp) {
            // ---- epilogue: this thread's output row (the tensor-memory loads are
            // warp-wide; rows with nothing to write discard them)
            const bool write = has && tok_begin <= lim;
            const bool finished = lim < a.part_tokens && !grouped;
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            const int64_t prow = pair * a.max_parts + part;
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                float ov[32];
                tmem_ld32(t_o + lane_off + 32 * q, ov);
                tmem_wait_ld();
                if (!write) continue;
                if (finished) {
                    uint4 *dst = reinterpret_cast<uint4 *>(a.out + pair * kTcD) + 4 * q;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_uint4(tc_bf16x2(ov[8 * i] * inv, ov[8 * i + 1] * inv),
                                            tc_bf16x2(ov[8 * i + 2] * inv, ov[8 * i + 3] * inv),
                                            tc_bf16x2(ov[8 * i + 4] * inv, ov[8 * i + 5] * inv),
                                            tc_bf16x2(ov[8 * i + 6] * inv, ov[8 * i + 7] * inv));
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(a.ws_acc + prow * kTcD) + 8 * q;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(ov[4 * i], ov[4 * i + 1], ov[4 * i + 2], ov[4 * i + 3]);
                }
            }
            if (write && !finished) *reinterpret_cast<float2 *>(a.ws_ml + prow * 2) = make_float2(m_run, l_run);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && sh.abort) tc_raise(a.err_flag, PA_FLAG_TIMEOUT);
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem) : "memory");
}

}  // namespace

namespace {

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_tiled() {
    static const EncodeTiled fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (EncodeTiled) nullptr;
        return reinterpret_cast<EncodeTiled>(p);
    }();
    return fn;
}

// A cache pool [N][Hkv][bs][128] bf16 seen as rows of 128 values, copied in boxes of
// 64 values x bs rows with the 128-byte swizzle.
bool pool_map(CUtensorMap *map, const void *pool, int rows, int bs) {
    const EncodeTiled fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kTcD, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kTcD * 2};
    const cuuint32_t box[2] = {64u, (cuuint32_t)bs};
    const cuuint32_t estr[2] = {1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(pool), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BS>
cudaError_t launch_tc_typed(const MultiArgs &a, bool merge, cudaStream_t stream) {
    CUtensorMap kmap, vmap;
    if ((int64_t)a.N * a.Hkv * BS >= (int64_t)INT32_MAX) return cudaErrorInvalidValue;  // TMA row coordinates
    const int rows = a.N * a.Hkv * BS;
    if (!pool_map(&kmap, a.k_cache, rows, BS) || !pool_map(&vmap, a.v_cache, rows, BS)) return cudaErrorInvalidValue;
    static std::atomic<bool> configured[64];  // per device: the shared-memory attribute is set
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev].load(std::memory_order_acquire)) {
        const cudaError_t e =
            cudaFuncSetAttribute(multi_tc_kernel<BS>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
        if (e != cudaSuccess) return e;
        configured[dev].store(true, std::memory_order_release);
    }
    dim3 grid(a.max_parts, a.Hkv * a.CB, a.S);
    multi_tc_kernel<BS><<<grid, kTcAllThreads, kTcSmem, stream>>>(a, kmap, vmap);
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess || a.max_parts == 1 || !merge) return err;
    return launch_multi_merge(a, kTcD, BS, stream);
}

struct tc_e4m3 {  // an fp8 (e4m3) cache entry
    uint8_t bits;
};

// 8-bit caches, prefill-shaped calls: each block a sequence attends (its first
// ceil(ctx / bs) table entries) is dequantised once -- code x scale, rounded to bf16 --
// into a bf16 pool in the workspace, block i of sequence s at s * Mq + i, and row s of
// an identity table in the workspace names it; the bf16 kernel then reads that pool.
// A table entry outside [0, N) is flagged and its block written as zeros.
// Where each sequence's dequantised blocks start in the pool: off[s] = sum over s' < s
// of the blocks its context covers, off[S] the total (one CTA; S values).
template <int BS>
__global__ void __launch_bounds__(256) pool_offsets_kernel(const __grid_constant__ MultiArgs a, int32_t *off) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ int wsum[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int carry = 0;
    for (int base = 0; base < a.S; base += 256) {
        const int s = base + tid;
        int n = 0;
        if (s < a.S) {
            const int ctx = min(max(a.context_lens[s], 0), min(a.M * BS, a.max_context_len));
            n = (ctx + BS - 1) / BS;
        }
        int v = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        if (lane == 31) wsum[warp] = v;
        __syncthreads();
        int before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            before += w < warp ? wsum[w] : 0;
            total += wsum[w];
        }
        if (s < a.S) off[s] = carry + before + v - n;
        carry += total;
        __syncthreads();
    }
    if (tid == 0) off[a.S] = carry;
}

// The blocks a sequence attends, dequantised to bf16 (code x scale, rounded once) into
// a pool of `cap` blocks, sequences back to back from off[s]; tab[s][i] is the pool slot
// of the sequence's block i (its block table for the tcgen05 kernel).  A block beyond
// the pool's capacity is left out (slot -1, read as zeros) and PA_FLAG_WORKSPACE_SHORT
// raised.
template <typename KV, int BS>
__global__ void __launch_bounds__(256) dequant_blocks_kernel(const __grid_constant__ MultiArgs a, int Mq,
                                                             uint16_t *kq, uint16_t *vq, int32_t *tab,
                                                             const int32_t *off, int64_t cap) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int i = blockIdx.x, s = blockIdx.y, tid = threadIdx.x;
    int ctx = a.context_lens[s];
    ctx = min(max(ctx, 0), min(a.M * BS, a.max_context_len));  // the attention kernel flags it
    const bool attended = i < (ctx + BS - 1) / BS;
    const int64_t dblk = (int64_t)off[s] + i;
    const bool fits = dblk < cap;
    if (tid == 0) {
        tab[(int64_t)s * Mq + i] = (attended && fits) ? (int32_t)dblk : -1;
        if (attended && !fits && a.err_flag) atomicOr(a.err_flag, PA_FLAG_WORKSPACE_SHORT);
    }
    if (!attended || !fits) return;
    const int b = a.block_tables[(int64_t)s * a.M + i];
    const bool valid = b >= 0 && b < a.N;
    if (!valid && tid == 0 && a.err_flag) atomicOr(a.err_flag, PA_FLAG_BLOCK_OUT_OF_RANGE);
    const int rows = a.Hkv * BS;  // the block's rows, all kv heads
#pragma unroll 1
    for (int kv = 0; kv < 2; ++kv) {
        const uint8_t *codes = static_cast<const uint8_t *>(kv ? a.v_cache : a.k_cache);
        const float *scales = kv ? a.v_scale : a.k_scale;
        uint16_t *dst = kv ? vq : kq;
        for (int p = tid; p < rows * (kTcD / 16); p += 256) {
            const int row = p / (kTcD / 16), q = p % (kTcD / 16);
            uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
            if (valid) {
                const int64_t src_row = (int64_t)b * rows + row;
                const uint4 c = __ldg(reinterpret_cast<const uint4 *>(codes + src_row * kTcD) + q);
                const float sc = __ldg(scales + src_row);
                codes_to_bf16<KV>(c, lo, hi);
                const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
                uint32_t o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
                    o[e] = tc_bf16x2(f.x * sc, f.y * sc);
                }
                lo = make_uint4(o[0], o[1], o[2], o[3]);
                hi = make_uint4(o[4], o[5], o[6], o[7]);
            }
            uint4 *out = reinterpret_cast<uint4 *>(dst + (dblk * rows + row) * kTcD) + 2 * q;
            out[0] = lo;
            out[1] = hi;
        }
    }
}

}  // namespace

cudaError_t launch_dequant_blocks(const MultiArgs &a, int bs, int kv_dtype, int Mq, uint16_t *kq, uint16_t *vq,
                                  int32_t *tab, int32_t *off, int64_t cap, cudaStream_t stream) {
    cudaError_t err = bs == 16 ? launch_dependent(pool_offsets_kernel<16>, dim3(1), dim3(256), 0, stream, a, off)
                               : launch_dependent(pool_offsets_kernel<32>, dim3(1), dim3(256), 0, stream, a, off);
    if (err != cudaSuccess) return err;
    const dim3 grid(Mq, a.S);
    const int32_t *coff = off;
    if (kv_dtype == PA_KV_INT8)
        return bs == 16 ? launch_dependent(dequant_blocks_kernel<int8_t, 16>, grid, dim3(256), 0, stream, a, Mq, kq, vq,
                                           tab, coff, cap)
                        : launch_dependent(dequant_blocks_kernel<int8_t, 32>, grid, dim3(256), 0, stream, a, Mq, kq, vq,
                                           tab, coff, cap);
    return bs == 16 ? launch_dependent(dequant_blocks_kernel<tc_e4m3, 16>, grid, dim3(256), 0, stream, a, Mq, kq, vq,
                                       tab, coff, cap)
                    : launch_dependent(dequant_blocks_kernel<tc_e4m3, 32>, grid, dim3(256), 0, stream, a, Mq, kq, vq,
                                       tab, coff, cap);
}

cudaError_t launch_multi_tc(const MultiArgs &a, int bs, cudaStream_t stream) {
    return bs == 16 ? launch_tc_typed<16>(a, true, stream) : launch_tc_typed<32>(a, true, stream);
}

int multi_tc_rows() { return kTcRows; }

cudaError_t launch_multi_tc_groups(const MultiArgs &a, int bs, cudaStream_t stream) {
    if (!a.group_prefix || !a.seq_group || !a.ws_acc || !a.ws_ml) return cudaErrorInvalidValue;
    return bs == 16 ? launch_tc_typed<16>(a, false, stream) : launch_tc_typed<32>(a, false, stream);
}

bool multi_tc_eligible(int D, int kv_dtype, int G, int max_query_len) {
    if (D != kTcD) return false;
    const int64_t cols = (int64_t)max_query_len * G;
    if (kv_dtype == PA_KV_BF16) return cols >= kTcMinCols;
    // 8-bit caches: through the dequantising pass, which pays where the products
    // dominate (prefill-shaped chunks)
    return (kv_dtype == PA_KV_INT8 || kv_dtype == PA_KV_FP8) && cols >= kTcRows / 2;
}

}  // namespace pa
