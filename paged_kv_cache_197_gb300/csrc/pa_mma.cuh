// Small inline-PTX helpers shared by the shared-memory tiled attention kernels
// (grouped prefix, multi-token): cp.async staging, ldmatrix, the bf16 m16n8k16
// tensor-core product, movmatrix and exp2.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

namespace pa {
namespace tiled {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared copy; src_bytes 0 fills the destination with zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

// 4-byte global -> shared copy (L1-allocating); src_bytes 0 writes a zero.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// c[16x8] += a[16x16] * b[16x8], bf16 operands, fp32 accumulators.
__device__ __forceinline__ void mma16816(float *c, const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(x));
    return d;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Two e4m3 codes (low byte first) as an fp16 pair; every e4m3 value is an fp16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t pair16) {
    uint32_t out;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
        : "=r"(out)
        : "r"(pair16));
    return out;
}

struct e4m3_tag {  // an fp8 (e4m3) cache entry
    uint8_t bits;
};

// 8-bit caches: sixteen codes of one row times the row's scale, as sixteen fp16 (two
// 16-byte words).  The codes become exact fp16 first -- int8 through the fp16 pattern
// 0x64XX = 1024 + XX with XX = x + 128, less 1152; fp8 (e4m3) by the hardware
// conversion (every e4m3 value is an fp16 value) -- then one fp16 multiply by the
// scale (rounded to fp16) per pair.
// Largest row scale whose staged values code x scale stay finite in fp16: the largest
// code (127 for int8, 448 for e4m3) times the scale must not pass fp16's 65504.  Rows
// with a larger scale are flagged (PA_FLAG_FP16_RANGE) by the kernels that stage them.
template <typename KV>
__host__ __device__ constexpr float max_f16_scale() {
    return std::is_same<KV, int8_t>::value ? 65504.0f / 127.0f : 65504.0f / 448.0f;
}

template <typename KV>
__device__ __forceinline__ void codes_to_f16(const uint4 &c, float scale, uint4 &lo, uint4 &hi) {
    const __half2 sc2 = __float2half2_rn(scale);
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (std::is_same<KV, int8_t>::value) {
            const uint32_t u = w[i] ^ 0x80808080u;
            const __half2 bias = __half2half2(__ushort_as_half(0x6480));  // 1152
            const uint32_t b0 = __byte_perm(u, 0x64646464u, 0x4140), b1 = __byte_perm(u, 0x64646464u, 0x4342);
            const __half2 h0 = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&b0), bias), sc2);
            const __half2 h1 = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&b1), bias), sc2);
            out[2 * i] = *reinterpret_cast<const uint32_t *>(&h0);
            out[2 * i + 1] = *reinterpret_cast<const uint32_t *>(&h1);
        } else {
            const uint32_t e0 = e4m3x2_to_f16x2(w[i] & 0xffffu), e1 = e4m3x2_to_f16x2(w[i] >> 16);
            const __half2 h0 = __hmul2(*reinterpret_cast<const __half2 *>(&e0), sc2);
            const __half2 h1 = __hmul2(*reinterpret_cast<const __half2 *>(&e1), sc2);
            out[2 * i] = *reinterpret_cast<const uint32_t *>(&h0);
            out[2 * i + 1] = *reinterpret_cast<const uint32_t *>(&h1);
        }
    }
    lo = make_uint4(out[0], out[1], out[2], out[3]);
    hi = make_uint4(out[4], out[5], out[6], out[7]);
}

// 8-bit caches: sixteen codes of one row as sixteen exact fp16 values (two 16-byte
// words), without the row's scale: int8 through the fp16 pattern 0x64XX = 1024 + XX
// with XX = x + 128, less 1152; fp8 (e4m3) by the hardware conversion.
template <typename KV>
__device__ __forceinline__ void codes_to_f16_exact(const uint4 &c, uint4 &lo, uint4 &hi) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    uint32_t out[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (std::is_same<KV, int8_t>::value) {
            const uint32_t u = w[i] ^ 0x80808080u;
            const __half2 bias = __half2half2(__ushort_as_half(0x6480));  // 1152
            const uint32_t b0 = __byte_perm(u, 0x64646464u, 0x4140), b1 = __byte_perm(u, 0x64646464u, 0x4342);
            const __half2 h0 = __hsub2(*reinterpret_cast<const __half2 *>(&b0), bias);
            const __half2 h1 = __hsub2(*reinterpret_cast<const __half2 *>(&b1), bias);
            out[2 * i] = *reinterpret_cast<const uint32_t *>(&h0);
            out[2 * i + 1] = *reinterpret_cast<const uint32_t *>(&h1);
        } else {
            out[2 * i] = e4m3x2_to_f16x2(w[i] & 0xffffu);
            out[2 * i + 1] = e4m3x2_to_f16x2(w[i] >> 16);
        }
    }
    lo = make_uint4(out[0], out[1], out[2], out[3]);
    hi = make_uint4(out[4], out[5], out[6], out[7]);
}

__device__ __forceinline__ void mma16816_f16(float *c, const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Exponent e with |x| < 2^e for a finite, positive, normal x.
__device__ __forceinline__ int exponent_above(float x) {
    return (int)((__float_as_uint(x) >> 23) & 0xffu) - 126;
}

}  // namespace tiled
}  // namespace pa
