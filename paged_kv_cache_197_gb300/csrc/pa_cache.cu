// Cache-writing kernels: append (reshape_and_cache), int8 quantise-and-append and
// copy-on-write block copy.  All three move whole 16-byte vectors; they are bound by
// launch latency at decode batch sizes and by HBM bandwidth beyond that.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void raise_flag(int *err_flag, int bit) {
    if (err_flag) atomicOr(err_flag, bit);
}

// One thread moves one 16-byte chunk (8 bf16) of one K or V row.
// Chunk index layout: ((t * Hkv + h) * 2 + kv) * chunks_per_row + c.
__global__ void __launch_bounds__(kThreads)
reshape_and_cache_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                         uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                         const int64_t *__restrict__ slot_mapping, int T, int Hkv,
                         int chunks_per_row, int bs, int N, int *err_flag) {
    // a programmatic dependent of the previous kernel on the stream: wait for it, then
    // let the next one launch (it waits for this grid in turn)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t total = (int64_t)T * Hkv * 2 * chunks_per_row;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % chunks_per_row);
        const int64_t row = i / chunks_per_row;  // (t * Hkv + h) * 2 + kv
        const int kv = (int)(row & 1);
        const int64_t th = row >> 1;  // t * Hkv + h
        const int h = (int)(th % Hkv);
        const int t = (int)(th / Hkv);
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;  // padding token
        if (slot >= (int64_t)N * bs) {
            if (c == 0 && kv == 0 && h == 0) raise_flag(err_flag, PA_FLAG_SLOT_OUT_OF_RANGE);
            continue;
        }
        const int64_t blk = slot / bs;
        const int off = (int)(slot % bs);
        const int64_t dst = ((blk * Hkv + h) * bs + off) * chunks_per_row + c;
        const int64_t src = th * chunks_per_row + c;
        if (kv == 0)
            k_cache[dst] = __ldg(key + src);
        else
            v_cache[dst] = __ldg(value + src);
    }
}

// One warp quantises one row (token t, kv head h, K or V) of D values: each lane
// holds D/32 consecutive values.  IEEE division and rintf (int8) or the round-to-
// nearest-even saturating e4m3 conversion (fp8) keep the codes identical to the CPU
// statement of the rule.
template <int D, bool FP8>
__global__ void __launch_bounds__(kThreads)
quantize_kv_kernel(const uint16_t *__restrict__ key, const uint16_t *__restrict__ value,
                   int8_t *__restrict__ k_cache, int8_t *__restrict__ v_cache,
                   float *__restrict__ k_scale, float *__restrict__ v_scale,
                   const int64_t *__restrict__ slot_mapping, int T, int Hkv, int bs, int N,
                   int *err_flag) {
    constexpr int PER_LANE = D / 32;  // 4 (D = 128) or 2 (D = 64)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)T * Hkv * 2;
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows;
         r += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        const int kv = (int)(r & 1);
        const int64_t th = r >> 1;
        const int h = (int)(th % Hkv);
        const int t = (int)(th / Hkv);
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= (int64_t)N * bs) {
            if (lane == 0 && kv == 0 && h == 0) raise_flag(err_flag, PA_FLAG_SLOT_OUT_OF_RANGE);
            continue;
        }
        const uint16_t *src = (kv == 0 ? key : value) + th * D + lane * PER_LANE;
        float x[PER_LANE];
        if constexpr (PER_LANE == 4) {
            const uint2 raw = *reinterpret_cast<const uint2 *>(src);
            x[0] = __uint_as_float(raw.x << 16);
            x[1] = __uint_as_float(raw.x & 0xffff0000u);
            x[2] = __uint_as_float(raw.y << 16);
            x[3] = __uint_as_float(raw.y & 0xffff0000u);
        } else {
            const uint32_t raw = *reinterpret_cast<const uint32_t *>(src);
            x[0] = __uint_as_float(raw << 16);
            x[1] = __uint_as_float(raw & 0xffff0000u);
        }
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < PER_LANE; ++j) amax = fmaxf(amax, fabsf(x[j]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float scale = amax > 0.0f ? __fdiv_rn(amax, FP8 ? 448.0f : 127.0f) : 1.0f;
        uint32_t packed = 0;
        if constexpr (FP8) {
#pragma unroll
            for (int j = 0; j < PER_LANE; j += 2) {
                const __nv_fp8x2_storage_t two = __nv_cvt_float2_to_fp8x2(
                    make_float2(__fdiv_rn(x[j], scale), __fdiv_rn(x[j + 1], scale)), __NV_SATFINITE,
                    __NV_E4M3);
                packed |= (uint32_t)two << (8 * j);
            }
        } else {
#pragma unroll
            for (int j = 0; j < PER_LANE; ++j) {
                float qv = rintf(__fdiv_rn(x[j], scale));
                qv = fminf(fmaxf(qv, -127.0f), 127.0f);
                packed |= ((uint32_t)(int)qv & 0xffu) << (8 * j);
            }
        }
        const int64_t blk = slot / bs;
        const int off = (int)(slot % bs);
        const int64_t row_idx = (blk * Hkv + h) * bs + off;
        int8_t *dst = (kv == 0 ? k_cache : v_cache) + row_idx * D + lane * PER_LANE;
        if constexpr (PER_LANE == 4)
            *reinterpret_cast<uint32_t *>(dst) = packed;
        else
            *reinterpret_cast<uint16_t *>(dst) = (uint16_t)packed;
        if (lane == 0) (kv == 0 ? k_scale : v_scale)[row_idx] = scale;
    }
}

// Up to kPairsPerLaunch (src, dst) pairs travel in the kernel parameters.
constexpr int kPairsPerLaunch = 256;
struct CopyPairs {
    int src[kPairsPerLaunch];
    int dst[kPairsPerLaunch];
};

// blockIdx.x: pair; blockIdx.y: 0 = K cache, 1 = V cache, 2 = scales (if any).
__global__ void __launch_bounds__(kThreads)
copy_blocks_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                   float *__restrict__ k_scale, float *__restrict__ v_scale, const CopyPairs pairs,
                   int64_t block_vecs, int scale_elems) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t src = pairs.src[blockIdx.x];
    const int64_t dst = pairs.dst[blockIdx.x];
    if (blockIdx.y < 2) {
        uint4 *cache = blockIdx.y == 0 ? k_cache : v_cache;
        const uint4 *from = cache + src * block_vecs;
        uint4 *to = cache + dst * block_vecs;
        for (int64_t i = threadIdx.x; i < block_vecs; i += blockDim.x) to[i] = from[i];
    } else {
        for (int i = threadIdx.x; i < scale_elems; i += blockDim.x) {
            k_scale[dst * scale_elems + i] = k_scale[src * scale_elems + i];
            v_scale[dst * scale_elems + i] = v_scale[src * scale_elems + i];
        }
    }
}

int grid_for(int64_t work_items, int per_block) {
    int64_t blocks = (work_items + per_block - 1) / per_block;
    if (blocks < 1) blocks = 1;
    if (blocks > 152 * 64) blocks = 152 * 64;  // grid-stride beyond 64 waves of CTAs
    return (int)blocks;
}

}  // namespace

cudaError_t launch_reshape_and_cache(const uint16_t *key, const uint16_t *value, uint16_t *k_cache,
                                     uint16_t *v_cache, const int64_t *slot_mapping, int T,
                                     int Hkv, int D, int bs, int N, int *err_flag,
                                     cudaStream_t stream) {
    const int chunks = D / 8;
    const int64_t items = (int64_t)T * Hkv * 2 * chunks;
    return launch_dependent(reshape_and_cache_kernel, dim3(grid_for(items, kThreads)), dim3(kThreads), 0,
                            stream, reinterpret_cast<const uint4 *>(key),
                            reinterpret_cast<const uint4 *>(value), reinterpret_cast<uint4 *>(k_cache),
                            reinterpret_cast<uint4 *>(v_cache), slot_mapping, T, Hkv, chunks, bs, N,
                            err_flag);
}

cudaError_t launch_quantize_kv(const uint16_t *key, const uint16_t *value, int8_t *k_cache,
                               int8_t *v_cache, float *k_scale, float *v_scale,
                               const int64_t *slot_mapping, int T, int Hkv, int D, int bs, int N,
                               int *err_flag, cudaStream_t stream) {
    const int64_t warps = (int64_t)T * Hkv * 2;
    const dim3 grid(grid_for(warps, kThreads / 32));
    return launch_dependent(D == 128 ? quantize_kv_kernel<128, false> : quantize_kv_kernel<64, false>, grid,
                            dim3(kThreads), 0, stream, key, value, k_cache, v_cache, k_scale, v_scale,
                            slot_mapping, T, Hkv, bs, N, err_flag);
}

cudaError_t launch_quantize_kv_fp8(const uint16_t *key, const uint16_t *value, uint8_t *k_cache,
                                   uint8_t *v_cache, float *k_scale, float *v_scale,
                                   const int64_t *slot_mapping, int T, int Hkv, int D, int bs,
                                   int N, int *err_flag, cudaStream_t stream) {
    const int64_t warps = (int64_t)T * Hkv * 2;
    const dim3 grid(grid_for(warps, kThreads / 32));
    int8_t *kc = reinterpret_cast<int8_t *>(k_cache), *vc = reinterpret_cast<int8_t *>(v_cache);
    return launch_dependent(D == 128 ? quantize_kv_kernel<128, true> : quantize_kv_kernel<64, true>, grid,
                            dim3(kThreads), 0, stream, key, value, kc, vc, k_scale, v_scale, slot_mapping, T,
                            Hkv, bs, N, err_flag);
}

cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, float *k_scale, float *v_scale,
                               const int64_t *block_mapping, int n, size_t block_bytes,
                               int scale_elems_per_block, cudaStream_t stream) {
    const int64_t block_vecs = (int64_t)(block_bytes / 16);
    for (int base = 0; base < n; base += kPairsPerLaunch) {
        const int count = n - base < kPairsPerLaunch ? n - base : kPairsPerLaunch;
        CopyPairs pairs;
        for (int i = 0; i < count; ++i) {
            pairs.src[i] = (int)block_mapping[2 * (base + i)];
            pairs.dst[i] = (int)block_mapping[2 * (base + i) + 1];
        }
        dim3 grid(count, k_scale ? 3 : 2);
        cudaError_t err = launch_dependent(copy_blocks_kernel, grid, dim3(kThreads), 0, stream,
                                           reinterpret_cast<uint4 *>(k_cache),
                                           reinterpret_cast<uint4 *>(v_cache), k_scale, v_scale, pairs,
                                           block_vecs, scale_elems_per_block);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace pa
