// pa_decode_noalloc: paged decode for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code running inside a CUDA-graph capture
// that forbids new allocations, a host process that hands this library a fixed
// memory budget, or a plugin whose host application owns every allocation.  For
// them this entry point keeps pa_decode's split-K scratch in a fixed array that is
// part of the library itself, so a call needs only its inputs and outputs.
//
// The array is a file-scope __device__ variable of PA_NOALLOC_SCRATCH_BYTES bytes:
// every GPU that loads the library holds it until the process exits.  Host code
// cannot use the array's name as a device address (it names a host-side stand-in),
// so the first call on each device looks up the real address with
// cudaGetSymbolAddress while that device is current, and later calls reuse it.
#include <mutex>

#include "pa_internal.cuh"

static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_address[kMaxDevices];  // device address of the array, per device

// Device address of the scratch array on the current device (looked up once).
pa_status scratch_address(void **out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return pa::fail(PA_ERR_CUDA, "pa_decode_noalloc: cudaGetDevice: %s", cudaGetErrorString(err));
    if (dev < 0 || dev >= kMaxDevices)
        return pa::fail(PA_ERR_UNSUPPORTED, "pa_decode_noalloc: device %d beyond %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_address[dev] == nullptr) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess || p == nullptr)
            return pa::fail(PA_ERR_CUDA, "pa_decode_noalloc: cudaGetSymbolAddress: %s",
                            cudaGetErrorString(err));
        g_scratch_address[dev] = p;
    }
    *out = g_scratch_address[dev];
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(pa_bf16 *out, const pa_bf16 *query, const void *k_cache,
                                       const void *v_cache, const float *k_scale,
                                       const float *v_scale, int kv_dtype,
                                       const int32_t *block_tables, int M,
                                       const int32_t *context_lens, int S, int Hq, int Hkv, int D,
                                       int bs, int N, float scale, int max_context_len,
                                       int *err_flag, void *stream) {
    const size_t need = pa_decode_workspace_size(S, Hq, Hkv, D, bs, kv_dtype, max_context_len);
    if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES)
        return pa::fail(PA_ERR_UNSUPPORTED,
                        "pa_decode_noalloc: these sizes need %zu bytes of scratch but the built-in "
                        "array holds %zu; use pa_decode with a caller-owned workspace",
                        need, (size_t)PA_NOALLOC_SCRATCH_BYTES);
    void *scratch = nullptr;
    if (need > 0) {
        pa_status st = scratch_address(&scratch);
        if (st != PA_OK) return st;
    }
    // Nothing in the scratch has to start at zero: the decode kernel writes every
    // partial result that the merge kernel later reads, in the same call.
    return pa_decode(out, query, k_cache, v_cache, k_scale, v_scale, kv_dtype, block_tables, M,
                     context_lens, S, Hq, Hkv, D, bs, N, scale, max_context_len, scratch,
                     need > 0 ? (size_t)PA_NOALLOC_SCRATCH_BYTES : 0, err_flag, stream);
}
