// Synchronous baseline for ap_scale: the classic tiled loop of
// "CUDA Async Copy and Pipeline Guide", section Implementation Comparison,
// "Before" kernel (and the load -> barrier -> compute -> barrier loop that
// opens "Asynchronous Data Movement"): one CTA per tile, every thread copies
// its elements into shared memory with ordinary loads, the CTA waits,
// multiplies, waits again, stores. Loading and computing alternate instead
// of overlapping; this kernel is what the pipelined ring is measured against.
#include "internal.h"

namespace ap {
namespace {

__global__ void scale_sync_kernel(const float* in, float* out, int64_t n_tiles,
                                  int64_t tile, float alpha) {
    extern __shared__ float tile_smem[];
    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        const float* src = in + t * tile;
        float* dst = out + t * tile;
        for (int64_t k = threadIdx.x; k < tile; k += blockDim.x) tile_smem[k] = src[k];  // synchronous copy
        __syncthreads();
        for (int64_t k = threadIdx.x; k < tile; k += blockDim.x) tile_smem[k] = tile_smem[k] * alpha;  // compute
        __syncthreads();
        for (int64_t k = threadIdx.x; k < tile; k += blockDim.x) dst[k] = tile_smem[k];  // store
        __syncthreads();  // the next tile may now overwrite the buffer
    }
}

}  // namespace

ap_status launch_scale_sync(const DeviceInfo& di, const float* in, float* out, int64_t n_tiles, int64_t tile,
                            float alpha, cudaStream_t stream) {
    const int64_t smem = 4 * tile;
    if (smem > di.smem_optin) return AP_ERR_SMEM;
    if (smem > 48 * 1024) {
        if (cudaFuncSetAttribute(scale_sync_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem)) != cudaSuccess)
            return AP_ERR_CUDA;
    }
    int64_t threads = tile < 1024 ? tile : 1024;
    threads = (threads + 31) / 32 * 32;
    const int64_t grid = n_tiles < 2147483647LL ? n_tiles : 2147483647LL;
    record_launch(PATH_SYNC, grid, tile, smem, 1, 0);
    scale_sync_kernel<<<static_cast<unsigned>(grid), static_cast<unsigned>(threads), static_cast<size_t>(smem),
                        stream>>>(in, out, n_tiles, tile, alpha);
    return cudaGetLastError() == cudaSuccess ? AP_OK : AP_ERR_CUDA;
}

}  // namespace ap
