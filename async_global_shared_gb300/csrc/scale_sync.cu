// Synchronous baseline for ap_scale: the classic tiled loop of
// "CUDA Async Copy and Pipeline Guide", section Implementation Comparison,
// "Before" kernel (and the load -> barrier -> compute -> barrier loop that
// opens "Asynchronous Data Movement"): one CTA per tile, every thread copies
// its elements into shared memory with ordinary loads, the CTA waits,
// multiplies, waits again, stores. Loading and computing alternate instead
// of overlapping; this kernel is what the pipelined ring is measured against.
#include "internal.h"
#include "ptx.cuh"

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

// The pages' own asynchronous version of the same tiled scale, kept as a
// second baseline: "CUDA Async Copy and Pipeline Guide", section
// Implementation Comparison, "After" kernel (and the two-stage pipeline of
// "Asynchronous Data Movement", section Double buffering): a two-stage
// double buffer of one tile each, every thread copying its own 4-byte
// element with an asynchronous copy (cp.async.ca, what memcpy_async becomes
// on this hardware), committing, waiting for the older group, a CTA barrier,
// compute, store. The page's kernel has every block walk every tile; here
// block b takes tiles b, b + grid, ... (the plain reading of splitting the
// work across blocks). Tiles of up to 1024 floats, one element per thread.
namespace ap {
namespace {

__global__ void scale_pages_async_kernel(const float* in, float* out, int64_t n_tiles, int tile, float alpha) {
    extern __shared__ __align__(16) float dbuf[];  // [2][tile]
    const int tid = threadIdx.x;
    const bool mine = tid < tile;
    const uint32_t base = ptx::smem_addr(dbuf);
    int64_t t = blockIdx.x;
    if (t >= n_tiles) return;
    // prologue: the first tile's copy in flight
    if (mine) ptx::cp_async_ca4(base + 4u * tid, in + t * tile + tid);
    ptx::cp_async_commit();
    int cur = 0;
    for (; t < n_tiles; t += gridDim.x) {
        const int64_t nxt = t + gridDim.x;
        if (nxt < n_tiles && mine) ptx::cp_async_ca4(base + 4u * ((cur ^ 1) * tile + tid), in + nxt * tile + tid);
        ptx::cp_async_commit();
        ptx::cp_async_wait_group<1>();  // this tile's copy has landed
        __syncthreads();
        if (mine) out[t * tile + tid] = dbuf[cur * tile + tid] * alpha;
        __syncthreads();  // the buffer may now be refilled
        cur ^= 1;
    }
    ptx::cp_async_wait_all();
}

}  // namespace

ap_status launch_scale_pages_async(const DeviceInfo& di, const float* in, float* out, int64_t n_tiles, int64_t tile,
                                   float alpha, cudaStream_t stream) {
    const int threads = static_cast<int>((tile + 31) / 32 * 32);
    int64_t grid = static_cast<int64_t>(di.sms) * (2048 / threads);  // full residency
    if (grid > n_tiles) grid = n_tiles;
    record_launch(PATH_PAGES_ASYNC, grid, tile, 8 * tile, 2, 0);
    scale_pages_async_kernel<<<static_cast<unsigned>(grid), threads, static_cast<size_t>(8 * tile), stream>>>(
        in, out, n_tiles, static_cast<int>(tile), alpha);
    return cudaGetLastError() == cudaSuccess ? AP_OK : AP_ERR_CUDA;
}

}  // namespace ap
