// Register-only FP32 fma throughput probe: the compute roof that bounds the
// Horner polynomial at high degree, measured under the same clocks and power
// limit as the streaming kernels instead of taken from a datasheet.
#include "internal.h"

namespace ap {
namespace {

constexpr int kProbeThreads = 512;
constexpr int kChains = 32;

// 32 independent chains per thread and an 8-fold unrolled 32-bit loop keep
// the loop overhead under 2 % of the issued instructions, so the rate this
// kernel reaches is the FMA pipe's, not the loop's.
__global__ void __launch_bounds__(kProbeThreads) fma_probe_kernel(float* out, int iters) {
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    float p[kChains];
    const float x = 0.999f + 1e-7f * static_cast<float>(threadIdx.x & 7);
    const float c = 1e-3f;
#pragma unroll
    for (int t = 0; t < kChains; ++t) p[t] = static_cast<float>(t) * 1e-2f;
#pragma unroll 8
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int t = 0; t < kChains; ++t) p[t] = fmaf(p[t], x, c);
    }
    float s = 0.0f;
#pragma unroll
    for (int t = 0; t < kChains; ++t) s += p[t];
    out[tid] = s;
}

}  // namespace

ap_status launch_fma_probe(const DeviceInfo& di, float* out, int64_t out_elems, int64_t iters, cudaStream_t stream) {
    int64_t blocks = static_cast<int64_t>(di.sms) * 2;
    if (blocks * kProbeThreads > out_elems) blocks = out_elems / kProbeThreads;
    if (blocks < 1) return AP_ERR_SHAPE;
    fma_probe_kernel<<<static_cast<unsigned>(blocks), kProbeThreads, 0, stream>>>(out, static_cast<int>(iters));
    return cudaGetLastError() == cudaSuccess ? AP_OK : AP_ERR_CUDA;
}

}  // namespace ap
