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

constexpr int kHornerChains = 24;
constexpr int kHornerCoefs = 128;

// The operand pattern of ap_poly's inner loop without its memory traffic: 24
// chains a thread, p_t = fma(p_t, x_t, c_k) with a distinct x_t per chain and
// c_k read from shared memory four at a time (the next four loaded one step
// ahead), 128 steps per iteration, 512 threads and one CTA per SM. The gap to
// the register-only probe is what a coefficient operand read from a register
// costs the FMA issue rate, not memory.
__global__ void __launch_bounds__(kProbeThreads, 1) fma_probe_horner_kernel(float* out, int iters) {
    __shared__ __align__(16) float buf[kHornerCoefs + 4];
    for (int k = threadIdx.x; k < kHornerCoefs + 4; k += blockDim.x)
        buf[k] = k < 4 ? 0.0f : 1e-3f * static_cast<float>(k & 7);
    __syncthreads();
    const float* cs = buf + 4;  // four zero floats before c[0]
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    float p[kHornerChains], x[kHornerChains];
#pragma unroll
    for (int t = 0; t < kHornerChains; ++t) {
        p[t] = static_cast<float>(t) * 1e-2f;
        x[t] = 0.999f + 1e-7f * static_cast<float>(threadIdx.x & 7) + 1e-8f * static_cast<float>(t);
    }
    for (int i = 0; i < iters; ++i) {
        float4 q = *reinterpret_cast<const float4*>(cs + kHornerCoefs - 4);
#pragma unroll 2
        for (int k = kHornerCoefs - 1; k >= 3; k -= 4) {
            const float4 next = *reinterpret_cast<const float4*>(cs + k - 7);
#pragma unroll
            for (int t = 0; t < kHornerChains; ++t) p[t] = fmaf(p[t], x[t], q.w);
#pragma unroll
            for (int t = 0; t < kHornerChains; ++t) p[t] = fmaf(p[t], x[t], q.z);
#pragma unroll
            for (int t = 0; t < kHornerChains; ++t) p[t] = fmaf(p[t], x[t], q.y);
#pragma unroll
            for (int t = 0; t < kHornerChains; ++t) p[t] = fmaf(p[t], x[t], q.x);
            q = next;
        }
    }
    float s = 0.0f;
#pragma unroll
    for (int t = 0; t < kHornerChains; ++t) s += p[t];
    out[tid] = s;
}

}  // namespace

ap_status launch_fma_probe_horner(const DeviceInfo& di, float* out, int64_t out_elems, int64_t iters,
                                  cudaStream_t stream) {
    int64_t blocks = static_cast<int64_t>(di.sms);
    if (blocks * kProbeThreads > out_elems) blocks = out_elems / kProbeThreads;
    if (blocks < 1) return AP_ERR_SHAPE;
    fma_probe_horner_kernel<<<static_cast<unsigned>(blocks), kProbeThreads, 0, stream>>>(out, static_cast<int>(iters));
    return cudaGetLastError() == cudaSuccess ? AP_OK : AP_ERR_CUDA;
}

ap_status launch_fma_probe(const DeviceInfo& di, float* out, int64_t out_elems, int64_t iters, cudaStream_t stream) {
    int64_t blocks = static_cast<int64_t>(di.sms) * 2;
    if (blocks * kProbeThreads > out_elems) blocks = out_elems / kProbeThreads;
    if (blocks < 1) return AP_ERR_SHAPE;
    fma_probe_kernel<<<static_cast<unsigned>(blocks), kProbeThreads, 0, stream>>>(out, static_cast<int>(iters));
    return cudaGetLastError() == cudaSuccess ? AP_OK : AP_ERR_CUDA;
}

}  // namespace ap
