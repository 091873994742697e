// Masked / zero-filling copy of 16-byte chunks through a per-thread cp.async
// pipeline: the three forms of "Asynchronous Copies" (TVM TIRx guide),
// section A Global-to-Shared Copy, chunk by chunk: a false predicate skips
// the copy and leaves the destination unchanged, a source size copies a byte
// prefix and zero-fills the rest, and an ignored source zero-fills the whole
// chunk.
//
// Each thread owns U chunks per stage and keeps S stages in flight with
// commit groups ("Asynchronous Data Movement", section Barriers and
// pipelines: acquire a stage, commit its copies, wait for the oldest, release
// it): issue stage t + S - 1, commit, wait until at most S - 1 groups are
// pending (so stage t has landed), store stage t. A thread reads back only
// the chunks it copied itself, so no CTA barrier is needed (the page's CTA
// barrier is for reading a neighbour's row).
#include <atomic>

#include "device_common.cuh"
#include "internal.h"

namespace ap {
namespace {

constexpr int kMcThreads = 256;
constexpr int kMcChunks = 4;  // chunks per thread per stage: 16 KiB per CTA stage
constexpr int kMcStageChunks = kMcThreads * kMcChunks;
constexpr int kMcMaxStages = 6;

struct McParams {
    const unsigned char* in;
    unsigned char* out;
    const signed char* codes;
    int64_t n_chunks;
    uint32_t* status;
    int64_t run_chunks;  // 0: persistent grid (CTA b takes stages b, b + grid, ...); else chunks a CTA takes
};

// This thread's codes of the stage at `base` (chunk base + tid + u * kMcThreads
// for u < kMcChunks), -1 past `limit` (the end of the CTA's chunks); loaded one
// iteration before they are needed so the load latency hides behind the
// current stage.
__device__ __forceinline__ void load_codes(const McParams& P, int64_t base, int64_t limit, int tid,
                                           int (&c)[kMcChunks]) {
#pragma unroll
    for (int u = 0; u < kMcChunks; ++u) {
        const int64_t k = base + tid + static_cast<int64_t>(u) * kMcThreads;
        c[u] = k < limit ? static_cast<int>(P.codes[k]) : -1;
    }
}

// Issue this thread's copies of a stage; its codes are kept in shared memory
// beside the data (each thread reads back only the codes it wrote).
__device__ __forceinline__ void issue_stage(const McParams& P, uint32_t slot, signed char* code, int64_t base,
                                            int tid, const int (&c)[kMcChunks]) {
#pragma unroll
    for (int u = 0; u < kMcChunks; ++u) {
        const int64_t k = base + tid + static_cast<int64_t>(u) * kMcThreads;
        code[tid + u * kMcThreads] = static_cast<signed char>(c[u]);
        const uint32_t dst = slot + 16u * static_cast<uint32_t>(tid + u * kMcThreads);
        const unsigned char* src = P.in + 16 * k;
        if (c[u] >= 0 && c[u] <= 16) {
            ptx::cp_async_cg16(dst, src, static_cast<uint32_t>(c[u]));  // prefix, zero fill
        } else if (c[u] == -2) {
            ptx::cp_async_cg16_ignore_src(dst, src, true);  // whole chunk zero
        }
        // c == -1 (or past the end): predicated off, nothing copied
    }
}

template <int S>
__global__ void __launch_bounds__(kMcThreads) masked_copy_kernel(const __grid_constant__ McParams P) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x;
    const uint32_t base_addr = ptx::smem_addr(smem);
    // This CTA's stages: a persistent grid's b, b + grid, ..., or the run of
    // consecutive stages in [first, limit).
    int64_t stride, first, limit;
    if (P.run_chunks == 0) {
        stride = static_cast<int64_t>(gridDim.x) * kMcStageChunks;
        first = static_cast<int64_t>(blockIdx.x) * kMcStageChunks;
        limit = P.n_chunks;
    } else {
        stride = kMcStageChunks;
        first = static_cast<int64_t>(blockIdx.x) * P.run_chunks;
        limit = first + P.run_chunks < P.n_chunks ? first + P.run_chunks : P.n_chunks;
    }
    signed char* codes = reinterpret_cast<signed char*>(smem + static_cast<size_t>(S) * kMcStageChunks * 16);

    // prologue: stages 0 .. S-2 in flight (empty groups keep the count right)
    int c[kMcChunks];
#pragma unroll
    for (int t = 0; t < S - 1; ++t) {
        load_codes(P, first + t * stride, limit, tid, c);
        issue_stage(P, base_addr + t * kMcStageChunks * 16u, codes + t * kMcStageChunks, first + t * stride, tid, c);
        ptx::cp_async_commit();
    }
    load_codes(P, first + (S - 1) * stride, limit, tid, c);
    int slot = 0;  // stage t's slot, t mod S
    for (int64_t base = first; base < limit; base += stride, slot = slot + 1 == S ? 0 : slot + 1) {
        const int next = slot == 0 ? S - 1 : slot - 1;  // (t + S - 1) mod S
        // acquire + commit the stage S - 1 ahead (its slot was released last iteration)
        issue_stage(P, base_addr + next * kMcStageChunks * 16u, codes + next * kMcStageChunks, base + (S - 1) * stride,
                    tid, c);
        ptx::cp_async_commit();
        load_codes(P, base + S * stride, limit, tid, c);  // for the next iteration
        // wait: at most S - 1 groups pending, so this thread's copies of stage t have landed
        ptx::cp_async_wait_group<S - 1>();
        const unsigned char* sl = smem + static_cast<size_t>(slot) * kMcStageChunks * 16;
#pragma unroll
        for (int u = 0; u < kMcChunks; ++u) {
            const int code = codes[slot * kMcStageChunks + tid + u * kMcThreads];
            const int64_t k = base + tid + static_cast<int64_t>(u) * kMcThreads;
            if (k >= limit || code == -1) continue;
            if (code < -2 || code > 16) {
                atomicCAS(P.status, 0u, 11u /* AP_ERR_ARG */ | (SITE_MASKED_CODE << 8));
                continue;
            }
            const uint4 v = *reinterpret_cast<const uint4*>(sl + 16 * (tid + u * kMcThreads));
            *reinterpret_cast<uint4*>(P.out + 16 * k) = v;
        }
        // release: the slot is refilled by this same thread next iteration
    }
    ptx::cp_async_wait_all();
}

template <int S>
ap_status launch_masked_s(const DeviceInfo& di, McParams P, int64_t run, cudaStream_t stream) {
    const int64_t stages_total = (P.n_chunks + kMcStageChunks - 1) / kMcStageChunks;
    int64_t grid;
    if (run > 0) {
        // runs of `run` consecutive stages per CTA, as many CTAs as that takes
        const int64_t cap = int64_t(1) << 30;
        if ((stages_total + run - 1) / run > cap) run = (stages_total + cap - 1) / cap;
        grid = (stages_total + run - 1) / run;
        P.run_chunks = run * kMcStageChunks;
    } else {
        // persistent: two CTAs per SM at every depth (measured on 2^26 plain
        // chunks: one CTA per SM 0.73 of the copy, two 0.95, three 0.86-0.92,
        // four 0.93)
        grid = static_cast<int64_t>(di.sms) * 2;
        if (grid > stages_total) grid = stages_total;
        P.run_chunks = 0;
    }
    if (grid < 1) grid = 1;
    const size_t smem = static_cast<size_t>(S) * kMcStageChunks * 17;  // data + one code byte per chunk
    static std::atomic<int> configured[64];  // attribute set on this device (setting twice is harmless)
    if (di.device < 0 || di.device >= 64) return AP_ERR_CUDA;
    if (!configured[di.device].load()) {
        if (cudaFuncSetAttribute(masked_copy_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kMcMaxStages * kMcStageChunks * 17)) != cudaSuccess)
            return AP_ERR_CUDA;
        configured[di.device] = 1;
    }
    record_launch(PATH_MASKED, grid, kMcStageChunks * 4, static_cast<int64_t>(smem), S, 0);
    record_ring_shape(P.run_chunks / kMcStageChunks, kMcThreads / 32, 1, 0);
    masked_copy_kernel<S><<<static_cast<unsigned>(grid), kMcThreads, smem, stream>>>(P);
    return cudaGetLastError() == cudaSuccess ? AP_OK : AP_ERR_CUDA;
}

}  // namespace

ap_status launch_masked_copy(const DeviceInfo& di, const Options& o, const float* in, float* out, int64_t n_chunks,
                             const signed char* codes, int stages, cudaStream_t stream) {
    McParams P{reinterpret_cast<const unsigned char*>(in), reinterpret_cast<unsigned char*>(out), codes, n_chunks,
               di.status, 0};
    // Schedule (AP_DBG_RING_RUN: 1 persistent, r >= 2 runs of r stages).
    // Automatic: at depths 2-4 (up to 68 KiB of shared memory a CTA, three
    // CTAs a SM) runs of one pipeline's worth of stages, so the grid streams
    // one narrow window of memory: plain chunks 0.976 -> 1.031-1.042 of the
    // copy, mixed codes 0.63 -> 0.67 (2^26 chunks). At depths 5-6 (two CTAs
    // a SM) a run's start is exposed and the persistent grid stays faster
    // (0.973 against 0.88-0.94).
    const int64_t run = o.ring_run >= 2 ? o.ring_run : (o.ring_run == 1 || stages > 4 ? 0 : stages);
    switch (stages) {
        case 2: return launch_masked_s<2>(di, P, run, stream);
        case 3: return launch_masked_s<3>(di, P, run, stream);
        case 4: return launch_masked_s<4>(di, P, run, stream);
        case 5: return launch_masked_s<5>(di, P, run, stream);
        default: return launch_masked_s<6>(di, P, run, stream);
    }
}

}  // namespace ap
