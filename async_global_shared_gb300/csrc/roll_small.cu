// Row shift of a small matrix in one CTA, the shape of the worked example in
// "Asynchronous Copies" (TVM TIRx guide), section A Global-to-Shared Copy:
// every thread issues 16-byte cp.async.cg copies of its piece of A into
// shared memory, commits them as one copy group, waits for its groups,
// the CTA synchronises (a CTA barrier alone would not wait for cp.async), and
// then each thread reads a row that another thread copied:
//     B[i, :] = shared[(i + shift) mod rows, :].
// For the 64 x 4 example the launch is one CTA of 64 threads and thread i
// copies row i and stores row i from row i + 1.
//
// Elements that are not inside a 16-byte aligned block of A (a misaligned
// base, a ragged end) are copied with 4-byte cp.async.ca; nothing outside A
// is read.
#include "internal.h"
#include "ptx.cuh"

namespace ap {
namespace {

__global__ void roll_small_kernel(const float* __restrict__ A, float* __restrict__ B, int64_t rows, int64_t cols,
                                  int64_t s, int vec) {
    extern __shared__ __align__(16) unsigned char sm[];
    const int64_t n = rows * cols;
    const uint64_t ia = reinterpret_cast<uint64_t>(A);
    const uint32_t lead = static_cast<uint32_t>(ia & 15);  // shared copy keeps A's alignment mod 16
    const uint32_t base = ptx::smem_addr(sm);
    const uint64_t i0 = ceil16(ia);
    const uint64_t i1 = floor16(ia + 4 * static_cast<uint64_t>(n));
    const int tid = threadIdx.x;
    const int nt = blockDim.x;

    if (i0 <= i1) {
        const int64_t chunks = static_cast<int64_t>((i1 - i0) >> 4);
        const uint32_t first = static_cast<uint32_t>(i0 - (ia - lead));
        for (int64_t q = tid; q < chunks; q += nt)
            ptx::cp_async_cg16(base + first + 16u * static_cast<uint32_t>(q),
                               reinterpret_cast<const void*>(i0 + 16 * static_cast<uint64_t>(q)), 16u);
        const int64_t h = static_cast<int64_t>((i0 - ia) >> 2);  // elements before the first boundary
        const int64_t t = static_cast<int64_t>((i1 - ia) >> 2);  // first element after the last boundary
        const int64_t edge = h + (n - t);
        for (int64_t k = tid; k < edge; k += nt) {
            const int64_t x = k < h ? k : t + (k - h);
            ptx::cp_async_ca4(base + lead + 4u * static_cast<uint32_t>(x), A + x);
        }
    } else {
        for (int64_t x = tid; x < n; x += nt) ptx::cp_async_ca4(base + lead + 4u * static_cast<uint32_t>(x), A + x);
    }
    ptx::cp_async_commit();
    ptx::cp_async_wait_all();
    __syncthreads();

    const int64_t off = s * cols;  // a shift by whole rows is a rotation of the flat matrix
    if (vec) {
        // A, B 16-byte aligned and cols a multiple of 4: one 16-byte piece per step.
        const float4* src = reinterpret_cast<const float4*>(sm);
        float4* dst = reinterpret_cast<float4*>(B);
        for (int64_t q = tid; q < n / 4; q += nt) {
            int64_t x = 4 * q + off;
            if (x >= n) x -= n;
            dst[q] = src[x / 4];
        }
    } else {
        const float* src = reinterpret_cast<const float*>(sm + lead);
        for (int64_t e = tid; e < n; e += nt) {
            int64_t x = e + off;
            if (x >= n) x -= n;
            B[e] = src[x];
        }
    }
}

}  // namespace

ap_status launch_roll_small(const DeviceInfo& di, const float* A, float* B, int64_t rows, int64_t cols, int64_t s,
                            cudaStream_t stream) {
    (void)di;
    const int64_t n = rows * cols;
    const uint64_t ia = reinterpret_cast<uint64_t>(A), ob = reinterpret_cast<uint64_t>(B);
    const int vec = ((ia & 15) == 0 && (ob & 15) == 0 && cols % 4 == 0) ? 1 : 0;
    int64_t threads = (n + 3) / 4;  // one 16-byte piece per thread (the example: one row each)
    threads = (threads + 31) / 32 * 32;
    if (threads < 32) threads = 32;
    if (threads > 1024) threads = 1024;
    const size_t smem = static_cast<size_t>(4 * n + 16);
    record_launch(PATH_ROLL_SMALL, 1, n, static_cast<int64_t>(smem), 0, (ia & 15) ? 1 : 0);
    roll_small_kernel<<<1, static_cast<unsigned>(threads), smem, stream>>>(A, B, rows, cols, s, vec);
    return cudaGetLastError() == cudaSuccess ? AP_OK : AP_ERR_CUDA;
}

}  // namespace ap
