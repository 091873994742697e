// CTA-to-CTA shared-memory hand-off inside a thread-block cluster,
// "Asynchronous Copies" (TVM TIRx guide), section Copies between CTAs: the
// sender bulk-copies a chunk of its shared memory into the shared memory of
// another CTA of the cluster with cp.async.bulk.shared::cluster.shared::cta;
// completion lands on a transaction barrier in the DESTINATION CTA, which
// registers the expected byte count and waits for its phase before reading;
// every barrier is initialised (and the initialisation fenced and published
// with a cluster barrier) before any CTA sends; all CTAs synchronise before
// any of them exits.
//
// Each cluster walks a sequence of groups of cluster_size chunks through a
// ring of S send slots and S receive slots per CTA. CTA rank r has three
// roles, one warp each for the two single-thread roles:
//   loader   (warp 0): waits credit[s], loads its chunk of the group from
//            global memory into send[s] (bulk copy, load_full[s]).
//   pusher   (warp 1): waits load_full[s], pushes send[s] into recv[s] of
//            rank (r-1) mod cs, completing on that CTA's recv_full[s].
//   receiver (8 warps): registers chunk_bytes on its recv_full[s], waits,
//            stores recv[s] to its output chunk with 16-byte stores, then
//            each warp arrives (remote, release.cluster) on credit[s] of
//            rank (r+1) mod cs, the CTA that sends to it.
// credit[s] therefore tells a sender both that its send[s] has been read
// (the data reached the receiver) and that the receiver's recv[s] is free,
// so the loader may refill send[s] and the pusher may overwrite recv[s].
#include <algorithm>

#include "device_common.cuh"
#include "internal.h"

namespace ap {
namespace {

constexpr int kExConsumerWarps = 8;
constexpr int kExConsumers = 32 * kExConsumerWarps;
constexpr int kExThreads = 64 + kExConsumers;

struct ExParams {
    const float* in;
    float* out;
    int64_t groups;        // whole groups of cluster_size chunks
    uint32_t chunk_bytes;  // multiple of 16
    int cs;                // cluster size
    int stages;            // ring slots per direction
    uint32_t tx_extra;
    uint64_t timeout_ns;
    uint32_t* status;
};

__global__ void __launch_bounds__(kExThreads, 1) exchange_kernel(const __grid_constant__ ExParams P) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int S = P.stages;
    const uint32_t CB = P.chunk_bytes;
    unsigned char* send = smem;
    unsigned char* recv = smem + static_cast<size_t>(S) * CB;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * static_cast<size_t>(S) * CB);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 3 * S);
    const uint32_t bar_base = ptx::smem_addr(bars);
    auto load_full = [&](int s) { return bar_base + 8u * static_cast<uint32_t>(s); };
    auto credit = [&](int s) { return bar_base + 8u * static_cast<uint32_t>(S + s); };
    auto recv_full = [&](int s) { return bar_base + 8u * static_cast<uint32_t>(2 * S + s); };

    const uint32_t cs = static_cast<uint32_t>(P.cs);
    const uint32_t rank = ptx::cluster_ctarank();
    const uint32_t dst_rank = (rank + cs - 1) % cs;  // receives this CTA's chunk
    const uint32_t src_rank = (rank + 1) % cs;       // sends this CTA its chunk
    const int64_t cid = ptx::cluster_id_x();
    const int64_t ncl = ptx::nclusters_x();
    const int64_t count = cid < P.groups ? (P.groups - cid + ncl - 1) / ncl : 0;
    const int64_t E = CB / 4;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(load_full(s), 1);
            ptx::mbar_init(credit(s), kExConsumerWarps);
            ptx::mbar_init(recv_full(s), 1);
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    ptx::cluster_sync();  // every CTA's barriers exist before anyone sends

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (warp == 0) {
        if (lane == 0) {
            int64_t i = 0;
            for (; i < count; ++i) {
                const int s = static_cast<int>(i % S);
                const uint32_t ph = static_cast<uint32_t>((i / S) & 1);
                const int64_t grp = cid + i * ncl;
                const int w = wait_phase<true>(credit(s), ph ^ 1u, P.timeout_ns, abort_flag);
                if (w != WAIT_OK) {
                    if (w == WAIT_TIMEOUT) raise_timeout(P.status, SITE_EX_LOADER_CREDIT, abort_flag);
                    break;
                }
                ptx::mbar_arrive_expect_tx(load_full(s), CB + P.tx_extra);
                ptx::bulk_g2s(ptx::smem_addr(send + static_cast<size_t>(s) * CB),
                              P.in + (grp * P.cs + rank) * E, CB, load_full(s));
            }
            for (int64_t k = i > S ? i - S : 0; k < i; ++k) {
                if (wait_phase<false>(load_full(static_cast<int>(k % S)), static_cast<uint32_t>((k / S) & 1),
                                      P.timeout_ns, nullptr) != WAIT_OK)
                    raise_timeout(P.status, SITE_EX_DRAIN, abort_flag);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t peer_recv = ptx::mapa(ptx::smem_addr(recv), dst_rank);
            const uint32_t peer_bars = ptx::mapa(bar_base, dst_rank);
            for (int64_t i = 0; i < count; ++i) {
                const int s = static_cast<int>(i % S);
                const uint32_t ph = static_cast<uint32_t>((i / S) & 1);
                const int w = wait_phase<false>(load_full(s), ph, P.timeout_ns, abort_flag);
                if (w != WAIT_OK) {
                    if (w == WAIT_TIMEOUT) raise_timeout(P.status, SITE_EX_PUSHER_LOADED, abort_flag);
                    break;
                }
                ptx::bulk_s2s_cluster(peer_recv + static_cast<uint32_t>(s) * CB,
                                      ptx::smem_addr(send + static_cast<size_t>(s) * CB), CB,
                                      peer_bars + 8u * static_cast<uint32_t>(2 * S + s));
            }
        }
    } else {
        const int cw = warp - 2;
        const int ct = threadIdx.x - 64;
        const bool leader = (cw == 0 && lane == 0);
        const uint32_t peer_credit = ptx::mapa(credit(0), src_rank);
        int64_t i = 0;
        int64_t armed = 0;  // items [0, armed) have their expected bytes registered
        for (; i < count; ++i) {
            const int s = static_cast<int>(i % S);
            const uint32_t ph = static_cast<uint32_t>((i / S) & 1);
            const int64_t grp = cid + i * ncl;
            if (leader) {
                ptx::mbar_arrive_expect_tx(recv_full(s), CB);
                armed = i + 1;
            }
            int w = WAIT_OK;
            if (lane == 0) {
                w = wait_phase<true>(recv_full(s), ph, P.timeout_ns, abort_flag);
                if (w == WAIT_TIMEOUT) raise_timeout(P.status, SITE_EX_RECEIVER_FULL, abort_flag);
            }
            w = __shfl_sync(0xffffffffu, w, 0);
            if (w != WAIT_OK) break;
            __syncwarp();
            const float4* src = reinterpret_cast<const float4*>(recv + static_cast<size_t>(s) * CB);
            float4* dst = reinterpret_cast<float4*>(P.out + (grp * P.cs + rank) * E);
            const int64_t nq = CB / 16;
            int64_t q = ct;
            for (; q + 3 * kExConsumers < nq; q += 4 * kExConsumers) {
                const float4 a = src[q];
                const float4 b = src[q + kExConsumers];
                const float4 c = src[q + 2 * kExConsumers];
                const float4 d = src[q + 3 * kExConsumers];
                dst[q] = a;
                dst[q + kExConsumers] = b;
                dst[q + 2 * kExConsumers] = c;
                dst[q + 3 * kExConsumers] = d;
            }
            for (; q < nq; q += kExConsumers) dst[q] = src[q];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_remote(peer_credit + 8u * static_cast<uint32_t>(s));
        }
        if (leader && i < count) {
            // Gave up early: chunks a peer already sent may still be landing in
            // recv[]. Wait for them (bounded) before the final cluster barrier.
            for (int64_t k = i; k < count && k < i + S; ++k) {
                const int s = static_cast<int>(k % S);
                if (k >= armed) ptx::mbar_arrive_expect_tx(recv_full(s), CB);
                if (wait_phase<true>(recv_full(s), static_cast<uint32_t>((k / S) & 1), P.timeout_ns, nullptr) !=
                    WAIT_OK)
                    raise_timeout(P.status, SITE_EX_DRAIN, abort_flag);
            }
        }
    }
    __syncwarp();
    ptx::cluster_sync();  // no CTA leaves while a peer may still write its shared memory
}

}  // namespace

ap_status launch_exchange(const DeviceInfo& di, const Options& o, const float* in, float* out, int64_t n, int cs,
                          int64_t chunk_bytes, cudaStream_t stream) {
    const int64_t budget = di.smem_optin - 256;
    int64_t S = budget / (2 * chunk_bytes);
    if (S < 1) return AP_ERR_SMEM;
    if (S > 4) S = 4;
    const int64_t smem = 2 * S * chunk_bytes + 3 * 8 * S + 16;
    if (smem > di.smem_optin) return AP_ERR_SMEM;

    static bool configured[64] = {false};
    if (di.device < 0 || di.device >= 64) return AP_ERR_CUDA;
    if (!configured[di.device]) {
        if (cudaFuncSetAttribute(exchange_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, di.smem_optin) !=
            cudaSuccess)
            return AP_ERR_CUDA;
        configured[di.device] = true;
    }

    const int64_t groups = (4 * n) / (static_cast<int64_t>(cs) * chunk_bytes);
    ExParams P{in, out, groups, static_cast<uint32_t>(chunk_bytes), cs, static_cast<int>(S),
               static_cast<uint32_t>(o.tx_extra), static_cast<uint64_t>(o.timeout_ns), di.status};

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kExThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(cs), 1, 1);
    int max_clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, exchange_kernel, &cfg) != cudaSuccess || max_clusters < 1)
        return AP_ERR_CUDA;
    int64_t ncl = std::min<int64_t>(groups, max_clusters);
    if (o.grid > 0) ncl = std::max<int64_t>(1, std::min<int64_t>(ncl, o.grid / cs));
    cfg.gridDim = dim3(static_cast<unsigned>(ncl * cs), 1, 1);
    record_launch(PATH_EXCHANGE, ncl * cs, chunk_bytes / 4, smem, S, 0);
    if (cudaLaunchKernelEx(&cfg, exchange_kernel, P) != cudaSuccess) return AP_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? AP_OK : AP_ERR_CUDA;
}

}  // namespace ap
