// On-device tuning of the ring's shape: "CUDA Async Copy and Pipeline Guide",
// FAQ: how many stages to use is a trade of latency hiding against shared
// memory, and the sweet spot is found by profiling. ap_autotune times the
// ring over the caller's buffers for every stage size and CTAs-per-SM count
// that fits, under both schedules (a persistent grid, or runs of consecutive
// stages per CTA; the ring depth is the caller's), keeps the fastest, and
// installs it for later calls of that operation and depth on this device.
#include <algorithm>
#include <mutex>
#include <vector>

#include "internal.h"

namespace ap {
namespace {

struct TunedKey {
    int device;
    int kind;
    int stages;
};

std::mutex g_tuned_mutex;
std::vector<std::pair<TunedKey, RingShape>> g_tuned;

}  // namespace

bool tuned_shape(int device, OpKind kind, int stages, RingShape* out) {
    std::lock_guard<std::mutex> lock(g_tuned_mutex);
    for (const auto& e : g_tuned) {
        if (e.first.device == device && e.first.kind == kind && e.first.stages == stages) {
            *out = e.second;
            return true;
        }
    }
    return false;
}

void set_tuned_shape(int device, OpKind kind, int stages, const RingShape& shape) {
    std::lock_guard<std::mutex> lock(g_tuned_mutex);
    for (auto& e : g_tuned) {
        if (e.first.device == device && e.first.kind == kind && e.first.stages == stages) {
            e.second = shape;
            return;
        }
    }
    g_tuned.push_back({TunedKey{device, static_cast<int>(kind), stages}, shape});
}

void clear_tuned_shapes() {
    std::lock_guard<std::mutex> lock(g_tuned_mutex);
    g_tuned.clear();
}

ap_status autotune_ring(const DeviceInfo& di, const Options& base, OpKind kind, const float* in, float* out,
                        int64_t n, int64_t off, int64_t unit, int stages, const OpArgs& op, RingShape* best,
                        double* best_gbs, cudaStream_t stream) {
    static const int64_t kPayloadKiB[] = {8, 12, 16, 24, 32, 48, 64, 96};
    const int warp_choices[2] = {8, 16};
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess) return AP_ERR_CUDA;
    if (cudaEventCreate(&e1) != cudaSuccess) {
        cudaEventDestroy(e0);
        return AP_ERR_CUDA;
    }
    double best_ms = -1.0;
    ap_status result = AP_OK;
    // Time one shape (median of three launches after a warm-up); a shape
    // whose ring does not fit in shared memory is skipped.
    auto try_shape = [&](const RingShape& sh) {
        Options o = base;
        o.stage_bytes = sh.payload;
        o.ctas_per_sm = sh.ctas_per_sm;
        o.ring_run = sh.run > 0 ? sh.run : 1;  // 1: the persistent grid
        o.consumer_warps = sh.consumer_warps;
        o.consumer_groups = sh.groups;
        ap_status st = launch_ring(di, o, in, out, n, off, unit, stages, op, false, stream);  // warm-up
        if (st == AP_ERR_SMEM) return;
        if (st != AP_OK) {
            result = st;
            return;
        }
        float ms_rep[3];
        for (int r = 0; r < 3 && result == AP_OK; ++r) {
            if (cudaEventRecord(e0, stream) != cudaSuccess) result = AP_ERR_CUDA;
            st = launch_ring(di, o, in, out, n, off, unit, stages, op, false, stream);
            if (st != AP_OK) result = st;
            if (cudaEventRecord(e1, stream) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
                cudaEventElapsedTime(&ms_rep[r], e0, e1) != cudaSuccess)
                result = AP_ERR_CUDA;
        }
        if (result != AP_OK) return;
        std::sort(ms_rep, ms_rep + 3);
        if (best_ms < 0.0 || ms_rep[1] < best_ms) {
            best_ms = ms_rep[1];
            *best = sh;
        }
    };
    // The built-in shape first (so the choice is never slower than it),
    // then every stage size under both schedules: a persistent grid of
    // cps = 1..4 CTAs per SM, or (cps 0) runs of `runs[r]` consecutive
    // stages per CTA.
    try_shape(auto_ring_shape(kind, stages, kind == OP_POLY ? op.degree : 0));
    const int64_t runs[3] = {stages, 2 * static_cast<int64_t>(stages), 4 * static_cast<int64_t>(stages)};
    for (int wi = 0; wi < 2 && result == AP_OK; ++wi) {
        const int warps = warp_choices[wi];
        if (kind != OP_POLY && warps != 8) continue;  // data movement: 8 consumer warps
        for (int64_t kib : kPayloadKiB) {
            for (int64_t sched = 1; sched <= 7 && result == AP_OK; ++sched) {
                const int64_t cps = sched <= 4 ? sched : 0;
                const int64_t run = sched <= 4 ? 0 : runs[sched - 5];
                // the ring of one CTA, and cps of them per SM, must fit in shared memory
                const int64_t per_cta = static_cast<int64_t>(stages) * (kib * 1024 + 176) + 16 * stages + 4096;
                if (per_cta > di.smem_optin || cps * (per_cta + 1024) > kSmemPerSM) continue;
                if (kind == OP_POLY && cps > 1) continue;  // 16 warps x 92 registers: one CTA per SM
                try_shape(RingShape{kib * 1024, cps > 0 ? cps : 1, warps, run});
            }
            if (result != AP_OK) break;
        }
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (result != AP_OK) return result;
    if (best_ms <= 0.0) return AP_ERR_SMEM;
    *best_gbs = 8.0 * static_cast<double>(n) / (best_ms * 1e-3) / 1e9;
    return AP_OK;
}

}  // namespace ap
