// Host-side interfaces between the C-ABI entry points (api.cu) and the
// per-kernel launchers (one translation unit per kernel family).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "asyncpipe.h"
#include "asyncpipe_debug.h"
#include "stream_plan.h"

namespace ap {

// Per-device facts, looked up once per device.
struct DeviceInfo {
    int device;
    int sms;                 // streaming multiprocessors
    int smem_optin;          // max dynamic shared memory per CTA (opt-in), bytes
    uint32_t* status;        // device address of this device's status word
};

// Snapshot of the process-wide tuning / fault-injection settings.
struct Options {
    int64_t force_path;
    int64_t tx_extra;
    int64_t timeout_ns;
    int64_t stage_bytes;
    int64_t grid;
    int64_t ctas_per_sm;
    int64_t roll_stages;
    int64_t consumer_warps;
    int64_t ex_tma_store;
    int64_t device_checks;
    int64_t ex_group;
    int64_t strict_align;
    int64_t ex_lanes;
    int64_t ex_batch;
    int64_t ex_send_slots;
    int64_t ring_run;
    int64_t consumer_groups;
};

Options options();

// cuTensorMapEncodeTiled through the runtime's driver entry point (nullptr if
// the driver lacks it).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// What a launcher reports about the launch it made (AP_DBG_LAST_*).
void record_launch(int64_t path, int64_t grid, int64_t stage_elems, int64_t smem, int64_t stages, int64_t flags);
// The ring's schedule and consumer layout for the same launch (run 0:
// persistent grid), recorded after record_launch.
void record_ring_shape(int64_t run, int64_t warps, int64_t groups, int64_t chains);

enum Path : int64_t {
    PATH_RING = 1,
    PATH_ROLL_SMALL = 2,
    PATH_SYNC = 3,
    PATH_EXCHANGE = 4,
    PATH_MASKED = 5,
    PATH_PAGES_ASYNC = 6
};

// Arguments of the per-element compute of a ring call.
enum OpKind { OP_COPY, OP_SCALE, OP_POLY };
struct OpArgs {
    OpKind kind;
    float alpha;
    int degree;
    const float* coeffs;  // host, degree + 1
};

// Ring stage elements for a payload of `payload_bytes`, a multiple of
// lcm(4, unit) when that fits (so a stage holds whole tiles / rows).
int64_t stage_elems_for(int64_t payload_bytes, int64_t unit);

// Default ring shape for an op and ring depth: stage payload bytes, CTAs
// per SM the grid is sized for, consumer warps per CTA, and the schedule:
// run = 0 is a persistent grid of SMs x ctas_per_sm CTAs, CTA b taking stages
// b, b + grid, ...; run >= 2 gives every CTA `run` consecutive stages and
// launches as many CTAs as that takes (the hardware starts them in order as
// earlier ones finish; ctas_per_sm is then unused).
struct RingShape {
    int64_t payload;
    int64_t ctas_per_sm;
    int64_t consumer_warps;
    int64_t run = 0;
    int64_t groups = 0;  // ap_poly's consumer groups (0: the launcher's rule)
};
RingShape auto_ring_shape(OpKind kind, int stages, int degree);

// Shapes installed by ap_autotune, per device, operation and ring depth;
// they take the place of auto_ring_shape's defaults.
bool tuned_shape(int device, OpKind kind, int stages, RingShape* out);
void set_tuned_shape(int device, OpKind kind, int stages, const RingShape& shape);
void clear_tuned_shapes();

// Time every fitting (stage size, CTAs per SM, consumer warps) on the given
// buffers; the fastest goes to *best with its GB/s (8 bytes per element).
ap_status autotune_ring(const DeviceInfo& di, const Options& base, OpKind kind, const float* in, float* out,
                        int64_t n, int64_t off, int64_t unit, int stages, const OpArgs& op, RingShape* best,
                        double* best_gbs, cudaStream_t stream);

// tensor asks for the tensor-map producer; where tensor_ok() refuses the
// buffers, the 1-D bulk producer runs instead.
ap_status launch_ring(const DeviceInfo& di, const Options& o, const float* in, float* out, int64_t n, int64_t off,
                      int64_t unit, int stages, const OpArgs& op, bool tensor, cudaStream_t stream);

ap_status launch_roll_small(const DeviceInfo& di, const float* A, float* B, int64_t rows, int64_t cols, int64_t s,
                            cudaStream_t stream);

ap_status launch_scale_sync(const DeviceInfo& di, const float* in, float* out, int64_t n_tiles, int64_t tile,
                            float alpha, cudaStream_t stream);

ap_status launch_scale_pages_async(const DeviceInfo& di, const float* in, float* out, int64_t n_tiles, int64_t tile,
                                   float alpha, cudaStream_t stream);

ap_status launch_masked_copy(const DeviceInfo& di, const Options& o, const float* in, float* out, int64_t n_chunks,
                             const signed char* codes, int stages, cudaStream_t stream);

ap_status launch_fma_probe(const DeviceInfo& di, float* out, int64_t out_elems, int64_t iters, cudaStream_t stream);
ap_status launch_fma_probe_horner(const DeviceInfo& di, float* out, int64_t out_elems, int64_t iters,
                                  cudaStream_t stream);

// `groups` whole groups of cs chunks starting at in/out; rank r receives
// rank (r + shift) mod cs, or with a2a every rank sends sub-block j of its
// chunk (chunk_bytes / cs bytes each) to rank j (shift unused).
ap_status launch_exchange(const DeviceInfo& di, const Options& o, const float* in, float* out, int64_t groups, int cs,
                          int64_t chunk_bytes, int64_t shift, bool a2a, cudaStream_t stream);

// Largest chunk accepted by ap_cluster_exchange for this much shared memory.
constexpr int64_t kSmemOptinGB300 = 232448;  // 227 KiB per CTA on compute capability 10.x
constexpr int64_t kSmemPerSM = 233472;       // 228 KiB per SM
constexpr int64_t kRollSmallMaxBytes = 32 * 1024;

}  // namespace ap
