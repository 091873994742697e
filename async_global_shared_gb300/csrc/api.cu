// C-ABI entry points of libasyncpipe: argument validation (before any CUDA
// call), per-device set-up, dispatch to the kernel launchers, the device
// status word, the tuning hooks and the host emulator of the ring's data
// movement.
#include <atomic>
#include <cstdlib>
#include <string>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"

namespace ap {

// One status word per device that loads the library: the first error a
// kernel records since the last ap_check. Not an allocation: a static
// device variable of the library's module.
__device__ uint32_t g_status_word;

namespace {

// ------------------------------------------------------------------ options

std::atomic<int64_t> g_force_path{0};
std::atomic<int64_t> g_tx_extra{0};
std::atomic<int64_t> g_timeout_ns{0};
std::atomic<int64_t> g_stage_bytes{0};
std::atomic<int64_t> g_grid{0};
std::atomic<int64_t> g_ctas_per_sm{0};
std::atomic<int64_t> g_roll_stages{0};
std::atomic<int64_t> g_consumer_warps{0};
std::atomic<int64_t> g_ex_tma_store{0};
std::atomic<int64_t> g_device_checks{0};
std::atomic<int64_t> g_ex_group{0};
std::atomic<int64_t> g_strict_align{0};
std::atomic<int64_t> g_ex_lanes{0};
std::atomic<int64_t> g_ex_batch{0};
std::atomic<int64_t> g_ex_send_slots{0};
std::atomic<int64_t> g_ring_run{0};
std::atomic<int64_t> g_consumer_groups{0};

std::atomic<int64_t> g_last_path{0}, g_last_grid{0}, g_last_stage_elems{0}, g_last_smem{0}, g_last_stages{0},
    g_last_flags{0}, g_last_site{0}, g_last_run{0}, g_last_warps{0}, g_last_groups{0}, g_last_chains{0};

constexpr int64_t kDefaultTimeoutNs = 2000000000LL;  // 2 s

int64_t env_timeout() {
    static const int64_t v = [] {
        const char* s = std::getenv("AP_WAIT_TIMEOUT_NS");
        if (s == nullptr || *s == '\0') return int64_t(0);
        const long long x = std::atoll(s);
        return x > 0 ? static_cast<int64_t>(x) : int64_t(0);
    }();
    return v;
}

// AP_FORCE_PATH=auto|ring|small|tensor (also bulk = ring, cpasync = small, or
// 0..3): the path a call takes when ap_debug_set has not chosen one.
int64_t env_force_path() {
    static const int64_t v = [] {
        const char* s = std::getenv("AP_FORCE_PATH");
        if (s == nullptr || *s == '\0') return int64_t(0);
        const std::string x(s);
        if (x == "ring" || x == "bulk" || x == "1") return int64_t(1);
        if (x == "small" || x == "cpasync" || x == "2") return int64_t(2);
        if (x == "tensor" || x == "3") return int64_t(3);
        return int64_t(0);
    }();
    return v;
}

// ------------------------------------------------------------------ devices

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
bool g_dev_ready[kMaxDevices];
DeviceInfo g_dev[kMaxDevices];
ap_status g_dev_err[kMaxDevices];

ap_status current_device(DeviceInfo* out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return AP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_dev_ready[dev]) {
        DeviceInfo di{};
        di.device = dev;
        ap_status st = AP_OK;
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
            st = AP_ERR_CUDA;
        } else if (major != 10 || minor != 3) {
            st = AP_ERR_UNSUPPORTED_DEVICE;
        } else {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
                st = AP_ERR_CUDA;
            } else {
                di.status = static_cast<uint32_t*>(p);
            }
        }
        if (st == AP_ERR_CUDA) return st;  // not cached: may succeed later
        g_dev[dev] = di;
        g_dev_err[dev] = st;
        g_dev_ready[dev] = true;
    }
    *out = g_dev[dev];
    return g_dev_err[dev];
}

// ------------------------------------------------------------------ validation

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }

// Byte ranges [a, a+na) and [b, b+nb) overlap.
bool overlap(const void* a, int64_t na, const void* b, int64_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + static_cast<uintptr_t>(nb) && y < x + static_cast<uintptr_t>(na);
}

constexpr int64_t kMaxElems = int64_t(1) << 40;  // keeps every byte offset far from overflow

bool valid_stages(int stages) { return stages >= AP_MIN_STAGES && stages <= AP_MAX_STAGES; }

bool aligned16(const void* a, const void* b) {
    return ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 15) == 0;
}

}  // namespace

// cuTensorMapEncodeTiled, looked up once through the runtime (no -lcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

Options options() {
    Options o;
    const int64_t fp = g_force_path.load();
    o.force_path = fp != 0 ? fp : env_force_path();
    o.tx_extra = g_tx_extra.load();
    const int64_t t = g_timeout_ns.load();
    o.timeout_ns = t > 0 ? t : (env_timeout() > 0 ? env_timeout() : kDefaultTimeoutNs);
    o.stage_bytes = g_stage_bytes.load();
    o.grid = g_grid.load();
    o.ctas_per_sm = g_ctas_per_sm.load();
    o.roll_stages = g_roll_stages.load();
    o.consumer_warps = g_consumer_warps.load();
    o.ex_tma_store = g_ex_tma_store.load();
    o.device_checks = g_device_checks.load();
    o.ex_group = g_ex_group.load();
    o.strict_align = g_strict_align.load();
    o.ex_lanes = g_ex_lanes.load();
    o.ex_batch = g_ex_batch.load();
    o.ex_send_slots = g_ex_send_slots.load();
    o.ring_run = g_ring_run.load();
    o.consumer_groups = g_consumer_groups.load();
    return o;
}

void record_launch(int64_t path, int64_t grid, int64_t stage_elems, int64_t smem, int64_t stages, int64_t flags) {
    g_last_path = path;
    g_last_grid = grid;
    g_last_stage_elems = stage_elems;
    g_last_smem = smem;
    g_last_stages = stages;
    g_last_flags = flags;
    g_last_run = g_last_warps = g_last_groups = g_last_chains = 0;
}

void record_ring_shape(int64_t run, int64_t warps, int64_t groups, int64_t chains) {
    g_last_run = run;
    g_last_warps = warps;
    g_last_groups = groups;
    g_last_chains = chains;
}

}  // namespace ap

using namespace ap;

extern "C" {

const char* ap_status_string(ap_status s) {
    switch (s) {
        case AP_OK: return "AP_OK";
        case AP_ERR_NULL: return "AP_ERR_NULL";
        case AP_ERR_SHAPE: return "AP_ERR_SHAPE";
        case AP_ERR_ALIGN: return "AP_ERR_ALIGN";
        case AP_ERR_ALIAS: return "AP_ERR_ALIAS";
        case AP_ERR_STAGES: return "AP_ERR_STAGES";
        case AP_ERR_CLUSTER: return "AP_ERR_CLUSTER";
        case AP_ERR_SMEM: return "AP_ERR_SMEM";
        case AP_ERR_CUDA: return "AP_ERR_CUDA";
        case AP_ERR_DEVICE_TIMEOUT: return "AP_ERR_DEVICE_TIMEOUT";
        case AP_ERR_UNSUPPORTED_DEVICE: return "AP_ERR_UNSUPPORTED_DEVICE";
        case AP_ERR_ARG: return "AP_ERR_ARG";
    }
    return "AP_ERR_UNKNOWN";
}

ap_status ap_scale(const float* in, float* out, int64_t n_tiles, int64_t tile_elems, float alpha, int stages,
                   cudaStream_t stream) {
    if (!valid_stages(stages)) return AP_ERR_STAGES;
    if (n_tiles < 0 || tile_elems < 1) return AP_ERR_SHAPE;
    if (n_tiles > 0 && tile_elems > kMaxElems / n_tiles) return AP_ERR_SHAPE;
    const int64_t n = n_tiles * tile_elems;
    if (n == 0) return AP_OK;
    if (in == nullptr || out == nullptr) return AP_ERR_NULL;
    if (!aligned4(in) || !aligned4(out)) return AP_ERR_ALIGN;
    if (in != out && overlap(in, 4 * n, out, 4 * n)) return AP_ERR_ALIAS;
    const Options o = options();
    if (o.strict_align && !aligned16(in, out)) return AP_ERR_ALIGN;
    DeviceInfo di;
    const ap_status st = current_device(&di);
    if (st != AP_OK) return st;
    OpArgs op{OP_SCALE, alpha, 0, nullptr};
    return launch_ring(di, o, in, out, n, 0, tile_elems, stages, op, o.force_path == 3, stream);
}

ap_status ap_scale_sync(const float* in, float* out, int64_t n_tiles, int64_t tile_elems, float alpha,
                        cudaStream_t stream) {
    if (n_tiles < 0 || tile_elems < 1) return AP_ERR_SHAPE;
    if (n_tiles > 0 && tile_elems > kMaxElems / n_tiles) return AP_ERR_SHAPE;
    const int64_t n = n_tiles * tile_elems;
    if (n == 0) return AP_OK;
    if (in == nullptr || out == nullptr) return AP_ERR_NULL;
    if (!aligned4(in) || !aligned4(out)) return AP_ERR_ALIGN;
    if (in != out && overlap(in, 4 * n, out, 4 * n)) return AP_ERR_ALIAS;
    if (4 * tile_elems > kSmemOptinGB300) return AP_ERR_SMEM;
    DeviceInfo di;
    const ap_status st = current_device(&di);
    if (st != AP_OK) return st;
    return launch_scale_sync(di, in, out, n_tiles, tile_elems, alpha, stream);
}

ap_status ap_row_roll(const float* A, float* B, int64_t rows, int64_t cols, int64_t shift, cudaStream_t stream) {
    if (rows < 0 || cols < 0) return AP_ERR_SHAPE;
    if (rows > 0 && cols > kMaxElems / rows) return AP_ERR_SHAPE;
    const int64_t n = rows * cols;
    if (n == 0) return AP_OK;
    if (A == nullptr || B == nullptr) return AP_ERR_NULL;
    if (!aligned4(A) || !aligned4(B)) return AP_ERR_ALIGN;
    if (overlap(A, 4 * n, B, 4 * n)) return AP_ERR_ALIAS;
    const Options o = options();
    if (o.strict_align && !aligned16(A, B)) return AP_ERR_ALIGN;
    // Ring depth 2 (16 KiB stages in runs of 4) measured best for the
    // 2^26 x 4 shift, aligned and with either base 4 bytes off: 1.045 of the
    // copy against 1.035-1.037 at depth 3 and 1.032-1.034 at depth 4.
    const int stages = o.roll_stages > 0 ? static_cast<int>(o.roll_stages) : 2;
    if (!valid_stages(stages)) return AP_ERR_STAGES;
    DeviceInfo di;
    const ap_status st = current_device(&di);
    if (st != AP_OK) return st;
    const int64_t s = ((shift % rows) + rows) % rows;
    const bool small = 4 * n <= kRollSmallMaxBytes;
    if (small && (o.force_path == 0 || o.force_path == 2)) {
        return launch_roll_small(di, A, B, rows, cols, s, stream);
    }
    OpArgs op{OP_COPY, 1.0f, 0, nullptr};
    // The tensor-map producer on request (it falls back to the 1-D bulk
    // producer where the matrix misses its alignment rules).
    return launch_ring(di, o, A, B, n, s * cols, cols, stages, op, o.force_path == 3, stream);
}

ap_status ap_poly(const float* in, float* out, int64_t n, const float* coeffs, int degree, int stages,
                  cudaStream_t stream) {
    if (!valid_stages(stages)) return AP_ERR_STAGES;
    if (degree < 0 || degree > AP_POLY_MAX_DEGREE) return AP_ERR_ARG;
    if (n < 0 || n > kMaxElems) return AP_ERR_SHAPE;
    if (n == 0) return AP_OK;
    if (in == nullptr || out == nullptr || coeffs == nullptr) return AP_ERR_NULL;
    if (!aligned4(in) || !aligned4(out)) return AP_ERR_ALIGN;
    if (in != out && overlap(in, 4 * n, out, 4 * n)) return AP_ERR_ALIAS;
    const Options o = options();
    if (o.strict_align && !aligned16(in, out)) return AP_ERR_ALIGN;
    DeviceInfo di;
    const ap_status st = current_device(&di);
    if (st != AP_OK) return st;
    OpArgs op{OP_POLY, 0.0f, degree, coeffs};
    return launch_ring(di, o, in, out, n, 0, 1, stages, op, o.force_path == 3, stream);
}

ap_status ap_cluster_exchange(const float* in, float* out, int64_t n, int cluster_size, int64_t chunk_bytes,
                              cudaStream_t stream) {
    if (cluster_size != 1 && cluster_size != 2 && cluster_size != 4 && cluster_size != 8) return AP_ERR_CLUSTER;
    if (chunk_bytes < 16 || chunk_bytes % 16 != 0) return AP_ERR_SHAPE;
    if (2 * chunk_bytes + 256 > kSmemOptinGB300) return AP_ERR_SMEM;
    if (n < 0 || n > kMaxElems) return AP_ERR_SHAPE;
    if ((4 * n) % (static_cast<int64_t>(cluster_size) * chunk_bytes) != 0) return AP_ERR_SHAPE;
    if (n == 0) return AP_OK;
    if (in == nullptr || out == nullptr) return AP_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(in) & 15) || (reinterpret_cast<uintptr_t>(out) & 15)) return AP_ERR_ALIGN;
    if (overlap(in, 4 * n, out, 4 * n)) return AP_ERR_ALIAS;
    DeviceInfo di;
    const ap_status st = current_device(&di);
    if (st != AP_OK) return st;
    const int64_t groups = (4 * n) / (static_cast<int64_t>(cluster_size) * chunk_bytes);
    return launch_exchange(di, options(), in, out, groups, cluster_size, chunk_bytes, 1, false, stream);
}

ap_status ap_cluster_all_to_all(const float* in, float* out, int64_t n, int cluster_size, int64_t chunk_bytes,
                                cudaStream_t stream) {
    if (cluster_size < 1 || cluster_size > AP_MAX_CLUSTER_NONPORTABLE) return AP_ERR_CLUSTER;
    if (chunk_bytes < 16 * cluster_size || chunk_bytes % (16 * cluster_size) != 0) return AP_ERR_SHAPE;
    if (n < 0 || n > kMaxElems) return AP_ERR_SHAPE;
    if ((4 * n) % (static_cast<int64_t>(cluster_size) * chunk_bytes) != 0) return AP_ERR_SHAPE;
    if (n == 0) return AP_OK;
    if (in == nullptr || out == nullptr) return AP_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(in) & 15) || (reinterpret_cast<uintptr_t>(out) & 15)) return AP_ERR_ALIGN;
    if (overlap(in, 4 * n, out, 4 * n)) return AP_ERR_ALIAS;
    DeviceInfo di;
    const ap_status st = current_device(&di);
    if (st != AP_OK) return st;
    const int64_t groups = (4 * n) / (static_cast<int64_t>(cluster_size) * chunk_bytes);
    return launch_exchange(di, options(), in, out, groups, cluster_size, chunk_bytes, 0, true, stream);
}

ap_status ap_cluster_exchange_ex(const float* in, float* out, int64_t n, int cluster_size, int64_t chunk_bytes,
                                 int64_t shift, cudaStream_t stream) {
    if (cluster_size < 1 || cluster_size > AP_MAX_CLUSTER_NONPORTABLE) return AP_ERR_CLUSTER;
    if (chunk_bytes < 16 || chunk_bytes % 16 != 0) return AP_ERR_SHAPE;
    if (2 * chunk_bytes + 256 > kSmemOptinGB300) return AP_ERR_SMEM;
    if (n < 0 || n > kMaxElems) return AP_ERR_SHAPE;
    if ((4 * n) % chunk_bytes != 0) return AP_ERR_SHAPE;
    if (n == 0) return AP_OK;
    if (in == nullptr || out == nullptr) return AP_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(in) & 15) || (reinterpret_cast<uintptr_t>(out) & 15)) return AP_ERR_ALIGN;
    if (overlap(in, 4 * n, out, 4 * n)) return AP_ERR_ALIAS;
    DeviceInfo di;
    const ap_status st = current_device(&di);
    if (st != AP_OK) return st;
    const Options o = options();
    const int64_t chunks = (4 * n) / chunk_bytes;
    const int64_t groups = chunks / cluster_size;
    const int64_t m = chunks % cluster_size;  // chunks of the short last group
    if (groups > 0) {
        const ap_status s1 = launch_exchange(di, o, in, out, groups, cluster_size, chunk_bytes, shift, false, stream);
        if (s1 != AP_OK) return s1;
    }
    if (m > 0) {
        // The short last group runs as one cluster of m CTAs.
        const int64_t off = groups * cluster_size * (chunk_bytes / 4);
        return launch_exchange(di, o, in + off, out + off, 1, static_cast<int>(m), chunk_bytes, shift, false, stream);
    }
    return AP_OK;
}

ap_status ap_masked_copy(const float* in, float* out, int64_t n_chunks, const int8_t* codes, int stages,
                         cudaStream_t stream) {
    if (!valid_stages(stages)) return AP_ERR_STAGES;
    if (n_chunks < 0 || n_chunks > kMaxElems / 4) return AP_ERR_SHAPE;
    if (n_chunks == 0) return AP_OK;
    if (in == nullptr || out == nullptr || codes == nullptr) return AP_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(in) & 15) || (reinterpret_cast<uintptr_t>(out) & 15)) return AP_ERR_ALIGN;
    if (in != out && overlap(in, 16 * n_chunks, out, 16 * n_chunks)) return AP_ERR_ALIAS;
    DeviceInfo di;
    const ap_status st = current_device(&di);
    if (st != AP_OK) return st;
    return launch_masked_copy(di, options(), in, out, n_chunks, reinterpret_cast<const signed char*>(codes), stages,
                              stream);
}

ap_status ap_autotune(ap_tune_op op, const float* in, float* out, int64_t n, int stages, int degree,
                      ap_ring_shape* chosen, cudaStream_t stream) {
    if (op != AP_TUNE_SCALE && op != AP_TUNE_ROW_ROLL && op != AP_TUNE_POLY) return AP_ERR_ARG;
    if (!valid_stages(stages)) return AP_ERR_STAGES;
    if (op == AP_TUNE_POLY && (degree < 0 || degree > AP_POLY_MAX_DEGREE)) return AP_ERR_ARG;
    if (n < (int64_t(1) << 16) || n > kMaxElems || n % 4 != 0) return AP_ERR_SHAPE;
    if (in == nullptr || out == nullptr || chosen == nullptr) return AP_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(in) & 15) || (reinterpret_cast<uintptr_t>(out) & 15)) return AP_ERR_ALIGN;
    if (overlap(in, 4 * n, out, 4 * n)) return AP_ERR_ALIAS;
    DeviceInfo di;
    const ap_status st = current_device(&di);
    if (st != AP_OK) return st;
    // probe operations: scale by 2 over 256-float tiles; the row shift of an
    // (n / 4) x 4 matrix by one row; Horner with coefficients 1 / (k + 2)
    std::vector<float> coeffs(static_cast<size_t>(degree) + 1);
    for (int k = 0; k <= degree; ++k) coeffs[k] = 1.0f / static_cast<float>(k + 2);
    OpArgs args{OP_SCALE, 2.0f, 0, nullptr};
    int64_t off = 0, unit = 256;
    if (op == AP_TUNE_ROW_ROLL) {
        args = OpArgs{OP_COPY, 1.0f, 0, nullptr};
        off = 4;
        unit = 4;
    } else if (op == AP_TUNE_POLY) {
        args = OpArgs{OP_POLY, 0.0f, degree, coeffs.data()};
        unit = 1;
    }
    RingShape best{};
    double gbs = 0.0;
    const ap_status r = autotune_ring(di, options(), args.kind, in, out, n, off, unit, stages, args, &best, &gbs, stream);
    if (r != AP_OK) return r;
    set_tuned_shape(di.device, args.kind, stages, best);
    chosen->stage_bytes = best.payload;
    chosen->ctas_per_sm = static_cast<int>(best.ctas_per_sm);
    chosen->consumer_warps = static_cast<int>(best.consumer_warps);
    chosen->stages_per_cta = static_cast<int>(best.run);
    chosen->consumer_groups = static_cast<int>(best.groups);
    chosen->gbs = gbs;
    return AP_OK;
}

ap_status ap_autotune_reset(void) {
    clear_tuned_shapes();
    return AP_OK;
}

ap_status ap_check(cudaStream_t stream) {
    DeviceInfo di;
    const ap_status st = current_device(&di);
    if (st != AP_OK) return st;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return AP_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, di.status, sizeof(word), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return AP_ERR_CUDA;
    if (cudaMemsetAsync(di.status, 0, sizeof(uint32_t), stream) != cudaSuccess) return AP_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return AP_ERR_CUDA;
    g_last_site = static_cast<int64_t>((word >> 8) & 0xff);
    if (word == 0) return AP_OK;
    return static_cast<ap_status>(word & 0xff);
}

ap_status ap_debug_set(int key, int64_t value) {
    if (value < 0) return AP_ERR_ARG;
    switch (key) {
        case AP_DBG_FORCE_PATH:
            if (value > 3) return AP_ERR_ARG;
            g_force_path = value;
            return AP_OK;
        case AP_DBG_EXPECT_TX_EXTRA:
            if (value > 4096) return AP_ERR_ARG;
            g_tx_extra = value;
            return AP_OK;
        case AP_DBG_TIMEOUT_NS: g_timeout_ns = value; return AP_OK;
        case AP_DBG_STAGE_BYTES:
            if (value != 0 && (value < 16 || value > 200 * 1024)) return AP_ERR_ARG;
            g_stage_bytes = value;
            return AP_OK;
        case AP_DBG_GRID: g_grid = value; return AP_OK;
        case AP_DBG_CTAS_PER_SM:
            if (value > 8) return AP_ERR_ARG;
            g_ctas_per_sm = value;
            return AP_OK;
        case AP_DBG_ROLL_STAGES:
            if (value != 0 && !valid_stages(static_cast<int>(value))) return AP_ERR_ARG;
            g_roll_stages = value;
            return AP_OK;
        case AP_DBG_CONSUMER_WARPS:
            if (value != 0 && value != 8 && value != 12 && value != 16) return AP_ERR_ARG;
            g_consumer_warps = value;
            return AP_OK;
        case AP_DBG_EXCHANGE_STORE:
            if (value > 2) return AP_ERR_ARG;
            g_ex_tma_store = value;
            return AP_OK;
        case AP_DBG_DEVICE_CHECKS:
            if (value > 1) return AP_ERR_ARG;
            g_device_checks = value;
            return AP_OK;
        case AP_DBG_EXCHANGE_GROUP:
            if (value != 0 && value != 1 && value != 2 && value != 4 && value != 8) return AP_ERR_ARG;
            g_ex_group = value;
            return AP_OK;
        case AP_DBG_STRICT_ALIGN:
            if (value > 1) return AP_ERR_ARG;
            g_strict_align = value;
            return AP_OK;
        case AP_DBG_EXCHANGE_LANES:
            if (value != 0 && value != 1 && value != 2 && value != 4) return AP_ERR_ARG;
            g_ex_lanes = value;
            return AP_OK;
        case AP_DBG_EXCHANGE_BATCH:
            if (value > 256) return AP_ERR_ARG;
            g_ex_batch = value;
            return AP_OK;
        case AP_DBG_EXCHANGE_SEND_SLOTS:
            if (value > 16 || (value & (value - 1)) != 0) return AP_ERR_ARG;  // 0, 1 or a power of two up to 16
            g_ex_send_slots = value;
            return AP_OK;
        case AP_DBG_RING_RUN:
            if (value > (int64_t(1) << 20)) return AP_ERR_ARG;
            g_ring_run = value;
            return AP_OK;
        case AP_DBG_CONSUMER_GROUPS:
            if (value > 3) return AP_ERR_ARG;
            g_consumer_groups = value;
            return AP_OK;
        default: return AP_ERR_ARG;
    }
}

int64_t ap_debug_get(int key) {
    const Options o = options();
    switch (key) {
        case AP_DBG_FORCE_PATH: return o.force_path;
        case AP_DBG_EXPECT_TX_EXTRA: return o.tx_extra;
        case AP_DBG_TIMEOUT_NS: return o.timeout_ns;
        case AP_DBG_STAGE_BYTES: return o.stage_bytes;
        case AP_DBG_GRID: return o.grid;
        case AP_DBG_CTAS_PER_SM: return o.ctas_per_sm;
        case AP_DBG_ROLL_STAGES: return o.roll_stages;
        case AP_DBG_CONSUMER_WARPS: return o.consumer_warps;
        case AP_DBG_EXCHANGE_STORE: return o.ex_tma_store;
        case AP_DBG_DEVICE_CHECKS: return o.device_checks;
        case AP_DBG_EXCHANGE_GROUP: return o.ex_group;
        case AP_DBG_STRICT_ALIGN: return o.strict_align;
        case AP_DBG_EXCHANGE_LANES: return o.ex_lanes;
        case AP_DBG_EXCHANGE_BATCH: return o.ex_batch;
        case AP_DBG_EXCHANGE_SEND_SLOTS: return o.ex_send_slots;
        case AP_DBG_RING_RUN: return o.ring_run;
        case AP_DBG_CONSUMER_GROUPS: return o.consumer_groups;
        case AP_DBG_LAST_PATH: return g_last_path.load();
        case AP_DBG_LAST_GRID: return g_last_grid.load();
        case AP_DBG_LAST_STAGE_ELEMS: return g_last_stage_elems.load();
        case AP_DBG_LAST_SMEM: return g_last_smem.load();
        case AP_DBG_LAST_STAGES: return g_last_stages.load();
        case AP_DBG_LAST_FLAGS: return g_last_flags.load();
        case AP_DBG_LAST_SITE: return g_last_site.load();
        case AP_DBG_LAST_RUN: return g_last_run.load();
        case AP_DBG_LAST_WARPS: return g_last_warps.load();
        case AP_DBG_LAST_GROUPS: return g_last_groups.load();
        case AP_DBG_LAST_CHAINS: return g_last_chains.load();
        default: return -1;
    }
}

ap_status ap_debug_scale_pages_async(const float* in, float* out, int64_t n_tiles, int64_t tile_elems, float alpha,
                                     cudaStream_t stream) {
    if (n_tiles < 0 || tile_elems < 1 || tile_elems > 1024) return AP_ERR_SHAPE;
    const int64_t n = n_tiles * tile_elems;
    if (n == 0) return AP_OK;
    if (in == nullptr || out == nullptr) return AP_ERR_NULL;
    if (!aligned4(in) || !aligned4(out)) return AP_ERR_ALIGN;
    if (in != out && overlap(in, 4 * n, out, 4 * n)) return AP_ERR_ALIAS;
    DeviceInfo di;
    const ap_status st = current_device(&di);
    if (st != AP_OK) return st;
    return launch_scale_pages_async(di, in, out, n_tiles, tile_elems, alpha, stream);
}

ap_status ap_debug_fma_probe(float* out, int64_t out_elems, int64_t iters, cudaStream_t stream) {
    if (out == nullptr) return AP_ERR_NULL;
    if (out_elems < 1 || iters < 1 || iters > (int64_t(1) << 24)) return AP_ERR_SHAPE;
    if (!aligned4(out)) return AP_ERR_ALIGN;
    DeviceInfo di;
    const ap_status st = current_device(&di);
    if (st != AP_OK) return st;
    return launch_fma_probe(di, out, out_elems, iters, stream);
}

ap_status ap_debug_fma_probe_horner(float* out, int64_t out_elems, int64_t iters, cudaStream_t stream) {
    if (out == nullptr) return AP_ERR_NULL;
    if (out_elems < 1 || iters < 1 || iters > (int64_t(1) << 20)) return AP_ERR_SHAPE;
    if (!aligned4(out)) return AP_ERR_ALIGN;
    DeviceInfo di;
    const ap_status st = current_device(&di);
    if (st != AP_OK) return st;
    return launch_fma_probe_horner(di, out, out_elems, iters, stream);
}

}  // extern "C"

namespace {

// Host emulation of one ring call's data movement (see asyncpipe_debug.h). It
// follows the kernel step by step: the producer's copies into a stage slot,
// then the consumers' reads and stores through the slot descriptor, using the
// same planning functions.
ap_status emulate_ring(const StreamGeom& g, const float* in_host, float* out_host) {
    const int64_t n = g.n;
    const uint64_t in_addr = g.in_addr, out_addr = g.out_addr;
    const uint64_t in_end = in_addr + 4 * static_cast<uint64_t>(n);
    unsigned char* slot = static_cast<unsigned char*>(std::malloc(g.slot_bytes));
    unsigned char* written = static_cast<unsigned char*>(std::malloc(g.slot_bytes));
    unsigned char* out_done = static_cast<unsigned char*>(std::calloc(static_cast<size_t>(n), 1));
    if (!slot || !written || !out_done) {
        std::free(slot);
        std::free(written);
        std::free(out_done);
        return AP_ERR_SHAPE;
    }
    const unsigned char* src_bytes = reinterpret_cast<const unsigned char*>(in_host);
    ap_status result = AP_OK;
    auto fail = [&]() { result = AP_ERR_SHAPE; };
    // copy global [ga, ga + bytes) into slot [dst, dst + bytes); bytes past
    // src_valid are zero (the zero-filling copies)
    auto gcopy = [&](uint32_t dst, uint64_t ga, uint32_t bytes, uint32_t src_valid) {
        if (ga < in_addr || ga + src_valid > in_end || dst + bytes > g.slot_bytes) return fail();
        for (uint32_t b = 0; b < bytes; ++b) {
            slot[dst + b] = b < src_valid ? src_bytes[ga - in_addr + b] : 0;
            written[dst + b] = 1;
        }
    };
    RegularStages reg;
    make_regular(g, &reg);
    for (int64_t j = 0; j < g.n_stages && result == AP_OK; ++j) {
        std::memset(slot, 0xA5, g.slot_bytes);
        std::memset(written, 0, g.slot_bytes);
        StagePlan sp;
        plan_stage(g, j, &sp);
        if (j >= 1 && j < reg.end) {
            // the producer's shortcut for a regular stage must give the same
            // copy and descriptor as the full plan
            SlotDesc d, full_d;
            const uint64_t src = regular_stage(g, reg, j, &d);
            make_slot_desc(sp, &full_d);
            const Span& s0 = sp.span[0];
            if (sp.nspans != 1 || s0.bulk_src != src || s0.bulk_bytes != reg.bytes || s0.bulk_dst != 0 ||
                s0.head_end != s0.x0 || s0.tail_begin != s0.x1 || std::memcmp(&d, &full_d, sizeof(d)) != 0) {
                fail();
                break;
            }
        }
        for (int k = 0; k < sp.nspans && result == AP_OK; ++k) {
            const Span& sn = sp.span[k];
            if (g.box_bytes != 0) {
                // tensor-map boxes: one 2-D box of whole lines of the line
                // view, or 1-D boxes from the span's first element (on a
                // 16-byte boundary; what lies past n arrives as zeros)
                if (sn.bulk_dst % 128) {
                    fail();
                    break;
                }
                if (sn.line_y >= 0) {
                    const int64_t e0 = g.line_r + sn.line_y * kFlatBoxElems;
                    if (g.line_h <= 0 || sp.nspans != 1 || e0 != sn.x0 || sn.line_y + g.line_h > g.line_rows ||
                        sn.bulk_bytes != 4 * kFlatBoxElems * g.line_h) {
                        fail();
                        break;
                    }
                    gcopy(sn.bulk_dst, in_addr + 4 * static_cast<uint64_t>(e0), sn.bulk_bytes, sn.bulk_bytes);
                    continue;
                }
                if (sn.x0 % 4 || sn.bulk_bytes % g.box_bytes ||
                    sn.bulk_bytes != boxes_for(g, sn.x1 - sn.x0) * g.box_bytes) {
                    fail();
                    break;
                }
                const int64_t e_end = sn.x0 + static_cast<int64_t>(sn.bulk_bytes / 4);
                for (int64_t e = sn.x0; e < e_end && result == AP_OK; ++e) {
                    const uint32_t dst = sn.bulk_dst + static_cast<uint32_t>(4 * (e - sn.x0));
                    gcopy(dst, in_addr + 4 * static_cast<uint64_t>(e < n ? e : 0), 4, e < n ? 4u : 0u);
                }
                continue;
            }
            for (int64_t x = sn.x0; x < sn.head_end; ++x)
                gcopy(sn.region + sn.lead + static_cast<uint32_t>(4 * (x - sn.x0)), in_addr + 4 * x, 4, 4);
            if (sn.tail_begin < sn.x1) {
                if (sn.tail_dst % 16) fail();
                gcopy(sn.tail_dst, in_addr + 4 * g.t_in, 16, static_cast<uint32_t>(4 * (n - g.t_in)));
            }
            if (sn.bulk_bytes) {
                if (sn.bulk_src % 16 || sn.bulk_dst % 16 || sn.bulk_bytes % 16) fail();
                gcopy(sn.bulk_dst, sn.bulk_src, sn.bulk_bytes, sn.bulk_bytes);
            }
        }
        if (result != AP_OK) break;
        // consumers: the kernel reads the descriptor the producer wrote
        SlotDesc dsc;
        make_slot_desc(sp, &dsc);
        auto read = [&](int64_t e) -> float {
            const uint32_t o = desc_offset_of_output(dsc, e);
            float v = 0.0f;
            if (o != smem_offset_of_output(sp, e) || o + 4 > g.slot_bytes || !written[o] || !written[o + 3]) {
                fail();
                return v;
            }
            std::memcpy(&v, slot + o, 4);
            return v;
        };
        auto store = [&](int64_t e, float v) {
            if (e < 0 || e >= n || out_done[e]) return fail();
            out_done[e] = 1;
            out_host[e] = v;
        };
        const int64_t ngroups = (dsc.e_end - dsc.e_al) >> 2;
        const uint32_t o0 = dsc.off0 + static_cast<uint32_t>(4 * (dsc.e_al - dsc.lo));
        for (int64_t q = 0; q < ngroups && result == AP_OK; ++q) {
            const int64_t e = dsc.e_al + 4 * q;
            if ((out_addr + 4 * static_cast<uint64_t>(e)) % 16) fail();
            if (dsc.mode == MODE_VEC) {
                const uint32_t o = o0 + static_cast<uint32_t>(16 * q);
                if (o % 16 || o != smem_offset_of_output(sp, e)) fail();
            } else if (dsc.mode == MODE_SHIFTED) {
                // the kernel reads two aligned words per group and picks the
                // four inputs out of them: check the words and the picks
                const uint32_t d = o0 & 15u;
                const uint32_t w = o0 - d + static_cast<uint32_t>(16 * q);
                const uint32_t region_end =
                    sp.span[0].region + static_cast<uint32_t>((4 * sp.len1 + 32 + 15) & ~int64_t(15));
                if (sp.nspans != 1 || d == 0 || d % 4 || w + 32 > region_end || w + 32 > g.slot_bytes) {
                    fail();
                    break;
                }
                for (int t = 0; t < 4; ++t) {
                    const uint32_t pick = w + d + 4u * static_cast<uint32_t>(t);
                    if (pick != smem_offset_of_output(sp, e + t)) fail();
                }
            } else if (sp.nspans != 2) {
                fail();  // the per-element path is only for stages that wrap
            }
            for (int t = 0; t < 4; ++t) store(e + t, read(e + t));
        }
        for (int64_t e = sp.lo; e < sp.e_al; ++e) store(e, read(e));
        for (int64_t e = sp.e_end; e < sp.hi; ++e) store(e, read(e));
        if (sp.e_al - sp.lo > 3 || sp.hi - sp.e_end > 3) fail();  // the kernel handles <= 3 + 3 scalars
    }
    for (int64_t e = 0; e < n && result == AP_OK; ++e)
        if (!out_done[e]) fail();
    std::free(slot);
    std::free(written);
    std::free(out_done);
    return result;
}

}  // namespace

extern "C" {

ap_status ap_debug_emulate_ring(const float* in_host, float* out_host, int64_t n, int64_t off, int in_mis,
                                int out_mis, int64_t stage_elems) {
    if (n < 0 || off < 0 || (n > 0 && off >= n)) return AP_ERR_SHAPE;
    if (in_mis < 0 || in_mis > 12 || in_mis % 4 || out_mis < 0 || out_mis > 12 || out_mis % 4) return AP_ERR_ALIGN;
    if (stage_elems < 4 || stage_elems % 4) return AP_ERR_SHAPE;
    if (n == 0) return AP_OK;
    if (in_host == nullptr || out_host == nullptr) return AP_ERR_NULL;
    // Pretend device addresses with the requested low bits.
    StreamGeom g;
    make_geom(&g, (uint64_t(1) << 40) + static_cast<uint64_t>(in_mis), (uint64_t(3) << 40) + static_cast<uint64_t>(out_mis),
              n, off, stage_elems);
    return emulate_ring(g, in_host, out_host);
}

ap_status ap_debug_emulate_ring_tensor(const float* in_host, float* out_host, int64_t rows, int64_t cols,
                                       int64_t shift, int64_t line_boxes, int64_t stage_elems) {
    if (rows < 1 || cols < 1 || cols > kMaxElems / rows) return AP_ERR_SHAPE;
    if (line_boxes != 0 && line_boxes != 1) return AP_ERR_ARG;
    if (stage_elems < kFlatBoxElems || stage_elems % kFlatBoxElems) return AP_ERR_SHAPE;
    const int64_t n = rows * cols;
    const int64_t s = ((shift % rows) + rows) % rows;
    if (!tensor_ok(uint64_t(1) << 40, uint64_t(3) << 40, n, s * cols)) return AP_ERR_ALIGN;
    if (in_host == nullptr || out_host == nullptr) return AP_ERR_NULL;
    StreamGeom g;
    make_geom_tensor(&g, uint64_t(1) << 40, uint64_t(3) << 40, n, s * cols, stage_elems, line_boxes != 0);
    return emulate_ring(g, in_host, out_host);
}

}  // extern "C"
