/*
 * libasyncpipe: asynchronous global->shared tile streaming on GB300 (sm_103a).
 *
 * Every streaming call runs one persistent CUDA kernel whose CTAs walk a
 * sequence of tiles. A producer warp loads the next tiles from global memory
 * into a ring of shared-memory stages with bulk asynchronous copies
 * (cp.async.bulk, completion tracked by an mbarrier with expected transaction
 * bytes); consumer warps wait for a stage, compute on it from shared memory,
 * store the result with coalesced 16-byte stores and release the stage. The
 * load of tile t+1 therefore overlaps the compute and store of tile t, which
 * is the point of "Asynchronous Data Movement" (knowledge-base page, opening
 * section and section Double buffering): a plain tiled loop alternates load
 * and compute instead of overlapping them.
 *
 * Conventions shared by every call:
 *  - Pointers named in/out/A/B point to float32 data owned by the caller that
 *    the device can access: device memory, or pinned host memory mapped into
 *    the device's address space (as cudaHostAlloc memory is under unified
 *    addressing), which the kernels then read and write over the host link.
 *    They must be 4-byte aligned (AP_ERR_ALIGN otherwise). Any
 *    other misalignment is not an error: the bulk path needs 16-byte aligned
 *    addresses, so the few elements before the first and after the last
 *    16-byte boundary of a buffer are fetched with 4-byte cp.async.ca and one
 *    zero-filling 16-byte cp.async.cg instead ("Asynchronous Data Movement",
 *    section Alignment requirements; "Asynchronous Copies", section A
 *    Global-to-Shared Copy). No call reads or writes a byte outside the
 *    caller's ranges.
 *  - `stream` is a CUDA stream (0 = the legacy default stream). Calls are
 *    stream-ordered and return as soon as the kernel is queued. Argument
 *    errors are returned at once, before any CUDA call; errors raised inside
 *    a kernel (a bounded wait that gave up) are reported by ap_check().
 *  - A call with zero elements is a no-op that returns AP_OK and touches no
 *    pointer.
 *  - The streaming calls (scale, sync scale, row shift, poly, the cluster
 *    calls, the masked copy) may be captured into a CUDA graph on a capturing
 *    stream once each has run on the device outside capture (the first call
 *    sets one-time kernel attributes); a replay runs them with the pointers
 *    and sizes of the capture. ap_check synchronises its stream and
 *    ap_autotune times launches, so neither may be captured.
 *  - The library allocates no device memory. Its only device state is one
 *    status word per device, a static __device__ variable of the library.
 *  - Runs only on compute capability 10.3 devices (GB300):
 *    AP_ERR_UNSUPPORTED_DEVICE elsewhere.
 */
#ifndef ASYNCPIPE_H
#define ASYNCPIPE_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ap_status {
    AP_OK = 0,
    AP_ERR_NULL = 1,               /* a required pointer is NULL */
    AP_ERR_SHAPE = 2,              /* negative or inconsistent sizes, size overflow */
    AP_ERR_ALIGN = 3,              /* pointer not aligned as the call requires */
    AP_ERR_ALIAS = 4,              /* input and output overlap in a way the call forbids */
    AP_ERR_STAGES = 5,             /* ring depth outside [AP_MIN_STAGES, AP_MAX_STAGES] */
    AP_ERR_CLUSTER = 6,            /* cluster size not supported by the call */
    AP_ERR_SMEM = 7,               /* the requested tiles do not fit in shared memory */
    AP_ERR_CUDA = 8,               /* a CUDA runtime call failed (launch, sync, attribute) */
    AP_ERR_DEVICE_TIMEOUT = 9,     /* a kernel wait gave up (reported by ap_check) */
    AP_ERR_UNSUPPORTED_DEVICE = 10,/* current device is not compute capability 10.3 */
    AP_ERR_ARG = 11                /* other invalid argument (degree, debug key) */
} ap_status;

#define AP_MIN_STAGES 2
#define AP_MAX_STAGES 6
#define AP_POLY_MAX_DEGREE 1023
#define AP_MAX_CLUSTER 8
#define AP_MAX_CLUSTER_NONPORTABLE 16

/*
 * ap_scale: out[i] = alpha * in[i] for i < n_tiles * tile_elems.
 * Source: "CUDA Async Copy and Pipeline Guide", section Implementation
 * Comparison: the "After" kernel double-buffers 256-float tiles through a
 * two-stage pipeline and stores 2.0f times each element.
 *  in, out     device float32 arrays of n_tiles * tile_elems elements. They may
 *              be the same array (in place); any other overlap is AP_ERR_ALIAS.
 *  n_tiles     number of tiles (>= 0); tile_elems elements per tile (>= 1).
 *              Tiles are the logical unit; a ring stage holds a whole number
 *              of tiles where the tile size allows, which does not change
 *              the result (the operation is elementwise).
 *  alpha       one fp32 multiply per element, rounded to nearest even.
 *  stages      ring depth, AP_MIN_STAGES..AP_MAX_STAGES (the pipeline's
 *              number of shared-memory buffers).
 */
ap_status ap_scale(const float* in, float* out, int64_t n_tiles, int64_t tile_elems,
                   float alpha, int stages, cudaStream_t stream);

/*
 * ap_scale_sync: the same result as ap_scale, computed by the synchronous
 * baseline: one CTA per tile; every thread loads its elements into shared
 * memory, the block synchronises, multiplies, synchronises, stores.
 * Source: "CUDA Async Copy and Pipeline Guide", section Implementation
 * Comparison, the "Before" kernel. Kept as the baseline the pipelined kernel
 * is measured against. Arguments as ap_scale; tile_elems * 4 bytes must fit
 * in one CTA's shared memory (AP_ERR_SMEM otherwise).
 */
ap_status ap_scale_sync(const float* in, float* out, int64_t n_tiles, int64_t tile_elems,
                        float alpha, cudaStream_t stream);

/*
 * ap_row_roll: B[i, :] = A[(i + shift) mod rows, :] for a row-major
 * rows x cols float32 matrix.
 * Source: "Asynchronous Copies" (TVM TIRx guide), section A Global-to-Shared
 * Copy: each thread copies one row into shared memory and reads the next
 * thread's row; shift = 1 reproduces that example (torch.roll(A, -1, 0)).
 *  A, B        device arrays of rows * cols floats; they must not overlap.
 *  rows, cols  >= 0 (an empty matrix is a no-op).
 *  shift       any value; reduced modulo rows into [0, rows).
 * Small matrices (at most 32 KiB) run in one CTA that copies the matrix with
 * 16-byte cp.async.cg (commit group, wait group, CTA barrier) and reads the
 * shifted rows from shared memory. Larger ones stream through the ring: the
 * tile of output rows [r0, r1) loads input rows [r0 + shift, r1 + shift),
 * i.e. its own rows plus the halo that belongs to the next tile, wrapping to
 * row 0 with a second bulk copy at the end of the matrix.
 */
ap_status ap_row_roll(const float* A, float* B, int64_t rows, int64_t cols, int64_t shift,
                      cudaStream_t stream);

/*
 * ap_poly: out[i] = p(in[i]) with p(x) = sum_k coeffs[k] x^k, evaluated by
 * Horner's rule with one fmaf per step: p = c[K]; p = fmaf(p, x, c[k]) for
 * k = K-1 .. 0. Degree K sets the arithmetic intensity (K fma per element,
 * 8 bytes of traffic per element).
 * Source: the per-tile compute is left open by "Asynchronous Data Movement"
 * (section Double buffering, "compute on tile[cur]"), and "CUDA Async Copy
 * and Pipeline Guide" (Common Performance Issues) names too little work per
 * copy as a pitfall; the Horner chain is this library's tunable compute.
 *  in, out     as ap_scale (in place allowed), n elements (>= 0).
 *  coeffs      HOST array of degree + 1 floats, lowest power first; copied
 *              into the kernel parameters, so it may be freed on return.
 *  degree      0..AP_POLY_MAX_DEGREE (AP_ERR_ARG otherwise).
 *  stages      ring depth as ap_scale.
 */
ap_status ap_poly(const float* in, float* out, int64_t n, const float* coeffs, int degree,
                  int stages, cudaStream_t stream);

/*
 * ap_cluster_exchange: shared-memory hand-off between the CTAs of a
 * thread-block cluster. The input is cut into chunks of chunk_bytes; every
 * cluster_size consecutive chunks form one group. For each group a cluster
 * of cluster_size CTAs loads the group (CTA rank r loads chunk r into its own
 * shared memory), rank r bulk-copies its chunk into the shared memory of rank
 * (r - 1) mod cluster_size (cp.async.bulk.shared::cluster, completed on the
 * receiver's transaction barrier that expects chunk_bytes), and every CTA
 * stores what it received:
 *     out chunk (g * cs + r) = in chunk (g * cs + (r + 1) mod cs).
 * Source: "Asynchronous Copies" (TVM TIRx guide), section Copies between
 * CTAs. The direction (rank r receives from rank r + 1) follows the same
 * page's row shift, where each thread reads its neighbour's row.
 *  in, out       device arrays of n floats, 16-byte aligned (AP_ERR_ALIGN),
 *                not overlapping (AP_ERR_ALIAS).
 *  n             >= 0; n * 4 must be a multiple of cluster_size * chunk_bytes.
 *  cluster_size  1, 2, 4 or 8 (AP_ERR_CLUSTER otherwise).
 *  chunk_bytes   multiple of 16, >= 16; two chunks per ring stage must fit in
 *                shared memory (AP_ERR_SMEM otherwise, about 113 KiB max).
 *                Chunks under 8 KiB move in batches: one tensor-map box gathers
 *                a rank's chunk from several consecutive groups (chunks of at
 *                most 256 floats or a multiple of 256).
 */
ap_status ap_cluster_exchange(const float* in, float* out, int64_t n, int cluster_size,
                              int64_t chunk_bytes, cudaStream_t stream);

/*
 * ap_cluster_exchange_ex: the cluster hand-off generalised to any cluster
 * size from 1 to 16, any distance within the cluster, and a short last group.
 * The input is cut into chunks of chunk_bytes; consecutive runs of
 * cluster_size chunks form groups, the last group holding the
 * m = chunks mod cluster_size leftover chunks when that is not zero. Within a
 * group of m members (m = cluster_size for whole groups) member r receives
 * member (r + shift) mod m:
 *     out chunk (g * cs + r) = in chunk (g * cs + (r + shift) mod m).
 * shift = 1 with whole groups is ap_cluster_exchange. Source: "Asynchronous
 * Copies" (TVM TIRx guide), section Copies between CTAs, a CTA copying a
 * chunk into another CTA of its cluster; the pages fix neither the distance
 * nor how a short last cluster behaves, and this call defines both.
 *  in, out       as ap_cluster_exchange (16-byte aligned, not overlapping).
 *  n             >= 0; n * 4 must be a multiple of chunk_bytes (AP_ERR_SHAPE).
 *  cluster_size  1..16 (AP_ERR_CLUSTER otherwise; sizes above 8 use the
 *                non-portable cluster attribute and return AP_ERR_CLUSTER if
 *                the device cannot place such a cluster).
 *  chunk_bytes   as ap_cluster_exchange.
 *  shift         any value, reduced modulo the group's member count.
 * A short last group runs as a second launch with a cluster of m CTAs.
 */
ap_status ap_cluster_exchange_ex(const float* in, float* out, int64_t n, int cluster_size,
                                 int64_t chunk_bytes, int64_t shift, cudaStream_t stream);

/*
 * ap_cluster_all_to_all: every CTA of a cluster sends a piece of its chunk to
 * every CTA of the cluster. The input is cut into chunks of chunk_bytes and
 * every cluster_size consecutive chunks form one group; each chunk is
 * cluster_size equal sub-blocks of B = chunk_bytes / cluster_size bytes.
 * CTA rank r of the group's cluster loads chunk r, bulk-copies its sub-block j
 * into the shared memory of rank j (cp.async.bulk.shared::cluster, completed
 * on rank j's transaction barrier, which expects the bytes of every sender),
 * and each CTA stores what it received:
 *     out chunk (g * cs + d), sub-block r = in chunk (g * cs + r), sub-block d,
 * the block transpose of each group's cs x cs sub-blocks. Source: "Asynchronous
 * Copies" (TVM TIRx guide), section Copies between CTAs (a CTA copies shared
 * memory into another CTA of its cluster; the receiver waits on its own
 * transaction barrier); the pages describe one sender and one receiver, and
 * this call extends the pattern to all pairs of the cluster.
 *  in, out       device arrays of n floats, 16-byte aligned (AP_ERR_ALIGN),
 *                not overlapping (AP_ERR_ALIAS).
 *  n             >= 0; n * 4 must be a multiple of cluster_size * chunk_bytes
 *                (AP_ERR_SHAPE).
 *  cluster_size  1..16 (AP_ERR_CLUSTER otherwise; sizes above 8 use the
 *                non-portable cluster attribute and return AP_ERR_CLUSTER if
 *                the device cannot place such a cluster). 1 is a plain copy.
 *  chunk_bytes   a multiple of 16 * cluster_size (AP_ERR_SHAPE), so that every
 *                sub-block is whole 16-byte units.
 */
ap_status ap_cluster_all_to_all(const float* in, float* out, int64_t n, int cluster_size,
                                int64_t chunk_bytes, cudaStream_t stream);

/*
 * ap_masked_copy: predicated / zero-filling copy of 16-byte chunks. For chunk
 * k (floats 4k .. 4k+3) with code c = codes[k]:
 *     0..16  the first c bytes of in chunk k are copied, the remaining
 *            16 - c bytes of out chunk k are set to zero (16: plain copy);
 *     -2     out chunk k is set to zero, the source is not read;
 *     -1     out chunk k is left unchanged (the copy is predicated off).
 * Source: "Asynchronous Copies" (TVM TIRx guide), section A Global-to-Shared
 * Copy, which names exactly these three forms of the 16-byte copy (a false
 * predicate, a source size, an ignored source). The chunks stream through a
 * per-thread cp.async pipeline of `stages` commit groups into shared memory
 * and out with 16-byte stores; at depths 2-4 each CTA takes one pipeline's
 * worth of consecutive stages (1024 chunks a stage), at 5-6 a persistent
 * grid of two CTAs a SM walks them.
 *  in, out     device arrays of 4 * n_chunks floats, 16-byte aligned
 *              (AP_ERR_ALIGN); in == out is allowed, other overlap is not.
 *  n_chunks    >= 0.
 *  codes       DEVICE array of n_chunks int8 codes. A code outside -2..16
 *              leaves its chunk unchanged and makes ap_check report AP_ERR_ARG.
 *  stages      commit groups in flight per thread, AP_MIN_STAGES..AP_MAX_STAGES.
 */
ap_status ap_masked_copy(const float* in, float* out, int64_t n_chunks, const int8_t* codes, int stages,
                         cudaStream_t stream);

/*
 * ap_autotune: choose the ring's stage size, schedule and consumer warps by
 * timing them on this device. Source: "CUDA Async Copy and Pipeline Guide",
 * FAQ: more stages hide more latency but use more shared memory, and the
 * sweet spot is found by profiling. For the given ring depth the call runs
 * the operation over in/out for every stage size from 8 to 96 KiB, under
 * both schedules: a persistent grid of 1-4 CTAs per SM (whose shared memory
 * fits), and CTAs that each take a run of depth, 2 x depth or 4 x depth
 * consecutive stages, and the built-in shape for that operation and depth.
 * Three timed launches each (CUDA events on `stream`, median); it keeps the
 * fastest and installs it:
 * later calls of that operation with that depth on this device use it
 * instead of the built-in defaults (explicit ap_debug_set settings still
 * win). Blocks until the timing is done.
 *  op      AP_TUNE_SCALE (ap_scale, alpha 2, 256-float tiles), AP_TUNE_ROW_ROLL
 *          (ap_row_roll of an (n / 4) x 4 matrix by one row), AP_TUNE_POLY
 *          (ap_poly of the given degree; the choice is kept for every degree).
 *  in, out device buffers of n floats, 16-byte aligned, not overlapping. out
 *          is overwritten; in is only read.
 *  n       elements, a multiple of 4, at least 65536 (larger than the L2,
 *          256 MiB or more, gives the choice that holds for streaming work).
 *  chosen  receives the chosen shape and its rate (8 bytes per element / time).
 * ap_autotune_reset forgets every installed choice.
 */
typedef enum ap_tune_op { AP_TUNE_SCALE = 1, AP_TUNE_ROW_ROLL = 2, AP_TUNE_POLY = 3 } ap_tune_op;

typedef struct ap_ring_shape {
    int64_t stage_bytes; /* payload of one ring stage */
    int ctas_per_sm;     /* persistent grid: resident CTAs per SM the grid is sized for */
    int consumer_warps;  /* consumer warps per CTA */
    int stages_per_cta;  /* 0: persistent grid; r: every CTA takes r consecutive stages */
    int consumer_groups; /* ap_poly: consumer groups taking stages in turn (1-3; 0: two for 16
                            warps at even depths of 4 or more, else one) */
    double gbs;          /* measured rate of the chosen shape, GB/s */
} ap_ring_shape;

ap_status ap_autotune(ap_tune_op op, const float* in, float* out, int64_t n, int stages, int degree,
                      ap_ring_shape* chosen, cudaStream_t stream);
ap_status ap_autotune_reset(void);

/*
 * ap_check: waits for `stream`, then returns and clears the device status
 * word of the current device: AP_ERR_DEVICE_TIMEOUT if a kernel's bounded
 * wait gave up since the last check, AP_ERR_ARG if ap_masked_copy met a bad
 * code, AP_ERR_SHAPE if the device-checked ring (asyncpipe_debug.h) found an
 * access out of range, AP_ERR_CUDA if the stream reported an error, AP_OK
 * otherwise. The status word is shared by all streams of the
 * device (the first error since the last check wins).
 */
ap_status ap_check(cudaStream_t stream);

/* ap_status_string: a static, human-readable name for a status code. */
const char* ap_status_string(ap_status s);

#ifdef __cplusplus
}
#endif

#endif /* ASYNCPIPE_H */
