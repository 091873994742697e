/*
 * libasyncpipe tuning, fault-injection and inspection hooks.
 *
 * None of these is needed to use the library; they exist for tests and for
 * measuring the ring at other stage sizes. The pages define no API, so these
 * calls cite no passage. Settings are process-wide, apply to calls made
 * after they are set, and are read without locking (set them before
 * launching work from several threads).
 */
#ifndef ASYNCPIPE_DEBUG_H
#define ASYNCPIPE_DEBUG_H

#include <stdint.h>

#include "asyncpipe.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ap_debug_key {
    /* settable */
    AP_DBG_FORCE_PATH = 1,      /* (when 0, the environment variable AP_FORCE_PATH = auto, ring or
                                   bulk, small or cpasync, tensor, or 0..3, read once, decides) 0 auto; 1 always the ring (also for small row shifts);
                                   2 small one-CTA row shift when it fits; 3 ring with a tensor-map
                                   producer (cp.async.bulk.tensor) for ap_row_roll, ap_scale and
                                   ap_poly where input and output are 16-byte aligned and every span
                                   starts on a 16-byte boundary (shift * cols a multiple of 4, and
                                   rows * cols too for a nonzero shift): each stage one 2-D box of
                                   1 KiB lines of the input where it fits, else 1-D boxes of 256
                                   floats; the 1-D bulk producer otherwise */
    AP_DBG_EXPECT_TX_EXTRA = 2, /* bytes added to every stage's expected transaction count:
                                   the barrier then never completes and the consumers' bounded
                                   waits give up (fault injection; 0 = off) */
    AP_DBG_TIMEOUT_NS = 3,      /* limit of every kernel wait in ns (0 = default 2 s, or the
                                   AP_WAIT_TIMEOUT_NS environment variable) */
    AP_DBG_STAGE_BYTES = 4,     /* ring stage payload in bytes (0 = automatic) */
    AP_DBG_GRID = 5,            /* cap on the number of CTAs of ring kernels (0 = automatic) */
    AP_DBG_CTAS_PER_SM = 6,     /* resident ring CTAs per SM the grid is sized for (0 = 1) */
    AP_DBG_ROLL_STAGES = 7,     /* ring depth used by ap_row_roll (0 = 2) */
    AP_DBG_CONSUMER_WARPS = 8,  /* consumer warps per ring CTA: 8, 12 or 16 (0 = automatic) */
    AP_DBG_EXCHANGE_STORE = 9,  /* cluster exchange receiver: 0 automatic, 1 one thread handing each
                                   piece to a shared->global bulk copy, 2 receiver warps with 16-byte
                                   stores (AP_DBG_EXCHANGE_GROUP warps per piece) */
    AP_DBG_DEVICE_CHECKS = 11,  /* 1: ring kernels verify, before every stage, that each copy and each
                                   shared/global range they touch lies inside the caller's buffers and
                                   the stage slot; a violation makes ap_check report AP_ERR_SHAPE (site
                                   in AP_DBG_LAST_SITE) and nothing out of range is accessed */
    /* read-only: what the last call on this process launched */
    AP_DBG_LAST_PATH = 100,     /* 1 ring, 2 small row shift, 3 synchronous, 4 cluster exchange,
                                   5 masked copy, 6 the pages' asynchronous tiled scale */
    AP_DBG_LAST_GRID = 101,     /* CTAs launched */
    AP_DBG_LAST_STAGE_ELEMS = 102, /* elements per ring stage (chunk elements for exchange) */
    AP_DBG_LAST_SMEM = 103,     /* dynamic shared memory per CTA, bytes */
    AP_DBG_LAST_STAGES = 104,   /* ring depth */
    AP_DBG_EXCHANGE_GROUP = 13, /* cluster exchange, warp-store receiver: warps that store one piece
                                   together, 1, 2, 4 or 8 (the eight receiver warps take pieces in
                                   turn, 8 / value at once); 0 = automatic */
    AP_DBG_STRICT_ALIGN = 14,   /* 1: ap_scale, ap_poly and ap_row_roll return AP_ERR_ALIGN for
                                   buffers that are not 16-byte aligned instead of taking the
                                   cp.async edge fallback (checked before any CUDA call) */
    AP_DBG_EXCHANGE_LANES = 15, /* cluster exchange: threads that load and threads that push, 1, 2
                                   or 4 each, lane l taking items l, l + lanes, ... (reduced to a
                                   divisor of the ring depth); 0 = automatic */
    AP_DBG_EXCHANGE_BATCH = 16, /* cluster exchange, batched form (one tensor-map box gathers a rank's
                                   chunk, or sub-block, from several consecutive groups): 0 automatic
                                   (sub-blocks under 8 KiB), 1 never, 2..256 groups per item (rounded
                                   so an item is whole 128-byte units); applies where a sub-block is at
                                   most 256 floats or a multiple of 256 */
    AP_DBG_EXCHANGE_SEND_SLOTS = 17, /* cluster exchange, split rings: 2, 4, 8 or 16 send buffers, each
                                   freed as soon as its piece has landed, beside as many receive slots
                                   as fit (a multiple of it, and of the cluster size in the
                                   all-to-all; where none fits, one ring depth); 1 never split;
                                   0 automatic (the all-to-all splits where its ring depth is a power
                                   of two, with that many send buffers) */
    AP_DBG_RING_RUN = 18,       /* schedule of the ring calls and of ap_masked_copy: 0 automatic; 1 a
                                   persistent grid (SMs x CTAs per SM CTAs, CTA b taking stages b,
                                   b + grid, ...); r = 2 .. 2^20 every CTA takes r consecutive stages
                                   (masked copy: of 1024 chunks) and as many CTAs launch as that
                                   takes. AP_DBG_GRID, when set, implies the persistent grid for the
                                   ring calls */
    AP_DBG_CONSUMER_GROUPS = 19, /* ap_poly: consumer groups that take stages in turn (group g the
                                   stages g, g + groups, ...): 0 automatic, or 1, 2, 3 where the count
                                   divides the consumer warps (16: 1 or 2; 12: 1, 2 or 3; 8: 1) and the
                                   ring depth; other counts make ap_poly return AP_ERR_ARG */
    AP_DBG_LAST_SITE = 106,     /* where the error ap_check last reported was raised (kernel site code) */
    AP_DBG_LAST_RUN = 107,      /* ring: consecutive stages per CTA, 0 for the persistent grid */
    AP_DBG_LAST_WARPS = 108,    /* ring: consumer warps per CTA */
    AP_DBG_LAST_GROUPS = 109,   /* ring: consumer groups taking stages in turn */
    AP_DBG_LAST_CHAINS = 110,   /* ap_poly: Horner chains a consumer thread runs per round in whole
                                   aligned stages (16, 24 or 32); 0 for other calls */
    AP_DBG_LAST_FLAGS = 105     /* bit 0: some stage used cp.async edge copies (misaligned head
                                   or unaligned tail); bit 1: some stage used the scalar
                                   shared-memory path (input/output alignments differ or wrap);
                                   bit 2: the tensor-map producer ran; bit 3: with the line
                                   view (2-D boxes of whole stages) set up beside the flat map */
} ap_debug_key;

/* Set a settable key. AP_ERR_ARG for an unknown key or a negative value. */
ap_status ap_debug_set(int key, int64_t value);

/* Read any key; -1 for an unknown key. */
int64_t ap_debug_get(int key);

/*
 * The pages' own asynchronous tiled scale, kept as a measured baseline: a
 * two-stage double buffer of one tile per CTA, every thread copying its own
 * 4-byte element with cp.async, commit, wait for the older group, CTA
 * barrier, compute, store ("CUDA Async Copy and Pipeline Guide",
 * Implementation Comparison, "After" kernel; CTA b takes tiles b, b + grid,
 * ...). Same arguments and result as ap_scale; tile_elems at most 1024.
 */
ap_status ap_debug_scale_pages_async(const float* in, float* out, int64_t n_tiles, int64_t tile_elems, float alpha,
                                     cudaStream_t stream);

/*
 * FP32 FMA throughput probe: each thread of a grid sized to the device runs
 * 32 independent fmaf chains of `iters` steps on registers only and writes
 * one float (the chains' sum) to out[thread]; the number of threads launched
 * is min(out_elems, SMs * 1024) rounded down to whole CTAs of 512. Timing a
 * call gives the achievable fma rate that bounds ap_poly at high degree.
 * out is a device array of out_elems floats.
 */
ap_status ap_debug_fma_probe(float* out, int64_t out_elems, int64_t iters, cudaStream_t stream);

/*
 * As ap_debug_fma_probe, in the operand pattern of ap_poly's Horner loop:
 * 24 chains a thread, each step fmaf(p_t, x_t, c_k) with a distinct x_t per
 * chain and the coefficient c_k read from shared memory four at a time, 128
 * steps per iteration. One CTA of 512 threads per SM; the number of threads
 * launched is min(out_elems, SMs * 512) rounded down to whole CTAs, each
 * running iters * 128 * 24 fmaf and writing one float to out[thread]. iters
 * at most 2^20 (else AP_ERR_SHAPE). The rate it reaches is the compute roof
 * of a polynomial whose coefficients are only known at run time.
 */
ap_status ap_debug_fma_probe_horner(float* out, int64_t out_elems, int64_t iters, cudaStream_t stream);

/*
 * Host emulation of one ring call's data movement, for checking the
 * kernel's index arithmetic without a GPU. It runs the same tile planning
 * code the kernel runs (stage ranges, bulk spans, cp.async edges, shared
 * memory offsets) on host arrays that stand for device buffers located at
 * byte addresses whose low four bits are in_mis and out_mis, and performs
 * out[e] = in[(e + off) mod n]. It checks every bulk copy (16-byte aligned
 * source and destination, size a multiple of 16, inside the input), every
 * cp.async edge copy, every shared-memory access (inside its stage slot) and
 * every vector store (16-byte aligned), and returns AP_ERR_SHAPE at the
 * first violation, AP_OK otherwise.
 *  in_host, out_host  n floats each (host memory).
 *  in_mis, out_mis    0, 4, 8 or 12.
 *  stage_elems        elements per stage (multiple of 4, >= 4).
 */
ap_status ap_debug_emulate_ring(const float* in_host, float* out_host, int64_t n, int64_t off,
                                int in_mis, int out_mis, int64_t stage_elems);

/*
 * As ap_debug_emulate_ring, for the tensor-map producer:
 * B[i, :] = A[(i + shift) mod rows, :] for a rows x cols matrix at 16-byte
 * aligned addresses (shift 0 is the plain stream of scale and poly). Spans
 * load as whole 1-D boxes of 256 floats of the flat input (floats past its
 * end arrive as zeros, as the copy engine writes them); with line_boxes = 1 a
 * stage whose single span starts on a line of the line view (1 KiB lines from
 * element (shift mod rows) * cols mod 256) and stays inside its whole lines
 * loads as one 2-D box instead. (shift mod rows) * cols must be a multiple
 * of 4, and rows * cols too when that shift is not 0 (else AP_ERR_ALIGN);
 * stage_elems a multiple of 256; line_boxes 0 or 1 (else AP_ERR_ARG).
 * Checks every box (first coordinate on a 16-byte boundary, a 2-D box inside
 * the line view, destination 128-byte aligned and inside the slot) and every
 * consumer access.
 */
ap_status ap_debug_emulate_ring_tensor(const float* in_host, float* out_host, int64_t rows, int64_t cols,
                                       int64_t shift, int64_t line_boxes, int64_t stage_elems);

#ifdef __cplusplus
}
#endif

#endif /* ASYNCPIPE_DEBUG_H */
