// The streaming ring: a warp-specialised kernel in which one producer thread
// keeps up to S stages of input in flight with bulk asynchronous copies while
// the consumer warps (8 for the data-movement ops; 16 or 12 for the
// polynomial, in one to three groups that take stages in turn) compute on the
// oldest landed stage and store it.
//
// Protocol per ring slot s (two mbarriers, "Asynchronous Data Movement",
// section Barriers and pipelines: acquire, commit, wait, release):
//   producer: wait empty[s]            (acquire: the slot's previous tile is consumed)
//             cp.async edge copies, cp.async.mbarrier.arrive(full[s])
//             arrive.expect_tx(full[s], bulk bytes) + cp.async.bulk into the slot
//                                      (commit: the barrier now tracks the copies)
//   consumer: wait full[s]             (wait: every byte of the tile has landed)
//             ld.shared -> compute -> 16-byte st.global
//             arrive empty[s]          (release)
// The producer runs up to S tiles ahead, so the load of tile t+1 overlaps the
// compute and store of tile t ("Asynchronous Data Movement", section Double
// buffering; "CUDA Async Copy and Pipeline Guide", section Implementation
// Comparison, "After" kernel).
//
// GB300 choices that differ from the pages' 256-float, one-block sketch:
// a stage holds tens of KiB (many of the pages' tiles) so that each SM keeps
// enough bytes in flight to cover HBM latency; memory-bound work runs as CTAs
// that each take a short run of consecutive stages, started in index order so
// the grid streams one narrow window of memory, and fma-bound work as a
// persistent grid (CTA b takes stages b, b + grid, ...); the copy is a single
// bulk-copy instruction per stage issued by one thread (the TMA engine
// generates the addresses, "Asynchronous Data Movement", section The Tensor
// Memory Accelerator) instead of every thread copying a few bytes.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <type_traits>

#include "device_common.cuh"
#include "internal.h"

namespace ap {
namespace {


// Each op: stage() copies whatever the op reads from shared memory (only
// the polynomial's coefficients) before the ring starts; apply() transforms
// N values held in registers.
// kGroups: 16-byte groups a consumer thread keeps in flight per iteration
// (4 groups = 16 values; the polynomial wants 8, i.e. 32 independent Horner
// chains, where registers allow).
struct OpCopyDev {
    static constexpr int kGroups = 4;
    __device__ __forceinline__ void stage(float*, int, int) const {}
    template <int N>
    __device__ __forceinline__ void apply(float (&)[N], const float*) const {}
};

struct OpScaleDev {
    static constexpr int kGroups = 4;
    float alpha;
    __device__ __forceinline__ void stage(float*, int, int) const {}
    template <int N>
    __device__ __forceinline__ void apply(float (&v)[N], const float*) const {
#pragma unroll
        for (int t = 0; t < N; ++t) v[t] = alpha * v[t];
    }
};

// Horner's rule, one fmaf per step, N independent chains per thread so the
// FMA pipe sees N-way instruction-level parallelism. The coefficients are
// read from shared memory four at a time (one 16-byte broadcast load per four
// fma steps per chain), highest power first.
struct OpPolyDev {
    static constexpr int kGroups = 8;
    int degree;
    int six_groups;  // 1: 16 consumer warps take six groups (24 chains) a round
    float c[AP_POLY_MAX_DEGREE + 1];
    __device__ __forceinline__ void stage(float* cs, int tid, int nthreads) const {
        for (int k = tid; k <= degree; k += nthreads) cs[k] = c[k];
        if (tid < 4) cs[tid - 4] = 0.0f;
    }
    // Four Horner steps with the coefficients of one aligned 16-byte word,
    // highest power (q.w) first.
    template <int N>
    __device__ __forceinline__ static void steps4(float (&p)[N], const float (&v)[N], const float4 q) {
#pragma unroll
        for (int t = 0; t < N; ++t) p[t] = fmaf(p[t], v[t], q.w);
#pragma unroll
        for (int t = 0; t < N; ++t) p[t] = fmaf(p[t], v[t], q.z);
#pragma unroll
        for (int t = 0; t < N; ++t) p[t] = fmaf(p[t], v[t], q.y);
#pragma unroll
        for (int t = 0; t < N; ++t) p[t] = fmaf(p[t], v[t], q.x);
    }
    template <int N>
    __device__ __forceinline__ void apply(float (&v)[N], const float* cs) const {
        const float top = cs[degree];
        if (degree == 0) {
#pragma unroll
            for (int t = 0; t < N; ++t) v[t] = top;
            return;
        }
        // The first step reads c[K] straight from `top`, so no chain starts
        // with a register copy.
        float p[N];
        const float c1 = cs[degree - 1];
#pragma unroll
        for (int t = 0; t < N; ++t) p[t] = fmaf(top, v[t], c1);
        int k = degree - 2;
        {
            // Scalar steps until k + 1 is a multiple of 4: r <= k + 1 of
            // them, written out rather than looped (degree 128: +0.1-0.2 %,
            // degree 32 at depth 6 +0.9 %).
            const int r = (k + 1) & 3;
            if (r >= 3) {
                const float ck = cs[k];
                --k;
#pragma unroll
                for (int t = 0; t < N; ++t) p[t] = fmaf(p[t], v[t], ck);
            }
            if (r >= 2) {
                const float ck = cs[k];
                --k;
#pragma unroll
                for (int t = 0; t < N; ++t) p[t] = fmaf(p[t], v[t], ck);
            }
            if (r >= 1) {
                const float ck = cs[k];
                --k;
#pragma unroll
                for (int t = 0; t < N; ++t) p[t] = fmaf(p[t], v[t], ck);
            }
        }
        // Steps k down to 0 from whole aligned 16-byte words (k + 1 is a
        // multiple of four), each word loaded ahead of its use; a load past
        // c[0] reads the four zero floats staged below it. The loop's shape
        // is chosen by chain count, each form measured at degrees 32 and 128
        // against the others (GB300, 2^30 floats): with 16 chains one word a
        // trip; with 24, and with 32 below degree 64, an odd word alone and
        // then two words a trip with one exit test; with 32 from degree 64,
        // the odd words one at a time and then four a trip (0.84 -> 0.856 of
        // the register-only fma rate at ring depth 6). The same change to
        // another chain count cost it 1-5 %.
        if (k >= 3) {
            const float4* w = reinterpret_cast<const float4*>(cs + k - 3);
            const float4* const w0 = reinterpret_cast<const float4*>(cs);
            if constexpr (N >= 32) {
                if (degree >= 64) {
                    for (int r = ((k + 1) >> 2) & 3; r > 0; --r) {
                        const float4 q = *w;
                        --w;
                        steps4(p, v, q);
                    }
                    if (w >= w0) {
                        float4 q0 = w[0];
                        do {
                            const float4 q1 = w[-1];
                            steps4(p, v, q0);
                            const float4 q2 = w[-2];
                            steps4(p, v, q1);
                            const float4 q3 = w[-3];
                            steps4(p, v, q2);
                            q0 = w[-4];
                            steps4(p, v, q3);
                            w -= 4;
                        } while (w >= w0);
                    }
#pragma unroll
                    for (int t = 0; t < N; ++t) v[t] = p[t];
                    return;
                }
            }
            if constexpr (N >= 24) {
                if (((k + 1) >> 2) & 1) {
                    const float4 q = *w;
                    --w;
                    steps4(p, v, q);
                }
                if (w >= w0) {
                    float4 q0 = w[0];
                    do {
                        const float4 q1 = w[-1];
                        steps4(p, v, q0);
                        q0 = w[-2];
                        steps4(p, v, q1);
                        w -= 2;
                    } while (w >= w0);
                }
            } else {
                float4 q = *w;
#pragma unroll 2
                for (; k >= 3; k -= 4) {
                    const float4 next = *reinterpret_cast<const float4*>(cs + k - 7);
                    steps4(p, v, q);
                    q = next;
                }
            }
        }
#pragma unroll
        for (int t = 0; t < N; ++t) v[t] = p[t];
    }
};

template <class Op>
struct RingParams {
    CUtensorMap tmap;        // tensor-map mode: the input as a flat 1-D tensor (boxes of 256 floats)
    CUtensorMap tmap_lines;  // tensor-map mode: the line view (2-D boxes of one stage), if g.line_h > 0
    const float* in;
    float* out;
    StreamGeom g;
    int stages;
    uint32_t tx_extra;
    uint64_t timeout_ns;
    uint32_t* status;
    uint32_t coef_off;  // byte offset of the op's staged data in dynamic shared memory
    uint32_t groups;    // consumer groups taking alternate stages: 1, or 2 (see ring_kernel)
    int64_t run;        // 0: persistent grid, CTA b takes stages b, b + grid, ...; else `run` stages a CTA
    RegularStages reg;  // stages the producer plans by the regular-stage shortcut
    Op op;
};

__device__ __forceinline__ float lds_f32(const unsigned char* slot, uint32_t off) {
    return *reinterpret_cast<const float*>(slot + off);
}

// Groups q, q + kConsumers, ..., U at a time while U whole groups remain;
// advances q past them. Idx is the index type (see consume_stage).
template <int U, int kConsumers, class Idx, class Op>
__device__ __forceinline__ void vec_groups(const RingParams<Op>& P, const float4* src, float4* dst, Idx& q, Idx ngroups,
                                           const float* cs) {
    for (; q + (U - 1) * kConsumers < ngroups; q += U * kConsumers) {
        float v[4 * U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float4 t = src[q + u * kConsumers];
            v[4 * u + 0] = t.x;
            v[4 * u + 1] = t.y;
            v[4 * u + 2] = t.z;
            v[4 * u + 3] = t.w;
        }
        P.op.apply(v, cs);
#pragma unroll
        for (int u = 0; u < U; ++u)
            dst[q + u * kConsumers] = make_float4(v[4 * u + 0], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
    }
}

// Relatively misaligned stage: output group q takes floats kSkip .. kSkip + 3
// of the aligned 16-byte words q and q + 1 of the slot, U groups a round.
template <int U, int kSkip, int kConsumers, class Op>
__device__ __forceinline__ void shifted_groups(const RingParams<Op>& P, const float4* w, float4* dst, int& q,
                                               int ngroups, const float* cs) {
    for (; q + (U - 1) * kConsumers < ngroups; q += U * kConsumers) {
        float v[4 * U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float4 a = w[q + u * kConsumers];
            const float4 b = w[q + u * kConsumers + 1];
            const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) v[4 * u + t] = f[kSkip + t];
        }
        P.op.apply(v, cs);
#pragma unroll
        for (int u = 0; u < U; ++u)
            dst[q + u * kConsumers] = make_float4(v[4 * u + 0], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
    }
}

template <int kSkip, int kConsumers, class Op>
__device__ __forceinline__ void shifted_stage(const RingParams<Op>& P, const float4* w, float4* dst, int ngroups,
                                              const float* cs, int ct) {
    int q = ct;
    shifted_groups<4, kSkip, kConsumers>(P, w, dst, q, ngroups, cs);
    shifted_groups<1, kSkip, kConsumers>(P, w, dst, q, ngroups, cs);
}

// ---------------------------------------------------------------- checked build
// With kChecks the kernel verifies, for every stage, that each copy it is about
// to issue and each shared/global range its consumers will touch lies inside
// the caller's buffers and the stage slot; a violation is recorded in the
// status word (AP_ERR_SHAPE and the site), the CTA aborts, and nothing is
// accessed. Used by the tests as a stand-in for a memory checker.

__device__ __forceinline__ void check_fail(uint32_t* status, uint32_t site, volatile int* abort_flag) {
    atomicCAS(status, 0u, kStatusShape | (site << 8));
    *abort_flag = 1;
}

// The copies the producer issues for one stage.
__device__ __forceinline__ bool producer_plan_ok(const StreamGeom& g, const StagePlan& sp) {
    const uint64_t lo = g.in_addr, hi = g.in_addr + 4 * static_cast<uint64_t>(g.n);
    for (int k = 0; k < sp.nspans; ++k) {
        const Span& sn = sp.span[k];
        if (sn.x0 < 0 || sn.x1 > g.n || sn.x0 >= sn.x1) return false;
        if (g.box_bytes != 0) {
            if (sn.bulk_dst % 128 || sn.bulk_dst + static_cast<uint64_t>(sn.bulk_bytes) > g.slot_bytes) return false;
            if (sn.line_y >= 0) {  // one 2-D box of whole lines inside the line view
                if (g.line_h <= 0 || sp.nspans != 1 || sn.x0 != g.line_r + sn.line_y * kFlatBoxElems) return false;
                if (sn.line_y + g.line_h > g.line_rows || sn.bulk_bytes != 4 * kFlatBoxElems * g.line_h) return false;
                continue;
            }
            if (sn.x0 % 4 != 0) return false;
            if (sn.bulk_bytes % g.box_bytes || boxes_for(g, sn.x1 - sn.x0) * g.box_bytes != sn.bulk_bytes) return false;
            if (sn.x0 + (boxes_for(g, sn.x1 - sn.x0) - 1) * g.box_elems > 0x7fffffffll) return false;  // int32
            continue;
        }
        if (sn.bulk_bytes) {
            if (sn.bulk_src % 16 || sn.bulk_dst % 16 || sn.bulk_bytes % 16) return false;
            if (sn.bulk_src < lo || sn.bulk_src + sn.bulk_bytes > hi) return false;
            if (sn.bulk_dst + static_cast<uint64_t>(sn.bulk_bytes) > g.slot_bytes) return false;
        }
        if (sn.head_end > sn.x0 && sn.region + sn.lead + 4 * static_cast<uint64_t>(sn.head_end - sn.x0) > g.slot_bytes)
            return false;
        if (sn.tail_begin < sn.x1 && (sn.tail_dst % 16 || sn.tail_dst + 16ull > g.slot_bytes)) return false;
    }
    return true;
}

// The shared-memory and output ranges the consumers touch for one stage.
__device__ __forceinline__ bool consumer_desc_ok(const StreamGeom& g, const SlotDesc& d, uint64_t out_addr) {
    if (d.lo < 0 || d.lo > d.e_al || d.e_al > d.e_end || d.e_end > d.hi || d.hi > g.n) return false;
    if ((d.e_end - d.e_al) % 4 || d.e_al - d.lo > 3 || d.hi - d.e_end > 3) return false;
    if (d.e_end > d.e_al && (out_addr + 4 * static_cast<uint64_t>(d.e_al)) % 16) return false;
    const uint64_t ngroups = static_cast<uint64_t>(d.e_end - d.e_al) / 4;
    const uint64_t o0 = d.off0 + 4 * static_cast<uint64_t>(d.e_al - d.lo);
    if (d.mode == MODE_VEC) {
        if (o0 % 16 || o0 + 16 * ngroups > g.slot_bytes) return false;
    } else if (d.mode == MODE_SHIFTED) {
        if (o0 % 4 != 0 || o0 % 16 == 0) return false;  // 4, 8 or 12 bytes off the 16-byte grid
        if ((o0 & ~15ull) + 16 * ngroups + 16 > g.slot_bytes) return false;
    }
    const uint64_t L = static_cast<uint64_t>(d.hi - d.lo);
    const uint64_t l1 = d.len1 < static_cast<int64_t>(L) ? static_cast<uint64_t>(d.len1) : L;
    if (d.off0 + 4 * l1 > g.slot_bytes) return false;
    if (L > l1 && d.off1 + 4 * (L - l1) > g.slot_bytes) return false;
    return true;
}

// kConsumers threads take the stage; kRegLimited: the kernel runs 16
// consumer warps, whose register budget caps a thread at 24 chains.
template <int kConsumers, bool kRegLimited, class Op>
__device__ __forceinline__ void consume_stage(const RingParams<Op>& P, const SlotDesc& d, const unsigned char* slot,
                                              const float* cs, int ct) {
    // A stage holds fewer than 2^31 16-byte groups (it fits in shared memory).
    const int ngroups = static_cast<int>((d.e_end - d.e_al) >> 2);
    float* __restrict__ out = P.out;
    const uint32_t o0 = d.off0 + static_cast<uint32_t>(4 * (d.e_al - d.lo));  // input of the first group
    if (d.mode == MODE_VEC) {
        const float4* src = reinterpret_cast<const float4*>(slot + o0);
        float4* dst = reinterpret_cast<float4*>(out + d.e_al);
        int q = ct;
        // 17 warps (16 consumers + producer) leave at most 96 registers a
        // thread, too few for 32 chains: 16 chains there, or 24 (six groups)
        // where the op asks for them (a polynomial of degree 44 or more, 34 in
        // two consumer groups, whose stages are whole rounds of six groups a
        // thread: 1.5-4 % faster;
        // the 16-chain loop stays faster at low degree and for a six-plus-two
        // split). The choice is the host's: a per-stage test here cost the
        // low-degree loop 2 %.
        // Group indices are 32-bit, except in the 24-chain rounds: measured
        // on the 2^30-float polynomial, 32-bit indices made the other rounds
        // 1-8 % faster at degrees 8-128 but the 24-chain rounds 9 % slower
        // (degree 128, 96 KiB stages), so those keep 64-bit ones.
        constexpr int kG = kRegLimited ? 4 : Op::kGroups;
        if constexpr (kRegLimited && Op::kGroups > 4) {
            if (P.op.six_groups) {
                int64_t q6 = q;
                vec_groups<6, kConsumers, int64_t>(P, src, dst, q6, static_cast<int64_t>(ngroups), cs);
                q = static_cast<int>(q6);
            }
        }
        // The narrower rounds only where groups remain: a stage of whole
        // rounds (the automatic shapes) then pays one test instead of one per
        // loop (2^30-float polynomial: degree 128 +0.3-0.6 % at every depth,
        // degree 32 at depth 6 +1.9 %).
        if (q < ngroups) {
            vec_groups<kG, kConsumers, int>(P, src, dst, q, ngroups, cs);
            if (q < ngroups) {
                if (kG > 4) vec_groups<4, kConsumers, int>(P, src, dst, q, ngroups, cs);
                vec_groups<2, kConsumers, int>(P, src, dst, q, ngroups, cs);
                vec_groups<1, kConsumers, int>(P, src, dst, q, ngroups, cs);
            }
        }
    } else if (d.mode == MODE_SHIFTED) {
        // Input 4/8/12 bytes off the output's 16-byte grid: two aligned
        // 16-byte shared loads per group (bank-conflict free) instead of four
        // 4-byte loads that conflict four ways across the warp. Copy and
        // scale take four groups a round with the shift a compile-time
        // constant (2-3 % faster than one group a round). The polynomial
        // keeps one group a round: the larger loop changed the register
        // allocation of its whole kernel and cost the aligned loop 2-4 % at
        // degree 32.
        const uint32_t sh = o0 & 15u;
        const float4* w = reinterpret_cast<const float4*>(slot + (o0 - sh));
        float4* dst = reinterpret_cast<float4*>(out + d.e_al);
        if constexpr (Op::kGroups > 4) {
            for (int q = ct; q < ngroups; q += kConsumers) {
                const float4 a = w[q];
                const float4 b = w[q + 1];
                float v[4];
                if (sh == 4) {
                    v[0] = a.y, v[1] = a.z, v[2] = a.w, v[3] = b.x;
                } else if (sh == 8) {
                    v[0] = a.z, v[1] = a.w, v[2] = b.x, v[3] = b.y;
                } else {
                    v[0] = a.w, v[1] = b.x, v[2] = b.y, v[3] = b.z;
                }
                P.op.apply(v, cs);
                dst[q] = make_float4(v[0], v[1], v[2], v[3]);
            }
        } else if (sh == 4) {
            shifted_stage<1, kConsumers>(P, w, dst, ngroups, cs, ct);
        } else if (sh == 8) {
            shifted_stage<2, kConsumers>(P, w, dst, ngroups, cs, ct);
        } else {
            shifted_stage<3, kConsumers>(P, w, dst, ngroups, cs, ct);
        }
    } else {
        for (int64_t q = ct; q < ngroups; q += kConsumers) {
            const int64_t e = d.e_al + 4 * q;
            float v[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) v[t] = lds_f32(slot, desc_offset_of_output(d, e + t));
            P.op.apply(v, cs);
            *reinterpret_cast<float4*>(out + e) = make_float4(v[0], v[1], v[2], v[3]);
        }
    }
    // The first stage's unaligned head and the last stage's tail (<= 3 each).
    const int64_t nh = d.e_al - d.lo;
    const int64_t nt = d.hi - d.e_end;
    if (ct < nh + nt) {
        const int64_t e = ct < nh ? d.lo + ct : d.e_end + (ct - nh);
        float v[1] = {lds_f32(slot, desc_offset_of_output(d, e))};
        P.op.apply(v, cs);
        out[e] = v[0];
    }
}

// kConsumerWarps consumer warps plus one producer warp per CTA.
// kGroups consumer groups take alternate stages: 1, or 2 groups of 8 warps
// for the 16-warp polynomial at even ring depths of 4 or more (chosen on the
// host). With two, a thread takes twice the values of a stage, and one
// group's wait and release overlap the other's fma work: degree 32 at depth
// 4 goes from 0.95 to 1.0 of the copy; at depth 2 one group is faster.
template <class Op, int kConsumerWarps, bool kChecks, int kGroups>
__global__ void __launch_bounds__(32 * (kConsumerWarps + 1), 1) ring_kernel(const __grid_constant__ RingParams<Op> P) {
    constexpr int kConsumers = 32 * kConsumerWarps;
    constexpr bool kRegLimited = kConsumerWarps >= 16;
    constexpr int groups = kGroups;
    extern __shared__ __align__(128) unsigned char smem[];
    const int S = P.stages;
    const uint32_t slot_bytes = P.g.slot_bytes;
    SlotDesc* descs = reinterpret_cast<SlotDesc*>(smem + static_cast<size_t>(S) * slot_bytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(descs + S);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * S);
    const uint32_t smem_base = ptx::smem_addr(smem);
    const uint32_t bar_base = ptx::smem_addr(bars);
    auto full = [&](int s) { return bar_base + 8u * static_cast<uint32_t>(s); };
    auto empty = [&](int s) { return bar_base + 8u * static_cast<uint32_t>(S + s); };

    float* cs = reinterpret_cast<float*>(smem + P.coef_off) + 4;  // the op's data, after 16 bytes of zeros
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full(s), 1);
            ptx::mbar_init(empty(s), kConsumerWarps / groups);
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    P.op.stage(cs, threadIdx.x, blockDim.x);
    __syncthreads();

    const int64_t T = P.g.n_stages;
    const int64_t G = gridDim.x;
    // This CTA's stages: j0, j0 + step, ... (count of them). Persistent grid:
    // b, b + G, b + 2G, ...; otherwise the run of stages [b run, b run + run).
    int64_t j0, step, count;
    if (P.run == 0) {
        j0 = blockIdx.x;
        step = G;
        count = j0 < T ? (T - j0 + G - 1) / G : 0;
    } else {
        j0 = static_cast<int64_t>(blockIdx.x) * P.run;
        step = 1;
        count = j0 < T ? (T - j0 < P.run ? T - j0 : P.run) : 0;
    }
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (warp == 0) {
        if (lane != 0) return;
        // ------------------------------------------------ producer (one thread)
        if (P.g.box_bytes != 0) {
            // box destinations must be 128-byte aligned: refuse (status, no copy) otherwise
            if (smem_base & 127u) {
                atomicCAS(P.status, 0u, kStatusAlign | (SITE_RING_TENSOR_ALIGN << 8));
                *abort_flag = 1;
                return;
            }
            ptx::prefetch_tensormap(&P.tmap);
            if (P.g.line_h > 0) ptx::prefetch_tensormap(&P.tmap_lines);
        }
        int64_t issued = 0;
        int s = 0;        // slot of stage `issued`: issued mod S
        uint32_t ph = 0;  // its phase: (issued / S) mod 2
        for (int64_t j = j0; issued < count; j += step, ++issued) {
            const int w = wait_phase<false>(empty(s), ph ^ 1u, P.timeout_ns, abort_flag);
            if (w != WAIT_OK) {
                if (w == WAIT_TIMEOUT) raise_timeout(P.status, SITE_RING_PRODUCER_EMPTY, abort_flag);
                break;
            }
            const uint32_t slot = smem_base + static_cast<uint32_t>(s) * slot_bytes;
            if (j >= 1 && j < P.reg.end) {
                // a regular stage: one bulk copy to the slot's start
                SlotDesc d;
                const uint64_t src = regular_stage(P.g, P.reg, j, &d);
                if (kChecks) {  // the shortcut must agree with the full plan
                    StagePlan sp;
                    plan_stage(P.g, j, &sp);
                    SlotDesc full_d;
                    make_slot_desc(sp, &full_d);
                    if (!producer_plan_ok(P.g, sp) || sp.nspans != 1 || sp.span[0].bulk_src != src ||
                        sp.span[0].bulk_bytes != P.reg.bytes || sp.span[0].bulk_dst != 0 ||
                        sp.span[0].head_end != sp.span[0].x0 || sp.span[0].tail_begin != sp.span[0].x1 ||
                        full_d.lo != d.lo || full_d.hi != d.hi || full_d.e_al != d.e_al || full_d.e_end != d.e_end ||
                        full_d.len1 != d.len1 || full_d.off0 != d.off0 || full_d.mode != d.mode) {
                        check_fail(P.status, SITE_CHECK_PRODUCER, abort_flag);
                        break;
                    }
                }
                descs[s] = d;  // published to the consumers by the arrive below
                ptx::mbar_arrive_expect_tx(full(s), P.reg.bytes + P.tx_extra);
                ptx::bulk_g2s(slot, reinterpret_cast<const void*>(src), P.reg.bytes, full(s));
                if (++s == S) s = 0, ph ^= 1u;
                continue;
            }
            StagePlan sp;
            plan_stage(P.g, j, &sp);
            if (kChecks && !producer_plan_ok(P.g, sp)) {
                check_fail(P.status, SITE_CHECK_PRODUCER, abort_flag);
                break;
            }
            make_slot_desc(sp, &descs[s]);  // published to the consumers by the arrive below
            bool edges = false;
            uint32_t tx = 0;
            for (int k = 0; k < sp.nspans; ++k) {
                const Span& sn = sp.span[k];
                for (int64_t x = sn.x0; x < sn.head_end; ++x) {
                    ptx::cp_async_ca4(slot + sn.region + sn.lead + static_cast<uint32_t>(4 * (x - sn.x0)), P.in + x);
                    edges = true;
                }
                if (sn.tail_begin < sn.x1) {
                    ptx::cp_async_cg16(slot + sn.tail_dst, P.in + P.g.t_in,
                                       static_cast<uint32_t>(4 * (P.g.n - P.g.t_in)));
                    edges = true;
                }
                tx += sn.bulk_bytes;
            }
            if (edges) ptx::cp_async_mbar_arrive(full(s));
            ptx::mbar_arrive_expect_tx(full(s), tx + P.tx_extra);
            for (int k = 0; k < sp.nspans; ++k) {
                const Span& sn = sp.span[k];
                if (sn.bulk_bytes == 0) continue;
                if (P.g.box_bytes != 0) {
                    // tensor-map mode: the stage as one 2-D box of the line
                    // view, else whole 1-D boxes from the span's first element
                    if (sn.line_y >= 0) {
                        ptx::tensor_g2s_2d(slot + sn.bulk_dst, &P.tmap_lines, 0, static_cast<int32_t>(sn.line_y),
                                           full(s));
                    } else {
                        const uint32_t nbox = sn.bulk_bytes / P.g.box_bytes;
                        const int32_t be = static_cast<int32_t>(P.g.box_elems);
                        const int32_t x0 = static_cast<int32_t>(sn.x0);
                        for (uint32_t b = 0; b < nbox; ++b)
                            ptx::tensor_g2s_1d(slot + sn.bulk_dst + b * P.g.box_bytes, &P.tmap,
                                               x0 + static_cast<int32_t>(b) * be, full(s));
                    }
                    continue;
                }
                ptx::bulk_g2s(slot + sn.bulk_dst, reinterpret_cast<const void*>(sn.bulk_src), sn.bulk_bytes, full(s));
            }
            if (++s == S) s = 0, ph ^= 1u;
        }
        // Never leave with copies in flight: wait (bounded) for the last
        // S tiles issued. Tiles already consumed return at once.
        for (int64_t k = issued > S ? issued - S : 0; k < issued; ++k) {
            if (!drain_wait<false>(full(static_cast<int>(k % S)), static_cast<uint32_t>((k / S) & 1), P.timeout_ns,
                                   P.status, SITE_RING_DRAIN, abort_flag))
                break;
        }
        return;
    }

    // ---------------------------------------------------- consumers
    // With two groups, group g takes stages g, g + 2, ...; for an even ring
    // depth (the host's condition) every use of a slot then falls to the
    // same group, so each group waits on its slots' phases in order exactly
    // as a single group does. (With an odd depth a group could see the phase
    // of the slot's use two laps back as complete.)
    const int grp = (warp - 1) / (kConsumerWarps / groups);
    const int ct = threadIdx.x - 32 - grp * (kConsumers / groups);
    int s = grp;      // slot of stage i: i mod S
    uint32_t ph = 0;  // its phase: (i / S) mod 2
    for (int64_t i = grp; i < count; i += groups) {
        int w = WAIT_OK;
        if (lane == 0) {
            w = wait_phase<false>(full(s), ph, P.timeout_ns, abort_flag);
            if (w == WAIT_TIMEOUT) raise_timeout(P.status, SITE_RING_CONSUMER_FULL, abort_flag);
        }
        w = __shfl_sync(0xffffffffu, w, 0);
        if (w != WAIT_OK) break;
        __syncwarp();  // orders lane 0's observation of the phase before the other lanes' reads
        const SlotDesc d = descs[s];
        if (kChecks && !consumer_desc_ok(P.g, d, reinterpret_cast<uint64_t>(P.out))) {
            if (lane == 0) check_fail(P.status, SITE_CHECK_CONSUMER, abort_flag);
            break;
        }
        consume_stage<kConsumers / groups, kRegLimited>(P, d, smem + static_cast<size_t>(s) * slot_bytes, cs, ct);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty(s));
        s += groups;
        if (s >= S) s -= S, ph ^= 1u;
    }
}

template <class Op, int kConsumerWarps, bool kChecks, int kGroups = 1>
ap_status launch_ring_op(const DeviceInfo& di, const RingParams<Op>& P, int64_t grid, int64_t smem,
                         cudaStream_t stream) {
    // Raise the kernel's dynamic shared-memory limit once per device.
    static std::atomic<int64_t> configured[64];  // limit already set on this device (setting twice is harmless)
    const int d = di.device;
    if (d < 0 || d >= 64) return AP_ERR_CUDA;
    auto kernel = ring_kernel<Op, kConsumerWarps, kChecks, kGroups>;
    if (configured[d].load() < smem) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, di.smem_optin) != cudaSuccess)
            return AP_ERR_CUDA;
        configured[d] = di.smem_optin;
    }
    kernel<<<static_cast<unsigned>(grid), 32 * (kConsumerWarps + 1), static_cast<size_t>(smem), stream>>>(P);
    return cudaGetLastError() == cudaSuccess ? AP_OK : AP_ERR_CUDA;
}

template <class Op, bool kChecks>
ap_status launch_ring_checks(const DeviceInfo& di, int64_t warps, const RingParams<Op>& P, int64_t grid, int64_t smem,
                             cudaStream_t stream) {
    if (warps == 16) {
        if constexpr (std::is_same<Op, OpPolyDev>::value) {
            if (P.groups == 2) return launch_ring_op<Op, 16, kChecks, 2>(di, P, grid, smem, stream);
        }
        return launch_ring_op<Op, 16, kChecks>(di, P, grid, smem, stream);
    }
    if (warps == 12) {
        if constexpr (std::is_same<Op, OpPolyDev>::value) {
            if (P.groups == 2) return launch_ring_op<Op, 12, kChecks, 2>(di, P, grid, smem, stream);
            if (P.groups == 3) return launch_ring_op<Op, 12, kChecks, 3>(di, P, grid, smem, stream);
        }
        return launch_ring_op<Op, 12, kChecks>(di, P, grid, smem, stream);
    }
    return launch_ring_op<Op, 8, kChecks>(di, P, grid, smem, stream);
}

template <class Op>
ap_status launch_ring_warps(const DeviceInfo& di, int64_t warps, bool checks, const RingParams<Op>& P, int64_t grid,
                            int64_t smem, cudaStream_t stream) {
    if (checks) return launch_ring_checks<Op, true>(di, warps, P, grid, smem, stream);
    return launch_ring_checks<Op, false>(di, warps, P, grid, smem, stream);
}

}  // namespace

int64_t stage_elems_for(int64_t payload_bytes, int64_t unit) {
    int64_t se = payload_bytes / 4;
    if (se < 4) se = 4;
    int64_t l = 4;
    if (unit > 0 && unit <= se) {
        int64_t a = unit, b = 4;
        while (b) {
            const int64_t t = a % b;
            a = b;
            b = t;
        }
        l = unit / a * 4;  // lcm(unit, 4)
    }
    if (l <= se) return se / l * l;
    return se / 4 * 4;
}

RingShape auto_ring_shape(OpKind kind, int stages, int degree) {
    // Measured on GB300 (2^28-float scale and row shift, 2^30-float
    // polynomial at degrees 0-128, every ring depth 2-6; medians of
    // interleaved repetitions). Two schedules: a persistent grid (run 0), and
    // runs of consecutive stages per CTA (run r), as many CTAs as that takes,
    // which the hardware starts in index order as earlier ones finish, so the
    // grid reads and writes one narrow window of memory at any moment. Runs
    // win wherever the kernel is bound by memory: 1.03-1.05 of the copy
    // against 0.96-1.0 for the persistent grid. Where the fma work bounds it,
    // a CTA must keep its SM busy across stages and the persistent grid wins
    // (a run's first load is exposed with one 16-warp CTA per SM).
    if (kind == OP_POLY) {
        const int64_t r = 2 * static_cast<int64_t>(stages);  // runs: every slot filled twice
        // Bands by degree at each depth, chosen from sweeps at degrees 0-32
        // (every few degrees), 64, 80, 96 and 128; the best shape moves
        // jaggedly with the degree near the crossover, so each band is the
        // measured best of its neighbourhood.
        switch (stages) {
            case 2:
                // 0-15: 1.05 of the copy; 16-26: 96 KiB runs 1.00-1.045 (64 KiB
                // runs fell to 0.93 at 26); 27-31: 64 KiB persistent 1.01-1.03
                // (96 KiB 0.92-1.0); from 32 96 KiB persistent (1.038 at 32,
                // 0.874 of the register-only fma rate at 128)
                if (degree <= 15) return RingShape{64 * 1024, 1, 16, 4};
                if (degree <= 26) return RingShape{96 * 1024, 1, 16, 4};
                if (degree <= 31) return RingShape{64 * 1024, 1, 16};
                return RingShape{96 * 1024, 1, 16};
            case 3:
                // 0-1: 32 KiB runs (1.06); 2-14: 48 KiB runs (1.05, where 32
                // KiB runs fell to 0.97 at 14); 15-26: 64 KiB runs (0.99-1.044);
                // 27-29: 48 KiB persistent (1.0-1.046); then persistent stages of
                // 64 KiB (0.98-1.01 at 30-32); from degree 64 one 24-chain round
                // a stage (48 KiB: 0.860 of the register-only fma rate at
                // degree 128, 0.839 with 64 KiB; +0.3-1 % at 64-79)
                if (degree <= 1) return RingShape{32 * 1024, 1, 16, r};
                if (degree <= 14) return RingShape{48 * 1024, 1, 16, r};
                if (degree <= 26) return RingShape{64 * 1024, 1, 16, r};
                if (degree <= 29) return RingShape{48 * 1024, 1, 16};
                if (degree < 64) return RingShape{64 * 1024, 1, 16};
                return RingShape{48 * 1024, 1, 16};
            case 4:
                // 0-16: 32 KiB runs (1.047-1.055); 17-26: 48 KiB runs (1.01-1.045,
                // where 32 KiB runs fell to 0.92); 27-31: 32 KiB persistent in two
                // consumer groups (0.99-1.03); from 32 48 KiB persistent in two
                // groups (1.042 at 32, 0.872 of the register-only rate at 128)
                if (degree <= 16) return RingShape{32 * 1024, 1, 16, r};
                if (degree <= 26) return RingShape{48 * 1024, 1, 16, r};
                return RingShape{degree <= 31 ? 32 * 1024 : 48 * 1024, 1, 16};
            case 5:
                // 0-18: 32 KiB runs (1.05 falling to 1.0); 19-22: 12 consumer
                // warps persistent (1.0-1.025, runs 0.96-0.98); 23-25: 40 KiB
                // persistent (1.04 at 24); above 32 KiB persistent (1.0 at 26,
                // 0.92 at 32)
                if (degree <= 18) return RingShape{32 * 1024, 1, 16, r};
                if (degree <= 22) return RingShape{32 * 1024, 1, 12};
                if (degree <= 25) return RingShape{40 * 1024, 1, 16};
                return RingShape{32 * 1024, 1, 16};
            default:
                // 0-12: 24 KiB runs (1.05); 13-26: 32 KiB runs (1.044 falling
                // to 0.98); 27-30: 24 KiB persistent, 16 warps in two groups
                // (0.97-1.036, against 0.90-0.95 for the shapes either side);
                // from 31 the persistent grid with 12 consumer warps in three
                // groups, each taking every third stage in two rounds of 32
                // chains (degree 32: 1.02 of the copy; degree 128: 0.853 of
                // the register-only fma rate, against 0.836 with 16 warps in
                // two groups)
                if (degree <= 12) return RingShape{24 * 1024, 1, 16, r};
                if (degree <= 26) return RingShape{32 * 1024, 1, 16, r};
                if (degree <= 30) return RingShape{24 * 1024, 1, 16, 0, 2};
                return RingShape{32 * 1024, 1, 12, 0, 3};
        }
    }
    // Scale and row shift: runs of 2 S consecutive 16 KiB stages per CTA (each
    // slot of the ring filled twice): 1.03-1.05 of the copy at every depth,
    // where the persistent grid reached 0.97-1.0 (2^28 floats).
    return RingShape{16 * 1024, 1, 8, 2 * static_cast<int64_t>(stages)};
}

namespace {

template <class Op>
void fill_params(RingParams<Op>& P, const float* in, float* out, const StreamGeom& g, int stages, uint32_t tx_extra,
                 uint64_t timeout, uint32_t* status, int64_t coef_off, const CUtensorMap& tmap,
                 const CUtensorMap& tmap_lines) {
    P.tmap = tmap;
    P.tmap_lines = tmap_lines;
    P.in = in;
    P.out = out;
    P.g = g;
    P.stages = stages;
    P.tx_extra = tx_extra;
    P.timeout_ns = timeout;
    P.status = status;
    P.coef_off = static_cast<uint32_t>(coef_off);
    P.groups = 1;
    P.run = 0;
    make_regular(g, &P.reg);
}

}  // namespace

ap_status launch_ring(const DeviceInfo& di, const Options& o, const float* in, float* out, int64_t n, int64_t off,
                      int64_t unit, int stages, const OpArgs& op, bool tensor, cudaStream_t stream) {
    RingShape shape;
    if (tensor || !tuned_shape(di.device, op.kind, stages, &shape)) shape = auto_ring_shape(op.kind, stages, op.kind == OP_POLY ? op.degree : 0);
    const int64_t payload = o.stage_bytes > 0 ? o.stage_bytes : shape.payload;
    const int64_t cps = o.ctas_per_sm > 0 ? o.ctas_per_sm : shape.ctas_per_sm;
    const int64_t warps = o.consumer_warps > 0 ? o.consumer_warps : shape.consumer_warps;
    int64_t se = stage_elems_for(payload, unit);
    StreamGeom g;
    CUtensorMap tmap, tmap_lines;
    std::memset(&tmap, 0, sizeof(tmap));
    std::memset(&tmap_lines, 0, sizeof(tmap_lines));
    const bool use_tensor = tensor && tensor_ok(reinterpret_cast<uint64_t>(in), reinterpret_cast<uint64_t>(out), n, off);
    if (use_tensor) {
        // Whole 1 KiB boxes per stage; automatic stages give up boxes until
        // the ring (each slot two boxes larger than its stage) fits in shared
        // memory.
        se = std::max<int64_t>(kFlatBoxElems, se / kFlatBoxElems * kFlatBoxElems);
        if (o.stage_bytes == 0) {
            auto ring_bytes = [&](int64_t e) {
                return static_cast<int64_t>(stages) * (4 * e + 8 * kFlatBoxElems + 256 + 64) + 16 * stages + 16;
            };
            while (se > kFlatBoxElems && ring_bytes(se) > di.smem_optin) se -= kFlatBoxElems;
        }
        make_geom_tensor(&g, reinterpret_cast<uint64_t>(in), reinterpret_cast<uint64_t>(out), n, off, se, true);
        auto encode = tensor_map_encoder();
        if (encode == nullptr) return AP_ERR_CUDA;
        const cuuint32_t estr[2] = {1, 1};
        const cuuint64_t dims[1] = {static_cast<cuuint64_t>(n)};
        const cuuint64_t strides[1] = {0};  // a rank-1 tensor has no strides; never read
        const cuuint32_t box[1] = {static_cast<cuuint32_t>(kFlatBoxElems)};
        CUresult r = encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 1, const_cast<float*>(in), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r == CUDA_SUCCESS && g.line_h > 0) {
            // line_rows lines of 256 floats from element line_r (16-byte aligned: off % 4 == 0)
            const cuuint64_t ldims[2] = {static_cast<cuuint64_t>(kFlatBoxElems), static_cast<cuuint64_t>(g.line_rows)};
            const cuuint64_t lstrides[1] = {static_cast<cuuint64_t>(4 * kFlatBoxElems)};
            const cuuint32_t lbox[2] = {static_cast<cuuint32_t>(kFlatBoxElems), static_cast<cuuint32_t>(g.line_h)};
            r = encode(&tmap_lines, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(in) + g.line_r, ldims,
                       lstrides, lbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        }
        if (r != CUDA_SUCCESS) return AP_ERR_CUDA;
    } else {
        make_geom(&g, reinterpret_cast<uint64_t>(in), reinterpret_cast<uint64_t>(out), n, off, se);
    }
    const int64_t coef_off =
        static_cast<int64_t>(stages) * (g.slot_bytes + static_cast<int64_t>(sizeof(SlotDesc))) + 2 * 8 * stages + 16;
    const int64_t coef_bytes = op.kind == OP_POLY ? 16 + (4 * (op.degree + 1) + 15) / 16 * 16 : 0;
    const int64_t smem = coef_off + coef_bytes;
    if (smem > di.smem_optin) return AP_ERR_SMEM;
    // Schedule: a persistent grid, or runs of consecutive stages (a grid cap
    // asks for the persistent grid). Runs are lengthened where the grid would
    // pass 2^30 CTAs.
    int64_t run = o.ring_run == 1 ? 0 : (o.ring_run > 1 ? o.ring_run : shape.run);
    if (o.grid > 0) run = 0;
    int64_t grid;
    if (run > 0) {
        const int64_t cap = int64_t(1) << 30;
        if ((g.n_stages + run - 1) / run > cap) run = (g.n_stages + cap - 1) / cap;
        grid = (g.n_stages + run - 1) / run;
    } else {
        grid = std::min<int64_t>(g.n_stages, static_cast<int64_t>(di.sms) * cps);
        if (o.grid > 0) grid = std::min<int64_t>(grid, o.grid);
    }
    if (grid < 1) grid = 1;

    const uint64_t ia = g.in_addr, oa = g.out_addr;
    int64_t flags = 0;
    if (g.h_in > 0 || g.t_in < n) flags |= 1;
    if (((ia + 4 * static_cast<uint64_t>(off) - oa) & 15) != 0 || off != 0) flags |= 2;
    if (use_tensor) flags |= g.line_h > 0 ? 4 | 8 : 4;
    record_launch(PATH_RING, grid, se, smem, stages, flags);
    record_ring_shape(run, warps, 1, 0);

    const uint64_t timeout = static_cast<uint64_t>(o.timeout_ns);
    const uint32_t tx_extra = static_cast<uint32_t>(o.tx_extra);
    switch (op.kind) {
        case OP_COPY: {
            RingParams<OpCopyDev> P;
            fill_params(P, in, out, g, stages, tx_extra, timeout, di.status, coef_off, tmap, tmap_lines);
            P.run = run;
            return launch_ring_warps(di, warps, o.device_checks != 0, P, grid, smem, stream);
        }
        case OP_SCALE: {
            RingParams<OpScaleDev> P;
            fill_params(P, in, out, g, stages, tx_extra, timeout, di.status, coef_off, tmap, tmap_lines);
            P.run = run;
            P.op.alpha = op.alpha;
            return launch_ring_warps(di, warps, o.device_checks != 0, P, grid, smem, stream);
        }
        case OP_POLY: {
            RingParams<OpPolyDev> P;
            fill_params(P, in, out, g, stages, tx_extra, timeout, di.status, coef_off, tmap, tmap_lines);
            P.run = run;
            P.op.degree = op.degree;
            // 24-chain rounds (16 consumer warps): from degree 64 wherever a
            // group's share of a stage is whole rounds; below it the 16-chain
            // loop is faster.
            P.groups = warps == 16 && stages % 2 == 0 && stages >= 4 ? 2 : 1;
            if (o.consumer_warps == 0 && shape.groups > 0) P.groups = static_cast<uint32_t>(shape.groups);
            if (o.consumer_groups > 0) {
                // an explicit count must divide the warps (16: 1 or 2; 12: 1, 2 or 3; 8: 1) and the ring
                // depth (8 warps in two groups measured 0.78-0.80 of the fma rate at degree 128)
                const int64_t gcount = o.consumer_groups;
                if (warps % gcount != 0 || stages % gcount != 0 || (warps == 8 && gcount > 1)) return AP_ERR_ARG;
                P.groups = static_cast<uint32_t>(gcount);
            }
            // 24 chains a thread where a group's share of a stage is whole
            // rounds of six 16-byte groups, from the degree where they beat 16
            // chains (2^30 floats: from 34 in two groups at depth 4, +2-3 % at
            // degrees 34-63 but -2 % at 33; from 44 in one group at depth 2,
            // +1.3-2.5 % at 48-63 but -0.4-1 % at 33-40)
            const int64_t round_groups = 6 * 32 * 16 / P.groups;
            const bool whole_rounds = warps == 16 && (se / 4) % round_groups == 0;
            P.op.six_groups = whole_rounds && op.degree >= (P.groups == 2 ? 34 : 44) ? 1 : 0;
            record_ring_shape(run, warps, P.groups, warps == 16 ? (P.op.six_groups ? 24 : 16) : 32);
            for (int k = 0; k <= AP_POLY_MAX_DEGREE; ++k) P.op.c[k] = k <= op.degree ? op.coeffs[k] : 0.0f;
            return launch_ring_warps(di, warps, o.device_checks != 0, P, grid, smem, stream);
        }
    }
    return AP_ERR_ARG;
}

}  // namespace ap
