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
// ring of S send slots and S receive slots per CTA. A chunk moves as P
// equal pieces (each a ring item), so the load, the hand-off and the store
// of one chunk overlap each other; piece q of a chunk lands as piece q of the
// receiver's output chunk, so the result is the same as moving whole chunks.
// CTA rank r has three roles, one warp each for the two single-thread roles
// (rank r receives from rank r + shift, 1 for ap_cluster_exchange):
//   loader   (warp 0): waits credit[s], loads the next piece of its chunk of
//            the group from global memory into send[s] (bulk copy, load_full[s]).
//   pusher   (warp 1): waits load_full[s], pushes send[s] into recv[s] of
//            rank (r - shift) mod cs, completing on that CTA's recv_full[s].
//   receiver (8 warps in groups of 1, 2, 4 or 8, a piece per group in turn):
//            waits on recv_full[s], stores recv[s] to its output chunk with
//            16-byte stores, arms recv_full[s] with the bytes of the slot's
//            next item, then arrives (remote) on credit[s] of rank
//            (r + shift) mod cs, the CTA that sends to it. In the TMA-store
//            form one thread instead hands recv[s] to a shared->global bulk
//            copy and credits the slot once that copy has read it.
// Before the final cluster barrier each pusher waits (bounded) for the
// credits of its last S pieces, so no copy is in flight when a CTA leaves.
// credit[s] therefore tells a sender both that its send[s] has been read
// (the data reached the receiver) and that the receiver's recv[s] is free,
// so the loader may refill send[s] and the pusher may overwrite recv[s].
//
// Split form (a separate instantiation): the send ring has SS buffers, a
// power of two dividing S. The receiver then also arrives (remote) on
// sent[b] of the sender as soon as a piece has landed, b = i mod SS; the
// loader refills send[b] on that signal instead of the credit, and the pusher
// waits for credit[s] before it pushes into the receiver's slot s. A send
// buffer is then free once its piece has arrived, not once it is stored.
//
// All-to-all form (a2a): each chunk is cs sub-blocks; sub-block j of rank r's
// chunk goes to rank j as sub-block r of its output chunk. The senders go
// round-robin: item i of every CTA goes to rank (r + i) mod cs, so each
// receiver takes exactly one piece per item, from rank (d - i) mod cs. With
// S a multiple of cs, items i and i + S of a sender go to the same receiver
// and slot, so every (receiver, slot) pair has one fixed sender and the
// credit protocol above holds unchanged, with the peer chosen per item.
#include <algorithm>
#include <atomic>
#include <cstring>

#include "device_common.cuh"
#include "internal.h"

namespace ap {
namespace {

constexpr int kExConsumerWarps = 8;
constexpr int kExConsumers = 32 * kExConsumerWarps;
constexpr int kExThreads = 64 + kExConsumers;
constexpr int64_t kExMaxSlots = 16;

struct ExParams {
    // Batched form: the input and output as 5-D tensors {e0, e1, nsub, cs,
    // groups} (e0 * e1 floats = one sub-block; nsub = cs sub-blocks per chunk
    // in the all-to-all, else 1), so that one box gathers a rank's sub-block
    // from `batch` consecutive groups.
    CUtensorMap tin;
    CUtensorMap tout;
    int batch;             // groups per item in the batched form; 0: items are pieces of chunks
    const float* in;
    float* out;
    int64_t groups;        // whole groups of cluster_size chunks (batched form: batches of `batch` groups)
    uint32_t chunk_bytes;  // multiple of 16
    uint32_t piece_bytes;  // divides chunk_bytes, multiple of 16
    int pieces;            // chunk_bytes / piece_bytes
    int cs;                // cluster size
    int shift;             // rank r receives from rank (r + shift) mod cs, 0 <= shift < cs
    int stages;            // receive slots (a multiple of cs in the all-to-all form); send slots too, unless split
    int send_slots;        // split form: send slots, a power of two dividing stages (else equal to stages)
    int tma_store;         // receiver stores with bulk copies (1) or with the receiver warps (0)
    int a2a;               // 1: all-to-all (shift unused, pieces = cs x sub_pieces)
    int rgroup;            // receiver warps per piece in the warp-store form: 1, 2, 4 or 8
    int lanes;             // loader and pusher threads each (1, 2 or 4; divides stages)
    int sub_pieces;        // all-to-all: pieces per sub-block (chunk_bytes / cs / piece_bytes)
    uint32_t tx_extra;
    uint64_t timeout_ns;
    uint32_t* status;
};

// A CTA's items in order, without divisions (a 64-bit division per item in
// the single-thread roles would cost them more than moving a piece): item i
// uses ring slot s = i mod S in phase ph = (i / S) mod 2, and is piece
// il = i mod NP of group grp = cid + (i / NP) * ncl; in the all-to-all form
// q = il mod cs picks the peer and t = il / cs the piece of the sub-block.
struct ItemCursor {
    int s = 0;
    uint32_t ph = 0;
    uint32_t round = 0;  // i / S: how many items used slot s before this one
    int64_t grp;
    int64_t il = 0;
    int q = 0;
    int64_t t = 0;
    __device__ explicit ItemCursor(int64_t cid) : grp(cid) {}
    // Advance by L = 1, 2 or 4 items, without a loop (the single-thread roles
    // pay for every instruction per item).
    __device__ __forceinline__ void advance(int L, int S, int64_t NP, int cs, int64_t ncl) {
        next(S, NP, cs, ncl);
        if (L > 1) {
            next(S, NP, cs, ncl);
            if (L > 2) {
                next(S, NP, cs, ncl);
                next(S, NP, cs, ncl);
            }
        }
    }
    __device__ __forceinline__ void next(int S, int64_t NP, int cs, int64_t ncl) {
        if (++s == S) {
            s = 0;
            ph ^= 1u;
            ++round;
        }
        if (++il == NP) {
            il = 0;
            q = 0;
            t = 0;
            grp += ncl;
        } else if (++q == cs) {
            q = 0;
            ++t;
        }
    }
};

// kBatched: items are batches of groups moved with tensor-map boxes (a
// separate instantiation, so that the single-thread roles of the plain form
// carry no branch for it: they are bound by their per-item latency).
// kSplit: the send ring has its own, smaller depth SS (a power of two dividing
// S). The receiver then tells the sender twice: when a piece has landed (its
// send buffer may be refilled: sent[b], b = i mod SS) and, as before, when its
// receive slot is free (credit[s]); the loader waits on sent[b] and the pusher
// on credit[s]. More receive slots then fit beside a short send ring.
// kMinBlocks: CTAs an SM must hold, which caps the registers a thread (three:
// 64, where the other forms use about 90 and an SM holds two of them).
template <bool kBatched, bool kSplit, int kMinBlocks = 1>
__global__ void __launch_bounds__(kExThreads, kMinBlocks) exchange_kernel(const __grid_constant__ ExParams P) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int S = P.stages;
    const int SS = kSplit ? P.send_slots : S;
    const uint32_t CB = P.piece_bytes;  // ring slot = one piece
    const int64_t NP = P.pieces;
    unsigned char* send = smem;
    unsigned char* recv = smem + static_cast<size_t>(SS) * CB;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(SS + S) * CB);
    const int nbars = kSplit ? 4 * S : 3 * S;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + nbars);
    // taken[s]: items of slot s the receivers have finished with; group_bad[g]:
    // a wait of receiver group g failed (warp-store form)
    volatile uint32_t* taken = reinterpret_cast<volatile uint32_t*>(bars + nbars) + 4;
    volatile uint32_t* group_bad = taken + kExMaxSlots;
    const uint32_t bar_base = ptx::smem_addr(bars);
    auto load_full = [&](int s) { return bar_base + 8u * static_cast<uint32_t>(s); };
    auto credit = [&](int s) { return bar_base + 8u * static_cast<uint32_t>(S + s); };
    auto recv_full = [&](int s) { return bar_base + 8u * static_cast<uint32_t>(2 * S + s); };
    auto sent = [&](int b) { return bar_base + 8u * static_cast<uint32_t>(3 * S + b); };  // split form only
    // load_full is indexed by the send buffer: the slot, or b in the split form

    const uint32_t cs = static_cast<uint32_t>(P.cs);
    const uint32_t rank = ptx::cluster_ctarank();
    const uint32_t sh = static_cast<uint32_t>(P.shift);
    const uint32_t dst_rank = (rank + cs - sh) % cs;  // receives this CTA's chunk
    const uint32_t src_rank = (rank + sh) % cs;       // sends this CTA its chunk
    const int64_t cid = ptx::cluster_id_x();
    const int64_t ncl = ptx::nclusters_x();
    const int64_t count = (cid < P.groups ? (P.groups - cid + ncl - 1) / ncl : 0) * NP;
    // Byte offset of the piece of item c (a cursor) in this CTA's chunk: piece
    // il; in the all-to-all form piece t of sub-block blk, where blk is the
    // receiver (rank + q) mod cs for the piece this CTA sends, and the sender
    // (rank - q) mod cs for the piece it receives (that sender wrote its
    // sub-block `rank`, which lands as sub-block `sender` here).
    const int64_t sub_bytes = static_cast<int64_t>(CB) * P.sub_pieces;
    auto item_off = [&](const ItemCursor& c, uint32_t blk) -> int64_t {
        const int64_t base = (c.grp * P.cs + rank) * static_cast<int64_t>(P.chunk_bytes);
        if (!P.a2a) return base + c.il * static_cast<int64_t>(CB);
        return base + blk * sub_bytes + c.t * static_cast<int64_t>(CB);
    };
    auto a2a_dst = [&](const ItemCursor& c) {
        const uint32_t d = rank + static_cast<uint32_t>(c.q);
        return d >= cs ? d - cs : d;
    };
    auto a2a_src = [&](const ItemCursor& c) {
        const uint32_t q = static_cast<uint32_t>(c.q);
        return rank >= q ? rank - q : rank + cs - q;
    };
    const unsigned char* in_bytes = reinterpret_cast<const unsigned char*>(P.in);
    unsigned char* out_bytes = reinterpret_cast<unsigned char*>(P.out);
    // Load item c into send slot s: one box of this rank's (sub-block of its)
    // chunk from `batch` groups, or one bulk copy of a piece.
    auto load_item = [&](const ItemCursor& c, int s) {
        const uint32_t dst = ptx::smem_addr(send + static_cast<size_t>(s) * CB);
        if constexpr (kBatched) {
            ptx::tensor_g2s_5d(dst, &P.tin, 0, 0, P.a2a ? static_cast<int32_t>(a2a_dst(c)) : 0,
                               static_cast<int32_t>(rank), static_cast<int32_t>(c.grp * P.batch), load_full(s));
        } else {
            ptx::bulk_g2s(dst, in_bytes + item_off(c, a2a_dst(c)), CB, load_full(s));
        }
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(load_full(s), 1);
            ptx::mbar_init(credit(s), 1);  // one arrival per item: the warp (or thread) that stored it
            ptx::mbar_init(recv_full(s), 1);
            if (kSplit) ptx::mbar_init(sent(s), 1);  // one arrival per item: its receiver, once it landed
        }
        *abort_flag = 0;
        for (int s = 0; s < S; ++s) taken[s] = 0;
        for (int g = 0; g < kExConsumerWarps; ++g) group_bad[g] = 0;
        ptx::fence_mbar_init();
    }
    if (kBatched && threadIdx.x == 0) {
        ptx::prefetch_tensormap(&P.tin);
        ptx::prefetch_tensormap(&P.tout);
    }
    __syncthreads();
    ptx::cluster_sync();  // every CTA's barriers exist before anyone sends

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Loader and pusher: L lanes each (S a multiple of L), lane l taking
    // items l, l + L, ...; items i and i + S then belong to the same lane, so
    // every lane walks its own slots in order and no phase can alias. Each
    // lane drains its own copies.
    const int L = P.lanes;
    // First item of this lane at or after k0 (lane l takes items = l mod L).
    auto lane_first = [&](int64_t k0) -> int64_t {
        if (k0 <= lane) return lane;
        const int64_t r = (k0 - lane) % L;
        return r == 0 ? k0 : k0 + (L - r);
    };
    if (warp == 0) {
        if (L == 1 && lane == 0) {
            // one lane: the plain loop (measured faster than the lane loop at
            // one lane: these threads are bound by their per-item latency)
            int64_t i = 0;
            ItemCursor c(cid);
            int b = 0;         // split form: send buffer of item i
            uint32_t bph = 0;  // and the parity of its use
            for (; i < count; ++i, c.next(S, NP, P.cs, ncl)) {
                const int s = c.s;
                const int w = kSplit ? wait_phase<true>(sent(b), bph ^ 1u, P.timeout_ns, abort_flag)
                                     : wait_phase<true>(credit(s), c.ph ^ 1u, P.timeout_ns, abort_flag);
                if (w != WAIT_OK) {
                    if (w == WAIT_TIMEOUT) raise_timeout(P.status, SITE_EX_LOADER_CREDIT, abort_flag);
                    break;
                }
                const int sb = kSplit ? b : s;
                ptx::mbar_arrive_expect_tx(load_full(sb), CB + P.tx_extra);
                load_item(c, sb);
                if constexpr (kSplit) {
                    if (++b == SS) {
                        b = 0;
                        bph ^= 1u;
                    }
                }
            }
            for (int64_t k = i > SS ? i - SS : 0; k < i; ++k) {
                if (!drain_wait<false>(load_full(static_cast<int>(k % SS)), static_cast<uint32_t>((k / SS) & 1),
                                       P.timeout_ns, P.status, SITE_EX_DRAIN, abort_flag))
                    break;
            }
        } else if (L > 1 && lane < L) {
            ItemCursor c(cid);
            for (int k = 0; k < lane; ++k) c.next(S, NP, P.cs, ncl);
            int b = lane;  // split form: SS is a multiple of L, so b stays this lane's
            uint32_t bph = 0;
            int64_t i = lane;
            for (; i < count; i += L) {
                const int s = c.s;
                const int w = kSplit ? wait_phase<true>(sent(b), bph ^ 1u, P.timeout_ns, abort_flag)
                                     : wait_phase<true>(credit(s), c.ph ^ 1u, P.timeout_ns, abort_flag);
                if (w != WAIT_OK) {
                    if (w == WAIT_TIMEOUT) raise_timeout(P.status, SITE_EX_LOADER_CREDIT, abort_flag);
                    break;
                }
                const int sb = kSplit ? b : s;
                ptx::mbar_arrive_expect_tx(load_full(sb), CB + P.tx_extra);
                load_item(c, sb);
                c.advance(L, S, NP, P.cs, ncl);
                if constexpr (kSplit) {
                    b += L;
                    if (b >= SS) {
                        b -= SS;
                        bph ^= 1u;
                    }
                }
            }
            for (int64_t k = lane_first(i - SS); k < i; k += L) {
                if (!drain_wait<false>(load_full(static_cast<int>(k % SS)), static_cast<uint32_t>((k / SS) & 1),
                                       P.timeout_ns, P.status, SITE_EX_DRAIN, abort_flag))
                    break;
            }
        }
    } else if (warp == 1) {
        if (L == 1 && lane == 0) {
            uint32_t peer_recv = ptx::mapa(ptx::smem_addr(recv), dst_rank);
            uint32_t peer_bars = ptx::mapa(bar_base, dst_rank);
            ItemCursor c(cid);
            int64_t i = 0;
            int b = 0;
            uint32_t bph = 0;
            for (; i < count; ++i, c.next(S, NP, P.cs, ncl)) {
                if (P.a2a) {
                    peer_recv = ptx::mapa(ptx::smem_addr(recv), a2a_dst(c));
                    peer_bars = ptx::mapa(bar_base, a2a_dst(c));
                }
                const int s = c.s;
                const int sb = kSplit ? b : s;
                int w = wait_phase<false>(load_full(sb), kSplit ? bph : c.ph, P.timeout_ns, abort_flag);
                if (w != WAIT_OK) {
                    if (w == WAIT_TIMEOUT) raise_timeout(P.status, SITE_EX_PUSHER_LOADED, abort_flag);
                    break;
                }
                if constexpr (kSplit) {  // the receiver's slot s is free (item i - S consumed)
                    w = wait_phase<true>(credit(s), c.ph ^ 1u, P.timeout_ns, abort_flag);
                    if (w != WAIT_OK) {
                        if (w == WAIT_TIMEOUT) raise_timeout(P.status, SITE_EX_PUSHER_CREDIT, abort_flag);
                        break;
                    }
                    if (++b == SS) {
                        b = 0;
                        bph ^= 1u;
                    }
                }
                ptx::bulk_s2s_cluster(peer_recv + static_cast<uint32_t>(s) * CB,
                                      ptx::smem_addr(send + static_cast<size_t>(sb) * CB), CB,
                                      peer_bars + 8u * static_cast<uint32_t>(2 * S + s));
            }
            // credits of the last S pieces pushed (see the lane loop below)
            for (int64_t k = i > S ? i - S : 0; k < i; ++k) {
                if (!drain_wait<true>(credit(static_cast<int>(k % S)), static_cast<uint32_t>((k / S) & 1),
                                      P.timeout_ns, P.status, SITE_EX_DRAIN, abort_flag))
                    break;
            }
        } else if (L > 1 && lane < L) {
            uint32_t peer_recv = ptx::mapa(ptx::smem_addr(recv), dst_rank);
            uint32_t peer_bars = ptx::mapa(bar_base, dst_rank);
            ItemCursor c(cid);
            for (int k = 0; k < lane; ++k) c.next(S, NP, P.cs, ncl);
            int b = lane;
            uint32_t bph = 0;
            int64_t i = lane;
            for (; i < count; i += L) {
                if (P.a2a) {
                    peer_recv = ptx::mapa(ptx::smem_addr(recv), a2a_dst(c));
                    peer_bars = ptx::mapa(bar_base, a2a_dst(c));
                }
                const int s = c.s;
                const int sb = kSplit ? b : s;
                int w = wait_phase<false>(load_full(sb), kSplit ? bph : c.ph, P.timeout_ns, abort_flag);
                if (w != WAIT_OK) {
                    if (w == WAIT_TIMEOUT) raise_timeout(P.status, SITE_EX_PUSHER_LOADED, abort_flag);
                    break;
                }
                if constexpr (kSplit) {
                    w = wait_phase<true>(credit(s), c.ph ^ 1u, P.timeout_ns, abort_flag);
                    if (w != WAIT_OK) {
                        if (w == WAIT_TIMEOUT) raise_timeout(P.status, SITE_EX_PUSHER_CREDIT, abort_flag);
                        break;
                    }
                    b += L;
                    if (b >= SS) {
                        b -= SS;
                        bph ^= 1u;
                    }
                }
                ptx::bulk_s2s_cluster(peer_recv + static_cast<uint32_t>(s) * CB,
                                      ptx::smem_addr(send + static_cast<size_t>(sb) * CB), CB,
                                      peer_bars + 8u * static_cast<uint32_t>(2 * S + s));
                c.advance(L, S, NP, P.cs, ncl);
            }
            // Before the final cluster barrier: every piece this lane pushed
            // has been taken by its receiver (its credit, bounded), so no push
            // is still reading this CTA's shared memory or landing in a peer's
            // when a CTA of the cluster leaves. Item k's credit completes
            // phase k / S.
            for (int64_t k = lane_first(i - S); k < i; k += L) {
                if (!drain_wait<true>(credit(static_cast<int>(k % S)), static_cast<uint32_t>((k / S) & 1),
                                      P.timeout_ns, P.status, SITE_EX_DRAIN, abort_flag))
                    break;
            }
        }
    } else if (kBatched || P.tma_store) {
        // Receiver, TMA-store form (always, in the batched form): one thread
        // registers, waits and hands each received piece to the bulk-copy
        // engine (shared -> global); a slot is credited back once the engine
        // has finished reading it.
        if (warp == 2 && lane == 0) {
            const uint32_t credit0 = ptx::mapa(credit(0), src_rank);
            const int lag = S > 2 ? 2 : S - 1;  // bulk stores left reading before a slot is credited
            uint32_t prev1 = 0, prev2 = 0;      // peer credit addresses owed for items i - 1 and i - 2
            ItemCursor c(cid);
            int64_t i = 0;
            for (; i < count; ++i, c.next(S, NP, P.cs, ncl)) {
                const int s = c.s;
                ptx::mbar_arrive_expect_tx(recv_full(s), CB);
                const int w = wait_phase<true>(recv_full(s), c.ph, P.timeout_ns, abort_flag);
                if (w != WAIT_OK) {
                    if (w == WAIT_TIMEOUT) raise_timeout(P.status, SITE_EX_RECEIVER_FULL, abort_flag);
                    break;
                }
                if constexpr (kSplit)  // the piece has landed: its sender may refill the send buffer
                    ptx::mbar_arrive_remote_relaxed(ptx::mapa(sent(s & (SS - 1)), P.a2a ? a2a_src(c) : src_rank));
                const uint32_t src = ptx::smem_addr(recv + static_cast<size_t>(s) * CB);
                if constexpr (kBatched) {
                    // the sender's sub-block lands as sub-block `sender` of this rank's chunks
                    ptx::tensor_s2g_5d(&P.tout, 0, 0, P.a2a ? static_cast<int32_t>(a2a_src(c)) : 0,
                                       static_cast<int32_t>(rank), static_cast<int32_t>(c.grp * P.batch), src);
                } else {
                    ptx::bulk_s2g(out_bytes + item_off(c, a2a_src(c)), src, CB);
                }
                ptx::bulk_commit();
                if (lag == 2) {
                    ptx::bulk_wait_read<2>();
                } else if (lag == 1) {
                    ptx::bulk_wait_read<1>();
                } else {
                    ptx::bulk_wait_read<0>();
                }
                const uint32_t cur =
                    (P.a2a ? ptx::mapa(credit(0), a2a_src(c)) : credit0) + 8u * static_cast<uint32_t>(s);
                // credit the item whose store has now finished reading its slot
                if (lag == 2) {
                    if (i >= 2) ptx::mbar_arrive_remote_relaxed(prev2);
                } else if (lag == 1) {
                    if (i >= 1) ptx::mbar_arrive_remote_relaxed(prev1);
                } else {
                    ptx::mbar_arrive_remote_relaxed(cur);
                }
                prev2 = prev1;
                prev1 = cur;
            }
            ptx::bulk_wait_read<0>();
            if (lag == 2 && i >= 2) ptx::mbar_arrive_remote_relaxed(prev2);
            if (lag >= 1 && i >= 1) ptx::mbar_arrive_remote_relaxed(prev1);
            ptx::bulk_wait_all();
        }
    } else {
        // Receivers in groups of G warps (G = 1, 2, 4 or 8), one piece per
        // group in turn: group g takes items g, g + 8/G, ..., so 8/G pieces
        // drain at once and each is split over 32 G threads. The slot's
        // expected bytes for item k are registered by the group that consumed
        // item k - S (the first S at the start), right after that phase
        // completed and before the sender is credited, so every phase is
        // armed exactly once. A group waits on item k's phase only once
        // taken[s] shows item k - S consumed: a barrier's phase is known by its
        // parity alone, and a group that ran two phases ahead would take the
        // older completed phase for its own. The warps of a group agree on
        // every wait's outcome at a named barrier before any of them goes on,
        // so none is left waiting there.
        const int G = P.rgroup;
        const int NG = kExConsumerWarps / G;
        const int cw = warp - 2;
        const int grp = cw / G;
        const int gt = (cw % G) * 32 + lane;  // thread within the group
        const bool head = (cw % G == 0) && lane == 0;
        if (cw == 0 && lane == 0) {
            for (int64_t k = 0; k < count && k < S; ++k) ptx::mbar_arrive_expect_tx(recv_full(static_cast<int>(k)), CB);
        }
        uint32_t peer_credit = ptx::mapa(credit(0), src_rank);
        ItemCursor c(cid);
        for (int k = 0; k < grp; ++k) c.next(S, NP, P.cs, ncl);
        for (int64_t i = grp; i < count; i += NG) {
            const int s = c.s;
            int w = WAIT_OK;
            if (lane == 0) {
                if (taken[s] < c.round) {  // bounded wait for item k - S to be consumed
                    const uint64_t t0 = ptx::globaltimer_ns();
                    while (taken[s] < c.round) {
                        if (*abort_flag) {
                            w = WAIT_ABORTED;
                            break;
                        }
                        if (ptx::globaltimer_ns() - t0 > P.timeout_ns) {
                            w = WAIT_TIMEOUT;
                            break;
                        }
                    }
                }
                if (w == WAIT_OK) w = wait_phase<true>(recv_full(s), c.ph, P.timeout_ns, abort_flag);
                if (w == WAIT_TIMEOUT) raise_timeout(P.status, SITE_EX_RECEIVER_FULL, abort_flag);
            }
            w = __shfl_sync(0xffffffffu, w, 0);
            if (G > 1) {
                if (lane == 0 && w != WAIT_OK) group_bad[grp] = 1;
                ptx::named_barrier_sync(1 + grp, 32 * G);
                if (group_bad[grp]) w = WAIT_ABORTED;
            }
            if (w != WAIT_OK) break;
            __syncwarp();
            if constexpr (kSplit) {  // the piece has landed: its sender may refill the send buffer
                if (head)
                    ptx::mbar_arrive_remote_relaxed(ptx::mapa(sent(s & (SS - 1)), P.a2a ? a2a_src(c) : src_rank));
            }
            const float4* src = reinterpret_cast<const float4*>(recv + static_cast<size_t>(s) * CB);
            float4* dst = reinterpret_cast<float4*>(out_bytes + item_off(c, a2a_src(c)));
            if (P.a2a) peer_credit = ptx::mapa(credit(0), a2a_src(c));
            const int64_t nq = CB / 16;
            const int stride = 32 * G;
            int64_t q = gt;
            for (; q + 3 * stride < nq; q += 4 * stride) {
                const float4 a = src[q];
                const float4 b = src[q + stride];
                const float4 e = src[q + 2 * stride];
                const float4 f = src[q + 3 * stride];
                dst[q] = a;
                dst[q + stride] = b;
                dst[q + 2 * stride] = e;
                dst[q + 3 * stride] = f;
            }
            for (; q < nq; q += stride) dst[q] = src[q];
            if (G > 1) {
                ptx::named_barrier_sync(1 + grp, 32 * G);
            } else {
                __syncwarp();
            }
            // Credit the slot back to its sender, whose next bulk copy (the
            // async proxy) then overwrites it. The arrive is relaxed, and no
            // proxy fence precedes it, because every read of the slot has
            // already returned its data: each thread's stores took the loaded
            // registers as operands, and all of the group's stores were
            // issued before the group barrier above, so no load of the slot is
            // still outstanding when the credit leaves. Measured on 2^28
            // floats: a release arrive, which also waits for the global
            // stores, cost 22-50 % of the bandwidth (cs 2: 1.01 -> 0.50 of
            // the copy), and a fence.proxy.async before the relaxed arrive
            // 2.3 % at cs 2.
            if (head) {
                if (i + S < count) ptx::mbar_arrive_expect_tx(recv_full(s), CB);
                __threadfence_block();
                taken[s] = c.round + 1;
                ptx::mbar_arrive_remote_relaxed(peer_credit + 8u * static_cast<uint32_t>(s));
            }
            for (int k = 0; k < NG; ++k) c.next(S, NP, P.cs, ncl);
        }
    }
    __syncwarp();
    ptx::cluster_sync();  // no CTA leaves while a peer may still write its shared memory
}

}  // namespace

ap_status launch_exchange(const DeviceInfo& di, const Options& o, const float* in, float* out, int64_t groups, int cs,
                          int64_t chunk_bytes, int64_t shift, bool a2a, cudaStream_t stream) {
    // Piece: the largest multiple of 16 dividing chunk_bytes that is at most
    // the target (8 KiB, or the stage-bytes setting), and two CTAs per SM
    // (three for the all-to-all below). Measured on GB300 with 32 KiB chunks:
    // the loader and pusher are single threads with a fixed cost per piece,
    // so pieces much below 8 KiB starve them, and a second CTA per SM doubles
    // those threads; whole 32 KiB chunks leave too few slots in flight.
    const int64_t target = o.stage_bytes > 0 ? o.stage_bytes : 8192;
    // Shared memory per CTA when `cps` CTAs share an SM (228 KiB per SM, 1 KiB
    // reserved per CTA): more resident CTAs let clusters of 8 fill more SMs.
    // The all-to-all over clusters of 8 or 16 with sub-blocks of 4 KiB or
    // more (pieces, not batches) runs three CTAs per SM, in the instantiation
    // whose registers let three fit. Clusters of 8 then hold 8 send and 8
    // receive slots of 4 KiB a CTA, and the loads in flight per SM go from 64
    // to 96 KiB (2^28 floats, 32 KiB chunks: 0.935 -> 0.966 of the copy;
    // 64 KiB chunks: 0.934 -> 0.972); clusters of 16 with 64 KiB chunks
    // (2 KiB pieces) 0.68 -> 0.74. Two receiver warps per 4 KiB piece then
    // take it to 0.977 (below). The other forms lost up to 4 % with that
    // register cap, and the all-to-all at 4 CTAs gained nothing from a third
    // CTA.
    const bool a2a_three =
        a2a && (cs == 8 || cs == 16) && o.ctas_per_sm == 0 && o.ex_batch < 2 && chunk_bytes / cs >= 4096;
    const int64_t cps = o.ctas_per_sm > 0 ? o.ctas_per_sm : a2a_three ? 3 : 2;
    int64_t budget = std::min<int64_t>(di.smem_optin, kSmemPerSM / cps - 1024) - 512;
    // A piece divides the chunk (all-to-all: the sub-block of chunk_bytes / cs).
    const int64_t span = a2a ? chunk_bytes / cs : chunk_bytes;
    const int64_t units = span / 16;
    int64_t piece = 0, S = 0;
    if (!a2a) {
        int64_t piece_units = 1;
        for (int64_t d = 1; d * d <= units; ++d) {
            if (units % d) continue;
            const int64_t a = d, b = units / d;
            if (16 * a <= target && a > piece_units) piece_units = a;
            if (16 * b <= target && b > piece_units) piece_units = b;
        }
        piece = 16 * piece_units;
        S = std::min<int64_t>(budget / (2 * piece), kExMaxSlots);
        if (S < 1) return AP_ERR_SMEM;
    } else {
        // All-to-all: S a multiple of cs and at least 2. Measured on GB300
        // (2^28 floats, 32 KiB chunks): pieces under 4 KiB cost the
        // single-thread loader and pusher more per byte than the ring hides,
        // and at equal bytes in flight more slots win (the receiver warps
        // take one item each). So: pieces that divide the sub-block and stay
        // within the target, at least 4 KiB where the sub-block allows; the
        // most bytes in flight (S x piece); on a tie the smaller piece.
        int64_t largest = 0;
        for (int64_t d = 1; d <= units; ++d)
            if (units % d == 0 && 16 * d <= target) largest = 16 * d;
        // (If no such piece leaves a ring of cs slots, any smaller piece.)
        for (const int64_t floor_piece : {std::min<int64_t>(4096, largest), int64_t(16)}) {
            for (int64_t d = 1; d <= units; ++d) {
                if (units % d || 16 * d > target || 16 * d < floor_piece) continue;
                const int64_t p = 16 * d;
                int64_t slots = std::min<int64_t>(budget / (2 * p), kExMaxSlots);
                slots -= slots % cs;
                if (slots < 2) continue;
                if (slots * p > S * piece) {
                    piece = p;
                    S = slots;
                }
            }
            if (S > 0) break;
        }
        if (S == 0) return AP_ERR_SMEM;
    }
    // Batched form: a sub-block (the chunk, outside the all-to-all) under
    // 8 KiB makes items too small for the single-thread roles (256-byte chunks:
    // 0.04 of the copy as pieces), so an item gathers a rank's sub-block from
    // `batch` consecutive groups with one tensor-map box (about 8 KiB), pushes
    // it as one bulk copy and stores it with one tensor-map box; the engine
    // clips the last, partial batch at the tensor's edge. Needs a sub-block of
    // at most 256 floats or a multiple of 256 (a box extent is at most 256),
    // and a batch of whole 128-byte multiples (box destinations).
    const int64_t nsub = a2a ? cs : 1;
    const int64_t sub = chunk_bytes / nsub;
    const int64_t sub_e = sub / 4;
    // Automatic: fixed neighbour for chunks under 8 KiB, items of 8 KiB; the
    // all-to-all for sub-blocks under 4 KiB (at 4 KiB plain pieces already run
    // at the copy's rate), items sized for a ring of min(16, 2 cs) slots.
    // tight: items sized for a ring of cs slots instead of about 2 cs
    auto plan_batch = [&](int64_t bud, bool tight) -> int64_t {
        if (o.ex_batch == 1 || (o.ex_batch < 2 && sub >= (a2a ? 4096 : 8192)) || !(sub_e <= 256 || sub_e % 256 == 0) ||
            groups >= (int64_t(1) << 31) || tensor_map_encoder() == nullptr)
            return 0;
        const int64_t ring = tight ? cs : std::min<int64_t>(16, 2 * cs);
        const int64_t item_target = a2a ? std::min<int64_t>(8192, bud / (2 * ring)) : 8192;
        int64_t m = 128;  // smallest batch step keeping batch * sub a multiple of 128
        while (m > 1 && (sub * (m / 2)) % 128 == 0) m /= 2;
        int64_t b = o.ex_batch >= 2 ? o.ex_batch : std::max<int64_t>(1, item_target / sub);
        b = std::min<int64_t>(256, (b + m - 1) / m * m);
        if (b > 256 - 256 % m) b = 256 - 256 % m;
        const int64_t min_slots = a2a ? std::max<int64_t>(2, cs) : 2;
        while (b > m && 2 * min_slots * b * sub > bud) b -= m;
        return (b >= 2 && 2 * min_slots * b * sub <= bud) ? b : 0;
    };
    int64_t batch = plan_batch(budget, false);
    if (batch == 0 && a2a && cs >= 8) {
        // Large clusters: a ring of cs slots still leaves room for batches at
        // two CTAs per SM (8 CTAs, 16 KiB chunks: 0.96 of the copy against
        // 0.85 at one CTA per SM); where the usual ring fits a batch it is
        // faster (smaller chunks lost 1-5 % with cs slots).
        batch = plan_batch(budget, true);
    }
    if (batch == 0 && a2a && o.ctas_per_sm == 0 && plan_batch(kSmemPerSM - 1024 - 512, false) > 0) {
        // Large clusters with small sub-blocks: one CTA per SM leaves room for
        // batches (16 CTAs, 32 KiB chunks: 0.79 of the copy against 0.68 as
        // 2 KiB pieces at two CTAs per SM).
        budget = std::min<int64_t>(di.smem_optin, kSmemPerSM - 1024) - 512;
        batch = plan_batch(budget, false);
    }
    int64_t work = groups;  // what the clusters walk: groups, or batches of groups
    if (batch > 0) {
        piece = batch * sub;
        S = std::min<int64_t>(budget / (2 * piece), kExMaxSlots);
        if (a2a) S -= S % cs;
        work = (groups + batch - 1) / batch;
    }
    // Split form: a send ring of SS buffers beside S receive slots, S now as
    // many as fit (a multiple of SS, and of cs in the all-to-all). Automatic
    // for the all-to-all where the ring depth is a power of two, with the
    // send ring as deep as that depth: freeing a send buffer as soon as its
    // piece lands, rather than once it is stored and credited, measured 1-4 %
    // faster there (8 CTAs, 16 KiB chunks: 1.0 of the copy against 0.96; 32 KiB
    // chunks: 0.94 against 0.92, with 16 receive slots). Shallower send rings
    // were slower (the loader then waits out a whole load, push and landing),
    // and the fixed neighbour gained nothing.
    int64_t SS = 0;  // 0: one depth for both rings
    const int64_t want = o.ex_send_slots == 1 ? 0
                         : o.ex_send_slots > 1 ? o.ex_send_slots
                         : (a2a && S >= 2 && (S & (S - 1)) == 0) ? S
                                                                : 0;
    if (want > 0) {
        int64_t m = want;
        if (a2a) {
            int64_t x = cs, y = want;  // lcm(cs, want)
            while (y) {
                const int64_t t = x % y;
                x = y;
                y = t;
            }
            m = cs / x * want;
        }
        int64_t S2 = std::min<int64_t>(budget / piece - want, kExMaxSlots);
        S2 -= S2 % m;
        if (S2 >= std::max<int64_t>(want, 2)) {
            SS = want;
            S = S2;
        }
    }
    const int64_t smem = (SS > 0 ? SS + S : 2 * S) * piece + (SS > 0 ? 4 : 3) * 8 * S + 16 + 4 * kExMaxSlots +
                         4 * kExConsumerWarps;  // + abort flag, taken[], group_bad[]
    if (smem > di.smem_optin) return AP_ERR_SMEM;

    // Receiver form, unless set: measured on GB300 (2^28 floats, 32 KiB chunks;
    // 8-64 KiB for clusters of 4 and 8). Fixed neighbour (one sender, pieces
    // arrive in order): all eight warps on every piece for clusters of 1-2
    // (1.01 of the copy; bulk stores 0.96-1.0), bulk stores for 3-5 and 8
    // (0.97-1.0 and 0.99, against 0.95-0.99 and 0.95-0.96 with eight warps),
    // four warps per piece for 6-7 (0.96, against 0.87-0.94 either other
    // way), one warp per piece from 9 (16: 0.85, against 0.76). All-to-all
    // (pieces from every sender, in no fixed order, so in-order draining waits
    // on the slowest sender): bulk stores for clusters of 1-2 (1.01-1.02), one
    // warp per piece from 3 up (0.91-1.01; eight warps per piece: 0.53-0.56),
    // two with 4 KiB pieces at three CTAs per SM (clusters of 8, 32 and 64 KiB
    // chunks: 0.977 against 0.960 with one and 0.89-0.90 with four).
    const bool fixed_bulk = !a2a && (cs == 3 || cs == 4 || cs == 5 || cs == 8);
    const bool tma_store =
        batch > 0 || o.ex_tma_store == 1 || (o.ex_tma_store == 0 && ((a2a && cs <= 2) || fixed_bulk));
    const int64_t rgroup = o.ex_group > 0        ? o.ex_group
                           : a2a                 ? (cps >= 3 && piece >= 4096 ? 2 : 1)
                           : (cs <= 5 || cs == 8) ? kExConsumerWarps
                           : cs <= 7             ? 4
                                                 : 1;
    if (rgroup != 1 && rgroup != 2 && rgroup != 4 && rgroup != 8) return AP_ERR_ARG;
    // Loader and pusher lanes, unless set: four for all-to-all pieces of 2 KiB
    // or less, where the single-thread roles' per-item latency sets the rate
    // (clusters of 16, 32 KiB chunks: 0.68 of the copy against 0.40 with one
    // lane), else one (at 4 KiB pieces the one-lane loop is 3-10 % faster).
    // A count that does not divide the ring depth falls back to one that does.
    int64_t lanes = o.ex_lanes > 0 ? o.ex_lanes : (a2a && piece <= 2048 ? 4 : 1);
    while (lanes > 1 && (S % lanes != 0 || (SS > 0 && SS % lanes != 0))) lanes /= 2;

    static std::atomic<bool> configured[64];  // attributes set on this device (setting twice is harmless)
    if (di.device < 0 || di.device >= 64) return AP_ERR_CUDA;
    if (!configured[di.device].load()) {
        for (auto kernel : {exchange_kernel<false, false>, exchange_kernel<true, false>, exchange_kernel<false, true>,
                            exchange_kernel<true, true>, exchange_kernel<false, true, 3>}) {
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, di.smem_optin) !=
                    cudaSuccess ||
                cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
                return AP_ERR_CUDA;
        }
        configured[di.device] = true;
    }
    // Split pieces planned for three CTAs per SM take the instantiation that
    // lets three fit.
    auto kernel = batch > 0 ? (SS > 0 ? exchange_kernel<true, true> : exchange_kernel<true, false>)
                  : SS > 0  ? (cps >= 3 ? exchange_kernel<false, true, 3> : exchange_kernel<false, true>)
                            : exchange_kernel<false, false>;

    CUtensorMap tin, tout;
    std::memset(&tin, 0, sizeof(tin));
    std::memset(&tout, 0, sizeof(tout));
    if (batch > 0) {
        const int64_t e0 = std::min<int64_t>(sub_e, 256);
        const cuuint64_t dims[5] = {static_cast<cuuint64_t>(e0), static_cast<cuuint64_t>(sub_e / e0),
                                    static_cast<cuuint64_t>(nsub), static_cast<cuuint64_t>(cs),
                                    static_cast<cuuint64_t>(groups)};
        const cuuint64_t strides[4] = {static_cast<cuuint64_t>(4 * e0), static_cast<cuuint64_t>(sub),
                                       static_cast<cuuint64_t>(chunk_bytes),
                                       static_cast<cuuint64_t>(cs) * static_cast<cuuint64_t>(chunk_bytes)};
        const cuuint32_t box[5] = {static_cast<cuuint32_t>(e0), static_cast<cuuint32_t>(sub_e / e0), 1, 1,
                                   static_cast<cuuint32_t>(batch)};
        const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        auto encode = tensor_map_encoder();
        for (int k = 0; k < 2; ++k) {
            if (encode(k == 0 ? &tin : &tout, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5,
                       k == 0 ? const_cast<float*>(in) : out, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                       CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return AP_ERR_CUDA;
        }
    }
    ExParams P{tin,
               tout,
               static_cast<int>(batch),
               in,
               out,
               work,
               static_cast<uint32_t>(chunk_bytes),
               static_cast<uint32_t>(piece),
               static_cast<int>(batch > 0 ? nsub : chunk_bytes / piece),
               cs,
               static_cast<int>(((shift % cs) + cs) % cs),
               static_cast<int>(S),
               static_cast<int>(SS > 0 ? SS : S),
               tma_store ? 1 : 0,
               a2a ? 1 : 0,
               static_cast<int>(rgroup),
               static_cast<int>(lanes),
               static_cast<int>(a2a && batch == 0 ? span / piece : 1),
               static_cast<uint32_t>(o.tx_extra),
               static_cast<uint64_t>(o.timeout_ns),
               di.status};

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
    if (cudaOccupancyMaxActiveClusters(&max_clusters, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();  // clear: an unsupported cluster shape is an argument error, not a sticky one
        return cs > AP_MAX_CLUSTER ? AP_ERR_CLUSTER : AP_ERR_CUDA;
    }
    if (max_clusters < 1) return AP_ERR_CLUSTER;
    // Persistent clusters: as many as fit, cluster c taking groups c, c +
    // clusters, .... (Clusters that each take a run of consecutive groups, the
    // ring's schedule for memory-bound work, measured 0.43-0.92 of the copy
    // against 0.80-1.02: a cluster's start, barrier set-up and two cluster
    // barriers, and the fill and drain of its ring, are paid per run.)
    int64_t ncl = std::min<int64_t>(work, max_clusters);
    if (o.grid > 0) ncl = std::max<int64_t>(1, std::min<int64_t>(ncl, o.grid / cs));
    cfg.gridDim = dim3(static_cast<unsigned>(ncl * cs), 1, 1);
    record_launch(PATH_EXCHANGE, ncl * cs, piece / 4, smem, S, batch > 0 ? 4 : 0);
    if (cudaLaunchKernelEx(&cfg, kernel, P) != cudaSuccess) return AP_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? AP_OK : AP_ERR_CUDA;
}

}  // namespace ap
