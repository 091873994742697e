// Tile planning for the streaming ring, shared by the kernels, the host
// launchers and the host emulator (ap_debug_emulate_ring).
//
// Every ring call computes out[e] = f(in[(e + off) mod n]) for e in [0, n):
// off = 0 for scale and polynomial, off = shift * cols for the row shift of a
// row-major matrix (a shift by whole rows is a rotation of the flat array).
//
// Output tiles ("stages"). Output element e belongs to stage j when
//   j == 0: e in [0, out_head + se)          j >= 1: e in [out_head + j*se, out_head + (j+1)*se)
// (clipped to n), where out_head (0..3) counts the outputs before the first
// 16-byte aligned output address and se is a multiple of 4. So every stage
// after the first starts on a 16-byte boundary of `out`, and a stage's
// outputs are whole 16-byte groups except the first stage's head and the
// last stage's tail.
//
// Input spans. Stage j reads inputs [a, a + L) with a = (lo + off) mod n; if
// that runs past n it wraps, and the stage has a second span [0, ...). (For
// the row shift these are the tile's rows shifted by `shift`: its own rows
// plus the halo rows of the following tile, wrapping to row 0.)
//
// Shared-memory layout of a span. A span is placed in its region of the
// stage slot so that shared-memory addresses are congruent to global
// addresses modulo 16: input element x sits at
//   region + (in_addr + 4x) - floor16(in_addr + 4*x0).
// The span's elements between the buffer's first and last 16-byte boundaries
// (I0 = ceil16(in_addr), I1 = floor16(in_addr + 4n)) arrive with ONE bulk
// copy of their 16-byte-aligned enclosing range, which never leaves
// [I0, I1) and so never leaves the caller's buffer. Elements before I0 (at
// most 3, only near element 0) use 4-byte cp.async.ca; elements at or after
// I1 (at most 3, only near element n-1) use one 16-byte cp.async.cg whose
// source size is the tail's byte count (the rest of the 16 is zero-filled).
// If the buffer holds no aligned 16-byte block at all, every element is a
// 4-byte copy.
//
// Tensor-map mode (input and output 16-byte aligned, every span starting on
// a 16-byte boundary). The input is described twice to the copy engine: as a
// flat 1-D tensor of n floats, loaded in boxes of 256 floats (1 KiB), and as a
// 2-D "line view" of 1 KiB lines starting at element line_r = off mod 256,
// loaded in boxes of one whole stage (se / 256 lines). A stage with a single
// span that starts on a line of the view and whose box stays inside the
// view's whole lines takes ONE 2-D box; the others (the stage that wraps past
// n, the one that reaches the ragged end) take 1-D boxes. One copy-engine
// instruction per stage matters: boxes issued back to back by one thread are
// accepted about one per 25 ns on GB300, so 1 KiB boxes cannot keep a stage
// ring fed from one producer thread.
#pragma once

#include <cstdint>

#ifdef __CUDACC__
#define AP_HD __host__ __device__ __forceinline__
#else
#define AP_HD inline
#endif

namespace ap {

AP_HD uint64_t floor16(uint64_t a) { return a & ~uint64_t(15); }
AP_HD uint64_t ceil16(uint64_t a) { return (a + 15) & ~uint64_t(15); }

struct StreamGeom {
    uint64_t in_addr;     // byte address of input element 0 (4-byte aligned)
    uint64_t out_addr;    // byte address of output element 0 (4-byte aligned)
    int64_t n;            // elements of each buffer (> 0)
    int64_t off;          // output e reads input (e + off) mod n, 0 <= off < n
    int64_t se;           // stage elements, a multiple of 4, >= 4
    int64_t out_head;     // outputs before the first 16-byte aligned output, min(n, 0..3)
    int64_t n_stages;     // number of stages covering [0, n)
    int64_t h_in;         // inputs [0, h_in) lie before I0 (4-byte copies)
    int64_t t_in;         // inputs [t_in, n) lie at or after I1 (one zero-filling 16-byte copy)
    uint32_t slot_bytes;  // shared-memory bytes of one stage slot (multiple of 16)
    // Tensor-map mode (box_bytes != 0; 0 = 1-D bulk copies).
    uint32_t box_bytes;   // bytes of one flat 1-D box (1024), 0 in bulk mode
    int64_t box_elems;    // floats of one flat 1-D box (256)
    int64_t line_r;       // first element of the line view (off mod 256)
    int64_t line_rows;    // whole 1 KiB lines in the line view
    int64_t line_h;       // lines of one 2-D box (se / 256); 0: no line view
};

// Bytes of a stage slot for stages of `se` elements: two regions, each the
// span's bytes plus up to 12 bytes of alignment lead and 15 of trailing
// rounding, each rounded to 16.
AP_HD uint32_t slot_bytes_for(int64_t se) { return static_cast<uint32_t>(4 * se + 112); }

AP_HD void make_geom(StreamGeom* g, uint64_t in_addr, uint64_t out_addr, int64_t n, int64_t off, int64_t se) {
    g->in_addr = in_addr;
    g->out_addr = out_addr;
    g->n = n;
    g->off = off;
    g->se = se;
    const int64_t oh = static_cast<int64_t>(((16 - (out_addr & 15)) & 15) >> 2);
    g->out_head = oh < n ? oh : n;
    if (n <= 0) {
        g->n_stages = 0;
    } else if (n <= g->out_head + se) {
        g->n_stages = 1;
    } else {
        g->n_stages = 1 + (n - g->out_head - se + se - 1) / se;
    }
    const uint64_t i0 = ceil16(in_addr);
    const uint64_t i1 = floor16(in_addr + 4 * static_cast<uint64_t>(n));
    if (i0 <= i1) {
        g->h_in = static_cast<int64_t>((i0 - in_addr) >> 2);
        g->t_in = static_cast<int64_t>((i1 - in_addr) >> 2);
    } else {
        g->h_in = n;
        g->t_in = n;
    }
    g->slot_bytes = slot_bytes_for(se);
    g->box_bytes = 0;
    g->box_elems = 0;
    g->line_r = 0;
    g->line_rows = 0;
    g->line_h = 0;
}

// Floats in one box of the flat 1-D tensor map, and in one line of the line
// view: the largest box extent a dimension may have (256), 1 KiB.
constexpr int64_t kFlatBoxElems = 256;

// Whether the tensor-map producer can stream n floats read at offset off:
// input and output 16-byte aligned, and every span starting on a 16-byte
// boundary (off a multiple of 4; n too when off != 0, for the span that
// starts after the wrap), with box coordinates inside int32.
AP_HD bool tensor_ok(uint64_t in_addr, uint64_t out_addr, int64_t n, int64_t off) {
    if (((in_addr | out_addr) & 15) != 0 || n <= 0 || off < 0 || off >= n) return false;
    return off % 4 == 0 && (off == 0 || n % 4 == 0) && n <= 0x7fffffffll - 2 * kFlatBoxElems;
}

// Tensor-map geometry (tensor_ok holds; se a multiple of 256). Spans load as
// whole 1-D boxes from their first element (the last may run past the span,
// or past n, where the engine writes zeros), so each region is sized for
// whole boxes: slot = 4 se + 2 box_bytes + 256, regions 128-byte aligned. With
// `lines`, the line view covers the whole lines from element off mod 256 and a
// 2-D box is one stage (it fills region 0, 4 se bytes).
AP_HD void make_geom_tensor(StreamGeom* g, uint64_t in_addr, uint64_t out_addr, int64_t n, int64_t off, int64_t se,
                            bool lines) {
    make_geom(g, in_addr, out_addr, n, off, se);
    g->box_elems = kFlatBoxElems;
    g->box_bytes = static_cast<uint32_t>(4 * kFlatBoxElems);
    g->slot_bytes = static_cast<uint32_t>(4 * se + 2 * static_cast<int64_t>(g->box_bytes) + 256);
    if (lines) {
        g->line_r = off % kFlatBoxElems;
        g->line_rows = (n - g->line_r) / kFlatBoxElems;
        g->line_h = se / kFlatBoxElems;
        if (g->line_rows < g->line_h || g->line_h > 256) g->line_h = 0;
    }
}

AP_HD int64_t boxes_for(const StreamGeom& g, int64_t len) { return (len + g.box_elems - 1) / g.box_elems; }

struct Span {
    int64_t x0, x1;        // input elements [x0, x1)
    int64_t line_y;        // tensor-map mode: first line of its one 2-D box, -1 for 1-D boxes
    uint32_t region;       // slot-relative byte offset of the span's region (multiple of 16)
    uint32_t lead;         // (in_addr + 4*x0) mod 16: byte offset of x0 inside the region
    int64_t head_end;      // [x0, head_end): 4-byte cp.async.ca copies
    int64_t tail_begin;    // [tail_begin, x1): covered by the buffer-tail cp.async.cg
    uint32_t tail_dst;     // slot-relative destination of the tail copy (multiple of 16)
    uint32_t bulk_dst;     // slot-relative destination of the bulk copy (multiple of 16)
    uint32_t bulk_bytes;   // multiple of 16; 0 when the span has no bulk part
    uint64_t bulk_src;     // global source of the bulk copy (multiple of 16)
};

struct StagePlan {
    int64_t lo, hi;        // outputs [lo, hi)
    int64_t len1;          // outputs [lo, lo + len1) read span 0, the rest span 1
    int nspans;            // 1, or 2 when the input wraps past n
    Span span[2];
    int64_t e_al, e_end;   // outputs [e_al, e_end) are whole 16-byte aligned groups
    bool vec;              // each group's 4 inputs form one aligned 16-byte word in shared memory
};

AP_HD void plan_span(const StreamGeom& g, int64_t x0, int64_t x1, uint32_t region, Span* s) {
    s->x0 = x0;
    s->x1 = x1;
    s->region = region;
    s->line_y = -1;
    if (g.box_bytes != 0) {  // whole boxes from an aligned first element: no edges
        s->lead = 0;
        s->head_end = x0;
        s->tail_begin = x1;
        s->tail_dst = 0;
        s->bulk_src = 0;
        s->bulk_dst = region;
        s->bulk_bytes = static_cast<uint32_t>(boxes_for(g, x1 - x0) * g.box_bytes);
        return;
    }
    const uint64_t g0 = g.in_addr + 4 * static_cast<uint64_t>(x0);
    const uint64_t a0 = floor16(g0);
    s->lead = static_cast<uint32_t>(g0 - a0);
    const int64_t hb = (x0 < g.h_in) ? (x1 < g.h_in ? x1 : g.h_in) : x0;
    const int64_t tb = (x1 > g.t_in) ? (x0 > g.t_in ? x0 : g.t_in) : x1;
    s->head_end = hb;
    s->tail_begin = tb;
    const uint64_t i1 = g.in_addr + 4 * static_cast<uint64_t>(g.t_in);
    s->tail_dst = (tb < x1) ? region + static_cast<uint32_t>(i1 - a0) : 0u;
    if (tb > hb) {
        const uint64_t b0 = floor16(g.in_addr + 4 * static_cast<uint64_t>(hb));
        const uint64_t b1 = ceil16(g.in_addr + 4 * static_cast<uint64_t>(tb));
        s->bulk_src = b0;
        s->bulk_dst = region + static_cast<uint32_t>(b0 - a0);
        s->bulk_bytes = static_cast<uint32_t>(b1 - b0);
    } else {
        s->bulk_src = 0;
        s->bulk_dst = 0;
        s->bulk_bytes = 0;
    }
}

AP_HD int64_t stage_lo(const StreamGeom& g, int64_t j) { return j == 0 ? 0 : g.out_head + j * g.se; }

AP_HD void plan_stage(const StreamGeom& g, int64_t j, StagePlan* p) {
    const int64_t lo = stage_lo(g, j);
    int64_t hi = g.out_head + (j + 1) * g.se;
    if (hi > g.n) hi = g.n;
    p->lo = lo;
    p->hi = hi;
    const int64_t L = hi - lo;
    int64_t a = lo + g.off;
    if (a >= g.n) a -= g.n;
    int64_t len1 = g.n - a;
    if (len1 > L) len1 = L;
    p->len1 = len1;
    plan_span(g, a, a + len1, 0u, &p->span[0]);
    if (len1 < L) {
        p->nspans = 2;
        const uint32_t r2 = g.box_bytes != 0
                                ? static_cast<uint32_t>(boxes_for(g, len1) * g.box_bytes)
                                : static_cast<uint32_t>((4 * len1 + 32 + 15) & ~int64_t(15));
        plan_span(g, 0, L - len1, r2, &p->span[1]);
    } else {
        p->nspans = 1;
        // one 2-D box of the line view for the whole stage where it fits
        const int64_t rel = a - g.line_r;
        if (g.line_h > 0 && rel >= 0 && rel % kFlatBoxElems == 0 && rel / kFlatBoxElems + g.line_h <= g.line_rows) {
            p->span[0].line_y = rel / kFlatBoxElems;
            p->span[0].bulk_bytes = static_cast<uint32_t>(4 * kFlatBoxElems * g.line_h);
        }
    }
    int64_t e_al = lo > g.out_head ? lo : g.out_head;
    if (e_al > hi) e_al = hi;
    p->e_al = e_al;
    p->e_end = e_al + ((hi - e_al) & ~int64_t(3));
    p->vec = (p->nspans == 1) && (((p->span[0].lead + 4 * (e_al - lo)) & 15) == 0);
}

// Slot-relative shared-memory byte offset of the input of the first aligned
// output group (output e_al).
AP_HD uint32_t group_input_offset(const StagePlan& p) {
    return p.span[0].region + p.span[0].lead + static_cast<uint32_t>(4 * (p.e_al - p.lo));
}

// Stages whose inputs lie in one span but 4, 8 or 12 bytes off the 16-byte
// grid relative to the output: group q's four inputs are the last 16 - d
// bytes of the aligned word at w0 + 16q and the first d bytes of the next
// word (w0 = group_input_offset - d). Both words lie inside the span's
// region: the next word of the last group ends at most lead + 4L + 16 bytes
// into a region of at least 4L + 32 bytes.
AP_HD bool shifted_words(const StagePlan& p) { return !p.vec && p.nspans == 1; }

// What the consumers of a stage need, computed once by the producer and
// stored beside the stage's slot (so consumer threads spend their issue
// slots on the stage's data, not on re-planning it).
enum SlotMode : uint32_t { MODE_VEC = 0, MODE_SHIFTED = 1, MODE_SCALAR = 2 };

struct SlotDesc {
    int64_t lo, hi;        // outputs [lo, hi)
    int64_t e_al, e_end;   // whole aligned 16-byte output groups [e_al, e_end)
    int64_t len1;          // outputs [lo, lo + len1) read span 0
    uint32_t off0, off1;   // slot offsets of span 0's and span 1's first input (region + lead)
    uint32_t mode;         // SlotMode
    uint32_t pad_[3];
};
static_assert(sizeof(SlotDesc) == 64, "slot descriptor is 64 bytes");

AP_HD void make_slot_desc(const StagePlan& p, SlotDesc* d) {
    d->lo = p.lo;
    d->hi = p.hi;
    d->e_al = p.e_al;
    d->e_end = p.e_end;
    d->len1 = p.len1;
    d->off0 = p.span[0].region + p.span[0].lead;
    d->off1 = p.nspans == 2 ? p.span[1].region + p.span[1].lead : 0u;
    d->mode = p.vec ? MODE_VEC : (p.nspans == 1 ? MODE_SHIFTED : MODE_SCALAR);
    d->pad_[0] = d->pad_[1] = d->pad_[2] = 0;
}

// Slot offset of the input that output e reads, from a descriptor.
AP_HD uint32_t desc_offset_of_output(const SlotDesc& d, int64_t e) {
    const int64_t q = e - d.lo;
    if (q < d.len1) return d.off0 + static_cast<uint32_t>(4 * q);
    return d.off1 + static_cast<uint32_t>(4 * (q - d.len1));
}

// Slot-relative shared-memory byte offset of the input that output e reads.
AP_HD uint32_t smem_offset_of_output(const StagePlan& p, int64_t e) {
    const int64_t q = e - p.lo;
    if (q < p.len1) return p.span[0].region + p.span[0].lead + static_cast<uint32_t>(4 * q);
    return p.span[1].region + p.span[1].lead + static_cast<uint32_t>(4 * (q - p.len1));
}

// Regular stages. Every stage j in [1, end) is a whole stage of se outputs
// whose one input span neither wraps past n nor reaches the buffer's
// unaligned tail (its start is past the unaligned head since j >= 1). Such a
// stage's plan is stage 1's moved by j - 1 stages: one bulk copy of `bytes`
// from src1 + 4 se (j - 1) to slot offset 0, and a descriptor whose first
// input sits at slot offset off0 in mode `mode` (VEC or SHIFTED). The
// producer takes this shortcut for them instead of planning each stage from
// the geometry (about ten instructions instead of a few hundred, which
// matters when the consumer warps leave the producer few issue slots).
// Bulk (not tensor-map) mode only; end = 0 when no stage qualifies.
struct RegularStages {
    int64_t end;     // regular stages are [1, end)
    uint64_t src1;   // bulk source of stage 1
    uint32_t bytes;  // bulk bytes of a regular stage
    uint32_t off0;   // slot offset of a regular stage's first input
    uint32_t mode;   // its consumer mode
    uint32_t pad_;
};

AP_HD void make_regular(const StreamGeom& g, RegularStages* r) {
    r->end = 0;
    r->src1 = 0;
    r->bytes = 0;
    r->off0 = 0;
    r->mode = MODE_VEC;
    r->pad_ = 0;
    if (g.box_bytes != 0 || g.n_stages < 3) return;
    // stage j reads [lo + off, lo + off + se) with lo = out_head + j se: it
    // is regular while lo + off + se <= min(n, t_in)
    const int64_t lim = (g.n < g.t_in ? g.n : g.t_in) - g.out_head - g.off - g.se;
    if (lim < g.se) return;
    int64_t end = lim / g.se + 1;
    if (end > g.n_stages) end = g.n_stages;
    StagePlan sp;
    plan_stage(g, 1, &sp);
    const Span& sn = sp.span[0];
    if (sp.nspans != 1 || sp.hi - sp.lo != g.se || sn.head_end != sn.x0 || sn.tail_begin != sn.x1 ||
        sn.bulk_bytes == 0 || sn.bulk_dst != 0 || sp.e_al != sp.lo || sp.e_end != sp.hi)
        return;
    SlotDesc d;
    make_slot_desc(sp, &d);
    if (d.mode == MODE_SCALAR) return;
    r->end = end;
    r->src1 = sn.bulk_src;
    r->bytes = sn.bulk_bytes;
    r->off0 = d.off0;
    r->mode = d.mode;
}

// The bulk source and the descriptor of regular stage j (1 <= j < r.end).
AP_HD uint64_t regular_stage(const StreamGeom& g, const RegularStages& r, int64_t j, SlotDesc* d) {
    const int64_t lo = g.out_head + j * g.se;
    d->lo = lo;
    d->hi = lo + g.se;
    d->e_al = lo;
    d->e_end = lo + g.se;
    d->len1 = g.se;
    d->off0 = r.off0;
    d->off1 = 0;
    d->mode = r.mode;
    d->pad_[0] = d->pad_[1] = d->pad_[2] = 0;
    return r.src1 + 4 * static_cast<uint64_t>(g.se) * static_cast<uint64_t>(j - 1);
}

}  // namespace ap
