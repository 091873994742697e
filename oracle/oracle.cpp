// CPU oracle for the asynchronous global->shared streaming path.
//
// TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct
// definition of what each streaming operation computes. Only the test suite,
// the smoke check and the benchmark's CPU-baseline leg may load it. The CUDA
// library never includes, links or calls anything here, and this file shares
// no header, helper or constant with it.
//
// Asynchronous copy changes when bytes move, never which bytes, so each
// operation's result has a plain definition that is written out below as the
// simplest loop. Built with -O2 -ffp-contract=off -fno-fast-math so that the
// compiler neither fuses a*b+c (GCC's default on aarch64) nor reorders
// floating-point work.
//
// Parity status: every function below is pinned by tests that do not call it
// twice (worked example, library routines, exact rational arithmetic,
// closed forms and invariants); nothing here is "parity unpinned".

#include <cmath>
#include <cstdint>
#include <cstring>

extern "C" {

// Elementwise scale y = alpha * x.
// "CUDA Async Copy and Pipeline Guide", Implementation Comparison (Before and
// After kernels): every element of a 256-float tile is multiplied by 2.0f and
// stored; the asynchronous version computes the same product. One fp32
// multiply, rounded to nearest even.
void orc_scale(const float* in, float* out, int64_t n, float alpha) {
    for (int64_t i = 0; i < n; ++i) {
        out[i] = alpha * in[i];
    }
}

// Row shift B[i, :] = A[(i + shift) mod rows, :] of a row-major rows x cols
// matrix.
// "Asynchronous Copies" (TVM TIRx), section A Global-to-Shared Copy: each of 64
// threads copies one 4-float row into shared memory and then reads the next
// thread's row, (tid + 1) % 64; the page checks the result against
// torch.roll(a, shifts=-1, dims=0). shift = 1 is that example; any other shift
// is reduced modulo rows into [0, rows).
// Returns 0, or -1 for rows < 1 or cols < 1 with a non-empty matrix.
int orc_row_roll(const float* A, float* B, int64_t rows, int64_t cols, int64_t shift) {
    if (rows == 0 || cols == 0) return 0;
    if (rows < 0 || cols < 0) return -1;
    const int64_t s = ((shift % rows) + rows) % rows;
    for (int64_t i = 0; i < rows; ++i) {
        const int64_t src_row = (i + s) % rows;
        for (int64_t j = 0; j < cols; ++j) {
            B[i * cols + j] = A[src_row * cols + j];
        }
    }
    return 0;
}

// Polynomial p(x) = sum_k c[k] x^k of degree K, evaluated by Horner's rule with
// one fused multiply-add per step:
//   p = c[K];  for k = K-1 .. 0:  p = fma(p, x, c[k]).
// The pages leave the per-tile compute open ("compute on tile[cur]" in
// "Asynchronous Data Movement", section Double buffering) and name "not enough
// work to hide copy latency" as a pitfall ("CUDA Async Copy and Pipeline
// Guide", Common Performance Issues); the Horner chain is the library's
// tunable-intensity stand-in for that compute. Coefficients are in ascending
// order of power; degree 0 gives the constant c[0].
int orc_poly(const float* in, float* out, int64_t n, const float* coeffs, int degree) {
    if (degree < 0) return -1;
    for (int64_t i = 0; i < n; ++i) {
        const float x = in[i];
        float p = coeffs[degree];
        for (int k = degree - 1; k >= 0; --k) {
            p = std::fma(p, x, coeffs[k]);
        }
        out[i] = p;
    }
    return 0;
}

// Cluster hand-off: the input is cut into chunks of chunk_bytes, and every run
// of cluster_size consecutive chunks is one cluster's share. Within a cluster
// the chunk of rank r is handed to rank (r - 1) mod cluster_size, so that
//   out chunk (g*cs + r) = in chunk (g*cs + (r + 1) mod cs).
// "Asynchronous Copies" (TVM TIRx), section Copies between CTAs: a CTA copies
// a shared-memory chunk into another CTA of its thread-block cluster. The
// direction follows the same page's row-shift convention, where each thread
// reads its neighbour (tid + 1).
// Returns 0, or -1 when the sizes do not form whole clusters of whole chunks.
int orc_cluster_exchange(const float* in, float* out, int64_t n, int cluster_size,
                         int64_t chunk_bytes) {
    if (cluster_size < 1 || chunk_bytes < 4 || chunk_bytes % 4 != 0 || n < 0) return -1;
    const int64_t E = chunk_bytes / 4;
    const int64_t cs = cluster_size;
    if (n % (E * cs) != 0) return -1;
    const int64_t chunks = n / E;
    for (int64_t c = 0; c < chunks; ++c) {
        const int64_t group = c / cs;
        const int64_t r = c % cs;
        const int64_t src = group * cs + (r + 1) % cs;
        std::memcpy(out + c * E, in + src * E, (size_t)E * sizeof(float));
    }
    return 0;
}

// Generalised cluster hand-off: clusters of any size, any shift within the
// cluster, and a last group with fewer chunks. The input is cut into chunks of
// chunk_bytes; consecutive runs of cluster_size chunks form groups, the last
// group holding the m = chunks mod cluster_size leftover chunks when that is
// not zero. Within a group of m members, member r receives member
// (r + shift) mod m:
//   out chunk (g*cs + r) = in chunk (g*cs + (r + shift) mod m).
// shift = 1 with whole groups is orc_cluster_exchange. Same page and section
// as above: a CTA copies a chunk into another CTA of its cluster; the library
// extends the fixed neighbour to any distance and to a short last cluster.
// Returns 0, or -1 for sizes that are not whole chunks.
int orc_cluster_exchange_ex(const float* in, float* out, int64_t n, int cluster_size, int64_t chunk_bytes,
                            int64_t shift) {
    if (cluster_size < 1 || chunk_bytes < 4 || chunk_bytes % 4 != 0 || n < 0) return -1;
    const int64_t E = chunk_bytes / 4;
    if (n % E != 0) return -1;
    const int64_t chunks = n / E;
    const int64_t cs = cluster_size;
    for (int64_t c = 0; c < chunks; ++c) {
        const int64_t group = c / cs;
        const int64_t first = group * cs;
        const int64_t left = chunks - first;
        const int64_t m = left < cs ? left : cs;  // members of this group
        const int64_t r = c - first;
        const int64_t s = ((shift % m) + m) % m;
        const int64_t src = first + (r + s) % m;
        std::memcpy(out + c * E, in + src * E, (size_t)E * sizeof(float));
    }
    return 0;
}

// All-to-all inside each group of cluster_size consecutive chunks. Chunk c of
// a group (the CTA of rank c) holds cluster_size equal sub-blocks; sub-block j
// goes to the CTA of rank j, which stores it as sub-block c of its own output
// chunk. With E = chunk_bytes / 4 floats per chunk and B = E / cluster_size
// per sub-block:
//   out[(g*cs + d)*E + r*B + k] = in[(g*cs + r)*E + d*B + k]
// for every group g, receiver d, sender r and 0 <= k < B, i.e. each group is a
// cs x cs matrix of sub-blocks and the result is its block transpose.
// "Asynchronous Copies" (TVM TIRx guide), section Copies between CTAs: a CTA
// bulk-copies shared memory into another CTA of its cluster and the receiver
// waits on its own transaction barrier for the bytes it expects; here every
// CTA sends to every CTA and each receiver expects the bytes of all senders.
// Returns 0, or -1 for sizes that are not whole groups of whole sub-blocks.
int orc_cluster_all_to_all(const float* in, float* out, int64_t n, int cluster_size, int64_t chunk_bytes) {
    if (cluster_size < 1 || chunk_bytes < 4 || chunk_bytes % 4 != 0 || n < 0) return -1;
    const int64_t E = chunk_bytes / 4;
    const int64_t cs = cluster_size;
    if (E % cs != 0 || n % (E * cs) != 0) return -1;
    const int64_t B = E / cs;
    const int64_t groups = n / (E * cs);
    for (int64_t g = 0; g < groups; ++g) {
        for (int64_t d = 0; d < cs; ++d) {
            for (int64_t r = 0; r < cs; ++r) {
                const float* src = in + (g * cs + r) * E + d * B;
                float* dst = out + (g * cs + d) * E + r * B;
                for (int64_t k = 0; k < B; ++k) dst[k] = src[k];
            }
        }
    }
    return 0;
}

// Masked / zero-filling chunk copy over 16-byte chunks. For chunk k with
// code c = codes[k]:
//   c in 0..16  copy the first c bytes of in chunk k, write zeros to the rest
//               of out chunk k (c = 16 is a plain copy, c = 0 all zeros);
//   c == -2     write zeros to the whole out chunk (the source is ignored);
//   c == -1     leave out chunk k unchanged (the copy is predicated off).
// "Asynchronous Copies" (TVM TIRx guide), section A Global-to-Shared Copy: a
// false predicate skips the copy and leaves the destination unchanged, a source
// size copies a byte prefix and zero-fills the rest, and ignoring the source
// zero-fills the whole chunk. Returns 0, or -1 for a code outside -2..16.
int orc_masked_copy(const float* in, float* out, int64_t n_chunks, const signed char* codes) {
    const unsigned char* src = reinterpret_cast<const unsigned char*>(in);
    unsigned char* dst = reinterpret_cast<unsigned char*>(out);
    for (int64_t k = 0; k < n_chunks; ++k) {
        const int c = codes[k];
        if (c < -2 || c > 16) return -1;
        if (c == -1) continue;
        const int keep = c < 0 ? 0 : c;
        for (int b = 0; b < 16; ++b) {
            dst[16 * k + b] = b < keep ? src[16 * k + b] : 0;
        }
    }
    return 0;
}

}  // extern "C"
