// Layout of the per-chunk factor workspace shared by the factor kernel (writer)
// and the tensor-core chunk scan (reader).
//
// One slot per (chunk, V head): the lower-triangular factors
// Tw = diag(exp(G_C - G)) (I + N)^-1 diag(beta) and PTw = P (I + N)^-1 diag(beta)
// (G_C = G of the chunk's last row) and the chunk's gates, fp32:
//   [0, 2304)      Tw   rows packed in 8-float chunks: row t keeps chunks
//                        0 .. t/8 (columns 0 .. 8 (t/8) + 7, zeros right of the diagonal)
//   [2304, 4608)   PTw  same packing
//   [4608, 4672)   G log2(e)   (inclusive running sum of g; padding rows repeat the last)
//   [4672, 4736)   beta        (0 on padding rows)
//   [4736, 4800)   exp(G)
// Chunk c of sequence s lives in slot floor(cu[s] / 64) + s + c; slots of
// different sequences never collide and every slot index is below
// ceil(T_total / 64) + n_seqs.
#pragma once

#include <stdint.h>

namespace gdr {
namespace fac {

constexpr int C = 64;                // tokens per chunk
constexpr int TRI_FLOATS = 2304;     // 8 * sum_t (t/8 + 1)
constexpr int OFF_T = 0;
constexpr int OFF_PT = TRI_FLOATS;
constexpr int OFF_G = 2 * TRI_FLOATS;
constexpr int OFF_BETA = OFF_G + C;
constexpr int OFF_EG = OFF_BETA + C;
constexpr int SLOT_FLOATS = OFF_EG + C;  // 4800
constexpr int SLOT_BYTES = SLOT_FLOATS * 4;  // 19200, a multiple of 16

// First float of row t in a packed triangle.
__host__ __device__ constexpr int tri8_base(int t) {
    return 8 * (4 * (t >> 3) * ((t >> 3) + 1) + (t & 7) * ((t >> 3) + 1));
}
static_assert(tri8_base(64) == TRI_FLOATS, "packed triangle size");
static_assert(SLOT_BYTES % 16 == 0, "slots must keep 16-byte alignment");

__host__ __device__ constexpr int64_t n_slots(int64_t t_total, int64_t n_seqs) {
    return (t_total + C - 1) / C + n_seqs;
}
__host__ __device__ constexpr int64_t slot_base(int64_t seq_start, int64_t s) { return seq_start / C + s; }

}  // namespace fac
}  // namespace gdr
