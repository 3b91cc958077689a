// Layout of the per-chunk factor workspace shared by the factor kernel (writer)
// and the tensor-core chunk scan (reader).
//
// One slot per (chunk, V head), 17 152 bytes, holding the chunk's
// Tw = diag(exp(G_C - G)) (I + N)^-1 diag(beta) and PTw = P (I + N)^-1 diag(beta)
// (G_C = G of the chunk's last row) ready to be the A operand of a tcgen05 MMA:
//   [0, 16384)       the operand tile: 128 rows (Tw rows 0-63, then PTw rows
//                    64-127) of 64 fp16 in the 128-byte-swizzled K-major layout:
//                    16-byte chunk j of row r at r * 128 + 16 (j ^ (r % 8)); zeros
//                    above the diagonal
//   [16384, 16640)   exp(G), 64 fp32 (G: inclusive running sum of g; padding rows
//                    repeat the last)
//   [16640, 17152)   with the fused q/k L2 normalisation: 1 / |k_t| then 1 / |q_t|
//                    (64 fp32 each, |x| = sqrt(sum x^2 + 1e-6)) of the chunk's rows,
//                    the row scales the chunk scan applies; unwritten otherwise
// A bulk copy of the tile to a 1024-byte aligned shared-memory address yields
// the operand as it is.
//
// Chunk c of sequence s lives in slot floor(cu[s] / 64) + s + c; slots of
// different sequences never collide and every slot index is below
// ceil(T_total / 64) + n_seqs.
//
// After the slots (at x_region_offset, 1024-byte aligned) one X tile per
// (slot, QK head): for the slot of chunk c >= 1 of a sequence,
//   X = [K; Q]_c K_{c-1}ᵀ        (128 x 64: the chunk's K rows, then its Q rows,
//                                 against the previous chunk's 64 key tokens)
// as one fp16 tile of 128 rows of 128 bytes in the same 128-byte-swizzled
// K-major layout.  The slot of a sequence's first chunk has no X.
#pragma once

#include <stdint.h>

namespace gdr {
namespace fac {

constexpr int C = 64;                  // tokens per chunk
constexpr int TILE_BYTES = 16384;      // 128 rows x 64 fp16
constexpr int OFF_T = 0;               // bytes
constexpr int OFF_EG = TILE_BYTES;
constexpr int OFF_RK = OFF_EG + C * 4;      // row scales 1 / |k_t|, then 1 / |q_t|
constexpr int GATE_BYTES = 3 * C * 4;       // exp(G), 1 / |k|, 1 / |q|: what the scan copies per chunk
constexpr int SLOT_BYTES = OFF_EG + GATE_BYTES;  // 17152, a multiple of 16
static_assert(SLOT_BYTES % 16 == 0, "slots must keep 16-byte alignment");

// Byte offset of the 16-bit element (row r, column j) in a 128-byte-swizzled
// K-major tile of 128-byte rows.
__host__ __device__ constexpr uint32_t sw128_elem(int r, int j) {
    return (uint32_t)(r * 128 + ((((j >> 3) ^ (r & 7)) & 7) << 4) + (j & 7) * 2);
}

__host__ __device__ constexpr int64_t n_slots(int64_t t_total, int64_t n_seqs) {
    return (t_total + C - 1) / C + n_seqs;
}
__host__ __device__ constexpr int64_t slot_base(int64_t seq_start, int64_t s) { return seq_start / C + s; }

constexpr int X_BYTES = 16384;                // 128 rows x 64 fp16
__host__ __device__ constexpr int64_t x_region_offset(int64_t n_slots_total, int64_t h_v) {
    return (n_slots_total * h_v * SLOT_BYTES + 1023) / 1024 * 1024;
}
__host__ __device__ constexpr int64_t workspace_bytes(int64_t n_slots_total, int64_t h_v, int64_t h_qk) {
    return x_region_offset(n_slots_total, h_v) + n_slots_total * h_qk * X_BYTES;
}

}  // namespace fac
}  // namespace gdr
