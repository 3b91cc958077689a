// Chunk scan of the chunked prefill on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA): carries the state from chunk to chunk, using the
// state-independent factors that the factor kernel stored for every chunk
// beforehand: the gates, Tw = diag(exp(G_C - G)) T diag(beta) and
// PTw = P T diag(beta) with T = (I + N)^-1, and X_c = [K; Q]_{c+1} K_cᵀ.
//
// Shapes: d_k = d_v = 128, 64-token chunks, bf16 q/k/v, fp32 state, fp32 or
// bf16 output.  Four CTAs share one (sequence, V head); CTA `cb` owns state
// columns [32 cb, 32 cb + 32), keeps its 128 x 32 block of the state on chip
// for the whole sequence (fp32 in registers, bf16 hi/lo copies in shared
// memory as MMA operands) and walks the chunks in order.  Per chunk c (the
// chunkwise-parallel form of the Qwen3.5-9B NPU model card, "How it works"),
// with S_c the state before the chunk and gamma_c = G_C its total log decay:
//   A_c   = [K S_c; Q S_c]                          (an accumulator, see below)
//   R     = V - diag(e^G) K S_c
//   MMA2  [D~; P D] = [Tw; PTw] R                   A = [Tw; PTw], B = R (both fp16)
//         (D = T diag(beta) R is the chunk's delta correction, D~ = diag(exp(G_C - G)) D)
//   O     = scale (diag(e^G) Q S_c + P D)
//   MMA3  Y = K_cᵀ D~                                A = Kᵀ, B = [D~_hi | D~_lo]
//   S_c+1 = e^gamma_c S_c + Y
// The next chunk's accumulator is formed by lookahead.  Since
// S_c+1 = e^gamma_c S_c + K_cᵀ D~_c,
//   A_c+1 = [K; Q]_c+1 (e^gamma_c S_c) + X_c D~_c,        X_c = [K; Q]_c+1 K_cᵀ:
// MMA1' (the first term) is issued as soon as S_c is known, in the shadow of
// MMA2, and only MMA_X = X_c D~ (four token k-steps) lies between one chunk's
// D~ and the next chunk's R.  The chunk-to-chunk path is MMA_X, R, MMA2, D~:
// two dependent MMA groups per chunk; MMA3 and the state update run beside it.
// Precision: the state-sized products keep ~2^-16 relative precision: K and Q
// are exact in bf16, and the B operands of MMA1' and MMA3 carry the bf16 hi and
// lo halves of S' and of D~ side by side (N = 64; a tcgen05 MMA of N <= 64
// costs about the same as one of N = 32); the reader adds the two partial
// products.  MMA2 and MMA_X take fp16 operands instead (2^-11 relative
// rounding of Tw, PTw, X, R and D~), one pass of four k-steps each where bf16
// hi/lo splits of both sides needed two (a tcgen05 MMA costs the same in fp16
// as in bf16).  Their fp16 B tiles keep the N = 64 column map with the second
// half zero.  The rounding of Tw and PTw dominates the error this adds: on
// Qwen3.5-9B shapes up to ~1e-2 of the output RMS (max-abs) and ~2.5e-4 of the
// state (relative Frobenius), not growing with the number of chunks, since
// each chunk's rounding enters the state once and decays with it.  The fp16
// range: R and D~ scale with v and the state (the factors do not), so each CTA
// multiplies them by a power of two sigma, chosen once from its first V tile and
// initial state (sigma_exponent), and takes it out where they leave the fp16
// domain (the state update, the outputs): exact, and the relative accuracy no
// longer depends on the data's scale.
//
// Warp roles (448 threads; every role waits only on mbarriers and its own
// named barriers, so no role can stall another's issue):
//   warps 0-7, the "chain": warp w owns TMEM lanes 32 (w % 4) .. + 31 (chunk
//     rows: K/T rows in lanes 0-63, Q/PT rows in lanes 64-127) and columns
//     16 (w / 4) .. + 15 of the CTA's 32.  The warps of lanes 0-63 form R and D~
//     (the chunk-to-chunk path); the others form and store the outputs;
//   warps 8-11, the "loader": own the state (thread i: row i, in registers),
//     update it from Y and write S' while MMA2 runs;
//   warp 12 issues every MMA (converged, one elected lane);
//   warp 13, one thread, issues every copy: K, Q and V tiles three chunks deep
//     by TMA; the [Tw; PTw] and X operand tiles about two chunks ahead and the
//     gates two ahead by bulk copy, prefetched into L2 two chunks before.
// Every mbarrier wait is bounded; on timeout the thread records
// GDR_ERR_DEVICE_TIMEOUT and raises the CTA's abort flag, every role leaves its
// loop at its next wait or role barrier, and the CTA frees its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdr_common.cuh"
#include "gdr_factor_layout.h"
#include "gdr_internal.h"
#include "tc_ptx.cuh"

namespace gdr {

static __device__ int32_t g_device_error;

namespace {

using namespace tc;

constexpr int C = 64;
constexpr int D = 128;
constexpr int BV = 32;           // state columns per CTA
constexpr int NCOL = D / BV;     // CTAs per (sequence, V head)
constexpr int NCHAIN = 256;      // warps 0-7
constexpr int NLOAD = 128;       // warps 8-11
constexpr int NISSUE = 32;       // warp 12
constexpr int NCOPY = 32;        // warp 13
constexpr int NTHREADS = NCHAIN + NLOAD + NISSUE + NCOPY;
constexpr int NKQ = 3;           // K/Q/V ring depth (chunks)
constexpr uint32_t BAR_CHAIN = 1, BAR_LOW = 2, BAR_LOAD = 3, BAR_SIG = 4, BAR_OUT = 5;  // named barriers
constexpr int NLOW = 128;        // chain threads of TMEM lanes 0-63 (warps 0, 1, 4, 5)

// Shared memory map, bytes from a 1024-byte aligned base.
constexpr uint32_t KQ_BYTES = 32768;  // [K rows 0-63; Q rows 64-127] x 2 K-halves, 128-B swizzled rows
constexpr uint32_t V_BYTES = 64 * BV * 2;                 // 64 tokens x 32 columns, 64-B swizzled rows
constexpr uint32_t OFF_KQ = 0;
constexpr uint32_t OFF_V = OFF_KQ + NKQ * KQ_BYTES;
// The operand ring: NOP slots of one 16 KB A-operand tile (K-major 128 x 64 fp16,
// 128-byte swizzled), filled in the order the MMAs read them: per chunk c the
// [Tw; PTw] tile (MMA2), then, unless c is the last chunk, X_c (MMA_X).  Item i
// of that sequence sits in slot i % NOP, so each copy can start as soon as the
// item NOP places earlier has been read: two chunks ahead of its use.  With
// NOP = 4 the item that frees a slot is the previous use of the same full
// barrier (two per kind, by chunk parity), and the issuer has waited for that
// use before issuing the MMAs that free the slot: no full barrier can complete
// a phase its waiter has not yet seen.
constexpr int NOP = 4;
constexpr uint32_t OP_BYTES = 16384;
constexpr uint32_t OFF_OPS = OFF_V + NKQ * V_BYTES;
constexpr uint32_t OFF_S = OFF_OPS + NOP * OP_BYTES;      // [S'_hi | S'_lo]: 128 (k) rows x 64 bf16, MN-major
constexpr uint32_t OFF_R = OFF_S + 16384;                 // [R | 0]: 64 (token) rows x 64 fp16, MN-major
constexpr uint32_t OFF_DT = OFF_R + 8192;                 // [D~ | 0]: 64 rows x 64 fp16
constexpr uint32_t OFF_DT2 = OFF_DT + 8192;               // [D~_hi | D~_lo]: 64 rows x 64 bf16 (MMA3)
// per chunk: exp(G) (64 floats), then, with the fused q/k L2 norm, 1 / |k| and
// 1 / |q| of its rows (64 each): two chunks' worth
constexpr uint32_t OFF_GATES = OFF_DT2 + 8192;
constexpr uint32_t OFF_SMALL = OFF_GATES + 2 * fac::GATE_BYTES;
constexpr uint32_t SM_BARS = OFF_SMALL;                   // NBARS x uint64
constexpr uint32_t SM_TMEM = OFF_SMALL + 192;
constexpr uint32_t SM_ABORT = OFF_SMALL + 200;
constexpr uint32_t SM_SIGMA = OFF_SMALL + 208;   // the operand scale sigma (fp32)
constexpr uint32_t SM_WMAX = OFF_SMALL + 224;    // 4 floats: per K-row warp, max |V_0| and |S_0|
constexpr uint32_t SM_ROWMAX = OFF_SMALL + 256;  // 128 floats: per state row, max |S_0| over the CTA's columns
// The output staging tile: a chunk's 64 rows of the CTA's 32 columns (fp32: 128-byte
// rows; bf16: 64-byte rows), written by the Q / PT-row threads and stored by whole rows.
constexpr uint32_t OFF_OUT = OFF_SMALL + 256 + 512;
constexpr uint32_t SMEM_USED = OFF_OUT + 64 * BV * 4;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for aligning the base
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_V % 1024 == 0 && OFF_OPS % 1024 == 0 && OFF_S % 1024 == 0 &&
                  OFF_R % 1024 == 0 && OFF_DT % 1024 == 0 && OFF_DT2 % 1024 == 0 && OFF_GATES % 16 == 0,
              "operand tiles must be 1 KB aligned, bulk copies 16 B aligned");
static_assert(OFF_OUT % 16 == 0, "16-byte staging rows");

// mbarriers.  Each completes one phase per use; no waiter can fall two phases
// behind (the comments give what orders the next use after every wait).
constexpr int B_KQ_FULL = 0;                // NKQ: K, Q, V tiles landed
constexpr int B_KQ_EMPTY = B_KQ_FULL + NKQ; // NKQ: MMA3 of the chunk done (its tiles free)
constexpr int B_G_FULL = B_KQ_EMPTY + NKQ; // 2: a chunk's gates landed
constexpr int B_G_EMPTY = B_G_FULL + 2;     // 2: chain and loader done with a chunk's gates
constexpr int B_A_FULL = B_G_EMPTY + 2;    // 2: a chunk's [Tw; PTw] tile landed
constexpr int B_X_FULL = B_A_FULL + 2;     // 2: a chunk's X tile landed
constexpr int B_OP_FREE = B_X_FULL + 2;    // NOP: an operand-ring slot's MMAs have read it
constexpr int B_S_READY = B_OP_FREE + NOP; // S_c formed and S' = e^gamma_c S_c written (for MMA1')
constexpr int B_ACC = B_S_READY + 1;        // a chunk's accumulator A_c complete
constexpr int B_MMA2 = B_ACC + 1;           // [D~; P D] ready
constexpr int B_Y = B_MMA2 + 1;             // Kᵀ D~ ready
constexpr int B_SIG = B_Y + 1;              // the operand scale sigma is set (once, chunk 0)
constexpr int NBARS = B_SIG + 1;
static_assert(NBARS * 8 <= 192, "barrier space");

// TMEM columns (fp32 accumulators, lane = row).  Each holds the products of a
// thread's 16 columns in 32 consecutive columns: [hi-part | lo-part] of a bf16
// hi/lo B tile (MMA1', MMA3), which the reader adds, or [product | 0] of an fp16
// B tile (MMA2; MMA_X adds into A's hi part).
constexpr uint32_t TM_ACC = 0;     // + 64 (c % 2): A_c = [K S; Q S] of chunk c
constexpr uint32_t TM_D = 128;     // [D~; P D] = [Tw; PTw] R
constexpr uint32_t TM_Y = 192;     // Kᵀ D~
constexpr uint32_t TM_COLS = 256;  // allocation (a power of two)
constexpr int NLOW_SYNC = NLOW + NISSUE;     // BAR_LOW: the K / T-row threads and the issuing warp
constexpr int NCHAIN_SYNC = NCHAIN + NISSUE; // BAR_CHAIN: the chain and the issuing warp

constexpr uint32_t KQV_TX = 2 * 16384 + V_BYTES;
constexpr long long kWaitLimit = 4000000000LL;  // SM clocks (about 2 s)

constexpr uint32_t IDESC_N64 = idesc_bf16_f32(128, 64, 0, 1);   // MMA1': A K-major, B MN-major
constexpr uint32_t IDESC16_N64 = idesc_f16_f32(128, 64, 0, 1);  // MMA2, MMA_X
constexpr uint32_t IDESC_Y = idesc_bf16_f32(128, 64, 1, 1);     // MMA3: A MN-major (Kᵀ), B MN-major

// One run of the scan over chunks [c_lo, c_hi) of every sequence, from and into
// `state`, writing outputs to `o`; with v_zero the values are taken as zero (the
// run then carries only its initial state).  A launch walks up to kMaxTcRuns
// independent runs side by side (the segments of the two-level scan).
struct TcParams {
    int h_qk, h_v, n_seqs, n_runs;
    int qk_norm;  // fused q/k L2 normalisation: rows of [K S; Q S] and of D~ take the slot's row scales
    float scale;
    const int32_t *cu_seqlens;
    const uint8_t *ws;     // factor slots
    const uint8_t *xs;     // X tiles
    TcRun runs[kMaxTcRuns];
};

struct Ctx {
    uint8_t *sm;
    uint32_t sbase;
    uint32_t tmem;
    volatile int *abort_flag;
    __device__ uint32_t bar(int i) const { return sbase + SM_BARS + 8 * i; }
    __device__ float *fsmall(uint32_t off) const { return reinterpret_cast<float *>(sm + off); }
    __device__ const float *gates(int gb) const {
        return reinterpret_cast<const float *>(sm + OFF_GATES + fac::GATE_BYTES * gb);
    }
};

__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

// Barrier among `count` threads that also ORs a predicate across them.
__device__ __forceinline__ bool named_sync_or(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Bounded wait that also gives up as soon as any thread of the CTA has raised
// the abort flag.  Returns false on either.  It spins on the non-blocking test:
// a phase that has completed is found sooner than by a blocking try_wait, and a
// thread parked by try_wait wakes later after the phase completes than a
// spinning one notices it (the chain's waits are on the chunk-to-chunk path).
__device__ bool wait_or_abort(const Ctx &x, uint32_t bar, uint32_t parity) {
    if (mbar_test_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_test_wait(bar, parity)) return true;
        if (*x.abort_flag) return false;
        if (clock64() - t0 > kWaitLimit) {
            *x.abort_flag = 1;
            atomicCAS(&g_device_error, 0, (int32_t)GDR_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
}

// The operand scale of a CTA, from the largest magnitude M of its first V tile
// and initial state: 1 while M is in [2^-4, 2^13), where the fp16 tiles R and D~
// (which scale with v and the state; the factors do not) keep away from fp16's
// subnormals and its maximum; otherwise the power of two sigma with sigma M in
// [8, 16), so that they sit in the middle of fp16's range whatever the data's
// scale.  Exact: multiplying by a power of two changes no mantissa.  (1 also
// when M is zero, NaN or inf.)
__device__ __forceinline__ int sigma_exponent(float M) {
    if (!(M > 0.f) || !(M <= 3.0e38f)) return 0;
    int e = ((__float_as_int(M) >> 23) & 0xff) - 127;  // floor(log2 M) (M normal)
    if (e >= -4 && e < 13) return 0;
    e = e < -120 ? -120 : (e > 120 ? 120 : e);
    return 3 - e;
}

// This thread's 16 columns of one accumulator ([hi-part | lo-part] in TMEM
// columns [32 g, 32 g + 32)), summed: one TMEM load.
__device__ __forceinline__ void acc_sum1(uint32_t lanebase, uint32_t c0, int j0, float *out) {
    float r[32];
    tmem_ld32(lanebase + c0 + 2 * j0, r);
#pragma unroll
    for (int j = 0; j < 16; ++j) out[j] = r[j] + r[16 + j];
}
// The same for the product of an fp16 B tile: the second 16 columns are zero.
__device__ __forceinline__ void acc_prod(uint32_t lanebase, uint32_t c0, int j0, float *out) {
    tmem_ld16(lanebase + c0 + 2 * j0, out);
}

// Columns j0 .. j0+15 of row `row` of an N = 64 MN-major B operand with
// 128-byte rows: group g = j0 / 16 keeps the hi parts in 16-byte chunks 4g, 4g+1
// and the lo parts in 4g+2, 4g+3 (so each accumulator row has a thread's hi and
// lo partial products in 32 consecutive columns).  The fp16 tiles use chunks
// 4g, 4g+1 alone; 4g+2, 4g+3 stay zero.
__device__ __forceinline__ void store_hilo_row16(uint8_t *tile, int row, int j0, const float *x) {
    const int g4 = (j0 >> 4) * 4;
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
        uint32_t h[4], l[4];
        hilo_words(x + 8 * ch, h, l);
        *reinterpret_cast<uint4 *>(tile + sw128_offset(row, g4 + ch)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4 *>(tile + sw128_offset(row, g4 + 2 + ch)) = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

__device__ __forceinline__ void store_f16_row16(uint8_t *tile, int row, int j0, const float *x) {
    const int g4 = (j0 >> 4) * 4;
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
        const float *w = x + 8 * ch;
        *reinterpret_cast<uint4 *>(tile + sw128_offset(row, g4 + ch)) =
            make_uint4(pack_f16x2(w[0], w[1]), pack_f16x2(w[2], w[3]), pack_f16x2(w[4], w[5]), pack_f16x2(w[6], w[7]));
    }
}

// One ring stage: K and Q (d_k halves, 128-byte swizzled) and this CTA's V columns.
// (With zero values the V tile is not loaded: the chain does not read it.)
__device__ __forceinline__ void issue_kq_loads(const Ctx &x, int kb, int tok, int hq, int h, int cb,
                                               const CUtensorMap *tmK, const CUtensorMap *tmQ,
                                               const CUtensorMap *tmV, bool v_zero) {
    const uint32_t bar = x.bar(B_KQ_FULL + kb);
    mbar_arrive_expect_tx(bar, v_zero ? KQV_TX - V_BYTES : KQV_TX);
    const uint32_t kq = x.sbase + OFF_KQ + kb * KQ_BYTES;
    tma_load_3d(kq, tmK, bar, 0, hq, tok);
    tma_load_3d(kq + 16384, tmK, bar, 64, hq, tok);
    tma_load_3d(kq + 8192, tmQ, bar, 0, hq, tok);
    tma_load_3d(kq + 16384 + 8192, tmQ, bar, 64, hq, tok);
    if (!v_zero) tma_load_3d(x.sbase + OFF_V + kb * V_BYTES, tmV, bar, cb * BV, h, tok);
}

// The barrier that item i's copy completes (item 2 c + 1 is X_c) and the parity
// of its use by chunk c = i / 2.
__device__ __forceinline__ uint32_t op_full_bar(const Ctx &x, int i) {
    return x.bar(((i & 1) ? B_X_FULL : B_A_FULL) + ((i >> 1) & 1));
}
__device__ __forceinline__ uint32_t op_full_parity(int i) { return (uint32_t)(i >> 2) & 1u; }
// Item i of the operand ring: the 16 KB tile at `src` into slot i % NOP.
__device__ __forceinline__ void issue_op_load(const Ctx &x, int i, const uint8_t *src) {
    const uint32_t bar = op_full_bar(x, i);
    mbar_arrive_expect_tx(bar, OP_BYTES);
    bulk_load(x.sbase + OFF_OPS + (i % NOP) * OP_BYTES, src, OP_BYTES, bar);
}
// A slot's exp(G) (64 floats; with the fused L2 norm also its row scales) into
// gates ring buffer gb.
__device__ __forceinline__ void issue_gates_load(const Ctx &x, const uint8_t *slot, int gb, bool qk_norm) {
    const uint32_t bytes = qk_norm ? fac::GATE_BYTES : 256u;
    mbar_arrive_expect_tx(x.bar(B_G_FULL + gb), bytes);
    bulk_load(x.sbase + OFF_GATES + fac::GATE_BYTES * gb, slot + fac::OFF_EG, bytes, x.bar(B_G_FULL + gb));
}
// Operand-ring items: 2 c is the [Tw; PTw] tile of chunk c, 2 c + 1 X_c (only
// while c + 1 < nchunks).
__device__ __forceinline__ bool op_exists(int i, int nchunks) {
    const int c = i >> 1;
    return (i & 1) ? c + 1 < nchunks : c < nchunks;
}

__device__ __forceinline__ uint32_t lane_base(uint32_t tmem, int warp) {
    return tmem + ((uint32_t)((warp & 3) * 32) << 16);
}

// The sequence a CTA takes: the sequences in order of decreasing length (ties by
// index), so that the longest chains start in the first wave of CTAs when a packed
// prefill has more CTAs than SMs (a scheduling simulation of 8 packed sequences of
// 790-8079 tokens: 2.6% off the chunk-scan launch).  For 2..32 sequences each warp
// ranks the lengths with shuffles (every lane of the warp takes part); otherwise
// the sequences go in order.
__device__ __forceinline__ int seq_of_rank(const int32_t *cu, int n_seqs, int r) {
    if (n_seqs <= 1 || n_seqs > 32) return r;
    const int lane = threadIdx.x & 31;
    const int len = lane < n_seqs ? cu[lane + 1] - cu[lane] : -1;
    int rank = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const int lj = __shfl_sync(0xffffffffu, len, j);
        rank += (j < n_seqs && (lj > len || (lj == len && j < lane))) ? 1 : 0;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, lane < n_seqs && rank == r);
    return __ffs(hit) - 1;
}

// ================================ copies ============================================
// Warp 13, one thread: every copy into shared memory, in the order in which the
// chain frees the buffers.  Before the loop: the K/Q/V tiles of chunks 0-2,
// operand items 0-3 (each with an L2 prefetch of the item four places on), the
// gates of chunks 0 and 1.  Per chunk c, in the order the buffers come free:
// chunk c+2's K/Q/V tiles (MMA3 of chunk c-1 issued), [Tw; PTw] of chunk c+2
// (MMA2 of chunk c done), the gates of chunk c+2 (the chain and the loader done
// with chunk c's), X_c+2 (MMA_X of chunk c done).
__device__ void copy_role(const Ctx &x, const TcParams &p, int64_t t0, int nchunks, int64_t slot0, int h,
                          int hq, int cb, const CUtensorMap *tmK, const CUtensorMap *tmQ, const CUtensorMap *tmV,
                          bool v_zero) {
    const uint8_t *fsrc = p.ws + ((size_t)slot0 * p.h_v + h) * fac::SLOT_BYTES;
    const size_t fstride = (size_t)p.h_v * fac::SLOT_BYTES;
    // X tiles of chunk c (X_c = [K; Q]_c+1 K_cᵀ) sit with the slot of chunk c + 1
    const uint8_t *xsrc = p.xs + ((size_t)(slot0 + 1) * p.h_qk + hq) * fac::X_BYTES;
    const size_t xstride = (size_t)p.h_qk * fac::X_BYTES;
    auto op_src = [&](int i) -> const uint8_t * {
        const int c = i >> 1;
        return (i & 1) ? xsrc + c * xstride : fsrc + c * fstride + fac::OFF_T;
    };
    bool bad = false;
    // item i once item i - NOP (same slot) has been read
    auto next_op = [&](int i) {
        if (bad || !op_exists(i, nchunks)) return;
        if (i >= NOP) bad = !wait_or_abort(x, x.bar(B_OP_FREE + i % NOP), (uint32_t)(i / NOP - 1) & 1u);
        if (!bad) issue_op_load(x, i, op_src(i));
        // two chunks ahead; a [Tw; PTw] tile with the slot's exp(G) after it
        if (!bad && op_exists(i + 4, nchunks)) prefetch_l2(op_src(i + 4), (i & 1) ? OP_BYTES : fac::SLOT_BYTES);
    };
    for (int c = 0; c < nchunks && c < NKQ; ++c)
        issue_kq_loads(x, c, (int)(t0 + c * C), hq, h, cb, tmK, tmQ, tmV, v_zero);
    // launched as a programmatic dependent of the factor launch: everything above
    // reads only inputs; the workspace is read after that grid has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int i = 0; i < NOP; ++i) next_op(i);
    for (int c = 0; c < nchunks && c < 2; ++c) issue_gates_load(x, fsrc + c * fstride, c, p.qk_norm != 0);
    for (int c = 0; c < nchunks && !bad; ++c) {
        if (c >= 1 && c - 1 + NKQ < nchunks) {
            const int kb = (c - 1) % NKQ;
            bad = !wait_or_abort(x, x.bar(B_KQ_EMPTY + kb), (uint32_t)((c - 1) / NKQ) & 1u);
            if (!bad) issue_kq_loads(x, kb, (int)(t0 + (c - 1 + NKQ) * C), hq, h, cb, tmK, tmQ, tmV, v_zero);
        }
        next_op(2 * c + NOP);
        if (!bad && c + 2 < nchunks) {
            bad = !wait_or_abort(x, x.bar(B_G_EMPTY + (c & 1)), (uint32_t)(c >> 1) & 1u);
            if (!bad) issue_gates_load(x, fsrc + (c + 2) * fstride, c & 1, p.qk_norm != 0);
        }
        next_op(2 * c + NOP + 1);
    }
}

// ================================ loader ============================================
// The loader warps own the state: thread lt keeps row lt (a d_k index) of the
// CTA's 128 x 32 block in registers, reads its row of each Y = K_cᵀ D~_c from
// TMEM (warp 8 + i reads lanes 32 i .. 32 i + 31) and writes the bf16 hi/lo
// operand S' = e^gamma_c S_c that MMA1' reads.  Per chunk c:
//   S_c = e^gamma_c-1 S_c-1 + Y_c-1 (once MMA3 of chunk c-1 is done; for c = 0,
//   once A_0 has read the S_0 tile), S' = e^gamma_c S_c.
// SC: the CTA's operand scale sigma is not 1 (compile-time, see chain_loop): Y
// comes in units of sigma (D~ does) and S' goes out in them.
template <bool SC>
__device__ __forceinline__ void loader_loop(const Ctx &x, int nchunks, int lt, float *Sg, float (&Sr)[32], float sig,
                                            float isig, bool bad, bool &ok) {
    const uint32_t lb = lane_base(x.tmem, lt >> 5);  // warp 8 + i: lanes 32 i ..
    float eGC_prev = 1.f;  // exp(gamma) of the previous chunk
    for (int c = 0; c < nchunks; ++c) {
        const int gb = c & 1;
        if (!bad) bad = !wait_or_abort(x, x.bar(B_G_FULL + gb), (uint32_t)(c >> 1) & 1u);
        const float eGC = x.gates(gb)[C - 1];
        if (c > 0) {
            if (!bad) bad = !wait_or_abort(x, x.bar(B_Y), (uint32_t)(c - 1) & 1u);
            tc_fence_after_sync();
            if (!bad) {
#pragma unroll
                for (int g2 = 0; g2 < 2; ++g2) {
                    float y[16];
                    acc_sum1(lb, TM_Y, 16 * g2, y);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        Sr[16 * g2 + j] = fmaf(eGC_prev, Sr[16 * g2 + j], SC ? y[j] * isig : y[j]);
                }
            }
        } else if (!bad) {
            bad = !wait_or_abort(x, x.bar(B_ACC), 0u);  // A_0 has read the S_0 tile
        }
        if (!bad && c + 1 < nchunks) {
            const float f = SC ? sig * eGC : eGC;
#pragma unroll
            for (int g2 = 0; g2 < 2; ++g2) {
                float sp[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) sp[j] = f * Sr[16 * g2 + j];
                store_hilo_row16(x.sm + OFF_S, lt, 16 * g2, sp);
            }
            fence_proxy_async_smem();
        }
        tc_fence_before_sync();
        named_sync(BAR_LOAD, NLOAD);
        // every chunk, also the last: the issuer waits for it before MMA3, so Y of this
        // chunk cannot complete before this role has waited for Y of the last; and
        // before it releases this chunk's gates
        if (lt == 0 && !bad) mbar_arrive(x.bar(B_S_READY));
        eGC_prev = eGC;
        if (named_sync_or(BAR_LOAD, NLOAD, bad || *x.abort_flag)) {
            bad = true;
            break;
        }
    }
    // the state after the last chunk
    if (!bad) bad = !wait_or_abort(x, x.bar(B_Y), (uint32_t)(nchunks - 1) & 1u);
    tc_fence_after_sync();
    if (!bad) {
#pragma unroll
        for (int g2 = 0; g2 < 2; ++g2) {
            float y[16];
            acc_sum1(lb, TM_Y, 16 * g2, y);
#pragma unroll
            for (int j = 0; j < 16; ++j) Sr[16 * g2 + j] = fmaf(eGC_prev, Sr[16 * g2 + j], SC ? y[j] * isig : y[j]);
        }
    }
    ok = !bad;
    if (ok && *x.abort_flag == 0) {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4 *>(Sg + j) = make_float4(Sr[j], Sr[j + 1], Sr[j + 2], Sr[j + 3]);
    }
}

// The loader warps own the state (see loader_loop); they first wait for the
// operand scale the chain sets before its loop.
__device__ void loader_role(const Ctx &x, int nchunks, int lt, float *Sg, bool &ok) {
    float Sr[32];  // state row lt, the CTA's 32 columns (S_0 was loaded into the S tile)
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
        const float4 v = *reinterpret_cast<const float4 *>(Sg + j);
        Sr[j] = v.x;
        Sr[j + 1] = v.y;
        Sr[j + 2] = v.z;
        Sr[j + 3] = v.w;
    }
    bool bad = !wait_or_abort(x, x.bar(B_SIG), 0u);
    const float sig = bad ? 1.f : *x.fsmall(SM_SIGMA);
    if (sig == 1.f)
        loader_loop<false>(x, nchunks, lt, Sg, Sr, 1.f, 1.f, bad, ok);
    else
        loader_loop<true>(x, nchunks, lt, Sg, Sr, sig, 1.f / sig, bad, ok);
}

// Row t's 16 outputs (columns j0 .. j0+15 of the CTA's 32) into the staging tile: fp32
// rows of eight 16-byte pieces, bf16 rows of four, the piece index XOR-swizzled by the
// row so that a warp's writes (32 rows, one piece each) and the row-wise reads below
// spread over the banks.
__device__ __forceinline__ void stage_out_row(uint8_t *st, int t, int j0, const float *ov, bool bf16) {
    if (bf16) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int ch = (j0 >> 3) + q;
            const float *w = ov + 8 * q;
            *reinterpret_cast<uint4 *>(st + t * 64 + ((ch ^ ((t >> 1) & 3)) << 4)) =
                make_uint4(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]), pack_bf16x2(w[4], w[5]),
                           pack_bf16x2(w[6], w[7]));
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int ch = (j0 >> 2) + q;
            *reinterpret_cast<float4 *>(st + t * 128 + ((ch ^ (t & 7)) << 4)) =
                make_float4(ov[4 * q], ov[4 * q + 1], ov[4 * q + 2], ov[4 * q + 3]);
        }
    }
}

// The chunk's rows below L from the staging tile to the output, one 16-byte piece per
// thread (q: 0..127 over the Q / PT-row threads) and step: a warp writes four whole
// 128-byte rows (fp32) or eight 64-byte rows (bf16) at a time.  (Stored straight from
// the threads' registers, each warp instruction touched 32 rows at 16 bytes each, and
// the chunk scan took 4% longer.)
__device__ __forceinline__ void store_out_rows(const TcParams &p, const TcRun &run, const uint8_t *st, int64_t c0,
                                               int L, int h, int cb, int q) {
    if (run.out_bf16) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int k = q + 128 * i, r = k >> 2, ch = k & 3;
            if (r < L) {
                const uint4 w = *reinterpret_cast<const uint4 *>(st + r * 64 + ((ch ^ ((r >> 1) & 3)) << 4));
                const size_t off = ((size_t)(c0 + r) * p.h_v + h) * D + cb * BV + ch * 8;
                *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(run.o) + off) = w;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = q + 128 * i, r = k >> 3, ch = k & 7;
            if (r < L) {
                const float4 w = *reinterpret_cast<const float4 *>(st + r * 128 + ((ch ^ (r & 7)) << 4));
                const size_t off = ((size_t)(c0 + r) * p.h_v + h) * D + cb * BV + ch * 4;
                *reinterpret_cast<float4 *>(reinterpret_cast<float *>(run.o) + off) = w;
            }
        }
    }
}

// ================================= issuer ===========================================
// Warp 12 issues every MMA: the whole warp runs the issue code and its waits,
// converged, and one elected lane issues (a lone divergent thread blocks
// several times longer per MMA).  Per chunk c, in the tensor pipe's order:
//   MMA2 (once the K / T-row warps hand it R at BAR_LOW),
//   MMA1' = [K; Q]_c+1 S' into A_c+1 (once the loader has written S'),
//   MMA_X = X_c D~ into A_c+1 and MMA3 = K_cᵀ D~ (once the chain has written
//   D~, read [D~; P D], at BAR_CHAIN).

// [K; Q] (a ring stage) times a [hi | lo] B operand: 8 k-steps over d_k.
__device__ __forceinline__ void issue_kq_times(uint32_t d_tmem, uint32_t kq, uint64_t dB) {
    const uint64_t a0 = smem_desc_sw128(kq, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
        mma_bf16(d_tmem, desc_add(a0, (ks >> 2) * 16384 + (ks & 3) * 32), desc_add(dB, ks * 2048), IDESC_N64,
                 ks > 0);
}

// The EMPTY / FREE commits are made only for buffers that will be filled again.
__device__ void issuer_role(const Ctx &x, int nchunks, int lane) {
    const uint32_t tmem = x.tmem;
    const uint64_t dS = smem_desc(x.sbase + OFF_S, 8192, 1024, kSwizzle128);
    const uint64_t dR = smem_desc(x.sbase + OFF_R, 8192, 1024, kSwizzle128);
    const uint64_t dDT = smem_desc(x.sbase + OFF_DT, 8192, 1024, kSwizzle128);
    const uint64_t dDT2 = smem_desc(x.sbase + OFF_DT2, 8192, 1024, kSwizzle128);
    const uint64_t dOp0 = smem_desc_sw128(x.sbase + OFF_OPS, 16, 1024);
    bool bad = false;  // warp-uniform
    // operand item i (fp16) times the fp16 B tile, four k-steps, into d_tmem: the
    // item is awaited by the whole warp and its slot released once read (if reused)
    auto op_mmas = [&](int i, uint32_t d_tmem, uint64_t dB, bool acc_first) {
        bad = bad || __any_sync(0xffffffffu, !wait_or_abort(x, op_full_bar(x, i), op_full_parity(i)));
        if (bad) return;
        tc_fence_after_sync();
        if (elect_one()) {
            const int slot = i % NOP;
            const uint64_t dA = desc_add(dOp0, slot * OP_BYTES);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(d_tmem, desc_add(dA, ks * 32), desc_add(dB, ks * 2048), IDESC16_N64, acc_first || ks > 0);
            if (op_exists(i + NOP, nchunks)) mma_commit(x.bar(B_OP_FREE + slot));
        }
        __syncwarp();
    };
    // A_0 = [K; Q]_0 [S_hi | S_lo] (the S tile holds S_0)
    bad = __any_sync(0xffffffffu, !wait_or_abort(x, x.bar(B_KQ_FULL + 0), 0u));
    if (!bad) {
        tc_fence_after_sync();
        if (elect_one()) {
            issue_kq_times(tmem + TM_ACC, x.sbase + OFF_KQ, dS);
            mma_commit(x.bar(B_ACC));
        }
        __syncwarp();
    }
    for (int c = 0; c < nchunks; ++c) {
        const int kb = c % NKQ, ab = c & 1;
        const uint32_t par = (uint32_t)c & 1u;
        const bool more = c + 1 < nchunks;
        named_sync(BAR_LOW, NLOW_SYNC);  // R written
        // ---- MMA2: [D~; P D] = [Tw; PTw] R ----------------------------------------------
        op_mmas(2 * c, tmem + TM_D, dR, false);
        if (!bad) {
            if (elect_one()) mma_commit(x.bar(B_MMA2));
            __syncwarp();
        }
        // ---- MMA1': A_c+1 = [K; Q]_c+1 [S'_hi | S'_lo] -------------------------------------
        if (!bad) bad = __any_sync(0xffffffffu, !wait_or_abort(x, x.bar(B_S_READY), par));
        if (more && !bad) {
            bad = __any_sync(0xffffffffu, !wait_or_abort(x, x.bar(B_KQ_FULL + (c + 1) % NKQ),
                                                         (uint32_t)((c + 1) / NKQ) & 1u));
            if (!bad) {
                tc_fence_after_sync();
                if (elect_one())
                    issue_kq_times(tmem + TM_ACC + 64 * (ab ^ 1), x.sbase + OFF_KQ + ((c + 1) % NKQ) * KQ_BYTES, dS);
                __syncwarp();
            }
        }
        // D~ written
        const bool stop = named_sync_or(BAR_CHAIN, NCHAIN_SYNC, bad || *x.abort_flag);
        if (stop) break;
        if (lane == 0) mbar_arrive(x.bar(B_G_EMPTY + (c & 1)));  // the chain has read the gates of chunk c
        // ---- MMA_X: A_c+1 += X_c D~; MMA3: Y = K_cᵀ D~ -----------------------------------
        if (more) op_mmas(2 * c + 1, tmem + TM_ACC + 64 * (ab ^ 1), dDT, true);
        if (!bad) {
            tc_fence_after_sync();
            if (elect_one()) {
                if (more) mma_commit(x.bar(B_ACC));
                const uint64_t a0 = smem_desc_sw128(x.sbase + OFF_KQ + kb * KQ_BYTES, 16384, 1024);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(tmem + TM_Y, desc_add(a0, ks * 2048), desc_add(dDT2, ks * 2048), IDESC_Y, ks > 0);
                mma_commit(x.bar(B_Y));
                // every MMA reading this chunk's tiles is issued
                if (c + NKQ < nchunks) mma_commit(x.bar(B_KQ_EMPTY + kb));
            }
            __syncwarp();
        }
    }
}

// ================================= chain ============================================
// The chunk loop of the chain.  QKN: the fused q/k L2 normalisation (row scales
// from the slots); SC: the CTA's operand scale sigma is not 1 (data outside
// fp16's comfortable range).  Both are compile-time, so the default loop carries
// no code for either.
template <bool QKN, bool SC>
__device__ void chain_loop(const Ctx &x, const TcParams &p, const TcRun &run, int64_t t0, int64_t t1, int nchunks,
                           int h, int cb, int tid, float sig, float isig, bool bad, bool &ok) {
    const int warp = tid >> 5, lane = tid & 31;
    const int j0 = 16 * (warp >> 2);           // this thread's 16 columns of the CTA's 32
    const int row = ((warp & 3) << 5) + lane;  // TMEM lane
    const bool low = row < 64;                 // K / T rows (on the chunk-to-chunk path)
    const int t = row & 63;
    const uint32_t lb = lane_base(x.tmem, warp);
    // every thread runs every named barrier of every chunk; only the CTA-wide
    // stop decided at BAR_CHAIN ends the loop early
    for (int c = 0; c < nchunks; ++c) {
        const int kb = c % NKQ, gb = c & 1, ab = c & 1;
        const int64_t c0 = t0 + (int64_t)c * C;
        const int L = (int)((t1 - c0) < C ? (t1 - c0) : C);
        const uint32_t par = (uint32_t)c & 1u;
        if (!bad) bad = !wait_or_abort(x, x.bar(B_KQ_FULL + kb), (uint32_t)(c / NKQ) & 1u);  // V
        if (!bad) bad = !wait_or_abort(x, x.bar(B_G_FULL + gb), (uint32_t)(c >> 1) & 1u);
        const float egt = x.gates(gb)[t];
        // with the fused L2 norm: this row's scale, 1 / |k_t| (K / T rows) or 1 / |q_t| (Q / PT rows)
        float rsc = 1.f;
        if constexpr (QKN) rsc = x.gates(gb)[(low ? 64 : 128) + t];
        // ---- A_c complete: R = V - e^G K S_c ---------------------------------------------
        if (!bad) bad = !wait_or_abort(x, x.bar(B_ACC), par);
        tc_fence_after_sync();
        float qse[16];  // lanes 64-127: e^G Q S, kept for the output
        {
            float ks[16];
            if (!bad) acc_sum1(lb, TM_ACC + 64 * ab, j0, ks);
            if constexpr (QKN) {
#pragma unroll
                for (int j = 0; j < 16; ++j) ks[j] *= rsc;
            }
            if (low) {
                if (!bad) {
                    // R = V - e^G K S in fp16; with the operand scale, sigma (V - e^G K S)
                    // (A_0 came from the unscaled S_0 tile, every later A is in units of sigma)
                    const uint8_t *vt = x.sm + OFF_V + kb * V_BYTES;
                    const float ea = SC ? -egt * (c == 0 ? sig : 1.f) : -egt;
                    float r[16];
#pragma unroll
                    for (int ch = 0; ch < 2; ++ch) {
                        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                        if (!run.v_zero) load_bf16_chunk64(vt, t, (j0 >> 3) + ch, v);
#pragma unroll
                        for (int e = 0; e < 8; ++e) r[8 * ch + e] = fmaf(ea, ks[8 * ch + e], SC ? sig * v[e] : v[e]);
                    }
                    store_f16_row16(x.sm + OFF_R, t, j0, r);
                    fence_proxy_async_smem();
                }
                tc_fence_before_sync();
                named_sync(BAR_LOW, NLOW_SYNC);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) qse[j] = egt * ks[j];
            }
        }
        // ---- [D~; P D] from MMA2 ----------------------------------------------------------
        if (!bad) bad = !wait_or_abort(x, x.bar(B_MMA2), par);
        tc_fence_after_sync();
        float ov[16];
        {
            float d[16];
            if (!bad) acc_prod(lb, TM_D, j0, d);
            if (low) {
                if (!bad) {
                    // with the fused L2 norm both products take diag(1 / |k|) D~ (K^T of
                    // the normalised keys; X holds the raw keys' products)
                    if constexpr (QKN) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) d[j] *= rsc;
                    }
                    // D~ in fp16 (MMA_X) and as bf16 hi/lo (MMA3)
                    store_f16_row16(x.sm + OFF_DT, t, j0, d);
                    store_hilo_row16(x.sm + OFF_DT2, t, j0, d);
                    fence_proxy_async_smem();
                }
            } else if constexpr (SC) {
                // O = scale (e^G Q S + P D); P D is in units of sigma, so is e^G Q S after chunk 0
                const float fq = p.scale * (c == 0 ? 1.f : isig), fd = p.scale * isig;
#pragma unroll
                for (int j = 0; j < 16; ++j) ov[j] = fmaf(fq, qse[j], fd * d[j]);
            } else {
                // O = scale (e^G Q S + P D)
#pragma unroll
                for (int j = 0; j < 16; ++j) ov[j] = p.scale * (qse[j] + d[j]);
            }
        }
        tc_fence_before_sync();
        const bool stop = named_sync_or(BAR_CHAIN, NCHAIN_SYNC, bad || *x.abort_flag);
        if (stop) {
            bad = true;
            break;
        }
        // outputs of the chunk's real rows (after the barrier, so no proxy fence waits on
        // them), staged and stored by whole rows.  The staging tile is rewritten only after
        // BAR_CHAIN of the next chunk, which every Q / PT-row thread reaches after its reads.
        if (!low) {
            stage_out_row(x.sm + OFF_OUT, t, j0, ov, run.out_bf16 != 0);
            named_sync(BAR_OUT, NCHAIN - NLOW);
            store_out_rows(p, run, x.sm + OFF_OUT, c0, L, h, cb, ((warp >> 2) << 6) | ((warp & 1) << 5) | lane);
        }
    }
    ok = !bad;
}

// Warps 0-7.  Warp w owns TMEM lanes 32 (w % 4) .. + 31 (chunk rows: K/T rows
// in lanes 0-63, Q/PT rows in lanes 64-127) and columns 16 (w / 4) .. + 15 of
// the CTA's 32.  Per chunk: the K / T-row warps form R from A_c and hand it to
// the issuer (BAR_LOW), then write D~ from MMA2's accumulator; the Q / PT-row
// warps form the outputs and store them after the chunk's last barrier.
// Before the loop the K / T-row threads set the CTA's operand scale from the
// first V tile and the initial state's row maxima (every one of them takes part,
// also after an abort, and one publishes it on B_SIG); the Q / PT-row threads
// wait for it.  Then every chain thread runs the loop for that scale.
template <bool QKN>
__device__ void chain_role(const Ctx &x, const TcParams &p, const TcRun &run, int64_t t0, int64_t t1, int nchunks,
                           int h, int cb, int tid, bool &ok) {
    const int warp = tid >> 5, lane = tid & 31;
    const bool low = (warp & 3) < 2;
    const int t = (((warp & 3) << 5) + lane) & 63;
    const int j0 = 16 * (warp >> 2);
    bool bad = false;
    float sig = 1.f;
    if (low) {
        const int kidx = ((warp >> 2) << 6) + ((warp & 3) << 5) + lane;  // 0 .. 127
        float mx = x.fsmall(SM_ROWMAX)[kidx];
        if (!bad) bad = !wait_or_abort(x, x.bar(B_KQ_FULL + 0), 0u);  // the first V tile
        if (!bad && !run.v_zero) {
            float v[16];
            const uint8_t *vt = x.sm + OFF_V;
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) load_bf16_chunk64(vt, t, (j0 >> 3) + ch, v + 8 * ch);
#pragma unroll
            for (int j = 0; j < 16; ++j) mx = fmaxf(mx, fabsf(v[j]));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (lane == 0) x.fsmall(SM_WMAX)[kidx >> 5] = mx;
        named_sync(BAR_SIG, NLOW);
        const float *wm = x.fsmall(SM_WMAX);
        sig = ldexpf(1.f, sigma_exponent(fmaxf(fmaxf(wm[0], wm[1]), fmaxf(wm[2], wm[3]))));
        if (kidx == 0) {
            *x.fsmall(SM_SIGMA) = sig;
            mbar_arrive(x.bar(B_SIG));  // release: the Q / PT-row threads and the state warps read it
        }
    } else {
        if (!bad) bad = !wait_or_abort(x, x.bar(B_SIG), 0u);
        if (!bad) sig = *x.fsmall(SM_SIGMA);
    }
    if (sig == 1.f)
        chain_loop<QKN, false>(x, p, run, t0, t1, nchunks, h, cb, tid, 1.f, 1.f, bad, ok);
    else
        chain_loop<QKN, true>(x, p, run, t0, t1, nchunks, h, cb, tid, sig, 1.f / sig, bad, ok);
}

template <bool QKN>
__device__ __forceinline__ void prefill_tc_body(const CUtensorMap &tmK, const CUtensorMap &tmQ,
                                                const CUtensorMap &tmV, const TcParams &p) {
    extern __shared__ uint8_t smem_raw[];
    Ctx x;
    x.sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    x.sbase = smem_u32(x.sm);
    x.abort_flag = reinterpret_cast<volatile int *>(x.sm + SM_ABORT);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(x.sm + SM_TMEM);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int per_run = p.n_seqs * p.h_v * NCOL;
    const int ri = (int)blockIdx.x / per_run, bi = (int)blockIdx.x % per_run;
    TcRun run = p.runs[0];
#pragma unroll
    for (int i = 1; i < kMaxTcRuns; ++i)  // static indices only: the table stays in the parameter space
        if (i == ri) run = p.runs[i];
    const int cb = bi % NCOL;
    const int h = (bi / NCOL) % p.h_v;
    const int s = seq_of_rank(p.cu_seqlens, p.n_seqs, (bi / NCOL) / p.h_v);
    const int hq = h / (p.h_v / p.h_qk);
    const int64_t ts0 = p.cu_seqlens[s], t1 = p.cu_seqlens[s + 1];
    if (t1 <= ts0) return;  // empty sequence: the state stays as it is
    const int nch_all = (int)((t1 - ts0 + C - 1) / C);
    const int c_end = nch_all < run.c_hi ? nch_all : run.c_hi;
    if (run.c_lo >= c_end) return;  // no chunk of this sequence in this run: its state stays as it is
    const int nchunks = c_end - run.c_lo;
    const int64_t t0 = ts0 + (int64_t)run.c_lo * C;
    const int64_t slot0 = fac::slot_base(ts0, s) + run.c_lo;
    // a programmatic dependent launch queued behind this one (the factors of a
    // later chunk range) may start as soon as every CTA of this grid runs
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (tid == 0) {
        for (int i = 0; i < NBARS; ++i) mbar_init(x.bar(i), 1);
        *x.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_holder), TM_COLS);
        tmem_relinquish();
    }
    // loader thread lt: state row lt (a d_k index), the CTA's 32 columns
    const int lt = tid - NCHAIN;
    const bool loader = lt >= 0 && lt < NLOAD;
    const bool issuer = warp == (NCHAIN + NLOAD) / 32;
    float *Sg = run.state + (((size_t)s * p.h_v + h) * D + (loader ? lt : 0)) * D + cb * BV;
    if (loader) {
        // S_0 into the S tile (the loader role reads its row again into registers)
        float rmax = 0.f;
#pragma unroll
        for (int g2 = 0; g2 < 2; ++g2) {
            float s0[16];
#pragma unroll
            for (int j = 0; j < 16; j += 4) {
                const float4 v = *reinterpret_cast<const float4 *>(Sg + 16 * g2 + j);
                s0[j] = v.x;
                s0[j + 1] = v.y;
                s0[j + 2] = v.z;
                s0[j + 3] = v.w;
            }
            store_hilo_row16(x.sm + OFF_S, lt, 16 * g2, s0);
#pragma unroll
            for (int j = 0; j < 16; ++j) rmax = fmaxf(rmax, fabsf(s0[j]));
        }
        x.fsmall(SM_ROWMAX)[lt] = rmax;  // read by the chain when it sets the operand scale
        fence_proxy_async_smem();
    } else if (tid < NCHAIN) {
        // the zero second halves of the fp16 R and D~ tiles (16 KB, contiguous)
        uint4 *z = reinterpret_cast<uint4 *>(x.sm + OFF_R) + 4 * tid;
#pragma unroll
        for (int i = 0; i < 4; ++i) z[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    x.tmem = *tmem_holder;

    bool ok = true;
    if (tid < NCHAIN)
        chain_role<QKN>(x, p, run, t0, t1, nchunks, h, cb, tid, ok);
    else if (loader)
        loader_role(x, nchunks, lt, Sg, ok);
    else if (issuer)
        issuer_role(x, nchunks, lane);
    else if (lane == 0)
        copy_role(x, p, t0, nchunks, slot0, h, hq, cb, &tmK, &tmQ, &tmV, run.v_zero != 0);

    tc_fence_before_sync();
    __syncthreads();
    if (*x.abort_flag && tid == NCHAIN) {
        // let any tile, factor or X load still in flight land before the shared memory is released
        for (int i = 0; i < NKQ; ++i) {
            mbar_wait_bounded(x.bar(B_KQ_FULL + i), 0, kWaitLimit / 16);
            mbar_wait_bounded(x.bar(B_KQ_FULL + i), 1, kWaitLimit / 16);
        }
        for (int b = B_G_FULL; b < B_G_FULL + 2; ++b) {
            mbar_wait_bounded(x.bar(b), 0, kWaitLimit / 16);
            mbar_wait_bounded(x.bar(b), 1, kWaitLimit / 16);
        }
        for (int b = B_A_FULL; b < B_A_FULL + 4; ++b) {
            mbar_wait_bounded(x.bar(b), 0, kWaitLimit / 16);
            mbar_wait_bounded(x.bar(b), 1, kWaitLimit / 16);
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(x.tmem, TM_COLS);
    }
}

template <bool QKN>
__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmV, TcParams p) {
    prefill_tc_body<QKN>(tmK, tmQ, tmV, p);
}

// ============================ decode blocks (mixed launch) ===========================
// A chunk-scan launch can carry one decode step of another batch (continuous
// batching: prefill chunks and decode steps in one launch).  The blocks after
// the scan's CTAs take the SMs the scan leaves free and walk the batch's
// (sequence, V head) pairs, block j taking pairs j, j + n_blocks, ...  Each
// step is the one-token rule of gdr_decode.cu with the same arithmetic, in the
// same order (so the results are bit-identical to gdr_decode_step's): with
// d = exp(g), y = S^T k, z = S^T q, delta = beta (v - d y),
//     o = scale (d z + (q.k) delta),      S' = d S + k delta^T.
// A block uses the CTA's large shared memory as a ring of three state buffers,
// filled three pairs ahead by bulk copies (the state and the q, k, v rows), and
// splits each pair's work between two warp groups so that consecutive pairs
// overlap: warps 0-7 (thread t: column quad t % 32 of every 8th row) form the
// row groups' partial S^T k and S^T q, sum them through a table, and write
// delta and o; warps 8-13 then write S' = d S + k delta^T of that pair from the
// buffer while warps 0-7 go on to the next pair, and one of them refills the
// buffer once every element has been read.
struct DecBatch {
    int n_pairs;   // batch * h_v (0: no decode blocks)
    int n_blocks;  // decode blocks after the scan's CTAs
    int h_qk, h_v;
    int in_bf16, out_bf16, qk_norm, beta_logits;
    float scale;
    const void *q, *k, *v;
    const float *g, *beta;
    float *state;
    void *o;
};

constexpr int DEC_NBUF = 3;
constexpr int DEC_NT = 256;                          // the reducing group (warps 0-7)
constexpr int DEC_NW = NTHREADS - DEC_NT;            // the writing group (warps 8-13)
constexpr uint32_t DEC_SBYTES = D * D * 4;           // one state
constexpr uint32_t DEC_VEC = 512;                    // room for one q, k or v row (fp32 at most)
constexpr uint32_t DEC_PAR = (D + 4) * 4;            // delta (D floats), then d and 1 / |k|
constexpr uint32_t DEC_BUF = DEC_SBYTES + 3 * DEC_VEC + DEC_PAR;
constexpr uint32_t DEC_OFF_RED = DEC_NBUF * DEC_BUF;           // [8][D] partial sums
constexpr uint32_t DEC_OFF_SMALL = DEC_OFF_RED + 8 * D * 4;    // s_qk, s_rk, s_rq
constexpr uint32_t DEC_OFF_BARS = DEC_OFF_SMALL + 16;          // full[DEC_NBUF], reduced[DEC_NBUF]
constexpr uint32_t DEC_OFF_FLAG = DEC_OFF_BARS + 16 * DEC_NBUF;
constexpr uint32_t DEC_BAR_R = 1, DEC_BAR_W = 2;               // named barriers of the two groups
static_assert(DEC_OFF_FLAG + 16 <= SMEM_USED, "the decode ring fits in the scan's shared memory");
static_assert(DEC_BUF % 16 == 0 && DEC_NW % 32 == 0, "alignment and whole warps");

__device__ __forceinline__ float dec_in(const uint8_t *row, int i, int is_bf16) {
    return is_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(row)[i])
                   : reinterpret_cast<const float *>(row)[i];
}

__device__ __forceinline__ void dec_issue(const DecBatch &d, uint8_t *sm, int buf, int pr) {
    const uint32_t bar = smem_u32(sm + DEC_OFF_BARS + 8 * buf);
    const uint32_t dst = smem_u32(sm + (size_t)buf * DEC_BUF);
    const int b = pr / d.h_v, h = pr - b * d.h_v, hq = h / (d.h_v / d.h_qk);
    const uint32_t rowb = (uint32_t)D * (d.in_bf16 ? 2u : 4u);
    mbar_arrive_expect_tx(bar, DEC_SBYTES + 3 * rowb);
    const uint8_t *S = reinterpret_cast<const uint8_t *>(d.state + (size_t)pr * D * D);
#pragma unroll
    for (uint32_t i = 0; i < 4; ++i) bulk_load(dst + i * 16384u, S + i * 16384u, 16384u, bar);
    const size_t qk_off = ((size_t)b * d.h_qk + hq) * rowb;
    bulk_load(dst + DEC_SBYTES, reinterpret_cast<const uint8_t *>(d.q) + qk_off, rowb, bar);
    bulk_load(dst + DEC_SBYTES + DEC_VEC, reinterpret_cast<const uint8_t *>(d.k) + qk_off, rowb, bar);
    bulk_load(dst + DEC_SBYTES + 2 * DEC_VEC, reinterpret_cast<const uint8_t *>(d.v) + (size_t)pr * rowb, rowb,
              bar);
}

__device__ void decode_blocks(const DecBatch &d, int dblk) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int npairs = dblk < d.n_pairs ? (d.n_pairs - dblk + d.n_blocks - 1) / d.n_blocks : 0;
    float *red = reinterpret_cast<float *>(sm + DEC_OFF_RED);
    float *small = reinterpret_cast<float *>(sm + DEC_OFF_SMALL);
    volatile int *stop = reinterpret_cast<volatile int *>(sm + DEC_OFF_FLAG);
    auto full_bar = [&](int b) { return smem_u32(sm + DEC_OFF_BARS + 8 * b); };
    auto reduced_bar = [&](int b) { return smem_u32(sm + DEC_OFF_BARS + 8 * (DEC_NBUF + b)); };
    const bool producer = tid == DEC_NT;  // the writing group's first thread
    if (producer) {
        for (int i = 0; i < 2 * DEC_NBUF; ++i) mbar_init(smem_u32(sm + DEC_OFF_BARS + 8 * i), 1);
        fence_mbar_init();
        *stop = 0;
        for (int i = 0; i < DEC_NBUF && i < npairs; ++i) dec_issue(d, sm, i, dblk + i * d.n_blocks);
    }
    __syncthreads();
    constexpr int Q4 = D / 4, RSTEP = DEC_NT / Q4, NR = D / RSTEP;
    if (tid < DEC_NT) {
        // ---- the reducing group: partial sums, delta and o of every pair, in order
        const int cq = tid % Q4, rg = tid / Q4;
        for (int i = 0; i < npairs; ++i) {
            const int buf = i % DEC_NBUF, pr = dblk + i * d.n_blocks;
            uint8_t *base = sm + (size_t)buf * DEC_BUF;
            const float4 *sS = reinterpret_cast<const float4 *>(base);
            const uint8_t *qrow = base + DEC_SBYTES, *krow = qrow + DEC_VEC, *vrow = krow + DEC_VEC;
            float *par = reinterpret_cast<float *>(base + DEC_SBYTES + 3 * DEC_VEC);
            const float dgate = __expf(d.g[pr]);
            const float bt = beta_of(d.beta[pr], d.beta_logits);
            if (!mbar_wait_bounded(full_bar(buf), (uint32_t)(i / DEC_NBUF) & 1u, kWaitLimit)) {
                *stop = 1;
                atomicCAS(&g_device_error, 0, (int32_t)GDR_ERR_DEVICE_TIMEOUT);
            }
            named_sync(DEC_BAR_R, DEC_NT);
            if (*stop) break;
            float vv[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) vv[c] = dec_in(vrow, 4 * cq + c, d.in_bf16);
            if (d.qk_norm && warp < 2) {
                const uint8_t *xr = warp == 0 ? krow : qrow;
                float ss = 0.f;
                for (int j = lane; j < D; j += 32) {
                    const float xv = dec_in(xr, j, d.in_bf16);
                    ss = fmaf(xv, xv, ss);
                }
                ss = warp_sum(ss);
                if (lane == 0) small[warp == 0 ? 1 : 2] = l2norm_scale(ss);
            }
            float4 y = make_float4(0.f, 0.f, 0.f, 0.f), z = y;
#pragma unroll
            for (int k = 0; k < NR; ++k) {
                const int r = rg + k * RSTEP;
                const float4 sv = sS[r * Q4 + cq];
                const float kr = dec_in(krow, r, d.in_bf16), qr = dec_in(qrow, r, d.in_bf16);
                y.x = fmaf(sv.x, kr, y.x);
                y.y = fmaf(sv.y, kr, y.y);
                y.z = fmaf(sv.z, kr, y.z);
                y.w = fmaf(sv.w, kr, y.w);
                z.x = fmaf(sv.x, qr, z.x);
                z.y = fmaf(sv.y, qr, z.y);
                z.z = fmaf(sv.z, qr, z.z);
                z.w = fmaf(sv.w, qr, z.w);
            }
            *reinterpret_cast<float4 *>(red + rg * D + 4 * cq) = y;
            if (warp == 0) {
                float pq = 0.f;
                for (int j = lane; j < D; j += 32) pq = fmaf(dec_in(krow, j, d.in_bf16), dec_in(qrow, j, d.in_bf16), pq);
                pq = warp_sum(pq);
                if (lane == 0) small[0] = pq;
            }
            named_sync(DEC_BAR_R, DEC_NT);
            const float rk = d.qk_norm ? small[1] : 1.f, rq = d.qk_norm ? small[2] : 1.f;
            float delta[4], zt[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float ys = 0.f;
#pragma unroll 8
                for (int w = 0; w < RSTEP; ++w) ys += red[w * D + 4 * cq + c];
                delta[c] = bt * (vv[c] - dgate * rk * ys);
            }
            named_sync(DEC_BAR_R, DEC_NT);
            *reinterpret_cast<float4 *>(red + rg * D + 4 * cq) = z;
            named_sync(DEC_BAR_R, DEC_NT);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float zs = 0.f;
#pragma unroll 8
                for (int w = 0; w < RSTEP; ++w) zs += red[w * D + 4 * cq + c];
                zt[c] = rq * zs;
            }
            if (rg == 0) {
                const float qk = small[0] * rq * rk;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    store_out(d.o, (size_t)pr * D + 4 * cq + c, d.scale * fmaf(dgate, zt[c], qk * delta[c]),
                              d.out_bf16);
                    par[4 * cq + c] = delta[c];
                }
                if (cq == 0) {
                    par[D] = dgate;
                    par[D + 1] = rk;
                }
            }
            named_sync(DEC_BAR_R, DEC_NT);  // every read of the table and of `small` is done; delta is written
            if (tid == 0) mbar_arrive(reduced_bar(buf));  // release: delta, d, 1 / |k| for the writing group
        }
    } else {
        // ---- the writing group: S' = d S + k delta^T of every pair, then the refill
        const int wt = tid - DEC_NT;
        for (int i = 0; i < npairs; ++i) {
            const int buf = i % DEC_NBUF, pr = dblk + i * d.n_blocks;
            const uint8_t *base = sm + (size_t)buf * DEC_BUF;
            const float4 *sS = reinterpret_cast<const float4 *>(base);
            const uint8_t *krow = base + DEC_SBYTES + DEC_VEC;
            const float *par = reinterpret_cast<const float *>(base + DEC_SBYTES + 3 * DEC_VEC);
            bool ok = mbar_wait_bounded(reduced_bar(buf), (uint32_t)(i / DEC_NBUF) & 1u, kWaitLimit);
            if (!ok || *stop) {
                if (!ok) atomicCAS(&g_device_error, 0, (int32_t)GDR_ERR_DEVICE_TIMEOUT);
                *stop = 1;
                break;
            }
            const float dgate = par[D], rk = par[D + 1];
            float4 *Sg = reinterpret_cast<float4 *>(d.state + (size_t)pr * D * D);
            for (int e = wt; e < D * Q4; e += DEC_NW) {
                const int r = e / Q4, cq = e - r * Q4;
                const float4 sv = sS[e];
                const float4 dl = *reinterpret_cast<const float4 *>(par + 4 * cq);
                const float kr = rk * dec_in(krow, r, d.in_bf16);
                __stcs(&Sg[e], make_float4(fmaf(dgate, sv.x, kr * dl.x), fmaf(dgate, sv.y, kr * dl.y),
                                           fmaf(dgate, sv.z, kr * dl.z), fmaf(dgate, sv.w, kr * dl.w)));
            }
            named_sync(DEC_BAR_W, DEC_NW);  // every read of this buffer is done
            if (producer && i + DEC_NBUF < npairs) dec_issue(d, sm, buf, dblk + (i + DEC_NBUF) * d.n_blocks);
        }
    }
    __syncthreads();
    if (producer && *stop) {
        // let the copies in flight land before the shared memory is released
        for (int b = 0; b < DEC_NBUF; ++b) {
            mbar_wait_bounded(full_bar(b), 0, kWaitLimit / 16);
            mbar_wait_bounded(full_bar(b), 1, kWaitLimit / 16);
        }
    }
}

template <bool QKN>
__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_tc_mixed_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmV, TcParams p, DecBatch d) {
    const int n_scan = p.n_runs * p.n_seqs * p.h_v * NCOL;
    if ((int)blockIdx.x >= n_scan) {
        decode_blocks(d, (int)blockIdx.x - n_scan);
        return;
    }
    prefill_tc_body<QKN>(tmK, tmQ, tmV, p);
}

}  // namespace

cudaError_t launch_prefill_tc_runs(const Args &a, const TcRun *runs, int n_runs, const float *ws, cudaStream_t s,
                                   bool overlap, const Args *dec, int dec_blocks) {
    if (a.n_seqs == 0 || a.t_total == 0 || n_runs == 0) return cudaSuccess;  // nothing to walk
    if (dec && (dec->n_seqs <= 0 || dec_blocks <= 0 || dec->d != D)) return cudaErrorInvalidValue;
    if (n_runs < 0 || n_runs > kMaxTcRuns) return cudaErrorInvalidValue;
    CUtensorMap tmK, tmQ, tmV;
    if (!encode_bf16_3d(&tmK, a.k, D, (uint64_t)a.h_qk, (uint64_t)a.t_total, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_bf16_3d(&tmQ, a.q, D, (uint64_t)a.h_qk, (uint64_t)a.t_total, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_bf16_3d(&tmV, a.v, D, (uint64_t)a.h_v, (uint64_t)a.t_total, BV, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(prefill_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SMEM_BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(prefill_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)SMEM_BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(prefill_tc_mixed_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)SMEM_BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(prefill_tc_mixed_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    TcParams p = {};
    p.h_qk = a.h_qk;
    p.h_v = a.h_v;
    p.n_seqs = a.n_seqs;
    p.n_runs = n_runs;
    p.qk_norm = a.qk_norm;
    p.scale = a.scale;
    p.cu_seqlens = a.cu_seqlens;
    p.ws = reinterpret_cast<const uint8_t *>(ws);
    p.xs = reinterpret_cast<const uint8_t *>(ws) + fac::x_region_offset(fac::n_slots(a.t_total, a.n_seqs), a.h_v);
    for (int i = 0; i < n_runs; ++i) p.runs[i] = runs[i];
    cudaLaunchConfig_t cfg = {};
    const unsigned n_scan = (unsigned)n_runs * (unsigned)a.n_seqs * (unsigned)a.h_v * (unsigned)NCOL;
    cfg.gridDim = dim3(n_scan + (dec ? (unsigned)dec_blocks : 0u));
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = overlap ? &attr : nullptr;
    cfg.numAttrs = overlap ? 1 : 0;
    if (dec) {
        DecBatch d = {};
        d.n_pairs = dec->n_seqs * dec->h_v;
        d.n_blocks = dec_blocks;
        d.h_qk = dec->h_qk;
        d.h_v = dec->h_v;
        d.in_bf16 = dec->in_bf16;
        d.out_bf16 = dec->out_bf16;
        d.qk_norm = dec->qk_norm;
        d.beta_logits = dec->beta_logits;
        d.scale = dec->scale;
        d.q = dec->q;
        d.k = dec->k;
        d.v = dec->v;
        d.g = dec->g;
        d.beta = dec->beta;
        d.state = dec->state;
        d.o = dec->o;
        return a.qk_norm ? cudaLaunchKernelEx(&cfg, prefill_tc_mixed_kernel<true>, tmK, tmQ, tmV, p, d)
                         : cudaLaunchKernelEx(&cfg, prefill_tc_mixed_kernel<false>, tmK, tmQ, tmV, p, d);
    }
    return a.qk_norm ? cudaLaunchKernelEx(&cfg, prefill_tc_kernel<true>, tmK, tmQ, tmV, p)
                     : cudaLaunchKernelEx(&cfg, prefill_tc_kernel<false>, tmK, tmQ, tmV, p);
}

cudaError_t launch_prefill_tc(const Args &a, const float *ws, cudaStream_t s, bool overlap, const Args *dec,
                              int dec_blocks) {
    TcRun run = {};
    run.c_lo = a.c_lo;
    run.c_hi = a.c_hi;
    run.out_bf16 = a.out_bf16;
    run.v_zero = 0;
    run.state = a.state;
    run.o = a.o;
    return launch_prefill_tc_runs(a, &run, 1, ws, s, overlap, dec, dec_blocks);
}

int32_t *device_error_word() {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess) return nullptr;
    return reinterpret_cast<int32_t *>(ptr);
}

cudaError_t read_clear_device_error(cudaStream_t s, int32_t *code) {
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    int32_t v = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v));
    if (e != cudaSuccess) return e;
    if (v != 0) {
        const int32_t zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    }
    *code = v;
    return e;
}

}  // namespace gdr
