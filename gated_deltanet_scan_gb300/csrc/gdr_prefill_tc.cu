// Chunk scan of the chunked prefill on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA): carries the state from chunk to chunk, using the
// state-independent factors that the factor kernel stored for every chunk
// beforehand: the gates and Tw = diag(exp(G_C - G)) T diag(beta),
// PTw = P T diag(beta), with T = (I + N)^-1.
//
// Shapes: d_k = d_v = 128, 64-token chunks, bf16 q/k/v, fp32 state, fp32 or
// bf16 output.  Four CTAs share one (sequence, V head); CTA `cb` owns state
// columns [32 cb, 32 cb + 32), keeps its 128 x 32 block of the state on chip
// for the whole sequence (fp32 in registers, bf16 hi/lo copies in shared
// memory as MMA operands) and walks the chunks in order.  Per chunk (the
// chunkwise-parallel form of the Qwen3.5-9B NPU model card, "How it works"):
//   MMA1  [K S; Q S] = [K; Q] S                      A = K/Q tile, B = [S_hi | S_lo]
//   R     = V - diag(e^G) K S
//   MMA2  [D~; P D] = [Tw; PTw] R                    A = [Tw; PTw]_hi and _lo, B = [R_hi | R_lo]
//         (D = T diag(beta) R is the chunk's delta correction, D~ = diag(exp(G_C - G)) D)
//   O     = scale (diag(e^G) Q S + P D)
//   MMA3  Y = Kᵀ D~                                  A = Kᵀ, B = [D~_hi | D~_lo]
//   S    <- exp(G_C) S + Y
// A tcgen05 MMA of N <= 64 costs the same as one of N = 32 (about 50 cycles of
// issue each), so each B operand carries its bf16 hi and lo halves side by side
// (N = 64) and the partial products are summed when the accumulator is read:
// every product that feeds the state keeps ~2^-16 relative precision with
// 8 + 8 + 4 MMAs per chunk, all issued by one thread into one accumulator per
// group (more issuing threads, each with its own accumulator, measured slower:
// the readers' extra TMEM loads and sums cost more than the issue they save).
//
// Warp roles (384 threads).  Warps 0-7, the "chain": warp w owns TMEM lanes
// 32 (w % 4) .. + 31 (state rows, or chunk rows: K/T rows in lanes 0-63, Q/PT
// rows in lanes 64-127) and columns 16 (w / 4) .. + 15 of the CTA's 32.  Only
// warps of lanes 0-63 sit on the chunk-to-chunk path between MMA1 and MMA3;
// the others form the outputs meanwhile, and lane 0 of warp 2 issues every
// MMA (so no K/T-row warp ever waits behind an MMA issue).  Warps 8-11, the "loader": one
// thread issues the TMA loads (K, Q and V tiles three chunks deep, factor
// slots two deep); all four unpack a chunk's packed fp32 [T; PT] into the
// bf16 hi/lo operand tiles while the chain runs the chunk before.  Every
// mbarrier wait is bounded; on timeout the thread records
// GDR_ERR_DEVICE_TIMEOUT, raises the CTA's abort flag, and both roles leave
// their loops together at their next role barrier.
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
constexpr int NTHREADS = NCHAIN + NLOAD;
constexpr int NKQ = 3;           // K/Q/V ring depth (chunks)
constexpr int NF = 2;            // factor ring depth (chunks)
constexpr uint32_t BAR_CHAIN = 1, BAR_LOW = 2, BAR_LOAD = 3;  // named barriers
constexpr int NLOW = 128;        // chain threads of TMEM lanes 0-63 (warps 0, 1, 4, 5)

// Shared memory map, bytes from a 1024-byte aligned base.
constexpr uint32_t KQ_BYTES = 32768;  // [K rows 0-63; Q rows 64-127] x 2 K-halves, 128-B swizzled rows
constexpr uint32_t V_BYTES = 64 * BV * 2;                 // 64 tokens x 32 columns, 64-B swizzled rows
constexpr uint32_t OFF_KQ = 0;
constexpr uint32_t OFF_V = OFF_KQ + NKQ * KQ_BYTES;
constexpr uint32_t OFF_F = OFF_V + NKQ * V_BYTES;         // factor slots (fac::SLOT_BYTES each)
constexpr uint32_t OFF_ATP = ((OFF_F + NF * fac::SLOT_BYTES + 1023) / 1024) * 1024;
constexpr uint32_t OFF_ATP_LO = OFF_ATP + 16384;          // [T; PT] hi / lo, K-major 128 x 64 bf16
constexpr uint32_t OFF_S = OFF_ATP + 32768;               // [S_hi | S_lo]: 128 (k) rows x 64 bf16, MN-major
constexpr uint32_t OFF_R = OFF_S + 16384;                 // [R_hi | R_lo]: 64 (token) rows x 64 bf16
constexpr uint32_t OFF_DT = OFF_R + 8192;                 // [D~_hi | D~_lo]: 64 rows x 64 bf16
constexpr uint32_t OFF_SMALL = OFF_DT + 8192;
constexpr uint32_t SM_BARS = OFF_SMALL;                   // NBARS x uint64
constexpr uint32_t SM_TMEM = OFF_SMALL + 192;
constexpr uint32_t SM_ABORT = OFF_SMALL + 200;
constexpr uint32_t SMEM_USED = OFF_SMALL + 256;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for aligning the base
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_V % 1024 == 0 && OFF_ATP % 1024 == 0 && OFF_S % 1024 == 0 && OFF_R % 1024 == 0 &&
                  OFF_DT % 1024 == 0 && OFF_F % 16 == 0,
              "operand tiles must be 1 KB aligned, bulk copies 16 B aligned");

// mbarriers
constexpr int B_KQ_FULL = 0;                // NKQ: K, Q, V tiles landed
constexpr int B_KQ_EMPTY = B_KQ_FULL + NKQ; // NKQ: chain done with the tiles
constexpr int B_F_FULL = B_KQ_EMPTY + NKQ;  // NF: factor slot landed
constexpr int B_F_EMPTY = B_F_FULL + NF;    // NF: chain done with the slot (its gates)
constexpr int B_ATP_FULL = B_F_EMPTY + NF;  // [T; PT] operand tiles unpacked
constexpr int B_ATP_FREE = B_ATP_FULL + 1;  // MMA2 has read them
// MMA1, MMA2, MMA3 each complete one phase of their own barrier per chunk, so a
// warp that reaches a wait late can never see a later group's phase instead.
constexpr int B_MMA1 = B_ATP_FREE + 1, B_MMA2 = B_MMA1 + 1, B_MMA3 = B_MMA2 + 1;
constexpr int NBARS = B_MMA3 + 1;
static_assert(NBARS * 8 <= 192, "barrier space");

// TMEM columns (fp32 accumulators, lane = row).  Each holds [hi-part | lo-part]
// products of a thread's 16 columns in 32 consecutive columns; readers add the
// two halves.
constexpr uint32_t TM_KS = 0;    // [K S; Q S]
constexpr uint32_t TM_D = 64;    // [D; P D] = [T; PT]_hi R + [T; PT]_lo R
constexpr uint32_t TM_Y = 128;   // Kᵀ D~
constexpr uint32_t TM_COLS = 256;  // allocation (a power of two)
constexpr int ISSUE_WARP = 2;          // lane 0 issues every MMA; a Q / PT-row warp (TMEM lanes 64-95)
constexpr int NLOW_SYNC = NLOW + 32;  // BAR_LOW: the K / T-row threads and the issuing warp

constexpr uint32_t KQV_TX = 2 * 16384 + V_BYTES;
constexpr long long kWaitLimit = 4000000000LL;  // SM clocks (about 2 s)

constexpr uint32_t IDESC_N64 = idesc_bf16_f32(128, 64, 0, 1);  // A K-major, B MN-major
constexpr uint32_t IDESC_Y = idesc_bf16_f32(128, 64, 1, 1);    // A MN-major (Kᵀ), B MN-major

struct TcParams {
    int h_qk, h_v, out_bf16;
    int c_lo, c_hi;  // chunks of each sequence to process; the state is read before and written after them
    float scale;
    const int32_t *cu_seqlens;
    const float *ws;  // factor slots
    float *state;
    void *o;
};

struct Ctx {
    uint8_t *sm;
    uint32_t sbase;
    uint32_t tmem;
    volatile int *abort_flag;
    __device__ uint32_t bar(int i) const { return sbase + SM_BARS + 8 * i; }
    __device__ const float *fslot(int fb) const {
        return reinterpret_cast<const float *>(sm + OFF_F + fb * fac::SLOT_BYTES);
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
// the abort flag.  Returns false on either.
__device__ bool wait_or_abort(const Ctx &x, uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*x.abort_flag) return false;
        if (clock64() - t0 > kWaitLimit) {
            *x.abort_flag = 1;
            atomicCAS(&g_device_error, 0, (int32_t)GDR_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
}

// This thread's 16 columns of one accumulator ([hi-part | lo-part] in TMEM
// columns [32 g, 32 g + 32)), summed: one TMEM load.
__device__ __forceinline__ void acc_sum1(uint32_t lanebase, uint32_t c0, int j0, float *out) {
    float r[32];
    tmem_ld32(lanebase + c0 + 2 * j0, r);
#pragma unroll
    for (int j = 0; j < 16; ++j) out[j] = r[j] + r[16 + j];
}

// Columns j0 .. j0+15 of row `row` of an N = 64 MN-major B operand with
// 128-byte rows: group g = j0 / 16 keeps the hi parts in 16-byte chunks 4g, 4g+1
// and the lo parts in 4g+2, 4g+3 (so each accumulator row has a thread's hi and
// lo partial products in 32 consecutive columns).
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

__device__ __forceinline__ void issue_kq_loads(const Ctx &x, int kb, int tok, int hq, int h, int cb,
                                               const CUtensorMap *tmK, const CUtensorMap *tmQ,
                                               const CUtensorMap *tmV) {
    const uint32_t bar = x.bar(B_KQ_FULL + kb);
    mbar_arrive_expect_tx(bar, KQV_TX);
    const uint32_t kq = x.sbase + OFF_KQ + kb * KQ_BYTES;
    tma_load_3d(kq, tmK, bar, 0, hq, tok);
    tma_load_3d(kq + 16384, tmK, bar, 64, hq, tok);
    tma_load_3d(kq + 8192, tmQ, bar, 0, hq, tok);
    tma_load_3d(kq + 16384 + 8192, tmQ, bar, 64, hq, tok);
    tma_load_3d(x.sbase + OFF_V + kb * V_BYTES, tmV, bar, cb * BV, h, tok);
}

__device__ __forceinline__ void issue_factor_load(const Ctx &x, int fb, const float *src) {
    const uint32_t bar = x.bar(B_F_FULL + fb);
    mbar_arrive_expect_tx(bar, fac::SLOT_BYTES);
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            x.sbase + OFF_F + fb * fac::SLOT_BYTES),
        "l"(reinterpret_cast<uint64_t>(src)), "r"((uint32_t)fac::SLOT_BYTES), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint32_t lane_base(uint32_t tmem, int warp) {
    return tmem + ((uint32_t)((warp & 3) * 32) << 16);
}

// ================================ loader ============================================
// One thread issues every TMA; all 128 unpack [T; PT] (packed fp32 triangles)
// into the hi/lo K-major operand tiles.  Rows t and 63 - t of T (or of PT)
// hold 9 chunks of 8 between them; two threads share each such pair, 5 and 4
// chunks, so every thread does the same work.  Chunks right of a row's
// diagonal chunk stay zero from the start.
__device__ void loader_role(const Ctx &x, const TcParams &p, int64_t t0, int nchunks, int64_t slot0, int h,
                            int hq, int cb, const CUtensorMap *tmK, const CUtensorMap *tmQ,
                            const CUtensorMap *tmV, int lt) {
    const float *fsrc = p.ws + ((size_t)slot0 * p.h_v + h) * fac::SLOT_FLOATS;
    const size_t fstride = (size_t)p.h_v * fac::SLOT_FLOATS;
    if (lt == 0) {
        for (int c = 0; c < nchunks && c < NKQ; ++c) issue_kq_loads(x, c, (int)(t0 + c * C), hq, h, cb, tmK, tmQ, tmV);
        for (int c = 0; c < nchunks && c < NF; ++c) issue_factor_load(x, c, fsrc + c * fstride);
    }
    const int pr = lt >> 1, hf = lt & 1;
    const int ta = pr & 31, tb = 63 - ta, nch_a = (ta >> 3) + 1;
    const int mat = pr < 32 ? fac::OFF_T : fac::OFF_PT, rbase = pr < 32 ? 0 : 64;
    uint8_t *hi = x.sm + OFF_ATP, *lo = x.sm + OFF_ATP_LO;
    for (int c = 0; c < nchunks; ++c) {
        const int fb = c % NF;
        bool bad = !wait_or_abort(x, x.bar(B_F_FULL + fb), (uint32_t)(c / NF) & 1u);
        if (c > 0 && !bad) bad = !wait_or_abort(x, x.bar(B_ATP_FREE), (uint32_t)(c - 1) & 1u);
        if (!bad) {
            const float *f = x.fslot(fb) + mat;
#pragma unroll
            for (int i = 0; i < 5; ++i) {
                const int k = 5 * hf + i;
                if (k < 9) {
                    const bool in_a = k < nch_a;
                    const int t = in_a ? ta : tb, j = in_a ? k : k - nch_a;
                    const float *src = f + fac::tri8_base(t) + 8 * j;
                    const float4 u = *reinterpret_cast<const float4 *>(src);
                    const float4 v = *reinterpret_cast<const float4 *>(src + 4);
                    const float xv[8] = {u.x, u.y, u.z, u.w, v.x, v.y, v.z, v.w};
                    uint32_t hw[4], lw[4];
                    hilo_words(xv, hw, lw);
                    const uint32_t off = sw128_offset(rbase + t, j);
                    *reinterpret_cast<uint4 *>(hi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4 *>(lo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
            }
            fence_proxy_async_smem();
        }
        named_sync(BAR_LOAD, NLOAD);
        if (lt == 0 && !bad) {
            mbar_arrive(x.bar(B_ATP_FULL));
            // refill the ring slots the chain released with chunk c-1
            if (c >= 1) {
                const int kb = (c - 1) % NKQ, pf = (c - 1) % NF;
                if (c - 1 + NKQ < nchunks) {
                    bad = !wait_or_abort(x, x.bar(B_KQ_EMPTY + kb), (uint32_t)((c - 1) / NKQ) & 1u);
                    if (!bad) issue_kq_loads(x, kb, (int)(t0 + (c - 1 + NKQ) * C), hq, h, cb, tmK, tmQ, tmV);
                }
                if (!bad && c - 1 + NF < nchunks) {
                    bad = !wait_or_abort(x, x.bar(B_F_EMPTY + pf), (uint32_t)((c - 1) / NF) & 1u);
                    if (!bad) issue_factor_load(x, pf, fsrc + (c - 1 + NF) * fstride);
                }
            }
        }
        if (named_sync_or(BAR_LOAD, NLOAD, bad || *x.abort_flag)) break;
    }
}

// Row t of chunk c0 of the output (16 columns at j0 of the CTA's block).
__device__ __forceinline__ void store_out_row(const TcParams &p, int64_t c0, int t, int h, int cb, int j0,
                                              const float *ov) {
    const size_t off = ((size_t)(c0 + t) * p.h_v + h) * D + cb * BV + j0;
    if (p.out_bf16) {
        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.o) + off);
#pragma unroll
        for (int j = 0; j < 16; j += 8)
            dst[j / 8] = make_uint4(pack_bf16x2(ov[j], ov[j + 1]), pack_bf16x2(ov[j + 2], ov[j + 3]),
                                    pack_bf16x2(ov[j + 4], ov[j + 5]), pack_bf16x2(ov[j + 6], ov[j + 7]));
    } else {
        float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.o) + off);
#pragma unroll
        for (int j = 0; j < 16; j += 4) dst[j / 4] = make_float4(ov[j], ov[j + 1], ov[j + 2], ov[j + 3]);
    }
}

// ================================= chain ============================================
// One thread, lane 0 of warp 2, issues every MMA.  That warp holds Q / PT rows,
// which are off the chunk-to-chunk path: the K / T-row warps never wait behind
// an MMA issue, and the issuing warp joins the K / T-row barrier (BAR_LOW) that
// hands it R and D~.  It stores a chunk's outputs only after the next chunk's
// MMA1 has been issued (global stores ahead of it delay the issue).
__device__ void chain_role(const Ctx &x, const TcParams &p, int64_t t0, int64_t t1, int nchunks, int h,
                           int cb, float *Sr, int tid, bool &ok) {
    const int warp = tid >> 5, lane = tid & 31;
    const int j0 = 16 * (warp >> 2);           // this thread's 16 columns of the CTA's 32
    const int row = ((warp & 3) << 5) + lane;  // TMEM lane
    const bool low = row < 64;                 // K / T rows (on the chunk-to-chunk path)
    const int t = row & 63;
    const bool iwarp = warp == ISSUE_WARP;     // joins BAR_LOW
    const bool issuer = iwarp && lane == 0;
    const uint32_t lb = lane_base(x.tmem, warp);
    const uint32_t tmem = x.tmem;
    const uint64_t dS = smem_desc(x.sbase + OFF_S, 8192, 1024, kSwizzle128);
    const uint64_t dR = smem_desc(x.sbase + OFF_R, 8192, 1024, kSwizzle128);
    const uint64_t dDT = smem_desc(x.sbase + OFF_DT, 8192, 1024, kSwizzle128);
    const uint64_t dAh = smem_desc_sw128(x.sbase + OFF_ATP, 16, 1024);
    const uint64_t dAl = smem_desc_sw128(x.sbase + OFF_ATP_LO, 16, 1024);
    bool bad = false;
    float ov[16];      // lanes 64-127: a chunk's outputs, stored after its last barrier
    int64_t ov_c0 = 0; // first token of the chunk whose outputs ov holds
    int ov_len = 0;    // its number of real rows (0: nothing pending)
    for (int c = 0; c < nchunks; ++c) {
        const int kb = c % NKQ, fb = c % NF;
        const int64_t c0 = t0 + (int64_t)c * C;
        const int L = (int)((t1 - c0) < C ? (t1 - c0) : C);
        const uint32_t kq = x.sbase + OFF_KQ + kb * KQ_BYTES;
        const uint32_t par = (uint32_t)c & 1u;
        bad = !wait_or_abort(x, x.bar(B_KQ_FULL + kb), (uint32_t)(c / NKQ) & 1u);
        // ---- MMA1: [K S; Q S] = [K; Q] [S_hi | S_lo], 8 k-steps over d_k ----------------
        if (issuer && !bad) {
            tc_fence_after_sync();
            const uint64_t a0 = smem_desc_sw128(kq, 16, 1024);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16(tmem + TM_KS, desc_add(a0, (ks >> 2) * 16384 + (ks & 3) * 32), desc_add(dS, ks * 2048),
                         IDESC_N64, ks > 0);
            mma_commit(x.bar(B_MMA1));
        }
        if (iwarp && t < ov_len) store_out_row(p, ov_c0, t, h, cb, j0, ov);
        if (!bad) bad = !wait_or_abort(x, x.bar(B_F_FULL + fb), (uint32_t)(c / NF) & 1u);
        const float *egs = x.fslot(fb) + fac::OFF_EG;  // exp(G)
        const float egt = egs[t], eGC = egs[C - 1];
        if (issuer && !bad) bad = !wait_or_abort(x, x.bar(B_ATP_FULL), par);
        if (!bad) bad = !wait_or_abort(x, x.bar(B_MMA1), par);
        tc_fence_after_sync();
        float qse[16];  // lanes 64-127: e^G Q S, kept for the output
        {
            float ks[16];
            if (!bad) acc_sum1(lb, TM_KS, j0, ks);
            if (low) {
                if (!bad) {
                    // R = V - e^G K S as [R_hi | R_lo]
                    const uint8_t *vt = x.sm + OFF_V + kb * V_BYTES;
                    float r[16];
#pragma unroll
                    for (int ch = 0; ch < 2; ++ch) {
                        float v[8];
                        load_bf16_chunk64(vt, t, (j0 >> 3) + ch, v);
#pragma unroll
                        for (int e = 0; e < 8; ++e) r[8 * ch + e] = fmaf(-egt, ks[8 * ch + e], v[e]);
                    }
                    store_hilo_row16(x.sm + OFF_R, t, j0, r);
                    fence_proxy_async_smem();
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) qse[j] = egt * ks[j];
            }
        }
        if (low || iwarp) {
            tc_fence_before_sync();
            named_sync(BAR_LOW, NLOW_SYNC);
        }
        // ---- MMA2: [D~; P D] = [Tw; PTw]_hi [R_hi | R_lo] + [Tw; PTw]_lo [R_hi | R_lo] -----
        if (issuer && !bad) {
            tc_fence_after_sync();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16(tmem + TM_D, desc_add(ks < 4 ? dAh : dAl, (ks & 3) * 32), desc_add(dR, (ks & 3) * 2048),
                         IDESC_N64, ks > 0);
            mma_commit(x.bar(B_MMA2));
            mma_commit(x.bar(B_ATP_FREE));
        }
        if (!bad) bad = !wait_or_abort(x, x.bar(B_MMA2), par);
        tc_fence_after_sync();
        {
            float d[16];
            if (!bad) acc_sum1(lb, TM_D, j0, d);
            if (low) {
                if (!bad) {
                    // D~ as [D~_hi | D~_lo]
                    store_hilo_row16(x.sm + OFF_DT, t, j0, d);
                    fence_proxy_async_smem();
                }
            } else {
                // O = scale (e^G Q S + P D)
#pragma unroll
                for (int j = 0; j < 16; ++j) ov[j] = p.scale * (qse[j] + d[j]);
            }
        }
        if (low || iwarp) {
            tc_fence_before_sync();
            named_sync(BAR_LOW, NLOW_SYNC);
        }
        // ---- MMA3: Y = Kᵀ [D~_hi | D~_lo], 4 token k-steps ------------------------------
        if (issuer && !bad) {
            tc_fence_after_sync();
            const uint64_t a0 = smem_desc_sw128(kq, 16384, 1024);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(tmem + TM_Y, desc_add(a0, ks * 2048), desc_add(dDT, ks * 2048), IDESC_Y, ks > 0);
            mma_commit(x.bar(B_MMA3));
        }
        if (!bad) bad = !wait_or_abort(x, x.bar(B_MMA3), par);
        tc_fence_after_sync();
        if (!bad) {
            // S <- exp(G_C) S + Kᵀ D~, and its [S_hi | S_lo] operand copy
            float y[16];
            acc_sum1(lb, TM_Y, j0, y);
#pragma unroll
            for (int j = 0; j < 16; ++j) Sr[j] = fmaf(eGC, Sr[j], y[j]);
            store_hilo_row16(x.sm + OFF_S, row, j0, Sr);
            fence_proxy_async_smem();
        }
        tc_fence_before_sync();
        const bool stop = named_sync_or(BAR_CHAIN, NCHAIN, bad || *x.abort_flag);
        if (tid == 0 && !stop) {
            mbar_arrive(x.bar(B_KQ_EMPTY + kb));
            mbar_arrive(x.bar(B_F_EMPTY + fb));
        }
        if (stop) {
            bad = true;
            break;
        }
        // outputs of the chunk's real rows (after the barrier, so no proxy fence waits on them)
        if (!low && !iwarp && t < L) store_out_row(p, c0, t, h, cb, j0, ov);
        ov_c0 = c0;
        ov_len = L;
    }
    if (!bad && iwarp && t < ov_len) store_out_row(p, ov_c0, t, h, cb, j0, ov);
    ok = !bad;
}

__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmV, TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    Ctx x;
    x.sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    x.sbase = smem_u32(x.sm);
    x.abort_flag = reinterpret_cast<volatile int *>(x.sm + SM_ABORT);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(x.sm + SM_TMEM);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cb = blockIdx.x % NCOL;
    const int h = (blockIdx.x / NCOL) % p.h_v;
    const int s = (blockIdx.x / NCOL) / p.h_v;
    const int hq = h / (p.h_v / p.h_qk);
    const int64_t ts0 = p.cu_seqlens[s], t1 = p.cu_seqlens[s + 1];
    if (t1 <= ts0) return;  // empty sequence: the state stays as it is
    const int nch_all = (int)((t1 - ts0 + C - 1) / C);
    const int c_end = nch_all < p.c_hi ? nch_all : p.c_hi;
    if (p.c_lo >= c_end) return;  // no chunk of this sequence in this launch: its state stays as it is
    const int nchunks = c_end - p.c_lo;
    const int64_t t0 = ts0 + (int64_t)p.c_lo * C;
    const int64_t slot0 = fac::slot_base(ts0, s) + p.c_lo;
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
    // chain thread: state row `srow` (a d_k index), columns [j0, j0 + 16) of the CTA's block
    const int srow = ((warp & 3) << 5) + lane, j0 = 16 * ((warp >> 2) & 1);
    float Sr[16];
    float *Sg = p.state + (((size_t)s * p.h_v + h) * D + srow) * D + cb * BV + j0;
    if (tid < NCHAIN) {
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(Sg + j);
            Sr[j] = v.x;
            Sr[j + 1] = v.y;
            Sr[j + 2] = v.z;
            Sr[j + 3] = v.w;
        }
        store_hilo_row16(x.sm + OFF_S, srow, j0, Sr);
        fence_proxy_async_smem();
    } else {
        // [T; PT] operand tiles: zero once (right of each row's diagonal chunk stays zero)
        for (int i = tid - NCHAIN; i < 32768 / 16; i += NLOAD)
            reinterpret_cast<uint4 *>(x.sm + OFF_ATP)[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    x.tmem = *tmem_holder;

    bool ok = true;
    if (tid < NCHAIN)
        chain_role(x, p, t0, t1, nchunks, h, cb, Sr, tid, ok);
    else
        loader_role(x, p, t0, nchunks, slot0, h, hq, cb, &tmK, &tmQ, &tmV, tid - NCHAIN);

    if (tid < NCHAIN) {
        if (ok && *x.abort_flag == 0) {
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                *reinterpret_cast<float4 *>(Sg + j) = make_float4(Sr[j], Sr[j + 1], Sr[j + 2], Sr[j + 3]);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (*x.abort_flag && tid == NCHAIN) {
        // let any tile or factor load still in flight land before the shared memory is released
        for (int i = 0; i < NKQ; ++i) {
            mbar_wait_bounded(x.bar(B_KQ_FULL + i), 0, kWaitLimit / 16);
            mbar_wait_bounded(x.bar(B_KQ_FULL + i), 1, kWaitLimit / 16);
        }
        for (int i = 0; i < NF; ++i) {
            mbar_wait_bounded(x.bar(B_F_FULL + i), 0, kWaitLimit / 16);
            mbar_wait_bounded(x.bar(B_F_FULL + i), 1, kWaitLimit / 16);
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(x.tmem, TM_COLS);
    }
}

}  // namespace

cudaError_t launch_prefill_tc(const Args &a, const float *ws, cudaStream_t s) {
    if (a.n_seqs == 0 || a.t_total == 0) return cudaSuccess;  // every sequence empty: state unchanged
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
        e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    TcParams p;
    p.h_qk = a.h_qk;
    p.h_v = a.h_v;
    p.out_bf16 = a.out_bf16;
    p.c_lo = a.c_lo;
    p.c_hi = a.c_hi;
    p.scale = a.scale;
    p.cu_seqlens = a.cu_seqlens;
    p.ws = ws;
    p.state = a.state;
    p.o = a.o;
    const unsigned grid = (unsigned)a.n_seqs * (unsigned)a.h_v * (unsigned)NCOL;
    prefill_tc_kernel<<<grid, NTHREADS, SMEM_BYTES, s>>>(tmK, tmQ, tmV, p);
    return cudaGetLastError();
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
