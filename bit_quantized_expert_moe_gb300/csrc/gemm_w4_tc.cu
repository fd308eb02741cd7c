// Stage 3, prefill regime: grouped W4A16 GEMM on the 5th-generation tensor
// cores (tcgen05, TMEM accumulators, TMA).
//
// "Performance and verification", section "Why it is fast": a prompt's
// expert products are batched into grouped tensor-core GEMMs; "Measured
// results", section Speed: prompts run fastest with the 4-bit weights widened
// to 16-bit for a dense GEMM.  Here the dequantisation happens tile by tile on
// chip, never in HBM: the widened weights go from registers straight into
// tensor memory, where the MMA reads its A operand.
//
// Shapes (swap-AB: weight rows are the MMA's M, tokens its N):
//   D[m][n] = sum_k A[m][k] * B[n][k]     M = 256 weight rows, N <= 256 tokens
//   A = dequantised weights (fp16, written by the dequant warps into tensor
//       memory: lane = row, a 32-bit column = two consecutive K elements)
//   B = activation rows of one expert segment (fp16, TMA, SW128 K-major)
// The GEMM runs on CTA pairs (2-SM clusters, tcgen05 cta_group::2): each CTA
// dequantises its own 128 weight rows into its own tensor memory and loads
// half of the token tile, one or two threads of the even CTA issue the pair's
// MMAs, and each CTA drains its 128 rows of the accumulator.  Per 64 K an SM
// then receives 16 KB of activations and 4 KB of codes (36 KB for one CTA
// alone): the rate at which an SM's copies land, not the tensor pipe, bounded
// the one-CTA kernel.
// The pipeline moves in units of 128 K (two 64-K sub-stages, one scale
// group): one barrier round, one copy of codes, one copy of activations and
// one wait per unit.  The shared-memory ring holds one unit more than tensor
// memory holds A units, so the copies are issued one unit earlier.
// The operands are fp16 rather than bf16: bf16 activations convert to fp16
// exactly inside fp16's range (values outside set the error word), and a
// weight is q s - fl16(z s) rounded once to fp16, which keeps 3 more bits than
// bf16 would.  Both operands hold K interleaved in groups of 8 (k8_interleave),
// the order in which the dequantisation takes a packed word apart.
// A work item is (token tile of one expert, pair of 128-row weight blocks);
// CTA rank r of the pair takes block 2 j + r of the item's pair j.  A
// persistent pair walks items pair, pair + pairs, ...
//
// gate_up: the 128 A rows of a block hold 64 gate rows and the 64 matching up
// rows, interleaved by 16 inside each 32-lane TMEM quarter, so one thread's
// lane and the lane 16 above it carry gate and up of the same feature; the
// epilogue pairs them with one shuffle and writes h = SiLU(g) * u (fp16).
// down: 128 consecutive rows of W2; the epilogue writes y rows (fp16 for the
// layer's own combine, bf16 when y is the caller's output).
//
// Warp roles (896 threads per CTA): 0 TMA producer, 1 TMEM owner and (even
// CTA) MMA issuer 0, 2 (even CTA) MMA issuer 1, 3 idle, 4-11 dequantisation
// (warp w: TMEM lane quarter w % 4, half (w - 4) / 4 of each sub-stage's K),
// 12-27 epilogue (warp w: lane quarter w % 4, every fourth 32-column block).
// With one accumulator the next item's MMAs wait until both CTAs' epilogues
// have read it, so four warps per quarter cut that wait.
// Barriers: each CTA's copies land on its own full[u]; both CTAs' dequant
// warps arrive on the even CTA's afull[a] and both epilogues on its
// accempty; MMA completion (empty[u], aempty[a], accfull, done) is signalled
// to both CTAs at once.
// TMEM: the fp32 accumulator in columns 0..255, A unit a in columns
// 256 + 64 a .. + 63 (the same columns in both CTAs).
// Every wait is bounded in time; a timeout sets the error word, every role
// leaves its loop, in-flight copies and MMAs are drained, and both CTAs meet
// before TMEM is freed.
#include <cstdio>

#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;                  // A rows per CTA (256 per pair)
constexpr int BK = 64;                   // K per sub-stage: one 128-byte swizzle row of fp16
constexpr int UK = 2 * BK;               // K per pipeline unit (= the scale group)
constexpr int BN = TILE_ROWS;            // max tokens per item (256)
constexpr int B_BYTES = BN / 2 * BK * 2; // 16 KB: one CTA's half of the token tile, one sub-stage
constexpr int P_BYTES = BM * UK / 2;     // 8 KB of packed codes per unit
constexpr int UNIT_BYTES = 2 * B_BYTES + P_BYTES;
// A CTA's half of the token tile arrives in one copy: a box of 64 rows when
// the half is at most 64 rows, else of 128 (an SM's copies land at a limited
// rate of operations, not only of bytes)
constexpr int B_BOX_ROWS = 64;
constexpr int B_BOX_BYTES = B_BOX_ROWS * BK * 2;
constexpr int THREADS = 896;
constexpr int DQ_WARP0 = 4, DQ_WARPS = 8;
constexpr int EP_WARP0 = 12, EP_WARPS = 16;
constexpr uint32_t TMEM_COLS = 512;      // accumulator (256 columns) + 4 A units of 64 columns
constexpr uint32_t A_COL0 = 256;         // first TMEM column of A unit 0
constexpr uint32_t A_UNIT_COLS = UK / 2;
constexpr int A_UNITS = 4;
constexpr int MAX_UNITS = 6;
constexpr uint32_t SPLIT_N = BN / 2;     // tiles of at most this many tokens split K between two MMA issuers
constexpr size_t BAR_BYTES = 512;        // barriers (8 (2 SU + 2 A_UNITS + 9) bytes), TMEM slot, abort flag

struct TcParams {
    int E, d, f, R;
    int K;        // reduction length (d for gate_up, f for down)
    int NFB;      // 128-row weight blocks per expert (even: taken in pairs)
    const uint16_t* wsc;   // scales [E * rows_per_expert][K/128]
    const uint16_t* wz;    // zeros
    const Tile* tiles;
    const DevPlan* plan;
    uint16_t* out;         // h [R][f] (fp16) or y [R][d]
    int out_ld;            // f or d
    int out_f16;           // down: 1 = fp16 y, 0 = bf16 y
    const float* row_w;
    uint32_t* err;
};

__host__ __device__ constexpr size_t scale_bytes(int K) { return (size_t)2 * 2 * BM * (K / 128) * 2; }
__host__ __device__ constexpr size_t tc_smem_bytes(int SU, int K) {
    return (size_t)SU * UNIT_BYTES + scale_bytes(K) + BAR_BYTES + 1024;
}

// Item -> expert, token rows and this CTA's weight block (rank 0 / 1 of the pair).
template <bool GATEUP>
__device__ __forceinline__ void item_rows(const TcParams& p, int item, int& e, int& row0, int& nrows,
                                          int& fb) {
    const int npb = p.NFB >> 1;
    const int ti = item / npb;
    fb = 2 * (item - ti * npb) + (int)tc::cluster_ctarank();
    const Tile t = p.tiles[ti];
    e = t.expert;
    row0 = t.row0;
    nrows = t.nrows;
}

// Global weight row of A row r of block fb of expert e.
template <bool GATEUP>
__device__ __forceinline__ size_t a_global_row(const TcParams& p, int e, int fb, int r) {
    if (GATEUP) {
        const int q = r >> 5, i = r & 31;
        const size_t base = (size_t)e * 2 * p.f + (size_t)fb * 64 + 16 * q;
        return (i < 16) ? base + i : base + p.f + (i - 16);
    } else {
        return (size_t)e * p.d + (size_t)fb * BM + r;
    }
}

// Row of a unit's packed-code buffer that holds A row r.
template <bool GATEUP>
__device__ __forceinline__ int a_packed_row(int r) {
    if (GATEUP) {
        const int q = r >> 5, i = r & 31;
        return (i < 16) ? 16 * q + i : 64 + 16 * q + (i - 16);
    } else {
        return r;
    }
}

// Wait that ignores the abort flag (used to drain in-flight work at teardown).
__device__ __forceinline__ void mbar_drain_wait(uint32_t bar, uint32_t parity, uint32_t* err) {
    if (tc::mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = globaltimer_ns();
    while (!tc::mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > tc::WAIT_LIMIT_NS) { set_error(err, ERRBIT_TIMEOUT); return; }
    }
}

template <bool GATEUP, int SU>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
tc_grouped_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                  const __grid_constant__ CUtensorMap map_x2, TcParams p) {
    static_assert(SU <= MAX_UNITS && A_COL0 + A_UNIT_COLS * A_UNITS <= TMEM_COLS, "A units exceed tensor memory");
    constexpr int NBAR = 2 * SU + 2 * A_UNITS + 9;
    static_assert(8 * NBAR + 8 <= BAR_BYTES, "barrier area too small");
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* gbase = smem_raw + (base - raw);

    // shared memory: per unit slot two 16 KB activation sub-stages (128B-swizzled
    // K-major), then the units' codes ([128 rows][16 words]), the scales and zeros,
    // the barriers
    const uint32_t sB = base;
    const uint32_t sP = base + SU * 2 * B_BYTES;
    const int G = p.K / 128;
    uint16_t* sScale = reinterpret_cast<uint16_t*>(gbase + SU * UNIT_BYTES);  // [2][BM][G]
    uint16_t* sZero = sScale + 2 * BM * G;                                    // [2][BM][G]
    const uint32_t bars = base + SU * UNIT_BYTES + (uint32_t)scale_bytes(p.K);
    // barrier layout: full[SU], empty[SU], afull[A_UNITS], aempty[A_UNITS], accfull[2],
    // accempty[2], done, qsync[4] (one accumulator: only accfull[0] and accempty[0] are used)
    const uint32_t bar_full = bars, bar_empty = bars + 8 * SU, bar_afull = bars + 16 * SU;
    const uint32_t bar_aempty = bar_afull + 8 * A_UNITS, bar_accfull = bar_aempty + 8 * A_UNITS;
    const uint32_t bar_accempty = bar_accfull + 16, bar_done = bar_accempty + 16;
    const uint32_t bar_qsync = bar_done + 8;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + SU * UNIT_BYTES + scale_bytes(p.K) + 8 * NBAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NU = p.K / UK;  // units per item (even: K is a multiple of 256)
    const uint32_t rank = tc::cluster_ctarank();
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int n_items = p.plan->n_tiles * (p.NFB >> 1);

    if (threadIdx.x == 0) {
        // afull and accempty count both CTAs' warps (only the even CTA's are used)
        for (int u = 0; u < SU; ++u) {
            tc::mbar_init(bar_full + 8 * u, 1);
            tc::mbar_init(bar_empty + 8 * u, 1);
        }
        for (int a = 0; a < A_UNITS; ++a) {
            tc::mbar_init(bar_afull + 8 * a, 2 * DQ_WARPS);
            tc::mbar_init(bar_aempty + 8 * a, 1);
        }
        // accfull and done: one commit from each of the two MMA issuers
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(bar_accfull + 8 * b, 2);
            tc::mbar_init(bar_accempty + 8 * b, 2 * EP_WARPS);
        }
        tc::mbar_init(bar_done, 2);
        for (int q4 = 0; q4 < 4; ++q4) tc::mbar_init(bar_qsync + 8 * q4, 2);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc_pair(smem_u32((const void*)tmem_slot), TMEM_COLS);
        tc::tmem_relinquish_pair();
    }
    // both CTAs' barriers are initialised and the tensor memory allocated
    // before either CTA signals the other
    tc::tc_fence_before();
    tc::cluster_sync();
    tc::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the even CTA's afull[0] and accempty in the cluster's shared window
    const uint32_t afull_lead = tc::mapa_shared(bar_afull, 0), accempty_lead = tc::mapa_shared(bar_accempty, 0);

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            tc::tma_prefetch_desc(&map_w);
            tc::tma_prefetch_desc(&map_x);
            tc::tma_prefetch_desc(&map_x2);
            int gu = 0;  // units issued so far
            uint32_t issued_mask = 0, issued_phase = 0;  // per unit slot: last issued phase parity
            bool ok = true;
            for (int item = pair; ok && item < n_items; item += npairs) {
                int e, row0, nrows, fb;
                item_rows<GATEUP>(p, item, e, row0, nrows, fb);
                // this CTA's half of the MMA's N (nrows rounded up to 16)
                const int half = ceil_div(nrows, 16) * 8;
                const int brow0 = row0 + (int)rank * half;
                const bool big = half > B_BOX_ROWS;
                const int wrow_a = e * p.d + fb * BM;  // down: first weight row of the block
                for (int ku = 0; ku < NU; ++ku, ++gu) {
                    const int u = gu % SU;
                    const uint32_t pu = (uint32_t)(gu / SU) & 1u;
                    if (!tc::mbar_wait(bar_empty + 8 * u, pu ^ 1, abort_flag, p.err)) { ok = false; break; }
                    const uint32_t fbar = bar_full + 8 * u;
                    tc::mbar_arrive_expect_tx(fbar, P_BYTES + 2 * (big ? 2 : 1) * B_BOX_BYTES);
                    const uint32_t dp = sP + u * P_BYTES;
                    // the unit's 128 rows of codes in one box: gate_up's 64 gate and
                    // 64 up rows (3D map over the expert halves), down's 128 rows
                    if (GATEUP)
                        tc::tma_load_3d(dp, &map_w, fbar, ku * (UK / 8), fb * 64, 2 * e);
                    else
                        tc::tma_load_2d(dp, &map_w, fbar, ku * (UK / 8), wrow_a);
                    const uint32_t db = sB + u * 2 * B_BYTES;
                    // both sub-stages of the activation half in one box of a 3D view
                    // {64 K, rows, K / 64}: the box lands as two 128B-swizzled tiles
                    // of 64 (half <= 64, tiles 8 KB apart) or 128 rows (16 KB apart)
                    tc::tma_load_3d(db, big ? &map_x2 : &map_x, fbar, 0, brow0, ku * 2);
                    issued_mask |= 1u << u;
                    issued_phase = (issued_phase & ~(1u << u)) | (pu << u);
                }
            }
            // drain: every issued unit's copies must have landed before exit
            for (int u = 0; u < SU; ++u)
                if (issued_mask >> u & 1u) mbar_drain_wait(bar_full + 8 * u, (issued_phase >> u) & 1u, p.err);
        }
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------- MMA issuers (even CTA of the pair)
        // Issuer 0 (warp 1) takes every unit of a tile of more than 128
        // tokens.  A tile of at most 128 tokens splits its K between the two
        // issuers, alternate units each, into accumulators in columns 0.. and
        // 128.. that the epilogue adds: at small N the issue of the MMAs, not
        // the tensor pipe, bounds a unit, and two issuers double it.
        const int iss = warp - 1;
        if (lane == 0 && rank == 0) {
            int ic = 0;
            bool ok = true;
            for (int item = pair, g = 0; ok && item < n_items; item += npairs, ++ic, g += NU) {
                int e, row0, nrows, fb;
                item_rows<GATEUP>(p, item, e, row0, nrows, fb);
                const int N = ceil_div(nrows, 16) * 16;
                const bool split = N <= SPLIT_N;
                const uint32_t idesc = tc::idesc_f16_f32(2 * BM, N);
                // both CTAs' epilogues have read the accumulator
                if (!tc::mbar_wait_cluster(bar_accempty, (ic & 1) ^ 1, abort_flag, p.err)) { ok = false; break; }
                tc::tc_fence_after();
                if (split || iss == 0) {
                    const uint32_t d_tmem = tmem_base + (split ? SPLIT_N * (uint32_t)iss : 0u);
                    const int ku0 = split ? iss : 0;
                    for (int ku = ku0; ku < NU; ku += split ? 2 : 1) {
                        const int gu = g + ku, a = gu % A_UNITS, u = gu % SU;
                        // both CTAs' A of the unit are in tensor memory, which
                        // also means both CTAs' copies of the unit have landed
                        if (!tc::mbar_wait_cluster(bar_afull + 8 * a, (uint32_t)(gu / A_UNITS) & 1u, abort_flag, p.err)) {
                            ok = false;
                            break;
                        }
                        tc::tc_fence_after();
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t a0 = tmem_base + A_COL0 + A_UNIT_COLS * a + BK / 2 * h;
                            // the second sub-stage follows the first: 64 rows (8 KB)
                            // later for halves of at most 64 rows, else 128 (16 KB)
                            const uint32_t b0 = sB + u * 2 * B_BYTES + h * (split ? B_BYTES / 2 : B_BYTES);
#pragma unroll
                            for (int ks = 0; ks < BK / 16; ++ks) {
                                tc::mma_f16_tmem_a_pair(d_tmem, a0 + 8 * ks, tc::sw128_kmajor_desc(b0 + ks * 32), idesc,
                                                        !(ku == ku0 && h == 0 && ks == 0));
                            }
                        }
                        tc::mma_commit_pair(bar_empty + 8 * u);
                        tc::mma_commit_pair(bar_aempty + 8 * a);
                    }
                }
                if (!ok) break;
                tc::mma_commit_pair(bar_accfull);
            }
            // drain: every issued MMA completes (in both CTAs) before TMEM is released
            if (pair < n_items) {
                tc::mma_commit_pair(bar_done);
                mbar_drain_wait(bar_done, 0, p.err);
            }
        } else if (lane == 0 && iss == 0 && pair < n_items) {
            // odd CTA: its tensor and shared memory stay in use until the
            // even CTA's last MMAs have completed
            mbar_drain_wait(bar_done, 0, p.err);
        }
    } else if (warp >= DQ_WARP0 && warp < DQ_WARP0 + DQ_WARPS) {
        // ------------------------------------------------------ dequantisers
        // Warp w owns A row r = 32 (w % 4) + lane (its TMEM lane) and half
        // hk = (w - 4) / 4 of every sub-stage's K: 4 packed words (32 codes)
        // per sub-stage, widened in registers and stored as 16 TMEM columns.  The two
        // warps of a lane quarter share its rows' scales and zeros: warp hk
        // prefetches array hk (scales, zeros) of the next item into the other
        // half of a double buffer (4-byte cp.async).  They meet on a named
        // mbarrier at every item start, after which both are done with the
        // previous item's buffer (the one the next prefetch overwrites), and
        // again once both copies of this item have landed.  Every wait is
        // bounded and warp-uniform, so a warp whose partner gave up leaves too.
        const int q = warp & 3, hk = (warp - DQ_WARP0) >> 2;
        const int r = 32 * q + lane;
        const int prow = a_packed_row<GATEUP>(r);
        const uint32_t t_lane = (uint32_t)(32 * q) << 16;
        const uint32_t qbar = bar_qsync + 8 * q;  // the quarter's two warps meet here
        uint32_t qphase = 0;
        auto quarter_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(qbar);
            const bool r = tc::mbar_wait(qbar, qphase, abort_flag, p.err);
            qphase ^= 1u;
            return __all_sync(0xffffffffu, r);
        };
        uint16_t* const s_dst = hk ? sZero : sScale;
        const uint16_t* const s_src = hk ? p.wz : p.wsc;
        auto prefetch_scales = [&](int item, int buf) {
            int e, row0, nrows, fb;
            item_rows<GATEUP>(p, item, e, row0, nrows, fb);
            const int pairs = G / 2;
            for (int idx = lane; idx < 32 * pairs; idx += 32) {
                const int rr = 32 * q + idx / pairs, gp = idx % pairs;
                const size_t grow = a_global_row<GATEUP>(p, e, fb, rr);
                cp_async4(smem_u32(s_dst + ((size_t)buf * BM + rr) * G + 2 * gp), s_src + grow * G + 2 * gp);
            }
        };
        int gu = 0;  // units consumed so far
        int ic = 0;
        bool ok = true;
        if (pair < n_items) prefetch_scales(pair, 0);
        cp_async_commit();
        for (int item = pair; ok && item < n_items; item += npairs, ++ic) {
            const int sbuf = ic & 1;
            // both warps are done with the buffer the next prefetch overwrites
            if (!quarter_sync()) break;
            if (item + npairs < n_items) prefetch_scales(item + npairs, sbuf ^ 1);
            cp_async_commit();
            cp_async_wait<1>();
            // both warps' copies of this item's scales and zeros have landed
            if (!quarter_sync()) break;
            for (int ku = 0; ku < NU; ++ku, ++gu) {
                const int u = gu % SU, a = gu % A_UNITS;
                // the unit's copies have landed and the MMAs that read A unit a
                // the previous time have completed
                ok = tc::mbar_wait(bar_full + 8 * u, (uint32_t)(gu / SU) & 1u, abort_flag, p.err) &&
                     tc::mbar_wait(bar_aempty + 8 * a, ((uint32_t)(gu / A_UNITS) & 1u) ^ 1u, abort_flag, p.err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                // as f16x2: (s, s) and (-fl16(z s), -fl16(z s)) of this row's group ku
                const size_t si = ((size_t)sbuf * BM + r) * G + ku;
                const uint32_t sb = sScale[si];
                const float zs = half_bits_to_float((uint16_t)sb) * half_bits_to_float(sZero[si]);
                const uint32_t s2 = sb * 0x10001u;
                const uint32_t nzs2 = (uint32_t)float_to_f16_bits(-zs) * 0x10001u;
                // this row's 4 words of the half in each sub-stage: codes 32 hk .. 32 hk + 31
                uint4 pw[2];
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    pw[h] = *reinterpret_cast<const uint4*>(gbase + (sP - base) + u * P_BYTES + prow * (UK / 2) + h * 32 + hk * 16);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t words[4] = {pw[h].x, pw[h].y, pw[h].z, pw[h].w};
                    uint32_t o[16];
#pragma unroll
                    for (int wi = 0; wi < 4; ++wi) {
                        // the 8 codes of one word in the operand order (k0,k4)
                        // (k1,k5) (k2,k6) (k3,k7): masking a nibble into the
                        // mantissa of 1024.0 (bits 0-3) or 64.0 (bits 4-7) gives
                        // 1024 + q or 64 + q exactly, minus the base gives q
                        // exactly, and one fma gives q s - fl16(z s) rounded once
                        const uint32_t word = words[wi], ws = word >> 8;
                        o[4 * wi + 0] = hfma2_u32(hsub2_u32(lop_mask_or(word, 0x000F000Fu, 0x64006400u), 0x64006400u), s2, nzs2);
                        o[4 * wi + 1] = hfma2_u32(hsub2_u32(lop_mask_or(word, 0x00F000F0u, 0x54005400u), 0x54005400u), s2, nzs2);
                        o[4 * wi + 2] = hfma2_u32(hsub2_u32(lop_mask_or(ws, 0x000F000Fu, 0x64006400u), 0x64006400u), s2, nzs2);
                        o[4 * wi + 3] = hfma2_u32(hsub2_u32(lop_mask_or(ws, 0x00F000F0u, 0x54005400u), 0x54005400u), s2, nzs2);
                    }
                    tc::tmem_st_32x32b_x16(tmem_base + t_lane + A_COL0 + A_UNIT_COLS * a + BK / 2 * h + 16 * hk, o);
                }
                tc::tmem_st_wait();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive_cluster(afull_lead + 8 * a);
            }
        }
        cp_async_wait<0>();
    } else if (warp >= EP_WARP0) {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;                 // TMEM lane quarter
        const int eh = (warp - EP_WARP0) >> 2;  // column blocks eh, eh + EP_WARPS / 4, ...
        int ic = 0;
        for (int item = pair; item < n_items; item += npairs, ++ic) {
            int e, row0, nrows, fb;
            item_rows<GATEUP>(p, item, e, row0, nrows, fb);
            const uint32_t aph = ic & 1;
            bool ok = tc::mbar_wait(bar_accfull, aph, abort_flag, p.err);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc::tc_fence_after();
            const int ncb = ceil_div(nrows, 32);
            // K split between the two MMA issuers: the sum of two accumulators
            const bool split = ceil_div(nrows, 16) * 16 <= SPLIT_N;
            // this warp's last block (< eh: none)
            constexpr int EP_STEP = EP_WARPS / 4;
            const int last = ncb - 1 < eh ? -1 : eh + EP_STEP * ((ncb - 1 - eh) / EP_STEP);
            for (int cb = eh; cb < ncb; cb += EP_STEP) {
                uint32_t v[32];
                const uint32_t ta = tmem_base + cb * 32 + ((uint32_t)(32 * q) << 16);
                tc::tmem_ld_32x32b_x32(ta, v);
                tc::tmem_ld_wait();
                if (split) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t t[16];
                        tc::tmem_ld_32x32b_x16(ta + SPLIT_N + 16 * hh, t);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            v[16 * hh + j] = __float_as_uint(__uint_as_float(v[16 * hh + j]) + __uint_as_float(t[j]));
                    }
                }
                if (cb == last) {
                    // every column read: the MMA warp may start the next item
                    tc::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive_cluster(accempty_lead);
                }
                // out-of-range fp16 values are collected per column block and
                // reported once (a branch per element costs more than the math)
                uint32_t bad = 0;
                if (GATEUP) {
                    const bool lo_half = lane < 16;
                    const int feat = fb * 64 + 16 * q + (lane & 15);
                    // h is the down GEMM's operand: K interleaved in groups of 8
                    const int hcol = (feat & ~7) | k8_pos(feat & 7);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const uint32_t send = lo_half ? v[16 + j] : v[j];
                        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 16);
                        const float g = __uint_as_float(lo_half ? v[j] : recv);
                        const float u = __uint_as_float(lo_half ? recv : v[16 + j]);
                        const int col = cb * 32 + (lo_half ? j : 16 + j);
                        const uint16_t hb = float_to_f16_bits(silu(g) * u);
                        const bool valid = col < nrows;  // later columns hold the next expert's rows
                        bad |= valid & ((hb & 0x7C00u) == 0x7C00u);
                        if (valid) p.out[(size_t)(row0 + col) * p.out_ld + hcol] = hb;
                    }
                } else {
                    const int feat = fb * BM + 32 * q + lane;
                    uint16_t* outp = p.out + (size_t)(row0 + cb * 32) * p.out_ld + feat;
                    const int ncol = min(32, nrows - cb * 32);
                    if (p.row_w) {
                        const float* rw = p.row_w + row0 + cb * 32;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < ncol) {
                                const float y = __uint_as_float(v[j]) * rw[j];
                                const uint16_t yb = p.out_f16 ? float_to_f16_bits(y) : float_to_bf16_bits(y);
                                bad |= p.out_f16 && ((yb & 0x7C00u) == 0x7C00u);
                                outp[(size_t)j * p.out_ld] = yb;
                            }
                    } else if (p.out_f16) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < ncol) {
                                const uint16_t yb = float_to_f16_bits(__uint_as_float(v[j]));
                                bad |= ((yb & 0x7C00u) == 0x7C00u);
                                outp[(size_t)j * p.out_ld] = yb;
                            }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < ncol) outp[(size_t)j * p.out_ld] = float_to_bf16_bits(__uint_as_float(v[j]));
                    }
                }
                if (bad) set_error(p.err, ERRBIT_F16_RANGE);
            }
            if (last < eh) {
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive_cluster(accempty_lead);
            }
        }
    }

    // neither CTA frees its tensor memory or exits while the other may still
    // signal its barriers or use its memory
    __syncwarp();
    tc::tc_fence_before();
    tc::cluster_sync();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn get_encode() {
    static EncodeFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(ptr);
    }
    return fn;
}

// 2D map over a row-major [rows][cols] array.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, size_t esize, const void* ptr, uint64_t cols,
              uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
    EncodeFn enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * esize};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Activation rows [R][K] fp16 as a 3D view {64 K elements, rows, K / 64
// chunks}: a box {64, box_rows, 2} is one unit's two sub-stages of box_rows
// rows, each a 128B-swizzled K-major tile.
bool make_x_map(CUtensorMap* m, const void* ptr, int K, int R, uint32_t box_rows) {
    EncodeFn enc = get_encode();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)BK, (cuuint64_t)R, (cuuint64_t)(K / BK)};
    const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)BK * 2};
    const cuuint32_t box[3] = {BK, box_rows, 2}, estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr size_t TC_SMEM_LIMIT = 232448;

// Units of the shared-memory ring for a reduction length: 5 when they fit
// (one more than the A units in tensor memory), else 4.  A unit must be
// refilled while the MMAs of the units ahead of it run: the copy latency
// (about a microsecond) plus the dequantisation has to fit in SU - 1 units'
// MMA time, so the deeper ring keeps the tensor pipe fed.
int tc_units(int K) { return tc_smem_bytes(5, K) <= TC_SMEM_LIMIT ? 5 : 4; }

template <bool GATEUP, int SU>
cudaError_t launch_impl(int E, int d, int f, int R, const TcIn& in, cudaStream_t s) {
    TcParams p{};
    p.E = E;
    p.d = d;
    p.f = f;
    p.R = R;
    p.K = GATEUP ? d : f;
    p.NFB = GATEUP ? f / 64 : d / BM;
    p.wsc = GATEUP ? in.w13_s : in.w2_s;
    p.wz = GATEUP ? in.w13_z : in.w2_z;
    p.tiles = in.tiles;
    p.plan = in.plan;
    p.out = GATEUP ? in.h16 : in.y_out;
    p.out_ld = GATEUP ? f : d;
    p.out_f16 = GATEUP ? 1 : in.y_f16;
    p.row_w = GATEUP ? nullptr : in.row_w;
    p.err = in.err;

    const uint64_t rows_w = (uint64_t)E * (GATEUP ? 2 * (uint64_t)f : (uint64_t)d);
    CUtensorMap map_w, map_x, map_x2;
    if (GATEUP) {
        // codes as [expert * 2 + (gate, up)][feature][K / 8 words]: box = 8 words
        // of 64 features of both halves
        EncodeFn enc = get_encode();
        const cuuint64_t dims[3] = {(cuuint64_t)p.K / 8, (cuuint64_t)f, (cuuint64_t)E * 2};
        const cuuint64_t strides[2] = {(cuuint64_t)p.K / 2, (cuuint64_t)f * p.K / 2};
        const cuuint32_t box[3] = {UK / 8, 64, 2}, estr[3] = {1, 1, 1};
        if (!enc || enc(&map_w, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t*>(in.w13_q), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    } else if (!make_map(&map_w, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, in.w2_q, (uint64_t)p.K / 8, rows_w, UK / 8, BM,
                         CU_TENSOR_MAP_SWIZZLE_NONE)) {
        return cudaErrorInvalidValue;
    }
    if (!make_x_map(&map_x, GATEUP ? in.x16 : in.h16, p.K, R, B_BOX_ROWS) ||
        !make_x_map(&map_x2, GATEUP ? in.x16 : in.h16, p.K, R, 2 * B_BOX_ROWS))
        return cudaErrorInvalidValue;

    const size_t smem = tc_smem_bytes(SU, p.K);
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(tc_grouped_kernel<GATEUP, SU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)TC_SMEM_LIMIT);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    // one CTA pair per pair of SMs that can hold one (clusters of 2 SMs)
    static int max_pairs = 0;
    if (max_pairs == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(num_sms() & ~1));
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = smem;
        int nc = 0;
        if (cudaOccupancyMaxActiveClusters(&nc, tc_grouped_kernel<GATEUP, SU>, &cfg) != cudaSuccess || nc < 1) {
            (void)cudaGetLastError();
            nc = num_sms() / 2;
        }
        max_pairs = std::max(1, nc);
    }
    const int max_items = tc_max_tiles(R, E) * (p.NFB / 2);
    const int grid = 2 * std::max(1, std::min(max_pairs, max_items));
    tc_grouped_kernel<GATEUP, SU><<<grid, THREADS, smem, s>>>(map_w, map_x, map_x2, p);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

bool make_tensor_map_u32(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims, const uint64_t* strides,
                         const uint32_t* box) {
    EncodeFn enc = get_encode();
    if (!enc || rank < 1 || rank > 5) return false;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], estr[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        estr[i] = 1;
        if (i + 1 < rank) gs[i] = strides[i];
    }
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, (cuuint32_t)rank, const_cast<void*>(ptr), gd, gs, bx, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tensor_map_u16(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims, const uint64_t* strides,
                         const uint32_t* box) {
    EncodeFn enc = get_encode();
    if (!enc || rank < 1 || rank > 5) return false;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], estr[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        estr[i] = 1;
        if (i + 1 < rank) gs[i] = strides[i];
    }
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, (cuuint32_t)rank, const_cast<void*>(ptr), gd, gs, bx, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tensor_map_3d(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                        uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
    const uint64_t dims[3] = {d0, d1, d2}, strides[2] = {s1, s2};
    const uint32_t box[3] = {b0, b1, b2};
    return make_tensor_map_u32(m, ptr, 3, dims, strides, box);
}

int tc_max_tiles(int R, int E) { return ceil_div(R, TILE_ROWS) + std::min(R, E); }

bool tc_supported(int E, int d, int f) {
    (void)E;
    if (d % 256 || f % 256) return false;
    const int Kmax = std::max(d, f);
    return tc_smem_bytes(4, Kmax) <= TC_SMEM_LIMIT && d <= 8192 && f <= 8192;
}

cudaError_t launch_tc_gateup(int E, int d, int f, int R, const TcIn& in, cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    return tc_units(d) == 5 ? launch_impl<true, 5>(E, d, f, R, in, s) : launch_impl<true, 4>(E, d, f, R, in, s);
}

cudaError_t launch_tc_down(int E, int d, int f, int R, const TcIn& in, cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    return tc_units(f) == 5 ? launch_impl<false, 5>(E, d, f, R, in, s) : launch_impl<false, 4>(E, d, f, R, in, s);
}

}  // namespace moe
