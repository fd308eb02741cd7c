// The whole MoE layer for a few tokens (decode) in one persistent kernel.
//
// With T <= 8 tokens the layer is a stream of the routed experts' int4 weights
// past a handful of activation vectors: "Performance and verification"
// (bloomery docs/performance.md), section "Why it is fast", fetches each
// expert's weights once per batch and computes on the packed codes directly;
// "Measured results" (vllm-omni docs/edge/results.md), section Fidelity, fixes
// the W4A16 g128 format.  The kernel is built so that the weight stream never
// waits on anything but routing:
//
//   phase 0  every CTA routes all T tokens itself (top-k of the logits held
//            in shared memory, softmax over the selection) and sorts the T*k
//            assignments by expert (a rank per assignment from comparisons
//            with all the others), so no CTA waits for another to learn which
//            experts are needed.  CTA 0 writes the routing to topk_ids_out.
//   phase 1  gate_up: the CTA takes a contiguous share of the tiles
//            (touched expert u, 8 features) and computes, for each token routed
//            to u, the 8 gate and 8 up dot products over d_model, then
//            h = SiLU(gate) * up (fp16) into a global scratch.  Inside the CTA
//            the 8 consumer pairs split the tiles' chunks evenly; a tile cut
//            between two pairs is finished from their partial sums.
//   barrier  one grid-wide arrival on a 64-bit counter in the workspace header
//            (all CTAs are co-resident: one per SM, cooperative launch); the
//            producer keeps loading phase-2 weights while it is pending.
//   phase 2  down + combine: the CTA takes a contiguous share of one
//            token's units (16 output features); for each of the token's k
//            experts it forms 16 down-projection dot products over d_ff,
//            scaled by the routing weight; the pairs' partial sums of a unit
//            are added in pair order in fp32 and written to out as bf16.
//
// Inner loop.  One warp holds the A fragment of an m16n8k16 MMA (16 weight
// rows x 16 codes) in registers, dequantised straight from the packed words:
// ORing a nibble into the mantissa of an fp16 constant gives 1024 + q (nibble
// at bits 0..3 of a half, constant 0x6400) or 64 + q (bits 4..7, constant
// 0x5400) exactly, so one word becomes four f16x2 registers with four LOP3 and
// one shift.  The B fragment (8 columns = the tokens of the expert, zero for
// unused columns) holds the activations in fp16.  Per group of 128 codes the
// MMAs accumulate sum((offset + q) * x) in fp32; the group epilogue removes the
// offsets and applies zero and scale:
//     sum((q - z) * s * x) = s * (acc - C1 - z * C2),
//     C1 = 1024 * sum(x over even k) + 64 * sum(x over odd k),   C2 = sum(x),
// with C1 and C2 computed once per (token, group) from the same fp16 values.
//
// Pipeline.  NQ independent pipelines (3 or 4, see Shape): producer warp
// CW + i owns 1/NQ of the ring's slots and feeds consumer pairs 2i and 2i + 1,
// in chunk order.  A chunk is 16 weight rows x 4 lines of 128 B (2 groups
// each; one TMA box, 128-byte swizzle) plus the rows' fp16 scales and zeros
// (TMA boxes, plain bulk copies or 4-byte cp.async, by shape and
// instantiation), all completing the chunk's full mbarrier.  Consumer warps 0 .. CW - 1 form pairs; each warp
// of a pair takes half of a chunk's groups, loading each group's codes into
// registers right before its math and releasing the slot after the last
// group's loads; the two halves are added through shared memory.
// Every wait is bounded (2 s), after which the kernel records a timeout in the
// workspace error word, raises the CTA's abort flag and winds down.
#include <cfloat>
#include <climits>

#include "decode_ops.cuh"
#include "fastdiv.h"

namespace moe {
namespace {

using namespace dec;
using tc::WAIT_LIMIT_NS;

// Warp layout of one instantiation: NQ producer pipelines (producer warp
// CW + i feeds consumer pairs 2i and 2i + 1), 2 NQ pairs, 4 NQ consumer warps.
// Small layers take NQ = 3 (12 consumer warps: 128 registers each instead of
// 96, and fewer warps sharing a sub-partition when every pair computes at
// once); layers with megabytes of weights per CTA take NQ = 4 (more math in
// flight).
template <int NQ_>
struct Shape {
    static constexpr int NQ = NQ_;
    static constexpr int NPAIR = 2 * NQ_;
    static constexpr int CW = 2 * NPAIR;
    static constexpr int PRODUCER_WARP = CW;
    static constexpr int NTHREADS = 32 * (CW + NQ_);
    static constexpr int CONSUMER_THREADS = 32 * CW;
};
constexpr uint32_t FULL_ARRIVALS = 1;          // lane 0's expect_tx arrival (cp.async arrivals are counted)
// Each pipeline numbers its chunks in issue order and indexes its "full"
// barriers by chunk number modulo NFQ (not by ring slot: the pipeline's two
// pairs consume different chunks, so a pair may wait for chunk q before the
// chunk that last used q's slot has been consumed).  The pipeline's producer
// issues in order and issues chunk x only once chunk x - ns4 (ns4: its slots)
// has been consumed, so every chunk up to x - ns4 has landed by then; a pair's
// next chunk is at most 2 past its previous one, so with NFQ >= ns4 + 3 the
// previous use of q's barrier (chunk q - NFQ) has landed when q is waited on
// and the barrier's parity names q's phase unambiguously.
constexpr int NFQ = 64;
static_assert((NFQ & (NFQ - 1)) == 0, "NFQ must be a power of two");
constexpr int MAX_SLOTS = 32;

struct Tab {
    int32_t ids[MAX_R];    // routing, slot a = t*k + j
    float w[MAX_R];
    int32_t pos[MAX_R];    // permuted position of slot a
    int32_t ptok[MAX_R];   // token of permuted position i
    int32_t uexp[MAX_R];   // touched experts, ascending
    int32_t uoff[MAX_R];
    int32_t ucnt[MAX_R];
    int32_t first[MAX_R];  // sort scratch: 1 if assignment a is its expert's first
    int32_t n_uniq;
    int32_t abort;
    int32_t pad[30];
};

struct Params {
    const uint16_t* x;       // bf16 [T][d]
    const float* logits;     // fp32 [T][E]
    const uint16_t *w13_s, *w13_z, *w2_s, *w2_z;
    uint16_t* out;           // bf16 [T][d]
    int32_t* ids_out;        // [T][k] or null
    uint8_t* hb;             // fp16 [R][f], staged layout (see staged_offset)
    uint32_t* err;
    unsigned long long* bar_count;  // grid-barrier arrivals (only grows)
    int T, k, E, d, f;
    int nslot;                 // a multiple of the pipeline count NQ: pipeline i owns slots [i, i + 1) * nslot / NQ
    uint32_t off_sz, off_bars, off_xb, off_cx, off_hs, off_ch, off_red, off_red2, off_tab;
    int xb_stride, hs_stride;  // bytes per staged row
    // how the scales and zeros of gate_up / down reach a slot (SZ_*) and their
    // row stride there in bytes
    int sz13_mode, sz2_mode, sz13_rs, sz2_rs;
    // divisors fixed per launch (grid size, tokens, the two CTA counts a token
    // can have, chunks per tile of each phase, feature blocks, top-k, slots
    // per pipeline), for division without a runtime divide
    FastDiv fd_G, fd_T, fd_nct0, fd_nct1, fd_nch1, fd_nch2, fd_nfb1, fd_k, fd_ns4;
    FastDiv fd_xw, fd_hw;  // 16-byte words per activation row (d / 8) and per h row (f / 8)
};

// This warp's NG groups (gb .. gb + NG - 1 of the chunk whose codes are at sa
// and whose scales and zeros are at szs): the scales and zeros are copied
// into registers first, then each group's codes are loaded right before its
// math (the next group's loads overlap the current group's MMAs); the slot is
// given back after the last group's loads.
template <int NG>
__device__ __forceinline__ void consume_groups(float (&acc)[4], uint32_t sa, uint32_t szs, uint32_t rs, uint32_t empty,
                                               int gb, int g, int t, int gi0, uint32_t brow_a, uint32_t bact,
                                               uint32_t c0_a, uint32_t c1_a, float wscale) {
    // scales and zeros kept as fp16 pairs until use: sz[0..3] = s0, z0, s1, z1
    // (rows g and g + 8), word w holds groups 2w and 2w + 1 of this warp's NG
    constexpr int NW = (NG + 1) / 2;
    uint32_t sz[4][NW];
    const uint32_t szb = szs + (uint32_t)gb * 2 + (uint32_t)g * rs;
    const uint32_t sza[4] = {szb, szb + SZ_ARRAY, szb + 8 * rs, szb + SZ_ARRAY + 8 * rs};
    if constexpr (NG == 4) {
        // four groups' values of one row are 8 aligned bytes (gb is 0 or 4;
        // four groups per warp means 8 per chunk, so rows are 16 bytes)
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const float2 v = lds_f2(sza[a]);
            sz[a][0] = __float_as_uint(v.x);
            sz[a][1] = __float_as_uint(v.y);
        }
    } else {
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const uint32_t lo = lds_u16(sza[a] + 4 * w);
                const uint32_t hi = (2 * w + 1 < NG) ? lds_u16(sza[a] + 4 * w + 2) : 0u;
                sz[a][w] = lo | (hi << 16);
            }
    }
    // groups in pairs (two groups' MMAs interleaved: four independent
    // chains), each pair's codes loaded right before its math; the slot is
    // given back after the last codes are loaded
#pragma unroll
    for (int i = 0; i < NG; i += 2) {
        const bool two = i + 1 < NG;
        const uint32_t aoff0 = a_offset(gb + i, g, t);
        const uint4 wa0 = lds128(sa + aoff0), wb0 = lds128(sa + BOX_BYTES + aoff0);
        uint4 wa1 = wa0, wb1 = wb0;
        if (two) {
            const uint32_t aoff1 = a_offset(gb + i + 1, g, t);
            wa1 = lds128(sa + aoff1);
            wb1 = lds128(sa + BOX_BYTES + aoff1);
        }
        if (i + 2 >= NG) {
            __syncwarp();
            if ((threadIdx.x & 31) == 0) tc::mbar_arrive(empty);
        }
        const uint32_t gi = (uint32_t)(gi0 + gb + i);
        float v0[4], v1[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            v0[a] = (i & 1) ? half_hi(sz[a][i >> 1]) : half_lo(sz[a][i >> 1]);
            v1[a] = ((i + 1) & 1) ? half_hi(sz[a][(i + 1) >> 1]) : half_lo(sz[a][(i + 1) >> 1]);
        }
        v0[0] *= wscale;
        v0[2] *= wscale;
        v1[0] *= wscale;
        v1[2] *= wscale;
        if (two)
            compute_group2(acc, wa0, wb0, wa1, wb1, v0, v1, t, brow_a + 256u * gi, brow_a + 256u * (gi + 1), bact,
                           c0_a + 8u * gi, c1_a + 8u * gi, c0_a + 8u * (gi + 1), c1_a + 8u * (gi + 1));
        else
            compute_group(acc, wa0, wb0, v0[0], v0[1], v0[2], v0[3], t, brow_a + 256u * gi, bact, c0_a + 8u * gi,
                          c1_a + 8u * gi);
    }
}

// A chunk for this warp: wait for it, then take half of its gcv groups
// (gcv is even: d_model and d_ff are multiples of 256).
__device__ __forceinline__ void consume_chunk(float (&acc)[4], uint32_t full, uint32_t empty, uint32_t parity,
                                              uint32_t sa, uint32_t szs, uint32_t rs, int gcv, int half, int g, int t, int gi0, uint32_t brow_a,
                                              uint32_t bact, uint32_t c0_a, uint32_t c1_a, float wscale,
                                              volatile int* abort_flag, uint32_t* err) {
    const bool ready = tc::mbar_wait(full, parity, abort_flag, err);
    if (!ready) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) tc::mbar_arrive(empty);
        return;
    }
    const int ng = gcv >> 1, gb = half * ng;
    switch (ng) {
        case 4: consume_groups<4>(acc, sa, szs, rs, empty, gb, g, t, gi0, brow_a, bact, c0_a, c1_a, wscale); break;
        case 3: consume_groups<3>(acc, sa, szs, rs, empty, gb, g, t, gi0, brow_a, bact, c0_a, c1_a, wscale); break;
        case 2: consume_groups<2>(acc, sa, szs, rs, empty, gb, g, t, gi0, brow_a, bact, c0_a, c1_a, wscale); break;
        default: consume_groups<1>(acc, sa, szs, rs, empty, gb, g, t, gi0, brow_a, bact, c0_a, c1_a, wscale); break;
    }
}

// ------------------------------------------------------------------ kernel
template <int NQ_>
__global__ void __launch_bounds__(Shape<NQ_>::NTHREADS, 1)
decode_fused_kernel(const __grid_constant__ CUtensorMap map13, const __grid_constant__ CUtensorMap map2,
                    const __grid_constant__ CUtensorMap map13s, const __grid_constant__ CUtensorMap map13z,
                    const __grid_constant__ CUtensorMap map2s, const __grid_constant__ CUtensorMap map2z,
                    const Params p) {
    constexpr int NQ = Shape<NQ_>::NQ, NPAIR = Shape<NQ_>::NPAIR, CW = Shape<NQ_>::CW;
    constexpr int PRODUCER_WARP = Shape<NQ_>::PRODUCER_WARP, NTHREADS = Shape<NQ_>::NTHREADS;
    constexpr int CONSUMER_THREADS = Shape<NQ_>::CONSUMER_THREADS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sbase = smem_u32(sm);
    Tab& tab = *reinterpret_cast<Tab*>(sm + p.off_tab);
    volatile int* abort_flag = &tab.abort;
    const uint32_t szbase = sbase + p.off_sz;
    const uint32_t full0 = sbase + p.off_bars;            // [NQ][NFQ]
    const uint32_t empty0 = full0 + 8u * (NQ * NFQ);      // [nslot]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = p.T, k = p.k, R = T * k, E = p.E, d = p.d, f = p.f;
    const int Gd = d >> 7, Gf = f >> 7;
    const int G = gridDim.x, cta = blockIdx.x;
    const int nslot = p.nslot, ns4 = nslot / NQ;

    // ------------------------------------------------ phase 0: init, routing
    // The routed tokens' logits live in the ring, which is idle until the
    // producers start.
    float* lgs = reinterpret_cast<float*>(sm);
    const int nsort = T > 2 ? T : 2;  // warps that route (t < T) and sort (warps 0, 1)
    if (threadIdx.x == 0) tab.abort = 0;
    if (warp == PRODUCER_WARP) {
        for (int i = lane; i < NQ * NFQ; i += 32) tc::mbar_init(full0 + 8u * i, FULL_ARRIVALS);
        for (int i = lane; i < nslot; i += 32) tc::mbar_init(empty0 + 8u * i, 2);
        if (lane == 0) {
            tc::fence_mbar_init();
            tc::tma_prefetch_desc(&map13);
            tc::tma_prefetch_desc(&map2);
            if (p.sz13_mode == SZ_TMA) {
                tc::tma_prefetch_desc(&map13s);
                tc::tma_prefetch_desc(&map13z);
            }
            if (p.sz2_mode == SZ_TMA) {
                tc::tma_prefetch_desc(&map2s);
                tc::tma_prefetch_desc(&map2z);
            }
        }
    }
    // Launched as a programmatic dependent of the previous kernel on the
    // stream (when the driver accepts it), the CTA may start while that kernel
    // drains: everything above touches only this CTA's shared memory; from
    // here on global memory (inputs, workspace, outputs) is read and written,
    // so wait until the previous grid has completed and its writes are
    // visible.  (Without a programmatic dependency this returns at once.)
    // Before that, one warp asks L2 for this layer's logits and activations,
    // the first data the layer reads: a prefetch returns nothing, so it is
    // harmless even while the previous kernel may still write them.
    if (warp == 2) {
        const int lg_lines = (T * E * 4 + 127) / 128, x_lines = (T * d * 2 + 127) / 128;
        for (int i = lane; i < lg_lines; i += 32)
            asm volatile("prefetch.global.L2 [%0];" :: "l"(reinterpret_cast<const char*>(p.logits) + 128 * (size_t)i));
        for (int i = lane; i < x_lines; i += 32)
            asm volatile("prefetch.global.L2 [%0];" :: "l"(reinterpret_cast<const char*>(p.x) + 128 * (size_t)i));
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (warp < nsort) {
        if (warp < T) {
            // this token's logits into shared memory, then top-k
            float* lrow = lgs + warp * E;
            const float* src = p.logits + (size_t)warp * E;
            for (int e = lane; e < E; e += 32) lrow[e] = __ldg(src + e);
            __syncwarp();
            route_token(lrow, E, k, &tab.ids[warp * k], &tab.w[warp * k]);
            // the logits' ring bytes are overwritten by TMA once the producers start
            tc::fence_proxy_async_smem();
        }
        // every token routed: warps 0 and 1 sort while the other warps still
        // stage the activations
        bar_sync(15, 32 * nsort);
        if (warp < 2) {
            // Stable counting sort of the R <= 64 assignments by expert, one
            // thread per assignment a: its position is the number of
            // assignments with a smaller expert plus those of the same expert
            // before it; its expert's index in the ascending list of touched
            // experts is the number of distinct smaller experts.
            const int a = threadIdx.x;
            const bool va = a < R;
            const int ea = va ? tab.ids[a] : INT_MAX;
            int lt = 0, eqb = 0, eqall = 0;
            for (int b = 0; b < R; ++b) {
                const int eb = tab.ids[b];
                lt += eb < ea;
                eqall += eb == ea;
                eqb += (eb == ea) & (b < a);
            }
            const int first = (va && eqb == 0) ? 1 : 0;
            tab.first[a] = first;
            bar_sync(14, 64);
            int ui = 0, nu = 0;
            for (int b = 0; b < R; ++b) {
                const int fb = tab.first[b];
                nu += fb;
                ui += fb & (tab.ids[b] < ea);
            }
            if (va) {
                const int pos = lt + eqb;
                tab.pos[a] = pos;
                tab.ptok[pos] = (int)fd_div((uint32_t)a, p.fd_k);
            }
            if (first) {
                tab.uexp[ui] = ea;
                tab.uoff[ui] = lt;
                tab.ucnt[ui] = eqall;
            }
            if (a == 0) tab.n_uniq = nu;
        }
    } else if (warp < CW) {
        // activations -> fp16 in MMA order, plus C1/C2 per (token, group); the
        // C1/C2 row T is zero (B columns without a token)
        const int nthr = (CW - nsort) * 32, tid = (warp - nsort) * 32 + lane;
        const int wpr = d >> 3;  // 16-byte words per row (a multiple of 32)
        float2* cx = reinterpret_cast<float2*>(sm + p.off_cx);
        for (int wi = tid; wi < T * wpr; wi += nthr) {
            const int t = (int)fd_div((uint32_t)wi, p.fd_xw), wr = wi - t * wpr;
            const uint4 raw = __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)t * d) + wr);
            const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
            uint32_t q[4];
            bool bad = false;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                q[m] = pack_f16x2(__uint_as_float(rw[m] << 16), __uint_as_float(rw[m] & 0xFFFF0000u));
                bad |= f16x2_nonfinite(q[m]);
            }
            if (bad) set_error(p.err, ERRBIT_F16_RANGE);
            const uint4 o = k8_interleave(q[0], q[1], q[2], q[3]);
            sts128(sbase + p.off_xb + (uint32_t)(t * p.xb_stride) + staged_offset(wr * 8), o);
            const float2 c = halfwarp_sum(word_c1c2(o));
            if ((lane & 15) == 0) cx[t * Gd + (wr >> 4)] = c;
        }
        for (int i = tid; i < Gd; i += nthr) cx[T * Gd + i] = make_float2(0.f, 0.f);
    }
    __syncthreads();
    if (cta == 0 && p.ids_out)
        for (int a = threadIdx.x; a < R; a += NTHREADS) p.ids_out[a] = tab.ids[a];

    // work shares.  Phase 1: a contiguous share of the tiles (touched expert,
    // 8 features).  Phase 2: token tok gets the CTAs c with c * T / G == tok and
    // each of them a contiguous share of tok's units (16 output rows), so a
    // CTA stages the h rows of one token only.
    const int U = tab.n_uniq;
    const int nfb1 = f >> 3, nrb = d >> 4;
    const int N1 = U * nfb1;
    // (32-bit products: N1 <= 64 * 2048 times G < 2^12)
    const int a1 = (int)fd_div((uint32_t)(cta * N1), p.fd_G), b1 = (int)fd_div((uint32_t)((cta + 1) * N1), p.fd_G);
    const int tok = (int)fd_div((uint32_t)(cta * T), p.fd_G);
    const int c_lo = (int)fd_div((uint32_t)(tok * G + T - 1), p.fd_T);
    const int c_hi = (int)fd_div((uint32_t)((tok + 1) * G + T - 1), p.fd_T);
    const FastDiv fd_nct = (uint32_t)(c_hi - c_lo) == p.fd_nct0.d ? p.fd_nct0 : p.fd_nct1;
    const int r_lo = (int)fd_div((uint32_t)((cta - c_lo) * nrb), fd_nct);
    const int r_hi = (int)fd_div((uint32_t)((cta - c_lo + 1) * nrb), fd_nct);
    const int n1 = b1 - a1, n2u = r_hi - r_lo, n2t = n2u * k;
    const int nch1 = ceil_div(Gd, CHUNK_GROUPS), nch2 = ceil_div(Gf, CHUNK_GROUPS);

    // Work inside the CTA is split by chunks: a phase's W = tiles x chunks per
    // tile, in (tile, chunk) order, and pair P takes the chunks
    // [P W / NPAIR, (P + 1) W / NPAIR), so every pair streams the same number
    // of bytes.  A tile cut by a range boundary leaves partial sums that are
    // added after the phase (phase 1) or per (unit, pair) (phase 2).
    // Pipeline qp (producer warp PRODUCER_WARP + qp) feeds pairs 2qp and
    // 2qp + 1: its chunks are numbered in issue order, chunk i of pair 2qp, then
    // chunk i of pair 2qp + 1, then i + 1 ...; phase 2 continues after phase 1.
    auto rng = [](int P, int W) { return P * W / NPAIR; };
    const int W1 = n1 * nch1, W2 = n2t * nch2;

    // ---------------------------------------------------------- producers
    // Per chunk the pipeline waits until the chunk's slot is empty and issues
    // the TMA box of the codes.  The fp16 scales and zeros come by TMA or bulk
    // copies issued by lane 0 as well, or every lane copies its row's values
    // with 4-byte cp.async and a counted arrival, after which lane 0 arrives
    // (the codes' bytes were expected before their copy was issued); the host
    // picks the form per phase (sz13_mode, sz2_mode).  One warp per pipeline,
    // in chunk order: a slot's round r is waited on only after its round
    // r - 1 has completed, so every parity wait is exact.
    if (warp >= PRODUCER_WARP) {
        const int qp = warp - PRODUCER_WARP;
        const uint32_t fullq = full0 + 8u * (uint32_t)(qp * NFQ);
        const int slot0 = qp * ns4;
        // chunk number, its slot inside the pipeline and the slot's round, kept
        // incrementally (a runtime divide costs tens of dependent instructions)
        uint32_t qq = 0, sl = 0, round = 0;
        int ok = 1;
        auto advance = [&]() {
            ++qq;
            if (++sl == (uint32_t)ns4) {
                sl = 0;
                ++round;
            }
        };
        // A consumer that gave up releases its slot without the chunk having
        // landed, and only once the abort flag is raised; so a slot wait that
        // completes with the flag raised issues nothing more, and the drain of
        // each slot's last use below then covers every copy still in flight.
        auto slot_free = [&](uint32_t slot) -> int {
            if (round != 0 && !tc::mbar_wait(empty0 + 8u * slot, (round - 1) & 1u, abort_flag, p.err)) return 0;
            return *abort_flag ? 0 : 1;
        };
        // A pair's position in its chunk range: chunk c of tile (p0, p1) =
        // (touched-expert index, feature block) in phase 1, (unit, slot j) in
        // phase 2, and the tile's weight rows.  Tiles advance without division.
        struct Cur {
            int c, p0, p1, row0, row1, ex, fb8;
        };
        auto set_rows = [&](Cur& u, bool up) {
            if (up) {
                u.ex = tab.uexp[u.p0];
                u.fb8 = 8 * u.p1;
                u.row0 = u.ex * 2 * f + u.fb8;
                u.row1 = u.row0 + f;
            } else {
                u.row0 = tab.ids[tok * k + u.p1] * d + 16 * (r_lo + u.p0);
                u.row1 = u.row0 + 8;
            }
        };
        auto cur_init = [&](Cur& u, bool up, int x, int nch, bool any) {
            const int tl = (int)fd_div((uint32_t)x, up ? p.fd_nch1 : p.fd_nch2);
            u.c = x - tl * nch;
            const int a = up ? a1 + tl : tl;
            const FastDiv dv = up ? p.fd_nfb1 : p.fd_k;
            u.p0 = (int)fd_div((uint32_t)a, dv);
            u.p1 = a - u.p0 * (int)dv.d;
            u.ex = u.fb8 = 0;
            if (any) set_rows(u, up);
        };
        auto cur_next = [&](Cur& u, bool up, int nch, bool more) {
            if (++u.c < nch) return;
            u.c = 0;
            if (++u.p1 == (up ? nfb1 : k)) {
                u.p1 = 0;
                ++u.p0;
            }
            if (more) set_rows(u, up);
        };
        auto tma_codes = [&](bool up, uint32_t dst, uint32_t full, const Cur& u) {
            if (up)
                tc::tma_load_4d(dst, &map13, full, 0, u.c * LINES, u.fb8, 2 * u.ex);
            else
                tc::tma_load_3d(dst, &map2, full, 0, u.c * LINES, u.row0);
        };
        // one phase: the two pairs' chunk ranges interleaved (chunk i of pair
        // 2qp, then of pair 2qp + 1)
        auto run = [&](bool up, int W, int nch, int mode, const uint16_t* s_arr, const uint16_t* z_arr, int Gk) {
            const int xa = rng(2 * qp, W), xm = rng(2 * qp + 1, W), xz = rng(2 * qp + 2, W);
            const int len[2] = {xm - xa, xz - xm};
            const int lmax = max(len[0], len[1]);
            Cur cu[2];
            cur_init(cu[0], up, xa, nch, len[0] > 0);
            cur_init(cu[1], up, xm, nch, len[1] > 0);
            if (mode != SZ_CPASYNC) {
                // bytes per chunk: codes + two arrays of 16 rows (8 groups by TMA,
                // all Gk groups by bulk copy)
                const uint32_t tx = SLOT_CODE + (mode == SZ_TMA ? SLOT_SZ : 64u * (uint32_t)Gk);
                if (lane == 0) {
                    for (int i = 0; i < lmax && ok; ++i)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            if (i >= len[e] || !ok) continue;
                            Cur& u = cu[e];
                            const uint32_t full = fullq + 8u * (qq & (NFQ - 1));
                            const uint32_t slot = (uint32_t)slot0 + sl;
                            ok = slot_free(slot);
                            if (!ok) break;
                            const uint32_t dst = sbase + slot * SLOT_CODE, sdst = szbase + slot * SLOT_SZ;
                            tc::mbar_arrive_expect_tx(full, tx);
                            tma_codes(up, dst, full, u);
                            const int g0 = u.c * CHUNK_GROUPS;
                            if (mode == SZ_TMA) {
                                if (up) {
                                    tc::tma_load_3d(sdst, &map13s, full, g0, u.fb8, 2 * u.ex);
                                    tc::tma_load_3d(sdst + SZ_ARRAY, &map13z, full, g0, u.fb8, 2 * u.ex);
                                } else {
                                    tc::tma_load_2d(sdst, &map2s, full, g0, u.row0);
                                    tc::tma_load_2d(sdst + SZ_ARRAY, &map2z, full, g0, u.row0);
                                }
                            } else if (up) {
                                // 8 gate rows, then 8 up rows, of every group
                                const uint32_t hb = 16u * (uint32_t)Gk;
                                tc::bulk_load(sdst, s_arr + (size_t)u.row0 * Gk, hb, full);
                                tc::bulk_load(sdst + hb, s_arr + (size_t)u.row1 * Gk, hb, full);
                                tc::bulk_load(sdst + SZ_ARRAY, z_arr + (size_t)u.row0 * Gk, hb, full);
                                tc::bulk_load(sdst + SZ_ARRAY + hb, z_arr + (size_t)u.row1 * Gk, hb, full);
                            } else {
                                tc::bulk_load(sdst, s_arr + (size_t)u.row0 * Gk, 32u * (uint32_t)Gk, full);
                                tc::bulk_load(sdst + SZ_ARRAY, z_arr + (size_t)u.row0 * Gk, 32u * (uint32_t)Gk, full);
                            }
                            advance();
                            cur_next(u, up, nch, i + 1 < len[e]);
                        }
                }
                // the other lanes take over lane 0's state
                qq = __shfl_sync(0xffffffffu, qq, 0);
                sl = __shfl_sync(0xffffffffu, sl, 0);
                round = __shfl_sync(0xffffffffu, round, 0);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                return;
            }
            const int arr = lane >> 4, r = lane & 15;
            const uint16_t* base = arr ? z_arr : s_arr;
            for (int i = 0; i < lmax && ok; ++i)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    if (i >= len[e] || !ok) continue;
                    Cur& u = cu[e];
                    const uint32_t full = fullq + 8u * (qq & (NFQ - 1));
                    const uint32_t slot = (uint32_t)slot0 + sl;
                    int w = 1;
                    if (lane == 0) w = slot_free(slot);
                    // the warp follows lane 0's verdict; __syncwarp orders the
                    // wait before any lane's copies into the slot
                    ok = __shfl_sync(0xffffffffu, w, 0);
                    __syncwarp();
                    if (!ok) break;
                    // the codes' copy first: its bytes are expected before it is
                    // issued, and the phase still waits for lane 0's arrival
                    // below (decode layer 17.50 -> 17.38 us against issuing it
                    // after the scales)
                    if (lane == 0) {
                        tc::mbar_expect_tx(full, SLOT_CODE);
                        tma_codes(up, sbase + slot * SLOT_CODE, full, u);
                    }
                    const int grow = r < 8 ? u.row0 + r : u.row1 + (r - 8);
                    const int g0 = u.c * CHUNK_GROUPS;
                    const int gcv = min(CHUNK_GROUPS, Gk - g0);
                    const uint16_t* src = base + (size_t)grow * Gk + g0;
                    const uint32_t sdst = szbase + slot * SLOT_SZ + (uint32_t)(arr * SZ_ARRAY + r * 16);
                    for (int gi = 0; gi < (gcv >> 1); ++gi) cp_async4(sdst + 4u * gi, src + 2 * gi);
                    // counted arrivals before lane 0's, so the phase cannot
                    // complete before every lane's copies are tracked
                    tc::cp_async_mbar_arrive(full);
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(full);
                    advance();
                    cur_next(u, up, nch, i + 1 < len[e]);
                }
        };
        run(true, W1, nch1, p.sz13_mode, p.w13_s, p.w13_z, Gd);
        if (ok) run(false, W2, nch2, p.sz2_mode, p.w2_s, p.w2_z, Gf);
        if (p.sz13_mode == SZ_CPASYNC || p.sz2_mode == SZ_CPASYNC)
            asm volatile("cp.async.wait_all;" ::: "memory");  // this lane's copies have landed
        // drain: the last use of each of the pipeline's slots must have landed
        // before the CTA exits
        if (lane == 0) {
            const uint32_t first = qq > (uint32_t)ns4 ? qq - (uint32_t)ns4 : 0u;
            const uint64_t t0 = globaltimer_ns();
            for (uint32_t qx = first; qx < qq; ++qx) {
                const uint32_t full = fullq + 8u * (qx & (NFQ - 1));
                const uint32_t par = (qx / NFQ) & 1u;
                while (!tc::mbar_try_wait(full, par)) {
                    if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
                        set_error(p.err, ERRBIT_TIMEOUT);
                        qx = qq;
                        break;
                    }
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int pair = warp >> 1, half = warp & 1;
    const int qp = pair >> 1, e = pair & 1;
    const int g = lane >> 2, t4 = lane & 3;
    const uint32_t fullq = full0 + 8u * (uint32_t)(qp * NFQ);
    const int slot0 = qp * ns4;
    float* red = reinterpret_cast<float*>(sm + p.off_red);  // [pair][2][32 lanes][4]
    int rcount = 0;
    auto pair_reduce = [&](float (&acc)[4]) {
        float* rb = red + ((pair * 2 + (rcount & 1)) * 32 + lane) * 4;
        if (half == 1) *reinterpret_cast<float4*>(rb) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        bar_sync(2 + pair, 64);
        if (half == 0) {
            const float4 o = *reinterpret_cast<const float4*>(rb);
            acc[0] += o.x;
            acc[1] += o.y;
            acc[2] += o.z;
            acc[3] += o.w;
        }
        ++rcount;
    };
    // This pair's chunks of a phase: pipeline numbers qbase + 2i + e while the
    // partner pair also has an i-th chunk, then consecutive.  The slot index
    // inside the pipeline follows incrementally (steps of 1 or 2 <= ns4).
    struct Seq {
        uint32_t qq, sl;
        int i, lmin;
    };
    auto seq_start = [&](int W, uint32_t qbase) {
        const int len_me = rng(pair + 1, W) - rng(pair, W);
        const int len_pt = e ? rng(pair, W) - rng(pair - 1, W) : rng(pair + 2, W) - rng(pair + 1, W);
        Seq s;
        s.lmin = min(len_me, len_pt);
        s.i = 0;
        s.qq = qbase + (uint32_t)(s.lmin > 0 ? e : 0);
        s.sl = s.qq - fd_div(s.qq, p.fd_ns4) * (uint32_t)ns4;
        return s;
    };
    auto seq_chunk = [&](Seq& s, float (&acc)[4], int c, int Gk, uint32_t rs, uint32_t brow_a, uint32_t bact,
                         uint32_t c0_a, uint32_t c1_a, float wscale) {
        const uint32_t slot = (uint32_t)slot0 + s.sl;
        consume_chunk(acc, fullq + 8u * (s.qq & (NFQ - 1)), empty0 + 8u * slot, (s.qq / NFQ) & 1u,
                      sbase + slot * SLOT_CODE, szbase + slot * SLOT_SZ, rs, min(CHUNK_GROUPS, Gk - c * CHUNK_GROUPS),
                      half, g, t4, c * CHUNK_GROUPS, brow_a, bact, c0_a, c1_a, wscale, abort_flag, p.err);
        ++s.i;
        const uint32_t step = s.i <= s.lmin - 1 ? 2u : (s.i == s.lmin ? (uint32_t)(2 - e) : 1u);
        s.qq += step;
        s.sl += step;
        if (s.sl >= (uint32_t)ns4) s.sl -= (uint32_t)ns4;
    };
    const uint32_t xb = sbase + p.off_xb, cxa = sbase + p.off_cx;
    // partial sums of tiles cut by a range boundary: [pair][head, tail][32 lanes][4]
    // (aliases red2, which is used only after the grid barrier)
    float* part = reinterpret_cast<float*>(sm + p.off_red2);

    // phase 1: gate_up.  h = SiLU(gate) * up of tile tl (half 0 of a pair, from
    // acc = the pair's sums: rows g (gate) and g + 8 (up), columns 2 t4, 2 t4 + 1)
    // (feature block fb of the touched expert whose cnt tokens start at permuted
    // position off)
    auto h_epilogue_at = [&](int fb, int cnt, int off, const float (&acc)[4]) {
        const uint32_t hoff = staged_offset(8 * fb + g);
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
            const int colm = 2 * t4 + mm;
            if (colm < cnt) {
                const float h = silu(acc[mm]) * acc[2 + mm];
                const __half hh = __float2half_rn(h);
                if (__hisinf(hh) || __hisnan(hh)) set_error(p.err, ERRBIT_F16_RANGE);
                *reinterpret_cast<__half*>(p.hb + (size_t)(off + colm) * (f * 2) + hoff) = hh;
            }
        }
    };
    auto h_epilogue = [&](int tl, const float (&acc)[4]) {
        const int tau = a1 + tl, u = (int)fd_div((uint32_t)tau, p.fd_nfb1), fb = tau - u * nfb1;
        h_epilogue_at(fb, tab.ucnt[u], tab.uoff[u], acc);
    };
    {
        const int x_lo = rng(pair, W1), x_hi = rng(pair + 1, W1);
        Seq s = seq_start(W1, 0u);
        for (int x = x_lo; x < x_hi;) {
            const int tl = (int)fd_div((uint32_t)x, p.fd_nch1), c0 = x - tl * nch1, c1 = min(nch1, c0 + (x_hi - x));
            const int tau = a1 + tl, u = (int)fd_div((uint32_t)tau, p.fd_nfb1);
            const int cnt = tab.ucnt[u], off = tab.uoff[u];
            const int col = lane >> 2;
            // B columns without a token are not loaded (bact = 0) and read as zero
            const int brow = col < cnt ? tab.ptok[off + col] : 0;
            const int cr0 = 2 * t4 < cnt ? tab.ptok[off + 2 * t4] : T;
            const int cr1 = 2 * t4 + 1 < cnt ? tab.ptok[off + 2 * t4 + 1] : T;
            const uint32_t brow_a = xb + (uint32_t)(brow * p.xb_stride);
            const uint32_t c0_a = cxa + (uint32_t)(cr0 * Gd * 8), c1_a = cxa + (uint32_t)(cr1 * Gd * 8);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int c = c0; c < c1; ++c)
                seq_chunk(s, acc, c, Gd, (uint32_t)p.sz13_rs, brow_a, (uint32_t)(col < cnt), c0_a, c1_a, 1.0f);
            pair_reduce(acc);
            if (half == 0 && !*abort_flag) {
                if (c0 == 0 && c1 == nch1) {
                    // The 16-warp instantiation hands the tile's expert data on
                    // (large layer 75.4 -> 74.2 us); the 12-warp one looks it up
                    // again, which keeps fewer registers live across the chunk
                    // loop (17.55 us with the hand-on against 17.41).
                    if constexpr (NQ_ == 4)
                        h_epilogue_at(tau - u * nfb1, cnt, off, acc);
                    else
                        h_epilogue(tl, acc);
                } else {
                    // head piece (the tile began in an earlier range) or tail piece
                    float* pp = part + ((pair * 2 + (c0 > 0 ? 0 : 1)) * 32 + lane) * 4;
                    *reinterpret_cast<float4*>(pp) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                }
            }
            x += c1 - c0;
        }
    }
    bar_sync(1, CONSUMER_THREADS);
    // tiles cut by boundaries: the first boundary inside tile tc (that of pair
    // P = this pair, P >= 1) adds the pieces of the pairs P - 1, P, ... that
    // hold parts of tc, in pair order, and writes tc's h
    if (half == 0 && pair >= 1 && !*abort_flag) {
        const int xbd = rng(pair, W1);
        const int tc_ = (int)fd_div((uint32_t)xbd, p.fd_nch1);
        if (xbd < W1 && xbd - tc_ * nch1 != 0 && rng(pair - 1, W1) <= tc_ * nch1) {
            const int tstart = tc_ * nch1, tend = tstart + nch1;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int P2 = pair - 1; P2 < NPAIR; ++P2) {
                const int s0 = rng(P2, W1), s1 = rng(P2 + 1, W1);
                if (s0 >= tend) break;
                if (s1 <= s0) continue;
                const float4 v =
                    *reinterpret_cast<const float4*>(part + ((P2 * 2 + (s0 > tstart ? 0 : 1)) * 32 + lane) * 4);
                acc[0] += v.x;
                acc[1] += v.y;
                acc[2] += v.z;
                acc[3] += v.w;
            }
            h_epilogue(tc_, acc);
        }
    }

    // grid-wide barrier: every CTA's h is written before anyone reads it.  The
    // 64-bit arrival count only grows (G per launch), so a CTA's own arrival
    // tells it the count at which this launch's barrier opens and nothing has
    // to be reset afterwards.
    bar_sync(1, CONSUMER_THREADS);
    if (threadIdx.x == 0) {
        const uint64_t old = atom_add_release_gpu(p.bar_count, 1ull);
        const uint64_t target = (old / (uint64_t)G + 1) * (uint64_t)G;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t it = 1; ld_acquire_gpu64(p.bar_count) < target; ++it) {
            if ((it & 63u) == 0) {
                if (*abort_flag) break;
                if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
                    set_error(p.err, ERRBIT_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
            }
        }
    }
    bar_sync(1, CONSUMER_THREADS);

    // this CTA is in its last phase: the next kernel may be scheduled
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // stage token tok's k rows of h (slot j at row j) and their C1/C2 (the
    // C1/C2 row k is zero); clear the per-(unit, pair) partials
    const int zrow = k;
    const uint32_t hs = sbase + p.off_hs, cha = sbase + p.off_ch;
    float2* ch = reinterpret_cast<float2*>(sm + p.off_ch);
    float* red2 = reinterpret_cast<float*>(sm + p.off_red2);  // [unit][pair][16]
    if (!*abort_flag && n2u > 0) {
        const int tid = threadIdx.x;
        const int wpr = f >> 3;  // 16-byte words per row, a multiple of 32
        // h is stored in the staged order already.  The 16-warp instantiation
        // (over a megabyte of weights per CTA) copies first, all of a thread's
        // words in flight at once, then sums the words it copied (1.3 us less
        // per d_model 7168 layer); the 12-warp one loads and sums word by
        // word, which measured faster there (the copy form left its staging
        // time unchanged and slowed its phase loops by ~0.5 us per layer).
        if constexpr (NQ_ == 4) {
            const int nw = k * wpr;
            for (int wi = tid; wi < nw; wi += CONSUMER_THREADS) {
                const int lr = (int)fd_div((uint32_t)wi, p.fd_hw), wr = wi - lr * wpr;
                cp_async16(hs + (uint32_t)(lr * p.hs_stride) + 16u * wr,
                           p.hb + (size_t)tab.pos[tok * k + lr] * (f * 2) + 16 * (size_t)wr);
            }
            asm volatile("cp.async.wait_all;" ::: "memory");
            for (int wi = tid; wi < nw; wi += CONSUMER_THREADS) {
                const int lr = (int)fd_div((uint32_t)wi, p.fd_hw), wr = wi - lr * wpr;
                const uint4 o = lds128(hs + (uint32_t)(lr * p.hs_stride) + 16u * wr);
                // a staged word holds one word's 8 values in MMA order (staged_offset)
                const float2 c = halfwarp_sum(word_c1c2(o));
                if ((lane & 15) == 0) ch[lr * Gf + (wr >> 4)] = c;
            }
        } else {
            for (int wi = tid; wi < k * wpr; wi += CONSUMER_THREADS) {
                const int lr = (int)fd_div((uint32_t)wi, p.fd_hw), wr = wi - lr * wpr;
                const uint4 o = ldg_cg16(p.hb + (size_t)tab.pos[tok * k + lr] * (f * 2) + 16 * (size_t)wr);
                sts128(hs + (uint32_t)(lr * p.hs_stride) + 16u * wr, o);
                // a staged word holds one word's 8 values in MMA order (staged_offset)
                const float2 c = halfwarp_sum(word_c1c2(o));
                if ((lane & 15) == 0) ch[lr * Gf + (wr >> 4)] = c;
            }
        }
        for (int i = tid; i < Gf; i += CONSUMER_THREADS) ch[zrow * Gf + i] = make_float2(0.f, 0.f);
        for (int i = tid; i < n2u * NPAIR * 16; i += CONSUMER_THREADS) red2[i] = 0.f;
    }
    bar_sync(1, CONSUMER_THREADS);

    // phase 2: down tiles i2 = (unit ul, slot j); a pair's chunks accumulate
    // over the slots and K range it holds of a unit, one partial per (unit, pair)
    {
        const int x_lo = rng(pair, W2), x_hi = rng(pair + 1, W2);
        Seq s = seq_start(W2, (uint32_t)(rng(2 * qp + 2, W1) - rng(2 * qp, W1)));
        int cur = -1;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        auto flush = [&](int ul) {
            pair_reduce(acc);
            if (half == 0 && t4 == 0) {
                float* dst = red2 + (ul * NPAIR + pair) * 16;
                dst[g] = acc[0];
                dst[g + 8] = acc[2];
            }
        };
        const uint32_t bact = (uint32_t)((lane >> 2) == 0);  // column 0 is the token
        for (int x = x_lo; x < x_hi;) {
            const int i2 = (int)fd_div((uint32_t)x, p.fd_nch2), c0 = x - i2 * nch2, c1 = min(nch2, c0 + (x_hi - x));
            const int ul = (int)fd_div((uint32_t)i2, p.fd_k), j = i2 - ul * k;
            if (ul != cur) {
                if (cur >= 0) flush(cur);
                cur = ul;
                acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
            }
            const float wj = tab.w[tok * k + j];
            const int cr0 = t4 == 0 ? j : zrow;
            const uint32_t brow_a = hs + (uint32_t)(j * p.hs_stride);
            const uint32_t c0_a = cha + (uint32_t)(cr0 * Gf * 8), c1_a = cha + (uint32_t)(zrow * Gf * 8);
            for (int c = c0; c < c1; ++c) seq_chunk(s, acc, c, Gf, (uint32_t)p.sz2_rs, brow_a, bact, c0_a, c1_a, wj);
            x += c1 - c0;
        }
        if (cur >= 0) flush(cur);
    }
    bar_sync(1, CONSUMER_THREADS);

    // out[tok][16 rb + r] = the unit's partials, in pair order
    if (!*abort_flag) {
        for (int idx = threadIdx.x; idx < n2u * 16; idx += CONSUMER_THREADS) {
            const int ul = idx >> 4, r = idx & 15;
            float sum = 0.f;
#pragma unroll
            for (int P2 = 0; P2 < NPAIR; ++P2) sum += red2[(ul * NPAIR + P2) * 16 + r];
            p.out[(size_t)tok * d + 16 * (r_lo + ul) + r] = float_to_bf16_bits(sum);
        }
    }
}

struct Layout {
    int nslot;
    size_t smem;
    uint32_t off_sz, off_bars, off_xb, off_cx, off_hs, off_ch, off_red, off_red2, off_tab;
    int xb_stride, hs_stride;
};

bool plan_layout(int T, int k, int E, int d, int f, int G, int nq, Layout* L) {
    const int NQ = nq, NPAIR = 2 * nq;
    if (T < 1 || T > MAX_T || k < 1 || T * k > MAX_R || E < 1 || E > 1024 || G < T) return false;
    if (d % 256 || f % 256 || f >= 65536) return false;  // (a feature index is packed in 16 bits)
    Layout l{};
    l.xb_stride = 2 * d + ROW_PAD;
    l.hs_stride = 2 * f + ROW_PAD;
    // a token has at least G / T CTAs for its d / 16 units
    const int n2u_max = ceil_div(d / 16, G / T);
    size_t fixed = 0;
    auto take = [&](size_t bytes) {
        const size_t o = fixed;
        fixed = align_up(fixed + bytes, 128);
        return (uint32_t)o;
    };
    // offsets relative to the end of the ring and its barriers (rebased below).
    // The staged activations (+ C1/C2) are read in phase 1 only and the staged
    // h rows (+ C1/C2) are written after the grid barrier: one shared region.
    const size_t sx = align_up((size_t)T * l.xb_stride, 128) + (size_t)(T + 1) * (d / 128) * 8;
    const size_t sh = align_up((size_t)k * l.hs_stride, 128) + (size_t)(k + 1) * (f / 128) * 8;
    const uint32_t o_xb = take(std::max(sx, sh));
    const uint32_t o_cx = o_xb + (uint32_t)align_up((size_t)T * l.xb_stride, 128);
    const uint32_t o_hs = o_xb;
    const uint32_t o_ch = o_xb + (uint32_t)align_up((size_t)k * l.hs_stride, 128);
    const uint32_t o_red = take((size_t)NPAIR * 2 * 32 * 4 * 4);
    // red2 (phase 2) also holds phase 1's cut-tile pieces [pair][2][32][4]
    const uint32_t o_red2 = take(std::max((size_t)n2u_max * NPAIR * 16 * 4, (size_t)NPAIR * 2 * 32 * 4 * 4));
    const uint32_t o_tab = take(sizeof(Tab));
    if (fixed + 1024 >= SMEM_LIMIT) return false;
    const size_t avail = SMEM_LIMIT - 1024 - fixed;
    const size_t bar_fixed = align_up((size_t)8 * NQ * NFQ + 8 * MAX_SLOTS, 128);
    if (avail <= bar_fixed) return false;
    int nslot = (int)((avail - bar_fixed) / (SLOT_CODE + SLOT_SZ));
    nslot = std::min(nslot, MAX_SLOTS);
    nslot -= nslot % NQ;
    // two slots per pipeline at least (a consumer's slot index advances by at
    // most 2 per chunk), and the full-barrier bound NFQ >= slots + 3
    if (nslot < 2 * NQ || nslot / NQ + 3 > NFQ) return false;
    // phase-0 scratch in the ring: the routed tokens' logits
    if ((size_t)T * E * 4 > (size_t)nslot * SLOT_CODE) return false;  // routing scratch in the ring
    const uint32_t ring = (uint32_t)nslot * SLOT_CODE;
    const uint32_t szs = (uint32_t)nslot * SLOT_SZ;
    const uint32_t base = ring + szs + (uint32_t)bar_fixed;
    l.nslot = nslot;
    l.off_sz = ring;
    l.off_bars = ring + szs;
    l.off_xb = base + o_xb;
    l.off_cx = base + o_cx;
    l.off_hs = base + o_hs;
    l.off_ch = base + o_ch;
    l.off_red = base + o_red;
    l.off_red2 = base + o_red2;
    l.off_tab = base + o_tab;
    l.smem = 1024 + base + fixed;
    if (l.smem > SMEM_LIMIT) return false;
    *L = l;
    return true;
}

}  // namespace

// Pipelines for a layer: 3 while the routed weights per CTA are small (at most
// T k experts touched), else 4 (both measured on the benchmark workloads'
// shapes: 12 consumer warps win at d_model 2048, 16 at d_model 7168).
int pick_nq(int T, int k, int E, int d, int f, int G) {
    const double bytes = (double)std::min(T * k, E) * 3.0 * d * f * 0.53125 / G;
    return bytes <= 1.0e6 ? 3 : 4;
}

bool decode_fused_supported(int T, int k, int E, int d, int f) {
    Layout l;
    const int G = num_sms();
    return plan_layout(T, k, E, d, f, G, pick_nq(T, k, E, d, f, G), &l);
}

cudaError_t launch_decode_fused(const FusedIn& in, cudaStream_t s) {
    const moe_w4_layer& W = *in.L;
    const int E = W.E, d = W.d_model, f = W.d_ff;
    const int G = num_sms();
    const int nq = pick_nq(in.T, in.k, E, d, f, G);
    Layout l;
    if (!plan_layout(in.T, in.k, E, d, f, G, nq, &l)) return cudaErrorInvalidValue;
    // codes as 32-word lines: gate_up [expert * 2 + (gate, up)][feature][line][32
    // words], box 8 features of both halves; down [row][line][32 words], box 16 rows
    CUtensorMap m13, m2;
    const uint64_t d13[4] = {32, (uint64_t)d / 256, (uint64_t)f, (uint64_t)E * 2};
    const uint64_t s13[3] = {128, (uint64_t)d / 2, (uint64_t)f * d / 2};
    const uint32_t b13[4] = {32, LINES, 8, 2};
    if (!make_tensor_map_u32(&m13, W.w13_q, 4, d13, s13, b13)) return cudaErrorInvalidValue;
    if (!make_tensor_map_3d(&m2, W.w2_q, 32, (uint64_t)f / 256, (uint64_t)E * d, 128, (uint64_t)f / 2, 32, LINES, 16))
        return cudaErrorInvalidValue;
    // fp16 scales and zeros [rows][groups]: by TMA when a row is a multiple of
    // 16 bytes (groups % 8 == 0): gate_up {groups, feature, expert * 2 + half}
    // box {8, 8, 2}, down {groups, row} box {8, 16}; by bulk copies when a row
    // fits one chunk (groups < 8; 16-byte aligned arrays); else with cp.async.
    // In the 3-pipeline instantiation (little weight per CTA) gate_up's scales
    // and zeros always go by the producer lanes' 4-byte cp.async: measured on
    // the d_model 2048 layer 17.45 against 17.95 us per layer with the TMA
    // boxes (outputs identical); on the d_model 7168 layer (4 pipelines) the
    // TMA boxes are the faster, 75.4 against 79.4 us.
    CUtensorMap m13s = m13, m13z = m13, m2s = m2, m2z = m2;
    const uint64_t Gd = (uint64_t)d / 128, Gf = (uint64_t)f / 128;
    bool sz13 = Gd % 8 == 0 && nq == 4, sz2 = Gf % 8 == 0;
    auto a16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
    if (sz13) {
        const uint64_t dims[3] = {Gd, (uint64_t)f, (uint64_t)E * 2}, str[2] = {Gd * 2, (uint64_t)f * Gd * 2};
        const uint32_t box[3] = {CHUNK_GROUPS, 8, 2};
        sz13 = make_tensor_map_u16(&m13s, W.w13_s, 3, dims, str, box) &&
               make_tensor_map_u16(&m13z, W.w13_z, 3, dims, str, box);
    }
    if (sz2) {
        const uint64_t dims[2] = {Gf, (uint64_t)E * d}, str[1] = {Gf * 2};
        const uint32_t box[2] = {CHUNK_GROUPS, 16};
        sz2 = make_tensor_map_u16(&m2s, W.w2_s, 2, dims, str, box) && make_tensor_map_u16(&m2z, W.w2_z, 2, dims, str, box);
    }
    Params p{};
    p.x = in.x;
    p.logits = in.logits;
    p.w13_s = W.w13_s;
    p.w13_z = W.w13_z;
    p.w2_s = W.w2_s;
    p.w2_z = W.w2_z;
    p.out = in.out;
    p.ids_out = in.ids_out;
    p.hb = reinterpret_cast<uint8_t*>(in.hb);
    auto* hdr = static_cast<uint32_t*>(in.ws);
    p.err = hdr;
    p.bar_count = reinterpret_cast<unsigned long long*>(hdr + WS_BAR_COUNT_WORD);
    p.T = in.T;
    p.k = in.k;
    p.E = E;
    p.d = d;
    p.f = f;
    p.nslot = l.nslot;
    p.off_sz = l.off_sz;
    p.off_bars = l.off_bars;
    p.off_xb = l.off_xb;
    p.off_cx = l.off_cx;
    p.off_hs = l.off_hs;
    p.off_ch = l.off_ch;
    p.off_red = l.off_red;
    p.off_red2 = l.off_red2;
    p.off_tab = l.off_tab;
    p.xb_stride = l.xb_stride;
    p.hs_stride = l.hs_stride;
    const bool bulk13 = Gd < CHUNK_GROUPS && a16(W.w13_s) && a16(W.w13_z);
    const bool bulk2 = Gf < CHUNK_GROUPS && a16(W.w2_s) && a16(W.w2_z);
    p.sz13_mode = sz13 ? SZ_TMA : (bulk13 ? SZ_BULK : SZ_CPASYNC);
    p.sz2_mode = sz2 ? SZ_TMA : (bulk2 ? SZ_BULK : SZ_CPASYNC);
    p.sz13_rs = p.sz13_mode == SZ_BULK ? (int)Gd * 2 : 16;
    p.fd_G = make_fastdiv((uint32_t)G);
    p.fd_T = make_fastdiv((uint32_t)in.T);
    p.fd_nct0 = make_fastdiv((uint32_t)(G / in.T));
    p.fd_nct1 = make_fastdiv((uint32_t)(G / in.T + 1));
    p.fd_nch1 = make_fastdiv((uint32_t)ceil_div(d / 128, CHUNK_GROUPS));
    p.fd_nch2 = make_fastdiv((uint32_t)ceil_div(f / 128, CHUNK_GROUPS));
    p.fd_nfb1 = make_fastdiv((uint32_t)(f / 8));
    p.fd_k = make_fastdiv((uint32_t)in.k);
    p.fd_ns4 = make_fastdiv((uint32_t)(l.nslot / nq));
    p.fd_xw = make_fastdiv((uint32_t)(d / 8));
    p.fd_hw = make_fastdiv((uint32_t)(f / 8));
    p.sz2_rs = p.sz2_mode == SZ_BULK ? (int)Gf * 2 : 16;

    static bool configured[2] = {false, false};
    if (!configured[nq - 3]) {
        cudaError_t e = nq == 3 ? cudaFuncSetAttribute(decode_fused_kernel<3>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_LIMIT)
                                : cudaFuncSetAttribute(decode_fused_kernel<4>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_LIMIT);
        if (e != cudaSuccess) return e;
        configured[nq - 3] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G);
    cfg.blockDim = dim3(nq == 3 ? Shape<3>::NTHREADS : Shape<4>::NTHREADS);
    cfg.dynamicSmemBytes = l.smem;
    cfg.stream = s;
    // cooperative (the grid barrier needs every CTA resident) and, where the
    // driver accepts it, a programmatic dependent of the previous kernel on the
    // stream (the kernel waits for it before touching global memory)
    static int pdl_ok = 1;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_ok ? 2 : 1;
    auto launch = [&]() {
        return nq == 3 ? cudaLaunchKernelEx(&cfg, decode_fused_kernel<3>, m13, m2, m13s, m13z, m2s, m2z, p)
                       : cudaLaunchKernelEx(&cfg, decode_fused_kernel<4>, m13, m2, m13s, m13z, m2s, m2z, p);
    };
    cudaError_t e = launch();
    if (e != cudaSuccess && pdl_ok) {
        // not accepted together with the cooperative launch: plain launch
        (void)cudaGetLastError();
        pdl_ok = 0;
        cfg.numAttrs = 1;
        e = launch();
    }
    note_launch();
    return e;
}

}  // namespace moe
