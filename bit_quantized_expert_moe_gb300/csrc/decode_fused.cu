// The whole MoE layer for a few tokens (decode) in one persistent kernel.
//
// With T <= 8 tokens the layer is a stream of the routed experts' int4 weights
// past a handful of activation vectors: "Performance and verification"
// (bloomery docs/performance.md), section "Why it is fast", reads every routed
// expert once per batch and takes the dot products on the weights as stored;
// "Measured results" (vllm-omni docs/edge/results.md), section Fidelity, fixes
// the W4A16 g128 format.  The kernel is built so that the weight stream never
// waits on anything but routing:
//
//   phase 0  every CTA routes all T tokens itself (top-k of the logits held
//            in shared memory, softmax over the selection) and sorts the T*k
//            assignments by expert, so no CTA waits for another to learn which
//            experts are needed.  CTA 0 writes the routing to topk_ids_out.
//   phase 1  gate_up: the CTA takes a contiguous share of the tiles
//            (touched expert u, 8 features) and computes, for each token routed
//            to u, the 8 gate and 8 up dot products over d_model, then
//            h = SiLU(gate) * up (fp16) into a global scratch.
//   barrier  one grid-wide arrival on a 64-bit counter in the workspace header
//            (all CTAs are co-resident: one per SM, cooperative launch); the
//            producer keeps loading phase-2 weights while it is pending.
//   phase 2  down + combine: the CTA takes a contiguous share of the units
//            (token t, 16 output features); for each of t's k experts it forms
//            16 down-projection dot products over d_ff, scales them by the
//            routing weight, and the unit's k contributions are added in slot
//            order in fp32 and written to out as bf16.
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
// Pipeline.  Warps 16..19 are producers (chunk q belongs to warp 16 + q % 4,
// since issuing one chunk keeps a warp busy for about a thousand cycles):
// lane 0 issues 3D TMA boxes of the packed codes (16 rows x 4 lines of 128 B =
// 2 groups each, 128-byte swizzle) into a ring of slots and all lanes copy
// the matching fp16 scales and zeros with 4-byte cp.async, tracked by the
// chunk's full mbarrier.  Warps 0..15 form 8 pairs; a tile belongs to one pair
// and each warp of the pair takes half of every chunk's groups (the slot is
// released after the warp's last copy from it); the two halves are added
// through shared memory.
// Every wait is bounded (2 s), after which the kernel records a timeout in the
// workspace error word, raises the CTA's abort flag and winds down.
#include <cfloat>
#include <climits>

#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using tc::WAIT_LIMIT_NS;

constexpr int CW = 16;                          // consumer warps (8 pairs)
constexpr int NPAIR = CW / 2;
constexpr int PRODUCER_WARP = CW;               // first producer warp
constexpr int NPROD = 4;                        // producer warps: chunk q is issued by warp q % NPROD
static_assert((NPROD & (NPROD - 1)) == 0, "NPROD must be a power of two");
constexpr int NTHREADS = 32 * (CW + NPROD);
constexpr int CONSUMER_THREADS = 32 * CW;
constexpr int LINES = 4;                        // 128-byte lines (2 groups each) per chunk row
constexpr int CHUNK_GROUPS = 2 * LINES;         // groups of 128 codes per chunk
constexpr int BOX_BYTES = 8 * LINES * 128;      // one TMA box: 8 rows x 4 lines
constexpr int SLOT_CODE = 2 * BOX_BYTES;        // 16 rows of codes
constexpr int SZ_ARRAY = 16 * CHUNK_GROUPS * 2; // fp16 [16 rows][8 groups]
constexpr int SLOT_BYTES = SLOT_CODE + 1024;    // codes + scales + zeros, 1024-byte aligned
constexpr uint32_t FULL_ARRIVALS = 1 + 32;      // expect_tx arrival + 32 cp.async arrivals
// "Full" barriers are indexed by chunk number modulo NFULL, not by ring slot:
// the pairs consume different chunks, so a pair may wait for chunk q before
// the chunk that last used q's ring slot has been consumed.  A pair's next
// chunk is at most NPAIR * (chunks per tile + 1) past its previous one, so with
// NFULL >= nslot + NPAIR * (chunks per tile + 1) + 1 the previous use of q's
// barrier (chunk q - NFULL) has always landed when q is waited on, and the
// barrier's parity names q's phase unambiguously.
constexpr int NFULL = 256;
static_assert((NFULL & (NFULL - 1)) == 0, "NFULL must be a power of two");
constexpr int MAX_T = 8;
constexpr int MAX_R = 64;
constexpr int ROW_PAD = 64;                     // bytes after each staged activation row
constexpr size_t SMEM_LIMIT = 232448;
constexpr int MIN_SLOTS = 6;

struct Tab {
    int32_t ids[MAX_R];    // routing, slot a = t*k + j
    float w[MAX_R];
    int32_t pos[MAX_R];    // permuted position of slot a
    int32_t ptok[MAX_R];   // token of permuted position i
    int32_t uexp[MAX_R];   // touched experts, ascending
    int32_t uoff[MAX_R];
    int32_t ucnt[MAX_R];
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
    int nslot;
    uint32_t off_bars, off_xb, off_cx, off_hs, off_ch, off_red, off_red2, off_tab;
    uint32_t off_cnt;          // phase-0 counters inside the ring, after the logits
    int xb_stride, hs_stride;  // bytes per staged row
};

// ------------------------------------------------------------ small helpers
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ float2 lds_f2(uint32_t a) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ float lds_half(uint32_t a) {
    uint16_t h;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(a));
    return __half2float(__ushort_as_half(h));
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" :: "r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
}
__device__ __forceinline__ uint4 ldg_cg16(const void* p) {
    uint4 r;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
__device__ __forceinline__ uint64_t ld_acquire_gpu64(const unsigned long long* p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint64_t atom_add_release_gpu(unsigned long long* p, uint64_t v) {
    uint64_t old;
    asm volatile("atom.add.release.gpu.global.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
    return old;
}
__device__ __forceinline__ void bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}

// D = A * B + D, m16n8k16, fp16 inputs, fp32 accumulation.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ routing
// Order-preserving map of a finite fp32 value to uint32 (larger value, larger
// key; -0 is folded onto +0 so that equal values give equal keys).  Every
// finite value maps above 0x007FFFFF, so 0 can stand for "no candidate".
__device__ __forceinline__ uint32_t route_key(float v) {
    if (v == 0.0f) v = 0.0f;
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Top-k of one token by one warp, logits read once from shared memory (`row`)
// into registers (VPL per lane: experts lane, lane+32, ...): k rounds of
// (warp maximum of the keys, then the lowest expert id among the lanes
// holding it), i.e. a sort by (-logit, id) on the exact fp32 values (router
// ids must match exactly: "Performance and verification", section "How it is
// verified").  Lane j (and j+32) keeps slot j; the weights are the softmax of
// the k <= 64 selected logits, in fp32.  No shared-memory traffic and no
// data-dependent branch inside the rounds.
template <int VPL>
__device__ __forceinline__ void route_token_regs(const float* row, int E, int k, int32_t* out_ids, float* out_w) {
    const int lane = threadIdx.x & 31;
    uint32_t key[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        key[i] = e < E ? route_key(row[e]) : 0u;
    }
    float vmax = 0.f, v0 = 0.f, v1 = 0.f;
    int id0 = 0, id1 = 0;
    for (int j = 0; j < k; ++j) {
        uint32_t bk = key[0];
        int bi = 0;
#pragma unroll
        for (int i = 1; i < VPL; ++i) {
            const bool better = key[i] > bk;  // ascending e within the lane: ties keep the lower id
            bk = better ? key[i] : bk;
            bi = better ? i : bi;
        }
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
        const int win = __reduce_min_sync(0xffffffffu, (bk == kmax && bk != 0u) ? lane + 32 * bi : INT_MAX);
        const bool mine = (win & 31) == lane;
#pragma unroll
        for (int i = 0; i < VPL; ++i) key[i] = (mine && i == (win >> 5)) ? 0u : key[i];
        // the winning key back to its value (route_key is invertible on finite values)
        const float v = __uint_as_float((kmax & 0x80000000u) ? (kmax & 0x7FFFFFFFu) : ~kmax);
        vmax = (j == 0) ? v : vmax;
        if (lane == j) { id0 = win; v0 = v; }
        if (lane + 32 == j) { id1 = win; v1 = v; }
    }
    const float ex0 = lane < k ? expf(v0 - vmax) : 0.f;
    const float ex1 = lane + 32 < k ? expf(v1 - vmax) : 0.f;
    float sum = ex0;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (k > 32) {
        float s1 = ex1;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s1 += __shfl_xor_sync(0xffffffffu, s1, off);
        sum += s1;
    }
    const float inv_sum = 1.0f / sum;
    if (lane < k) {
        out_ids[lane] = id0;
        out_w[lane] = ex0 * inv_sum;
    }
    if (lane + 32 < k) {
        out_ids[lane + 32] = id1;
        out_w[lane + 32] = ex1 * inv_sum;
    }
    __syncwarp();
}

__device__ __forceinline__ void route_token(const float* row, int E, int k, int32_t* out_ids, float* out_w) {
    const int nv = (E + 31) >> 5;
    if (nv <= 1) route_token_regs<1>(row, E, k, out_ids, out_w);
    else if (nv <= 2) route_token_regs<2>(row, E, k, out_ids, out_w);
    else if (nv <= 4) route_token_regs<4>(row, E, k, out_ids, out_w);
    else if (nv <= 8) route_token_regs<8>(row, E, k, out_ids, out_w);
    else if (nv <= 16) route_token_regs<16>(row, E, k, out_ids, out_w);
    else route_token_regs<32>(row, E, k, out_ids, out_w);
}

// -------------------------------------------------------- staged activations
// Position of word w (0..15) of a group inside a staged activation row: the
// four words a thread reads in turn land in four different bank quads.
__device__ __forceinline__ int stage_word(int w) { return (w & 12) | ((w ^ (w >> 2)) & 3); }

// Byte offset of feature (or input column) c inside a staged row: group c/128
// (256 bytes), word (c/8)%16 at stage_word, then the eight values of the word
// in the order 0,4,1,5,2,6,3,7 (the k-pairs of the MMA's B fragment).
__device__ __forceinline__ uint32_t staged_offset(int c) {
    const int i = c & 7;
    const int pos = (i < 4) ? 2 * i : 2 * (i - 4) + 1;
    return (uint32_t)((c >> 7) * 256 + stage_word((c >> 3) & 15) * 16 + pos * 2);
}

// Eight fp16 values in natural order (four f16x2 registers (v0,v1), (v2,v3),
// (v4,v5), (v6,v7)) -> the staged word: (v0,v4), (v1,v5), (v2,v6), (v3,v7).
__device__ __forceinline__ uint4 to_mma_order(uint32_t p01, uint32_t p23, uint32_t p45, uint32_t p67) {
    uint4 o;
    o.x = __byte_perm(p01, p45, 0x5410);
    o.y = __byte_perm(p01, p45, 0x7632);
    o.z = __byte_perm(p23, p67, 0x5410);
    o.w = __byte_perm(p23, p67, 0x7632);
    return o;
}
// A staged word's contributions to (C1, C2).
__device__ __forceinline__ float2 word_c1c2(uint4 o) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&o.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&o.y));
    const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&o.z));
    const float2 e = __half22float2(*reinterpret_cast<const __half2*>(&o.w));
    const float even = (a.x + a.y) + (c.x + c.y);  // k = 0, 4, 2, 6
    const float odd = (b.x + b.y) + (e.x + e.y);   // k = 1, 5, 3, 7
    return make_float2(1024.0f * even + 64.0f * odd, even + odd);
}
// Sum over the 16 lanes of a half-warp (one group of 16 words).
__device__ __forceinline__ float2 halfwarp_sum(float2 v) {
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
        v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
        v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
    }
    return v;
}

// One group (128 codes) of one 16-row tile, as this warp takes it from a ring
// slot: the packed words of rows g and g + 8 (words 4t..4t+3 of the group)
// and the two rows' scales and zeros.  sa: slot address; gl: group inside the
// chunk.  Loading all of a chunk's groups first lets the warp give the slot
// back before it computes.
struct GroupA {
    uint4 wa, wb;
    float s0, z0, s1, z1;
};
__device__ __forceinline__ void load_group(GroupA& ga, uint32_t sa, int gl, int g, int t) {
    const int ell = gl >> 1;
    const uint32_t phys = (uint32_t)((((gl & 1) << 2) | t) ^ (((g & 1) << 2) | ell));
    const uint32_t aoff = (uint32_t)(g * 512 + ell * 128) + (phys << 4);
    ga.wa = lds128(sa + aoff);              // row g
    ga.wb = lds128(sa + BOX_BYTES + aoff);  // row g + 8
    const uint32_t szb = sa + SLOT_CODE + (uint32_t)(gl * 2);
    ga.s0 = lds_half(szb + g * 16);
    ga.z0 = lds_half(szb + SZ_ARRAY + g * 16);
    ga.s1 = lds_half(szb + (8 + g) * 16);
    ga.z1 = lds_half(szb + SZ_ARRAY + (8 + g) * 16);
}

// The group's 8 MMAs and its epilogue into acc.  bg: staged B row address of
// this lane's column at the group; c0, c1: C1/C2 addresses of columns 2t and
// 2t + 1 at the group; wscale: factor on the scales (routing weight in phase 2).
__device__ __forceinline__ void compute_group(float (&acc)[4], const GroupA& ga, int t, uint32_t bg, uint32_t c0,
                                              uint32_t c1, float wscale) {
    uint4 b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) b[i] = lds128(bg + ((uint32_t)stage_word(4 * t + i) << 4));
    const uint32_t A[4] = {ga.wa.x, ga.wa.y, ga.wa.z, ga.wa.w};
    const uint32_t Bw[4] = {ga.wb.x, ga.wb.y, ga.wb.z, ga.wb.w};
    float da[4] = {0.f, 0.f, 0.f, 0.f}, db[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t x = A[i], y = Bw[i];
        const uint32_t xs = x >> 8, ys = y >> 8;
        const uint32_t a0 = lop_mask_or(x, 0x000F000Fu, 0x64006400u);   // (q0, q4) + 1024
        const uint32_t a2 = lop_mask_or(x, 0x00F000F0u, 0x54005400u);   // (q1, q5) + 64
        const uint32_t a1 = lop_mask_or(y, 0x000F000Fu, 0x64006400u);
        const uint32_t a3 = lop_mask_or(y, 0x00F000F0u, 0x54005400u);
        mma16816(da, a0, a1, a2, a3, b[i].x, b[i].y);
        const uint32_t e0 = lop_mask_or(xs, 0x000F000Fu, 0x64006400u);  // (q2, q6) + 1024
        const uint32_t e2 = lop_mask_or(xs, 0x00F000F0u, 0x54005400u);  // (q3, q7) + 64
        const uint32_t e1 = lop_mask_or(ys, 0x000F000Fu, 0x64006400u);
        const uint32_t e3 = lop_mask_or(ys, 0x00F000F0u, 0x54005400u);
        mma16816(db, e0, e1, e2, e3, b[i].z, b[i].w);
    }
    const float s0 = ga.s0 * wscale, s1 = ga.s1 * wscale;
    const float2 ca = lds_f2(c0), cb = lds_f2(c1);
    acc[0] = fmaf(s0, (da[0] + db[0]) - fmaf(ga.z0, ca.y, ca.x), acc[0]);
    acc[1] = fmaf(s0, (da[1] + db[1]) - fmaf(ga.z0, cb.y, cb.x), acc[1]);
    acc[2] = fmaf(s1, (da[2] + db[2]) - fmaf(ga.z1, ca.y, ca.x), acc[2]);
    acc[3] = fmaf(s1, (da[3] + db[3]) - fmaf(ga.z1, cb.y, cb.x), acc[3]);
}

// A chunk for this warp: wait for it, then for each of this warp's groups
// (half of the chunk's gcv groups) copy the group into registers and compute
// it; the slot is given back right after the last group's copy, before its
// math.
__device__ __forceinline__ void consume_chunk(float (&acc)[4], uint32_t full, uint32_t empty, uint32_t parity,
                                              uint32_t sa, int gcv, int half, int g, int t, int gi0, uint32_t brow_a,
                                              uint32_t c0_a, uint32_t c1_a, float wscale, volatile int* abort_flag,
                                              uint32_t* err) {
    const bool ready = tc::mbar_wait(full, parity, abort_flag, err);
    const int ng = gcv >> 1, gb = half * ng;
    if (!ready) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) tc::mbar_arrive(empty);
        return;
    }
    for (int i = 0; i < ng; ++i) {
        GroupA ga;
        load_group(ga, sa, gb + i, g, t);
        if (i == ng - 1) {
            __syncwarp();
            if ((threadIdx.x & 31) == 0) tc::mbar_arrive(empty);
        }
        const int gi = gi0 + gb + i;
        compute_group(acc, ga, t, brow_a + 256u * gi, c0_a + 8u * gi, c1_a + 8u * gi, wscale);
    }
}

// ------------------------------------------------------------------ kernel
__global__ void __launch_bounds__(NTHREADS, 1)
decode_fused_kernel(const __grid_constant__ CUtensorMap map13, const __grid_constant__ CUtensorMap map2,
                    const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sbase = smem_u32(sm);
    Tab& tab = *reinterpret_cast<Tab*>(sm + p.off_tab);
    volatile int* abort_flag = &tab.abort;
    const uint32_t full0 = sbase + p.off_bars;
    const uint32_t empty0 = full0 + 8u * NFULL;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = p.T, k = p.k, R = T * k, E = p.E, d = p.d, f = p.f;
    const int Gd = d >> 7, Gf = f >> 7;
    const int G = gridDim.x, cta = blockIdx.x;
    const int nslot = p.nslot;

    // ------------------------------------------------ phase 0: init, routing
    // Scratch of phase 0 lives in the ring, which is idle until the producers
    // start: the routed tokens' logits, then per-expert counts of the first and
    // second 32 assignments and the touched-expert bitmask.
    float* lgs = reinterpret_cast<float*>(sm);
    int32_t* cnt_a = reinterpret_cast<int32_t*>(sm + p.off_cnt);
    int32_t* cnt_b = cnt_a + E;
    uint32_t* emask = reinterpret_cast<uint32_t*>(cnt_b + E);
    int32_t* wpre = reinterpret_cast<int32_t*>(emask + 32);
    if (threadIdx.x == 0) tab.abort = 0;
    if (warp == PRODUCER_WARP) {
        for (int i = lane; i < NFULL; i += 32) tc::mbar_init(full0 + 8u * i, FULL_ARRIVALS);
        for (int i = lane; i < nslot; i += 32) tc::mbar_init(empty0 + 8u * i, 2);
        if (lane == 0) {
            tc::fence_mbar_init();
            tc::tma_prefetch_desc(&map13);
            tc::tma_prefetch_desc(&map2);
        }
    } else if (warp == PRODUCER_WARP + 1) {
        for (int i = lane; i < 2 * E; i += 32) cnt_a[i] = 0;
        emask[lane] = 0;
    }
    if (warp < T) {
        // this token's logits into shared memory, then top-k
        float* lrow = lgs + warp * E;
        const float* src = p.logits + (size_t)warp * E;
        for (int e = lane; e < E; e += 32) lrow[e] = __ldg(src + e);
        __syncwarp();
        route_token(lrow, E, k, &tab.ids[warp * k], &tab.w[warp * k]);
    } else if (warp < CW) {
        // activations -> fp16 in MMA order, plus C1/C2 per (token, group)
        const int nthr = (CW - T) * 32, tid = (warp - T) * 32 + lane;
        const int wpr = d >> 3;  // 16-byte words per row (a multiple of 32)
        float2* cx = reinterpret_cast<float2*>(sm + p.off_cx);
        for (int wi = tid; wi < T * wpr; wi += nthr) {
            const int t = wi / wpr, wr = wi - t * wpr;
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
            const uint4 o = to_mma_order(q[0], q[1], q[2], q[3]);
            sts128(sbase + p.off_xb + (uint32_t)(t * p.xb_stride) + staged_offset(wr * 8), o);
            const float2 c = halfwarp_sum(word_c1c2(o));
            if ((lane & 15) == 0) cx[t * Gd + (wr >> 4)] = c;
        }
        // the zero row (index T): columns without a token
        for (int i = tid; i < (p.xb_stride >> 4); i += nthr)
            sts128(sbase + p.off_xb + (uint32_t)(T * p.xb_stride) + 16u * i, make_uint4(0, 0, 0, 0));
        for (int i = tid; i < Gd; i += nthr) cx[T * Gd + i] = make_float2(0.f, 0.f);
    }
    __syncthreads();
    if (warp == 0) {
        // stable counting sort of the R <= 64 assignments by expert: per-expert
        // counts of the two halves, the touched-expert bitmask (ascending expert
        // list by a warp scan), ranks inside an expert from __match_any_sync
        const int a0 = lane, a1 = lane + 32;
        const bool v0 = a0 < R, v1 = a1 < R;
        const int e0 = v0 ? tab.ids[a0] : 0, e1 = v1 ? tab.ids[a1] : 0;
        if (v0) {
            atomicAdd(&cnt_a[e0], 1);
            atomicOr(&emask[e0 >> 5], 1u << (e0 & 31));
        }
        if (v1) {
            atomicAdd(&cnt_b[e1], 1);
            atomicOr(&emask[e1 >> 5], 1u << (e1 & 31));
        }
        const uint32_t m0 = __match_any_sync(0xffffffffu, v0 ? e0 : -1 - lane);
        const uint32_t m1 = __match_any_sync(0xffffffffu, v1 ? e1 : -1 - lane);
        const uint32_t lt = (1u << lane) - 1u;
        __syncwarp();
        // ascending expert list: lane l owns bitmask word l
        const uint32_t w = emask[lane];
        int incl = __popc(w);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int U = __shfl_sync(0xffffffffu, incl, 31);
        int pre = incl - __popc(w);
        wpre[lane] = pre;
        for (uint32_t b = w; b; b &= b - 1) tab.uexp[pre++] = 32 * lane + (__ffs(b) - 1);
        __syncwarp();
        // expert counts and offsets in list order (U <= 64)
        const int c0 = lane < U ? cnt_a[tab.uexp[lane]] + cnt_b[tab.uexp[lane]] : 0;
        const int c1 = lane + 32 < U ? cnt_a[tab.uexp[lane + 32]] + cnt_b[tab.uexp[lane + 32]] : 0;
        int s0 = c0, s1 = c1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y0 = __shfl_up_sync(0xffffffffu, s0, o);
            const int y1 = __shfl_up_sync(0xffffffffu, s1, o);
            if (lane >= o) {
                s0 += y0;
                s1 += y1;
            }
        }
        const int tot0 = __shfl_sync(0xffffffffu, s0, 31);
        if (lane < U) {
            tab.ucnt[lane] = c0;
            tab.uoff[lane] = s0 - c0;
        }
        if (lane + 32 < U) {
            tab.ucnt[lane + 32] = c1;
            tab.uoff[lane + 32] = tot0 + s1 - c1;
        }
        __syncwarp();
        // permuted position of each assignment
        auto uidx = [&](int e) {
            return wpre[e >> 5] + __popc(emask[e >> 5] & ((1u << (e & 31)) - 1u));
        };
        if (v0) {
            const int pos = tab.uoff[uidx(e0)] + __popc(m0 & lt);
            tab.pos[a0] = pos;
            tab.ptok[pos] = a0 / k;
        }
        if (v1) {
            const int pos = tab.uoff[uidx(e1)] + cnt_a[e1] + __popc(m1 & lt);
            tab.pos[a1] = pos;
            tab.ptok[pos] = a1 / k;
        }
        if (lane == 0) tab.n_uniq = U;
    }
    __syncthreads();
    if (cta == 0 && p.ids_out)
        for (int a = threadIdx.x; a < R; a += NTHREADS) p.ids_out[a] = tab.ids[a];

    // work shares
    const int U = tab.n_uniq;
    const int nfb1 = f >> 3, nrb = d >> 4;
    const int N1 = U * nfb1, N2 = T * nrb;
    // (32-bit products: N1 <= 64 * 2048 and N2 <= 8 * 1024, times G < 2^12)
    const int a1 = cta * N1 / G, b1 = (cta + 1) * N1 / G;
    const int a2 = cta * N2 / G, b2 = (cta + 1) * N2 / G;
    const int n1 = b1 - a1, n2u = b2 - a2, n2t = n2u * k;
    const int nch1 = ceil_div(Gd, CHUNK_GROUPS), nch2 = ceil_div(Gf, CHUNK_GROUPS);

    // ---------------------------------------------------------- producers
    if (warp >= PRODUCER_WARP) {
        const uint32_t pw = (uint32_t)(warp - PRODUCER_WARP);
        // chunk counter q = round * nslot + slot, kept incrementally (no division
        // in the issue loop: a runtime divide costs tens of dependent instructions)
        uint32_t q = 0, slot = 0, round = 0;
        bool ok = true;
        auto advance = [&]() {
            ++q;
            if (++slot == (uint32_t)nslot) {
                slot = 0;
                ++round;
            }
        };
        auto issue = [&](const CUtensorMap* map, int row0, int row1, int chunk, const uint16_t* s_arr,
                         const uint16_t* z_arr, int Gk) {
            if ((q & (NPROD - 1)) != pw) {  // another producer warp's chunk
                advance();
                return;
            }
            const uint32_t full = full0 + 8u * (q & (NFULL - 1)), empty = empty0 + 8u * slot;
            if (round > 0) {
                // one lane waits and the warp follows its verdict; __syncwarp orders
                // the consumers' last reads of the slot before any lane's new copies
                int w = 1;
                if (lane == 0) w = tc::mbar_wait(empty, (round - 1) & 1u, abort_flag, p.err);
                w = __shfl_sync(0xffffffffu, w, 0);
                __syncwarp();
                if (!w) {
                    ok = false;
                    return;
                }
            }
            const uint32_t dst = sbase + (uint32_t)slot * SLOT_BYTES;
            if (lane == 0) {
                tc::mbar_arrive_expect_tx(full, SLOT_CODE);
                tc::tma_load_3d(dst, map, full, 0, chunk * LINES, row0);
                tc::tma_load_3d(dst + BOX_BYTES, map, full, 0, chunk * LINES, row1);
            }
            const int arr = lane >> 4, r = lane & 15;
            const uint16_t* base = arr ? z_arr : s_arr;
            const int grow = r < 8 ? row0 + r : row1 + (r - 8);
            const int g0 = chunk * CHUNK_GROUPS;
            const int gcv = min(CHUNK_GROUPS, Gk - g0);
            const uint16_t* src = base + (size_t)grow * Gk + g0;
            const uint32_t sdst = dst + SLOT_CODE + (uint32_t)(arr * SZ_ARRAY + r * 16);
            for (int i = 0; i < (gcv >> 1); ++i) cp_async4(sdst + 4u * i, src + 2 * i);
            tc::cp_async_mbar_arrive_noinc(full);
            advance();
        };
        // Issue order: tiles in batches of NPAIR (one per pair); inside a batch,
        // chunk c of every tile before chunk c + 1, so that every pair has data
        // in the ring at once (the consumers' chunk numbering follows it).
        // lane pp < NPAIR holds the first weight row of tile b0 + pp
        for (int b0 = 0; b0 < n1 && ok; b0 += NPAIR) {
            const int nb = min(NPAIR, n1 - b0);
            int my_rg = 0;
            if (lane < nb) {
                const int tau = a1 + b0 + lane, u = tau / nfb1, fb = tau - u * nfb1;
                my_rg = tab.uexp[u] * 2 * f + 8 * fb;
            }
            for (int c = 0; c < nch1 && ok; ++c)
                for (int pp = 0; pp < nb && ok; ++pp) {
                    const int rg = __shfl_sync(0xffffffffu, my_rg, pp);
                    issue(&map13, rg, rg + f, c, p.w13_s, p.w13_z, Gd);
                }
        }
        for (int b0 = 0; b0 < n2t && ok; b0 += NPAIR) {
            const int nb = min(NPAIR, n2t - b0);
            int my_rg = 0;
            if (lane < nb) {
                const int i2 = b0 + lane, ul = i2 / k, j = i2 - ul * k;
                const int ups = a2 + ul, t = ups / nrb, rb = ups - t * nrb;
                my_rg = tab.ids[t * k + j] * d + 16 * rb;
            }
            for (int c = 0; c < nch2 && ok; ++c)
                for (int pp = 0; pp < nb && ok; ++pp) {
                    const int rg = __shfl_sync(0xffffffffu, my_rg, pp);
                    issue(&map2, rg, rg + 8, c, p.w2_s, p.w2_z, Gf);
                }
        }
        // drain: the last use of every slot must have landed before the CTA exits
        // (each warp waits for its own chunks among the last nslot)
        const uint32_t issued = q;
        const uint32_t first = issued > (uint32_t)nslot ? issued - (uint32_t)nslot : 0u;
        for (uint32_t qq = first; qq < issued; ++qq) {
            if (qq % NPROD != pw) continue;
            const uint32_t full = full0 + 8u * (qq & (NFULL - 1));
            const uint32_t par = (qq / NFULL) & 1u;
            if (tc::mbar_try_wait(full, par)) continue;
            const uint64_t t0 = globaltimer_ns();
            while (!tc::mbar_try_wait(full, par)) {
                if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
                    set_error(p.err, ERRBIT_TIMEOUT);
                    break;
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int pair = warp >> 1, half = warp & 1;
    const int g = lane >> 2, t4 = lane & 3;
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
    const uint32_t xb = sbase + p.off_xb, cxa = sbase + p.off_cx;

    // phase 1: gate_up tiles
    for (int tl = pair; tl < n1; tl += NPAIR) {
        const int tau = a1 + tl, u = tau / nfb1, fb = tau - u * nfb1;
        const int cnt = tab.ucnt[u], off = tab.uoff[u];
        const int col = lane >> 2;
        const int brow = col < cnt ? tab.ptok[off + col] : T;
        const int cr0 = 2 * t4 < cnt ? tab.ptok[off + 2 * t4] : T;
        const int cr1 = 2 * t4 + 1 < cnt ? tab.ptok[off + 2 * t4 + 1] : T;
        const uint32_t brow_a = xb + (uint32_t)(brow * p.xb_stride);
        const uint32_t c0_a = cxa + (uint32_t)(cr0 * Gd * 8), c1_a = cxa + (uint32_t)(cr1 * Gd * 8);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const int b0 = tl - pair, nb = min(NPAIR, n1 - b0);
        for (int c = 0; c < nch1; ++c) {
            const uint32_t q = (uint32_t)(b0 * nch1 + c * nb + pair);  // interleaved issue order
            const int slot = (int)(q % (uint32_t)nslot);
            consume_chunk(acc, full0 + 8u * (q % NFULL), empty0 + 8u * slot, (q / NFULL) & 1u,
                          sbase + (uint32_t)slot * SLOT_BYTES, min(CHUNK_GROUPS, Gd - c * CHUNK_GROUPS), half, g,
                          t4, c * CHUNK_GROUPS, brow_a, c0_a, c1_a, 1.0f, abort_flag, p.err);
        }
        pair_reduce(acc);
        if (half == 0 && !*abort_flag) {
            // h = SiLU(gate) * up for feature 8 fb + g and columns 2 t4, 2 t4 + 1
            const uint32_t hoff = staged_offset(8 * fb + g);
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int colm = 2 * t4 + m;
                if (colm < cnt) {
                    const float h = silu(acc[m]) * acc[2 + m];
                    const __half hh = __float2half_rn(h);
                    if (__hisinf(hh) || __hisnan(hh)) set_error(p.err, ERRBIT_F16_RANGE);
                    *reinterpret_cast<__half*>(p.hb + (size_t)(off + colm) * (f * 2) + hoff) = hh;
                }
            }
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

    // stage the h rows of this CTA's tokens (<= 2 tokens x k slots) + C1/C2
    const int tok_lo = n2u > 0 ? a2 / nrb : 0;
    const int tok_hi = n2u > 0 ? (b2 - 1) / nrb : -1;
    const int nloc = (tok_hi - tok_lo + 1) * k;  // staged rows; row 2k is the zero row
    const int zrow = 2 * k;
    const uint32_t hs = sbase + p.off_hs, cha = sbase + p.off_ch;
    float2* ch = reinterpret_cast<float2*>(sm + p.off_ch);
    if (!*abort_flag) {
        const int tid = threadIdx.x;
        const int wpr = f >> 3;  // 16-byte words per row, a multiple of 32
        for (int wi = tid; wi < nloc * wpr; wi += CONSUMER_THREADS) {
            const int lr = wi / wpr, wr = wi - lr * wpr;
            const int a = (tok_lo + lr / k) * k + lr % k;
            const uint4 o = ldg_cg16(p.hb + (size_t)tab.pos[a] * (f * 2) + 16 * (size_t)wr);
            sts128(hs + (uint32_t)(lr * p.hs_stride) + 16u * wr, o);
            // a staged word holds one word's 8 values in MMA order (staged_offset)
            const float2 c = halfwarp_sum(word_c1c2(o));
            if ((lane & 15) == 0) ch[lr * Gf + (wr >> 4)] = c;
        }
        for (int i = tid; i < (p.hs_stride >> 4); i += CONSUMER_THREADS)
            sts128(hs + (uint32_t)(zrow * p.hs_stride) + 16u * i, make_uint4(0, 0, 0, 0));
        for (int i = tid; i < Gf; i += CONSUMER_THREADS) ch[zrow * Gf + i] = make_float2(0.f, 0.f);
    }
    bar_sync(1, CONSUMER_THREADS);

    // phase 2: down tiles (unit, slot j); one partial per (unit, pair)
    float* red2 = reinterpret_cast<float*>(sm + p.off_red2);  // [unit][pair][16]
    {
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
        const uint32_t qbase = (uint32_t)(n1 * nch1);
        for (int i2 = pair; i2 < n2t; i2 += NPAIR) {
            const int ul = i2 / k, j = i2 - ul * k;
            if (ul != cur) {
                if (cur >= 0) flush(cur);
                cur = ul;
                acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
            }
            const int ups = a2 + ul, t = ups / nrb;
            const int a = t * k + j;
            const float wj = tab.w[a];
            const int lr = (t - tok_lo) * k + j;
            const int brow = (lane >> 2) == 0 ? lr : zrow;
            const int cr0 = t4 == 0 ? lr : zrow;
            const uint32_t brow_a = hs + (uint32_t)(brow * p.hs_stride);
            const uint32_t c0_a = cha + (uint32_t)(cr0 * Gf * 8), c1_a = cha + (uint32_t)(zrow * Gf * 8);
            const int b0 = i2 - pair, nb = min(NPAIR, n2t - b0);
            for (int c = 0; c < nch2; ++c) {
                const uint32_t q = qbase + (uint32_t)(b0 * nch2 + c * nb + pair);  // interleaved issue order
                const int slot = (int)(q % (uint32_t)nslot);
                consume_chunk(acc, full0 + 8u * (q % NFULL), empty0 + 8u * slot, (q / NFULL) & 1u,
                              sbase + (uint32_t)slot * SLOT_BYTES, min(CHUNK_GROUPS, Gf - c * CHUNK_GROUPS), half, g,
                              t4, c * CHUNK_GROUPS, brow_a, c0_a, c1_a, wj, abort_flag, p.err);
            }
        }
        if (cur >= 0) flush(cur);
    }
    bar_sync(1, CONSUMER_THREADS);

    // out[t][16 rb + r] = contributions of the unit's slots, in slot order
    if (!*abort_flag) {
        const int nj = min(k, NPAIR);
        for (int idx = threadIdx.x; idx < n2u * 16; idx += CONSUMER_THREADS) {
            const int ul = idx >> 4, r = idx & 15;
            const int ups = a2 + ul, t = ups / nrb, rb = ups - t * nrb;
            float sum = 0.f;
            for (int j = 0; j < nj; ++j) sum += red2[(ul * NPAIR + (ul * k + j) % NPAIR) * 16 + r];
            p.out[(size_t)t * d + 16 * rb + r] = float_to_bf16_bits(sum);
        }
    }
}

struct Layout {
    int nslot;
    size_t smem;
    uint32_t off_bars, off_xb, off_cx, off_hs, off_ch, off_red, off_red2, off_tab, off_cnt;
    int xb_stride, hs_stride;
};

bool plan_layout(int T, int k, int E, int d, int f, int G, Layout* L) {
    if (T < 1 || T > MAX_T || k < 1 || T * k > MAX_R || E < 1 || E > 1024) return false;
    if (d % 256 || f % 256) return false;
    Layout l{};
    l.xb_stride = 2 * d + ROW_PAD;
    l.hs_stride = 2 * f + ROW_PAD;
    const int n2u_max = ceil_div(T * (d / 16), G) + 1;
    size_t fixed = 0;
    auto take = [&](size_t bytes) {
        const size_t o = fixed;
        fixed = align_up(fixed + bytes, 128);
        return (uint32_t)o;
    };
    // offsets relative to the end of the ring and its barriers (rebased below).
    // The staged activations (+ C1/C2) are read in phase 1 only and the staged
    // h rows (+ C1/C2) are written after the grid barrier: one shared region.
    const size_t sx = align_up((size_t)(T + 1) * l.xb_stride, 128) + (size_t)(T + 1) * (d / 128) * 8;
    const size_t sh = align_up((size_t)(2 * k + 1) * l.hs_stride, 128) + (size_t)(2 * k + 1) * (f / 128) * 8;
    const uint32_t o_xb = take(std::max(sx, sh));
    const uint32_t o_cx = o_xb + (uint32_t)align_up((size_t)(T + 1) * l.xb_stride, 128);
    const uint32_t o_hs = o_xb;
    const uint32_t o_ch = o_xb + (uint32_t)align_up((size_t)(2 * k + 1) * l.hs_stride, 128);
    const uint32_t o_red = take((size_t)NPAIR * 2 * 32 * 4 * 4);
    const uint32_t o_red2 = take((size_t)n2u_max * NPAIR * 16 * 4);
    const uint32_t o_tab = take(sizeof(Tab));
    if (fixed + 1024 >= SMEM_LIMIT) return false;
    const size_t avail = SMEM_LIMIT - 1024 - fixed;
    int nslot = (int)((avail - 8 * NFULL) / (SLOT_BYTES + 8));
    nslot = std::min(nslot, 32);
    if (nslot < MIN_SLOTS) return false;
    const int nch_max = ceil_div(std::max(d, f) / 128, CHUNK_GROUPS);
    if (nslot + NPAIR * (nch_max + 1) + 1 > NFULL) return false;
    // phase-0 scratch in the ring: logits, two count arrays, bitmask, word prefixes
    l.off_cnt = (uint32_t)align_up((size_t)T * E * 4, 16);
    if (l.off_cnt + (size_t)8 * E + 256 > (size_t)nslot * SLOT_BYTES) return false;
    const uint32_t ring = (uint32_t)nslot * SLOT_BYTES;
    const uint32_t bars = (uint32_t)align_up((size_t)8 * (NFULL + nslot), 128);
    l.nslot = nslot;
    l.off_bars = ring;
    l.off_xb = ring + bars + o_xb;
    l.off_cx = ring + bars + o_cx;
    l.off_hs = ring + bars + o_hs;
    l.off_ch = ring + bars + o_ch;
    l.off_red = ring + bars + o_red;
    l.off_red2 = ring + bars + o_red2;
    l.off_tab = ring + bars + o_tab;
    l.smem = 1024 + ring + bars + fixed;
    if (l.smem > SMEM_LIMIT) return false;
    *L = l;
    return true;
}

}  // namespace

bool decode_fused_supported(int T, int k, int E, int d, int f) {
    Layout l;
    return plan_layout(T, k, E, d, f, num_sms(), &l);
}

cudaError_t launch_decode_fused(const FusedIn& in, cudaStream_t s) {
    const moe_w4_layer& W = *in.L;
    const int E = W.E, d = W.d_model, f = W.d_ff;
    const int G = num_sms();
    Layout l;
    if (!plan_layout(in.T, in.k, E, d, f, G, &l)) return cudaErrorInvalidValue;
    // codes viewed as [rows][lines of 32 words][32 words]
    CUtensorMap m13, m2;
    if (!make_tensor_map_3d(&m13, W.w13_q, 32, (uint64_t)d / 256, (uint64_t)E * 2 * f, 128, (uint64_t)d / 2, 32,
                            LINES, 8))
        return cudaErrorInvalidValue;
    if (!make_tensor_map_3d(&m2, W.w2_q, 32, (uint64_t)f / 256, (uint64_t)E * d, 128, (uint64_t)f / 2, 32, LINES, 8))
        return cudaErrorInvalidValue;
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
    p.off_bars = l.off_bars;
    p.off_xb = l.off_xb;
    p.off_cx = l.off_cx;
    p.off_hs = l.off_hs;
    p.off_ch = l.off_ch;
    p.off_red = l.off_red;
    p.off_red2 = l.off_red2;
    p.off_tab = l.off_tab;
    p.off_cnt = l.off_cnt;
    p.xb_stride = l.xb_stride;
    p.hs_stride = l.hs_stride;

    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(decode_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SMEM_LIMIT);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = l.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, decode_fused_kernel, m13, m2, p);
    note_launch();
    return e;
}

}  // namespace moe
