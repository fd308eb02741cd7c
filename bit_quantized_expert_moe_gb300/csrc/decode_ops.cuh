// Device helpers of the decode regime: the int4 chunk format of the
// shared-memory ring, routing in registers (also used by the router kernel),
// the staged fp16 activation layout and the m16n8k16 group product on
// register-dequantised codes.  decode_fused.cu puts them together.
#pragma once

#include <cfloat>
#include <climits>

#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace dec {

constexpr int LINES = 4;                        // 128-byte lines (2 groups each) per chunk row
constexpr int CHUNK_GROUPS = 2 * LINES;         // groups of 128 codes per chunk
constexpr int BOX_BYTES = 8 * LINES * 128;      // 8 rows x 4 lines (rows g; rows g + 8 follow)
constexpr int SLOT_CODE = 2 * BOX_BYTES;        // one TMA box: 16 rows of codes (a multiple of the 1024-byte swizzle atom)
constexpr int SZ_ARRAY = 16 * CHUNK_GROUPS * 2; // fp16 [16 rows][8 groups]
constexpr int SLOT_SZ = 2 * SZ_ARRAY;           // scales, then zeros
constexpr int MAX_T = 8;
constexpr int MAX_R = 64;
constexpr int ROW_PAD = 64;                     // bytes after each staged activation row
constexpr size_t SMEM_LIMIT = 232448;
// Scales and zeros of a chunk: by TMA boxes where a row of groups is a
// multiple of 16 bytes (groups % 8 == 0; [16 rows][8 groups] in the slot), by
// plain bulk copies where a whole row fits one chunk (the chunk's rows are
// then contiguous: [16 rows][groups] in the slot), else by 4-byte cp.async.
enum { SZ_CPASYNC = 0, SZ_TMA = 1, SZ_BULK = 2 };

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
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
    uint16_t h;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(a));
    return h;
}
// 16-byte shared load done only by lanes with `active` set (others get zeros):
// lanes that skip it issue no shared-memory wavefronts.
__device__ __forceinline__ uint4 lds128_if(uint32_t a, uint32_t active) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %5, 0;\n\t"
        "@p ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n\t}"
        : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w) : "r"(a), "r"(active));
    return v;
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
    return (uint32_t)((c >> 7) * 256 + stage_word((c >> 3) & 15) * 16 + k8_pos(c & 7) * 2);
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

// Offset of this lane's 16 bytes of group gl of row g inside a slot's codes
// (row g + 8 is the same offset in the second box): the TMA box's 128-byte
// swizzle XORs the 16-byte unit index with the row's index inside the
// 1024-byte swizzle atom.
__device__ __forceinline__ uint32_t a_offset(int gl, int g, int t) {
    const int ell = gl >> 1;
    const uint32_t phys = (uint32_t)((((gl & 1) << 2) | t) ^ (((g & 1) << 2) | ell));
    return (uint32_t)(g * 512 + ell * 128) + (phys << 4);
}

// The group's 8 MMAs and its epilogue into acc.  wa, wb: this lane's packed
// words of rows g and g + 8; s0, z0, s1, z1: the two rows' scale and zero;
// bg: staged B row address of this lane's column at the group (loaded only
// where bact is set: B columns without a token are zero); c0, c1: C1/C2
// addresses of columns 2t and 2t + 1 at the group.
__device__ __forceinline__ void compute_group(float (&acc)[4], uint4 wa, uint4 wb, float s0, float z0, float s1,
                                              float z1, int t, uint32_t bg, uint32_t bact, uint32_t c0, uint32_t c1) {
    uint4 b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) b[i] = lds128_if(bg + ((uint32_t)stage_word(4 * t + i) << 4), bact);
    const uint32_t A[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t Bw[4] = {wb.x, wb.y, wb.z, wb.w};
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
    const float2 ca = lds_f2(c0), cb = lds_f2(c1);
    acc[0] = fmaf(s0, (da[0] + db[0]) - fmaf(z0, ca.y, ca.x), acc[0]);
    acc[1] = fmaf(s0, (da[1] + db[1]) - fmaf(z0, cb.y, cb.x), acc[1]);
    acc[2] = fmaf(s1, (da[2] + db[2]) - fmaf(z1, ca.y, ca.x), acc[2]);
    acc[3] = fmaf(s1, (da[3] + db[3]) - fmaf(z1, cb.y, cb.x), acc[3]);
}

// Two groups at once (gi0 and gi1 of the same rows): their 16 MMAs form four
// independent accumulation chains instead of two, so the tensor pipe sees
// twice the work in flight per warp.  Same arithmetic as compute_group.
__device__ __forceinline__ void compute_group2(float (&acc)[4], uint4 wa0, uint4 wb0, uint4 wa1, uint4 wb1,
                                               const float (&sz0)[4], const float (&sz1)[4], int t, uint32_t bg0,
                                               uint32_t bg1, uint32_t bact, uint32_t c00, uint32_t c10, uint32_t c01,
                                               uint32_t c11) {
    uint4 b0[4], b1[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t sw = (uint32_t)stage_word(4 * t + i) << 4;
        b0[i] = lds128_if(bg0 + sw, bact);
        b1[i] = lds128_if(bg1 + sw, bact);
    }
    const uint32_t A0[4] = {wa0.x, wa0.y, wa0.z, wa0.w}, B0[4] = {wb0.x, wb0.y, wb0.z, wb0.w};
    const uint32_t A1[4] = {wa1.x, wa1.y, wa1.z, wa1.w}, B1[4] = {wb1.x, wb1.y, wb1.z, wb1.w};
    float da0[4] = {0.f, 0.f, 0.f, 0.f}, db0[4] = {0.f, 0.f, 0.f, 0.f};
    float da1[4] = {0.f, 0.f, 0.f, 0.f}, db1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        {
            const uint32_t x = A0[i], y = B0[i];
            mma16816(da0, lop_mask_or(x, 0x000F000Fu, 0x64006400u), lop_mask_or(y, 0x000F000Fu, 0x64006400u),
                     lop_mask_or(x, 0x00F000F0u, 0x54005400u), lop_mask_or(y, 0x00F000F0u, 0x54005400u), b0[i].x,
                     b0[i].y);
        }
        {
            const uint32_t x = A1[i], y = B1[i];
            mma16816(da1, lop_mask_or(x, 0x000F000Fu, 0x64006400u), lop_mask_or(y, 0x000F000Fu, 0x64006400u),
                     lop_mask_or(x, 0x00F000F0u, 0x54005400u), lop_mask_or(y, 0x00F000F0u, 0x54005400u), b1[i].x,
                     b1[i].y);
        }
        {
            const uint32_t xs = A0[i] >> 8, ys = B0[i] >> 8;
            mma16816(db0, lop_mask_or(xs, 0x000F000Fu, 0x64006400u), lop_mask_or(ys, 0x000F000Fu, 0x64006400u),
                     lop_mask_or(xs, 0x00F000F0u, 0x54005400u), lop_mask_or(ys, 0x00F000F0u, 0x54005400u), b0[i].z,
                     b0[i].w);
        }
        {
            const uint32_t xs = A1[i] >> 8, ys = B1[i] >> 8;
            mma16816(db1, lop_mask_or(xs, 0x000F000Fu, 0x64006400u), lop_mask_or(ys, 0x000F000Fu, 0x64006400u),
                     lop_mask_or(xs, 0x00F000F0u, 0x54005400u), lop_mask_or(ys, 0x00F000F0u, 0x54005400u), b1[i].z,
                     b1[i].w);
        }
    }
    const float2 ca0 = lds_f2(c00), cb0 = lds_f2(c10), ca1 = lds_f2(c01), cb1 = lds_f2(c11);
    acc[0] = fmaf(sz0[0], (da0[0] + db0[0]) - fmaf(sz0[1], ca0.y, ca0.x), acc[0]);
    acc[1] = fmaf(sz0[0], (da0[1] + db0[1]) - fmaf(sz0[1], cb0.y, cb0.x), acc[1]);
    acc[2] = fmaf(sz0[2], (da0[2] + db0[2]) - fmaf(sz0[3], ca0.y, ca0.x), acc[2]);
    acc[3] = fmaf(sz0[2], (da0[3] + db0[3]) - fmaf(sz0[3], cb0.y, cb0.x), acc[3]);
    acc[0] = fmaf(sz1[0], (da1[0] + db1[0]) - fmaf(sz1[1], ca1.y, ca1.x), acc[0]);
    acc[1] = fmaf(sz1[0], (da1[1] + db1[1]) - fmaf(sz1[1], cb1.y, cb1.x), acc[1]);
    acc[2] = fmaf(sz1[2], (da1[2] + db1[2]) - fmaf(sz1[3], ca1.y, ca1.x), acc[2]);
    acc[3] = fmaf(sz1[2], (da1[3] + db1[3]) - fmaf(sz1[3], cb1.y, cb1.x), acc[3]);
}

__device__ __forceinline__ float half_lo(uint32_t v) { return __half2float(__ushort_as_half((uint16_t)(v & 0xFFFFu))); }
__device__ __forceinline__ float half_hi(uint32_t v) { return __half2float(__ushort_as_half((uint16_t)(v >> 16))); }

}  // namespace dec
}  // namespace moe
