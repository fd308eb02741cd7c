// Shared device helpers of the moe_w4 library (sm_103a only).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_w4.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "moe_w4 kernels are written for Blackwell (sm_103a)"
#endif

namespace moe {

// ---------------------------------------------------------------------------
// Workspace header: the first 256 bytes of every workspace.
// ---------------------------------------------------------------------------
constexpr uint32_t ERRBIT_RANGE = 1u;    // an expert id outside [0, E)
constexpr uint32_t ERRBIT_TIMEOUT = 2u;  // a bounded pipeline wait gave up
constexpr uint32_t ERRBIT_F16_RANGE = 4u;  // a value outside the fp16 range of the tensor-core regime
constexpr size_t WS_HEADER = 256;

struct WsHeader {
    uint32_t err;        // OR of ERRBIT_*; cleared by moe_get_device_error
    uint32_t reserved[63];
};
// Header word of the one-kernel decode layer (32-bit word index): the
// grid-barrier kernel's 64-bit arrival counter, in its own 64-byte sector.
constexpr int WS_BAR_COUNT_WORD = 16;

// Small device-side plan written by the permutation kernels (after the header).
struct DevPlan {
    int32_t n_uniq;      // experts with at least one row
    int32_t n_tiles;     // token tiles of the grouped GEMM
    int32_t pad[62];
};

__device__ __forceinline__ void set_error(uint32_t* err, uint32_t bit) {
    atomicOr(err, bit);
}

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ constexpr size_t align_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

// ---------------------------------------------------------------------------
// Bit tricks for int4 -> float (magic-number conversion).
//
// A float whose exponent field is that of 1.0 and whose mantissa holds a 4-bit
// code q at bit position p (p in 12..19) has the value 1 + q * 2^(p-23) exactly.
// Nibble i of a packed word sits at bit 4i; bits 12 and 16 are inside the
// window, the others are brought there by one shift or rotate per two nibbles:
//   w        : nibble 3 -> bit 12, nibble 4 -> bit 16
//   w << 8   : nibble 1 -> bit 12, nibble 2 -> bit 16
//   w >> 8   : nibble 5 -> bit 12, nibble 6 -> bit 16
//   rot16(w) : nibble 7 -> bit 12, nibble 0 -> bit 16
// So every odd code k is read as 1 + q_k * 2^-11 and every even code as
// 1 + q_k * 2^-7.  Callers undo the offsets and the 2^-11 / 2^-7 factors.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t lop_mask_or(uint32_t a, uint32_t mask, uint32_t bits) {
    uint32_t r;
    // (a & mask) | bits  (LUT 0xEA: (A & B) | C)
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(mask), "r"(bits));
    return r;
}

struct Nib8 {  // eight codes of one word as floats: .odd[i], .even[i] (see pair order)
    float2 p[4];  // p[m] = (odd code value, even code value) for pairs (3,4),(1,2),(5,6),(7,0)
};

__device__ __forceinline__ void nib8_magic(uint32_t w, float2 (&p)[4]) {
    constexpr uint32_t ONE = 0x3F800000u;
    uint32_t wl = w << 8, wr = w >> 8;
    uint32_t wt = __funnelshift_l(w, w, 16);
    p[0] = make_float2(__uint_as_float(lop_mask_or(w, 0x0000F000u, ONE)),
                       __uint_as_float(lop_mask_or(w, 0x000F0000u, ONE)));   // codes 3, 4
    p[1] = make_float2(__uint_as_float(lop_mask_or(wl, 0x0000F000u, ONE)),
                       __uint_as_float(lop_mask_or(wl, 0x000F0000u, ONE)));  // codes 1, 2
    p[2] = make_float2(__uint_as_float(lop_mask_or(wr, 0x0000F000u, ONE)),
                       __uint_as_float(lop_mask_or(wr, 0x000F0000u, ONE)));  // codes 5, 6
    p[3] = make_float2(__uint_as_float(lop_mask_or(wt, 0x0000F000u, ONE)),
                       __uint_as_float(lop_mask_or(wt, 0x000F0000u, ONE)));  // codes 7, 0
}

// fp16 operands of the int4 GEMMs keep K in groups of 8 interleaved as
// (0, 4, 1, 5, 2, 6, 3, 7): the order in which masking one packed word of 8
// codes yields them (nibbles 0 and 4, 1 and 5 of a word, then of the word
// shifted by 8).  A dot product is unchanged when both operands share the
// permutation.  Eight fp16 values in natural order as four f16x2 registers
// (v0,v1), (v2,v3), (v4,v5), (v6,v7) -> (v0,v4), (v1,v5), (v2,v6), (v3,v7).
__device__ __forceinline__ uint4 k8_interleave(uint32_t p01, uint32_t p23, uint32_t p45, uint32_t p67) {
    uint4 o;
    o.x = __byte_perm(p01, p45, 0x5410);
    o.y = __byte_perm(p01, p45, 0x7632);
    o.z = __byte_perm(p23, p67, 0x5410);
    o.w = __byte_perm(p23, p67, 0x7632);
    return o;
}
// Position of element k (0..7) of a group of 8 in that order.
__device__ __forceinline__ int k8_pos(int k) { return k < 4 ? 2 * k : 2 * k - 7; }

// f16x2 arithmetic on raw 32-bit registers (round to nearest even).
__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// Packed fp32x2 fused multiply-add (Blackwell FFMA2): d = a * b + c lane-wise.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    unsigned long long ra, rb, rc, rd;
    ra = *reinterpret_cast<unsigned long long*>(&a);
    rb = *reinterpret_cast<unsigned long long*>(&b);
    rc = *reinterpret_cast<unsigned long long*>(&c);
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
    return *reinterpret_cast<float2*>(&rd);
}

__device__ __forceinline__ float half_bits_to_float(uint16_t b) {
    return __half2float(__ushort_as_half(b));
}

// Two fp32 -> packed bf16x2 (round to nearest even): low half = lo, high half = hi.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two fp32 -> packed f16x2 (round to nearest even): low half = lo, high half = hi.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// True if either half of a packed f16x2 word is infinite or NaN.
__device__ __forceinline__ bool f16x2_nonfinite(uint32_t p) {
    return ((p & 0x7C00u) == 0x7C00u) || ((p & 0x7C000000u) == 0x7C000000u);
}

__device__ __forceinline__ uint16_t float_to_f16_bits(float v) {
    return __half_as_ushort(__float2half_rn(v));
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// SiLU(g) = g / (1 + e^-g) with the fast exponential and division (a few ulp;
// g -> -inf gives -0 since the quotient by an infinite denominator is 0).
__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte streaming load that bypasses L1 allocation (read-once weights).
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// cp.async (Ampere-style LDGSTS) helpers.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

}  // namespace moe
