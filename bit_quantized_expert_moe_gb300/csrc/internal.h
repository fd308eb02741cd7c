// Internal declarations shared by the library's translation units.
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace moe {

// ---------------------------------------------------------------- routing
cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                              cudaStream_t s);

// ------------------------------------------------------------ permutation
// Token tiles of the grouped tensor-core GEMM: one entry per (expert, <=256 rows).
constexpr int TILE_ROWS = 256;
struct Tile {
    int32_t expert;
    int32_t row0;    // first permuted row
    int32_t nrows;   // 1..TILE_ROWS
    int32_t pad;
};

struct AlignOut {
    int32_t* counts;    // [E]
    int32_t* offsets;   // [E+1]
    int32_t* sorted;    // [R]
    int32_t* inv;       // [R]
    int32_t* uniq;      // [E]  experts with rows, ascending
    Tile* tiles;        // [R/TILE_ROWS + E]
    DevPlan* plan;      // n_uniq, n_tiles
    uint16_t* x_perm;   // [R][d] or null
    int x_perm_f16;     // 1: write x_perm as fp16 in the tensor-core operand order (K interleaved
                        //    in groups of 8, k8_interleave); values outside fp16 set the error word
    int32_t* blockcnt;  // [nblocks][E] scratch for the multi-block path
    uint32_t* err;
};
constexpr int ALIGN_SMALL_MAX_R = 2048;   // single-CTA permutation up to this many rows
constexpr int ALIGN_BLOCK_ROWS = 1024;    // most assignments per CTA on the multi-block path
// Assignments per CTA on the multi-block path: the smallest of 32, 64 and 256
// (more CTAs for the stable placement and the row copy) whose per-block count
// table stays within 64 KB, else 1024.
int align_block_rows(int R, int E);
size_t align_blockcnt_bytes(int R, int E);
cudaError_t launch_align(const int32_t* ids, int T, int k, int E, const uint16_t* x, int d,
                         const AlignOut& o, cudaStream_t s);
// uniq list + tile list from an offsets array already on the device.
// bf16 -> fp16 copy of n elements (n % 8 == 0); out-of-range values set the error word.
// bf16 rows -> fp16 in the tensor-core operand order (K interleaved in groups of 8)
cudaError_t launch_bf16_to_f16(const uint16_t* in, uint16_t* out, size_t n, uint32_t* err, cudaStream_t s);
cudaError_t launch_plan_from_offsets(const int32_t* offsets, int E, int32_t* uniq, Tile* tiles,
                                     DevPlan* plan, cudaStream_t s);

// ---------------------------------------------------------------- combine
// y_perm is bf16 (y_f16 = false) or fp16 (y_f16 = true).
cudaError_t launch_combine(const uint16_t* y_perm, bool y_f16, const int32_t* inv, const float* w, int T, int k,
                           int d, uint16_t* out, cudaStream_t s);

// ------------------------------------------------- decode regime (GEMV)
struct GemvShape {
    int E, d, f;
    int R;          // rows (assignments) in the permuted order
    int max_uniq;   // upper bound on experts with rows: min(R, E)
};
struct GemvIn {
    const uint32_t *w13_q, *w2_q;
    const uint16_t *w13_s, *w13_z, *w2_s, *w2_z;
    const int32_t* offsets;
    const int32_t* uniq;
    const DevPlan* plan;
    const int32_t* sorted;   // gate_up input row i = x[sorted[i] / k] when non-null, else x[i]
    int k;
    const uint16_t* x;       // bf16 [*][d]
    float* h;                // fp32 [R][f] (written by gate_up, read by down)
    // down outputs: exactly one of (y_perm) or (out with topk_w, inv, T)
    uint16_t* y_perm;        // bf16 [R][d]
    const float* row_w;      // optional row scale for y_perm
    uint16_t* out;           // bf16 [T][d]: fused combine
    const float* topk_w;
    const int32_t* inv;
    int T;
    uint32_t* err;
};
bool gemv_supported(const GemvShape& sh, int T_tokens);
cudaError_t launch_gemv_gateup(const GemvShape& sh, const GemvIn& in, cudaStream_t s);
cudaError_t launch_gemv_down(const GemvShape& sh, const GemvIn& in, cudaStream_t s);

// ------------------------- decode regime: the whole layer in one kernel
// Routing, gate_up, down and combine of T <= 8 tokens in one cooperative
// persistent launch (decode_fused.cu).
struct FusedIn {
    const moe_w4_layer* L;
    const uint16_t* x;       // bf16 [T][d]
    const float* logits;     // fp32 [T][E]
    int T, k;
    uint16_t* out;           // bf16 [T][d]
    int32_t* ids_out;        // [T][k] or null
    uint16_t* hb;            // fp16 scratch, [T*k][f]
    void* ws;                // workspace (header: error word and the kernels' counters)
};
bool decode_fused_supported(int T, int k, int E, int d, int f);
cudaError_t launch_decode_fused(const FusedIn& in, cudaStream_t s);

// ---------------------------------------------- prefill regime (tcgen05)
struct TcIn {
    const uint32_t *w13_q, *w2_q;
    const uint16_t *w13_s, *w13_z, *w2_s, *w2_z;
    const Tile* tiles;
    const DevPlan* plan;
    const uint16_t* x16;     // fp16 [R][d]: permuted activations
    uint16_t* h16;           // fp16 [R][f]
    uint16_t* y_out;         // [R][d], fp16 if y_f16 else bf16
    int y_f16;
    const float* row_w;      // optional
    uint32_t* err;
};
bool tc_supported(int E, int d, int f);
int tc_max_tiles(int R, int E);
cudaError_t launch_tc_gateup(int E, int d, int f, int R, const TcIn& in, cudaStream_t s);
cudaError_t launch_tc_down(int E, int d, int f, int R, const TcIn& in, cudaStream_t s);

// 3D tensor map over 32-bit words: dims {d0, d1, d2} (d0 contiguous), byte
// strides s1 (dim 1) and s2 (dim 2), box {b0, b1, b2}, 128-byte swizzle.
bool make_tensor_map_3d(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                        uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2);
// Tensor map of rank 1..5 over 32-bit words: dims[0] contiguous, strides[i]
// the byte stride of dimension i + 1, box per dimension, 128-byte swizzle.
bool make_tensor_map_u32(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims, const uint64_t* strides,
                         const uint32_t* box);
// The same over 16-bit elements, without swizzle.
bool make_tensor_map_u16(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims, const uint64_t* strides,
                         const uint32_t* box);

// ----------------------------------------------------------- device info
int num_sms();
// Counts one kernel launch of this library (reported by moe_kernel_launches).
void note_launch(int n = 1);

}  // namespace moe
