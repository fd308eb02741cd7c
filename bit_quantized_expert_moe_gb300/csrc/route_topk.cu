// Stage 1: top-k expert selection and softmax over the selected logits.
//
// One warp per token.  Lane l holds the logits of experts l, l+32, l+64, ...
// Each of the k rounds picks the largest remaining logit with a warp
// arg-max whose tie rule is "lower expert id wins"; the comparisons are exact
// on the fp32 values, so the ids are exactly those of a sort by
// (-logit, id) (router ids must match exactly: "Performance and
// verification", section "How it is verified").  For k <= 64 the selected
// values stay in registers (route_topk_regs_kernel); larger k keeps them in
// the output arrays between rounds.
#include <cfloat>
#include <climits>

#include "decode_ops.cuh"
#include "internal.h"

namespace moe {
namespace {

// k <= 64: the selection in registers (order-preserving uint32 keys, k rounds
// of warp max and lowest id among the lanes holding it; lane j keeps slot j
// and j + 32) with one store of the ids and weights at the end.
template <int VPL>
__global__ void __launch_bounds__(256) route_topk_regs_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                              int32_t* __restrict__ ids, float* __restrict__ w) {
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    dec::route_token_regs<VPL>(logits + (size_t)t * E, E, k, ids + (size_t)t * k, w + (size_t)t * k);
}

__device__ __forceinline__ bool better(float v, int e, float bv, int be) {
    return (v > bv) || (v == bv && e < be);
}

template <int VPL>  // logits per lane: E <= 32 * VPL
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E,
                                                         int k, int32_t* __restrict__ ids,
                                                         float* __restrict__ w) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float* row = logits + (size_t)t * E;

    float v[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        v[i] = (e < E) ? row[e] : -FLT_MAX;
    }
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
        if (lane + 32 * i >= E) taken |= 1u << i;

    int32_t* out_ids = ids + (size_t)t * k;
    float* out_w = w + (size_t)t * k;
    float vmax = 0.f;
    for (int j = 0; j < k; ++j) {
        // lane-local best among the untaken
        float bv = -FLT_MAX;
        int be = INT_MAX, bi = -1;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int e = lane + 32 * i;
            if (!(taken >> i & 1u) && better(v[i], e, bv, be)) { bv = v[i]; be = e; bi = i; }
        }
        // warp arg-max (butterfly: every lane ends with the winner)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oe = __shfl_xor_sync(0xffffffffu, be, off);
            if (better(ov, oe, bv, be)) { bv = ov; be = oe; }
        }
        if (bi >= 0 && be == lane + 32 * bi) taken |= 1u << bi;
        if (j == 0) vmax = bv;
        if (lane == 0) {
            out_ids[j] = be;
            out_w[j] = bv;  // selected logit, turned into a weight below
        }
    }
    __syncwarp();
    // softmax over the k selected logits, fp32
    float sum = 0.f;
    for (int j = lane; j < k; j += 32) {
        const float ex = expf(out_w[j] - vmax);
        out_w[j] = ex;
        sum += ex;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    __syncwarp();
    const float inv_sum = 1.0f / sum;
    for (int j = lane; j < k; j += 32) out_w[j] = out_w[j] * inv_sum;
}

template <int VPL>
cudaError_t launch_vpl(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t s) {
    const int warps = 8;
    if (k <= 64)
        route_topk_regs_kernel<VPL><<<ceil_div(T, warps), warps * 32, 0, s>>>(logits, T, E, k, ids, w);
    else
        route_topk_kernel<VPL><<<ceil_div(T, warps), warps * 32, 0, s>>>(logits, T, E, k, ids, w);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                              cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (E <= 32) return launch_vpl<1>(logits, T, E, k, ids, w, s);
    if (E <= 64) return launch_vpl<2>(logits, T, E, k, ids, w, s);
    if (E <= 128) return launch_vpl<4>(logits, T, E, k, ids, w, s);
    if (E <= 256) return launch_vpl<8>(logits, T, E, k, ids, w, s);
    if (E <= 512) return launch_vpl<16>(logits, T, E, k, ids, w, s);
    return launch_vpl<32>(logits, T, E, k, ids, w, s);
}

}  // namespace moe
