// Stage 4: router-weighted combine back to token order.
//
// out[t][n] = sum_{j<k} w[t][j] * y_perm[inv[t*k+j]][n], fp32 accumulation in
// slot order j = 0..k-1, one rounding to bf16 at the end.  y_perm is bf16 at
// the C ABI and fp16 inside the layer (the tensor-core regime's output).  Each thread owns
// 8 consecutive features of one token (16-byte loads and stores); the grid is
// a multiple of the SM count and strides over (token, 8-feature chunk).
#include "internal.h"

namespace moe {
namespace {

template <bool Y_F16>
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ y_perm,
                                                      const int32_t* __restrict__ inv,
                                                      const float* __restrict__ w, int T, int k, int d,
                                                      uint16_t* __restrict__ out) {
    const int chunks = d / 8;
    const long long total = (long long)T * chunks;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(idx / chunks);
        const int c = (int)(idx % chunks);
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        // slots in batches of 8: every row load of a batch is in flight
        // before the first is used; the sum still runs in slot order
        for (int j0 = 0; j0 < k; j0 += 8) {
            uint4 v[8];
            float wj[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int j = j0 + jj;
                const int pos = j < k ? inv[(size_t)t * k + j] : -1;
                const bool ok = (unsigned)pos < (unsigned)(T * k);  // else not a permutation entry
                wj[jj] = ok ? w[(size_t)t * k + j] : 0.f;
                v[jj] = ok ? *reinterpret_cast<const uint4*>(y_perm + (size_t)pos * d + c * 8) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                if (j0 + jj >= k) break;
                const uint32_t u[4] = {v[jj].x, v[jj].y, v[jj].z, v[jj].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float lo, hi;
                    if (Y_F16) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
                        lo = f.x;
                        hi = f.y;
                    } else {
                        lo = __uint_as_float(u[i] << 16);
                        hi = __uint_as_float(u[i] & 0xFFFF0000u);
                    }
                    acc[2 * i] = fmaf(wj[jj], lo, acc[2 * i]);
                    acc[2 * i + 1] = fmaf(wj[jj], hi, acc[2 * i + 1]);
                }
            }
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        *reinterpret_cast<uint4*>(out + (size_t)t * d + c * 8) = o;
    }
}

}  // namespace

cudaError_t launch_combine(const uint16_t* y_perm, bool y_f16, const int32_t* inv, const float* w, int T, int k,
                           int d, uint16_t* out, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const long long work = (long long)T * (d / 8);
    const int per_wave = num_sms() * 8;  // 8 CTAs of 256 threads per SM
    const int blocks = (int)std::min<long long>(per_wave, (work + 255) / 256);
    if (y_f16)
        combine_kernel<true><<<blocks, 256, 0, s>>>(y_perm, inv, w, T, k, d, out);
    else
        combine_kernel<false><<<blocks, 256, 0, s>>>(y_perm, inv, w, T, k, d, out);
    note_launch();
    return cudaGetLastError();
}

}  // namespace moe
