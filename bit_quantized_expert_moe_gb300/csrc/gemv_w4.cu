// Stage 3, decode regime: W4A16 split-K GEMV on the CUDA cores.
//
// With a handful of rows per expert the layer is bound by the bytes of the
// experts' weights, which are read exactly once ("Performance and
// verification", section "Why it is fast": one fetch of an expert per batch;
// the packed 4-bit codes enter the arithmetic without being expanded first).
//
// Layout of the work:
//   * a thread owns one 32-element chunk c of the reduction axis (16 bytes of
//     packed codes per weight row) and one expert slot us; the CTA's threads
//     cover C = K/32 chunks x U expert slots;
//   * the CTA owns a contiguous range of output features and walks it; for
//     each feature every thread streams its 16-byte chunk of the weight row(s)
//     through a private cp.async ring (STAGES-1 rows in flight per thread);
//   * the thread's 32 activations of each token row stay in registers,
//     pre-scaled for the magic-number decode (see nib8_magic): the packed FMA
//     fma.rn.f32x2 accumulates an odd-code and an even-code product at once;
//   * the zero point and the fp16 scale are applied once per chunk:
//     sum (q - z) s x = s (sum q x - z sum x);
//   * partial sums of the C chunk-threads of a row are reduced through shared
//     memory in batches of FB features (8 lanes per output, shuffles).
// gate_up writes h = SiLU(g) * u in fp32; down either writes y_perm rows or,
// because one CTA sees every expert of its feature range, applies the router
// weights and writes the combined token rows directly (fixed slot order, no
// atomics).
#include <algorithm>

#include "internal.h"

namespace moe {
namespace {

constexpr int NT = 2;        // token rows of one expert handled per pass
constexpr int FB = 4;        // features per reduction batch
constexpr int STAGES = 4;    // cp.async ring depth per thread
constexpr int MAX_THREADS = 512;
constexpr int MAX_ROWS = 64; // rows (assignments) supported by this regime

struct XSlice {
    float2 p[4][4];  // [word][pair] = (x_odd * 2^11, x_even * 2^7), pairs (3,4),(1,2),(5,6),(7,0)
    float2 init;     // (-2^11 * sum x_odd, -2^7 * sum x_even): cancels the magic offsets
    float X;         // sum of the 32 activations
};

// The 32 activations of chunk c of a row: bf16 rows (gate_up input) or fp32
// rows (the down projection's input h).
template <typename TIn>
__device__ __forceinline__ void load_xslice(const TIn* __restrict__ row, int c, bool valid, XSlice& xs) {
    float xv[32];
    if (!valid) {
#pragma unroll
        for (int i = 0; i < 32; ++i) xv[i] = 0.f;
    } else if (sizeof(TIn) == 2) {
        const uint4* src = reinterpret_cast<const uint4*>(row + 32 * c);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const uint4 q = src[w];
            const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xv[8 * w + 2 * i] = __uint_as_float(u[i] << 16);
                xv[8 * w + 2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
            }
        }
    } else {
        const float4* src = reinterpret_cast<const float4*>(row + 32 * c);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 q = src[i];
            xv[4 * i] = q.x;
            xv[4 * i + 1] = q.y;
            xv[4 * i + 2] = q.z;
            xv[4 * i + 3] = q.w;
        }
    }
    float so = 0.f, se = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float x0 = xv[8 * w], x1 = xv[8 * w + 1], x2 = xv[8 * w + 2], x3 = xv[8 * w + 3];
        const float x4 = xv[8 * w + 4], x5 = xv[8 * w + 5], x6 = xv[8 * w + 6], x7 = xv[8 * w + 7];
        xs.p[w][0] = make_float2(x3 * 2048.f, x4 * 128.f);
        xs.p[w][1] = make_float2(x1 * 2048.f, x2 * 128.f);
        xs.p[w][2] = make_float2(x5 * 2048.f, x6 * 128.f);
        xs.p[w][3] = make_float2(x7 * 2048.f, x0 * 128.f);
        so += (x1 + x3) + (x5 + x7);
        se += (x0 + x2) + (x4 + x6);
    }
    xs.init = make_float2(-2048.f * so, -128.f * se);
    xs.X = so + se;
}

// Same, for NT slices sharing the decode of the weights.
__device__ __forceinline__ void chunk_dot_nt(const uint4& wq, const XSlice (&xs)[NT], float (&out)[NT]) {
    float2 acc[NT];
#pragma unroll
    for (int s = 0; s < NT; ++s) acc[s] = xs[s].init;
    const uint32_t words[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        float2 v[4];
        nib8_magic(words[w], v);
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int s = 0; s < NT; ++s) acc[s] = ffma2(v[m], xs[s].p[w][m], acc[s]);
    }
#pragma unroll
    for (int s = 0; s < NT; ++s) out[s] = acc[s].x + acc[s].y;
}

__device__ __forceinline__ float pick_half(uint32_t pair, int hi) {
    return half_bits_to_float((uint16_t)(hi ? (pair >> 16) : (pair & 0xFFFFu)));
}

struct KernelCfg {
    int C;        // chunks per weight row (K / 32)
    int Cp;       // padded row stride of the reduction buffer
    int U;        // expert slots per CTA
    int nthreads;
    int nfeat_max;
    int R;
};

// Dynamic shared memory layout (all 16-byte aligned):
//   ring  [STAGES][PARTS][nthreads] uint4
//   red   [2][FB * U * NT * G2 * Cp] float
//   yrow  [nfeat_max][R] float          (down, combine mode only)
template <bool GATEUP>
struct Smem {
    static constexpr int PARTS = GATEUP ? 3 : 2;
    static constexpr int G2 = GATEUP ? 2 : 1;
    __host__ __device__ static size_t ring_bytes(const KernelCfg& k) { return (size_t)STAGES * PARTS * k.nthreads * 16; }
    __host__ __device__ static size_t red_floats(const KernelCfg& k) { return (size_t)FB * k.U * NT * G2 * k.Cp; }
    static size_t bytes(const KernelCfg& k, bool combine) {
        size_t b = ring_bytes(k) + 2 * red_floats(k) * 4;
        if (combine) b += (size_t)k.nfeat_max * k.R * 4;
        return b;
    }
};

template <bool GATEUP>
__global__ void __launch_bounds__(MAX_THREADS, 1)
gemv_w4_kernel(GemvShape sh, GemvIn in, KernelCfg kc) {
    using SM = Smem<GATEUP>;
    extern __shared__ __align__(16) unsigned char smem[];
    uint4* ring = reinterpret_cast<uint4*>(smem);
    float* red = reinterpret_cast<float*>(smem + SM::ring_bytes(kc));
    float* yrow = red + 2 * SM::red_floats(kc);

    __shared__ int s_e[MAX_ROWS], s_seg[MAX_ROWS], s_cnt[MAX_ROWS];
    __shared__ int s_maxcnt;

    const int tid = threadIdx.x;
    const int C = kc.C, U = kc.U, Cp = kc.Cp;
    const int c = tid % C;
    const int us = tid / C;                  // may be >= U for padding threads
    const int K = GATEUP ? sh.d : sh.f;      // reduction length
    const int G = K / 128;                   // groups per row
    const int n_out = GATEUP ? sh.f : sh.d;  // features per expert
    const int n_uniq = in.plan->n_uniq;
    const bool combine = !GATEUP && in.out != nullptr;

    // feature range of this CTA
    const int nranges = gridDim.x;
    const int lo = (int)((long long)blockIdx.x * n_out / nranges);
    const int hi = (int)((long long)(blockIdx.x + 1) * n_out / nranges);
    const int nfeat = hi - lo;

    const uint32_t* wq = GATEUP ? in.w13_q : in.w2_q;
    const uint16_t* wsc = GATEUP ? in.w13_s : in.w2_s;
    const uint16_t* wz = GATEUP ? in.w13_z : in.w2_z;
    const size_t rows_per_expert = GATEUP ? 2 * (size_t)sh.f : (size_t)sh.d;
    const size_t wpr = (size_t)K / 8;        // words per row
    const int g = c >> 2;                    // this thread's group
    const int ghi = g & 1;

    // expert groups: gate_up takes one from blockIdx.y, down walks all of them
    const int ug_begin = GATEUP ? blockIdx.y * U : 0;
    const int ug_end = GATEUP ? min(n_uniq, ug_begin + U) : n_uniq;
    const int ug_step = U;

    for (int ug = ug_begin; ug < ug_end; ug += ug_step) {
        // ---- slot table for this expert group
        if (tid < U) {
            const int u = ug + tid;
            if (u < n_uniq) {
                const int e = in.uniq[u];
                s_e[tid] = e;
                s_seg[tid] = in.offsets[e];
                s_cnt[tid] = in.offsets[e + 1] - in.offsets[e];
            } else {
                s_e[tid] = 0;
                s_seg[tid] = 0;
                s_cnt[tid] = 0;
            }
        }
        if (tid == 0) s_maxcnt = 0;
        __syncthreads();
        if (tid < U) atomicMax(&s_maxcnt, s_cnt[tid]);
        __syncthreads();
        const int maxcnt = s_maxcnt;
        const bool active = (us < U) && (ug + us < n_uniq);
        const int my_e = active ? s_e[us] : 0;
        const int my_seg = active ? s_seg[us] : 0;
        const int my_cnt = active ? s_cnt[us] : 0;

        for (int p0 = 0; p0 < maxcnt; p0 += NT) {
            // ---- activations of this pass's rows
            XSlice xs[NT];
#pragma unroll
            for (int s = 0; s < NT; ++s) {
                const int r = p0 + s;
                const bool v = active && r < my_cnt;
                if (GATEUP) {
                    const uint16_t* row = nullptr;
                    if (v) {
                        const int i = my_seg + r;
                        const int src = in.sorted ? in.sorted[i] / in.k : i;
                        row = in.x + (size_t)src * sh.d;
                    }
                    load_xslice(row, c, v, xs[s]);
                } else {
                    const float* row = v ? in.h + (size_t)(my_seg + r) * sh.f : nullptr;
                    load_xslice(row, c, v, xs[s]);
                }
            }
            const bool loads = active && p0 < my_cnt;
            const size_t ebase = (size_t)my_e * rows_per_expert;

            auto issue = [&](int fi, int st) {
                const int n = lo + fi;
                uint4* r0 = ring + ((size_t)st * SM::PARTS) * kc.nthreads + tid;
                const size_t row_a = ebase + n;
                cp_async16(smem_u32(r0), wq + row_a * wpr + 4 * c);
                const size_t sa = row_a * G + (g & ~1);
                if (GATEUP) {
                    const size_t row_b = ebase + sh.f + n;
                    cp_async16(smem_u32(r0 + kc.nthreads), wq + row_b * wpr + 4 * c);
                    const uint32_t d2 = smem_u32(r0 + 2 * kc.nthreads);
                    const size_t sb = row_b * G + (g & ~1);
                    cp_async4(d2 + 0, wsc + sa);
                    cp_async4(d2 + 4, wz + sa);
                    cp_async4(d2 + 8, wsc + sb);
                    cp_async4(d2 + 12, wz + sb);
                } else {
                    const uint32_t d2 = smem_u32(r0 + kc.nthreads);
                    cp_async4(d2 + 0, wsc + sa);
                    cp_async4(d2 + 4, wz + sa);
                }
            };

#pragma unroll 1
            for (int st = 0; st < STAGES - 1; ++st) {
                if (loads && st < nfeat) issue(st, st);
                cp_async_commit();
            }
            int buf = 0;
            int batch0 = 0;  // first feature of the current reduction batch
#pragma unroll 1
            for (int fi = 0; fi < nfeat; ++fi) {
                {
                    const int nf = fi + STAGES - 1;
                    if (loads && nf < nfeat) issue(nf, nf % STAGES);
                    cp_async_commit();
                }
                cp_async_wait<STAGES - 1>();
                const int st = fi % STAGES;
                const uint4* r0 = ring + ((size_t)st * SM::PARTS) * kc.nthreads + tid;
                float* rb = red + (size_t)buf * SM::red_floats(kc);
                const int fb = fi - batch0;
                if (loads) {
                    if (GATEUP) {
                        const uint4 wg = r0[0], wu = r0[kc.nthreads], sz = r0[2 * kc.nthreads];
                        float dg[NT], du[NT];
                        chunk_dot_nt(wg, xs, dg);
                        chunk_dot_nt(wu, xs, du);
                        const float sg = pick_half(sz.x, ghi), zg = pick_half(sz.y, ghi);
                        const float su = pick_half(sz.z, ghi), zu = pick_half(sz.w, ghi);
#pragma unroll
                        for (int s = 0; s < NT; ++s) {
                            const int o = ((fb * U + us) * NT + s) * 2;
                            rb[(size_t)o * Cp + c] = sg * fmaf(-zg, xs[s].X, dg[s]);
                            rb[(size_t)(o + 1) * Cp + c] = su * fmaf(-zu, xs[s].X, du[s]);
                        }
                    } else {
                        const uint4 wd = r0[0], sz = r0[kc.nthreads];
                        float dd[NT];
                        chunk_dot_nt(wd, xs, dd);
                        const float sd = pick_half(sz.x, ghi), zd = pick_half(sz.y, ghi);
#pragma unroll
                        for (int s = 0; s < NT; ++s) {
                            const int o = (fb * U + us) * NT + s;
                            rb[(size_t)o * Cp + c] = sd * fmaf(-zd, xs[s].X, dd[s]);
                        }
                    }
                }
                // ---- reduce a full batch (or the tail)
                if (fb == FB - 1 || fi == nfeat - 1) {
                    __syncthreads();
                    const int nb = fb + 1;
                    const int O = nb * U * NT * SM::G2;
                    const int warp = tid >> 5, lane = tid & 31;
                    const int l8 = lane & 7, gq = lane >> 3;
                    const int nwarps = kc.nthreads >> 5;
                    for (int base = warp * 4; base < O; base += nwarps * 4) {
                        const int o = base + gq;
                        float sum = 0.f;
                        if (o < O)
                            for (int cc = l8; cc < C; cc += 8) sum += rb[(size_t)o * Cp + cc];
                        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
                        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                        if (GATEUP) {
                            const float other = __shfl_xor_sync(0xffffffffu, sum, 8);
                            if (o < O && (o & 1) == 0 && l8 == 0) {
                                const int rest = o >> 1;
                                const int s = rest % NT;
                                const int slot = (rest / NT) % U;
                                const int f_i = rest / (NT * U);
                                const int r = p0 + s;
                                if (ug + slot < n_uniq && r < s_cnt[slot]) {
                                    const int i = s_seg[slot] + r;
                                    in.h[(size_t)i * sh.f + lo + batch0 + f_i] = silu(sum) * other;
                                }
                            }
                        } else {
                            if (o < O && l8 == 0) {
                                const int s = o % NT;
                                const int slot = (o / NT) % U;
                                const int f_i = o / (NT * U);
                                const int r = p0 + s;
                                if (ug + slot < n_uniq && r < s_cnt[slot]) {
                                    const int i = s_seg[slot] + r;
                                    const int nl = batch0 + f_i;
                                    if (combine) {
                                        yrow[(size_t)nl * kc.R + i] = sum;
                                    } else {
                                        const float sc = in.row_w ? in.row_w[i] : 1.0f;
                                        in.y_perm[(size_t)i * sh.d + lo + nl] = float_to_bf16_bits(sum * sc);
                                    }
                                }
                            }
                        }
                    }
                    buf ^= 1;
                    batch0 = fi + 1;
                }
            }
            cp_async_wait<0>();
            __syncthreads();
        }
    }

    if (combine) {
        __syncthreads();
        const int T = in.T, k = in.k;
        for (int idx = tid; idx < nfeat * T; idx += blockDim.x) {
            const int nl = idx % nfeat;
            const int t = idx / nfeat;
            float acc = 0.f;
            for (int j = 0; j < k; ++j) {
                const int a = t * k + j;
                acc = fmaf(in.topk_w[a], yrow[(size_t)nl * kc.R + in.inv[a]], acc);
            }
            in.out[(size_t)t * sh.d + lo + nl] = float_to_bf16_bits(acc);
        }
    }
}

KernelCfg make_cfg(int K, int max_uniq, int R, int nfeat_max) {
    KernelCfg kc{};
    kc.C = K / 32;
    kc.U = std::max(1, std::min(max_uniq, MAX_THREADS / kc.C));
    kc.nthreads = (kc.C * kc.U + 31) / 32 * 32;
    kc.Cp = kc.C + ((8 - kc.C) % 32 + 32) % 32;
    kc.nfeat_max = nfeat_max;
    kc.R = R;
    return kc;
}

template <bool GATEUP>
cudaError_t launch(const GemvShape& sh, const GemvIn& in, const KernelCfg& kc, dim3 grid, bool combine,
                   cudaStream_t s) {
    const size_t smem = Smem<GATEUP>::bytes(kc, combine);
    static size_t configured = 0;
    if (smem > configured) {
        cudaError_t e = cudaFuncSetAttribute(gemv_w4_kernel<GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)std::max<size_t>(smem, 48 * 1024));
        if (e != cudaSuccess) return e;
        configured = smem;
    }
    gemv_w4_kernel<GATEUP><<<grid, kc.nthreads, smem, s>>>(sh, in, kc);
    note_launch();
    return cudaGetLastError();
}

constexpr size_t SMEM_LIMIT = 220 * 1024;

}  // namespace

bool gemv_supported(const GemvShape& sh, int T) {
    if (sh.R > MAX_ROWS || sh.R <= 0) return false;
    if (sh.d % 256 || sh.f % 256) return false;
    if (sh.d / 32 > MAX_THREADS || sh.f / 32 > MAX_THREADS) return false;
    const int nsm = num_sms();
    KernelCfg a = make_cfg(sh.d, sh.max_uniq, sh.R, 0);
    KernelCfg b = make_cfg(sh.f, sh.max_uniq, sh.R, ceil_div(sh.d, std::min(sh.d, nsm)));
    if (Smem<true>::bytes(a, false) > SMEM_LIMIT) return false;
    if (Smem<false>::bytes(b, true) > SMEM_LIMIT) return false;
    (void)T;
    return true;
}

cudaError_t launch_gemv_gateup(const GemvShape& sh, const GemvIn& in, cudaStream_t s) {
    const int nsm = num_sms();
    KernelCfg kc = make_cfg(sh.d, sh.max_uniq, sh.R, 0);
    const int GU = ceil_div(sh.max_uniq, kc.U);
    const int FR = std::max(1, std::min(sh.f, ceil_div(nsm, GU)));
    return launch<true>(sh, in, kc, dim3(FR, GU), false, s);
}

cudaError_t launch_gemv_down(const GemvShape& sh, const GemvIn& in, cudaStream_t s) {
    const int nsm = num_sms();
    const int ranges = std::min(sh.d, nsm);
    KernelCfg kc = make_cfg(sh.f, sh.max_uniq, sh.R, ceil_div(sh.d, ranges));
    return launch<false>(sh, in, kc, dim3(ranges), in.out != nullptr, s);
}

}  // namespace moe
