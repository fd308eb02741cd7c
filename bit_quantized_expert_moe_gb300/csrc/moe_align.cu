// Stage 2: token -> expert permutation (stable counting sort) and gather.
//
// The assignments a = t*k + j are grouped by expert so that the weights of an
// expert are fetched a single time per batch ("Performance and verification",
// section "Why it is fast").  Inside an expert's segment the assignments keep
// ascending a (a stable sort), so the permutation is unique and is compared
// bit-exactly.
//
// Small batches (R <= ALIGN_SMALL_MAX_R) use one CTA for everything.  Larger
// batches use two kernels: per-block histograms, then one CTA per block that
// sums the earlier blocks' counts and every block's counts straight from the
// count table, scans the totals into expert offsets, places its block's
// assignments in order (one warp, stable) and copies their activation rows
// (all warps; a separate row gather when there are too few blocks to fill
// the GPU).  Besides counts/offsets/sorted/inv, block 0 also emits the list
// of experts with rows (for the GEMV regime) and the token tiles (for the
// tensor-core regime).  An id outside [0, E) sets the range error bit and is
// skipped.
#include "internal.h"

namespace moe {
namespace {

constexpr int SCAN_THREADS = 1024;

// Exclusive block scan of one int per thread (blockDim.x == SCAN_THREADS).
// Returns the exclusive prefix; `total` receives the block total.
__device__ int block_exclusive_scan(int v, int& total) {
    __shared__ int warp_sums[32];
    __shared__ int s_total;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += n;
    }
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        const int ws = warp_sums[lane];
        int wincl = ws;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, wincl, off);
            if (lane >= off) wincl += n;
        }
        warp_sums[lane] = wincl - ws;  // exclusive prefix of the warp sums
        if (lane == 31) s_total = wincl;
    }
    __syncthreads();
    const int res = warp_sums[wid] + incl - v;
    total = s_total;
    __syncthreads();  // warp_sums / s_total are reused by the next call
    return res;
}

// Per-expert totals -> offsets, counts, uniq list and tiles (one CTA of
// SCAN_THREADS threads; thread e owns expert e).
__device__ void emit_plan(int cnt, int e, int E, int32_t* counts, int32_t* offsets, int32_t* uniq,
                          Tile* tiles, DevPlan* plan, int* s_offset_out) {
    int total;
    const bool live = e < E;
    const int c = live ? cnt : 0;
    const int off = block_exclusive_scan(c, total);
    if (live) {
        if (counts) counts[e] = c;
        if (offsets) offsets[e] = off;
    }
    if (threadIdx.x == 0 && offsets) offsets[E] = total;
    if (s_offset_out) *s_offset_out = off;
    // experts with rows, ascending id
    const int has = (live && c > 0) ? 1 : 0;
    int n_uniq;
    const int upos = block_exclusive_scan(has, n_uniq);
    if (has && uniq) uniq[upos] = e;
    // Token tiles of at most TILE_ROWS rows: first every expert's full tiles
    // in expert order, then each expert's last partial tile, largest first
    // (classes of 16 rows, the MMA's N step; expert order inside a class).
    // The grouped GEMM hands tiles to its CTA pairs round-robin, and a tile's
    // cost grows with its rows: this order ends the list with the cheapest
    // tiles and spreads the expensive ones evenly over the pairs.
    if (!tiles && !plan) return;  // the same for every thread of the block
    const int nfull = live ? c / TILE_ROWS : 0;
    const int rem = live ? c - nfull * TILE_ROWS : 0;
    int n_full;
    const int fpos = block_exclusive_scan(nfull, n_full);
    constexpr int NCLS = TILE_ROWS / 16;
    __shared__ int cls_cnt[SCAN_THREADS / 32][NCLS + 1];  // per warp, per class: count, then prefix
    __shared__ int cls_base[NCLS + 1];
    __shared__ int s_n_tiles;
    const int cls = rem > 0 ? ceil_div(rem, 16) : 0;      // 1..NCLS, 0: no partial tile
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < (SCAN_THREADS / 32) * (NCLS + 1); i += SCAN_THREADS) (&cls_cnt[0][0])[i] = 0;
    __syncthreads();
    const uint32_t peers = __match_any_sync(0xffffffffu, cls);
    const int lane_rank = __popc(peers & ((1u << lane) - 1u));
    if (lane_rank == 0) cls_cnt[wid][cls] = __popc(peers);
    __syncthreads();
    if (threadIdx.x <= NCLS) {
        int run = 0;
        for (int w = 0; w < SCAN_THREADS / 32; ++w) {
            const int v = cls_cnt[w][threadIdx.x];
            cls_cnt[w][threadIdx.x] = run;
            run += v;
        }
        cls_base[threadIdx.x] = run;  // class total for now
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int b = n_full;
        for (int k = NCLS; k >= 1; --k) {
            const int tot = cls_base[k];
            cls_base[k] = b;
            b += tot;
        }
        s_n_tiles = b;
    }
    __syncthreads();
    const int n_tiles = s_n_tiles;
    if (tiles) {
        for (int i = 0; i < nfull; ++i) {
            Tile tl;
            tl.expert = e;
            tl.row0 = off + i * TILE_ROWS;
            tl.nrows = TILE_ROWS;
            tl.pad = 0;
            tiles[fpos + i] = tl;
        }
        if (cls > 0) {
            Tile tl;
            tl.expert = e;
            tl.row0 = off + nfull * TILE_ROWS;
            tl.nrows = rem;
            tl.pad = 0;
            tiles[cls_base[cls] + cls_cnt[wid][cls] + lane_rank] = tl;
        }
    }
    if (threadIdx.x == 0 && plan) {
        plan->n_uniq = n_uniq;
        plan->n_tiles = n_tiles;
    }
}

// Stable placement of assignments [a0, a1) by one warp, walking them in
// ascending order 32 at a time.  The id of assignment a is ids[a - ibase];
// run[e] holds the next free position of e.  When pos_out is given,
// pos_out[a - ibase] receives a's position (-1 for an id outside [0, E)).
__device__ void warp_stable_scatter(const int32_t* __restrict__ ids, int ibase, int a0, int a1, int E, int* run,
                                    int32_t* __restrict__ sorted, int32_t* __restrict__ inv,
                                    uint32_t* err, int32_t* pos_out = nullptr) {
    const int lane = threadIdx.x & 31;
    const uint32_t lt = (1u << lane) - 1u;
    for (int base = a0; base < a1; base += 32) {
        const int a = base + lane;
        int e = (a < a1) ? ids[a - ibase] : -1;
        const bool valid = (a < a1) && e >= 0 && e < E;
        if (a < a1 && !valid) set_error(err, ERRBIT_RANGE);
        const int key = valid ? e : -1;
        const uint32_t peers = __match_any_sync(0xffffffffu, key);
        if (valid) {
            const int rank = __popc(peers & lt);
            const int pos = run[e] + rank;
            sorted[pos] = a;
            inv[a] = pos;
            if (pos_out) pos_out[a - ibase] = pos;
        } else if (pos_out && a < a1) {
            pos_out[a - ibase] = -1;
        }
        __syncwarp();
        if (valid && (__ffs(peers) - 1) == lane) run[e] += __popc(peers);
        __syncwarp();
    }
}

// bf16x2 -> f16x2 (exact inside fp16's range); sets *bad on overflow.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v, bool& bad) {
    const uint32_t r = pack_f16x2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
    bad |= f16x2_nonfinite(r);
    return r;
}

// One activation row (d elements) copied by a warp, 16 bytes per lane,
// converting bf16 to fp16 when TO_F16 (then in the tensor-core operand order:
// K interleaved in groups of 8, see k8_interleave).  8 vectors per lane at a
// time, all loads in flight before the stores.
template <bool TO_F16>
__device__ __forceinline__ void copy_row(const uint16_t* __restrict__ src_row, uint16_t* __restrict__ dst_row, int d,
                                         int lane, bool& bad) {
    const int vec = d / 8;  // 16-byte vectors per row
    const uint4* src = reinterpret_cast<const uint4*>(src_row);
    uint4* dst = reinterpret_cast<uint4*>(dst_row);
    for (int v0 = 0; v0 < vec; v0 += 256) {
        uint4 q[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int v = v0 + lane + 32 * u;
            if (v < vec) q[u] = src[v];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int v = v0 + lane + 32 * u;
            if (v >= vec) break;
            if (TO_F16)
                q[u] = k8_interleave(bf16x2_to_f16x2(q[u].x, bad), bf16x2_to_f16x2(q[u].y, bad),
                                     bf16x2_to_f16x2(q[u].z, bad), bf16x2_to_f16x2(q[u].w, bad));
            dst[v] = q[u];
        }
    }
}

// Copy rows x[sorted[i] / k] -> x_perm[i] for i in [i0, i1), one warp a row.
template <bool TO_F16>
__device__ void gather_rows(const uint16_t* __restrict__ x, int d, int k, const int32_t* __restrict__ sorted,
                            int i0, int i1, uint16_t* __restrict__ x_perm, int warp, int nwarps, uint32_t* err) {
    const int lane = threadIdx.x & 31;
    bool bad = false;
    for (int i = i0 + warp; i < i1; i += nwarps) {
        const int a = sorted[i];
        if (a < 0 || a >= i1) continue;  // a slot left unwritten by out-of-range ids
        copy_row<TO_F16>(x + (size_t)(a / k) * d, x_perm + (size_t)i * d, d, lane, bad);
    }
    if (TO_F16 && bad) set_error(err, ERRBIT_F16_RANGE);
}

__device__ void gather_any(const AlignOut& o, const uint16_t* x, int d, int k, int R, int warp, int nwarps) {
    if (o.x_perm_f16)
        gather_rows<true>(x, d, k, o.sorted, 0, R, o.x_perm, warp, nwarps, o.err);
    else
        gather_rows<false>(x, d, k, o.sorted, 0, R, o.x_perm, warp, nwarps, o.err);
}

// -------------------------------------------------------------- small path
__global__ void __launch_bounds__(SCAN_THREADS) align_small_kernel(const int32_t* __restrict__ ids, int R, int k, int E,
                                                                   const uint16_t* __restrict__ x, int d,
                                                                   AlignOut o) {
    __shared__ int cnt[1024];
    __shared__ int run[1024];
    const int tid = threadIdx.x;
    if (tid < E) cnt[tid] = 0;
    __syncthreads();
    for (int a = tid; a < R; a += SCAN_THREADS) {
        const int e = ids[a];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
        else set_error(o.err, ERRBIT_RANGE);
    }
    __syncthreads();
    int my_off = 0;
    emit_plan(tid < E ? cnt[tid] : 0, tid, E, o.counts, o.offsets, o.uniq, o.tiles, o.plan, &my_off);
    if (tid < E) run[tid] = my_off;
    __syncthreads();
    if (tid < 32) warp_stable_scatter(ids, 0, 0, R, E, run, o.sorted, o.inv, o.err);
    if (o.x_perm) {
        __syncthreads();
        gather_any(o, x, d, k, R, tid >> 5, SCAN_THREADS / 32);
    }
}

// -------------------------------------------------------- multi-block path
__global__ void __launch_bounds__(256) align_hist_kernel(const int32_t* __restrict__ ids, int R, int E, int rows,
                                                         int32_t* __restrict__ blockcnt, uint32_t* err) {
    __shared__ int cnt[1024];
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int a0 = blockIdx.x * rows;
    const int a1 = min(R, a0 + rows);
    for (int a = a0 + threadIdx.x; a < a1; a += blockDim.x) {
        const int e = ids[a];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
        else set_error(err, ERRBIT_RANGE);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) blockcnt[(size_t)blockIdx.x * E + e] = cnt[e];
}

// One CTA (SCAN_THREADS threads) per block of assignments b:
//  1. per expert e, the assignments to e in blocks before b and in all blocks,
//     read from the count table by SCAN_THREADS / E thread groups, each
//     summing a contiguous slice of the blocks with all its loads in flight;
//  2. the expert offsets (exclusive scan of the totals; block 0 also writes
//     counts, offsets, the experts with rows and the token tiles);
//  3. the stable placement of block b's assignments by warp 0 from
//     run[e] = offset[e] + (assignments to e in earlier blocks);
//  4. with COPY, every warp copies activation rows of the block's
//     assignments to their positions in x_perm.
template <bool COPY>
__global__ void __launch_bounds__(SCAN_THREADS) align_place_kernel(const int32_t* __restrict__ ids, int R, int k, int E,
                                                                   int rows, int nblocks,
                                                                   const int32_t* __restrict__ blockcnt,
                                                                   const uint16_t* __restrict__ x, int d, AlignOut o) {
    __shared__ int s_pre[SCAN_THREADS];
    __shared__ int s_tot[SCAN_THREADS];
    __shared__ int run[1024];
    __shared__ int32_t bid[ALIGN_BLOCK_ROWS];
    __shared__ int32_t pos[ALIGN_BLOCK_ROWS];
    const int tid = threadIdx.x, b = blockIdx.x;
    const int a0 = b * rows, a1 = min(R, a0 + rows);
    for (int a = a0 + tid; a < a1; a += SCAN_THREADS) bid[a - a0] = ids[a];
    const int groups = SCAN_THREADS / E;  // >= 1 since E <= 1024
    if (tid < groups * E) {
        const int e = tid % E, j = tid / E;
        const int b_lo = (int)((long long)j * nblocks / groups);
        const int b_hi = (int)((long long)(j + 1) * nblocks / groups);
        constexpr int BATCH = 16;
        int pre = 0, tot = 0;
        for (int c0 = b_lo; c0 < b_hi; c0 += BATCH) {
            int c[BATCH];
#pragma unroll
            for (int i = 0; i < BATCH; ++i) c[i] = c0 + i < b_hi ? blockcnt[(size_t)(c0 + i) * E + e] : 0;
#pragma unroll
            for (int i = 0; i < BATCH; ++i) {
                tot += c[i];
                if (c0 + i < b) pre += c[i];
            }
        }
        s_pre[tid] = pre;
        s_tot[tid] = tot;
    }
    __syncthreads();
    int pre = 0, tot = 0;
    if (tid < E)
        for (int j = 0; j < groups; ++j) {
            pre += s_pre[j * E + tid];
            tot += s_tot[j * E + tid];
        }
    const bool lead = b == 0;
    int off = 0;
    emit_plan(tot, tid, E, lead ? o.counts : nullptr, lead ? o.offsets : nullptr, lead ? o.uniq : nullptr,
              lead ? o.tiles : nullptr, lead ? o.plan : nullptr, &off);
    if (tid < E) run[tid] = off + pre;
    __syncthreads();
    if (tid < 32) warp_stable_scatter(bid, a0, a0, a1, E, run, o.sorted, o.inv, o.err, pos);
    if (COPY) {
        __syncthreads();
        const int lane = tid & 31;
        bool bad = false;
        for (int i = tid >> 5; i < a1 - a0; i += SCAN_THREADS / 32) {
            const int p = pos[i];
            if (p < 0) continue;
            const uint16_t* src = x + (size_t)((a0 + i) / k) * d;
            if (o.x_perm_f16)
                copy_row<true>(src, o.x_perm + (size_t)p * d, d, lane, bad);
            else
                copy_row<false>(src, o.x_perm + (size_t)p * d, d, lane, bad);
        }
        if (bad) set_error(o.err, ERRBIT_F16_RANGE);
    }
}

__global__ void __launch_bounds__(256) gather_kernel(const uint16_t* __restrict__ x, int d, int k, int R, AlignOut o) {
    const int warps = blockDim.x >> 5;
    gather_any(o, x, d, k, R, blockIdx.x * warps + (threadIdx.x >> 5), gridDim.x * warps);
}

__global__ void __launch_bounds__(256) bf16_to_f16_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                                                          size_t n16, uint32_t* err) {
    bool bad = false;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x) {
        const uint4 q = in[i];
        out[i] = k8_interleave(bf16x2_to_f16x2(q.x, bad), bf16x2_to_f16x2(q.y, bad), bf16x2_to_f16x2(q.z, bad),
                               bf16x2_to_f16x2(q.w, bad));
    }
    if (bad) set_error(err, ERRBIT_F16_RANGE);
}

__global__ void __launch_bounds__(SCAN_THREADS) plan_from_offsets_kernel(const int32_t* __restrict__ offsets, int E,
                                                                         int32_t* uniq, Tile* tiles, DevPlan* plan) {
    const int e = threadIdx.x;
    const int c = (e < E) ? offsets[e + 1] - offsets[e] : 0;
    emit_plan(c, e, E, nullptr, nullptr, uniq, tiles, plan, nullptr);
}

}  // namespace

int align_block_rows(int R, int E) {
    // the smallest of 32, 64, 256 whose per-block count table fits in 64 KB:
    // more placing CTAs (each copies its own rows once they are enough to
    // fill the GPU); else 1024
    for (const int rows : {32, 64, 256})
        if ((size_t)ceil_div(R, rows) * E * sizeof(int32_t) <= 65536) return rows;
    return ALIGN_BLOCK_ROWS;
}

size_t align_blockcnt_bytes(int R, int E) {
    if (R <= ALIGN_SMALL_MAX_R) return 0;
    return (size_t)ceil_div(R, align_block_rows(R, E)) * E * sizeof(int32_t);
}

cudaError_t launch_align(const int32_t* ids, int T, int k, int E, const uint16_t* x, int d,
                         const AlignOut& o, cudaStream_t s) {
    const int R = T * k;
    if (R <= ALIGN_SMALL_MAX_R) {
        align_small_kernel<<<1, SCAN_THREADS, 0, s>>>(ids, R, k, E, x, d, o);
        note_launch();
        return cudaGetLastError();
    }
    const int rows = align_block_rows(R, E);
    const int nb = ceil_div(R, rows);
    align_hist_kernel<<<nb, 256, 0, s>>>(ids, R, E, rows, o.blockcnt, o.err);
    note_launch();
    // the placing CTAs copy the rows themselves when they are enough to keep
    // most SMs busy; otherwise a separate gather spreads the copy
    const bool copy_in_place = o.x_perm && nb >= num_sms() / 2;
    if (copy_in_place)
        align_place_kernel<true><<<nb, SCAN_THREADS, 0, s>>>(ids, R, k, E, rows, nb, o.blockcnt, x, d, o);
    else
        align_place_kernel<false><<<nb, SCAN_THREADS, 0, s>>>(ids, R, k, E, rows, nb, o.blockcnt, x, d, o);
    note_launch();
    if (o.x_perm && !copy_in_place) {
        const int blocks = min(ceil_div(R, 8), 8 * num_sms());
        gather_kernel<<<blocks, 256, 0, s>>>(x, d, k, R, o);
        note_launch();
    }
    return cudaGetLastError();
}

cudaError_t launch_bf16_to_f16(const uint16_t* in, uint16_t* out, size_t n, uint32_t* err, cudaStream_t s) {
    const size_t n16 = n / 8;
    if (n16 == 0) return cudaSuccess;
    const int blocks = (int)std::min<size_t>((n16 + 255) / 256, (size_t)num_sms() * 8);
    bf16_to_f16_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const uint4*>(in), reinterpret_cast<uint4*>(out), n16, err);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_plan_from_offsets(const int32_t* offsets, int E, int32_t* uniq, Tile* tiles,
                                     DevPlan* plan, cudaStream_t s) {
    plan_from_offsets_kernel<<<1, SCAN_THREADS, 0, s>>>(offsets, E, uniq, tiles, plan);
    note_launch();
    return cudaGetLastError();
}

}  // namespace moe
