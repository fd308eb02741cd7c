// The whole MoE layer for a few tokens (decode) as one dataflow kernel.
//
// With T <= 8 tokens the layer is a stream of the routed experts' int4 weights
// past a handful of activation vectors: "Performance and verification"
// (bloomery docs/performance.md), section "Why it is fast", fetches each
// expert's weights once per batch and computes on the packed codes directly;
// "Measured results" (vllm-omni docs/edge/results.md), section Fidelity,
// fixes the W4A16 g128 format.  The kernel keeps that stream flowing from the
// first weight byte to the last, with no grid-wide synchronisation:
//
//   routing  every CTA routes all T tokens itself (top-k of the fp32 logits,
//            softmax over the selection) and sorts the T*k assignments by
//            expert: U touched experts, their token lists.
//   units    the layer is cut into units of work, numbered in one global
//            order: first the gate_up units (8 features of one touched expert:
//            its 8 gate and 8 up rows over d_model, SiLU(gate)*up for each of
//            the expert's tokens -> h), expert by expert, then the down units
//            (32 output rows of one touched expert over d_ff, for each of its
//            tokens -> y).  CTA c takes units c, c + G, c + 2G, ... (G CTAs)
//            and hands them to its NQ pipelines (one producer warp, four
//            consumer warps each) in turn: every SM gets the same share, and
//            all SMs work through the gate_up units expert after expert.
//   h        a gate_up unit writes its h values (fp16) to the workspace and
//            counts itself done in the expert's readiness counter.  A down
//            unit's producer streams the unit's weights first, then waits for
//            its expert's counter to be complete (all its h written) and copies
//            the expert's h rows into shared memory; by the time the down
//            units of an expert come up its gate_up units finished long ago.
//   combine  a down unit writes y (fp32) per assignment; the CTA's publisher
//            warp counts it in the counter of each (token, 32-row block) it
//            fed, and the token's k-th count sums all k y rows in slot order
//            (deterministic) into the bf16 output.  Every counter returns to
//            zero by the end of a call.
//   publish  consumers never wait on global memory: they store h or y and
//            hand the unit to the publisher warp through shared memory; it
//            makes batches of units visible with one gpu-scope fence and does
//            the counting and combining.
//
// A down unit waits only for gate_up units of lower index, which never wait
// on another CTA, so the waits cannot form a cycle; all CTAs must be resident
// for that (cooperative launch, one CTA per SM).
//
// Inner loop (decode_ops.cuh): one warp holds the A fragment of an m16n8k16
// MMA (16 weight rows x 16 codes) in registers, decoded from the packed words
// (1024 + q or 64 + q as fp16, exact); B holds the activations (or h) of the
// expert's tokens in fp16; per group of 128 codes the offsets, zero and scale
// are removed in fp32: sum((q - z) s x) = s (acc - C1 - z C2).
//
// Every wait is bounded (2 s); a wait that gives up records a timeout in the
// workspace error word, raises the CTA's and the grid's abort flags and the
// kernel winds down: producers issue nothing more and drain what they issued,
// consumers pass through their remaining barriers without work.
#include "decode_ops.cuh"
#include "fastdiv.h"

namespace moe {
namespace {

using namespace dec;
using tc::WAIT_LIMIT_NS;

template <int NQ_>
struct FlowShape {
    static constexpr int NQ = NQ_;                 // pipelines per CTA
    static constexpr int QW = 4;                   // consumer warps per pipeline
    static constexpr int CW = NQ_ * QW;            // consumer warps 0 .. CW - 1
    static constexpr int PRODUCER_WARP = CW;       // producer warps CW .. CW + NQ - 1
    static constexpr int PUBLISHER_WARP = CW + NQ_;
    static constexpr int NTHREADS = 32 * (CW + NQ_ + 1);
};

constexpr int NF = 64;          // "full" barriers per pipeline, indexed by chunk number mod NF
constexpr int MAX_SLOTS = 48;
constexpr int FG = 8;           // features per gate_up unit (8 gate + 8 up rows: one m16 tile)
constexpr int RD = 32;          // output rows per down unit (two m16 tiles)
constexpr int MAX_NHS = 2;      // h slots per pipeline
constexpr uint32_t GRID_WAIT_POLL = 16;
constexpr int NPUB = 128;       // publication queue entries
enum { PUB_GATEUP = 0, PUB_DOWN = 1, PUB_END = 2 };

// Units a CTA's consumers finished and whose results the publisher warp makes
// visible to the other CTAs: consumers write an entry and release its flag
// (the entry's index + 1); the publisher acquires entries in order.
struct PubQ {
    int32_t tail;            // next entry index (shared-memory atomic)
    int32_t head;            // first entry the publisher has not retired
    int32_t pad[30];
    int4 ent[NPUB];          // kind, touched expert, unit index inside the expert, 0
    uint32_t flag[NPUB];
};

// Named barriers: 0 is __syncthreads; 2 .. 2 + NQ - 1 the pipelines' quads.
constexpr int BAR_ROUTED = 8, BAR_SORTED = 9, BAR_CONSUMERS = 10, BAR_SORT2 = 11;

struct FlowTab {
    int32_t ids[MAX_R];     // routing, slot a = t*k + j
    float w[MAX_R];
    int32_t pa[MAX_R];      // assignment at permuted position i
    int32_t ptok[MAX_R];    // its token
    int32_t uexp[MAX_R];    // touched experts, ascending
    int32_t uoff[MAX_R];    // first permuted position of each
    int32_t ucnt[MAX_R];    // and its number of tokens
    int32_t first[MAX_R];   // sort scratch
    int32_t n_uniq;
    int32_t abort;
    int32_t pad[30];
};

struct FlowParams {
    const uint16_t* x;        // bf16 [T][d]
    const float* logits;      // fp32 [T][E]
    const uint16_t *w13_s, *w13_z, *w2_s, *w2_z;
    uint16_t* out;            // bf16 [T][d]
    int32_t* ids_out;         // [T][k] or null
    uint8_t* hb;              // fp16 [R][f] in the staged order, row = permuted position
    float* ybuf;              // fp32 [R][d], row = assignment
    uint32_t* hdr;            // workspace header (error word, queue counter, abort flag)
    uint32_t* ready;          // [MAX_R] gate_up units done per touched expert
    uint32_t* done;           // [MAX_R] down units done per touched expert
    uint32_t* ccnt;           // [T][d / RD] contributions per (token, row block)
    int T, k, E, d, f;
    int nslot, nhs, cmax;     // ring slots (multiple of NQ), h slots per pipeline, rows per h slot
    uint32_t off_sz, off_bars, off_desc, off_xb, off_cx, off_hs, off_red, off_tab, off_pub;
    int xb_stride, hs_stride, hs_bytes, hs_csum;
    int sz13_mode, sz2_mode, sz13_rs, sz2_rs;
    uint32_t clear_bytes;
    FastDiv fd_gpe, fd_dpe, fd_k, fd_xw, fd_gf;
};

__device__ __forceinline__ uint32_t ld_acquire_gpu32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_volatile32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.volatile.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ float ldg_cg_f32(const float* p) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ void bar_arrive(int id, int n) {
    asm volatile("bar.arrive %0, %1;" :: "r"(id), "r"(n) : "memory");
}
// Barrier over n threads that returns, to all of them, whether any passed a
// non-zero predicate.
__device__ __forceinline__ bool bar_red_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"((uint32_t)pred), "r"(id), "r"(n) : "memory");
    return r != 0;
}
__device__ __forceinline__ float half_bits(uint32_t h) { return __half2float(__ushort_as_half((uint16_t)h)); }
__device__ __forceinline__ void st_release_cta_u32(uint32_t* p, uint32_t v) {
    asm volatile("st.release.cta.shared.u32 [%0], %1;" :: "r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_cta_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void red_add_gpu(uint32_t* p, uint32_t v) {
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// One consumer quad's entry for the publisher (lane 0 of the quad's warp 0,
// after the unit's global stores are ordered before it by a warp or quad
// barrier).  Waits (bounded) while the queue is full.
__device__ __forceinline__ void pub_push(PubQ& q, int kind, int u, int idx, volatile int* abort_flag, uint32_t* err) {
    const int slot = atomicAdd(&q.tail, 1);
    const uint64_t t0 = globaltimer_ns();
    while (slot - *reinterpret_cast<volatile int32_t*>(&q.head) >= NPUB) {
        if (*abort_flag || globaltimer_ns() - t0 > tc::WAIT_LIMIT_NS) {
            if (!*abort_flag) set_error(err, ERRBIT_TIMEOUT);
            *abort_flag = 1;
            break;
        }
        __nanosleep(200);
    }
    q.ent[slot % NPUB] = make_int4(kind, u, idx, 0);
    st_release_cta_u32(&q.flag[slot % NPUB], (uint32_t)slot + 1u);
}

// Groups l0 .. l0 + n - 1 (chunk-local) of the chunk whose codes are at sa and
// whose scales and zeros are at szs (row stride rs bytes), for this lane's
// rows g and g + 8; gi0 is the chunk's first group along the reduction axis.
__device__ __forceinline__ void consume_range(float (&acc)[4], uint32_t sa, uint32_t szs, uint32_t rs, int l0, int n,
                                              int g, int t, int gi0, uint32_t brow_a, uint32_t bact, uint32_t c0_a,
                                              uint32_t c1_a) {
    const uint32_t szb = szs + (uint32_t)g * rs;
#pragma unroll 2
    for (int i = 0; i < n; ++i) {
        const int gl = l0 + i;
        const uint32_t aoff = a_offset(gl, g, t);
        const uint4 wa = lds128(sa + aoff), wb = lds128(sa + BOX_BYTES + aoff);
        const uint32_t sb = szb + 2u * (uint32_t)gl;
        const float s0 = half_bits(lds_u16(sb)), z0 = half_bits(lds_u16(sb + SZ_ARRAY));
        const float s1 = half_bits(lds_u16(sb + 8u * rs)), z1 = half_bits(lds_u16(sb + SZ_ARRAY + 8u * rs));
        const uint32_t gi = (uint32_t)(gi0 + gl);
        compute_group(acc, wa, wb, s0, z0, s1, z1, t, brow_a + 256u * gi, bact, c0_a + 8u * gi, c1_a + 8u * gi);
    }
}

template <int NQ_>
__global__ void __launch_bounds__(FlowShape<NQ_>::NTHREADS, 1)
decode_flow_kernel(const __grid_constant__ CUtensorMap map13, const __grid_constant__ CUtensorMap map2,
                   const __grid_constant__ CUtensorMap map13s, const __grid_constant__ CUtensorMap map13z,
                   const __grid_constant__ CUtensorMap map2s, const __grid_constant__ CUtensorMap map2z,
                   const FlowParams p) {
    constexpr int NQ = FlowShape<NQ_>::NQ, QW = FlowShape<NQ_>::QW, CW = FlowShape<NQ_>::CW;
    constexpr int PRODUCER_WARP = FlowShape<NQ_>::PRODUCER_WARP, PUBLISHER_WARP = FlowShape<NQ_>::PUBLISHER_WARP;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sbase = smem_u32(sm);
    FlowTab& tab = *reinterpret_cast<FlowTab*>(sm + p.off_tab);
    volatile int* abort_flag = &tab.abort;
    int32_t* desc = reinterpret_cast<int32_t*>(sm + p.off_desc);     // [nslot] unit of the chunk in each slot
    PubQ& pq = *reinterpret_cast<PubQ*>(sm + p.off_pub);
    const uint32_t szbase = sbase + p.off_sz;
    const uint32_t full0 = sbase + p.off_bars;                        // [NQ][NF]
    const uint32_t empty0 = full0 + 8u * (NQ * NF);                   // [MAX_SLOTS]
    const uint32_t hfull0 = empty0 + 8u * MAX_SLOTS;                  // [NQ][MAX_NHS]
    const uint32_t hempty0 = hfull0 + 8u * (NQ * MAX_NHS);            // [NQ][MAX_NHS]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = p.T, k = p.k, R = T * k, E = p.E, d = p.d, f = p.f;
    const int Gd = d >> 7, Gf = f >> 7;
    const int G = gridDim.x, cta = blockIdx.x;
    const int ns4 = p.nslot / NQ;
    const int nsort = T > 2 ? T : 2;  // warps that route (t < T) and sort (warps 0, 1)

    // ------------------------------------------------- setup and routing
    float* lgs = reinterpret_cast<float*>(sm);  // the routed tokens' logits, in the idle ring
    if (threadIdx.x == 0) tab.abort = 0;
    if (warp == PUBLISHER_WARP) {
        for (int i = lane; i < NPUB; i += 32) pq.flag[i] = 0u;
        if (lane == 0) pq.tail = pq.head = 0;
    }
    if (warp == PRODUCER_WARP) {
        for (int i = lane; i < NQ * NF; i += 32) tc::mbar_init(full0 + 8u * i, 1);
        for (int i = lane; i < p.nslot; i += 32) tc::mbar_init(empty0 + 8u * i, QW);
        for (int i = lane; i < NQ * MAX_NHS; i += 32) {
            tc::mbar_init(hfull0 + 8u * i, 1);
            tc::mbar_init(hempty0 + 8u * i, QW);
        }
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
    // stream (where the driver accepts it), the CTA may start while that
    // kernel drains: everything above touches only this CTA's shared memory.
    // From here on global memory is read and written, so wait until the
    // previous grid has completed and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (cta == 0 && threadIdx.x == 0) p.hdr[WS_CLEAR_WORD] = p.clear_bytes;

    if (warp < nsort) {
        if (warp < T) {
            float* lrow = lgs + warp * E;
            const float* src = p.logits + (size_t)warp * E;
            for (int e = lane; e < E; e += 32) lrow[e] = __ldg(src + e);
            __syncwarp();
            route_token(lrow, E, k, &tab.ids[warp * k], &tab.w[warp * k]);
            // the logits' ring bytes are overwritten by TMA once the producers start
            tc::fence_proxy_async_smem();
        }
        bar_sync(BAR_ROUTED, 32 * nsort);
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
            bar_sync(BAR_SORT2, 64);
            int ui = 0, nu = 0;
            for (int b = 0; b < R; ++b) {
                const int fb = tab.first[b];
                nu += fb;
                ui += fb & (tab.ids[b] < ea);
            }
            if (va) {
                const int pos = lt + eqb;
                tab.pa[pos] = a;
                tab.ptok[pos] = (int)fd_div((uint32_t)a, p.fd_k);
            }
            if (first) {
                tab.uexp[ui] = ea;
                tab.uoff[ui] = lt;
                tab.ucnt[ui] = eqall;
            }
            if (a == 0) tab.n_uniq = nu;
            bar_arrive(BAR_SORTED, 64 + 32 * (NQ + 1));  // the routing tables are complete
        }
    } else if (warp < CW) {
        // activations -> fp16 in MMA order, plus C1/C2 per (token, group); the
        // C1/C2 row T (B columns without a token) and every h slot's zero
        // C1/C2 row are zero
        const int nthr = (CW - nsort) * 32, tid = (warp - nsort) * 32 + lane;
        const int wpr = d >> 3;
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
            if (bad) set_error(p.hdr, ERRBIT_F16_RANGE);
            const uint4 o = k8_interleave(q[0], q[1], q[2], q[3]);
            sts128(sbase + p.off_xb + (uint32_t)(t * p.xb_stride) + staged_offset(wr * 8), o);
            const float2 c = halfwarp_sum(word_c1c2(o));
            if ((lane & 15) == 0) cx[t * Gd + (wr >> 4)] = c;
        }
        for (int i = tid; i < Gd; i += nthr) cx[T * Gd + i] = make_float2(0.f, 0.f);
        const int nzr = NQ * p.nhs * Gf;
        for (int i = tid; i < nzr; i += nthr) {
            const int hsi = i / Gf, gi = i - hsi * Gf;
            float2* cz = reinterpret_cast<float2*>(sm + p.off_hs + (size_t)hsi * p.hs_bytes + p.hs_csum);
            cz[p.cmax * Gf + gi] = make_float2(0.f, 0.f);
        }
    }

    const int gpe = f / FG, dpe = d / RD;  // units per touched expert

    // ---------------------------------------------------------- producers
    // Lane 0 issues every copy of the pipeline: the weight chunks of its units
    // in order and, for each down unit, the expert's h rows.  A down unit's
    // weights never wait for its h: its h copy is queued and issued, in unit
    // order, as soon as the expert's gate_up units have all written their h
    // and one of the pipeline's h slots is free; pending copies are served
    // between chunks and while the ring is full (the consumers need a down
    // unit's h only when they reach it).
    if (warp >= PRODUCER_WARP && warp < PUBLISHER_WARP) {
        bar_sync(BAR_SORTED, 64 + 32 * (NQ + 1));
        if (lane != 0) return;
        const int qp = warp - PRODUCER_WARP;
        const int U = tab.n_uniq;
        const int NG = U * gpe, N = NG + U * dpe;
        const uint32_t fullq = full0 + 8u * (uint32_t)(qp * NF);
        const uint32_t slot0 = (uint32_t)(qp * ns4);
        const int nch1 = ceil_div(Gd, CHUNK_GROUPS), nch2 = ceil_div(Gf, CHUNK_GROUPS);
        const uint32_t tx13 = SLOT_CODE + (p.sz13_mode == SZ_TMA ? SLOT_SZ : 64u * (uint32_t)Gd);
        const uint32_t tx2 = SLOT_CODE + (p.sz2_mode == SZ_TMA ? SLOT_SZ : 64u * (uint32_t)Gf);
        uint32_t* grid_abort = p.hdr + WS_ABORT_WORD;
        uint32_t qq = 0, sl = 0, round = 0, hq = 0;
        bool ok = true;
        auto raise_abort = [&]() {
            *abort_flag = 1;
            atomicExch(grid_abort, 1u);
        };
        // down units whose h copy is not issued yet, oldest first
        constexpr int PEND = 16;
        int pend[PEND];
        int np = 0, pf = 0;
        uint32_t pv = 0;     // the front unit's last readiness load (acquire)
        bool pv_set = false;
        // Issues pending h copies that can go now; with `block`, waits
        // (bounded) until every pending copy is issued.  False on abort.
        auto serve_h = [&](bool block) -> bool {
            const uint64_t t0 = block ? globaltimer_ns() : 0;
            for (uint32_t it = 1; np > 0; ++it) {
                const int u = pend[pf];
                const uint32_t hs = (uint32_t)p.nhs == 1 ? 0u : (hq & 1u);
                const uint32_t huse = (uint32_t)p.nhs == 1 ? hq : (hq >> 1);
                const bool slot_ok =
                    huse == 0 || tc::mbar_try_wait(hempty0 + 8u * (uint32_t)(qp * MAX_NHS + hs), (huse - 1) & 1u);
                const bool ready = pv_set && pv == (uint32_t)gpe;
                if (slot_ok && ready) {
                    // the h rows were written by other CTAs' generic stores,
                    // acquired above; the bulk copy reads them through the
                    // async proxy
                    fence_proxy_async_global();
                    const int cnt = tab.ucnt[u], off = tab.uoff[u];
                    const uint32_t hrow = 2u * (uint32_t)f;
                    const uint32_t hfull = hfull0 + 8u * (uint32_t)(qp * MAX_NHS + hs);
                    const uint32_t hdst = sbase + p.off_hs + (uint32_t)((qp * p.nhs + (int)hs) * p.hs_bytes);
                    tc::mbar_arrive_expect_tx(hfull, (uint32_t)cnt * hrow);
                    for (int r = 0; r < cnt; ++r)
                        tc::bulk_load(hdst + (uint32_t)(r * p.hs_stride), p.hb + (size_t)(off + r) * hrow, hrow, hfull);
                    ++hq;
                    pf = (pf + 1) % PEND;
                    --np;
                    pv_set = false;
                    continue;
                }
                if (!ready) {
                    pv = ld_acquire_gpu32(p.ready + u);  // checked on the next pass
                    pv_set = true;
                }
                if (!block) return true;
                __nanosleep(100);
                if ((it % GRID_WAIT_POLL) == 0) {
                    if (*abort_flag || ld_volatile32(grid_abort)) {
                        *abort_flag = 1;
                        return false;
                    }
                    if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
                        set_error(p.hdr, ERRBIT_TIMEOUT);
                        raise_abort();
                        return false;
                    }
                }
            }
            return true;
        };
        // The next ring slot is free: its previous chunk was consumed.  A slot
        // that consumers gave back because they gave up is released only
        // after the abort flag was raised, so nothing is issued into it.
        // Pending h copies are served while waiting.  (Only the CTA's flag in
        // shared memory is read per chunk: a global load there would cost an
        // L2 round trip on the issue path.)
        auto slot_wait = [&]() -> bool {
            if (round != 0) {
                const uint32_t bar = empty0 + 8u * (slot0 + sl), par = (round - 1) & 1u;
                const uint64_t t0 = globaltimer_ns();
                for (uint32_t it = 1;; ++it) {
                    if (np == 0 ? tc::mbar_try_wait_sleep(bar, par) : tc::mbar_try_wait_sleep_short(bar, par)) break;
                    if (!serve_h(false)) return false;
                    if ((it & 7u) == 0) {
                        if (*abort_flag) return false;
                        if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
                            set_error(p.hdr, ERRBIT_TIMEOUT);
                            raise_abort();
                            return false;
                        }
                    }
                }
            }
            return !*abort_flag;
        };
        auto advance = [&]() {
            ++qq;
            if (++sl == (uint32_t)ns4) {
                sl = 0;
                ++round;
            }
        };
        // one chunk: its unit number for the consumers, then the codes and
        // the scales and zeros
        auto issue = [&](int v, bool up, int c, int row0, int ex, int fb8) -> bool {
            if (!slot_wait()) return false;
            const uint32_t slot = slot0 + sl;
            desc[slot] = v;
            const uint32_t full = fullq + 8u * (qq & (NF - 1));
            const uint32_t dst = sbase + slot * SLOT_CODE, sdst = szbase + slot * SLOT_SZ;
            const int g0 = c * CHUNK_GROUPS;
            if (up) {
                tc::mbar_arrive_expect_tx(full, tx13);
                tc::tma_load_4d(dst, &map13, full, 0, c * LINES, fb8, 2 * ex);
                if (p.sz13_mode == SZ_TMA) {
                    tc::tma_load_3d(sdst, &map13s, full, g0, fb8, 2 * ex);
                    tc::tma_load_3d(sdst + SZ_ARRAY, &map13z, full, g0, fb8, 2 * ex);
                } else {
                    // 8 gate rows, then the 8 up rows, of every group
                    const uint32_t hbytes = 16u * (uint32_t)Gd;
                    const size_t r0 = (size_t)ex * 2 * f + fb8, r1 = r0 + f;
                    tc::bulk_load(sdst, p.w13_s + r0 * Gd, hbytes, full);
                    tc::bulk_load(sdst + hbytes, p.w13_s + r1 * Gd, hbytes, full);
                    tc::bulk_load(sdst + SZ_ARRAY, p.w13_z + r0 * Gd, hbytes, full);
                    tc::bulk_load(sdst + SZ_ARRAY + hbytes, p.w13_z + r1 * Gd, hbytes, full);
                }
            } else {
                tc::mbar_arrive_expect_tx(full, tx2);
                tc::tma_load_3d(dst, &map2, full, 0, c * LINES, row0);
                if (p.sz2_mode == SZ_TMA) {
                    tc::tma_load_2d(sdst, &map2s, full, g0, row0);
                    tc::tma_load_2d(sdst + SZ_ARRAY, &map2z, full, g0, row0);
                } else {
                    tc::bulk_load(sdst, p.w2_s + (size_t)row0 * Gf, 32u * (uint32_t)Gf, full);
                    tc::bulk_load(sdst + SZ_ARRAY, p.w2_z + (size_t)row0 * Gf, 32u * (uint32_t)Gf, full);
                }
            }
            advance();
            return true;
        };
        // This pipeline's units: the CTA takes units cta, cta + G, cta + 2G, ...
        // (every CTA the same share, within one unit, in the global order, so
        // all CTAs work through the gate_up units expert by expert at the
        // same pace) and hands them to its pipelines in turn.
        for (int v = cta + G * qp; v < N && ok; v += G * NQ) {
            if (v < NG) {
                const int u = (int)fd_div((uint32_t)v, p.fd_gpe), fb = v - u * gpe;
                const int ex = tab.uexp[u];
                for (int c = 0; c < nch1 && ok; ++c) ok = issue(v, true, c, 0, ex, fb * FG);
            } else {
                const int vd = v - NG;
                const int u = (int)fd_div((uint32_t)vd, p.fd_dpe), rb = vd - u * dpe;
                const int ex = tab.uexp[u];
                if (np == PEND) ok = serve_h(true);
                if (ok) {
                    pend[(pf + np) % PEND] = u;
                    ++np;
                }
                for (int m = 0; m < 2 && ok; ++m)
                    for (int c = 0; c < nch2 && ok; ++c) ok = issue(v, false, c, ex * d + rb * RD + m * 16, ex, 0);
                if (ok) ok = serve_h(false);
            }
        }
        if (ok) ok = serve_h(true);
        // end of this pipeline's stream
        if (ok && slot_wait()) {
            desc[slot0 + sl] = -1;
            tc::mbar_arrive(fullq + 8u * (qq & (NF - 1)));
            advance();
        }
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        // drain: the last use of each of the pipeline's ring slots and h
        // slots must have landed before the CTA exits
        const uint64_t t0 = globaltimer_ns();
        bool late = false;
        const uint32_t first = qq > (uint32_t)ns4 ? qq - (uint32_t)ns4 : 0u;
        for (uint32_t qx = first; qx < qq && !late; ++qx)
            while (!tc::mbar_try_wait(fullq + 8u * (qx & (NF - 1)), (qx / NF) & 1u))
                if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
                    late = true;
                    break;
                }
        const uint32_t hfirst = hq > (uint32_t)p.nhs ? hq - (uint32_t)p.nhs : 0u;
        for (uint32_t hx = hfirst; hx < hq && !late; ++hx) {
            const uint32_t hs = (uint32_t)p.nhs == 1 ? 0u : (hx & 1u);
            const uint32_t huse = (uint32_t)p.nhs == 1 ? hx : (hx >> 1);
            while (!tc::mbar_try_wait(hfull0 + 8u * (uint32_t)(qp * MAX_NHS + hs), huse & 1u))
                if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
                    late = true;
                    break;
                }
        }
        if (late) set_error(p.hdr, ERRBIT_TIMEOUT);
        return;
    }

    // ---------------------------------------------------------- publisher
    // Makes the results of this CTA's finished units visible to the other
    // CTAs, in batches: one gpu-scope fence, then a readiness increment per
    // gate_up unit, and per down unit a count in each of its tokens'
    // (token, row block) counters; the token's k-th count combines the k y
    // rows in slot order into the bf16 output.  The last down unit of an
    // expert returns the expert's counters to zero.
    if (warp == PUBLISHER_WARP) {
        bar_arrive(BAR_CONSUMERS, 32 * (CW + 1));  // the queue is initialised: consumers may push
        bar_sync(BAR_SORTED, 64 + 32 * (NQ + 1));
        const int U = tab.n_uniq;
        const int nrb = d / RD;
        int head = 0, ends = 0;
        uint64_t t_last = globaltimer_ns();  // lane 0's clock decides for the warp
        while (ends < NQ) {
            // the entries head .. head + n - 1 whose flags are released
            const int e_i = head + lane;
            const bool rdy = ld_acquire_cta_u32(&pq.flag[e_i % NPUB]) == (uint32_t)e_i + 1u;
            const uint32_t rmask = __ballot_sync(0xffffffffu, rdy);
            const int n = rmask == 0xffffffffu ? 32 : __ffs(~rmask) - 1;  // leading ready entries
            const uint64_t now = globaltimer_ns();
            if (n == 0) {
                // nothing new: bounded wait (consumers always end with an end entry)
                if (__shfl_sync(0xffffffffu, now - t_last > WAIT_LIMIT_NS ? 1 : 0, 0)) {
                    if (lane == 0) {
                        set_error(p.hdr, ERRBIT_TIMEOUT);
                        *abort_flag = 1;
                    }
                    break;
                }
                __nanosleep(100);
                continue;
            }
            t_last = now;
            const int4 en = lane < n ? pq.ent[e_i % NPUB] : make_int4(PUB_END + 1, 0, 0, 0);
            ends += __popc(__ballot_sync(0xffffffffu, lane < n && en.x == PUB_END));
            const bool live = !*abort_flag;
            const bool isg = lane < n && en.x == PUB_GATEUP && en.y >= 0 && en.y < U;
            const bool isd = lane < n && en.x == PUB_DOWN && en.y >= 0 && en.y < U && en.z >= 0 && en.z < nrb;
            fence_acq_rel_gpu();  // the units' stores before the counts below
            if (live && isg) red_add_gpu(p.ready + en.y, 1u);
            uint32_t lastm = 0;   // bit c: token column c of this lane's down unit completes its row block
            if (live && isd) {
                const int cnt = tab.ucnt[en.y], off = tab.uoff[en.y];
                uint32_t old[MAX_T];
#pragma unroll
                for (int c = 0; c < MAX_T; ++c)
                    if (c < cnt) old[c] = atomicAdd(p.ccnt + (size_t)tab.ptok[off + c] * nrb + en.z, 1u);
                const uint32_t od = atomicAdd(p.done + en.y, 1u);
#pragma unroll
                for (int c = 0; c < MAX_T; ++c)
                    if (c < cnt && old[c] == (uint32_t)k - 1u) {
                        atomicExch(p.ccnt + (size_t)tab.ptok[off + c] * nrb + en.z, 0u);
                        lastm |= 1u << c;
                    }
                if (od == (uint32_t)dpe - 1u) {
                    // every down unit of the expert is through its wait: reset
                    atomicExch(p.ready + en.y, 0u);
                    atomicExch(p.done + en.y, 0u);
                }
            }
            if (__any_sync(0xffffffffu, lastm != 0)) {
                fence_acq_rel_gpu();  // the other contributions' y rows after their counts
                for (uint32_t lm = __ballot_sync(0xffffffffu, lastm != 0); lm; lm &= lm - 1u) {
                    const int src = __ffs(lm) - 1;
                    const int su = __shfl_sync(0xffffffffu, en.y, src), srb = __shfl_sync(0xffffffffu, en.z, src);
                    for (uint32_t cm = __shfl_sync(0xffffffffu, lastm, src); cm; cm &= cm - 1u) {
                        const int tok = tab.ptok[tab.uoff[su] + __ffs(cm) - 1];
                        const int row = srb * RD + lane;
                        const float* ycol = p.ybuf + (size_t)tok * k * d + row;
                        float sum = 0.f;
                        for (int j0 = 0; j0 < k; j0 += 8) {
                            float yv[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                yv[j] = j0 + j < k ? ldg_cg_f32(ycol + (size_t)(j0 + j) * d) : 0.f;
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                if (j0 + j < k) sum = fmaf(tab.w[tok * k + j0 + j], yv[j], sum);
                        }
                        p.out[(size_t)tok * d + row] = float_to_bf16_bits(sum);
                    }
                }
            }
            head += n;
            __syncwarp();
            if (lane == 0) *reinterpret_cast<volatile int32_t*>(&pq.head) = head;
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    bar_sync(BAR_CONSUMERS, 32 * (CW + 1));
    if (cta == 0 && p.ids_out)
        for (int a = threadIdx.x; a < R; a += 32 * CW) p.ids_out[a] = tab.ids[a];
    const int qp = warp >> 2, w4 = warp & 3;
    const int g = lane >> 2, t4 = lane & 3;
    const int qbar = 2 + qp;
    const int U = tab.n_uniq;
    const int NG = U * gpe;
    const int nch1 = ceil_div(Gd, CHUNK_GROUPS), nch2 = ceil_div(Gf, CHUNK_GROUPS);
    const uint32_t fullq = full0 + 8u * (uint32_t)(qp * NF);
    const uint32_t slot0 = (uint32_t)(qp * ns4);
    const uint32_t xb = sbase + p.off_xb, cxa = sbase + p.off_cx;
    // partial sums for the unit's reduction: [2 (unit parity)][3 warps][2 tiles][32 lanes]
    float4* red = reinterpret_cast<float4*>(sm + p.off_red) + qp * (2 * 6 * 32);
    // every chunk's groups are split among the quad's four warps, so all four
    // compute each chunk as it lands
    auto my_groups = [&](int ng, int& lo, int& n) {
        lo = w4 * ng / QW;
        n = (w4 + 1) * ng / QW - lo;
    };
    uint32_t qq = 0, sl = 0, hq = 0, ucount = 0;
    auto slot_of = [&](int c) -> uint32_t {
        uint32_t s = sl + (uint32_t)c;
        while (s >= (uint32_t)ns4) s -= (uint32_t)ns4;
        return slot0 + s;
    };
    auto wait_chunk = [&](int c) -> bool {
        const uint32_t q = qq + (uint32_t)c;
        return tc::mbar_wait(fullq + 8u * (q & (NF - 1)), (q / NF) & 1u, abort_flag, p.hdr);
    };
    auto release = [&](uint32_t slot) {
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(empty0 + 8u * slot);
    };
    for (;;) {
        bool good = wait_chunk(0);
        const int v = good ? desc[slot_of(0)] : -1;
        // the quad takes the same branch: stop when any warp saw the end
        // marker or gave up
        if (bar_red_or(qbar, 32 * QW, v < 0)) break;
        float4* rb4 = red + (ucount & 1u) * (6 * 32);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        int nch;
        if (v < NG) {
            // ------------------------------------------------ gate_up unit
            nch = nch1;
            const int u = (int)fd_div((uint32_t)v, p.fd_gpe), fb = v - u * gpe;
            const int cnt = tab.ucnt[u], off = tab.uoff[u];
            const int col = lane >> 2;
            const int brow = col < cnt ? tab.ptok[off + col] : 0;
            const int cr0 = 2 * t4 < cnt ? tab.ptok[off + 2 * t4] : T;
            const int cr1 = 2 * t4 + 1 < cnt ? tab.ptok[off + 2 * t4 + 1] : T;
            const uint32_t brow_a = xb + (uint32_t)(brow * p.xb_stride);
            const uint32_t c0_a = cxa + (uint32_t)(cr0 * Gd * 8), c1_a = cxa + (uint32_t)(cr1 * Gd * 8);
            for (int c = 0; c < nch1; ++c) {
                if (c > 0) good &= wait_chunk(c);
                const uint32_t slot = slot_of(c);
                int l0, n;
                my_groups(min(CHUNK_GROUPS, Gd - c * CHUNK_GROUPS), l0, n);
                if (good && n > 0)
                    consume_range(acc, sbase + slot * SLOT_CODE, szbase + slot * SLOT_SZ, (uint32_t)p.sz13_rs, l0, n,
                                  g, t4, c * CHUNK_GROUPS, brow_a, (uint32_t)(col < cnt), c0_a, c1_a);
                release(slot);
            }
            // the four warps' partial sums, added in warp order
            if (w4 != 0) rb4[(w4 - 1) * 2 * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            bar_sync(qbar, 32 * QW);
            if (w4 == 0) {
#pragma unroll
                for (int i = 0; i < 3; ++i) {
                    const float4 o = rb4[i * 2 * 32 + lane];
                    acc[0] += o.x;
                    acc[1] += o.y;
                    acc[2] += o.z;
                    acc[3] += o.w;
                }
                if (good && !*abort_flag) {
                    // h = SiLU(gate) * up for feature fb*8 + g (rows g and g + 8
                    // of the tile), columns 2 t4 and 2 t4 + 1
                    const uint32_t hoff = staged_offset(fb * FG + g);
#pragma unroll
                    for (int mm = 0; mm < 2; ++mm) {
                        const int cm = 2 * t4 + mm;
                        if (cm < cnt) {
                            const __half hh = __float2half_rn(silu(acc[mm]) * acc[2 + mm]);
                            if (__hisinf(hh) || __hisnan(hh)) set_error(p.hdr, ERRBIT_F16_RANGE);
                            *reinterpret_cast<__half*>(p.hb + (size_t)(off + cm) * (f * 2) + hoff) = hh;
                        }
                    }
                    // this unit's h is written: the publisher counts it
                    __syncwarp();
                    if (lane == 0) pub_push(pq, PUB_GATEUP, u, fb, abort_flag, p.hdr);
                }
            }
        } else {
            // --------------------------------------------------- down unit
            nch = 2 * nch2;
            const int vd = v - NG;
            const int u = (int)fd_div((uint32_t)vd, p.fd_dpe), rb = vd - u * dpe;
            const int cnt = tab.ucnt[u], off = tab.uoff[u];
            const uint32_t hs = (uint32_t)p.nhs == 1 ? 0u : (hq & 1u);
            const uint32_t huse = (uint32_t)p.nhs == 1 ? hq : (hq >> 1);
            const uint32_t hsa = sbase + p.off_hs + (uint32_t)((qp * p.nhs + (int)hs) * p.hs_bytes);
            const uint32_t csa = hsa + (uint32_t)p.hs_csum;
            good &= tc::mbar_wait(hfull0 + 8u * (uint32_t)(qp * MAX_NHS + hs), huse & 1u, abort_flag, p.hdr);
            if (good) {
                // C1/C2 of the expert's h rows per group: a half-warp per (row, group)
                const int items = cnt * Gf;
                for (int base = 2 * w4; base < items; base += 2 * QW) {
                    const int item = base + (lane >> 4);
                    const bool act = item < items;
                    const int r = act ? (int)fd_div((uint32_t)item, p.fd_gf) : 0, gi = act ? item - r * Gf : 0;
                    const uint4 o = act ? lds128(hsa + (uint32_t)(r * p.hs_stride + gi * 256 + (lane & 15) * 16))
                                        : make_uint4(0u, 0u, 0u, 0u);
                    const float2 c = halfwarp_sum(word_c1c2(o));
                    if (act && (lane & 15) == 0) *reinterpret_cast<float2*>(sm + (csa - sbase) + (r * Gf + gi) * 8) = c;
                }
            }
            bar_sync(qbar, 32 * QW);
            const int col = lane >> 2;
            const uint32_t brow_a = hsa + (uint32_t)((col < cnt ? col : 0) * p.hs_stride);
            const int cr0 = 2 * t4 < cnt ? 2 * t4 : p.cmax, cr1 = 2 * t4 + 1 < cnt ? 2 * t4 + 1 : p.cmax;
            const uint32_t c0_a = csa + (uint32_t)(cr0 * Gf * 8), c1_a = csa + (uint32_t)(cr1 * Gf * 8);
            float acc1[4] = {0.f, 0.f, 0.f, 0.f};  // the second m16 tile (acc: the first)
            for (int ci = 0; ci < 2 * nch2; ++ci) {
                if (ci > 0) good &= wait_chunk(ci);
                const uint32_t slot = slot_of(ci);
                const int m = ci >= nch2 ? 1 : 0, c = ci - m * nch2;
                int l0, n;
                my_groups(min(CHUNK_GROUPS, Gf - c * CHUNK_GROUPS), l0, n);
                if (good && n > 0)
                    consume_range(m ? acc1 : acc, sbase + slot * SLOT_CODE, szbase + slot * SLOT_SZ,
                                  (uint32_t)p.sz2_rs, l0, n, g, t4, c * CHUNK_GROUPS, brow_a, (uint32_t)(col < cnt),
                                  c0_a, c1_a);
                release(slot);
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(hempty0 + 8u * (uint32_t)(qp * MAX_NHS + hs));
            ++hq;
            // the four warps' partial sums of both tiles, added in warp order
            if (w4 != 0) {
                rb4[((w4 - 1) * 2 + 0) * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                rb4[((w4 - 1) * 2 + 1) * 32 + lane] = make_float4(acc1[0], acc1[1], acc1[2], acc1[3]);
            }
            bar_sync(qbar, 32 * QW);
            const bool live = good && !*abort_flag;
            if (w4 == 0) {
#pragma unroll
                for (int i = 0; i < 3; ++i) {
                    const float4 o = rb4[(i * 2 + 0) * 32 + lane], o1 = rb4[(i * 2 + 1) * 32 + lane];
                    acc[0] += o.x;
                    acc[1] += o.y;
                    acc[2] += o.z;
                    acc[3] += o.w;
                    acc1[0] += o1.x;
                    acc1[1] += o1.y;
                    acc1[2] += o1.z;
                    acc1[3] += o1.w;
                }
                if (live) {
                    // y of rows rb*32 + m*16 + g (+ 8) for the assignments of
                    // columns 2 t4 and 2 t4 + 1
                    const int row = rb * RD + g;
#pragma unroll
                    for (int mm = 0; mm < 2; ++mm) {
                        const int cm = 2 * t4 + mm;
                        if (cm < cnt) {
                            float* yr = p.ybuf + (size_t)tab.pa[off + cm] * d;
                            yr[row] = acc[mm];
                            yr[row + 8] = acc[2 + mm];
                            yr[row + 16] = acc1[mm];
                            yr[row + 24] = acc1[2 + mm];
                        }
                    }
                }
            }
            // the unit's y rows are written (both m16 tiles): the publisher
            // counts them and combines completed row blocks
            bar_sync(qbar, 32 * QW);
            if (w4 == 0 && lane == 0 && live) pub_push(pq, PUB_DOWN, u, rb, abort_flag, p.hdr);
        }
        qq += (uint32_t)nch;
        sl += (uint32_t)nch;
        while (sl >= (uint32_t)ns4) sl -= (uint32_t)ns4;
        ++ucount;
    }
    if (w4 == 0 && lane == 0) pub_push(pq, PUB_END, 0, 0, abort_flag, p.hdr);
}

struct FlowLayout {
    int nslot, nhs;
    size_t smem;
    uint32_t off_sz, off_bars, off_desc, off_xb, off_cx, off_hs, off_red, off_tab, off_pub;
    int xb_stride, hs_stride, hs_bytes, hs_csum, cmax;
};

bool plan_flow(int T, int k, int E, int d, int f, int nq, int nhs, FlowLayout* L) {
    if (T < 1 || T > MAX_T || k < 1 || T * k > MAX_R || E < 1 || E > 1024) return false;
    if (d % 256 || f % 256 || f >= 65536) return false;
    FlowLayout l{};
    l.nhs = nhs;
    l.cmax = T;  // an expert has at most T tokens (a token's experts are distinct)
    l.xb_stride = 2 * d + ROW_PAD;
    l.hs_stride = 2 * f + ROW_PAD;
    const int Gd = d / 128, Gf = f / 128;
    l.hs_csum = (int)align_up((size_t)l.cmax * l.hs_stride, 128);
    l.hs_bytes = (int)align_up((size_t)l.hs_csum + (size_t)(l.cmax + 1) * Gf * 8, 128);
    size_t fixed = 0;
    auto take = [&](size_t bytes) {
        const size_t o = fixed;
        fixed = align_up(fixed + bytes, 128);
        return (uint32_t)o;
    };
    const uint32_t o_xb = take((size_t)T * l.xb_stride);
    const uint32_t o_cx = take((size_t)(T + 1) * Gd * 8);
    const uint32_t o_hs = take((size_t)nq * nhs * l.hs_bytes);
    const uint32_t o_red = take((size_t)nq * 2 * 6 * 32 * 16);
    const uint32_t o_tab = take(sizeof(FlowTab));
    const uint32_t o_desc = take((size_t)MAX_SLOTS * 4);
    const uint32_t o_pub = take(sizeof(PubQ));
    const size_t bars = align_up((size_t)8 * (nq * NF + MAX_SLOTS + 2 * nq * MAX_NHS), 128);
    if (fixed + bars + 1024 >= SMEM_LIMIT) return false;
    int nslot = (int)((SMEM_LIMIT - 1024 - fixed - bars) / (SLOT_CODE + SLOT_SZ));
    nslot = std::min(nslot, MAX_SLOTS);
    nslot -= nslot % nq;
    if (nslot < 2 * nq || nslot / nq > NF) return false;
    if ((size_t)T * E * 4 > (size_t)nslot * SLOT_CODE) return false;  // routing scratch in the ring
    const uint32_t ring = (uint32_t)nslot * SLOT_CODE, szs = (uint32_t)nslot * SLOT_SZ;
    const uint32_t base = ring + szs + (uint32_t)bars;
    l.nslot = nslot;
    l.off_sz = ring;
    l.off_bars = ring + szs;
    l.off_xb = base + o_xb;
    l.off_cx = base + o_cx;
    l.off_hs = base + o_hs;
    l.off_red = base + o_red;
    l.off_tab = base + o_tab;
    l.off_desc = base + o_desc;
    l.off_pub = base + o_pub;
    l.smem = 1024 + base + fixed;
    if (l.smem > SMEM_LIMIT) return false;
    *L = l;
    return true;
}

// Scales and zeros reach a slot by TMA (a row of groups a multiple of 16
// bytes) or, when a row of groups fits one chunk, by plain bulk copies.
bool sz_modes(int d, int f, int* m13, int* m2) {
    const int Gd = d / 128, Gf = f / 128;
    *m13 = Gd % 8 == 0 ? SZ_TMA : (Gd < CHUNK_GROUPS ? SZ_BULK : -1);
    *m2 = Gf % 8 == 0 ? SZ_TMA : (Gf < CHUNK_GROUPS ? SZ_BULK : -1);
    return *m13 >= 0 && *m2 >= 0;
}

int flow_nq(int T, int k, int E, int d, int f) {
    (void)T;
    (void)k;
    (void)E;
    (void)d;
    (void)f;
    return 3;
}

bool flow_plan_any(int T, int k, int E, int d, int f, int* nq, FlowLayout* L) {
    *nq = flow_nq(T, k, E, d, f);
    // two h slots per pipeline where the ring keeps at least four slots per pipeline
    return plan_flow(T, k, E, d, f, *nq, 2, L) && L->nslot / *nq >= 4 ? true
                                                                       : plan_flow(T, k, E, d, f, *nq, 1, L);
}

}  // namespace

size_t flow_counter_bytes(int T, int d) {
    return align_up((size_t)2 * MAX_R * 4 + (size_t)T * (d / RD) * 4, 256);
}

bool decode_flow_supported(int T, int k, int E, int d, int f) {
    int m13, m2, nq;
    FlowLayout l;
    return sz_modes(d, f, &m13, &m2) && flow_plan_any(T, k, E, d, f, &nq, &l);
}

cudaError_t launch_decode_flow(const FusedIn& in, cudaStream_t s) {
    const moe_w4_layer& W = *in.L;
    const int E = W.E, d = W.d_model, f = W.d_ff;
    const int G = num_sms();
    int nq, m13, m2;
    FlowLayout l;
    if (!sz_modes(d, f, &m13, &m2) || !flow_plan_any(in.T, in.k, E, d, f, &nq, &l)) return cudaErrorInvalidValue;
    // codes as 32-word lines: gate_up [expert * 2 + (gate, up)][feature][line][32
    // words], box 8 features of both halves; down [row][line][32 words], box 16 rows
    CUtensorMap m13m, m2m;
    const uint64_t d13[4] = {32, (uint64_t)d / 256, (uint64_t)f, (uint64_t)E * 2};
    const uint64_t s13[3] = {128, (uint64_t)d / 2, (uint64_t)f * d / 2};
    const uint32_t b13[4] = {32, LINES, 8, 2};
    if (!make_tensor_map_u32(&m13m, W.w13_q, 4, d13, s13, b13)) return cudaErrorInvalidValue;
    if (!make_tensor_map_3d(&m2m, W.w2_q, 32, (uint64_t)f / 256, (uint64_t)E * d, 128, (uint64_t)f / 2, 32, LINES, 16))
        return cudaErrorInvalidValue;
    CUtensorMap m13s = m13m, m13z = m13m, m2s = m2m, m2z = m2m;
    const uint64_t Gd = (uint64_t)d / 128, Gf = (uint64_t)f / 128;
    auto a16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
    if (m13 == SZ_TMA) {
        const uint64_t dims[3] = {Gd, (uint64_t)f, (uint64_t)E * 2}, str[2] = {Gd * 2, (uint64_t)f * Gd * 2};
        const uint32_t box[3] = {CHUNK_GROUPS, 8, 2};
        if (!make_tensor_map_u16(&m13s, W.w13_s, 3, dims, str, box) ||
            !make_tensor_map_u16(&m13z, W.w13_z, 3, dims, str, box))
            return cudaErrorInvalidValue;
    } else if (!a16(W.w13_s) || !a16(W.w13_z)) {
        return cudaErrorInvalidValue;
    }
    if (m2 == SZ_TMA) {
        const uint64_t dims[2] = {Gf, (uint64_t)E * d}, str[1] = {Gf * 2};
        const uint32_t box[2] = {CHUNK_GROUPS, 16};
        if (!make_tensor_map_u16(&m2s, W.w2_s, 2, dims, str, box) || !make_tensor_map_u16(&m2z, W.w2_z, 2, dims, str, box))
            return cudaErrorInvalidValue;
    } else if (!a16(W.w2_s) || !a16(W.w2_z)) {
        return cudaErrorInvalidValue;
    }
    FlowParams p{};
    p.x = in.x;
    p.logits = in.logits;
    p.w13_s = W.w13_s;
    p.w13_z = W.w13_z;
    p.w2_s = W.w2_s;
    p.w2_z = W.w2_z;
    p.out = in.out;
    p.ids_out = in.ids_out;
    p.hb = reinterpret_cast<uint8_t*>(in.hb);
    p.ybuf = in.ybuf;
    auto* hdr = static_cast<uint32_t*>(in.ws);
    p.hdr = hdr;
    p.ready = hdr + WS_HEADER / 4;
    p.done = p.ready + MAX_R;
    p.ccnt = p.done + MAX_R;
    p.T = in.T;
    p.k = in.k;
    p.E = E;
    p.d = d;
    p.f = f;
    p.nslot = l.nslot;
    p.nhs = l.nhs;
    p.cmax = l.cmax;
    p.off_sz = l.off_sz;
    p.off_bars = l.off_bars;
    p.off_desc = l.off_desc;
    p.off_pub = l.off_pub;
    p.off_xb = l.off_xb;
    p.off_cx = l.off_cx;
    p.off_hs = l.off_hs;
    p.off_red = l.off_red;
    p.off_tab = l.off_tab;
    p.xb_stride = l.xb_stride;
    p.hs_stride = l.hs_stride;
    p.hs_bytes = l.hs_bytes;
    p.hs_csum = l.hs_csum;
    p.sz13_mode = m13;
    p.sz2_mode = m2;
    p.sz13_rs = m13 == SZ_BULK ? (int)Gd * 2 : 16;
    p.sz2_rs = m2 == SZ_BULK ? (int)Gf * 2 : 16;
    p.clear_bytes = (uint32_t)(WS_HEADER + flow_counter_bytes(in.T, d));
    p.fd_gpe = make_fastdiv((uint32_t)(f / FG));
    p.fd_dpe = make_fastdiv((uint32_t)(d / RD));
    p.fd_k = make_fastdiv((uint32_t)in.k);
    p.fd_xw = make_fastdiv((uint32_t)(d / 8));
    p.fd_gf = make_fastdiv((uint32_t)Gf);

    static bool configured[2] = {false, false};
    if (!configured[nq - 3]) {
        cudaError_t e = nq == 3 ? cudaFuncSetAttribute(decode_flow_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       (int)SMEM_LIMIT)
                                : cudaFuncSetAttribute(decode_flow_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       (int)SMEM_LIMIT);
        if (e != cudaSuccess) return e;
        configured[nq - 3] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G);
    cfg.blockDim = dim3(nq == 3 ? FlowShape<3>::NTHREADS : FlowShape<4>::NTHREADS);
    cfg.dynamicSmemBytes = l.smem;
    cfg.stream = s;
    // cooperative (a down unit may wait for a gate_up unit of any CTA, so all
    // must be resident) and, where the driver accepts it, a programmatic
    // dependent of the previous kernel on the stream (the kernel waits for it
    // before touching global memory)
    static int pdl_ok = 1;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_ok ? 2 : 1;
    auto launch = [&]() {
        return nq == 3 ? cudaLaunchKernelEx(&cfg, decode_flow_kernel<3>, m13m, m2m, m13s, m13z, m2s, m2z, p)
                       : cudaLaunchKernelEx(&cfg, decode_flow_kernel<4>, m13m, m2m, m13s, m13z, m2s, m2z, p);
    };
    cudaError_t e = launch();
    if (e != cudaSuccess && pdl_ok) {
        (void)cudaGetLastError();
        pdl_ok = 0;
        cfg.numAttrs = 1;
        e = launch();
    }
    note_launch();
    return e;
}

}  // namespace moe
