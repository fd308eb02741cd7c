// The C ABI declared in include/moe_w4.h: argument checks, workspace carving,
// regime choice and the launch chains.  No allocation, no host sync (except
// moe_get_device_error).
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "internal.h"
#include "moe_w4.h"

namespace moe {

int num_sms() {
    static int n = 0;
    if (n == 0) {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
            n = v;
        else
            return 1;
    }
    return n;
}

static std::atomic<uint64_t> g_launches{0};
void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

namespace {

// Stage events of moe_profile_stages (per host thread).
struct StageProfile {
    cudaEvent_t* events = nullptr;
    int32_t capacity = 0;
    int32_t* cursor = nullptr;
};
thread_local StageProfile g_prof;

// Records the stage marks of one call: mark(i) for i in 0..5.
struct StageMarks {
    cudaEvent_t* ev = nullptr;
    cudaStream_t s;
    explicit StageMarks(cudaStream_t st) : s(st) {
        if (g_prof.events && g_prof.cursor && *g_prof.cursor + 6 <= g_prof.capacity) {
            ev = g_prof.events + *g_prof.cursor;
            *g_prof.cursor += 6;
        }
    }
    void mark(int i) {
        if (!ev) return;
        // inside a stream capture an external record becomes an event-record
        // node of the graph, so replays time the stages too; outside a capture
        // a plain record.  A failed record must not surface as a launch error.
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaStreamIsCapturing(s, &cs);
        const cudaError_t e = (cs == cudaStreamCaptureStatusActive)
                                  ? cudaEventRecordWithFlags(ev[i], s, cudaEventRecordExternal)
                                  : cudaEventRecord(ev[i], s);
        if (e != cudaSuccess) (void)cudaGetLastError();
    }
};

constexpr int DECODE_MAX_ROWS = 64;  // R = T*k at or below which the GEMV regime runs

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

enum class Regime { Auto, Decode, Prefill };

Regime regime_override() {
    const char* v = std::getenv("MOE_W4_REGIME");
    if (!v) return Regime::Auto;
    if (!std::strcmp(v, "decode")) return Regime::Decode;
    if (!std::strcmp(v, "prefill")) return Regime::Prefill;
    return Regime::Auto;
}

moe_status_t check_layer(const moe_w4_layer* L) {
    if (!L) return MOE_ERR_INVALID_ARG;
    if (L->E < 1 || L->E > 1024 || L->d_model <= 0 || L->d_ff <= 0) return MOE_ERR_INVALID_ARG;
    if (L->group != 128) return MOE_ERR_UNSUPPORTED;
    if (L->d_model % 256 || L->d_ff % 256 || L->d_model > 16384 || L->d_ff > 16384) return MOE_ERR_UNSUPPORTED;
    const void* ps[6] = {L->w13_q, L->w13_s, L->w13_z, L->w2_q, L->w2_s, L->w2_z};
    for (const void* p : ps) {
        if (!p) return MOE_ERR_INVALID_ARG;
        if (!aligned16(p)) return MOE_ERR_MISALIGNED;
    }
    return MOE_OK;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Bump allocator over a caller-provided workspace (256-byte aligned regions).
struct Carver {
    unsigned char* base;
    size_t off;
    explicit Carver(void* b) : base(static_cast<unsigned char*>(b)), off(WS_HEADER) {}
    template <class T>
    T* take(size_t count) {
        T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
        off = align_up(off + count * sizeof(T), 256);
        return p;
    }
};

struct PermScratch {
    DevPlan* plan;
    int32_t* uniq;
    Tile* tiles;
    int32_t* blockcnt;
};

PermScratch carve_perm(Carver& c, int R, int E) {
    PermScratch s;
    s.plan = c.take<DevPlan>(1);
    s.uniq = c.take<int32_t>(E);
    s.tiles = c.take<Tile>(tc_max_tiles(R, E));
    s.blockcnt = c.take<int32_t>(align_blockcnt_bytes(R, E) / sizeof(int32_t));
    return s;
}

struct LayerWs {
    PermScratch ps;
    int32_t *ids, *counts, *offsets, *sorted, *inv;
    float* w;
    float* h;             // fp32 [R][f] (GEMV regime) or fp16 [R][f] (tensor-core regime)
    uint16_t *x_perm, *y_perm;  // fp16 [R][d] (tensor-core regime)
    size_t bytes;
};

LayerWs carve_layer(void* ws, int T, int k, int E, int d, int f) {
    const int R = T * k;
    Carver c(ws);
    LayerWs l;
    l.ps = carve_perm(c, R, E);
    l.ids = c.take<int32_t>(R);
    l.w = c.take<float>(R);
    l.counts = c.take<int32_t>(E);
    l.offsets = c.take<int32_t>(E + 1);
    l.sorted = c.take<int32_t>(R);
    l.inv = c.take<int32_t>(R);
    l.h = c.take<float>((size_t)R * f);
    l.x_perm = c.take<uint16_t>((size_t)R * d);
    l.y_perm = c.take<uint16_t>((size_t)R * d);
    l.bytes = c.off;
    return l;
}

struct FfnWs {
    PermScratch ps;
    float* h;       // fp32 [R][f] (GEMV regime) or fp16 [R][f] (tensor-core regime)
    uint16_t* x16;  // fp16 copy of x_perm (tensor-core regime)
    size_t bytes;
};

FfnWs carve_ffn(void* ws, int R, int E, int d, int f) {
    Carver c(ws);
    FfnWs w;
    w.ps = carve_perm(c, R, E);
    w.h = c.take<float>((size_t)R * f);
    w.x16 = c.take<uint16_t>((size_t)R * d);
    w.bytes = c.off;
    return w;
}

// The decode regime of moe_layer_forward runs as one kernel when the shape
// allows (the grid-barrier kernel), else as the route/permute/GEMV chain;
// MOE_W4_DECODE_KERNEL=split forces the chain.
enum class DecodeKernel { Fused, Split };

DecodeKernel pick_decode_kernel(int T, int k, const moe_w4_layer* L) {
    const char* v = std::getenv("MOE_W4_DECODE_KERNEL");
    if (v && !std::strcmp(v, "split")) return DecodeKernel::Split;
    if (decode_fused_supported(T, k, L->E, L->d_model, L->d_ff)) return DecodeKernel::Fused;
    return DecodeKernel::Split;
}

bool choose_decode(int R, int T, const moe_w4_layer* L) {
    GemvShape sh{L->E, L->d_model, L->d_ff, R, std::min(R, L->E)};
    const Regime rg = regime_override();
    if (rg == Regime::Prefill) return false;
    if (!gemv_supported(sh, T)) return false;
    if (rg == Regime::Decode) return true;
    return R <= DECODE_MAX_ROWS;
}

uint32_t* err_word(void* ws) { return &static_cast<WsHeader*>(ws)->err; }

GemvIn gemv_in(const moe_w4_layer* L) {
    GemvIn in{};
    in.w13_q = L->w13_q;
    in.w13_s = L->w13_s;
    in.w13_z = L->w13_z;
    in.w2_q = L->w2_q;
    in.w2_s = L->w2_s;
    in.w2_z = L->w2_z;
    return in;
}

TcIn tc_in(const moe_w4_layer* L) {
    TcIn in{};
    in.w13_q = L->w13_q;
    in.w13_s = L->w13_s;
    in.w13_z = L->w13_z;
    in.w2_q = L->w2_q;
    in.w2_s = L->w2_s;
    in.w2_z = L->w2_z;
    return in;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_str(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_DEVICE_RANGE: return "MOE_ERR_DEVICE_RANGE";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
        case MOE_ERR_F16_RANGE: return "MOE_ERR_F16_RANGE";
        case MOE_ERR_SCRATCH_LIMIT: return "MOE_ERR_SCRATCH_LIMIT";
        case MOE_ERR_CAPTURE: return "MOE_ERR_CAPTURE";
    }
    return "MOE_ERR_UNKNOWN";
}

const char* moe_version(void) { return "moe_w4 1.0 sm_103a"; }

moe_status_t moe_route_topk(const float* logits, int32_t T, int32_t E, int32_t k, int32_t* topk_ids,
                            float* topk_w, cudaStream_t stream) {
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
    if ((int64_t)T * k >= (int64_t)1 << 31 || (int64_t)T * E >= (int64_t)1 << 31) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    if (!aligned16(logits) || !aligned16(topk_ids) || !aligned16(topk_w)) return MOE_ERR_MISALIGNED;
    return cuda_status(launch_route_topk(logits, T, E, k, topk_ids, topk_w, stream));
}

size_t moe_permute_workspace_size(int32_t T, int32_t k, int32_t E) {
    if (T < 0 || k < 1 || E < 1) return 0;
    Carver c(nullptr);
    carve_perm(c, T * k, E);
    return c.off;
}

moe_status_t moe_permute(const int32_t* topk_ids, int32_t T, int32_t k, int32_t E, const void* x_bf16,
                         int32_t d, int32_t* counts, int32_t* offsets, int32_t* sorted, int32_t* inv,
                         void* x_perm_bf16, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
    if ((int64_t)T * k >= (int64_t)1 << 31) return MOE_ERR_INVALID_ARG;
    if (!counts || !offsets || !workspace) return MOE_ERR_INVALID_ARG;
    if (x_perm_bf16 && (!x_bf16 || d <= 0 || d % 8)) return MOE_ERR_INVALID_ARG;
    const void* ps[] = {topk_ids, counts, offsets, sorted, inv, x_bf16, x_perm_bf16, workspace};
    for (const void* p : ps)
        if (p && !aligned16(p)) return MOE_ERR_MISALIGNED;
    if (T > 0 && (!topk_ids || !sorted || !inv)) return MOE_ERR_INVALID_ARG;
    if (workspace_bytes < moe_permute_workspace_size(T, k, E)) return MOE_ERR_WORKSPACE;
    const int R = T * k;
    Carver c(workspace);
    PermScratch s = carve_perm(c, R, E);
    AlignOut o{counts, offsets, sorted, inv, s.uniq, s.tiles, s.plan,
               static_cast<uint16_t*>(x_perm_bf16), 0, s.blockcnt, err_word(workspace)};
    return cuda_status(launch_align(topk_ids, T, k, E, static_cast<const uint16_t*>(x_bf16), d, o, stream));
}

size_t moe_expert_ffn_workspace_size(const moe_w4_layer* L, int32_t R) {
    if (check_layer(L) != MOE_OK || R < 0) return 0;
    return carve_ffn(nullptr, R, L->E, L->d_model, L->d_ff).bytes;
}

moe_status_t moe_expert_ffn_w4a16(const moe_w4_layer* L, const void* x_perm_bf16, const int32_t* offsets,
                                  int32_t R, const float* row_w, void* y_perm_bf16, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream) {
    moe_status_t st = check_layer(L);
    if (st != MOE_OK) return st;
    if (R < 0 || !offsets || !workspace) return MOE_ERR_INVALID_ARG;
    if (R > 0 && (!x_perm_bf16 || !y_perm_bf16)) return MOE_ERR_INVALID_ARG;
    const void* ps[] = {x_perm_bf16, offsets, row_w, y_perm_bf16, workspace};
    for (const void* p : ps)
        if (p && !aligned16(p)) return MOE_ERR_MISALIGNED;
    if (workspace_bytes < moe_expert_ffn_workspace_size(L, R)) return MOE_ERR_WORKSPACE;
    if (R == 0) return MOE_OK;
    const int E = L->E, d = L->d_model, f = L->d_ff;
    FfnWs w = carve_ffn(workspace, R, E, d, f);
    uint32_t* err = err_word(workspace);
    cudaError_t ce = launch_plan_from_offsets(offsets, E, w.ps.uniq, w.ps.tiles, w.ps.plan, stream);
    if (ce != cudaSuccess) return MOE_ERR_CUDA;
    if (choose_decode(R, R, L)) {
        GemvShape sh{E, d, f, R, std::min(R, E)};
        GemvIn in = gemv_in(L);
        in.offsets = offsets;
        in.uniq = w.ps.uniq;
        in.plan = w.ps.plan;
        in.sorted = nullptr;
        in.k = 1;
        in.x = static_cast<const uint16_t*>(x_perm_bf16);
        in.h = w.h;
        in.y_perm = static_cast<uint16_t*>(y_perm_bf16);
        in.row_w = row_w;
        in.err = err;
        ce = launch_gemv_gateup(sh, in, stream);
        if (ce == cudaSuccess) ce = launch_gemv_down(sh, in, stream);
        return cuda_status(ce);
    }
    if (!tc_supported(E, d, f)) return MOE_ERR_UNSUPPORTED;
    ce = launch_bf16_to_f16(static_cast<const uint16_t*>(x_perm_bf16), w.x16, (size_t)R * d, err, stream);
    if (ce != cudaSuccess) return MOE_ERR_CUDA;
    TcIn in = tc_in(L);
    in.tiles = w.ps.tiles;
    in.plan = w.ps.plan;
    in.x16 = w.x16;
    in.h16 = reinterpret_cast<uint16_t*>(w.h);
    in.y_out = static_cast<uint16_t*>(y_perm_bf16);
    in.y_f16 = 0;
    in.row_w = row_w;
    in.err = err;
    ce = launch_tc_gateup(E, d, f, R, in, stream);
    if (ce == cudaSuccess) ce = launch_tc_down(E, d, f, R, in, stream);
    return cuda_status(ce);
}

moe_status_t moe_combine(const void* y_perm_bf16, const int32_t* inv, const float* topk_w, int32_t T,
                         int32_t k, int32_t d, void* out_bf16, cudaStream_t stream) {
    if (T < 0 || k < 1 || d <= 0 || d % 8) return MOE_ERR_INVALID_ARG;
    if ((int64_t)T * k >= (int64_t)1 << 31) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!y_perm_bf16 || !inv || !topk_w || !out_bf16) return MOE_ERR_INVALID_ARG;
    if (!aligned16(y_perm_bf16) || !aligned16(inv) || !aligned16(topk_w) || !aligned16(out_bf16))
        return MOE_ERR_MISALIGNED;
    return cuda_status(launch_combine(static_cast<const uint16_t*>(y_perm_bf16), false, inv, topk_w, T, k, d,
                                      static_cast<uint16_t*>(out_bf16), stream));
}

size_t moe_layer_workspace_size(const moe_w4_layer* L, int32_t T, int32_t k) {
    if (check_layer(L) != MOE_OK || T < 0 || k < 1) return 0;
    return carve_layer(nullptr, T, k, L->E, L->d_model, L->d_ff).bytes;
}

moe_status_t moe_layer_forward(const moe_w4_layer* L, const void* x_bf16, const float* logits, int32_t T,
                               int32_t k, void* out_bf16, int32_t* topk_ids_out, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream) {
    moe_status_t st = check_layer(L);
    if (st != MOE_OK) return st;
    if (T < 0 || k < 1 || k > L->E) return MOE_ERR_INVALID_ARG;
    if ((int64_t)T * k >= (int64_t)1 << 31 || (int64_t)T * L->E >= (int64_t)1 << 31) return MOE_ERR_INVALID_ARG;
    if (!workspace) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x_bf16 || !logits || !out_bf16)) return MOE_ERR_INVALID_ARG;
    const void* ps[] = {x_bf16, logits, out_bf16, topk_ids_out, workspace};
    for (const void* p : ps)
        if (p && !aligned16(p)) return MOE_ERR_MISALIGNED;
    if (workspace_bytes < moe_layer_workspace_size(L, T, k)) return MOE_ERR_WORKSPACE;
    if (T == 0) return MOE_OK;

    const int E = L->E, d = L->d_model, f = L->d_ff, R = T * k;
    LayerWs w = carve_layer(workspace, T, k, E, d, f);
    uint32_t* err = err_word(workspace);
    int32_t* ids = topk_ids_out ? topk_ids_out : w.ids;
    const bool decode = choose_decode(R, T, L);
    if (!decode && !tc_supported(E, d, f)) return MOE_ERR_UNSUPPORTED;

    StageMarks marks(stream);
    marks.mark(0);
    const DecodeKernel dk = decode ? pick_decode_kernel(T, k, L) : DecodeKernel::Split;
    if (dk != DecodeKernel::Split) {
        // one kernel for the whole layer: every later stage mark sits after it
        FusedIn fi{L,
                   static_cast<const uint16_t*>(x_bf16),
                   logits,
                   T,
                   k,
                   static_cast<uint16_t*>(out_bf16),
                   topk_ids_out,
                   reinterpret_cast<uint16_t*>(w.h),
                   workspace};
        const cudaError_t fe = launch_decode_fused(fi, stream);
        for (int i = 1; i <= 5; ++i) marks.mark(i);
        return cuda_status(fe);
    }
    cudaError_t ce = launch_route_topk(logits, T, E, k, ids, w.w, stream);
    if (ce != cudaSuccess) return MOE_ERR_CUDA;
    marks.mark(1);
    AlignOut o{w.counts, w.offsets, w.sorted, w.inv, w.ps.uniq, w.ps.tiles, w.ps.plan,
               decode ? nullptr : w.x_perm, 1, w.ps.blockcnt, err};
    ce = launch_align(ids, T, k, E, static_cast<const uint16_t*>(x_bf16), d, o, stream);
    if (ce != cudaSuccess) return MOE_ERR_CUDA;
    marks.mark(2);

    if (decode) {
        GemvShape sh{E, d, f, R, std::min(R, E)};
        GemvIn in = gemv_in(L);
        in.offsets = w.offsets;
        in.uniq = w.ps.uniq;
        in.plan = w.ps.plan;
        in.sorted = w.sorted;
        in.k = k;
        in.x = static_cast<const uint16_t*>(x_bf16);
        in.h = w.h;
        in.out = static_cast<uint16_t*>(out_bf16);
        in.topk_w = w.w;
        in.inv = w.inv;
        in.T = T;
        in.err = err;
        ce = launch_gemv_gateup(sh, in, stream);
        marks.mark(3);
        if (ce == cudaSuccess) ce = launch_gemv_down(sh, in, stream);
        marks.mark(4);
        marks.mark(5);
        return cuda_status(ce);
    }
    TcIn in = tc_in(L);
    in.tiles = w.ps.tiles;
    in.plan = w.ps.plan;
    in.x16 = w.x_perm;
    in.h16 = reinterpret_cast<uint16_t*>(w.h);
    in.y_out = w.y_perm;
    in.y_f16 = 1;
    in.row_w = nullptr;
    in.err = err;
    ce = launch_tc_gateup(E, d, f, R, in, stream);
    marks.mark(3);
    if (ce == cudaSuccess) ce = launch_tc_down(E, d, f, R, in, stream);
    marks.mark(4);
    if (ce == cudaSuccess) ce = launch_combine(w.y_perm, true, w.inv, w.w, T, k, d, static_cast<uint16_t*>(out_bf16), stream);
    marks.mark(5);
    return cuda_status(ce);
}

moe_status_t moe_profile_stages(cudaEvent_t* events, int32_t capacity, int32_t* cursor) {
    if (events && (!cursor || capacity < 0)) return MOE_ERR_INVALID_ARG;
    g_prof.events = events;
    g_prof.capacity = events ? capacity : 0;
    g_prof.cursor = events ? cursor : nullptr;
    return MOE_OK;
}

uint64_t moe_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

moe_status_t moe_get_device_error(void* workspace, cudaStream_t stream) {
    if (!workspace) return MOE_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
    uint32_t e = 0;
    if (cudaMemcpy(&e, workspace, sizeof(e), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (e == 0) return MOE_OK;
    // the header: the error word and whatever a call that gave up left behind
    // (the grid-barrier kernel's arrival counter)
    if (cudaMemset(workspace, 0, WS_HEADER) != cudaSuccess) return MOE_ERR_CUDA;
    if (e & ERRBIT_TIMEOUT) return MOE_ERR_TIMEOUT;
    if (e & ERRBIT_RANGE) return MOE_ERR_DEVICE_RANGE;
    return MOE_ERR_F16_RANGE;
}

}  // extern "C"
