// moe_permute_noalloc: the permutation stage for callers that cannot allocate
// device memory.
//
// Some callers have no way to hand the library a workspace: a host runtime
// that plans all of its device memory up front and refuses any allocation
// after start-up (a fixed-pool inference server), code that runs where CUDA
// API calls that allocate are not allowed (a host function enqueued with
// cudaLaunchHostFunc), or a plain C program that only owns the buffers of its
// inputs and outputs.  For them this entry point keeps its scratch in a
// fixed-size array in device global memory that is part of the library
// image itself, so nothing is allocated or freed at call time.
//
// Properties of that array (MOE_NOALLOC_SCRATCH_BYTES, see include/moe_w4.h):
//   * every GPU that loads the library holds it until the process exits;
//   * every call on a device shares it and it keeps the last call's contents;
//     the permutation rewrites every byte it later reads (per-block counts,
//     plan, expert list, tiles), so nothing has to start at zero;
//   * calls that overlap on the GPU (different streams, or different host
//     threads on one device) race on it: serialise them.
// The array's name is only a host-side stand-in for the device copy, so the
// device address is looked up once per device with cudaGetSymbolAddress (on
// the first call made with that device current) and cached.  Make that first
// call before any stream capture: a first call on a capturing stream returns
// MOE_ERR_CAPTURE and does nothing.
#include <mutex>

#include "internal.h"
#include "moe_w4.h"

namespace moe {
namespace {

constexpr int NOALLOC_MAX_DEVICES = 64;

static __device__ __align__(256) unsigned char g_permute_scratch[MOE_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_dev[NOALLOC_MAX_DEVICES] = {};

// Device address of the scratch array on the current device (looked up once).
// The lookup may load the library's device code, which a stream capture in
// progress would not allow (it could invalidate the caller's capture), so a
// first call made on a capturing stream is refused with MOE_ERR_CAPTURE before
// any CUDA call other than the capture query.
moe_status_t scratch_address(cudaStream_t stream, unsigned char** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NOALLOC_MAX_DEVICES) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_dev[dev]) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return MOE_ERR_CUDA;
        if (cs != cudaStreamCaptureStatusNone) return MOE_ERR_CAPTURE;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        g_scratch_dev[dev] = p;
    }
    *out = static_cast<unsigned char*>(g_scratch_dev[dev]);
    return MOE_OK;
}

// Layout inside the array: error word (never read back here), plan, expert
// list, tiles, per-block counts -- 256-byte aligned regions.
struct NoallocLayout {
    size_t plan, uniq, tiles, blockcnt, end;
};

NoallocLayout layout(int R, int E) {
    NoallocLayout l;
    size_t off = WS_HEADER;
    l.plan = off;
    off = align_up(off + sizeof(DevPlan), 256);
    l.uniq = off;
    off = align_up(off + (size_t)E * sizeof(int32_t), 256);
    l.tiles = off;
    off = align_up(off + (size_t)tc_max_tiles(R, E) * sizeof(Tile), 256);
    l.blockcnt = off;
    off = align_up(off + align_blockcnt_bytes(R, E), 256);
    l.end = off;
    return l;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_permute_noalloc(const int32_t* topk_ids, int32_t T, int32_t k, int32_t E,
                                            const void* x_bf16, int32_t d, int32_t* counts, int32_t* offsets,
                                            int32_t* sorted, int32_t* inv, void* x_perm_bf16,
                                            cudaStream_t stream) {
    using namespace moe;
    if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
    if ((int64_t)T * k > MOE_NOALLOC_MAX_ROWS) return MOE_ERR_SCRATCH_LIMIT;
    if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
    if (x_perm_bf16 && (!x_bf16 || d <= 0 || d % 8)) return MOE_ERR_INVALID_ARG;
    const void* ps[] = {topk_ids, counts, offsets, sorted, inv, x_bf16, x_perm_bf16};
    for (const void* p : ps)
        if (p && !aligned16(p)) return MOE_ERR_MISALIGNED;
    if (T > 0 && (!topk_ids || !sorted || !inv)) return MOE_ERR_INVALID_ARG;
    const int R = T * k;
    const NoallocLayout l = layout(R, E);
    if (l.end > sizeof(g_permute_scratch)) return MOE_ERR_SCRATCH_LIMIT;
    unsigned char* base = nullptr;
    moe_status_t st = scratch_address(stream, &base);
    if (st != MOE_OK) return st;
    AlignOut o{counts,
               offsets,
               sorted,
               inv,
               reinterpret_cast<int32_t*>(base + l.uniq),
               reinterpret_cast<Tile*>(base + l.tiles),
               reinterpret_cast<DevPlan*>(base + l.plan),
               static_cast<uint16_t*>(x_perm_bf16),
               0,
               reinterpret_cast<int32_t*>(base + l.blockcnt),
               reinterpret_cast<uint32_t*>(base)};
    return launch_align(topk_ids, T, k, E, static_cast<const uint16_t*>(x_bf16), d, o, stream) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}
