// Token routing for callers that cannot allocate device memory.
//
// mlora_get_routing needs a handle, and mlora_create reserves the whole
// training workspace with cudaMalloc.  Some callers of the routing cannot do
// that: a process whose device memory is already owned by another allocator
// (a framework's caching allocator that reserved the HBM up front), or a
// latency-bound scheduler loop that must not call cudaMalloc/cudaFree,
// which can synchronise the device.  mlora_routing_noalloc serves them: the
// caller passes the inputs and the outputs, and the routing's scratch
// (per-block counts, the padded permutation, the inverse map, the tile and
// chunk bookkeeping) lives in the file-scope array below, which every GPU
// that loads this library holds until the process exits.
//
// Limits: at most MLORA_NOALLOC_MAX_TOKENS tokens and MLORA_NOALLOC_MAX_ADAPTERS
// adapters per call.  The array is shared by every call on a device and keeps
// the previous call's contents; each call re-initialises what must start
// fresh (the padded permutation is reset to -1, every other scratch entry is
// fully rewritten before it is read).  Two calls whose work overlaps on the
// GPU (different streams, or different host threads without ordering) race
// on the array: the caller must order them.
#include <mutex>

#include "internal.h"

namespace {

using namespace mlk;

constexpr int64_t NA_TOKENS = MLORA_NOALLOC_MAX_TOKENS;
constexpr int64_t NA_ADAPTERS = MLORA_NOALLOC_MAX_ADAPTERS;
constexpr int64_t NA_PAD = (NA_TOKENS + (TILE_M - 1) * NA_ADAPTERS + TILE_M - 1) / TILE_M * TILE_M;
constexpr int64_t NA_BLOCKS = (NA_TOKENS + ROUTE_BLOCK - 1) / ROUTE_BLOCK;
constexpr int64_t NA_CHUNKS = NA_PAD / GRAD_CHUNK + NA_ADAPTERS + 1;
// layout of the scratch array, in ints
constexpr int64_t OFF_BLK = 0;                                     // [NA_BLOCKS][n_adapters]
constexpr int64_t OFF_PERM = OFF_BLK + NA_BLOCKS * NA_ADAPTERS;      // [NA_PAD]
constexpr int64_t OFF_INV = OFF_PERM + NA_PAD;                       // [NA_TOKENS]
constexpr int64_t OFF_META = (OFF_INV + NA_TOKENS + 3) / 4 * 4;      // [4]
constexpr int64_t OFF_CHUNKS = OFF_META + 4;                         // int4 [NA_CHUNKS]
constexpr int64_t SCRATCH_INTS = OFF_CHUNKS + 4 * NA_CHUNKS;

constexpr int MAX_DEVICES = 64;

}  // namespace

// The routing scratch (about 0.6 MB).  In host code this name is only a
// stand-in for the device array: its device address is obtained with
// cudaGetSymbolAddress, per device, before any kernel receives it.
static __device__ __align__(256) int g_route_scratch[SCRATCH_INTS];

namespace {

std::mutex g_setup_mu;
int* g_scratch_ptr[MAX_DEVICES] = {nullptr};

// Device address of the scratch array on the current device; resolved on the
// first call made on that device.
cudaError_t scratch_for_current_device(int** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_route_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = static_cast<int*>(p);
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

int mlk_report_error(int code, const char* msg);   // defined with the rest of the C ABI

extern "C" int mlora_routing_noalloc(const int32_t* adapter_ids, int64_t n, int32_t n_adapters,
                                     int32_t* perm, int32_t* seg_off, int32_t* pad_off,
                                     int32_t* tile_ad, void* stream) {
    if (n < 0 || n > NA_TOKENS)
        return mlk_report_error(MLORA_E_ARG, "mlora_routing_noalloc: n must be in 0..MLORA_NOALLOC_MAX_TOKENS");
    if (n_adapters < 1 || n_adapters > NA_ADAPTERS)
        return mlk_report_error(MLORA_E_ARG,
                                     "mlora_routing_noalloc: n_adapters must be in 1..MLORA_NOALLOC_MAX_ADAPTERS");
    if ((n > 0 && (!adapter_ids || !perm)) || !seg_off || !pad_off || !tile_ad)
        return mlk_report_error(MLORA_E_ARG, "mlora_routing_noalloc: NULL input or output");
    int* base = nullptr;
    cudaError_t e = scratch_for_current_device(&base);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return mlk_report_error(MLORA_E_CUDA, "mlora_routing_noalloc: cannot resolve the scratch array");
    }
    const int64_t busy = n < n_adapters ? n : n_adapters;
    RouteBufs rb;
    rb.blk_cnt = base + OFF_BLK;
    rb.perm_pad = base + OFF_PERM;
    rb.inv = base + OFF_INV;
    rb.meta = base + OFF_META;
    rb.chunks = reinterpret_cast<int4*>(base + OFF_CHUNKS);
    rb.seg_off = seg_off;
    rb.pad_off = pad_off;
    rb.tile_ad = tile_ad;
    rb.max_pad = (int)((n + (TILE_M - 1) * busy + TILE_M - 1) / TILE_M * TILE_M);
    rb.max_tiles = (int)(n / TILE_M) + n_adapters + 1;
    rb.max_chunks = (int)NA_CHUNKS;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int64_t launches = 0;
    launch_routing(adapter_ids, n, n_adapters, rb, nullptr, nullptr, s, &launches);
    if (n > 0) launch_compact_perm(rb, n_adapters, perm, s, &launches);
    e = cudaGetLastError();
    if (e != cudaSuccess) return mlk_report_error(MLORA_E_CUDA, cudaGetErrorString(e));
    return MLORA_OK;
}
