// rlk_linear_logprob_static_ws: the full selected-token logprob for callers
// that cannot allocate device memory at call time.
//
// Who needs it.  A rollout engine typically reserves nearly all of the
// GPU's memory for its KV cache when it starts, so a cudaMalloc in the
// middle of serving can fail; and cudaFree synchronises the whole device,
// which stalls every other stream of a latency-bound decode loop.  Such a
// caller has its inputs and outputs already in place but no way to provide
// the extra workspace rlk_linear_logprob asks for.  This entry point takes
// that scratch from a fixed array compiled into the library instead.
//
// The scratch.  `g_static_ws` below is a file-scope __device__ array of
// RLK_STATIC_WS_BYTES (16 MiB).  Every GPU that loads the library holds its
// own copy for as long as the process lives.  Host code cannot use the
// array's name as a device address (on the host it names a stand-in
// object), so the device address is fetched once per device with
// cudaGetSymbolAddress, with that device current, on the first call made
// on that device; make that first call before any stream capture.
//
// Sharing.  All calls on one device use the same array, and it keeps
// whatever the previous call left in it.  Nothing in it has to start at
// zero: the logits stage writes every per-tile pair and target logit that
// the merge stage later reads.  Calls that overlap on the GPU (for example
// issued on two streams without ordering between them) race on the array;
// order them on one stream or synchronise between them.
//
// Everything else -- the kernels, the arithmetic, the bits -- is that of
// rlk_linear_logprob: this call runs the same two stages, rlk_tile_partials
// and rlk_tile_merge, on the built-in array.  It calls no cudaMalloc,
// cudaFree or other allocating routine.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/rlk.h"

namespace {

static __device__ __align__(256) uint8_t g_static_ws[RLK_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_ws_mutex;
void* g_ws_addr[kMaxDevices] = {nullptr};

// Device address of this device's copy of g_static_ws (set up on first use).
rlk_status_t static_ws_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RLK_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return RLK_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    if (g_ws_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || p == nullptr)
            return RLK_ERR_CUDA;
        g_ws_addr[dev] = p;
    }
    *out = g_ws_addr[dev];
    return RLK_OK;
}

}  // namespace

extern "C" rlk_status_t rlk_linear_logprob_static_ws(
    const void* hidden, const void* W, const int32_t* targets, const uint8_t* active_mask,
    int64_t T, int64_t H, int64_t V, int n_shards, float* out_logprob, float* out_lse,
    int32_t* dev_status, rlk_stream_t stream) {
    if (T == 0) return RLK_OK;
    if (T < 0 || T > RLK_MAX_ROWS) return RLK_ERR_INVALID_ARG;
    const size_t need = rlk_workspace_size(T, V, n_shards);
    if (need == 0) {
        // invalid V / n_shards: let the stage report the precise code
        return rlk_tile_partials(hidden, W, targets, active_mask, T, H, V, n_shards, nullptr, 0,
                                 dev_status, stream);
    }
    if (need > RLK_STATIC_WS_BYTES) return RLK_ERR_WORKSPACE;
    if (!out_logprob || !out_lse) return RLK_ERR_INVALID_ARG;
    void* ws = nullptr;
    rlk_status_t s = static_ws_address(&ws);
    if (s != RLK_OK) return s;
    s = rlk_tile_partials(hidden, W, targets, active_mask, T, H, V, n_shards, ws,
                          RLK_STATIC_WS_BYTES, dev_status, stream);
    if (s != RLK_OK) return s;
    return rlk_tile_merge(targets, active_mask, T, V, n_shards, out_logprob, out_lse, ws,
                          RLK_STATIC_WS_BYTES, dev_status, stream);
}
