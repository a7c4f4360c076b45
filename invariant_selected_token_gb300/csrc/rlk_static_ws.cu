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
// on that device.  Under CUDA's default lazy module loading that lookup is
// also what loads this file's module and with it the array's 16 MiB, so the
// first call on each device is the one that can still fail for lack of
// memory: make it at start-up, before the caller reserves the rest of the
// device's memory (a KV cache), and before any stream capture.  The cached
// address belongs to the device's primary context: do not reset the device
// (cudaDeviceReset) or switch to another context between calls.
//
// Sharing.  All calls on one device use the same array, and it keeps
// whatever the previous call left in it.  Nothing in it has to start at
// zero: the logits stage writes every per-tile pair and target logit that
// the merge stage later reads.  Calls that overlap on the GPU (for example
// issued on two streams without ordering between them) race on the array;
// order them on one stream or synchronise between them.
//
// Everything else -- the argument checks, the kernels, the arithmetic, the
// bits -- is that of rlk_linear_logprob: this call is rlk_linear_logprob on
// the built-in array.  It calls no cudaMalloc, cudaFree or other allocating
// routine.
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
    void* ws = nullptr;
    const rlk_status_t s = static_ws_address(&ws);
    if (s != RLK_OK) return s;
    // rlk_linear_logprob checks every argument in its own order and refuses a
    // batch whose workspace exceeds the array with RLK_ERR_WORKSPACE before
    // anything is launched, so both calls report the same codes.
    return rlk_linear_logprob(hidden, W, targets, active_mask, T, H, V, n_shards, out_logprob,
                              out_lse, ws, RLK_STATIC_WS_BYTES, dev_status, stream);
}
