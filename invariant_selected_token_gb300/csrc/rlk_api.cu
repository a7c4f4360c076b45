// Host side of the C-ABI (include/rlk.h): argument checks, the canonical
// tile tree on the host, workspace layout, TMA descriptor encoding and kernel
// dispatch.  Strict mode only: anything unsupported is refused with a
// status code, nothing falls back to another path ("vLLM RL-Kernel v0.1.0",
// strict path; the vime ablation-matrix issue, "strict: unsupported 时 fail
// closed").
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "rlk_internal.h"

#ifndef RLK_GIT_REV
#define RLK_GIT_REV "unknown"
#endif
#ifndef RLK_NVCC_VERSION
#define RLK_NVCC_VERSION "unknown"
#endif

namespace {

using rlk::kTileM;
using rlk::kTileN;
using rlk::kVocabTile;

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    int cc = 0;             // 10 * major + minor
    int mat_ctas_per_sm[2] = {0, 0};  // materialised-logits kernel, fp32 / bf16
    // backward: grad_hidden's split sum runs on this stream beside the grad_W
    // GEMM (created at the first backward that computes both); `side_mutex`
    // keeps one call's record / wait sequence on the two events whole
    cudaStream_t side = nullptr;
    cudaEvent_t ev_split = nullptr, ev_sum = nullptr;
    std::mutex side_mutex;
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int64_t n_tiles_of(int64_t V) { return (V + kVocabTile - 1) / kVocabTile; }

int log2_exact(int n) {
    int d = 0;
    while ((1 << d) < n) ++d;
    return (1 << d) == n ? d : -1;
}

int tree_depth(int64_t n_tiles) {
    int d = 0;
    while ((int64_t(1) << d) < n_tiles) ++d;
    return d;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Tile range [first, first + count) of node `index` at depth `depth` of the
// recursive bisection of [0, n_tiles) (the lower half takes the extra tile).
bool tree_node(int64_t n_tiles, int depth, int index, int64_t* first, int64_t* count) {
    int64_t f = 0, k = n_tiles;
    for (int b = depth - 1; b >= 0; --b) {
        if (k < 2) return false;
        const int64_t left = (k + 1) / 2;
        if ((index >> b) & 1) {
            f += left;
            k -= left;
        } else {
            k = left;
        }
    }
    *first = f;
    *count = k;
    return k >= 1;
}

struct Layout {
    size_t partials, tgt, records, total;
};

Layout layout_of(int64_t T, int64_t V, int n_shards) {
    Layout l;
    l.partials = 0;
    l.tgt = align256(size_t(T) * size_t(n_tiles_of(V)) * sizeof(float2));
    l.records = l.tgt + align256(size_t(T) * sizeof(float));
    l.total = l.records + align256(size_t(T) * size_t(n_shards) * sizeof(rlk_partial_t));
    return l;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

rlk_status_t shard_check(int64_t V, int n_shards) {
    if (V < 1) return RLK_ERR_INVALID_ARG;
    if (V > RLK_MAX_VOCAB) return RLK_ERR_UNSUPPORTED;
    const int d = log2_exact(n_shards);
    if (n_shards < 1 || n_shards > RLK_MAX_SHARDS || d < 0) return RLK_ERR_UNSUPPORTED;
    if (int64_t(n_shards) > n_tiles_of(V)) return RLK_ERR_UNSUPPORTED;
    return RLK_OK;
}

// Device of the calling thread: must be sm_103.  RLK_TEST_DEVICE_CC
// (e.g. "100") makes the check see another compute capability, so the
// refusal path can be exercised on real hardware without launching anything.
rlk_status_t device_check(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RLK_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return RLK_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& st = g_dev[dev];
    if (!st.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return RLK_ERR_CUDA;
        st.cc = major * 10 + minor;
        st.sm_count = sms;
        if (st.cc == 103) {
            if (rlk::prepare_tile_partials_kernels() != cudaSuccess) return RLK_ERR_CUDA;
            if (rlk::prepare_gemm_kernels() != cudaSuccess) return RLK_ERR_CUDA;
            if (rlk::prepare_mat_kernels(st.mat_ctas_per_sm) != cudaSuccess) return RLK_ERR_CUDA;
            if (rlk::prepare_tree_kernels() != cudaSuccess) return RLK_ERR_CUDA;
        }
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return RLK_ERR_CUDA;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        st.ready = true;
    }
    int cc = st.cc;
    if (const char* fake = std::getenv("RLK_TEST_DEVICE_CC")) cc = std::atoi(fake);
    if (cc != 103) return RLK_ERR_UNSUPPORTED;
    *out = &st;
    return RLK_OK;
}

// bf16 [rows][inner] row-major, boxes of 64 (inner) x box_rows, 128-byte swizzle.
rlk_status_t encode_bf16_map(CUtensorMap* map, const void* base, int64_t inner, int64_t rows,
                             uint32_t box_rows) {
    const cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(inner) * 2};
    const cuuint32_t box[2] = {cuuint32_t(rlk::kBlockK), box_rows};
    const cuuint32_t elem[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                                dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? RLK_OK : RLK_ERR_CUDA;
}

// RLK_TEST_DROP_STAGE=1 (the logits kernel) or 2 (the grad_hidden GEMM): CTA
// 0's producer skips its first pipeline stage, so its MMA wait runs out
// (bounded) and the kernel reports RLK_ERR_TIMEOUT -- the failure-detection
// tests' way to exercise the give-up path.
int test_drop_stage_code() {
    const char* f = std::getenv("RLK_TEST_DROP_STAGE");
    return f ? std::atoi(f) : 0;
}
bool test_drop_stage() { return test_drop_stage_code() == 1; }

// logits_out (with its row stride ld_logits): the saving forward, which
// also stores every row's fp32 logits; dbg: the debug dump (logits only).
rlk_status_t run_tile_partials(const void* hidden, const void* W, const int32_t* targets,
                               const uint8_t* active, int64_t T, int64_t H, int64_t V_local,
                               int64_t v_offset, float2* partials, float* tgt, float* dbg,
                               int32_t* status, cudaStream_t stream, const DeviceState* dev,
                               float* logits_out = nullptr, int64_t ld_logits = 0) {
    CUtensorMap map_h, map_w;
    // one token tile: load only the rows that exist (rounded up to a whole
    // 8-row swizzle atom); the MMA's other accumulator rows are discarded
    const int a_rows = T >= kTileM ? kTileM : int((T + 7) / 8 * 8);
    rlk_status_t s = encode_bf16_map(&map_h, hidden, H, T, uint32_t(a_rows));
    if (s != RLK_OK) return s;
    s = encode_bf16_map(&map_w, W, H, V_local, kTileN);
    if (s != RLK_OK) return s;
    rlk::TilePartialsArgs a;
    a.targets = targets;
    a.active = active;
    a.partials = partials;
    a.tgt_logit = tgt;
    a.dbg_logits = dbg;
    a.status = status;
    a.v_offset = v_offset;
    a.T = int(T);
    a.V_local = int(V_local);
    a.n_tiles = int(n_tiles_of(V_local));
    a.k_blocks = int(H / rlk::kBlockK);
    a.a_box_rows = a_rows;
    a.test_drop_stage = test_drop_stage() ? 1 : 0;
    a.lse = nullptr;
    a.grad = nullptr;
    a.G = nullptr;
    a.ldG = 0;
    a.V_total = V_local;
    a.logits_out = logits_out;
    a.ld_logits = ld_logits;
    const int epi = dbg != nullptr ? rlk::kEpiDebugLogits
                    : logits_out != nullptr ? rlk::kEpiSave
                                            : rlk::kEpiPartials;
    return rlk::launch_tile_partials(map_h, map_w, a, epi, dev->sm_count, stream) == cudaSuccess
               ? RLK_OK
               : RLK_ERR_CUDA;
}

// bf16 [rows][inner] row-major with row stride `stride_elems`, 64 x 64 boxes
// (MN-major GEMM operands: the inner dimension is M or N, rows are K).
rlk_status_t encode_bf16_mn_map(CUtensorMap* map, const void* base, int64_t inner, int64_t rows,
                                int64_t stride_elems) {
    const cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(stride_elems) * 2};
    const cuuint32_t box[2] = {64, 64};
    const cuuint32_t elem[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                                dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? RLK_OK : RLK_ERR_CUDA;
}

// K-major bf16 operand [rows][inner] with row stride `stride_elems`, boxes 64 x box_rows.
rlk_status_t encode_bf16_k_map(CUtensorMap* map, const void* base, int64_t inner, int64_t rows,
                               int64_t stride_elems, uint32_t box_rows) {
    const cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(stride_elems) * 2};
    const cuuint32_t box[2] = {cuuint32_t(rlk::kBlockK), box_rows};
    const cuuint32_t elem[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                                dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? RLK_OK : RLK_ERR_CUDA;
}

constexpr int kGradHiddenSplits = 8;

int64_t grad_ld(int64_t V) { return (V + 7) / 8 * 8; }

struct BackwardLayout {
    size_t G, parts, total;
};

BackwardLayout backward_layout_of(int64_t T, int64_t H, int64_t V) {
    BackwardLayout l;
    l.G = 0;
    l.parts = align256(size_t(T) * size_t(grad_ld(V)) * 2);
    l.total = l.parts + align256(size_t(kGradHiddenSplits) * size_t(T) * size_t(H) * 4);
    return l;
}

rlk_status_t common_checks(const void* hidden, const void* W, const int32_t* targets, int64_t T,
                           int64_t H) {
    if (T < 0 || T > RLK_MAX_ROWS) return RLK_ERR_INVALID_ARG;
    if (T > 0 && (!hidden || !W || !targets)) return RLK_ERR_INVALID_ARG;
    if (H < rlk::kBlockK || H % rlk::kBlockK != 0 || H > (int64_t(1) << 20)) return RLK_ERR_UNSUPPORTED;
    if (!aligned(hidden, 16) || !aligned(W, 16) || !aligned(targets, 4)) return RLK_ERR_ALIGNMENT;
    return RLK_OK;
}

// Tile tree over a full-vocabulary workspace (layout_of(T, V, n_shards)):
// shard records, then lse (and logprob when targets is not null).
rlk_status_t run_tile_tree(const int32_t* targets, const uint8_t* active, int64_t T, int64_t V,
                           int n_shards, float* out_logprob, float* out_lse, uint8_t* ws,
                           const Layout& l, int32_t* status, cudaStream_t stream,
                           const DeviceState* dev) {
    const int64_t nt = n_tiles_of(V);
    rlk::TileTreeArgs a;
    std::memset(&a, 0, sizeof(a));
    a.partials = reinterpret_cast<const float2*>(ws + l.partials);
    a.ld = nt;
    a.tgt_logit = reinterpret_cast<const float*>(ws + l.tgt);
    a.targets = targets;
    a.active = active;
    a.status = status;
    a.T = int(T);
    a.n_tiles = int(nt);
    a.depth = tree_depth(nt);
    a.shard_depth = log2_exact(n_shards);
    a.n_shards = n_shards;
    a.shard_mode = 0;
    for (int r = 0; r < n_shards; ++r) {
        int64_t b = 0, e = 0;
        int64_t first = 0, count = 0;
        tree_node(nt, log2_exact(n_shards), r, &first, &count);
        b = first * kVocabTile;
        e = (first + count) * kVocabTile < V ? (first + count) * kVocabTile : V;
        a.shard_vbegin[r] = b;
        a.shard_vbegin[r + 1] = e;
    }
    a.V_total = V;
    a.out_logprob = out_logprob;
    a.out_lse = out_lse;
    a.records = reinterpret_cast<rlk_partial_t*>(ws + l.records);
    return rlk::launch_tile_tree(a, dev->sm_count, stream) == cudaSuccess ? RLK_OK : RLK_ERR_CUDA;
}

// Checks shared by the two materialised-logits calls.
rlk_status_t mat_checks(const void* logits, int dtype, int64_t ld, int64_t T, int64_t V) {
    if (T < 0 || T > RLK_MAX_ROWS) return RLK_ERR_INVALID_ARG;
    if (V < 1 || ld < V) return RLK_ERR_INVALID_ARG;
    if (V > RLK_MAX_VOCAB) return RLK_ERR_UNSUPPORTED;
    if (dtype != RLK_DTYPE_F32 && dtype != RLK_DTYPE_BF16) return RLK_ERR_UNSUPPORTED;
    if (T > 0 && !logits) return RLK_ERR_INVALID_ARG;
    if (!aligned(logits, dtype == RLK_DTYPE_F32 ? 4 : 2)) return RLK_ERR_ALIGNMENT;
    return RLK_OK;
}

// Argument checks shared by the two backward calls (T == 0 passes).
rlk_status_t backward_checks(const void* hidden, const void* W, const int32_t* targets,
                             const float* grad_logprob, const float* lse, int64_t T, int64_t H,
                             int64_t V, const float* grad_hidden, const float* grad_W,
                             const void* workspace, size_t workspace_bytes) {
    rlk_status_t s = common_checks(hidden, W, targets, T, H);
    if (s != RLK_OK) return s;
    if (V < 1) return RLK_ERR_INVALID_ARG;
    if (V > RLK_MAX_VOCAB) return RLK_ERR_UNSUPPORTED;
    if (T == 0) return RLK_OK;
    if (!grad_logprob || !lse || !workspace || (!grad_hidden && !grad_W))
        return RLK_ERR_INVALID_ARG;
    if (!aligned(workspace, 256) || !aligned(grad_logprob, 4) || !aligned(lse, 4) ||
        !aligned(grad_hidden, 4) || !aligned(grad_W, 4))
        return RLK_ERR_ALIGNMENT;
    if (workspace_bytes < backward_layout_of(T, H, V).total) return RLK_ERR_WORKSPACE;
    return RLK_OK;
}

// Step 3 of both backward calls: grad_W = G^T h (K = T ascending, one range).
rlk_status_t grad_w_gemm(const void* hidden, int64_t T, int64_t H, int64_t V, uint16_t* G,
                         int64_t ldG, float* grad_W, int32_t* dev_status, cudaStream_t st,
                         const DeviceState* dev) {
    rlk_status_t s = RLK_OK;
    CUtensorMap map_gt, map_hmn;
    if ((s = encode_bf16_mn_map(&map_gt, G, V, T, ldG)) != RLK_OK) return s;
    if ((s = encode_bf16_mn_map(&map_hmn, hidden, H, T, H)) != RLK_OK) return s;
    rlk::GemmArgs g;
    std::memset(&g, 0, sizeof(g));
    g.out = grad_W;
    g.ld_out = H;
    g.split_stride = 0;
    g.M = int(V);
    g.N = int(H);
    g.k_blocks = int((T + rlk::kBlockK - 1) / rlk::kBlockK);
    g.kb_per_split = g.k_blocks;
    g.splits = 1;
    g.vec_store = aligned(grad_W, 16);
    // bands of hidden-feature tiles whose hidden columns take ~32 MB of L2
    const int64_t band_bytes = int64_t(32) << 20;
    const int64_t per_tile = T * 256 * 2;  // one 256-feature tile of the T hidden rows
    g.n_band = int(band_bytes / per_tile > 1 ? band_bytes / per_tile : 1);
    g.n_fastest = true;
    g.status = dev_status;
    if (rlk::launch_gemm_f32(map_gt, map_hmn, true, true, g, dev->sm_count, st) != cudaSuccess)
        return RLK_ERR_CUDA;
    return RLK_OK;
}

// Steps 2 and 3 of both backward calls: the two GEMMs from G.
rlk_status_t backward_gemms(const void* hidden, const void* W, int64_t T, int64_t H, int64_t V,
                            uint16_t* G, int64_t ldG, uint8_t* parts, float* grad_hidden,
                            float* grad_W, int32_t* dev_status, cudaStream_t st,
                            DeviceState* dev) {
    rlk_status_t s = RLK_OK;
    // 2. grad_hidden = G W: K = V in kGradHiddenSplits fixed ranges, then a fixed-order sum.
    //    Feature tiles fastest, in bands of 8: the ~152 CTAs running together cover about
    //    19 token tiles x 8 feature tiles of one K range, sharing each G slice (19 k
    //    columns) and each W slice through L2.  Against all 16 feature tiles per band
    //    (9.5 token tiles at a time), each wave re-reads less of the range's W slice, which
    //    is larger than L2: at T = 4096, 5.76 GB of DRAM reads instead of 6.60 GB.
    if (grad_hidden) {
        CUtensorMap map_g, map_wmn;
        if ((s = encode_bf16_k_map(&map_g, G, V, T, ldG, kTileM)) != RLK_OK) return s;
        if ((s = encode_bf16_mn_map(&map_wmn, W, H, V, H)) != RLK_OK) return s;
        const int kb = int((V + rlk::kBlockK - 1) / rlk::kBlockK);
        const int splits = kb < kGradHiddenSplits ? kb : kGradHiddenSplits;
        rlk::GemmArgs g;
        std::memset(&g, 0, sizeof(g));
        g.out = reinterpret_cast<float*>(parts);
        g.ld_out = H;
        g.split_stride = T * H;
        g.M = int(T);
        g.N = int(H);
        g.k_blocks = kb;
        g.kb_per_split = (kb + splits - 1) / splits;
        g.splits = (kb + g.kb_per_split - 1) / g.kb_per_split;
        g.vec_store = true;
        g.n_fastest = true;
        g.n_band = 8;
        g.test_drop_stage = test_drop_stage_code() == 2 ? 1 : 0;
        g.status = dev_status;
        if (rlk::launch_gemm_f32(map_g, map_wmn, false, true, g, dev->sm_count, st) != cudaSuccess)
            return RLK_ERR_CUDA;
        if (!grad_W) {
            if (rlk::launch_sum_splits(g.out, g.split_stride, g.splits, T * H, grad_hidden,
                                       dev->sm_count, st) != cudaSuccess)
                return RLK_ERR_CUDA;
        } else {
            // the memory-bound split sum beside the tensor-bound grad_W GEMM, on the
            // side stream: forked after grad_hidden's GEMM, joined after grad_W's
            std::lock_guard<std::mutex> lock(dev->side_mutex);
            if (!dev->side) {
                if (cudaStreamCreateWithFlags(&dev->side, cudaStreamNonBlocking) != cudaSuccess ||
                    cudaEventCreateWithFlags(&dev->ev_split, cudaEventDisableTiming) != cudaSuccess ||
                    cudaEventCreateWithFlags(&dev->ev_sum, cudaEventDisableTiming) != cudaSuccess)
                    return RLK_ERR_CUDA;
            }
            if (cudaEventRecord(dev->ev_split, st) != cudaSuccess ||
                cudaStreamWaitEvent(dev->side, dev->ev_split, 0) != cudaSuccess)
                return RLK_ERR_CUDA;
            if (rlk::launch_sum_splits(g.out, g.split_stride, g.splits, T * H, grad_hidden,
                                       dev->sm_count, dev->side) != cudaSuccess ||
                cudaEventRecord(dev->ev_sum, dev->side) != cudaSuccess)
                return RLK_ERR_CUDA;
            s = grad_w_gemm(hidden, T, H, V, G, ldG, grad_W, dev_status, st, dev);
            if (cudaStreamWaitEvent(st, dev->ev_sum, 0) != cudaSuccess) return RLK_ERR_CUDA;
            return s;
        }
    }

    // 3. grad_W = G^T h: K = T ascending, one range
    if (grad_W) return grad_w_gemm(hidden, T, H, V, G, ldG, grad_W, dev_status, st, dev);
    return RLK_OK;
}

}  // namespace

extern "C" {

const char* rlk_contract_id(void) { return "rlk-linlogp-v1"; }

const char* rlk_build_fingerprint(void) {
    return "rlk-linlogp-v1; rev=" RLK_GIT_REV "; nvcc=" RLK_NVCC_VERSION
           "; arch=sm_103a; flags=-O3 -ftz=false -prec-div=true -prec-sqrt=true -fmad=false";
}

const char* rlk_status_string(int status) {
    switch (status) {
        case RLK_OK: return "RLK_OK";
        case RLK_ERR_INVALID_ARG: return "RLK_ERR_INVALID_ARG";
        case RLK_ERR_UNSUPPORTED: return "RLK_ERR_UNSUPPORTED";
        case RLK_ERR_ALIGNMENT: return "RLK_ERR_ALIGNMENT";
        case RLK_ERR_WORKSPACE: return "RLK_ERR_WORKSPACE";
        case RLK_ERR_CUDA: return "RLK_ERR_CUDA";
        case RLK_ERR_TARGET_RANGE: return "RLK_ERR_TARGET_RANGE";
        case RLK_ERR_TIMEOUT: return "RLK_ERR_TIMEOUT";
        default: return "RLK_ERR_UNKNOWN";
    }
}

rlk_status_t rlk_shard_range(int64_t V, int n_shards, int shard, int64_t* v_begin,
                             int64_t* v_end) {
    if (!v_begin || !v_end) return RLK_ERR_INVALID_ARG;
    const rlk_status_t s = shard_check(V, n_shards);
    if (s != RLK_OK) return s;
    if (shard < 0 || shard >= n_shards) return RLK_ERR_INVALID_ARG;
    int64_t first = 0, count = 0;
    if (!tree_node(n_tiles_of(V), log2_exact(n_shards), shard, &first, &count))
        return RLK_ERR_UNSUPPORTED;
    *v_begin = first * kVocabTile;
    const int64_t e = (first + count) * kVocabTile;
    *v_end = e < V ? e : V;
    return RLK_OK;
}

size_t rlk_workspace_size(int64_t T, int64_t V, int n_shards) {
    if (T < 0 || T > RLK_MAX_ROWS || shard_check(V, n_shards) != RLK_OK) return 0;
    return layout_of(T, V, n_shards).total;
}

rlk_status_t rlk_tile_partials(const void* hidden, const void* W, const int32_t* targets,
                               const uint8_t* active_mask, int64_t T, int64_t H, int64_t V,
                               int n_shards, void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, rlk_stream_t stream) {
    rlk_status_t s = common_checks(hidden, W, targets, T, H);
    if (s != RLK_OK) return s;
    if ((s = shard_check(V, n_shards)) != RLK_OK) return s;
    if (T == 0) return RLK_OK;
    if (!workspace) return RLK_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return RLK_ERR_ALIGNMENT;
    const Layout l = layout_of(T, V, n_shards);
    if (workspace_bytes < l.total) return RLK_ERR_WORKSPACE;
    DeviceState* dev = nullptr;
    if ((s = device_check(&dev)) != RLK_OK) return s;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    return run_tile_partials(hidden, W, targets, active_mask, T, H, V, 0,
                             reinterpret_cast<float2*>(ws + l.partials),
                             reinterpret_cast<float*>(ws + l.tgt), nullptr, dev_status,
                             reinterpret_cast<cudaStream_t>(stream), dev);
}

rlk_status_t rlk_tile_merge(const int32_t* targets, const uint8_t* active_mask, int64_t T,
                            int64_t V, int n_shards, float* out_logprob, float* out_lse,
                            void* workspace, size_t workspace_bytes, int32_t* dev_status,
                            rlk_stream_t stream) {
    if (T < 0 || T > RLK_MAX_ROWS) return RLK_ERR_INVALID_ARG;
    rlk_status_t s = shard_check(V, n_shards);
    if (s != RLK_OK) return s;
    if (T == 0) return RLK_OK;
    if (!targets || !out_logprob || !out_lse || !workspace) return RLK_ERR_INVALID_ARG;
    if (!aligned(workspace, 256) || !aligned(targets, 4) || !aligned(out_logprob, 4) ||
        !aligned(out_lse, 4))
        return RLK_ERR_ALIGNMENT;
    const Layout l = layout_of(T, V, n_shards);
    if (workspace_bytes < l.total) return RLK_ERR_WORKSPACE;
    DeviceState* dev = nullptr;
    if ((s = device_check(&dev)) != RLK_OK) return s;
    return run_tile_tree(targets, active_mask, T, V, n_shards, out_logprob, out_lse,
                         static_cast<uint8_t*>(workspace), l, dev_status,
                         reinterpret_cast<cudaStream_t>(stream), dev);
}

rlk_status_t rlk_linear_logprob(const void* hidden, const void* W, const int32_t* targets,
                                const uint8_t* active_mask, int64_t T, int64_t H, int64_t V,
                                int n_shards, float* out_logprob, float* out_lse,
                                void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                rlk_stream_t stream) {
    if (T > 0 && (!out_logprob || !out_lse)) return RLK_ERR_INVALID_ARG;
    rlk_status_t s = rlk_tile_partials(hidden, W, targets, active_mask, T, H, V, n_shards,
                                       workspace, workspace_bytes, dev_status, stream);
    if (s != RLK_OK) return s;
    return rlk_tile_merge(targets, active_mask, T, V, n_shards, out_logprob, out_lse, workspace,
                          workspace_bytes, dev_status, stream);
}

rlk_status_t rlk_linear_logprob_save_logits(const void* hidden, const void* W,
                                           const int32_t* targets, const uint8_t* active_mask,
                                           int64_t T, int64_t H, int64_t V, int n_shards,
                                           float* out_logprob, float* out_lse, float* logits,
                                           int64_t ld_logits, void* workspace,
                                           size_t workspace_bytes, int32_t* dev_status,
                                           rlk_stream_t stream) {
    rlk_status_t s = common_checks(hidden, W, targets, T, H);
    if (s != RLK_OK) return s;
    if ((s = shard_check(V, n_shards)) != RLK_OK) return s;
    if (T == 0) return RLK_OK;
    if (!out_logprob || !out_lse || !logits || !workspace || ld_logits < V)
        return RLK_ERR_INVALID_ARG;
    if (!aligned(workspace, 256) || !aligned(logits, 16) || ld_logits % 4 != 0)
        return RLK_ERR_ALIGNMENT;
    const Layout l = layout_of(T, V, n_shards);
    if (workspace_bytes < l.total) return RLK_ERR_WORKSPACE;
    DeviceState* dev = nullptr;
    if ((s = device_check(&dev)) != RLK_OK) return s;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    s = run_tile_partials(hidden, W, targets, active_mask, T, H, V, 0,
                          reinterpret_cast<float2*>(ws + l.partials),
                          reinterpret_cast<float*>(ws + l.tgt), nullptr, dev_status, st, dev,
                          logits, ld_logits);
    if (s != RLK_OK) return s;
    return run_tile_tree(targets, active_mask, T, V, n_shards, out_logprob, out_lse, ws, l,
                         dev_status, st, dev);
}

rlk_status_t rlk_linear_logprob_shard(const void* hidden, const void* W_shard,
                                      const int32_t* targets, const uint8_t* active_mask,
                                      int64_t T, int64_t H, int64_t V_total, int n_shards,
                                      int shard, rlk_partial_t* out_partial, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status,
                                      rlk_stream_t stream) {
    rlk_status_t s = common_checks(hidden, W_shard, targets, T, H);
    if (s != RLK_OK) return s;
    int64_t vb = 0, ve = 0;
    if ((s = rlk_shard_range(V_total, n_shards, shard, &vb, &ve)) != RLK_OK) return s;
    if (T == 0) return RLK_OK;
    if (!out_partial || !workspace) return RLK_ERR_INVALID_ARG;
    if (!aligned(workspace, 256) || !aligned(out_partial, 16)) return RLK_ERR_ALIGNMENT;
    const int64_t V_local = ve - vb;
    const Layout l = layout_of(T, V_local, 1);
    if (workspace_bytes < l.total) return RLK_ERR_WORKSPACE;
    DeviceState* dev = nullptr;
    if ((s = device_check(&dev)) != RLK_OK) return s;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    s = run_tile_partials(hidden, W_shard, targets, active_mask, T, H, V_local, vb,
                          reinterpret_cast<float2*>(ws + l.partials),
                          reinterpret_cast<float*>(ws + l.tgt), nullptr, dev_status, st, dev);
    if (s != RLK_OK) return s;
    const int64_t nt = n_tiles_of(V_local);
    rlk::TileTreeArgs a;
    std::memset(&a, 0, sizeof(a));
    a.partials = reinterpret_cast<const float2*>(ws + l.partials);
    a.ld = nt;
    a.tgt_logit = reinterpret_cast<const float*>(ws + l.tgt);
    a.targets = targets;
    a.active = active_mask;
    a.status = dev_status;
    a.T = int(T);
    a.n_tiles = int(nt);
    a.depth = tree_depth(nt);
    a.shard_depth = 0;
    a.n_shards = 1;
    a.shard_mode = 1;
    a.own_begin = vb;
    a.own_end = ve;
    a.V_total = V_total;
    a.records = out_partial;
    return rlk::launch_tile_tree(a, dev->sm_count, st) == cudaSuccess ? RLK_OK : RLK_ERR_CUDA;
}

rlk_status_t rlk_lse_merge(const rlk_partial_t* const* partials, int n_shards, int64_t T,
                           const uint8_t* active_mask, float* out_logprob, float* out_lse,
                           int32_t* dev_status, rlk_stream_t stream) {
    if (T < 0 || T > RLK_MAX_ROWS) return RLK_ERR_INVALID_ARG;
    if (n_shards < 1 || n_shards > RLK_MAX_SHARDS || log2_exact(n_shards) < 0)
        return RLK_ERR_UNSUPPORTED;
    if (T == 0) return RLK_OK;
    if (!partials || !out_logprob || !out_lse) return RLK_ERR_INVALID_ARG;
    rlk::ShardMergeArgs a;
    std::memset(&a, 0, sizeof(a));
    for (int r = 0; r < n_shards; ++r) {
        if (!partials[r]) return RLK_ERR_INVALID_ARG;
        if (!aligned(partials[r], 16)) return RLK_ERR_ALIGNMENT;
        a.parts[r] = partials[r];
    }
    DeviceState* dev = nullptr;
    rlk_status_t s = device_check(&dev);
    if (s != RLK_OK) return s;
    a.n_shards = n_shards;
    a.T = int(T);
    a.active = active_mask;
    a.out_logprob = out_logprob;
    a.out_lse = out_lse;
    a.status = dev_status;
    return rlk::launch_shard_merge(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? RLK_OK
               : RLK_ERR_CUDA;
}

rlk_status_t rlk_debug_logits(const void* hidden, const void* W, int64_t T, int64_t H, int64_t V,
                              float* out_logits, int32_t* dev_status, rlk_stream_t stream) {
    // targets are not read in this mode; pass W as a stand-in non-null pointer for the checks
    rlk_status_t s = common_checks(hidden, W, reinterpret_cast<const int32_t*>(W), T, H);
    if (s != RLK_OK) return s;
    if (V < 1) return RLK_ERR_INVALID_ARG;
    if (V > RLK_MAX_VOCAB) return RLK_ERR_UNSUPPORTED;
    if (T == 0) return RLK_OK;
    if (!out_logits) return RLK_ERR_INVALID_ARG;
    if (!aligned(out_logits, 4)) return RLK_ERR_ALIGNMENT;
    DeviceState* dev = nullptr;
    if ((s = device_check(&dev)) != RLK_OK) return s;
    return run_tile_partials(hidden, W, nullptr, nullptr, T, H, V, 0, nullptr, nullptr, out_logits,
                             dev_status, reinterpret_cast<cudaStream_t>(stream), dev);
}

rlk_status_t rlk_logits_logprob(const void* logits, int logits_dtype, int64_t ld,
                                const int32_t* targets, const uint8_t* active_mask, int64_t T,
                                int64_t V, int n_shards, float* out_logprob, float* out_lse,
                                void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                rlk_stream_t stream) {
    rlk_status_t s = mat_checks(logits, logits_dtype, ld, T, V);
    if (s != RLK_OK) return s;
    if ((s = shard_check(V, n_shards)) != RLK_OK) return s;
    if (T == 0) return RLK_OK;
    if (!targets || !out_logprob || !out_lse || !workspace) return RLK_ERR_INVALID_ARG;
    if (!aligned(workspace, 256) || !aligned(targets, 4)) return RLK_ERR_ALIGNMENT;
    const Layout l = layout_of(T, V, n_shards);
    if (workspace_bytes < l.total) return RLK_ERR_WORKSPACE;
    DeviceState* dev = nullptr;
    if ((s = device_check(&dev)) != RLK_OK) return s;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (rlk::launch_mat_tile_partials(logits, logits_dtype, ld, targets, active_mask, int(T),
                                      int(V), reinterpret_cast<float2*>(ws + l.partials),
                                      reinterpret_cast<float*>(ws + l.tgt),
                                      dev->sm_count * dev->mat_ctas_per_sm[logits_dtype], st) !=
        cudaSuccess)
        return RLK_ERR_CUDA;
    return run_tile_tree(targets, active_mask, T, V, n_shards, out_logprob, out_lse, ws, l,
                         dev_status, st, dev);
}

rlk_status_t rlk_log_softmax(const void* logits, int logits_dtype, int64_t ld,
                             const uint8_t* active_mask, int64_t T, int64_t V, float* out,
                             float* out_lse, void* workspace, size_t workspace_bytes,
                             int32_t* dev_status, rlk_stream_t stream) {
    rlk_status_t s = mat_checks(logits, logits_dtype, ld, T, V);
    if (s != RLK_OK) return s;
    if (T == 0) return RLK_OK;
    if (!out || !out_lse || !workspace) return RLK_ERR_INVALID_ARG;
    if (!aligned(workspace, 256) || !aligned(out, 4) || !aligned(out_lse, 4))
        return RLK_ERR_ALIGNMENT;
    const Layout l = layout_of(T, V, 1);
    if (workspace_bytes < l.total) return RLK_ERR_WORKSPACE;
    DeviceState* dev = nullptr;
    if ((s = device_check(&dev)) != RLK_OK) return s;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (rlk::launch_mat_tile_partials(logits, logits_dtype, ld, nullptr, active_mask, int(T),
                                      int(V), reinterpret_cast<float2*>(ws + l.partials),
                                      reinterpret_cast<float*>(ws + l.tgt),
                                      dev->sm_count * dev->mat_ctas_per_sm[logits_dtype], st) !=
        cudaSuccess)
        return RLK_ERR_CUDA;
    if ((s = run_tile_tree(nullptr, active_mask, T, V, 1, nullptr, out_lse, ws, l, dev_status,
                           st, dev)) != RLK_OK)
        return s;
    return rlk::launch_log_softmax_out(logits, logits_dtype, ld, out_lse, active_mask, int(T),
                                       int(V), out, dev->sm_count, st) == cudaSuccess
               ? RLK_OK
               : RLK_ERR_CUDA;
}

size_t rlk_backward_workspace_size(int64_t T, int64_t H, int64_t V) {
    if (T < 0 || T > RLK_MAX_ROWS || H < rlk::kBlockK || H % rlk::kBlockK != 0 || V < 1 ||
        V > RLK_MAX_VOCAB)
        return 0;
    return backward_layout_of(T, H, V).total;
}

rlk_status_t rlk_linear_logprob_backward(const void* hidden, const void* W,
                                         const int32_t* targets, const uint8_t* active_mask,
                                         const float* grad_logprob, const float* lse, int64_t T,
                                         int64_t H, int64_t V, float* grad_hidden, float* grad_W,
                                         void* workspace, size_t workspace_bytes,
                                         int32_t* dev_status, rlk_stream_t stream) {
    rlk_status_t s = backward_checks(hidden, W, targets, grad_logprob, lse, T, H, V, grad_hidden,
                                     grad_W, workspace, workspace_bytes);
    if (s != RLK_OK || T == 0) return s;
    DeviceState* dev = nullptr;
    if ((s = device_check(&dev)) != RLK_OK) return s;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const BackwardLayout l = backward_layout_of(T, H, V);
    uint16_t* G = reinterpret_cast<uint16_t*>(ws + l.G);
    const int64_t ldG = grad_ld(V);

    // 1. logits again, then G = g (onehot - softmax) in bf16 (the forward's lse)
    CUtensorMap map_h, map_w;
    const int a_rows = T >= kTileM ? kTileM : int((T + 7) / 8 * 8);
    if ((s = encode_bf16_map(&map_h, hidden, H, T, uint32_t(a_rows))) != RLK_OK) return s;
    if ((s = encode_bf16_map(&map_w, W, H, V, kTileN)) != RLK_OK) return s;
    rlk::TilePartialsArgs a;
    std::memset(&a, 0, sizeof(a));
    a.targets = targets;
    a.active = active_mask;
    a.status = dev_status;
    a.v_offset = 0;
    a.T = int(T);
    a.V_local = int(V);
    a.n_tiles = int(n_tiles_of(V));
    a.k_blocks = int(H / rlk::kBlockK);
    a.a_box_rows = a_rows;
    a.lse = lse;
    a.grad = grad_logprob;
    a.G = G;
    a.ldG = ldG;
    a.V_total = V;
    if (rlk::launch_tile_partials(map_h, map_w, a, rlk::kEpiGrad, dev->sm_count, st) !=
        cudaSuccess)
        return RLK_ERR_CUDA;
    return backward_gemms(hidden, W, T, H, V, G, ldG, ws + l.parts, grad_hidden, grad_W,
                          dev_status, st, dev);
}

rlk_status_t rlk_linear_logprob_backward_from_logits(
    const float* logits, int64_t ld_logits, const void* hidden, const void* W,
    const int32_t* targets, const uint8_t* active_mask, const float* grad_logprob,
    const float* lse, int64_t T, int64_t H, int64_t V, float* grad_hidden, float* grad_W,
    void* workspace, size_t workspace_bytes, int32_t* dev_status, rlk_stream_t stream) {
    rlk_status_t s = backward_checks(hidden, W, targets, grad_logprob, lse, T, H, V, grad_hidden,
                                     grad_W, workspace, workspace_bytes);
    if (s != RLK_OK || T == 0) return s;
    if (!logits || ld_logits < V) return RLK_ERR_INVALID_ARG;
    if (!aligned(logits, 16) || ld_logits % 4 != 0) return RLK_ERR_ALIGNMENT;
    DeviceState* dev = nullptr;
    if ((s = device_check(&dev)) != RLK_OK) return s;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const BackwardLayout l = backward_layout_of(T, H, V);
    uint16_t* G = reinterpret_cast<uint16_t*>(ws + l.G);
    const int64_t ldG = grad_ld(V);
    // 1. G = g (onehot - softmax) in bf16 from the saved logits (the forward's lse)
    if (rlk::launch_grad_from_logits(logits, ld_logits, targets, active_mask, grad_logprob, lse,
                                     int(T), int(V), G, ldG, dev_status, dev->sm_count,
                                     st) != cudaSuccess)
        return RLK_ERR_CUDA;
    return backward_gemms(hidden, W, T, H, V, G, ldG, ws + l.parts, grad_hidden, grad_W,
                          dev_status, st, dev);
}

rlk_status_t rlk_rmsnorm(const void* x, const void* residual, const void* gamma, float eps,
                         int64_t T, int64_t H, void* out, void* residual_out,
                         rlk_stream_t stream) {
    if (T < 0 || T > RLK_MAX_ROWS) return RLK_ERR_INVALID_ARG;
    if (H < 64 || H % 64 != 0 || H > 8192) return RLK_ERR_UNSUPPORTED;
    if (!(eps > 0.0f) || !(eps < 3.0e38f)) return RLK_ERR_INVALID_ARG;
    if (T == 0) return RLK_OK;
    if (!x || !gamma || !out || (residual_out && !residual)) return RLK_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(residual, 16) || !aligned(gamma, 16) || !aligned(out, 16) ||
        !aligned(residual_out, 16))
        return RLK_ERR_ALIGNMENT;
    DeviceState* dev = nullptr;
    rlk_status_t s = device_check(&dev);
    if (s != RLK_OK) return s;
    rlk::RmsNormArgs a;
    a.x = static_cast<const uint16_t*>(x);
    a.res = static_cast<const uint16_t*>(residual);
    a.gamma = static_cast<const uint16_t*>(gamma);
    a.eps = eps;
    a.T = int(T);
    a.H = int(H);
    a.y = static_cast<uint16_t*>(out);
    a.res_out = static_cast<uint16_t*>(residual_out);
    return rlk::launch_rmsnorm(a, dev->sm_count, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? RLK_OK
               : RLK_ERR_CUDA;
}

rlk_status_t rlk_debug_primitive_hash(int which, uint32_t first, uint64_t count,
                                      uint64_t* out_hash, rlk_stream_t stream) {
    if (which < 0 || which > 3 || !out_hash) return RLK_ERR_INVALID_ARG;
    if (uint64_t(first) + count > (uint64_t(1) << 32)) return RLK_ERR_INVALID_ARG;
    if (!aligned(out_hash, 8)) return RLK_ERR_ALIGNMENT;
    DeviceState* dev = nullptr;
    rlk_status_t s = device_check(&dev);
    if (s != RLK_OK) return s;
    return rlk::launch_primitive_hash(which, first, count, out_hash, dev->sm_count,
                                      reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? RLK_OK
               : RLK_ERR_CUDA;
}

}  // extern "C"
