// Selected-token logprob and full log_softmax on materialised logits.
//
// The RL-Kernel blog's own example operator is log_softmax over logits that
// already exist in memory (the blog on bitwise consistency with RL-Kernel +
// vime on AMD, sections 4.2-4.3: rl_kernel.log_softmax with a fixed
// reduction tree, fp32 accumulation).  These kernels apply the same numeric
// contract as the fused path to a [T, V] fp32 or bf16 logits matrix:
//
//   k_mat_tile_partials  a warp per run of (token, 128-column tile)s: lane l holds
//                        columns 4l..4l+3; the pairwise tree over the column
//                        index is levels 1-2 inside the lane and levels 3-7
//                        across lanes (xor 1, 2, 4, 8, 16; lower lane left),
//                        which is exactly the contract's 128-slot tree.  The
//                        (m, s) pairs and the target logit go to the same
//                        workspace layout the fused path uses, so the tile
//                        tree kernel finishes the job unchanged.
//   k_log_softmax_out    out[t, v] = RN(l[t, v] - lse[t]).
//
// Given the fused path's own fp32 logits, this path returns the fused path's
// bits.  It is HBM-bound: each logit is read once (twice for log_softmax,
// which also writes T x V floats).
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "rlk_contract.cuh"
#include "rlk_internal.h"

namespace rlk {
namespace {

constexpr int kMatWarps = 8;

// Four consecutive logits of one row as fp32 (bf16 widens exactly).  Columns
// at or beyond `ncols` read as -inf (they are not part of the tile).
// `vec` says rows are aligned for one 16-byte (fp32) / 8-byte (bf16) load
// per lane; otherwise the same four values are read one by one.
template <int kDtype>
__device__ __forceinline__ void load4(const void* row, int64_t c0, int ncols, int lane, bool vec,
                                      float (&x)[4]) {
    const int c = 4 * lane;
    if (kDtype == RLK_DTYPE_F32) {
        const float* p = static_cast<const float*>(row) + c0 + c;
        if (vec && c + 3 < ncols) {
            const float4 q = *reinterpret_cast<const float4*>(p);
            x[0] = q.x; x[1] = q.y; x[2] = q.z; x[3] = q.w;
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) x[i] = (c + i < ncols) ? p[i] : -CUDART_INF_F;
        }
    } else {
        const __nv_bfloat16* p = static_cast<const __nv_bfloat16*>(row) + c0 + c;
        if (vec && c + 3 < ncols) {
            const uint2 q = *reinterpret_cast<const uint2*>(p);
            x[0] = __uint_as_float(q.x << 16);
            x[1] = __uint_as_float(q.x & 0xFFFF0000u);
            x[2] = __uint_as_float(q.y << 16);
            x[3] = __uint_as_float(q.y & 0xFFFF0000u);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                x[i] = (c + i < ncols) ? __bfloat162float(p[i]) : -CUDART_INF_F;
        }
    }
}

// (m, s) of one 128-column tile held 4 columns per lane, plus the target pick.
template <int kDtype>
__device__ __forceinline__ float2 tile_pair(const float (&x)[4], int lane) {
    float m = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    // levels 1-2 of the 128-slot tree inside the lane (padding gives exp(-inf) = +0)
    const float e0 = contract_exp(__fsub_rn(x[0], m));
    const float e1 = contract_exp(__fsub_rn(x[1], m));
    const float e2 = contract_exp(__fsub_rn(x[2], m));
    const float e3 = contract_exp(__fsub_rn(x[3], m));
    float s = __fadd_rn(__fadd_rn(e0, e1), __fadd_rn(e2, e3));
    // levels 3-7 across lanes, the lower lane's partial on the left
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float other = __shfl_xor_sync(0xffffffffu, s, o);
        s = (lane & o) ? __fadd_rn(other, s) : __fadd_rn(s, other);
    }
    return make_float2(m, s);
}

// Warps walk runs of kRun consecutive tiles of one row (no per-tile index
// division), two tiles in flight per step.
template <int kDtype>
__global__ void __launch_bounds__(kMatWarps * 32)
    k_mat_tile_partials(const void* logits, int64_t ld, bool vec, const int32_t* targets,
                        const uint8_t* active, int T, int V, int n_tiles, float2* partials,
                        float* tgt_logit) {
    constexpr int kRun = 16;
    const int lane = threadIdx.x & 31;
    const int runs_per_row = (n_tiles + kRun - 1) / kRun;
    const int64_t n_runs = static_cast<int64_t>(T) * runs_per_row;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kMatWarps;
    const int elem = kDtype == RLK_DTYPE_F32 ? 4 : 2;
    for (int64_t run = static_cast<int64_t>(blockIdx.x) * kMatWarps + (threadIdx.x >> 5);
         run < n_runs; run += stride) {
        const int t = static_cast<int>(run / runs_per_row);
        const int j0 = static_cast<int>(run - static_cast<int64_t>(t) * runs_per_row) * kRun;
        if (active && active[t] == 0) continue;
        const int j1 = min(n_tiles, j0 + kRun);
        const void* row = static_cast<const uint8_t*>(logits) + static_cast<int64_t>(t) * ld * elem;
        const int64_t tg = targets ? static_cast<int64_t>(targets[t]) : -1;
        float2* prow = partials + static_cast<int64_t>(t) * n_tiles;
        for (int j = j0; j < j1; j += 2) {
            const bool two = j + 1 < j1;
            const int64_t c0 = static_cast<int64_t>(j) * kVocabTile;
            const int nc0 = min(kVocabTile, V - static_cast<int>(c0));
            const int nc1 = two ? min(kVocabTile, V - static_cast<int>(c0) - kVocabTile) : 0;
            float x[4], y[4];
            load4<kDtype>(row, c0, nc0, lane, vec, x);
            if (two) load4<kDtype>(row, c0 + kVocabTile, nc1, lane, vec, y);
            const int64_t tl = tg - c0 - 4 * lane;
            if (tl >= 0 && tl < 4 && 4 * lane + tl < nc0)
                tgt_logit[t] = tl == 0 ? x[0] : tl == 1 ? x[1] : tl == 2 ? x[2] : x[3];
            const float2 p0 = tile_pair<kDtype>(x, lane);
            if (lane == 0) prow[j] = p0;
            if (two) {
                const int64_t tl1 = tl - kVocabTile;
                if (tl1 >= 0 && tl1 < 4 && 4 * lane + tl1 < nc1)
                    tgt_logit[t] = tl1 == 0 ? y[0] : tl1 == 1 ? y[1] : tl1 == 2 ? y[2] : y[3];
                const float2 p1 = tile_pair<kDtype>(y, lane);
                if (lane == 0) prow[j + 1] = p1;
            }
        }
    }
}

template <int kDtype>
__global__ void __launch_bounds__(256)
    k_log_softmax_out(const void* logits, int64_t ld, bool vec, const float* lse,
                      const uint8_t* active, int T, int V, float* out) {
    const int elem = kDtype == RLK_DTYPE_F32 ? 4 : 2;
    const int64_t groups_per_row = (V + 3) / 4;
    const int64_t n = static_cast<int64_t>(T) * groups_per_row;
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < n;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(g / groups_per_row);
        const int c = static_cast<int>(g - static_cast<int64_t>(t) * groups_per_row) * 4;
        float* o = out + static_cast<int64_t>(t) * V + c;
        const bool act = active ? active[t] != 0 : true;
        const float l0 = lse[t];
        const void* row = static_cast<const uint8_t*>(logits) + static_cast<int64_t>(t) * ld * elem;
        float x[4];
        // column group c/4 of the row, read the same way the tile kernel reads it
        load4<kDtype>(row, 0, V, c / 4, vec, x);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (c + i < V) o[i] = act ? __fsub_rn(x[i], l0) : 0.0f;
    }
}

bool rows_vector_aligned(const void* logits, int dtype, int64_t ld) {
    const uintptr_t a = dtype == RLK_DTYPE_F32 ? 16 : 8;
    return (reinterpret_cast<uintptr_t>(logits) % a) == 0 && ld % 4 == 0;
}

}  // namespace

cudaError_t launch_mat_tile_partials(const void* logits, int dtype, int64_t ld,
                                     const int32_t* targets, const uint8_t* active, int T, int V,
                                     float2* partials, float* tgt_logit, int num_sms,
                                     cudaStream_t stream) {
    const int n_tiles = (V + kVocabTile - 1) / kVocabTile;
    const bool vec = rows_vector_aligned(logits, dtype, ld);
    const int64_t runs = static_cast<int64_t>(T) * ((n_tiles + 15) / 16);
    int64_t blocks = (runs + kMatWarps - 1) / kMatWarps;
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    if (blocks > cap) blocks = cap;
    if (dtype == RLK_DTYPE_F32)
        k_mat_tile_partials<RLK_DTYPE_F32><<<static_cast<int>(blocks), kMatWarps * 32, 0, stream>>>(
            logits, ld, vec, targets, active, T, V, n_tiles, partials, tgt_logit);
    else
        k_mat_tile_partials<RLK_DTYPE_BF16><<<static_cast<int>(blocks), kMatWarps * 32, 0, stream>>>(
            logits, ld, vec, targets, active, T, V, n_tiles, partials, tgt_logit);
    return cudaGetLastError();
}

cudaError_t launch_log_softmax_out(const void* logits, int dtype, int64_t ld, const float* lse,
                                   const uint8_t* active, int T, int V, float* out, int num_sms,
                                   cudaStream_t stream) {
    const int64_t n = static_cast<int64_t>(T) * ((V + 3) / 4);
    const bool vec = rows_vector_aligned(logits, dtype, ld);
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    if (blocks > cap) blocks = cap;
    if (dtype == RLK_DTYPE_F32)
        k_log_softmax_out<RLK_DTYPE_F32><<<static_cast<int>(blocks), 256, 0, stream>>>(
            logits, ld, vec, lse, active, T, V, out);
    else
        k_log_softmax_out<RLK_DTYPE_BF16><<<static_cast<int>(blocks), 256, 0, stream>>>(
            logits, ld, vec, lse, active, T, V, out);
    return cudaGetLastError();
}

}  // namespace rlk
