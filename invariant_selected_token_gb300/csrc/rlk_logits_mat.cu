// Selected-token logprob and full log_softmax on materialised logits.
//
// The RL-Kernel blog's own example operator is log_softmax over logits that
// already exist in memory (the blog on bitwise consistency with RL-Kernel +
// vime on AMD, sections 4.2-4.3: rl_kernel.log_softmax with a fixed
// reduction tree, fp32 accumulation).  These kernels apply the same numeric
// contract as the fused path to a [T, V] fp32 or bf16 logits matrix:
//
//   k_mat_tile_partials  a warp stages 32 tiles of one row in shared memory,
//                        then each lane reduces one whole 128-column tile in
//                        registers with the contract's in-tile pairwise tree
//                        (the fused epilogue's arithmetic, run two values per
//                        instruction with the packed fp32 operations).  The
//                        next slice's copies are in flight while a slice is
//                        reduced.  The (m, s) pairs and the target logit go
//                        to the same workspace layout the fused path uses, so
//                        the tile tree kernel finishes the job unchanged.
//   k_log_softmax_out    out[t, v] = RN(l[t, v] - lse[t]).
//
// Given the fused path's own fp32 logits, this path returns the fused path's
// bits.  fp32 logits are HBM-bound (each logit is read once, twice for
// log_softmax, which also writes T x V floats); bf16 logits, half the bytes,
// are bound by the FMA pipe: the contract's exp, the subtraction of the max
// and the tree add are 14 FMA-pipe lane operations per logit.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "rlk_contract.cuh"
#include "rlk_internal.h"

namespace rlk {
namespace {

constexpr int kMatWarps = 4;

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

// Thread-per-tile reduction from shared memory.  A warp stages a slice of
// one row -- 32 consecutive 128-column tiles -- with coalesced loads into
// shared memory (tile i at a 132-float pitch, so the later per-thread reads
// are free of bank conflicts), then lane i reduces tile i in registers with
// the contract's in-tile pairwise tree, exactly as the fused path's epilogue
// does.  No cross-lane reduction remains.
constexpr int kSliceTiles = 32;
// Staged tile pitch in elements: a multiple of 16 bytes (16-byte copies and
// reads stay aligned) that is an odd number of 16-byte chunks (consecutive
// lanes' 16-byte reads fall in different bank groups): 132 fp32 = 33 chunks,
// 136 bf16 = 17 chunks.
template <int kDtype>
struct Pitch {
    static constexpr int value = kDtype == RLK_DTYPE_F32 ? kVocabTile + 4 : kVocabTile + 8;
};

// Copy the slice's real columns into shared memory in their input type
// (element e of the slice at tile e/128, column e%128, tile pitch kPitch
// elements).  Aligned rows use asynchronous 16-byte copies, all in flight
// at once: lane l's i-th copy is chunk l + 32 i, and since 32 chunks span
// whole tiles, its source advances 512 bytes and its destination a fixed
// number of tile pitches per step.  A row tail or an unaligned row falls
// back to plain loads.  The asynchronous copies are complete after
// stage_wait().
template <int kDtype>
__device__ __forceinline__ void stage_issue(const void* row, int64_t c0, int ncols_total, int lane,
                                            bool vec, void* sm_raw) {
    constexpr int kElem = kDtype == RLK_DTYPE_F32 ? 4 : 2;
    constexpr int kPitch = Pitch<kDtype>::value;
    constexpr int kPerChunk = 16 / kElem;                              // elements per copy
    constexpr uint32_t kDstStep = (32 * kPerChunk / kVocabTile) * kPitch * kElem;
    const uint8_t* src = static_cast<const uint8_t*>(row) + c0 * kElem;
    uint8_t* sm = static_cast<uint8_t*>(sm_raw);
    const int full_chunks = vec ? ncols_total / kPerChunk : 0;
    const int e0 = lane * kPerChunk;
    uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(
        sm + ((e0 / kVocabTile) * kPitch + e0 % kVocabTile) * kElem));
    const uint8_t* from = src + e0 * kElem;
    for (int ch = lane; ch < full_chunks; ch += 32) {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(from) : "memory");
        dst += kDstStep;
        from += 512;
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    for (int e = full_chunks * kPerChunk + lane; e < ncols_total; e += 32) {
        uint8_t* d = sm + ((e / kVocabTile) * kPitch + e % kVocabTile) * kElem;
        if (kDtype == RLK_DTYPE_F32)
            *reinterpret_cast<float*>(d) = reinterpret_cast<const float*>(src)[e];
        else
            *reinterpret_cast<uint16_t*>(d) = reinterpret_cast<const uint16_t*>(src)[e];
    }
}

__device__ __forceinline__ void stage_wait() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncwarp();
}

// A staged fp32 tile as 64 pairs (columns 2k, 2k+1).
__device__ __forceinline__ void read_tile_pairs_f32(const void* sm_raw, int tile, uint64_t (&P)[64]) {
    const float* p = static_cast<const float*>(sm_raw) + tile * Pitch<RLK_DTYPE_F32>::value;
#pragma unroll
    for (int c = 0; c < kVocabTile; c += 4) {
        const ulonglong2 q = *reinterpret_cast<const ulonglong2*>(p + c);
        P[c / 2] = q.x;
        P[c / 2 + 1] = q.y;
    }
}

// Eight staged bf16 values (16 bytes) as four words; the asm keeps each read
// where it stands, so no tile is held in registers between the two passes.
__device__ __forceinline__ uint4 lds128(const void* p) {
    uint4 q;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(q.x), "=r"(q.y), "=r"(q.z), "=r"(q.w)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
    return q;
}

// A bf16 word (two columns) widened exactly to an fp32 pair.
__device__ __forceinline__ uint64_t widen_bf16x2(uint32_t w) {
    return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ __nv_bfloat162 as_bf162(uint32_t w) {
    __nv_bfloat162 b;
    memcpy(&b, &w, 4);
    return b;
}
__device__ __forceinline__ uint32_t as_u32(__nv_bfloat162 b) {
    uint32_t w;
    memcpy(&w, &b, 4);
    return w;
}

// Second pass over a staged bf16 tile: the packed tree of the exps, reading
// pairs j..j+3 and j+32..j+35 as they are needed.  The exps run on (column
// 2j, column 64+2j) and (2j+1, 64+2j+1) pairs, so the two level-1 sums s_j
// and s_j+32 come out of one packed add (299.6 against 303.4 us with the
// exps on (2j, 2j+1) pairs and two scalar adds).
template <bool kUnderflow>
__device__ __forceinline__ float bf16_tile_sum(const uint16_t* tile, uint64_t neg_m) {
    TreeX2 tree;
#pragma unroll
    for (int j0 = 0; j0 < 32; j0 += 4) {
        const uint4 lo = lds128(tile + 2 * j0);
        const uint4 hi = lds128(tile + 64 + 2 * j0);
        const uint32_t L[4] = {lo.x, lo.y, lo.z, lo.w};
        const uint32_t H[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint64_t even = f2_pack(__uint_as_float(L[i] << 16), __uint_as_float(H[i] << 16));
            const uint64_t odd = f2_pack(__uint_as_float(L[i] & 0xFFFF0000u),
                                         __uint_as_float(H[i] & 0xFFFF0000u));
            tree.push_node(j0 + i, f2_add(contract_exp_x2<kUnderflow>(f2_add(even, neg_m)),
                                          contract_exp_x2<kUnderflow>(f2_add(odd, neg_m))));
        }
    }
    return tree.total();
}

// A staged bf16 tile reduced straight from shared memory in two passes: max
// and min two columns per instruction on the bf16 pairs (bf16 widens
// exactly and monotonically, so the widened max is the fp32 max of the
// widened values; the min propagates NaN), then the exps and the tree.
// When the tile holds no NaN and its smallest value is within 86 of its max,
// every exp argument lies in [-86, 0] and the exps take their shorter form
// (no underflow select, the scaling by 2^n an exponent add); the bits are
// the same either way.
__device__ __forceinline__ MaxSum bf16_tile_reduce(const uint16_t* tile) {
    __nv_bfloat162 mx[2], mn[2];
#pragma unroll
    for (int c = 0; c < kVocabTile; c += 8) {
        const uint4 q = lds128(tile + c);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 b = as_bf162(w[i]);
            if (c == 0 && i < 2) {
                mx[i] = b;
                mn[i] = b;
            } else {
                mx[i & 1] = __hmax2(mx[i & 1], b);
                mn[i & 1] = __hmin2_nan(mn[i & 1], b);
            }
        }
    }
    const uint64_t mx2 = widen_bf16x2(as_u32(__hmax2(mx[0], mx[1])));
    const uint64_t mn2 = widen_bf16x2(as_u32(__hmin2_nan(mn[0], mn[1])));
    float a, b, c, d;
    f2_unpack(mx2, a, b);
    f2_unpack(mn2, c, d);
    MaxSum out;
    out.m = fmaxf(a, b);
    const uint64_t neg_m = f2_splat(-out.m);
    // NaN in c or d (or a NaN difference) fails the comparison
    if (__fsub_rn(c, out.m) >= -86.0f && __fsub_rn(d, out.m) >= -86.0f)
        out.s = bf16_tile_sum<false>(tile, neg_m);
    else
        out.s = bf16_tile_sum<true>(tile, neg_m);
    return out;
}

// Staged element c of a tile as fp32.
template <int kDtype>
__device__ __forceinline__ float staged_value(const void* sm_raw, int tile, int c) {
    constexpr int kPitch = Pitch<kDtype>::value;
    if (kDtype == RLK_DTYPE_F32) return static_cast<const float*>(sm_raw)[tile * kPitch + c];
    return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(sm_raw)[tile * kPitch + c]) << 16);
}

// fp32: three CTAs per SM -- the slices fill shared memory at three, and the
// register cap (168) that three imply costs no spills.  bf16: five CTAs per
// SM (96 registers) -- the tile is reduced from shared memory,
// not held in registers, and the other warps cover a warp's staging (four
// CTAs: 331 us, five: 307 us, six: 308 us at T = 4096).
template <int kDtype>
constexpr int mat_ctas_per_sm() { return kDtype == RLK_DTYPE_F32 ? 3 : 5; }

template <int kDtype>
__global__ void __launch_bounds__(kMatWarps * 32, mat_ctas_per_sm<kDtype>())
    k_mat_tile_partials(const void* logits, int64_t ld, bool vec, const int32_t* targets,
                        const uint8_t* active, int T, int V, int n_tiles, float2* partials,
                        float* tgt_logit) {
    extern __shared__ float4 mat_smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    constexpr int kElem = kDtype == RLK_DTYPE_F32 ? 4 : 2;
    void* sm = reinterpret_cast<uint8_t*>(mat_smem) +
               warp * (kSliceTiles * Pitch<kDtype>::value * kElem);
    const int slices_per_row = (n_tiles + kSliceTiles - 1) / kSliceTiles;
    // The warp's tasks are (row t, slice s of 32 tiles) in row-major order,
    // every gridDim.x * kMatWarps-th one; the position advances by a fixed
    // (rows, slices) step instead of dividing a task index per task.
    // Inactive rows are skipped.  The row index stays in 32 bits: T is at most
    // RLK_MAX_ROWS = 2^31 - 2^20 and a step passes the last row by less than
    // one grid stride (at most kMatMaxBlocks * kMatWarps = 2^20 tasks).
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kMatWarps;
    const int step_t = static_cast<int>(stride / slices_per_row);
    const int step_s = static_cast<int>(stride - static_cast<int64_t>(step_t) * slices_per_row);
    auto advance = [&](int& t, int& s) {
        t += step_t;
        s += step_s;
        if (s >= slices_per_row) {
            s -= slices_per_row;
            ++t;
        }
    };
    auto skip_inactive = [&](int& t, int& s) {
        while (t < T && active && active[t] == 0) advance(t, s);
    };
    auto issue = [&](int t, int s) {
        const int64_t c0 = static_cast<int64_t>(s) * (kSliceTiles * kVocabTile);
        const int ncols_total = min(kSliceTiles * kVocabTile, V - static_cast<int>(c0));
        const void* row = static_cast<const uint8_t*>(logits) + static_cast<int64_t>(t) * ld * kElem;
        stage_issue<kDtype>(row, c0, ncols_total, lane, vec, sm);
    };
    const int first = static_cast<int>(blockIdx.x) * kMatWarps + warp;
    int t = first / slices_per_row, s = first - (first / slices_per_row) * slices_per_row;
    skip_inactive(t, s);
    if (t < T) issue(t, s);
    while (t < T) {
        stage_wait();
        const int j = s * kSliceTiles + lane;
        const bool own = j < n_tiles;
        const int ncols = own ? min(kVocabTile, V - j * kVocabTile) : 0;
        if (own && targets) {
            const int64_t tl = static_cast<int64_t>(targets[t]) - static_cast<int64_t>(j) * kVocabTile;
            if (tl >= 0 && tl < ncols) tgt_logit[t] = staged_value<kDtype>(sm, lane, static_cast<int>(tl));
        }
        int nt = t, ns = s;
        advance(nt, ns);
        skip_inactive(nt, ns);
        if constexpr (kDtype == RLK_DTYPE_BF16) {
            if (own) {
                // columns past the vocabulary are not part of the tile: -inf
                // (bf16 0xFF80) in the lane's own staged tile
                uint16_t* tile = static_cast<uint16_t*>(sm) + lane * Pitch<kDtype>::value;
                for (int c = ncols; c < kVocabTile; ++c) tile[c] = 0xFF80u;
                const MaxSum r = bf16_tile_reduce(tile);
                partials[static_cast<int64_t>(t) * n_tiles + j] = make_float2(r.m, r.s);
            }
            __syncwarp();  // every lane is done with its tile: the buffer is free
            if (nt < T) issue(nt, ns);
            t = nt;
            s = ns;
            continue;
        }
        uint64_t P[64];
        if (own) read_tile_pairs_f32(sm, lane, P);
        __syncwarp();  // every lane has its tile: the buffer is free
        if (nt < T) issue(nt, ns);
        if (own) {
            // columns past the vocabulary are not part of the tile: -inf, whose
            // exp is +0, so their tree partners pass through unchanged
            if (ncols < kVocabTile) {
#pragma unroll
                for (int k = 0; k < 64; ++k) {
                    float a, b;
                    f2_unpack(P[k], a, b);
                    P[k] = f2_pack(2 * k < ncols ? a : -CUDART_INF_F,
                                   2 * k + 1 < ncols ? b : -CUDART_INF_F);
                }
            }
            const MaxSum r = tile_reduce_x2(P);
            partials[static_cast<int64_t>(t) * n_tiles + j] = make_float2(r.m, r.s);
        }
        t = nt;
        s = ns;
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

// The backward's G from saved fp32 logits: one thread per 8 columns of a row
// (two 16-byte loads, one 16-byte store), the arithmetic of the fused
// gradient epilogue (contract_grad_x2) on the same fp32 logits, so G has the
// same bits.  Inactive rows get zeros; an active row whose target is out of
// range sets RLK_ERR_TARGET_RANGE (its G has no target column).
__global__ void __launch_bounds__(256)
    k_grad_from_logits(const float* logits, int64_t ld, const int32_t* targets,
                       const uint8_t* active, const float* grad, const float* lse, int T, int V,
                       uint16_t* G, int64_t ldG, int32_t* status) {
    const int64_t groups_per_row = (V + 7) / 8;
    const int64_t n = static_cast<int64_t>(T) * groups_per_row;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(i / groups_per_row);
        const int c = static_cast<int>(i - static_cast<int64_t>(t) * groups_per_row) * 8;
        const bool valid = active ? active[t] != 0 : true;
        const int64_t tg = targets[t];
        if (valid && c == 0 && (tg < 0 || tg >= V) && status)
            atomicOr(status, 1 << RLK_ERR_TARGET_RANGE);
        const int64_t tl = tg - c;
        const uint64_t neg_lse = f2_splat(valid ? -lse[t] : 0.0f);
        const uint64_t g2 = f2_splat(valid ? grad[t] : 0.0f);
        const float* src = logits + static_cast<int64_t>(t) * ld + c;
        float x[8];
        if (c + 8 <= V) {
            const float4 a = *reinterpret_cast<const float4*>(src);
            const float4 b = *reinterpret_cast<const float4*>(src + 4);
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
            x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) x[k] = c + k < V ? src[k] : 0.0f;
        }
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = contract_grad_x2(f2_pack(x[2 * k], x[2 * k + 1]), neg_lse, g2, 2 * k == tl,
                                    2 * k + 1 == tl, valid);
        uint16_t* dst = G + static_cast<int64_t>(t) * ldG + c;
        if (c + 8 <= V) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (c + k < V) dst[k] = static_cast<uint16_t>(w[k / 2] >> (16 * (k & 1)));
        }
    }
}

// one slice per warp: fp32 4 warps x 32 tiles x 132 x 4 B = 66 KB (3 CTAs per
// SM), bf16 4 x 32 x 136 x 2 B = 34 KB (6 CTAs per SM)
template <int kDtype>
constexpr int mat_smem_bytes() {
    return kMatWarps * kSliceTiles * Pitch<kDtype>::value * (kDtype == RLK_DTYPE_F32 ? 4 : 2);
}

// Largest grid of the materialised-logits kernel (the walk's step bound).
constexpr int64_t kMatMaxBlocks = int64_t(1) << 18;

// Every row starts on a 16-byte boundary (16-byte copies of whole chunks).
bool rows_vector_aligned(const void* logits, int dtype, int64_t ld) {
    const int64_t row_bytes = ld * (dtype == RLK_DTYPE_F32 ? 4 : 2);
    return (reinterpret_cast<uintptr_t>(logits) % 16) == 0 && row_bytes % 16 == 0;
}

}  // namespace

cudaError_t prepare_mat_kernels(int* ctas_per_sm) {
    cudaError_t e = cudaFuncSetAttribute(k_mat_tile_partials<RLK_DTYPE_F32>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         mat_smem_bytes<RLK_DTYPE_F32>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_mat_tile_partials<RLK_DTYPE_BF16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 mat_smem_bytes<RLK_DTYPE_BF16>());
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &ctas_per_sm[0], k_mat_tile_partials<RLK_DTYPE_F32>, kMatWarps * 32,
            mat_smem_bytes<RLK_DTYPE_F32>());
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &ctas_per_sm[1], k_mat_tile_partials<RLK_DTYPE_BF16>, kMatWarps * 32,
            mat_smem_bytes<RLK_DTYPE_BF16>());
    if (e == cudaSuccess && (ctas_per_sm[0] < 1 || ctas_per_sm[1] < 1)) e = cudaErrorInvalidConfiguration;
    return e;
}

cudaError_t launch_mat_tile_partials(const void* logits, int dtype, int64_t ld,
                                     const int32_t* targets, const uint8_t* active, int T, int V,
                                     float2* partials, float* tgt_logit, int resident_ctas,
                                     cudaStream_t stream) {
    const int n_tiles = (V + kVocabTile - 1) / kVocabTile;
    const bool vec = rows_vector_aligned(logits, dtype, ld);
    const int64_t tasks = static_cast<int64_t>(T) * ((n_tiles + kSliceTiles - 1) / kSliceTiles);
    int64_t blocks = (tasks + kMatWarps - 1) / kMatWarps;
    // fp32: one resident wave, each warp overlapping its next slice's copies
    // with its reduction.  bf16: a warp per task (up to 2^20 tasks per walk
    // step), so the block scheduler hands out work as warps finish; one
    // persistent wave with a fixed walk left a quarter of the warp slots
    // idle on average (348 against 308 us at T = 4096).
    if (dtype == RLK_DTYPE_F32 && blocks > resident_ctas) {
        blocks = resident_ctas;
        // a walk stride that is a multiple of the slices per row would give
        // every warp a fixed slice index, and the warps of a row's short last
        // slice little work (one CTA fewer: 420 -> 417 us at V = 151936)
        const int64_t slices_per_row = (n_tiles + kSliceTiles - 1) / kSliceTiles;
        if (blocks > 1 && (blocks * kMatWarps) % slices_per_row == 0) --blocks;
    }
    if (blocks > kMatMaxBlocks) blocks = kMatMaxBlocks;
    if (dtype == RLK_DTYPE_F32)
        k_mat_tile_partials<RLK_DTYPE_F32><<<static_cast<int>(blocks), kMatWarps * 32,
                                             mat_smem_bytes<RLK_DTYPE_F32>(), stream>>>(logits, ld, vec, targets, active, T, V,
                                                       n_tiles, partials, tgt_logit);
    else
        k_mat_tile_partials<RLK_DTYPE_BF16><<<static_cast<int>(blocks), kMatWarps * 32,
                                              mat_smem_bytes<RLK_DTYPE_BF16>(), stream>>>(logits, ld, vec, targets, active, T, V,
                                                        n_tiles, partials, tgt_logit);
    return cudaGetLastError();
}

cudaError_t launch_grad_from_logits(const float* logits, int64_t ld, const int32_t* targets,
                                    const uint8_t* active, const float* grad, const float* lse,
                                    int T, int V, uint16_t* G, int64_t ldG, int32_t* status,
                                    int num_sms, cudaStream_t stream) {
    const int64_t n = static_cast<int64_t>(T) * ((V + 7) / 8);
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    if (blocks > cap) blocks = cap;
    k_grad_from_logits<<<static_cast<int>(blocks), 256, 0, stream>>>(logits, ld, targets, active,
                                                                     grad, lse, T, V, G, ldG,
                                                                     status);
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
