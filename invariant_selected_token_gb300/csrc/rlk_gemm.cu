// Deterministic bf16 GEMM with fp32 output for the backward pass:
//   grad_hidden = G · W   (M = T, N = H, K = V; G K-major, W MN-major)
//   grad_W      = Gᵀ · h  (M = V, N = H, K = T; Gᵀ MN-major, h MN-major)
// where G = g (onehot - softmax) is the bf16 logit gradient (the blog on
// bitwise consistency, sections 3.3 and 4.2: the kernel must provide a
// backward with the same numeric discipline as its forward).
//
// The same persistent, warp-specialised tcgen05 pipeline as the forward
// logits kernel: warp 0 TMA producer (4-stage ring, 128-byte swizzle), warp
// 1 TMEM owner + single-thread MMA issue (kind::f16, M=128, N=256, fp32
// accumulator, K ascending in steps of 16), warps 2-5 epilogue (TMEM -> fp32
// rows in global memory).  An operand is K-major (K contiguous: one 64 x rows
// box per stage) or MN-major (M/N contiguous: boxes of 64 MN elements x 64 K
// rows, one per 64-wide MN atom).
//
// Determinism: every output element is one accumulator over a fixed K range
// in ascending order.  A GEMM may be cut into `splits` fixed K ranges
// (independent of M, N and of the scheduler); each range writes its own fp32
// partial and k_sum_splits adds the partials in a fixed pairwise order.
#include <cstdint>
#include <cuda_runtime.h>

#include "rlk_internal.h"
#include "rlk_ptx.cuh"

namespace rlk {
namespace {

constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr uint32_t kBytesA = kBM * kBK * 2;  // 16 KB
constexpr uint32_t kBytesB = kBN * kBK * 2;  // 32 KB
constexpr uint32_t kAtomBytes = 64 * kBK * 2;  // one MN-major box: 64 MN x 64 K = 8 KB
constexpr uint32_t kTmemCols = 512;
// Epilogue staging: each epilogue warp turns its 32 rows x 32 columns of fp32
// results around in shared memory (row pitch 36 floats: the eight rows a
// 16-byte access phase touches fall in distinct bank quads), so that every
// global store instruction writes whole 128-byte row segments.
constexpr int kTrPitch = 36;
constexpr uint32_t kTrBytes = 4 * 32 * kTrPitch * 4;  // four epilogue warps, 18 KB
constexpr int kSmemBytes = kStages * (kBytesA + kBytesB) + 1024 + 256 + kTrBytes;

__device__ __forceinline__ void report(int32_t* status, int code) {
    if (status) atomicOr(status, 1 << code);
}

// MN-major, 128-byte swizzle: 64-element MN atoms LBO = 8 KB apart (one TMA
// box each), 8-row K groups SBO = 1024 B apart.
__device__ __forceinline__ uint64_t smem_desc_mn_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(kAtomBytes >> 4) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

template <bool kAmn, bool kBmn>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_f32(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               const GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sA = smem;
    uint8_t* sB = smem + kStages * kBytesA;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + kStages * kBytesB);
    uint64_t* empty = full + kStages;
    uint64_t* acc_full = empty + kStages;
    uint64_t* acc_empty = acc_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* transpose = reinterpret_cast<float*>(sB + kStages * kBytesB + 256);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_m = (g.M + kBM - 1) / kBM;
    const int num_n = (g.N + kBN - 1) / kBN;
    const int tiles_per_split = num_m * num_n;
    const int total = tiles_per_split * g.splits;
    constexpr uint32_t idesc = ptx::idesc_bf16_f32(kBM, kBN) | (kAmn ? (1u << 15) : 0u) |
                               (kBmn ? (1u << 16) : 0u);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&acc_full[b], 1);
            ptx::mbar_init(&acc_empty[b], 4 * 32);
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tensormap(&map_a);
        ptx::prefetch_tensormap(&map_b);
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    // work unit -> (split, n tile, m tile).  m fastest: CTAs running side by
    // side share one B slice through L2; n fastest: they share one A slice
    // (both backward GEMMs, whose A -- the logit gradient -- is the large
    // streamed operand).
    // With n_band, the N tiles are taken in bands: every M tile visits a band's N
    // tiles before the next band, so the band's B columns stay in L2 while A
    // streams (grad_W at T = 8192: the hidden rows are 64 MB, two bands of 32 MB).
    const int n_band = (g.n_band > 0 && g.n_band < num_n) ? g.n_band : num_n;
    auto decode = [&](int unit, int& split, int& n_blk, int& m_blk) {
        split = unit / tiles_per_split;
        const int r = unit - split * tiles_per_split;
        if (g.n_fastest) {
            const int full = num_m * n_band;  // units of a full band
            const int band = r / full;
            const int first_n = band * n_band;
            const int nb = min(n_band, num_n - first_n);
            const int within = r - band * full;
            m_blk = within / nb;
            n_blk = first_n + (within - m_blk * nb);
        } else {
            n_blk = r / num_m;
            m_blk = r - n_blk * num_m;
        }
    };

    if (warp == 0) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            if (g.test_drop_stage && blockIdx.x == 0) {
                // test only: leave stage 0 unfilled; the MMA's bounded wait gives up
                stage = 1;
            }
            for (int unit = blockIdx.x; unit < total && !*abort_flag; unit += gridDim.x) {
                int split, n_blk, m_blk;
                decode(unit, split, n_blk, m_blk);
                const int kb0 = split * g.kb_per_split;
                const int kb1 = min(g.k_blocks, kb0 + g.kb_per_split);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
                        *abort_flag = 1;
                        report(g.status, RLK_ERR_TIMEOUT);
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(&full[stage], kBytesA + kBytesB);
                    uint8_t* a_dst = sA + stage * kBytesA;
                    uint8_t* b_dst = sB + stage * kBytesB;
                    if (kAmn) {
                        for (int i = 0; i < kBM / 64; ++i)
                            ptx::tma_load_2d(a_dst + i * kAtomBytes, &map_a, &full[stage],
                                             m_blk * kBM + i * 64, kb * kBK);
                    } else {
                        ptx::tma_load_2d(a_dst, &map_a, &full[stage], kb * kBK, m_blk * kBM);
                    }
                    if (kBmn) {
                        for (int i = 0; i < kBN / 64; ++i)
                            ptx::tma_load_2d(b_dst + i * kAtomBytes, &map_b, &full[stage],
                                             n_blk * kBN + i * 64, kb * kBK);
                    } else {
                        ptx::tma_load_2d(b_dst, &map_b, &full[stage], kb * kBK, n_blk * kBN);
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            for (int unit = blockIdx.x; unit < total && !*abort_flag; unit += gridDim.x) {
                int split, n_blk, m_blk;
                decode(unit, split, n_blk, m_blk);
                const int kb0 = split * g.kb_per_split;
                const int kb1 = min(g.k_blocks, kb0 + g.kb_per_split);
                if (!ptx::mbar_wait(&acc_empty[acc], acc_phase ^ 1u, abort_flag)) {
                    *abort_flag = 1;
                    report(g.status, RLK_ERR_TIMEOUT);
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * kBN;
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!ptx::mbar_wait(&full[stage], phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint32_t a0 = ptx::smem_addr(sA + stage * kBytesA);
                    const uint32_t b0 = ptx::smem_addr(sB + stage * kBytesB);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        // K-major: 16 elements = 32 B along the swizzled row;
                        // MN-major: 16 K rows of 128 B = 2048 B
                        const uint64_t da = kAmn ? smem_desc_mn_sw128(a0 + kk * 2048)
                                                 : ptx::smem_desc_k_sw128(a0 + kk * 32);
                        const uint64_t db = kBmn ? smem_desc_mn_sw128(b0 + kk * 2048)
                                                 : ptx::smem_desc_k_sw128(b0 + kk * 32);
                        ptx::mma_bf16(d_tmem, da, db, idesc, (kb != kb0 || kk) ? 1u : 0u);
                    }
                    ptx::mma_commit(&empty[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) {
                    *abort_flag = 1;
                    report(g.status, RLK_ERR_TIMEOUT);
                    break;
                }
                ptx::mma_commit(&acc_full[acc]);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
        }
    } else {
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        float* tr = transpose + quad * (32 * kTrPitch);  // this warp's 32 x 32 staging tile
        uint32_t acc = 0, acc_phase = 0;
        for (int unit = blockIdx.x; unit < total; unit += gridDim.x) {
            int split, n_blk, m_blk;
            decode(unit, split, n_blk, m_blk);
            if (!ptx::mbar_wait(&acc_full[acc], acc_phase, abort_flag)) {
                *abort_flag = 1;
                report(g.status, RLK_ERR_TIMEOUT);
                break;
            }
            ptx::tc_fence_after_sync();
            const int m = m_blk * kBM + row;
            const int n0 = n_blk * kBN;
            float* out_split = g.out + static_cast<int64_t>(split) * g.split_stride;
            float* dst = out_split + static_cast<int64_t>(m) * g.ld_out + n0;
            const bool row_ok = m < g.M;
            const bool vec = g.vec_store && n0 + kBN <= g.N;
            // staged stores: in pass i, lanes 8j..8j+7 write row 4i + j of the warp's 32
            // rows, 4 consecutive columns each (one 128-byte segment per row)
            const int st_row = lane >> 3;
            const int st_col = (lane & 7) * 4;
#pragma unroll 1
            for (int q = 0; q < kBN / 32; ++q) {
                float v[32];
                __syncwarp();
                ptx::tmem_load_32cols(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                          acc * kBN + q * 32,
                                      v);
                if (vec) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4*>(tr + lane * kTrPitch + i) =
                            make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int r = 4 * i + st_row;
                        const int mr = m_blk * kBM + quad * 32 + r;
                        const float4 x = *reinterpret_cast<const float4*>(tr + r * kTrPitch + st_col);
                        if (mr < g.M)
                            *reinterpret_cast<float4*>(out_split + static_cast<int64_t>(mr) * g.ld_out +
                                                       n0 + q * 32 + st_col) = x;
                    }
                } else if (row_ok) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (n0 + q * 32 + i < g.N) dst[q * 32 + i] = v[i];
                }
            }
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(&acc_empty[acc]);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        const uint64_t t0 = ptx::globaltimer();
        while (ptx::globaltimer() - t0 < 1000000ull) {
        }
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
}

// out[i] = pairwise sum over the split partials, fixed order:
// ((p0 + p1) + (p2 + p3)) + ((p4 + p5) + (p6 + p7)); absent partials pass through.
__global__ void k_sum_splits(const float* parts, int64_t split_stride, int splits, int64_t n,
                             float* out) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float v[8];
#pragma unroll
        for (int s = 0; s < 8; ++s) v[s] = s < splits ? parts[s * split_stride + i] : 0.0f;
#pragma unroll
        for (int w = 1; w < 8; w <<= 1)
#pragma unroll
            for (int s = 0; s + w < 8; s += 2 * w)
                if (s + w < splits) v[s] = __fadd_rn(v[s], v[s + w]);
        out[i] = v[0];
    }
}

}  // namespace

cudaError_t prepare_gemm_kernels() {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(k_gemm_f32<false, true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)) !=
        cudaSuccess)
        return e;
    return cudaFuncSetAttribute(k_gemm_f32<true, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

cudaError_t launch_gemm_f32(const CUtensorMap& map_a, const CUtensorMap& map_b, bool a_mn,
                            bool b_mn, const GemmArgs& g, int num_sms, cudaStream_t stream) {
    const int64_t units = static_cast<int64_t>((g.M + kBM - 1) / kBM) * ((g.N + kBN - 1) / kBN) *
                          g.splits;
    const int grid = static_cast<int>(units < num_sms ? units : num_sms);
    if (!b_mn) return cudaErrorInvalidValue;
    if (a_mn)
        k_gemm_f32<true, true><<<grid, kThreads, kSmemBytes, stream>>>(map_a, map_b, g);
    else
        k_gemm_f32<false, true><<<grid, kThreads, kSmemBytes, stream>>>(map_a, map_b, g);
    return cudaGetLastError();
}

cudaError_t launch_sum_splits(const float* parts, int64_t split_stride, int splits, int64_t n,
                              float* out, int num_sms, cudaStream_t stream) {
    int64_t blocks = (n + 255) / 256;
    if (blocks > num_sms * 8) blocks = num_sms * 8;
    k_sum_splits<<<static_cast<int>(blocks), 256, 0, stream>>>(parts, split_stride, splits, n, out);
    return cudaGetLastError();
}

}  // namespace rlk
