// Strict RMSNorm producing the head's hidden states ("vLLM RL-Kernel v0.1.0:
// ROCm 上でのビット単位のトレーニング-ロールアウト一貫性", strict-path table, row
// "RMSNorm": reduction domain, epsilon, residual add, output boundary).
//
// Contract, per row:
//   x'   = bf16_RN(RN(x + r))                       residual add (optional)
//   s    = pairwise tree over nextpow2(H) feature slots of RN(x'_i * x'_i)
//          (products of bf16 values are exact in fp32; slots >= H absent)
//   a    = RN(RN(s / H) + eps)
//   rstd = rlk_rsqrt(a)
//   y_i  = bf16_RN(RN(RN(x'_i * rstd) * gamma_i))
//
// Layout: element i = 256 k + 8 l + j is lane l's j-th value of column group
// k, so each lane reads 16 contiguous bytes per group (a warp reads 512
// contiguous bytes) and the tree's levels fall as: 1-3 over j inside the
// lane, 4-8 over l across lanes (xor 1..16, lower lane on the left), then
// over the groups -- the contract's pairwise tree over the feature index,
// whatever the row's position in the batch.  Three kernels share it:
//   k_rmsnorm          one warp per row (rows of at most 256 features);
//   k_rmsnorm_team     rows of 512 .. 4096 features split across a team of
//                      warps, each holding whole groups; the team's partial
//                      sums are the top levels of the same tree;
//   k_rmsnorm_grouped  one warp per row, group by group (rows wider than 4096
//                      features, whose x and residual do not fit in
//                      registers together).
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "rlk_contract.cuh"
#include "rlk_internal.h"

namespace rlk {
namespace {


__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}

constexpr int kRmsWarps = 4;
// Warps per row for rows of 512 .. 4096 features (measured at H = 4096, T =
// 4096: one warp per row 38 us, two 33.6 us, four 27.3 us, eight 27.2 us).
#ifndef RLK_RMS_TEAM
#define RLK_RMS_TEAM 8
#endif

__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b) {
    return pack_bf16(__fadd_rn(bf16_lo(a), bf16_lo(b)), __fadd_rn(bf16_hi(a), bf16_hi(b)));
}

// kK column groups of 256 features per row (nextpow2(H) / 256, 1 .. 16).
// All of a row's loads are issued before any of its stores, so they are in
// flight together.  out / residual_out may be x / residual themselves: every
// element is read before the same element is written, and rows are disjoint.
template <int kK>
__global__ void __launch_bounds__(kRmsWarps * 32)
    k_rmsnorm(const uint16_t* x, const uint16_t* res, const uint16_t* gamma, float eps, int T,
              int H, uint16_t* y, uint16_t* res_out) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * kRmsWarps;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * kRmsWarps + (threadIdx.x >> 5); t < T;
         t += warps) {
        uint4 v[kK];  // x' of this lane, 8 bf16 per group
#pragma unroll
        for (int k = 0; k < kK; ++k) {
            const int i0 = 256 * k + 8 * lane;
            v[k] = i0 < H ? *reinterpret_cast<const uint4*>(x + t * H + i0) : make_uint4(0u, 0u, 0u, 0u);
        }
        if (res) {
            uint4 r[kK];
#pragma unroll
            for (int k = 0; k < kK; ++k) {
                const int i0 = 256 * k + 8 * lane;
                r[k] = i0 < H ? *reinterpret_cast<const uint4*>(res + t * H + i0)
                              : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int k = 0; k < kK; ++k) {
                v[k].x = add_bf16x2(v[k].x, r[k].x);
                v[k].y = add_bf16x2(v[k].y, r[k].y);
                v[k].z = add_bf16x2(v[k].z, r[k].z);
                v[k].w = add_bf16x2(v[k].w, r[k].w);
            }
            if (res_out) {
#pragma unroll
                for (int k = 0; k < kK; ++k) {
                    const int i0 = 256 * k + 8 * lane;
                    if (i0 < H) *reinterpret_cast<uint4*>(res_out + t * H + i0) = v[k];
                }
            }
        }
        float part[kK];
#pragma unroll
        for (int k = 0; k < kK; ++k) {
            // levels 1-3: pairs (0,1),(2,3),(4,5),(6,7), then pairs of those; absent
            // groups (i0 >= H) hold +0, which passes every partner through
            const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
            float s2[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float a = bf16_lo(w[p]), b = bf16_hi(w[p]);
                s2[p] = __fadd_rn(__fmul_rn(a, a), __fmul_rn(b, b));
            }
            part[k] = __fadd_rn(__fadd_rn(s2[0], s2[1]), __fadd_rn(s2[2], s2[3]));
        }
        // levels 4-8 across lanes, lower lane on the left
#pragma unroll
        for (int k = 0; k < kK; ++k) {
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float other = __shfl_xor_sync(0xffffffffu, part[k], o);
                part[k] = (lane & o) ? __fadd_rn(other, part[k]) : __fadd_rn(part[k], other);
            }
        }
        // remaining levels over the column groups
#pragma unroll
        for (int w = kK / 2; w >= 1; w >>= 1) {
#pragma unroll
            for (int i = 0; i < w; ++i) part[i] = __fadd_rn(part[2 * i], part[2 * i + 1]);
        }
        const float mean = __fdiv_rn(part[0], static_cast<float>(H));
        const float rstd = contract_rsqrt(__fadd_rn(mean, eps));
        uint16_t* yr = y + t * H;
#pragma unroll
        for (int k = 0; k < kK; ++k) {
            const int i0 = 256 * k + 8 * lane;
            if (i0 < H) {
                const uint4 g = *reinterpret_cast<const uint4*>(gamma + i0);
                const uint32_t xw[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
                const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
                uint32_t o[4];
#pragma unroll
                for (int p = 0; p < 4; ++p)
                    o[p] = pack_bf16(__fmul_rn(__fmul_rn(bf16_lo(xw[p]), rstd), bf16_lo(gw[p])),
                                     __fmul_rn(__fmul_rn(bf16_hi(xw[p]), rstd), bf16_hi(gw[p])));
                *reinterpret_cast<uint4*>(yr + i0) = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
}

// kK = 2 .. 16: each row is split between kW warps (a team), warp w taking
// column groups [w kK/kW, (w+1) kK/kW) -- fewer registers per lane, so more
// rows in flight per SM.  The contract's tree over the column groups is
// perfect, so its top log2(kW) levels combine the warps' sums pairwise in
// order ((w0 + w1) + (w2 + w3) for four): each warp forms its part as the
// one-warp kernel does, and the team combines the parts through shared
// memory (a named barrier per team; two slots alternate between rows, and a
// team's warps are never more than one row apart).
__host__ __device__ constexpr int team_cta_threads(int kW) { return 32 * kW > 128 ? 32 * kW : 128; }

template <int kK, int kW>
__global__ void __launch_bounds__(team_cta_threads(kW))
    k_rmsnorm_team(const uint16_t* x, const uint16_t* res, const uint16_t* gamma, float eps, int T,
                   int H, uint16_t* y, uint16_t* res_out) {
    constexpr int kTeams = team_cta_threads(kW) / (32 * kW);
    constexpr int kPart = kK / kW;  // column groups per warp
    __shared__ float parts[kTeams][2][kW];  // [team][slot][warp]
    const int lane = threadIdx.x & 31;
    const int team = threadIdx.x / (32 * kW);
    const int w = (threadIdx.x >> 5) % kW;
    const int g0 = w * kPart;  // first column group of this warp
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kTeams;
    int slot = 0;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * kTeams + team; t < T; t += stride) {
        uint4 v[kPart];
#pragma unroll
        for (int k = 0; k < kPart; ++k) {
            const int i0 = 256 * (g0 + k) + 8 * lane;
            v[k] = i0 < H ? *reinterpret_cast<const uint4*>(x + t * H + i0) : make_uint4(0u, 0u, 0u, 0u);
        }
        if (res) {
            uint4 r[kPart];
#pragma unroll
            for (int k = 0; k < kPart; ++k) {
                const int i0 = 256 * (g0 + k) + 8 * lane;
                r[k] = i0 < H ? *reinterpret_cast<const uint4*>(res + t * H + i0)
                              : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int k = 0; k < kPart; ++k) {
                v[k].x = add_bf16x2(v[k].x, r[k].x);
                v[k].y = add_bf16x2(v[k].y, r[k].y);
                v[k].z = add_bf16x2(v[k].z, r[k].z);
                v[k].w = add_bf16x2(v[k].w, r[k].w);
            }
            if (res_out) {
#pragma unroll
                for (int k = 0; k < kPart; ++k) {
                    const int i0 = 256 * (g0 + k) + 8 * lane;
                    if (i0 < H) *reinterpret_cast<uint4*>(res_out + t * H + i0) = v[k];
                }
            }
        }
        float part[kPart];
#pragma unroll
        for (int k = 0; k < kPart; ++k) {
            const uint32_t q[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
            float s2[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float a = bf16_lo(q[p]), b = bf16_hi(q[p]);
                s2[p] = __fadd_rn(__fmul_rn(a, a), __fmul_rn(b, b));
            }
            part[k] = __fadd_rn(__fadd_rn(s2[0], s2[1]), __fadd_rn(s2[2], s2[3]));
        }
#pragma unroll
        for (int k = 0; k < kPart; ++k) {
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float other = __shfl_xor_sync(0xffffffffu, part[k], o);
                part[k] = (lane & o) ? __fadd_rn(other, part[k]) : __fadd_rn(part[k], other);
            }
        }
#pragma unroll
        for (int n = kPart / 2; n >= 1; n >>= 1) {
#pragma unroll
            for (int i = 0; i < n; ++i) part[i] = __fadd_rn(part[2 * i], part[2 * i + 1]);
        }
        if (lane == 0) parts[team][slot][w] = part[0];
        asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(32 * kW) : "memory");
        float p[kW];
#pragma unroll
        for (int i = 0; i < kW; ++i) p[i] = parts[team][slot][i];
#pragma unroll
        for (int n = kW / 2; n >= 1; n >>= 1) {
#pragma unroll
            for (int i = 0; i < n; ++i) p[i] = __fadd_rn(p[2 * i], p[2 * i + 1]);
        }
        slot ^= 1;
        const float mean = __fdiv_rn(p[0], static_cast<float>(H));
        const float rstd = contract_rsqrt(__fadd_rn(mean, eps));
        uint16_t* yr = y + t * H;
#pragma unroll
        for (int k = 0; k < kPart; ++k) {
            const int i0 = 256 * (g0 + k) + 8 * lane;
            if (i0 < H) {
                const uint4 g = *reinterpret_cast<const uint4*>(gamma + i0);
                const uint32_t xw[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
                const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
                uint32_t o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    o[q] = pack_bf16(__fmul_rn(__fmul_rn(bf16_lo(xw[q]), rstd), bf16_lo(gw[q])),
                                     __fmul_rn(__fmul_rn(bf16_hi(xw[q]), rstd), bf16_hi(gw[q])));
                *reinterpret_cast<uint4*>(yr + i0) = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
}

// Rows wider than 4096 features (kK = 32): x and the residual of a row do
// not fit in registers together, so the row is read group by group, each
// group's residual store after its own loads.
template <int kK>
__global__ void __launch_bounds__(256)
    k_rmsnorm_grouped(const uint16_t* x, const uint16_t* res, const uint16_t* gamma, float eps, int T,
              int H, uint16_t* y, uint16_t* res_out) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         t < T; t += warps) {
        const uint16_t* xr = x + t * H;
        uint4 v[kK];  // x' of this lane, 8 bf16 per group
        float part[kK];
#pragma unroll
        for (int k = 0; k < kK; ++k) {
            const int i0 = 256 * k + 8 * lane;
            if (i0 < H) {
                uint4 q = *reinterpret_cast<const uint4*>(xr + i0);
                if (res) {
                    const uint4 r = *reinterpret_cast<const uint4*>(res + t * H + i0);
                    q.x = pack_bf16(__fadd_rn(bf16_lo(q.x), bf16_lo(r.x)), __fadd_rn(bf16_hi(q.x), bf16_hi(r.x)));
                    q.y = pack_bf16(__fadd_rn(bf16_lo(q.y), bf16_lo(r.y)), __fadd_rn(bf16_hi(q.y), bf16_hi(r.y)));
                    q.z = pack_bf16(__fadd_rn(bf16_lo(q.z), bf16_lo(r.z)), __fadd_rn(bf16_hi(q.z), bf16_hi(r.z)));
                    q.w = pack_bf16(__fadd_rn(bf16_lo(q.w), bf16_lo(r.w)), __fadd_rn(bf16_hi(q.w), bf16_hi(r.w)));
                    if (res_out) *reinterpret_cast<uint4*>(res_out + t * H + i0) = q;
                }
                v[k] = q;
                // levels 1-3: pairs (0,1),(2,3),(4,5),(6,7), then pairs of those
                const uint32_t w[4] = {q.x, q.y, q.z, q.w};
                float s2[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const float a = bf16_lo(w[p]), b = bf16_hi(w[p]);
                    s2[p] = __fadd_rn(__fmul_rn(a, a), __fmul_rn(b, b));
                }
                part[k] = __fadd_rn(__fadd_rn(s2[0], s2[1]), __fadd_rn(s2[2], s2[3]));
            } else {
                v[k] = make_uint4(0u, 0u, 0u, 0u);
                part[k] = 0.0f;  // absent slots: +0 passes every partner through
            }
        }
        // levels 4-8 across lanes, lower lane on the left
#pragma unroll
        for (int k = 0; k < kK; ++k) {
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float other = __shfl_xor_sync(0xffffffffu, part[k], o);
                part[k] = (lane & o) ? __fadd_rn(other, part[k]) : __fadd_rn(part[k], other);
            }
        }
        // remaining levels over the column groups
#pragma unroll
        for (int w = kK / 2; w >= 1; w >>= 1) {
#pragma unroll
            for (int i = 0; i < w; ++i) part[i] = __fadd_rn(part[2 * i], part[2 * i + 1]);
        }
        const float mean = __fdiv_rn(part[0], static_cast<float>(H));
        const float rstd = contract_rsqrt(__fadd_rn(mean, eps));
        uint16_t* yr = y + t * H;
#pragma unroll
        for (int k = 0; k < kK; ++k) {
            const int i0 = 256 * k + 8 * lane;
            if (i0 < H) {
                const uint4 g = *reinterpret_cast<const uint4*>(gamma + i0);
                const uint32_t xw[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
                const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
                uint32_t o[4];
#pragma unroll
                for (int p = 0; p < 4; ++p)
                    o[p] = pack_bf16(__fmul_rn(__fmul_rn(bf16_lo(xw[p]), rstd), bf16_lo(gw[p])),
                                     __fmul_rn(__fmul_rn(bf16_hi(xw[p]), rstd), bf16_hi(gw[p])));
                *reinterpret_cast<uint4*>(yr + i0) = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
}

template <int kK>
cudaError_t launch_k(const RmsNormArgs& a, int num_sms, cudaStream_t stream) {
    if constexpr (kK >= 2 && kK <= 16) {
        constexpr int kW = (kK >= RLK_RMS_TEAM) ? RLK_RMS_TEAM : kK;  // warps per row
        constexpr int kTeams = team_cta_threads(kW) / (32 * kW);
        int64_t blocks = (static_cast<int64_t>(a.T) + kTeams - 1) / kTeams;
        if (blocks > static_cast<int64_t>(num_sms) * 32) blocks = static_cast<int64_t>(num_sms) * 32;
        k_rmsnorm_team<kK, kW><<<static_cast<int>(blocks), team_cta_threads(kW), 0, stream>>>(
            a.x, a.res, a.gamma, a.eps, a.T, a.H, a.y, a.res_out);
    } else if constexpr (kK <= 16) {
        int64_t blocks = (static_cast<int64_t>(a.T) + kRmsWarps - 1) / kRmsWarps;
        if (blocks > static_cast<int64_t>(num_sms) * 32) blocks = static_cast<int64_t>(num_sms) * 32;
        k_rmsnorm<kK><<<static_cast<int>(blocks), kRmsWarps * 32, 0, stream>>>(
            a.x, a.res, a.gamma, a.eps, a.T, a.H, a.y, a.res_out);
    } else {
        int64_t blocks = (static_cast<int64_t>(a.T) + 7) / 8;
        if (blocks > static_cast<int64_t>(num_sms) * 16) blocks = static_cast<int64_t>(num_sms) * 16;
        k_rmsnorm_grouped<kK><<<static_cast<int>(blocks), 256, 0, stream>>>(
            a.x, a.res, a.gamma, a.eps, a.T, a.H, a.y, a.res_out);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rmsnorm(const RmsNormArgs& a, int num_sms, cudaStream_t stream) {
    int slots = 1;
    while (slots < a.H) slots *= 2;
    const int k = slots <= 256 ? 1 : slots / 256;
    switch (k) {
        case 1: return launch_k<1>(a, num_sms, stream);
        case 2: return launch_k<2>(a, num_sms, stream);
        case 4: return launch_k<4>(a, num_sms, stream);
        case 8: return launch_k<8>(a, num_sms, stream);
        case 16: return launch_k<16>(a, num_sms, stream);
        case 32: return launch_k<32>(a, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace rlk
