// Fixed-order merges of the per-tile (max, sum-exp) pairs: the tile tree,
// the shard records, the final log-sum-exp and logprob, and the separate
// cross-shard merge ("cross-rank LSE merge" and "fixed rank reduction
// order" in the strict-path table of "vLLM RL-Kernel v0.1.0: ROCm 上での
// ビット単位のトレーニング-ロールアウト一貫性").
//
// The contract's tile tree is a recursive bisection of the tile range (a
// node of k tiles gives ceil(k/2) to its left child).  This kernel
// evaluates exactly that tree as a perfect binary tree over 2^depth slots:
// walking the bisection down to single slots places every tile in one slot
// and leaves the remaining slots empty (always in right subtrees).  An empty
// slot carries (-inf, 0), which the merge passes through bit for bit, so
// every non-empty node of the perfect tree holds the bits of the
// corresponding bisection node.
//
// One warp per token.  Lane l owns slots [l*L, (l+1)*L), L = 2^max(0,
// depth-5): it merges them in registers (levels 1..log2 L), then five
// shuffle levels pair lane l with lane l^1, l^2, ..., always with the lower
// lane as the left operand.  The shard nodes (depth log2 n_shards) appear
// after the shuffle level that completes them; their records are written
// from there, and the levels above them are the regular pairwise merge of
// the records in shard order -- the same merges rlk_lse_merge performs.
#include <cstdint>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "rlk_contract.cuh"
#include "rlk_internal.h"

namespace rlk {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ void report(int32_t* status, int code) {
    if (status) atomicOr(status, 1 << code);
}

// Tile held by slot `s` of the depth-`depth` perfect tree over n tiles, or -1.
__device__ __forceinline__ int slot_tile(int s, int depth, int n) {
    int first = 0, k = n;
    for (int b = depth - 1; b >= 0; --b) {
        const int left = (k + 1) >> 1;
        if ((s >> b) & 1) {
            first += left;
            k -= left;
        } else {
            k = left;
        }
    }
    return k == 1 ? first : -1;
}

template <int kLogL>
__global__ void __launch_bounds__(kWarps * 32) k_tile_tree(const TileTreeArgs a) {
    constexpr int L = 1 << kLogL;
    constexpr int kSlots = 32 * L;
    __shared__ int16_t slot_of[kSlots];
    for (int s = threadIdx.x; s < kSlots; s += blockDim.x)
        slot_of[s] = static_cast<int16_t>(s < (1 << a.depth) ? slot_tile(s, a.depth, a.n_tiles) : -1);
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    // shuffle level after which lane r << shard_level holds shard r's node
    const int shard_level = (a.depth < 5 ? a.depth : 5) - a.shard_depth;

    for (int t = blockIdx.x * kWarps + warp; t < a.T; t += gridDim.x * kWarps) {
        const bool act = a.active ? (a.active[t] != 0) : true;
        if (!act) {
            if (a.shard_mode) {
                if (lane == 0) a.records[t] = rlk_partial_t{0.0f, 0.0f, 0.0f, 0u};
            } else {
                if (lane < a.n_shards)
                    a.records[static_cast<int64_t>(lane) * a.T + t] =
                        rlk_partial_t{0.0f, 0.0f, 0.0f, 0u};
                if (lane == 0) {
                    a.out_logprob[t] = 0.0f;
                    a.out_lse[t] = 0.0f;
                }
            }
            continue;
        }
        const float2* row = a.partials + static_cast<int64_t>(t) * a.ld;
        MaxSum v[L];
#pragma unroll
        for (int j = 0; j < L; ++j) {
            const int tile = slot_of[lane * L + j];
            if (tile >= 0) {
                const float2 p = row[tile];
                v[j].m = p.x;
                v[j].s = p.y;
            } else {
                v[j].m = -CUDART_INF_F;
                v[j].s = 0.0f;
            }
        }
#pragma unroll
        for (int w = L / 2; w >= 1; w >>= 1) {
#pragma unroll
            for (int i = 0; i < w; ++i) v[i] = contract_merge(v[2 * i], v[2 * i + 1]);
        }
        MaxSum x = v[0];
        MaxSum shard = x;
#pragma unroll
        for (int lv = 0; lv < 5; ++lv) {
            if (lv == shard_level) shard = x;
            MaxSum o;
            o.m = __shfl_xor_sync(0xffffffffu, x.m, 1 << lv);
            o.s = __shfl_xor_sync(0xffffffffu, x.s, 1 << lv);
            x = (lane & (1 << lv)) ? contract_merge(o, x) : contract_merge(x, o);
        }
        if (shard_level == 5) shard = x;

        const int64_t tg = a.targets[t];
        if (a.shard_mode) {
            if (lane == 0) {
                const bool owned = tg >= a.own_begin && tg < a.own_end;
                a.records[t] = rlk_partial_t{x.m, x.s, owned ? a.tgt_logit[t] : 0.0f,
                                             owned ? 1u : 0u};
            }
            continue;
        }
        const bool holds_shard = (lane & ((1 << shard_level) - 1)) == 0 &&
                                 (lane >> shard_level) < a.n_shards;
        if (holds_shard) {
            const int r = lane >> shard_level;
            const bool owned = tg >= a.shard_vbegin[r] && tg < a.shard_vbegin[r + 1];
            a.records[static_cast<int64_t>(r) * a.T + t] =
                rlk_partial_t{shard.m, shard.s, owned ? a.tgt_logit[t] : 0.0f, owned ? 1u : 0u};
        }
        if (lane == 0) {
            if (tg >= 0 && tg < a.V_total) {
                const float lse = __fadd_rn(x.m, contract_log(x.s));
                a.out_lse[t] = lse;
                a.out_logprob[t] = __fsub_rn(a.tgt_logit[t], lse);
            } else {
                a.out_lse[t] = CUDART_NAN_F;
                a.out_logprob[t] = CUDART_NAN_F;
                report(a.status, RLK_ERR_TARGET_RANGE);
            }
        }
    }
}

// Records of n_shards shards (a power of two) merged pairwise in shard
// order, one thread per token.
__global__ void __launch_bounds__(256) k_shard_merge(const ShardMergeArgs a) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= a.T) return;
    if (a.active && a.active[t] == 0) {
        a.out_logprob[t] = 0.0f;
        a.out_lse[t] = 0.0f;
        return;
    }
    MaxSum v[RLK_MAX_SHARDS];
    int owners = 0;
    float tgt = 0.0f;
    for (int r = 0; r < a.n_shards; ++r) {
        const rlk_partial_t p = a.parts[r][t];
        v[r].m = p.m;
        v[r].s = p.s;
        if (p.owned) {
            ++owners;
            tgt = p.tgt;
        }
    }
    for (int w = a.n_shards / 2; w >= 1; w >>= 1)
        for (int i = 0; i < w; ++i) v[i] = contract_merge(v[2 * i], v[2 * i + 1]);
    if (owners == 1) {
        const float lse = __fadd_rn(v[0].m, contract_log(v[0].s));
        a.out_lse[t] = lse;
        a.out_logprob[t] = __fsub_rn(tgt, lse);
    } else {
        a.out_lse[t] = CUDART_NAN_F;
        a.out_logprob[t] = CUDART_NAN_F;
        report(a.status, RLK_ERR_TARGET_RANGE);
    }
}

template <int kLogL>
cudaError_t launch_tree(const TileTreeArgs& a, cudaStream_t stream) {
    int blocks = (a.T + kWarps - 1) / kWarps;
    if (blocks > 4096) blocks = 4096;
    k_tile_tree<kLogL><<<blocks, kWarps * 32, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tile_tree(const TileTreeArgs& a, cudaStream_t stream) {
    const int log_l = a.depth > 5 ? a.depth - 5 : 0;
    switch (log_l) {
        case 0: return launch_tree<0>(a, stream);
        case 1: return launch_tree<1>(a, stream);
        case 2: return launch_tree<2>(a, stream);
        case 3: return launch_tree<3>(a, stream);
        case 4: return launch_tree<4>(a, stream);
        case 5: return launch_tree<5>(a, stream);
        case 6: return launch_tree<6>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_shard_merge(const ShardMergeArgs& a, cudaStream_t stream) {
    const int blocks = (a.T + 255) / 256;
    k_shard_merge<<<blocks, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace rlk
