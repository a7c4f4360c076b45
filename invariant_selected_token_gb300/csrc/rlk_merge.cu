// Fixed-order merges of the per-tile (max, sum-exp) pairs: the tile tree,
// the shard records, the final log-sum-exp and logprob, and the separate
// cross-shard merge ("cross-rank LSE merge" and "fixed rank reduction
// order" in the strict-path table of "vLLM RL-Kernel v0.1.0: ROCm 上での
// ビット単位のトレーニング-ロールアウト一貫性").
//
// The contract's tile tree is a recursive bisection of the tile range (a
// node of k tiles gives ceil(k/2) to its left child).  These kernels
// evaluate exactly that tree as a perfect binary tree over 2^depth slots:
// walking the bisection down to single slots places every tile in one slot
// and leaves the remaining slots empty (always in right subtrees).  An empty
// slot carries (-inf, 0), which the merge passes through bit for bit, so
// every non-empty node of the perfect tree holds the bits of the
// corresponding bisection node.
//
// A token's slots are spread over P threads (P = 32: one warp per token,
// for large batches; P = 256: one CTA per token, for small batches where the
// tree's latency is the cost).  Thread u owns slots [u*L, (u+1)*L) and merges
// them in registers (levels 1 .. log2 L); the levels above pair thread u with
// u^1, u^2, ... (shuffles inside a warp, shared memory across warps), always
// with the lower thread as the left operand.  The shard nodes (depth
// log2 n_shards) are complete after the level that finishes them; their
// records are written from there, and the levels above them are the pairwise
// merge of the records in shard order -- the same merges rlk_lse_merge
// performs.  Both layouts run the same merges on the same operands, so the
// choice between them never changes a bit.
#include <cstdint>
#include <cstdlib>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "rlk_contract.cuh"
#include "rlk_internal.h"
#include "rlk_ptx.cuh"

namespace rlk {
namespace {

// batches up to this many tokens use one CTA per token
constexpr int kCtaTreeMaxTokens = 256;

__device__ __forceinline__ void report(int32_t* status, int code) {
    if (status) atomicOr(status, 1 << code);
}

// The slots a thread owns form one node of the perfect tree; its tiles are a
// contiguous run (the bisection keeps tile order): `first` tile, `count` tiles.
struct SlotRun {
    int first;
    int count;
};

// Node of thread u when a token's 2^max(depth, log2 P) slots are spread over
// P = 2^kLogP threads.  The contract's tree occupies the first 2^depth slots;
// walking its bisection down u's bits (most significant first) gives the
// node.  With fewer slots than threads, thread u holds slot u alone.
template <int kLogP>
__device__ __forceinline__ SlotRun slot_run(int u, int depth, int n_tiles) {
    SlotRun r;
    r.first = 0;
    r.count = n_tiles;
    int levels = kLogP;
    if (depth < kLogP) {
        if (u >= (1 << depth)) {
            r.count = 0;
            return r;
        }
        levels = depth;
    }
    for (int b = levels - 1; b >= 0; --b) {
        const int left = (r.count + 1) >> 1;
        if ((u >> b) & 1) {
            r.first += left;
            r.count -= left;
        } else {
            r.count = left;
        }
    }
    return r;
}

// Load a thread's L slots of one token's tile pairs and merge them in
// registers (levels 1 .. log2 L of the perfect tree).  In a bisection of k
// tiles over 2^h slots (larger half first), slot j holds a tile exactly when
// the h-bit reversal of j is below k, and the tiles fill the held slots in
// order.
template <int L>
__device__ __forceinline__ MaxSum merge_own_slots(const float2* row, const SlotRun& run) {
    constexpr int kLogL = (L >= 64) ? 6 : (L >= 32) ? 5 : (L >= 16) ? 4 : (L >= 8) ? 3
                        : (L >= 4) ? 2 : (L >= 2) ? 1 : 0;
    MaxSum v[L];
    int rel = 0;
#pragma unroll
    for (int j = 0; j < L; ++j) {
        const int rev = kLogL ? static_cast<int>(__brev(static_cast<unsigned>(j)) >> (32 - kLogL)) : 0;
        if (rev < run.count) {
            const float2 p = row[run.first + rel];
            ++rel;
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
    return v[0];
}

// One merge level across lanes: partner lane ^ (1 << lv), the lower lane left.
__device__ __forceinline__ MaxSum shuffle_level(MaxSum x, int lane, int lv) {
    MaxSum o;
    o.m = __shfl_xor_sync(0xffffffffu, x.m, 1 << lv);
    o.s = __shfl_xor_sync(0xffffffffu, x.s, 1 << lv);
    return (lane & (1 << lv)) ? contract_merge(o, x) : contract_merge(x, o);
}

__device__ __forceinline__ void write_inactive(const TileTreeArgs& a, int t) {
    if (a.shard_mode) {
        a.records[t] = rlk_partial_t{0.0f, 0.0f, 0.0f, 0u};
    } else {
        for (int r = 0; r < a.n_shards; ++r)
            a.records[static_cast<int64_t>(r) * a.T + t] = rlk_partial_t{0.0f, 0.0f, 0.0f, 0u};
        if (a.out_logprob) a.out_logprob[t] = 0.0f;
        a.out_lse[t] = 0.0f;
    }
}

__device__ __forceinline__ void write_shard_record(const TileTreeArgs& a, int t, int r, MaxSum n) {
    const int64_t tg = a.targets ? a.targets[t] : -1;
    const bool owned = a.targets && tg >= a.shard_vbegin[r] && tg < a.shard_vbegin[r + 1];
    a.records[static_cast<int64_t>(r) * a.T + t] =
        rlk_partial_t{n.m, n.s, owned ? a.tgt_logit[t] : 0.0f, owned ? 1u : 0u};
}

// Root of a token's tree -> its shard-mode record, or the final lse / logprob.
__device__ __forceinline__ void finish_token(const TileTreeArgs& a, int t, MaxSum root) {
    if (!a.targets) {  // log_softmax: the log-sum-exp alone
        a.out_lse[t] = __fadd_rn(root.m, contract_log(root.s));
        return;
    }
    const int64_t tg = a.targets[t];
    if (a.shard_mode) {
        const bool owned = tg >= a.own_begin && tg < a.own_end;
        a.records[t] = rlk_partial_t{root.m, root.s, owned ? a.tgt_logit[t] : 0.0f,
                                     owned ? 1u : 0u};
        return;
    }
    if (tg >= 0 && tg < a.V_total) {
        const float lse = __fadd_rn(root.m, contract_log(root.s));
        a.out_lse[t] = lse;
        a.out_logprob[t] = __fsub_rn(a.tgt_logit[t], lse);
    } else {
        a.out_lse[t] = CUDART_NAN_F;
        a.out_logprob[t] = CUDART_NAN_F;
        report(a.status, RLK_ERR_TARGET_RANGE);
    }
}

// One warp per token.  Lane l owns slots [l*L, (l+1)*L).
template <int kLogL>
__global__ void __launch_bounds__(256) k_tile_tree(const TileTreeArgs a) {
    constexpr int L = 1 << kLogL;
    constexpr int kWarps = 8;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const SlotRun run = slot_run<5>(lane, a.depth, a.n_tiles);
    // cross-lane level after which lane r << shard_level holds shard r's node
    const int shard_level = (a.depth < 5 ? a.depth : 5) - a.shard_depth;
    ptx::grid_dependency_wait();   // the tile pairs are the previous kernel's output
    ptx::grid_dependents_launch();

    for (int t = blockIdx.x * kWarps + warp; t < a.T; t += gridDim.x * kWarps) {
        const bool act = a.active ? (a.active[t] != 0) : true;
        if (!act) {
            if (lane == 0) write_inactive(a, t);
            continue;
        }
        MaxSum x = merge_own_slots<L>(a.partials + static_cast<int64_t>(t) * a.ld, run);
        MaxSum shard = x;
#pragma unroll
        for (int lv = 0; lv < 5; ++lv) {
            if (lv == shard_level) shard = x;
            x = shuffle_level(x, lane, lv);
        }
        if (shard_level == 5) shard = x;
        if (!a.shard_mode && (lane & ((1 << shard_level) - 1)) == 0 &&
            (lane >> shard_level) < a.n_shards)
            write_shard_record(a, t, lane >> shard_level, shard);
        if (lane == 0) finish_token(a, t, x);
    }
}

// One 256-thread CTA per token.  Thread u owns slots [u*L, (u+1)*L); five
// shuffle levels inside each warp, then the eight warp nodes merge pairwise
// in shared memory (levels 5, 6, 7).
template <int kLogL>
__global__ void __launch_bounds__(256) k_tile_tree_cta(const TileTreeArgs a) {
    constexpr int L = 1 << kLogL;
    __shared__ MaxSum warp_node[8];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const SlotRun run = slot_run<8>(tid, a.depth, a.n_tiles);
    const int shard_level = (a.depth < 8 ? a.depth : 8) - a.shard_depth;
    ptx::grid_dependency_wait();   // the tile pairs are the previous kernel's output
    ptx::grid_dependents_launch();

    for (int t = blockIdx.x; t < a.T; t += gridDim.x) {
        const bool act = a.active ? (a.active[t] != 0) : true;
        if (!act) {
            if (tid == 0) write_inactive(a, t);
            continue;
        }
        MaxSum x = merge_own_slots<L>(a.partials + static_cast<int64_t>(t) * a.ld, run);
        MaxSum shard = x;
#pragma unroll
        for (int lv = 0; lv < 5; ++lv) {
            if (lv == shard_level) shard = x;
            x = shuffle_level(x, lane, lv);
        }
        if (!a.shard_mode && shard_level < 5 && (tid & ((1 << shard_level) - 1)) == 0 &&
            (tid >> shard_level) < a.n_shards)
            write_shard_record(a, t, tid >> shard_level, shard);
        if (lane == 0) warp_node[warp] = x;
        __syncthreads();
        if (tid == 0) {
            MaxSum v[8];
#pragma unroll
            for (int w = 0; w < 8; ++w) v[w] = warp_node[w];
#pragma unroll
            for (int lv = 5; lv < 8; ++lv) {
                const int stride = 1 << (lv - 5);
                if (!a.shard_mode && lv == shard_level) {
                    for (int r = 0; r < a.n_shards; ++r) write_shard_record(a, t, r, v[r * stride]);
                }
#pragma unroll
                for (int i = 0; i < 8; i += 2 * stride) v[i] = contract_merge(v[i], v[i + stride]);
            }
            if (!a.shard_mode && shard_level == 8) write_shard_record(a, t, 0, v[0]);
            finish_token(a, t, v[0]);
        }
        __syncthreads();
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

// Launched with programmatic dependent launch: the grid may start while the
// logits kernel finishes, and waits for it before reading the tile pairs.
template <typename Kernel>
cudaError_t launch_dependent(Kernel kernel, int blocks, const TileTreeArgs& a,
                             cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <int kLogL>
cudaError_t launch_warp_tree(const TileTreeArgs& a, cudaStream_t stream) {
    int blocks = (a.T + 7) / 8;
    if (blocks > 4096) blocks = 4096;
    return launch_dependent(k_tile_tree<kLogL>, blocks, a, stream);
}

template <int kLogL>
cudaError_t launch_cta_tree(const TileTreeArgs& a, cudaStream_t stream) {
    const int blocks = a.T < 65535 ? a.T : 65535;
    return launch_dependent(k_tile_tree_cta<kLogL>, blocks, a, stream);
}

}  // namespace

// RLK_TEST_TREE_THREADS=32|256 forces one layout; tests use it to show that
// the layout never changes a bit.
cudaError_t launch_tile_tree(const TileTreeArgs& a, cudaStream_t stream) {
    bool per_cta = a.T <= kCtaTreeMaxTokens;
    if (const char* f = std::getenv("RLK_TEST_TREE_THREADS")) per_cta = std::atoi(f) == 256;
    if (per_cta) {
        switch (a.depth > 8 ? a.depth - 8 : 0) {
            case 0: return launch_cta_tree<0>(a, stream);
            case 1: return launch_cta_tree<1>(a, stream);
            case 2: return launch_cta_tree<2>(a, stream);
            case 3: return launch_cta_tree<3>(a, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (a.depth > 5 ? a.depth - 5 : 0) {
        case 0: return launch_warp_tree<0>(a, stream);
        case 1: return launch_warp_tree<1>(a, stream);
        case 2: return launch_warp_tree<2>(a, stream);
        case 3: return launch_warp_tree<3>(a, stream);
        case 4: return launch_warp_tree<4>(a, stream);
        case 5: return launch_warp_tree<5>(a, stream);
        case 6: return launch_warp_tree<6>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_shard_merge(const ShardMergeArgs& a, cudaStream_t stream) {
    const int blocks = (a.T + 255) / 256;
    k_shard_merge<<<blocks, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace rlk
