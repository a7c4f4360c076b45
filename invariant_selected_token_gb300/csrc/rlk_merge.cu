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

// Merge a thread's node of one token's tree: its L = 2^kLogL slots of the
// perfect tree (levels 1 .. kLogL).  In a bisection of k tiles over 2^h
// slots (larger half first), slot j holds a tile exactly when the h-bit
// reversal of j is below k, and the tiles fill the held slots in order.  A
// thread's node holds between L/2 and L tiles (bisection keeps the nodes of
// one depth within one tile of each other, and the tree has 2^depth slots
// for at most 2^depth and more than 2^(depth-1) tiles), so every even slot
// 2i holds a tile (its reversal is that of i, below L/2), and the odd slot
// 2i+1 holds one exactly when the (h-1)-bit reversal of i is below k - L/2.
// Level 1 therefore merges a pair only where the odd slot is held -- a
// lone even slot is its own level-1 node, as in the bisection tree, whose
// nodes never see an empty operand -- and levels 2 .. kLogL, over nodes that
// all hold tiles, run as a binary counter (a node is formed as soon as both
// children exist).  load(k) returns tile k's (max, sum) pair; `present`
// says whether the node holds any tile (only L = 1 nodes can be empty).
template <int kLogL, typename Load>
__device__ __forceinline__ MaxSum merge_run(const SlotRun& run, Load load, bool& present) {
    MaxSum x;
    if constexpr (kLogL == 0) {
        present = run.count > 0;
        x.m = -CUDART_INF_F;
        x.s = 0.0f;
        if (present) {
            const float2 p = load(run.first);
            x.m = p.x;
            x.s = p.y;
        }
    } else {
        constexpr int kPairs = 1 << (kLogL - 1);
        const int odd_limit = run.count - kPairs;
        MaxSum pend[kLogL];
        int rel = 0;
#pragma unroll
        for (int i = 0; i < kPairs; ++i) {
            const float2 p = load(run.first + rel);
            ++rel;
            x.m = p.x;
            x.s = p.y;
            const int rev =
                kLogL > 1 ? static_cast<int>(__brev(static_cast<unsigned>(i)) >> (33 - kLogL)) : 0;
            if (rev < odd_limit) {
                const float2 q = load(run.first + rel);
                ++rel;
                MaxSum y;
                y.m = q.x;
                y.s = q.y;
                x = contract_merge(x, y);
            }
            int level = 0;
#pragma unroll
            for (; level < kLogL - 1; ++level) {
                if (!(i & (1 << level))) break;
                x = contract_merge(pend[level], x);  // left sibling + this node
            }
            if (level < kLogL - 1) pend[level] = x;
        }
        present = true;
    }
    return x;
}

// One merge level across lanes: partner lane ^ (1 << lv), the lower lane
// left; a side without tiles leaves the other unchanged.
__device__ __forceinline__ MaxSum shuffle_level(MaxSum x, bool& xp, int lane, int lv) {
    MaxSum o;
    o.m = __shfl_xor_sync(0xffffffffu, x.m, 1 << lv);
    o.s = __shfl_xor_sync(0xffffffffu, x.s, 1 << lv);
    const bool op = __shfl_xor_sync(0xffffffffu, xp ? 1 : 0, 1 << lv) != 0;
    MaxSum r = x;
    if (xp && op) r = (lane & (1 << lv)) ? contract_merge(o, x) : contract_merge(x, o);
    else if (op) r = o;
    xp = xp || op;
    return r;
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

// One warp per token, kTreeWarps warps per CTA.  The warp copies the
// token's row of tile pairs into shared memory (coalesced 8-byte copies:
// rows are n_tiles pairs apart, so only 8-byte aligned), then lane l merges
// its node of the tree (slots [l*L, (l+1)*L), a contiguous run of tiles)
// from there, and five shuffle levels finish the token.
constexpr int kTreeWarps = 4;

template <int kLogL>
__global__ void __launch_bounds__(kTreeWarps * 32) k_tile_tree(const TileTreeArgs a) {
    extern __shared__ float2 tree_rows[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    float2* row_sm = tree_rows + static_cast<int64_t>(warp) * a.n_tiles;
    const SlotRun run = slot_run<5>(lane, a.depth, a.n_tiles);
    // cross-lane level after which lane r << shard_level holds shard r's node
    const int shard_level = (a.depth < 5 ? a.depth : 5) - a.shard_depth;
    ptx::grid_dependency_wait();   // the tile pairs are the previous kernel's output
    ptx::grid_dependents_launch();

    for (int t = blockIdx.x * kTreeWarps + warp; t < a.T; t += gridDim.x * kTreeWarps) {
        const bool act = a.active ? (a.active[t] != 0) : true;
        if (!act) {
            if (lane == 0) write_inactive(a, t);
            continue;
        }
        const float2* row = a.partials + static_cast<int64_t>(t) * a.ld;
        __syncwarp();  // the previous token's reads of the buffer are done
        for (int k = lane; k < a.n_tiles; k += 32) {
            const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(row_sm + k));
            asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(row + k)
                         : "memory");
        }
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
        __syncwarp();
        bool xp;
        MaxSum x = merge_run<kLogL>(run, [&](int k) { return row_sm[k]; }, xp);
        MaxSum shard = x;
#pragma unroll
        for (int lv = 0; lv < 5; ++lv) {
            if (lv == shard_level) shard = x;
            x = shuffle_level(x, xp, lane, lv);
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
    __shared__ MaxSum warp_node[8];
    __shared__ bool warp_present[8];
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
        const float2* row = a.partials + static_cast<int64_t>(t) * a.ld;
        bool xp;
        MaxSum x = merge_run<kLogL>(run, [&](int k) { return row[k]; }, xp);
        MaxSum shard = x;
#pragma unroll
        for (int lv = 0; lv < 5; ++lv) {
            if (lv == shard_level) shard = x;
            x = shuffle_level(x, xp, lane, lv);
        }
        if (!a.shard_mode && shard_level < 5 && (tid & ((1 << shard_level) - 1)) == 0 &&
            (tid >> shard_level) < a.n_shards)
            write_shard_record(a, t, tid >> shard_level, shard);
        if (lane == 0) {
            warp_node[warp] = x;
            warp_present[warp] = xp;
        }
        __syncthreads();
        if (tid == 0) {
            MaxSum v[8];
            bool vp[8];
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                v[w] = warp_node[w];
                vp[w] = warp_present[w];
            }
#pragma unroll
            for (int lv = 5; lv < 8; ++lv) {
                const int stride = 1 << (lv - 5);
                if (!a.shard_mode && lv == shard_level) {
                    for (int r = 0; r < a.n_shards; ++r) write_shard_record(a, t, r, v[r * stride]);
                }
#pragma unroll
                for (int i = 0; i < 8; i += 2 * stride) {
                    if (vp[i] && vp[i + stride]) v[i] = contract_merge(v[i], v[i + stride]);
                    else if (vp[i + stride]) v[i] = v[i + stride];
                    vp[i] = vp[i] || vp[i + stride];
                }
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
cudaError_t launch_dependent(Kernel kernel, int blocks, int threads, size_t smem,
                             const TileTreeArgs& a, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

// Largest staged rows: RLK_MAX_VOCAB / 128 tiles per warp.
constexpr size_t kTreeSmemMax = size_t(kTreeWarps) * (RLK_MAX_VOCAB / kVocabTile) * sizeof(float2);

template <int kLogL>
cudaError_t launch_warp_tree(const TileTreeArgs& a, int num_sms, cudaStream_t stream) {
    const size_t smem = size_t(kTreeWarps) * a.n_tiles * sizeof(float2);
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_tile_tree<kLogL>,
                                                                  kTreeWarps * 32, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    int64_t blocks = (int64_t(a.T) + kTreeWarps - 1) / kTreeWarps;
    if (blocks > int64_t(per_sm) * num_sms) blocks = int64_t(per_sm) * num_sms;
    return launch_dependent(k_tile_tree<kLogL>, int(blocks), kTreeWarps * 32, smem, a, stream);
}

template <int kLogL>
cudaError_t launch_cta_tree(const TileTreeArgs& a, cudaStream_t stream) {
    const int blocks = a.T < 65535 ? a.T : 65535;
    return launch_dependent(k_tile_tree_cta<kLogL>, blocks, 256, 0, a, stream);
}

template <int kLogL>
cudaError_t allow_tree_smem() {
    return cudaFuncSetAttribute(k_tile_tree<kLogL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(kTreeSmemMax));
}

}  // namespace

cudaError_t prepare_tree_kernels() {
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = allow_tree_smem<0>();
    if (e == cudaSuccess) e = allow_tree_smem<1>();
    if (e == cudaSuccess) e = allow_tree_smem<2>();
    if (e == cudaSuccess) e = allow_tree_smem<3>();
    if (e == cudaSuccess) e = allow_tree_smem<4>();
    if (e == cudaSuccess) e = allow_tree_smem<5>();
    if (e == cudaSuccess) e = allow_tree_smem<6>();
    return e;
}

// RLK_TEST_TREE_THREADS=32|256 forces one layout; tests use it to show that
// the layout never changes a bit.
cudaError_t launch_tile_tree(const TileTreeArgs& a, int num_sms, cudaStream_t stream) {
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
        case 0: return launch_warp_tree<0>(a, num_sms, stream);
        case 1: return launch_warp_tree<1>(a, num_sms, stream);
        case 2: return launch_warp_tree<2>(a, num_sms, stream);
        case 3: return launch_warp_tree<3>(a, num_sms, stream);
        case 4: return launch_warp_tree<4>(a, num_sms, stream);
        case 5: return launch_warp_tree<5>(a, num_sms, stream);
        case 6: return launch_warp_tree<6>(a, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_shard_merge(const ShardMergeArgs& a, cudaStream_t stream) {
    const int blocks = (a.T + 255) / 256;
    k_shard_merge<<<blocks, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace rlk
