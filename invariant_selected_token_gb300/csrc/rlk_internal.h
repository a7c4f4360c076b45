// Internal launch interface between the host dispatcher (rlk_api.cu) and the
// kernels (rlk_logits.cu: logits GEMM + fused tile epilogue; rlk_merge.cu:
// tile tree, shard records, finalize, cross-shard merge).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/rlk.h"

namespace rlk {

constexpr int kTileM = 128;          // token rows per MMA tile
constexpr int kTileN = 256;          // vocabulary rows per MMA tile (two contract tiles)
constexpr int kVocabTile = RLK_VOCAB_TILE;
constexpr int kBlockK = RLK_K_BLOCK; // K elements per pipeline stage (one 128-byte swizzle row)
constexpr int kMaxTreeDepth = 11;    // 2048 tiles

struct TilePartialsArgs {
    const int32_t* targets;   // [T] global vocabulary ids
    const uint8_t* active;    // [T] or nullptr
    float2* partials;         // [T][n_tiles] (m, s); unused in debug mode
    float* tgt_logit;         // [T] target logit, written by the owning tile
    float* dbg_logits;        // [T][V_local], debug mode only
    int32_t* status;          // device status bits or nullptr
    int64_t v_offset;         // global vocabulary id of W row 0
    int T;
    int V_local;              // rows of W this launch covers
    int n_tiles;              // ceil(V_local / 128): row stride of partials
    int k_blocks;             // H / 64
    int a_box_rows;           // rows of the hidden TMA box: 128, or roundup(T, 8) when T <= 128
    int test_drop_stage;      // test only: CTA 0 never loads its first stage (wait runs out)
    // backward (gradient epilogue) only
    const float* lse;         // [T] forward log-sum-exp
    const float* grad;        // [T] dL/dlogprob
    uint16_t* G;              // bf16 [T][ldG] logit gradient
    int64_t ldG;
    int64_t V_total;          // for the target-range check
    // saving forward only: the fp32 logits [T][ld_logits] (16-byte aligned, ld % 4 == 0)
    float* logits_out;
    int64_t ld_logits;
};

// kEpiSave: kEpiPartials plus every row's fp32 logits stored for the backward
enum TileEpilogue { kEpiPartials = 0, kEpiDebugLogits = 1, kEpiGrad = 2, kEpiSave = 3 };

// hidden map: bf16 [T][H], box 64 x a_box_rows; weight map: bf16 [V_local][H], box 64 x 256.
cudaError_t launch_tile_partials(const CUtensorMap& map_hidden, const CUtensorMap& map_w,
                                 const TilePartialsArgs& a, int epilogue, int num_sms,
                                 cudaStream_t stream);
cudaError_t prepare_tile_partials_kernels();

struct TileTreeArgs {
    const float2* partials;   // [T][ld]
    int64_t ld;
    const float* tgt_logit;   // [T]
    const int32_t* targets;   // [T], or nullptr: lse only (no target, no logprob)
    const uint8_t* active;    // [T] or nullptr
    int32_t* status;
    int T;
    int n_tiles;              // leaves of this tree
    int depth;                // ceil(log2(n_tiles))
    int shard_depth;          // log2(n_shards) (full mode); 0 in shard mode
    int n_shards;
    int shard_mode;           // 0: full tree -> records + outputs; 1: one shard's record
    int64_t shard_vbegin[RLK_MAX_SHARDS + 1];  // vocabulary boundaries (full mode)
    int64_t own_begin, own_end;                 // ownership range (shard mode)
    int64_t V_total;
    float* out_logprob;       // [T] (full mode)
    float* out_lse;           // [T] (full mode)
    rlk_partial_t* records;   // full: [n_shards][T]; shard: [T]
};

cudaError_t launch_tile_tree(const TileTreeArgs& a, int num_sms, cudaStream_t stream);
// Sets the warp-per-token tree kernels' shared-memory limit (staged rows).
cudaError_t prepare_tree_kernels();

// materialised logits [T][ld] (fp32 or bf16) -> the same per-tile pairs / target logits
// resident_ctas: CTAs of the kernel (for this dtype) that fit on the device
// at once; the grid never exceeds it (one persistent wave).
cudaError_t launch_mat_tile_partials(const void* logits, int dtype, int64_t ld,
                                     const int32_t* targets, const uint8_t* active, int T, int V,
                                     float2* partials, float* tgt_logit, int resident_ctas,
                                     cudaStream_t stream);
// Sets the kernels' shared-memory limits and reports the CTAs per SM of
// k_mat_tile_partials for fp32 [0] and bf16 [1] logits.
cudaError_t prepare_mat_kernels(int* ctas_per_sm);
// G[t][v] (bf16, row stride ldG) from fp32 logits [T][ld] (16-byte aligned, ld % 4 == 0):
// the backward epilogue's arithmetic on the saved logits instead of recomputed ones
cudaError_t launch_grad_from_logits(const float* logits, int64_t ld, const int32_t* targets,
                                    const uint8_t* active, const float* grad, const float* lse,
                                    int T, int V, uint16_t* G, int64_t ldG, int32_t* status,
                                    int num_sms, cudaStream_t stream);
// out[t][v] = RN(l[t][v] - lse[t])
cudaError_t launch_log_softmax_out(const void* logits, int dtype, int64_t ld, const float* lse,
                                   const uint8_t* active, int T, int V, float* out, int num_sms,
                                   cudaStream_t stream);

struct GemmArgs {
    float* out;               // [splits][M][ld_out] fp32
    int64_t ld_out;
    int64_t split_stride;     // elements between split partials
    int M, N;
    int k_blocks;             // ceil(K / 64)
    int kb_per_split;
    int splits;
    bool vec_store;           // out rows 16-byte aligned
    bool n_fastest;           // raster: N tiles fastest (CTAs side by side share the A slice)
    int n_band;               // n_fastest: N tiles per band (all M tiles visit a band's
                              // N tiles before the next band); 0 = all N tiles
    int test_drop_stage;      // test only: CTA 0 never loads its first stage (wait runs out)
    int32_t* status;
};

// A MN-major or K-major, B MN-major; 128 x 256 tiles, fixed K ranges per split.
cudaError_t launch_gemm_f32(const CUtensorMap& map_a, const CUtensorMap& map_b, bool a_mn,
                            bool b_mn, const GemmArgs& g, int num_sms, cudaStream_t stream);
cudaError_t prepare_gemm_kernels();
cudaError_t launch_sum_splits(const float* parts, int64_t split_stride, int splits, int64_t n,
                              float* out, int num_sms, cudaStream_t stream);

struct RmsNormArgs {
    const uint16_t* x;        // bf16 [T][H]
    const uint16_t* res;      // bf16 [T][H] or nullptr
    const uint16_t* gamma;    // bf16 [H]
    float eps;
    int T, H;
    uint16_t* y;              // bf16 [T][H]
    uint16_t* res_out;        // bf16 [T][H] (x + res) or nullptr
};

cudaError_t launch_rmsnorm(const RmsNormArgs& a, int num_sms, cudaStream_t stream);

// Position-weighted hash of a contract primitive over fp32 bit patterns
// [first, first + count): which 0 exp, 1 exp two lanes at a time, 2 log, 3 rsqrt.
cudaError_t launch_primitive_hash(int which, uint32_t first, uint64_t count, uint64_t* out,
                                  int num_sms, cudaStream_t stream);

struct ShardMergeArgs {
    const rlk_partial_t* parts[RLK_MAX_SHARDS];
    int n_shards;
    int T;
    const uint8_t* active;
    float* out_logprob;
    float* out_lse;
    int32_t* status;
};

cudaError_t launch_shard_merge(const ShardMergeArgs& a, cudaStream_t stream);

}  // namespace rlk
