// Logits GEMM with the fused per-tile epilogue (the "local reduction" and
// "target ownership" of the strict-path table's Linear-logprob row, in
// "vLLM RL-Kernel v0.1.0: ROCm 上でのビット単位のトレーニング-ロールアウト一貫性").
//
// One persistent CTA per SM walks output tiles of 128 tokens x 256
// vocabulary rows, vocabulary-major within bands of 32 token tiles (all
// token tiles of a band run side by side on one W slice, so each 2 MB slice
// of W is read from HBM once per band and shared through L2).  Warp roles:
//   warp 0      TMA producer: 4-stage ring of (hidden 128x64, W 256x64) bf16
//               boxes, 128-byte swizzled;
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma kind::f16, M=128,
//               N=256, K=16, cta_group::1, fp32 accumulator in TMEM, K in
//               ascending order, the first step overwriting; two
//               accumulators (2 x 256 TMEM columns) so the epilogue of tile
//               i overlaps the mainloop of tile i+1;
//   warps 2-5   epilogue: one thread per token row (TMEM lane), 128 columns
//               per contract tile read with tcgen05.ld, reduced in registers
//               to (max, pairwise-tree sum of exp(logit - max)) and the
//               target's logit picked if the tile owns it.  The [T, V]
//               logits never reach HBM.
//
// Invariance: every logit comes from the same instruction sequence whatever
// T, the row position or the launch shape, so the per-tile values depend on
// the token and the tile only.  There is no split over K on any path.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "rlk_contract.cuh"
#include "rlk_internal.h"
#include "rlk_ptx.cuh"

namespace rlk {
namespace {

constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr uint32_t kStageBytesA = kTileM * kBlockK * 2;  // 16 KB
constexpr uint32_t kStageBytesB = kTileN * kBlockK * 2;  // 32 KB
constexpr uint32_t kTmemCols = 512;                      // two 256-column accumulators
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kTileM, kTileN);
constexpr int kSmemBytes = kStages * (kStageBytesA + kStageBytesB) + 1024 /*alignment slack*/
                           + 256 /*barriers, TMEM address, abort flag*/;
// The backward epilogue turns each warp's 32 rows x 64 columns of bf16 G
// around in shared memory before storing them, so that every store
// instruction writes whole 128-byte row segments.  Row pitch 72 elements
// (144 bytes, an odd number of 16-byte chunks): the eight rows one 16-byte
// access phase touches fall in distinct bank quads.
constexpr int kGradPitch = 72;
constexpr uint32_t kGradStageBytes = 4 * 32 * kGradPitch * 2;  // 18 KB
// The saving forward turns 32 rows x 32 columns of fp32 logits around the
// same way (pitch 36 floats, again 144 bytes) in the same 18 KB.
constexpr int kSavePitch = 36;
static_assert(4 * 32 * kSavePitch * 4 == kGradStageBytes, "one staging region for both");
__host__ __device__ constexpr bool staged_epi(int epi) { return epi == kEpiGrad || epi == kEpiSave; }
template <int kEpi>
constexpr int smem_bytes_of() {
    return kSmemBytes + (staged_epi(kEpi) ? static_cast<int>(kGradStageBytes) : 0);
}

// Ring depth for a hidden box of `a_rows` rows: as many (hidden box, W box)
// stages as fit in a CTA's shared memory (227 KB) next to the barriers and,
// for the backward, the G staging rows; at most kMaxStages.  A full 128-row
// box gives the 4 stages above; the small boxes of decode batches (at most
// 128 tokens, box rows roundup(T, 8)) give 6 stages up to 40 rows and 5 up
// to 104 (with the G staging: 16 and 72): a deeper W stream where the MMAs
// are nearly free.  Host and device compute it alike.
constexpr int kMaxStages = 6;
constexpr int kSmemLimit = 232448;
__host__ __device__ constexpr int ring_stages(int a_rows, bool grad) {
    const int budget = kSmemLimit - 1024 - 256 - (grad ? static_cast<int>(kGradStageBytes) : 0);
    const int n = budget / (a_rows * kBlockK * 2 + static_cast<int>(kStageBytesB));
    return n > kMaxStages ? kMaxStages : n;
}
template <int kEpi>
constexpr int ring_smem_bytes(int a_rows) {
    return ring_stages(a_rows, staged_epi(kEpi)) * (a_rows * kBlockK * 2 + static_cast<int>(kStageBytesB)) +
           1024 + 256 + (staged_epi(kEpi) ? static_cast<int>(kGradStageBytes) : 0);
}

__device__ __forceinline__ void report(int32_t* status, int code) {
    if (status) atomicOr(status, 1 << code);
}

// Reduce one 128-column contract tile held in registers (v[c] = logit of
// column c; columns at or beyond ncols are padding) to (max, sum).
// The sum is the contract's 128-slot pairwise tree: (0+1), (2+3), ..., then
// pairs of those, seven levels.  A padding column is set to -inf, whose exp
// is +0, and x + 0 = x exactly for the non-negative terms here, so padding
// slots pass their partner through unchanged, as the contract requires.
// The arithmetic runs two columns per instruction (tile_reduce_x2), with
// the scalar evaluation's bits.
__device__ __forceinline__ MaxSum reduce_tile(float (&v)[kVocabTile], int ncols) {
    if (ncols < kVocabTile) {
#pragma unroll
        for (int c = 0; c < kVocabTile; ++c)
            if (c >= ncols) v[c] = -CUDART_INF_F;
    }
    uint64_t P[kVocabTile / 2];
#pragma unroll
    for (int k = 0; k < kVocabTile / 2; ++k) P[k] = f2_pack(v[2 * k], v[2 * k + 1]);
    return tile_reduce_x2(P);
}

// Backward epilogue: G[t, c] = bf16_RN(RN(g_t * d)) with d = RN(1 - p) at the
// target and -p elsewhere, p = rlk_exp(RN(l - lse_t)) -- the gradient of
// g_t * logprob_t with respect to the logits, from the same fp32 logits and
// the same exp the forward used.  Inactive rows write zeros; rows at or
// beyond T write nothing.  Called by the whole warp (lane = row0 + lane's
// row): each full 64-column half of the tile goes through the warp's staging
// rows `stage` and out in 128-byte row segments; a ragged last half is
// stored element by element.
__device__ __forceinline__ void grad_tile(const float (&v)[kVocabTile], const TilePartialsArgs& a,
                                          int t, int c0, int ncols, bool valid, int64_t tl,
                                          uint16_t* stage, int lane, int row0) {
    const bool row_ok = t < a.T;
    const float lse = valid ? a.lse[t] : 0.0f;
    const float gt = valid ? a.grad[t] : 0.0f;
    const uint64_t neg_lse = f2_splat(-lse);  // RN(l - lse) = RN(l + (-lse))
    const uint64_t g2 = f2_splat(gt);
    uint16_t* dst = a.G + static_cast<int64_t>(t) * a.ldG + c0;
#pragma unroll
    for (int q = 0; q < kVocabTile / 8; ++q) {
        const int half = q / 8;
        const bool staged = half * 64 + 64 <= ncols;  // the same for the whole warp
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // columns c, c + 1, two per instruction with the scalar bits
            const int c = q * 8 + 2 * i;
            w[i] = contract_grad_x2(f2_pack(v[c], v[c + 1]), neg_lse, g2, c == tl, c + 1 == tl,
                                    valid);
        }
        if (staged) {
            *reinterpret_cast<uint4*>(stage + lane * kGradPitch + (q % 8) * 8) =
                make_uint4(w[0], w[1], w[2], w[3]);
        } else if (row_ok) {
            if (q * 8 + 8 <= ncols) {
                *reinterpret_cast<uint4*>(dst + q * 8) = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (q * 8 + i < ncols)
                        dst[q * 8 + i] = static_cast<uint16_t>(w[i / 2] >> (16 * (i & 1)));
            }
        }
        if (staged && q % 8 == 7) {
            // the half is staged: lanes 8j..8j+7 store row 4i + j, 16 bytes each
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = 4 * i + (lane >> 3);
                const int ch = lane & 7;
                const uint4 x = *reinterpret_cast<const uint4*>(stage + r * kGradPitch + ch * 8);
                if (row0 + r < a.T)
                    *reinterpret_cast<uint4*>(a.G + static_cast<int64_t>(row0 + r) * a.ldG + c0 +
                                              half * 64 + ch * 8) = x;
            }
            __syncwarp();  // the staging rows are free for the next half
        }
    }
}

// Saving forward: the tile's fp32 logits (its ncols real columns) into
// logits_out row t, read from TMEM a quarter at a time (taddr: the tile's
// first column) apart from the reduction's own copy, which keeps fewer
// values live (4 bytes of spills instead of 52; the training step 0.7 %
// faster).  Called by the whole warp (lane = row0 + lane's row): each full
// 32-column quarter goes through the warp's staging rows and out in
// 128-byte row segments; a ragged last quarter is stored element by
// element.  Rows at or beyond T store nothing.
__device__ __forceinline__ void save_tile(uint32_t taddr, const TilePartialsArgs& a,
                                          int t, int c0, int ncols, float* stage, int lane,
                                          int row0) {
#pragma unroll
    for (int q = 0; q < kVocabTile / 32; ++q) {
        float v[32];  // this quarter, read from TMEM again (fewer live registers)
        ptx::tmem_load_32cols(taddr + q * 32, v);
        if (q * 32 + 32 <= ncols) {  // the same for the whole warp
#pragma unroll
            for (int k = 0; k < 8; ++k)
                *reinterpret_cast<float4*>(stage + lane * kSavePitch + 4 * k) =
                    make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
            __syncwarp();
            // lanes 8j..8j+7 store row 4i + j, 16 bytes each
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = 4 * i + (lane >> 3);
                const int ch = lane & 7;
                const float4 x = *reinterpret_cast<const float4*>(stage + r * kSavePitch + ch * 4);
                if (row0 + r < a.T)
                    *reinterpret_cast<float4*>(a.logits_out + static_cast<int64_t>(row0 + r) * a.ld_logits +
                                               c0 + q * 32 + ch * 4) = x;
            }
            __syncwarp();  // the staging rows are free for the next quarter
        } else if (t < a.T) {
            float* dst = a.logits_out + static_cast<int64_t>(t) * a.ld_logits + c0 + q * 32;
#pragma unroll
            for (int c = 0; c < 32; ++c)
                if (q * 32 + c < ncols) dst[c] = v[c];
        }
    }
}

// Work-unit order.  Units are (W tile n, token tile mu).  The order is
// vocabulary-major inside bands of kBandTokenTiles token tiles: every W tile
// is visited by all of a band's token tiles before the next W tile, so W is
// read from HBM once per band while the band's hidden rows (4096 rows = 32
// MB at H = 4096) stay in L2.  One band covers T <= 4096; at T = 8192 a
// single band let the drifting CTAs keep W tiles and 64 MB of hidden rows
// alive together, and L2 sent 7.9 GB per launch to HBM instead of the 2.6 GB
// two bands read.
constexpr int kBandTokenTiles = 32;

struct UnitCoords {
    int n_blk;  // W tile
    int mu;     // token tile
};

// unit -> (W tile, token tile) for num_n W tiles, num_mu token tiles and
// band_mu token tiles per band (the last band may hold fewer).
__device__ __forceinline__ UnitCoords unit_coords(int unit, int num_n, int num_mu, int band_mu) {
    const int full = band_mu * num_n;  // units of a full band
    const int band = unit / full;
    const int first_mu = band * band_mu;
    const int mus = min(band_mu, num_mu - first_mu);  // token tiles of this band
    const int within = unit - band * full;
    UnitCoords c;
    c.n_blk = within / mus;
    c.mu = first_mu + (within - c.n_blk * mus);
    return c;
}

// Shared-memory rings of the logits kernel:
//   kRingFull   full 128-row hidden boxes, one ring of 4 (hidden, W) stages;
//   kRingSmall  hidden boxes of roundup(T, 8) < 128 rows (decode batches), one
//               ring of ring_stages() stages;
//   kRingSplit  full hidden boxes in a ring of 4 and W boxes in a ring of 5,
//               filled independently as their slots free up (W first), for
//               batches of two token tiles (128 < T <= 256): each W tile is then
//               shared by two CTAs and streamed from HBM while their MMAs run at
//               the same pace, and the extra W stage of lookahead pays
//               (232 -> 224 us at T = 256); at the tensor-bound sizes it cost
//               8 %, so no other size uses it.  Not with the G or logits
//               staging rows, which leave no room for the fifth W stage.
enum RingKind { kRingFull = 0, kRingSmall = 1, kRingSplit = 2 };
constexpr int kSplitStagesB = kStages + 1;
constexpr int kSplitSmemBytes = kStages * static_cast<int>(kStageBytesA) +
                                kSplitStagesB * static_cast<int>(kStageBytesB) + 1024 + 256;
static_assert(kSplitSmemBytes <= kSmemLimit, "split rings exceed shared memory");

template <int kEpi, int kRing>
__global__ void __launch_bounds__(kThreads, 1)
    k_tile_partials(const __grid_constant__ CUtensorMap map_hidden,
                    const __grid_constant__ CUtensorMap map_w, const TilePartialsArgs a) {
    constexpr bool kSplit = kRing == kRingSplit;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    // hidden slots are a_box_rows rows each; the MMA still reads 128 rows from a
    // slot, and the rows past the box (the next slots' or the W boxes' bytes,
    // inside this allocation) only feed accumulator rows that are never read
    const int S = kRing == kRingSmall ? ring_stages(a.a_box_rows, staged_epi(kEpi)) : kStages;
    const int SB = kSplit ? kSplitStagesB : S;  // W slots
    const uint32_t a_stage = kRing == kRingSmall
                                 ? static_cast<uint32_t>(a.a_box_rows) * kBlockK * 2
                                 : kStageBytesA;
    uint8_t* sA = smem;
    uint8_t* sB = smem + S * a_stage;
    // full/empty: the (hidden, W) stages, or the hidden ring alone when split;
    // fullB/emptyB: the W ring when split
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + SB * kStageBytesB);
    uint64_t* empty = full + kMaxStages;
    uint64_t* fullB = empty + kMaxStages;
    uint64_t* emptyB = fullB + kMaxStages;
    uint64_t* acc_full = emptyB + kMaxStages;
    uint64_t* acc_empty = acc_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // backward and saving forward only: per-epilogue-warp staging rows for
    // the G or logits stores
    uint16_t* grad_stage = reinterpret_cast<uint16_t*>(sB + SB * kStageBytesB + 256);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_m = (a.T + kTileM - 1) / kTileM;
    const int num_n = (a.V_local + kTileN - 1) / kTileN;
    // a work unit is one W tile and one token tile
    const int total = num_m * num_n;
    const int unit0 = static_cast<int>(blockIdx.x);
    const int ustride = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        if (kSplit)
            for (int s = 0; s < SB; ++s) {
                ptx::mbar_init(&fullB[s], 1);
                ptx::mbar_init(&emptyB[s], 1);
            }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&acc_full[b], 1);
            ptx::mbar_init(&acc_empty[b], 4 * 32);
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tensormap(&map_hidden);
        ptx::prefetch_tensormap(&map_w);
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // With programmatic dependent launch the set-up above overlaps the
    // previous kernel; nothing it wrote or reads is touched before this point.
    ptx::grid_dependency_wait();

    if (warp == 0) {
        if (lane == 0 && kSplit) {
            // ---------------- TMA producer, split rings: each ring is refilled as
            // soon as one of its slots is free (W first), so the W stream runs up
            // to five stages ahead of the MMAs and the hidden rows up to four.
            uint32_t sa = 0, pa = 0, sb = 0, pb = 0;
            if (a.test_drop_stage && blockIdx.x == 0) {
                // test only: leave hidden slot 0 unfilled; the MMA's bounded wait gives up
                sa = 1;
            }
            int ua = unit0, ka = 0, ub = unit0, kbb = 0;  // next k-block of each ring
            UnitCoords ca = unit_coords(ua, num_n, num_m, kBandTokenTiles);
            UnitCoords cb = ca;
            bool idle = false;
            uint64_t t_idle = 0;
            while ((ua < total || ub < total) && !*abort_flag) {
                bool did = false;
                if (ub < total && ptx::mbar_try_wait(ptx::smem_addr(&emptyB[sb]), pb ^ 1u)) {
                    ptx::mbar_arrive_expect_tx(&fullB[sb], kStageBytesB);
                    ptx::tma_load_2d(sB + sb * kStageBytesB, &map_w, &fullB[sb], kbb * kBlockK,
                                     cb.n_blk * kTileN);
                    if (++sb == static_cast<uint32_t>(SB)) {
                        sb = 0;
                        pb ^= 1u;
                    }
                    if (++kbb == a.k_blocks) {
                        kbb = 0;
                        ub += ustride;
                        if (ub < total) cb = unit_coords(ub, num_n, num_m, kBandTokenTiles);
                    }
                    did = true;
                }
                if (ua < total && ptx::mbar_try_wait(ptx::smem_addr(&empty[sa]), pa ^ 1u)) {
                    ptx::mbar_arrive_expect_tx(&full[sa], kStageBytesA);
                    ptx::tma_load_2d(sA + sa * kStageBytesA, &map_hidden, &full[sa], ka * kBlockK,
                                     ca.mu * kTileM);
                    if (++sa == static_cast<uint32_t>(S)) {
                        sa = 0;
                        pa ^= 1u;
                    }
                    if (++ka == a.k_blocks) {
                        ka = 0;
                        ua += ustride;
                        if (ua < total) ca = unit_coords(ua, num_n, num_m, kBandTokenTiles);
                    }
                    did = true;
                }
                if (did) {
                    idle = false;
                } else if (!idle) {
                    idle = true;
                    t_idle = ptx::globaltimer();
                } else if (ptx::globaltimer() - t_idle > ptx::kWaitLimitNs) {
                    *abort_flag = 1;
                    report(a.status, RLK_ERR_TIMEOUT);
                    break;
                }
            }
        } else if (lane == 0) {
            // ---------------- TMA producer
            // A batch of at most 128 tokens loads only its first roundup(T, 8)
            // hidden rows; the accumulator rows beyond them are never read.
            const uint32_t a_bytes = static_cast<uint32_t>(a.a_box_rows) * kBlockK * 2;
            uint32_t stage = 0, phase = 0;
            if (a.test_drop_stage && blockIdx.x == 0) {
                // test only: leave stage 0 unfilled; the MMA's bounded wait gives up
                stage = 1;
            }
            for (int unit = unit0; unit < total && !*abort_flag; unit += ustride) {
                const UnitCoords uc = unit_coords(unit, num_n, num_m, kBandTokenTiles);
                const int n_blk = uc.n_blk;
                const int m_blk = uc.mu;
                for (int kb = 0; kb < a.k_blocks; ++kb) {
                    if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
                        *abort_flag = 1;
                        report(a.status, RLK_ERR_TIMEOUT);
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(&full[stage], a_bytes + kStageBytesB);
                    ptx::tma_load_2d(sA + stage * a_stage, &map_hidden, &full[stage],
                                     kb * kBlockK, m_blk * kTileM);
                    ptx::tma_load_2d(sB + stage * kStageBytesB, &map_w, &full[stage],
                                     kb * kBlockK, n_blk * kTileN);
                    if (++stage == static_cast<uint32_t>(S)) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer (split rings: stage/phase track the hidden
            // ring, sb/pb the W ring)
            uint32_t stage = 0, phase = 0, sb = 0, pb = 0, acc = 0, acc_phase = 0;
            for (int unit = unit0; unit < total && !*abort_flag; unit += ustride) {
                if (!ptx::mbar_wait(&acc_empty[acc], acc_phase ^ 1u, abort_flag)) {
                    *abort_flag = 1;
                    report(a.status, RLK_ERR_TIMEOUT);
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * kTileN;
                bool ok = true;
                for (int kb = 0; kb < a.k_blocks; ++kb) {
                    if ((kSplit && !ptx::mbar_wait(&fullB[sb], pb, abort_flag)) ||
                        !ptx::mbar_wait(&full[stage], phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint32_t a0 = ptx::smem_addr(sA + stage * a_stage);
                    const uint32_t b0 = ptx::smem_addr(sB + (kSplit ? sb : stage) * kStageBytesB);
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk) {
                        // advance 16 bf16 = 32 bytes along K inside the swizzle row
                        ptx::mma_bf16(d_tmem, ptx::smem_desc_k_sw128(a0 + kk * 32),
                                      ptx::smem_desc_k_sw128(b0 + kk * 32), kIdesc,
                                      (kb | kk) != 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(&empty[stage]);
                    if (++stage == static_cast<uint32_t>(S)) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (kSplit) {
                        ptx::mma_commit(&emptyB[sb]);
                        if (++sb == static_cast<uint32_t>(SB)) {
                            sb = 0;
                            pb ^= 1u;
                        }
                    }
                }
                if (!ok) {
                    *abort_flag = 1;
                    report(a.status, RLK_ERR_TIMEOUT);
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
        // ---------------- epilogue (warps 2..5; TMEM lane quadrant = warp % 4)
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        uint32_t acc = 0, acc_phase = 0;
        for (int unit = unit0; unit < total; unit += ustride) {
            const UnitCoords uc = unit_coords(unit, num_n, num_m, kBandTokenTiles);
            const int n_blk = uc.n_blk;
            const int m_blk = uc.mu;
            // last unit of this CTA: let the next kernel (the tile tree) start
            // launching; it waits for this grid before reading anything
            if (unit + ustride >= total) ptx::grid_dependents_launch();
            if (!ptx::mbar_wait(&acc_full[acc], acc_phase, abort_flag)) {
                *abort_flag = 1;
                report(a.status, RLK_ERR_TIMEOUT);
                break;
            }
            ptx::tc_fence_after_sync();
            const int t = m_blk * kTileM + row;
            bool valid = t < a.T;
            if (valid && a.active) valid = a.active[t] != 0;
            const int64_t tg_local =
                (kEpi != kEpiDebugLogits && valid) ? static_cast<int64_t>(a.targets[t]) - a.v_offset
                                                   : -1;
            if (kEpi == kEpiGrad && valid && n_blk == 0 && (tg_local < 0 || tg_local >= a.V_total))
                report(a.status, RLK_ERR_TARGET_RANGE);
            if (__any_sync(0xffffffffu, kEpi == kEpiPartials ? valid : (t < a.T))) {
                // kEpiSave: every row below T stores its logits, active or not
#pragma unroll 1
                for (int sub = 0; sub < kTileN / kVocabTile; ++sub) {
                    const int j = n_blk * (kTileN / kVocabTile) + sub;
                    const int c0 = j * kVocabTile;
                    if (c0 >= a.V_local) break;
                    const int ncols = min(kVocabTile, a.V_local - c0);
                    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                           acc * kTileN + sub * kVocabTile;
                    __syncwarp();  // tcgen05.ld is warp-collective: reconverge first
                    if (kEpi == kEpiSave)
                        save_tile(taddr, a, t, c0, ncols,
                                  reinterpret_cast<float*>(grad_stage) + quad * (32 * kSavePitch),
                                  lane, m_blk * kTileM + quad * 32);
                    float v[kVocabTile];
#pragma unroll
                    for (int q = 0; q < kVocabTile / 32; ++q) {
                        float part[32];
                        ptx::tmem_load_32cols(taddr + q * 32, part);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[q * 32 + i] = part[i];
                    }
                    if (kEpi == kEpiDebugLogits) {
                        if (t < a.T) {
                            float* dst = a.dbg_logits + static_cast<int64_t>(t) * a.V_local + c0;
                            for (int c = 0; c < ncols; ++c) dst[c] = v[c];
                        }
                        continue;
                    }
                    if (kEpi == kEpiGrad) {
                        grad_tile(v, a, t, c0, ncols, valid, tg_local - c0,
                                  grad_stage + quad * (32 * kGradPitch), lane,
                                  m_blk * kTileM + quad * 32);
                        continue;
                    }
                    const int64_t tl = tg_local - c0;
                    const bool own = valid && tl >= 0 && tl < ncols;
                    if (__any_sync(0xffffffffu, own)) {
                        const int ti = own ? static_cast<int>(tl) : -1;
                        float tv = 0.0f;
#pragma unroll
                        for (int c = 0; c < kVocabTile; ++c) tv = (c == ti) ? v[c] : tv;
                        if (own) a.tgt_logit[t] = tv;
                    }
                    const MaxSum r = reduce_tile(v, ncols);
                    if (valid)
                        a.partials[static_cast<int64_t>(t) * a.n_tiles + j] = make_float2(r.m, r.s);
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
        // a wait gave up: let copies and MMAs already in flight land before
        // the shared memory and TMEM are released (bounded, ~1 ms)
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

template <int kEpi>
cudaError_t set_smem_attr() {
    cudaError_t e = cudaFuncSetAttribute(k_tile_partials<kEpi, kRingFull>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_bytes_of<kEpi>());
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_tile_partials<kEpi, kRingSmall>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if constexpr (!staged_epi(kEpi)) {
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_tile_partials<kEpi, kRingSplit>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kSplitSmemBytes);
    }
    return e;
}

template <int kEpi>
cudaError_t launch_epi(const CUtensorMap& map_hidden, const CUtensorMap& map_w,
                       const TilePartialsArgs& a, int num_sms, cudaStream_t stream) {
    const int num_m = (a.T + kTileM - 1) / kTileM;
    const int num_n = (a.V_local + kTileN - 1) / kTileN;
    const int64_t total = static_cast<int64_t>(num_m) * num_n;
    const int grid = static_cast<int>(total < num_sms ? total : num_sms);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    const int ring = a.a_box_rows < kTileM ? kRingSmall
                     : (num_m == 2 && !staged_epi(kEpi)) ? kRingSplit
                                                         : kRingFull;
    cfg.dynamicSmemBytes = ring == kRingSmall ? ring_smem_bytes<kEpi>(a.a_box_rows)
                           : ring == kRingSplit ? kSplitSmemBytes
                                                : smem_bytes_of<kEpi>();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (ring == kRingSmall)
        return cudaLaunchKernelEx(&cfg, k_tile_partials<kEpi, kRingSmall>, map_hidden, map_w, a);
    if constexpr (!staged_epi(kEpi)) {
        if (ring == kRingSplit)
            return cudaLaunchKernelEx(&cfg, k_tile_partials<kEpi, kRingSplit>, map_hidden, map_w, a);
    }
    return cudaLaunchKernelEx(&cfg, k_tile_partials<kEpi, kRingFull>, map_hidden, map_w, a);
}

}  // namespace

cudaError_t prepare_tile_partials_kernels() {
    cudaError_t e;
    if ((e = set_smem_attr<kEpiPartials>()) != cudaSuccess) return e;
    if ((e = set_smem_attr<kEpiDebugLogits>()) != cudaSuccess) return e;
    if ((e = set_smem_attr<kEpiSave>()) != cudaSuccess) return e;
    return set_smem_attr<kEpiGrad>();
}

cudaError_t launch_tile_partials(const CUtensorMap& map_hidden, const CUtensorMap& map_w,
                                 const TilePartialsArgs& a, int epilogue, int num_sms,
                                 cudaStream_t stream) {
    if (epilogue == kEpiDebugLogits)
        return launch_epi<kEpiDebugLogits>(map_hidden, map_w, a, num_sms, stream);
    if (epilogue == kEpiGrad) return launch_epi<kEpiGrad>(map_hidden, map_w, a, num_sms, stream);
    if (epilogue == kEpiSave) return launch_epi<kEpiSave>(map_hidden, map_w, a, num_sms, stream);
    return launch_epi<kEpiPartials>(map_hidden, map_w, a, num_sms, stream);
}

}  // namespace rlk
