/*
 * rlk.h -- C-ABI of the layout-invariant selected-token logprob ("strict-path
 * linear logprob") for NVIDIA GB300 (sm_103a).
 *
 * What it computes.  For each token t of a batch, with bf16 hidden state
 * h[t, :] and bf16 output-head weights W[v, :] over the whole vocabulary,
 *
 *     lse[t]     = log sum_v exp(h[t] . W[v])
 *     logprob[t] = h[t] . W[target[t]] - lse[t]
 *
 * ("vLLM RL-Kernel v0.1.0: ROCm 上でのビット単位のトレーニング-ロールアウト一貫性",
 * strict-path boundary table, row "Linear logprob": actual vocabulary range,
 * target ownership, local reduction, cross-rank LSE merge; the blog on
 * bitwise consistency with RL-Kernel + vime on AMD, section 3.1: log_softmax
 * read at the target, whose max and sum reductions fix the last bits).
 *
 * The numeric contract "rlk-linlogp-v1" fixes every reduction, merge order,
 * precision, rounding point and primitive (the same page, section
 * 数値実行契約), so a token's two results are bit-identical whatever batch it
 * sits in (1-row decode or a packed batch), whatever its row position, and
 * however the vocabulary is split into tree-aligned shards:
 *
 *   - logits are fp32 tensor-core dot products of bf16 inputs, K ascending in
 *     steps of 16, one accumulator, never split over K, never rounded to bf16;
 *   - the vocabulary is cut into tiles of 128 columns; each tile gives
 *     (m, s) = (max logit, pairwise-tree sum of exp(logit - m)) for its real
 *     columns (a last, shorter tile simply has fewer columns);
 *   - tiles merge along one fixed tree (recursive bisection of the tile
 *     index range, lower half taking the extra tile) with
 *     merge(L, R) = (hi.m, fma(lo.s, exp(lo.m - hi.m), hi.s)), hi = the
 *     operand with the larger m, L on a tie;
 *   - n_shards (1, 2, 4 or 8) shards are the nodes of that tree at depth
 *     log2(n_shards), so shard records merged in shard order give the same
 *     bits as the unsharded call;
 *   - lse = RN(m + log(s)), logprob = RN(target logit - lse);
 *   - exp and log are the library's own (Cody-Waite + degree-7 Taylor; atanh
 *     series), not the CUDA math library's.
 *
 * Conventions for every call below.
 *   - Pointers named as device pointers must point to device memory of the
 *     current CUDA device; the caller owns every buffer.  The library keeps
 *     no per-call state and allocates no device memory.
 *   - Calls are asynchronous and stream-ordered on `stream` (NULL = legacy
 *     default stream); outputs are valid once the stream reaches them.
 *   - Host-detectable errors are returned before anything is launched.
 *   - Device-detected errors are OR-ed into *dev_status (a device int32 the
 *     caller zeroes; may be NULL) as bit (1 << code): RLK_ERR_TARGET_RANGE
 *     for an active row whose target no shard owns (that row's outputs are
 *     NaN), RLK_ERR_TIMEOUT if a pipeline wait ran out (outputs undefined;
 *     the kernel returns instead of hanging).
 *   - T == 0 is a no-op returning RLK_OK; T < 0 or T > RLK_MAX_ROWS returns
 *     RLK_ERR_INVALID_ARG (kernels index rows in 32 bits and step past
 *     the last row by less than 2^20).
 *   - Inactive rows (active_mask[t] == 0) give out_logprob = out_lse = 0 and
 *     all-zero partial records; their hidden row and target are never used
 *     in any other row's result.  active_mask == NULL means all active.
 *   - Only sm_103 devices are supported; anything else returns
 *     RLK_ERR_UNSUPPORTED.  There is no fallback path.
 */
#ifndef RLK_H_
#define RLK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle type as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st* rlk_stream_t;

typedef enum rlk_status {
    RLK_OK = 0,
    RLK_ERR_INVALID_ARG = 1,   /* null pointer, negative size, T > RLK_MAX_ROWS, bad shard index */
    RLK_ERR_UNSUPPORTED = 2,   /* device not sm_103; H % 64 != 0 or H > 2^20; V > 262144; n_shards not in {1,2,4,8} or > tiles */
    RLK_ERR_ALIGNMENT = 3,     /* hidden/W not 16-byte aligned, workspace not 256-byte aligned */
    RLK_ERR_WORKSPACE = 4,     /* workspace smaller than rlk_workspace_size() */
    RLK_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed (launch, device query) */
    RLK_ERR_TARGET_RANGE = 6,  /* device-detected: active row whose target no shard owns */
    RLK_ERR_TIMEOUT = 7        /* device-detected: a bounded pipeline wait gave up */
} rlk_status_t;

/* Per-token record of one vocabulary shard (16 bytes). */
typedef struct rlk_partial {
    float m;          /* max logit over the shard's vocabulary range */
    float s;          /* sum of exp(logit - m) over the range, merged along the tile tree */
    float tgt;        /* the target's logit if this shard owns the target, else 0 */
    uint32_t owned;   /* 1 if target lies in [v_begin, v_end) of this shard, else 0 */
} rlk_partial_t;

#define RLK_VOCAB_TILE 128
#define RLK_MAX_SHARDS 8
#define RLK_MAX_VOCAB 262144          /* 2048 tiles */
#define RLK_K_BLOCK 64                /* H must be a multiple of this */
#define RLK_MAX_ROWS 2146435072       /* 2^31 - 2^20: the largest T (rows) any call takes */
#define RLK_DTYPE_F32 0               /* logits element types for the materialised-logits calls */
#define RLK_DTYPE_BF16 1

/* "rlk-linlogp-v1": names the numeric contract above. */
const char* rlk_contract_id(void);

/* Build fingerprint: source revision, nvcc version, arch and contract flags. */
const char* rlk_build_fingerprint(void);

/* Human-readable name of a status code. */
const char* rlk_status_string(int status);

/*
 * Vocabulary range [*v_begin, *v_end) of shard `shard` of `n_shards`: the
 * shard-th node at depth log2(n_shards) of the tile tree, in vocabulary ids
 * (the strict-path table's "actual vocabulary range").  Host only.
 * Errors: RLK_ERR_INVALID_ARG (null outputs, V < 1, shard out of range),
 * RLK_ERR_UNSUPPORTED (bad n_shards, V > RLK_MAX_VOCAB).
 */
rlk_status_t rlk_shard_range(int64_t V, int n_shards, int shard, int64_t* v_begin, int64_t* v_end);

/*
 * Bytes of device workspace rlk_linear_logprob needs for (T, V, n_shards);
 * it also covers rlk_linear_logprob_shard for any shard of that split.
 * Layout (each part 256-byte aligned): per-tile (m, s) float pairs [T][tiles],
 * target logits float [T], shard records rlk_partial_t [n_shards][T].
 * Returns 0 for invalid arguments.
 */
size_t rlk_workspace_size(int64_t T, int64_t V, int n_shards);

/*
 * Full selected-token logprob of T tokens over V vocabulary entries,
 * vocabulary split into n_shards tree-aligned shards merged in shard order
 * on this device (the boundary table's local reduction + cross-rank LSE
 * merge, with the ranks emulated as shards).  The per-shard records are
 * left in the workspace's record area.
 *
 *   hidden       device, bf16 [T][H] row-major, 16-byte aligned
 *   W            device, bf16 [V][H] row-major (vocabulary rows), 16-byte aligned
 *   targets      device, int32 [T], global vocabulary ids
 *   active_mask  device, uint8 [T] (nonzero = active) or NULL
 *   H            multiple of 64, at most 2^20
 *   V            1 .. RLK_MAX_VOCAB
 *   n_shards     1, 2, 4 or 8, and at most ceil(V / 128)
 *   out_logprob  device, float [T];  out_lse  device, float [T]
 *   workspace    device, 256-byte aligned, >= rlk_workspace_size(T, V, n_shards) bytes
 *   dev_status   device int32 or NULL (see conventions)
 */
rlk_status_t rlk_linear_logprob(const void* hidden, const void* W, const int32_t* targets,
                                const uint8_t* active_mask, int64_t T, int64_t H, int64_t V,
                                int n_shards, float* out_logprob, float* out_lse,
                                void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                rlk_stream_t stream);

/*
 * The part one vocabulary shard (one emulated TP rank) computes: its record
 * (m, s, tgt, owned) per token from its own weight rows only.
 *
 *   W_shard      device, bf16 rows [v_begin, v_end) of the full W (see
 *                rlk_shard_range), [v_end - v_begin][H] row-major, 16-byte aligned
 *   targets      global vocabulary ids; ownership is target in [v_begin, v_end)
 *   V_total      the full vocabulary size (defines the tile tree)
 *   out_partial  device, rlk_partial_t [T]
 *   workspace    >= rlk_workspace_size(T, v_end - v_begin, 1) bytes
 * Other arguments as rlk_linear_logprob.
 */
rlk_status_t rlk_linear_logprob_shard(const void* hidden, const void* W_shard,
                                      const int32_t* targets, const uint8_t* active_mask,
                                      int64_t T, int64_t H, int64_t V_total, int n_shards,
                                      int shard, rlk_partial_t* out_partial, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status,
                                      rlk_stream_t stream);

/*
 * Cross-shard LSE merge in fixed shard order (the boundary table's
 * "cross-rank LSE merge" and the distributed-aggregation row's fixed rank
 * reduction order): records merge pairwise (0,1),(2,3),... then pairs of
 * those; the target logit comes from the one owning shard.
 *
 *   partials     HOST array of n_shards DEVICE pointers, each rlk_partial_t [T], shard order
 *   n_shards     1, 2, 4 or 8
 *   out_logprob, out_lse  device, float [T]
 * An active row with no owning shard, or with more than one, gets NaN and
 * sets RLK_ERR_TARGET_RANGE in *dev_status.
 * The records may come from other processes: with the vocabulary split over
 * n ranks (rank r holding shard r's W rows and calling
 * rlk_linear_logprob_shard), gathering every rank's records in rank order and
 * merging them here on each rank gives every rank the unsharded call's bits.
 */
rlk_status_t rlk_lse_merge(const rlk_partial_t* const* partials, int n_shards, int64_t T,
                           const uint8_t* active_mask, float* out_logprob, float* out_lse,
                           int32_t* dev_status, rlk_stream_t stream);

/*
 * The two stages of rlk_linear_logprob as separate calls (same kernels,
 * same bits), so a caller can time or overlap them:
 *   rlk_tile_partials: logits GEMM + fused per-tile (m, s) and target pick,
 *                      into the workspace;
 *   rlk_tile_merge:    tile tree, shard records, final lse/logprob.
 * Arguments mean what they mean for rlk_linear_logprob; the workspace must
 * be the same buffer for both calls.
 */
rlk_status_t rlk_tile_partials(const void* hidden, const void* W, const int32_t* targets,
                               const uint8_t* active_mask, int64_t T, int64_t H, int64_t V,
                               int n_shards, void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, rlk_stream_t stream);
rlk_status_t rlk_tile_merge(const int32_t* targets, const uint8_t* active_mask, int64_t T,
                            int64_t V, int n_shards, float* out_logprob, float* out_lse,
                            void* workspace, size_t workspace_bytes, int32_t* dev_status,
                            rlk_stream_t stream);

/*
 * Diagnostic: the fp32 logits [T][V] exactly as the fused path sees them
 * (same kernel mainloop, the epilogue stores the accumulator instead of
 * reducing it).  out_logits: device, float [T][V] row-major.  Meant for
 * tests and for locating a divergence (the blog's advice to dump the
 * intermediate values, section 5.2).
 */
rlk_status_t rlk_debug_logits(const void* hidden, const void* W, int64_t T, int64_t H, int64_t V,
                              float* out_logits, int32_t* dev_status, rlk_stream_t stream);

/*
 * Diagnostic: evaluates one of the contract's primitives on the GPU over the
 * fp32 bit patterns [first, first + count) and writes
 *   sum_i (bits(f(x_i)) + 0x9E3779B9) * (2 i + 1)   (mod 2^64)
 * to *out_hash, so a caller can compare the device's primitive with another
 * implementation of the contract over a whole input range (any single
 * differing output changes the sum).  The primitives are the contract's
 * fixed exp, log and rsqrt ("vLLM RL-Kernel v0.1.0: ROCm 上でのビット単位の
 * トレーニング-ロールアウト一貫性", section 数値実行契約, item 6: the math
 * primitives are part of the contract); the check itself has no counterpart
 * in the pages.
 *   which     0: rlk_exp; 1: rlk_exp evaluated two values per instruction (the
 *             kernels' packed form; must equal 0); 2: rlk_log; 3: rlk_rsqrt
 *   first, count  first bit pattern and how many; first + count <= 2^32
 *   out_hash  device, one uint64_t, overwritten
 * Errors: RLK_ERR_INVALID_ARG for an unknown primitive, a range beyond 2^32
 * or a null out_hash; otherwise as the other calls.
 */
rlk_status_t rlk_debug_primitive_hash(int which, uint32_t first, uint64_t count,
                                      uint64_t* out_hash, rlk_stream_t stream);

/*
 * Selected-token logprob from logits that already exist in memory, under
 * the same contract (the blog's rl_kernel.log_softmax with a fixed reduction
 * tree, sections 4.2-4.3, read at the target).  Given the fp32 logits the
 * fused path computes (rlk_debug_logits), it returns the fused path's bits.
 *
 *   logits       device, [T][ld] row-major, elements RLK_DTYPE_F32 or RLK_DTYPE_BF16
 *                (bf16 widens exactly to fp32); only columns [0, V) are read
 *   ld           row stride in elements, >= V; logits aligned to their element
 *                size (when every row starts on a 16-byte boundary -- a 16-byte
 *                aligned base and ld * element size a multiple of 16 -- rows
 *                are copied in 16-byte pieces; the values and results are the
 *                same either way)
 *   workspace    >= rlk_workspace_size(T, V, n_shards) bytes, same layout as rlk_linear_logprob
 * Other arguments, outputs and errors as rlk_linear_logprob.
 */
rlk_status_t rlk_logits_logprob(const void* logits, int logits_dtype, int64_t ld,
                                const int32_t* targets, const uint8_t* active_mask, int64_t T,
                                int64_t V, int n_shards, float* out_logprob, float* out_lse,
                                void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                rlk_stream_t stream);

/*
 * Full log_softmax of materialised logits: out[t][v] = RN(l[t][v] - lse[t])
 * with lse from the contract's tile tree; out_lse[t] = lse[t].  Inactive rows
 * give zeros.  The same tree gives the same lse bits as rlk_linear_logprob.
 *
 *   out          device, float [T][V] row-major (dense, V columns)
 *   out_lse      device, float [T]
 *   workspace    >= rlk_workspace_size(T, V, 1) bytes
 * logits, logits_dtype, ld as rlk_logits_logprob.
 */
rlk_status_t rlk_log_softmax(const void* logits, int logits_dtype, int64_t ld,
                             const uint8_t* active_mask, int64_t T, int64_t V, float* out,
                             float* out_lse, void* workspace, size_t workspace_bytes,
                             int32_t* dev_status, rlk_stream_t stream);

/*
 * Backward of sum_t grad_logprob[t] * logprob[t] (the blog's requirement,
 * sections 3.3 and 4.2, that the kernel provide a backward with the same
 * numeric discipline as its forward):
 *
 *   G[t, v]        = bf16_RN(RN(g_t * d)), d = RN(1 - p) at the target, -p elsewhere,
 *                    p = rlk_exp(RN(logit[t, v] - lse[t])), from the same fp32 logits
 *   grad_hidden    = G · W   (fp32; the sum over v in 8 fixed ranges of ascending
 *                    vocabulary, each one accumulator, added pairwise in fixed order;
 *                    a token's row does not depend on the rest of the batch)
 *   grad_W         = Gᵀ · h  (fp32; the sum over t ascending in one accumulator)
 *
 *   lse           device, float [T]: the forward's out_lse for this batch
 *   grad_logprob  device, float [T]: dL/dlogprob
 *   grad_hidden   device, float [T][H], or NULL to skip
 *   grad_W        device, float [V][H], or NULL to skip (at least one is required)
 *   workspace     >= rlk_backward_workspace_size(T, H, V) bytes, 256-byte aligned
 *                 (holds G as bf16 [T][roundup(V, 8)] at offset 0)
 * Inactive rows contribute nothing (their G row is zero).  An active row
 * whose target lies outside [0, V) sets RLK_ERR_TARGET_RANGE and gets no
 * one-hot term.  Other arguments as rlk_linear_logprob.
 * When both gradients are asked for, grad_hidden's fixed-order split sum
 * runs beside the grad_W GEMM on a library stream, forked from `stream`
 * after grad_hidden's GEMM and joined back before the call's work on
 * `stream` ends (events; capturable in a CUDA graph).  The first such call
 * on a device creates that stream and its two events; they live for the
 * process.
 */
size_t rlk_backward_workspace_size(int64_t T, int64_t H, int64_t V);
rlk_status_t rlk_linear_logprob_backward(const void* hidden, const void* W,
                                         const int32_t* targets, const uint8_t* active_mask,
                                         const float* grad_logprob, const float* lse, int64_t T,
                                         int64_t H, int64_t V, float* grad_hidden, float* grad_W,
                                         void* workspace, size_t workspace_bytes,
                                         int32_t* dev_status, rlk_stream_t stream);

/*
 * Training pair that trades memory for the backward's second logits GEMM:
 * rlk_linear_logprob_save_logits is rlk_linear_logprob (same outputs, same
 * bits) that also stores every row's fp32 logits (the exact accumulator
 * values the epilogue reduces), and rlk_linear_logprob_backward_from_logits
 * forms G from those stored logits instead of recomputing them, then runs
 * the same two GEMMs: its grad_hidden and grad_W have the bits of
 * rlk_linear_logprob_backward on the same batch.  Same backward definition
 * as above (the blog's sections 3.3 and 4.2).
 *
 *   logits       device, float [T][ld_logits] row-major; written by the
 *                forward (columns [0, V) of every row below T, active or
 *                not), read by the backward; 16-byte aligned, ld_logits a
 *                multiple of 4 and >= V (else RLK_ERR_ALIGNMENT /
 *                RLK_ERR_INVALID_ARG); T * ld_logits * 4 bytes, owned by the
 *                caller (2.49 GB at T = 4096, V = 151936)
 * Forward: other arguments, outputs and errors as rlk_linear_logprob.
 * Backward: other arguments, outputs and errors as rlk_linear_logprob_backward
 * (hidden and W are still read: the GEMMs need them).
 */
rlk_status_t rlk_linear_logprob_save_logits(const void* hidden, const void* W,
                                           const int32_t* targets, const uint8_t* active_mask,
                                           int64_t T, int64_t H, int64_t V, int n_shards,
                                           float* out_logprob, float* out_lse, float* logits,
                                           int64_t ld_logits, void* workspace,
                                           size_t workspace_bytes, int32_t* dev_status,
                                           rlk_stream_t stream);
rlk_status_t rlk_linear_logprob_backward_from_logits(
    const float* logits, int64_t ld_logits, const void* hidden, const void* W,
    const int32_t* targets, const uint8_t* active_mask, const float* grad_logprob,
    const float* lse, int64_t T, int64_t H, int64_t V, float* grad_hidden, float* grad_W,
    void* workspace, size_t workspace_bytes, int32_t* dev_status, rlk_stream_t stream);

/*
 * Strict RMSNorm producing the hidden states the head consumes (the
 * strict-path table's "RMSNorm" row: reduction domain, epsilon, residual
 * add, output boundary).  Per row:
 *   x'   = bf16_RN(RN(x + residual))          (x itself when residual is NULL)
 *   s    = pairwise tree over nextpow2(H) feature slots of x'_i^2 (fp32)
 *   rstd = rlk_rsqrt(RN(RN(s / H) + eps))      (the library's own rsqrt)
 *   out  = bf16_RN(RN(RN(x'_i * rstd) * gamma_i))
 * A row's result does not depend on the batch around it.
 *
 *   x, residual  device, bf16 [T][H] (residual may be NULL), 16-byte aligned
 *   gamma        device, bf16 [H]
 *   eps          > 0
 *   out          device, bf16 [T][H]
 *   residual_out device, bf16 [T][H] receiving x' (the next residual stream), or NULL;
 *                requires residual
 * out may be x and residual_out may be residual (updated in place): every
 * element is read before it is written.  No other overlap is allowed.
 *   H            multiple of 64, at most 8192
 */
rlk_status_t rlk_rmsnorm(const void* x, const void* residual, const void* gamma, float eps,
                         int64_t T, int64_t H, void* out, void* residual_out, rlk_stream_t stream);

/*
 * Same result as rlk_linear_logprob (same kernels, same bits), for callers
 * that cannot allocate device memory when they call: e.g. a rollout engine
 * that reserved almost all GPU memory for its KV cache at start-up, or a
 * decode loop that cannot afford the device-wide synchronisation cudaFree
 * performs.  Instead of a caller workspace it uses a scratch array of
 * RLK_STATIC_WS_BYTES compiled into the library (one copy per GPU that
 * loads the library, held until the process exits).  The pages have no
 * counterpart to this call; it is a deployment convenience.
 *
 *   - Allocates nothing and calls no allocating routine.
 *   - Batches whose workspace (rlk_workspace_size(T, V, n_shards)) exceeds
 *     RLK_STATIC_WS_BYTES are refused with RLK_ERR_WORKSPACE; at V = 151936
 *     that is about 1700 tokens per call with 4 shards.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current).  Under CUDA's
 *     default lazy module loading that lookup also loads the array itself,
 *     so the first call on a device is the one that still needs 16 MiB of
 *     free device memory: make it at start-up, before reserving the rest of
 *     the memory (a KV cache), and before any stream capture.  Later calls
 *     need no free memory at all.
 *   - The looked-up address belongs to the device's primary context: do not
 *     reset the device (cudaDeviceReset) or call from another context
 *     between calls.
 *   - All calls on a device share the array: calls that overlap on the GPU
 *     (e.g. on two unordered streams) race; order them.  Nothing in the
 *     array needs to start at zero.
 * Other arguments and errors (and the order in which they are checked) as
 * rlk_linear_logprob; RLK_ERR_CUDA also if the address lookup fails.
 */
#define RLK_STATIC_WS_BYTES (16u << 20)
rlk_status_t rlk_linear_logprob_static_ws(const void* hidden, const void* W,
                                          const int32_t* targets, const uint8_t* active_mask,
                                          int64_t T, int64_t H, int64_t V, int n_shards,
                                          float* out_logprob, float* out_lse, int32_t* dev_status,
                                          rlk_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RLK_H_ */
