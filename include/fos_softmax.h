/*
 * fos_softmax.h -- C ABI of libfos_softmax.so: a fixed-order, batch-invariant row softmax
 * (forward, backward, per-head sink gradient) for NVIDIA GB300 (sm_103a).
 *
 * The operation sits between the QK and AV GEMMs of joint attention: it takes a
 * materialised score matrix, applies softmax along the key dimension and hands the
 * probabilities on ("[WS1][kernels] Add fixed-order joint-attention softmax for Qwen-Image",
 * Summary).  Its floating-point evaluation order is fixed, so a row gives the same bits
 * whatever its batch, its position in the batch or the launch geometry (same page, Summary:
 * "Fixed-order online softmax"; "Batch-invariant attention (standard softmax--cuda
 * version)", Acceptance Criteria).
 *
 * Layout.  Scores, P, dP and dScores are row-major [rows, ld] arrays of the I/O dtype, with
 * rows ordered [batch][heads][q_len] (row r has b = r / (heads*q_len), h = (r / q_len) %
 * heads, i = r % q_len) and ld >= key_len elements between row starts.  Columns key_len ..
 * ld-1 are never read or written.  LSE and delta are float32 [rows]; sink and d_sink are
 * float32 [heads].
 *
 * Short rows.  Rows of at most 8 tiles (2,048 keys) with 16-byte aligned rows are taken one
 * warp per row, forward and backward (warps_per_cta then counts those warps, stages their row
 * buffers per warp); the arithmetic is the same, so the bits are too.
 *
 * Long rows.  A row is normally staged whole in shared memory (up to about 57k fp32 / 113k
 * bf16 keys forward, half that backward).  Longer rows are read twice, in segments of
 * max(16, 2 x compute warps) tiles, by streaming kernels with the same per-tile arithmetic and
 * merge order, so a row gives the same bits either way; they need 16-byte aligned rows (base,
 * ld * size and key_len * size multiples of 16 bytes) and fit up to about 4.5 M (forward) /
 * 14 M (backward) bf16 keys.
 *
 * Masks.  Key j of row r is valid iff all of the given conditions hold:
 *   causal:        j <= key_len - q_len + i
 *                  ("Batch-invariant attention", Prefill / Decode / KV-cache Contract)
 *   kv_valid_len:  j <  kv_valid_len[b]   (values are clamped to [0, key_len])
 *   key_mask:      key_mask[b*key_len + j] != 0
 *   forward only:  scores[r, j] != -inf   (an input -inf acts as masked)
 * Masked keys take no part in any sum and their P / dScores are written as +0.
 * Scores equal to +inf or NaN are outside the contract (their rows come out NaN).
 *
 * Arithmetic contract (the same in every path of the library, so results are bit-identical
 * across batch size, row offset, CTAs, warps per CTA, pipeline depth and load path):
 *   - keys are cut into tiles of 256 (TILE_K), walked left to right; inside a tile lane l of
 *     a warp owns keys 8l..8l+7 and combines them in ascending order, and the 32 lane values
 *     are combined by a warp xor-shuffle tree with offsets 16, 8, 4, 2, 1;
 *   - exp(x) is evaluated as 2^(x * log2 e) with the hardware base-2 approximation
 *     (PTX ex2.approx.f32) after one float32 multiply by log2 e rounded to float32;
 *   - all intermediates are float32 with explicit round-to-nearest operations (no FMA
 *     contraction, no fast-math, no atomics, no split of a row across CTAs, no tensor cores);
 *   - the result is rounded to the I/O dtype once, at the final write.
 * fos_contract_fingerprint() spells out the full contract as a string.
 *
 * Ownership and streams.  The caller owns every buffer; all array pointers are DEVICE
 * pointers, except the data arrays of fos_softmax_step_host, which are HOST pointers.  The
 * library allocates no memory and never synchronises (fos_device_error excepted): each call
 * validates its arguments on the host, enqueues its work on `stream` on the current device
 * and returns.  The only state kept across calls is per device: kernel attributes, the
 * device error word, and the two streams and events of the host-buffer pipeline.  Output
 * buffers must not overlap inputs, except that probs may equal scores and dscores may equal
 * dprobs (in place).
 *
 * Errors.  Every entry point returns fos_status:
 *   FOS_ERR_INVALID      bad arguments (null required pointer, rows != batch*heads*q_len,
 *                        key_len < 1, ld < key_len, unknown dtype, causal with q_len >
 *                        key_len, bad launch options); nothing is launched.
 *   FOS_ERR_UNSUPPORTED  valid, but beyond what the kernels take (a row too long to stage
 *                        whose buffers do not allow bulk copies, a row whose tile statistics
 *                        exceed shared memory, or a forced load path the buffers do not
 *                        allow).
 *   FOS_ERR_CUDA         the launch failed (cudaGetLastError after the launch).
 *   FOS_ERR_TIMEOUT      reported by fos_device_error(): a bounded wait inside a kernel ran
 *                        out, the kernel stopped early and its outputs are not valid.
 *   FOS_ERR_INDEX        reported by fos_device_error() of the debug build only (the library
 *                        compiled with FOS_DEBUG, whose kernels check their stage offsets,
 *                        tensor-memory columns and row indices before using them): a check
 *                        failed and the access was skipped.
 * rows == 0 is valid and launches nothing (the array pointers may then be NULL).
 */
#ifndef FOS_SOFTMAX_H
#define FOS_SOFTMAX_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

/* I/O dtype of scores, P, dP and dScores. */
typedef enum fos_dtype {
  FOS_F32 = 0,  /* IEEE binary32 */
  FOS_BF16 = 1, /* bfloat16; rounded to nearest-even once, at the final write */
  FOS_F16 = 2   /* IEEE binary16; rounded to nearest-even once, at the final write */
} fos_dtype;

typedef enum fos_status {
  FOS_OK = 0,
  FOS_ERR_INVALID = 1,
  FOS_ERR_UNSUPPORTED = 2,
  FOS_ERR_CUDA = 3,
  FOS_ERR_TIMEOUT = 4,
  FOS_ERR_INDEX = 5 /* debug build only (compiled with FOS_DEBUG): an index check in a kernel
                       failed, the access was skipped and the outputs are not valid */
} fos_status;

/* Problem description shared by the three operations. */
typedef struct fos_desc {
  int64_t rows;                /* batch * heads * q_len */
  int64_t ld;                  /* elements between row starts, >= key_len */
  int32_t key_len;             /* L, keys per row, >= 1 */
  int32_t batch;               /* B */
  int32_t heads;               /* H */
  int32_t q_len;               /* Sq, query rows per (batch, head) */
  int32_t causal;              /* 0 or 1; key j of query i valid iff j <= L - Sq + i */
  int32_t reserved;            /* must be 0 */
  const int32_t *kv_valid_len; /* device [batch] or NULL: keys j >= kv_valid_len[b] masked */
  const uint8_t *key_mask;     /* device [batch * key_len] or NULL: 0 = masked */
  const float *sink;           /* device [heads] or NULL: per-head sink logit (off-by-one) */
} fos_desc;

/*
 * Optional launch options (pass NULL for the defaults).  None of them changes a result bit:
 * they exist so that tests can vary the launch geometry and exercise the bounded-wait path.
 */
typedef struct fos_launch {
  int32_t warps_per_cta; /* 0 = default (chosen from key_len); otherwise 1..16 */
  int32_t ctas;          /* 0 = default (persistent: SMs x resident CTAs); else >= 1 */
  int32_t stages;        /* 0 = default; rows in flight per CTA on the bulk-copy path, 1..16 */
  int32_t load_path;     /* 0 = auto, 1 = bulk copy (TMA) only, 2 = plain loads only,
                            3 = streaming: the row read twice in segments (the path taken
                            anyway by rows too long to stage; same bits) */
  int64_t wait_timeout_ns; /* 0 = default (2 s): limit of every bounded wait in a kernel */
  int32_t test_stall;    /* 0; 1 = CTA 0 waits on a copy that is never issued (test only) */
  int32_t generic;       /* 0 = auto; 1 = the general one-CTA-per-row kernels only: neither the
                            instances specialised for unmasked rows, nor the forward's row
                            groups, nor the one-warp-per-row kernels for rows of at most 8
                            tiles (same bits) */
  int32_t groups_per_cta; /* 0 = default; forward rows whose warps keep all their tiles'
                            exponentials (4, 6 or 8 tiles per warp, bulk copies): row groups of
                            warps_per_cta warps per CTA, 1..15, each with its own ring of
                            `stages` rows; FOS_ERR_UNSUPPORTED where that kernel does not apply
                            (same bits) */
  int32_t sink_fusion;    /* fos_softmax_bwd_sink only: 0 = the library's choice (the faster way
                            measured), 1 = the backward takes the sink terms by octets wherever
                            its kernel can, 2 = never (delta, then the sink-gradient kernel);
                            the same bits every way */
} fos_launch;

/*
 * Forward.  For each row: tile statistics (max, sum of exp) over keys 256t..256t+255,
 * online-softmax states merged left to right starting from (sink_h, 1) when a sink is given
 * and (-inf, 0) otherwise; LSE = M + log(S); P_j = exp(x_j - m_t) * (exp(m_t - M) / S) for
 * key j of tile t.  ("[WS1][kernels] Add fixed-order joint-attention softmax for
 * Qwen-Image", Summary; LSE: "Batch-invariant attention", Implementation; sink: "[ROCm] Jax
 * Add softmax sink (learnable off-by-one) support", Description.)
 *   scores  device [rows, ld] of dtype        (input)
 *   probs   device [rows, ld] of dtype        (output P; may equal scores)
 *   lse     device float [rows]               (output; -inf for a row with nothing valid)
 * Resources: besides shared memory, each CTA of the forward allocates tensor memory (tcgen05,
 * at most 256 of an SM's 512 columns) for its lifetime, and it frees it before exiting, on
 * error paths too.  A kernel of another stream that holds the SM's remaining columns makes the
 * forward's CTAs wait in their allocation until those are released.  No kernel of this library
 * waits on another kernel while it holds columns (fos_qk_scores and fos_pv_out free theirs
 * when their CTAs finish their own tiles), so such a wait between this library's kernels
 * always ends; a caller's kernel that holds columns until the softmax has run would never
 * see it run.
 */
fos_status fos_softmax_fwd(const fos_desc *desc, fos_dtype dtype, const void *scores,
                           void *probs, float *lse, cudaStream_t stream,
                           const fos_launch *launch);

/*
 * Backward (softmax VJP on the P given): delta = sum_j P_j dP_j with the forward's tile
 * layout (lane-local ascending fused multiply-adds, warp xor tree, tile partials added left
 * to right); dScores_j = P_j * (dP_j - delta), rounded once.  Only the mask inputs of desc
 * are used (the sink is not).  ("[WS1][kernels] Add fixed-order joint-attention softmax for
 * Qwen-Image", Summary, "Fixed-order backward".)
 *   probs    device [rows, ld] of dtype      (input P)
 *   dprobs   device [rows, ld] of dtype      (input dP)
 *   dscores  device [rows, ld] of dtype      (output; may equal dprobs)
 *   delta    device float [rows] or NULL     (output; needed later by fos_sink_grad)
 */
fos_status fos_softmax_bwd(const fos_desc *desc, fos_dtype dtype, const void *probs,
                           const void *dprobs, void *dscores, float *delta,
                           cudaStream_t stream, const fos_launch *launch);

/*
 * Sink gradient: d_sink[h] = -sum_r exp(sink_h - lse_r) * delta_r over the rows of head h,
 * taken in (b, i) order in chunks of 256 rows (lane-local ascending sums of 8, warp xor
 * tree, chunk partials added left to right); no atomics.  A head whose sink is -inf gets 0.
 * ("[ROCm] Jax Add softmax sink (learnable off-by-one) support": one sink value per head,
 * d_sink reduced per head; the CK code there accumulates with atomicAdd, which this
 * replaces by a fixed order.)
 *   desc->sink must be non-NULL (FOS_ERR_INVALID otherwise).
 *   lse, delta  device float [rows]  (inputs, as written by the forward and the backward)
 *   d_sink      device float [heads] (output)
 */
fos_status fos_sink_grad(const fos_desc *desc, const float *lse, const float *delta,
                         float *d_sink, cudaStream_t stream, const fos_launch *launch);

/*
 * The backward and the sink gradient in one call: the results of fos_softmax_bwd followed by
 * fos_sink_grad, bit for bit.  Staged rows of more than 8 tiles with at least four octets per
 * CTA are taken by octets, 8 consecutive positions (b, i) of one head: the backward writes each
 * octet's ascending float32 sum of c_r = -(exp(sink_h - lse_r) * delta_r) to the workspace and
 * a small kernel combines them per head by the sink gradient's own chunk tree and left-to-right
 * order, so delta and LSE are never read back and no atomic is used.  Otherwise the two
 * launches run (delta to the workspace when none is given): for rows of at most 8 tiles they
 * are the faster way (the one-warp kernel takes octets only when launch->sink_fusion is 1),
 * and rows streamed in segments take no octets.  ("[ROCm] Jax Add softmax sink (learnable
 * off-by-one) support", Description and review thread: d_sink reduced per head inside the
 * backward; there by atomicAdd into a zeroed buffer, here in a fixed order.)
 *   desc->sink    required (FOS_ERR_INVALID otherwise)
 *   probs, dprobs, dscores, delta  as fos_softmax_bwd (delta may be NULL)
 *   lse           device float [rows] (input, as written by the forward)
 *   d_sink        device float [heads] (output)
 *   workspace     device, 16-byte aligned, at least fos_bwd_sink_workspace_bytes(desc) bytes
 *                 (the octet sums, or delta when none is given and the octets are not taken);
 *                 owned by the caller, not to be touched until `stream` completes
 * heads == 0 is a no-op; rows == 0 writes d_sink = 0.
 */
fos_status fos_softmax_bwd_sink(const fos_desc *desc, fos_dtype dtype, const void *probs,
                                const void *dprobs, void *dscores, float *delta,
                                const float *lse, float *d_sink, void *workspace,
                                size_t workspace_bytes, cudaStream_t stream,
                                const fos_launch *launch);

/* Workspace bytes of fos_softmax_bwd_sink: 4 * max(rows, heads * ceil(batch * q_len / 8)),
 * rounded up to 256 (0 for an invalid description).  Host arithmetic only. */
size_t fos_bwd_sink_workspace_bytes(const fos_desc *desc);

/*
 * The sink gradient with the rows sharded by batch entry (one shard per device, say): each
 * shard writes the chunk partials of fos_sink_grad for its batch entries; the partials of all
 * shards, concatenated per head in chunk order (shard order), go through fos_sink_grad_merge,
 * which adds them left to right.  The result has the bits of fos_sink_grad on the whole batch,
 * because each chunk's partial is the same sum and the final additions happen in the same
 * order.  ("[ROCm] Jax Add softmax sink (learnable off-by-one) support": d_sink is a per-head
 * sum over batch and query rows; here the cross-shard step is a gather, not an all-reduce,
 * whose order would not be fixed.)
 *   batch_begin, batch_end  the shard's batch entries [b0, b1), 0 <= b0 <= b1 <= batch (an
 *                           empty shard is a no-op with no chunks); for a non-empty one the
 *                           shard's positions [b0*q_len, b1*q_len) of a head must start on a
 *                           multiple of 256 and end on one unless b1 == batch
 *                           (FOS_ERR_INVALID otherwise)
 *   lse, delta              device float [(b1-b0)*heads*q_len]: the shard's rows only
 *   partials                device float [heads][c1 - c0] (output), c0 = b0*q_len/256,
 *                           c1 = ceil(b1*q_len/256)
 *   desc                    the whole problem (batch = all shards); desc->sink required
 */
fos_status fos_sink_grad_partials(const fos_desc *desc, int32_t batch_begin, int32_t batch_end,
                                  const float *lse, const float *delta, float *partials,
                                  cudaStream_t stream, const fos_launch *launch);

/*
 * d_sink[h] = +0 + partials[h][0] + partials[h][1] + ... in float32, left to right, on the
 * host (no CUDA call): the merge of fos_sink_grad_partials' outputs.
 *   partials  host float [heads][nchunks], every shard's chunks in order
 *   d_sink    host float [heads] (output)
 * FOS_ERR_INVALID for negative sizes or missing pointers; heads == 0 is a no-op.
 */
fos_status fos_sink_grad_merge(int32_t heads, int64_t nchunks, const float *partials,
                               float *d_sink);

/*
 * The forward, the backward and (when d_sink is given) the sink gradient of one batch whose
 * data live in HOST memory: the same results, bit for bit, as fos_softmax_fwd on a device
 * copy of scores, fos_softmax_bwd on the P it produced and dprobs, and fos_sink_grad, with
 * every outcome copied back.  Rows are processed in chunks of `chunk_rows` (0 = about 16 MB
 * of one tensor per chunk) that cycle through three slots of `workspace`: the upload of one
 * chunk, the kernels of the previous one and the download of the one before that overlap on
 * three streams (two of them the library's own, ordered against `stream` by events).  This is
 * the data movement a caller with host-resident data needs around the softmax ("Batch-
 * invariant attention (standard softmax--cuda version)", Acceptance Criteria: the outputs
 * must not depend on how rows are batched; here they do not depend on the chunking either).
 *   scores, dprobs        host [rows, ld] of dtype  (inputs; page-locked memory lets the
 *                         copies overlap, pageable memory is correct but serialises them)
 *   probs, dscores        host [rows, ld] of dtype  (outputs; columns key_len..ld-1 of the
 *                         host rows are not written)
 *   lse, delta            host float [rows]         (outputs)
 *   d_sink                host float [heads] or NULL (output; needs desc->sink)
 *   desc->kv_valid_len, key_mask, sink stay DEVICE pointers, as in the other calls.
 *   workspace             device, 256-byte aligned, at least
 *                         fos_step_host_workspace_bytes(desc, dtype, chunk_rows) bytes;
 *                         owned by the caller, not to be touched until `stream` completes.
 * The call returns once everything is enqueued; the outputs are complete when `stream` is.
 * FOS_ERR_INVALID also for a missing or too small or misaligned workspace, a negative
 * chunk_rows, or d_sink without a sink.  rows == 0 is valid and enqueues nothing.  On
 * FOS_ERR_CUDA part of the pipeline may already be enqueued; the outputs are then undefined.
 */
fos_status fos_softmax_step_host(const fos_desc *desc, fos_dtype dtype, const void *scores,
                                 const void *dprobs, void *probs, float *lse, void *dscores,
                                 float *delta, float *d_sink, void *workspace,
                                 size_t workspace_bytes, int64_t chunk_rows, cudaStream_t stream,
                                 const fos_launch *launch);

/*
 * Device workspace bytes fos_softmax_step_host needs for this problem and chunk size
 * (0 = the default chunk): the full LSE and delta arrays, d_sink, and three slots of two
 * chunk tensors.  Host arithmetic only (no CUDA call).  Returns 0 for an invalid
 * description, dtype or chunk_rows, and for rows == 0.
 */
size_t fos_step_host_workspace_bytes(const fos_desc *desc, fos_dtype dtype, int64_t chunk_rows);

/* Bytes of the scratch array built into the library for fos_softmax_step_host_static. */
#define FOS_STEP_HOST_STATIC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * fos_softmax_step_host for callers that cannot allocate device memory: no workspace
 * argument; the step uses a scratch array of FOS_STEP_HOST_STATIC_SCRATCH_BYTES (32 MB) that
 * is part of the library and held by every GPU that loads it until the process exits.  Made
 * for a host application whose memory manager already owns the device memory it may use (a
 * serving engine that reserves its cache pool up front, a framework whose caching allocator
 * must account for every block), or a code path that must not call cudaMalloc / cudaFree
 * (cudaFree synchronises the whole device).  It calls neither, nor any routine that allocates
 * device memory.  The pages describe no counterpart of this entry point: it is data movement
 * around the softmax, not part of the method.
 *   Arguments as fos_softmax_step_host, minus the workspace.  chunk_rows = 0 takes the default
 *   chunk, shrunk until the LSE, delta and d_sink arrays and three slots of two chunk tensors
 *   fit the array.
 *   FOS_ERR_UNSUPPORTED when they do not fit even with the given (or a one-row) chunk: roughly
 *   8 * rows + 4 * heads + 6 * chunk_rows * ld * element size > 32 MB.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress) and
 * creates the pipeline's streams and events: make that first call before any stream capture.
 * Every call uses the same array, so calls that overlap on the GPU (on two streams with no
 * order between them) race; calls on one stream are ordered.  Nothing in the array needs to
 * start at zero: each call writes what it reads there.
 */
fos_status fos_softmax_step_host_static(const fos_desc *desc, fos_dtype dtype,
                                        const void *scores, const void *dprobs, void *probs,
                                        float *lse, void *dscores, float *delta, float *d_sink,
                                        int64_t chunk_rows, cudaStream_t stream,
                                        const fos_launch *launch);

/*
 * The QK contraction in front of the softmax: scores[b, h, i, j] = scale * sum_d q[b, h, i, d]
 * * k[b, h / (q_heads / kv_heads), j, d] on the tensor cores, the head dimension accumulated in
 * float32 in a fixed order (steps of 16, ascending), then multiplied by `scale` (one rounding)
 * and rounded once to the output dtype.  Each score depends only on its query row and key row,
 * so it has the same bits whatever the batch, the heads around it or its position.
 * ("Batch-invariant attention (standard softmax--cuda version)", Fixed Reduction Contract: one
 * writer per score, the head dimension in a fixed order; "[WS1][kernels] Add fixed-order
 * joint-attention softmax for Qwen-Image", Summary: the QK GEMM feeds the softmax.)
 */
typedef struct fos_qk_desc {
  int32_t batch;      /* B */
  int32_t q_heads;    /* Hq, a multiple of kv_heads */
  int32_t kv_heads;   /* Hkv >= 1; query head h reads key head h / (Hq / Hkv) */
  int32_t q_len;      /* Sq, query rows per (batch, query head) */
  int32_t kv_len;     /* Skv, keys per (batch, key head) */
  int32_t head_dim;   /* D: 64 or 128 */
  int64_t ld_scores;  /* elements between rows of scores, >= kv_len */
  float scale;        /* applied to the float32 sum (e.g. 1 / sqrt(D)) */
  int32_t tile_n;     /* 0 = default: one CTA per SM walks 128 x 128 tiles, one tile's stores
                         overlapping the next tile's copies and multiplies; 128 or 256: one CTA
                         per tile of that many keys.  No result bit depends on it: each score's
                         sum is the same sequence of instructions. */
} fos_qk_desc;

/*
 *   q       device [batch][q_heads][q_len][head_dim] of in_dtype (FOS_BF16 or FOS_F16), dense
 *   k       device [batch][kv_heads][kv_len][head_dim] of in_dtype, dense
 *   scores  device [batch][q_heads][q_len][ld_scores] of out_dtype (FOS_F32, FOS_BF16 or
 *           FOS_F16); columns kv_len .. ld_scores-1 are not written
 * q, k and scores must start on 16-byte boundaries and ld_scores * (size of out_dtype) must be
 * a multiple of 16 (FOS_ERR_UNSUPPORTED otherwise); scores must not overlap q or k.
 * FOS_ERR_INVALID for a bad description (negative sizes, q_heads not a multiple of kv_heads,
 * ld_scores < kv_len, tile_n not 0, 128 or 256) or dtype; FOS_ERR_UNSUPPORTED for another
 * head dimension or more than 65535 (batch x query heads) or query tiles of 128.  A problem with no score is a
 * no-op.  Resources: with tile_n = 0, one CTA per SM that allocates all 512 tensor-memory
 * columns (four accumulators); with tile_n given, tile_n columns per CTA.  Every CTA frees its
 * columns before it exits.  A bounded wait that runs out is reported by fos_device_error() as
 * FOS_ERR_TIMEOUT.
 */
fos_status fos_qk_scores(const fos_qk_desc *desc, fos_dtype in_dtype, fos_dtype out_dtype,
                         const void *q, const void *k, void *scores, cudaStream_t stream);

/*
 * The PV contraction behind the softmax: out[b, h, i, d] = scale * sum_j probs[b, h, i, j] *
 * v[b, h / (q_heads / kv_heads), j, d] on the tensor cores, the keys accumulated in float32 in a
 * fixed order (steps of 16, ascending from key 0), multiplied by scale (one rounding; scale 1 is
 * an exact no-op) and rounded once to the output dtype.  With (probs, v, scale) = (dScores, K,
 * the score scale) the same call gives the query gradient dQ.  Each output depends only on its
 * probability row and the value rows, so it has the same bits whatever the batch, the heads
 * around it or its row's position.  ("Batch-invariant attention (standard softmax--cuda
 * version)", Fixed Reduction Contract: one writer per output, the keys in a fixed order;
 * "[WS1][kernels] Add fixed-order joint-attention softmax for Qwen-Image", Summary: the softmax
 * feeds the AV GEMM.)
 */
typedef struct fos_pv_desc {
  int32_t batch;      /* B */
  int32_t q_heads;    /* Hq, a multiple of kv_heads */
  int32_t kv_heads;   /* Hkv >= 1; query head h reads value head h / (Hq / Hkv) */
  int32_t q_len;      /* Sq */
  int32_t kv_len;     /* Skv (>= 1 for fos_pv_out) */
  int32_t head_dim;   /* D: 64 or 128 */
  int64_t ld_probs;   /* elements between rows of probs (of `a` for fos_grad_kv), >= kv_len */
  float scale;        /* finite and nonzero: 1 for P V */
} fos_pv_desc;

/*
 *   probs  device [batch][q_heads][q_len][ld_probs] of in_dtype (FOS_BF16 or FOS_F16): P, as the
 *          forward writes it (columns kv_len .. ld_probs-1 are not read)
 *   v      device [batch][kv_heads][kv_len][head_dim] of in_dtype, dense
 *   out    device [batch][q_heads][q_len][head_dim] of out_dtype (FOS_F32, FOS_BF16, FOS_F16),
 *          dense; must not overlap probs or v
 * probs, v and out must start on 16-byte boundaries and ld_probs must be a multiple of 8
 * (FOS_ERR_UNSUPPORTED otherwise).  FOS_ERR_INVALID for a bad description (negative sizes,
 * kv_len < 1, q_heads not a multiple of kv_heads, ld_probs < kv_len, scale zero or not finite)
 * or dtype; FOS_ERR_UNSUPPORTED for another head dimension or more than 65535 (batch x query
 * heads).  A problem with no output is a no-op.  Resources: each CTA allocates head_dim
 * tensor-memory columns and frees them before it exits; a bounded wait that runs out is
 * reported by fos_device_error() as FOS_ERR_TIMEOUT.
 */
fos_status fos_pv_out(const fos_pv_desc *desc, fos_dtype in_dtype, fos_dtype out_dtype,
                      const void *probs, const void *v, void *out, cudaStream_t stream);

/*
 * The contraction behind the key and value gradients of attention:
 *   out[b, g, j, d] = scale * sum over the query heads h = g*G .. g*G + G - 1 (G = q_heads /
 *                     kv_heads, ascending) and the query positions i = 0 .. q_len - 1
 *                     (ascending, in steps of 16) of a[b, h, i, j] * m[b, h, i, d],
 * accumulated in float32 on the tensor cores, multiplied by scale (one rounding) and rounded once
 * to the output dtype.  (a, m, scale) = (P, dO, 1) gives dV, (dScores, Q, the score scale) dK.
 * Each output has one writer and depends only on its key's column of a and on m, so it has the
 * same bits whatever the batch or its key's position.  ("Batch-invariant attention (standard
 * softmax--cuda version)", GQA backward: each dK / dV element accumulates the group's query
 * heads, then the query positions, in a fixed order, with no atomics.)
 *   desc   as for fos_pv_out, ld_probs giving the row stride of a; kv_len >= 0
 *   a      device [batch][q_heads][q_len][ld_probs] of in_dtype (FOS_BF16 or FOS_F16); columns
 *          kv_len .. ld_probs-1 are not read
 *   m      device [batch][q_heads][q_len][head_dim] of in_dtype, dense
 *   out    device [batch][kv_heads][kv_len][head_dim] of out_dtype, dense; must not overlap a or m
 * Alignment and errors as for fos_pv_out (more than 65535 (batch x kv_heads) is
 * FOS_ERR_UNSUPPORTED).  q_len == 0 writes +0 to every output; a problem with no output is a
 * no-op.  Resources: each CTA allocates head_dim tensor-memory columns and frees them before it
 * exits; a bounded wait that runs out is reported by fos_device_error() as FOS_ERR_TIMEOUT.
 */
fos_status fos_grad_kv(const fos_pv_desc *desc, fos_dtype in_dtype, fos_dtype out_dtype,
                       const void *a, const void *m, void *out, cudaStream_t stream);

/*
 * Synchronises `stream`, then reports and clears the device error word of the current
 * device: FOS_ERR_TIMEOUT if a kernel's bounded wait ran out since the last call, FOS_ERR_INDEX
 * if an index check of the debug build failed, FOS_OK otherwise (FOS_ERR_CUDA if the
 * synchronisation itself failed).
 */
fos_status fos_device_error(cudaStream_t stream);

/* Static, NUL-terminated name of a status. */
const char *fos_status_string(fos_status status);

/* Static string naming the arithmetic contract: tile, lane layout, trees, exp form, arch. */
const char *fos_contract_fingerprint(void);

#ifdef __cplusplus
}
#endif

#endif /* FOS_SOFTMAX_H */
