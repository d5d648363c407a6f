/*
 * lora.h -- C ABI of liblora.so, the multi-LoRA batched linear layer for
 * GB300 (sm_103a).
 *
 * The layer (row-vector form, as in "Serving multiple LoRAs: segmented matrix
 * multiplies and adapter scheduling", section "Not merging the weights,
 * computing in batches"):
 *
 *     y[t,:] = x[t,:] W0 + s[a_t] * (x[t,:] A[a_t]) B[a_t]
 *
 * for a batch of T tokens that may each use a different adapter a_t, or none
 * (a_t = -1: base only, as in the "Replay" figure of "Serving many LoRA
 * adapters", blog.ecitis.org: "req C -> base only").  The base product runs
 * once for the whole batch; the adapter term is gathered per token (BGMV) or
 * per segment of tokens sorted by adapter (SGMV), first shrinking to rank r
 * and then expanding back ("Serving multiple LoRAs ...", the paragraph after
 * the toy script: shrink x -> xA, then expand and add into the base output).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Arrays are caller-owned DEVICE pointers to dense row-major storage.  Data
 *    pointers must be 16-byte aligned.  x and y must not alias.
 *  - Layouts (element type = dt for x, W0, A_pool, B_pool, y):
 *        x       [T, d_in]
 *        W0      [d_in, d_out]
 *        A_pool  [n_slots, d_in, r]     adapter a's A is A_pool[a]
 *        B_pool  [n_slots, r, d_out]    adapter a's B is B_pool[a]
 *        scale   [n_slots] float32      s[a] = alpha/r of adapter a; it
 *                travels with the adapter ("Serving many LoRA adapters",
 *                section "Correctness across tenants").  NULL means 1.0.
 *        slot_ids[T] int32              -1 = base only.  Any id outside
 *                [-1, n_slots) is treated as base only and sets
 *                LORA_DEVERR_BAD_SLOT in the workspace error word.
 *        v_partial [ksplit, T, r] float32: shrink output split over d_in into
 *                ksplit contiguous ranges; v = sum over the first index.  The
 *                scale is already applied (v = s * x A).
 *  - Shapes: T >= 0; d_in, d_out >= 8 and multiples of 8; r in {8,16,32,64,
 *    128}; 1 <= n_slots <= LORA_MAX_SLOTS; T <= LORA_MAX_TOKENS; 1 <= ksplit
 *    <= LORA_MAX_KSPLIT.  T = 0 is a valid empty batch (nothing is launched).
 *  - Workspace: every call takes a caller-owned device workspace `ws` of at
 *    least lora_workspace_bytes(op, ...) bytes.  Its first 16 bytes hold the
 *    sticky device error word; zero-fill the workspace once before first use.
 *    One workspace must not be used by two calls that run concurrently.
 *  - Streams: every call only enqueues work on `stream` (a cudaStream_t;
 *    NULL = the legacy default stream) and returns; nothing synchronises
 *    except lora_get_error.  The library allocates no memory and keeps no
 *    per-call global state.  Calls can be captured into CUDA graphs.
 *  - Errors: host-side validation failures return a status != LORA_OK and
 *    launch nothing.  LORA_ERR_CUDA reports a launch failure.  Data-dependent
 *    problems found on the device never trap: they set bits in the workspace
 *    error word, read back by lora_get_error.
 *  - dt: LORA_DTYPE_BF16 (bf16 storage, fp32 accumulation, tensor cores for
 *    the base product) or LORA_DTYPE_F32 (fp32 storage and arithmetic on CUDA
 *    cores; meant for small checks).
 */
#ifndef LORA_H_
#define LORA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LORA_OK = 0,
  LORA_ERR_INVALID_ARG = 1, /* null pointer, misaligned pointer, negative size */
  LORA_ERR_SHAPE = 2,       /* unsupported dimension (see conventions)          */
  LORA_ERR_DTYPE = 3,       /* unknown dtype                                     */
  LORA_ERR_WORKSPACE = 4,   /* ws NULL or smaller than lora_workspace_bytes      */
  LORA_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed              */
  LORA_ERR_DEVICE = 6       /* current device is not a GB300-class sm_103 GPU    */
} lora_status_t;

typedef enum { LORA_DTYPE_BF16 = 0, LORA_DTYPE_F32 = 1 } lora_dtype_t;

/* operation codes for lora_workspace_bytes */
typedef enum {
  LORA_OP_BUILD_SEGMENTS = 0,
  LORA_OP_BGMV_SHRINK = 1,
  LORA_OP_BGMV_EXPAND = 2,
  LORA_OP_SGMV_SHRINK = 3,
  LORA_OP_SGMV_EXPAND = 4,
  LORA_OP_LINEAR_FUSED = 5,
  LORA_OP_BASE_GEMM_EXPAND = 6,
  LORA_OP_LINEAR_FUSED_4BIT = 7,
  LORA_OP_LINEAR_FUSED_RAGGED = 8
} lora_op_t;

/* device error word bits */
#define LORA_DEVERR_BAD_SLOT 0x1u /* a slot id outside [-1, n_slots) was read   */
#define LORA_DEVERR_TIMEOUT 0x2u  /* a bounded on-chip wait gave up (no hang)   */
#define LORA_DEVERR_BAD_RANK 0x4u /* a ragged-pool entry (rank, offsets) read was out of range */
/* debug builds of the library only (-DLORA_DEBUG, liblora_debug.so): an index
 * handed from one kernel to another (segment offsets, perm rows, segment
 * slots) fell outside its buffer; it was replaced by 0, so nothing was read or
 * written outside a buffer.  Release builds never set it. */
#define LORA_DEVERR_BOUNDS 0x8u

#define LORA_MAX_SLOTS 16384
#define LORA_MAX_TOKENS (1 << 20)
#define LORA_MAX_KSPLIT 64

/* Bytes of workspace `op` needs for these sizes (>= 16; the error word). */
size_t lora_workspace_bytes(int32_t op, int32_t T, int32_t d_in, int32_t d_out, int32_t r,
                            int32_t n_slots);

/*
 * Segment builder (SGMV's sort step: "Serving multiple LoRAs ...", SGMV
 * bullet -- tokens of one adapter are placed together -- and its toy script,
 * which groups by a stable sort of the ids).
 *   perm     [T]   out: token indices, stably sorted by slot id; base-only
 *                  (and invalid) tokens come first.
 *   seg_slot [min(T, n_slots)] out: ids >= 0 present in the batch, ascending;
 *                  entries past n_seg are left untouched.
 *   seg_off  [min(T, n_slots) + 1] out: segment j is perm[seg_off[j] ..
 *                  seg_off[j+1]); seg_off[n_seg] = T; seg_off[0] is the count
 *                  of base-only tokens.
 *   n_seg    [1]   out: number of segments (device int; no host sync).
 * Bit-exact: equals a stable argsort of the ids followed by run-length
 * grouping.  One CTA; latency-bound.
 */
lora_status_t lora_build_segments(const int32_t* slot_ids, int32_t T, int32_t n_slots,
                                  int32_t* perm, int32_t* seg_slot, int32_t* seg_off,
                                  int32_t* n_seg, void* ws, size_t ws_bytes, void* stream);

/*
 * BGMV shrink ("Serving multiple LoRAs ...", BGMV bullet: each token gathers
 * its adapter's A by index): for every token t with a valid id,
 *   v_partial[s, t, :] = s[a_t] * x[t, K_s] A[a_t][K_s, :]
 * over the s-th of ksplit contiguous, 8-aligned ranges K_s of d_in.  Rows of
 * base-only tokens are written as zeros.  Overwrites v_partial.
 */
lora_status_t lora_bgmv_shrink(const void* x, const void* A_pool, const int32_t* slot_ids,
                               const float* scale, float* v_partial, int32_t T, int32_t d_in,
                               int32_t r, int32_t n_slots, int32_t ksplit, lora_dtype_t dt,
                               void* ws, size_t ws_bytes, void* stream);

/*
 * BGMV expand ("Serving multiple LoRAs ...", BGMV bullet: each token gathers
 * its own adapter's factors by index; the paragraph after the toy script:
 * the rank-r result is expanded with B and added into the base output):
 * y[t, :] += (sum_s v_partial[s, t, :]) B[a_t] for tokens with a valid id
 * (fp32 arithmetic, one rounding to dt per element).  Base-only rows of y
 * are not touched.  Accumulates into y.
 */
lora_status_t lora_bgmv_expand(const float* v_partial, int32_t ksplit, const void* B_pool,
                               const int32_t* slot_ids, void* y, int32_t T, int32_t r,
                               int32_t d_out, int32_t n_slots, lora_dtype_t dt, void* ws,
                               size_t ws_bytes, void* stream);

/*
 * SGMV shrink ("Serving Many LoRA Adapters", section "Punica: The Segmented
 * Gather-Scatter Kernel"; "Serving multiple LoRAs ...", SGMV bullet): the
 * shrink done segment by segment, each segment reading its adapter's A once.
 * Takes the outputs of lora_build_segments (device arrays; n_seg is read on
 * the device).  Same output contract as lora_bgmv_shrink: v_partial rows of
 * every token are written (zeros for base-only tokens).
 */
lora_status_t lora_sgmv_shrink(const void* x, const void* A_pool, const int32_t* perm,
                               const int32_t* seg_slot, const int32_t* seg_off,
                               const int32_t* n_seg, const float* scale, float* v_partial,
                               int32_t T, int32_t d_in, int32_t r, int32_t n_slots,
                               int32_t ksplit, lora_dtype_t dt, void* ws, size_t ws_bytes,
                               void* stream);

/*
 * SGMV expand ("Serving multiple LoRAs ...", SGMV bullet: one segment per
 * adapter, so its factors are read once for the segment; the paragraph
 * after the toy script: expand with B and add into the base output):
 * per segment, y[t, :] += (sum_s v_partial[s, t, :]) B[a] for the
 * segment's tokens, reading B[a] once per segment.  Accumulates into y;
 * base-only rows untouched.
 */
lora_status_t lora_sgmv_expand(const float* v_partial, int32_t ksplit, const void* B_pool,
                               const int32_t* perm, const int32_t* seg_slot,
                               const int32_t* seg_off, const int32_t* n_seg, void* y, int32_t T,
                               int32_t r, int32_t d_out, int32_t n_slots, lora_dtype_t dt,
                               void* ws, size_t ws_bytes, void* stream);

/*
 * The whole layer: y = x W0 + s (x A) B, y OVERWRITTEN and written once
 * ("Multi-LoRA batching and adapter paging", section "Walking through a
 * batch": the base product once for all rows, then each row's adapter term;
 * "Serving many LoRA adapters", "Replay" figure: segmented gather, grouped
 * GEMM, scatter add, one fused output).  Batches of up to 256 tokens
 * (decode) take the per-token BGMV path: for bf16 the base product split
 * over d_in into fp32 partials (lora_base_gemm_splitk), then one kernel that
 * computes each token's adapter term, adds the partials and stores y
 * (lora_bgmv_adapter_merge).  fp32 takes the BGMV shrink and a CUDA-core
 * layer kernel.  Larger batches (prefill) take the segment builder, the
 * segment-grouped SGMV shrink and a base GEMM whose tensor-memory
 * accumulator also takes the expand as extra K-blocks
 * (lora_base_gemm_expand).  Either way y is stored once.
 *
 * Overlap with the previous kernel (bf16 decode-sized batches): the first
 * kernel is launched as a programmatic dependent of whatever precedes it
 * in the stream.  If that kernel lets its dependents start early
 * (griddepcontrol.launch_dependents), this layer's W0 starts streaming
 * before it completes; everything else (x, the ids, the adapters, the
 * scales) is read only after it completed.  So W0 must not be written by a
 * kernel that lets its dependents start early and runs right before this
 * call.  The last kernel of this call lets the next one start early in the
 * same way, so consecutive layers overlap.
 */
lora_status_t lora_linear_fused(const void* x, const void* W0, const void* A_pool,
                                const void* B_pool, const int32_t* slot_ids, const float* scale,
                                void* y, int32_t T, int32_t d_in, int32_t d_out, int32_t r,
                                int32_t n_slots, lora_dtype_t dt, void* ws, size_t ws_bytes,
                                void* stream);

/*
 * BGMV expand into an fp32 adapter term (bf16 B only):
 *   delta[t, :] = (sum_s v_partial[s, t, :]) B[a_t]      for tokens with a valid id
 * delta [T, d_out] float32, rows of base-only tokens are not written.  This
 * is the expand of lora_linear_fused for decode-sized batches (T <= 256): it
 * runs while the base GEMM streams W0 and lora_base_gemm_delta adds it in
 * its epilogue ("Serving multiple LoRAs ...": the expand is added directly
 * to the base output; BGMV suits decode).  Workspace: the error word only.
 */
lora_status_t lora_bgmv_delta(const float* v_partial, int32_t ksplit, const void* B_pool,
                              const int32_t* slot_ids, float* delta, int32_t T, int32_t r,
                              int32_t d_out, int32_t n_slots, lora_dtype_t dt, void* ws,
                              size_t ws_bytes, void* stream);

/*
 * The whole BGMV adapter term of every token in one launch (bf16 only):
 *   delta[t, :] = scale[a_t] * (x[t, :] A[a_t]) B[a_t]    for tokens with a valid id
 * fp32 delta [T, d_out]; rows of base-only tokens are not written
 * ("Serving multiple LoRAs: segmented matrix multiplies and adapter
 * scheduling", BGMV bullet and the paragraph after the toy script: shrink to
 * rank r, then expand).  One thread-block cluster per token: its CTAs shrink
 * slices of d_in, sum the rank-r partials through distributed shared memory
 * in a fixed order (deterministic) and expand slices of d_out.
 * lora_bgmv_adapter_merge is the same kernel adding the base product, the
 * last kernel of lora_linear_fused for bf16 batches of up to 256 tokens.
 * T <= 65535.  scale may be null (1.0).  Workspace: the error word only.
 */
lora_status_t lora_bgmv_adapter(const void* x, const void* A_pool, const void* B_pool,
                                const int32_t* slot_ids, const float* scale, float* delta,
                                int32_t T, int32_t d_in, int32_t d_out, int32_t r,
                                int32_t n_slots, lora_dtype_t dt, void* ws, size_t ws_bytes,
                                void* stream);

/*
 * The merge form of lora_bgmv_adapter: the last kernel of lora_linear_fused
 * for bf16 batches of up to 256 tokens (bf16 only):
 *   y[t, :] = sum_s partial[s, t, :] + scale[a_t] (x[t, :] A[a_t]) B[a_t]   (a_t valid)
 *   y[t, :] = sum_s partial[s, t, :]                                        (base only)
 * partial [ksplit, T, d_out] fp32 is any split of the base product x W0
 * over d_in (lora_base_gemm_splitk writes one).  y [T, d_out] bf16 is
 * OVERWRITTEN, every row, rounded once ("Multi-LoRA batching and adapter
 * paging", section "Walking through a batch": the base product once for
 * all rows, each row then gets its own adapter term).  1 <= ksplit <=
 * LORA_MAX_KSPLIT; T <= 65535; scale may be null (1.0).  Workspace: the
 * error word only.
 */
lora_status_t lora_bgmv_adapter_merge(const void* x, const void* A_pool, const void* B_pool,
                                      const int32_t* slot_ids, const float* scale,
                                      const float* partial, int32_t ksplit, void* y, int32_t T,
                                      int32_t d_in, int32_t d_out, int32_t r, int32_t n_slots,
                                      lora_dtype_t dt, void* ws, size_t ws_bytes, void* stream);

/*
 * The shared base product split over d_in, on tcgen05 tensor cores with
 * the token dimension as the MMA's N (bf16 only):
 *   partial[s, t, :] = x[t, K_s] W0[K_s, :]      s = 0 .. S-1
 * where K_0 .. K_{S-1} are contiguous ranges of d_in that together cover it
 * ("Multi-LoRA batching and adapter paging", section "Walking through a
 * batch": one base product for the whole batch), so sum_s partial[s] =
 * x W0.  partial [S, T, d_out] (S = ksplit) fp32, caller-owned, fully
 * written.  1 <= ksplit <= the number of 192-row (T <= 64) or 128-row
 * (T > 64) blocks of d_in and <= LORA_MAX_KSPLIT, or ksplit == 0 for the
 * split lora_linear_fused uses (S = lora_decode_split(T, d_in, d_out);
 * 1 <= T <= 256 only).  Any T; it is built for T <= 256.  Workspace: the
 * error word only.
 */
lora_status_t lora_base_gemm_splitk(const void* x, const void* W0, float* partial, int32_t T,
                                    int32_t d_in, int32_t d_out, int32_t ksplit, lora_dtype_t dt,
                                    void* ws, size_t ws_bytes, void* stream);

/*
 * The ksplit lora_linear_fused uses for the base product of a bf16 batch of
 * 1 <= T <= 256 tokens: (d_out / 128 column tiles) x ksplit ~ 152 CTAs.  A
 * function of the shapes only: it is laid out for a 152-SM GB300 whatever
 * the current device, so results do not depend on the device.  0 for other
 * T or invalid dimensions.
 */
int32_t lora_decode_split(int32_t T, int32_t d_in, int32_t d_out);

/*
 * Diagnostic for tests of the failure path; the pages have no counterpart.
 * Enqueues the kernel of lora_base_gemm_splitk (ksplit 1) with its TMA
 * producer held back, so nothing ever arrives on the barrier its MMA issuer
 * waits on.  Each bounded wait of the kernel gives up after wait_us
 * microseconds (1 <= wait_us <= 2,000,000; the library's kernels otherwise
 * use 2 s); the kernel then sets LORA_DEVERR_TIMEOUT in the workspace error
 * word, writes nothing to partial, frees its tensor memory and returns, so
 * the device stays usable.  partial is [1, T, d_out] fp32 (not written);
 * 1 <= T <= 256.  Workspace: the error word only.
 */
lora_status_t lora_debug_gemm_wait_timeout(const void* x, const void* W0, float* partial,
                                           int32_t T, int32_t d_in, int32_t d_out,
                                           int32_t wait_us, void* ws, size_t ws_bytes,
                                           void* stream);

/*
 * The last kernel of lora_linear_fused on its own: the shared base product
 * with the expand folded into the same accumulator, given the shrink output.
 *   y[t, :] = x[t, :] W0 + (sum_s v_partial[s, t, :]) B[a_t]   (a_t valid)
 *   y[t, :] = x[t, :] W0                                       (base only)
 * y is OVERWRITTEN and written once.  v_partial is any shrink output
 * (lora_bgmv_shrink or lora_sgmv_shrink, scale applied).  bf16: tcgen05
 * tensor cores with the accumulator in tensor memory; fp32: CUDA cores.
 * Workspace: the 16-byte error word only.
 */
lora_status_t lora_base_gemm_expand(const void* x, const void* W0, const void* B_pool,
                                    const int32_t* slot_ids, const float* v_partial,
                                    int32_t ksplit, void* y, int32_t T, int32_t d_in,
                                    int32_t d_out, int32_t r, int32_t n_slots, lora_dtype_t dt,
                                    void* ws, size_t ws_bytes, void* stream);

/*
 * The whole layer (same contract and result as lora_linear_fused) for
 * callers that cannot allocate device memory: code running under a
 * framework whose allocator already owns the GPU's memory, plugins the host
 * process does not let allocate, and paths that forbid allocation once they
 * are running.  The pages have no counterpart; this is a library concern.
 *
 * Scratch: a fixed array of LORA_NOALLOC_SCRATCH_BYTES inside the library.
 * Its device memory is committed when the library's device code is loaded
 * on a GPU: under CUDA's lazy module loading (the default) that happens in
 * the first call on each device; with CUDA_MODULE_LOADING=EAGER, when the
 * process first uses the GPU.  It is held until the process exits.  Make
 * the first call on each device before an allocator reserves the rest of
 * its memory, or that first call may fail (LORA_ERR_CUDA).  Batches whose
 * scratch (lora_workspace_bytes(LORA_OP_LINEAR_FUSED, ...)) is larger are
 * refused with LORA_ERR_WORKSPACE, and every other invalid argument with
 * its status, before anything is enqueued.  The call allocates nothing (no
 * cudaMalloc, no allocating library routine).
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it; make that first call before any stream
 * capture.  Every call shares the one array: calls whose GPU work overlaps
 * (other streams, other threads) race on it.  Each call clears the error
 * word it keeps in the array; device error bits are not reported back (ids
 * outside [-1, n_slots) are still read as base-only).
 */
#define LORA_NOALLOC_SCRATCH_BYTES (8u << 20)
lora_status_t lora_linear_fused_noalloc(const void* x, const void* W0, const void* A_pool,
                                        const void* B_pool, const int32_t* slot_ids,
                                        const float* scale, void* y, int32_t T, int32_t d_in,
                                        int32_t d_out, int32_t r, int32_t n_slots,
                                        lora_dtype_t dt, void* stream);

/*
 * Ragged-rank adapter pools: each adapter keeps its own rank instead of being
 * zero-padded to the largest one ("Serving Many LoRA Adapters", section
 * "When It Falls Down": padding a rank-4 adapter to rank 64 costs 16x on its
 * term; "Serving multiple LoRAs ...", Exercise 2: kernels that take
 * variable ranks; "Serving many LoRA adapters", section "Batching across
 * different adapters": mixed ranks need ragged indexing or padding).
 *   A_flat, B_flat  bf16, flat.  Slot a holds A_a [d_in, rank[a]] row-major at
 *                   A_flat + a_off[a] and B_a [rank[a], d_out] row-major at
 *                   B_flat + b_off[a] (offsets in elements).
 *   a_off, b_off    [n_slots] int64, device; multiples of 8 (16-byte rows).
 *   rank            [n_slots] int32, device; each one of 8, 16, 32, 64, 128
 *                   and <= r_max.  An adapter of another rank is stored
 *                   zero-padded to the next of these (at most 2x its own
 *                   bytes, where padding to the largest rank costs up to 16x).
 *   a_elems, b_elems  the lengths of A_flat and B_flat in elements.
 *   r_max           one of 8, 16, 32, 64, 128: the largest rank allowed.
 * Each token costs its own adapter's rank: the kernel runs the body compiled
 * for that rank, so nothing of the larger ranks in the pool is read.  A slot entry
 * outside these rules (or one that would read past a pool's end) is not read:
 * LORA_DEVERR_BAD_RANK is set in the workspace error word and the token is
 * treated as base-only.  The results equal those of the zero-padded pool.
 *
 * lora_bgmv_adapter_ragged: the adapter term only, as lora_bgmv_adapter
 * (fp32 delta [T, d_out], base-only rows not written; T <= 65535; workspace:
 * the error word).  lora_linear_fused_ragged: the whole layer.
 *   - Up to 256 tokens: lora_linear_fused's bf16 decode path (the split-K
 *     base GEMM, then the merge kernel over the ragged pool, with the same
 *     programmatic overlap rules).
 *   - More tokens, with a workspace of lora_workspace_bytes(
 *     LORA_OP_LINEAR_FUSED_RAGGED, T, d_in, d_out, r_max, n_slots) bytes: the
 *     prefill route.  The adapters the batch uses are copied into the
 *     workspace as a dense pool at rank r_max (zero-padded), their tokens'
 *     ids remapped to it, and lora_linear_fused's prefill path runs over it
 *     (segments, SGMV shrink, the base GEMM with the expand in its
 *     accumulator): W0 is read once.  The result equals that of the
 *     zero-padded pool, as on the decode path.
 *   - More tokens with a workspace too small for that but of at least
 *     lora_workspace_bytes(LORA_OP_LINEAR_FUSED, 256, ...) bytes: the decode
 *     path over consecutive chunks of at most 256 tokens, which reads W0
 *     once per chunk.  (The prefill route's workspace can be the smaller of
 *     the two: the chunked route's holds the split-K partials.)
 *   LORA_OP_LINEAR_FUSED_RAGGED gives, for T <= 256, the decode path's
 *   workspace; for T > 256 the prefill route's (with n_c = min(T, n_slots):
 *   the prefill layout of lora_linear_fused for T tokens over n_c slots at
 *   rank r_max, plus n_c x (d_in + d_out) x r_max x 2 bytes of pool).
 * Both: bf16 only; LORA_ERR_INVALID_ARG for a null pointer, a pool, x or
 * output not 16-byte aligned, or a negative pool length.
 */
lora_status_t lora_bgmv_adapter_ragged(const void* x, const void* A_flat, const void* B_flat,
                                       const int64_t* a_off, const int64_t* b_off,
                                       const int32_t* rank, int64_t a_elems, int64_t b_elems,
                                       int32_t r_max, const int32_t* slot_ids,
                                       const float* scale, float* delta, int32_t T,
                                       int32_t d_in, int32_t d_out, int32_t n_slots,
                                       lora_dtype_t dt, void* ws, size_t ws_bytes, void* stream);
lora_status_t lora_linear_fused_ragged(const void* x, const void* W0, const void* A_flat,
                                       const void* B_flat, const int64_t* a_off,
                                       const int64_t* b_off, const int32_t* rank,
                                       int64_t a_elems, int64_t b_elems, int32_t r_max,
                                       const int32_t* slot_ids, const float* scale, void* y,
                                       int32_t T, int32_t d_in, int32_t d_out, int32_t n_slots,
                                       lora_dtype_t dt, void* ws, size_t ws_bytes, void* stream);

/*
 * 4-bit base matrix with bf16 adapters ("Serving Many LoRA Adapters", section
 * "When It Falls Down": QLoRA-style 4-bit base models served next to bf16
 * adapters, the base path passing through dequantisation).  Format (one
 * reading of "QLoRA style": a 16-entry codebook scaled by the absolute
 * maximum of each block of 64 weights):
 *   W0q     [d_out, d_in / 2] uint8, k contiguous per output column (the
 *           [out, in] orientation of a QLoRA weight): byte i of row n holds
 *           the codes of rows 2i (low nibble) and 2i + 1 (high nibble) of
 *           column n.
 *   absmax  [d_in / 64, d_out] bf16; the scale of rows [64b, 64b + 64) of a
 *           column.
 *   codebook [16] bf16; code c stands for codebook[c] (for NF4-like codes,
 *           values in [-1, 1]).
 *   deq(W0)[k, n] = bf16(codebook[code[k, n]] * absmax[k / 64, n]), the
 *           product rounded once to bf16.
 * Shapes: d_in a multiple of 64, d_out a multiple of 32; all pointers device
 * pointers, 16-byte aligned.
 *
 * lora_quantize_base_4bit: W0 [d_in, d_out] bf16 (finite) -> W0q, absmax:
 * absmax = max |W0| over each block; code = the codebook entry nearest
 * W0 / absmax (fp32 quotient and distances, ties to the lower code; an
 * all-zero block takes the entry nearest 0).  Done once per weight matrix.
 *
 * lora_base_gemm_4bit_splitk: partial [ksplit, T, d_out] fp32 with
 * partial[z] = x[:, K_z] deq(W0)[K_z, :] over ksplit contiguous ranges of
 * d_in, 1 <= ksplit <= min(d_in / 64, 64); the dequantisation runs in the
 * GEMM's mainloop on chip (into tensor memory, where the MMA reads it).
 * Workspace: the error word.
 *
 * lora_linear_fused_4bit: the whole layer, y = x deq(W0) + s (x A) B, for
 * bf16 batches.  Up to 256 tokens: the 4-bit split-K GEMM, then the merge
 * kernel of lora_linear_fused's decode path (bf16 adapters).  Larger
 * batches: W0 dequantised once into the workspace (the same bf16 values the
 * 4-bit GEMM feeds its MMAs), then lora_linear_fused's prefill path over it
 * (segments, SGMV shrink, the GEMM with the expand in its accumulator), so
 * the base is streamed once per call.  Same pools, ids, scale and
 * programmatic-overlap rules as lora_linear_fused (W0q, absmax and the
 * codebook play the part of W0 there); workspace:
 * lora_workspace_bytes(LORA_OP_LINEAR_FUSED_4BIT, T, d_in, d_out, r,
 * n_slots), which for T > 256 includes d_in x d_out x 2 bytes for the
 * dequantised W0.
 */
lora_status_t lora_quantize_base_4bit(const void* W0, const void* codebook, void* W0q,
                                      void* absmax, int32_t d_in, int32_t d_out, void* stream);
lora_status_t lora_base_gemm_4bit_splitk(const void* x, const void* W0q, const void* absmax,
                                         const void* codebook, float* partial, int32_t T,
                                         int32_t d_in, int32_t d_out, int32_t ksplit, void* ws,
                                         size_t ws_bytes, void* stream);
lora_status_t lora_linear_fused_4bit(const void* x, const void* W0q, const void* absmax,
                                     const void* codebook, const void* A_pool,
                                     const void* B_pool, const int32_t* slot_ids,
                                     const float* scale, void* y, int32_t T, int32_t d_in,
                                     int32_t d_out, int32_t r, int32_t n_slots, void* ws,
                                     size_t ws_bytes, void* stream);

/*
 * Uploads one adapter into pool slot `slot` (the data path of adapter
 * paging: "Multi-LoRA batching and adapter paging", section "Adapter
 * paging", and "Serving many LoRA adapters", section "Paging adapters": an
 * adapter moves from host memory into a slot of the resident pool while the
 * layer kernels keep running).  The adapter has rank r_a <= r; it is stored
 * zero-padded to the pool rank, which leaves every layer result unchanged:
 *   A_pool[slot][:, 0:r_a] = A_host [d_in, r_a]    A_pool[slot][:, r_a:r] = 0
 *   B_pool[slot][0:r_a, :] = B_host [r_a, d_out]   B_pool[slot][r_a:r, :] = 0
 *   scale[slot] = s                                 (skipped when scale is NULL)
 * A_host / B_host are host pointers, row-major and contiguous; pin them
 * (cudaHostAlloc) for the copies to be asynchronous and overlap kernels on
 * other streams.  Only enqueues work on `stream` (two copies, the zero
 * fills, and a one-thread kernel for the scale); the caller must not change
 * the host buffers until the stream has passed this call, and must not run
 * a layer that reads `slot` concurrently on another stream.  bf16 or fp32
 * pools (dt).  Errors: LORA_ERR_SHAPE for slot outside [0, n_slots), r_a
 * outside [1, r] or an invalid r / dims; LORA_ERR_INVALID_ARG for a null
 * pointer or a pool not 16-byte aligned.  No workspace.
 */
lora_status_t lora_slot_upload(void* A_pool, void* B_pool, float* scale, int32_t slot,
                               const void* A_host, const void* B_host, float s, int32_t d_in,
                               int32_t d_out, int32_t r, int32_t r_a, int32_t n_slots,
                               lora_dtype_t dt, void* stream);

/*
 * Synchronises `stream`, copies the workspace error word to *device_err and
 * clears it.  Returns LORA_ERR_CUDA if the stream reports an error.
 */
lora_status_t lora_get_error(void* ws, void* stream, int32_t* device_err);

/* Static, human-readable name of a status code. */
const char* lora_status_string(lora_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* LORA_H_ */
