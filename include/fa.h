/*
 * fa.h -- C ABI of libfa: exact, IO-aware tiled attention on one GB300
 * (sm_103a).
 *
 * The operation is scaled dot-product attention with an optional causal mask,
 *
 *     O = softmax(scale * Q K^T [+ mask]) V,
 *
 * as defined on "FlashAttention and the Kernel Era", section "The
 * Mathematics" (first equation), and on "FlashAttention 1, 2, and 3
 * Explained", section 1 (the S, P, O equations).  The forward pass computes it
 * block by block with the online-softmax rescaling of that page's section 2
 * and of "The Mathematics" (running max m and running sum l), so the N x N
 * score matrix never reaches HBM; only O and one float per query row (the
 * log-sum-exp) are written.  The backward pass recomputes S and P from Q, K, V
 * and that saved row statistic ("FlashAttention Kernel", the recomputation
 * bullets; "FlashAttention", the recomputation paragraph).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Layout is [B, N, H, d], row-major, contiguous (the flash_attn_func layout
 *    on the "Flash Attention" page, section "Code Example"): element
 *    (b, n, h, c) is at ((b*N + n)*H + h)*d + c.  Query-side tensors (q, o,
 *    dout, dq) have H = Hq heads; key/value-side tensors (k, v, dk, dv) have
 *    H = Hkv heads.  Tensors of the same call share B, N and d (Nq == Nk == N).
 *  - Element type: bf16 (IEEE bfloat16) for q, k, v, o, dout, dq, dk, dv;
 *    fp32 for lse and the backward workspace.  Outputs are rounded to nearest
 *    even from fp32 accumulators.
 *  - lse is [B, Hq, N] fp32: lse[b,h,i] = ln sum_j exp(scale * q_i . k_j) over
 *    the keys j visible to query i (natural log of the *scaled* scores).
 *  - GQA / MQA ("FlashAttention", the KV-cache bullets; "Flash Attention",
 *    "Key Technical Innovations"): query head h reads key/value head
 *    h / (Hq / Hkv); Hq must be a multiple of Hkv.  Hkv == Hq is plain
 *    multi-head attention, Hkv == 1 is multi-query attention.
 *  - causal != 0 masks key j from query i when j > i.  Since Nq == Nk the
 *    top-left and bottom-right alignments coincide.
 *  - d must be 64 or 128.  N >= 1 with no other restriction (ragged tails are
 *    masked).  B, Hq, Hkv >= 1.
 *  - All pointers are DEVICE pointers on the current CUDA device, 16-byte
 *    aligned (workspaces: 256-byte aligned).  The caller owns every buffer;
 *    the library allocates no device memory in these calls and keeps no
 *    pointer after a call returns.  The library itself holds, on every device
 *    where it is loaded, two static device arrays: a 4-byte status word (the
 *    watchdog's) and the 2^21-float (8 MiB) scratch of fa_bwd_noalloc.
 *  - Operand precision.  Every product is accumulated in fp32.  The scores
 *    S = Q K^T (forward) use the bf16 inputs as given.  Where a rounded
 *    intermediate feeds a product -- P in O += P V, and P, dS in the
 *    backward's dV, dK, dQ products -- the training forward and fa_bwd round
 *    it to fp16 and multiply it with an fp16 copy of the other operand (the
 *    bf16 inputs scaled by a power of two chosen from the tensor's largest
 *    magnitude, which makes the copy exact for every element above 2^-19 of
 *    that maximum, for maxima in [2^-25, 2^36]; the scaling is undone
 *    exactly).  fp16 keeps 3 more bits than bf16, which the peaked-row
 *    near-cancellation dS = P o (dP - D) needs.  fa_fwd (inference) and
 *    fa_bwd_noalloc round those intermediates to bf16 instead.
 *  - stream is a cudaStream_t (CUstream) handle, or NULL for the legacy
 *    default stream.  Calls enqueue work on it and return without waiting.
 *  - Errors: argument errors are detected on the host before any launch and
 *    return FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED with nothing enqueued.  A
 *    launch failure returns FA_ERR_CUDA (see fa_last_cuda_error).  Every wait
 *    inside the kernels is bounded; a wait that runs out records
 *    FA_ERR_DEVICE_TIMEOUT in a library-owned device status word, every
 *    other pending wait of the same launch then gives up too, the kernel
 *    returns (its outputs incomplete), and fa_get_device_error reports it.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,     /* null/misaligned pointer, bad size, Hq % Hkv != 0 */
    FA_ERR_UNSUPPORTED = 2,     /* d not in {64, 128}, or no sm_103 device */
    FA_ERR_CUDA = 3,            /* a CUDA runtime/driver call failed */
    FA_ERR_DEVICE_TIMEOUT = 4   /* a bounded in-kernel wait ran out */
} fa_status;

/*
 * Forward pass.
 *   q   [B, N, Hq, d]  bf16 in
 *   k   [B, N, Hkv, d] bf16 in
 *   v   [B, N, Hkv, d] bf16 in
 *   o   [B, N, Hq, d]  bf16 out: softmax(scale*QK^T [+mask]) V
 *   lse [B, Hq, N]     fp32 out: per-row log-sum-exp of the scaled scores
 *   H is the number of query heads (Hq).  scale is usually 1/sqrt(d).
 * Tiled with online softmax as on "FlashAttention 1, 2, and 3 Explained",
 * section 2 (the l and O update equations), parallel over (batch, head,
 * query block) as on "FlashAttention Kernel" (the FlashAttention-2 bullets).
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int Hkv, int N, int d, int causal, float scale,
                 void* stream);

/*
 * Forward pass for training: fa_fwd plus the low half of O, with P rounded
 * to fp16 for the P V product.
 *   o_lo [B, N, Hq, d] bf16 out (or NULL): bf16(O32 - O), where O32 is the
 *        fp32 output before rounding and O the bf16 value written to `o`.
 *        o + o_lo carries O to about 16 significant bits.
 *   workspace: the training workspace, fa_bwd_workspace_size(B, H, Hkv, N, d)
 *        bytes, 256-byte aligned, caller-owned, contents irrelevant on entry;
 *        NULL rounds P to bf16 as fa_fwd does.  The call leaves the fp16
 *        copies of q, k, v (and their maxima) in it, so that a backward on
 *        the same workspace and the same q, k, v skips them (fa_bwd_stage
 *        with FA_BWD_PREP_DOUT instead of FA_BWD_PREP).
 * fa_bwd forms D_i = sum_c dO_ic O_ic from o + o_lo when given it.  Both
 * matter when rows are peaked: there dS = P o (dP - D) is a near-cancellation
 * and the roundings of P and of O alone move dQ by more than the rounding of
 * the gradients themselves.  Other arguments and errors as fa_fwd.
 */
fa_status fa_fwd_train(const void* q, const void* k, const void* v, void* o, void* o_lo,
                       float* lse, void* workspace, int B, int H, int Hkv, int N, int d,
                       int causal, float scale, void* stream);

/*
 * Bytes of the training workspace (fa_fwd_train, fa_bwd): one fp32 per query row and head
 * (D_i = sum_c dO_ic * O_ic, 4 * B * H * N bytes), the fp16 copies of q, k,
 * v, dout (2 * B * N * (2 * H + 2 * Hkv) * d bytes) and 512 bytes of scale
 * data, each part rounded up to 256.  Returns 0 for invalid sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int Hkv, int N, int d);

/*
 * Backward pass of the loss L with dL/dO = dout.
 *   q, k, v, o, lse  as produced/consumed by fa_fwd (same B, H, Hkv, N, d,
 *                    causal and scale)
 *   o_lo             the o_lo written by fa_fwd_train, or NULL (then D is
 *                    formed from the bf16 o alone)
 *   dout [B, N, Hq, d]  bf16 in
 *   dq   [B, N, Hq, d]  bf16 out
 *   dk   [B, N, Hkv, d] bf16 out (summed over the Hq/Hkv query heads of a group)
 *   dv   [B, N, Hkv, d] bf16 out (same)
 *   workspace: device buffer of at least fa_bwd_workspace_size(B, H, Hkv,
 *              N, d) bytes, 256-byte aligned, owned by the caller; its
 *              contents on entry do not matter and are overwritten.
 * S and P are recomputed from q, k and lse ("FlashAttention Kernel",
 * recomputation bullets).  Every output element is written by exactly one
 * thread block; no atomics, so results are deterministic.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, void* workspace,
                 const void* o_lo, int B, int H, int Hkv, int N, int d, int causal,
                 float scale, void* stream);

/*
 * The steps of fa_bwd, callable one at a time (e.g. to time them).  `stages`
 * is a bitmask of FA_BWD_PREP (max |x| of q, k, v, dout and the fp16 copies
 * of q, k, v into the workspace), FA_BWD_PREP_DOUT (max |dout| only: the
 * workspace must hold fa_fwd_train's copies of the same q, k, v),
 * FA_BWD_DSUM (D = rowsum(dout * o) into the workspace; in a call with
 * FA_BWD_PREP or FA_BWD_PREP_DOUT it also takes max |dout|, which the prep
 * kernels then skip), FA_BWD_DQ (dq; it also writes the fp16 copy of dout and
 * the scales into the workspace) and FA_BWD_DKDV (dk, dv; it reads that copy);
 * set stages run in the order PREP(_DOUT), DSUM, DQ, DKDV.  Each stage reads
 * what the earlier stages wrote into the same workspace earlier on the stream,
 * so DKDV must follow a DQ of the same inputs.  fa_bwd(...) is
 * fa_bwd_stage(FA_BWD_PREP | FA_BWD_DSUM | FA_BWD_DKDV | FA_BWD_DQ, ...); a
 * training step that ran fa_fwd_train on the workspace can use
 * FA_BWD_PREP_DOUT | FA_BWD_DSUM | FA_BWD_DKDV | FA_BWD_DQ.
 * Arguments, ownership and errors are those of fa_bwd; pointers a stage does
 * not read or write must still be valid (they are checked, not dereferenced).
 */
enum { FA_BWD_DSUM = 1, FA_BWD_DKDV = 2, FA_BWD_DQ = 4, FA_BWD_PREP = 8, FA_BWD_PREP_DOUT = 16 };
fa_status fa_bwd_stage(int stages, const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv,
                       void* workspace, const void* o_lo, int B, int H, int Hkv, int N, int d,
                       int causal, float scale, void* stream);

/*
 * fa_bwd without a workspace argument, for callers that cannot allocate
 * device memory: a plug-in inside a host application that owns every device
 * allocation, or a loop that must not call cudaMalloc mid-step.  (The pages
 * have no counterpart; this is a library convenience.)
 *   Arguments, outputs and errors are those of fa_bwd minus `workspace`,
 *   except that P and dS are rounded to bf16, not fp16, before their
 *   products (there is no room for fp16 operand copies).
 *   Accuracy: on unpeaked inputs (N(0, 1)-like rows) the outputs meet the
 *   same bounds as fa_bwd (max-abs 2e-2 beyond bf16 output rounding, rel-L2
 *   5e-3).  On peaked rows -- a few keys far larger than the rest, where
 *   dS = P o (dP - D) nearly cancels and |K| is large -- the bf16 rounding of
 *   dS shows in dQ = dS K: rel-L2 stays within 5e-3 but max-abs can exceed
 *   2e-2 (measured 0.076 for dQ with 1% of the keys scaled by 8; the
 *   library test allows 0.15).  Use fa_bwd where that matters.
 *   D lives in a fixed array built into the library: 2^21 fp32 rows (8 MiB),
 *   held on every GPU that loads the library until the process exits.  Calls
 *   with B * H * N > 2^21 return FA_ERR_INVALID_ARG (with a message on
 *   stderr) and enqueue nothing.
 *   The first call on a device looks up the array's device address on that
 *   device (current device, no allocation); make that first call before any
 *   stream capture.
 *   All calls share the one array, and it keeps the last call's contents:
 *   calls whose work overlaps on the GPU (other streams, other threads) race
 *   on it and must be serialised by the caller.  Nothing in it needs to start
 *   at zero.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const void* dout, const float* lse, void* dq, void* dk, void* dv,
                         const void* o_lo, int B, int H, int Hkv, int N, int d, int causal,
                         float scale, void* stream);

/*
 * Split-KV forward (FlashDecoding): Nq queries against Nk keys and values,
 * the key range cut into splits that run as separate thread blocks, then an
 * exact merge of the splits' results ("FlashAttention Kernel", the
 * FlashDecoding mentions: parallel over the key/value length, then combined;
 * the merge is the two-block online-softmax update of "FlashAttention 1, 2,
 * and 3 Explained", section 2).  For decoding: the queries are the last Nq
 * positions of a sequence of Nk.
 *   q    [B, Nq, H, d]   bf16 in
 *   k, v [B, Nk, Hkv, d] bf16 in
 *   o    [B, Nq, H, d]   bf16 out
 *   lse  [B, H, Nq]      fp32 out, natural log of the scaled scores' sum
 *   causal: query i sees keys j <= i + Nk - Nq (needs Nq <= Nk; with
 *        Nq == Nk this is fa_fwd's mask)
 *   num_splits: number of key ranges, <= 0 for the library's choice (enough
 *        thread blocks for two per SM); clamped to the number of 128-key
 *        blocks, and reduced so that no range is empty.
 *   workspace: fa_fwd_splitkv_workspace_size(...) bytes (fp32 per-split
 *        results), 256-byte aligned, caller-owned; may be NULL when that size
 *        is 0 (one split: the kernel writes o and lse itself).
 * The g = H / Hkv query heads of a key/value head are processed together
 * (128 / g queries of all g heads per 128-row tile), so K and V are read from
 * HBM once.  d in {64, 128}; g <= 128.  Errors as fa_fwd; FA_ERR_INVALID_ARG
 * also for causal with Nq > Nk and for a missing workspace.
 */
fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                         void* workspace, int B, int H, int Hkv, int Nq, int Nk, int d,
                         int causal, float scale, int num_splits, void* stream);

/* The split count fa_fwd_splitkv uses for these arguments (0: invalid sizes). */
int fa_fwd_splitkv_num_splits(int B, int H, int Hkv, int Nq, int Nk, int d, int causal,
                              int num_splits);

/* Workspace bytes fa_fwd_splitkv needs for these arguments: 0 when it uses one
 * split (or the sizes are invalid), else (splits * B * H * Nq) * (d + 1) fp32
 * values, each part rounded up to 256 bytes. */
size_t fa_fwd_splitkv_workspace_size(int B, int H, int Hkv, int Nq, int Nk, int d, int causal,
                                     int num_splits);

/*
 * Block-sparse forward: fa_fwd computed only over the 128 x 128 blocks a
 * block mask selects ("FlashAttention Kernel": block-sparse FlashAttention
 * skips the blocks a sparsity mask zeroes).
 *   q, k, v, o, lse, B, H, Hkv, N, d, causal, scale: as fa_fwd
 *   block_mask: device bytes [H, nb, nb] with nb = ceil(N / 128); query i of
 *        head h may see key j only when block_mask[h][i / 128][j / 128] != 0
 *        (and, with causal, j <= i).  Read only.
 * A query row with no visible key gets o = 0 and lse = -inf.  Each thread
 * block takes two 128-query tiles of one head (the pipeline of fa_fwd), reads
 * their two mask rows once into shared memory, and each tile streams the K
 * and V blocks of its own row.  Errors as fa_fwd; FA_ERR_INVALID_ARG also for
 * a null block_mask; FA_ERR_UNSUPPORTED for N > 917,504 (mask rows longer
 * than 7,168 blocks).
 */
fa_status fa_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse,
                             const uint8_t* block_mask, int B, int H, int Hkv, int N, int d,
                             int causal, float scale, void* stream);

/*
 * FP8 (e4m3) forward, head dimension 128: fa_fwd with Q, K, V and P entering
 * the products as e4m3 values behind block quantisation ("FlashAttention and
 * the Kernel Era", the FP8 paragraph; "FlashAttention 1, 2, and 3 Explained",
 * section 4: FP8 with block quantisation and incoherent processing).
 *   q, k, v, o, lse, B, H, Hkv, N, causal, scale: as fa_fwd (bf16 in and out);
 *        d must be 128 (FA_ERR_UNSUPPORTED otherwise)
 *   workspace: fa_fwd_fp8_workspace_size(...) bytes, 256-byte aligned,
 *        caller-owned: the e4m3 copies (q and k with one scale per
 *        128-row block of each head, v transposed with one scale per head)
 *   flags: FA_FP8_ROTATE -- multiply the rows of q and k by a fixed
 *        random-sign Walsh-Hadamard matrix before quantising them (Q K^T is
 *        unchanged; outliers are spread over the row); FA_FP8_QUANTIZE_ONLY
 *        -- make the e4m3 copies and stop; FA_FP8_ATTEND_ONLY -- skip the
 *        copies and use those an earlier call with the same q, k, v and
 *        FA_FP8_ROTATE setting left in the workspace (e.g. a cache quantised
 *        once); not both
 * Accuracy: e4m3 keeps 4 significant bits, so O carries relative errors of a
 * few percent per element where bf16 carries a fraction of one.  The library
 * tests hold O to rel-L2 6e-2 and lse to 0.15 of the exact result on N(0, 1)
 * inputs with scale 1/sqrt(128), and to 5e-2 / 5e-2 on 0.5 N(0, 1) inputs.
 * Errors as fa_fwd.
 */
enum { FA_FP8_ROTATE = 1, FA_FP8_QUANTIZE_ONLY = 2, FA_FP8_ATTEND_ONLY = 4 };
fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                     void* workspace, int B, int H, int Hkv, int N, int d, int causal,
                     float scale, int flags, void* stream);

/* Bytes of the FP8 forward's workspace (0 for invalid sizes or d != 128). */
size_t fa_fwd_fp8_workspace_size(int B, int H, int Hkv, int N, int d);

/*
 * Synchronises `stream`, then reads and clears the device status word of the
 * current device.  Returns FA_OK, FA_ERR_DEVICE_TIMEOUT (a bounded wait ran
 * out in some kernel since the last call) or FA_ERR_CUDA (the synchronise
 * failed).
 */
fa_status fa_get_device_error(void* stream);

/* Static, human-readable name of a status code. */
const char* fa_status_string(fa_status s);

/* Text of the last CUDA error seen by this thread inside the library
 * (empty string if none).  Valid until the thread's next library call. */
const char* fa_last_cuda_error(void);

/*
 * Test hook for the watchdog: launches `num_blocks` thread blocks (clamped to
 * [1, 2^20]) whose first thread waits on a shared-memory barrier that nothing
 * ever signals, with the same bounded wait the attention kernels use, but a
 * limit of `timeout_ns` nanoseconds (clamped to [1e3, 5e9]).  The first wait
 * to run out records FA_ERR_DEVICE_TIMEOUT; every other block's wait then
 * gives up within microseconds (a failure ends the whole launch), so the
 * launch takes about one limit however many waves of blocks it has.  The GPU
 * stays usable.  Enqueued on `stream`; read the result with
 * fa_get_device_error.
 */
fa_status fa_debug_watchdog_probe(uint64_t timeout_ns, int num_blocks, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
