/*
 * gqa_attn.h -- C ABI of the fused attention-forward library for GB300 (sm_103a).
 *
 * Two regimes share one library:
 *   prefill: q_len = kv_len = S, optional causal mask, O = softmax(Q K^T * scale) V per head,
 *            computed as one fused kernel that never writes the score or probability matrix
 *            to device memory;
 *   decode:  one query token per sequence against a KV cache; the keys are split into chunks
 *            processed by separate thread blocks, and a second kernel merges the chunk results
 *            with their log-sum-exp weights.
 *
 * The operation (per batch b, query head h, query row i):
 *   g = h / (Hq / Hkv)                                      kv head of h (contiguous groups)
 *   s_j = scale * sum_d q[b,h,i,d] k[b,g,j,d]               scores
 *   visible keys: j < kv_len, and j <= i when causal        masked scores are -infinity
 *   O[b,h,i,:] = sum_j softmax(s)_j v[b,g,j,:]              row softmax, then P V
 *   LSE[b,h,i] = log sum_j exp(s_j)                         natural log, of the scaled scores
 * Sources: "Attention three-op fusion" (xdnf.cn/news/349386) section 1.1 (the S, P, O chain),
 * section 2.2-2.3 (online softmax with running max and sum, output correction, divide once at
 * the end), section 4.3 (causal and padding masks as -infinity) and section 4.4 (keys split
 * across thread blocks, partial results merged); "Hand-written Triton decoder"
 * (m.nlpx.cn/news/28229) section 2.1 (2 KV heads broadcast to 8 query heads, head dim 128)
 * and section 3.3 (partials in a separate buffer reduced by a second small kernel);
 * "triton-optimization" skill (skillsmp.com) section 3.5 (log-sum-exp = m + log of the sum).
 *
 * Conventions for every entry point:
 *   - All tensors are device pointers, row-major with the head dimension D innermost and
 *     contiguous; the caller owns them. The library never frees caller memory.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls are asynchronous on
 *     that stream; nothing is allocated and nothing synchronizes on the hot path, except the
 *     documented first-use growth of the library-owned decode workspace.
 *   - Arguments are checked on the host before anything is launched. A bad argument returns
 *     an error code and launches nothing. A launch failure returns ATTN_ERR_CUDA.
 *   - Conditions only the device can see (a sequence length above max_len, a pipeline wait
 *     that ran out) set bits of a per-device status word; read it with attn_device_status.
 *   - Results are deterministic for fixed inputs and shapes (no floating-point atomics).
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID = 1,     /* NULL pointer, non-positive size, Hq % Hkv != 0, bad dtype   */
    ATTN_ERR_UNSUPPORTED = 2, /* valid but not built: head dim or dtype combination          */
    ATTN_ERR_ALIGN = 3,       /* a tensor pointer is not 16-byte aligned                     */
    ATTN_ERR_WORKSPACE = 4,   /* workspace too small (or cannot grow while capturing)        */
    ATTN_ERR_CUDA = 5,        /* a CUDA runtime or driver call failed                        */
    ATTN_ERR_TIMEOUT = 6      /* reported through attn_device_status: a device wait expired  */
} attn_status;

/* Element types. */
typedef enum { ATTN_F32 = 0, ATTN_BF16 = 1 } attn_dtype;

/* Bits of the device status word (attn_device_status). */
#define ATTN_DEV_SEQLEN_CLAMPED 0x1u /* decode: a seqlens[b] was < 0 or > max_len; clamped   */
#define ATTN_DEV_WAIT_TIMEOUT 0x2u   /* a pipeline wait ran out; the block stopped          */
#define ATTN_DEV_INDEX_CHECK 0x4u    /* debug build only: an index check in a kernel failed
                                        and the access it guards was skipped               */

/*
 * attn_prefill -- causal or non-causal prefill, bf16 in, bf16 out.
 *   q   [B, Hq,  S, D] bf16        k, v [B, Hkv, S, D] bf16
 *   o   [B, Hq,  S, D] bf16        lse  [B, Hq, S] fp32, natural log; may be NULL
 *   scale multiplies the scores before the softmax (usually 1/sqrt(D)).
 *   causal != 0: query i sees keys 0..i.
 * Requires Hq % Hkv == 0, D in {64, 128}, 16-byte aligned pointers.
 * When the shape has fewer (256-row block, head) tiles than the GPU has SMs, the key range of
 * each row block is split over several thread blocks and a second kernel merges their results
 * by log-sum-exp weights.
 * Computes on tcgen05 tensor cores with fp32 accumulation and fp32 softmax state: Q K^T from
 * the bf16 inputs; P V with P rounded to fp16 and V converted bf16 -> fp16. Each (batch, kv
 * head) slab of V is scaled by a power of two 2^-e picked from its largest finite |v| (e = 0
 * unless that maximum is below 2^-9 or at least 2^16), and O is multiplied back by 2^e, so
 * every finite bf16 V gives the same result as unscaled arithmetic would. V must be finite:
 * an inf or NaN in V reaches rows whose probability for that key is 0 as NaN.
 * The conversion normally writes an fp16 copy of V (B*Hkv*S*D*2 bytes) once per call, which
 * the attention kernel then streams.
 * Scratch: a small V scale area (per slab: one int, plus one word per conversion block), the
 * split's partial results and the fp16 copy of V use the library-owned scratch buffer of the
 * device (grown with cudaMalloc on first use, outside stream capture; the buffer is shared with
 * the decode calls, so calls on different streams must be serialised, or use attn_prefill_ws).
 * A call that cannot have all of it (stream capture before the buffer has grown that far; a
 * copy above 1 GiB) runs unsplit and converts V on chip instead, with the same results. During
 * stream capture a buffer too small even for the V scale area (no earlier call of any kind on
 * the device) returns ATTN_ERR_WORKSPACE: reserve attn_prefill_workspace_bytes(...) with
 * attn_reserve_workspace_bytes, or make one call, before capturing.
 */
int attn_prefill(const void *q, const void *k, const void *v, void *o, float *lse, int B, int S,
                 int Hq, int Hkv, int D, float scale, int causal, void *stream);

/*
 * attn_prefill_ex -- prefill with explicit element types.
 *   in_dtype  ATTN_BF16: q, k, v bf16; D in {64, 128}; tensor-core kernel (as attn_prefill).
 *             ATTN_F32:  q, k, v fp32; D in {64, 128}; fp32 CUDA-core kernel (fp32 products,
 *                        sums and exponentials throughout).
 *   out_dtype ATTN_BF16 or ATTN_F32 for o (ATTN_F32 with bf16 inputs returns the fp32 result
 *             before the final rounding). fp32 inputs require out_dtype ATTN_F32.
 * Other arguments as attn_prefill.
 */
int attn_prefill_ex(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                    int S, int Hq, int Hkv, int D, float scale, int causal, int in_dtype,
                    int out_dtype, void *stream);

/*
 * attn_prefill_workspace_bytes -- bytes of scratch a bf16 prefill call of this shape uses on the
 * current device (the key split depends on its SM count): the V scale area, the split's partial
 * results when the shape is split, and the fp16 copy of V when it is at most 1 GiB. 0 for
 * invalid arguments (including D not in {64, 128}).
 */
size_t attn_prefill_workspace_bytes(int B, int S, int Hq, int Hkv, int D, int causal);

/*
 * attn_prefill_ws -- attn_prefill_ex for bf16 inputs with a caller-owned workspace, so calls on
 * different streams (each with its own workspace) may overlap. workspace: device memory,
 * 256-byte aligned (else ATTN_ERR_ALIGN), of workspace_bytes bytes; NULL = the library-owned
 * buffer, as attn_prefill. The call uses the first arrangement that fits: split + fp16 copy of
 * V, the copy alone, or neither (V converted on chip), all with the same results; with less than
 * the V scale area it returns ATTN_ERR_WORKSPACE and launches nothing. Nothing in the workspace
 * needs initialising, and the call never allocates. Calls sharing one workspace must not
 * overlap on the GPU.
 *   out_dtype ATTN_BF16 or ATTN_F32. Other arguments, layouts and numerics as attn_prefill.
 * Source: "Hand-written Triton decoder" (m.nlpx.cn/news/28229) section 3.3 (a split's partial
 * results go to a buffer that is allocated once and reused, never allocated per call).
 */
int attn_prefill_ws(const void *q, const void *k, const void *v, void *o, float *lse, int B, int S,
                    int Hq, int Hkv, int D, float scale, int causal, int out_dtype,
                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * attn_prefill_strided -- attn_prefill for bf16 operands in any layout whose head dim is
 * contiguous: each of q, k, v, o is described by its base pointer and three element strides
 * {batch, token, head}. Element (b, h, i, d) of q is q[b*qs[0] + i*qs[1] + h*qs[2] + d]; k, v and
 * o likewise with their own strides. Examples: [B, H, S, D] contiguous is {H*S*D, D, S*D};
 * [B, S, H, D] contiguous is {S*H*D, H*D, D}; the output of a fused QKV projection
 * [B, S, Hq + 2*Hkv, D] gives q = base, k = base + Hq*D, v = base + (Hq + Hkv)*D, all with the
 * strides {S*(Hq+2*Hkv)*D, (Hq+2*Hkv)*D, D}. The operands are read in place (no copy).
 *   q_strides, k_strides, v_strides, o_strides: host arrays of 3 int64, each > 0 and a multiple
 *   of 16 bytes (8 bf16 elements; 4 for an fp32 o), else ATTN_ERR_ALIGN; NULL: ATTN_ERR_INVALID.
 *   o bf16 or fp32 by out_dtype; lse [B, Hq, S] fp32 contiguous, or NULL.
 * Other arguments, requirements and numerics as attn_prefill (D in {64, 128}). Overlapping o
 * elements (strides that alias) are the caller's error.
 * Sources: "Attention three-op fusion" (xdnf.cn/news/349386) section 6.1, second item (after the
 * projection weights are merged Q, K and V sit in one contiguous buffer; the kernel's address
 * arithmetic follows that layout instead of three separate tensors); "Hand-written Triton
 * decoder" (m.nlpx.cn/news/28229) section 2.2, operations 2, 3 and 9 (one projection writes
 * q, k and v side by side; splitting q into heads and merging the heads' outputs back into the
 * hidden layout are stride changes, not kernels).
 */
int attn_prefill_strided(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                         int S, int Hq, int Hkv, int D, const long long *q_strides,
                         const long long *k_strides, const long long *v_strides,
                         const long long *o_strides, float scale, int causal, int out_dtype,
                         void *stream);

/*
 * attn_chunk -- a chunk of Sq new query tokens per sequence against a bf16 KV cache (chunked
 * prefill, verification of speculative tokens). The chunk is the last Sq tokens of each
 * sequence and is already in the cache, so query i of sequence b sits at position
 * p = seqlens[b] - Sq + i; it sees cache rows j < seqlens[b], and with causal != 0 only j <= p.
 * A query with p < 0 sees nothing: o = 0, lse = -inf.
 *   q        [B, Hq, Sq, D] bf16
 *   kcache   [B, Hkv, max_len, D] bf16, vcache likewise; rows >= seqlens[b] are masked (their
 *            contents never reach the result, NaN included)
 *   seqlens  [B] int32, device memory; values outside [0, max_len] are clamped and flagged
 *            (ATTN_DEV_SEQLEN_CLAMPED)
 *   o        [B, Hq, Sq, D], bf16 or fp32 by out_dtype; lse [B, Hq, Sq] fp32 or NULL
 * Requires Hq % Hkv == 0, D in {64, 128}. Same tensor-core kernel as attn_prefill (with
 * seqlens[b] = Sq = S, max_len = S it computes exactly attn_prefill's result), including the
 * fp16 copy of V in the library-owned scratch (B*Hkv*max_len*D*2 bytes; only the key tiles
 * below each seqlens[b] are written) and the same fallback when the scratch is unavailable.
 * Sources: "Hand-written Triton decoder" (m.nlpx.cn/news/28229) section 1.4 (speculative
 * decoding and beam search reuse the attention kernels with several new tokens);
 * "Attention three-op fusion" (xdnf.cn/news/349386) section 4.3 (causal and padding masks).
 */
int attn_chunk(const void *q, const void *kcache, const void *vcache, const int *seqlens,
               void *o, float *lse, int B, int Sq, int Hq, int Hkv, int D, int max_len,
               float scale, int causal, int out_dtype, void *stream);

/*
 * attn_chunk_strided -- attn_chunk for operands in any layout whose head dim is contiguous,
 * described as for attn_prefill_strided by three int64 element strides {batch, token, head}
 * per operand: q and o over Sq tokens, the caches over max_len rows. Element (b, g, r, d) of
 * kcache is kcache[b*k_strides[0] + r*k_strides[1] + g*k_strides[2] + d]; e.g. caches stored
 * [B, max_len, Hkv, D] have strides {max_len*Hkv*D, Hkv*D, D}. NULL stride arrays return
 * ATTN_ERR_INVALID; strides that are not positive multiples of 16 bytes, ATTN_ERR_ALIGN. The
 * fp16 copy of V it makes (as attn_chunk) is contiguous. Other arguments as attn_chunk.
 */
int attn_chunk_strided(const void *q, const void *kcache, const void *vcache, const int *seqlens,
                       void *o, float *lse, int B, int Sq, int Hq, int Hkv, int D, int max_len,
                       const long long *q_strides, const long long *k_strides,
                       const long long *v_strides, const long long *o_strides, float scale,
                       int causal, int out_dtype, void *stream);

/*
 * attn_prefill_varlen -- batched prefill of sequences of different lengths, padded to S tokens.
 * Sequence b holds seqlens[b] valid tokens at positions 0 .. seqlens[b]-1 of q, k, v; keys at
 * or past seqlens[b] are masked (their contents never reach the result); padding rows
 * (i >= seqlens[b]) get o = 0 and lse = -inf.
 *   q [B, Hq, S, D] bf16, k/v [B, Hkv, S, D] bf16, seqlens [B] int32 (device, clamped to
 *   [0, S] and flagged with ATTN_DEV_SEQLEN_CLAMPED), o [B, Hq, S, D] bf16 or fp32 by
 *   out_dtype, lse [B, Hq, S] fp32 or NULL. Requires Hq % Hkv == 0, D in {64, 128}.
 * Source: "Attention three-op fusion" (xdnf.cn/news/349386) section 4.3 (padding mask: positions
 * at or past the sequence length get score -infinity) and section 6.1 (dynamic shapes).
 */
int attn_prefill_varlen(const void *q, const void *k, const void *v, const int *seqlens, void *o,
                        float *lse, int B, int S, int Hq, int Hkv, int D, float scale, int causal,
                        int out_dtype, void *stream);

/*
 * attn_prefill_varlen_strided -- attn_prefill_varlen for operands in any layout whose head dim
 * is contiguous ({batch, token, head} element strides per operand, as attn_prefill_strided;
 * e.g. q, k, v as head slices of a padded fused QKV projection output [B, S, Hq+2*Hkv, D], o
 * written into a [B, S, Hq, D] buffer). NULL stride arrays return ATTN_ERR_INVALID; strides
 * that are not positive multiples of 16 bytes, ATTN_ERR_ALIGN. Other arguments as
 * attn_prefill_varlen.
 */
int attn_prefill_varlen_strided(const void *q, const void *k, const void *v, const int *seqlens,
                                void *o, float *lse, int B, int S, int Hq, int Hkv, int D,
                                const long long *q_strides, const long long *k_strides,
                                const long long *v_strides, const long long *o_strides,
                                float scale, int causal, int out_dtype, void *stream);

/*
 * attn_decode -- one query token per sequence against a bf16 KV cache.
 *   q        [B, Hq, D] bf16
 *   kcache   [B, Hkv, max_len, D] bf16, vcache likewise; rows >= seqlens[b] are never read
 *   seqlens  [B] int32, device memory: valid cache rows of sequence b (including the newest
 *            token, already written); 0 gives o = 0 (and lse = -inf)
 *   o        [B, Hq, D] bf16
 * Requires Hq % Hkv == 0, D in {64, 128}, max_len >= 1.
 * Scratch for the per-chunk partial results comes from a library-owned buffer per device.
 * The first call for a larger shape grows it: cudaMalloc of a new buffer at least twice as
 * large; the old one stays allocated until the process exits, so CUDA graphs captured with it
 * remain valid. During stream capture it cannot grow and the call returns ATTN_ERR_WORKSPACE
 * instead, so reserve it first with attn_reserve_workspace. Calls on different streams of one
 * device share that buffer: serialise them, or use attn_decode_ex with your own workspace.
 */
int attn_decode(const void *q, const void *kcache, const void *vcache, const int *seqlens,
                void *o, int B, int Hq, int Hkv, int D, int max_len, float scale, void *stream);

/*
 * attn_decode_ex -- decode with an optional fp32 LSE output [B, Hq] (lse may be NULL), a
 * caller-owned device workspace of at least attn_decode_workspace_bytes(...) bytes (16-byte
 * aligned; NULL = the library-owned buffer, as attn_decode), and out_dtype ATTN_BF16 or
 * ATTN_F32 for o. A workspace that is too small returns ATTN_ERR_WORKSPACE.
 */
int attn_decode_ex(const void *q, const void *kcache, const void *vcache, const int *seqlens,
                   void *o, float *lse, int B, int Hq, int Hkv, int D, int max_len, float scale,
                   void *workspace, size_t workspace_bytes, int out_dtype, void *stream);

/*
 * attn_decode_noalloc -- attn_decode_ex for callers that cannot allocate device memory.
 * The pages describe no such variant; it exists for code that runs where cudaMalloc is not
 * available to it: under a memory manager that owns the whole device, in a process whose
 * allocator is frozen after start-up, or in a plug-in that is handed tensors but no allocator.
 * It allocates nothing and takes no workspace: the per-chunk partial results go to a fixed
 * device array of ATTN_DECODE_NOALLOC_SCRATCH_BYTES bytes inside the library, which every GPU
 * that loads the library keeps until the process exits.
 *   Arguments as attn_decode_ex, without workspace/workspace_bytes.
 *   Batches up to 1024: the key list is split over as many warps as the array has room for
 *   (up to the full grid), so any shape with B * Hq up to about 8000 at D = 128 (about 15800 at
 *   D = 64) runs; a grid smaller than the full one only lowers parallelism. Larger batches (the
 *   chunked kernel): the shape's partials, attn_decode_workspace_bytes(...), must fit in the
 *   array.
 *   Otherwise it returns ATTN_ERR_WORKSPACE and launches nothing.
 *   The first call on each device looks up the array's device address (with that device
 *   current); make that first call before any stream capture.
 *   All calls on a device share the one array and it keeps the last call's contents: calls
 *   that overlap on the GPU (different streams, no ordering between them) race and give wrong
 *   results. Nothing in it needs to start at zero.
 */
#define ATTN_DECODE_NOALLOC_SCRATCH_BYTES (4u * 1024u * 1024u)
int attn_decode_noalloc(const void *q, const void *kcache, const void *vcache, const int *seqlens,
                        void *o, float *lse, int B, int Hq, int Hkv, int D, int max_len,
                        float scale, int out_dtype, void *stream);

/*
 * attn_decode_rope -- one decode step that first places the new token: rotary position
 * embedding (rotate-half form) of the new query and key at position p = seqlens[b] - 1, the
 * rotated key (rounded to bf16) and the value stored at cache row p, then decode as attn_decode
 * with the rotated query (kept in fp32, not rounded).
 *   q      [B, Hq, D] bf16, not yet rotated     k_new, v_new [B, Hkv, D] bf16, k_new not rotated
 *   cos_t, sin_t  [max_len, D/2] fp32 tables, row p used for position p:
 *                 [x1 | x2] -> [x1 cos - x2 sin | x1 sin + x2 cos] on the two halves of a head
 *   kcache, vcache [B, Hkv, max_len, D] bf16, row seqlens[b]-1 overwritten
 *   seqlens [B] int32 (device): lengths including the new token
 *   o [B, Hq, D] bf16 or fp32 by out_dtype, lse [B, Hq] fp32 or NULL
 * q, k_new, v_new, cos_t, sin_t must be 16-byte aligned (else ATTN_ERR_ALIGN).
 * Batches up to 1024: one kernel does everything. The query is rotated as it is loaded; the
 * warp whose key slice ends a sequence substitutes the rotated key (rounded to bf16) and the
 * value for the cache row it just read, and writes both to the cache. Larger batches: a small
 * kernel rotates q (kept in fp32) and stores the key and value first, then the decode runs.
 * Scratch (partials; the rotated queries for large batches) comes from the library-owned
 * buffer, grown on first use as for attn_decode. Requires D in {64, 128}.
 * Sources: "triton-optimization" skill (skillsmp.com) section 3.4 (RoPE on the two halves of a
 * head with precomputed cos/sin tables, q and k in one kernel); "Hand-written Triton decoder"
 * (m.nlpx.cn/news/28229) section 1.2 (RoPE computed in fp32 while q and k are loaded) and
 * section 2.2 (RoPE and the KV-cache store are operators of the decode step).
 */
int attn_decode_rope(const void *q, const void *k_new, const void *v_new, const float *cos_t,
                     const float *sin_t, void *kcache, void *vcache, const int *seqlens, void *o,
                     float *lse, int B, int Hq, int Hkv, int D, int max_len, float scale,
                     int out_dtype, void *stream);

/* Workspace bytes attn_decode_ex needs for this shape (0 for invalid arguments).
 * Depends only on the arguments, not on the device. */
size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int D, int max_len);

/* Keys per chunk (one thread block each) that decode uses for this shape (0 if invalid). */
int attn_decode_chunk_len(int B, int Hkv, int max_len);

/* Grow the library-owned decode workspace of the current device to fit this shape. Call it
 * before capturing attn_decode in a CUDA graph (a graph keeps the buffer it was captured with;
 * growing later allocates a new one and keeps the old). */
int attn_reserve_workspace(int B, int Hq, int Hkv, int D, int max_len);

/* Grow the library-owned scratch buffer of the current device (shared by prefill and decode) to
 * at least `bytes`, e.g. attn_prefill_workspace_bytes(...) before capturing a prefill in a CUDA
 * graph. Not during stream capture. Returns ATTN_OK or ATTN_ERR_CUDA. */
int attn_reserve_workspace_bytes(size_t bytes);

/* Debugging aid for the failure path: every pipeline wait of the prefill and decode kernels
 * launched after this call gives up after `cycles` SM clock cycles instead of the default bound
 * (about 2 s; cycles <= 0 restores it). The bound is an argument of each launch (a CUDA graph
 * keeps the one it was captured with). A wait that runs out sets ATTN_DEV_WAIT_TIMEOUT, the block
 * lets the copies and tensor-core work it started finish, and returns without writing its
 * results. A bound of a few cycles makes a wait that is not satisfied at its first probe give up,
 * which lets a test exercise that path without a fault. Process-wide; returns ATTN_OK. */
int attn_debug_set_wait_limit(long long cycles);

/* Synchronise `stream`, then read and clear the current device's status word into *status
 * (bits ATTN_DEV_*). Returns ATTN_OK, or ATTN_ERR_CUDA if the synchronisation failed. */
int attn_device_status(void *stream, unsigned int *status);

/* Static text for a return code. */
const char *attn_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int attn_version(void);

/*
 * attn_debug_build -- 1 in the debug build of this library, 0 otherwise. The pages give no
 * debug build; it serves the checking of this implementation. The debug build (built on
 * demand and loaded by the Python binding when GQA_ATTN_DEBUG=1) compiles in device-side
 * checks of the kernels' index arithmetic: where a cache row range, a partial-result row or a
 * block's work item would fall outside its buffer, the kernel sets ATTN_DEV_INDEX_CHECK in
 * the status word and skips that access instead of trapping. Same entry points, same results;
 * the checks cost a little speed.
 */
int attn_debug_build(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H */
