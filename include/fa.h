/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library, libfa.so.
 *
 * Two operations, both the exact attention O = softmax(scale * Q K^T [+ mask]) V
 * computed with an online softmax so that S and P never reach HBM:
 *
 *   fa_fwd     prefill / forward.  Q is cut into tiles of query rows, K/V are
 *              streamed in tiles while a running max m and sum l are kept and
 *              the normalisation is deferred to the end ("[CUDA 优化实战] fmha
 *              sm120 : 超越 torch.sdpa(flash-attention-2)", section 1 "flash
 *              attention" and section 2 "fmha 实现"), with GQA, an optional
 *              top-left causal mask and a per-row log-sum-exp output.
 *
 *   fa_decode  split-KV flash decoding for a single query row per head: the M
 *              keys are cut into chunks, each chunk yields a partial O_c
 *              (normalised inside the chunk) and lse_c, and an LSE-weighted
 *              merge combines them ("CUDA 实现 Flash Decoding：解码阶段并行度重建
 *              与性能剖析", section 2.2 Steps 1 and 2, section 3 "两段式 kernel").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Layouts are contiguous, heads inner: q and o [B, N, Hq, d]; k and v
 *    [B, M, Hkv, d]; lse [B, Hq, N] fp32.  Decode uses N = 1: q/o [B, 1, Hq, d],
 *    lse [B, Hq].
 *  - Element type: fp16 or bf16 for q, k, v and o (all four the same); all
 *    arithmetic accumulates in fp32.  o is rounded to nearest-even.
 *  - GQA: query head h reads kv head h / (Hq / Hkv); Hq % Hkv must be 0.
 *  - Causal (fa_fwd only): key j is visible to query i iff j <= i (top-left
 *    aligned, so no row is ever empty).
 *  - lse is the natural log of sum_j exp(scale * q_i . k_j) over the visible
 *    keys, in fp32 ("Tensor Core 迁移计划", cross-cutting concerns: the LSE
 *    output stays fp32).  lse may be NULL; it is then not written.
 *  - Pointers are DEVICE pointers owned by the caller (the library never
 *    allocates, frees or keeps them); q, k, v, o must be 16-byte aligned, lse
 *    4-byte aligned.  The output buffers must not overlap the inputs.
 *  - Calls are asynchronous on `stream` (NULL = legacy default stream) on the
 *    current CUDA device, which must be compute capability 10.3 (GB300).
 *  - The return value reports argument errors (checked before any CUDA call)
 *    and launch errors; it does not synchronise.  Device-side failures of the
 *    bounded waits are reported later by fa_get_last_device_status().
 *  - Errors are return codes; nothing asserts or aborts the process.
 */
#ifndef FA_H
#define FA_H

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
struct CUstream_st;
typedef struct CUstream_st* fa_stream_t;

typedef enum {
    FA_FP16 = 0,
    FA_BF16 = 1
} fa_dtype;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, Hq % Hkv != 0,
                                 misaligned pointer, bad scale, size overflow */
    FA_ERR_UNSUPPORTED = 2,   /* d not in {64, 128}, unknown dtype, device not sm_103 */
    FA_ERR_CUDA = 3,          /* a CUDA runtime/driver call or kernel launch failed */
    FA_ERR_NO_MEMORY = 4,     /* the decode workspace could not be allocated */
    FA_ERR_TIMEOUT = 5,       /* a device-side bounded wait expired (see below) */
    FA_ERR_SCRATCH_LIMIT = 6  /* the problem needs more than the static scratch of
                                 fa_decode_noalloc holds */
} fa_status;

/*
 * Exact attention forward (prefill).
 *
 *   q   [B, N, Hq, d]   fp16/bf16, device
 *   k   [B, M, Hkv, d]  same type
 *   v   [B, M, Hkv, d]  same type
 *   o   [B, N, Hq, d]   same type, written
 *   lse [B, Hq, N]      fp32, written unless NULL
 *   causal  0 = full attention, 1 = top-left causal mask
 *   scale   multiplies the logits; must be finite and > 0 (usually 1/sqrt(d))
 *
 * Limits: B, Hq, Hkv, N, M >= 1; d in {64, 128}; B*N*Hq*d and B*M*Hkv*d
 * below 2^40 elements.  Returns FA_OK once the work is enqueued.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int Hq, int Hkv, int N, int M, int d, int causal,
                 float scale, fa_dtype dtype, fa_stream_t stream);

/*
 * fa_fwd on host-resident tensors: the same operation, arguments, layouts and
 * results, with q, k, v, o and lse in host memory.  The problem is cut into
 * independent chunks of (b, a group of kv heads with their query heads), about
 * four in all (one per batch entry when B >= 4).  Chunk c's inputs are copied to
 * the device on an internal stream while chunk c-1 runs fa_fwd on `stream` and
 * chunk c-2's o and lse are copied back on another internal stream, so the
 * transfers overlap the kernels.  Each chunk gives exactly what fa_fwd gives for
 * those heads.
 *
 * Host memory should be page-locked (pinned) for the copies to overlap;
 * pageable memory works, with copies that do not overlap.  Returns FA_OK once
 * the work is enqueued; `stream` is ordered after the last copy back, so
 * synchronize it before reading o and lse, and keep the inputs unchanged until
 * then.  Calls on one stream must come from one host thread at a time.
 *
 * Workspace: two chunks' device staging per (device, stream), from the same
 * cached buffer as fa_decode; two internal streams and a few events per
 * (device, stream), released by fa_release_workspaces().
 * Errors: as fa_fwd.
 */
fa_status fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int Hq, int Hkv, int N, int M, int d, int causal,
                      float scale, fa_dtype dtype, fa_stream_t stream);

/*
 * Split-KV flash decoding (one query row per head).
 *
 *   q   [B, 1, Hq, d]   fp16/bf16, device
 *   k   [B, M, Hkv, d]  same type
 *   v   [B, M, Hkv, d]  same type
 *   o   [B, 1, Hq, d]   same type, written
 *   lse [B, Hq]         fp32, written unless NULL
 *   chunk   keys per split (>= 1); the split count is nc = ceil(M / chunk),
 *           the last chunk may be short.
 *
 * Two kernels run back to back on `stream`: the chunk kernel writes nc fp32
 * partials (O_c, lse_c) per (b, h) into a workspace, the merge kernel combines
 * them.  The workspace (B*Hq*nc*(d+1) fp32 values) is owned by the library:
 * one buffer per (device, stream), allocated on first use, grown on demand
 * (growing synchronises the device) and kept until fa_release_workspaces().
 * Calls on the same stream are ordered by the stream; calls on different
 * streams use different buffers.  FA_ERR_NO_MEMORY if it cannot be allocated.
 */
fa_status fa_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int Hq, int Hkv, int M, int d, int chunk,
                    float scale, fa_dtype dtype, fa_stream_t stream);

/*
 * Split-KV decode in a single launch.  Same arguments, layouts, results and
 * errors as fa_decode; the chunk partials are merged by the chunk kernel
 * itself instead of a second kernel.  Each persistent CTA walks the chunks
 * s, s + S, s + 2S, ... of one (b, kv head) (S CTAs per (b, kv head), as many
 * as fit in one wave) and merges its chunks with the LSE weights of "CUDA 实现
 * Flash Decoding" section 2.2 Step 2.  When one pass over a K/V tile serves all
 * query heads of the kv head (Hq/Hkv <= 4 for 16-bit inputs) it does so on the
 * fly, carrying the running max, sum and accumulators from chunk to chunk; else
 * it merges the chunk partials it wrote.  The last of the S CTAs to finish
 * merges the S results into o and lse.  The merge is associative, so the result
 * is the same up to rounding order.  The page's section 8 lists this single
 * launch as its fourth lever.
 *
 * Workspace: the same per-(device, stream) buffer as fa_decode, plus room for
 * one merged result per CTA (at most B*Hq*nc*(d+1) fp32), plus B*Hkv int
 * tickets that are zeroed when allocated and reset by the kernel itself; after
 * a call that reported FA_ERR_TIMEOUT call fa_release_workspaces() before the
 * next call on that stream.
 */
fa_status fa_decode_fused(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int Hq, int Hkv, int M, int d, int chunk,
                          float scale, fa_dtype dtype, fa_stream_t stream);

/*
 * Split-KV decode that allocates no device memory.  The pages have no
 * counterpart: this entry point exists for callers that cannot call
 * cudaMalloc -- code running while a CUDA graph is captured, processes whose
 * device memory must all come from their own pool, hosts that forbid
 * allocation after start-up.
 *
 * Same arguments, layouts, results and argument errors as fa_decode, but the
 * fp32 chunk partials live in one array of static device memory of
 * FA_DECODE_NOALLOC_SCRATCH_BYTES bytes, which every GPU that loads the
 * library's module holds until the process exits.  A problem needing more
 * than that -- B*Hq*ceil(M/chunk)*(d+1)*4 bytes -- returns
 * FA_ERR_SCRATCH_LIMIT before any launch (B=2, Hq=8, M=65536, chunk=128,
 * d=128 needs 4.2 MB).  The call makes no cudaMalloc, cudaFree or other
 * allocating call.
 *
 * The first call on a device looks up the array's device address and that
 * of the library's status word (cudaGetSymbolAddress, once per device, with
 * that device current) and applies the launch attributes of every decode
 * kernel variant (each head dim, type and GQA group): make that first call
 * before any stream capture starts.  All calls share the one array and it
 * keeps the previous call's contents; nothing in it needs to start at zero,
 * but calls that overlap on the GPU (e.g. on two streams with no ordering
 * between them) race on it and give undefined results.  The kernels' waits
 * take the limit of fa_set_wait_timeout_ns() at the time of the call, and an
 * expired wait is reported by fa_get_last_device_status(), whose status word
 * (static device memory as well) every entry point shares.
 */
#define FA_DECODE_NOALLOC_SCRATCH_BYTES (8u << 20)
fa_status fa_decode_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int M, int d, int chunk,
                            float scale, fa_dtype dtype, fa_stream_t stream);

/*
 * Backward of fa_fwd: the gradients dQ, dK, dV of O = softmax(scale Q K^T
 * [+ causal]) V for an upstream gradient dO.  "Tensor Core 迁移计划" (phase
 * 2) names the backward's contractions dV = P^T dO, dP = dO V^T and dQ, dK
 * from dS; dS = P o (dP - D) with D_i = dO_i . O_i is the softmax's Jacobian,
 * and P is recomputed from the forward's LSE (nothing of size N x M is kept).
 *
 *   q, k, v, o   the forward's inputs and output (layouts as fa_fwd).
 *   lse          device, [B, Hq, N] fp32: the natural-log LSE fa_fwd wrote
 *                for the same q, k, v, causal and scale (required).
 *   dout         device, [B, N, Hq, d]: dL/dO, of `dtype`.
 *   dq           device, [B, N, Hq, d] out; dk, dv device, [B, M, Hkv, d] out,
 *                of `dtype` (with GQA, dk/dv of a kv head sum over the query
 *                heads that read it).
 *   others       as fa_fwd.
 * P and dS enter the tensor core as fp16/bf16 (as P does in the forward);
 * every accumulation is fp32.  Three launches on `stream`: D = rowsum(dO o O)
 * (also zeroing the fp32 dQ accumulator), the main kernel, and the dQ
 * conversion.  Workspace: B*N*Hq*(d+1) fp32 values in the library's
 * per-(device, stream) buffer (the one fa_decode uses), allocated or grown on
 * demand (growing synchronises the device).
 * Errors: as fa_fwd; FA_ERR_INVALID_ARG also for a NULL or misaligned lse,
 * dout, dq, dk or dv; FA_ERR_NO_MEMORY if the workspace cannot be allocated.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N,
                 int M, int d, int causal, float scale, fa_dtype dtype, fa_stream_t stream);

/*
 * Split-KV decode over an FP8 (e4m3) K/V cache with one fp32 scale per kv
 * head.  FP8 and INT8/INT4 KV quantisation are named as the next memory-side
 * step in the closing "TODO" section of "[CUDA 优化实战] fmha sm120 : 超越
 * torch.sdpa(flash-attention-2)", and as lever 1 (the only lever that halves
 * the bytes) in section 8 of "CUDA 实现 Flash Decoding：解码阶段并行度重建与
 * 性能剖析".  This is not exact attention over the original 16-bit K/V: it is
 * exact attention over the dequantised cache
 *     K[b][j][h][:] = k_scale[h] * e4m3(k8[b][j][h][:]),
 *     V[b][j][h][:] = v_scale[h] * e4m3(v8[b][j][h][:]),
 * computed like fa_decode: the same chunks and the same LSE-weighted merge.
 * When one pass over a K/V tile serves all query heads of a kv head
 * (Hq/Hkv = 1, 2 or 4), each persistent chunk-kernel CTA merges its chunks on
 * the fly (running max, sum and accumulators carried from chunk to chunk).  It
 * leaves one partial per query head, and the merge kernel combines those few
 * partials rather than one per chunk.  The merge is associative, so only the
 * rounding order differs.
 *
 *   q, o, lse   as fa_decode; q and o are fp16 or bf16 (`dtype`).
 *   k8, v8      device, [B, M, Hkv, d] bytes, each an OCP e4m3 value (bias 7,
 *               no infinities, 0x7f/0xff are NaN); 16-byte aligned.
 *   k_scale,    device, Hkv fp32 each, finite; the kernel applies k_scale once
 *   v_scale     per score and v_scale once per output row.
 *   others      as fa_decode.
 * Errors: as fa_decode, plus FA_ERR_INVALID_ARG for a NULL scale pointer or
 * one not 4-byte aligned.  The workspace is fa_decode's.
 */
fa_status fa_decode_fp8(const void* q, const void* k8, const void* v8, const float* k_scale,
                        const float* v_scale, void* o, float* lse, int B, int Hq, int Hkv, int M,
                        int d, int chunk, float scale, fa_dtype dtype, fa_stream_t stream);

/*
 * Split-KV decode over a paged K/V cache addressed through a block table, the
 * layout paged attention needs to plug into an inference server (the closing
 * "TODO" section of "[CUDA 优化实战] fmha sm120 : 超越
 * torch.sdpa(flash-attention-2)", "attention with kv cache block").  Key j of
 * sequence b is row j % page_size of page block_table[b][j / page_size]; the
 * result is fa_decode's on the gathered K/V of the first seq_lens[b] keys, up
 * to rounding order.  As in fa_decode_fp8, when Hq/Hkv is 1, 2 or 4 each
 * persistent chunk-kernel CTA merges its chunks on the fly, and the merge
 * kernel combines one partial per CTA.
 *
 *   q, o, lse          as fa_decode (one query row per (b, h)).
 *   k_cache, v_cache   device, [num_pages, page_size, Hkv, d] of `dtype`,
 *                      16-byte aligned.
 *   block_table        device int32 [B, max_pages_per_seq], row-major.  Every
 *                      entry that covers a key below seq_lens[b] must lie in
 *                      [0, num_pages); the library cannot check device data,
 *                      and an entry outside that range reads its rows as
 *                      zeros (the copy engine's bounds), never out of bounds.
 *   seq_lens           device int32 [B]: keys of sequence b, taken as
 *                      min(seq_lens[b], max_seq_len); 0 (or negative) gives
 *                      o = 0 and lse = -inf for that sequence.
 *   max_seq_len        upper bound of seq_lens (sizes the chunk grid); > 0.
 *   page_size          a power of two, 8 <= page_size <= 65536.
 *   max_pages_per_seq  >= ceil(max_seq_len / page_size).
 *   chunk              keys per chunk, a multiple of min(page_size, 128), so
 *                      that every copy of keys starts on a page boundary.
 * Errors: FA_ERR_INVALID_ARG for NULL or misaligned pointers, non-positive
 * sizes, a page size or chunk outside the rules above, or Hq % Hkv != 0;
 * FA_ERR_UNSUPPORTED as fa_decode.  Workspace: fa_decode's, sized with
 * M = max_seq_len.
 */
fa_status fa_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                          const int* block_table, const int* seq_lens, void* o, float* lse, int B,
                          int Hq, int Hkv, int max_seq_len, int num_pages, int page_size,
                          int max_pages_per_seq, int d, int chunk, float scale, fa_dtype dtype,
                          fa_stream_t stream);

/* Static, human-readable name of a status code (never NULL). */
const char* fa_status_string(fa_status status);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word.  Every spin-wait inside the kernels of every entry point (the
 * allocation-free decode included) is bounded; when one expires the kernel
 * records FA_ERR_TIMEOUT there, drains its own in-flight copies and
 * tensor-core work, frees its tensor memory and returns (its outputs are then
 * undefined).  The word is static device memory, one per device: reading and
 * clearing it allocates nothing.  Returns FA_OK, FA_ERR_TIMEOUT, or
 * FA_ERR_CUDA if the synchronisation itself failed.
 */
fa_status fa_get_last_device_status(fa_stream_t stream);

/*
 * Sets the limit of every device-side wait, in nanoseconds, for launches made
 * after the call by any entry point (process-wide; default 2e9 = 2 s; 0
 * restores the default).  The limit travels with each launch as an argument,
 * so a captured CUDA graph keeps the limit in force when it was captured.
 */
void fa_set_wait_timeout_ns(unsigned long long ns);

/*
 * Test hook for the bounded-wait path: launches one CTA that waits on a
 * shared-memory barrier nobody arrives on, under the current wait limit, so
 * that the wait expires and the kernel records FA_ERR_TIMEOUT in the status
 * word.  It faults nothing and leaves the context usable.
 */
fa_status fa_selftest_wait_timeout(fa_stream_t stream);

/* Frees every decode workspace the library holds (synchronises each device used). */
void fa_release_workspaces(void);

/* ABI version of this header, 1. */
int fa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
