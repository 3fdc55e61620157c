/*
 * libbwattn: exact scaled-dot-product attention on one GB300 (sm_103a).
 *
 *   O = softmax(Q K^T * scale) V,  scale normally 1/sqrt(d)
 *
 * computed with the online-softmax recurrence (a running max m, running sum l and an
 * unnormalised output o, rescaled by exp(m - m_new) tile by tile), so that the score matrix
 * never reaches device memory. Sources, by page title and section:
 *   - "Attention from the kernel's side: FlashAttention, online softmax and fused dequant":
 *     "The online softmax" (the recurrence), "FlashAttention: what never touches memory"
 *     (Q tile resident, K/V tiles streamed, O written once), "Prefill and decode are
 *     different problems" (GQA reuse, flash-decoding split over the KV axis).
 *   - "Attention kernels" (llm-inference-explained): "Maths" (the recurrence and the merge
 *     rule for two partial states (m, l, o)), "Concept" (split-K decode).
 *   - "Attention Computation in Practice": section 5, "The four attention kernels you
 *     actually use" (prefill, decode, append/mixed with cu_seqlens, cross attention),
 *     "GQA in the kernel" (query head h reads KV head h / (Hq / Hkv)), "Masking variants"
 *     (causal j <= i and the skip / full / diagonal rule per block pair).
 *
 * Conventions shared by every call:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller, contiguous in the layout
 *     given, 16-byte aligned (attn_fwd_host alone takes host pointers). The library never
 *     allocates or frees memory and never synchronises the host.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*; NULL = the
 *     legacy default stream) and returns a status code. Argument checks happen on the host
 *     before any CUDA call, so a rejected call has no side effect.
 *   - Causal masking with Nq != Nk is aligned to the end: query i sees key j iff
 *     j <= i + (Nk - Nq). A query that sees no key gets O = 0 and LSE = -inf.
 *   - LSE (log-sum-exp) is the natural log of sum_j exp(scale * q.k_j) over the visible keys,
 *     written as fp32. Passing lse = NULL skips it.
 *   - Inputs are bf16 (IEEE bfloat16) unless a dtype argument says otherwise; arithmetic is
 *     fp32 (tensor cores with fp32 accumulation for bf16 inputs, fp32 FMA for fp32 inputs).
 *   - State kept across calls: a device status word that records a timed-out internal wait
 *     (see bwattn_get_status); rings of per-launch device counters (the prefill's item
 *     counters, the decode's merge tickets), each launch taking its share when it is enqueued
 *     and leaving it reset; the static scratch of attn_decode_static; the streams and events
 *     of attn_fwd_host. Calls are thread-safe and may be captured into CUDA graphs (except
 *     attn_fwd_host).
 *   - Limit of those rings, per device: a share is handed out again after 4096 further
 *     prefill launches (item counters) or 65,536 further merge tickets (a fused-merge decode
 *     takes one ticket per (sequence, KV head, row group)). Calls still running when their
 *     share comes round again would share it and corrupt each other's scheduling or merge:
 *     keep fewer launches than that in flight on one device at a time, counting every replay
 *     of a captured graph that runs concurrently with other calls.
 */
#ifndef BWATTN_H
#define BWATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---- */
#define BWATTN_OK 0
#define BWATTN_ERR_INVALID_ARG 1 /* null pointer, size out of range, Hq % Hkv != 0, misaligned pointer, workspace too small */
#define BWATTN_ERR_UNSUPPORTED 2 /* valid arguments outside what the kernels implement (dtype / head dim / group size) */
#define BWATTN_ERR_CUDA 3        /* a CUDA runtime call or kernel launch failed; see bwattn_last_cuda_error() */
#define BWATTN_ERR_TIMEOUT 4     /* a kernel gave up an internal wait; reported by bwattn_get_status() */

/* ---- dtypes ---- */
#define BWATTN_DTYPE_FP32 0
#define BWATTN_DTYPE_BF16 1

/*
 * attn_fwd: prefill / cross attention over dense batches.
 * ("Attention Computation in Practice", section 5, kernel classes 1 and 4;
 *  "Attention from the kernel's side", "FlashAttention: what never touches memory".)
 *
 *   q, o : [B, Hq, Nq, d]        (dtype; o has the same dtype as q)
 *   k, v : [B, Hkv, Nk, d]       (dtype)
 *   lse  : [B, Hq, Nq] fp32, may be NULL
 *   causal: 0 = no mask (cross attention), 1 = causal aligned to the end
 *   scale: multiplies q.k before the softmax; must be finite and > 0
 *   dtype: BWATTN_DTYPE_BF16 (tcgen05 tensor-core kernel, d in {64, 128, 256}: the fast
 *          kernels' head dims, "Production implications"; d = 256 keeps one query tile per
 *          CTA because its fp32 O tile fills half of tensor memory) or
 *          BWATTN_DTYPE_FP32 (fp32 FMA kernel, d in {64, 128})
 * Query head h reads KV head h / (Hq / Hkv). Nq = 0 or B = 0 is a valid no-op; Nk = 0 gives
 * O = 0 and LSE = -inf. Errors: INVALID_ARG for null / misaligned pointers, negative sizes,
 * Hq % Hkv != 0, bad scale; UNSUPPORTED for other d or dtype.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
             int Nk, int d, int causal, float scale, int dtype, void* stream);

/*
 * attn_fwd_host: attn_fwd on HOST-resident tensors (same shapes, layouts, dtypes and errors),
 * copies included. The (sequence, KV head) units are cut into up to 8 chunks; each chunk's
 * copies in, kernel and copies out run on library-owned streams so that transfers overlap
 * kernels (no counterpart on the pages; it is the host-memory end of the same computation).
 *
 *   q, k, v, o, lse : HOST pointers in the attn_fwd layouts; page-locked memory is needed for
 *                     the copies to overlap (pageable memory works, serialised); lse may be NULL
 *   workspace       : DEVICE buffer, 256-byte aligned, of at least
 *                     attn_fwd_host_workspace_size(B, Hq, Hkv, Nq, Nk, d, dtype) bytes (two
 *                     chunks of staging); contents undefined on exit
 *   stream          : the work starts after everything already queued on it, and work queued on
 *                     it afterwards starts after the last copy out; the host buffers must stay
 *                     valid until then
 * Calls from several host threads are serialised while they enqueue (the streams are shared).
 * On an error return after copies were queued (a CUDA error part way through), the call first
 * waits on the host for its own streams, so no copy from or to the host buffers is still
 * running when it returns; the outputs are then undefined.
 */
int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                  int Nk, int d, int causal, float scale, int dtype, void* workspace, size_t workspace_bytes,
                  void* stream);
size_t attn_fwd_host_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d, int dtype);

/*
 * attn_fwd_window: causal prefill with a sliding window ("Attention Computation in Practice",
 * "Masking variants": sliding window i - W < j <= i). Same layouts, dtypes and errors as
 * attn_fwd with causal = 1; query i sees keys j with i' - window < j <= i', i' = i + (Nk - Nq).
 * K/V tiles entirely outside every row's window are not read. window >= 1, else INVALID_ARG;
 * window >= Nk gives the plain causal result.
 */
int attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                    int Nk, int d, int window, float scale, int dtype, void* stream);

/*
 * attn_decode_workspace_size: bytes of caller-provided workspace attn_decode needs for the
 * per-split partial states (m, l, o[d]) in fp32.
 */
size_t attn_decode_workspace_size(int B, int Hq, int d, int num_splits);

/*
 * attn_decode: single-query decode against a contiguous KV cache, split over the KV axis
 * (flash-decoding), partial states merged with the two-state merge rule.
 * ("Attention from the kernel's side", "Prefill and decode are different problems";
 *  "Attention kernels", "Maths", second display; "Attention Computation in Practice",
 *  section 5, kernel class 2 and "PagedAttention's kernel difference", contiguous form.)
 *
 *   q, o     : [B, Hq, d] bf16 (the one new query of each sequence)
 *   kcache,
 *   vcache   : [B, Hkv, nk_cap, d] bf16
 *   nk       : [B] int32 DEVICE array, valid keys per sequence, 0 <= nk[b] <= nk_cap;
 *              every valid key is visible (the new token's K/V are already in the cache)
 *   num_splits: KV slices per (sequence, KV head), 1..1024; slices past nk[b] are empty
 *   scale    : finite, > 0
 *   lse      : [B, Hq] fp32, may be NULL
 *   workspace: device buffer of at least attn_decode_workspace_size(B, Hq, d, num_splits)
 *              bytes; contents on entry are ignored, on exit undefined. Must not be shared
 *              by calls that may overlap on the GPU.
 * The g = Hq / Hkv query heads of a group are packed against each K/V tile, so every cache
 * byte is read once. Supported: d in {64, 128, 256} ("Production implications": the fast
 * kernels' head dims), 1 <= g <= 32. Errors as for attn_fwd, plus INVALID_ARG when the
 * workspace is NULL or too small.
 */
int attn_decode(const void* q, const void* kcache, const void* vcache, void* o, const int32_t* nk, int B, int Hq,
                int Hkv, int nk_cap, int d, int num_splits, float scale, float* lse, void* workspace,
                size_t workspace_bytes, void* stream);

/*
 * attn_decode_paged: single-query decode against a paged KV cache: the cache is a pool of
 * fixed-size pages and a per-sequence block table lists which page holds each run of
 * page_size consecutive keys. ("Attention Computation in Practice", "PagedAttention's kernel
 * difference": block_table[b] = [17, 3, 92, ...], read block 17, then 3, ...; the kernel takes
 * the table as an argument and gathers.) Same split-K pass and merge as attn_decode.
 *
 *   q, o        : [B, Hq, d] bf16
 *   k_pages,
 *   v_pages     : [num_pages, page_size, Hkv, d] bf16 (a page holds page_size consecutive keys
 *                 of every KV head)
 *   block_table : [B, max_pages_per_seq] int32 DEVICE array; key j of sequence b is row
 *                 j % page_size of page block_table[b][j / page_size]. Entries outside
 *                 [0, num_pages) are clamped into the pool (wrong data, never an out-of-bounds read)
 *   nk          : [B] int32 DEVICE array, 0 <= nk[b] <= max_pages_per_seq * page_size
 *   page_size   : a multiple of 16, 16..1024
 *   workspace   : at least attn_decode_workspace_size(B, Hq, d, num_splits) bytes
 * Supported: d in {64, 128, 256}, 1 <= g <= 32. Errors as for attn_decode.
 */
int attn_decode_paged(const void* q, const void* k_pages, const void* v_pages, void* o, const int32_t* block_table,
                      const int32_t* nk, int B, int Hq, int Hkv, int page_size, int num_pages, int max_pages_per_seq,
                      int d, int num_splits, float scale, float* lse, void* workspace, size_t workspace_bytes,
                      void* stream);

/*
 * attn_decode_fp8 / attn_decode_paged_fp8: attn_decode / attn_decode_paged against an FP8 KV
 * cache, each code turned into its value inside the kernel as it is loaded ("Attention from the
 * kernel's side", "Why a quantised cache needs a fused kernel": a separate dequantise pass would
 * move more bytes than the 16-bit cache it replaces; rule 3 of "Rules I use"). The pages' own
 * format (TBQ4) belongs to another project; this is the generic FP8 form:
 *
 *   kcache, vcache /
 *   k_pages, v_pages : the layouts of attn_decode / attn_decode_paged with one byte per element,
 *                      an OCP FP8 E4M3 code (bias 7, no infinities, S.1111.111 = NaN, max 448)
 *   k_scale, v_scale : [Hkv, d] fp32 DEVICE arrays, 16-byte aligned; the cached value of channel
 *                      c of KV head h is e4m3(code) * k_scale[h * d + c] (v_scale for V)
 *   q, o, lse, nk, block_table, page_size, num_splits, scale, workspace: as for attn_decode /
 *                      attn_decode_paged (same workspace size)
 * The cache is read exactly once; arithmetic is f16 x f16 products of the codes against
 * q * k_scale (rescaled per query row by a power of two) with fp32 accumulation. Supported:
 * d = 128, 1 <= g <= 32. Errors as for attn_decode, plus INVALID_ARG for NULL or unaligned
 * scales.
 */
int attn_decode_fp8(const void* q, const void* kcache, const void* vcache, const float* k_scale,
                    const float* v_scale, void* o, const int32_t* nk, int B, int Hq, int Hkv, int nk_cap, int d,
                    int num_splits, float scale, float* lse, void* workspace, size_t workspace_bytes, void* stream);

int attn_decode_paged_fp8(const void* q, const void* k_pages, const void* v_pages, const float* k_scale,
                          const float* v_scale, void* o, const int32_t* block_table, const int32_t* nk, int B, int Hq,
                          int Hkv, int page_size, int num_pages, int max_pages_per_seq, int d, int num_splits,
                          float scale, float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_decode_static: the same single-query split-K decode as attn_decode, for callers that
 * cannot allocate device memory. The pages have no counterpart to this entry point; it exists
 * for deployment. Some callers cannot call cudaMalloc or hand the library a workspace: a
 * plugin or inference-engine host that gives a kernel only its input and output buffers, code
 * whose device memory is entirely owned by another allocator, or a latency-critical loop that
 * cannot afford cudaMalloc's implicit device-wide synchronisation. This call takes the same
 * arguments as attn_decode minus the workspace, and keeps its per-split partial states in a
 * fixed array of BWATTN_DECODE_STATIC_SCRATCH_BYTES inside the library, which every GPU that
 * loads the library holds until the process exits. It allocates nothing.
 *   - Limit: the partials must fit the array, i.e.
 *     attn_decode_workspace_size(B, Hq, d, num_splits) <= BWATTN_DECODE_STATIC_SCRATCH_BYTES
 *     (about B * Hq * num_splits <= 16,000 at d = 128); larger calls return
 *     BWATTN_ERR_UNSUPPORTED without launching anything.
 *   - The first call on each device looks up the array's device address (once per device,
 *     with that device current); make that first call before any stream capture.
 *   - Every call on a device shares the one array, and the array keeps the last call's
 *     contents. Nothing in it needs to start at zero (each call writes every partial it later
 *     reads), but calls that overlap on the GPU (other streams, other host threads) race on it:
 *     order them, e.g. on one stream.
 * Errors otherwise as for attn_decode.
 */
#define BWATTN_DECODE_STATIC_SCRATCH_BYTES (8u * 1024u * 1024u)
int attn_decode_static(const void* q, const void* kcache, const void* vcache, void* o, const int32_t* nk, int B,
                       int Hq, int Hkv, int nk_cap, int d, int num_splits, float scale, float* lse, void* stream);

/*
 * attn_varlen_workspace_size: bytes of workspace attn_varlen needs, from the host-side
 * bounds it is given.
 */
size_t attn_varlen_workspace_size(int num_seqs, int max_seqlen_k, int Hq, int Hkv, int d);

/*
 * attn_varlen: packed batches of sequences with different lengths (append / mixed:
 * speculative verify, chunked prefill), described by prefix sums of the lengths.
 * ("Attention Computation in Practice", section 5, kernel class 3, "varlen kernels with
 *  cu_seqlens".)
 *
 *   q, o         : [total_q, Hq, d] bf16, sequence s owns rows cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1
 *   k, v         : [total_k, Hkv, d] bf16, sequence s owns rows cu_seqlens_k[s] .. cu_seqlens_k[s+1]-1
 *   total_q,
 *   total_k      : host-side row counts of the packed tensors (= cu_seqlens_*[num_seqs]); they
 *                  bound every tensor-core load, so no copy ever reads past the buffers
 *   lse          : [total_q, Hq] fp32, may be NULL
 *   cu_seqlens_q,
 *   cu_seqlens_k : [num_seqs + 1] int32 DEVICE arrays, non-decreasing, [0] = 0
 *   max_seqlen_q,
 *   max_seqlen_k : host-side upper bounds of the per-sequence lengths (grid sizing); a
 *                  sequence longer than its bound is not processed correctly
 *   causal       : 1 = causal aligned to each sequence's end, 0 = none
 *   workspace    : device buffer of at least attn_varlen_workspace_size(...) bytes
 * Sequences whose n_q * (Hq / Hkv) <= 32 run on the split-K decode kernel (all query heads
 * of a KV group packed in one tile); the others run on the tcgen05 prefill kernel. When both
 * run, the split-K pass is a programmatic dependent launch that starts on the SMs the prefill
 * leaves; it still completes after the prefill, so work queued on `stream` after the call sees
 * the whole output.
 * Supported: d in {64, 128, 256}, 1 <= g <= 32. Errors as for attn_decode.
 */
int attn_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_seqlens_q,
                const int32_t* cu_seqlens_k, int num_seqs, int total_q, int total_k, int max_seqlen_q,
                int max_seqlen_k, int Hq, int Hkv, int d, int causal, float scale, void* workspace,
                size_t workspace_bytes, void* stream);

/*
 * attn_varlen_window: attn_varlen with causal = 1 and a sliding window of `window` keys ending
 * at each query's causal limit (aligned to each sequence's end). window >= 1, else INVALID_ARG.
 */
int attn_varlen_window(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_seqlens_q,
                       const int32_t* cu_seqlens_k, int num_seqs, int total_q, int total_k, int max_seqlen_q,
                       int max_seqlen_k, int Hq, int Hkv, int d, int window, float scale, void* workspace,
                       size_t workspace_bytes, void* stream);

/* ---- status and diagnostics ---- */

/* The cudaError_t of the last failing CUDA call made by this thread inside the library (0 if none). */
int bwattn_last_cuda_error(void);

/* Short text for a status code (static storage). */
const char* bwattn_status_string(int status);

/*
 * bwattn_get_status: synchronises `stream`, then returns BWATTN_ERR_TIMEOUT if any kernel of
 * this library on the current device gave up an internal wait since the last
 * bwattn_clear_status(), else BWATTN_OK (or BWATTN_ERR_CUDA if the synchronisation failed).
 * A kernel that gives up a wait writes no further output and leaves the context usable.
 */
int bwattn_get_status(void* stream);

/* bwattn_clear_status: resets the device status word (ordered on `stream`). */
int bwattn_clear_status(void* stream);

/*
 * bwattn_set_wait_timeout_ns: the bound on any single internal wait of a kernel (default
 * 2e9 ns); applies to launches made after the call, from any thread.
 */
void bwattn_set_wait_timeout_ns(uint64_t ns);

/*
 * bwattn_test_wait_timeout: launches a one-CTA kernel that waits on a barrier nothing ever
 * arrives at, bounded by the current wait timeout, so a test can check that a timed-out wait
 * returns BWATTN_ERR_TIMEOUT through bwattn_get_status() with the context still usable.
 */
int bwattn_test_wait_timeout(void* stream);

/* Number of kernels this library has launched successfully in this process (all threads). */
uint64_t bwattn_launch_count(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int bwattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BWATTN_H */
