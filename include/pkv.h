/*
 * pkv.h -- C ABI of the paged-KV attention library (libpkv.so, sm_103a).
 *
 * The library implements the per-decoder-layer paged-KV attention path of the
 * minimal vLLM-style engine nano-vllm, as described on the page
 * "13. 读一个最小推理引擎：nano-vllm" (commit bb823b3):
 *
 *   1. pkv_kv_cache_write      -- scatter each scheduled token's K and V into
 *                                 the paged cache by slot; slot -1 is skipped.
 *   2. pkv_paged_attn_prefill  -- causal GQA attention of a varlen batch whose
 *                                 sequences may be chunked or prefix-cached,
 *                                 reading K/V through block tables.
 *   3. pkv_paged_attn_decode   -- one-query-token GQA attention over a batch,
 *                                 reading K/V through block tables.
 *
 * Conventions shared by every call
 * --------------------------------
 * - bf16 tensors are passed as pointers to raw bfloat16 bit patterns
 *   (pkv_bf16).  Integer metadata is int32.
 * - Every pointer argument is a DEVICE pointer owned by the caller.  The
 *   library never allocates, frees or retains memory.  Scratch memory, where a
 *   call needs some, is passed in by the caller (`workspace`), sized by the
 *   matching *_workspace_bytes function.
 * - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *   asynchronous on that stream; they never synchronise the host and never
 *   read device data on the host, so they can be captured in a CUDA graph.
 * - The cache of one layer is a pair of tensors k_cache, v_cache of shape
 *   (num_blocks, block_size, num_kv_heads, head_dim), C-contiguous
 *   (page section "第五站：执行准备与 KV 容量": one preallocated cache of shape
 *   (2, layers, blocks, block_size, kv_heads, head_dim); one layer's K or V is
 *   one slice of it).  Logical position p of a sequence with block table row
 *   `bt` lives at slot bt[p / block_size] * block_size + p % block_size
 *   (same section, slot mapping).
 * - Supported shapes: block_size == 256 (the page's default, "第二站"),
 *   head_dim == 128, num_kv_heads in [1, 8], num_q_heads a multiple of
 *   num_kv_heads with group size num_q_heads / num_kv_heads in [1, 16], and
 *   num_q_heads <= 64.  Other shapes return PKV_ERR_UNSUPPORTED.
 * - GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
 * - Return value (pkv_status, an int-sized enum): PKV_OK, or a negative
 *   status for a host-side argument error (nothing is launched) or a launch
 *   error.  Faults inside a kernel
 *   surface at the caller's next synchronisation.  Invalid device-side values
 *   that the host cannot see (an out-of-range slot or block id, a bounded wait
 *   that timed out) never fault: the offending access is skipped or clamped
 *   and a bit is set in the library's device error word, readable with
 *   pkv_device_error().
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols of the C ABI are exported even when the library is built with
 * hidden default visibility. */
#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

typedef uint16_t pkv_bf16; /* raw bfloat16 bit pattern */

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_NULL = -1,        /* a required pointer is NULL */
  PKV_ERR_SHAPE = -2,       /* inconsistent or negative sizes */
  PKV_ERR_UNSUPPORTED = -3, /* shape outside the supported set (see above) */
  PKV_ERR_WORKSPACE = -4,   /* workspace NULL or smaller than required */
  PKV_ERR_CUDA = -5,        /* a CUDA runtime/driver call or launch failed */
  PKV_ERR_ALIGN = -6        /* a pointer or stride breaks 16-byte alignment */
} pkv_status;

/* Bits of the device error word (pkv_device_error). */
#define PKV_DEVERR_SLOT_RANGE 0x1u   /* kv write: slot < -1 or >= num_blocks*block_size */
#define PKV_DEVERR_BLOCK_RANGE 0x2u  /* a block table entry outside [0, num_blocks) */
#define PKV_DEVERR_LEN_RANGE 0x4u    /* a context/sequence length outside its stated bound */
#define PKV_DEVERR_WAIT_TIMEOUT 0x8u /* a bounded pipeline wait gave up */

/* Human-readable name of a status code.  Never NULL. */
PKV_API const char* pkv_status_string(int status);

/* Library ABI version (major * 100 + minor). */
PKV_API int pkv_version(void);

/*
 * KV-cache write (page section "第六站：注意力层": before attention, in
 * prefill and decode alike, a small kernel copies every scheduled token's K
 * and V into the paged cache; slot -1 marks CUDA-graph padding and is
 * skipped).
 *
 *   k, v           [num_tokens, num_kv_heads, head_dim] bf16; token i's row
 *                  of num_kv_heads*head_dim contiguous elements starts at
 *                  element i * k_token_stride (resp. v_token_stride).
 *                  Strides are in elements, >= num_kv_heads*head_dim.
 *   slot_mapping   [num_tokens] int32: destination slot of token i, or -1.
 *                  Slots of one call must be distinct (duplicate slots give
 *                  an unspecified one of the rows).  Out-of-range slots are
 *                  skipped and flag PKV_DEVERR_SLOT_RANGE.
 *   k_cache, v_cache  (num_blocks, block_size, num_kv_heads, head_dim) bf16,
 *                  modified in place: row `slot` receives token i's row
 *                  bit-exactly; every other element is left untouched.
 * Pointers and strides must give 16-byte aligned rows (PKV_ERR_ALIGN
 * otherwise).  num_tokens == 0 is a no-op.
 */
PKV_API pkv_status pkv_kv_cache_write(const pkv_bf16* k, int64_t k_token_stride, const pkv_bf16* v,
                       int64_t v_token_stride, const int32_t* slot_mapping, int32_t num_tokens,
                       pkv_bf16* k_cache, pkv_bf16* v_cache, int32_t num_blocks, int32_t block_size,
                       int32_t num_kv_heads, int32_t head_dim, void* stream);

/*
 * Scratch bytes pkv_paged_attn_decode (and the fused-write variant) needs for
 * `batch` sequences on the CUDA device that is current when this is called.
 * The size depends on that device's SM count (the decode kernel splits the
 * batch's tokens into one equal share per SM and keeps one partial result
 * per (sequence or share boundary, query head)), so query it with the device
 * the decode will run on current.  `max_context_len` is accepted so that the
 * query takes the decode call's own bounds; the size does not depend on it.
 * Returns 0 for a negative batch, num_q_heads <= 0, or when the device cannot
 * be queried.
 */
PKV_API size_t pkv_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t max_context_len);

/*
 * Decode attention (page section "第六站：注意力层": decode attends from one
 * new token per sequence to that sequence's history, reading it from the
 * paged cache through the block table; "第五站": CUDA-graph pad rows).
 *
 *   q             [batch, num_q_heads, head_dim] bf16, 16-byte aligned.
 *   k_cache, v_cache  as in pkv_kv_cache_write (already holding the new
 *                 token: call pkv_kv_cache_write first).
 *   context_lens  [batch] int32: L_b, the tokens of sequence b to attend to,
 *                 the new one included.  L_b == 0 marks a pad row: its output
 *                 is zeros and nothing is read for it.  L_b must be <=
 *                 max_context_len and <= max_blocks_per_seq * block_size;
 *                 a larger (or negative) L_b flags PKV_DEVERR_LEN_RANGE and
 *                 is clamped to that bound (or to 0).
 *   block_tables  [batch, max_blocks_per_seq] int32, row b lists sequence b's
 *                 physical blocks in logical order; entries at index
 *                 >= ceil(L_b / block_size) are never read.
 *   scale         multiplies q.k before the softmax (usually 1/sqrt(head_dim)).
 *   out           [batch, num_q_heads, head_dim] bf16:
 *                 out[b,h] = sum_t softmax_t(scale * q[b,h].K[t]) V[t], with
 *                 K, V the kv head h / (num_q_heads/num_kv_heads) rows of the
 *                 first L_b logical positions.  Accumulation is fp32; the
 *                 probabilities are rounded to bf16 before the V product.
 *   workspace     >= pkv_decode_workspace_bytes(batch, num_q_heads, max_context_len)
 *                 device bytes, 256-byte aligned, contents need not be
 *                 initialised; overwritten by the call.  Two calls that may
 *                 run concurrently need two workspaces.
 */
PKV_API pkv_status pkv_paged_attn_decode(const pkv_bf16* q, const pkv_bf16* k_cache, const pkv_bf16* v_cache,
                          const int32_t* context_lens, const int32_t* block_tables,
                          int32_t max_blocks_per_seq, int32_t batch, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                          int32_t num_blocks, int32_t max_context_len, float scale, pkv_bf16* out,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * Decode attention with the KV-cache write fused in: the same result as
 * pkv_kv_cache_write(k_new, v_new, slot_mapping, ...) followed by
 * pkv_paged_attn_decode(...), in one call (page section "第六站：注意力层":
 * write the step's K/V first, then attend).  Each sequence's new K/V row is
 * written by the kernel that then reads it, which saves the separate write
 * launch and its pass over the new rows.
 *
 *   k_new, v_new   [batch, num_kv_heads, head_dim] bf16, row b at element
 *                  b * k_token_stride (resp. v_token_stride); 16-byte aligned.
 *   slot_mapping   [batch] int32: the slot of position context_lens[b] - 1
 *                  (the new token), or -1 for a padding row.  A slot that is
 *                  neither is not written and flags PKV_DEVERR_SLOT_RANGE
 *                  (writing it could race with the attention's own reads).
 *   k_cache, v_cache  written at those slots, read as in pkv_paged_attn_decode.
 * Every other argument is as in pkv_paged_attn_decode.
 */
PKV_API pkv_status pkv_paged_attn_decode_fused_write(
    const pkv_bf16* q, const pkv_bf16* k_new, int64_t k_token_stride, const pkv_bf16* v_new,
    int64_t v_token_stride, const int32_t* slot_mapping, pkv_bf16* k_cache, pkv_bf16* v_cache,
    const int32_t* context_lens, const int32_t* block_tables, int32_t max_blocks_per_seq,
    int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
    int32_t num_blocks, int32_t max_context_len, float scale, pkv_bf16* out, void* workspace,
    size_t workspace_bytes, void* stream);

/*
 * Varlen causal prefill attention (page sections "第二站" -- every step
 * computes from num_cached_tokens onward; "第三站" -- only the first sequence
 * of a step may be a split chunk; "第六站" -- with prefix hits or a chunk
 * continuation the block table is passed so the whole context is read from
 * the paged cache).
 *
 *   q             [total_q, num_q_heads, head_dim] bf16, packed: sequence i
 *                 owns rows cu_seqlens_q[i] .. cu_seqlens_q[i+1]-1.
 *   cu_seqlens_q  [num_seqs+1] int32, cu_seqlens_q[0] == 0, n_i = difference.
 *   cu_seqlens_k  [num_seqs+1] int32, L_i = difference = tokens of sequence i
 *                 in the cache after the write (cached + new).
 *                 c_i = L_i - n_i >= 0 is num_cached_tokens; query row j of
 *                 sequence i sits at position c_i + j and attends to keys
 *                 0 .. c_i + j (causal mask aligned bottom-right).
 *   block_tables  [num_seqs, max_blocks_per_seq] int32.
 *   max_seqlen_q, max_seqlen_k  host-known upper bounds of n_i and L_i;
 *                 max_seqlen_q sizes the launch (a sequence with more new
 *                 tokens flags PKV_DEVERR_LEN_RANGE and its leading query
 *                 tiles are not computed).  A sequence with c_i < 0 or
 *                 L_i > max_blocks_per_seq * block_size flags the same bit
 *                 and is skipped.
 *   out           [total_q, num_q_heads, head_dim] bf16.
 * Accumulation is fp32; probabilities are rounded to bf16 before the V
 * product.  total_q == 0 is a no-op.
 */
PKV_API pkv_status pkv_paged_attn_prefill(const pkv_bf16* q, const pkv_bf16* k_cache, const pkv_bf16* v_cache,
                           const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q,
                           int32_t max_seqlen_k, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale,
                           pkv_bf16* out, void* stream);

/*
 * Prefill attention with the KV-cache write fused in: the same result as
 * pkv_kv_cache_write(k_new, v_new, slot_mapping, ...) of the step's total_q
 * new tokens followed by pkv_paged_attn_prefill(...), in one call (page
 * section "第六站：注意力层": in prefill and decode alike the step's K/V are
 * written into the cache first, then attention reads the cache).  Every SM
 * writes a share of the new rows, then waits at a grid-wide barrier for all
 * others before the first cache read, so the write costs no launch of its own
 * and its rows are still in L2 when attention reads them.
 *
 *   k_new, v_new   [total_q, num_kv_heads, head_dim] bf16, token i's row at
 *                  element i * k_token_stride (resp. v_token_stride);
 *                  16-byte aligned, strides multiples of 8 elements.
 *   slot_mapping   [total_q] int32: the cache slot of new token i, or -1
 *                  (skipped).  Out-of-range slots are skipped and flag
 *                  PKV_DEVERR_SLOT_RANGE.
 *   k_cache, v_cache  written at those slots, then read as in
 *                  pkv_paged_attn_prefill.
 *   workspace      >= pkv_prefill_fused_workspace_bytes() bytes, 16-byte
 *                  aligned, ZEROED before its first use (e.g. by cudaMemset
 *                  when allocated); every call leaves it ready for the next.
 *                  Two calls that may run concurrently need two workspaces.
 *                  If a call reports PKV_DEVERR_WAIT_TIMEOUT, zero it again.
 * Every other argument is as in pkv_paged_attn_prefill.  Up to a stated
 * max_seqlen_q of 2048 the call uses the persistent kernel (one CTA per SM,
 * launched cooperatively so that all of them are resident at the barrier); a
 * launch that cannot be co-resident returns PKV_ERR_CUDA.  Above 2048 it
 * launches the KV write and then the long-prompt attention kernel on the
 * stream (two launches, faster there) and leaves the workspace untouched;
 * the results are the same either way.
 */
PKV_API size_t pkv_prefill_fused_workspace_bytes(void);
PKV_API pkv_status pkv_paged_attn_prefill_fused_write(
    const pkv_bf16* q, const pkv_bf16* k_new, int64_t k_token_stride, const pkv_bf16* v_new,
    int64_t v_token_stride, const int32_t* slot_mapping, pkv_bf16* k_cache, pkv_bf16* v_cache,
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, const int32_t* block_tables,
    int32_t max_blocks_per_seq, int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q,
    int32_t max_seqlen_k, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
    int32_t num_blocks, float scale, pkv_bf16* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Decode attention without caller scratch: the same computation and
 * arguments as pkv_paged_attn_decode, minus `workspace`/`workspace_bytes`.
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory themselves -- for example a plugin inside a
 * host engine that owns every device allocation and forbids plugins from
 * allocating once serving has started, or a C caller that only holds the raw
 * tensor pointers it was handed.  Such callers cannot obtain the workspace
 * pkv_paged_attn_decode asks for.
 *
 * Scratch lives in one fixed array inside the library, PKV_DECODE_STATIC_SCRATCH_BYTES
 * (8 MiB) per GPU, held by every GPU that loads the library until the process
 * exits.  A call whose batch needs more than that
 * (pkv_decode_workspace_bytes(batch, num_q_heads, max_context_len) > 8 MiB, e.g.
 * batch above 855 at 16 query heads on a 152-SM GPU) returns PKV_ERR_WORKSPACE
 * and launches nothing.  The call allocates nothing and frees nothing.
 *
 * The first call on a device looks up that array's device address (with the
 * device current) and caches it; make that first call before any stream
 * capture (a first call made while `stream` is being captured returns
 * PKV_ERR_CUDA and leaves the capture untouched).  The cached address belongs
 * to the device's primary context as it was at that first call: resetting
 * the device (cudaDeviceReset) afterwards is not supported by this call.  Every call on a device shares the one array and it keeps the
 * previous call's contents; no part of it needs to start at zero.  Calls
 * that can overlap on the GPU (different streams without ordering between
 * them) race on the array and give undefined results: order them, or use
 * pkv_paged_attn_decode with one workspace per stream.
 */
#define PKV_DECODE_STATIC_SCRATCH_BYTES ((size_t)8 << 20)
PKV_API pkv_status pkv_paged_attn_decode_noalloc(const pkv_bf16* q, const pkv_bf16* k_cache,
                                          const pkv_bf16* v_cache, const int32_t* context_lens,
                                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                                          int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                          int32_t max_context_len, float scale, pkv_bf16* out,
                                          void* stream);

/*
 * Step metadata on the device (page section "第五站：执行准备与 KV 容量":
 * prepare_prefill / prepare_decode build the slot mapping with
 * slot = block_table[p / block_size] * block_size + p % block_size and feed
 * only the tokens from num_cached_tokens onward, "第二站"; the varlen attention
 * calls take cumulative lengths, "第六站").
 *
 * Inputs, one entry per sequence i (num_seqs S):
 *   block_ids, table_offsets [S+1]  sequence i's block table is
 *                 block_ids[table_offsets[i] .. table_offsets[i+1]-1].
 *   num_cached [S]   c_i, tokens already in the cache (prefix hits and earlier
 *                 chunks; L_i - 1 for a decode step).
 *   seq_lens [S]     L_i, tokens in the cache after this step (c_i < L_i).
 *   token_capacity   entries of slot_mapping (host-known bound of the new
 *                 tokens, sum of L_i - c_i; extra entries are set to -1).
 * Outputs:
 *   cu_seqlens_q [S+1], cu_seqlens_k [S+1]  prefix sums of L_i - c_i and L_i;
 *   context_lens [S] = L_i;  slot_mapping [token_capacity]: the slot of each
 *   new token, sequence by sequence, positions c_i .. L_i-1, then -1;
 *   block_tables [S, max_blocks_per_seq]: the tables packed, -1 padded.
 * A sequence whose table is shorter than ceil(L_i / block_size) blocks (the
 * decode rule: a token at a position that is a multiple of block_size opens a
 * new block) or whose lengths are inconsistent contributes no tokens and
 * flags PKV_DEVERR_LEN_RANGE; more tokens than token_capacity also flag it.
 */
PKV_API pkv_status pkv_prepare_metadata(const int32_t* block_ids, const int32_t* table_offsets,
                                 const int32_t* num_cached, const int32_t* seq_lens, int32_t num_seqs,
                                 int32_t token_capacity, int32_t max_blocks_per_seq, int32_t block_size,
                                 int32_t num_blocks, int32_t* cu_seqlens_q, int32_t* cu_seqlens_k,
                                 int32_t* context_lens, int32_t* slot_mapping, int32_t* block_tables,
                                 void* stream);

/*
 * Exponential-race sampling of the next token (page section "其余部分":
 * temperature-only sampling that divides the probabilities by exponentially
 * distributed random numbers and takes the largest quotient -- equivalent to
 * sampling by probability; temperature 0 is not allowed).
 *
 *   logits        [batch, vocab] float32, row b at element b * row_stride.
 *   temperatures  [batch] float32, each finite and > 0 (otherwise that row's
 *                 token is -1 and PKV_DEVERR_LEN_RANGE is set).
 *   seed, offset  select the random numbers: token i of row b uses output word
 *                 i % 4 of Philox4x32-10 (counter {i/4, b, offset_lo,
 *                 offset_hi}, key {seed_lo, seed_hi}; Salmon et al., SC 2011)
 *                 as U = ((word >> 9) + 0.5) / 2^23, E = -ln U.  Use a new
 *                 offset (or seed) for every step.
 *   out_tokens    [batch] int32: argmax_i softmax(logits / T)_i / E_i (ties go
 *                 to the smaller index; computed as the argmax of
 *                 l_i log2(e) / T - log2(-log2 U_i)).
 *   workspace     >= pkv_sample_workspace_bytes(batch, vocab) bytes, 256-byte
 *                 aligned, need not be initialised.
 */
PKV_API size_t pkv_sample_workspace_bytes(int32_t batch, int32_t vocab);
PKV_API pkv_status pkv_sample_exponential_race(const float* logits, int64_t row_stride, const float* temperatures,
                                        int32_t batch, int32_t vocab, uint64_t seed, uint64_t offset,
                                        int32_t* out_tokens, void* workspace, size_t workspace_bytes,
                                        void* stream);

/*
 * Read (and, if `clear` is nonzero, reset) the device error word of the
 * current device.  Synchronises the device.  *out receives an OR of
 * PKV_DEVERR_* bits set by kernels since the last clear.
 */
PKV_API pkv_status pkv_device_error(uint32_t* out, int clear);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
