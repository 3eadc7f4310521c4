/*
 * pkv.h -- C ABI of libpkv, paged-KV attention for a GB300 (sm_103a).
 *
 * The library implements the data-parallel hot path of LLM decoding in an
 * audio-LLM ASR server: appending new key/value rows to a paged KV cache,
 * batched decode attention over that cache, and chunked-prefill attention.
 *
 * Sources of the operations (titles of the pages they come from):
 *  - "FunASR vLLM Inference Engine Guide", section 2 "vLLM Engine Architecture"
 *    and the table "Why vLLM?": the LLM engine runs PagedAttention over a KV
 *    cache that is allocated on demand, with continuous batching and CUDA
 *    graphs.
 *  - "Fun-ASR-Nano Native Runtime Design", section "Decoder And Prompt": the
 *    decoder is a Qwen3-0.6B with 28 layers and 16 query / 8 KV heads.
 *  - "Optimizing ASR for 90-minute multi-speaker audio" (MOSS-TD in
 *    SGLang-Omni): section "Time spent: profiling" (decode takes over 94% of
 *    the time on long audio), section "Chunked prefill for long audio"
 *    (4096-token prefill chunks interleaved with decode steps) and section
 *    "Autoregressive decoding" (decode replayed as CUDA graphs over batches
 *    padded to buckets 1, 2, 4, 8, ...).
 *
 * Data layout (a reading; no page gives one):
 *  - k_pages, v_pages: bf16 [num_pages][num_kv_heads][page_size][head_dim],
 *    K and V in separate pools. One (page, KV head) tile is contiguous.
 *  - Logical position j of request b is page block_table[b][j / page_size],
 *    slot j % page_size. A slot index s names page s / page_size, slot
 *    s % page_size.
 *  - Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *  - q and out: bf16, row-major [rows][num_q_heads][head_dim].
 *  - block_table: int32 [rows][max_pages_per_seq]; entries past a request's
 *    last page are never read.
 *
 * Supported geometry:
 *  - Every call: num_q_heads = 16, num_kv_heads = 8, head_dim = 128,
 *    page_size = 16 (the Qwen3 decoder; the tuned kernels).
 *  - pkv_append, pkv_decode_attn, pkv_decode_append_attn,
 *    pkv_decode_append_rope_attn and pkv_prefill_chunk_attn also take
 *    page_size = 16, head_dim 64 or 128,
 *    any num_kv_heads and num_q_heads = G * num_kv_heads with G from 1 to 8
 *    (other decoder backbones; decode runs the same persistent split-KV
 *    kernel with the head counts read at run time, early prefetch included;
 *    prefill runs its tensor-core kernel on pairs of query heads).
 *  - Anything else returns PKV_ERR_UNSUPPORTED.
 *
 * Conventions for every entry point:
 *  - Every pointer argument except `desc` is DEVICE memory owned by the
 *    caller; `desc` is a host pointer read during the call only. The library
 *    never allocates, frees or synchronises, and keeps no state between calls
 *    apart from a per-device cache of the SM count. The one exception is
 *    pkv_decode_attn_noalloc, which owns a fixed device array per GPU and has
 *    no status word the caller can read (see its own block).
 *  - Work is enqueued on `stream` (NULL = the legacy default stream) and is
 *    ordered with the caller's other work on that stream. No call reads
 *    device memory from the host, so the calls can be captured in a CUDA graph.
 *  - Return value: PKV_OK, or a negative PKV_ERR_* code when the arguments are
 *    rejected on the host (nothing is launched) or the launch fails.
 *  - Errors found on the device (a page id outside the pool, a length beyond
 *    the block table, a wait that ran out of time) are written to the status
 *    word at the start of the workspace; the first error wins. The kernel
 *    skips the offending access and stays within the caller's buffers.
 *    Read the word with pkv_read_status().
 *  - A workspace must be zero-filled once before its first use
 *    (pkv_workspace_init); the kernels leave it ready for the next call. Calls
 *    that may run concurrently (different streams) need separate workspaces.
 *  - After any call whose status word is not PKV_OK, run pkv_workspace_init on
 *    the workspace again before its next use. A call that stopped early (a
 *    bounded wait that ran out, a skipped access) may leave split counters
 *    above zero or tagged partial records behind, and the next call would
 *    take them for its own.
 *  - Split merge of decode batches: the CTA that merges a (request, KV head)
 *    waits, with a bound, for the partial records of CTAs with lower block
 *    indices. This relies on the hardware starting a grid's CTAs in
 *    block-index order, which NVIDIA GPUs do but CUDA does not promise. Were
 *    it not so, the wait would run out after about one second and report
 *    PKV_ERR_DEVICE_TIMEOUT; it never hangs.
 *  - A workspace serves one kind of attention call: decode calls
 *    (pkv_decode_attn, pkv_decode_append_attn) or prefill calls
 *    (pkv_prefill_chunk_attn), not both: each kind relies on its own split
 *    scratch (counters, and for decode tagged records) having been left
 *    cleared by the previous call of that kind. pkv_append uses only the
 *    status word and may share either.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st* pkv_stream_t;

typedef struct pkv_cache_desc {
  int32_t num_q_heads;  /* query heads (16; see "Supported geometry") */
  int32_t num_kv_heads; /* KV heads (8) */
  int32_t head_dim;     /* 128 (or 64) */
  int32_t page_size;    /* tokens per page (16) */
  int32_t num_pages;    /* pages in each of k_pages / v_pages */
} pkv_cache_desc;

enum {
  PKV_OK = 0,
  PKV_ERR_NULL_ARG = -1,            /* a required pointer is NULL */
  PKV_ERR_BAD_SHAPE = -2,           /* a size is negative, zero where it may not be, or inconsistent */
  PKV_ERR_UNSUPPORTED = -3,         /* geometry the call does not serve, or no sm_103 device */
  PKV_ERR_WORKSPACE_TOO_SMALL = -4, /* workspace_bytes below the matching *_workspace_bytes() */
  PKV_ERR_CUDA = -5,                /* a CUDA runtime call or the launch failed */
  PKV_ERR_DEVICE_TIMEOUT = -6,      /* device: a bounded wait for a copy ran out (status word only) */
  PKV_ERR_OUT_OF_BOUNDS = -7,       /* device: page id, slot or length outside the pool/table (status word only) */
  PKV_ERR_MISALIGNED = -8           /* a buffer is not 16-byte aligned */
};

/* Bytes of the status header at the start of every workspace. */
#define PKV_STATUS_BYTES 256

/* Zero a workspace (cudaMemsetAsync on `stream`). Call once after allocating it. */
int pkv_workspace_init(void* workspace, size_t workspace_bytes, pkv_stream_t stream);

/*
 * Read the status word of a workspace: waits for `stream`, then copies the
 * word to the host. For tests and debugging only (it synchronises).
 * Returns the device status (PKV_OK or a PKV_ERR_* code), or PKV_ERR_CUDA.
 */
int pkv_read_status(const void* workspace, pkv_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* pkv_status_string(int status);

/*
 * pkv_append -- write the key and value rows of new tokens into their slots.
 *
 * Source: the KV cache grows by one row per generated token and by a chunk of
 * rows per prefill chunk ("FunASR vLLM Inference Engine Guide", section 2:
 * PagedAttention with on-demand allocation; "Optimizing ASR for 90-minute
 * multi-speaker audio", section "LLM prefill").
 *
 *  k_new, v_new:  bf16 [n_tokens][num_kv_heads][head_dim], 16-byte aligned.
 *  slot_mapping:  int32 [n_tokens]; token t goes to slot slot_mapping[t];
 *                 a negative slot skips the token; a slot >= num_pages *
 *                 page_size sets PKV_ERR_OUT_OF_BOUNDS and is skipped.
 *  n_tokens:      >= 0 (0 launches nothing).
 *  k_pages, v_pages: the pools, updated in place. Bit-exact copy.
 *  workspace:     may be NULL (device errors then go unreported); otherwise
 *                 at least PKV_STATUS_BYTES.
 */
int pkv_append(const void* k_new, const void* v_new, const int32_t* slot_mapping, int32_t n_tokens,
               void* k_pages, void* v_pages, const pkv_cache_desc* desc, pkv_stream_t stream,
               void* workspace, size_t workspace_bytes);

/*
 * Workspace bytes pkv_decode_attn needs for `batch` requests on the current
 * device: the status header, one counter per (request, KV head), and the
 * split-KV partial records (two areas of two 1056-byte records per CTA of the
 * launch grid, one per merge scheme). Returns 0 for unsupported arguments.
 */
size_t pkv_decode_workspace_bytes(const pkv_cache_desc* desc, int32_t batch, int32_t max_pages_per_seq);

/*
 * pkv_decode_attn -- decode attention over the paged KV cache.
 *
 * Source: PagedAttention decoding ("FunASR vLLM Inference Engine Guide",
 * section 2); decode dominates long-audio serving ("Optimizing ASR for
 * 90-minute multi-speaker audio", section "Time spent: profiling").
 *
 * For every request b and query head h:
 *   out[b][h] = sum_j softmax_j(scale * <q[b][h], k_j>) v_j,  j < seq_lens[b],
 * with k_j, v_j the rows of KV head h / (num_q_heads / num_kv_heads) at
 * logical position j. seq_lens counts the token appended this step (append
 * first). A request with seq_lens[b] == 0 (a padding row of a graph bucket)
 * gets an all-zero output row. Inputs bf16, fp32 accumulation, bf16 output.
 * The split of long contexts over CTAs and the merge of the partial results
 * happen inside the call; the result does not depend on page placement.
 *
 *  q:            bf16 [batch][num_q_heads][head_dim]
 *  k_pages, v_pages: bf16 pools (see layout above), 16-byte aligned
 *  block_table:  int32 [batch][max_pages_per_seq]
 *  seq_lens:     int32 [batch], 0 <= seq_lens[b] <= max_pages_per_seq * page_size
 *                (larger values are clamped and set PKV_ERR_OUT_OF_BOUNDS)
 *  out:          bf16 [batch][num_q_heads][head_dim]
 *  scale:        softmax scale (1/sqrt(head_dim) for the Qwen3 decoder)
 *  batch:        >= 0 (0 launches nothing), max_pages_per_seq >= 1;
 *                batch * max_pages_per_seq * max(num_kv_heads, 8) < 2^31
 *                (PKV_ERR_BAD_SHAPE beyond; the same for the fused calls)
 *  workspace:    >= pkv_decode_workspace_bytes(desc, batch, max_pages_per_seq)
 */
int pkv_decode_attn(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
                    const int32_t* seq_lens, void* out, float scale, pkv_stream_t stream,
                    const pkv_cache_desc* desc, int32_t batch, int32_t max_pages_per_seq, void* workspace,
                    size_t workspace_bytes);

/*
 * pkv_decode_append_attn -- one decode step of one layer: KV append fused into
 * decode attention (one launch instead of pkv_append + pkv_decode_attn).
 *
 * Source: each generated token adds one K/V row per layer to the paged cache
 * and then attends over the whole cache ("FunASR vLLM Inference Engine Guide",
 * section 2; "Optimizing ASR for 90-minute multi-speaker audio", section
 * "Autoregressive decoding").
 *
 * For every request b with seq_lens[b] > 0, the rows k_new[b][g][:] and
 * v_new[b][g][:] of every KV head g are written at logical position
 * seq_lens[b] - 1 (page block_table[b][(seq_lens[b]-1) / page_size], slot
 * (seq_lens[b]-1) % page_size), bit-exactly; then out is computed exactly as
 * by pkv_decode_attn over seq_lens[b] positions, the new one included. The
 * result equals pkv_append with slot_mapping[b] = that slot followed by
 * pkv_decode_attn.
 *
 *  k_new, v_new: bf16 [batch][num_kv_heads][head_dim], 16-byte aligned
 *  k_pages, v_pages: the pools, updated in place at the new slots only
 *  flags:        0 or PKV_DECODE_EARLY_PREFETCH (see below); other bits are
 *                rejected with PKV_ERR_UNSUPPORTED
 *  other arguments and the workspace: as for pkv_decode_attn
 */
int pkv_decode_append_attn(const void* q, const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                           const int32_t* block_table, const int32_t* seq_lens, void* out, float scale,
                           pkv_stream_t stream, const pkv_cache_desc* desc, int32_t batch, int32_t max_pages_per_seq,
                           void* workspace, size_t workspace_bytes, uint32_t flags);

/*
 * Flag for pkv_decode_append_attn. Every kernel of the library is launched
 * with programmatic stream serialisation and normally waits for the previous
 * kernel in the stream before it reads any argument. With this flag the
 * caller promises that the previous kernel writes neither k_pages / v_pages
 * nor block_table nor seq_lens (the usual case in a decode step, where the
 * previous kernel produces q, k_new and v_new): the call then reads those
 * while that kernel is still finishing and starts copying pages into shared
 * memory, and waits for it only before it reads q / k_new / v_new or writes
 * anything. Pass 0 when the promise does not hold (for example right after
 * pkv_append or a prefill chunk that wrote the same pool).
 */
#define PKV_DECODE_EARLY_PREFETCH 1u

/*
 * pkv_decode_append_rope_attn -- pkv_decode_append_attn with the rotary
 * position embedding of the new token applied on the way: one launch for the
 * step that precedes decode attention in a RoPE decoder and the attention.
 *
 * Source: the decoder is a Qwen3-style causal LM with RoPE theta 1e6
 * ("Fun-ASR-Nano Native Runtime Design", section "Decoder And Prompt"). The
 * pages name RoPE and theta only; the rotate-half form of Qwen3 decoders is
 * taken: dims i and i + head_dim/2 form a pair rotated by the angle of
 * (position, i).
 *
 * For every request b with seq_lens[b] > 0, at position p = seq_lens[b] - 1,
 * with c = rope_cos_sin[p][i] and s = rope_cos_sin[p][head_dim/2 + i]:
 *  - the key row written is k_new[b][g] rotated and rounded to bf16 (ties to
 *    even), each pair (x1, x2) = (k[i], k[i + head_dim/2]) evaluated in fp32
 *    as y1 = fmaf(x1, c, -(x2 * s)), y2 = fmaf(x2, c, x1 * s), each product
 *    rounded to fp32 first (so the written bits are defined exactly);
 *  - every query row q[b][h] is rotated the same way in fp32, then rounded to
 *    bf16 (ties to even), the operand precision of the score product;
 *  - v_new is written unchanged; everything else is as pkv_decode_append_attn.
 *
 *  rope_cos_sin: fp32 [rope_max_pos][head_dim], row p = cos(p w_i) for
 *                i < head_dim/2, then sin(p w_i) (w_i = theta^(-2i/head_dim));
 *                caller-owned device memory, 16-byte aligned, read only
 *                (pkv_rope_table builds it).
 *                A position >= rope_max_pos is reported as
 *                PKV_ERR_OUT_OF_BOUNDS in the status word and clamped to the
 *                last row.
 *  rope_max_pos: rows of the table (>= 1)
 *  other arguments, flags and the workspace: as for pkv_decode_append_attn
 */
int pkv_decode_append_rope_attn(const void* q, const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                                const int32_t* block_table, const int32_t* seq_lens, const float* rope_cos_sin,
                                int32_t rope_max_pos, void* out, float scale, pkv_stream_t stream,
                                const pkv_cache_desc* desc, int32_t batch, int32_t max_pages_per_seq, void* workspace,
                                size_t workspace_bytes, uint32_t flags);

/*
 * pkv_rope_table -- build the cos/sin table the RoPE decode call reads.
 *
 * Source: the decoder's rotary position embedding with theta 1e6
 * ("Fun-ASR-Nano Native Runtime Design", section "Decoder And Prompt"), in the
 * rotate-half form of Qwen3 decoders (the pages name RoPE and theta only).
 *
 * Writes table[p][i] = cos(p w_i) and table[p][head_dim/2 + i] = sin(p w_i)
 * for p < max_pos, i < head_dim/2, w_i = theta^(-2i / head_dim); each angle
 * and its cosine and sine are evaluated in double and rounded to float once.
 *
 *  table:     fp32 [max_pos][head_dim], caller-owned device memory, 16-byte
 *             aligned, written on `stream`
 *  max_pos:   >= 1 rows (positions 0 .. max_pos - 1)
 *  head_dim:  even, 2 .. 1024 (the decode calls use 64 or 128)
 *  theta:     > 0 (1e6 for the Qwen3 decoder)
 * Returns PKV_ERR_BAD_SHAPE for other sizes, PKV_ERR_MISALIGNED for an
 * unaligned table; nothing is written then.
 */
int pkv_rope_table(float* table, int32_t max_pos, int32_t head_dim, double theta, pkv_stream_t stream);

/*
 * Workspace bytes pkv_prefill_chunk_attn needs: the status header, split
 * counters (num_seqs x head pairs x ceil(max_q_len / 128) x 2 ints, with
 * num_kv_heads x ceil(G / 2) head pairs) and two partial records per SM of the
 * current device (for each of the 2 query heads of a pair: 128 rows x
 * head_dim dims of fp16 O / l, then fp32 max and sum per row: 67,584 bytes at
 * head_dim 128), for query tiles whose key range is cut between CTAs.
 */
size_t pkv_prefill_workspace_bytes(const pkv_cache_desc* desc, int32_t num_seqs, int32_t max_q_len);

/*
 * pkv_prefill_chunk_attn -- causal attention of prefill chunks over the cache.
 *
 * Source: "Optimizing ASR for 90-minute multi-speaker audio", section
 * "Chunked prefill for long audio": a long prompt is prefilled in 4096-token
 * chunks, one per scheduler step, between other requests' decode steps.
 *
 * Request n owns query rows cu_q_lens[n] .. cu_q_lens[n+1]-1 of q; its chunk
 * follows prefix_lens[n] cached tokens, and row i of the chunk (absolute
 * position prefix_lens[n] + i) attends keys 0 .. prefix_lens[n] + i of the
 * request (bottom-right causal alignment). The chunk's own K/V rows must
 * already be in the pool (pkv_append first). bf16 inputs, fp32 accumulation on
 * the tensor cores, the softmax weights rounded to bf16 before they multiply
 * V, bf16 output.
 *
 *  q, out:       bf16 [total_q][num_q_heads][head_dim]
 *  block_table:  int32 [num_seqs][max_pages_per_seq]
 *  prefix_lens:  int32 [num_seqs]
 *  cu_q_lens:    int32 [num_seqs + 1], cu_q_lens[0] = 0, non-decreasing,
 *                cu_q_lens[num_seqs] <= total_q
 *  total_q:      rows of q and out (host value; bounds every access)
 *  max_q_len:    host-side upper bound on any chunk length (sizes the grid
 *                and the workspace). A chunk longer than
 *                128 * ceil(max_q_len / 128) rows sets PKV_ERR_OUT_OF_BOUNDS
 *                in the status word; its rows past that bound are not
 *                computed.
 *  workspace:    >= pkv_prefill_workspace_bytes(...), zeroed once by
 *                pkv_workspace_init (the call leaves its counters at zero)
 * Limits: num_pages * num_kv_heads * page_size < 2^31 rows per pool;
 * num_seqs <= 1024 (PKV_ERR_UNSUPPORTED beyond).
 */
int pkv_prefill_chunk_attn(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
                           const int32_t* prefix_lens, const int32_t* cu_q_lens, int32_t num_seqs, int32_t total_q,
                           void* out, float scale, pkv_stream_t stream, const pkv_cache_desc* desc,
                           int32_t max_pages_per_seq, int32_t max_q_len, void* workspace, size_t workspace_bytes);

/*
 * Workspace bytes pkv_mixed_step_attn needs: the prefill workspace of the
 * chunk part (see pkv_prefill_workspace_bytes), then one counter per (decode
 * request, KV head) and, where a decode context spans more than 64 pages,
 * partial records of its 64-page chunks (1056 bytes each). Returns 0 for
 * unsupported arguments.
 */
size_t pkv_mixed_workspace_bytes(const pkv_cache_desc* desc, int32_t num_seqs, int32_t max_q_len, int32_t dec_batch,
                                 int32_t dec_max_pages_per_seq);

/*
 * pkv_mixed_step_attn -- one scheduler step that interleaves chunked prefill
 * with decode: the attention of prefill chunks and of decode requests over
 * the same paged cache, in one launch.
 *
 * Source: a long prompt is prefilled in 4096-token chunks, one per scheduler
 * step, between other requests' decode steps ("Optimizing ASR for 90-minute
 * multi-speaker audio", section "Chunked prefill for long audio"); running
 * the chunk and the decode batch as one kernel is the step the same page's
 * section "后续计划" (future work) leaves open with CUDA-graph capture of
 * chunked prefill.
 *
 * Computes exactly what pkv_prefill_chunk_attn computes for the chunk
 * arguments (q .. max_q_len) and what pkv_decode_attn computes for the decode
 * arguments (dec_*), both over k_pages / v_pages; results are within the same
 * tolerance as those calls but not bit-identical to them (the work is split
 * differently). All K/V rows, the chunks' and the decode tokens', must already
 * be in the pools (pkv_append first). The decode requests run in CTAs of their
 * own, one per chunk of up to 64 pages of a (request, KV head), that the
 * hardware starts on the SMs the chunk leaves free (the tail of a short chunk;
 * for a long cached prefix the chunk's persistent schedule keeps a few SMs for
 * them, in proportion to their pages); chunks of one context are merged by
 * log-sum-exp.
 *
 *  chunk arguments: as for pkv_prefill_chunk_attn; num_seqs = 0 (or total_q =
 *                   0, max_q_len = 0) means no chunk, and q, out, block_table,
 *                   prefix_lens and cu_q_lens may then be NULL
 *  dec_q, dec_out:  bf16 [dec_batch][16][128], 16-byte aligned
 *  dec_block_table: int32 [dec_batch][dec_max_pages_per_seq]
 *  dec_seq_lens:    int32 [dec_batch]; 0 gives an all-zero output row; larger
 *                   than dec_max_pages_per_seq * 16 is clamped and set
 *                   PKV_ERR_OUT_OF_BOUNDS
 *  dec_batch:       0 .. 1024 (0: the call is pkv_prefill_chunk_attn)
 *  workspace:       >= pkv_mixed_workspace_bytes(desc, num_seqs, max_q_len,
 *                   dec_batch, dec_max_pages_per_seq), zeroed once by
 *                   pkv_workspace_init (the call leaves its counters at zero);
 *                   serves mixed-step calls only
 * Geometry: 16 query / 8 KV heads, head_dim 128, page 16 (PKV_ERR_UNSUPPORTED
 * otherwise).
 */
int pkv_mixed_step_attn(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
                        const int32_t* prefix_lens, const int32_t* cu_q_lens, int32_t num_seqs, int32_t total_q,
                        void* out, int32_t max_pages_per_seq, int32_t max_q_len, const void* dec_q,
                        const int32_t* dec_block_table, const int32_t* dec_seq_lens, void* dec_out, int32_t dec_batch,
                        int32_t dec_max_pages_per_seq, float scale, pkv_stream_t stream, const pkv_cache_desc* desc,
                        void* workspace, size_t workspace_bytes);

/*
 * pkv_decode_attn_noalloc -- pkv_decode_attn without a caller-provided workspace.
 *
 * The source pages have no counterpart to this call: it exists for callers
 * that may not allocate device memory where they run decode attention (for
 * example a plug-in inside a host runtime that owns all device memory through
 * its own pool, or a serving loop that reserves memory once at start-up and
 * must not allocate, or implicitly synchronise, afterwards). The caller still
 * passes q, the pools, the block table, the lengths and out, with the same
 * meaning and layout as for pkv_decode_attn; the split-KV scratch comes from a
 * fixed array inside the library instead of a workspace.
 *
 *  - The scratch is one device array of PKV_NOALLOC_SCRATCH_BYTES (2 MiB).
 *    Every GPU that loads the library holds it until the process exits. The
 *    call itself allocates and frees nothing.
 *  - Geometry: 16 query / 8 KV heads, head_dim 128, page size 16 only (the
 *    tuned decode kernel); other geometries return PKV_ERR_UNSUPPORTED.
 *  - Limit: batch <= PKV_NOALLOC_MAX_BATCH (256), and the scratch must cover
 *    the device's split partials (it does for up to ~240 SMs; a GB300 has 152).
 *    Larger requests return PKV_ERR_WORKSPACE_TOO_SMALL without launching.
 *  - The first call on a device, and the first call in each other context
 *    on it, looks up the array's device address (each context loads its own
 *    copy of the array): a one-time set-up; make that first call before any
 *    CUDA-graph capture. The call is not supported after cudaDeviceReset in
 *    the same process: the device's primary context may come back under the
 *    same handle while the array has moved.
 *  - Every call uses the same array and it keeps the previous call's
 *    contents; each call zeroes the status word, the split counters and records on
 *    `stream` before its kernel. Calls whose kernels overlap on the GPU (on
 *    different streams, or in parallel graph branches) race on the array:
 *    issue them in order on one stream.
 *  - Device-side errors are not reported: the status word lives in the
 *    library's array and no call reads it back. A page id outside the pool or
 *    a length beyond the block table is skipped as in pkv_decode_attn. A
 *    bounded wait of the split merge that runs out (see the convention on the
 *    split merge above) leaves the output rows of the affected (request, KV
 *    head) unwritten: `out` keeps whatever it held there, with no signal.
 *    Callers that need to see such errors use pkv_decode_attn.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (2u << 20)
#define PKV_NOALLOC_MAX_BATCH 256

int pkv_decode_attn_noalloc(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
                            const int32_t* seq_lens, void* out, float scale, pkv_stream_t stream,
                            const pkv_cache_desc* desc, int32_t batch, int32_t max_pages_per_seq);

/*
 * pkv_selftest_wait_timeout -- diagnostic of the bounded device waits.
 *
 * Not a step of the attention path (the pages have no counterpart): it runs
 * one CTA that waits, through the same bounded-wait helper the kernels use,
 * on a shared-memory barrier that nothing ever completes, for at most
 * limit_cycles SM clock cycles (<= 2^32), and then writes
 * PKV_ERR_DEVICE_TIMEOUT into the workspace status word. Shows that a wait
 * which runs out ends the kernel with an error the host can read
 * (pkv_read_status) and leaves the context usable.
 */
int pkv_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int64_t limit_cycles, pkv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
