/*
 * libfattn -- exact tiled attention, paged attention and the fused KV-cache
 * append for one NVIDIA GB300 GPU (sm_103a).
 *
 * The operations follow "Fast Attention Kernels and Operator Fusion":
 *   - section "FlashAttention-Style Kernels", attention equation
 *       Attention(Q, K, V) = softmax(Q K^T / sqrt(d) + M) V,
 *     computed tile by tile with running softmax statistics so the T x T score
 *     matrix never reaches device memory (same section, the paragraph on
 *     processing queries, keys and values in tiles);
 *   - section "Paged Attention Kernels": keys and values stored in fixed
 *     16-token blocks, a per-sequence block table translating logical block
 *     numbers to physical ones (the section's example maps logical blocks
 *     0 1 2 3 to physical 17 4 29 8), and a kernel that reads every key and
 *     value through that table;
 *   - section "Operator Fusion", fusion list item on updating the KV cache
 *     while transforming key and value tensors (the fused append).
 *
 * Conventions shared by every call
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise.  The
 *     caller owns all buffers, including workspaces; the library allocates no
 *     device memory in any call.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream); they do
 *     not synchronise the host.  Errors found on the device (a block-table
 *     entry outside the pool, a slot outside the cache, an inconsistent length,
 *     a bounded wait that expired) are recorded in a per-device error word and
 *     read with fa_get_error().
 *   - bf16 tensors are IEEE bfloat16 stored as 16-bit words.  Accumulation is
 *     fp32; outputs are bf16 rounded to nearest even.
 *   - Grouped-query attention: query head h reads kv head h / (Hq / Hkv).
 *   - Causal masking with Tq <= Tk is bottom-right aligned: query i sits at
 *     position i + Tk - Tq and sees keys j <= i + Tk - Tq.
 *   - A query row that sees no key at all produces output 0 and LSE -inf.
 *   - Supported: head dim d in {64, 128}; block_size 16; Hq % Hkv == 0;
 *     sm_103a devices.  Anything else returns FA_ERR_UNSUPPORTED before any
 *     launch; malformed arguments return FA_ERR_INVALID_ARG.  No call falls
 *     back to the CPU.
 */
#ifndef FATTN_H
#define FATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fa_stream_t; /* same type as cudaStream_t */

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1, /* null pointer, negative size, misaligned buffer */
    FA_ERR_UNSUPPORTED = 2, /* head dim, block size, GQA ratio or device not supported */
    FA_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed */
    FA_ERR_TIMEOUT = 4,     /* a bounded device-side wait expired (read by fa_get_error) */
    FA_ERR_BOUNDS = 5,      /* device-side index check failed (read by fa_get_error) */
    FA_ERR_WORKSPACE = 6,   /* workspace missing or smaller than the size query says */
    FA_ERR_NO_BLOCKS = 7    /* the block pool has no free block left */
} fa_status;

typedef enum { FA_BF16 = 0, FA_F32 = 1 } fa_dtype;

/* Human-readable name of a status code (static storage; never NULL). */
const char* fa_status_string(fa_status status);

/*
 * fa_prefill -- contiguous attention over [B, T, H, d] tensors.
 * Passage: "FlashAttention-Style Kernels" (attention equation with M = 0, or
 * the causal mask when `causal` != 0; tile-by-tile processing).
 *   q   bf16 [B, T, Hq, d] row-major, 16-byte aligned
 *   k,v bf16 [B, T, Hkv, d]
 *   out bf16 [B, T, Hq, d], 32-byte aligned (written; may not alias the inputs)
 *   lse fp32 [B, Hq, T] natural-log log-sum-exp of each row's scores, or NULL
 *   scale multiplies Q K^T (1/sqrt(d) for the textbook form); must be finite
 *         and > 0 (FA_ERR_INVALID_ARG otherwise)
 * Tq = Tk = T.  T may be any positive length (ragged final tile).
 */
fa_status fa_prefill(const void* q, const void* k, const void* v, void* out, int B, int T,
                     int Hq, int Hkv, int d, int causal, float scale, float* lse,
                     fa_stream_t stream);

/*
 * fa_prefill_rows -- fa_prefill for a window of query rows: rows
 * [q0, q0 + Tq) of every sequence against keys [0, Tk) (a chunk of a longer
 * prefill whose keys and values are already in place).
 * Passage: "FlashAttention-Style Kernels" (each query tile is combined with
 * the key tiles it can see; the causal mask keeps key j for query i when
 * j <= i, positions counted from the start of the sequence).
 *   q, k, v, out, B, T, Hq, Hkv, d, causal, scale: as fa_prefill (the buffers
 *       hold whole sequences; only rows [q0, q0 + Tq) of q and out, and rows
 *       [0, Tk) of k and v, are read or written)
 *   q0  a multiple of 128; 0 <= q0, q0 + Tq <= T
 *   Tk  1 <= Tk <= T; with causal != 0, Tk >= q0 + Tq (every key a row can see)
 * The rows written equal, bit for bit, the same rows of fa_prefill over the
 * whole problem when Tk covers them (the same query tiles meet the same key
 * tiles in the same order).  FA_ERR_INVALID_ARG for a window outside those
 * bounds; other errors as fa_prefill.
 */
fa_status fa_prefill_rows(const void* q, const void* k, const void* v, void* out, int B, int T, int Hq,
                          int Hkv, int d, int causal, float scale, int q0, int Tq, int Tk,
                          fa_stream_t stream);

/*
 * fa_prefill_host -- fa_prefill with the inputs and the output in host memory.
 * Passage: "FlashAttention-Style Kernels" (same computation as fa_prefill);
 * the copies are the runtime around it.
 *   q_host, k_host, v_host  bf16 [B, T, Hq|Hkv, d] in host memory (page-locked
 *                           memory lets the copies overlap; pageable works)
 *   out_host                bf16 [B, T, Hq, d] in host memory (written)
 *   q, k, v, out            device buffers of the same shapes, with
 *                           fa_prefill's alignment rules; the caller owns them
 *                           and they are overwritten (q, k, v with the inputs)
 * The key and value rows are copied in first, then the query rows in row
 * chunks (rows [c*R, (c+1)*R) of every sequence, R = max(128, T/4 rounded up
 * to a multiple of 128)) from the last chunk to the first, on a
 * library-owned stream; each chunk's attention runs on `stream` as soon as
 * its query rows are in, and its output is copied out on a second
 * library-owned stream, so copies in both directions overlap the kernels.
 * One launch per chunk.  The output equals fa_prefill's for the whole batch
 * bit for bit.
 * Ordered on `stream` like any other call: it starts after the work already
 * queued there, and work queued after it sees out_host written; the host is
 * not synchronised.  The library-owned streams are per device and shared by
 * every call on it (the enqueue is serialised); while a graph capture holding
 * this call is open, another host thread must not call it on the same device.  No LSE output.  Errors: as fa_prefill, plus
 * FA_ERR_INVALID_ARG for a NULL host pointer; FA_ERR_CUDA if a copy or event
 * call fails while the pipeline is being queued (work queued before the
 * failure still runs).
 */
fa_status fa_prefill_host(const void* q_host, const void* k_host, const void* v_host, void* out_host,
                          void* q, void* k, void* v, void* out, int B, int T, int Hq, int Hkv, int d,
                          int causal, float scale, fa_stream_t stream);

/*
 * fa_prefill_masked -- as fa_prefill plus an additive mask M.
 * Passage: "FlashAttention-Style Kernels", attention equation with additive M.
 *   mask fp32 [T, T] row-major, broadcast over batch and heads; -inf allowed.
 *        Added to the causal mask when `causal` != 0.
 *   ws   device workspace of at least fa_prefill_masked_workspace_size(T)
 *        bytes; holds the per-tile mask classes (all -inf: tile skipped; all
 *        zero: mask not read; each row restricted to one run of keys: the run
 *        applied as a column limit, mask not read; otherwise mask read and
 *        added), the rows' runs and the tile order.  Contents need not be
 *        initialised.
 */
size_t fa_prefill_masked_workspace_size(int T);
fa_status fa_prefill_masked(const void* q, const void* k, const void* v, const float* mask,
                            void* out, int B, int T, int Hq, int Hkv, int d, int causal,
                            float scale, float* lse, void* ws, size_t ws_bytes,
                            fa_stream_t stream);

/*
 * fa_mask_tile_classes -- classes of the 128 x 128 tiles of an additive mask
 * (the first pass of fa_prefill_masked, callable alone).
 * Passage: "FlashAttention-Style Kernels", attention equation with additive M
 * (a tile of M that is -inf everywhere contributes nothing; a tile that is 0
 * everywhere leaves the scores unchanged; a tile of 0 and -inf only, whose
 * zeros form one run in each row, only limits each row to an interval of keys).
 *   mask      fp32 [Tq, Tk] row-major, 16-byte aligned
 *   cls       uint8 [ceil(Tq/128), ceil(Tk/128)] row-major (written): 0 when
 *             every in-range element of the tile is -inf, 1 when every one is
 *             exactly 0 (either sign), 3 when every one is 0 or -inf and the
 *             zeros of each row are one contiguous run (possibly empty), 2
 *             otherwise; edge tiles cover only in-range elements
 *   intervals NULL, or uint8 [ceil(Tq/128), ceil(Tk/128), 128, 2] (written for
 *             class-3 tiles only): row r of the tile has its zeros at tile
 *             columns [lo, hi) (lo = hi = 0 for a row without a zero and for
 *             rows past Tq)
 * One read of M.  Empty masks are a no-op.  FA_ERR_UNSUPPORTED when Tq needs
 * more than 65535 tile rows.
 */
fa_status fa_mask_tile_classes(const float* mask, int Tq, int Tk, uint8_t* cls, uint8_t* intervals,
                               fa_stream_t stream);

/*
 * fa_stage_bf16 -- fp32 -> bf16 conversion, round to nearest even.  Used to
 * stage fp32 q/k/v for the bf16 attention kernels.
 *   src fp32 [n], dst bf16 [n]; both 16-byte aligned.
 */
fa_status fa_stage_bf16(const float* src, void* dst, size_t n, fa_stream_t stream);

/*
 * fa_cache_append -- fused write of new keys and values into the paged cache.
 * Passage: "Operator Fusion", fusion list (updating the KV cache while
 * transforming key and value tensors); "Paged Attention Kernels" (block
 * storage).
 *   k, v         [N, Hkv, d] in `in_dtype` (fp32 inputs are rounded to bf16, RNE)
 *   k_cache, v_cache bf16 [num_blocks, Hkv, 16, d]
 *   slot_mapping int32 [N]: token i goes to slot s = slot_mapping[i], i.e.
 *                block s / 16, offset s % 16.  s < 0 skips the token;
 *                s >= num_blocks * 16 sets FA_ERR_BOUNDS and skips it.
 * Exact: bf16 inputs are copied bit for bit.
 */
fa_status fa_cache_append(const void* k, const void* v, void* k_cache, void* v_cache,
                          const int32_t* slot_mapping, int N, int Hkv, int d, int num_blocks,
                          fa_dtype in_dtype, fa_stream_t stream);

/*
 * fa_cache_append_rope -- the append above fused with rotary position
 * embeddings of queries and keys, in one launch.
 * Passage: "Operator Fusion", fusion list (applying rotary position
 * embeddings to queries and keys; updating the KV cache while transforming
 * key and value tensors).  The pages name this fusion but not the rotation;
 * the reading implemented is the rotate-half form: channel j (j < d/2) pairs
 * with channel j + d/2 and both turn by the angle of table row positions[i]:
 *   y_j = x_j c - x_{j+d/2} s,   y_{j+d/2} = x_{j+d/2} c + x_j s,
 * c = cos_sin[pos][j], s = cos_sin[pos][d/2 + j], computed in fp32 and
 * rounded once to bf16 (RNE).
 *   q            [N, Hq, d] in `in_dtype`; rotated rows go to q_out bf16 [N, Hq, d]
 *   k, v         [N, Hkv, d] in `in_dtype`; k rotated, v unchanged (fp32
 *                values rounded to bf16, RNE), both written to slot
 *                slot_mapping[i] as fa_cache_append places them
 *   positions    int32 [N], 0 <= positions[i] < max_pos (else FA_ERR_BOUNDS is
 *                recorded and token i is skipped entirely)
 *   cos_sin      fp32 [max_pos, d], caller-owned (the angles are the caller's
 *                choice of rotary base and position scaling)
 *   slot_mapping int32 [N], as for fa_cache_append (s < 0: the query is still
 *                rotated, the cache is not written)
 * All pointers 16-byte aligned; d = 64 or 128.
 */
fa_status fa_cache_append_rope(const void* q, const void* k, const void* v, const int32_t* positions,
                               const float* cos_sin, int max_pos, void* q_out, void* k_cache,
                               void* v_cache, const int32_t* slot_mapping, int N, int Hq, int Hkv,
                               int d, int num_blocks, fa_dtype in_dtype, fa_stream_t stream);

/*
 * fa_cache_append_fp8 / fa_paged_attn_fp8 -- the 8-bit (E4M3) KV cache.
 * Passage: page 3, "Key Details" (the fused kernels use the GPU's 16-bit or
 * 8-bit matrix-multiply-accumulate units); the pages fix no format or scale
 * convention.  Reading: E4M3 (1 sign, 4
 * exponent bits, bias 7, 3 mantissa bits, largest finite 448, S.1111.111 NaN),
 * one scale per cache: code = E4M3(x / scale), division in binary32, round to
 * nearest even, saturating at +-448; the cached value is E4M3 * scale.
 *   k_cache uint8 [num_blocks, Hkv, 16, d]   (a token's d codes contiguous)
 *   v_cache uint8 [num_blocks, Hkv, d, 16]   (a channel's 16 tokens contiguous)
 * fa_cache_append_fp8: k, v [N, Hkv, d] in `in_dtype`, slot_mapping as for
 *   fa_cache_append; exact (bit-reproducible codes).  d = 128.
 * fa_paged_attn_fp8: fa_paged_attn over these caches for decode rows only
 *   ((Hq/Hkv) * max_q_len <= 16, else FA_ERR_UNSUPPORTED); the split-KV decode
 *   kernel reads half the bytes of the bf16 cache, converts E4M3 to f16
 *   (exactly) in registers, and computes in f16 MMAs with fp32 accumulation
 *   (queries are converted bf16 -> f16: |q| must stay below 65504); k_scale
 *   is folded into the score scale, v_scale multiplies the output.  Same
 *   workspace as fa_paged_attn.  d = 128; scales finite and > 0.
 */
fa_status fa_cache_append_fp8(const void* k, const void* v, void* k_cache, void* v_cache,
                              const int32_t* slot_mapping, int N, int Hkv, int d, int num_blocks,
                              float k_scale, float v_scale, fa_dtype in_dtype, fa_stream_t stream);
fa_status fa_paged_attn_fp8(const void* q, const void* k_cache, const void* v_cache, float k_scale,
                            float v_scale, const int32_t* block_table, const int32_t* ctx_lens,
                            const int32_t* q_lens, void* out, int num_seqs, int max_blocks_per_seq,
                            int num_blocks, int Hq, int Hkv, int d, int block_size, int causal,
                            float scale, int total_q, int max_q_len, void* ws, size_t ws_bytes,
                            fa_stream_t stream);

/*
 * fa_paged_attn -- attention of packed queries against the paged cache.
 * Passage: "Paged Attention Kernels" (logical positions translated through
 * the block table; 16-token blocks); "FlashAttention-Style Kernels" (the
 * attention it computes; prefill processes many queries, decode one or a few
 * while reading the growing cache).
 *   q            bf16 [total_q, Hq, d], sequences packed in order
 *   k_cache, v_cache bf16 [num_blocks, Hkv, 16, d]
 *   block_table  int32 [num_seqs, max_blocks_per_seq]; entries past
 *                ceil(ctx_lens[s] / 16) are never read
 *   ctx_lens     int32 [num_seqs]: tokens of sequence s in the cache, the new
 *                chunk included (its queries sit at ctx - q_len .. ctx - 1)
 *   q_lens       int32 [num_seqs], 0 <= q_lens[s] <= ctx_lens[s];
 *                sum(q_lens) must equal total_q
 *   out          bf16 [total_q, Hq, d], 32-byte aligned
 *   max_q_len    host-side upper bound on every q_lens[s] (total_q is always
 *                a valid bound); used to skip launching a kernel that would
 *                find no work and to size the decode kernel's partial slots
 *                ((Hq/Hkv) * max_q_len <= 6 rows keeps its deeper ring); a
 *                decode chunk above the bound is reported as FA_ERR_BOUNDS
 *                (fa_get_error) and its rows are not valid
 *   block_size   must be 16
 *   scale        finite and > 0, multiplies Q K^T
 *   ws           workspace of at least fa_paged_attn_workspace_size(...) bytes
 *                (split partials and scheduling lists); contents need not be
 *                initialised
 * Sequences whose (Hq/Hkv) * q_len <= 16 take the bandwidth-bound split-KV
 * decode kernel followed by a log-sum-exp merge; longer chunks take the
 * tensor-core kernel.  Both read K/V only through the block table.  When a
 * call may take both paths (Hq/Hkv <= 16 and max_q_len above the decode
 * size), the tensor-core path's work list is built on a library-owned stream
 * of the device, forked from and joined back to `stream` with events, beside
 * the decode kernel: the call stays ordered on `stream` and capturable, but
 * while a graph capture holding such a call is open, another host thread must
 * not make such a call on the same device (that stream is part of the capture).
 */
size_t fa_paged_attn_workspace_size(int num_seqs, int max_blocks_per_seq, int Hq, int Hkv, int d,
                                    int total_q);
fa_status fa_paged_attn(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_table, const int32_t* ctx_lens,
                        const int32_t* q_lens, void* out, int num_seqs, int max_blocks_per_seq,
                        int num_blocks, int Hq, int Hkv, int d, int block_size, int causal,
                        float scale, int total_q, int max_q_len, void* ws, size_t ws_bytes,
                        fa_stream_t stream);

/*
 * fa_paged_attn_noalloc -- fa_paged_attn for callers that cannot allocate
 * device memory.  The pages have no counterpart: this is a convenience of the
 * library, not part of the method.
 *
 * Some callers cannot call cudaMalloc: a process whose device memory was
 * reserved up front by another runtime's pool (a fresh allocation would fail
 * or fragment that pool), or a plugin interface that hands over inputs and
 * outputs but no scratch space.  This entry point takes the same arguments as
 * fa_paged_attn minus the workspace and uses instead a fixed scratch array of
 * FA_NOALLOC_SCRATCH_BYTES (32 MiB) that the library keeps on every GPU that
 * loads it, until the process exits.  It calls no allocator.
 *   - Problems whose fa_paged_attn_workspace_size(...) exceeds
 *     FA_NOALLOC_SCRATCH_BYTES are rejected with FA_ERR_WORKSPACE before any
 *     launch (the scheduling lists grow with num_seqs and total_q; decode
 *     partials take a fixed ~21 MB).
 *   - The first call on a device looks up the scratch array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.
 *   - Every call on a device shares the one array, which keeps the last call's
 *     contents.  Nothing in it has to start at zero: each call writes what it
 *     later reads.  Calls that overlap on the GPU (different streams, or
 *     different host threads without ordering) race on it and must not be
 *     issued.
 * Everything else -- arguments, layouts, results, errors -- is as for
 * fa_paged_attn.
 */
#define FA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
fa_status fa_paged_attn_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_table, const int32_t* ctx_lens,
                                const int32_t* q_lens, void* out, int num_seqs,
                                int max_blocks_per_seq, int num_blocks, int Hq, int Hkv, int d,
                                int block_size, int causal, float scale, int total_q,
                                int max_q_len, fa_stream_t stream);

/*
 * fa_pool_* -- host-side pool of cache blocks with prefix sharing.
 * Passage: "Paged Attention Kernels" (a logical sequence is a block table;
 * blocks are allocated on demand, returned to a pool when a request ends,
 * and shared when sequences have a common prefix).
 * Bookkeeping only (no device memory is touched; all arrays are host
 * memory).  Blocks are ids 0 .. num_blocks-1 of the caches fa_cache_append
 * writes; every block has a reference count, and a block shared by several
 * sequences is always full, so it is never written again.
 *   _create      pool of num_blocks blocks; tables are max_blocks_per_seq wide
 *   _add_seq     new empty sequence, id in *seq
 *   _fork        new sequence *child holding the first prefix_len tokens of
 *                `parent` (0 <= prefix_len <= parent's length): the full blocks
 *                of the prefix are shared; when prefix_len % 16 != 0 the block
 *                with the prefix tail is copied on write -- the child gets a
 *                fresh block and (*copy_src, *copy_dst) name the copy the caller
 *                must run (fa_copy_blocks) before writing to the child; else
 *                both are -1
 *   _append      slots for n new tokens of `seq` (slots[i] = block * 16 +
 *                offset, for fa_cache_append), taking blocks from the free
 *                list as needed; all or nothing
 *   _release     ends a sequence; its blocks' counts drop and blocks reaching
 *                0 return to the free list; the id may be reused
 *   _tables      block-table rows [n, max_blocks_per_seq] (unused entries -1,
 *                never read by the kernels) and lengths of n sequences
 *   _num_free, _refcount, _seq_len  queries (-1 on a bad argument)
 * Errors: FA_ERR_INVALID_ARG (bad id, length beyond max_blocks_per_seq * 16,
 * null pointer), FA_ERR_NO_BLOCKS (no free block; the pool is unchanged; also
 * host memory for the pool itself).  A pool is thread-safe.
 */
typedef struct fa_block_pool fa_block_pool;
fa_status fa_pool_create(fa_block_pool** pool, int num_blocks, int max_blocks_per_seq);
void fa_pool_destroy(fa_block_pool* pool);
fa_status fa_pool_add_seq(fa_block_pool* pool, int* seq);
fa_status fa_pool_fork(fa_block_pool* pool, int parent, int prefix_len, int* child, int* copy_src,
                       int* copy_dst);
fa_status fa_pool_append(fa_block_pool* pool, int seq, int n, int32_t* slots);
fa_status fa_pool_release(fa_block_pool* pool, int seq);
fa_status fa_pool_tables(const fa_block_pool* pool, const int* seqs, int n, int32_t* table,
                         int32_t* ctx_lens);
int fa_pool_num_free(const fa_block_pool* pool);
int fa_pool_refcount(const fa_block_pool* pool, int block);
int fa_pool_seq_len(const fa_block_pool* pool, int seq);

/*
 * fa_copy_blocks -- device side of the pool's copy on write: for each of the
 * n pairs (device int32 [n, 2]) copies block pairs[i][0] onto pairs[i][1] in
 * both caches (bf16 [num_blocks, Hkv, 16, d], 16-byte aligned).  A block id
 * outside [0, num_blocks) records FA_ERR_BOUNDS and that pair is skipped.
 * Exact (bit copy).
 */
fa_status fa_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int n, int Hkv, int d,
                         int num_blocks, fa_stream_t stream);

/*
 * fa_decode_graph_* -- a decode step recorded once as a CUDA graph and
 * replayed with one submission.
 * Passage: "Fusion and CUDA Graphs with torch.compile" (a CUDA Graph records
 * the sequence of GPU operations and replays it with one CPU submission,
 * reducing launch overhead; replay requires stable memory addresses and
 * compatible shapes; most useful for repeated small-batch work such as
 * decode).
 * _create captures fa_cache_append (skipped when n_new == 0) followed by
 * fa_paged_attn with exactly these arguments on a private stream and
 * instantiates the graph; nothing runs.  Every pointer and size is fixed from
 * then on: between replays the caller rewrites buffer contents only (new
 * rows, slot mapping, block table, context lengths, which the kernels read on
 * the device); a change of any size needs a new graph.  Argument meaning,
 * layout and errors are those of the two captured calls (their status is
 * returned, and no graph is made); FA_ERR_CUDA if capture or instantiation
 * fails.  Call the two entry points once eagerly on the same device before
 * the first capture: first-use setup inside the library is not capturable.
 * _launch replays on `stream` (asynchronous; fa_get_error reports device-side
 * errors as for the eager calls).  _kernel_count is the number of kernels one
 * replay runs.  _destroy frees the graph (NULL is ignored).  The handle is
 * not thread-safe; replays of one handle must not overlap on the GPU.
 */
typedef struct fa_decode_graph fa_decode_graph;
fa_status fa_decode_graph_create(fa_decode_graph** out, const void* k_new, const void* v_new,
                                 const int32_t* slot_mapping, int n_new, fa_dtype in_dtype,
                                 const void* q, void* k_cache, void* v_cache,
                                 const int32_t* block_table, const int32_t* ctx_lens,
                                 const int32_t* q_lens, void* attn_out, int num_seqs,
                                 int max_blocks_per_seq, int num_blocks, int Hq, int Hkv, int d,
                                 int causal, float scale, int total_q, int max_q_len, void* ws,
                                 size_t ws_bytes);
fa_status fa_decode_graph_launch(fa_decode_graph* graph, fa_stream_t stream);
int fa_decode_graph_kernel_count(const fa_decode_graph* graph);
void fa_decode_graph_destroy(fa_decode_graph* graph);

/*
 * fa_get_error -- synchronises `stream`, then returns and clears the current
 * device's error word: FA_OK, FA_ERR_BOUNDS or FA_ERR_TIMEOUT (FA_ERR_BOUNDS
 * when both were recorded), or FA_ERR_CUDA if synchronisation itself failed.
 */
fa_status fa_get_error(fa_stream_t stream);

/*
 * fa_debug_gather_kv -- test hook for the block-table translation alone.
 * Passage: "Paged Attention Kernels" (translate logical positions through
 * the block table).  Writes out[s][t][h][:] = cache[block_table[s][t/16]][h][t%16][:]
 * for t < ctx_lens[s]; positions t >= ctx_lens[s] are left untouched.
 *   cache bf16 [num_blocks, Hkv, 16, d]; out bf16 [num_seqs, max_ctx, Hkv, d]
 */
fa_status fa_debug_gather_kv(const void* cache, const int32_t* block_table,
                             const int32_t* ctx_lens, void* out, int num_seqs,
                             int max_blocks_per_seq, int num_blocks, int Hkv, int d, int max_ctx,
                             fa_stream_t stream);

/*
 * fa_debug_set_wait_limit -- bound, in nanoseconds, on every device-side
 * pipeline wait of later launches (default 4e9).  A wait that runs out sets
 * FA_ERR_TIMEOUT and the kernel exits cleanly.  Host-side setting; not
 * synchronised with launches already queued.
 */
void fa_debug_set_wait_limit(unsigned long long nanoseconds);

/*
 * fa_debug_force_timeout -- test hook for failure detection.  While enabled,
 * every pipelined kernel launched afterwards begins each of its roles with a
 * wait on a barrier that nothing ever arrives on; the wait runs out after the
 * current wait limit, the kernel records FA_ERR_TIMEOUT, drains the copies it
 * issued, releases its tensor memory and exits.  No fault, trap or hang is
 * involved.  Host-side setting.
 */
void fa_debug_force_timeout(int enable);

/* Number of kernels the last successful call on this host thread launched. */
int fa_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* FATTN_H */
