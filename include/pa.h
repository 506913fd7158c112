/*
 * pa.h -- C ABI of the GB300 paged KV-cache decode-attention library (libpa.so).
 *
 * Two operations on a paged KV cache, both asynchronous on a caller stream:
 *
 *   pa_cache_write  append the new token's K/V rows at the slots a block
 *                   manager handed out (optionally quantising them to INT8);
 *   pa_decode       single-token decode attention of every sequence's query
 *                   heads over that sequence's paged K/V history.
 *
 * Sources (web pages; cited by title and section):
 *  [F] "LLM 推理底层：KV Cache 显存几何、GQA/MLA 压缩与 PagedAttention 调度"
 *      (blog.faulkner.fun)
 *  [Q] "【infra之路】10-PagedAttention 与 KV Cache 管理" (qwbw.cn)
 *  [G] "kv-cache-guide" (guijiagi.com)
 *  [T] "KV Cache 显存管理全景：内存碎片拟合推导、vLLM PagedAttention 虚拟内存与
 *      Prefix Caching" (talentme.airsota.com)
 *  [H] "LLM 推理引擎设计：KV Cache、PagedAttention 与连续批处理" (hx.sn.cn)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is a DEVICE pointer (memory the GPU can read or
 *    write), except where a comment says otherwise. Tensors are dense and
 *    row-major in the shapes given. The caller owns every buffer; the library
 *    allocates no device memory and keeps no pointer after a call returns.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). Calls only enqueue work: none of them synchronises the device or
 *    reads device memory from the host.
 *  - Alignment: tensors of bf16 or int8 rows (k, v, q, out, the pools) must
 *    start on a 16-byte boundary, fp32 scales on 16 bytes for pa_decode and
 *    4 bytes for pa_cache_write, slot_mapping on 8 bytes and the decode
 *    workspace on 256 bytes; otherwise PA_ERR_ALIGNMENT.
 *  - Errors the host can see (null pointers, unsupported shapes, a workspace
 *    that is too small, a failed launch) are returned before or at launch and
 *    nothing is enqueued when the return value is not PA_OK.
 *  - Errors only the GPU can see (a block id outside the pool, a slot outside
 *    the pool, a context length the block table cannot hold) never trap or
 *    fault: the kernel skips the offending unit of work and ORs a PA_DEV_* bit
 *    into *dev_status when dev_status is not NULL. Read dev_status after the
 *    stream has finished and turn it into a status with
 *    pa_status_from_device(). What was skipped: a bad slot is not written; a
 *    bad block contributes nothing to its sequence's attention; a bad context
 *    length gives that sequence an all-zero output.
 *
 * Pool layout (the block layout [num_blocks, H, block_size, D] that [G] §7.1
 * gives for PagedAttention):
 *   k_cache, v_cache : [num_blocks][n_kv][block_size][d_h]  bf16 or int8 codes
 *                      [num_blocks][n_kv][block_size][d_h/2] bytes for INT4
 *   k_scale, v_scale : [num_blocks][n_kv][block_size]       fp32 (INT8, INT4)
 * so the 16 rows of one (block, kv head) pair are one contiguous tile.
 * Token j of a sequence lives in physical block block_table[j / block_size] at
 * offset j % block_size ([F] "逻辑块与物理块映射"); its slot is
 * phys * block_size + offset.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. PA_OK is zero; every error is negative. */
typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_NULL = -1,        /* a required pointer is NULL */
    PA_ERR_SHAPE = -2,       /* a size is out of range (n_h % n_kv != 0, count <= 0, ...) */
    PA_ERR_DTYPE = -3,       /* kv_dtype is not a pa_kv_dtype value */
    PA_ERR_UNSUPPORTED = -4, /* a valid but unsupported geometry (d_h, block_size, group size) */
    PA_ERR_BAD_BLOCK = -5,   /* device: a block table entry outside [0, num_blocks) */
    PA_ERR_BAD_SLOT = -6,    /* device: a slot >= num_blocks * block_size */
    PA_ERR_WORKSPACE = -7,   /* workspace NULL or smaller than pa_decode_workspace_size() */
    PA_ERR_CUDA = -8,        /* a CUDA runtime or driver call failed */
    PA_ERR_BAD_CONTEXT = -9, /* device: a context length < 0 or > max_blocks_per_seq * block_size */
    PA_ERR_TIMEOUT = -10,    /* device: a pipeline wait gave up after about one second */
    PA_ERR_ALIGNMENT = -11,  /* a pointer lacks the alignment its entry point documents */
    PA_ERR_OUT_OF_BLOCKS = -12, /* allocator: not enough free blocks; nothing was changed */
    PA_ERR_STATE = -13       /* allocator: a table names a block outside the pool or one
                                that no holder references */
} pa_status;

/* Bits the kernels OR into *dev_status. */
#define PA_DEV_BAD_BLOCK 0x1
#define PA_DEV_BAD_SLOT 0x2
#define PA_DEV_BAD_CONTEXT 0x4
#define PA_DEV_TIMEOUT 0x8

/* Element type of the cached K/V. */
typedef enum pa_kv_dtype {
    PA_KV_BF16 = 0, /* bf16 rows, stored as given */
    PA_KV_INT8 = 1, /* int8 codes + one fp32 scale per (token, kv head), [G] §4.2 */
    PA_KV_INT4 = 2  /* int4 codes, two per byte (element 2i in the low nibble of
                       byte i, two's complement), + one fp32 scale per (token,
                       kv head), [G] §4.2 with num_bits = 4 */
} pa_kv_dtype;

/* Attention and pool geometry of one layer.
 *   n_h        query heads per token
 *   n_kv       KV heads per token; n_h % n_kv == 0, and g = n_h / n_kv query
 *              heads share one KV head ([F] table "注意力头架构演进", GQA row);
 *              query head h reads KV head h / g. g = 1 is MHA.
 *   d_h        head dimension: 64 or 128
 *   block_size tokens per physical block: 16 (the vLLM default, [Q] §5)
 *   num_blocks physical blocks in the pool
 *   kv_dtype   a pa_kv_dtype value
 * Supported group sizes g: 1, 2, 4, 8, 16. */
typedef struct pa_geom {
    int64_t num_blocks;
    int32_t n_h;
    int32_t n_kv;
    int32_t d_h;
    int32_t block_size;
    int32_t kv_dtype;
    int32_t reserved; /* must be 0 */
} pa_geom;

/*
 * pa_cache_write -- slot-mapped append of new K/V rows.
 *
 * [T] 第三章 `write_kv` and [F] "逻辑块与物理块映射": the row of token t goes to
 * physical block slot/block_size at offset slot%block_size, for every KV head:
 *     k_cache[s / bs][h][s % bs][:] = k[t][h][:]     (same for v)
 * Only the new rows are written; history stays untouched (the cached K/V of
 * earlier tokens never change, [F] "自回归解码与 KV Cache 的物理来源").
 *
 * INT8 (geom.kv_dtype == PA_KV_INT8), [G] §4.2 `quantize_kv_cache`, per
 * (token, head) row of d_h values, in IEEE fp32:
 *     scale = max_d |x_d| / 127
 *     code  = clamp(round_half_even(x / scale), -128, 127)
 * and scale is stored in k_scale/v_scale[s / bs][h][s % bs]. A row of zeros
 * stores scale 0 and zero codes.
 * INT4 (PA_KV_INT4), the same with num_bits = 4:
 *     scale = max_d |x_d| / 7,  code = clamp(round_half_even(x / scale), -8, 7)
 * packed two per byte as the pa_kv_dtype comment says.
 *
 *   k, v          bf16 [num_tokens][n_kv][d_h]      new rows (read)
 *   slot_mapping  int64 [num_tokens]                 slot of each row; < 0 = skip
 *   num_tokens    >= 0 (0 enqueues nothing)
 *   k_cache, v_cache  pool (written), layout above
 *   k_scale, v_scale  fp32 scales (written, INT8/INT4); must be NULL for PA_KV_BF16
 *   dev_status    optional int32 device word for PA_DEV_BAD_SLOT
 * Duplicate non-negative slots in one call leave the slot's content undefined.
 */
pa_status pa_cache_write(const void *k, const void *v, const int64_t *slot_mapping,
                         int64_t num_tokens, void *k_cache, void *v_cache, float *k_scale,
                         float *v_scale, pa_geom geom, int32_t *dev_status, void *stream);

/*
 * Bytes of device workspace pa_decode needs for num_seqs sequences on the
 * CURRENT device (it depends on the SM count). num_ctas = 0 asks for the
 * library's default grid; a positive value sizes the workspace for
 * pa_decode_ex with that many CTAs. Returns 0 for an invalid geometry.
 */
size_t pa_decode_workspace_size(pa_geom geom, int32_t num_seqs, int32_t num_ctas);

/*
 * Zero a workspace (cudaMemsetAsync on `stream`).
 *
 * Workspace layout: the first round_up(4 * num_seqs * n_kv, 256) bytes are
 * one int32 counter per (sequence, kv head); they must be zero when pa_decode
 * starts, and every pa_decode leaves them zero again when its kernel ends. The
 * rest is scratch for split partial results. So zero a workspace once before
 * its first use, and again before a call whose num_seqs * n_kv is larger than
 * any earlier call's on it.
 */
pa_status pa_decode_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/*
 * pa_decode -- decode attention over the paged KV cache.
 *
 * For every sequence b < num_seqs and query head h < n_h ([F] eq. for o_t in
 * "自回归解码与 KV Cache 的物理来源"; [Q] §3.4 `paged_attention`):
 *     kv   = h / g
 *     s_j  = scale * < q[b][h][:], K_b[j][kv][:] >          for j < ctx_b
 *     out[b][h][:] = sum_j softmax(s)_j * V_b[j][kv][:]
 * where K_b[j] is read through the block table (token j in block
 * block_tables[b][j / bs] at offset j % bs) and ctx_b = context_lens[b]
 * counts the whole history INCLUDING the new token, which the caller appends
 * with pa_cache_write first. INT8 rows are read as code * scale (fp32),
 * [G] §4.2 `dequantize_kv`. The pages use scale = 1 / sqrt(d_h).
 * Accumulation is fp32; the output is rounded to bf16. ctx_b == 0 gives a
 * zero row. Long contexts are split across CTAs and merged with a
 * log-sum-exp reduction, so results do not depend on how the work was split
 * beyond fp32 rounding.
 *
 *   q                bf16 [num_seqs][n_h][d_h]
 *   k_cache, v_cache pool, layout above (read)
 *   k_scale, v_scale fp32 scales for PA_KV_INT8, else NULL
 *   block_tables     int32 [num_seqs][max_blocks_per_seq]; entries past a
 *                    sequence's ceil(ctx/bs) blocks are never read
 *   context_lens     int32 [num_seqs] (device memory; not read by the host)
 *   num_seqs         0..8192 (0 enqueues nothing)
 *   scale            softmax scale applied to q.k
 *   out              bf16 [num_seqs][n_h][d_h] (written)
 *   workspace        >= pa_decode_workspace_size(geom, num_seqs, 0) bytes,
 *                    256-byte aligned, counter area zero on entry (see
 *                    pa_decode_workspace_init). Calls that share a workspace
 *                    must be ordered on one stream.
 *   dev_status       optional int32 device word (PA_DEV_* bits)
 */
pa_status pa_decode(const void *q, const void *k_cache, const void *v_cache,
                    const float *k_scale, const float *v_scale, const int32_t *block_tables,
                    int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                    float scale, void *out, void *workspace, size_t workspace_bytes, pa_geom geom,
                    int32_t *dev_status, void *stream);

/* pa_decode with an explicit CTA count (num_ctas > 0) instead of the
 * library's default of one wave of resident CTAs. Results agree with
 * pa_decode within fp32 rounding; this exists to test split invariance and
 * to tune the split. The workspace must be sized for the same num_ctas. */
pa_status pa_decode_ex(const void *q, const void *k_cache, const void *v_cache,
                       const float *k_scale, const float *v_scale, const int32_t *block_tables,
                       int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                       float scale, void *out, void *workspace, size_t workspace_bytes,
                       pa_geom geom, int32_t *dev_status, void *stream, int32_t num_ctas);

/*
 * Options of pa_decode_opt (zero-initialise, then set what is needed).
 *
 *   window    > 0: sliding-window attention ([G] §5.1 `SlidingWindowKVCache`:
 *             only the latest w tokens are kept and attended). Sequence b
 *             attends positions [max(0, ctx_b - window), ctx_b). Block-table
 *             entries of logical blocks wholly before that start are never
 *             read (a windowed cache may have released them). 0 = attend all.
 *   n_sink    INT8/INT4 pools only, 0..16: attention-sink rows ([G] §4.3: the first
 *             k tokens, typically 4, stay unquantised in an INT8 cache). An
 *             attended position j < n_sink takes its K and V from the bf16
 *             rows sink_k/sink_v[b][kv head][j][:] instead of the pool; the
 *             pool's codes for those positions are not read. 0 = none.
 *   sink_k, sink_v  bf16 [num_seqs][n_kv][n_sink][d_h] (device, read;
 *             2-byte aligned), required when n_sink > 0, else NULL.
 *             pa_sink_write fills them.
 *   num_ctas  > 0: the CTA count as in pa_decode_ex; 0: the default.
 *   share_prefix  1 or 2: sequences whose block tables start with the same
 *             physical blocks (prefix caching, [F] "Prefix Caching 与
 *             Copy-on-Write") have those blocks attended once per group: a
 *             first kernel cuts runs of neighbouring sequences sharing >= 8
 *             leading full blocks into groups (of at most 8 sequences for
 *             g <= 2, 16/g otherwise), neighbours in the batch's order (1:
 *             sharers must be adjacent) or, with 2, in an order by a hash
 *             of each sequence's first 8 table entries (sharers anywhere in
 *             the batch; the sort costs a few microseconds more); a second
 *             kernel attends each group's shared
 *             blocks once with all the group's query rows and, in the same
 *             launch, each sequence's remaining blocks, and the last piece of
 *             a sequence to finish merges the softmax states (log-sum-exp).
 *             The result equals pa_decode's up to rounding. A batch whose
 *             2 * num_seqs units' tables do not fit the kernel's shared
 *             memory (thousands of sequences at d_h 128) is decoded without
 *             sharing, with the same result. Not with a window or sink rows;
 *             g <= 8. The workspace is
 *             pa_decode_opt_workspace_size(geom, num_seqs, opts).
 */
typedef struct pa_decode_opts {
    int32_t window;
    int32_t n_sink;
    const void *sink_k;
    const void *sink_v;
    int32_t num_ctas;
    int32_t share_prefix; /* 1, 2: attend shared prefixes once per group (below) */
    int32_t reserved;     /* must be 0 */
} pa_decode_opts;

/* Workspace bytes pa_decode_opt needs for these options (0 if invalid). */
size_t pa_decode_opt_workspace_size(pa_geom geom, int32_t num_seqs, const pa_decode_opts *opts);

/*
 * The shared-prefix groups of a batch, as pa_decode_opt with share_prefix
 * finds them (its first kernel), written to the caller's device buffers:
 *   skip    int32 [num_seqs]: leading blocks sequence b's group shares, 0 if
 *           b is in no group;
 *   groups  int32 [3 * num_seqs]: for groups s = 0 .. NG-1 (first, members,
 *           shared blocks), then zeros;
 *   order   int32 [num_seqs]: the order the groups are cut in (mode 1: the
 *           batch's own; mode 2: by a hash of each sequence's first 8 table
 *           entries, ties by index); member j of group s is sequence
 *           order[first + j].
 * g is the query heads per kv head (1, 2, 4 or 8): groups hold at most 8
 * sequences for g <= 2, 16/g otherwise. block_tables and context_lens are as
 * for pa_decode; mode is pa_decode_opts.share_prefix (1 or 2).
 * Asynchronous on `stream`; num_seqs == 0 does nothing.
 * Errors: PA_ERR_SHAPE (num_seqs outside 0..8192, max_blocks_per_seq <= 0,
 * another mode),
 * PA_ERR_UNSUPPORTED (other g), PA_ERR_NULL, PA_ERR_CUDA. The pages have no
 * counterpart: it exposes the grouping the shared-prefix decode uses.
 */
pa_status pa_share_groups(const int32_t *block_tables, int32_t max_blocks_per_seq,
                          const int32_t *context_lens, int32_t num_seqs, int32_t g,
                          int32_t mode, int32_t *skip, int32_t *groups, int32_t *order,
                          void *stream);

/* pa_decode with options (opts may be NULL: plain pa_decode). Extra
 * errors: PA_ERR_SHAPE for window < 0, n_sink outside 0..16, n_sink > 0 on
 * a bf16 pool, num_ctas < 0 or reserved != 0; PA_ERR_NULL for missing sink
 * rows; PA_ERR_ALIGNMENT for odd sink pointers. The workspace is sized as
 * for pa_decode_ex with the same num_ctas (0: pa_decode's size). */
pa_status pa_decode_opt(const void *q, const void *k_cache, const void *v_cache,
                        const float *k_scale, const float *v_scale, const int32_t *block_tables,
                        int32_t max_blocks_per_seq, const int32_t *context_lens,
                        int32_t num_seqs, float scale, void *out, void *workspace,
                        size_t workspace_bytes, pa_geom geom, const pa_decode_opts *opts,
                        int32_t *dev_status, void *stream);

/*
 * pa_decode_mq -- multi-query decode: n_q new tokens per sequence attend in
 * one pass, as when a target model verifies a k-token draft ([H] §6
 * "投机解码": the large model checks the draft tokens in one parallel
 * forward) or processes one chunk of a chunked prefill ([F] "Chunked
 * Prefill"). The n_q tokens of sequence b are its last n_q positions
 * ctx_b - n_q .. ctx_b - 1 (their K/V already written with pa_cache_write);
 * new token i attends causally to positions 0 .. ctx_b - n_q + i. A token
 * whose range is empty (ctx_b < n_q - i) gets a zero output.
 *
 *   q    bf16 [num_seqs][n_q][n_h][d_h]; out the same shape
 *   n_q  1 (pa_decode), or 2, 4, 8 with g * n_q <= 16, on bf16, INT8 and
 *        INT4 pools (PA_ERR_UNSUPPORTED otherwise)
 * Every other argument is pa_decode's (k_scale/v_scale for INT8/INT4 pools). All n_q * g query rows of a kv head
 * read each K/V tile once: the bytes moved are those of one decode step.
 * The workspace is pa_decode_mq_workspace_size(geom, num_seqs, n_q, 0).
 */
pa_status pa_decode_mq(const void *q, const void *k_cache, const void *v_cache,
                       const float *k_scale, const float *v_scale, const int32_t *block_tables,
                       int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                       int32_t n_q, float scale, void *out, void *workspace,
                       size_t workspace_bytes, pa_geom geom, int32_t *dev_status, void *stream);

/* pa_decode_mq with the work split over exactly num_ctas CTAs (> 0), as
 * pa_decode_ex does for pa_decode; the workspace is
 * pa_decode_mq_workspace_size(geom, num_seqs, n_q, num_ctas). */
pa_status pa_decode_mq_ex(const void *q, const void *k_cache, const void *v_cache,
                          const float *k_scale, const float *v_scale,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          const int32_t *context_lens, int32_t num_seqs, int32_t n_q,
                          float scale, void *out, void *workspace, size_t workspace_bytes,
                          pa_geom geom, int32_t *dev_status, void *stream, int32_t num_ctas);

/* Workspace bytes pa_decode_mq needs (num_ctas 0: the default grid); 0 when
 * the geometry or n_q is not supported. */
size_t pa_decode_mq_workspace_size(pa_geom geom, int32_t num_seqs, int32_t n_q,
                                   int32_t num_ctas);

/*
 * pa_sink_write -- store bf16 attention-sink rows of new tokens.
 *
 * For each row t with 0 <= positions[t] < n_sink and 0 <= seq_rows[t] <
 * num_seqs: sink_k[seq_rows[t]][h][positions[t]][:] = k[t][h][:] for every
 * kv head h (same for v). Other rows are skipped. Call it beside
 * pa_cache_write for the same tokens; the INT8 pool keeps its own codes.
 *
 *   k, v        bf16 [num_tokens][n_kv][d_h] (16-byte aligned)
 *   seq_rows    int32 [num_tokens]: the batch row of each token's sequence
 *   positions   int32 [num_tokens]: each token's position in its sequence
 *   sink_k, sink_v  bf16 [num_seqs][n_kv][n_sink][d_h] (written, 16-byte aligned)
 *   n_sink      1..16
 */
pa_status pa_sink_write(const void *k, const void *v, const int32_t *seq_rows,
                        const int32_t *positions, int64_t num_tokens, void *sink_k, void *sink_v,
                        int32_t n_sink, int32_t num_seqs, pa_geom geom, void *stream);

/*
 * pa_kv_read_probe -- read the K/V bytes a decode of this batch reads, and
 * nothing more, to measure what the scattered access pattern allows.
 * The pages have no counterpart: it is a measurement aid that times plain
 * 16-byte loads of the same physical blocks, through the same block tables,
 * as pa_decode would read (every block of ctx_b tokens of every sequence),
 * without arithmetic.
 *
 *   heads_per_read  kv heads read together as one contiguous run of a block
 *                   (1: the (block, head) tiles one by one; n_kv: all heads
 *                   of a block); must divide n_kv
 *   num_ctas        grid size (> 0)
 *   sink            uint32 [num_ctas], written: an XOR of every word read
 * Other arguments as pa_decode (INT8/INT4 pools also read their scales;
 * bf16 pools take NULL scales). Blocks outside the pool and context lengths
 * outside [0, max_blocks_per_seq * 16] are skipped.
 */
pa_status pa_kv_read_probe(const void *k_cache, const void *v_cache, const float *k_scale,
                           const float *v_scale, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *context_lens,
                           int32_t num_seqs, int32_t heads_per_read, int32_t num_ctas,
                           uint32_t *sink, pa_geom geom, void *stream);

/*
 * pa_decode_noalloc -- pa_decode without a caller workspace, for callers that
 * cannot allocate device memory (for example a plugin whose host framework
 * owns all device memory and forbids allocating inside its execute callback).
 * The pages have no counterpart: this is a deployment convenience.
 *
 * Same arguments and results as pa_decode, minus workspace/workspace_bytes.
 * The split scratch lives in one fixed array of PA_NOALLOC_SCRATCH_BYTES that
 * every GPU loading the library holds until the process exits; nothing is
 * allocated per call. A batch whose pa_decode_workspace_size(geom, num_seqs, 0)
 * exceeds that size is refused with PA_ERR_WORKSPACE before anything is
 * enqueued (use pa_decode with a workspace of its own instead).
 * The first call on a device looks up the array's device address (which may
 * load the library's device code) and keeps it for the life of the process;
 * make that first call before any stream capture. cudaDeviceReset on a
 * device unloads the array with the context, so the kept address goes stale:
 * after a reset, reload the library before calling this entry point again. Each call clears the array's counter area on `stream`, then runs
 * the decode there. All calls on a device share the one array, so calls whose
 * GPU work can overlap (different streams without ordering) race and give
 * wrong results: order them on one stream.
 */
#define PA_NOALLOC_SCRATCH_BYTES (8u << 20)
pa_status pa_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                            const float *k_scale, const float *v_scale,
                            const int32_t *block_tables, int32_t max_blocks_per_seq,
                            const int32_t *context_lens, int32_t num_seqs, float scale, void *out,
                            pa_geom geom, int32_t *dev_status, void *stream);

/* Default CTA count pa_decode uses for this geometry on the current device
 * (>= 1), or a negative pa_status. */
int32_t pa_decode_default_ctas(pa_geom geom, int32_t num_seqs);

/* Host-only: how pa_decode splits work. The W = n_kv * sum_b ceil(ctx_b / bs)
 * (sequence, kv head, block) items are laid out sequence-major, kv-head next;
 * with G = min(num_ctas, W), CTA c < G takes items [floor(c*W/G),
 * floor((c+1)*W/G)) and CTAs c >= G do nothing. For item x this returns the
 * CTA that owns it. Exposed so the split can be checked on a CPU. */
int32_t pa_plan_owner(int64_t item, int64_t total_items, int32_t num_ctas);

/* Human-readable name of a status. Never NULL. */
const char *pa_status_string(pa_status status);

/* The status a device word stands for (first bit set wins: BAD_BLOCK,
 * BAD_SLOT, BAD_CONTEXT, TIMEOUT), PA_OK for 0. */
pa_status pa_status_from_device(int32_t dev_word);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int32_t pa_version(void);

/*
 * pa_wait_selftest -- exercise the failure path of the bounded pipeline
 * waits: one CTA waits, with the decode kernel's wait primitive, on a shared
 * barrier that nothing arrives on; after limit_us microseconds the wait gives
 * up, PA_DEV_TIMEOUT is ORed into *dev_status (device, int32) and the kernel
 * returns. Nothing faults or hangs and the context stays usable: read
 * *dev_status after the stream finishes (pa_status_from_device gives
 * PA_ERR_TIMEOUT). Errors: PA_ERR_NULL without dev_status, PA_ERR_SHAPE for
 * limit_us outside 1..1000000, PA_ERR_CUDA if the launch fails.
 */
pa_status pa_wait_selftest(int32_t *dev_status, int32_t limit_us, void *stream);

/*
 * pa_block_copy -- the device half of copy-on-write ([F] "Prefix Caching 与
 * Copy-on-Write": a branch that appends to a shared, partly filled last
 * block gets a new block holding a copy of the filled slots; [T] 考点 4:
 * only that one 16-token block is copied).
 *
 * For each pair p: every kv head and all block_size slots of block
 * pairs[p][0] are copied to block pairs[p][1], in k_cache and v_cache and,
 * for PA_KV_INT8, in k_scale and v_scale. Copying all slots is the plainest
 * reading: slots past the filled ones hold nothing a reader may use.
 *
 *   k_cache, v_cache  pool (read and written), layout above
 *   k_scale, v_scale  fp32 scales for PA_KV_INT8, NULL for PA_KV_BF16
 *   pairs         int32 [num_pairs][2] device array of (source, destination)
 *                 block ids, as pa_allocator_append_slots hands them out.
 *                 Destinations are distinct and none is a source of another
 *                 pair (otherwise the result is undefined).
 *   num_pairs     >= 0 (0 enqueues nothing)
 *   dev_status    optional; a pair with a block id outside [0, num_blocks)
 *                 is skipped and sets PA_DEV_BAD_BLOCK
 */
pa_status pa_block_copy(void *k_cache, void *v_cache, float *k_scale, float *v_scale,
                        const int32_t *pairs, int32_t num_pairs, pa_geom geom,
                        int32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
