/*
 * kvq.h -- C ABI of libkvq.so: decode-phase attention over a quantized KV cache
 * on one GB300 (sm_103a).
 *
 * What is computed.  K is kept as an 8-bit payload, four codes packed per
 * 32-bit word, with one fp16 scale per 32 head-dim elements ("Flash Attention
 * for llama.cpp on RDNA3", first paragraph: only the 8-bit K payload and fp16
 * scales are stored, and four 8-bit values fill one 32-bit word for the dot4
 * instruction).  V is kept as q4_0 or q8_0 blocks of 32 with an fp16 scale (the
 * V formats of that page's VRAM and KLD tables).  The cache of a sequence is a
 * list of append-only segments: new tokens go into the last one, filled tokens
 * are never copied or moved (BitLLM summary, "What differs").  A query is
 * quantized per 32-block with the K rule, so q.k is a sum over blocks of exact
 * int32 dot products scaled by the two fp16 scales (BitLLM summary, "How to
 * use": the MatMul stays in the integer domain and casts are deferred);
 * softmax and the P.V product over dequantized V are then evaluated in fp32.
 *
 * Quantization rules (bit-exact contract):
 *   int8 (K, Q, q8_0 V): s = fp16_rn(absmax/127); c = clamp(round_half_away(x/s), -127, 127);
 *                        s == 0 gives all-zero codes.
 *   q4_0 (V):            d = fp16_rn(absmax/8); q = clamp(round_half_away(x/d) + 8, 0, 15);
 *                        value (q-8)*d; d == 0 gives q = 8.
 * x/s is the correctly rounded fp32 quotient; absmax is over the 32 fp16 inputs.
 *
 * Memory.  The library allocates nothing.  Every pointer marked "device" is
 * caller-owned device memory of the current CUDA device; every pointer marked
 * "host" is caller-owned host memory read during the call only.  Work is
 * enqueued on `stream` (a cudaStream_t; NULL = legacy default stream) and is
 * asynchronous: no call synchronizes the host.  Kernels are chained with
 * programmatic dependent launch (set KVQ_PDL=0 in the environment to launch
 * them plainly); calls can be captured into CUDA graphs once the first call on
 * the device has run outside capture (it caches device attributes).  Other
 * environment knobs steer the launch plan only, never the arithmetic's
 * definition: KVQ_SPLIT (force the split chunk), KVQ_SPLIT_WARPS, KVQ_ROW_TILE,
 * KVQ_PREFILL=0 and KVQ_TC_ROWS (which kernel takes long query chunks), and
 * KVQ_PREFILL_BALANCE / KVQ_PREFILL_CTA_COST (the uneven two-way split of a
 * one-wave tcgen05 launch).  A plan with more splits changes the order of the
 * fp32 sums, within the stated tolerance.
 *
 * Errors.  Arguments are validated before anything is enqueued; a failed
 * validation returns a status and changes no state (kvq_append bumps segment
 * lengths only on success).  A launch failure returns KVQ_ERR_CUDA.  Faults
 * during execution surface at the caller's next synchronization.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_QBLOCK 32          /* quantization block (head-dim elements)          */
#define KVQ_HEAD_DIM 128       /* the only head_dim the library supports          */
#define KVQ_SEG_ALIGN 64       /* segment capacity must be a multiple of this     */
#define KVQ_MAX_ROWS 32        /* query rows one attention CTA takes (row tile)   */
#define KVQ_MAX_T_Q 4096       /* query tokens per sequence per call              */
#define KVQ_MAX_T_Q_APPEND 8   /* ... when the call also appends them (fused)     */
#define KVQ_MAX_HEADS 256      /* n_q_heads and n_kv_heads limit                  */
#define KVQ_MAX_CALLS 16       /* decode calls fused by kvq_decode_attn_multi     */

typedef enum kvq_status {
    KVQ_OK = 0,
    KVQ_ERR_INVALID_ARG = 1,   /* a pointer, size or layout rule is violated      */
    KVQ_ERR_UNSUPPORTED = 2,   /* no sm_103 device, or a size the kernels lack    */
    KVQ_ERR_CAPACITY = 3,      /* kvq_append: the open segment is too small       */
    KVQ_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required      */
    KVQ_ERR_CUDA = 5,          /* a CUDA runtime call or kernel launch failed     */
    KVQ_ERR_TIMEOUT = 6        /* a kernel gave up waiting for its own copies     */
} kvq_status;

typedef enum kvq_vtype {
    KVQ_V_Q4_0 = 0,            /* 16 bytes of nibbles + fp16 scale per 32 values  */
    KVQ_V_Q8_0 = 1             /* 32 int8 + fp16 scale per 32 values              */
} kvq_vtype;

/*
 * K format.  KVQ_K_I8 (the default): int8 codes + fp16 scale per 32 values,
 * and the query is quantized per 32-block the same way, so q.k is a sum of
 * exact integer block dots ("Flash Attention for llama.cpp on RDNA3", first
 * paragraph).  KVQ_K_F16: K kept as its fp16 values and the query used
 * unquantized (the F16 K / q4_0 V configuration of the same page's title and
 * KLD tables), score = sm_scale * q.k with fp32 accumulation.  F16 K supports
 * kvq_append and the decode calls without fused append (k16_new / v16_new
 * must be NULL) and not kvq_debug_qk.
 */
typedef enum kvq_ktype {
    KVQ_K_I8 = 0,
    KVQ_K_F16 = 1
} kvq_ktype;

/*
 * Segment layout (the stride-1 axis and packing of a segment's code bytes,
 * chosen per segment: BitLLM summary, "How it works" and "What differs", where
 * a layout is picked per sequence length by a cost model and a new layout only
 * ever applies to a new append-only segment).
 *   KVQ_LAYOUT_TILES  16-token tiles with the code bytes permuted into the
 *                     order the attention kernel's MMA lanes read them (see
 *                     "Tiles" below).  Every fragment read is one
 *                     conflict-free 16-byte load; a tile is the unit of every
 *                     copy, so a segment's last partly filled tile is read
 *                     whole.  The default.
 *   KVQ_LAYOUT_ROWS   one row per token in element order: K row j = code of
 *                     element j, q4_0 V row = the 32-blocks' 16 bytes in the
 *                     usual q4_0 order, q8_0 V row = codes in element order
 *                     (the order of the row sizes below).  Copies move exactly
 *                     the filled rows; the kernel then permutes each staged
 *                     tile into the tile order in shared memory (extra unpack
 *                     instructions).  int8 K only.
 * kvq_layout_cost / kvq_choose_layout weigh the two per segment.
 */
typedef enum kvq_layout {
    KVQ_LAYOUT_TILES = 0,
    KVQ_LAYOUT_ROWS = 1
} kvq_layout;

/*
 * One append-only segment of one sequence.  All four arrays are device memory,
 * 16-byte aligned and head-major: kv head h owns cap token rows starting at row
 * h*cap, and token t of the segment is row t of its head.  Row sizes (and, for
 * KVQ_LAYOUT_ROWS, the byte order of each row):
 *   k_q  int8 codes, head_dim bytes per row (F16 K: fp16 values, 2*head_dim
 *        bytes per row)
 *   k_s  fp16 scales, head_dim/32 per row, plain [kv_head][token][block] order
 *        (F16 K: unused, may be NULL)
 *   v_q  q4_0: head_dim/2 bytes per row, in each 32-block byte j holds element j
 *              (low nibble) and element j+16 (high nibble);
 *        q8_0: int8 codes, head_dim bytes per row
 *   v_s  fp16 scales, as k_s
 * Tiles.  Tokens 16T..16T+15 of a head form tile T, one contiguous run of 16
 * rows in every array.  Scales keep row order inside a tile; the code bytes of
 * k_q and v_q are permuted inside the tile so that the attention kernel copies
 * a tile with one bulk copy and reads it with conflict-free 16-byte loads.
 * With u = token % 16 (sub = u/8, gu = u%8, cu = gu/2, e = u%2) and j the byte
 * of the row in the logical order above, byte j of token u sits at tile offset
 *   k_q       ((2*sub + j/64)*32 + 4*gu + (j%32)/8)*16 + 8*((j/32)%2) + j%8
 *   v_q q4_0  (sub*32 + 4*((j%16)/2) + cu)*16 + 4*(j/16) + 2*e + j%2
 *   v_q q8_0  ((2*sub + j/64)*32 + 4*((j%32)/4) + cu)*16 + 8*((j/32)%2)
 *             + 4*((j%4)/2) + 2*(j%2) + e
 * and for F16 K, with j the element (not byte) of the row, the fp16 value of
 * element j of token u sits at byte offset (a 4096-byte tile)
 *   k_q f16   (j/16)*512 + (4*(u%8) + (j%8)/2)*16 + 4*(u/8 + 2*((j%16)/8)) + 2*(j%2)
 * (head_dim 128), for segments of KVQ_LAYOUT_TILES.  Segments of
 * KVQ_LAYOUT_ROWS keep every row in the element order above.  Only kvq_append
 * and the fused append write code bytes, so callers never see the
 * permutation unless they read the arrays themselves.
 * cap  : capacity in tokens, a positive multiple of KVQ_SEG_ALIGN.
 * len  : tokens filled, 0..cap (host bookkeeping; kvq_append advances it).
 * pos0 : absolute position of the segment's token 0.  Segment k+1 of a sequence
 *        must start where segment k ends: pos0[k+1] == pos0[k] + len[k]; the
 *        first segment starts at 0.  Only the last segment of a sequence is
 *        open for appends.
 * layout: kvq_layout of this segment's code bytes (0 = KVQ_LAYOUT_TILES); the
 *        segments of one sequence may differ.
 */
typedef struct kvq_segment {
    void *k_q;
    void *k_s;
    void *v_q;
    void *v_s;
    int32_t cap;
    int32_t len;
    int32_t pos0;
    int32_t layout;
} kvq_segment;

/*
 * Host descriptor of a batch of caches that share shape and V format.
 * segs is a host array [n_seqs * max_segs]; sequence b uses segs[b*max_segs ..
 * b*max_segs + n_segs[b] - 1].  n_segs is a host array [n_seqs], each in
 * 0..max_segs and at most 64 (a sequence with no segment has no positions).
 * All of it is caller-owned.
 */
typedef struct kvq_cache {
    int32_t n_seqs;
    int32_t n_kv_heads;
    int32_t head_dim;          /* must be KVQ_HEAD_DIM                            */
    int32_t v_type;            /* kvq_vtype                                       */
    int32_t max_segs;
    int32_t *n_segs;
    kvq_segment *segs;
    int32_t k_type;            /* kvq_ktype (0 = KVQ_K_I8)                        */
    int32_t reserved;
} kvq_cache;

/*
 * kvq_append -- quantize new fp16 K/V tokens into the open (last) segment of
 * each listed sequence (steps "append-quantize K" and "append-quantize V"; the
 * int8 rule above for K and q8_0 V, the q4_0 rule for q4_0 V).
 *
 *  c        host descriptor; on success segs[last].len of every listed sequence
 *           grows by its n_new.
 *  n_seqs_in number of listed sequences (0 is a no-op).
 *  seq_ids  host [n_seqs_in], distinct sequence indices in [0, c->n_seqs).
 *  n_new    host [n_seqs_in], tokens to append per listed sequence (>= 0).
 *  k16, v16 device fp16 [sum(n_new)][n_kv_heads][head_dim], token-major, the
 *           tokens of seq_ids[0] first, 16-byte aligned.
 *  stream   cudaStream_t.
 * Every listed sequence with n_new > 0 needs at least one segment.
 * Returns KVQ_ERR_CAPACITY (nothing enqueued, nothing changed) if some open
 * segment lacks room; the caller then adds a segment and retries.
 */
kvq_status kvq_append(kvq_cache *c, int32_t n_seqs_in, const int32_t *seq_ids,
                      const int32_t *n_new, const void *k16, const void *v16,
                      void *stream);

/*
 * kvq_decode_attn -- split-KV decode attention of every sequence of c.
 *
 *  q16       device fp16 [n_seqs][t_q][n_q_heads][head_dim], 16-byte aligned.
 *            The t_q query tokens of a sequence are its last t_q positions.
 *  n_q_heads query heads.
 *  t_q       query tokens per sequence, 1..KVQ_MAX_T_Q: one decode token,
 *            a few tokens to verify (speculative decoding), or a chunk of
 *            prompt tokens (chunked prefill over the cache, causal_tail set).
 *            A kv head's t_q x (query heads of it) rows are attended in row
 *            tiles of up to KVQ_MAX_ROWS rows, one CTA per tile and split;
 *            each tile streams the positions its split covers.
 *  causal_tail nonzero: query token i sees positions 0 .. L-t_q+i (a causal mask
 *            among the t_q newest positions); zero: every query token sees
 *            0 .. L-1.
 *  seq_lens  device int32 [n_seqs]: L of each sequence (positions, including
 *            the t_q new ones).  Positions at or beyond max_len, or beyond the
 *            last segment's capacity, are ignored.
 *  max_len   host: upper bound of seq_lens, sizes the grid.
 *  head_map  host int32 [n_q_heads]: kv head read by each query head, or NULL
 *            for contiguous groups (query head h reads kv head
 *            h / (n_q_heads/n_kv_heads)).
 *  sm_scale  softmax scale applied to q.k (e.g. 1/sqrt(head_dim)).
 *  out       device fp32 [n_seqs][t_q][n_q_heads][head_dim], 16-byte aligned:
 *            softmax(q.k*sm_scale).v
 *  lse       device fp32 [n_seqs][t_q][n_q_heads]: natural log of
 *            sum_t exp(sm_scale*q.k_t).  A row that sees no position gets
 *            out = 0 and lse = -inf.
 *  workspace device scratch for the split partials, 256-byte aligned, at
 *            least kvq_decode_workspace_size() bytes; NULL is allowed when
 *            that size is 0.
 *  workspace_bytes size of workspace; KVQ_ERR_WORKSPACE if it is too small.
 * Launches (per group of at most 64 sequences): the split-KV attention kernel
 * and, when a sequence is split, the log-sum-exp combine kernel.  It is
 * kvq_decode_attn_multi with one call.
 */
kvq_status kvq_decode_attn(const kvq_cache *c, const void *q16, int32_t n_q_heads,
                           int32_t t_q, int32_t causal_tail, const int32_t *seq_lens,
                           int32_t max_len, const int32_t *head_map, float sm_scale,
                           float *out, float *lse, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * kvq_decode_workspace_size -- bytes of workspace kvq_decode_attn needs for
 * these arguments on the current device (0 when no sequence is split).  It
 * depends on the device's SM count, n_seqs, the heads, t_q, max_len and the
 * host segment lengths, so query it again after any of them changes.
 *  bytes  host out.
 */
kvq_status kvq_decode_workspace_size(const kvq_cache *c, int32_t n_q_heads, int32_t t_q,
                                     int32_t max_len, const int32_t *head_map, size_t *bytes);

/*
 * One decode call for kvq_decode_attn_multi: the arguments of kvq_decode_attn
 * that belong to one cache, with the same meaning and rules, plus an optional
 * fused append:
 *  k16_new, v16_new  NULL, or device fp16 [n_seqs][t_q][n_kv_heads][head_dim]
 *            (16-byte aligned): the step's t_q new tokens of every sequence.
 *            The call then does what kvq_append of these tokens followed by
 *            the decode would do, in the attention kernel itself: the tokens
 *            are quantized by the append rules and stored at the end of each
 *            sequence's open segment, and the decode sees them.  Every
 *            sequence needs an open segment with room for t_q more tokens
 *            (else KVQ_ERR_CAPACITY, nothing enqueued); seq_lens must already
 *            count the new tokens; the host len of each open segment grows by
 *            t_q when the call succeeds.  A cache that receives tokens may
 *            appear in only one call of a kvq_decode_attn_multi.
 */
typedef struct kvq_decode_desc {
    const kvq_cache *cache;
    const void *q16;
    int32_t n_q_heads;
    int32_t t_q;
    int32_t causal_tail;
    const int32_t *seq_lens;
    int32_t max_len;
    const int32_t *head_map;
    float sm_scale;
    float *out;
    float *lse;
    const void *k16_new;
    const void *v16_new;
} kvq_decode_desc;

/*
 * kvq_decode_attn_multi -- n (0..KVQ_MAX_CALLS) decode calls, e.g. the main
 * and the draft model's caches of one speculative-decoding step, enqueued as
 * one split-attention launch (and one combine) instead of one per call.  Each
 * call computes exactly what kvq_decode_attn computes for it; the calls may
 * use different caches, head counts, head maps, t_q and scales, but caches with
 * different V formats go to separate launches.  Splits are planned over all
 * calls together, so the GPU fills with the calls' positions at once.
 *  calls      host array [n] (read during the call only).
 *  workspace  as kvq_decode_attn, at least kvq_decode_multi_workspace_size().
 * Errors: as kvq_decode_attn (and kvq_append for a fused append), checked for
 * every call before anything is enqueued.  The pages describe single-cache decode only; fusing calls is the
 * library's own launch plan.
 */
kvq_status kvq_decode_attn_multi(int32_t n, const kvq_decode_desc *calls, void *workspace,
                                 size_t workspace_bytes, void *stream);

/*
 * kvq_decode_multi_workspace_size -- bytes of workspace kvq_decode_attn_multi
 * needs for these calls (q16, seq_lens, out and lse are not read).
 *  bytes  host out.
 */
kvq_status kvq_decode_multi_workspace_size(int32_t n, const kvq_decode_desc *calls, size_t *bytes);

/*
 * kvq_decode_attn_noalloc -- kvq_decode_attn for callers that cannot allocate
 * device memory.  (The pages have no counterpart: this is a library-usage
 * variant, not a step of the method.)  Typical callers: code recorded into a
 * CUDA graph or running inside a latency-critical decode loop, where a
 * cudaMalloc (which may synchronize the device) is not allowed, and runtimes
 * whose memory manager owns all device memory and has no way to hand over a
 * temporary buffer.  Inputs and outputs are still passed by the caller; only
 * the split partials go to a scratch array inside the library.
 *
 *  The scratch is one file-scope device array of KVQ_NOALLOC_SCRATCH_BYTES
 *  (32 MiB) that every GPU loading the library holds until the process exits.
 *  The call allocates nothing and calls no allocating routine.  If this call's
 *  partials would need more than KVQ_NOALLOC_SCRATCH_BYTES it returns
 *  KVQ_ERR_WORKSPACE and enqueues nothing (kvq_decode_workspace_size gives the
 *  need; roughly rows x splits x 516 bytes).
 *  The first call on a device looks up the array's device address (once per
 *  device, with that device current); make that first call before any stream
 *  capture.  All calls share the array and it keeps the last call's contents;
 *  nothing in it has to start at zero, because every partial a call reads was
 *  written earlier in the same call.  Calls whose work overlaps on the GPU
 *  (other streams, or other host threads) race on the array: serialize them.
 * Other arguments and results as kvq_decode_attn.
 */
#define KVQ_NOALLOC_SCRATCH_BYTES (32u << 20)
kvq_status kvq_decode_attn_noalloc(const kvq_cache *c, const void *q16, int32_t n_q_heads,
                                   int32_t t_q, int32_t causal_tail, const int32_t *seq_lens,
                                   int32_t max_len, const int32_t *head_map, float sm_scale,
                                   float *out, float *lse, void *stream);

/*
 * kvq_wait_timeouts -- the attention kernel bounds every wait for a copy it
 * issued; a wait that gives up (which no correct run does) makes the kernel
 * drain its copies, write NaN for the CTA's rows and bump a per-device
 * counter.  This call reads that counter for the current device into *count
 * (host; synchronizes with the device) and returns KVQ_ERR_TIMEOUT when it is
 * nonzero, KVQ_OK otherwise.  The pages have no counterpart: it is the
 * library's own hang guard.
 */
kvq_status kvq_wait_timeouts(uint32_t *count);

/*
 * kvq_reset_wait_timeouts -- set the current device's wait counter of
 * kvq_wait_timeouts back to 0 (synchronizes with the device).  The pages have
 * no counterpart.
 */
kvq_status kvq_reset_wait_timeouts(void);

/*
 * Per-segment layout cost model (BitLLM summary, "How it works": a layout is
 * scored as alpha1 * Bytes / BW + alpha2 * UnpackOps, both weights fitted once
 * per GPU by a microbenchmark; "What differs": the layout is chosen by the
 * expected length, a new layout only for a new segment).  The library's
 * terms for one kv head of a segment of n tokens read by the attention kernel:
 *   Bytes      KVQ_LAYOUT_TILES: whole 16-token tiles, ceil(n/16)*16 rows;
 *              KVQ_LAYOUT_ROWS: n code rows plus the scale rows rounded up
 *              to a pair (a row: 128 K bytes + 64 (q4_0) or 128 (q8_0) V
 *              bytes + 16 bytes of scales);
 *   UnpackOps  tiles: 0; rows: ops_rows_per_tile per staged tile (the
 *              in-shared-memory permute into the tile order).
 * cost = us_per_byte * Bytes + us_per_op * UnpackOps, in microseconds; the
 * layout-independent work (the same number of tiles computed either way) is
 * left out.  kvq_layout_model_default() gives the coefficients fitted on a
 * GB300 (layout_calib.py beside the package; its record layout_model.json
 * holds every measured point).  On that GPU the tiles cost less at every
 * segment length.
 */
typedef struct kvq_layout_model {
    double us_per_byte;         /* time per HBM byte moved by the copies    */
    double us_per_op;           /* time per unpack warp-instruction         */
    double ops_rows_per_tile;   /* rows-layout unpack instructions per tile */
} kvq_layout_model;

/* The fitted GB300 coefficients.  m: host out. */
kvq_status kvq_layout_model_default(kvq_layout_model *m);

/*
 * kvq_layout_cost -- modelled cost (us) of one attention pass over one kv head
 * of a segment of n_tokens (>= 1) tokens in `layout` with V format v_type,
 * under model m (NULL: the default).  cost_us: host out.
 */
kvq_status kvq_layout_cost(int32_t layout, int32_t v_type, int32_t n_tokens, const kvq_layout_model *m,
                           double *cost_us);

/*
 * kvq_choose_layout -- the layout of lower modelled cost for a new segment
 * expected to hold n_tokens tokens (ties and int8-K-only rules: F16 K and
 * ties give KVQ_LAYOUT_TILES).  layout: host out.
 */
kvq_status kvq_choose_layout(int32_t k_type, int32_t v_type, int32_t n_tokens, const kvq_layout_model *m,
                             int32_t *layout);

/* Short English text of a status code (static storage). */
const char *kvq_status_string(kvq_status s);

/*
 * kvq_debug_qk -- TEST HOOK, not part of the decode path: runs the attention
 * kernel that kvq_decode_attn picks for these arguments (the split-KV kernel,
 * or the tcgen05 kernel for more than KVQ_MAX_ROWS query rows per kv head)
 * with its outputs replaced by dumps of the quantized query and the raw
 * per-block integer scores as that kernel computed them, so tests can compare
 * them bit for bit with an independent implementation.
 *
 *  q_codes   device int8 [n_seqs][t_q][n_q_heads][head_dim]
 *  q_scales  device fp16 bits [n_seqs][t_q][n_q_heads][head_dim/32]
 *  scores    device int32 [n_seqs][t_q][n_q_heads][max_len][head_dim/32]:
 *            I_b = sum over the 32 elements of block b of q_code*k_code, for
 *            every position < L of the sequence (causal masking is not applied
 *            here); other entries are left untouched.
 *  kernel    host out (may be NULL): the kernel that produced the dumps,
 *            0 the split-KV kernel, 1 the tcgen05 kernel.
 * Other arguments as kvq_decode_attn.
 */
kvq_status kvq_debug_qk(const kvq_cache *c, const void *q16, int32_t n_q_heads,
                        int32_t t_q, const int32_t *seq_lens, int32_t max_len,
                        const int32_t *head_map, int8_t *q_codes, uint16_t *q_scales,
                        int32_t *scores, int32_t *kernel, void *stream);

/*
 * kvq_debug_lose_stage -- TEST HOOK, not part of the decode path: the decode
 * call of kvq_decode_attn (same arguments and rules) on a test flavour of the
 * split-KV kernel in which warp 0 of the first CTA arms the barrier of its
 * second copy stage without issuing that stage's copies.  Its bounded wait on
 * that stage (a short limit here) runs out, which drives the give-up path of
 * kvq_wait_timeouts: the warp waits for every copy it did issue, the CTA's
 * query rows come out as NaN (after the combine, every query row of kv head 0
 * of sequence 0 when that CTA is its first split), the wait counter grows by
 * one, and the device stays usable.  Nothing faults and nothing waits without
 * a limit.  The flavour exists for the 16-warp, <= 8-row form with int8 K and
 * q4_0 V: calls that plan otherwise, or whose first CTA's warp 0 has fewer
 * than two copy stages of work, return KVQ_ERR_UNSUPPORTED or lose no stage.
 * The pages have no counterpart: it tests the library's own hang guard.
 */
kvq_status kvq_debug_lose_stage(const kvq_cache *c, const void *q16, int32_t n_q_heads,
                                int32_t t_q, int32_t causal_tail, const int32_t *seq_lens,
                                int32_t max_len, const int32_t *head_map, float sm_scale,
                                float *out, float *lse, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * kvq_debug_plan -- TEST HOOK, not part of the decode path: the launches that
 * kvq_decode_attn_multi would make for `calls`, worked out on the host for a
 * device with n_sms SMs on which ctas_per_sm[i] split-kernel CTAs fit per SM:
 *   i = 0  the <= 8-row kernel, 16 warps;  1  the same with 8 warps;
 *   i = 2  16-row tiles;                   3  32-row tiles.
 * It reads the calls' host descriptors and the same environment knobs as the
 * decode call (KVQ_SPLIT, KVQ_SPLIT_WARPS, KVQ_ROW_TILE, KVQ_PREFILL,
 * KVQ_TC_ROWS, KVQ_PREFILL_BALANCE, KVQ_PREFILL_CTA_COST).  It
 * touches no device and dereferences no device pointer, so segments and
 * k16_new / v16_new may hold any non-null 16-byte-aligned address; q16,
 * seq_lens, out and lse may be NULL.
 *
 *  out              host [max_out]: launch i for i < min(*n_out, max_out), in
 *                   launch order (may be NULL when max_out is 0)
 *  n_out            host: launches of the plan
 *  workspace_bytes  host: what kvq_decode_multi_workspace_size would report
 *  n_pre_appends    host: calls whose step tokens go through a separate append
 *                   launch first (the tcgen05 kernel has no fused append)
 * Errors: the argument checks of kvq_decode_attn_multi (pointers aside), and
 * KVQ_ERR_INVALID_ARG for n_sms < 1, ctas_per_sm NULL or an entry < 1, or a
 * NULL n_out / workspace_bytes / n_pre_appends.
 */
typedef struct kvq_plan_launch {
    int32_t kernel;     /* 0 split kernel, 1 tcgen05 prefill kernel */
    int32_t n_tiles8;   /* split kernel: 8-row query tiles per CTA (1, 2 or 4); else 0 */
    int32_t warps;      /* split kernel: warps per CTA; else 0 */
    int32_t chunk;      /* kv positions per split (after the first, see chunk0) */
    int32_t chunk0;     /* kv positions of the first split: chunk, except on a
                           one-wave tcgen05 launch split unevenly (large first
                           pieces on every busy SM, small second pieces taken
                           by the SMs that would idle) */
    int32_t n_ctas;     /* CTAs of the attention launch */
    int32_t n_rows;     /* query rows of the combine launch (0: no combine launch) */
} kvq_plan_launch;

kvq_status kvq_debug_plan(int32_t n, const kvq_decode_desc *calls, int32_t n_sms,
                          const int32_t *ctas_per_sm, kvq_plan_launch *out,
                          int32_t max_out, int32_t *n_out, size_t *workspace_bytes,
                          int32_t *n_pre_appends);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
