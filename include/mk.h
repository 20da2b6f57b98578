/*
 * mk.h -- C ABI of libmk: a dense Llama/Qwen-style decoder forward pass run as
 * one persistent GB300 (sm_103a) kernel whose operators synchronise on
 * individual tiles of the intermediate tensors.
 *
 * Sources of the operations:
 *  - "MegaOps: A Kernel Overlapping Framework with PyTorch-like Modularity and
 *    Megakernel Performance" (arXiv 2611.16248), Abstract: dependencies are
 *    enforced on individual tiles of the intermediate tensor a producer writes
 *    and a consumer reads; weights are prefetched while the preceding operator
 *    runs; the comparison point is the kernel-per-operator paradigm; the models
 *    are dense Llama3 and Qwen3, decode and prefill.
 *  - "Lecture 112: Production Megakernels for Real-World Inference", Key
 *    takeaways and Technical details: an on-device interpreter whose cores
 *    atomically pop instructions from a global queue in DRAM; barriers held as
 *    tensors; shapes, extents and barriers expressed symbolically in the
 *    sequence length S and context length P so the work queue is built once;
 *    memory pipelining across output tiles; the host stays out of the hot loop.
 *
 * Conventions for every entry point:
 *  - All tensors are caller-owned DEVICE memory unless a name ends in _host.
 *    bf16 tensors are passed as raw 16-bit words; weights are [out, in]
 *    row-major, 16-byte aligned.  The library never copies or repacks weights;
 *    they must stay valid and unchanged while the plan lives.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Calls are asynchronous on `stream`; one plan is driven by one stream at a
 *    time.
 *  - Return value: MK_OK or an MK_ERR_* code.  Argument errors are returned
 *    before anything is launched.  Errors raised on the device (a wait that ran
 *    out of time, an out-of-range token or position) are latched in a device
 *    status word, returned by mk_status(), and every later launch on that plan
 *    returns the latched code without launching until mk_plan_reset().
 */
#ifndef MK_H
#define MK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MK_OK = 0,
  MK_ERR_INVALID_ARG = 1, /* bad pointer, size or shape; nothing launched      */
  MK_ERR_CUDA = 2,        /* a CUDA runtime call failed                          */
  MK_ERR_TIMEOUT = 3,     /* a device-side wait exceeded its limit (latched)     */
  MK_ERR_BOUNDS = 4,      /* a token/position/operand out of range (latched)     */
  MK_ERR_UNSUPPORTED = 5, /* shape not supported by this build                   */
  MK_ERR_NO_DEVICE = 6    /* no usable CUDA device                               */
};

enum { MK_DECODE = 0, MK_PREFILL = 1 };

typedef struct mk_plan mk_plan; /* opaque, library-owned */

/* Model shape.  Llama-3: qk_norm = 0.  Qwen3: qk_norm = 1 (per-head RMSNorm of
 * q and k over head_dim, same eps, applied before RoPE).  tied_embeddings = 1
 * makes the LM head read the embedding matrix. */
typedef struct {
  int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
  float rms_eps, rope_theta;
  int qk_norm;
  int tied_embeddings;
} mk_model_cfg;

/* Device pointers to bf16 weights.  The per-layer fields point to HOST arrays
 * of n_layers device pointers (copied at plan creation).  q_norm/k_norm may be
 * NULL when qk_norm == 0; lm_head may be NULL when tied_embeddings == 1. */
typedef struct {
  const void *embed;      /* [vocab, hidden]                 */
  const void *final_norm; /* [hidden]                        */
  const void *lm_head;    /* [vocab, hidden] or NULL if tied */
  const void *const *attn_norm; /* [hidden]                  */
  const void *const *wq;        /* [n_q_heads*head_dim, hidden]  */
  const void *const *wk;        /* [n_kv_heads*head_dim, hidden] */
  const void *const *wv;        /* [n_kv_heads*head_dim, hidden] */
  const void *const *wo;        /* [hidden, n_q_heads*head_dim]  */
  const void *const *q_norm;    /* [head_dim] or NULL            */
  const void *const *k_norm;    /* [head_dim] or NULL            */
  const void *const *ffn_norm;  /* [hidden]                      */
  const void *const *w_gate;    /* [ffn, hidden]                 */
  const void *const *w_up;      /* [ffn, hidden]                 */
  const void *const *w_down;    /* [hidden, ffn]                 */
} mk_weight_ptrs;

/* Build the tile DAG, the instruction queues and the barrier tensors for up to
 * max_batch sequences of up to max_ctx cached positions (queue extents are
 * symbolic in batch, S and P, so nothing is rebuilt when those change), and
 * allocate the plan's device scratch (activations, barrier counters, RoPE
 * table).  Uses the current CUDA device.  *out receives the plan. */
int mk_plan_create(const mk_model_cfg *cfg, const mk_weight_ptrs *w, int max_batch, int max_ctx,
                   mk_plan **out);
void mk_plan_destroy(mk_plan *plan);

/* Bytes of the KV cache the caller must allocate:
 * bf16 [n_layers][2 (k, v)][max_batch][n_kv_heads][max_ctx][head_dim].
 * Keys are stored after RoPE (and after the q/k norm when enabled). */
size_t mk_kv_cache_bytes(const mk_plan *plan);

/* One decode step for `batch` (1..max_batch) sequences, one persistent launch.
 * tokens[b]: new token id of sequence b (device int32 [batch]).
 * positions[b]: number of tokens already cached for sequence b (device int32
 *   [batch]); the new token attends over positions[b]+1 keys and its k/v are
 *   written to cache slot positions[b] of sequence slot b.  Must be < max_ctx.
 * logits: device float [batch, vocab].  */
int mk_decode_step(mk_plan *plan, const int32_t *tokens, const int32_t *positions, int batch,
                   void *kv_cache, float *logits, void *stream);

/* Same step with HOST buffers: copies tokens/positions in, runs the step, copies
 * logits [batch, vocab] out, and waits for the stream.  Host buffers should be
 * pinned for full speed.  Returns the device status after the wait. */
int mk_decode_step_host(mk_plan *plan, const int32_t *tokens_host, const int32_t *positions_host,
                        int batch, void *kv_cache, float *logits_host, void *stream);

/* Device memory that mk_decode_step_noalloc may use: a file-scope array of
 * this many bytes is part of the library image, so every GPU that loads libmk
 * holds it until the process exits. */
#define MK_NOALLOC_SCRATCH_BYTES (16u << 20)

/* A decode step for callers that must not allocate device memory when they
 * run it -- for example a serving process that handed (nearly) all device
 * memory to its own pool and KV cache at start-up, or code running under an
 * external memory manager that forbids new device allocations.  The paper has
 * no counterpart: it is the persistent launch of mk_decode_step without a plan
 * object.  The caller passes what mk_plan_create and mk_decode_step take (the
 * model shape, the weights, the cache geometry max_batch x max_ctx, then the
 * step's tokens, positions, KV cache and logits, same layouts).  Activations,
 * barrier counters, the instruction queue and the RoPE table go into the
 * static array above; nothing here calls cudaMalloc, cudaFree or any other
 * device allocator (the queue is built in ordinary host memory and copied in).
 *  - Shapes whose scratch exceeds MK_NOALLOC_SCRATCH_BYTES return
 *    MK_ERR_UNSUPPORTED before any device work.
 *  - The first call on a device (with that device current) looks up the
 *    array's device address and sets the kernel's shared-memory limit.
 *  - A call on a stream that is being captured into a graph returns
 *    MK_ERR_INVALID_ARG before any device work (the call copies host data
 *    that a replayed graph would read after it is gone).
 *  - The host-side plan and RoPE table are kept from the previous call with
 *    the same (shape, max_batch, max_ctx, device SM count), and the array's
 *    queue, bytecode, RoPE table and layer table are re-copied only when the
 *    previous call on the device left another shape's (or other weights') in
 *    it; repeated calls with one shape cost a memset and the launch.
 *  - All calls share the one array and find the previous call's contents;
 *    each call clears its own counters and control words.  Calls whose work
 *    overlaps on the GPU (several streams or threads) race on the array:
 *    serialise them.
 *  - Device-side errors (an out-of-range token or position) are not reported
 *    here; the logits are then undefined.
 * Returns MK_OK once the step is queued on `stream`. */
int mk_decode_step_noalloc(const mk_model_cfg *cfg, const mk_weight_ptrs *w, int max_batch,
                           int max_ctx, const int32_t *tokens, const int32_t *positions, int batch,
                           void *kv_cache, float *logits, void *stream);

/* Prefill one prompt of `len` tokens (1..max_ctx) into sequence slot 0 of the
 * cache at positions 0..len-1, causal; writes the last token's logits
 * (device float [vocab]). */
int mk_prefill(mk_plan *plan, const int32_t *tokens, int len, void *kv_cache, float *logits,
               void *stream);

/* The same tile routines launched kernel-per-operator on `stream` (one launch
 * per operator per layer, ordered by the stream), the comparison point.  mode is
 * MK_DECODE (batch_or_len = batch, positions used) or MK_PREFILL (batch_or_len =
 * prompt length, positions ignored).  use_graph = 1 captures the launches into
 * a CUDA graph on first use for these pointers and replays it. */
int mk_run_per_op(mk_plan *plan, int mode, int use_graph, const int32_t *tokens,
                  const int32_t *positions, int batch_or_len, void *kv_cache, float *logits,
                  void *stream);

/* Wait for `stream`, then return the plan's device status word (MK_OK or the
 * first latched MK_ERR_*). */
int mk_status(mk_plan *plan, void *stream);
/* Clear a latched error and the barrier counters (after a timeout). */
int mk_plan_reset(mk_plan *plan, void *stream);
const char *mk_status_string(int code);

/* Plan facts, for tests and measurement. */
typedef struct {
  uint32_t n_instr_decode;  /* instructions in the decode queue            */
  uint32_t n_instr_prefill; /* instructions in the prefill queue (0: none) */
  uint32_t n_barriers;      /* uint32 counters in the barrier tensor       */
  uint32_t n_launches_per_op_decode; /* kernel launches of one per-op step */
  uint32_t n_ctas;          /* CTAs of a persistent launch                  */
  uint32_t n_splits;        /* split-KV partitions per (sequence, kv head)  */
  uint64_t weight_bytes;    /* bf16 weight bytes one decode step streams    */
  uint64_t scratch_bytes;   /* device scratch owned by the plan             */
  uint32_t decode_path;     /* 0: CUDA-core decode interpreter; 1: tensor-core
                               batched decode (batches the former does not
                               take, up to 32 sequences)                     */
  uint64_t queue_hash;      /* FNV-1a hash of the decode queue as the device
                               holds it (mk_plan_get_stats only; reading it
                               back waits for the device)                    */
} mk_plan_stats;
int mk_plan_get_stats(const mk_plan *plan, mk_plan_stats *out);

/* Test-only: mk_plan_create for a device of n_sms SMs (1 .. the current
 * device's count; 0 = the device's own): the plan's projection tiling is cut
 * for n_sms SMs and its persistent launches use n_sms CTAs.  Results must not
 * depend on it ("MegaOps", Abstract: scheduling changes only when independent
 * tiles run, not what they compute); schedule-invariance tests compare plans
 * built for several counts.  Errors as mk_plan_create; n_sms above the device's
 * count is MK_ERR_INVALID_ARG. */
int mk_plan_create_for_sms(const mk_model_cfg *cfg, const mk_weight_ptrs *w, int max_batch,
                           int max_ctx, int n_sms, mk_plan **out);

/* Host-only check (no GPU needed): build the plan's queues for this shape,
 * optionally in a seeded random topological order, and run them through a
 * sequential simulator of the barrier counters.  Returns MK_OK if every wait is
 * satisfied when reached and every barrier receives exactly the releases its
 * waiters expect; fills *out (n_ctas/scratch_bytes are 0). */
int mk_plan_check(const mk_model_cfg *cfg, int max_batch, int max_ctx, uint64_t queue_perm_seed,
                  mk_plan_stats *out);

/* Prefill of `batch` prompts ("MegaOps", Abstract: prefill of the dense
 * Llama3/Qwen3 decoders, here for several prompts):
 * prompt b (tokens[b * stride .. b * stride + lens[b])) goes to sequence slot
 * b of the cache and its last token's logits to logits[b].  The prompts'
 * 128-token blocks go end to end into ONE persistent launch of the prefill
 * queue ("Lecture 112" summary, Key takeaways: one queue whose extents are
 * symbolic), so every weight tile is streamed once for all of them: a table
 * gives each block its cache slot, its prompt's first block, length and
 * token offset (RoPE positions, cache rows and causal attention stay within
 * the prompt).  When the blocks exceed the plan's context (sum over b of
 * ceil(lens[b] / 128) > ceil(max_ctx / 128)), consecutive prompts are packed
 * into as few such launches as fit.  Then each prompt's last token runs its
 * LM-head tiles.  Results are bit-identical to prompt-by-prompt calls.
 *   tokens  device int32 [batch][stride]
 *   lens    HOST int32 [batch], 1 <= lens[b] <= min(stride, max_ctx)
 *   batch   1 .. max_batch of the plan
 *   logits  device float [batch][V]
 * Argument errors: MK_ERR_INVALID_ARG (nothing launched); device errors are
 * latched as for mk_prefill. */
int mk_prefill_batch(mk_plan *plan, const int32_t *tokens, const int32_t *lens, int batch,
                     int stride, void *kv_cache, float *logits, void *stream);

/* Chunked prefill mixed with decode in the tensor-core prefill kernel
 * ("Lecture 112" summary, Key takeaways: one queue with symbolic extents
 * serves both; "MegaOps", Abstract: decode and prefill of the same decoder).
 * Chunk i is chunks[4 i .. 4 i + 3] = {slot, pos0, len, tok}: `len` tokens
 * (tokens[tok .. tok + len), device int32) of the sequence in cache slot
 * `slot`, at cache positions pos0 .. pos0 + len - 1, the positions below pos0
 * already cached.  A decode token is a chunk of length 1; a prompt's
 * continuation a longer one.  The chunks' 128-token blocks share one
 * persistent launch (as for mk_prefill_batch): every row attends to its
 * sequence's keys 0 .. its own position (the cached ones and its chunk's
 * earlier ones) and writes its key and value to the cache.  logits[i]
 * (device float [n][V]) receives the logits after chunk i's last token.
 *   chunks  HOST int32 [n][4]; 0 <= slot < max_batch, len >= 1,
 *           pos0 + len <= max_ctx; a later chunk of a slot must start where
 *           the slot's previous chunk ends (else MK_ERR_INVALID_ARG)
 * Errors as mk_prefill. */
int mk_prefill_chunks(mk_plan *plan, const int32_t *tokens, const int32_t *chunks, int n,
                      void *kv_cache, float *logits, void *stream);

/* Prefill with the logits of EVERY prompt token ("MegaOps", Abstract:
 * prefill of the dense Llama3/Qwen3 decoders).  Same as mk_prefill, except that the final RMSNorm and the LM
 * head run for all len tokens inside the same persistent launch, as
 * tensor-core GEMM tiles (128 tokens x 256 vocabulary rows) that wait on the
 * last layer's tiles of their own 128-token block.
 *   logits  device float [len][V], row-major, caller-owned; row i = the
 *           logits after token i (row len - 1 = mk_prefill's logits).
 * Errors as mk_prefill. */
int mk_prefill_logits(mk_plan *plan, const int32_t *tokens, int len, void *kv_cache, float *logits,
                      void *stream);

/* Chunked prefill mixed with decode in ONE persistent launch ("Lecture 112"
 * summary, Key takeaways: one queue with symbolic extents serves both; the
 * MegaOps Abstract's decode and prefill of the same decoder).  A decode step
 * whose columns name their cache slot: column c is the token tokens[c] of the
 * sequence in slot slots[c] at position positions[c].  Several columns of one
 * slot at consecutive positions are a prompt chunk: every column's key and
 * value are in the cache before any column's attention reads it (the
 * attention tiles wait on the whole projection), so column c attends to the
 * slot's keys 0..positions[c], its own chunk's earlier tokens included.
 * Columns of other slots are ordinary decode steps.
 *   slots   device int32 [batch], 0 <= slots[c] < max_batch (else
 *           MK_ERR_BOUNDS is latched); no two columns may share
 *           (slot, position)
 *   tokens, positions, batch, kv_cache, logits: as mk_decode_step (logits
 *           [batch][V]: every column's, the chunk's included)
 * Plans of the tensor-core batched path only (mk_plan_stats.decode_path = 1;
 * others: MK_ERR_UNSUPPORTED). */
int mk_decode_step_slots(mk_plan *plan, const int32_t *tokens, const int32_t *positions,
                         const int32_t *slots, int batch, void *kv_cache, float *logits,
                         void *stream);

/* Greedy decode of n_steps tokens of one sequence in ONE persistent launch
 * (the host stays out of the loop: "Lecture 112" summary, Practical
 * implications).  Step s (0 <= s < n_steps) is the decode step of
 * mk_decode_step at position position[0] + s; step 0 reads token[0], every
 * later step the token the previous step chose: the index of the largest
 * logit (the smallest index among equal logits), computed on the device from
 * the LM-head tiles as they finish: each CTA keeps the running maximum of the
 * LM-head tiles it finished in a step in one word of its own, and step s + 1
 * reads the token once the CTAs' words account for every LM-head tile of
 * step s.  The queue runs n_steps times with a tag per step.
 *   token       device int32 [1]      first input token
 *   position    device int32 [1]      tokens already cached (index of token)
 *   n_steps     1 .. 64               position[0] + n_steps <= max_ctx, else
 *                                     MK_ERR_BOUNDS is latched
 *   out_tokens  device int32 [n_steps] out_tokens[s] = the token step s chose
 *   logits      device float [V]      the last step's logits
 * Cache slots position[0] .. position[0] + n_steps - 1 are written.  Batch-1
 * plans of the CUDA-core path with the batch-1 register kernel and a
 * vocabulary below 2^18 rows only (other plans: MK_ERR_UNSUPPORTED); the
 * caller's buffers follow mk_decode_step's rules.  Asynchronous on
 * `stream`. */
int mk_decode_steps(mk_plan *plan, const int32_t *token, const int32_t *position, int n_steps,
                    void *kv_cache, int32_t *out_tokens, float *logits, void *stream);

/* Composition of the decode step ("One Megakernel is Not Enough", Abstract:
 * one megakernel is not always the fastest; Lecture 112 summary, Practical
 * implications: the LM head may stay a separate operator).
 * MK_LM_FUSED (default): one persistent launch runs every tile of the step,
 * the LM head included.  MK_LM_SEPARATE: the persistent launch runs the
 * layers, then the LM-head tiles run as one kernel-per-operator launch on the
 * same stream (stream order replaces their counter waits).  Results are
 * bit-identical in both modes.  Applies to mk_decode_step and
 * mk_decode_step_host calls made after it; returns MK_ERR_INVALID_ARG for a
 * null plan or an unknown mode. */
enum { MK_LM_FUSED = 0, MK_LM_SEPARATE = 1 };
int mk_plan_set_lm_mode(mk_plan *plan, int mode);

/* Test and measurement options.  force_ctas > 0 launches that many persistent
 * CTAs (<= the co-resident limit); queue_perm_seed != 0 rebuilds the decode
 * queue in a seeded random topological order; trace = 1 records one 128-byte
 * record per instruction (mk_trace_copy); wait_limit_ns bounds every device-side wait
 * (0 = default 2 s). */
int mk_plan_set_debug(mk_plan *plan, int force_ctas, uint64_t queue_perm_seed, int trace,
                      uint64_t wait_limit_ns);

/* Test-only fault injection, made on the host: instruction `index` of the
 * persistent queue (pop order) no longer releases its barrier, so the
 * consumers of that barrier wait until their bounded wait gives up and the
 * launch ends with MK_ERR_TIMEOUT latched.  The next mk_plan_set_debug()
 * rebuilds the queue; mk_plan_reset() clears the latched error. */
int mk_plan_debug_drop_release(mk_plan *plan, uint32_t index);

/* Test-only: the tensor-core tile routine (tcgen05.mma with TMEM accumulators,
 * TMA-fed 128-byte-swizzled operands) on one plain GEMM, synchronous:
 *   C[M][N] (device f32) = A[M][K] (device bf16) * B^T (device bf16),
 * row-major, 16-byte aligned; N % 128 == 0, K % 64 == 0.  b_layout 0: B is
 * [N][K] (K contiguous, as weights are stored); b_layout 1: B is [K][N] (N
 * contiguous, as the V cache is read by prefill attention).  This is the
 * contraction the batched-decode and prefill projections run ("MegaOps",
 * Abstract: the dense Llama3/Qwen3 projections).  Returns MK_OK, an argument
 * error, or MK_ERR_TIMEOUT if a bounded wait inside the kernel gave up. */
int mk_debug_gemm_bf16(const void *A, const void *B, float *C, int M, int N, int K, int b_layout,
                       void *stream);

/* Copy the trace of the last traced launch (mk_plan_set_debug(trace = 1)):
 * 16 x uint64 per instruction (128 bytes), indexed by queue position, times in
 * %globaltimer ns.  CUDA-core decode: {smid | (op | layer << 8) << 32, consumer
 * took it, its waits were satisfied, done, producer posted it, ns spent waiting
 * for operand stages, first operand stage ready, ns the producer waited for free
 * stages, then for GEMV tiles: last stage consumed (batch-1 tiles), finisher
 * took it (batch-1 tiles), instruction reached every consumer warp, hand-off
 * buffer free (batch-1 tiles); for attention tiles: inputs rotated, scores
 * done, partial stored, and for combining instructions every split's max and
 * sum in; then consumer loop top
 * before the instruction was taken, and for batch-1 GEMV tiles: consumer warp
 * 7 reached the hand-off, finisher added the partial sums, consumer warp 0
 * finished the hand-off}.  Tensor-core batched
 * decode (mk_plan_stats.decode_path = 1): {smid | (op | layer << 8) << 32,
 * compute warps took it, inputs ready (GEMM: accumulator full; otherwise
 * dependencies met), done, producer posted it, producer's dependency wait met,
 * producer issued its last stage, first MMA issued, last MMA committed, then
 * for attention splits: first key block ready, last key block done; 0 x 5}.
 * *n_records receives the count copied.  Waits for the device. */
int mk_trace_copy(mk_plan *plan, void *host_buf, size_t bytes, size_t *n_records);

#ifdef __cplusplus
}
#endif
#endif /* MK_H */
