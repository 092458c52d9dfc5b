/*
 * mk.h -- C ABI of the GB300 persistent decode megakernel library (libmk.so).
 *
 * Batch-1 autoregressive decode of a Qwen3-style decoder run as ONE
 * cooperatively launched kernel that loops over layers and decode steps
 * without exiting (page A, section "The idea: one kernel that never exits":
 * a single resident kernel that takes the whole GPU and runs the decode loop
 * itself instead of a chain of per-op launches).
 * Around that loop: a batched prompt prefill on tensor cores (mk_prefill), a
 * streaming mailbox the kernel fills with each greedy id while it runs
 * (mk_decode_start / mk_mailbox_read), and the per-op ablation of the same
 * math, plain or replayed from a CUDA graph (MK_DECODE_PER_OP*).
 *
 * Sources cited below:
 *   page A = "Porting a 1,200-line persistent CUDA megakernel to Qwen3-TTS:
 *            ~25 ms to first audio chunk" (dev.to)
 *   page B = "I made a single CUDA kernel speak: streaming Qwen3-TTS at 50ms
 *            latency on an RTX 5090" (theaicatchup.com)
 *
 * Conventions for every entry point:
 *   - Return value: MK_OK (0) or a negative MK_ERR_* code.  Nothing aborts the
 *     process.  mk_error_string() names a code.
 *   - "device" pointers are CUDA global-memory addresses on the handle's device
 *     (the device current at mk_create); "host" pointers are ordinary host memory.
 *   - Streams are passed as `mk_stream` (a cudaStream_t); NULL is the legacy
 *     default stream.
 *   - A handle is not thread-safe: one caller at a time.
 */
#ifndef MK_H
#define MK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define MK_OK               0
#define MK_ERR_INVALID_ARG (-1)  /* bad pointer, size or option, checked on the host */
#define MK_ERR_UNSUPPORTED (-2)  /* shape or launch geometry this build does not handle */
#define MK_ERR_KV_FULL     (-3)  /* position + forwards would pass max_seq (host check) */
#define MK_ERR_BAD_TOKEN   (-4)  /* id >= vocab_in, or a sentinel row outside the buffer
                                    (found on the device; later forwards are skipped) */
#define MK_ERR_TIMEOUT     (-5)  /* a device wait (grid barrier, ring, merge) ran past
                                    its time budget; the kernel returned early */
#define MK_ERR_NUMERIC     (-6)  /* a logit was NaN or infinite */
#define MK_ERR_CUDA        (-7)  /* a CUDA runtime call failed */
#define MK_ERR_NO_MEMORY   (-8)  /* a device allocation failed */
#define MK_ERR_BAD_POSITION (-9) /* an MRoPE position-stream value outside the rotary table */

typedef struct mk_handle mk_handle;
typedef void *mk_stream; /* cudaStream_t */

/* ---- model description ---------------------------------------------------
 * Qwen3-style decoder (page B, "Why Does a Single Kernel Even Matter for
 * TTS?": the TTS talker has the dimensions, layer count and heads of
 * Qwen3-0.6B; vocab, RoPE frequencies and the untied head differ).  The page's
 * kernel bakes these into compile-time constants (page A, "Porting it to
 * Qwen3-TTS-1.7B"); here they are runtime fields checked at mk_create, with
 * head_dim a template parameter of the kernel.
 *
 * Limits checked by mk_create (MK_ERR_UNSUPPORTED otherwise):
 *   head_dim in {64, 128}; n_q_heads % n_kv_heads == 0 with group size
 *   n_q_heads / n_kv_heads in {1, 2, 4, 8} and group * head_dim <= 512;
 *   every GEMV input width (hidden, n_q_heads * head_dim, intermediate) is
 *   K = KPT * T with KPT in {8, 12, 16, 24} and T in {32, 64, 128, 256};
 *   rope_modes 1 and 2 need mrope_sections summing to head_dim / 2.       */
typedef struct {
  int32_t n_layers;
  int32_t hidden;          /* H */
  int32_t n_q_heads;       /* Hq */
  int32_t n_kv_heads;      /* Hkv */
  int32_t head_dim;        /* d */
  int32_t intermediate;    /* I, SiLU-gated MLP width */
  int32_t vocab;           /* V, rows of the LM head */
  int32_t vocab_in;        /* rows of the input embedding table */
  float rms_eps;           /* RMSNorm epsilon inside the root (Qwen3: 1e-6) */
  float rope_theta;        /* rotary base (Qwen3: 1e6) */
  int32_t rope_mode;       /* 0 = RoPE, 1 = sectioned MRoPE (page A, "Porting it to
                              Qwen3-TTS-1.7B": the talker's rotary positions come in
                              sections, one position stream each): contiguous runs of
                              pairs per stream; 2 = interleaved MRoPE:
                              pair i with i % 3 = s in {1, 2} follows stream s while
                              i < 3 * mrope_sections[s], every other pair stream 0 */
  int32_t mrope_sections[3]; /* rotary pairs driven by position streams 0, 1, 2 */
  int32_t max_seq;         /* KV-cache capacity in positions */
  int32_t rope_positions;  /* rows of the host-built cos/sin table; 0 = 2*max_seq + 8
                              (page B, "So, What's the Catch with These Megakernels?":
                              the rotary frequencies come from tables the host
                              builds, not from the kernel) */
  uint32_t flags;          /* reserved, must be 0 */
} mk_config;

/* Per-layer weights: device pointers to bf16, row-major [out][in] (the
 * torch.nn.Linear layout), each 16-byte aligned.  Norm gains are [H] or [d].
 *   wq [Hq*d][H], wk/wv [Hkv*d][H], wo [H][Hq*d],
 *   w_gate/w_up [I][H], w_down [H][I].
 * BORROWED: the caller keeps them alive and unchanged until mk_destroy. */
typedef struct {
  const void *attn_norm, *wq, *wk, *wv, *q_norm, *k_norm, *wo;
  const void *mlp_norm, *w_gate, *w_up, *w_down;
} mk_layer_weights;

typedef struct {
  const void *embed;      /* [vocab_in][H] bf16, device, borrowed */
  const void *lm_head;    /* [vocab][H] bf16, or NULL = tied to embed (requires
                             vocab == vocab_in); page A, "Porting it to Qwen3-TTS-1.7B":
                             the text model ties them, the talker does not */
  const void *final_norm; /* [H] bf16 */
  const mk_layer_weights *layers; /* HOST array of n_layers entries, read at mk_create */
} mk_weights;

/* ---- per-call options (all optional; pass NULL for defaults) ------------ */
#define MK_DECODE_PER_OP 1u  /* run the same math as one ordinary kernel launch per
                                phase: this kernel relaunched once per phase (the
                                launch-overhead ablation; page A, "The idea: one kernel
                                that never exits": a conventional decode step is a long
                                chain of separate kernel launches) */
#define MK_DECODE_STREAM 4u    /* publish each forward's greedy id to the handle's
                                host-mapped mailbox the moment it is chosen, so the
                                host can consume ids while the launch still runs
                                (page A, "Porting a 1,200-line persistent CUDA
                                megakernel...": the talker streams audio tokens out
                                chunk by chunk); see mk_decode_start */
#define MK_DECODE_PER_OP_GRAPH 2u /* the same per-phase launches, captured once per
                                handle as a CUDA graph of one forward and replayed
                                once per forward (the ablation without host launch
                                cost); the first such call captures and instantiates */

typedef struct {
  uint32_t flags;             /* MK_DECODE_* bits */
  const float *embeds;        /* device [n_embed_rows][H] fp32 precomputed input rows;
                                 id -(r+1) selects row r (page B, "Why Does a Single
                                 Kernel Even Matter for TTS?": a non-negative id is
                                 looked up, any other input comes precomputed from a
                                 buffer) */
  int32_t n_embed_rows;
  const int32_t *pos3;        /* device [3][n_in + n_steps] position streams for MRoPE;
                                 NULL = the slot index in every stream */
  float *logits;              /* device [n_in + n_steps][vocab] fp32 out, or NULL */
  float *hidden;              /* device [n_in + n_steps][n_layers + 1][H] fp32 out, or NULL:
                                 the input row then the residual stream after each layer */
  uint64_t *trace;            /* device [n_fwd][5*n_layers + 1][grid][4] %globaltimer stamps
                                 of each CTA's thread 0 per phase: start, input in
                                 registers, tiles and epilogue done, phase left (the LM
                                 phase: after the grid barrier that closes the forward);
                                 or NULL */
  int32_t attn_chunks;        /* split-KV chunks per kv head; 0 = the library's policy
                                 (at least 4, one per 48 cached positions up to 8, then
                                 one per 256 positions up to grid / n_kv_heads; up to 8
                                 chunks merge by polling, more by the last CTA) */
  int64_t spin_ns;            /* budget of every device wait; 0 = 1 s */
  int32_t fault_skip_barrier; /* test hook: N > 0 makes CTA 0 skip its arrival at the
                                 grid barrier that closes forward N - 1 (persistent path
                                 only), so the other CTAs time out; 0 = off (a zeroed
                                 struct runs normally) */
  /* Talker inputs summed inside the kernel.  When codes != NULL a negative id
     -(r+1) selects code row r: the forward's input is
       sum_{j<n_books} books[j][codes[r][j]] + text[text_ids[r]]
     accumulated in fp32 in table order (codebook 0 .. n_books-1, then text) --
     the same sum mk_embed_sum writes, so the result is bitwise that of the
     embeds path fed by mk_embed_sum (page B, "Why Does a Single Kernel Even
     Matter for TTS?": each talker input is the 17-way codebook + text sum).
     codes and embeds are exclusive.  A code or text id out of range
     gives MK_ERR_BAD_TOKEN. */
  const void *books;          /* device bf16 [n_books][book_rows][H] */
  int32_t n_books;            /* 0 .. 64 */
  int32_t book_rows;
  const void *text;           /* device bf16 [text_rows][H] */
  int32_t text_rows;
  const int32_t *codes;       /* device int32 [n_code_rows][n_books] */
  const int32_t *text_ids;    /* device int32 [n_code_rows] */
  int32_t n_code_rows;
} mk_decode_opts;

typedef struct {
  int32_t grid;          /* CTAs = SMs of the device, one per SM */
  int32_t threads;       /* per CTA: consumer warps + 1 producer warp */
  int32_t stages;        /* shared-memory ring stages */
  int32_t stage_bytes;
  int32_t smem_bytes;    /* dynamic shared memory per CTA */
  int32_t position;      /* next KV slot */
  int32_t max_chunks;    /* split-KV chunk capacity per kv head */
  int64_t weight_bytes;  /* bf16 bytes streamed per forward (layers + head) */
  int64_t kv_bytes;      /* KV-cache allocation */
  int32_t plan;          /* decode kernel: 0 the general one (layouts chosen at run time,
                            phases out of line), 1 compiled for hidden 1024 / MLP 3072 /
                            16:8 heads of 128, 2 for hidden 2048 / MLP 6144 / 16:8 heads of 128 */
} mk_info;

/* Validate cfg, allocate the KV cache [L][Hkv][max_seq][d] bf16 (keys and
 * values), scratch, barrier/error words and the cos/sin table (built on the
 * host in double precision), and check that one CTA per SM fits.  *out gets
 * the handle.  The pages fix no interface beyond the model constants and the
 * token-id-or-buffer input (page A, "Porting it to Qwen3-TTS-1.7B"; page B,
 * "Why Does a Single Kernel Even Matter for TTS?"); the handle holds what the
 * persistent kernel keeps between calls (page A, "The idea: one kernel that
 * never exits": the KV cache and the step loop's state).  Errors:
 * MK_ERR_INVALID_ARG, MK_ERR_UNSUPPORTED, MK_ERR_NO_MEMORY, MK_ERR_CUDA
 * (nothing is leaked on failure). */
int mk_create(const mk_config *cfg, const mk_weights *w, mk_handle **out);

/* Forget the cached context: the cursor returns to slot 0 and the last id to 0
 * (a new sequence; the KV cache of page A, "The idea: one kernel that never
 * exits", starts empty).  Enqueued on `stream`; returns after the stream
 * completes.  Errors: MK_ERR_INVALID_ARG (NULL, or a started decode not yet
 * waited for), MK_ERR_CUDA. */
int mk_reset_kv(mk_handle *h, mk_stream stream);

/* Run n_in + n_steps forwards from the handle's cursor in ONE cooperative launch.
 * Forward i < n_in consumes d_in_ids[i] (device int32; a negative id picks a
 * row of opts->embeds); forward i >= n_in consumes the greedy id of forward
 * i-1 (for i == 0, the last id of the previous call).  d_out_ids[i] (device
 * int32, n_in + n_steps entries) receives the greedy argmax of forward i,
 * lowest index on ties.  Blocks until `stream` completes and returns the
 * device status.  After an error the cached context is undefined: call
 * mk_reset_kv.  Errors: all codes above. */
int mk_decode(mk_handle *h, const int32_t *d_in_ids, int32_t n_in, int32_t n_steps,
              int32_t *d_out_ids, const mk_decode_opts *opts, mk_stream stream);

/* Batched prompt prefill: the n forwards of mk_decode(h, d_in_ids, n, 0, ...)
 * computed all at once per layer instead of one token per forward -- the
 * projections as the library's own tcgen05 tensor-core GEMMs with fp32
 * accumulation in tensor memory (each fp32 activation enters as three bf16
 * terms, hi + mid + lo: all 24 bits, each in its own accumulator), then
 * QK-norm, RoPE / MRoPE,
 * the bf16 KV append and causal attention over the cache in the library's own
 * kernels.  It fills the same KV cache and advances the same cursor, so a
 * following mk_decode(h, NULL, 0, n_steps, ...) continues from the prompt's
 * greedy id (page A, "Porting a 1,200-line persistent CUDA megakernel to
 * Qwen3-TTS": the time to the first chunk is what the listener waits for).
 *   d_in_ids: device int32 [n] (negative ids pick rows of opts->embeds).
 *   d_out_ids: device int32 [n] greedy ids after every prompt token, or NULL
 *   (then only the last token's logits are computed).  opts: embeds, pos3,
 *   logits ([n][vocab]) and hidden ([n][L+1][H]) as for mk_decode; flags,
 *   trace and code rows must be unset.  Not bitwise equal to mk_decode (other
 *   summation orders); both follow the oracle within the parity tolerance.
 * The first call of a handle creates its scratch for 256-token chunks (tens
 * of MB at the 0.6B shape, plus V x 256 fp32 logits when every id is wanted)
 * and the TMA descriptors of every weight matrix; the launch sequence of each
 * prompt length is captured as a CUDA graph on its first use and replayed
 * afterwards (the call's ids, cursor and output pointers are read from device
 * memory, so a replay serves any call of that length; at most 8 lengths are
 * kept per handle, the least recently used replaced).
 * Blocks until `stream` completes.  Errors: MK_ERR_INVALID_ARG, MK_ERR_KV_FULL,
 * MK_ERR_BAD_TOKEN, MK_ERR_BAD_POSITION, MK_ERR_NUMERIC, MK_ERR_NO_MEMORY,
 * MK_ERR_UNSUPPORTED, MK_ERR_CUDA. */
int mk_prefill(mk_handle *h, const int32_t *d_in_ids, int32_t n, int32_t *d_out_ids,
               const mk_decode_opts *opts, mk_stream stream);

/* mk_decode without the wait: enqueue the launch on `stream` and return.  Same
 * arguments and argument errors as mk_decode; the device status comes from
 * mk_decode_wait, which must be called exactly once before the handle's next
 * call (another mk_decode / mk_decode_start / mk_reset_kv first gives
 * MK_ERR_INVALID_ARG).  With MK_DECODE_STREAM in opts->flags the mailbox is
 * reset to zero ids before the launch and every forward's id appears in it as
 * soon as the kernel has chosen it (mk_mailbox_read). */
int mk_decode_start(mk_handle *h, const int32_t *d_in_ids, int32_t n_in, int32_t n_steps,
                    int32_t *d_out_ids, const mk_decode_opts *opts, mk_stream stream);

/* Wait for the launch mk_decode_start enqueued; returns its status exactly as
 * mk_decode would and advances the cursor on success.  MK_ERR_INVALID_ARG when
 * nothing is pending. */
int mk_decode_wait(mk_handle *h);

/* Non-blocking read of the streaming mailbox: *n_out = ids the current (or last)
 * MK_DECODE_STREAM launch has published so far -- ids 0 .. *n_out-1 of that call,
 * each final -- and the first min(*n_out, cap) of them are copied to dst (host
 * memory).  The mailbox is host-mapped pinned memory the handle owns (max_seq
 * ids); the kernel writes an id, fences at system scope, then raises the count,
 * and this read takes the count with acquire ordering before the ids. */
int mk_mailbox_read(mk_handle *h, int32_t *dst, int32_t cap, int32_t *n_out);

/* mk_decode with HOST id buffers: copies h_in_ids to the device, decodes and
 * copies the ids back to h_out_ids (n_in + n_steps entries) -- the token-id
 * input of page B, "Why Does a Single Kernel Even Matter for TTS?", from host
 * memory.  The copies use handle-owned staging; at most max_seq ids per call.
 * Errors: as mk_decode. */
int mk_decode_host(mk_handle *h, const int32_t *h_in_ids, int32_t n_in, int32_t n_steps,
                   int32_t *h_out_ids, const mk_decode_opts *opts, mk_stream stream);

/* Launch geometry, cursor and byte counts of a handle (the bytes one forward
 * streams: the quantity page B, "Why Does a Single Kernel Even Matter for
 * TTS?", measures the kernel's bandwidth use by).  MK_ERR_INVALID_ARG on NULL. */
int mk_get_info(const mk_handle *h, mk_info *info);

/* The decode kernel mk_create would pick for this shape on a device with n_sm
 * multiprocessors (one CTA each), as mk_info.plan: 0 the general kernel, 1 the
 * one compiled for hidden 1024 / MLP 3072 / 16:8 heads of 128, 2 the one for
 * hidden 2048 / MLP 6144 / 16:8 heads of 128.  Runs the same shape checks and
 * layout choice as mk_create, needs no device and allocates nothing (the
 * compiled instantiations are an implementation choice; the pages have no
 * counterpart of this call).  Errors: MK_ERR_INVALID_ARG (NULL pointers,
 * n_sm < 1, a config mk_create rejects as invalid), MK_ERR_UNSUPPORTED. */
int mk_plan_for(const mk_config *cfg, int32_t n_sm, int32_t *plan);

/* Talker input rows: out[r] = sum_{j<n_books} books[j][codes[r][j]] + text[text_ids[r]],
 * accumulated in fp32 in table order (page B, "Why Does a Single Kernel Even
 * Matter for TTS?": each talker input is the sum of the 16 codebook embeddings
 * and the text embedding).
 * books: device bf16 [n_books][book_rows][H]; text: device bf16 [text_rows][H];
 * codes: device int32 [n][n_books]; text_ids: device int32 [n]; out: device fp32
 * [n][H].  Ids out of range give MK_ERR_BAD_TOKEN.  Blocks until `stream` completes. */
int mk_embed_sum(const void *books, int32_t n_books, int32_t book_rows, const void *text,
                 int32_t text_rows, int32_t hidden, const int32_t *codes,
                 const int32_t *text_ids, int32_t n, float *out, mk_stream stream);

/* mk_embed_sum for callers that cannot allocate device memory -- for example a
 * host that runs inside another allocator's fixed memory pool, or a streaming
 * thread that must not call cudaMalloc because it can block and synchronise the
 * device mid-stream.  The pages have no counterpart of this entry point.
 * Same arguments, result and errors as mk_embed_sum, and it allocates nothing:
 * its scratch (one status word per output row) is a 16 KB static device array
 * that every GPU loading the library holds until the process exits.
 *   - n may be at most 4096; larger n gives MK_ERR_INVALID_ARG.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address; make that first call before any stream capture.
 *   - All calls share the array, which keeps the last call's contents; each
 *     call clears the words it uses.  Calls from several host threads are
 *     serialised; calls that overlap on the GPU (e.g. issued on different
 *     streams by other means) would race on the array. */
int mk_embed_sum_noalloc(const void *books, int32_t n_books, int32_t book_rows, const void *text,
                         int32_t text_rows, int32_t hidden, const int32_t *codes,
                         const int32_t *text_ids, int32_t n, float *out, mk_stream stream);

/* Free everything the handle owns (not the borrowed weights): the end of the
 * handle lifecycle that mk_create starts.  NULL is a no-op; always MK_OK. */
int mk_destroy(mk_handle *h);

/* Static string naming a status code (the error words the kernel sets instead
 * of trapping, so that a failed step never takes the GPU down; the pages
 * define no error model).  Unknown codes give "unknown error". */
const char *mk_error_string(int code);

#ifdef __cplusplus
}
#endif
#endif /* MK_H */
