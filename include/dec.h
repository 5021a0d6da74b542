/*
 * dec.h -- C ABI of the GB300 persistent MoE decode engine.
 *
 * One call of dec_step runs a whole decode step (every layer, the LM head and the greedy
 * argmax) as ONE launch of one persistent, warp-specialised kernel, instead of a chain of
 * per-operator kernels. This is the execution model described on the page "Ultra-High
 * Interactivity on NVIDIA GPUs? TileRT on InferenceX", section "But What Exactly is TileRT?"
 * (the host launches once, warp groups specialise on data movement and compute, stages overlap
 * at tile granularity and intermediates stay in registers, shared memory and L2), applied to the
 * per-layer decode recipe of "vLLM's Kimi K3 Backend Hits 842 Tokens per Second", section "Four
 * changes drive the gains" (shape-aware small-N GEMV, split-K at larger batches, the shared
 * expert overlapped with routing, weight prefetch ahead of use).
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" are CUDA device pointers; "host" pointers are CPU memory.
 *  - bf16 tensors are passed as 16-bit bit patterns (any type with that layout).
 *  - FP8 matrices are OCP E4M3 codes, row-major [rows][cols], with fp32 block scales
 *    [ceil(rows/128)][ceil(cols/128)]; element (r, c) means scale[r/128][c/128] * e4m3(W[r][c]).
 *  - A `stream` argument is a cudaStream_t; NULL means the engine's own (non-blocking) stream,
 *    so the legacy default stream must be passed as cudaStreamLegacy. Consecutive steps of one
 *    engine share its counters, exchange buffers and KV cache, so they must not overlap: when a
 *    call queues work on a different stream than the engine's previous work, the library makes
 *    the new stream wait for the old one (an event), so calls of one engine run in call order
 *    whatever streams they are given. Work of other engines and other libraries is never waited
 *    for: no entry point synchronises the whole device.
 *  - Entry points that queue device work require the engine's device to be the current CUDA
 *    device (DEC_ERR_ARG otherwise).
 *  - Every call returns a dec_status. Errors found on the device (a wait that ran out of time,
 *    a failed bounds check) are reported by the next call that synchronises (dec_sync,
 *    dec_generate, dec_prefill_kv, dec_export_kv) and POISON the engine: later calls return
 *    DEC_ERR_POISONED. dec_last_error() gives a human-readable reason.
 *  - No call falls back to a CPU path: shapes the kernel does not handle give
 *    DEC_ERR_UNSUPPORTED.
 *  - The engine is not thread-safe; use one engine per host thread.
 */
#ifndef DEC_H
#define DEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dec_engine dec_engine; /* opaque, owned by the library */

typedef enum {
  DEC_OK = 0,
  DEC_ERR_ARG = -1,         /* bad argument (NULL, out of range, batch > max_batch, ...) */
  DEC_ERR_CUDA = -2,        /* a CUDA runtime call failed */
  DEC_ERR_OOM = -3,         /* device allocation failed */
  DEC_ERR_TIMEOUT = -4,     /* a device-side wait ran out of time; engine poisoned */
  DEC_ERR_UNSUPPORTED = -5, /* model shape or batch the kernel does not implement */
  DEC_ERR_POISONED = -6,    /* an earlier device error made the engine unusable */
  DEC_ERR_DEVICE = -7,      /* a device-side consistency check failed; engine poisoned */
  DEC_ERR_CAPACITY = -8     /* a sequence would exceed max_ctx */
} dec_status;

/* Model shape. The layer is a pre-norm decoder: RMSNorm -> q/k/v projection -> RoPE (half-split
   pairing) -> GQA attention over a bf16 KV cache -> output projection + residual -> RMSNorm ->
   FFN + residual. The FFN is either a dense SwiGLU of width dense_ffn (n_experts == 0), or a
   sigmoid-routed MoE: top_k of n_experts SwiGLU experts of width moe_inter with gates normalised
   over the selected scores, plus n_shared (0 or 1) always-on experts of the same width.
   ("Kimi K3: The Manos, The Mythos, The Legendos": GQA; the expert as SwiGLU; top-k over router
   scores; the residual x_{l+1} = x_l + f(x_l).) vocab == 0 builds a headless stack that maps a
   bf16 hidden state to a bf16 hidden state (no embedding, LM head or argmax). */
typedef struct {
  int32_t n_layers;   /* >= 1 */
  int32_t hidden;     /* multiple of 128 */
  int32_t n_heads;    /* query heads */
  int32_t n_kv_heads; /* KV heads; n_heads / n_kv_heads must be 2 or 4 */
  int32_t head_dim;   /* 64 or 128 */
  int32_t n_experts;  /* 0 for a dense FFN, else <= 128 */
  int32_t top_k;      /* 1..16, <= n_experts */
  int32_t moe_inter;  /* expert SwiGLU width, multiple of 128 */
  int32_t n_shared;   /* 0 or 1 */
  int32_t dense_ffn;  /* dense SwiGLU width (multiple of 128) when n_experts == 0, else 0 */
  int32_t vocab;      /* 0: headless stack */
  int32_t max_ctx;    /* KV positions per sequence */
  int32_t max_batch;  /* sequences decoded together, 1..64 (8 and more: the wide kernels) */
  float rms_eps;
  float rope_theta;
} dec_model_cfg;

/* An FP8-E4M3 matrix with its fp32 block scales (both device pointers, borrowed). */
typedef struct {
  const void* w;
  const float* scale;
} dec_fp8_mat;

/* One layer's weights. Matrix shapes (rows x cols): wq [n_heads*head_dim x hidden],
   wk/wv [n_kv_heads*head_dim x hidden], wo [hidden x n_heads*head_dim],
   router [n_experts x hidden], gate/up [inter x hidden], down [hidden x inter].
   The expert and shared arrays are HOST arrays of device matrices. */
typedef struct {
  const void* attn_norm; /* device bf16 [hidden] */
  dec_fp8_mat wq, wk, wv, wo;
  const void* ffn_norm; /* device bf16 [hidden] */
  dec_fp8_mat router;
  const dec_fp8_mat* expert_gate; /* host array [n_experts] */
  const dec_fp8_mat* expert_up;
  const dec_fp8_mat* expert_down;
  const dec_fp8_mat* shared_gate; /* host array [n_shared] */
  const dec_fp8_mat* shared_up;
  const dec_fp8_mat* shared_down;
  dec_fp8_mat ffn_gate, ffn_up, ffn_down; /* dense FFN */
} dec_layer_weights;

typedef struct {
  const void* embed;      /* device bf16 [vocab][hidden] (vocab > 0) */
  const void* final_norm; /* device bf16 [hidden] (vocab > 0) */
  dec_fp8_mat lm_head;    /* [vocab x hidden] (vocab > 0) */
  const dec_layer_weights* layers; /* host array [n_layers] */
} dec_weights;

/* Host-only check of a model shape (no CUDA needed). DEC_OK, DEC_ERR_ARG (inconsistent) or
   DEC_ERR_UNSUPPORTED (consistent but not implemented by the kernel). */
dec_status dec_validate_cfg(const dec_model_cfg* cfg);

/* Build an engine on the current CUDA device: validates the shape, copies every weight into
   library-owned memory (repacked into the kernel's tile order; the caller may free its buffers
   once the call returns), builds the RoPE table (angles in double on the host), allocates the
   KV cache [n_layers][max_batch][n_kv_heads][max_ctx][head_dim] bf16 x2 and the workspace, and
   checks that one CTA per SM can be co-resident. An engine of max_batch >= 5 also builds the
   wide kernel's buffers and two tensor maps over the K and V caches (the driver's
   cuTensorMapEncodeTiled, reached through the runtime; DEC_ERR_CUDA if it is missing). All
   sequence lengths start at 0. Work is queued on `stream` and synchronised before return. *out
   receives the engine (NULL on failure).
   Environment, read here: DEC_TIMEOUT_MS bounds every device-side wait (default 1000);
   DEC_INFLIGHT / DEC_WIDE_INFLIGHT set how many ring slots one CTA keeps in flight (defaults 2
   and 4; tuning only); DEC_WIDE_MIN_BATCH (2..9, default 5) is the smallest decode batch that
   runs the wide kernel (tuning and tests);
   DEC_TEST_SKIP_ARRIVAL=1 (tests of the failure path only) makes the CTA holding the first
   q/k/v tile withhold that partial sum's arrival in layer 0 (in a step of 5 tokens or more:
   CTA 0 its arrival at the first grid barrier), so the waits for it run out after
   DEC_TIMEOUT_MS and the step ends with DEC_ERR_TIMEOUT instead of hanging;
   DEC_EPOCH_LIMIT lowers the number of steps after which a step first zeroes the engine's
   cross-step counters and flags (a cudaMemsetAsync on the step's stream) and restarts its epoch
   (default 2^30 / the largest number of k blocks of a row block), so tests can make it happen. */
dec_status dec_init(const dec_model_cfg* cfg, const dec_weights* weights, void* stream,
                    dec_engine** out);

/* Fill the KV cache of sequence slots [seq, seq + n_seq).
   Token mode (k_import == NULL): token_ids is device int32 [n_seq][n_tokens]; appending to each
   slot's current length, the engine runs the decode kernel over the prompt and discards the
   logits: for one slot (n_seq == 1) in launches of up to DEC_MAX_STEP_TOKENS consecutive
   positions each (as dec_step_positions: every launch streams the weights once for all of its
   positions), for several slots one launch per position with the slots side by side. This is
   decode-engine prefill as on the pages' prefill/decode split, not a compute-bound prefill
   engine.
   Import mode (k_import != NULL): copies an external KV state, device bf16
   [n_layers][n_kv_heads][n_tokens][head_dim] for K (post-RoPE) and V, into positions
   0..n_tokens of every slot in the range and sets their length to n_tokens (the handoff of a KV
   cache produced elsewhere, as in the TileRT page's section "PD Disaggregated Engine with vLLM
   and TileRT"). n_tokens == 0 is a no-op in both modes. Synchronises. */
typedef struct {
  int32_t seq;
  int32_t n_seq;
  const int32_t* token_ids; /* device, token mode */
  int32_t n_tokens;
  const void* k_import; /* device, import mode */
  const void* v_import;
} dec_ctx;
dec_status dec_prefill_kv(dec_engine* eng, const dec_ctx* ctx);

/* Token-mode prefill that allocates no device memory. The pages have no counterpart: this is a
   property of the library boundary, not of the method. dec_prefill_kv's token mode stages the
   step-major token ids in a buffer it takes with cudaMalloc and returns with cudaFree; a caller
   that may not allocate device memory while serving (a framework whose caching allocator holds
   the device's free memory, or a loop in which cudaFree's implicit device-wide synchronisation
   would stall other streams) calls this instead. The ids are staged in a file-scope device
   array of DEC_NOALLOC_PREFILL_MAX_IDS int32 (256 KiB), one per device.
   - ctx must be token mode (k_import and v_import NULL); anything else is DEC_ERR_ARG.
   - n_seq * n_tokens > DEC_NOALLOC_PREFILL_MAX_IDS returns DEC_ERR_ARG, with the sizes in
     dec_last_error(), before any work is queued; split longer prompts into several calls.
   - The first call on a device does a one-time setup: with that device current it looks up the
     array's device address (cudaGetSymbolAddress) and caches it. Make that first call before
     any stream capture begins.
   - Nothing needs to start at zero: a call writes every id it reads before reading it.
   - The array is shared by all engines on a device: overlapping calls (two host threads, or two
     engines on one device) race on it; the caller must serialise them. Within one engine the
     call is stream-ordered after the engine's earlier work (no device-wide synchronisation).
   - The engine's device must be the current device (DEC_ERR_ARG otherwise).
   Results, capacity checks and synchronisation are those of dec_prefill_kv's token mode. */
#define DEC_NOALLOC_PREFILL_MAX_IDS 65536
dec_status dec_prefill_kv_noalloc(dec_engine* eng, const dec_ctx* ctx);

/* One decode step of `batch` sequences in slots [seq0, seq0 + batch). Token b is written at
   position length[seq0 + b] and attends over positions 0..length (inclusive); the lengths grow
   by one. Exactly one kernel launch on `stream`; nothing is synchronised.
     tokens      device int32 [batch]         input ids (vocab > 0)
     hidden_in   device bf16 [batch][hidden]  input hidden states (vocab == 0; also accepted
                                              with vocab > 0 in place of tokens)
     logits      device fp32 [batch][vocab]   caller-owned output, may be NULL
     next_tokens device int32 [batch]         greedy argmax (lowest id on ties), may be NULL
     hidden_out  device bf16 [batch][hidden]  final residual stream (before the final norm),
                                              may be NULL
   batch == 0 is a no-op. Errors: DEC_ERR_ARG, DEC_ERR_CAPACITY (a length would pass max_ctx),
   DEC_ERR_POISONED, DEC_ERR_CUDA (launch failure).
   Batches of 5 .. 64 (engines built with max_batch >= 5) run the wide kernel: every GEMV on the
   tensor cores with all of the step's tokens as the N dimension, tokens grouped per routed expert
   (an expert's products kept for the tokens routed to it), attention as bf16 tensor-core products
   on KV tiles loaded by tensor-map copies, phases separated by grid barriers
   ("vLLM's Kimi K3 Backend Hits 842 Tokens per Second", section "A narrow deployment lane":
   decode batches up to 64). Same arguments, results and errors. */
typedef struct {
  const int32_t* tokens;
  const void* hidden_in;
  int32_t batch;
  int32_t seq0;
  float* logits;
  int32_t* next_tokens;
  void* hidden_out;
  void* stream;
} dec_step_args;
dec_status dec_step_ex(dec_engine* eng, const dec_step_args* args);

/* The most tokens one launch takes (sequences side by side, or positions of one sequence). */
#define DEC_MAX_STEP_TOKENS 8

/* Several consecutive positions of ONE sequence in one launch ("vLLM's Kimi K3 Backend Hits 842
   Tokens per Second", section "Throughput holds across the tested range": verifying speculative
   drafts; also chunked prefill). tokens is device int32 [n], 1 <= n <= DEC_MAX_STEP_TOKENS;
   token j is written at position length[seq] + j and attends over positions 0 .. length + j
   (causal: the keys and values of the earlier tokens of the same launch included); the slot's
   length grows by n. logits device fp32 [n][vocab] and next_tokens device int32 [n] (the argmax
   after each position) are optional. One launch on `stream`; nothing is synchronised.
   Requires vocab > 0. Errors: DEC_ERR_ARG, DEC_ERR_CAPACITY, DEC_ERR_POISONED, DEC_ERR_CUDA. */
dec_status dec_step_positions(dec_engine* eng, int32_t seq, const int32_t* tokens, int32_t n,
                              float* logits, int32_t* next_tokens, void* stream);

/* Speculative-decoding verify step: as dec_step_positions with tokens = [t0, d1, .., d(n-1)], t0
   the sequence's next input token and d the draft. The kernel accepts draft d(j+1) while it equals
   the argmax after position length + j, writes the accepted count m (0 <= m < n) to the host
   int *n_accepted, and keeps the positions length .. length + m in the cache: the slot's length
   becomes length + m + 1, and next_tokens[m] (if given) is the next input token. Synchronises
   with `stream` (the caller needs m to go on). */
dec_status dec_verify(dec_engine* eng, int32_t seq, const int32_t* tokens, int32_t n, float* logits,
                      int32_t* next_tokens, int32_t* n_accepted, void* stream);

/* The plain form: slots [0, batch), token input, logits/next_tokens outputs (may be NULL). */
dec_status dec_step(dec_engine* eng, const int32_t* token_ids, int32_t batch, float* logits,
                    int32_t* next_tokens, void* stream);

/* Greedy generation from HOST buffers: copies first_tokens (host int32 [batch]) to the device,
   runs n_steps greedy decode steps of slots [0, batch) in ONE launch of a resident kernel ("Ultra-
   High Interactivity on NVIDIA GPUs? TileRT on InferenceX", section "But What Exactly is
   TileRT?": the host launches once and execution stays on the GPU for the decode lifecycle):
   step i's argmax becomes step i+1's input through device memory and a flag, and the producer
   warps stream the next step's first weights while the LM head finishes. Copies the generated
   tokens back to out_tokens (host int32 [n_steps][batch]) and synchronises. Requires vocab > 0
   and length + n_steps <= max_ctx for every slot (DEC_ERR_CAPACITY otherwise). (A generation of
   more steps than the engine's epoch period takes one launch per period; batches of 5 and more
   take one wide-kernel launch per step, the tokens still chained on the device.) */
dec_status dec_generate(dec_engine* eng, const int32_t* first_tokens, int32_t batch,
                        int32_t n_steps, int32_t* out_tokens, void* stream);

/* The same resident generation with DEVICE buffers (first_tokens device int32 [batch],
   out_tokens device int32 [n_steps][batch]); queued on `stream`, nothing synchronised. */
dec_status dec_generate_device(dec_engine* eng, const int32_t* first_tokens, int32_t batch,
                               int32_t n_steps, int32_t* out_tokens, void* stream);

/* Sequence lengths (positions already in the cache). Setting a length rewinds or advances a
   slot without touching the cache contents. */
dec_status dec_set_length(dec_engine* eng, int32_t seq, int32_t length);
dec_status dec_get_length(dec_engine* eng, int32_t seq, int32_t* length);

/* Copy positions [pos0, pos0 + n) of one slot and layer out of the KV cache into device bf16
   buffers k_out/v_out [n_kv_heads][n][head_dim]. Synchronises. */
dec_status dec_export_kv(dec_engine* eng, int32_t seq, int32_t layer, int32_t pos0, int32_t n,
                         void* k_out, void* v_out);

/* Wait for all queued engine work and read the device status word. */
dec_status dec_sync(dec_engine* eng);

/* Engine facts for tools and benchmarks. */
typedef struct {
  int32_t grid;           /* persistent CTAs (one per SM) */
  int32_t threads;        /* threads per CTA */
  int32_t smem_bytes;     /* dynamic shared memory per CTA */
  int32_t ring_slots;     /* stages of the shared-memory weight ring */
  int32_t stages_per_layer;
  int64_t weight_bytes;   /* repacked weight bytes held by the engine */
  int64_t kv_bytes;       /* KV cache bytes */
  int64_t workspace_bytes;
  int64_t launches;       /* kernel launches issued by this engine so far */
  int32_t wide_min_batch; /* decode steps of at least this many tokens run the wide kernel
                             (a value above max_batch: none does) */
} dec_info;
dec_status dec_get_info(dec_engine* eng, dec_info* out);

/* Routing of the most recent step at one layer (MoE models): copies the selected experts
   (score-descending) into host idx [R][top_k] and their normalised gates into host gates
   [R][top_k], R = max(DEC_MAX_STEP_TOKENS, max_batch), one row per token of the step; rows >=
   the step's token count are stale. Synchronises. */
dec_status dec_get_routing(dec_engine* eng, int32_t layer, int32_t* idx, float* gates);

/* The router logits (fp32, before the sigmoid) the most recent step selected from at one layer
   (MoE models): host logits [R][n_experts], R = max(DEC_MAX_STEP_TOKENS, max_batch); rows >=
   the step's token count are stale. With
   dec_get_routing this lets a caller check that a selection is the top_k of its own logits
   (ties to the lower expert index). Synchronises. */
dec_status dec_get_router_logits(dec_engine* eng, int32_t layer, float* logits);

/* Diagnostics of the last step, recorded only by a library built with DEC_TRACE=1 /
   DEC_STAMPS=1 (`DEC_DIAG=1` when running latency_moe_decode_gb300/build.py; the default build
   records nothing, its words stay zero: the stores cost the step ~4% in instruction fetch).
   Per-step trace written by CTA 0: (event code, %globaltimer ns) pairs in host_buf[2i], [2i+1].
   code = what << 4 | event; what: 0 q/k/v GEMV, 1 output projection, 2 router, 3 shared-expert
   (or dense FFN) gate/up, 4 routed gate/up, 5 down projections, 6 LM head, 7 attention, 8 grid
   barrier, 9 routing wait, 10 step; event: 0 begin, 1 last tile consumed, 2 finalisers done
   (barrier: its site). Words [512 - 128, 512) hold CTA 0's producer trace in the same format.
   With DEC_STAMPS=1, words from 512 on hold per-CTA %globaltimer stamps of the first 8 layers:
   word
   512 + (layer * 16 + point) * grid + cta, for the points q/k/v tiles consumed (0), q/k/v done
   (1), attention merged (2), attention outputs ready (3), output-projection tiles consumed (4)
   and done (5), x_mid ready (6), router partials published (7), routing known (8), gate/up
   tiles consumed (9) and done (10), SwiGLU rows ready (11), down tiles consumed (12) and done
   (13), layer barrier passed (14). Copies up to n words and returns the count in *n_written.
   Synchronises. */
dec_status dec_get_trace(dec_engine* eng, uint64_t* host_buf, int32_t n, int32_t* n_written);

/* Per-layer timing of the most recent step, recorded in every build by one thread of the first
   CTA: host_buf[l] is the %globaltimer time (ns) at which the input of layer l was final, as
   that CTA saw it (l = 0: the step start; l = n_layers: the final norm's input), and
   host_buf[n_layers + 1] the time that CTA finished the step. So host_buf[l + 1] - host_buf[l]
   is layer l's time on the critical path and the last difference the LM head's tail. Copies
   min(n, n_layers + 2) words and returns the count in *n_written. Synchronises with the
   engine's work. */
dec_status dec_get_layer_times(dec_engine* eng, uint64_t* host_buf, int32_t n, int32_t* n_written);

/* Reason for the last failing call on this engine ("" if none). Valid until the next call. */
const char* dec_last_error(const dec_engine* eng);

/* Fixed string naming a status code. */
const char* dec_status_string(dec_status s);

/* Release every device buffer of the engine (synchronises first). NULL is a no-op. */
void dec_destroy(dec_engine* eng);

#ifdef __cplusplus
}
#endif
#endif /* DEC_H */
