/* llmq — GB300-native per-token decode step of a Llama/Qwen-style decoder with
 * group-64 4-bit weights (W4A16), behind a plain C ABI.
 *
 * The operation is the decode step the aot-llm page ("p10node/aot-llm") draws
 * in its sequence diagram and "static pipeline": embedding -> [RMSNorm ->
 * q/k/v matvec -> RoPE -> attention over the KV cache -> o matvec + residual
 * -> RMSNorm -> gate/up -> SwiGLU -> down + residual] x L -> RMSNorm -> logits
 * -> greedy choice. Weights are "packed group-64 W4A16" (llmopt page); the KV
 * cache is bf16 appended from f32 (zynfer page, stage M4). The shape of the
 * API follows aot-llm's C library section (open a model, evaluate tokens, read
 * n_vocab logits, reset a context) and the pytensor-ml issue's "immutable
 * model, mutable context" and "fail at load with the missing capability named".
 *
 * Conventions for every entry point:
 *   - returns LLM_OK (0) or a negative llm_status; llm_last_error() then holds
 *     a one-line reason. LLM_ERR_CUDA and LLM_ERR_TIMEOUT poison the model
 *     (every later call returns the same error); all other errors leave it
 *     usable.
 *   - a model is not thread-safe: the caller serialises calls on one model.
 *   - output pointers marked "host or device" may point to either; the call
 *     is synchronous when any output is in host memory.
 *   - all device memory is owned by the library and allocated once, in
 *     llm_model_create; no call in the token loop allocates.
 */
#ifndef LLMQ_H
#define LLMQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LLMQ_ABI_VERSION 1

typedef enum {
  LLM_OK = 0,
  LLM_ERR_INVALID_ARG = -1,   /* null pointer, out-of-range index, bad size */
  LLM_ERR_UNSUPPORTED = -2,   /* config the kernels do not cover; message names it */
  LLM_ERR_OOM = -3,           /* device allocation failed at create */
  LLM_ERR_CTX_FULL = -4,      /* position would reach max_seq */
  LLM_ERR_CUDA = -5,          /* CUDA runtime error (poisons the model) */
  LLM_ERR_TIMEOUT = -6,       /* a device-side wait hit its limit (poisons the model) */
  LLM_ERR_NAN = -7,           /* the logit reduction saw a NaN */
  LLM_ERR_NOT_FOUND = -8      /* tensor name unknown */
} llm_status;

typedef enum { LLM_F32 = 0, LLM_BF16 = 1, LLM_F16 = 2, LLM_Q4G64 = 3 } llm_dtype;

/* llm_config.flags */
#define LLM_NO_GRAPH 1u       /* launch the step's kernels one by one (debugging) */
#define LLM_NO_PDL   2u       /* no programmatic dependent launch between kernels */
#define LLM_MULTI_KERNEL 4u   /* one kernel per phase instead of the persistent step kernel */
#define LLM_TEST_EXPIRE_WAIT 0x80000000u  /* test only: every grid barrier of the persistent step
                                 waits for one arrival too many with a 1 ms limit, so the first one
                                 expires; the call returns LLM_ERR_TIMEOUT (nothing faults or hangs) */
#define LLM_DEBUG_BATCH_HIDDEN 16u  /* keep every layer's residual of the last batched decode step
                                 for llm_debug_hidden_batch (adds L+1 device copies to the step) */
#define LLM_W4A8 64u          /* 4-bit weights x int8 activations in the batch-1 paths: every 4-bit GEMV
                                 input quantized once per 32-input block (fp16 scale amax/127, codes
                                 round(x/scale) clamped to +-127) and dotted in integers; the batched
                                 kernels keep their fp16 tensor-core inputs. Not with LLM_DATAFLOW_STEP */
#define LLM_KV_Q8 128u        /* grouped int8 K/V cache (llmopt README, "Current compiler and runtime":
                                 grouped-Q8 attention state): each 32 values of a (position, kv head)
                                 row stored as int8 codes with one fp16 scale fp16(amax/127), codes
                                 round(x/scale) half away from zero clamped to +-127, decided in fp32;
                                 attention reads the codes and scales. Persistent step only (not with
                                 LLM_MULTI_KERNEL or LLM_DATAFLOW_STEP); llm_kv_write quantizes its bf16
                                 rows the same way, llm_kv_read_q8 reads codes and scales */
#define LLM_DATAFLOW_STEP 8u  /* greedy batch-1 steps on the flag-synchronised persistent kernel (phases
                                 wait on flagged words instead of grid barriers; slower than the
                                 default grid-barrier step on GB300, kept for comparison) */

typedef struct {
  int32_t abi_version;        /* must equal LLMQ_ABI_VERSION */
  int32_t dim, n_layers, n_heads, n_kv_heads, head_dim, ffn_dim, vocab;
  float   norm_eps;           /* RMSNorm epsilon */
  int32_t rope_neox;          /* 0: rotate pairs (2i, 2i+1); 1: pairs (i, i + head_dim/2) */
  double  rope_theta;         /* RoPE base: theta_i = base^(-2i/head_dim) */
  int32_t qk_norm;            /* 1: per-head RMSNorm of q and k before RoPE (Qwen3) */
  int32_t tied_embedding;     /* 1: LM head is the bf16 embedding table */
  int32_t max_seq;            /* KV capacity per sequence (positions) */
  int32_t max_batch;          /* number of sequences (independent caches) */
  uint32_t flags;             /* LLM_NO_GRAPH | LLM_NO_PDL | LLM_MULTI_KERNEL | LLM_DATAFLOW_STEP |
                                 LLM_DEBUG_BATCH_HIDDEN | LLM_W4A8 | LLM_KV_Q8 | LLM_TEST_EXPIRE_WAIT */
} llm_config;

/* One input tensor in the canonical layout, host memory, caller-owned, only
 * read during llm_model_create (the caller may free it afterwards).
 *   LLM_Q4G64 linear [rows=out][cols=in], cols % 64 == 0:
 *       codes  uint8 [rows][cols/2], element 2j in the low nibble of byte j,
 *                    element 2j+1 in the high nibble;
 *       scales fp16  [rows][cols/64];  mins fp16 [rows][cols/64];
 *       weight w[r][c] = scale[r][c/64] * q + min[r][c/64].
 *   LLM_F32 / LLM_BF16 dense [rows][cols] in `data` (norm weights: rows = 1).
 * Names: "embed" (f32, or bf16 when tied) [vocab][dim]; "final_norm";
 * per layer l: "L{l}.attn_norm", "L{l}.ffn_norm", "L{l}.q_norm", "L{l}.k_norm"
 * (qk_norm only, [head_dim]); q4 "L{l}.wq" [n_heads*head_dim][dim],
 * "L{l}.wk", "L{l}.wv" [n_kv_heads*head_dim][dim], "L{l}.wo"
 * [dim][n_heads*head_dim], "L{l}.w_gate", "L{l}.w_up" [ffn_dim][dim],
 * "L{l}.w_down" [dim][ffn_dim]; "lm_head" q4 [vocab][dim] when untied. */
typedef struct {
  const char* name;
  int32_t dtype;              /* llm_dtype */
  int64_t rows, cols;
  const void* codes;          /* LLM_Q4G64 */
  const void* scales;
  const void* mins;
  const void* data;           /* LLM_F32 / LLM_BF16 */
} llm_tensor;

typedef struct llm_model llm_model;

typedef struct {
  int64_t device_bytes;       /* all device memory owned by the model */
  int64_t weight_stream_bytes;/* repacked weight bytes read per decode step */
  int64_t kv_bytes_per_pos;   /* bf16 K+V bytes per cached position, all layers */
  int32_t kernels_per_step;   /* kernel nodes in one batch-1 step */
  int32_t n_sm;               /* SMs of the device the model lives on */
} llm_stats;

/* Validate the config, repack the 4-bit weights into the GPU tile layout, copy
 * everything to the device, size all buffers and capture the step graph.
 * cuda_stream: cudaStream_t to run on, or NULL for a stream the model owns.
 * Errors: INVALID_ARG, UNSUPPORTED (head_dim not 64/128, cols % 64, heads not
 * divisible, missing tensor...), NOT_FOUND, OOM, CUDA. On error *out = NULL.
 * Source: aot-llm README, "Library output" and its C example (aot_open: the model opened once, weights
 * ready); pytensor-ml issue #53, "Acceptance rules that apply to every PR" (fail at load with the
 * missing capability named). */
int llm_model_create(const llm_config* cfg, const llm_tensor* tensors, int32_t n_tensors,
                     void* cuda_stream, llm_model** out);

/* Free every device allocation of the model. NULL is accepted.
 * Source: no page counterpart: the model owns its device memory (pytensor-ml issue #53, "Already
 * here": immutable model, mutable context). */
void llm_model_destroy(llm_model* m);

/* Append n tokens (host array) to sequence seq at positions len..len+n-1 and
 * return the last position's fp32 logits [vocab] and greedy token. Runs n
 * decode steps. logits_out / argmax_out: host or device, may be NULL.
 * Errors: INVALID_ARG, CTX_FULL (len + n > max_seq), NAN, CUDA, TIMEOUT.
 * Source: aot-llm README C example (aot_eval of n prompt tokens, then aot_logits: n_vocab floats); the
 * static pipeline emitted for every model (aot-llm README) run once per token. */
int llm_prefill(llm_model* m, int32_t seq, const int32_t* tokens, int32_t n,
                float* logits_out, int32_t* argmax_out);

/* The same contract as llm_prefill, computed as batched prompt processing
 * (aot-llm "Batched prompt processing": each weight row read once per chunk of
 * tokens; llmopt "prefill-style GEMM"): chunks of up to 32 tokens go through
 * the batched pipeline (4-bit skinny GEMMs on the tensor cores, fp32
 * accumulation) with the chunk's rows appending their k, v to the cache first
 * and then attending causally over it. Equal to token-by-token prefill within
 * floating-point tolerance (a different summation order); the greedy token is
 * the argmax of the returned logits. llm_debug_hidden is not updated.
 * Errors as llm_prefill. */
int llm_prefill_batched(llm_model* m, int32_t seq, const int32_t* tokens, int32_t n,
                        float* logits_out, int32_t* argmax_out);

/* One decode step of sequence seq for `token` at position len; len += 1.
 * logits_out [vocab] fp32 and argmax_out (lowest index wins ties): host or
 * device, may be NULL. Errors as llm_prefill.
 * Source: aot-llm README, "The static pipeline emitted for every model" and its C example (one token
 * through aot_eval, aot_logits); pytensor-ml issue #53 (one-token append to the cache). */
int llm_decode_step(llm_model* m, int32_t seq, int32_t token, float* logits_out,
                    int32_t* argmax_out);

/* n_steps greedy steps starting from first_token; each step's argmax feeds the
 * next step on the device (no host round trip per step). tokens_out
 * [n_steps] (host or device) receives the token chosen at each step.
 * Source: zynfer PR #100, stage M3 (one command buffer per forward, 2 waits per token instead of 476:
 * the step runs on the device without a host round trip). */
int llm_decode_greedy(llm_model* m, int32_t seq, int32_t first_token, int32_t n_steps,
                      int32_t* tokens_out);

/* Sampled instead of greedy next-token choice for the batch-1 calls
 * (llm_prefill, llm_prefill_batched, llm_decode_step, llm_decode_greedy), from
 * the options the aot-llm page lists ("Generated binary options": temperature,
 * 0 = greedy; top-k; top-p; seed). Keep the top_k largest logits (ties: lower
 * token id), p = softmax((l - l_max) / temperature), keep the shortest prefix
 * whose cumulative probability reaches top_p, and take the first token whose
 * cumulative probability exceeds u times the prefix total. The draw u for the
 * token after position pos of sequence seq is Philox4x32-10 (Salmon et al.,
 * SC 2011) of counter (pos, seq, 0, 0) and key (seed low, seed high word):
 * u = (x0 >> 8) / 2^24, reproducible from the seed. The chosen token is what
 * argmax_out / tokens_out return and what llm_decode_greedy feeds back.
 * temperature 0 restores the greedy choice. llm_decode_step_batch stays
 * greedy. Errors: INVALID_ARG (temperature < 0 or not finite; when sampling,
 * top_k outside 1..64 or top_p outside (0, 1]). */
int llm_set_sampling(llm_model* m, float temperature, int32_t top_k, float top_p, uint64_t seed);

/* One decode step for sequences 0..n_seq-1 at once (n_seq == max_batch >= 2,
 * at most 32), each at its own position (its cache may come from
 * llm_kv_write or llm_prefill). The 4-bit matvecs become skinny GEMMs (fp32
 * register tiles, each weight dequantised once for every sequence); attention
 * runs over every sequence's own cache length. tokens [n_seq] (host or
 * device), or NULL to continue every sequence from its previous greedy token
 * on the device; logits_out [n_seq][vocab] and argmax_out [n_seq]: host or
 * device, may be NULL. Synchronous when tokens or an output are host memory.
 * Errors: UNSUPPORTED (max_batch < 2), INVALID_ARG, CTX_FULL, NAN, CUDA.
 * Source: no page decodes several sequences at once; this applies the batched prompt path of the
 * aot-llm README ("Batched prompt processing": each weight row read once for a chunk of tokens) to one
 * token of each sequence. */
int llm_decode_step_batch(llm_model* m, const int32_t* tokens, int32_t n_seq,
                          float* logits_out, int32_t* argmax_out);

/* Forget the cache of sequence seq (-1: all); its length becomes 0.
 * Source: aot-llm README C example (aot_ctx_reset). */
int llm_kv_reset(llm_model* m, int32_t seq);

/* Copy bf16 keys/values [n][n_kv_heads][head_dim] (host or device) into
 * positions pos0..pos0+n-1 of one layer of sequence seq; keys are stored as
 * given (already rotated). The sequence length becomes max(len, pos0 + n).
 * Errors: INVALID_ARG, CTX_FULL.
 * Source: aot-llm README (aot_ctx_save / aot_ctx_load move a conversation's cache between processes);
 * zynfer PR #100, stage M4 (bf16 KV cache appended from f32). */
int llm_kv_write(llm_model* m, int32_t seq, int32_t layer, int32_t pos0, int32_t n,
                 const uint16_t* k_bf16, const uint16_t* v_bf16);

/* Read back bf16 keys/values [n][n_kv_heads][head_dim] (host or device).
 * Source: as llm_kv_write. */
int llm_kv_read(llm_model* m, int32_t seq, int32_t layer, int32_t pos0, int32_t n,
                uint16_t* k_bf16, uint16_t* v_bf16);

/* Read back an int8 cache (LLM_KV_Q8 models): codes k, v [n][n_kv_heads][head_dim]
 * and fp16 scale bits ks, vs [n][n_kv_heads][head_dim / 32], host or device.
 * Source: llmopt README, "Current compiler and runtime" (grouped-Q8 attention state). */
int llm_kv_read_q8(llm_model* m, int32_t seq, int32_t layer, int32_t pos0, int32_t n, int8_t* k, uint16_t* ks,
                   int8_t* v, uint16_t* vs);

/* Current cache length of sequence seq, or a negative llm_status.
 * Source: pytensor-ml issue #53, "Already here" (the cache and its one-token append). */
int llm_kv_len(const llm_model* m, int32_t seq);

/* Residual stream after the embedding and after every layer of the last
 * batch-1 step: out [(n_layers+1)][dim] fp32, host or device.
 * Source: pytensor-ml issue #53, "Acceptance rules that apply to every PR" (an independent oracle, the
 * cached output checked at every step). */
int llm_debug_hidden(llm_model* m, float* out);

/* Residual stream of every sequence after the embedding and after every layer
 * of the last llm_decode_step_batch: out [(n_layers+1)][max_batch][dim] fp32,
 * host or device. Needs a model created with LLM_DEBUG_BATCH_HIDDEN
 * (else LLM_ERR_UNSUPPORTED).
 * Source: as llm_debug_hidden. */
int llm_debug_hidden_batch(llm_model* m, float* out);

/* Undo the repack of one 4-bit tensor: write its canonical codes [rows][cols/2],
 * scales and mins [rows][cols/64] (host) from the device copy.
 * Source: aot-llm README, testing section (every dot product and weight type checked against a scalar
 * reference). */
int llm_debug_unpack(llm_model* m, const char* name, uint8_t* codes, uint16_t* scales,
                     uint16_t* mins);

/* Test hook: the nth device allocation (counted from 1) made by the models
 * created after this call fails as if cudaMalloc had run out of memory, so
 * llm_model_create returns LLM_ERR_OOM naming the buffer and frees what it
 * had allocated. nth <= 0 disarms it. Process-wide; returns LLM_OK.
 * Source: zynfer PR #100, stage M6 (allocation behaviour tested with a failing allocator). */
int llm_debug_fail_alloc(int32_t nth);

/* Sizes and counts of the model (host struct).
 * Source: zynfer PR #100, stages M2-M4 (bytes per token for the roofline estimate). */
int llm_model_stats(const llm_model* m, llm_stats* out);

/* One launch of a decode step, as timed by llm_profile_step. */
typedef struct {
  int32_t kind;               /* 0 4-bit GEMV, 1 bf16 GEMV, 2 attention, 3 logits/argmax */
  int32_t layer;              /* -1 for the LM head and the argmax */
  int64_t bytes;              /* algorithmic HBM bytes: weight units, or K/V rows read */
  float   ms;                 /* CUDA-event duration on the model's stream */
} llm_kernel_time;

/* Run one decode step of `token` like llm_decode_step, but eagerly and
 * without programmatic dependent launch, with a CUDA event pair around every
 * kernel. Writes up to max_out records (launch order) and returns the number
 * of launches, or a negative llm_status. Meant for measurement, not the token
 * loop (it creates and destroys events).
 * Source: zynfer PR #100, stage M2 (per-family timing and a roofline JSON). */
int llm_profile_step(llm_model* m, int32_t seq, int32_t token, llm_kernel_time* out, int32_t max_out);

/* Time back-to-back launches of the batch-1 step's kernels of sequence seq
 * (programmatic dependent launch between them, CUDA events on the model's
 * stream) on the buffers the last step left. which = 0 q|k|v GEMV, 1
 * attention, 2 o GEMV, 3 gate|up GEMV, 4 down GEMV: that kernel for `layer`,
 * or for every layer in turn when layer = -1 (so that a weight set larger than
 * L2 is streamed); 5 the LM-head GEMV; 6 every 4-bit/bf16 GEMV of one step in
 * step order. The list is launched n times. Attention launches re-append the
 * last position with the values already there. Writes the mean milliseconds
 * per launch and the mean algorithmic bytes per launch. Needs at least one
 * completed step of seq.
 * Source: as llm_profile_step. */
int llm_time_kernel(llm_model* m, int32_t seq, int32_t which, int32_t layer, int32_t n, float* ms,
                    int64_t* bytes);

/* On a model without LLM_DATAFLOW_STEP, in a library built with
 * LLMQ_PHASE_STAMPS=1 (else LLM_ERR_UNSUPPORTED): one step (n_steps = 1) of
 * the grid-barrier persistent step, recording per (phase, CTA) the clock64
 * stamps 0 phase start, 1 grid barrier passed, 2 input built, 3 weight units
 * done, 4 arrival issued (0 where a phase has no such point), and with
 * LLMQ_UNIT_STAMPS=1 also 5..8 the largest and summed per-warp cycles waiting
 * for units and in unit dots; values 12..15 of phase 0's records hold
 * (%globaltimer, clock64) at each CTA's start and end; out [phases][n_sm][16].
 * Otherwise: run n_steps (1..8) greedy steps of sequence seq from first_token through the
 * flag-synchronised step kernel in one launch and record, for every (step,
 * phase, CTA), 16 values: the SM cycle counter (clock64) when the phase's
 * input build starts, when its inputs have all arrived, when the build is
 * done, when the phase's weight units are done and when its outputs are
 * published (the LM head's stays 0); the largest and the summed per-warp
 * cycles spent waiting for weight units and computing unit dots; values 12..15
 * of the CTA's (step 0, phase 0) record hold (%globaltimer ns, clock64) at the
 * kernel's start and end, which map its cycles onto one time line.
 * out [n_steps][phases][n_sm][16] (host); phases are the four GEMVs of every
 * layer (q|k|v, o with the attention in its build, gate|up, down) and the LM
 * head. Returns the number of records (n_steps * phases * n_sm) or a negative
 * llm_status (UNSUPPORTED when the step kernel does not cover these
 * positions). len += n_steps. For measurement, not the token loop.
 * Source: as llm_profile_step. */
int llm_phase_times(llm_model* m, int32_t seq, int32_t first_token, int32_t n_steps, uint64_t* out,
                    int64_t max_out);

/* Wait for all queued work of the model and report device-side errors.
 * Source: pytensor-ml issue #53, "Acceptance rules that apply to every PR" (errors reported, not
 * swallowed). */
int llm_sync(llm_model* m);

/* Last error text of the model (m may be NULL: the last create error of this
 * thread). Never NULL; owned by the library.
 * Source: as llm_sync. */
const char* llm_last_error(const llm_model* m);

/* Kernel-level check: y = W x through the same repack and dequant-GEMV kernel
 * the decode step uses (plain store epilogue). w: one LLM_Q4G64 or LLM_BF16
 * tensor (host, cols a multiple of 64 up to 8192); x [cols], y [rows] fp32
 * host arrays. Allocates and frees its
 * own device memory; not for the token loop.
 * Source: aot-llm README, testing section (every matrix product against a float reference). */
int llm_op_matvec(const llm_tensor* w, const float* x, float* y);

/* llm_op_matvec in the W4A8 numerics of LLM_W4A8 (Q4G64 tensors only): x is
 * quantized per 32-input block to int8 with an fp16 scale (aot-llm README,
 * implementation notes: the f32 activation vector quantized once to Q8_0,
 * integer dot products scaled back to f32), each block's integer sums
 * scaled by its d and the group's scale and min. */
int llm_op_matvec_w4a8(const llm_tensor* w, const float* x, float* y);

/* y = W x with one weight matrix already resident in model m, without any
 * device allocation. No page has a counterpart: it exists for callers that
 * cannot call cudaMalloc at this point -- a process whose device memory was
 * handed to its own pool at start-up (a new cudaMalloc would fail or bypass
 * the pool's accounting), or a latency-critical loop where cudaMalloc/cudaFree
 * would stall (cudaFree synchronises the device). The caller passes x [cols]
 * and y [rows] as fp32 device buffers (y must not overlap x) on the model's
 * device, which must be the current device; `name` is a 4-bit tensor stored
 * as a contiguous row range ("L{l}.wq", "L{l}.wk", "L{l}.wv", "L{l}.wo",
 * "L{l}.w_down", "lm_head") or "embed" for a tied bf16 LM head.
 * Scratch (split-row-tile partial sums, arrival counters, a status word) lives
 * in one file-scope device array of 4 MiB + 128 KiB + 256 B that every GPU
 * loading the library keeps until exit; a matrix needing more partial-sum or
 * counter space is rejected with LLM_ERR_UNSUPPORTED naming both sizes (the
 * model stays usable). The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) and keeps it for the process: it does not
 * survive cudaDeviceReset, after which this call must not be used again.
 * Every call shares the array and clears its counters and status on
 * `cuda_stream` (NULL: the legacy default stream) before the kernel: calls
 * whose work overlaps on the GPU race on it, so serialise them. The call is
 * synchronous -- it reads the status word back and synchronises
 * `cuda_stream`, returning after y is written -- so it cannot be captured
 * into a graph: on a capturing stream it returns LLM_ERR_INVALID_ARG without
 * touching the stream or the model. Device ordinals of 64 and above:
 * LLM_ERR_UNSUPPORTED. */
int llm_matvec_noalloc(const llm_model* m, const char* name, const float* x, float* y, void* cuda_stream);

#ifdef __cplusplus
}
#endif
#endif /* LLMQ_H */
