/*
 * sab.h -- C ABI of libsab.so: streaming chunk attention over a rolling ring
 * KV cache, for NVIDIA GB300 (sm_103a).
 *
 * What the library computes
 * -------------------------
 * Streaming autoregressive video-diffusion world models generate a video
 * chunk by chunk.  Inside every transformer block the queries of the current
 * chunk attend
 *   - bidirectionally to the keys of their own chunk, and
 *   - causally to the keys of the W chunks before it, held in a rolling KV
 *     cache, plus optionally a permanent sink / reference chunk.
 * ("WanToFight: Real-Time Generative Game Engine for Multi-Player Combat
 * Interaction", section 三, table "模型组件", rows "Block-Causal Attention" and
 * "Rolling KV Cache"; "Matrix-Game 4.0: Harnessing Video Models for Real-Time
 * Playable Game Worlds", sections "前置知识 / 因果自回归与 KV 缓存" and
 * "技术新颖性".)  The cache is a ring: chunk c lives in slot c mod R and a new
 * chunk overwrites the oldest slot in place ("Matrix-Game 4.0", section
 * "技术新颖性": in-place overwrite of the oldest slot instead of a whole-window
 * copy).  Optionally the KV cache is stored as FP8 E4M3 with one fp32 scale
 * per (batch, head, chunk) and tensor ("Matrix-Game 4.0", section
 * "技术新颖性": 8-bit keys/values per window interval).
 *
 * For query token i of chunk c and visible key set J(c):
 *   s_ij  = softmax_scale * <q_i, k_j>
 *   O_i   = sum_j softmax_j(s_ij) v_j,   LSE_i = ln sum_{j in J(c)} exp(s_ij)
 * J(c) = sink tokens (if used) + tokens of chunks max(0, c-W) .. c.
 *
 * Conventions for every call
 * --------------------------
 * - Element types: Q, K, V, O are bf16 (stored as uint16 bit patterns); LSE is
 *   fp32; the FP8 cache stores E4M3 codes as uint8 and fp32 scales.
 * - Token-major tensors ("[B, L, H, D]") are contiguous, row-major, last index
 *   fastest: element (b, t, h, d) at ((b*L + t)*H + h)*D + d.  This is the
 *   layout a fused QKV projection produces.
 * - Pointers named "device" point to device memory of the current CUDA device;
 *   every device pointer must be 16-byte aligned.  The caller owns all device
 *   memory (ring, inputs, outputs, workspace); the library owns only the small
 *   host handle of a ring.
 * - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *   asynchronous on that stream and never synchronises the host, except
 *   sab_get_last_device_error.  No call allocates device memory.
 * - Arguments are validated before anything is enqueued: on any error code
 *   nothing is launched and no memory is touched.  No C++ exception crosses
 *   this ABI.
 * - Supported shapes: head_dim D in {64, 128}; chunk_tokens >= 1; every other
 *   extent >= 1 and small enough that row counts fit in int32.
 */
#ifndef SAB_H_
#define SAB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SAB_OK = 0,
  SAB_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad shape or value   */
  SAB_ERR_UNSUPPORTED = 2,   /* valid request this build does not implement   */
  SAB_ERR_OUT_OF_RANGE = 3,  /* chunk not held by the ring / bad chunk order  */
  SAB_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required    */
  SAB_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed             */
  SAB_ERR_TIMEOUT = 6,       /* a device-side pipeline wait gave up (see sab_get_last_device_error) */
  SAB_ERR_BOUNDS = 7         /* debug builds: a device-side index check failed (ditto) */
} sab_status;

/*
 * KV cache element type.
 *   SAB_KV_BF16        keys and values in bf16.
 *   SAB_KV_FP8_E4M3    keys and values as E4M3 codes, one fp32 absmax scale
 *                      (amax / 448) per (batch, head, chunk) and tensor.
 *   SAB_KV_INT8K_FP8V  keys as INT8 codes with scale amax / 127 (symmetric,
 *                      round half to even, clamped to +-127), values as E4M3
 *                      codes with scale amax / 448 ("Matrix-Game 4.0", section
 *                      "技术新颖性": each window interval caches INT8 keys and
 *                      FP8 values; only the changed interval is re-quantised).
 * Both 8-bit forms keep one byte per element in the ring and are expanded
 * exactly to bf16 on chip; the scales are applied in fp32.
 */
typedef enum { SAB_KV_BF16 = 0, SAB_KV_FP8_E4M3 = 1, SAB_KV_INT8K_FP8V = 2 } sab_kv_dtype;

/* Shape of one ring KV cache with `num_layers` independent per-layer rings. */
typedef struct {
  int num_layers;    /* transformer blocks sharing the ring geometry (>= 1)       */
  int batch;         /* B                                                          */
  int heads;         /* H                                                          */
  int head_dim;      /* D, 64 or 128                                               */
  int chunk_tokens;  /* Lc, tokens per chunk                                       */
  int ring_slots;    /* R, cached chunks (the rolling window's capacity)          */
  int has_sink;      /* 1: reserve a permanent sink/reference slot, else 0         */
  int kv_dtype;      /* sab_kv_dtype                                               */
} sab_ring_desc;

typedef struct sab_ring sab_ring; /* opaque host handle */

/*
 * Device memory layout of a ring (informative; use sab_kv_ring_layer_ptrs):
 * per layer, 256-byte aligned regions
 *   K codes  [B][H][(has_sink + R) * Lc][D]   (bf16, or one byte: E4M3 / INT8)
 *   V codes  same                             (bf16, or one byte: E4M3)
 *   K scales [B][H][has_sink + R] fp32        (8-bit forms only)
 *   V scales same                             (8-bit forms only)
 * Rows [0, Lc) hold the sink when has_sink; slot r holds rows
 * [(has_sink + r) * Lc, (has_sink + r + 1) * Lc).
 */

/* Bytes of device memory a ring with this shape needs; 0 if the shape is invalid. */
size_t sab_kv_ring_bytes(const sab_ring_desc* desc);

/*
 * Create a ring on caller-owned device memory `dev_mem` (`bytes` >=
 * sab_kv_ring_bytes, 256-byte aligned).  Enqueues a zero fill of the whole
 * region on `stream` (so slots never written hold finite zeros) and returns a
 * new host handle in *out.  The handle records, per layer, the newest chunk
 * appended (none yet) and whether the sink is set.
 */
sab_status sab_kv_ring_create(const sab_ring_desc* desc, void* dev_mem, size_t bytes,
                              void* stream, sab_ring** out);

/* Free the host handle only (the device memory stays the caller's). NULL is a no-op. */
sab_status sab_kv_ring_destroy(sab_ring* ring);

/* Copy of the descriptor the ring was created with. */
sab_status sab_kv_ring_get_desc(const sab_ring* ring, sab_ring_desc* desc);

/*
 * Device pointers of layer `layer`'s regions (any output may be NULL).  The
 * scale pointers are NULL for a BF16 ring.  Intended for checkpointing and
 * tests: the memory is the caller's.
 */
sab_status sab_kv_ring_layer_ptrs(const sab_ring* ring, int layer, void** k, void** v,
                                  float** k_scale, float** v_scale);

/*
 * Write the sink / reference chunk of `layer` ("Matrix-Game 4.0", section
 * "前置知识 / 因果自回归与 KV 缓存": recent window plus a reference frame; it is
 * never evicted).  K, V: device, token-major [B, Lc, H, D] bf16.  For an FP8
 * ring they are quantised exactly as sab_kv_ring_append does.
 * Errors: INVALID_ARG (null/misaligned, layer out of range),
 * UNSUPPORTED (ring has no sink slot).
 */
sab_status sab_kv_ring_set_sink(sab_ring* ring, int layer, const void* K, const void* V,
                                void* stream);

/*
 * Append chunk `chunk` of layer `layer` into slot chunk mod R, overwriting
 * that slot in place ("Matrix-Game 4.0", section "技术新颖性").  K, V: device,
 * token-major [B, Lc, H, D] bf16; they are transposed to the head-major slot
 * rows.  The copy is bit-exact for a BF16 ring.  For an FP8 ring each (b, h)
 * block of Lc x D values is quantised with amax = max |x|,
 * scale = amax / 448 (fp32, round-to-nearest division; 1 when amax = 0),
 * code = E4M3(x / scale) rounded to nearest even with saturation to +-448;
 * the scale is stored beside the slot.  An INT8K_FP8V ring quantises K the
 * same way with scale = amax / 127 and code = round-half-even(x / scale)
 * clamped to [-127, 127] (two's complement byte), and V as E4M3.
 * `chunk` must be >= 0 and, after the first append of that layer, equal to
 * the newest appended chunk (an in-place rewrite, e.g. the clean re-run of a
 * chunk) or one more.  Errors: INVALID_ARG, OUT_OF_RANGE (chunk order).
 */
sab_status sab_kv_ring_append(sab_ring* ring, int layer, long long chunk, const void* K,
                              const void* V, void* stream);

/* Slot of `chunk` in `layer`'s ring: chunk mod R if the chunk is held, else OUT_OF_RANGE. */
sab_status sab_kv_ring_slot_of(const sab_ring* ring, int layer, long long chunk, int* slot);

/*
 * Host-side state for checkpoint/resume, one entry per layer: the newest
 * appended chunk (-1: none), how many chunks the ring holds (0..R; they are
 * newest-held+1 .. newest) and whether the sink is set.  A caller that saves
 * the ring's device memory and this state can restore both and continue the
 * stream.  set_state validates every entry (held <= R, held <= newest+1,
 * held == 0 iff newest == -1) before changing anything.
 */
sab_status sab_kv_ring_get_state(const sab_ring* ring, long long* newest_chunk /*[num_layers]*/,
                                 int* held /*[num_layers]*/, int* sink_set /*[num_layers]*/);
sab_status sab_kv_ring_set_state(sab_ring* ring, const long long* newest_chunk, const int* held,
                                 const int* sink_set);

/*
 * Workspace bytes sab_chunk_attention needs for `num_splits` KV partitions
 * (0 when num_splits == 1; num_splits == 0 sizes it for any automatic choice).  The workspace holds per-split partial outputs
 * and LSEs plus one arrival counter per query tile; the counters must be zero
 * before the first call (zero-fill the workspace once after allocating it);
 * every call leaves them zero again, also one whose device waits gave up
 * (SAB_ERR_TIMEOUT from sab_get_last_device_error: its outputs are then not
 * valid, but the workspace needs no re-zeroing).
 */
size_t sab_chunk_attention_workspace(const sab_ring* ring, int num_splits);

/*
 * Attention of chunk `chunk`'s queries over the ring of layer `layer`.
 *   Q      device, token-major [B, Lc, H, D] bf16 (the chunk's queries).
 *   K_cur, V_cur
 *          device, token-major [B, Lc, H, D] bf16: the current chunk's keys
 *          and values computed fresh at this denoise step; or both NULL when
 *          the current chunk was already appended to the ring.
 *   window W >= 0: previous chunks attended (visible chunks c-W .. c).
 *   use_sink  1 to attend to the sink (the ring must have one, and it must be set).
 *   num_splits >= 1: KV partitions computed in parallel and merged by
 *          log-sum-exp inside the same kernel ("Matrix-Game 4.0", section
 *          "技术新颖性": the window is cut into intervals whose partial outputs
 *          are merged with log-sum-exp): one CTA per (128-query tile, b, h,
 *          partition); each partition writes its normalised partial rows and
 *          LSEs to the workspace and the last one of a query tile to finish
 *          merges them.  1 runs each query tile over the whole key set (no
 *          merge).  0 lets the library choose S in 1..8 (and at most half the
 *          key tiles) to fill the SMs: the S that minimises, in units of one
 *          key tile's time, waves * ceil(key tiles / S) + 5 (waves - 1) plus
 *          1 + 0.4 S for the merge when S > 1, where waves =
 *          ceil(tiles * S / SMs) and tiles = B * H * ceil(Lc / 128).
 *   softmax_scale  usually 1/sqrt(D).
 *   O      device, token-major [B, Lc, H, D] bf16 (output).
 *   LSE    device, [B, H, Lc] fp32, natural log of sum exp(s) (output; may be NULL).
 *   workspace/ws_bytes  device scratch, >= sab_chunk_attention_workspace.
 * Every chunk in max(0, c-W) .. c-1 (and c itself when K_cur is NULL) must be
 * held by the ring: OUT_OF_RANGE otherwise.  With an 8-bit ring (FP8_E4M3
 * or INT8K_FP8V) the kernel expands the codes to bf16 on chip (exact: every
 * E4M3 value and every integer in [-127, 127] is a bf16 value) and applies
 * the per-(batch, head, chunk) scales in fp32 (the K scale to the scores,
 * the V scale to the probabilities); this path needs head_dim 128,
 * chunk_tokens >= 128 and K_cur == V_cur == NULL (append the current chunk
 * first): UNSUPPORTED otherwise.  Device-side pipeline waits are
 * bounded; a wait that gives up is reported by sab_get_last_device_error.
 */
sab_status sab_chunk_attention(const sab_ring* ring, int layer, long long chunk, const void* Q,
                               const void* K_cur, const void* V_cur, int window, int use_sink,
                               int num_splits, float softmax_scale, void* O, float* LSE,
                               void* workspace, size_t ws_bytes, void* stream);

/*
 * Chunk attention over an E4M3 cache with 8-bit tensor-core products
 * ("Matrix-Game 4.0: Harnessing Video Models for Real-Time Playable Game
 * Worlds", sections 前置知识 / FP8 量化与 CUDA Graph and 技术新颖性: attention in
 * FP8 over an 8-bit KV cache).  Same key set and arguments as
 * sab_chunk_attention with K_cur = V_cur = NULL (the current chunk appended
 * first); num_splits, workspace and ws_bytes as there (0 = the library picks
 * the split count, and a workspace of sab_chunk_attention_workspace bytes is
 * then required).  The cached codes are used by the tensor cores as stored.
 * Each query row is quantised on chip to E4M3 with its own absmax scale
 * (amax / 448, fp32 division, round to nearest even, satfinite -- the cache's
 * rule applied per row); the probabilities are rounded to E4M3 as
 * P * (vs / vs_ref) * 2^3 (vs: the key's V scale, vs_ref: the largest V scale
 * of the key set; the running max lags by at most 2^5.75, so the values stay
 * below 2^8.75 < 448) and the row sums are kept in fp32 from the unrounded
 * values.  S = Q8 K8^T and O += P8 V8 accumulate in fp32; the splits' partial
 * rows merge by log-sum-exp in fp32.  O and LSE as in sab_chunk_attention.
 * Requires a SAB_KV_FP8_E4M3 ring (UNSUPPORTED otherwise), D = 128.
 * Errors: as sab_chunk_attention.
 */
sab_status sab_chunk_attention_fp8mma(const sab_ring* ring, int layer, long long chunk, const void* Q, int window,
                                      int use_sink, int num_splits, float softmax_scale, void* O, float* LSE,
                                      void* workspace, size_t ws_bytes, void* stream);

/*
 * Gradients of block-causal attention (training / causal adaptation:
 * "WanToFight", section 训练流程 / Stage 2; the same mask as
 * sab_block_causal_attention).  For a loss with gradient dO with respect to
 * O = softmax(scale Q K^T + mask) V, with P recomputed from the forward's LSE
 * and delta_i = sum_d dO_id O_id:
 *   dV = P^T dO,  dS = P * (dO V^T - delta),  dQ = scale dS K,  dK = scale dS^T Q.
 * Q, K, V, O, dO  device, token-major [B, L, H, D] bf16 (O and LSE as the
 *          forward produced them).  LSE: device [B, H, L] fp32.
 * dQ, dK, dV  device, token-major [B, L, H, D] bf16 (outputs).
 * workspace  device scratch of sab_block_causal_attention_backward_workspace
 *          bytes (delta), 256-byte aligned; no zero-fill needed.
 * D must be 64 or 128.  Errors: INVALID_ARG, WORKSPACE, CUDA.
 */
size_t sab_block_causal_attention_backward_workspace(int B, int L, int H);
sab_status sab_block_causal_attention_backward(const void* Q, const void* K, const void* V, const void* O,
                                               const void* dO, const float* LSE, int B, int L, int H, int D,
                                               int chunk_tokens, int window, float softmax_scale, void* dQ,
                                               void* dK, void* dV, void* workspace, size_t ws_bytes,
                                               void* stream);

/*
 * Block-causal attention behind a variable-length memory prefix (training
 * with compressed memory: "WorldPlay2: Extending Real-Time Interactive World
 * Models in Control and Horizon", Figure 3 and section 方法步骤详情, training
 * stage 3, where the padded variable-length memory is attended with a mask).
 * Each sample's L tokens are mem_pad memory positions, of which the first
 * mem_len[b] are real and the rest padding, then target tokens in chunks of
 * chunk_tokens (target token t is in chunk (t - mem_pad) / chunk_tokens).
 * A real memory query sees the real memory; a target query of chunk c sees
 * the real memory and the target chunks c - window .. c; padding sees nothing
 * and is seen by nothing, so padded rows get O = 0 and LSE = -inf (and zero
 * gradients).
 * Q, K, V, O  device, token-major [B, L, H, D] bf16, 16-byte aligned.
 * mem_len     device int32 [B], 4-byte aligned; values are clamped to
 *             [0, mem_pad] on the device.  May be NULL when mem_pad == 0
 *             (then this is sab_block_causal_attention with one split).
 * LSE         device [B, H, L] fp32 or NULL.  No workspace; one query tile
 *             of 128 rows per CTA.  D must be 64 or 128.
 * Errors: INVALID_ARG (pointers, sizes, mem_pad outside [0, L]), CUDA.
 */
sab_status sab_memory_prefix_attention(const void* Q, const void* K, const void* V, int B, int L, int H, int D,
                                       int mem_pad, const int* mem_len, int chunk_tokens, int window,
                                       float softmax_scale, void* O, float* LSE, void* stream);

/*
 * Gradients of sab_memory_prefix_attention (same formulas and arguments as
 * sab_block_causal_attention_backward, plus mem_pad and mem_len as above;
 * the workspace size is sab_block_causal_attention_backward_workspace).
 */
sab_status sab_memory_prefix_attention_backward(const void* Q, const void* K, const void* V, const void* O,
                                                const void* dO, const float* LSE, int B, int L, int H, int D,
                                                int mem_pad, const int* mem_len, int chunk_tokens, int window,
                                                float softmax_scale, void* dQ, void* dK, void* dV, void* workspace,
                                                size_t ws_bytes, void* stream);

/*
 * Fused Q/K normalisation and rotary embedding of one chunk, with the K/V
 * append ("WorldPlay2: Extending Real-Time Interactive World Models in
 * Control and Horizon", section 方法步骤详情: QKRoPE and QKV fusion;
 * "Matrix-Game 4.0", section 实验结果: a fused RoPE kernel).  The pages give
 * no formulas; the plain ones of a Wan-style video DiT are used:
 *   q' = RoPE(RMSNorm_q(q)), k' = RoPE(RMSNorm_k(k)), v' = v, where
 *   RMSNorm(x) = x / sqrt(mean(x^2) + eps) * gamma over each token's H*D
 *   values (gamma NULL: 1), and RoPE rotates the interleaved pairs
 *   (2i, 2i+1) of every head by pos * base^(-2i / band): the head dimension
 *   is split into bands (band_t, band_h, band_w) rotated by the token's
 *   frame, row and column in the chunk's latent grid (frames x height x
 *   width = chunk_tokens; token t of chunk c is at frame
 *   c * frames + t / (height * width)).  band_h = band_w = 0 with
 *   height = width = 1 is the one-dimensional embedding over the token index.
 * Q, K, V  device, token-major [B, Lc, H, D] bf16 (the QKV projection's
 *          output; shape from the ring).  gamma_q, gamma_k: device [H*D] fp32
 *          or NULL.  Q_out: device [B, Lc, H, D] bf16.  K_out, V_out: device
 *          [B, Lc, H, D] bf16 or NULL (k' and a copy of v).
 * append   1: also store k', v into slot chunk mod R of `layer`, with the
 *          rules and chunk-order check of sab_kv_ring_append -- fused into
 *          the same kernel for a BF16 ring; an 8-bit ring needs K_out and
 *          V_out and runs its quantiser on them.  0: no ring write (the
 *          chunk index still sets the positions).
 * Computed in fp32, rounded to bf16 once.  Errors: INVALID_ARG (pointers,
 * bands not even or not summing to head_dim, grid not matching chunk_tokens,
 * base <= 1, eps <= 0), OUT_OF_RANGE (chunk order when appending).
 */
typedef struct {
  int frames, height, width;    /* latent grid of one chunk                     */
  int band_t, band_h, band_w;   /* rotary bands of head_dim (even, sum = D)     */
  float base;                   /* rotary base, e.g. 10000                      */
  float eps;                    /* RMSNorm epsilon, e.g. 1e-6                   */
} sab_rope_desc;

sab_status sab_qk_norm_rope(sab_ring* ring, int layer, long long chunk, const void* Q, const void* K, const void* V,
                            const float* gamma_q, const float* gamma_k, const sab_rope_desc* rope, void* Q_out,
                            void* K_out, void* V_out, int append, void* stream);

/*
 * Graph-capturable streaming ("Matrix-Game 4.0", section "前置知识 / FP8 量化
 * 与 CUDA Graph": a whole chunk's GPU work is recorded once as a graph and
 * replayed with one launch per chunk, removing the per-kernel CPU launch
 * cost).  The three calls below read the chunk index from `d_chunk`, one
 * int64 in device memory, when their kernels run -- not when they are
 * launched -- so a chunk step (every layer's and denoise step's attention,
 * the ring appends and one sab_chunk_counter_add) captured once with
 * cudaStreamBeginCapture on `stream` replays correctly for every later chunk.
 *
 * sab_chunk_attention_dev: as sab_chunk_attention for chunk *d_chunk.  The
 *   key set is planned on the device by the same rule; the caller guarantees
 *   the stream discipline the host check enforces for sab_chunk_attention
 *   (every chunk the window needs was appended, in order, through
 *   sab_kv_ring_append_dev; *d_chunk >= 0).  Checked at the call: everything
 *   independent of the chunk, and that the window fits the ring (window <= R
 *   with K_cur, <= R - 1 without).  A chunk index that breaks the discipline
 *   gives wrong results but no out-of-range access: every key row read lies
 *   inside the layer's ring.  num_splits 0 sizes the automatic choice for a
 *   full window.
 * sab_kv_ring_append_dev: as sab_kv_ring_append into slot (*d_chunk mod R).
 *   The host handle's chunk bookkeeping (sab_kv_ring_get_state, the order
 *   check of sab_kv_ring_append) is not updated: drive a ring either through
 *   the _dev calls or through the host-indexed calls, not both.
 * sab_chunk_counter_add: *d_chunk += delta, as a kernel on `stream` (ordered
 *   after the work before it on the stream).
 * d_chunk: device pointer, 8-byte aligned; INVALID_ARG otherwise.
 */
sab_status sab_chunk_attention_dev(const sab_ring* ring, int layer, const long long* d_chunk, const void* Q,
                                   const void* K_cur, const void* V_cur, int window, int use_sink, int num_splits,
                                   float softmax_scale, void* O, float* LSE, void* workspace, size_t ws_bytes,
                                   void* stream);
sab_status sab_kv_ring_append_dev(sab_ring* ring, int layer, const long long* d_chunk, const void* K,
                                  const void* V, void* stream);
sab_status sab_chunk_counter_add(long long* d_chunk, long long delta, void* stream);

/*
 * sab_chunk_attention without a caller workspace.  The method itself has no
 * counterpart of this entry point; it exists for callers that cannot
 * allocate device memory -- for instance a plugin whose host application
 * owns every device allocation through its own pool, or a real-time stream
 * that forbids allocation once it is running -- and so cannot hand over the
 * workspace that a split (num_splits >= 2) merge needs.
 *
 * Arguments and results are those of sab_chunk_attention (num_splits >= 1,
 * no automatic choice).  With num_splits >= 2 the partial outputs, partial
 * LSEs and arrival counters of the split merge live in one library-owned
 * device array of 8 MiB (a file-scope __device__ array: every GPU that loads
 * the library holds it until the process exits).  A request whose merge
 * needs more -- num_splits * B * H * ceil-to-128(Lc) * (D + 1) * 4 bytes,
 * roughly -- returns SAB_ERR_WORKSPACE and launches nothing.
 * The call allocates nothing (no cudaMalloc/cudaFree or allocating library
 * routine); it clears the counters with cudaMemsetAsync on `stream`.
 * The first call on a device looks up the array's device address (with
 * that device current); make that first call before any stream capture.
 * Every call shares the one array, which keeps the previous call's partials:
 * calls whose executions overlap on the GPU (different streams, or devices
 * sharing nothing but this array's name) race -- serialise them.
 */
sab_status sab_chunk_attention_noalloc(const sab_ring* ring, int layer, long long chunk, const void* Q,
                                       const void* K_cur, const void* V_cur, int window, int use_sink,
                                       int num_splits, float softmax_scale, void* O, float* LSE, void* stream);

/*
 * Block-causal attention over whole sequences (training / causal-adaptation
 * shape; "WanToFight", section "训练流程 / Stage 2": the dense mask is replaced
 * by a block-causal one, bidirectional inside a chunk, each chunk seeing
 * itself and the `window` chunks before it).  Token t is in chunk
 * t / chunk_tokens; query i sees key j iff 0 <= chunk(i) - chunk(j) <= window.
 *   Q, K, V  device, token-major [B, L, H, D] bf16;  O likewise (output);
 *   LSE      device, [B, H, L] fp32 (output; may be NULL).
 *   num_splits / workspace as for sab_chunk_attention (size from
 *   sab_block_causal_attention_workspace).
 */
size_t sab_block_causal_attention_workspace(int B, int L, int H, int D, int num_splits);
sab_status sab_block_causal_attention(const void* Q, const void* K, const void* V, int B, int L,
                                      int H, int D, int chunk_tokens, int window, int num_splits,
                                      float softmax_scale, void* O, float* LSE, void* workspace,
                                      size_t ws_bytes, void* stream);

/*
 * Synchronise `stream`, then report and clear the device error word that
 * bounded pipeline waits set when they give up (SAB_ERR_TIMEOUT) and that the
 * index checks of a debug build set (SAB_ERR_BOUNDS, reported first when both
 * are recorded), or SAB_ERR_CUDA if the stream itself reports an error.
 * SAB_OK otherwise.
 */
sab_status sab_get_last_device_error(void* stream);

/*
 * Debug builds (no counterpart in the method).  A library compiled with
 * -DSAB_DEBUG_BOUNDS (libsab_debug.so) checks, in every kernel before it
 * issues a copy or a store, each global index it is about to form: the ring
 * slot rows of an append (inside the (batch, head) block, on a slot
 * boundary), the scale entry of an 8-bit append, every key run of an
 * attention CTA against the rows of its source, the FP8 scale entries it
 * reads, its workspace tile and counter, and the row ranges of the backward
 * tiles.  The checks are uniform over a CTA: a CTA that fails one records
 * SAB_ERR_BOUNDS in the device error word and leaves through the same path as
 * a CTA whose wait gave up (no copy, no store; split-merge counters still
 * return to zero).  Nothing traps.  Release builds compile the checks out.
 *
 * sab_debug_bounds_enabled: 1 in a debug build, 0 otherwise.
 * sab_debug_inject_bounds_error: makes the next launch of the named kind
 * carry an index past its buffer, so that its device check has to catch it
 * (the forged index points inside memory the caller owns in the forms the
 * self-test uses: one slot past the ring rows for an append, one slot past
 * the ring for an attention key run, one tile fewer than the workspace holds
 * for a split tile).  what: SAB_DEBUG_INJECT_APPEND_SLOT,
 * SAB_DEBUG_INJECT_KEY_ROW or SAB_DEBUG_INJECT_WS_TILE; 0 cancels a pending
 * injection.  Host-side only: nothing is launched.  Errors: UNSUPPORTED in a
 * release build, INVALID_ARG for another `what`.
 */
enum {
  SAB_DEBUG_INJECT_APPEND_SLOT = 1, /* next ring append (BF16 or 8-bit) */
  SAB_DEBUG_INJECT_KEY_ROW = 2,     /* next streaming chunk attention */
  SAB_DEBUG_INJECT_WS_TILE = 3      /* next split (num_splits >= 2) chunk attention */
};
int sab_debug_bounds_enabled(void);
sab_status sab_debug_inject_bounds_error(int what);

/*
 * Self-test of the device-side failure detection (no counterpart in the
 * method): launches one CTA on `stream` whose pipeline wait -- the same
 * bounded mbarrier wait every kernel of the library uses -- waits on a
 * barrier that nothing ever completes.  After timeout_ns (1 ms .. 2 s;
 * INVALID_ARG otherwise) the wait gives up, records its site and the kernel
 * returns; a following sab_get_last_device_error reports SAB_ERR_TIMEOUT and
 * clears the record.  Nothing faults, traps or hangs, and the context stays
 * usable.
 */
sab_status sab_selftest_bounded_wait(unsigned long long timeout_ns, void* stream);

/*
 * Self-test of the split merge's recovery (no counterpart in the method):
 * runs sab_chunk_attention with the same arguments and num_splits >= 2 (the
 * merge through the caller's workspace), in which split `abort_split`
 * (0 <= abort_split < num_splits) reports itself at the merge exactly as a
 * split whose bounded wait gave up does.  The merge of every query tile is
 * then skipped (O and LSE of this call are not valid),
 * sab_get_last_device_error reports SAB_ERR_TIMEOUT, and every arrival
 * counter of the workspace is zero again, so the next call on the same
 * workspace needs no re-zeroing.  Nothing faults, traps or hangs.
 * Errors: INVALID_ARG (num_splits < 2 or > 256, abort_split out of range),
 * then those of sab_chunk_attention.
 */
sab_status sab_selftest_split_abort(const sab_ring* ring, int layer, long long chunk, const void* Q,
                                    const void* K_cur, const void* V_cur, int window, int use_sink, int num_splits,
                                    float softmax_scale, void* O, float* LSE, void* workspace, size_t ws_bytes,
                                    int abort_split, void* stream);

/* Static, human-readable name of a status code. */
const char* sab_status_string(sab_status status);

/* Library version string. */
const char* sab_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SAB_H_ */
