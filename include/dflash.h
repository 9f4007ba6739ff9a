/*
 * dflash.h -- C ABI of libdflash: one DFlash block-diffusion draft + verify step on
 * one GB300 (sm_103a).
 *
 * The step, as the DFlash pages describe it:
 *   - DFlash wiki (aisparkup.com/wiki/dflash), "타깃 모델 피처 컨디셔닝" items 1-3:
 *     hidden features of several target layers are fused by a light projection
 *     (dflash_fuse_features), injected into the KV cache of every drafter layer
 *     (dflash_inject_kv), and a block of future tokens is predicted from that context
 *     in one parallel forward pass (dflash_draft_block); the drafter reuses the
 *     target's embedding and LM head (dflash_lm_head_argmax).
 *   - NVIDIA blog "Boost inference performance up to 15x on NVIDIA Blackwell using
 *     DFlash speculative decoding", section "How does DFlash speculative decoding
 *     work?": the target verifies the block in parallel and the longest valid prefix is
 *     accepted (dflash_verify_greedy); verification keeps the target's output
 *     distribution (dflash_verify_sample, temperature > 0 with supplied uniforms).
 *
 * Conventions shared by every call:
 *   - Every tensor argument is a DEVICE pointer owned by the caller, row-major, with
 *     the element type given by dflash_config.dtype (DFLASH_BF16 or DFLASH_F32) unless
 *     the argument says otherwise (int32 indices, fp32 statistics).  Tensor pointers
 *     must be 16-byte aligned.  Arrays of per-layer pointers (dflash_weights members,
 *     k_pool / v_pool) are HOST arrays of n_layers device pointers.
 *   - Matrices follow the [out, in] convention: y = x W^T.
 *   - The handle borrows the weights (the caller keeps them alive and unchanged until
 *     dflash_destroy); it owns a device error word and a RoPE cos/sin table.
 *   - Hot-path calls allocate nothing: scratch comes from a caller-provided workspace
 *     of at least dflash_workspace_size() bytes that was zeroed once by
 *     dflash_workspace_init() (the library keeps its control words at zero after every
 *     call that completes without a device error).  One workspace serves one stream at
 *     a time; calls that share a workspace or a handle must not overlap on the GPU.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).  Every
 *     call only enqueues work and returns; a returned status covers host-side
 *     validation and the kernel launches.  Problems found on the device (an index out
 *     of range, a position past the RoPE table, a bounded wait that ran out) set the
 *     handle's error word, the kernel that found them returns early, and outputs of
 *     that call are unspecified; read and clear the word with dflash_get_device_error.
 *   - A handle belongs to the device that was current at dflash_create; every call on
 *     it must be made with that device current (EINVAL otherwise).
 *   - No call throws; the message of the last failing call on this thread is
 *     available from dflash_last_error().
 *   - KV cache: per drafter layer, one K pool and one V pool, each
 *     [num_pages][n_kv_heads][page_size][head_dim] (page_size = 16).  A token at cache
 *     slot s lives in page s / page_size at offset s % page_size.  Slots of a
 *     sequence's last page past its context length are read (with zero weight): they
 *     must hold finite values, e.g. a pool zeroed once at allocation.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DFLASH_API __attribute__((visibility("default")))
#else
#define DFLASH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dflash_status {
  DFLASH_OK = 0,
  DFLASH_EINVAL = 1,        /* bad argument: null/misaligned pointer, bad size      */
  DFLASH_EUNSUPPORTED = 2,  /* valid but outside what the kernels implement          */
  DFLASH_EWORKSPACE = 3,    /* workspace smaller than dflash_workspace_size()        */
  DFLASH_ECUDA = 4,         /* a CUDA runtime/driver call failed                     */
  DFLASH_EDEVICE = 5        /* the device error word is set (dflash_get_device_error) */
} dflash_status;

typedef enum dflash_dtype { DFLASH_F32 = 0, DFLASH_BF16 = 1 } dflash_dtype;

/* Storage of the projection weights (fusion, Q/K/V/O, gate/up/down, LM head; the
 * embedding and the norm gains stay in the dtype).  NATIVE: the config dtype.  FP8:
 * packed FP8 E4M3 matrices (dflash_pack_fp8), bf16 configs only; their projections
 * run on the weight-streaming kernel, whose tiles take at most 32 activation rows
 * (larger row counts run as several such tiles). */
typedef enum dflash_weight_format { DFLASH_WEIGHTS_NATIVE = 0, DFLASH_WEIGHTS_FP8 = 1 }
    dflash_weight_format;

/* Device error codes (the first error of a call wins). */
enum {
  DFLASH_DEV_OK = 0,
  DFLASH_DEV_BAD_INDEX = 1,     /* page id, slot, token id or draft token out of range */
  DFLASH_DEV_BAD_POSITION = 2,  /* position outside [0, max_position)                  */
  DFLASH_DEV_TIMEOUT = 3        /* a bounded on-device wait ran out                     */
};

/* Drafter shape.  d_model = d, fused input width = n_target_layers * target_width
 * (target layer l in columns [l*target_width, (l+1)*target_width)), q width =
 * n_q_heads * head_dim, kv width = n_kv_heads * head_dim.  page_size must be 16;
 * head_dim must be even and divide 128 (64 or 128 for bf16).
 * max_position bounds every RoPE position (context and block).  rope_theta: base of
 * the rotary frequencies theta^(-2j/head_dim); rms_eps: epsilon of every RMSNorm. */
typedef struct dflash_config {
  int32_t d_model, n_layers, n_q_heads, n_kv_heads, head_dim, ffn_dim, vocab;
  int32_t block_size, n_target_layers, target_width, page_size, max_position;
  float rope_theta, rms_eps;
  int32_t dtype; /* dflash_dtype of weights, activations, KV cache and target logits */
  int32_t weight_format; /* dflash_weight_format of the projection weights             */
} dflash_config;

/* Borrowed device weights ([out, in] matrices, [d] RMSNorm gains).  Per-layer members
 * are host arrays of n_layers device pointers; the handle copies those arrays.  With
 * weight_format FP8 the projection matrices are packed FP8 buffers (dflash_pack_fp8). */
typedef struct dflash_weights {
  /* both NULL: a handle without fusion (a plain transformer, e.g. a target model) */
  const void* w_fuse;   /* [d, n_target_layers*target_width]  feature fusion        */
  const void* g_fuse;   /* [d]                                 fusion RMSNorm gain   */
  const void* const* g_attn;  /* [d]              pre-attention RMSNorm gain       */
  const void* const* w_q;     /* [n_q_heads*head_dim, d]                           */
  const void* const* w_k;     /* [n_kv_heads*head_dim, d] (block and injected K)   */
  const void* const* w_v;     /* [n_kv_heads*head_dim, d] (block and injected V)   */
  const void* const* w_o;     /* [d, n_q_heads*head_dim]                           */
  const void* const* g_mlp;   /* [d]              pre-MLP RMSNorm gain             */
  const void* const* w_gate;  /* [ffn_dim, d]                                      */
  const void* const* w_up;    /* [ffn_dim, d]                                      */
  const void* const* w_down;  /* [d, ffn_dim]                                      */
  const void* g_final;  /* [d]       final RMSNorm gain                             */
  const void* embed;    /* [vocab, d] target embedding (reused)                      */
  const void* lm_head;  /* [vocab, d] target LM head (reused)                        */
} dflash_weights;

typedef struct dflash_handle_s* dflash_handle;

/* Creates a handle on the current device: validates the shape, copies the pointer
 * arrays, allocates the error word and the RoPE table (the only allocations of the
 * library) and prepares the TMA descriptors of the weights.  Returns EUNSUPPORTED for
 * shapes the kernels do not cover: bf16 needs head_dim 64 or 128, d_model, ffn_dim and
 * the fused input width multiples of 8, q and kv widths multiples of 128, and
 * block_size * (n_q_heads / n_kv_heads) a multiple of 16 up to 128; both dtypes need
 * block_size <= 16. */
DFLASH_API dflash_status dflash_create(const dflash_config* cfg, const dflash_weights* w,
                            dflash_handle* out);
DFLASH_API dflash_status dflash_destroy(dflash_handle h);

/* Workspace bytes for calls with at most max_rows rows (dflash_fuse_features /
 * dflash_inject_kv: n; dflash_draft_block / dflash_lm_head_argmax: batch*block_size),
 * at most max_batch sequences (dflash_draft_block, dflash_inject_inputs,
 * dflash_target_forward, verification) and page tables at most max_pages wide. */
DFLASH_API dflash_status dflash_workspace_size(dflash_handle h, int32_t max_rows, int32_t max_batch,
                                    int32_t max_pages, size_t* bytes);

/* Zeroes the workspace's control words (enqueued on stream).  Needed once before the
 * first use of a workspace and again after any call that set the device error word. */
DFLASH_API dflash_status dflash_workspace_init(dflash_handle h, void* ws, size_t ws_bytes,
                                    void* stream);

/* [DFlash wiki, item 1] fused = RMSNorm(x_cat W_fuse^T) * g_fuse.
 * x_cat [n, n_target_layers*target_width] -> fused [n, d].  n >= 0 (0 = no-op). */
DFLASH_API dflash_status dflash_fuse_features(dflash_handle h, const void* x_cat, int32_t n,
                                   void* fused, void* ws, size_t ws_bytes, void* stream);

/* [DFlash wiki, item 2; DFlash FAQ 1 (opensource-hub.com/ko/library/z-lab-dflash)]
 * writes the context features of n tokens into every layer's cache:
 * K_l = RoPE(fused W_k,l^T, positions), V_l = fused W_v,l^T, at cache `slots`.
 * Exactly one of x_cat [n, n_target_layers*target_width] (fused here first) and
 * fused [n, d] is non-NULL.  positions [n] int32 in [0, max_position); slots [n] int32
 * in [0, num_pages*page_size).  k_pool / v_pool: host arrays of n_layers pool
 * pointers.  fused_out [n, d] (optional, may be NULL) receives the fused features
 * when x_cat is given. */
DFLASH_API dflash_status dflash_inject_kv(dflash_handle h, const void* x_cat, const void* fused,
                               int32_t n, const int32_t* positions, const int32_t* slots,
                               int32_t num_pages, void* const* k_pool, void* const* v_pool,
                               void* fused_out, void* ws, size_t ws_bytes, void* stream);

/* [DFlash wiki, "블록 확산으로 병렬 드래프팅" and item 3; NVIDIA blog, how it works]
 * one parallel drafter forward pass over `batch` blocks of block_size tokens.
 * block_ids [batch, block_size] int32 (mask id for masked slots); ctx_lens [batch]
 * int32 = context tokens already in the cache (block token i sits at position
 * ctx_lens[b] + i); page_table [batch, max_pages] int32 (entries past a sequence's
 * last page are ignored); num_pages = pool size.  Each layer: RMSNorm, Q/K/V
 * projections, RoPE, bidirectional grouped-query attention over [the sequence's
 * cached context ; the block], output projection + residual, RMSNorm, SwiGLU MLP +
 * residual.  final_hidden [batch*block_size, d] = final RMSNorm output. */
DFLASH_API dflash_status dflash_draft_block(dflash_handle h, const int32_t* block_ids,
                                 const int32_t* ctx_lens, const int32_t* page_table,
                                 int32_t max_pages, int32_t batch, int32_t num_pages,
                                 void* const* k_pool, void* const* v_pool,
                                 void* final_hidden, void* ws, size_t ws_bytes,
                                 void* stream);

/* [DFlash wiki, item 2; NVIDIA blog, how it works: the injected K/V come from the same
 * key-value projections as the block's own]  dflash_inject_kv of n_inj new context rows
 * (x_cat, positions, slots as there) followed by dflash_draft_block, in one call: the
 * same results.  When the block's rows plus the new rows fit one weight-streaming tile
 * (bf16, batch * block_size + n_inj <= 64) every layer's W_k and W_v are read once:
 * that layer's Q/K/V projection runs over [the block's normed rows ; the fused new
 * rows] and writes the new rows' K (RoPE) and V into the cache, and the attention
 * fetches the pages of the newest n_inj positions of each sequence only after those
 * writes (the new rows must be each sequence's newest context positions).  Otherwise
 * the two calls run one after the other.  fused_out (optional) as in
 * dflash_inject_kv. */
DFLASH_API dflash_status dflash_inject_draft(dflash_handle h, const void* x_cat, int32_t n_inj,
                                  const int32_t* positions, const int32_t* slots,
                                  const int32_t* block_ids, const int32_t* ctx_lens,
                                  const int32_t* page_table, int32_t max_pages, int32_t batch,
                                  int32_t num_pages, void* const* k_pool, void* const* v_pool,
                                  void* fused_out, void* final_hidden, void* ws, size_t ws_bytes,
                                  void* stream);

/* [DFlash FAQ 1 (opensource-hub.com/ko/library/z-lab-dflash): the input-fusion
 * ablation, where the fused hidden features are the drafter's input rather than being
 * injected into every layer's K/V; the FAQ attributes KV injection's shorter draft
 * prefill to the context skipping that full per-token processing]
 * Input-fusion counterpart of dflash_inject_kv for `batch` sequences of block_size new
 * context rows each: x_cat [batch*block_size, n_target_layers*target_width] (row b*S+i
 * = token ctx_lens[b] + i of sequence b) is fused as in dflash_fuse_features, and the
 * fused rows are then the layer-0 input of the drafter's layer stack: each layer takes
 * RMSNorm, Q/K/V + RoPE at positions ctx_lens[b] + i, causal attention over [the
 * sequence's ctx_lens[b] cached tokens ; the new rows 0..i], output projection +
 * residual, RMSNorm, SwiGLU MLP + residual, and writes its K/V of the new rows into its
 * cache at those positions (the last layer stops after its K/V).  ctx_lens are the
 * tokens already in the cache (the caller advances them by block_size afterwards);
 * page_table / num_pages / pools as in dflash_draft_block, with pages allocated up to
 * position ctx_lens[b] + block_size - 1.  fused_out [batch*block_size, d] (optional)
 * receives the fused rows.  A context of any length is prefilled chunk by chunk
 * (causal attention makes that identical to one pass; a ragged last chunk may carry
 * padding rows, whose cache entries lie past the context and are overwritten later). */
DFLASH_API dflash_status dflash_inject_inputs(dflash_handle h, const void* x_cat,
                                   const int32_t* ctx_lens, const int32_t* page_table,
                                   int32_t max_pages, int32_t batch, int32_t num_pages,
                                   void* const* k_pool, void* const* v_pool, void* fused_out,
                                   void* ws, size_t ws_bytes, void* stream);

/* [DFlash wiki, 사용법: spec_generate(..., target=target); NVIDIA blog, how it works:
 * the target verifies the drafted block in one parallel pass]  The target side of the
 * speculative loop, for a handle created without fusion weights (w_fuse = g_fuse =
 * NULL: a plain transformer with the same layer structure).  One causal pass over
 * block_size tokens per sequence: ids [batch, block_size] at positions ctx_lens[b] + i,
 * each layer attending causally over [the ctx_lens[b] cached tokens ; tokens 0..i] and
 * writing its K/V of the tokens into its cache at those positions.  taps [batch*S,
 * n_taps*d] (optional): column block t = the residual stream after layer tap_layers[t]
 * (1-based, host array), rounded to the config dtype -- the multi-layer hidden features
 * the drafter fuses.  logits [batch*S, vocab] fp32 (optional): the final RMSNorm and LM
 * head of every token. */
DFLASH_API dflash_status dflash_target_forward(dflash_handle h, const int32_t* ids,
                                   const int32_t* ctx_lens, const int32_t* page_table,
                                   int32_t max_pages, int32_t batch, int32_t num_pages,
                                   void* const* k_pool, void* const* v_pool,
                                   const int32_t* tap_layers, int32_t n_taps, void* taps,
                                   float* logits, void* ws, size_t ws_bytes, void* stream);

/* State of the greedy speculative loop (device pointers unless marked host).  Both
 * caches hold the tokens before each sequence's anchor (ctx_lens[b] of them) and share
 * one page table, whose pages must reach position ctx_lens[b] + block_size - 1 at every
 * step. */
typedef struct dflash_spec_state {
  int32_t batch;
  int32_t* block_ids;          /* [batch, S]: the anchor (last emitted token) in slot 0,
                                  mask_id after it; rewritten by every step            */
  int32_t* ctx_lens;           /* [batch]: tokens in both caches; advanced by each step */
  const int32_t* page_table;   /* [batch, max_pages] (both caches)                      */
  int32_t max_pages, num_pages;
  void* const* d_k_pool;       /* host array [drafter n_layers] of drafter K pools      */
  void* const* d_v_pool;
  void* const* t_k_pool;       /* host array [target n_layers] of target K pools        */
  void* const* t_v_pool;
  const int32_t* tap_layers;   /* host [drafter n_target_layers]: the target layers
                                  (1-based) whose outputs the drafter fuses, in order   */
  int32_t mask_id;
  int32_t* generated;          /* [batch, max_new]: emitted tokens, appended            */
  int32_t max_new;
  int32_t* n_generated;        /* [batch]: tokens in `generated` (stops at max_new)     */
  int32_t* n_emitted;          /* [batch]: tokens the last step emitted (1..S)          */
  int32_t* drafts;             /* [batch, S] or NULL: the last step's drafted tokens    */
  int32_t* step;               /* [1]: step counter, advanced by every step             */
  const float* plant_u;        /* [plant_steps, batch, S] or NULL: see dflash_spec_step */
  int32_t plant_steps;
  float plant_p;
} dflash_spec_state;

/* Workspace of dflash_spec_step for `batch` sequences and page tables max_pages wide;
 * zero its control words once with dflash_spec_workspace_init before the first step
 * (and again after a step that set a device error). */
DFLASH_API dflash_status dflash_spec_workspace_size(dflash_handle drafter, dflash_handle target,
                                         int32_t batch, int32_t max_pages, size_t* bytes);
DFLASH_API dflash_status dflash_spec_workspace_init(dflash_handle drafter, dflash_handle target,
                                         int32_t batch, int32_t max_pages, void* ws,
                                         size_t ws_bytes, void* stream);

/* [DFlash wiki, 사용법: spec_generate; NVIDIA blog, "How does DFlash speculative
 * decoding work?": draft a block in one pass, verify it with the target in one pass,
 * accept the longest valid prefix]  One step of greedy speculative decoding, entirely
 * on the device (no host synchronisation, so a CUDA graph can hold it):
 *   1. the drafter drafts the block [anchor, mask, ...] at positions ctx_lens[b] + i
 *      over its cache (dflash_draft_block) and takes the LM-head argmax d_0..d_{S-1};
 *   2. the target (a handle without fusion weights, d_model = the drafter's
 *      target_width, same vocab, block_size and dtype) runs causally over [anchor,
 *      d_1, ..., d_{S-1}] (dflash_target_forward): its cache, the tap features of the
 *      block's tokens and fp32 logits;
 *   3. with plant_u given, a synthetic stand-in for a trained drafter/target pair: row
 *      i < S-1 of the target logits gets logit[d_{i+1}] = row max + 1 when
 *      plant_u[step mod plant_steps, b, i] < plant_p;
 *   4. t_i = argmax of target row i (lowest index); n = leading i < S-1 with
 *      d_{i+1} = t_i; the step emits t_0..t_n (n accepted drafts and the target's
 *      token) into `generated`, n_emitted[b] = n + 1;
 *   5. the block's tap features are fused and injected into the drafter's cache at
 *      positions ctx_lens[b] + i (rows past the accepted ones are overwritten later),
 *      the anchor becomes t_n and ctx_lens[b] advances by n + 1.
 * The emitted tokens are exactly the target's own greedy continuation (without
 * planting).  Before the first step: both caches hold the context (prompt tokens but
 * the last, e.g. by dflash_target_forward and dflash_inject_kv of its taps), the
 * anchor is the prompt's last token and the workspace is initialised. */
DFLASH_API dflash_status dflash_spec_step(dflash_handle drafter, dflash_handle target,
                                          const dflash_spec_state* s, void* ws,
                                          size_t ws_bytes, void* stream);

/* [DFlash wiki: the drafter reuses the target's LM head] per row r of hidden
 * [rows, d]: tokens[r] = argmax_v (hidden W_lm^T)[r, v], lowest index among equal
 * maxima; the logits never reach memory.  Optional fp32 outputs (NULL to skip):
 * max_logit[r] = the maximum logit, lse[r] = log sum_v exp(logit_v / temperature)
 * (temperature > 0; ignored when lse is NULL). */
DFLASH_API dflash_status dflash_lm_head_argmax(dflash_handle h, const void* hidden, int32_t rows,
                                    float temperature, int32_t* tokens, float* max_logit,
                                    float* lse, void* ws, size_t ws_bytes, void* stream);

/* [NVIDIA blog, how it works: accept the longest valid prefix] greedy verification of
 * `batch` drafted blocks.  draft [batch, block_size] int32; target_logits
 * [batch, block_size, vocab] (dtype of the config), row i scoring block slot i.
 * t_i = argmax of row i (lowest index on ties); n = number of leading slots with
 * draft == t; outputs: out_tokens [batch, block_size] int32 = t_0..t_min(n, S-1) then
 * -1 padding; n_accepted [batch] = n; n_emitted [batch] = min(n + 1, block_size). */
DFLASH_API dflash_status dflash_verify_greedy(dflash_handle h, const int32_t* draft,
                                   const void* target_logits, int32_t batch,
                                   int32_t* out_tokens, int32_t* n_accepted,
                                   int32_t* n_emitted, void* ws, size_t ws_bytes,
                                   void* stream);

/* [DFlash wiki, 성능 비교: sampling at temperature 1; NVIDIA blog: verification keeps
 * the target's output distribution] verification at temperature tau > 0 with
 * supplied uniforms [batch, block_size, 2] fp32 in [0, 1).  p_i = softmax(target_i /
 * tau), q_i = softmax(z_i / tau) with z the drafter's logits (z_i = final_hidden_i
 * W_lm^T, draft_max / draft_lse from dflash_lm_head_argmax at the same tau).  Slot i
 * is accepted iff u[i,0] < p_i(d_i) / q_i(d_i); at the first rejection n the emitted
 * token is the lowest v with sum_{w<=v} r_w >= u[n,1] * sum(r), r = max(0, p_n - q_n)
 * (r = p_n if that is all zero).  Outputs as dflash_verify_greedy, out_tokens =
 * d_0..d_{n-1} then the sampled token. */
DFLASH_API dflash_status dflash_verify_sample(dflash_handle h, const int32_t* draft,
                                   const void* final_hidden, const float* draft_max,
                                   const float* draft_lse, const void* target_logits,
                                   const float* uniforms, float temperature, int32_t batch,
                                   int32_t* out_tokens, int32_t* n_accepted,
                                   int32_t* n_emitted, void* ws, size_t ws_bytes,
                                   void* stream);

/* Greedy verification that allocates nothing and takes no workspace.  The paper has no
 * counterpart: this exists for callers that cannot call cudaMalloc where they verify a
 * block (a host runtime that owns only fixed buffers, a memory budget frozen at that
 * point, a plain C caller without an allocator).  Same inputs, outputs and results as
 * dflash_verify_greedy; its scratch is one fixed 256 KiB device array of the library
 * (held by every GPU that loads the library until exit), so batch * block_size must
 * not exceed 16384 (larger requests return DFLASH_EUNSUPPORTED with a message).  The
 * first call on a device looks up that array's device address (cudaGetSymbolAddress,
 * with the device current); make that first call before any stream capture.  Each call
 * clears the array's counters on `stream` before use.  All calls share the one array:
 * calls whose work overlaps on the GPU (other streams, other threads) race. */
DFLASH_API dflash_status dflash_verify_greedy_static(dflash_handle h, const int32_t* draft,
                                                     const void* target_logits, int32_t batch,
                                                     int32_t* out_tokens, int32_t* n_accepted,
                                                     int32_t* n_emitted, void* stream);

/* [NVIDIA blog, Blackwell Ultra paragraph: low-precision tensor formats] Packed FP8
 * form of a weight matrix [rows, cols] ([out, in]): e4m3 codes, row stride
 * round_up(cols, 16) bytes, then at the next 256-byte boundary rows fp32 scales.  Row
 * n's scale is the power of two s_n = 2^e, e the smallest integer with
 * max_k |w[n,k]| <= 448 * 2^e (1 for an all-zero row), and its codes are
 * e4m3(w[n,k] / s_n) rounded to nearest, ties to even (the division is exact), so the
 * matrix stands for codes * s_n.  dflash_fp8_packed_bytes gives the buffer size;
 * dflash_pack_fp8 quantizes a bf16 device matrix w into the device buffer `packed` on
 * the current device (enqueued on stream). */
DFLASH_API dflash_status dflash_fp8_packed_bytes(int32_t rows, int32_t cols, size_t* bytes);
DFLASH_API dflash_status dflash_pack_fp8(const void* w, int32_t rows, int32_t cols, void* packed,
                                         void* stream);

/* Test hook for the bounded waits (no counterpart in the pages).  With enable != 0,
 * the CTA that finishes a projection tile split between CTAs waits for one more
 * published piece than can ever arrive, gives up after 10 ms, raises
 * DFLASH_DEV_TIMEOUT in the error word and goes on (no copy is abandoned and no kernel
 * leaves early; the outputs of such calls are unspecified).  Split tiles occur in
 * every projection whose work is cut between CTAs (batch-1 blocks always are).  After
 * disabling it, re-initialise the workspace (dflash_workspace_init) before the next
 * call. */
DFLASH_API dflash_status dflash_test_force_timeout(dflash_handle h, int32_t enable);

/* Synchronizes the device, returns the handle's error word in *code (DFLASH_DEV_*)
 * and zeroes it when clear != 0. */
DFLASH_API dflash_status dflash_get_device_error(dflash_handle h, int32_t* code, int32_t clear);

/* Message of the last failing call on this thread ("" if none). */
DFLASH_API const char* dflash_last_error(void);

/* Number of kernels the last call on this thread enqueued. */
DFLASH_API int32_t dflash_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_H */
