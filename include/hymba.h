/*
 * hymba.h -- C ABI of the B300 (sm_103a) forward pass of Hymba's fused
 * hybrid-head layer.
 *
 * The operation ("Hymba: A Hybrid-head Architecture for Small Language
 * Models", section 2.1, eq. 3):
 *
 *     Y = W_out( beta1 * norm(M_attn X~) + beta2 * norm(M_ssm X~) )
 *
 * X~ is the input with the M learned meta-token rows prepended (section 2.3).
 * One shared input projection W_in yields Q, K, V, the SSM input x and the
 * gate z.  M_attn is causal GQA softmax attention whose key set is the window
 * of the last `window` tokens (0 = global) united with the meta prefix
 * (section 2.2).  M_ssm is a causal depthwise conv1d + SiLU followed by the
 * selective scan
 *     h_t = exp(delta_t * A) (.) h_{t-1} + delta_t * B_t * u_t,
 *     y_t = C_t . h_t + D (.) u_t,     g = y (.) silu(z),
 * with [dt | B | C] = u W_x^T, delta = softplus(dt W_dt^T + dt_bias),
 * A = -exp(A_log).  norm is RMSNorm over the d_inner channels of a row
 * (no weight of its own).  Layers can share K/V with the previous layer
 * (section 2.2), in which case they have no K/V projection.
 *
 * Conventions for every entry point:
 *  - All tensors are dense row-major ("C order") with the shapes given below.
 *    Pointers named "device" must point to device memory of the current CUDA
 *    device; the library never dereferences them on the host.
 *  - The caller owns every buffer.  The library allocates no memory, keeps no
 *    pointer after a call returns and keeps no state between calls apart
 *    from kernel attributes and occupancy figures it caches per device (and
 *    the per-device static scratch of hymba_layer_decode_static); calls on
 *    different streams and different devices are independent.
 *  - Calls are stream-ordered and asynchronous: inputs must stay valid and
 *    outputs must not be read until `stream` reaches the call.  `stream` is a
 *    cudaStream_t passed as void* (NULL = the legacy default stream).
 *  - Argument errors are detected on the host before anything is launched;
 *    the call then returns the error code and leaves every buffer untouched.
 *    No C++ exception crosses the ABI.
 *  - `dev_status` (may be NULL) is a device int32 that kernels set to a
 *    nonzero hymba_status when a bounded wait gives up (HYMBA_ERR_TIMEOUT)
 *    or an fp16 intermediate overflows (HYMBA_ERR_RANGE).  The caller zeroes
 *    it before the call and reads it afterwards.
 */
#ifndef HYMBA_H
#define HYMBA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HYMBA_ABI_VERSION 1

#if defined(__GNUC__)
#define HYMBA_API __attribute__((visibility("default")))
#else
#define HYMBA_API
#endif

typedef enum hymba_status {
  HYMBA_OK = 0,
  HYMBA_ERR_INVALID = 1,      /* null pointer, bad shape, misaligned buffer,
                                 kv_shared/kv_in mismatch                     */
  HYMBA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (see per-call)     */
  HYMBA_ERR_WORKSPACE = 3,    /* ws too small (query the *_workspace call)    */
  HYMBA_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed         */
  HYMBA_ERR_TIMEOUT = 5,      /* asynchronous: a bounded wait gave up         */
  HYMBA_ERR_RANGE = 6         /* asynchronous: |value| > 65504 in an fp16
                                 intermediate (bf16 path)                     */
} hymba_status;

typedef enum hymba_dtype {
  HYMBA_F32 = 0,   /* fp32 inputs/weights, fp32 SIMT arithmetic throughout   */
  HYMBA_BF16 = 1   /* bf16 inputs/weights; tensor-core MMAs with fp32
                      accumulation; intermediate activations stored as fp16;
                      scan state, delta, B, C, norms and Y in fp32            */
} hymba_dtype;

/* Shape and flags of one layer call.  L = n_meta + n_tokens.
 * P_in = n_q_heads*head_dim + (kv_shared ? 0 : n_kv_heads*(head_dim+v_head_dim))
 *        + 2*d_inner  (rows of W_in).                                       */
typedef struct hymba_layer_desc {
  int32_t batch;        /* B >= 1                                            */
  int32_t n_tokens;     /* T >= 1 real tokens (1 for decode)                 */
  int32_t n_meta;       /* M >= 0 meta rows at the start of X~               */
  int32_t d_model;      /* d                                                 */
  int32_t n_q_heads;    /* Hq; n_q_heads % n_kv_heads == 0                   */
  int32_t n_kv_heads;   /* Hkv (GQA groups; query head h uses KV head
                           h / (Hq/Hkv))                                     */
  int32_t head_dim;     /* dh of Q and K (even)                              */
  int32_t v_head_dim;   /* dv; n_q_heads * v_head_dim == d_inner             */
  int32_t d_inner;      /* di, width of both branches                        */
  int32_t d_state;      /* N                                                 */
  int32_t d_conv;       /* k, conv width (1..8)                              */
  int32_t dt_rank;      /* R                                                 */
  int32_t window;       /* keys incl. self visible in the window; 0 = global */
  int32_t kv_shared;    /* 1: no K/V projection; K/V come from kv_in (prefill)
                           or shared_cache (decode)                          */
  int32_t residual;     /* 0: none; 1: Y += X~ (the layer input, desc.dtype);
                           2: Y += Y (y holds an fp32 residual stream on
                           entry and is updated in place)                    */
  int32_t dtype;        /* hymba_dtype                                       */
  float rope_theta;     /* RoPE base (rotate-half pairs, absolute positions
                           counting the meta rows); 0 disables RoPE          */
  float eps;            /* RMSNorm epsilon (1e-6 in the reference workloads) */
  uint32_t wait_limit_us; /* bound on any single in-kernel wait; 0 = 2 s     */
  int32_t fusion;       /* 0: beta-weighted sum of the branches (eq. 3),
                           W_out [d, di]; 1: concatenation of the normalised,
                           beta-scaled branches (the appendix B ablation),
                           W_out [d, 2*di]                                    */
  int32_t reserved0;    /* must be 0                                         */
  int32_t reserved;     /* must be 0                                         */
} hymba_layer_desc;

/* Layer parameters (device pointers).  Matrices are in desc.dtype, vectors
 * are fp32.  W_in rows: [Q (Hq*dh) | K (Hkv*dh) | V (Hkv*dv) | x (di) | z (di)]
 * (no K/V rows when kv_shared).  W_x rows: [dt (R) | B (N) | C (N)].          */
typedef struct hymba_layer_weights {
  const void* W_in;     /* [P_in, d]                                         */
  const void* W_out;    /* [d, di]                                           */
  const void* W_x;      /* [R + 2N, di]                                      */
  const void* W_dt;     /* [di, R]                                           */
  const float* dt_bias; /* [di]                                              */
  const float* A_log;   /* [di, N]; A = -exp(A_log)                          */
  const float* D;       /* [di]                                              */
  const float* conv_w;  /* [di, k]; tap k-1 multiplies the newest row        */
  const float* conv_b;  /* [di]                                              */
  const float* beta1;   /* [di] attention-branch scale                       */
  const float* beta2;   /* [di] SSM-branch scale                             */
} hymba_layer_weights;

/* K/V of a layer, post-RoPE, exported for (or imported by) a KV-sharing
 * consumer.  Element type: fp16 on the HYMBA_BF16 path, fp32 on HYMBA_F32.  */
typedef struct hymba_kv {
  void* k;              /* [B, L, Hkv, dh] device                            */
  void* v;              /* [B, L, Hkv, dv] device                            */
} hymba_kv;

/* Decode state of one layer (device pointers).  K/V entries are in
 * desc.dtype (bf16 or fp32), post-RoPE.  Real token number p (0-based, not
 * counting meta rows) lives in slot p % cap.  A sliding-window layer needs
 * cap >= window; a global layer needs cap > the largest position it will
 * reach (no wrap).  A KV-sharing consumer layer's own cache needs only
 * ssm_state, conv_state and pos (its K/V pointers may be NULL).             */
typedef struct hymba_cache {
  void* k_ring;         /* [B, cap, Hkv, dh]                                 */
  void* v_ring;         /* [B, cap, Hkv, dv]                                 */
  void* k_meta;         /* [M, Hkv, dh], shared by the batch                 */
  void* v_meta;         /* [M, Hkv, dv]                                      */
  float* ssm_state;     /* [B, di, N] fp32                                   */
  float* conv_state;    /* [B, di, k-1] fp32, oldest row first               */
  int32_t* pos;         /* [B] real tokens already consumed                  */
  int32_t cap;          /* ring slots                                        */
  int32_t reserved;     /* must be 0                                         */
} hymba_cache;

/* Bytes of scratch memory hymba_layer_fwd needs for `d` (0 on invalid d):
 * the intermediates of eq. 3 of the Hymba page (section 2.1) -- the shared
 * projection [Q|K|V|x|z], the conv output, [dt|B|C], both branch outputs
 * and their normalised sum -- plus fp16 copies of W_out, W_x and W_dt.
 * A pure function of the descriptor; launches nothing.                     */
HYMBA_API size_t hymba_layer_fwd_workspace(const hymba_layer_desc* d);

/* Prefill forward of one layer over X~ (Hymba page, section 2.1 eq. 3;
 * meta tokens section 2.3; window / KV sharing section 2.2).  "Hymba page"
 * is "Hymba: A Hybrid-head Architecture for Small Language Models" throughout.
 *   x        [B, L, d] device, desc.dtype: X~ with the M meta rows first.
 *            Meta rows must be identical across the batch when cache_out is
 *            given (the cache keeps one copy of the meta K/V).
 *   y        [B, L, d] device fp32: Y for every row (meta rows included).
 *   cache_out (may be NULL) host struct of device buffers receiving the
 *            decode state: the last min(T, cap) tokens' K/V in their slots,
 *            meta K/V, final SSM state, conv tail (last k-1 pre-conv x rows)
 *            and pos = T.  Requires cap >= window (SWA) or cap >= T (global).
 *            Not allowed with kv_shared except for its ssm/conv/pos fields.
 *            Continuous batching: to admit a new sequence into row b of a
 *            running batch's cache, prefill it alone (desc.batch = 1, its own
 *            n_tokens) with cache_out pointing at row b -- k_ring + b*cap*Hkv*dh,
 *            v_ring + b*cap*Hkv*dv, ssm_state + b*di*N, conv_state +
 *            b*di*(k-1), pos + b elements -- and the batch's shared meta K/V
 *            (rewritten with the same values: the meta rows are identical for
 *            every sequence).  Rows are independent, so the other rows'
 *            state is untouched and the next decode step runs them all, each
 *            at its own pos.
 *   kv_in    non-NULL exactly when desc.kv_shared: the producer's K/V.
 *   kv_out   (may be NULL) receives this layer's post-RoPE K/V.
 *   ws       device scratch of ws_bytes >= hymba_layer_fwd_workspace(d),
 *            256-byte aligned; contents on entry are ignored.
 * Supported: HYMBA_F32 any shape (SIMT); HYMBA_BF16 needs d, P_in, d_inner,
 * Hkv*dh and Hkv*dv multiples of 8 and 16-byte aligned buffers.
 * Returns HYMBA_OK or a synchronous error code; asynchronous errors go to
 * dev_status.                                                               */
HYMBA_API hymba_status hymba_layer_fwd(const hymba_layer_desc* d, const hymba_layer_weights* w,
                             const void* x, float* y, const hymba_cache* cache_out,
                             const hymba_kv* kv_in, const hymba_kv* kv_out,
                             void* ws, size_t ws_bytes, int32_t* dev_status,
                             void* stream);

/* hymba_layer_fwd that also records CUDA events on `stream` around its
 * stages, for profiling: events[0] before the first launch and events[k]
 * after stage k, stages being 1 weight conversion, 2 input projection (+RoPE),
 * 3 K/V export, 4 attention, 5 conv+SiLU, 6 x_proj, 7 dt_proj+softplus,
 * 8 selective scan+gate, 9 norm/beta/sum, 10 output projection, 11 cache
 * emission (HYMBA_FWD_EVENTS events in all; extra events are not recorded,
 * missing ones are skipped).  events are cudaEvent_t handles created by the
 * caller; n_events >= 0.  Otherwise identical to hymba_layer_fwd.            */
#define HYMBA_FWD_EVENTS 12
HYMBA_API hymba_status hymba_layer_fwd_events(const hymba_layer_desc* d, const hymba_layer_weights* w,
                                              const void* x, float* y, const hymba_cache* cache_out,
                                              const hymba_kv* kv_in, const hymba_kv* kv_out, void* ws,
                                              size_t ws_bytes, int32_t* dev_status, void* const* events,
                                              int32_t n_events, void* stream);

/* ---------------------------------------------------------------------------
 * Meta-prefix precompute.  The M meta tokens are learned vectors prepended
 * to every input (Hymba page, section 2.3), so their rows of a layer are the same
 * for every sequence: hymba_meta_prefill runs the layer once over those M
 * rows and keeps what the real tokens need from them; hymba_layer_fwd_meta
 * then runs the layer over the real tokens of a whole batch from that
 * state.  The result equals hymba_layer_fwd on [meta rows | tokens] (rows M..
 * of Y) without recomputing the prefix B times.
 * Supported on HYMBA_BF16 with head_dim 64, v_head_dim 64 or 128 and n_meta a
 * positive multiple of 64 (HYMBA_ERR_UNSUPPORTED otherwise).
 * ------------------------------------------------------------------------- */
typedef struct hymba_meta {
  void* k;              /* [M, Hkv, dh] fp16, post-RoPE (a KV-sharing layer
                           points at its producer's meta K/V)                */
  void* v;              /* [M, Hkv, dv] fp16                                 */
  float* ssm_state;     /* [di, N] fp32: the SSM state after the meta rows   */
  float* conv_tail;     /* [di, k-1] fp32: the last k-1 x rows, oldest first */
  float* y;             /* [M, d] fp32: Y of the meta rows                   */
} hymba_meta;

/* Bytes of scratch memory hymba_meta_prefill needs (desc.batch and
 * desc.n_tokens are ignored: one copy of the meta rows is processed).        */
HYMBA_API size_t hymba_meta_prefill_workspace(const hymba_layer_desc* d);

/* Runs the layer over the M meta rows alone and fills `meta` (every buffer
 * device memory owned by the caller).
 *   x_meta   [M, d] device, bf16: the meta rows of X~.
 *   kv_in    non-NULL exactly when desc.kv_shared: the producer layer's meta
 *            K/V ([M, Hkv, dh] / [M, Hkv, dv] fp16); meta->k / meta->v are
 *            then not written.
 * Errors as hymba_layer_fwd.                                                */
HYMBA_API hymba_status hymba_meta_prefill(const hymba_layer_desc* d, const hymba_layer_weights* w,
                                          const void* x_meta, const hymba_meta* meta, const hymba_kv* kv_in,
                                          void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Bytes of scratch memory hymba_layer_fwd_meta needs for `d`.              */
HYMBA_API size_t hymba_layer_fwd_meta_workspace(const hymba_layer_desc* d);

/* Prefill of the real tokens from a hymba_meta_prefill state.
 *   x        [B, T, d] device bf16: the real tokens only (no meta rows).
 *   y        [B, T, d] device fp32: Y of the real tokens (position M + t);
 *            residual 1 adds x, residual 2 updates y in place.
 *   meta     the state written by hymba_meta_prefill with the same weights.
 *   cache_out, kv_in, kv_out as hymba_layer_fwd, with the K/V of kv_in and
 *            kv_out holding the T real rows ([B, T, Hkv, .]); the meta K/V of
 *            cache_out are copied from meta->k / meta->v.  With cache_out,
 *            T >= k-1 is not required: the conv tail falls back on
 *            meta->conv_tail.                                               */
HYMBA_API hymba_status hymba_layer_fwd_meta(const hymba_layer_desc* d, const hymba_layer_weights* w,
                                            const hymba_meta* meta, const void* x, float* y,
                                            const hymba_cache* cache_out, const hymba_kv* kv_in,
                                            const hymba_kv* kv_out, void* ws, size_t ws_bytes,
                                            int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------
 * Full residual block around the hybrid-head layer.  The Hymba pages give no
 * block structure of their own; this follows the residual pattern and gated
 * MLP of "Griffin: Mixing Gated Linear Recurrences with Local Attention for
 * Efficient Language Models" (section 2.1 residual block, section 2.2 MLP
 * block):
 *     x = x + Layer(RMSNorm(x; norm1))
 *     x = x + W_down (GeLU(W_gate h) * (W_up h)),  h = RMSNorm(x; norm2)
 * RMSNorm(x; w) = x / sqrt(mean(x^2) + eps) * w over the d channels of a row;
 * GeLU(v) = v Phi(v) (exact, erf).  The sub-block inputs are stored in bf16
 * (the layer's input type); the stream x stays fp32.
 * Supported on HYMBA_BF16 (the layer's own constraints), d % 8 == 0 and
 * d_ff % 8 == 0.
 * ------------------------------------------------------------------------- */
typedef struct hymba_block_weights {
  hymba_layer_weights mix;  /* the hybrid-head layer                          */
  const float* norm1;       /* [d] fp32: RMSNorm weight before the layer      */
  const float* norm2;       /* [d] fp32: RMSNorm weight before the MLP        */
  const void* W_gu;         /* [2*d_ff, d] bf16: gate and up rows interleaved,
                               row 2j = W_gate row j, row 2j+1 = W_up row j    */
  const void* W_down;       /* [d, d_ff] bf16                                 */
} hymba_block_weights;

/* Bytes of scratch memory hymba_block_fwd needs (0 on invalid). */
HYMBA_API size_t hymba_block_fwd_workspace(const hymba_layer_desc* d, int32_t d_ff);

/* One residual block over the whole stream (meta rows included).
 *   d        the layer's descriptor; desc.residual must be 0 (the block adds
 *            the stream itself).
 *   x        [B, L, d] device fp32, the residual stream: read, then
 *            overwritten with the block's output.
 *   d_ff     the MLP width F.
 * Errors as hymba_layer_fwd; HYMBA_ERR_RANGE in *dev_status if an fp16
 * intermediate (layer activations, the MLP's gated hidden layer) overflows. */
HYMBA_API hymba_status hymba_block_fwd(const hymba_layer_desc* d, const hymba_block_weights* w, int32_t d_ff,
                                       float* x, void* ws, size_t ws_bytes, int32_t* dev_status,
                                       void* stream);

/* ---------------------------------------------------------------------------
 * Residual stack of hybrid-head layers over one batch (the stacks of the
 * Hymba page's 300M-parameter design roadmap, section 2 and Table 1;
 * consecutive layers may share K/V, section 2.2):
 *     X_{l+1} = X_l + Y_l(X_l),   X_0 = x
 * The stream X_l is kept in fp32.  Layer 0 reads x (bf16); each later layer
 * reads the stream rounded to fp16 (its matmul operand type; W_in is
 * converted to fp16 for it, exact for every bf16 value in fp16's normal
 * range).  A layer with desc.kv_shared reads the previous layer's post-RoPE
 * K/V.  The Hymba pages describe no pre-norm or FFN for this stack.  Errors
 * add HYMBA_ERR_RANGE (dev_status) if the stream leaves fp16's range.
 * ------------------------------------------------------------------------- */

/* Bytes of scratch memory hymba_stack_fwd needs (0 on invalid descs).      */
HYMBA_API size_t hymba_stack_fwd_workspace(int32_t n_layers, const hymba_layer_desc* descs);

/* Runs n_layers (1..256) layers back to back on `stream`.
 *   descs    [n_layers] host array: HYMBA_BF16, the same batch, n_tokens,
 *            n_meta and d_model in every layer; residual must be 0 (the
 *            stack adds the stream itself); layer 0 may not be kv_shared,
 *            and a kv_shared layer has its producer's n_kv_heads, head_dim
 *            and v_head_dim.
 *   weights  [n_layers] host array of device-pointer structs.
 *   x        [B, L, d] device bf16: X_0 with the meta rows first.
 *   y        [B, L, d] device fp32 (must not overlap x): the stream after
 *            the last layer.
 *   ws       device scratch, ws_bytes >= hymba_stack_fwd_workspace().
 * Errors as hymba_layer_fwd, every descriptor validated before anything is
 * launched.                                                                 */
HYMBA_API hymba_status hymba_stack_fwd(int32_t n_layers, const hymba_layer_desc* descs,
                                       const hymba_layer_weights* weights, const void* x, float* y, void* ws,
                                       size_t ws_bytes, int32_t* dev_status, void* stream);

/* Bytes of scratch memory hymba_layer_decode needs for `d` (0 on invalid):
 * one row per sequence of the same intermediates as the prefill, the
 * split-K partial sums of x_proj / out_proj and the key-split partials of
 * the decode attention (the step of the Hymba page, sections 2.2-2.3, whose
 * cost is the bytes it reads: "Griffin: Mixing Gated Linear Recurrences with
 * Local Attention for Efficient Language Models", section 4.1, eq. 5).
 * A pure function of the descriptor; launches nothing.                     */
HYMBA_API size_t hymba_layer_decode_workspace(const hymba_layer_desc* d);

/* One decode step for B sequences (desc.n_tokens must be 1): eq. 3 of the
 * Hymba page (section 2.1) for one new row per sequence, with the attention
 * branch reading a window-bounded cache plus the meta-token K/V (sections 2.2
 * and 2.3: SWA keeps only the last `window` tokens, the meta tokens act as a
 * learned cache prefix; consecutive layers may share K/V) and the SSM branch
 * advancing its carried state by one step of the recurrence.  Its time is the
 * bytes it moves over the memory bandwidth ("Griffin: ...", section 4.1,
 * eq. 5: decode is memory-bound, the cache and the weights are read once per
 * step).  The token of
 * sequence b sits at absolute position M + pos[b]; its K/V go into slot
 * pos[b] % cap of `cache` (skipped for a kv_shared layer, which reads the
 * producer's `shared_cache`, already updated for this token); attention sees
 * the meta K/V plus the last min(pos+1, window) ring entries (pos+1 for a
 * global layer); ssm_state and conv_state are advanced in place; pos[b] is
 * incremented at the end.
 *   x_new    [B, d] device, desc.dtype.      y  [B, d] device fp32.
 * A global layer needs pos[b] + 1 <= cap: a token past a full global cache
 * is not stored (the write is skipped on the device, never out of bounds)
 * and attends to the first cap cached entries only.                         */
HYMBA_API hymba_status hymba_layer_decode(const hymba_layer_desc* d, const hymba_layer_weights* w,
                                const void* x_new, float* y, const hymba_cache* cache,
                                const hymba_cache* shared_cache, void* ws, size_t ws_bytes,
                                int32_t* dev_status, void* stream);

/* Size of the library's built-in decode scratch buffer (32 MiB), used by
 * hymba_layer_decode_static.                                                */
#define HYMBA_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* hymba_layer_decode for callers that cannot allocate device memory.  No
 * counterpart in the paper: it exists for integration only.
 *
 * Some callers cannot call cudaMalloc at the point where they run a decode
 * step: a plugin inside a host framework that owns all device memory and
 * hands out none, or a serving loop whose memory is fully reserved by its
 * KV-cache pool and where cudaMalloc would fail or stall the device.  This
 * entry point takes the same arguments as hymba_layer_decode minus the
 * workspace: its scratch lives in one statically sized device buffer that the
 * library declares (HYMBA_STATIC_SCRATCH_BYTES per GPU that loads the
 * library, held until the process exits).  It allocates nothing.
 *   - Shapes whose decode workspace (hymba_layer_decode_workspace) exceeds
 *     HYMBA_STATIC_SCRATCH_BYTES are rejected with HYMBA_ERR_WORKSPACE before
 *     anything is launched; hymba_layer_decode_workspace gives a shape's
 *     need (the 1.5B-shaped decode at batch 128 fits).
 *   - The first call on a device looks up that device's address of the
 *     buffer (cudaGetSymbolAddress, with that device current); make that first
 *     call before any stream capture.
 *   - Every call, on every stream, uses the same buffer: calls whose
 *     execution overlaps on the GPU race on it and give wrong results.
 *     Serialise them (one stream, or events).  The buffer keeps the last
 *     call's contents; the decode step writes every scratch byte it reads, so
 *     nothing has to start at zero.
 * Other arguments, errors and effects are those of hymba_layer_decode.       */
HYMBA_API hymba_status hymba_layer_decode_static(const hymba_layer_desc* d, const hymba_layer_weights* w,
                                                 const void* x_new, float* y, const hymba_cache* cache,
                                                 const hymba_cache* shared_cache, int32_t* dev_status,
                                                 void* stream);

/* hymba_layer_decode that also records CUDA events on `stream` around its
 * stages (bf16 path): events[0] before the first launch, events[k] after
 * stage k: 1 weight conversion, 2 input projection (+RoPE), 3 ring append,
 * 4 attention, 5 conv step, 6 x_proj, 7 dt_proj+softplus, 8 scan step,
 * 9 norm/beta/sum, 10 output projection, 11 position advance
 * (HYMBA_DECODE_EVENTS events).  Otherwise identical to hymba_layer_decode. */
#define HYMBA_DECODE_EVENTS 12
HYMBA_API hymba_status hymba_layer_decode_events(const hymba_layer_desc* d, const hymba_layer_weights* w,
                                                 const void* x_new, float* y, const hymba_cache* cache,
                                                 const hymba_cache* shared_cache, void* ws, size_t ws_bytes,
                                                 int32_t* dev_status, void* const* events, int32_t n_events,
                                                 void* stream);

/* Human-readable name of a status code (static storage, never NULL; unknown
 * codes give "unknown hymba_status").  No counterpart in the paper: the
 * error channel of this interface.                                          */
HYMBA_API const char* hymba_status_str(hymba_status s);

/* HYMBA_ABI_VERSION of the built library.                                   */
HYMBA_API int32_t hymba_abi_version(void);

/* ---------------------------------------------------------------------------
 * Component entry points used by the parity tests.  Each runs exactly one of
 * the kernels hymba_layer_fwd uses, on caller buffers, on `stream`.
 * ------------------------------------------------------------------------- */

/* C[M, N] (fp32, row stride ldc) = A[M, K] . B[N, K]^T on the tcgen05 GEMM
 * (Hymba page, section 2.1: the shared input projection and W_out are these
 * GEMMs).  ab_dtype 1 = bf16 operands, 2 = fp16 operands, 3 = fp16 A with
 * bf16 B converted to fp16 in shared memory (the decode step's weights, read
 * once and never copied; a bf16 value outside fp16's normal range rounds as
 * a float-to-half conversion does).  K-major rows,
 * 16-byte aligned, lda/ldb (elements) multiples of 8.                        */
HYMBA_API hymba_status hymba_test_gemm(int32_t M, int32_t N, int32_t K, int32_t ab_dtype,
                             const void* A, int32_t lda, const void* B, int32_t ldb,
                             float* C, int32_t ldc, int32_t* dev_status, void* stream);

/* The bf16-path causal depthwise conv + SiLU kernel alone (the SSM heads'
 * short convolution, section 2.1): u[b,t,c] = silu(conv_b[c] + sum_j
 * conv_w[c,j] x[b, t-k+1+j, c]) with x = 0 before row 0 of each sequence.
 * x fp16 [B, L, ld_x] (di valid columns), u fp16 [B, L, di]; conv_w [di, k],
 * conv_b [di] fp32.  HYMBA_ERR_UNSUPPORTED unless di % 8 == 0, 2 <= k <= 4,
 * ld_x % 8 == 0 and x, u 16-byte aligned.                                    */
HYMBA_API hymba_status hymba_test_conv(int32_t B, int32_t L, int32_t di, int32_t k,
                                       const void* x, int32_t ld_x, void* u,
                                       const float* conv_w, const float* conv_b,
                                       int32_t* dev_status, void* stream);

/* The bf16-path selective scan + gate kernel alone (SSM recurrence of the
 * hybrid head, section 2.1).  u, z: fp16 [B, L, di] (row strides ld_u, ld_z);
 * delta: fp32 [B, L, di]; BC: fp32 [B, L, 2N] ([B | C]); A_log [di, N], D [di]
 * fp32.  g: fp16 [B, L, di] = (C.h + D u) silu(z); h_out [B, di, N] fp32
 * final state (may be NULL).  threads_per_channel: how many threads share
 * one channel's states (1, 2 or 4); channels_per_thread: how many adjacent
 * channels one thread runs over those states (0 or 1, or 2 with two or four
 * threads per channel); both 0 = the choice hymba_layer_fwd makes.  Other
 * combinations: HYMBA_ERR_INVALID.                                         */
HYMBA_API hymba_status hymba_test_scan(int32_t B, int32_t L, int32_t di, int32_t N,
                             const void* u, int32_t ld_u, const void* z, int32_t ld_z,
                             const float* delta, const float* BC, const float* A_log,
                             const float* D, void* g, float* h_out,
                             int32_t threads_per_channel, int32_t channels_per_thread,
                             void* stream);

/* The same scan with the dt projection fused in, as hymba_layer_fwd runs it:
 * delta = softplus(dtr . W_dt^T + dt_bias) is computed inside the kernel.
 * dtr fp16 [B, L, ld_dtr] (R valid columns, ld_dtr % 8 == 0), W_dt bf16
 * [di, R], dt_bias fp32 [di]; other arguments as hymba_test_scan.
 * HYMBA_ERR_UNSUPPORTED unless di % 16 == 0, N == 16, R <= 128.             */
HYMBA_API hymba_status hymba_test_scan_fused(int32_t B, int32_t L, int32_t di, int32_t N, int32_t R,
                                             const void* u, int32_t ld_u, const void* z, int32_t ld_z,
                                             const void* dtr, int32_t ld_dtr, const void* W_dt,
                                             const float* dt_bias, const float* BC, const float* A_log,
                                             const float* D, void* g, float* h_out,
                                             int32_t threads_per_channel, int32_t channels_per_thread,
                                             void* stream);

/* The bf16-path attention kernel alone (section 2.2 window + section 2.3 meta
 * prefix): Q [B, L, Hq, dh], K [B, L, Hkv, dh], V [B, L, Hkv, dv] fp16 ->
 * O [B, L, Hq*dv] fp16.  use_tc: 1 = tcgen05 flash kernel, 0 = SIMT kernel. */
HYMBA_API hymba_status hymba_test_attention(int32_t B, int32_t L, int32_t M, int32_t Hq, int32_t Hkv,
                                  int32_t dh, int32_t dv, int32_t window, int32_t use_tc,
                                  const void* Q, const void* K, const void* V, void* O,
                                  int32_t* dev_status, void* stream);

/* Failure-detection check: one block waits on an mbarrier that nothing
 * arrives on, for at most limit_us, then writes HYMBA_ERR_TIMEOUT to
 * *dev_status and returns.  No paper counterpart.                           */
HYMBA_API hymba_status hymba_test_wait_timeout(uint32_t limit_us, int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* HYMBA_H */
