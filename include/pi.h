/*
 * pi.h -- C ABI of the neuron-aware sparse FFN decode path (one GPU, sm_103a).
 *
 * Per decode layer the path computes, for each token x (length d):
 *   1. predictor:  u = P1 x,  s = P2 u + b,  neuron k predicted active iff s_k > tau
 *   2. compaction: the ascending list of predicted-active storage rows
 *   3. FC1:        h_j = ReLU(W1[idx_j] . x + b1[idx_j])     (gated: * (Wu[idx_j] . x))
 *   4. FC2:        y = b2 + sum_j h_j * W2t[idx_j, :]
 * following the pages describing PowerInfer (PowerInfer summary (CSDN)):
 * section "Background" (FC1, ReLU, FC2 as products of the input with neurons,
 * i.e. rows/columns of the weight matrices), section "Adaptive sparse
 * predictor" (an input/hidden/output predictor of which neurons fire),
 * section "Neuron-aware operator" (decide whether a neuron is active, then
 * process only its row or column, with no dense-format conversion) and section
 * "Neuron placement and management" (a table maps each stored neuron to its
 * original position).
 *
 * Conventions for every entry point:
 *  - Every pointer argument except the descriptors is DEVICE memory owned by
 *    the caller; the library allocates nothing and keeps no pointer after the
 *    call returns.  Descriptors (pi_layer_desc, pi_layer_weights) are HOST
 *    structs read during the call only.
 *  - All calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream).  Device-side counts stay on the device:
 *    no call synchronises the host except pi_last_device_status.
 *  - Arguments are validated on the host before anything is launched; a bad
 *    argument returns PI_ERR_INVALID_ARG and launches nothing.  A failed launch
 *    returns PI_ERR_CUDA.
 *  - Binary16 data is passed as pi_half (IEEE 754 binary16 bit patterns).
 *  - Per-neuron arrays (W1, Wu, W2t, their scales, b1, P2 rows, table) are in
 *    STORAGE order: storage row k holds original neuron table[k].
 *  - Masks: bit k of a mask is bit (k % 32) of 32-bit word k / 32; a batch of
 *    B masks is B consecutive runs of ceil(F/32) words.
 *  - Alignment: every weight, x and workspace pointer 16-byte aligned;
 *    d % 8 == 0 (fp16) and d % 32 == 0 (INT4); rank % 8 == 0.
 *  - Calls on distinct streams with distinct outputs and workspaces may run
 *    concurrently; calls sharing a workspace must be stream-ordered.
 *  - A workspace must be zero-filled (e.g. cudaMemset) before its first use;
 *    the library keeps it consistent from then on.  pi_ffn_layer and
 *    pi_ffn_stack exchange data between thread blocks through it with bounded
 *    waits: a wait that exceeds 2 s makes the kernel return early and sets the
 *    device status read by pi_last_device_status (PI_ERR_TIMEOUT).
 */
#ifndef PI_H
#define PI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(PI_BUILD) && defined(__GNUC__)
#define PI_API __attribute__((visibility("default")))
#else
#define PI_API
#endif

typedef uint16_t pi_half; /* IEEE 754 binary16 bit pattern */

typedef enum {
    PI_OK = 0,
    PI_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or descriptor      */
    PI_ERR_UNSUPPORTED = 2, /* valid request this build does not implement       */
    PI_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed              */
    PI_ERR_TIMEOUT = 4,     /* a bounded device-side wait expired                */
    PI_ERR_WORKSPACE = 5    /* workspace NULL, misaligned or smaller than needed */
} pi_status;

typedef enum {
    PI_W_F16 = 0,     /* rows of d binary16 values                                    */
    PI_W_INT4_G32 = 1 /* rows of d/2 bytes of INT4 codes (even element in the low      */
                      /* nibble, two's complement, value q*scale) + d/32 binary16 scales */
} pi_wdtype;

typedef struct {
    int d;            /* model width                                  */
    int ffn;          /* FFN width F (number of neurons)              */
    int rank;         /* predictor rank r                             */
    int batch;        /* tokens B processed together (1..32)          */
    pi_wdtype wdtype; /* FC1/FC2 weight format (Wu is always fp16)    */
    int gated;        /* 1: h = ReLU(Wg x + bg) * (Wu x)              */
} pi_layer_desc;

typedef struct {
    const void *w1;          /* [F, d] fp16, or [F, d/2] INT4 codes (gate rows when gated) */
    const pi_half *w1_scales; /* [F, d/32] (INT4 only, else NULL)                           */
    const pi_half *b1;       /* [F]  FC1 (gate) bias, also the predictor bias              */
    const pi_half *wu;       /* [F, d] fp16 up-projection rows (gated only, else NULL)     */
    const void *w2t;         /* [F, d] fp16 or INT4 codes: row k = neuron k's FC2 column   */
    const pi_half *w2t_scales; /* [F, d/32] (INT4 only, else NULL)                         */
    const pi_half *b2;       /* [d]                                                        */
    const pi_half *p1;       /* [r, d] predictor input layer                               */
    const pi_half *p2;       /* [F, r] predictor output layer (storage order)              */
    const int32_t *table;    /* [F] storage row -> original neuron id                      */
} pi_layer_weights;

/* Bytes of workspace pi_predict, pi_sparse_fc1, pi_sparse_fc2 and pi_ffn_layer need for
 * `desc` (0 if the descriptor is invalid). */
PI_API size_t pi_workspace_bytes(const pi_layer_desc *desc);

/*
 * Predictor (PowerInfer summary (CSDN), section "Adaptive sparse predictor").
 *   u_b = P1 x_b (fp32), s_b = P2 u_b + bpred (fp32), mask_b bit k = s_bk > tau.
 * x: [B, d] fp16.  mask: [B, ceil(F/32)] uint32 (bits past F are 0).
 * workspace: >= pi_workspace_bytes(desc) bytes, 16-byte aligned.
 * For 16 <= B <= 32, fp16 weights, d % 128 == 0 and rank % 16 == 0 both
 * products run on the tcgen05 tensor cores; u enters P2 u as two fp16 halves
 * hi = fp16(u), lo = fp16(u - hi), which keeps fp32 accuracy.
 */
PI_API pi_status pi_predict(const pi_layer_desc *desc, const pi_half *x, const pi_half *p1,
                     const pi_half *p2, const pi_half *bpred, float tau, uint32_t *mask,
                     void *workspace, size_t ws_bytes, void *stream);

/*
 * Active-neuron compaction (section "Neuron-aware operator": first decide
 * which neurons are active; section "Neuron placement and management": the
 * table gives each stored neuron's original position).
 * For B == 1 compacts mask; for B > 1 compacts the union (bitwise OR) of the
 * B masks.  idx: [F] int32, ascending storage rows, first *d_count valid.
 * orig_idx (nullable, requires table): table[idx].  d_count: [1] int32.
 */
PI_API pi_status pi_compact(const pi_layer_desc *desc, const uint32_t *mask, const int32_t *table,
                     int32_t *idx, int32_t *orig_idx, int32_t *d_count, void *stream);

/*
 * Row-gathered FC1 with fused bias and ReLU (section "Background"; section
 * "Neuron-aware operator": only the rows of active neurons are read).
 *   h[j*B + b] = ReLU(W1[idx_j] . x_b + b1[idx_j])  (gated: times Wu[idx_j] . x_b)
 * for j < *d_count; when B > 1 and mask != NULL, h[j*B+b] = 0 wherever token
 * b's own mask bit idx_j is 0.  h: [F*B] fp32 (neuron-major).
 * For 16 <= B <= 32, fp16 weights and d % 128 == 0 the rows are gathered once
 * for all B tokens and multiplied on the tcgen05 tensor cores (fp16 x fp16
 * products, fp32 accumulation); so are INT4 rows of a ReLU layer at B = 16
 * with d % 256 == 0 (codes as exact fp16 integers, group scales applied per
 * 32-element group); INT4 at 2 <= B <= 16 otherwise streams on CUDA cores;
 * the rest runs on CUDA cores in chunks of <= 8 tokens.
 * workspace: >= pi_workspace_bytes(desc) bytes, 16-byte aligned (partial
 * sums of the tensor-core split).
 */
PI_API pi_status pi_sparse_fc1(const pi_layer_desc *desc, const pi_half *x, const pi_layer_weights *w,
                        const int32_t *idx, const int32_t *d_count, const uint32_t *mask,
                        float *h, void *workspace, size_t ws_bytes, void *stream);

/*
 * FC2 as a gather-accumulate over W2t rows (section "Background"; section
 * "Neuron-aware operator": only the columns of active neurons, stored as rows).
 *   y[b*d + c] = b2[c] + sum_{j < *d_count} h[j*B + b] * W2t[idx_j, c]   (fp32)
 * Reduced without atomics in a fixed order (bitwise reproducible).
 * Under the same conditions as pi_sparse_fc1 the tensor cores take it, with h
 * split into fp16 hi = fp16(h) and lo = fp16(h - hi) so that fp32 accuracy is
 * kept.  INT4 rows at B = 16: the codes are the exact fp16 A operand and the
 * row's group scale moves into B, one (hi, lo) pair of h * scale per token and
 * 32-column group, lo = fp16((h * scale - hi) * 2^11) (scaled out again in the
 * epilogue).
 */
PI_API pi_status pi_sparse_fc2(const pi_layer_desc *desc, const float *h, const int32_t *idx,
                        const int32_t *d_count, const pi_layer_weights *w, float *y,
                        void *workspace, size_t ws_bytes, void *stream);

/*
 * pi_sparse_fc2 for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point: it exists for callers such as a
 * plug-in inside a host framework that owns the whole device memory pool and
 * offers no allocation hook, or a service with a fixed device-memory budget
 * that forbids allocation after start-up, which therefore cannot pass the
 * workspace pi_sparse_fc2 needs.  Same arguments and result as pi_sparse_fc2
 * without the workspace; the FC2 partial sums live in an 8 MiB array inside
 * the library that every GPU loading the library holds until process exit.
 *  - Returns PI_ERR_WORKSPACE when the FC2 partial sums of `desc` exceed that
 *    array (2 Mi floats).  They are, with G the SM count: splits x batch x d
 *    floats on the per-token path; G x (ceil(d/128/G) + 2) x T x 128 floats on
 *    the streamed fp16 path (T = 2, 4 or 8 tokens) and on the batch 16..32
 *    tensor-core path (T = 16 or 32) and on the INT4 tensor-core path at 16
 *    tokens (T = 16); G x (ceil(d/256/G) + 2) x T x 256 on the streamed INT4
 *    path (T = 4, 8 or 16).  Allocates nothing in any case.
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any
 *    stream capture.
 *  - All calls share the one array: calls whose executions overlap on the GPU
 *    (different streams, or concurrent host threads) race and give wrong
 *    results; keep them ordered on one stream.
 */
PI_API pi_status pi_sparse_fc2_noalloc(const pi_layer_desc *desc, const float *h, const int32_t *idx,
                                       const int32_t *d_count, const pi_layer_weights *w, float *y,
                                       void *stream);

/*
 * Second tier of a layer's FC rows (PowerInfer summary (CSDN), sections
 * "Neuron placement and management" and "GPU-CPU hybrid execution": the hot
 * neurons stay in GPU memory and the cold ones in the host's memory).  Storage
 * rows 0 .. n_hot-1 (the hot prefix of the neuron table) are read from the
 * pi_layer_weights arrays, rows n_hot .. F-1 from these arrays at row
 * k - n_hot.  The arrays may be host memory that the GPU addresses directly
 * (pinned and mapped, as from cudaHostAlloc; on a Grace-Blackwell system the
 * Grace memory, read over NVLink-C2C) or device memory; they are read with
 * plain 16-byte loads, never with bulk copies.  Same element layout as the
 * pi_layer_weights arrays; 16-byte aligned.
 */
typedef struct {
    int n_hot;                 /* 0 .. F                                              */
    const void *w1;            /* [F - n_hot, d] fp16 or [F - n_hot, d/2] INT4 codes   */
    const pi_half *w1_scales;  /* [F - n_hot, d/32] (INT4 only, else NULL)             */
    const pi_half *wu;         /* [F - n_hot, d] fp16 (gated only, else NULL)          */
    const void *w2t;           /* [F - n_hot, d] fp16 or INT4 codes                    */
    const pi_half *w2t_scales; /* [F - n_hot, d/32] (INT4 only, else NULL)             */
} pi_cold_tier;

/*
 * pi_sparse_fc1 / pi_sparse_fc2 with the rows of `cold` for the storage rows
 * from cold->n_hot on (same results; the per-token CUDA-core kernels, in
 * chunks of <= 8 tokens, for every batch size).  pi_sparse_fc1_tiered needs no
 * workspace; pi_sparse_fc2_tiered takes pi_workspace_bytes(desc) bytes.
 * PI_ERR_INVALID_ARG if n_hot is outside 0..F or a needed pointer is NULL or
 * misaligned.
 */
PI_API pi_status pi_sparse_fc1_tiered(const pi_layer_desc *desc, const pi_half *x, const pi_layer_weights *w,
                                      const pi_cold_tier *cold, const int32_t *idx, const int32_t *d_count,
                                      const uint32_t *mask, float *h, void *stream);
PI_API pi_status pi_sparse_fc2_tiered(const pi_layer_desc *desc, const float *h, const int32_t *idx,
                                      const int32_t *d_count, const pi_layer_weights *w, const pi_cold_tier *cold,
                                      float *y, void *workspace, size_t ws_bytes, void *stream);
/* One decode layer whose cold FC rows live in `cold`: predictor (weights in
 * w) -> compaction -> pi_sparse_fc1_tiered -> pi_sparse_fc2_tiered.  The
 * workspace holds the same intermediates as for pi_ffn_layer. */
PI_API pi_status pi_ffn_layer_tiered(const pi_layer_desc *desc, const pi_half *x, const pi_layer_weights *w,
                                     const pi_cold_tier *cold, float tau, void *workspace, size_t ws_bytes,
                                     float *y, void *stream);

/*
 * One whole decode layer: predictor -> compaction -> FC1 -> FC2 on `stream`.
 * x: [B, d] fp16; y: [B, d] fp32.  The per-token masks, the union index list
 * and its count are left in the workspace (see pi_workspace_layout).
 */
PI_API pi_status pi_ffn_layer(const pi_layer_desc *desc, const pi_half *x, const pi_layer_weights *w,
                       float tau, void *workspace, size_t ws_bytes, float *y, void *stream);

/*
 * One decode step through a stack of n_layers (1..96) layers that share d,
 * ffn, wdtype and gated; desc->rank is the largest rank and ranks[l] (NULL:
 * all desc->rank) the rank of layer l.  Layer l computes y_l from x_l exactly
 * as pi_ffn_layer does, and the next layer's input is the normalisation of
 * its output, x_{l+1} = fp16(y_l / sqrt(mean(y_l^2) + eps)) (as
 * pi_rmsnorm_half).  layers: HOST array of n_layers weight sets (device
 * pointers inside).  x: [B, d] fp16 input of layer 0; y: [B, d] fp32 output
 * of the last layer; x_trace (nullable): [n_layers-1, B, d] fp16, the inputs
 * of layers 1..n_layers-1; layer_counts (nullable): [n_layers, 2] int32, per
 * layer the number of predicted-active neurons and the number of those whose
 * FC1 output is non-zero (for any token of the batch).  The workspace
 * intermediates are the last layer's.
 */
PI_API pi_status pi_ffn_stack(const pi_layer_desc *desc, int n_layers, const pi_layer_weights *layers,
                              const int *ranks, const pi_half *x, float tau, float eps, void *workspace,
                              size_t ws_bytes, float *y, pi_half *x_trace, int32_t *layer_counts,
                              void *stream);

/* Offsets (bytes) of the intermediates pi_ffn_layer leaves in the workspace. */
typedef struct {
    size_t mask;  /* uint32 [B, ceil(F/32)] per-token masks         */
    size_t idx;   /* int32 [F] ascending active rows (union if B>1) */
    size_t count; /* int32 [1]                                      */
    size_t h;     /* float [F*B] FC1 outputs                        */
    size_t total; /* == pi_workspace_bytes                          */
} pi_workspace_layout_t;
PI_API pi_status pi_workspace_layout(const pi_layer_desc *desc, pi_workspace_layout_t *out);

/*
 * Inter-layer normalisation of a decode stack: x_out[b, c] =
 * fp16(y[b, c] / sqrt(mean_c(y[b, :]^2) + eps)) with round-to-nearest-even.
 * y: [B, d] fp32, 16-byte aligned; x_out: [B, d] fp16, 8-byte aligned; d a
 * multiple of 4 (else PI_ERR_INVALID_ARG).  One block per token.
 */
PI_API pi_status pi_rmsnorm_half(int d, int batch, const float *y, float eps, pi_half *x_out,
                          void *stream);

/*
 * Head-sparse self-attention block of one decode step (PowerInfer summary
 * (CSDN), section "Background", paragraph on activation sparsity: in the
 * self-attention block about half of the heads contribute little for a given
 * input; unite.ai page, section on adaptive sparsity predictors: each layer
 * has one activity predictor for its MLP block and one for its self-attention
 * block, and only the neurons predicted active are computed).  The block's
 * neurons are its heads.  For each sequence b (one new token x_b at cache
 * position pos[b]):
 *   1. head mask: u = P1 x_b, s = P2 u + bp, head h active iff s_h > tau
 *      (the predictor of pi_predict with F = heads);
 *   2. k_g = Wk_g x_b + bk_g and v_g = Wv_g x_b + bv_g for EVERY KV head g,
 *      stored as binary16 (round to nearest even) at position pos[b] of the
 *      caches, so later tokens find a complete cache;
 *   3. for each active head h (KV head g = h / (heads / kv_heads)):
 *      q = Wq_h x_b + bq_h;  a_t = softmax_t(q . K_g[t] / sqrt(head_dim)) over
 *      t = 0 .. pos[b] (the token's own key included);  o_h = sum_t a_t V_g[t];
 *   4. y_b = bo + sum over active h of Wo[:, h*dh .. h*dh+dh-1] o_h.
 * A head that is not active for the token adds nothing to y_b: its query,
 * its pass over the cache and its Wo columns are skipped.  Arithmetic in fp32
 * on fp16 weights and caches; the output projection is reduced in a fixed
 * order (bitwise reproducible).
 */
typedef struct {
    int d;         /* model width (multiple of 8)                                  */
    int heads;     /* query heads H (1 .. 1024)                                    */
    int kv_heads;  /* key/value heads KVH, dividing H (H: multi-head attention)    */
    int head_dim;  /* dh: 64 or 128                                                */
    int rank;      /* head predictor rank (multiple of 8)                          */
    int batch;     /* sequences B, one new token each (1 .. 32)                    */
    int max_seq;   /* cache capacity smax per sequence and KV head                 */
} pi_attn_desc;

typedef struct {
    const pi_half *wqkv; /* [(H + 2 KVH) dh, d]: query rows of head h at h*dh, key rows of KV
                            head g at (H + g) dh, value rows at (H + KVH + g) dh            */
    const pi_half *bqkv; /* [(H + 2 KVH) dh] (zeros for a model without biases)           */
    const pi_half *wot;  /* [H dh, d]: Wo transposed, row j = column j of Wo              */
    const pi_half *bo;   /* [d]                                                           */
    const pi_half *p1;   /* [rank, d]  head predictor input layer                         */
    const pi_half *p2;   /* [H, rank]  head predictor output layer                        */
    const pi_half *bp;   /* [H]        head predictor bias                                */
} pi_attn_weights;

/* Bytes of workspace pi_attn_heads needs for `desc` (0 if it is invalid). */
PI_API size_t pi_attn_workspace_bytes(const pi_attn_desc *desc);

/*
 * x: [B, d] fp16.  kcache, vcache: [B, KVH, max_seq, head_dim] fp16 (in:
 * positions below pos[b] of sequence b; out: position pos[b] written).
 * pos: [B] int32 on the device.  head_mask: [B, ceil(H/32)] uint32 out (the
 * predicted-active heads).  y: [B, d] fp32 out.  All 16-byte aligned.
 * The workspace needs no zero fill.  A pos[b] outside 0 .. max_seq-1 leaves
 * sequence b's cache untouched and its y equal to bo, and sets the device
 * status read by pi_last_device_status to PI_ERR_INVALID_ARG.
 */
PI_API pi_status pi_attn_heads(const pi_attn_desc *desc, const pi_half *x, const pi_attn_weights *w,
                               pi_half *kcache, pi_half *vcache, const int32_t *pos, float tau,
                               uint32_t *head_mask, float *y, void *workspace, size_t ws_bytes,
                               void *stream);

/* How one pi_ffn_stack step of `desc` (n_layers layers with the given ranks,
 * NULL: all desc->rank) is executed on the current device.  Diagnostics: lets a
 * caller or a test see which streaming mode the batch-1 persistent kernel
 * takes for a shape.  Host only, launches nothing. */
typedef struct {
    int fused;         /* 1: one persistent launch per decode step (batch 1)      */
    int ctas;          /* its thread blocks (one per SM)                          */
    int pred_in_smem;  /* 1: a block's share of the predictor is copied whole into
                          shared memory before it is used                         */
    int p2_ring_slots; /* else: a block's P2 rows stream through this many slots of
                          16 rows (a rank whose ring cannot hold two slots runs
                          on the per-step kernels: fused = 0)                     */
    int fc_row_slots;  /* FC weight rows a block holds in shared memory at once; a
                          block whose predicted neurons need more rows (gated: 3
                          per neuron, else 2) streams them through a ring          */
    int smem_bytes;    /* dynamic shared memory per block                         */
} pi_stack_plan_t;
PI_API pi_status pi_stack_plan(const pi_layer_desc *desc, int n_layers, const int *ranks, pi_stack_plan_t *out);
/* The same plan for a device with `sm_count` SMs (1..4096) instead of the
 * current device: host only, no device is queried, so the plan can be checked
 * where there is no GPU.  PI_ERR_INVALID_ARG for a bad descriptor, layer count,
 * rank or SM count. */
PI_API pi_status pi_stack_plan_for(const pi_layer_desc *desc, int n_layers, const int *ranks, int sm_count,
                                   pi_stack_plan_t *out);

/* Number of kernel launches one pi_ffn_layer call issues for `desc` (-1 if
 * the descriptor is invalid). */
PI_API int pi_launches_per_layer(const pi_layer_desc *desc);

PI_API const char *pi_status_string(pi_status s);

/* Synchronises `stream`, then returns and clears the device status word set
 * by bounded device-side waits (PI_OK or PI_ERR_TIMEOUT). */
PI_API pi_status pi_last_device_status(void *stream);

/* Diagnostics: sets the limit of the bounded device-side waits of the launches
 * that follow (grid barriers and copy/MMA stage waits; 1 ns .. 10 s; 0 restores
 * the default 2 s).  Process-wide, for every device.  A short limit makes the
 * kernels take their failure path: the wait gives up, the device status
 * becomes PI_ERR_TIMEOUT, the block waits (always up to 2 s) for its own copies
 * and tensor-core operations in flight, frees its tensor memory and returns.
 * For testing that path; outputs of a call that timed out are undefined, and
 * a workspace used by pi_ffn_layer or pi_ffn_stack must be zero-filled again
 * before its next use. */
PI_API pi_status pi_debug_set_wait_timeout(long long timeout_ns);

/* Diagnostics: launches one wait on a word that nothing writes, bounded by
 * timeout_ns (1 ns .. 10 s).  The wait gives up, and the device status becomes
 * PI_ERR_TIMEOUT (read it with pi_last_device_status); the GPU context stays
 * usable.  For testing the bounded-wait path. */
PI_API pi_status pi_debug_wait_timeout(long long timeout_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PI_H */
