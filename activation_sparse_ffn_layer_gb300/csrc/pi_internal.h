// pi_internal.h -- launchers shared between the C-ABI layer and the kernel files.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/pi.h"

namespace pi {

// Launch `kernel` with programmatic dependent launch allowed, so that its grid
// is scheduled while the previous kernel on the stream finishes; the kernel
// must begin with pdl_entry() (or wait with griddepcontrol.wait before it
// reads another kernel's output or writes global memory).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Work split chosen for one layer descriptor on the current device.  Both the
// workspace size and every launch are derived from it, so they always agree.
struct Plan {
    int d, F, r, B;
    bool int4, gated;
    int W;          // mask words per token, ceil(F/32)
    int nsm;        // SMs of the device
    int u_splits;   // predictor P1 x: splits of d (partial sums reduced in fixed order)
    int u_seg;      // elements of d per split (multiple of 8)
    int fc2_cols;   // columns per FC2 block
    int fc2_tiles;  // ceil(d / fc2_cols)
    int fc2_splits; // neuron splits of FC2 (partials reduced in fixed order)
    // workspace offsets (bytes, 256-aligned); the fused exchange region comes first
    size_t xchg_bytes, rmax_su;
    bool fused;     // pi_ffn_layer / pi_ffn_stack take the fused persistent kernel
    bool tc;        // FC1 / FC2 take the tcgen05 batched path (batch 16..32, fp16 weights)
    bool st;        // ... or the CUDA-core streamed batched path (batch 2..8, fp16 weights)
    bool st4;       // ... or its INT4 variant (batch 2..16, ReLU FFN)
    bool fc1_tc4;   // INT4 FC1 on the tensor cores (codes as fp16, group scales in the epilogue; batch 16-32)
    bool proj;      // rows are a plain projection (bias, no activation): the
                    // query/key/value rows of the attention block, not FFN rows
    int pred;       // predictor path (its weights are fp16 for every weight type):
                    // 2 tcgen05 (batch 16..32), 1 streamed CUDA cores (batch 2..8), 0 chunked
    // predictor of a small batch in one pass over P2 (16-row warp units, all
    // tokens at once): up to 2 tokens at any rank, up to 4 up to rank 512
    // (past that the streamed kernel is faster at 3-4 tokens)
    bool pred_units() const { return pred != 2 && (B <= 2 || (B <= 4 && r <= 512)); }
    size_t part_floats;  // split partial sums: the largest need of the predictor, FC1 and FC2 paths taken
    size_t off_mask, off_idx, off_count, off_h, off_upart, off_part, off_xbuf, off_live, off_uhl, total;
};

// sm_count > 0 plans for a device with that many SMs instead of the current one
bool make_plan(const pi_layer_desc& desc, Plan* p, int sm_count = 0);

// Limit of the bounded device-side waits of the next launches: 2 s, unless a
// caller set another one with pi_debug_set_wait_timeout.  Draining a CTA's own
// copies and MMAs after a failed wait always gets kDrainTimeoutNs, so a short
// wait limit never lets a CTA leave with its copies in flight.
long long wait_timeout_ns();
constexpr long long kDrainTimeoutNs = 2000000000ll;

struct LayerPtrs {
    const void* w1;
    const __half* w1s;
    const __half* b1;
    const __half* wu;
    const void* w2t;
    const __half* w2ts;
    const __half* b2;
    const __half* p1;
    const __half* p2;
    const int32_t* table;
};

// Second tier of a layer's FC rows: storage rows k >= n_hot are read from
// these arrays at row k - n_hot (n_hot >= F: no second tier).
struct ColdPtrs {
    int n_hot;
    const void* w1;
    const __half* w1s;
    const __half* wu;
    const void* w2t;
    const __half* w2ts;
};
inline ColdPtrs no_cold_tier() { return ColdPtrs{0x7fffffff, nullptr, nullptr, nullptr, nullptr, nullptr}; }

// FC1 / FC2 on the per-token CUDA-core kernels (token chunks of <= 8) with a
// second tier of rows; plain 16-byte loads, so the second tier may be host
// memory the GPU addresses directly.
cudaError_t launch_fc1_chunked(const Plan& p, const __half* x, const LayerPtrs& w, const ColdPtrs& cold,
                               const int32_t* idx, const int32_t* count, const uint32_t* mask, float* h,
                               cudaStream_t s);
cudaError_t launch_fc2_chunked(const Plan& p, const float* h, const int32_t* idx, const int32_t* count,
                               const LayerPtrs& w, const ColdPtrs& cold, float* partial, float* y, cudaStream_t s);

// ws: the layer workspace (u partial sums and, on the tcgen05 path, u hi | lo rows)
cudaError_t launch_predict(const Plan& p, const __half* x, const __half* p1, const __half* p2,
                           const __half* bpred, float tau, uint32_t* mask, void* ws, cudaStream_t s);
cudaError_t launch_compact(const Plan& p, const uint32_t* mask, const int32_t* table, int32_t* idx,
                           int32_t* orig, int32_t* count, cudaStream_t s);
// live (nullable): FC1 marks listed rows whose h is non-zero for some token
// (tcgen05 path only); FC2 may then skip the other rows' W2t reads.
cudaError_t launch_fc1(const Plan& p, const __half* x, const LayerPtrs& w, const int32_t* idx,
                       const int32_t* count, const uint32_t* mask, float* partial, float* h, int32_t* live,
                       cudaStream_t s);
cudaError_t launch_fc2(const Plan& p, const float* h, const int32_t* idx, const int32_t* count,
                       const LayerPtrs& w, const int32_t* live, float* partial, float* y, cudaStream_t s);
// ---- head-sparse attention block (pi_attn.cu) ----
struct AttnPlan {
    int d, H, KVH, dh, B, smax, WH, nsplit;
    Plan pred;   // head predictor (F = heads)
    Plan proj;   // query/key/value projections (F = rows of Wqkv)
    Plan out;    // output projection (F = rows of Wo^T)
    size_t off_pred, off_slot, off_cnt, off_idx, off_proj, off_ppart, off_apart, off_fpart, total;
};
bool make_attn_plan(const pi_attn_desc& a, AttnPlan* out);
cudaError_t launch_attn(const AttnPlan& q, const __half* x, const pi_attn_weights& w, __half* kcache,
                        __half* vcache, const int32_t* pos, float tau, uint32_t* head_mask, float* y, void* ws,
                        cudaStream_t s);

// partial-sum floats of the FC2 path launch_fc2 takes for this plan (FC2 alone)
size_t fc2_part_floats(const Plan& p);
cudaError_t launch_rmsnorm(int d, int B, const float* y, float eps, __half* x, cudaStream_t s);
// out[0] = *count, out[1] = listed neurons whose h is non-zero for some token
cudaError_t launch_count_active(const Plan& p, const int32_t* count, const float* h, int32_t* out, cudaStream_t s);

// ---- tcgen05 batched path (pi_tc.cu) ----
bool tc_supported(const Plan& p);
bool tc_pred_supported(const Plan& p);   // predictor only (any weight type)
int tc_tokens(const Plan& p);       // N of the MMAs: batch rounded up to 16 or 32
size_t tc_part_floats(const Plan& p);  // partial tiles of the stream-K splits
size_t tc_fc2_part_floats(const Plan& p);  // ... of the FC2 split alone
size_t tc_uhl_bytes(const Plan& p);    // u as fp16 hi | lo rows
cudaError_t launch_predict_tc(const Plan& p, const __half* x, const __half* p1, const __half* p2,
                              const __half* bpred, float tau, uint32_t* mask, float* part, __half* uhl,
                              cudaStream_t s);
cudaError_t launch_fc1_tc(const Plan& p, const __half* x, const LayerPtrs& w, const int32_t* idx,
                          const int32_t* count, const uint32_t* mask, float* part, float* h, int32_t* live,
                          cudaStream_t s);
// INT4 FC2 at 16 tokens on the tensor cores (plans with fc1_tc4)
cudaError_t launch_fc2_tc4(const Plan& p, const float* h, const int32_t* idx, const int32_t* count,
                           const LayerPtrs& w, const int32_t* live, float* partial, float* y, cudaStream_t s);
cudaError_t launch_fc2_tc(const Plan& p, const float* h, const int32_t* idx, const int32_t* count,
                          const LayerPtrs& w, const int32_t* live, float* partial, float* y, cudaStream_t s);
bool tc4_supported(const Plan& p);
cudaError_t launch_fc1_tc4(const Plan& p, const __half* x, const LayerPtrs& w, const int32_t* idx,
                           const int32_t* count, const uint32_t* mask, float* part, float* h, int32_t* live,
                           cudaStream_t s);

// fixed-order finishing of the stream-K partials (shared by the batched paths):
// nt = partial columns per token group, G = CTAs of the split, slots = tiles per
// CTA, nk = K-chunks per FC1 row, tw = FC2 column-tile width, nb tokens from b0
cudaError_t launch_fc1_finish(const Plan& p, int nt, int G, int slots, int nk, const float* part,
                              const int32_t* count, const int32_t* idx, const __half* b1, const uint32_t* mask,
                              float* h, int32_t* live, cudaStream_t s);
cudaError_t launch_fc2_reduce(const Plan& p, int nt, int G, int slots, int tw, int nb, int b0, const float* part,
                              const int32_t* count, const __half* b2, float* y, cudaStream_t s);

// ---- CUDA-core streamed batched path (pi_stream.cu, batch 2..8, fp16 weights) ----
bool st_supported(const Plan& p);
bool st_pred_supported(const Plan& p);   // predictor only (any weight type)
int st_tokens(const Plan& p);          // token slots of the kernels: 2, 4 or 8
size_t st_part_floats(const Plan& p);
size_t st_fc2_part_floats(const Plan& p);
size_t st_u_bytes(const Plan& p);      // u as fp32 rows [B][r]
cudaError_t launch_predict_st(const Plan& p, const __half* x, const __half* p1, const __half* p2,
                              const __half* bpred, float tau, uint32_t* mask, float* part, float* u32,
                              cudaStream_t s);
cudaError_t launch_fc1_st(const Plan& p, const __half* x, const LayerPtrs& w, const int32_t* idx,
                          const int32_t* count, const uint32_t* mask, float* part, float* h, int32_t* live,
                          cudaStream_t s);
cudaError_t launch_fc2_st(const Plan& p, const float* h, const int32_t* idx, const int32_t* count,
                          const LayerPtrs& w, const int32_t* live, float* partial, float* y, cudaStream_t s);

// ---- CUDA-core streamed batched path for INT4 weights (pi_stream4.cu, batch 2..16) ----
bool st4_supported(const Plan& p);
size_t st4_part_floats(const Plan& p);
size_t st4_fc2_part_floats(const Plan& p);
cudaError_t launch_fc1_st4(const Plan& p, const __half* x, const LayerPtrs& w, const int32_t* idx,
                           const int32_t* count, const uint32_t* mask, float* part, float* h, int32_t* live,
                           cudaStream_t s);
cudaError_t launch_fc2_st4(const Plan& p, const float* h, const int32_t* idx, const int32_t* count,
                           const LayerPtrs& w, const int32_t* live, float* partial, float* y, cudaStream_t s);

// ---- fused persistent stack (batch 1) ----
struct FusedStackArgs {
    int L, d, F, G;
    bool int4, gated;
    float tau, eps;
    long long timeout_ns;
    const LayerPtrs* layers;  // [L]
    const int* ranks;         // [L]
    const __half* x_in;       // [d]
    float* y_out;             // [d]
    __half* x_trace;          // nullable [L-1][d]
    void* xchg;               // exchange region (zero-filled before first use)
    size_t rmax_su;           // capacity of the u-partial exchange, entries
    uint32_t* mask_out;
    int32_t* idx_out;
    int32_t* count_out;
    float* h_out;
    int32_t* layer_counts;    // nullable [L][2] (zeroed by the caller of launch_fused)
};
size_t fused_workspace_bytes(int d, int F, size_t rmax_su, int G);
bool fused_supported(int d, int F, int rmax, bool int4, bool gated, int G);
cudaError_t launch_fused(const FusedStackArgs& a, cudaStream_t s);
// How a stack step would run on the fused kernel (shapes and ranks of `a`
// only; its pointers are not read).  False if the fused kernel cannot take it.
struct FusedStackConfig {
    int pred_smem;   // predictor slices staged whole in shared memory
    int ring_slots;  // else P2 units stream through this many slots
    int fc_slots;    // FC row slots
    int smem_bytes;  // dynamic shared memory per CTA
};
bool fused_stack_config(const FusedStackArgs& a, FusedStackConfig* out);
cudaError_t launch_wait_nothing(long long timeout_ns, cudaStream_t s);
cudaError_t read_and_clear_status(int* out, cudaStream_t s);
// Device address of the status word that bounded waits set on expiry (current device).
int* status_word();

// Argument checks of pi_sparse_fc2 (without its workspace) and the weight
// pointer bundle, shared with the allocation-free FC2 entry point.
bool fc2_args_ok(const Plan& p, const float* h, const int32_t* idx, const int32_t* d_count,
                 const pi_layer_weights* w, const float* y);
LayerPtrs layer_ptrs(const pi_layer_weights* w);

}  // namespace pi
