// pi_api.cu -- the extern "C" boundary: argument validation, work planning,
// workspace layout and launch sequencing.  No arithmetic of the path lives
// here; every step runs in the kernels.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "pi_internal.h"

namespace pi {

namespace {

constexpr size_t kAlign = 256;
size_t up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

int device_sms() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

bool make_plan(const pi_layer_desc& desc, Plan* p, int sm_count) {
    if (desc.d <= 0 || desc.d % 8 != 0 || desc.ffn <= 0 || desc.rank <= 0 || desc.rank % 8 != 0 ||
        desc.batch < 1 || desc.batch > 32 || desc.d > (1 << 16) || desc.rank > 8192 ||
        desc.ffn > (1 << 22))
        return false;
    if (desc.wdtype != PI_W_F16 && desc.wdtype != PI_W_INT4_G32) return false;
    if (desc.wdtype == PI_W_INT4_G32 && desc.d % 32 != 0) return false;
    if (desc.gated != 0 && desc.gated != 1) return false;
    Plan q{};
    q.d = desc.d;
    q.F = desc.ffn;
    q.r = desc.rank;
    q.B = desc.batch;
    q.int4 = desc.wdtype == PI_W_INT4_G32;
    q.gated = desc.gated == 1;
    q.W = (q.F + 31) / 32;
    q.nsm = sm_count > 0 ? sm_count : device_sms();
    if (q.nsm <= 0) q.nsm = 1;
    // predictor P1 x: enough (row, split) warps to cover the GPU twice, splits >= 256 elements
    const int row_blocks = (q.r + 7) / 8;
    int us = (2 * q.nsm + row_blocks - 1) / row_blocks;
    const int max_us = (q.d + 255) / 256;
    if (us > max_us) us = max_us;
    if (us < 1) us = 1;
    q.u_seg = ((q.d / 8 + us - 1) / us) * 8;
    q.u_splits = (q.d + q.u_seg - 1) / q.u_seg;
    // FC2: a block covers 256 threads x (8 fp16 | 16 INT4) columns
    q.fc2_cols = 256 * (q.int4 ? 16 : 8);
    q.fc2_tiles = (q.d + q.fc2_cols - 1) / q.fc2_cols;
    int s2 = (2 * q.nsm + q.fc2_tiles - 1) / q.fc2_tiles;
    const int max_s2 = (q.F + 7) / 8;
    if (s2 > max_s2) s2 = max_s2;
    q.fc2_splits = s2 < 1 ? 1 : s2;
    // fused exchange region first (its epoch word stays at offset 0 for every
    // descriptor that shares the workspace), then the per-step buffers
    q.rmax_su = (size_t)16 * q.nsm + 2 * (size_t)q.r;
    q.xchg_bytes = up(fused_workspace_bytes(q.d, q.F, q.rmax_su, q.nsm));
    q.fused = q.B == 1 && fused_supported(q.d, q.F, q.r, q.int4, q.gated, q.nsm);
    q.tc = tc_supported(q);
    q.st = !q.tc && st_supported(q);
    q.st4 = !q.tc && !q.st && st4_supported(q);
    q.fc1_tc4 = q.st4 && tc4_supported(q);
    q.pred = tc_pred_supported(q) ? 2 : (st_pred_supported(q) ? 1 : 0);
    {
        // partial sums of whichever paths the plan takes (the stream-K sizes
        // cover the predictor and both FFN products)
        size_t part = (size_t)q.fc2_splits * q.B * q.d;
        if (q.pred == 2 || q.tc) part = std::max(part, tc_part_floats(q));
        if (q.pred == 1 || q.st) part = std::max(part, st_part_floats(q));
        if (q.st4) part = std::max(part, st4_part_floats(q));
        if (q.fc1_tc4) part = std::max(part, tc_part_floats(q));
        q.part_floats = part;
    }
    size_t off = q.xchg_bytes;
    q.off_mask = off;  off = up(off + sizeof(uint32_t) * (size_t)q.B * q.W);
    q.off_idx = off;   off = up(off + sizeof(int32_t) * (size_t)q.F);
    q.off_count = off; off = up(off + sizeof(int32_t) * 4);
    q.off_h = off;     off = up(off + sizeof(float) * (size_t)q.F * q.B);
    q.off_upart = off; off = up(off + sizeof(float) * (size_t)q.u_splits * q.B * q.r);
    q.off_part = off;  off = up(off + sizeof(float) * q.part_floats);
    q.off_xbuf = off;  off = up(off + sizeof(uint16_t) * 2 * (size_t)q.B * q.d);
    q.off_live = off;  off = up(off + sizeof(int32_t) * (size_t)q.F);
    q.off_uhl = off;   off = up(off + (q.pred == 2 ? tc_uhl_bytes(q) : q.pred == 1 ? st_u_bytes(q) : 0));
    q.total = off;
    *p = q;
    return true;
}

namespace {

pi_status from_cuda(cudaError_t e) { return e == cudaSuccess ? PI_OK : PI_ERR_CUDA; }

bool weights_ok(const Plan& p, const pi_layer_weights* w, bool need_w1, bool need_w2, bool need_pred) {
    if (!w) return false;
    if (need_w1) {
        if (!w->w1 || !w->b1 || !aligned16(w->w1)) return false;
        if (p.int4 && (!w->w1_scales || !aligned16(w->w1_scales))) return false;
        if (p.gated && (!w->wu || !aligned16(w->wu))) return false;
    }
    if (need_w2) {
        if (!w->w2t || !w->b2 || !aligned16(w->w2t)) return false;
        if (p.int4 && (!w->w2t_scales || !aligned16(w->w2t_scales))) return false;
    }
    if (need_pred) {
        if (!w->p1 || !w->p2 || !w->b1 || !aligned16(w->p1) || !aligned16(w->p2)) return false;
    }
    return true;
}

LayerPtrs ptrs(const pi_layer_weights* w) {
    LayerPtrs l;
    l.w1 = w->w1;
    l.w1s = reinterpret_cast<const __half*>(w->w1_scales);
    l.b1 = reinterpret_cast<const __half*>(w->b1);
    l.wu = reinterpret_cast<const __half*>(w->wu);
    l.w2t = w->w2t;
    l.w2ts = reinterpret_cast<const __half*>(w->w2t_scales);
    l.b2 = reinterpret_cast<const __half*>(w->b2);
    l.p1 = reinterpret_cast<const __half*>(w->p1);
    l.p2 = reinterpret_cast<const __half*>(w->p2);
    l.table = w->table;
    return l;
}

template <typename T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

}  // namespace

bool fc2_args_ok(const Plan& p, const float* h, const int32_t* idx, const int32_t* d_count,
                 const pi_layer_weights* w, const float* y) {
    return h && idx && d_count && y && aligned16(y) && weights_ok(p, w, false, true, false);
}

LayerPtrs layer_ptrs(const pi_layer_weights* w) { return ptrs(w); }

constexpr int kMaxStackLayers = 96;
constexpr long long kWaitTimeoutNs = 2000000000ll;  // 2 s per wait
std::atomic<long long> g_wait_override_ns{0};

long long wait_timeout_ns() {
    const long long v = g_wait_override_ns.load(std::memory_order_relaxed);
    return v > 0 ? v : kWaitTimeoutNs;
}

// One decode step through n layers: the fused persistent kernel when the plan
// allows it, else the per-step kernels with the normalisation between layers.
cudaError_t run_stack(const Plan& p, int n, const LayerPtrs* lp, const int* ranks, const __half* x, float tau,
                      float eps, void* ws, float* y, __half* x_trace, int32_t* layer_counts, cudaStream_t s) {
    if (layer_counts) {
        cudaError_t e = cudaMemsetAsync(layer_counts, 0, sizeof(int32_t) * 2 * (size_t)n, s);
        if (e != cudaSuccess) return e;
    }
    uint32_t* mask = at<uint32_t>(ws, p.off_mask);
    int32_t* idx = at<int32_t>(ws, p.off_idx);
    int32_t* cnt = at<int32_t>(ws, p.off_count);
    float* h = at<float>(ws, p.off_h);
    if (p.fused) {
        int rk[kMaxStackLayers];
        for (int l = 0; l < n; ++l) rk[l] = ranks ? ranks[l] : p.r;
        FusedStackArgs a{};
        a.L = n;
        a.d = p.d;
        a.F = p.F;
        a.G = p.nsm;
        a.int4 = p.int4;
        a.gated = p.gated;
        a.tau = tau;
        a.eps = eps;
        a.timeout_ns = wait_timeout_ns();
        a.layers = lp;
        a.ranks = rk;
        a.x_in = x;
        a.y_out = y;
        a.x_trace = x_trace;
        a.xchg = ws;
        a.rmax_su = p.rmax_su;
        a.mask_out = mask;
        a.idx_out = idx;
        a.count_out = cnt;
        a.h_out = h;
        a.layer_counts = layer_counts;
        FusedStackConfig fc{};
        if (fused_stack_config(a, &fc)) return launch_fused(a, s);
        // ranks too large for the persistent kernel's P2 ring: the per-step kernels
    }
    const __half* cur = x;
    __half* xbuf = at<__half>(ws, p.off_xbuf);
    for (int l = 0; l < n; ++l) {
        Plan q = p;
        q.r = ranks ? ranks[l] : p.r;
        const LayerPtrs& w = lp[l];
        cudaError_t e = launch_predict(q, cur, w.p1, w.p2, w.b1, tau, mask, ws, s);
        if (e == cudaSuccess) e = launch_compact(q, mask, nullptr, idx, nullptr, cnt, s);
        int32_t* live = at<int32_t>(ws, p.off_live);
        if (e == cudaSuccess)
            e = launch_fc1(q, cur, w, idx, cnt, q.B > 1 ? mask : nullptr, at<float>(ws, p.off_part), h, live, s);
        if (e == cudaSuccess && layer_counts) e = launch_count_active(q, cnt, h, layer_counts + 2 * l, s);
        if (e == cudaSuccess)
            e = launch_fc2(q, h, idx, cnt, w, (q.tc || q.st || q.st4) ? live : nullptr, at<float>(ws, p.off_part), y, s);
        if (e != cudaSuccess) return e;
        if (l + 1 < n) {
            __half* nxt = x_trace ? x_trace + (size_t)l * p.B * p.d : xbuf + (size_t)(l % 2) * p.B * p.d;
            e = launch_rmsnorm(p.d, p.B, y, eps, nxt, s);
            if (e != cudaSuccess) return e;
            cur = nxt;
        }
    }
    return cudaSuccess;
}

}  // namespace pi

using namespace pi;

extern "C" {

size_t pi_workspace_bytes(const pi_layer_desc* desc) {
    Plan p;
    if (!desc || !make_plan(*desc, &p)) return 0;
    return p.total;
}

pi_status pi_workspace_layout(const pi_layer_desc* desc, pi_workspace_layout_t* out) {
    Plan p;
    if (!desc || !out || !make_plan(*desc, &p)) return PI_ERR_INVALID_ARG;
    out->mask = p.off_mask;
    out->idx = p.off_idx;
    out->count = p.off_count;
    out->h = p.off_h;
    out->total = p.total;
    return PI_OK;
}

pi_status pi_predict(const pi_layer_desc* desc, const pi_half* x, const pi_half* p1, const pi_half* p2,
                     const pi_half* bpred, float tau, uint32_t* mask, void* workspace, size_t ws_bytes,
                     void* stream) {
    Plan p;
    if (!desc || !make_plan(*desc, &p)) return PI_ERR_INVALID_ARG;
    if (!x || !p1 || !p2 || !bpred || !mask || !aligned16(x) || !aligned16(p1) || !aligned16(p2))
        return PI_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || ws_bytes < p.total) return PI_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return from_cuda(launch_predict(p, reinterpret_cast<const __half*>(x), reinterpret_cast<const __half*>(p1),
                                    reinterpret_cast<const __half*>(p2), reinterpret_cast<const __half*>(bpred),
                                    tau, mask, workspace, s));
}

pi_status pi_compact(const pi_layer_desc* desc, const uint32_t* mask, const int32_t* table, int32_t* idx,
                     int32_t* orig_idx, int32_t* d_count, void* stream) {
    Plan p;
    if (!desc || !make_plan(*desc, &p)) return PI_ERR_INVALID_ARG;
    if (!mask || !idx || !d_count || (orig_idx && !table)) return PI_ERR_INVALID_ARG;
    return from_cuda(launch_compact(p, mask, table, idx, orig_idx, d_count, static_cast<cudaStream_t>(stream)));
}

pi_status pi_sparse_fc1(const pi_layer_desc* desc, const pi_half* x, const pi_layer_weights* w,
                        const int32_t* idx, const int32_t* d_count, const uint32_t* mask, float* h,
                        void* workspace, size_t ws_bytes, void* stream) {
    Plan p;
    if (!desc || !make_plan(*desc, &p)) return PI_ERR_INVALID_ARG;
    if (!x || !aligned16(x) || !idx || !d_count || !h || !weights_ok(p, w, true, false, false))
        return PI_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || ws_bytes < p.total) return PI_ERR_WORKSPACE;
    if ((size_t)8 * p.d * sizeof(uint16_t) > 200 * 1024) return PI_ERR_UNSUPPORTED;
    return from_cuda(launch_fc1(p, reinterpret_cast<const __half*>(x), ptrs(w), idx, d_count, mask,
                                at<float>(workspace, p.off_part), h, nullptr, static_cast<cudaStream_t>(stream)));
}

pi_status pi_sparse_fc2(const pi_layer_desc* desc, const float* h, const int32_t* idx, const int32_t* d_count,
                        const pi_layer_weights* w, float* y, void* workspace, size_t ws_bytes, void* stream) {
    Plan p;
    if (!desc || !make_plan(*desc, &p)) return PI_ERR_INVALID_ARG;
    if (!h || !idx || !d_count || !y || !aligned16(y) || !weights_ok(p, w, false, true, false))
        return PI_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || ws_bytes < p.total) return PI_ERR_WORKSPACE;
    return from_cuda(launch_fc2(p, h, idx, d_count, ptrs(w), nullptr, at<float>(workspace, p.off_part), y,
                                static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// Checks the second tier against the plan and converts it (no second tier
// when every row is hot).
bool cold_ok(const Plan& p, const pi_cold_tier* c, bool need_w1, bool need_w2, ColdPtrs* out) {
    if (!c || c->n_hot < 0 || c->n_hot > p.F) return false;
    ColdPtrs k = no_cold_tier();
    if (c->n_hot == p.F) {
        *out = k;
        return true;
    }
    if (need_w1) {
        if (!c->w1 || !aligned16(c->w1)) return false;
        if (p.int4 && !c->w1_scales) return false;
        if (p.gated && (!c->wu || !aligned16(c->wu))) return false;
    }
    if (need_w2) {
        if (!c->w2t || !aligned16(c->w2t)) return false;
        if (p.int4 && !c->w2t_scales) return false;
    }
    k.n_hot = c->n_hot;
    k.w1 = c->w1;
    k.w1s = reinterpret_cast<const __half*>(c->w1_scales);
    k.wu = reinterpret_cast<const __half*>(c->wu);
    k.w2t = c->w2t;
    k.w2ts = reinterpret_cast<const __half*>(c->w2t_scales);
    *out = k;
    return true;
}

}  // namespace

extern "C" {

pi_status pi_sparse_fc1_tiered(const pi_layer_desc* desc, const pi_half* x, const pi_layer_weights* w,
                               const pi_cold_tier* cold, const int32_t* idx, const int32_t* d_count,
                               const uint32_t* mask, float* h, void* stream) {
    Plan p;
    if (!desc || !make_plan(*desc, &p)) return PI_ERR_INVALID_ARG;
    ColdPtrs c;
    if (!x || !aligned16(x) || !idx || !d_count || !h || !weights_ok(p, w, true, false, false) ||
        !cold_ok(p, cold, true, false, &c))
        return PI_ERR_INVALID_ARG;
    if ((size_t)8 * p.d * sizeof(uint16_t) > 200 * 1024) return PI_ERR_UNSUPPORTED;
    return from_cuda(launch_fc1_chunked(p, reinterpret_cast<const __half*>(x), ptrs(w), c, idx, d_count,
                                        p.B > 1 ? mask : nullptr, h, static_cast<cudaStream_t>(stream)));
}

pi_status pi_sparse_fc2_tiered(const pi_layer_desc* desc, const float* h, const int32_t* idx,
                               const int32_t* d_count, const pi_layer_weights* w, const pi_cold_tier* cold,
                               float* y, void* workspace, size_t ws_bytes, void* stream) {
    Plan p;
    if (!desc || !make_plan(*desc, &p)) return PI_ERR_INVALID_ARG;
    ColdPtrs c;
    if (!h || !idx || !d_count || !y || !aligned16(y) || !weights_ok(p, w, false, true, false) ||
        !cold_ok(p, cold, false, true, &c))
        return PI_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || ws_bytes < p.total) return PI_ERR_WORKSPACE;
    return from_cuda(launch_fc2_chunked(p, h, idx, d_count, ptrs(w), c, at<float>(workspace, p.off_part), y,
                                        static_cast<cudaStream_t>(stream)));
}

pi_status pi_ffn_layer_tiered(const pi_layer_desc* desc, const pi_half* x, const pi_layer_weights* w,
                              const pi_cold_tier* cold, float tau, void* workspace, size_t ws_bytes, float* y,
                              void* stream) {
    Plan p;
    if (!desc || !make_plan(*desc, &p)) return PI_ERR_INVALID_ARG;
    ColdPtrs c;
    if (!x || !aligned16(x) || !y || !aligned16(y) || !weights_ok(p, w, true, true, true) ||
        !cold_ok(p, cold, true, true, &c))
        return PI_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || ws_bytes < p.total) return PI_ERR_WORKSPACE;
    if ((size_t)8 * p.d * sizeof(uint16_t) > 200 * 1024) return PI_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const LayerPtrs l = ptrs(w);
    const __half* xh = reinterpret_cast<const __half*>(x);
    uint32_t* mask = at<uint32_t>(workspace, p.off_mask);
    int32_t* idx = at<int32_t>(workspace, p.off_idx);
    int32_t* cnt = at<int32_t>(workspace, p.off_count);
    float* h = at<float>(workspace, p.off_h);
    cudaError_t e = launch_predict(p, xh, l.p1, l.p2, l.b1, tau, mask, workspace, s);
    if (e == cudaSuccess) e = launch_compact(p, mask, nullptr, idx, nullptr, cnt, s);
    if (e == cudaSuccess) e = launch_fc1_chunked(p, xh, l, c, idx, cnt, p.B > 1 ? mask : nullptr, h, s);
    if (e == cudaSuccess) e = launch_fc2_chunked(p, h, idx, cnt, l, c, at<float>(workspace, p.off_part), y, s);
    return from_cuda(e);
}

pi_status pi_ffn_layer(const pi_layer_desc* desc, const pi_half* x, const pi_layer_weights* w, float tau,
                       void* workspace, size_t ws_bytes, float* y, void* stream) {
    Plan p;
    if (!desc || !make_plan(*desc, &p)) return PI_ERR_INVALID_ARG;
    if (!x || !aligned16(x) || !y || !aligned16(y) || !weights_ok(p, w, true, true, true))
        return PI_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || ws_bytes < p.total) return PI_ERR_WORKSPACE;
    if ((size_t)8 * p.d * sizeof(uint16_t) > 200 * 1024) return PI_ERR_UNSUPPORTED;
    const LayerPtrs l = ptrs(w);
    return from_cuda(run_stack(p, 1, &l, nullptr, reinterpret_cast<const __half*>(x), tau, 0.f, workspace, y,
                               nullptr, nullptr, static_cast<cudaStream_t>(stream)));
}

pi_status pi_ffn_stack(const pi_layer_desc* desc, int n_layers, const pi_layer_weights* layers, const int* ranks,
                       const pi_half* x, float tau, float eps, void* workspace, size_t ws_bytes, float* y,
                       pi_half* x_trace, int32_t* layer_counts, void* stream) {
    Plan p;
    if (!desc || !make_plan(*desc, &p)) return PI_ERR_INVALID_ARG;
    if (n_layers < 1 || n_layers > kMaxStackLayers || !layers || !x || !aligned16(x) || !y || !aligned16(y) ||
        !(eps >= 0.f))
        return PI_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || ws_bytes < p.total) return PI_ERR_WORKSPACE;
    if ((size_t)8 * p.d * sizeof(uint16_t) > 200 * 1024) return PI_ERR_UNSUPPORTED;
    LayerPtrs lp[kMaxStackLayers];
    for (int l = 0; l < n_layers; ++l) {
        if (!weights_ok(p, &layers[l], true, true, true)) return PI_ERR_INVALID_ARG;
        if (ranks && (ranks[l] <= 0 || ranks[l] % 8 != 0 || ranks[l] > p.r)) return PI_ERR_INVALID_ARG;
        lp[l] = ptrs(&layers[l]);
    }
    return from_cuda(run_stack(p, n_layers, lp, ranks, reinterpret_cast<const __half*>(x), tau, eps, workspace, y,
                               reinterpret_cast<__half*>(x_trace), layer_counts, static_cast<cudaStream_t>(stream)));
}

pi_status pi_rmsnorm_half(int d, int batch, const float* y, float eps, pi_half* x_out, void* stream) {
    if (d <= 0 || d % 4 != 0 || batch <= 0 || !y || !x_out || !(eps >= 0.f) || !aligned16(y) ||
        (reinterpret_cast<uintptr_t>(x_out) & 7u) != 0)
        return PI_ERR_INVALID_ARG;
    return from_cuda(launch_rmsnorm(d, batch, y, eps, reinterpret_cast<__half*>(x_out),
                                    static_cast<cudaStream_t>(stream)));
}

namespace {
pi_status stack_plan(const pi_layer_desc* desc, int n_layers, const int* ranks, int sm_count, pi_stack_plan_t* out) {
    Plan p;
    if (!desc || !out || !make_plan(*desc, &p, sm_count)) return PI_ERR_INVALID_ARG;
    if (n_layers < 1 || n_layers > kMaxStackLayers) return PI_ERR_INVALID_ARG;
    *out = pi_stack_plan_t{};
    if (!p.fused) return PI_OK;
    int rk[kMaxStackLayers];
    for (int l = 0; l < n_layers; ++l) {
        rk[l] = ranks ? ranks[l] : p.r;
        if (rk[l] <= 0 || rk[l] % 8 != 0 || rk[l] > p.r) return PI_ERR_INVALID_ARG;
    }
    FusedStackArgs a{};
    a.L = n_layers;
    a.d = p.d;
    a.F = p.F;
    a.G = p.nsm;
    a.int4 = p.int4;
    a.gated = p.gated;
    a.ranks = rk;
    a.rmax_su = p.rmax_su;
    FusedStackConfig c{};
    if (!fused_stack_config(a, &c)) return PI_OK;
    out->fused = 1;
    out->ctas = p.nsm;
    out->pred_in_smem = c.pred_smem;
    out->p2_ring_slots = c.ring_slots;
    out->fc_row_slots = c.fc_slots;
    out->smem_bytes = c.smem_bytes;
    return PI_OK;
}
}  // namespace

pi_status pi_stack_plan(const pi_layer_desc* desc, int n_layers, const int* ranks, pi_stack_plan_t* out) {
    return stack_plan(desc, n_layers, ranks, 0, out);
}

pi_status pi_stack_plan_for(const pi_layer_desc* desc, int n_layers, const int* ranks, int sm_count,
                            pi_stack_plan_t* out) {
    if (sm_count < 1 || sm_count > 4096) return PI_ERR_INVALID_ARG;
    return stack_plan(desc, n_layers, ranks, sm_count, out);
}

int pi_launches_per_layer(const pi_layer_desc* desc) {
    Plan p;
    if (!desc || !make_plan(*desc, &p)) return -1;
    int chunks = 0;
    for (int b0 = 0; b0 < p.B;) {
        const int left = p.B - b0;
        b0 += left >= 8 ? 8 : left >= 4 ? 4 : left >= 2 ? 2 : 1;
        ++chunks;
    }
    if (p.fused) {
        // one persistent kernel, when its P2 ring fits the rank
        const int rk[1] = {p.r};
        FusedStackArgs a{};
        a.L = 1;
        a.d = p.d;
        a.F = p.F;
        a.G = p.nsm;
        a.int4 = p.int4;
        a.gated = p.gated;
        a.ranks = rk;
        a.rmax_su = p.rmax_su;
        FusedStackConfig c{};
        if (fused_stack_config(a, &c)) return 1;
    }
    // predictor: 2 per token chunk; compaction: 1; then FC1 + FC2 + the FC2
    // reduction (tcgen05 path: all tokens at once) or FC1 and FC2 per chunk + 1
    // tcgen05 path: predictor u + finish + s, compaction, FC1 + finish, FC2 + reduction
    // predictor: u GEMM + finish + s GEMM on the streamed paths, else 2 per token chunk
    const int pred = (p.pred == 2 && p.r % 16 == 0) ? 3 : p.pred_units() ? 2 : p.pred == 1 ? 3 : 2 * chunks;
    // FC1 + finish and FC2 + reduction on the streamed paths, else 1 per chunk each + 1
    const int ffn = (p.tc || p.st || p.st4) ? 4 : chunks + chunks + 1;
    return pred + 1 + ffn;
}

const char* pi_status_string(pi_status s) {
    switch (s) {
        case PI_OK: return "ok";
        case PI_ERR_INVALID_ARG: return "invalid argument";
        case PI_ERR_UNSUPPORTED: return "unsupported request";
        case PI_ERR_CUDA: return "CUDA error";
        case PI_ERR_TIMEOUT: return "device-side wait timed out";
        case PI_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    }
    return "unknown status";
}

size_t pi_attn_workspace_bytes(const pi_attn_desc* desc) {
    AttnPlan q;
    if (!desc || !make_attn_plan(*desc, &q)) return 0;
    return q.total;
}

pi_status pi_attn_heads(const pi_attn_desc* desc, const pi_half* x, const pi_attn_weights* w, pi_half* kcache,
                        pi_half* vcache, const int32_t* pos, float tau, uint32_t* head_mask, float* y,
                        void* workspace, size_t ws_bytes, void* stream) {
    AttnPlan q;
    if (!desc || !make_attn_plan(*desc, &q)) return PI_ERR_INVALID_ARG;
    if (!x || !w || !kcache || !vcache || !pos || !head_mask || !y || !aligned16(x) || !aligned16(kcache) ||
        !aligned16(vcache) || !aligned16(y) || !aligned16(head_mask))
        return PI_ERR_INVALID_ARG;
    if (!w->wqkv || !w->bqkv || !w->wot || !w->bo || !w->p1 || !w->p2 || !w->bp || !aligned16(w->wqkv) ||
        !aligned16(w->wot) || !aligned16(w->p1) || !aligned16(w->p2))
        return PI_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || ws_bytes < q.total) return PI_ERR_WORKSPACE;
    return from_cuda(launch_attn(q, reinterpret_cast<const __half*>(x), *w, reinterpret_cast<__half*>(kcache),
                                 reinterpret_cast<__half*>(vcache), pos, tau, head_mask, y, workspace,
                                 static_cast<cudaStream_t>(stream)));
}

pi_status pi_last_device_status(void* stream) {
    int v = 0;
    if (read_and_clear_status(&v, static_cast<cudaStream_t>(stream)) != cudaSuccess) return PI_ERR_CUDA;
    return v == 0 ? PI_OK : static_cast<pi_status>(v);
}

pi_status pi_debug_set_wait_timeout(long long timeout_ns) {
    if (timeout_ns < 0 || timeout_ns > 10000000000ll) return PI_ERR_INVALID_ARG;
    g_wait_override_ns.store(timeout_ns, std::memory_order_relaxed);
    return PI_OK;
}

pi_status pi_debug_wait_timeout(long long timeout_ns, void* stream) {
    if (timeout_ns <= 0 || timeout_ns > 10000000000ll) return PI_ERR_INVALID_ARG;
    return from_cuda(launch_wait_nothing(timeout_ns, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
