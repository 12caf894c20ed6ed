// pi_attn.cu -- the head-sparse self-attention block of one decode step.
//
// The pages describing PowerInfer note that in the self-attention block about
// half of the heads contribute little for a given input (PowerInfer summary
// (CSDN), section "Background", paragraph on activation sparsity), and that
// each layer has one activity predictor for its MLP block and one for its
// self-attention block, so that only the neurons predicted active are
// computed (unite.ai page, section on adaptive sparsity predictors).  Here the
// block's neurons are its heads:
//
//   head mask   the low-rank predictor of the FFN path with F = heads
//               (launch_predict)
//   row list    k_attn_list: query rows of the heads active for some token
//               of the batch, then every key and value row
//   projections the FFN's FC1 row paths with the activation left out
//               (launch_fc1 on a plan of projection rows: the per-token
//               kernel up to 4 tokens and at 9..15, streamed at 5..8,
//               tcgen05 at 16..32)
//   attention   k_attn_decode: per (head, token, split of the positions) a
//               pass over the key and value cache with a running softmax
//   combine     k_attn_combine: the splits of each active (head, token) are
//               merged into o_h, written where the output projection reads it;
//               the token's keys and values go into the cache as binary16
//   output      the FC2 gather-accumulate over the rows of Wo^T of the active
//               heads (launch_fc2)
//
// A head that is not predicted active for a token adds nothing to that
// token's output: its query, its pass over the cache and its output-projection
// rows are skipped.  The token's keys and values are projected for every KV
// head and stored, so the cache stays complete for later tokens.
#include <cuda_runtime.h>
#include <math.h>

#include "pi_common.cuh"
#include "pi_internal.h"

namespace pi {
namespace {

constexpr int kAttnThreads = 128;
constexpr int kMaxHeads = 1024;

PI_DEV bool head_on(const uint32_t* mask, int WH, int b, int h) {
    return (mask[(size_t)b * WH + (h >> 5)] >> (h & 31)) & 1u;
}

// Slot of every head in the union of the batch's head masks (-1: no token
// uses it), and the row list of the projections: the dh query rows of each
// union head in ascending head order, then every key and value row.
// cnt[0] = rows projected, cnt[1] = query rows (= rows of Wo^T read later).
__global__ void __launch_bounds__(256) k_attn_list(const uint32_t* __restrict__ mask, int B, int WH, int H,
                                                    int KVH, int dh, int* __restrict__ slot,
                                                    int32_t* __restrict__ idx, int32_t* __restrict__ cnt) {
    pdl_entry();
    __shared__ uint32_t un[kMaxHeads / 32];
    __shared__ int base[kMaxHeads / 32 + 1];
    __shared__ int sl[kMaxHeads];
    for (int w = threadIdx.x; w < WH; w += blockDim.x) {
        uint32_t v = 0;
        for (int b = 0; b < B; ++b) v |= mask[(size_t)b * WH + w];
        un[w] = v;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int w = 0; w < WH; ++w) {
            base[w] = acc;
            acc += __popc(un[w]);
        }
        base[WH] = acc;
    }
    __syncthreads();
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        const uint32_t word = un[h >> 5];
        const int bit = (word >> (h & 31)) & 1u;
        const int s = bit ? base[h >> 5] + __popc(word & ((1u << (h & 31)) - 1u)) : -1;
        sl[h] = s;
        slot[h] = s;
    }
    __syncthreads();
    const int nq = base[WH] * dh;
    for (int p = threadIdx.x; p < H * dh; p += blockDim.x) {
        const int h = p / dh, i = p - h * dh;
        if (sl[h] >= 0) idx[sl[h] * dh + i] = p;
    }
    for (int j = threadIdx.x; j < 2 * KVH * dh; j += blockDim.x) idx[nq + j] = H * dh + j;
    if (threadIdx.x == 0) {
        cnt[0] = nq + 2 * KVH * dh;
        cnt[1] = nq;
    }
}

// One (head, token, split of the positions) per block of 128 threads.  A group
// of DH/8 lanes takes one position at a time (16 bytes of the key and of the
// value row per lane); each group keeps a running maximum m, sum l and
// unnormalised output o over its positions, and the block merges its groups
// into the split's (m, l, o[DH]).  Positions below pos come from the cache;
// position pos is the token's own key and value, read from the projections
// and rounded to binary16 as the cache will hold them.
template <int DH>
__global__ void __launch_bounds__(kAttnThreads) k_attn_decode(
    const float* __restrict__ proj, const int* __restrict__ slot, const int32_t* __restrict__ cnt,
    const uint32_t* __restrict__ mask, int WH, const __half* __restrict__ kcache,
    const __half* __restrict__ vcache, const int32_t* __restrict__ pos, int B, int H, int KVH, int smax,
    int nsplit, float scale, float* __restrict__ part, int* status) {
    pdl_entry();
    constexpr int LPP = DH / 8;          // lanes per position
    constexpr int PPW = 32 / LPP;        // positions per warp step
    constexpr int GROUPS = (kAttnThreads / 32) * PPW;
    constexpr int U = 4;                 // positions per group requested at once
    __shared__ float sm_m[GROUPS], sm_l[GROUPS];
    __shared__ __align__(16) float sm_o[GROUPS][DH];
    const int h = blockIdx.x, b = blockIdx.y, sp = blockIdx.z;
    if (!head_on(mask, WH, b, h)) return;
    const int p = pos[b];
    if (p < 0 || p >= smax) {
        if (threadIdx.x == 0 && sp == 0) atomicExch(status, (int)PI_ERR_INVALID_ARG);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane / LPP, li = lane % LPP;
    const int gid = warp * PPW + grp;
    const int nq = cnt[1];
    const int s = slot[h];
    const int g = h / (H / KVH);
    const int n = p + 1;
    const int chunk = (n + nsplit - 1) / nsplit;
    const int t0 = sp * chunk;
    const int t1 = min(n, t0 + chunk);
    float q[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) q[e] = proj[(size_t)(s * DH + 8 * li + e) * B + b] * scale;
    float m = -INFINITY, l = 0.f, o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = 0.f;
    auto update = [&](const uint4& kw, const uint4& vw, bool valid) {
        float kf[8], vf[8];
        h8_to_f8(kw, kf);
        h8_to_f8(vw, vf);
        float sc = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) sc = fmaf(q[e], kf[e], sc);
#pragma unroll
        for (int off = LPP / 2; off > 0; off >>= 1) sc += __shfl_xor_sync(FULL, sc, off);
        if (valid) {
            const float mn = fmaxf(m, sc);
            const float corr = expf(m - mn);
            const float pw = expf(sc - mn);
            l = l * corr + pw;
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = fmaf(o[e], corr, pw * vf[e]);
            m = mn;
        }
    };
    const size_t kvbase = ((size_t)b * KVH + g) * smax * DH;
    const __half* Kb = kcache + kvbase + 8 * li;
    const __half* Vb = vcache + kvbase + 8 * li;
    const int tc1 = min(t1, p);   // cached positions of this split: [t0, tc1)
    const int stride = GROUPS;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    // every lane of a warp runs the same number of steps (the shuffles need
    // the whole warp); positions past the range are loaded as zeros and not used
    const int steps = tc1 > t0 ? (tc1 - t0 + stride - 1) / stride : 0;
    for (int k0 = 0; k0 < steps; k0 += U) {
        uint4 kw[U], vw[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = t0 + (k0 + u) * stride + gid;
            const bool ok = k0 + u < steps && t < tc1;
            kw[u] = ok ? ld_stream16(Kb + (size_t)t * DH) : zero;
            vw[u] = ok ? ld_stream16(Vb + (size_t)t * DH) : zero;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = t0 + (k0 + u) * stride + gid;
            if (k0 + u < steps) update(kw[u], vw[u], t < tc1);
        }
    }
    if (t0 <= p && p < t1 && warp == 0) {
        // the token's own key and value (position p), group 0 of warp 0
        uint32_t kh[4], vh[4];
        const float* kp = proj + (size_t)(nq + g * DH + 8 * li) * B + b;
        const float* vp = proj + (size_t)(nq + KVH * DH + g * DH + 8 * li) * B + b;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __half2 k2 = __floats2half2_rn(kp[(size_t)(2 * e) * B], kp[(size_t)(2 * e + 1) * B]);
            const __half2 v2 = __floats2half2_rn(vp[(size_t)(2 * e) * B], vp[(size_t)(2 * e + 1) * B]);
            kh[e] = *reinterpret_cast<const uint32_t*>(&k2);
            vh[e] = *reinterpret_cast<const uint32_t*>(&v2);
        }
        update(make_uint4(kh[0], kh[1], kh[2], kh[3]), make_uint4(vh[0], vh[1], vh[2], vh[3]), grp == 0);
    }
    if (li == 0) {
        sm_m[gid] = m;
        sm_l[gid] = l;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) sm_o[gid][8 * li + e] = o[e];
    __syncthreads();
    float* out = part + (((size_t)b * H + h) * nsplit + sp) * (DH + 2);
    float M = -INFINITY;
    for (int k = 0; k < GROUPS; ++k) M = fmaxf(M, sm_m[k]);
    for (int i = threadIdx.x; i < DH; i += blockDim.x) {
        float O = 0.f;
        if (M != -INFINITY)
            for (int k = 0; k < GROUPS; ++k)
                if (sm_m[k] != -INFINITY) O = fmaf(sm_o[k][i], expf(sm_m[k] - M), O);
        out[i] = O;
    }
    if (threadIdx.x == 0) {
        float L = 0.f;
        if (M != -INFINITY)
            for (int k = 0; k < GROUPS; ++k)
                if (sm_m[k] != -INFINITY) L = fmaf(sm_l[k], expf(sm_m[k] - M), L);
        out[DH] = M;
        out[DH + 1] = L;
    }
}

// Blocks x < H: head x.  For each token whose mask has the head (and a
// union head with the token's bit clear: zero) the splits are merged,
// o = sum_k O_k e^(m_k - M) / sum_k l_k e^(m_k - M), and written over the
// head's query values in the projections, which is where the output
// projection reads its inputs (list position slot*DH + i).  Blocks x >= H: KV
// head x - H of token y: its key and value, rounded to binary16, go into the
// cache at position pos.
template <int DH>
__global__ void __launch_bounds__(DH) k_attn_combine(float* __restrict__ proj, const int* __restrict__ slot,
                                                     const int32_t* __restrict__ cnt,
                                                     const uint32_t* __restrict__ mask, int WH,
                                                     const float* __restrict__ part, int nsplit,
                                                     const int32_t* __restrict__ pos, int B, int H, int KVH,
                                                     int smax, __half* __restrict__ kcache,
                                                     __half* __restrict__ vcache) {
    pdl_entry();
    const int b = blockIdx.y, i = threadIdx.x;
    const int p = pos[b];
    const bool pos_ok = p >= 0 && p < smax;
    if (blockIdx.x < H) {
        const int h = blockIdx.x;
        const int s = slot[h];
        if (s < 0) return;
        float* dst = proj + (size_t)(s * DH + i) * B + b;
        if (!pos_ok || !head_on(mask, WH, b, h)) {
            *dst = 0.f;
            return;
        }
        const float* pp = part + ((size_t)b * H + h) * nsplit * (DH + 2);
        float M = -INFINITY;
        for (int k = 0; k < nsplit; ++k) M = fmaxf(M, pp[(size_t)k * (DH + 2) + DH]);
        float O = 0.f, L = 0.f;
        for (int k = 0; k < nsplit; ++k) {
            const float mk = pp[(size_t)k * (DH + 2) + DH];
            if (mk == -INFINITY) continue;
            const float f = expf(mk - M);
            O = fmaf(pp[(size_t)k * (DH + 2) + i], f, O);
            L = fmaf(pp[(size_t)k * (DH + 2) + DH + 1], f, L);
        }
        *dst = O / L;
    } else {
        if (!pos_ok) return;
        const int g = blockIdx.x - H;
        const int nq = cnt[1];
        const size_t at = (((size_t)b * KVH + g) * smax + p) * DH + i;
        kcache[at] = __float2half_rn(proj[(size_t)(nq + g * DH + i) * B + b]);
        vcache[at] = __float2half_rn(proj[(size_t)(nq + KVH * DH + g * DH + i) * B + b]);
    }
}

}  // namespace

bool make_attn_plan(const pi_attn_desc& a, AttnPlan* out) {
    if (a.d <= 0 || a.d % 8 != 0 || a.d > (1 << 16) || a.heads < 1 || a.heads > kMaxHeads || a.kv_heads < 1 ||
        a.heads % a.kv_heads != 0 || (a.head_dim != 64 && a.head_dim != 128) || a.rank <= 0 || a.rank % 8 != 0 ||
        a.rank > 8192 || a.batch < 1 || a.batch > 32 || a.max_seq < 1 || a.max_seq > (1 << 20))
        return false;
    AttnPlan q{};
    q.d = a.d;
    q.H = a.heads;
    q.KVH = a.kv_heads;
    q.dh = a.head_dim;
    q.B = a.batch;
    q.smax = a.max_seq;
    q.WH = (q.H + 31) / 32;
    const int rows = (q.H + 2 * q.KVH) * q.dh;
    // head predictor: the FFN predictor with F = heads, on its per-token kernels
    if (!make_plan(pi_layer_desc{a.d, a.heads, a.rank, a.batch, PI_W_F16, 0}, &q.pred)) return false;
    q.pred.pred = 0;
    // projections: rows of Wqkv; output projection: rows of Wo^T
    if (!make_plan(pi_layer_desc{a.d, rows, 8, a.batch, PI_W_F16, 0}, &q.proj)) return false;
    q.proj.proj = true;
    // the projection rows are long contiguous runs (whole heads): up to 4
    // tokens the per-token row kernel (a warp per row, one token chunk)
    // streams them faster than the streamed tile path, which wins at 5..8
    if (q.B <= 4) q.proj.st = false;
    if (!make_plan(pi_layer_desc{a.d, a.heads * a.head_dim, 8, a.batch, PI_W_F16, 0}, &q.out)) return false;
    // splits of the positions: about four blocks per SM for a batch whose
    // tokens use half of the heads, at least 32 positions per split
    const int nsm = q.proj.nsm;
    int ns = (8 * nsm + q.B * q.H - 1) / (q.B * q.H);
    const int max_ns = (q.smax + 31) / 32;
    if (ns > max_ns) ns = max_ns;
    if (ns > 64) ns = 64;
    q.nsplit = ns < 1 ? 1 : ns;
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    size_t off = 0;
    q.off_pred = off;  off = up(off + q.pred.total);
    q.off_slot = off;  off = up(off + sizeof(int) * (size_t)q.H);
    q.off_cnt = off;   off = up(off + sizeof(int32_t) * 4);
    q.off_idx = off;   off = up(off + sizeof(int32_t) * (size_t)rows);
    q.off_proj = off;  off = up(off + sizeof(float) * (size_t)rows * q.B);
    q.off_ppart = off; off = up(off + sizeof(float) * q.proj.part_floats);
    q.off_apart = off; off = up(off + sizeof(float) * (size_t)q.B * q.H * q.nsplit * (q.dh + 2));
    q.off_fpart = off; off = up(off + sizeof(float) * fc2_part_floats(q.out));
    q.total = off;
    *out = q;
    return true;
}

cudaError_t launch_attn(const AttnPlan& q, const __half* x, const pi_attn_weights& w, __half* kcache,
                        __half* vcache, const int32_t* pos, float tau, uint32_t* head_mask, float* y, void* ws,
                        cudaStream_t s) {
    char* base = static_cast<char*>(ws);
    int* slot = reinterpret_cast<int*>(base + q.off_slot);
    int32_t* cnt = reinterpret_cast<int32_t*>(base + q.off_cnt);
    int32_t* idx = reinterpret_cast<int32_t*>(base + q.off_idx);
    float* proj = reinterpret_cast<float*>(base + q.off_proj);
    float* apart = reinterpret_cast<float*>(base + q.off_apart);
    float* fpart = reinterpret_cast<float*>(base + q.off_fpart);
    const __half* wqkv = reinterpret_cast<const __half*>(w.wqkv);
    cudaError_t e = launch_predict(q.pred, x, reinterpret_cast<const __half*>(w.p1),
                                   reinterpret_cast<const __half*>(w.p2), reinterpret_cast<const __half*>(w.bp),
                                   tau, head_mask, base + q.off_pred, s);
    if (e != cudaSuccess) return e;
    launch_pdl(k_attn_list, 1, 256, 0, s, static_cast<const uint32_t*>(head_mask), q.B, q.WH, q.H, q.KVH, q.dh,
               slot, idx, cnt);
    LayerPtrs pw{};
    pw.w1 = wqkv;
    pw.b1 = reinterpret_cast<const __half*>(w.bqkv);
    e = launch_fc1(q.proj, x, pw, idx, cnt, nullptr, reinterpret_cast<float*>(base + q.off_ppart), proj, nullptr, s);
    if (e != cudaSuccess) return e;
    const float scale = 1.0f / sqrtf((float)q.dh);
    const dim3 ga(q.H, q.B, q.nsplit), gc(q.H + q.KVH, q.B);
    int* status = status_word();
    if (q.dh == 128) {
        launch_pdl(k_attn_decode<128>, ga, kAttnThreads, 0, s, static_cast<const float*>(proj),
                   static_cast<const int*>(slot), static_cast<const int32_t*>(cnt),
                   static_cast<const uint32_t*>(head_mask), q.WH, static_cast<const __half*>(kcache),
                   static_cast<const __half*>(vcache), pos, q.B, q.H, q.KVH, q.smax, q.nsplit, scale, apart, status);
        launch_pdl(k_attn_combine<128>, gc, 128, 0, s, proj, static_cast<const int*>(slot),
                   static_cast<const int32_t*>(cnt), static_cast<const uint32_t*>(head_mask), q.WH,
                   static_cast<const float*>(apart), q.nsplit, pos, q.B, q.H, q.KVH, q.smax, kcache, vcache);
    } else {
        launch_pdl(k_attn_decode<64>, ga, kAttnThreads, 0, s, static_cast<const float*>(proj),
                   static_cast<const int*>(slot), static_cast<const int32_t*>(cnt),
                   static_cast<const uint32_t*>(head_mask), q.WH, static_cast<const __half*>(kcache),
                   static_cast<const __half*>(vcache), pos, q.B, q.H, q.KVH, q.smax, q.nsplit, scale, apart, status);
        launch_pdl(k_attn_combine<64>, gc, 64, 0, s, proj, static_cast<const int*>(slot),
                   static_cast<const int32_t*>(cnt), static_cast<const uint32_t*>(head_mask), q.WH,
                   static_cast<const float*>(apart), q.nsplit, pos, q.B, q.H, q.KVH, q.smax, kcache, vcache);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    LayerPtrs lw{};
    lw.w2t = w.wot;
    lw.b2 = reinterpret_cast<const __half*>(w.bo);
    return launch_fc2(q.out, proj, idx, cnt + 1, lw, nullptr, fpart, y, s);
}

}  // namespace pi
