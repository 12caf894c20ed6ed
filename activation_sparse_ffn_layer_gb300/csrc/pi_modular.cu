// pi_modular.cu -- the decode path as separate kernels (one per step).
//
//   predictor       k_predict_u (P1 x, split over d) + k_predict_s (P2 u + b > tau, ballot)
//   compaction      k_compact   (popcount + block scan, ascending rows)
//   FC1             k_fc1       (row gather, 16-byte loads, warp-shuffle dot products,
//                                bias + ReLU (+ gate) fused)
//   FC2             k_fc2_part  (gather-accumulate over W2t rows, neuron splits)
//                   k_fc2_reduce(fixed-order sum of the splits + b2: no atomics)
//   normalisation   k_rmsnorm
//
// The math follows the PowerInfer summary (CSDN), sections "Background"
// (FC1 -> ReLU -> FC2, neurons are rows/columns), "Neuron-aware operator"
// (test each neuron, touch only active rows/columns), "Adaptive sparse
// predictor" and "Neuron placement and management" (neuron table).
#include <cuda_runtime.h>

#include "pi_common.cuh"
#include "pi_internal.h"

namespace pi {

// ------------------------------------------------------------------ predictor

// upart[s][b][i] = sum over split s of d of P1[i, c] x_b[c]; one warp per row.
template <int TB>
__global__ void __launch_bounds__(256) k_predict_u(const __half* __restrict__ x, int B, int b0,
                                                   const __half* __restrict__ p1, int d, int r,
                                                   int seg, float* __restrict__ upart) {
    pdl_entry();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x * 8 + warp;
    const int s = blockIdx.y;
    if (i >= r) return;
    const int c0 = s * seg;
    const int c1 = min(d, c0 + seg);
    float acc[TB];
#pragma unroll
    for (int t = 0; t < TB; ++t) acc[t] = 0.f;
    const __half* row = p1 + (size_t)i * d;
#pragma unroll 2
    for (int c = c0 + lane * 8; c < c1; c += 256) {
        float wf[8];
        h8_to_f8(ld_stream16(row + c), wf);
#pragma unroll
        for (int t = 0; t < TB; ++t) {
            float xf[8];
            h8_to_f8(__ldg(reinterpret_cast<const uint4*>(x + (size_t)(b0 + t) * d + c)), xf);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[t] = fmaf(wf[e], xf[e], acc[t]);
        }
    }
#pragma unroll
    for (int t = 0; t < TB; ++t) acc[t] = warp_sum(acc[t]);
    if (lane == 0) {
#pragma unroll
        for (int t = 0; t < TB; ++t) upart[((size_t)s * B + b0 + t) * r + i] = acc[t];
    }
}

// mask[b][w] bit e = (P2[32w+e] . u_b + bias[32w+e] > tau).  One warp per mask
// word; G lanes share a row of P2 (16-byte loads), 32/G rows per step.
template <int TB>
__global__ void __launch_bounds__(128) k_predict_s(const __half* __restrict__ p2,
                                                   const __half* __restrict__ bias,
                                                   const float* __restrict__ upart, int usplits,
                                                   int B, int b0, int r, int F, int W, float tau,
                                                   uint32_t* __restrict__ mask) {
    pdl_entry();
    extern __shared__ __align__(16) float us[];  // [TB][r]
    for (int e = threadIdx.x; e < TB * r; e += blockDim.x) {
        const int t = e / r, i = e - t * r;
        float v = 0.f;
        for (int s = 0; s < usplits; ++s) v += upart[((size_t)s * B + b0 + t) * r + i];
        us[e] = v;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int w = blockIdx.x * 4 + warp;
    if (w >= W) return;
    const int nvec = r / 8;
    int G = 1;
    while (G * 2 <= nvec && G * 2 <= 32) G *= 2;
    const int rpp = 32 / G;
    const int g = lane / G, t = lane % G;
    uint32_t bits[TB];
#pragma unroll
    for (int tt = 0; tt < TB; ++tt) bits[tt] = 0u;
    for (int step = 0; step < G; ++step) {
        const int k = w * 32 + step * rpp + g;
        float acc[TB];
#pragma unroll
        for (int tt = 0; tt < TB; ++tt) acc[tt] = 0.f;
        if (k < F) {
            const __half* row = p2 + (size_t)k * r;
            for (int v = t; v < nvec; v += G) {
                float pf[8];
                h8_to_f8(ld_stream16(row + v * 8), pf);
#pragma unroll
                for (int tt = 0; tt < TB; ++tt) {
                    const float4* u4 = reinterpret_cast<const float4*>(us + tt * r + v * 8);
                    const float4 a = u4[0], b = u4[1];
                    acc[tt] = fmaf(pf[0], a.x, acc[tt]);
                    acc[tt] = fmaf(pf[1], a.y, acc[tt]);
                    acc[tt] = fmaf(pf[2], a.z, acc[tt]);
                    acc[tt] = fmaf(pf[3], a.w, acc[tt]);
                    acc[tt] = fmaf(pf[4], b.x, acc[tt]);
                    acc[tt] = fmaf(pf[5], b.y, acc[tt]);
                    acc[tt] = fmaf(pf[6], b.z, acc[tt]);
                    acc[tt] = fmaf(pf[7], b.w, acc[tt]);
                }
            }
        }
        for (int o = G / 2; o > 0; o >>= 1) {
#pragma unroll
            for (int tt = 0; tt < TB; ++tt) acc[tt] += __shfl_xor_sync(FULL, acc[tt], o);
        }
        const float bk = (k < F) ? __half2float(bias[k]) : 0.f;
#pragma unroll
        for (int tt = 0; tt < TB; ++tt) {
            const bool pred = (t == 0) && (k < F) && (acc[tt] + bk > tau);
            const uint32_t bal = __ballot_sync(FULL, pred);
            for (int gg = 0; gg < rpp; ++gg)
                if ((bal >> (gg * G)) & 1u) bits[tt] |= 1u << (step * rpp + gg);
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int tt = 0; tt < TB; ++tt) mask[(size_t)(b0 + tt) * W + w] = bits[tt];
    }
}

// TB tokens (1..4): mask bits of 16-row units.  A warp takes unit m (rows 16m
// .. 16m+15), its lanes the rows' 8-element vectors v = lane, lane + 32, ...;
// the 16 rows' vectors of one step are requested before any arithmetic on them
// and used for every token.  A halving butterfly then leaves row k's dot
// product in lanes 2k', 2k'+1 (k = fold16_row), and one ballot per token gives
// the unit's 16 mask bits, stored as the low or high half of mask word m / 2
// (every unit up to 2 W is written, the ones past F as zeros).  u is the sum of
// the split partials, staged per block.
template <int TB>
__global__ void __launch_bounds__(256) k_predict_s1(const __half* __restrict__ p2, const __half* __restrict__ bias,
                                                    const float* __restrict__ upart, int usplits, int B, int b0,
                                                    int r, int F, int W, float tau, uint32_t* __restrict__ mask) {
    extern __shared__ __align__(16) float us[];  // [TB][r]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m = blockIdx.x * 8 + warp;
    const int nvec = r / 8;
    // this lane's vectors of the unit's 16 rows at step vi0 (zero past F or r)
    auto load = [&](int vi0, uint4 (&w)[16]) {
        const int vi = vi0 + lane;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int row = 16 * m + k;
            w[k] = m < 2 * W && vi < nvec && row < F ? ld_stream16(p2 + (size_t)row * r + vi * 8)
                                                     : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    // the first step's rows do not depend on u: they are requested before
    // this grid waits for the one that writes the u partials (launched as its
    // programmatic dependent)
    uint4 w[16];
    load(0, w);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    for (int e = threadIdx.x; e < TB * r; e += blockDim.x) {
        const int t = e / r, i = e - t * r;
        float v = 0.f;
        for (int s = 0; s < usplits; ++s) v += upart[((size_t)s * B + b0 + t) * r + i];
        us[e] = v;
    }
    __syncthreads();
    if (m >= 2 * W) return;
    float v[TB][16];
#pragma unroll
    for (int t = 0; t < TB; ++t)
#pragma unroll
        for (int k = 0; k < 16; ++k) v[t][k] = 0.f;
    for (int vi0 = 0; vi0 < nvec; vi0 += 32) {
        const int vi = vi0 + lane;
        const bool vok = vi < nvec;
        if (vi0 > 0) load(vi0, w);
        if (vok) {
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                float wf[8];
                h8_to_f8(w[k], wf);
#pragma unroll
                for (int t = 0; t < TB; ++t) {
                    const float4 ua = reinterpret_cast<const float4*>(us + t * r + vi * 8)[0];
                    const float4 ub = reinterpret_cast<const float4*>(us + t * r + vi * 8)[1];
                    float a = v[t][k];
                    a = fmaf(wf[0], ua.x, a);
                    a = fmaf(wf[1], ua.y, a);
                    a = fmaf(wf[2], ua.z, a);
                    a = fmaf(wf[3], ua.w, a);
                    a = fmaf(wf[4], ub.x, a);
                    a = fmaf(wf[5], ub.y, a);
                    a = fmaf(wf[6], ub.z, a);
                    a = fmaf(wf[7], ub.w, a);
                    v[t][k] = a;
                }
            }
        }
    }
    const int k = 16 * m + fold16_row(lane);
    const float bk = __half2float(bias[k < F ? k : 0]);
#pragma unroll
    for (int t = 0; t < TB; ++t) {
        const float tot = fold16(v[t], lane);
        const bool pred = (lane & 1) == 0 && k < F && tot + bk > tau;
        const unsigned bal = __ballot_sync(FULL, pred);
        if (lane == 0) {
            unsigned bits = 0;
#pragma unroll
            for (int L = 0; L < 32; L += 2) bits |= ((bal >> L) & 1u) << fold16_row(L);
            reinterpret_cast<uint16_t*>(mask + (size_t)(b0 + t) * W)[m] = (uint16_t)bits;
        }
    }
}

// ----------------------------------------------------------------- compaction

// One block of 1024 threads: each thread takes one mask word (OR over the
// batch), counts its bits, an exclusive block scan gives its output offset.
__global__ void __launch_bounds__(1024) k_compact(const uint32_t* __restrict__ mask, int B, int W,
                                                  int F, const int32_t* __restrict__ table,
                                                  int32_t* __restrict__ idx,
                                                  int32_t* __restrict__ orig,
                                                  int32_t* __restrict__ count) {
    pdl_entry();
    __shared__ int wsum[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int base = 0;
    for (int w0 = 0; w0 < W; w0 += 1024) {
        const int w = w0 + threadIdx.x;
        uint32_t bits = 0u;
        if (w < W) {
            // tokens' words requested 8 at a time (independent loads in flight)
#pragma unroll 8
            for (int b = 0; b < B; ++b) bits |= __ldg(mask + (size_t)b * W + w);
            if (w == W - 1 && (F & 31)) bits &= (1u << (F & 31)) - 1u;
        }
        const int c = __popc(bits);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(FULL, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int v = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(FULL, v, o);
                if (lane >= o) v += u;
            }
            wsum[lane] = v;  // inclusive prefix over warps
        }
        __syncthreads();
        int off = base + incl - c + (warp > 0 ? wsum[warp - 1] : 0);
        while (bits) {
            const int p = __ffs(bits) - 1;
            bits &= bits - 1u;
            const int k = w * 32 + p;
            idx[off] = k;
            if (orig) orig[off] = table[k];
            ++off;
        }
        base += wsum[31];
        __syncthreads();
    }
    if (threadIdx.x == 0) *count = base;
}

// ------------------------------------------------------------------------ FC1

// KIND 0: fp16 rows; 1: fp16 gate + up rows (gated); 2: INT4 group-32 rows;
// 3: fp16 rows as a plain projection (bias, no activation: the query, key and
// value rows of the head-sparse attention block).
// One warp per listed neuron (grid-stride), x for TB tokens staged in smem.
template <int TB, int KIND>
__global__ void __launch_bounds__(256) k_fc1(const __half* __restrict__ x, int B, int b0, int d,
                                             LayerPtrs w, ColdPtrs cold, const int32_t* __restrict__ idx,
                                             const int32_t* __restrict__ count,
                                             const uint32_t* __restrict__ mask, int W,
                                             float* __restrict__ h) {
    pdl_entry();
    const int n = *count;
    if (n == 0) return;  // nothing predicted active: skip the layer's FC1 entirely
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __half* xs = reinterpret_cast<__half*>(smem_raw);
    const int nv = d / 8;
    const uint4* xg = reinterpret_cast<const uint4*>(x + (size_t)b0 * d);
    for (int e = threadIdx.x; e < TB * nv; e += blockDim.x) reinterpret_cast<uint4*>(xs)[e] = xg[e];
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nw = (gridDim.x * blockDim.x) >> 5;
    for (int j = gw; j < n; j += nw) {
        const int k = idx[j];
        float acc[TB], accu[TB];
#pragma unroll
        for (int t = 0; t < TB; ++t) acc[t] = accu[t] = 0.f;
        if (KIND != 2) {
            // the row's words are requested U per lane at a time; products of
            // fp16 weights and fp16 x are exact in fp32
            // rows past the hot tier come from the second tier
            const bool hot = k < cold.n_hot;
            const size_t kr = hot ? (size_t)k : (size_t)(k - cold.n_hot);
            const __half* w1b = static_cast<const __half*>(hot ? w.w1 : cold.w1);
            const uint4* row = reinterpret_cast<const uint4*>(w1b + kr * d);
            const uint4* rowu = KIND == 1 ? reinterpret_cast<const uint4*>((hot ? w.wu : cold.wu) + kr * d) : nullptr;
            constexpr int U = (KIND == 1 || TB >= 4) ? 8 : 16;
            for (int cb = lane; cb < nv; cb += 32 * U) {
                uint4 wv[U], uv[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = cb + 32 * u;
                    wv[u] = c < nv ? ld_stream16(row + c) : make_uint4(0u, 0u, 0u, 0u);
                    if (KIND == 1) uv[u] = c < nv ? ld_stream16(rowu + c) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = cb + 32 * u;
                    if (c >= nv) break;
#pragma unroll
                    for (int t = 0; t < TB; ++t) {
                        const uint4 xw = reinterpret_cast<const uint4*>(xs + (size_t)t * d)[c];
                        acc[t] += dot8hh(wv[u], xw);
                        if (KIND == 1) accu[t] += dot8hh(uv[u], xw);
                    }
                }
            }
        } else {
            // groups of 32 codes (16 bytes) and their scales, U per lane at a
            // time; codes become exact fp16 integers, products exact in fp32
            const int ng = d / 32;
            const bool hot = k < cold.n_hot;
            const size_t kr = hot ? (size_t)k : (size_t)(k - cold.n_hot);
            const uint4* row = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(hot ? w.w1 : cold.w1) +
                                                              kr * (d / 2));
            const __half* sc = (hot ? w.w1s : cold.w1s) + kr * ng;
            constexpr int U = 8;
            for (int gb = lane; gb < ng; gb += 32 * U) {
                uint4 qv[U];
                float sv[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int g = gb + 32 * u;
                    qv[u] = g < ng ? ld_stream16(row + g) : make_uint4(0u, 0u, 0u, 0u);
                    sv[u] = g < ng ? __half2float(sc[g]) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int g = gb + 32 * u;
                    if (g >= ng) break;
                    const uint32_t qw[4] = {qv[u].x, qv[u].y, qv[u].z, qv[u].w};
                    float part[TB];
#pragma unroll
                    for (int t = 0; t < TB; ++t) part[t] = 0.f;
#pragma unroll
                    for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
                        for (int t = 0; t < TB; ++t)
                            part[t] += dotq8h(qw[wi], *reinterpret_cast<const uint4*>(xs + (size_t)t * d + g * 32 + wi * 8));
                    }
#pragma unroll
                    for (int t = 0; t < TB; ++t) acc[t] = fmaf(sv[u], part[t], acc[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < TB; ++t) {
            acc[t] = warp_sum(acc[t]);
            if (KIND == 1) accu[t] = warp_sum(accu[t]);
        }
        const float bk = __half2float(w.b1[k]);
#pragma unroll
        for (int t = 0; t < TB; ++t) {
            if (lane == t) {
                const float z = acc[t] + bk;
                float hv = KIND == 3 ? z : (z > 0.f ? z : 0.f);
                if (KIND == 1) hv *= accu[t];
                if (mask != nullptr && B > 1 && !((mask[(size_t)(b0 + t) * W + (k >> 5)] >> (k & 31)) & 1u))
                    hv = 0.f;
                h[(size_t)j * B + b0 + t] = hv;
            }
        }
    }
}

// ------------------------------------------------------------------------ FC2

// part[s][b][c] = sum over listed neurons j of split s of h[j][b] * W2t[idx_j][c].
// Block (column tile, split); each thread owns CPT consecutive columns.  Rows
// whose h is zero for every token of the block are not read: ReLU already
// removed those neurons from FC2.
template <int TB, bool INT4>
__global__ void __launch_bounds__(256) k_fc2_part(const float* __restrict__ h, int B, int b0,
                                                  const int32_t* __restrict__ idx,
                                                  const int32_t* __restrict__ count, int d,
                                                  const void* __restrict__ w2t,
                                                  const __half* __restrict__ w2ts, ColdPtrs cold,
                                                  float* __restrict__ part) {
    pdl_entry();
    constexpr int CPT = INT4 ? 16 : 8;
    constexpr int CH = 256;
    const int n = *count;
    const int S = gridDim.y, s = blockIdx.y;
    const int chunk = (n + S - 1) / S;
    const int j0 = min(n, s * chunk), j1 = min(n, j0 + chunk);
    const int c = (blockIdx.x * blockDim.x + threadIdx.x) * CPT;
    const bool active = c < d;
    __shared__ int sidx[CH];
    __shared__ float sh[CH * TB];
    float acc[TB][CPT];
#pragma unroll
    for (int t = 0; t < TB; ++t)
#pragma unroll
        for (int e = 0; e < CPT; ++e) acc[t][e] = 0.f;
    for (int base = j0; base < j1; base += CH) {
        const int cnt = min(CH, j1 - base);
        __syncthreads();
        for (int e = threadIdx.x; e < cnt; e += blockDim.x) {
            float any = 0.f;
            for (int t = 0; t < TB; ++t) {
                const float v = h[(size_t)(base + e) * B + b0 + t];
                sh[e * TB + t] = v;
                any = fmaxf(any, fabsf(v));
            }
            sidx[e] = any > 0.f ? idx[base + e] : -1;
        }
        __syncthreads();
        if (!active) continue;
        // rows in batches of U: the batch's loads are all requested before the
        // first is used; the products are added in row order as before
        constexpr int U = TB <= 2 ? 8 : 4;
        for (int t0 = 0; t0 < cnt; t0 += U) {
            int kk[U];
#pragma unroll
            for (int u = 0; u < U; ++u) kk[u] = t0 + u < cnt ? sidx[t0 + u] : -1;
            if (!INT4) {
                uint4 wv[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    // rows past the hot tier come from the second tier
                    const int k = kk[u];
                    const bool hot = k < cold.n_hot;
                    const size_t kr = hot ? (size_t)k : (size_t)(k - cold.n_hot);
                    wv[u] = k >= 0 ? ld_stream16(static_cast<const __half*>(hot ? w2t : cold.w2t) + kr * d + c)
                                   : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (kk[u] < 0) continue;
                    float wf[8];
                    h8_to_f8(wv[u], wf);
#pragma unroll
                    for (int tb = 0; tb < TB; ++tb) {
                        const float hv = sh[(t0 + u) * TB + tb];
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[tb][e] = fmaf(hv, wf[e], acc[tb][e]);
                    }
                }
            } else {
                uint2 qv[U];
                float sv[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int k = kk[u];
                    const bool hot = k < cold.n_hot;
                    const size_t kr = hot ? (size_t)k : (size_t)(k - cold.n_hot);
                    qv[u] = k >= 0 ? ld_stream8(static_cast<const uint8_t*>(hot ? w2t : cold.w2t) + kr * (d / 2) + c / 2)
                                   : make_uint2(0u, 0u);
                    sv[u] = k >= 0 ? __half2float((hot ? w2ts : cold.w2ts)[kr * (d / 32) + c / 32]) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (kk[u] < 0) continue;
                    float qa[8], qb[8];
                    q8_to_f8(qv[u].x, qa);
                    q8_to_f8(qv[u].y, qb);
#pragma unroll
                    for (int tb = 0; tb < TB; ++tb) {
                        const float hv = sh[(t0 + u) * TB + tb] * sv[u];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            acc[tb][e] = fmaf(hv, qa[e], acc[tb][e]);
                            acc[tb][8 + e] = fmaf(hv, qb[e], acc[tb][8 + e]);
                        }
                    }
                }
            }
        }
    }
    if (!active) return;
#pragma unroll
    for (int tb = 0; tb < TB; ++tb) {
        float4* dst = reinterpret_cast<float4*>(part + ((size_t)s * B + b0 + tb) * d + c);
#pragma unroll
        for (int e = 0; e < CPT / 4; ++e)
            dst[e] = make_float4(acc[tb][4 * e], acc[tb][4 * e + 1], acc[tb][4 * e + 2], acc[tb][4 * e + 3]);
    }
}

// y[b][c] = b2[c] + sum_{s = 0..S-1} part[s][b][c], in a fixed order: a block
// takes 32 consecutive float4 of y (lanes), its warps the splits s = w, w + 8,
// ... (a warp's loads of one split are 512 contiguous bytes) with all of a
// lane's loads of a round in flight; the 8 warp sums are added in warp order.
__global__ void __launch_bounds__(256) k_fc2_reduce(const float* __restrict__ part, int S, int B,
                                                    int d, const __half* __restrict__ b2,
                                                    float* __restrict__ y) {
    pdl_entry();
    __shared__ float4 red[8][32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total4 = B * d / 4;
    const int e4 = blockIdx.x * 32 + lane;
    const bool ok = e4 < total4;
    const float4* p = reinterpret_cast<const float4*>(part) + (ok ? e4 : 0);
    const size_t stride = (size_t)total4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    constexpr int QB = 10;
    for (int s0 = warp; s0 < S; s0 += 8 * QB) {
        float4 v[QB];
#pragma unroll
        for (int b = 0; b < QB; ++b) {
            const int sp = s0 + 8 * b;
            if (ok && sp < S) v[b] = p[(size_t)sp * stride];
        }
#pragma unroll
        for (int b = 0; b < QB; ++b) {
            const int sp = s0 + 8 * b;
            if (ok && sp < S) {
                acc.x += v[b].x;
                acc.y += v[b].y;
                acc.z += v[b].z;
                acc.w += v[b].w;
            }
        }
    }
    red[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && ok) {
        const int c = (e4 * 4) % d;
        float4 t = red[0][lane];
        for (int w = 1; w < 8; ++w) {
            t.x += red[w][lane].x;
            t.y += red[w][lane].y;
            t.z += red[w][lane].z;
            t.w += red[w][lane].w;
        }
        t.x += __half2float(b2[c]);
        t.y += __half2float(b2[c + 1]);
        t.z += __half2float(b2[c + 2]);
        t.w += __half2float(b2[c + 3]);
        reinterpret_cast<float4*>(y)[e4] = t;
    }
}

// -------------------------------------------------------------- normalisation

// x_b = fp16(y_b / sqrt(mean(y_b^2) + eps)): one block of 1024 threads per
// token; each thread keeps its float4 words of y in registers between the
// sum of squares and the scaling (d % 4 == 0), the block sum in a fixed order.
constexpr int kNormThreads = 1024;
constexpr int kNormWords = 4;   // float4 words per thread held in registers (d <= 16384)
__global__ void __launch_bounds__(kNormThreads) k_rmsnorm(const float* __restrict__ y, int d, float eps,
                                                          __half* __restrict__ x) {
    pdl_entry();
    __shared__ float red[32];
    const float4* yb = reinterpret_cast<const float4*>(y + (size_t)blockIdx.x * d);
    const int n4 = d / 4;
    float4 v[kNormWords];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < kNormWords; ++k) {
        const int i4 = threadIdx.x + k * kNormThreads;
        v[k] = i4 < n4 ? __ldg(yb + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < kNormWords; ++k) ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
    for (int i4 = threadIdx.x + kNormWords * kNormThreads; i4 < n4; i4 += kNormThreads) {
        const float4 t = __ldg(yb + i4);
        ss += t.x * t.x + t.y * t.y + t.z * t.z + t.w * t.w;
    }
    ss = warp_sum(ss);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (warp == 0) {
        float t = red[lane];
        t = warp_sum(t);
        if (lane == 0) red[0] = t;
    }
    __syncthreads();
    const float scale = rsqrtf(red[0] / (float)d + eps);
    __half2* xb = reinterpret_cast<__half2*>(x + (size_t)blockIdx.x * d);
    auto put = [&](int i4, const float4& t) {
        xb[2 * i4] = __halves2half2(__float2half_rn(t.x * scale), __float2half_rn(t.y * scale));
        xb[2 * i4 + 1] = __halves2half2(__float2half_rn(t.z * scale), __float2half_rn(t.w * scale));
    };
#pragma unroll
    for (int k = 0; k < kNormWords; ++k) {
        const int i4 = threadIdx.x + k * kNormThreads;
        if (i4 < n4) put(i4, v[k]);
    }
    for (int i4 = threadIdx.x + kNormWords * kNormThreads; i4 < n4; i4 += kNormThreads) put(i4, __ldg(yb + i4));
}

// out[0] = n, out[1] = number of listed neurons with a non-zero h for some token
__global__ void __launch_bounds__(256) k_count_active(const int32_t* __restrict__ count, const float* __restrict__ h,
                                                      int B, int32_t* __restrict__ out) {
    pdl_entry();
    const int n = *count;
    int nz = 0;
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
        bool any = false;
        for (int b = 0; b < B; ++b) any |= h[(size_t)j * B + b] != 0.f;
        nz += any ? 1 : 0;
    }
    for (int o = 16; o > 0; o >>= 1) nz += __shfl_xor_sync(FULL, nz, o);
    __shared__ int red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = nz;
    __syncthreads();
    if (threadIdx.x == 0) {
        int t = 0;
        for (int w = 0; w < 8; ++w) t += red[w];
        out[0] = n;
        out[1] = t;
    }
}

// ------------------------------------------------------------------ launchers

namespace {

template <typename F>
cudaError_t for_token_chunks(int B, F&& f) {
    for (int b0 = 0; b0 < B;) {
        const int left = B - b0;
        const int tb = left >= 8 ? 8 : left >= 4 ? 4 : left >= 2 ? 2 : 1;
        cudaError_t e = f(b0, tb);
        if (e != cudaSuccess) return e;
        b0 += tb;
    }
    return cudaSuccess;
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t launch_predict(const Plan& p, const __half* x, const __half* p1, const __half* p2,
                           const __half* bpred, float tau, uint32_t* mask, void* ws, cudaStream_t s) {
    if (p.pred == 2 && p.r % 16 == 0)
        return launch_predict_tc(p, x, p1, p2, bpred, tau, mask,
                                 reinterpret_cast<float*>(static_cast<char*>(ws) + p.off_part),
                                 reinterpret_cast<__half*>(static_cast<char*>(ws) + p.off_uhl), s);
    if (p.pred_units()) {
        // the whole batch in one chunk: P2 is read once for every token
        float* upart = reinterpret_cast<float*>(static_cast<char*>(ws) + p.off_upart);
        const dim3 gu((p.r + 7) / 8, p.u_splits);
        const int tb = p.B, b0 = 0;
        cudaError_t e = cudaSuccess;
        const size_t sm1 = (size_t)tb * p.r * sizeof(float);
        const dim3 gs((2 * p.W + 7) / 8);
#define PI_PRED1(TBV)                                                                                        \
    if (tb == TBV) {                                                                                          \
        launch_pdl(k_predict_u<TBV>, gu, 256, 0, s, x, p.B, b0, p1, p.d, p.r, p.u_seg, upart);                 \
        e = set_smem(k_predict_s1<TBV>, sm1);                                                                 \
        if (e != cudaSuccess) return e;                                                                       \
        e = launch_pdl(k_predict_s1<TBV>, gs, 256, sm1, s, p2, bpred, static_cast<const float*>(upart),      \
                       p.u_splits, p.B, b0, p.r, p.F, p.W, tau, mask);                                        \
    }
        PI_PRED1(1) PI_PRED1(2) PI_PRED1(3) PI_PRED1(4)
#undef PI_PRED1
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    if (p.pred == 1)
        return launch_predict_st(p, x, p1, p2, bpred, tau, mask,
                                 reinterpret_cast<float*>(static_cast<char*>(ws) + p.off_part),
                                 reinterpret_cast<float*>(static_cast<char*>(ws) + p.off_uhl), s);
    float* upart = reinterpret_cast<float*>(static_cast<char*>(ws) + p.off_upart);
    return for_token_chunks(p.B, [&](int b0, int tb) -> cudaError_t {
        dim3 gu((p.r + 7) / 8, p.u_splits);
        const int ws = (p.W + 3) / 4;
        const size_t sm = (size_t)tb * p.r * sizeof(float);
#define PI_PRED(TBV)                                                                               \
    case TBV: {                                                                                    \
        launch_pdl(k_predict_u<TBV>, gu, 256, 0, s, x, p.B, b0, p1, p.d, p.r, p.u_seg, upart);             \
        cudaError_t e = set_smem(k_predict_s<TBV>, sm);                                            \
        if (e != cudaSuccess) return e;                                                            \
        launch_pdl(k_predict_s<TBV>, ws, 128, sm, s, p2, bpred, upart, p.u_splits, p.B, b0, p.r, p.F, p.W, \
                                             tau, mask);                                           \
        break;                                                                                     \
    }
        switch (tb) {
            PI_PRED(1)
            PI_PRED(2)
            PI_PRED(4)
            PI_PRED(8)
        }
#undef PI_PRED
        return cudaGetLastError();
    });
}

cudaError_t launch_compact(const Plan& p, const uint32_t* mask, const int32_t* table, int32_t* idx,
                           int32_t* orig, int32_t* count, cudaStream_t s) {
    launch_pdl(k_compact, 1, 1024, 0, s, mask, p.B, p.W, p.F, table, idx, orig, count);
    return cudaGetLastError();
}

cudaError_t launch_fc1_chunked(const Plan& p, const __half* x, const LayerPtrs& w, const ColdPtrs& cold,
                               const int32_t* idx, const int32_t* count, const uint32_t* mask, float* h,
                               cudaStream_t s) {
    const int kind = p.proj ? 3 : p.int4 ? 2 : (p.gated ? 1 : 0);
    return for_token_chunks(p.B, [&](int b0, int tb) -> cudaError_t {
        const size_t sm = (size_t)tb * p.d * sizeof(__half);
        const int blocks_max = (p.F + 7) / 8;
        int grid = p.nsm * 4;
        if (grid > blocks_max) grid = blocks_max;
        cudaError_t e = cudaSuccess;
#define PI_FC1(TBV, KV)                                                                       \
    if (tb == TBV && kind == KV) {                                                            \
        e = set_smem(k_fc1<TBV, KV>, sm);                                                     \
        if (e != cudaSuccess) return e;                                                       \
        launch_pdl(k_fc1<TBV, KV>, grid, 256, sm, s, x, p.B, b0, p.d, w, cold, idx, count, mask, p.W, h); \
    }
        PI_FC1(1, 0) PI_FC1(2, 0) PI_FC1(4, 0) PI_FC1(8, 0)
        PI_FC1(1, 1) PI_FC1(2, 1) PI_FC1(4, 1) PI_FC1(8, 1)
        PI_FC1(1, 2) PI_FC1(2, 2) PI_FC1(4, 2) PI_FC1(8, 2)
        PI_FC1(1, 3) PI_FC1(2, 3) PI_FC1(4, 3) PI_FC1(8, 3)
#undef PI_FC1
        return cudaGetLastError();
    });
}

cudaError_t launch_fc1(const Plan& p, const __half* x, const LayerPtrs& w, const int32_t* idx,
                       const int32_t* count, const uint32_t* mask, float* partial, float* h, int32_t* live,
                       cudaStream_t s) {
    if (p.tc) return launch_fc1_tc(p, x, w, idx, count, mask, partial, h, live, s);
    if (p.st) return launch_fc1_st(p, x, w, idx, count, mask, partial, h, live, s);
    if (p.fc1_tc4) return launch_fc1_tc4(p, x, w, idx, count, mask, partial, h, live, s);
    if (p.st4) return launch_fc1_st4(p, x, w, idx, count, mask, partial, h, live, s);
    return launch_fc1_chunked(p, x, w, no_cold_tier(), idx, count, mask, h, s);
}

cudaError_t launch_fc2_chunked(const Plan& p, const float* h, const int32_t* idx, const int32_t* count,
                               const LayerPtrs& w, const ColdPtrs& cold, float* partial, float* y, cudaStream_t s) {
    cudaError_t e = for_token_chunks(p.B, [&](int b0, int tb) -> cudaError_t {
        dim3 grid(p.fc2_tiles, p.fc2_splits);
#define PI_FC2(TBV, IV)                                                                       \
    if (tb == TBV && p.int4 == IV)                                                            \
        launch_pdl(k_fc2_part<TBV, IV>, grid, 256, 0, s, h, p.B, b0, idx, count, p.d, w.w2t, w.w2ts, \
                   cold, partial);
        PI_FC2(1, false) PI_FC2(2, false) PI_FC2(4, false) PI_FC2(8, false)
        PI_FC2(1, true) PI_FC2(2, true) PI_FC2(4, true) PI_FC2(8, true)
#undef PI_FC2
        return cudaGetLastError();
    });
    if (e != cudaSuccess) return e;
    const int total4 = p.B * p.d / 4;
    launch_pdl(k_fc2_reduce, (total4 + 31) / 32, 256, 0, s, partial, p.fc2_splits, p.B, p.d, w.b2, y);
    return cudaGetLastError();
}

cudaError_t launch_fc2(const Plan& p, const float* h, const int32_t* idx, const int32_t* count,
                       const LayerPtrs& w, const int32_t* live, float* partial, float* y, cudaStream_t s) {
    if (p.tc) return launch_fc2_tc(p, h, idx, count, w, live, partial, y, s);
    if (p.st) return launch_fc2_st(p, h, idx, count, w, live, partial, y, s);
    if (p.fc1_tc4) return launch_fc2_tc4(p, h, idx, count, w, live, partial, y, s);
    if (p.st4) return launch_fc2_st4(p, h, idx, count, w, live, partial, y, s);
    return launch_fc2_chunked(p, h, idx, count, w, no_cold_tier(), partial, y, s);
}

size_t fc2_part_floats(const Plan& p) {
    if (p.tc) return tc_fc2_part_floats(p);
    if (p.st) return st_fc2_part_floats(p);
    if (p.fc1_tc4) return tc_fc2_part_floats(p);
    if (p.st4) return st4_fc2_part_floats(p);
    return (size_t)p.fc2_splits * p.B * p.d;
}

cudaError_t launch_count_active(const Plan& p, const int32_t* count, const float* h, int32_t* out, cudaStream_t s) {
    launch_pdl(k_count_active, 1, 256, 0, s, count, h, p.B, out);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm(int d, int B, const float* y, float eps, __half* x, cudaStream_t s) {
    launch_pdl(k_rmsnorm, B, kNormThreads, 0, s, y, d, eps, x);
    return cudaGetLastError();
}

}  // namespace pi
