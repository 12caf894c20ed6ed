// pi_stream.cu -- the batched union path on CUDA cores (batch 2..8, fp16
// weights).
//
// Same work as the tensor-core path (PowerInfer summary (CSDN), section
// "Neuron-aware operator": only the rows of active neurons are processed; here
// the union's rows of W1 and W2t are read once for all tokens), with the same streamed structure: one CTA per SM,
// 4 loader warps fill a ring of stages with cp.async (paired K-chunks: 256
// contiguous bytes of a row per visit), the (tile x K-chunk) or (column tile x
// row) space is split evenly over the CTAs ("stream-K"), and fixed-order finish
// kernels add the per-CTA partial tiles.  At 2..8 tokens a weight element
// feeds at most 8 fused multiply-adds, which the SMs' CUDA cores sustain at
// HBM rate, so 8 compute warps do the products instead of tcgen05:
//   row GEMMs (FC1, gated FC1, predictor u and s): lane (rg, c) of compute
//     warp w owns rows 4w + rg + 32i (i < 4) and 16-byte chunk c of each
//     K-chunk; x is converted once per chunk and used for 4 rows, partial sums
//     are combined over the 8 chunk lanes by shuffles;
//   FC2: lane (mc, rg) owns 8 columns (chunk mc) and rows rg + 16i of each
//     64-row stage; partial sums are combined over the 16 row-group lanes.
// Shared rows use pitches of an odd number of 16-byte units, so the 8 lanes
// of a shared-memory phase always touch 8 different bank groups.  Every wait
// is bounded (status word; own copies drained before the CTA leaves).
#include <cuda_runtime.h>

#include "pi_common.cuh"
#include "pi_internal.h"
#include "pi_pipe.cuh"

namespace pi {
namespace {

using namespace pipe;

constexpr int kSThreads = 384;   // warps 0-3 load, 4-11 compute
constexpr int kSLoaders = 128;
constexpr int kSCompute = 8;     // compute warps
constexpr int kSBudget = 210 * 1024;
constexpr int kPitch = 144;      // shared bytes of one row's 64 fp16 (128 + 16)
constexpr int kTileS = 128 * kPitch;

// ------------------------------------------------------------------ row GEMMs
//   MODE 0  FC1            A = W1 rows (gathered),        Bop = x (fp16)
//   MODE 1  FC1 gated      A = Wg and Wu rows (gathered), Bop = x (fp16)
//   MODE 2  predictor u    A = P1 rows,                   Bop = x (fp16)
//   MODE 3  predictor s    A = P2 rows,                   Bop = u (fp32); whole
//           tiles per CTA, mask bits set with atomicOr (the caller zeroes them)
template <int MODE, int TB>
struct SCfg {
    static constexpr bool GATHER = MODE <= 1;
    static constexpr bool DIRECT = MODE == 3;
    static constexpr int NA = MODE == 1 ? 2 : 1;
    static constexpr int XE = DIRECT ? 4 : 2;          // bytes per B-operand element
    static constexpr int XROW = 64 * XE;               // one token's K-chunk
    static constexpr int STAGE = NA * kTileS + TB * XROW;
    static constexpr int S0 = kSBudget / STAGE > 12 ? 12 : kSBudget / STAGE;
    static constexpr int S = S0 & ~1;
    static constexpr int LAGP = S / 2 >= 4 ? S / 2 - 2 : S / 2 - 1;
    static constexpr int COLS = NA * TB;
    static constexpr size_t SMEM = (size_t)S * STAGE + 16;
};

struct SArgs {
    const __half* a0;      // A rows (row length K)
    const __half* a1;      // up-projection rows (gated FC1)
    const int32_t* idx;    // gathered row ids (FC1)
    const int32_t* count;  // device row count (FC1), else R rows
    int R;
    const void* bop;       // B operand rows [B][K] (fp16 x, or fp32 u)
    int K, B;
    float* part;           // modes 0-2: [G][slots][COLS][128]
    int slots;
    const __half* bias;    // mode 3
    float tau;
    uint32_t* mask;        // mode 3: [B][W], zero on entry
    int W;
    int* status;
    long long timeout_ns;
};

template <int MODE, int TB>
__global__ void __launch_bounds__(kSThreads, 1) k_rows_st(SArgs a) {
    pdl_entry();
    using C = SCfg<MODE, TB>;
    extern __shared__ __align__(16) unsigned char ring[];
    __shared__ __align__(8) unsigned long long full[C::S], empty[C::S];
    __shared__ int abort_flag;
    __shared__ int srow[128];

    const int R = a.count != nullptr ? *a.count : a.R;
    const int G = gridDim.x, g = blockIdx.x;
    const int ntile = (R + 127) / 128;
    const int nk = (a.K + 63) / 64;
    const long long U = (long long)ntile * nk;
    const long long u0 = U * g / G, u1 = U * (g + 1) / G;
    int npiece;
    if (C::DIRECT)
        npiece = ntile > g ? (ntile - 1 - g) / G + 1 : 0;
    else
        npiece = u0 < u1 ? (int)((u1 - 1) / nk - u0 / nk) + 1 : 0;
    if (npiece == 0) return;
    auto span = [&](int p) {
        Span sp;
        if (C::DIRECT) {
            sp.tile = g + p * G;
            sp.kc0 = 0;
            sp.kc1 = nk;
        } else {
            sp.tile = (int)(u0 / nk) + p;
            const long long lo = (long long)sp.tile * nk;
            sp.kc0 = (int)((u0 > lo ? u0 : lo) - lo);
            sp.kc1 = (int)((u1 < lo + nk ? u1 : lo + nk) - lo);
        }
        return sp;
    };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp == 4) {
        if (lane == 0) {
            for (int s = 0; s < C::S; ++s) {
                bar_init(&full[s], kSLoaders / 32);
                bar_init(&empty[s], kSCompute);
            }
            abort_flag = 0;
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
    } else if (warp < 4) {
        const Span s0 = span(0);
        const int rows = R - 128 * s0.tile < 128 ? R - 128 * s0.tile : 128;
        srow[tid] = tid < rows ? (C::GATHER ? a.idx[128 * s0.tile + tid] : 128 * s0.tile + tid) : -1;
    }
    __syncthreads();
    const Ctl ctl{a.status, a.timeout_ns, &abort_flag};

    if (warp < 4) {
        // ---- loaders (as in the tensor-core row kernel; rows at kPitch)
        const int t = tid, w = t >> 5, l = t & 31;
        int total = 0;
        for (int p = 0; p < npiece; ++p) {
            const Span sp = span(p);
            total += sp.kc1 - sp.kc0;
        }
        int pc = 0;
        Span sp = span(0);
        int ks = sp.kc0;
        long long pr[16], sr[8];
        auto take_rows = [&]() {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int rid = srow[2 * (4 * i + w) + (l >> 4)];
                pr[i] = rid >= 0 ? (long long)rid * a.K : -1;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int rid = srow[4 * (4 * i + w) + (l >> 3)];
                sr[i] = rid >= 0 ? (long long)rid * a.K : -1;
            }
        };
        auto load_rows = [&]() {
            loaders_sync_any(false);
            const int rows = R - 128 * sp.tile < 128 ? R - 128 * sp.tile : 128;
            srow[t] = t < rows ? (C::GATHER ? a.idx[128 * sp.tile + t] : 128 * sp.tile + t) : -1;
            loaders_sync_any(false);
            take_rows();
        };
        auto next_piece = [&]() {
            if (ks == sp.kc1 && pc + 1 < npiece) {
                ++pc;
                sp = span(pc);
                ks = sp.kc0;
                load_rows();
            }
        };
        auto copy_a = [&](unsigned char* st, int row, long long base, int kchunk, int c) {
            if (base < 0) return;
            const unsigned off = row * kPitch + c * 16;
            const long long gofs = base + kchunk * 64 + c * 8;
            cp16(st + off, a.a0 + gofs);
            if (MODE == 1) cp16(st + kTileS + off, a.a1 + gofs);
        };
        auto copy_b = [&](unsigned char* st, int kchunk) {
            const int k0 = kchunk * 64;
            const int kvalid = a.K - k0 < 64 ? a.K - k0 : 64;
            constexpr int CPR = C::XROW / 16;   // 16-byte chunks per token row
            for (int pp = t; pp < a.B * CPR; pp += kSLoaders) {
                const int tok = pp / CPR, kx = pp % CPR;
                if (kx * (16 / C::XE) < kvalid)
                    cp16(st + C::NA * kTileS + tok * C::XROW + kx * 16,
                         static_cast<const unsigned char*>(a.bop) + ((size_t)tok * a.K + k0) * C::XE + kx * 16);
            }
        };
        take_rows();
        const int npairs = (total + 1) / 2;
        bool ok = true;
        for (int it = 0; it < total; it += 2) {
            const int ng = total - it < 2 ? total - it : 2;
            bool good = true;
            for (int u = 0; u < ng; ++u) {
                const int st = it + u;
                if (good && st >= C::S && !bar_wait(&empty[st % C::S], ((st / C::S) - 1) & 1, ctl)) good = false;
            }
            if (loaders_sync_any(!good)) {
                ok = false;
                break;
            }
            unsigned char* s0 = ring + (size_t)(it % C::S) * C::STAGE;
            unsigned char* s1 = ring + (size_t)((it + 1) % C::S) * C::STAGE;
            if (ng == 2 && ks + 1 < sp.kc1) {
                const int u = (l >> 3) & 1, c = l & 7;
                if (c * 8 < a.K - (ks + u) * 64) {
                    unsigned char* sd = u ? s1 : s0;
#pragma unroll
                    for (int i = 0; i < 16; ++i) copy_a(sd, 2 * (4 * i + w) + (l >> 4), pr[i], ks + u, c);
                }
                copy_b(s0, ks);
                copy_b(s1, ks + 1);
                ks += 2;
                next_piece();
            } else {
                for (int u = 0; u < ng; ++u) {
                    unsigned char* st = u == 0 ? s0 : s1;
                    if ((l & 7) * 8 < a.K - ks * 64) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) copy_a(st, 4 * (4 * i + w) + (l >> 3), sr[i], ks, l & 7);
                    }
                    copy_b(st, ks);
                    ++ks;
                    next_piece();
                }
            }
            cp_commit();
            const int pd = it / 2 - C::LAGP;
            if (pd >= 0) {
                cp_wait<C::LAGP>();
                warp_arrive(&full[(2 * pd) % C::S]);
                if (2 * pd + 1 < total) warp_arrive(&full[(2 * pd + 1) % C::S]);
            }
        }
        if (ok) {
            const int first = npairs - C::LAGP < 0 ? 0 : npairs - C::LAGP;
            for (int pd = first; pd < npairs; ++pd) {
                const int newer = npairs - 1 - pd;
                if (newer >= 3)
                    cp_wait<3>();
                else if (newer == 2)
                    cp_wait<2>();
                else if (newer == 1)
                    cp_wait<1>();
                else
                    cp_wait<0>();
                warp_arrive(&full[(2 * pd) % C::S]);
                if (2 * pd + 1 < total) warp_arrive(&full[(2 * pd + 1) % C::S]);
            }
        }
        cp_wait_all();
    } else {
        // ---- compute warps
        const int cw = warp - 4, rg = lane >> 3, c = lane & 7;
        float acc[C::NA][4][TB];
#pragma unroll
        for (int q = 0; q < C::NA; ++q)
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int t = 0; t < TB; ++t) acc[q][i][t] = 0.f;
        int it = 0;
        for (int p = 0; p < npiece; ++p) {
            const Span sp = span(p);
            bool ok = true;
            for (int ks = sp.kc0; ks < sp.kc1; ++ks, ++it) {
                const int s = it % C::S;
                if (!bar_wait(&full[s], (it / C::S) & 1, ctl)) {
                    ok = false;
                    break;
                }
                const unsigned char* st = ring + (size_t)s * C::STAGE;
                if (c * 8 < a.K - ks * 64) {
                    float wv[C::NA][4][8];
#pragma unroll
                    for (int q = 0; q < C::NA; ++q)
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            h8_to_f8(*reinterpret_cast<const uint4*>(st + q * kTileS +
                                                                     (4 * cw + rg + 32 * i) * kPitch + c * 16),
                                     wv[q][i]);
                    const unsigned char* xs = st + C::NA * kTileS + c * 8 * C::XE;
#pragma unroll
                    for (int t = 0; t < TB; ++t) {
                        if (t < a.B) {
                            float xv[8];
                            if (C::DIRECT) {
                                const float4 x0 = reinterpret_cast<const float4*>(xs + t * C::XROW)[0];
                                const float4 x1 = reinterpret_cast<const float4*>(xs + t * C::XROW)[1];
                                xv[0] = x0.x; xv[1] = x0.y; xv[2] = x0.z; xv[3] = x0.w;
                                xv[4] = x1.x; xv[5] = x1.y; xv[6] = x1.z; xv[7] = x1.w;
                            } else {
                                h8_to_f8(*reinterpret_cast<const uint4*>(xs + t * C::XROW), xv);
                            }
#pragma unroll
                            for (int q = 0; q < C::NA; ++q)
#pragma unroll
                                for (int i = 0; i < 4; ++i)
#pragma unroll
                                    for (int e = 0; e < 8; ++e) acc[q][i][t] = fmaf(wv[q][i][e], xv[e], acc[q][i][t]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) bar_arrive(&empty[s]);
            }
            if (!ok) break;
            // piece done: sum over the 8 chunk lanes (every lane gets the total)
#pragma unroll
            for (int q = 0; q < C::NA; ++q)
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int t = 0; t < TB; ++t) {
                        float v = acc[q][i][t];
                        v += __shfl_xor_sync(FULL, v, 1);
                        v += __shfl_xor_sync(FULL, v, 2);
                        v += __shfl_xor_sync(FULL, v, 4);
                        acc[q][i][t] = v;
                    }
            if (C::DIRECT) {
                // s = P2 u + b > tau: the chunk-0 lanes of the warp hold rows
                // 4cw + rg + 32i; one ballot per (i, token) gives their 4 bits
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int k = 128 * sp.tile + 4 * cw + rg + 32 * i;
                    const float bk = (c == 0 && k < R) ? __half2float(a.bias[k]) : 0.f;
                    const int word = 4 * sp.tile + i;
#pragma unroll
                    for (int t = 0; t < TB; ++t) {
                        const bool on = c == 0 && k < R && t < a.B && acc[0][i][t] + bk > a.tau;
                        const unsigned bal = __ballot_sync(FULL, on);
                        const unsigned bits4 = (bal & 1u) | ((bal >> 7) & 2u) | ((bal >> 14) & 4u) | ((bal >> 21) & 8u);
                        if (lane == 0 && bits4 != 0u && word < a.W)
                            atomicOr(a.mask + (size_t)t * a.W + word, bits4 << (4 * cw));
                    }
                }
            } else if (c == 0) {
                if (p < a.slots) {
                    float* dst = a.part + ((size_t)g * a.slots + p) * C::COLS * 128;
#pragma unroll
                    for (int q = 0; q < C::NA; ++q)
#pragma unroll
                        for (int i = 0; i < 4; ++i)
#pragma unroll
                            for (int t = 0; t < TB; ++t)
                                if (t < a.B) dst[(size_t)(q * TB + t) * 128 + 4 * cw + rg + 32 * i] = acc[q][i][t];
                } else if (rg == 0) {
                    atomicExch(a.status, (int)PI_ERR_WORKSPACE);
                }
            }
#pragma unroll
            for (int q = 0; q < C::NA; ++q)
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int t = 0; t < TB; ++t) acc[q][i][t] = 0.f;
        }
    }
}

// u[t][i] = sum of the P1 x partials in ascending CTA order, fp32 rows [B][r].
__global__ void __launch_bounds__(256) k_u_finish32(const float* __restrict__ part, int slots, int G, int nk, int r,
                                                    int B, int NT, float* __restrict__ u) {
    pdl_entry();
    __shared__ int slot[kMaxCtas];
    __shared__ int rng[2];
    const int i0 = blockIdx.x * 32;
    const int lane = threadIdx.x & 31, t = threadIdx.x >> 5;
    cover_setup((long long)((r + 127) / 128) * nk, G, nk, i0 >> 7, slot, rng);
    __syncthreads();
    const int i = i0 + lane;
    if (i >= r || t >= B) return;
    u[(size_t)t * r + i] = sum_cover(part, slot, rng, slots, NT, t, i & 127);
}

// ------------------------------------------------------------------------ FC2
// y[t, c] = sum_j W2t[idx_j, c] h[j, t]; stages of 64 gathered rows x 128
// columns (row pitch 272 bytes), h rows copied raw ([64][hp] fp32, hp odd).
constexpr int kPitch2 = 272;
constexpr int kTile2 = 64 * kPitch2;

template <int TB>
struct SCfg2 {
    static constexpr int HP = TB | 1;                   // padded h row (floats)
    static constexpr int RAW = 64 * HP * 4;
    static constexpr int IDX = 64 * 2 * 4;              // row ids + live flags
    static constexpr int STAGE = kTile2 + RAW;
    static constexpr int S = kSBudget / (STAGE + IDX) > 10 ? 10 : kSBudget / (STAGE + IDX);
    static constexpr int LAG = S - 2;
    static constexpr size_t SMEM = (size_t)S * (STAGE + IDX) + 16;
};

struct SArgs2 {
    const float* h;        // [count][B]
    const int32_t* idx;
    const int32_t* count;
    const __half* w2t;
    const int32_t* live;   // nullable
    float* part;           // [G][slots][TB][128]
    int* status;
    long long timeout_ns;
    int B, d, slots;
};

struct Piece2 {
    int ct, j0, j1;
};
constexpr int kMaxPieces2 = 16;
PI_DEV void piece2(long long u0, long long u1, int n, int which, Piece2* out) {
    const int ct = (int)(u0 / n) + which;
    const long long lo = (long long)ct * n, hi = lo + n;
    const long long a = u0 > lo ? u0 : lo, b = u1 < hi ? u1 : hi;
    out->ct = ct;
    out->j0 = (int)(a - lo);
    out->j1 = (int)(b - lo);
}

template <int TB>
__global__ void __launch_bounds__(kSThreads, 1) k_fc2_st(SArgs2 a) {
    pdl_entry();
    using C = SCfg2<TB>;
    extern __shared__ __align__(16) unsigned char ring[];
    __shared__ __align__(8) unsigned long long full[C::S], empty[C::S];
    __shared__ int abort_flag;

    const int n = *a.count;
    const int G = gridDim.x, g = blockIdx.x;
    const int nct = a.d / 128;
    const long long U = (long long)nct * n;
    const long long u0 = U * g / G, u1 = U * (g + 1) / G;
    if (u0 >= u1) return;
    const int npiece = (int)((u1 - 1) / n - u0 / n) + 1;
    // this CTA's pieces, computed once (64-bit divisions stay out of the loops)
    __shared__ Piece2 ptab[kMaxPieces2];
    if (npiece > kMaxPieces2) {
        if (threadIdx.x == 0) atomicExch(a.status, (int)PI_ERR_WORKSPACE);
        return;
    }
    if (threadIdx.x < npiece) piece2(u0, u1, n, threadIdx.x, &ptab[threadIdx.x]);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < C::S; ++s) {
            bar_init(&full[s], kSLoaders / 32);
            bar_init(&empty[s], kSCompute);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const Ctl ctl{a.status, a.timeout_ns, &abort_flag};
    int32_t* sidx = reinterpret_cast<int32_t*>(ring + (size_t)C::S * C::STAGE);
    int32_t* slive = sidx + C::S * 64;

    if (warp < 4) {
        // ---- loaders: per stage 64 W2t rows x 256 bytes (2 rows x 256 contiguous
        // bytes per warp instruction) and the h rows; row ids run a ring ahead
        const int t = tid, w = t >> 5, l = t & 31;
        int total = 0;
        for (int p = 0; p < npiece; ++p) {
            const Piece2 pc = ptab[p];
            total += (pc.j1 - pc.j0 + 63) / 64;
        }
        int fq = 0, fpiece = 0, fst = 0;
        auto copy_ids = [&]() {
            const Piece2 pc = ptab[fpiece];
            const int jb = pc.j0 + 64 * fst;
            const int kk = t & 63;
            const int j = jb + kk;
            if (j < pc.j1) {
                if (t < 64)
                    cp4(sidx + (fq % C::S) * 64 + kk, a.idx + j);
                else if (a.live != nullptr)
                    cp4(slive + (fq % C::S) * 64 + kk, a.live + j);
            }
            ++fq;
            if (64 * (++fst) >= pc.j1 - pc.j0) {
                ++fpiece;
                fst = 0;
            }
        };
        while (fq < total && fq <= C::LAG) copy_ids();
        cp_commit();
        cp_wait_all();
        loaders_sync_any(false);
        int it = 0;
        bool ok = true;
        for (int pi_ = 0; pi_ < npiece && ok; ++pi_) {
            const Piece2 pc = ptab[pi_];
            const int nst = (pc.j1 - pc.j0 + 63) / 64;
            const int col0 = pc.ct * 128;
            for (int st = 0; st < nst; ++st, ++it) {
                const int s = it % C::S;
                bool good = true;
                if (it >= C::S) good = bar_wait(&empty[s], ((it / C::S) - 1) & 1, ctl);
                unsigned char* sb = ring + (size_t)s * C::STAGE;
                const int jb = pc.j0 + 64 * st;
                const int nrow = pc.j1 - jb < 64 ? pc.j1 - jb : 64;
                if (good) {
                    // W2t rows: lane (row half r2 = l >> 4, chunk c16 = l & 15)
#pragma unroll 4
                    for (int i = 0; i < 8; ++i) {
                        const int kk = 2 * (4 * i + w) + (l >> 4), c16 = l & 15;
                        unsigned char* dst = sb + kk * kPitch2 + c16 * 16;
                        const bool in = kk < nrow;
                        const bool alive = a.live == nullptr || (in && slive[s * 64 + kk] != 0);
                        if (in && alive)
                            cp16(dst, a.w2t + (size_t)sidx[s * 64 + kk] * a.d + col0 + c16 * 8);
                        else
                            *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    // h rows into [64][HP]; rows past the piece are zero
                    float* raw = reinterpret_cast<float*>(sb + kTile2);
                    for (int e = t; e < 64 * a.B; e += kSLoaders) {
                        const int kk = e / a.B, tok = e - kk * a.B;
                        if (kk < nrow)
                            cp4(raw + kk * C::HP + tok, a.h + (size_t)(jb + kk) * a.B + tok);
                        else
                            raw[kk * C::HP + tok] = 0.f;
                    }
                    if (fq < total) copy_ids();
                }
                cp_commit();
                if (it >= C::LAG) cp_wait<C::LAG>();
                // every loader's copies of stage it - LAG (and the ids of stage
                // it + 1) have landed; stop together
                if (loaders_sync_any(!good || *(volatile int*)&abort_flag)) {
                    ok = false;
                    break;
                }
                if (it >= C::LAG) warp_arrive(&full[(it - C::LAG) % C::S]);
            }
        }
        cp_wait_all();
        if (!loaders_sync_any(!ok || *(volatile int*)&abort_flag)) {
            for (int q = it - C::LAG < 0 ? 0 : it - C::LAG; q < it; ++q) warp_arrive(&full[q % C::S]);
        }
    } else {
        // ---- compute warps: lane (mc = 2cw + (lane >> 4), rg = lane & 15)
        const int cw = warp - 4, mc = 2 * cw + (lane >> 4), rg = lane & 15;
        float acc[8][TB];
#pragma unroll
        for (int e = 0; e < 8; ++e)
#pragma unroll
            for (int t = 0; t < TB; ++t) acc[e][t] = 0.f;
        int it = 0;
        for (int p = 0; p < npiece; ++p) {
            const Piece2 pc = ptab[p];
            const int nst = (pc.j1 - pc.j0 + 63) / 64;
            bool ok = true;
            for (int st = 0; st < nst; ++st, ++it) {
                const int s = it % C::S;
                if (!bar_wait(&full[s], (it / C::S) & 1, ctl)) {
                    ok = false;
                    break;
                }
                const unsigned char* sb = ring + (size_t)s * C::STAGE;
                const float* raw = reinterpret_cast<const float*>(sb + kTile2);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int kk = rg + 16 * i;
                    float wf[8];
                    h8_to_f8(*reinterpret_cast<const uint4*>(sb + kk * kPitch2 + mc * 16), wf);
#pragma unroll
                    for (int t = 0; t < TB; ++t) {
                        if (t < a.B) {
                            const float hv = raw[kk * C::HP + t];
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc[e][t] = fmaf(hv, wf[e], acc[e][t]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) bar_arrive(&empty[s]);
            }
            if (!ok) break;
            // sum over the 16 row-group lanes of this column chunk
#pragma unroll
            for (int e = 0; e < 8; ++e)
#pragma unroll
                for (int t = 0; t < TB; ++t) {
                    float v = acc[e][t];
                    v += __shfl_xor_sync(FULL, v, 1);
                    v += __shfl_xor_sync(FULL, v, 2);
                    v += __shfl_xor_sync(FULL, v, 4);
                    v += __shfl_xor_sync(FULL, v, 8);
                    acc[e][t] = v;
                }
            if (rg == 0) {
                if (p < a.slots) {
                    float* dst = a.part + ((size_t)g * a.slots + p) * TB * 128 + mc * 8;
#pragma unroll
                    for (int t = 0; t < TB; ++t)
                        if (t < a.B) {
                            float4* o = reinterpret_cast<float4*>(dst + (size_t)t * 128);
                            o[0] = make_float4(acc[0][t], acc[1][t], acc[2][t], acc[3][t]);
                            o[1] = make_float4(acc[4][t], acc[5][t], acc[6][t], acc[7][t]);
                        }
                } else {
                    atomicExch(a.status, (int)PI_ERR_WORKSPACE);
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e)
#pragma unroll
                for (int t = 0; t < TB; ++t) acc[e][t] = 0.f;
        }
    }
}

template <typename K>
cudaError_t prep_st(K kernel, size_t smem) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

int cdiv(int a, int b) { return (a + b - 1) / b; }
int slots_of(int tiles, int G) { return cdiv(tiles, G) + 2; }
int u_grid_st(const Plan& p) {
    const int units = cdiv(p.r, 128) * cdiv(p.d, 64);
    const int G = p.nsm > 0 ? p.nsm : 1;
    return units / 8 < 1 ? 1 : (units / 8 < G ? units / 8 : G);
}

template <int MODE, int TB>
cudaError_t launch_rows(const SArgs& a, int grid, cudaStream_t s) {
    using C = SCfg<MODE, TB>;
    cudaError_t e = prep_st(k_rows_st<MODE, TB>, C::SMEM);
    if (e != cudaSuccess) return e;
    launch_pdl(k_rows_st<MODE, TB>, grid, kSThreads, C::SMEM, s, a);
    return cudaGetLastError();
}
template <int MODE>
cudaError_t launch_rows_tb(const SArgs& a, int tb, int grid, cudaStream_t s) {
    if (tb == 2) return launch_rows<MODE, 2>(a, grid, s);
    if (tb == 4) return launch_rows<MODE, 4>(a, grid, s);
    return launch_rows<MODE, 8>(a, grid, s);
}

}  // namespace

bool st_pred_supported(const Plan& p) { return p.B >= 2 && p.B <= 8 && p.d % 128 == 0 && p.nsm <= kMaxCtas; }

bool st_supported(const Plan& p) { return !p.int4 && st_pred_supported(p); }

int st_tokens(const Plan& p) { return p.B <= 2 ? 2 : (p.B <= 4 ? 4 : 8); }

size_t st_part_floats(const Plan& p) {
    const size_t G = p.nsm > 0 ? p.nsm : 1, tb = st_tokens(p);
    const size_t fc1 = G * slots_of(cdiv(p.F, 128), (int)G) * (p.gated ? 2 : 1) * tb * 128;
    const size_t fc2 = G * slots_of(p.d / 128, (int)G) * tb * 128;
    const size_t pu = (size_t)u_grid_st(p) * slots_of(cdiv(p.r, 128), u_grid_st(p)) * tb * 128;
    size_t m = fc1 > fc2 ? fc1 : fc2;
    return m > pu ? m : pu;
}

size_t st_fc2_part_floats(const Plan& p) {
    const size_t G = p.nsm > 0 ? p.nsm : 1;
    return G * slots_of(p.d / 128, (int)G) * st_tokens(p) * 128;
}

size_t st_u_bytes(const Plan& p) { return (size_t)p.B * p.r * sizeof(float); }

cudaError_t launch_predict_st(const Plan& p, const __half* x, const __half* p1, const __half* p2,
                              const __half* bpred, float tau, uint32_t* mask, float* part, float* u32,
                              cudaStream_t s) {
    int* status = status_word();
    if (status == nullptr) return cudaErrorInvalidDevice;
    const int tb = st_tokens(p), Gu = u_grid_st(p);
    SArgs a{};
    a.a0 = p1;
    a.R = p.r;
    a.bop = x;
    a.K = p.d;
    a.B = p.B;
    a.part = part;
    a.slots = slots_of(cdiv(p.r, 128), Gu);
    a.status = status;
    a.timeout_ns = wait_timeout_ns();
    cudaError_t e = launch_rows_tb<2>(a, tb, Gu, s);
    if (e != cudaSuccess) return e;
    launch_pdl(k_u_finish32, cdiv(p.r, 32), 256, 0, s, part, a.slots, Gu, cdiv(p.d, 64), p.r, p.B, tb, u32);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(mask, 0, sizeof(uint32_t) * (size_t)p.B * p.W, s);
    if (e != cudaSuccess) return e;
    SArgs b{};
    b.a0 = p2;
    b.R = p.F;
    b.bop = u32;
    b.K = p.r;
    b.B = p.B;
    b.bias = bpred;
    b.tau = tau;
    b.mask = mask;
    b.W = p.W;
    b.status = status;
    b.timeout_ns = wait_timeout_ns();
    return launch_rows_tb<3>(b, tb, p.nsm, s);
}

cudaError_t launch_fc1_st(const Plan& p, const __half* x, const LayerPtrs& w, const int32_t* idx,
                          const int32_t* count, const uint32_t* mask, float* part, float* h, int32_t* live,
                          cudaStream_t s) {
    int* status = status_word();
    if (status == nullptr) return cudaErrorInvalidDevice;
    const int tb = st_tokens(p), G = p.nsm;
    SArgs a{};
    a.a0 = static_cast<const __half*>(w.w1);
    a.a1 = w.wu;
    a.idx = idx;
    a.count = count;
    a.bop = x;
    a.K = p.d;
    a.B = p.B;
    a.part = part;
    a.slots = slots_of(cdiv(p.F, 128), G);
    a.status = status;
    a.timeout_ns = wait_timeout_ns();
    cudaError_t e = p.gated ? launch_rows_tb<1>(a, tb, G, s) : launch_rows_tb<0>(a, tb, G, s);
    if (e != cudaSuccess) return e;
    return launch_fc1_finish(p, tb, G, a.slots, cdiv(p.d, 64), part, count, idx, w.b1, mask, h, live, s);
}

cudaError_t launch_fc2_st(const Plan& p, const float* h, const int32_t* idx, const int32_t* count,
                          const LayerPtrs& w, const int32_t* live, float* partial, float* y, cudaStream_t s) {
    int* status = status_word();
    if (status == nullptr) return cudaErrorInvalidDevice;
    const int tb = st_tokens(p), G = p.nsm;
    const int slots = slots_of(p.d / 128, G);
    SArgs2 a{h, idx, count, static_cast<const __half*>(w.w2t), live, partial, status, wait_timeout_ns(), p.B, p.d, slots};
    cudaError_t e;
#define PI_FC2ST(TBV)                                                     \
    if (tb == TBV) {                                                      \
        e = prep_st(k_fc2_st<TBV>, SCfg2<TBV>::SMEM);                     \
        if (e != cudaSuccess) return e;                                   \
        launch_pdl(k_fc2_st<TBV>, G, kSThreads, SCfg2<TBV>::SMEM, s, a);           \
    }
    PI_FC2ST(2) else PI_FC2ST(4) else PI_FC2ST(8)
#undef PI_FC2ST
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_fc2_reduce(p, tb, G, slots, 128, p.B, 0, partial, count, w.b2, y, s);
}

}  // namespace pi
