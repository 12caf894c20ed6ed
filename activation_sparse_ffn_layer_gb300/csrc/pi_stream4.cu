// pi_stream4.cu -- the batched union path for INT4 group-32 weights on CUDA
// cores (batch 2..16, ReLU FFN).
//
// Same streamed structure as the fp16 batched kernels (loader warps filling a
// cp.async ring, stream-K split over the CTAs, fixed-order finish kernels),
// with the INT4 rows dequantised in registers (PowerInfer summary (CSDN),
// section "Introduction": 4-bit quantised models; the code q of an element is
// a signed 4-bit integer, its value q * s with one fp16 scale s per 32 consecutive
// elements of the row).  A stage holds 256 elements of each of 128 rows (FC1)
// or 256 columns of each of 64 rows (FC2): 128 bytes of codes followed by the
// 16 bytes of the 8 scales, a 144-byte pitch (9 x 16 bytes: the 8 lanes of a
// shared-memory phase touch 8 different bank groups).
//   FC1: lane (rg, c) of compute warp w owns rows 4w + rg + 32i (i < 4) and
//        scale group c of the stage; each group is done in two 16-element
//        halves (acc += s * sum q x), partial sums combined over the 8 group
//        lanes by shuffles.
//   FC2: lane (mc, rg) owns 8 columns (chunk mc of 32) and rows rg + 8i of the
//        64-row stage; partial sums combined over the 8 row-group lanes.
#include <cuda_runtime.h>

#include "pi_common.cuh"
#include "pi_internal.h"
#include "pi_pipe.cuh"

namespace pi {
namespace {

using namespace pipe;

constexpr int kQThreads = 384;   // warps 0-3 load, 4-11 compute
constexpr int kQLoaders = 128;
constexpr int kQCompute = 8;
constexpr int kQBudget = 210 * 1024;
constexpr int kQPitch = 144;     // 128 bytes of codes + 16 bytes of scales
constexpr int kQTile = 128 * kQPitch;
constexpr int kQTile2 = 64 * kQPitch;

// Barriers of the 256 compute threads (ids 0 and 1 are the CTA's and the
// loaders'): a plain one, and one that ORs a flag so all take the same branch
PI_DEV void compute_sync() { asm volatile("bar.sync 2, 256;" ::: "memory"); }
PI_DEV bool compute_sync_any(bool v) {
    unsigned r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, 2, 256, q;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(r)
        : "r"((unsigned)v)
        : "memory");
    return r != 0;
}

// 16 codes (low nibble first) of one 64-bit word -> exact floats
PI_DEV void q16_to_f16(uint2 w, float (&f)[16]) {
    float a[8], b[8];
    q8_to_f8(w.x, a);
    q8_to_f8(w.y, b);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        f[e] = a[e];
        f[8 + e] = b[e];
    }
}

// ------------------------------------------------------------------------ FC1

template <int TB>
struct Q1Cfg {
    // one token's 256 fp16 of x: 8 groups of 32 at an 80-byte pitch, so the 8 group lanes of a
    // shared-memory phase read 8 disjoint bank quads
    static constexpr int XROW = 8 * 80;
    static constexpr int STAGE = kQTile + TB * XROW;
    // the stage's x converted to fp32 once for all compute lanes: per token 8
    // groups of 32 floats at a 36-float pitch (8 group lanes hit 8 bank quads)
    // (for 8 tokens and more; with 4 the lanes convert their own x words)
    static constexpr bool PRE = TB >= 8;
    static constexpr int XF_GROUP = 36;
    static constexpr int XF_TOKEN = 8 * XF_GROUP;
    static constexpr int XF = PRE ? TB * XF_TOKEN * 4 : 0;
    static constexpr int S0 = (kQBudget - XF) / STAGE > 12 ? 12 : (kQBudget - XF) / STAGE;
    static constexpr int S = S0 & ~1;
    static constexpr int LAGP = S / 2 >= 4 ? S / 2 - 2 : S / 2 - 1;
    static constexpr size_t SMEM = (size_t)S * STAGE + XF + 16;
};

struct Q1Args {
    const uint8_t* codes;   // [F][d/2]
    const __half* scales;   // [F][d/32]
    const int32_t* idx;
    const int32_t* count;
    const __half* x;        // [B][d]
    int K, B;
    float* part;            // [G][slots][TB][128]
    int slots;
    int* status;
    long long timeout_ns;
};

template <int TB>
__global__ void __launch_bounds__(kQThreads, 1) k_fc1_st4(Q1Args a) {
    pdl_entry();
    using C = Q1Cfg<TB>;
    extern __shared__ __align__(16) unsigned char ring[];
    __shared__ __align__(8) unsigned long long full[C::S], empty[C::S];
    __shared__ int abort_flag;
    __shared__ int srow[128];

    const int R = *a.count;
    const int G = gridDim.x, g = blockIdx.x;
    const int ntile = (R + 127) / 128;
    const int nk = a.K / 256;
    const long long U = (long long)ntile * nk;
    const long long u0 = U * g / G, u1 = U * (g + 1) / G;
    const int npiece = u0 < u1 ? (int)((u1 - 1) / nk - u0 / nk) + 1 : 0;
    if (npiece == 0) return;
    auto span = [&](int p) {
        Span sp;
        sp.tile = (int)(u0 / nk) + p;
        const long long lo = (long long)sp.tile * nk;
        sp.kc0 = (int)((u0 > lo ? u0 : lo) - lo);
        sp.kc1 = (int)((u1 < lo + nk ? u1 : lo + nk) - lo);
        return sp;
    };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp == 4) {
        if (lane == 0) {
            for (int s = 0; s < C::S; ++s) {
                bar_init(&full[s], kQLoaders);
                bar_init(&empty[s], kQCompute);
            }
            abort_flag = 0;
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
    } else if (warp < 4) {
        const Span s0 = span(0);
        const int rows = R - 128 * s0.tile < 128 ? R - 128 * s0.tile : 128;
        srow[tid] = tid < rows ? a.idx[128 * s0.tile + tid] : -1;
    }
    __syncthreads();
    const Ctl ctl{a.status, a.timeout_ns, &abort_flag};
    const size_t cpr = (size_t)a.K / 2, spr = (size_t)a.K / 32;   // code bytes, scales per row
    float* xsf = reinterpret_cast<float*>(ring + (size_t)C::S * C::STAGE);   // [TB][XF_TOKEN] fp32 x

    if (warp < 4) {
        const int t = tid, w = t >> 5, l = t & 31;
        int total = 0;
        for (int p = 0; p < npiece; ++p) {
            const Span sp = span(p);
            total += sp.kc1 - sp.kc0;
        }
        int pc = 0;
        Span sp = span(0);
        int ks = sp.kc0;
        int pr[16], sr[8], own;
        auto take_rows = [&]() {
#pragma unroll
            for (int i = 0; i < 16; ++i) pr[i] = srow[2 * (4 * i + w) + (l >> 4)];
#pragma unroll
            for (int i = 0; i < 8; ++i) sr[i] = srow[4 * (4 * i + w) + (l >> 3)];
            own = srow[t];
        };
        auto load_rows = [&]() {
            loaders_sync_any(false);
            const int rows = R - 128 * sp.tile < 128 ? R - 128 * sp.tile : 128;
            srow[t] = t < rows ? a.idx[128 * sp.tile + t] : -1;
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
        // this thread's row's 8 scales of K-chunk kchunk, and x
        auto copy_scales_x = [&](unsigned char* st, int kchunk) {
            if (own >= 0) cp16(st + t * kQPitch + 128, a.scales + (size_t)own * spr + kchunk * 8);
            const int k0 = kchunk * 256;
            for (int pp = t; pp < a.B * 32; pp += kQLoaders) {
                const int tok = pp >> 5, kx = pp & 31;
                cp16(st + kQTile + tok * C::XROW + (kx >> 2) * 80 + (kx & 3) * 16,
                     a.x + (size_t)tok * a.K + k0 + kx * 8);
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
                // both K-chunks of a row back to back: 2 rows x 256 bytes of codes per instruction
                const int u = (l >> 3) & 1, c = l & 7;
                unsigned char* sd = u ? s1 : s0;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int row = 2 * (4 * i + w) + (l >> 4);
                    if (pr[i] >= 0)
                        cp16(sd + row * kQPitch + c * 16, a.codes + (size_t)pr[i] * cpr + (size_t)(ks + u) * 128 + c * 16);
                }
                copy_scales_x(s0, ks);
                copy_scales_x(s1, ks + 1);
                ks += 2;
                next_piece();
            } else {
                for (int u = 0; u < ng; ++u) {
                    unsigned char* st = u == 0 ? s0 : s1;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int row = 4 * (4 * i + w) + (l >> 3);
                        if (sr[i] >= 0)
                            cp16(st + row * kQPitch + (l & 7) * 16,
                                 a.codes + (size_t)sr[i] * cpr + (size_t)ks * 128 + (l & 7) * 16);
                    }
                    copy_scales_x(st, ks);
                    ++ks;
                    next_piece();
                }
            }
            cp_commit();
            const int pd = it / 2 - C::LAGP;
            if (pd >= 0) {
                cp_wait<C::LAGP>();
                bar_arrive(&full[(2 * pd) % C::S]);
                if (2 * pd + 1 < total) bar_arrive(&full[(2 * pd + 1) % C::S]);
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
                bar_arrive(&full[(2 * pd) % C::S]);
                if (2 * pd + 1 < total) bar_arrive(&full[(2 * pd + 1) % C::S]);
            }
        }
        cp_wait_all();
    } else {
        const int cw = warp - 4, rg = lane >> 3, c = lane & 7;
        float acc[4][TB];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int tt = 0; tt < TB; ++tt) acc[i][tt] = 0.f;
        int it = 0;
        for (int p = 0; p < npiece; ++p) {
            const Span sp = span(p);
            bool ok = true;
            for (int ks = sp.kc0; ks < sp.kc1; ++ks, ++it) {
                const int s = it % C::S;
                // every compute thread has left the previous stage (its x scratch is
                // free); stop together if a wait failed
                const bool got = bar_wait(&full[s], (it / C::S) & 1, ctl);
                if (C::PRE ? compute_sync_any(!got) : !got) {
                    ok = false;
                    break;
                }
                const unsigned char* st = ring + (size_t)s * C::STAGE;
                if (C::PRE) {
                    // convert the stage's x once: thread tc takes 8-element words tc, tc + 256, ...
                    const int tc = tid - 128;
                    for (int wdx = tc; wdx < a.B * 32; wdx += 256) {
                        const int tok = wdx >> 5, kx = wdx & 31, grp = kx >> 2;
                        float xv8[8];
                        h8_to_f8(*reinterpret_cast<const uint4*>(st + kQTile + tok * C::XROW + grp * 80 + (kx & 3) * 16),
                                 xv8);
                        float4* o = reinterpret_cast<float4*>(xsf + tok * C::XF_TOKEN + grp * C::XF_GROUP + (kx & 3) * 8);
                        o[0] = make_float4(xv8[0], xv8[1], xv8[2], xv8[3]);
                        o[1] = make_float4(xv8[4], xv8[5], xv8[6], xv8[7]);
                    }
                    compute_sync();
                }
                float sc[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    sc[i] = __half2float(*reinterpret_cast<const __half*>(st + (4 * cw + rg + 32 * i) * kQPitch + 128 +
                                                                         c * 2));
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    // odd rows take the halves in the other order: the 16 lanes of an
                    // 8-byte phase then cover all 32 banks
                    const int half = hh ^ (rg & 1);
                    float q[4][16];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        q16_to_f16(*reinterpret_cast<const uint2*>(st + (4 * cw + rg + 32 * i) * kQPitch + c * 16 +
                                                                   half * 8),
                                   q[i]);
                    const float* xs = xsf + c * C::XF_GROUP + half * 16;
                    const unsigned char* xh = st + kQTile + c * 80 + half * 32;
#pragma unroll
                    for (int tt = 0; tt < TB; ++tt) {
                        if (tt < a.B) {
                            float xv[16];
                            if (C::PRE) {
#pragma unroll
                                for (int v4 = 0; v4 < 4; ++v4) {
                                    const float4 x4 = reinterpret_cast<const float4*>(xs + tt * C::XF_TOKEN)[v4];
                                    xv[4 * v4] = x4.x;
                                    xv[4 * v4 + 1] = x4.y;
                                    xv[4 * v4 + 2] = x4.z;
                                    xv[4 * v4 + 3] = x4.w;
                                }
                            } else {
                                h8_to_f8(*reinterpret_cast<const uint4*>(xh + tt * C::XROW),
                                         *reinterpret_cast<float(*)[8]>(xv));
                                h8_to_f8(*reinterpret_cast<const uint4*>(xh + tt * C::XROW + 16),
                                         *reinterpret_cast<float(*)[8]>(xv + 8));
                            }
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                float pt = q[i][0] * xv[0];
#pragma unroll
                                for (int e = 1; e < 16; ++e) pt = fmaf(q[i][e], xv[e], pt);
                                acc[i][tt] = fmaf(sc[i], pt, acc[i][tt]);
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) bar_arrive(&empty[s]);
            }
            if (!ok) break;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int tt = 0; tt < TB; ++tt) {
                    float v = acc[i][tt];
                    v += __shfl_xor_sync(FULL, v, 1);
                    v += __shfl_xor_sync(FULL, v, 2);
                    v += __shfl_xor_sync(FULL, v, 4);
                    acc[i][tt] = v;
                }
            if (c == 0) {
                if (p < a.slots) {
                    float* dst = a.part + ((size_t)g * a.slots + p) * TB * 128;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int tt = 0; tt < TB; ++tt)
                            if (tt < a.B) dst[(size_t)tt * 128 + 4 * cw + rg + 32 * i] = acc[i][tt];
                } else if (rg == 0) {
                    atomicExch(a.status, (int)PI_ERR_WORKSPACE);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int tt = 0; tt < TB; ++tt) acc[i][tt] = 0.f;
        }
    }
}

// ------------------------------------------------------------------------ FC2

template <int TB>
struct Q2Cfg {
    // padded h row (floats): odd for TB <= 8 (lanes read one float of 8 rows);
    // 20 for TB = 16 (lanes read their row's 16 floats as 4 float4 from 4 rows)
    static constexpr int HP = TB == 16 ? 20 : (TB | 1);
    static constexpr int RAW = 64 * HP * 4;
    static constexpr int IDX = 64 * 2 * 4;
    static constexpr int STAGE = kQTile2 + RAW;
    static constexpr int S = kQBudget / (STAGE + IDX) > 12 ? 12 : kQBudget / (STAGE + IDX);
    static constexpr int LAG = S - 2;
    static constexpr size_t SMEM = (size_t)S * (STAGE + IDX) + 16;
};

struct Q2Args {
    const float* h;          // [count][B]
    const int32_t* idx;
    const int32_t* count;
    const uint8_t* codes;    // [F][d/2]
    const __half* scales;    // [F][d/32]
    const int32_t* live;     // nullable
    float* part;             // [G][slots][TB][256]
    int* status;
    long long timeout_ns;
    int B, b0, nb, d, slots;  // tokens [b0, b0 + nb) of the B in h
};

struct QPiece {
    int ct, j0, j1;
};
constexpr int kQMaxPieces = 16;

template <int TB>
__global__ void __launch_bounds__(kQThreads, 1) k_fc2_st4(Q2Args a) {
    pdl_entry();
    using C = Q2Cfg<TB>;
    extern __shared__ __align__(16) unsigned char ring[];
    __shared__ __align__(8) unsigned long long full[C::S], empty[C::S];
    __shared__ int abort_flag;
    __shared__ QPiece ptab[kQMaxPieces];

    const int n = *a.count;
    const int G = gridDim.x, g = blockIdx.x;
    const int nct = a.d / 256;
    const long long U = (long long)nct * n;
    const long long u0 = U * g / G, u1 = U * (g + 1) / G;
    if (u0 >= u1) return;
    const int npiece = (int)((u1 - 1) / n - u0 / n) + 1;
    if (npiece > kQMaxPieces) {
        if (threadIdx.x == 0) atomicExch(a.status, (int)PI_ERR_WORKSPACE);
        return;
    }
    if (threadIdx.x < npiece) {
        const int ct = (int)(u0 / n) + threadIdx.x;
        const long long lo = (long long)ct * n, hi = lo + n;
        const long long aa = u0 > lo ? u0 : lo, bb = u1 < hi ? u1 : hi;
        ptab[threadIdx.x] = QPiece{ct, (int)(aa - lo), (int)(bb - lo)};
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < C::S; ++s) {
            bar_init(&full[s], kQLoaders);
            bar_init(&empty[s], kQCompute);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const Ctl ctl{a.status, a.timeout_ns, &abort_flag};
    int32_t* sidx = reinterpret_cast<int32_t*>(ring + (size_t)C::S * C::STAGE);
    int32_t* slive = sidx + C::S * 64;
    const size_t cpr = (size_t)a.d / 2, spr = (size_t)a.d / 32;

    if (warp < 4) {
        const int t = tid, w = t >> 5, l = t & 31;
        int total = 0;
        for (int p = 0; p < npiece; ++p) total += (ptab[p].j1 - ptab[p].j0 + 63) / 64;
        int fq = 0, fpiece = 0, fst = 0;
        auto copy_ids = [&]() {
            const QPiece pc = ptab[fpiece];
            const int kk = t & 63;
            const int j = pc.j0 + 64 * fst + kk;
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
            const QPiece pc = ptab[pi_];
            const int nst = (pc.j1 - pc.j0 + 63) / 64;
            const int col0 = pc.ct * 256;
            for (int st = 0; st < nst; ++st, ++it) {
                const int s = it % C::S;
                bool good = true;
                if (it >= C::S) good = bar_wait(&empty[s], ((it / C::S) - 1) & 1, ctl);
                unsigned char* sb = ring + (size_t)s * C::STAGE;
                const int jb = pc.j0 + 64 * st;
                const int nrow = pc.j1 - jb < 64 ? pc.j1 - jb : 64;
                if (good) {
                    // codes: 4 rows x 128 bytes per warp instruction; scales: one row per thread
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int kk = 4 * (4 * i + w) + (l >> 3), c8 = l & 7;
                        unsigned char* dst = sb + kk * kQPitch + c8 * 16;
                        const bool in = kk < nrow;
                        const bool alive = a.live == nullptr || (in && slive[s * 64 + kk] != 0);
                        if (in && alive)
                            cp16(dst, a.codes + (size_t)sidx[s * 64 + kk] * cpr + col0 / 2 + c8 * 16);
                        else
                            *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    if (t < 64) {
                        unsigned char* dst = sb + t * kQPitch + 128;
                        const bool in = t < nrow && (a.live == nullptr || slive[s * 64 + t] != 0);
                        if (in)
                            cp16(dst, a.scales + (size_t)sidx[s * 64 + t] * spr + col0 / 32);
                        else
                            *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    float* raw = reinterpret_cast<float*>(sb + kQTile2);
                    for (int e = t; e < 64 * a.nb; e += kQLoaders) {
                        const int kk = e / a.nb, tok = e - kk * a.nb;
                        if (kk < nrow)
                            cp4(raw + kk * C::HP + tok, a.h + (size_t)(jb + kk) * a.B + a.b0 + tok);
                        else
                            raw[kk * C::HP + tok] = 0.f;
                    }
                    if (fq < total) copy_ids();
                }
                cp_commit();
                if (it >= C::LAG) cp_wait<C::LAG>();
                if (loaders_sync_any(!good || *(volatile int*)&abort_flag)) {
                    ok = false;
                    break;
                }
                if (it >= C::LAG) bar_arrive(&full[(it - C::LAG) % C::S]);
            }
        }
        cp_wait_all();
        if (!loaders_sync_any(!ok || *(volatile int*)&abort_flag)) {
            for (int q = it - C::LAG < 0 ? 0 : it - C::LAG; q < it; ++q) bar_arrive(&full[q % C::S]);
        }
    } else {
        // TB <= 8: lane (mc = 4cw + (lane >> 3), rg = lane & 7) owns 8 columns and rows rg + 8i;
        // TB = 16: lane (mq = 8cw + (lane & 7), rg = lane >> 3) owns 4 columns and rows rg + 4i
        // (all 16 tokens in one pass: the W2t rows are read once)
        constexpr int CPL = TB == 16 ? 4 : 8;   // columns per lane
        constexpr int NRG = TB == 16 ? 4 : 8;   // row groups (lanes sharing the columns)
        const int cw = warp - 4;
        const int col0 = TB == 16 ? (8 * cw + (lane & 7)) * 4 : (4 * cw + (lane >> 3)) * 8;
        const int rg = TB == 16 ? lane >> 3 : lane & 7;
        float acc[CPL][TB];
#pragma unroll
        for (int e = 0; e < CPL; ++e)
#pragma unroll
            for (int tt = 0; tt < TB; ++tt) acc[e][tt] = 0.f;
        int it = 0;
        for (int p = 0; p < npiece; ++p) {
            const QPiece pc = ptab[p];
            const int nst = (pc.j1 - pc.j0 + 63) / 64;
            bool ok = true;
            for (int st = 0; st < nst; ++st, ++it) {
                const int s = it % C::S;
                if (!bar_wait(&full[s], (it / C::S) & 1, ctl)) {
                    ok = false;
                    break;
                }
                const unsigned char* sb = ring + (size_t)s * C::STAGE;
                const float* raw = reinterpret_cast<const float*>(sb + kQTile2);
#pragma unroll 4
                for (int i = 0; i < 64 / NRG; ++i) {
                    const int kk = rg + NRG * i;
                    const unsigned char* rowp = sb + kk * kQPitch;
                    const uint32_t cwd = TB == 16 ? (uint32_t)*reinterpret_cast<const uint16_t*>(rowp + col0 / 2)
                                                  : *reinterpret_cast<const uint32_t*>(rowp + col0 / 2);
                    const float scl = __half2float(*reinterpret_cast<const __half*>(rowp + 128 + (col0 / 32) * 2));
                    float qf[8];
                    q8_to_f8(cwd, qf);
                    float hv[TB];
                    if (TB == 16) {
#pragma unroll
                        for (int v4 = 0; v4 < TB / 4; ++v4) {
                            const float4 h4 = reinterpret_cast<const float4*>(raw + kk * C::HP)[v4];
                            hv[4 * v4] = h4.x;
                            hv[4 * v4 + 1] = h4.y;
                            hv[4 * v4 + 2] = h4.z;
                            hv[4 * v4 + 3] = h4.w;
                        }
                    } else {
#pragma unroll
                        for (int tt = 0; tt < TB; ++tt) hv[tt] = raw[kk * C::HP + tt];
                    }
#pragma unroll
                    for (int tt = 0; tt < TB; ++tt) {
                        if (tt < a.nb) {
                            const float hs = hv[tt] * scl;
#pragma unroll
                            for (int e = 0; e < CPL; ++e) acc[e][tt] = fmaf(hs, qf[e], acc[e][tt]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) bar_arrive(&empty[s]);
            }
            if (!ok) break;
#pragma unroll
            for (int e = 0; e < CPL; ++e)
#pragma unroll
                for (int tt = 0; tt < TB; ++tt) {
                    float v = acc[e][tt];
                    if (TB == 16) {
                        v += __shfl_xor_sync(FULL, v, 8);
                        v += __shfl_xor_sync(FULL, v, 16);
                    } else {
                        v += __shfl_xor_sync(FULL, v, 1);
                        v += __shfl_xor_sync(FULL, v, 2);
                        v += __shfl_xor_sync(FULL, v, 4);
                    }
                    acc[e][tt] = v;
                }
            if (rg == 0) {
                if (p < a.slots) {
                    float* dst = a.part + ((size_t)g * a.slots + p) * TB * 256 + col0;
#pragma unroll
                    for (int tt = 0; tt < TB; ++tt)
                        if (tt < a.nb) {
                            float4* o = reinterpret_cast<float4*>(dst + (size_t)tt * 256);
#pragma unroll
                            for (int e4 = 0; e4 < CPL / 4; ++e4)
                                o[e4] = make_float4(acc[4 * e4][tt], acc[4 * e4 + 1][tt], acc[4 * e4 + 2][tt],
                                                    acc[4 * e4 + 3][tt]);
                        }
                } else {
                    atomicExch(a.status, (int)PI_ERR_WORKSPACE);
                }
            }
#pragma unroll
            for (int e = 0; e < CPL; ++e)
#pragma unroll
                for (int tt = 0; tt < TB; ++tt) acc[e][tt] = 0.f;
        }
    }
}

template <typename K>
cudaError_t prep_q(K kernel, size_t smem) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}
int qdiv(int a, int b) { return (a + b - 1) / b; }
int qslots(int tiles, int G) { return qdiv(tiles, G) + 2; }
int q1_tokens(int B) { return B <= 4 ? 4 : (B <= 8 ? 8 : 16); }
int q2_tokens(int B) { return B <= 4 ? 4 : (B <= 8 ? 8 : 16); }

}  // namespace

bool st4_supported(const Plan& p) {
    return p.int4 && !p.gated && p.B >= 2 && p.B <= 16 && p.d % 256 == 0 && p.nsm <= kMaxCtas;
}

size_t st4_part_floats(const Plan& p) {
    const size_t G = p.nsm > 0 ? p.nsm : 1;
    const size_t fc1 = G * qslots(qdiv(p.F, 128), (int)G) * q1_tokens(p.B) * 128;
    const size_t fc2 = G * qslots(p.d / 256, (int)G) * q2_tokens(p.B) * 256;
    return fc1 > fc2 ? fc1 : fc2;
}

size_t st4_fc2_part_floats(const Plan& p) {
    const size_t G = p.nsm > 0 ? p.nsm : 1;
    return G * qslots(p.d / 256, (int)G) * q2_tokens(p.B) * 256;
}

cudaError_t launch_fc1_st4(const Plan& p, const __half* x, const LayerPtrs& w, const int32_t* idx,
                           const int32_t* count, const uint32_t* mask, float* part, float* h, int32_t* live,
                           cudaStream_t s) {
    int* status = status_word();
    if (status == nullptr) return cudaErrorInvalidDevice;
    const int tb = q1_tokens(p.B), G = p.nsm;
    Q1Args a{static_cast<const uint8_t*>(w.w1), w.w1s, idx, count, x, p.d, p.B, part,
             qslots(qdiv(p.F, 128), G), status, wait_timeout_ns()};
    cudaError_t e;
#define PI_Q1(TBV)                                                       \
    if (tb == TBV) {                                                     \
        e = prep_q(k_fc1_st4<TBV>, Q1Cfg<TBV>::SMEM);                    \
        if (e != cudaSuccess) return e;                                  \
        launch_pdl(k_fc1_st4<TBV>, G, kQThreads, Q1Cfg<TBV>::SMEM, s, a);         \
    }
    PI_Q1(4) else PI_Q1(8) else PI_Q1(16)
#undef PI_Q1
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_fc1_finish(p, tb, G, a.slots, p.d / 256, part, count, idx, w.b1, mask, h, live, s);
}

cudaError_t launch_fc2_st4(const Plan& p, const float* h, const int32_t* idx, const int32_t* count,
                           const LayerPtrs& w, const int32_t* live, float* part, float* y, cudaStream_t s) {
    int* status = status_word();
    if (status == nullptr) return cudaErrorInvalidDevice;
    const int tb = q2_tokens(p.B), G = p.nsm;
    const int slots = qslots(p.d / 256, G);
    for (int b0 = 0; b0 < p.B; b0 += tb) {
        const int nb = p.B - b0 < tb ? p.B - b0 : tb;
        Q2Args a{h, idx, count, static_cast<const uint8_t*>(w.w2t), w.w2ts, live, part, status, wait_timeout_ns(),
                 p.B, b0, nb, p.d, slots};
        cudaError_t e;
#define PI_Q2(TBV)                                                       \
        if (tb == TBV) {                                                 \
            e = prep_q(k_fc2_st4<TBV>, Q2Cfg<TBV>::SMEM);                \
            if (e != cudaSuccess) return e;                              \
            launch_pdl(k_fc2_st4<TBV>, G, kQThreads, Q2Cfg<TBV>::SMEM, s, a);     \
        }
        PI_Q2(4) else PI_Q2(8) else PI_Q2(16)
#undef PI_Q2
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        e = launch_fc2_reduce(p, tb, G, slots, 256, nb, b0, part, count, w.b2, y, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace pi
