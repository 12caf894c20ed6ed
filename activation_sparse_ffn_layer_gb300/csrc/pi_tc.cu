// pi_tc.cu -- the batched union path on the tcgen05 tensor cores (batch 16..32,
// fp16 weights).
//
// At batch B the union of the B tokens' predicted neurons is gathered once and
// both FFN products become dense contractions over the gathered rows
// (PowerInfer (arXiv 2312.12456) §5 "Neuron-aware Inference Engine": only the
// activated rows of W1 and columns of W2 are processed; §4.3 / Figure 6 for the
// row-per-neuron layout):
//
//   FC1   Z[j, t] = sum_k W1[idx_j, k] x[t, k]        M = 128 listed neurons,
//                                                      N = tokens, K = d
//   FC2   y[t, c] = sum_j h[j, t] W2t[idx_j, c]       M = 128 columns of y,
//                                                      N = tokens (hi | lo), K = j
//
// One CTA per SM, three warp roles:
//   warps 0-3  load: cp.async 16-byte copies of the gathered rows straight into
//              the tensor cores' shared-memory operand layout (no swizzle:
//              8 rows x 16 bytes per core matrix), a ring of stages;
//   warp  8    one thread issues tcgen05.mma (fp16 x fp16 -> fp32 in TMEM);
//   warps 4-7  drain the TMEM accumulators (tcgen05.ld) and apply the epilogue.
// Ring slots are handed over with mbarriers: loaders arrive on `full` after
// their copies landed; tcgen05.commit arrives on `empty` when the MMAs that
// read a slot are done.  Two accumulator buffers let the epilogue of one tile
// overlap the MMAs of the next.  Every wait is bounded: on expiry the status
// word becomes PI_ERR_TIMEOUT, the CTA drains its own copies and MMAs, frees
// its tensor memory and returns.
//
// FC1 work split: each CTA takes an equal contiguous share of the union list,
// cut into tiles of at most 128 rows, so every SM streams the same bytes.
// FC2 work split: the (column tile x union row) space is cut into equal
// contiguous ranges per CTA ("stream-K"); each CTA writes one partial tile per
// column tile it touches and a fixed-order reduction adds the partials to b2.
//
// FC2 feeds h to the tensor cores as two fp16 halves, hi = fp16(h) and
// lo = fp16(h - hi), placed as extra N columns: hi + lo carries 22 bits of h,
// so the product keeps fp32-level accuracy.  Weights and x are fp16 already,
// and fp16 x fp16 products are exact in the fp32 accumulator.
#include <cuda_runtime.h>

#include "pi_common.cuh"
#include "pi_internal.h"

namespace pi {
namespace {

constexpr int kTcThreads = 288;      // warps 0-3 load, 4-7 epilogue, 8 MMA
constexpr int kLoaders = 128;
constexpr int kRingBudget = 200 * 1024;
constexpr int kTileA = 16384;        // 128 x 64 fp16 operand tile

PI_DEV unsigned long long tc_timer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
PI_DEV unsigned su32(const void* p) { return static_cast<unsigned>(__cvta_generic_to_shared(p)); }

PI_DEV void bar_init(unsigned long long* b, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}
PI_DEV void bar_arrive(unsigned long long* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
PI_DEV bool bar_try(unsigned long long* b, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n .reg .pred q;\n mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n selp.u32 %0, 1, 0, q;\n}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

struct Ctl {
    int* status;
    long long timeout_ns;
    int* abort_flag;  // shared memory
};

// Wait (bounded) for the phase with this parity.  False on expiry or when
// another role of the CTA already gave up.
PI_DEV bool bar_wait(unsigned long long* b, unsigned parity, const Ctl& c) {
    if (bar_try(b, parity)) return true;
    const unsigned long long t0 = tc_timer();
    for (;;) {
        if (bar_try(b, parity)) return true;
        if (*(volatile int*)c.abort_flag) return false;
        if ((long long)(tc_timer() - t0) > c.timeout_ns) {
            atomicExch(c.status, (int)PI_ERR_TIMEOUT);
            *(volatile int*)c.abort_flag = 1;
            return false;
        }
    }
}
// Bounded wait that ignores the abort flag (used while draining).
PI_DEV void bar_drain(unsigned long long* b, unsigned parity, long long timeout_ns) {
    const unsigned long long t0 = tc_timer();
    while (!bar_try(b, parity) && (long long)(tc_timer() - t0) <= timeout_ns) {
    }
}

PI_DEV void cp16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(su32(dst)), "l"(src) : "memory");
}
PI_DEV void cp4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(su32(dst)), "l"(src) : "memory");
}
PI_DEV void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
PI_DEV void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
PI_DEV void cp_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// generic-proxy writes to shared memory -> visible to the tensor cores
PI_DEV void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// Barrier of the 128 loader threads that also ORs a flag over them, so every
// loader takes the same branch afterwards.
PI_DEV bool loaders_sync_any(bool v) {
    unsigned r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, 1, 128, q;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(r)
        : "r"((unsigned)v)
        : "memory");
    return r != 0;
}

PI_DEV void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
PI_DEV void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, no swizzle: start, leading-dimension byte
// offset (between core matrices adjacent in K for K-major operands, in K for
// MN-major ones), stride-dimension byte offset (between core matrices adjacent
// in M/N), fixed version field 1 at bit 46.
PI_DEV uint64_t sdesc(unsigned addr, unsigned lbo, unsigned sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}
// Instruction descriptor of kind::f16: fp32 D, fp16 A and B, A major-ness,
// B K-major, N >> 3 at bit 17, M >> 4 at bit 24.
PI_DEV unsigned idesc_f16(int M, int N, bool a_mn_major) {
    return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((unsigned)(N >> 3) << 17) | ((unsigned)(M >> 4) << 24);
}
PI_DEV void mma_f16(unsigned tmem_d, uint64_t a, uint64_t b, unsigned idesc, unsigned accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
PI_DEV void mma_commit(unsigned long long* b) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(b))
                 : "memory");
}
// 16 consecutive fp32 columns of this thread's TMEM lane
PI_DEV void tmem_ld16(unsigned taddr, float* v) {
    unsigned r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
PI_DEV void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

PI_DEV void tmem_alloc(unsigned* slot, unsigned cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(slot)), "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
PI_DEV void tmem_free(unsigned base, unsigned cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols) : "memory");
}

PI_DEV unsigned char* align1024(unsigned char* p) {
    return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

constexpr int tmem_cols_for(int c) { return c <= 32 ? 32 : c <= 64 ? 64 : c <= 128 ? 128 : 256; }

// ------------------------------------------------------------------------ FC1

template <bool GATED, int NT>
struct Fc1Cfg {
    static constexpr int NA = GATED ? 2 : 1;            // operand tiles per stage (gate, up)
    static constexpr int X = NT * 128;                   // NT tokens x 64 fp16
    static constexpr int STAGE = NA * kTileA + X;
    static constexpr int S = kRingBudget / STAGE > 8 ? 8 : kRingBudget / STAGE;
    static constexpr int LAG = S - 2;                    // stages whose copies stay in flight
    static constexpr int ACC = NA * NT;                  // TMEM columns per accumulator buffer
    static constexpr int TMEM = tmem_cols_for(2 * ACC);
    static constexpr size_t SMEM = (size_t)S * STAGE + 1024;
};

struct TcFc1Args {
    const __half* x;
    const __half* w1;
    const __half* wu;
    const __half* b1;
    const int32_t* idx;
    const int32_t* count;
    const uint32_t* mask;  // per-token masks [B][W] (nullable)
    float* h;              // [count][B]
    uint8_t* live;         // nullable [F]: 1 where some token's h is non-zero
    int* status;
    long long timeout_ns;
    int B, d, W;
};

// h[j, t] = act(W1[idx_j] . x_t + b1[idx_j]) for the union list, zero where
// token t's own mask does not list idx_j.
template <bool GATED, int NT>
__global__ void __launch_bounds__(kTcThreads, 1) k_fc1_tc(TcFc1Args a) {
    using C = Fc1Cfg<GATED, NT>;
    extern __shared__ unsigned char dsm[];
    __shared__ __align__(8) unsigned long long full[C::S], empty[C::S], accf[2], acce[2], drain;
    __shared__ unsigned tmem_slot;
    __shared__ int abort_flag;

    const int n = *a.count;
    const int G = gridDim.x, g = blockIdx.x;
    const int r0 = (int)((long long)n * g / G), r1 = (int)((long long)n * (g + 1) / G);
    const int len = r1 - r0;
    if (len <= 0) return;
    const int ntile = (len + 127) / 128;
    const int nk = a.d / 64;
    const int total = ntile * nk;
    unsigned char* ring = align1024(dsm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < C::S; ++s) {
            bar_init(&full[s], kLoaders);
            bar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            bar_init(&accf[b], 1);
            bar_init(&acce[b], 128);
        }
        bar_init(&drain, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 8) tmem_alloc(&tmem_slot, C::TMEM);
    tc_before();
    __syncthreads();
    tc_after();
    const unsigned tmem = tmem_slot;
    const Ctl ctl{a.status, a.timeout_ns, &abort_flag};
    auto tile_lo = [&](int i) { return r0 + (int)((long long)len * i / ntile); };

    if (warp < 4) {
        // ---- loaders: thread t copies chunk kc of 8 rows per stage (each warp
        // instruction covers 8 rows x 64 contiguous bytes; the 8 lanes of a
        // shared-memory phase hit 8 different banks groups)
        const int t = tid, w = t >> 5, l = t & 31;
        const int kc = 4 * (w & 1) + (l >> 3);
        const int rb = w >> 1;
        int it = 0;
        bool ok = true;
        for (int i = 0; i < ntile && ok; ++i) {
            const int tr0 = tile_lo(i), rows = tile_lo(i + 1) - tr0;
            const __half* src[8];
            const __half* srcu[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int row = 8 * (2 * q + rb) + (l & 7);
                src[q] = nullptr;
                srcu[q] = nullptr;
                if (row < rows) {
                    const size_t k = (size_t)a.idx[tr0 + row];
                    src[q] = a.w1 + k * a.d + kc * 8;
                    if (GATED) srcu[q] = a.wu + k * a.d + kc * 8;
                }
            }
            for (int ks = 0; ks < nk; ++ks, ++it) {
                const int s = it % C::S;
                if (it >= C::S && !bar_wait(&empty[s], ((it / C::S) - 1) & 1, ctl)) {
                    ok = false;
                    break;
                }
                unsigned char* st = ring + (size_t)s * C::STAGE;
                const int k0 = ks * 64;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (src[q] != nullptr) {
                        const int row = 8 * (2 * q + rb) + (l & 7);
                        const unsigned off = kc * 2048 + (row >> 3) * 128 + (row & 7) * 16;
                        cp16(st + off, src[q] + k0);
                        if (GATED) cp16(st + kTileA + off, srcu[q] + k0);
                    }
                }
#pragma unroll
                for (int p = t; p < NT * 8; p += kLoaders) {
                    const int gg = p >> 5, ll = p & 31;
                    const int tok = 8 * (gg >> 1) + (ll & 7), kx = 4 * (gg & 1) + (ll >> 3);
                    if (tok < a.B)
                        cp16(st + C::NA * kTileA + kx * (NT * 16) + (tok >> 3) * 128 + (tok & 7) * 16,
                             a.x + (size_t)tok * a.d + k0 + kx * 8);
                }
                cp_commit();
                if (it >= C::LAG) {
                    cp_wait<C::LAG>();
                    fence_async_smem();
                    bar_arrive(&full[(it - C::LAG) % C::S]);
                }
            }
        }
        cp_wait_all();
        if (ok) {
            fence_async_smem();
            for (int q = total - C::LAG < 0 ? 0 : total - C::LAG; q < total; ++q) bar_arrive(&full[q % C::S]);
        }
    } else if (warp < 8) {
        // ---- epilogue: TMEM lane m = row m of the tile
        const int e = warp - 4, m = 32 * e + lane;
        for (int i = 0; i < ntile; ++i) {
            const int b = i & 1;
            if (!bar_wait(&accf[b], (i >> 1) & 1, ctl)) break;
            tc_after();
            float z[NT], zu[GATED ? NT : 1];
            const unsigned ta = tmem + ((unsigned)(32 * e) << 16) + (unsigned)(b * C::ACC);
#pragma unroll
            for (int c = 0; c < NT; c += 16) {
                tmem_ld16(ta + c, z + c);
                if (GATED) tmem_ld16(ta + NT + c, zu + c);
            }
            tmem_wait_ld();
            tc_before();
            bar_arrive(&acce[b]);
            const int tr0 = tile_lo(i), rows = tile_lo(i + 1) - tr0;
            if (m < rows) {
                const int j = tr0 + m;
                const int k = a.idx[j];
                const float bk = __half2float(a.b1[k]);
                float* hrow = a.h + (size_t)j * a.B;
                bool any = false;
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if (t < a.B) {
                        float v = z[t] + bk;
                        v = v > 0.f ? v : 0.f;
                        if (GATED) v *= zu[t];
                        if (a.mask != nullptr && !((a.mask[(size_t)t * a.W + (k >> 5)] >> (k & 31)) & 1u)) v = 0.f;
                        hrow[t] = v;
                        any |= v != 0.f;
                    }
                }
                if (a.live != nullptr) a.live[j] = any ? 1 : 0;
            }
        }
    } else if (lane == 0) {
        // ---- MMA issuer
        const unsigned idesc = idesc_f16(128, NT, false);
        int it = 0;
        bool ok = true;
        for (int i = 0; i < ntile && ok; ++i) {
            const int b = i & 1;
            if (i >= 2 && !bar_wait(&acce[b], ((i >> 1) - 1) & 1, ctl)) {
                ok = false;
                break;
            }
            tc_after();
            const unsigned dcol = tmem + (unsigned)(b * C::ACC);
            for (int ks = 0; ks < nk; ++ks, ++it) {
                const int s = it % C::S;
                if (!bar_wait(&full[s], (it / C::S) & 1, ctl)) {
                    ok = false;
                    break;
                }
                tc_after();
                const unsigned sa = su32(ring + (size_t)s * C::STAGE);
                const unsigned sx = sa + C::NA * kTileA;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t bd = sdesc(sx + kk * 2 * NT * 16, NT * 16, 128);
                    const unsigned acc = (ks | kk) ? 1u : 0u;
                    mma_f16(dcol, sdesc(sa + kk * 4096, 2048, 128), bd, idesc, acc);
                    if (GATED) mma_f16(dcol + NT, sdesc(sa + kTileA + kk * 4096, 2048, 128), bd, idesc, acc);
                }
                mma_commit(&empty[s]);
            }
            if (ok) mma_commit(&accf[b]);
        }
        if (ok) {
            // every slot's last release has arrived before the CTA may exit
            for (int s = 0; s < C::S && s < total; ++s) {
                const int last = s + ((total - 1 - s) / C::S) * C::S;
                bar_drain(&empty[s], (last / C::S) & 1, a.timeout_ns);
            }
        } else {
            mma_commit(&drain);
            bar_drain(&drain, 0, a.timeout_ns);
        }
    }
    tc_before();
    __syncthreads();
    if (warp == 8) {
        tc_after();
        tmem_free(tmem, C::TMEM);
    }
}

// ------------------------------------------------------------------------ FC2

template <int NT>
struct Fc2Cfg {
    static constexpr int BOP = 2 * NT * 64 * 2;          // (hi | lo) tokens x 64 rows fp16
    static constexpr int RAW = 64 * NT * 4;              // 64 rows x B fp32 of h, as copied
    static constexpr int STAGE = kTileA + BOP + RAW;
    static constexpr int S = kRingBudget / STAGE > 8 ? 8 : kRingBudget / STAGE;
    static constexpr int LAG = S - 2;
    static constexpr int ACC = 2 * NT;
    static constexpr int TMEM = tmem_cols_for(2 * ACC);
    static constexpr size_t SMEM = (size_t)S * STAGE + 1024;
};

struct TcFc2Args {
    const float* h;        // [count][B]
    const int32_t* idx;
    const int32_t* count;
    const __half* w2t;
    const uint8_t* live;   // nullable: rows with live == 0 have h == 0 for every token
    float* part;           // [G][slots][NT][128]
    int* status;
    long long timeout_ns;
    int B, d, slots;
};

struct Piece {
    int ct, j0, j1;
};

// Pieces of CTA g: the column tiles its range [u0, u1) of the (tile, row)
// space touches, with the row interval inside each.
PI_DEV int fc2_piece(long long u0, long long u1, int n, int which, Piece* out) {
    const int ct0 = (int)(u0 / n);
    const int ct = ct0 + which;
    const long long lo = (long long)ct * n, hi = lo + n;
    const long long a = u0 > lo ? u0 : lo, b = u1 < hi ? u1 : hi;
    out->ct = ct;
    out->j0 = (int)(a - lo);
    out->j1 = (int)(b - lo);
    return ct - ct0;
}

template <int NT>
__global__ void __launch_bounds__(kTcThreads, 1) k_fc2_tc(TcFc2Args a) {
    using C = Fc2Cfg<NT>;
    extern __shared__ unsigned char dsm[];
    __shared__ __align__(8) unsigned long long full[C::S], empty[C::S], accf[2], acce[2], drain;
    __shared__ unsigned tmem_slot;
    __shared__ int abort_flag;

    const int n = *a.count;
    const int G = gridDim.x, g = blockIdx.x;
    const int nct = a.d / 128;
    const long long U = (long long)nct * n;
    const long long u0 = U * g / G, u1 = U * (g + 1) / G;
    if (u0 >= u1) return;
    const int npiece = (int)((u1 - 1) / n - u0 / n) + 1;
    unsigned char* ring = align1024(dsm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < C::S; ++s) {
            bar_init(&full[s], kLoaders);
            bar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            bar_init(&accf[b], 1);
            bar_init(&acce[b], 128);
        }
        bar_init(&drain, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 8) tmem_alloc(&tmem_slot, C::TMEM);
    tc_before();
    __syncthreads();
    tc_after();
    const unsigned tmem = tmem_slot;
    const Ctl ctl{a.status, a.timeout_ns, &abort_flag};

    if (warp < 4) {
        // ---- loaders: thread t copies 16-byte column chunk mc of 8 rows per
        // stage; 64 rows x B floats of h are copied raw and converted to
        // (hi, lo) fp16 once every loader's copies of the stage have landed
        const int t = tid, w = t >> 5, l = t & 31;
        const int mc = 4 * w + (l >> 3);
        const bool vec = (a.B & 3) == 0 && (reinterpret_cast<uintptr_t>(a.h) & 15) == 0;
        int it = 0;     // stage being issued
        int cv = 0;     // next stage to convert and publish
        int cv_piece = 0, cv_st = 0;
        bool ok = true;
        auto convert = [&](int q, const Piece& pc, int st) {
            unsigned char* sb = ring + (size_t)(q % C::S) * C::STAGE;
            const float* raw = reinterpret_cast<const float*>(sb + kTileA + C::BOP);
            const int jb = pc.j0 + 64 * st;
            const int nrow = pc.j1 - jb < 64 ? pc.j1 - jb : 64;
#pragma unroll
            for (int p = t; p < NT * 8; p += kLoaders) {
                const int tok = p % NT, kc = p / NT;
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const int r = 8 * kc + e;
                    const float v0 = (tok < a.B && r < nrow) ? raw[r * a.B + tok] : 0.f;
                    const float v1 = (tok < a.B && r + 1 < nrow) ? raw[(r + 1) * a.B + tok] : 0.f;
                    const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
                    const __half l0 = __float2half_rn(v0 - __half2float(h0));
                    const __half l1 = __float2half_rn(v1 - __half2float(h1));
                    hi[e >> 1] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
                    lo[e >> 1] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
                }
                unsigned char* bo = sb + kTileA + kc * (2 * NT * 16);
                *reinterpret_cast<uint4*>(bo + (tok >> 3) * 128 + (tok & 7) * 16) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                const int tl = NT + tok;
                *reinterpret_cast<uint4*>(bo + (tl >> 3) * 128 + (tl & 7) * 16) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        };
        // publish stage cv: every loader's copies for it have landed
        auto publish = [&]() {
            Piece pc;
            fc2_piece(u0, u1, n, cv_piece, &pc);
            convert(cv, pc, cv_st);
            fence_async_smem();
            bar_arrive(&full[cv % C::S]);
            ++cv;
            if (64 * (++cv_st) >= pc.j1 - pc.j0) {
                ++cv_piece;
                cv_st = 0;
            }
        };
        for (int pi_ = 0; pi_ < npiece && ok; ++pi_) {
            Piece pc;
            fc2_piece(u0, u1, n, pi_, &pc);
            const int nst = (pc.j1 - pc.j0 + 63) / 64;
            const int col0 = pc.ct * 128;
            for (int st = 0; st < nst; ++st, ++it) {
                const int s = it % C::S;
                bool good = true;
                if (it >= C::S) good = bar_wait(&empty[s], ((it / C::S) - 1) & 1, ctl);
                unsigned char* sb = ring + (size_t)s * C::STAGE;
                const int jb = pc.j0 + 64 * st;
                if (good) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int kk = 8 * q + (l & 7);
                        const int j = jb + kk;
                        unsigned char* dst = sb + mc * 128 + (kk >> 3) * 2048 + (kk & 7) * 16;
                        bool take = j < pc.j1;
                        if (take && a.live != nullptr) take = a.live[j] != 0;
                        if (take)
                            cp16(dst, a.w2t + (size_t)a.idx[j] * a.d + col0 + mc * 8);
                        else
                            *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    const int nrow = pc.j1 - jb < 64 ? pc.j1 - jb : 64;
                    unsigned char* raw = sb + kTileA + C::BOP;
                    const float* hsrc = a.h + (size_t)jb * a.B;
                    if (vec) {
                        for (int c = t; c < nrow * a.B / 4; c += kLoaders) cp16(raw + 16 * c, hsrc + 4 * c);
                    } else {
                        for (int c = t; c < nrow * a.B; c += kLoaders) cp4(raw + 4 * c, hsrc + c);
                    }
                }
                cp_commit();
                if (it >= C::LAG) cp_wait<C::LAG>();
                // every loader's copies of stage it - LAG have landed; stop together
                if (loaders_sync_any(!good || *(volatile int*)&abort_flag)) {
                    ok = false;
                    break;
                }
                if (it >= C::LAG) publish();
            }
        }
        cp_wait_all();
        if (!loaders_sync_any(!ok || *(volatile int*)&abort_flag)) {
            while (cv < it) publish();
        }
    } else if (warp < 8) {
        // ---- epilogue: TMEM lane m = column col0 + m; hi and lo halves summed
        const int e = warp - 4, m = 32 * e + lane;
        for (int p = 0; p < npiece; ++p) {
            const int b = p & 1;
            if (!bar_wait(&accf[b], (p >> 1) & 1, ctl)) break;
            tc_after();
            float vh[NT], vl[NT];
            const unsigned ta = tmem + ((unsigned)(32 * e) << 16) + (unsigned)(b * C::ACC);
#pragma unroll
            for (int c = 0; c < NT; c += 16) {
                tmem_ld16(ta + c, vh + c);
                tmem_ld16(ta + NT + c, vl + c);
            }
            tmem_wait_ld();
            tc_before();
            bar_arrive(&acce[b]);
            if (p < a.slots) {
                float* dst = a.part + (((size_t)g * a.slots + p) * NT) * 128 + m;
#pragma unroll
                for (int t = 0; t < NT; ++t)
                    if (t < a.B) dst[(size_t)t * 128] = vh[t] + vl[t];
            } else if (lane == 0) {
                atomicExch(a.status, (int)PI_ERR_WORKSPACE);
            }
        }
    } else if (lane == 0) {
        // ---- MMA issuer: A = W2t rows (M = 128 columns, MN-major), B = h (hi | lo)
        const unsigned idesc = idesc_f16(128, 2 * NT, true);
        int it = 0;
        bool ok = true;
        for (int p = 0; p < npiece && ok; ++p) {
            Piece pc;
            fc2_piece(u0, u1, n, p, &pc);
            const int nst = (pc.j1 - pc.j0 + 63) / 64;
            const int b = p & 1;
            if (p >= 2 && !bar_wait(&acce[b], ((p >> 1) - 1) & 1, ctl)) {
                ok = false;
                break;
            }
            tc_after();
            const unsigned dcol = tmem + (unsigned)(b * C::ACC);
            for (int st = 0; st < nst; ++st, ++it) {
                const int s = it % C::S;
                if (!bar_wait(&full[s], (it / C::S) & 1, ctl)) {
                    ok = false;
                    break;
                }
                tc_after();
                const unsigned sa = su32(ring + (size_t)s * C::STAGE);
                const unsigned sbop = sa + kTileA;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = sdesc(sa + kk * 4096, 2048, 128);
                    const uint64_t bd = sdesc(sbop + kk * 2 * (2 * NT * 16), 2 * NT * 16, 128);
                    mma_f16(dcol, ad, bd, idesc, (st | kk) ? 1u : 0u);
                }
                mma_commit(&empty[s]);
            }
            if (ok) mma_commit(&accf[b]);
        }
        if (ok) {
            for (int s = 0; s < C::S && s < it; ++s) {
                const int last = s + ((it - 1 - s) / C::S) * C::S;
                bar_drain(&empty[s], (last / C::S) & 1, a.timeout_ns);
            }
        } else {
            mma_commit(&drain);
            bar_drain(&drain, 0, a.timeout_ns);
        }
    }
    tc_before();
    __syncthreads();
    if (warp == 8) {
        tc_after();
        tmem_free(tmem, C::TMEM);
    }
}

// y[t, c] = b2[c] + sum over the CTAs whose range touches column tile c / 128
// of their partial (ascending CTA order: reproducible).
__global__ void __launch_bounds__(256) k_fc2_tc_reduce(const float* __restrict__ part, int slots, int G,
                                                       const int32_t* __restrict__ count, int B, int NT, int d,
                                                       const __half* __restrict__ b2, float* __restrict__ y) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= B * d) return;
    const int t = e / d, c = e - t * d;
    float acc = __half2float(b2[c]);
    const int n = *count;
    if (n > 0) {
        const int nct = d / 128, ct = c / 128, m = c % 128;
        const long long U = (long long)nct * n;
        const long long lo = (long long)ct * n, hi = lo + n;
        long long gs = lo * G / U;
        int gg = (int)gs;
        while (gg > 0 && U * gg / G > lo) --gg;          // u0(gg) <= lo
        while (gg < G && U * (gg + 1) / G <= lo) ++gg;   // first range reaching past lo
        for (; gg < G; ++gg) {
            const long long u0 = U * gg / G, u1 = U * (gg + 1) / G;
            if (u0 >= hi) break;
            if (u0 >= u1) continue;
            const int slot = ct - (int)(u0 / n);
            if (slot < slots) acc += part[(((size_t)gg * slots + slot) * NT + t) * 128 + m];
        }
    }
    y[e] = acc;
}

template <typename K>
cudaError_t prep(K kernel, size_t smem) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

constexpr long long kTcTimeoutNs = 2000000000ll;

}  // namespace

bool tc_supported(const Plan& p) { return !p.int4 && p.B >= 16 && p.B <= 32 && p.d % 128 == 0; }

int tc_tokens(const Plan& p) { return p.B <= 16 ? 16 : 32; }

int tc_slots(const Plan& p) { return (p.d / 128) / (p.nsm > 0 ? p.nsm : 1) + 2; }

size_t tc_part_floats(const Plan& p) { return (size_t)p.nsm * tc_slots(p) * tc_tokens(p) * 128; }

cudaError_t launch_fc1_tc(const Plan& p, const __half* x, const LayerPtrs& w, const int32_t* idx,
                          const int32_t* count, const uint32_t* mask, float* h, uint8_t* live, cudaStream_t s) {
    int* status = status_word();
    if (status == nullptr) return cudaErrorInvalidDevice;
    TcFc1Args a{x, static_cast<const __half*>(w.w1), w.wu, w.b1, idx, count, mask, h, live, status, kTcTimeoutNs,
                p.B, p.d, p.W};
    const int grid = p.nsm;
#define PI_FC1TC(GV, NV)                                                          \
    {                                                                             \
        cudaError_t e = prep(k_fc1_tc<GV, NV>, Fc1Cfg<GV, NV>::SMEM);            \
        if (e != cudaSuccess) return e;                                           \
        k_fc1_tc<GV, NV><<<grid, kTcThreads, Fc1Cfg<GV, NV>::SMEM, s>>>(a);        \
        return cudaGetLastError();                                                \
    }
    const int nt = tc_tokens(p);
    if (p.gated) {
        if (nt == 16) PI_FC1TC(true, 16)
        PI_FC1TC(true, 32)
    }
    if (nt == 16) PI_FC1TC(false, 16)
    PI_FC1TC(false, 32)
#undef PI_FC1TC
}

cudaError_t launch_fc2_tc(const Plan& p, const float* h, const int32_t* idx, const int32_t* count,
                          const LayerPtrs& w, const uint8_t* live, float* partial, float* y, cudaStream_t s) {
    int* status = status_word();
    if (status == nullptr) return cudaErrorInvalidDevice;
    const int slots = tc_slots(p), nt = tc_tokens(p);
    TcFc2Args a{h, idx, count, static_cast<const __half*>(w.w2t), live, partial, status, kTcTimeoutNs,
                p.B, p.d, slots};
    const int grid = p.nsm;
    cudaError_t e;
    if (nt == 16) {
        e = prep(k_fc2_tc<16>, Fc2Cfg<16>::SMEM);
        if (e != cudaSuccess) return e;
        k_fc2_tc<16><<<grid, kTcThreads, Fc2Cfg<16>::SMEM, s>>>(a);
    } else {
        e = prep(k_fc2_tc<32>, Fc2Cfg<32>::SMEM);
        if (e != cudaSuccess) return e;
        k_fc2_tc<32><<<grid, kTcThreads, Fc2Cfg<32>::SMEM, s>>>(a);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int total = p.B * p.d;
    k_fc2_tc_reduce<<<(total + 255) / 256, 256, 0, s>>>(partial, slots, grid, count, p.B, nt, p.d, w.b2, y);
    return cudaGetLastError();
}

}  // namespace pi
