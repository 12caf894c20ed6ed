// pi_fused.cu -- the whole decode step of a layer stack in ONE persistent,
// cooperative launch (one CTA per SM), batch 1.
//
// Per layer (PowerInfer summary (CSDN): "Adaptive sparse predictor",
// "Neuron-aware operator", "Background"):
//   A  u-partials  = P1[i, segment] . x              (items spread over all warps)
//   B  mask bits   = (P2 u + b > tau) of this CTA's own rows, then FC1 of its
//      own predicted rows (bias + ReLU [+ gate]) and the FC2 gather-accumulate
//      of those neurons into a private partial y -- no exchange of the mask:
//      a CTA computes the FFN of exactly the neurons it predicted
//   D  y columns   = b2 + sum of all partials (fixed order), sum of squares
//   (next layer)   x = fp16(y / sqrt(mean(y^2) + eps))
// with one grid barrier after each phase (three per layer; the last layer's
// third is the end of the grid).  Rows are owned in
// pieces of 8: the pieces of round k (G consecutive pieces) go to the CTAs in
// ascending order for even k and descending order for odd k, so that the hot
// rows at the start of the table spread over all CTAs.
//
// The barrier is a single counter: each CTA adds 1 with release semantics and
// spins (one thread, acquire loads) until the count reaches the barrier's
// target.  Targets are relative to an epoch kept in the workspace and advanced
// by every launch, so the counter is never reset.  Every wait is bounded by a
// wall-clock limit: on expiry the status word becomes PI_ERR_TIMEOUT and the
// kernel returns (the other CTAs then time out at their next barrier).
// Exchanged data is written with plain stores and read with L2-only loads.
//
// Weights move into shared memory by bulk copies (TMA): a CTA's predictor slice
// of the next layer is requested while the current layer's partial sums are
// reduced, and its FC rows stream through a ring of row slots.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "pi_common.cuh"
#include "pi_internal.h"

namespace pi {

__device__ int g_pi_status = 0;

namespace {

constexpr int kThreads = 256;
constexpr int kCols = 8 * kThreads;   // fp16 FC2 columns of one chunk (8 per thread)
constexpr int kWarps = kThreads / 32;
constexpr int kBarriersPerLayer = 3;
constexpr int kMaxUnits = 64;   // 16-row units (two 8-row pieces) per CTA
constexpr int kRingMax = 8;   // P2 ring slots at most
constexpr int kMaxFcSlots = 32;   // FC row ring slots at most
constexpr int kPrefetchUnits = 4; // P2 units brought into L2 during the u barrier

PI_DEV unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
PI_DEV unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
PI_DEV float4 ld_cg4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

// ---- shared-memory mbarrier + 1D bulk copy (TMA) helpers
PI_DEV unsigned smem_u32(const void* p) { return static_cast<unsigned>(__cvta_generic_to_shared(p)); }
PI_DEV void mbar_init(unsigned long long* mbar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(mbar)), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
PI_DEV void mbar_arrive_expect_tx(unsigned long long* mbar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(mbar)), "r"(bytes) : "memory");
}
PI_DEV bool mbar_test(unsigned long long* mbar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n .reg .pred q;\n mbarrier.test_wait.parity.shared::cta.b64 q, [%1], %2;\n selp.u32 %0, 1, 0, q;\n}"
        : "=r"(ok)
        : "r"(smem_u32(mbar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// global -> shared bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned)
PI_DEV void bulk_g2s(void* dst, const void* src, unsigned bytes, unsigned long long* mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(mbar))
                 : "memory");
}
// Bring the 128-byte lines that hold [p, p + bytes) into L2 through the
// load/store path (no registers written, nothing to wait for): thread t of n
// takes lines t, t + n, ...
PI_DEV void prefetch_lines(const void* p, size_t bytes, int t, int n) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(p) & ~(uintptr_t)127;
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(p) + bytes;
    for (uintptr_t a = a0 + (uintptr_t)t * 128; a < a1; a += (uintptr_t)n * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
}

// Before leaving after a failure: wait (bounded) for this CTA's own bulk copy
// still in flight, so none lands in shared memory after the CTA has exited.
PI_DEV void mbar_drain(unsigned long long* mbar, unsigned parity, long long timeout_ns) {
    const unsigned long long t0 = globaltimer();
    while (!mbar_test(mbar, parity) && (long long)(globaltimer() - t0) <= timeout_ns) {
    }
}

// Wait (bounded) until the mbarrier phase with this parity has completed.
// The spinning part stays out of line: the kernel waits at many places, and
// one copy of the loop keeps its code (fetched afresh every layer) small.
__device__ __noinline__ bool mbar_wait_slow(unsigned long long* mbar, unsigned parity, long long timeout_ns, int* bad) {
    const unsigned long long t0 = globaltimer();
    while (!mbar_test(mbar, parity)) {
        if ((long long)(globaltimer() - t0) > timeout_ns || *(volatile int*)bad) {
            atomicExch(&g_pi_status, (int)PI_ERR_TIMEOUT);
            *(volatile int*)bad = 1;
            return false;
        }
    }
    return true;
}
PI_DEV bool mbar_wait(unsigned long long* mbar, unsigned parity, long long timeout_ns, int* bad) {
    return mbar_test(mbar, parity) || mbar_wait_slow(mbar, parity, timeout_ns, bad);
}

// Grid barrier number `k` of this launch.  Returns false (and sets the status
// word) if the wait exceeded timeout_ns or another CTA already failed.  Warp 0
// runs between() after this CTA's arrival, before waiting for the others.
template <typename Between>
PI_DEV bool grid_sync(unsigned* counter, unsigned target, long long timeout_ns, int* bad, Between&& between) {
    __syncthreads();
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(counter) : "memory");
        __syncwarp();
        between();
    }
    if (threadIdx.x == 0) {
        unsigned v = ld_acquire(counter);
        if ((int)(v - target) < 0) {
            const unsigned long long t0 = globaltimer();
            int polls = 0;
            while ((int)((v = ld_acquire(counter)) - target) < 0) {
                if (++polls == 32) {
                    polls = 0;
                    if ((long long)(globaltimer() - t0) > timeout_ns || *(volatile int*)&g_pi_status != 0) {
                        atomicExch(&g_pi_status, (int)PI_ERR_TIMEOUT);
                        *bad = 1;
                        break;
                    }
                }
            }
        }
    }
    __syncthreads();
    return *(volatile int*)bad == 0;
}

}  // namespace

struct FusedLayer {
    const void* w1;
    const __half* w1s;
    const __half* b1;
    const __half* wu;
    const void* w2t;
    const __half* w2ts;
    const __half* b2;
    const __half* p1;
    const __half* p2;
    int r;    // predictor rank
    int su;   // splits of d in the P1 x items
    int seg;  // elements per split (multiple of 8)
};

constexpr int kMaxFusedLayers = 96;

struct FusedParams {
    int L, d, F, M, W;   // M = ceil(F / 16) mask units, W = ceil(F / 32) mask words
    float tau, eps;
    long long timeout_ns;
    const __half* x_in;     // [d]
    float* y_out;           // [d]
    __half* x_trace;        // nullable [L-1][d]: normalised inputs of layers 1..L-1
    unsigned long long* epoch;  // [1] barriers completed by earlier launches
    unsigned* counter;          // [1] barrier arrivals (mod 2^32)
    float* xu;                  // [max su*r]
    float* xyp;                 // [G][d]
    float* xy;                  // [d]
    float* xss;                 // [G]
    uint32_t* mask_out;         // [W] mask of the last layer (written by the owners of its pieces)
    int32_t* idx_out;           // [F]
    int32_t* count_out;         // [1]
    float* h_out;               // [F]
    int32_t* layer_counts;      // nullable [L][2]: predicted-active, non-zero FC1 output
    int pred_smem;              // 1: each CTA's predictor slice is bulk-copied to shared memory
    int p1s_bytes, p2s_bytes, b1s_bytes;  // capacities of the shared predictor buffers
    int stage_bytes;            // shared staging region (predictor slices, then this CTA's FC rows)
    int ring_slots;             // without pred_smem: P2 units stream through this many slots of
    int ring_unit;              // ring_unit bytes (16 rows of the largest rank) in the staging region
    int fc_slots;               // FC row slots (one weight row each) in the staging region
    FusedLayer layers[kMaxFusedLayers];
};

// Dynamic smem layout (bytes): x half[d] | u / ustage float[max(rmax, usmax)]
//   | scratch | m16 int[M] | upre int[M+1] | lidx int[cap] | lh float[cap]
//   | P1 slice | P2 slice | bias slice   (the last three only with pred_smem)
// lidx / lh hold this CTA's own active rows from the end of its mask units to
// the end of FC2 (to the end of the step in the last layer, where m16 / upre
// then take the whole mask for the list positions); the P2 ring, idle then,
// spans m16 .. lh together with the staging region.  The u partials are
// staged where u goes: thread i reads entries i, r + i, ... of the staging and
// then writes u[i], which no other thread reads.  The scratch holds FC1's warp
// sums of 128 rows (gated: and of the up rows) and the reduction's float4 sums.
struct SmemPlan {
    int d, rmax, usmax, M, cap, gated;
    int p1s = 0, p2s = 0, b1s = 0;  // shared predictor buffers (bytes, 16-aligned), 0 if unused
    int stage = 0;                  // staging region (bytes, 16-aligned): the predictor buffers
                                    // up to the mask bits, then the ring of this CTA's FC rows
    __host__ __device__ int off_u() const { return ((d * 2 + 15) / 16) * 16; }
    __host__ __device__ int off_ust() const { return off_u(); }
    __host__ __device__ int off_scr() const {
        return ((off_u() + (((rmax > usmax ? rmax : usmax) + 3) / 4) * 16 + 15) / 16) * 16;
    }
    __host__ __device__ int off_m16() const { return off_scr() + (gated ? 8192 : 4096); }
    __host__ __device__ int off_upre() const { return off_m16() + ((M + 1) / 2) * 8; }
    __host__ __device__ int off_lidx() const { return off_upre() + (M + 1) * 4; }
    __host__ __device__ int off_lh() const { return off_lidx() + cap * 4; }
    __host__ __device__ int off_stage() const { return ((off_lh() + cap * 4 + 15) / 16) * 16; }
    __host__ __device__ int off_p1s() const { return off_stage(); }
    __host__ __device__ int off_p2s() const { return off_p1s() + p1s; }
    __host__ __device__ int off_b1s() const { return off_p2s() + p2s; }
    __host__ __device__ int bytes() const { return off_stage() + stage; }
};

// Halving butterfly over a warp: v[b] is this lane's partial sum of row b
// (N = 8 or 4 rows); on return lane L holds the warp's total of row
// fold_row<N>(L) (a fixed order: 9 shuffles for 8 rows, 6 for 4).
template <int N>
PI_DEV int fold_row(int lane) {
    return N == 8 ? ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1)
                  : ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
}
template <int N>
PI_DEV float fold(float (&v)[N], int lane) {
    int o = 16;
#pragma unroll
    for (int n = N / 2; n >= 1; n /= 2, o /= 2) {
        const bool hi = lane & o;
#pragma unroll
        for (int k = 0; k < n; ++k) {
            const float send = hi ? v[k] : v[k + n];
            const float keep = hi ? v[k + n] : v[k];
            v[k] = keep + __shfl_xor_sync(FULL, send, o);
        }
    }
    for (; o >= 1; o /= 2) v[0] += __shfl_xor_sync(FULL, v[0], o);
    return v[0];
}

// Block-wide exclusive scan of one int per thread (kThreads threads).
PI_DEV int block_exscan(int v, int* scr, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) scr[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kWarps ? scr[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(FULL, w, o);
            if (lane >= o) w += t;
        }
        if (lane < kWarps) scr[lane] = w;
    }
    __syncthreads();
    const int base = warp > 0 ? scr[warp - 1] : 0;
    *total = scr[kWarps - 1];
    __syncthreads();
    return base + incl - v;
}

#ifdef PI_PHASE_TRACE
// Phase timestamps of every CTA: [layer][slot][cta] globaltimer ns and clock64.
constexpr int kTraceSlots = 16;
constexpr int kTraceCtas = 256;
__device__ unsigned long long g_pi_trace[96 * kTraceSlots * kTraceCtas];
__device__ unsigned long long g_pi_trace_clk[96 * kTraceSlots * kTraceCtas];
#define PI_STAMP(l, k)                                                              \
    do {                                                                            \
        if (tid == 0) {                                                             \
            g_pi_trace[((l) * kTraceSlots + (k)) * kTraceCtas + c] = globaltimer(); \
            g_pi_trace_clk[((l) * kTraceSlots + (k)) * kTraceCtas + c] = clock64(); \
        }                                                                           \
    } while (0)
#else
#define PI_STAMP(l, k) \
    do {               \
    } while (0)
#endif

// KIND 0: fp16 rows; 1: fp16 gate + up rows; 2: INT4 group-32 rows.
// NCH: kCols-column chunks of d that each thread covers in FC2 (fp16 rows).
// PS: each CTA's predictor slices are staged whole in shared memory (else P2
// streams through the ring of 16-row slots); fixed at compile time, so
// a kernel holds the code of one mode only (measured 3-5 % faster per layer
// than one kernel branching at run time: the code of each phase is fetched
// afresh every layer).
template <int KIND, int NCH, bool PS>
__global__ void __launch_bounds__(kThreads, 1) k_fused_stack(const __grid_constant__ FusedParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int G = gridDim.x, c = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = p.d, F = p.F, M = p.M;
    const long long tmo = p.timeout_ns;
    int rmax = 8, usmax = 8;
    for (int l = 0; l < p.L; ++l) {
        rmax = max(rmax, p.layers[l].r);
        usmax = max(usmax, p.layers[l].r * p.layers[l].su);
    }
    // this CTA's own 8-row pieces: own piece i is global piece piece_of(i)
    const int P = (F + 7) / 8;
    auto piece_of = [&](int i) { return i * G + ((i & 1) ? G - 1 - c : c); };
    const int npc = P / G + (piece_of(P / G) < P ? 1 : 0);
    const int nunits = (npc + 1) / 2;   // unit k = own pieces 2k, 2k+1
    const int cap = 16 * ((P + 2 * G - 1) / (2 * G));
    SmemPlan sp{d, rmax, usmax, M, cap, KIND == 1};
    sp.p1s = PS ? p.p1s_bytes : 0;
    sp.p2s = PS ? p.p2s_bytes : 0;
    sp.b1s = PS ? p.b1s_bytes : 0;
    sp.stage = p.stage_bytes;
    __half* xh = reinterpret_cast<__half*>(smem);   // the layer input, exactly fp16
    float* us = reinterpret_cast<float*>(smem + sp.off_u());
    float* ust = reinterpret_cast<float*>(smem + sp.off_ust());
    uint16_t* m16 = reinterpret_cast<uint16_t*>(smem + sp.off_m16());
    int* upre = reinterpret_cast<int*>(smem + sp.off_upre());
    int* lidx = reinterpret_cast<int*>(smem + sp.off_lidx());
    float* lh = reinterpret_cast<float*>(smem + sp.off_lh());
    float* red = reinterpret_cast<float*>(smem + sp.off_scr());
    int* scr = reinterpret_cast<int*>(smem + sp.off_scr());
    __half* p1s = reinterpret_cast<__half*>(smem + sp.off_p1s());
    __half* p2s = reinterpret_cast<__half*>(smem + sp.off_p2s());
    __half* b1s = reinterpret_cast<__half*>(smem + sp.off_b1s());
    unsigned char* stage = smem + sp.off_stage();
    unsigned char* ring = smem + sp.off_m16();   // P2 ring (phase B; spans m16 .. stage)
    // bytes of one staged weight row: fp16 row, or INT4 codes followed by the scales
    const int wrow = KIND == 2 ? d / 2 + d / 16 : 2 * d;
    const int fc1_rows = KIND == 1 ? 2 : 1;   // gate and up rows when gated
    __shared__ int bad;
    __shared__ float rs_s;
    __shared__ uint16_t ubits[kMaxUnits];   // mask bits of this CTA's units (bit kk = row kk)
    __shared__ int ubase[kMaxUnits];        // list position of each unit's first active row
    __shared__ int nmine_s;
    __shared__ __align__(8) unsigned long long pred_mbar;
    __shared__ __align__(8) unsigned long long fc_full[kMaxFcSlots];   // FC row ring
    __shared__ __align__(8) unsigned long long w1_mbar, w2_mbar;       // FC rows when all fit
    __shared__ __align__(8) unsigned long long ring_full[kRingMax];   // P2 unit ring
    __shared__ int ring_uses[kRingMax];                                // copies issued per slot
    const int ns = p.ring_slots;
    if (tid == 0) {
        bad = 0;
        mbar_init(&pred_mbar, 1);
        for (int q = 0; q < kMaxFcSlots; ++q) mbar_init(&fc_full[q], 1);
        mbar_init(&w1_mbar, 1);
        mbar_init(&w2_mbar, 1);
        for (int q = 0; q < kRingMax; ++q) {
            mbar_init(&ring_full[q], 1);
            ring_uses[q] = 0;
        }
    }
    unsigned fseq = 0;    // ring FC row copies of earlier layers (the ring's running element index)
    unsigned fc_hi = 0;   // ring FC row copies issued so far
    unsigned w12_uses = 0;      // phases armed on w1_mbar / w2_mbar
    bool w12_pending = false;   // ... of which the last is not yet waited for

    // barrier targets: the counter holds G arrivals per barrier ever completed
    const unsigned long long ebase = __ldcg(p.epoch);
    unsigned nbar = 0;
    auto sync = [&]() -> bool {
        ++nbar;
        return grid_sync(p.counter, (unsigned)((ebase + nbar) * (unsigned long long)G), tmo, &bad, [] {});
    };
    auto sync_then = [&](auto between) -> bool {
        ++nbar;
        return grid_sync(p.counter, (unsigned)((ebase + nbar) * (unsigned long long)G), tmo, &bad, between);
    };
    // CTA 0 advances the epoch when it leaves, by every barrier this launch
    // schedules (also after a failure: the counts then no longer matter, the
    // status word reports the failure)
    int inflight = -1;   // layer whose predictor copy is issued but not yet waited for
    auto leave = [&]() {
        if (inflight >= 0) mbar_drain(&pred_mbar, (unsigned)(inflight & 1), kDrainTimeoutNs);
        for (int q = 0; q < ns; ++q)
            if (ring_uses[q] > 0) mbar_drain(&ring_full[q], (unsigned)((ring_uses[q] - 1) & 1), kDrainTimeoutNs);
        if (w12_pending) {
            mbar_drain(&w1_mbar, (w12_uses - 1) & 1u, kDrainTimeoutNs);
            mbar_drain(&w2_mbar, (w12_uses - 1) & 1u, kDrainTimeoutNs);
        }
        // the last copy issued into each FC row slot
        const unsigned S = (unsigned)p.fc_slots;
        for (unsigned g = fc_hi > S ? fc_hi - S : 0u; g < fc_hi; ++g) mbar_drain(&fc_full[g % S], (g / S) & 1u, kDrainTimeoutNs);
        if (c == 0 && tid == 0) {
            const unsigned long long next = ebase + (unsigned long long)kBarriersPerLayer * p.L - 1;
            __stcg(p.epoch, next);
        }
    };

    // This CTA's share of layer l's predictor: P1 items [q0, q1) (item q =
    // row q/su, segment q%su; consecutive items are contiguous in memory) and
    // the P2 rows of its own pieces.
    // (sizes here are far below 2^32 / G, so 32-bit unsigned arithmetic is exact)
    auto item_range = [&](const FusedLayer& ly, int* q0, int* q1) {
        const unsigned items = (unsigned)(ly.r * ly.su);
        *q0 = (int)(items * (unsigned)c / (unsigned)G);
        *q1 = (int)(items * (unsigned)(c + 1) / (unsigned)G);
    };
    // element offset of item q in P1
    auto item_off = [&](const FusedLayer& ly, int q) -> size_t {
        const int i = q / ly.su, sg = q % ly.su;
        return (size_t)i * d + (size_t)sg * ly.seg;
    };
    // warp 0: bulk-copy layer l's predictor slice into shared memory (lane 0
    // arms the mbarrier with the total, then the lanes issue the copies)
    auto issue_predictor = [&](int l) {
        const FusedLayer& ly = p.layers[l];
        int q0, q1;
        item_range(ly, &q0, &q1);
        const size_t e0 = item_off(ly, q0), e1 = q1 < ly.r * ly.su ? item_off(ly, q1) : (size_t)ly.r * d;
        const unsigned b_p1 = (unsigned)(2 * (e1 - e0));
        // own piece i: its rows of P2 at p2s row 8i, its bias (whole pieces only) at b1s[8i]
        unsigned b_p2 = 0, b_b1 = 0;
        for (int i = 0; i < npc; ++i) {
            const int rows = min(8, F - 8 * piece_of(i));
            b_p2 += (unsigned)(2 * ly.r * rows);
            b_b1 += rows == 8 ? 16u : 0u;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (lane == 0) mbar_arrive_expect_tx(&pred_mbar, b_p1 + b_p2 + b_b1);
        __syncwarp();
        if (b_p1 && lane == 0) bulk_g2s(p1s, ly.p1 + e0, b_p1, &pred_mbar);
        for (int i = lane; i < npc; i += 32) {
            const int rb = 8 * piece_of(i);
            const int rows = min(8, F - rb);
            bulk_g2s(p2s + (size_t)8 * i * ly.r, ly.p2 + (size_t)rb * ly.r, (unsigned)(2 * ly.r * rows), &pred_mbar);
            if (rows == 8) bulk_g2s(b1s + 8 * i, ly.b1 + rb, 16u, &pred_mbar);
        }
    };
    // P2 ring (no shared predictor slices): unit k (own pieces 2k, 2k+1, rows
    // 16 apart in the slot) goes to slot k % ns; issued by one thread (the first
    // ns units of a layer by thread 0, later ones by the warp that owns the
    // slot), which counts the slot's uses.
    auto issue_unit = [&](const FusedLayer& ly, int k) {
        const int q = k % ns;
        unsigned bytes = 0;
        for (int h = 0; h < 2 && 2 * k + h < npc; ++h) bytes += (unsigned)(2 * ly.r * min(8, F - 8 * piece_of(2 * k + h)));
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(&ring_full[q], bytes);
        for (int h = 0; h < 2 && 2 * k + h < npc; ++h) {
            const int rb = 8 * piece_of(2 * k + h);
            bulk_g2s(ring + (size_t)q * p.ring_unit + (size_t)16 * h * ly.r, ly.p2 + (size_t)rb * ly.r,
                     (unsigned)(2 * ly.r * min(8, F - rb)), &ring_full[q]);
        }
        ring_uses[q] += 1;
    };
    // uses of slot q in one layer (every layer has the same units)
    auto ring_per_layer = [&](int q) { return nunits > q ? (nunits - 1 - q) / ns + 1 : 0; };
    __syncthreads();
    if (PS) {
        if (warp == 0) issue_predictor(0);
        inflight = 0;
    } else if (tid == 0) {
        for (int k = 0; k < ns && k < nunits; ++k) issue_unit(p.layers[0], k);
    }

    // phase-D columns of this CTA: a contiguous range of 4-column groups
    const int ng4 = d / 4;
    const int g0 = (int)(((long long)ng4 * c) / G), g1 = (int)(((long long)ng4 * (c + 1)) / G);
    const int ngm = g1 - g0;

    for (int l = 0; l < p.L; ++l) {
        const FusedLayer& ly = p.layers[l];
        const int r = ly.r;
        // warp 0, after this CTA's arrival at the barrier that ends FC2 (its FC
        // rows are read by then): bring in layer l+1's predictor slices
        auto issue_next = [&]() {
            if (l + 1 < p.L) {
                if (PS)
                    issue_predictor(l + 1);
                else if (lane == 0)
                    for (int k = 0; k < ns && k < nunits; ++k) issue_unit(p.layers[l + 1], k);
            }
        };
        PI_STAMP(l, 0);

        // ---------------------------------------------------------- phase A
        if (l == 0) {
            for (int i = tid; i < d; i += kThreads) xh[i] = p.x_in[i];
        } else {
            // float4 of y per thread, all requested at once: fp16 rows have
            // d <= NCH * kCols (2 NCH of them); INT4 rows to d = 12288 (wider ones loop)
            constexpr int NY = KIND == 2 ? 12 : 2 * NCH;
            float4 yv[NY];
#pragma unroll
            for (int b = 0; b < NY; ++b) {
                const int i4 = tid + b * kThreads;
                if (i4 < d / 4) yv[b] = ld_cg4(p.xy + i4 * 4);
            }
            if (warp == 0) {
                float s = 0.f;
                for (int q = lane; q < G; q += 32) s += __ldcg(p.xss + q);
                s = warp_sum(s);
                if (lane == 0) rs_s = rsqrtf(s / (float)d + p.eps);
            }
            __syncthreads();
            const float rs = rs_s;
            auto put_x = [&](int i4, const float4& y4) {
                const __half h0 = __float2half_rn(y4.x * rs), h1 = __float2half_rn(y4.y * rs);
                const __half h2 = __float2half_rn(y4.z * rs), h3 = __float2half_rn(y4.w * rs);
                reinterpret_cast<uint2*>(xh)[i4] =
                    make_uint2((uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16),
                               (uint32_t)__half_as_ushort(h2) | ((uint32_t)__half_as_ushort(h3) << 16));
                if (p.x_trace && c == 0) {
                    __half* xt = p.x_trace + (size_t)(l - 1) * d + i4 * 4;
                    xt[0] = h0;
                    xt[1] = h1;
                    xt[2] = h2;
                    xt[3] = h3;
                }
            };
#pragma unroll
            for (int b = 0; b < NY; ++b) {
                const int i4 = tid + b * kThreads;
                if (i4 < d / 4) put_x(i4, yv[b]);
            }
            // columns past the register-prefetched ones
            for (int i4 = tid + NY * kThreads; i4 < d / 4; i4 += kThreads) put_x(i4, ld_cg4(p.xy + i4 * 4));
        }
        __syncthreads();
        PI_STAMP(l, 1);
        {
            // this CTA's items [q0, q1), at most one per warp
            int q0, q1;
            item_range(ly, &q0, &q1);
            if (PS && mbar_wait(&pred_mbar, (unsigned)(l & 1), tmo, &bad)) inflight = -1;
            for (int q = q0 + warp; q < q1; q += kWarps) {
                const int i = q / ly.su, sg = q % ly.su;
                const int c0 = sg * ly.seg, c1 = min(d, c0 + ly.seg);
                const __half* row = PS ? p1s + (item_off(ly, q) - item_off(ly, q0)) - c0
                                                : ly.p1 + (size_t)i * d;
                float acc = 0.f;
                if (PS) {
#pragma unroll 4
                    for (int e = c0 + lane * 8; e < c1; e += 256)
                        acc += dot8hh(*reinterpret_cast<const uint4*>(row + e), *reinterpret_cast<const uint4*>(xh + e));
                } else {
#pragma unroll 8
                    for (int e = c0 + lane * 8; e < c1; e += 256)
                        acc += dot8hh(ld_stream16(row + e), *reinterpret_cast<const uint4*>(xh + e));
                }
                acc = warp_sum(acc);
                if (lane == 0) p.xu[(size_t)sg * r + i] = acc;
            }
        }
        PI_STAMP(l, 8);
        // warp 0, after this CTA's arrival at the barrier that publishes u (HBM
        // is idle while the grid waits): the P2 units the ring reaches right
        // after its prefilled ones are brought into L2
        auto prefetch_next_units = [&]() {
            const int u0 = min(ns, nunits), u1 = min(nunits, u0 + kPrefetchUnits);
            for (int i = 2 * u0; i < min(npc, 2 * u1); ++i) {
                const int rb = 8 * piece_of(i);
                prefetch_lines(ly.p2 + (size_t)rb * ly.r, (size_t)2 * ly.r * min(8, F - rb), lane, 32);
            }
        };
        if (!PS) {
            if (!sync_then(prefetch_next_units)) break;
        } else if (!sync()) break;
        PI_STAMP(l, 2);

        // ---------------------------------------------------------- phase B
        {
            const int nw = r * ly.su;  // multiple of 8: float4 loads
            for (int w4 = tid; w4 < nw / 4; w4 += kThreads)
                reinterpret_cast<float4*>(ust)[w4] = ld_cg4(p.xu + w4 * 4);
            __syncthreads();
            PI_STAMP(l, 9);
            for (int i = tid; i < r; i += kThreads) {
                float acc = 0.f;
                for (int s = 0; s < ly.su; ++s) acc += ust[s * r + i];
                us[i] = acc;
            }
        }
        __syncthreads();
        PI_STAMP(l, 10);
        {
            const int nvec = r / 8;
            const int vpl = (nvec + 31) / 32;
            // this CTA's units: one warp per unit of 16 rows (own pieces 2k and
            // 2k+1, local row kk = 8 * piece + row in piece).  Lane L
            // accumulates, for each of the 16 rows, the products of the row's
            // vectors L, L+32, ... with u; a halving butterfly then leaves the
            // full dot product of row (L >> 1) in lanes L (16 shuffles for 16
            // rows), and one ballot forms the unit's 16 mask bits.
            // With the P2 ring, warp q < ns owns slot q and takes units q, q+ns,
            // ...: each slot's copies are waited for, read and refilled in
            // order by one warp, so a wait never sees an older phase of its slot.
            const int mstep = PS ? kWarps : ns;
            const bool unit_warp = PS || warp < ns;
            for (int m = warp; unit_warp && m < nunits; m += mstep) {
                // first rows of the unit's two pieces (F: no second piece)
                const int pb0 = 8 * piece_of(2 * m);
                const int pb1 = 2 * m + 1 < npc ? 8 * piece_of(2 * m + 1) : F;
                const __half* p2r = nullptr;   // this unit's rows in the ring
                if (!PS) {
                    if (!mbar_wait(&ring_full[warp], (unsigned)((l * ring_per_layer(warp) + m / ns) & 1), tmo, &bad))
                        break;
                    p2r = reinterpret_cast<const __half*>(ring + (size_t)warp * p.ring_unit);
                }
                float v[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) v[k] = 0.f;
                for (int e = 0; e < vpl; ++e) {
                    const int vi = lane + 32 * e;
                    const bool vok = vi < nvec;
                    const int vc = vok ? vi : nvec - 1;   // clamped: loads stay in bounds, result masked
                    float uf[8];
                    {
                        const float4 a = reinterpret_cast<const float4*>(us + vc * 8)[0];
                        const float4 b = reinterpret_cast<const float4*>(us + vc * 8)[1];
                        const float z = vok ? 1.f : 0.f;
                        uf[0] = a.x * z; uf[1] = a.y * z; uf[2] = a.z * z; uf[3] = a.w * z;
                        uf[4] = b.x * z; uf[5] = b.y * z; uf[6] = b.z * z; uf[7] = b.w * z;
                    }
                    // 8 rows' vectors are requested before any arithmetic on them
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint4 w[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            // rows past F (short last piece, missing second piece) read
                            // a row in bounds; their result is never used
                            const int kk = 8 * h + k;
                            w[k] = PS ? *reinterpret_cast<const uint4*>(p2s + (size_t)(16 * m + kk) * r + vc * 8)
                                      : *reinterpret_cast<const uint4*>(p2r + (size_t)kk * r + vc * 8);
                        }
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            float wf[8];
                            h8_to_f8(w[k], wf);
#pragma unroll
                            for (int t = 0; t < 8; ++t) v[8 * h + k] = fmaf(wf[t], uf[t], v[8 * h + k]);
                        }
                    }
                }
                // butterfly: after the step with offset o, a lane keeps the half of
                // its values selected by its bit o and adds the partner's copy
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const bool hi = lane & 16;
                    const float send = hi ? v[k] : v[k + 8];
                    const float keep = hi ? v[k + 8] : v[k];
                    v[k] = keep + __shfl_xor_sync(FULL, send, 16);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const bool hi = lane & 8;
                    const float send = hi ? v[k] : v[k + 4];
                    const float keep = hi ? v[k + 4] : v[k];
                    v[k] = keep + __shfl_xor_sync(FULL, send, 8);
                }
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const bool hi = lane & 4;
                    const float send = hi ? v[k] : v[k + 2];
                    const float keep = hi ? v[k + 2] : v[k];
                    v[k] = keep + __shfl_xor_sync(FULL, send, 4);
                }
                {
                    const bool hi = lane & 2;
                    const float send = hi ? v[0] : v[1];
                    const float keep = hi ? v[1] : v[0];
                    v[0] = keep + __shfl_xor_sync(FULL, send, 2);
                }
                v[0] += __shfl_xor_sync(FULL, v[0], 1);
                // lane L now holds row k = 8*b16 + 4*b8 + 2*b4 + b2 of the unit
                const int k = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
                const int row = (k < 8 ? pb0 : pb1) + (k & 7);
                bool pred = false;
                if (row < F && (lane & 1) == 0) {
                    // staged bias of whole pieces
                    const bool staged = PS && (k < 8 ? pb0 + 8 <= F : pb1 + 8 <= F);
                    const float bk = staged ? __half2float(b1s[16 * m + k]) : __half2float(ly.b1[row]);
                    pred = v[0] + bk > p.tau;
                }
                const unsigned bal = __ballot_sync(FULL, pred);
                // the unit's slot is read: refill it with unit m + ns of this layer
                if (!PS && lane == 0 && m + ns < nunits) issue_unit(ly, m + ns);
                if (lane == 0) {
                    unsigned bits = 0;
                    // the bit of row kk(L) sits at ballot position L (even lanes)
#pragma unroll
                    for (int L2 = 0; L2 < 32; L2 += 2) {
                        const int kk = ((L2 >> 4) & 1) * 8 + ((L2 >> 3) & 1) * 4 + ((L2 >> 2) & 1) * 2 + ((L2 >> 1) & 1);
                        bits |= ((bal >> L2) & 1u) << kk;
                    }
                    ubits[m] = (uint16_t)bits;
                    if (l == p.L - 1) {
                        uint8_t* mb = reinterpret_cast<uint8_t*>(p.mask_out);
                        mb[pb0 / 8] = (uint8_t)(bits & 0xFFu);
                        if (pb1 < F) mb[pb1 / 8] = (uint8_t)(bits >> 8);
                    }
                }
            }
            if (l == p.L - 1 && c == 0) {
                // mask bytes past the last piece
                uint8_t* mb = reinterpret_cast<uint8_t*>(p.mask_out);
                for (int b = P + tid; b < 4 * p.W; b += kThreads) mb[b] = 0;
            }
        }
        __syncthreads();
        PI_STAMP(l, 3);

        if (*(volatile int*)&bad) break;

        // ---------------------------------------------------------- phase B, FFN
        // this CTA's active rows, in unit order (a fixed order: FC2 sums them in
        // it): warp 0 scans the units' counts, then thread (unit m, row kk) places
        // its row, with its FC1 bias when the predictor slice holds it (read
        // before the FC rows overwrite the slice)
        if (warp == 0) {
            int base = 0;
            for (int m0 = 0; m0 < nunits; m0 += 32) {
                const int m = m0 + lane;
                const int cnt = m < nunits ? __popc((unsigned)ubits[m]) : 0;
                int incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int t = __shfl_up_sync(FULL, incl, o);
                    if (lane >= o) incl += t;
                }
                if (m < nunits) ubase[m] = base + incl - cnt;
                base += __shfl_sync(FULL, incl, 31);
            }
            if (lane == 0) nmine_s = base;
        }
        __syncthreads();
        for (int t = tid; t < 16 * nunits; t += kThreads) {
            const int m = t >> 4, kk = t & 15;
            const unsigned bits = ubits[m];
            if ((bits >> kk) & 1u) {
                const int pos = ubase[m] + __popc(bits & ((1u << kk) - 1u));
                const int rb = 8 * piece_of(2 * m + (kk >> 3));
                lidx[pos] = rb + (kk & 7);
                if (PS)
                    lh[pos] = rb + 8 <= F ? __half2float(b1s[16 * m + kk]) : __half2float(ly.b1[rb + (kk & 7)]);
            }
        }
        __syncthreads();
        if (p.layer_counts && tid == 0 && nmine_s) atomicAdd(p.layer_counts + 2 * l, nmine_s);
        const int nmine = nmine_s;
        PI_STAMP(l, 12);
        // FC rows stream through a ring of S row slots in the staging region
        // (which held this layer's predictor slices or P2 ring, read by now):
        // the sequence is this CTA's FC1 rows (gated: gate and up row of each
        // neuron), then its W2t rows; element i lands in slot (fseq + i) % S.
        // Bulk copies run up to S elements ahead; a batch's slots are refilled
        // as soon as the whole CTA has read them.  W2t rows of neurons whose FC1
        // output turns out to be zero are loaded but not used.
        const int S = p.fc_slots;
        const int fc1n = nmine * fc1_rows;
        const int T = fc1n + nmine;
        // all rows fit: element i sits in slot i, the FC1 rows complete on one
        // mbarrier and the W2t rows on another (no per-row waits)
        const bool fits = T <= S;
        auto slot_of = [&](int i) { return fits ? i : (int)((fseq + (unsigned)i) % (unsigned)S); };
        // slot and wait parity of element i, advanced one element at a time (no
        // division per row); take() waits for the element in ring mode (every
        // thread) and returns its row
        struct Cursor {
            int slot;
            unsigned par;
        };
        auto cursor_at = [&](int i) {
            const unsigned g = fits ? (unsigned)i : fseq + (unsigned)i;
            return Cursor{(int)(g % (unsigned)S), (g / (unsigned)S) & 1u};
        };
        auto step = [&](Cursor& cu) {
            if (++cu.slot == S) {
                cu.slot = 0;
                cu.par ^= 1u;
            }
        };
        auto take = [&](Cursor& cu) -> const unsigned char* {
            const unsigned char* r = stage + (size_t)cu.slot * wrow;
            step(cu);
            return r;
        };
        // ring mode: every thread waits for the n elements from cu on (a plain
        // loop of its own, outside the unrolled row loops)
        auto wait_n = [&](Cursor cu, int n) {
            if (fits) return;
            for (int e = 0; e < n; ++e) {
                mbar_wait(&fc_full[cu.slot], cu.par, tmo, &bad);
                step(cu);
            }
        };
        // row copies are spread over the warps (a warp issues its bulk copies one
        // after the other): elements [a, b) go to threads (warp, lane) in the order
        // warp + kWarps * lane
        const int qspread = warp + kWarps * lane;
        auto issue_range = [&](int a, int b) {
            if (a + qspread >= b) return;
            if (!fits) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            for (int i = a + qspread; i < b; i += kThreads) {
                const int sl = slot_of(i);
                unsigned long long* mb = fits ? (i < fc1n ? &w1_mbar : &w2_mbar) : &fc_full[sl];
                unsigned char* dst = stage + (size_t)sl * wrow;
                const size_t k = (size_t)lidx[i < fc1n ? i / fc1_rows : i - fc1n];
                if (!fits) mbar_arrive_expect_tx(mb, (unsigned)wrow);
                if (KIND != 2) {
                    const __half* src = i >= fc1n ? static_cast<const __half*>(ly.w2t)
                                        : (KIND == 1 && (i & 1)) ? ly.wu
                                                                 : static_cast<const __half*>(ly.w1);
                    bulk_g2s(dst, src + k * d, 2u * d, mb);
                } else {
                    const bool w2 = i >= fc1n;
                    const uint8_t* codes = static_cast<const uint8_t*>(w2 ? ly.w2t : ly.w1);
                    const __half* scales = w2 ? ly.w2ts : ly.w1s;
                    bulk_g2s(dst, codes + k * (d / 2), (unsigned)(d / 2), mb);
                    bulk_g2s(dst + d / 2, scales + k * (d / 32), (unsigned)(d / 16), mb);
                }
            }
        };
        int issued = min(S, T);
        if (fits) {
            if (tid == 0 && T > 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive_expect_tx(&w1_mbar, (unsigned)(fc1n * wrow));
                mbar_arrive_expect_tx(&w2_mbar, (unsigned)(nmine * wrow));
            }
            __syncthreads();
            if (T > 0) {
                ++w12_uses;
                w12_pending = true;
            }
        } else {
            fc_hi = fseq + (unsigned)issued;
        }
        // FC1 rows first (spread over the warps on their own, so they are queued first)
        issue_range(0, min(issued, fc1n));
        issue_range(fc1n, issued);
        PI_STAMP(l, 13);
        // after a batch ending at element e has been read by every thread (ring mode)
        auto refill = [&](int e) {
            const int hi = min(T, e + S);
            if (hi > issued) {
                issue_range(issued, hi);
                issued = hi;
                fc_hi = fseq + (unsigned)issued;
            }
        };

        // FC1, the whole CTA on rbn neurons at a time: thread t takes the 8-element
        // words t, t + kThreads, ... of the rows (x read once per word and batch);
        // fold reduces a warp's partials, and the kWarps warp sums of a row are
        // added in a fixed order
        {
            if (!PS)
                for (int q = tid; q < nmine; q += kThreads) lh[q] = __half2float(ly.b1[lidx[q]]);
            float* part = red;           // [128 rows][kWarps]
            float* partu = red + 1024;   // gated: up-projection partials
            const int nwd = d / 8;
            constexpr int RB = KIND == 1 ? 4 : 8;
            const int rbn = max(1, min(RB, S / (2 * fc1_rows)));   // half the slots per batch
            if (fits && nmine > 0 && mbar_wait(&w1_mbar, (w12_uses - 1) & 1u, tmo, &bad)) w12_pending = false;
            PI_STAMP(l, 14);
            Cursor cu = cursor_at(0);
            for (int qb = 0; qb < nmine; qb += 128) {
                const int qe = min(nmine, qb + 128);
                for (int q0 = qb; q0 < qe; q0 += rbn) {
                    const int q1 = min(qe, q0 + rbn);
                    wait_n(cu, (q1 - q0) * fc1_rows);
                    const unsigned char* rw[RB];
                    const unsigned char* ru[RB];
#pragma unroll
                    for (int b = 0; b < RB; ++b) {
                        rw[b] = ru[b] = stage;
                        if (q0 + b < q1) {
                            rw[b] = take(cu);
                            if (KIND == 1) ru[b] = take(cu);
                        }
                    }
                    float v[RB], vu[RB];
#pragma unroll
                    for (int b = 0; b < RB; ++b) v[b] = vu[b] = 0.f;
                    for (int wd = tid; wd < nwd; wd += kThreads) {
                        const uint4 xv = reinterpret_cast<const uint4*>(xh)[wd];
#pragma unroll
                        for (int b = 0; b < RB; ++b) {
                            const int q = q0 + b;
                            if (q >= q1) break;
                            const unsigned char* row = rw[b];
                            if (KIND != 2) {
                                v[b] += dot8hh(reinterpret_cast<const uint4*>(row)[wd], xv);
                                if (KIND == 1) vu[b] += dot8hh(reinterpret_cast<const uint4*>(ru[b])[wd], xv);
                            } else {
                                const uint32_t cw = reinterpret_cast<const uint32_t*>(row)[wd];
                                const float sc = __half2float(reinterpret_cast<const __half*>(row + d / 2)[wd >> 2]);
                                v[b] = fmaf(sc, dotq8h(cw, xv), v[b]);
                            }
                        }
                    }
                    const int rb = fold_row<RB>(lane);
                    const float tv = fold<RB>(v, lane);
                    const float tu = KIND == 1 ? fold<RB>(vu, lane) : 0.f;
                    if ((lane & (32 / RB - 1)) == 0 && q0 + rb < q1) {
                        part[(q0 - qb + rb) * kWarps + warp] = tv;
                        if (KIND == 1) partu[(q0 - qb + rb) * kWarps + warp] = tu;
                    }
                    if (issued < T) {   // the batch's slots are read by every thread: refill them
                        __syncthreads();
                        refill(q1 * fc1_rows);
                    }
                }
                __syncthreads();
                for (int q = qb + tid; q < qe; q += kThreads) {
                    float z = 0.f, zu = 0.f;
#pragma unroll
                    for (int w = 0; w < kWarps; ++w) {
                        z += part[(q - qb) * kWarps + w];
                        if (KIND == 1) zu += partu[(q - qb) * kWarps + w];
                    }
                    z += lh[q];
                    float hv = z > 0.f ? z : 0.f;
                    if (KIND == 1) hv *= zu;
                    lh[q] = hv;
                }
                __syncthreads();
            }
            if (p.layer_counts) {
                int nz = 0;
                for (int q = tid; q < nmine; q += kThreads) nz += lh[q] != 0.f ? 1 : 0;
                nz = __reduce_add_sync(FULL, nz);
                if (lane == 0 && nz) atomicAdd(p.layer_counts + 2 * l + 1, nz);
            }
        }
        PI_STAMP(l, 4);

        // FC2: the whole CTA accumulates its neurons' W2t rows (rb2 rows per
        // batch); rows whose FC1 output is zero are skipped (ReLU removed them)
        if (KIND != 2) {
            constexpr int RB2 = NCH == 1 ? 8 : (NCH == 2 ? 4 : 2);
            const int rb2 = max(1, min(RB2, S / 2));
            float acc[NCH][8];
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[ch][e] = 0.f;
            if (fits && nmine > 0) mbar_wait(&w2_mbar, (w12_uses - 1) & 1u, tmo, &bad);
            PI_STAMP(l, 15);
            Cursor cu = cursor_at(fc1n);
            for (int q0 = 0; q0 < nmine; q0 += rb2) {
                const int q1 = min(nmine, q0 + rb2);
                wait_n(cu, q1 - q0);
                const unsigned char* rr[RB2];
#pragma unroll
                for (int b = 0; b < RB2; ++b) rr[b] = q0 + b < q1 ? take(cu) : stage;
                uint4 wv[RB2][NCH];
                float hv[RB2];
#pragma unroll
                for (int b = 0; b < RB2; ++b) {
                    const int q = q0 + b;
                    const unsigned char* r = rr[b];
                    hv[b] = q < q1 ? lh[q] : 0.f;
                    if (hv[b] != 0.f) {
                        const __half* row = reinterpret_cast<const __half*>(r);
#pragma unroll
                        for (int ch = 0; ch < NCH; ++ch) {
                            const int col = ch * kCols + tid * 8;
                            if (col < d) wv[b][ch] = *reinterpret_cast<const uint4*>(row + col);
                        }
                    }
                }
#pragma unroll
                for (int b = 0; b < RB2; ++b) {
                    if (hv[b] == 0.f) continue;
#pragma unroll
                    for (int ch = 0; ch < NCH; ++ch) {
                        const int col = ch * kCols + tid * 8;
                        if (col < d) {
                            float wf[8];
                            h8_to_f8(wv[b][ch], wf);
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc[ch][e] = fmaf(hv[b], wf[e], acc[ch][e]);
                        }
                    }
                }
                if (issued < T) {
                    __syncthreads();
                    refill(fc1n + q1);
                }
            }
            float* dst = p.xyp + (size_t)c * d;
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
                const int col = ch * kCols + tid * 8;
                if (col < d) {
                    float4* o = reinterpret_cast<float4*>(dst + col);
                    __stcg(o, make_float4(acc[ch][0], acc[ch][1], acc[ch][2], acc[ch][3]));
                    __stcg(o + 1, make_float4(acc[ch][4], acc[ch][5], acc[ch][6], acc[ch][7]));
                }
            }
        } else {
            // INT4: a thread owns scale groups tid and tid + kThreads (32
            // consecutive columns each)
            constexpr int NG = 2;
            const int rb2 = max(1, min(2, S / 2));
            float acc[NG][32];
#pragma unroll
            for (int g = 0; g < NG; ++g)
#pragma unroll
                for (int e = 0; e < 32; ++e) acc[g][e] = 0.f;
            if (fits && nmine > 0) mbar_wait(&w2_mbar, (w12_uses - 1) & 1u, tmo, &bad);
            PI_STAMP(l, 15);
            Cursor cu = cursor_at(fc1n);
            for (int q0 = 0; q0 < nmine; q0 += rb2) {
                const int q1 = min(nmine, q0 + rb2);
                wait_n(cu, q1 - q0);
                const unsigned char* rr[2];
#pragma unroll
                for (int b = 0; b < 2; ++b) rr[b] = q0 + b < q1 ? take(cu) : stage;
                uint4 wv[2][NG];
                float hs[2][NG];
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    const int q = q0 + b;
                    const unsigned char* row = rr[b];
                    const float hv = q < q1 ? lh[q] : 0.f;
#pragma unroll
                    for (int g = 0; g < NG; ++g) {
                        const int col = (tid + g * kThreads) * 32;
                        hs[b][g] = 0.f;
                        if (hv != 0.f && col < d) {
                            wv[b][g] = *reinterpret_cast<const uint4*>(row + col / 2);
                            hs[b][g] = hv * __half2float(reinterpret_cast<const __half*>(row + d / 2)[col / 32]);
                        }
                    }
                }
#pragma unroll
                for (int b = 0; b < 2; ++b)
#pragma unroll
                    for (int g = 0; g < NG; ++g) {
                        if (hs[b][g] == 0.f) continue;
                        const uint32_t qw[4] = {wv[b][g].x, wv[b][g].y, wv[b][g].z, wv[b][g].w};
#pragma unroll
                        for (int wi = 0; wi < 4; ++wi) {
                            float qf[8];
                            q8_to_f8(qw[wi], qf);
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc[g][wi * 8 + e] = fmaf(hs[b][g], qf[e], acc[g][wi * 8 + e]);
                        }
                    }
                if (issued < T) {
                    __syncthreads();
                    refill(fc1n + q1);
                }
            }
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                const int col = (tid + g * kThreads) * 32;
                if (col < d) {
                    float4* o = reinterpret_cast<float4*>(p.xyp + (size_t)c * d + col);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        __stcg(o + e, make_float4(acc[g][4 * e], acc[g][4 * e + 1], acc[g][4 * e + 2], acc[g][4 * e + 3]));
                }
            }
        }
        if (!fits) fseq += (unsigned)T;
        // (both FC mbarriers of the fitting case are waited for by every thread by now)
        if (!*(volatile int*)&bad) w12_pending = false;
        PI_STAMP(l, 5);
        if (l + 1 < p.L && PS) inflight = l + 1;
        if (!sync_then(issue_next)) break;
        PI_STAMP(l, 6);

        // ---------------------------------------------------------- phase D
        {
            // this CTA's ngm 4-column groups, gpw = 32 / lpg at a time: the lpg
            // lanes of a group in warp w add the partial rows q = lpg w + sub,
            // + lpg kWarps, ... (a warp's loads of one row are consecutive 16-byte
            // words), every load of a lane in flight at once (lpg grows when a
            // CTA has few groups, so the rows per lane stay few); the lanes of a
            // group are then combined by a fixed xor order, the warps' sums in
            // warp order, and b2 added last
            float4* red4 = reinterpret_cast<float4*>(red);   // [kWarps][gpw]
            const int lpg = ngm <= 16 ? 2 : 1;
            const int gpw = 32 / lpg;
            float ss_local = 0.f;   // warp 0, lane L < gpw: squares of its groups, in chunk order
            // with at most one group per warp, a warp takes a group with its lanes
            // over all G partial rows (one round of loads, a fixed xor-tree)
            if (ngm <= kWarps) {
                if (warp < ngm) {
                    const int col = (g0 + warp) * 4;
                    __half b2v[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) b2v[e] = lane == 0 ? __ldg(ly.b2 + col + e) : __float2half(0.f);
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    constexpr int NB = 5;   // one round for up to 160 partial rows
                    for (int q0 = lane; q0 < G; q0 += NB * 32) {
                        float4 v[NB];
#pragma unroll
                        for (int b = 0; b < NB; ++b) {
                            const int q = q0 + b * 32;
                            if (q < G) v[b] = ld_cg4(p.xyp + (size_t)q * d + col);
                        }
#pragma unroll
                        for (int b = 0; b < NB; ++b) {
                            const int q = q0 + b * 32;
                            if (q < G) {
                                acc.x += v[b].x;
                                acc.y += v[b].y;
                                acc.z += v[b].z;
                                acc.w += v[b].w;
                            }
                        }
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        acc.x += __shfl_xor_sync(FULL, acc.x, o);
                        acc.y += __shfl_xor_sync(FULL, acc.y, o);
                        acc.z += __shfl_xor_sync(FULL, acc.z, o);
                        acc.w += __shfl_xor_sync(FULL, acc.w, o);
                    }
                    if (lane == 0) {
                        const float4 yv = make_float4(acc.x + __half2float(b2v[0]), acc.y + __half2float(b2v[1]),
                                                      acc.z + __half2float(b2v[2]), acc.w + __half2float(b2v[3]));
                        __stcg(reinterpret_cast<float4*>(p.xy + col), yv);
                        if (l == p.L - 1) *reinterpret_cast<float4*>(p.y_out + col) = yv;
                        red[kWarps * 32 + warp] = yv.x * yv.x + yv.y * yv.y + yv.z * yv.z + yv.w * yv.w;
                    }
                }
                __syncthreads();
                if (warp == 0 && lane < ngm) ss_local = red[kWarps * 32 + lane];
            }
            for (int gc = 0; gc < ngm && ngm > kWarps; gc += gpw) {
                const int gl = lane / lpg, sub = lane % lpg;
                const bool ok = gc + gl < ngm;
                const int col = (g0 + (ok ? gc + gl : gc)) * 4;
                // b2 of the group that lane L of warp 0 finishes, requested before the partials
                const bool fin = warp == 0 && lane < gpw && gc + lane < ngm;
                const int fcol = (g0 + gc + (fin ? lane : 0)) * 4;
                __half b2v[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) b2v[e] = fin ? __ldg(ly.b2 + fcol + e) : __float2half(0.f);
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                constexpr int QB = 10;
                const int qstep = kWarps * lpg;
                for (int q0 = warp * lpg + sub; q0 < G; q0 += QB * qstep) {
                    float4 v[QB];
#pragma unroll
                    for (int b = 0; b < QB; ++b) {
                        const int q = q0 + b * qstep;
                        if (ok && q < G) v[b] = ld_cg4(p.xyp + (size_t)q * d + col);
                    }
#pragma unroll
                    for (int b = 0; b < QB; ++b) {
                        const int q = q0 + b * qstep;
                        if (ok && q < G) {
                            acc.x += v[b].x;
                            acc.y += v[b].y;
                            acc.z += v[b].z;
                            acc.w += v[b].w;
                        }
                    }
                }
                for (int o = 1; o < lpg; o <<= 1) {
                    acc.x += __shfl_xor_sync(FULL, acc.x, o);
                    acc.y += __shfl_xor_sync(FULL, acc.y, o);
                    acc.z += __shfl_xor_sync(FULL, acc.z, o);
                    acc.w += __shfl_xor_sync(FULL, acc.w, o);
                }
                if (sub == 0) red4[warp * gpw + gl] = acc;
                __syncthreads();
                if (fin) {
                    float4 yv = red4[lane];
                    for (int w = 1; w < kWarps; ++w) {
                        const float4 t = red4[w * gpw + lane];
                        yv.x += t.x;
                        yv.y += t.y;
                        yv.z += t.z;
                        yv.w += t.w;
                    }
                    yv.x += __half2float(b2v[0]);
                    yv.y += __half2float(b2v[1]);
                    yv.z += __half2float(b2v[2]);
                    yv.w += __half2float(b2v[3]);
                    __stcg(reinterpret_cast<float4*>(p.xy + fcol), yv);
                    if (l == p.L - 1) *reinterpret_cast<float4*>(p.y_out + fcol) = yv;
                    ss_local += yv.x * yv.x + yv.y * yv.y + yv.z * yv.z + yv.w * yv.w;
                }
                __syncthreads();   // red4 is reused by the next chunk
            }
            if (l + 1 < p.L && warp == 0) {
                // fixed-order sum of squares of this CTA's columns
                const float t = warp_sum(ss_local);
                if (lane == 0) __stcg(p.xss + c, t);
            }
        }
        PI_STAMP(l, 7);
        // the next layer's input needs every CTA's columns of y; after the last
        // layer the end of the grid publishes them
        if (l + 1 < p.L && !sync()) break;
    }
    // (a failure anywhere left the loop early with bad set; the code of the
    // last layer's list and of the exit stays out of the layer loop)
    __syncthreads();
    if (!*(volatile int*)&bad) {
        // the active list of the last layer in storage order: every CTA scans the
        // whole mask (complete since the last barrier) and places its own rows
        for (int w = tid; w < p.W; w += kThreads) reinterpret_cast<uint32_t*>(m16)[w] = __ldcg(p.mask_out + w);
        __syncthreads();
        const int per = (M + kThreads - 1) / kThreads;
        int cnt = 0;
        for (int e = 0; e < per; ++e) {
            const int m = tid * per + e;
            if (m < M) cnt += __popc((unsigned)m16[m]);
        }
        int total;
        int run = block_exscan(cnt, scr, &total);
        for (int e = 0; e < per; ++e) {
            const int m = tid * per + e;
            if (m < M) {
                upre[m] = run;
                run += __popc((unsigned)m16[m]);
            }
        }
        __syncthreads();
        const int nmine = nmine_s;
        for (int q = tid; q < nmine; q += kThreads) {
            const int k = lidx[q];
            const int pos = upre[k >> 4] + __popc((unsigned)m16[k >> 4] & ((1u << (k & 15)) - 1u));
            p.idx_out[pos] = k;
            p.h_out[pos] = lh[q];
        }
        if (c == 0 && tid == 0) *p.count_out = total;
    }
    leave();
}

// A wait on a counter nothing increments: exercises the bounded-wait path.
__device__ unsigned g_never_incremented = 0u;

__global__ void k_wait_nothing(long long timeout_ns) {
    __shared__ int bad;
    if (threadIdx.x == 0) bad = 0;
    // target 2 with one arrival: the count never gets there
    (void)grid_sync(&g_never_incremented, g_never_incremented + 2u, timeout_ns, &bad, [] {});
    if (threadIdx.x == 0) atomicSub(&g_never_incremented, 1u);
}

// ------------------------------------------------------------------ host side

namespace {

template <int KIND, int NCH>
cudaError_t launch_kind(const FusedParams& prm, int G, size_t smem, cudaStream_t s) {
    auto kern = prm.pred_smem ? k_fused_stack<KIND, NCH, true> : k_fused_stack<KIND, NCH, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, prm);
}

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

// own units (two 8-row pieces) of a CTA at most
int max_units(int F, int G) { return ((F + 7) / 8 + 2 * G - 1) / (2 * G); }

// exchange region: epoch | counter | xu | xyp | xy | xss
struct XchgLayout {
    size_t counter, xu, xyp, xy, xss, total;
    XchgLayout(int d, int F, size_t rmax_su, int G) {
        size_t off = 256;
        counter = off;
        off += 256;
        xu = off;
        off += up256(4ull * rmax_su);
        xyp = off;
        off += up256(4ull * (size_t)G * d);
        xy = off;
        off += up256(4ull * d);
        xss = off;
        off += up256(4ull * G);
        total = off;
    }
};

SmemPlan smem_plan(int d, int F, int rmax, size_t rmax_su, int G, bool gated) {
    return SmemPlan{d, rmax < 8 ? 8 : rmax, (int)rmax_su, (F + 15) / 16, 16 * max_units(F, G), gated};
}

}  // namespace

size_t fused_workspace_bytes(int d, int F, size_t rmax_su, int G) { return XchgLayout(d, F, rmax_su, G).total; }

// FC row slots of the staging region: at least two batches of one neuron's rows
int fc_slots_for(int d, bool int4, int stage_bytes) {
    const int wrow = int4 ? d / 2 + d / 16 : 2 * d;
    const int n = stage_bytes / wrow;
    return n < kMaxFcSlots ? n : kMaxFcSlots;
}

bool fused_supported(int d, int F, int rmax, bool int4, bool gated, int G) {
    if (d % 8 != 0 || G < 1) return false;
    if (int4 && d % 256 != 0) return false;                  // 16-byte bulk copies of the scale rows
    if (!int4 && d > 4 * kCols) return false;              // FC2: 8 columns per thread and chunk
    if (int4 && (d % 32 != 0 || d > 64 * kThreads)) return false;  // FC2: two groups per thread
    if (max_units(F, G) > kMaxUnits) return false;
    const size_t rmax_su = (size_t)16 * G + 2 * (size_t)rmax;
    const SmemPlan sp = smem_plan(d, F, rmax, rmax_su, G, gated);
    const long long room = 227ll * 1024 - 1024 - sp.off_stage();
    if (room <= 0) return false;
    return fc_slots_for(d, int4, (int)(room / 16 * 16)) >= (gated ? 4 : 2);
}

// Work split and shared-memory plan of one stack step (no pointers needed:
// the layers' ranks and the shapes decide it).  Returns false if the stack
// cannot run on the fused kernel.
static bool plan_fused(const FusedStackArgs& a, FusedParams* out, size_t* smem_out) {
    if (a.L < 1 || a.L > kMaxFusedLayers || max_units(a.F, a.G) > kMaxUnits) return false;
    FusedParams& prm = *out;
    const int G = a.G;
    prm.L = a.L;
    prm.d = a.d;
    prm.F = a.F;
    prm.M = (a.F + 15) / 16;
    prm.W = (a.F + 31) / 32;
    int rmax = 8;
    for (int l = 0; l < a.L; ++l) {
        FusedLayer& f = prm.layers[l];
        f.r = a.ranks[l];
        // at most one (row, split) item per warp of the grid; splits >= 256 elements
        int su = (kWarps * G) / f.r;
        const int max_su = (a.d + 255) / 256;
        if (su > max_su) su = max_su;
        if (su < 1) su = 1;
        f.seg = ((a.d / 8 + su - 1) / su) * 8;
        f.su = (a.d + f.seg - 1) / f.seg;
        if ((size_t)f.su * f.r > a.rmax_su) return false;
        rmax = f.r > rmax ? f.r : rmax;
    }
    // the u-partial staging buffer as the kernel sizes it: the largest r * su
    size_t usmax = 8;
    for (int l = 0; l < a.L; ++l) usmax = std::max(usmax, (size_t)prm.layers[l].r * prm.layers[l].su);
    SmemPlan sp = smem_plan(a.d, a.F, rmax, usmax, G, a.gated);
    // shared predictor slices when they fit: P1 items, P2 units and bias of one CTA
    {
        size_t p1b = 16;
        for (int l = 0; l < a.L; ++l) {
            const FusedLayer& f = prm.layers[l];
            const size_t items = (size_t)f.r * f.su;
            p1b = std::max(p1b, ((items + G - 1) / G) * (size_t)f.seg * 2);
        }
        const size_t units = (size_t)max_units(a.F, G);
        const size_t p2b = units * 16 * (size_t)rmax * 2, b1b = units * 16 * 2;
        auto r16 = [](size_t v) { return (int)((v + 15) / 16 * 16); };
        SmemPlan with = sp;
        with.p1s = r16(p1b);
        with.p2s = r16(p2b);
        with.b1s = r16(b1b);
        if ((size_t)with.off_stage() + with.p1s + with.p2s + with.b1s <= 227 * 1024 - 1024) {
            sp = with;
            prm.pred_smem = 1;
            prm.p1s_bytes = with.p1s;
            prm.p2s_bytes = with.p2s;
            prm.b1s_bytes = with.b1s;
        }
    }
    // the staging region takes the rest of shared memory (leaving room for the
    // kernel's static shared variables); it must at least hold the predictor slices
    {
        const int pred = sp.p1s + sp.p2s + sp.b1s;
        const long long room = 227ll * 1024 - 1024 - sp.off_stage();
        const int st = (int)(room / 16 * 16);
        sp.stage = st > pred ? st : pred;
        prm.stage_bytes = sp.stage;
        prm.fc_slots = fc_slots_for(a.d, a.int4, sp.stage);
        if (prm.fc_slots < (a.gated ? 4 : 2)) return false;
        // predictor slices too large for shared memory: stream P2 in 16-row units
        // through the mask/list buffers and the staging region
        const int unit = 16 * rmax * 2;
        const int slots = prm.stage_bytes > 0 ? (prm.stage_bytes + sp.off_stage() - sp.off_m16()) / unit : 0;
        if (!prm.pred_smem) {
            if (slots < 2) return false;   // neither fits: the per-step kernels run the stack
            prm.ring_slots = slots < kRingMax ? slots : kRingMax;
            prm.ring_unit = unit;
        }
    }
    const size_t smem = sp.bytes();
    if (smem > 227 * 1024) return false;
    *smem_out = smem;
    return true;
}

bool fused_stack_config(const FusedStackArgs& a, FusedStackConfig* out) {
    FusedParams prm = {};
    size_t smem = 0;
    if (!plan_fused(a, &prm, &smem)) return false;
    out->pred_smem = prm.pred_smem;
    out->ring_slots = prm.ring_slots;
    out->fc_slots = prm.fc_slots;
    out->smem_bytes = (int)smem;
    return true;
}

cudaError_t launch_fused(const FusedStackArgs& a, cudaStream_t s) {
    FusedParams prm = {};
    size_t smem = 0;
    if (!plan_fused(a, &prm, &smem)) return cudaErrorInvalidValue;
    const int G = a.G;
    prm.tau = a.tau;
    prm.eps = a.eps;
    prm.timeout_ns = a.timeout_ns;
    prm.x_in = a.x_in;
    prm.y_out = a.y_out;
    prm.x_trace = a.x_trace;
    const XchgLayout xl(a.d, a.F, a.rmax_su, G);
    char* ws = static_cast<char*>(a.xchg);
    prm.epoch = reinterpret_cast<unsigned long long*>(ws);
    prm.counter = reinterpret_cast<unsigned*>(ws + xl.counter);
    prm.xu = reinterpret_cast<float*>(ws + xl.xu);
    prm.xyp = reinterpret_cast<float*>(ws + xl.xyp);
    prm.xy = reinterpret_cast<float*>(ws + xl.xy);
    prm.xss = reinterpret_cast<float*>(ws + xl.xss);
    prm.mask_out = a.mask_out;
    prm.idx_out = a.idx_out;
    prm.count_out = a.count_out;
    prm.h_out = a.h_out;
    prm.layer_counts = a.layer_counts;
    for (int l = 0; l < a.L; ++l) {
        const LayerPtrs& w = a.layers[l];
        FusedLayer& f = prm.layers[l];
        f.w1 = w.w1;
        f.w1s = w.w1s;
        f.b1 = w.b1;
        f.wu = w.wu;
        f.w2t = w.w2t;
        f.w2ts = w.w2ts;
        f.b2 = w.b2;
        f.p1 = w.p1;
        f.p2 = w.p2;
    }
    if (a.int4) return launch_kind<2, 4>(prm, G, smem, s);
    const int nch = (a.d + kCols - 1) / kCols;
    if (a.gated) {
        if (nch == 1) return launch_kind<1, 1>(prm, G, smem, s);
        if (nch == 2) return launch_kind<1, 2>(prm, G, smem, s);
        return launch_kind<1, 4>(prm, G, smem, s);
    }
    if (nch == 1) return launch_kind<0, 1>(prm, G, smem, s);
    if (nch == 2) return launch_kind<0, 2>(prm, G, smem, s);
    return launch_kind<0, 4>(prm, G, smem, s);
}

cudaError_t launch_wait_nothing(long long timeout_ns, cudaStream_t s) {
    k_wait_nothing<<<1, 32, 0, s>>>(timeout_ns);
    return cudaGetLastError();
}

int* status_word() {
    static std::mutex mu;
    static int* cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_pi_status) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<int*>(ptr);
    }
    return cache[dev];
}

cudaError_t read_and_clear_status(int* out, cudaStream_t s) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_pi_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    *out = v;
    if (v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_pi_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

}  // namespace pi

#ifdef PI_PHASE_TRACE
extern "C" __attribute__((visibility("default"))) int pi_debug_read_trace(unsigned long long* host,
                                                                          unsigned long long* clk, int n) {
    if (n > 96 * pi::kTraceSlots * pi::kTraceCtas) n = 96 * pi::kTraceSlots * pi::kTraceCtas;
    if (cudaMemcpyFromSymbol(host, pi::g_pi_trace, sizeof(unsigned long long) * n) != cudaSuccess) return -1;
    if (cudaMemcpyFromSymbol(clk, pi::g_pi_trace_clk, sizeof(unsigned long long) * n) != cudaSuccess) return -1;
    return n;
}
#endif
