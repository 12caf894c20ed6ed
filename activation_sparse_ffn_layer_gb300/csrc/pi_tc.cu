// pi_tc.cu -- the batched union path on the tcgen05 tensor cores (batch 16..32,
// fp16 weights, and the FC1 of INT4 weights).
//
// At batch B the union of the B tokens' predicted neurons is gathered once and
// both FFN products become dense contractions over the gathered rows
// (PowerInfer summary (CSDN), section "Neuron-aware operator": only the rows
// and columns of active neurons are processed; section "Background": a neuron
// is a row of W1 and a column of W2, stored here as a row of W2t):
//
//   FC1   Z[j, t] = sum_k W1[idx_j, k] x[t, k]        M = 128 listed neurons,
//                                                      N = tokens, K = d
//   FC2   y[t, c] = sum_j h[j, t] W2t[idx_j, c]       M = 128 columns of y,
//                                                      N = tokens (hi | lo), K = j
//
// One CTA per SM, three warp roles:
//   warps 0-3  load: cp.async 16-byte copies of the gathered rows straight into
//              the tensor cores' shared-memory operand layouts (A tiles with
//              the 128-byte swizzle, B as 8 x 16-byte core matrices), a ring
//              of stages; for INT4 rows they also convert the codes to fp16
//              and store the A operand into tensor memory (tcgen05.st);
//   warp  8    one thread issues tcgen05.mma (fp16 x fp16 -> fp32 in TMEM);
//   warps 4-7  drain the TMEM accumulators (tcgen05.ld) and apply the epilogue.
// Ring slots are handed over with mbarriers: loaders arrive on `full` after
// their copies landed; tcgen05.commit arrives on `empty` when the MMAs that
// read a slot are done.  Two accumulator buffers let the epilogue of one tile
// overlap the MMAs of the next.  Every wait is bounded: on expiry the status
// word becomes PI_ERR_TIMEOUT, the CTA drains its own copies and MMAs, frees
// its tensor memory and returns.
//
// FC1 work split: the (128-row tile x K-chunk) space is cut into equal
// contiguous ranges per CTA ("stream-K"; INT4 in quads of four K-chunks), so
// every SM streams the same bytes; a finish kernel adds the partial tiles.
// FC2 work split: the (column tile x union row) space is cut into equal
// contiguous ranges per CTA ("stream-K"); each CTA writes one partial tile per
// column tile it touches and a fixed-order reduction adds the partials to b2.
//
// FC2 feeds h to the tensor cores as two fp16 halves, hi = fp16(h) and
// lo = fp16(h - hi), placed as extra N columns: hi + lo carries 22 bits of h,
// so the product keeps fp32-level accuracy.  Weights and x are fp16 already,
// and fp16 x fp16 products are exact in the fp32 accumulator.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "pi_common.cuh"
#include "pi_internal.h"
#include "pi_pipe.cuh"

namespace pi {
namespace {

using namespace pipe;

constexpr int kTcThreads = 288;      // warps 0-3 load, 4-7 epilogue, 8 MMA
constexpr int kLoaders = 128;
constexpr int kRingBudget = 220 * 1024;
constexpr int kTileA = 16384;        // 128 x 64 fp16 operand tile

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
// Same for the 128-byte-swizzled K-major layout: rows of 128 bytes (64 fp16
// of K), 8-row atoms of 1024 bytes (1024-byte aligned), 16-byte chunk c of row
// r stored at chunk position c ^ (r % 8); K-steps advance the start by 32 bytes.
PI_DEV uint64_t sdesc_sw128(unsigned addr) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// 128-byte-swizzled MN-major layout (the W2t tile of FC2): atoms of 8 K-rows x
// 64 MN-elements (1024 bytes, 1024-byte aligned), 16-byte chunk c of row k at
// position c ^ (k % 8); lbo = bytes between atoms adjacent in MN, sbo = bytes
// between 8-row groups adjacent in K.
PI_DEV uint64_t sdesc_sw128_mn(unsigned addr, unsigned lbo, unsigned sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
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
// Same with the A operand in tensor memory (row m of A in lane m, two fp16
// per 32-bit column along K)
PI_DEV void mma_f16_ta(unsigned tmem_d, unsigned tmem_a, uint64_t b, unsigned idesc, unsigned accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
// 2-D tiled TMA load of the box at (x = inner element, y = row) into shared
// memory, completing on the barrier (the tensor map carries shape, box and swizzle)
PI_DEV void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, unsigned long long* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            su32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(su32(bar))
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
// 32 consecutive 32-bit columns of this thread's TMEM lane
PI_DEV void tmem_st32(unsigned taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
PI_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

constexpr int kLoaderWarps = kLoaders / 32;   // arrivals on a stage's `full` barrier

PI_DEV void tmem_alloc(unsigned* slot, unsigned cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(slot)), "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
PI_DEV void tmem_free(unsigned base, unsigned cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols) : "memory");
}

constexpr int tmem_cols_for(int c) { return c <= 32 ? 32 : c <= 64 ? 64 : c <= 128 ? 128 : c <= 256 ? 256 : 512; }

// ------------------------------------------------- row-tile GEMMs (FC1, predictor)
//
// D[m, t] = sum_k A[row(m), k] Bop[t, k] over 128-row tiles of A (rows
// gathered through idx, or contiguous), K in chunks of 64, N = tokens.
//   MODE 0  FC1            A = W1 rows (gathered),          Bop = x
//   MODE 1  FC1 gated      A = Wg and Wu rows (gathered),   Bop = x
//   MODE 2  predictor u    A = P1 rows,                     Bop = x
//   MODE 3  predictor s    A = P2 rows,                     Bop = u (hi | lo fp16)
//   MODE 4  FC1, INT4 rows A = W1 codes as exact fp16 integers, Bop = x;
//                          each group of 32 along K has its own TMEM
//                          accumulator, which the epilogue scales by the
//                          row's group scale and adds up in registers
// Modes 0-2 split the (tile x K-chunk) space evenly over the CTAs and write
// one partial tile per tile touched; a finish kernel adds the partials of each
// tile in ascending CTA order and applies the epilogue.  Mode 3 has short K
// (the rank) and many tiles: each CTA takes whole tiles and thresholds s in
// its own epilogue (mask bits by warp ballot: a warp's 32 TMEM lanes are the
// 32 rows of one mask word).

template <int MODE, int NT>
struct RowsCfg {
    static constexpr bool Q4 = MODE == 4;
    static constexpr bool GATHER = MODE <= 1 || Q4;
    static constexpr bool DIRECT = MODE == 3;
    static constexpr int NA = MODE == 1 ? 2 : 1;            // A operand tiles per stage
    static constexpr int NACC = MODE == 1 ? 2 : 1;          // accumulators (gate and up)
    static constexpr int NB = DIRECT ? 2 * NT : NT;          // B operand rows
    static constexpr int X = NB * 128;                       // NB rows x 64 fp16
    static constexpr int STAGE = Q4 ? 0 : NA * kTileA + X;   // INT4: A in TMEM, x read from the raw ring
    // even ring of stages, filled two K-chunks at a time (256 contiguous bytes
    // of every row per visit); LAGP pairs of copies stay in flight.  INT4: 8
    // A stages in TMEM (32 columns each), fed from a ring of RQ raw quads in
    // shared memory (per row 128 bytes of codes at a 144-byte pitch, then the
    // quad's x, which the MMAs read in place)
    static constexpr int S0 = Q4 ? 0 : kRingBudget / STAGE > 12 ? 12 : kRingBudget / STAGE;
    static constexpr int S = Q4 ? 8 : S0 & ~1;
    static constexpr int LAGP = S / 2 >= 4 ? S / 2 - 2 : S / 2 - 1;
    static constexpr int KQ = Q4 ? 4 : 1;                    // K-chunks per unit of the split
    static constexpr int RAWQ = 128 * 144 + 4 * X;
    static constexpr int RQ0 = Q4 ? (kRingBudget - S * STAGE) / RAWQ : 0;
    static constexpr int RQ = RQ0 > 8 ? 8 : RQ0;
    static constexpr int CS = Q4 ? 4 : 1;                    // INT4: TMEM accumulator slots, 2 groups of 32 each
    static constexpr int ACOL = 2 * CS * NB;                 // INT4: first TMEM column of the S A stages (32 each)
    static constexpr int ACC = NACC * NB;                    // TMEM columns per accumulator buffer
    static constexpr int COLS = NACC * NT;                   // partial columns (modes 0-2, 4)
    static constexpr int TMEM = tmem_cols_for(Q4 ? ACOL + 32 * S : 2 * ACC);
    static constexpr size_t SMEM = (size_t)S * STAGE + (size_t)RQ * RAWQ + 1024;
    static_assert(!Q4 || RQ >= 2 + S / 4, "INT4 raw ring too shallow");
    static_assert(!Q4 || S >= CS, "INT4: a stage barrier must not run a phase ahead of the epilogue");
};

struct TcRowsArgs {
    CUtensorMap tma_a;     // modes 2-3 with use_tma: A rows [R][K] fp16, box 64 x 128, 128-byte swizzle
    CUtensorMap tma_b;     // ... and the B operand rows [bop_rows][K], box 64 x NB
    int use_tma;           // 1: one thread loads A and B tiles by TMA (contiguous A rows)
    const __half* a0;      // A rows (row length K)
    const __half* a1;      // up-projection rows (gated FC1)
    const uint8_t* q;      // mode 4: W1 codes [F][K/2]
    const __half* qs;      // mode 4: W1 group scales [F][K/32]
    const int32_t* idx;    // gathered row ids (FC1)
    const int32_t* count;  // device row count (FC1), else R rows
    int R;
    const __half* bop;     // B operand rows [bop_rows][K] fp16
    int bop_rows;
    int K, B;
    float* part;           // modes 0-2: [G][slots][COLS][128]
    int slots;
    const __half* bias;    // mode 3: s threshold
    float tau;
    uint32_t* mask;        // mode 3: [B][W]
    int W;
    int* status;
    long long timeout_ns;
};

// cp.async.wait_group with a count known only at run time (0 .. 11)
PI_DEV void cp_wait_n(int n) {
    switch (n) {
        case 0: cp_wait<0>(); break;
        case 1: cp_wait<1>(); break;
        case 2: cp_wait<2>(); break;
        case 3: cp_wait<3>(); break;
        case 4: cp_wait<4>(); break;
        case 5: cp_wait<5>(); break;
        case 6: cp_wait<6>(); break;
        case 7: cp_wait<7>(); break;
        case 8: cp_wait<8>(); break;
        case 9: cp_wait<9>(); break;
        case 10: cp_wait<10>(); break;
        default: cp_wait<11>(); break;
    }
}

// 8 INT4 codes (element e in bits 4e..4e+3, two's complement) as 8 fp16
// integers in element order, three operations per pair: byte b of w (elements
// 2b and 2b+1, sign-flipped to n = q + 8) is spread to both halves, the low
// half keeps bits 0-3 and the high half bits 4-7 under the fp16 pattern of
// 1024, giving 1024 + n and 1024 + 16 n; one fp16 fma with (1, 1/16) and
// (-1032, -72) returns q for both, exactly (every intermediate is an fp16
// integer or a multiple of 1/16 below 128).
PI_DEV uint4 q8_f16(uint32_t w) {
    const uint32_t u = w ^ 0x88888888u;
    const uint32_t scale = 0x2C003C00u;   // (1, 1/16)
    const uint32_t offset = 0xD480E408u;  // (-1032, -72)
    uint32_t r[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        uint32_t t = (__byte_perm(u, 0u, 0x1111u * (unsigned)b) & 0x00F0000Fu) | 0x64006400u;
        const __half2 q = __hfma2(*reinterpret_cast<const __half2*>(&t), *reinterpret_cast<const __half2*>(&scale),
                                  *reinterpret_cast<const __half2*>(&offset));
        r[b] = *reinterpret_cast<const uint32_t*>(&q);
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// Loaders of the INT4 FC1 (mode 4).  The CTA's K range is split in quads of
// four K-chunks.  A quad of a 128-row tile is copied by all 128 loaders with
// cp.async into a raw ring entry, RQ-2 quads ahead: per row the 128 contiguous
// bytes of codes (eight lanes per row, so a warp instruction reads four rows'
// runs) at a 144-byte pitch, then the quad's x in the B-tile layout, which the
// MMAs read in place.  For each chunk of the current quad, once the stage is
// free, loader t writes row t's 64 codes as fp16 into TMEM lane t of the
// stage's A columns (tcgen05.st, so shared memory carries only the raw copies
// and x) and arrives on `full`.  A barrier per quad makes every
// loader's copies visible; an entry is refilled only after the MMAs of its
// previous quad have completed (the stage waits of the quad after it).
template <typename C, typename SpanOf>
PI_DEV void q4_loader(const TcRowsArgs& a, unsigned char* ring, const SpanOf& span, int npiece, int R,
                      const int* srow, unsigned tmem, unsigned long long* full, unsigned long long* empty,
                      const Ctl& ctl) {
    static_assert(C::S % 4 == 0, "stages must be a multiple of a quad");
    const int t = threadIdx.x;
    unsigned char* raw = ring + (size_t)C::S * C::STAGE;
    const size_t cpr = (size_t)a.K / 2;   // code bytes per row
    int nquad = 0;
    for (int p = 0; p < npiece; ++p) {
        const Span sp = span(p);
        nquad += (sp.kc1 - sp.kc0) / 4;
    }
    // x rows of padded tokens stay zero in every entry (never copied)
    for (int pp = t; pp < C::RQ * 4 * C::NB * 8; pp += kLoaders) {
        const int e = pp / (4 * C::NB * 8), q = pp % (C::NB * 8), c = (pp / (C::NB * 8)) % 4;
        const int gg = q >> 5, ll = q & 31;
        const int tok = 8 * (gg >> 1) + (ll & 7), kx = 4 * (gg & 1) + (ll >> 3);
        if (tok >= a.bop_rows)
            *reinterpret_cast<uint4*>(raw + (size_t)e * C::RAWQ + 128 * 144 + c * C::X + kx * (C::NB * 16) +
                                      (tok >> 3) * 128 + (tok & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    // issue cursor and the row ids it copies: rows (t >> 3) + 16 i of the tile
    int ip = 0;
    Span isp = span(0);
    int iq = isp.kc0 / 4;
    int crow[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) crow[i] = srow[(t >> 3) + 16 * i];
    auto issue = [&](int qn) {
        unsigned char* b = raw + (size_t)(qn % C::RQ) * C::RAWQ;
        const size_t co = (size_t)iq * 128 + (t & 7) * 16;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (crow[i] >= 0) cp16(b + ((t >> 3) + 16 * i) * 144 + (t & 7) * 16, a.q + (size_t)crow[i] * cpr + co);
        const int k0 = iq * 256;
#pragma unroll
        for (int pp = t; pp < 4 * C::NB * 8; pp += kLoaders) {
            const int c = pp / (C::NB * 8), q = pp % (C::NB * 8);
            const int gg = q >> 5, ll = q & 31;
            const int tok = 8 * (gg >> 1) + (ll & 7), kx = 4 * (gg & 1) + (ll >> 3);
            if (tok < a.bop_rows)
                cp16(b + 128 * 144 + c * C::X + kx * (C::NB * 16) + (tok >> 3) * 128 + (tok & 7) * 16,
                     a.bop + (size_t)tok * a.K + k0 + c * 64 + kx * 8);
        }
        cp_commit();
        if (++iq == isp.kc1 / 4 && ip + 1 < npiece) {
            ++ip;
            isp = span(ip);
            iq = isp.kc0 / 4;
            const int base = 128 * isp.tile;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int rr = base + (t >> 3) + 16 * i;
                crow[i] = rr < R ? __ldg(a.idx + rr) : -1;
            }
        }
    };
    const int ahead = C::RQ - 1 - C::S / 4;
    int issued = 0;
    while (issued < nquad && issued < ahead) issue(issued++);
    // conversion cursor
    int cp = 0;
    Span csp = span(0);
    int cq = csp.kc0 / 4;
    int j = 0;
    bool stop = false;
    const int lane = t & 31;
    const unsigned tlane = tmem + ((unsigned)(t & ~31) << 16) + (unsigned)C::ACOL;
    for (int qd = 0; qd < nquad; ++qd) {
        cp_wait_n(issued - 1 - qd);             // this thread's copies of quad qd have landed
        if (loaders_sync_any(stop)) break;      // and everyone's; a warp that gave up stops all
        const unsigned char* b = raw + (size_t)(qd % C::RQ) * C::RAWQ;
        const bool valid = 128 * csp.tile + t < R;
        // two chunks per step: 16 independent conversions keep the warp busy
#pragma unroll 1
        for (int c = 0; c < 4; c += 2, j += 2) {
            const int s0 = j % C::S, s1 = (j + 1) % C::S;
            if (j >= C::S) {   // lane 0 waits for the stages' previous MMAs for the warp
                bool good = true;
                if (lane == 0)
                    good = bar_wait(&empty[s0], ((j / C::S) - 1) & 1, ctl) &&
                           bar_wait(&empty[s1], (((j + 1) / C::S) - 1) & 1, ctl);
                if (!__shfl_sync(FULL, good ? 1 : 0, 0)) {
                    stop = true;
                    break;
                }
            }
            // the stage waits of this quad's first chunk cover the MMAs of
            // quad qd-1-S/4: its entry can take quad qd + ahead
            if (c == 0 && issued < nquad) issue(issued++);
            uint32_t av[2][32];
            if (valid) {
                const uint4* src = reinterpret_cast<const uint4*>(b + t * 144 + c * 32);
                const uint4 q0 = src[0], q1 = src[1], q2 = src[2], q3 = src[3];
                const uint32_t cw[16] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w,
                                         q2.x, q2.y, q2.z, q2.w, q3.x, q3.y, q3.z, q3.w};
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const uint4 h = q8_f16(cw[e]);
                    av[e >> 3][4 * (e & 7)] = h.x;
                    av[e >> 3][4 * (e & 7) + 1] = h.y;
                    av[e >> 3][4 * (e & 7) + 2] = h.z;
                    av[e >> 3][4 * (e & 7) + 3] = h.w;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) av[0][e] = av[1][e] = 0u;
            }
            tc_after();   // after the stages' previous MMAs (waited for above)
            tmem_st32(tlane + (unsigned)(32 * s0), av[0]);
            tmem_st32(tlane + (unsigned)(32 * s1), av[1]);
            tmem_wait_st();
            tc_before();
            warp_arrive(&full[s0]);
            warp_arrive(&full[s1]);
        }
        if (++cq == csp.kc1 / 4 && cp + 1 < npiece) {
            ++cp;
            csp = span(cp);
            cq = csp.kc0 / 4;
        }
    }
    cp_wait_all();
}

// MMA issuer of the INT4 FC1.  Chunk j owns accumulator slot j % CS: two
// TMEM accumulators of NB columns, one per group of 32 along K (K-steps 0-1
// and 2-3 of the stage's A columns in TMEM against the x chunk in the raw
// ring).  One
// commit per chunk, on `empty[j % S]`, frees the stage for the loaders and
// tells the epilogue that the chunk's two accumulators are final; the slot is
// reused once the epilogue has read it (`cempty`).  The issuing thread runs a
// chain of dependent instructions, so the loop keeps it short: one wait per
// barrier per chunk and descriptors advanced by adding the byte offset >> 4.
template <typename C>
PI_DEV bool q4_mma(unsigned char* ring, int total, unsigned tmem, unsigned long long* full,
                   unsigned long long* empty, unsigned long long* cempty, const Ctl& ctl, int& it) {
    const unsigned idesc = idesc_f16(128, C::NB, false);
    const uint64_t bd0 = sdesc(su32(ring + (size_t)C::S * C::STAGE) + 128 * 144, C::NB * 16, 128);
    int qslot = 0;
    for (it = 0; it < total; ++it) {
        const int s = it % C::S, cs = it % C::CS;
        if (!bar_wait(&full[s], (it / C::S) & 1, ctl)) return false;
        if (it >= C::CS && !bar_wait(&cempty[cs], ((it / C::CS) - 1) & 1, ctl)) return false;
        tc_after();
        const unsigned ta = tmem + (unsigned)(C::ACOL + 32 * s);
        const uint64_t bd = bd0 + (uint64_t)((qslot * C::RAWQ + (it & 3) * C::X) >> 4);
        const unsigned dcol = tmem + (unsigned)(2 * cs * C::NB);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_f16_ta(dcol + (unsigned)((kk >> 1) * C::NB), ta + (unsigned)(8 * kk),
                       bd + (uint64_t)((kk * 2 * C::NB * 16) >> 4), idesc, (unsigned)(kk & 1));
        mma_commit(&empty[s]);
        if ((it & 3) == 3) qslot = qslot + 1 == C::RQ ? 0 : qslot + 1;
    }
    return true;
}

// Epilogue of the INT4 FC1: TMEM lane m = row m of the tile.  For each chunk
// in order it waits for the chunk's commit, reads its two group accumulators,
// frees the slot and adds them times the row's group scales (read from global
// memory, a quad of eight scales two quads ahead) into register sums; at the
// end of a piece the sums are its partial tile.
template <typename C, int NT, typename SpanOf>
PI_DEV void q4_epilogue(const TcRowsArgs& a, const SpanOf& span, int npiece, int R, int g, unsigned tmem,
                        unsigned long long* empty, unsigned long long* cempty, const Ctl& ctl) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = warp - 4, m = 32 * e + lane;
    const size_t spr = (size_t)a.K / 32;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    const unsigned tl = tmem + ((unsigned)(32 * e) << 16);
    int j = 0;
    for (int p = 0; p < npiece; ++p) {
        const Span sp = span(p);
        const int r = 128 * sp.tile + m;
        const int rid = r < R ? __ldg(a.idx + r) : -1;
        const uint4* sq = reinterpret_cast<const uint4*>(a.qs + (size_t)(rid < 0 ? 0 : rid) * spr) + sp.kc0 / 4;
        const int nq = (sp.kc1 - sp.kc0) / 4;
        float z[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) z[t] = 0.f;
        uint4 s_cur = rid >= 0 ? __ldg(sq) : zero;
        uint4 s_next = rid >= 0 && nq > 1 ? __ldg(sq + 1) : zero;
        for (int q = 0; q < nq; ++q) {
            const uint4 sc = s_cur;
            s_cur = s_next;
            s_next = rid >= 0 && q + 2 < nq ? __ldg(sq + q + 2) : zero;
            const uint32_t sw[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
            for (int c = 0; c < 4; ++c, ++j) {
                const int s = j % C::S, cs = j % C::CS;
                if (!__all_sync(FULL, bar_wait(&empty[s], (j / C::S) & 1, ctl))) return;
                tc_after();
                float v0[NT], v1[NT];
#pragma unroll
                for (int k = 0; k < NT; k += 16) {
                    tmem_ld16(tl + (unsigned)(2 * cs * C::NB + k), v0 + k);
                    tmem_ld16(tl + (unsigned)((2 * cs + 1) * C::NB + k), v1 + k);
                }
                tmem_wait_ld();
                tc_before();
                __syncwarp();
                if (lane == 0) bar_arrive(&cempty[cs]);
                const float s0 = __half2float(__ushort_as_half((unsigned short)(sw[c] & 0xFFFFu)));
                const float s1 = __half2float(__ushort_as_half((unsigned short)(sw[c] >> 16)));
#pragma unroll
                for (int t = 0; t < NT; ++t) z[t] = fmaf(s1, v1[t], fmaf(s0, v0[t], z[t]));
            }
        }
        if (p < a.slots) {
            float* dst = a.part + ((size_t)g * a.slots + p) * C::COLS * 128 + m;
#pragma unroll
            for (int t = 0; t < NT; ++t)
                if (t < a.B) dst[(size_t)t * 128] = z[t];
        } else if (lane == 0) {
            atomicExch(a.status, (int)PI_ERR_WORKSPACE);
        }
    }
}

template <int MODE, int NT>
__global__ void __launch_bounds__(kTcThreads, 1) k_rows_tc(const __grid_constant__ TcRowsArgs a) {
    pdl_entry();
    using C = RowsCfg<MODE, NT>;
    // contiguous A rows (predictor P1, P2) may come by TMA: one thread issues
    // the A and B tiles of each stage (128-byte swizzle, the MMA layout)
    const bool TMA = (MODE == 2 || MODE == 3) && a.use_tma != 0;
    extern __shared__ unsigned char dsm[];
    __shared__ __align__(8) unsigned long long full[C::S], empty[C::S], accf[2], acce[2], drain;
    __shared__ __align__(8) unsigned long long cempty[C::CS];   // INT4 accumulator slots read
    __shared__ unsigned tmem_slot;
    __shared__ int abort_flag;
    __shared__ int srow[128];  // A row ids of the current tile (-1 past the end)

    const int R = a.count != nullptr ? *a.count : a.R;
    const int G = gridDim.x, g = blockIdx.x;
    const int ntile = (R + 127) / 128;
    const int nk = (a.K + 63) / 64;
    const int nu = C::Q4 ? nk / C::KQ : nk;   // units per tile (INT4: quads; K % 256 == 0)
    const long long U = (long long)ntile * nu;
    const long long u0 = U * g / G, u1 = U * (g + 1) / G;
    int npiece;
    if (C::DIRECT)
        npiece = ntile > g ? (ntile - 1 - g) / G + 1 : 0;
    else
        npiece = u0 < u1 ? (int)((u1 - 1) / nu - u0 / nu) + 1 : 0;
    if (npiece == 0) return;
    auto span = [&](int p) {
        Span s;
        if (C::DIRECT) {
            s.tile = g + p * G;
            s.kc0 = 0;
            s.kc1 = nk;
        } else {
            s.tile = (int)(u0 / nu) + p;
            const long long lo = (long long)s.tile * nu;
            s.kc0 = C::KQ * (int)((u0 > lo ? u0 : lo) - lo);
            s.kc1 = C::KQ * (int)((u1 < lo + nu ? u1 : lo + nu) - lo);
        }
        return s;
    };
    unsigned char* ring = align1024(dsm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // warp 8 sets up barriers and tensor memory while the loaders fetch the
    // first tile's row ids
    if (warp == 8) {
        if (lane == 0) {
            for (int s = 0; s < C::S; ++s) {
                bar_init(&full[s], TMA ? 1 : kLoaderWarps);
                bar_init(&empty[s], 1);
            }
            for (int b = 0; b < 2; ++b) {
                bar_init(&accf[b], 1);
                bar_init(&acce[b], 128);
            }
            if (C::Q4)
                for (int q = 0; q < C::CS; ++q) bar_init(&cempty[q], 4);
            bar_init(&drain, 1);
            abort_flag = 0;
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncwarp();
        tmem_alloc(&tmem_slot, C::TMEM);
    } else if (warp < 4) {
        const Span s0 = span(0);
        const int rows = R - 128 * s0.tile < 128 ? R - 128 * s0.tile : 128;
        srow[tid] = tid < rows ? (C::GATHER ? a.idx[128 * s0.tile + tid] : 128 * s0.tile + tid) : -1;
    }
    tc_before();
    __syncthreads();
    tc_after();
    const unsigned tmem = tmem_slot;
    const Ctl ctl{a.status, a.timeout_ns, &abort_flag};

    if (warp < 4 && C::Q4) {
        if constexpr (C::Q4) q4_loader<C>(a, ring, span, npiece, R, srow, tmem, full, empty, ctl);
    } else if (warp < 4 && TMA) {
        // ---- TMA producer (one thread): stage it = (piece, K-chunk) in order
        if (tid == 0) {
            constexpr unsigned kBytes = (unsigned)(C::NA * kTileA + C::X);
            int it = 0;
            bool ok = true;
            for (int p = 0; p < npiece && ok; ++p) {
                const Span sp = span(p);
                for (int ks = sp.kc0; ks < sp.kc1; ++ks, ++it) {
                    const int s = it % C::S;
                    if (it >= C::S && !bar_wait(&empty[s], ((it / C::S) - 1) & 1, ctl)) {
                        ok = false;
                        break;
                    }
                    unsigned char* st = ring + (size_t)s * C::STAGE;
                    bar_arrive_expect_tx(&full[s], kBytes);
                    tma_load_2d(st, &a.tma_a, 64 * ks, 128 * sp.tile, &full[s]);
                    tma_load_2d(st + C::NA * kTileA, &a.tma_b, 64 * ks, 0, &full[s]);
                }
            }
            // every copy issued has landed before the CTA may exit
            for (int s = 0; s < C::S && s < it; ++s) {
                const int last = s + ((it - 1 - s) / C::S) * C::S;
                bar_drain(&full[s], (last / C::S) & 1, kDrainTimeoutNs);
            }
        }
    } else if (warp < 4) {
        // ---- loaders.  A tiles use the 128-byte-swizzled layout, so the 8
        // lanes of one shared-memory phase copy the 8 chunks of one row's 128
        // bytes without bank conflicts.  Stages go out in pairs: a warp
        // instruction copies 2 rows x 256 contiguous bytes (both K-chunks).
        const int t = tid, w = t >> 5, l = t & 31;
        int total = 0;
        for (int p = 0; p < npiece; ++p) {
            const Span sp = span(p);
            total += sp.kc1 - sp.kc0;
        }
        int pc = 0;
        Span sp = span(0);
        int ks = sp.kc0;
        // this thread's rows: pair issue (16 rows) and single-stage issue (8 rows)
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
            loaders_sync_any(false);  // nobody still reads the previous tile's ids
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
        // chunk c of K-chunk kchunk of `row` (element offset base, -1: none)
        // into the A tile(s) of slot st
        auto copy_a = [&](unsigned char* st, int row, long long base, int kchunk, int c) {
            if (base < 0) return;
            const unsigned off = (row >> 3) * 1024 + (row & 7) * 128 + ((c ^ (row & 7)) << 4);
            const long long gofs = base + kchunk * 64 + c * 8;
            cp16(st + off, a.a0 + gofs);
            if (MODE == 1) cp16(st + kTileA + off, a.a1 + gofs);
        };
        // B operand chunk of K-chunk kchunk into slot st (no swizzle)
        auto copy_b = [&](unsigned char* st, int kchunk) {
            const int k0 = kchunk * 64;
            const int kvalid = a.K - k0 < 64 ? a.K - k0 : 64;
#pragma unroll
            for (int pp = t; pp < C::NB * 8; pp += kLoaders) {
                const int gg = pp >> 5, ll = pp & 31;
                const int tok = 8 * (gg >> 1) + (ll & 7), kx = 4 * (gg & 1) + (ll >> 3);
                if (tok < a.bop_rows && kx * 8 < kvalid)
                    cp16(st + C::NA * kTileA + kx * (C::NB * 16) + (tok >> 3) * 128 + (tok & 7) * 16,
                         a.bop + (size_t)tok * a.K + k0 + kx * 8);
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
            if (loaders_sync_any(!good)) {  // stop together
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
                fence_async_smem();
                warp_arrive(&full[(2 * pd) % C::S]);
                if (2 * pd + 1 < total) warp_arrive(&full[(2 * pd + 1) % C::S]);
            }
        }
        if (ok) {
            // release the pairs still in flight one by one, oldest first
            const int first = npairs - C::LAGP < 0 ? 0 : npairs - C::LAGP;
            for (int pd = first; pd < npairs; ++pd) {
                const int newer = npairs - 1 - pd;  // groups committed after pair pd
                if (newer >= 3)
                    cp_wait<3>();
                else if (newer == 2)
                    cp_wait<2>();
                else if (newer == 1)
                    cp_wait<1>();
                else
                    cp_wait<0>();
                fence_async_smem();
                warp_arrive(&full[(2 * pd) % C::S]);
                if (2 * pd + 1 < total) warp_arrive(&full[(2 * pd + 1) % C::S]);
            }
        }
        cp_wait_all();
    } else if (warp < 8 && C::Q4) {
        if constexpr (C::Q4) q4_epilogue<C, NT>(a, span, npiece, R, g, tmem, empty, cempty, ctl);
    } else if (warp < 8) {
        // ---- epilogue: TMEM lane m = row m of the tile
        const int e = warp - 4, m = 32 * e + lane;
        for (int p = 0; p < npiece; ++p) {
            const int b = p & 1;
            if (!bar_wait(&accf[b], (p >> 1) & 1, ctl)) break;
            tc_after();
            const unsigned ta = tmem + ((unsigned)(32 * e) << 16) + (unsigned)(b * C::ACC);
            const Span sp = span(p);
            if (C::DIRECT) {
                float vh[NT], vl[NT];
#pragma unroll
                for (int c = 0; c < NT; c += 16) {
                    tmem_ld16(ta + c, vh + c);
                    tmem_ld16(ta + NT + c, vl + c);
                }
                tmem_wait_ld();
                tc_before();
                bar_arrive(&acce[b]);
                const int k = 128 * sp.tile + m;
                const float bk = k < R ? __half2float(a.bias[k]) : 0.f;
                const int word = (128 * sp.tile + 32 * e) >> 5;
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const bool on = k < R && (vh[t] + vl[t]) + bk > a.tau;
                    const unsigned bits = __ballot_sync(FULL, on);
                    if (lane == 0 && t < a.B && word < a.W) a.mask[(size_t)t * a.W + word] = bits;
                }
            } else {
                float v[C::NACC][NT];
#pragma unroll
                for (int q = 0; q < C::NACC; ++q)
#pragma unroll
                    for (int c = 0; c < NT; c += 16) tmem_ld16(ta + q * C::NB + c, v[q] + c);
                tmem_wait_ld();
                tc_before();
                bar_arrive(&acce[b]);
                if (p < a.slots) {
                    float* dst = a.part + ((size_t)g * a.slots + p) * C::COLS * 128 + m;
#pragma unroll
                    for (int q = 0; q < C::NACC; ++q)
#pragma unroll
                        for (int t = 0; t < NT; ++t)
                            if (t < a.B) dst[(size_t)(q * NT + t) * 128] = v[q][t];
                } else if (lane == 0) {
                    atomicExch(a.status, (int)PI_ERR_WORKSPACE);
                }
            }
        }
    } else if (lane == 0) {
        // ---- MMA issuer
        const unsigned idesc = idesc_f16(128, C::NB, false);
        int it = 0;
        bool ok = true;
        if constexpr (C::Q4) {
            int total = 0;
            for (int p = 0; p < npiece; ++p) {
                const Span sp = span(p);
                total += sp.kc1 - sp.kc0;
            }
            ok = q4_mma<C>(ring, total, tmem, full, empty, cempty, ctl, it);
        }
        const uint64_t ad0 = sdesc_sw128(su32(ring));
        // B: swizzled like A when it comes by TMA, else core matrices of 8 rows
        const uint64_t bd0 = TMA ? sdesc_sw128(su32(ring) + C::NA * kTileA)
                                 : sdesc(su32(ring) + C::NA * kTileA, C::NB * 16, 128);
        const uint64_t bstep = TMA ? 2u : (uint64_t)((2 * C::NB * 16) >> 4);   // per K-step of 16
        for (int p = 0; p < npiece && ok && !C::Q4; ++p) {
            const Span sp = span(p);
            const int b = p & 1;
            if (p >= 2 && !bar_wait(&acce[b], ((p >> 1) - 1) & 1, ctl)) {
                ok = false;
                break;
            }
            tc_after();
            const unsigned dcol = tmem + (unsigned)(b * C::ACC);
            for (int ks = sp.kc0; ks < sp.kc1; ++ks, ++it) {
                const int s = it % C::S;
                if (!bar_wait(&full[s], (it / C::S) & 1, ctl)) {
                    ok = false;
                    break;
                }
                tc_after();
                // descriptors advance by byte offset >> 4 from stage 0's: the
                // issuing thread is one dependent chain, so its loop stays short
                const uint64_t so = (uint64_t)((s * C::STAGE) >> 4);
                const uint64_t ad = ad0 + so, bd = bd0 + so;
                const unsigned first = ks > sp.kc0 ? 1u : 0u;
                if (64 * ks + 64 <= a.K) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bk = bd + bstep * (uint64_t)kk;
                        const unsigned acc = kk > 0 ? 1u : first;
                        mma_f16(dcol, ad + (uint64_t)(2 * kk), bk, idesc, acc);
                        if (MODE == 1) mma_f16(dcol + C::NB, ad + (uint64_t)((kTileA >> 4) + 2 * kk), bk, idesc, acc);
                    }
                } else {
                    const int ksteps = (a.K - 64 * ks) / 16;
                    for (int kk = 0; kk < ksteps; ++kk) {
                        const uint64_t bk = bd + bstep * (uint64_t)kk;
                        const unsigned acc = kk > 0 ? 1u : first;
                        mma_f16(dcol, ad + (uint64_t)(2 * kk), bk, idesc, acc);
                        if (MODE == 1) mma_f16(dcol + C::NB, ad + (uint64_t)((kTileA >> 4) + 2 * kk), bk, idesc, acc);
                    }
                }
                mma_commit(&empty[s]);
            }
            if (ok) mma_commit(&accf[b]);
        }
        if (ok) {
            // every slot's last release has arrived before the CTA may exit
            for (int s = 0; s < C::S && s < it; ++s) {
                const int last = s + ((it - 1 - s) / C::S) * C::S;
                bar_drain(&empty[s], (last / C::S) & 1, kDrainTimeoutNs);
            }
        } else {
            mma_commit(&drain);
            bar_drain(&drain, 0, kDrainTimeoutNs);
        }
    }
    tc_before();
    __syncthreads();
    if (warp == 8) {
        tc_after();
        tmem_free(tmem, C::TMEM);
    }
}

// h[j, t] = act(Z[j, t] + b1[idx_j]) (gated: times Zu[j, t]), zero where token
// t's own mask does not list idx_j; live[j] = some h[j, :] != 0.  act is ReLU
// for FFN rows and the identity for projection rows (RELU = false).
// Block: 32 consecutive rows (lane) x B tokens (warp).
template <bool GATED, bool RELU>
__global__ void __launch_bounds__(1024) k_fc1_finish(const float* __restrict__ part, int slots, int G, int nk,
                                                     const int32_t* __restrict__ count, int B, int NT,
                                                     const int32_t* __restrict__ idx, const __half* __restrict__ b1,
                                                     const uint32_t* __restrict__ mask, int W,
                                                     float* __restrict__ h, int32_t* __restrict__ live) {
    pdl_entry();
    __shared__ int slot[kMaxCtas];
    __shared__ int rng[2];
    __shared__ int any[32];
    const int n = *count;
    const int j0 = blockIdx.x * 32;
    if (j0 >= n) return;
    const int lane = threadIdx.x & 31, t = threadIdx.x >> 5;
    cover_setup((long long)((n + 127) / 128) * nk, G, nk, j0 >> 7, slot, rng);
    if (threadIdx.x < 32) any[threadIdx.x] = 0;
    __syncthreads();
    const int j = j0 + lane;
    const int cols = (GATED ? 2 : 1) * NT;
    if (j < n) {
        const int m = j & 127;
        const int k = idx[j];
        float v = sum_cover(part, slot, rng, slots, cols, t, m) + __half2float(b1[k]);
        if (RELU) v = v > 0.f ? v : 0.f;
        if (GATED) v *= sum_cover(part, slot, rng, slots, cols, NT + t, m);
        if (mask != nullptr && !((mask[(size_t)t * W + (k >> 5)] >> (k & 31)) & 1u)) v = 0.f;
        h[(size_t)j * B + t] = v;
        if (v != 0.f) any[lane] = 1;
    }
    __syncthreads();
    if (t == 0 && j < n && live != nullptr) live[j] = any[lane] ? 1 : 0;
}

// u[t, i] = sum of the P1 x partials, stored as fp16 hi = fp16(u) and
// lo = fp16(u - hi) rows: uhl[t][i] = hi, uhl[NT + t][i] = lo (zero rows for
// padded tokens t >= B).  Block: 32 consecutive i (lane) x NT tokens (warp).
__global__ void __launch_bounds__(1024) k_u_finish(const float* __restrict__ part, int slots, int G, int nk, int r,
                                                   int B, int NT, __half* __restrict__ uhl) {
    pdl_entry();
    __shared__ int slot[kMaxCtas];
    __shared__ int rng[2];
    const int i0 = blockIdx.x * 32;
    const int lane = threadIdx.x & 31, t = threadIdx.x >> 5;
    cover_setup((long long)((r + 127) / 128) * nk, G, nk, i0 >> 7, slot, rng);
    __syncthreads();
    const int i = i0 + lane;
    if (i >= r) return;
    const float u = t < B ? sum_cover(part, slot, rng, slots, NT, t, i & 127) : 0.f;
    const __half hi = __float2half_rn(u);
    uhl[(size_t)t * r + i] = hi;
    uhl[(size_t)(NT + t) * r + i] = __float2half_rn(u - __half2float(hi));
}

// ------------------------------------------------------------------------ FC2

template <int NT>
struct Fc2Cfg {
    static constexpr int BOP = 2 * NT * 64 * 2;          // (hi | lo) tokens x 64 rows fp16
    static constexpr int RAW = 64 * NT * 4;              // 64 rows x B fp32 of h, as copied
    static constexpr int STAGE = kTileA + BOP + RAW;
    static constexpr int IDX = 64 * 2 * 4;               // 64 row ids + 64 live flags (int32)
    static constexpr int S = kRingBudget / (STAGE + IDX) > 8 ? 8 : kRingBudget / (STAGE + IDX);
    static constexpr int LAG = S - 2;
    static constexpr int ACC = 2 * NT;
    static constexpr int TMEM = tmem_cols_for(2 * ACC);
    static constexpr size_t SMEM = (size_t)S * (STAGE + IDX) + 1024;
};

struct TcFc2Args {
    const float* h;        // [count][B]
    const int32_t* idx;
    const int32_t* count;
    const __half* w2t;
    const int32_t* live;   // nullable: rows with live == 0 have h == 0 for every token
    float* part;           // [G][slots][NT][128]
    int* status;
    long long timeout_ns;
    int B, d, slots;
};

struct Piece {
    int ct, j0, j1;
};
constexpr int kMaxPieces = 16;   // pieces of one CTA's stream-K range

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
    pdl_entry();
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
    // this CTA's pieces, computed once (64-bit divisions stay out of the loops)
    __shared__ Piece ptab[kMaxPieces];
    if (npiece > kMaxPieces) {
        if (threadIdx.x == 0) atomicExch(a.status, (int)PI_ERR_WORKSPACE);
        return;
    }
    if (threadIdx.x < npiece) fc2_piece(u0, u1, n, threadIdx.x, &ptab[threadIdx.x]);
    unsigned char* ring = align1024(dsm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < C::S; ++s) {
            bar_init(&full[s], kLoaderWarps);
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
            const Piece pc = ptab[cv_piece];
            convert(cv, pc, cv_st);
            fence_async_smem();
            warp_arrive(&full[cv % C::S]);
            ++cv;
            if (64 * (++cv_st) >= pc.j1 - pc.j0) {
                ++cv_piece;
                cv_st = 0;
            }
        };
        // Row ids and live flags of stage q sit in a small ring (slot q % S),
        // copied LAG + 1 stages ahead of use, so no loader waits on them.
        int32_t* sidx = reinterpret_cast<int32_t*>(ring + (size_t)C::S * C::STAGE);
        int32_t* slive = sidx + C::S * 64;
        int total = 0;
        for (int p = 0; p < npiece; ++p) {
            const Piece pc = ptab[p];
            total += (pc.j1 - pc.j0 + 63) / 64;
        }
        int fq = 0, fpiece = 0, fst = 0;  // next stage whose row ids to copy
        auto copy_ids = [&]() {
            const Piece pc = ptab[fpiece];
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
        for (int pi_ = 0; pi_ < npiece && ok; ++pi_) {
            const Piece pc = ptab[pi_];
            const int nst = (pc.j1 - pc.j0 + 63) / 64;
            const int col0 = pc.ct * 128;
            for (int st = 0; st < nst; ++st, ++it) {
                const int s = it % C::S;
                bool good = true;
                if (it >= C::S) good = bar_wait(&empty[s], ((it / C::S) - 1) & 1, ctl);
                unsigned char* sb = ring + (size_t)s * C::STAGE;
                const int jb = pc.j0 + 64 * st;
                if (good) {
                    // W2t tile, 128-byte-swizzled MN-major: a warp instruction
                    // copies 2 rows x 256 contiguous bytes (lane: row half
                    // l >> 4, 16-byte column chunk c16 = l & 15)
                    const int c16 = l & 15;
                    int kv[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int kk = 2 * (4 * q + w) + (l >> 4);
                        const bool in = jb + kk < pc.j1;
                        const bool alive = a.live == nullptr || slive[s * 64 + kk] != 0;
                        kv[q] = (in && alive) ? sidx[s * 64 + kk] : -1;
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int kk = 2 * (4 * q + w) + (l >> 4);
                        unsigned char* dst = sb + (c16 >> 3) * 1024 + (kk >> 3) * 2048 + (kk & 7) * 128 +
                                             (((c16 & 7) ^ (kk & 7)) << 4);
                        if (kv[q] >= 0)
                            cp16(dst, a.w2t + (size_t)kv[q] * a.d + col0 + c16 * 8);
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
                    if (fq < total) copy_ids();  // ids of stage it + LAG + 1
                }
                cp_commit();
                if (it >= C::LAG) cp_wait<C::LAG>();
                // every loader's copies of stage it - LAG (and the ids of stage
                // it + 1) have landed; stop together
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
            const Piece pc = ptab[p];
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
                    const uint64_t ad = sdesc_sw128_mn(sa + kk * 4096, 1024, 2048);
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
                bar_drain(&empty[s], (last / C::S) & 1, kDrainTimeoutNs);
            }
        } else {
            mma_commit(&drain);
            bar_drain(&drain, 0, kDrainTimeoutNs);
        }
    }
    tc_before();
    __syncthreads();
    if (warp == 8) {
        tc_after();
        tmem_free(tmem, C::TMEM);
    }
}

// ------------------------------------------------------------ FC2, INT4 rows
//
// y[t, c] = sum_j h[j, t] q[j, c] s[j, c / 32] with the stream-K split of the
// fp16 FC2.  The W2t codes enter the MMA as exact fp16 integers (A: 128
// columns x 64 rows per stage, MN-major, as the fp16 rows), and the group
// scale, which changes along the rows (K) and along the 32-column groups of
// the tile (M), moves into the B operand: for each of the tile's four groups g
// and token t, B holds v = h[j, t] s[j, g] as hi = fp16(v) and
// lo = fp16((v - hi) 2^11), N = 4 groups x 16 tokens x (hi | lo) = 128.  An
// accumulator column (g, t, .) is meaningful only for the tile's columns of
// group g; epilogue warp e owns TMEM lanes 32e .. 32e+31 (group e) and reads
// its columns (e, t, hi | lo): y = D_hi + 2^-11 D_lo.  Scaling lo up keeps it
// out of the fp16 subnormals wherever hi is normal, so the pair carries about
// 22 bits of v.
//
// Eight loader warps (two per SM sub-partition: the per-stage work is a chain
// of dependent shared-memory loads and conversions that one warp per
// sub-partition cannot overlap) copy each stage's codes (64 rows x 64 bytes),
// scales (64 rows x 4) and h rows raw into a ring of RQ entries LAG stages
// ahead, with the row ids and live flags copied LAG + 1 stages ahead of that.
// In one loop step they wait for stage cv's copies, then issue stage cv + LAG
// and write stage cv's A and B operands in the same instruction stream (the
// two are independent, so their latencies overlap), fence the operands for the
// tensor cores and arrive on `full`.
constexpr int kQLoaderWarps = 8;
constexpr int kQLoaders = 32 * kQLoaderWarps;
constexpr int kQThreads = kQLoaders + 128 + 32;   // loaders, 4 epilogue warps, MMA warp

// barrier 1 over the kQLoaders loader threads, OR of a flag
PI_DEV bool qloaders_sync_any(bool v) {
    unsigned r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, 1, %2, q;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(r)
        : "r"((unsigned)v), "n"(kQLoaders)
        : "memory");
    return r != 0;
}

template <int NT>
struct Fc2qCfg {
    static constexpr int N = 8 * NT;                     // 4 groups x NT tokens x (hi | lo)
    static constexpr int BOP = N * 64 * 2;
    static constexpr int STAGE = kTileA + BOP;
    static constexpr int S = 4;
    static constexpr int LAG = 6;
    static constexpr int RQ = LAG + 1;                   // raw entries
    static constexpr int IDR = 2 * LAG + 2;              // row-id slots
    static constexpr int RCODE = 64 * 64;
    static constexpr int RSC = 64 * 8;
    static constexpr int RVAL = 64 * 4;
    static constexpr int RH = 64 * NT * 4;
    static constexpr int RAW = RCODE + RSC + RVAL + RH;
    static constexpr int IDS = 64 * 2 * 4;               // 64 row ids + 64 live flags
    static constexpr int ACC = N;
    static constexpr int TMEM = tmem_cols_for(2 * ACC);
    static constexpr size_t SMEM = (size_t)S * STAGE + (size_t)RQ * RAW + (size_t)IDR * IDS + 1024;
    static_assert(STAGE % 1024 == 0 && RAW % 16 == 0, "stage alignment");
    static_assert(NT == 16 && kQLoaders == 256, "thread mappings below assume 16 tokens, 256 loaders");
};

struct TcFc2qArgs {
    const float* h;        // [count][B]
    const int32_t* idx;
    const int32_t* count;
    const uint8_t* q;      // W2t codes [F][d/2]
    const __half* qs;      // W2t group scales [F][d/32]
    const int32_t* live;   // nullable
    float* part;           // [G][slots][NT][128]
    int* status;
    long long timeout_ns;
    int B, d, slots;
};

template <int NT>
__global__ void __launch_bounds__(kQThreads, 1) k_fc2q_tc(TcFc2qArgs a) {
    pdl_entry();
    using C = Fc2qCfg<NT>;
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
    __shared__ Piece ptab[kMaxPieces];
    if (npiece > kMaxPieces) {
        if (threadIdx.x == 0) atomicExch(a.status, (int)PI_ERR_WORKSPACE);
        return;
    }
    if (threadIdx.x < npiece) fc2_piece(u0, u1, n, threadIdx.x, &ptab[threadIdx.x]);
    unsigned char* ring = align1024(dsm);
    unsigned char* raw0 = ring + (size_t)C::S * C::STAGE;
    int32_t* ids0 = reinterpret_cast<int32_t*>(raw0 + (size_t)C::RQ * C::RAW);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int kEpi = kQLoaderWarps, kMma = kQLoaderWarps + 4;

    if (tid == 0) {
        for (int s = 0; s < C::S; ++s) {
            bar_init(&full[s], kQLoaderWarps);
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
    if (warp == kMma) tmem_alloc(&tmem_slot, C::TMEM);
    tc_before();
    __syncthreads();
    tc_after();
    const unsigned tmem = tmem_slot;
    const Ctl ctl{a.status, a.timeout_ns, &abort_flag};

    if (warp < kEpi) {
        const int t = tid;
        const bool vec = (a.B & 3) == 0 && (reinterpret_cast<uintptr_t>(a.h) & 15) == 0;
        const size_t cpr = (size_t)a.d / 2, spr = (size_t)a.d / 32;
        int total = 0;
        for (int p = 0; p < npiece; ++p) total += (ptab[p].j1 - ptab[p].j0 + 63) / 64;
        // cursors: row-id copies, raw copies, conversions (piece, stage in piece)
        int fq = 0, fpiece = 0, fst = 0;
        int ipc = 0, ist = 0;
        int cpc = 0, cst = 0;
        auto copy_ids = [&]() {
            const Piece pc = ptab[fpiece];
            const int kk = t & 63;
            const int j = pc.j0 + 64 * fst + kk;
            int32_t* sl = ids0 + (fq % C::IDR) * 128;
            if (j < pc.j1) {
                if (t < 64)
                    cp4(sl + kk, a.idx + j);
                else if (t < 128 && a.live != nullptr)
                    cp4(sl + 64 + kk, a.live + j);
            }
            ++fq;
            if (64 * (++fst) >= pc.j1 - pc.j0) {
                ++fpiece;
                fst = 0;
            }
        };
        auto issue = [&](int q) {
            const Piece pc = ptab[ipc];
            const int jb = pc.j0 + 64 * ist;
            const int nrow = pc.j1 - jb < 64 ? pc.j1 - jb : 64;
            const int col0 = pc.ct * 128;
            const int32_t* sl = ids0 + (q % C::IDR) * 128;
            unsigned char* rw = raw0 + (size_t)(q % C::RQ) * C::RAW;
            {   // codes: 16-byte chunk t of the stage, row t / 4
                const int r = t >> 2, part = t & 3;
                if (r < nrow && (a.live == nullptr || sl[64 + r] != 0))
                    cp16(rw + r * 64 + part * 16, a.q + (size_t)sl[r] * cpr + col0 / 2 + part * 16);
            }
            if (t < 64) {
                const bool ok = t < nrow && (a.live == nullptr || sl[64 + t] != 0);
                reinterpret_cast<int*>(rw + C::RCODE + C::RSC)[t] = ok ? 1 : 0;
                if (ok) cp8(rw + C::RCODE + 8 * t, a.qs + (size_t)sl[t] * spr + col0 / 32);
            }
            unsigned char* hd = rw + C::RCODE + C::RSC + C::RVAL;
            const float* hsrc = a.h + (size_t)jb * a.B;
            if (vec) {
                for (int c = t; c < nrow * a.B / 4; c += kQLoaders) cp16(hd + 16 * c, hsrc + 4 * c);
            } else {
                for (int c = t; c < nrow * a.B; c += kQLoaders) cp4(hd + 4 * c, hsrc + c);
            }
            if (64 * (++ist) >= pc.j1 - pc.j0) {
                ++ipc;
                ist = 0;
            }
        };
        auto convert = [&](int q) {
            const unsigned char* rw = raw0 + (size_t)(q % C::RQ) * C::RAW;
            unsigned char* sb = ring + (size_t)(q % C::S) * C::STAGE;
            // A: word c of row r holds columns 8c .. 8c+7 of the tile
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int w = t + kQLoaders * i, r = w >> 4, c = w & 15;
                const uint4 hv = q8_f16(*reinterpret_cast<const uint32_t*>(rw + r * 64 + 4 * c));
                *reinterpret_cast<uint4*>(sb + (c >> 3) * 1024 + (r >> 3) * 2048 + (r & 7) * 128 +
                                          (((c & 7) ^ (r & 7)) << 4)) = hv;
            }
            // B: rows 8 kc .. 8 kc + 7 of token tok, groups 2 gp and 2 gp + 1
            const int tok = t & 15, kc = (t >> 4) & 7, gp = t >> 7;
            const int* val = reinterpret_cast<const int*>(rw + C::RCODE + C::RSC);
            const float* hr = reinterpret_cast<const float*>(rw + C::RCODE + C::RSC + C::RVAL);
            float hv[8];
            uint32_t sw[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int r = 8 * kc + e;
                const bool ok = tok < a.B && val[r] != 0;
                hv[e] = ok ? hr[r * a.B + tok] : 0.f;
                sw[e] = ok ? reinterpret_cast<const uint32_t*>(rw + C::RCODE + 8 * r)[gp] : 0u;
            }
            unsigned char* bo = sb + kTileA + kc * (C::N * 16);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int grp = 2 * gp + u;
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    const float s0 = __half2float(__ushort_as_half((unsigned short)(sw[2 * e2] >> (16 * u))));
                    const float s1 = __half2float(__ushort_as_half((unsigned short)(sw[2 * e2 + 1] >> (16 * u))));
                    const float v0 = hv[2 * e2] * s0, v1 = hv[2 * e2 + 1] * s1;
                    const __half2 h2 = __floats2half2_rn(v0, v1);
                    const float2 bk = __half22float2(h2);
                    const __half2 l2 = __floats2half2_rn((v0 - bk.x) * 2048.f, (v1 - bk.y) * 2048.f);
                    hi[e2] = *reinterpret_cast<const uint32_t*>(&h2);
                    lo[e2] = *reinterpret_cast<const uint32_t*>(&l2);
                }
                const int nh = 2 * NT * grp + tok, nl = nh + NT;
                *reinterpret_cast<uint4*>(bo + (nh >> 3) * 128 + (nh & 7) * 16) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(bo + (nl >> 3) * 128 + (nl & 7) * 16) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            if (64 * (++cst) >= ptab[cpc].j1 - ptab[cpc].j0) {
                ++cpc;
                cst = 0;
            }
        };
        while (fq < total && fq <= C::LAG) copy_ids();
        cp_commit();
        cp_wait_all();
        qloaders_sync_any(false);
        bool ok = true;
        for (int q = 0; q < total + C::LAG; ++q) {
            const int cv = q - C::LAG;
            if (cv >= 0) {
                // this thread's copies of stage cv (and the ids of stage q) have
                // landed; every loader's, after the barrier
                cp_wait<C::LAG - 1>();
                if (qloaders_sync_any(!ok || *(volatile int*)&abort_flag)) {
                    ok = false;
                    break;
                }
                if (cv >= C::S) {   // the MMAs of stage cv - S have released the operand stage
                    bool good = true;
                    if (lane == 0) good = bar_wait(&empty[cv % C::S], ((cv / C::S) - 1) & 1, ctl);
                    if (!__shfl_sync(FULL, good ? 1 : 0, 0)) {
                        ok = false;
                        cp_commit();
                        continue;   // the next barrier stops every loader
                    }
                }
            }
            if (q < total) {
                issue(q);
                if (fq < total) copy_ids();   // ids of stage q + LAG + 1
            }
            if (cv >= 0) convert(cv);
            cp_commit();
            if (cv >= 0) {
                fence_async_smem();
                warp_arrive(&full[cv % C::S]);
            }
        }
        cp_wait_all();
    } else if (warp < kMma) {
        // ---- epilogue: TMEM lane m = column col0 + m, group e = m / 32
        const int e = warp - kEpi, m = 32 * e + lane;
        for (int p = 0; p < npiece; ++p) {
            const int b = p & 1;
            if (!bar_wait(&accf[b], (p >> 1) & 1, ctl)) break;
            tc_after();
            float vh[NT], vl[NT];
            const unsigned ta = tmem + ((unsigned)(32 * e) << 16) + (unsigned)(b * C::ACC + 2 * NT * e);
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
                    if (t < a.B) dst[(size_t)t * 128] = fmaf(vl[t], 1.0f / 2048.0f, vh[t]);
            } else if (lane == 0) {
                atomicExch(a.status, (int)PI_ERR_WORKSPACE);
            }
        }
    } else if (lane == 0) {
        // ---- MMA issuer: A = W2t codes (M = 128 columns, MN-major), B = h s (hi | lo per group)
        const unsigned idesc = idesc_f16(128, C::N, true);
        int it = 0;
        bool ok = true;
        for (int p = 0; p < npiece && ok; ++p) {
            const Piece pc = ptab[p];
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
                    const uint64_t ad = sdesc_sw128_mn(sa + kk * 4096, 1024, 2048);
                    const uint64_t bd = sdesc(sbop + kk * 2 * (C::N * 16), C::N * 16, 128);
                    mma_f16(dcol, ad, bd, idesc, (st | kk) ? 1u : 0u);
                }
                mma_commit(&empty[s]);
            }
            if (ok) mma_commit(&accf[b]);
        }
        if (ok) {
            for (int s = 0; s < C::S && s < it; ++s) {
                const int last = s + ((it - 1 - s) / C::S) * C::S;
                bar_drain(&empty[s], (last / C::S) & 1, kDrainTimeoutNs);
            }
        } else {
            mma_commit(&drain);
            bar_drain(&drain, 0, kDrainTimeoutNs);
        }
    }
    tc_before();
    __syncthreads();
    if (warp == kMma) {
        tc_after();
        tmem_free(tmem, C::TMEM);
    }
}

// y[b0 + t, c] = b2[c] + sum over the CTAs whose range touches column tile
// c / tw of their partial (ascending CTA order: reproducible), for the nb
// tokens of this pass.  Block: the tw columns of one tile x 1024 / tw tokens.
__global__ void __launch_bounds__(1024) k_fc2_tc_reduce(const float* __restrict__ part, int slots, int G,
                                                        const int32_t* __restrict__ count, int nb, int b0, int NT,
                                                        int d, int tw, const __half* __restrict__ b2,
                                                        float* __restrict__ y) {
    pdl_entry();
    __shared__ int slot[kMaxCtas];
    __shared__ int rng[2];
    const int ct = blockIdx.x;
    const int m = threadIdx.x % tw, t = blockIdx.y * (1024 / tw) + threadIdx.x / tw;
    const int n = *count;
    const int c = ct * tw + m;
    if (n == 0) {  // uniform over the block
        if (t < nb) y[(size_t)(b0 + t) * d + c] = __half2float(b2[c]);
        return;
    }
    cover_setup((long long)(d / tw) * n, G, n, ct, slot, rng);
    __syncthreads();
    if (t >= nb) return;
    y[(size_t)(b0 + t) * d + c] = __half2float(b2[c]) + sum_cover(part, slot, rng, slots, NT, t, m, tw);
}

template <typename K>
cudaError_t prep(K kernel, size_t smem) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}


}  // namespace

namespace {
int ceil_div(int a, int b) { return (a + b - 1) / b; }

// cuTensorMapEncodeTiled, looked up once through the runtime (the library
// links only the CUDA runtime)
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// Tensor map of `rows` fp16 rows of `inner` elements (row stride inner * 2
// bytes) read in boxes of 64 elements x box_rows rows with the 128-byte
// swizzle of the MMA operand tiles; rows and columns past the end read as zero.
bool rows_tensor_map(CUtensorMap* m, const void* base, int inner, int rows, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
    if (fn == nullptr || (reinterpret_cast<uintptr_t>(base) & 15) != 0 || (inner * 2) % 16 != 0) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
    const cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
int slots_for(int tiles, int G) { return ceil_div(tiles, G) + 2; }
// CTAs of the u = P1 x split.  P1 is small: at least 8 K-chunks per CTA keeps
// the number of partials per u element (the finish kernel's fan-in) low.
int u_grid(const Plan& p) {
    const int units = ceil_div(p.r, 128) * ceil_div(p.d, 64);
    const int G = p.nsm > 0 ? p.nsm : 1;
    return units / 8 < 1 ? 1 : (units / 8 < G ? units / 8 : G);
}
}  // namespace

// The INT4 batched plan covers 2 <= B <= 16 (its FC2 runs on CUDA cores);
// FC1 moves to the tensor cores at 16 tokens, one N = 16 tile.
bool tc4_supported(const Plan& p) {
    return p.int4 && !p.gated && p.B == 16 && p.d % 256 == 0 && p.nsm <= kMaxCtas;
}

bool tc_pred_supported(const Plan& p) { return p.B >= 16 && p.B <= 32 && p.d % 128 == 0 && p.nsm <= kMaxCtas; }

bool tc_supported(const Plan& p) { return !p.int4 && tc_pred_supported(p); }

int tc_tokens(const Plan& p) { return p.B <= 16 ? 16 : 32; }

size_t tc_part_floats(const Plan& p) {
    const size_t G = p.nsm > 0 ? p.nsm : 1, nt = tc_tokens(p);
    const size_t fc1 = G * slots_for(ceil_div(p.F, 128), (int)G) * (p.gated ? 2 : 1) * nt * 128;
    const size_t fc2 = G * slots_for(p.d / 128, (int)G) * nt * 128;
    const size_t pu = (size_t)u_grid(p) * slots_for(ceil_div(p.r, 128), u_grid(p)) * nt * 128;
    size_t m = fc1 > fc2 ? fc1 : fc2;
    return m > pu ? m : pu;
}

size_t tc_fc2_part_floats(const Plan& p) {
    const size_t G = p.nsm > 0 ? p.nsm : 1;
    return G * slots_for(p.d / 128, (int)G) * tc_tokens(p) * 128;
}

size_t tc_uhl_bytes(const Plan& p) { return (size_t)2 * tc_tokens(p) * p.r * sizeof(__half); }

namespace {

template <int MODE, int NT>
cudaError_t launch_rows(const TcRowsArgs& a, int grid, cudaStream_t s) {
    using C = RowsCfg<MODE, NT>;
    cudaError_t e = prep(k_rows_tc<MODE, NT>, C::SMEM);
    if (e != cudaSuccess) return e;
    launch_pdl(k_rows_tc<MODE, NT>, grid, kTcThreads, C::SMEM, s, a);
    return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_rows_nt(const TcRowsArgs& a, int nt, int grid, cudaStream_t s) {
    return nt == 16 ? launch_rows<MODE, 16>(a, grid, s) : launch_rows<MODE, 32>(a, grid, s);
}

}  // namespace

cudaError_t launch_predict_tc(const Plan& p, const __half* x, const __half* p1, const __half* p2,
                              const __half* bpred, float tau, uint32_t* mask, float* part, __half* uhl,
                              cudaStream_t s) {
    int* status = status_word();
    if (status == nullptr) return cudaErrorInvalidDevice;
    const int G = p.nsm, nt = tc_tokens(p);
    // u = P1 x (stream-K over (r tiles x d chunks)), finished into fp16 hi | lo rows
    const int Gu = u_grid(p);
    TcRowsArgs a{};
    a.a0 = p1;
    a.R = p.r;
    a.bop = x;
    a.bop_rows = p.B;
    a.K = p.d;
    // P1 rows and x by TMA (the loaders' gather path stays for a failed encode)
    a.use_tma = rows_tensor_map(&a.tma_a, p1, p.d, p.r, 128) && rows_tensor_map(&a.tma_b, x, p.d, p.B, nt) ? 1 : 0;
    a.B = p.B;
    a.part = part;
    a.slots = slots_for(ceil_div(p.r, 128), Gu);
    a.status = status;
    a.timeout_ns = wait_timeout_ns();
    cudaError_t e = launch_rows_nt<2>(a, nt, Gu, s);
    if (e != cudaSuccess) return e;
    launch_pdl(k_u_finish, ceil_div(p.r, 32), 32 * nt, 0, s, part, a.slots, Gu, ceil_div(p.d, 64), p.r, p.B, nt, uhl);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // s = P2 u + b > tau over whole 128-row tiles, mask words by ballot
    TcRowsArgs b{};
    b.a0 = p2;
    b.R = p.F;
    b.bop = uhl;
    b.bop_rows = 2 * nt;
    b.K = p.r;
    b.use_tma = rows_tensor_map(&b.tma_a, p2, p.r, p.F, 128) && rows_tensor_map(&b.tma_b, uhl, p.r, 2 * nt, 2 * nt)
                    ? 1 : 0;
    b.B = p.B;
    b.bias = bpred;
    b.tau = tau;
    b.mask = mask;
    b.W = p.W;
    b.status = status;
    b.timeout_ns = wait_timeout_ns();
    return launch_rows_nt<3>(b, nt, G, s);
}

cudaError_t launch_fc1_tc(const Plan& p, const __half* x, const LayerPtrs& w, const int32_t* idx,
                          const int32_t* count, const uint32_t* mask, float* part, float* h, int32_t* live,
                          cudaStream_t s) {
    int* status = status_word();
    if (status == nullptr) return cudaErrorInvalidDevice;
    const int G = p.nsm, nt = tc_tokens(p);
    TcRowsArgs a{};
    a.a0 = static_cast<const __half*>(w.w1);
    a.a1 = w.wu;
    a.idx = idx;
    a.count = count;
    a.bop = x;
    a.bop_rows = p.B;
    a.K = p.d;
    a.B = p.B;
    a.part = part;
    a.slots = slots_for(ceil_div(p.F, 128), G);
    a.status = status;
    a.timeout_ns = wait_timeout_ns();
    cudaError_t e = p.gated ? launch_rows_nt<1>(a, nt, G, s) : launch_rows_nt<0>(a, nt, G, s);
    if (e != cudaSuccess) return e;
    return launch_fc1_finish(p, nt, G, a.slots, ceil_div(p.d, 64), part, count, idx, w.b1, mask, h, live, s);
}

cudaError_t launch_fc1_tc4(const Plan& p, const __half* x, const LayerPtrs& w, const int32_t* idx,
                           const int32_t* count, const uint32_t* mask, float* part, float* h, int32_t* live,
                           cudaStream_t s) {
    int* status = status_word();
    if (status == nullptr) return cudaErrorInvalidDevice;
    const int G = p.nsm, nt = tc_tokens(p);
    TcRowsArgs a{};
    a.q = static_cast<const uint8_t*>(w.w1);
    a.qs = w.w1s;
    a.idx = idx;
    a.count = count;
    a.bop = x;
    a.bop_rows = p.B;
    a.K = p.d;
    a.B = p.B;
    a.part = part;
    a.slots = slots_for(ceil_div(p.F, 128), G);
    a.status = status;
    a.timeout_ns = wait_timeout_ns();
    cudaError_t e = launch_rows<4, 16>(a, G, s);
    if (e != cudaSuccess) return e;
    return launch_fc1_finish(p, nt, G, a.slots, p.d / 256, part, count, idx, w.b1, mask, h, live, s);
}

cudaError_t launch_fc1_finish(const Plan& p, int nt, int G, int slots, int nk, const float* part,
                              const int32_t* count, const int32_t* idx, const __half* b1, const uint32_t* mask,
                              float* h, int32_t* live, cudaStream_t s) {
    const int blocks = ceil_div(p.F, 32);
    if (p.gated)
        launch_pdl(k_fc1_finish<true, true>, blocks, 32 * p.B, 0, s, part, slots, G, nk, count, p.B, nt, idx, b1, mask,
                   p.W, h, live);
    else if (p.proj)
        launch_pdl(k_fc1_finish<false, false>, blocks, 32 * p.B, 0, s, part, slots, G, nk, count, p.B, nt, idx, b1, mask,
                   p.W, h, live);
    else
        launch_pdl(k_fc1_finish<false, true>, blocks, 32 * p.B, 0, s, part, slots, G, nk, count, p.B, nt, idx, b1, mask,
                   p.W, h, live);
    return cudaGetLastError();
}

cudaError_t launch_fc2_reduce(const Plan& p, int nt, int G, int slots, int tw, int nb, int b0, const float* part,
                              const int32_t* count, const __half* b2, float* y, cudaStream_t s) {
    const int tpb = 1024 / tw;
    launch_pdl(k_fc2_tc_reduce, dim3(p.d / tw, ceil_div(nb, tpb)), 1024, 0, s, part, slots, G, count, nb, b0, nt, p.d, tw,
                                                                        b2, y);
    return cudaGetLastError();
}

cudaError_t launch_fc2_tc4(const Plan& p, const float* h, const int32_t* idx, const int32_t* count,
                           const LayerPtrs& w, const int32_t* live, float* partial, float* y, cudaStream_t s) {
    int* status = status_word();
    if (status == nullptr) return cudaErrorInvalidDevice;
    const int G = p.nsm;
    const int slots = slots_for(p.d / 128, G);
    TcFc2qArgs a{h, idx, count, static_cast<const uint8_t*>(w.w2t), w.w2ts, live, partial, status,
                 wait_timeout_ns(), p.B, p.d, slots};
    cudaError_t e = prep(k_fc2q_tc<16>, Fc2qCfg<16>::SMEM);
    if (e != cudaSuccess) return e;
    launch_pdl(k_fc2q_tc<16>, G, kQThreads, Fc2qCfg<16>::SMEM, s, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    launch_pdl(k_fc2_tc_reduce, dim3(p.d / 128, ceil_div(p.B, 8)), 1024, 0, s, static_cast<const float*>(partial),
               slots, G, count, p.B, 0, 16, p.d, 128, w.b2, y);
    return cudaGetLastError();
}

cudaError_t launch_fc2_tc(const Plan& p, const float* h, const int32_t* idx, const int32_t* count,
                          const LayerPtrs& w, const int32_t* live, float* partial, float* y, cudaStream_t s) {
    int* status = status_word();
    if (status == nullptr) return cudaErrorInvalidDevice;
    const int G = p.nsm, nt = tc_tokens(p);
    const int slots = slots_for(p.d / 128, G);
    TcFc2Args a{h, idx, count, static_cast<const __half*>(w.w2t), live, partial, status, wait_timeout_ns(),
                p.B, p.d, slots};
    cudaError_t e;
    if (nt == 16) {
        e = prep(k_fc2_tc<16>, Fc2Cfg<16>::SMEM);
        if (e != cudaSuccess) return e;
        launch_pdl(k_fc2_tc<16>, G, kTcThreads, Fc2Cfg<16>::SMEM, s, a);
    } else {
        e = prep(k_fc2_tc<32>, Fc2Cfg<32>::SMEM);
        if (e != cudaSuccess) return e;
        launch_pdl(k_fc2_tc<32>, G, kTcThreads, Fc2Cfg<32>::SMEM, s, a);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    launch_pdl(k_fc2_tc_reduce, dim3(p.d / 128, ceil_div(p.B, 8)), 1024, 0, s, partial, slots, G, count, p.B, 0, nt, p.d,
                                                                        128, w.b2, y);
    return cudaGetLastError();
}

}  // namespace pi
