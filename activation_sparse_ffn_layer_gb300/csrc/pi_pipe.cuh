// pi_pipe.cuh -- device helpers of the streamed batched kernels (pi_tc.cu,
// pi_stream.cu): mbarriers with bounded waits, cp.async copies, the loaders'
// uniform-abort barrier, and the stream-K work split with its fixed-order
// partial sums.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pi_common.cuh"
#include "../../include/pi.h"

namespace pi {
namespace pipe {

PI_DEV unsigned long long wall_ns() {
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
// One arrival per warp on a barrier that counts warps: __syncwarp orders
// every lane's prior shared-memory writes (cp.async results its own wait has
// completed, or stores it fenced for the async proxy) before lane 0's
// release.  A hundred arrivals on one barrier word would serialise.
PI_DEV void warp_arrive(unsigned long long* b) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) bar_arrive(b);
}
// one arrival that also expects `bytes` of asynchronous copies (TMA) on the barrier
PI_DEV void bar_arrive_expect_tx(unsigned long long* b, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
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
    const unsigned long long t0 = wall_ns();
    for (;;) {
        if (bar_try(b, parity)) return true;
        if (*(volatile int*)c.abort_flag) return false;
        if ((long long)(wall_ns() - t0) > c.timeout_ns) {
            atomicExch(c.status, (int)PI_ERR_TIMEOUT);
            *(volatile int*)c.abort_flag = 1;
            return false;
        }
    }
}
// Bounded wait that ignores the abort flag (used while draining).
PI_DEV void bar_drain(unsigned long long* b, unsigned parity, long long timeout_ns) {
    const unsigned long long t0 = wall_ns();
    while (!bar_try(b, parity) && (long long)(wall_ns() - t0) <= timeout_ns) {
    }
}

// cp.async copies carry no compiler memory clobber: their shared-memory
// results are only read after cp_wait / cp_wait_all (which have one), and
// leaving it off lets the compiler keep row ids in registers across copies.
PI_DEV void cp16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(su32(dst)), "l"(src));
}
PI_DEV void cp4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(su32(dst)), "l"(src));
}
PI_DEV void cp8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(su32(dst)), "l"(src));
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

PI_DEV unsigned char* align1024(unsigned char* p) {
    return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

struct Span {
    int tile, kc0, kc1;
};

// The CTAs of a stream-K split (CTA g owns units [U*g/G, U*(g+1)/G)) that
// touch tile `tile` (units [tile*nk, (tile+1)*nk)) form one contiguous range
// [rng[0], rng[1]]; slot[g] is the partial slot CTA g wrote for the tile (-1:
// empty share).  All threads of the block take part; the caller syncs after.
constexpr int kMaxCtas = 1024;
PI_DEV void cover_setup(long long U, int G, int nk, int tile, int* slot, int* rng) {
    const long long lo = (long long)tile * nk, hi = lo + nk;
    if (threadIdx.x == 0) {
        rng[0] = G;
        rng[1] = -1;
    }
    __syncthreads();
    for (int g = threadIdx.x; g < G && g < kMaxCtas; g += blockDim.x) {
        const long long u0 = U * g / G, u1 = U * (g + 1) / G;
        const bool hit = u0 < u1 && u0 < hi && u1 > lo;
        slot[g] = hit ? tile - (int)(u0 / nk) : -1;
        if (hit) {
            atomicMin(&rng[0], g);
            atomicMax(&rng[1], g);
        }
    }
}

// Ascending-CTA sum; loads go out eight at a time so their latencies overlap.
PI_DEV float sum_cover(const float* __restrict__ part, const int* slot, const int* rng, int slots, int cols,
                       int col, int m, int tw = 128) {
    float acc = 0.f;
    for (int g0 = rng[0]; g0 <= rng[1]; g0 += 8) {
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int g = g0 + k;
            const int sl = g <= rng[1] ? slot[g] : -1;
            v[k] = (sl >= 0 && sl < slots) ? __ldcg(part + (((size_t)g * slots + sl) * cols + col) * tw + m) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) acc += v[k];
    }
    return acc;
}

}  // namespace pipe
}  // namespace pi
