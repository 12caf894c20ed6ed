// pi_common.cuh -- small device helpers shared by the sparse-FFN kernels.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#define PI_DEV __device__ __forceinline__

namespace pi {

constexpr unsigned FULL = 0xffffffffu;

// 16-byte streaming load of read-only data that is touched once per token
// (no L1 allocation).
PI_DEV uint4 ld_stream16(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

PI_DEV uint2 ld_stream8(const void* p) {
    uint2 v;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p));
    return v;
}

// Eight binary16 values packed in a uint4 -> eight floats.
PI_DEV void h8_to_f8(const uint4& v, float (&f)[8]) {
    const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __half22float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

// Eight signed 4-bit codes of one 32-bit word (element e in bits 4e..4e+3,
// two's complement) -> exact floats, via the float whose low mantissa bits
// are the biased code: as_float(0x4B000000 | n) == 2^23 + n.
PI_DEV void q8_to_f8(uint32_t w, float (&f)[8]) {
    const uint32_t u = w ^ 0x88888888u;  // n = code + 8, in 0..15
#pragma unroll
    for (int e = 0; e < 8; ++e)
        f[e] = __uint_as_float(((u >> (4 * e)) & 0xFu) | 0x4B000000u) - 8388616.0f;
}

// f32 result of a*b + c for binary16 a and b (the low 16 bits of a16, b16):
// the product is exact, so this equals fmaf on the values widened to fp32.
PI_DEV float fma_h(uint32_t a16, uint32_t b16, float c) {
    float d;
    const unsigned short a = (unsigned short)a16, b = (unsigned short)b16;
    asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
    return d;
}
// dot of 8 fp16 weights with 8 fp16 x values: exact products summed in
// element order in fp32, with no conversion instructions
PI_DEV float dot8hh(const uint4& w, const uint4& x) {
    float acc = fma_h(w.x, x.x, -0.f);
    acc = fma_h(w.x >> 16, x.x >> 16, acc);
    acc = fma_h(w.y, x.y, acc);
    acc = fma_h(w.y >> 16, x.y >> 16, acc);
    acc = fma_h(w.z, x.z, acc);
    acc = fma_h(w.z >> 16, x.z >> 16, acc);
    acc = fma_h(w.w, x.w, acc);
    acc = fma_h(w.w >> 16, x.w >> 16, acc);
    return acc;
}
// dot of 8 INT4 codes (element e in bits 4e..4e+3, two's complement) with 8
// fp16 x values.  A code pair becomes exact fp16 integers without
// conversions: with n = q + 8, the half 0x6400 | n holds 1024 + n, and one
// half-precision subtraction of 1032 leaves q.  The pairs are elements
// (e, e + 4), which sit 16 bits apart in the word; the products are summed in
// element order.
PI_DEV float dotq8h(uint32_t cw, const uint4& x) {
    const uint32_t u = cw ^ 0x88888888u;
    const __half2 k = __halves2half2(__ushort_as_half((unsigned short)0x6408u), __ushort_as_half((unsigned short)0x6408u));
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t m = ((u >> (4 * i)) & 0x000F000Fu) | 0x64006400u;
        const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&m), k);
        q[i] = *reinterpret_cast<const uint32_t*>(&v);
    }
    float acc = fma_h(q[0], x.x, -0.f);         // element 0
    acc = fma_h(q[1], x.x >> 16, acc);           // 1
    acc = fma_h(q[2], x.y, acc);                 // 2
    acc = fma_h(q[3], x.y >> 16, acc);           // 3
    acc = fma_h(q[0] >> 16, x.z, acc);           // 4
    acc = fma_h(q[1] >> 16, x.z >> 16, acc);     // 5
    acc = fma_h(q[2] >> 16, x.w, acc);           // 6
    acc = fma_h(q[3] >> 16, x.w >> 16, acc);     // 7
    return acc;
}

// Halving butterfly over a warp for 16 rows: v[k] is this lane's partial sum
// of row k.  After the step with offset o a lane keeps the half of its values
// selected by its bit o and adds the partner's copy of them, so on return
// lanes L and L ^ 1 hold the warp's total of row fold16_row(L) (a fixed order:
// 16 shuffles for 16 rows).
PI_DEV int fold16_row(int lane) {
    return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
}
PI_DEV float fold16(float (&v)[16], int lane) {
#pragma unroll
    for (int n = 8, o = 16; n >= 1; n /= 2, o /= 2) {
        const bool hi = lane & o;
#pragma unroll
        for (int k = 0; k < n; ++k) {
            const float send = hi ? v[k] : v[k + n];
            const float keep = hi ? v[k + n] : v[k];
            v[k] = keep + __shfl_xor_sync(FULL, send, o);
        }
    }
    return v[0] + __shfl_xor_sync(FULL, v[0], 1);
}

// Programmatic dependent launch: a kernel launched with launch_pdl may be
// scheduled while the previous kernel on its stream is still running.  Its
// first statement waits until that kernel has completed and its memory is
// visible, then lets the next kernel be scheduled in turn.  Nothing before
// it reads another kernel's output or writes global memory.
PI_DEV void pdl_entry() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
}

PI_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    return v;
}

}  // namespace pi
