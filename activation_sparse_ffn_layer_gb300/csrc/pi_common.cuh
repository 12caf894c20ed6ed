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

PI_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    return v;
}

}  // namespace pi
