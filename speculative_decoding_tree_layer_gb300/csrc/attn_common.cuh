// attn_common.cuh -- pieces shared by the attention tree-verify kernels:
// exact conversion of int8 / 4-bit codes to fp16 and the block quantiser
// that writes the tree's keys and values into the cache (the cluster and
// distributed-shared-memory helpers come from cluster.cuh).
#pragma once

#include "cluster.cuh"
#include "common.cuh"

namespace dflv {
namespace attn {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- exact code -> fp16
// fp16 with exponent field 25 (0x6400 = 1024) has unit spacing on
// [1024, 2048): the bit pattern 0x6400 | u is exactly 1024 + u for u < 1024.
DFLV_DEVINL uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
// four int8 codes -> {c0,c1}, {c2,c3} as exact fp16x2
DFLV_DEVINL void i8x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;  // code + 128 in [1, 255]
    const uint32_t l = prmt(u, 0x64646464u, 0x5140u);
    const uint32_t h = prmt(u, 0x64646464u, 0x5342u);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    __half2 lh = __hsub2(*reinterpret_cast<const __half2*>(&l), bias);
    __half2 hh = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
    lo = *reinterpret_cast<uint32_t*>(&lh);
    hi = *reinterpret_cast<uint32_t*>(&hh);
}
// four 4-bit codes (one per byte, low nibble) -> value - 8 as exact fp16x2
DFLV_DEVINL void u4x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t l = prmt(w, 0x64646464u, 0x5140u);
    const uint32_t h = prmt(w, 0x64646464u, 0x5342u);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1032
    __half2 lh = __hsub2(*reinterpret_cast<const __half2*>(&l), bias);
    __half2 hh = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
    lo = *reinterpret_cast<uint32_t*>(&lh);
    hi = *reinterpret_cast<uint32_t*>(&hh);
}

// ---------------------------------------------------------------- block quantiser
// One 32-value block of a tree row (bf16) -> codes + fp16 scale in the cache.
template <int TYPE>
DFLV_DEVINL void quantize_block(const uint16_t* __restrict__ src, uint8_t* __restrict__ codes,
                                uint16_t* __restrict__ scale) {
    float x[32];
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(src + j));
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            x[j + 2 * e] = bf16_bits_to_float((uint16_t)(ww[e] & 0xffff));
            x[j + 2 * e + 1] = bf16_bits_to_float((uint16_t)(ww[e] >> 16));
        }
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(x[j]));
    constexpr float qmax = (TYPE == DFLV_KV_Q8_0) ? 127.f : 7.f;
    const float d = __fdiv_rn(amax, qmax);
    const float id = (d != 0.f) ? __frcp_rn(d) : 0.f;
    *scale = __half_as_ushort(__float2half_rn(d));
    if constexpr (TYPE == DFLV_KV_Q8_0) {
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float r = fminf(fmaxf(roundf(__fmul_rn(x[j], id)), -127.f), 127.f);
            const uint32_t c = (uint32_t)(uint8_t)(int8_t)(int)r;
            if ((j & 3) == 0) w[j >> 2] = 0;
            w[j >> 2] |= c << (8 * (j & 3));
        }
        reinterpret_cast<uint4*>(codes)[0] = make_uint4(w[0], w[1], w[2], w[3]);
        reinterpret_cast<uint4*>(codes)[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
        uint32_t code[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
            code[j] = (uint32_t)((int)fminf(fmaxf(roundf(__fmul_rn(x[j], id)), -8.f), 7.f) + 8);
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if ((j & 3) == 0) w[j >> 2] = 0;
            w[j >> 2] |= (code[j] | (code[j + 16] << 4)) << (8 * (j & 3));
        }
        *reinterpret_cast<uint4*>(codes) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}


}  // namespace attn
}  // namespace dflv
