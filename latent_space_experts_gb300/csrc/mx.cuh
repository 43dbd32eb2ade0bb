// MXFP8 activations and the block-scaled tensor-core MMA of the MXFP4 layer ("Stable Latent
// MoE" concept note, 训练基础设施: MXFP4 weights with MXFP8 activations), sm_103a.
//
// MXFP8 here is the OCP Microscaling block format with FP8 E4M3 elements: 32 consecutive
// values along K share the scale 2^e, e = floor(log2 max |v|) - 8 (8 = the largest E4M3
// exponent), clamped to [-127, 127] (-127 for an all-zero block), stored as the E8M0 byte
// e + 127; each value is v * 2^-e rounded to the nearest E4M3 value, ties to the even
// mantissa, saturating at 448.
//
// The MMA is tcgen05.mma kind::mxf8f6f4 with block scaling: A = E2M1 weights (expanded by TMA
// into one byte per value, 16 values in each 16-byte chunk), B = E4M3 activations, K = 32 per
// instruction, one E8M0 scale per row of A and per column of B for those 32 values.  Scales
// live in tensor memory, four bytes (four K = 32 steps) to a 32-bit column:
//   A: row r of the M = 128 tile at lane r, column base + r / 32;
//   B: column n of the tile at lane 32 q + n % 32 of every lane quadrant q, column base + n / 32;
// the byte is picked by the scale-ID fields of the instruction descriptor.
#pragma once

#include <stdint.h>

namespace slmoe {

// E8M0 exponent e of an MXFP8 block from its largest magnitude (fp32): the exponent field
// minus 127 + 8; a zero or subnormal maximum (field 0) gives -127.  (Finite inputs: the
// field is at most 254, so e <= 119.)
__device__ __forceinline__ int mx8_exp(float amax) {
    const int e = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 135;
    return e < -127 ? -127 : e;
}
// 2^-e for e in [-127, 119] (a normal fp32 number).
__device__ __forceinline__ float mx8_inv_scale(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }
// Two fp32 values -> two E4M3 codes (round to nearest even, saturating): lo in bits 0..7.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
// One block of 32 values held by one thread: 8 words of codes (value 4i + j in byte j of
// word i) and the returned E8M0 byte.  v * 2^-e is exact (a power-of-two scaling; a result
// below the fp32 normal range is far below E4M3's smallest value and rounds to zero anyway).
__device__ __forceinline__ uint32_t mx8_quant32(const float (&v)[32], uint32_t (&w)[8]) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int e = mx8_exp(amax);
    const float s = mx8_inv_scale(e);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        w[i] = e4m3x2(v[4 * i] * s, v[4 * i + 1] * s) | (e4m3x2(v[4 * i + 2] * s, v[4 * i + 3] * s) << 16);
    return (uint32_t)(e + 127);
}

// Instruction descriptor of kind::mxf8f6f4 with block scaling: A E2M1 and B E4M3, both
// K-major, E8M0 scales, fp32 D, shape M x N; id = the byte of the scale columns (the K = 32
// step inside a 128-wide K block).
__host__ __device__ constexpr uint32_t idesc_mx(int M, int N, int id) {
    return ((uint32_t)id << 4) | (5u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
           ((uint32_t)(M >> 4) << 24) | ((uint32_t)id << 29);
}
__device__ __forceinline__ void umma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}
// Stores of one / eight 32-bit TMEM columns in this thread's lane (warp-wide, the warp's
// lane quadrant).
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

}  // namespace slmoe
