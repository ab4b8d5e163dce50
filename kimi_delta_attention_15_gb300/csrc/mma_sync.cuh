// Warp-level tf32 MMA (m16n8k8) for the small 16x16 blocks of the chunk
// algorithm, whose operands are built in registers with per-block decay
// factors. Fragment layout (PTX ISA, mma.m16n8k8 .tf32), g = lane / 4,
// t = lane % 4:
//   A 16x8 row-major: a0 (g, t), a1 (g+8, t), a2 (g, t+4), a3 (g+8, t+4)
//   B 8x8  col-major: b0 (k=t, n=g), b1 (k=t+4, n=g)
//   C 16x8:           c0 (g, 2t), c1 (g, 2t+1), c2 (g+8, 2t), c3 (g+8, 2t+1)
#pragma once
#include <cstdint>

namespace kda {

// x rounded to tf32 (nearest, ties away from zero), as bits: the same rounding as
// tf32_round_bits in umma.cuh, and as the cvt.rna.tf32.f32 conversion
__device__ __forceinline__ uint32_t tf32_bits(float x) {
    return (__float_as_uint(x) + (x != x ? 0u : 0x1000u)) & 0xffffe000u;
}

__device__ __forceinline__ void mma_tf32_16x8x8(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace kda

namespace kda {

// Operands split exactly by masking: x = hi + lo, hi = x with the 13 mantissa bits below
// tf32 cleared, lo = x - hi (exact in fp32).
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
    hi = __float_as_uint(x) & 0xffffe000u;
    lo = __float_as_uint(x - __uint_as_float(hi));
}
// Single tf32 products, for products whose outputs stay well inside their tolerances
// without the split (measured against the fp64 reference): the fp32 operands go in
// unconverted and the tensor core reads their top 19 bits (truncation toward zero),
// which costs no instruction.
struct Frag4t { uint32_t r[4]; };
struct Frag2t { uint32_t r[2]; };
__device__ __forceinline__ Frag4t frag4t(float a0, float a1, float a2, float a3) {
    return Frag4t{{__float_as_uint(a0), __float_as_uint(a1), __float_as_uint(a2), __float_as_uint(a3)}};
}
__device__ __forceinline__ Frag2t frag2t(float b0, float b1) { return Frag2t{{__float_as_uint(b0), __float_as_uint(b1)}}; }
__device__ __forceinline__ void mma1(float (&c)[4], const Frag4t& a, const Frag2t& b) {
    mma_tf32_16x8x8(c, a.r[0], a.r[1], a.r[2], a.r[3], b.r[0], b.r[1]);
}
__device__ __forceinline__ void mma1(float (&c)[4], const Frag4t& a, uint32_t b0, uint32_t b1) {
    mma_tf32_16x8x8(c, a.r[0], a.r[1], a.r[2], a.r[3], b0, b1);
}

// Fragments straight from shared memory with ldmatrix: an 8x8 b16 matrix is an 8x4
// tile of 32-bit values, and lane i receives the word (row i/4, column i%4) of each
// matrix, the layout of the tf32 A and B fragments. Every lane passes the address of
// one 16-byte row (lanes 8m .. 8m+7: the rows of matrix m).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* row) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(row))));
}
// A fragment (16 x 8, rows r0.., columns k0..) of a row-major fp32 tile with row
// stride ld floats (16-byte aligned rows), as fp32 bit patterns
__device__ __forceinline__ Frag4t ldsm_a(const float* tile, int ld, int r0, int k0) {
    const int lane = threadIdx.x & 31, m = lane >> 3;
    Frag4t f;
    ldsm_x4(f.r, tile + (size_t)(r0 + (m & 1) * 8 + (lane & 7)) * ld + k0 + (m >> 1) * 4);
    return f;
}
// B fragments of the n-tiles n0.. and n0+8.. at columns k0.. of a tile stored with
// n as its row index (row stride ld floats), as fp32 bit patterns
__device__ __forceinline__ void ldsm_b2(Frag2t& b0, Frag2t& b1, const float* tile, int ld, int n0, int k0) {
    const int lane = threadIdx.x & 31, m = lane >> 3;
    uint32_t r[4];
    ldsm_x4(r, tile + (size_t)(n0 + (m >> 1) * 8 + (lane & 7)) * ld + k0 + (m & 1) * 4);
    b0 = Frag2t{{r[0], r[1]}};
    b1 = Frag2t{{r[2], r[3]}};
}


}  // namespace kda

#include <cuda_bf16.h>
namespace kda {
// About fp32-accurate products in two MMAs ("tf32 + bf16 cross terms"), where the gate
// gradient needs more than tf32: with the masked split a = a_hi + a_lo, b = b_hi + b_lo,
//   a b ~ a_hi b_hi            (one tf32 m16n8k8 product, exact operands)
//       + a b_lo + a_lo b      (one bf16 m16n8k16 product: the two cross terms side by side
//                               along k, a and b_lo in the first 8 slots, a_lo and b in the
//                               last 8)
// The cross terms are 2^-11 of the product, so their bf16 operands (8 bits) leave an error
// of about 2^-20 of a b, the accuracy of the three-product "3xTF32" split (hi hi + hi lo +
// lo hi) at two thirds of its MMAs; the measured output errors against the fp64 reference
// are the same. The bf16 k slots are permuted so that each thread's bf16 pairs are exactly
// the values of its tf32 fragments: slot 2t <-> k = t, slot 2t+1 <-> k = t+4 (fragment
// layouts of mma.m16n8k16 .bf16, PTX ISA).
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
struct Frag4x { uint32_t hi[4], lo[4], bf[4]; };   // bf: [a | a_lo] pairs (k = t, t + 4)
struct Frag2x { uint32_t hi[2], bf[2]; };
__device__ __forceinline__ Frag4x frag4x(float a0, float a1, float a2, float a3) {
    Frag4x f;
    split_tf32(a0, f.hi[0], f.lo[0]); split_tf32(a1, f.hi[1], f.lo[1]);
    split_tf32(a2, f.hi[2], f.lo[2]); split_tf32(a3, f.hi[3], f.lo[3]);
    f.bf[0] = pack_bf16(a0, a2);
    f.bf[1] = pack_bf16(a1, a3);
    f.bf[2] = pack_bf16(__uint_as_float(f.lo[0]), __uint_as_float(f.lo[2]));
    f.bf[3] = pack_bf16(__uint_as_float(f.lo[1]), __uint_as_float(f.lo[3]));
    return f;
}
__device__ __forceinline__ Frag2x frag2x(float b0, float b1) {
    Frag2x f;
    uint32_t l[2];
    split_tf32(b0, f.hi[0], l[0]); split_tf32(b1, f.hi[1], l[1]);
    f.bf[0] = pack_bf16(__uint_as_float(l[0]), __uint_as_float(l[1]));
    f.bf[1] = pack_bf16(b0, b1);
    return f;
}
__device__ __forceinline__ void mma_bf16_16x8x16(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
__device__ __forceinline__ void mma2x(float (&c)[4], const Frag4x& a, const Frag2x& b) {
    mma_bf16_16x8x16(c, a.bf, b.bf);
    mma_tf32_16x8x8(c, a.hi[0], a.hi[1], a.hi[2], a.hi[3], b.hi[0], b.hi[1]);
}
}  // namespace kda
