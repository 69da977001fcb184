// Register-level tensor-core fragments shared by the kernels that multiply NVFP4 weights held in
// registers (mma.sync m16n8k16, f16 operands, fp32 accumulation): the one-launch decode kernel
// and the narrow-group arm of the tcgen05 grouped GEMM.
#pragma once
#include "internal.cuh"

namespace moe {

// D += A B for one m16n8k16 tile.  Fragment layout (lane = 4 * grp + tig): A registers {row grp,
// K 2tig..+1}, {row grp + 8, same K}, {row grp, K 2tig + 8..+9}, {row grp + 8, same K}; B registers
// {K 2tig..+1, column grp}, {K 2tig + 8..+9, column grp}; D {row grp, columns 2tig, 2tig + 1},
// {row grp + 8, same}.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two e4m3 bytes of w as an f16x2 pair of their values times 2^-8 (sel = 0x0404 | lo << 4 |
// hi << 12 puts byte lo into the low half and byte hi into the high half), with integer
// operations only: a byte's seven low bits placed at f16 bits 7..13 make the f16 exponent field
// the e4m3 exponent and the f16 mantissa's top bits the e4m3 mantissa, so every finite code,
// subnormals included, maps exactly to its value x 2^-8 (the biases differ by 8); the sign goes
// to bit 15.  Callers multiply their results by 2^8.
__device__ __forceinline__ __half2 e4m3_pair_f16x2_2m8(uint32_t w, uint32_t sel) {
  const uint32_t b = __byte_perm(w, 0u, sel);   // [0, lo, 0, hi]: each byte in its half's high byte
  const uint32_t f = (b & 0x80008000u) | ((b >> 1) & 0x3FFF3FFFu);
  return *reinterpret_cast<const __half2*>(&f);
}
constexpr float kScaleUnbias = 256.0f;   // 2^8, undoes the scales' 2^-8

// The lane's selector for e4m3_pair_f16x2_2m8 over a 32-bit word of block scales that covers two
// 32-element pieces (64 K): piece 2p + s of the word uses block 2 (2p + s) + tig / 2, i.e. byte
// 2 s + tig / 2 of the word -- the low half for the even piece, the high half for the odd one.
__device__ __forceinline__ uint32_t scale_pair_sel(int tig) {
  return 0x0404u | (static_cast<uint32_t>(tig >> 1) << 4) | ((2u + static_cast<uint32_t>(tig >> 1)) << 12);
}

// K order of the MMAs over a 16-byte piece of a weight row (32 elements, two NVFP4 blocks): lane
// tig of a quad takes the piece's word tig, i.e. elements 8 tig .. 8 tig + 7, of which the first
// MMA of the piece uses 8 tig .. + 3 as its K positions (2 tig, 2 tig + 1 | 2 tig + 8, 2 tig + 9)
// and the second MMA 8 tig + 4 .. + 7.  The B operand is read in the same order (the lane's 16
// bytes of activations at elements 8 tig .. 8 tig + 7 of the piece), so each dot product is the
// piece's own; the lane's elements all lie in block 2 q + tig / 2 of piece q and share one scale.
// w: the lane's word of the row, s: the scale in both halves; r[0], r[1] feed the first MMA,
// r[2], r[3] the second (e2m1 x e4m3 is exact in f16).
__device__ __forceinline__ void piece_frag(uint32_t w, __half2 s, uint32_t (&r)[4]) {
  e2m1x8_to_f16x2(w, r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 p = __hmul2(*reinterpret_cast<const __half2*>(&r[i]), s);
    r[i] = *reinterpret_cast<const uint32_t*>(&p);
  }
}

}  // namespace moe
