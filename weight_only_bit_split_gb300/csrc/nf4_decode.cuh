// NF4 code decoding shared by the tensor-core NF4 kernels: a 16-entry f16
// codebook held as byte planes in registers, and the byte-permute lookup of
// eight 4-bit codes at a time (bitsandbytes issue #1842: codes index a
// 16-entry codebook; two codes per byte, the first element in the high
// nibble).
#pragma once

#include <cstdint>

namespace wobs {

// PTX prmt, default mode: selector nibble bits 0-2 pick one of the eight
// source bytes, bit 3 replicates that byte's sign bit over the result byte.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
// Codebook held as byte planes: lo/hi bytes of the f16 entries 0..7 (A) and
// 8..15 (B), two registers each.
struct Planes {
  uint32_t la0, la1, lb0, lb1, ha0, ha1, hb0, hb1;
};

// Byte planes of a 16-entry f16 table given as eight f16x2 words (word i =
// entries 2i in the low half, 2i + 1 in the high half).
__device__ __forceinline__ Planes planes_from_pairs(const uint32_t (&w)[8]) {
  Planes p;
  p.la0 = prmt(w[0], w[1], 0x6420u);
  p.ha0 = prmt(w[0], w[1], 0x7531u);
  p.la1 = prmt(w[2], w[3], 0x6420u);
  p.ha1 = prmt(w[2], w[3], 0x7531u);
  p.lb0 = prmt(w[4], w[5], 0x6420u);
  p.hb0 = prmt(w[4], w[5], 0x7531u);
  p.lb1 = prmt(w[6], w[7], 0x6420u);
  p.hb1 = prmt(w[6], w[7], 0x7531u);
  return p;
}

// Register variant: the low 3 bits of each code select a byte in the A and B
// planes, the high bit (spread to a byte mask by sign replication) picks A or
// B, and byte permutes pair the low and high bytes into f16 values.
__device__ __forceinline__ void decode_planes(uint32_t w, const Planes& p, uint32_t (&r)[4]) {
  const uint32_t s = w & 0x77777777u;
  const uint32_t w4 = w << 4;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t sel = h ? (s >> 16) : s;
    const uint32_t m = prmt(w4, w, h ? 0xFBEAu : 0xD9C8u);   // byte i = 0xFF where code i >= 8
    const uint32_t la = prmt(p.la0, p.la1, sel), lb = prmt(p.lb0, p.lb1, sel);
    const uint32_t ha = prmt(p.ha0, p.ha1, sel), hb = prmt(p.hb0, p.hb1, sel);
    const uint32_t lo = (la & ~m) | (lb & m);
    const uint32_t hi = (ha & ~m) | (hb & m);
    r[2 * h] = prmt(lo, hi, 0x4051u);
    r[2 * h + 1] = prmt(lo, hi, 0x6273u);
  }
}

}  // namespace wobs
