// Layout shared by the block-scaled decode rail's kernels (T <= 8 tokens on
// prepacked weights): the decode prologue in route_bucket.cu writes the x
// operand in this layout, the expert kernels in decode_mx.cu read it and write
// the down operand in it.
//
// An activation operand chunk (128 K positions) is a block of npad rows, row
// n = t * kDecTerms + term for token t and E2M1 term `term` (rows past
// T * kDecTerms are zero), of four 32-blocks of 16 bytes in the MXFP4 byte
// layout (byte i = column i low nibble, column 16 + i high nibble), so that the
// MMA pairs every activation code with the weight code of the same column. A
// chunk is stored as the 64-byte-swizzled image the MMA reads (block kb of row
// n at n*64 + 16*(kb ^ ((n >> 1) & 3))): one contiguous copy of npad * 64 bytes
// lands it in shared memory ready for the MMA. Its E8M0 scales form one
// 512-byte atom per chunk: byte 16*(n%32) + 4*(n/32) + kb for row n and K-block
// kb, the order tcgen05.cp.32x128b.warpx4 copies into tensor memory.
#pragma once

#include <cstdint>

namespace moe {
namespace dmx {

// E2M1 terms per activation on the decode rail: x enters gate/up as eight
// terms and w*h enters down as eight (each term takes about 2.5 bits of the
// residual: eight leave ~1e-7 of the block's largest value).
constexpr int kDecTerms = 8;

__host__ __device__ inline int npad_for(int T) { return ((T * kDecTerms + 15) / 16) * 16; }

// Byte offset of (row n, K-block kb, byte i) inside an operand chunk of npad * 64 bytes.
__host__ __device__ inline int chunk_off(int n, int kb, int i) { return n * 64 + 16 * (kb ^ ((n >> 1) & 3)) + i; }
// Byte offset of (row n, K-block kb in 0..3) inside a 512-byte scale atom.
__host__ __device__ inline int atom_off(int n, int kb) { return 16 * (n & 31) + 4 * (n >> 5) + kb; }

}  // namespace dmx
}  // namespace moe
