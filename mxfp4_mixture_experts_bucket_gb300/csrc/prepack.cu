// Prepacked MXFP4 weights for the block-scaled tensor-core rails.
//
// The weights stay MXFP4 ("dasLLAMA: dig the last two board reds green",
// section "gpt-oss: mx4 kernels to the lab-winning shape": blocks of 32 E2M1
// codes sharing one E8M0 exponent); only their placement in memory changes, so
// that one contiguous bulk copy brings a weight tile into shared memory in the
// operand layout of tcgen05.mma kind::mxf4 (64-byte-swizzled rows, so that the
// tensor core's reads of eight rows spread over all shared-memory banks) and
// one 512-byte copy its scales.
//
//   qs_p: tile by tile, NK = ceil(C/128) chunks of 64 bytes per row: expert e,
//        128-row tile t (rows_t = 128, or R - 128t for the last tile) starts at
//        byte (e*R + 128t) * NK*64; inside it chunk j (columns 128j..128j+127)
//        starts at rows_t * 64 * j and is the 64-byte-swizzled image of its
//        rows: block kb of tile row m at m*64 + 16*(kb ^ ((m >> 1) & 3)), the 16
//        bytes as stored (byte i = column i low nibble, column 16+i high);
//        blocks past C/32 are zero.
//   sf_p [E][ceil(R/128)][NK][512], NK = ceil(C/128): one atom per tile and
//        chunk, byte 16*(m%32) + 4*(m/32) + kb = E8M0 of tile row m, block
//        4j+kb; 127 (a scale of 1) where the row or the block does not exist.
//
// The source may hold two matrices' rows interleaved (gate/up of gpt-oss, one
// [2R][C] plane per expert): with row stride rs = 2 row r of the matrix is
// source row 2r of the plane starting at `qs` (pass qs one row further for
// the odd rows).
//
// The atom is the order tcgen05.cp.32x128b.warpx4 copies into tensor memory
// (32 rows of 16 bytes, each row replicated into the four lane quarters): row m
// of the tile then finds its four scale bytes in lane m, column m/32.
#include "moe_common.cuh"

namespace moe {

// One thread per 16-byte block of the output (expert e, row, block b < 4*NK):
// the stored block, or zero past the last column.
__global__ void __launch_bounds__(256) prepack_qs_kernel(const uint8_t* __restrict__ qs, int E, int R, int C,
                                                         int rs, uint8_t* __restrict__ qs_p) {
  const int nb = C / 32, NK = (C + 127) / 128, nbp = 4 * NK;
  const size_t total = (size_t)E * R * nbp;
  for (size_t p = (size_t)blockIdx.x * blockDim.x + threadIdx.x; p < total; p += (size_t)gridDim.x * blockDim.x) {
    const int b = (int)(p % nbp);
    const size_t er = p / nbp;
    const int row = (int)(er % R);
    const int e = (int)(er / R);
    const int t = row >> 7, m = row & 127;
    const int rows_t = min(128, R - 128 * t);
    const int j = b >> 2, kb = b & 3;
    const size_t dst = ((size_t)e * R + 128 * (size_t)t) * ((size_t)NK * 64) + (size_t)rows_t * 64 * j +
                       (size_t)(m * 64 + 16 * (kb ^ ((m >> 1) & 3)));
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (b < nb) v = __ldg(reinterpret_cast<const uint4*>(qs + ((size_t)e * R + row) * rs * (C / 2)) + b);
    *reinterpret_cast<uint4*>(qs_p + dst) = v;
  }
}

__global__ void __launch_bounds__(256) prepack_sf_kernel(const uint8_t* __restrict__ sc, int E, int R, int C,
                                                         int rs, uint8_t* __restrict__ sf_p) {
  const int NK = (C + 127) / 128, nb = C / 32, NT = (R + 127) / 128;
  const size_t total = (size_t)E * NT * NK * 512;
  for (size_t p = (size_t)blockIdx.x * blockDim.x + threadIdx.x; p < total; p += (size_t)gridDim.x * blockDim.x) {
    const int byte = (int)(p & 511);
    size_t rest = p >> 9;
    const int j = (int)(rest % NK);
    rest /= NK;
    const int t = (int)(rest % NT);
    const int e = (int)(rest / NT);
    const int l = byte >> 4, q = (byte >> 2) & 3, kb = byte & 3;
    const int row = 128 * t + 32 * q + l, b = 4 * j + kb;
    uint8_t v = 127;
    if (row < R && b < nb) v = sc[((size_t)e * R + row) * rs * nb + b];
    sf_p[p] = v;
  }
}

size_t packed_qs_bytes(int E, int R, int C) { return (size_t)E * R * ((C + 127) / 128) * 64; }
size_t packed_sf_bytes(int E, int R, int C) {
  return (size_t)E * ((R + 127) / 128) * ((C + 127) / 128) * 512;
}

cudaError_t launch_prepack(const uint8_t* qs, const uint8_t* sc, int E, int R, int C, uint8_t* qs_p,
                           uint8_t* sf_p, Launch L, int rs) {
  const int cap = device_sm_count() * 8;
  auto blocks_for = [&](size_t n) {
    size_t b = (n + 255) / 256;
    if (b > (size_t)cap) b = cap;
    return (int)(b < 1 ? 1 : b);
  };
  const size_t nq = (size_t)E * R * ((C + 127) / 128) * 4, ns = packed_sf_bytes(E, R, C);
  cudaError_t err = launch_kernel(prepack_qs_kernel, dim3(blocks_for(nq)), dim3(256), 0, L, qs, E, R, C, rs, qs_p);
  if (err != cudaSuccess) return err;
  return launch_kernel(prepack_sf_kernel, dim3(blocks_for(ns)), dim3(256), 0, L, sc, E, R, C, rs, sf_p);
}

}  // namespace moe
