// MXFP8 (OCP Microscaling Formats v1.0, MXFP8 E4M3): shared definitions of the kernels
// that write or read MX data (dispatch, the offline weight quantiser, the grouped GEMM).
//
// Scale of a 1x32 block: X = 2^s with s = floor(log2(amax)) - 8 (8 = exponent of 448, the
// largest e4m3 normal), clamped to [-127, 127]; stored as the UE8M0 code s + 127. An
// all-zero block takes s = -127. Elements are e4m3_rn_satfinite(v * 2^-s).
//
// Scale atoms: the codes of a matrix with K columns are kept in 512-byte atoms of 128 rows
// x one 128-column K stage (four blocks of 32). Atom (a, ks) starts at byte
// (a * (K / 128) + ks) * 512, and row i of the atom's 128, block kb of the stage's four, is
// at byte (i % 32) * 16 + (i / 32) * 4 + kb. That is the order in which the block-scaled
// tcgen05.mma (M = 128, scale_vec::1X) reads scale factors from tensor memory after one
// tcgen05.cp 32x128b.warpx4 of the atom: the copy gives every lane quarter the atom's 32 x
// 16 bytes, and rows 32q..32q+31 read column q, byte = the MMA's scale-factor id.
//
// Atom rows of a grouped matrix: group g (routed expert g < E, or the shared expert g = E
// with offsets[E] = T*k) starts at atom row ceil((offsets[g] + 127 * g) / 128), so every
// group's first row begins an atom of its own and groups never share one; row r of group g
// is row (r - offsets[g]) % 128 of atom row base(g) + (r - offsets[g]) / 128.
#pragma once

#include <stdint.h>

#include "moe_internal.cuh"

namespace moe {

__host__ __device__ __forceinline__ int64_t mx_group_atom_base(int64_t group_offset, int g) {
  return (group_offset + 127 * (int64_t)g + 127) / 128;
}

// Atom rows the activations of a layer need (dispatched rows, or h).
inline int64_t mx_act_atom_rows(const moe_config_t& c) {
  return ceil_div(routed_rows(c) + 127 * (int64_t)c.E, 128) + (c.n_shared ? ceil_div(c.T, 128) : 0) + 2;
}

// Byte offset of (atom row a, stage ks, atom row-in-tile i) for a K of ks_total stages;
// add the block index kb (0..3) inside the stage.
__host__ __device__ __forceinline__ int64_t mx_atom_byte(int64_t a, int ks, int ks_total, int i) {
  return ((a * ks_total + ks) << 9) + (i & 31) * 16 + (i >> 5) * 4;
}

#ifdef __CUDACC__
// s for a block whose largest magnitude is amax (finite, >= 0).
__device__ __forceinline__ int mx_scale_exp(float amax) {
  const int eb = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
  if (eb == 0) return -127;  // zero or subnormal: floor(log2 amax) - 8 < -127
  const int s = eb - 127 - 8;
  return s < -127 ? -127 : s;  // eb <= 254 for finite amax, so s <= 119
}

// 2^-s as an fp32 (normal for s in [-127, 119]).
__device__ __forceinline__ float mx_inv_scale(int s) { return __uint_as_float((uint32_t)(127 - s) << 23); }
#endif

}  // namespace moe
