// bwd_common.cuh -- pieces shared by the backward kernels of bwd.cu (the deterministic
// dK/dV and dQ kernels) and bwd_fused.cu (the fused dK/dV/dQ kernel): warp roles, tile
// geometry, and the 16-bit row writers of the epilogues.
#pragma once

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace attn {

// Warp roles of the two gradient kernels: warp 0 TMA, warp 1 TMEM owner + MMA issuer,
// warps 2-3 idle, then kEw warpgroups of element-wise work, warpgroup w owning 32
// of the 128 columns of every tile (four warps per scheduler keep the exponentials'
// latency hidden).
constexpr int kEw = 4;
constexpr int kEwCols = 128 / kEw;  // tile columns per element-wise warpgroup
constexpr int kBwdThreads = 128 * (1 + kEw);

// ------------------------------------------------------------------ shared layout pieces

template <int D>
struct BwdTiles {
  static constexpr int KB = D / 64;
  static constexpr int TILE = kTileM * D * 2;
  static constexpr int BLK = kTileM * 128;
};

// 128 x 32 fp32 block of this thread's row (rescaled) -> 16-bit, into a
// 128B-swizzled staging tile (the layout the TMA store map expects).
template <int D, bool BF16>
__device__ __forceinline__ void stage_row_chunk(uint8_t* stage, int row, int cc, const uint32_t (&v)[32],
                                                float mul) {
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    pk[i] = pack2<BF16>(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
  const int kb = (cc * 32) / 64;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int ch = ((cc * 32) % 64) / 8 + q;
    uint4* dst = reinterpret_cast<uint4*>(stage + kb * BwdTiles<D>::BLK + row * 128 + ((ch ^ (row & 7)) << 4));
    *dst = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
  }
}

// Write zero rows k0 .. k0+127 (those below n) of a packed [T][H][D] gradient for head hh.
template <int D>
__device__ __forceinline__ void zero_rows_packed(void* base, int H, int hh, int t0, int k0, int n) {
  for (int r = threadIdx.x; r < kTileN; r += blockDim.x) {
    if (k0 + r >= n) continue;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(base) + ((static_cast<size_t>(t0 + k0 + r) * H + hh) * D) * 2);
    for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
  }
}

// 32 columns (chunk cc) of this thread's row, scaled, to a packed [T][H][D] tensor row.
template <int D, bool BF16>
__device__ __forceinline__ void store_row_chunk_packed(void* base, size_t row_elem, int cc, const uint32_t (&v)[32],
                                                       float mul) {
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    pk[i] = pack2<BF16>(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
  uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(base) + (row_elem + cc * 32) * 2);
#pragma unroll
  for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
}

}  // namespace attn
