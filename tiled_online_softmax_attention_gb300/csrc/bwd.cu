// bwd.cu -- backward attention kernels for sm_103a.
//
// The backward pass recomputes the probabilities tile by tile from the saved
// row logsumexp instead of storing P ("Understanding FlashAttention, Part 2",
// section 2.4, Fig 20; "FlashAttention hardware-aware analysis" (huaweicloud),
// section four, part 1).  With LSE2 = lse * log2(e) and c = scale * log2(e):
//
//   P   = ex2(c S - LSE2)            S = Q K^T, recomputed
//   dV  = P^T dO                     (Part 2, section 2.4, Fig 17)
//   dP  = dO V^T
//   dS  = P * (dP - D),  D_i = rowsum(dO_i * O_i)   (softmax Jacobian, Fig 18)
//   dQ  = scale dS K,    dK = scale dS^T Q          (Fig 19)
//
// Three kernels, all deterministic (no atomics):
//   bwd_pre   D and LSE2 per row into the workspace (rows padded to whole
//             tiles: padding rows get LSE2 = +inf and D = 0, so their P and dS
//             are exactly 0 without any per-element test).
//   bwd_dkdv  one CTA per 128-key tile: K_j, V_j stay in shared memory, Q_i and
//             dO_i stream through a TMA ring; S^T, dP^T, dV and dK live in
//             tensor memory; P^T and dS^T go back to tensor memory in 16 bits
//             and feed the dV and dK products directly.
//   bwd_dq    one CTA per 128-query tile: Q_i, dO_i stay, K_j and V_j stream;
//             S, dP and dQ in tensor memory, dS in 16 bits feeds dQ.
// Recomputing S and dP in both tile orders costs two extra N x N x d products
// (seven instead of five) and buys independence from floating-point atomics.
#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kBwdThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 elementwise + epilogue

// ------------------------------------------------------------------ bwd_pre

template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __grid_constant__ BwdArgs a) {
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(a.BH) * a.Npad;
  if (warp_global >= rows) return;
  const int bh = static_cast<int>(warp_global / a.Npad);
  const int r = static_cast<int>(warp_global % a.Npad);
  float dsum = 0.f;
  float l2 = INFINITY;
  if (r < a.N) {
    const size_t base = (static_cast<size_t>(bh) * a.N + r) * D;
    constexpr int PER = D / 32;  // 16-bit elements per lane (2 or 4)
    const uint16_t* op = reinterpret_cast<const uint16_t*>(a.o) + base + lane * PER;
    const uint16_t* dp = reinterpret_cast<const uint16_t*>(a.dout) + base + lane * PER;
    uint16_t ov[PER], dv[PER];
    if constexpr (PER == 4) {
      *reinterpret_cast<uint2*>(ov) = *reinterpret_cast<const uint2*>(op);
      *reinterpret_cast<uint2*>(dv) = *reinterpret_cast<const uint2*>(dp);
    } else {
      *reinterpret_cast<uint32_t*>(ov) = *reinterpret_cast<const uint32_t*>(op);
      *reinterpret_cast<uint32_t*>(dv) = *reinterpret_cast<const uint32_t*>(dp);
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      float x, y;
      if constexpr (BF16) {
        x = __uint_as_float(static_cast<uint32_t>(ov[i]) << 16);
        y = __uint_as_float(static_cast<uint32_t>(dv[i]) << 16);
      } else {
        x = __half2float(__ushort_as_half(ov[i]));
        y = __half2float(__ushort_as_half(dv[i]));
      }
      dsum = fmaf(x, y, dsum);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
    l2 = a.lse[static_cast<size_t>(bh) * a.N + r] * 1.4426950408889634f;
  }
  if (lane == 0) {
    const size_t w = static_cast<size_t>(bh) * a.Npad + r;
    a.delta[w] = dsum;
    a.lse2[w] = l2;
  }
}

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

// ------------------------------------------------------------------ bwd_dkdv

template <int D>
struct DkdvLayout {
  using T = BwdTiles<D>;
  static constexpr int STAGES = (D == 128) ? 2 : 3;
  static constexpr int STAGE_BYTES = 2 * T::TILE + 2 * 512;  // Q_i, dO_i, LSE2_i, D_i
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = T::TILE;
  static constexpr int OFF_ST = 2 * T::TILE;
  static constexpr int OFF_BAR = OFF_ST + STAGES * STAGE_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  // per-stage offsets
  static constexpr int S_Q = 0, S_DO = T::TILE, S_L = 2 * T::TILE, S_D = 2 * T::TILE + 512;
  // tensor memory columns
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 256 + D, TM_COLS = 512;
};

enum : int {
  K_KVFULL = 0,
  K_STFULL = 1,
  K_PFULL = 2,
  K_MM2 = 3,
  K_DRAIN = 4,
  K_QFULL = 5,   // + stage
  K_EMPTY = 9,   // + stage
  K_COUNT = 13
};

template <int D, bool BF16>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_dkdv_kernel(const __grid_constant__ BwdArgs a) {
  using L = DkdvLayout<D>;
  using T = BwdTiles<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bars = sb + L::OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 8 * K_COUNT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_BAR + 8 * K_COUNT + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_t = (a.N + kTileN - 1) / kTileN;
  const int kt = static_cast<int>(blockIdx.x) / a.BH;  // low key tiles see the most queries
  const int bh = static_cast<int>(blockIdx.x) % a.BH;
  const int k0 = kt * kTileN;
  const int i_begin = a.causal ? kt : 0;               // query tiles before the key tile are masked out
  const int n_iter = n_t - i_begin;

  if (threadIdx.x == 0) {
    mbar_init(bar(K_KVFULL), 1);
    mbar_init(bar(K_STFULL), 1);
    mbar_init(bar(K_PFULL), 128);
    mbar_init(bar(K_MM2), 1);
    mbar_init(bar(K_DRAIN), 1);
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(bar(K_QFULL + s), 1);
      mbar_init(bar(K_EMPTY + s), 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), L::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, a.dev_status, a.wait_limit_ns};
  auto stage_base = [&](int s) -> uint32_t { return sb + L::OFF_ST + s * L::STAGE_BYTES; };

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
      prefetch_tmap(&a.tm_do);
      mbar_arrive_expect_tx(bar(K_KVFULL), 2 * T::TILE);
      for (int kb = 0; kb < T::KB; ++kb) {
        tma_load_3d(sb + L::OFF_K + kb * T::BLK, &a.tm_k, bar(K_KVFULL), kb * 64, k0, bh);
        tma_load_3d(sb + L::OFF_V + kb * T::BLK, &a.tm_v, bar(K_KVFULL), kb * 64, k0, bh);
      }
      int issued = 0;
      for (int t = 0; t < n_iter; ++t) {
        const int s = t % L::STAGES;
        const int q0 = (i_begin + t) * kTileM;
        if (t >= L::STAGES && !mbar_wait(bar(K_EMPTY + s), ((t / L::STAGES) - 1) & 1, wc)) break;
        const uint32_t st = stage_base(s);
        mbar_arrive_expect_tx(bar(K_QFULL + s), 2 * T::TILE + 1024);
        for (int kb = 0; kb < T::KB; ++kb) {
          tma_load_3d(st + L::S_Q + kb * T::BLK, &a.tm_q, bar(K_QFULL + s), kb * 64, q0, bh);
          tma_load_3d(st + L::S_DO + kb * T::BLK, &a.tm_do, bar(K_QFULL + s), kb * 64, q0, bh);
        }
        const size_t w = static_cast<size_t>(bh) * a.Npad + q0;
        bulk_load(st + L::S_L, a.lse2 + w, 512, bar(K_QFULL + s));
        bulk_load(st + L::S_D, a.delta + w, 512, bar(K_QFULL + s));
        issued = t + 1;
      }
      mbar_wait(bar(K_KVFULL), 0, wc);
      for (int t = (issued > L::STAGES ? issued - L::STAGES : 0); t < issued; ++t)
        mbar_wait(bar(K_QFULL + t % L::STAGES), (t / L::STAGES) & 1, wc);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16(kTileM, kTileN, BF16, false, false);  // K-major x K-major
      constexpr uint32_t idesc_g = idesc_f16(kTileM, D, BF16, false, true);        // TMEM x MN-major
      bool ok = mbar_wait(bar(K_KVFULL), 0, wc);
      for (int t = 0; ok && t < n_iter; ++t) {
        const int s = t % L::STAGES;
        if (!mbar_wait(bar(K_QFULL + s), (t / L::STAGES) & 1, wc)) { ok = false; break; }
        // S^T, dP^T overwrite the columns that held P^T, dS^T of the previous tile.
        if (t > 0 && !mbar_wait(bar(K_MM2), (t - 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t st = stage_base(s);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * T::BLK + (k & 3) * 32;
          mma_ss(tmem + L::TM_S, sdesc_sw128(sb + L::OFF_K + off, 16, 1024),
                 sdesc_sw128(st + L::S_Q + off, 16, 1024), idesc_s, k > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * T::BLK + (k & 3) * 32;
          mma_ss(tmem + L::TM_DP, sdesc_sw128(sb + L::OFF_V + off, 16, 1024),
                 sdesc_sw128(st + L::S_DO + off, 16, 1024), idesc_s, k > 0 ? 1u : 0u);
        }
        tc_commit(bar(K_STFULL));
        if (!mbar_wait(bar(K_PFULL), t & 1, wc)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kTileM / 16; ++k) {
          const uint32_t acc = (t > 0 || k > 0) ? 1u : 0u;
          mma_ts(tmem + L::TM_DV, tmem + L::TM_S + k * 8, sdesc_sw128(st + L::S_DO + k * 2048, T::BLK, 1024),
                 idesc_g, acc);
          mma_ts(tmem + L::TM_DK, tmem + L::TM_DP + k * 8, sdesc_sw128(st + L::S_Q + k * 2048, T::BLK, 1024),
                 idesc_g, acc);
        }
        tc_commit(bar(K_MM2));
        tc_commit(bar(K_EMPTY + s));
      }
      tc_commit(bar(K_DRAIN));
      mbar_wait(bar(K_DRAIN), 0, wc);
    }
  } else {
    const int wq = warp & 3;
    const int row = wq * 32 + lane;    // key row within the tile == TMEM lane
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float sl2 = a.scale_log2;
    bool ok = n_iter > 0;
    for (int t = 0; t < n_iter; ++t) {
      const int s = t % L::STAGES;
      const int qt = i_begin + t;
      if (!mbar_wait_warp(bar(K_QFULL + s), (t / L::STAGES) & 1, wc)) { ok = false; break; }
      if (!mbar_wait_warp(bar(K_STFULL), t & 1, wc)) { ok = false; break; }
      tc_fence_after();
      const float* lse2 = reinterpret_cast<const float*>(smem + L::OFF_ST + s * L::STAGE_BYTES + L::S_L);
      const float* dlt = reinterpret_cast<const float*>(smem + L::OFF_ST + s * L::STAGE_BYTES + L::S_D);
      // causal diagonal tile: query c sees key `row` only if c >= row
      const int first_visible = (a.causal && qt == kt) ? row : 0;
#pragma unroll
      for (int ch = 0; ch < kTileM / 32; ++ch) {
        uint32_t sv[32], dpv[32];
        tmem_ld_x32(t_lane + L::TM_S + ch * 32, sv);
        tmem_ld_x32(t_lane + L::TM_DP + ch * 32, dpv);
        uint32_t ppk[16], dpk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int c = ch * 32 + i;
          float p0 = ex2(fmaf(__uint_as_float(sv[i]), sl2, -lse2[c]));
          float p1 = ex2(fmaf(__uint_as_float(sv[i + 1]), sl2, -lse2[c + 1]));
          if (c < first_visible) p0 = 0.f;
          if (c + 1 < first_visible) p1 = 0.f;
          const float d0 = p0 * (__uint_as_float(dpv[i]) - dlt[c]);
          const float d1 = p1 * (__uint_as_float(dpv[i + 1]) - dlt[c + 1]);
          ppk[i / 2] = pack2<BF16>(p0, p1);
          dpk[i / 2] = pack2<BF16>(d0, d1);
        }
        // 16-bit P^T / dS^T overwrite columns of S^T / dP^T this thread has already read.
        tmem_st_x16(t_lane + L::TM_S + ch * 16, ppk);
        tmem_st_x16(t_lane + L::TM_DP + ch * 16, dpk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(K_PFULL));
    }
    if (ok) ok = mbar_wait_warp(bar(K_MM2), (n_iter - 1) & 1, wc);
    if (ok) {
      tc_fence_after();
      // All products are done: the stage-0 Q and dO buffers become staging tiles.
      uint8_t* st_dk = smem + L::OFF_ST + L::S_Q;
      uint8_t* st_dv = smem + L::OFF_ST + L::S_DO;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t v[32];
        tmem_ld_x32(t_lane + L::TM_DV + cc * 32, v);
        stage_row_chunk<D, BF16>(st_dv, row, cc, v, 1.f);
        tmem_ld_x32(t_lane + L::TM_DK + cc * 32, v);
        stage_row_chunk<D, BF16>(st_dk, row, cc, v, a.scale);
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128);
    if (warp == 2 && lane == 0 && !*abort_flag) {
      for (int kb = 0; kb < T::KB; ++kb) {
        tma_store_3d(&a.tm_dk, sb + L::OFF_ST + L::S_Q + kb * T::BLK, kb * 64, k0, bh);
        tma_store_3d(&a.tm_dv, sb + L::OFF_ST + L::S_DO + kb * T::BLK, kb * 64, k0, bh);
      }
      bulk_commit();
      bulk_wait_read_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TM_COLS);
  }
}

// ------------------------------------------------------------------ bwd_dq

template <int D>
struct DqLayout {
  using T = BwdTiles<D>;
  static constexpr int STAGES = (D == 128) ? 2 : 4;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = T::TILE;
  static constexpr int OFF_K = 2 * T::TILE;
  static constexpr int OFF_V = OFF_K + STAGES * T::TILE;
  static constexpr int OFF_BAR = OFF_V + STAGES * T::TILE;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DQ = 256, TM_DS = 384, TM_COLS = 512;
};

enum : int {
  Q_QFULL = 0,
  Q_SFULL = 1,
  Q_SFREE = 2,
  Q_DSFULL = 3,
  Q_DQDONE = 4,
  Q_DRAIN = 5,
  Q_KVFULL = 6,  // + stage
  Q_EMPTY = 10,  // + stage
  Q_COUNT = 14
};

template <int D, bool BF16>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdArgs a) {
  using L = DqLayout<D>;
  using T = BwdTiles<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bars = sb + L::OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 8 * Q_COUNT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_BAR + 8 * Q_COUNT + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_t = (a.N + kTileM - 1) / kTileM;
  const int qt = n_t - 1 - static_cast<int>(blockIdx.x) / a.BH;  // longest causal tiles first
  const int bh = static_cast<int>(blockIdx.x) % a.BH;
  const int q0 = qt * kTileM;
  const int n_kv = a.causal ? qt + 1 : n_t;

  if (threadIdx.x == 0) {
    mbar_init(bar(Q_QFULL), 1);
    mbar_init(bar(Q_SFULL), 1);
    mbar_init(bar(Q_SFREE), 128);
    mbar_init(bar(Q_DSFULL), 128);
    mbar_init(bar(Q_DQDONE), 1);
    mbar_init(bar(Q_DRAIN), 1);
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(bar(Q_KVFULL + s), 1);
      mbar_init(bar(Q_EMPTY + s), 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), L::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, a.dev_status, a.wait_limit_ns};

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
      prefetch_tmap(&a.tm_do);
      mbar_arrive_expect_tx(bar(Q_QFULL), 2 * T::TILE);
      for (int kb = 0; kb < T::KB; ++kb) {
        tma_load_3d(sb + L::OFF_Q + kb * T::BLK, &a.tm_q, bar(Q_QFULL), kb * 64, q0, bh);
        tma_load_3d(sb + L::OFF_DO + kb * T::BLK, &a.tm_do, bar(Q_QFULL), kb * 64, q0, bh);
      }
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % L::STAGES;
        if (j >= L::STAGES && !mbar_wait(bar(Q_EMPTY + s), ((j / L::STAGES) - 1) & 1, wc)) break;
        mbar_arrive_expect_tx(bar(Q_KVFULL + s), 2 * T::TILE);
        for (int kb = 0; kb < T::KB; ++kb) {
          tma_load_3d(sb + L::OFF_K + s * T::TILE + kb * T::BLK, &a.tm_k, bar(Q_KVFULL + s), kb * 64, j * kTileN, bh);
          tma_load_3d(sb + L::OFF_V + s * T::TILE + kb * T::BLK, &a.tm_v, bar(Q_KVFULL + s), kb * 64, j * kTileN, bh);
        }
        issued = j + 1;
      }
      mbar_wait(bar(Q_QFULL), 0, wc);
      for (int j = (issued > L::STAGES ? issued - L::STAGES : 0); j < issued; ++j)
        mbar_wait(bar(Q_KVFULL + j % L::STAGES), (j / L::STAGES) & 1, wc);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16(kTileM, kTileN, BF16, false, false);
      constexpr uint32_t idesc_g = idesc_f16(kTileM, D, BF16, false, true);
      bool ok = mbar_wait(bar(Q_QFULL), 0, wc);
      auto issue_dq = [&](int t) -> bool {
        const int s = t % L::STAGES;
        if (!mbar_wait(bar(Q_DSFULL), t & 1, wc)) return false;
        tc_fence_after();
        const uint32_t kbase = sb + L::OFF_K + s * T::TILE;
#pragma unroll
        for (int k = 0; k < kTileN / 16; ++k)
          mma_ts(tmem + L::TM_DQ, tmem + L::TM_DS + k * 8, sdesc_sw128(kbase + k * 2048, T::BLK, 1024), idesc_g,
                 (t > 0 || k > 0) ? 1u : 0u);
        tc_commit(bar(Q_DQDONE));
        tc_commit(bar(Q_EMPTY + s));
        return true;
      };
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j % L::STAGES;
        if (!mbar_wait(bar(Q_KVFULL + s), (j / L::STAGES) & 1, wc)) { ok = false; break; }
        if (j > 0 && !mbar_wait(bar(Q_SFREE), (j - 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t kbase = sb + L::OFF_K + s * T::TILE;
        const uint32_t vbase = sb + L::OFF_V + s * T::TILE;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * T::BLK + (k & 3) * 32;
          mma_ss(tmem + L::TM_S, sdesc_sw128(sb + L::OFF_Q + off, 16, 1024), sdesc_sw128(kbase + off, 16, 1024),
                 idesc_s, k > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * T::BLK + (k & 3) * 32;
          mma_ss(tmem + L::TM_DP, sdesc_sw128(sb + L::OFF_DO + off, 16, 1024), sdesc_sw128(vbase + off, 16, 1024),
                 idesc_s, k > 0 ? 1u : 0u);
        }
        tc_commit(bar(Q_SFULL));
        if (j > 0 && !issue_dq(j - 1)) { ok = false; break; }
      }
      if (ok) issue_dq(n_kv - 1);
      tc_commit(bar(Q_DRAIN));
      mbar_wait(bar(Q_DRAIN), 0, wc);
    }
  } else {
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const int grow = q0 + row;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float sl2 = a.scale_log2;
    const size_t w = static_cast<size_t>(bh) * a.Npad + grow;   // grow < Npad always
    const float lse2 = a.lse2[w];
    const float dlt = a.delta[w];
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!mbar_wait_warp(bar(Q_SFULL), j & 1, wc)) { ok = false; break; }
      tc_fence_after();
      const int kbeg = j * kTileN;
      int lim = a.N - kbeg;                               // keys past the end
      if (a.causal) lim = min(lim, grow - kbeg + 1);      // keys after this query
      uint32_t dsp[64];
#pragma unroll
      for (int ch = 0; ch < kTileN / 32; ++ch) {
        uint32_t sv[32], dpv[32];
        tmem_ld_x32(t_lane + L::TM_S + ch * 32, sv);
        tmem_ld_x32(t_lane + L::TM_DP + ch * 32, dpv);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int c = ch * 32 + i;
          float p0 = ex2(fmaf(__uint_as_float(sv[i]), sl2, -lse2));
          float p1 = ex2(fmaf(__uint_as_float(sv[i + 1]), sl2, -lse2));
          if (c >= lim) p0 = 0.f;
          if (c + 1 >= lim) p1 = 0.f;
          dsp[c / 2] = pack2<BF16>(p0 * (__uint_as_float(dpv[i]) - dlt), p1 * (__uint_as_float(dpv[i + 1]) - dlt));
        }
      }
      tc_fence_before();
      mbar_arrive(bar(Q_SFREE));
      if (j > 0) {
        if (!mbar_wait_warp(bar(Q_DQDONE), (j - 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
      }
      tmem_st_x64(t_lane + L::TM_DS, dsp);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(Q_DSFULL));
    }
    if (ok) ok = mbar_wait_warp(bar(Q_DQDONE), (n_kv - 1) & 1, wc);
    if (ok) {
      tc_fence_after();
      uint8_t* stage = smem + L::OFF_Q;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t v[32];
        tmem_ld_x32(t_lane + L::TM_DQ + cc * 32, v);
        stage_row_chunk<D, BF16>(stage, row, cc, v, a.scale);
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128);
    if (warp == 2 && lane == 0 && !*abort_flag) {
      for (int kb = 0; kb < T::KB; ++kb) tma_store_3d(&a.tm_dq, sb + L::OFF_Q + kb * T::BLK, kb * 64, q0, bh);
      bulk_commit();
      bulk_wait_read_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TM_COLS);
  }
}

template <int D, bool BF16>
cudaError_t launch_pre_t(const BwdArgs& a, cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(a.BH) * a.Npad;
  const int64_t blocks = (rows * 32 + 255) / 256;
  bwd_pre_kernel<D, BF16><<<static_cast<unsigned>(blocks), 256, 0, st>>>(a);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_dkdv_t(const BwdArgs& a, cudaStream_t st) {
  auto k = bwd_dkdv_kernel<D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, DkdvLayout<D>::SMEM);
  if (e != cudaSuccess) return e;
  const int n_t = (a.N + kTileN - 1) / kTileN;
  k<<<n_t * a.BH, kBwdThreads, DkdvLayout<D>::SMEM, st>>>(a);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_dq_t(const BwdArgs& a, cudaStream_t st) {
  auto k = bwd_dq_kernel<D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, DqLayout<D>::SMEM);
  if (e != cudaSuccess) return e;
  const int n_t = (a.N + kTileM - 1) / kTileM;
  k<<<n_t * a.BH, kBwdThreads, DqLayout<D>::SMEM, st>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ bounded-wait self-test

__global__ void wait_selftest_kernel(int* dev_status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t b;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&b), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const WaitCtl wc{&abort_flag, dev_status, limit_ns};
  // Nothing ever arrives on this barrier: the wait must give up and report.
  if (threadIdx.x == 0) (void)mbar_wait(smem_u32(&b), 0, wc);
  __syncthreads();
}

}  // namespace

#define ATTN_DISPATCH(fn)                                                   \
  if (d == 128) return bf16 ? fn<128, true>(a, s) : fn<128, false>(a, s); \
  return bf16 ? fn<64, true>(a, s) : fn<64, false>(a, s);

cudaError_t launch_bwd_pre(const BwdArgs& a, int d, bool bf16, cudaStream_t s) { ATTN_DISPATCH(launch_pre_t) }
cudaError_t launch_bwd_dkdv(const BwdArgs& a, int d, bool bf16, cudaStream_t s) { ATTN_DISPATCH(launch_dkdv_t) }
cudaError_t launch_bwd_dq(const BwdArgs& a, int d, bool bf16, cudaStream_t s) { ATTN_DISPATCH(launch_dq_t) }
#undef ATTN_DISPATCH

cudaError_t launch_wait_selftest(int* dev_status, uint64_t limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(dev_status, limit_ns);
  return cudaGetLastError();
}

}  // namespace attn
