// bwd256.cu -- backward attention kernels for head dimension 256 (sm_103a).
//
// The same gradients as bwd.cu ("Understanding FlashAttention, Part 2", section 2.4,
// Figs 16-20: P recomputed from the saved logsumexp, dV = P^T dO, dP = dO V^T,
// dS = P (dP - D), dQ = scale dS K, dK = scale dS^T Q), for the head dimension 256 the
// huaweicloud page's section five, part 1 lists.
//
// At d = 256 one 128-row tile of Q, K, V or dO takes 64 KB of shared memory and one
// gradient accumulator 256 tensor-memory columns, so bwd.cu's fused dK/dV kernel
// (K, V, Q, dO tiles and four accumulators at once) does not fit.  Three kernels:
//   dV   one CTA per 128-key tile: K stays; per query tile S^T = K Q^T, P^T, and
//        dV += P^T dO (two 128-column halves)
//   dK   one CTA per 128-key tile: K and V stay; S^T, dP^T = V dO^T, dS^T, and
//        dK += dS^T Q
//   dQ   one CTA per 128-query tile: Q and dO stay; per key tile S, dP, dS and
//        dQ += dS K
// Everything that streams does so in 32 KB column halves (128 rows x 128 columns)
// through a ring of slots, in exactly the order the MMA warp consumes them; a tensor
// needed twice in one step (Q in dK, K in dQ) is fetched twice.  This costs products
// (16 half-tile units per step against 10 algorithmic) and load traffic, and buys a fit.
//
// Warp roles as in bwd.cu: warp 0 TMA, warp 1 TMEM owner + MMA issuer, warps 2-3 idle,
// four element-wise warpgroups of 32 columns each.  Every wait is bounded.
#include "common.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int D2 = 256;
constexpr int kEw2 = 4;
constexpr int kEwCols2 = 128 / kEw2;
constexpr int kThreads2 = 128 * (1 + kEw2);
constexpr int kBlk = kTileM * 128;        // one 128-row x 64-column block (16 KB)
constexpr int kTile = kTileM * D2 * 2;    // one 128-row x 256-column tile (64 KB)
constexpr int kHalf = kTileM * 128 * 2;   // one 128-row x 128-column half (32 KB)

// Barriers (shared by the three kernels; unused ones are simply never waited on).
enum : int {
  R_STAT = 0,     // stationary tiles loaded
  R_SFULL = 1,    // S / S^T computed
  R_DPFULL = 2,   // dP / dP^T computed
  R_PREADY = 3,   // P^T written (element-wise threads)
  R_DSREADY = 4,  // dS / dS^T written (element-wise threads)
  R_DONE = 5,
  R_DRAIN = 6,
  R_FULL = 7,     // + ring slot
  R_EMPTY = 11,   // + ring slot
  R_COUNT = 15
};

template <int NSLOT, int STATIONARY>
struct Layout256 {
  static constexpr int OFF_ST = 0;                              // STATIONARY 64 KB tiles
  static constexpr int OFF_RING = STATIONARY * kTile;           // NSLOT halves
  static constexpr int OFF_L = OFF_RING + NSLOT * kHalf;        // 16 warps x (LSE2[32], D[32])
  static constexpr int OFF_BAR = OFF_L + 4096;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  static_assert(NSLOT * kHalf >= kTile, "the epilogue stages a 256-column tile over the ring");
};

// Common prologue: barriers, TMEM allocation.  Returns the TMEM base address.
__device__ __forceinline__ uint32_t prologue256(uint32_t bars, int nslot, volatile int* abort_flag,
                                                uint32_t* tmem_slot, int ew_count) {
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(bars + 8 * R_STAT, 1);
    mbar_init(bars + 8 * R_SFULL, 1);
    mbar_init(bars + 8 * R_DPFULL, 1);
    mbar_init(bars + 8 * R_PREADY, ew_count);
    mbar_init(bars + 8 * R_DSREADY, ew_count);
    mbar_init(bars + 8 * R_DONE, 1);
    mbar_init(bars + 8 * R_DRAIN, 1);
    for (int s = 0; s < nslot; ++s) {
      mbar_init(bars + 8 * (R_FULL + s), 1);
      mbar_init(bars + 8 * (R_EMPTY + s), 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return *tmem_slot;
}

// Ring of 32 KB half tiles.  Item c sits in slot c % NSLOT; the producer and the MMA
// warp walk the same item sequence.
template <int NSLOT>
struct Ring {
  uint32_t sb, bars;
  int c = 0;
  __device__ uint32_t slot_addr(int item) const { return sb + (item % NSLOT) * kHalf; }
  __device__ uint32_t full(int item) const { return bars + 8 * (R_FULL + item % NSLOT); }
  __device__ uint32_t empty(int item) const { return bars + 8 * (R_EMPTY + item % NSLOT); }
};

// Producer: load column half `half` (columns 128 half .. +127) of the 128-row tile at
// `row` of head `bh` as the ring's next item, once the item NSLOT earlier has been
// released.
template <int NSLOT>
__device__ __forceinline__ bool load_half(Ring<NSLOT>& r, const CUtensorMap* m, int half, int row, int bh,
                                          const WaitCtl& wc) {
  const int c = r.c;
  if (c >= NSLOT && !mbar_wait(r.empty(c), ((c / NSLOT) - 1) & 1, wc)) return false;
  mbar_arrive_expect_tx(r.full(c), kHalf);
  for (int b = 0; b < 2; ++b) tma_load_3d(r.slot_addr(c) + b * kBlk, m, r.full(c), 128 * half + 64 * b, row, bh);
  ++r.c;
  return true;
}

// Element-wise warps of the key-tile kernels: each stages the 32 per-query values its
// warpgroup needs (LSE2, and D when `dl` is given) in its own 256-byte slice of shared
// memory, read back as broadcast float4s.  The lane's own values are fetched before the
// wait for S^T, so the global load overlaps it.
struct RowStage {
  float* w;  // this warp's slice: [0, 32) LSE2, [32, 64) D
  __device__ void put(float l, float d) {
    __syncwarp();
    w[threadIdx.x & 31] = l;
    w[32 + (threadIdx.x & 31)] = d;
    __syncwarp();
  }
  __device__ const float4* lse4() const { return reinterpret_cast<const float4*>(w); }
  __device__ const float4* d4() const { return reinterpret_cast<const float4*>(w + 32); }
};

// S^T-style product over d = 256 as two halves: D (+)= A_stat[:, half] B_half^T, both
// K-major; A is a stationary 4-block tile, B the ring item.
__device__ __forceinline__ void mma_half_kk(uint32_t d_tmem, uint32_t a_stat, uint32_t b_item, int half,
                                            uint32_t idesc, bool first) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const int k = 8 * half + kk;
    const uint32_t aoff = (k >> 2) * kBlk + (k & 3) * 32;
    const uint32_t boff = (kk >> 2) * kBlk + (kk & 3) * 32;
    mma_ss(d_tmem, sdesc_sw128(a_stat + aoff, 16, 1024), sdesc_sw128(b_item + boff, 16, 1024), idesc,
           (first && kk == 0) ? 0u : 1u);
  }
}

// Gradient product into one 128-column half: D (+)= A_tmem B_half, A the 16-bit P^T /
// dS^T / dS written by warpgroup w at a_tmem + 32w (16 columns), B MN-major.
__device__ __forceinline__ void mma_half_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_item, uint32_t idesc,
                                            bool first) {
#pragma unroll
  for (int k = 0; k < kTileM / 16; ++k)
    mma_ts(d_tmem, a_tmem + kEwCols2 * (k >> 1) + 8 * (k & 1), sdesc_sw128(b_item + k * 2048, kBlk, 1024), idesc,
           (first && k == 0) ? 0u : 1u);
}

// Epilogue: this thread's row of a 256-column fp32 accumulator (its warpgroup's 64
// columns), scaled, as 16-bit into a 128B-swizzled staging tile; then one thread
// stores the tile with TMA.
template <bool BF16>
__device__ __forceinline__ void stage_acc256(uint8_t* stage, uint32_t t_acc, int row, int h, float mul) {
#pragma unroll 1
  for (int cc = 2 * h; cc < 2 * h + 2; ++cc) {
    uint32_t v[32];
    tmem_ld_x32(t_acc + cc * 32, v);
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      pk[i] = pack2<BF16>(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
    const int kb = (cc * 32) / 64;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int ch = ((cc * 32) % 64) / 8 + q;
      uint4* dst = reinterpret_cast<uint4*>(stage + kb * kBlk + row * 128 + ((ch ^ (row & 7)) << 4));
      *dst = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
  }
}

// ------------------------------------------------------------------ dV
// TMEM: S^T at 0 (P^T over its first columns), dV at 256..511 (halves at 256, 384).
template <bool BF16>
__global__ void __launch_bounds__(kThreads2, 1) bwd256_dv_kernel(const __grid_constant__ BwdArgs a) {
  constexpr int NSLOT = 4;
  using L = Layout256<NSLOT, 1>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bars = sb + L::OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 8 * R_COUNT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_BAR + 8 * R_COUNT + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_t = (a.N + kTileM - 1) / kTileM, n_tk = (a.Nk + kTileN - 1) / kTileN;
  const WorkItem wi = work_item<2>(static_cast<int>(blockIdx.x), a.BH, n_tk);
  const int bh = wi.bh, k0 = wi.rank * kTileN;
  const int i_begin = a.causal ? max(0, k0 - a.cofs) / kTileM : 0;
  const int n_iter = n_t - i_begin;
  const uint32_t tmem = prologue256(bars, NSLOT, abort_flag, tmem_slot, 128 * kEw2);
  const WaitCtl wc{abort_flag, a.dev_status, a.wait_limit_ns};
  constexpr uint32_t TM_S = 0, TM_DV = 256;

  if (warp == 0 && lane == 0) {
    mbar_arrive_expect_tx(bar(R_STAT), kTile);
    for (int b = 0; b < 4; ++b) tma_load_3d(sb + L::OFF_ST + b * kBlk, &a.tm_k, bar(R_STAT), 64 * b, k0, bh);
    Ring<NSLOT> r{sb + L::OFF_RING, bars};
    bool ok = true;
    for (int t = 0; ok && t < n_iter; ++t) {  // per query tile: Q halves, then dO halves
      const int q0 = (i_begin + t) * kTileM;
      ok = load_half(r, &a.tm_q, 0, q0, bh, wc) && load_half(r, &a.tm_q, 1, q0, bh, wc) &&
           load_half(r, &a.tm_do, 0, q0, bh, wc) && load_half(r, &a.tm_do, 1, q0, bh, wc);
    }
    mbar_wait(bar(R_STAT), 0, wc);
    for (int c = (r.c > NSLOT ? r.c - NSLOT : 0); c < r.c; ++c) mbar_wait(r.full(c), (c / NSLOT) & 1, wc);
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc_s = idesc_f16(kTileM, kTileM, BF16, false, false);
    constexpr uint32_t idesc_g = idesc_f16(kTileM, 128, BF16, false, true);
    Ring<NSLOT> r{sb + L::OFF_RING, bars};
    auto next = [&]() -> bool { return mbar_wait(r.full(r.c), (r.c / NSLOT) & 1, wc); };
    auto release = [&]() { tc_commit(r.empty(r.c)); ++r.c; };
    bool ok = mbar_wait(bar(R_STAT), 0, wc);
    auto issue_st = [&]() -> bool {  // S^T = K Q^T over both column halves
      for (int h = 0; h < 2; ++h) {
        if (!next()) return false;
        tc_fence_after();
        mma_half_kk(tmem + TM_S, sb + L::OFF_ST, r.slot_addr(r.c), h, idesc_s, h == 0);
        release();
      }
      tc_commit(bar(R_SFULL));
      return true;
    };
    if (ok && n_iter > 0) ok = issue_st();
    for (int t = 0; ok && t < n_iter; ++t) {
      if (!(ok = mbar_wait(bar(R_PREADY), t & 1, wc))) break;
      for (int h = 0; ok && h < 2; ++h) {  // dV[:, half] += P^T dO[:, half]
        if (!(ok = next())) break;
        tc_fence_after();
        mma_half_ts(tmem + TM_DV + 128 * h, tmem + TM_S, r.slot_addr(r.c), idesc_g, t == 0);
        release();
      }
      if (ok && t + 1 < n_iter) ok = issue_st();  // overwrites P^T(t) after dV(t) read it
    }
    if (ok) tc_commit(bar(R_DONE));
    tc_commit(bar(R_DRAIN));
    mbar_wait(bar(R_DRAIN), 0, wc);
  } else if (warp >= 4) {
    const int h = (warp >> 2) - 1, wq = warp & 3, row = wq * 32 + lane;  // row: key within the tile
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float sl2 = a.scale_log2;
    RowStage rs{reinterpret_cast<float*>(smem + L::OFF_L) + (warp - 4) * 64};
    bool ok = true;
    for (int t = 0; t < n_iter; ++t) {
      const int qt = i_begin + t;
      const float my_l = a.lse2[static_cast<size_t>(bh) * a.Npad + qt * kTileM + kEwCols2 * h + lane];
      if (!(ok = mbar_wait_warp(bar(R_SFULL), t & 1, wc))) break;
      tc_fence_after();
      rs.put(my_l, 0.f);
      const float4* l4 = rs.lse4();
      const int first_visible = a.causal ? k0 + row - a.cofs - qt * kTileM - kEwCols2 * h : 0;
      uint32_t sv[kEwCols2];
      tmem_ld_x32(t_lane + TM_S + kEwCols2 * h, sv);
      float p[kEwCols2];
#pragma unroll
      for (int v = 0; v < kEwCols2 / 4; ++v) {
        const float4 lv = l4[v];
        p[4 * v + 0] = ex2(fmaf(__uint_as_float(sv[4 * v + 0]), sl2, -lv.x));
        p[4 * v + 1] = ex2(fmaf(__uint_as_float(sv[4 * v + 1]), sl2, -lv.y));
        p[4 * v + 2] = ex2(fmaf(__uint_as_float(sv[4 * v + 2]), sl2, -lv.z));
        p[4 * v + 3] = ex2(fmaf(__uint_as_float(sv[4 * v + 3]), sl2, -lv.w));
      }
      if (first_visible > 0) {
#pragma unroll
        for (int c = 0; c < kEwCols2; ++c)
          if (c < first_visible) p[c] = 0.f;
      }
      uint32_t pk[kEwCols2 / 2];
#pragma unroll
      for (int c = 0; c < kEwCols2; c += 2) pk[c / 2] = pack2<BF16>(p[c], p[c + 1]);
      tmem_st_x16(t_lane + TM_S + kEwCols2 * h, pk);  // over columns this thread has read
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(R_PREADY));
    }
    if (ok) ok = mbar_wait_warp(bar(R_DONE), 0, wc);
    if (ok) {
      tc_fence_after();
      stage_acc256<BF16>(smem + L::OFF_RING, t_lane + TM_DV, row, h, 1.f);
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128 * kEw2);
    if (warp == 4 && lane == 0 && ok && !*abort_flag) {
      for (int b = 0; b < 4; ++b) tma_store_3d(&a.tm_dv, sb + L::OFF_RING + b * kBlk, 64 * b, k0, bh);
      bulk_commit();
      bulk_wait_read_all();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ dK
// TMEM: S^T at 0, dP^T at 128 (dS^T over its first columns), dK at 256..511.
template <bool BF16>
__global__ void __launch_bounds__(kThreads2, 1) bwd256_dk_kernel(const __grid_constant__ BwdArgs a) {
  constexpr int NSLOT = 2;
  using L = Layout256<NSLOT, 2>;  // K, V stationary
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bars = sb + L::OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 8 * R_COUNT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_BAR + 8 * R_COUNT + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_t = (a.N + kTileM - 1) / kTileM, n_tk = (a.Nk + kTileN - 1) / kTileN;
  const WorkItem wi = work_item<2>(static_cast<int>(blockIdx.x), a.BH, n_tk);
  const int bh = wi.bh, k0 = wi.rank * kTileN;
  const int i_begin = a.causal ? max(0, k0 - a.cofs) / kTileM : 0;
  const int n_iter = n_t - i_begin;
  const uint32_t tmem = prologue256(bars, NSLOT, abort_flag, tmem_slot, 128 * kEw2);
  const WaitCtl wc{abort_flag, a.dev_status, a.wait_limit_ns};
  constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DK = 256;
  const uint32_t st_k = sb + L::OFF_ST, st_v = sb + L::OFF_ST + kTile;

  if (warp == 0 && lane == 0) {
    mbar_arrive_expect_tx(bar(R_STAT), 2 * kTile);
    for (int b = 0; b < 4; ++b) {
      tma_load_3d(st_k + b * kBlk, &a.tm_k, bar(R_STAT), 64 * b, k0, bh);
      tma_load_3d(st_v + b * kBlk, &a.tm_v, bar(R_STAT), 64 * b, k0, bh);
    }
    Ring<NSLOT> r{sb + L::OFF_RING, bars};
    bool ok = true;
    for (int t = 0; ok && t < n_iter; ++t) {  // Q halves, dO halves, Q halves again
      const int q0 = (i_begin + t) * kTileM;
      ok = load_half(r, &a.tm_q, 0, q0, bh, wc) && load_half(r, &a.tm_q, 1, q0, bh, wc) && load_half(r, &a.tm_do, 0, q0, bh, wc) &&
           load_half(r, &a.tm_do, 1, q0, bh, wc) && load_half(r, &a.tm_q, 0, q0, bh, wc) &&
           load_half(r, &a.tm_q, 1, q0, bh, wc);
    }
    mbar_wait(bar(R_STAT), 0, wc);
    for (int c = (r.c > NSLOT ? r.c - NSLOT : 0); c < r.c; ++c) mbar_wait(r.full(c), (c / NSLOT) & 1, wc);
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc_s = idesc_f16(kTileM, kTileM, BF16, false, false);
    constexpr uint32_t idesc_g = idesc_f16(kTileM, 128, BF16, false, true);
    Ring<NSLOT> r{sb + L::OFF_RING, bars};
    auto next = [&]() -> bool { return mbar_wait(r.full(r.c), (r.c / NSLOT) & 1, wc); };
    auto release = [&]() { tc_commit(r.empty(r.c)); ++r.c; };
    bool ok = mbar_wait(bar(R_STAT), 0, wc);
    for (int t = 0; ok && t < n_iter; ++t) {
      for (int h = 0; ok && h < 2; ++h) {  // S^T = K Q^T (overwrites S^T(t-1), read before dS^T(t-1))
        if (!(ok = next())) break;
        tc_fence_after();
        mma_half_kk(tmem + TM_S, st_k, r.slot_addr(r.c), h, idesc_s, h == 0);
        release();
      }
      if (!ok) break;
      tc_commit(bar(R_SFULL));
      for (int h = 0; ok && h < 2; ++h) {  // dP^T = V dO^T (overwrites dS^T(t-1), read by dK(t-1))
        if (!(ok = next())) break;
        tc_fence_after();
        mma_half_kk(tmem + TM_DP, st_v, r.slot_addr(r.c), h, idesc_s, h == 0);
        release();
      }
      if (!ok) break;
      tc_commit(bar(R_DPFULL));
      if (!(ok = mbar_wait(bar(R_DSREADY), t & 1, wc))) break;
      for (int h = 0; ok && h < 2; ++h) {  // dK[:, half] += dS^T Q[:, half]
        if (!(ok = next())) break;
        tc_fence_after();
        mma_half_ts(tmem + TM_DK + 128 * h, tmem + TM_DP, r.slot_addr(r.c), idesc_g, t == 0);
        release();
      }
    }
    if (ok) tc_commit(bar(R_DONE));
    tc_commit(bar(R_DRAIN));
    mbar_wait(bar(R_DRAIN), 0, wc);
  } else if (warp >= 4) {
    const int h = (warp >> 2) - 1, wq = warp & 3, row = wq * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float sl2 = a.scale_log2;
    RowStage rs{reinterpret_cast<float*>(smem + L::OFF_L) + (warp - 4) * 64};
    bool ok = true;
    for (int t = 0; t < n_iter; ++t) {
      const int qt = i_begin + t;
      const size_t wrow = static_cast<size_t>(bh) * a.Npad + qt * kTileM + kEwCols2 * h + lane;
      const float my_l = a.lse2[wrow], my_d = a.delta[wrow];
      if (!(ok = mbar_wait_warp(bar(R_SFULL), t & 1, wc))) break;
      tc_fence_after();
      rs.put(my_l, my_d);
      const float4* l4 = rs.lse4();
      const float4* d4 = rs.d4();
      const int first_visible = a.causal ? k0 + row - a.cofs - qt * kTileM - kEwCols2 * h : 0;
      float p[kEwCols2];
      {
        uint32_t sv[kEwCols2];
        tmem_ld_x32(t_lane + TM_S + kEwCols2 * h, sv);
#pragma unroll
        for (int v = 0; v < kEwCols2 / 4; ++v) {
          const float4 lv = l4[v];
          p[4 * v + 0] = ex2(fmaf(__uint_as_float(sv[4 * v + 0]), sl2, -lv.x));
          p[4 * v + 1] = ex2(fmaf(__uint_as_float(sv[4 * v + 1]), sl2, -lv.y));
          p[4 * v + 2] = ex2(fmaf(__uint_as_float(sv[4 * v + 2]), sl2, -lv.z));
          p[4 * v + 3] = ex2(fmaf(__uint_as_float(sv[4 * v + 3]), sl2, -lv.w));
        }
      }
      if (first_visible > 0) {
#pragma unroll
        for (int c = 0; c < kEwCols2; ++c)
          if (c < first_visible) p[c] = 0.f;
      }
      if (!(ok = mbar_wait_warp(bar(R_DPFULL), t & 1, wc))) break;
      tc_fence_after();
      {
        uint32_t dv[kEwCols2], ds[kEwCols2 / 2];
        tmem_ld_x32(t_lane + TM_DP + kEwCols2 * h, dv);
#pragma unroll
        for (int v = 0; v < kEwCols2 / 4; ++v) {
          const float4 dd = d4[v];
          ds[2 * v] = pack2<BF16>(p[4 * v] * (__uint_as_float(dv[4 * v]) - dd.x),
                                  p[4 * v + 1] * (__uint_as_float(dv[4 * v + 1]) - dd.y));
          ds[2 * v + 1] = pack2<BF16>(p[4 * v + 2] * (__uint_as_float(dv[4 * v + 2]) - dd.z),
                                      p[4 * v + 3] * (__uint_as_float(dv[4 * v + 3]) - dd.w));
        }
        tmem_st_x16(t_lane + TM_DP + kEwCols2 * h, ds);  // over columns this thread has read
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(R_DSREADY));
    }
    if (ok) ok = mbar_wait_warp(bar(R_DONE), 0, wc);
    if (ok) {
      tc_fence_after();
      stage_acc256<BF16>(smem + L::OFF_RING, t_lane + TM_DK, row, h, a.scale);
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128 * kEw2);
    if (warp == 4 && lane == 0 && ok && !*abort_flag) {
      for (int b = 0; b < 4; ++b) tma_store_3d(&a.tm_dk, sb + L::OFF_RING + b * kBlk, 64 * b, k0, bh);
      bulk_commit();
      bulk_wait_read_all();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ dQ
// TMEM: S at 0, dP at 128 (dS over its first columns), dQ at 256..511.
template <bool BF16>
__global__ void __launch_bounds__(kThreads2, 1) bwd256_dq_kernel(const __grid_constant__ BwdArgs a) {
  constexpr int NSLOT = 2;
  using L = Layout256<NSLOT, 2>;  // Q, dO stationary
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bars = sb + L::OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 8 * R_COUNT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_BAR + 8 * R_COUNT + 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_t = (a.N + kTileM - 1) / kTileM;
  const WorkItem wi = work_item<2>(static_cast<int>(blockIdx.x), a.BH, n_t);
  const int bh = wi.bh, qt = n_t - 1 - wi.rank, q0 = qt * kTileM;
  const int n_kv = visible_key_tiles(qt, a.Nk, a.causal, a.cofs);
  const uint32_t tmem = prologue256(bars, NSLOT, abort_flag, tmem_slot, 128 * kEw2);
  const WaitCtl wc{abort_flag, a.dev_status, a.wait_limit_ns};
  constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DQ = 256;
  const uint32_t st_q = sb + L::OFF_ST, st_do = sb + L::OFF_ST + kTile;

  if (warp == 0 && lane == 0) {
    mbar_arrive_expect_tx(bar(R_STAT), 2 * kTile);
    for (int b = 0; b < 4; ++b) {
      tma_load_3d(st_q + b * kBlk, &a.tm_q, bar(R_STAT), 64 * b, q0, bh);
      tma_load_3d(st_do + b * kBlk, &a.tm_do, bar(R_STAT), 64 * b, q0, bh);
    }
    Ring<NSLOT> r{sb + L::OFF_RING, bars};
    bool ok = true;
    for (int j = 0; ok && j < n_kv; ++j) {  // K halves, V halves, K halves again
      const int kr = j * kTileN;
      ok = load_half(r, &a.tm_k, 0, kr, bh, wc) && load_half(r, &a.tm_k, 1, kr, bh, wc) &&
           load_half(r, &a.tm_v, 0, kr, bh, wc) && load_half(r, &a.tm_v, 1, kr, bh, wc) &&
           load_half(r, &a.tm_k, 0, kr, bh, wc) && load_half(r, &a.tm_k, 1, kr, bh, wc);
    }
    mbar_wait(bar(R_STAT), 0, wc);
    for (int c = (r.c > NSLOT ? r.c - NSLOT : 0); c < r.c; ++c) mbar_wait(r.full(c), (c / NSLOT) & 1, wc);
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc_s = idesc_f16(kTileM, kTileN, BF16, false, false);
    constexpr uint32_t idesc_g = idesc_f16(kTileM, 128, BF16, false, true);
    Ring<NSLOT> r{sb + L::OFF_RING, bars};
    auto next = [&]() -> bool { return mbar_wait(r.full(r.c), (r.c / NSLOT) & 1, wc); };
    auto release = [&]() { tc_commit(r.empty(r.c)); ++r.c; };
    bool ok = mbar_wait(bar(R_STAT), 0, wc);
    for (int j = 0; ok && j < n_kv; ++j) {
      for (int h = 0; ok && h < 2; ++h) {  // S = Q K^T (overwrites S(j-1), read before dS(j-1))
        if (!(ok = next())) break;
        tc_fence_after();
        mma_half_kk(tmem + TM_S, st_q, r.slot_addr(r.c), h, idesc_s, h == 0);
        release();
      }
      if (!ok) break;
      tc_commit(bar(R_SFULL));
      for (int h = 0; ok && h < 2; ++h) {  // dP = dO V^T (overwrites dS(j-1), read by dQ(j-1))
        if (!(ok = next())) break;
        tc_fence_after();
        mma_half_kk(tmem + TM_DP, st_do, r.slot_addr(r.c), h, idesc_s, h == 0);
        release();
      }
      if (!ok) break;
      tc_commit(bar(R_DPFULL));
      if (!(ok = mbar_wait(bar(R_DSREADY), j & 1, wc))) break;
      for (int h = 0; ok && h < 2; ++h) {  // dQ[:, half] += dS K[:, half]
        if (!(ok = next())) break;
        tc_fence_after();
        mma_half_ts(tmem + TM_DQ + 128 * h, tmem + TM_DP, r.slot_addr(r.c), idesc_g, j == 0);
        release();
      }
    }
    if (ok) tc_commit(bar(R_DONE));
    tc_commit(bar(R_DRAIN));
    mbar_wait(bar(R_DRAIN), 0, wc);
  } else if (warp >= 4) {
    const int h = (warp >> 2) - 1, wq = warp & 3, row = wq * 32 + lane, grow = q0 + row;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float sl2 = a.scale_log2;
    const size_t w = static_cast<size_t>(bh) * a.Npad + grow;  // grow < Npad always
    const float lse2 = a.lse2[w], dlt = a.delta[w];
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!(ok = mbar_wait_warp(bar(R_SFULL), j & 1, wc))) break;
      tc_fence_after();
      const int kbeg = j * kTileN + kEwCols2 * h;
      int lim = a.Nk - kbeg;                                     // keys past the end
      if (a.causal) lim = min(lim, grow + a.cofs - kbeg + 1);  // keys after this query
      float p[kEwCols2];
      {
        uint32_t sv[kEwCols2];
        tmem_ld_x32(t_lane + TM_S + kEwCols2 * h, sv);
#pragma unroll
        for (int e = 0; e < kEwCols2; ++e) p[e] = ex2(fmaf(__uint_as_float(sv[e]), sl2, -lse2));
      }
      if (lim < kEwCols2) {
#pragma unroll
        for (int c = 0; c < kEwCols2; ++c)
          if (c >= lim) p[c] = 0.f;
      }
      if (!(ok = mbar_wait_warp(bar(R_DPFULL), j & 1, wc))) break;
      tc_fence_after();
      {
        uint32_t dv[kEwCols2], ds[kEwCols2 / 2];
        tmem_ld_x32(t_lane + TM_DP + kEwCols2 * h, dv);
#pragma unroll
        for (int e = 0; e < kEwCols2; e += 2)
          ds[e / 2] = pack2<BF16>(p[e] * (__uint_as_float(dv[e]) - dlt), p[e + 1] * (__uint_as_float(dv[e + 1]) - dlt));
        tmem_st_x16(t_lane + TM_DP + kEwCols2 * h, ds);  // over columns this thread has read
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(R_DSREADY));
    }
    if (ok) ok = mbar_wait_warp(bar(R_DONE), 0, wc);
    if (ok) {
      tc_fence_after();
      stage_acc256<BF16>(smem + L::OFF_RING, t_lane + TM_DQ, row, h, a.scale);
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128 * kEw2);
    if (warp == 4 && lane == 0 && ok && !*abort_flag) {
      for (int b = 0; b < 4; ++b) tma_store_3d(&a.tm_dq, sb + L::OFF_RING + b * kBlk, 64 * b, q0, bh);
      bulk_commit();
      bulk_wait_read_all();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <class K>
cudaError_t launch256(K k, int smem, int grid, const BwdArgs& a, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k<<<grid, kThreads2, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd256_dkdv(const BwdArgs& a, bool bf16, cudaStream_t s) {
  const int grid = (a.Nk + kTileN - 1) / kTileN * a.BH;
  cudaError_t e = bf16 ? launch256(bwd256_dv_kernel<true>, Layout256<4, 1>::SMEM, grid, a, s)
                       : launch256(bwd256_dv_kernel<false>, Layout256<4, 1>::SMEM, grid, a, s);
  if (e != cudaSuccess) return e;
  return bf16 ? launch256(bwd256_dk_kernel<true>, Layout256<2, 2>::SMEM, grid, a, s)
              : launch256(bwd256_dk_kernel<false>, Layout256<2, 2>::SMEM, grid, a, s);
}

cudaError_t launch_bwd256_dq(const BwdArgs& a, bool bf16, cudaStream_t s) {
  const int grid = (a.N + kTileM - 1) / kTileM * a.BH;
  return bf16 ? launch256(bwd256_dq_kernel<true>, Layout256<2, 2>::SMEM, grid, a, s)
              : launch256(bwd256_dq_kernel<false>, Layout256<2, 2>::SMEM, grid, a, s);
}

}  // namespace attn
