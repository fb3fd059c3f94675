// bwd_pair.cu -- dK and dV for d = 128 on CTA pairs (tcgen05 cta_group::2) for sm_103a.
//
// The arithmetic is bwd_dkdv_kernel's (bwd.cu): per 128-key tile, for every visible
// 128-query tile, recompute S^T = K Q^T and P^T = 2^(S^T scale log2 e - LSE2), then
// dP^T = V dO^T, dS^T = P^T (dP^T - D), dV += P^T dO and dK += scale dS^T Q ("Understanding
// FlashAttention, Part 2", section 2.4).  What changes is who issues the products.  Two
// CTAs on neighbouring SMs form a cluster and take two consecutive key tiles, one each;
// one elected lane of the even CTA's issuing warp issues every product of both as an
// M = 256 pair product (tcgen05.mma.cta_group::2):
//
//   S^T, dP^T   A = K or V, each CTA its own 128 keys; B = Q or dO split along N (the
//               queries): each CTA supplies 64 of the tile's 128 query rows (all d)
//   dV, dK      A = P^T or dS^T from each CTA's tensor memory; B = dO or Q split along N
//               (d): each CTA supplies its 64 of the 128 columns for all 128 query rows
//
// so each CTA holds two views of every Q and dO tile (its query half with all columns,
// and its column half with all rows: 32 KB per tensor, what one CTA held before) and each
// SM reads half of every B operand per product step (per query tile ~128 KB of operand
// reads instead of ~192 KB, with the same 64 KB of TMA writes: in the one-CTA kernel
// those needed close to the SM's whole shared-memory bandwidth at the tensor core's
// rate).  Each CTA computes its own keys' P^T and dS^T with the one-CTA kernel's
// element-wise warpgroups and writes its own dK and dV.
//
// Hand-offs that gate a product (P^T written, dS^T written) arrive on the even CTA's
// barriers from the warps of both CTAs (the partner's through cluster addresses); every
// product completion is committed to both CTAs' barriers at once; the K, V, Q and dO
// copies of both CTAs complete on the even CTA's barriers (which expect the bytes of
// both), the per-query LSE2 and D rows on each CTA's own.  All waits are bounded; the
// first to expire raises the abort flag of both CTAs.  Causal pairs visit the query
// tiles of their earlier key tile: the later tile's first one is then wholly masked.
#include "bwd_common.cuh"

namespace attn {
namespace {

struct DkdvPairLayout {
  static constexpr int D = 128;
  static constexpr int TILE = kTileM * D * 2;        // 128 rows x 128 columns: 32 KB
  static constexpr int BLK = kTileM * 128;           // 128 rows x 64 columns: 16 KB
  static constexpr int BLK_H = 64 * 128;             // 64 rows x 64 columns: 8 KB
  static constexpr int STAGES = 2;
  // a stage: Q's query half (2 blocks of 64 rows), Q's column half (1 block of 128 rows),
  // the same for dO, then LSE2 and D of the tile's 128 queries
  static constexpr int S_QN = 0, S_QD = 2 * BLK_H, S_DON = 2 * BLK_H + BLK, S_DOD = 4 * BLK_H + BLK;
  static constexpr int S_L = 4 * BLK_H + 2 * BLK, S_D = S_L + 512;
  static constexpr int STAGE_BYTES = S_D + 512;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TILE;
  static constexpr int OFF_ST = 2 * TILE;
  static constexpr int OFF_BAR = OFF_ST + STAGES * STAGE_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 384, TM_COLS = 512;
  static_assert(S_QD + BLK == S_DON && S_DON + 2 * BLK_H == S_DOD, "stage layout");
};

enum : int {
  R_KVFULL = 0,   // both CTAs' K and V landed (CTA 0)
  R_SFULL = 1,    // S^T computed (both CTAs)
  R_DPFULL = 2,   // dP^T computed (both CTAs)
  R_PREADY = 3,   // P^T written by the pair's 32 element-wise warps (CTA 0)
  R_DSREADY = 4,  // dS^T written by the pair's 32 element-wise warps (CTA 0)
  R_DONE = 5,     // every product done (both CTAs)
  R_DRAIN = 6,    // (CTA 0)
  R_QFULL = 7,    // + stage: both CTAs' Q views landed (CTA 0)
  R_DOFULL = 9,   // + stage: both CTAs' dO views landed (CTA 0)
  R_ROWS = 11,    // + stage: this CTA's LSE2 and D rows landed (each CTA)
  R_EMPTY = 13,   // + stage: the stage's products done (both CTAs)
  R_COUNT = 15
};

// Bounded wait for the pair (as in the pair forward): an expired wait also raises the
// partner's abort flag.
struct PairWaitB {
  volatile int* abort;
  uint32_t peer_abort;
  int* dev_status;
  uint64_t limit_ns;
};

static __device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, const PairWaitB& w) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((n & 31) == 0) {
      if (*w.abort) return false;
      if (globaltimer_ns() - t0 > w.limit_ns) {
        *w.abort = 1;
        st_cluster_u32(w.peer_abort, 1u);
        if (w.dev_status) atomicExch(w.dev_status, kStatusTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool bwait_warp(uint32_t bar, uint32_t parity, const PairWaitB& w) {
  return __all_sync(0xffffffffu, bwait(bar, parity, w));
}

template <bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kBwdThreads, 1)
    bwd_dkdv_pair_kernel(const __grid_constant__ BwdArgs a) {
  using L = DkdvPairLayout;
  constexpr int D = L::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bars = sb + L::OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 8 * R_COUNT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_BAR + 8 * R_COUNT + 8);

  const uint32_t rank = cluster_ctarank();  // 0: the CTA that issues the products
  const bool lead = rank == 0;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_tk = (a.Nk + kTileN - 1) / kTileN;
  const int n_kp = (n_tk + 1) / 2;  // key-tile pairs per head
  const WorkItem wi = work_item(static_cast<int>(blockIdx.x >> 1), a.BH, n_kp);
  const int bh = wi.bh;
  const int kp = wi.rank;  // low key tiles see the most queries: they go first
  const int k0 = (2 * kp + static_cast<int>(rank)) * kTileN;  // this CTA's key tile
  const int n_t = (a.N + kTileM - 1) / kTileM;
  // the query tiles of the pair's earlier key tile
  const int i_begin = a.causal ? max(0, 2 * kp * kTileN - a.cofs) / kTileM : 0;
  const int n_iter = n_t - i_begin;

  if (threadIdx.x == 0) {
    mbar_init(bar(R_KVFULL), 1);
    mbar_init(bar(R_SFULL), 1);
    mbar_init(bar(R_DPFULL), 1);
    mbar_init(bar(R_PREADY), 2 * 4 * kEw);
    mbar_init(bar(R_DSREADY), 2 * 4 * kEw);
    mbar_init(bar(R_DONE), 1);
    mbar_init(bar(R_DRAIN), 1);
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(bar(R_QFULL + s), 1);
      mbar_init(bar(R_DOFULL + s), 1);
      mbar_init(bar(R_ROWS + s), 1);
      mbar_init(bar(R_EMPTY + s), 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), L::TM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before either touches the other's
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const PairWaitB wc{abort_flag, mapa_shared(smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u), a.dev_status,
                     a.wait_limit_ns};
  auto lead_bar = [&](int b) -> uint32_t { return mapa_shared(bar(b), 0); };
  auto stage_base = [&](int s) -> uint32_t { return sb + L::OFF_ST + s * L::STAGE_BYTES; };
  const int r64 = 64 * static_cast<int>(rank);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- TMA producer
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_qh);
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
      prefetch_tmap(&a.tm_do);
      prefetch_tmap(&a.tm_doh);
      if (lead) mbar_arrive_expect_tx(bar(R_KVFULL), 2 * 2 * L::TILE);
      for (int kb = 0; kb < 2; ++kb) {
        tma_load_3d_pair(sb + L::OFF_K + kb * L::BLK, &a.tm_k, lead_bar(R_KVFULL), kb * 64, k0, bh);
        tma_load_3d_pair(sb + L::OFF_V + kb * L::BLK, &a.tm_v, lead_bar(R_KVFULL), kb * 64, k0, bh);
      }
      int issued = 0;
      for (int t = 0; t < n_iter; ++t) {
        const int s = t % L::STAGES;
        const int q0 = (i_begin + t) * kTileM;
        if (t >= L::STAGES && !bwait(bar(R_EMPTY + s), ((t / L::STAGES) - 1) & 1, wc)) break;
        const uint32_t st = stage_base(s);
        if (lead) {
          mbar_arrive_expect_tx(bar(R_QFULL + s), 2 * L::TILE);
          mbar_arrive_expect_tx(bar(R_DOFULL + s), 2 * L::TILE);
        }
        mbar_arrive_expect_tx(bar(R_ROWS + s), 1024);
        for (int kb = 0; kb < 2; ++kb)  // Q's query half: rows q0 + 64 rank .. +63, all columns
          tma_load_3d_pair(st + L::S_QN + kb * L::BLK_H, &a.tm_qh, lead_bar(R_QFULL + s), kb * 64, q0 + r64, bh);
        tma_load_3d_pair(st + L::S_QD, &a.tm_q, lead_bar(R_QFULL + s), r64, q0, bh);  // column half
        const size_t w = static_cast<size_t>(bh) * a.Npad + q0;
        bulk_load(st + L::S_L, a.lse2 + w, 512, bar(R_ROWS + s));
        bulk_load(st + L::S_D, a.delta + w, 512, bar(R_ROWS + s));
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d_pair(st + L::S_DON + kb * L::BLK_H, &a.tm_doh, lead_bar(R_DOFULL + s), kb * 64, q0 + r64,
                           bh);
        tma_load_3d_pair(st + L::S_DOD, &a.tm_do, lead_bar(R_DOFULL + s), r64, q0, bh);
        issued = t + 1;
      }
      // Every copy lands before the CTA can exit: this CTA's rows here, both CTAs' tiles on
      // CTA 0's barriers (the partner leaves only after the final cluster barrier).
      for (int t = (issued > L::STAGES ? issued - L::STAGES : 0); t < issued; ++t) {
        bwait(bar(R_ROWS + t % L::STAGES), (t / L::STAGES) & 1, wc);
        if (lead) {
          bwait(bar(R_QFULL + t % L::STAGES), (t / L::STAGES) & 1, wc);
          bwait(bar(R_DOFULL + t % L::STAGES), (t / L::STAGES) & 1, wc);
        }
      }
      if (lead) bwait(bar(R_KVFULL), 0, wc);
    }
  } else if (warp == 1 && lead) {
    // ------------------------------------------------------------ pair product issuer
    // (the whole warp runs it, one elected lane issues)
    constexpr uint32_t idesc_s = idesc_f16(2 * kTileM, kTileM, BF16, false, false);  // keys x queries
    constexpr uint32_t idesc_g = idesc_f16(2 * kTileM, D, BF16, false, true);        // TMEM x MN-major
    constexpr uint16_t kBoth = 3;
    auto issue_st = [&](int t) {
      const uint32_t st = stage_base(t % L::STAGES);
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        mma_ss_pair_w(tmem + L::TM_S, sdesc_sw128(sb + L::OFF_K + (k >> 2) * L::BLK + (k & 3) * 32, 16, 1024),
                      sdesc_sw128(st + L::S_QN + (k >> 2) * L::BLK_H + (k & 3) * 32, 16, 1024), idesc_s,
                      k > 0 ? 1u : 0u);
      tc_commit_pair_w(bar(R_SFULL), kBoth);
    };
    bool ok = bwait_warp(bar(R_KVFULL), 0, wc);
    if (ok && n_iter > 0 && (ok = bwait_warp(bar(R_QFULL + 0), 0, wc))) {
      tc_fence_after();
      issue_st(0);
    }
    for (int t = 0; ok && t < n_iter; ++t) {
      const int s = t % L::STAGES;
      const uint32_t st = stage_base(s);
      if (!(ok = bwait_warp(bar(R_DOFULL + s), (t / L::STAGES) & 1, wc))) break;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        mma_ss_pair_w(tmem + L::TM_DP, sdesc_sw128(sb + L::OFF_V + (k >> 2) * L::BLK + (k & 3) * 32, 16, 1024),
                      sdesc_sw128(st + L::S_DON + (k >> 2) * L::BLK_H + (k & 3) * 32, 16, 1024), idesc_s,
                      k > 0 ? 1u : 0u);
      tc_commit_pair_w(bar(R_DPFULL), kBoth);
      if (!(ok = bwait_warp(bar(R_PREADY), t & 1, wc))) break;
      tc_fence_after();
      // 16-query steps; P^T of warpgroup w at S^T + 32w; B = dO's column half (MN-major)
#pragma unroll
      for (int k = 0; k < kTileM / 16; ++k)
        mma_ts_pair_w(tmem + L::TM_DV, tmem + L::TM_S + kEwCols * (k >> 1) + 8 * (k & 1),
                      sdesc_sw128(st + L::S_DOD + k * 2048, L::BLK, 1024), idesc_g, (t > 0 || k > 0) ? 1u : 0u);
      if (t + 1 < n_iter) {  // S^T(t+1) over P^T(t), issued after dV(t), which reads it
        if (!(ok = bwait_warp(bar(R_QFULL + (t + 1) % L::STAGES), ((t + 1) / L::STAGES) & 1, wc))) break;
        tc_fence_after();
        issue_st(t + 1);
      }
      if (!(ok = bwait_warp(bar(R_DSREADY), t & 1, wc))) break;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < kTileM / 16; ++k)
        mma_ts_pair_w(tmem + L::TM_DK, tmem + L::TM_DP + kEwCols * (k >> 1) + 8 * (k & 1),
                      sdesc_sw128(st + L::S_QD + k * 2048, L::BLK, 1024), idesc_g, (t > 0 || k > 0) ? 1u : 0u);
      tc_commit_pair_w(bar(R_EMPTY + s), kBoth);
    }
    if (ok) tc_commit_pair_w(bar(R_DONE), kBoth);
    tc_commit_pair_w(bar(R_DRAIN), 1);
    bwait_warp(bar(R_DRAIN), 0, wc);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ element-wise (own keys)
    const int h = (warp >> 2) - 1;      // this warpgroup's 32 query columns of every tile
    const int wq = warp & 3;
    const int row = wq * 32 + lane;     // key row within the tile == TMEM lane
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t t_s = t_lane + L::TM_S + kEwCols * h, t_dp = t_lane + L::TM_DP + kEwCols * h;
    const float sl2 = a.scale_log2;
    // One arrival per warp on CTA 0's barrier b.
    auto arrive_lead_warp = [&](int b) {
      __syncwarp();
      if (lane == 0) {
        if (lead)
          mbar_arrive(bar(b));
        else
          mbar_arrive_cluster(lead_bar(b));
      }
    };
    bool ok = true;
    for (int t = 0; t < n_iter; ++t) {
      const int s = t % L::STAGES;
      const int qt = i_begin + t;
      if (!(ok = bwait_warp(bar(R_ROWS + s), (t / L::STAGES) & 1, wc))) break;
      if (!(ok = bwait_warp(bar(R_SFULL), t & 1, wc))) break;
      tc_fence_after();
      const float4* l4 = reinterpret_cast<const float4*>(smem + L::OFF_ST + s * L::STAGE_BYTES + L::S_L) + (kEwCols / 4) * h;
      const float4* d4 = reinterpret_cast<const float4*>(smem + L::OFF_ST + s * L::STAGE_BYTES + L::S_D) + (kEwCols / 4) * h;
      // causal: query column c (query qt*128 + 32h + c) sees key k0 + row only if
      // qt*128 + 32h + c + cofs >= k0 + row
      const int first_visible = a.causal ? k0 + row - a.cofs - qt * kTileM - kEwCols * h : 0;
      float p[kEwCols];
      {
        uint32_t sv[kEwCols];
        tmem_ld_x32(t_s, sv);
        const uint64_t nsl2 = f32x2_pack(-sl2, -sl2);
#pragma unroll
        for (int v = 0; v < kEwCols / 4; ++v) {
          const float4 lv = l4[v];
          float x0, x1, x2, x3;
          f32x2_unpack(f32x2_fma(f32x2_pack(__uint_as_float(sv[4 * v]), __uint_as_float(sv[4 * v + 1])), nsl2,
                                 f32x2_pack(lv.x, lv.y)), x0, x1);
          f32x2_unpack(f32x2_fma(f32x2_pack(__uint_as_float(sv[4 * v + 2]), __uint_as_float(sv[4 * v + 3])), nsl2,
                                 f32x2_pack(lv.z, lv.w)), x2, x3);
          p[4 * v + 0] = ex2(-x0);
          p[4 * v + 1] = ex2(-x1);
          p[4 * v + 2] = ex2(-x2);
          p[4 * v + 3] = ex2(-x3);
        }
      }
      if (first_visible > 0) {
#pragma unroll
        for (int c = 0; c < kEwCols; ++c)
          if (c < first_visible) p[c] = 0.f;
      }
      {
        uint32_t pk[kEwCols / 2];
#pragma unroll
        for (int c = 0; c < kEwCols; c += 2) pk[c / 2] = pack2<BF16>(p[c], p[c + 1]);
        tmem_st_x16(t_s, pk);  // over columns this thread has read
      }
      tmem_st_wait();
      tc_fence_before();
      arrive_lead_warp(R_PREADY);
      if (!(ok = bwait_warp(bar(R_DPFULL), t & 1, wc))) break;
      tc_fence_after();
      {
        uint32_t dv[kEwCols], dk[kEwCols / 2];
        tmem_ld_x32(t_dp, dv);
#pragma unroll
        for (int v = 0; v < kEwCols / 4; ++v) {
          const float4 dd = d4[v];
          float a0, a1, b0, b1;
          f32x2_unpack(f32x2_mul(f32x2_pack(p[4 * v], p[4 * v + 1]),
                                 f32x2_sub(f32x2_pack(__uint_as_float(dv[4 * v]), __uint_as_float(dv[4 * v + 1])),
                                           f32x2_pack(dd.x, dd.y))), a0, a1);
          f32x2_unpack(f32x2_mul(f32x2_pack(p[4 * v + 2], p[4 * v + 3]),
                                 f32x2_sub(f32x2_pack(__uint_as_float(dv[4 * v + 2]), __uint_as_float(dv[4 * v + 3])),
                                           f32x2_pack(dd.z, dd.w))), b0, b1);
          dk[2 * v] = pack2<BF16>(a0, a1);
          dk[2 * v + 1] = pack2<BF16>(b0, b1);
        }
        tmem_st_x16(t_dp, dk);
      }
      tmem_st_wait();
      tc_fence_before();
      arrive_lead_warp(R_DSREADY);
    }
    if (ok) ok = bwait_warp(bar(R_DONE), 0, wc);
    // Epilogue: warpgroups 0-1 write dV, 2-3 write scale * dK (each half of the d columns),
    // through swizzled 32 KB staging tiles over stage 0 (every product of both CTAs is done).
    const int which = h >> 1;  // 0: dV, 1: dK
    uint8_t* stage = smem + L::OFF_ST + (which == 0 ? L::S_DON : L::S_QN);
    if (ok) {
      tc_fence_after();
      const uint32_t col = (which == 0) ? L::TM_DV : L::TM_DK;
      const float mul = (which == 0) ? 1.f : a.scale;
#pragma unroll
      for (int cc = (h & 1) * (D / 64); cc < ((h & 1) + 1) * (D / 64); ++cc) {
        uint32_t v[32];
        tmem_ld_x32(t_lane + col + cc * 32, v);
        stage_row_chunk<D, BF16>(stage, row, cc, v, mul);
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1 + which, 256);
    if ((h & 1) == 0 && (warp & 3) == 0 && lane == 0 && ok && !*abort_flag && k0 < a.Nk) {
      const CUtensorMap* m = (which == 0) ? &a.tm_dv : &a.tm_dk;
      for (int kb = 0; kb < 2; ++kb) tma_store_3d(m, smem_u32(stage) + kb * L::BLK, kb * 64, k0, bh);
      bulk_commit();
      bulk_wait_read_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the pair's products and copies are done before its tensor memory goes
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, L::TM_COLS);
  }
}

template <bool BF16>
cudaError_t launch_dkdv_pair_t(const BwdArgs& a, cudaStream_t st) {
  auto k = bwd_dkdv_pair_kernel<BF16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, DkdvPairLayout::SMEM);
  if (e != cudaSuccess) return e;
  const int n_tk = (a.Nk + kTileN - 1) / kTileN;
  k<<<dim3(2 * ((n_tk + 1) / 2) * a.BH), kBwdThreads, DkdvPairLayout::SMEM, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkdv_pair(const BwdArgs& a, bool bf16, cudaStream_t s) {
  return bf16 ? launch_dkdv_pair_t<true>(a, s) : launch_dkdv_pair_t<false>(a, s);
}

}  // namespace attn
