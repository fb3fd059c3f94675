// bwd_fused.cu -- the fused backward for d = 64 and 128: one CTA per 128-key tile
// computes dK and dV as the deterministic dK/dV kernel does and, from the same dS tile,
// adds each query tile's dQ contribution into a float32 accumulator in the workspace.
// Five N x N x d products per (key tile, query tile) pair -- the algorithm's count
// ("Understanding FlashAttention, Part 2", section 2.4, Figs 16-20: dQ accumulates over
// the key tiles while dK and dV stay with their key tile) -- against seven for the
// deterministic two-kernel backward, which recomputes S and dP in the query-tile order.
//
// Per query tile t the MMA warp issues, in this order,
//   dV += P^T dO | dP^T(t) = V dO^T | S^T(t+1) = K Q^T | dQ(t) = dS K | dK += dS^T Q
// P^T(t+1) = ex2(c S^T - LSE2) is computed while dQ(t) and dK(t) run; dS^T(t) =
// P^T (dP^T - D) while S^T(t+1) runs.  dS^T goes to a 128 x 128 16-bit
// shared-memory tile laid out [key][query] with the 128-byte swizzle: read K-major it
// is the A operand of dK (rows = keys), read MN-major it is the A operand of dQ (rows =
// queries), so both products take it without a transpose.  dQ(t) accumulates in the
// tensor-memory columns of dP^T, which are free once every element-wise thread has read
// dP^T(t); the element-wise warps read dQ(t) out while dK(t) and dV(t+1) run and add it to
// the accumulator through per-warp staging areas and TMA bulk reductions
// (cp.reduce.async.bulk .add.f32), and only then may
// dP^T(t+1) take the columns back.  The element-wise order per tile is therefore
//   P^T(t) | read out dQ(t-1) | dS^T(t)
// and the reductions, which the memory pipeline throttles, are issued while dP^T(t) runs.
//
// The accumulator's summation order depends on which CTA's reduction reaches a value
// first: dQ is not bit-for-bit reproducible from run to run (dK and dV are).  The
// deterministic kernels of bwd.cu stay available for callers that need identical bytes.
//
// DROP (dropout with the forward's keep mask, Z = keep * 256 / (256 - t)):
//   dV = (P o Z)^T dO,  dS = P o (Z o dP - D)   (D = rowsum(dO o O) with the dropped-out O)
// A thread owns a key and 32 queries, while one Philox call covers 16 keys of one query:
// each lane draws one query's bits over the warp's 32 keys (or reads them, as one word,
// from the keep bits the forward stored), and a warp transpose of the 32 x 32 bit block
// hands every lane its key's bits over the 32 queries.
#include <cuda_fp16.h>

#include "bwd_common.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kSmemMax = 232448;  // opt-in shared memory per CTA
constexpr int kStatusLayout = 3;  // ATTN_ERR_CUDA: the shared-memory window is misaligned

// Shared memory: K, V (stationary), STAGES x (Q, LSE2, D), one dO tile, the dS tile, the
// dQ staging area (2 KB per element-wise warp: half of the warp's 32 x 32 float32 share
// of dQ(t) at a time), barriers.  dO is read only by dV(t) and dP^T(t), which run back to
// back, so one buffer suffices: dO(t+1) is loaded once dP^T(t) is done and is not needed
// before dV(t+1), three products later.  At d = 128 this is 226.25 KB; dynamic shared
// memory starts 1024-byte aligned in practice and the slack below the opt-in limit
// covers a start misaligned by up to SLACK bytes (a kernel that finds more reports
// ATTN_ERR_CUDA and returns at once).
template <int D>
struct FusedLayout {
  using T = BwdTiles<D>;
  static constexpr int STAGES = (D == 128) ? 2 : 3;
  static constexpr int STAGE_BYTES = T::TILE + 2 * 512;  // Q, LSE2, D
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = T::TILE;
  static constexpr int OFF_ST = 2 * T::TILE;
  static constexpr int OFF_DO = OFF_ST + STAGES * STAGE_BYTES;
  static constexpr int OFF_DS = OFF_DO + T::TILE;
  static constexpr int DS_BYTES = kTileN * kTileM * 2;
  static constexpr int CHUNK = 32 * (D / 4) * 4;           // one warp's share of dQ(t): 32 rows x D/4 columns
  static constexpr int OFF_STG = OFF_DS + DS_BYTES;
  static constexpr int STG_BYTES = 16 * CHUNK / 2;         // half a share per element-wise warp
  static constexpr int OFF_BAR = OFF_STG + STG_BYTES;
  static constexpr int NEED = OFF_BAR + 256;
  static constexpr int SMEM = NEED + 1024 < kSmemMax ? NEED + 1024 : kSmemMax;
  static constexpr int SLACK = SMEM - NEED;
  static_assert(SLACK >= 0, "shared memory");
  static constexpr int S_Q = 0, S_L = T::TILE, S_D = T::TILE + 512;
  // dQ(t) shares dP^T's columns (see the file header)
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 256 + D, TM_DQ = TM_DP, TM_COLS = 512;
};

enum : int {
  F_KVFULL = 0,
  F_SFULL = 1,    // S^T computed (MMA commit)
  F_DPFULL = 2,   // dP^T computed (MMA commit)
  F_PREADY = 3,   // P^T written to tensor memory (all element-wise threads)
  F_DSREADY = 4,  // dS^T written to shared memory (all element-wise threads)
  F_DQFULL = 5,   // dQ(t) computed (MMA commit)
  F_DQFREE = 6,   // dQ(t) read out of tensor memory (all element-wise threads)
  F_DONE = 7,
  F_DRAIN = 8,
  F_DOFULL = 9,   // dO(t) loaded
  F_DOFREE = 10,  // dP^T(t), the last reader of dO(t), done (MMA commit)
  F_QFULL = 11,   // + stage: Q(t), LSE2, D loaded
  F_EMPTY = 14,   // + stage: dK(t), the last reader of Q(t), done (MMA commit)
  F_COUNT = 17
};
static_assert(8 * F_COUNT + 16 <= 256, "barrier area");

// TMA tensor reduction (add, float32) of one staged box into the accumulator at
// (column c0, row c1) (bulk-group completion).
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* m, uint32_t src, int c0, int c1) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(src), "r"(c0), "r"(c1)
               : "memory");
}

// This warp's share of dQ(t) -- rows 32 wq .. 32 wq + 31 of the query tile (one per lane),
// columns (D/4) h .. (D/4)(h+1) - 1 -- added to the accumulator.  The share goes through
// the warp's staging area in two halves of 16 rows; each half is one box of the
// accumulator's tensor map, handed to the TMA unit as one reduction.  Before a half is
// written, the previous reduction must have finished reading the area.  The area is
// swizzled as the map expects (16-byte piece c of row r at piece c ^ (r mod 8) of a
// 128-byte row at d = 128, c ^ ((r / 2) mod 4) of a 64-byte row at d = 64), which also
// spreads the 16 lanes' stores over all banks.
template <int D>
__device__ __forceinline__ void dq_stage_reduce(const CUtensorMap* acc, int col0, int row0, uint8_t* stg, int lane,
                                                const uint32_t* v) {
  constexpr int ROW_BYTES = D;  // D/4 floats
  constexpr int PIECES = D / 16;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
    if ((lane >> 4) == half) {
      const int r = lane & 15;
      const int sw = (D == 128) ? (r & 7) : ((r >> 1) & 3);
#pragma unroll
      for (int c = 0; c < PIECES; ++c)
        *reinterpret_cast<uint4*>(stg + r * ROW_BYTES + ((c ^ sw) << 4)) =
            make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
      fence_proxy_async_smem();
    }
    __syncwarp();
    if (lane == 0) {
      tma_reduce_add_2d(acc, smem_u32(stg), col0, row0 + 16 * half);
      bulk_commit();
    }
  }
}

template <int D, bool BF16, bool VARLEN, bool DROP>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_fused_kernel(const __grid_constant__ BwdArgs a) {
  using L = FusedLayout<D>;
  using T = BwdTiles<D>;
  extern __shared__ uint8_t smem_raw[];
  const uintptr_t raw = reinterpret_cast<uintptr_t>(smem_raw);
  const uintptr_t aligned = (raw + 1023) & ~static_cast<uintptr_t>(1023);
  if (aligned - raw > static_cast<uintptr_t>(L::SLACK)) {
    if (threadIdx.x == 0 && a.dev_status) atomicExch(a.dev_status, kStatusLayout);
    return;
  }
  uint8_t* smem = reinterpret_cast<uint8_t*>(aligned);
  const uint32_t sb = smem_u32(smem);
  const uint32_t bars = sb + L::OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 8 * F_COUNT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_BAR + 8 * F_COUNT + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_tk = (a.Nk + kTileN - 1) / kTileN;
  const WorkItem wi = work_item(static_cast<int>(blockIdx.x), a.BH, n_tk);
  const int bh = wi.bh;
  const int kt = wi.rank;  // low key tiles see the most queries: they go first
  const int k0 = kt * kTileN;
  int N = a.N, cofs = a.cofs, hh = 0, tq0 = 0, tk0 = 0, Nk = a.Nk;
  if constexpr (VARLEN) {
    const SeqView sv = seq_view(a, bh);
    N = sv.N, Nk = sv.Nk, cofs = sv.cofs, hh = sv.hh, tq0 = sv.tq0, tk0 = sv.tk0;
    if (k0 >= Nk) return;  // this key tile lies past the sequence's keys (whole CTA)
    if (sv.degenerate || N <= 0) {
      zero_rows_packed<D>(a.dk_out, a.H, hh, tk0, k0, Nk);
      zero_rows_packed<D>(a.dv_out, a.H, hh, tk0, k0, Nk);
      return;  // the accumulator rows stay zero: dQ = 0
    }
  }
  const int n_t = (N + kTileM - 1) / kTileM;
  const int i_begin = a.causal ? max(0, k0 - cofs) / kTileM : 0;
  const int n_iter = n_t - i_begin;

  if (threadIdx.x == 0) {
    mbar_init(bar(F_KVFULL), 1);
    mbar_init(bar(F_SFULL), 1);
    mbar_init(bar(F_DPFULL), 1);
    mbar_init(bar(F_PREADY), 128 * kEw);
    mbar_init(bar(F_DSREADY), 128 * kEw);
    mbar_init(bar(F_DQFULL), 1);
    mbar_init(bar(F_DQFREE), 128 * kEw);
    mbar_init(bar(F_DONE), 1);
    mbar_init(bar(F_DRAIN), 1);
    mbar_init(bar(F_DOFULL), 1);
    mbar_init(bar(F_DOFREE), 1);
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(bar(F_QFULL + s), 1);
      mbar_init(bar(F_EMPTY + s), 1);
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
      prefetch_tmap(&a.tm_dqacc);
      mbar_arrive_expect_tx(bar(F_KVFULL), 2 * T::TILE);
      for (int kb = 0; kb < T::KB; ++kb) {
        tma_load_3d(sb + L::OFF_K + kb * T::BLK, &a.tm_k, bar(F_KVFULL), kb * 64, VARLEN ? hh : k0,
                    VARLEN ? tk0 + k0 : bh);
        tma_load_3d(sb + L::OFF_V + kb * T::BLK, &a.tm_v, bar(F_KVFULL), kb * 64, VARLEN ? hh : k0,
                    VARLEN ? tk0 + k0 : bh);
      }
      int issued = 0, do_issued = 0;
      for (int t = 0; t < n_iter; ++t) {
        const int s = t % L::STAGES;
        const int q0 = (i_begin + t) * kTileM;
        if (t >= L::STAGES && !mbar_wait(bar(F_EMPTY + s), ((t / L::STAGES) - 1) & 1, wc)) break;
        const uint32_t st = stage_base(s);
        mbar_arrive_expect_tx(bar(F_QFULL + s), T::TILE + 1024);
        for (int kb = 0; kb < T::KB; ++kb)
          tma_load_3d(st + L::S_Q + kb * T::BLK, &a.tm_q, bar(F_QFULL + s), kb * 64, VARLEN ? hh : q0,
                      VARLEN ? tq0 + q0 : bh);
        const size_t w = static_cast<size_t>(bh) * a.Npad + q0;
        bulk_load(st + L::S_L, a.lse2 + w, 512, bar(F_QFULL + s));
        bulk_load(st + L::S_D, a.delta + w, 512, bar(F_QFULL + s));
        issued = t + 1;
        if (t > 0 && !mbar_wait(bar(F_DOFREE), (t - 1) & 1, wc)) break;
        mbar_arrive_expect_tx(bar(F_DOFULL), T::TILE);
        for (int kb = 0; kb < T::KB; ++kb)
          tma_load_3d(sb + L::OFF_DO + kb * T::BLK, &a.tm_do, bar(F_DOFULL), kb * 64, VARLEN ? hh : q0,
                      VARLEN ? tq0 + q0 : bh);
        do_issued = t + 1;
      }
      mbar_wait(bar(F_KVFULL), 0, wc);
      for (int t = (issued > L::STAGES ? issued - L::STAGES : 0); t < issued; ++t)
        mbar_wait(bar(F_QFULL + t % L::STAGES), (t / L::STAGES) & 1, wc);
      if (do_issued > 0) mbar_wait(bar(F_DOFULL), (do_issued - 1) & 1, wc);
    }
  } else if (warp == 1) {
    // The whole warp runs the issuing loop; one elected lane issues each product.
    constexpr uint32_t idesc_s = idesc_f16(kTileM, kTileM, BF16, false, false);  // K-major x K-major
    constexpr uint32_t idesc_g = idesc_f16(kTileM, D, BF16, false, true);        // K-major A x MN-major B
    constexpr uint32_t idesc_q = idesc_f16(kTileM, D, BF16, true, true);         // MN-major A x MN-major B
    const uint32_t ds = sb + L::OFF_DS;
    auto issue_st = [&](int t) {
      const uint32_t st = stage_base(t % L::STAGES);
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * T::BLK + (k & 3) * 32;
        mma_ss_w(tmem + L::TM_S, sdesc_sw128(sb + L::OFF_K + off, 16, 1024), sdesc_sw128(st + L::S_Q + off, 16, 1024),
                 idesc_s, k > 0 ? 1u : 0u);
      }
      tc_commit_w(bar(F_SFULL));
    };
    bool ok = mbar_wait_warp(bar(F_KVFULL), 0, wc);
    if (ok && n_iter > 0 && (ok = mbar_wait_warp(bar(F_QFULL + 0), 0, wc))) {
      tc_fence_after();
      issue_st(0);
    }
    for (int t = 0; ok && t < n_iter; ++t) {
      const int s = t % L::STAGES;
      const uint32_t st = stage_base(s);
      if (!(ok = mbar_wait_warp(bar(F_PREADY), t & 1, wc) && mbar_wait_warp(bar(F_DOFULL), t & 1, wc))) break;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < kTileM / 16; ++k)  // 16-query steps; P^T of warpgroup w at S^T + 32w
        mma_ts_w(tmem + L::TM_DV, tmem + L::TM_S + kEwCols * (k >> 1) + 8 * (k & 1),
                 sdesc_sw128(sb + L::OFF_DO + k * 2048, T::BLK, 1024), idesc_g, (t > 0 || k > 0) ? 1u : 0u);
      // dP^T(t) takes dQ(t-1)'s columns once the element-wise warps have read them; dK(t-1)
      // and dV(t) run meanwhile.
      if (t > 0 && !(ok = mbar_wait_warp(bar(F_DQFREE), (t - 1) & 1, wc))) break;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * T::BLK + (k & 3) * 32;
        mma_ss_w(tmem + L::TM_DP, sdesc_sw128(sb + L::OFF_V + off, 16, 1024),
                 sdesc_sw128(sb + L::OFF_DO + off, 16, 1024), idesc_s, k > 0 ? 1u : 0u);
      }
      tc_commit_w(bar(F_DPFULL));
      tc_commit_w(bar(F_DOFREE));
      if (t + 1 < n_iter) {  // S^T(t+1) over P^T(t): issued after dV(t), which reads it
        if (!(ok = mbar_wait_warp(bar(F_QFULL + (t + 1) % L::STAGES), ((t + 1) / L::STAGES) & 1, wc))) break;
        tc_fence_after();
        issue_st(t + 1);
      }
      if (!(ok = mbar_wait_warp(bar(F_DSREADY), t & 1, wc))) break;
      tc_fence_after();
      // dQ(t) = dS K: A = dS read MN-major from the [key][query] tile (16-key steps of
      // 16 rows), B = K MN-major (d contiguous).
#pragma unroll
      for (int k = 0; k < kTileN / 16; ++k)
        mma_ss_w(tmem + L::TM_DQ, sdesc_sw128(ds + k * 2048, T::BLK, 1024),
                 sdesc_sw128(sb + L::OFF_K + k * 2048, T::BLK, 1024), idesc_q, k > 0 ? 1u : 0u);
      tc_commit_w(bar(F_DQFULL));
      // dK += dS^T Q: A = dS^T read K-major from the same tile (16-query steps).
#pragma unroll
      for (int k = 0; k < kTileM / 16; ++k)
        mma_ss_w(tmem + L::TM_DK, sdesc_sw128(ds + (k >> 2) * T::BLK + (k & 3) * 32, 16, 1024),
                 sdesc_sw128(st + L::S_Q + k * 2048, T::BLK, 1024), idesc_g, (t > 0 || k > 0) ? 1u : 0u);
      tc_commit_w(bar(F_EMPTY + s));
    }
    if (ok) tc_commit_w(bar(F_DONE));
    tc_commit_w(bar(F_DRAIN));
    mbar_wait_warp(bar(F_DRAIN), 0, wc);
  } else if (warp >= 4) {
    const int h = (warp >> 2) - 1;   // this warpgroup's 32 query columns of every tile
    const int wq = warp & 3;
    const int row = wq * 32 + lane;  // key row within the tile == TMEM lane (query row for dQ)
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t t_s = t_lane + L::TM_S + kEwCols * h, t_dp = t_lane + L::TM_DP + kEwCols * h;
    const float sl2 = a.scale_log2;
    uint8_t* ds_tile = smem + L::OFF_DS;
    uint8_t* stg = smem + L::OFF_STG + (warp - 4) * (L::CHUNK / 2);
    // Reads dQ(t) (this thread's query row, the warpgroup's D/4 columns) out of tensor
    // memory, frees the columns and adds the warp's share to the accumulator.
    auto drain = [&](int t) -> bool {
      if (!mbar_wait_warp(bar(F_DQFULL), t & 1, wc)) return false;
      tc_fence_after();
      uint32_t v[D / 4];
      if constexpr (D == 128)
        tmem_ld_x32(t_lane + L::TM_DQ + (D / 4) * h, v);
      else
        tmem_ld_x16(t_lane + L::TM_DQ + (D / 4) * h, v);
      tc_fence_before();
      mbar_arrive(bar(F_DQFREE));
      // rows of this warp in the accumulator: head bh's padded rows; rows past the end hold
      // zeros (their dS is zero) and add nothing
      dq_stage_reduce<D>(&a.tm_dqacc, (D / 4) * h, bh * a.Npad + (i_begin + t) * kTileM + 32 * wq, stg, lane, v);
      return true;
    };
    bool ok = true;
    for (int t = 0; t < n_iter; ++t) {
      const int s = t % L::STAGES;
      const int qt = i_begin + t;
      uint32_t keepbits = 0xffffffffu;  // bit c: query column 32h + c keeps this thread's key
      if constexpr (DROP) {
        // lane L draws query qt*128 + 32h + L's bits over keys k0 + 32wq .. +31
        const uint32_t qi = static_cast<uint32_t>(qt * kTileM + kEwCols * h + lane);
        const uint32_t jg = static_cast<uint32_t>((k0 + 32 * wq) / 16);
        uint32_t mine;
        if (a.keep_bits != nullptr)  // the forward's stored decisions (same bits, no draw)
          mine = a.keep_bits[(static_cast<size_t>(bh) * n_tk + kt) * 4 * a.bits_rows +
                             static_cast<size_t>(wq) * a.bits_rows + qi];
        else
          mine = dropout_keep16(jg, qi, static_cast<uint32_t>(bh), a.drop_t, a.seed_lo, a.seed_hi) |
                 (dropout_keep16(jg + 1, qi, static_cast<uint32_t>(bh), a.drop_t, a.seed_lo, a.seed_hi) << 16);
        keepbits = warp_transpose32(mine);
      }
      if (!(ok = mbar_wait_warp(bar(F_QFULL + s), (t / L::STAGES) & 1, wc))) break;
      if (!(ok = mbar_wait_warp(bar(F_SFULL), t & 1, wc))) break;
      tc_fence_after();
      const float4* l4 =
          reinterpret_cast<const float4*>(smem + L::OFF_ST + s * L::STAGE_BYTES + L::S_L) + (kEwCols / 4) * h;
      const float4* d4 =
          reinterpret_cast<const float4*>(smem + L::OFF_ST + s * L::STAGE_BYTES + L::S_D) + (kEwCols / 4) * h;
      // Query column c sees key k0 + row only if the key exists (in a packed batch the
      // rows past the sequence's last key hold the next sequence's keys, which must not
      // reach dQ) and, causal, if qt*128 + 32h + c + cofs >= k0 + row.
      const int first_visible = k0 + row >= Nk ? kEwCols
                                : a.causal    ? k0 + row - cofs - qt * kTileM - kEwCols * h
                                              : 0;
      float p[kEwCols];
      {  // P^T = 2^-(lse2 - s sl2) (overlaps dQ(t-1) and dK(t-1))
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
        if constexpr (DROP) {  // dV takes P o Z
          const float zs = a.drop_scale;
#pragma unroll
          for (int c = 0; c < kEwCols; c += 2)
            pk[c / 2] = pack2<BF16>(((keepbits >> c) & 1u) ? p[c] * zs : 0.f,
                                    ((keepbits >> (c + 1)) & 1u) ? p[c + 1] * zs : 0.f);
        } else {
#pragma unroll
          for (int c = 0; c < kEwCols; c += 2) pk[c / 2] = pack2<BF16>(p[c], p[c + 1]);
        }
        tmem_st_x16(t_s, pk);  // over columns this thread has read
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(F_PREADY));
      // dQ(t-1) out of tensor memory (it completed before dK(t-1); dP^T(t) waits for it).
      if (t > 0 && !(ok = drain(t - 1))) break;
      // dS^T = P^T (dP^T - D) into the shared [key][query] tile (overlaps S^T(t+1)).
      if (!(ok = mbar_wait_warp(bar(F_DPFULL), t & 1, wc))) break;
      tc_fence_after();
      {
        uint32_t dv[kEwCols], dk[kEwCols / 2];
        tmem_ld_x32(t_dp, dv);
        if constexpr (DROP) {  // dP <- Z o dP
          const float zs = a.drop_scale;
#pragma unroll
          for (int c = 0; c < kEwCols; ++c)
            dv[c] = __float_as_uint(((keepbits >> c) & 1u) ? __uint_as_float(dv[c]) * zs : 0.f);
        }
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
        // queries 32h .. 32h+31 of key row `row`: 64 bytes in block h/2, 16-byte chunks
        // (h%2)*4 .. +3 of the row, swizzled by the row's low three bits
        uint8_t* base = ds_tile + (h >> 1) * T::BLK + row * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int ch = (h & 1) * 4 + c;
          *reinterpret_cast<uint4*>(base + ((ch ^ (row & 7)) << 4)) =
              make_uint4(dk[4 * c], dk[4 * c + 1], dk[4 * c + 2], dk[4 * c + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(F_DSREADY));
    }
    if (ok && n_iter > 0) ok = drain(n_iter - 1);
    if (lane == 0) bulk_wait_all();  // this warp's bulk reductions are done
    if (ok) ok = mbar_wait_warp(bar(F_DONE), 0, wc);
    // Epilogue: warpgroups 0-1 write dV, 2-3 write scale * dK, as the dK/dV kernel does.
    const int which = h >> 1;
    uint8_t* stage = smem + (which == 0 ? L::OFF_DO : L::OFF_ST + L::S_Q);
    if (ok) {
      tc_fence_after();
      const uint32_t col = (which == 0) ? L::TM_DV : L::TM_DK;
      const float mul = (which == 0) ? 1.f : a.scale;
#pragma unroll
      for (int cc = (h & 1) * (D / 64); cc < ((h & 1) + 1) * (D / 64); ++cc) {
        uint32_t v[32];
        tmem_ld_x32(t_lane + col + cc * 32, v);
        if constexpr (VARLEN) {
          if (k0 + row < Nk)
            store_row_chunk_packed<D, BF16>(which == 0 ? a.dv_out : a.dk_out,
                                            (static_cast<size_t>(tk0 + k0 + row) * a.H + hh) * D, cc, v, mul);
        } else {
          stage_row_chunk<D, BF16>(stage, row, cc, v, mul);
        }
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1 + which, 256);
    if (!VARLEN && (h & 1) == 0 && (warp & 3) == 0 && lane == 0 && ok && !*abort_flag) {
      const CUtensorMap* m = (which == 0) ? &a.tm_dv : &a.tm_dk;
      for (int kb = 0; kb < T::KB; ++kb) tma_store_3d(m, smem_u32(stage) + kb * T::BLK, kb * 64, k0, bh);
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

// dQ = scale * accumulator, rounded to the 16-bit type: one thread per 8 columns of a row
// (two float32 vector loads, one 16-byte store; consecutive threads cover consecutive
// columns, so both sides are coalesced).
template <int D, bool BF16, bool VARLEN>
__global__ void __launch_bounds__(256) bwd_dq_finish_kernel(const __grid_constant__ BwdArgs a) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = idx / (D / 8);
  const int u = static_cast<int>(idx % (D / 8));
  if (row >= static_cast<int64_t>(a.BH) * a.Npad) return;
  const int bh = static_cast<int>(row / a.Npad), r = static_cast<int>(row % a.Npad);
  int N = a.N, hh = 0, tq0 = 0;
  if constexpr (VARLEN) {
    const SeqView sv = seq_view(a, bh);
    N = sv.N, hh = sv.hh, tq0 = sv.tq0;
  }
  if (r >= N) return;
  const float4* src = reinterpret_cast<const float4*>(a.dq_acc + row * D + u * 8);
  const float4 x0 = src[0], x1 = src[1];
  const float sc = a.scale;
  const uint4 out = make_uint4(pack2<BF16>(x0.x * sc, x0.y * sc), pack2<BF16>(x0.z * sc, x0.w * sc),
                               pack2<BF16>(x1.x * sc, x1.y * sc), pack2<BF16>(x1.z * sc, x1.w * sc));
  size_t elem;
  if constexpr (VARLEN)
    elem = (static_cast<size_t>(tq0 + r) * a.H + hh) * D + u * 8;
  else
    elem = (static_cast<size_t>(bh) * a.N + r) * D + u * 8;
  *reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.dq) + elem * 2) = out;
}

template <int D, bool BF16, bool VARLEN, bool DROP>
cudaError_t launch_fused_t(const BwdArgs& a, cudaStream_t st) {
  auto k = bwd_fused_kernel<D, BF16, VARLEN, DROP>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, FusedLayout<D>::SMEM);
  if (e != cudaSuccess) return e;
  const int n_tk = (a.Nk + kTileN - 1) / kTileN;
  k<<<n_tk * a.BH, kBwdThreads, FusedLayout<D>::SMEM, st>>>(a);
  return cudaGetLastError();
}

template <int D, bool BF16, bool VARLEN>
cudaError_t launch_finish_t(const BwdArgs& a, cudaStream_t st) {
  const int64_t threads = static_cast<int64_t>(a.BH) * a.Npad * (D / 8);
  bwd_dq_finish_kernel<D, BF16, VARLEN><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_fused_d(const BwdArgs& a, bool varlen, cudaStream_t s) {
  if (a.drop_t > 0)
    return varlen ? launch_fused_t<D, BF16, true, true>(a, s) : launch_fused_t<D, BF16, false, true>(a, s);
  return varlen ? launch_fused_t<D, BF16, true, false>(a, s) : launch_fused_t<D, BF16, false, false>(a, s);
}

}  // namespace

// a.drop_t > 0 selects the dropout kernels.
cudaError_t launch_bwd_fused(const BwdArgs& a, int d, bool bf16, bool varlen, cudaStream_t s) {
  if (d == 128) return bf16 ? launch_fused_d<128, true>(a, varlen, s) : launch_fused_d<128, false>(a, varlen, s);
  return bf16 ? launch_fused_d<64, true>(a, varlen, s) : launch_fused_d<64, false>(a, varlen, s);
}

cudaError_t launch_bwd_dq_finish(const BwdArgs& a, int d, bool bf16, bool varlen, cudaStream_t s) {
  if (varlen) {
    if (d == 128) return bf16 ? launch_finish_t<128, true, true>(a, s) : launch_finish_t<128, false, true>(a, s);
    return bf16 ? launch_finish_t<64, true, true>(a, s) : launch_finish_t<64, false, true>(a, s);
  }
  if (d == 128) return bf16 ? launch_finish_t<128, true, false>(a, s) : launch_finish_t<128, false, false>(a, s);
  return bf16 ? launch_finish_t<64, true, false>(a, s) : launch_finish_t<64, false, false>(a, s);
}

}  // namespace attn
