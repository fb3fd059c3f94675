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
//
// DROP (dropout, with the forward's keep mask and scale Z = keep * 256 / (256 - t)):
//   dV = (P o Z)^T dO,  dS = P o (Z o dP - D); D = rowsum(dO o O) still equals
//   sum_k P_ik Z_ik dP_ik because O is the dropped-out output.
#include <cuda_fp16.h>

#include "bwd_common.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

// ------------------------------------------------------------------ bwd_pre

// D = D/8 lanes per row, 16 bytes of O and of dO per lane; a warp covers 32/(D/8) rows
// per step and kPreUnroll steps with every load issued before any arithmetic.
constexpr int kPreUnroll = 4;

template <int D, bool BF16>
__device__ __forceinline__ float dot8(const uint4& x, const uint4& y) {
  const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float x0, x1, y0, y1;
    if constexpr (BF16) {
      x0 = __uint_as_float(xs[i] << 16);
      x1 = __uint_as_float(xs[i] & 0xffff0000u);
      y0 = __uint_as_float(ys[i] << 16);
      y1 = __uint_as_float(ys[i] & 0xffff0000u);
    } else {
      const float2 xf = __half22float2(*reinterpret_cast<const __half2*>(&xs[i]));
      const float2 yf = __half22float2(*reinterpret_cast<const __half2*>(&ys[i]));
      x0 = xf.x, x1 = xf.y, y0 = yf.x, y1 = yf.y;
    }
    acc = fmaf(x0, y0, acc);
    acc = fmaf(x1, y1, acc);
  }
  return acc;
}

// VARLEN: rows (bh, r) of one packed sequence read token tq0 + r of head hh; rows past
// the sequence, and every row of a degenerate sequence, get LSE2 = +inf and D = 0.
template <int D, bool BF16, bool VARLEN>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __grid_constant__ BwdArgs a) {
  constexpr int LPR = D / 8;         // lanes per row
  constexpr int RPW = 32 / LPR;      // rows per warp step
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t rows = static_cast<int64_t>(a.BH) * a.Npad;
  const int sub = lane / LPR, col = lane % LPR;
  uint4 ov[kPreUnroll], dv[kPreUnroll];
  int64_t rr[kPreUnroll];
#pragma unroll
  for (int u = 0; u < kPreUnroll; ++u) {
    rr[u] = (warp_global * kPreUnroll + u) * RPW + sub;
    ov[u] = dv[u] = make_uint4(0, 0, 0, 0);
    if (rr[u] < rows) {
      const int bh = static_cast<int>(rr[u] / a.Npad), r = static_cast<int>(rr[u] % a.Npad);
      bool valid = r < a.N;
      size_t off = ((static_cast<size_t>(bh) * a.N + r) * D) * 2 + col * 16;
      if constexpr (VARLEN) {
        const SeqView sv = seq_view(a, bh);
        valid = r < sv.N && !sv.degenerate;
        off = ((static_cast<size_t>(sv.tq0 + r) * a.H + sv.hh) * D) * 2 + col * 16;
      }
      if (valid) {
        ov[u] = *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.o) + off);
        dv[u] = *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.dout) + off);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kPreUnroll; ++u) {
    float dsum = dot8<D, BF16>(ov[u], dv[u]);
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
    if (col == 0 && rr[u] < rows) {
      const int bh = static_cast<int>(rr[u] / a.Npad), r = static_cast<int>(rr[u] % a.Npad);
      const size_t w = static_cast<size_t>(bh) * a.Npad + r;
      bool valid = r < a.N;
      size_t li = static_cast<size_t>(bh) * a.N + r;
      if constexpr (VARLEN) {
        const SeqView sv = seq_view(a, bh);
        valid = r < sv.N && !sv.degenerate;
        li = static_cast<size_t>(sv.hh) * a.Tq + sv.tq0 + r;
      }
      a.delta[w] = valid ? dsum : 0.f;
      a.lse2[w] = valid ? a.lse[li] * 1.4426950408889634f : INFINITY;
    }
  }
  if (a.dq_acc != nullptr) {
    // The fused backward's dQ accumulator starts at zero: each block clears as many of its
    // values as its rows hold (the accumulator is B*H*Npad*D floats, covered block by block).
    constexpr int64_t kBlockRows = (256 / 32) * kPreUnroll * RPW;
    const int64_t beg = static_cast<int64_t>(blockIdx.x) * kBlockRows * D;
    const int64_t n = min(kBlockRows * D, rows * D - beg);
    float4* z = reinterpret_cast<float4*>(a.dq_acc + beg);
    for (int64_t i = threadIdx.x; i < n / 4; i += blockDim.x) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// ------------------------------------------------------------------ bwd_dkdv
//
// Element-wise warpgroup w handles queries 32w..32w+31 of every tile (every
// tensor-core product keeps N >= 128: the tcgen05.mma issue cost does not shrink
// below N = 128).  Per query tile the MMA
// warp issues, in this order,
//   S^T = K Q^T | dP^T = V dO^T | dV += P^T dO | dK += dS^T Q
// and the element-wise work is split in two phases so that each overlaps a
// product: P^T = ex2(c S^T - LSE2) while dP^T is computed, then
// dS^T = P^T (dP^T - D) while dV is computed.  P^T and dS^T go back as 16-bit
// pairs over the first half of each warpgroup's own S^T / dP^T columns.  The next
// tile's S^T / dP^T overwrite those columns; one thread issues every product and
// the tensor core executes one thread's MMAs in order.

template <int D>
struct DkdvLayout {
  using T = BwdTiles<D>;
  static constexpr int STAGES = (D == 128) ? 2 : 3;
  static constexpr int STAGE_BYTES = 2 * T::TILE + 2 * 512;  // Q_i, dO_i, LSE2_i, D_i
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = T::TILE;
  static constexpr int OFF_ST = 2 * T::TILE;
  static constexpr int OFF_BAR = OFF_ST + STAGES * STAGE_BYTES;
  static constexpr int OFF_DROP = OFF_BAR + 256;           // dropout: 1 KB per element-wise warp
  static constexpr int DROP_BYTES = 32 * 4 * kEw * 32;
  static constexpr int SMEM = OFF_DROP + 1024;             // + DROP_BYTES with dropout
  static constexpr int S_Q = 0, S_DO = T::TILE, S_L = 2 * T::TILE, S_D = 2 * T::TILE + 512;
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 256 + D, TM_COLS = 512;
};

enum : int {
  K_KVFULL = 0,
  K_SFULL = 1,    // S^T computed (MMA commit)
  K_DPFULL = 2,   // dP^T computed (MMA commit)
  K_PREADY = 3,   // P^T written (all element-wise threads)
  K_DSREADY = 4,  // dS^T written (all element-wise threads)
  K_DONE = 5,
  K_DRAIN = 6,
  K_QFULL = 7,    // + stage: Q_i, LSE2_i, D_i landed
  K_EMPTY = 11,   // + stage
  K_DOFULL = 15,  // + stage: dO_i landed (apart from Q_i: S^T(t+1), issued before dP^T(t+1),
                  //   needs only Q_i, so the stage's dO copy is not on that product's path)
  K_COUNT = 19
};

// The dK/dV CTA for work unit `block` (its body; the kernels below launch it).  `a` is
// the kernel's __grid_constant__ parameter, so the tensor maps stay in parameter space.
template <int D, bool BF16, bool DROP, bool VARLEN>
__device__ __forceinline__ void dkdv_body(const BwdArgs& a, int block) {
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
  const int n_tk = (a.Nk + kTileN - 1) / kTileN;  // key tiles (of the longest sequence)
  const WorkItem wi = work_item(block, a.BH, n_tk);
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
      return;
    }
  }
  const int n_t = (N + kTileM - 1) / kTileM;  // query tiles
  // Query tiles wholly before the key tile's first key (query i sees key j iff
  // j <= i + cofs) are masked out.
  const int i_begin = a.causal ? max(0, k0 - cofs) / kTileM : 0;
  const int n_iter = n_t - i_begin;

  if (threadIdx.x == 0) {
    mbar_init(bar(K_KVFULL), 1);
    mbar_init(bar(K_SFULL), 1);
    mbar_init(bar(K_DPFULL), 1);
    mbar_init(bar(K_PREADY), 128 * kEw);
    mbar_init(bar(K_DSREADY), 128 * kEw);
    mbar_init(bar(K_DONE), 1);
    mbar_init(bar(K_DRAIN), 1);
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(bar(K_QFULL + s), 1);
      mbar_init(bar(K_EMPTY + s), 1);
      mbar_init(bar(K_DOFULL + s), 1);
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
        tma_load_3d(sb + L::OFF_K + kb * T::BLK, &a.tm_k, bar(K_KVFULL), kb * 64, VARLEN ? hh : k0,
                    VARLEN ? tk0 + k0 : bh);
        tma_load_3d(sb + L::OFF_V + kb * T::BLK, &a.tm_v, bar(K_KVFULL), kb * 64, VARLEN ? hh : k0,
                    VARLEN ? tk0 + k0 : bh);
      }
      int issued = 0;
      for (int t = 0; t < n_iter; ++t) {
        const int s = t % L::STAGES;
        const int q0 = (i_begin + t) * kTileM;
        if (t >= L::STAGES && !mbar_wait(bar(K_EMPTY + s), ((t / L::STAGES) - 1) & 1, wc)) break;
        const uint32_t st = stage_base(s);
        mbar_arrive_expect_tx(bar(K_QFULL + s), T::TILE + 1024);
        mbar_arrive_expect_tx(bar(K_DOFULL + s), T::TILE);
        for (int kb = 0; kb < T::KB; ++kb)
          tma_load_3d(st + L::S_Q + kb * T::BLK, &a.tm_q, bar(K_QFULL + s), kb * 64, VARLEN ? hh : q0,
                      VARLEN ? tq0 + q0 : bh);
        const size_t w = static_cast<size_t>(bh) * a.Npad + q0;
        bulk_load(st + L::S_L, a.lse2 + w, 512, bar(K_QFULL + s));
        bulk_load(st + L::S_D, a.delta + w, 512, bar(K_QFULL + s));
        for (int kb = 0; kb < T::KB; ++kb)
          tma_load_3d(st + L::S_DO + kb * T::BLK, &a.tm_do, bar(K_DOFULL + s), kb * 64, VARLEN ? hh : q0,
                      VARLEN ? tq0 + q0 : bh);
        issued = t + 1;
      }
      mbar_wait(bar(K_KVFULL), 0, wc);
      for (int t = (issued > L::STAGES ? issued - L::STAGES : 0); t < issued; ++t) {
        mbar_wait(bar(K_QFULL + t % L::STAGES), (t / L::STAGES) & 1, wc);
        mbar_wait(bar(K_DOFULL + t % L::STAGES), (t / L::STAGES) & 1, wc);
      }
    }
  } else if (warp == 1) {
    // The whole warp runs the issuing loop; one elected lane issues each product.
    constexpr uint32_t idesc_s = idesc_f16(kTileM, kTileM, BF16, false, false);  // K-major x K-major
    constexpr uint32_t idesc_g = idesc_f16(kTileM, D, BF16, false, true);        // TMEM x MN-major
    // S^T of the next query tile goes between dV and dK: S^T(t+1) overwrites P^T(t),
    // which dV(t) (issued before it) reads, and the element-wise warps keep P(t) in
    // registers for dS^T(t).  So the P^T work of a tile overlaps dK(t-1) and dP^T(t),
    // and the dS^T work overlaps dV(t) and S^T(t+1): two products each instead of one.
    auto issue_st = [&](int t) {
      const uint32_t st = stage_base(t % L::STAGES);
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * T::BLK + (k & 3) * 32;
        mma_ss_w(tmem + L::TM_S, sdesc_sw128(sb + L::OFF_K + off, 16, 1024), sdesc_sw128(st + L::S_Q + off, 16, 1024),
                 idesc_s, k > 0 ? 1u : 0u);
      }
      tc_commit_w(bar(K_SFULL));
    };
    bool ok = mbar_wait_warp(bar(K_KVFULL), 0, wc);
    if (ok && n_iter > 0 && (ok = mbar_wait_warp(bar(K_QFULL + 0), 0, wc))) {
      tc_fence_after();
      issue_st(0);
    }
    for (int t = 0; ok && t < n_iter; ++t) {
      const int s = t % L::STAGES;
      const uint32_t st = stage_base(s);
      if (!(ok = mbar_wait_warp(bar(K_DOFULL + s), (t / L::STAGES) & 1, wc))) break;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * T::BLK + (k & 3) * 32;
        mma_ss_w(tmem + L::TM_DP, sdesc_sw128(sb + L::OFF_V + off, 16, 1024),
                 sdesc_sw128(st + L::S_DO + off, 16, 1024), idesc_s, k > 0 ? 1u : 0u);
      }
      tc_commit_w(bar(K_DPFULL));
      if (!(ok = mbar_wait_warp(bar(K_PREADY), t & 1, wc))) break;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < kTileM / 16; ++k)  // 16-query steps; P^T of warpgroup w at S^T + 32w
        mma_ts_w(tmem + L::TM_DV, tmem + L::TM_S + kEwCols * (k >> 1) + 8 * (k & 1),
                 sdesc_sw128(st + L::S_DO + k * 2048, T::BLK, 1024), idesc_g, (t > 0 || k > 0) ? 1u : 0u);
      if (t + 1 < n_iter) {
        if (!(ok = mbar_wait_warp(bar(K_QFULL + (t + 1) % L::STAGES), ((t + 1) / L::STAGES) & 1, wc))) break;
        tc_fence_after();
        issue_st(t + 1);
      }
      if (!(ok = mbar_wait_warp(bar(K_DSREADY), t & 1, wc))) break;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < kTileM / 16; ++k)
        mma_ts_w(tmem + L::TM_DK, tmem + L::TM_DP + kEwCols * (k >> 1) + 8 * (k & 1),
                 sdesc_sw128(st + L::S_Q + k * 2048, T::BLK, 1024), idesc_g, (t > 0 || k > 0) ? 1u : 0u);
      tc_commit_w(bar(K_EMPTY + s));
    }
    if (ok) tc_commit_w(bar(K_DONE));
    tc_commit_w(bar(K_DRAIN));
    mbar_wait_warp(bar(K_DRAIN), 0, wc);
  } else if (warp >= 4) {
    const int h = (warp >> 2) - 1;      // this warpgroup's 32 query columns of every tile
    const int wq = warp & 3;
    const int row = wq * 32 + lane;     // key row within the tile == TMEM lane
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t t_s = t_lane + L::TM_S + kEwCols * h, t_dp = t_lane + L::TM_DP + kEwCols * h;
    const float sl2 = a.scale_log2;
    // dropout: this warp's 32 x 32 block of keep bytes goes through 1 KB of shared memory
    // (written by query, read by key) so that each thread gets its key's 32 queries
    uint8_t* dbuf = smem + L::OFF_DROP + (warp - 4) * 1024;
    bool ok = true;
    for (int t = 0; t < n_iter; ++t) {
      const int s = t % L::STAGES;
      const int qt = i_begin + t;
      uint32_t keepbits = 0xffffffffu;  // bit c: query column c keeps this key
      if constexpr (DROP) {
        // Lane L takes query qt*128 + 32h + L's decisions for keys k0 + 32wq .. +31.
        const uint32_t qi = static_cast<uint32_t>(qt * kTileM + kEwCols * h + lane);
        if (!VARLEN && a.keep_bits != nullptr) {
          // the forward's stored decisions (one 32-key word per row), transposed so that
          // each thread holds its key's 32 queries
          keepbits = warp_transpose32(a.keep_bits[(static_cast<size_t>(bh) * n_tk + kt) * 4 * a.bits_rows +
                                                  static_cast<size_t>(wq) * a.bits_rows + qi]);
        } else {
          // drawn: lane L's keep bytes go through 1 KB of shared memory (written by query,
          // read by key)
          const uint32_t jg = static_cast<uint32_t>((k0 + 32 * wq) / 16);
          uint32_t w0[4], w1[4];
          philox4x32_10(jg, qi, static_cast<uint32_t>(bh), 0u, a.seed_lo, a.seed_hi, w0);
          philox4x32_10(jg + 1, qi, static_cast<uint32_t>(bh), 0u, a.seed_lo, a.seed_hi, w1);
          uint4* dst = reinterpret_cast<uint4*>(dbuf + lane * 32);
          dst[0] = make_uint4(w0[0], w0[1], w0[2], w0[3]);
          dst[1] = make_uint4(w1[0], w1[1], w1[2], w1[3]);
          __syncwarp();
          keepbits = 0;
#pragma unroll
          for (int c = 0; c < kEwCols; ++c) keepbits |= (dbuf[c * 32 + lane] >= a.drop_t ? 1u : 0u) << c;
          __syncwarp();  // the buffer is rewritten for the next tile
        }
      }
      if (!(ok = mbar_wait_warp(bar(K_QFULL + s), (t / L::STAGES) & 1, wc))) break;
      if (!(ok = mbar_wait_warp(bar(K_SFULL), t & 1, wc))) break;
      tc_fence_after();
      const float4* l4 =
          reinterpret_cast<const float4*>(smem + L::OFF_ST + s * L::STAGE_BYTES + L::S_L) + (kEwCols / 4) * h;
      const float4* d4 =
          reinterpret_cast<const float4*>(smem + L::OFF_ST + s * L::STAGE_BYTES + L::S_D) + (kEwCols / 4) * h;
      // causal: query column c (query qt*128 + 32h + c) sees key k0 + row only if
      // qt*128 + 32h + c + cofs >= k0 + row
      const int first_visible = a.causal ? k0 + row - cofs - qt * kTileM - kEwCols * h : 0;
      float p[kEwCols];
      // Phase 1: P^T for this warpgroup's queries (overlaps the dP^T product).
      {
        // p = 2^(s sl2 - lse2) as 2^-(lse2 - s sl2): one paired fma per two columns, and
        // bit-identical to the scalar form (round-to-nearest is symmetric under negation).
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
      mbar_arrive(bar(K_PREADY));
      // Phase 2: dS^T = P^T (dP^T - D) (overlaps the dV product).
      if (!(ok = mbar_wait_warp(bar(K_DPFULL), t & 1, wc))) break;
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
        for (int v = 0; v < kEwCols / 4; ++v) {  // paired sub and mul, two columns each
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
      mbar_arrive(bar(K_DSREADY));
    }
    if (ok) ok = mbar_wait_warp(bar(K_DONE), 0, wc);
    // Epilogue: warpgroups 0-1 write dV, 2-3 write scale * dK (each half of the d
    // columns), through swizzled staging tiles over the stage-0 dO / Q buffers
    // (every product is done).
    const int which = h >> 1;  // 0: dV, 1: dK
    uint8_t* stage = smem + L::OFF_ST + (which == 0 ? L::S_DO : L::S_Q);
    if (ok) {
      tc_fence_after();
      const uint32_t col = (which == 0) ? L::TM_DV : L::TM_DK;
      const float mul = (which == 0) ? 1.f : a.scale;
#pragma unroll
      for (int cc = (h & 1) * (D / 64); cc < ((h & 1) + 1) * (D / 64); ++cc) {
        uint32_t v[32];
        tmem_ld_x32(t_lane + col + cc * 32, v);
        if constexpr (VARLEN) {  // rows of this sequence only, straight to global memory
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

// ------------------------------------------------------------------ bwd_dq
//
// Same warp roles; element-wise warpgroup w handles keys 32w..32w+31 of every
// key tile.  Q and dO sit in tensor memory for the whole loop (copied there once),
// dS goes over the first half of each warpgroup's dP columns, and S has its own
// columns, so the MMA warp issues the next tile's S as soon as the element-wise
// warps have read this one:
//   S(j) | dP(j) | S(j+1) | dQ += dS(j) K_j | dP(j+1) | S(j+2) | ...
// P = ex2(c S - LSE2) is computed while dP runs, dS = P (dP - D) while the next S
// runs; dP(j+1) comes after dQ(j), which reads dS(j) from dP(j)'s columns.
//
// K and V stream through separate rings: K(j) is read by S(j) and dQ(j), V(j) only by
// dP(j), and S(j+1) is issued about when dQ(j-1) frees K's slot.  With one shared
// two-slot ring every S waited a whole load; three K slots give each K load an
// iteration of slack, and V's two slots free at dP(j), well ahead of dP(j+2).

template <int D>
struct DqLayout {
  using T = BwdTiles<D>;
  static constexpr int KST = (D == 128) ? 3 : 4;  // K ring slots
  static constexpr int VST = (D == 128) ? 2 : 4;  // V ring slots
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = T::TILE;
  static constexpr int OFF_K = 2 * T::TILE;
  static constexpr int OFF_V = OFF_K + KST * T::TILE;
  static constexpr int OFF_BAR = OFF_V + VST * T::TILE;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  // Q and dO are copied into tensor memory once (16-bit pairs) and feed S = Q K^T and
  // dP = dO V^T from there, so those products read only K or V from shared memory: with
  // both operands in shared memory a 128 x 128 x 16 product reads 8 KB, 64 cycles of the
  // SM's 128 B/cycle, and the kernel was bound by shared-memory bandwidth.  dS goes over
  // the first half of each warpgroup's own dP columns.
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DQ = 256, TM_Q = 384, TM_DO = 384 + D / 2, TM_COLS = 512;
};

enum : int {
  Q_QFULL = 0,
  Q_SFULL = 1,    // S computed (MMA commit)
  Q_DPFULL = 2,   // dP computed (MMA commit)
  Q_SCONS = 3,    // S read by every element-wise thread
  Q_DSREADY = 4,  // dS written by every element-wise thread
  Q_DONE = 5,
  Q_DRAIN = 6,
  Q_KFULL = 7,    // + K slot
  Q_KEMPTY = 11,  // + K slot
  Q_VFULL = 15,   // + V slot
  Q_VEMPTY = 19,  // + V slot
  Q_QTM = 23,     // Q and dO copied into tensor memory (all element-wise threads)
  Q_COUNT = 24
};

// The dQ CTA for work unit `block` (its body; the kernels below launch it).
template <int D, bool BF16, bool DROP, bool VARLEN>
__device__ __forceinline__ void dq_body(const BwdArgs& a, int block) {
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
  const WorkItem wi = work_item(block, a.BH, n_t);
  const int bh = wi.bh;
  const int qt = n_t - 1 - wi.rank;  // longest causal tiles first
  const int q0 = qt * kTileM;
  int N = a.N, Nk = a.Nk, cofs = a.cofs, hh = 0, tq0 = 0, tk0 = 0;
  if constexpr (VARLEN) {
    const SeqView sv = seq_view(a, bh);
    N = sv.N, Nk = sv.Nk, cofs = sv.cofs, hh = sv.hh, tq0 = sv.tq0, tk0 = sv.tk0;
    if (q0 >= sv.N) return;  // this query tile lies past the sequence's end (whole CTA)
    if (sv.degenerate) {
      zero_rows_packed<D>(a.dq_out, a.H, hh, tq0, q0, sv.N);
      return;
    }
  }
  const int n_kv = visible_key_tiles(qt, Nk, a.causal, cofs);

  if (threadIdx.x == 0) {
    mbar_init(bar(Q_QFULL), 1);
    mbar_init(bar(Q_SFULL), 1);
    mbar_init(bar(Q_DPFULL), 1);
    mbar_init(bar(Q_SCONS), 128 * kEw);
    mbar_init(bar(Q_QTM), 128 * kEw);
    mbar_init(bar(Q_DSREADY), 128 * kEw);
    mbar_init(bar(Q_DONE), 1);
    mbar_init(bar(Q_DRAIN), 1);
    for (int s = 0; s < L::KST; ++s) {
      mbar_init(bar(Q_KFULL + s), 1);
      mbar_init(bar(Q_KEMPTY + s), 1);
    }
    for (int s = 0; s < L::VST; ++s) {
      mbar_init(bar(Q_VFULL + s), 1);
      mbar_init(bar(Q_VEMPTY + s), 1);
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
        tma_load_3d(sb + L::OFF_Q + kb * T::BLK, &a.tm_q, bar(Q_QFULL), kb * 64, VARLEN ? hh : q0,
                    VARLEN ? tq0 + q0 : bh);
        tma_load_3d(sb + L::OFF_DO + kb * T::BLK, &a.tm_do, bar(Q_QFULL), kb * 64, VARLEN ? hh : q0,
                    VARLEN ? tq0 + q0 : bh);
      }
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        // K(j) waits for dQ(j - KST) to free its slot, V(j) for dP(j - VST); in the
        // tensor core's order dQ(j - 3) precedes dP(j - 2), so neither wait holds up a
        // load the other could have started.
        const int ks = j % L::KST;
        if (j >= L::KST && !mbar_wait(bar(Q_KEMPTY + ks), ((j / L::KST) - 1) & 1, wc)) break;
        mbar_arrive_expect_tx(bar(Q_KFULL + ks), T::TILE);
        for (int kb = 0; kb < T::KB; ++kb)
          tma_load_3d(sb + L::OFF_K + ks * T::TILE + kb * T::BLK, &a.tm_k, bar(Q_KFULL + ks), kb * 64,
                      VARLEN ? hh : j * kTileN, VARLEN ? tk0 + j * kTileN : bh);
        k_issued = j + 1;
        const int vs = j % L::VST;
        if (j >= L::VST && !mbar_wait(bar(Q_VEMPTY + vs), ((j / L::VST) - 1) & 1, wc)) break;
        mbar_arrive_expect_tx(bar(Q_VFULL + vs), T::TILE);
        for (int kb = 0; kb < T::KB; ++kb)
          tma_load_3d(sb + L::OFF_V + vs * T::TILE + kb * T::BLK, &a.tm_v, bar(Q_VFULL + vs), kb * 64,
                      VARLEN ? hh : j * kTileN, VARLEN ? tk0 + j * kTileN : bh);
        v_issued = j + 1;
      }
      mbar_wait(bar(Q_QFULL), 0, wc);
      for (int j = (k_issued > L::KST ? k_issued - L::KST : 0); j < k_issued; ++j)
        mbar_wait(bar(Q_KFULL + j % L::KST), (j / L::KST) & 1, wc);
      for (int j = (v_issued > L::VST ? v_issued - L::VST : 0); j < v_issued; ++j)
        mbar_wait(bar(Q_VFULL + j % L::VST), (j / L::VST) & 1, wc);
    }
  } else if (warp == 1) {
    // The whole warp runs the issuing loop; one elected lane issues each product.
    constexpr uint32_t idesc_s = idesc_f16(kTileM, kTileN, BF16, false, false);
    constexpr uint32_t idesc_g = idesc_f16(kTileM, D, BF16, false, true);
    auto k_full = [&](int j) { return mbar_wait_warp(bar(Q_KFULL + j % L::KST), (j / L::KST) & 1, wc); };
    auto v_full = [&](int j) { return mbar_wait_warp(bar(Q_VFULL + j % L::VST), (j / L::VST) & 1, wc); };
    auto issue_s = [&](int j) {  // S = Q K^T, Q from tensor memory (16 elements = 8 columns per step)
      const uint32_t kbase = sb + L::OFF_K + (j % L::KST) * T::TILE;
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * T::BLK + (k & 3) * 32;
        mma_ts_w(tmem + L::TM_S, tmem + L::TM_Q + 8 * k, sdesc_sw128(kbase + off, 16, 1024), idesc_s, k > 0 ? 1u : 0u);
      }
      tc_commit_w(bar(Q_SFULL));
    };
    auto issue_dp = [&](int j) {  // dP = dO V^T, dO from tensor memory
      const uint32_t vbase = sb + L::OFF_V + (j % L::VST) * T::TILE;
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * T::BLK + (k & 3) * 32;
        mma_ts_w(tmem + L::TM_DP, tmem + L::TM_DO + 8 * k, sdesc_sw128(vbase + off, 16, 1024), idesc_s,
                 k > 0 ? 1u : 0u);
      }
      tc_commit_w(bar(Q_DPFULL));
      tc_commit_w(bar(Q_VEMPTY + j % L::VST));
    };
    bool ok = mbar_wait_warp(bar(Q_QTM), 0, wc) && k_full(0);
    if (ok) {
      tc_fence_after();
      issue_s(0);
      ok = v_full(0);
    }
    if (ok) {
      tc_fence_after();
      issue_dp(0);
    }
    for (int j = 0; ok && j < n_kv; ++j) {
      if (j + 1 < n_kv) {
        // The next S may overwrite S(j) once both warpgroups have read it.
        if (!(ok = k_full(j + 1) && mbar_wait_warp(bar(Q_SCONS), j & 1, wc))) break;
        tc_fence_after();
        issue_s(j + 1);
      }
      if (!(ok = mbar_wait_warp(bar(Q_DSREADY), j & 1, wc))) break;
      tc_fence_after();
      const uint32_t kbase = sb + L::OFF_K + (j % L::KST) * T::TILE;
#pragma unroll
      for (int k = 0; k < kTileN / 16; ++k)  // 16-key steps; dS of warpgroup w's keys at dP + 32w
        mma_ts_w(tmem + L::TM_DQ, tmem + L::TM_DP + kEwCols * (k >> 1) + 8 * (k & 1),
                 sdesc_sw128(kbase + k * 2048, T::BLK, 1024), idesc_g, (j > 0 || k > 0) ? 1u : 0u);
      tc_commit_w(bar(Q_KEMPTY + j % L::KST));
      if (j + 1 < n_kv) {  // dP(j) was read before dS(j) was published
        if (!(ok = v_full(j + 1))) break;
        tc_fence_after();
        issue_dp(j + 1);
      }
    }
    if (ok) tc_commit_w(bar(Q_DONE));
    tc_commit_w(bar(Q_DRAIN));
    mbar_wait_warp(bar(Q_DRAIN), 0, wc);
  } else if (warp >= 4) {
    const int h = (warp >> 2) - 1;  // this warpgroup's 32 key columns of every tile
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const int grow = q0 + row;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float sl2 = a.scale_log2;
    const size_t w = static_cast<size_t>(bh) * a.Npad + grow;  // grow < Npad always
    const float lse2 = a.lse2[w];
    const float dlt = a.delta[w];
    bool ok = mbar_wait_warp(bar(Q_QFULL), 0, wc);
    if (ok) {
      // Copy this row's D/4 columns of Q and of dO (warpgroup h's share) from the
      // 128-byte-swizzled shared tiles into tensor memory.
      constexpr int CPW = D / kEw;  // columns per warpgroup: 32 (d = 128) or 16 (d = 64)
      const int c0 = CPW * h;
      const int kb = c0 / 64, ch0 = (c0 % 64) / 8;
      uint32_t qv[CPW / 2], ov[CPW / 2];
#pragma unroll
      for (int q = 0; q < CPW / 8; ++q) {
        const int off = kb * T::BLK + row * 128 + (((ch0 + q) ^ (row & 7)) << 4);
        const uint4 a4 = *reinterpret_cast<const uint4*>(smem + L::OFF_Q + off);
        const uint4 b4 = *reinterpret_cast<const uint4*>(smem + L::OFF_DO + off);
        qv[4 * q] = a4.x, qv[4 * q + 1] = a4.y, qv[4 * q + 2] = a4.z, qv[4 * q + 3] = a4.w;
        ov[4 * q] = b4.x, ov[4 * q + 1] = b4.y, ov[4 * q + 2] = b4.z, ov[4 * q + 3] = b4.w;
      }
      if constexpr (CPW == 32) {
        tmem_st_x16(t_lane + L::TM_Q + CPW / 2 * h, qv);
        tmem_st_x16(t_lane + L::TM_DO + CPW / 2 * h, ov);
      } else {
        tmem_st_x8(t_lane + L::TM_Q + CPW / 2 * h, qv);
        tmem_st_x8(t_lane + L::TM_DO + CPW / 2 * h, ov);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(Q_QTM));
    }
    for (int j = 0; ok && j < n_kv; ++j) {
      uint32_t keepw[8];  // dropout: bit 0 of byte (c % 4) of word c / 4 set if key column c is kept
      if constexpr (DROP) {
        if (!VARLEN && a.keep_bits != nullptr) {
          // the forward's stored word for this row and the warpgroup's 32 keys, one bit
          // per key spread to one byte per key
          const size_t n_tk = (a.Nk + kTileN - 1) / kTileN;
          const uint32_t bits = a.keep_bits[(static_cast<size_t>(bh) * n_tk + j) * 4 * a.bits_rows +
                                            static_cast<size_t>(h) * a.bits_rows + grow];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t x = (bits >> (4 * q)) & 0xFu;
            keepw[q] = (x & 1u) | ((x & 2u) << 7) | ((x & 4u) << 14) | ((x & 8u) << 21);
          }
        } else {
          const uint32_t jg = static_cast<uint32_t>((j * kTileN + kEwCols * h) / 16);
          uint32_t w[4];
          const uint32_t tt = a.drop_t * 0x01010101u;
          philox4x32_10(jg, static_cast<uint32_t>(grow), static_cast<uint32_t>(bh), 0u, a.seed_lo, a.seed_hi, w);
#pragma unroll
          for (int q = 0; q < 4; ++q) keepw[q] = __vcmpgeu4(w[q], tt);
          philox4x32_10(jg + 1, static_cast<uint32_t>(grow), static_cast<uint32_t>(bh), 0u, a.seed_lo, a.seed_hi, w);
#pragma unroll
          for (int q = 0; q < 4; ++q) keepw[4 + q] = __vcmpgeu4(w[q], tt);
        }
      }
      if (!(ok = mbar_wait_warp(bar(Q_SFULL), j & 1, wc))) break;
      tc_fence_after();
      const int kbeg = j * kTileN + kEwCols * h;
      int lim = Nk - kbeg;                                   // keys past the end
      if (a.causal) lim = min(lim, grow + cofs - kbeg + 1);  // keys after this query
      float p[kEwCols];
      {
        uint32_t sv[kEwCols];
        tmem_ld_x32(t_lane + L::TM_S + kEwCols * h, sv);
        tc_fence_before();
        mbar_arrive(bar(Q_SCONS));
        const uint64_t sl2x2 = f32x2_pack(sl2, sl2), nl2 = f32x2_pack(-lse2, -lse2);
#pragma unroll
        for (int e = 0; e < kEwCols; e += 2) {  // one paired fma per two columns
          float x0, x1;
          f32x2_unpack(f32x2_fma(f32x2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sl2x2, nl2), x0, x1);
          p[e] = ex2(x0);
          p[e + 1] = ex2(x1);
        }
      }
      if (lim < kEwCols) {
#pragma unroll
        for (int c = 0; c < kEwCols; ++c)
          if (c >= lim) p[c] = 0.f;
      }
      if (!(ok = mbar_wait_warp(bar(Q_DPFULL), j & 1, wc))) break;
      tc_fence_after();
      {
        uint32_t dv[kEwCols], dsp[kEwCols / 2];
        tmem_ld_x32(t_lane + L::TM_DP + kEwCols * h, dv);
        if constexpr (DROP) {  // dP <- Z o dP
          const float zs = a.drop_scale;
#pragma unroll
          for (int e = 0; e < kEwCols; ++e)
            dv[e] = __float_as_uint(((keepw[e / 4] >> (8 * (e % 4))) & 1u) ? __uint_as_float(dv[e]) * zs : 0.f);
        }
        const uint64_t dlt2 = f32x2_pack(dlt, dlt);
#pragma unroll
        for (int e = 0; e < kEwCols; e += 2) {  // paired sub and mul
          float a0, a1;
          f32x2_unpack(f32x2_mul(f32x2_pack(p[e], p[e + 1]),
                                 f32x2_sub(f32x2_pack(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])), dlt2)),
                       a0, a1);
          dsp[e / 2] = pack2<BF16>(a0, a1);
        }
        // dS goes over the first half of this warpgroup's dP columns, which this thread
        // has read; dP(j+1) is issued after dQ(j), the product that reads dS(j).
        tmem_st_x16(t_lane + L::TM_DP + kEwCols * h, dsp);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(Q_DSREADY));
    }
    if (ok) ok = mbar_wait_warp(bar(Q_DONE), 0, wc);
    if (ok) {
      tc_fence_after();
      uint8_t* stage = smem + L::OFF_Q;  // Q is no longer read once every product is done
#pragma unroll
      for (int c32 = h; c32 < D / 32; c32 += kEw) {  // this warpgroup's 32-column chunks
        uint32_t v[32];
        tmem_ld_x32(t_lane + L::TM_DQ + c32 * 32, v);
        if constexpr (VARLEN) {  // rows of this sequence only, straight to global memory
          if (grow < N)
            store_row_chunk_packed<D, BF16>(a.dq_out, (static_cast<size_t>(tq0 + grow) * a.H + hh) * D, c32, v,
                                            a.scale);
        } else {
          stage_row_chunk<D, BF16>(stage, row, c32, v, a.scale);
        }
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128 * kEw);
    if (!VARLEN && warp == 4 && lane == 0 && ok && !*abort_flag) {
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

template <int D, bool BF16, bool DROP, bool VARLEN>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_dkdv_kernel(const __grid_constant__ BwdArgs a) {
  dkdv_body<D, BF16, DROP, VARLEN>(a, static_cast<int>(blockIdx.x));
}

template <int D, bool BF16, bool DROP, bool VARLEN>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdArgs a) {
  dq_body<D, BF16, DROP, VARLEN>(a, static_cast<int>(blockIdx.x));
}

// Both gradient stages in one grid: the first n_dkdv CTAs are dK/dV units, the rest dQ
// units.  The two stages are independent once the preparation pass has run, and the
// block scheduler starts the dQ CTAs as the dK/dV CTAs retire, so the end of one stage
// overlaps the start of the other instead of draining the GPU between two launches.
template <int D, bool BF16, bool DROP>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_grads_kernel(const __grid_constant__ BwdArgs a, int n_dkdv) {
  const int b = static_cast<int>(blockIdx.x);
  if (b < n_dkdv)
    dkdv_body<D, BF16, DROP, false>(a, b);
  else
    dq_body<D, BF16, DROP, false>(a, b - n_dkdv);
}

template <int D, bool BF16, bool VARLEN = false>
cudaError_t launch_pre_t(const BwdArgs& a, cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(a.BH) * a.Npad;
  const int64_t rows_per_block = (256 / 32) * kPreUnroll * (32 / (D / 8));
  const int64_t blocks = (rows + rows_per_block - 1) / rows_per_block;
  bwd_pre_kernel<D, BF16, VARLEN><<<static_cast<unsigned>(blocks), 256, 0, st>>>(a);
  return cudaGetLastError();
}

template <int D, bool BF16, bool DROP = false, bool VARLEN = false>
cudaError_t launch_dkdv_t(const BwdArgs& a, cudaStream_t st) {
  auto k = bwd_dkdv_kernel<D, BF16, DROP, VARLEN>;
  constexpr int smem = DkdvLayout<D>::SMEM + (DROP ? DkdvLayout<D>::DROP_BYTES : 0);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int n_tk = (a.Nk + kTileN - 1) / kTileN;
  k<<<n_tk * a.BH, kBwdThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <int D, bool BF16, bool DROP = false, bool VARLEN = false>
cudaError_t launch_dq_t(const BwdArgs& a, cudaStream_t st) {
  auto k = bwd_dq_kernel<D, BF16, DROP, VARLEN>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, DqLayout<D>::SMEM);
  if (e != cudaSuccess) return e;
  const int n_t = (a.N + kTileM - 1) / kTileM;
  k<<<n_t * a.BH, kBwdThreads, DqLayout<D>::SMEM, st>>>(a);
  return cudaGetLastError();
}

template <int D, bool BF16, bool DROP = false>
cudaError_t launch_grads_t(const BwdArgs& a, cudaStream_t st) {
  auto k = bwd_grads_kernel<D, BF16, DROP>;
  constexpr int smem_kv = DkdvLayout<D>::SMEM + (DROP ? DkdvLayout<D>::DROP_BYTES : 0);
  constexpr int smem = smem_kv > DqLayout<D>::SMEM ? smem_kv : DqLayout<D>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int n_dkdv = (a.Nk + kTileN - 1) / kTileN * a.BH;
  const int n_dq = (a.N + kTileM - 1) / kTileM * a.BH;
  k<<<n_dkdv + n_dq, kBwdThreads, smem, st>>>(a, n_dkdv);
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

cudaError_t launch_bwd_pre(const BwdArgs& a, int d, bool bf16, cudaStream_t s) {
  if (d == 256) return bf16 ? launch_pre_t<256, true>(a, s) : launch_pre_t<256, false>(a, s);
  ATTN_DISPATCH(launch_pre_t)
}
cudaError_t launch_bwd_dkdv(const BwdArgs& a, int d, bool bf16, cudaStream_t s) { ATTN_DISPATCH(launch_dkdv_t) }
cudaError_t launch_bwd_dq(const BwdArgs& a, int d, bool bf16, cudaStream_t s) { ATTN_DISPATCH(launch_dq_t) }
cudaError_t launch_bwd_grads(const BwdArgs& a, int d, bool bf16, cudaStream_t s) { ATTN_DISPATCH(launch_grads_t) }
#undef ATTN_DISPATCH

#define ATTN_DISPATCH_DROP(fn)                                                          \
  if (d == 128) return bf16 ? fn<128, true, true>(a, s) : fn<128, false, true>(a, s); \
  return bf16 ? fn<64, true, true>(a, s) : fn<64, false, true>(a, s);

cudaError_t launch_bwd_dkdv_dropout(const BwdArgs& a, int d, bool bf16, cudaStream_t s) {
  ATTN_DISPATCH_DROP(launch_dkdv_t)
}
cudaError_t launch_bwd_dq_dropout(const BwdArgs& a, int d, bool bf16, cudaStream_t s) {
  ATTN_DISPATCH_DROP(launch_dq_t)
}
cudaError_t launch_bwd_grads_dropout(const BwdArgs& a, int d, bool bf16, cudaStream_t s) {
  ATTN_DISPATCH_DROP(launch_grads_t)
}
#undef ATTN_DISPATCH_DROP

cudaError_t launch_bwd_pre_varlen(const BwdArgs& a, int d, bool bf16, cudaStream_t s) {
  if (d == 256) return bf16 ? launch_pre_t<256, true, true>(a, s) : launch_pre_t<256, false, true>(a, s);
  if (d == 128) return bf16 ? launch_pre_t<128, true, true>(a, s) : launch_pre_t<128, false, true>(a, s);
  return bf16 ? launch_pre_t<64, true, true>(a, s) : launch_pre_t<64, false, true>(a, s);
}
// The varlen gradient launchers: a.drop_t > 0 selects the dropout kernels.
cudaError_t launch_bwd_dkdv_varlen(const BwdArgs& a, int d, bool bf16, cudaStream_t s) {
  if (a.drop_t > 0) {
    if (d == 128) return bf16 ? launch_dkdv_t<128, true, true, true>(a, s) : launch_dkdv_t<128, false, true, true>(a, s);
    return bf16 ? launch_dkdv_t<64, true, true, true>(a, s) : launch_dkdv_t<64, false, true, true>(a, s);
  }
  if (d == 128) return bf16 ? launch_dkdv_t<128, true, false, true>(a, s) : launch_dkdv_t<128, false, false, true>(a, s);
  return bf16 ? launch_dkdv_t<64, true, false, true>(a, s) : launch_dkdv_t<64, false, false, true>(a, s);
}
cudaError_t launch_bwd_dq_varlen(const BwdArgs& a, int d, bool bf16, cudaStream_t s) {
  if (a.drop_t > 0) {
    if (d == 128) return bf16 ? launch_dq_t<128, true, true, true>(a, s) : launch_dq_t<128, false, true, true>(a, s);
    return bf16 ? launch_dq_t<64, true, true, true>(a, s) : launch_dq_t<64, false, true, true>(a, s);
  }
  if (d == 128) return bf16 ? launch_dq_t<128, true, false, true>(a, s) : launch_dq_t<128, false, false, true>(a, s);
  return bf16 ? launch_dq_t<64, true, false, true>(a, s) : launch_dq_t<64, false, false, true>(a, s);
}

cudaError_t launch_wait_selftest(int* dev_status, uint64_t limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(dev_status, limit_ns);
  return cudaGetLastError();
}

}  // namespace attn
