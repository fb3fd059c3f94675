// fwd.cu -- forward attention kernel for sm_103a.
//
// One CTA computes one 128-row query tile of one (batch, head) and streams the
// K/V tiles of that head through shared memory (FA2 loop order: queries outer,
// keys inner; "FlashAttention hardware-aware analysis" (huaweicloud), section
// four, part 2).  Per key tile j:
//
//   S_j   = Q K_j^T                 tcgen05.mma, SMEM x SMEM -> TMEM (fp32)
//   m_new = max(m, rowmax S_j)      online-softmax recurrence (huaweicloud page,
//   P_j   = exp(S_j - m_new)        section two; "Understanding online softmax in
//   l     = l e^(m-m_new) + rowsum  Flash Attention from scratch", section 3.1),
//   O     = O e^(m-m_new) + P_j V_j in the base-2 domain: exponents are
//                                   scale*log2(e)*S, so exp becomes ex2
//
// O stays in tensor memory for the whole loop and is divided by l once at the
// end (deferred normalisation; hotelren.com FA1/FA2 comparison, section 2.1.2).
// The row logsumexp m + ln l is saved for the backward pass.  Nothing of size
// N x N ever leaves the SM.
//
// Warp roles (192 threads):
//   warp 0     TMA producer: Q once, then K_j and V_j into a STAGES-deep ring
//   warp 1     TMEM owner and MMA issuer (one elected lane)
//   warps 2-5  softmax: thread r owns query row r (TMEM lane r): masks, row max,
//              ex2, row sum, P -> TMEM (16-bit), O rescale, epilogue
//
// Tensor memory (512 columns): S at 0..127 (fp32), P at 128..191 (16-bit pairs),
// O at 256..256+d-1 (fp32).
//
// Causal: key tiles wholly above the diagonal are never loaded (the huaweicloud
// page's section five, part 3); only the diagonal tile and the ragged last tile
// are masked.  The grid is walked longest-tile-first.
#include "common.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

template <int D>
struct FwdLayout {
  static constexpr int KB = D / 64;                  // 64-column (128-byte) blocks per row
  static constexpr int TILE = kTileM * D * 2;        // bytes of one 128 x D 16-bit tile
  static constexpr int BLK = kTileM * 128;           // bytes of one 128-row x 64-col block
  static constexpr int STAGES = (D == 128) ? 3 : 4;  // K/V ring depth
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE;
  static constexpr int OFF_V = OFF_K + STAGES * TILE;
  static constexpr int OFF_BAR = OFF_V + STAGES * TILE;
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = OFF_BAR + BAR_BYTES + 1024;  // + alignment slack
  static constexpr uint32_t TM_S = 0, TM_P = 128, TM_O = 256, TM_COLS = 512;
};

constexpr int kFwdThreads = 192;

// Barrier slots (uint64 each) after OFF_BAR.
enum : int {
  B_QFULL = 0,
  B_SFULL = 1,
  B_SFREE = 2,
  B_PFULL = 3,
  B_ORDY = 4,
  B_DRAIN = 5,
  B_KFULL = 6,   // + stage
  B_VFULL = 10,  // + stage
  B_EMPTY = 14,  // + stage
  B_COUNT = 18
};

template <int D, bool BF16>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_kernel(const __grid_constant__ FwdArgs a) {
  using L = FwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t sQ = sb + L::OFF_Q;
  const uint32_t sK = sb + L::OFF_K;
  const uint32_t sV = sb + L::OFF_V;
  const uint32_t bars = sb + L::OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 8 * B_COUNT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_BAR + 8 * B_COUNT + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_qt = (a.N + kTileM - 1) / kTileM;
  const int qt = n_qt - 1 - static_cast<int>(blockIdx.x) / a.BH;  // longest causal tiles first
  const int bh = static_cast<int>(blockIdx.x) % a.BH;
  const int q0 = qt * kTileM;
  const int n_kt = (a.N + kTileN - 1) / kTileN;
  const int n_kv = a.causal ? min(qt + 1, n_kt) : n_kt;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_SFREE), 128);
    mbar_init(bar(B_PFULL), 128);
    mbar_init(bar(B_ORDY), 1);
    mbar_init(bar(B_DRAIN), 1);
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_EMPTY + s), 1);
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
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
      prefetch_tmap(&a.tm_o);
      mbar_arrive_expect_tx(bar(B_QFULL), L::TILE);
      for (int kb = 0; kb < L::KB; ++kb) tma_load_3d(sQ + kb * L::BLK, &a.tm_q, bar(B_QFULL), kb * 64, q0, bh);
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % L::STAGES;
        if (j >= L::STAGES && !mbar_wait(bar(B_EMPTY + s), ((j / L::STAGES) - 1) & 1, wc)) break;
        const uint32_t dk = sK + s * L::TILE, dv = sV + s * L::TILE;
        mbar_arrive_expect_tx(bar(B_KFULL + s), L::TILE);
        for (int kb = 0; kb < L::KB; ++kb) tma_load_3d(dk + kb * L::BLK, &a.tm_k, bar(B_KFULL + s), kb * 64, j * kTileN, bh);
        mbar_arrive_expect_tx(bar(B_VFULL + s), L::TILE);
        for (int kb = 0; kb < L::KB; ++kb) tma_load_3d(dv + kb * L::BLK, &a.tm_v, bar(B_VFULL + s), kb * 64, j * kTileN, bh);
        issued = j + 1;
      }
      // Let every copy this thread started land before the CTA can exit.
      mbar_wait(bar(B_QFULL), 0, wc);
      for (int j = (issued > L::STAGES ? issued - L::STAGES : 0); j < issued; ++j) {
        const int s = j % L::STAGES, ph = (j / L::STAGES) & 1;
        mbar_wait(bar(B_KFULL + s), ph, wc);
        mbar_wait(bar(B_VFULL + s), ph, wc);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f16(kTileM, kTileN, BF16, false, false);
      constexpr uint32_t idesc_pv = idesc_f16(kTileM, D, BF16, false, true);
      bool ok = mbar_wait(bar(B_QFULL), 0, wc);
      auto issue_pv = [&](int t) -> bool {
        const int s = t % L::STAGES, ph = (t / L::STAGES) & 1;
        if (!mbar_wait(bar(B_PFULL), t & 1, wc)) return false;
        if (!mbar_wait(bar(B_VFULL + s), ph, wc)) return false;
        tc_fence_after();
        const uint32_t v_base = sV + s * L::TILE;
#pragma unroll
        for (int k = 0; k < kTileN / 16; ++k) {
          // 16 keys = two 8-row groups of 128 bytes; d blocks are L::BLK apart.
          const uint64_t bd = sdesc_sw128(v_base + k * 2048, L::BLK, 1024);
          mma_ts(tmem + L::TM_O, tmem + L::TM_P + k * 8, bd, idesc_pv, (t > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit(bar(B_ORDY));
        tc_commit(bar(B_EMPTY + s));
        return true;
      };
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j % L::STAGES, ph = (j / L::STAGES) & 1;
        if (!mbar_wait(bar(B_KFULL + s), ph, wc)) { ok = false; break; }
        if (j > 0 && !mbar_wait(bar(B_SFREE), (j - 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t k_base = sK + s * L::TILE;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * L::BLK + (k & 3) * 32;
          const uint64_t ad = sdesc_sw128(sQ + off, 16, 1024);
          const uint64_t bd = sdesc_sw128(k_base + off, 16, 1024);
          mma_ss(tmem + L::TM_S, ad, bd, idesc_qk, k > 0 ? 1u : 0u);
        }
        tc_commit(bar(B_SFULL));
        if (j > 0 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok) issue_pv(n_kv - 1);
      // Drain: nothing may still write tensor memory when it is released.
      tc_commit(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0, wc);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int wq = warp & 3;                     // TMEM lane quarter of this warp
    const int row = wq * 32 + lane;              // row in the tile == TMEM lane
    const int grow = q0 + row;                   // row in the sequence
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float sl2 = a.scale_log2;
    float m = -INFINITY;  // running max of scale*log2(e)*S
    float l = 0.f;        // running sum of ex2(.. - m)
    bool ok = true;

    for (int j = 0; j < n_kv; ++j) {
      if (!mbar_wait_warp(bar(B_SFULL), j & 1, wc)) { ok = false; break; }
      tc_fence_after();
      float s[128];
      {
        uint32_t sr[128];
        tmem_ld_x128(t_lane + L::TM_S, sr);
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
      }
      tc_fence_before();
      mbar_arrive(bar(B_SFREE));

      const int k0 = j * kTileN;
      const bool tail = k0 + kTileN > a.N;
      const bool diag = a.causal && (k0 + kTileN - 1 > q0);
      if (tail || diag) {
        int lim = a.N - k0;                       // keys past the end of the sequence
        if (a.causal) lim = min(lim, grow - k0 + 1);  // keys after this query
#pragma unroll
        for (int c = 0; c < kTileN; ++c)
          if (c >= lim) s[c] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < kTileN; ++c) mx = fmaxf(mx, s[c]);
      const float m_new = fmaxf(m, mx * sl2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // a row with nothing visible yet
      const float alpha = ex2(m - m_use);                     // 0 on the first tile
      float rs = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < kTileN; c += 2) {
        const float p0 = ex2(fmaf(s[c], sl2, -m_use));
        const float p1 = ex2(fmaf(s[c + 1], sl2, -m_use));
        rs += p0 + p1;
        pk[c / 2] = pack2<BF16>(p0, p1);
      }
      l = fmaf(l, alpha, rs);
      m = m_new;

      if (j > 0) {
        // O and the P columns are busy until the previous P V product is done.
        if (!mbar_wait_warp(bar(B_ORDY), (j - 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld_x32(t_lane + L::TM_O + cc * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st_x32(t_lane + L::TM_O + cc * 32, o);
          }
        }
      }
      tmem_st_x64(t_lane + L::TM_P, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL));
    }

    // ---------------------------------------------------------- epilogue
    if (ok) ok = mbar_wait_warp(bar(B_ORDY), (n_kv - 1) & 1, wc);
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      uint8_t* stage = smem + L::OFF_Q;  // Q is no longer read once the last S is done
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld_x32(t_lane + L::TM_O + cc * 32, o);
        uint32_t pkd[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pkd[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
        // 32 columns = four 16-byte chunks of the 128B-swizzled row.
        const int kb = (cc * 32) / 64;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int ch = ((cc * 32) % 64) / 8 + q;
          uint4* dst = reinterpret_cast<uint4*>(stage + kb * L::BLK + row * 128 + ((ch ^ (row & 7)) << 4));
          *dst = make_uint4(pkd[4 * q], pkd[4 * q + 1], pkd[4 * q + 2], pkd[4 * q + 3]);
        }
      }
      if (grow < a.N) {
        // natural-log logsumexp of the scaled scores: (m + log2 l) * ln 2
        a.lse[static_cast<size_t>(bh) * a.N + grow] = (m + __log2f(l)) * 0.69314718055994531f;
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128);
    if (warp == 2 && lane == 0 && !*abort_flag) {
      for (int kb = 0; kb < L::KB; ++kb) tma_store_3d(&a.tm_o, sQ + kb * L::BLK, kb * 64, q0, bh);
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
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t st) {
  using L = FwdLayout<D>;
  auto k = fwd_kernel<D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  const int n_qt = (a.N + kTileM - 1) / kTileM;
  dim3 grid(n_qt * a.BH);
  k<<<grid, kFwdThreads, L::SMEM, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, int d, bool bf16, cudaStream_t s) {
  if (d == 128) return bf16 ? launch_fwd_t<128, true>(a, s) : launch_fwd_t<128, false>(a, s);
  return bf16 ? launch_fwd_t<64, true>(a, s) : launch_fwd_t<64, false>(a, s);
}

}  // namespace attn
