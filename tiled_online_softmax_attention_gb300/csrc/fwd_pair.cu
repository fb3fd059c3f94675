// fwd_pair.cu -- the d = 128 forward on CTA pairs (tcgen05 cta_group::2) for sm_103a.
//
// The arithmetic is fwd_kernel's (fwd.cu): online softmax in the base-2 domain with a
// lazily moved reference maximum, P kept in tensor memory, O divided by l once at the end
// ("FlashAttention hardware-aware analysis" (huaweicloud), sections two and four;
// "Understanding online softmax in Flash Attention from scratch", section 3.1).  What
// changes is how the products are shared and pipelined.
//
// Two CTAs on neighbouring SMs form a cluster and take two consecutive 128-row query
// tiles of one (batch, head), one each.  One thread of the even CTA issues every product
// of both as an M = 256 pair product (tcgen05.mma.cta_group::2):
//
//   S(j)  = [Q of CTA 0 ; Q of CTA 1] K_j^T     each CTA supplies its 128 query rows and
//                                              64 of the 128 keys (0-63 / 64-127)
//   O    += [P of CTA 0 ; P of CTA 1] V_j       P from each CTA's tensor memory; each CTA
//                                              supplies 64 of V's 128 columns
//
// and every CTA receives its own 128 rows of S and O, all columns, in its own tensor
// memory.  Per 128 x 128 x 16 step an SM reads 6 KB of operands from shared memory for S
// (Q 4 KB, half of K 2 KB) and 2 KB of V for P V, and its TMA unit writes half of each K/V
// tile: about 96 KB of shared-memory traffic per key tile and 128 query rows where a
// one-CTA kernel needs 160 KB (more than the SM moves in the time the tensor core takes).
// That is what lets a CTA hold a single query tile: the tensor memory left over holds
// kBuf score buffers, and S(j+1) .. S(j+kBuf-1) are computed while the softmax works on
// S(j), so neither waits for the other's hand-offs (one query tile per CTA and no
// double-buffering would leave the tensor core idle during every softmax; the one-CTA
// kernel instead alternates two query tiles, which puts the P -> P V -> next S hand-offs
// on the critical path).
//
// Per key tile j the issuer runs P V(j) once P(j) is written and O rescaled, then S(j+kBuf)
// into the buffer P(j) was read from (the tensor core executes one thread's products in
// order).  The issuing warp waits on two barriers per key tile (the step being ready, and
// the next key tile's K/V slot): on this GPU each wait costs ~130 cycles even when its
// phase is already complete, during which the tensor core drains the issued products, so
// the hand-offs that gate one product share a barrier and a key tile's K and V halves
// share a slot.  The two query tiles of a cluster visit the key tiles of the later one; under
// the causal mask CTA 0's last key tile is then wholly masked for its rows (one product
// of its ~N/128).
//
// Warp roles per CTA (384 threads):
//   warp 0          TMA producer: its Q, then its halves of K_j and V_j into a ring of
//                   32 KB slots; both CTAs' copies complete on CTA 0's barriers
//   warp 1          tensor-memory allocation for the pair; in CTA 0, the product issuer
//                   (the whole warp runs it, one elected lane issues)
//   warpgroup 1     softmax (thread r owns row r = tensor-memory lane r)
//   warpgroup 2     O rescale when a reference max moves, then the epilogue
// Every barrier that feeds a product sits in CTA 0 and counts the warps of both CTAs
// (the partner's arrive through cluster addresses); every product completion is committed
// to both CTAs' barriers at once.  The barriers of the score buffers (and of the P V
// products that read them) are per buffer: with kBuf steps in flight, a single barrier
// could be two phases ahead of, or behind, its waiter, which a parity wait cannot tell.  All waits are bounded; the first to
// expire raises the abort flag of both CTAs.
#include "common.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kBuf = 3;  // score buffers in tensor memory

struct PairLayout {
  static constexpr int D = 128;
  static constexpr int QTILE = kTileM * D * 2;  // 128 query rows: 32 KB
  static constexpr int QBLK = kTileM * 128;     // 128 rows x 128 bytes (64 columns)
  static constexpr int HALF = 64 * D * 2;       // half a K or V tile: 16 KB
  static constexpr int KBLK = 64 * 128;         // 64 key rows x 128 bytes
  static constexpr int SLOT = 2 * HALF;         // one key tile's halves: K at 0, V at HALF
  static constexpr int NSLOT = 5;               // ring slots, key tile j in slot j mod NSLOT
  static constexpr int OFF_Q = 0;               // Q (later O's staging)
  static constexpr int OFF_KV = QTILE;
  static constexpr int OFF_AUX = OFF_KV + NSLOT * SLOT;
  static constexpr int AUX_BAR = 0;             // up to 64 mbarriers
  static constexpr int AUX_ALPHA = 512;         // float[kBuf][128]: rescale factor per row and step
  static constexpr int AUX_M = AUX_ALPHA + 512 * kBuf;
  static constexpr int AUX_L = AUX_M + 512;
  static constexpr int AUX_MISC = AUX_L + 512;  // abort flag, TMEM address
  static constexpr int AUX_BYTES = AUX_MISC + 64;
  static constexpr int SMEM = OFF_AUX + AUX_BYTES + 1024;
  static constexpr uint32_t TM_COLS = 512;
  static constexpr uint32_t tm_s(int b) { return 128u * b; }
  static constexpr uint32_t TM_O = 128u * kBuf;
  static_assert(TM_O + D <= TM_COLS, "score buffers and O must fit the tensor memory");
};

constexpr int kPairThreads = 384;
constexpr float kPairRescaleThreshold = 8.0f;  // log2 units, as in fwd_kernel

enum : int {
  P_Q = 0,         // both CTAs' Q landed (CTA 0)
  P_DRAIN = 1,     // every product done (CTA 0)
  P_FIN = 2,       // final m, l published (within a CTA)
  P_SFULL = 4,     // + b: S in buffer b computed (both CTAs)
  P_READY = 8,     // + b: the step in buffer b may run P V: P written by the pair's eight
                   //      softmax warps and O rescaled by its eight correction warps (CTA 0)
  P_STAT = 12,     // + b: rescale factors of the step in buffer b published (within a CTA)
  P_ODONE = 16,    // + b: P V of the step in buffer b done (both CTAs)
  P_KVFULL = 20,   // + slot: both CTAs' K and V halves landed (CTA 0)
  P_KVEMPTY = 28,  // + slot: the slot's products done (both CTAs)
  P_COUNT = 36
};
static_assert(kBuf <= 4 && P_KVFULL + PairLayout::NSLOT <= P_KVEMPTY && P_KVEMPTY + PairLayout::NSLOT <= P_COUNT &&
                  P_COUNT <= 64 && PairLayout::NSLOT >= kBuf + 2,
              "barrier map and ring depth");

// Bounded wait for the pair: like mbar_wait, acquiring at cluster scope, and an expired
// wait raises the partner's abort flag too, so that neither CTA waits out its own limits
// on work the other has abandoned.
struct PairWait {
  volatile int* abort;  // this CTA's flag
  uint32_t peer_abort;  // the partner's flag (cluster address)
  int* dev_status;
  uint64_t limit_ns;
};

static __device__ __forceinline__ bool pwait(uint32_t bar, uint32_t parity, const PairWait& w) {
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

__device__ __forceinline__ bool pwait_warp(uint32_t bar, uint32_t parity, const PairWait& w) {
  return __all_sync(0xffffffffu, pwait(bar, parity, w));
}

template <bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    fwd_pair_kernel(const __grid_constant__ FwdArgs a) {
  using L = PairLayout;
  constexpr int D = L::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  uint8_t* aux = smem + L::OFF_AUX;
  const uint32_t bars = sb + L::OFF_AUX + L::AUX_BAR;
  auto bar = [&](int b) -> uint32_t { return bars + 8u * b; };
  float* alpha_s = reinterpret_cast<float*>(aux + L::AUX_ALPHA);
  float* m_s = reinterpret_cast<float*>(aux + L::AUX_M);
  float* l_s = reinterpret_cast<float*>(aux + L::AUX_L);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(aux + L::AUX_MISC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aux + L::AUX_MISC + 8);

  const uint32_t rank = cluster_ctarank();  // 0: the CTA that issues the products
  const bool lead = rank == 0;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_t = (a.N + kTileM - 1) / kTileM;
  const int n_sup = (n_t + 1) / 2;  // query-tile pairs per head
  const WorkItem wi = work_item(static_cast<int>(blockIdx.x >> 1), a.BH, n_sup);
  const int bh = wi.bh;
  const int sp = n_sup - 1 - wi.rank;  // longest causal pair first
  const int qt = 2 * sp + static_cast<int>(rank);  // this CTA's query tile (past the end for
                                                   // CTA 1 of an odd last pair)
  // Key tiles the pair visits: those of its later tile (the last one that exists).
  const int n_kv = visible_key_tiles(min(2 * sp + 1, n_t - 1), a.Nk, a.causal, a.cofs);

  if (threadIdx.x == 0) {
    mbar_init(bar(P_Q), 1);
    mbar_init(bar(P_DRAIN), 1);
    mbar_init(bar(P_FIN), 4);
    for (int b = 0; b < kBuf; ++b) {
      mbar_init(bar(P_SFULL + b), 1);
      mbar_init(bar(P_READY + b), 16);
      mbar_init(bar(P_STAT + b), 4);
      mbar_init(bar(P_ODONE + b), 1);
    }
    for (int s = 0; s < L::NSLOT; ++s) {
      mbar_init(bar(P_KVFULL + s), 1);
      mbar_init(bar(P_KVEMPTY + s), 1);
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
  const PairWait wc{abort_flag, mapa_shared(smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u), a.dev_status,
                    a.wait_limit_ns};
  auto lead_bar = [&](int b) -> uint32_t { return mapa_shared(bar(b), 0); };
  // One arrival per warp on CTA 0's barrier b (a hand-off that feeds a product).
  auto arrive_lead_warp = [&](int b) {
    __syncwarp();
    if (lane == 0) {
      if (lead)
        mbar_arrive(bar(b));
      else
        mbar_arrive_cluster(lead_bar(b));
    }
  };
  // Step j uses score buffer j mod kBuf; its barriers there are in phase j / kBuf.
  auto buf_of = [](int j) { return j % kBuf; };
  auto use_parity = [](int j) { return static_cast<uint32_t>((j / kBuf) & 1); };
  const int wg = warp >> 2;

  // Register split: 120 (control) + 224 (softmax) + 120 (correction) per lane triple,
  // within the 168 x 384 threads of the launch.
  if (wg == 0) {
    setmaxnreg_dec<120>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_kh);
      prefetch_tmap(&a.tm_v);
      prefetch_tmap(&a.tm_o);
      if (lead) mbar_arrive_expect_tx(bar(P_Q), 2 * L::QTILE);
      for (int kb = 0; kb < 2; ++kb)
        tma_load_3d_pair(sb + L::OFF_Q + kb * L::QBLK, &a.tm_q, lead_bar(P_Q), kb * 64, qt * kTileM, bh);
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % L::NSLOT;
        if (j >= L::NSLOT && !pwait(bar(P_KVEMPTY + s), ((j / L::NSLOT) - 1) & 1, wc)) break;
        if (lead) mbar_arrive_expect_tx(bar(P_KVFULL + s), 2 * L::SLOT);
        const uint32_t dst = sb + L::OFF_KV + s * L::SLOT;
        // K_j: this CTA's 64 keys, both 64-column blocks; V_j: all 128 keys, its 64 columns
        for (int kb = 0; kb < 2; ++kb)
          tma_load_3d_pair(dst + kb * L::KBLK, &a.tm_kh, lead_bar(P_KVFULL + s), kb * 64,
                           j * kTileN + 64 * static_cast<int>(rank), bh);
        tma_load_3d_pair(dst + L::HALF, &a.tm_v, lead_bar(P_KVFULL + s), 64 * static_cast<int>(rank), j * kTileN, bh);
        issued = j + 1;
      }
      if (lead) {
        // Every copy of both CTAs completes on these barriers: let them land before
        // either CTA can exit (the partner leaves only after the final cluster barrier).
        pwait(bar(P_Q), 0, wc);
        for (int j = (issued > L::NSLOT ? issued - L::NSLOT : 0); j < issued; ++j)
          pwait(bar(P_KVFULL + j % L::NSLOT), (j / L::NSLOT) & 1, wc);
      }
    } else if (warp == 1 && lead) {
      // ---------------------------------------------------------- pair product issuer
      constexpr uint32_t idesc_qk = idesc_f16(2 * kTileM, kTileN, BF16, false, false);
      constexpr uint32_t idesc_pv = idesc_f16(2 * kTileM, D, BF16, false, true);
      constexpr uint16_t kBoth = 3;
      auto full = [&](int j) { return pwait_warp(bar(P_KVFULL + j % L::NSLOT), (j / L::NSLOT) & 1, wc); };
      auto issue_s = [&](int j) {  // S(j) into buffer j mod kBuf
        const uint32_t kbase = sb + L::OFF_KV + (j % L::NSLOT) * L::SLOT;
        if (elect_one_sync()) {
#pragma unroll
          for (int k = 0; k < D / 16; ++k)
            mma_ss_pair(tmem + L::tm_s(buf_of(j)), sdesc_sw128(sb + L::OFF_Q + (k >> 2) * L::QBLK + (k & 3) * 32, 16, 1024),
                        sdesc_sw128(kbase + (k >> 2) * L::KBLK + (k & 3) * 32, 16, 1024), idesc_qk, k > 0 ? 1u : 0u);
          tc_commit_pair(bar(P_SFULL + buf_of(j)), kBoth);
        }
        __syncwarp();
      };
      auto issue_pv = [&](int j) {  // O += P(j) V_j; key tile j's slot is then free
        const uint32_t vbase = sb + L::OFF_KV + (j % L::NSLOT) * L::SLOT + L::HALF;
        // 16 keys per step: 8 columns of packed P, 16 rows (2 KB) of this CTA's V half
        if (elect_one_sync()) {
#pragma unroll
          for (int k = 0; k < kTileN / 16; ++k)
            mma_ts_pair(tmem + L::TM_O, tmem + L::tm_s(buf_of(j)) + k * 8, sdesc_sw128(vbase + k * 2048, L::HALF, 1024),
                        idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
          tc_commit_pair(bar(P_ODONE + buf_of(j)), kBoth);
          tc_commit_pair(bar(P_KVEMPTY + j % L::NSLOT), kBoth);
        }
        __syncwarp();
      };
      bool ok = pwait_warp(bar(P_Q), 0, wc);
      for (int j = 0; ok && j < min(kBuf, n_kv); ++j) {
        if (!(ok = full(j))) break;
        tc_fence_after();
        issue_s(j);
      }
      // Per key tile: P V(j) once its step is ready (its slot was waited for by S(j)), then
      // S(j + kBuf) into the buffer P(j) was read from.
      for (int j = 0; ok && j < n_kv; ++j) {
        if (!(ok = pwait_warp(bar(P_READY + buf_of(j)), use_parity(j), wc))) break;
        tc_fence_after();
        issue_pv(j);
        if (j + kBuf < n_kv) {
          if (!(ok = full(j + kBuf))) break;
          tc_fence_after();
          issue_s(j + kBuf);
        }
      }
      // Drain: nothing may still write either CTA's tensor memory when it is released.
      tc_commit_pair_w(bar(P_DRAIN), 1);
      pwait_warp(bar(P_DRAIN), 0, wc);
    }
  } else if (wg == 1) {
    // ------------------------------------------------------------ softmax
    setmaxnreg_inc<224>();
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const int grow = qt * kTileM + row;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float tsc = a.scale_log2;
    float m = -INFINITY;  // reference max (scale*log2(e) units)
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int b = buf_of(j);
      if (!pwait_warp(bar(P_SFULL + b), use_parity(j), wc)) { ok = false; break; }
      tc_fence_after();
      const uint32_t t_s = t_lane + L::tm_s(b);
      float s[128];
      {
        uint32_t sr[128];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld_x32_async(t_s + 32 * q, sr + 32 * q);
        tmem_ld_wait(sr);
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
      }
      const int k0 = j * kTileN;
      const bool tail = k0 + kTileN > a.Nk;
      const bool diag = a.causal && (k0 + kTileN - 1 > qt * kTileM + a.cofs);
      if (tail || diag) {
        int lim = a.Nk - k0;
        if (a.causal) lim = min(lim, grow + a.cofs - k0 + 1);
#pragma unroll
        for (int c = 0; c < kTileN; ++c)
          if (c >= lim) s[c] = -INFINITY;
      }
      // A tree of three-input maxima: with one softmax warp per SM sub-partition nothing
      // hides the latency of a 127-long chain.
      const float mx = rowmax128(s) * tsc;
      const float m_new = (mx - m > kPairRescaleThreshold) ? mx : m;
      const float alpha = (m_new == m) ? 1.f : ex2(m - m_new);  // 0 on the first visible tile
      alpha_s[b * 128 + row] = alpha;
      mbar_arrive_warp(bar(P_STAT + b));
      m = m_new;
      const float m_use = (m == -INFINITY) ? 0.f : m;
      uint32_t pk[64];
      const uint64_t tsc2 = f32x2_pack(tsc, tsc), negm2 = f32x2_pack(-m_use, -m_use);
      uint64_t acc2[2] = {0ull, 0ull};
#pragma unroll
      for (int c = 0; c < kTileN; c += 2) {
        float x0, x1;
        f32x2_unpack(f32x2_fma(f32x2_pack(s[c], s[c + 1]), tsc2, negm2), x0, x1);
        const float p0 = ex2(x0);
        const float p1 = ex2(x1);
        acc2[(c / 2) & 1] = f32x2_add(acc2[(c / 2) & 1], f32x2_pack(p0, p1));
        pk[c / 2] = pack2<BF16>(p0, p1);
      }
      float a0, a1, b0, b1;
      f32x2_unpack(acc2[0], a0, a1);
      f32x2_unpack(acc2[1], b0, b1);
      l = fmaf(l, alpha, (a0 + a1) + (b0 + b1));
      tmem_st_x64(t_s, pk);
      tmem_st_wait();
      tc_fence_before();
      arrive_lead_warp(P_READY + b);
    }
    if (ok) {
      m_s[row] = (m == -INFINITY) ? 0.f : m;
      l_s[row] = l;
      mbar_arrive_warp(bar(P_FIN));
    }
  } else {
    // ------------------------------------------------------------ correction + epilogue
    setmaxnreg_dec<120>();
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t t_o = tmem + (static_cast<uint32_t>(wq * 32) << 16) + L::TM_O;
    bool ok = true;
    for (int j = 0; ok && j < n_kv; ++j) {
      const int b = buf_of(j);
      if (!(ok = pwait_warp(bar(P_STAT + b), use_parity(j), wc))) break;
      const float alpha = alpha_s[b * 128 + row];
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O holds the sum up to key tile j-1: wait for that product, then rescale.  (Its
        // buffer's previous product, P V(j-1-kBuf), is done: S(j) was issued after it.)
        if (!(ok = pwait_warp(bar(P_ODONE + buf_of(j - 1)), use_parity(j - 1), wc))) break;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld_x32(t_o + cc * 32, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st_x32(t_o + cc * 32, o);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      arrive_lead_warp(P_READY + b);
    }
    // Epilogue: O / l -> 16-bit -> swizzled staging over Q -> TMA store; logsumexp.
    const bool ok_e = ok && pwait_warp(bar(P_FIN), 0, wc) &&
                      pwait_warp(bar(P_ODONE + buf_of(n_kv - 1)), use_parity(n_kv - 1), wc);
    const int q0 = qt * kTileM;
    if (ok_e) {
      tc_fence_after();
      const float mf = m_s[row];
      const float lf = l_s[row];
      const float inv_l = 1.f / lf;
      uint8_t* stage = smem + L::OFF_Q;  // Q is no longer read by either CTA
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld_x32(t_o + cc * 32, o);
        uint32_t pkd[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pkd[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
        const int kb = (cc * 32) / 64;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int ch = ((cc * 32) % 64) / 8 + q;
          uint4* dst = reinterpret_cast<uint4*>(stage + kb * L::QBLK + row * 128 + ((ch ^ (row & 7)) << 4));
          *dst = make_uint4(pkd[4 * q], pkd[4 * q + 1], pkd[4 * q + 2], pkd[4 * q + 3]);
        }
      }
      if (q0 + row < a.N) a.lse[static_cast<size_t>(bh) * a.N + q0 + row] = (mf + __log2f(lf)) * 0.69314718055994531f;
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128);
    if (warp == 8 && lane == 0) {
      if (ok_e && !*abort_flag && q0 < a.N) {
        for (int kb = 0; kb < 2; ++kb) tma_store_3d(&a.tm_o, sb + L::OFF_Q + kb * L::QBLK, kb * 64, q0, bh);
        bulk_commit();
      }
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
cudaError_t launch_pair_t(const FwdArgs& a, cudaStream_t st) {
  auto k = fwd_pair_kernel<BF16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, PairLayout::SMEM);
  if (e != cudaSuccess) return e;
  const int n_t = (a.N + kTileM - 1) / kTileM;
  k<<<dim3(2 * ((n_t + 1) / 2) * a.BH), kPairThreads, PairLayout::SMEM, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_pair(const FwdArgs& a, bool bf16, cudaStream_t s) {
  return bf16 ? launch_pair_t<true>(a, s) : launch_pair_t<false>(a, s);
}

}  // namespace attn
