// fwd_persist.cu -- the d = 64 forward on a persistent grid for sm_103a.
//
// The arithmetic is fwd_kernel's (fwd.cu) for d = 64 with 16-bit inputs: online softmax
// in the base-2 domain with a lazily moved reference maximum, P kept in tensor memory,
// O divided by l once at the end ("FlashAttention hardware-aware analysis" (huaweicloud),
// sections two and four; "Understanding online softmax in Flash Attention from scratch",
// section 3.1), and the same product order: the two O tiles take 128 tensor-memory
// columns, S/P has three 128-column buffers, S_i(j) goes to buffer (2j + i) mod 3, and per
// key tile the issuer runs S_0(j+1), P_0 V(j), S_1(j+1), P_1 V(j).
//
// What changes is the schedule (huaweicloud section four, part 2: FA2's work partitioning
// over the SMs).  A work unit is two consecutive query tiles of one (batch, head), as
// before, and the grid still has one CTA per unit in longest-first order, but a CTA does
// not stop after its unit: it asks the hardware scheduler to cancel the launch of the next
// CTA that has not started (cluster launch control, clusterlaunchcontrol.try_cancel) and
// runs that CTA's unit itself, until an answer cancels nothing.  The order of the units is
// the hardware's launch order, so the longest-first greedy schedule stays, and no counter
// in memory is needed.  Within a CTA the units follow each other without a break:
//
//   * barrier phases carry over from one unit to the next (nothing is re-initialised):
//     every role counts, per barrier, the phases of the units it has finished;
//   * Q has two sets of two tiles (unit u uses set u mod 2), so the next unit's Q is
//     loaded while this one still computes; the epilogue stages O over its own unit's Q
//     (every S product of the unit is done by then), and the producer reloads a set once
//     the O stores of the unit before have read it;
//   * the producer asks for unit u+1 once it has issued unit u's last K/V load (about
//     the ring's depth, four key tiles, before unit u ends: asking when unit u starts
//     would hold every CTA's next unit a whole unit ahead, and the grid's tail would then
//     leave SMs idle beside CTAs that still hold a unit), then loads its Q and K/V as the
//     ring frees up; the issuer starts unit u+1's products right after unit u's last P V,
//     and the only hand-off between units is O: P_i V(0) of unit u+1 (accumulate = 0)
//     waits until the epilogue of unit u has read O_i out of tensor memory.
//
// Each role sets its register budget once (setmaxnreg) and loops over the units inside
// the role.  The answer to each request lands in one of four 16-byte slots; every role
// reads it to learn the next unit (or that there is none), and the producer reuses a
// slot only after all readers have arrived on its "read" barrier.  The four correction
// warps use named barriers in their epilogue, so they leave the unit loop together (a
// named barrier with an AND reduction).  Every mbarrier wait is bounded as everywhere
// else.  Query-tile counts must be even (every unit has two real tiles); the launcher
// refuses other shapes.
#include "common.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kPThreads = 512;
constexpr float kPRescaleThreshold = 8.0f;  // log2 units, as in fwd_kernel

struct PersistLayout {
  static constexpr int D = 64;
  static constexpr int TILE = kTileM * D * 2;  // one 128-row tile: 16 KB (one 128-byte block per row)
  static constexpr int NSLOT = 8;              // K/V ring entries, one tile each
  static constexpr int OFF_Q = 0;              // Q set s, tile i at (2 s + i) * TILE (later O's staging)
  static constexpr int OFF_KV = 4 * TILE;
  static constexpr int OFF_AUX = OFF_KV + NSLOT * TILE;
  static constexpr int AUX_BAR = 0;            // up to 64 mbarriers
  static constexpr int AUX_CLC = 512;          // four 16-byte answers
  static constexpr int AUX_ALPHA = 576;        // float[2][2][128]: rescale factor per slot, tile, row
  static constexpr int AUX_M = AUX_ALPHA + 2048;
  static constexpr int AUX_L = AUX_M + 1024;
  static constexpr int AUX_MISC = AUX_L + 1024;  // abort flag, TMEM address
  static constexpr int AUX_BYTES = AUX_MISC + 64;
  static constexpr int SMEM = OFF_AUX + AUX_BYTES + 1024;
  static constexpr uint32_t TM_COLS = 512;
  static constexpr uint32_t tm_o(int i) { return 256u + D * i; }
  static constexpr uint32_t tm_sbuf(int b) { return b < 2 ? 128u * b : 384u; }
};

enum : int {
  U_Q = 0,         // + 2 set + tile: the Q tile landed
  U_STFREE = 4,    // + set: the O stores of the set's last unit have read it
  U_SFULL = 6,     // + 3 tile + buffer: S of that tile computed into that buffer
  U_PFULL = 12,    // + tile: P written (softmax)
  U_STAT = 14,     // + tile: rescale factors of this key tile published (softmax)
  U_CORR = 16,     // + tile: O rescaled if needed (correction)
  U_ODONE = 18,    // + tile: P V done
  U_OLAST = 20,    // + tile: every product of the tile in this unit done (once per unit)
  U_FIN = 22,      // + tile: final m, l published (softmax)
  U_OFREE = 24,    // + tile: the epilogue has read O, m and l of the tile
  U_DRAIN = 26,
  U_CLC = 27,      // + slot (4): an answer landed
  U_CLCREAD = 31,  // + slot (4): every reader has read it
  U_KVFULL = 35,   // + ring slot (up to 8)
  U_KVEMPTY = 43,  // + ring slot (up to 8)
  U_COUNT = 51
};
static_assert(U_KVFULL + PersistLayout::NSLOT <= U_KVEMPTY && U_KVEMPTY + PersistLayout::NSLOT <= U_COUNT &&
                  8 * U_COUNT <= PersistLayout::AUX_CLC,
              "barrier map");

// Warps that read every answer besides the producer: the issuer, 8 softmax, 4 correction.
constexpr uint32_t kClcReaders = 13;

// One unit: (batch, head), its pair of query tiles and the key tiles each visits.
struct Unit {
  int bh, pr, n0, n1;
};

__device__ __forceinline__ Unit unit_of(const FwdArgs& a, int x) {
  const int n_pairs = ((a.N + kTileM - 1) / kTileM) / 2;
  const WorkItem wi = work_item(x, a.BH, n_pairs);
  const int pr = n_pairs - 1 - wi.rank;  // longest causal pair first
  return {wi.bh, pr, visible_key_tiles(2 * pr, a.Nk, a.causal, a.cofs),
          visible_key_tiles(2 * pr + 1, a.Nk, a.causal, a.cofs)};
}

// S products of tile i in one unit of n_i key tiles that land in buffer b: S_i(j) goes to
// buffer (2j + i) mod 3, so those with j = j_b mod 3, j_b = 2 (b - i) mod 3.
__device__ __forceinline__ int tile_buf_uses(int n_i, int i, int b) {
  const int jb = (2 * (b - i) % 3 + 3) % 3;
  return (n_i + 2 - jb) / 3;
}

template <bool BF16>
__global__ void __launch_bounds__(kPThreads, 1) fwd_persist_kernel(const __grid_constant__ FwdArgs a) {
  using L = PersistLayout;
  constexpr int D = L::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  uint8_t* aux = smem + L::OFF_AUX;
  const uint32_t bars = sb + L::OFF_AUX + L::AUX_BAR;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * i; };
  auto resp = [&](int slot) -> uint32_t { return sb + L::OFF_AUX + L::AUX_CLC + 16u * slot; };
  float* alpha_s = reinterpret_cast<float*>(aux + L::AUX_ALPHA);
  float* m_s = reinterpret_cast<float*>(aux + L::AUX_M);
  float* l_s = reinterpret_cast<float*>(aux + L::AUX_L);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(aux + L::AUX_MISC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aux + L::AUX_MISC + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(bar(U_Q + i), 1);
    for (int s = 0; s < 2; ++s) mbar_init(bar(U_STFREE + s), 1);
    for (int b = 0; b < 6; ++b) mbar_init(bar(U_SFULL + b), 1);
    for (int i = 0; i < 2; ++i) mbar_init(bar(U_OLAST + i), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(U_PFULL + i), 4);
      mbar_init(bar(U_STAT + i), 4);
      mbar_init(bar(U_CORR + i), 4);
      mbar_init(bar(U_ODONE + i), 1);
      mbar_init(bar(U_FIN + i), 4);
      mbar_init(bar(U_OFREE + i), 4);
    }
    mbar_init(bar(U_DRAIN), 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(bar(U_CLC + s), 1);
      mbar_init(bar(U_CLCREAD + s), kClcReaders);
    }
    for (int s = 0; s < L::NSLOT; ++s) {
      mbar_init(bar(U_KVFULL + s), 1);
      mbar_init(bar(U_KVEMPTY + s), 1);
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
  const int wg = warp >> 2;
  // The unit after unit u (the answer to the request made as u started), or -1; every
  // lane of the calling warp calls it, and one arrival per warp marks the slot read.
  auto next_unit = [&](int u, bool& ok) -> int {
    const int slot = u & 3;
    if (!(ok = mbar_wait_warp(bar(U_CLC + slot), (u >> 2) & 1, wc))) return -1;
    // (broadcast from lane 0: the value is the same in every lane, and the compiler can
    // then keep everything derived from it in uniform registers)
    const int x = __shfl_sync(0xffffffffu, clc_cancelled_x(resp(slot)), 0);
    mbar_arrive_warp(bar(U_CLCREAD + slot));
    return x;
  };

  // Register split: 64 (control) + 2 x 184 (softmax) + 80 (correction) per lane quadruple
  // = 128 x 512 threads, the launch allotment.
  if (wg == 0) {
    setmaxnreg_dec<64>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- TMA producer
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
      prefetch_tmap(&a.tm_o);
      int x = static_cast<int>(blockIdx.x);
      int ld = 0;            // K/V loads issued, over all units
      int u = 0;
      bool asked = false;    // a request whose answer has not been waited for
      for (;; ++u) {
        const Unit un = unit_of(a, x);
        const int set = u & 1;
        if (u >= 2 && !mbar_wait(bar(U_STFREE + set), ((u >> 1) - 1) & 1, wc)) break;
        for (int i = 0; i < 2; ++i) {
          mbar_arrive_expect_tx(bar(U_Q + 2 * set + i), L::TILE);
          tma_load_3d(sb + L::OFF_Q + (2 * set + i) * L::TILE, &a.tm_q, bar(U_Q + 2 * set + i), 0,
                      (2 * un.pr + i) * kTileM, un.bh);
        }
        bool ok = true;
        for (int l = 0; l < 2 * un.n1; ++l, ++ld) {  // K_j, V_j alternately
          const int s = ld % L::NSLOT;
          if (ld >= L::NSLOT && !(ok = mbar_wait(bar(U_KVEMPTY + s), ((ld / L::NSLOT) - 1) & 1, wc))) break;
          mbar_arrive_expect_tx(bar(U_KVFULL + s), L::TILE);
          tma_load_3d(sb + L::OFF_KV + s * L::TILE, (l & 1) ? &a.tm_v : &a.tm_k, bar(U_KVFULL + s), 0,
                      (l >> 1) * kTileN, un.bh);
        }
        if (!ok) break;
        // Every load of this unit is issued: ask for the unit after it (slot u mod 4, once
        // that slot's earlier answer has been read by every role).
        const int slot = u & 3;
        if (u >= 4 && !mbar_wait(bar(U_CLCREAD + slot), ((u >> 2) - 1) & 1, wc)) break;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar(U_CLC + slot), 16);
        clc_try_cancel(resp(slot), bar(U_CLC + slot));
        asked = true;
        if (!mbar_wait(bar(U_CLC + slot), (u >> 2) & 1, wc)) break;
        asked = false;
        x = clc_cancelled_x(resp(slot));
        if (x < 0) break;
      }
      // Let every copy and answer this thread started land before the CTA can exit.
      if (asked) mbar_wait(bar(U_CLC + (u & 3)), (u >> 2) & 1, wc);
      for (int v = (u > 1 ? u - 1 : 0); v <= u; ++v)
        for (int i = 0; i < 2; ++i) mbar_wait(bar(U_Q + 2 * (v & 1) + i), (v >> 1) & 1, wc);
      for (int l = (ld > L::NSLOT ? ld - L::NSLOT : 0); l < ld; ++l)
        mbar_wait(bar(U_KVFULL + l % L::NSLOT), (l / L::NSLOT) & 1, wc);
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer (the whole
      // warp runs it, one elected lane issues)
      constexpr uint32_t idesc_qk = idesc_f16(kTileM, kTileN, BF16, false, false);
      constexpr uint32_t idesc_pv = idesc_f16(kTileM, D, BF16, false, true);
      int x = static_cast<int>(blockIdx.x);
      uint32_t ldb = 0;                 // the unit's first K/V load
      uint32_t par_p = 0, par_c = 0;    // bit i: parity of tile i's P V products / U_CORR phases so far
      bool ok = true;
      for (int u = 0; ok; ++u) {
        const Unit un = unit_of(a, x);
        const int n0 = un.n0, n1 = un.n1;
        // Per-unit constants, captured by value: the Q tiles of this unit's set, the
        // unit's first ring load, the phase parities it starts from.
        const uint32_t q_base = sb + L::OFF_Q + static_cast<uint32_t>(2 * (u & 1)) * L::TILE;
        const uint32_t q_bar = bar(U_Q + 2 * (u & 1));
        const uint32_t q_par = static_cast<uint32_t>(u >> 1) & 1u;
        const uint32_t lb = ldb, pp = par_p, pc = par_c;
        const bool first = u == 0;
        const uint32_t of_par = static_cast<uint32_t>(u - 1) & 1u;
        auto slot_of = [=](uint32_t l) { return (lb + l) % L::NSLOT; };
        auto full = [=, &wc](uint32_t l) {
          return mbar_wait_warp(bar(U_KVFULL + static_cast<int>((lb + l) % L::NSLOT)), ((lb + l) / L::NSLOT) & 1u, wc);
        };
        auto issue_s = [=](int i, int j) {
          const uint32_t qb = q_base + static_cast<uint32_t>(i) * L::TILE;
          const uint32_t kbase = sb + L::OFF_KV + slot_of(2u * j) * L::TILE;
          const int b = (2 * j + i) % 3;
          if (elect_one_sync()) {
#pragma unroll
            for (int k = 0; k < D * 2 / 32; ++k)
              mma_ss(tmem + L::tm_sbuf(b), sdesc_sw128(qb + k * 32, 16, 1024), sdesc_sw128(kbase + k * 32, 16, 1024),
                     idesc_qk, k > 0 ? 1u : 0u);
            tc_commit(bar(U_SFULL + 3 * i + b));
          }
          __syncwarp();
        };
        auto issue_pv = [=](int i, int j) {
          const uint32_t vbase = sb + L::OFF_KV + slot_of(2u * j + 1u) * L::TILE;
          const int b = (2 * j + i) % 3;
          // One MMA per 16 keys: 8 columns of packed P, 16 rows (2 KB) of V.
          if (elect_one_sync()) {
#pragma unroll
            for (int k = 0; k < kTileN / 16; ++k)
              mma_ts(tmem + L::tm_o(i), tmem + L::tm_sbuf(b) + k * 8, sdesc_sw128(vbase + k * 2048, kTileM * 128, 1024),
                     idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
            tc_commit(bar(U_ODONE + i));
          }
          __syncwarp();
        };
        // P_i V(j) may run: P written, O rescaled for it, and for j = 0 the previous
        // unit's O_i read out by its epilogue.
        auto pv_ready = [=, &wc](int i, int j) {
          if (!mbar_wait_warp(bar(U_PFULL + i), ((pp >> i) + static_cast<uint32_t>(j)) & 1u, wc)) return false;
          if (j > 0) return mbar_wait_warp(bar(U_CORR + i), ((pc >> i) + static_cast<uint32_t>(j) - 1u) & 1u, wc);
          return first || mbar_wait_warp(bar(U_OFREE + i), of_par, wc);
        };
        ok = mbar_wait_warp(q_bar, q_par, wc) && full(0);
        if (ok) {
          tc_fence_after();
          issue_s(0, 0);
          ok = mbar_wait_warp(q_bar + 8, q_par, wc);
        }
        if (ok) {
          tc_fence_after();
          issue_s(1, 0);
          tc_commit_w(bar(U_KVEMPTY + static_cast<int>(slot_of(0))));
        }
        for (int j = 0; ok && j < n1; ++j) {
          // S_0(j+1) | P_0 V(j) | S_1(j+1) | P_1 V(j).  V(j) is waited for before S_0(j+1)
          // is issued, so that nothing stands between that product and the wait for P_0(j):
          // tile 0's softmax, which S_0(j+1) lets run on, cannot complete P_0(j+1) first
          // (two phases of U_PFULL ahead of a parity wait).
          const bool k_next = j + 1 < n1;
          if (!(ok = full(2u * j + 1u))) break;
          if (k_next && !(ok = full(2u * j + 2u))) break;
          if (j + 1 < n0) {
            tc_fence_after();
            issue_s(0, j + 1);
          }
          if (j < n0) {
            if (!(ok = pv_ready(0, j))) break;
            tc_fence_after();
            issue_pv(0, j);
            if (j == n0 - 1) tc_commit_w(bar(U_OLAST + 0));
          }
          if (k_next) {
            tc_fence_after();
            issue_s(1, j + 1);
            tc_commit_w(bar(U_KVEMPTY + static_cast<int>(slot_of(2u * j + 2u))));
          }
          if (!(ok = pv_ready(1, j))) break;
          tc_fence_after();
          issue_pv(1, j);
          tc_commit_w(bar(U_KVEMPTY + static_cast<int>(slot_of(2u * j + 1u))));
        }
        if (!ok) break;
        tc_commit_w(bar(U_OLAST + 1));
        ldb += 2u * static_cast<uint32_t>(n1);
        par_p ^= (static_cast<uint32_t>(n0) & 1u) | ((static_cast<uint32_t>(n1) & 1u) << 1);
        par_c ^= (static_cast<uint32_t>(n0 - 1) & 1u) | ((static_cast<uint32_t>(n1 - 1) & 1u) << 1);
        x = next_unit(u, ok);
        if (x < 0) break;
      }
      // Drain: nothing may still write tensor memory when it is released.
      tc_commit_w(bar(U_DRAIN));
      mbar_wait_warp(bar(U_DRAIN), 0, wc);
    }
  } else if (wg <= 2) {
    // ------------------------------------------------------------ softmax of tile i
    setmaxnreg_inc<184>();
    const int i = wg - 1;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t t_lane_s = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float tsc = a.scale_log2;
    int x = static_cast<int>(blockIdx.x);
    uint32_t par_s = 0;        // bit b: parity of this tile's S products into buffer b so far
    int cum_a = 0;             // rescale factors published so far (U_STAT phases)
    bool ok = true;
    for (int u = 0; ok; ++u) {
      const Unit un = unit_of(a, x);
      const int n_i = i ? un.n1 : un.n0;
      const int grow = (2 * un.pr + i) * kTileM + row;
      float m = -INFINITY;  // reference max (scale*log2(e) units) used by the exponentials
      float l = 0.f;        // row sum of ex2(. - m)
      for (int j = 0; j < n_i; ++j) {
        const int b = (2 * j + i) % 3;
        // (each tile has its own barrier per buffer: waited for in order, every phase)
        if (!(ok = mbar_wait_warp(bar(U_SFULL + 3 * i + b), ((par_s >> b) ^ (j / 3)) & 1, wc))) break;
        tc_fence_after();
        const uint32_t t_s = t_lane_s + L::tm_sbuf(b);
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
        const bool diag = a.causal && (k0 + kTileN - 1 > (2 * un.pr + i) * kTileM + a.cofs);
        if (tail || diag) {
          int lim = a.Nk - k0;                                  // keys past the end
          if (a.causal) lim = min(lim, grow + a.cofs - k0 + 1);  // keys after this query
#pragma unroll
          for (int c = 0; c < kTileN; ++c)
            if (c >= lim) s[c] = -INFINITY;
        }
        float mx = s[0];
#pragma unroll
        for (int c = 1; c < kTileN; ++c) mx = fmaxf(mx, s[c]);
        mx *= tsc;
        // Move the reference max only when it is exceeded by more than the threshold.
        const float m_new = (mx - m > kPRescaleThreshold) ? mx : m;
        const float alpha = (m_new == m) ? 1.f : ex2(m - m_new);  // 0 on the first tile
        if (j > 0) {
          // Two slots: the correction may still be reading the previous factor (at the
          // start of a unit it is finishing the last unit's epilogue).
          alpha_s[(((cum_a + j - 1) & 1) * 2 + i) * 128 + row] = alpha;
          mbar_arrive_warp(bar(U_STAT + i));
        }
        m = m_new;
        const float m_use = (m == -INFINITY) ? 0.f : m;  // a row with nothing visible yet
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
        float rs;
        {
          float a0, a1, b0, b1;
          f32x2_unpack(acc2[0], a0, a1);
          f32x2_unpack(acc2[1], b0, b1);
          rs = (a0 + a1) + (b0 + b1);
        }
        l = fmaf(l, alpha, rs);
        tmem_st_x64(t_s, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(bar(U_PFULL + i));
      }
      if (!ok) break;
      // The previous unit's epilogue has read m and l (and O) of this tile.
      if (u > 0 && !(ok = mbar_wait_warp(bar(U_OFREE + i), (u - 1) & 1, wc))) break;
      m_s[i * 128 + row] = (m == -INFINITY) ? 0.f : m;
      l_s[i * 128 + row] = l;
      mbar_arrive_warp(bar(U_FIN + i));
      cum_a += n_i - 1;
      for (int b = 0; b < 3; ++b) par_s ^= static_cast<uint32_t>(tile_buf_uses(n_i, i, b) & 1) << b;
      x = next_unit(u, ok);
      if (x < 0) break;
    }
  } else {
    // ------------------------------------------------------------ correction + epilogue
    setmaxnreg_dec<80>();
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    int x = static_cast<int>(blockIdx.x);
    int cum_p[2] = {0, 0}, cum_c[2] = {0, 0};
    for (int u = 0;; ++u) {
      const Unit un = unit_of(a, x);
      const int n_kv[2] = {un.n0, un.n1};
      bool ok = true;
      for (int j = 1; ok && j < un.n1; ++j) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (j >= n_kv[i]) continue;
          if (!(ok = mbar_wait_warp(bar(U_STAT + i), (cum_c[i] + j - 1) & 1, wc))) break;
          const float alpha = alpha_s[(((cum_c[i] + j - 1) & 1) * 2 + i) * 128 + row];
          // Every step waits for P_i V(j-1) first, rescaling or not: that product is issued
          // only once the issuer has consumed U_CORR's previous phase, so this arrival can
          // never put U_CORR two phases ahead of the issuer's parity wait.
          if (!(ok = mbar_wait_warp(bar(U_ODONE + i), (cum_p[i] + j - 1) & 1, wc))) break;
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
            // O_i holds the sum up to key tile j-1 (that product is done): rescale.
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < D / 16; ++cc) {
              uint32_t o[16];
              tmem_ld_x16(t_lane + L::tm_o(i) + cc * 16, o);
#pragma unroll
              for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_st_x16(t_lane + L::tm_o(i) + cc * 16, o);
            }
            tmem_st_wait();
          }
          tc_fence_before();
          mbar_arrive_warp(bar(U_CORR + i));
        }
      }
      // Epilogue: O_i / l -> 16-bit -> swizzled staging over Q_i of this unit's set (no
      // product reads it any more once U_OLAST + i has completed) -> TMA store; logsumexp.
      const int set = u & 1;
#pragma unroll 1
      for (int i = 0; i < 2; ++i) {
        // Every product of the tile in this unit done (one phase per unit, waited for in
        // order: the per-step U_ODONE phases are not all observed here, and a parity wait
        // may only ever be one phase ahead of the barrier).
        const bool ok_i = ok && mbar_wait_warp(bar(U_FIN + i), u & 1, wc) &&
                          mbar_wait_warp(bar(U_OLAST + i), u & 1, wc);
        const int q0 = (2 * un.pr + i) * kTileM;
        if (ok_i) {
          tc_fence_after();
          const float mf = m_s[i * 128 + row];
          const float lf = l_s[i * 128 + row];
          const float inv_l = 1.f / lf;
          uint8_t* stage = smem + L::OFF_Q + (2 * set + i) * L::TILE;
#pragma unroll
          for (int cc = 0; cc < D / 16; ++cc) {
            uint32_t o[16];
            tmem_ld_x16(t_lane + L::tm_o(i) + cc * 16, o);
            uint32_t pkd[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              pkd[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const int ch = cc * 2 + q;
              uint4* dst = reinterpret_cast<uint4*>(stage + row * 128 + ((ch ^ (row & 7)) << 4));
              *dst = make_uint4(pkd[4 * q], pkd[4 * q + 1], pkd[4 * q + 2], pkd[4 * q + 3]);
            }
          }
          // O_i, m and l are read: the next unit may overwrite them.
          tc_fence_before();
          mbar_arrive_warp(bar(U_OFREE + i));
          // natural-log logsumexp of the scaled scores: (m + log2 l) * ln 2
          if (q0 + row < a.N) a.lse[static_cast<size_t>(un.bh) * a.N + q0 + row] = (mf + __log2f(lf)) * 0.69314718055994531f;
          fence_proxy_async_smem();
        }
        ok = ok && ok_i;
      }
      named_bar_sync(1, 128);
      if (warp == 12 && lane == 0) {
        if (ok && !*abort_flag) {
          for (int i = 0; i < 2; ++i)
            tma_store_3d(&a.tm_o, sb + L::OFF_Q + (2 * set + i) * L::TILE, 0, (2 * un.pr + i) * kTileM, un.bh);
          bulk_commit();
          bulk_wait_read_all();
        }
        mbar_arrive(bar(U_STFREE + set));  // the producer may load the unit after next's Q here
      }
      for (int i = 0; i < 2; ++i) {
        cum_p[i] += n_kv[i];
        cum_c[i] += n_kv[i] - 1;
      }
      if (ok) x = next_unit(u, ok);
      // the four warps leave together (the epilogue's named barriers count all of them)
      if (!named_bar_and(2, 128, ok && x >= 0)) break;
    }
    if (warp == 12 && lane == 0) bulk_wait_read_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TM_COLS);
  }
}

template <bool BF16>
cudaError_t launch_persist_t(const FwdArgs& a, cudaStream_t st) {
  auto k = fwd_persist_kernel<BF16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, PersistLayout::SMEM);
  if (e != cudaSuccess) return e;
  const int n_t = (a.N + kTileM - 1) / kTileM;
  if (n_t % 2 != 0) return cudaErrorInvalidValue;
  k<<<dim3((n_t / 2) * a.BH), kPThreads, PersistLayout::SMEM, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_persist(const FwdArgs& a, bool bf16, cudaStream_t s) {
  return bf16 ? launch_persist_t<true>(a, s) : launch_persist_t<false>(a, s);
}

}  // namespace attn
