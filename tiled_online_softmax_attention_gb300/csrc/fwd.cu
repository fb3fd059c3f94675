// fwd.cu -- forward attention kernel for sm_103a.
//
// One CTA computes two 128-row query tiles (Q0, Q1) of one (batch, head) and
// streams that head's K/V tiles through shared memory once for both (FA2 loop
// order: queries outer, keys inner; "FlashAttention hardware-aware analysis"
// (huaweicloud), section four, part 2).  Per key tile j and query tile i:
//
//   S_i   = Q_i K_j^T               tcgen05.mma, SMEM x SMEM -> TMEM (fp32)
//   m_new = max(m, rowmax S_i)      online-softmax recurrence (huaweicloud page,
//   P_i   = exp(S_i - m_new)        section two; "Understanding online softmax in
//   l     = l e^(m-m_new) + rowsum  Flash Attention from scratch", section 3.1),
//   O_i   = O_i e^(m-m_new) + P_i V_j   in the base-2 domain (exponents are
//                                   scale*log2(e)*S, so exp becomes ex2)
//
// O_i stays in tensor memory for the whole loop and is divided by l once at the
// end (deferred normalisation; hotelren.com FA1/FA2 comparison, section 2.1.2).
// The row logsumexp m + ln l is saved for the backward pass.  Nothing of size
// N x N ever leaves the SM.
//
// The two query tiles exist so that the tensor core always has work: while the
// softmax warps of tile 0 turn S_0 into P_0, the MMA warp runs P_1 V and
// Q_1 K^T for tile 1, and the other way round.  The MMA issue order per key
// tile is PV_0(j), S_0(j+1), PV_1(j), S_1(j+1).  S_i(j+1) overwrites the
// columns P_i(j) was read from by PV_i(j); the two products are issued by one
// thread in that order and the tensor core executes one thread's MMAs in order.
//
// Rescaling is lazy: a row's reference maximum only moves when the new row max
// exceeds it by more than 2^8 (in exp2 units), so exponentials stay <= 256 and
// the O rescale (a TMEM read-modify-write) is skipped on almost every tile.
// Because O, l and the final logsumexp all use the same reference maximum, the
// result is exact; only the moment of rescaling changes.
//
// Warp roles (512 threads, four warpgroups):
//   warpgroup 0  warp 0 TMA producer (Q0, Q1 once; then K_j, V_j into a ring),
//                warp 1 TMEM owner and MMA issuer (the warp runs the loop, one elected
//                lane issues each product)
//   warpgroup 1  softmax of query tile 0 (thread r owns row r = TMEM lane r)
//   warpgroup 2  softmax of query tile 1
//   warpgroup 3  correction (O rescale when a reference max moves) and the
//                epilogue of both tiles (O / l -> 16-bit -> swizzled SMEM -> TMA store)
//
// Tensor memory (512 columns): S_0 at 0, S_1 at 128 (fp32; P_i is written as
// 16-bit pairs over the first 64 columns of S_i), O_0 at 256, O_1 at 256 + d.
//
// Causal: key tiles wholly above the diagonal are never loaded (the huaweicloud
// page's section five, part 3); only diagonal and ragged tiles are masked.  The
// grid is walked in groups of heads, longest query pairs first (work_item).
#include "common.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

template <int D, bool FP8>
struct FwdLayout {
  static constexpr int ELEM = FP8 ? 1 : 2;           // input bytes per element
  static constexpr int KB_IN = D * ELEM / 128;       // 128-byte blocks per input row
  static constexpr int KB = D / 64;                  // 128-byte blocks per 16-bit output row
  static constexpr int TILE = kTileM * D * ELEM;     // bytes of one 128-row input tile
  static constexpr int OTILE = kTileM * D * 2;       // bytes of one 128-row 16-bit output tile
  static constexpr int BLK = kTileM * 128;           // bytes of one 128-row x 128-byte block
  static constexpr int NSLOT = (TILE == 32768) ? 4 : 8;  // K/V ring entries, one tile each
  static constexpr int OFF_Q = 0;                    // Q_i at i * OTILE (later O_i's staging)
  static constexpr int OFF_KV = 2 * OTILE;
  static constexpr int OFF_AUX = OFF_KV + NSLOT * TILE;
  static constexpr int AUX_BAR = 0;                  // up to 64 mbarriers
  static constexpr int AUX_ALPHA = 512;              // float[2][128]: rescale factor per row
  static constexpr int AUX_M = AUX_ALPHA + 1024;     // float[2][128]: final reference max
  static constexpr int AUX_L = AUX_M + 1024;         // float[2][128]: final row sum
  static constexpr int AUX_MISC = AUX_L + 1024;      // abort flag, TMEM address
  static constexpr int AUX_BYTES = AUX_MISC + 64;
  static constexpr int SMEM = OFF_AUX + AUX_BYTES + 1024;  // + alignment slack
  static constexpr uint32_t TM_O = 256, TM_COLS = 512;
  static constexpr uint32_t tm_s(int i) { return 128u * i; }
  static constexpr uint32_t tm_o(int i) { return TM_O + D * i; }
  // d = 64: the O tiles end at column 384, and S/P buffer 2 (see ROT) takes 384 .. 511
  static constexpr uint32_t tm_sbuf(int b) { return b < 2 ? 128u * b : 384u; }
};

constexpr int kFwdThreads = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// E4M3 inputs.  The second product reads P as E4M3, so P is formed on a scale where the
// format is accurate: P~ = 2^(w - m + kPExp), with w = the log2-domain score plus
// log2 of its key block's V scale (the V scale is folded into P, see the softmax) and
// m the row's reference max of w.  kPExp is an integer, so the entry at the reference
// max is exactly 2^6 and every entry within 2^-12 of it is a normal E4M3 number
// (relative rounding error <= 2^-4); the reference max moves when exceeded by more than
// 2^2.5, so P~ <= 2^8.5 < 448, the largest E4M3 value.
constexpr float kRescaleThresholdFp8 = 2.5f;
constexpr float kPExp = 6.0f;

enum : int {
  B_Q = 0,         // + tile
  B_SFULL = 2,     // + tile: S_i computed (MMA commit)
  B_PFULL = 4,     // + tile: P_i written (softmax warpgroup) and, but with ROT, O_i rescaled
                   //   for it (correction warpgroup): the one hand-off P_i V_j waits for
  B_STAT = 6,      // + tile: rescale factors of this key tile published (softmax warpgroup)
  B_CORR = 8,      // + tile: O_i rescaled if needed (correction warpgroup; ROT only)
  B_ODONE = 10,    // + tile: P_i V_j done (MMA commit)
  B_FIN = 12,      // + tile: final m, l published (softmax warpgroup)
  B_DRAIN = 14,
  B_SFULL2 = 15,   // S/P buffer 2 computed (d = 64, ROT)
  B_KVFULL = 16,   // + slot
  B_KVEMPTY = 24,  // + slot
  B_COUNT = 32
};

// FP8: Q, K, V are E4M3 with one float32 scale per 128-row block of each head (FP8 with
// per-block scale factors, huaweicloud page, section four, part 3); S = Q8 K8^T runs on
// kind::f8f6f4, the per-tile factor q_scale * k_scale joins the softmax scale, and P~ V8
// runs on kind::f8f6f4 with P~ in E4M3.  The output stays 16-bit.
//
// DROP: dropout on the probabilities ("Understanding FlashAttention, Part 2", section 2.4
// names it): P(i, j) is kept iff byte j mod 16 of Philox4x32-10 at counter
// (j / 16, i, bh, 0), keyed by the seed, is >= a.drop_t; the row sum l keeps every
// probability (dropout follows the softmax) and the epilogue scales O by
// 256 / (256 - drop_t).  With packed sequences i and j are positions within the
// sequence and bh = b * H + h, so a packed batch draws the padded batch's mask.
//
// VARLEN: variable-length packed sequences ([tokens][H][d] with offsets): the CTA reads
// its sequence's token range, loads tiles at (column, head, token) coordinates, masks
// with the sequence's own lengths and writes O rows with plain stores, so that a
// partial last tile never touches the next sequence's rows.
//
// SPLIT: the CTA covers one of a.n_splits contiguous ranges of the pair's key tiles and
// writes its range's normalised partial O (fp32) and logsumexp instead of the output;
// merge_kernel combines the ranges with the two-block merge of the huaweicloud page's
// section two.  With VARLEN too, the partials sit in the packed layout ([split][token]
// [head]), and a degenerate sequence's ranges are all empty (lse = -inf).
// ROT (d = 64, whole pairs): the two O tiles take only 128 tensor-memory columns, so S/P
// has three 128-column buffers instead of one per tile.  S_i(j) goes to buffer
// (2 j + i) mod 3; S_0(j+1) then lands in the buffer P_1(j-1) was read from and can be
// issued before PV_0(j), and S_1(j+1) in the buffer of P_0(j), right after PV_0(j).  The
// MMA order per key tile becomes S_0(j+1), PV_0(j), S_1(j+1), PV_1(j): a query tile's
// next scores are ready when its softmax finishes the current tile, instead of waiting
// for the current tile's P V and the next Q K^T (at d = 64 those products are short and
// the chain S -> P -> PV -> S set the pace).
// The CTA's body; PAD: its pair's second query tile lies wholly past the last query
// (a sequence of an odd number of tiles, or a few queries against many keys), so only
// tile 0 runs.  `a` is the kernel's __grid_constant__ parameter.
template <int D, bool BF16, bool SPLIT, bool FP8, bool DROP, bool VARLEN, bool PAD>
__device__ __forceinline__ void fwd_body(const FwdArgs& a) {
  static_assert(!(FP8 && SPLIT) && (!FP8 || D == 128), "E4M3 inputs: d = 128, no split");
  static_assert(!DROP || (!FP8 && !SPLIT), "dropout: 16-bit inputs, no split");
  static_assert(!VARLEN || !FP8, "packed sequences: 16-bit inputs");
  using L = FwdLayout<D, FP8>;
  constexpr bool ROT = (D == 64) && !FP8 && !PAD;
  // S/P buffer of query tile i at key step j, its completion barrier and the parity of
  // its use (the number of earlier S products into the same buffer, mod 2)
  auto sbuf = [](int i, int j) -> int { return ROT ? (2 * j + i) % 3 : i; };
  auto sfull_bar = [](int b) -> int { return b < 2 ? B_SFULL + b : B_SFULL2; };
  auto sfull_parity = [](int i, int j) -> uint32_t {
    return ROT ? static_cast<uint32_t>(((2 * j + i) / 3) & 1) : static_cast<uint32_t>(j & 1);
  };
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  uint8_t* aux = smem + L::OFF_AUX;
  const uint32_t bars = sb + L::OFF_AUX + L::AUX_BAR;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * i; };
  float* alpha_s = reinterpret_cast<float*>(aux + L::AUX_ALPHA);
  float* m_s = reinterpret_cast<float*>(aux + L::AUX_M);
  float* l_s = reinterpret_cast<float*>(aux + L::AUX_L);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(aux + L::AUX_MISC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aux + L::AUX_MISC + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_t = (a.N + kTileM - 1) / kTileM;    // query tiles
  const int n_tk = (a.Nk + kTileN - 1) / kTileN;  // key tiles
  const int n_pairs = (n_t + 1) / 2;
  const int split = SPLIT ? static_cast<int>(blockIdx.x) % a.n_splits : 0;
  const WorkItem wi = work_item(static_cast<int>(blockIdx.x) / (SPLIT ? a.n_splits : 1), a.BH, n_pairs);
  const int bh = wi.bh;
  const int pr = n_pairs - 1 - wi.rank;  // longest causal pair first
  // Lengths this CTA works with: one sequence's in VARLEN mode, else the kernel
  // parameters themselves (read through accessors so that the plain kernel keeps using
  // the parameters directly; holding them in registers measured 4 % slower).  Plus where
  // the rows sit: the head and the first query / key token of the sequence.
  int vN = 0, vNk = 0, vcofs = 0;
  int hh = 0, tq0 = 0, tk0 = 0;
  if constexpr (VARLEN) {
    // The offsets are the caller's; seq_view clamps them so that a malformed table
    // cannot send a store outside o or lse.
    const SeqView sv = seq_view(a, bh);
    hh = sv.hh;
    tq0 = sv.tq0;
    tk0 = sv.tk0;
    vN = sv.N;
    vNk = sv.Nk;
    vcofs = sv.cofs;
    const int N = vN;
    if (2 * pr * kTileM >= N) return;  // this pair lies past the sequence's end (whole CTA)
    if (sv.degenerate) {
      // No key at all, or causal rows that would see none: O = 0 and lse = -inf for the
      // pair's rows (documented), without starting the pipeline.
      for (int r = threadIdx.x; r < 2 * kTileM; r += blockDim.x) {
        const int gr = 2 * pr * kTileM + r;
        if (gr >= N) continue;
        if constexpr (SPLIT) {  // every range is empty: the merge writes O = 0, lse = -inf
          a.part_lse[(static_cast<size_t>(split) * a.Tq + tq0 + gr) * a.H + hh] = -INFINITY;
          continue;
        }
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.o) + ((static_cast<size_t>(tq0 + gr) * a.H + hh) * D) * 2);
        for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
        a.lse[static_cast<size_t>(hh) * a.Tq + tq0 + gr] = -INFINITY;
      }
      return;
    }
  }
  auto N_ = [&]() -> int {
    if constexpr (VARLEN) return vN; else return a.N;
  };
  auto Nk_ = [&]() -> int {
    if constexpr (VARLEN) return vNk; else return a.Nk;
  };
  auto cofs_ = [&]() -> int {
    if constexpr (VARLEN) return vcofs; else return a.cofs;
  };
  // TMA coordinates of query row r / key row r: (row, bh) or, packed, (head, token)
  auto qc1 = [&](int r) { return VARLEN ? hh : r; };
  auto qc2 = [&](int r) { return VARLEN ? tq0 + r : bh; };
  auto kc1 = [&](int r) { return VARLEN ? hh : r; };
  auto kc2 = [&](int r) { return VARLEN ? tk0 + r : bh; };
  // Split-KV partial row of query row r (part_lse index; part_o rows hold D floats):
  // [split][BH][N], or packed [split][Tq][H] like O itself.
  auto prow_of = [&](int r) -> size_t {
    if constexpr (VARLEN)
      return (static_cast<size_t>(split) * a.Tq + tq0 + r) * a.H + hh;
    else
      return (static_cast<size_t>(split) * a.BH + bh) * a.N + r;
  };
  int n_kv[2];  // key tiles each query tile visits, starting at key tile kv0
#pragma unroll
  for (int i = 0; i < 2; ++i) n_kv[i] = visible_key_tiles(2 * pr + i, Nk_(), a.causal, cofs_());
  int kv0 = 0;
  if constexpr (SPLIT) {
    // Ranges cut tile 0's visible tiles evenly; tile 1's one extra causal tile joins the
    // last range.  A pair with fewer tiles than ranges leaves the surplus ranges empty.
    const int ns = min(a.n_splits, n_kv[0]);
    if (split >= ns) {
      for (int r = threadIdx.x; r < 2 * kTileM; r += blockDim.x) {
        const int grow = 2 * pr * kTileM + r;
        if (grow < N_()) a.part_lse[prow_of(grow)] = -INFINITY;
      }
      return;
    }
    kv0 = split * n_kv[0] / ns;
    const int hi0 = (split + 1) * n_kv[0] / ns;
    n_kv[1] = (split == ns - 1 ? n_kv[1] : hi0) - kv0;
    n_kv[0] = hi0 - kv0;
  }
  if constexpr (PAD) n_kv[1] = 0;  // the padding tile visits no key tile
  const int n_steps = PAD ? n_kv[0] : n_kv[1];  // key tiles the pair visits (n_kv[1] >= n_kv[0])

  // Warpgroup hand-offs arrive once per warp for 16-bit tiles and once per thread for
  // E4M3 tiles: each measured about 1 % faster than the other form on its own path.
  constexpr uint32_t kWgArrivals = FP8 ? 128 : 4;
  auto arrive_wg = [&](uint32_t b) {
    if constexpr (FP8)
      mbar_arrive(b);
    else
      mbar_arrive_warp(b);
  };
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_Q + i), 1);
      mbar_init(bar(B_SFULL + i), 1);
      mbar_init(bar(B_PFULL + i), ROT ? kWgArrivals : 2 * kWgArrivals);
      mbar_init(bar(B_STAT + i), kWgArrivals);
      mbar_init(bar(B_CORR + i), kWgArrivals);
      mbar_init(bar(B_ODONE + i), 1);
      mbar_init(bar(B_FIN + i), kWgArrivals);
    }
    mbar_init(bar(B_DRAIN), 1);
    if (ROT) mbar_init(bar(B_SFULL2), 1);
    for (int s = 0; s < L::NSLOT; ++s) {
      mbar_init(bar(B_KVFULL + s), 1);
      mbar_init(bar(B_KVEMPTY + s), 1);
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
      for (int i = 0; i < 2; ++i) {
        mbar_arrive_expect_tx(bar(B_Q + i), L::TILE);
        for (int kb = 0; kb < L::KB_IN; ++kb)
          tma_load_3d(sb + L::OFF_Q + i * L::OTILE + kb * L::BLK, &a.tm_q, bar(B_Q + i), kb * (128 / L::ELEM),
                      qc1((2 * pr + i) * kTileM), qc2((2 * pr + i) * kTileM));
      }
      const int n_loads = 2 * n_steps;  // K_j, V_j alternately
      int issued = 0;
      for (int ld = 0; ld < n_loads; ++ld) {
        const int s = ld % L::NSLOT;
        if (ld >= L::NSLOT && !mbar_wait(bar(B_KVEMPTY + s), ((ld / L::NSLOT) - 1) & 1, wc)) break;
        const CUtensorMap* m = (ld & 1) ? &a.tm_v : &a.tm_k;
        mbar_arrive_expect_tx(bar(B_KVFULL + s), L::TILE);
        for (int kb = 0; kb < L::KB_IN; ++kb)
          tma_load_3d(sb + L::OFF_KV + s * L::TILE + kb * L::BLK, m, bar(B_KVFULL + s), kb * (128 / L::ELEM),
                      kc1((kv0 + (ld >> 1)) * kTileN), kc2((kv0 + (ld >> 1)) * kTileN));
        issued = ld + 1;
      }
      // Let every copy this thread started land before the CTA can exit.
      mbar_wait(bar(B_Q + 0), 0, wc);
      mbar_wait(bar(B_Q + 1), 0, wc);
      for (int ld = (issued > L::NSLOT ? issued - L::NSLOT : 0); ld < issued; ++ld)
        mbar_wait(bar(B_KVFULL + ld % L::NSLOT), (ld / L::NSLOT) & 1, wc);
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer (the whole
      // warp runs it, one elected lane issues)
      constexpr uint32_t idesc_qk =
          FP8 ? idesc_e4m3(kTileM, kTileN, false, false) : idesc_f16(kTileM, kTileN, BF16, false, false);
      constexpr uint32_t idesc_pv = FP8 ? idesc_e4m3(kTileM, D, false, true) : idesc_f16(kTileM, D, BF16, false, true);
      auto full = [&](int ld) { return mbar_wait_warp(bar(B_KVFULL + ld % L::NSLOT), (ld / L::NSLOT) & 1, wc); };
      auto issue_s = [&](int i, int j) {
        const uint32_t qb = sb + L::OFF_Q + i * L::OTILE;
        const uint32_t kbase = sb + L::OFF_KV + ((2 * j) % L::NSLOT) * L::TILE;
        // One MMA per 32 bytes of the rows (K = 16 16-bit or 32 8-bit elements).
        const uint32_t d_s = FP8 ? tmem + L::tm_s(i) : tmem + L::tm_sbuf(sbuf(i, j));
        const uint32_t cb = bar(sfull_bar(sbuf(i, j)));
        if (elect_one_sync()) {
#pragma unroll
          for (int k = 0; k < D * L::ELEM / 32; ++k) {
            const uint32_t off = (k >> 2) * L::BLK + (k & 3) * 32;
            if constexpr (FP8)
              mma_ss_f8(d_s, sdesc_sw128(qb + off, 16, 1024), sdesc_sw128(kbase + off, 16, 1024), idesc_qk, k > 0 ? 1u : 0u);
            else
              mma_ss(d_s, sdesc_sw128(qb + off, 16, 1024), sdesc_sw128(kbase + off, 16, 1024), idesc_qk, k > 0 ? 1u : 0u);
          }
          tc_commit(cb);
        }
        __syncwarp();
      };
      auto issue_pv = [&](int i, int j) {
        const uint32_t vbase = sb + L::OFF_KV + ((2 * j + 1) % L::NSLOT) * L::TILE;
        // One MMA per 32 keys' bytes of P (8 TMEM columns); V advances 32 / ELEM key rows.
        const uint32_t a_p = FP8 ? tmem + L::tm_s(i) : tmem + L::tm_sbuf(sbuf(i, j));
        if (elect_one_sync()) {
#pragma unroll
          for (int k = 0; k < kTileN * L::ELEM / 32; ++k) {
            if constexpr (FP8)
              mma_ts_f8(tmem + L::tm_o(i), a_p + k * 8, sdesc_sw128(vbase + k * (4096 / L::ELEM), L::BLK, 1024), idesc_pv,
                        (j > 0 || k > 0) ? 1u : 0u);
            else
              mma_ts(tmem + L::tm_o(i), a_p + k * 8, sdesc_sw128(vbase + k * (4096 / L::ELEM), L::BLK, 1024), idesc_pv,
                     (j > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit(bar(B_ODONE + i));
        }
        __syncwarp();
      };
      constexpr bool has1 = !PAD;
      bool ok = mbar_wait_warp(bar(B_Q + 0), 0, wc) && full(0);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        ok = mbar_wait_warp(bar(B_Q + 1), 0, wc);
      }
      if (ok) {
        tc_fence_after();
        if (has1) issue_s(1, 0);
        tc_commit_w(bar(B_KVEMPTY + 0));
      }
      for (int j = 0; ROT && ok && j < n_steps; ++j) {
        // S_0(j+1) | PV_0(j) | S_1(j+1) | PV_1(j)  (see ROT above).  V(j) is waited for
        // before S_0(j+1) is issued, so that nothing stands between that product and the
        // wait for P_0(j): tile 0's softmax, which S_0(j+1) lets run on, cannot complete
        // P_0(j+1) first (B_PFULL two phases ahead of a parity wait).
        const bool k_next = j + 1 < n_steps;  // K(j+1) is read by S_1(j+1) at least
        if (!(ok = full(2 * j + 1))) break;
        if (k_next && !(ok = full(2 * j + 2))) break;
        if (j + 1 < n_kv[0]) {
          tc_fence_after();
          issue_s(0, j + 1);
        }
        if (j < n_kv[0]) {
          if (!(ok = mbar_wait_warp(bar(B_PFULL + 0), j & 1, wc) && (j == 0 || mbar_wait_warp(bar(B_CORR + 0), (j - 1) & 1, wc))))
            break;
          tc_fence_after();
          issue_pv(0, j);
        }
        if (k_next) {
          tc_fence_after();
          issue_s(1, j + 1);
          tc_commit_w(bar(B_KVEMPTY + (2 * j + 2) % L::NSLOT));
        }
        if (!(ok = mbar_wait_warp(bar(B_PFULL + 1), j & 1, wc) && (j == 0 || mbar_wait_warp(bar(B_CORR + 1), (j - 1) & 1, wc))))
          break;
        tc_fence_after();
        issue_pv(1, j);
        tc_commit_w(bar(B_KVEMPTY + (2 * j + 1) % L::NSLOT));
      }
      for (int j = 0; !ROT && ok && j < n_steps; ++j) {
        bool v_ready = false, k_next_ready = false;
        if (j < n_kv[0]) {
          if (!(ok = full(2 * j + 1) && mbar_wait_warp(bar(B_PFULL + 0), j & 1, wc)))
            break;
          v_ready = true;
          tc_fence_after();
          issue_pv(0, j);
          if (j + 1 < n_kv[0]) {
            if (!(ok = full(2 * j + 2))) break;
            k_next_ready = true;
            tc_fence_after();
            issue_s(0, j + 1);
          }
        }
        if (has1) {
          if (!(ok = (v_ready || full(2 * j + 1)) && mbar_wait_warp(bar(B_PFULL + 1), j & 1, wc)))
            break;
          tc_fence_after();
          issue_pv(1, j);
        }
        tc_commit_w(bar(B_KVEMPTY + (2 * j + 1) % L::NSLOT));
        if (j + 1 < n_steps) {
          if (has1) {  // (without tile 1, tile 0's S(j+1) above was the slot's last use)
            if (!(ok = k_next_ready || full(2 * j + 2))) break;
            tc_fence_after();
            issue_s(1, j + 1);
          }
          tc_commit_w(bar(B_KVEMPTY + (2 * j + 2) % L::NSLOT));
        }
      }
      // Drain: nothing may still write tensor memory when it is released.
      tc_commit_w(bar(B_DRAIN));
      mbar_wait_warp(bar(B_DRAIN), 0, wc);
    }
  } else if (wg <= 2) {
    // ------------------------------------------------------------ softmax of tile i
    setmaxnreg_inc<184>();
    const int i = wg - 1;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const int grow = (2 * pr + i) * kTileM + row;
    const uint32_t t_lane_s = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    float sl2 = a.scale_log2;
    float m = -INFINITY;  // reference max (scale*log2(e) units) used by the exponentials
    float l = 0.f;        // row sum of ex2(. - m)
    bool ok = true;
    // E4M3: block scales of this query tile and of the next key tile (loaded a tile ahead).
    float ks_next = 1.f, vs_next = 1.f;
    if constexpr (FP8) {
      const int qt = 2 * pr + i;  // the second tile of the last pair may lie past the end
      if (qt < n_t) sl2 *= a.q_scale[static_cast<size_t>(bh) * n_t + qt];
      if (n_kv[i] > 0) {
        ks_next = a.k_scale[static_cast<size_t>(bh) * n_tk + kv0];
        vs_next = a.v_scale[static_cast<size_t>(bh) * n_tk + kv0];
      }
    }
    for (int j = 0; j < n_kv[i]; ++j) {
      float tsc = sl2, gj = 0.f, inv_vs = 1.f;  // score factor; log2 and inverse of V's scale
      if constexpr (FP8) {
        tsc = sl2 * ks_next;
        gj = __log2f(vs_next);
        inv_vs = 1.f / vs_next;
        if (j + 1 < n_kv[i]) {
          ks_next = a.k_scale[static_cast<size_t>(bh) * n_tk + kv0 + j + 1];
          vs_next = a.v_scale[static_cast<size_t>(bh) * n_tk + kv0 + j + 1];
        }
      }
      // Dropout keep masks of this row's 128 keys, drawn while S is being computed:
      // keep[g] holds 0xFF in every byte (key 16g + 4q + b in byte b of word q) kept.
      uint32_t keep[8][4];
      if constexpr (DROP) {
        const uint32_t tt = a.drop_t * 0x01010101u;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          uint32_t w[4];
          philox4x32_10(static_cast<uint32_t>((kv0 + j) * (kTileN / 16) + g), static_cast<uint32_t>(grow),
                        static_cast<uint32_t>(bh), 0u, a.seed_lo, a.seed_hi, w);
#pragma unroll
          for (int q = 0; q < 4; ++q) keep[g][q] = __vcmpgeu4(w[q], tt);
        }
        if (a.keep_bits != nullptr && grow < N_()) {
          // The row's 128 decisions as four 32-key words for the backward: the top bit of
          // each 0x00 / 0xFF byte of keep[g][q] gathered by one multiply (bits 7, 15, 23, 31
          // land on 28..31 and nothing else reaches those bits).
          uint32_t* kb = a.keep_bits + (static_cast<size_t>(bh) * n_tk + kv0 + j) * 4 * a.bits_rows + grow;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            uint32_t word = 0;
#pragma unroll
            for (int gg = 0; gg < 2; ++gg)
#pragma unroll
              for (int q = 0; q < 4; ++q)
                word |= (((keep[2 * w + gg][q] & 0x80808080u) * 0x00204081u) >> 28) << (16 * gg + 4 * q);
            kb[static_cast<size_t>(w) * a.bits_rows] = word;
          }
        }
      }
      if (!mbar_wait_warp(bar(sfull_bar(sbuf(i, j))), sfull_parity(i, j), wc)) { ok = false; break; }
      tc_fence_after();
      const uint32_t t_s = t_lane_s + L::tm_sbuf(sbuf(i, j));
      float s[128];
      {
        // Four loads in flight, one wait: a TMEM load issued while the tensor core
        // runs the other tile's products takes several times its idle latency.
        uint32_t sr[128];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld_x32_async(t_s + 32 * q, sr + 32 * q);
        tmem_ld_wait(sr);
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
      }
      const int k0 = (kv0 + j) * kTileN;
      const bool tail = k0 + kTileN > Nk_();
      const bool diag = a.causal && (k0 + kTileN - 1 > (2 * pr + i) * kTileM + cofs_());
      if (tail || diag) {
        int lim = Nk_() - k0;                                   // keys past the end of the sequence
        if (a.causal) lim = min(lim, grow + cofs_() - k0 + 1);  // keys after this query
#pragma unroll
        for (int c = 0; c < kTileN; ++c)
          if (c >= lim) s[c] = -INFINITY;
      }
      // Row max: a tree for E4M3 tiles; one running chain for 16-bit tiles, where the
      // tree measured 2 % slower (the chain's latency hides behind the other tile's MMAs).
      float mx;
      if constexpr (FP8) {
        mx = rowmax128(s);
      } else {
        mx = s[0];
#pragma unroll
        for (int c = 1; c < kTileN; ++c) mx = fmaxf(mx, s[c]);
      }
      if constexpr (FP8)
        mx = mx * tsc + gj;  // tsc > 0: the max of the scaled scores, plus V's block term
      else
        mx *= tsc;
      // Move the reference max only when it is exceeded by more than the threshold.
      const float m_new = (mx - m > (FP8 ? kRescaleThresholdFp8 : kRescaleThreshold)) ? mx : m;
      const float alpha = (m_new == m) ? 1.f : ex2(m - m_new);  // 0 on the first tile
      if (j > 0) {
        alpha_s[i * 128 + row] = alpha;
        arrive_wg(bar(B_STAT + i));
      }
      m = m_new;
      const float m_use = (m == -INFINITY) ? 0.f : m;  // a row with nothing visible yet
      float rs = 0.f;  // row sum of this tile's exponentials
      if constexpr (FP8) {
        // P~ = 2^(S tsc + g_j - m + kPExp) carries V's block scale, so P~ V8 accumulates
        // the dequantised product; the row sum takes it out again (l = sum P~ / vscale_j),
        // and O / l is then the softmax average of the dequantised V rows.
        const float bias = gj + kPExp - m_use;
        uint32_t pk[32];
        const uint64_t tsc2 = f32x2_pack(tsc, tsc), bias2 = f32x2_pack(bias, bias);
        uint64_t acc2[2] = {0ull, 0ull};
#pragma unroll
        for (int c = 0; c < kTileN; c += 4) {
          float x0, x1, x2, x3;
          f32x2_unpack(f32x2_fma(f32x2_pack(s[c], s[c + 1]), tsc2, bias2), x0, x1);
          f32x2_unpack(f32x2_fma(f32x2_pack(s[c + 2], s[c + 3]), tsc2, bias2), x2, x3);
          const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
          acc2[0] = f32x2_add(acc2[0], f32x2_pack(p0, p1));
          acc2[1] = f32x2_add(acc2[1], f32x2_pack(p2, p3));
          pk[c / 4] = pack4_e4m3(p0, p1, p2, p3);
        }
        {
          float a0, a1, b0, b1;
          f32x2_unpack(acc2[0], a0, a1);
          f32x2_unpack(acc2[1], b0, b1);
          rs = (a0 + a1) + (b0 + b1);
        }
        l = fmaf(l, alpha, rs * inv_vs);
        tmem_st_x32(t_s, pk);
      } else {
        // The softmax warps are issue-bound here: the exponent arguments and the row sum
        // go through paired f32x2 instructions (two columns each, two running sums),
        // which measured 8-9 % faster for the whole kernel than the scalar forms.
        uint32_t pk[64];
        const uint64_t tsc2 = f32x2_pack(tsc, tsc), negm2 = f32x2_pack(-m_use, -m_use);
        uint64_t acc2[2] = {0ull, 0ull};  // (+0, +0) pairs
#pragma unroll
        for (int c = 0; c < kTileN; c += 2) {
          float x0, x1;
          f32x2_unpack(f32x2_fma(f32x2_pack(s[c], s[c + 1]), tsc2, negm2), x0, x1);
          const float p0 = ex2(x0);
          const float p1 = ex2(x1);
          acc2[(c / 2) & 1] = f32x2_add(acc2[(c / 2) & 1], f32x2_pack(p0, p1));
          pk[c / 2] = pack2<BF16>(p0, p1);
          if constexpr (DROP)  // both 16-bit halves: all ones if kept, zero if dropped
            pk[c / 2] &= __byte_perm(keep[c / 16][(c % 16) / 4], 0u, (c % 4) ? 0x3322u : 0x1100u);
        }
        {
          float a0, a1, b0, b1;
          f32x2_unpack(acc2[0], a0, a1);
          f32x2_unpack(acc2[1], b0, b1);
          rs = (a0 + a1) + (b0 + b1);
        }
        l = fmaf(l, alpha, rs);
        tmem_st_x64(t_s, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      arrive_wg(bar(B_PFULL + i));
    }
    if (ok) {
      // E4M3: l carries the factor 2^kPExp of P~; the logsumexp is m - kPExp + log2 l.
      m_s[i * 128 + row] = (m == -INFINITY) ? 0.f : (FP8 ? m - kPExp : m);
      l_s[i * 128 + row] = l;
      arrive_wg(bar(B_FIN + i));
    }
  } else {
    // ------------------------------------------------------------ correction + epilogue
    setmaxnreg_dec<80>();
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    bool ok = true;
    // Without ROT the correction arrives on B_PFULL for every step, the first one too
    // (nothing to rescale there), so that P_i V_j waits on one barrier; with ROT, S_i(j+1)
    // is issued before P_i V_j, so the softmax's next arrival could land in the phase the
    // correction has not yet reached, and the two hand-offs keep their own barriers.
    for (int j = ROT ? 1 : 0; ok && j < n_steps; ++j) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (j >= n_kv[i]) continue;
        if (j == 0) {
          arrive_wg(bar(B_PFULL + i));
          continue;
        }
        if (!(ok = mbar_wait_warp(bar(B_STAT + i), (j - 1) & 1, wc))) break;
        const float alpha = alpha_s[i * 128 + row];
        // With ROT every step waits for P_i V(j-1) first, rescaling or not: that product is
        // issued only once the issuer has consumed B_CORR's previous phase, so this arrival
        // can never put B_CORR two phases ahead of the issuer's parity wait (tile i's softmax,
        // running on ahead, would otherwise let the two arrivals land back to back).
        const bool rescale = __any_sync(0xffffffffu, alpha != 1.f);
        if (ROT || rescale)
          if (!(ok = mbar_wait_warp(bar(B_ODONE + i), (j - 1) & 1, wc))) break;
        if (rescale) {
          // O_i holds the sum up to key tile j-1 (that product is done): rescale.
          tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld_x32(t_lane + L::tm_o(i) + cc * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st_x32(t_lane + L::tm_o(i) + cc * 32, o);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        arrive_wg(bar(ROT ? B_CORR + i : B_PFULL + i));
      }
    }
    // Epilogue: O_i / l -> 16-bit -> swizzled staging over Q_i -> TMA store; logsumexp.
#pragma unroll 1
    for (int i = 0; i < 2; ++i) {
      if (PAD && i == 1) continue;  // the padding tile: nothing to store
      const bool ok_i = ok && mbar_wait_warp(bar(B_FIN + i), 0, wc) &&
                        mbar_wait_warp(bar(B_ODONE + i), (n_kv[i] - 1) & 1, wc);
      const int q0 = (2 * pr + i) * kTileM;
      if (SPLIT && ok_i) {
        tc_fence_after();
        const float mf = m_s[i * 128 + row];
        const float lf = l_s[i * 128 + row];
        const float inv_l = 1.f / lf;
        const size_t prow = prow_of(q0 + row);
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld_x32(t_lane + L::tm_o(i) + cc * 32, o);
          if (q0 + row < N_()) {
            float4* dst = reinterpret_cast<float4*>(a.part_o + prow * D + cc * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_float4(__uint_as_float(o[4 * q]) * inv_l, __uint_as_float(o[4 * q + 1]) * inv_l,
                                   __uint_as_float(o[4 * q + 2]) * inv_l, __uint_as_float(o[4 * q + 3]) * inv_l);
          }
        }
        if (q0 + row < N_()) a.part_lse[prow] = (mf + __log2f(lf)) * 0.69314718055994531f;
      }
      if (!SPLIT && ok_i) {
        tc_fence_after();
        const float mf = m_s[i * 128 + row];
        const float lf = l_s[i * 128 + row];
        const float inv_l = (DROP ? a.drop_scale : 1.f) / lf;
        uint8_t* stage = smem + L::OFF_Q + i * L::OTILE;  // Q_i is no longer read
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld_x32(t_lane + L::tm_o(i) + cc * 32, o);
          uint32_t pkd[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pkd[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
          if constexpr (VARLEN) {  // this row of this sequence, straight to global memory
            if (q0 + row < N_()) {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.o) +
                                                    ((static_cast<size_t>(tq0 + q0 + row) * a.H + hh) * D + cc * 32) * 2);
#pragma unroll
              for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pkd[4 * q], pkd[4 * q + 1], pkd[4 * q + 2], pkd[4 * q + 3]);
            }
          } else {
            const int kb = (cc * 32) / 64;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int ch = ((cc * 32) % 64) / 8 + q;
              uint4* dst = reinterpret_cast<uint4*>(stage + kb * L::BLK + row * 128 + ((ch ^ (row & 7)) << 4));
              *dst = make_uint4(pkd[4 * q], pkd[4 * q + 1], pkd[4 * q + 2], pkd[4 * q + 3]);
            }
          }
        }
        // natural-log logsumexp of the scaled scores: (m + log2 l) * ln 2
        if (q0 + row < N_()) {
          const size_t li = VARLEN ? static_cast<size_t>(hh) * a.Tq + tq0 + q0 + row : static_cast<size_t>(bh) * N_() + q0 + row;
          a.lse[li] = (mf + __log2f(lf)) * 0.69314718055994531f;
        }
        fence_proxy_async_smem();
      }
      ok = ok && ok_i;
      named_bar_sync(1, 128);
      if (!SPLIT && !VARLEN && warp == 12 && lane == 0 && ok_i && !*abort_flag && q0 < N_()) {
        for (int kb = 0; kb < L::KB; ++kb)
          tma_store_3d(&a.tm_o, sb + L::OFF_Q + i * L::OTILE + kb * L::BLK, kb * 64, q0, bh);
        bulk_commit();
      }
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

template <int D, bool BF16, bool SPLIT, bool FP8, bool DROP, bool VARLEN>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_kernel(const __grid_constant__ FwdArgs a) {
  // Which body this CTA runs: the same pair and length the body derives.
  const int n_pairs = ((a.N + kTileM - 1) / kTileM + 1) / 2;
  const WorkItem wi = work_item(static_cast<int>(blockIdx.x) / (SPLIT ? a.n_splits : 1), a.BH, n_pairs);
  const int pr = n_pairs - 1 - wi.rank;
  int N = a.N;
  if constexpr (VARLEN) N = seq_view(a, wi.bh).N;
  if ((2 * pr + 1) * kTileM >= N)
    fwd_body<D, BF16, SPLIT, FP8, DROP, VARLEN, true>(a);
  else
    fwd_body<D, BF16, SPLIT, FP8, DROP, VARLEN, false>(a);
}

template <int D, bool BF16, bool SPLIT, bool FP8 = false, bool DROP = false, bool VARLEN = false>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t st) {
  using L = FwdLayout<D, FP8>;
  auto k = fwd_kernel<D, BF16, SPLIT, FP8, DROP, VARLEN>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  const int n_t = (a.N + kTileM - 1) / kTileM;
  const int n_pairs = (n_t + 1) / 2;
  k<<<dim3(n_pairs * a.BH * (SPLIT ? a.n_splits : 1)), kFwdThreads, L::SMEM, st>>>(a);
  return cudaGetLastError();
}

// Merge of the split-KV partials, one warp per row: M = max_s lse_s,
// O = sum_s e^(lse_s - M) O_s / sum_s e^(lse_s - M), lse = M + ln sum_s e^(lse_s - M);
// a row whose ranges are all empty (a degenerate packed sequence) gets O = 0, lse = -inf.
// Rows are (bh, query) or, VARLEN, (token, head) of the packed layout; tokens outside
// cu_q[0] .. cu_q[B] belong to no sequence and are left untouched.
template <int D, bool BF16, bool VARLEN = false>
__global__ void __launch_bounds__(256) merge_kernel(const __grid_constant__ FwdArgs a) {
  constexpr int PER = D / 32;  // columns per lane
  const int lane = threadIdx.x & 31;
  const int64_t rows = VARLEN ? static_cast<int64_t>(a.Tq) * a.H : static_cast<int64_t>(a.BH) * a.N;
  const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (r >= rows) return;
  if constexpr (VARLEN) {
    const int64_t tok = r / a.H;
    const int B = a.BH / a.H;
    if (tok < min(max(a.cu_q[0], 0), a.Tq) || tok >= min(max(a.cu_q[B], 0), a.Tq)) return;
  }
  float mx = -INFINITY;
  for (int s = 0; s < a.n_splits; ++s) mx = fmaxf(mx, a.part_lse[s * rows + r]);
  float acc[PER];
#pragma unroll
  for (int c = 0; c < PER; ++c) acc[c] = 0.f;
  float den = 0.f;
  for (int s = 0; s < a.n_splits; ++s) {
    const float ls = a.part_lse[s * rows + r];
    if (ls == -INFINITY) continue;  // an empty range contributes nothing
    const float wgt = __expf(ls - mx);
    den += wgt;
    const float* src = a.part_o + (s * rows + r) * D + lane * PER;
    if constexpr (PER == 8) {
      const float4 v0 = *reinterpret_cast<const float4*>(src), v1 = *reinterpret_cast<const float4*>(src + 4);
      const float vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[c] = fmaf(wgt, vv[c], acc[c]);
    } else if constexpr (PER == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      acc[0] = fmaf(wgt, v.x, acc[0]);
      acc[1] = fmaf(wgt, v.y, acc[1]);
      acc[2] = fmaf(wgt, v.z, acc[2]);
      acc[3] = fmaf(wgt, v.w, acc[3]);
    } else {
      const float2 v = *reinterpret_cast<const float2*>(src);
      acc[0] = fmaf(wgt, v.x, acc[0]);
      acc[1] = fmaf(wgt, v.y, acc[1]);
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  uint32_t pk[PER / 2];
#pragma unroll
  for (int c = 0; c < PER; c += 2) pk[c / 2] = pack2<BF16>(acc[c] * inv, acc[c + 1] * inv);
  uint8_t* dst = static_cast<uint8_t*>(a.o) + (r * D + lane * PER) * 2;
  if constexpr (PER == 8)
    *reinterpret_cast<uint4*>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  else if constexpr (PER == 4)
    *reinterpret_cast<uint2*>(dst) = make_uint2(pk[0], pk[1]);
  else
    *reinterpret_cast<uint32_t*>(dst) = pk[0];
  if (lane == 0) {
    const int64_t li = VARLEN ? (r % a.H) * a.Tq + r / a.H : r;  // packed lse is [H][Tq]
    a.lse[li] = den > 0.f ? mx + __logf(den) : -INFINITY;
  }
}

template <int D, bool BF16, bool VARLEN = false>
cudaError_t launch_split_t(const FwdArgs& a, cudaStream_t st) {
  cudaError_t e;
  if constexpr (D == 256)
    e = launch_fwd256_split(a, BF16, VARLEN, st);  // the partials of fwd256.cu's kernel
  else
    e = launch_fwd_t<D, BF16, true, false, false, VARLEN>(a, st);
  if (e != cudaSuccess) return e;
  const int64_t rows = VARLEN ? static_cast<int64_t>(a.Tq) * a.H : static_cast<int64_t>(a.BH) * a.N;
  merge_kernel<D, BF16, VARLEN><<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, int d, bool bf16, cudaStream_t s) {
  if (d == 128) return bf16 ? launch_fwd_t<128, true, false>(a, s) : launch_fwd_t<128, false, false>(a, s);
  return bf16 ? launch_fwd_t<64, true, false>(a, s) : launch_fwd_t<64, false, false>(a, s);
}

cudaError_t launch_fwd_split(const FwdArgs& a, int d, bool bf16, cudaStream_t s) {
  if (d == 256) return bf16 ? launch_split_t<256, true>(a, s) : launch_split_t<256, false>(a, s);
  if (d == 128) return bf16 ? launch_split_t<128, true>(a, s) : launch_split_t<128, false>(a, s);
  return bf16 ? launch_split_t<64, true>(a, s) : launch_split_t<64, false>(a, s);
}

cudaError_t launch_fwd_varlen_split(const FwdArgs& a, int d, bool bf16, cudaStream_t s) {
  if (d == 256) return bf16 ? launch_split_t<256, true, true>(a, s) : launch_split_t<256, false, true>(a, s);
  if (d == 128) return bf16 ? launch_split_t<128, true, true>(a, s) : launch_split_t<128, false, true>(a, s);
  return bf16 ? launch_split_t<64, true, true>(a, s) : launch_split_t<64, false, true>(a, s);
}

cudaError_t launch_fwd_dropout(const FwdArgs& a, int d, bool bf16, cudaStream_t s) {
  if (d == 128)
    return bf16 ? launch_fwd_t<128, true, false, false, true>(a, s) : launch_fwd_t<128, false, false, false, true>(a, s);
  return bf16 ? launch_fwd_t<64, true, false, false, true>(a, s) : launch_fwd_t<64, false, false, false, true>(a, s);
}

// a.drop_t > 0 selects the dropout kernels.
cudaError_t launch_fwd_varlen(const FwdArgs& a, int d, bool bf16, cudaStream_t s) {
  if (a.drop_t > 0) {
    if (d == 128)
      return bf16 ? launch_fwd_t<128, true, false, false, true, true>(a, s)
                  : launch_fwd_t<128, false, false, false, true, true>(a, s);
    return bf16 ? launch_fwd_t<64, true, false, false, true, true>(a, s)
                : launch_fwd_t<64, false, false, false, true, true>(a, s);
  }
  if (d == 128)
    return bf16 ? launch_fwd_t<128, true, false, false, false, true>(a, s)
                : launch_fwd_t<128, false, false, false, false, true>(a, s);
  return bf16 ? launch_fwd_t<64, true, false, false, false, true>(a, s)
              : launch_fwd_t<64, false, false, false, false, true>(a, s);
}

cudaError_t launch_fwd_fp8(const FwdArgs& a, int d, bool bf16_out, cudaStream_t s) {
  if (d != 128) return cudaErrorInvalidValue;
  return bf16_out ? launch_fwd_t<128, true, false, true>(a, s) : launch_fwd_t<128, false, false, true>(a, s);
}

}  // namespace attn
