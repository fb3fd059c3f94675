// fwd256.cu -- forward attention kernel for head dimension 256 (sm_103a).
//
// The same computation as fwd.cu (online softmax over 128-key tiles, O kept in tensor
// memory and divided by l once at the end, logsumexp saved; huaweicloud page, sections
// two and four; "Understanding online softmax in Flash Attention from scratch", section
// 3.1), for the head dimension 256 the huaweicloud page's section five, part 1 lists
// next to 64 and 128.
//
// At d = 256 one query tile's O takes 256 of the 512 tensor-memory columns, so a CTA
// owns one 128-row query tile instead of two.  The tensor core is kept busy by double-
// buffering S instead: while the softmax warps turn S(j) into P(j), the MMA warp runs
// P(j-1) V(j-1) and Q K(j+1)^T.  The MMA issue order is S(0), S(1), PV(0), S(2), PV(1),
// S(3), ...; S(j+2) overwrites the columns P(j) was read from by PV(j), issued just
// before it by the same thread (the tensor core executes one thread's MMAs in order).
// K and V tiles go through a two-slot ring in exactly that consumption order, so
// K(j+2) is fetched as soon as S(j+1) has read its slot.
//
// Warp roles (256 threads):
//   warpgroup 0  warp 0 TMA producer, warp 1 TMEM owner and MMA issuer (one lane)
//   warpgroup 1  softmax (thread r owns row r = TMEM lane r), the rare O rescale when a
//                row's reference max moves, and the epilogue
//
// Tensor memory: S buffers at columns 0 and 128 (fp32; P as 16-bit pairs over the first
// 64 columns of its buffer), O at 256..511.  Shared memory: Q (64 KB, later O's staging
// tile) and two 64 KB K/V slots.
#include "common.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int D256 = 256;
constexpr int kF256Threads = 256;
constexpr float kRescaleThreshold256 = 8.0f;  // log2 units, as in fwd.cu

struct F256Layout {
  static constexpr int KB = D256 / 64;                // 64-column (128-byte) blocks per row
  static constexpr int BLK = kTileM * 128;            // one 128-row x 64-column block
  static constexpr int TILE = kTileM * D256 * 2;      // 64 KB
  static constexpr int NSLOT = 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = TILE;
  static constexpr int OFF_AUX = OFF_KV + NSLOT * TILE;
  static constexpr int AUX_BAR = 0;                   // mbarriers
  static constexpr int AUX_MISC = 256;                // abort flag, TMEM address
  static constexpr int AUX_BYTES = AUX_MISC + 64;
  static constexpr int SMEM = OFF_AUX + AUX_BYTES + 1024;
  static constexpr uint32_t TM_O = 256, TM_COLS = 512;
};

// One S-full and one P-full barrier per S buffer: with S issued two tiles ahead, the
// softmax may finish P(j+1) before the MMA warp has seen P(j), so a single P barrier
// could complete two phases between two of the MMA warp's polls.  Per buffer, the next
// phase needs S(j+2), which the MMA warp issues only after it has seen P(j).
enum : int {
  F_Q = 0,
  F_SFULL = 1,   // + buffer: S in that buffer computed (MMA commit)
  F_PFULL = 3,   // + buffer: P written over that buffer (128 softmax arrivals)
  F_ODONE = 5,   // P V done (MMA commit)
  F_DRAIN = 6,
  F_KVFULL = 7,  // + slot
  F_KVEMPTY = 9, // + slot
  F_COUNT = 11
};

// VARLEN: variable-length packed sequences ([tokens][H][d], offsets cu_q, cu_k), as in
// fwd.cu: the CTA reads its sequence's token range, loads tiles at (column, head, token)
// coordinates, masks with the sequence's own lengths and writes O rows with plain stores.
// DROP: dropout on the probabilities with fwd.cu's keep rule (key j of query i in head bh
// kept iff byte j % 16 of Philox((j / 16, i, bh, 0), seed) is >= drop_t); l sums every
// probability and the kept ones are scaled by drop_scale at the end.
// SPLIT: as in fwd.cu, the CTA covers one of a.n_splits contiguous ranges of its query
// tile's visible key tiles and writes the range's normalised partial O (fp32) and
// logsumexp for the merge kernel; a range past the tile's key tiles writes lse = -inf
// (with VARLEN: partials in the packed layout, every range of a degenerate sequence empty).
template <bool BF16, bool VARLEN, bool DROP, bool SPLIT>
__global__ void __launch_bounds__(kF256Threads, 1) fwd256_kernel(const __grid_constant__ FwdArgs a) {
  static_assert(!SPLIT || !DROP, "split-KV: no dropout");
  using L = F256Layout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  uint8_t* aux = smem + L::OFF_AUX;
  const uint32_t bars = sb + L::OFF_AUX + L::AUX_BAR;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(aux + L::AUX_MISC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aux + L::AUX_MISC + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_t = (a.N + kTileM - 1) / kTileM;
  const int split = SPLIT ? static_cast<int>(blockIdx.x) % a.n_splits : 0;
  const WorkItem wi = work_item<2>(static_cast<int>(blockIdx.x) / (SPLIT ? a.n_splits : 1), a.BH, n_t);
  const int bh = wi.bh;
  const int qt = n_t - 1 - wi.rank;  // longest causal tile first
  // Lengths and positions: the sequence's own (VARLEN), else the kernel parameters, read
  // through accessors so that the plain kernel keeps using the parameters directly.
  int vN = 0, vNk = 0, vcofs = 0, hh = 0, tq0 = 0, tk0 = 0;
  if constexpr (VARLEN) {
    const SeqView sv = seq_view(a, bh);
    vN = sv.N;
    vNk = sv.Nk;
    vcofs = sv.cofs;
    hh = sv.hh;
    tq0 = sv.tq0;
    tk0 = sv.tk0;
    const int N = vN;
    if (qt * kTileM >= N) return;  // this tile lies past the sequence's end (whole CTA)
    if (sv.degenerate) {           // no key, or causal rows that would see none: O = 0, lse = -inf
      for (int r = threadIdx.x; r < kTileM; r += blockDim.x) {
        const int gr = qt * kTileM + r;
        if (gr >= N) continue;
        if constexpr (SPLIT) {  // every range is empty: the merge writes O = 0, lse = -inf
          a.part_lse[(static_cast<size_t>(split) * a.Tq + tq0 + gr) * a.H + hh] = -INFINITY;
          continue;
        }
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.o) + ((static_cast<size_t>(tq0 + gr) * a.H + hh) * D256) * 2);
        for (int c = 0; c < D256 / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
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
  // Split-KV partial row of query row r (part_lse index; part_o rows hold 256 floats):
  // [split][BH][N], or packed [split][Tq][H] like O itself.
  auto prow_of = [&](int r) -> size_t {
    if constexpr (VARLEN)
      return (static_cast<size_t>(split) * a.Tq + tq0 + r) * a.H + hh;
    else
      return (static_cast<size_t>(split) * a.BH + bh) * a.N + r;
  };
  int n_kv = visible_key_tiles(qt, Nk_(), a.causal, cofs_());
  int kv0 = 0;  // first key tile of this CTA's range
  if constexpr (SPLIT) {
    const int ns = min(a.n_splits, n_kv);  // n_kv >= 1: every query sees key 0
    if (split >= ns) {                     // an empty range (whole CTA, before any barrier)
      for (int r = threadIdx.x; r < kTileM; r += blockDim.x) {
        const int grow = qt * kTileM + r;
        if (grow < N_()) a.part_lse[prow_of(grow)] = -INFINITY;
      }
      return;
    }
    kv0 = split * n_kv / ns;
    n_kv = (split + 1) * n_kv / ns - kv0;
  }
  // TMA coordinates of row r of Q (or K, V): (row, head-batch) or, packed, (head, token)
  auto qy = [&](int r) { return VARLEN ? hh : r; };
  auto qz = [&](int r) { return VARLEN ? tq0 + r : bh; };
  auto ky = [&](int r) { return VARLEN ? hh : r; };
  auto kz = [&](int r) { return VARLEN ? tk0 + r : bh; };

  if (threadIdx.x == 0) {
    mbar_init(bar(F_Q), 1);
    mbar_init(bar(F_SFULL + 0), 1);
    mbar_init(bar(F_SFULL + 1), 1);
    mbar_init(bar(F_PFULL + 0), 128);
    mbar_init(bar(F_PFULL + 1), 128);
    mbar_init(bar(F_ODONE), 1);
    mbar_init(bar(F_DRAIN), 1);
    for (int s = 0; s < L::NSLOT; ++s) {
      mbar_init(bar(F_KVFULL + s), 1);
      mbar_init(bar(F_KVEMPTY + s), 1);
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

  // The ring's load order equals the MMA warp's consumption order:
  // K0, K1, then V_j, K_{j+2} for j = 0, 1, ...  Item c uses slot c % 2.
  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    prefetch_tmap(&a.tm_q);
    prefetch_tmap(&a.tm_k);
    prefetch_tmap(&a.tm_v);
    prefetch_tmap(&a.tm_o);
    mbar_arrive_expect_tx(bar(F_Q), L::TILE);
    for (int kb = 0; kb < L::KB; ++kb)
      tma_load_3d(sb + L::OFF_Q + kb * L::BLK, &a.tm_q, bar(F_Q), kb * 64, qy(qt * kTileM), qz(qt * kTileM));
    int c = 0;
    bool ok = true;
    auto load = [&](const CUtensorMap* m, int tile) {
      const int s = c & 1;
      if (c >= 2 && !(ok = mbar_wait(bar(F_KVEMPTY + s), ((c >> 1) - 1) & 1, wc))) return;
      mbar_arrive_expect_tx(bar(F_KVFULL + s), L::TILE);
      for (int kb = 0; kb < L::KB; ++kb)
        tma_load_3d(sb + L::OFF_KV + s * L::TILE + kb * L::BLK, m, bar(F_KVFULL + s), kb * 64,
                    ky((kv0 + tile) * kTileN), kz((kv0 + tile) * kTileN));
      ++c;
    };
    load(&a.tm_k, 0);
    if (ok && n_kv > 1) load(&a.tm_k, 1);
    for (int j = 0; ok && j < n_kv; ++j) {
      load(&a.tm_v, j);
      if (ok && j + 2 < n_kv) load(&a.tm_k, j + 2);
    }
    // Let every copy this thread started land before the CTA can exit.
    mbar_wait(bar(F_Q), 0, wc);
    for (int i = (c > L::NSLOT ? c - L::NSLOT : 0); i < c; ++i) mbar_wait(bar(F_KVFULL + (i & 1)), (i >> 1) & 1, wc);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (the whole
    // warp runs it, one elected lane issues)
    constexpr uint32_t idesc_qk = idesc_f16(kTileM, kTileN, BF16, false, false);
    constexpr uint32_t idesc_pv = idesc_f16(kTileM, D256, BF16, false, true);
    int c = 0;
    auto full = [&]() -> bool { return mbar_wait_warp(bar(F_KVFULL + (c & 1)), (c >> 1) & 1, wc); };
    auto release = [&]() {
      tc_commit_w(bar(F_KVEMPTY + (c & 1)));
      ++c;
    };
    auto issue_s = [&](int buf) {
      const uint32_t kbase = sb + L::OFF_KV + (c & 1) * L::TILE;
#pragma unroll
      for (int k = 0; k < D256 / 16; ++k) {
        const uint32_t off = (k >> 2) * L::BLK + (k & 3) * 32;
        mma_ss_w(tmem + 128u * buf, sdesc_sw128(sb + L::OFF_Q + off, 16, 1024), sdesc_sw128(kbase + off, 16, 1024),
                 idesc_qk, k > 0 ? 1u : 0u);
      }
      tc_commit_w(bar(F_SFULL + buf));
      release();
    };
    auto issue_pv = [&](int j) {
      const uint32_t vbase = sb + L::OFF_KV + (c & 1) * L::TILE;
#pragma unroll
      for (int k = 0; k < kTileN / 16; ++k)
        mma_ts_w(tmem + L::TM_O, tmem + 128u * (j & 1) + k * 8, sdesc_sw128(vbase + k * 2048, L::BLK, 1024), idesc_pv,
                 (j > 0 || k > 0) ? 1u : 0u);
      tc_commit_w(bar(F_ODONE));
      release();
    };
    bool ok = mbar_wait_warp(bar(F_Q), 0, wc) && full();
    if (ok) {
      tc_fence_after();
      issue_s(0);
    }
    if (ok && n_kv > 1 && (ok = full())) {
      tc_fence_after();
      issue_s(1);
    }
    for (int j = 0; ok && j < n_kv; ++j) {
      if (!(ok = mbar_wait_warp(bar(F_PFULL + (j & 1)), (j >> 1) & 1, wc) && full())) break;
      tc_fence_after();
      issue_pv(j);
      if (j + 2 < n_kv) {
        if (!(ok = full())) break;
        tc_fence_after();
        issue_s(j & 1);
      }
    }
    // Drain: nothing may still write tensor memory when it is released.
    tc_commit_w(bar(F_DRAIN));
    mbar_wait_warp(bar(F_DRAIN), 0, wc);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax, rescale, epilogue
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const int grow = qt * kTileM + row;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float sl2 = a.scale_log2;
    float m = -INFINITY;  // reference max (scale*log2(e) units) used by the exponentials
    float l = 0.f;        // row sum of ex2(. - m)
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int buf = j & 1;
      // Keep masks of this row's 128 keys, drawn while S is being computed: keep[g][q]
      // has 0xFF in byte b if key 16g + 4q + b is kept.
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
      }
      if (!mbar_wait_warp(bar(F_SFULL + buf), (j >> 1) & 1, wc)) { ok = false; break; }
      tc_fence_after();
      float s[128];
      {
        uint32_t sr[128];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld_x32_async(t_lane + 128u * buf + 32 * q, sr + 32 * q);
        tmem_ld_wait(sr);
#pragma unroll
        for (int cc = 0; cc < 128; ++cc) s[cc] = __uint_as_float(sr[cc]);
      }
      const int k0 = (kv0 + j) * kTileN;
      const bool tail = k0 + kTileN > Nk_();
      const bool diag = a.causal && (k0 + kTileN - 1 > qt * kTileM + cofs_());
      if (tail || diag) {
        int lim = Nk_() - k0;                                   // keys past the end of the sequence
        if (a.causal) lim = min(lim, grow + cofs_() - k0 + 1);  // keys after this query
#pragma unroll
        for (int cc = 0; cc < kTileN; ++cc)
          if (cc >= lim) s[cc] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int cc = 1; cc < kTileN; ++cc) mx = fmaxf(mx, s[cc]);
      mx *= sl2;
      // Move the reference max only when it is exceeded by more than 2^8.
      const float m_new = (mx - m > kRescaleThreshold256) ? mx : m;
      const float alpha = (m_new == m) ? 1.f : ex2(m - m_new);  // 0 on the first tile
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O holds the sum up to key tile j-1: wait for that product, then rescale.
        if (!mbar_wait_warp(bar(F_ODONE), (j - 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < D256 / 32; ++cc) {
          uint32_t o[32];
          tmem_ld_x32(t_lane + L::TM_O + cc * 32, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st_x32(t_lane + L::TM_O + cc * 32, o);
        }
        tmem_st_wait();
      }
      m = m_new;
      const float m_use = (m == -INFINITY) ? 0.f : m;  // a row with nothing visible yet
      // Paired f32x2 arithmetic for the exponent arguments and the row sum (fewer
      // issue slots for the softmax warps; see the d <= 128 forward).
      uint32_t pk[64];
      const uint64_t sl2x2 = f32x2_pack(sl2, sl2), negm2 = f32x2_pack(-m_use, -m_use);
      uint64_t acc2[2] = {0ull, 0ull};
#pragma unroll
      for (int cc = 0; cc < kTileN; cc += 2) {
        float x0, x1;
        f32x2_unpack(f32x2_fma(f32x2_pack(s[cc], s[cc + 1]), sl2x2, negm2), x0, x1);
        const float p0 = ex2(x0);
        const float p1 = ex2(x1);
        acc2[(cc / 2) & 1] = f32x2_add(acc2[(cc / 2) & 1], f32x2_pack(p0, p1));
        pk[cc / 2] = pack2<BF16>(p0, p1);
        if constexpr (DROP)  // both 16-bit halves: all ones if kept, zero if dropped
          pk[cc / 2] &= __byte_perm(keep[cc / 16][(cc % 16) / 4], 0u, (cc % 4) ? 0x3322u : 0x1100u);
      }
      float rs;
      {
        float a0, a1, b0, b1;
        f32x2_unpack(acc2[0], a0, a1);
        f32x2_unpack(acc2[1], b0, b1);
        rs = (a0 + a1) + (b0 + b1);
      }
      l = fmaf(l, alpha, rs);
      tmem_st_x64(t_lane + 128u * buf, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(F_PFULL + buf));
    }
    // Epilogue: O / l -> 16-bit -> swizzled staging over Q -> TMA store; logsumexp.
    // It waits for the MMA warp's drain commit, not for a parity of F_ODONE: when the
    // last softmax ends, P(n-2) V may still be running (S(n-1) was issued before it), so
    // F_ODONE can be two phases short of the last product and a parity wait would alias.
    // (The rescale's wait above is safe: P(j-2) V precedes S(j), which softmax j has seen.)
    ok = ok && mbar_wait_warp(bar(F_DRAIN), 0, wc);
    if (SPLIT && ok) {  // this range's normalised partial O and logsumexp, one row per thread
      tc_fence_after();
      const float inv_l = 1.f / l;
      const size_t prow = prow_of(grow);
#pragma unroll 1
      for (int cc = 0; cc < D256 / 32; ++cc) {
        uint32_t o[32];
        tmem_ld_x32(t_lane + L::TM_O + cc * 32, o);
        if (grow < N_()) {
          float4* dst = reinterpret_cast<float4*>(a.part_o + prow * D256 + cc * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(__uint_as_float(o[4 * q]) * inv_l, __uint_as_float(o[4 * q + 1]) * inv_l,
                                 __uint_as_float(o[4 * q + 2]) * inv_l, __uint_as_float(o[4 * q + 3]) * inv_l);
        }
      }
      if (grow < N_()) a.part_lse[prow] = ((m == -INFINITY ? 0.f : m) + __log2f(l)) * 0.69314718055994531f;
    }
    if (!SPLIT && ok) {
      tc_fence_after();
      const float inv_l = (DROP ? a.drop_scale : 1.f) / l;
      uint8_t* stage = smem + L::OFF_Q;  // every S product has read Q by now
#pragma unroll 1
      for (int cc = 0; cc < D256 / 32; ++cc) {
        uint32_t o[32];
        tmem_ld_x32(t_lane + L::TM_O + cc * 32, o);
        uint32_t pkd[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pkd[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
        if constexpr (VARLEN) {  // this row of this sequence, straight to global memory
          if (grow < N_()) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.o) +
                                                  ((static_cast<size_t>(tq0 + grow) * a.H + hh) * D256 + cc * 32) * 2);
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
      if (grow < N_()) {  // natural-log logsumexp of the scaled scores: (m + log2 l) * ln 2
        const size_t li = VARLEN ? static_cast<size_t>(hh) * a.Tq + tq0 + grow : static_cast<size_t>(bh) * a.N + grow;
        a.lse[li] = ((m == -INFINITY ? 0.f : m) + __log2f(l)) * 0.69314718055994531f;
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128);
    if (!VARLEN && !SPLIT && warp == 4 && lane == 0 && ok && !*abort_flag) {
      for (int kb = 0; kb < L::KB; ++kb) tma_store_3d(&a.tm_o, sb + L::OFF_Q + kb * L::BLK, kb * 64, qt * kTileM, bh);
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

template <bool BF16, bool VARLEN = false, bool DROP = false, bool SPLIT = false>
cudaError_t launch_fwd256_t(const FwdArgs& a, cudaStream_t st) {
  auto k = fwd256_kernel<BF16, VARLEN, DROP, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, F256Layout::SMEM);
  if (e != cudaSuccess) return e;
  const int n_t = (a.N + kTileM - 1) / kTileM;
  k<<<dim3(n_t * a.BH * (SPLIT ? a.n_splits : 1)), kF256Threads, F256Layout::SMEM, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

// a.drop_t > 0 selects the dropout kernel.
cudaError_t launch_fwd256(const FwdArgs& a, bool bf16, cudaStream_t s) {
  if (a.drop_t > 0) return bf16 ? launch_fwd256_t<true, false, true>(a, s) : launch_fwd256_t<false, false, true>(a, s);
  return bf16 ? launch_fwd256_t<true>(a, s) : launch_fwd256_t<false>(a, s);
}

// The split-KV partials only (of a padded or, varlen, a packed batch); the caller runs
// the merge.
cudaError_t launch_fwd256_split(const FwdArgs& a, bool bf16, bool varlen, cudaStream_t s) {
  if (varlen)
    return bf16 ? launch_fwd256_t<true, true, false, true>(a, s) : launch_fwd256_t<false, true, false, true>(a, s);
  return bf16 ? launch_fwd256_t<true, false, false, true>(a, s) : launch_fwd256_t<false, false, false, true>(a, s);
}

cudaError_t launch_fwd256_varlen(const FwdArgs& a, bool bf16, cudaStream_t s) {
  if (a.drop_t > 0) return bf16 ? launch_fwd256_t<true, true, true>(a, s) : launch_fwd256_t<false, true, true>(a, s);
  return bf16 ? launch_fwd256_t<true, true>(a, s) : launch_fwd256_t<false, true>(a, s);
}

}  // namespace attn
