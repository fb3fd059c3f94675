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
// The MMA warp runs one product ahead of the element-wise warps: the next step's S (or
// S^T) is issued as soon as the element-wise warps have read the current one into
// registers, so it overlaps their dS work (dV kernel: S^T is double-buffered in tensor
// memory and the next S^T overlaps the P^T work).
//
// Warp roles as in bwd.cu: warp 0 TMA, warp 1 TMEM owner + MMA issuer, warps 2-3 idle,
// four element-wise warpgroups of 32 columns each.  Every wait is bounded.
//
// DROP (dropout, the forward's keep rule, Z = keep * 256 / (256 - t)): dV = (P o Z)^T dO
// and dS = P o (Z o dP - D), as in bwd.cu.  The key-tile kernels need the keep bits by
// key row: each lane draws one query's 32 keep bytes and 32 warp ballots transpose the
// 32 x 32 bit block, so no shared memory is spent on it.
#include "common.cuh"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int D2 = 256;
constexpr int kEw2 = 4;
constexpr int kEwCols2 = 128 / kEw2;
constexpr int kThreads2 = 128 * (1 + kEw2);
constexpr int kEwThreads2 = 128 * kEw2;
constexpr int kBlk = kTileM * 128;        // one 128-row x 64-column block (16 KB)
constexpr int kTile = kTileM * D2 * 2;    // one 128-row x 256-column tile (64 KB)
constexpr int kHalf = kTileM * 128 * 2;   // one 128-row x 128-column half (32 KB)
constexpr int kSmemMax = 232448;          // opt-in shared memory per CTA
constexpr int kStatusLayout = 3;          // ATTN_ERR_CUDA: the shared-memory window is misaligned

// Barriers (shared by the three kernels; unused ones are never waited on).
enum : int {
  R_STAT = 0,     // stationary tiles loaded
  R_SFULL = 1,    // + buffer: S / S^T computed (the dV kernel has two buffers)
  R_DPFULL = 3,   // dP / dP^T computed
  R_PREADY = 4,   // + buffer: P^T written (dV kernel)
  R_SREAD = 6,    // S / S^T read into registers (dK, dQ kernels)
  R_DSREADY = 7,  // dS / dS^T written
  R_DONE = 8,
  R_DRAIN = 9,
  R_FULL = 10,    // + ring slot (at most 5)
  R_EMPTY = 15,   // + ring slot
  R_COUNT = 20
};
constexpr int kMaxSlots = R_EMPTY - R_FULL;

// Shared memory: STATIONARY 64 KB tiles, NSLOT 32 KB ring slots, LBYTES of per-query
// values staged by the element-wise warps, the barriers.  Dynamic shared memory starts
// 1024-byte aligned in practice; the slack left below the opt-in limit covers a
// misaligned start up to SLACK bytes, and a kernel that finds more reports
// kStatusLayout and returns before touching anything.
template <int NSLOT, int STATIONARY, int LBYTES>
struct Layout256 {
  static_assert(NSLOT <= kMaxSlots, "ring slots");
  static constexpr int OFF_ST = 0;
  static constexpr int OFF_RING = STATIONARY * kTile;
  static constexpr int OFF_L = OFF_RING + NSLOT * kHalf;
  static constexpr int OFF_BAR = OFF_L + LBYTES;
  static constexpr int NEED = OFF_BAR + 256;
  static constexpr int SMEM = NEED + 1024 < kSmemMax ? NEED + 1024 : kSmemMax;
  static constexpr int SLACK = SMEM - NEED;
  static_assert(SLACK >= 0, "shared memory");
  static_assert(8 * R_COUNT + 16 <= 256, "barrier area");
  static_assert(NSLOT * kHalf >= kTile, "the epilogue stages a 256-column tile over the ring");
};

// Common CTA state of the three kernels.
struct Cta {
  uint8_t* smem;
  uint32_t sb, bars, tmem;
  volatile int* abort_flag;
};

// Aligns the layout, initialises the barriers and allocates all 512 TMEM columns.
// Returns false (status reported, nothing else done) when the slack does not cover
// the shared-memory window's misalignment; uniform over the CTA.
template <class L, int NSLOT>
__device__ __forceinline__ bool cta_setup(uint8_t* raw, int* dev_status, Cta& c) {
  const uintptr_t p = reinterpret_cast<uintptr_t>(raw);
  const uintptr_t al = (p + 1023) & ~static_cast<uintptr_t>(1023);
  if (al - p > static_cast<uintptr_t>(L::SLACK)) {
    if (threadIdx.x == 0 && dev_status) atomicExch(dev_status, kStatusLayout);
    return false;
  }
  c.smem = reinterpret_cast<uint8_t*>(al);
  c.sb = smem_u32(c.smem);
  c.bars = c.sb + L::OFF_BAR;
  c.abort_flag = reinterpret_cast<volatile int*>(c.smem + L::OFF_BAR + 8 * R_COUNT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(c.smem + L::OFF_BAR + 8 * R_COUNT + 8);
  if (threadIdx.x == 0) {
    for (int i = 0; i < R_FULL; ++i) {
      const bool ew = i == R_PREADY || i == R_PREADY + 1 || i == R_SREAD || i == R_DSREADY;
      mbar_init(c.bars + 8 * i, ew ? kEwThreads2 : 1);
    }
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(c.bars + 8 * (R_FULL + s), 1);
      mbar_init(c.bars + 8 * (R_EMPTY + s), 1);
    }
    *c.abort_flag = 0;
    fence_barrier_init();
  }
  if ((threadIdx.x >> 5) == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  c.tmem = *tmem_slot;
  return true;
}

__device__ __forceinline__ void teardown256(uint32_t tmem) {
  tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
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

// Producer: the two column halves (columns 0..127, 128..255) of a 128-row tile, as the
// ring's next two items, each once the item NSLOT earlier has been released.  (y, z) are
// the tile's TMA coordinates: (first row, head-batch), or (head, first token) in a packed
// [tokens][H][d] tensor.
template <int NSLOT>
__device__ __forceinline__ bool load_tile(Ring<NSLOT>& r, const CUtensorMap* m, int y, int z,
                                          const WaitCtl& wc) {
  for (int half = 0; half < 2; ++half) {
    const int c = r.c;
    if (c >= NSLOT && !mbar_wait(r.empty(c), ((c / NSLOT) - 1) & 1, wc)) return false;
    mbar_arrive_expect_tx(r.full(c), kHalf);
    for (int b = 0; b < 2; ++b) tma_load_3d(r.slot_addr(c) + b * kBlk, m, r.full(c), 128 * half + 64 * b, y, z);
    ++r.c;
  }
  return true;
}

// Producer's end: the stationary tiles and the last items have landed (no copy in
// flight when the CTA exits).
template <int NSLOT>
__device__ __forceinline__ void producer_drain(const Ring<NSLOT>& r, uint32_t stat_bar, const WaitCtl& wc) {
  mbar_wait(stat_bar, 0, wc);
  for (int c = (r.c > NSLOT ? r.c - NSLOT : 0); c < r.c; ++c) mbar_wait(r.full(c), (c / NSLOT) & 1, wc);
}

// The MMA warp's side of the ring (the whole warp calls it; one elected lane issues).
template <int NSLOT>
struct RingUse {
  Ring<NSLOT> r;
  const WaitCtl* wc;
  __device__ bool next() { return mbar_wait_warp(r.full(r.c), (r.c / NSLOT) & 1, *wc); }
  __device__ uint32_t addr() const { return r.slot_addr(r.c); }
  __device__ void release() {
    tc_commit_w(r.empty(r.c));
    ++r.c;
  }
};

// D = A_stat B^T over d = 256, both K-major: A a stationary 4-block tile, B the next two
// ring items (its column halves); commits `done` once issued.
template <int NSLOT>
__device__ __forceinline__ bool mma_kk256(RingUse<NSLOT>& u, uint32_t d_tmem, uint32_t a_stat, uint32_t idesc,
                                          uint32_t done) {
  for (int h = 0; h < 2; ++h) {
    if (!u.next()) return false;
    tc_fence_after();
    const uint32_t b_item = u.addr();
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int k = 8 * h + kk;
      const uint32_t aoff = (k >> 2) * kBlk + (k & 3) * 32;
      const uint32_t boff = (kk >> 2) * kBlk + (kk & 3) * 32;
      mma_ss_w(d_tmem, sdesc_sw128(a_stat + aoff, 16, 1024), sdesc_sw128(b_item + boff, 16, 1024), idesc,
               (h == 0 && kk == 0) ? 0u : 1u);
    }
    u.release();
  }
  tc_commit_w(done);
  return true;
}

// acc[:, 128h .. 128h+127] (+)= A_tmem B_h for both halves h: A the 16-bit operand the
// element-wise warpgroups wrote (warpgroup w: 16 columns at a_tmem + 32w), B the next two
// ring items (rows = the contraction, MN-major).
template <int NSLOT>
__device__ __forceinline__ bool mma_ts256(RingUse<NSLOT>& u, uint32_t acc, uint32_t a_tmem, uint32_t idesc,
                                          bool first) {
  for (int h = 0; h < 2; ++h) {
    if (!u.next()) return false;
    tc_fence_after();
    const uint32_t b_item = u.addr();
#pragma unroll
    for (int k = 0; k < kTileM / 16; ++k)
      mma_ts_w(acc + 128 * h, a_tmem + kEwCols2 * (k >> 1) + 8 * (k & 1), sdesc_sw128(b_item + k * 2048, kBlk, 1024),
               idesc, (first && k == 0) ? 0u : 1u);
    u.release();
  }
  return true;
}

// The key-tile kernels' element-wise warps need 32 per-query values (LSE2, D) per
// warpgroup: each warp stages them in its own 128-byte slice of shared memory (the
// lane's own value fetched from global memory beforehand) and reads them back as
// broadcast float4s.
struct RowStage {
  float* w;
  __device__ const float4* put(float x) {
    __syncwarp();
    w[threadIdx.x & 31] = x;
    __syncwarp();
    return reinterpret_cast<const float4*>(w);
  }
};

// The lengths a CTA works with and where its rows sit: the kernel parameters, or (VARLEN)
// one packed sequence's (seq_view), whose rows are token t0 + r of head hh.
struct Lens {
  int N, Nk, cofs, hh, tq0, tk0;
  bool degenerate;
};
template <bool VARLEN>
__device__ __forceinline__ Lens lens_of(const BwdArgs& a, int bh) {
  if constexpr (VARLEN) {
    const SeqView v = seq_view(a, bh);
    return {v.N, v.Nk, v.cofs, v.hh, v.tq0, v.tk0, v.degenerate || v.N <= 0};
  } else {
    return {a.N, a.Nk, a.cofs, 0, 0, 0, false};
  }
}

// Zero rows r0 .. min(r0 + 128, n) - 1 of head hh of a packed [T][H][256] tensor whose
// sequence starts at token t0 (the gradients of a sequence that has no softmax).
__device__ __forceinline__ void zero_rows256(void* base, int H, int hh, int t0, int r0, int n) {
  for (int r = threadIdx.x; r < kTileM; r += blockDim.x) {
    if (r0 + r >= n) continue;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(base) + ((static_cast<size_t>(t0 + r0 + r) * H + hh) * D2) * 2);
    for (int c = 0; c < D2 / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
  }
}

// P for this thread's 32 columns from S in registers: 2^(s scale log2e - lse2), lse2 one
// per column (lse4) or one for the row (lse_row, when lse4 is null).
__device__ __forceinline__ void softmax_cols(const uint32_t (&sv)[kEwCols2], float sl2, const float4* lse4,
                                             float lse_row, float (&p)[kEwCols2]) {
  // Paired fma per two columns; per column lse2 as 2^-(lse2 - s sl2), bit-identical to
  // the scalar form since round-to-nearest is symmetric under negation.
  if (lse4) {
    const uint64_t nsl2 = f32x2_pack(-sl2, -sl2);
#pragma unroll
    for (int v = 0; v < kEwCols2 / 4; ++v) {
      const float4 lv = lse4[v];
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
  } else {
    const uint64_t sl2x2 = f32x2_pack(sl2, sl2), nl2 = f32x2_pack(-lse_row, -lse_row);
#pragma unroll
    for (int e = 0; e < kEwCols2; e += 2) {
      float x0, x1;
      f32x2_unpack(f32x2_fma(f32x2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sl2x2, nl2), x0, x1);
      p[e] = ex2(x0);
      p[e + 1] = ex2(x1);
    }
  }
}

// Dropout keep bits, key-tile kernels: for this thread's key k_base + lane (k_base a
// multiple of 16; all 32 lanes call it together), bit c set iff query q_base + c keeps
// it.  Lane L draws query q_base + L's bits over the warp's 32 keys; ballot c collects
// key c's bits over the 32 queries and lane c keeps it.
__device__ __forceinline__ uint32_t keep_bits_by_key(const BwdArgs& a, int bh, int q_base, int k_base) {
  const int lane = threadIdx.x & 31;
  const uint32_t jg = static_cast<uint32_t>(k_base / 16), qi = static_cast<uint32_t>(q_base + lane);
  const uint32_t mine = dropout_keep16(jg, qi, static_cast<uint32_t>(bh), a.drop_t, a.seed_lo, a.seed_hi) |
                        (dropout_keep16(jg + 1, qi, static_cast<uint32_t>(bh), a.drop_t, a.seed_lo, a.seed_hi) << 16);
  uint32_t bits = 0;
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const uint32_t b = __ballot_sync(0xffffffffu, (mine >> c) & 1u);
    if (lane == c) bits = b;
  }
  return bits;
}

// Dropout keep bits, query-tile kernel: bit e set iff query i keeps key k_base + e.
__device__ __forceinline__ uint32_t keep_bits_by_query(const BwdArgs& a, int bh, int i, int k_base) {
  const uint32_t jg = static_cast<uint32_t>(k_base / 16);
  return dropout_keep16(jg, static_cast<uint32_t>(i), static_cast<uint32_t>(bh), a.drop_t, a.seed_lo, a.seed_hi) |
         (dropout_keep16(jg + 1, static_cast<uint32_t>(i), static_cast<uint32_t>(bh), a.drop_t, a.seed_lo,
                         a.seed_hi) << 16);
}

// dP <- Z o dP over this thread's 32 columns (bit e of keep: column e kept).
__device__ __forceinline__ void drop_scale_cols(uint32_t (&dv)[kEwCols2], uint32_t keep, float zs) {
#pragma unroll
  for (int e = 0; e < kEwCols2; ++e)
    dv[e] = __float_as_uint(((keep >> e) & 1u) ? __uint_as_float(dv[e]) * zs : 0.f);
}

// Zero p[e] for e < lo and for e >= hi (the masked columns).
__device__ __forceinline__ void mask_cols(float (&p)[kEwCols2], int lo, int hi) {
  if (lo > 0 || hi < kEwCols2) {
#pragma unroll
    for (int e = 0; e < kEwCols2; ++e)
      if (e < lo || e >= hi) p[e] = 0.f;
  }
}

// Epilogue: this thread's row of a 256-column fp32 accumulator (its warpgroup's 64
// columns), scaled, as 16-bit into a 128B-swizzled staging tile over the ring; then one
// TMA store of the 128 x 256 tile at row `row0` of head `bh`.
// VARLEN: the rows go straight to the packed tensor `out` (row r0 + row of the sequence
// at token t0, head hh; rows >= n are not written) instead of through a TMA store.
template <bool BF16, bool VARLEN>
__device__ __forceinline__ void epilogue256(bool ok, const Cta& c, int off_ring, uint32_t t_acc, int row, int h,
                                            float mul, uint32_t done_bar, const WaitCtl& wc, const CUtensorMap* m,
                                            int row0, int bh, void* out, int H, int hh, int t0, int n) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* stage = c.smem + off_ring;
  if (ok) ok = mbar_wait_warp(done_bar, 0, wc);
  if constexpr (VARLEN) {
    if (ok) {
      tc_fence_after();
      const size_t elem0 = (static_cast<size_t>(t0 + row0 + row) * H + hh) * D2;
#pragma unroll 1
      for (int cc = 2 * h; cc < 2 * h + 2; ++cc) {
        uint32_t v[32];
        tmem_ld_x32(t_acc + cc * 32, v);  // every lane loads (warp-wide); only rows < n store
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack2<BF16>(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
        if (row0 + row < n) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(out) + (elem0 + cc * 32) * 2);
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
    }
    return;
  }
  if (ok) {
    tc_fence_after();
#pragma unroll 1
    for (int cc = 2 * h; cc < 2 * h + 2; ++cc) {
      uint32_t v[32];
      tmem_ld_x32(t_acc + cc * 32, v);
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        pk[i] = pack2<BF16>(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int ch = (cc & 1) * 4 + q;  // 16-byte chunk within the 64-column block cc / 2
        uint4* dst = reinterpret_cast<uint4*>(stage + (cc >> 1) * kBlk + row * 128 + ((ch ^ (row & 7)) << 4));
        *dst = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
    }
    fence_proxy_async_smem();
  }
  named_bar_sync(1, kEwThreads2);
  if (warp == 4 && lane == 0 && ok && !*c.abort_flag) {
    for (int b = 0; b < 4; ++b) tma_store_3d(m, c.sb + off_ring + b * kBlk, 64 * b, row0, bh);
    bulk_commit();
    bulk_wait_read_all();
  }
}

// ------------------------------------------------------------------ dV
// TMEM: S^T in two buffers at 0 and 128 (P^T over the first columns of each), dV at
// 256..511.  MMA order: S^T(0) | S^T(1) dV(0) | S^T(2) dV(1) | ...; ring items
// Q(0) | Q(1) dO(0) | Q(2) dO(1) | ...
constexpr int kDvSlots = 5;
using LayoutDv = Layout256<kDvSlots, 1, 16 * 128>;

template <bool BF16, bool VARLEN, bool DROP>
__global__ void __launch_bounds__(kThreads2, 1) bwd256_dv_kernel(const __grid_constant__ BwdArgs a) {
  constexpr int NSLOT = kDvSlots;
  using L = LayoutDv;
  extern __shared__ uint8_t smem_raw[];
  const int n_tk = (a.Nk + kTileN - 1) / kTileN;  // key tiles (of the longest sequence)
  const WorkItem wi = work_item<2>(static_cast<int>(blockIdx.x), a.BH, n_tk);
  const int bh = wi.bh, k0 = wi.rank * kTileN;
  const Lens q = lens_of<VARLEN>(a, bh);
  if (VARLEN && k0 >= q.Nk) return;  // past the sequence's keys (whole CTA)
  if (VARLEN && q.degenerate) {      // no softmax for this sequence: zero gradients
    zero_rows256(a.dv_out, a.H, q.hh, q.tk0, k0, q.Nk);
    return;
  }
  Cta c;
  if (!cta_setup<L, NSLOT>(smem_raw, a.dev_status, c)) return;
  auto bar = [&](int i) -> uint32_t { return c.bars + 8u * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_t = (q.N + kTileM - 1) / kTileM;
  const int i_begin = a.causal ? max(0, k0 - q.cofs) / kTileM : 0;
  const int n_iter = n_t - i_begin;
  auto qy = [&](int r) { return VARLEN ? q.hh : r; };  // TMA coordinates of query row r
  auto qz = [&](int r) { return VARLEN ? q.tq0 + r : bh; };
  const WaitCtl wc{c.abort_flag, a.dev_status, a.wait_limit_ns};
  constexpr uint32_t TM_DV = 256;

  if (warp == 0 && lane == 0) {
    mbar_arrive_expect_tx(bar(R_STAT), kTile);
    for (int b = 0; b < 4; ++b)
      tma_load_3d(c.sb + L::OFF_ST + b * kBlk, &a.tm_k, bar(R_STAT), 64 * b, VARLEN ? q.hh : k0,
                  VARLEN ? q.tk0 + k0 : bh);
    Ring<NSLOT> r{c.sb + L::OFF_RING, c.bars};
    bool ok = n_iter <= 0 || load_tile(r, &a.tm_q, qy(i_begin * kTileM), qz(i_begin * kTileM), wc);
    for (int t = 0; ok && t < n_iter; ++t) {
      const int q0 = (i_begin + t) * kTileM;
      if (t + 1 < n_iter) ok = load_tile(r, &a.tm_q, qy(q0 + kTileM), qz(q0 + kTileM), wc);
      ok = ok && load_tile(r, &a.tm_do, qy(q0), qz(q0), wc);
    }
    producer_drain(r, bar(R_STAT), wc);
  } else if (warp == 1) {  // the whole warp runs the issuing loop, one elected lane issues
    constexpr uint32_t idesc_s = idesc_f16(kTileM, kTileM, BF16, false, false);
    constexpr uint32_t idesc_g = idesc_f16(kTileM, 128, BF16, false, true);
    RingUse<NSLOT> u{Ring<NSLOT>{c.sb + L::OFF_RING, c.bars}, &wc};
    const uint32_t kst = c.sb + L::OFF_ST;
    bool ok = mbar_wait_warp(bar(R_STAT), 0, wc);
    if (ok && n_iter > 0) ok = mma_kk256(u, c.tmem, kst, idesc_s, bar(R_SFULL));
    for (int t = 0; ok && t < n_iter; ++t) {
      const uint32_t buf = 128u * (t & 1);
      // S^T(t+1) into the other buffer (its P^T(t-1) was read by dV(t-1), issued earlier)
      if (t + 1 < n_iter && !(ok = mma_kk256(u, c.tmem + (128u - buf), kst, idesc_s, bar(R_SFULL + ((t + 1) & 1)))))
        break;
      if (!(ok = mbar_wait_warp(bar(R_PREADY + (t & 1)), (t >> 1) & 1, wc))) break;
      ok = mma_ts256(u, c.tmem + TM_DV, c.tmem + buf, idesc_g, t == 0);
    }
    if (ok) tc_commit_w(bar(R_DONE));
    tc_commit_w(bar(R_DRAIN));
    mbar_wait_warp(bar(R_DRAIN), 0, wc);
  } else if (warp >= 4) {
    const int h = (warp >> 2) - 1, wq = warp & 3, row = wq * 32 + lane;  // row: key within the tile
    const uint32_t t_lane = c.tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float sl2 = a.scale_log2;
    RowStage rs{reinterpret_cast<float*>(c.smem + L::OFF_L) + (warp - 4) * 32};
    bool ok = true;
    for (int t = 0; t < n_iter; ++t) {
      const int qt = i_begin + t;
      const uint32_t col = 128u * (t & 1) + kEwCols2 * h;
      const float my_l = a.lse2[static_cast<size_t>(bh) * a.Npad + qt * kTileM + kEwCols2 * h + lane];
      uint32_t keep = 0xffffffffu;  // bit c: query column c keeps this key
      if constexpr (DROP) keep = keep_bits_by_key(a, bh, qt * kTileM + kEwCols2 * h, k0 + 32 * wq);
      if (!(ok = mbar_wait_warp(bar(R_SFULL + (t & 1)), (t >> 1) & 1, wc))) break;
      tc_fence_after();
      const float4* l4 = rs.put(my_l);
      float p[kEwCols2];
      {
        uint32_t sv[kEwCols2];
        tmem_ld_x32(t_lane + col, sv);
        softmax_cols(sv, sl2, l4, 0.f, p);
      }
      if (a.causal) mask_cols(p, k0 + row - q.cofs - qt * kTileM - kEwCols2 * h, kEwCols2);
      uint32_t pk[kEwCols2 / 2];
      if constexpr (DROP) {  // dV takes P o Z
        const float zs = a.drop_scale;
#pragma unroll
        for (int e = 0; e < kEwCols2; e += 2)
          pk[e / 2] = pack2<BF16>(((keep >> e) & 1u) ? p[e] * zs : 0.f, ((keep >> (e + 1)) & 1u) ? p[e + 1] * zs : 0.f);
      } else {
#pragma unroll
        for (int e = 0; e < kEwCols2; e += 2) pk[e / 2] = pack2<BF16>(p[e], p[e + 1]);
      }
      tmem_st_x16(t_lane + col, pk);  // over columns this thread has read
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(R_PREADY + (t & 1)));
    }
    epilogue256<BF16, VARLEN>(ok, c, L::OFF_RING, t_lane + TM_DV, row, h, 1.f, bar(R_DONE), wc, &a.tm_dv, k0, bh,
                              a.dv_out, a.H, q.hh, q.tk0, q.Nk);
  }
  teardown256(c.tmem);
}

// ------------------------------------------------------------------ dK
// TMEM: S^T at 0, dP^T at 128 (dS^T over its first columns), dK at 256..511.  MMA order:
// S^T(0) dP^T(0) | S^T(1) dK(0) dP^T(1) | S^T(2) dK(1) dP^T(2) | ...; ring items
// Q(0) dO(0) | Q(1) Q(0) dO(1) | Q(2) Q(1) dO(2) | ...
constexpr int kDkSlots = 3;
using LayoutDk = Layout256<kDkSlots, 2, 16 * 128>;

template <bool BF16, bool VARLEN, bool DROP>
__global__ void __launch_bounds__(kThreads2, 1) bwd256_dk_kernel(const __grid_constant__ BwdArgs a) {
  constexpr int NSLOT = kDkSlots;
  using L = LayoutDk;
  extern __shared__ uint8_t smem_raw[];
  const int n_tk = (a.Nk + kTileN - 1) / kTileN;  // key tiles (of the longest sequence)
  const WorkItem wi = work_item<2>(static_cast<int>(blockIdx.x), a.BH, n_tk);
  const int bh = wi.bh, k0 = wi.rank * kTileN;
  const Lens q = lens_of<VARLEN>(a, bh);
  if (VARLEN && k0 >= q.Nk) return;  // past the sequence's keys (whole CTA)
  if (VARLEN && q.degenerate) {      // no softmax for this sequence: zero gradients
    zero_rows256(a.dk_out, a.H, q.hh, q.tk0, k0, q.Nk);
    return;
  }
  Cta c;
  if (!cta_setup<L, NSLOT>(smem_raw, a.dev_status, c)) return;
  auto bar = [&](int i) -> uint32_t { return c.bars + 8u * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_t = (q.N + kTileM - 1) / kTileM;
  const int i_begin = a.causal ? max(0, k0 - q.cofs) / kTileM : 0;
  const int n_iter = n_t - i_begin;
  auto qy = [&](int r) { return VARLEN ? q.hh : r; };  // TMA coordinates of query row r
  auto qz = [&](int r) { return VARLEN ? q.tq0 + r : bh; };
  const WaitCtl wc{c.abort_flag, a.dev_status, a.wait_limit_ns};
  constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DK = 256;
  const uint32_t st_k = c.sb + L::OFF_ST, st_v = c.sb + L::OFF_ST + kTile;

  if (warp == 0 && lane == 0) {
    mbar_arrive_expect_tx(bar(R_STAT), 2 * kTile);
    for (int b = 0; b < 4; ++b) {
      tma_load_3d(st_k + b * kBlk, &a.tm_k, bar(R_STAT), 64 * b, VARLEN ? q.hh : k0, VARLEN ? q.tk0 + k0 : bh);
      tma_load_3d(st_v + b * kBlk, &a.tm_v, bar(R_STAT), 64 * b, VARLEN ? q.hh : k0, VARLEN ? q.tk0 + k0 : bh);
    }
    Ring<NSLOT> r{c.sb + L::OFF_RING, c.bars};
    const int q_first = i_begin * kTileM;
    bool ok = n_iter <= 0 || (load_tile(r, &a.tm_q, qy(q_first), qz(q_first), wc) &&
                              load_tile(r, &a.tm_do, qy(q_first), qz(q_first), wc));
    for (int t = 0; ok && t < n_iter; ++t) {
      const int q0 = (i_begin + t) * kTileM;
      if (t + 1 < n_iter) ok = load_tile(r, &a.tm_q, qy(q0 + kTileM), qz(q0 + kTileM), wc);
      ok = ok && load_tile(r, &a.tm_q, qy(q0), qz(q0), wc);
      if (ok && t + 1 < n_iter) ok = load_tile(r, &a.tm_do, qy(q0 + kTileM), qz(q0 + kTileM), wc);
    }
    producer_drain(r, bar(R_STAT), wc);
  } else if (warp == 1) {  // the whole warp runs the issuing loop, one elected lane issues
    constexpr uint32_t idesc_s = idesc_f16(kTileM, kTileM, BF16, false, false);
    constexpr uint32_t idesc_g = idesc_f16(kTileM, 128, BF16, false, true);
    RingUse<NSLOT> u{Ring<NSLOT>{c.sb + L::OFF_RING, c.bars}, &wc};
    bool ok = mbar_wait_warp(bar(R_STAT), 0, wc);
    if (ok && n_iter > 0)
      ok = mma_kk256(u, c.tmem + TM_S, st_k, idesc_s, bar(R_SFULL)) &&
           mma_kk256(u, c.tmem + TM_DP, st_v, idesc_s, bar(R_DPFULL));
    for (int t = 0; ok && t < n_iter; ++t) {
      if (t + 1 < n_iter) {  // S^T(t+1) once S^T(t) is in registers
        if (!(ok = mbar_wait_warp(bar(R_SREAD), t & 1, wc))) break;
        tc_fence_after();
        if (!(ok = mma_kk256(u, c.tmem + TM_S, st_k, idesc_s, bar(R_SFULL)))) break;
      }
      if (!(ok = mbar_wait_warp(bar(R_DSREADY), t & 1, wc))) break;
      tc_fence_after();
      if (!(ok = mma_ts256(u, c.tmem + TM_DK, c.tmem + TM_DP, idesc_g, t == 0))) break;
      // dP^T(t+1) overwrites dS^T(t) after dK(t), issued above, has read it
      if (t + 1 < n_iter && !(ok = mma_kk256(u, c.tmem + TM_DP, st_v, idesc_s, bar(R_DPFULL)))) break;
    }
    if (ok) tc_commit_w(bar(R_DONE));
    tc_commit_w(bar(R_DRAIN));
    mbar_wait_warp(bar(R_DRAIN), 0, wc);
  } else if (warp >= 4) {
    const int h = (warp >> 2) - 1, wq = warp & 3, row = wq * 32 + lane;
    const uint32_t t_lane = c.tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float sl2 = a.scale_log2;
    RowStage rs{reinterpret_cast<float*>(c.smem + L::OFF_L) + (warp - 4) * 32};
    bool ok = true;
    for (int t = 0; t < n_iter; ++t) {
      const int qt = i_begin + t;
      const size_t wrow = static_cast<size_t>(bh) * a.Npad + qt * kTileM + kEwCols2 * h + lane;
      const float my_l = a.lse2[wrow], my_d = a.delta[wrow];
      uint32_t keep = 0xffffffffu;  // bit c: query column c keeps this key
      if constexpr (DROP) keep = keep_bits_by_key(a, bh, qt * kTileM + kEwCols2 * h, k0 + 32 * wq);
      if (!(ok = mbar_wait_warp(bar(R_SFULL), t & 1, wc))) break;
      tc_fence_after();
      float p[kEwCols2];
      {
        const float4* l4 = rs.put(my_l);
        uint32_t sv[kEwCols2];
        tmem_ld_x32(t_lane + TM_S + kEwCols2 * h, sv);
        tc_fence_before();
        mbar_arrive(bar(R_SREAD));
        softmax_cols(sv, sl2, l4, 0.f, p);
      }
      if (a.causal) mask_cols(p, k0 + row - q.cofs - qt * kTileM - kEwCols2 * h, kEwCols2);
      const float4* d4 = rs.put(my_d);
      if (!(ok = mbar_wait_warp(bar(R_DPFULL), t & 1, wc))) break;
      tc_fence_after();
      {
        uint32_t dv[kEwCols2], ds[kEwCols2 / 2];
        tmem_ld_x32(t_lane + TM_DP + kEwCols2 * h, dv);
        if constexpr (DROP) drop_scale_cols(dv, keep, a.drop_scale);
#pragma unroll
        for (int v = 0; v < kEwCols2 / 4; ++v) {  // paired sub and mul, two columns each
          const float4 dd = d4[v];
          float a0, a1, b0, b1;
          f32x2_unpack(f32x2_mul(f32x2_pack(p[4 * v], p[4 * v + 1]),
                                 f32x2_sub(f32x2_pack(__uint_as_float(dv[4 * v]), __uint_as_float(dv[4 * v + 1])),
                                           f32x2_pack(dd.x, dd.y))), a0, a1);
          f32x2_unpack(f32x2_mul(f32x2_pack(p[4 * v + 2], p[4 * v + 3]),
                                 f32x2_sub(f32x2_pack(__uint_as_float(dv[4 * v + 2]), __uint_as_float(dv[4 * v + 3])),
                                           f32x2_pack(dd.z, dd.w))), b0, b1);
          ds[2 * v] = pack2<BF16>(a0, a1);
          ds[2 * v + 1] = pack2<BF16>(b0, b1);
        }
        tmem_st_x16(t_lane + TM_DP + kEwCols2 * h, ds);  // over columns this thread has read
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(R_DSREADY));
    }
    epilogue256<BF16, VARLEN>(ok, c, L::OFF_RING, t_lane + TM_DK, row, h, a.scale, bar(R_DONE), wc, &a.tm_dk, k0, bh,
                              a.dk_out, a.H, q.hh, q.tk0, q.Nk);
  }
  teardown256(c.tmem);
}

// ------------------------------------------------------------------ dQ
// TMEM: S at 0, dP at 128 (dS over its first columns), dQ at 256..511.  MMA order:
// S(0) dP(0) | S(1) dQ(0) dP(1) | ...; ring items K(0) V(0) | K(1) K(0) V(1) | ...
constexpr int kDqSlots = 3;
using LayoutDq = Layout256<kDqSlots, 2, 0>;

template <bool BF16, bool VARLEN, bool DROP>
__global__ void __launch_bounds__(kThreads2, 1) bwd256_dq_kernel(const __grid_constant__ BwdArgs a) {
  constexpr int NSLOT = kDqSlots;
  using L = LayoutDq;
  extern __shared__ uint8_t smem_raw[];
  const int n_t = (a.N + kTileM - 1) / kTileM;  // query tiles (of the longest sequence)
  const WorkItem wi = work_item<2>(static_cast<int>(blockIdx.x), a.BH, n_t);
  const int bh = wi.bh, qt = n_t - 1 - wi.rank, q0 = qt * kTileM;
  const Lens q = lens_of<VARLEN>(a, bh);
  if (VARLEN && q0 >= q.N) return;  // past the sequence's queries (whole CTA)
  if (VARLEN && q.degenerate) {     // no softmax for this sequence: zero gradients
    zero_rows256(a.dq_out, a.H, q.hh, q.tq0, q0, q.N);
    return;
  }
  Cta c;
  if (!cta_setup<L, NSLOT>(smem_raw, a.dev_status, c)) return;
  auto bar = [&](int i) -> uint32_t { return c.bars + 8u * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_kv = visible_key_tiles(qt, q.Nk, a.causal, q.cofs);
  auto ky = [&](int r) { return VARLEN ? q.hh : r; };  // TMA coordinates of key row r
  auto kz = [&](int r) { return VARLEN ? q.tk0 + r : bh; };
  const WaitCtl wc{c.abort_flag, a.dev_status, a.wait_limit_ns};
  constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DQ = 256;
  const uint32_t st_q = c.sb + L::OFF_ST, st_do = c.sb + L::OFF_ST + kTile;

  if (warp == 0 && lane == 0) {
    mbar_arrive_expect_tx(bar(R_STAT), 2 * kTile);
    for (int b = 0; b < 4; ++b) {
      tma_load_3d(st_q + b * kBlk, &a.tm_q, bar(R_STAT), 64 * b, VARLEN ? q.hh : q0, VARLEN ? q.tq0 + q0 : bh);
      tma_load_3d(st_do + b * kBlk, &a.tm_do, bar(R_STAT), 64 * b, VARLEN ? q.hh : q0, VARLEN ? q.tq0 + q0 : bh);
    }
    Ring<NSLOT> r{c.sb + L::OFF_RING, c.bars};
    bool ok = n_kv <= 0 || (load_tile(r, &a.tm_k, ky(0), kz(0), wc) && load_tile(r, &a.tm_v, ky(0), kz(0), wc));
    for (int j = 0; ok && j < n_kv; ++j) {
      const int kr = j * kTileN;
      if (j + 1 < n_kv) ok = load_tile(r, &a.tm_k, ky(kr + kTileN), kz(kr + kTileN), wc);
      ok = ok && load_tile(r, &a.tm_k, ky(kr), kz(kr), wc);
      if (ok && j + 1 < n_kv) ok = load_tile(r, &a.tm_v, ky(kr + kTileN), kz(kr + kTileN), wc);
    }
    producer_drain(r, bar(R_STAT), wc);
  } else if (warp == 1) {  // the whole warp runs the issuing loop, one elected lane issues
    constexpr uint32_t idesc_s = idesc_f16(kTileM, kTileN, BF16, false, false);
    constexpr uint32_t idesc_g = idesc_f16(kTileM, 128, BF16, false, true);
    RingUse<NSLOT> u{Ring<NSLOT>{c.sb + L::OFF_RING, c.bars}, &wc};
    bool ok = mbar_wait_warp(bar(R_STAT), 0, wc);
    if (ok && n_kv > 0)
      ok = mma_kk256(u, c.tmem + TM_S, st_q, idesc_s, bar(R_SFULL)) &&
           mma_kk256(u, c.tmem + TM_DP, st_do, idesc_s, bar(R_DPFULL));
    for (int j = 0; ok && j < n_kv; ++j) {
      if (j + 1 < n_kv) {  // S(j+1) once S(j) is in registers
        if (!(ok = mbar_wait_warp(bar(R_SREAD), j & 1, wc))) break;
        tc_fence_after();
        if (!(ok = mma_kk256(u, c.tmem + TM_S, st_q, idesc_s, bar(R_SFULL)))) break;
      }
      if (!(ok = mbar_wait_warp(bar(R_DSREADY), j & 1, wc))) break;
      tc_fence_after();
      if (!(ok = mma_ts256(u, c.tmem + TM_DQ, c.tmem + TM_DP, idesc_g, j == 0))) break;
      // dP(j+1) overwrites dS(j) after dQ(j), issued above, has read it
      if (j + 1 < n_kv && !(ok = mma_kk256(u, c.tmem + TM_DP, st_do, idesc_s, bar(R_DPFULL)))) break;
    }
    if (ok) tc_commit_w(bar(R_DONE));
    tc_commit_w(bar(R_DRAIN));
    mbar_wait_warp(bar(R_DRAIN), 0, wc);
  } else if (warp >= 4) {
    const int h = (warp >> 2) - 1, wq = warp & 3, row = wq * 32 + lane, grow = q0 + row;
    const uint32_t t_lane = c.tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float sl2 = a.scale_log2;
    const size_t w = static_cast<size_t>(bh) * a.Npad + grow;  // grow < Npad always
    const float lse2 = a.lse2[w], dlt = a.delta[w];
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      uint32_t keep = 0xffffffffu;  // bit e: this query keeps key column e
      if constexpr (DROP) keep = keep_bits_by_query(a, bh, grow, j * kTileN + kEwCols2 * h);
      if (!(ok = mbar_wait_warp(bar(R_SFULL), j & 1, wc))) break;
      tc_fence_after();
      float p[kEwCols2];
      {
        uint32_t sv[kEwCols2];
        tmem_ld_x32(t_lane + TM_S + kEwCols2 * h, sv);
        tc_fence_before();
        mbar_arrive(bar(R_SREAD));
        softmax_cols(sv, sl2, nullptr, lse2, p);
      }
      const int kbeg = j * kTileN + kEwCols2 * h;
      int lim = q.Nk - kbeg;                                     // keys past the end
      if (a.causal) lim = min(lim, grow + q.cofs - kbeg + 1);  // keys after this query
      mask_cols(p, 0, lim);
      if (!(ok = mbar_wait_warp(bar(R_DPFULL), j & 1, wc))) break;
      tc_fence_after();
      {
        uint32_t dv[kEwCols2], ds[kEwCols2 / 2];
        tmem_ld_x32(t_lane + TM_DP + kEwCols2 * h, dv);
        if constexpr (DROP) drop_scale_cols(dv, keep, a.drop_scale);
        const uint64_t dlt2 = f32x2_pack(dlt, dlt);
#pragma unroll
        for (int e = 0; e < kEwCols2; e += 2) {  // paired sub and mul
          float a0, a1;
          f32x2_unpack(f32x2_mul(f32x2_pack(p[e], p[e + 1]),
                                 f32x2_sub(f32x2_pack(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])), dlt2)),
                       a0, a1);
          ds[e / 2] = pack2<BF16>(a0, a1);
        }
        tmem_st_x16(t_lane + TM_DP + kEwCols2 * h, ds);  // over columns this thread has read
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(R_DSREADY));
    }
    epilogue256<BF16, VARLEN>(ok, c, L::OFF_RING, t_lane + TM_DQ, row, h, a.scale, bar(R_DONE), wc, &a.tm_dq, q0, bh,
                              a.dq_out, a.H, q.hh, q.tq0, q.N);
  }
  teardown256(c.tmem);
}

template <class K>
cudaError_t launch256(K k, int smem, int grid, const BwdArgs& a, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k<<<grid, kThreads2, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

template <bool VARLEN, bool DROP = false>
cudaError_t launch_dkdv256_t(const BwdArgs& a, bool bf16, cudaStream_t s) {
  const int grid = (a.Nk + kTileN - 1) / kTileN * a.BH;
  cudaError_t e = bf16 ? launch256(bwd256_dv_kernel<true, VARLEN, DROP>, LayoutDv::SMEM, grid, a, s)
                       : launch256(bwd256_dv_kernel<false, VARLEN, DROP>, LayoutDv::SMEM, grid, a, s);
  if (e != cudaSuccess) return e;
  return bf16 ? launch256(bwd256_dk_kernel<true, VARLEN, DROP>, LayoutDk::SMEM, grid, a, s)
              : launch256(bwd256_dk_kernel<false, VARLEN, DROP>, LayoutDk::SMEM, grid, a, s);
}

template <bool VARLEN, bool DROP = false>
cudaError_t launch_dq256_t(const BwdArgs& a, bool bf16, cudaStream_t s) {
  const int grid = (a.N + kTileM - 1) / kTileM * a.BH;
  return bf16 ? launch256(bwd256_dq_kernel<true, VARLEN, DROP>, LayoutDq::SMEM, grid, a, s)
              : launch256(bwd256_dq_kernel<false, VARLEN, DROP>, LayoutDq::SMEM, grid, a, s);
}

// a.drop_t > 0 selects the dropout kernels.
cudaError_t launch_bwd256_dkdv(const BwdArgs& a, bool bf16, cudaStream_t s) {
  return a.drop_t > 0 ? launch_dkdv256_t<false, true>(a, bf16, s) : launch_dkdv256_t<false>(a, bf16, s);
}
cudaError_t launch_bwd256_dq(const BwdArgs& a, bool bf16, cudaStream_t s) {
  return a.drop_t > 0 ? launch_dq256_t<false, true>(a, bf16, s) : launch_dq256_t<false>(a, bf16, s);
}
cudaError_t launch_bwd256_dkdv_varlen(const BwdArgs& a, bool bf16, cudaStream_t s) {
  return a.drop_t > 0 ? launch_dkdv256_t<true, true>(a, bf16, s) : launch_dkdv256_t<true>(a, bf16, s);
}
cudaError_t launch_bwd256_dq_varlen(const BwdArgs& a, bool bf16, cudaStream_t s) {
  return a.drop_t > 0 ? launch_dq256_t<true, true>(a, bf16, s) : launch_dq256_t<true>(a, bf16, s);
}

}  // namespace attn
