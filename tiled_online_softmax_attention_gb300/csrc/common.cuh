// common.cuh -- launch parameters shared by the host API (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

// Tiles: 128 query rows x 128 keys for every kernel (one TMEM lane per row).
constexpr int kTileM = 128;
constexpr int kTileN = 128;

struct FwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_o;  // 3-D maps over [B*H][N][d], 128-byte boxes x 128 rows, 128B swizzle
  CUtensorMap tm_kh;                   // the pair kernel (fwd_pair.cu): K with 64-row boxes (half a key tile)
  void* o;                             // [B*H][N][d] output (the merge kernel writes it directly)
  float* lse;                          // [B*H][N]
  int* dev_status;                     // nullable
  int N;                               // queries per head
  int Nk;                              // keys per head (tm_k, tm_v rows)
  int cofs;                            // causal: query i sees keys j <= i + cofs (cofs = Nk - N)
  int BH;
  int causal;
  float scale_log2;                    // scale * log2(e)
  uint64_t wait_limit_ns;
  // split-KV only: n_splits key ranges per query-tile pair, each writing its normalised
  // partial output and logsumexp for the merge kernel
  int n_splits;
  float* part_o;                       // [n_splits][B*H][N][d] fp32
  float* part_lse;                     // [n_splits][B*H][N] fp32 (natural log; -inf: empty range)
  // E4M3 inputs only: one scale per 128-row block of each head, [B*H][ceil(N/128)]
  const float* q_scale;                // [B*H][ceil(N/128)]
  const float* k_scale;                // [B*H][ceil(Nk/128)]
  const float* v_scale;
  // dropout only: keep (bh, i, j) iff its Philox byte >= drop_t; kept ones scaled by drop_scale
  uint32_t drop_t;
  uint32_t seed_lo, seed_hi;
  float drop_scale;                    // 256 / (256 - drop_t)
  // dropout keep bits written by the forward (nullable; d <= 128, not packed): bit b of word
  // ((bh * n_tk + j) * 4 + w) * bits_rows + i is the keep decision of query i and key
  // 128 j + 32 w + b (n_tk key tiles, bits_rows = N rounded up to 128)
  uint32_t* keep_bits;
  int bits_rows;
  // variable-length packed sequences only: tensors [tokens][H][d] (maps over (d, H, tokens)),
  // sequence b = bh / H owns query tokens cu_q[b] .. cu_q[b+1]-1 and key tokens
  // cu_k[b] .. cu_k[b+1]-1; N and Nk are the longest lengths (grid size); lse is [H][Tq]
  int H;
  int Tq;
  const int* cu_q;
  const int* cu_k;
};

// Key tiles query tile qt (rows qt*128 .. qt*128+127) has to visit: every key tile when
// not causal, else those holding a key j <= the tile's last row + cofs.
__host__ __device__ __forceinline__ int visible_key_tiles(int qt, int Nk, int causal, int cofs) {
  const int n_tk = (Nk + 127) / 128;
  if (!causal) return n_tk;
  const int last = qt * 128 + 127 + cofs;
  return min(last / 128 + 1, n_tk);
}

struct BwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // inputs, as in FwdArgs
  CUtensorMap tm_dq, tm_dk, tm_dv;      // outputs
  CUtensorMap tm_qh, tm_doh;            // the pair dK/dV kernel (bwd_pair.cu): Q and dO with 64-row boxes
  const void* o;                        // [B*H][N][d] forward output
  const void* dout;                     // [B*H][N][d]
  const float* lse;                     // [B*H][N]
  float* lse2;                          // workspace [B*H][Npad]: lse * log2(e); +inf on padding rows
  float* delta;                         // workspace [B*H][Npad]: rowsum(dO * O); 0 on padding rows
  int* dev_status;
  int N;                                // queries per head
  int Nk;                               // keys per head
  int cofs;                             // causal: query i sees keys j <= i + cofs (cofs = Nk - N)
  int Npad;                             // N rounded up to a multiple of 128
  int BH;
  int causal;
  float scale;
  float scale_log2;
  uint64_t wait_limit_ns;
  // dropout only, as in FwdArgs (keep_bits: the forward's stored decisions, read by the
  // backward kernels instead of drawing; nullable)
  uint32_t drop_t;
  uint32_t seed_lo, seed_hi;
  float drop_scale;
  const uint32_t* keep_bits;
  int bits_rows;
  // variable-length packed sequences only, as in FwdArgs (N, Nk: the longest lengths;
  // Npad: N rounded up; lse [H][Tq]; the workspace keeps [B*H][Npad])
  int H;
  int Tq;
  const int* cu_q;
  const int* cu_k;
  void* dq_out;                         // packed gradients, written row by row
  void* dk_out;
  void* dv_out;
  // fused backward only: float32 dQ accumulator in the workspace, [B*H][Npad][d] (row
  // major), zeroed by the preparation pass; nullptr for the deterministic kernels.  The
  // 2-D map over it ({d, B*H*Npad}, box {d/4, 16}, 128- or 64-byte swizzle) carries the
  // TMA bulk reductions of the fused kernel.
  float* dq_acc;
  CUtensorMap tm_dqacc;
  void* dq;                             // fused backward: dQ [B*H][N][d] (the finishing pass writes it)
};

// One packed sequence as a kernel sees it: lengths clamped to the caller's bounds, the
// first query and key tokens, the head, and whether it is degenerate (no key, or causal
// with fewer keys than queries: every row of it gets O = 0, lse = -inf, zero gradients).
struct SeqView {
  int N, Nk, cofs, hh, tq0, tk0;
  bool degenerate;
};
template <class Args>
__device__ __forceinline__ SeqView seq_view(const Args& a, int bh) {
  const int b = bh / a.H;
  SeqView v;
  v.hh = bh % a.H;
  v.tq0 = min(max(a.cu_q[b], 0), a.Tq);
  v.tk0 = max(a.cu_k[b], 0);
  v.N = min(min(max(a.cu_q[b + 1], v.tq0), a.Tq) - v.tq0, a.N);
  v.Nk = min(max(a.cu_k[b + 1] - v.tk0, 0), a.Nk);
  v.cofs = a.causal ? v.Nk - v.N : 0;
  v.degenerate = v.Nk <= 0 || (a.causal && v.Nk < v.N);
  return v;
}

// Order in which CTAs take work.  Heads go in groups of up to kGroup: within a group
// the CTAs walk the tile index (rank 0 first), so the CTAs running at one time
// share a few heads' K/V in L2, and the longest causal tiles of every group start
// before its short ones (no long tile is left for the end of the grid).  Groups of 8
// suit d <= 128; at d = 256 a head's K/V is twice as large and groups of 2 measured
// fastest (8 overflowed L2: 5x the input bytes read from DRAM).
struct WorkItem {
  int bh;    // (batch, head)
  int rank;  // 0 .. n_units-1 in dispatch order within the head
};
template <int kGroup = 8>
__device__ __forceinline__ WorkItem work_item(int x, int BH, int n_units) {
  const int full = BH / kGroup;
  const int per_group = kGroup * n_units;
  int g, y, gs;
  if (x < full * per_group) {
    g = x / per_group;
    y = x % per_group;
    gs = kGroup;
  } else {
    g = full;
    y = x - full * per_group;
    gs = BH - full * kGroup;
  }
  return {g * kGroup + y % gs, y / gs};
}

// Launchers (fwd.cu / bwd.cu); return the CUDA launch status.
cudaError_t launch_fwd(const FwdArgs& a, int d, bool bf16, cudaStream_t s);
// d = 128 on CTA pairs (fwd_pair.cu); needs tm_kh; not split, E4M3, dropout or packed
cudaError_t launch_fwd_pair(const FwdArgs& a, bool bf16, cudaStream_t s);
// d = 64 on a persistent grid (fwd_persist.cu); an even number of query tiles; not split,
// dropout or packed
cudaError_t launch_fwd_persist(const FwdArgs& a, bool bf16, cudaStream_t s);
cudaError_t launch_fwd_split(const FwdArgs& a, int d, bool bf16, cudaStream_t s);
cudaError_t launch_fwd_varlen_split(const FwdArgs& a, int d, bool bf16, cudaStream_t s);  // packed batches
cudaError_t launch_fwd_fp8(const FwdArgs& a, int d, bool bf16_out, cudaStream_t s);
cudaError_t launch_fwd256(const FwdArgs& a, bool bf16, cudaStream_t s);
cudaError_t launch_fwd256_split(const FwdArgs& a, bool bf16, bool varlen, cudaStream_t s);  // partials only
cudaError_t launch_fwd256_varlen(const FwdArgs& a, bool bf16, cudaStream_t s);
cudaError_t launch_fwd_dropout(const FwdArgs& a, int d, bool bf16, cudaStream_t s);
cudaError_t launch_fwd_varlen(const FwdArgs& a, int d, bool bf16, cudaStream_t s);
cudaError_t launch_bwd_dkdv_dropout(const BwdArgs& a, int d, bool bf16, cudaStream_t s);
cudaError_t launch_bwd_dq_dropout(const BwdArgs& a, int d, bool bf16, cudaStream_t s);
cudaError_t launch_bwd_pre_varlen(const BwdArgs& a, int d, bool bf16, cudaStream_t s);
cudaError_t launch_bwd_dkdv_varlen(const BwdArgs& a, int d, bool bf16, cudaStream_t s);
cudaError_t launch_bwd_dq_varlen(const BwdArgs& a, int d, bool bf16, cudaStream_t s);
cudaError_t launch_bwd_pre(const BwdArgs& a, int d, bool bf16, cudaStream_t s);
cudaError_t launch_bwd_dkdv(const BwdArgs& a, int d, bool bf16, cudaStream_t s);
cudaError_t launch_bwd_dq(const BwdArgs& a, int d, bool bf16, cudaStream_t s);
// d = 128 dK/dV on CTA pairs (bwd_pair.cu); needs tm_qh, tm_doh; not dropout or packed
cudaError_t launch_bwd_dkdv_pair(const BwdArgs& a, bool bf16, cudaStream_t s);
// dK/dV and dQ in one grid (the preparation pass must have run)
cudaError_t launch_bwd_grads(const BwdArgs& a, int d, bool bf16, cudaStream_t s);
cudaError_t launch_bwd_grads_dropout(const BwdArgs& a, int d, bool bf16, cudaStream_t s);
cudaError_t launch_bwd256_dkdv(const BwdArgs& a, bool bf16, cudaStream_t s);  // d = 256: dV, then dK
cudaError_t launch_bwd256_dq(const BwdArgs& a, bool bf16, cudaStream_t s);
cudaError_t launch_bwd256_dkdv_varlen(const BwdArgs& a, bool bf16, cudaStream_t s);
cudaError_t launch_bwd256_dq_varlen(const BwdArgs& a, bool bf16, cudaStream_t s);
// The fused backward (bwd_fused.cu): dK, dV and the float32 dQ accumulator in one pass over
// each key tile's query tiles (five products per tile pair), then dQ = scale * accumulator.
cudaError_t launch_bwd_fused(const BwdArgs& a, int d, bool bf16, bool varlen, cudaStream_t s);
cudaError_t launch_bwd_dq_finish(const BwdArgs& a, int d, bool bf16, bool varlen, cudaStream_t s);
cudaError_t launch_wait_selftest(int* dev_status, uint64_t limit_ns, cudaStream_t s);

}  // namespace attn
