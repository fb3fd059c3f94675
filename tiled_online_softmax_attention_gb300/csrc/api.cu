// api.cu -- the C ABI declared in include/attn.h: argument validation, TMA
// descriptor encoding and kernel dispatch.  Nothing here allocates device
// memory or keeps state between calls (the driver entry point for the tensor
// map encoder is looked up once and cached).
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <initializer_list>
#include <vector>

#include "../../include/attn.h"
#include "common.cuh"

namespace {

using attn::kTileM;

constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s per wait; a healthy wait takes microseconds

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Which kernel runs the d = 128 forward without dropout: the CTA-pair kernel (fwd_pair.cu)
// when the mask is not causal and every query tile visits at least 48 key tiles, else the
// one-CTA kernel.  Measured on B=1, H=32, N=16384: pair 1513 against 1444 TFLOP/s
// non-causal, but 1420 against 1437 causal; on B=2, H=16, N=8192 causal 1285 against 1367,
// and N=4096 causal 853 against 955 (the pair kernel's twice as many CTAs each pay their
// own start-up and epilogue, which the causal mask's short rows cannot amortise).
// ATTN_FWD_CTA_PAIR=1 or =0 (read on every call) forces one or the other.
bool fwd_use_pair(int Nk, int causal) {
  const char* s = std::getenv("ATTN_FWD_CTA_PAIR");
  if (s && (s[0] == '0' || s[0] == '1') && s[1] == 0) return s[0] == '1';
  return !causal && (Nk + attn::kTileN - 1) / attn::kTileN >= 48;
}

// The d = 64 forward without dropout on the persistent grid (fwd_persist.cu) when
// ATTN_FWD_PERSIST=1 (read on every call) and the query tiles pair up evenly.  The same
// bytes as fwd_kernel; measured 159.7 against 172.3 us on B=32, H=12, N=1024 non-causal,
// level on B=8, H=12, N=1024, and slower on causal and long rows (2797 against 2619 us on
// B=1, H=32, N=16384), so it is not the default.
bool fwd_use_persist(int N) {
  const char* s = std::getenv("ATTN_FWD_PERSIST");
  const bool even = ((N + attn::kTileM - 1) / attn::kTileM) % 2 == 0;
  return even && s && s[0] == '1' && s[1] == 0;
}

// The d = 128 dK/dV stage without dropout on CTA pairs (bwd_pair.cu) when
// ATTN_BWD_CTA_PAIR=1 (read on every call), else the one-CTA kernel.  Both give the same
// bytes; the pair kernel measured 0.774 against 0.716 ms on B=2, H=16, N=8192 causal and
// 1.473 against 1.407 ms non-causal (its hand-offs cross SMs, which costs more than the
// halved operand reads save), so it is not the default.
bool bwd_use_pair() {
  const char* s = std::getenv("ATTN_BWD_CTA_PAIR");
  return s && s[0] == '1' && s[1] == 0;
}

uint64_t wait_limit_ns() {
  static uint64_t v = [] {
    const char* s = std::getenv("ATTN_WAIT_LIMIT_NS");
    if (!s) return kDefaultWaitLimitNs;
    const unsigned long long x = std::strtoull(s, nullptr, 10);
    return x ? static_cast<uint64_t>(x) : kDefaultWaitLimitNs;
  }();
  return v;
}

// 3-D map over a [BH][N][d] 16-bit tensor: box {64, rows, 1} (rows = 128 but for the
// pair forward's half key tiles), 128-byte swizzle, out-of-range rows read as zero and
// are dropped on store.
bool make_map(CUtensorMap* m, const void* base, int BH, int N, int d, bool bf16, int rows = kTileM) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D map over a packed [T][H][d] 16-bit tensor, dimensions (d, H, T): box {64, 1, 128}
// puts 128 tokens of one head in shared memory exactly as make_map's box does.
bool make_map_packed(CUtensorMap* m, const void* base, int H, int T, int d, bool bf16) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(H) * d * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kTileM)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D map over a [BH][N][d] tensor of E4M3 bytes: box {128, 128, 1} (one 128-byte row
// block at d = 128), 128-byte swizzle, zero fill past the end.
bool make_map_e4m3(CUtensorMap* m, const void* base, int BH, int N, int d) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N) * d};
  cuuint32_t box[3] = {128, static_cast<cuuint32_t>(kTileM), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D map over the fused backward's float32 dQ accumulator [rows][d]: box {d/4, 16} (one
// element-wise warp's columns, half its 32 rows), swizzled like the staging area the
// kernel writes (128-byte rows at d = 128, 64-byte rows at d = 64).
bool make_map_acc(CUtensorMap* m, const void* base, int64_t rows, int d) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 4};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(d / 4), 16};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Dropout parameters: t = round(256 p) in 0..255 (0 = no dropout) and the 64-bit seed.
struct Dropout {
  uint32_t t = 0;
  uint64_t seed = 0;
};

// p must be finite and in [0, 1) with round(256 p) <= 255.
bool dropout_from_p(float p, uint64_t seed, Dropout* out) {
  if (!(std::isfinite(p) && p >= 0.f && p < 1.f)) return false;
  const long t = std::lround(256.0 * static_cast<double>(p));
  if (t > 255) return false;
  out->t = static_cast<uint32_t>(t);
  out->seed = seed;
  return true;
}

template <class Args>
void set_dropout(Args& a, const Dropout& dr) {
  a.drop_t = dr.t;
  a.seed_lo = static_cast<uint32_t>(dr.seed);
  a.seed_hi = static_cast<uint32_t>(dr.seed >> 32);
  a.drop_scale = 256.f / static_cast<float>(256 - static_cast<int>(dr.t));
}
bool aligned4(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// d = 256 is accepted only where the caller says so (all but the FP8 forward).
// Nk = key length.
attn_status check_sizes(int B, int H, int N, int d, attn_dtype dt, float scale, bool allow_d256 = false,
                        int Nk = -1) {
  if (Nk < 0) Nk = N;
  if (B < 1 || H < 1 || N < 1 || Nk < 1) return ATTN_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && !(allow_d256 && d == 256)) return ATTN_ERR_UNSUPPORTED;
  if (dt != ATTN_BF16 && dt != ATTN_FP16) return ATTN_ERR_UNSUPPORTED;
  const int64_t total = static_cast<int64_t>(B) * H * (N > Nk ? N : Nk) * d;
  if (total >= (int64_t(1) << 31)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

attn_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (major != 10 || minor != 3) return ATTN_ERR_UNSUPPORTED;  // built for sm_103a only
  return ATTN_OK;
}

// A tensor argument and its size in bytes.
struct Buf {
  const void* p;
  size_t bytes;
};

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace

extern "C" {

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
  }
  return "ATTN_ERR_UNKNOWN";
}

}  // extern "C"

namespace {

// The forward for Nq queries against Nk keys (Nk = Nq for attn_fwd).
attn_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int Nk,
                     int d, attn_dtype dt, int causal, float scale, int* dev_status, void* stream,
                     const Dropout& dr = Dropout{}, uint32_t* keep_bits = nullptr) {
  attn_status st = check_sizes(B, H, N, d, dt, scale, true, Nk);
  if (st != ATTN_OK) return st;
  if (causal && Nk < N) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_INVALID_ARG;
  const size_t qb = static_cast<size_t>(B) * H * N * d * 2, kb = static_cast<size_t>(B) * H * Nk * d * 2;
  const size_t lb = static_cast<size_t>(B) * H * N * 4;
  for (const void* in : {q, k, v}) {
    const size_t ib = in == q ? qb : kb;
    if (overlaps(in, ib, o, qb) || overlaps(in, ib, lse, lb)) return ATTN_ERR_INVALID_ARG;
  }
  if (overlaps(o, qb, lse, lb)) return ATTN_ERR_INVALID_ARG;
  if ((st = check_device()) != ATTN_OK) return st;

  attn::FwdArgs a{};
  const bool bf16 = dt == ATTN_BF16;
  const int BH = B * H;
  if (!make_map(&a.tm_q, q, BH, N, d, bf16) || !make_map(&a.tm_k, k, BH, Nk, d, bf16) ||
      !make_map(&a.tm_v, v, BH, Nk, d, bf16) || !make_map(&a.tm_o, o, BH, N, d, bf16))
    return ATTN_ERR_CUDA;
  a.lse = lse;
  a.dev_status = dev_status;
  a.N = N;
  a.Nk = Nk;
  a.cofs = causal ? Nk - N : 0;
  a.BH = BH;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_limit_ns = wait_limit_ns();
  set_dropout(a, dr);
  a.keep_bits = keep_bits;
  a.bits_rows = static_cast<int>((static_cast<size_t>(N) + kTileM - 1) / kTileM * kTileM);
  const bool pair = d == 128 && dr.t == 0 && fwd_use_pair(Nk, causal);
  if (pair && !make_map(&a.tm_kh, k, BH, Nk, d, bf16, 64)) return ATTN_ERR_CUDA;
  const bool persist = d == 64 && dr.t == 0 && fwd_use_persist(N);
  const cudaError_t e = d == 256  ? attn::launch_fwd256(a, bf16, static_cast<cudaStream_t>(stream))
                        : dr.t > 0 ? attn::launch_fwd_dropout(a, d, bf16, static_cast<cudaStream_t>(stream))
                        : pair     ? attn::launch_fwd_pair(a, bf16, static_cast<cudaStream_t>(stream))
                        : persist  ? attn::launch_fwd_persist(a, bf16, static_cast<cudaStream_t>(stream))
                                   : attn::launch_fwd(a, d, bf16, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                     int d, attn_dtype dt, int causal, float scale, int* dev_status, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, N, N, d, dt, causal, scale, dev_status, stream);
}

attn_status attn_fwd_rect(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                          int Nk, int d, attn_dtype dt, int causal, float scale, int* dev_status, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, Nq, Nk, d, dt, causal, scale, dev_status, stream);
}

}  // extern "C"

namespace {

// The packed-batch forward, with or without dropout; n_splits > 0: split-KV through the
// workspace (no dropout then).
attn_status fwd_varlen_impl(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_q,
                            const int* cu_k, int B, int H, int max_q, int max_k, int Tq, int Tk, int d,
                            attn_dtype dt, int causal, float scale, int* dev_status, void* stream,
                            const Dropout& dr, void* workspace = nullptr, size_t workspace_bytes = 0,
                            int n_splits = 0) {
  attn_status st = check_sizes(1, H, Tq > Tk ? Tq : Tk, d, dt, scale, true);  // d = 256 too
  if (st != ATTN_OK) return st;
  if (B < 1 || max_q < 1 || max_k < 1 || Tq < 1 || Tk < 1) return ATTN_ERR_INVALID_ARG;
  if (n_splits < 0 || n_splits > 64 || (n_splits > 0 && dr.t > 0)) return ATTN_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * H * ((max_q + 127) / 128) * (n_splits > 0 ? n_splits : 1) >= (int64_t(1) << 31))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned4(cu_q) ||
      !aligned4(cu_k) || (n_splits > 0 && !aligned16(workspace)))
    return ATTN_ERR_INVALID_ARG;
  const size_t qb = static_cast<size_t>(Tq) * H * d * 2, kb = static_cast<size_t>(Tk) * H * d * 2;
  const size_t lb = static_cast<size_t>(H) * Tq * 4, cb = static_cast<size_t>(B + 1) * 4;
  const size_t wb = n_splits > 0 ? attn_fwd_varlen_splitkv_workspace_bytes(H, Tq, d, n_splits) : 0;
  if (n_splits > 0 && (wb == 0 || workspace_bytes < wb)) return ATTN_ERR_INVALID_ARG;
  for (const void* in : {q, k, v, static_cast<const void*>(cu_q), static_cast<const void*>(cu_k)}) {
    const size_t ib = in == q ? qb : (in == k || in == v) ? kb : cb;
    if (overlaps(in, ib, o, qb) || overlaps(in, ib, lse, lb) || (wb && overlaps(in, ib, workspace, wb)))
      return ATTN_ERR_INVALID_ARG;
  }
  if (overlaps(o, qb, lse, lb)) return ATTN_ERR_INVALID_ARG;
  if (wb && (overlaps(o, qb, workspace, wb) || overlaps(lse, lb, workspace, wb))) return ATTN_ERR_INVALID_ARG;
  if ((st = check_device()) != ATTN_OK) return st;

  attn::FwdArgs a{};
  const bool bf16 = dt == ATTN_BF16;
  if (!make_map_packed(&a.tm_q, q, H, Tq, d, bf16) || !make_map_packed(&a.tm_k, k, H, Tk, d, bf16) ||
      !make_map_packed(&a.tm_v, v, H, Tk, d, bf16) || !make_map_packed(&a.tm_o, o, H, Tq, d, bf16))
    return ATTN_ERR_CUDA;
  a.o = o;
  a.lse = lse;
  a.dev_status = dev_status;
  a.N = max_q;
  a.Nk = max_k;
  a.BH = B * H;
  a.H = H;
  a.Tq = Tq;
  a.cu_q = cu_q;
  a.cu_k = cu_k;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_limit_ns = wait_limit_ns();
  set_dropout(a, dr);
  if (n_splits > 0) {
    a.n_splits = n_splits;
    a.part_o = static_cast<float*>(workspace);
    a.part_lse = static_cast<float*>(workspace) + static_cast<size_t>(n_splits) * Tq * H * d;
    if (attn::launch_fwd_varlen_split(a, d, bf16, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  const cudaError_t e = d == 256 ? attn::launch_fwd256_varlen(a, bf16, static_cast<cudaStream_t>(stream))
                                 : attn::launch_fwd_varlen(a, d, bf16, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_q,
                            const int* cu_k, int B, int H, int max_q, int max_k, int Tq, int Tk, int d,
                            attn_dtype dt, int causal, float scale, int* dev_status, void* stream) {
  return fwd_varlen_impl(q, k, v, o, lse, cu_q, cu_k, B, H, max_q, max_k, Tq, Tk, d, dt, causal, scale, dev_status,
                         stream, Dropout{});
}

size_t attn_fwd_varlen_splitkv_workspace_bytes(int H, int Tq, int d, int n_splits) {
  if (H < 1 || Tq < 1 || (d != 64 && d != 128 && d != 256) || n_splits < 1 || n_splits > 64) return 0;
  return static_cast<size_t>(n_splits) * Tq * H * (static_cast<size_t>(d) + 1) * sizeof(float);
}

attn_status attn_fwd_varlen_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                                    void* workspace, size_t workspace_bytes, const int* cu_q, const int* cu_k,
                                    int B, int H, int max_q, int max_k, int Tq, int Tk, int d, attn_dtype dt,
                                    int causal, float scale, int n_splits, int* dev_status, void* stream) {
  if (n_splits < 1) return ATTN_ERR_INVALID_ARG;
  return fwd_varlen_impl(q, k, v, o, lse, cu_q, cu_k, B, H, max_q, max_k, Tq, Tk, d, dt, causal, scale, dev_status,
                         stream, Dropout{}, workspace, workspace_bytes, n_splits);
}

attn_status attn_fwd_varlen_dropout(const void* q, const void* k, const void* v, void* o, float* lse,
                                    const int* cu_q, const int* cu_k, int B, int H, int max_q, int max_k, int Tq,
                                    int Tk, int d, attn_dtype dt, int causal, float scale, float p_drop,
                                    uint64_t seed, int* dev_status, void* stream) {
  Dropout dr;
  if (!dropout_from_p(p_drop, seed, &dr)) return ATTN_ERR_INVALID_ARG;
  return fwd_varlen_impl(q, k, v, o, lse, cu_q, cu_k, B, H, max_q, max_k, Tq, Tk, d, dt, causal, scale, dev_status,
                         stream, dr);
}

attn_status attn_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                             int d, attn_dtype dt, int causal, float scale, float p_drop, uint64_t seed,
                             int* dev_status, void* stream) {
  Dropout dr;
  if (!dropout_from_p(p_drop, seed, &dr)) return ATTN_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, B, H, N, N, d, dt, causal, scale, dev_status, stream, dr);
}

size_t attn_dropout_bits_bytes(int B, int H, int Nq, int Nk) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return 0;
  const size_t rows = (static_cast<size_t>(Nq) + kTileM - 1) / kTileM * kTileM;
  const size_t tiles = (static_cast<size_t>(Nk) + kTileM - 1) / kTileM;
  return static_cast<size_t>(B) * H * tiles * 4 * rows * sizeof(uint32_t);
}

attn_status attn_fwd_dropout_bits(const void* q, const void* k, const void* v, void* o, float* lse, void* keep_bits,
                                  size_t keep_bits_bytes, int B, int H, int N, int d, attn_dtype dt, int causal,
                                  float scale, float p_drop, uint64_t seed, int* dev_status, void* stream) {
  Dropout dr;
  if (!dropout_from_p(p_drop, seed, &dr) || dr.t == 0) return ATTN_ERR_INVALID_ARG;
  const size_t need = attn_dropout_bits_bytes(B, H, N, N);
  if (need == 0 || keep_bits_bytes < need || !aligned16(keep_bits)) return ATTN_ERR_INVALID_ARG;
  if (d == 256) return ATTN_ERR_UNSUPPORTED;
  const size_t qb = static_cast<size_t>(B) * H * N * d * 2, lb = static_cast<size_t>(B) * H * N * 4;
  for (const Buf& b : {Buf{q, qb}, Buf{k, qb}, Buf{v, qb}, Buf{o, qb}, Buf{lse, lb}})
    if (b.p && overlaps(b.p, b.bytes, keep_bits, need)) return ATTN_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, B, H, N, N, d, dt, causal, scale, dev_status, stream, dr,
                  static_cast<uint32_t*>(keep_bits));
}

attn_status attn_fwd_rect_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                  int Nq, int Nk, int d, attn_dtype dt, int causal, float scale, float p_drop,
                                  uint64_t seed, int* dev_status, void* stream) {
  Dropout dr;
  if (!dropout_from_p(p_drop, seed, &dr)) return ATTN_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, B, H, Nq, Nk, d, dt, causal, scale, dev_status, stream, dr);
}

attn_status attn_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* q_scale,
                         const float* k_scale, const float* v_scale, void* o, float* lse, int B, int H, int N,
                         int d, attn_dtype out_dt, int causal, float scale, int* dev_status, void* stream) {
  attn_status st = check_sizes(B, H, N, d, out_dt, scale);
  if (st != ATTN_OK) return st;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned4(q_scale) || !aligned4(k_scale) || !aligned4(v_scale)) return ATTN_ERR_INVALID_ARG;
  const int n_t = (N + kTileM - 1) / kTileM;
  const size_t ib = static_cast<size_t>(B) * H * N * d, ob = ib * 2, lb = static_cast<size_t>(B) * H * N * 4;
  const size_t sb = static_cast<size_t>(B) * H * n_t * 4;
  for (const void* in : {q8, k8, v8})
    if (overlaps(in, ib, o, ob) || overlaps(in, ib, lse, lb)) return ATTN_ERR_INVALID_ARG;
  for (const void* sc : {static_cast<const void*>(q_scale), static_cast<const void*>(k_scale),
                         static_cast<const void*>(v_scale)})
    if (overlaps(sc, sb, o, ob) || overlaps(sc, sb, lse, lb)) return ATTN_ERR_INVALID_ARG;
  if (overlaps(o, ob, lse, lb)) return ATTN_ERR_INVALID_ARG;
  if ((st = check_device()) != ATTN_OK) return st;

  attn::FwdArgs a{};
  const bool bf16 = out_dt == ATTN_BF16;
  const int BH = B * H;
  if (!make_map_e4m3(&a.tm_q, q8, BH, N, d) || !make_map_e4m3(&a.tm_k, k8, BH, N, d) ||
      !make_map_e4m3(&a.tm_v, v8, BH, N, d) || !make_map(&a.tm_o, o, BH, N, d, bf16))
    return ATTN_ERR_CUDA;
  a.o = o;
  a.lse = lse;
  a.dev_status = dev_status;
  a.N = N;
  a.Nk = N;
  a.BH = BH;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_limit_ns = wait_limit_ns();
  a.q_scale = q_scale;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  if (attn::launch_fwd_fp8(a, d, bf16, static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

size_t attn_fwd_splitkv_workspace_bytes(int B, int H, int N, int d, int n_splits) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128 && d != 256) || n_splits < 1 || n_splits > 64) return 0;
  return static_cast<size_t>(n_splits) * B * H * N * (static_cast<size_t>(d) + 1) * sizeof(float);
}

attn_status attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                             size_t workspace_bytes, int B, int H, int N, int d, attn_dtype dt, int causal,
                             float scale, int n_splits, int* dev_status, void* stream) {
  return attn_fwd_splitkv_rect(q, k, v, o, lse, workspace, workspace_bytes, B, H, N, N, d, dt, causal, scale,
                               n_splits, dev_status, stream);
}

attn_status attn_fwd_splitkv_rect(const void* q, const void* k, const void* v, void* o, float* lse,
                                  void* workspace, size_t workspace_bytes, int B, int H, int Nq, int Nk, int d,
                                  attn_dtype dt, int causal, float scale, int n_splits, int* dev_status,
                                  void* stream) {
  attn_status st = check_sizes(B, H, Nq, d, dt, scale, true, Nk);
  if (st != ATTN_OK) return st;
  if (causal && Nk < Nq) return ATTN_ERR_INVALID_ARG;
  if (n_splits < 1 || n_splits > 64) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(workspace))
    return ATTN_ERR_INVALID_ARG;
  const size_t need = attn_fwd_splitkv_workspace_bytes(B, H, Nq, d, n_splits);
  if (workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
  const size_t qb = static_cast<size_t>(B) * H * Nq * d * 2, kb = static_cast<size_t>(B) * H * Nk * d * 2;
  const size_t lb = static_cast<size_t>(B) * H * Nq * 4;
  const void* ins[] = {q, k, v};
  const size_t in_bytes[] = {qb, kb, kb};
  for (int i = 0; i < 3; ++i)
    if (overlaps(ins[i], in_bytes[i], o, qb) || overlaps(ins[i], in_bytes[i], lse, lb) ||
        overlaps(ins[i], in_bytes[i], workspace, need))
      return ATTN_ERR_INVALID_ARG;
  if (overlaps(o, qb, lse, lb) || overlaps(o, qb, workspace, need) || overlaps(lse, lb, workspace, need))
    return ATTN_ERR_INVALID_ARG;
  if ((st = check_device()) != ATTN_OK) return st;

  attn::FwdArgs a{};
  const bool bf16 = dt == ATTN_BF16;
  const int BH = B * H;
  if (!make_map(&a.tm_q, q, BH, Nq, d, bf16) || !make_map(&a.tm_k, k, BH, Nk, d, bf16) ||
      !make_map(&a.tm_v, v, BH, Nk, d, bf16) || !make_map(&a.tm_o, o, BH, Nq, d, bf16))
    return ATTN_ERR_CUDA;
  a.o = o;
  a.lse = lse;
  a.dev_status = dev_status;
  a.N = Nq;
  a.Nk = Nk;
  a.cofs = causal ? Nk - Nq : 0;
  a.BH = BH;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_limit_ns = wait_limit_ns();
  a.n_splits = n_splits;
  a.part_o = static_cast<float*>(workspace);
  a.part_lse = static_cast<float*>(workspace) + static_cast<size_t>(n_splits) * BH * Nq * d;
  if (attn::launch_fwd_split(a, d, bf16, static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

size_t attn_bwd_deterministic_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128 && d != 256)) return 0;
  const size_t npad = (static_cast<size_t>(N) + kTileM - 1) / kTileM * kTileM;
  return 2 * static_cast<size_t>(B) * H * npad * sizeof(float);
}

size_t attn_bwd_workspace_bytes(int B, int H, int N, int d) {
  const size_t base = attn_bwd_deterministic_workspace_bytes(B, H, N, d);
  if (base == 0 || d == 256) return base;
  // + the fused backward's float32 dQ accumulator, d values per padded row
  return base + base / 2 * static_cast<size_t>(d);
}

}  // extern "C"

namespace {


// Validation shared by the backward entry points: every input and output 16-byte
// aligned and non-null, no output overlapping an input, the logsumexp, the workspace
// or another output, and (when the call writes the workspace) no input or the
// logsumexp inside the workspace, which must hold `need` bytes (the workspace size of the
// path the call takes).
attn_status check_bwd(std::initializer_list<Buf> ins, const float* lse, std::initializer_list<Buf> outs,
                      const void* ws, size_t ws_bytes, bool ws_out, int B, int H, int N, int Nk, int d,
                      attn_dtype dt, float scale, int causal, size_t need) {
  attn_status st = check_sizes(B, H, N, d, dt, scale, true, Nk);
  if (st != ATTN_OK) return st;
  if (causal && Nk < N) return ATTN_ERR_INVALID_ARG;
  for (const Buf& b : ins)
    if (!aligned16(b.p)) return ATTN_ERR_INVALID_ARG;
  for (const Buf& b : outs)
    if (!aligned16(b.p)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(ws)) return ATTN_ERR_INVALID_ARG;
  if (lse && !aligned16(lse)) return ATTN_ERR_INVALID_ARG;
  if (need == 0 || ws_bytes < need) return ATTN_ERR_INVALID_ARG;
  const size_t lb = static_cast<size_t>(B) * H * N * 4;
  const std::vector<Buf> o(outs);
  for (size_t i = 0; i < o.size(); ++i) {
    for (const Buf& in : ins)
      if (overlaps(in.p, in.bytes, o[i].p, o[i].bytes)) return ATTN_ERR_INVALID_ARG;
    if ((lse && overlaps(lse, lb, o[i].p, o[i].bytes)) || overlaps(ws, need, o[i].p, o[i].bytes))
      return ATTN_ERR_INVALID_ARG;
    for (size_t j = i + 1; j < o.size(); ++j)  // identical pointers are an overlap too
      if (o[i].p == o[j].p || overlaps(o[i].p, o[i].bytes, o[j].p, o[j].bytes)) return ATTN_ERR_INVALID_ARG;
  }
  if (ws_out) {
    for (const Buf& in : ins)
      if (overlaps(in.p, in.bytes, ws, need)) return ATTN_ERR_INVALID_ARG;
    if (lse && overlaps(lse, lb, ws, need)) return ATTN_ERR_INVALID_ARG;
  }
  return check_device();
}

void fill_bwd(attn::BwdArgs& a, const void* ws, int B, int H, int N, int Nk, int causal, float scale,
              int* dev_status, const Dropout& dr = Dropout{}) {
  set_dropout(a, dr);
  const int BH = B * H;
  const int npad = static_cast<int>((static_cast<size_t>(N) + kTileM - 1) / kTileM * kTileM);
  a.lse2 = static_cast<float*>(const_cast<void*>(ws));
  a.delta = static_cast<float*>(const_cast<void*>(ws)) + static_cast<size_t>(BH) * npad;
  a.dev_status = dev_status;
  a.N = N;
  a.Nk = Nk;
  a.cofs = causal ? Nk - N : 0;
  a.Npad = npad;
  a.BH = BH;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_limit_ns = wait_limit_ns();
}

size_t qbytes(int B, int H, int N, int d) { return static_cast<size_t>(B) * H * N * d * 2; }

// The fused backward's dQ accumulator: the d float32 values per padded row that follow
// the two per-row values in a workspace of attn_bwd_workspace_bytes().
float* dq_accumulator(void* ws, int B, int H, int N) {
  const size_t npad = (static_cast<size_t>(N) + kTileM - 1) / kTileM * kTileM;
  return static_cast<float*>(ws) + 2 * static_cast<size_t>(B) * H * npad;
}

// Fills the per-row values (and, when the workspace holds the fused backward's dQ
// accumulator, clears the accumulator).
attn_status prepare_impl(const void* o, const void* dout, const float* lse, void* workspace, size_t workspace_bytes,
                         int B, int H, int N, int d, attn_dtype dt, void* stream) {
  if (!lse) return ATTN_ERR_INVALID_ARG;
  const size_t qb = qbytes(B, H, N, d);
  const size_t small = attn_bwd_deterministic_workspace_bytes(B, H, N, d);
  attn_status st = check_bwd({{o, qb}, {dout, qb}}, lse, {}, workspace, workspace_bytes, true, B, H, N, N, d, dt,
                             1.f, 0, small);
  if (st != ATTN_OK) return st;
  const size_t full = attn_bwd_workspace_bytes(B, H, N, d);
  const bool with_acc = d != 256 && workspace_bytes >= full;
  if (with_acc && (overlaps(o, qb, workspace, full) || overlaps(dout, qb, workspace, full) ||
                   overlaps(lse, static_cast<size_t>(B) * H * N * 4, workspace, full)))
    return ATTN_ERR_INVALID_ARG;
  attn::BwdArgs a{};
  fill_bwd(a, workspace, B, H, N, N, 0, 1.f, nullptr);
  a.dq_acc = with_acc ? dq_accumulator(workspace, B, H, N) : nullptr;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  if (attn::launch_bwd_pre(a, d, dt == ATTN_BF16, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

attn_status dkdv_impl(const void* q, const void* k, const void* v, const void* dout, const void* workspace,
                      size_t workspace_bytes, void* dk, void* dv, int B, int H, int N, int Nk, int d, attn_dtype dt,
                      int causal, float scale, int* dev_status, void* stream, const Dropout& dr = Dropout{}) {
  const size_t qb = qbytes(B, H, N, d), kb = qbytes(B, H, Nk, d);
  attn_status st = check_bwd({{q, qb}, {k, kb}, {v, kb}, {dout, qb}}, nullptr, {{dk, kb}, {dv, kb}}, workspace,
                             workspace_bytes, false, B, H, N, Nk, d, dt, scale, causal,
                             attn_bwd_deterministic_workspace_bytes(B, H, N, d));
  if (st != ATTN_OK) return st;
  attn::BwdArgs a{};
  const bool bf16 = dt == ATTN_BF16;
  const int BH = B * H;
  if (!make_map(&a.tm_q, q, BH, N, d, bf16) || !make_map(&a.tm_k, k, BH, Nk, d, bf16) ||
      !make_map(&a.tm_v, v, BH, Nk, d, bf16) || !make_map(&a.tm_do, dout, BH, N, d, bf16) ||
      !make_map(&a.tm_dk, dk, BH, Nk, d, bf16) || !make_map(&a.tm_dv, dv, BH, Nk, d, bf16))
    return ATTN_ERR_CUDA;
  fill_bwd(a, workspace, B, H, N, Nk, causal, scale, dev_status, dr);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool pair = d == 128 && dr.t == 0 && bwd_use_pair();
  if (pair && (!make_map(&a.tm_qh, q, BH, N, d, bf16, 64) || !make_map(&a.tm_doh, dout, BH, N, d, bf16, 64)))
    return ATTN_ERR_CUDA;
  const cudaError_t e = d == 256  ? attn::launch_bwd256_dkdv(a, bf16, s)
                        : pair    ? attn::launch_bwd_dkdv_pair(a, bf16, s)
                        : dr.t > 0 ? attn::launch_bwd_dkdv_dropout(a, d, bf16, s)
                                   : attn::launch_bwd_dkdv(a, d, bf16, s);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

attn_status dq_impl(const void* q, const void* k, const void* v, const void* dout, const void* workspace,
                    size_t workspace_bytes, void* dq, int B, int H, int N, int Nk, int d, attn_dtype dt, int causal,
                    float scale, int* dev_status, void* stream, const Dropout& dr = Dropout{}) {
  const size_t qb = qbytes(B, H, N, d), kb = qbytes(B, H, Nk, d);
  attn_status st = check_bwd({{q, qb}, {k, kb}, {v, kb}, {dout, qb}}, nullptr, {{dq, qb}}, workspace,
                             workspace_bytes, false, B, H, N, Nk, d, dt, scale, causal,
                             attn_bwd_deterministic_workspace_bytes(B, H, N, d));
  if (st != ATTN_OK) return st;
  attn::BwdArgs a{};
  const bool bf16 = dt == ATTN_BF16;
  const int BH = B * H;
  if (!make_map(&a.tm_q, q, BH, N, d, bf16) || !make_map(&a.tm_k, k, BH, Nk, d, bf16) ||
      !make_map(&a.tm_v, v, BH, Nk, d, bf16) || !make_map(&a.tm_do, dout, BH, N, d, bf16) ||
      !make_map(&a.tm_dq, dq, BH, N, d, bf16))
    return ATTN_ERR_CUDA;
  fill_bwd(a, workspace, B, H, N, Nk, causal, scale, dev_status, dr);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = d == 256 ? attn::launch_bwd256_dq(a, bf16, s)
                        : dr.t > 0 ? attn::launch_bwd_dq_dropout(a, d, bf16, s)
                                   : attn::launch_bwd_dq(a, d, bf16, s);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

// The fused stage: dK, dV and the dQ accumulator (the preparation pass, with the
// accumulator cleared, must have run on the same workspace).
attn_status fused_impl(const void* q, const void* k, const void* v, const void* dout, void* workspace,
                       size_t workspace_bytes, void* dk, void* dv, int B, int H, int N, int Nk, int d, attn_dtype dt,
                       int causal, float scale, int* dev_status, void* stream, const Dropout& dr = Dropout{},
                       const uint32_t* keep_bits = nullptr) {
  if (d == 256) return ATTN_ERR_UNSUPPORTED;
  const size_t qb = qbytes(B, H, N, d), kb = qbytes(B, H, Nk, d);
  attn_status st = check_bwd({{q, qb}, {k, kb}, {v, kb}, {dout, qb}}, nullptr, {{dk, kb}, {dv, kb}}, workspace,
                             workspace_bytes, true, B, H, N, Nk, d, dt, scale, causal,
                             attn_bwd_workspace_bytes(B, H, N, d));
  if (st != ATTN_OK) return st;
  attn::BwdArgs a{};
  const bool bf16 = dt == ATTN_BF16;
  const int BH = B * H;
  if (!make_map(&a.tm_q, q, BH, N, d, bf16) || !make_map(&a.tm_k, k, BH, Nk, d, bf16) ||
      !make_map(&a.tm_v, v, BH, Nk, d, bf16) || !make_map(&a.tm_do, dout, BH, N, d, bf16) ||
      !make_map(&a.tm_dk, dk, BH, Nk, d, bf16) || !make_map(&a.tm_dv, dv, BH, Nk, d, bf16))
    return ATTN_ERR_CUDA;
  fill_bwd(a, workspace, B, H, N, Nk, causal, scale, dev_status, dr);
  a.keep_bits = keep_bits;
  a.bits_rows = a.Npad;
  a.dq_acc = dq_accumulator(workspace, B, H, N);
  if (!make_map_acc(&a.tm_dqacc, a.dq_acc, static_cast<int64_t>(BH) * a.Npad, d)) return ATTN_ERR_CUDA;
  if (attn::launch_bwd_fused(a, d, bf16, false, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

// dQ = scale * accumulator, rounded to the 16-bit type.
attn_status finish_impl(const void* workspace, size_t workspace_bytes, void* dq, int B, int H, int N, int d,
                        attn_dtype dt, float scale, void* stream) {
  if (d == 256) return ATTN_ERR_UNSUPPORTED;
  const size_t qb = qbytes(B, H, N, d);
  attn_status st = check_bwd({}, nullptr, {{dq, qb}}, workspace, workspace_bytes, false, B, H, N, N, d, dt, scale,
                             0, attn_bwd_workspace_bytes(B, H, N, d));
  if (st != ATTN_OK) return st;
  attn::BwdArgs a{};
  fill_bwd(a, workspace, B, H, N, N, 0, scale, nullptr);
  a.dq_acc = dq_accumulator(const_cast<void*>(workspace), B, H, N);
  a.dq = dq;
  if (attn::launch_bwd_dq_finish(a, d, dt == ATTN_BF16, false, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

// The whole backward.  d <= 128 with dropout drawn here takes the fused path (five
// products per tile pair, the keep bits drawn once, dQ through a float32 accumulator);
// without dropout, or with the forward's stored keep bits (nothing to draw twice), the two
// deterministic kernels measured as fast or faster on this GPU (the fused kernel's dQ
// reductions compete with its shared-memory operand traffic) and run instead; d = 256
// uses its three deterministic kernels.
attn_status bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                     void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int N,
                     int Nk, int d, attn_dtype dt, int causal, float scale, int* dev_status, void* stream,
                     const Dropout& dr = Dropout{}, bool deterministic = false, const uint32_t* keep_bits = nullptr) {
  if (!lse) return ATTN_ERR_INVALID_ARG;
  const size_t qb = qbytes(B, H, N, d), kb = qbytes(B, H, Nk, d);
  const size_t need = deterministic ? attn_bwd_deterministic_workspace_bytes(B, H, N, d)
                                    : attn_bwd_workspace_bytes(B, H, N, d);
  attn_status st = check_bwd({{q, qb}, {k, kb}, {v, kb}, {o, qb}, {dout, qb}}, lse, {{dq, qb}, {dk, kb}, {dv, kb}},
                             workspace, workspace_bytes, true, B, H, N, Nk, d, dt, scale, causal, need);
  if (st != ATTN_OK) return st;
  const bool fused = !deterministic && d != 256 && dr.t > 0 && keep_bits == nullptr;
  // the deterministic path does not read past the per-row values: prepare only those
  const size_t prep_bytes = fused ? workspace_bytes : attn_bwd_deterministic_workspace_bytes(B, H, N, d);
  if ((st = prepare_impl(o, dout, lse, workspace, prep_bytes, B, H, N, d, dt, stream)) != ATTN_OK) return st;
  if (fused) {
    if ((st = fused_impl(q, k, v, dout, workspace, workspace_bytes, dk, dv, B, H, N, Nk, d, dt, causal, scale,
                         dev_status, stream, dr, keep_bits)) != ATTN_OK)
      return st;
    return finish_impl(workspace, workspace_bytes, dq, B, H, N, d, dt, scale, stream);
  }
  if (d == 256) {
    if ((st = dkdv_impl(q, k, v, dout, workspace, workspace_bytes, dk, dv, B, H, N, Nk, d, dt, causal, scale,
                        dev_status, stream, dr)) != ATTN_OK)
      return st;
    return dq_impl(q, k, v, dout, workspace, workspace_bytes, dq, B, H, N, Nk, d, dt, causal, scale, dev_status,
                   stream, dr);
  }
  // d <= 128: dK/dV and dQ as one grid (arguments already validated above)
  attn::BwdArgs a{};
  const bool bf16 = dt == ATTN_BF16;
  const int BH = B * H;
  if (!make_map(&a.tm_q, q, BH, N, d, bf16) || !make_map(&a.tm_k, k, BH, Nk, d, bf16) ||
      !make_map(&a.tm_v, v, BH, Nk, d, bf16) || !make_map(&a.tm_do, dout, BH, N, d, bf16) ||
      !make_map(&a.tm_dq, dq, BH, N, d, bf16) || !make_map(&a.tm_dk, dk, BH, Nk, d, bf16) ||
      !make_map(&a.tm_dv, dv, BH, Nk, d, bf16))
    return ATTN_ERR_CUDA;
  fill_bwd(a, workspace, B, H, N, Nk, causal, scale, dev_status, dr);
  a.keep_bits = keep_bits;
  a.bits_rows = a.Npad;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = dr.t > 0 ? attn::launch_bwd_grads_dropout(a, d, bf16, s) : attn::launch_bwd_grads(a, d, bf16, s);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

attn_status attn_bwd_prepare(const void* o, const void* dout, const float* lse, void* workspace,
                             size_t workspace_bytes, int B, int H, int N, int d, attn_dtype dt, void* stream) {
  return prepare_impl(o, dout, lse, workspace, workspace_bytes, B, H, N, d, dt, stream);
}

attn_status attn_bwd_dkdv(const void* q, const void* k, const void* v, const void* dout, const void* workspace,
                          size_t workspace_bytes, void* dk, void* dv, int B, int H, int N, int d, attn_dtype dt,
                          int causal, float scale, int* dev_status, void* stream) {
  return dkdv_impl(q, k, v, dout, workspace, workspace_bytes, dk, dv, B, H, N, N, d, dt, causal, scale, dev_status,
                   stream);
}

attn_status attn_bwd_dq(const void* q, const void* k, const void* v, const void* dout, const void* workspace,
                        size_t workspace_bytes, void* dq, int B, int H, int N, int d, attn_dtype dt, int causal,
                        float scale, int* dev_status, void* stream) {
  return dq_impl(q, k, v, dout, workspace, workspace_bytes, dq, B, H, N, N, d, dt, causal, scale, dev_status,
                 stream);
}

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                     int B, int H, int N, int d, attn_dtype dt, int causal, float scale, int* dev_status,
                     void* stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, N, d, dt, causal, scale,
                  dev_status, stream);
}

attn_status attn_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                   const float* lse, void* dq, void* dk, void* dv, void* workspace,
                                   size_t workspace_bytes, int B, int H, int N, int d, attn_dtype dt, int causal,
                                   float scale, int* dev_status, void* stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, N, d, dt, causal, scale,
                  dev_status, stream, Dropout{}, true);
}

attn_status attn_bwd_dkdvdq(const void* q, const void* k, const void* v, const void* dout, void* workspace,
                            size_t workspace_bytes, void* dk, void* dv, int B, int H, int N, int d, attn_dtype dt,
                            int causal, float scale, int* dev_status, void* stream) {
  return fused_impl(q, k, v, dout, workspace, workspace_bytes, dk, dv, B, H, N, N, d, dt, causal, scale, dev_status,
                    stream);
}

attn_status attn_bwd_dq_finish(const void* workspace, size_t workspace_bytes, void* dq, int B, int H, int N, int d,
                               attn_dtype dt, float scale, void* stream) {
  return finish_impl(workspace, workspace_bytes, dq, B, H, N, d, dt, scale, stream);
}

attn_status attn_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const void* dout,
                             const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                             int B, int H, int N, int d, attn_dtype dt, int causal, float scale, float p_drop,
                             uint64_t seed, int* dev_status, void* stream) {
  Dropout dr;
  if (!dropout_from_p(p_drop, seed, &dr)) return ATTN_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, N, d, dt, causal, scale,
                  dev_status, stream, dr);
}

attn_status attn_bwd_dropout_bits(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                  const float* lse, const void* keep_bits, size_t keep_bits_bytes, void* dq, void* dk,
                                  void* dv, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                                  attn_dtype dt, int causal, float scale, float p_drop, int* dev_status,
                                  void* stream) {
  Dropout dr;
  if (!dropout_from_p(p_drop, 0, &dr) || dr.t == 0) return ATTN_ERR_INVALID_ARG;
  const size_t need = attn_dropout_bits_bytes(B, H, N, N);
  if (need == 0 || keep_bits_bytes < need || !aligned16(keep_bits)) return ATTN_ERR_INVALID_ARG;
  if (d == 256) return ATTN_ERR_UNSUPPORTED;
  const size_t qb = static_cast<size_t>(B) * H * N * d * 2;
  for (const Buf& b : {Buf{dq, qb}, Buf{dk, qb}, Buf{dv, qb}, Buf{workspace, workspace_bytes}})
    if (b.p && overlaps(b.p, b.bytes, keep_bits, need)) return ATTN_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, N, N, d, dt, causal, scale,
                  dev_status, stream, dr, false, static_cast<const uint32_t*>(keep_bits));
}

}  // extern "C"

namespace {

// The packed-batch backward, with or without dropout.
attn_status bwd_varlen_impl(const void* q, const void* k, const void* v, const void* o, const void* dout,
                            const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                            const int* cu_q, const int* cu_k, int B, int H, int max_q, int max_k, int Tq, int Tk,
                            int d, attn_dtype dt, int causal, float scale, int* dev_status, void* stream,
                            const Dropout& dr) {
  attn_status st = check_sizes(1, H, Tq > Tk ? Tq : Tk, d, dt, scale, true);  // H * tokens * d < 2^31
  if (st != ATTN_OK) return st;
  if (B < 1 || max_q < 1 || max_k < 1 || Tq < 1 || Tk < 1) return ATTN_ERR_INVALID_ARG;
  const int64_t tiles = static_cast<int64_t>(B) * H * ((max_q > max_k ? max_q : max_k) + kTileM - 1) / kTileM;
  if (tiles >= (int64_t(1) << 31)) return ATTN_ERR_INVALID_ARG;  // grid sizes
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace) || !aligned4(cu_q) ||
      !aligned4(cu_k))
    return ATTN_ERR_INVALID_ARG;
  // the workspace rows are the padded rows of the longest sequence, per (sequence, head)
  const size_t need = attn_bwd_workspace_bytes(B, H, max_q, d);
  if (need == 0 || workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
  const size_t qb = static_cast<size_t>(Tq) * H * d * 2, kb = static_cast<size_t>(Tk) * H * d * 2;
  const size_t cb = static_cast<size_t>(B + 1) * 4, lb = static_cast<size_t>(H) * Tq * 4;
  const Buf ins[] = {{q, qb}, {k, kb}, {v, kb}, {o, qb}, {dout, qb}, {cu_q, cb}, {cu_k, cb}, {lse, lb}};
  const Buf outs[] = {{dq, qb}, {dk, kb}, {dv, kb}, {workspace, need}};
  for (int i = 0; i < 4; ++i) {
    for (const Buf& in : ins)
      if (overlaps(in.p, in.bytes, outs[i].p, outs[i].bytes)) return ATTN_ERR_INVALID_ARG;
    for (int j = i + 1; j < 4; ++j)
      if (overlaps(outs[i].p, outs[i].bytes, outs[j].p, outs[j].bytes)) return ATTN_ERR_INVALID_ARG;
  }
  if ((st = check_device()) != ATTN_OK) return st;

  attn::BwdArgs a{};
  const bool bf16 = dt == ATTN_BF16;
  if (!make_map_packed(&a.tm_q, q, H, Tq, d, bf16) || !make_map_packed(&a.tm_k, k, H, Tk, d, bf16) ||
      !make_map_packed(&a.tm_v, v, H, Tk, d, bf16) || !make_map_packed(&a.tm_do, dout, H, Tq, d, bf16))
    return ATTN_ERR_CUDA;
  fill_bwd(a, workspace, B, H, max_q, max_k, causal, scale, dev_status, dr);
  a.cofs = 0;  // per sequence, from the offsets
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.H = H;
  a.Tq = Tq;
  a.cu_q = cu_q;
  a.cu_k = cu_k;
  a.dq_out = dq;
  a.dk_out = dk;
  a.dv_out = dv;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d != 256 && dr.t > 0) {  // the fused path: dK, dV and a float32 dQ accumulator, then dQ from it
    a.dq_acc = dq_accumulator(workspace, B, H, max_q);
    a.dq = dq;
    if (!make_map_acc(&a.tm_dqacc, a.dq_acc, static_cast<int64_t>(B) * H * a.Npad, d)) return ATTN_ERR_CUDA;
    if (attn::launch_bwd_pre_varlen(a, d, bf16, s) != cudaSuccess ||
        attn::launch_bwd_fused(a, d, bf16, true, s) != cudaSuccess ||
        attn::launch_bwd_dq_finish(a, d, bf16, true, s) != cudaSuccess)
      return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  if (attn::launch_bwd_pre_varlen(a, d, bf16, s) != cudaSuccess) return ATTN_ERR_CUDA;
  const cudaError_t e = d == 256 ? (attn::launch_bwd256_dkdv_varlen(a, bf16, s) == cudaSuccess
                                        ? attn::launch_bwd256_dq_varlen(a, bf16, s)
                                        : cudaErrorLaunchFailure)
                                 : (attn::launch_bwd_dkdv_varlen(a, d, bf16, s) == cudaSuccess
                                        ? attn::launch_bwd_dq_varlen(a, d, bf16, s)
                                        : cudaErrorLaunchFailure);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dout,
                            const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                            const int* cu_q, const int* cu_k, int B, int H, int max_q, int max_k, int Tq, int Tk,
                            int d, attn_dtype dt, int causal, float scale, int* dev_status, void* stream) {
  return bwd_varlen_impl(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, cu_q, cu_k, B, H, max_q,
                         max_k, Tq, Tk, d, dt, causal, scale, dev_status, stream, Dropout{});
}

attn_status attn_bwd_varlen_dropout(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                    const float* lse, void* dq, void* dk, void* dv, void* workspace,
                                    size_t workspace_bytes, const int* cu_q, const int* cu_k, int B, int H,
                                    int max_q, int max_k, int Tq, int Tk, int d, attn_dtype dt, int causal,
                                    float scale, float p_drop, uint64_t seed, int* dev_status, void* stream) {
  Dropout dr;
  if (!dropout_from_p(p_drop, seed, &dr)) return ATTN_ERR_INVALID_ARG;
  return bwd_varlen_impl(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, cu_q, cu_k, B, H, max_q,
                         max_k, Tq, Tk, d, dt, causal, scale, dev_status, stream, dr);
}

attn_status attn_bwd_rect(const void* q, const void* k, const void* v, const void* o, const void* dout,
                          const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                          int B, int H, int Nq, int Nk, int d, attn_dtype dt, int causal, float scale,
                          int* dev_status, void* stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, Nq, Nk, d, dt, causal, scale,
                  dev_status, stream);
}

attn_status attn_bwd_rect_dropout(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                  const float* lse, void* dq, void* dk, void* dv, void* workspace,
                                  size_t workspace_bytes, int B, int H, int Nq, int Nk, int d, attn_dtype dt,
                                  int causal, float scale, float p_drop, uint64_t seed, int* dev_status,
                                  void* stream) {
  Dropout dr;
  if (!dropout_from_p(p_drop, seed, &dr)) return ATTN_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, Nq, Nk, d, dt, causal, scale,
                  dev_status, stream, dr);
}

attn_status attn_selftest_bounded_wait(int* dev_status, uint64_t limit_ns, void* stream) {
  if (!dev_status) return ATTN_ERR_INVALID_ARG;
  if (limit_ns < 1000ull) limit_ns = 1000ull;
  if (limit_ns > 1000000000ull) limit_ns = 1000000000ull;
  attn_status st = check_device();
  if (st != ATTN_OK) return st;
  if (attn::launch_wait_selftest(dev_status, limit_ns, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // extern "C"
