// The C ABI of libkdkl.so (declared in include/kdkl.h): argument checks,
// workspace layout, TMA descriptor set-up and the chunk loop that drives the
// kernels.  Host code only; every arithmetic step runs in the kernels.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "kd_host_state.h"
#include "kd_internal.h"

namespace kd {

// ------------------------------------------------------------ profiling ---

struct ProfRec {
  const char* name;
  cudaEvent_t start, stop;
};
static std::vector<ProfRec> g_prof;
static int g_prof_used = 0;
static bool g_prof_on = false;

void prof_before(const char* name, cudaStream_t s) {
  if (!g_prof_on || g_prof_used >= int(g_prof.size())) return;
  g_prof[g_prof_used].name = name;
  cudaEventRecord(g_prof[g_prof_used].start, s);
}

void prof_after(cudaStream_t s) {
  if (!g_prof_on || g_prof_used >= int(g_prof.size())) return;
  cudaEventRecord(g_prof[g_prof_used].stop, s);
  ++g_prof_used;
}

// ------------------------------------------------------------ tensor maps ---

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

static bool load_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

static bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                         uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  if (!load_encode()) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_mn2_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint64_t row_stride_bytes,
                        uint32_t box_rows) {
  if (!load_encode() || cols % 64 != 0) return false;
  const cuuint64_t dims[3] = {64, rows, cols / 64};
  const cuuint64_t strides[2] = {row_stride_bytes, 128};
  const cuuint32_t box[3] = {64, box_rows, 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_dz_blocked(CUtensorMap* map, const void* base, uint64_t rows, uint64_t rows_pad, uint64_t nvb,
                          uint32_t box_rows, uint32_t box_depth) {
  if (!load_encode()) return false;
  const cuuint64_t dims[3] = {64, rows, nvb};
  const cuuint64_t strides[2] = {128, rows_pad * 128};
  const cuuint32_t box[3] = {64, box_rows, box_depth};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                       uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  return make_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, inner, outer, row_stride_bytes, box_inner,
                      box_outer);
}

bool make_tmap_2d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                      uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  return make_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, inner, outer, row_stride_bytes, box_inner,
                      box_outer);
}

// ---------------------------------------------------------- device check ---

static PerDevice<int> g_dev_ok;  // per device: 1 = sm_103, 0 = another architecture

// The current device is an sm_103 GPU (the kernels are built for sm_103a only).
static kd_status check_device() {
  int dev = 0, ok = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KD_ERR_CUDA;
  const int rc = g_dev_ok.get(dev, &ok, [](int d, int* v) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess)
      return 1;
    *v = (major == 10 && minor == 3) ? 1 : 0;
    return 0;
  });
  if (rc < 0) return KD_ERR_UNSUPPORTED;  // an ordinal beyond the per-device tables
  if (rc > 0) return KD_ERR_CUDA;
  return ok ? KD_OK : KD_ERR_UNSUPPORTED;
}

// -------------------------------------------------------------- layout ---

static inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct KlLayout {
  size_t ids_sorted, p_sorted, negent, kl, partials, dz, gh_part, total;
  int64_t ldz, rows_pad, nvb;
  int n_groups;
};

static int choose_n_group(int64_t V) {
  (void)V;
  return 1;
}

static KlLayout kl_layout(int64_t N, int64_t d, int64_t V, int K, int64_t chunk) {
  KlLayout L{};
  const int64_t c = chunk < N ? chunk : N;
  L.rows_pad = (c + BM - 1) / BM * BM;
  L.ldz = (V + 7) / 8 * 8;
  const int n_tiles = int((V + BN - 1) / BN);
  const int g = choose_n_group(V);
  L.n_groups = (n_tiles + g - 1) / g;
  size_t off = sizeof(Ctrl);
  L.ids_sorted = off; off = align_up(off + size_t(L.rows_pad) * K * 4, 256);
  L.p_sorted = off;   off = align_up(off + size_t(L.rows_pad) * K * 4, 256);
  L.negent = off;     off = align_up(off + size_t(L.rows_pad) * 4, 256);
  L.kl = off;         off = align_up(off + size_t(N) * 4, 256);
  L.partials = off;   off = align_up(off + size_t(L.n_groups) * L.rows_pad * 16, 256);
  L.nvb = (V + 63) / 64;
  L.dz = off;         off = align_up(off + size_t(L.nvb) * L.rows_pad * 128, 256);
  L.gh_part = off;    off = align_up(off + size_t(KD_MAX_SPLITS) * L.rows_pad * size_t(d) * 4, 256);
  L.total = off;
  return L;
}

// CTA pairs (GemmProblem::cta_pair, clusters of two) for every launch with at least two
// row tiles (measured on the gpt-oss shape: 342k against 295k tokens/s for single-CTA
// tiles).  The loss epilogues also need an even number of row tiles (no phantom tile
// writing past the chunk); the gradient products check their rows themselves.
static void set_cluster(GemmProblem& p) {
  const bool loss_epi = (p.epi == EPI_LSE || p.epi == EPI_DZ || p.epi == EPI_LSE_Z);
  p.cta_pair = (p.m_tiles >= 2 && !(loss_epi && p.m_tiles % 2 != 0)) ? 1 : 0;
  p.cluster = p.cta_pair ? 2 : 1;
}

// Number of K splits for a product of `tiles` output tiles with `k_blocks` steps of
// BK each: the fewest waves of `grid` persistent CTAs per unit of work, with a small
// charge per split for the extra partial traffic.
// The loss sweeps and the teacher projection (both operands K-major) build depth-2
// K-major boxes (a_k3d / b_k3d) for CTA pairs.
static_assert(pair_kblocks(0, 0) == 2, "K-major operand pairs take two k-blocks per pair stage");

static int choose_splits(int64_t tiles, int k_blocks, int grid) {
  int best = 1;
  double best_cost = 1e300;
  for (int S = 1; S <= KD_MAX_SPLITS; ++S) {
    if (S > 1 && k_blocks / S < 32) break;
    const double waves = double((tiles * S + grid - 1) / grid) / S;
    const double cost = waves * (1.0 + 0.005 * (S - 1));
    if (cost < best_cost - 1e-12) {
      best_cost = cost;
      best = S;
    }
  }
  return best;
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static kd_status check_kl_args(const void* H, const void* W, const int32_t* ids, const float* tlog, int64_t N,
                               int64_t d, int64_t V, int K, int64_t chunk, float tau, const void* ws,
                               size_t ws_bytes) {
  if (N < 1 || d < 8 || V < 1 || K < 1 || chunk < BM) return KD_ERR_INVALID_ARG;
  if (d % 8 != 0 || chunk % BM != 0) return KD_ERR_INVALID_ARG;
  if (K > KD_MAX_K || int64_t(K) > V) return KD_ERR_INVALID_ARG;
  if (V > 0x7fffffffLL || N > 0x7fffffffLL || d > 0x7fffffffLL) return KD_ERR_INVALID_ARG;
  if (!(tau > 0.f) || !isfinite(tau)) return KD_ERR_INVALID_ARG;
  if (!H || !W || !ids || !tlog) return KD_ERR_INVALID_ARG;
  if (!aligned(H, 16) || !aligned(W, 16) || !aligned(ids, 4) || !aligned(tlog, 4)) return KD_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return KD_ERR_WORKSPACE;
  if (ws_bytes < kl_layout(N, d, V, K, chunk).total) return KD_ERR_WORKSPACE;
  return KD_OK;
}

static kd_status map_cuda(cudaError_t e) { return e == cudaSuccess ? KD_OK : KD_ERR_CUDA; }

}  // namespace kd

using namespace kd;

extern "C" {

const char* kd_status_string(int status) {
  switch (status) {
    case KD_OK: return "KD_OK";
    case KD_ERR_INVALID_ARG: return "KD_ERR_INVALID_ARG";
    case KD_ERR_UNSUPPORTED: return "KD_ERR_UNSUPPORTED";
    case KD_ERR_WORKSPACE: return "KD_ERR_WORKSPACE";
    case KD_ERR_CUDA: return "KD_ERR_CUDA";
    case KD_ERR_TIMEOUT: return "KD_ERR_TIMEOUT";
    case KD_ERR_DEVICE: return "KD_ERR_DEVICE";
    case KD_ERR_IO: return "KD_ERR_IO";
    default: return "KD_ERR_UNKNOWN";
  }
}

int kd_version(void) { return 100; }

size_t kd_topk_cache_workspace(int64_t N, int64_t V, int K) {
  (void)V;
  if (N < 1 || K < 1) return sizeof(Ctrl);
  return sizeof(Ctrl) + align_up(topk_scratch_bytes(N, K), 256);
}

int kd_topk_cache(const void* logits_bf16, int64_t N, int64_t V, int64_t ld, int K, int32_t* ids_out,
                  float* vals_out, float* lse_out, float* dropped_out, void* ws, size_t ws_bytes, void* stream) {
  if (N < 1 || V < 1 || K < 1 || K > KD_MAX_K || int64_t(K) > V || ld < V) return KD_ERR_INVALID_ARG;
  if (V > 0x7fffffffLL || ld % 8 != 0) return KD_ERR_INVALID_ARG;
  if (!logits_bf16 || !ids_out || !vals_out) return KD_ERR_INVALID_ARG;
  if (!aligned(logits_bf16, 16) || !aligned(ids_out, 4) || !aligned(vals_out, 4)) return KD_ERR_INVALID_ARG;
  if ((lse_out && !aligned(lse_out, 4)) || (dropped_out && !aligned(dropped_out, 4))) return KD_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256) || ws_bytes < kd_topk_cache_workspace(N, V, K)) return KD_ERR_WORKSPACE;
  kd_status st = check_device();
  if (st != KD_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Ctrl* ctrl = static_cast<Ctrl*>(ws);
  return map_cuda(launch_topk(static_cast<const uint16_t*>(logits_bf16), N, V, ld, K, ids_out, vals_out, lse_out,
                              dropped_out, &ctrl->err, static_cast<uint8_t*>(ws) + sizeof(Ctrl), s));
}

size_t kd_fused_kl_workspace(int64_t N, int64_t d, int64_t V, int K, int64_t chunk) {
  if (N < 1 || d < 1 || V < 1 || K < 1 || chunk < 1) return 0;
  return kl_layout(N, d, V, K, chunk).total;
}

// Teacher workspace: control block | the chunk's bf16 logits [rows_pad, ldz] | per-tile row
// maxima [rows_pad, ldt] | per-tile row sums [rows_pad, ldt] (fp32) | the chunk's row
// logsumexp [rows_pad] | the top-K scratch of one chunk.
static size_t teacher_topk_ws(int64_t N, int64_t V, int K, int64_t chunk) {
  const int64_t c = chunk < N ? chunk : N;
  const int64_t rows_pad = (c + BM - 1) / BM * BM;
  const int64_t ldz = (V + 7) / 8 * 8;
  const int64_t ldt = ((V + BN - 1) / BN + 7) / 8 * 8;  // per-tile row maxima of the logits
  return sizeof(Ctrl) + align_up(size_t(rows_pad) * size_t(ldz) * 2, 256) +
         align_up(size_t(rows_pad) * size_t(ldt) * 2, 256) + align_up(size_t(rows_pad) * size_t(ldt) * 4, 256) +
         align_up(size_t(rows_pad) * 4, 256) + align_up(topk_scratch_bytes(c, K), 256);
}

size_t kd_teacher_topk_workspace(int64_t N, int64_t dt, int64_t V, int K, int64_t chunk) {
  if (N < 1 || dt < 1 || V < 1 || K < 1 || chunk < 1) return 0;
  return teacher_topk_ws(N, V, K, chunk);
}

int kd_teacher_topk(const void* Ht_bf16, const void* Wt_bf16, int64_t N, int64_t dt, int64_t V, int K,
                    int64_t chunk, int32_t* ids_out, float* vals_out, float* lse_out, float* dropped_out, void* ws,
                    size_t ws_bytes, void* stream) {
  if (N < 1 || dt < 8 || dt % 8 != 0 || V < 1 || K < 1 || K > KD_MAX_K || int64_t(K) > V) return KD_ERR_INVALID_ARG;
  if (chunk < BM || chunk % BM != 0 || V > 0x7fffffffLL || N > 0x7fffffffLL || dt > 0x7fffffffLL)
    return KD_ERR_INVALID_ARG;
  if (!Ht_bf16 || !Wt_bf16 || !ids_out || !vals_out) return KD_ERR_INVALID_ARG;
  if (!aligned(Ht_bf16, 16) || !aligned(Wt_bf16, 16) || !aligned(ids_out, 4) || !aligned(vals_out, 4))
    return KD_ERR_INVALID_ARG;
  if ((lse_out && !aligned(lse_out, 4)) || (dropped_out && !aligned(dropped_out, 4))) return KD_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return KD_ERR_WORKSPACE;
  if (ws_bytes < teacher_topk_ws(N, V, K, chunk)) return KD_ERR_WORKSPACE;
  kd_status st = check_device();
  if (st != KD_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(w8);
  uint16_t* zbuf = reinterpret_cast<uint16_t*>(w8 + sizeof(Ctrl));
  const int64_t ldz = (V + 7) / 8 * 8;
  // each chunk row's maximum over every BN-column tile of its logits, from the projection's
  // epilogue: their K-th largest starts the row's top-K selection
  const int ntiles = int((V + BN - 1) / BN);
  const int64_t ldt = (int64_t(ntiles) + 7) / 8 * 8;
  const int64_t crows = chunk < N ? chunk : N;
  const size_t rows_pad = size_t((crows + BM - 1) / BM * BM);
  uint16_t* tmax = reinterpret_cast<uint16_t*>(w8 + sizeof(Ctrl) + align_up(rows_pad * size_t(ldz) * 2, 256));
  float* tsum = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(tmax) + align_up(rows_pad * size_t(ldt) * 2, 256));
  float* lse_chunk = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(tsum) + align_up(rows_pad * size_t(ldt) * 4, 256));
  void* tk_scratch = reinterpret_cast<uint8_t*>(lse_chunk) + align_up(rows_pad * 4, 256);
  // the row logsumexp (asked for, or needed by the dropped mass) comes from the projection's
  // epilogue in per-tile pieces, so that the selection below runs without it
  const bool tile_lse = (lse_out != nullptr || dropped_out != nullptr) && topk_takes_known_lse(K);
  const uint16_t* Ht = static_cast<const uint16_t*>(Ht_bf16);
  const int grid_max = gemm_max_grid();
  // Wt boxes: BN rows for single CTAs, BN / 2 for a CTA pair's halves
  alignas(64) CUtensorMap tw[2], th, tw2, th2;
  for (int i = 0; i < 2; ++i)
    if (!make_tmap_2d_bf16(&tw[i], Wt_bf16, uint64_t(dt), uint64_t(V), uint64_t(dt) * 2, BK, BN >> i))
      return KD_ERR_CUDA;
  const bool dt64 = dt % 64 == 0;  // two k-blocks per box for CTA pairs
  if (dt64 && !make_tmap_mn2_bf16(&tw2, Wt_bf16, uint64_t(dt), uint64_t(V), uint64_t(dt) * 2, BN / 2))
    return KD_ERR_CUDA;
  for (int64_t c0 = 0; c0 < N; c0 += chunk) {
    const int n = int((N - c0) < chunk ? (N - c0) : chunk);
    // the chunk's teacher logits, fp32 on the tensor cores, rounded once to bf16
    if (!make_tmap_2d_bf16(&th, Ht + c0 * dt, uint64_t(dt), uint64_t(n), uint64_t(dt) * 2, BK, BM))
      return KD_ERR_CUDA;
    if (dt64 && !make_tmap_mn2_bf16(&th2, Ht + c0 * dt, uint64_t(dt), uint64_t(n), uint64_t(dt) * 2, BM))
      return KD_ERR_CUDA;
    GemmProblem p{};
    p.M = n; p.N = int(V); p.K = int(dt);
    p.a_mn = 0; p.b_mn = 0; p.epi = EPI_STORE;
    p.m_tiles = (n + BM - 1) / BM;
    p.n_tiles = int((V + BN - 1) / BN);
    p.n_group = 1;
    p.k_splits = 1;
    set_cluster(p);
    p.n_units = ((p.m_tiles + p.cluster - 1) / p.cluster) * p.n_tiles;
    p.C = zbuf; p.ldc = ldz; p.c_bf16 = 1; p.err = &ctrl->err;
    p.c_tma = 1;   // bf16 logits written as TMA boxes into the row-major chunk buffer
    p.tile_max = tmax;
    p.ld_tile_max = ldt;
    p.tile_sum = tile_lse ? tsum : nullptr;
    p.m_fast = 1;  // Wt (larger than L2) read once per chunk, the chunk of Ht kept in L2
    alignas(64) CUtensorMap tz;
    if (!make_tmap_2d_bf16(&tz, zbuf, uint64_t(V), uint64_t(n), uint64_t(ldz) * 2, 64, 32)) return KD_ERR_CUDA;
    p.a_k3d = p.b_k3d = p.cta_pair && dt64;
    cudaError_t e = launch_gemm(p, p.a_k3d ? th2 : th, p.b_k3d ? tw2 : tw[p.cta_pair], tz, grid_max, s);
    if (e != cudaSuccess) return KD_ERR_CUDA;
    float* lse_rows = nullptr;
    if (tile_lse) {
      lse_rows = lse_out ? lse_out + c0 : lse_chunk;
      e = launch_tile_lse(tmax, tsum, ldt, ntiles, n, lse_rows, s);
      if (e != cudaSuccess) return KD_ERR_CUDA;
    }
    // exact top-K (and dropped mass; row logsumexp when not known already) of those bf16 logits
    e = launch_topk(zbuf, n, V, ldz, K, ids_out + c0 * K, vals_out + c0 * K,
                    (lse_out && !tile_lse) ? lse_out + c0 : nullptr, dropped_out ? dropped_out + c0 : nullptr,
                    &ctrl->err, tk_scratch, s, tmax, ldt, ntiles, lse_rows);
    if (e != cudaSuccess) return KD_ERR_CUDA;
  }
  return KD_OK;
}

size_t kd_chunked_kl_logits_bytes(int64_t N, int64_t V) {
  if (N < 1 || V < 1) return 0;
  return size_t((V + 63) / 64) * size_t(N) * 128;
}

}  // extern "C"

// Forward pass of both modes: z_store == NULL is the fused chunked loss; otherwise
// each chunk's raw logits are also written (bf16, blocked) for a backward pass that
// reads them instead of recomputing them.
static int fwd_impl(const void* H_bf16, const void* W_bf16, const int32_t* t_ids, const float* t_logits,
                    const uint8_t* mask, int64_t N, int64_t d, int64_t V, int K, int64_t chunk, float tau,
                    float* loss_out, float* lse_out, float* kl_per_token_out, void* z_store, size_t z_bytes,
                    void* ws, size_t ws_bytes, void* stream) {
  kd_status st = check_kl_args(H_bf16, W_bf16, t_ids, t_logits, N, d, V, K, chunk, tau, ws, ws_bytes);
  if (st != KD_OK) return st;
  if (!loss_out || !lse_out || !aligned(loss_out, 4) || !aligned(lse_out, 4)) return KD_ERR_INVALID_ARG;
  if (kl_per_token_out && !aligned(kl_per_token_out, 4)) return KD_ERR_INVALID_ARG;
  st = check_device();
  if (st != KD_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const KlLayout L = kl_layout(N, d, V, K, chunk);
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(w8);
  int32_t* ids_sorted = reinterpret_cast<int32_t*>(w8 + L.ids_sorted);
  float* p_sorted = reinterpret_cast<float*>(w8 + L.p_sorted);
  float* negent = reinterpret_cast<float*>(w8 + L.negent);
  float* kl = kl_per_token_out ? kl_per_token_out : reinterpret_cast<float*>(w8 + L.kl);
  float4* partials = reinterpret_cast<float4*>(w8 + L.partials);
  const float inv_tau = 1.0f / tau;
  const uint16_t* H = static_cast<const uint16_t*>(H_bf16);

  alignas(64) CUtensorMap tw, tw_half, th, tz;
  if (!make_tmap_2d_bf16(&tw, W_bf16, uint64_t(d), uint64_t(V), uint64_t(d) * 2, BK, BN)) return KD_ERR_CUDA;
  if (!make_tmap_2d_bf16(&tw_half, W_bf16, uint64_t(d), uint64_t(V), uint64_t(d) * 2, BK, BN / 2))
    return KD_ERR_CUDA;
  alignas(64) CUtensorMap tw2, th2;
  const bool d64 = d % 64 == 0;  // two k-blocks per box for CTA pairs
  if (d64 && !make_tmap_mn2_bf16(&tw2, W_bf16, uint64_t(d), uint64_t(V), uint64_t(d) * 2, BN / 2)) return KD_ERR_CUDA;
  if (z_store) {
    (void)z_bytes;
    if (!make_tmap_dz_blocked(&tz, z_store, uint64_t(N), uint64_t(N), uint64_t((V + 63) / 64), 32))
      return KD_ERR_CUDA;
  }

  cudaError_t e = launch_count_valid(mask, N, &ctrl->n_valid, s);
  if (e != cudaSuccess) return KD_ERR_CUDA;
  const int grid_max = gemm_max_grid();
  for (int64_t c0 = 0; c0 < N; c0 += chunk) {
    const int n = int((N - c0) < chunk ? (N - c0) : chunk);
    e = launch_teacher_prologue(t_ids + c0 * K, t_logits + c0 * K, n, K, V, inv_tau, ids_sorted, p_sorted, negent,
                                &ctrl->err, c0, s);
    if (e != cudaSuccess) return KD_ERR_CUDA;
    if (!make_tmap_2d_bf16(&th, H + c0 * d, uint64_t(d), uint64_t(n), uint64_t(d) * 2, BK, BM)) return KD_ERR_CUDA;
    if (d64 && !make_tmap_mn2_bf16(&th2, H + c0 * d, uint64_t(d), uint64_t(n), uint64_t(d) * 2, BM))
      return KD_ERR_CUDA;
    GemmProblem p{};
    p.M = n; p.N = int(V); p.K = int(d);
    p.a_mn = 0; p.b_mn = 0; p.epi = z_store ? EPI_LSE_Z : EPI_LSE;
    p.z_row0 = int(c0);
    p.m_tiles = (n + BM - 1) / BM;
    p.n_tiles = int((V + BN - 1) / BN);
    p.n_group = choose_n_group(V);
    set_cluster(p);
    p.n_units = ((p.m_tiles + p.cluster - 1) / p.cluster) * ((p.n_tiles + p.n_group - 1) / p.n_group);
    p.k_splits = 1;
    p.ids_sorted = ids_sorted; p.p_sorted = p_sorted; p.Kt = K; p.inv_tau = inv_tau;
    p.partials = partials; p.rows = n; p.err = &ctrl->err;
    p.a_k3d = p.b_k3d = p.cta_pair && d64;
    e = launch_gemm(p, p.a_k3d ? th2 : th,
                    p.b_k3d ? tw2 : (p.cta_pair ? tw_half : tw), z_store ? tz : tw,
                    grid_max, s);
    if (e != cudaSuccess) return KD_ERR_CUDA;
    e = launch_lse_combine(partials, L.n_groups, n, negent, inv_tau, lse_out + c0, kl + c0, s);
    if (e != cudaSuccess) return KD_ERR_CUDA;
  }
  e = launch_loss_reduce(kl, mask, N, &ctrl->n_valid, loss_out, s);
  return map_cuda(e);
}

// Backward pass of both modes: z_store == NULL recomputes each chunk's logits on
// the tensor cores (fused); otherwise dZ is formed from the stored logits.
static int bwd_impl(const void* H_bf16, const void* W_bf16, const int32_t* t_ids, const float* t_logits,
                    const uint8_t* mask, int64_t N, int64_t d, int64_t V, int K, int64_t chunk, float tau,
                    const float* lse, const float* grad_loss, const void* z_store, void* grad_H, int grad_H_is_fp32,
                    float* grad_W, void* ws, size_t ws_bytes, void* stream) {
  kd_status st = check_kl_args(H_bf16, W_bf16, t_ids, t_logits, N, d, V, K, chunk, tau, ws, ws_bytes);
  if (st != KD_OK) return st;
  if (!lse || !grad_loss || !grad_H || !grad_W) return KD_ERR_INVALID_ARG;
  if (!aligned(lse, 4) || !aligned(grad_loss, 4) || !aligned(grad_H, 16) || !aligned(grad_W, 16))
    return KD_ERR_INVALID_ARG;
  st = check_device();
  if (st != KD_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const KlLayout L = kl_layout(N, d, V, K, chunk);
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(w8);
  int32_t* ids_sorted = reinterpret_cast<int32_t*>(w8 + L.ids_sorted);
  float* p_sorted = reinterpret_cast<float*>(w8 + L.p_sorted);
  float* negent = reinterpret_cast<float*>(w8 + L.negent);
  uint16_t* dz = reinterpret_cast<uint16_t*>(w8 + L.dz);
  const float inv_tau = 1.0f / tau;
  const uint16_t* H = static_cast<const uint16_t*>(H_bf16);
  const size_t gh_elt = grad_H_is_fp32 ? 4 : 2;

  alignas(64) CUtensorMap tw_k, tw_k_half, tw_mn, tw_mn2, th_k, th_mn, th_mn2, tdz_k, tdz_mn, tdz_st, tgw;
  // CTA-pair launches take pair_kblocks(a_mn, b_mn) 64-deep k-blocks per ring stage: boxes of
  // 64 kq (grad_H) / 64 kr (grad_W) rows for MN-major operands, that depth for K-major
  // ones (suffix _p); the dZ recompute takes two (tw_k2, th_k2: depth-2 boxes)
  alignas(64) CUtensorMap tw_k2, tw_mn_p, th_k2, th_mn_p, tdz_k_p, tdz_mn_p;
  const int kq = pair_kblocks(0, 1), kr = pair_kblocks(1, 1);  // grad_H, grad_W
  const bool d64 = d % 64 == 0;  // 3-D two-block views of W and H need whole 64-column blocks
  if (!make_tmap_2d_bf16(&tw_k, W_bf16, uint64_t(d), uint64_t(V), uint64_t(d) * 2, BK, BN)) return KD_ERR_CUDA;
  if (!make_tmap_2d_bf16(&tw_k_half, W_bf16, uint64_t(d), uint64_t(V), uint64_t(d) * 2, BK, BN / 2))
    return KD_ERR_CUDA;
  if (!make_tmap_2d_f32(&tgw, grad_W, uint64_t(d), uint64_t(V), uint64_t(d) * 4, 32, 32)) return KD_ERR_CUDA;
  if (!make_tmap_2d_bf16(&tw_mn, W_bf16, uint64_t(d), uint64_t(V), uint64_t(d) * 2, 64, BK)) return KD_ERR_CUDA;
  if (d64 && !make_tmap_mn2_bf16(&tw_mn2, W_bf16, uint64_t(d), uint64_t(V), uint64_t(d) * 2, BK * kq))
    return KD_ERR_CUDA;
  if (!make_tmap_2d_bf16(&tw_mn_p, W_bf16, uint64_t(d), uint64_t(V), uint64_t(d) * 2, 64, BK * kq)) return KD_ERR_CUDA;
  if (d64 && !make_tmap_mn2_bf16(&tw_k2, W_bf16, uint64_t(d), uint64_t(V), uint64_t(d) * 2, BN / 2))
    return KD_ERR_CUDA;

  cudaError_t e = launch_count_valid(mask, N, &ctrl->n_valid, s);
  if (e != cudaSuccess) return KD_ERR_CUDA;
  const int grid_max = gemm_max_grid();
  for (int64_t c0 = 0; c0 < N; c0 += chunk) {
    const int n = int((N - c0) < chunk ? (N - c0) : chunk);
    e = launch_teacher_prologue(t_ids + c0 * K, t_logits + c0 * K, n, K, V, inv_tau, ids_sorted, p_sorted, negent,
                                &ctrl->err, c0, s);
    if (e != cudaSuccess) return KD_ERR_CUDA;
    const uint16_t* Hc = H + c0 * d;
    if (!make_tmap_2d_bf16(&th_k, Hc, uint64_t(d), uint64_t(n), uint64_t(d) * 2, BK, BM)) return KD_ERR_CUDA;
    if (!make_tmap_2d_bf16(&th_mn, Hc, uint64_t(d), uint64_t(n), uint64_t(d) * 2, 64, BK)) return KD_ERR_CUDA;
    if (d64 && !make_tmap_mn2_bf16(&th_mn2, Hc, uint64_t(d), uint64_t(n), uint64_t(d) * 2, BK * kr))
      return KD_ERR_CUDA;
    if (!make_tmap_2d_bf16(&th_mn_p, Hc, uint64_t(d), uint64_t(n), uint64_t(d) * 2, 64, BK * kr)) return KD_ERR_CUDA;
    if (d64 && !make_tmap_mn2_bf16(&th_k2, Hc, uint64_t(d), uint64_t(n), uint64_t(d) * 2, BM)) return KD_ERR_CUDA;
    // dZ in blocked layout [vocab/64][row][64]: each box below is one contiguous run
    if (!make_tmap_dz_blocked(&tdz_k, dz, uint64_t(n), uint64_t(L.rows_pad), uint64_t(L.nvb), BM)) return KD_ERR_CUDA;
    if (!make_tmap_dz_blocked(&tdz_mn, dz, uint64_t(n), uint64_t(L.rows_pad), uint64_t(L.nvb), BK)) return KD_ERR_CUDA;
    if (!make_tmap_dz_blocked(&tdz_k_p, dz, uint64_t(n), uint64_t(L.rows_pad), uint64_t(L.nvb), BM, kq))
      return KD_ERR_CUDA;
    if (!make_tmap_dz_blocked(&tdz_mn_p, dz, uint64_t(n), uint64_t(L.rows_pad), uint64_t(L.nvb), BK * kr, 2))
      return KD_ERR_CUDA;
    if (!make_tmap_dz_blocked(&tdz_st, dz, uint64_t(n), uint64_t(L.rows_pad), uint64_t(L.nvb), 32)) return KD_ERR_CUDA;

    if (z_store) {
      // forward-chunked: dZ from the logits the forward pass kept
      e = launch_dz_from_z(static_cast<const uint16_t*>(z_store), N, c0, n, V, L.nvb, L.rows_pad, lse + c0,
                           mask ? mask + c0 : nullptr, grad_loss, &ctrl->n_valid, inv_tau, ids_sorted, p_sorted, K,
                           dz, s);
      if (e != cudaSuccess) return KD_ERR_CUDA;
    } else {
    // B1: recompute the chunk's logits, dZ -> bf16 workspace
    GemmProblem p{};
    p.M = n; p.N = int(V); p.K = int(d);
    p.a_mn = 0; p.b_mn = 0; p.epi = EPI_DZ;
    p.m_tiles = (n + BM - 1) / BM;
    p.n_tiles = int((V + BN - 1) / BN);
    p.n_group = 1;
    set_cluster(p);
    p.n_units = ((p.m_tiles + p.cluster - 1) / p.cluster) * p.n_tiles;
    p.k_splits = 1;
    p.ids_sorted = ids_sorted; p.p_sorted = p_sorted; p.Kt = K; p.inv_tau = inv_tau;
    p.lse = lse + c0; p.mask = mask ? mask + c0 : nullptr; p.grad_loss = grad_loss; p.n_valid = &ctrl->n_valid;
    p.dz = dz; p.ldz = L.ldz; p.rows = n; p.err = &ctrl->err;
    p.a_k3d = p.b_k3d = p.cta_pair && d64;
    e = launch_gemm(p, p.a_k3d ? th_k2 : th_k,
                    p.b_k3d ? tw_k2 : (p.cta_pair ? tw_k_half : tw_k), tdz_st,
                    grid_max, s);
    if (e != cudaSuccess) return KD_ERR_CUDA;
    }

    // B2: grad_H rows of the chunk = dZ W  (A = dZ K-major over V, B = W with d contiguous)
    GemmProblem q{};
    q.M = n; q.N = int(d); q.K = int(V);
    q.a_mn = 0; q.b_mn = 1; q.epi = EPI_STORE;
    q.m_tiles = (n + BM - 1) / BM;
    q.n_tiles = int((d + BN - 1) / BN);
    q.n_group = 1;
    q.a_blocked = 1;
    q.k_splits = choose_splits(int64_t(q.m_tiles) * q.n_tiles, int((V + BK - 1) / BK), grid_max);
    set_cluster(q);
    q.n_units = ((q.m_tiles + q.cluster - 1) / q.cluster) * q.n_tiles * q.k_splits;
    void* gh_out = static_cast<uint8_t*>(grad_H) + size_t(c0) * d * gh_elt;
    if (q.k_splits == 1) {
      q.C = gh_out;
      q.ldc = d; q.c_bf16 = grad_H_is_fp32 ? 0 : 1;
    } else {
      q.C = w8 + L.gh_part;  // fp32 partial per split, summed in split order below
      q.ldc = d; q.c_bf16 = 0;
      q.split_stride = L.rows_pad * d;
    }
    q.err = &ctrl->err;
    q.b_box2 = q.cta_pair && d64;
    e = launch_gemm(q, q.cta_pair ? tdz_k_p : tdz_k, q.b_box2 ? tw_mn2 : (q.cta_pair ? tw_mn_p : tw_mn), tw_mn,
                    grid_max, s);
    if (e != cudaSuccess) return KD_ERR_CUDA;
    if (q.k_splits > 1) {
      e = launch_split_reduce(reinterpret_cast<const float*>(w8 + L.gh_part), q.k_splits, L.rows_pad * d,
                              int64_t(n) * d, gh_out, grad_H_is_fp32 ? 0 : 1, s);
      if (e != cudaSuccess) return KD_ERR_CUDA;
    }

    // B3: grad_W += dZ^T H_c  (A = dZ with V contiguous, B = H_c with d contiguous)
    GemmProblem r{};
    r.M = int(V); r.N = int(d); r.K = n;
    r.a_mn = 1; r.b_mn = 1; r.epi = EPI_ACCUM;
    r.m_tiles = int((V + BM - 1) / BM);
    r.n_tiles = int((d + BN - 1) / BN);
    r.n_group = 1;
    r.a_blocked = 1;
    r.k_splits = 1;
    set_cluster(r);
    r.n_units = ((r.m_tiles + r.cluster - 1) / r.cluster) * r.n_tiles;
    r.C = grad_W; r.ldc = d; r.c_bf16 = 0; r.err = &ctrl->err;
    r.b_box2 = r.cta_pair && d64;
    e = launch_gemm(r, r.cta_pair ? tdz_mn_p : tdz_mn, r.b_box2 ? th_mn2 : (r.cta_pair ? th_mn_p : th_mn), tgw,
                    grid_max, s);
    if (e != cudaSuccess) return KD_ERR_CUDA;
  }
  return KD_OK;
}

extern "C" {

int kd_fused_kl_fwd(const void* H_bf16, const void* W_bf16, const int32_t* t_ids, const float* t_logits,
                    const uint8_t* mask, int64_t N, int64_t d, int64_t V, int K, int64_t chunk, float tau,
                    float* loss_out, float* lse_out, float* kl_per_token_out, void* ws, size_t ws_bytes,
                    void* stream) {
  return fwd_impl(H_bf16, W_bf16, t_ids, t_logits, mask, N, d, V, K, chunk, tau, loss_out, lse_out,
                  kl_per_token_out, nullptr, 0, ws, ws_bytes, stream);
}

int kd_fused_kl_bwd(const void* H_bf16, const void* W_bf16, const int32_t* t_ids, const float* t_logits,
                    const uint8_t* mask, int64_t N, int64_t d, int64_t V, int K, int64_t chunk, float tau,
                    const float* lse, const float* grad_loss, void* grad_H, int grad_H_is_fp32, float* grad_W,
                    void* ws, size_t ws_bytes, void* stream) {
  return bwd_impl(H_bf16, W_bf16, t_ids, t_logits, mask, N, d, V, K, chunk, tau, lse, grad_loss, nullptr, grad_H,
                  grad_H_is_fp32, grad_W, ws, ws_bytes, stream);
}

int kd_chunked_kl_fwd(const void* H_bf16, const void* W_bf16, const int32_t* t_ids, const float* t_logits,
                      const uint8_t* mask, int64_t N, int64_t d, int64_t V, int K, int64_t chunk, float tau,
                      float* loss_out, float* lse_out, float* kl_per_token_out, void* z_store, size_t z_bytes,
                      void* ws, size_t ws_bytes, void* stream) {
  if (!z_store || !aligned(z_store, 16) || N < 1 || V < 1) return KD_ERR_INVALID_ARG;
  if (z_bytes < kd_chunked_kl_logits_bytes(N, V)) return KD_ERR_INVALID_ARG;
  return fwd_impl(H_bf16, W_bf16, t_ids, t_logits, mask, N, d, V, K, chunk, tau, loss_out, lse_out,
                  kl_per_token_out, z_store, z_bytes, ws, ws_bytes, stream);
}

int kd_chunked_kl_bwd(const void* H_bf16, const void* W_bf16, const int32_t* t_ids, const float* t_logits,
                      const uint8_t* mask, int64_t N, int64_t d, int64_t V, int K, int64_t chunk, float tau,
                      const float* lse, const float* grad_loss, const void* z_store, size_t z_bytes, void* grad_H,
                      int grad_H_is_fp32, float* grad_W, void* ws, size_t ws_bytes, void* stream) {
  if (!z_store || !aligned(z_store, 16) || N < 1 || V < 1) return KD_ERR_INVALID_ARG;
  if (z_bytes < kd_chunked_kl_logits_bytes(N, V)) return KD_ERR_INVALID_ARG;
  return bwd_impl(H_bf16, W_bf16, t_ids, t_logits, mask, N, d, V, K, chunk, tau, lse, grad_loss, z_store, grad_H,
                  grad_H_is_fp32, grad_W, ws, ws_bytes, stream);
}

int kd_get_device_error(void* ws, void* stream, int64_t* detail_out) {
  if (ws == nullptr) {
    // the scratch array of the allocation-free forward on the current device
    kd_status st = static_scratch_address(&ws);
    if (st != KD_OK) return st;
  }
  if (!aligned(ws, 256)) return KD_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return KD_ERR_CUDA;
  uint32_t w[2] = {0, 0};
  if (cudaMemcpy(w, ws, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return KD_ERR_CUDA;
  if (cudaMemset(ws, 0, sizeof(w)) != cudaSuccess) return KD_ERR_CUDA;
  if (detail_out) *detail_out = int64_t(w[1]);
  if (w[0] == KD_DEVERR_NONE) return KD_OK;
  if (w[0] == KD_DEVERR_TIMEOUT) return KD_ERR_TIMEOUT;
  return KD_ERR_DEVICE;
}

size_t kd_gemm_workspace(void) { return sizeof(Ctrl); }

int kd_check_wait_timeout(void* ws, size_t ws_bytes, int64_t limit_ns, void* stream) {
  if (!ws || !aligned(ws, 256) || ws_bytes < sizeof(Ctrl)) return KD_ERR_WORKSPACE;
  if (limit_ns < 1000 || limit_ns > 1000000000LL) return KD_ERR_INVALID_ARG;
  kd_status st = check_device();
  if (st != KD_OK) return st;
  return map_cuda(launch_wait_timeout(&static_cast<Ctrl*>(ws)->err, uint64_t(limit_ns),
                                      static_cast<cudaStream_t>(stream)));
}

int kd_gemm_bf16(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K, int a_mn, int b_mn,
                 int accumulate, void* ws, size_t ws_bytes, void* stream) {
  if (M < 1 || N < 1 || K < 1 || M > 0x7fffffffLL || N > 0x7fffffffLL || K > 0x7fffffffLL)
    return KD_ERR_INVALID_ARG;
  if (!A || !B || !C || !aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16)) return KD_ERR_INVALID_ARG;
  if (N % 4 != 0) return KD_ERR_INVALID_ARG;
  if ((a_mn ? M : K) % 8 != 0 || (b_mn ? N : K) % 8 != 0) return KD_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256) || ws_bytes < kd_gemm_workspace()) return KD_ERR_WORKSPACE;
  kd_status st = check_device();
  if (st != KD_OK) return st;
  alignas(64) CUtensorMap ta, tb, tc;
  GemmProblem p{};
  p.epi = accumulate ? EPI_ACCUM : EPI_STORE;
  p.m_tiles = int((M + BM - 1) / BM);
  set_cluster(p);
  bool ok;
  if (p.cta_pair) {
    // kk 64-deep k-blocks per ring stage; each operand in one box where whole 64-column
    // blocks allow (MN-major: both column blocks; K-major: kk = 2 k-blocks, depth 2)
    const int kk = pair_kblocks(a_mn ? 1 : 0, b_mn ? 1 : 0);
    p.a_box2 = a_mn && M % 64 == 0;
    p.a_k3d = kk == 2 && !a_mn && K % 64 == 0;
    p.b_box2 = b_mn && N % 64 == 0;
    p.b_k3d = kk == 2 && !b_mn && K % 64 == 0;
    ok = a_mn ? (p.a_box2 ? make_tmap_mn2_bf16(&ta, A, uint64_t(M), uint64_t(K), uint64_t(M) * 2, BK * kk)
                          : make_tmap_2d_bf16(&ta, A, uint64_t(M), uint64_t(K), uint64_t(M) * 2, 64, BK * kk))
              : (p.a_k3d ? make_tmap_mn2_bf16(&ta, A, uint64_t(K), uint64_t(M), uint64_t(K) * 2, BM)
                         : make_tmap_2d_bf16(&ta, A, uint64_t(K), uint64_t(M), uint64_t(K) * 2, BK, BM));
    ok = ok && (b_mn ? (p.b_box2 ? make_tmap_mn2_bf16(&tb, B, uint64_t(N), uint64_t(K), uint64_t(N) * 2, BK * kk)
                                 : make_tmap_2d_bf16(&tb, B, uint64_t(N), uint64_t(K), uint64_t(N) * 2, 64, BK * kk))
                     : (p.b_k3d ? make_tmap_mn2_bf16(&tb, B, uint64_t(K), uint64_t(N), uint64_t(K) * 2, BN / 2)
                                : make_tmap_2d_bf16(&tb, B, uint64_t(K), uint64_t(N), uint64_t(K) * 2, BK, BN / 2)));
  } else {
    ok = a_mn ? make_tmap_2d_bf16(&ta, A, uint64_t(M), uint64_t(K), uint64_t(M) * 2, 64, BK)
              : make_tmap_2d_bf16(&ta, A, uint64_t(K), uint64_t(M), uint64_t(K) * 2, BK, BM);
    ok = ok && (b_mn ? make_tmap_2d_bf16(&tb, B, uint64_t(N), uint64_t(K), uint64_t(N) * 2, 64, BK)
                     : make_tmap_2d_bf16(&tb, B, uint64_t(K), uint64_t(N), uint64_t(K) * 2, BK, BN));
  }
  ok = ok && make_tmap_2d_f32(&tc, C, uint64_t(N), uint64_t(M), uint64_t(N) * 4, 32, 32);
  if (!ok) return KD_ERR_CUDA;
  p.M = int(M); p.N = int(N); p.K = int(K);
  p.a_mn = a_mn ? 1 : 0; p.b_mn = b_mn ? 1 : 0;
  p.n_tiles = int((N + BN - 1) / BN);
  p.n_group = 1;
  p.k_splits = 1;
  p.m_fast = N > M ? 1 : 0;  // B larger than A: share B tiles in flight, read B once
  p.n_units = ((p.m_tiles + p.cluster - 1) / p.cluster) * p.n_tiles;
  p.C = C; p.ldc = N; p.c_bf16 = 0;
  p.err = &static_cast<Ctrl*>(ws)->err;
  return map_cuda(launch_gemm(p, ta, tb, tc, gemm_max_grid(), static_cast<cudaStream_t>(stream)));
}

int kd_profile_begin(int capacity) {
  if (capacity < 1) return KD_ERR_INVALID_ARG;
  if (int(g_prof.size()) < capacity) {
    size_t old = g_prof.size();
    g_prof.resize(size_t(capacity));
    for (size_t i = old; i < g_prof.size(); ++i) {
      if (cudaEventCreate(&g_prof[i].start) != cudaSuccess || cudaEventCreate(&g_prof[i].stop) != cudaSuccess)
        return KD_ERR_CUDA;
    }
  }
  g_prof_used = 0;
  g_prof_on = true;
  return KD_OK;
}

int kd_profile_end(void) {
  g_prof_on = false;
  return KD_OK;
}

int kd_profile_read(const char** names, float* ms, int n) {
  for (int i = 0; i < g_prof_used && i < n; ++i) {
    if (cudaEventSynchronize(g_prof[i].stop) != cudaSuccess) return -KD_ERR_CUDA;
    float t = 0.f;
    cudaEventElapsedTime(&t, g_prof[i].start, g_prof[i].stop);
    if (names) names[i] = g_prof[i].name;
    if (ms) ms[i] = t;
  }
  return g_prof_used;
}

}  // extern "C"
