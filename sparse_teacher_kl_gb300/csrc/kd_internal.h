// Internal declarations shared by the translation units of libkdkl.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kdkl.h"
#include "kd_host_state.h"

namespace kd {

// Device error word codes (first word of every workspace; the second word
// holds a detail, the third a launch tag).
constexpr uint32_t KD_DEVERR_NONE = 0;
constexpr uint32_t KD_DEVERR_TIMEOUT = 1;
constexpr uint32_t KD_DEVERR_BAD_ID = 2;
constexpr uint32_t KD_DEVERR_BOUNDS = 3;  // KD_DEBUG builds: a computed index out of range (skipped)

// Upper bound on any single wait inside a kernel.  A healthy wait lasts
// microseconds; this only stops a kernel that would otherwise hang.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Workspace control block at offset 0 of every workspace.
struct Ctrl {
  uint32_t err;        // KD_DEVERR_*
  uint32_t err_detail;
  uint32_t topk_reselected;  // top-K: rows selected a second time after a speculative start
  uint32_t pad0;
  int32_t n_valid;     // number of valid positions of the current call
  uint32_t pad1[59];
};
static_assert(sizeof(Ctrl) == 256, "control block is 256 bytes");

// GEMM engine geometry: one CTA computes a 128 x 256 fp32 tile in tensor
// memory, K staged 64 bf16 (128 B, one swizzle row) at a time.
constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int STAGE_A_BYTES = BM * BK * 2;  // 16 KB
constexpr int STAGE_B_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = STAGE_A_BYTES + STAGE_B_BYTES;
constexpr int GEMM_THREADS = 192;           // TMA warp, MMA warp, 4 epilogue warps
constexpr int STAGING_BYTES = 4 * 2 * 4096; // per epilogue warp: two 32 x 128 B output boxes
constexpr int TMEM_COLS = 512;              // two 256-column fp32 accumulators

// Epilogue kinds of the GEMM engine.
enum EpiKind : int {
  EPI_LSE = 0,    // forward: online logsumexp + teacher-id gather -> partials
  EPI_DZ = 1,     // backward: dZ = scale * (softmax - p) -> bf16 [rows, ldz]
  EPI_STORE = 2,  // C = acc -> fp32 or bf16
  EPI_ACCUM = 3,  // C += acc (fp32)
  EPI_LSE_Z = 4,  // forward-chunked: EPI_LSE plus the raw logits z -> bf16, blocked [V/64][N][64]
};

// 64-deep k-blocks per ring stage of a CTA-pair launch: two when both operands are
// K-major (the loss sweeps and the teacher projection: each stage one depth-2 box per
// operand), one otherwise (the gradient products, MN-major operands: more, shallower
// stages measured faster there).  The tensor maps of a pair launch are sized for this.
constexpr int pair_kblocks(int a_mn, int b_mn) { return (a_mn == 0 && b_mn == 0) ? 2 : 1; }

struct GemmProblem {
  int M, N, K;           // logical GEMM sizes
  int a_mn, b_mn;        // operand major-ness (0 = K-major)
  int epi;               // EpiKind
  // tile schedule: tiles are (m_blk, n_blk); n_group consecutive n tiles form
  // one unit processed by one CTA in order (used by EPI_LSE).
  int m_tiles, n_tiles, n_group, n_units;
  // split-K (EPI_STORE): the K range is cut into k_splits nearly equal parts; the
  // partial of split s goes to C + s * split_stride (elements).
  int k_splits;
  int64_t split_stride;
  // blocked dZ: operand A (a_blocked) or the EPI_DZ output is the 3-D blocked layout
  // dZ[vocab / 64][row][vocab % 64] (see make_tmap_dz_blocked), so that every TMA box
  // of it is one contiguous run of memory.
  int a_blocked;
  // a_box2 / b_box2 (CTA pairs, MN-major operand): the operand's two 64-column blocks of
  // a stage come in one TMA box of depth 2 from a 3-D map (64, k, blocks), 8 KB apart in
  // shared memory as the MMA reads them; 0: two boxes from a 2-D (or depth-1) map.
  int a_box2, b_box2;
  // a_k3d / b_k3d (CTA pairs with two k-blocks per stage, K-major operand): both come in
  // one box of depth 2 from a 3-D view (64, rows, K / 64); 0: one box per k-block.
  int a_k3d, b_k3d;
  int z_row0;                 // EPI_LSE_Z: row of the stored logits that chunk row 0 maps to
  // cluster: CTAs per cluster, 2 for CTA pairs (cta_pair = 1), else 1.  The CTAs of a
  // pair take consecutive m tiles of the same n tile; n_units counts pairs' units.
  int cluster;
  // cta_pair = 1 (cluster = 2): each pair computes one 256 x 256 tile with tcgen05
  // cta_group::2 MMAs (A split by rows, B by columns between the two CTAs, each CTA
  // loading its own halves; K-major B map box 64 x 128).
  int cta_pair;
  // EPI_STORE / EPI_ACCUM
  void* C;
  int64_t ldc;
  int c_bf16;
  // c_tma = 1 (EPI_STORE, bf16 C, k_splits = 1): the epilogue writes 32 x 64 boxes staged
  // in shared memory with TMA stores through tmap_c (row-major C, box 64 x 32, 128-byte
  // swizzle), clipped at the matrix edges; 0: direct 16-byte stores.
  int c_tma;
  // tile_max (c_tma = 1 only; NULL: none): per row of C and per BN-column tile, the largest
  // bf16-rounded value of the row inside the tile (columns < N; bf16 bits, -inf for a tile
  // of NaNs), at tile_max[row * ld_tile_max + tile] for rows < M.
  uint16_t* tile_max;
  int64_t ld_tile_max;
  // tile_sum (with tile_max; NULL: none): per row and BN-column tile, the sum of
  // 2^((z - m) log2 e) over the row's bf16-rounded values z in the tile (columns < N), m
  // the tile's maximum above (NaN if one of them is NaN), at tile_sum[row * ld_tile_max +
  // tile] for rows < M: with tile_max, the row's logsumexp in pieces.
  float* tile_sum;
  // m_fast = 1 (EPI_STORE / EPI_ACCUM with k_splits = 1): units walk m fastest, so the CTAs
  // in flight share one B tile while the A operand stays in L2 (for a small A and a B
  // larger than L2, as in the teacher projection); 0: n fastest (they share one A slab).
  int m_fast;
  // EPI_LSE / EPI_DZ (rows = tokens of the chunk, cols = vocabulary)
  const int32_t* ids_sorted;  // [rows, K] ascending
  const float* p_sorted;      // [rows, K] teacher probabilities matching ids_sorted
  int Kt;                     // teacher K
  float inv_tau;
  float4* partials;           // EPI_LSE: [n_units_per_row, rows] (m2, s, G, 0)
  const float* lse;           // EPI_DZ: [rows] natural-log lse (chunk-relative pointer)
  const uint8_t* mask;        // EPI_DZ: [rows] or null (chunk-relative pointer)
  const float* grad_loss;     // EPI_DZ: device scalar
  const int32_t* n_valid;     // EPI_DZ: device scalar
  uint16_t* dz;               // EPI_DZ: bf16 [rows, ldz]
  int64_t ldz;
  int rows;                   // valid rows of A (tokens in this chunk) for LSE/DZ
  uint32_t* err;
};

// Host helpers (kd_tma.cpp part of kd_abi.cu).
bool make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                       uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);
// dZ chunk in blocked layout: [nvb = ceil(V/64)][rows_pad][64] bf16; dims {64, rows, nvb},
// box {64, box_rows, 1}, 128-byte swizzle.
bool make_tmap_dz_blocked(CUtensorMap* map, const void* base, uint64_t rows, uint64_t rows_pad, uint64_t nvb,
                          uint32_t box_rows, uint32_t box_depth = 1);
// 3-D view (64, rows, cols / 64) of a row-major bf16 matrix whose column count is a
// multiple of 64, box (64, box_rows, 2): two 64-column blocks per TMA box (two k-blocks
// of a K-major operand, or two column blocks of an MN-major one).
bool make_tmap_mn2_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint64_t row_stride_bytes,
                        uint32_t box_rows);
bool make_tmap_2d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                      uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);

// Raise a kernel's dynamic shared-memory limit to `bytes` once per device (safe from
// several host threads; `done` is the kernel's own per-device record).
inline cudaError_t smem_attr_once(PerDevice<int>& done, const void* func, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int v = 0;
  const int rc = done.get(dev, &v, [&](int, int* out) {
    *out = 1;
    return int(cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
  });
  return rc == 0 ? cudaSuccess : (rc > 0 ? cudaError_t(rc) : cudaErrorInvalidDevice);
}

// Launchers (return a cudaError_t).
// tc: output map for the epilogues that write through TMA (EPI_ACCUM: fp32 C,
// box 32 x 32; EPI_DZ: bf16 dZ, box 64 x 32; both 128-byte swizzle); ignored
// by the others.
cudaError_t launch_gemm(const GemmProblem& p, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                        int grid, cudaStream_t s);
int gemm_max_grid();

// Top-K of every row of X [N, ld] bf16 (columns [0, V)): ids and values [N, K], optionally
// the row logsumexp lse [N] and the dropped teacher mass dropped [N] (NULL: not wanted).
// err: the workspace control block's error word (its third word counts rows that a
// speculative start made select twice).  scratch: topk_scratch_bytes(N, K) bytes, 256-byte
// aligned.  tile_max (NULL: none): per row, the maxima of ntiles disjoint column ranges of
// the row (bf16 bits, [N, ld_tile_max]); with ntiles >= K their K-th largest is a lower
// bound of the row's K-th largest value and starts the row.  lse_known (NULL: none; only
// where topk_takes_known_lse(K)): the rows' logsumexp, already computed, for the dropped
// mass; the selection then computes none (lse must be NULL).
size_t topk_scratch_bytes(int64_t N, int K);
bool topk_takes_known_lse(int K);
cudaError_t launch_topk(const uint16_t* X, int64_t N, int64_t V, int64_t ld, int K, int32_t* ids,
                        float* vals, float* lse, float* dropped, uint32_t* err, void* scratch, cudaStream_t s,
                        const uint16_t* tile_max = nullptr, int64_t ld_tile_max = 0, int ntiles = 0,
                        const float* lse_known = nullptr);
// Row logsumexp [rows] from the per-tile maxima and sums of a projection's epilogue
// (GemmProblem::tile_max, tile_sum; ntiles of them per row, row stride ld).
cudaError_t launch_tile_lse(const uint16_t* tile_max, const float* tile_sum, int64_t ld, int ntiles, int64_t rows,
                            float* lse, cudaStream_t s);

cudaError_t launch_count_valid(const uint8_t* mask, int64_t N, int32_t* n_valid, cudaStream_t s);
cudaError_t launch_teacher_prologue(const int32_t* ids, const float* tlog, int rows, int K, int64_t V,
                                    float inv_tau, int32_t* ids_sorted, float* p_sorted, float* negent,
                                    uint32_t* err, int64_t row0, cudaStream_t s);
cudaError_t launch_lse_combine(const float4* partials, int n_units_per_row, int rows, const float* negent,
                               float inv_tau, float* lse_out, float* kl_out, cudaStream_t s);
cudaError_t launch_loss_reduce(const float* kl, const uint8_t* mask, int64_t N, const int32_t* n_valid,
                               float* loss_out, cudaStream_t s);

cudaError_t launch_wait_timeout(uint32_t* err, uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_dz_from_z(const uint16_t* z, int64_t N, int64_t c0, int rows, int64_t V, int64_t nvb,
                             int64_t rows_pad, const float* lse, const uint8_t* mask, const float* grad_loss,
                             const int32_t* n_valid, float inv_tau, const int32_t* ids_sorted, const float* p_sorted,
                             int K, uint16_t* dz, cudaStream_t s);
cudaError_t launch_split_reduce(const float* parts, int splits, int64_t split_stride, int64_t count, void* out,
                                int out_bf16, cudaStream_t s);

constexpr int KD_MAX_SPLITS = 8;

// Device address of the library's own scratch array (kd_fused_kl_fwd_static) on the
// current device, looked up once per device and context.
kd_status static_scratch_address(void** out);

// Profiling hooks (kd_abi.cu): bracket a launch with events when enabled.
void prof_before(const char* name, cudaStream_t s);
void prof_after(cudaStream_t s);

}  // namespace kd
