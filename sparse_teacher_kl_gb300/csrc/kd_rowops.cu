// Row-wise steps around the projection engine: the sparse teacher prologue,
// the merge of per-unit logsumexp partials into per-position KL, the masked
// token-mean reduction and the valid-position count.  All O(N * K) or
// O(N * V / 256) work, a small share of a step.
#include <math.h>
#include <stdint.h>

#include "kd_device.cuh"
#include "kd_internal.h"

namespace kd {

// ---------------------------------------------------------- valid count ---

__global__ void kd_count_valid_kernel(const uint8_t* __restrict__ mask, int64_t N, int32_t* __restrict__ n_valid) {
  __shared__ int32_t warp_sums[32];
  int32_t c = 0;
  if (mask == nullptr) {
    if (threadIdx.x == 0) *n_valid = int32_t(N);
    return;
  }
  for (int64_t i = threadIdx.x; i < N; i += blockDim.x) c += mask[i] != 0;
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x < 32) {
    c = (threadIdx.x < (blockDim.x >> 5)) ? warp_sums[threadIdx.x] : 0;
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (threadIdx.x == 0) *n_valid = c;
  }
}

cudaError_t launch_count_valid(const uint8_t* mask, int64_t N, int32_t* n_valid, cudaStream_t s) {
  prof_before("kd_count_valid", s);
  kd_count_valid_kernel<<<1, 1024, 0, s>>>(mask, N, n_valid);
  prof_after(s);
  return cudaGetLastError();
}

// ------------------------------------------------------ teacher prologue ---
// [ART] fused-loss paragraph (the teacher stays sparse) and offline-cache
// paragraph: per position, p = softmax(t / tau) over the K cached logits (the
// mass outside them dropped), its negative entropy sum_k p_k log p_k, and the
// (id, p) pairs ordered by id so that the projection epilogue meets them in
// vocabulary order.  One warp per position.

constexpr int PRO_WARPS = 4;

// Warp: sort the 32 E entries a[] of the warp ascending, in registers: a bitonic network over
// positions p = lane E + i; a partner within the lane is swapped in place, one in another
// lane (distance >= E) comes by shuffle.
template <int E>
__device__ __forceinline__ void warp_sort_regs_asc(unsigned long long (&a)[E]) {
  const uint32_t lane = threadIdx.x & 31u;
#pragma unroll
  for (int k = 2; k <= 32 * E; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= E) {
#pragma unroll
        for (int i = 0; i < E; ++i) {
          const uint32_t p = lane * E + i;
          const unsigned long long o = __shfl_xor_sync(0xffffffffu, a[i], uint32_t(j / E));
          const bool asc = (p & uint32_t(k)) == 0;
          const bool lower = (p & uint32_t(j)) == 0;
          a[i] = (asc == lower) ? (a[i] < o ? a[i] : o) : (a[i] < o ? o : a[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < E; ++i) {
          if ((i & j) == 0) {
            const uint32_t p = lane * E + i;
            const bool asc = (p & uint32_t(k)) == 0;
            const unsigned long long x = a[i], y = a[i + j];
            const bool swap = asc ? (x > y) : (x < y);
            a[i] = swap ? y : x;
            a[i + j] = swap ? x : y;
          }
        }
      }
    }
  }
}

// E = KP / 32 entries per lane, KP the power of two >= max(K, 32); entry k of the row is
// held by lane k / E.
template <int E>
__global__ void __launch_bounds__(PRO_WARPS * 32)
    kd_teacher_prologue_kernel(const int32_t* __restrict__ ids, const float* __restrict__ tlog, int rows, int K,
                               int64_t V, float inv_tau, int32_t* __restrict__ ids_sorted,
                               float* __restrict__ p_sorted, float* __restrict__ negent,
                               uint32_t* __restrict__ err, int64_t row0) {
  const uint32_t lane = threadIdx.x & 31u;
  const int row = blockIdx.x * PRO_WARPS + int(threadIdx.x >> 5);
  if (row >= rows) return;
  const int32_t* idr = ids + size_t(row) * K;
  const float* tr = tlog + size_t(row) * K;

  float t[E];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int k = int(lane) * E + i;
    t[i] = k < K ? tr[k] * inv_tau : -INFINITY;
    m = fmaxf(m, t[i]);
  }
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i)
    if (int(lane) * E + i < K) s += expf(t[i] - m);
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float log_s = logf(s);
  float h = 0.f;
  bool bad = false;
  unsigned long long a[E];
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int k = int(lane) * E + i;
    a[i] = ~0ull;  // padding sorts after every entry
    if (k < K) {
      const float lp = t[i] - m - log_s;
      const float pk = expf(lp);
      if (pk > 0.f) h += pk * lp;
      const int32_t id = idr[k];
      bad |= (id < 0) || (int64_t(id) >= V);
      a[i] = (static_cast<unsigned long long>(uint32_t(id)) << 32) | __float_as_uint(pk);
    }
  }
  for (int o = 16; o > 0; o >>= 1) h += __shfl_xor_sync(0xffffffffu, h, o);
  if (__any_sync(0xffffffffu, bad) && lane == 0) raise_error(err, KD_DEVERR_BAD_ID, uint32_t(row0 + row));
  warp_sort_regs_asc<E>(a);  // ascending by id
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const int k = int(lane) * E + i;
    if (k < K) {
      ids_sorted[size_t(row) * K + k] = int32_t(uint32_t(a[i] >> 32));
      p_sorted[size_t(row) * K + k] = __uint_as_float(uint32_t(a[i]));
    }
  }
  if (lane == 0) negent[row] = h;
}

cudaError_t launch_teacher_prologue(const int32_t* ids, const float* tlog, int rows, int K, int64_t V,
                                    float inv_tau, int32_t* ids_sorted, float* p_sorted, float* negent,
                                    uint32_t* err, int64_t row0, cudaStream_t s) {
  const int grid = (rows + PRO_WARPS - 1) / PRO_WARPS;
  prof_before("kd_teacher_prologue", s);
#define KD_PROLOGUE(E_)                                                                                          \
  kd_teacher_prologue_kernel<E_><<<grid, PRO_WARPS * 32, 0, s>>>(ids, tlog, rows, K, V, inv_tau, ids_sorted, \
                                                                 p_sorted, negent, err, row0)
  if (K <= 32) KD_PROLOGUE(1);
  else if (K <= 64) KD_PROLOGUE(2);
  else if (K <= 128) KD_PROLOGUE(4);
  else if (K <= 256) KD_PROLOGUE(8);
  else if (K <= 512) KD_PROLOGUE(16);
  else KD_PROLOGUE(32);
#undef KD_PROLOGUE
  prof_after(s);
  return cudaGetLastError();
}

// ------------------------------------------------------- lse combine ---
// Merge the per-unit (max, sum, gather) partials of each position into
//   lse_t = ln 2 * (M + log2 sum_u s_u 2^(m_u - M)),  KL_t = negent_t - G_t + lse_t
// ([ART] fused-loss paragraph: the running accumulator of the fused loss).

// Block = 32 rows x 8 unit phases: thread (x, y) folds the partials of row x from units
// y, y + 8, ... into one running (max, scaled sum, gather) in a single pass (each load a
// 512-byte coalesced row of partials across the warp), then the 8 phases are merged in
// shared memory.
constexpr int LC_ROWS = 32, LC_PHASES = 8;

__global__ void __launch_bounds__(LC_ROWS * LC_PHASES)
    kd_lse_combine_kernel(const float4* __restrict__ partials, int n_units, int rows, int rows_pad,
                          const float* __restrict__ negent, float* __restrict__ lse_out,
                          float* __restrict__ kl_out) {
  __shared__ float sm_m[LC_PHASES][LC_ROWS], sm_s[LC_PHASES][LC_ROWS], sm_g[LC_PHASES][LC_ROWS];
  const int x = threadIdx.x, y = threadIdx.y;
  const int r = blockIdx.x * LC_ROWS + x;
  float M = -INFINITY, S = 0.f, G = 0.f;
  if (r < rows) {
#pragma unroll 4
    for (int u = y; u < n_units; u += LC_PHASES) {
      const float4 q = partials[size_t(u) * rows_pad + r];
      G += q.z;
      if (q.x != -INFINITY) {
        if (q.x > M) {
          S = S * exp2f(M - q.x) + q.y;
          M = q.x;
        } else {
          S += q.y * exp2f(q.x - M);
        }
      }
    }
  }
  sm_m[y][x] = M;
  sm_s[y][x] = S;
  sm_g[y][x] = G;
  __syncthreads();
  if (y == 0 && r < rows) {
    for (int k = 1; k < LC_PHASES; ++k) {
      const float m2 = sm_m[k][x], s2 = sm_s[k][x];
      G += sm_g[k][x];
      if (m2 != -INFINITY) {
        if (m2 > M) {
          S = S * exp2f(M - m2) + s2;
          M = m2;
        } else {
          S += s2 * exp2f(m2 - M);
        }
      }
    }
    const float lse = (M + log2f(S)) * 0.69314718055994531f;
    lse_out[r] = lse;
    kl_out[r] = negent[r] - G + lse;
  }
}

cudaError_t launch_lse_combine(const float4* partials, int n_units_per_row, int rows, const float* negent,
                               float inv_tau, float* lse_out, float* kl_out, cudaStream_t s) {
  (void)inv_tau;
  const int rows_pad = ((rows + BM - 1) / BM) * BM;
  prof_before("kd_lse_combine", s);
  kd_lse_combine_kernel<<<(rows + LC_ROWS - 1) / LC_ROWS, dim3(LC_ROWS, LC_PHASES), 0, s>>>(
      partials, n_units_per_row, rows, rows_pad, negent, lse_out, kl_out);
  prof_after(s);
  return cudaGetLastError();
}

// ------------------------------------------------------- loss reduce ---
// loss = sum over valid positions of KL_t / N_valid, 0 if none ([ART] drop-in
// KL term; the token mean with a padding mask).  One block, fixed summation
// order in fp64, so the result is deterministic.

__global__ void __launch_bounds__(1024)
    kd_loss_reduce_kernel(const float* __restrict__ kl, const uint8_t* __restrict__ mask, int64_t N,
                          const int32_t* __restrict__ n_valid, float* __restrict__ loss_out) {
  __shared__ double sh[1024];
  double acc = 0.0;
  for (int64_t i = threadIdx.x; i < N; i += blockDim.x)
    if (mask == nullptr || mask[i] != 0) acc += double(kl[i]);
  sh[threadIdx.x] = acc;
  __syncthreads();
  for (int w = blockDim.x >> 1; w > 0; w >>= 1) {
    if (int(threadIdx.x) < w) sh[threadIdx.x] += sh[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int nv = *n_valid;
    *loss_out = nv > 0 ? float(sh[0] / double(nv)) : 0.f;
  }
}

cudaError_t launch_loss_reduce(const float* kl, const uint8_t* mask, int64_t N, const int32_t* n_valid,
                               float* loss_out, cudaStream_t s) {
  prof_before("kd_loss_reduce", s);
  kd_loss_reduce_kernel<<<1, 1024, 0, s>>>(kl, mask, N, n_valid, loss_out);
  prof_after(s);
  return cudaGetLastError();
}

// ------------------------------------------- dZ from stored logits ---
// Forward-chunked backward ([ART] fused-loss paragraph, second formulation: the
// chunk's student logits were kept by the forward pass, so the backward reads
// them instead of recomputing the projection):
//   dZ_t,v = grad_loss * mask_t / (N_valid * tau) * (2^(z_t,v log2e / tau - lse_t log2e) - p_t,v)
// Both z and dZ use the blocked layout [V/64][rows][64].  The dense part runs over
// contiguous 16-byte vectors; the K cached ids of each row are then rewritten
// with their teacher probability subtracted (one rounding, as in the fused path).

__device__ __forceinline__ float dz_rowscale(const uint8_t* mask, int t, const float* grad_loss,
                                             const int32_t* n_valid, float inv_tau) {
  const int nv = *n_valid;
  const bool valid = (mask == nullptr) || (mask[t] != 0);
  return (valid && nv > 0) ? (*grad_loss) * inv_tau / float(nv) : 0.f;
}

// dZ of one chunk from its kept bf16 logits: both in the blocked layout [V/64][rows][64].
// A thread owns one (row, 8-column group) of a 64-column block, so its row constants are
// computed once, and walks vocabulary blocks gridDim.y apart, four loads in flight;
// consecutive threads cover consecutive 16-byte pieces of one block (coalesced).
__global__ void __launch_bounds__(256) kd_dz_from_z_kernel(const uint16_t* __restrict__ z, int64_t N, int64_t c0,
                                                           int rows, int64_t V, int64_t nvb, int64_t rows_pad,
                                                           const float* __restrict__ lse,
                                                           const uint8_t* __restrict__ mask,
                                                           const float* __restrict__ grad_loss,
                                                           const int32_t* __restrict__ n_valid, float inv_tau,
                                                           uint16_t* __restrict__ dz) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= rows * 8) return;
  const int t = r >> 3, j8 = r & 7;
  const float scale2 = 1.4426950408889634f * inv_tau;
  const float lse2 = lse[t] * 1.4426950408889634f;
  const float rs = dz_rowscale(mask, t, grad_loss, n_valid, inv_tau);
  const uint16_t* zr = z + (c0 + t) * 64 + j8 * 8;  // + vb * N * 64
  uint16_t* dr = dz + int64_t(t) * 64 + j8 * 8;     // + vb * rows_pad * 64
  auto one = [&](int64_t vb, const uint4& zin) {
    const int64_t v0 = vb * 64 + j8 * 8;
    const uint32_t w[4] = {zin.x, zin.y, zin.z, zin.w};
    float q[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float zv = __uint_as_float((w[e >> 1] >> (16 * (e & 1))) << 16);
      q[e] = (v0 + e < V) ? rs * ex2_approx(fmaf(zv, scale2, -lse2)) : 0.f;
    }
    uint4 out;
    out.x = pack_bf16x2(q[0], q[1]);
    out.y = pack_bf16x2(q[2], q[3]);
    out.z = pack_bf16x2(q[4], q[5]);
    out.w = pack_bf16x2(q[6], q[7]);
    *reinterpret_cast<uint4*>(dr + vb * rows_pad * 64) = out;
  };
  const int64_t step = gridDim.y;
  int64_t vb = blockIdx.y;
  for (; vb + 3 * step < nvb; vb += 4 * step) {
    uint4 zin[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) zin[u] = __ldcs(reinterpret_cast<const uint4*>(zr + (vb + u * step) * N * 64));
#pragma unroll
    for (int u = 0; u < 4; ++u) one(vb + u * step, zin[u]);
  }
  for (; vb < nvb; vb += step) one(vb, __ldcs(reinterpret_cast<const uint4*>(zr + vb * N * 64)));
}

__global__ void kd_dz_fixup_kernel(const uint16_t* __restrict__ z, int64_t N, int64_t c0, int rows, int64_t V,
                                   int64_t rows_pad, const float* __restrict__ lse, const uint8_t* __restrict__ mask,
                                   const float* __restrict__ grad_loss, const int32_t* __restrict__ n_valid,
                                   float inv_tau, const int32_t* __restrict__ ids_sorted,
                                   const float* __restrict__ p_sorted, int K, uint16_t* __restrict__ dz) {
  const float scale2 = 1.4426950408889634f * inv_tau;
  const int64_t total = int64_t(rows) * K;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
    const int t = int(i / K);
    const int32_t v = ids_sorted[i];
    if (v < 0 || int64_t(v) >= V) continue;  // reported by the prologue
    const int64_t vb = v >> 6, j = v & 63;
    const float zv = __uint_as_float(uint32_t(z[(vb * N + c0 + t) * 64 + j]) << 16);
    const float q = ex2_approx(fmaf(zv, scale2, -lse[t] * 1.4426950408889634f));
    const float rs = dz_rowscale(mask, t, grad_loss, n_valid, inv_tau);
    const uint32_t packed = pack_bf16x2(rs * (q - p_sorted[i]), 0.f);
    dz[(vb * rows_pad + t) * 64 + j] = uint16_t(packed & 0xFFFFu);
  }
}

cudaError_t launch_dz_from_z(const uint16_t* z, int64_t N, int64_t c0, int rows, int64_t V, int64_t nvb,
                             int64_t rows_pad, const float* lse, const uint8_t* mask, const float* grad_loss,
                             const int32_t* n_valid, float inv_tau, const int32_t* ids_sorted, const float* p_sorted,
                             int K, uint16_t* dz, cudaStream_t s) {
  // rows * 8 threads in x; enough vocabulary-block strides in y for ~8 blocks of 256 per SM
  const int gx = (rows * 8 + 255) / 256;
  int gy = (8 * gemm_max_grid() + gx - 1) / gx;
  if (int64_t(gy) > nvb) gy = int(nvb);
  if (gy > 65535) gy = 65535;
  prof_before("kd_dz_from_z", s);
  kd_dz_from_z_kernel<<<dim3(gx, gy), 256, 0, s>>>(z, N, c0, rows, V, nvb, rows_pad, lse, mask, grad_loss, n_valid,
                                                    inv_tau, dz);
  prof_after(s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prof_before("kd_dz_fixup", s);
  kd_dz_fixup_kernel<<<(rows * K + 255) / 256, 256, 0, s>>>(z, N, c0, rows, V, rows_pad, lse, mask, grad_loss,
                                                            n_valid, inv_tau, ids_sorted, p_sorted, K, dz);
  prof_after(s);
  return cudaGetLastError();
}

// -------------------------------------------------- split-K reduction ---
// out[i] = sum over s of parts[s * stride + i], in split order (deterministic),
// to bf16 or fp32.  count and stride are multiples of 4.

__global__ void kd_split_reduce_kernel(const float4* __restrict__ parts, int splits, int64_t stride4,
                                       int64_t count4, void* __restrict__ out, int out_bf16) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < count4; i += int64_t(gridDim.x) * blockDim.x) {
    float4 a = parts[i];
    for (int sp = 1; sp < splits; ++sp) {
      const float4 b = parts[sp * stride4 + i];
      a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
    }
    if (out_bf16) {
      uint2 v;
      v.x = pack_bf16x2(a.x, a.y);
      v.y = pack_bf16x2(a.z, a.w);
      reinterpret_cast<uint2*>(out)[i] = v;
    } else {
      reinterpret_cast<float4*>(out)[i] = a;
    }
  }
}

cudaError_t launch_split_reduce(const float* parts, int splits, int64_t split_stride, int64_t count, void* out,
                                int out_bf16, cudaStream_t s) {
  const int64_t count4 = count / 4;
  int grid = int((count4 + 255) / 256);
  const int cap = 4 * gemm_max_grid();
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  prof_before("kd_split_reduce", s);
  kd_split_reduce_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const float4*>(parts), splits, split_stride / 4,
                                              count4, out, out_bf16);
  prof_after(s);
  return cudaGetLastError();
}

// ------------------------------------------------- bounded-wait check ---
// Waits on an mbarrier that nothing ever arrives at, with the same bounded
// wait the projection engine uses, so that a test can see the wait give up and
// report KD_ERR_TIMEOUT through the workspace error word.

__global__ void kd_wait_timeout_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_wait(&bar, 0, &abort_flag, err, 0x7e57u, limit_ns);
  }
  __syncthreads();
}

cudaError_t launch_wait_timeout(uint32_t* err, uint64_t limit_ns, cudaStream_t s) {
  prof_before("kd_wait_timeout", s);
  kd_wait_timeout_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  prof_after(s);
  return cudaGetLastError();
}

// ------------------------------------------------- row logsumexp of tiles ---
// A row's logsumexp from the per-tile pieces the teacher projection's epilogue leaves: per
// BN-column tile t its largest stored value m_t (bf16 bits) and s_t = the sum of
// 2^((z - m_t) log2 e) over its stored values z.  lse = M + ln(sum_t s_t 2^((m_t - M) log2 e)),
// M the row's largest m_t.  One warp per row; a NaN in any tile's sum makes the row's NaN.

constexpr int TL_WARPS = 8;

__global__ void __launch_bounds__(TL_WARPS * 32)
    kd_tile_lse_kernel(const uint16_t* __restrict__ tile_max, const float* __restrict__ tile_sum, int64_t ld,
                       int ntiles, int64_t rows, float* __restrict__ lse) {
  const int64_t row = int64_t(blockIdx.x) * TL_WARPS + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = int(threadIdx.x & 31u);
  const uint16_t* tm = tile_max + row * ld;
  const float* ts = tile_sum + row * ld;
  float M = -INFINITY;
  for (int t = lane; t < ntiles; t += 32) M = fmaxf(M, __uint_as_float(uint32_t(tm[t]) << 16));
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float S = 0.f;
  for (int t = lane; t < ntiles; t += 32) {
    const float m = __uint_as_float(uint32_t(tm[t]) << 16), q = ts[t];
    S += m == -INFINITY ? (q != q ? q : 0.f) : q * ex2_approx((m - M) * 1.4426950408889634f);
  }
  for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
  if (lane == 0) lse[row] = M == -INFINITY ? (S != S ? S : -INFINITY) : M + log2f(S) * 0.69314718055994531f;
}

cudaError_t launch_tile_lse(const uint16_t* tile_max, const float* tile_sum, int64_t ld, int ntiles, int64_t rows,
                            float* lse, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  prof_before("kd_tile_lse", s);
  kd_tile_lse_kernel<<<unsigned((rows + TL_WARPS - 1) / TL_WARPS), TL_WARPS * 32, 0, s>>>(tile_max, tile_sum, ld,
                                                                                          ntiles, rows, lse);
  prof_after(s);
  return cudaGetLastError();
}

}  // namespace kd
