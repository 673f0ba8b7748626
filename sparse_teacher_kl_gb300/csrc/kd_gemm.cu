// The projection engine: a persistent, warp-specialised bf16 GEMM on the
// fifth-generation tensor cores (tcgen05.mma, fp32 accumulators in tensor
// memory), fed by TMA, with the loss arithmetic fused into the epilogue.
//
// One CTA per SM.  Warp 0 issues TMA loads into a shared-memory ring, warp 1
// owns tensor memory and issues the MMAs (one thread), warps 2..5 drain finished
// accumulators (128 rows x 256 columns per CTA) from tensor memory while the next
// tile is being multiplied into the other half of it (512 columns, double-buffered).
// A product with at least two row tiles runs as CTA pairs (clusters of two): each
// pair computes a 256 x 256 tile with tcgen05 cta_group::2 MMAs, every CTA loading
// its own half of both operands with plain (non-multicast) TMA copies.
//
// Epilogues (the loss steps of the fused chunked KL, [ART] paragraph on the
// second fix; [DAI] "As duas inovações" item 2):
//   EPI_LSE   z = H_c W^T never leaves the chip: per row, a running max and
//             sum of 2^((z - max) log2e / tau) across the vocabulary tiles of a
//             unit, plus sum_k p_k z_id_k for the cached ids that fall in them;
//             one (max, sum, gather) partial per row and unit.
//   EPI_DZ    the backward recompute: dZ = scale * (2^(z log2e/tau - lse log2e)
//             - p on the cached ids), rounded to bf16 into a [rows, ldz] buffer.
//   EPI_LSE_Z as EPI_LSE, and also writes the raw logits (bf16) out for a
//             backward pass that does not recompute them (forward-chunked mode).
//   EPI_STORE / EPI_ACCUM  plain C = acc / C += acc for the gradient products.
#include <math.h>
#include <stdio.h>

#include "kd_device.cuh"
#include "kd_host_state.h"
#include "kd_internal.h"

namespace kd {

constexpr int MAX_STAGES = 6;
// EPI_ACCUM with a reduction depth K up to this adds its output through shared memory and
// TMA reduce-adds (tmap_c: fp32 C, 32 x 32 boxes, 128-byte swizzle); deeper, each thread adds
// its own row with vector reductions.
constexpr int ACCUM_STAGED_MAX_K = 2048;

struct __align__(8) GemmSmemTail {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
};

// Shared-memory ring per CTA.  One CTA per tile (CG = 1): a stage holds A 128 x 64 and
// B 256 x 64 (48 KB), 4 stages.  CTA pair per tile (CG = 2, tcgen05 cta_group::2): each
// CTA holds its 128 rows of A and its 128 columns of B for KKB 64-deep k-blocks: two
// when both operands are K-major (64 KB, 3 stages; every operand of a stage in one
// depth-2 TMA box), else one (32 KB, PAIR_ONE_BLOCK_STAGES stages).
constexpr int PAIR_ONE_BLOCK_STAGES = 6;

template <int CG, int KKB>
struct Geo {
  static constexpr int kKB = KKB;  // 64-deep k-blocks per stage
  static constexpr int kStages = CG == 1 ? STAGES : (KKB == 2 ? 3 : PAIR_ONE_BLOCK_STAGES);
  static constexpr int kA = STAGE_A_BYTES * kKB;
  static constexpr int kB = (CG == 2 ? STAGE_B_BYTES / 2 : STAGE_B_BYTES) * kKB;
  static constexpr int kStage = kA + kB;
  static constexpr size_t kSmem =
      1024 /*alignment slack*/ + size_t(kStages) * kStage + STAGING_BYTES + sizeof(GemmSmemTail);
  static_assert(CG == 2 || KKB == 1, "two k-blocks per stage only for CTA pairs");
  static_assert(kStages <= MAX_STAGES, "barrier arrays");
  static_assert(kSmem <= 232448, "shared memory budget of one CTA");
};

// Unit u -> tile coordinates.  LSE/DZ walk the vocabulary (n) slowly so that
// every CTA in flight reads the same few W tiles while the small H chunk stays
// in L2; the gradient products walk n fastest so that CTAs in flight share A.
// K ranges are in steps of kkb 64-deep k-blocks (one ring stage each).
__device__ __forceinline__ void unit_coords(const GemmProblem& p, int u, uint32_t crank, int kkb, int& m_blk,
                                            int& n_first, int& n_count, int& kb_lo, int& kb_hi, int& split) {
  const int k_blocks = ((p.K + BK - 1) / BK + kkb - 1) / kkb;
  const int m_groups = (p.m_tiles + p.cluster - 1) / p.cluster;
  if (p.epi == EPI_LSE || p.epi == EPI_DZ || p.epi == EPI_LSE_Z) {
    const int g = u / m_groups;
    m_blk = (u - g * m_groups) * p.cluster + int(crank);
    n_first = g * p.n_group;
    n_count = min(p.n_group, p.n_tiles - n_first);
    kb_lo = 0;
    kb_hi = k_blocks;
    split = 0;
  } else if (p.m_fast) {
    // n slowest, m fastest (no split): the CTAs in flight share a few B tiles, each
    // read from HBM once, and the A operand stays in L2
    const int n = u / m_groups;
    m_blk = (u - n * m_groups) * p.cluster + int(crank);
    n_first = n;
    n_count = 1;
    kb_lo = 0;
    kb_hi = k_blocks;
    split = 0;
  } else {
    // split slowest, then m, then n: the CTAs in flight share one K range, so each
    // A slab is read by all n tiles and each B slab by all m tiles from L2.
    const int per_split = m_groups * p.n_tiles;
    split = u / per_split;
    const int r = u - split * per_split;
    const int mg = r / p.n_tiles;
    m_blk = mg * p.cluster + int(crank);
    n_first = r - mg * p.n_tiles;
    n_count = 1;
    kb_lo = int((int64_t(k_blocks) * split) / p.k_splits);
    kb_hi = int((int64_t(k_blocks) * (split + 1)) / p.k_splits);
  }
}

template <int EPI, int CG, int KKB>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    kd_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                   const __grid_constant__ CUtensorMap tmap_c, const GemmProblem p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using G = Geo<CG, KKB>;
  uint8_t* stage_base = smem;
  uint8_t* staging = smem + size_t(G::kStages) * G::kStage;  // 1024-aligned output boxes of the epilogue warps
  GemmSmemTail* tail = reinterpret_cast<GemmSmemTail*>(staging + STAGING_BYTES);
  volatile uint32_t* abort_flag = &tail->abort_flag;

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const uint32_t crank = CG == 2 ? cluster_ctarank() : 0u;
  const int u_first = int(blockIdx.x) / p.cluster;
  const int u_step = int(gridDim.x) / p.cluster;

  if (threadIdx.x == 0) {
    for (int s = 0; s < G::kStages; ++s) {
      mbar_init(&tail->full[s], 1);
      // released once by the MMA thread (for a pair: the first CTA's, on both CTAs)
      mbar_init(&tail->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tail->tfull[a], 1);
      // the pair's MMA thread waits for both CTAs' epilogues
      mbar_init(&tail->tempty[a], (CG == 2 && crank == 0) ? 256u : 128u);
    }
    mbar_init(&tail->drain, 1);
    tail->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmap_a);
    tma_prefetch_map(&tmap_b);
    if (EPI == EPI_DZ || EPI == EPI_LSE_Z) tma_prefetch_map(&tmap_c);
  }
  if (warp == 1) {
    if (CG == 2) tmem_alloc_pair(&tail->tmem_base, TMEM_COLS); else tmem_alloc(&tail->tmem_base, TMEM_COLS);
  }
  tc_fence_before();
  __syncthreads();
  if (CG == 2) cluster_sync();  // the peer's barriers exist before any commit or copy reaches them
  tc_fence_after();
  const uint32_t tmem_base = tail->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int u = u_first; u < p.n_units && ok; u += u_step) {
        int m_blk, n_first, n_count, kb_lo, kb_hi, split;
        unit_coords(p, u, crank, G::kKB, m_blk, n_first, n_count, kb_lo, kb_hi, split);
        for (int nb = n_first; nb < n_first + n_count && ok; ++nb) {
          for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
            const uint32_t s = it % G::kStages;
            const uint32_t ph = (it / G::kStages) & 1u;
            if (!mbar_wait(&tail->empty[s], ph ^ 1u, abort_flag, p.err, 0x100u)) {
              ok = false;
              break;
            }
            uint8_t* sa = stage_base + size_t(s) * G::kStage;
            uint8_t* sb = sa + G::kA;
            if (CG == 2) {
              // both CTAs' halves complete on the first CTA's barrier, where the MMA waits
              const uint32_t bar0 = mapa_u32(&tail->full[s], 0);
              if (crank == 0) mbar_arrive_expect_tx(&tail->full[s], 2 * G::kStage);
              // stage kb = k-blocks kKB kb .. kKB kb + kKB - 1, elements k0 .. k0 + 64 kKB - 1
              const int k0 = kb * BK * G::kKB;
              if (p.a_blocked) {
                // blocked dZ [vocab/64][row][64]: K-major takes 128 rows of kKB vocabulary
                // blocks, MN-major two vocabulary blocks of 64 kKB rows (tokens)
                if (p.a_mn == 0) tma_load_3d_pair(sa, &tmap_a, bar0, 0, m_blk * BM, kb * G::kKB);
                else tma_load_3d_pair(sa, &tmap_a, bar0, 0, k0, m_blk * (BM / 64));
              } else if (p.a_mn == 0) {
                if (p.a_k3d) {
                  tma_load_3d_pair(sa, &tmap_a, bar0, 0, m_blk * BM, kb * G::kKB);
                } else {
#pragma unroll
                  for (int j = 0; j < G::kKB; ++j)
                    tma_load_2d_pair(sa + j * (G::kA / G::kKB), &tmap_a, bar0, k0 + j * BK, m_blk * BM);
                }
              } else if (p.a_box2) {
                tma_load_3d_pair(sa, &tmap_a, bar0, 0, k0, m_blk * (BM / 64));
              } else {
#pragma unroll
                for (int j = 0; j < BM / 64; ++j)
                  tma_load_2d_pair(sa + j * (G::kA / 2), &tmap_a, bar0, m_blk * BM + j * 64, k0);
              }
              // this CTA's 128 columns of the pair's 256-column B tile
              const int col = nb * BN + int(crank) * (BN / 2);
              if (p.b_mn == 0) {
                if (p.b_k3d) {
                  tma_load_3d_pair(sb, &tmap_b, bar0, 0, col, kb * G::kKB);
                } else {
#pragma unroll
                  for (int j = 0; j < G::kKB; ++j)
                    tma_load_2d_pair(sb + j * (G::kB / G::kKB), &tmap_b, bar0, k0 + j * BK, col);
                }
              } else if (p.b_box2) {
                tma_load_3d_pair(sb, &tmap_b, bar0, 0, k0, col / 64);
              } else {
#pragma unroll
                for (int j = 0; j < BN / 128; ++j)
                  tma_load_2d_pair(sb + j * (G::kB / 2), &tmap_b, bar0, col + j * 64, k0);
              }
              continue;
            }
            mbar_arrive_expect_tx(&tail->full[s], G::kStage);
            if (p.a_blocked) {
              // blocked dZ [vocab/64][row][64]: K-major A walks vocabulary blocks; MN-major
              // A takes the two 64-wide vocabulary blocks of its 128 rows
              if (p.a_mn == 0) {
                tma_load_3d(sa, &tmap_a, &tail->full[s], 0, m_blk * BM, kb);
              } else {
#pragma unroll
                for (int j = 0; j < BM / 64; ++j)
                  tma_load_3d(sa + j * 8192, &tmap_a, &tail->full[s], 0, kb * BK, m_blk * (BM / 64) + j);
              }
            } else if (p.a_mn == 0) {
              tma_load_2d(sa, &tmap_a, &tail->full[s], kb * BK, m_blk * BM);
            } else {
#pragma unroll
              for (int j = 0; j < BM / 64; ++j)
                tma_load_2d(sa + j * 8192, &tmap_a, &tail->full[s], m_blk * BM + j * 64, kb * BK);
            }
            if (p.b_mn == 0) {
              tma_load_2d(sb, &tmap_b, &tail->full[s], kb * BK, nb * BN);
            } else {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j)
                tma_load_2d(sb + j * 8192, &tmap_b, &tail->full[s], nb * BN + j * 64, kb * BK);
            }
          }
        }
      }
      if (!ok && (CG == 1 || crank == 0)) {
        // Let the copies already issued land before the CTA can exit (for a pair, all of
        // them complete on the first CTA's barriers).
        const uint32_t first = it > uint32_t(G::kStages) ? it - G::kStages : 0;
        for (uint32_t j = first; j < it; ++j) {
          volatile uint32_t never = 0;
          mbar_wait(&tail->full[j % G::kStages], (j / G::kStages) & 1u, &never, nullptr, 0);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && (CG == 1 || crank == 0)) {  // a pair's MMAs are issued by its first CTA
      const uint32_t idesc = idesc_bf16_f32(BM * CG, BN, p.a_mn, p.b_mn);
      // A 16-deep step kk of a stage: K-major operands hold each k-block as rows of 128 B
      // (the second k-block kA / 2 or kB / 2 further on), MN-major ones hold each 64-column
      // block as kKB * 64 rows of 128 B (LBO between the blocks).
      const uint32_t a_lbo = p.a_mn ? uint32_t(BK * G::kKB * 128) : 16u;
      const uint32_t b_lbo = p.b_mn ? uint32_t(BK * G::kKB * 128) : 16u;
      uint32_t it = 0, acc_it = 0;
      bool ok = true;
      for (int u = u_first; u < p.n_units && ok; u += u_step) {
        int m_blk, n_first, n_count, kb_lo, kb_hi, split;
        unit_coords(p, u, crank, G::kKB, m_blk, n_first, n_count, kb_lo, kb_hi, split);
        for (int nb = n_first; nb < n_first + n_count && ok; ++nb, ++acc_it) {
          const uint32_t a = acc_it & 1u;
          const uint32_t aph = (acc_it >> 1) & 1u;
          if (!mbar_wait(&tail->tempty[a], aph ^ 1u, abort_flag, p.err, 0x200u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + a * BN;
          for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
            const uint32_t s = it % G::kStages;
            const uint32_t ph = (it / G::kStages) & 1u;
            if (!mbar_wait(&tail->full[s], ph, abort_flag, p.err, 0x300u)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(stage_base + size_t(s) * G::kStage);
            const uint32_t sb = sa + G::kA;
            // 16-deep steps of this stage inside K (a pair's last stage may hold one
            // k-block of zeros past the end of K: skip its MMAs)
            const int ksteps = (p.K - kb * BK * G::kKB + 15) / 16;
#pragma unroll
            for (int k = 0; k < G::kKB * (BK / 16); ++k) {
              if (CG == 2 && k >= BK / 16 && k >= ksteps) break;
              const uint32_t a_off = p.a_mn ? uint32_t(k) * 2048u : uint32_t(k >> 2) * (G::kA / G::kKB) + (k & 3) * 32u;
              const uint32_t b_off = p.b_mn ? uint32_t(k) * 2048u : uint32_t(k >> 2) * (G::kB / G::kKB) + (k & 3) * 32u;
              const uint64_t ad = sdesc_sw128(sa + a_off, a_lbo);
              const uint64_t bd = sdesc_sw128(sb + b_off, b_lbo);
              if (CG == 2) umma_bf16_pair(d_tmem, ad, bd, idesc, (kb != kb_lo || k != 0) ? 1u : 0u);
              else umma_bf16(d_tmem, ad, bd, idesc, (kb != kb_lo || k != 0) ? 1u : 0u);
            }
            if (CG == 2) umma_commit_pair_mc(&tail->empty[s], 0x3);
            else umma_commit(&tail->empty[s]);
          }
          if (ok) {
            if (CG == 2) umma_commit_pair_mc(&tail->tfull[a], 0x3); else umma_commit(&tail->tfull[a]);
          }
        }
      }
      // Drain: every MMA issued above has completed once this arrives.
      if (CG == 2) umma_commit_pair_mc(&tail->drain, 0x1); else umma_commit(&tail->drain);
      volatile uint32_t never = 0;
      mbar_wait(&tail->drain, 0, &never, p.err, 0x400u);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const uint32_t quarter = warp & 3u;  // tensor-memory lane quarter this warp may access
    const int r_local = int(quarter * 32u + lane);
    const uint32_t t_lane = tmem_base + ((quarter * 32u) << 16);
    const float scale2 = 1.4426950408889634f * p.inv_tau;  // log2(e) / tau
    uint8_t* my_staging = staging + quarter * 8192u;        // two 4 KB boxes of this warp
    uint32_t sbuf = 0;
    uint32_t acc_it = 0;
    bool ok = true;
    for (int u = u_first; u < p.n_units && ok; u += u_step) {
      int m_blk, n_first, n_count, kb_lo, kb_hi, split;
      unit_coords(p, u, crank, G::kKB, m_blk, n_first, n_count, kb_lo, kb_hi, split);
      const int row = m_blk * BM + r_local;

      // Per-row state for the loss epilogues.
      float run_m = -INFINITY, run_s = 0.f, run_g = 0.f;
      int cur = 0;
      int nid = 0x7fffffff;
      float np_ = 0.f;
      const int32_t* ids_row = nullptr;
      const float* p_row = nullptr;
      float lse2 = 0.f, rowscale = 0.f;
      if (EPI == EPI_LSE || EPI == EPI_DZ || EPI == EPI_LSE_Z) {
        const bool row_ok = row < p.rows;
        cur = p.Kt;
        if (row_ok) {
          ids_row = p.ids_sorted + size_t(row) * p.Kt;
          p_row = p.p_sorted + size_t(row) * p.Kt;
          const int v_lo = n_first * BN;
          int lo = 0, hi = p.Kt;  // first entry with id >= v_lo
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(ids_row + mid) < v_lo) lo = mid + 1; else hi = mid;
          }
          cur = lo;
          if (cur < p.Kt) {
            nid = __ldg(ids_row + cur);
            np_ = __ldg(p_row + cur);
          }
        }
        if (EPI == EPI_DZ && row_ok) {
          lse2 = p.lse[row] * 1.4426950408889634f;
          const int nv = *p.n_valid;
          const bool valid = (p.mask == nullptr) || (p.mask[row] != 0);
          rowscale = (valid && nv > 0) ? (*p.grad_loss) * p.inv_tau / float(nv) : 0.f;
        }
      }

      for (int nb = n_first; nb < n_first + n_count; ++nb, ++acc_it) {
        const uint32_t a = acc_it & 1u;
        const uint32_t aph = (acc_it >> 1) & 1u;
        float tmax = -INFINITY;  // EPI_STORE with tile_max: the row's largest value in this tile
        float tsm = -INFINITY, tss = 0.f;  // with tile_sum: running maximum and sum, rounded values
        // the tensor-memory loads below are warp-collective: decide per warp
        const bool got = mbar_wait(&tail->tfull[a], aph, abort_flag, p.err, 0x500u);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t_acc = t_lane + a * BN;

#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t raw[32];
          tmem_ld_32x32b_x32(t_acc + c * 32, raw);
          tmem_ld_wait();
          float x[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(raw[i]);
          const int col0 = nb * BN + c * 32;

          if (EPI == EPI_LSE_Z) {
            // forward-chunked: keep this tile's raw logits (bf16) for the backward pass
            uint8_t* box = my_staging + sbuf * 4096u;
            if ((c & 1) == 0) {
              if (lane == 0) bulk_wait_read<1>();
              __syncwarp();
            }
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
              uint4 v;
              v.x = pack_bf16x2(x[g8 * 8 + 0], x[g8 * 8 + 1]);
              v.y = pack_bf16x2(x[g8 * 8 + 2], x[g8 * 8 + 3]);
              v.z = pack_bf16x2(x[g8 * 8 + 4], x[g8 * 8 + 5]);
              v.w = pack_bf16x2(x[g8 * 8 + 6], x[g8 * 8 + 7]);
              const uint32_t j = uint32_t((c & 1) * 4 + g8);
              *reinterpret_cast<uint4*>(box + lane * 128u + ((j ^ (lane & 7u)) * 16u)) = v;
            }
            if (c & 1) {
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d(&tmap_c, box, 0, p.z_row0 + m_blk * BM + int(quarter) * 32, (col0 - 32) / 64);
                bulk_commit();
              }
              sbuf ^= 1u;
            }
          }
          if (EPI == EPI_LSE || EPI == EPI_LSE_Z) {
            if (row < p.rows) {
              // columns past the vocabulary do not exist
              if (col0 + 32 > p.N) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (col0 + i >= p.N) x[i] = -INFINITY;
              }
              float cm = x[0];
#pragma unroll
              for (int i = 1; i < 32; ++i) cm = fmaxf(cm, x[i]);
              if (cm != -INFINITY) {
                if (cm > run_m) {
                  run_s *= ex2_approx((run_m - cm) * scale2);
                  run_m = cm;
                }
                const float off = -run_m * scale2;
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                  s0 += ex2_approx(fmaf(x[i], scale2, off));
                  s1 += ex2_approx(fmaf(x[i + 1], scale2, off));
                }
                run_s += s0 + s1;
              }
              while (nid < col0 + 32) {
                run_g = fmaf(np_, select32(x, uint32_t(nid - col0)), run_g);
                ++cur;
                if (cur < p.Kt) {
                  nid = __ldg(ids_row + cur);
                  np_ = __ldg(p_row + cur);
                } else {
                  nid = 0x7fffffff;
                }
              }
            }
          } else if (EPI == EPI_DZ) {
            float q[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) q[i] = 0.f;
            if (row < p.rows) {
#pragma unroll
              for (int i = 0; i < 32; ++i) q[i] = ex2_approx(fmaf(x[i], scale2, -lse2));
              while (nid < col0 + 32) {
                const int off = nid - col0;
#pragma unroll
                for (int i = 0; i < 32; ++i) q[i] = (i == off) ? q[i] - np_ : q[i];
                ++cur;
                if (cur < p.Kt) {
                  nid = __ldg(ids_row + cur);
                  np_ = __ldg(p_row + cur);
                } else {
                  nid = 0x7fffffff;
                }
              }
              if (col0 + 32 > p.N) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (col0 + i >= p.N) q[i] = 0.f;
              }
            }
            // Stage bf16 dZ for this warp's 32 rows: two 32-column chunks fill one 32 x 64
            // box (128-byte rows, 128-byte swizzle), written out by one TMA store that clips
            // rows past the chunk and columns past the vocabulary.
            uint8_t* box = my_staging + sbuf * 4096u;
            if ((c & 1) == 0) {
              if (lane == 0) bulk_wait_read<1>();
              __syncwarp();
            }
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
              uint4 v;
              v.x = pack_bf16x2(q[g8 * 8 + 0] * rowscale, q[g8 * 8 + 1] * rowscale);
              v.y = pack_bf16x2(q[g8 * 8 + 2] * rowscale, q[g8 * 8 + 3] * rowscale);
              v.z = pack_bf16x2(q[g8 * 8 + 4] * rowscale, q[g8 * 8 + 5] * rowscale);
              v.w = pack_bf16x2(q[g8 * 8 + 6] * rowscale, q[g8 * 8 + 7] * rowscale);
              const uint32_t j = uint32_t((c & 1) * 4 + g8);
              *reinterpret_cast<uint4*>(box + lane * 128u + ((j ^ (lane & 7u)) * 16u)) = v;
            }
            if (c & 1) {
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d(&tmap_c, box, 0, m_blk * BM + int(quarter) * 32, (col0 - 32) / 64);
                bulk_commit();
              }
              sbuf ^= 1u;
            }
          } else if (EPI == EPI_ACCUM) {
            // C[row, col0 .. col0+31] += acc, each element exactly one addition per launch, as
            // a read-modify-write in L2 that nothing waits on.
            if (p.K <= ACCUM_STAGED_MAX_K) {
              // A shallow reduction leaves the launch bound by this read-modify-write: the
              // warp's 32 x 32 block goes to shared memory (two alternating 4 KB boxes, 128-byte
              // rows, 16-byte chunks swizzled by row, as tmap_c's 128-byte swizzle lays them
              // out) and one TMA reduce-add per box adds it to C, clipped at the edges.
              uint8_t* box = my_staging + (uint32_t(c) & 1u) * 4096u;
              if (lane == 0) bulk_wait_read<1>();  // this box's reduce from two chunks ago has read it
              __syncwarp();
#pragma unroll
              for (int g4 = 0; g4 < 8; ++g4)
                *reinterpret_cast<float4*>(box + lane * 128u + ((uint32_t(g4) ^ (lane & 7u)) * 16u)) =
                    make_float4(x[g4 * 4 + 0], x[g4 * 4 + 1], x[g4 * 4 + 2], x[g4 * 4 + 3]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_reduce_add_2d(&tmap_c, box, col0, m_blk * BM + int(quarter) * 32);
                bulk_commit();
              }
            } else if (row < p.M) {
              // deeper: fire-and-forget vector reductions of the thread's own row, which leave
              // the TMA unit to the operand loads
              float* dst = reinterpret_cast<float*>(p.C) + size_t(row) * p.ldc + col0;
#pragma unroll
              for (int g4 = 0; g4 < 8; ++g4) {
                if (col0 + g4 * 4 + 4 <= p.N)
                  red_add_v4(dst + g4 * 4, x[g4 * 4 + 0], x[g4 * 4 + 1], x[g4 * 4 + 2], x[g4 * 4 + 3]);
              }
            }
          } else if (p.c_tma) {
            // EPI_STORE through TMA: two 32-column chunks fill one 32 x 64 bf16 box of this
            // warp's 32 rows (128-byte rows, 128-byte swizzle); the store clips rows past M
            // and columns past N.
            uint8_t* box = my_staging + sbuf * 4096u;
            if ((c & 1) == 0) {
              if (lane == 0) bulk_wait_read<1>();
              __syncwarp();
            }
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
              uint4 v;
              v.x = pack_bf16x2(x[g8 * 8 + 0], x[g8 * 8 + 1]);
              v.y = pack_bf16x2(x[g8 * 8 + 2], x[g8 * 8 + 3]);
              v.z = pack_bf16x2(x[g8 * 8 + 4], x[g8 * 8 + 5]);
              v.w = pack_bf16x2(x[g8 * 8 + 6], x[g8 * 8 + 7]);
              const uint32_t j = uint32_t((c & 1) * 4 + g8);
              *reinterpret_cast<uint4*>(box + lane * 128u + ((j ^ (lane & 7u)) * 16u)) = v;
            }
            if (p.tile_max) {
              // rounding to bf16 is monotonic: the largest of the fp32 values, rounded, is the
              // largest stored value (fmaxf skips NaNs)
              float cm = -INFINITY;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (col0 + i < p.N) cm = fmaxf(cm, x[i]);
              tmax = fmaxf(tmax, cm);
              if (p.tile_sum) {
                // sum of 2^((z - m) log2 e) over the stored (rounded) values z, m the running
                // maximum of those values: the tile's maximum once the tile is done
                constexpr float kL2E = 1.4426950408889634f;
                if (cm != -INFINITY) {
                  const float cr = __uint_as_float(pack_bf16x2(cm, cm) << 16);
                  if (cr > tsm) {
                    tss *= ex2_approx((tsm - cr) * kL2E);  // 0 while nothing was summed
                    tsm = cr;
                  }
                  const float off = -tsm * kL2E;
                  float s0 = 0.f, s1 = 0.f;
#pragma unroll
                  for (int i = 0; i < 32; i += 2) {
                    const uint32_t w = pack_bf16x2(x[i], x[i + 1]);
                    const float e0 = ex2_approx(fmaf(__uint_as_float(w << 16), kL2E, off));
                    const float e1 = ex2_approx(fmaf(__uint_as_float(w & 0xFFFF0000u), kL2E, off));
                    s0 += col0 + i < p.N ? e0 : 0.f;
                    s1 += col0 + i + 1 < p.N ? e1 : 0.f;
                  }
                  tss += s0 + s1;
                } else {
#pragma unroll
                  for (int i = 0; i < 32; ++i)  // no number here: a NaN still makes the sum NaN
                    if (col0 + i < p.N && x[i] != x[i]) tss = x[i];
                }
              }
            }
            if (c & 1) {
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tmap_c, box, col0 - 32, m_blk * BM + int(quarter) * 32);
                bulk_commit();
              }
              sbuf ^= 1u;
            }
          } else {
            // EPI_STORE: C[row, col0 + i]
            if (row < p.M) {
              if (p.c_bf16) {
                uint16_t* dst =
                    reinterpret_cast<uint16_t*>(p.C) + size_t(split) * p.split_stride + size_t(row) * p.ldc + col0;
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                  // whole 8-column groups that start inside the matrix; the row stride ldc is
                  // a multiple of 8, so a group ending past column N stays inside its row
                  if (col0 + g8 * 8 < p.N && col0 + g8 * 8 + 8 <= p.ldc) {
                    uint4 v;
                    v.x = pack_bf16x2(x[g8 * 8 + 0], x[g8 * 8 + 1]);
                    v.y = pack_bf16x2(x[g8 * 8 + 2], x[g8 * 8 + 3]);
                    v.z = pack_bf16x2(x[g8 * 8 + 4], x[g8 * 8 + 5]);
                    v.w = pack_bf16x2(x[g8 * 8 + 6], x[g8 * 8 + 7]);
                    *reinterpret_cast<uint4*>(dst + g8 * 8) = v;
                  }
                }
              } else {
                float* dst =
                    reinterpret_cast<float*>(p.C) + size_t(split) * p.split_stride + size_t(row) * p.ldc + col0;
#pragma unroll
                for (int g4 = 0; g4 < 8; ++g4) {
                  if (col0 + g4 * 4 < p.N && col0 + g4 * 4 + 4 <= p.ldc) {
                    *reinterpret_cast<float4*>(dst + g4 * 4) =
                        make_float4(x[g4 * 4 + 0], x[g4 * 4 + 1], x[g4 * 4 + 2], x[g4 * 4 + 3]);
                  }
                }
              }
            }
          }
        }
        tc_fence_before();
        if (CG == 2 && crank != 0) mbar_arrive_remote(mapa_u32(&tail->tempty[a], 0));
        else mbar_arrive(&tail->tempty[a]);
        if (EPI == EPI_STORE && p.tile_max && ok && row < p.M) {
          p.tile_max[size_t(row) * p.ld_tile_max + nb] = uint16_t(pack_bf16x2(tmax, tmax) & 0xFFFFu);
          if (p.tile_sum) p.tile_sum[size_t(row) * p.ld_tile_max + nb] = tss;
        }
      }
      if ((EPI == EPI_LSE || EPI == EPI_LSE_Z) && ok && row < p.rows) {
        const int g = n_first / p.n_group;
        p.partials[size_t(g) * (p.m_tiles * BM) + row] =
            make_float4(run_m * scale2, run_s, run_g * p.inv_tau, 0.f);
      }
    }
    if ((EPI == EPI_DZ || EPI == EPI_LSE_Z || (EPI == EPI_STORE && p.c_tma) || (EPI == EPI_ACCUM && p.K <= ACCUM_STAGED_MAX_K)) && lane == 0)
      bulk_wait_all();  // output boxes done before exit
  }

  tc_fence_before();
  __syncthreads();
  if (CG == 2) cluster_sync();  // no commit or remote arrival of the peer can still target this CTA
  tc_fence_after();
  if (warp == 1) {
    if (CG == 2) tmem_dealloc_pair(tmem_base, TMEM_COLS); else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

static PerDevice<int> g_num_sms;

int gemm_max_grid() {
  int dev = 0, n = 1;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  g_num_sms.get(dev, &n, [](int d, int* v) {
    if (cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) return 1;
    if (*v <= 0) *v = 1;
    return 0;
  });
  return n;
}

// One launch of the engine.  CG = 1: `grid` single CTAs (at most one per unit).  CG = 2:
// clusters of two CTAs, as many pairs as can be resident at once (at most one per unit).
// The kernel's shared-memory attribute and the resident pair count are set up once per
// device (each template instance has its own).
template <int EPI, int CG, int KKB = 1>
static cudaError_t launch_one(const GemmProblem& p, const CUtensorMap& ta, const CUtensorMap& tb,
                              const CUtensorMap& tc, int grid, cudaStream_t s) {
  static PerDevice<int> max_pairs;  // CG = 2: resident clusters; CG = 1: 1 once set up
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int resident = 1;
  const int rc = max_pairs.get(dev, &resident, [](int, int* v) {
    cudaError_t r = cudaFuncSetAttribute(kd_gemm_kernel<EPI, CG, KKB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(Geo<CG, KKB>::kSmem));
    if (r != cudaSuccess) return int(r);
    *v = 1;
    if (CG == 2) {
      cudaLaunchConfig_t q = {};
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = 2;
      qa[0].val.clusterDim.y = 1;
      qa[0].val.clusterDim.z = 1;
      q.attrs = qa;
      q.numAttrs = 1;
      q.blockDim = dim3(GEMM_THREADS, 1, 1);
      q.dynamicSmemBytes = Geo<CG, KKB>::kSmem;
      q.gridDim = dim3(unsigned((gemm_max_grid() / 2) * 2), 1, 1);
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kd_gemm_kernel<EPI, CG, KKB>, &q) == cudaSuccess && n >= 1) *v = n;
    }
    return 0;
  });
  if (rc != 0) return rc > 0 ? cudaError_t(rc) : cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = Geo<CG, KKB>::kSmem;
  cfg.stream = s;
  if (CG == 2) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int pairs = grid / 2;
    if (pairs > resident) pairs = resident;
    if (pairs > p.n_units) pairs = p.n_units;
    if (pairs < 1) pairs = 1;
    cfg.gridDim = dim3(unsigned(pairs * 2), 1, 1);
  } else {
    if (grid > p.n_units) grid = p.n_units;
    cfg.gridDim = dim3(unsigned(grid), 1, 1);
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
  }
  e = cudaLaunchKernelEx(&cfg, kd_gemm_kernel<EPI, CG, KKB>, ta, tb, tc, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

static const char* gemm_name(int epi, int a_mn, int b_mn) {
  switch (epi) {
    case EPI_LSE: return "kd_proj_lse_fwd";
    case EPI_LSE_Z: return "kd_proj_lse_z_fwd";
    case EPI_DZ: return "kd_proj_dz_bwd";
    case EPI_STORE: return (a_mn == 0 && b_mn == 1) ? "kd_gemm_dz_w" : "kd_gemm_store";
    default: return (a_mn == 1 && b_mn == 1) ? "kd_gemm_dzT_h" : "kd_gemm_accum";
  }
}

cudaError_t launch_gemm(const GemmProblem& p, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                        int grid, cudaStream_t s) {
  if (p.n_units <= 0) return cudaSuccess;
  // CTA pairs run as clusters of two; everything else as single CTAs
  if (p.cluster != (p.cta_pair ? 2 : 1)) return cudaErrorInvalidValue;
  prof_before(gemm_name(p.epi, p.a_mn, p.b_mn), s);
  cudaError_t e;
  if (p.cta_pair) {
    const bool two = pair_kblocks(p.a_mn, p.b_mn) == 2;
    switch (p.epi) {
      // the loss sweeps read H and W K-major: always two k-blocks per stage
      case EPI_LSE: e = two ? launch_one<EPI_LSE, 2, 2>(p, ta, tb, tc, grid, s) : cudaErrorInvalidValue; break;
      case EPI_LSE_Z: e = two ? launch_one<EPI_LSE_Z, 2, 2>(p, ta, tb, tc, grid, s) : cudaErrorInvalidValue; break;
      case EPI_DZ: e = two ? launch_one<EPI_DZ, 2, 2>(p, ta, tb, tc, grid, s) : cudaErrorInvalidValue; break;
      case EPI_STORE:
        e = two ? launch_one<EPI_STORE, 2, 2>(p, ta, tb, tc, grid, s) : launch_one<EPI_STORE, 2, 1>(p, ta, tb, tc, grid, s);
        break;
      default:
        e = two ? launch_one<EPI_ACCUM, 2, 2>(p, ta, tb, tc, grid, s) : launch_one<EPI_ACCUM, 2, 1>(p, ta, tb, tc, grid, s);
        break;
    }
  } else {
    switch (p.epi) {
      case EPI_LSE: e = launch_one<EPI_LSE, 1>(p, ta, tb, tc, grid, s); break;
      case EPI_LSE_Z: e = launch_one<EPI_LSE_Z, 1>(p, ta, tb, tc, grid, s); break;
      case EPI_DZ: e = launch_one<EPI_DZ, 1>(p, ta, tb, tc, grid, s); break;
      case EPI_STORE: e = launch_one<EPI_STORE, 1>(p, ta, tb, tc, grid, s); break;
      default: e = launch_one<EPI_ACCUM, 1>(p, ta, tb, tc, grid, s); break;
    }
  }
  prof_after(s);
  return e;
}

}  // namespace kd
