// Offline top-K teacher cache: the K largest logits of every row of a dense
// bf16 [N, V] teacher-logits matrix, with their token ids ([ART] paragraph on
// the first fix; [DAI] "As duas inovações" item 1; [EPO] "Los dos cambios
// propuestos", first item).
//
// HBM-bound: every logit is read once (twice for a row whose guessed starting
// threshold, below, turned out too high).  Each element becomes a 48-bit
// composite
//   (order-preserving 16-bit key of the bf16 value) << 32 | (~column)
// which is unique per element and orders by value descending, then column
// ascending; the top-K are the K largest composites, so the result is exact with
// any number of ties.  A threshold key T is valid once at least K elements seen so
// far reach it: later elements then need key > T (an equal key comes with a larger
// column and ranks below those K).  Two kernels:
//  * K <= 256 (the pages' top-100): one warp per row, no block barrier (the
//    warp-per-row section below);
//  * 256 < K <= 1024: one CTA per row (grid-strided): the row streams through in
//    segments of 4096 elements into a shared candidate buffer; when it passes half
//    full, the K-th largest key in it is found with two byte histograms and only
//    what reaches it is kept; the survivors are sorted once at the end.
//
// Optionally the same pass also takes the full-row logsumexp of the teacher
// logits, so that the probability mass the cache drops, 1 - sum_k e^(t_k - lse),
// can be reported per position ([ART] paragraph on the top-K limitation).
#include <stdint.h>
#include <stdlib.h>

#include "kd_device.cuh"
#include "kd_internal.h"

namespace kd {

constexpr int TK_THREADS = 512;
constexpr int TK_VEC = 8;                      // bf16 per 16-byte load
constexpr int TK_SEG = TK_THREADS * TK_VEC;    // elements per segment
constexpr int TK_CHECK = 1;                    // segments between two looks at the buffer fill
constexpr int TK_CAP = 2 * TK_SEG;             // candidate buffer entries (a power of two: sort_desc)
constexpr int TK_PIPE = 4;                     // segments in flight per thread
constexpr int TK_ROUND = 8;                    // entries per thread per compaction round

static_assert((TK_CAP & (TK_CAP - 1)) == 0, "the bitonic sort pads the buffer to a power of two");
static_assert(TK_CAP >= (TK_CHECK + 1) * TK_SEG, "room for one check window after a compaction");

struct TopkSmem {
  unsigned long long buf[TK_CAP];
  uint32_t hist[256];
  float red_m[TK_THREADS / 32];
  float red_s[TK_THREADS / 32];
  uint32_t count;
  uint32_t sel_bin;
  uint32_t sel_need;
  uint32_t sel_above;
  uint32_t* err;  // the workspace error word (checked builds report bad indices there)
};

// bf16 bits -> unsigned key with the same order as the values (-0 == +0).
__device__ __forceinline__ uint32_t bf16_key(uint32_t b) {
  b &= 0xFFFFu;
  if (b == 0x8000u) b = 0u;
  return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}

__device__ __forceinline__ uint32_t comp_key(unsigned long long c) { return uint32_t(c >> 32); }

// Warp 0 finds, scanning bins from the top, the bin where the running count
// reaches `target`; stores the bin, the count still needed inside it and the
// count strictly above it.
__device__ void find_bin_from_top(TopkSmem& sm, uint32_t target) {
  if (threadIdx.x < 32) {
    const uint32_t lane = threadIdx.x;
    uint32_t local[8];
    uint32_t sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      local[j] = sm.hist[255 - (lane * 8 + j)];
      sum += local[j];
    }
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= uint32_t(o)) incl += t;
    }
    const uint32_t excl = incl - sum;
    if (excl < target && target <= incl) {
      uint32_t run = excl;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (run < target && target <= run + local[j]) {
          sm.sel_bin = 255 - (lane * 8 + j);
          sm.sel_need = target - run;
          sm.sel_above = run;
        }
        run += local[j];
      }
    }
  }
}

// K-th largest key among buf[0, count) (count >= K); also returns how many
// entries have key >= that value.
// hist[bin] += 1 for every lane with a valid bin, one atomic per distinct bin per warp
// (the keys near the top of a row fall in very few bins).  All 32 lanes call it.
__device__ __forceinline__ void hist_add_warp(uint32_t* hist, bool valid, uint32_t bin) {
  const uint32_t b = valid ? bin : 0xFFFFFFFFu;
  const uint32_t peers = __match_any_sync(0xffffffffu, b);
  if (valid && lane_id() == uint32_t(__ffs(peers) - 1)) atomicAdd(&hist[bin], uint32_t(__popc(peers)));
}

__device__ uint32_t kth_largest_key(TopkSmem& sm, uint32_t count, uint32_t K, uint32_t& count_ge) {
  for (int i = threadIdx.x; i < 256; i += TK_THREADS) sm.hist[i] = 0;
  __syncthreads();
  for (uint32_t base = threadIdx.x & ~31u; base < count; base += TK_THREADS) {
    const uint32_t i = base + lane_id();
    hist_add_warp(sm.hist, i < count, i < count ? comp_key(sm.buf[i]) >> 8 : 0u);
  }
  __syncthreads();
  find_bin_from_top(sm, K);
  __syncthreads();
  const uint32_t b1 = sm.sel_bin, need = sm.sel_need, above1 = sm.sel_above;
  __syncthreads();
  for (int i = threadIdx.x; i < 256; i += TK_THREADS) sm.hist[i] = 0;
  __syncthreads();
  for (uint32_t base = threadIdx.x & ~31u; base < count; base += TK_THREADS) {
    const uint32_t i = base + lane_id();
    const uint32_t k = i < count ? comp_key(sm.buf[i]) : 0u;
    hist_add_warp(sm.hist, i < count && (k >> 8) == b1, k & 255u);
  }
  __syncthreads();
  find_bin_from_top(sm, need);
  __syncthreads();
  const uint32_t b2 = sm.sel_bin;
  count_ge = above1 + sm.sel_above + sm.hist[b2];
  __syncthreads();
  return (b1 << 8) | b2;
}

// Append `c` (if `take`) to sm.buf with one shared atomic per warp.
__device__ __forceinline__ void warp_append(TopkSmem& sm, bool take, unsigned long long c) {
  const uint32_t ballot = __ballot_sync(0xffffffffu, take);
  if (ballot == 0) return;
  const uint32_t lane = lane_id();
  uint32_t base = 0;
  if (lane == 0) base = atomicAdd(&sm.count, uint32_t(__popc(ballot)));
  base = __shfl_sync(0xffffffffu, base, 0);
  const uint32_t at = base + __popc(ballot & ((1u << lane) - 1u));
  if (take && KD_DCHECK(at < uint32_t(TK_CAP), sm.err, 0x7001)) sm.buf[at] = c;
}

// Keep only the entries with key >= T, in place: rounds of TK_ROUND entries per
// thread are read into registers before any survivor of that round is written, and
// survivors never outnumber the entries read so far, so no unread entry is overwritten.
__device__ void filter_ge(TopkSmem& sm, uint32_t count, uint32_t T) {
  __syncthreads();
  if (threadIdx.x == 0) sm.count = 0;
  for (uint32_t base = 0; base < count; base += TK_ROUND * TK_THREADS) {
    unsigned long long held[TK_ROUND];
#pragma unroll
    for (int j = 0; j < TK_ROUND; ++j) {
      const uint32_t i = base + threadIdx.x + j * TK_THREADS;
      held[j] = (i < count) ? sm.buf[i] : 0ull;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < TK_ROUND; ++j) {
      const uint32_t i = base + threadIdx.x + j * TK_THREADS;
      warp_append(sm, i < count && comp_key(held[j]) >= T, held[j]);
    }
    __syncthreads();
  }
}

// Sort buf[0, count) descending (bitonic over the next power of two, padded
// with 0, which is below every real composite).
__device__ void sort_desc(TopkSmem& sm, uint32_t count) {
  uint32_t P = 1;
  while (P < count) P <<= 1;
  for (uint32_t i = count + threadIdx.x; i < P; i += TK_THREADS) sm.buf[i] = 0ull;
  __syncthreads();
  for (uint32_t k = 2; k <= P; k <<= 1) {
    for (uint32_t j = k >> 1; j > 0; j >>= 1) {
      for (uint32_t i = threadIdx.x; i < P; i += TK_THREADS) {
        const uint32_t ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = sm.buf[i], b = sm.buf[ixj];
          const bool desc = (i & k) == 0;
          if (desc ? (a < b) : (a > b)) {
            sm.buf[i] = b;
            sm.buf[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

// Bring the buffer back to at most TK_CAP - TK_CHECK * TK_SEG entries, all of them able
// to reach the top K; returns the new acceptance threshold (key must exceed it).
__device__ int compact(TopkSmem& sm, uint32_t K) {
  const uint32_t count = sm.count;
  uint32_t count_ge = 0;
  const uint32_t T = kth_largest_key(sm, count, K, count_ge);
  if (count_ge <= uint32_t(TK_CAP - TK_CHECK * TK_SEG)) {
    if (count_ge < count) filter_ge(sm, count, T);
    return int(T);
  }
  // Too many ties at T: order fully and keep exactly the K best.
  sort_desc(sm, count);
  if (threadIdx.x == 0) sm.count = K;
  __syncthreads();
  return int(comp_key(sm.buf[K - 1]));
}

__device__ __forceinline__ uint4 load_seg(const uint16_t* xr, int64_t V, int seg) {
  const int64_t i0 = int64_t(seg) * TK_SEG + int64_t(threadIdx.x) * TK_VEC;
  if (i0 + TK_VEC <= V) return __ldcs(reinterpret_cast<const uint4*>(xr + i0));
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int e = 0; e < TK_VEC; ++e)
    if (i0 + e < V) w[e >> 1] |= uint32_t(xr[i0 + e]) << (16 * (e & 1));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void __launch_bounds__(TK_THREADS, 2)
    kd_topk_kernel(const uint16_t* __restrict__ X, int64_t N, int64_t V, int64_t ld, int K,
                   int32_t* __restrict__ ids_out, float* __restrict__ vals_out, float* __restrict__ lse_out,
                   uint32_t* err) {
  extern __shared__ __align__(16) uint8_t tk_smem_raw[];
  TopkSmem& sm = *reinterpret_cast<TopkSmem*>(tk_smem_raw);
  if (threadIdx.x == 0) sm.err = err;  // read after the first barrier below
  const int nseg = int((V + TK_SEG - 1) / TK_SEG);

  for (int64_t row = blockIdx.x; row < N; row += gridDim.x) {
    const uint16_t* xr = X + row * ld;
    if (threadIdx.x == 0) sm.count = 0;
    int thresh = -1;  // accept every element until the first compaction
    // optional full-row logsumexp (base 2, per thread: running max and scaled sum)
    float lm = -INFINITY, ls = 0.f;
    uint4 pipe[TK_PIPE];
#pragma unroll
    for (int j = 0; j < TK_PIPE; ++j)
      if (j < nseg) pipe[j] = load_seg(xr, V, j);
    __syncthreads();

    // Candidate test in the float domain: key(x) > T  <=>  x > value(T) for ordinary
    // values (-0 and +0 compare equal either way); !(x <= tv) also lets NaN through to
    // the exact key test.  tv = NaN before the first compaction accepts everything.
    float tv = __int_as_float(0x7fc00000);
    int seg_start = 0;
    if (K <= TK_THREADS / 2 && nseg >= 2) {
      // Quick start: the K-th largest of the 512 per-thread maxima over the first two
      // segments is a key that at least K elements reach, so every element of the top K
      // has a key >= it.  Keep the elements of those segments that reach it; later
      // elements need a strictly larger key (an equal key with a larger column ranks
      // below those K).  This replaces compacting a buffer of 8192 entries.
      const int64_t i0a = int64_t(threadIdx.x) * TK_VEC;
      const int64_t i0b = int64_t(TK_SEG) + i0a;
      const uint32_t wa[4] = {pipe[0].x, pipe[0].y, pipe[0].z, pipe[0].w};
      const uint32_t wb[4] = {pipe[1].x, pipe[1].y, pipe[1].z, pipe[1].w};
      uint32_t ka[TK_VEC], kb[TK_VEC];
      uint32_t tmax = 0;
#pragma unroll
      for (int e = 0; e < TK_VEC; ++e) {
        ka[e] = (i0a + e < V) ? bf16_key(wa[e >> 1] >> (16 * (e & 1))) : 0u;
        kb[e] = (i0b + e < V) ? bf16_key(wb[e >> 1] >> (16 * (e & 1))) : 0u;
        tmax = max(tmax, max(ka[e], kb[e]));
      }
      if (lse_out != nullptr) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t* w = h ? wb : wa;
          const int64_t i0 = h ? i0b : i0a;
          float x2[TK_VEC];
          float vm = -INFINITY;
#pragma unroll
          for (int e = 0; e < TK_VEC; ++e) {
            const float xv = __uint_as_float((e & 1) ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16));
            x2[e] = (i0 + e < V) ? xv * 1.4426950408889634f : -INFINITY;
            vm = fmaxf(vm, x2[e]);
          }
          const float nm = fmaxf(lm, vm);
          if (nm != -INFINITY) {
            float acc = ls * ex2_approx(lm - nm);
#pragma unroll
            for (int e = 0; e < TK_VEC; ++e) acc += ex2_approx(x2[e] - nm);
            ls = acc;
            lm = nm;
          }
        }
      }
      sm.buf[threadIdx.x] = static_cast<unsigned long long>(tmax) << 32;
      __syncthreads();
      uint32_t count_ge = 0;
      const uint32_t T = kth_largest_key(sm, TK_THREADS, uint32_t(K), count_ge);
      if (threadIdx.x == 0) sm.count = 0;
      __syncthreads();
#pragma unroll
      for (int e = 0; e < TK_VEC; ++e)
        warp_append(sm, (i0a + e < V) && ka[e] >= T,
                    (static_cast<unsigned long long>(ka[e]) << 32) | uint32_t(~uint32_t(i0a + e)));
#pragma unroll
      for (int e = 0; e < TK_VEC; ++e)
        warp_append(sm, (i0b + e < V) && kb[e] >= T,
                    (static_cast<unsigned long long>(kb[e]) << 32) | uint32_t(~uint32_t(i0b + e)));
      thresh = int(T);
      const uint32_t tb = (T & 0x8000u) ? (T & 0x7FFFu) : (~T & 0xFFFFu);
      tv = __uint_as_float(tb << 16);
      if (TK_PIPE < nseg) pipe[0] = load_seg(xr, V, TK_PIPE);
      if (TK_PIPE + 1 < nseg) pipe[1] = load_seg(xr, V, TK_PIPE + 1);
      seg_start = 2;
      __syncthreads();
      const uint32_t cnt = sm.count;
      __syncthreads();
      if (cnt > uint32_t(TK_CAP - TK_CHECK * TK_SEG)) {  // many ties at T: make room first
        thresh = compact(sm, uint32_t(K));
        const uint32_t tb2 = (uint32_t(thresh) & 0x8000u) ? (uint32_t(thresh) & 0x7FFFu)
                                                          : (~uint32_t(thresh) & 0xFFFFu);
        tv = __uint_as_float(tb2 << 16);
      }
    }
    for (int base = 0; base < nseg; base += TK_PIPE) {
#pragma unroll
      for (int j = 0; j < TK_PIPE; ++j) {
        const int seg = base + j;
        if (seg < nseg && seg >= seg_start) {
          const uint4 v = pipe[j];
          if (seg + TK_PIPE < nseg) pipe[j] = load_seg(xr, V, seg + TK_PIPE);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
          const int64_t i0 = int64_t(seg) * TK_SEG + int64_t(threadIdx.x) * TK_VEC;
          float xf[TK_VEC];
#pragma unroll
          for (int e = 0; e < TK_VEC; ++e)
            xf[e] = __uint_as_float((e & 1) ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16));
          if (lse_out != nullptr) {
            float vm = -INFINITY;
            float x2[TK_VEC];
#pragma unroll
            for (int e = 0; e < TK_VEC; ++e) {
              x2[e] = (i0 + e < V) ? xf[e] * 1.4426950408889634f : -INFINITY;
              vm = fmaxf(vm, x2[e]);
            }
            const float nm = fmaxf(lm, vm);
            if (nm != -INFINITY) {
              float acc = ls * ex2_approx(lm - nm);
#pragma unroll
              for (int e = 0; e < TK_VEC; ++e) acc += ex2_approx(x2[e] - nm);
              ls = acc;
              lm = nm;
            }
          }
          uint32_t take = 0;
#pragma unroll
          for (int e = 0; e < TK_VEC; ++e) {
            if (!(xf[e] <= tv) && i0 + e < V) {
              const uint32_t key = bf16_key(w[e >> 1] >> (16 * (e & 1)));
              if (int(key) > thresh) take |= 1u << e;
            }
          }
          if (__any_sync(0xffffffffu, take != 0)) {
#pragma unroll
            for (int e = 0; e < TK_VEC; ++e) {
              const uint32_t key = bf16_key(w[e >> 1] >> (16 * (e & 1)));
              const unsigned long long c =
                  (static_cast<unsigned long long>(key) << 32) | uint32_t(~uint32_t(i0 + e));
              warp_append(sm, (take >> e) & 1u, c);
            }
          }
          if ((seg % TK_CHECK) == TK_CHECK - 1 || seg == nseg - 1) {
            __syncthreads();
            const uint32_t cnt = sm.count;
            __syncthreads();  // every thread has read the count before anyone appends again
            if (cnt > uint32_t(TK_CAP - TK_CHECK * TK_SEG)) {
              thresh = compact(sm, uint32_t(K));
              // float form of the new threshold key (its bf16 value)
              const uint32_t tb = (uint32_t(thresh) & 0x8000u) ? (uint32_t(thresh) & 0x7FFFu)
                                                               : (~uint32_t(thresh) & 0xFFFFu);
              tv = __uint_as_float(tb << 16);
            }
          }
        }
      }
    }

    if (lse_out != nullptr) {
      // merge the threads' (max, sum) pairs: warp shuffles, then warp 0 over the warps
      for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, lm, o);
        const float os = __shfl_xor_sync(0xffffffffu, ls, o);
        const float nm = fmaxf(lm, om);
        if (nm != -INFINITY) {
          ls = ls * ex2_approx(lm - nm) + os * ex2_approx(om - nm);
          lm = nm;
        }
      }
      if ((threadIdx.x & 31) == 0) {
        sm.red_m[threadIdx.x >> 5] = lm;
        sm.red_s[threadIdx.x >> 5] = ls;
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        float M = -INFINITY, S = 0.f;
        for (int i = 0; i < TK_THREADS / 32; ++i) {
          const float nm = fmaxf(M, sm.red_m[i]);
          if (nm != -INFINITY) {
            S = S * exp2f(M - nm) + sm.red_s[i] * exp2f(sm.red_m[i] - nm);
            M = nm;
          }
        }
        lse_out[row] = (M + log2f(S)) * 0.69314718055994531f;
      }
    }

    // Final: keep the candidates that can be in the top K, order them, emit K.
    __syncthreads();
    uint32_t count = sm.count;
    __syncthreads();
    if (count > uint32_t(K)) {
      uint32_t count_ge = 0;
      const uint32_t T = kth_largest_key(sm, count, uint32_t(K), count_ge);
      if (count_ge < count) filter_ge(sm, count, T);
      count = sm.count;
    }
    sort_desc(sm, count);
    for (int j = threadIdx.x; j < K; j += TK_THREADS) {
      const uint32_t col = ~uint32_t(sm.buf[j]);
      ids_out[row * K + j] = int32_t(col);
      if (KD_DCHECK(int64_t(col) < V, sm.err, 0x7002)) vals_out[row * K + j] = __uint_as_float(uint32_t(xr[col]) << 16);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Warp-per-row path for K <= TW_MAXK (the pages' top-100 cache).  The same selection,
// run by one warp per row so that no block barrier is ever taken:
//  * the copy engine streams the row: each warp owns a ring of RING slots of GRP warp
//    steps (a step is 256 elements, 16 bytes per lane); lane 0 fills a slot with one bulk
//    copy completing on the slot's mbarrier, RING groups ahead of its use, running on
//    into the warp's next row while the current one is finished; every lane fences its
//    reads of a slot before the warp barrier after which the slot is refilled;
//  * a first threshold (key >= it) before any element is kept, the first of these that
//    applies: the K-th largest of per-tile row maxima a producer supplies (the teacher
//    projection's epilogue); a guess from the warp's previous row, verified when the row
//    ends (a row short of K entries at or above it is selected again from its start);
//    the K-th largest of the 8-element vector maxima of the row's first RING x GRP steps,
//    which the ring already holds when the row begins (quick start);
//  * each lane tests its 8 values with one packed bf16 max against the threshold, GRP
//    steps at a time with one vote; a vector that passes is queued whole in shared
//    memory, and the warp filters BATCH queued vectors at a time (one per lane) with
//    exact comparisons;
//  * the warp keeps the row's best K so far as a sorted list and merges each drained
//    batch into it (a bitonic sort across the lanes and a rank merge); once it holds K
//    entries its last key is the threshold, exact after every drain: one warp sees the
//    whole row, so the threshold is as tight as the prefix allows, and the list is the
//    answer when the row ends.
// Elements past V read as -inf and are dropped by their column.

constexpr int TW_MAXK = 256;
constexpr int TW_STEP = 32 * TK_VEC;         // elements per warp step
constexpr int TW_GROUP = 4;                  // steps tested together (one vote)
constexpr int TW_QUEUE = 64;                 // queued vectors per warp (ring)
constexpr float TW_LOG2E = 1.4426950408889634f;
// Margin of a guessed threshold below the previous row's K-th value, in units of that
// row's spacing between its (K/2)-th and K-th values (about rank 2.8 K for normal rows).
constexpr float TW_GUESS_MARGIN = 1.5f;

// A configuration: CAP candidate entries per warp, WARPS rows in flight per block (one
// block per SM), BATCH queued vectors filtered per drain (at most 8 * BATCH new
// entries), MAXK the largest K it serves.  The top list (<= MAXK) and one drain's
// entries fit in the buffer, and its bitonic sort pads to a power of two within it.
template <int CAP_, int WARPS_, int BATCH_, int MAXK_>
struct TwCfg {
  static constexpr int CAP = CAP_;
  static constexpr int WARPS = WARPS_;
  static constexpr int BATCH = BATCH_;
  static constexpr int MAXK = MAXK_;
  static_assert((CAP & (CAP - 1)) == 0, "the bitonic sort pads to a power of two within the buffer");
  static_assert(MAXK + 8 * BATCH <= CAP && MAXK <= TW_MAXK && MAXK % 32 == 0, "a drain fits after the list");
  static_assert(BATCH <= 32 && BATCH + 32 <= TW_QUEUE, "one vector per lane; the queue holds a batch and a step");
};

template <int CAP>
struct TopkWarpSmem {
  unsigned long long buf[CAP];
  uint4 qv[TW_QUEUE];
  uint32_t qcol[TW_QUEUE];
  uint32_t hist[256];
  uint32_t* err;  // the workspace error word (checked builds report bad indices there)
};

__device__ __forceinline__ void warp_find_bin(const uint32_t* h, uint32_t target, uint32_t& bin, uint32_t& need,
                                              uint32_t& above) {
  const uint32_t lane = lane_id();
  uint32_t local[8];
  uint32_t sum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    local[j] = h[255 - (lane * 8 + j)];
    sum += local[j];
  }
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= uint32_t(o)) incl += t;
  }
  const uint32_t excl = incl - sum;
  uint32_t b = 0, nd = 0, ab = 0;
  const bool mine = excl < target && target <= incl;
  if (mine) {
    uint32_t run = excl;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (run < target && target <= run + local[j] && nd == 0) {
        b = 255 - (lane * 8 + j);
        nd = target - run;
        ab = run;
      }
      run += local[j];
    }
  }
  const uint32_t owner = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
  bin = __shfl_sync(0xffffffffu, b, owner);
  need = __shfl_sync(0xffffffffu, nd, owner);
  above = __shfl_sync(0xffffffffu, ab, owner);
}

// Warp: K-th largest key among reg[0, cnt) (cnt >= K) and how many keys reach it.
__device__ uint32_t warp_kth_largest(const unsigned long long* reg, uint32_t cnt, uint32_t K, uint32_t* h,
                                     uint32_t& count_ge) {
  const uint32_t lane = lane_id();
  for (uint32_t i = lane; i < 256; i += 32) h[i] = 0;
  __syncwarp();
  for (uint32_t base = 0; base < cnt; base += 32) {
    const uint32_t i = base + lane;
    hist_add_warp(h, i < cnt, i < cnt ? comp_key(reg[i]) >> 8 : 0u);
  }
  __syncwarp();
  uint32_t b1, need, above1;
  warp_find_bin(h, K, b1, need, above1);
  __syncwarp();
  for (uint32_t i = lane; i < 256; i += 32) h[i] = 0;
  __syncwarp();
  for (uint32_t base = 0; base < cnt; base += 32) {
    const uint32_t i = base + lane;
    const uint32_t k = i < cnt ? comp_key(reg[i]) : 0u;
    hist_add_warp(h, i < cnt && (k >> 8) == b1, k & 255u);
  }
  __syncwarp();
  uint32_t b2, need2, above2;
  warp_find_bin(h, need, b2, need2, above2);
  count_ge = above1 + above2 + h[b2];
  __syncwarp();
  return (b1 << 8) | b2;
}

// Warp: K-th largest key among the bf16 values src[0, cnt) in global memory (cnt >= K).
__device__ uint32_t warp_kth_largest_bf16(const uint16_t* src, uint32_t cnt, uint32_t K, uint32_t* h) {
  const uint32_t lane = lane_id();
  for (uint32_t i = lane; i < 256; i += 32) h[i] = 0;
  __syncwarp();
  for (uint32_t base = 0; base < cnt; base += 32) {
    const uint32_t i = base + lane;
    hist_add_warp(h, i < cnt, i < cnt ? bf16_key(__ldg(src + i)) >> 8 : 0u);
  }
  __syncwarp();
  uint32_t b1, need, above1;
  warp_find_bin(h, K, b1, need, above1);
  __syncwarp();
  for (uint32_t i = lane; i < 256; i += 32) h[i] = 0;
  __syncwarp();
  for (uint32_t base = 0; base < cnt; base += 32) {
    const uint32_t i = base + lane;
    const uint32_t k = i < cnt ? bf16_key(__ldg(src + i)) : 0u;
    hist_add_warp(h, i < cnt && (k >> 8) == b1, k & 255u);
  }
  __syncwarp();
  uint32_t b2, need2, above2;
  warp_find_bin(h, need, b2, need2, above2);
  __syncwarp();
  return (b1 << 8) | b2;
}

// Warp: keep the entries of reg[0, cnt) with key >= T, in place (each round of 256 is
// read before any survivor of it is written); returns the new count.
__device__ uint32_t warp_filter_ge(unsigned long long* reg, uint32_t cnt, uint32_t T) {
  const uint32_t lane = lane_id();
  uint32_t out = 0;
  for (uint32_t base = 0; base < cnt; base += 256) {
    unsigned long long held[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t i = base + lane + 32u * j;
      held[j] = i < cnt ? reg[i] : 0ull;
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t i = base + lane + 32u * j;
      const bool take = i < cnt && comp_key(held[j]) >= T;
      const uint32_t bal = __ballot_sync(0xffffffffu, take);
      if (take) reg[out + __popc(bal & ((1u << lane) - 1u))] = held[j];
      out += __popc(bal);
    }
    __syncwarp();
  }
  return out;
}

// Warp: sort reg[0, cnt) descending (bitonic, padded with 0 up to a power of two).
__device__ void warp_sort_desc(unsigned long long* reg, uint32_t cnt) {
  const uint32_t lane = lane_id();
  uint32_t P = 32;
  while (P < cnt) P <<= 1;
  for (uint32_t i = cnt + lane; i < P; i += 32) reg[i] = 0ull;
  __syncwarp();
  for (uint32_t k = 2; k <= P; k <<= 1) {
    for (uint32_t j = k >> 1; j > 0; j >>= 1) {
      for (uint32_t i = lane; i < P; i += 32) {
        const uint32_t ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = reg[i], b = reg[ixj];
          if (((i & k) == 0) ? (a < b) : (a > b)) {
            reg[i] = b;
            reg[ixj] = a;
          }
        }
      }
      __syncwarp();
    }
  }
}

// 16 bytes of warp step `st` for this lane, read directly; elements past V read as -inf.
// Out of line: only the lanes at the ragged end of a row come here.
__device__ __noinline__ uint4 load_step(const uint16_t* xr, int64_t V, int st) {
  const int64_t i0 = int64_t(st) * TW_STEP + int64_t(lane_id()) * TK_VEC;
  if (i0 + TK_VEC <= V) return __ldcs(reinterpret_cast<const uint4*>(xr + i0));
  uint32_t w[4] = {0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u};
#pragma unroll
  for (int e = 0; e < TK_VEC; ++e)
    if (i0 + e < V) {
      const int sh = 16 * (e & 1);
      w[e >> 1] = (w[e >> 1] & ~(0xFFFFu << sh)) | (uint32_t(xr[i0 + e]) << sh);
    }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Largest of the 8 bf16 in v, widened to float (NaN if one of them is NaN).
__device__ __forceinline__ float vec_max(const uint4& v) {
  uint32_t m = bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w));
  m = bmax2(m, __byte_perm(m, 0u, 0x1032));
  return __uint_as_float(m & 0xFFFF0000u);
}

__device__ __forceinline__ float key_to_float(uint32_t key) {
  const uint32_t b = (key & 0x8000u) ? (key & 0x7FFFu) : (~key & 0xFFFFu);
  return __uint_as_float(b << 16);
}

// Key of the largest bf16 value <= x (x finite): x rounded toward -infinity.
__device__ __forceinline__ uint32_t key_floor(float x) {
  const uint32_t f = __float_as_uint(x);
  uint32_t b = f >> 16;
  if ((f & 0x80000000u) && (f & 0xFFFFu)) ++b;  // negative: round the magnitude up
  return bf16_key(b);
}

// Per-warp selection state (warp-uniform).
struct WarpSel {
  uint32_t cnt;   // entries in buf
  uint32_t qh;    // queue head (ring index of the oldest queued vector)
  uint32_t nq;    // queued vectors
  uint32_t wth;   // threshold key
  bool ge;        // until the list holds K entries: key >= wth is a candidate (wth = 0: every element)
  float tv;       // pre-test bound: a vector can hold a candidate only if its maximum is > tv
};

// Warp: merge the T (<= 32) candidates buf[nt, nt + T) into the top list buf[0, nt)
// (composites, sorted descending, nt <= K <= 32 * SLOTS), keeping the K best, in place.
// The candidates come from later columns than every list entry and lie in column order,
// so ranks need only 32-bit keys: a list entry outranks a candidate of equal key, and of
// two equal candidates the earlier one wins.  The candidates are sorted across the lanes
// by (key, -index) as one 32-bit word (bitonic, empty lanes last); every element's new
// place is its index plus the number of elements of the other list above it (binary
// searches over 32-bit keys); nothing is written until everything is read.  `keys`
// (>= 32 words) holds the sorted candidate keys.  Returns min(nt + T, K).
template <int SLOTS>
__device__ uint32_t warp_merge_top(unsigned long long* buf, uint32_t* keys, uint32_t nt, uint32_t T, uint32_t K) {
  const uint32_t lane = lane_id();
  const uint32_t* key_hi = reinterpret_cast<const uint32_t*>(buf) + 1;  // high word of buf[i] at [2 i]
  uint32_t s = lane < T ? (key_hi[2 * (nt + lane)] << 16) | (0xFFFFu - lane) : 0u;
#pragma unroll
  for (uint32_t k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (uint32_t j = k >> 1; j > 0; j >>= 1) {
      const uint32_t o = __shfl_xor_sync(0xffffffffu, s, j);
      const bool desc = (lane & k) == 0;
      const bool low = (lane & j) == 0;
      s = (low == desc) ? max(s, o) : min(s, o);
    }
  }
  // sorted candidate `lane`: its key, its composite, its place
  const uint32_t ck = s >> 16;
  const unsigned long long c = lane < T ? buf[nt + (0xFFFFu - (s & 0xFFFFu))] : 0ull;
  uint32_t lo = 0, hi = nt;  // list entries with key >= ck
  while (lo < hi) {
    const uint32_t mid = (lo + hi) >> 1;
    if (key_hi[2 * mid] >= ck) lo = mid + 1; else hi = mid;
  }
  const uint32_t cpos = lane + lo;
  keys[lane] = ck;
  __syncwarp();
  unsigned long long tv[SLOTS];
  uint32_t tpos[SLOTS];
#pragma unroll
  for (int m = 0; m < SLOTS; ++m) {
    const uint32_t j = lane + 32u * m;
    tv[m] = 0ull;
    tpos[m] = K;
    if (j < nt) {
      tv[m] = buf[j];
      const uint32_t tk = uint32_t(tv[m] >> 32);
      uint32_t a = 0, b = T;  // candidates with a key above tk
      while (a < b) {
        const uint32_t mid = (a + b) >> 1;
        if (keys[mid] > tk) a = mid + 1; else b = mid;
      }
      tpos[m] = j + a;
    }
  }
  __syncwarp();
  if (lane < T && cpos < K) buf[cpos] = c;
#pragma unroll
  for (int m = 0; m < SLOTS; ++m)
    if (tpos[m] < K) buf[tpos[m]] = tv[m];
  __syncwarp();
  return nt + T < K ? nt + T : K;
}

// Warp: filter the nb (<= BATCH) oldest queued vectors, one per lane, and merge what
// passes into the top list.  For values other than NaN, key(x) > wth exactly when
// x > value(wth) (-0 and +0 have one key), and the same for >=, so the test is a float
// compare; a vector holding a NaN, or a threshold key that is a NaN pattern, takes the
// key path.  Once the list holds K entries its last key is the threshold (later
// elements need a larger key: an equal key comes with a larger column).  Out of line:
// it runs once per BATCH queued vectors, and one copy of it keeps the streaming loop
// small in the instruction cache.
template <class C>
__device__ __noinline__ WarpSel warp_drain(TopkWarpSmem<C::CAP>& ws, WarpSel st, uint32_t nb, uint32_t V32,
                                           uint32_t K) {
  const uint32_t lane = lane_id();
  uint32_t take = 0, col0 = 0;
  unsigned long long lo = 0, hi = 0;
  if (lane < nb) {
    const uint32_t q = (st.qh + lane) & (TW_QUEUE - 1);
    const uint4 v = ws.qv[q];
    col0 = ws.qcol[q];
    lo = (static_cast<unsigned long long>(v.y) << 32) | v.x;
    hi = (static_cast<unsigned long long>(v.w) << 32) | v.z;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const float t = key_to_float(st.wth);
    if (st.ge && st.wth == 0) {
      take = 0xFFu;  // every element
    } else if (vec_max(v) == vec_max(v) && t == t) {
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float a = __uint_as_float(w[h] << 16), b = __uint_as_float(w[h] & 0xFFFF0000u);
        if (st.ge ? a >= t : a > t) take |= 1u << (2 * h);
        if (st.ge ? b >= t : b > t) take |= 2u << (2 * h);
      }
    } else {
#pragma unroll
      for (int e = 0; e < TK_VEC; ++e) {
        const uint32_t key = bf16_key(w[e >> 1] >> (16 * (e & 1)));
        if (st.ge ? key >= st.wth : key > st.wth) take |= 1u << e;
      }
    }
    if (col0 + TK_VEC > V32) take &= (V32 > col0 ? (1u << (V32 - col0)) - 1u : 0u);
  }
  // exclusive prefix of the per-lane counts (<= 8: four bits) and the warp total
  const uint32_t c = __popc(take);
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t pre = 0, tot = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t bb = __ballot_sync(0xffffffffu, (c >> b) & 1u);
    pre += uint32_t(__popc(bb & lt)) << b;
    tot += uint32_t(__popc(bb)) << b;
  }
  uint32_t pos = st.cnt + pre;  // after the top list
  while (take) {
    const uint32_t e = __ffs(take) - 1;
    take &= take - 1;
    const uint32_t bits = uint32_t(((e & 4) ? hi : lo) >> (16 * (e & 3))) & 0xFFFFu;
    if (KD_DCHECK(pos < uint32_t(C::CAP), ws.err, 0x7101))
      ws.buf[pos] = (static_cast<unsigned long long>(bf16_key(bits)) << 32) | uint32_t(~(col0 + e));
    ++pos;
  }
  st.qh = (st.qh + nb) & (TW_QUEUE - 1);
  st.nq -= nb;
  __syncwarp();
  if (tot == 0) return st;
  if (!KD_DCHECK(st.cnt + tot <= uint32_t(C::CAP), ws.err, 0x7102)) return st;
  if (tot <= 32) {
    st.cnt = warp_merge_top<C::MAXK / 32>(ws.buf, ws.hist, st.cnt, tot, K);
  } else {  // a large batch: select and sort the whole list
    uint32_t cnt = st.cnt + tot;
    if (cnt > K) {
      uint32_t cge = 0;
      const uint32_t T = warp_kth_largest(ws.buf, cnt, K, ws.hist, cge);
      if (cge < cnt) cnt = warp_filter_ge(ws.buf, cnt, T);
    }
    warp_sort_desc(ws.buf, cnt);
    st.cnt = cnt < K ? cnt : K;
  }
  if (st.cnt >= K) {
    st.wth = comp_key(ws.buf[K - 1]);
    st.ge = false;
    st.tv = key_to_float(st.wth);
  }
  return st;
}

// Warp: the top list (sorted; K entries whenever V >= K) to the row's outputs; values
// are read back from the row (exact bits, -0 kept).
__device__ __noinline__ void warp_finish(const unsigned long long* top, uint32_t cnt, uint32_t K, const uint16_t* xr,
                                         uint32_t V32, uint32_t* err, int32_t* ids_row, float* vals_row) {
  (void)V32;
  (void)err;
  for (uint32_t j = lane_id(); j < K; j += 32) {
    if (j < cnt) {
      const uint32_t col = ~uint32_t(top[j]);
      ids_row[j] = int32_t(col);
      if (KD_DCHECK(col < V32, err, 0x7301)) vals_row[j] = __uint_as_float(uint32_t(xr[col]) << 16);
    } else {
      ids_row[j] = -1;
      vals_row[j] = -INFINITY;
    }
  }
}

// Sum over the 8 values x of v of 2^(x log2 e - b), b = lm log2 e: each word's pair of
// values goes through one packed f32x2 multiply-add and one packed add.
__device__ __forceinline__ float lse_terms(const uint4& v, float b) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  unsigned long long l2e2, nb2, acc;
  asm("mov.b64 %0, {%1, %1};" : "=l"(l2e2) : "r"(__float_as_uint(TW_LOG2E)));
  asm("mov.b64 %0, {%1, %1};" : "=l"(nb2) : "r"(__float_as_uint(-b)));
  asm("mov.b64 %0, {%1, %1};" : "=l"(acc) : "r"(0u));
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    unsigned long long x, t, e;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "r"(w[h] << 16), "r"(w[h] & 0xFFFF0000u));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(t) : "l"(x), "l"(l2e2), "l"(nb2));
    uint32_t t0, t1;
    asm("mov.b64 {%0, %1}, %2;" : "=r"(t0), "=r"(t1) : "l"(t));
    asm("mov.b64 %0, {%1, %2};"
        : "=l"(e)
        : "r"(__float_as_uint(ex2_approx(__uint_as_float(t0)))), "r"(__float_as_uint(ex2_approx(__uint_as_float(t1)))));
    asm("add.rn.f32x2 %0, %0, %1;" : "+l"(acc) : "l"(e));
  }
  uint32_t a0, a1;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(a0), "=r"(a1) : "l"(acc));
  return __uint_as_float(a0) + __uint_as_float(a1);
}

// One group of TW_GROUP steps of a lane, vectors v[0 ..]: the packed pre-test of each
// against the warp's threshold (st.tv is NaN while every element is a candidate), one
// vote for the group, and, when a vector passed, its queueing and a drain every BATCH
// queued.  s0 = the group's first step; `live` = the group's steps that exist.
template <class C, bool WITH_LSE>
__device__ __forceinline__ void test_group(TopkWarpSmem<C::CAP>& ws, WarpSel& st, const uint4* v, int s0,
                                           uint32_t live, float& lm, float& ls, uint32_t V32, uint32_t K) {
  const uint32_t lane = lane_id();
  float vm[TW_GROUP];
  uint32_t pass = 0;
#pragma unroll
  for (int k = 0; k < TW_GROUP; ++k) {
    vm[k] = vec_max(v[k]);
    if (((live >> k) & 1u) && !(vm[k] <= st.tv)) pass |= 1u << k;
  }
  if (WITH_LSE) {
    float gm = -INFINITY;
#pragma unroll
    for (int k = 0; k < TW_GROUP; ++k)
      if ((live >> k) & 1u) gm = fmaxf(gm, vm[k]);
    if (gm > lm) {
      ls *= ex2_approx((lm - gm) * TW_LOG2E);
      lm = gm;
    }
    if (lm != -INFINITY) {
      const float b = lm * TW_LOG2E;
#pragma unroll
      for (int k = 0; k < TW_GROUP; ++k)
        if ((live >> k) & 1u) ls += lse_terms(v[k], b);
    }
  }
  if (__any_sync(0xffffffffu, pass != 0)) {
#pragma unroll
    for (int k = 0; k < TW_GROUP; ++k) {
      const bool p = (pass >> k) & 1u;
      const uint32_t bal = __ballot_sync(0xffffffffu, p);
      if (bal != 0) {
        if (p) {
          const uint32_t q = (st.qh + st.nq + __popc(bal & ((1u << lane) - 1u))) & (TW_QUEUE - 1);
          ws.qv[q] = v[k];
          ws.qcol[q] = uint32_t(s0 + k) * TW_STEP + lane * TK_VEC;
        }
        st.nq += __popc(bal);  // < BATCH + 32 <= TW_QUEUE
        if (st.nq >= uint32_t(C::BATCH)) {
          __syncwarp();
          do {
            st = warp_drain<C>(ws, st, C::BATCH, V32, K);
          } while (st.nq >= uint32_t(C::BATCH));
        }
      }
    }
  }
}

// Ring feeding: (RING - 1) x GRP x 512 bytes per warp stay in flight whatever the
// register schedule.  A row's last group copies whole 16-byte vectors only; the one lane
// whose vector straddles the end of the row (and the lanes past it) read theirs directly.

template <int CAP_, int WARPS_, int BATCH_, int MAXK_, int RING_, int GRP_>
struct TmaCfg : TwCfg<CAP_, WARPS_, BATCH_, MAXK_> {
  static constexpr int RING = RING_;
  static constexpr int GRP = GRP_;
  static_assert(GRP == TW_GROUP, "a slot is one tested group");
  static_assert((RING & (RING - 1)) == 0, "slots wrap with a mask");
};
using TmSmallK = TmaCfg<512, 15, 24, 128, 4, 4>;   // K <= 128
using TmLargeK = TmaCfg<1024, 12, 32, 256, 4, 4>;  // K <= 256

template <class C>
struct TopkTmaSmem {
  uint4 ring[C::RING][C::GRP][32];
  TopkWarpSmem<C::CAP> sel;
  uint64_t full[C::RING];
  uint32_t abort;  // set by a timed-out wait
  uint32_t never;  // stays 0: the flag of the bounded waits after an abort
};

// Bulk copy global -> shared of `bytes` (a multiple of 16), completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Orders this thread's shared-memory accesses so far before the async-proxy operations
// (bulk copies) that follow it, in this thread or, after a barrier, in another.
__device__ __forceinline__ void fence_proxy_async_cta() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The lane's vectors of warp steps s0 .. s0 + TW_GROUP - 1 of a row, read directly
// (past the row: -inf, nothing read).
__device__ __forceinline__ void load_group(uint4* v, const uint16_t* xr, int64_t V, int s0) {
#pragma unroll
  for (int k = 0; k < TW_GROUP; ++k) {
    const int64_t i0 = int64_t(s0 + k) * TW_STEP + int64_t(lane_id()) * TK_VEC;
    v[k] = i0 + TK_VEC <= V ? __ldcs(reinterpret_cast<const uint4*>(xr + i0)) : load_step(xr, V, s0 + k);
  }
}

// Warp: the whole selection of one row again, read directly from global memory (the next
// group's loads in flight while a group is tested), every element a candidate until the
// list holds K.  Out of line: it runs only after a guessed threshold turned out too high.
template <class C>
__device__ __noinline__ WarpSel warp_reselect(TopkWarpSmem<C::CAP>& ws, const uint16_t* xr, int64_t V, int nst,
                                              uint32_t V32, uint32_t K) {
  WarpSel st;
  st.cnt = 0;
  st.qh = 0;
  st.nq = 0;
  st.wth = 0;
  st.ge = true;
  st.tv = key_to_float(0);
  float lm = -INFINITY, ls = 0.f;  // unused: no logsumexp here
  uint4 a[TW_GROUP], b[TW_GROUP];
  load_group(a, xr, V, 0);
  for (int s0 = 0; s0 < nst; s0 += TW_GROUP) {
    if (s0 + TW_GROUP < nst) load_group(b, xr, V, s0 + TW_GROUP);
    const uint32_t live = nst - s0 >= TW_GROUP ? (1u << TW_GROUP) - 1u : (1u << (nst - s0)) - 1u;
    test_group<C, false>(ws, st, a, s0, live, lm, ls, V32, K);
#pragma unroll
    for (int k = 0; k < TW_GROUP; ++k) a[k] = b[k];
  }
  __syncwarp();
  while (st.nq > 0) st = warp_drain<C>(ws, st, min(st.nq, uint32_t(C::BATCH)), V32, K);
  return st;
}

template <class C, bool WITH_LSE>
__global__ void __launch_bounds__(C::WARPS * 32, 1)
    kd_topk_tma_kernel(const uint16_t* __restrict__ X, int64_t N, int64_t V, int64_t ld, int K,
                       int32_t* __restrict__ ids_out, float* __restrict__ vals_out, float* __restrict__ lse_out,
                       uint32_t* err, int guesses, const uint32_t* guess_in, uint32_t* guess_out,
                       const uint16_t* __restrict__ tile_max, int64_t ld_tile_max, int ntiles) {
  extern __shared__ __align__(16) uint8_t tkt_smem_raw[];
  constexpr int GSTEPS = C::GRP;
  constexpr uint32_t GBYTES = uint32_t(C::GRP) * TW_STEP * 2;
  const uint32_t lane = lane_id();
  TopkTmaSmem<C>& ts = reinterpret_cast<TopkTmaSmem<C>*>(tkt_smem_raw)[threadIdx.x >> 5];
  TopkWarpSmem<C::CAP>& ws = ts.sel;
  const int64_t nwarps = int64_t(gridDim.x) * C::WARPS;
  const int nst = int((V + TW_STEP - 1) / TW_STEP);
  const int ngr = (nst + GSTEPS - 1) / GSTEPS;  // groups per row
  const uint32_t V32 = uint32_t(V), Ku = uint32_t(K);
  // this lane's vector in a row's last step is not a whole 16 bytes inside the row
  const bool tail_lane = int64_t(nst - 1) * TW_STEP + int64_t(lane) * TK_VEC + TK_VEC > V;

  if (lane == 0) {
    for (int r = 0; r < C::RING; ++r) mbar_init(&ts.full[r], 1);
    ts.abort = 0;
    ts.never = 0;
    ws.err = err;
    fence_mbar_init();
  }
  __syncwarp();

  int64_t row = int64_t(blockIdx.x) * C::WARPS + (threadIdx.x >> 5);
  // Producer: the warp's rows one after another, group by group.
  int64_t prow = row;
  int pg = 0;
  uint32_t issued = 0;
  auto issue = [&](uint32_t slot) {
    if (prow < N) {
      if (lane == 0) {
        const int64_t e0 = int64_t(pg) * GSTEPS * TW_STEP;
        const int64_t left = V - e0;
        uint32_t bytes = left >= int64_t(GSTEPS) * TW_STEP ? GBYTES : uint32_t(left * 2) & ~15u;
        if (!KD_DCHECK(e0 >= 0 && e0 + bytes / 2 <= V && bytes <= GBYTES, err, 0x7401)) bytes = 0;
        mbar_arrive_expect_tx(&ts.full[slot], bytes);  // 0 bytes: the phase completes on the arrival
        if (bytes != 0) bulk_g2s(&ts.ring[slot][0][0], X + prow * ld + e0, bytes, &ts.full[slot]);
      }
      ++issued;
      if (++pg == ngr) {
        pg = 0;
        prow += nwarps;
      }
    }
  };
  for (int r = 0; r < C::RING; ++r) issue(uint32_t(r));

  uint32_t gidx = 0;  // groups consumed
  bool ok = true;
  // Guessed threshold for the warp's next row (0: none) and the margin factor behind it.
  const int64_t gw = int64_t(blockIdx.x) * C::WARPS + (threadIdx.x >> 5);  // this warp's guess word
  const bool may_guess = guesses != 0 && K >= 16;
  uint32_t guess = (may_guess && guess_in && gw < KD_TOPK_MAX_WARPS) ? guess_in[gw] : 0u;
  float margin = TW_GUESS_MARGIN;
  for (; row < N; row += nwarps) {
    const uint16_t* xr = X + row * ld;
    WarpSel st;
    st.cnt = 0;
    st.qh = 0;
    st.nq = 0;
    st.wth = 0;
    st.ge = true;
    st.tv = key_to_float(0);
    float lm = -INFINITY, ls = 0.f;

    // Tile start (maxima of ntiles >= K disjoint column ranges of every row given, as the
    // teacher projection emits them): their K-th largest is reached by at least K elements,
    // so every element of the top K has a key >= it, an exact first threshold.
    // Guessed start (when enabled: every row after a warp's first, K >= 16): the threshold
    // is a key taken from the previous row's best K (below).  If at least K elements reach it, the top K
    // all do and the row is selected exactly; if not, the list ends short of K and the row
    // is selected again from its start with no threshold.
    // Quick start (otherwise): the ring holds this row's first RING groups (none of them the
    // row's last).  The K-th largest of their per-lane vector maxima is reached by at least
    // K elements, so every element of the top K has a key >= it: those groups are then
    // consumed with that threshold (>=), and the rest of the row with the raised ones.
    const bool tiles = tile_max != nullptr && ntiles >= K;
    const bool guessed = !tiles && guess != 0u;
    if (tiles) {
      const uint32_t T = warp_kth_largest_bf16(tile_max + row * ld_tile_max, uint32_t(ntiles), Ku, ws.hist);
      if (T != 0) {
        st.wth = T;
        st.tv = key_to_float(T - 1u == 0x7FFFu ? 0x7FFEu : T - 1u);
      }
    } else if (guessed) {
      st.wth = guess;
      st.tv = key_to_float(guess - 1u == 0x7FFFu ? 0x7FFEu : guess - 1u);
    } else if (ngr > C::RING && K <= C::RING * C::GRP * 32) {
      for (int r = 0; r < C::RING && ok; ++r) {
        const uint32_t u = gidx + uint32_t(r);
        ok = mbar_wait(&ts.full[u & (C::RING - 1)], (u / C::RING) & 1u, &ts.abort, err, 0x72u);
      }
      if (!ok) break;
#pragma unroll
      for (int r = 0; r < C::RING; ++r) {
#pragma unroll
        for (int k = 0; k < C::GRP; ++k) {
          const uint4 v = ts.ring[(gidx + r) & (C::RING - 1)][k][lane];
          const float m = vec_max(v);
          uint32_t key;
          if (m == m) {
            key = bf16_key(__float_as_uint(m) >> 16);
          } else {  // a NaN hides the maximum: take the exact keys
            key = 0;
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) key = max(key, max(bf16_key(w[h]), bf16_key(w[h] >> 16)));
          }
          ws.buf[(r * C::GRP + k) * 32 + lane] = static_cast<unsigned long long>(key) << 32;
        }
      }
      __syncwarp();
      uint32_t cge = 0;
      const uint32_t T0 = warp_kth_largest(ws.buf, uint32_t(C::RING * C::GRP * 32), Ku, ws.hist, cge);
      if (T0 != 0) {
        st.wth = T0;
        // pre-test bound just below value(T0) (the -0/+0 key is 0x8000: step past -0)
        st.tv = key_to_float(T0 - 1u == 0x7FFFu ? 0x7FFEu : T0 - 1u);
      }
    }

    for (int g = 0; g < ngr; ++g, ++gidx) {
      const uint32_t slot = gidx & (C::RING - 1);
      if (!mbar_wait(&ts.full[slot], (gidx / C::RING) & 1u, &ts.abort, err, 0x70u)) {
        ok = false;
        break;
      }
      uint4 v[GSTEPS];
#pragma unroll
      for (int k = 0; k < GSTEPS; ++k) v[k] = ts.ring[slot][k][lane];
      const int s0 = g * GSTEPS;
      uint32_t live = (1u << GSTEPS) - 1u;
      if (g == ngr - 1) {  // the row's last group
        live = nst - s0 >= GSTEPS ? live : (1u << (nst - s0)) - 1u;
        if (tail_lane) {
#pragma unroll
          for (int k = 0; k < GSTEPS; ++k)
            if (s0 + k == nst - 1) v[k] = load_step(xr, V, nst - 1);
        }
      }
      // The slot is refilled by the async proxy: every lane's reads of it are ordered before
      // the refill (a proxy fence in each lane, then the warp barrier before lane 0 issues).
      fence_proxy_async_cta();
      __syncwarp();
      issue(slot);
      test_group<C, WITH_LSE>(ws, st, v, s0, live, lm, ls, V32, Ku);
    }
    if (!ok) break;
    __syncwarp();
    while (st.nq > 0) st = warp_drain<C>(ws, st, min(st.nq, uint32_t(C::BATCH)), V32, Ku);
    if (guessed && st.cnt < Ku) {
      // fewer than K elements reach the guess (the logsumexp of the pass is complete)
      st = warp_reselect<C>(ws, xr, V, nst, V32, Ku);
      margin *= 4.f;  // a wider margin for the rows after a miss
    }
    if (may_guess) {
      // Next guess: the K-th best value lowered by margin x (its distance to the (K/2)-th).
      // For tails like the normal's or the logistic's the top order statistics are spaced
      // about logarithmically in rank, so margin m lands near rank 2^m K of a row like this.
      const float vk = key_to_float(comp_key(ws.buf[K - 1]));
      const float vh = key_to_float(comp_key(ws.buf[K / 2 - 1]));
      const float g = vk - margin * (vh - vk);
      guess = (g > -INFINITY && g < INFINITY) ? key_floor(g) : 0u;  // none after a NaN or an infinity
    }

    if (WITH_LSE) {
      for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, lm, o);
        const float os = __shfl_xor_sync(0xffffffffu, ls, o);
        const float nm = fmaxf(lm, om);
        if (nm != -INFINITY) {
          ls = ls * ex2_approx((lm - nm) * TW_LOG2E) + os * ex2_approx((om - nm) * TW_LOG2E);
          lm = nm;
        }
      }
      if (lane == 0) lse_out[row] = lm + log2f(ls) * 0.69314718055994531f;
    }
    warp_finish(ws.buf, st.cnt, Ku, xr, V32, err, ids_out + row * K, vals_out + row * K);
    __syncwarp();
  }
  if (!ok) {  // a wait timed out: let this warp's copies still in flight land (bounded) before leaving
    for (uint32_t u = gidx; u < issued; ++u)
      mbar_wait(&ts.full[u & (C::RING - 1)], (u / C::RING) & 1u, &ts.never, err, 0x71u, 10000000ull);
  }
  if (guess_out && gw < KD_TOPK_MAX_WARPS && lane == 0) guess_out[gw] = guess;
}

// Guessed starting thresholds are speculative: a row whose guess was too high is read a
// second time by its warp alone, at the end of that warp's work, so a few misses decide
// the launch's duration.  They pay off only when consecutive rows have about the same
// scale (0.52 against 0.65 ms on 8192 rows of N(0, 2) over 151936 columns, K = 100) and
// cost when it varies (0.77 ms with the rows' scales 5 % apart): off unless
// KD_TOPK_GUESS=1 is set in the environment.
static int topk_guesses() {
  static int on = -1;
  if (on < 0) {
    const char* v = getenv("KD_TOPK_GUESS");
    on = (v && v[0] == '1') ? 1 : 0;
  }
  return on;
}

template <class C>
cudaError_t launch_topk_tma(const uint16_t* X, int64_t N, int64_t V, int64_t ld, int K, int32_t* ids, float* vals,
                            float* lse, uint32_t* err, cudaStream_t s, const uint32_t* guess_in, uint32_t* guess_out,
                            const uint16_t* tile_max, int64_t ld_tile_max, int ntiles) {
  static PerDevice<int> attr_plain, attr_lse;
  const int smem = int(C::WARPS * sizeof(TopkTmaSmem<C>));
  cudaError_t e = smem_attr_once(attr_plain, reinterpret_cast<const void*>(kd_topk_tma_kernel<C, false>), smem);
  if (e == cudaSuccess)
    e = smem_attr_once(attr_lse, reinterpret_cast<const void*>(kd_topk_tma_kernel<C, true>), smem);
  if (e != cudaSuccess) return e;
  int grid = gemm_max_grid();  // one block of C::WARPS row-streaming warps per SM
  if (int64_t(grid) * C::WARPS > N) grid = int((N + C::WARPS - 1) / C::WARPS);
  if (grid > KD_TOPK_MAX_WARPS / C::WARPS) guess_in = guess_out = nullptr;  // more warps than guess words
  const int guesses = topk_guesses();
  if (lse)
    kd_topk_tma_kernel<C, true><<<grid, C::WARPS * 32, smem, s>>>(X, N, V, ld, K, ids, vals, lse, err, guesses,
                                                                   guess_in, guess_out, tile_max, ld_tile_max, ntiles);
  else
    kd_topk_tma_kernel<C, false><<<grid, C::WARPS * 32, smem, s>>>(X, N, V, ld, K, ids, vals, lse, err, guesses,
                                                                    guess_in, guess_out, tile_max, ld_tile_max, ntiles);
  return cudaSuccess;
}

cudaError_t launch_topk(const uint16_t* X, int64_t N, int64_t V, int64_t ld, int K, int32_t* ids, float* vals,
                        float* lse, uint32_t* err, cudaStream_t s, const uint32_t* guess_in, uint32_t* guess_out,
                        const uint16_t* tile_max, int64_t ld_tile_max, int ntiles) {
  static PerDevice<int> attr;
  const int smem = int(sizeof(TopkSmem));
  cudaError_t ea = smem_attr_once(attr, reinterpret_cast<const void*>(kd_topk_kernel), smem);
  if (ea != cudaSuccess) return ea;
  int grid = 2 * gemm_max_grid();
  if (int64_t(grid) > N) grid = int(N);
  if (grid <= 0) return cudaSuccess;
  prof_before("kd_topk_cache", s);
  if (K <= TmSmallK::MAXK) {
    cudaError_t e = launch_topk_tma<TmSmallK>(X, N, V, ld, K, ids, vals, lse, err, s, guess_in, guess_out, tile_max,
                                              ld_tile_max, ntiles);
    if (e != cudaSuccess) return e;
  } else if (K <= TmLargeK::MAXK) {
    cudaError_t e = launch_topk_tma<TmLargeK>(X, N, V, ld, K, ids, vals, lse, err, s, guess_in, guess_out, tile_max,
                                              ld_tile_max, ntiles);
    if (e != cudaSuccess) return e;
  } else {
    kd_topk_kernel<<<grid, TK_THREADS, smem, s>>>(X, N, V, ld, K, ids, vals, lse, err);
  }
  prof_after(s);
  return cudaGetLastError();
}

}  // namespace kd
