// Offline top-K teacher cache: the K largest logits of every row of a dense
// bf16 [N, V] teacher-logits matrix, with their token ids ([ART] paragraph on
// the first fix; [DAI] "As duas inovações" item 1; [EPO] "Los dos cambios
// propuestos", first item).
//
// HBM-bound: every logit is read once (twice for a row whose speculative start,
// below, turned out too high).  Every element's rank is a unique composite of the
// order-preserving 16-bit key of its bf16 value and its column, which orders by
// value descending, then column ascending; the top K are the K largest composites,
// so the result is exact with any number of ties.  A threshold key T is valid once
// at least K elements seen so far reach it: later elements then need key > T (an
// equal key comes with a larger column and ranks below those K).  Kernels:
//  * K <= 256 (the pages' top-100): a streaming kernel, one warp per row and no
//    block barrier, that hands each row's best candidates to the workspace, and an
//    emit kernel that sorts them and writes the outputs (the warp-per-row section
//    below);
//  * 256 < K <= 1024: one CTA per row (grid-strided): the row streams through in
//    segments of 4096 elements into a shared candidate buffer; when it passes half
//    full, the K-th largest key in it is found with two byte histograms and only
//    what reaches it is kept; the survivors are sorted once at the end.
//
// Optionally the same pass also takes the full-row logsumexp of the teacher
// logits and the probability mass the cache drops, 1 - sum_k e^(t_k - lse), per
// position ([ART] paragraph on the top-K limitation).
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
  float lse_row;  // the row's logsumexp, for the dropped mass
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
                   float* __restrict__ dropped_out, uint32_t* err) {
  extern __shared__ __align__(16) uint8_t tk_smem_raw[];
  TopkSmem& sm = *reinterpret_cast<TopkSmem*>(tk_smem_raw);
  if (threadIdx.x == 0) sm.err = err;  // read after the first barrier below
  const int nseg = int((V + TK_SEG - 1) / TK_SEG);
  const bool want_lse = lse_out != nullptr || dropped_out != nullptr;

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
      if (want_lse) {
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
          if (want_lse) {
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

    if (want_lse) {
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
        sm.lse_row = (M + log2f(S)) * 0.69314718055994531f;
        if (lse_out) lse_out[row] = sm.lse_row;
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
    float part = 0.f;  // this thread's share of sum_k exp(v_k - lse) (at most two terms)
    for (int j = threadIdx.x; j < K; j += TK_THREADS) {
      const uint32_t col = ~uint32_t(sm.buf[j]);
      ids_out[row * K + j] = int32_t(col);
      if (KD_DCHECK(int64_t(col) < V, sm.err, 0x7002)) {
        const float v = __uint_as_float(uint32_t(xr[col]) << 16);
        vals_out[row * K + j] = v;
        if (dropped_out) part += expf(v - sm.lse_row);
      }
    }
    if (dropped_out) {
      // the teacher probability outside the K kept logits: 1 - sum over the block
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      __syncthreads();
      if ((threadIdx.x & 31) == 0) sm.red_s[threadIdx.x >> 5] = part;
      __syncthreads();
      if (threadIdx.x == 0) {
        float tot = 0.f;
        for (int i = 0; i < TK_THREADS / 32; ++i) tot += sm.red_s[i];
        dropped_out[row] = 1.f - tot;
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Warp-per-row path for K <= TW_MAXK (the pages' top-100 cache): two kernels.
//
// kd_topk_stream_kernel, one warp per row, no block barrier; it reads every logit once:
//  * the copy engine streams the row: each warp owns a ring of RING slots of TW_GROUP warp
//    steps (a step is 256 elements, 16 bytes per lane); lane 0 fills a slot with one bulk
//    copy completing on the slot's mbarrier, RING groups ahead of its use, running on into
//    the warp's next row while the current one is finished; every lane fences its reads
//    of a slot before the warp barrier after which the slot is refilled;
//  * a first threshold before any element is kept: the K-th largest of per-tile row
//    maxima a producer supplies (the teacher projection's epilogue; exact), else from the
//    row's first TW_QS groups (4096 elements), which the ring holds when the row begins:
//    the K-th largest of their 512 vector maxima (T0; at least K elements reach it: exact),
//    raised by a speculative step (below) when that helps;
//  * the pre-test: per step, each lane's 8 values reduced by three packed bf16 maxima
//    and compared with the threshold by one packed unordered compare (a NaN passes);
//  * a vector that passes is queued in the lane's own shared-memory queue (no warp vote
//    per vector); when a lane's queue is nearly full the warp drains every queue: each
//    lane tests the elements of all its queued vectors exactly, one prefix sum over the
//    lanes' counts places the ones that pass in a candidate buffer (one slot at a time,
//    with raises between slots, when they would not fit); the threshold is then raised to
//    the K-th largest key of the buffer, and the buffer is filtered to what reaches it
//    when it runs short of room (not after the row's last drain: the hand-over below
//    finds that key itself);
//  * when the row ends: the K-th largest key T of the buffer, and the candidates that
//    reach it (K of them, or a few more on ties) handed to a per-row slot of the
//    workspace; the warp goes on with its next row.
// kd_topk_emit_kernel, one warp per row: sorts the row's handed-over candidates in
// registers (a bitonic network across the lanes) and writes the first K: ids, values (the
// candidates carry their bf16 bits) and, when asked, the dropped teacher mass.
//
// The K-th largest key of a set of keys is found by bisection between the smallest and the
// largest key present (steps of a per-lane count and a warp sum), in registers.
//
// Speculative start.  Among the 512 vector maxima of the row's first 4096 elements, the
// K-th largest T0 and the (K/4)-th largest T1 locate and scale the row's upper tail; the
// start T0 + c (T1 - T0) is invariant to the row's offset and scale.  A simulation of
// rows of normal, logistic, Gumbel and uniform values (offset and scale varying per row)
// put the row's K-th value above T0 + c (T1 - T0) in 99.5 % of rows or more for c up to
// 1.1 (uniform) and 1.8 (the others); c = TW_SPEC_C puts the start near rank 5 K of a
// normal row.  At least K elements must reach the start for the selection to be exact:
// a row where fewer do (its buffer ends short of K) is selected again from its start with
// T0, and that warp makes no further speculative starts in the launch.  The control
// block's third word counts such rows.

constexpr int TW_MAXK = 256;
constexpr int TW_STEP = 32 * TK_VEC;   // elements per warp step
constexpr int TW_GROUP = 4;            // steps per ring slot, tested together
constexpr int TW_HAND = 256;           // candidates handed over per row, at most
constexpr float TW_LOG2E = 1.4426950408889634f;
constexpr float TW_SPEC_C = 1.3f;      // speculative start: T0 + c (T1 - T0)
constexpr int TW_SPEC_MIN_K = 16;      // smaller K: too few vector maxima above T1 to place it
constexpr int TW_QS = 4;               // groups whose vector maxima place the start: 4096 elements

// A configuration: CAP candidate entries per warp, WARPS rows in flight per block (one block
// per SM), QL queued vectors per lane, MAXK the largest K it serves, RING ring slots.  A
// queue slot adds at most 256 elements, and a filtered buffer over CAP - 256 entries (ties)
// is cut to its best K; both fit, and the bitonic sort pads to a power of two within CAP.
template <int CAP_, int WARPS_, int QL_, int MAXK_, int RING_>
struct TwCfg {
  static constexpr int CAP = CAP_;
  static constexpr int WARPS = WARPS_;
  static constexpr int QL = QL_;
  static constexpr int MAXK = MAXK_;
  static constexpr int RING = RING_;
  static_assert(CAP == 512, "the bisection selects hold the buffer as 16 keys per lane");
  static_assert(CAP >= MAXK + TW_STEP, "a slot's elements fit after a cut list");
  static_assert(MAXK <= TW_MAXK && MAXK <= TW_HAND && MAXK <= RING * TW_GROUP * 32, "limits of K");
  static_assert(QL >= 2 * TW_GROUP, "a group's vectors fit in a lane's queue after the drain check");
  static_assert(RING >= TW_QS, "the ring holds the groups of the quick start");
};
using TmSmallK = TwCfg<512, 11, 12, 128, 4>;   // K <= 128
using TmLargeK = TwCfg<512, 11, 12, 256, 4>;   // K <= 256

template <class C>
struct TwSmem {                             // one warp's part of the block's shared memory
  uint4 ring[C::RING][TW_GROUP][32];        // bulk-copy ring: slot, step, lane
  union {
    uint4 qv[C::QL][32];                    // per-lane queues: slot j of lane l at [j][l]
    uint32_t hist[256];                     // byte histograms (K-th of the tile maxima), used at a
  };                                        // row's start, while the queues are empty
  uint32_t qcol[C::QL][32];                 // first column of each queued vector
  unsigned long long buf[C::CAP];           // candidates (cand_make)
  uint64_t full[C::RING];
  uint32_t abort;                           // set by a timed-out wait
  uint32_t never;                           // stays 0: the flag of the bounded waits after an abort
  uint32_t* err;                            // the workspace error word (checked builds report there)
  uint32_t pad[2];
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

// A candidate of the warp path as one 64-bit word that orders like the element's rank:
// key (16 bits) | ~column (32) | the bf16 bits (16), so the value, -0 and NaN payloads
// included, travels with it.
__device__ __forceinline__ unsigned long long cand_make(uint32_t bits, uint32_t col) {
  return (static_cast<unsigned long long>(bf16_key(bits)) << 48) | (static_cast<unsigned long long>(~col) << 16) |
         (bits & 0xFFFFu);
}
__device__ __forceinline__ uint32_t cand_key(unsigned long long c) { return uint32_t(c >> 48); }
__device__ __forceinline__ uint32_t cand_col(unsigned long long c) { return ~uint32_t(c >> 16); }
__device__ __forceinline__ uint32_t cand_bits(unsigned long long c) { return uint32_t(c) & 0xFFFFu; }

// Warp: for each of R ranks r, the largest key T_r that at least r of the warp's keys reach
// (the r-th largest key), and how many reach it.  Each lane holds E keys, kp[i] = key + 1
// (0: no key).  Bisection on the warp's counts over [smallest key, largest key + 1), the
// keys present: count(>= lo) >= r > count(>= hi) holds from the start, and each step halves
// the bracket until it is one key wide (a handful of steps for keys that lie close, 16 for
// keys spread over the whole 16-bit range); rank must not exceed the number of keys.
// lo_hint: per rank a warp-uniform kp value that at least rank[r] keys reach, a higher start
// for the bracket (0: none).
template <int E, int R>
__device__ __forceinline__ void warp_rank_keys(const uint32_t (&kp)[E], const uint32_t (&rank)[R], uint32_t (&T)[R],
                                               uint32_t (&count_ge)[R], const uint32_t (&lo_hint)[R]) {
  uint32_t n = 0, kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    n += kp[i] != 0u ? 1u : 0u;
    kmin = min(kmin, kp[i] != 0u ? kp[i] : 0xFFFFFFFFu);
    kmax = max(kmax, kp[i]);
  }
  n = __reduce_add_sync(0xffffffffu, n);
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (n == 0u) {  // no keys (not a caller's case): T = 0, nothing reaches it
    kmin = 1u;
    kmax = 1u;
  }
  uint32_t lo[R], hi[R], clo[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    lo[r] = kmin;        // keys + 1 >= lo: all n of them
    hi[r] = kmax + 1u;   // none
    clo[r] = n;
    if (lo_hint[r] > kmin && lo_hint[r] <= kmax) {
      uint32_t c = 0;
#pragma unroll
      for (int i = 0; i < E; ++i) c += kp[i] >= lo_hint[r] ? 1u : 0u;
      lo[r] = lo_hint[r];
      clo[r] = __reduce_add_sync(0xffffffffu, c);
    }
  }
#pragma unroll 1
  for (;;) {
    bool open = false;
#pragma unroll
    for (int r = 0; r < R; ++r) open |= hi[r] - lo[r] > 1u;
    if (!open) break;  // lo and hi come from warp sums: the exit is warp-uniform
    uint32_t mid[R], c[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      mid[r] = (lo[r] + hi[r]) >> 1;
      c[r] = 0;
    }
#pragma unroll
    for (int i = 0; i < E; ++i)
#pragma unroll
      for (int r = 0; r < R; ++r) c[r] += kp[i] >= mid[r] ? 1u : 0u;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      c[r] = __reduce_add_sync(0xffffffffu, c[r]);
      if (hi[r] - lo[r] > 1u) {
        if (c[r] >= rank[r]) {
          lo[r] = mid[r];
          clo[r] = c[r];
        } else {
          hi[r] = mid[r];
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    T[r] = lo[r] - 1u;
    count_ge[r] = clo[r];
  }
}

// Warp: the K-th largest key of the buffer's cnt entries (K <= cnt <= 32 E) and how many
// entries reach it.
template <int E>
__device__ __forceinline__ uint32_t buf_rank_key_e(const unsigned long long* buf, uint32_t cnt, uint32_t K,
                                                   uint32_t& count_ge) {
  const uint32_t lane = lane_id();
  uint32_t kp[E];
  const uint32_t* hw = reinterpret_cast<const uint32_t*>(buf) + 1;  // high word of buf[i] at [2 i]
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const uint32_t j = lane + 32u * i;
    kp[i] = j < cnt ? (hw[2 * j] >> 16) + 1u : 0u;
  }
  const uint32_t rank[1] = {K};
  uint32_t T[1], cge[1];
  const uint32_t none[1] = {0u};
  warp_rank_keys<E, 1>(kp, rank, T, cge, none);
  count_ge = cge[0];
  return T[0];
}

// The same for any cnt up to CAP = 512, holding 8 or 16 keys per lane: (key, count reaching it).
__device__ __noinline__ uint2 buf_rank_key(const unsigned long long* buf, uint32_t cnt, uint32_t K) {
  uint32_t cge = 0;
  const uint32_t T = cnt <= 256u ? buf_rank_key_e<8>(buf, cnt, K, cge) : buf_rank_key_e<16>(buf, cnt, K, cge);
  return make_uint2(T, cge);
}

// Warp: keep the entries of buf[0, cnt) whose key reaches T, in place (each round of 256 is
// read before any survivor of it is written); returns the new count.
__device__ uint32_t buf_filter_ge(unsigned long long* buf, uint32_t cnt, uint32_t T) {
  const uint32_t lane = lane_id();
  uint32_t out = 0;
  for (uint32_t base = 0; base < cnt; base += 256) {
    unsigned long long held[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t i = base + lane + 32u * j;
      held[j] = i < cnt ? buf[i] : 0ull;
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t i = base + lane + 32u * j;
      const bool take = i < cnt && cand_key(held[j]) >= T;
      const uint32_t bal = __ballot_sync(0xffffffffu, take);
      if (take) buf[out + __popc(bal & ((1u << lane) - 1u))] = held[j];
      out += __popc(bal);
    }
    __syncwarp();
  }
  return out;
}

// Largest of the 8 bf16 of v, as a packed pair: each half the maximum of four (NaN if one is NaN).
__device__ __forceinline__ uint32_t vec_max2(const uint4& v) { return bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w)); }

// Some half of the packed bf16 pair m is > (ge: >=) the packed threshold t2, or is NaN.
__device__ __forceinline__ bool half_passes(uint32_t m, uint32_t t2, bool ge) {
  uint32_t r;
  if (ge)
    asm("{\n\t.reg .pred p, q;\n\tsetp.geu.bf16x2 p|q, %1, %2;\n\tor.pred p, p, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(m), "r"(t2));
  else
    asm("{\n\t.reg .pred p, q;\n\tsetp.gtu.bf16x2 p|q, %1, %2;\n\tor.pred p, p, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(m), "r"(t2));
  return r != 0;
}

// bf16 bits of the value whose key is `key`, twice (a packed threshold for half_passes).
// Key 0 (below every element) gives a NaN pattern, which every compare passes.
__device__ __forceinline__ uint32_t key_pair(uint32_t key) {
  const uint32_t b = (key & 0x8000u) ? (key & 0x7FFFu) : (~key & 0xFFFFu);
  return b | (b << 16);
}

// Per-warp selection state (warp-uniform).
struct Sel {
  uint32_t cnt;   // entries in buf
  uint32_t thr;   // threshold key
  uint32_t thr2;  // key_pair(thr)
  bool ge;        // a candidate needs key >= thr (until K entries are known to reach a key), else key > thr
};

__device__ __forceinline__ void sel_set(Sel& st, uint32_t key, bool ge) {
  st.thr = key;
  st.thr2 = key_pair(key);
  st.ge = ge;
}

// Bits e of the elements of v that pass the threshold exactly.  For values other than NaN,
// key(x) > thr exactly when x > value(thr) (-0 and +0 have one key), and the same for >=, so
// the test is a float compare; a vector holding a NaN, or a NaN threshold, takes the key path.
__device__ __forceinline__ uint32_t elem_mask(const uint4& v, const Sel& st) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t take = 0;
  uint32_t m = vec_max2(v);
  m = bmax2(m, __byte_perm(m, 0u, 0x1032));
  const float mx = __uint_as_float(m & 0xFFFF0000u);
  const float t = key_to_float(st.thr);
  if (mx == mx && t == t) {
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
      if (st.ge ? key >= st.thr : key > st.thr) take |= 1u << e;
    }
  }
  return take;
}

// Warp: the K-th largest key T of the buffer (cnt >= K) becomes the threshold.  With
// `strict` (every element queued so far is in the buffer), a later element needs key > T:
// an equal key comes with a larger column and ranks below those K.  Part-way through a
// drain, queue slots still to come may hold elements of earlier columns than some in the
// buffer, so an element with key T may still outrank one of those K: key >= T.  With
// `cut`, the buffer is also filtered to the entries that reach T, and cut to its best K
// (an element it drops has K entries above it) when ties leave less than a slot's room.
template <class C>
__device__ __noinline__ Sel tw_raise(TwSmem<C>& ws, Sel st, uint32_t K, bool cut, bool strict) {
  const uint2 tc = buf_rank_key(ws.buf, st.cnt, K);
  const uint32_t T = tc.x, cge = tc.y;
  if (cut && cge < st.cnt) st.cnt = buf_filter_ge(ws.buf, st.cnt, T);
  if (cut && st.cnt > uint32_t(C::CAP - TW_STEP)) {
    warp_sort_desc(ws.buf, st.cnt);
    st.cnt = K;
  }
  sel_set(st, T, !strict);
  return st;
}

// Warp: move every lane's queued vectors (nq of them in this lane) into the candidate
// buffer one queue slot at a time, keeping the elements that pass the threshold exactly and
// raising the threshold before a slot that might not fit.  The selection state goes in and
// out by value (out of line, a reference would keep it in local memory).
template <class C>
__device__ __noinline__ Sel tw_drain_slots(TwSmem<C>& ws, Sel st, uint32_t nq, uint32_t V32, uint32_t K) {
  const uint32_t lane = lane_id();
  const uint32_t slots = __reduce_max_sync(0xffffffffu, nq);
  for (uint32_t j = 0; j < slots; ++j) {
    if (st.cnt + TW_STEP > uint32_t(C::CAP)) st = tw_raise(ws, st, K, true, false);  // room for a slot's elements
    uint32_t take = 0, col0 = 0;
    unsigned long long lo = 0, hi = 0;
    if (j < nq && KD_DCHECK(j < uint32_t(C::QL), ws.err, 0x7102)) {
      const uint4 v = ws.qv[j][lane];
      col0 = ws.qcol[j][lane];
      lo = (static_cast<unsigned long long>(v.y) << 32) | v.x;
      hi = (static_cast<unsigned long long>(v.w) << 32) | v.z;
      take = elem_mask(v, st);
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
    uint32_t pos = st.cnt + pre;
    while (take) {
      const uint32_t e = __ffs(take) - 1;
      take &= take - 1;
      const uint32_t bits = uint32_t(((e & 4) ? hi : lo) >> (16 * (e & 3))) & 0xFFFFu;
      if (KD_DCHECK(pos < uint32_t(C::CAP), ws.err, 0x7101)) ws.buf[pos] = cand_make(bits, col0 + e);
      ++pos;
    }
    st.cnt += tot;
    __syncwarp();
  }
  return st;
}

// The lane's queued vectors tested exactly against the threshold: for each of its nq slots
// the bits of the elements that pass (elements past the row's end never do), eight bits per
// slot, slots 0-7 in mw[0] and 8-15 in mw[1]; returns how many pass.
template <class C>
__device__ __forceinline__ uint32_t queue_masks(const TwSmem<C>& ws, const Sel& st, uint32_t nq, uint32_t V32,
                                                unsigned long long (&mw)[2]) {
  static_assert(C::QL <= 16, "two 64-bit words of slot masks");
  const uint32_t lane = lane_id();
  uint32_t n = 0;
  mw[0] = 0ull;
  mw[1] = 0ull;
#pragma unroll 1
  for (uint32_t j = 0; j < nq; ++j) {
    const uint4 v = ws.qv[j][lane];
    const uint32_t col0 = ws.qcol[j][lane];
    uint32_t take = elem_mask(v, st);
    if (col0 + TK_VEC > V32) take &= (V32 > col0 ? (1u << (V32 - col0)) - 1u : 0u);
    const unsigned long long t = static_cast<unsigned long long>(take) << (8 * (j & 7u));
    if (j < 8u) mw[0] |= t; else mw[1] |= t;
    n += uint32_t(__popc(take));
  }
  return n;
}

// Warp: move every lane's queued vectors into the candidate buffer, keeping the elements that
// pass the threshold exactly, then (with `raise`: more of the row is still to come) raise the
// threshold once the buffer holds K entries.  A row's last drain leaves the buffer as it is:
// the hand-over finds the same K-th key itself.
// Every lane tests all its vectors first (no warp operation between them), one prefix sum
// over the lanes' counts places them, and each lane writes its own.  When they do not all
// fit, they go one queue slot at a time, the threshold raised between slots.  (Raising it on
// the buffer first would not help: every drain ends with the threshold at the buffer's K-th
// key, and the buffer is unchanged until the next drain.)
template <class C>
__device__ __noinline__ Sel tw_drain(TwSmem<C>& ws, Sel st, uint32_t nq, uint32_t V32, uint32_t K, bool raise) {
  static_assert(8 * C::QL < 128, "a lane's passing count fits the seven-bit prefix sum");
  const uint32_t lane = lane_id();
  unsigned long long mw[2];
  const uint32_t n = queue_masks<C>(ws, st, nq, V32, mw);
  const uint32_t tot = __reduce_add_sync(0xffffffffu, n);
  if (st.cnt + tot > uint32_t(C::CAP)) {
    st = tw_drain_slots(ws, st, nq, V32, K);
  } else {
    const uint32_t lt = (1u << lane) - 1u;
    uint32_t pre = 0;
#pragma unroll
    for (int b = 0; b < 7; ++b) pre += uint32_t(__popc(__ballot_sync(0xffffffffu, (n >> b) & 1u) & lt)) << b;
    uint32_t pos = st.cnt + pre;
#pragma unroll 1
    for (uint32_t j = 0; j < nq; ++j) {
      uint32_t take = uint32_t((j < 8u ? mw[0] : mw[1]) >> (8 * (j & 7u))) & 0xFFu;
      if (take) {
        const uint4 v = ws.qv[j][lane];
        const uint32_t col0 = ws.qcol[j][lane];
        const unsigned long long lo = (static_cast<unsigned long long>(v.y) << 32) | v.x;
        const unsigned long long hi = (static_cast<unsigned long long>(v.w) << 32) | v.z;
        do {
          const uint32_t e = __ffs(take) - 1;
          take &= take - 1;
          const uint32_t bits = uint32_t(((e & 4) ? hi : lo) >> (16 * (e & 3))) & 0xFFFFu;
          if (KD_DCHECK(pos < uint32_t(C::CAP), ws.err, 0x7101)) ws.buf[pos] = cand_make(bits, col0 + e);
          ++pos;
        } while (take);
      }
    }
    st.cnt += tot;
    __syncwarp();
  }
  if (raise && st.cnt >= K) st = tw_raise(ws, st, K, st.cnt > uint32_t(C::CAP / 2), true);
  return st;
}

// Row logsumexp, per lane: an offset lm (natural units) and, per step of a group, a packed
// pair of partial sums of e^(x - lm) = 2^(x log2 e - lm log2 e); four independent chains.
// The offset moves only when a group's maximum passes it by more than TW_LSE_SLACK, so that
// every term stays below e^TW_LSE_SLACK and the rescale of the sums is rare.
constexpr float TW_LSE_SLACK = 8.f;

struct LseAcc {
  float lm;                               // offset (-inf: nothing seen yet)
  unsigned long long acc[TW_GROUP];       // packed f32x2 partial sums
};

__device__ __forceinline__ unsigned long long f32x2_splat(float x) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "r"(__float_as_uint(x)));
  return r;
}

__device__ __forceinline__ void lse_init(LseAcc& a) {
  a.lm = -INFINITY;
#pragma unroll
  for (int k = 0; k < TW_GROUP; ++k) a.acc[k] = 0ull;
}

// Add the live steps' vectors of one group; gm = the group's largest value.
__device__ __forceinline__ void lse_group(LseAcc& a, const uint4* v, uint32_t live, float gm) {
  if (gm > a.lm + TW_LSE_SLACK) {  // also the first finite value (lm = -inf); never a NaN
    const unsigned long long f = f32x2_splat(a.lm == -INFINITY ? 0.f : ex2_approx((a.lm - gm) * TW_LOG2E));
#pragma unroll
    for (int k = 0; k < TW_GROUP; ++k) asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(a.acc[k]) : "l"(f));
    a.lm = gm;
  }
  if (a.lm == -INFINITY) return;  // every value so far is -inf: every term is 0
  const unsigned long long l2e2 = f32x2_splat(TW_LOG2E), nb2 = f32x2_splat(-a.lm * TW_LOG2E);
#pragma unroll
  for (int k = 0; k < TW_GROUP; ++k) {
    if ((live >> k) & 1u) {
      const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
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
        asm("add.rn.f32x2 %0, %0, %1;" : "+l"(a.acc[k]) : "l"(e));
      }
    }
  }
}

// The lane's (offset, sum) pair.
__device__ __forceinline__ float lse_sum(const LseAcc& a) {
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < TW_GROUP; ++k) {
    uint32_t lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(a.acc[k]));
    s += __uint_as_float(lo) + __uint_as_float(hi);
  }
  return s;
}

// One group of TW_GROUP steps of a lane, vectors v[0 ..]: the packed pre-test of each against
// the threshold; the vectors that pass go to the lane's queue (predicated stores), and the
// warp drains the queues when one of them has less than a group's room left.  s0 = the
// group's first step; `live` = its steps that exist (the row's last group may have fewer).
template <class C, bool WITH_LSE>
__device__ __forceinline__ void tw_group(TwSmem<C>& ws, Sel& st, uint32_t& nq, const uint4* v, int s0,
                                         uint32_t live, LseAcc& la, uint32_t V32, uint32_t K) {
  const uint32_t lane = lane_id();
  uint32_t m[TW_GROUP];
#pragma unroll
  for (int k = 0; k < TW_GROUP; ++k) m[k] = ((live >> k) & 1u) ? vec_max2(v[k]) : 0xFF80FF80u;  // -inf pair
  if (WITH_LSE) {
    uint32_t g = bmax2(bmax2(m[0], m[1]), bmax2(m[2], m[3]));
    g = bmax2(g, __byte_perm(g, 0u, 0x1032));
    lse_group(la, v, live, __uint_as_float(g & 0xFFFF0000u));
  }
  // nq <= QL - TW_GROUP when a group starts, so every slot addressed below is inside the queue
#pragma unroll
  for (int k = 0; k < TW_GROUP; ++k) {
    if (half_passes(m[k], st.thr2, st.ge) && KD_DCHECK(nq < uint32_t(C::QL), ws.err, 0x7103)) {
      ws.qv[nq][lane] = v[k];
      ws.qcol[nq][lane] = uint32_t(s0 + k) * TW_STEP + lane * TK_VEC;
      ++nq;
    }
  }
  if (__any_sync(0xffffffffu, nq > uint32_t(C::QL - TW_GROUP))) {
    __syncwarp();
    st = tw_drain(ws, st, nq, V32, K, true);
    nq = 0;
  }
}

// Warp: hand the row's best candidates over (cnt >= K entries in the buffer): those whose
// key reaches the K-th largest key (K of them, more on ties, cut to the best K when ties
// make more than TW_HAND), written to hand[0 ..], their count to *hand_cnt.
template <class C>
__device__ __noinline__ void tw_hand_over(TwSmem<C>& ws, Sel st, uint32_t K, unsigned long long* hand,
                                         uint32_t* hand_cnt) {
  const uint32_t lane = lane_id();
  uint32_t cge = st.cnt;
  uint32_t T = 0;
  if (st.cnt > K) {
    const uint2 tc = buf_rank_key(ws.buf, st.cnt, K);
    T = tc.x;
    cge = tc.y;
  }
  if (cge > uint32_t(TW_HAND)) {  // ties at T: order the buffer and keep exactly the best K
    warp_sort_desc(ws.buf, st.cnt);
    for (uint32_t i = lane; i < K; i += 32) hand[i] = ws.buf[i];
    if (lane == 0) *hand_cnt = K;
    __syncwarp();
    return;
  }
  uint32_t out = 0;
  for (uint32_t base = 0; base < st.cnt; base += 32) {
    const uint32_t i = base + lane;
    const unsigned long long c = i < st.cnt ? ws.buf[i] : 0ull;
    const bool take = i < st.cnt && cand_key(c) >= T;
    const uint32_t bal = __ballot_sync(0xffffffffu, take);
    const uint32_t at = out + __popc(bal & ((1u << lane) - 1u));
    if (take && KD_DCHECK(at < uint32_t(TW_HAND), ws.err, 0x7104)) hand[at] = c;
    out += __popc(bal);
  }
  if (lane == 0) *hand_cnt = out;
  __syncwarp();
}

// Warp: the selection of one row again, read directly from global memory (the next group's
// loads in flight while a group is tested), from the exact start T0.  Out of line: it runs
// only after a speculative start left fewer than K elements.
template <class C>
__device__ __noinline__ Sel tw_reselect(TwSmem<C>& ws, const uint16_t* xr, int64_t V, int nst, uint32_t T0,
                                        uint32_t V32, uint32_t K) {
  Sel st;
  st.cnt = 0;
  sel_set(st, T0, true);
  uint32_t nq = 0;
  LseAcc la;  // unused: the logsumexp pass is already complete
  lse_init(la);
  uint4 a[TW_GROUP], b[TW_GROUP];
  load_group(a, xr, V, 0);
  for (int s0 = 0; s0 < nst; s0 += TW_GROUP) {
    if (s0 + TW_GROUP < nst) load_group(b, xr, V, s0 + TW_GROUP);
    const uint32_t live = nst - s0 >= TW_GROUP ? (1u << TW_GROUP) - 1u : (1u << (nst - s0)) - 1u;
    tw_group<C, false>(ws, st, nq, a, s0, live, la, V32, K);
#pragma unroll
    for (int k = 0; k < TW_GROUP; ++k) a[k] = b[k];
  }
  if (__any_sync(0xffffffffu, nq > 0)) st = tw_drain(ws, st, nq, V32, K, false);
  return st;
}

template <class C, bool WITH_LSE>
__global__ void __launch_bounds__(C::WARPS * 32, 1)
    kd_topk_stream_kernel(const uint16_t* __restrict__ X, int64_t N, int64_t V, int64_t ld, int K,
                          unsigned long long* __restrict__ hand, uint32_t* __restrict__ hand_cnt,
                          float* __restrict__ lse_out, uint32_t* err, const uint16_t* __restrict__ tile_max,
                          int64_t ld_tile_max, int ntiles) {
  extern __shared__ __align__(16) uint8_t tkt_smem_raw[];
  constexpr uint32_t GBYTES = uint32_t(TW_GROUP) * TW_STEP * 2;
  const uint32_t lane = lane_id();
  TwSmem<C>& ws = reinterpret_cast<TwSmem<C>*>(tkt_smem_raw)[threadIdx.x >> 5];
  const int64_t nwarps = int64_t(gridDim.x) * C::WARPS;
  const int nst = int((V + TW_STEP - 1) / TW_STEP);
  const int ngr = (nst + TW_GROUP - 1) / TW_GROUP;  // groups per row
  const uint32_t V32 = uint32_t(V), Ku = uint32_t(K);
  // this lane's vector in a row's last step is not a whole 16 bytes inside the row
  const bool tail_lane = int64_t(nst - 1) * TW_STEP + int64_t(lane) * TK_VEC + TK_VEC > V;

  if (lane == 0) {
    for (int r = 0; r < C::RING; ++r) mbar_init(&ws.full[r], 1);
    ws.abort = 0;
    ws.never = 0;
    ws.err = err;
    fence_mbar_init();
  }
  __syncwarp();

  int64_t row = int64_t(blockIdx.x) * C::WARPS + (threadIdx.x >> 5);
  // Producer: the warp's rows one after another, group by group.  A row's last group copies
  // the whole 16-byte vectors that remain (possibly none).
  const uint32_t last_bytes = uint32_t((V - int64_t(ngr - 1) * TW_GROUP * TW_STEP) * 2) & ~15u;
  int64_t prow = row;
  const uint16_t* psrc = X + prow * ld;  // the producer's current group
  int pg = 0;
  uint32_t issued = 0;
  auto issue = [&](uint32_t slot) {
    if (prow < N) {
      if (lane == 0) {
        uint32_t bytes = pg < ngr - 1 ? GBYTES : last_bytes;
        if (!KD_DCHECK(psrc + bytes / 2 <= X + prow * ld + V, err, 0x7401)) bytes = 0;
        mbar_arrive_expect_tx(&ws.full[slot], bytes);  // 0 bytes: the phase completes on the arrival
        if (bytes != 0) bulk_g2s(&ws.ring[slot][0][0], psrc, bytes, &ws.full[slot]);
      }
      ++issued;
      psrc += TW_GROUP * TW_STEP;
      if (++pg == ngr) {
        pg = 0;
        prow += nwarps;
        psrc = X + prow * ld;
      }
    }
  };
  for (int r = 0; r < C::RING; ++r) issue(uint32_t(r));

  uint32_t gidx = 0;  // groups consumed
  bool ok = true;
  bool may_speculate = K >= TW_SPEC_MIN_K;
  for (; row < N; row += nwarps) {
    const uint16_t* xr = X + row * ld;
    Sel st;
    st.cnt = 0;
    sel_set(st, 0u, true);  // key >= 0: every element, until a start applies
    uint32_t nq = 0;
    LseAcc la;
    lse_init(la);
    uint32_t T0 = 0;        // exact start (0: none)
    bool speculative = false;

    const bool tiles = tile_max != nullptr && ntiles >= K;
    if (tiles) {
      // The K-th largest of the row's tile maxima (ntiles >= K disjoint column ranges) is
      // reached by at least K elements: an exact start near the row's K-th value.
      const uint32_t T = warp_kth_largest_bf16(tile_max + row * ld_tile_max, uint32_t(ntiles), Ku, ws.hist);
      if (T != 0) sel_set(st, T, true);
    } else if (ngr > TW_QS) {
      // The ring holds this row's first TW_QS groups (none of them the row's last).
      for (int r = 0; r < TW_QS && ok; ++r) {
        const uint32_t u = gidx + uint32_t(r);
        ok = mbar_wait(&ws.full[u % C::RING], (u / C::RING) & 1u, &ws.abort, err, 0x72u);
      }
      if (!ok) break;
      static_assert(TW_QS * TW_GROUP == 16, "the bracket bounds below take 16 keys per lane");
      uint32_t kp[TW_QS * TW_GROUP];  // the lane's vector maxima keys + 1
#pragma unroll
      for (int r = 0; r < TW_QS; ++r) {
#pragma unroll
        for (int k = 0; k < TW_GROUP; ++k) {
          const uint4 v = ws.ring[(gidx + r) % C::RING][k][lane];
          const float mx = vec_max(v);
          uint32_t key;
          if (mx == mx) {
            key = bf16_key(__float_as_uint(mx) >> 16);
          } else {  // a NaN hides the maximum: take the exact keys
            key = 0;
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) key = max(key, max(bf16_key(w[h]), bf16_key(w[h] >> 16)));
          }
          kp[r * TW_GROUP + k] = key + 1u;
        }
      }
      const uint32_t rank[2] = {Ku, Ku / 4 > 0 ? Ku / 4 : 1u};
      // Lower bounds for the bracket: when every lane has g keys that reach b (the smallest
      // of its g group maxima, groups of 16 / g consecutive keys), 32 g keys reach the smallest
      // b of the warp; g is the least power of two with 32 g >= rank.
      // lb[l]: the lane's smallest maximum over groups of 16 >> l keys (lb[0] its largest key)
      uint32_t p2[8], p4[4], lb[5];
#pragma unroll
      for (int i = 0; i < 8; ++i) p2[i] = max(kp[2 * i], kp[2 * i + 1]);
#pragma unroll
      for (int i = 0; i < 4; ++i) p4[i] = max(p2[2 * i], p2[2 * i + 1]);
      const uint32_t p8a = max(p4[0], p4[1]), p8b = max(p4[2], p4[3]);
      lb[0] = max(p8a, p8b);
      lb[1] = min(p8a, p8b);
      lb[2] = min(min(p4[0], p4[1]), min(p4[2], p4[3]));
      lb[3] = p2[0];
#pragma unroll
      for (int i = 1; i < 8; ++i) lb[3] = min(lb[3], p2[i]);
      lb[4] = kp[0];
#pragma unroll
      for (int i = 1; i < 16; ++i) lb[4] = min(lb[4], kp[i]);
      uint32_t hint[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const uint32_t g = (rank[r] + 31u) / 32u;
        const uint32_t b = g <= 1u ? lb[0] : g <= 2u ? lb[1] : g <= 4u ? lb[2] : g <= 8u ? lb[3] : lb[4];
        hint[r] = __reduce_min_sync(0xffffffffu, b);
      }
      uint32_t T[2], cge[2];
      warp_rank_keys<TW_QS * TW_GROUP, 2>(kp, rank, T, cge, hint);
      T0 = T[0];
      uint32_t start = T0;
      if (may_speculate) {
        const uint32_t T1 = T[1];
        const bool finite = T0 > 0x007Fu && T1 < 0xFF80u;  // both keys of finite values
        if (finite && T1 > T0) {
          const float v0 = key_to_float(T0), v1 = key_to_float(T1);
          const uint32_t Ts = key_floor(fmaf(TW_SPEC_C, v1 - v0, v0));
          if (Ts > T0) {
            start = Ts;
            speculative = true;
          }
        }
      }
      if (start != 0) sel_set(st, start, true);
    }

    for (int g = 0; g < ngr; ++g, ++gidx) {
      const uint32_t slot = gidx % C::RING;
      if (!mbar_wait(&ws.full[slot], (gidx / C::RING) & 1u, &ws.abort, err, 0x70u)) {
        ok = false;
        break;
      }
      uint4 v[TW_GROUP];
#pragma unroll
      for (int k = 0; k < TW_GROUP; ++k) v[k] = ws.ring[slot][k][lane];
      const int s0 = g * TW_GROUP;
      uint32_t live = (1u << TW_GROUP) - 1u;
      if (g == ngr - 1) {  // the row's last group
        live = nst - s0 >= TW_GROUP ? live : (1u << (nst - s0)) - 1u;
        if (tail_lane) {
#pragma unroll
          for (int k = 0; k < TW_GROUP; ++k)
            if (s0 + k == nst - 1) v[k] = load_step(xr, V, nst - 1);
        }
      }
      // The slot is refilled by the async proxy: every lane's reads of it are ordered before
      // the refill (a proxy fence in each lane, then the warp barrier before lane 0 issues).
      fence_proxy_async_cta();
      __syncwarp();
      issue(slot);
      tw_group<C, WITH_LSE>(ws, st, nq, v, s0, live, la, V32, Ku);
    }
    if (!ok) break;
    if (__any_sync(0xffffffffu, nq > 0)) st = tw_drain(ws, st, nq, V32, Ku, false);
    if (speculative && st.cnt < Ku) {
      // fewer than K elements reach the speculative start: select the row again from T0
      st = tw_reselect(ws, xr, V, nst, T0, V32, Ku);
      may_speculate = false;
      if (lane == 0) atomicAdd(err + 2, 1u);
    }
    if (WITH_LSE) {
      float lm = la.lm, ls = lse_sum(la);
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
    tw_hand_over(ws, st, Ku, hand + row * TW_HAND, hand_cnt + row);
  }
  if (!ok) {  // a wait timed out: let this warp's copies still in flight land (bounded) before leaving
    for (uint32_t u = gidx; u < issued; ++u)
      mbar_wait(&ws.full[u % C::RING], (u / C::RING) & 1u, &ws.never, err, 0x71u, 10000000ull);
  }
}

// Warp: sort the 32 E candidates a[] of the warp descending, in registers: a bitonic network
// over positions p = lane E + i; a partner within the lane is swapped in place, one in
// another lane (distance >= E) comes by shuffle.
template <int E>
__device__ __forceinline__ void warp_sort_regs_desc(unsigned long long (&a)[E]) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int k = 2; k <= 32 * E; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= E) {
        const uint32_t lm = uint32_t(j / E);
#pragma unroll
        for (int i = 0; i < E; ++i) {
          const uint32_t p = lane * E + i;
          const unsigned long long o = __shfl_xor_sync(0xffffffffu, a[i], lm);
          const bool desc = (p & uint32_t(k)) == 0;
          const bool lower = (p & uint32_t(j)) == 0;
          const bool keep_max = desc == lower;
          a[i] = keep_max ? (a[i] > o ? a[i] : o) : (a[i] < o ? a[i] : o);
        }
      } else {
#pragma unroll
        for (int i = 0; i < E; ++i) {
          if ((i & j) == 0) {
            const uint32_t p = lane * E + i;
            const bool desc = (p & uint32_t(k)) == 0;
            const unsigned long long x = a[i], y = a[i + j];
            const bool swap = desc ? (x < y) : (x > y);
            a[i] = swap ? y : x;
            a[i + j] = swap ? x : y;
          }
        }
      }
    }
  }
}

// Warp: sort one row's handed-over candidates (cnt <= 32 E) and write the first K.
template <int E>
__device__ __forceinline__ void emit_row(const unsigned long long* hand, uint32_t cnt, uint32_t K, int32_t* ids_row,
                                         float* vals_row, const float* lse, float* dropped) {
  const uint32_t lane = lane_id();
  unsigned long long a[E];
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const uint32_t p = lane * E + i;
    a[i] = p < cnt ? hand[p] : 0ull;  // 0 ranks below every candidate (its ~column is never 0)
  }
  warp_sort_regs_desc<E>(a);
  float s = 0.f, comp = 0.f;
  const float l = dropped ? *lse : 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    const uint32_t p = lane * E + i;
    if (p < K) {
      const bool real = p < cnt;
      ids_row[p] = real ? int32_t(cand_col(a[i])) : -1;
      const float v = real ? __uint_as_float(cand_bits(a[i]) << 16) : -INFINITY;
      vals_row[p] = v;
      if (dropped && real) {  // compensated running sum of exp(v_k - lse)
        const float y = expf(v - l) - comp;
        const float t = s + y;
        comp = (t - s) - y;
        s = t;
      }
    }
  }
  if (dropped) {
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) *dropped = 1.f - s;
  }
}

constexpr int EMIT_WARPS = 8;

__global__ void __launch_bounds__(EMIT_WARPS * 32)
    kd_topk_emit_kernel(const unsigned long long* __restrict__ hand, const uint32_t* __restrict__ hand_cnt,
                        int64_t N, int K, int32_t* __restrict__ ids_out, float* __restrict__ vals_out,
                        const float* __restrict__ lse, float* __restrict__ dropped_out, uint32_t* err) {
  const int64_t nwarps = int64_t(gridDim.x) * EMIT_WARPS;
  for (int64_t row = int64_t(blockIdx.x) * EMIT_WARPS + (threadIdx.x >> 5); row < N; row += nwarps) {
    uint32_t cnt = hand_cnt[row];
    // at most TW_HAND (a row the streaming kernel never reached, after a timed-out wait it
    // reported, holds no count: its outputs are not defined, but nothing is read past its slot)
    if (!KD_DCHECK(cnt <= uint32_t(TW_HAND), err, 0x7501) || cnt > uint32_t(TW_HAND)) cnt = TW_HAND;
    const unsigned long long* h = hand + row * TW_HAND;
    int32_t* ids_row = ids_out + row * K;
    float* vals_row = vals_out + row * K;
    float* d = dropped_out ? dropped_out + row : nullptr;
    if (cnt <= 128u && K <= 128)
      emit_row<4>(h, cnt, uint32_t(K), ids_row, vals_row, lse ? lse + row : nullptr, d);
    else
      emit_row<8>(h, cnt, uint32_t(K), ids_row, vals_row, lse ? lse + row : nullptr, d);
  }
}

// Streaming-kernel shared memory and its per-device attribute.
template <class C>
static cudaError_t launch_topk_stream(const uint16_t* X, int64_t N, int64_t V, int64_t ld, int K,
                                      unsigned long long* hand, uint32_t* hand_cnt, float* lse, uint32_t* err,
                                      cudaStream_t s, const uint16_t* tile_max, int64_t ld_tile_max, int ntiles) {
  static PerDevice<int> attr_plain, attr_lse;
  const int smem = int(C::WARPS * sizeof(TwSmem<C>));
  cudaError_t e = smem_attr_once(attr_plain, reinterpret_cast<const void*>(kd_topk_stream_kernel<C, false>), smem);
  if (e == cudaSuccess)
    e = smem_attr_once(attr_lse, reinterpret_cast<const void*>(kd_topk_stream_kernel<C, true>), smem);
  if (e != cudaSuccess) return e;
  int grid = gemm_max_grid();  // one block of C::WARPS row-streaming warps per SM
  if (int64_t(grid) * C::WARPS > N) grid = int((N + C::WARPS - 1) / C::WARPS);
  if (lse)
    kd_topk_stream_kernel<C, true><<<grid, C::WARPS * 32, smem, s>>>(X, N, V, ld, K, hand, hand_cnt, lse, err,
                                                                      tile_max, ld_tile_max, ntiles);
  else
    kd_topk_stream_kernel<C, false><<<grid, C::WARPS * 32, smem, s>>>(X, N, V, ld, K, hand, hand_cnt, lse, err,
                                                                       tile_max, ld_tile_max, ntiles);
  return cudaGetLastError();
}

bool topk_takes_known_lse(int K) { return K <= TW_MAXK; }

size_t topk_scratch_bytes(int64_t N, int K) {
  if (K > TW_MAXK) return 0;
  // per row: TW_HAND candidates, their count, the logsumexp (for the dropped mass)
  return size_t(N) * TW_HAND * 8 + (size_t(N) * 4 + 255) / 256 * 256 + size_t(N) * 4;
}

cudaError_t launch_topk(const uint16_t* X, int64_t N, int64_t V, int64_t ld, int K, int32_t* ids, float* vals,
                        float* lse, float* dropped, uint32_t* err, void* scratch, cudaStream_t s,
                        const uint16_t* tile_max, int64_t ld_tile_max, int ntiles, const float* lse_known) {
  if (N <= 0) return cudaSuccess;
  prof_before("kd_topk_cache", s);
  if (K <= TW_MAXK) {
    uint8_t* w8 = static_cast<uint8_t*>(scratch);
    unsigned long long* hand = reinterpret_cast<unsigned long long*>(w8);
    uint32_t* hand_cnt = reinterpret_cast<uint32_t*>(w8 + size_t(N) * TW_HAND * 8);
    float* lse_ws = reinterpret_cast<float*>(w8 + size_t(N) * TW_HAND * 8 + (size_t(N) * 4 + 255) / 256 * 256);
    // the dropped mass needs the logsumexp: given, else computed by the selection
    float* lse_rows = lse_known ? nullptr : (lse ? lse : (dropped ? lse_ws : nullptr));
    const float* lse_emit = lse_known ? lse_known : lse_rows;
    cudaError_t e = K <= TmSmallK::MAXK
                        ? launch_topk_stream<TmSmallK>(X, N, V, ld, K, hand, hand_cnt, lse_rows, err, s, tile_max,
                                                       ld_tile_max, ntiles)
                        : launch_topk_stream<TmLargeK>(X, N, V, ld, K, hand, hand_cnt, lse_rows, err, s, tile_max,
                                                       ld_tile_max, ntiles);
    if (e != cudaSuccess) return e;
    int grid = 4 * gemm_max_grid();
    if (int64_t(grid) * EMIT_WARPS > N) grid = int((N + EMIT_WARPS - 1) / EMIT_WARPS);
    kd_topk_emit_kernel<<<grid, EMIT_WARPS * 32, 0, s>>>(hand, hand_cnt, N, K, ids, vals, lse_emit, dropped, err);
  } else {
    static PerDevice<int> attr;
    const int smem = int(sizeof(TopkSmem));
    cudaError_t ea = smem_attr_once(attr, reinterpret_cast<const void*>(kd_topk_kernel), smem);
    if (ea != cudaSuccess) return ea;
    int grid = 2 * gemm_max_grid();
    if (int64_t(grid) > N) grid = int(N);
    kd_topk_kernel<<<grid, TK_THREADS, smem, s>>>(X, N, V, ld, K, ids, vals, lse, dropped, err);
  }
  prof_after(s);
  return cudaGetLastError();
}

}  // namespace kd
