// Span builder and row schedule ("perf(megatron): add block-sparse fused
// LM-head backward", SkyRL PR #2376: "What does this PR do?" - ordered active
// spans; Bugbot "Overview" - spans coalesced with gaps <= 128; "How it works" -
// spans are used without reordering tokens).
//
// The page builds spans on the host before the device copy; here they are
// built on the device (edge detection + block scans + stream compaction), so a
// training step never waits on the host and the calls can be graph-captured.
//
// Kernels:
//   spans_build_kernel   mask -> spans[S][2], S                 (one CTA)
//   rowmap_count_kernel, rowmap_write_kernel
//                        spans + mask -> validated row schedule (one CTA per
//                        4096 tokens, two passes)
//   gather_rows_kernel   hidden rows of the schedule -> packed copy
//   combine_kernel       per-vocab-tile softmax partials -> lse, entropy, logp
//   zero_unpacked_rows_kernel  dhidden rows that no GEMM tile writes -> 0
#include "eas_device.cuh"
#include "eas_kernels.h"

namespace eas {

namespace {

constexpr int kScanThreads = 1024;
constexpr int kScanItems = 16;
constexpr int kScanWarps = kScanThreads / 32;

// Block-wide exclusive sum (and the block total) of one int per thread.
__device__ __forceinline__ int block_excl_sum(int v, int* sm, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < kScanWarps) ? sm[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sm[lane] = w;
  }
  __syncthreads();
  const int before = warp ? sm[warp - 1] : 0;
  total = sm[kScanWarps - 1];
  __syncthreads();
  return before + x - v;
}

// Block-wide exclusive max (identity -1) and the block maximum.
__device__ __forceinline__ long long block_excl_max(long long v, long long* sm, long long& all) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = max(x, y);
  }
  long long excl = __shfl_up_sync(0xffffffffu, x, 1);
  if (lane == 0) excl = -1;
  if (lane == 31) sm[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long w = (lane < kScanWarps) ? sm[lane] : -1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w = max(w, y);
    }
    sm[lane] = w;
  }
  __syncthreads();
  const long long before = warp ? sm[warp - 1] : -1;
  all = sm[kScanWarps - 1];
  __syncthreads();
  return max(before, excl);
}

}  // namespace

// One CTA walks the mask in tiles of kScanThreads * kScanItems tokens.  A token
// t starts a span when it is active and the previous active token p is absent
// or more than max_gap tokens away (t - p - 1 > max_gap); at that point the
// previous span ends at p + 1.  The last span ends after the last active token.
__global__ void __launch_bounds__(kScanThreads)
spans_build_kernel(const uint8_t* __restrict__ mask, long long T, int max_gap,
                   int* __restrict__ spans, long long cap, int* __restrict__ num_spans,
                   DevStatus* st) {
  __shared__ int sm_i[32];
  __shared__ long long sm_l[32];
  long long carry_last = -1;   // last active token before the current tile
  long long carry_count = 0;   // spans started before the current tile
  const long long tile = static_cast<long long>(kScanThreads) * kScanItems;
  for (long long base = 0; base < T; base += tile) {
    const long long t0 = base + static_cast<long long>(threadIdx.x) * kScanItems;
    uint32_t bits = 0;
#pragma unroll
    for (int i = 0; i < kScanItems; ++i) {
      const long long t = t0 + i;
      if (t < T && mask[t] != 0) bits |= 1u << i;
    }
    long long my_last = -1;
#pragma unroll
    for (int i = 0; i < kScanItems; ++i)
      if (bits & (1u << i)) my_last = t0 + i;
    long long tile_max;
    long long prev = block_excl_max(my_last, sm_l, tile_max);
    prev = max(prev, carry_last);
    int cnt = 0;
    uint32_t starts = 0;
    long long p = prev;
#pragma unroll
    for (int i = 0; i < kScanItems; ++i) {
      if (bits & (1u << i)) {
        const long long t = t0 + i;
        if (p < 0 || t - p - 1 > static_cast<long long>(max_gap)) {
          starts |= 1u << i;
          ++cnt;
        }
        p = t;
      }
    }
    int total;
    const int excl = block_excl_sum(cnt, sm_i, total);
    long long k = carry_count + excl;
    p = prev;
#pragma unroll
    for (int i = 0; i < kScanItems; ++i) {
      if (bits & (1u << i)) {
        const long long t = t0 + i;
        if (starts & (1u << i)) {
          if (k < cap) spans[2 * k] = static_cast<int>(t);
          if (k >= 1 && k - 1 < cap) spans[2 * (k - 1) + 1] = static_cast<int>(p + 1);
          ++k;
        }
        p = t;
      }
    }
    carry_count += total;
    carry_last = max(carry_last, tile_max);
  }
  if (threadIdx.x == 0) {
    if (carry_count > 0 && carry_count - 1 < cap)
      spans[2 * (carry_count - 1) + 1] = static_cast<int>(carry_last + 1);
    *num_spans = static_cast<int>(carry_count);
    if (carry_count > cap) report(st, kStSpanCapacity, 1, static_cast<int>(carry_count));
  }
}

// Validates the spans and lists the rows the kernels work on, in span order:
//   row_map[r] = token of packed row r (r < R), -1 for r in [R, R_pad), R_pad =
//   R rounded up to 256 (a whole number of tensor-core tiles of either shape);
//   pack_of[t] = packed row of token t, or -1.
// A row is listed when it lies in a span and (policy EAS_ROWS_SPAN, or the
// token is active).  Spans must be sorted, disjoint, inside [0, T) and cover
// every active token; otherwise nothing is listed (R = 0) and the status word
// reads kStInvalidSpans.  Active tokens whose target lies outside [t_lo, t_hi)
// set kStInvalidArg (their outputs are then meaningless; nothing is read out
// of bounds).
//
// Two passes over tiles of kRmTile tokens, one CTA per tile:
//   rowmap_count_kernel  validates, counts each tile's listed rows into
//                        tile_rows[tile]; the CTA that finishes last turns
//                        the counts into exclusive offsets and writes R, R_pad;
//   rowmap_write_kernel  writes row_map / pack_of of its tile from its offset.
namespace {

constexpr int kRmThreads = 256;
constexpr int kRmItems = 16;
constexpr int kRmTile = kRmThreads * kRmItems;   // 4096 tokens per CTA
constexpr int kRmWarps = kRmThreads / 32;

// Block-wide exclusive sum of one long long per thread (kRmThreads threads);
// `total` receives the block's sum.
__device__ __forceinline__ long long rm_excl_sum(long long v, long long* sm, long long& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long w = (lane < kRmWarps) ? sm[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kRmWarps) sm[lane] = w;
  }
  __syncthreads();
  const long long before = warp ? sm[warp - 1] : 0;
  total = sm[kRmWarps - 1];
  __syncthreads();
  return before + x - v;
}

// The listed rows among this thread's kRmItems tokens starting at t0: bit i
// of the result is set when token t0 + i is listed.  `uncovered` is set when
// an active token lies outside every span.
__device__ __forceinline__ uint32_t rm_select(const uint8_t* __restrict__ mask,
                                              const int* __restrict__ spans, int S, long long T,
                                              long long t0, int span_rows, bool& uncovered) {
  // largest k with start_k <= t0 (or -1)
  int lo = 0, hi = S;  // search in [lo, hi)
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<long long>(spans[2 * mid]) <= t0) lo = mid + 1; else hi = mid;
  }
  int k = lo - 1;
  uint32_t sel = 0;
#pragma unroll 4
  for (int i = 0; i < kRmItems; ++i) {
    const long long t = t0 + i;
    if (t >= T) break;
    while (k + 1 < S && static_cast<long long>(spans[2 * (k + 1)]) <= t) ++k;
    const bool covered = (k >= 0) && (t < static_cast<long long>(spans[2 * k + 1]));
    const bool active = mask[t] != 0;
    if (active && !covered) uncovered = true;
    if (covered && (span_rows || active)) sel |= 1u << i;
  }
  return sel;
}

// Span count after the capacity check (0 when num_spans is out of range).
__device__ __forceinline__ int rm_span_count(const int* num_spans, long long cap) {
  const int S_raw = *num_spans;
  return (S_raw < 0 || static_cast<long long>(S_raw) > cap) ? 0 : S_raw;
}

}  // namespace

__global__ void __launch_bounds__(kRmThreads)
rowmap_count_kernel(const uint8_t* __restrict__ mask, const int* __restrict__ spans,
                    const int* __restrict__ num_spans, long long cap, long long T, int span_rows,
                    const int* __restrict__ targets, int t_lo, int t_hi,
                    long long* __restrict__ tile_rows, Sched* sched, DevStatus* st) {
  __shared__ long long sm_l[32];
  __shared__ int last;
  const int S_raw = *num_spans;
  const int S = rm_span_count(num_spans, cap);
  if (S != S_raw && blockIdx.x == 0 && threadIdx.x == 0) {
    report(st, S_raw < 0 ? kStInvalidSpans : kStSpanCapacity, 2, S_raw);
    atomicExch(&sched->bad, 1);
  }
  // span validity: sorted, non-empty, inside [0, T)
  for (long long k = static_cast<long long>(blockIdx.x) * kRmThreads + threadIdx.x; k < S;
       k += static_cast<long long>(gridDim.x) * kRmThreads) {
    const int s = spans[2 * k], e = spans[2 * k + 1];
    bool ok = (s >= 0) && (s < e) && (static_cast<long long>(e) <= T);
    if (k > 0) ok = ok && (spans[2 * k - 1] <= s);
    if (!ok) atomicExch(&sched->bad, 1);
  }
  const long long t0 = static_cast<long long>(blockIdx.x) * kRmTile +
                       static_cast<long long>(threadIdx.x) * kRmItems;
  bool uncovered = false;
  const uint32_t sel = rm_select(mask, spans, S, T, t0, span_rows, uncovered);
  if (targets != nullptr) {
    for (int i = 0; i < kRmItems; ++i) {
      const long long t = t0 + i;
      if (t >= T) break;
      if (mask[t] != 0) {
        const int tg = targets[t];
        if (tg < t_lo || tg >= t_hi) report(st, kStInvalidArg, 3, static_cast<int>(t));
      }
    }
  }
  if (uncovered) atomicExch(&sched->bad, 1);
  __threadfence();     // this thread's flags before the CTA's ticket below
  long long total;
  rm_excl_sum(__popc(sel), sm_l, total);
  if (threadIdx.x == 0) {
    tile_rows[blockIdx.x] = total;
    __threadfence();
    last = (atomicAdd(&sched->ticket, 1) == static_cast<int>(gridDim.x) - 1);
  }
  __syncthreads();
  if (!last) return;
  // the last CTA: every count and every `bad` flag of the grid is visible
  __threadfence();
  const int n = gridDim.x;
  long long carry = 0;
  for (int base = 0; base < n; base += kRmThreads) {
    const int i = base + threadIdx.x;
    const long long v = (i < n) ? *reinterpret_cast<volatile long long*>(&tile_rows[i]) : 0;
    long long part;
    const long long ex = rm_excl_sum(v, sm_l, part);
    if (i < n) tile_rows[i] = carry + ex;
    carry += part;
  }
  if (threadIdx.x == 0) {
    const bool bad = *reinterpret_cast<volatile int*>(&sched->bad) != 0;
    if (bad) report(st, kStInvalidSpans, 2, -1);
    sched->R = bad ? 0 : static_cast<int>(carry);
    sched->R_pad = bad ? 0 : static_cast<int>((carry + 255) / 256 * 256);
    sched->S = S_raw;
  }
}

__global__ void __launch_bounds__(kRmThreads)
rowmap_write_kernel(const uint8_t* __restrict__ mask, const int* __restrict__ spans,
                    const int* __restrict__ num_spans, long long cap, long long T, int span_rows,
                    const long long* __restrict__ tile_rows, int* __restrict__ row_map,
                    int* __restrict__ pack_of, const Sched* __restrict__ sched) {
  __shared__ long long sm_l[32];
  const long long t0 = static_cast<long long>(blockIdx.x) * kRmTile +
                       static_cast<long long>(threadIdx.x) * kRmItems;
  if (sched->bad) {
    for (int i = 0; i < kRmItems; ++i)
      if (t0 + i < T) pack_of[t0 + i] = -1;
    return;
  }
  const int S = rm_span_count(num_spans, cap);
  bool uncovered = false;
  const uint32_t sel = rm_select(mask, spans, S, T, t0, span_rows, uncovered);
  long long total;
  long long idx = tile_rows[blockIdx.x] + rm_excl_sum(__popc(sel), sm_l, total);
  for (int i = 0; i < kRmItems; ++i) {
    const long long t = t0 + i;
    if (t >= T) break;
    if (sel & (1u << i)) {
      row_map[idx] = static_cast<int>(t);
      pack_of[t] = static_cast<int>(idx);
      ++idx;
    } else {
      pack_of[t] = -1;
    }
  }
  if (blockIdx.x == gridDim.x - 1) {
    const long long R = sched->R, R_pad = sched->R_pad;
    for (long long r = R + threadIdx.x; r < R_pad; r += kRmThreads) row_map[r] = -1;
  }
}

// dst[r, :] = src[row_map[r], :] for r < R_pad (zeros for pad rows).  One
// 16-byte vector per thread per step; `vec_per_row` = H * sizeof(elem) / 16.
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                   const int* __restrict__ row_map, const Sched* __restrict__ sched,
                   long long vec_per_row) {
  const int R_pad = sched->R_pad;
  for (long long r = blockIdx.x; r < R_pad; r += gridDim.x) {
    const int t = row_map[r];
    uint4* d = dst + r * vec_per_row;
    if (t < 0) {
      for (long long i = threadIdx.x; i < vec_per_row; i += blockDim.x) d[i] = make_uint4(0, 0, 0, 0);
    } else {
      const uint4* s = src + static_cast<long long>(t) * vec_per_row;
      for (long long i = threadIdx.x; i < vec_per_row; i += blockDim.x) d[i] = __ldg(s + i);
    }
  }
}

// Folds the per-vocab-tile partials of each packed row into lse, entropy and
// logp.  Partials are kept in base-2 units: with y = z log2(e), partial n of
// row r holds, over the tile's valid columns, m = max y, s = sum 2^(y - m),
// u = sum 2^(y - m) (y - m).  Two states merge as
//   M = max(m_a, m_b), S = sum_i s_i 2^(m_i - M), U = sum_i 2^(m_i - M) (u_i + (m_i - M) s_i)
// so that S = sum_v exp(z_v - M ln2) and U ln2 = sum_v exp(z_v - M ln2) (z_v - M ln2):
//   lse = M ln2 + log S,  H = log S - (U / S) ln2,  logp = z_target - lse.
// A block handles 32 tokens; its 8 thread groups fold the tiles n = g, g+8,
// ... of each token (coalesced across the 32 tokens), then group 0 merges the
// 8 states in a fixed order.  Tokens without a packed row, or with mask 0,
// get zeros.
namespace {
constexpr int kCombTok = 32;
constexpr int kCombGroups = 8;

struct Lse3 {
  float m, s, u;
};

__device__ __forceinline__ void lse_merge(Lse3& a, float m, float s, float u) {
  if (s == 0.f) return;
  if (a.s == 0.f) {
    a.m = m; a.s = s; a.u = u;
    return;
  }
  if (m > a.m) {
    const float d = a.m - m;               // < 0
    const float f = ex2_approx(d);
    a.u = f * (a.u + d * a.s) + u;
    a.s = f * a.s + s;
    a.m = m;
  } else {
    const float d = m - a.m;               // <= 0
    const float f = ex2_approx(d);
    a.s += f * s;
    a.u += f * (u + d * s);
  }
}
// Group g's fold of packed row r over the tiles n = g, g + 8, g + 16, ...
// Four accumulators take every fourth of those tiles, so four tiles' loads
// are in flight at once, and merge in a fixed order at the end.
__device__ __forceinline__ Lse3 fold_tiles(const float* __restrict__ pm,
                                           const float* __restrict__ ps,
                                           const float* __restrict__ pu, int n_tiles,
                                           long long stride, int r, int g) {
  Lse3 a[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) a[j] = Lse3{0.f, 0.f, 0.f};
  int n = g;
  for (; n + 3 * kCombGroups < n_tiles; n += 4 * kCombGroups) {
    float m[4], sv[4], u[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const long long o = static_cast<long long>(n + j * kCombGroups) * stride + r;
      m[j] = pm[o];
      sv[j] = ps[o];
      u[j] = pu[o];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) lse_merge(a[j], m[j], sv[j], u[j]);
  }
  // at most three tiles remain
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    if (n < n_tiles) {
      const long long o = static_cast<long long>(n) * stride + r;
      lse_merge(a[j], pm[o], ps[o], pu[o]);
      n += kCombGroups;
    }
  }
#pragma unroll
  for (int j = 1; j < 4; ++j) lse_merge(a[0], a[j].m, a[j].s, a[j].u);
  return a[0];
}
}  // namespace

__global__ void __launch_bounds__(kCombTok * kCombGroups)
combine_kernel(const float* __restrict__ pm, const float* __restrict__ ps,
               const float* __restrict__ pu, const float* __restrict__ zt, int n_tiles,
               long long stride, const int* __restrict__ pack_of, const uint8_t* __restrict__ mask,
               long long T, float* __restrict__ logprob, float* __restrict__ entropy,
               float* __restrict__ lse) {
  __shared__ Lse3 st[kCombGroups][kCombTok];
  const int x = threadIdx.x % kCombTok, g = threadIdx.x / kCombTok;
  for (long long t0 = static_cast<long long>(blockIdx.x) * kCombTok; t0 < T;
       t0 += static_cast<long long>(gridDim.x) * kCombTok) {
    const long long t = t0 + x;
    int r = -1;
    if (t < T) {
      r = pack_of[t];
      if (r >= 0 && mask[t] == 0) r = -1;
    }
    Lse3 a{0.f, 0.f, 0.f};
    if (r >= 0) a = fold_tiles(pm, ps, pu, n_tiles, stride, r, g);
    st[g][x] = a;
    __syncthreads();
    if (g == 0 && t < T) {
      if (r < 0) {
        logprob[t] = 0.f;
        entropy[t] = 0.f;
        if (lse) lse[t] = 0.f;
      } else {
        Lse3 acc = st[0][x];
        for (int k = 1; k < kCombGroups; ++k) lse_merge(acc, st[k][x].m, st[k][x].s, st[k][x].u);
        const float logS = logf(acc.s);
        const float l = fmaf(acc.m, kLn2, logS);
        if (lse) lse[t] = l;
        entropy[t] = logS - (acc.u / acc.s) * kLn2;
        logprob[t] = zt[r] - l;
      }
    }
    __syncthreads();
  }
}

// Vocabulary-parallel forward, shard side: the same fold as combine_kernel,
// stopped before the logarithm.  stats[t] = (M, S, U, z_t) in base-2 units
// over this shard's columns, z_t the target logit when the target lies in the
// shard (else 0).  Inactive or unscheduled tokens get (0, 0, 0, 0).
__global__ void __launch_bounds__(kCombTok * kCombGroups)
combine_stats_kernel(const float* __restrict__ pm, const float* __restrict__ ps,
                     const float* __restrict__ pu, const float* __restrict__ zt, int n_tiles,
                     long long stride, const int* __restrict__ pack_of,
                     const uint8_t* __restrict__ mask, const int* __restrict__ targets, int t_off,
                     int v_shard, long long T, float4* __restrict__ stats) {
  __shared__ Lse3 st[kCombGroups][kCombTok];
  const int x = threadIdx.x % kCombTok, g = threadIdx.x / kCombTok;
  for (long long t0 = static_cast<long long>(blockIdx.x) * kCombTok; t0 < T;
       t0 += static_cast<long long>(gridDim.x) * kCombTok) {
    const long long t = t0 + x;
    int r = -1;
    if (t < T) {
      r = pack_of[t];
      if (r >= 0 && mask[t] == 0) r = -1;
    }
    Lse3 a{0.f, 0.f, 0.f};
    if (r >= 0) a = fold_tiles(pm, ps, pu, n_tiles, stride, r, g);
    st[g][x] = a;
    __syncthreads();
    if (g == 0 && t < T) {
      if (r < 0) {
        stats[t] = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        Lse3 acc = st[0][x];
        for (int k = 1; k < kCombGroups; ++k) lse_merge(acc, st[k][x].m, st[k][x].s, st[k][x].u);
        const int tl = targets[t] - t_off;
        const float z = (tl >= 0 && tl < v_shard) ? zt[r] : 0.f;
        stats[t] = make_float4(acc.m, acc.s, acc.u, z);
      }
    }
    __syncthreads();
  }
}

// Vocabulary-parallel forward, gather side: merges the statistics of
// n_shards shards in shard order (stats is [n_shards][T]) and finishes
// lse = M ln2 + log S, H = log S - (U / S) ln2, logp = z_t - lse, with z_t
// the sum of the shards' z slots (only the owning shard's is nonzero).
__global__ void __launch_bounds__(256)
combine_shards_kernel(const float4* __restrict__ stats, int n_shards, long long T,
                      const uint8_t* __restrict__ mask, float* __restrict__ logprob,
                      float* __restrict__ entropy, float* __restrict__ lse) {
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < T;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    if (mask[t] == 0) {
      logprob[t] = 0.f;
      entropy[t] = 0.f;
      if (lse) lse[t] = 0.f;
      continue;
    }
    Lse3 acc{0.f, 0.f, 0.f};
    float z = 0.f;
    for (int k = 0; k < n_shards; ++k) {
      const float4 v = stats[static_cast<long long>(k) * T + t];
      lse_merge(acc, v.x, v.y, v.z);
      z += v.w;
    }
    const float logS = logf(acc.s);
    const float l = fmaf(acc.m, kLn2, logS);
    if (lse) lse[t] = l;
    entropy[t] = logS - (acc.u / acc.s) * kLn2;
    logprob[t] = z - l;
  }
}

// Rows of dhidden that no GEMM tile writes (tokens outside the row schedule)
// are set to zero.  `vec_per_row` 16-byte vectors per row.
__global__ void __launch_bounds__(256)
zero_unpacked_rows_kernel(uint4* __restrict__ out, const int* __restrict__ pack_of, long long T,
                          long long vec_per_row) {
  for (long long t = blockIdx.x; t < T; t += gridDim.x) {
    if (pack_of[t] >= 0) continue;
    uint4* d = out + t * vec_per_row;
    for (long long i = threadIdx.x; i < vec_per_row; i += blockDim.x) d[i] = make_uint4(0, 0, 0, 0);
  }
}

// ------------------------------------------------------------ launchers --

cudaError_t launch_spans_build(const uint8_t* mask, long long T, int max_gap, int* spans,
                               long long cap, int* num_spans, DevStatus* st, cudaStream_t s) {
  spans_build_kernel<<<1, kScanThreads, 0, s>>>(mask, T, max_gap, spans, cap, num_spans, st);
  return cudaGetLastError();
}

long long rowmap_tiles(long long T) { return (T + kRmTile - 1) / kRmTile; }

cudaError_t launch_rowmap(const uint8_t* mask, const int* spans, const int* num_spans,
                          long long cap, long long T, int span_rows, const int* targets, int t_lo,
                          int t_hi, int* row_map, int* pack_of, long long* tile_rows,
                          Sched* sched, DevStatus* st, cudaStream_t s) {
  const long long n = rowmap_tiles(T);
  if (n <= 0) return cudaSuccess;
  if (n > 0x7fffffffLL) return cudaErrorInvalidValue;
  rowmap_count_kernel<<<static_cast<unsigned>(n), kRmThreads, 0, s>>>(
      mask, spans, num_spans, cap, T, span_rows, targets, t_lo, t_hi, tile_rows, sched, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  rowmap_write_kernel<<<static_cast<unsigned>(n), kRmThreads, 0, s>>>(
      mask, spans, num_spans, cap, T, span_rows, tile_rows, row_map, pack_of, sched);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void* src, void* dst, const int* row_map, const Sched* sched,
                               long long T_pad, long long row_bytes, int num_sms, cudaStream_t s) {
  if (T_pad == 0) return cudaSuccess;
  const long long grid = T_pad < 8LL * num_sms ? T_pad : 8LL * num_sms;
  gather_rows_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(
      static_cast<const uint4*>(src), static_cast<uint4*>(dst), row_map, sched, row_bytes / 16);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* pm, const float* ps, const float* pu, const float* zt,
                           int n_tiles, long long stride, const int* pack_of, const uint8_t* mask,
                           long long T, float* logprob, float* entropy, float* lse, int num_sms,
                           cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  long long grid = (T + kCombTok - 1) / kCombTok;
  if (grid > 32LL * num_sms) grid = 32LL * num_sms;
  combine_kernel<<<static_cast<unsigned>(grid), kCombTok * kCombGroups, 0, s>>>(pm, ps, pu, zt, n_tiles, stride,
                                                             pack_of, mask, T, logprob, entropy,
                                                             lse);
  return cudaGetLastError();
}

cudaError_t launch_combine_stats(const float* pm, const float* ps, const float* pu,
                                 const float* zt, int n_tiles, long long stride, const int* pack_of,
                                 const uint8_t* mask, const int* targets, int t_off, int v_shard,
                                 long long T, float4* stats, int num_sms, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  long long grid = (T + kCombTok - 1) / kCombTok;
  if (grid > 32LL * num_sms) grid = 32LL * num_sms;
  combine_stats_kernel<<<static_cast<unsigned>(grid), kCombTok * kCombGroups, 0, s>>>(
      pm, ps, pu, zt, n_tiles, stride, pack_of, mask, targets, t_off, v_shard, T, stats);
  return cudaGetLastError();
}

cudaError_t launch_combine_shards(const float4* stats, int n_shards, long long T,
                                  const uint8_t* mask, float* logprob, float* entropy, float* lse,
                                  int num_sms, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  long long grid = (T + 255) / 256;
  if (grid > 16LL * num_sms) grid = 16LL * num_sms;
  combine_shards_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(stats, n_shards, T, mask,
                                                                    logprob, entropy, lse);
  return cudaGetLastError();
}

cudaError_t launch_zero_unpacked_rows(void* out, const int* pack_of, long long T,
                                      long long row_bytes, int num_sms, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const long long grid = T < 8LL * num_sms ? T : 8LL * num_sms;
  zero_unpacked_rows_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(
      static_cast<uint4*>(out), pack_of, T, row_bytes / 16);
  return cudaGetLastError();
}

}  // namespace eas

namespace eas {

// Failure-detection self-test: one warp waits on an mbarrier that nothing
// arrives on, once with the CTA-scope wait and once with the cluster-scope
// wait the GEMM kernel uses.  Each bounded wait runs out after `budget`
// clocks and reports kStTimeout (where = 90 / 91) instead of hanging.
__global__ void selftest_wait_kernel(long long budget, DevStatus* st) {
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait(&bar[0], 0, &abort_flag, budget)) report(st, kStTimeout, 90, 0);
    abort_flag = 0;
    long long t0 = clock64();
    bool done = false;
    while (!done && clock64() - t0 <= budget) {
      uint32_t ok;
      asm volatile(
          "{\n\t.reg .pred p;\n\t"
          "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
          "selp.u32 %0, 1, 0, p;\n\t}"
          : "=r"(ok)
          : "r"(smem_u32(&bar[1])), "r"(0)
          : "memory");
      done = ok != 0;
    }
    if (!done) report(st, kStTimeout, 91, 0);
    // complete both phases so that nothing is left pending at exit
    mbar_arrive(&bar[0]);
    mbar_arrive(&bar[1]);
  }
}

cudaError_t launch_selftest_wait(long long budget, DevStatus* st, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(budget, st);
  return cudaGetLastError();
}

}  // namespace eas

namespace eas {

// Context-parallel token layout ("How it works": forward mask and spans come
// from a CP-aware packed layout; diagram: "CP-local ordered spans").  Every
// packed segment [offs[k], offs[k+1]) has a length that is a multiple of 2*cp
// and is cut into 2*cp equal chunks; rank `rank` holds chunk `rank` then chunk
// 2*cp-1-rank of each segment, segments in order.  For each local token i:
//   l2g[i] = its global token index, local_mask[i] = mask[l2g[i]].
// Offsets that are not a valid layout report kStInvalidLayout; every access
// stays in bounds regardless.
__global__ void __launch_bounds__(256)
cp_local_kernel(const uint8_t* __restrict__ mask, const int* __restrict__ offs, int n_segs,
                long long T, int cp, int rank, uint8_t* __restrict__ local_mask,
                int* __restrict__ l2g, DevStatus* st) {
  const long long n_local = T / cp;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long tid = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  for (long long k = tid; k < n_segs; k += stride) {
    const long long L = static_cast<long long>(offs[k + 1]) - offs[k];
    if (L < 0 || L % (2LL * cp) != 0) report(st, kStInvalidLayout, 95, static_cast<int>(k));
  }
  if (tid == 0 && (offs[0] != 0 || static_cast<long long>(offs[n_segs]) != T))
    report(st, kStInvalidLayout, 96, -1);
  for (long long i = tid; i < n_local; i += stride) {
    int lo = 0, hi = n_segs;              // largest k with offs[k] / cp <= i
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (static_cast<long long>(offs[mid]) / cp <= i) lo = mid; else hi = mid;
    }
    const long long s0 = offs[lo];
    const long long c = (static_cast<long long>(offs[lo + 1]) - s0) / (2LL * cp);
    const long long p = i - s0 / cp;
    const long long g = (p < c) ? s0 + rank * c + p : s0 + (2LL * cp - 1 - rank) * c + (p - c);
    if (g >= 0 && g < T) {
      l2g[i] = static_cast<int>(g);
      local_mask[i] = mask[g];
    } else {
      l2g[i] = -1;
      local_mask[i] = 0;
      report(st, kStInvalidLayout, 97, static_cast<int>(i));
    }
  }
}

cudaError_t launch_cp_local(const uint8_t* mask, const int* offs, int n_segs, long long T, int cp,
                            int rank, uint8_t* local_mask, int* l2g, DevStatus* st, int num_sms,
                            cudaStream_t s) {
  const long long work = T / cp > n_segs ? T / cp : n_segs;
  long long grid = (work + 255) / 256;
  if (grid < 1) grid = 1;
  if (grid > 8LL * num_sms) grid = 8LL * num_sms;
  cp_local_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(mask, offs, n_segs, T, cp, rank,
                                                              local_mask, l2g, st);
  return cudaGetLastError();
}

}  // namespace eas
