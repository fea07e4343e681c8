// Tensor-core (tcgen05) GEMMs of the block-sparse fused LM-head, bf16 inputs,
// fp32 accumulation in TMEM, operands fed by TMA from HBM.
//
// One persistent, warp-specialised kernel serves the four contractions of the
// path ("perf(megatron): add block-sparse fused LM-head backward", SkyRL PR
// #2376, "What does this PR do?" / "How it works" / diagram):
//
//   kind        A (M x K)                 B (N x K)               epilogue
//   kTcFwd      Hp [R, H]   K-major       W [V, H]    K-major     online softmax partials
//   kTcDLogits  Hp [R, H]   K-major       W_c         K-major     d-logits -> bf16 staging
//   kTcDHidden  dZ_c [R,Vc] K-major       W_c [Vc, H] MN-major    fp32 accumulate / dhidden
//   kTcDWeight  dZ_c^T      MN-major      Hp [R, H]   MN-major    dW rows (fp32)
//
// Hp is the row-packed copy of hidden (rows of the ordered spans), so every M
// tile is dense; tile counts come from live extents only (greptile "Wide-tail
// grid exceeds live split": programs must not outrun the live split width).
//
// A launch carries up to kMaxTcJobs independent jobs (e.g. dW and dHidden of
// chunk c next to the d-logits of chunk c+1).  Their tiles form one list that
// the CTA pairs draw from through a global atomic counter, so a pair that
// finishes early takes more work and the jobs fill each other's tails.
//
// A cluster of two CTAs (the two SMs of a TPC) computes each tile with
// tcgen05.mma.cta_group::2: CTA r loads A rows [128r, 128r+128) and, of every
// 256-column block of B, columns [128r, 128r+128).  The forward and the e4m3
// kinds compute 256 x 256 tiles: the bf16 forward in seven 32 KB stages of
// K = 64, the e4m3 ones in three 64 KB stages of two k-blocks; each CTA's
// TMEM holds two 128 x 256 fp32 accumulators (all 512 columns), so the
// epilogue of tile i overlaps the mainloop of tile i+1.  The bf16 backward
// computes 256 x 512 tiles as two staggered 256-column halves in TMEM columns
// [0, 256) and [256, 512), fed by four 48 KB stages that share each A k-block
// between the halves (see PipeGeo); its epilogues stage their output in the
// remaining 32 KB and write it with TMA.  A K-major operand comes in one 2-D
// TMA box per k-block, an MN-major one (dHidden's B, dW's A and B) in one 3-D
// box {64 columns, 64 k-rows, 2 column blocks}.  When the last m-tile of a
// job over the packed rows holds at most 128 real rows, the bf16 backward
// (d-logits, dHidden) computes it as a 128-row pair MMA (64 rows per CTA,
// half the tensor time) instead of carrying the padding rows through the
// tensor pipe; its results are bit-identical to those of a full tile.  CTA
// layout (192 threads): warp 0 = TMA producer (lane 0; on the even CTA it also
// fetches tile indices and publishes them to both CTAs), warp 1 = MMA issuer
// (lane 0 of the even CTA) and TMEM owner, warps 2..5 = epilogue, one
// accumulator row per thread (warp w reads TMEM lanes 32*(w%4) .. +31).  Every
// mbarrier wait is bounded; on expiry a CTA raises its abort flag, lets its
// in-flight copies and MMAs land, frees TMEM and reports kStTimeout in the
// status word.
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "eas_device.cuh"
#include "eas_kernels.h"

namespace eas {

namespace {

constexpr int kRing = 4;                      // tile indices in flight
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;

struct TileCoord {
  int m, n;
};

// Band raster: group_m consecutive m-tiles sweep all n-tiles together, so the
// B tiles they share stay in L2 while the A band is reused across n.
__device__ __forceinline__ TileCoord raster(int t, int num_m, int num_n, int group_m) {
  const int band_tiles = group_m * num_n;
  const int band = t / band_tiles;
  const int m_first = band * group_m;
  int gm = num_m - m_first;
  if (gm > group_m) gm = group_m;
  const int in = t - band * band_tiles;
  TileCoord c;
  c.m = m_first + in % gm;
  c.n = in / gm;
  return c;
}

// Per-job extents, identical in every thread.
struct JobShape {
  int num_m, num_n, num_kb, tiles, first;
  int num_nb;      // 256-column blocks of N (a wide tile's half h is block 2n + h)
};

struct Work {
  int job;
  TileCoord tc;
};

__device__ __forceinline__ Work locate(int t, const JobShape (&js)[kMaxTcJobs], int n_jobs,
                                       const TcArgs& a) {
  int j = 0;
  while (j + 1 < n_jobs && t >= js[j + 1].first) ++j;
  Work w;
  w.job = j;
  w.tc = raster(t - js[j].first, js[j].num_m, js[j].num_n, a.jobs[j].group_m > 0 ? a.jobs[j].group_m : 1);
  return w;
}

// ------------------------------------------------------------ epilogues --

// Forward: per-row online softmax statistics over the tile's valid columns,
// in base-2 units (y = z log2 e): m = max y, s = sum 2^(y-m), u = sum
// 2^(y-m)(y-m); plus the target logit when the target falls in this tile.
template <bool kScaled>
__device__ __forceinline__ void epi_fwd(const TcArgs& a, uint32_t tbase, bool k_empty,
                                        long long r0, int n_blk, int row, int tgt,
                                        float rscale, const float* __restrict__ wscale) {
  const int n0 = n_blk * kTcBN;
  int valid = a.V - n0;
  if (valid > kTcBN) valid = kTcBN;
  float m2 = -INFINITY, s = 0.f, u2 = 0.f;
  float ztv = 0.f;
  bool found = false;
#pragma unroll 1
  for (int c = 0; c < kTcBN / 32; ++c) {
    if (c * 32 >= valid) break;
    float v[32];
    if (k_empty) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0.f;
    } else {
      tmem_ld32(tbase + c * 32, v);
    }
    const int cvalid = valid - c * 32;   // > 0
    if constexpr (kScaled) {
      // e4m3 operands: z = acc * scale(row) * scale(column)
      const float* wsc = wscale + n0 + c * 32;
      if (cvalid >= 32 && (reinterpret_cast<uintptr_t>(wsc) & 15u) == 0) {
        // the 32 column scales as eight 16-byte loads (one line, shared by
        // every lane of the warp)
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 w4 = __ldg(reinterpret_cast<const float4*>(wsc) + q);
          v[4 * q] *= rscale * w4.x;
          v[4 * q + 1] *= rscale * w4.y;
          v[4 * q + 2] *= rscale * w4.z;
          v[4 * q + 3] *= rscale * w4.w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= rscale * (j < cvalid ? __ldg(wsc + j) : 0.f);
      }
    }
    const int tj = tgt - (n0 + c * 32);
    if (static_cast<unsigned>(tj) < static_cast<unsigned>(cvalid < 32 ? cvalid : 32)) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j == tj) ztv = v[j];
      found = true;
    }
    float cmax = -INFINITY;
    if (cvalid >= 32) {
#pragma unroll
      for (int j = 0; j < 32; ++j) cmax = fmaxf(cmax, v[j]);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < cvalid) cmax = fmaxf(cmax, v[j]);
    }
    const float mnew = fmaxf(m2, cmax * kLog2e);
    if (s == 0.f) {
      m2 = mnew;
    } else if (mnew > m2) {
      const float d = m2 - mnew;
      const float f = ex2_approx(d);
      u2 = f * (u2 + d * s);
      s *= f;
      m2 = mnew;
    }
    if (cvalid >= 32) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float d = fmaf(v[j], kLog2e, -m2);
        const float e = ex2_approx(d);
        s += e;
        u2 = fmaf(e, d, u2);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (j < cvalid) {
          const float d = fmaf(v[j], kLog2e, -m2);
          const float e = ex2_approx(d);
          s += e;
          u2 = fmaf(e, d, u2);
        }
      }
    }
  }
  const long long r = r0 + row;
  const long long o = static_cast<long long>(n_blk) * a.part_stride + r;
  a.part_m[o] = m2;
  a.part_s[o] = s;
  a.part_u[o] = u2;
  if (found) a.zt[r] = ztv;
}

struct RowScalars {
  float lse2;    // lse * log2 e
  float gh2;     // g_H * ln 2
  float c1;      // g_lp + g_H * H
  float glp;
  int tgt;       // chunk-local target column, or -1 outside the chunk
  bool active;
  float hs;      // e4m3 d-logits: scale of the row's quantised hidden
};

// TMA store of a shared-memory box to the map's coordinates (c0, c1), as one
// bulk async-group of the issuing thread.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* smem_src, int c0,
                                             int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(smem_src)), "r"(c0), "r"(c1)
      : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, const void* smem_src,
                                                  int c0, int c1) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(smem_src)), "r"(c0), "r"(c1)
      : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d_pair_hint(void* smem_dst, const CUtensorMap* map,
                                                      uint32_t bar, int c0, int c1,
                                                      uint64_t policy);
// Coalesced row stores.  tcgen05.ld (32x32b) hands each lane one row of the
// tile, so a lane storing its own row would touch 32 rows (32 memory lines)
// per warp store.  octet_transpose regroups a chunk across each group of 8
// lanes: on entry lane i of an octet holds 16-byte blocks b = 0..7 of its own
// row (x[4b .. 4b+3]); on exit it holds block i of the octet's rows p = 0..7
// (x[4p .. 4p+3]), so every store instruction writes 4 rows x 128 contiguous
// bytes.  Three butterfly stages (lane xor 1, 2, 4) each swap half the blocks.
template <typename T>
__device__ __forceinline__ void octet_transpose(T (&x)[32], int i) {
#pragma unroll
  for (int s = 1; s < 8; s <<= 1) {
    const bool hi = (i & s) != 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      if (b & s) continue;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const T send = hi ? x[4 * b + w] : x[4 * (b | s) + w];
        const T recv = __shfl_xor_sync(0xffffffffu, send, s);
        if (hi) x[4 * b + w] = recv;
        else x[4 * (b | s) + w] = recv;
      }
    }
  }
}

// d-logits of 32 columns of one row, packed to bf16 pairs: dZ = g_lp (onehot
// - p) - g_H p (z - lse + H), p = exp(z - lse), written as -p (g_H (z - lse)
// + g_lp + g_H H) + g_lp onehot.  Inactive rows and columns past the live
// width are exact zeros.
template <bool kScaled>
__device__ __forceinline__ void dlogits_chunk(const TcJob& jb, uint32_t taddr, bool k_empty,
                                              int col0, const RowScalars& rs, uint32_t* pk,
                                              const float* __restrict__ wsc) {
  // tcgen05.ld is warp-collective: only warp-uniform conditions (live width,
  // empty K) may skip it; per-row activity is applied afterwards.
  if (col0 >= jb.vc_live) {
#pragma unroll
    for (int j = 0; j < 16; ++j) pk[j] = 0u;
    return;
  }
  float v[32];
  if (k_empty) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = 0.f;
  } else {
    tmem_ld32(taddr, v);
  }
  if (!rs.active) {
#pragma unroll
    for (int j = 0; j < 16; ++j) pk[j] = 0u;
    return;
  }
  const int cvalid = jb.vc_live - col0;
  const int tj = rs.tgt - col0;
  if constexpr (kScaled) {
    // e4m3 operands: z = acc * scale(row) * scale(vocabulary row); wsc points
    // at the scale of this chunk's column col0
    if (cvalid >= 32 && (reinterpret_cast<uintptr_t>(wsc) & 15u) == 0) {
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        const float4 w4 = __ldg(reinterpret_cast<const float4*>(wsc) + q4);
        v[4 * q4] *= rs.hs * w4.x;
        v[4 * q4 + 1] *= rs.hs * w4.y;
        v[4 * q4 + 2] *= rs.hs * w4.z;
        v[4 * q4 + 3] *= rs.hs * w4.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= rs.hs * (j < cvalid ? __ldg(wsc + j) : 0.f);
    }
  }
  float d[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float x2 = fmaf(v[j], kLog2e, -rs.lse2);    // (z - lse) log2 e
    const float p = ex2_approx(x2);
    const float w = fmaf(rs.gh2, x2, rs.c1);           // g_H (z - lse) + g_lp + g_H H
    d[j] = -p * w;
  }
  // the target column and the live-width edge fall in few chunks: branch
  // around them instead of selecting on every element
  if (static_cast<unsigned>(tj) < 32u) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j == tj) d[j] += rs.glp;
  }
  if (cvalid < 32) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j >= cvalid) d[j] = 0.f;
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(d[2 * j], d[2 * j + 1]);
}

// d-logits tile rows into the bf16 staging buffer, 64 columns (128 bytes of a
// row) per round: the warp's 32 rows go to a 4 KB shared-memory box in the
// 128-byte swizzled layout (16-byte chunk j of row l at chunk j ^ (l & 7)),
// and lane 0 writes the box with a TMA store.  Two boxes per warp (q = warp
// quadrant) alternate; `cnt` counts the warp's boxes so far.  The warp covers
// tile columns [c0, c0 + ncol) of rows r0 + (row & ~31) .. + 31.
template <bool kScaled>
__device__ __forceinline__ void epi_dlogits(const TcJob& jb, uint32_t tbase, bool k_empty,
                                            long long r0, int n_blk, int q, int row, int c0,
                                            int ncol, const RowScalars& rs, uint8_t* sEpi,
                                            uint32_t& cnt, const float* __restrict__ wscale) {
  const int n0 = n_blk * kTcBN + c0;
  const int lane = row & 31;
#pragma unroll 1
  for (int c = 0; c < ncol / 64; ++c) {
    uint32_t pk[32];
    const float* wsc = kScaled ? wscale + jb.v0 + n0 + c * 64 : nullptr;
    dlogits_chunk<kScaled>(jb, tbase + c * 64, k_empty, n0 + c * 64, rs, pk, wsc);
    dlogits_chunk<kScaled>(jb, tbase + c * 64 + 32, k_empty, n0 + c * 64 + 32, rs, pk + 16,
                           kScaled ? wsc + 32 : nullptr);
    uint8_t* box = sEpi + ((cnt & 1u) * 4 + q) * 4096;
    if (lane == 0) bulk_wait_read<1>();     // the box's previous store has read it
    __syncwarp();
    uint8_t* rowp = box + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<uint4*>(rowp + ((j ^ (lane & 7)) << 4)) =
          make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tma_store_2d(&jb.tmD, box, n0 + c * 64, static_cast<int>(r0) + (row & ~31));
    ++cnt;
  }
}

// dHidden of a chunk before the last: the warp's 32 rows x 32 columns of fp32
// go to a 4 KB shared-memory box (128-byte swizzled) and lane 0 adds the box
// into the fp32 accumulator [T_pad][H] with a TMA reduce-add (a TMA store on
// the first chunk), so the L2 does the read-modify-write.  Each accumulator
// element receives one add per launch, in chunk order across launches, so
// the sum is deterministic.
__device__ __forceinline__ void epi_dhidden_acc(const TcArgs& a, const TcJob& jb, uint32_t tbase,
                                                bool k_empty, long long r0, int n_blk, int q,
                                                int row, int c0, int ncol, uint8_t* sEpi,
                                                uint32_t& cnt) {
  const int n0 = n_blk * kTcBN + c0;
  const int lane = row & 31;
#pragma unroll 1
  for (int c = 0; c < ncol / 32; ++c) {
    if (n0 + c * 32 >= a.H) break;
    float v[32];
    if (k_empty) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0.f;
    } else {
      tmem_ld32(tbase + c * 32, v);
    }
    uint8_t* box = sEpi + ((cnt & 1u) * 4 + q) * 4096;
    if (lane == 0) bulk_wait_read<1>();
    __syncwarp();
    uint8_t* rowp = box + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<float4*>(rowp + ((j ^ (lane & 7)) << 4)) =
          make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      const int rr = static_cast<int>(r0) + (row & ~31);
      if (jb.first_chunk) tma_store_2d(&jb.tmD, box, n0 + c * 32, rr);
      else tma_reduce_add_2d(&jb.tmD, box, n0 + c * 32, rr);
    }
    ++cnt;
  }
}

// dHidden of the last chunk (or the only one): this chunk's product plus the
// accumulator (unless it is also the first chunk), converted to bf16 and
// scattered to the rows' tokens (zeros for gap rows whose mask byte is 0).
__device__ __forceinline__ void epi_dhidden_last(const TcArgs& a, const TcJob& jb, uint32_t tbase,
                                            bool k_empty, long long r0, int n_blk, int row, int c0,
                                            int ncol, int tok, bool active) {
  const int n0 = n_blk * kTcBN + c0;
  const int lane = row & 31;
  const int i = lane & 7;
  const long long r_oct = r0 + (row & ~31) + (lane & ~7);
  float* acc = a.acc + r_oct * a.H + n0;
  // token and activity of the octet's rows p = 0..7 (row p lives in lane
  // (lane & ~7) + p)
  int tok_p[8];
  uint32_t act_bits = 0;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    tok_p[p] = __shfl_sync(0xffffffffu, tok, (lane & ~7) + p);
    if (__shfl_sync(0xffffffffu, active ? 1 : 0, (lane & ~7) + p)) act_bits |= 1u << p;
  }
#pragma unroll 1
  for (int c = 0; c < ncol / 32; ++c) {
    if (n0 + c * 32 >= a.H) break;
    float v[32];
    if (k_empty) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0.f;
    } else {
      tmem_ld32(tbase + c * 32, v);
    }
    octet_transpose(v, i);
    if (!jb.first_chunk) {
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        const float4 x = reinterpret_cast<const float4*>(acc + p * a.H + c * 32)[i];
        v[4 * p] += x.x;
        v[4 * p + 1] += x.y;
        v[4 * p + 2] += x.z;
        v[4 * p + 3] += x.w;
      }
    }
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      if (tok_p[p] < 0) continue;
      const bool on = (act_bits >> p) & 1u;
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.dhidden) +
                         static_cast<long long>(tok_p[p]) * a.H + n0 + c * 32;
      reinterpret_cast<uint2*>(o)[i] =
          make_uint2(on ? pack_bf16x2(v[4 * p], v[4 * p + 1]) : 0u,
                     on ? pack_bf16x2(v[4 * p + 2], v[4 * p + 3]) : 0u);
    }
  }
}

// dW rows of this chunk: every vocabulary row of the chunk is overwritten.
__device__ __forceinline__ void epi_dweight(const TcArgs& a, const TcJob& jb, uint32_t tbase,
                                            bool k_empty, long long r0, int n_blk, int row) {
  const int n0 = n_blk * kTcBN;
  const int lane = row & 31;
  const int i = lane & 7;
  const int m_oct = static_cast<int>(r0) + (row & ~31) + (lane & ~7);   // chunk-local vocab row
  float* outp = a.dW + (static_cast<long long>(jb.v0) + m_oct) * a.H + n0;
#pragma unroll 1
  for (int c = 0; c < kTcBN / 32; ++c) {
    if (n0 + c * 32 >= a.H) break;
    float v[32];
    if (k_empty) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0.f;
    } else {
      tmem_ld32(tbase + c * 32, v);    // warp-collective: every lane loads
    }
    octet_transpose(v, i);
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      if (m_oct + p >= jb.vc_live) continue;
      reinterpret_cast<float4*>(outp + static_cast<long long>(p) * a.H + c * 32)[i] =
          make_float4(v[4 * p], v[4 * p + 1], v[4 * p + 2], v[4 * p + 3]);
    }
  }
}

// ----------------------------------------------------------------- kernel --

// =====================================================================
// The CTA-pair kernel.  Against one CTA per 128 x 256 tile, the pair halves
// the B bytes each SM moves from L2 and reads from shared memory per k-step.
//
// Synchronisation (each line: barrier, where it lives, who arrives):
//   full[s]   leader   leader producer's expect_tx (the stage's bytes of both
//                      CTAs) + both CTAs' TMA bytes
//   empty[s]  both     leader MMA commit, multicast to both CTAs
//   tfull[b]  both     leader MMA commit, multicast to both CTAs (b = the
//                      tile's parity for 256 x 256 tiles, the half of a wide
//                      tile)
//   tempty[b] leader   4 epilogue warps of each CTA (the peer's arrive remotely)
//   rfull[i]  both     leader fetcher (local arrive + remote arrive)
//   rempty[i] leader   leader MMA + 4 leader epilogue warps + peer producer
//                      + 4 peer epilogue warps
// =====================================================================

constexpr int kPHalf = 128;                       // rows (of A) / columns (of B) per CTA
constexpr int kPM = 256;                          // rows of a pair tile
constexpr int kPKBlockBytes = kPHalf * 128;       // one 128-byte-swizzled k-block: 16 KB

// Pipeline stage geometry of an instantiation.  A stage holds kSub k-blocks
// of each operand.  The backward keeps 32 KB for the epilogues' TMA staging
// (two 4 KB boxes per epilogue warp).  The e4m3 instantiations, whose MMAs
// finish a k-block in half the time, compute 256 x 256 tiles in three stages
// of two k-blocks (64 KB): half as many stage boundaries per unit of work.
//
// The bf16 backward instantiation computes 256 x 512 tiles ("wide"): a stage
// holds one k-block of A and of both 256-column halves of B (48 KB per CTA,
// four stages), and the two halves accumulate in TMEM columns [0, 256) and
// [256, 512).  A 256 x 256 tile needs 32 KB per CTA per 512-cycle k-block,
// 64 B per SM-clock, about what an SM takes in; sharing each A stage between
// two halves brings that to 24 KB per half-tile's k-block, and the operand
// traffic's power goes to the clock.  The halves run staggered: half 0 alone
// for its first kWideStagger k-blocks, then both, then half 1 alone for its
// first kWideStagger k-blocks.  Half 0's epilogue then runs under half 1's
// last k-blocks and half 1's under the next tile's first ones, as the two
// TMEM buffers of a 256 x 256 tile would.
constexpr int kWideStagger = 16;   // k-blocks each half of a wide tile runs alone

template <int kMode>
struct PipeGeo {
  static constexpr bool kWide = (kMode == 1);
  static constexpr int kTileN = kWide ? 2 * kTcBN : kTcBN;
  static constexpr int kSub = (kMode >= 2) ? 2 : 1;
  static constexpr int kStages = (kMode >= 2) ? 3 : kWide ? 4 : 7;
  static constexpr int kABytes = kSub * kPKBlockBytes;
  static constexpr int kBBytes = (kWide ? 2 : 1) * kSub * kPKBlockBytes;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kEpiBytes = (kMode == 1 || kMode == 3) ? 32768 : 0;
  // 128-row last m-tiles: the bf16 backward kinds (d-logits, dHidden)
  static constexpr bool kHalfTiles = (kMode == 1);
  static constexpr int kSmemBytes = kStages * kStageBytes + kEpiBytes + 1024 + 512;
};
// the backward's MN-major operands come in TMA boxes of one k-block's 64
// k-rows (the host builds those tensor maps)
static_assert(PipeGeo<1>::kSub == 1, "MN-major boxes span one k-block");

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared::cluster address of the same shared-memory location in CTA `rank`.
__device__ __forceinline__ uint32_t map_rank(const void* p, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
  return out;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cl(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait with cluster-scope acquire (for barriers other CTAs arrive on).
__device__ __forceinline__ bool mbar_wait_cl(uint64_t* bar, uint32_t parity, volatile int* abort,
                                             long long budget) {
  if (mbar_try_wait_cl(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > budget) {
      *abort = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// TMA load into this CTA's shared memory whose completion bytes are counted
// on a barrier of either CTA of the pair (`bar` is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map,
                                                 uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// 3-D TMA load: coordinates (c0, c1, c2) of the map's three dimensions.
__device__ __forceinline__ void tma_load_3d_pair(void* smem_dst, const CUtensorMap* map,
                                                 uint32_t bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// The same load with an L2 eviction-priority hint (a createpolicy policy).
// Only the bf16 forward uses it: its band of Hp rows is kept (evict-last)
// while W streams past (evict-first), which cut its DRAM bytes on long_256k
// from 181 to 155 GB and the step by 0.5 %.  The same hints on the backward
// jobs added DRAM traffic, since the streamed operand is shared by the band's
// tiles of one wave.
__device__ __forceinline__ void tma_load_2d_pair_hint(void* smem_dst, const CUtensorMap* map,
                                                      uint32_t bar, int c0, int c1,
                                                      uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

// e4m3 k-block: 128 one-byte elements per 128-byte swizzle row.
constexpr int kKbFp8 = 128;

// Instruction descriptor of kind::f8f6f4 with e4m3 A/B (format code 0), an
// fp32 accumulator, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_e4m3_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the barrier at `bar`'s offset in both CTAs of the pair when
// the pair MMAs issued so far complete.
__device__ __forceinline__ void umma_commit_pair_both(uint64_t* bar) {
  const uint16_t mask = 3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)), "h"(mask)
      : "memory");
}

__device__ __forceinline__ void umma_commit_pair_local(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// One instantiation per family of jobs, so that each carries only the code
// its jobs run (the kernel's size measurably costs throughput):
//   kMode 0: bf16 forward (kTcFwd), 3: e4m3 d-logits (kTcDLogitsFp8, the e4m3
//   backward's recompute), 1: bf16 backward (kTcDLogits, kTcDHidden,
//   kTcDWeight), 2: e4m3 forward (kTcFwdFp8).
template <int kMode>
__global__ void __launch_bounds__(kThreads, 1) tc_pair_kernel(const __grid_constant__ TcArgs a) {
  constexpr bool kFp8 = (kMode == 2 || kMode == 3);
  constexpr bool kFwd = (kMode == 0 || kMode == 2);
  using G = PipeGeo<kMode>;
  constexpr int kPStages = G::kStages;
  constexpr int kPABytes = G::kABytes;
  constexpr int kPBBytes = G::kBBytes;
  constexpr int kPStageBytes = G::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kPStages * kPABytes;
  uint8_t* sEpi = sB + kPStages * kPBBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sEpi + G::kEpiBytes);
  uint64_t* empty = full + kPStages;
  uint64_t* tfull = empty + kPStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* rfull = tempty + 2;
  uint64_t* rempty = rfull + kRing;
  uint64_t* drain = rempty + kRing;
  int* ring = reinterpret_cast<int*>(drain + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ring + kRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = (rank == 0);
  const Sched* sched = static_cast<const Sched*>(a.sched);
  DevStatus* st = static_cast<DevStatus*>(a.status);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 8);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&rfull[i], 1);
      mbar_init(&rempty[i], 10);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    for (int j = 0; j < a.n_jobs; ++j) {
      tma_prefetch_desc(&a.jobs[j].tmA);
      tma_prefetch_desc(&a.jobs[j].tmB);
    }
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync_all();     // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Launched with programmatic stream serialisation, the prologue above may
  // run while the previous kernel of the stream finishes; nothing it touched
  // is that kernel's output.  Every read of global memory comes after this
  // wait, which returns once the previous grid has completed and its writes
  // are visible (and at once for a launch without the attribute).  Dependents
  // are then released: their CTAs find a free SM only when a CTA of this grid
  // exits (one CTA per SM), and wait here in turn.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  JobShape js[kMaxTcJobs];
  int total = 0;
#pragma unroll
  for (int j = 0; j < kMaxTcJobs; ++j) {
    js[j] = JobShape{0, 0, 0, 0, total, 0};
    if (j < a.n_jobs) {
      const TcJob& jb = a.jobs[j];
      const int M = jb.M_fixed > 0 ? jb.M_fixed : sched->R_pad;
      // a reduction over packed rows (dW) stops at the last k-block holding a
      // real row; rows from R to R_pad are zero in both operands
      const int K = jb.K_fixed > 0 ? jb.K_fixed : sched->R;
      js[j].num_m = (M + kPM - 1) / kPM;
      js[j].num_n = (jb.N + G::kTileN - 1) / G::kTileN;
      js[j].num_nb = (jb.N + kTcBN - 1) / kTcBN;
      constexpr int kse = G::kSub * (kFp8 ? kKbFp8 : kTcBK);   // K per stage
      js[j].num_kb = (K + kse - 1) / kse;
      js[j].tiles = js[j].num_m * js[j].num_n;
      total += js[j].tiles;
    }
  }
  // The last m-tile of the jobs over the packed rows (M = R_pad) holds at most
  // 128 real rows: the backward instantiation runs it as a 128-row tile.
  bool last_half = false;
  if constexpr (G::kHalfTiles) {
    const int last = sched->R - (sched->R_pad / kPM - 1) * kPM;
    last_half = last > 0 && last <= kPHalf;
  }

  // shared::cluster addresses of the leader's barriers and the peer's ring
  const uint32_t full_leader0 = map_rank(&full[0], 0);
  const uint32_t tempty_leader0 = map_rank(&tempty[0], 0);
  const uint32_t rempty_leader0 = map_rank(&rempty[0], 0);
  const uint32_t ring_peer0 = map_rank(&ring[0], 1);
  const uint32_t rfull_peer0 = map_rank(&rfull[0], 1);

  if (warp == 0) {
    // ------------------------------------------------ fetcher (leader) + TMA producer (both)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int slot = it % kRing;
        const uint32_t rph = (it / kRing) & 1;
        int t;
        if (leader) {
          if (!mbar_wait_cl(&rempty[slot], rph ^ 1u, abort_flag, a.budget)) {
            report(st, kStTimeout, 11, it);
            ok = false;
            break;
          }
          const int got = atomicAdd(a.tile_counter, 1);
          t = (got < total) ? got : -1;
          ring[slot] = t;
          st_cluster_u32(ring_peer0 + 4 * slot, static_cast<uint32_t>(t));
          mbar_arrive(&rfull[slot]);
          mbar_arrive_cluster(rfull_peer0 + 8 * slot);
        } else {
          if (!mbar_wait_cl(&rfull[slot], rph, abort_flag, a.budget)) {
            report(st, kStTimeout, 12, it);
            ok = false;
            break;
          }
          t = ring[slot];
          mbar_arrive_cluster(rempty_leader0 + 8 * slot);
        }
        if (t < 0) break;
        const Work w = locate(t, js, a.n_jobs, a);
        const TcJob& jb = a.jobs[w.job];
        const int kind = jb.kind;
        // a 128-row tile: each CTA's A operand is 64 rows (the box still
        // loads 128, of which the MMA reads the first 64)
        const bool half = last_half && a.jobs[w.job].M_fixed <= 0 && w.tc.m == js[w.job].num_m - 1;
        const int mrow = w.tc.m * kPM + static_cast<int>(rank) * (half ? kPHalf / 2 : kPHalf);
        if constexpr (G::kWide) {
          // k-steps of a wide tile: half 0 alone for k-blocks [0, jst), both
          // halves for [jst, Kb), half 1 alone for [0, jst); a tile whose
          // second half lies past N runs half 0 only
          const int Kb = js[w.job].num_kb;
          const bool has1 = 2 * w.tc.n + 1 < js[w.job].num_nb;
          const int jst = Kb < kWideStagger ? Kb : kWideStagger;
          const int S = has1 ? Kb + jst : Kb;
          const int ncol0 = w.tc.n * G::kTileN + static_cast<int>(rank) * kPHalf;
          for (int sidx = 0; sidx < S; ++sidx) {
            const int kb = sidx < Kb ? sidx : sidx - Kb;
            const uint32_t hm = !has1 ? 1u : (sidx < jst ? 1u : (sidx < Kb ? 3u : 2u));
            if (!mbar_wait_cl(&empty[stage], phase ^ 1u, abort_flag, a.budget)) {
              report(st, kStTimeout, 13, t);
              ok = false;
              break;
            }
            uint8_t* dA = sA + stage * kPABytes;
            uint8_t* dB = sB + stage * kPBBytes;
            const uint32_t bar = full_leader0 + 8 * stage;
            const uint32_t nbh = (hm == 3u) ? 2u : 1u;
            if (leader)
              mbar_arrive_expect_tx(&full[stage], 2u * (kPABytes + nbh * kPKBlockBytes));
            const int k0 = kb * kTcBK;
            if (kind == kTcDLogits) {
              tma_load_2d_pair(dA, &jb.tmA, bar, k0, mrow);
#pragma unroll
              for (int h = 0; h < 2; ++h)
                if ((hm >> h) & 1u)
                  tma_load_2d_pair(dB + h * kPKBlockBytes, &jb.tmB, bar, k0,
                                   jb.v0 + ncol0 + h * kTcBN);
            } else if (kind == kTcDHidden) {
              tma_load_2d_pair(dA, &jb.tmA, bar, k0, mrow);
#pragma unroll
              for (int h = 0; h < 2; ++h)
                if ((hm >> h) & 1u)
                  tma_load_3d_pair(dB + h * kPKBlockBytes, &jb.tmB, bar, 0, jb.v0 + k0,
                                   (ncol0 + h * kTcBN) >> 6);
            } else {
              tma_load_3d_pair(dA, &jb.tmA, bar, 0, k0, mrow >> 6);
#pragma unroll
              for (int h = 0; h < 2; ++h)
                if ((hm >> h) & 1u)
                  tma_load_3d_pair(dB + h * kPKBlockBytes, &jb.tmB, bar, 0, k0,
                                   (ncol0 + h * kTcBN) >> 6);
            }
            if (++stage == kPStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        } else {
          const int ncol = w.tc.n * kTcBN + static_cast<int>(rank) * kPHalf; // this CTA's B columns
          for (int kb = 0; kb < js[w.job].num_kb; ++kb) {
            if (!mbar_wait_cl(&empty[stage], phase ^ 1u, abort_flag, a.budget)) {
              report(st, kStTimeout, 13, t);
              ok = false;
              break;
            }
            uint8_t* dA = sA + stage * kPABytes;
            uint8_t* dB = sB + stage * kPBBytes;
            const uint32_t bar = full_leader0 + 8 * stage;
            if (leader) mbar_arrive_expect_tx(&full[stage], 2 * kPStageBytes);
            constexpr int kblk = kFp8 ? kKbFp8 : kTcBK;      // K of one k-block
            const int k0 = kb * G::kSub * kblk;
            if constexpr (kFwd && !kFp8) {
              uint64_t keep, stream;
              asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
              asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(stream));
              tma_load_2d_pair_hint(dA, &jb.tmA, bar, k0, mrow, keep);
              tma_load_2d_pair_hint(dB, &jb.tmB, bar, k0, jb.v0 + ncol, stream);
            } else if (kFwd || kMode == 3 || kind == kTcDLogits) {
#pragma unroll
              for (int sb = 0; sb < G::kSub; ++sb) {
                tma_load_2d_pair(dA + sb * kPKBlockBytes, &jb.tmA, bar, k0 + sb * kblk, mrow);
                tma_load_2d_pair(dB + sb * kPKBlockBytes, &jb.tmB, bar, k0 + sb * kblk,
                                 jb.v0 + ncol);
              }
            } else if (kind == kTcDHidden) {
              tma_load_2d_pair(dA, &jb.tmA, bar, k0, mrow);
              tma_load_3d_pair(dB, &jb.tmB, bar, 0, jb.v0 + k0, ncol >> 6);
            } else {
              tma_load_3d_pair(dA, &jb.tmA, bar, 0, k0, mrow >> 6);
              tma_load_3d_pair(dB, &jb.tmB, bar, 0, k0, ncol >> 6);
            }
            if (++stage == kPStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok && leader) {
        for (int s2 = 0; s2 < kPStages; ++s2) {
          const uint32_t par = (s2 < stage) ? phase : (phase ^ 1u);
          long long t0 = clock64();
          while (!mbar_try_wait_cl(&full[s2], par) && clock64() - t0 < a.budget) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (leader only)
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int it = 0;; ++it) {
        const int slot = it % kRing;
        if (!mbar_wait_cl(&rfull[slot], (it / kRing) & 1, abort_flag, a.budget)) {
          report(st, kStTimeout, 14, it);
          break;
        }
        const int t = ring[slot];
        mbar_arrive(&rempty[slot]);
        if (t < 0) break;
        const Work w = locate(t, js, a.n_jobs, a);
        const int kind = a.jobs[w.job].kind;
        const bool a_mn = (kMode == 1) && (kind == kTcDWeight);
        const bool b_mn = (kMode == 1) && (kind == kTcDHidden || kind == kTcDWeight);
        const bool half = last_half && a.jobs[w.job].M_fixed <= 0 && w.tc.m == js[w.job].num_m - 1;
        const int mm = half ? kPHalf : kPM;
        const uint32_t idesc = kFp8 ? idesc_e4m3_f32(kPM, kTcBN)
                                    : a_mn ? idesc_bf16_f32(kPM, kTcBN, true, true)
                                    : (b_mn ? idesc_bf16_f32(mm, kTcBN, false, true)
                                            : idesc_bf16_f32(mm, kTcBN, false, false));
        const uint32_t a_lbo = a_mn ? 8192 : 16, a_step = a_mn ? 2048 : 32;
        const uint32_t b_lbo = b_mn ? 8192 : 16, b_step = b_mn ? 2048 : 32;
        if constexpr (G::kWide) {
          // TMEM half h of a tile: its epilogue's arrival on tempty[h] frees it
          // for the next tile (one phase per tile), its last MMA's commit on
          // tfull[h] hands it to the epilogue
          const int Kb = js[w.job].num_kb;
          const bool has1 = 2 * w.tc.n + 1 < js[w.job].num_nb;
          const int jst = Kb < kWideStagger ? Kb : kWideStagger;
          const int S = has1 ? Kb + jst : Kb;
          const uint32_t tph = it & 1;
          if (!mbar_wait_cl(&tempty[0], tph ^ 1u, abort_flag, a.budget)) {
            report(st, kStTimeout, 15, t);
            break;
          }
          tc_fence_after();
          bool ok = true;
          for (int sidx = 0; sidx < S; ++sidx) {
            const uint32_t hm = !has1 ? 1u : (sidx < jst ? 1u : (sidx < Kb ? 3u : 2u));
            if (has1 && sidx == jst) {
              if (!mbar_wait_cl(&tempty[1], tph ^ 1u, abort_flag, a.budget)) {
                report(st, kStTimeout, 15, t);
                ok = false;
                break;
              }
              tc_fence_after();
            }
            if (!mbar_wait_cl(&full[stage], phase, abort_flag, a.budget)) {
              report(st, kStTimeout, 16, t);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(sA + stage * kPABytes);
            const uint32_t b_addr = smem_u32(sB + stage * kPBBytes);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (!((hm >> h) & 1u)) continue;
              const bool first = (h == 0) ? (sidx == 0) : (sidx == jst);
              const uint32_t d_tmem = tmem_base + h * kTcBN;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t adesc = sdesc_sw128(a_addr + k * a_step, a_lbo, 1024);
                const uint64_t bdesc =
                    sdesc_sw128(b_addr + h * kPKBlockBytes + k * b_step, b_lbo, 1024);
                umma_bf16_pair(d_tmem, adesc, bdesc, idesc, (first && k == 0) ? 0u : 1u);
              }
            }
            umma_commit_pair_both(&empty[stage]);
            if (sidx == Kb - 1) umma_commit_pair_both(&tfull[0]);
            if (has1 && sidx == S - 1) umma_commit_pair_both(&tfull[1]);
            if (++stage == kPStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          if (Kb == 0) {
            mbar_arrive(&tfull[0]);
            mbar_arrive_cluster(map_rank(&tfull[0], 1));
          }
          if (Kb == 0 || !has1) {
            // nothing accumulates in half 1: hand it over once its previous
            // tile's epilogue has released it, keeping one phase per tile
            if (!mbar_wait_cl(&tempty[1], tph ^ 1u, abort_flag, a.budget)) {
              report(st, kStTimeout, 15, t);
              break;
            }
            mbar_arrive(&tfull[1]);
            mbar_arrive_cluster(map_rank(&tfull[1], 1));
          }
        } else {
          const int buf = it & 1;
          const uint32_t tph = (it >> 1) & 1;
          if (!mbar_wait_cl(&tempty[buf], tph ^ 1u, abort_flag, a.budget)) {
            report(st, kStTimeout, 15, t);
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * kTcBN;
          const int num_kb = js[w.job].num_kb;
          bool ok = true;
          for (int kb = 0; kb < num_kb; ++kb) {
            if (!mbar_wait_cl(&full[stage], phase, abort_flag, a.budget)) {
              report(st, kStTimeout, 16, t);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(sA + stage * kPABytes);
            const uint32_t b_addr = smem_u32(sB + stage * kPBBytes);
            // four MMAs per 128-byte k-block: K = 16 bf16 or 32 e4m3 each, so
            // the K-major descriptors advance 32 bytes either way, and a whole
            // k-block between the k-blocks of a stage
#pragma unroll
            for (int k = 0; k < 4 * G::kSub; ++k) {
              const uint32_t kbo = (k / 4) * kPKBlockBytes;
              const uint64_t adesc = sdesc_sw128(a_addr + kbo + (k % 4) * a_step, a_lbo, 1024);
              const uint64_t bdesc = sdesc_sw128(b_addr + kbo + (k % 4) * b_step, b_lbo, 1024);
              if constexpr (kFp8)
                umma_e4m3_pair(d_tmem, adesc, bdesc, idesc, (kb > 0 || k > 0) ? 1u : 0u);
              else
                umma_bf16_pair(d_tmem, adesc, bdesc, idesc, (kb > 0 || k > 0) ? 1u : 0u);
            }
            umma_commit_pair_both(&empty[stage]);
            if (++stage == kPStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          if (num_kb == 0) {
            mbar_arrive(&tfull[buf]);
            mbar_arrive_cluster(map_rank(&tfull[buf], 1));
          } else {
            umma_commit_pair_both(&tfull[buf]);
          }
        }
      }
      umma_commit_pair_local(drain);
      long long t0 = clock64();
      while (!mbar_try_wait(drain, 0) && clock64() - t0 < a.budget) {
      }
    }
  } else {
    // ------------------------------------------------ epilogue warps (both CTAs)
    const int q = warp & 3;
    uint32_t epi_cnt = 0;
    for (int it = 0;; ++it) {
      const int slot = it % kRing;
      if (!mbar_wait_cl(&rfull[slot], (it / kRing) & 1, abort_flag, a.budget)) {
        report(st, kStTimeout, 17, it);
        break;
      }
      const int t = ring[slot];
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&rempty[slot]);
        else mbar_arrive_cluster(rempty_leader0 + 8 * slot);
      }
      if (t < 0) break;
      const Work w = locate(t, js, a.n_jobs, a);
      const TcJob& jb = a.jobs[w.job];
      const int kind = jb.kind;
      const bool k_empty = (js[w.job].num_kb == 0);
      const int buf = it & 1;
      const uint32_t tph = (it >> 1) & 1;
      // Rows and columns this warp holds.  A 256-row tile gives CTA r rows
      // [128r, 128r + 128), TMEM lane = row.  A 128-row tile (the last m-tile
      // of a job with at most 128 real rows there, computed by a 128 x 256
      // pair MMA) gives CTA r rows [64r, 64r + 64): TMEM lanes 0..63 hold
      // their columns 0..127 and lanes 64..127 the same rows' columns 128..255.
      const bool half = last_half && a.jobs[w.job].M_fixed <= 0 && w.tc.m == js[w.job].num_m - 1;
      const int hcol = half ? (q >> 1) : 0;
      const int row = (half ? (q & 1) : q) * 32 + lane;
      const int c0 = hcol * (kTcBN / 2);
      const int ncol = half ? kTcBN / 2 : kTcBN;
      const long long r0 = static_cast<long long>(w.tc.m) * kPM +
                           static_cast<long long>(rank) * (half ? kPHalf / 2 : kPHalf);
      const long long r = r0 + row;
      int tok = -1;
      if (kind != kTcDWeight) tok = a.row_map[r];
      int tgt = -1;
      RowScalars rs;
      rs.active = false;
      bool active = false;
      float rscale = 0.f;
      if (kFwd) {
        if (tok >= 0) {
          tgt = a.targets[tok] - a.t_off;
          if constexpr (kFp8) rscale = a.hscale[tok];
        }
      } else if (kMode == 3 || kind == kTcDLogits) {
        active = (tok >= 0) && (a.mask[tok] != 0);
        rs.active = active;
        if (active) {
          if constexpr (kMode == 3) rs.hs = a.hscale[tok];
          const float l = a.lse[tok], h = a.ent[tok], gl = a.g_lp[tok], gh = a.g_h[tok];
          rs.lse2 = l * kLog2e;
          rs.gh2 = gh * kLn2;
          rs.c1 = fmaf(gh, h, gl);
          rs.glp = gl;
          const int tg = a.targets[tok] - a.t_off - jb.v0;
          rs.tgt = (tg >= 0 && tg < jb.vc_live) ? tg : -1;
        }
      } else if (kind == kTcDHidden) {
        active = (tok >= 0) && (a.mask[tok] != 0);
      }
      // a wide tile hands over its two halves one after the other (TMEM
      // columns [0, 256) then [256, 512), one barrier phase per tile each)
      bool dead = false;
      for (int h = 0; h < (G::kWide ? 2 : 1); ++h) {
        const int hb = G::kWide ? h : buf;
        const uint32_t hph = G::kWide ? (static_cast<uint32_t>(it) & 1u) : tph;
        if (!mbar_wait_cl(&tfull[hb], hph, abort_flag, a.budget)) {
          report(st, kStTimeout, 18, t);
          dead = true;
          break;
        }
        tc_fence_after();
        const int n_blk = G::kWide ? 2 * w.tc.n + h : w.tc.n;     // 256-column block of N
        if (!G::kWide || n_blk < js[w.job].num_nb) {
          const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + hb * kTcBN;
          if constexpr (kMode == 3) {
            epi_dlogits<true>(jb, tbase, k_empty, r0, n_blk, q, row, c0, ncol, rs, sEpi, epi_cnt,
                              a.wscale);
          } else if constexpr (kFp8) {
            epi_fwd<true>(a, tbase, k_empty, r0, n_blk, row, tgt, rscale, a.wscale);
          } else if constexpr (kFwd) {
            epi_fwd<false>(a, tbase, k_empty, r0, n_blk, row, tgt, 0.f, nullptr);
          } else {
            if (kind == kTcDLogits)
              epi_dlogits<false>(jb, tbase, k_empty, r0, n_blk, q, row, c0, ncol, rs, sEpi, epi_cnt,
                                 nullptr);
            else if (kind == kTcDHidden) {
              if (jb.last_chunk)
                epi_dhidden_last(a, jb, tbase, k_empty, r0, n_blk, row, c0, ncol, tok, active);
              else
                epi_dhidden_acc(a, jb, tbase, k_empty, r0, n_blk, q, row, c0, ncol, sEpi, epi_cnt);
            }
            else epi_dweight(a, jb, tbase, k_empty, r0, n_blk, row);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(&tempty[hb]);
          else mbar_arrive_cluster(tempty_leader0 + 8 * hb);
        }
      }
      if (dead) break;
    }
    if (!kFwd && lane == 0) bulk_wait_all();   // every staged d-logits box written
  }

  tc_fence_before();
  cluster_sync_all();     // both CTAs done with TMEM and with each other's barriers
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kTmemCols)
                 : "memory");
  }
}

}  // namespace

size_t tc_smem_bytes() {
  size_t m = PipeGeo<0>::kSmemBytes;
  if (PipeGeo<1>::kSmemBytes > m) m = PipeGeo<1>::kSmemBytes;
  if (PipeGeo<2>::kSmemBytes > m) m = PipeGeo<2>::kSmemBytes;
  if (PipeGeo<3>::kSmemBytes > m) m = PipeGeo<3>::kSmemBytes;
  return m;
}

int tc_tile_rows() { return kPM; }

cudaError_t launch_tc_gemm(const TcArgs& args, int grid, cudaStream_t s) {
  if (grid <= 0) return cudaSuccess;
  if (args.n_jobs < 1 || args.n_jobs > kMaxTcJobs) return cudaErrorInvalidValue;
  // the jobs of one launch belong to one family (see tc_pair_kernel)
  auto family = [](int kind) {
    return kind == kTcFwd ? 0 : kind == kTcFwdFp8 ? 2 : kind == kTcDLogitsFp8 ? 3 : 1;
  };
  const int mode = family(args.jobs[0].kind);
  for (int j = 1; j < args.n_jobs; ++j)
    if (family(args.jobs[j].kind) != mode) return cudaErrorInvalidValue;
  // the large dynamic shared memory is opted into once per device and
  // instantiation (one bit per device ordinal; a repeated opt-in is harmless)
  static std::atomic<uint64_t> configured[4];
  void (*kern)(TcArgs) = mode == 0   ? tc_pair_kernel<0>
                         : mode == 1 ? tc_pair_kernel<1>
                         : mode == 2 ? tc_pair_kernel<2>
                                     : tc_pair_kernel<3>;
  const int smem = mode == 0   ? PipeGeo<0>::kSmemBytes
                   : mode == 1 ? PipeGeo<1>::kSmemBytes
                   : mode == 2 ? PipeGeo<2>::kSmemBytes
                               : PipeGeo<3>::kSmemBytes;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
  if (bit == 0 || (configured[mode].load(std::memory_order_acquire) & bit) == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[mode].fetch_or(bit, std::memory_order_release);
  }
  const int clusters = (grid + 1) / 2;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the CTA prologue (barrier set-up, TMEM
  // allocation, descriptor prefetch) overlaps the previous kernel's last
  // wave; the kernel waits for that grid before its first global read
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, args);
}

}  // namespace eas
