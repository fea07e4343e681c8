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
// the CTAs draw from through a global atomic counter, so a CTA that finishes
// early takes more work and the jobs fill each other's tails.
//
// CTA layout (192 threads): warp 0 = tile fetcher + TMA producer (one lane),
// warp 1 = MMA issuer (one lane) and TMEM owner, warps 2..5 = epilogue, one
// accumulator row per thread (warp w reads TMEM lanes 32*(w%4) .. +31).  The
// producer publishes each tile index in a small shared ring that the MMA and
// epilogue roles read in order.  Four smem stages of A 128x64 + B 256x64 bf16
// (48 KB each, 128-byte swizzle); two 128x256 fp32 accumulators in TMEM (all
// 512 columns) so the epilogue of tile i overlaps the mainloop of tile i+1.
// Every mbarrier wait is bounded; on expiry the CTA raises an abort flag,
// drains its in-flight copies and MMAs, frees TMEM and reports kStTimeout.
#include "eas_device.cuh"
#include "eas_kernels.h"

namespace eas {

namespace {

constexpr int kStages = 4;
constexpr int kRing = 4;                      // tile indices in flight
constexpr int kABytes = kTcBM * kTcBK * 2;   // 16 KB
constexpr int kBBytes = kTcBN * kTcBK * 2;   // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align slack*/ + 512 /*barriers*/;

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
__device__ __forceinline__ void epi_fwd(const TcArgs& a, uint32_t tbase, bool k_empty, int m_blk,
                                        int n_blk, int row, int tgt) {
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
    const int tj = tgt - (n0 + c * 32);
    if (static_cast<unsigned>(tj) < 32u) {
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
  const long long r = static_cast<long long>(m_blk) * kTcBM + row;
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
};

// d-logits of one row: dZ = g_lp (onehot - p) - g_H p (z - lse + H), p =
// exp(z - lse), written as -p (g_H (z - lse) + g_lp + g_H H) + g_lp onehot.
// Inactive rows and columns past the live width are written as exact zeros.
__device__ __forceinline__ void epi_dlogits(const TcArgs& a, const TcJob& jb, uint32_t tbase,
                                            bool k_empty, int m_blk, int n_blk, int row,
                                            const RowScalars& rs) {
  const long long r = static_cast<long long>(m_blk) * kTcBM + row;
  const int n0 = n_blk * kTcBN;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(jb.dz) + r * a.ldz + n0;
#pragma unroll 1
  for (int c = 0; c < kTcBN / 32; ++c) {
    uint32_t pk[16];
    const int col0 = n0 + c * 32;
    // tcgen05.ld is warp-collective: only warp-uniform conditions (live
    // width, empty K) may skip it; per-row activity is applied afterwards.
    if (col0 >= jb.vc_live) {
#pragma unroll
      for (int j = 0; j < 16; ++j) pk[j] = 0u;
    } else {
      float v[32];
      if (k_empty) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.f;
      } else {
        tmem_ld32(tbase + c * 32, v);
      }
      if (!rs.active) {
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = 0u;
      } else {
        const int cvalid = jb.vc_live - col0;
        const int tj = rs.tgt - col0;
        float d[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float x2 = fmaf(v[j], kLog2e, -rs.lse2);    // (z - lse) log2 e
          const float p = ex2_approx(x2);
          const float w = fmaf(rs.gh2, x2, rs.c1);           // g_H (z - lse) + g_lp + g_H H
          float dz = -p * w;
          if (j == tj) dz += rs.glp;
          d[j] = (j < cvalid) ? dz : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(d[2 * j], d[2 * j + 1]);
      }
    }
    uint4* o = reinterpret_cast<uint4*>(out + c * 32);
#pragma unroll
    for (int q = 0; q < 4; ++q) o[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
  }
}

// dHidden: accumulate this chunk's product into the fp32 accumulator; the
// last chunk converts to bf16 and scatters the row to its token (zeros for
// gap rows whose mask byte is 0).
__device__ __forceinline__ void epi_dhidden(const TcArgs& a, const TcJob& jb, uint32_t tbase,
                                            bool k_empty, int m_blk, int n_blk, int row, int tok,
                                            bool active) {
  const long long r = static_cast<long long>(m_blk) * kTcBM + row;
  const int n0 = n_blk * kTcBN;
  float* accp = a.acc + r * a.H + n0;
  __nv_bfloat16* outp =
      (tok >= 0) ? static_cast<__nv_bfloat16*>(a.dhidden) + static_cast<long long>(tok) * a.H + n0
                 : nullptr;
#pragma unroll 1
  for (int c = 0; c < kTcBN / 32; ++c) {
    if (n0 + c * 32 >= a.H) break;
    float v[32];
    if (k_empty) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0.f;
    } else {
      tmem_ld32(tbase + c * 32, v);
    }
    float4* ap = reinterpret_cast<float4*>(accp + c * 32);
    if (!jb.first_chunk) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 x = ap[q];
        v[4 * q] += x.x;
        v[4 * q + 1] += x.y;
        v[4 * q + 2] += x.z;
        v[4 * q + 3] += x.w;
      }
    }
    if (!jb.last_chunk) {
#pragma unroll
      for (int q = 0; q < 8; ++q) ap[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    } else if (outp != nullptr) {
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) pk[j] = active ? pack_bf16x2(v[2 * j], v[2 * j + 1]) : 0u;
      uint4* o = reinterpret_cast<uint4*>(outp + c * 32);
#pragma unroll
      for (int q = 0; q < 4; ++q) o[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
  }
}

// dW rows of this chunk: every vocabulary row of the chunk is overwritten.
__device__ __forceinline__ void epi_dweight(const TcArgs& a, const TcJob& jb, uint32_t tbase,
                                            bool k_empty, int m_blk, int n_blk, int row) {
  const int m = m_blk * kTcBM + row;
  const int n0 = n_blk * kTcBN;
  const bool live = m < jb.vc_live;
  float* outp = a.dW + (static_cast<long long>(jb.v0) + m) * a.H + n0;
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
    if (live) {
      float4* o = reinterpret_cast<float4*>(outp + c * 32);
#pragma unroll
      for (int q = 0; q < 8; ++q) o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
  }
}

// ----------------------------------------------------------------- kernel --

__global__ void __launch_bounds__(kThreads, 1) tc_gemm_kernel(const __grid_constant__ TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kStages * kBBytes);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* rfull = tempty + 2;
  uint64_t* rempty = rfull + kRing;
  uint64_t* drain = rempty + kRing;
  int* ring = reinterpret_cast<int*>(drain + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ring + kRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Sched* sched = static_cast<const Sched*>(a.sched);
  DevStatus* st = static_cast<DevStatus*>(a.status);

  JobShape js[kMaxTcJobs];
  int total = 0;
#pragma unroll
  for (int j = 0; j < kMaxTcJobs; ++j) {
    js[j] = JobShape{0, 0, 0, 0, total};
    if (j < a.n_jobs) {
      const TcJob& jb = a.jobs[j];
      const int M = jb.M_fixed > 0 ? jb.M_fixed : sched->R_pad;
      const int K = jb.K_fixed > 0 ? jb.K_fixed : sched->R_pad;
      js[j].num_m = (M + kTcBM - 1) / kTcBM;
      js[j].num_n = (jb.N + kTcBN - 1) / kTcBN;
      js[j].num_kb = (K + kTcBK - 1) / kTcBK;
      js[j].tiles = js[j].num_m * js[j].num_n;
      total += js[j].tiles;
    }
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&rfull[i], 1);
      mbar_init(&rempty[i], 1 + 4);     // MMA thread + 4 epilogue warps
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
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------ tile fetcher + TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int slot = it % kRing;
        const uint32_t rph = (it / kRing) & 1;
        if (!mbar_wait(&rempty[slot], rph ^ 1u, abort_flag, a.budget)) {
          report(st, kStTimeout, 1, it);
          ok = false;
          break;
        }
        const int t = atomicAdd(a.tile_counter, 1);
        ring[slot] = (t < total) ? t : -1;
        mbar_arrive(&rfull[slot]);
        if (t >= total) break;
        const Work w = locate(t, js, a.n_jobs, a);
        const TcJob& jb = a.jobs[w.job];
        const int kind = jb.kind;
        for (int kb = 0; kb < js[w.job].num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.budget)) {
            report(st, kStTimeout, 2, t);
            ok = false;
            break;
          }
          uint8_t* dA = sA + stage * kABytes;
          uint8_t* dB = sB + stage * kBBytes;
          mbar_arrive_expect_tx(&full[stage], kStageBytes);
          const int k0 = kb * kTcBK;
          if (kind == kTcFwd || kind == kTcDLogits) {
            tma_load_2d(dA, &jb.tmA, &full[stage], k0, w.tc.m * kTcBM);
            tma_load_2d(dB, &jb.tmB, &full[stage], k0, jb.v0 + w.tc.n * kTcBN);
          } else if (kind == kTcDHidden) {
            tma_load_2d(dA, &jb.tmA, &full[stage], k0, w.tc.m * kTcBM);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tma_load_2d(dB + j * 8192, &jb.tmB, &full[stage], w.tc.n * kTcBN + j * 64, jb.v0 + k0);
          } else {
#pragma unroll
            for (int j = 0; j < 2; ++j)
              tma_load_2d(dA + j * 8192, &jb.tmA, &full[stage], w.tc.m * kTcBM + j * 64, k0);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tma_load_2d(dB + j * 8192, &jb.tmB, &full[stage], w.tc.n * kTcBN + j * 64, k0);
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let every copy this thread issued land before the CTA exits: the
        // last use of stage s had parity `phase` if s < stage, else phase^1.
        for (int s = 0; s < kStages; ++s) {
          const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
          long long t0 = clock64();
          while (!mbar_try_wait(&full[s], par) && clock64() - t0 < a.budget) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int it = 0;; ++it) {
        const int slot = it % kRing;
        if (!mbar_wait(&rfull[slot], (it / kRing) & 1, abort_flag, a.budget)) {
          report(st, kStTimeout, 3, it);
          break;
        }
        const int t = ring[slot];
        mbar_arrive(&rempty[slot]);
        if (t < 0) break;
        const Work w = locate(t, js, a.n_jobs, a);
        const int kind = a.jobs[w.job].kind;
        const bool a_mn = (kind == kTcDWeight);
        const bool b_mn = (kind == kTcDHidden || kind == kTcDWeight);
        const uint32_t idesc = a_mn ? idesc_bf16_f32(kTcBM, kTcBN, true, true)
                                    : (b_mn ? idesc_bf16_f32(kTcBM, kTcBN, false, true)
                                            : idesc_bf16_f32(kTcBM, kTcBN, false, false));
        const uint32_t a_lbo = a_mn ? 8192 : 16, a_step = a_mn ? 2048 : 32;
        const uint32_t b_lbo = b_mn ? 8192 : 16, b_step = b_mn ? 2048 : 32;
        const int buf = it & 1;
        const uint32_t tph = (it >> 1) & 1;
        if (!mbar_wait(&tempty[buf], tph ^ 1u, abort_flag, a.budget)) {
          report(st, kStTimeout, 4, t);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * kTcBN;
        const int num_kb = js[w.job].num_kb;
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, a.budget)) {
            report(st, kStTimeout, 5, t);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + stage * kABytes);
          const uint32_t b_addr = smem_u32(sB + stage * kBBytes);
#pragma unroll
          for (int k = 0; k < kTcBK / 16; ++k) {
            const uint64_t adesc = sdesc_sw128(a_addr + k * a_step, a_lbo, 1024);
            const uint64_t bdesc = sdesc_sw128(b_addr + k * b_step, b_lbo, 1024);
            umma_bf16(d_tmem, adesc, bdesc, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (num_kb == 0)
          mbar_arrive(&tfull[buf]);
        else
          umma_commit(&tfull[buf]);
      }
      // Wait for every MMA this thread issued before TMEM is released.
      umma_commit(drain);
      long long t0 = clock64();
      while (!mbar_try_wait(drain, 0) && clock64() - t0 < a.budget) {
      }
    }
  } else {
    // ------------------------------------------------ epilogue warps
    const int q = warp & 3;               // TMEM lane quarter of this warp
    const int row = q * 32 + lane;        // accumulator row of this thread
    for (int it = 0;; ++it) {
      const int slot = it % kRing;
      if (!mbar_wait(&rfull[slot], (it / kRing) & 1, abort_flag, a.budget)) {
        report(st, kStTimeout, 6, it);
        break;
      }
      const int t = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&rempty[slot]);
      if (t < 0) break;
      const Work w = locate(t, js, a.n_jobs, a);
      const TcJob& jb = a.jobs[w.job];
      const int kind = jb.kind;
      const bool k_empty = (js[w.job].num_kb == 0);
      const int buf = it & 1;
      const uint32_t tph = (it >> 1) & 1;
      // per-row operands, fetched before waiting on the accumulator
      const long long r = static_cast<long long>(w.tc.m) * kTcBM + row;
      int tok = -1;
      if (kind != kTcDWeight) tok = a.row_map[r];
      int tgt = -1;
      RowScalars rs;
      rs.active = false;
      bool active = false;
      if (kind == kTcFwd) {
        if (tok >= 0) tgt = a.targets[tok];
      } else if (kind == kTcDLogits) {
        active = (tok >= 0) && (a.mask[tok] != 0);
        rs.active = active;
        if (active) {
          const float l = a.lse[tok], h = a.ent[tok], gl = a.g_lp[tok], gh = a.g_h[tok];
          rs.lse2 = l * kLog2e;
          rs.gh2 = gh * kLn2;
          rs.c1 = fmaf(gh, h, gl);
          rs.glp = gl;
          const int tg = a.targets[tok] - jb.v0;
          rs.tgt = (tg >= 0 && tg < jb.vc_live) ? tg : -1;
        }
      } else if (kind == kTcDHidden) {
        active = (tok >= 0) && (a.mask[tok] != 0);
      }
      if (!mbar_wait(&tfull[buf], tph, abort_flag, a.budget)) {
        report(st, kStTimeout, 7, t);
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * kTcBN;
      if (kind == kTcFwd) epi_fwd(a, tbase, k_empty, w.tc.m, w.tc.n, row, tgt);
      else if (kind == kTcDLogits) epi_dlogits(a, jb, tbase, k_empty, w.tc.m, w.tc.n, row, rs);
      else if (kind == kTcDHidden) epi_dhidden(a, jb, tbase, k_empty, w.tc.m, w.tc.n, row, tok, active);
      else epi_dweight(a, jb, tbase, k_empty, w.tc.m, w.tc.n, row);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

size_t tc_smem_bytes() { return kSmemBytes; }

cudaError_t launch_tc_gemm(const TcArgs& args, int grid, cudaStream_t s) {
  if (grid <= 0) return cudaSuccess;
  if (args.n_jobs < 1 || args.n_jobs > kMaxTcJobs) return cudaErrorInvalidValue;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  tc_gemm_kernel<<<grid, kThreads, kSmemBytes, s>>>(args);
  return cudaGetLastError();
}

}  // namespace eas
