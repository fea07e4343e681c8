// fp32 path of the fused LM-head: the same four contractions and epilogues as
// the tensor-core path (forward softmax partials, d-logits, dHidden, dW), on
// CUDA cores with fp32 FMA so that fp32 inputs keep fp32 accuracy end to end
// (d-logits are staged in fp32 too).  Tiles of 64 x 64 outputs, K in steps of
// 16 through shared memory; 256 threads, 4 x 4 outputs each (rows ty + 16 i,
// columns tx + 16 j), so the 16 threads that share a row form a half-warp and
// reduce row statistics with shuffles.
#include "eas_device.cuh"
#include "eas_kernels.h"

namespace eas {

namespace {

constexpr int BM = kSimtBM, BN = kSimtBN, BK = 16;

struct Operand {
  const float* p;
  long long s_mn;   // stride between rows of the M (or N) index
  long long s_k;    // stride along K
};

__device__ __forceinline__ Operand op_a(const SimtArgs& a) {
  if (a.kind == kTcDWeight) return {a.A, 1, a.lda};       // dZ^T: A(m,k) = dz[k, m]
  return {a.A, a.lda, 1};                                 // Hp or dZ rows
}

__device__ __forceinline__ Operand op_b(const SimtArgs& a) {
  if (a.kind == kTcFwd || a.kind == kTcDLogits)
    return {a.B + static_cast<long long>(a.v0) * a.ldb, a.ldb, 1};          // W rows
  if (a.kind == kTcDHidden)
    return {a.B + static_cast<long long>(a.v0) * a.ldb, 1, a.ldb};          // W^T
  return {a.B, 1, a.ldb};                                                   // Hp^T
}

__global__ void __launch_bounds__(256) simt_gemm_kernel(const SimtArgs a) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const Sched* sched = static_cast<const Sched*>(a.sched);
  const int M = a.M_fixed > 0 ? a.M_fixed : sched->R_pad;
  const int K = a.K_fixed > 0 ? a.K_fixed : sched->R_pad;
  const int num_m = (M + BM - 1) / BM;
  const int num_n = (a.N + BN - 1) / BN;
  const long long tiles = static_cast<long long>(num_m) * num_n;
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const Operand A = op_a(a), B = op_b(a);

  for (long long t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int mb = static_cast<int>(t % num_m);
    const int nb = static_cast<int>(t / num_m);
    const int m0 = mb * BM, n0 = nb * BN;
    float c[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) c[i][j] = 0.f;

    for (int k0 = 0; k0 < K; k0 += BK) {
      // 64 x 16 elements of each operand, 4 per thread
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int idx = tid + e * 256;
        const int kk = idx & 15, mm = idx >> 4;
        const int gm = m0 + mm, gk = k0 + kk;
        float va = 0.f;
        if (gm < M && gk < K) va = A.p[gm * A.s_mn + gk * A.s_k];
        As[kk][mm] = va;
        const int gn = n0 + mm;
        float vb = 0.f;
        if (gn < a.N && gk < K) vb = B.p[gn * B.s_mn + gk * B.s_k];
        Bs[kk][mm] = vb;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < BK; ++kk) {
        float ra[4], rb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) ra[i] = As[kk][ty + 16 * i];
#pragma unroll
        for (int j = 0; j < 4; ++j) rb[j] = Bs[kk][tx + 16 * j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) c[i][j] = fmaf(ra[i], rb[j], c[i][j]);
      }
      __syncthreads();
    }

    // ------------------------------------------------------------ epilogues
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int m = m0 + ty + 16 * i;
      const bool mrow = m < M;
      if (a.kind == kTcFwd) {
        // row statistics over this tile's valid columns (base-2 units)
        const int tok = mrow ? a.row_map[m] : -1;
        const int tgt = (tok >= 0) ? a.targets[tok] - a.t_off : -1;
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (n0 + tx + 16 * j < a.V) mx = fmaxf(mx, c[i][j] * kLog2e);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float s = 0.f, u = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int n = n0 + tx + 16 * j;
          if (n < a.V) {
            const float d = fmaf(c[i][j], kLog2e, -mx);
            const float e = ex2_approx(d);
            s += e;
            u = fmaf(e, d, u);
          }
          if (n == tgt && mrow) a.zt[m] = c[i][j];
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
          s += __shfl_xor_sync(0xffffffffu, s, o);
          u += __shfl_xor_sync(0xffffffffu, u, o);
        }
        if (tx == 0 && mrow) {
          const long long off = static_cast<long long>(nb) * a.part_stride + m;
          a.part_m[off] = mx;
          a.part_s[off] = s;
          a.part_u[off] = u;
        }
      } else if (a.kind == kTcDLogits) {
        if (!mrow) continue;
        const int tok = a.row_map[m];
        const bool active = (tok >= 0) && (a.mask[tok] != 0);
        float l = 0.f, h = 0.f, gl = 0.f, gh = 0.f;
        int tg = -1;
        if (active) {
          l = a.lse[tok];
          h = a.ent[tok];
          gl = a.g_lp[tok];
          gh = a.g_h[tok];
          tg = a.targets[tok] - a.t_off - a.v0;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int n = n0 + tx + 16 * j;
          if (n >= a.N) continue;
          float dz = 0.f;
          if (active) {
            const float x = c[i][j] - l;                 // z - lse
            const float p = ex2_approx(x * kLog2e);
            dz = -p * fmaf(gh, x + h, gl);
            if (n == tg) dz += gl;
          }
          a.dz[static_cast<long long>(m) * a.ldz + n] = dz;
        }
      } else if (a.kind == kTcDHidden) {
        if (!mrow) continue;
        const int tok = a.row_map[m];
        const bool active = (tok >= 0) && (a.mask[tok] != 0);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int n = n0 + tx + 16 * j;
          if (n >= a.N) continue;
          float v = c[i][j];
          float* accp = a.acc + static_cast<long long>(m) * a.H + n;
          if (!a.first_chunk) v += *accp;
          if (!a.last_chunk) {
            *accp = v;
          } else if (tok >= 0) {
            a.dhidden[static_cast<long long>(tok) * a.H + n] = active ? v : 0.f;
          }
        }
      } else {   // kTcDWeight
        if (m >= a.vc_live) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int n = n0 + tx + 16 * j;
          if (n >= a.N) continue;
          a.dW[(static_cast<long long>(a.v0) + m) * a.H + n] = c[i][j];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_simt_gemm(const SimtArgs& args, long long max_tiles, cudaStream_t s) {
  if (max_tiles <= 0) return cudaSuccess;
  long long grid = max_tiles < 4096 ? max_tiles : 4096;
  simt_gemm_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(args);
  return cudaGetLastError();
}

}  // namespace eas
