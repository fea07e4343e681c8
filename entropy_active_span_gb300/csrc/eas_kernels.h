// Internal launchers shared by the C-ABI layer (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace eas {

struct DevStatus;
struct Sched;

// ---- span builder and row schedule (eas_sched.cu) ----
cudaError_t launch_spans_build(const uint8_t* mask, long long T, int max_gap, int* spans,
                               long long cap, int* num_spans, DevStatus* st, cudaStream_t s);
// Row schedule in two passes over tiles of 4096 tokens; tile_rows holds
// rowmap_tiles(T) entries of scratch.
long long rowmap_tiles(long long T);
cudaError_t launch_rowmap(const uint8_t* mask, const int* spans, const int* num_spans,
                          long long cap, long long T, int span_rows, const int* targets, int t_lo,
                          int t_hi, int* row_map, int* pack_of, long long* tile_rows,
                          Sched* sched, DevStatus* st, cudaStream_t s);
cudaError_t launch_gather_rows(const void* src, void* dst, const int* row_map, const Sched* sched,
                               long long T_pad, long long row_bytes, int num_sms, cudaStream_t s);
cudaError_t launch_combine(const float* pm, const float* ps, const float* pu, const float* zt,
                           int n_tiles, long long stride, const int* pack_of, const uint8_t* mask,
                           long long T, float* logprob, float* entropy, float* lse, int num_sms,
                           cudaStream_t s);
// Per-token statistics of one vocabulary shard instead of final outputs:
// stats[t] = (M, S, U, z_target if the target lies in the shard else 0).
cudaError_t launch_combine_stats(const float* pm, const float* ps, const float* pu,
                                 const float* zt, int n_tiles, long long stride, const int* pack_of,
                                 const uint8_t* mask, const int* targets, int t_off, int v_shard,
                                 long long T, float4* stats, int num_sms, cudaStream_t s);
cudaError_t launch_combine_shards(const float4* stats, int n_shards, long long T,
                                  const uint8_t* mask, float* logprob, float* entropy, float* lse,
                                  int num_sms, cudaStream_t s);
cudaError_t launch_zero_unpacked_rows(void* out, const int* pack_of, long long T,
                                      long long row_bytes, int num_sms, cudaStream_t s);
cudaError_t launch_selftest_wait(long long budget, DevStatus* st, cudaStream_t s);
cudaError_t launch_cp_local(const uint8_t* mask, const int* offs, int n_segs, long long T, int cp,
                            int rank, uint8_t* local_mask, int* l2g, DevStatus* st, int num_sms,
                            cudaStream_t s);

// ---- tcgen05 GEMMs with fused epilogues, bf16 (eas_gemm_tc.cu) ----

// Tensor-core tiles: 256 x 256 outputs per CTA pair (128 x 256 per CTA in
// TMEM), K in blocks of 64 bf16 (one 128-byte swizzle row).
constexpr int kTcBM = 128;    // accumulator rows held by one CTA
constexpr int kTcBN = 256;
constexpr int kTcBK = 64;

enum TcKind : int {
  kTcFwd = 0,      // Z = Hp W^T -> per-tile softmax partials (+ target logit)
  kTcDLogits = 1,  // Z = Hp W_c^T -> dZ_c (bf16 staging)
  kTcDHidden = 2,  // dHacc (+)= dZ_c W_c -> fp32 accumulator / final dhidden
  kTcDWeight = 3,  // dW_c = dZ_c^T Hp -> fp32 dW rows
  kTcFwdFp8 = 4,   // as kTcFwd with e4m3 operands and per-row scales
  kTcDLogitsFp8 = 5,  // as kTcDLogits with e4m3 operands and per-row scales
};

// One contraction of a launch.  A launch runs up to kMaxTcJobs jobs; their
// tiles form one list (job 0's tiles first) that the CTAs draw from with an
// atomic counter, so jobs with no dependency between them share the machine
// and fill each other's tails.
struct TcJob {
  CUtensorMap tmA;   // A operand (see TcKind for the layout of each kind)
  CUtensorMap tmB;   // B operand
  CUtensorMap tmD;   // TMA store target: the d-logits staging (dlogits), the fp32
                     // accumulator (dhidden before the last chunk)
  int kind;
  int M_fixed;       // > 0: rows of the problem; 0: R_pad from sched
  int N;             // columns of the problem
  int K_fixed;       // > 0: reduction length; 0: the packed row count R from sched
  int group_m;       // m-tiles per raster band
  int v0;            // first vocabulary row of the chunk (B row / k offset)
  int vc_live;       // live columns of this chunk (dlogits / dweight)
  int first_chunk;   // dhidden: first chunk (store, do not accumulate)
  int last_chunk;    // dhidden: last chunk (convert and scatter to dhidden)
};

constexpr int kMaxTcJobs = 3;

struct TcArgs {
  TcJob jobs[kMaxTcJobs];
  int n_jobs;
  const void* sched; // Sched*: packed row count R, R_pad
  void* status;      // DevStatus*
  int* tile_counter; // zero before the launch; one atomic per tile
  long long budget;  // clocks before a pipeline wait gives up
  // epilogue operands shared by the jobs
  const int* row_map;     // packed row -> token (or -1)
  const int* targets;     // [T]
  int t_off;              // first vocabulary id of W's rows (vocabulary shard), else 0
  const uint8_t* mask;    // [T]
  const float* lse;       // [T]
  const float* ent;       // [T]
  const float* g_lp;      // [T]
  const float* g_h;       // [T]
  float* part_m;          // fwd partials, [n_vtiles][stride]
  float* part_s;
  float* part_u;
  float* zt;              // [stride]
  long long part_stride;
  int V;                  // vocabulary size (fwd column bound)
  long long ldz;          // staging row pitch
  float* acc;             // fp32 dHidden accumulator [T_pad][H]
  void* dhidden;          // bf16 [T][H]
  int H;
  float* dW;              // fp32 [V][H]
  const float* hscale;    // e4m3 kinds: per-token scale of hidden [T]
  const float* wscale;    // e4m3 kinds: per-row scale of W [V]
};

size_t tc_smem_bytes();
// Rows of one tensor-core tile (256 for the CTA-pair kernel, else 128).
int tc_tile_rows();
cudaError_t launch_tc_gemm(const TcArgs& args, int grid, cudaStream_t s);

// ---- fp32 SIMT GEMMs with the same epilogues (eas_simt.cu) ----
constexpr int kSimtBM = 64;
constexpr int kSimtBN = 64;

struct SimtArgs {
  int kind;               // TcKind values
  const float* A;         // see launch_simt_gemm
  const float* B;
  long long lda, ldb;
  const void* sched;
  int M_fixed, N, K_fixed;
  int v0;
  const int* row_map;
  const int* targets;
  int t_off;
  const uint8_t* mask;
  const float* lse;
  const float* ent;
  const float* g_lp;
  const float* g_h;
  float* part_m;
  float* part_s;
  float* part_u;
  float* zt;
  long long part_stride;
  int V;
  int vc_live;
  float* dz;
  long long ldz;
  float* acc;
  float* dhidden;
  int H;
  int first_chunk;
  int last_chunk;
  float* dW;
};

cudaError_t launch_simt_gemm(const SimtArgs& args, long long max_tiles, cudaStream_t s);

}  // namespace eas

namespace eas {
// ---- e4m3 quantisation (eas_fp8.cu) ----
cudaError_t launch_quantize_rows_e4m3(const void* src, int src_is_bf16, long long R, long long H,
                                      uint8_t* dst, float* scale, int num_sms, cudaStream_t s);
// ---- helpers the C-ABI translation units share (eas_api.cu) ----
size_t lmhead_fwd_workspace_bytes(long long T, long long H, long long V, int dtype);
void set_last_error(const char* msg);
}  // namespace eas
