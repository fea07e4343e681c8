// C ABI of the block-sparse fused LM-head (declared in include/eas.h).
//
// Host side only: argument checks, the workspace layout, TMA tensor maps, and
// the stream-ordered launch sequence of each call.  No call allocates memory
// or synchronises the host (except eas_read_device_status).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <deque>
#include <atomic>
#include <mutex>

#include "../../include/eas.h"
#include "eas_device.cuh"
#include "eas_kernels.h"

using namespace eas;

namespace {

thread_local char g_err[512] = "";

eas_status fail(eas_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

eas_status cuda_fail(cudaError_t e, const char* what) {
  return fail(EAS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define EAS_CUDA(call, what)                  \
  do {                                        \
    cudaError_t e_ = (call);                  \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

inline long long round_up(long long x, long long m) { return (x + m - 1) / m * m; }
inline long long cdiv(long long x, long long m) { return (x + m - 1) / m; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ------------------------------------------------------------ device info

struct DevInfo {
  int sms = 0;
  int major = 0, minor = 0;
};

eas_status device_info(DevInfo* out) {
  static std::mutex mu;
  static DevInfo cache[64];
  static bool have[64] = {};
  int dev = 0;
  EAS_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(EAS_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lk(mu);
  if (!have[dev]) {
    DevInfo d;
    EAS_CUDA(cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev), "sm count");
    EAS_CUDA(cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev), "cc");
    EAS_CUDA(cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev), "cc");
    cache[dev] = d;
    have[dev] = true;
  }
  *out = cache[dev];
  if (out->major != 10 || out->minor != 3)
    return fail(EAS_ERR_UNSUPPORTED, "built for sm_103a; device is sm_%d%d", out->major,
                out->minor);
  return EAS_OK;
}

long long wait_budget() {
  static long long b = [] {
    const char* s = getenv("EAS_WAIT_BUDGET_CYCLES");
    long long v = s ? atoll(s) : 0;
    return v > 0 ? v : (1LL << 31);   // ~1 s at 2 GHz
  }();
  return b;
}

// ------------------------------------------------------------ tracing
//
// When enabled, every kernel launch of the library is bracketed by a pair of
// CUDA events on its stream, tagged with the kernel's kind; eas_trace_read()
// returns the durations.  Off by default; meant for eager (not captured)
// launches.  Backward tensor-core launches are named by their jobs:
// dlogits_gemm_tc (d-logits of chunk 0), bwd_chunk_gemm_tc (dW and dHidden of
// chunk c-1 with the d-logits of chunk c), dproj_gemm_tc (dW and dHidden of
// the last chunk); the e4m3 backward runs dlogits_gemm_tc_e4m3 (d-logits of a
// chunk) and dproj_gemm_tc (dW and dHidden of that chunk) per chunk.

enum TraceKind : int {
  kTrSpans = 0, kTrRowmap, kTrGather, kTrFwdGemm, kTrCombine, kTrZeroRows,
  kTrDLogitsGemm, kTrDProjGemm, kTrUnused, kTrSimtFwd, kTrSimtDLogits,
  kTrSimtDHidden, kTrSimtDWeight, kTrMemset, kTrBwdChunkGemm, kTrDLogitsFp8Gemm, kTrCount
};

const char* const kTraceNames[kTrCount] = {
    "spans_build", "rowmap", "gather_rows", "fwd_gemm_tc", "combine", "zero_rows",
    "dlogits_gemm_tc", "dproj_gemm_tc", "unused", "fwd_gemm_simt",
    "dlogits_gemm_simt", "dhidden_gemm_simt", "dweight_gemm_simt", "memset",
    "bwd_chunk_gemm_tc", "dlogits_gemm_tc_e4m3"};

struct TraceRec {
  int kind;
  cudaEvent_t a, b;
};

std::mutex g_trace_mu;
std::atomic<bool> g_trace_on{false};   // read unlocked on every launch
std::deque<TraceRec> g_trace_pool;    // events are created once and reused; a deque
                                      // keeps records in place as it grows
size_t g_trace_used = 0;

class Trace {
 public:
  Trace(int kind, cudaStream_t s) : s_(s) {
    if (!g_trace_on.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lk(g_trace_mu);
    if (!g_trace_on.load(std::memory_order_relaxed)) return;
    if (g_trace_used == g_trace_pool.size()) {
      TraceRec r{kind, nullptr, nullptr};
      if (cudaEventCreate(&r.a) != cudaSuccess) return;
      if (cudaEventCreate(&r.b) != cudaSuccess) {
        cudaEventDestroy(r.a);
        return;
      }
      g_trace_pool.push_back(r);
    }
    rec_ = &g_trace_pool[g_trace_used++];
    rec_->kind = kind;
    cudaEventRecord(rec_->a, s_);
  }
  ~Trace() {
    if (rec_) cudaEventRecord(rec_->b, s_);
  }

 private:
  cudaStream_t s_;
  TraceRec* rec_ = nullptr;
};

// ------------------------------------------------------------ tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

eas_status get_encoder(EncodeTiledFn* fn) {
  static EncodeTiledFn f = nullptr;
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                           cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) f = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!f) return fail(EAS_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(err));
  *fn = f;
  return EAS_OK;
}

// 2-D tensor [rows][cols] with row pitch `ld` elements, 128-byte swizzle, box
// of 128 bytes (64 bf16 or 128 one-byte elements) x box_rows rows;
// out-of-range elements read as zero.
eas_status make_map_2d(CUtensorMap* m, CUtensorMapDataType type, int esize, const void* base,
                       long long cols, long long rows, long long ld, int box_rows) {
  EncodeTiledFn enc;
  eas_status s = get_encoder(&enc);
  if (s != EAS_OK) return s;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esize};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, type, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(EAS_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for [%lld x %lld] ld %lld",
                static_cast<int>(r), rows, cols, ld);
  return EAS_OK;
}

eas_status make_map_bf16(CUtensorMap* m, const void* base, long long cols, long long rows,
                         long long ld, int box_rows) {
  return make_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, cols, rows, ld, box_rows);
}

// MN-major operand [rows = k][cols = m or n] as a 3-D map {64 columns, rows,
// 64-column blocks}: one box {64, 64 k-rows, 2 blocks} lands in shared memory
// as two 8 KB blocks [block][k-row][64 columns], the layout of two 2-D boxes.
// Columns past `cols` in the last block are read from the row's padding
// (within ld); blocks and rows past the end read as zero.
eas_status make_map_bf16_mn3(CUtensorMap* m, const void* base, long long cols, long long rows,
                             long long ld) {
  EncodeTiledFn enc;
  eas_status s = get_encoder(&enc);
  if (s != EAS_OK) return s;
  if (ld < (cols + 63) / 64 * 64) return fail(EAS_ERR_INVALID_ARG, "row pitch below block width");
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>((cols + 63) / 64)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, 128};
  cuuint32_t box[3] = {64, 64, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(EAS_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (%d) for [%lld x %lld] ld %lld",
                static_cast<int>(r), rows, cols, ld);
  return EAS_OK;
}

eas_status make_map_u8(CUtensorMap* m, const void* base, long long cols, long long rows,
                       long long ld, int box_rows) {
  return make_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, cols, rows, ld, box_rows);
}

size_t elem_size(eas_dtype dt) { return dt == EAS_BF16 ? 2 : dt == EAS_E4M3 ? 1 : 4; }

// ---------------------------------------------------------- workspace layout

struct Layout {
  long long T_pad;
  int vt;              // vocabulary tile width of the forward partials
  int n_vt;
  long long vc;        // vocabulary chunk of the backward
  int n_chunks;
  long long ldz;       // staging row pitch (elements)
  size_t status, sched, head_end;                // cleared at the start of each call
  size_t row_map, pack_of, tile_rows, hp;        // common part
  size_t pm, ps, pu, zt, fwd_counter;             // forward part
  size_t dz, dz2, acc, counters;                  // backward part (two staging buffers)
  size_t fwd_end, bwd_end, total;
};

size_t align_up(size_t x) { return (x + 1023) / 1024 * 1024; }

Layout layout(long long T, long long H, long long V, eas_dtype dt, long long chunk) {
  Layout L;
  const size_t esz = elem_size(dt);
  L.T_pad = round_up(T, 256);
  L.vt = (dt == EAS_FP32) ? kSimtBN : kTcBN;
  L.n_vt = static_cast<int>(cdiv(V, L.vt));
  if (chunk <= 0) chunk = EAS_DEFAULT_VOCAB_CHUNK;
  L.vc = chunk < V ? chunk : V;
  L.n_chunks = static_cast<int>(cdiv(V, L.vc));
  L.ldz = (dt == EAS_BF16) ? round_up(L.vc, kTcBN) : round_up(L.vc, kSimtBN);
  size_t o = 0;
  L.status = o; o = align_up(o + sizeof(DevStatus));
  L.sched = o; o = align_up(o + sizeof(Sched));
  L.head_end = o;
  L.row_map = o; o = align_up(o + 4 * static_cast<size_t>(L.T_pad > 0 ? L.T_pad : 1));
  L.pack_of = o; o = align_up(o + 4 * static_cast<size_t>(T > 0 ? T : 1));
  L.tile_rows = o; o = align_up(o + 8 * static_cast<size_t>(rowmap_tiles(T > 0 ? T : 1)));
  L.hp = o; o = align_up(o + esz * static_cast<size_t>(L.T_pad) * H);
  const size_t common = o;
  L.pm = o; o = align_up(o + 4 * static_cast<size_t>(L.n_vt) * L.T_pad);
  L.ps = o; o = align_up(o + 4 * static_cast<size_t>(L.n_vt) * L.T_pad);
  L.pu = o; o = align_up(o + 4 * static_cast<size_t>(L.n_vt) * L.T_pad);
  L.zt = o; o = align_up(o + 4 * static_cast<size_t>(L.T_pad));
  L.fwd_counter = o; o = align_up(o + sizeof(int));
  L.fwd_end = o;
  o = common;
  L.dz = o; o = align_up(o + esz * static_cast<size_t>(L.T_pad) * L.ldz);
  L.dz2 = o;
  if (dt == EAS_BF16 && L.n_chunks > 1) o = align_up(o + esz * static_cast<size_t>(L.T_pad) * L.ldz);
  L.acc = o;
  if (L.n_chunks > 1) o = align_up(o + 4 * static_cast<size_t>(L.T_pad) * H);
  L.counters = o; o = align_up(o + sizeof(int) * static_cast<size_t>(2 * L.n_chunks + 1));
  L.bwd_end = o;
  L.total = L.fwd_end > L.bwd_end ? L.fwd_end : L.bwd_end;
  return L;
}

// The e4m3 backward's packed e4m3 rows [T_pad][H] (one byte each), placed
// after the bf16 layout, which holds its bf16 packed rows, staging and
// accumulator.
size_t fp8_rows_offset(const Layout& L) { return align_up(L.total); }
size_t fp8_bwd_total(const Layout& L, long long H) {
  return fp8_rows_offset(L) + align_up(static_cast<size_t>(L.T_pad) * static_cast<size_t>(H));
}

// e4m3 operands of the e4m3 backward's recompute.
struct Fp8Operands {
  const uint8_t* hidden;   // [T, H] codes
  const float* hscale;     // [T]
  const uint8_t* weight;   // [V, H] codes
  const float* wscale;     // [V]
};

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

eas_status check_shape(long long T, long long H, long long V, eas_dtype dt) {
  if (T < 0 || T > 0x7fffff00LL) return fail(EAS_ERR_INVALID_ARG, "T=%lld out of range", T);
  if (V < 1 || V > 0x7fffff00LL) return fail(EAS_ERR_INVALID_ARG, "V=%lld out of range", V);
  if (H < 1 || H > (1LL << 20)) return fail(EAS_ERR_INVALID_ARG, "H=%lld out of range", H);
  if (dt != EAS_BF16 && dt != EAS_FP32 && dt != EAS_E4M3)
    return fail(EAS_ERR_INVALID_ARG, "dtype %d", (int)dt);
  if (dt == EAS_E4M3 && H % 128 != 0)
    return fail(EAS_ERR_UNSUPPORTED, "e4m3 path needs H %% 128 == 0 (H=%lld)", H);
  if (dt == EAS_BF16 && H % 64 != 0)
    return fail(EAS_ERR_UNSUPPORTED, "bf16 path needs H %% 64 == 0 (H=%lld)", H);
  if (dt == EAS_FP32 && H % 4 != 0)
    return fail(EAS_ERR_UNSUPPORTED, "fp32 path needs H %% 4 == 0 (H=%lld)", H);
  return EAS_OK;
}

// Common prologue of forward and backward: status clear, span validation and
// row schedule, packed copy of hidden.
// Active tokens' targets must lie in [t_lo, t_hi) (checked on the device).
eas_status prologue(const void* hidden, const uint8_t* mask, const int32_t* spans,
                    const int32_t* num_spans, int64_t cap, long long T, long long H,
                    eas_dtype dt, uint32_t flags, const int32_t* targets, long long t_lo,
                    long long t_hi, void* ws, const Layout& L, const DevInfo& di,
                    cudaStream_t s) {
  {
    Trace tr_(kTrMemset, s);
    EAS_CUDA(cudaMemsetAsync(at<char>(ws, L.status), 0, L.head_end, s), "clear status");
  }
  if (T == 0) return EAS_OK;
  {
    Trace tr_(kTrRowmap, s);
    EAS_CUDA(launch_rowmap(mask, spans, num_spans, cap, T, (flags & EAS_ROWS_SPAN) ? 1 : 0,
                           targets, static_cast<int>(t_lo),
                           static_cast<int>(t_hi < 0x7fffffffLL ? t_hi : 0x7fffffffLL),
                           at<int>(ws, L.row_map), at<int>(ws, L.pack_of),
                           at<long long>(ws, L.tile_rows), at<Sched>(ws, L.sched),
                           at<DevStatus>(ws, L.status), s),
             "rowmap");
  }
  const long long row_bytes = H * static_cast<long long>(elem_size(dt));
  {
    Trace tr_(kTrGather, s);
    EAS_CUDA(launch_gather_rows(hidden, at<char>(ws, L.hp), at<int>(ws, L.row_map),
                                at<Sched>(ws, L.sched), L.T_pad, row_bytes, di.sms, s),
             "gather");
  }
  return EAS_OK;
}

// Raster band height (m-tiles) of a job whose A slab, one m-tile's operand
// over the whole K, is bytes_per_mtile.  While the slabs of a band fit in
// kBandBytes they are meant to stay in L2 while B streams past, and the band
// is as tall as that allows.  When one slab is already larger (dW at large R:
// K = R rows), no slab stays in L2; the band is then kWaveBands m-tiles tall,
// so that the ~76 tiles running at once (4 m-tiles x ~19 n-tiles) share
// their A and B k-blocks as they advance through K together.  On long_256k
// that took the dW DRAM traffic from Hp re-read once per vocabulary tile to
// once per 4, about a third of the step's DRAM bytes, and the step 1.5 %
// faster under the power cap (bands of 8, 12 and 16: 1.2, 1.0 and 0.5 %).
constexpr long long kBandBytes = 48LL << 20;
constexpr int kWaveBands = 4;

int group_for(long long bytes_per_mtile, long long num_m) {
  long long g = bytes_per_mtile > 0 ? kBandBytes / bytes_per_mtile : num_m;
  if (g < 1) g = kWaveBands;
  if (g > num_m) g = num_m;
  return static_cast<int>(g > 0 ? g : 1);
}

int grid_for(long long tiles, int sms) {
  return static_cast<int>(tiles < sms ? tiles : sms);
}

}  // namespace

// =====================================================================
extern "C" {

size_t eas_spans_workspace_size(int64_t T) {
  (void)T;
  return 1024;
}

eas_status eas_build_active_spans(const uint8_t* mask, int64_t T, int32_t max_gap,
                                  int32_t* spans, int64_t cap, int32_t* num_spans, void* ws,
                                  size_t ws_bytes, void* stream) {
  if (T < 0 || T > 0x7fffff00LL) return fail(EAS_ERR_INVALID_ARG, "T=%lld out of range", (long long)T);
  if (max_gap < 0) return fail(EAS_ERR_INVALID_ARG, "max_gap must be >= 0");
  if (cap < 0) return fail(EAS_ERR_INVALID_ARG, "cap must be >= 0");
  if (!num_spans || (T > 0 && !mask) || (cap > 0 && !spans))
    return fail(EAS_ERR_INVALID_ARG, "null pointer");
  if (!ws || ws_bytes < eas_spans_workspace_size(T)) return fail(EAS_ERR_WORKSPACE, "workspace too small");
  if (!aligned(ws, 16)) return fail(EAS_ERR_INVALID_ARG, "workspace not 16-byte aligned");
  DevInfo di;
  eas_status st = device_info(&di);
  if (st != EAS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  {
    Trace tr_(kTrMemset, s);
    EAS_CUDA(cudaMemsetAsync(ws, 0, sizeof(DevStatus), s), "clear status");
  }
  {
    Trace tr_(kTrSpans, s);
    EAS_CUDA(launch_spans_build(mask, T, max_gap, spans, cap, num_spans, static_cast<DevStatus*>(ws), s),
             "spans_build");
  }
  return EAS_OK;
}

size_t eas_lmhead_workspace_size(int64_t T, int64_t H, int64_t V, eas_dtype dtype,
                                 int64_t vocab_chunk) {
  if (T < 0 || H < 1 || V < 1) return 0;
  return layout(T, H, V, dtype, vocab_chunk).total;
}

// Forward of the rows of `weight`, whose first row is vocabulary id t_off.
// With stats == nullptr it writes the final logprob / entropy / lse (the whole
// vocabulary); otherwise it writes each token's shard statistics to stats.
static eas_status fwd_impl(const void* hidden, const void* weight, const int32_t* targets,
                           const uint8_t* mask, const int32_t* spans, const int32_t* num_spans,
                           int64_t cap, int64_t T, int64_t H, int64_t V, eas_dtype dtype,
                           uint32_t flags, float* logprob, float* entropy, float* lse,
                           float* stats, int64_t t_off, const float* hscale,
                           const float* wscale, void* ws, size_t ws_bytes, void* stream) {
  eas_status st = check_shape(T, H, V, dtype);
  if (st != EAS_OK) return st;
  if ((dtype == EAS_E4M3) != (hscale != nullptr && wscale != nullptr))
    return fail(EAS_ERR_INVALID_ARG,
                "e4m3 operands are taken (with their scales) by eas_lmhead_fwd_fp8 only");
  if (flags > 1u) return fail(EAS_ERR_INVALID_ARG, "unknown flags %u", flags);
  if (cap < 0) return fail(EAS_ERR_INVALID_ARG, "cap must be >= 0");
  if (!weight || !num_spans || !ws) return fail(EAS_ERR_INVALID_ARG, "null pointer");
  if (T > 0 && (!hidden || !targets || !mask || (cap > 0 && !spans)))
    return fail(EAS_ERR_INVALID_ARG, "null pointer");
  if (T > 0 && (stats ? !aligned(stats, 16) : (!logprob || !entropy)))
    return fail(EAS_ERR_INVALID_ARG, "null or misaligned output");
  if (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(ws, 256))
    return fail(EAS_ERR_INVALID_ARG, "hidden/weight must be 16-byte and ws 256-byte aligned");
  const Layout L = layout(T, H, V, dtype, 0);
  if (ws_bytes < L.fwd_end) return fail(EAS_ERR_WORKSPACE, "workspace %zu < %zu", ws_bytes, L.fwd_end);
  DevInfo di;
  st = device_info(&di);
  if (st != EAS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  st = prologue(hidden, mask, spans, num_spans, cap, T, H, dtype, flags, targets, 0,
                stats ? 0x7fffffffLL : static_cast<long long>(V), ws, L, di, s);
  if (st != EAS_OK || T == 0) return st;
  const Sched* sched = at<Sched>(ws, L.sched);
  const long long num_m_max = L.T_pad / tc_tile_rows();

  if (dtype == EAS_BF16 || dtype == EAS_E4M3) {
    const bool fp8 = (dtype == EAS_E4M3);
    TcArgs a;
    memset(&a, 0, sizeof(a));
    TcJob& j = a.jobs[0];
    st = fp8 ? make_map_u8(&j.tmA, at<char>(ws, L.hp), H, L.T_pad, H, 128)
             : make_map_bf16(&j.tmA, at<char>(ws, L.hp), H, L.T_pad, H, 128);
    if (st != EAS_OK) return st;
    st = fp8 ? make_map_u8(&j.tmB, weight, H, V, H, 128)
             : make_map_bf16(&j.tmB, weight, H, V, H, tc_tile_rows() == 256 ? 128 : 256);
    if (st != EAS_OK) return st;
    j.kind = fp8 ? kTcFwdFp8 : kTcFwd;
    a.hscale = hscale;
    a.wscale = wscale;
    j.M_fixed = 0;
    j.N = static_cast<int>(V);
    j.K_fixed = static_cast<int>(H);
    j.group_m = group_for(tc_tile_rows() * H * static_cast<long long>(elem_size(dtype)), num_m_max);
    a.n_jobs = 1;
    a.sched = sched;
    a.status = at<DevStatus>(ws, L.status);
    a.tile_counter = at<int>(ws, L.fwd_counter);
    a.budget = wait_budget();
    a.row_map = at<int>(ws, L.row_map);
    a.targets = targets;
    a.t_off = static_cast<int>(t_off);
    a.part_m = at<float>(ws, L.pm);
    a.part_s = at<float>(ws, L.ps);
    a.part_u = at<float>(ws, L.pu);
    a.zt = at<float>(ws, L.zt);
    a.part_stride = L.T_pad;
    a.V = static_cast<int>(V);
    a.H = static_cast<int>(H);
    {
      Trace tr_(kTrMemset, s);
      EAS_CUDA(cudaMemsetAsync(at<char>(ws, L.fwd_counter), 0, sizeof(int), s), "clear counter");
    }
    {
      Trace tr_(kTrFwdGemm, s);
      EAS_CUDA(launch_tc_gemm(a, grid_for(num_m_max * L.n_vt, di.sms), s), "fwd gemm");
    }
  } else {
    SimtArgs a;
    memset(&a, 0, sizeof(a));
    a.kind = kTcFwd;
    a.A = at<float>(ws, L.hp);
    a.lda = H;
    a.B = static_cast<const float*>(weight);
    a.ldb = H;
    a.sched = sched;
    a.M_fixed = 0;
    a.N = static_cast<int>(V);
    a.K_fixed = static_cast<int>(H);
    a.row_map = at<int>(ws, L.row_map);
    a.targets = targets;
    a.t_off = static_cast<int>(t_off);
    a.part_m = at<float>(ws, L.pm);
    a.part_s = at<float>(ws, L.ps);
    a.part_u = at<float>(ws, L.pu);
    a.zt = at<float>(ws, L.zt);
    a.part_stride = L.T_pad;
    a.V = static_cast<int>(V);
    a.H = static_cast<int>(H);
    {
      Trace tr_(kTrSimtFwd, s);
      EAS_CUDA(launch_simt_gemm(a, cdiv(L.T_pad, kSimtBM) * L.n_vt, s), "fwd simt");
    }
  }
  {
    Trace tr_(kTrCombine, s);
    if (stats) {
      EAS_CUDA(launch_combine_stats(at<float>(ws, L.pm), at<float>(ws, L.ps), at<float>(ws, L.pu),
                                    at<float>(ws, L.zt), L.n_vt, L.T_pad, at<int>(ws, L.pack_of),
                                    mask, targets, static_cast<int>(t_off), static_cast<int>(V), T,
                                    reinterpret_cast<float4*>(stats), di.sms, s),
               "combine stats");
    } else {
      EAS_CUDA(launch_combine(at<float>(ws, L.pm), at<float>(ws, L.ps), at<float>(ws, L.pu),
                              at<float>(ws, L.zt), L.n_vt, L.T_pad, at<int>(ws, L.pack_of), mask, T,
                              logprob, entropy, lse, di.sms, s),
               "combine");
    }
  }
  return EAS_OK;
}

eas_status eas_lmhead_fwd(const void* hidden, const void* weight, const int32_t* targets,
                          const uint8_t* mask, const int32_t* spans, const int32_t* num_spans,
                          int64_t cap, int64_t T, int64_t H, int64_t V, eas_dtype dtype,
                          uint32_t flags, float* logprob, float* entropy, float* lse, void* ws,
                          size_t ws_bytes, void* stream) {
  return fwd_impl(hidden, weight, targets, mask, spans, num_spans, cap, T, H, V, dtype, flags,
                  logprob, entropy, lse, nullptr, 0, nullptr, nullptr, ws, ws_bytes, stream);
}

eas_status eas_lmhead_fwd_fp8(const uint8_t* hidden_e4m3, const float* hidden_scale,
                              const uint8_t* weight_e4m3, const float* weight_scale,
                              const int32_t* targets, const uint8_t* mask, const int32_t* spans,
                              const int32_t* num_spans, int64_t cap, int64_t T, int64_t H,
                              int64_t V, uint32_t flags, float* logprob, float* entropy,
                              float* lse, void* ws, size_t ws_bytes, void* stream) {
  if (!weight_scale || (T > 0 && !hidden_scale)) return fail(EAS_ERR_INVALID_ARG, "null scale");
  return fwd_impl(hidden_e4m3, weight_e4m3, targets, mask, spans, num_spans, cap, T, H, V,
                  EAS_E4M3, flags, logprob, entropy, lse, nullptr, 0,
                  hidden_scale ? hidden_scale : weight_scale, weight_scale, ws, ws_bytes, stream);
}

eas_status eas_quantize_rows_e4m3(const void* src, eas_dtype src_dtype, int64_t R, int64_t H,
                                  uint8_t* dst, float* scale, void* stream) {
  if (src_dtype != EAS_BF16 && src_dtype != EAS_FP32)
    return fail(EAS_ERR_INVALID_ARG, "source must be bf16 or fp32");
  if (R < 0 || H < 1) return fail(EAS_ERR_INVALID_ARG, "bad shape");
  if (R > 0 && (!src || !dst || !scale)) return fail(EAS_ERR_INVALID_ARG, "null pointer");
  DevInfo di;
  eas_status st = device_info(&di);
  if (st != EAS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  EAS_CUDA(launch_quantize_rows_e4m3(src, src_dtype == EAS_BF16, R, H, dst, scale, di.sms, s),
           "quantize");
  return EAS_OK;
}

eas_status eas_lmhead_fwd_shard(const void* hidden, const void* weight_shard, int64_t v_lo,
                                const int32_t* targets, const uint8_t* mask, const int32_t* spans,
                                const int32_t* num_spans, int64_t cap, int64_t T, int64_t H,
                                int64_t V_shard, eas_dtype dtype, uint32_t flags, float* stats,
                                void* ws, size_t ws_bytes, void* stream) {
  if (v_lo < 0 || v_lo > 0x7fffff00LL) return fail(EAS_ERR_INVALID_ARG, "v_lo out of range");
  if (T > 0 && !stats) return fail(EAS_ERR_INVALID_ARG, "null stats");
  return fwd_impl(hidden, weight_shard, targets, mask, spans, num_spans, cap, T, H, V_shard, dtype,
                  flags, nullptr, nullptr, nullptr, stats, v_lo, nullptr, nullptr, ws, ws_bytes,
                  stream);
}

eas_status eas_lmhead_combine_shards(const float* stats, int32_t n_shards, int64_t T,
                                     const uint8_t* mask, float* logprob, float* entropy,
                                     float* lse, void* stream) {
  if (n_shards < 1) return fail(EAS_ERR_INVALID_ARG, "n_shards must be >= 1");
  if (T < 0 || T > 0x7fffff00LL) return fail(EAS_ERR_INVALID_ARG, "T out of range");
  if (T > 0 && (!stats || !mask || !logprob || !entropy))
    return fail(EAS_ERR_INVALID_ARG, "null pointer");
  if (T > 0 && !aligned(stats, 16)) return fail(EAS_ERR_INVALID_ARG, "stats not 16-byte aligned");
  DevInfo di;
  eas_status st = device_info(&di);
  if (st != EAS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Trace tr_(kTrCombine, s);
  EAS_CUDA(launch_combine_shards(reinterpret_cast<const float4*>(stats), n_shards, T, mask,
                                 logprob, entropy, lse, di.sms, s),
           "combine shards");
  return EAS_OK;
}

// Backward through the rows of `weight`, whose first row is vocabulary id
// t_off (0 for the whole vocabulary).
static eas_status bwd_impl(const float* g_logprob, const float* g_entropy, const void* hidden,
                           const void* weight, const int32_t* targets, const uint8_t* mask,
                           const int32_t* spans, const int32_t* num_spans, int64_t cap,
                           const float* lse, const float* entropy, int64_t T, int64_t H, int64_t V,
                           eas_dtype dtype, uint32_t flags, int64_t vocab_chunk, void* dhidden,
                           float* dweight, int64_t t_off, bool sharded, const Fp8Operands* f8,
                           void* ws, size_t ws_bytes, void* stream) {
  eas_status st = check_shape(T, H, V, dtype);
  if (st != EAS_OK) return st;
  if (dtype == EAS_E4M3)
    return fail(EAS_ERR_UNSUPPORTED,
                "the backward takes bf16 or fp32 operands (e4m3: eas_lmhead_bwd_fp8)");
  if (f8) {
    if (dtype != EAS_BF16) return fail(EAS_ERR_INVALID_ARG, "the e4m3 backward projects in bf16");
    if (H % 128 != 0)
      return fail(EAS_ERR_UNSUPPORTED, "e4m3 path needs H %% 128 == 0 (H=%lld)", (long long)H);
    if (flags & EAS_REUSE_FWD_ROWS)
      return fail(EAS_ERR_INVALID_ARG,
                  "the e4m3 backward packs its own rows (EAS_REUSE_FWD_ROWS not accepted)");
    if (T > 0 && (!f8->hidden || !f8->hscale)) return fail(EAS_ERR_INVALID_ARG, "null pointer");
    if (!f8->weight || !f8->wscale) return fail(EAS_ERR_INVALID_ARG, "null pointer");
    if (!aligned(f8->hidden, 16) || !aligned(f8->weight, 16))
      return fail(EAS_ERR_INVALID_ARG, "e4m3 operands must be 16-byte aligned");
  }
  const bool reuse = (flags & EAS_REUSE_FWD_ROWS) != 0;
  flags &= ~EAS_REUSE_FWD_ROWS;
  if (flags > 1u) return fail(EAS_ERR_INVALID_ARG, "unknown flags %u", flags);
  if (cap < 0) return fail(EAS_ERR_INVALID_ARG, "cap must be >= 0");
  if (vocab_chunk < 0) return fail(EAS_ERR_INVALID_ARG, "vocab_chunk must be >= 0");
  if (!weight || !dweight || !num_spans || !ws) return fail(EAS_ERR_INVALID_ARG, "null pointer");
  if (T > 0 && (!hidden || !targets || !mask || !g_logprob || !g_entropy || !lse || !entropy ||
                !dhidden || (cap > 0 && !spans)))
    return fail(EAS_ERR_INVALID_ARG, "null pointer");
  if (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(dhidden, 16) ||
      !aligned(dweight, 16) || !aligned(ws, 256))
    return fail(EAS_ERR_INVALID_ARG, "tensors must be 16-byte and ws 256-byte aligned");
  const Layout L = layout(T, H, V, dtype, vocab_chunk);
  const size_t need = f8 ? fp8_bwd_total(L, H) : L.bwd_end;
  if (ws_bytes < need) return fail(EAS_ERR_WORKSPACE, "workspace %zu < %zu", ws_bytes, need);
  DevInfo di;
  st = device_info(&di);
  if (st != EAS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (!reuse) {
    st = prologue(hidden, mask, spans, num_spans, cap, T, H, dtype, flags, targets, 0,
                  sharded ? 0x7fffffffLL : static_cast<long long>(V), ws, L, di, s);
    if (st != EAS_OK) return st;
  }
  if (f8 && T > 0) {
    Trace tr_(kTrGather, s);
    EAS_CUDA(launch_gather_rows(f8->hidden, at<char>(ws, fp8_rows_offset(L)),
                                at<int>(ws, L.row_map), at<Sched>(ws, L.sched), L.T_pad, H,
                                di.sms, s),
             "gather e4m3 rows");
  }
  // (with reuse, the row schedule and packed rows of the preceding forward
  // stay where that call's layout put them: the shared part of the layout
  // does not depend on vocab_chunk; the status word is kept)
  {
    Trace tr_(kTrMemset, s);
    EAS_CUDA(cudaMemsetAsync(at<char>(ws, L.counters), 0, sizeof(int) * (2 * L.n_chunks + 1), s),
             "clear counters");
  }
  if (T == 0) {
    {
      Trace tr_(kTrMemset, s);
      EAS_CUDA(cudaMemsetAsync(dweight, 0, sizeof(float) * V * H, s), "zero dW");
    }
    return EAS_OK;
  }
  const size_t esz = (dtype == EAS_BF16) ? 2 : 4;
  {
    Trace tr_(kTrZeroRows, s);
    EAS_CUDA(launch_zero_unpacked_rows(dhidden, at<int>(ws, L.pack_of), T, H * esz, di.sms, s),
             "zero rows");
  }
  const Sched* sched = at<Sched>(ws, L.sched);
  const long long num_m_max = L.T_pad / tc_tile_rows();

  if (dtype == EAS_BF16) {
    CUtensorMap hp_k, w_k, w_mn, hp_mn;
    if ((st = make_map_bf16(&hp_k, at<char>(ws, L.hp), H, L.T_pad, H, 128)) != EAS_OK) return st;
    if ((st = make_map_bf16(&w_k, weight, H, V, H, tc_tile_rows() == 256 ? 128 : 256)) != EAS_OK)
      return st;
    if ((st = make_map_bf16_mn3(&w_mn, weight, H, V, H)) != EAS_OK) return st;
    if ((st = make_map_bf16_mn3(&hp_mn, at<char>(ws, L.hp), H, L.T_pad, H)) != EAS_OK) return st;
    TcArgs base;
    memset(&base, 0, sizeof(base));
    base.sched = sched;
    base.status = at<DevStatus>(ws, L.status);
    base.budget = wait_budget();
    base.row_map = at<int>(ws, L.row_map);
    base.targets = targets;
    base.t_off = static_cast<int>(t_off);
    base.mask = mask;
    base.lse = lse;
    base.ent = entropy;
    base.g_lp = g_logprob;
    base.g_h = g_entropy;
    base.V = static_cast<int>(V);
    base.H = static_cast<int>(H);
    base.ldz = L.ldz;
    base.acc = at<float>(ws, L.acc);
    base.dhidden = dhidden;
    base.dW = dweight;
    void* staging[2] = {at<char>(ws, L.dz), at<char>(ws, L.n_chunks > 1 ? L.dz2 : L.dz)};
    // dW and dHidden of chunk p, reading staging buffer p%2
    auto add_projections = [&](TcArgs& a, int p, long long& tiles) -> eas_status {
      const long long v0 = p * L.vc;
      const long long live = (V - v0) < L.vc ? (V - v0) : L.vc;
      void* dz = staging[p % 2];
      CUtensorMap dz_k, dz_mn;
      eas_status e;
      if ((e = make_map_bf16(&dz_k, dz, live, L.T_pad, L.ldz, 128)) != EAS_OK) return e;
      if ((e = make_map_bf16_mn3(&dz_mn, dz, live, L.T_pad, L.ldz)) != EAS_OK) return e;
      TcJob& w = a.jobs[a.n_jobs++];
      w.tmA = dz_mn;
      w.tmB = hp_mn;
      w.kind = kTcDWeight;
      w.M_fixed = static_cast<int>(live);
      w.N = static_cast<int>(H);
      w.K_fixed = 0;
      w.group_m = group_for(tc_tile_rows() * L.T_pad * 2LL, cdiv(live, tc_tile_rows()));
      w.v0 = static_cast<int>(v0);
      w.vc_live = static_cast<int>(live);
      tiles += cdiv(live, tc_tile_rows()) * cdiv(H, kTcBN);
      TcJob& h = a.jobs[a.n_jobs++];
      h.tmA = dz_k;
      h.tmB = w_mn;
      h.kind = kTcDHidden;
      h.M_fixed = 0;
      h.N = static_cast<int>(H);
      h.K_fixed = static_cast<int>(live);
      h.group_m = group_for(tc_tile_rows() * live * 2LL, num_m_max);
      h.v0 = static_cast<int>(v0);
      h.vc_live = static_cast<int>(live);
      h.first_chunk = (p == 0);
      if (p != L.n_chunks - 1 &&
          (e = make_map_2d(&h.tmD, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, at<float>(ws, L.acc), H,
                           L.T_pad, H, 32)) != EAS_OK)
        return e;
      h.last_chunk = (p == L.n_chunks - 1);
      tiles += num_m_max * cdiv(H, kTcBN);
      return EAS_OK;
    };
    // d-logits of chunk c into staging buffer c%2, from bf16 or e4m3 operands
    auto add_dlogits = [&](TcArgs& a, int c, long long& tiles, bool e4m3,
                           const CUtensorMap& tmA, const CUtensorMap& tmB) -> eas_status {
      const long long v0 = c * L.vc;
      const long long live = (V - v0) < L.vc ? (V - v0) : L.vc;
      TcJob& d = a.jobs[a.n_jobs++];
      d.tmA = tmA;
      d.tmB = tmB;
      d.kind = e4m3 ? kTcDLogitsFp8 : kTcDLogits;
      d.M_fixed = 0;
      d.N = static_cast<int>(live);
      d.K_fixed = static_cast<int>(H);
      d.group_m = group_for(tc_tile_rows() * H * (e4m3 ? 1LL : 2LL), num_m_max);
      d.v0 = static_cast<int>(v0);
      d.vc_live = static_cast<int>(live);
      eas_status e = make_map_bf16(&d.tmD, staging[c % 2], L.ldz, L.T_pad, L.ldz, 32);
      if (e != EAS_OK) return e;
      tiles += num_m_max * cdiv(live, kTcBN);
      return EAS_OK;
    };
    if (!f8) {
      // Launch c (0..n) runs dW and dHidden of chunk c-1 (reading staging
      // buffer (c-1)%2) next to the d-logits of chunk c (writing buffer c%2):
      // the jobs of one launch are independent and share the machine, and
      // each launch boundary orders a chunk's d-logits before its projections.
      for (int c = 0; c <= L.n_chunks; ++c) {
        TcArgs a = base;
        a.tile_counter = at<int>(ws, L.counters) + c;
        long long tiles = 0;
        int trace_kind = kTrDLogitsGemm;
        // projections of the previous chunk: dW (longest tiles when R is
        // large) and dHidden first, the short d-logits tiles last
        if (c > 0) {
          if ((st = add_projections(a, c - 1, tiles)) != EAS_OK) return st;
          trace_kind = kTrDProjGemm;
        }
        if (c < L.n_chunks) {
          if ((st = add_dlogits(a, c, tiles, false, hp_k, w_k)) != EAS_OK) return st;
          if (c > 0) trace_kind = kTrBwdChunkGemm;
        }
        Trace tr_(trace_kind, s);
        EAS_CUDA(launch_tc_gemm(a, grid_for(tiles, di.sms), s), "backward gemm");
      }
    } else {
      // e4m3 recompute: the d-logits GEMM runs in its own instantiation, so
      // each chunk is two launches, the e4m3 d-logits, then dW and dHidden
      CUtensorMap hp8_k, w8_k;
      if ((st = make_map_u8(&hp8_k, at<char>(ws, fp8_rows_offset(L)), H, L.T_pad, H, 128)) !=
          EAS_OK)
        return st;
      if ((st = make_map_u8(&w8_k, f8->weight, H, V, H, 128)) != EAS_OK) return st;
      for (int c = 0; c < L.n_chunks; ++c) {
        {
          TcArgs a = base;
          a.tile_counter = at<int>(ws, L.counters) + 2 * c;
          a.hscale = f8->hscale;
          a.wscale = f8->wscale;
          long long tiles = 0;
          if ((st = add_dlogits(a, c, tiles, true, hp8_k, w8_k)) != EAS_OK) return st;
          Trace tr_(kTrDLogitsFp8Gemm, s);
          EAS_CUDA(launch_tc_gemm(a, grid_for(tiles, di.sms), s), "backward gemm (e4m3)");
        }
        {
          TcArgs a = base;
          a.tile_counter = at<int>(ws, L.counters) + 2 * c + 1;
          long long tiles = 0;
          if ((st = add_projections(a, c, tiles)) != EAS_OK) return st;
          Trace tr_(kTrDProjGemm, s);
          EAS_CUDA(launch_tc_gemm(a, grid_for(tiles, di.sms), s), "backward gemm");
        }
      }
    }
  } else {
    SimtArgs base;
    memset(&base, 0, sizeof(base));
    base.sched = sched;
    base.row_map = at<int>(ws, L.row_map);
    base.targets = targets;
    base.t_off = static_cast<int>(t_off);
    base.mask = mask;
    base.lse = lse;
    base.ent = entropy;
    base.g_lp = g_logprob;
    base.g_h = g_entropy;
    base.V = static_cast<int>(V);
    base.H = static_cast<int>(H);
    base.dz = at<float>(ws, L.dz);
    base.ldz = L.ldz;
    base.acc = at<float>(ws, L.acc);
    base.dhidden = static_cast<float*>(dhidden);
    base.dW = dweight;
    for (int c = 0; c < L.n_chunks; ++c) {
      const long long v0 = c * L.vc;
      const long long live = (V - v0) < L.vc ? (V - v0) : L.vc;
      SimtArgs a = base;
      a.kind = kTcDLogits;
      a.A = at<float>(ws, L.hp);
      a.lda = H;
      a.B = static_cast<const float*>(weight);
      a.ldb = H;
      a.M_fixed = 0;
      a.N = static_cast<int>(live);
      a.K_fixed = static_cast<int>(H);
      a.v0 = static_cast<int>(v0);
      a.vc_live = static_cast<int>(live);
      {
        Trace tr_(kTrSimtDLogits, s);
        EAS_CUDA(launch_simt_gemm(a, cdiv(L.T_pad, kSimtBM) * cdiv(live, kSimtBN), s), "dlogits simt");
      }
      SimtArgs h = base;
      h.kind = kTcDHidden;
      h.A = at<float>(ws, L.dz);
      h.lda = L.ldz;
      h.B = static_cast<const float*>(weight);
      h.ldb = H;
      h.M_fixed = 0;
      h.N = static_cast<int>(H);
      h.K_fixed = static_cast<int>(live);
      h.v0 = static_cast<int>(v0);
      h.vc_live = static_cast<int>(live);
      h.first_chunk = (c == 0);
      h.last_chunk = (c == L.n_chunks - 1);
      {
        Trace tr_(kTrSimtDHidden, s);
        EAS_CUDA(launch_simt_gemm(h, cdiv(L.T_pad, kSimtBM) * cdiv(H, kSimtBN), s), "dhidden simt");
      }
      SimtArgs w = base;
      w.kind = kTcDWeight;
      w.A = at<float>(ws, L.dz);
      w.lda = L.ldz;
      w.B = at<float>(ws, L.hp);
      w.ldb = H;
      w.M_fixed = static_cast<int>(live);
      w.N = static_cast<int>(H);
      w.K_fixed = 0;
      w.v0 = static_cast<int>(v0);
      w.vc_live = static_cast<int>(live);
      {
        Trace tr_(kTrSimtDWeight, s);
        EAS_CUDA(launch_simt_gemm(w, cdiv(live, kSimtBM) * cdiv(H, kSimtBN), s), "dweight simt");
      }
    }
  }
  return EAS_OK;
}

eas_status eas_lmhead_bwd(const float* g_logprob, const float* g_entropy, const void* hidden,
                          const void* weight, const int32_t* targets, const uint8_t* mask,
                          const int32_t* spans, const int32_t* num_spans, int64_t cap,
                          const float* lse, const float* entropy, int64_t T, int64_t H, int64_t V,
                          eas_dtype dtype, uint32_t flags, int64_t vocab_chunk, void* dhidden,
                          float* dweight, void* ws, size_t ws_bytes, void* stream) {
  return bwd_impl(g_logprob, g_entropy, hidden, weight, targets, mask, spans, num_spans, cap, lse,
                  entropy, T, H, V, dtype, flags, vocab_chunk, dhidden, dweight, 0, false, nullptr,
                  ws, ws_bytes, stream);
}

size_t eas_lmhead_bwd_fp8_workspace_size(int64_t T, int64_t H, int64_t V, int64_t vocab_chunk) {
  if (T < 0 || H < 1 || V < 1) return 0;
  return fp8_bwd_total(layout(T, H, V, EAS_BF16, vocab_chunk), H);
}

eas_status eas_lmhead_bwd_fp8(const float* g_logprob, const float* g_entropy, const void* hidden,
                              const void* weight, const uint8_t* hidden_e4m3,
                              const float* hidden_scale, const uint8_t* weight_e4m3,
                              const float* weight_scale, const int32_t* targets,
                              const uint8_t* mask, const int32_t* spans, const int32_t* num_spans,
                              int64_t cap, const float* lse, const float* entropy, int64_t T,
                              int64_t H, int64_t V, uint32_t flags, int64_t vocab_chunk,
                              void* dhidden, float* dweight, void* ws, size_t ws_bytes,
                              void* stream) {
  const Fp8Operands f8{hidden_e4m3, hidden_scale, weight_e4m3, weight_scale};
  return bwd_impl(g_logprob, g_entropy, hidden, weight, targets, mask, spans, num_spans, cap, lse,
                  entropy, T, H, V, EAS_BF16, flags, vocab_chunk, dhidden, dweight, 0, false, &f8,
                  ws, ws_bytes, stream);
}

eas_status eas_lmhead_bwd_shard(const float* g_logprob, const float* g_entropy,
                                const void* hidden, const void* weight_shard, int64_t v_lo,
                                const int32_t* targets, const uint8_t* mask, const int32_t* spans,
                                const int32_t* num_spans, int64_t cap, const float* lse,
                                const float* entropy, int64_t T, int64_t H, int64_t V_shard,
                                eas_dtype dtype, uint32_t flags, int64_t vocab_chunk,
                                void* dhidden_partial, float* dweight_shard, void* ws,
                                size_t ws_bytes, void* stream) {
  if (v_lo < 0 || v_lo > 0x7fffff00LL) return fail(EAS_ERR_INVALID_ARG, "v_lo out of range");
  return bwd_impl(g_logprob, g_entropy, hidden, weight_shard, targets, mask, spans, num_spans, cap,
                  lse, entropy, T, H, V_shard, dtype, flags, vocab_chunk, dhidden_partial,
                  dweight_shard, v_lo, true, nullptr, ws, ws_bytes, stream);
}

eas_status eas_cp_local_layout(const uint8_t* mask, const int32_t* seg_offsets, int32_t n_segs,
                               int64_t T, int32_t cp_size, int32_t cp_rank, uint8_t* local_mask,
                               int32_t* local_to_global, void* ws, size_t ws_bytes,
                               void* stream) {
  if (T < 0 || T > 0x7fffff00LL) return fail(EAS_ERR_INVALID_ARG, "T out of range");
  if (cp_size < 1 || cp_rank < 0 || cp_rank >= cp_size)
    return fail(EAS_ERR_INVALID_ARG, "cp_rank %d outside [0, cp_size=%d)", cp_rank, cp_size);
  if (T % (2LL * cp_size) != 0)
    return fail(EAS_ERR_INVALID_ARG, "T=%lld is not a multiple of 2*cp_size", (long long)T);
  if (n_segs < 1) return fail(EAS_ERR_INVALID_ARG, "n_segs must be >= 1");
  if (!seg_offsets || (T > 0 && (!mask || !local_mask || !local_to_global)))
    return fail(EAS_ERR_INVALID_ARG, "null pointer");
  if (!ws || ws_bytes < sizeof(DevStatus)) return fail(EAS_ERR_WORKSPACE, "workspace too small");
  if (!aligned(ws, 16)) return fail(EAS_ERR_INVALID_ARG, "workspace not 16-byte aligned");
  DevInfo di;
  eas_status st = device_info(&di);
  if (st != EAS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  EAS_CUDA(cudaMemsetAsync(ws, 0, sizeof(DevStatus), s), "clear status");
  EAS_CUDA(launch_cp_local(mask, seg_offsets, n_segs, T, cp_size, cp_rank, local_mask,
                           local_to_global, static_cast<DevStatus*>(ws), di.sms, s),
           "cp layout");
  return EAS_OK;
}

eas_status eas_selftest_wait_timeout(int64_t budget_cycles, void* ws, size_t ws_bytes,
                                     void* stream) {
  if (budget_cycles < 1 || budget_cycles > (1LL << 34))
    return fail(EAS_ERR_INVALID_ARG, "budget_cycles out of range");
  if (!ws || ws_bytes < sizeof(DevStatus)) return fail(EAS_ERR_WORKSPACE, "workspace too small");
  if (!aligned(ws, 16)) return fail(EAS_ERR_INVALID_ARG, "workspace not 16-byte aligned");
  DevInfo di;
  eas_status st = device_info(&di);
  if (st != EAS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  EAS_CUDA(cudaMemsetAsync(ws, 0, sizeof(DevStatus), s), "clear status");
  EAS_CUDA(launch_selftest_wait(budget_cycles, static_cast<DevStatus*>(ws), s), "selftest");
  return EAS_OK;
}

eas_status eas_read_device_status(const void* ws, void* stream) {
  if (!ws) return fail(EAS_ERR_INVALID_ARG, "null workspace");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevStatus h;
  EAS_CUDA(cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, s), "read status");
  EAS_CUDA(cudaStreamSynchronize(s), "stream sync");
  if (h.code != 0)
    return fail(static_cast<eas_status>(h.code), "device status %d (where %d, info %d)", h.code,
                h.where, h.info);
  return EAS_OK;
}

void eas_trace_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  g_trace_on.store(on != 0, std::memory_order_relaxed);
  if (on != 0) g_trace_used = 0;
}

int32_t eas_trace_read(int32_t* kinds, float* ms, int32_t cap) {
  std::lock_guard<std::mutex> lk(g_trace_mu);
  const int32_t n = static_cast<int32_t>(g_trace_used);
  for (int32_t i = 0; i < n && i < cap; ++i) {
    const TraceRec& r = g_trace_pool[i];
    float t = -1.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
      t = -1.f;
    if (kinds) kinds[i] = r.kind;
    if (ms) ms[i] = t;
  }
  return n;
}

const char* eas_kernel_name(int32_t kind) {
  return (kind >= 0 && kind < kTrCount) ? kTraceNames[kind] : "unknown";
}

const char* eas_last_error(void) { return g_err; }

const char* eas_status_string(eas_status s) {
  switch (s) {
    case EAS_OK: return "EAS_OK";
    case EAS_ERR_INVALID_ARG: return "EAS_ERR_INVALID_ARG";
    case EAS_ERR_INVALID_SPANS: return "EAS_ERR_INVALID_SPANS";
    case EAS_ERR_UNSUPPORTED: return "EAS_ERR_UNSUPPORTED";
    case EAS_ERR_WORKSPACE: return "EAS_ERR_WORKSPACE";
    case EAS_ERR_CUDA: return "EAS_ERR_CUDA";
    case EAS_ERR_TIMEOUT: return "EAS_ERR_TIMEOUT";
    case EAS_ERR_SPAN_CAPACITY: return "EAS_ERR_SPAN_CAPACITY";
    case EAS_ERR_INVALID_LAYOUT: return "EAS_ERR_INVALID_LAYOUT";
  }
  return "EAS_UNKNOWN";
}

int32_t eas_version(void) { return 100; }

}  // extern "C"

namespace eas {

// Forward-only workspace requirement (the larger backward part excluded).
size_t lmhead_fwd_workspace_bytes(long long T, long long H, long long V, int dtype) {
  if (T < 0 || H < 1 || V < 1) return 0;
  return layout(T, H, V, static_cast<eas_dtype>(dtype), 0).fwd_end;
}

// Replaces this thread's eas_last_error() message.
void set_last_error(const char* msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }

}  // namespace eas
