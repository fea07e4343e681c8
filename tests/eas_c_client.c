/*
 * A plain C (C11) caller of the library's C ABI (include/eas.h), so the boundary
 * is exercised by something other than the Python binding.
 *
 *   eas_c_client host
 *       host-side checks only (no GPU touched): version, workspace sizes,
 *       argument errors returned before any device work.
 *   eas_c_client run DIR T H V
 *       reads DIR/hidden.bf16 [T,H], DIR/weight.bf16 [V,H], DIR/targets.i32,
 *       DIR/mask.u8, DIR/glp.f32, DIR/gh.f32 [T]; builds the spans (max gap
 *       128), runs the forward and the backward on the GPU in bf16 and writes
 *       DIR/{logprob,entropy,lse}.f32 [T], DIR/dhidden.bf16 [T,H],
 *       DIR/dweight.f32 [V,H] and DIR/spans.i32 (the span count, then the
 *       start/end pairs).
 * Exit status 0 on success; on failure a line naming the call and the
 * library's error text goes to stderr.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "eas.h"

static int fail(const char* what, eas_status st) {
  fprintf(stderr, "%s: %s (%s)\n", what, eas_status_string(st), eas_last_error());
  return 1;
}

static int cuda_fail(const char* what, cudaError_t e) {
  fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
  return 1;
}

static int host_checks(void) {
  eas_status st;
  if (eas_version() <= 0) return fail("eas_version", EAS_OK);
  if (eas_spans_workspace_size(1024) == 0) return fail("eas_spans_workspace_size", EAS_OK);
  if (eas_lmhead_workspace_size(1024, 128, 1000, EAS_BF16, 0) == 0)
    return fail("eas_lmhead_workspace_size", EAS_OK);
  /* a negative token count is rejected before any device work */
  st = eas_lmhead_fwd(NULL, NULL, NULL, NULL, NULL, NULL, 0, -1, 128, 1000, EAS_BF16,
                      EAS_ROWS_ACTIVE, NULL, NULL, NULL, NULL, 0, NULL);
  if (st != EAS_ERR_INVALID_ARG) return fail("eas_lmhead_fwd(T=-1)", st);
  if (eas_last_error()[0] == '\0') return fail("eas_last_error", st);
  /* H not a multiple of 64 is not supported in bf16 */
  st = eas_lmhead_fwd(NULL, NULL, NULL, NULL, NULL, NULL, 0, 16, 100, 1000, EAS_BF16,
                      EAS_ROWS_ACTIVE, NULL, NULL, NULL, NULL, 0, NULL);
  if (st != EAS_ERR_UNSUPPORTED) return fail("eas_lmhead_fwd(H=100)", st);
  if (eas_status_string(EAS_OK) == NULL) return fail("eas_status_string", EAS_OK);
  printf("host checks ok, version %d\n", (int)eas_version());
  return 0;
}

static void* read_file(const char* dir, const char* name, size_t bytes) {
  char path[4096];
  FILE* f;
  void* p = malloc(bytes > 0 ? bytes : 1);
  snprintf(path, sizeof(path), "%s/%s", dir, name);
  f = fopen(path, "rb");
  if (!f || !p || fread(p, 1, bytes, f) != bytes) {
    fprintf(stderr, "cannot read %zu bytes from %s\n", bytes, path);
    exit(1);
  }
  fclose(f);
  return p;
}

static void write_file(const char* dir, const char* name, const void* p, size_t bytes) {
  char path[4096];
  FILE* f;
  snprintf(path, sizeof(path), "%s/%s", dir, name);
  f = fopen(path, "wb");
  if (!f || fwrite(p, 1, bytes, f) != bytes) {
    fprintf(stderr, "cannot write %s\n", path);
    exit(1);
  }
  fclose(f);
}

/* device buffer of `bytes`, holding a copy of `h` unless h is NULL */
static int to_device(void** d, const void* h, size_t bytes) {
  cudaError_t e = cudaMalloc(d, bytes > 0 ? bytes : 1);
  if (e != cudaSuccess) return cuda_fail("cudaMalloc", e);
  if (bytes > 0 && h != NULL) {
    e = cudaMemcpy(*d, h, bytes, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail("cudaMemcpy to device", e);
  }
  return 0;
}

static int to_host(void* h, const void* d, size_t bytes) {
  cudaError_t e = cudaMemcpy(h, d, bytes, cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? 0 : cuda_fail("cudaMemcpy to host", e);
}

static int run(const char* dir, int64_t T, int64_t H, int64_t V) {
  const size_t th = (size_t)(T * H), vh = (size_t)(V * H);
  const int64_t cap = (T + 1) / 2;
  void *hidden = read_file(dir, "hidden.bf16", th * 2), *weight = read_file(dir, "weight.bf16", vh * 2);
  void *targets = read_file(dir, "targets.i32", (size_t)T * 4), *mask = read_file(dir, "mask.u8", (size_t)T);
  void *glp = read_file(dir, "glp.f32", (size_t)T * 4), *gh = read_file(dir, "gh.f32", (size_t)T * 4);
  void *d_hidden, *d_weight, *d_targets, *d_mask, *d_glp, *d_gh;
  void *d_spans, *d_ns, *d_sws, *d_ws, *d_lp, *d_ent, *d_lse, *d_dh, *d_dw;
  const size_t sws_bytes = eas_spans_workspace_size(T);
  const size_t ws_bytes = eas_lmhead_workspace_size(T, H, V, EAS_BF16, 0);
  eas_status st;
  cudaError_t e;
  int32_t ns = 0;
  float* out;
  int32_t* spans_h;

  if (to_device(&d_hidden, hidden, th * 2) || to_device(&d_weight, weight, vh * 2) ||
      to_device(&d_targets, targets, (size_t)T * 4) || to_device(&d_mask, mask, (size_t)T) ||
      to_device(&d_glp, glp, (size_t)T * 4) || to_device(&d_gh, gh, (size_t)T * 4) ||
      to_device(&d_spans, NULL, (size_t)cap * 8) || to_device(&d_ns, NULL, 4) ||
      to_device(&d_sws, NULL, sws_bytes) || to_device(&d_ws, NULL, ws_bytes) ||
      to_device(&d_lp, NULL, (size_t)T * 4) || to_device(&d_ent, NULL, (size_t)T * 4) ||
      to_device(&d_lse, NULL, (size_t)T * 4) || to_device(&d_dh, NULL, th * 2) ||
      to_device(&d_dw, NULL, vh * 4))
    return 1;

  st = eas_build_active_spans((const uint8_t*)d_mask, T, 128, (int32_t*)d_spans, cap,
                              (int32_t*)d_ns, d_sws, sws_bytes, NULL);
  if (st != EAS_OK) return fail("eas_build_active_spans", st);
  st = eas_read_device_status(d_sws, NULL);
  if (st != EAS_OK) return fail("span status", st);

  st = eas_lmhead_fwd(d_hidden, d_weight, (const int32_t*)d_targets, (const uint8_t*)d_mask,
                      (const int32_t*)d_spans, (const int32_t*)d_ns, cap, T, H, V, EAS_BF16,
                      EAS_ROWS_ACTIVE, (float*)d_lp, (float*)d_ent, (float*)d_lse, d_ws, ws_bytes,
                      NULL);
  if (st != EAS_OK) return fail("eas_lmhead_fwd", st);
  st = eas_read_device_status(d_ws, NULL);
  if (st != EAS_OK) return fail("forward status", st);

  st = eas_lmhead_bwd((const float*)d_glp, (const float*)d_gh, d_hidden, d_weight,
                      (const int32_t*)d_targets, (const uint8_t*)d_mask, (const int32_t*)d_spans,
                      (const int32_t*)d_ns, cap, (const float*)d_lse, (const float*)d_ent, T, H,
                      V, EAS_BF16, EAS_ROWS_ACTIVE, 0, d_dh, (float*)d_dw, d_ws, ws_bytes, NULL);
  if (st != EAS_OK) return fail("eas_lmhead_bwd", st);
  st = eas_read_device_status(d_ws, NULL);
  if (st != EAS_OK) return fail("backward status", st);
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail("cudaDeviceSynchronize", e);

  out = (float*)malloc(vh * 4 > th * 2 ? vh * 4 : th * 2);
  if (!out) return 1;
  if (to_host(out, d_lp, (size_t)T * 4)) return 1;
  write_file(dir, "logprob.f32", out, (size_t)T * 4);
  if (to_host(out, d_ent, (size_t)T * 4)) return 1;
  write_file(dir, "entropy.f32", out, (size_t)T * 4);
  if (to_host(out, d_lse, (size_t)T * 4)) return 1;
  write_file(dir, "lse.f32", out, (size_t)T * 4);
  if (to_host(out, d_dh, th * 2)) return 1;
  write_file(dir, "dhidden.bf16", out, th * 2);
  if (to_host(out, d_dw, vh * 4)) return 1;
  write_file(dir, "dweight.f32", out, vh * 4);
  if (to_host(&ns, d_ns, 4)) return 1;
  spans_h = (int32_t*)malloc(((size_t)cap * 2 + 1) * 4);
  if (!spans_h) return 1;
  spans_h[0] = ns;
  if (ns > 0 && to_host(spans_h + 1, d_spans, (size_t)ns * 8)) return 1;
  write_file(dir, "spans.i32", spans_h, ((size_t)ns * 2 + 1) * 4);
  printf("ran T=%lld H=%lld V=%lld, %d spans\n", (long long)T, (long long)H, (long long)V, (int)ns);
  return 0;
}

int main(int argc, char** argv) {
  if (argc == 2 && strcmp(argv[1], "host") == 0) return host_checks();
  if (argc == 6 && strcmp(argv[1], "run") == 0)
    return run(argv[2], atoll(argv[3]), atoll(argv[4]), atoll(argv[5]));
  fprintf(stderr, "usage: eas_c_client host | run DIR T H V\n");
  return 2;
}
