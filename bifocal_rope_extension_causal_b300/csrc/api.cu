// C ABI of libjetlong.so (declared in include/jetlong.h): argument
// validation, workspace carving, and the launches of the CUDA path.  The
// library allocates no device memory; every buffer is the caller's.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "../../include/jetlong.h"
#include "internal.h"
#include "positions.cuh"
#include "rope_math.cuh"

namespace jl {

__device__ int g_device_status = 0;

int* device_status_ptr() {
  int* ptr = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_device_status) != cudaSuccess) return nullptr;
  return ptr;
}

namespace {

thread_local char t_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof(t_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(JL_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

float resolve_scale(float s, int d) { return s > 0.f ? s : 1.0f / sqrtf(static_cast<float>(d)); }

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace

int set_error(int code, const char* msg) { return fail(code, "%s", msg); }

RopeFreqs make_rope_freqs(int d, double theta) {
  RopeFreqs f{};
  for (int i = 0; i < d / 2 && i < kMaxHalfDim; ++i) f.w[i] = pow(theta, -2.0 * i / d);
  return f;
}

AngleTable make_angle_table(int d, double theta) {
  AngleTable t{};
  const RopeFreqs f = make_rope_freqs(d, theta);
  for (int i = 0; i < d / 2 && i < kMaxHalfDim; ++i) {
    for (int l = 0; l < 3; ++l) {
      // x = 2^(10 l) omega exactly; r = x mod 2 pi in [-pi, pi], with 2 pi as
      // the nearest double plus its remainder (each fma rounds once).
      const double x = ldexp(f.w[i], 10 * l);
      const double m = rint(x / kTwoPiHi);
      double r = fma(-m, kTwoPiHi, x);
      r = fma(-m, kTwoPiLo, r);
      uint32_t bits;
      float hi = static_cast<float>(r);
      memcpy(&bits, &hi, 4);
      bits &= 0xfffffc00u;  // 14 significant bits
      memcpy(&hi, &bits, 4);
      t.hi[l][i] = hi;
      t.lo[l][i] = static_cast<float>(r - static_cast<double>(hi));
    }
  }
  return t;
}

}  // namespace jl

using namespace jl;

extern "C" {

int64_t jl_group_size(int64_t L, int64_t w_pretrained) {
  if (L < 0 || w_pretrained <= 0) return -1;
  return jl::group_size(L, w_pretrained);
}

size_t jl_bifocal_prefill_workspace_size(int B, int L, int Hq, int Hkv, int d, int w_pretrained) {
  if (B < 1 || L < 1 || Hq < 1 || Hkv < 1 || d < 1 || w_pretrained < 1) return 0;
  const bool bif = jl::group_size(L, w_pretrained) > 1;
  const size_t qbytes = align_up(static_cast<size_t>(B) * Hq * L * d * 2);
  const size_t kbytes = align_up(static_cast<size_t>(B) * Hkv * L * d * 2);
  return (bif ? 2 : 1) * (qbytes + kbytes) + align_up(rope_table_bytes(d));
}

namespace {

// Shared validation of the prefill-family arguments; 0 if fine.
int check_prefill_shape(const char* who, int B, int L, int Hq, int Hkv, int d, int w0,
                        int w_pretrained) {
  if (B < 1 || L < 1 || Hq < 1 || Hkv < 1)
    return fail(JL_ERR_INVALID, "%s: need B, L, Hq, Hkv >= 1 (got %d, %d, %d, %d)", who, B, L, Hq, Hkv);
  if (Hq % Hkv != 0) return fail(JL_ERR_INVALID, "%s: Hq %% Hkv != 0 (%d, %d)", who, Hq, Hkv);
  if (w0 < 0 || w_pretrained < 1) return fail(JL_ERR_INVALID, "%s: need w0 >= 0, w_pretrained >= 1", who);
  if (d != 64 && d != 128) return fail(JL_ERR_UNSUPPORTED, "%s: head dim %d (supported: 64, 128)", who, d);
  if (L > kMaxRopePosition)
    return fail(JL_ERR_UNSUPPORTED, "%s: positions up to 2^30 - 1 are supported (L = %d)", who, L);
  return JL_OK;
}

int check_workspace(const char* who, const void* ws, size_t bytes, size_t need) {
  if (!ws || bytes < need || (reinterpret_cast<uintptr_t>(ws) % kAlign))
    return fail(JL_ERR_WORKSPACE, "%s: workspace needs %zu bytes, 256-byte aligned (got %zu)", who, need,
                bytes);
  return JL_OK;
}

// Workspace carving: Q_abs, K_abs, then (G > 1) Q_rem, K_rem, then the
// rotation tables.
struct PrefillWs {
  unsigned char *qa, *ka, *qr, *kr, *tables;
};
PrefillWs carve(const void* workspace, int B, int L, int Hq, int Hkv, int d, bool bif) {
  auto* ws = static_cast<unsigned char*>(const_cast<void*>(workspace));
  const size_t qbytes = align_up(static_cast<size_t>(B) * Hq * L * d * 2);
  const size_t kbytes = align_up(static_cast<size_t>(B) * Hkv * L * d * 2);
  PrefillWs w;
  w.qa = ws;
  w.ka = ws + qbytes;
  w.qr = bif ? ws + qbytes + kbytes : w.qa;
  w.kr = bif ? ws + 2 * qbytes + kbytes : w.ka;
  w.tables = ws + (bif ? 2 : 1) * (qbytes + kbytes);
  return w;
}

}  // namespace

int jl_bifocal_rope(const void* q, const void* k, int B, int L, int Hq, int Hkv, int d,
                    int w_pretrained, double rope_theta, void* k_rot_out, void* workspace,
                    size_t workspace_bytes, void* cuda_stream) {
  t_err[0] = '\0';
  if (!q || !k) return fail(JL_ERR_INVALID, "rope: null q/k pointer");
  int rc = check_prefill_shape("rope", B, L, Hq, Hkv, d, 0, w_pretrained);
  if (rc != JL_OK) return rc;
  if (!(rope_theta > 0.0) || !isfinite(rope_theta)) return fail(JL_ERR_INVALID, "rope: rope_theta must be > 0");
  if (!aligned16(q) || !aligned16(k) || (k_rot_out && !aligned16(k_rot_out)))
    return fail(JL_ERR_INVALID, "rope: every pointer must be 16-byte aligned");
  rc = check_workspace("rope", workspace, workspace_bytes,
                       jl_bifocal_prefill_workspace_size(B, L, Hq, Hkv, d, w_pretrained));
  if (rc != JL_OK) return rc;
  const int G = static_cast<int>(jl::group_size(L, w_pretrained));
  const bool bif = G > 1;
  const PrefillWs w = carve(workspace, B, L, Hq, Hkv, d, bif);
  auto stream = static_cast<cudaStream_t>(cuda_stream);
  const RopeFreqs fr = make_rope_freqs(d, rope_theta);
  const TensorView none{nullptr, 0, 0, 0, 0};
  cudaError_t e = launch_rope_tables(w.tables, d, fr, stream);
  if (e != cudaSuccess) return cuda_fail(e, "rope: rotation tables");
  e = launch_rope_prepass(q, B, L, Hq, d, G, 0, w.tables, head_major(w.qa, Hq, L, d),
                          bif ? head_major(w.qr, Hq, L, d) : none, none, stream);
  if (e != cudaSuccess) return cuda_fail(e, "rope: pre-pass (Q)");
  e = launch_rope_prepass(k, B, L, Hkv, d, G, 0, w.tables, head_major(w.ka, Hkv, L, d),
                          bif ? head_major(w.kr, Hkv, L, d) : none,
                          k_rot_out ? cache_layout(k_rot_out, L, Hkv, d, L) : none, stream);
  if (e != cudaSuccess) return cuda_fail(e, "rope: pre-pass (K)");
  return JL_OK;
}

}  // extern "C"

namespace {

// jl_bifocal_attention with a given pipeline wait limit (0: the default) and
// kernel (cta_pair: the CTA-pair kernel, head dim 128).
int attention_call(const void* v, void* o, float* lse, int B, int L, int Hq, int Hkv, int d, int w0,
                   int w_pretrained, float softmax_scale, const void* workspace, size_t workspace_bytes,
                   long long wait_limit, bool cta_pair, void* cuda_stream) {
  if (!v || !o) return fail(JL_ERR_INVALID, "attention: null v/o pointer");
  int rc = check_prefill_shape("attention", B, L, Hq, Hkv, d, w0, w_pretrained);
  if (rc != JL_OK) return rc;
  if (!aligned16(v) || !aligned16(o) || (lse && !aligned16(lse)))
    return fail(JL_ERR_INVALID, "attention: every pointer must be 16-byte aligned");
  rc = check_workspace("attention", workspace, workspace_bytes,
                       jl_bifocal_prefill_workspace_size(B, L, Hq, Hkv, d, w_pretrained));
  if (rc != JL_OK) return rc;
  const int G = static_cast<int>(jl::group_size(L, w_pretrained));
  const PrefillWs w = carve(workspace, B, L, Hq, Hkv, d, G > 1);
  PrefillArgs a;
  a.qa = head_major(w.qa, Hq, L, d);
  a.qr = head_major(w.qr, Hq, L, d);
  a.ka = head_major(w.ka, Hkv, L, d);
  a.kr = head_major(w.kr, Hkv, L, d);
  a.v = cache_layout(v, L, Hkv, d, L);
  a.o = o; a.lse = lse;
  a.B = B; a.Lq = L; a.Lk = L; a.q_base = 0; a.Hq = Hq; a.Hkv = Hkv; a.d = d; a.w0 = w0; a.G = G;
  a.scale_log2 = resolve_scale(softmax_scale, d) * kLog2e;
  a.wait_limit = wait_limit;
  a.cta_pair = cta_pair;
  const cudaError_t e = launch_prefill_attention(a, static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return cuda_fail(e, "attention: kernel launch");
  return JL_OK;
}

}  // namespace

extern "C" {

int jl_bifocal_attention(const void* v, void* o, float* lse, int B, int L, int Hq, int Hkv, int d,
                         int w0, int w_pretrained, float softmax_scale, const void* workspace,
                         size_t workspace_bytes, void* cuda_stream) {
  t_err[0] = '\0';
  return attention_call(v, o, lse, B, L, Hq, Hkv, d, w0, w_pretrained, softmax_scale, workspace, workspace_bytes,
                        0, false, cuda_stream);
}

int jl_bifocal_attention_cta_pair(const void* v, void* o, float* lse, int B, int L, int Hq, int Hkv, int d,
                                  int w0, int w_pretrained, float softmax_scale, const void* workspace,
                                  size_t workspace_bytes, void* cuda_stream) {
  t_err[0] = '\0';
  if (d != 128) return fail(JL_ERR_UNSUPPORTED, "attention_cta_pair: head dim 128 only (d = %d)", d);
  return attention_call(v, o, lse, B, L, Hq, Hkv, d, w0, w_pretrained, softmax_scale, workspace, workspace_bytes,
                        0, true, cuda_stream);
}

}  // extern "C"

namespace {

int selftest_wait_limit(const void* q, const void* k, const void* v, void* o, float* lse, int B, int L, int Hq,
                        int Hkv, int d, int w0, int w_pretrained, double rope_theta, long long limit_cycles,
                        void* workspace, size_t workspace_bytes, bool cta_pair, void* cuda_stream) {
  if (limit_cycles < 1 || limit_cycles > 4000000000LL)
    return fail(JL_ERR_INVALID, "selftest: limit_cycles must be in [1, 4e9]");
  if (!q || !k || !v || !o) return fail(JL_ERR_INVALID, "selftest: null q/k/v/o pointer");
  if (cta_pair && d != 128) return fail(JL_ERR_UNSUPPORTED, "selftest: the CTA-pair kernel takes head dim 128 only");
  int rc = jl_bifocal_rope(q, k, B, L, Hq, Hkv, d, w_pretrained, rope_theta, nullptr, workspace,
                           workspace_bytes, cuda_stream);
  if (rc != JL_OK) return rc;
  return attention_call(v, o, lse, B, L, Hq, Hkv, d, w0, w_pretrained, 0.f, workspace, workspace_bytes,
                        limit_cycles, cta_pair, cuda_stream);
}

}  // namespace

extern "C" {

int jl_selftest_prefill_wait_limit(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                   int L, int Hq, int Hkv, int d, int w0, int w_pretrained, double rope_theta,
                                   long long limit_cycles, void* workspace, size_t workspace_bytes,
                                   void* cuda_stream) {
  t_err[0] = '\0';
  return selftest_wait_limit(q, k, v, o, lse, B, L, Hq, Hkv, d, w0, w_pretrained, rope_theta, limit_cycles,
                             workspace, workspace_bytes, false, cuda_stream);
}

int jl_selftest_prefill_pair_wait_limit(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                        int L, int Hq, int Hkv, int d, int w0, int w_pretrained,
                                        double rope_theta, long long limit_cycles, void* workspace,
                                        size_t workspace_bytes, void* cuda_stream) {
  t_err[0] = '\0';
  return selftest_wait_limit(q, k, v, o, lse, B, L, Hq, Hkv, d, w0, w_pretrained, rope_theta, limit_cycles,
                             workspace, workspace_bytes, true, cuda_stream);
}

int jl_bifocal_prefill(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int L, int Hq, int Hkv, int d, int w0, int w_pretrained, double rope_theta,
                       float softmax_scale, void* k_rot_out, void* workspace,
                       size_t workspace_bytes, void* cuda_stream) {
  t_err[0] = '\0';
  if (!q || !k || !v || !o) return fail(JL_ERR_INVALID, "prefill: null q/k/v/o pointer");
  int rc = check_prefill_shape("prefill", B, L, Hq, Hkv, d, w0, w_pretrained);
  if (rc != JL_OK) return rc;
  if (!aligned16(v) || !aligned16(o) || (lse && !aligned16(lse)))
    return fail(JL_ERR_INVALID, "prefill: every pointer must be 16-byte aligned");
  rc = jl_bifocal_rope(q, k, B, L, Hq, Hkv, d, w_pretrained, rope_theta, k_rot_out, workspace,
                       workspace_bytes, cuda_stream);
  if (rc != JL_OK) return rc;
  return jl_bifocal_attention(v, o, lse, B, L, Hq, Hkv, d, w0, w_pretrained, softmax_scale,
                              workspace, workspace_bytes, cuda_stream);
}

size_t jl_bifocal_prefill_three_pass_workspace_size(int B, int L, int Hq, int Hkv, int d,
                                                    int w_pretrained) {
  const size_t base = jl_bifocal_prefill_workspace_size(B, L, Hq, Hkv, d, w_pretrained);
  if (base == 0) return 0;
  const size_t obytes = align_up(static_cast<size_t>(B) * L * Hq * d * 2);
  const size_t lbytes = align_up(static_cast<size_t>(B) * Hq * L * sizeof(float));
  return base + 2 * obytes + 3 * lbytes;
}

int jl_bifocal_prefill_three_pass(const void* q, const void* k, const void* v, void* o, float* lse,
                                  int B, int L, int Hq, int Hkv, int d, int w0, int w_pretrained,
                                  double rope_theta, float softmax_scale, void* workspace,
                                  size_t workspace_bytes, void* cuda_stream) {
  t_err[0] = '\0';
  if (!q || !k || !v || !o) return fail(JL_ERR_INVALID, "three_pass: null q/k/v/o pointer");
  int rc = check_prefill_shape("three_pass", B, L, Hq, Hkv, d, w0, w_pretrained);
  if (rc != JL_OK) return rc;
  if (!aligned16(v) || !aligned16(o) || (lse && !aligned16(lse)))
    return fail(JL_ERR_INVALID, "three_pass: every pointer must be 16-byte aligned");
  rc = check_workspace("three_pass", workspace, workspace_bytes,
                       jl_bifocal_prefill_three_pass_workspace_size(B, L, Hq, Hkv, d, w_pretrained));
  if (rc != JL_OK) return rc;
  rc = jl_bifocal_rope(q, k, B, L, Hq, Hkv, d, w_pretrained, rope_theta, nullptr, workspace,
                       workspace_bytes, cuda_stream);
  if (rc != JL_OK) return rc;
  auto stream = static_cast<cudaStream_t>(cuda_stream);
  const int G = static_cast<int>(jl::group_size(L, w_pretrained));
  const PrefillWs w = carve(workspace, B, L, Hq, Hkv, d, G > 1);
  auto* extra = static_cast<unsigned char*>(workspace) +
                jl_bifocal_prefill_workspace_size(B, L, Hq, Hkv, d, w_pretrained);
  const size_t obytes = align_up(static_cast<size_t>(B) * L * Hq * d * 2);
  const size_t lbytes = align_up(static_cast<size_t>(B) * Hq * L * sizeof(float));
  void* o_a = extra;
  void* o_c = extra + obytes;
  float* lse_a = reinterpret_cast<float*>(extra + 2 * obytes);
  float* lse_b = reinterpret_cast<float*>(extra + 2 * obytes + lbytes);
  float* lse_c = reinterpret_cast<float*>(extra + 2 * obytes + 2 * lbytes);

  PrefillArgs a;
  a.v = cache_layout(v, L, Hkv, d, L);
  a.B = B; a.Lq = L; a.Lk = L; a.q_base = 0; a.Hq = Hq; a.Hkv = Hkv; a.d = d; a.G = G;
  a.scale_log2 = resolve_scale(softmax_scale, d) * kLog2e;
  const TensorView q_abs = head_major(w.qa, Hq, L, d), q_rem = head_major(w.qr, Hq, L, d);
  const TensorView k_abs = head_major(w.ka, Hkv, L, d), k_rem = head_major(w.kr, Hkv, L, d);
  // A: local window, absolute rotations.
  a.qa = a.qr = q_abs; a.ka = a.kr = k_abs;
  a.w0 = w0; a.window_only = true; a.o = o_a; a.lse = lse_a;
  cudaError_t e = launch_prefill_attention(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "three_pass: pass A");
  // B: every causal key, aliased rotations (w0 = L: all pairs in one phase).
  a.qa = a.qr = q_rem; a.ka = a.kr = k_rem;
  a.w0 = L; a.window_only = false; a.o = o; a.lse = lse_b;
  e = launch_prefill_attention(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "three_pass: pass B");
  // C: local window, aliased rotations.
  a.w0 = w0; a.window_only = true; a.o = o_c; a.lse = lse_c;
  e = launch_prefill_attention(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "three_pass: pass C");
  e = launch_three_pass_merge(o_a, lse_a, o, lse_b, o_c, lse_c, lse, B, L, Hq, d, stream);
  if (e != cudaSuccess) return cuda_fail(e, "three_pass: merge");
  return JL_OK;
}

namespace {

// Copy streams and events of the host-buffer prefill, created once per
// device (the library never allocates device memory).
constexpr int kPipeEvents = 256;
struct HostPipe {
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t ev[kPipeEvents] = {};
  int next = 0;
};
constexpr int kPipeDevices = 64;
std::mutex g_pipe_mu;      // creation of the per-device pipes
std::mutex g_enqueue_mu;   // one host thread at a time enqueues (shares the event pool)
HostPipe g_pipe[kPipeDevices];

HostPipe* host_pipe(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kPipeDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe& p = g_pipe[dev];
  if (!p.ready) {
    if ((*err = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking)) != cudaSuccess) return nullptr;
    if ((*err = cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking)) != cudaSuccess) return nullptr;
    for (int i = 0; i < kPipeEvents; ++i)
      if ((*err = cudaEventCreateWithFlags(&p.ev[i], cudaEventDisableTiming)) != cudaSuccess) return nullptr;
    p.ready = true;
  }
  return &p;
}

// Device buffers of the host-buffer prefill after the prefill workspace:
// q, k, v, o copies ([B, L, H, d] bf16) and the log-sum-exp staging (chunk c
// of sequence b as [Hq][rows] at b * Hq * L + c * Hq * C floats).
struct HostWs {
  unsigned char *q, *k, *v, *o;
  float* lse;
};
HostWs carve_host(void* workspace, int B, int L, int Hq, int Hkv, int d, int w_pretrained) {
  auto* ws = static_cast<unsigned char*>(workspace) + jl_bifocal_prefill_workspace_size(B, L, Hq, Hkv, d, w_pretrained);
  const size_t qb = align_up(static_cast<size_t>(B) * L * Hq * d * 2);
  const size_t kb = align_up(static_cast<size_t>(B) * L * Hkv * d * 2);
  HostWs h;
  h.q = ws;
  h.k = ws + qb;
  h.v = ws + qb + kb;
  h.o = ws + qb + 2 * kb;
  h.lse = reinterpret_cast<float*>(ws + 2 * qb + 2 * kb);
  return h;
}

TensorView rows_of(TensorView t, int r0, int rows, int d) {
  t.base = static_cast<const unsigned char*>(t.base) + static_cast<size_t>(r0) * d * 2;
  t.rows = rows;
  return t;
}

}  // namespace

size_t jl_bifocal_prefill_host_workspace_size(int B, int L, int Hq, int Hkv, int d, int w_pretrained) {
  const size_t base = jl_bifocal_prefill_workspace_size(B, L, Hq, Hkv, d, w_pretrained);
  if (base == 0) return 0;
  const size_t qb = align_up(static_cast<size_t>(B) * L * Hq * d * 2);
  const size_t kb = align_up(static_cast<size_t>(B) * L * Hkv * d * 2);
  return base + 2 * qb + 2 * kb + align_up(static_cast<size_t>(B) * Hq * L * sizeof(float));
}

int jl_bifocal_prefill_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                            float* lse_host, int B, int L, int Hq, int Hkv, int d, int w0, int w_pretrained,
                            double rope_theta, float softmax_scale, int n_chunks, void* workspace,
                            size_t workspace_bytes, void* cuda_stream) {
  t_err[0] = '\0';
  if (!q_host || !k_host || !v_host || !o_host) return fail(JL_ERR_INVALID, "prefill_host: null q/k/v/o pointer");
  int rc = check_prefill_shape("prefill_host", B, L, Hq, Hkv, d, w0, w_pretrained);
  if (rc != JL_OK) return rc;
  if (!(rope_theta > 0.0) || !isfinite(rope_theta)) return fail(JL_ERR_INVALID, "prefill_host: rope_theta must be > 0");
  if (n_chunks < 0) return fail(JL_ERR_INVALID, "prefill_host: n_chunks must be >= 0");
  rc = check_workspace("prefill_host", workspace, workspace_bytes,
                       jl_bifocal_prefill_host_workspace_size(B, L, Hq, Hkv, d, w_pretrained));
  if (rc != JL_OK) return rc;
  cudaError_t e = cudaSuccess;
  HostPipe* pipe = host_pipe(&e);
  if (pipe == nullptr) return cuda_fail(e, "prefill_host: copy streams");
  auto stream = static_cast<cudaStream_t>(cuda_stream);
  std::lock_guard<std::mutex> lock(g_enqueue_mu);
  auto event = [&]() {
    cudaEvent_t ev = pipe->ev[pipe->next];
    pipe->next = (pipe->next + 1) % kPipeEvents;
    return ev;
  };
  // Query chunks of C rows, C a multiple of 256 (the attention kernel's
  // query-tile pair), so each chunk's tiles are those of a single call.
  const int nc_req = n_chunks > 0 ? n_chunks : std::min(16, std::max(1, L / 8192));
  int C = (L + nc_req - 1) / nc_req;
  C = (C + 255) / 256 * 256;
  const int nc = (L + C - 1) / C;

  const int G = static_cast<int>(jl::group_size(L, w_pretrained));
  const bool bif = G > 1;
  const PrefillWs w = carve(workspace, B, L, Hq, Hkv, d, bif);
  const HostWs h = carve_host(workspace, B, L, Hq, Hkv, d, w_pretrained);
  const RopeFreqs fr = make_rope_freqs(d, rope_theta);
  const TensorView none{nullptr, 0, 0, 0, 0};
  const size_t qrow = static_cast<size_t>(Hq) * d * 2, krow = static_cast<size_t>(Hkv) * d * 2;
  const float scale_log2 = resolve_scale(softmax_scale, d) * kLog2e;

  // The copy streams start after the work already queued on the caller's stream.
  cudaEvent_t ev = event();
  if ((e = cudaEventRecord(ev, stream)) != cudaSuccess) return cuda_fail(e, "prefill_host: event");
  cudaStreamWaitEvent(pipe->h2d, ev, 0);
  cudaStreamWaitEvent(pipe->d2h, ev, 0);
  // Every exit from here on (errors included) makes the caller's stream wait
  // for both copy streams, so no copy is still in flight on the workspace or
  // the host buffers once that stream has synchronised.
  auto join = [&]() {
    cudaEvent_t j = event();
    cudaEventRecord(j, pipe->d2h);
    cudaStreamWaitEvent(stream, j, 0);
    j = event();
    cudaEventRecord(j, pipe->h2d);
    cudaStreamWaitEvent(stream, j, 0);
  };
  auto fail_joined = [&](cudaError_t err, const char* what) {
    join();
    return cuda_fail(err, what);
  };
  if ((e = launch_rope_tables(w.tables, d, fr, stream)) != cudaSuccess) return fail_joined(e, "prefill_host: tables");
  for (int b = 0; b < B; ++b) {
    const size_t qoff = static_cast<size_t>(b) * L * qrow, koff = static_cast<size_t>(b) * L * krow;
    const TensorView qa = head_major(w.qa + static_cast<size_t>(b) * Hq * L * d * 2, Hq, L, d);
    const TensorView qr = head_major(w.qr + static_cast<size_t>(b) * Hq * L * d * 2, Hq, L, d);
    const TensorView ka = head_major(w.ka + static_cast<size_t>(b) * Hkv * L * d * 2, Hkv, L, d);
    const TensorView kr = head_major(w.kr + static_cast<size_t>(b) * Hkv * L * d * 2, Hkv, L, d);
    for (int c = 0; c < nc; ++c) {
      const int r0 = c * C, rows = std::min(C, L - r0);
      // 1. Chunk rows of q, k, v in.
      const size_t qo = qoff + static_cast<size_t>(r0) * qrow, ko = koff + static_cast<size_t>(r0) * krow;
      e = cudaMemcpyAsync(h.q + qo, static_cast<const unsigned char*>(q_host) + qo, rows * qrow,
                          cudaMemcpyHostToDevice, pipe->h2d);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(h.k + ko, static_cast<const unsigned char*>(k_host) + ko, rows * krow,
                            cudaMemcpyHostToDevice, pipe->h2d);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(h.v + ko, static_cast<const unsigned char*>(v_host) + ko, rows * krow,
                            cudaMemcpyHostToDevice, pipe->h2d);
      if (e != cudaSuccess) return fail_joined(e, "prefill_host: copy in");
      ev = event();
      cudaEventRecord(ev, pipe->h2d);
      cudaStreamWaitEvent(stream, ev, 0);
      // 2. Rotations of the chunk's rows (the call's G).
      e = launch_rope_prepass(h.q + qo, 1, rows, Hq, d, G, r0, w.tables, rows_of(qa, r0, rows, d),
                              bif ? rows_of(qr, r0, rows, d) : none, none, stream);
      if (e == cudaSuccess)
        e = launch_rope_prepass(h.k + ko, 1, rows, Hkv, d, G, r0, w.tables, rows_of(ka, r0, rows, d),
                                bif ? rows_of(kr, r0, rows, d) : none, none, stream);
      if (e != cudaSuccess) return fail_joined(e, "prefill_host: pre-pass");
      // 3. The chunk's query rows over keys 0 .. r0 + rows - 1.
      PrefillArgs a;
      a.qa = rows_of(qa, r0, rows, d);
      a.qr = bif ? rows_of(qr, r0, rows, d) : a.qa;
      a.ka = rows_of(ka, 0, r0 + rows, d);
      a.kr = bif ? rows_of(kr, 0, r0 + rows, d) : a.ka;
      a.v = cache_layout(h.v + koff, L, Hkv, d, r0 + rows);
      a.o = h.o + qo;
      float* lse_stage = h.lse + static_cast<size_t>(b) * Hq * L + static_cast<size_t>(c) * Hq * C;
      a.lse = lse_host ? lse_stage : nullptr;
      a.B = 1; a.Lq = rows; a.Lk = r0 + rows; a.q_base = r0; a.Hq = Hq; a.Hkv = Hkv; a.d = d; a.w0 = w0; a.G = G;
      a.scale_log2 = scale_log2;
      if ((e = launch_prefill_attention(a, stream)) != cudaSuccess) return fail_joined(e, "prefill_host: attention");
      ev = event();
      cudaEventRecord(ev, stream);
      cudaStreamWaitEvent(pipe->d2h, ev, 0);
      // 4. The chunk's outputs out.
      e = cudaMemcpyAsync(static_cast<unsigned char*>(o_host) + qo, h.o + qo, rows * qrow, cudaMemcpyDeviceToHost,
                          pipe->d2h);
      if (e == cudaSuccess && lse_host)
        e = cudaMemcpy2DAsync(lse_host + static_cast<size_t>(b) * Hq * L + r0, static_cast<size_t>(L) * sizeof(float),
                              lse_stage, static_cast<size_t>(rows) * sizeof(float), rows * sizeof(float), Hq,
                              cudaMemcpyDeviceToHost, pipe->d2h);
      if (e != cudaSuccess) return fail_joined(e, "prefill_host: copy out");
    }
  }
  // The caller's stream resumes after the last copy out (and the last copy in).
  join();
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "prefill_host: stream ordering");
  return JL_OK;
}

size_t jl_bifocal_prefill_chunk_workspace_size(int B, int C, int P0, int Hq, int Hkv, int d,
                                               int w_pretrained) {
  if (B < 1 || C < 1 || P0 < 0 || Hq < 1 || Hkv < 1 || d < 1 || w_pretrained < 1) return 0;
  const int Lk = P0 + C;
  const bool bif = jl::group_size(Lk, w_pretrained) > 1;
  const size_t qbytes = align_up(static_cast<size_t>(B) * Hq * C * d * 2);
  const size_t krbytes = align_up(static_cast<size_t>(B) * Hkv * Lk * d * 2);
  return (bif ? 2 : 1) * qbytes + (bif ? krbytes : 0) + align_up(rope_table_bytes(d));
}

int jl_bifocal_prefill_chunk(const void* q, const void* k, const void* v, void* k_cache, void* v_cache,
                             int P0, int Lcap, void* o, float* lse, int B, int C, int Hq, int Hkv, int d,
                             int w0, int w_pretrained, double rope_theta, float softmax_scale,
                             void* workspace, size_t workspace_bytes, void* cuda_stream) {
  t_err[0] = '\0';
  if (!q || !k || !v || !k_cache || !v_cache || !o)
    return fail(JL_ERR_INVALID, "prefill_chunk: null q/k/v/cache/o pointer");
  if (C < 1 || P0 < 0) return fail(JL_ERR_INVALID, "prefill_chunk: need C >= 1 and P0 >= 0");
  if (static_cast<long long>(P0) + C > Lcap)
    return fail(JL_ERR_INVALID, "prefill_chunk: P0 + C = %lld exceeds Lcap = %d", static_cast<long long>(P0) + C, Lcap);
  if (static_cast<long long>(P0) + C > kMaxRopePosition)
    return fail(JL_ERR_UNSUPPORTED, "prefill_chunk: positions up to 2^30 - 1 are supported");
  int rc = check_prefill_shape("prefill_chunk", B, C, Hq, Hkv, d, w0, w_pretrained);
  if (rc != JL_OK) return rc;
  if (!(rope_theta > 0.0) || !isfinite(rope_theta))
    return fail(JL_ERR_INVALID, "prefill_chunk: rope_theta must be > 0");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(o) || (lse && !aligned16(lse)))
    return fail(JL_ERR_INVALID, "prefill_chunk: every pointer must be 16-byte aligned");
  rc = check_workspace("prefill_chunk", workspace, workspace_bytes,
                       jl_bifocal_prefill_chunk_workspace_size(B, C, P0, Hq, Hkv, d, w_pretrained));
  if (rc != JL_OK) return rc;
  const int Lk = P0 + C;
  const int G = static_cast<int>(jl::group_size(Lk, w_pretrained));
  const bool bif = G > 1;
  auto* ws = static_cast<unsigned char*>(workspace);
  const size_t qbytes = align_up(static_cast<size_t>(B) * Hq * C * d * 2);
  void* qa = ws;
  void* qr = bif ? ws + qbytes : qa;
  void* kr = bif ? ws + 2 * qbytes : nullptr;
  const size_t krbytes = align_up(static_cast<size_t>(B) * Hkv * Lk * d * 2);
  void* tables = ws + (bif ? 2 * qbytes + krbytes : qbytes);
  auto stream = static_cast<cudaStream_t>(cuda_stream);
  const RopeFreqs fr = make_rope_freqs(d, rope_theta);
  cudaError_t e = launch_rope_tables(tables, d, fr, stream);
  if (e != cudaSuccess) return cuda_fail(e, "prefill_chunk: rotation tables");
  const TensorView none{nullptr, 0, 0, 0, 0};
  const size_t row_elems = static_cast<size_t>(Hkv) * d;
  auto* kc = static_cast<__nv_bfloat16_raw*>(k_cache);
  // 1. Queries at positions P0 .. P0+C-1, both rotations.
  e = launch_rope_prepass(q, B, C, Hq, d, G, P0, tables, head_major(qa, Hq, C, d),
                                      bif ? head_major(qr, Hq, C, d) : none, none, stream);
  if (e != cudaSuccess) return cuda_fail(e, "prefill_chunk: pre-pass (Q)");
  // 2. New keys: absolute rotation appended to the cache, aliased rotation
  //    into rows P0.. of K_rem.
  TensorView kr_all = bif ? head_major(kr, Hkv, Lk, d) : none;
  TensorView kr_new = kr_all;
  if (bif) kr_new.base = static_cast<const unsigned char*>(kr) + static_cast<size_t>(P0) * d * 2;
  TensorView kc_new = cache_layout(kc + static_cast<size_t>(P0) * row_elems, Lcap, Hkv, d, C);
  e = launch_rope_prepass(k, B, C, Hkv, d, G, P0, tables, none, kr_new, kc_new, stream);
  if (e != cudaSuccess) return cuda_fail(e, "prefill_chunk: pre-pass (K)");
  // 3. Cached keys 0 .. P0-1: aliased rotation by the correction R_{f(k)-k}.
  if (bif && P0 > 0) {
    e = launch_rope_correct(k_cache, B, P0, Lcap, Hkv, d, G, tables, kr_all, stream);
    if (e != cudaSuccess) return cuda_fail(e, "prefill_chunk: correction pass");
  }
  // 4. New values appended to the value cache.
  e = cudaMemcpy2DAsync(static_cast<unsigned char*>(v_cache) + static_cast<size_t>(P0) * row_elems * 2,
                        static_cast<size_t>(Lcap) * row_elems * 2, v, static_cast<size_t>(C) * row_elems * 2,
                        static_cast<size_t>(C) * row_elems * 2, B, cudaMemcpyDeviceToDevice, stream);
  if (e != cudaSuccess) return cuda_fail(e, "prefill_chunk: value append");
  // 5. Attention of the C query rows over keys 0 .. P0+C-1.
  PrefillArgs a;
  a.qa = head_major(qa, Hq, C, d);
  a.qr = head_major(qr, Hq, C, d);
  a.ka = cache_layout(k_cache, Lcap, Hkv, d, Lk);
  a.kr = bif ? kr_all : a.ka;
  a.v = cache_layout(v_cache, Lcap, Hkv, d, Lk);
  a.o = o; a.lse = lse;
  a.B = B; a.Lq = C; a.Lk = Lk; a.q_base = P0; a.Hq = Hq; a.Hkv = Hkv; a.d = d; a.w0 = w0; a.G = G;
  a.scale_log2 = resolve_scale(softmax_scale, d) * kLog2e;
  e = launch_prefill_attention(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "prefill_chunk: attention kernel");
  return JL_OK;
}

size_t jl_bifocal_decode_workspace_size(int B, int Hq, int d, int Lcap) {
  if (B < 1 || Hq < 1 || d < 1 || Lcap < 1) return 0;
  return align_up(decode_workspace_bytes(B, Hq, d, Lcap));
}

}  // extern "C"

namespace jl {

// Validation shared by the decode entry points; L is the (largest) length.
int check_decode_args(const char* who, const void* q, const void* k_cache, const void* v_cache, int L, int Lcap,
                      const void* o, int B, int Hq, int Hkv, int d, int w0, int w_pretrained, double rope_theta) {
  if (!q || !k_cache || !v_cache || !o) return fail(JL_ERR_INVALID, "%s: null q/cache/o pointer", who);
  if (B < 1 || Hq < 1 || Hkv < 1 || Lcap < 1) return fail(JL_ERR_INVALID, "%s: need B, Hq, Hkv, Lcap >= 1", who);
  if (L < 1 || L > Lcap) return fail(JL_ERR_INVALID, "%s: need 1 <= L <= Lcap (got L=%d, Lcap=%d)", who, L, Lcap);
  if (Hq % Hkv != 0) return fail(JL_ERR_INVALID, "%s: Hq %% Hkv != 0 (%d, %d)", who, Hq, Hkv);
  if (w0 < 0 || w_pretrained < 1) return fail(JL_ERR_INVALID, "%s: need w0 >= 0, w_pretrained >= 1", who);
  if (!(rope_theta > 0.0) || !isfinite(rope_theta)) return fail(JL_ERR_INVALID, "%s: rope_theta must be > 0", who);
  if (d != 64 && d != 128) return fail(JL_ERR_UNSUPPORTED, "%s: head dim %d (supported: 64, 128)", who, d);
  if (!decode_supported(Hq, Hkv, d))
    return fail(JL_ERR_UNSUPPORTED, "%s: need 1 <= Hq/Hkv <= 8 query heads per KV head (got %d)", who, Hq / Hkv);
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o))
    return fail(JL_ERR_INVALID, "%s: every pointer must be 16-byte aligned", who);
  return JL_OK;
}

int decode_call(const char* who, const void* q, const void* k_cache, const void* v_cache, const int* seqlens,
                int L, int Lcap, void* o, float* lse, int B, int Hq, int Hkv, int d, int w0, int w_pretrained,
                double rope_theta, float softmax_scale, float* partials, void* cuda_stream) {
  DecodeArgs a;
  a.q = q; a.k_cache = k_cache; a.v_cache = v_cache; a.o = o; a.lse = lse;
  a.part = partials;
  a.seqlens = seqlens;
  a.B = B; a.L = L; a.Lcap = Lcap; a.Hq = Hq; a.Hkv = Hkv; a.d = d; a.w0 = w0;
  a.G = static_cast<int>(jl::group_size(L, w_pretrained));
  a.wp = w_pretrained;
  a.scale_log2 = resolve_scale(softmax_scale, d) * kLog2e;
  a.ang = make_angle_table(d, rope_theta);
  const cudaError_t e = launch_decode(a, static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return fail(JL_ERR_CUDA, "%s: launch: %s", who, cudaGetErrorString(e));
  return JL_OK;
}

}  // namespace jl

namespace {

int run_decode(const char* who, const void* q, const void* k_cache, const void* v_cache, const int* seqlens,
               int L, int Lcap, void* o, float* lse, int B, int Hq, int Hkv, int d, int w0, int w_pretrained,
               double rope_theta, float softmax_scale, void* workspace, size_t workspace_bytes,
               void* cuda_stream) {
  int rc = check_decode_args(who, q, k_cache, v_cache, L, Lcap, o, B, Hq, Hkv, d, w0, w_pretrained, rope_theta);
  if (rc != JL_OK) return rc;
  rc = check_workspace(who, workspace, workspace_bytes, jl_bifocal_decode_workspace_size(B, Hq, d, Lcap));
  if (rc != JL_OK) return rc;
  return decode_call(who, q, k_cache, v_cache, seqlens, L, Lcap, o, lse, B, Hq, Hkv, d, w0, w_pretrained,
                     rope_theta, softmax_scale, static_cast<float*>(workspace), cuda_stream);
}

}  // namespace

extern "C" {

int jl_bifocal_decode(const void* q, const void* k_cache, const void* v_cache, int L, int Lcap,
                      void* o, float* lse, int B, int Hq, int Hkv, int d, int w0, int w_pretrained,
                      double rope_theta, float softmax_scale, void* workspace,
                      size_t workspace_bytes, void* cuda_stream) {
  t_err[0] = '\0';
  return run_decode("decode", q, k_cache, v_cache, nullptr, L, Lcap, o, lse, B, Hq, Hkv, d, w0, w_pretrained,
                    rope_theta, softmax_scale, workspace, workspace_bytes, cuda_stream);
}

int jl_bifocal_decode_varlen(const void* q, const void* k_cache, const void* v_cache,
                             const int* seqlens, int max_len, int Lcap, void* o, float* lse, int B,
                             int Hq, int Hkv, int d, int w0, int w_pretrained, double rope_theta,
                             float softmax_scale, void* workspace, size_t workspace_bytes,
                             void* cuda_stream) {
  t_err[0] = '\0';
  if (!seqlens || (reinterpret_cast<uintptr_t>(seqlens) % alignof(int)))
    return fail(JL_ERR_INVALID, "decode_varlen: seqlens must be a non-null, int-aligned device pointer");
  return run_decode("decode_varlen", q, k_cache, v_cache, seqlens, max_len, Lcap, o, lse, B, Hq, Hkv, d, w0,
                    w_pretrained, rope_theta, softmax_scale, workspace, workspace_bytes, cuda_stream);
}

int jl_device_status(void* cuda_stream) {
  t_err[0] = '\0';
  auto stream = static_cast<cudaStream_t>(cuda_stream);
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "status: stream sync");
  int h = 0;
  e = cudaMemcpyFromSymbol(&h, g_device_status, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "status: read");
  if (h != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "status: clear");
    const char* what = h == 30 ? "a per-sequence length was outside [1, Lcap] and was clamped"
                               : "a bounded device wait ran out; the kernel skipped its remaining work";
    return fail(JL_ERR_TIMEOUT, "device status %d: %s", h, what);
  }
  return JL_OK;
}

const char* jl_last_error(void) { return t_err; }

}  // extern "C"
