// Launchers shared between the C-ABI layer (api.cu) and the kernel files.
// Host-only declarations; no torch types anywhere in this library.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace jl {

constexpr int kMaxHalfDim = 64;  // d <= 128

// omega_i = theta^(-2i/d), i < d/2, in double (passed by value to kernels).
struct RopeFreqs {
  double w[kMaxHalfDim];
};
RopeFreqs make_rope_freqs(int d, double theta);

// Per-frequency angle tables for float-only rotary angles (decode): level l
// holds phi_l = (2^(10 l) omega_i) mod 2 pi, reduced in double on the host
// and split as hi + lo, hi keeping 14 significant bits so that d * hi is
// exact in float for any 10-bit integer d.
struct AngleTable {
  float hi[3][kMaxHalfDim];
  float lo[3][kMaxHalfDim];
};
AngleTable make_angle_table(int d, double theta);

// A bf16 tensor addressed as [B, H, rows, d]: element (b, h, row, e) lives at
// base + b * sb + h * sh + row * sr + e (strides in elements).  Head-major
// workspace tensors [B, H, L, d] and cache-layout tensors [B, Lcap, H, d]
// are both described this way.
struct TensorView {
  const void* base;
  long long sb, sh, sr;
  int rows;
};
inline TensorView head_major(const void* base, int H, int L, int d) {
  return {base, static_cast<long long>(H) * L * d, static_cast<long long>(L) * d, d, L};
}
inline TensorView cache_layout(const void* base, int Lcap, int H, int d, int rows) {
  return {base, static_cast<long long>(Lcap) * H * d, d, static_cast<long long>(H) * d, rows};
}

// ---- RoPE pre-pass (rope_prepass.cu) ---------------------------------------
// Rotation tables: rows 0..1023 hold R_j, rows 1024..2047 R_{j 2^10}, rows
// 2048..3071 R_{j 2^20} (positions below 2^30), each row d/2 float4
// {cos hi, cos lo, sin hi, sin lo}.  Built per call into caller workspace.
constexpr int kRopeTableRows = 3 * 1024;
constexpr int kMaxRopePosition = (1 << 30) - 1;
inline size_t rope_table_bytes(int d) { return static_cast<size_t>(kRopeTableRows) * (d / 2) * 16; }
cudaError_t launch_rope_tables(void* tables, int d, const RopeFreqs& freqs, cudaStream_t stream);

// Rotates x [B, C, H, d] (raw; row p is position pos0 + p) at the absolute
// positions into `abs` and at the aliased positions f(pos) = pos / G into
// `rem`, also writing the absolute rotation into `cache` (rows p of each
// view; a view with a null base is skipped).  Every element is the exact
// rotation rounded to bf16; `tables` come from launch_rope_tables.
cudaError_t launch_rope_prepass(const void* x, int B, int C, int H, int d, int G, int pos0,
                                const void* tables, TensorView abs, TensorView rem,
                                TensorView cache, cudaStream_t stream);

// Turns keys already rotated at their absolute positions k (cache [B, Lcap,
// H, d], rows 0 .. P0-1) into keys rotated at f(k) = k / G by the
// correction rotation R_{f(k) - k}; writes rows 0 .. P0-1 of `rem`
// (exactly rounded, as above).
cudaError_t launch_rope_correct(const void* k_cache, int B, int P0, int Lcap, int H, int d, int G,
                                const void* tables, TensorView rem, cudaStream_t stream);

// ---- Prefill attention over pre-rotated operands (prefill_tc.cu) -------------
// Query rows 0 .. Lq-1 sit at positions q_base .. q_base+Lq-1 and attend
// causally to keys 0 .. q_base+row (Lk = q_base + Lq key rows).
struct PrefillArgs {
  TensorView qa, qr;  // R_q x_q and R_f(q) x_q (qr == qa when G == 1); rows = Lq
  TensorView ka, kr;  // R_k x_k and R_f(k) x_k (kr == ka when G == 1); rows = Lk
  TensorView v;       // values; rows = Lk
  void* o;            // bf16 [B, Lq, Hq, d]
  float* lse;         // fp32 [B, Hq, Lq] or nullptr
  int B, Lq, Lk, q_base, Hq, Hkv, d, w0, G;
  float scale_log2;   // softmax scale * log2(e)
  // Window-only mode (the local views of the three-pass form): score only
  // the pairs with 0 <= q - k <= w0, with the qa/ka rotations.
  bool window_only = false;
  // Clock cycles a pipeline wait may take before the CTA gives up (records a
  // status code and skips its remaining work); 0 selects the default
  // (about 2 s).  Only the test-support entry point sets it.
  long long wait_limit = 0;
  // Head dim 128 only: run on CTA pairs (prefill_pair.cu) instead of the
  // single-CTA kernel; the A/B counterpart, slower on B300.
  bool cta_pair = false;
};
cudaError_t launch_prefill_attention(const PrefillArgs& a, cudaStream_t stream);
// Head dim 128 on CTA pairs (prefill_pair.cu); `status` is the device status word.
cudaError_t launch_prefill_attention_pair(const PrefillArgs& a, int* status, cudaStream_t stream);

// ---- Three-pass merge (three_pass.cu) ----------------------------------------
// o = (wA oA + wB o - wC oC) / (wA + wB - wC), w_X = exp(lse_X - max(lse_A, lse_B)),
// in place on o ([B, L, Hq, d] bf16); lse_out [B, Hq, L] (nullable) gets the
// merged log-sum-exp.
cudaError_t launch_three_pass_merge(const void* o_a, const float* lse_a, void* o, const float* lse_b,
                                    const void* o_c, const float* lse_c, float* lse_out, int B, int L,
                                    int Hq, int d, cudaStream_t stream);

// ---- Decode (decode.cu) ------------------------------------------------------
struct DecodeArgs {
  const void* q;        // bf16 [B, Hq, d] raw
  const void* k_cache;  // bf16 [B, Lcap, Hkv, d]
  const void* v_cache;  // bf16 [B, Lcap, Hkv, d]
  void* o;              // bf16 [B, Hq, d]
  float* lse;           // fp32 [B, Hq] or nullptr
  float* part;          // workspace: partial outputs and statistics
  const int* seqlens;   // per-sequence lengths [B] on the device, or nullptr
  int B, L, Lcap, Hq, Hkv, d, w0, G, wp;  // L: the length, or the largest one with seqlens
  float scale_log2;
  AngleTable ang;
};
int decode_max_splits();
// Largest number of key slices one decode launch uses on the current device:
// min(SM count, decode_max_splits()).
int decode_slice_cap();
// Bytes of partials a decode call needs (device-independent upper bound) and
// the tighter bound for the current device's slice cap.
size_t decode_workspace_bytes(int B, int Hq, int d, int Lcap);
size_t decode_scratch_bytes(int B, int Hq, int d);
// Head layouts the decode kernels take: d in {64, 128}, Hq / Hkv in 1..8.
bool decode_supported(int Hq, int Hkv, int d);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

// ---- TMA descriptors (tma_host.cu) -------------------------------------------
// Encode a tiled bf16 tensor map: dims[0] innermost; strides_bytes[i] is the
// byte stride of dimension i+1; box[i] the tile extent.  False on failure.
bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128);

// ---- Errors and shared checks (api.cu) -------------------------------------------
// Record `msg` as this thread's jl_last_error() message; returns `code`.
int set_error(int code, const char* msg);
// Argument checks of the decode entry points (JL_OK, or the error code with
// the message recorded); `who` prefixes the message.
int check_decode_args(const char* who, const void* q, const void* k_cache, const void* v_cache, int L, int Lcap,
                      const void* o, int B, int Hq, int Hkv, int d, int w0, int w_pretrained, double rope_theta);
// Launches the decode kernels of a checked call with the partials at
// `partials` (at least decode_scratch_bytes(B, Hq, d) bytes); JL_OK or
// JL_ERR_CUDA with the message recorded.
int decode_call(const char* who, const void* q, const void* k_cache, const void* v_cache, const int* seqlens,
                int L, int Lcap, void* o, float* lse, int B, int Hq, int Hkv, int d, int w0, int w_pretrained,
                double rope_theta, float softmax_scale, float* partials, void* cuda_stream);

// ---- Device status word (api.cu) ----------------------------------------------
// Device address of the library's status word; kernels with bounded waits set
// it (non-zero) when a wait runs out.  nullptr if it cannot be resolved.
int* device_status_ptr();

}  // namespace jl
