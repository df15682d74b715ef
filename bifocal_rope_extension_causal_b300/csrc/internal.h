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

// ---- RoPE pre-pass (rope_prepass.cu) ---------------------------------------
// Rotates x [B, L, H, d] (raw) at absolute positions into out_abs [B, H, L, d]
// and, if out_rem != nullptr, at aliased positions f(p) = p / G into out_rem
// [B, H, L, d]; if out_cache != nullptr also writes the absolute rotation in
// the input layout [B, L, H, d].
cudaError_t launch_rope_prepass(const void* x, int B, int L, int H, int d, int G,
                                const RopeFreqs& freqs, void* out_abs, void* out_rem,
                                void* out_cache, cudaStream_t stream);

// ---- Prefill attention over pre-rotated operands (prefill_*.cu) -------------
struct PrefillArgs {
  const void* qa;  // bf16 [B, Hq, L, d]  R_q x_q
  const void* qr;  // bf16 [B, Hq, L, d]  R_f(q) x_q   (== qa when G == 1)
  const void* ka;  // bf16 [B, Hkv, L, d] R_k x_k
  const void* kr;  // bf16 [B, Hkv, L, d] R_f(k) x_k  (== ka when G == 1)
  const void* v;   // bf16 [B, L, Hkv, d]
  void* o;         // bf16 [B, L, Hq, d]
  float* lse;      // fp32 [B, Hq, L] or nullptr
  int B, L, Hq, Hkv, d, w0, G;
  float scale_log2;  // softmax scale * log2(e)
};
cudaError_t launch_prefill_attention(const PrefillArgs& a, cudaStream_t stream);

// ---- Decode (decode.cu) ------------------------------------------------------
struct DecodeArgs {
  const void* q;        // bf16 [B, Hq, d] raw
  const void* k_cache;  // bf16 [B, Lcap, Hkv, d]
  const void* v_cache;  // bf16 [B, Lcap, Hkv, d]
  void* o;              // bf16 [B, Hq, d]
  float* lse;           // fp32 [B, Hq] or nullptr
  float* part;          // workspace: partial outputs and statistics
  int B, L, Lcap, Hq, Hkv, d, w0, G;
  float scale_log2;
  RopeFreqs freqs;
};
int decode_max_splits();
size_t decode_workspace_bytes(int B, int Hq, int d, int Lcap);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

// ---- TMA descriptors (tma_host.cu) -------------------------------------------
// Encode a tiled bf16 tensor map: dims[0] innermost; strides_bytes[i] is the
// byte stride of dimension i+1; box[i] the tile extent.  False on failure.
bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128);

// ---- Errors (api.cu) -----------------------------------------------------------
// Record `msg` as this thread's jl_last_error() message; returns `code`.
int set_error(int code, const char* msg);

// ---- Device status word (api.cu) ----------------------------------------------
// Device address of the library's status word; kernels with bounded waits set
// it (non-zero) when a wait runs out.  nullptr if it cannot be resolved.
int* device_status_ptr();

}  // namespace jl
