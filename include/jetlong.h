/*
 * jetlong.h -- C ABI of libjetlong.so: causal bifocal-RoPE attention
 * (dynamic bifocal RoPE, "Jet-Long: Efficient Long-Context Extension with
 * Dynamic Bifocal RoPE") on one NVIDIA B300 (sm_103a).
 *
 * What the library computes.  For a query at position q and a key at
 * position k <= q (0-based positions, causal):
 *
 *   local  (q - k <= w0):  S(q,k) = <R_q x_q,       R_k x_k>
 *   remote (q - k >  w0):  S(q,k) = <R_f(q) x_q,    R_f(k) x_k>
 *
 * with f(x) = floor(x / G) and G = max(1, ceil(L / w_pretrained))
 * (paper digest page, section "Method": bifocal score Eq. 1, dynamic group
 * size and alias map Eqs. 2-3).  R_p is rotate-half RoPE: coordinate pair
 * (x_i, x_{i+d/2}) is turned by the angle p * theta^(-2i/d) (RoFormer).
 * The output is softmax(scale * S) V over keys k <= q, and the per-row
 * natural-log log-sum-exp lse = log sum_k exp(scale * S(q,k)).
 *
 * Conventions shared by every entry point:
 *  - Tensors are CALLER-OWNED device pointers (cudaMalloc / torch); the
 *    library allocates no device memory.  bf16 is IEEE bfloat16, fp32 is
 *    IEEE float.  Every tensor is dense row-major in the layout stated.
 *  - Calls are asynchronous on `cuda_stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  A return of JL_OK means the work was
 *    launched; device-side faults surface at the caller's next sync.
 *  - On error nothing is launched and a message is available from
 *    jl_last_error() (thread-local, valid until the next call).
 *  - No CPU fallback: without a CUDA device every compute call returns
 *    JL_ERR_CUDA.
 */
#ifndef JETLONG_H_
#define JETLONG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define JL_OK               0
#define JL_ERR_INVALID     -1  /* bad argument: null pointer, negative size, ...   */
#define JL_ERR_UNSUPPORTED -2  /* legal but not implemented (head dim, group, ...) */
#define JL_ERR_CUDA        -3  /* a CUDA runtime call or launch failed             */
#define JL_ERR_TIMEOUT     -4  /* a bounded device-side wait ran out (see status)  */
#define JL_ERR_WORKSPACE   -5  /* workspace pointer null or workspace_bytes small  */

/*
 * Dynamic group size G = max(1, ceil(L / w_pretrained))  (digest page,
 * "Method", Eq. 2): the smallest integer g >= 1 with floor((L-1)/g) <
 * w_pretrained, so every aliased position lies in the pretrained window.
 * Pure host function, no device work.  Returns G >= 1 (L == 0 gives 1),
 * or -1 if L < 0 or w_pretrained <= 0.
 */
int64_t jl_group_size(int64_t L, int64_t w_pretrained);

/*
 * Bytes of device workspace jl_bifocal_prefill needs for these sizes.
 * Returns 0 for invalid sizes.  Layout after jl_bifocal_rope, each part
 * starting on a 256-byte boundary: Q_abs bf16 [B, Hq, L, d], K_abs bf16
 * [B, Hkv, L, d], then (only when G > 1) Q_rem [B, Hq, L, d] and K_rem
 * [B, Hkv, L, d], then the per-call rotation tables (3 * 1024 * d/2 float4).
 * Every rotated element is the exact rotation R_p x (p = the absolute or the
 * aliased position) rounded to bf16, round to nearest even.  Positions are
 * supported up to 2^30 - 1.
 */
size_t jl_bifocal_prefill_workspace_size(int B, int L, int Hq, int Hkv, int d,
                                         int w_pretrained);

/*
 * Causal bifocal-RoPE attention over a whole prompt (prefill), one G for
 * the whole call, G = jl_group_size(L, w_pretrained).
 *
 *  q     bf16 [B, L, Hq,  d]  raw (pre-RoPE) queries
 *  k     bf16 [B, L, Hkv, d]  raw (pre-RoPE) keys
 *  v     bf16 [B, L, Hkv, d]  values
 *  o     bf16 [B, L, Hq,  d]  output (written)
 *  lse   fp32 [B, Hq, L]      natural-log LSE of the scaled scores; may be NULL
 *  d     head dim, 64 or 128; Hq % Hkv == 0 (query head h reads KV head
 *        h / (Hq / Hkv)); B, L, Hq, Hkv >= 1
 *  w0    local window (>= 0): q - k <= w0 scores at absolute positions
 *  w_pretrained  pretrained context length (>= 1)
 *  rope_theta    RoPE base (> 0)
 *  softmax_scale <= 0 selects 1/sqrt(d)
 *  k_rot_out     NULL, or bf16 [B, L, Hkv, d] receiving R_k x_k (keys rotated
 *                at their absolute position), the form a KV cache stores
 *                for jl_bifocal_decode
 *  workspace     device buffer of >= jl_bifocal_prefill_workspace_size bytes,
 *                256-byte aligned; contents on entry are ignored
 *
 * Inputs are read-only; o, lse, k_rot_out and the workspace are written.
 * Buffers must not overlap.  Every pointer must be 16-byte aligned.
 */
int jl_bifocal_prefill(const void* q, const void* k, const void* v,
                       void* o, float* lse,
                       int B, int L, int Hq, int Hkv, int d,
                       int w0, int w_pretrained, double rope_theta,
                       float softmax_scale, void* k_rot_out,
                       void* workspace, size_t workspace_bytes,
                       void* cuda_stream);

/*
 * The two stages of jl_bifocal_prefill, callable separately (same arguments,
 * same workspace).  jl_bifocal_rope rotates q and k at absolute and aliased
 * positions into the workspace (and writes k_rot_out if not NULL);
 * jl_bifocal_attention then runs the routed causal attention over the
 * workspace and v.  Calling both in order on one stream is exactly
 * jl_bifocal_prefill.  jl_bifocal_attention reads nothing but the workspace
 * written by a jl_bifocal_rope call with the same B, L, Hq, Hkv, d and
 * w_pretrained.
 */
int jl_bifocal_rope(const void* q, const void* k,
                    int B, int L, int Hq, int Hkv, int d,
                    int w_pretrained, double rope_theta, void* k_rot_out,
                    void* workspace, size_t workspace_bytes, void* cuda_stream);

int jl_bifocal_attention(const void* v, void* o, float* lse,
                         int B, int L, int Hq, int Hkv, int d,
                         int w0, int w_pretrained, float softmax_scale,
                         const void* workspace, size_t workspace_bytes,
                         void* cuda_stream);

/*
 * The same computation as jl_bifocal_attention (same arguments, workspace,
 * results and error behaviour) on a second kernel design, kept as its A/B
 * counterpart: each tensor-core operation is shared by a cluster of two CTAs
 * (tcgen05 cta_group::2, M = 256), so that each CTA holds one 128-row query
 * tile with a double-buffered score tile.  Head dim 128 only
 * (JL_ERR_UNSUPPORTED otherwise).  Outputs are within the same bounds of the
 * oracle; on B300 it is slower than jl_bifocal_attention (paper digest page,
 * "Method", Eq. 1 for what it computes).
 */
int jl_bifocal_attention_cta_pair(const void* v, void* o, float* lse,
                                  int B, int L, int Hq, int Hkv, int d,
                                  int w0, int w_pretrained, float softmax_scale,
                                  const void* workspace, size_t workspace_bytes,
                                  void* cuda_stream);

/*
 * Chunked prefill against an absolute-position KV cache: the prompt arrives
 * in chunks, and each chunk attends to everything before it through the
 * cache that earlier calls filled (this entry point, jl_bifocal_prefill's
 * k_rot_out, or decode-side appends).
 *
 * The cache holds positions [0, P0): keys rotated at their absolute
 * positions, R_k x_k, and values.  The chunk is C raw tokens at positions
 * [P0, P0 + C).  With G = jl_group_size(P0 + C, w_pretrained) (one G for the
 * call, from the total length after the chunk), query p in the chunk attends
 * to keys 0 .. p with the bifocal score; cached keys reach their aliased
 * rotation through the correction R_{f(k)-k} (digest page, "KV cache
 * invariant") -- positions [0, P0) of the cache are only read.  The chunk's
 * rotated keys and its values are appended to the cache at [P0, P0 + C).
 * The result equals rows [P0, P0 + C) of a jl_bifocal_prefill over the first
 * P0 + C tokens when both see the same G.
 *
 *  q        bf16 [B, C, Hq, d]   raw chunk queries
 *  k, v     bf16 [B, C, Hkv, d]  raw chunk keys, values
 *  k_cache  bf16 [B, Lcap, Hkv, d]  rows [0, P0) read, rows [P0, P0+C) written
 *  v_cache  bf16 [B, Lcap, Hkv, d]  same
 *  P0 >= 0, C >= 1, P0 + C <= Lcap
 *  o        bf16 [B, C, Hq, d];  lse fp32 [B, Hq, C] (may be NULL)
 *  workspace >= jl_bifocal_prefill_chunk_workspace_size(...) bytes
 */
size_t jl_bifocal_prefill_chunk_workspace_size(int B, int C, int P0, int Hq, int Hkv, int d,
                                               int w_pretrained);

int jl_bifocal_prefill_chunk(const void* q, const void* k, const void* v,
                             void* k_cache, void* v_cache, int P0, int Lcap,
                             void* o, float* lse,
                             int B, int C, int Hq, int Hkv, int d,
                             int w0, int w_pretrained, double rope_theta,
                             float softmax_scale,
                             void* workspace, size_t workspace_bytes,
                             void* cuda_stream);

/*
 * Three-pass form of the same prefill (digest page, "Method", Eq. 7), kept
 * as an A/B counterpart of the routed single pass: three causal attention
 * passes over the pre-rotated operands,
 *   A  the local window (0 <= q - k <= w0) at absolute rotations,
 *   B  every causal key at aliased rotations (written into o / a private lse),
 *   C  the local window at aliased rotations,
 * merged by inclusion-exclusion, o = (e^lA oA + e^lB oB - e^lC oC) /
 * (e^lA + e^lB - e^lC), lse = log(e^lA + e^lB - e^lC).  Mathematically
 * identical to jl_bifocal_prefill; numerically, the merge subtracts C's mass
 * from B's, so its error grows where the local window holds most of the
 * aliased-rotation mass.  It scores the window pairs three times.
 *
 * Fidelity: this A/B form does NOT always meet the acceptance bound of the
 * routed prefill (O max-abs 2e-2 against the fp64 reference).  On random
 * inputs the two forms agree to about 3e-3 (O) and 4e-6 (LSE), but where
 * each query's own window dominates (queries close to their own keys) the
 * measured O max-abs error of the three-pass form reached 2.7e-2, against
 * 1.5e-2 for jl_bifocal_prefill on the same inputs.  Use jl_bifocal_prefill
 * when the bound matters; this entry point exists for comparison.
 *
 * Arguments, layouts and errors as jl_bifocal_prefill (no k_rot_out);
 * workspace >= jl_bifocal_prefill_three_pass_workspace_size(...) bytes, which
 * holds the rotated operands, oA, oC and the three log-sum-exps.
 */
size_t jl_bifocal_prefill_three_pass_workspace_size(int B, int L, int Hq, int Hkv, int d,
                                                    int w_pretrained);

int jl_bifocal_prefill_three_pass(const void* q, const void* k, const void* v,
                                  void* o, float* lse,
                                  int B, int L, int Hq, int Hkv, int d,
                                  int w0, int w_pretrained, double rope_theta,
                                  float softmax_scale,
                                  void* workspace, size_t workspace_bytes,
                                  void* cuda_stream);

/*
 * The same prefill with q, k, v, o and lse in HOST memory: the library copies
 * the inputs in and the outputs out itself, pipelined by query chunks so that
 * the copies overlap the kernels.  Chunk c (rows r0 .. r0 + rows - 1, rows a
 * multiple of 256 except the last) is copied in on a library copy stream,
 * rotated, attended over keys 0 .. r0 + rows - 1 with the call's single G,
 * and its o and lse rows are copied out on a second copy stream while the
 * next chunk computes.  Results are bit-identical to jl_bifocal_prefill on
 * the same data.
 *
 *  q_host  bf16 [B, L, Hq, d], k_host / v_host bf16 [B, L, Hkv, d]  (read)
 *  o_host  bf16 [B, L, Hq, d]; lse_host fp32 [B, Hq, L] or NULL       (written)
 *  n_chunks  query chunks per sequence; 0 picks min(16, max(1, L / 8192))
 *  workspace >= jl_bifocal_prefill_host_workspace_size(...) bytes (device):
 *            the prefill workspace plus device copies of q, k, v, o and lse
 *  other arguments as jl_bifocal_prefill
 *
 * Asynchronous on cuda_stream like every call: the host outputs are complete
 * once the stream has synchronised, and the host buffers must stay valid
 * until then.  Page-locked host buffers are needed for the copies to overlap;
 * pageable ones are correct but serialise.  The two copy streams and an
 * event pool are created on the first call on each device and kept; calls
 * from several host threads are serialised while they enqueue.
 */
size_t jl_bifocal_prefill_host_workspace_size(int B, int L, int Hq, int Hkv, int d,
                                              int w_pretrained);

int jl_bifocal_prefill_host(const void* q_host, const void* k_host, const void* v_host,
                            void* o_host, float* lse_host,
                            int B, int L, int Hq, int Hkv, int d,
                            int w0, int w_pretrained, double rope_theta,
                            float softmax_scale, int n_chunks,
                            void* workspace, size_t workspace_bytes,
                            void* cuda_stream);

/*
 * Bytes of device workspace jl_bifocal_decode needs (per-split partial
 * softmax statistics and outputs) for caches of up to Lcap positions.
 * Returns 0 for invalid sizes.
 */
size_t jl_bifocal_decode_workspace_size(int B, int Hq, int d, int Lcap);

/*
 * One new query token against an absolute-position KV cache (decode), with
 * the on-the-fly correction rotation of the digest page's "KV cache
 * invariant" (Delta_q = f(q) - q, Delta_k = f(k) - k, R_a R_b = R_{a+b}):
 * the cache is read, never rewritten, whatever G is.
 *
 *  q        bf16 [B, Hq, d]          raw (pre-RoPE) query of the token at
 *                                    position L-1
 *  k_cache  bf16 [B, Lcap, Hkv, d]   key j holds R_j x_j (rotated at its
 *                                    absolute position j); read-only
 *  v_cache  bf16 [B, Lcap, Hkv, d]   values; read-only
 *  L        number of valid cache positions INCLUDING the new token
 *           (1 <= L <= Lcap); G = jl_group_size(L, w_pretrained)
 *  o        bf16 [B, Hq, d]   output
 *  lse      fp32 [B, Hq]      natural-log LSE; may be NULL
 *  d        64 or 128; Hkv >= 1 and Hq % Hkv == 0 with 1 <= Hq / Hkv <= 8
 *           (query head h reads KV head h / (Hq / Hkv)); other layouts
 *           return JL_ERR_UNSUPPORTED
 *  workspace >= jl_bifocal_decode_workspace_size(B, Hq, d, Lcap) bytes
 *
 *   local  (L-1 - j <= w0):  s_j = <R_{L-1} x_q, K_j>
 *   remote (L-1 - j >  w0):  s_j = <R_{f(L-1)} x_q, R_{f(j)-j} K_j>
 */
int jl_bifocal_decode(const void* q, const void* k_cache, const void* v_cache,
                      int L, int Lcap, void* o, float* lse,
                      int B, int Hq, int Hkv, int d,
                      int w0, int w_pretrained, double rope_theta,
                      float softmax_scale,
                      void* workspace, size_t workspace_bytes,
                      void* cuda_stream);

/*
 * Batched decode with one length per sequence: sequence b holds
 * seqlens[b] valid cache positions (its new token at position seqlens[b]-1)
 * and uses its own G = jl_group_size(seqlens[b], w_pretrained).  Same
 * arguments and kernels as jl_bifocal_decode otherwise.
 *
 *  seqlens  int32 [B] on the DEVICE; each value in [1, max_len] (values
 *           outside [1, Lcap] are clamped and reported by jl_device_status)
 *  max_len  largest value of seqlens (<= Lcap); sizes the key split
 *  workspace >= jl_bifocal_decode_workspace_size(B, Hq, d, Lcap) bytes
 */
int jl_bifocal_decode_varlen(const void* q, const void* k_cache, const void* v_cache,
                             const int* seqlens, int max_len, int Lcap, void* o, float* lse,
                             int B, int Hq, int Hkv, int d,
                             int w0, int w_pretrained, double rope_theta,
                             float softmax_scale,
                             void* workspace, size_t workspace_bytes,
                             void* cuda_stream);

/*
 * jl_bifocal_decode for callers that cannot allocate device memory.  There is
 * no counterpart on the paper's pages: this is a deployment variant.
 *
 * Same arguments, semantics and kernels as jl_bifocal_decode minus the
 * workspace: the split-K partials live in a fixed 16 MiB scratch array that
 * is part of the library image (every GPU that loads the library holds it
 * until the process exits).  A call needs min(SM count, 512) * B * Hq *
 * (d + 2) * 4 bytes of it, so on a 148-SM B300 it serves B * Hq <= 218 at
 * d = 128 (B * Hq <= 425 at d = 64); larger sizes return JL_ERR_UNSUPPORTED
 * with a message, after the same argument checks (and error codes) as
 * jl_bifocal_decode.  The entry point itself calls no allocator of any kind.
 *  - The first call on each device (with that device current) resolves the
 *    scratch array's device address; make that first call before any stream
 *    capture.
 *  - Every call shares the one array: calls whose kernels overlap on the GPU
 *    (other streams, unordered threads) race and corrupt each other's
 *    results.  Order them on one stream.
 *  - Nothing in the array needs to start at zero; each call writes every
 *    slot it reads.
 */
int jl_bifocal_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                              int L, int Lcap, void* o, float* lse,
                              int B, int Hq, int Hkv, int d,
                              int w0, int w_pretrained, double rope_theta,
                              float softmax_scale, void* cuda_stream);

/* Size in bytes of the fixed scratch array of jl_bifocal_decode_noalloc. */
size_t jl_bifocal_decode_noalloc_scratch_bytes(void);

/*
 * Synchronises `cuda_stream`, then reads and clears the library's device
 * status word, which a kernel sets when one of its bounded waits on a
 * barrier runs out (it then skips its remaining work instead of hanging) or
 * when jl_bifocal_decode_varlen had to clamp a length.  Returns JL_OK,
 * JL_ERR_TIMEOUT (the code and its meaning in jl_last_error) or JL_ERR_CUDA.
 */
int jl_device_status(void* cuda_stream);

/*
 * Exercises the failure path of jl_device_status without faulting the GPU:
 * launches one thread that waits, with the library's bounded wait, on a
 * barrier nothing arrives on.  After `limit_cycles` clock cycles (1 .. 4e9)
 * the wait gives up, the status word is set and the kernel returns; the next
 * jl_device_status on the stream then reports JL_ERR_TIMEOUT.  The paper has
 * no counterpart: this is test support for the bounded waits.
 */
int jl_selftest_bounded_wait(long long limit_cycles, void* cuda_stream);

/*
 * Test support for the bounded waits of the prefill pipeline: exactly
 * jl_bifocal_prefill (no k_rot_out, default softmax scale), except that every
 * wait of the attention kernel's pipeline gives up after `limit_cycles`
 * clock cycles (1 .. 4e9) instead of about 2 s.  With a small limit the
 * waits run out: the CTAs record a status code, let their bulk copies and
 * tensor-core work finish, free their tensor memory and return, so the next
 * jl_device_status on the stream reports JL_ERR_TIMEOUT and the context stays
 * usable; o and lse are then incomplete.  The paper has no counterpart.
 */
int jl_selftest_prefill_wait_limit(const void* q, const void* k, const void* v,
                                   void* o, float* lse,
                                   int B, int L, int Hq, int Hkv, int d,
                                   int w0, int w_pretrained, double rope_theta,
                                   long long limit_cycles,
                                   void* workspace, size_t workspace_bytes,
                                   void* cuda_stream);

/*
 * The same test support for the CTA-pair attention kernel
 * (jl_bifocal_attention_cta_pair, d = 128 only; JL_ERR_UNSUPPORTED
 * otherwise): with a small limit both CTAs of a pair give up, tell each
 * other, drain their copies and tensor-core work, meet at the cluster
 * barrier, free the pair's tensor memory and return.
 */
int jl_selftest_prefill_pair_wait_limit(const void* q, const void* k, const void* v,
                                        void* o, float* lse,
                                        int B, int L, int Hq, int Hkv, int d,
                                        int w0, int w_pretrained, double rope_theta,
                                        long long limit_cycles,
                                        void* workspace, size_t workspace_bytes,
                                        void* cuda_stream);

/* Message of the last error on this thread ("" if none). Never NULL. */
const char* jl_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* JETLONG_H_ */
