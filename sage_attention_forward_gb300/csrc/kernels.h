// Host-side launchers of the device kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>
#include <mutex>

namespace sa {

// The unique id (cuCtxGetId) of the CUDA context current on the calling thread; when none
// is current yet, the current device's primary context is made current first, as the
// runtime's next call would.  Ids are never reused within a process.
cudaError_t current_context_id(unsigned long long* id);

// A value made once per CUDA context and cached, thread-safe.  Keyed by the context id,
// so a device that was reset, or a second context on the same device, makes its own
// value; the cache keeps the last 64 contexts (an older one simply makes it again).
template <class T>
class PerContext {
 public:
  // make: cudaError_t(T*), called with the context current; its value is cached on success
  template <class F>
  cudaError_t get(F&& make, T* out) {
    unsigned long long id = 0;
    cudaError_t e = current_context_id(&id);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu_);
    for (int i = 0; i < kSlots && i < n_; ++i)
      if (ids_[i] == id) {
        *out = vals_[i];
        return cudaSuccess;
      }
    T v{};
    e = make(&v);
    if (e != cudaSuccess) return e;
    ids_[n_ % kSlots] = id;
    vals_[n_ % kSlots] = v;
    ++n_;
    *out = v;
    return cudaSuccess;
  }

 private:
  static constexpr int kSlots = 64;
  std::mutex mu_;
  unsigned long long ids_[kSlots] = {};
  T vals_[kSlots] = {};
  int n_ = 0;
};

// A set-up step run once per CUDA context (e.g. a kernel attribute).
class ContextOnce {
 public:
  template <class F>
  cudaError_t run(F&& step) {
    char done = 0;
    return cache_.get([&](char* v) {
      cudaError_t e = step();
      *v = 1;
      return e;
    }, &done);
  }

 private:
  PerContext<char> cache_;
};

// Number of SMs of the current device (cached per context).
int device_sm_count();

// The attention forward kernel, three modes (attn_fwd.cu).  BF16 flash attention:
// Q, K, V through [B, S, H, 128] BF16 tensor maps.
// withhold_loads: the failure-path self-test (the producer loads nothing).
cudaError_t launch_attn_fwd_bf16(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v, void* o,
                                 long long o_sb, long long o_ss, long long o_sh, int B, int S, int H, float c_log2,
                                 cudaStream_t stream, bool withhold_loads = false);
// Timing instrumentation: per-SM {clock64, globaltimer} into out[n_slots][2] (cleared first).
cudaError_t launch_sm_clock_probe(unsigned long long* out, int n_slots, int num_sms, cudaStream_t stream);
// The device error word all three modes record bounded-wait timeouts in.
cudaError_t read_and_clear_err_attn(uint32_t* out);

// Sage prepare (sage_prepare.cu)
struct PrepareArgs {
  const void* x[3];          // q, k, v (BF16)
  long long str[3][3];       // element strides (b, s, h)
  int B, S, H;
  long long S_pad;
  const void* q_norm_w;
  const void* k_norm_w;
  float rms_eps;
  const void* rope_cos;
  const void* rope_sin;
  int rope_dim;
  int8_t* q_i8;
  int8_t* k_i8;
  uint8_t* v_fp8;
  float* q_scale;
  float* k_scale;
  float* v_scale;
  float c_log2;
  uint32_t* vmax;            // workspace: B*H*128 words
  float* k_mean = nullptr;   // K smoothing: output [B*H*128] (nullptr: no smoothing)
  float* k_partial = nullptr;  // K smoothing workspace: [B*H, S_pad/32, 128] block sums
  void* q16 = nullptr;       // when set: Q/K codes written as FP16 [B*H, S_pad, 128] here, not as INT8
  void* k16 = nullptr;
  bool skip_v = false;       // V not prepared (the 16-bit P V mode reads the BF16 input)
  bool skip_q = false;       // Q not prepared (the forward quantises Q as it loads it)
  bool skip_k = false;       // K not prepared either (the forward codes K as well; needs skip_q)
  void* q_mean16 = nullptr;  // Q smoothing: output, binary16 [B*H, S_pad/32, 128] block means in step units
                             // (nullptr: no Q smoothing); the FP16 codes (q16) are then f16(code + mean)
};
cudaError_t launch_sage_prepare(const PrepareArgs& a, cudaStream_t stream);
// Q's score operand with Q smoothing, f16(code + mean), from the INT8 codes and the block means.
cudaError_t launch_widen_q_mean(const int8_t* q8, const void* qmean16, void* q16, long long n_codes, int num_sms,
                               cudaStream_t stream);
// e4m3 codes of n binary32 values through the prepare's and the attention's packing.
cudaError_t launch_e4m3_encode(const float* x, uint8_t* y, long long n, int num_sms, cudaStream_t stream);

// Device address, in the current context, of the static scratch used by the
// allocation-free prepare entry point; it holds kNoAllocMaxHeads * 128 words.
// Looked up on the first call in each context and cached.
constexpr int kNoAllocMaxHeads = 2048;
cudaError_t noalloc_prepare_scratch(uint32_t** out);

// Sage attention on prepared tensors (attn_fwd.cu)
size_t sage_attn_smem_bytes();
cudaError_t launch_sage_widen(const int8_t* q8, const int8_t* k8, void* q16, void* k16, long long n_codes,
                              int num_sms, cudaStream_t stream);
cudaError_t launch_sage_attn(const CUtensorMap& tm_q16, const CUtensorMap& tm_k16, const CUtensorMap& tm_v8,
                             const float* q_scale, const float* k_scale, const float* v_scale, void* o,
                             long long o_sb, long long o_ss, long long o_sh, int B, int S, int H, long long S_pad,
                             cudaStream_t stream);
// The 16-bit P V mode: V is the BF16 input through a [B, S, H, 128] tensor map.
cudaError_t launch_sage_attn_pv16(const CUtensorMap& tm_q16, const CUtensorMap& tm_k16,
                                  const CUtensorMap& tm_v_bf16, const float* q_scale, const float* k_scale, void* o,
                                  long long o_sb, long long o_ss, long long o_sh, int B, int S, int H,
                                  long long S_pad, cudaStream_t stream);

// Quantise-on-load of Q: the forward reads BF16 Q through a [B, S, H, 128] tensor
// map and each softmax thread turns its own row into the codes and the scale the
// prepare would have written (optional RMSNorm + RoPE first, the same arithmetic).
struct QLoadArgs {
  const void* q_norm_w = nullptr;   // BF16 [128], or nullptr: no RMSNorm
  const void* k_norm_w = nullptr;   // the same for K (K coded on load)
  float rms_eps = 0.0f;
  const void* rope_cos = nullptr;   // BF16 [S, rope_dim], or nullptr: no RoPE
  const void* rope_sin = nullptr;
  int rope_dim = 0;
  float c_log2 = 0.0f;              // fl32(softmax_scale * log2 e), folded into Q's scales
};
cudaError_t launch_sage_attn_qload(const CUtensorMap& tm_q_bf16, const CUtensorMap& tm_k16,
                                   const CUtensorMap& tm_v8, const QLoadArgs& qa, const float* k_scale,
                                   const float* v_scale, void* o, long long o_sb, long long o_ss, long long o_sh,
                                   int B, int S, int H, long long S_pad, cudaStream_t stream);
// K coded on load as well: K through a BF16 [B, S, H, 128] tensor map, coded per tile by the
// softmax warpgroups (the prepare's arithmetic); the block scales never leave shared memory.
cudaError_t launch_sage_attn_qkload(const CUtensorMap& tm_q_bf16, const CUtensorMap& tm_k_bf16,
                                    const CUtensorMap& tm_v8, const QLoadArgs& qa, const float* v_scale, void* o,
                                    long long o_sb, long long o_ss, long long o_sh, int B, int S, int H,
                                    long long S_pad, cudaStream_t stream);
cudaError_t launch_sage_attn_pv16_qkload(const CUtensorMap& tm_q_bf16, const CUtensorMap& tm_k_bf16,
                                         const CUtensorMap& tm_v_bf16, const QLoadArgs& qa, void* o, long long o_sb,
                                         long long o_ss, long long o_sh, int B, int S, int H, long long S_pad,
                                         cudaStream_t stream);
cudaError_t launch_sage_attn_pv16_qload(const CUtensorMap& tm_q_bf16, const CUtensorMap& tm_k16,
                                        const CUtensorMap& tm_v_bf16, const QLoadArgs& qa, const float* k_scale,
                                        void* o, long long o_sb, long long o_ss, long long o_sh, int B, int S, int H,
                                        long long S_pad, cudaStream_t stream);

}  // namespace sa
