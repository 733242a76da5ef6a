// C ABI of the library (declared in include/sageattn.h): argument validation,
// TMA tensor-map encoding and kernel launches.  No allocation happens here.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/sageattn.h"
#include "kernels.h"

namespace {

thread_local char g_msg[512] = "";

attn_status fail(attn_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return s;
}

attn_status fail_cuda(cudaError_t e, const char* what) {
  return fail(ATTN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr double kLog2e = 1.4426950408889634;

// ------------------------------------------------------------------ device check
constexpr int kMaxDevices = 64;
int g_dev_ok[kMaxDevices];  // 0 unknown, 1 sm_103, -1 other
std::mutex g_dev_mu;

attn_status check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_dev_ok[dev] == 0) {
    int major = 0, minor = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
    g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    if (g_dev_ok[dev] < 0) {
      g_dev_ok[dev] = -1;
      return fail(ATTN_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev, major,
                  minor);
    }
  }
  if (g_dev_ok[dev] < 0) return fail(ATTN_ERR_UNSUPPORTED, "device %d is not an sm_103 device", dev);
  return ATTN_OK;
}

// ------------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

attn_status get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  return ATTN_OK;
}

// BF16 [B, S, H, 128] with element strides (b, s, h): a 4-D map (d, s, h, b),
// box 64 channels (128 bytes, 128-byte swizzle) x 128 rows.  Rows past S read as zero.
attn_status tmap_bhsd_bf16(CUtensorMap* m, const void* ptr, int B, int S, int H, const long long str[3]) {
  cuuint64_t dims[4] = {128, (cuuint64_t)S, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)str[1] * 2, (cuuint64_t)str[2] * 2, (cuuint64_t)str[0] * 2};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled (BF16 [B,S,H,128]) failed: %d", (int)r);
  return ATTN_OK;
}

// FP16 tensor [n2, n1, 128] (contiguous): a 3-D map with a 64 x 128 element
// box (128 bytes wide, 128-byte swizzle).
attn_status tmap_f16_rows(CUtensorMap* m, const void* ptr, long long n1, long long n2) {
  cuuint64_t dims[3] = {128, (cuuint64_t)n1, (cuuint64_t)n2};
  cuuint64_t strides[2] = {256, (cuuint64_t)(256 * n1)};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled (FP16 rows) failed: %d", (int)r);
  return ATTN_OK;
}

// Byte tensor [n2, n1, n0] (contiguous rows of n0 bytes): a 3-D map with a
// 128 x 128 byte box, 128-byte swizzle.
attn_status tmap_bytes_3d(CUtensorMap* m, const void* ptr, long long n0, long long n1, long long n2) {
  cuuint64_t dims[3] = {(cuuint64_t)n0, (cuuint64_t)n1, (cuuint64_t)n2};
  cuuint64_t strides[2] = {(cuuint64_t)n0, (cuuint64_t)(n0 * n1)};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled (bytes) failed: %d", (int)r);
  return ATTN_OK;
}

// ------------------------------------------------------------------ validation
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The kernels run one CTA per (head, 128 padded positions) at most, numbered along
// grid.x: B * H * S_pad / 128 must stay below 2^31.
attn_status check_grid(int B, int H, long long S_pad) {
  if ((long long)B * H * (S_pad / 128) > 0x7fffffffLL)
    return fail(ATTN_ERR_INVALID_ARG, "B=%d H=%d S_pad=%lld: B*H*S_pad/128 must be below 2^31", B, H, S_pad);
  return ATTN_OK;
}

// B = 0 or H = 0 (no query rows at all) is a valid empty problem: *empty is set and the
// caller returns ATTN_OK without touching its pointers.  S = 0 is an error: attention over
// no keys is undefined.
attn_status check_shape(int B, int S, int H, int D, bool* empty) {
  *empty = false;
  if (D != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dimension D=%d; only D=128 is supported", D);
  if (B < 0 || H < 0) return fail(ATTN_ERR_INVALID_ARG, "B=%d H=%d must be >= 0", B, H);
  if (S < 1) return fail(ATTN_ERR_INVALID_ARG, "S=%d: attention needs at least one key (S >= 1)", S);
  if (B == 0 || H == 0) {
    *empty = true;
    return ATTN_OK;
  }
  return check_grid(B, H, ((long long)S + 127) / 128 * 128);
}

// Strides of a [B, S, H, 128] tensor; a dimension of extent 1 gets a harmless
// stand-in stride (never used to form an address).
attn_status check_strides(const char* name, const void* ptr, const int64_t* in, int B, int S, int H,
                          long long out[3]) {
  if (ptr == nullptr) return fail(ATTN_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(ptr)) return fail(ATTN_ERR_ALIGNMENT, "%s is not 16-byte aligned", name);
  if (in == nullptr) return fail(ATTN_ERR_INVALID_ARG, "%s strides are NULL", name);
  const int ext[3] = {B, S, H};
  const char* dn[3] = {"batch", "sequence", "head"};
  for (int i = 0; i < 3; ++i) {
    long long s = in[i];
    if (ext[i] == 1) s = 128;
    if (s <= 0) return fail(ATTN_ERR_INVALID_ARG, "%s %s stride %lld must be positive", name, dn[i], (long long)in[i]);
    if (s % 8 != 0)
      return fail(ATTN_ERR_ALIGNMENT, "%s %s stride %lld is not a multiple of 8 elements", name, dn[i], s);
    if (s >= (1ll << 38)) return fail(ATTN_ERR_INVALID_ARG, "%s %s stride %lld too large", name, dn[i], s);
    out[i] = s;
  }
  return ATTN_OK;
}

}  // namespace

namespace sa {
namespace {
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;
}  // namespace

cudaError_t current_context_id(unsigned long long* id) {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  });
  if (!g_ctx_current || !g_ctx_id) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (ctx == nullptr) {
    // nothing current on this thread yet: make the current device's primary context
    // current, as the runtime's next call would
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);
    if (e != cudaSuccess) return e;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  }
  if (g_ctx_id(ctx, id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  return cudaSuccess;
}

int device_sm_count() {
  static PerContext<int> cache;
  int n = 0;
  cudaError_t e = cache.get([](int* v) {
    int dev = 0, m = 0;
    cudaError_t r = cudaGetDevice(&dev);
    if (r == cudaSuccess) r = cudaDeviceGetAttribute(&m, cudaDevAttrMultiProcessorCount, dev);
    if (r == cudaSuccess && m <= 0) r = cudaErrorInvalidValue;
    *v = m;
    return r;
  }, &n);
  return e == cudaSuccess ? n : 148;
}
}  // namespace sa

namespace {

#define TRY(x)                          \
  do {                                  \
    attn_status _s = (x);               \
    if (_s != ATTN_OK) return _s;       \
  } while (0)

}  // namespace

extern "C" {

attn_status attn_fwd_bf16(const void* q, const void* k, const void* v, void* o, int B, int S, int H, int D,
                          const int64_t q_str[3], const int64_t k_str[3], const int64_t v_str[3],
                          const int64_t o_str[3], float softmax_scale, attn_stream_t stream) {
  bool empty = false;
  TRY(check_shape(B, S, H, D, &empty));
  if (empty) return ATTN_OK;
  long long qs[3], ks[3], vs[3], os[3];
  TRY(check_strides("q", q, q_str, B, S, H, qs));
  TRY(check_strides("k", k, k_str, B, S, H, ks));
  TRY(check_strides("v", v, v_str, B, S, H, vs));
  TRY(check_strides("o", o, o_str, B, S, H, os));
  if (!std::isfinite(softmax_scale)) return fail(ATTN_ERR_INVALID_ARG, "softmax_scale is not finite");
  TRY(check_device());
  TRY(get_encoder());
  CUtensorMap tq, tk, tv;
  TRY(tmap_bhsd_bf16(&tq, q, B, S, H, qs));
  TRY(tmap_bhsd_bf16(&tk, k, B, S, H, ks));
  TRY(tmap_bhsd_bf16(&tv, v, B, S, H, vs));
  const float c = (float)((double)softmax_scale * kLog2e);
  cudaError_t e = sa::launch_attn_fwd_bf16(tq, tk, tv, o, os[0], os[1], os[2], B, S, H, c, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail_cuda(e, "attn_fwd_bf16 launch");
  return ATTN_OK;
}

int64_t sage_padded_len(int64_t S) { return S <= 0 ? 0 : ((S + 127) / 128) * 128; }

size_t sage_prepare_workspace_size(int B, int H) {
  if (B < 1 || H < 1) return 0;
  return (size_t)B * (size_t)H * 128 * sizeof(uint32_t);
}

// Inputs and options of the prepare stage (shape already checked, not empty): strides,
// softmax scale, S_pad, RMSNorm and RoPE arguments; fills the input side of `a`.
static attn_status prepare_inputs(const void* q, const void* k, const void* v, int B, int S, int H,
                                  const int64_t q_str[3], const int64_t k_str[3], const int64_t v_str[3],
                                  float softmax_scale, const void* q_norm_w, const void* k_norm_w, float rms_eps,
                                  const void* rope_cos, const void* rope_sin, int rope_dim, int64_t S_pad,
                                  sa::PrepareArgs& a) {
  TRY(check_strides("q", q, q_str, B, S, H, a.str[0]));
  TRY(check_strides("k", k, k_str, B, S, H, a.str[1]));
  TRY(check_strides("v", v, v_str, B, S, H, a.str[2]));
  if (!std::isfinite(softmax_scale)) return fail(ATTN_ERR_INVALID_ARG, "softmax_scale is not finite");
  if (S_pad < S || S_pad % 128 != 0)
    return fail(ATTN_ERR_INVALID_ARG, "S_pad=%lld must be a multiple of 128 and >= S=%d", (long long)S_pad, S);
  if (S_pad / 32 > (1ll << 30)) return fail(ATTN_ERR_INVALID_ARG, "S_pad=%lld too large", (long long)S_pad);
  TRY(check_grid(B, H, S_pad));
  if (H > 65535) return fail(ATTN_ERR_INVALID_ARG, "H=%d: the prepare takes at most 65535 heads per batch entry", H);
  if ((q_norm_w == nullptr) != (k_norm_w == nullptr))
    return fail(ATTN_ERR_INVALID_ARG, "q_norm_w and k_norm_w must both be given or both be NULL");
  if (q_norm_w && (!aligned16(q_norm_w) || !aligned16(k_norm_w)))
    return fail(ATTN_ERR_ALIGNMENT, "RMSNorm weights must be 16-byte aligned");
  if (q_norm_w && !(rms_eps >= 0.0f && std::isfinite(rms_eps)))
    return fail(ATTN_ERR_INVALID_ARG, "rms_eps must be finite and >= 0");
  if (!(rope_dim == 0 || rope_dim == 32 || rope_dim == 64 || rope_dim == 96 || rope_dim == 128))
    return fail(ATTN_ERR_INVALID_ARG, "rope_dim=%d must be one of 0, 32, 64, 96, 128", rope_dim);
  if (rope_dim > 0) {
    if (!rope_cos || !rope_sin) return fail(ATTN_ERR_INVALID_ARG, "rope_dim > 0 needs rope_cos and rope_sin");
    if (!aligned16(rope_cos) || !aligned16(rope_sin))
      return fail(ATTN_ERR_ALIGNMENT, "RoPE tables must be 16-byte aligned");
  }
  a.x[0] = q;
  a.x[1] = k;
  a.x[2] = v;
  a.B = B;
  a.S = S;
  a.H = H;
  a.S_pad = S_pad;
  a.q_norm_w = q_norm_w;
  a.k_norm_w = k_norm_w;
  a.rms_eps = rms_eps;
  a.rope_cos = rope_dim > 0 ? rope_cos : nullptr;
  a.rope_sin = rope_dim > 0 ? rope_sin : nullptr;
  a.rope_dim = rope_dim;
  a.c_log2 = (float)((double)softmax_scale * kLog2e);
  return ATTN_OK;
}

// The six prepare outputs: present and 16-byte aligned; then stored into `a`.
static attn_status prepare_outputs(int8_t* q_i8, int8_t* k_i8, uint8_t* v_fp8, float* q_scale, float* k_scale,
                                   float* v_scale, sa::PrepareArgs& a) {
  struct {
    const char* n;
    const void* p;
  } outs[] = {{"q_i8", q_i8}, {"k_i8", k_i8}, {"v_fp8", v_fp8},
              {"q_scale", q_scale}, {"k_scale", k_scale}, {"v_scale", v_scale}};
  for (auto& t : outs) {
    if (!t.p) return fail(ATTN_ERR_INVALID_ARG, "%s is NULL", t.n);
    if (!aligned16(t.p)) return fail(ATTN_ERR_ALIGNMENT, "%s is not 16-byte aligned", t.n);
  }
  a.q_i8 = q_i8;
  a.k_i8 = k_i8;
  a.v_fp8 = v_fp8;
  a.q_scale = q_scale;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  return ATTN_OK;
}

static attn_status prepare_checked(const char* who, const void* q, const void* k, const void* v, int B, int S, int H, int D,
                         const int64_t q_str[3], const int64_t k_str[3], const int64_t v_str[3],
                         float softmax_scale, const void* q_norm_w, const void* k_norm_w, float rms_eps,
                         const void* rope_cos, const void* rope_sin, int rope_dim, int64_t S_pad, int8_t* q_i8,
                         int8_t* k_i8, uint8_t* v_fp8, float* q_scale, float* k_scale, float* v_scale,
                         void* workspace, size_t workspace_bytes, size_t workspace_needed, float* k_mean,
                         void* q_mean16, attn_stream_t stream) {
  bool empty = false;
  TRY(check_shape(B, S, H, D, &empty));
  if (empty) return ATTN_OK;
  sa::PrepareArgs a;
  TRY(prepare_inputs(q, k, v, B, S, H, q_str, k_str, v_str, softmax_scale, q_norm_w, k_norm_w, rms_eps, rope_cos,
                     rope_sin, rope_dim, S_pad, a));
  TRY(prepare_outputs(q_i8, k_i8, v_fp8, q_scale, k_scale, v_scale, a));
  if (!workspace) return fail(ATTN_ERR_INVALID_ARG, "workspace is NULL");
  if (!aligned16(workspace)) return fail(ATTN_ERR_ALIGNMENT, "workspace is not 16-byte aligned");
  if (workspace_bytes < workspace_needed)
    return fail(ATTN_ERR_INVALID_ARG, "%s: workspace_bytes=%zu < %zu required", who, workspace_bytes,
                workspace_needed);
  TRY(check_device());
  a.vmax = reinterpret_cast<uint32_t*>(workspace);
  a.q_mean16 = q_mean16;
  if (k_mean != nullptr) {
    a.k_mean = k_mean;
    // block sums after the V maxima, 16-byte aligned (B*H*128 words is a multiple of 4)
    a.k_partial = reinterpret_cast<float*>(a.vmax + (size_t)B * H * 128);
  }
  cudaError_t e = sa::launch_sage_prepare(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail_cuda(e, who);
  return ATTN_OK;
}

attn_status sage_prepare(const void* q, const void* k, const void* v, int B, int S, int H, int D,
                         const int64_t q_str[3], const int64_t k_str[3], const int64_t v_str[3],
                         float softmax_scale, const void* q_norm_w, const void* k_norm_w, float rms_eps,
                         const void* rope_cos, const void* rope_sin, int rope_dim, int64_t S_pad, int8_t* q_i8,
                         int8_t* k_i8, uint8_t* v_fp8, float* q_scale, float* k_scale, float* v_scale,
                         void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  return prepare_checked("sage_prepare", q, k, v, B, S, H, D, q_str, k_str, v_str, softmax_scale, q_norm_w,
                         k_norm_w, rms_eps, rope_cos, rope_sin, rope_dim, S_pad, q_i8, k_i8, v_fp8, q_scale,
                         k_scale, v_scale, workspace, workspace_bytes, sage_prepare_workspace_size(B, H), nullptr,
                         nullptr, stream);
}

attn_status sage_prepare_noalloc(const void* q, const void* k, const void* v, int B, int S, int H, int D,
                                 const int64_t q_str[3], const int64_t k_str[3], const int64_t v_str[3],
                                 float softmax_scale, const void* q_norm_w, const void* k_norm_w, float rms_eps,
                                 const void* rope_cos, const void* rope_sin, int rope_dim, int64_t S_pad,
                                 int8_t* q_i8, int8_t* k_i8, uint8_t* v_fp8, float* q_scale, float* k_scale,
                                 float* v_scale, attn_stream_t stream) {
  bool empty = false;
  TRY(check_shape(B, S, H, D, &empty));
  if (empty) return ATTN_OK;
  if ((long long)B * H > sa::kNoAllocMaxHeads)
    return fail(ATTN_ERR_INVALID_ARG,
                "sage_prepare_noalloc: B*H=%lld heads exceeds the %d heads its static scratch holds; use "
                "sage_prepare with a caller-allocated workspace",
                (long long)B * H, sa::kNoAllocMaxHeads);
  // the same validation as sage_prepare, short of the workspace
  sa::PrepareArgs a;
  TRY(prepare_inputs(q, k, v, B, S, H, q_str, k_str, v_str, softmax_scale, q_norm_w, k_norm_w, rms_eps, rope_cos,
                     rope_sin, rope_dim, S_pad, a));
  TRY(prepare_outputs(q_i8, k_i8, v_fp8, q_scale, k_scale, v_scale, a));
  TRY(check_device());
  uint32_t* scratch = nullptr;
  cudaError_t e = sa::noalloc_prepare_scratch(&scratch);
  if (e != cudaSuccess) return fail_cuda(e, "sage_prepare_noalloc: looking up the static scratch");
  a.vmax = scratch;  // zeroed on the stream by the launcher before the kernels use it
  e = sa::launch_sage_prepare(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail_cuda(e, "sage_prepare_noalloc launch");
  return ATTN_OK;
}

size_t sage_prepare_smooth_k_workspace_size(int B, int H, int64_t S_pad) {
  if (B < 1 || H < 1 || S_pad < 1) return 0;
  const size_t bh = (size_t)B * (size_t)H;
  return bh * 128 * sizeof(uint32_t) + bh * (size_t)(S_pad / 32) * 128 * sizeof(float);
}

attn_status sage_prepare_smooth_k(const void* q, const void* k, const void* v, int B, int S, int H, int D,
                                  const int64_t q_str[3], const int64_t k_str[3], const int64_t v_str[3],
                                  float softmax_scale, const void* q_norm_w, const void* k_norm_w, float rms_eps,
                                  const void* rope_cos, const void* rope_sin, int rope_dim, int64_t S_pad,
                                  int8_t* q_i8, int8_t* k_i8, uint8_t* v_fp8, float* q_scale, float* k_scale,
                                  float* v_scale, float* k_mean, void* workspace, size_t workspace_bytes,
                                  attn_stream_t stream) {
  bool empty = false;
  TRY(check_shape(B, S, H, D, &empty));
  if (empty) return ATTN_OK;
  if (k_mean == nullptr) return fail(ATTN_ERR_INVALID_ARG, "sage_prepare_smooth_k: k_mean is NULL");
  if (!aligned16(k_mean)) return fail(ATTN_ERR_ALIGNMENT, "sage_prepare_smooth_k: k_mean is not 16-byte aligned");
  return prepare_checked("sage_prepare_smooth_k", q, k, v, B, S, H, D, q_str, k_str, v_str, softmax_scale,
                         q_norm_w, k_norm_w, rms_eps, rope_cos, rope_sin, rope_dim, S_pad, q_i8, k_i8, v_fp8,
                         q_scale, k_scale, v_scale, workspace, workspace_bytes,
                         sage_prepare_smooth_k_workspace_size(B, H, S_pad), k_mean, nullptr, stream);
}

attn_status sage_prepare_smoothed(const void* q, const void* k, const void* v, int B, int S, int H, int D,
                                  const int64_t q_str[3], const int64_t k_str[3], const int64_t v_str[3],
                                  float softmax_scale, const void* q_norm_w, const void* k_norm_w, float rms_eps,
                                  const void* rope_cos, const void* rope_sin, int rope_dim, int64_t S_pad,
                                  int smooth_q, int smooth_k, int8_t* q_i8, int8_t* k_i8, uint8_t* v_fp8,
                                  float* q_scale, float* k_scale, float* v_scale, void* q_mean, float* k_mean,
                                  void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  bool empty = false;
  TRY(check_shape(B, S, H, D, &empty));
  if (empty) return ATTN_OK;
  if ((smooth_q != 0 && smooth_q != 1) || (smooth_k != 0 && smooth_k != 1))
    return fail(ATTN_ERR_INVALID_ARG, "smooth_q=%d and smooth_k=%d must be 0 or 1", smooth_q, smooth_k);
  if (smooth_q) {
    if (q_mean == nullptr) return fail(ATTN_ERR_INVALID_ARG, "sage_prepare_smoothed: smooth_q needs q_mean");
    if (!aligned16(q_mean)) return fail(ATTN_ERR_ALIGNMENT, "sage_prepare_smoothed: q_mean is not 16-byte aligned");
  }
  if (smooth_k) {
    if (k_mean == nullptr) return fail(ATTN_ERR_INVALID_ARG, "sage_prepare_smoothed: smooth_k needs k_mean");
    if (!aligned16(k_mean)) return fail(ATTN_ERR_ALIGNMENT, "sage_prepare_smoothed: k_mean is not 16-byte aligned");
  }
  const size_t need = smooth_k ? sage_prepare_smooth_k_workspace_size(B, H, S_pad) : sage_prepare_workspace_size(B, H);
  return prepare_checked("sage_prepare_smoothed", q, k, v, B, S, H, D, q_str, k_str, v_str, softmax_scale, q_norm_w,
                         k_norm_w, rms_eps, rope_cos, rope_sin, rope_dim, S_pad, q_i8, k_i8, v_fp8, q_scale, k_scale,
                         v_scale, workspace, workspace_bytes, need, smooth_k ? k_mean : nullptr,
                         smooth_q ? q_mean : nullptr, stream);
}

size_t sage_attn_workspace_size(int B, int H, int64_t S_pad) {
  if (B < 1 || H < 1 || S_pad < 1) return 0;
  return (size_t)4 * (size_t)B * (size_t)H * (size_t)S_pad * 128;
}

// The two-call forwards: the codes widened to the FP16 score operands (Q's carrying its
// block means with Q smoothing), then the attention kernel in the chosen P V mode.
static attn_status attn_fwd_prepared(const char* who, const int8_t* q_i8, const void* q_mean, const int8_t* k_i8,
                                     const float* q_scale, const float* k_scale, const uint8_t* v_fp8,
                                     const float* v_scale, const void* v, const int64_t v_str[3], int pv_bf16,
                                     void* o, const int64_t o_str[3], int B, int S, int H, int D, int64_t S_pad,
                                     void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  bool empty = false;
  TRY(check_shape(B, S, H, D, &empty));
  if (empty) return ATTN_OK;
  if (S_pad < S || S_pad % 128 != 0)
    return fail(ATTN_ERR_INVALID_ARG, "S_pad=%lld must be a multiple of 128 and >= S=%d", (long long)S_pad, S);
  if (S_pad > (1ll << 31) - 256) return fail(ATTN_ERR_INVALID_ARG, "S_pad=%lld too large", (long long)S_pad);
  TRY(check_grid(B, H, S_pad));
  struct In {
    const char* n;
    const void* p;
    bool needed;
  } ins[] = {{"q_i8", q_i8, true},        {"k_i8", k_i8, true},          {"q_scale", q_scale, true},
             {"k_scale", k_scale, true},  {"workspace", workspace, true}, {"v_fp8", v_fp8, !pv_bf16},
             {"v_scale", v_scale, !pv_bf16}, {"q_mean", q_mean, q_mean != nullptr}};
  for (const In& t : ins) {
    if (!t.needed) continue;
    if (!t.p) return fail(ATTN_ERR_INVALID_ARG, "%s is NULL", t.n);
    if (!aligned16(t.p)) return fail(ATTN_ERR_ALIGNMENT, "%s is not 16-byte aligned", t.n);
  }
  if (workspace_bytes < sage_attn_workspace_size(B, H, S_pad))
    return fail(ATTN_ERR_INVALID_ARG, "workspace_bytes=%zu < %zu required", workspace_bytes,
                sage_attn_workspace_size(B, H, S_pad));
  long long vs[3], os[3];
  if (pv_bf16) TRY(check_strides("v", v, v_str, B, S, H, vs));
  TRY(check_strides("o", o, o_str, B, S, H, os));
  TRY(check_device());
  TRY(get_encoder());
  const long long bh = (long long)B * H;
  const long long n_codes = bh * S_pad * 128;
  uint8_t* q16 = reinterpret_cast<uint8_t*>(workspace);
  uint8_t* k16 = q16 + 2 * n_codes;
  CUtensorMap tq, tk, tv;
  TRY(tmap_f16_rows(&tq, q16, S_pad, bh));
  TRY(tmap_f16_rows(&tk, k16, S_pad, bh));
  if (pv_bf16) TRY(tmap_bhsd_bf16(&tv, v, B, S, H, vs));
  else TRY(tmap_bytes_3d(&tv, v_fp8, S_pad, 128, bh));
  cudaError_t e = sa::launch_sage_widen(q_i8, k_i8, q16, k16, n_codes, sa::device_sm_count(), (cudaStream_t)stream);
  if (e == cudaSuccess && q_mean != nullptr)   // Q's operand again, now with its block means
    e = sa::launch_widen_q_mean(q_i8, q_mean, q16, n_codes, sa::device_sm_count(), (cudaStream_t)stream);
  if (e != cudaSuccess) return fail_cuda(e, who);
  if (pv_bf16)
    e = sa::launch_sage_attn_pv16(tq, tk, tv, q_scale, k_scale, o, os[0], os[1], os[2], B, S, H, S_pad,
                                  (cudaStream_t)stream);
  else
    e = sa::launch_sage_attn(tq, tk, tv, q_scale, k_scale, v_scale, o, os[0], os[1], os[2], B, S, H, S_pad,
                             (cudaStream_t)stream);
  if (e != cudaSuccess) return fail_cuda(e, who);
  return ATTN_OK;
}

attn_status sage_attn_fwd(const int8_t* q_i8, const int8_t* k_i8, const uint8_t* v_fp8, const float* q_scale,
                          const float* k_scale, const float* v_scale, void* o, const int64_t o_str[3], int B,
                          int S, int H, int D, int64_t S_pad, void* workspace, size_t workspace_bytes,
                          attn_stream_t stream) {
  return attn_fwd_prepared("sage_attn_fwd", q_i8, nullptr, k_i8, q_scale, k_scale, v_fp8, v_scale, nullptr, nullptr,
                           0, o, o_str, B, S, H, D, S_pad, workspace, workspace_bytes, stream);
}

attn_status sage_attn_fwd_pv16(const int8_t* q_i8, const int8_t* k_i8, const float* q_scale, const float* k_scale,
                               const void* v, const int64_t v_str[3], void* o, const int64_t o_str[3], int B, int S,
                               int H, int D, int64_t S_pad, void* workspace, size_t workspace_bytes,
                               attn_stream_t stream) {
  return attn_fwd_prepared("sage_attn_fwd_pv16", q_i8, nullptr, k_i8, q_scale, k_scale, nullptr, nullptr, v, v_str,
                           1, o, o_str, B, S, H, D, S_pad, workspace, workspace_bytes, stream);
}

attn_status sage_attn_fwd_smooth_q(const int8_t* q_i8, const void* q_mean, const int8_t* k_i8,
                                   const uint8_t* v_fp8, const float* q_scale, const float* k_scale,
                                   const float* v_scale, void* o, const int64_t o_str[3], int B, int S, int H, int D,
                                   int64_t S_pad, void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  if (q_mean == nullptr) return fail(ATTN_ERR_INVALID_ARG, "q_mean is NULL");
  return attn_fwd_prepared("sage_attn_fwd_smooth_q", q_i8, q_mean, k_i8, q_scale, k_scale, v_fp8, v_scale, nullptr,
                           nullptr, 0, o, o_str, B, S, H, D, S_pad, workspace, workspace_bytes, stream);
}

attn_status sage_attn_fwd_pv16_smooth_q(const int8_t* q_i8, const void* q_mean, const int8_t* k_i8,
                                        const float* q_scale, const float* k_scale, const void* v,
                                        const int64_t v_str[3], void* o, const int64_t o_str[3], int B, int S, int H,
                                        int D, int64_t S_pad, void* workspace, size_t workspace_bytes,
                                        attn_stream_t stream) {
  if (q_mean == nullptr) return fail(ATTN_ERR_INVALID_ARG, "q_mean is NULL");
  return attn_fwd_prepared("sage_attn_fwd_pv16_smooth_q", q_i8, q_mean, k_i8, q_scale, k_scale, nullptr, nullptr, v,
                           v_str, 1, o, o_str, B, S, H, D, S_pad, workspace, workspace_bytes, stream);
}

// Workspace of sage_attention: consecutive 256-byte aligned pieces.
// The one-call op's workspace: Q's FP16 codes and scales (unless the forward codes Q
// as it loads it), K's, V's codes and scales (FP8 mode), the smoothing buffers.
struct FusedLayout {
  size_t q16, q_scale, q_mean, k16, k_scale, v_fp8, v_scale, vmax, k_mean, k_partial, total;
};
static FusedLayout fused_layout(int B, int H, int64_t S_pad, int smooth_k, int pv_bf16, int q_on_load) {
  FusedLayout L{};
  const size_t bh = (size_t)B * (size_t)H, nblk = (size_t)(S_pad / 32);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += (bytes + 255) & ~size_t(255);
    return at;
  };
  if (!q_on_load) {
    L.q16 = take(bh * (size_t)S_pad * 128 * 2);
    L.q_scale = take(bh * nblk * 4);
    L.q_mean = take(bh * nblk * 128 * 2);   // used with Q smoothing only
  }
  if (q_on_load < 2) {
    L.k16 = take(bh * (size_t)S_pad * 128 * 2);
    L.k_scale = take(bh * nblk * 4);
  }
  if (!pv_bf16) {
    L.v_fp8 = take(bh * 128 * (size_t)S_pad);
    L.v_scale = take(bh * 128 * 4);
    L.vmax = take(bh * 128 * 4);
  }
  if (smooth_k) {
    L.k_mean = take(bh * 128 * 4);
    L.k_partial = take(bh * nblk * 128 * 4);
  }
  L.total = off;
  return L;
}

size_t sage_attention_workspace_size(int B, int H, int64_t S_pad, int smooth_k, int pv_bf16, int q_on_load) {
  if (B < 1 || H < 1 || S_pad < 1) return 0;
  return fused_layout(B, H, S_pad, smooth_k, pv_bf16, q_on_load).total;
}

attn_status sage_attention(const void* q, const void* k, const void* v, int B, int S, int H, int D,
                           const int64_t q_str[3], const int64_t k_str[3], const int64_t v_str[3],
                           float softmax_scale, const void* q_norm_w, const void* k_norm_w, float rms_eps,
                           const void* rope_cos, const void* rope_sin, int rope_dim, int smooth_q, int smooth_k,
                           int pv_bf16, int q_on_load, void* o, const int64_t o_str[3], void* workspace,
                           size_t workspace_bytes, attn_stream_t stream) {
  bool empty = false;
  TRY(check_shape(B, S, H, D, &empty));
  if (empty) return ATTN_OK;
  if ((smooth_q != 0 && smooth_q != 1) || (smooth_k != 0 && smooth_k != 1) || (pv_bf16 != 0 && pv_bf16 != 1) ||
      q_on_load < 0 || q_on_load > 2)
    return fail(ATTN_ERR_INVALID_ARG, "smooth_q=%d, smooth_k=%d and pv_bf16=%d must be 0 or 1, q_on_load=%d 0, 1 or 2",
                smooth_q, smooth_k, pv_bf16, q_on_load);
  if (smooth_q && q_on_load)
    return fail(ATTN_ERR_UNSUPPORTED, "smooth_q with q_on_load: the forward codes Q without block means");
  if (smooth_k && q_on_load == 2)
    return fail(ATTN_ERR_UNSUPPORTED, "smooth_k with K coded on load: the sequence mean of K needs its own pass");
  const int64_t S_pad = sage_padded_len(S);
  sa::PrepareArgs a;
  TRY(prepare_inputs(q, k, v, B, S, H, q_str, k_str, v_str, softmax_scale, q_norm_w, k_norm_w, rms_eps, rope_cos,
                     rope_sin, rope_dim, S_pad, a));
  long long os[3];
  TRY(check_strides("o", o, o_str, B, S, H, os));
  const FusedLayout L = fused_layout(B, H, S_pad, smooth_k, pv_bf16, q_on_load);
  // with the 16-bit P V and Q and K coded on load nothing is prepared: no workspace at all
  if (L.total > 0 && !workspace) return fail(ATTN_ERR_INVALID_ARG, "workspace is NULL");
  if (!aligned16(workspace)) return fail(ATTN_ERR_ALIGNMENT, "workspace is not 16-byte aligned");
  if (workspace_bytes < L.total)
    return fail(ATTN_ERR_INVALID_ARG, "sage_attention: workspace_bytes=%zu < %zu required", workspace_bytes, L.total);
  TRY(check_device());
  TRY(get_encoder());
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  if (!q_on_load) {
    a.q16 = ws + L.q16;
    a.q_scale = reinterpret_cast<float*>(ws + L.q_scale);
  }
  if (q_on_load < 2) {
    a.k16 = ws + L.k16;
    a.k_scale = reinterpret_cast<float*>(ws + L.k_scale);
  }
  a.skip_q = q_on_load != 0;  // else the forward codes Q as it loads it
  a.skip_k = q_on_load == 2;  // ... and K
  a.skip_v = pv_bf16 != 0;
  // Q smoothing: the means go to the workspace; the FP16 Q operand already carries them
  if (smooth_q) a.q_mean16 = ws + L.q_mean;
  if (!pv_bf16) {
    a.v_fp8 = ws + L.v_fp8;
    a.v_scale = reinterpret_cast<float*>(ws + L.v_scale);
    a.vmax = reinterpret_cast<uint32_t*>(ws + L.vmax);
  }
  if (smooth_k) {
    a.k_mean = reinterpret_cast<float*>(ws + L.k_mean);
    a.k_partial = reinterpret_cast<float*>(ws + L.k_partial);
  }
  // (nothing to prepare when the forward codes Q and K and V stays in BF16)
  cudaError_t e = (q_on_load == 2 && pv_bf16) ? cudaSuccess : sa::launch_sage_prepare(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail_cuda(e, "sage_attention prepare");
  const long long bh = (long long)B * H;
  CUtensorMap tq, tk, tv;
  if (q_on_load == 2) {
    // Q and K are coded by the forward: both through their BF16 [B, S, H, 128] maps
    TRY(tmap_bhsd_bf16(&tq, q, B, S, H, a.str[0]));
    TRY(tmap_bhsd_bf16(&tk, k, B, S, H, a.str[1]));
    sa::QLoadArgs qa;
    qa.q_norm_w = a.q_norm_w;
    qa.k_norm_w = a.k_norm_w;
    qa.rms_eps = a.rms_eps;
    qa.rope_cos = a.rope_cos;
    qa.rope_sin = a.rope_sin;
    qa.rope_dim = a.rope_dim;
    qa.c_log2 = a.c_log2;
    if (pv_bf16) {
      TRY(tmap_bhsd_bf16(&tv, v, B, S, H, a.str[2]));
      e = sa::launch_sage_attn_pv16_qkload(tq, tk, tv, qa, o, os[0], os[1], os[2], B, S, H, S_pad, (cudaStream_t)stream);
    } else {
      TRY(tmap_bytes_3d(&tv, a.v_fp8, S_pad, 128, bh));
      e = sa::launch_sage_attn_qkload(tq, tk, tv, qa, a.v_scale, o, os[0], os[1], os[2], B, S, H, S_pad,
                                      (cudaStream_t)stream);
    }
    if (e != cudaSuccess) return fail_cuda(e, "sage_attention launch");
    return ATTN_OK;
  }
  TRY(tmap_f16_rows(&tk, a.k16, S_pad, bh));
  if (!q_on_load) {
    TRY(tmap_f16_rows(&tq, a.q16, S_pad, bh));
    if (pv_bf16) {
      TRY(tmap_bhsd_bf16(&tv, v, B, S, H, a.str[2]));
      e = sa::launch_sage_attn_pv16(tq, tk, tv, a.q_scale, a.k_scale, o, os[0], os[1], os[2], B, S, H, S_pad,
                                    (cudaStream_t)stream);
    } else {
      TRY(tmap_bytes_3d(&tv, a.v_fp8, S_pad, 128, bh));
      e = sa::launch_sage_attn(tq, tk, tv, a.q_scale, a.k_scale, a.v_scale, o, os[0], os[1], os[2], B, S, H,
                               S_pad, (cudaStream_t)stream);
    }
    if (e != cudaSuccess) return fail_cuda(e, "sage_attention launch");
    return ATTN_OK;
  }
  TRY(tmap_bhsd_bf16(&tq, q, B, S, H, a.str[0]));
  sa::QLoadArgs qa;
  qa.q_norm_w = a.q_norm_w;
  qa.rms_eps = a.rms_eps;
  qa.rope_cos = a.rope_cos;
  qa.rope_sin = a.rope_sin;
  qa.rope_dim = a.rope_dim;
  qa.c_log2 = a.c_log2;
  if (pv_bf16) {
    TRY(tmap_bhsd_bf16(&tv, v, B, S, H, a.str[2]));
    e = sa::launch_sage_attn_pv16_qload(tq, tk, tv, qa, a.k_scale, o, os[0], os[1], os[2], B, S, H, S_pad,
                                        (cudaStream_t)stream);
  } else {
    TRY(tmap_bytes_3d(&tv, a.v_fp8, S_pad, 128, bh));
    e = sa::launch_sage_attn_qload(tq, tk, tv, qa, a.k_scale, a.v_scale, o, os[0], os[1], os[2], B, S, H, S_pad,
                                   (cudaStream_t)stream);
  }
  if (e != cudaSuccess) return fail_cuda(e, "sage_attention launch");
  return ATTN_OK;
}

attn_status attn_selftest_wait_timeout(const void* q, const void* k, const void* v, void* o,
                                       attn_stream_t stream) {
  const int64_t st[3] = {128 * 128, 128, 128};   // [1, 128, 1, 128] contiguous
  long long qs[3], ks[3], vs[3], os[3];
  TRY(check_strides("q", q, st, 1, 128, 1, qs));
  TRY(check_strides("k", k, st, 1, 128, 1, ks));
  TRY(check_strides("v", v, st, 1, 128, 1, vs));
  TRY(check_strides("o", o, st, 1, 128, 1, os));
  TRY(check_device());
  TRY(get_encoder());
  // start from a clean error word, so that the status below is this launch's
  attn_status pre = attn_get_device_status(stream);
  if (pre != ATTN_OK && pre != ATTN_ERR_DEVICE_TIMEOUT) return pre;
  CUtensorMap tq, tk, tv;
  TRY(tmap_bhsd_bf16(&tq, q, 1, 128, 1, qs));
  TRY(tmap_bhsd_bf16(&tk, k, 1, 128, 1, ks));
  TRY(tmap_bhsd_bf16(&tv, v, 1, 128, 1, vs));
  const float c = (float)(0.08838834764831845 * kLog2e);
  cudaError_t e = sa::launch_attn_fwd_bf16(tq, tk, tv, o, os[0], os[1], os[2], 1, 128, 1, c, (cudaStream_t)stream,
                                           /*withhold_loads=*/true);
  if (e != cudaSuccess) return fail_cuda(e, "attn_selftest_wait_timeout launch");
  return attn_get_device_status(stream);
}

attn_status attn_get_device_status(attn_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
  uint32_t w = 0;
  e = sa::read_and_clear_err_attn(&w);
  if (e != cudaSuccess) return fail_cuda(e, "reading the device error word");
  if (w)
    return fail(ATTN_ERR_DEVICE_TIMEOUT,
                "an attention kernel gave up on a bounded wait (bits 0x%x: 1 TMA load, 2 MMA commit, 4 hand-off; "
                "0x100 a check build's TMEM-maximum mismatch)", w);
  return ATTN_OK;
}

attn_status attn_sm_clock_sample(uint64_t* out, int n_slots, attn_stream_t stream) {
  if (out == nullptr) return fail(ATTN_ERR_INVALID_ARG, "out is NULL");
  if (!aligned16(out)) return fail(ATTN_ERR_ALIGNMENT, "out is not 16-byte aligned");
  if (n_slots < 1) return fail(ATTN_ERR_INVALID_ARG, "n_slots=%d must be >= 1", n_slots);
  TRY(check_device());
  cudaError_t e = sa::launch_sm_clock_probe(reinterpret_cast<unsigned long long*>(out), n_slots,
                                            sa::device_sm_count(), (cudaStream_t)stream);
  if (e != cudaSuccess) return fail_cuda(e, "attn_sm_clock_sample launch");
  return ATTN_OK;
}

attn_status sage_e4m3_encode(const float* x, uint8_t* y, int64_t n, attn_stream_t stream) {
  if (n < 0) return fail(ATTN_ERR_INVALID_ARG, "sage_e4m3_encode: n=%lld must be >= 0", (long long)n);
  if (n == 0) return ATTN_OK;
  if (x == nullptr || y == nullptr) return fail(ATTN_ERR_INVALID_ARG, "sage_e4m3_encode: x or y is NULL");
  TRY(check_device());
  cudaError_t e = sa::launch_e4m3_encode(x, y, (long long)n, sa::device_sm_count(), (cudaStream_t)stream);
  if (e != cudaSuccess) return fail_cuda(e, "sage_e4m3_encode launch");
  return ATTN_OK;
}

const char* attn_last_error(void) { return g_msg; }

const char* attn_status_name(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_ALIGNMENT: return "ATTN_ERR_ALIGNMENT";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_DEVICE_TIMEOUT: return "ATTN_ERR_DEVICE_TIMEOUT";
  }
  return "ATTN_UNKNOWN_STATUS";
}

}  // extern "C"
